// The MXFP8 MoE SwiGLU layer, forward and backward, composed from the
// library's kernels on the caller's stream ("1.5x faster MoE training on
// Blackwell with MXFP8 kernels built from scratch", Overview: the MoE layer
// rebuilt on MXFP8 kernels for both passes; pytorch/ao "mxfp8 moe training"
// PR, Next steps: stay in MXFP8 from the token shuffle through the grouped
// GEMM).  No host synchronization anywhere: group sizes never leave the
// device.
//
// Forward:  route -> map -> permute+quantize x -> GEMM1 (+SwiGLU, quantize h)
//           -> GEMM2 -> combine.
// Backward: gate grad; gather+quantize dY (row and column) -> dgrad2 (dh) ->
//           SwiGLU backward + quantize (row and column) -> wgrad2 -> dgrad1 ->
//           gather+column-quantize x -> wgrad1 -> combine (unit gates).
#include "common.cuh"

extern "C" mx_status moe_gather_quant(const void *x, const float *gate, const int32_t *src, int64_t T, int64_t H,
                                      int32_t k, int64_t rows_cap, int32_t mode, int32_t elem, uint8_t *q_row,
                                      uint8_t *s_row, uint8_t *q_col, uint8_t *s_col, const int32_t *row_limit,
                                      mx_stream stream);
extern "C" mx_status moe_gate_grad(const void *dOut, const void *y, const int32_t *dst, int64_t T, int64_t H,
                                   int32_t k, float *d_gate, mx_stream stream);

namespace mxmoe {

struct Carver {
  uint8_t *base;
  int64_t off = 0;
  template <class T>
  T *take(int64_t bytes) {
    T *p = reinterpret_cast<T *>(base ? base + off : nullptr);
    off += round_up(bytes, 256);
    return p;
  }
};

struct WeightsView {
  uint8_t *w13_cq, *w13_cs;  // [E, 2F, H] (forward GEMM1 B), scales (E*2F, H)
  uint8_t *w13_rq, *w13_rs;  // [E, H, 2F] (dgrad1 B), scales (E*H, 2F)
  uint8_t *w2_cq, *w2_cs;    // [E, H, F] (forward GEMM2 B), scales (E*H, F)
  uint8_t *w2_rq, *w2_rs;    // [E, F, H] (dgrad2 B), scales (E*F, H)
};

static int64_t carve_weights(void *base, int64_t H, int64_t F, int64_t E, WeightsView *v) {
  Carver c{static_cast<uint8_t *>(base)};
  v->w13_cq = c.take<uint8_t>(E * 2 * F * H);
  v->w13_cs = c.take<uint8_t>(mx_scale_bytes(E * 2 * F, H, MX_SCALE_SWIZZLED));
  v->w13_rq = c.take<uint8_t>(E * H * 2 * F);
  v->w13_rs = c.take<uint8_t>(mx_scale_bytes(E * H, 2 * F, MX_SCALE_SWIZZLED));
  v->w2_cq = c.take<uint8_t>(E * H * F);
  v->w2_cs = c.take<uint8_t>(mx_scale_bytes(E * H, F, MX_SCALE_SWIZZLED));
  v->w2_rq = c.take<uint8_t>(E * F * H);
  v->w2_rs = c.take<uint8_t>(mx_scale_bytes(E * F, H, MX_SCALE_SWIZZLED));
  return c.off;
}

struct Workspace {
  int32_t *counts, *offsets, *dst, *src;
  void *map_ws;
  int64_t map_ws_bytes;
  uint8_t *xq, *xs;      // permuted, quantized x: [R, H]
  uint16_t *ab;          // saved a | b: [R, 2F] bf16
  uint8_t *hq, *hs;      // quantized h: [R, F]
  uint16_t *y;           // GEMM2 output: [R, H] bf16
  // backward scratch
  uint8_t *dy_rq, *dy_rs;    // [R, H]
  uint8_t *dy_cq, *dy_cs;    // [H, R]
  float *dh;                 // [R, F]
  uint8_t *dab_rq, *dab_rs;  // [R, 2F]
  uint8_t *dab_cq, *dab_cs;  // [2F, R]
  uint8_t *h_cq, *h_cs;      // [F, R]
  uint8_t *xp_cq, *xp_cs;    // [H, R]
  uint16_t *dxp;             // [R, H] bf16
  int64_t R;
};

static int64_t carve_ws(void *base, int64_t T, int64_t H, int64_t F, int32_t E, int32_t k, Workspace *w) {
  Carver c{static_cast<uint8_t *>(base)};
  const int64_t R = moe_rows_cap(T, k, E);
  w->R = R;
  w->counts = c.take<int32_t>(E * 4);
  w->offsets = c.take<int32_t>((E + 1) * 4);
  w->dst = c.take<int32_t>(T * k * 4);
  w->src = c.take<int32_t>(R * 4);
  w->map_ws_bytes = moe_permute_map_workspace_size(T, k, E);
  w->map_ws = c.take<uint8_t>(w->map_ws_bytes);
  w->xq = c.take<uint8_t>(R * H);
  w->xs = c.take<uint8_t>(mx_scale_bytes(R, H, MX_SCALE_SWIZZLED));
  w->ab = c.take<uint16_t>(R * 2 * F * 2);
  w->hq = c.take<uint8_t>(R * F);
  w->hs = c.take<uint8_t>(mx_scale_bytes(R, F, MX_SCALE_SWIZZLED));
  w->y = c.take<uint16_t>(R * H * 2);
  w->dy_rq = c.take<uint8_t>(R * H);
  w->dy_rs = c.take<uint8_t>(mx_scale_bytes(R, H, MX_SCALE_SWIZZLED));
  w->dy_cq = c.take<uint8_t>(H * R);
  w->dy_cs = c.take<uint8_t>(mx_scale_bytes(H, R, MX_SCALE_SWIZZLED));
  w->dh = c.take<float>(R * F * 4);
  w->dab_rq = c.take<uint8_t>(R * 2 * F);
  w->dab_rs = c.take<uint8_t>(mx_scale_bytes(R, 2 * F, MX_SCALE_SWIZZLED));
  w->dab_cq = c.take<uint8_t>(2 * F * R);
  w->dab_cs = c.take<uint8_t>(mx_scale_bytes(2 * F, R, MX_SCALE_SWIZZLED));
  w->h_cq = c.take<uint8_t>(F * R);
  w->h_cs = c.take<uint8_t>(mx_scale_bytes(F, R, MX_SCALE_SWIZZLED));
  w->xp_cq = c.take<uint8_t>(H * R);
  w->xp_cs = c.take<uint8_t>(mx_scale_bytes(H, R, MX_SCALE_SWIZZLED));
  w->dxp = c.take<uint16_t>(R * H * 2);
  return c.off;
}

static mx_status check_dims(int64_t T, int64_t H, int64_t F, int32_t E, int32_t k) {
  if (T < 0 || H < 1 || F < 1 || E < 1 || E > 256 || k < 1 || k > E || k > 8) return MX_ERR_INVALID_ARG;
  if (H % 256 || F % 256) return MX_ERR_SHAPE;
  return MX_OK;
}

}  // namespace mxmoe

using namespace mxmoe;

#define MX_TRY(expr)                     \
  do {                                   \
    mx_status _s = (expr);               \
    if (_s != MX_OK) return _s;          \
  } while (0)

extern "C" int64_t moe_layer_weights_size(int64_t H, int64_t F, int32_t E) {
  if (H < 1 || F < 1 || E < 1) return -1;
  WeightsView v;
  return carve_weights(nullptr, H, F, E, &v);
}

extern "C" int64_t moe_layer_workspace_size(int64_t T, int64_t H, int64_t F, int32_t E, int32_t k) {
  if (check_dims(T, H, F, E, k) == MX_ERR_INVALID_ARG) return -1;
  Workspace w;
  return carve_ws(nullptr, T, H, F, E, k, &w);
}

extern "C" mx_status moe_layer_prep_weights(const void *W13, const void *W2, int64_t H, int64_t F, int32_t E,
                                            void *wq, int64_t wq_bytes, mx_stream stream) {
  MX_HOST_CHECK(W13 && W2 && wq, MX_ERR_INVALID_ARG);
  MX_TRY(check_dims(1, H, F, E, 1));
  MX_HOST_CHECK(wq_bytes >= moe_layer_weights_size(H, F, E), MX_ERR_WORKSPACE);
  WeightsView v;
  carve_weights(wq, H, F, E, &v);
  // W13[e] is [H, 2F]: ROW blocks run along 2F (dgrad1), COL blocks along H (forward)
  MX_TRY(mx_quantize(W13, E, H, 2 * F, MX_MODE_BOTH, MX_SCALE_SWIZZLED, MX_ELEM_E4M3, v.w13_rq, v.w13_rs, v.w13_cq,
                     v.w13_cs, stream));
  // W2[e] is [F, H]: ROW blocks along H (dgrad2), COL blocks along F (forward)
  MX_TRY(mx_quantize(W2, E, F, H, MX_MODE_BOTH, MX_SCALE_SWIZZLED, MX_ELEM_E4M3, v.w2_rq, v.w2_rs, v.w2_cq, v.w2_cs,
                     stream));
  return MX_OK;
}

extern "C" mx_status moe_layer_fwd(const void *x, const float *logits, int32_t *ids, float *gate, const void *wq,
                                   int64_t T, int64_t H, int64_t F, int32_t E, int32_t k, void *ws,
                                   int64_t ws_bytes, void *out, int32_t *dev_status, mx_stream stream) {
  MX_HOST_CHECK(wq && ws && (T == 0 || (x && ids && out)), MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(!logits || gate, MX_ERR_INVALID_ARG);
  MX_TRY(check_dims(T, H, F, E, k));
  MX_HOST_CHECK(ws_bytes >= moe_layer_workspace_size(T, H, F, E, k), MX_ERR_WORKSPACE);
  WeightsView v;
  carve_weights(const_cast<void *>(wq), H, F, E, &v);
  Workspace w;
  carve_ws(ws, T, H, F, E, k, &w);
  const int64_t R = w.R;
  if (logits) MX_TRY(moe_route(logits, T, E, k, ids, gate, stream));
  MX_TRY(moe_permute_map(ids, T, k, E, R, w.counts, w.offsets, w.dst, w.src, w.map_ws, w.map_ws_bytes, dev_status,
                         stream));
  MX_TRY(moe_permute(MX_PERMUTE_BF16_QUANT, x, nullptr, T, H, k, w.dst, w.src, R, w.xq, w.xs, MX_SCALE_SWIZZLED,
                     stream));
  MX_TRY(moe_gemm1_swiglu(w.xq, w.xs, v.w13_cq, v.w13_cs, w.offsets, E, R, F, H, w.ab, w.hq, w.hs, dev_status,
                          stream));
  MX_TRY(mx_grouped_gemm(MX_GEMM_FWD, w.hq, w.hs, v.w2_cq, v.w2_cs, w.offsets, E, R, H, F, w.y, MX_OUT_BF16,
                         MX_ELEM_E4M3, MX_ELEM_E4M3, dev_status, stream));
  MX_TRY(moe_unpermute(w.y, w.dst, gate, T, H, k, out, stream));
  return MX_OK;
}

extern "C" mx_status moe_layer_bwd(const void *x, const void *dOut, const float *gate, const void *wq, int64_t T,
                                   int64_t H, int64_t F, int32_t E, int32_t k, int32_t grad_elem,
                                   int32_t wgrad_dtype, void *ws, int64_t ws_bytes, void *dX, void *dW13, void *dW2,
                                   float *d_gate, int32_t *dev_status, mx_stream stream) {
  MX_HOST_CHECK(wq && ws && dW13 && dW2 && (T == 0 || (x && dOut && dX)), MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(grad_elem == MX_ELEM_E4M3 || grad_elem == MX_ELEM_E5M2, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(wgrad_dtype == MX_OUT_F32 || wgrad_dtype == MX_OUT_BF16, MX_ERR_INVALID_ARG);
  const int32_t ge = grad_elem, e4 = MX_ELEM_E4M3;
  MX_TRY(check_dims(T, H, F, E, k));
  MX_HOST_CHECK(ws_bytes >= moe_layer_workspace_size(T, H, F, E, k), MX_ERR_WORKSPACE);
  WeightsView v;
  carve_weights(const_cast<void *>(wq), H, F, E, &v);
  Workspace w;
  carve_ws(ws, T, H, F, E, k, &w);
  const int64_t R = w.R;
  if (d_gate) MX_TRY(moe_gate_grad(dOut, w.y, w.dst, T, H, k, d_gate, stream));
  // dY rows = gate * dOut, quantized along H (dgrad2) and along tokens (wgrad2)
  // (rows past offsets[E], the end of the routed rows, are skipped on the device)
  const int32_t *row_limit = w.offsets + E;
  MX_TRY(moe_gather_quant(dOut, gate, w.src, T, H, k, R, MX_MODE_BOTH, ge, w.dy_rq, w.dy_rs, w.dy_cq, w.dy_cs,
                          row_limit, stream));
  // dh = dY W2^T : B = W2[e] [F, H] quantized along H
  MX_TRY(mx_grouped_gemm(MX_GEMM_DGRAD, w.dy_rq, w.dy_rs, v.w2_rq, v.w2_rs, w.offsets, E, R, F, H, w.dh,
                         MX_OUT_F32, ge, e4, dev_status, stream));
  MX_TRY(moe_swiglu_bwd(w.dh, w.ab, R, F, ge, w.dab_rq, w.dab_rs, w.dab_cq, w.dab_cs, w.h_cq, w.h_cs, row_limit,
                        stream));
  // dW2[e] = h^T dY over the expert's tokens -> [F, H]
  MX_TRY(mx_grouped_gemm(MX_GEMM_WGRAD, w.h_cq, w.h_cs, w.dy_cq, w.dy_cs, w.offsets, E, R, F, H, dW2, wgrad_dtype,
                         e4, ge, dev_status, stream));
  // dxp = dab W13^T : B = W13[e] [H, 2F] quantized along 2F
  MX_TRY(mx_grouped_gemm(MX_GEMM_DGRAD, w.dab_rq, w.dab_rs, v.w13_rq, v.w13_rs, w.offsets, E, R, H, 2 * F, w.dxp,
                         MX_OUT_BF16, ge, e4, dev_status, stream));
  // x permuted (bf16) and quantized along tokens for wgrad1
  MX_TRY(moe_gather_quant(x, nullptr, w.src, T, H, k, R, MX_MODE_COL, e4, nullptr, nullptr, w.xp_cq, w.xp_cs,
                          row_limit, stream));
  // dW13[e] = xp^T dab over the expert's tokens -> [H, 2F]
  MX_TRY(mx_grouped_gemm(MX_GEMM_WGRAD, w.xp_cq, w.xp_cs, w.dab_cq, w.dab_cs, w.offsets, E, R, H, 2 * F, dW13,
                         wgrad_dtype, e4, ge, dev_status, stream));
  MX_TRY(moe_unpermute(w.dxp, w.dst, nullptr, T, H, k, dX, stream));
  return MX_OK;
}
