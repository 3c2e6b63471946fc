// Router, expert grouping map, token permute / unpermute and the gate
// gradient.
//
// The pytorch/ao "mxfp8 moe training" PR (Next steps) asks for an MXFP8 token
// shuffle: routed tokens are grouped by expert while staying in MXFP8, so the
// grouped GEMM can consume them without a dequantize.  Groups are padded to a
// multiple of 128 rows so that every 128-row GEMM tile belongs to one expert
// and every 32-row block of a column-wise scale stays inside one group.
//
// All kernels here are HBM- or latency-bound; none uses tensor cores.
#include "common.cuh"

#include <mutex>

namespace mxmoe {

constexpr int MAP_CHUNK = 1024;  // routed pairs per CTA in the map kernels
constexpr int MAP_MAX_E = 256;

// ---------------------------------------------------------------------------
// router: one thread per token
// ---------------------------------------------------------------------------
__global__ void k_route(const float *__restrict__ logits, int64_t T, int E, int k, int32_t *ids, float *gate) {
  pdl_enter();
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  const float *l = logits + t * E;
  float m = -INFINITY;
  for (int e = 0; e < E; ++e) m = fmaxf(m, l[e]);
  float sum = 0.f;
  for (int e = 0; e < E; ++e) sum += expf(l[e] - m);
  // k rounds of selection: the largest logit not yet taken, ties to the lower id
  uint32_t taken[MAP_MAX_E / 32] = {0};
  for (int j = 0; j < k; ++j) {
    int best = -1;
    float bv = 0.f;
    for (int e = 0; e < E; ++e) {
      if (taken[e >> 5] & (1u << (e & 31))) continue;
      const float v = l[e];
      if (best < 0 || v > bv) {
        best = e;
        bv = v;
      }
    }
    taken[best >> 5] |= 1u << (best & 31);
    ids[t * k + j] = best;
    gate[t * k + j] = expf(bv - m) / sum;
  }
}

// ---------------------------------------------------------------------------
// grouping map: count per chunk -> scan -> stable ranks
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(MAP_CHUNK) k_map_count(const int32_t *__restrict__ ids, int64_t n, int E,
                                                         int32_t *chunk_counts, int32_t *dev_status) {
  pdl_enter();
  __shared__ int32_t hist[MAP_MAX_E];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t i = (int64_t)blockIdx.x * MAP_CHUNK + threadIdx.x;
  if (i < n) {
    const int e = ids[i];
    if (e >= 0 && e < E)
      atomicAdd(&hist[e], 1);
    else
      set_status(dev_status, MX_ERR_DEVICE);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_counts[(int64_t)blockIdx.x * E + e] = hist[e];
}

// one CTA of MAP_MAX_E threads: thread e owns expert e
__global__ void __launch_bounds__(MAP_MAX_E) k_map_scan(const int32_t *__restrict__ chunk_counts, int64_t nchunks,
                                                        int E, int64_t rows_cap, int32_t *chunk_base,
                                                        int32_t *counts, int32_t *offsets, int32_t *src) {
  pdl_enter();
  __shared__ int32_t s_pad[MAP_MAX_E + 1];
  __shared__ int32_t s_cnt[MAP_MAX_E];
  const int e = threadIdx.x;
  int32_t total = 0;
  if (e < E) {
    for (int64_t c = 0; c < nchunks; ++c) {
      chunk_base[c * E + e] = total;  // relative to the group start for now
      total += chunk_counts[c * E + e];
    }
    s_cnt[e] = total;
  }
  s_pad[e] = (e < E) ? (total + 127) / 128 * 128 : 0;
  __syncthreads();
  // exclusive scan of padded sizes (E <= 256: a serial scan by thread 0 is cheap)
  if (e == 0) {
    int32_t run = 0;
    for (int i = 0; i < E; ++i) {
      const int32_t p = s_pad[i];
      s_pad[i] = run;
      run += p;
    }
    s_pad[E] = run;
  }
  __syncthreads();
  if (e < E) {
    counts[e] = s_cnt[e];
    offsets[e] = s_pad[e];
    for (int64_t c = 0; c < nchunks; ++c) chunk_base[c * E + e] += s_pad[e];
  }
  if (e == 0) offsets[E] = s_pad[E];
  // pad rows of every group, then every row past the last group
  for (int g = 0; g < E; ++g) {
    const int32_t lo = s_pad[g] + s_cnt[g], hi = s_pad[g + 1];
    for (int32_t r = lo + e; r < hi; r += blockDim.x) src[r] = -1;
  }
  for (int64_t r = s_pad[E] + e; r < rows_cap; r += blockDim.x) src[r] = -1;
}

__global__ void __launch_bounds__(MAP_CHUNK) k_map_assign(const int32_t *__restrict__ ids, int64_t n, int E,
                                                          const int32_t *__restrict__ chunk_base, int32_t *dst,
                                                          int32_t *src) {
  pdl_enter();
  __shared__ int32_t warp_cnt[MAP_CHUNK / 32][MAP_MAX_E];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  for (int i = tid; i < (MAP_CHUNK / 32) * MAP_MAX_E; i += blockDim.x) (&warp_cnt[0][0])[i] = 0;
  __syncthreads();
  const int64_t i = (int64_t)blockIdx.x * MAP_CHUNK + tid;
  int e = -1;
  if (i < n) {
    e = ids[i];
    if (e < 0 || e >= E) e = -1;
  }
  // rank among earlier lanes of this warp with the same expert
  const uint32_t peers = __match_any_sync(0xffffffffu, e);
  const int rank_w = __popc(peers & ((1u << lane) - 1u));
  if (e >= 0 && rank_w == 0) warp_cnt[w][e] = __popc(peers);
  __syncthreads();
  // exclusive prefix over warps, per expert
  for (int x = tid; x < E; x += blockDim.x) {
    int32_t run = 0;
    for (int ww = 0; ww < MAP_CHUNK / 32; ++ww) {
      const int32_t c = warp_cnt[ww][x];
      warp_cnt[ww][x] = run;
      run += c;
    }
  }
  __syncthreads();
  if (i < n) {
    if (e >= 0) {
      const int32_t row = chunk_base[(int64_t)blockIdx.x * E + e] + warp_cnt[w][e] + rank_w;
      dst[i] = row;
      src[row] = (int32_t)i;
    } else {
      dst[i] = -1;
    }
  }
}

// ---------------------------------------------------------------------------
// permute (scatter): one warp per token row, plus one warp per row of the
// output that might be padding (it zeroes the row if src says so)
// ---------------------------------------------------------------------------
// One 32-byte store (a whole sector per lane); p must be 32-byte aligned.
__device__ __forceinline__ void st_global_32B(void *p, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3,
                                              uint32_t w4, uint32_t w5, uint32_t w6, uint32_t w7) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w0), "r"(w1), "r"(w2),
               "r"(w3), "r"(w4), "r"(w5), "r"(w6), "r"(w7)
               : "memory");
}

struct PermuteArgs {
  int kind;
  const uint8_t *x;        // fp8 [T,H] or bf16 [T,H]
  const uint8_t *x_scales; // plain [T, H/32] (FP8 kind)
  int64_t T, H;
  int k;
  const int32_t *dst, *src;
  int64_t rows_cap;
  uint8_t *out, *out_scales;
  int swizzled;
};

__device__ __forceinline__ int64_t scale_off(const PermuteArgs &a, int64_t r, int64_t c) {
  const int64_t nb = a.H / 32;
  return a.swizzled ? sf_swizzle_offset(r, c, round_up(nb, 4)) : r * nb + c;
}

__global__ void __launch_bounds__(256) k_permute(PermuteArgs a) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nb = a.H / 32;
  if (w < a.T) {
    const int64_t t = w;
    int32_t rows[8];
    for (int j = 0; j < a.k; ++j) rows[j] = a.dst[t * a.k + j];
    if (a.kind == MX_PERMUTE_FP8) {
      const uint4 *xs = reinterpret_cast<const uint4 *>(a.x + t * a.H);
      const int64_t nc = a.H / 16;
      for (int64_t c0 = lane; c0 < nc; c0 += 32 * 4) {  // four 16-byte loads in flight per lane
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (c0 + 32 * u < nc) v[u] = __ldg(xs + c0 + 32 * u);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (c0 + 32 * u < nc)
            for (int j = 0; j < a.k; ++j)
              if (rows[j] >= 0) reinterpret_cast<uint4 *>(a.out + (int64_t)rows[j] * a.H)[c0 + 32 * u] = v[u];
      }
      // Scales: the blocks 4i .. 4i+3 of a row are 4 contiguous bytes in both
      // layouts (plain: r * nb + c; swizzled: c & 3 is the lowest field), so
      // a lane moves one 32-bit word when the arrays allow 4-byte access.
      const uint8_t *xsc = a.x_scales + t * nb;
      if (nb % 4 == 0 && ((uintptr_t)xsc & 3) == 0 && ((uintptr_t)a.out_scales & 3) == 0) {
        for (int64_t c4 = lane; c4 < nb / 4; c4 += 32) {
          const uint32_t w = *reinterpret_cast<const uint32_t *>(xsc + 4 * c4);
          for (int j = 0; j < a.k; ++j)
            if (rows[j] >= 0) *reinterpret_cast<uint32_t *>(a.out_scales + scale_off(a, rows[j], 4 * c4)) = w;
        }
      } else {
        for (int64_t c = lane; c < nb; c += 32) {
          const uint8_t sc = xsc[c];
          for (int j = 0; j < a.k; ++j)
            if (rows[j] >= 0) a.out_scales[scale_off(a, rows[j], c)] = sc;
        }
      }
    } else if (a.kind == MX_PERMUTE_BF16) {
      const uint4 *xs = reinterpret_cast<const uint4 *>(a.x + t * a.H * 2);
      for (int64_t c = lane; c < a.H / 8; c += 32) {
        const uint4 v = __ldg(xs + c);
        for (int j = 0; j < a.k; ++j)
          if (rows[j] >= 0) reinterpret_cast<uint4 *>(a.out + (int64_t)rows[j] * a.H * 2)[c] = v;
      }
    } else {  // BF16_QUANT: quantize 32-element blocks while moving them
      const uint4 *xs = reinterpret_cast<const uint4 *>(a.x + t * a.H * 2);
      const bool words = nb % 4 == 0 && ((uintptr_t)a.out_scales & 3) == 0;  // scales as 32-bit words
      for (int64_t b = lane; b < nb; b += 32) {
        float f[32];
        uint32_t am2 = 0;  // packed |bf16| maximum of the block
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 v = __ldg(xs + b * 4 + q);
          am2 = vmax_u16x2(am2, vmax_u16x2(vmax_u16x2(v.x & 0x7fff7fffu, v.y & 0x7fff7fffu),
                                           vmax_u16x2(v.z & 0x7fff7fffu, v.w & 0x7fff7fffu)));
          f[8 * q + 0] = bf16_lo(v.x);
          f[8 * q + 1] = bf16_hi(v.x);
          f[8 * q + 2] = bf16_lo(v.y);
          f[8 * q + 3] = bf16_hi(v.y);
          f[8 * q + 4] = bf16_lo(v.z);
          f[8 * q + 5] = bf16_hi(v.z);
          f[8 * q + 6] = bf16_lo(v.w);
          f[8 * q + 7] = bf16_hi(v.w);
        }
        const MxScale s = mx_scale_from_amax_bits(max(am2 << 16, am2 & 0xffff0000u));
        uint32_t wd[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          wd[i] = s.bad ? 0x7f7f7f7fu : scale_pack_e4m3x4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3], s.inv);
        for (int j = 0; j < a.k; ++j) {
          if (rows[j] < 0) continue;
          uint8_t *o = a.out + (int64_t)rows[j] * a.H + b * 32;
          if (((uintptr_t)o & 31) == 0) {  // a whole sector per lane
            st_global_32B(o, wd[0], wd[1], wd[2], wd[3], wd[4], wd[5], wd[6], wd[7]);
          } else {
            reinterpret_cast<uint4 *>(o)[0] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
            reinterpret_cast<uint4 *>(o)[1] = make_uint4(wd[4], wd[5], wd[6], wd[7]);
          }
          if (!words) a.out_scales[scale_off(a, rows[j], b)] = (uint8_t)s.byte;
        }
        if (words) {
          // lanes 4i .. 4i+3 hold blocks b .. b+3 (b % 4 == 0 for lane 4i):
          // their scale bytes leave as one 32-bit word from lane 4i.  The
          // four lanes of a group are active together (nb % 4 == 0).
          const unsigned m = __activemask();
          const uint32_t s1 = __shfl_down_sync(m, s.byte, 1, 4), s2 = __shfl_down_sync(m, s.byte, 2, 4),
                         s3 = __shfl_down_sync(m, s.byte, 3, 4);
          const uint32_t w = s.byte | (s1 << 8) | (s2 << 16) | (s3 << 24);
          if ((lane & 3) == 0)
            for (int j = 0; j < a.k; ++j)
              if (rows[j] >= 0) *reinterpret_cast<uint32_t *>(a.out_scales + scale_off(a, rows[j], b)) = w;
        }
      }
    }
    return;
  }
  const int64_t r = w - a.T;  // candidate pad row
  if (r >= a.rows_cap || a.src[r] >= 0) return;
  const int64_t row_bytes = a.kind == MX_PERMUTE_BF16 ? a.H * 2 : a.H;
  uint4 *o = reinterpret_cast<uint4 *>(a.out + r * row_bytes);
  for (int64_t c = lane; c < row_bytes / 16; c += 32) o[c] = make_uint4(0, 0, 0, 0);
  if (a.kind != MX_PERMUTE_BF16)
    for (int64_t c = lane; c < nb; c += 32) a.out_scales[scale_off(a, r, c)] = 0;
}
// ---------------------------------------------------------------------------
// unpermute / combine: one warp per token, 8 bf16 per lane-step
// ---------------------------------------------------------------------------
// U chunks of 8 per lane with all their K row loads issued first (8 loads
// in flight per lane for every k); the per-element arithmetic and its order
// are the plain definition's.
template <int K>
__global__ void __launch_bounds__(256) k_unpermute(const uint16_t *__restrict__ y, const int32_t *__restrict__ dst,
                                                   const float *__restrict__ gate, int64_t T, int64_t H,
                                                   uint16_t *out) {
  pdl_enter();
  constexpr int U = K >= 8 ? 1 : 8 / K;
  const int lane = threadIdx.x & 31;
  const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  int32_t rows[K];
  float g[K];
#pragma unroll
  for (int j = 0; j < K; ++j) {
    rows[j] = dst[t * K + j];
    g[j] = gate ? gate[t * K + j] : 1.0f;
  }
  const int64_t nc = H / 8;
  for (int64_t c0 = lane; c0 < nc; c0 += 32 * U) {
    uint4 v[U][K];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int j = 0; j < K; ++j) {
        v[u][j] = make_uint4(0, 0, 0, 0);
        if (c0 + 32 * u < nc && rows[j] >= 0)
          v[u][j] = __ldg(reinterpret_cast<const uint4 *>(y + (int64_t)rows[j] * H) + c0 + 32 * u);
      }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (c0 + 32 * u >= nc) break;
      float acc[8];
#pragma unroll
      for (int j = 0; j < K; ++j) {
        const uint4 w = v[u][j];
        const float f[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                            bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float p = gate ? __fmul_rn(g[j], f[i]) : f[i];
          acc[i] = (j == 0) ? p : __fadd_rn(acc[i], p);
        }
      }
      uint4 o;
      o.x = pack_bf16x2(acc[0], acc[1]);
      o.y = pack_bf16x2(acc[2], acc[3]);
      o.z = pack_bf16x2(acc[4], acc[5]);
      o.w = pack_bf16x2(acc[6], acc[7]);
      reinterpret_cast<uint4 *>(out + t * H)[c0 + 32 * u] = o;
    }
  }
}

// ---------------------------------------------------------------------------
// gate gradient: one warp per routed pair, fp32 accumulation, fixed order
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_gate_grad(const uint16_t *__restrict__ dOut, const uint16_t *__restrict__ y,
                                                   const int32_t *__restrict__ dst, int64_t T, int64_t H, int k,
                                                   float *d_gate) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int64_t p = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (p >= T * k) return;
  const int64_t t = p / k;
  const int32_t row = dst[p];
  float acc = 0.f;
  if (row >= 0) {
    const uint4 *a = reinterpret_cast<const uint4 *>(dOut + t * H);
    const uint4 *b = reinterpret_cast<const uint4 *>(y + (int64_t)row * H);
    const int64_t nc = H / 8;
    for (int64_t c0 = lane; c0 < nc; c0 += 32 * 4) {  // four chunk pairs in flight per lane
      uint4 u[4], v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (c0 + 32 * q < nc) {
          u[q] = __ldg(a + c0 + 32 * q);
          v[q] = __ldg(b + c0 + 32 * q);
        }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (c0 + 32 * q >= nc) break;
        acc = fmaf(bf16_lo(u[q].x), bf16_lo(v[q].x), acc);
        acc = fmaf(bf16_hi(u[q].x), bf16_hi(v[q].x), acc);
        acc = fmaf(bf16_lo(u[q].y), bf16_lo(v[q].y), acc);
        acc = fmaf(bf16_hi(u[q].y), bf16_hi(v[q].y), acc);
        acc = fmaf(bf16_lo(u[q].z), bf16_lo(v[q].z), acc);
        acc = fmaf(bf16_hi(u[q].z), bf16_hi(v[q].z), acc);
        acc = fmaf(bf16_lo(u[q].w), bf16_lo(v[q].w), acc);
        acc = fmaf(bf16_hi(u[q].w), bf16_hi(v[q].w), acc);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) d_gate[p] = acc;
}

}  // namespace mxmoe

using namespace mxmoe;

extern "C" mx_status moe_route(const float *logits, int64_t T, int32_t E, int32_t k, int32_t *ids, float *gate,
                               mx_stream stream) {
  MX_HOST_CHECK(T == 0 || (logits && ids && gate), MX_ERR_INVALID_ARG);  // T = 0: nothing to read or write
  MX_HOST_CHECK(T >= 0 && E >= 1 && E <= MAP_MAX_E && k >= 1 && k <= E && k <= 8, MX_ERR_INVALID_ARG);
  mx_status st = check_device_cached();
  if (st != MX_OK) return st;
  if (T == 0) return MX_OK;
  (void)launch_k(k_route, (unsigned)((T + 127) / 128), 128, 0, stream, logits, T, E, k, ids, gate);
  return launch_status();
}

extern "C" int64_t moe_rows_cap(int64_t T, int32_t k, int32_t E) {
  if (T < 0 || k < 1 || E < 1) return -1;
  return round_up(T * k + (int64_t)E * 127, 128);
}

extern "C" int64_t moe_permute_map_workspace_size(int64_t T, int32_t k, int32_t E) {
  if (T < 0 || k < 1 || E < 1) return -1;
  const int64_t nchunks = (T * k + MAP_CHUNK - 1) / MAP_CHUNK;
  return round_up(2 * nchunks * E * (int64_t)sizeof(int32_t), 256);
}

extern "C" mx_status moe_permute_map(const int32_t *ids, int64_t T, int32_t k, int32_t E, int64_t rows_cap,
                                     int32_t *counts, int32_t *offsets, int32_t *dst, int32_t *src, void *workspace,
                                     int64_t workspace_bytes, int32_t *dev_status, mx_stream stream) {
  MX_HOST_CHECK(counts && offsets && src && (T == 0 || (ids && dst)), MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(T >= 0 && k >= 1 && k <= 8 && E >= 1 && E <= MAP_MAX_E, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(rows_cap >= moe_rows_cap(T, k, E), MX_ERR_SHAPE);
  const int64_t need = moe_permute_map_workspace_size(T, k, E);
  MX_HOST_CHECK(workspace != nullptr || need == 0, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(workspace_bytes >= need, MX_ERR_WORKSPACE);
  mx_status st = check_device_cached();
  if (st != MX_OK) return st;
  const int64_t n = T * k;
  const int64_t nchunks = (n + MAP_CHUNK - 1) / MAP_CHUNK;
  int32_t *chunk_counts = static_cast<int32_t *>(workspace);
  int32_t *chunk_base = chunk_counts + nchunks * E;
  if (nchunks > 0) (void)launch_k(k_map_count, (unsigned)nchunks, MAP_CHUNK, 0, stream, ids, n, E, chunk_counts, dev_status);
  (void)launch_k(k_map_scan, 1, MAP_MAX_E, 0, stream, chunk_counts, nchunks, E, rows_cap, chunk_base, counts, offsets, src);
  if (nchunks > 0) (void)launch_k(k_map_assign, (unsigned)nchunks, MAP_CHUNK, 0, stream, ids, n, E, chunk_base, dst, src);
  return launch_status();
}

// ---------------------------------------------------------------------------
// Allocation-free grouping map: the same three kernels, with their per-chunk
// count/base scratch in a fixed array of this library's device memory instead
// of a caller workspace (see moe_permute_map_noalloc in mxmoe.h).
// ---------------------------------------------------------------------------
static __device__ __align__(256) int32_t g_noalloc_map_scratch[MOE_NOALLOC_SCRATCH_BYTES / sizeof(int32_t)];

namespace {
std::mutex g_noalloc_mu;
int32_t *g_noalloc_ptr[64];  // device address of the array, per device

// Host code must not pass the array's name to a kernel: on the host it is a
// stand-in symbol, not a device address.  Look the address up once per device
// (with that device current) and hand the kernels that pointer.
mx_status noalloc_scratch(int32_t **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MX_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_map_scratch) != cudaSuccess || p == nullptr) return MX_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<int32_t *>(p);
  }
  *out = g_noalloc_ptr[dev];
  return MX_OK;
}
}  // namespace

extern "C" mx_status moe_permute_map_noalloc(const int32_t *ids, int64_t T, int32_t k, int32_t E, int64_t rows_cap,
                                             int32_t *counts, int32_t *offsets, int32_t *dst, int32_t *src,
                                             int32_t *dev_status, mx_stream stream) {
  MX_HOST_CHECK(counts && offsets && src && (T == 0 || (ids && dst)), MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(T >= 0 && k >= 1 && k <= 8 && E >= 1 && E <= MAP_MAX_E, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(rows_cap >= moe_rows_cap(T, k, E), MX_ERR_SHAPE);
  MX_HOST_CHECK(moe_permute_map_workspace_size(T, k, E) <= (int64_t)MOE_NOALLOC_SCRATCH_BYTES, MX_ERR_SCRATCH_LIMIT);
  mx_status st = check_device_cached();
  if (st != MX_OK) return st;
  int32_t *scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != MX_OK) return st;
  const int64_t n = T * k;
  const int64_t nchunks = (n + MAP_CHUNK - 1) / MAP_CHUNK;
  int32_t *chunk_counts = scratch;
  int32_t *chunk_base = scratch + nchunks * E;
  if (nchunks > 0) (void)launch_k(k_map_count, (unsigned)nchunks, MAP_CHUNK, 0, stream, ids, n, E, chunk_counts, dev_status);
  (void)launch_k(k_map_scan, 1, MAP_MAX_E, 0, stream, chunk_counts, nchunks, E, rows_cap, chunk_base, counts, offsets, src);
  if (nchunks > 0) (void)launch_k(k_map_assign, (unsigned)nchunks, MAP_CHUNK, 0, stream, ids, n, E, chunk_base, dst, src);
  return launch_status();
}

extern "C" mx_status moe_permute(int32_t kind, const void *x, const uint8_t *x_scales, int64_t T, int64_t H,
                                 int32_t k, const int32_t *dst, const int32_t *src, int64_t rows_cap, void *out,
                                 uint8_t *out_scales, int32_t scale_layout, mx_stream stream) {
  MX_HOST_CHECK(kind == MX_PERMUTE_FP8 || kind == MX_PERMUTE_BF16 || kind == MX_PERMUTE_BF16_QUANT,
                MX_ERR_INVALID_ARG);
  // T = 0: no token rows (x, x_scales, dst may be NULL); the pad rows are still zeroed
  MX_HOST_CHECK(src && out && (T == 0 || (x && dst)), MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(kind == MX_PERMUTE_BF16 || (out_scales != nullptr), MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(kind != MX_PERMUTE_FP8 || T == 0 || x_scales != nullptr, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(scale_layout == MX_SCALE_PLAIN || scale_layout == MX_SCALE_SWIZZLED, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(T >= 0 && H > 0 && k >= 1 && k <= 8 && rows_cap >= 0, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(H % 32 == 0, MX_ERR_SHAPE);
  MX_HOST_CHECK(!(kind != MX_PERMUTE_BF16 && scale_layout == MX_SCALE_SWIZZLED) || (H % 128 == 0 && rows_cap % 128 == 0),
                MX_ERR_SHAPE);
  MX_HOST_CHECK(aligned16(x) && aligned16(out), MX_ERR_ALIGNMENT);
  mx_status st = check_device_cached();
  if (st != MX_OK) return st;
  PermuteArgs a;
  a.kind = kind;
  a.x = static_cast<const uint8_t *>(x);
  a.x_scales = x_scales;
  a.T = T;
  a.H = H;
  a.k = k;
  a.dst = dst;
  a.src = src;
  a.rows_cap = rows_cap;
  a.out = static_cast<uint8_t *>(out);
  a.out_scales = out_scales;
  a.swizzled = scale_layout == MX_SCALE_SWIZZLED;
  const int64_t warps = T + rows_cap;
  if (warps == 0) return MX_OK;
  (void)launch_k(k_permute, (unsigned)((warps + 7) / 8), 256, 0, stream, a);
  return launch_status();
}

extern "C" mx_status moe_unpermute(const void *y, const int32_t *dst, const float *gate, int64_t T, int64_t H,
                                   int32_t k, void *out, mx_stream stream) {
  MX_HOST_CHECK(T == 0 || (y && dst && out), MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(T >= 0 && H > 0 && k >= 1 && k <= 8, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(H % 8 == 0, MX_ERR_SHAPE);
  MX_HOST_CHECK(aligned16(y) && aligned16(out), MX_ERR_ALIGNMENT);
  mx_status st = check_device_cached();
  if (st != MX_OK) return st;
  if (T == 0) return MX_OK;
  const unsigned grid = (unsigned)((T + 7) / 8);
  const uint16_t *yy = static_cast<const uint16_t *>(y);
  uint16_t *oo = static_cast<uint16_t *>(out);
  switch (k) {
    case 1: (void)launch_k(k_unpermute<1>, grid, 256, 0, stream, yy, dst, gate, T, H, oo); break;
    case 2: (void)launch_k(k_unpermute<2>, grid, 256, 0, stream, yy, dst, gate, T, H, oo); break;
    case 3: (void)launch_k(k_unpermute<3>, grid, 256, 0, stream, yy, dst, gate, T, H, oo); break;
    case 4: (void)launch_k(k_unpermute<4>, grid, 256, 0, stream, yy, dst, gate, T, H, oo); break;
    case 5: (void)launch_k(k_unpermute<5>, grid, 256, 0, stream, yy, dst, gate, T, H, oo); break;
    case 6: (void)launch_k(k_unpermute<6>, grid, 256, 0, stream, yy, dst, gate, T, H, oo); break;
    case 7: (void)launch_k(k_unpermute<7>, grid, 256, 0, stream, yy, dst, gate, T, H, oo); break;
    default: (void)launch_k(k_unpermute<8>, grid, 256, 0, stream, yy, dst, gate, T, H, oo); break;
  }
  return launch_status();
}

extern "C" mx_status moe_gate_grad(const void *dOut, const void *y, const int32_t *dst, int64_t T, int64_t H,
                                   int32_t k, float *d_gate, mx_stream stream) {
  MX_HOST_CHECK(T == 0 || (dOut && y && dst && d_gate), MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(T >= 0 && H > 0 && k >= 1 && k <= 8, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(H % 8 == 0, MX_ERR_SHAPE);
  MX_HOST_CHECK(aligned16(dOut) && aligned16(y), MX_ERR_ALIGNMENT);
  mx_status st = check_device_cached();
  if (st != MX_OK) return st;
  if (T == 0) return MX_OK;
  (void)launch_k(k_gate_grad, (unsigned)((T * k + 7) / 8), 256, 0, stream, static_cast<const uint16_t *>(dOut),
                                                               static_cast<const uint16_t *>(y), dst, T, H, k, d_gate);
  return launch_status();
}
