// MXFP8 quantize kernels.
//
// Block quantization per OCP Microscaling Formats (MX) v1.0, section 6.3
// (32-element blocks, E8M0 scale 2^(floor(log2 amax) - 8), E4M3 elements cast
// with round-to-nearest-even and saturation), row-wise and column-wise, as the
// "1.5x faster MoE training on Blackwell with MXFP8 kernels built from
// scratch" article (Key Questions Answered: microscaling; Common Pitfalls:
// quantization overhead) and the pytorch/ao "mxfp8 moe training" PR stack
// (Stacked PRs: quant kernels) describe.
//
// HBM-bound.  One CTA owns a tile of 128 rows x 64 columns of the input:
//   phase 1  coalesced 16-byte loads; each 32-element row block lives in 4
//            consecutive lanes, so the ROW result needs only two shuffles;
//            the tile is staged in shared memory for the column pass;
//   phase 2  each thread walks 32 rows of one column in shared memory
//            (conflict-free: a warp reads 64 contiguous bytes per row) and
//            writes the 32 E4M3 bytes of that column block contiguously into
//            the transposed COL output.
#include "common.cuh"

namespace mxmoe {

constexpr int QT_ROWS = 128;
constexpr int QT_COLS = 64;
constexpr int QT_THREADS = 256;

struct QuantArgs {
  const uint16_t *x;
  int64_t rows, cols;
  // gather mode: output row r takes input row src[r] / k (zero when src[r] < 0),
  // multiplied by gate[src[r]] (fp32 product rounded to bf16) when gate != NULL
  const int32_t *src;
  const float *gate;
  int k;
  const int32_t *row_limit;  // gather mode, nullable: rows at or past *row_limit are skipped
  uint8_t *q_row, *s_row, *q_col, *s_col;
  int64_t s_row_stride, s_col_stride;  // bytes per batch entry
  int32_t swizzled;
};

template <bool ROW, bool COL, bool GATHER, bool E5 = false>
// E5: E5M2 elements (the gradient option); otherwise E4M3.
// 6 resident CTAs per SM (registers capped at 42): 1.5-2% faster than the
// register-limited 5, measured side by side in one process.  The row amax on
// packed bf16 pairs and the packed fp32x2 scaling each save ~2.5% (the kernel
// is close to issue-bound), measured the same way.
__global__ void __launch_bounds__(QT_THREADS, 6) k_quantize_bf16(QuantArgs a) {
  pdl_enter();
  __shared__ __align__(16) uint16_t tile[QT_ROWS][QT_COLS];
  // COL output staged as [64 columns][128 rows] bytes (+16 pad per row: the
  // 16-byte writes of 8 consecutive columns then fall in distinct banks)
  __shared__ __align__(16) uint8_t qcol[QT_COLS][QT_ROWS + 16];
  __shared__ __align__(16) uint8_t scol[QT_COLS][4];
  constexpr int ITERS = (QT_ROWS * QT_COLS / 8) / QT_THREADS;  // 4 chunks of 8 per thread
  const int tid = threadIdx.x;
  const int64_t b = blockIdx.z;
  // COL-only mode walks row bands fastest: CTAs resident together then cover
  // neighbouring row bands of the same columns and the transposed writes form
  // long runs (measured 13% faster); with ROW output, column tiles fastest
  // keep the row-major reads and writes contiguous instead.
  const int64_t row0 = (int64_t)(ROW ? blockIdx.y : blockIdx.x) * QT_ROWS;
  const int64_t col0 = (int64_t)(ROW ? blockIdx.x : blockIdx.y) * QT_COLS;
  // This thread's chunks: tile rows it * 32 + tr (it < ITERS), columns
  // tc .. tc + 7.  64-bit bases once per CTA, 32-bit offsets inside the tile
  // (the host bounds rows and cols so that they fit).
  const int tr = tid >> 3, tc = (tid & 7) * 8;
  const int64_t gc = col0 + tc;
  const bool col_ok = gc < a.cols;
  const uint32_t ucols = (uint32_t)a.cols;
  const int64_t tile_off = (b * a.rows + row0) * a.cols + gc;  // element (row0 + tr, gc) minus tr rows
  const uint32_t t_off = (uint32_t)tr * ucols;

  if (GATHER && a.row_limit && row0 >= __ldg(a.row_limit)) return;  // past the last routed row

  // ---- phase 0: every load of this thread in flight at once ----
  // (gather mode: all source indices first, then the rows and their gates,
  // so phase 1 never waits on a dependent load)
  uint4 v[ITERS];
  int32_t sidx[ITERS];
  float gv[ITERS];
  if (GATHER) {
#pragma unroll
    for (int it = 0; it < ITERS; ++it) {
      const int64_t gr = row0 + it * 32 + tr;
      sidx[it] = (gr < a.rows && col_ok) ? a.src[gr] : -1;
    }
  }
#pragma unroll
  for (int it = 0; it < ITERS; ++it) {
    const bool valid = col_ok && row0 + it * 32 + tr < a.rows;
    v[it] = make_uint4(0, 0, 0, 0);
    if (GATHER) {
      gv[it] = 1.0f;
      if (sidx[it] >= 0) {
        const int32_t t = a.k == 1 ? sidx[it] : sidx[it] / a.k;
        v[it] = __ldg(reinterpret_cast<const uint4 *>(a.x + (int64_t)t * a.cols + gc));
        if (a.gate) gv[it] = __ldg(a.gate + sidx[it]);
      }
    } else if (valid) {
      v[it] = __ldg(reinterpret_cast<const uint4 *>(a.x + tile_off + (t_off + (uint32_t)(it * 32) * ucols)));
    }
  }

  // row-scale position of this thread's blocks: row r = row0 + it*32 + tr,
  // block column c = gc / 32.  row0 is a multiple of 128 and col0 of 64, so
  // in the swizzled layout r >> 7 = row0 >> 7, r & 31 = tr,
  // (r & 127) >> 5 = it, c >> 2 = col0 >> 7 and c & 3 = ((col0 >> 5) & 3) +
  // ((tid & 7) >> 2): the offset is a per-CTA base plus it * 4.
  const int64_t cblocks = a.cols / 32;
  int64_t rs_base = 0;
  uint32_t rs_step = 0;
  if (ROW) {
    if (a.swizzled) {
      rs_base = ((row0 >> 7) * (round_up(cblocks, 4) >> 2) + (col0 >> 7)) * 512 + tr * 16 + ((col0 >> 5) & 3) +
                ((tid & 7) >> 2);
      rs_step = 4;
    } else {
      rs_base = (row0 + tr) * cblocks + (gc >> 5);
      rs_step = (uint32_t)(32 * cblocks);
    }
  }

  // ---- phase 1: ROW quant (a 32-element block = 4 consecutive lanes), stage ----
#pragma unroll
  for (int it = 0; it < ITERS; ++it) {
    const int r = it * 32 + tr;
    const bool valid = col_ok && row0 + r < a.rows;
    uint4 w = v[it];
    if (GATHER && a.gate) {
      if (sidx[it] >= 0) {
        const float g = gv[it];
        w.x = pack_bf16x2(g * bf16_lo(w.x), g * bf16_hi(w.x));
        w.y = pack_bf16x2(g * bf16_lo(w.y), g * bf16_hi(w.y));
        w.z = pack_bf16x2(g * bf16_lo(w.z), g * bf16_hi(w.z));
        w.w = pack_bf16x2(g * bf16_lo(w.w), g * bf16_hi(w.w));
      }
    }
    if (COL) *reinterpret_cast<uint4 *>(&tile[r][tc]) = w;
    if (ROW) {
      const float f[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                          bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
      // block amax on the packed bf16 pairs (sign bits cleared), as an fp32 pattern
      uint32_t am = vmax_u16x2(vmax_u16x2(w.x & 0x7fff7fffu, w.y & 0x7fff7fffu),
                               vmax_u16x2(w.z & 0x7fff7fffu, w.w & 0x7fff7fffu));
      am = max(am << 16, am & 0xffff0000u);
      am = max(am, __shfl_xor_sync(0xffffffffu, am, 1));
      am = max(am, __shfl_xor_sync(0xffffffffu, am, 2));
      const MxScale s = mx_scale_from_amax_bits_t<E5>(am);
      uint2 o;
      o.x = s.bad ? 0x7f7f7f7fu : scale_pack_fp8x4<E5>(f[0], f[1], f[2], f[3], s.inv);
      o.y = s.bad ? 0x7f7f7f7fu : scale_pack_fp8x4<E5>(f[4], f[5], f[6], f[7], s.inv);
      if (valid) {
        *reinterpret_cast<uint2 *>(a.q_row + tile_off + (t_off + (uint32_t)(it * 32) * ucols)) = o;
        if ((tid & 3) == 0) a.s_row[b * a.s_row_stride + rs_base + it * rs_step] = (uint8_t)s.byte;
      }
    }
  }
  if (!COL) return;
  __syncthreads();

  // ---- phase 2: COL quant from shared memory into the staged output ----
  {
    const int col = tid & (QT_COLS - 1);
    const int rb = tid / QT_COLS;  // 0..3
    float f[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) f[i] = __uint_as_float((uint32_t)tile[rb * 32 + i][col] << 16);
    uint32_t am = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) am = max(am, abs_bits(f[i]));
    const MxScale s = mx_scale_from_amax_bits_t<E5>(am);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      w[i] = s.bad ? 0x7f7f7f7fu : scale_pack_fp8x4<E5>(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3], s.inv);
    uint4 *dst = reinterpret_cast<uint4 *>(&qcol[col][rb * 32]);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    scol[col][rb] = (uint8_t)s.byte;
  }
  __syncthreads();

  // ---- phase 3: full-line writes of the transposed output and its scales ----
  const int nrows_valid = (int)min((int64_t)QT_ROWS, a.rows - row0);  // multiple of 32
  uint8_t *qc = a.q_col + (b * a.cols + col0) * a.rows + row0;      // (col0, row0) of the COL output
  const int part = tid & 7;                                         // 8 x 16 bytes per staged row
#pragma unroll
  for (int it = 0; it < (QT_COLS * QT_ROWS / 16) / QT_THREADS; ++it) {
    const int cc = it * (QT_THREADS / 8) + (tid >> 3);
    if (col0 + cc < a.cols && part * 16 < nrows_valid)
      *reinterpret_cast<uint4 *>(qc + (int64_t)cc * a.rows + part * 16) =
          *reinterpret_cast<const uint4 *>(&qcol[cc][part * 16]);
  }
  if (tid < QT_COLS && col0 + tid < a.cols) {
    // column gc = col0 + tid, block rows row0/32 + i: row0 is a multiple of
    // 128, so the (up to) four scale bytes are consecutive in both layouts
    const int64_t gcs = col0 + tid, rblocks = a.rows / 32;
    const int64_t off = a.swizzled ? ((gcs >> 7) * (round_up(rblocks, 4) >> 2) + (row0 >> 7)) * 512 +
                                         (gcs & 31) * 16 + ((gcs & 127) >> 5) * 4
                                   : gcs * rblocks + (row0 >> 5);
    uint8_t *sc = a.s_col + b * a.s_col_stride + off;
    for (int i = 0; i < nrows_valid / 32; ++i) sc[i] = scol[tid][i];
  }
}

// ---------------------------------------------------------------------------
// SwiGLU backward + quantization (see moe_swiglu_bwd in mxmoe.h).
// Tile: 128 rows x 32 columns of F, 256 threads.
//   phase 1  two (row, 8-column) chunks per thread, all loads issued first;
//            da, db, h in fp32, two columns per packed f32x2 instruction;
//            ROW quant of da and db (4 lanes per block); da, db, h staged
//            in shared memory;
//   phase 2  COL quant of the three staged matrices (32 x 4 column blocks
//            each) into a staged transposed tile;
//   phase 3  full 128-byte line writes of the transposed tiles and their
//            scales.
// The kernel issues about as many instructions as its bytes take at HBM
// speed, so the arithmetic is packed: the products and fused multiply-adds
// of two columns share one f32x2 instruction (each lane is an IEEE fp32
// operation, identical to the scalar one) and a block amax takes one
// max-of-magnitudes per element.  Measured side by side on the layer's
// 17792 x 8192 case, bytes identical: 6% faster than the scalar form.  (A
// lane-per-column variant without the fp32 staging, and 16-byte staging
// stores, were both slower.)
// ---------------------------------------------------------------------------
constexpr int SB_ROWS = 128;
constexpr int SB_COLS = 32;
constexpr int SB_THREADS = 256;
constexpr int SB_VAL_STRIDE = SB_COLS + 1;            // fp32 staging row (padded: conflict-free)
constexpr int SB_Q_STRIDE = SB_ROWS + 16;             // transposed byte row (padded)
constexpr int SB_SMEM = 3 * SB_ROWS * SB_VAL_STRIDE * 4 + 3 * SB_COLS * SB_Q_STRIDE + 3 * SB_COLS * 4;

// packed fp32 pairs (lane 0 = the first element)
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// max(|a|, |b|) as a magnitude (its sign bit is meaningless: callers take
// abs_bits of the result); NaN in either input gives NaN, so abs_bits of a
// chain of these is the block's abs_bits maximum with NaN and Inf above
// every finite value, as mx_scale_from_amax_bits_t expects.
__device__ __forceinline__ float max_mag(float a, float b) {
  float r;
  asm("max.NaN.xorsign.abs.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// The sigmoid pieces of sigmoid_parts for two bf16 values at once: the same
// operations, with the products and fused multiply-adds packed.
struct SigParts2 {
  uint64_t s, oms, back;
};
__device__ __forceinline__ SigParts2 sigmoid_parts2(float a0, float a1) {
  const float aa0 = fminf(fabsf(a0), 256.0f), aa1 = fminf(fabsf(a1), 256.0f);
  const bool far0 = a0 < -64.0f, far1 = a1 < -64.0f;
  const uint64_t aa = f2_pack(aa0, aa1);
  const uint64_t arg = f2_fma(aa, f2_pack(-LOG2E_HI, -LOG2E_HI), f2_pack(far0 ? 64.0f : 0.0f, far1 ? 64.0f : 0.0f));
  float x0, x1;
  f2_unpack(arg, x0, x1);
  const uint64_t t0 = f2_pack(ex2_approx(x0), ex2_approx(x1));
  const uint64_t y = f2_mul(aa, f2_pack(LOG2E_REM_LN, LOG2E_REM_LN));
  const uint64_t q = f2_fma(y, f2_fma(f2_pack(0.5f, 0.5f), y, f2_pack(-1.0f, -1.0f)), f2_pack(1.0f, 1.0f));
  const uint64_t t = f2_mul(t0, q);
  float u0, u1;
  f2_unpack(f2_add(f2_pack(1.0f, 1.0f), t), u0, u1);
  const uint64_t r = f2_pack(rcp_approx(far0 ? 1.0f : u0), rcp_approx(far1 ? 1.0f : u1));
  const uint64_t tr = f2_mul(t, r);
  float r0, r1, tr0, tr1;
  f2_unpack(r, r0, r1);
  f2_unpack(tr, tr0, tr1);
  SigParts2 p;
  p.s = f2_pack(a0 >= 0.0f ? r0 : tr0, a1 >= 0.0f ? r1 : tr1);
  p.oms = f2_pack(a0 >= 0.0f ? tr0 : r0, a1 >= 0.0f ? tr1 : r1);
  p.back = f2_pack(far0 ? 0x1p-64f : 1.0f, far1 ? 0x1p-64f : 1.0f);
  return p;
}

// da, db, h of two columns (d, a, b packed): the operations of the scalar
// reading, in the same order,
//   silu = a s,  h = (silu b) back,  db = (d silu) back,
//   da = (((d b) s) (1 + a oms)) back
__device__ __forceinline__ void swiglu_bwd2(uint64_t d, float a0, float a1, uint64_t b, uint64_t &da, uint64_t &db,
                                            uint64_t &h) {
  const SigParts2 p = sigmoid_parts2(a0, a1);
  const uint64_t a = f2_pack(a0, a1);
  const uint64_t silu = f2_mul(a, p.s);
  const uint64_t g = f2_fma(a, p.oms, f2_pack(1.0f, 1.0f));
  da = f2_mul(f2_mul(f2_mul(f2_mul(d, b), p.s), g), p.back);
  db = f2_mul(f2_mul(d, silu), p.back);
  h = f2_mul(f2_mul(silu, b), p.back);
}

template <bool E5>  // E5: [da|db] with E5M2 elements (the gradient option); h stays E4M3
__global__ void __launch_bounds__(SB_THREADS) k_swiglu_bwd(const float *__restrict__ dh, const uint16_t *__restrict__ ab,
                                                           int64_t rows, int64_t F, uint8_t *dab_rq, uint8_t *dab_rs,
                                                           uint8_t *dab_cq, uint8_t *dab_cs, uint8_t *h_cq,
                                                           uint8_t *h_cs, const int32_t *__restrict__ row_limit) {
  pdl_enter();
  extern __shared__ __align__(16) uint8_t sb_smem[];
  float *vals = reinterpret_cast<float *>(sb_smem);                          // [3][128][33]
  uint8_t *qst = sb_smem + 3 * SB_ROWS * SB_VAL_STRIDE * 4;                    // [3][32][144]
  uint8_t *sst = qst + 3 * SB_COLS * SB_Q_STRIDE;                             // [3][32][4]
  const int tid = threadIdx.x;
  const int64_t row0 = (int64_t)blockIdx.x * SB_ROWS;  // row bands fastest (see k_quantize_bf16)
  const int64_t f0 = (int64_t)blockIdx.y * SB_COLS;
  if (row_limit && row0 >= __ldg(row_limit)) return;  // past the last routed row: nothing to do
  const int64_t twoF = 2 * F;
  const int64_t cb2 = twoF / 32;

  // 512 chunks (128 rows x 4 chunks of 8): this thread's are tile rows
  // it * 64 + rt, columns ch * 8 .. + 7.  64-bit bases once, 32-bit offsets
  // inside the tile (the host bounds F).
  const int rt = tid >> 2, ch = tid & 3;
  const int64_t gf = f0 + ch * 8;
  const uint32_t uF = (uint32_t)F, u2F = 2u * uF;
  const float *dh_t = dh + row0 * F + gf;
  const uint16_t *ab_t = ab + row0 * twoF + gf;
  uint8_t *dab_t = dab_rq + row0 * twoF + gf;
  ulonglong2 d0[2], d1[2];  // dh columns 0..3 and 4..7 as packed pairs
  uint4 av[2], bv[2];
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const uint32_t r = (uint32_t)(it * 64 + rt);
    d0[it] = *reinterpret_cast<const ulonglong2 *>(dh_t + r * uF);
    d1[it] = *reinterpret_cast<const ulonglong2 *>(dh_t + r * uF + 4);
    av[it] = *reinterpret_cast<const uint4 *>(ab_t + r * u2F);
    bv[it] = *reinterpret_cast<const uint4 *>(ab_t + r * u2F + uF);
  }
  // row-scale offsets (swizzled): r >> 7 = row0 >> 7, r & 31 = rt & 31,
  // (r & 127) >> 5 = 2 * it + (rt >> 5); block column f0 / 32 for da and
  // (F + f0) / 32 for db
  const int64_t ca = f0 >> 5, cbk = (F + f0) >> 5, cp4 = round_up(cb2, 4);
  const int64_t rs_row = (row0 >> 7) * (cp4 >> 2);
  const int64_t rs_a = (rs_row + (ca >> 2)) * 512 + (rt & 31) * 16 + (rt >> 5) * 4 + (ca & 3);
  const int64_t rs_b = (rs_row + (cbk >> 2)) * 512 + (rt & 31) * 16 + (rt >> 5) * 4 + (cbk & 3);
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int r = it * 64 + rt;
    const uint64_t dp[4] = {d0[it].x, d0[it].y, d1[it].x, d1[it].y};
    const uint32_t aw[4] = {av[it].x, av[it].y, av[it].z, av[it].w};
    const uint32_t bw[4] = {bv[it].x, bv[it].y, bv[it].z, bv[it].w};
    float da[8], db[8], hh[8];
    float ma = 0.0f, mb = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint64_t da2, db2, h2;
      swiglu_bwd2(dp[j], bf16_lo(aw[j]), bf16_hi(aw[j]), f2_pack(bf16_lo(bw[j]), bf16_hi(bw[j])), da2, db2, h2);
      f2_unpack(da2, da[2 * j], da[2 * j + 1]);
      f2_unpack(db2, db[2 * j], db[2 * j + 1]);
      f2_unpack(h2, hh[2 * j], hh[2 * j + 1]);
      ma = max_mag(ma, max_mag(da[2 * j], da[2 * j + 1]));
      mb = max_mag(mb, max_mag(db[2 * j], db[2 * j + 1]));
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      vals[(0 * SB_ROWS + r) * SB_VAL_STRIDE + ch * 8 + i] = da[i];
      vals[(1 * SB_ROWS + r) * SB_VAL_STRIDE + ch * 8 + i] = db[i];
      vals[(2 * SB_ROWS + r) * SB_VAL_STRIDE + ch * 8 + i] = hh[i];
    }
    ma = max_mag(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
    ma = max_mag(ma, __shfl_xor_sync(0xffffffffu, ma, 2));
    mb = max_mag(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
    mb = max_mag(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
    const MxScale sa = mx_scale_from_amax_bits_t<E5>(abs_bits(ma)), sbb = mx_scale_from_amax_bits_t<E5>(abs_bits(mb));
    uint2 oa, ob;
    oa.x = sa.bad ? 0x7f7f7f7fu : scale_pack_fp8x4<E5>(da[0], da[1], da[2], da[3], sa.inv);
    oa.y = sa.bad ? 0x7f7f7f7fu : scale_pack_fp8x4<E5>(da[4], da[5], da[6], da[7], sa.inv);
    ob.x = sbb.bad ? 0x7f7f7f7fu : scale_pack_fp8x4<E5>(db[0], db[1], db[2], db[3], sbb.inv);
    ob.y = sbb.bad ? 0x7f7f7f7fu : scale_pack_fp8x4<E5>(db[4], db[5], db[6], db[7], sbb.inv);
    *reinterpret_cast<uint2 *>(dab_t + (uint32_t)r * u2F) = oa;
    *reinterpret_cast<uint2 *>(dab_t + (uint32_t)r * u2F + uF) = ob;
    if (ch == 0) {
      dab_rs[rs_a + it * 8] = (uint8_t)sa.byte;
      dab_rs[rs_b + it * 8] = (uint8_t)sbb.byte;
    }
  }
  __syncthreads();

  // COL: 3 matrices x 32 columns x 4 row blocks = 384 items
  for (int item = tid; item < 3 * SB_COLS * 4; item += SB_THREADS) {
    const int m = item / (SB_COLS * 4);
    const int rem = item % (SB_COLS * 4);
    const int col = rem % SB_COLS, rb = rem / SB_COLS;
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = vals[(m * SB_ROWS + rb * 32 + i) * SB_VAL_STRIDE + col];
    float mm[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) mm[i] = max_mag(v[2 * i], v[2 * i + 1]);
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
      for (int i = 0; i < w; ++i) mm[i] = max_mag(mm[i], mm[i + w]);
    const uint32_t am = abs_bits(mm[0]);
    // matrices 0, 1 ([da|db]) in the gradient format, 2 (h) in E4M3
    const bool e5 = E5 && m < 2;
    const MxScale s = e5 ? mx_scale_from_amax_bits_t<true>(am) : mx_scale_from_amax_bits_t<false>(am);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      w[i] = s.bad ? 0x7f7f7f7fu
             : e5  ? scale_pack_fp8x4<true>(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3], s.inv)
                   : scale_pack_fp8x4<false>(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3], s.inv);
    uint4 *dst = reinterpret_cast<uint4 *>(qst + (m * SB_COLS + col) * SB_Q_STRIDE + rb * 32);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    sst[(m * SB_COLS + col) * 4 + rb] = (uint8_t)s.byte;
  }
  __syncthreads();

  // full-line writes: 3 x 32 transposed rows of 128 bytes
  const int64_t rblocks_total = rows / 32;
#pragma unroll
  for (int it = 0; it < (3 * SB_COLS * 8) / SB_THREADS; ++it) {
    const int c = it * SB_THREADS + tid;
    const int mr = c >> 3, part = c & 7;  // mr = m * 32 + col
    const int m = mr / SB_COLS, col = mr % SB_COLS;
    const uint4 val = *reinterpret_cast<const uint4 *>(qst + mr * SB_Q_STRIDE + part * 16);
    if (m < 2) {
      const int64_t orow = (m == 0 ? 0 : F) + f0 + col;
      *reinterpret_cast<uint4 *>(dab_cq + orow * rows + row0 + part * 16) = val;
    } else {
      *reinterpret_cast<uint4 *>(h_cq + (f0 + col) * rows + row0 + part * 16) = val;
    }
  }
  for (int i = tid; i < 3 * SB_COLS * 4; i += SB_THREADS) {
    // one scale byte per (transposed row, row block); the 4 row blocks of a
    // transposed row are 4 consecutive bytes of the tiled layout
    const int mr = i >> 2, rb = i & 3;
    const int m = mr / SB_COLS, col = mr % SB_COLS;
    const uint8_t sc = sst[i];
    const int64_t orow = (m == 1 ? F : 0) + f0 + col;
    uint8_t *base = m < 2 ? dab_cs : h_cs;
    base[sf_swizzle_offset(orow, row0 / 32 + rb, round_up(rblocks_total, 4))] = sc;
  }
}

// ---------------------------------------------------------------------------
// MXFP8 dequantize (see mx_dequantize in mxmoe.h).  HBM-bound: a CTA of
// DQ_THREADS threads covers DQ_COLS columns of one row; a thread takes
// DQ_CHUNKS runs of 16 consecutive E4M3 bytes (16-byte loads, all issued
// before any math; a warp's load reads 512 contiguous bytes) and the scale
// byte of each run's 32-element block.  E4M3 -> f16 pairs (exact: every E4M3
// value is an f16 value) -> fp32, times 2^(s - 127) built from the scale
// byte's bits: all exact in fp32.  Each lane writes whole 32-byte sectors.
// Four runs per thread and the 32-byte stores measured 18% (bf16) and 34%
// (fp32) faster than one run with 16-byte stores.
// ---------------------------------------------------------------------------
constexpr int DQ_THREADS = 128;
constexpr int DQ_CHUNKS = 4;
constexpr int DQ_COLS = DQ_THREADS * 16 * DQ_CHUNKS;

// two fp8 bytes -> fp32 pair, exactly (every E4M3 and E5M2 value, +-Inf and
// NaN included, is an f16 value)
template <bool E5>
__device__ __forceinline__ float2 fp8x2_to_f32x2(uint32_t two_bytes) {
  uint32_t h2;
  if (E5)
    asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)two_bytes));
  else
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)two_bytes));
  return __half22float2(*reinterpret_cast<const __half2 *>(&h2));
}

// 2^(b - 127) for an E8M0 byte: fp32 exponent field b for b >= 1; 2^-127 is
// the fp32 subnormal 0x00400000; 0xFF is NaN.
__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
  return __uint_as_float(b == 0xffu ? 0x7fc00000u : b == 0u ? 0x00400000u : b << 23);
}

template <bool F32>
__device__ __forceinline__ void dq_store16(void *out, int64_t idx, const float (&v)[16]) {
  // whole 32-byte sectors per lane when the output allows it
  if (F32) {
    float *o = static_cast<float *>(out) + idx;
    if (((uintptr_t)o & 31) == 0) {
#pragma unroll
      for (int i = 0; i < 2; ++i)
        asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(o + 8 * i), "f"(v[8 * i]),
                     "f"(v[8 * i + 1]), "f"(v[8 * i + 2]), "f"(v[8 * i + 3]), "f"(v[8 * i + 4]), "f"(v[8 * i + 5]),
                     "f"(v[8 * i + 6]), "f"(v[8 * i + 7])
                     : "memory");
    } else {
      float4 *o4 = reinterpret_cast<float4 *>(o);
#pragma unroll
      for (int i = 0; i < 4; ++i) o4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
  } else {
    uint16_t *o = static_cast<uint16_t *>(out) + idx;
    uint32_t w8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w8[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    if (((uintptr_t)o & 31) == 0) {
      asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(o), "r"(w8[0]), "r"(w8[1]),
                   "r"(w8[2]), "r"(w8[3]), "r"(w8[4]), "r"(w8[5]), "r"(w8[6]), "r"(w8[7])
                   : "memory");
    } else {
      uint4 *o4 = reinterpret_cast<uint4 *>(o);
      o4[0] = make_uint4(w8[0], w8[1], w8[2], w8[3]);
      o4[1] = make_uint4(w8[4], w8[5], w8[6], w8[7]);
    }
  }
}

template <bool F32, bool E5>
__global__ void __launch_bounds__(DQ_THREADS) k_dequantize(const uint8_t *__restrict__ q, const uint8_t *__restrict__ s,
                                                           int64_t rows, int64_t cols, int64_t s_stride, int swizzled,
                                                           void *out) {
  pdl_enter();
  const int64_t grow = blockIdx.x;  // row over all batch entries
  const int64_t b = grow / rows, r = grow - b * rows;
  const int64_t cblocks = cols / 32;
  const uint8_t *sb = s + b * s_stride;
  // DQ_CHUNKS chunks of 16 per thread, DQ_THREADS * 16 elements apart (each
  // load instruction of a warp stays 512 contiguous bytes); loads first
  uint4 w[DQ_CHUNKS];
  uint32_t sbyte[DQ_CHUNKS];
#pragma unroll
  for (int j = 0; j < DQ_CHUNKS; ++j) {
    const int64_t c0 = (int64_t)blockIdx.y * DQ_COLS + j * (DQ_THREADS * 16) + threadIdx.x * 16;
    if (c0 < cols) {
      const int64_t c = c0 >> 5;
      sbyte[j] = __ldg(sb + (swizzled ? sf_swizzle_offset(r, c, round_up(cblocks, 4)) : r * cblocks + c));
      w[j] = __ldg(reinterpret_cast<const uint4 *>(q + grow * cols + c0));
    }
  }
#pragma unroll
  for (int j = 0; j < DQ_CHUNKS; ++j) {
    const int64_t c0 = (int64_t)blockIdx.y * DQ_COLS + j * (DQ_THREADS * 16) + threadIdx.x * 16;
    if (c0 >= cols) continue;
    const float sc = e8m0_to_f32(sbyte[j]);
    const uint32_t wd[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
    float v[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 lo = fp8x2_to_f32x2<E5>(wd[i] & 0xffffu), hi = fp8x2_to_f32x2<E5>(wd[i] >> 16);
      v[4 * i] = lo.x * sc;
      v[4 * i + 1] = lo.y * sc;
      v[4 * i + 2] = hi.x * sc;
      v[4 * i + 3] = hi.y * sc;
    }
    dq_store16<F32>(out, grow * cols + c0, v);
  }
}

// ---------------------------------------------------------------------------
// Row-max-scaled FP8 (see fp8_quantize_rowmax in mxmoe.h): one CTA per row.
// The row is read once from HBM into shared memory (16-byte loads, 8 bf16
// each) while each thread keeps the largest |x| bit pattern it saw; a warp
// shuffle and a shared-memory step give the row's amax.  Then s = amax / 448
// and every element x / s (the IEEE fp32 division the reading defines; see
// rowmax_cast2 for how the kernel reaches the same bytes mostly without
// dividing) is cast to E4M3 with round-to-nearest-even and saturation, 16
// bytes per store.  HBM-bound: 2 bytes read and 1 written per element.
// ---------------------------------------------------------------------------
// E4M3(RN(x / s)) for the two bf16 values of a word, without a division in
// the common case.  q = RN(x * y) with y = RN(1/s) lies within 3 * 2^-24 of
// x / s (relative), and so does RN(x / s).  The E4M3 cast is monotone: when
// both ends of the bracket q * (1 -+ 2^-21) cast to the same byte, so does
// every value between them, RN(x / s) included.  Otherwise (about one element
// in 2^16, where the bracket straddles an E4M3 rounding decision) the byte
// comes from the IEEE division itself; so does every byte of a row whose
// scale is so small (below 2^-128, a row of bf16 subnormals) that 1/s
// overflows.
__device__ __forceinline__ uint16_t rowmax_cast2(float a, float b, float s, float y) {
  const float qa = a * y, qb = b * y;
  constexpr float lo = 1.0f - 0x1p-21f, hi = 1.0f + 0x1p-21f;
  const uint16_t c0 = cvt_e4m3x2(qa * lo, qb * lo), c1 = cvt_e4m3x2(qa * hi, qb * hi);
  return c0 == c1 && y <= 0x1.fffffep127f ? c0 : cvt_e4m3x2(__fdiv_rn(a, s), __fdiv_rn(b, s));
}
__device__ __forceinline__ uint32_t rowmax_cast4(uint32_t w0, uint32_t w1, float s, float y) {
  return (uint32_t)rowmax_cast2(bf16_lo(w0), bf16_hi(w0), s, y) |
         ((uint32_t)rowmax_cast2(bf16_lo(w1), bf16_hi(w1), s, y) << 16);
}

constexpr int RM_THREADS = 128;
constexpr int RM_BATCH = 4;  // 16-byte loads in flight per thread

__global__ void __launch_bounds__(RM_THREADS) k_quantize_rowmax(const uint16_t *__restrict__ x, int64_t cols,
                                                                uint8_t *__restrict__ q, float *__restrict__ scale) {
  pdl_enter();
  extern __shared__ __align__(16) uint4 rm_row[];  // cols / 8 chunks
  __shared__ uint32_t red[RM_THREADS / 32];
  const int tid = threadIdx.x;
  const int64_t r = blockIdx.x;
  const int nch = (int)(cols / 8);
  const uint4 *src = reinterpret_cast<const uint4 *>(x + r * cols);
  uint32_t am = 0;
  for (int i0 = tid; i0 < nch; i0 += RM_THREADS * RM_BATCH) {
    uint4 v[RM_BATCH];
#pragma unroll
    for (int b = 0; b < RM_BATCH; ++b) {  // every load of the batch issued before any use
      const int i = i0 + b * RM_THREADS;
      v[b] = i < nch ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int b = 0; b < RM_BATCH; ++b) {
      const int i = i0 + b * RM_THREADS;
      if (i < nch) rm_row[i] = v[b];
      const uint32_t m = vmax_u16x2(vmax_u16x2(v[b].x & 0x7fff7fffu, v[b].y & 0x7fff7fffu),
                                    vmax_u16x2(v[b].z & 0x7fff7fffu, v[b].w & 0x7fff7fffu));
      am = max(am, max(m << 16, m & 0xffff0000u));  // as fp32 bit patterns
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) am = max(am, __shfl_xor_sync(0xffffffffu, am, o));
  if ((tid & 31) == 0) red[tid >> 5] = am;
  __syncthreads();
  am = red[0];
#pragma unroll
  for (int w = 1; w < RM_THREADS / 32; ++w) am = max(am, red[w]);
  const bool bad = am >= 0x7f800000u;  // NaN or Inf in the row
  const float amax = __uint_as_float(am);
  const float s = bad ? __uint_as_float(0x7fc00000u) : (am == 0 ? 1.0f : __fdiv_rn(amax, 448.0f));
  const float y = __frcp_rn(s);  // correctly rounded 1 / s
  if (tid == 0) scale[r] = s;
  uint4 *dst = reinterpret_cast<uint4 *>(q + r * cols);
  for (int i = tid; i < nch / 2; i += RM_THREADS) {
    const uint4 a = rm_row[2 * i], b = rm_row[2 * i + 1];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = bad ? 0x7f7f7f7fu : rowmax_cast4(w[2 * j], w[2 * j + 1], s, y);
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// The quantize kernel for one combination of outputs, gather mode and
// element format (E5: E5M2).
template <bool GATHER>
static void launch_quantize(const QuantArgs &a, bool row, bool col, bool e5, dim3 grid, mx_stream stream) {
  if (e5) {
    if (row && col) (void)launch_k(k_quantize_bf16<true, true, GATHER, true>, grid, QT_THREADS, 0, stream, a);
    else if (row) (void)launch_k(k_quantize_bf16<true, false, GATHER, true>, grid, QT_THREADS, 0, stream, a);
    else (void)launch_k(k_quantize_bf16<false, true, GATHER, true>, grid, QT_THREADS, 0, stream, a);
  } else {
    if (row && col) (void)launch_k(k_quantize_bf16<true, true, GATHER, false>, grid, QT_THREADS, 0, stream, a);
    else if (row) (void)launch_k(k_quantize_bf16<true, false, GATHER, false>, grid, QT_THREADS, 0, stream, a);
    else (void)launch_k(k_quantize_bf16<false, true, GATHER, false>, grid, QT_THREADS, 0, stream, a);
  }
}

}  // namespace mxmoe

using namespace mxmoe;

extern "C" mx_status fp8_quantize_rowmax(const void *x, int64_t rows, int64_t cols, uint8_t *q, float *row_scale,
                                         mx_stream stream) {
  MX_HOST_CHECK(rows >= 0 && cols > 0, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(rows == 0 || (x && q && row_scale), MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(cols % 16 == 0 && cols <= 102400 && rows < (int64_t)1 << 31, MX_ERR_SHAPE);
  MX_HOST_CHECK(aligned16(x) && aligned16(q) && aligned4(row_scale), MX_ERR_ALIGNMENT);
  mx_status st = check_device_cached();
  if (st != MX_OK) return st;
  if (rows == 0) return MX_OK;
  const int smem = (int)(cols * 2);
  if (smem > 48 * 1024) {
    static int set[64];
    int dev = 0;
    MX_CUDA_TRY(cudaGetDevice(&dev));
    if (dev >= 0 && dev < 64 && !set[dev]) {
      MX_CUDA_TRY(cudaFuncSetAttribute(k_quantize_rowmax, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024));
      set[dev] = 1;
    }
  }
  (void)launch_k(k_quantize_rowmax, (unsigned)rows, RM_THREADS, smem, stream, static_cast<const uint16_t *>(x), cols, q,
                                                                   row_scale);
  return launch_status();
}

extern "C" int64_t mx_scale_bytes(int64_t rows, int64_t cols, int32_t layout) {
  if (rows < 0 || cols < 0 || cols % 32) return -1;
  if (layout == MX_SCALE_SWIZZLED) return round_up(rows, 128) * round_up(cols / 32, 4);
  return rows * (cols / 32);
}

extern "C" mx_status mx_quantize(const void *x, int64_t batch, int64_t rows, int64_t cols, int32_t mode,
                                 int32_t scale_layout, int32_t elem, uint8_t *q_row, uint8_t *s_row, uint8_t *q_col,
                                 uint8_t *s_col, mx_stream stream) {
  MX_HOST_CHECK(x != nullptr, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(mode == MX_MODE_ROW || mode == MX_MODE_COL || mode == MX_MODE_BOTH, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(scale_layout == MX_SCALE_PLAIN || scale_layout == MX_SCALE_SWIZZLED, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(elem == MX_ELEM_E4M3 || elem == MX_ELEM_E5M2, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(batch >= 1 && rows >= 1 && cols >= 1, MX_ERR_INVALID_ARG);
  const bool row = mode & MX_MODE_ROW, col = mode & MX_MODE_COL;
  MX_HOST_CHECK(!row || (q_row && s_row), MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(!col || (q_col && s_col), MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(cols % 32 == 0 && (!col || rows % 32 == 0), MX_ERR_SHAPE);
  MX_HOST_CHECK(aligned16(x) && (!row || aligned16(q_row)) && (!col || aligned16(q_col)), MX_ERR_ALIGNMENT);
  MX_HOST_CHECK(rows / QT_ROWS < 65535 && cols / QT_COLS < 65535 && batch < 65535, MX_ERR_SHAPE);
  mx_status st = check_device_cached();
  if (st != MX_OK) return st;
  QuantArgs a;
  a.src = nullptr;
  a.gate = nullptr;
  a.k = 1;
  a.row_limit = nullptr;
  a.x = static_cast<const uint16_t *>(x);
  a.rows = rows;
  a.cols = cols;
  a.q_row = q_row;
  a.s_row = s_row;
  a.q_col = q_col;
  a.s_col = s_col;
  a.s_row_stride = mx_scale_bytes(rows, cols, scale_layout);
  a.s_col_stride = mx_scale_bytes(cols, rows, scale_layout);
  a.swizzled = scale_layout == MX_SCALE_SWIZZLED;
  // swizzled layouts carry zero padding that the kernel does not visit
  if (a.swizzled) {
    if (row && (rows % 128 || (cols / 32) % 4))
      MX_CUDA_TRY(cudaMemsetAsync(s_row, 0, a.s_row_stride * batch, stream));
    if (col && (cols % 128 || (rows / 32) % 4))
      MX_CUDA_TRY(cudaMemsetAsync(s_col, 0, a.s_col_stride * batch, stream));
  }
  const unsigned nrb = (unsigned)((rows + QT_ROWS - 1) / QT_ROWS), ncb = (unsigned)((cols + QT_COLS - 1) / QT_COLS);
  const dim3 grid = row ? dim3(ncb, nrb, (unsigned)batch) : dim3(nrb, ncb, (unsigned)batch);
  launch_quantize<false>(a, row, col, elem == MX_ELEM_E5M2, grid, stream);
  return launch_status();
}

extern "C" mx_status mx_dequantize(const uint8_t *q, const uint8_t *s, int64_t batch, int64_t rows, int64_t cols,
                                   int32_t scale_layout, int32_t elem, int32_t out_dtype, void *out,
                                   mx_stream stream) {
  MX_HOST_CHECK(q && s && out, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(scale_layout == MX_SCALE_PLAIN || scale_layout == MX_SCALE_SWIZZLED, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(elem == MX_ELEM_E4M3 || elem == MX_ELEM_E5M2, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(out_dtype == MX_OUT_BF16 || out_dtype == MX_OUT_F32, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(batch >= 1 && rows > 0 && cols > 0, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(cols % 32 == 0, MX_ERR_SHAPE);
  MX_HOST_CHECK(batch * rows < (int64_t)1 << 31 && (cols + DQ_COLS - 1) / DQ_COLS < 65535, MX_ERR_SHAPE);
  MX_HOST_CHECK(aligned16(q) && aligned16(out), MX_ERR_ALIGNMENT);
  mx_status st = check_device_cached();
  if (st != MX_OK) return st;
  const dim3 grid((unsigned)(batch * rows), (unsigned)((cols + DQ_COLS - 1) / DQ_COLS));
  const int64_t s_stride = mx_scale_bytes(rows, cols, scale_layout);
  const int swz = scale_layout == MX_SCALE_SWIZZLED;
  const bool e5 = elem == MX_ELEM_E5M2;
  if (out_dtype == MX_OUT_F32 && e5)
    (void)launch_k(k_dequantize<true, true>, grid, DQ_THREADS, 0, stream, q, s, rows, cols, s_stride, swz, out);
  else if (out_dtype == MX_OUT_F32)
    (void)launch_k(k_dequantize<true, false>, grid, DQ_THREADS, 0, stream, q, s, rows, cols, s_stride, swz, out);
  else if (e5)
    (void)launch_k(k_dequantize<false, true>, grid, DQ_THREADS, 0, stream, q, s, rows, cols, s_stride, swz, out);
  else
    (void)launch_k(k_dequantize<false, false>, grid, DQ_THREADS, 0, stream, q, s, rows, cols, s_stride, swz, out);
  return launch_status();
}

extern "C" mx_status moe_gather_quant(const void *x, const float *gate, const int32_t *src, int64_t T, int64_t H,
                                      int32_t k, int64_t rows_cap, int32_t mode, int32_t elem, uint8_t *q_row,
                                      uint8_t *s_row, uint8_t *q_col, uint8_t *s_col, const int32_t *row_limit,
                                      mx_stream stream) {
  MX_HOST_CHECK(src && (T == 0 || x), MX_ERR_INVALID_ARG);  // T = 0: every row is a zero pad row
  MX_HOST_CHECK(mode == MX_MODE_ROW || mode == MX_MODE_COL || mode == MX_MODE_BOTH, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(elem == MX_ELEM_E4M3 || elem == MX_ELEM_E5M2, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(T >= 0 && H > 0 && k >= 1 && rows_cap >= 0, MX_ERR_INVALID_ARG);
  const bool row = mode & MX_MODE_ROW, col = mode & MX_MODE_COL;
  MX_HOST_CHECK(!row || (q_row && s_row), MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(!col || (q_col && s_col), MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(H % 128 == 0 && rows_cap % 128 == 0 && H / QT_COLS < 65535, MX_ERR_SHAPE);
  MX_HOST_CHECK(aligned16(x) && (!row || aligned16(q_row)) && (!col || aligned16(q_col)), MX_ERR_ALIGNMENT);
  mx_status st = check_device_cached();
  if (st != MX_OK) return st;
  if (rows_cap == 0) return MX_OK;
  QuantArgs a;
  a.x = static_cast<const uint16_t *>(x);
  a.rows = rows_cap;
  a.cols = H;
  a.src = src;
  a.gate = gate;
  a.k = k;
  a.row_limit = row_limit;
  a.q_row = q_row;
  a.s_row = s_row;
  a.q_col = q_col;
  a.s_col = s_col;
  a.s_row_stride = 0;
  a.s_col_stride = 0;
  a.swizzled = 1;
  const unsigned nrb = (unsigned)(rows_cap / QT_ROWS), ncb = (unsigned)(H / QT_COLS);
  MX_HOST_CHECK(nrb < 65535 || !row, MX_ERR_SHAPE);
  const dim3 grid = row ? dim3(ncb, nrb, 1) : dim3(nrb, ncb, 1);
  launch_quantize<true>(a, row, col, elem == MX_ELEM_E5M2, grid, stream);
  return launch_status();
}

extern "C" mx_status moe_swiglu_bwd(const float *dh, const void *ab, int64_t rows, int64_t F, int32_t grad_elem,
                                    uint8_t *dab_rq, uint8_t *dab_rs, uint8_t *dab_cq, uint8_t *dab_cs, uint8_t *h_cq,
                                    uint8_t *h_cs, const int32_t *row_limit, mx_stream stream) {
  MX_HOST_CHECK(dh && ab && dab_rq && dab_rs && dab_cq && dab_cs && h_cq && h_cs, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(grad_elem == MX_ELEM_E4M3 || grad_elem == MX_ELEM_E5M2, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(rows >= 0 && F > 0, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(rows % SB_ROWS == 0 && F % SB_COLS == 0 && F / SB_COLS < 65535, MX_ERR_SHAPE);
  MX_HOST_CHECK(aligned16(dh) && aligned16(ab) && aligned16(dab_rq) && aligned16(dab_cq) && aligned16(h_cq),
                MX_ERR_ALIGNMENT);
  mx_status st = check_device_cached();
  if (st != MX_OK) return st;
  if (rows == 0) return MX_OK;
  static int smem_set[64];
  int dev = 0;
  MX_CUDA_TRY(cudaGetDevice(&dev));
  if (dev >= 0 && dev < 64 && !smem_set[dev]) {
    MX_CUDA_TRY(cudaFuncSetAttribute(k_swiglu_bwd<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SB_SMEM));
    MX_CUDA_TRY(cudaFuncSetAttribute(k_swiglu_bwd<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SB_SMEM));
    smem_set[dev] = 1;
  }
  dim3 grid((unsigned)(rows / SB_ROWS), (unsigned)(F / SB_COLS));
  const uint16_t *abp = static_cast<const uint16_t *>(ab);
  if (grad_elem == MX_ELEM_E5M2)
    (void)launch_k(k_swiglu_bwd<true>, grid, SB_THREADS, SB_SMEM, stream, dh, abp, rows, F, dab_rq, dab_rs, dab_cq, dab_cs, h_cq,
                                                              h_cs, row_limit);
  else
    (void)launch_k(k_swiglu_bwd<false>, grid, SB_THREADS, SB_SMEM, stream, dh, abp, rows, F, dab_rq, dab_rs, dab_cq, dab_cs, h_cq,
                                                               h_cs, row_limit);
  return launch_status();
}
