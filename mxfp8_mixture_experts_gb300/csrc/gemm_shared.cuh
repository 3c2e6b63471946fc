// Pieces shared by the two grouped-GEMM kernels (one CTA per tile, and a CTA
// pair per 256-row tile): parameters, the tcgen05 instruction descriptor, the
// epilogue conversions and stores, and the tensor-map helpers.
#pragma once

#include "common.cuh"

namespace mxmoe {
namespace gemm {

constexpr int BM = 128;  // rows of one CTA's accumulator (TMEM lanes)
constexpr int BN = 256;  // accumulator columns (TMEM columns)
constexpr int BK = 128;  // fp8 elements (= bytes) per row per pipeline stage
constexpr int MAX_E = 1024;
constexpr uint64_t WAIT_TIMEOUT_NS = 2000000000ull;
constexpr int NUM_EPI_WARPS = 8;

enum { EPI_BF16 = 0, EPI_F32 = 1, EPI_GLU = 2 };
enum { OP_ROWS = 0, OP_TOKENS = 1 };

struct Params {
  int op, epi, E;
  int64_t M_cap, N, K;  // see mx_grouped_gemm; for EPI_GLU N = F (output feature pairs)
  const int32_t *offsets;
  const uint8_t *sA, *sB;
  void *C;
  uint16_t *ab;
  uint8_t *hq, *hs;
  int32_t *dev_status;
  uint32_t idesc_fmt;  // element formats of A and B as instruction-descriptor bits (idesc_formats)
};

// Instruction descriptor, kind::mxf8f6f4 with block scales: E4M3 x E4M3 (format
// 0 in bits 7-9 and 10-12), both operands K-major (bits 15, 16 clear), N>>3 in
// bits 17-22, UE8M0 scales (bit 23), M>>4 in bits 24-28.  Bits 4-5 (B) and
// 29-30 (A) pick the byte, i.e. the 32-wide K block, of the 32-bit scale
// column in TMEM; they are OR-ed in per MMA.
__host__ __device__ constexpr uint32_t idesc_mxf8(int M, int N) {
  return (0u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 4) << 24);
}
// Element formats of the two operands in the same descriptor: A's in bits
// 7-9, B's in bits 10-12, E4M3 = 0 and E5M2 = 1 (kind::mxf8f6f4 takes the two
// independently).
__host__ __device__ constexpr uint32_t idesc_formats(int a_e5m2, int b_e5m2) {
  return ((uint32_t)(a_e5m2 ? 1 : 0) << 7) | ((uint32_t)(b_e5m2 ? 1 : 0) << 10);
}

// h = silu(a) * b = a * sigma(a) * b in fp32 for bf16 a, b (sigma from
// sigmoid_parts: within a few fp32 ulps of the exact value over the whole
// bf16 range of a that matters, with one final rounding into the subnormal
// range for very negative a).
__device__ __forceinline__ float swiglu_h(float a, float b) {
  const SigParts p = sigmoid_parts(a);
  return ((a * p.s) * b) * p.back;
}

// Validate the group offsets (identically in every CTA): non-decreasing,
// multiples of 128, last one within M_cap.
__device__ __forceinline__ int offsets_ok(const int32_t *off, int E, int64_t M_cap) {
  for (int i = 0; i < E; ++i)
    if (off[i + 1] < off[i] || (off[i] & (BM - 1))) return 0;
  if (off[0] < 0 || (off[E] & (BM - 1)) || off[E] > M_cap) return 0;
  return 1;
}

__device__ __forceinline__ int upper_group(const int32_t *pref, int E, int64_t x) {
  int lo = 0, hi = E;  // largest e with pref[e] <= x
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pref[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

// Zero the output columns [col0, col0 + ncols) of row `orow` (empty wgrad
// group); ncols is a multiple of 8.
__device__ __forceinline__ void epi_zero(const Params &p, int64_t orow, int64_t col0, int ncols = 128) {
  const int64_t ldc = p.op == OP_ROWS ? p.N : p.K;
  if (p.epi == EPI_F32) {
    float4 *c = reinterpret_cast<float4 *>(static_cast<float *>(p.C) + orow * ldc + col0);
    for (int j = 0; j < ncols / 4; ++j) c[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  } else {
    uint4 *c = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.C) + orow * ldc + col0);
    for (int j = 0; j < ncols / 8; ++j) c[j] = make_uint4(0, 0, 0, 0);
  }
}

// Store one thread's accumulator slice.
//   EPI_F32 / EPI_BF16: r[0..127] = columns [col0, col0+128) of row `orow`.
//   EPI_GLU: r[0..63] = a, r[64..127] = b for features [col0, col0+64) of row
//   `orow`; a, b are rounded to bf16 and saved, h = silu(a) * b is quantized
//   (two 32-element blocks) into hq / hs.
__device__ __forceinline__ void epi_store(const Params &p, int64_t orow, int64_t col0, const uint32_t (&r)[128]) {
  if (p.epi == EPI_F32) {
    const int64_t ldc = p.op == OP_ROWS ? p.N : p.K;
    float4 *c = reinterpret_cast<float4 *>(static_cast<float *>(p.C) + orow * ldc + col0);
#pragma unroll
    for (int j = 0; j < 32; ++j)
      c[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]), __uint_as_float(r[4 * j + 2]),
                         __uint_as_float(r[4 * j + 3]));
  } else if (p.epi == EPI_BF16) {
    const int64_t ldc = p.op == OP_ROWS ? p.N : p.K;
    uint4 *c = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.C) + orow * ldc + col0);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint32_t *v = r + 8 * j;
      c[j] = make_uint4(pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1])),
                        pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3])),
                        pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5])),
                        pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7])));
    }
  } else {
    const int64_t F = p.N;
    uint4 *pa = reinterpret_cast<uint4 *>(p.ab + orow * 2 * F + col0);
    uint4 *pb = reinterpret_cast<uint4 *>(p.ab + orow * 2 * F + F + col0);
    uint4 *ph = reinterpret_cast<uint4 *>(p.hq + orow * F + col0);
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      float hv[32];
      uint32_t am = 0;
#pragma unroll
      for (int j = 0; j < 32; j += 8) {
        float av[8], bv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          av[i] = round_bf16(__uint_as_float(r[blk * 32 + j + i]));
          bv[i] = round_bf16(__uint_as_float(r[64 + blk * 32 + j + i]));
          hv[j + i] = swiglu_h(av[i], bv[i]);
          am = max(am, abs_bits(hv[j + i]));
        }
        pa[(blk * 32 + j) / 8] = make_uint4(pack_bf16x2(av[0], av[1]), pack_bf16x2(av[2], av[3]),
                                            pack_bf16x2(av[4], av[5]), pack_bf16x2(av[6], av[7]));
        pb[(blk * 32 + j) / 8] = make_uint4(pack_bf16x2(bv[0], bv[1]), pack_bf16x2(bv[2], bv[3]),
                                            pack_bf16x2(bv[4], bv[5]), pack_bf16x2(bv[6], bv[7]));
      }
      const MxScale s = mx_scale_from_amax_bits(am);
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        w[i] = s.bad ? 0x7f7f7f7fu
                     : pack_e4m3x4(hv[4 * i] * s.inv, hv[4 * i + 1] * s.inv, hv[4 * i + 2] * s.inv,
                                   hv[4 * i + 3] * s.inv);
      ph[blk * 2] = make_uint4(w[0], w[1], w[2], w[3]);
      ph[blk * 2 + 1] = make_uint4(w[4], w[5], w[6], w[7]);
      p.hs[sf_swizzle_offset(orow, col0 / 32 + blk, round_up(F / 32, 4))] = (uint8_t)s.byte;
    }
  }
}

// host
mx_status make_map_u8_128x128(CUtensorMap *m, const void *base, int64_t inner, int64_t outer);
mx_status make_map_u8_128x128_swz(CUtensorMap *m, const void *base, int64_t inner, int64_t outer, int swizzle);
// 2-D uint8 map over [outer, inner], boxes of 128 bytes x box_rows
mx_status make_map_u8_box_swz(CUtensorMap *m, const void *base, int64_t inner, int64_t outer, int box_rows,
                              int swizzle);
mx_status make_map_sf_chunks(CUtensorMap *m, const void *base, int64_t nchunks);
mx_status make_map_store_64b(CUtensorMap *m, void *base, bool f32, int64_t cols, int64_t rows);
mx_status make_map_store_64b_u8(CUtensorMap *m, void *base, int64_t cols, int64_t rows);
mx_status launch_1cta(const Params &p, const uint8_t *A, int64_t a_inner, int64_t a_outer, const uint8_t *B,
                      int64_t b_inner, int64_t b_outer, int64_t max_tiles, mx_stream stream);
mx_status launch_pair(const Params &p, const uint8_t *A, int64_t a_inner, int64_t a_outer, const uint8_t *B,
                      int64_t b_inner, int64_t b_outer, int64_t sfa_bytes, int64_t sfb_bytes, mx_stream stream);

}  // namespace gemm
}  // namespace mxmoe
