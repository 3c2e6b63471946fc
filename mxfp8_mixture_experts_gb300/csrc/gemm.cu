// Block-scaled MXFP8 grouped GEMM on the sm_100-family 5th-generation tensor
// cores (tcgen05), written for GB300 (sm_103a).
//
// "1.5x faster MoE training on Blackwell with MXFP8 kernels built from
// scratch", Key Questions Answered: the tcgen05.mma block-scaled MMA
// accumulates in tensor memory (TMEM) and runs asynchronously; moving data
// between TMEM and registers costs latency and the fp32 CUDA cores are far
// slower than the tensor cores, so the scales are applied inside the MMA (no
// software dequantize) and the epilogue reads TMEM exactly once.
// pytorch/ao "mxfp8 moe training" PR, Next steps: the grouped GEMM takes
// pre-quantized operands together with their E8M0 scales.
//
// Kernel structure (one persistent CTA per SM, 320 threads):
//   warp 0      TMA producer: per 128-wide K step, one 128x128 A tile, two
//               128x128 B tiles (128-byte swizzle) and the matching E8M0
//               scale chunks (512 B each, already in the MMA's tile layout)
//               into a 4-stage shared-memory ring.
//   warp 1      allocates TMEM; one thread copies the scale chunks into TMEM
//               (tcgen05.cp 32x128b.warpx4) and issues 4 block-scaled MMAs
//               (M=128, N=256, K=32 each) per stage; tcgen05.commit frees the
//               stage and, after the last K step, signals the epilogue.
//   warps 2..9  epilogue: tcgen05.ld of the 128x256 fp32 accumulator (each
//               warp a 32-lane quarter x 128 columns), release of the
//               accumulator to the MMA warp, then the conversion and global
//               stores (bf16, fp32, or the fused SwiGLU + MXFP8 quantize).
// Group offsets stay on the device: every CTA walks the same static tile
// schedule derived from them (no host synchronization).
#include "gemm_shared.cuh"
#include <cstdlib>

#include <mutex>

namespace mxmoe {
namespace gemm {

// one-CTA variant: 128 x 256 tile per CTA, 4-stage ring
constexpr int STAGES = 4;
constexpr int A_TILE = BM * BK;          // 16 KB
constexpr int B_HALF = 128 * BK;         // 16 KB (one TMA box)
constexpr int B_TILE = BN * BK;          // 32 KB
constexpr int SF_STAGE = 512 + 1024;     // SFA chunk + two SFB chunks
constexpr uint32_t STAGE_TX = A_TILE + B_TILE + SF_STAGE;
constexpr int NUM_THREADS = 320;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;
constexpr uint32_t SF_COL = 256;  // per stage: SFA 4 columns, SFB 8 columns

constexpr int SMEM_A = 0;
constexpr int SMEM_B = SMEM_A + STAGES * A_TILE;
constexpr int SMEM_SF = SMEM_B + STAGES * B_TILE;
constexpr int SMEM_BAR = SMEM_SF + STAGES * SF_STAGE;
constexpr int SMEM_OFFS = SMEM_BAR + 256;
constexpr int SMEM_TOTAL = SMEM_OFFS + (MAX_E + 1) * 4;
constexpr int SMEM_ALLOC = SMEM_TOTAL + 1024;  // slack to align the base to 1024

__host__ __device__ constexpr uint32_t idesc_base() { return idesc_mxf8(BM, BN); }

struct Tile {
  int64_t a_row, b_row0, b_row1;  // TMA row coordinates
  int64_t k0;                     // first contraction coordinate
  int num_k;                      // 128-wide K steps (0: empty wgrad group)
  int64_t sfa_base, sfb_base0, sfb_base1;  // byte offsets of the k=0 scale chunks
  int64_t out_row, out_col;       // output position of the tile's top-left
  int e;
};

__device__ __forceinline__ int64_t num_tiles(const Params &p, const int32_t *off) {
  if (p.op == OP_ROWS) {
    const int64_t n_tiles = p.epi == EPI_GLU ? p.N / 128 : p.N / BN;
    return (int64_t)(off[p.E] / BM) * n_tiles;
  }
  return (int64_t)p.E * (p.N / BM) * (p.K / BN);
}

__device__ __forceinline__ Tile decode_tile(const Params &p, const int32_t *off, int64_t t) {
  Tile tl;
  if (p.op == OP_ROWS) {
    const int64_t n_tiles = p.epi == EPI_GLU ? p.N / 128 : p.N / BN;
    const int64_t mt = t / n_tiles, nt = t % n_tiles;
    const int64_t row = mt * BM;
    const int e = upper_group(off, p.E, row);
    const int64_t kblocks = p.K / BK;
    tl.e = e;
    tl.a_row = row;
    if (p.epi == EPI_GLU) {  // B rows: W1 part then W3 part of the same 128 output features
      tl.b_row0 = (int64_t)e * 2 * p.N + nt * 128;
      tl.b_row1 = tl.b_row0 + p.N;
      tl.out_col = nt * 128;
    } else {
      tl.b_row0 = (int64_t)e * p.N + nt * BN;
      tl.b_row1 = tl.b_row0 + 128;
      tl.out_col = nt * BN;
    }
    tl.k0 = 0;
    tl.num_k = (int)kblocks;
    tl.sfa_base = (row / 128) * kblocks * 512;
    tl.sfb_base0 = (tl.b_row0 / 128) * kblocks * 512;
    tl.sfb_base1 = (tl.b_row1 / 128) * kblocks * 512;
    tl.out_row = row;
  } else {
    const int64_t rt_n = p.N / BM, ct_n = p.K / BN;
    const int64_t per_e = rt_n * ct_n;
    const int e = (int)(t / per_e);
    const int64_t rem = t % per_e;
    const int64_t rt = rem / ct_n, ct = rem % ct_n;
    const int64_t kblocks = p.M_cap / BK;  // scale chunks per row tile
    tl.e = e;
    tl.a_row = rt * BM;
    tl.b_row0 = ct * BN;
    tl.b_row1 = tl.b_row0 + 128;
    tl.k0 = off[e];
    tl.num_k = (off[e + 1] - off[e]) / BK;
    tl.sfa_base = (rt * kblocks + off[e] / BK) * 512;
    tl.sfb_base0 = ((tl.b_row0 / 128) * kblocks + off[e] / BK) * 512;
    tl.sfb_base1 = ((tl.b_row1 / 128) * kblocks + off[e] / BK) * 512;
    tl.out_row = (int64_t)e * p.N + rt * BM;
    tl.out_col = ct * BN;
  }
  return tl;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_grouped_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, Params p) {
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + SMEM_BAR);
  uint64_t *empty = full + STAGES;
  uint64_t *tmem_full = empty + STAGES;
  uint64_t *tmem_empty = tmem_full + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tmem_empty + 1);
  int32_t *s_flag = reinterpret_cast<int32_t *>(tmem_slot + 1);
  int32_t *s_off = reinterpret_cast<int32_t *>(smem + SMEM_OFFS);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // group offsets -> shared memory, validated identically by every CTA
  for (int i = threadIdx.x; i <= p.E; i += NUM_THREADS) s_off[i] = p.offsets[i];
  __syncthreads();
  if (threadIdx.x == 0) {
    const int ok = offsets_ok(s_off, p.E, p.M_cap);
    *s_flag = ok;
    if (!ok && blockIdx.x == 0) set_status(p.dev_status, MX_ERR_DEVICE);
  }
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tmem_full, 1);
    mbar_init(tmem_empty, NUM_EPI_WARPS);
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  __syncthreads();
  if (!*s_flag) return;
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int64_t ntiles = num_tiles(p, s_off);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // the whole warp runs the loop; one elected lane issues the copies
    {
      int stage = 0;
      uint32_t phase = 0;
      bool dead = false;
      for (int64_t t = blockIdx.x; t < ntiles && !dead; t += gridDim.x) {
        const Tile tl = decode_tile(p, s_off, t);
        for (int kb = 0; kb < tl.num_k; ++kb) {
          if (!mbar_wait_warp(&empty[stage], phase ^ 1, WAIT_TIMEOUT_NS)) {
            if (lane == 0) set_status(p.dev_status, MX_ERR_TIMEOUT);
            dead = true;
            break;
          }
          if (elect_one_sync()) {
            uint8_t *sa = smem + SMEM_A + stage * A_TILE;
            uint8_t *sb = smem + SMEM_B + stage * B_TILE;
            uint8_t *sf = smem + SMEM_SF + stage * SF_STAGE;
            const int32_t kc = (int32_t)(tl.k0 + (int64_t)kb * BK);
            mbar_arrive_expect_tx(&full[stage], STAGE_TX);
            tma_load_2d(sa, &tmA, &full[stage], kc, (int32_t)tl.a_row);
            tma_load_2d(sb, &tmB, &full[stage], kc, (int32_t)tl.b_row0);
            tma_load_2d(sb + B_HALF, &tmB, &full[stage], kc, (int32_t)tl.b_row1);
            bulk_load(sf, p.sA + tl.sfa_base + (int64_t)kb * 512, 512, &full[stage]);
            bulk_load(sf + 512, p.sB + tl.sfb_base0 + (int64_t)kb * 512, 512, &full[stage]);
            bulk_load(sf + 1024, p.sB + tl.sfb_base1 + (int64_t)kb * 512, 512, &full[stage]);
          }
          __syncwarp();
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // the whole warp runs the loop and waits; one elected lane issues
    {
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool dead = false;
      const uint32_t d_tmem = tmem_base + ACC_COL;
      for (int64_t t = blockIdx.x; t < ntiles && !dead; t += gridDim.x) {
        const Tile tl = decode_tile(p, s_off, t);
        if (tl.num_k == 0) continue;
        if (!mbar_wait_warp(tmem_empty, acc_phase ^ 1, WAIT_TIMEOUT_NS)) {
          if (lane == 0) set_status(p.dev_status, MX_ERR_TIMEOUT);
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < tl.num_k; ++kb) {
          if (!mbar_wait_warp(&full[stage], phase, WAIT_TIMEOUT_NS)) {
            if (lane == 0) set_status(p.dev_status, MX_ERR_TIMEOUT);
            dead = true;
            break;
          }
          tc_fence_after();
          if (elect_one_sync()) {
          const uint32_t sa = smem_u32(smem + SMEM_A + stage * A_TILE);
          const uint32_t sb = smem_u32(smem + SMEM_B + stage * B_TILE);
          const uint32_t sf = smem_u32(smem + SMEM_SF + stage * SF_STAGE);
          const uint32_t sfa_t = tmem_base + SF_COL + stage * 12;
          const uint32_t sfb_t = sfa_t + 4;
          tc_cp_32x128b_warpx4(sfa_t, smem_desc(sf, 0, 128, 0));
          tc_cp_32x128b_warpx4(sfb_t, smem_desc(sf + 512, 0, 128, 0));
          tc_cp_32x128b_warpx4(sfb_t + 4, smem_desc(sf + 1024, 0, 128, 0));
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {
            const uint64_t ad = smem_desc(sa + kk * 32, 16, 1024, 2);
            const uint64_t bd = smem_desc(sb + kk * 32, 16, 1024, 2);
            const uint32_t id = idesc_base() | p.idesc_fmt | ((uint32_t)kk << 4) | ((uint32_t)kk << 29);
            tc_mma_mxf8(d_tmem, ad, bd, id, sfa_t, sfb_t, (kb | kk) != 0);
          }
          tc_commit(&empty[stage]);
          }
          __syncwarp();
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (dead) break;
        if (elect_one_sync()) tc_commit(tmem_full);
        __syncwarp();
        acc_phase ^= 1;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;             // TMEM lane quarter this warp may read
    const int h = (warp - 2) >> 2;      // which half of the columns
    const int row_in_tile = q * 32 + lane;
    const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + ACC_COL;
    uint32_t acc_phase = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
      const Tile tl = decode_tile(p, s_off, t);
      const int64_t orow = tl.out_row + row_in_tile;
      if (tl.num_k == 0) {  // empty wgrad group: the output block is zero
        epi_zero(p, orow, tl.out_col + h * 128);
        continue;
      }
      if (!mbar_wait_warp(tmem_full, acc_phase, WAIT_TIMEOUT_NS)) {
        if (lane == 0) set_status(p.dev_status, MX_ERR_TIMEOUT);
        break;
      }
      tc_fence_after();
      uint32_t r[128];
      if (p.epi == EPI_GLU) {
        // a columns [h*64, h*64+64), b columns [128 + h*64, ...)
        MX_TMEM_LD_32x32b_x32(t_row + h * 64, r);
        MX_TMEM_LD_32x32b_x32(t_row + h * 64 + 32, (r + 32));
        MX_TMEM_LD_32x32b_x32(t_row + 128 + h * 64, (r + 64));
        MX_TMEM_LD_32x32b_x32(t_row + 128 + h * 64 + 32, (r + 96));
      } else {
        MX_TMEM_LD_32x32b_x32(t_row + h * 128, r);
        MX_TMEM_LD_32x32b_x32(t_row + h * 128 + 32, (r + 32));
        MX_TMEM_LD_32x32b_x32(t_row + h * 128 + 64, (r + 64));
        MX_TMEM_LD_32x32b_x32(t_row + h * 128 + 96, (r + 96));
      }
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tmem_empty);
      acc_phase ^= 1;
      epi_store(p, orow, tl.out_col + (p.epi == EPI_GLU ? h * 64 : h * 128), r);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// 2-D uint8 map over [outer, inner] (inner contiguous), 128x128 boxes, 128-byte swizzle
mx_status make_map_u8_128x128(CUtensorMap *m, const void *base, int64_t inner, int64_t outer) {
  return make_map_u8_128x128_swz(m, base, inner, outer, (int)CU_TENSOR_MAP_SWIZZLE_128B);
}

mx_status make_map_u8_128x128_swz(CUtensorMap *m, const void *base, int64_t inner, int64_t outer, int swizzle) {
  return make_map_u8_box_swz(m, base, inner, outer, 128, swizzle);
}

mx_status make_map_u8_box_swz(CUtensorMap *m, const void *base, int64_t inner, int64_t outer, int box_rows,
                              int swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return MX_ERR_CUDA;
  if (box_rows < 1 || box_rows > 256) return MX_ERR_INVALID_ARG;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)inner};
  cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, (CUtensorMapSwizzle)swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MX_OK : MX_ERR_CUDA;
}

// a swizzled scale array seen as [nchunks, 128] uint32: one box = one 512-byte
// chunk (128 rows x 4 scale columns)
mx_status make_map_sf_chunks(CUtensorMap *m, const void *base, int64_t nchunks) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return MX_ERR_CUDA;
  cuuint64_t dims[2] = {128, (cuuint64_t)nchunks};
  cuuint64_t strides[1] = {512};
  cuuint32_t box[2] = {128, 1};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MX_OK : MX_ERR_CUDA;
}

// output store map: [rows, cols] fp32 or bf16, boxes of 32 rows x 64 bytes,
// 64-byte swizzle (matches the epilogue's staging layout)
mx_status make_map_store_64b(CUtensorMap *m, void *base, bool f32, int64_t cols, int64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return MX_ERR_CUDA;
  const int64_t esz = f32 ? 4 : 2;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(cols * esz)};
  cuuint32_t box[2] = {(cuuint32_t)(64 / esz), 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MX_OK : MX_ERR_CUDA;
}

// uint8 variant: [rows, cols] bytes, boxes of 32 rows x 64 bytes, 64-byte swizzle
mx_status make_map_store_64b_u8(CUtensorMap *m, void *base, int64_t cols, int64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return MX_ERR_CUDA;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols};
  cuuint32_t box[2] = {64, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MX_OK : MX_ERR_CUDA;
}

static std::mutex g_mu;
static int g_smem_set[64];
static int g_num_sms[64];

static mx_status prepare(int *num_sms) {
  int dev = 0;
  MX_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return MX_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_smem_set[dev]) {
    MX_CUDA_TRY(cudaFuncSetAttribute(k_grouped_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC));
    MX_CUDA_TRY(cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev));
    g_smem_set[dev] = 1;
  }
  *num_sms = g_num_sms[dev];
  return MX_OK;
}

mx_status launch_1cta(const Params &p, const uint8_t *A, int64_t a_inner, int64_t a_outer, const uint8_t *B,
                      int64_t b_inner, int64_t b_outer, int64_t max_tiles, mx_stream stream) {
  int sms = 0;
  mx_status st = prepare(&sms);
  if (st != MX_OK) return st;
  CUtensorMap ma, mb;
  st = make_map_u8_128x128(&ma, A, a_inner, a_outer);
  if (st != MX_OK) return st;
  st = make_map_u8_128x128(&mb, B, b_inner, b_outer);
  if (st != MX_OK) return st;
  int64_t grid = max_tiles < sms ? max_tiles : sms;
  if (grid < 1) grid = 1;
  (void)launch_k(k_grouped_gemm, (unsigned)grid, NUM_THREADS, SMEM_ALLOC, stream, ma, mb, p);
  return launch_status();
}

// Which kernel runs: the CTA-pair kernel by default; MXMOE_GEMM_CTAS=1 selects
// the one-CTA kernel (both compute the same values).
static bool use_pair() {
  static int v = -1;
  if (v < 0) {
    const char *e = std::getenv("MXMOE_GEMM_CTAS");
    v = (e && e[0] == '1') ? 0 : 1;
  }
  return v == 1;
}

static mx_status dispatch(const Params &p, const uint8_t *A, int64_t a_inner, int64_t a_outer, const uint8_t *B,
                          int64_t b_inner, int64_t b_outer, int64_t tiles_1cta, int64_t sfa_bytes, int64_t sfb_bytes,
                          mx_stream stream) {
  const bool pair_ok = p.op == OP_ROWS || (p.N % 256 == 0);
  if (use_pair() && pair_ok) return launch_pair(p, A, a_inner, a_outer, B, b_inner, b_outer, sfa_bytes, sfb_bytes, stream);
  return launch_1cta(p, A, a_inner, a_outer, B, b_inner, b_outer, tiles_1cta, stream);
}

}  // namespace gemm
}  // namespace mxmoe

using namespace mxmoe;

extern "C" mx_status mx_grouped_gemm(int32_t op, const uint8_t *A, const uint8_t *sA, const uint8_t *B,
                                     const uint8_t *sB, const int32_t *offsets, int32_t E, int64_t M_cap, int64_t N,
                                     int64_t K, void *C, int32_t c_dtype, int32_t elem_a, int32_t elem_b,
                                     int32_t *dev_status, mx_stream stream) {
  MX_HOST_CHECK(op == MX_GEMM_FWD || op == MX_GEMM_DGRAD || op == MX_GEMM_WGRAD, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK((elem_a == MX_ELEM_E4M3 || elem_a == MX_ELEM_E5M2) && (elem_b == MX_ELEM_E4M3 || elem_b == MX_ELEM_E5M2),
                MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(A && sA && B && sB && offsets && C, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(c_dtype == MX_OUT_BF16 || c_dtype == MX_OUT_F32, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(E >= 1 && E <= gemm::MAX_E && M_cap >= 0 && N > 0 && K > 0, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(M_cap % 128 == 0 && N % 256 == 0 && K % 128 == 0, MX_ERR_SHAPE);
  MX_HOST_CHECK(M_cap < (int64_t)1 << 31 && N < (int64_t)1 << 31 && K < (int64_t)1 << 31, MX_ERR_SHAPE);
  MX_HOST_CHECK(aligned16(A) && aligned16(B) && aligned16(sA) && aligned16(sB) && aligned16(C), MX_ERR_ALIGNMENT);
  mx_status st = check_device_cached();
  if (st != MX_OK) return st;
  gemm::Params p;
  p.E = E;
  p.M_cap = M_cap;
  p.N = N;
  p.offsets = offsets;
  p.sA = sA;
  p.sB = sB;
  p.C = C;
  p.ab = nullptr;
  p.hq = nullptr;
  p.hs = nullptr;
  p.dev_status = dev_status;
  p.idesc_fmt = gemm::idesc_formats(elem_a == MX_ELEM_E5M2, elem_b == MX_ELEM_E5M2);
  p.epi = c_dtype == MX_OUT_F32 ? gemm::EPI_F32 : gemm::EPI_BF16;
  if (op == MX_GEMM_WGRAD) {
    MX_HOST_CHECK(N % 128 == 0 && K % 256 == 0, MX_ERR_SHAPE);
    p.op = gemm::OP_TOKENS;
    p.K = K;
    if (M_cap == 0) return cudaMemsetAsync(C, 0, (size_t)E * N * K * (c_dtype == MX_OUT_F32 ? 4 : 2), stream) ==
                                   cudaSuccess ? MX_OK : MX_ERR_CUDA;
    const int64_t tiles = (int64_t)E * (N / 128) * (K / 256);
    return gemm::dispatch(p, A, M_cap, N, B, M_cap, K, tiles, N * M_cap / 32, K * M_cap / 32, stream);
  }
  if (M_cap == 0) return MX_OK;
  p.op = gemm::OP_ROWS;
  p.K = K;
  const int64_t tiles = (M_cap / 128) * (N / 256);
  return gemm::dispatch(p, A, K, M_cap, B, K, (int64_t)E * N, tiles, M_cap * K / 32, (int64_t)E * N * K / 32, stream);
}

extern "C" mx_status moe_gemm1_swiglu(const uint8_t *A, const uint8_t *sA, const uint8_t *B, const uint8_t *sB,
                                      const int32_t *offsets, int32_t E, int64_t M_cap, int64_t F, int64_t H,
                                      void *ab, uint8_t *hq, uint8_t *hs, int32_t *dev_status, mx_stream stream) {
  MX_HOST_CHECK(A && sA && B && sB && offsets && ab && hq && hs, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(E >= 1 && E <= gemm::MAX_E && M_cap >= 0 && F > 0 && H > 0, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(M_cap % 128 == 0 && F % 128 == 0 && H % 128 == 0, MX_ERR_SHAPE);
  MX_HOST_CHECK(aligned16(A) && aligned16(B) && aligned16(sA) && aligned16(sB) && aligned16(ab) && aligned16(hq),
                MX_ERR_ALIGNMENT);
  mx_status st = check_device_cached();
  if (st != MX_OK) return st;
  if (M_cap == 0) return MX_OK;
  gemm::Params p;
  p.op = gemm::OP_ROWS;
  p.epi = gemm::EPI_GLU;
  p.E = E;
  p.M_cap = M_cap;
  p.N = F;
  p.K = H;
  p.offsets = offsets;
  p.sA = sA;
  p.sB = sB;
  p.C = nullptr;
  p.ab = static_cast<uint16_t *>(ab);
  p.hq = hq;
  p.hs = hs;
  p.dev_status = dev_status;
  p.idesc_fmt = gemm::idesc_formats(0, 0);
  const int64_t tiles = (M_cap / 128) * (F / 128);
  return gemm::dispatch(p, A, H, M_cap, B, H, (int64_t)E * 2 * F, tiles, M_cap * H / 32, (int64_t)E * 2 * F * H / 32,
                        stream);
}
