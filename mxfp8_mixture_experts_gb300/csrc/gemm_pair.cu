// Block-scaled MXFP8 grouped GEMM, CTA-pair variant (tcgen05 cta_group::2).
//
// Same contraction as the one-CTA kernel in gemm.cu ("1.5x faster MoE
// training on Blackwell with MXFP8 kernels built from scratch", Key Questions
// Answered: block-scaled tcgen05.mma with TMEM accumulators), arranged for the
// bandwidth of one SM: two CTAs on neighbouring SMs form a cluster and compute
// one 256-row tile with M=256 MMAs.  Each CTA stages its own 128 rows of A and
// its own half of the B tile.
//
// One SM takes in 64 bytes of operands per MMA cycle (a 128 x 256 one-CTA
// tile needs 96), so the pair runs close to the tensor peak; with 6 operand
// stages in shared memory the loads run far enough ahead to cross tile
// boundaries without starving the MMA.  (Measured alternatives that lost:
// 256 x 128 tiles with two TMEM accumulators, which raise the L2-to-SM
// traffic per FLOP by half; direct global stores from registers; a second
// staging buffer per epilogue warp in place of the sixth stage.)
//
// Roles per CTA (320 threads): warp 0 loads (TMA, completion counted on the
// even CTA's barrier), warp 1 of the even CTA issues the scale copies, MMAs
// and commits for the pair, warps 2..9 drain the CTA's own 128-row slice of
// the accumulator (bf16/fp32 outputs leave through swizzled shared-memory
// staging and TMA tensor stores, so each global write is a full 64-byte row
// segment).  Row groups are 128-row aligned; a group with an odd number of
// 128-row tiles ends in a "lone" tile.  With bf16 or fp32 outputs the pair
// computes it transposed: the 256 weight rows of the column tile are the
// M=256 operand (each CTA its own 128, as the B half it loads for a full
// tile) and the lone tile's 128 rows are an N=128 operand (64 per CTA), so
// no product is computed twice; each CTA stores its 128 output columns, one
// per TMEM lane, as coalesced row segments.  In the SwiGLU epilogue the two
// halves of a feature pair would land in different CTAs, so there the pair
// computes the lone tile with both halves on the same rows and the even CTA
// stores it.
#include "gemm_shared.cuh"

#include <mutex>

namespace mxmoe {
namespace gemm {

constexpr int P_THREADS = 320;
constexpr uint32_t P_TMEM_COLS = 512;
constexpr int P_EPI_BUF = 2048;  // 32 rows x 64 bytes, 64-byte swizzle

struct PairCfg {
  static constexpr int TN = 256;                       // MMA N: tile columns
  static constexpr int STAGES = 6;
  static constexpr int EPI_BUFS = 1;                   // store staging buffers per epilogue warp
  static constexpr int A_TILE = 128 * BK;              // 16 KB: this CTA's 128 rows of A
  static constexpr int B_TILE = 128 * BK;              // 16 KB: this CTA's half of the B tile
  static constexpr int SF_STAGE = 3 * 512;             // own SFA chunk + both SFB chunks
  static constexpr uint32_t STAGE_TX = A_TILE + B_TILE + SF_STAGE;
  static constexpr uint32_t TR_STAGE_TX = A_TILE + B_TILE / 2 + 2 * 512;  // transposed lone tile
  static constexpr uint32_t ACC_COL = 0;               // accumulator: TMEM columns [0, 256)
  static constexpr uint32_t SF_COL = 256;              // scales: 12 columns per stage from here
  static constexpr uint32_t SF_COLS = 12;
  static constexpr int SMEM_A = 0;
  static constexpr int SMEM_B = SMEM_A + STAGES * A_TILE;
  static constexpr int SMEM_SF = SMEM_B + STAGES * B_TILE;
  static constexpr int SMEM_EPI = SMEM_SF + STAGES * SF_STAGE;
  static constexpr int SMEM_BAR = SMEM_EPI + NUM_EPI_WARPS * EPI_BUFS * P_EPI_BUF;
  static constexpr int SMEM_OFFS = SMEM_BAR + 256;
  static constexpr int SMEM_PP = SMEM_OFFS + (MAX_E + 1) * 4;
  static constexpr int SMEM_TOTAL = SMEM_PP + (MAX_E + 1) * 4;
  static constexpr int SMEM_ALLOC = SMEM_TOTAL + 1024;
  static_assert(SF_COL + STAGES * SF_COLS <= P_TMEM_COLS, "TMEM columns");
  static_assert((2 * STAGES + 2) * 8 + 8 <= 256, "barrier area");
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory");
};

struct PairTile {
  int64_t a_row;           // this CTA's A rows (TMA row coordinate)
  int64_t b_row;           // this CTA's rows of the B tile
  int64_t b_row0, b_row1;  // the two 128-row halves of the B tile (scale chunks)
  int64_t k0;
  int num_k;
  int64_t sfa_chunk, sfb_chunk0, sfb_chunk1;  // chunk index of the k=0 scales
  int64_t out_row, out_col;                   // this CTA's output rows / first column
  bool store;                                 // false: lone tile, odd CTA
  bool tr;                                    // transposed lone tile (see the header)
};

__device__ __forceinline__ int64_t pair_tiles(const Params &p, const int32_t *pp) {
  if (p.op == OP_ROWS) return (int64_t)pp[p.E] * (p.epi == EPI_GLU ? p.N / 128 : p.N / BN);
  return (int64_t)p.E * (p.N / 256) * (p.K / BN);
}

__device__ __forceinline__ PairTile decode_pair(const Params &p, const int32_t *off, const int32_t *pp, int64_t t,
                                                uint32_t rank) {
  PairTile tl;
  if (p.op == OP_ROWS) {
    const int64_t n_tiles = p.epi == EPI_GLU ? p.N / 128 : p.N / BN;
    // tiles of group e are [pp[e] * n_tiles, pp[e+1] * n_tiles)
    const int e = upper_group(pp, p.E, t / n_tiles);
    const int64_t local = t - (int64_t)pp[e] * n_tiles;
    const int64_t np_e = pp[e + 1] - pp[e];
    const int64_t n_e = (off[e + 1] - off[e]) / BM;
    const int64_t b_rows = p.epi == EPI_GLU ? 2 * p.N : p.N;
    // Raster within the group: when its rows are fewer than the weight rows,
    // walk the row pairs fastest so that each weight tile is read from HBM
    // once while the (smaller) activation slab stays in L2; otherwise walk
    // the column tiles fastest and keep each activation row pair in L2.
    const bool rows_fastest = n_e * BM < b_rows;
    const int64_t j = rows_fastest ? local % np_e : local / n_tiles;
    const int64_t nt = rows_fastest ? local / np_e : local % n_tiles;
    const int64_t mt0 = off[e] / BM + 2 * j;
    const bool lone = (2 * j + 1 == n_e);
    const int64_t my_mt = mt0 + (lone ? 0 : rank);
    const int64_t kblocks = p.K / BK;
    tl.a_row = my_mt * BM;
    if (p.epi == EPI_GLU) {
      // GEMM1: output features [nt*128, nt*128+128) need W1 rows (first F
      // rows of the expert's 2F) and the matching W3 rows (F further on)
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
    tl.tr = lone && p.epi != EPI_GLU;
    if (tl.tr) {
      // M side: this CTA's 128 weight rows; N side: 64 of the lone tile's 128
      // rows; the accumulator is [weight row, token row]
      tl.a_row = rank == 0 ? tl.b_row0 : tl.b_row1;
      tl.b_row = mt0 * BM + rank * 64;
      tl.sfa_chunk = (tl.a_row / 128) * kblocks;
      tl.sfb_chunk0 = tl.sfb_chunk1 = mt0 * kblocks;
      tl.out_row = mt0 * BM;
      tl.out_col += rank * 128;
      tl.store = true;
      return tl;
    }
    tl.sfa_chunk = my_mt * kblocks;
    tl.sfb_chunk0 = (tl.b_row0 / 128) * kblocks;
    tl.sfb_chunk1 = (tl.b_row1 / 128) * kblocks;
    tl.out_row = (mt0 + rank) * BM;
    tl.store = !(lone && rank == 1);
  } else {
    // token-grouped (wgrad): output [e*N + 256-row tile, 256-column tile],
    // contraction over the group's tokens [off[e], off[e+1])
    const int64_t rt_n = p.N / 256, ct_n = p.K / BN;
    const int64_t per_e = rt_n * ct_n;
    const int e = (int)(t / per_e);
    const int64_t rem = t % per_e;
    // The group's A slab is N x tokens, its B slab K x tokens: walk the tiles
    // of the smaller slab fastest, so it is the one re-read from L2 and the
    // larger one streams from HBM once.
    const bool rows_fastest = p.N <= p.K;
    const int64_t rt = rows_fastest ? rem % rt_n : rem / ct_n;
    const int64_t ct = rows_fastest ? rem / rt_n : rem % ct_n;
    const int64_t kblocks = p.M_cap / BK;
    const int64_t kc0 = off[e] / BK;
    tl.a_row = rt * 256 + rank * 128;
    tl.b_row0 = ct * BN;
    tl.b_row1 = tl.b_row0 + 128;
    tl.k0 = off[e];
    tl.num_k = (off[e + 1] - off[e]) / BK;
    tl.sfa_chunk = (tl.a_row / 128) * kblocks + kc0;
    tl.sfb_chunk0 = (tl.b_row0 / 128) * kblocks + kc0;
    tl.sfb_chunk1 = (tl.b_row1 / 128) * kblocks + kc0;
    tl.out_row = (int64_t)e * p.N + rt * 256 + rank * 128;
    tl.out_col = ct * BN;
    tl.store = true;
    tl.tr = false;
  }
  tl.b_row = rank == 0 ? tl.b_row0 : tl.b_row1;
  return tl;
}

// One warp's 32 rows x 64 bytes: wait until the store that last used `buf`
// has read it (at most NBUF - 1 newer stores pending), write the rows (16-byte
// chunk j of row i at chunk j ^ ((i>>1)&3), the 64-byte swizzle of the store
// map), then one lane issues the TMA store.
template <int NBUF>
__device__ __forceinline__ void stage_and_store(const CUtensorMap *map, uint8_t *buf, const uint4 (&v)[4], int lane,
                                                int x, int y) {
  if (lane == 0) bulk_wait_group_read<NBUF - 1>();
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint4 *>(buf + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) = v[j];
  fence_proxy_async();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, buf, x, y);
    bulk_commit_group();
  }
}

// SwiGLU epilogue of GEMM1 for one thread's row: r[0..63] = a, r[64..127] =
// b for features [f0, f0 + 64).  a and b are rounded to bf16 and saved; h =
// silu(a) * b in fp32 is quantized in two 32-element blocks.  The warp's 32
// rows leave as five 64-byte-wide TMA stores (two of a, two of b, one of h);
// the two scale bytes of the row are stored directly.
template <int NBUF>
__device__ __forceinline__ void glu_epilogue(const Params &p, const CUtensorMap *tmAB, const CUtensorMap *tmH,
                                             uint8_t *ebuf, int &nstore, int lane, int64_t orow, int y, int f0,
                                             const uint32_t (&r)[128]) {
  const int64_t F = p.N;
  uint4 hv4[4];
#pragma unroll
  for (int blk = 0; blk < 2; ++blk) {
    float hv[32];
    uint32_t am = 0;
    uint4 va[4], vb[4];
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
      va[j / 8] = make_uint4(pack_bf16x2(av[0], av[1]), pack_bf16x2(av[2], av[3]), pack_bf16x2(av[4], av[5]),
                             pack_bf16x2(av[6], av[7]));
      vb[j / 8] = make_uint4(pack_bf16x2(bv[0], bv[1]), pack_bf16x2(bv[2], bv[3]), pack_bf16x2(bv[4], bv[5]),
                             pack_bf16x2(bv[6], bv[7]));
    }
    stage_and_store<NBUF>(tmAB, ebuf + (nstore++ % NBUF) * P_EPI_BUF, va, lane, f0 + blk * 32, y);
    stage_and_store<NBUF>(tmAB, ebuf + (nstore++ % NBUF) * P_EPI_BUF, vb, lane, (int)F + f0 + blk * 32, y);
    const MxScale s = mx_scale_from_amax_bits(am);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      w[i] = s.bad ? 0x7f7f7f7fu
                   : pack_e4m3x4(hv[4 * i] * s.inv, hv[4 * i + 1] * s.inv, hv[4 * i + 2] * s.inv,
                                 hv[4 * i + 3] * s.inv);
    hv4[blk * 2] = make_uint4(w[0], w[1], w[2], w[3]);
    hv4[blk * 2 + 1] = make_uint4(w[4], w[5], w[6], w[7]);
    p.hs[sf_swizzle_offset(orow, f0 / 32 + blk, round_up(F / 32, 4))] = (uint8_t)s.byte;
  }
  stage_and_store<NBUF>(tmH, ebuf + (nstore++ % NBUF) * P_EPI_BUF, hv4, lane, f0, y);
}

__global__ void __launch_bounds__(P_THREADS, 1)
    k_grouped_gemm_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                        const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmH,
                        const __grid_constant__ CUtensorMap tmA64, Params p) {
  pdl_enter();
  using C = PairCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::SMEM_BAR);
  uint64_t *empty = full + C::STAGES;
  uint64_t *tmem_full = empty + C::STAGES;
  uint64_t *tmem_empty = tmem_full + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tmem_empty + 1);
  int32_t *s_flag = reinterpret_cast<int32_t *>(tmem_slot + 1);
  int32_t *s_off = reinterpret_cast<int32_t *>(smem + C::SMEM_OFFS);
  int32_t *s_pp = reinterpret_cast<int32_t *>(smem + C::SMEM_PP);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int64_t cid = cluster_id_x(), ncl = nclusters_x();

  for (int i = threadIdx.x; i <= p.E; i += P_THREADS) s_off[i] = p.offsets[i];
  __syncthreads();
  if (threadIdx.x == 0) {
    const int ok = offsets_ok(s_off, p.E, p.M_cap);
    *s_flag = ok;
    if (!ok && blockIdx.x == 0) set_status(p.dev_status, MX_ERR_DEVICE);
    // pairs of 128-row tiles per group (a trailing odd tile is a lone pair)
    int32_t run = 0;
    for (int e = 0; e < p.E; ++e) {
      s_pp[e] = run;
      run += ok ? ((s_off[e + 1] - s_off[e]) / BM + 1) / 2 : 0;
    }
    s_pp[p.E] = run;
  }
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tmem_full, 1);
    mbar_init(tmem_empty, 2 * NUM_EPI_WARPS);
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmSFA);
    prefetch_tmap(&tmSFB);
    prefetch_tmap(&tmC);
    if (p.epi == EPI_GLU) prefetch_tmap(&tmH);
    else prefetch_tmap(&tmA64);
  }
  __syncthreads();
  if (!*s_flag) return;  // identical decision in both CTAs of the pair
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, P_TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised, TMEM allocated in both
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int64_t ntiles = pair_tiles(p, s_pp);

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    // the whole warp runs the loop; one elected lane issues the copies
    {
      const uint32_t leader_full0 = mapa_shared(smem_u32(&full[0]), 0);
      int stage = 0;
      uint32_t phase = 0;
      bool dead = false;
      for (int64_t t = cid; t < ntiles && !dead; t += ncl) {
        const PairTile tl = decode_pair(p, s_off, s_pp, t, rank);
        for (int kb = 0; kb < tl.num_k; ++kb) {
          if (!mbar_wait_warp(&empty[stage], phase ^ 1, WAIT_TIMEOUT_NS)) {
            if (lane == 0) set_status(p.dev_status, MX_ERR_TIMEOUT);
            dead = true;
            break;
          }
          if (elect_one_sync()) {
            if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * (tl.tr ? C::TR_STAGE_TX : C::STAGE_TX));
            const uint32_t bar = leader_full0 + stage * 8;
            uint8_t *sa = smem + C::SMEM_A + stage * C::A_TILE;
            uint8_t *sb = smem + C::SMEM_B + stage * C::B_TILE;
            uint8_t *sf = smem + C::SMEM_SF + stage * C::SF_STAGE;
            const int32_t kc = (int32_t)(tl.k0 + (int64_t)kb * BK);
            if (tl.tr) {
              // weights as the M operand, 64 token rows as this CTA's N half
              tma_load_2d_pair(sa, &tmB, bar, kc, (int32_t)tl.a_row);
              tma_load_2d_pair(sb, &tmA64, bar, kc, (int32_t)tl.b_row);
              tma_load_2d_pair(sf, &tmSFB, bar, 0, (int32_t)(tl.sfa_chunk + kb));
              tma_load_2d_pair(sf + 512, &tmSFA, bar, 0, (int32_t)(tl.sfb_chunk0 + kb));
            } else {
              tma_load_2d_pair(sa, &tmA, bar, kc, (int32_t)tl.a_row);
              tma_load_2d_pair(sb, &tmB, bar, kc, (int32_t)tl.b_row);
              tma_load_2d_pair(sf, &tmSFA, bar, 0, (int32_t)(tl.sfa_chunk + kb));
              tma_load_2d_pair(sf + 512, &tmSFB, bar, 0, (int32_t)(tl.sfb_chunk0 + kb));
              tma_load_2d_pair(sf + 1024, &tmSFB, bar, 0, (int32_t)(tl.sfb_chunk1 + kb));
            }
          }
          __syncwarp();
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    // the whole warp runs the loop and waits; one elected lane issues
    if (rank == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool dead = false;
      const uint32_t idesc_full = idesc_mxf8(2 * BM, C::TN) | p.idesc_fmt;
      // transposed lone tile: N = 128, and the operands' formats trade places
      const uint32_t idesc_tr = idesc_mxf8(2 * BM, 128) | (((p.idesc_fmt >> 7) & 7u) << 10) |
                                (((p.idesc_fmt >> 10) & 7u) << 7);
      const uint32_t d_tmem = tmem_base + C::ACC_COL;
      for (int64_t t = cid; t < ntiles && !dead; t += ncl) {
        const PairTile tl = decode_pair(p, s_off, s_pp, t, rank);
        if (tl.num_k == 0) continue;
        const uint32_t idesc = tl.tr ? idesc_tr : idesc_full;
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
            const uint32_t sa = smem_u32(smem + C::SMEM_A + stage * C::A_TILE);
            const uint32_t sb = smem_u32(smem + C::SMEM_B + stage * C::B_TILE);
            const uint32_t sf = smem_u32(smem + C::SMEM_SF + stage * C::SF_STAGE);
            const uint32_t sfa_t = tmem_base + C::SF_COL + stage * C::SF_COLS;
            const uint32_t sfb_t = sfa_t + 4;
            // scales of this stage -> TMEM (in tensor-pipe order before the MMAs that read them)
            tc_cp_32x128b_warpx4_pair(sfa_t, smem_desc(sf, 0, 128, 0));
            tc_cp_32x128b_warpx4_pair(sfb_t, smem_desc(sf + 512, 0, 128, 0));
            if (!tl.tr) tc_cp_32x128b_warpx4_pair(sfb_t + 4, smem_desc(sf + 1024, 0, 128, 0));
#pragma unroll
            for (int kk = 0; kk < BK / 32; ++kk) {
              const uint64_t ad = smem_desc(sa + kk * 32, 16, 1024, 2);
              const uint64_t bd = smem_desc(sb + kk * 32, 16, 1024, 2);
              const uint32_t id = idesc | ((uint32_t)kk << 4) | ((uint32_t)kk << 29);
              tc_mma_mxf8_pair(d_tmem, ad, bd, id, sfa_t, sfb_t, (kb | kk) != 0);
            }
            tc_commit_pair(&empty[stage], 0x3);
          }
          __syncwarp();
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (dead) break;
        if (elect_one_sync()) tc_commit_pair(tmem_full, 0x3);
        __syncwarp();
        acc_phase ^= 1;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    // warp w drains TMEM lanes 32*(w%4).. (its sub-partition) and one half of
    // the accumulator's columns
    constexpr int EC = C::TN / 2;  // columns per epilogue warp
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const int row_in_tile = q * 32 + lane;
    const uint32_t leader_tmem_empty = mapa_shared(smem_u32(tmem_empty), 0);
    uint8_t *ebuf = smem + C::SMEM_EPI + (warp - 2) * C::EPI_BUFS * P_EPI_BUF;
    int nstore = 0;
    uint32_t acc_phase = 0;
    for (int64_t t = cid; t < ntiles; t += ncl) {
      const PairTile tl = decode_pair(p, s_off, s_pp, t, rank);
      const int64_t orow = tl.out_row + row_in_tile;
      if (tl.num_k == 0) {
        epi_zero(p, orow, tl.out_col + h * EC, EC);
        continue;
      }
      if (!mbar_wait_warp(tmem_full, acc_phase, WAIT_TIMEOUT_NS)) {
        if (lane == 0) set_status(p.dev_status, MX_ERR_TIMEOUT);
        break;
      }
      tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + C::ACC_COL;
      uint32_t r[EC];
      if (tl.tr) {
        // transposed lone tile: lane = output column out_col + q*32 + lane,
        // accumulator columns [h*64, h*64 + 64) = token rows out_row + h*64 + j
        MX_TMEM_LD_32x32b_x32(t_row + h * 64, r);
        MX_TMEM_LD_32x32b_x32(t_row + h * 64 + 32, (r + 32));
        tc_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(leader_tmem_empty);
        acc_phase ^= 1;
        const int64_t row0 = tl.out_row + h * 64;
        const int64_t col = tl.out_col + q * 32 + lane;
        if (p.epi == EPI_F32) {
          float *c = static_cast<float *>(p.C) + row0 * p.N + col;
#pragma unroll
          for (int j = 0; j < 64; ++j) c[j * p.N] = __uint_as_float(r[j]);
        } else {
          uint16_t *c = static_cast<uint16_t *>(p.C) + row0 * p.N + col;
#pragma unroll
          for (int j = 0; j < 64; ++j) c[j * p.N] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[j])));
        }
        continue;
      }
      if (p.epi == EPI_GLU) {
        // GEMM1: columns [0,128) hold a, [128,256) the matching b
        MX_TMEM_LD_32x32b_x32(t_row + h * 64, r);
        MX_TMEM_LD_32x32b_x32(t_row + h * 64 + 32, (r + 32));
        MX_TMEM_LD_32x32b_x32(t_row + 128 + h * 64, (r + 64));
        MX_TMEM_LD_32x32b_x32(t_row + 128 + h * 64 + 32, (r + 96));
      } else {
#pragma unroll
        for (int c = 0; c < EC / 32; ++c) MX_TMEM_LD_32x32b_x32(t_row + h * EC + c * 32, (r + c * 32));
      }
      tc_wait_ld();  // the accumulator is in registers: the MMA may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(leader_tmem_empty);
      acc_phase ^= 1;
      if (!tl.store) continue;
      const int y = (int)(tl.out_row + q * 32);
      if (p.epi == EPI_GLU) {
        glu_epilogue<C::EPI_BUFS>(p, &tmC, &tmH, ebuf, nstore, lane, orow, y, (int)(tl.out_col + h * 64), r);
        continue;
      }
      // 64-byte row segments: fp32 16 columns, bf16 32 columns per chunk
      const int x0 = (int)(tl.out_col + h * EC);
      if (p.epi == EPI_F32) {
#pragma unroll
        for (int c = 0; c < EC / 16; ++c) {
          uint4 v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j)
            v[j] = make_uint4(r[c * 16 + 4 * j], r[c * 16 + 4 * j + 1], r[c * 16 + 4 * j + 2], r[c * 16 + 4 * j + 3]);
          stage_and_store<C::EPI_BUFS>(&tmC, ebuf + (nstore % C::EPI_BUFS) * P_EPI_BUF, v, lane, x0 + c * 16, y);
          ++nstore;
        }
      } else {
#pragma unroll
        for (int c = 0; c < EC / 32; ++c) {
          uint4 v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t *w = r + c * 32 + 8 * j;
            v[j] = make_uint4(pack_bf16x2(__uint_as_float(w[0]), __uint_as_float(w[1])),
                              pack_bf16x2(__uint_as_float(w[2]), __uint_as_float(w[3])),
                              pack_bf16x2(__uint_as_float(w[4]), __uint_as_float(w[5])),
                              pack_bf16x2(__uint_as_float(w[6]), __uint_as_float(w[7])));
          }
          stage_and_store<C::EPI_BUFS>(&tmC, ebuf + (nstore % C::EPI_BUFS) * P_EPI_BUF, v, lane, x0 + c * 32, y);
          ++nstore;
        }
      }
    }
    if (lane == 0) bulk_wait_group_all();
    __syncwarp();
  }

  __syncwarp();
  tc_fence_before();
  cluster_sync();  // no MMA reads this CTA's shared memory or TMEM after this point
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, P_TMEM_COLS);
  }
}

static std::mutex g_pmu;
static int g_psmem_set[64];
static int g_pclusters[64];

// attr: room for two attributes (the CTA pair, and programmatic dependent
// launch as for every kernel of the library, see pdl_enter)
static void pair_config(cudaLaunchConfig_t *cfg, cudaLaunchAttribute *attr, int grid, mx_stream stream) {
  *cfg = cudaLaunchConfig_t{};
  cfg->gridDim = dim3(grid, 1, 1);
  cfg->blockDim = dim3(P_THREADS, 1, 1);
  cfg->dynamicSmemBytes = PairCfg::SMEM_ALLOC;
  cfg->stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg->attrs = attr;
  cfg->numAttrs = pdl_enabled() ? 2 : 1;
}

mx_status launch_pair(const Params &p, const uint8_t *A, int64_t a_inner, int64_t a_outer, const uint8_t *B,
                      int64_t b_inner, int64_t b_outer, int64_t sfa_bytes, int64_t sfb_bytes, mx_stream stream) {
  int dev = 0;
  MX_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return MX_ERR_CUDA;
  int clusters = 0;
  {
    // the persistent grid is as many CTA pairs as can be resident at once
    std::lock_guard<std::mutex> lk(g_pmu);
    if (!g_psmem_set[dev]) {
      MX_CUDA_TRY(cudaFuncSetAttribute(k_grouped_gemm_pair, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       PairCfg::SMEM_ALLOC));
      int sms = 0;
      MX_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
      cudaLaunchConfig_t cfg;
      cudaLaunchAttribute attr[2];
      pair_config(&cfg, attr, (sms / 2) * 2, nullptr);
      cfg.numAttrs = 1;  // the occupancy query needs the cluster shape only
      int n = 0;
      MX_CUDA_TRY(cudaOccupancyMaxActiveClusters(&n, k_grouped_gemm_pair, &cfg));
      if (n < 1) return MX_ERR_CUDA;
      g_pclusters[dev] = n < sms / 2 ? n : sms / 2;
      g_psmem_set[dev] = 1;
    }
    clusters = g_pclusters[dev];
  }
  CUtensorMap ma, mb, msa, msb, mc, mh, ma64;
  mx_status st = make_map_u8_128x128(&ma, A, a_inner, a_outer);
  if (st == MX_OK) st = make_map_u8_box_swz(&ma64, A, a_inner, a_outer, 64, (int)CU_TENSOR_MAP_SWIZZLE_128B);
  if (st == MX_OK) st = make_map_u8_128x128(&mb, B, b_inner, b_outer);
  if (st == MX_OK) st = make_map_sf_chunks(&msa, p.sA, sfa_bytes / 512);
  if (st == MX_OK) st = make_map_sf_chunks(&msb, p.sB, sfb_bytes / 512);
  if (st == MX_OK && p.epi != EPI_GLU) {
    const int64_t rows = p.op == OP_ROWS ? p.M_cap : (int64_t)p.E * p.N;
    const int64_t ldc = p.op == OP_ROWS ? p.N : p.K;
    st = make_map_store_64b(&mc, p.C, p.epi == EPI_F32, ldc, rows);
    mh = mc;  // unused outside the SwiGLU epilogue
  } else if (st == MX_OK) {
    // SwiGLU: a|b bf16 [M_cap, 2F] and h E4M3 [M_cap, F]
    st = make_map_store_64b(&mc, p.ab, false, 2 * p.N, p.M_cap);
    if (st == MX_OK) st = make_map_store_64b_u8(&mh, p.hq, p.N, p.M_cap);
  }
  if (st != MX_OK) return st;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  pair_config(&cfg, attr, 2 * clusters, stream);
  MX_CUDA_TRY(cudaLaunchKernelEx(&cfg, k_grouped_gemm_pair, ma, mb, msa, msb, mc, mh, ma64, p));
  return launch_status();
}

}  // namespace gemm
}  // namespace mxmoe
