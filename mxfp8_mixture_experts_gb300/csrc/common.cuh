// Shared device/host helpers for libmxmoe: status plumbing, MXFP8 block
// encoding, and thin inline-PTX wrappers for mbarrier, TMA (cp.async.bulk*)
// and the tcgen05 tensor-core instructions of sm_100-family GPUs.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mxmoe.h"

#define MX_HOST_CHECK(cond, code) \
  do {                            \
    if (!(cond)) return (code);   \
  } while (0)

#define MX_CUDA_TRY(expr)                       \
  do {                                          \
    cudaError_t _e = (expr);                    \
    if (_e != cudaSuccess) return MX_ERR_CUDA;  \
  } while (0)

namespace mxmoe {

// ---------------------------------------------------------------------------
// host-side validation helpers
// ---------------------------------------------------------------------------
static inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

mx_status check_device_cached();  // defined in api.cu
mx_status launch_status();        // cudaGetLastError -> mx_status
bool pdl_enabled();               // defined in api.cu (MXMOE_PDL=0 at process start turns it off)

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialization and begins with pdl_enter(): the
// wait makes the previous grid of the stream complete, with its writes
// visible, before any thread of this grid touches global memory; the trigger
// then lets the next grid's CTAs be scheduled, which happens once every CTA
// of this grid has issued it (all of them resident), so the next grid's
// launch overlaps this grid's tail instead of following its completion.  A
// grid waiting in pdl_enter() never holds resources its predecessor still
// needs: the predecessor's CTAs were all resident before it was scheduled.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                            Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------------------
// device status word
// ---------------------------------------------------------------------------
__device__ __forceinline__ void set_status(int32_t *st, int32_t code) {
  if (st) atomicCAS(st, 0, code);
}

// ---------------------------------------------------------------------------
// MXFP8 block encoding (OCP MX v1.0 section 6.3 with E4M3 elements)
//
// The block scale exponent is floor(log2 amax) - 8.  For an fp32 amax that is
// its exponent field minus 127 minus 8; the scale byte (exponent + 127) is
// therefore exp_field - 8, clamped at 0 (the exponent's -127 floor, which also
// covers zero and fp32 subnormals).  The elements are cast from x * 2^-e with
// the hardware's round-to-nearest-even, saturating conversion.
// ---------------------------------------------------------------------------
struct MxScale {
  uint32_t byte;   // E8M0 scale byte (0xFF when the block holds NaN/Inf)
  float inv;       // 2^-e as fp32 (exact power of two)
  bool bad;        // block holds NaN or Inf
};

// amax_bits: max over the block of (float_bits & 0x7fffffff), compared as
// unsigned integers (NaN patterns compare above +Inf).  E5: E5M2 elements,
// whose largest power of two is 2^15 (the scale exponent is then
// floor(log2 amax) - 15); otherwise E4M3 (2^8).
template <bool E5>
__device__ __forceinline__ MxScale mx_scale_from_amax_bits_t(uint32_t amax_bits) {
  constexpr uint32_t EMAX = E5 ? 15u : 8u;
  MxScale s;
  uint32_t ef = amax_bits >> 23;            // biased exponent of amax
  s.bad = amax_bits >= 0x7f800000u;
  uint32_t b = ef >= EMAX ? ef - EMAX : 0u;  // = max(floor(log2 amax) - EMAX, -127) + 127
  s.byte = s.bad ? 0xffu : b;
  // 2^-e = 2^(127 - b): biased fp32 exponent 254 - b (b <= 246 for finite inputs)
  s.inv = __uint_as_float((254u - (s.bad ? 127u : b)) << 23);
  return s;
}
__device__ __forceinline__ MxScale mx_scale_from_amax_bits(uint32_t amax_bits) {
  return mx_scale_from_amax_bits_t<false>(amax_bits);
}

// two fp32 -> two E4M3 bytes (lo = first argument), RNE + saturate to +-448
__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// two fp32 -> two E5M2 bytes (lo = first argument), RNE + saturate to +-57344
__device__ __forceinline__ uint16_t cvt_e5m2x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
template <bool E5>
__device__ __forceinline__ uint16_t cvt_fp8x2(float lo, float hi) {
  return E5 ? cvt_e5m2x2(lo, hi) : cvt_e4m3x2(lo, hi);
}

// four fp32 already multiplied by the inverse scale -> packed 4 bytes
template <bool E5>
__device__ __forceinline__ uint32_t pack_fp8x4(float a, float b, float c, float d) {
  return (uint32_t)cvt_fp8x2<E5>(a, b) | ((uint32_t)cvt_fp8x2<E5>(c, d) << 16);
}
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  return pack_fp8x4<false>(a, b, c, d);
}

__device__ __forceinline__ uint32_t abs_bits(float v) { return __float_as_uint(v) & 0x7fffffffu; }

// 2^x on the hardware's approximate base-2 exponential (ex2.approx).
__device__ __forceinline__ float ex2_approx(float x) {
  float e;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(x));
  return e;
}

// 1/x on the hardware's approximate reciprocal (rcp.approx, within 1 ulp).
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// The sigmoid of a bf16 value a, in pieces that keep fp32 accuracy over the
// whole range the SwiGLU kernels see:
//   s    = sigma(a) * 2^k        (k = 64 when a < -64, else 0)
//   oms  = 1 - sigma(a)
//   back = 2^-k
// so silu(a) * b = ((a * s) * b) * back, with the multiply by `back` the only
// rounding that may enter the fp32 subnormal range.
//
// t = e^-|a| = 2^(-|a| log2 e).  log2 e is split as LOG2E_HI (16 significant
// bits) plus a remainder: a has 8 significant bits, so |a| * LOG2E_HI is
// exact in fp32 and the exponential's argument carries no rounding error (the
// constant-splitting of Cody and Waite, 1980).  The remainder enters as the
// factor e^-y with y = |a| (1 - LOG2E_HI ln 2), |y| < 1.3e-3, taken as
// 1 - y + y^2/2 (error below 4e-10).  Then sigma(a) = 1/(1+t) for a >= 0 and
// t/(1+t) for a < 0, and 1 - sigma(a) the other one: no cancellation on
// either side.  For a < -64 the exponential is taken 2^64 higher, which keeps
// t and s in the normal range down to a = -128 (1 + t is then 1 in fp32).
// |a| is capped at 256 (t is 0 beyond); NaN propagates through the caller's
// products with a.
constexpr float LOG2E_HI = 0x1.7154p+0f;          // 23637 / 16384
constexpr float LOG2E_REM_LN = 0x1.480fb6p-18f;   // 1 - LOG2E_HI * ln 2
struct SigParts {
  float s, oms, back;
};
__device__ __forceinline__ SigParts sigmoid_parts(float a) {
  const float aa = fminf(fabsf(a), 256.0f);
  const bool far = a < -64.0f;
  const float t0 = ex2_approx(fmaf(aa, -LOG2E_HI, far ? 64.0f : 0.0f));  // exact argument
  const float y = aa * LOG2E_REM_LN;
  const float t = t0 * fmaf(y, fmaf(0.5f, y, -1.0f), 1.0f);               // e^-|a| (* 2^64 if far)
  const float r = rcp_approx(far ? 1.0f : 1.0f + t);
  const float tr = t * r;
  SigParts p;
  p.s = a >= 0.0f ? r : tr;
  p.oms = a >= 0.0f ? tr : r;
  p.back = far ? 0x1p-64f : 1.0f;
  return p;
}

// Two-lane 16-bit integer max.  On bf16 pairs with the sign bits cleared
// (& 0x7fff7fff) it is the per-half |x| maximum, NaN and Inf patterns above
// every finite value, exactly as abs_bits on fp32.
__device__ __forceinline__ uint32_t vmax_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Four fp32 scaled by `inv` (an exact power of two: every product is exact
// or an IEEE round-to-nearest result, as with scalar multiplies) in two packed
// fp32x2 multiplies, then cast to E4M3 (E5: E5M2) and packed, first element
// lowest.
template <bool E5>
__device__ __forceinline__ uint32_t scale_pack_fp8x4(float a, float b, float c, float d, float inv) {
  uint64_t x, y, s2, r1, r2;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a), "f"(b));
  asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(c), "f"(d));
  asm("mov.b64 %0, {%1, %1};" : "=l"(s2) : "f"(inv));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r1) : "l"(x), "l"(s2));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r2) : "l"(y), "l"(s2));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r1));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(c), "=f"(d) : "l"(r2));
  return pack_fp8x4<E5>(a, b, c, d);
}
__device__ __forceinline__ uint32_t scale_pack_e4m3x4(float a, float b, float c, float d, float inv) {
  return scale_pack_fp8x4<false>(a, b, c, d, inv);
}

// bf16 helpers (storage as uint16)
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // RNE
  return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ float round_bf16(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// swizzled scale offset: tiles of 128 rows x 4 scale columns (512 B)
__host__ __device__ __forceinline__ int64_t sf_swizzle_offset(int64_t r, int64_t c, int64_t cols_p4) {
  return ((r >> 7) * (cols_p4 >> 2) + (c >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (c & 3);
}
__host__ __device__ __forceinline__ int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

// ---------------------------------------------------------------------------
// shared-memory addresses, fences
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// One try_wait: returns once the phase with `parity` has completed or after
// an implementation-defined time limit, whichever comes first.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
#ifdef MX_TRYWAIT_SUSPEND_NS
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"((uint32_t)MX_TRYWAIT_SUSPEND_NS)
      : "memory");
#else
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
#endif
  return ok != 0;
}

// Bounded wait: spins on try_wait (which itself suspends for a while per
// call) until the phase with `parity` completed or `timeout_ns` of global
// time passed.  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 256; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > timeout_ns) return false;
  }
}

// Warp-uniform bounded wait: every lane of the warp calls it and all get the
// same answer.  Single-thread roles (TMA issue, MMA issue) run their loops
// with the whole warp and let one elected lane issue: a loop whose waits run
// in one divergent lane stalls the tensor pipe between MMA batches.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity, uint64_t timeout_ns) {
  if (__any_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (__any_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    const int expired = (globaltimer_ns() - t0) > timeout_ns;
    if (__shfl_sync(0xffffffffu, expired, 0)) return false;
  }
}

// true in exactly one lane of the (fully active) warp
__device__ __forceinline__ bool elect_one_sync() {
  uint32_t pred = 0;
  asm volatile("{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}" : "=r"(pred));
  return pred != 0;
}

// ---------------------------------------------------------------------------
// clusters (CTA pairs)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t nclusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// shared::cluster address of the same shared-memory location in CTA `rank`
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// arrive on an mbarrier given by a shared::cluster address (any CTA of the cluster)
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Arrive with no memory ordering.  For a signal that only says "my reads of
// TMEM are done" after tcgen05.wait::ld: the values are already in registers,
// so nothing needs to become visible, and the cluster-scope release of the
// plain arrive (measured at ~2000 cycles per arrive on GB300) is avoided.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// TMA / bulk copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, uint64_t *bar, int32_t x,
                                            int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
      "[%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}
// CTA-pair form: the completion is signalled on `cluster_bar`, an mbarrier
// that may live in the peer CTA of the pair (the MMA-issuing CTA)
__device__ __forceinline__ void tma_load_2d_pair(void *smem_dst, const CUtensorMap *map, uint32_t cluster_bar,
                                                 int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(cluster_bar), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gmem_src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// shared -> global tensor store (2-D box), tracked with bulk async-groups
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *smem_src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(smem_src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until at most N of this thread's bulk groups still read shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_group_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores, tensor memory)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *smem_result, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_result)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *smem_result, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_result)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// pair forms of commit / copy / MMA, issued by one thread of the even CTA
__device__ __forceinline__ void tc_commit_pair(uint64_t *bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}
__device__ __forceinline__ void tc_cp_32x128b_warpx4_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void tc_mma_mxf8_pair(uint32_t d_taddr, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t sfa_taddr, uint32_t sfb_taddr, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_taddr),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_taddr), "r"(sfb_taddr)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// arrive on an mbarrier once all prior tcgen05 async ops of this thread finish
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// copy a 32-row x 128-bit smem block into TMEM lanes 0..31 (4 columns),
// replicated into the other three 32-lane quarters
__device__ __forceinline__ void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// D(tmem) (+)= A(smem) . B(smem)^T with per-32-K block scales from TMEM
__device__ __forceinline__ void tc_mma_mxf8(uint32_t d_taddr, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa_taddr, uint32_t sfb_taddr, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_taddr),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_taddr), "r"(sfb_taddr)
      : "memory");
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 columns of 32-bit: thread i gets lane (base lane + i), columns c..c+31
#define MX_TMEM_LD_32x32b_x32(taddr, r)                                                                       \
  asm volatile(                                                                                               \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17," \
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"                                      \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),       \
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), \
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),            \
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),            \
        "=r"(r[30]), "=r"(r[31])                                                                              \
      : "r"(taddr)                                                                                            \
      : "memory")

// Shared-memory matrix descriptor (tcgen05 "matrix descriptor"): start
// address, leading/stride byte offsets (16-byte units), descriptor version 1
// (bits 46..48 = 0b001), swizzle mode in bits 61..63 (0 none, 2 = 128-byte).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint32_t swizzle) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3ffffu) >> 4);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3fffu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3fffu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(swizzle & 7u) << 61;
  return d;
}

}  // namespace mxmoe
