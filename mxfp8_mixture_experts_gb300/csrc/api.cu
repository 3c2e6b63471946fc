// Library-level entry points: status strings, ABI version, device check.
#include "common.cuh"

#include <cstdlib>

#include <mutex>

namespace mxmoe {

static std::mutex g_dev_mu;
static int g_dev_ok[64];  // 0 unknown, 1 ok, 2 unsupported

mx_status check_device_cached() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MX_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_dev_ok[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return MX_ERR_CUDA;
    // the binary carries sm_103a code only
    g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : 2;
  }
  return g_dev_ok[dev] == 1 ? MX_OK : MX_ERR_UNSUPPORTED_DEVICE;
}

mx_status launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

bool pdl_enabled() {
  static const bool on = [] {
    const char *v = std::getenv("MXMOE_PDL");
    return !(v && v[0] == '0');
  }();
  return on;
}

// One warp waits, with the kernels' own bounded warp-wide wait, on an mbarrier
// that nothing ever arrives on; when the limit passes it records
// MX_ERR_TIMEOUT and exits.  Nothing is in flight when it returns.
__global__ void k_selftest_wait_timeout(uint64_t timeout_ns, int32_t *dev_status) {
  pdl_enter();
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (!mbar_wait_warp(&bar, 0, timeout_ns) && threadIdx.x == 0) set_status(dev_status, MX_ERR_TIMEOUT);
}

// The SwiGLU kernels' sigmoid pieces (sigmoid_parts), evaluated on bf16 inputs:
// out[3i] = s, out[3i+1] = 1 - sigma, out[3i+2] = back (sigma = s * back).
__global__ void k_selftest_sigmoid(const uint16_t *__restrict__ a, int64_t n, float *__restrict__ out) {
  pdl_enter();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const SigParts p = sigmoid_parts(__uint_as_float((uint32_t)a[i] << 16));
    out[3 * i] = p.s;
    out[3 * i + 1] = p.oms;
    out[3 * i + 2] = p.back;
  }
}

}  // namespace mxmoe

extern "C" mx_status mx_selftest_sigmoid(const void *a, int64_t n, float *out, mx_stream stream) {
  MX_HOST_CHECK(n >= 0 && (n == 0 || (a && out)), MX_ERR_INVALID_ARG);
  mx_status st = mxmoe::check_device_cached();
  if (st != MX_OK) return st;
  if (n == 0) return MX_OK;
  const int64_t blocks = (n + 255) / 256;
  (void)mxmoe::launch_k(mxmoe::k_selftest_sigmoid, (unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, stream, 
      static_cast<const uint16_t *>(a), n, out);
  return mxmoe::launch_status();
}

extern "C" mx_status mx_selftest_wait_timeout(int64_t timeout_ns, int32_t *dev_status, mx_stream stream) {
  MX_HOST_CHECK(dev_status != nullptr, MX_ERR_INVALID_ARG);
  MX_HOST_CHECK(timeout_ns > 0 && timeout_ns <= 100000000, MX_ERR_INVALID_ARG);  // at most 100 ms
  mx_status st = mxmoe::check_device_cached();
  if (st != MX_OK) return st;
  (void)mxmoe::launch_k(mxmoe::k_selftest_wait_timeout, 1, 32, 0, stream, (uint64_t)timeout_ns, dev_status);
  return mxmoe::launch_status();
}

extern "C" const char *mx_status_string(mx_status s) {
  switch (s) {
    case MX_OK: return "MX_OK";
    case MX_ERR_INVALID_ARG: return "MX_ERR_INVALID_ARG: null pointer, unknown enum or negative size";
    case MX_ERR_SHAPE: return "MX_ERR_SHAPE: a dimension breaks the multiple-of-32/128/256 rule";
    case MX_ERR_ALIGNMENT:
      return "MX_ERR_ALIGNMENT: a device pointer breaks its alignment rule (16 bytes; 4 for word-written scales)";
    case MX_ERR_UNSUPPORTED_DEVICE: return "MX_ERR_UNSUPPORTED_DEVICE: the current device is not sm_103";
    case MX_ERR_CUDA: return "MX_ERR_CUDA: a CUDA call failed";
    case MX_ERR_DEVICE: return "MX_ERR_DEVICE: the device found an expert id out of range or bad group offsets";
    case MX_ERR_TIMEOUT: return "MX_ERR_TIMEOUT: a bounded pipeline wait expired on the device";
    case MX_ERR_WORKSPACE: return "MX_ERR_WORKSPACE: workspace smaller than the size query returned";
    case MX_ERR_SCRATCH_LIMIT:
      return "MX_ERR_SCRATCH_LIMIT: the problem needs more scratch than the allocation-free entry point's fixed array";
    default: return "unknown mx_status";
  }
}

extern "C" int32_t mx_abi_version(void) { return 4; }

extern "C" mx_status mx_check_device(void) { return mxmoe::check_device_cached(); }
