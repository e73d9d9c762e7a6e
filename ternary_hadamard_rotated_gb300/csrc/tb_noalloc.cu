// Decode GEMV entry point that allocates nothing.
//
// Some callers cannot hand this library a workspace: code that runs while a CUDA graph
// is being captured (where cudaMalloc is not allowed), plugins living inside a host
// runtime that owns every byte of device memory through its own pool, or services that
// forbid any allocation after start-up so their memory footprint stays fixed.  For them,
// tb_packed_linear_gemv_noalloc runs the same decode GEMV as tb_packed_linear (M <= 8),
// with the state of its split schedule (counters and fp32 parts of output tiles shared by
// several SMs) kept in a fixed array compiled into this library instead of a caller's
// workspace.  Every GPU that loads the library holds that array (about 2 MiB) until the
// process exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "tb_common.cuh"
#include "tb_host.h"

namespace tb {

int launch_gemv_tma(const __half* x, int64_t M, int64_t K, const int8_t* signs, int block,
                    const uint32_t* w, const __half* scales, const __half* biases, int64_t N,
                    __half* y, void* workspace, size_t ws_bytes, int32_t* status, cudaStream_t s);
size_t gemv_fixup_bytes();
size_t gemv_fixup_counter_bytes();

// split-schedule state for up to 256 SMs: counters (1 KiB) + fp32 parts [256][2][128 rows][8 tokens]
constexpr size_t kStaticScratchBytes = 1024 + (size_t)256 * 2 * 128 * 8 * 4;
constexpr int64_t kNoallocMaxTokens = 8;

}  // namespace tb

// A host-side name of device memory: host code must not pass it to a kernel directly (its
// address is obtained per device with cudaGetSymbolAddress below).
static __device__ __align__(256) unsigned char g_tb_gemv_scratch[tb::kStaticScratchBytes];

namespace tb {

// The driver's cuCtxGetCurrent, resolved once through the runtime (the library does not link
// libcuda itself); null if the driver does not offer it.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
static CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of g_tb_gemv_scratch on the current device.  It is looked up once per device
// and context: a context created after a reset (cudaDeviceReset, or the primary context torn
// down and made again) loads the module anew, so the address is looked up again when the
// current context is not the one it was found under.  (Without the driver's cuCtxGetCurrent
// it is looked up on every call.)
static int static_scratch(void** out) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  static CUcontext under[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    if (e != cudaSuccess) record_cuda_error(e);
    return TB_ERR_CUDA;
  }
  CtxGetCurrentFn get = ctx_get_current();
  CUcontext ctx = nullptr;
  if (get && get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (ctx && addr[dev] && under[dev] == ctx) {
    *out = addr[dev];
    return TB_OK;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_tb_gemv_scratch);  // binds the device's context if none is
  if (e != cudaSuccess || !p) {
    if (e != cudaSuccess) record_cuda_error(e);
    return TB_ERR_CUDA;
  }
  if (get && get(&ctx) == CUDA_SUCCESS && ctx) {
    addr[dev] = p;
    under[dev] = ctx;
  }
  *out = p;
  return TB_OK;
}

}  // namespace tb

extern "C" int tb_packed_linear_gemv_noalloc(const uint16_t* x, int64_t M, int64_t K,
                                             const int8_t* signs, int block, const uint32_t* w,
                                             const uint16_t* scales, const uint16_t* biases,
                                             int64_t N, uint16_t* y, int32_t* dev_status,
                                             void* stream) {
  using namespace tb;
  if (!x || !w || !scales || !y) return TB_ERR_NULL;  // biases may be NULL: each is -scale
  if (block != 0 && block != kBlock) return TB_ERR_UNSUPPORTED;
  if (M < 1 || N < 1 || K < kBlock || K % kBlock) return TB_ERR_SHAPE;
  if (M > kNoallocMaxTokens) return TB_ERR_TOO_LARGE;
  if (!aligned16(x) || !aligned16(w) || !aligned16(scales) || (biases && !aligned16(biases)) ||
      !aligned16(y) || (signs && !aligned16(signs)))
    return TB_ERR_ALIGN;
  DeviceFacts f;
  int rc = device_facts(&f);
  if (rc != TB_OK) return rc;
  if (f.sms > 256 || gemv_fixup_bytes() > kStaticScratchBytes) return TB_ERR_TOO_LARGE;
  void* scratch = nullptr;
  rc = static_scratch(&scratch);
  if (rc != TB_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the array keeps whatever the previous call left: its counters must start at zero (the
  // parts behind them are written before they are read)
  cudaError_t e = cudaMemsetAsync(scratch, 0, gemv_fixup_counter_bytes(), s);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return TB_ERR_CUDA;
  }
  return launch_gemv_tma(reinterpret_cast<const __half*>(x), M, K, block ? signs : nullptr, block, w,
                         reinterpret_cast<const __half*>(scales), reinterpret_cast<const __half*>(biases),
                         N, reinterpret_cast<__half*>(y), scratch, kStaticScratchBytes, dev_status, s);
}
