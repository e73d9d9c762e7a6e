// Status strings, CUDA error capture and per-device facts for the C ABI.
#include <cuda_runtime.h>
#include <stdio.h>
#include <string.h>

#include <map>
#include <mutex>

#include "tb_host.h"

namespace tb {

static thread_local char g_last_cuda_error[256] = "";

void record_cuda_error(cudaError_t e) {
  snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", cudaGetErrorName(e),
           cudaGetErrorString(e));
}

int ensure_dynamic_smem(const void* func, int device, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> set;
  std::lock_guard<std::mutex> lock(mu);
  int& have = set[{func, device}];
  if (have >= bytes) return TB_OK;
  const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return TB_ERR_CUDA;
  }
  have = bytes;
  return TB_OK;
}

int device_facts(DeviceFacts* f) {
  static std::mutex mu;
  static DeviceFacts cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    if (e != cudaSuccess) record_cuda_error(e);
    return TB_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev].device != dev) {
    DeviceFacts d;
    d.device = dev;
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      return TB_ERR_CUDA;
    }
    cache[dev] = d;
  }
  *f = cache[dev];
  return TB_OK;
}

}  // namespace tb

extern "C" const char* tb_status_string(int status) {
  switch (status) {
    case TB_OK: return "ok";
    case TB_ERR_NULL: return "a required pointer is NULL";
    case TB_ERR_SHAPE: return "shape out of range or not a required multiple";
    case TB_ERR_UNSUPPORTED: return "unsupported block size or algorithm";
    case TB_ERR_VALUE: return "invalid argument value";
    case TB_ERR_CUDA: return "CUDA error (see tb_last_cuda_error)";
    case TB_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case TB_ERR_WORKSPACE: return "workspace missing or too small";
    case TB_ERR_TOO_LARGE: return "problem exceeds the fixed scratch of the no-allocation entry point";
    default: return "unknown status";
  }
}

extern "C" const char* tb_last_cuda_error(void) { return tb::g_last_cuda_error; }

extern "C" int tb_version(void) { return 100; }
