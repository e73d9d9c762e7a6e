// Host-side helpers of the C ABI: argument checks, CUDA error capture, device facts.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/tb.h"

namespace tb {

// remember the text of a CUDA error for tb_last_cuda_error()
void record_cuda_error(cudaError_t e);

inline int check_launch() {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return TB_ERR_CUDA;
  }
  return TB_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// streaming multiprocessors and opt-in shared memory of the current device
struct DeviceFacts {
  int device = -1;
  int sms = 0;
  int smem_optin = 0;
};
int device_facts(DeviceFacts* f);

}  // namespace tb
