// Host-side helpers of the C ABI: argument checks, CUDA error capture, device facts.
#pragma once

#include <cudaTypedefs.h>
#include <cuda_fp16.h>
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

// Hadamard block sizes the transform accepts (the pack's loader takes 512 .. 4096); 1024 is the
// pack's own and the one the fused kernels run, the others go through a separate transform
inline bool supported_block(int block) {
  return block == 512 || block == 1024 || block == 2048 || block == 4096;
}

// y = fwht(x) over blocks of `block` (a supported size; K a multiple of it); y may equal x
int launch_fwht(const __half* x, __half* y, const int8_t* signs, int64_t M, int64_t K, int block,
                int inverse, cudaStream_t s);

// cuTensorMapEncodeTiled, looked up once (thread-safe); null when the driver lacks it
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// streaming multiprocessors and opt-in shared memory of the current device
struct DeviceFacts {
  int device = -1;
  int sms = 0;
  int smem_optin = 0;
};
int device_facts(DeviceFacts* f);

// cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes), made only when
// bytes exceeds what was set before for this kernel on this device (a driver call per launch
// costs host time that a stream of small launches does not hide)
int ensure_dynamic_smem(const void* func, int device, int bytes);

}  // namespace tb
