// Device-side generator of the synthetic ternary codes and group scales.
//
// Same definition as tb_inputs/__init__.py (SplitMix64 counters, integer thresholds,
// correctly rounded fp32 steps without contraction), so a row drawn here equals the
// row the host draws for the same (seed, row, column).  It holds none of the layer's
// arithmetic: it only fills the int8 codes and fp16 scales the packer consumes.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define GAMMA 0x9E3779B97F4A7C15ull

__host__ __device__ static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static uint64_t stream_key(uint64_t seed, uint64_t stream) {
  const uint64_t base = seed * 2ull + stream;
  return mix64(base * GAMMA + GAMMA);
}

// codes for rows [row0, row0 + nrows) of an [N, K] matrix; 16 codes per thread
__global__ void fill_codes_kernel(int8_t* __restrict__ out, uint64_t key, int64_t row0, int64_t nrows,
                                  int64_t K) {
  const int64_t n16 = nrows * K / 16;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t base = row0 * K + i * 16;  // global counter of the first code
    uint32_t packed[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t v = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint64_t h = mix64(key + (uint64_t)(base + 4 * q + e + 1) * GAMMA);
        const uint32_t u = (uint32_t)(h >> 40);
        const int t = u < 6375342u ? -1 : (u < 10401874u ? 0 : 1);
        v |= ((uint32_t)(uint8_t)(int8_t)t) << (8 * e);
      }
      packed[q] = v;
    }
    reinterpret_cast<uint4*>(out)[i] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  }
}

__global__ void fill_scales_kernel(__half* __restrict__ out, uint64_t key, int64_t row0, int64_t nrows,
                                   int64_t G) {
  const int64_t n = nrows * G;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t h = mix64(key + (uint64_t)(row0 * G + i + 1) * GAMMA);
    const uint32_t u = (uint32_t)(h >> 40);
    float f = __fmul_rn((float)u, 1.0f / 16777216.0f);
    f = __fmul_rn(0.015f, f);
    f = __fadd_rn(0.005f, f);
    out[i] = __float2half_rn(f);
  }
}

extern "C" int tbs_fill_codes(int8_t* out, uint64_t seed, int64_t row0, int64_t nrows, int64_t K,
                              void* stream) {
  if (!out || nrows < 1 || K % 16) return -2;
  const int64_t n16 = nrows * K / 16;
  int64_t blocks = (n16 + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  fill_codes_kernel<<<(int)blocks, 256, 0, (cudaStream_t)stream>>>(out, stream_key(seed, 0), row0,
                                                                   nrows, K);
  return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

extern "C" int tbs_fill_scales(uint16_t* out, uint64_t seed, int64_t row0, int64_t nrows, int64_t G,
                               void* stream) {
  if (!out || nrows < 1 || G < 1) return -2;
  const int64_t n = nrows * G;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  fill_scales_kernel<<<(int)blocks, 256, 0, (cudaStream_t)stream>>>(
      reinterpret_cast<__half*>(out), stream_key(seed, 1), row0, nrows, G);
  return cudaGetLastError() == cudaSuccess ? 0 : -5;
}
