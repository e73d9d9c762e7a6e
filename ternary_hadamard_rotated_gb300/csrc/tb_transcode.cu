// Lossless transcoding of the GGUF block formats of the same trits into the W2-g128 container.
//
// [ARCH] kwkr.cn/news/564617, section "打包格式的工程MLX 2.25 bits 与 GGUF 的两种装箱": PQ2_0 keeps
// each trit in a 2-bit slot (34 bytes per 128 weights), PTQ1_0 packs the trits densely (28 bytes);
// the transcoder takes the scale from the block header, sets the bias to its negation and
// rearranges the codes into uint32 words.  The byte layout inside a block is not on the page;
// the reading used: the fp16 scale first; PQ2_0 slot i at bits 2(i % 4) of byte 2 + i/4 with
// q = t + 1; PTQ1_0 byte 2 + j = sum_i (t[5j+i] + 1) 3^i over the trits 5j .. 5j+4 below 128.
//
// One thread per block (128 weights): the block's bytes in, eight uint32 words, the scale and
// the bias out.  Memory-bound: 34 or 28 bytes read and 36 written per 128 weights.
#include <cuda_runtime.h>

#include "tb_common.cuh"
#include "tb_host.h"

namespace tb {

constexpr int kPq2Bytes = 34;
constexpr int kPtq1Bytes = 28;

// PQ2_0: with the slot order above, the 32 code bytes are the little-endian bytes of the eight
// W2 words; a slot holding 3 (both bits set) is not a trit
__global__ void __launch_bounds__(256) transcode_pq2_0_kernel(const uint16_t* __restrict__ blk,
                                                             int64_t n_blocks, uint32_t* __restrict__ w,
                                                             uint16_t* __restrict__ scales,
                                                             uint16_t* __restrict__ biases,
                                                             int32_t* __restrict__ status) {
  bool bad = false;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_blocks;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint16_t* p = blk + i * (kPq2Bytes / 2);  // 2-byte aligned: 34 = 2 * 17
    uint16_t h[17];
#pragma unroll
    for (int k = 0; k < 17; ++k) h[k] = __ldg(p + k);
    uint32_t wd[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      wd[k] = (uint32_t)h[1 + 2 * k] | ((uint32_t)h[2 + 2 * k] << 16);
      bad |= (wd[k] & (wd[k] >> 1) & 0x55555555u) != 0;
    }
    uint4* dst = reinterpret_cast<uint4*>(w + i * 8);
    dst[0] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
    dst[1] = make_uint4(wd[4], wd[5], wd[6], wd[7]);
    scales[i] = h[0];
    if (biases) biases[i] = h[0] ^ 0x8000u;
  }
  if (bad) set_status(status, TB_DEV_BAD_CODE);
}

// PTQ1_0: five base-3 digits per byte (first trit least significant).  A table in shared memory
// maps each byte to its five codes q = t + 1 as ten bits, two per trit (bit 31 set for a byte of
// 243 or more); the ten bits go to code positions 5j .. 5j+4 of the block's eight words, which
// for some j straddle two words.  A digit past trit 127 (the last byte above 26) is invalid.
__global__ void __launch_bounds__(256) transcode_ptq1_0_kernel(const uint32_t* __restrict__ blk,
                                                              int64_t n_blocks, uint32_t* __restrict__ w,
                                                              uint16_t* __restrict__ scales,
                                                              uint16_t* __restrict__ biases,
                                                              int32_t* __restrict__ status) {
  __shared__ uint32_t lut[256];
  {
    uint32_t v = threadIdx.x, e = 0;
#pragma unroll
    for (int d = 0; d < 5; ++d) {
      const uint32_t v3 = (v * 171u) >> 9;  // v / 3 for v < 256
      e |= (v - 3u * v3) << (2 * d);
      v = v3;
    }
    lut[threadIdx.x] = threadIdx.x >= 243 ? 0x80000000u : e;
  }
  __syncthreads();
  bool bad = false;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_blocks;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t* p = blk + i * (kPtq1Bytes / 4);  // 4-byte aligned: 28 = 4 * 7
    uint32_t u[7];
#pragma unroll
    for (int k = 0; k < 7; ++k) u[k] = __ldg(p + k);
    const uint8_t* b = reinterpret_cast<const uint8_t*>(u);
    uint32_t wd[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int j = 0; j < 26; ++j) {
      const uint32_t v = b[2 + j];
      const uint32_t e = lut[v];
      bad |= (e >> 31) != 0;
      const int k = 5 * j, sh = 2 * (k & 15);
      if (j < 25) {
        wd[k >> 4] |= e << sh;
        if (sh > 22) wd[(k >> 4) + 1] |= (e & 0x3FFu) >> (32 - sh);
      } else {  // trits 125..127, then two digits that must be zero
        bad |= v > 26u;
        wd[7] |= (e & 0x3Fu) << sh;
      }
    }
    uint4* dst = reinterpret_cast<uint4*>(w + i * 8);
    dst[0] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
    dst[1] = make_uint4(wd[4], wd[5], wd[6], wd[7]);
    const uint16_t d = (uint16_t)(u[0] & 0xFFFFu);
    scales[i] = d;
    if (biases) biases[i] = d ^ 0x8000u;
  }
  if (bad) set_status(status, TB_DEV_BAD_CODE);
}

// The other direction, W2 words and group scales -> GGUF blocks, in the scale-only reading (each
// bias is the pack's -scale and is not read).  A code of 3 is not a trit: it is flagged, PQ2_0
// keeps it in its slot and PTQ1_0 writes it as 2.
__global__ void __launch_bounds__(256) encode_pq2_0_kernel(const uint32_t* __restrict__ w,
                                                          const uint16_t* __restrict__ scales,
                                                          int64_t n_blocks, uint16_t* __restrict__ blk,
                                                          int32_t* __restrict__ status) {
  bool bad = false;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_blocks;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4* src = reinterpret_cast<const uint4*>(w + i * 8);
    const uint4 a = __ldg(src), b = __ldg(src + 1);
    const uint32_t wd[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint16_t* p = blk + i * (kPq2Bytes / 2);
    p[0] = __ldg(scales + i);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      bad |= (wd[k] & (wd[k] >> 1) & 0x55555555u) != 0;
      p[1 + 2 * k] = (uint16_t)(wd[k] & 0xFFFFu);
      p[2 + 2 * k] = (uint16_t)(wd[k] >> 16);
    }
  }
  if (bad) set_status(status, TB_DEV_BAD_CODE);
}

__global__ void __launch_bounds__(256) encode_ptq1_0_kernel(const uint32_t* __restrict__ w,
                                                           const uint16_t* __restrict__ scales,
                                                           int64_t n_blocks, uint32_t* __restrict__ blk,
                                                           int32_t* __restrict__ status) {
  bool bad = false;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_blocks;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4* src = reinterpret_cast<const uint4*>(w + i * 8);
    const uint4 a = __ldg(src), b = __ldg(src + 1);
    const uint32_t wd[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t out[7] = {(uint32_t)__ldg(scales + i), 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int j = 0; j < 26; ++j) {  // byte 2 + j: trits 5j .. 5j+4 below 128, first the least significant
      uint32_t v = 0;
#pragma unroll
      for (int d = 4; d >= 0; --d) {
        const int p = 5 * j + d;
        if (p >= 128) continue;
        uint32_t q = (wd[p >> 4] >> (2 * (p & 15))) & 3u;
        bad |= q == 3u;
        q = q == 3u ? 2u : q;
        v = 3u * v + q;
      }
      const int byte = 2 + j;
      out[byte >> 2] |= v << (8 * (byte & 3));
    }
    uint32_t* p = blk + i * (kPtq1Bytes / 4);
#pragma unroll
    for (int k = 0; k < 7; ++k) p[k] = out[k];
  }
  if (bad) set_status(status, TB_DEV_BAD_CODE);
}

}  // namespace tb

extern "C" int tb_transcode_gguf(const uint8_t* blocks, int format, int64_t N, int64_t K, uint32_t* w,
                                 uint16_t* scales, uint16_t* biases, int32_t* dev_status, void* stream) {
  using namespace tb;
  if (!blocks || !w || !scales) return TB_ERR_NULL;  // biases may be NULL (not written)
  if (format != TB_FMT_PQ2_0 && format != TB_FMT_PTQ1_0) return TB_ERR_UNSUPPORTED;
  if (N < 1 || K < kGroup || K % kGroup) return TB_ERR_SHAPE;
  const uintptr_t ba = reinterpret_cast<uintptr_t>(blocks);
  if ((format == TB_FMT_PQ2_0 && (ba & 1u)) || (format == TB_FMT_PTQ1_0 && (ba & 3u)) ||
      !aligned16(w) || (reinterpret_cast<uintptr_t>(scales) & 1u) ||
      (biases && (reinterpret_cast<uintptr_t>(biases) & 1u)))
    return TB_ERR_ALIGN;
  DeviceFacts f;
  int rc = device_facts(&f);
  if (rc != TB_OK) return rc;
  const int64_t n_blocks = N * (K / kGroup);
  int64_t grid = (n_blocks + 255) / 256;
  const int64_t cap = (int64_t)f.sms * 16;
  if (grid > cap) grid = cap;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (format == TB_FMT_PQ2_0)
    transcode_pq2_0_kernel<<<(int)grid, 256, 0, s>>>(reinterpret_cast<const uint16_t*>(blocks), n_blocks, w,
                                                      scales, biases, dev_status);
  else
    transcode_ptq1_0_kernel<<<(int)grid, 256, 0, s>>>(reinterpret_cast<const uint32_t*>(blocks), n_blocks, w,
                                                       scales, biases, dev_status);
  return check_launch();
}

extern "C" int tb_encode_gguf(const uint32_t* w, const uint16_t* scales, int64_t N, int64_t K, int format,
                              uint8_t* blocks, int32_t* dev_status, void* stream) {
  using namespace tb;
  if (!w || !scales || !blocks) return TB_ERR_NULL;
  if (format != TB_FMT_PQ2_0 && format != TB_FMT_PTQ1_0) return TB_ERR_UNSUPPORTED;
  if (N < 1 || K < kGroup || K % kGroup) return TB_ERR_SHAPE;
  const uintptr_t ba = reinterpret_cast<uintptr_t>(blocks);
  if ((format == TB_FMT_PQ2_0 && (ba & 1u)) || (format == TB_FMT_PTQ1_0 && (ba & 3u)) || !aligned16(w) ||
      (reinterpret_cast<uintptr_t>(scales) & 1u))
    return TB_ERR_ALIGN;
  DeviceFacts f;
  int rc = device_facts(&f);
  if (rc != TB_OK) return rc;
  const int64_t n_blocks = N * (K / kGroup);
  int64_t grid = (n_blocks + 255) / 256;
  const int64_t cap = (int64_t)f.sms * 16;
  if (grid > cap) grid = cap;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (format == TB_FMT_PQ2_0)
    encode_pq2_0_kernel<<<(int)grid, 256, 0, s>>>(w, scales, n_blocks, reinterpret_cast<uint16_t*>(blocks),
                                                  dev_status);
  else
    encode_ptq1_0_kernel<<<(int)grid, 256, 0, s>>>(w, scales, n_blocks, reinterpret_cast<uint32_t*>(blocks),
                                                   dev_status);
  return check_launch();
}
