// Embedding path of the Packed layer: gather a packed row, dequantise, inverse FWHT.
//
// [ARCH] kwkr.cn/news/564617, section "Hadamard 旋转把量化误差抹平的免费午餐":
//   an embedding module looks its rows up, dequantises them and returns the inverse
//   transform of the result (the Hadamard transform first, the signs last).
// [PACK] lpnh.cn/news/2438023, section "文本模型加载artifact.load_model 与 Packed 模块":
//   embed_tokens rows are restored with mx.dequantize, then the inverse Hadamard
//   transform is applied (transform first, signs last).
//
// One warp per (token, 1024-block): each lane decodes 32 consecutive weights from two
// packed words and its group's scale/bias (exact {-s, 0, s} in fp32), the warp runs
// the 1024-point transform (registers + one shared-memory transpose), multiplies by
// the signs and writes fp16.  An id outside [0, V) writes zeros and flags the status.
#include <cuda_runtime.h>

#include "tb_common.cuh"
#include "tb_host.h"

namespace tb {

constexpr int kEmbWarps = 8;

__global__ void __launch_bounds__(kEmbWarps * 32) embed_kernel(
    const int32_t* __restrict__ ids, int64_t T, const uint32_t* __restrict__ w,
    const __half* __restrict__ scales, const __half* __restrict__ biases, int64_t V, int64_t D,
    const int8_t* __restrict__ signs, int rotate, __half* __restrict__ out,
    int32_t* __restrict__ status) {
  __shared__ float scratch[kEmbWarps][kWarpScratchFloats];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nchunk = (D + kBlock - 1) / kBlock;
  const int64_t G = D / kGroup;
  for (int64_t it = blockIdx.x * (int64_t)kEmbWarps + warp; it < T * nchunk;
       it += (int64_t)gridDim.x * kEmbWarps) {
    const int64_t t = it / nchunk, b = it - t * nchunk;
    // the signs of this lane's 32 elements (layout A) do not depend on the id: loaded first
    int4 sg[2] = {make_int4(0, 0, 0, 0), make_int4(0, 0, 0, 0)};
    if (rotate && signs) {
      const int4* sp = reinterpret_cast<const int4*>(signs + b * kBlock + lane * 32);
      sg[0] = __ldg(sp);
      sg[1] = __ldg(sp + 1);
    }
    const int64_t id = ids[t];
    const bool ok = id >= 0 && id < V;
    if (!ok && b == 0 && lane == 0) set_status(status, TB_DEV_BAD_ID);
    const int64_t k0 = b * kBlock + lane * 32;  // first element of this lane (layout A)
    const bool in = k0 < D;
    float v[32];
    if (ok && in) {
      const uint2 wd = *reinterpret_cast<const uint2*>(w + id * (D / kCodesPerWord) + k0 / kCodesPerWord);
      const int64_t grp = id * G + k0 / kGroup;
      // no biases given: each is the pack's -scale
      const float s = __half2float(scales[grp]), bb = biases ? __half2float(biases[grp]) : -s;
#pragma unroll
      for (int r = 0; r < 32; ++r) {
        const uint32_t word = r < 16 ? wd.x : wd.y;
        const float q = (float)((word >> (2 * (r & 15))) & 3u);
        v[r] = fmaf(s, q, bb);  // exact for the pack's b = -s: {-s, 0, s}
      }
    } else {
#pragma unroll
      for (int r = 0; r < 32; ++r) v[r] = 0.f;
    }
    __half* orow = out + t * D + b * kBlock;
    if (rotate) {
      wht1024_a_to_b(v, scratch[warp], lane);     // v[j] = element j*32 + lane
      transpose_b_to_a(v, scratch[warp], lane);   // back to v[r] = element lane*32 + r
      const int8_t* sp = reinterpret_cast<const int8_t*>(sg);
#pragma unroll
      for (int r = 0; r < 32; ++r) {
        const float f = v[r] * kInvSqrtBlock;
        v[r] = sp[r] < 0 ? -f : f;
      }
    }
    if (in) {
      uint4* dst = reinterpret_cast<uint4*>(orow + lane * 32);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        dst[q4] = make_uint4(pack_half2(v[8 * q4], v[8 * q4 + 1]), pack_half2(v[8 * q4 + 2], v[8 * q4 + 3]),
                             pack_half2(v[8 * q4 + 4], v[8 * q4 + 5]), pack_half2(v[8 * q4 + 6], v[8 * q4 + 7]));
    }
  }
}

}  // namespace tb

extern "C" int tb_embed_lookup(const int32_t* ids, int64_t T, const uint32_t* w,
                               const uint16_t* scales, const uint16_t* biases, int64_t V,
                               int64_t D, const int8_t* signs, int block, uint16_t* out,
                               int32_t* dev_status, void* stream) {
  using namespace tb;
  if (T < 0 || V < 1 || D < kGroup || D % kGroup) return TB_ERR_SHAPE;
  if (block != 0 && !supported_block(block)) return TB_ERR_UNSUPPORTED;
  if (block && D % block) return TB_ERR_SHAPE;
  if (T == 0) return TB_OK;
  if (!ids || !w || !scales || !out) return TB_ERR_NULL;  // biases may be NULL
  if (!aligned16(w) || !aligned16(scales) || (biases && !aligned16(biases)) || !aligned16(out) ||
      (signs && !aligned16(signs)))
    return TB_ERR_ALIGN;
  DeviceFacts f;
  int rc = device_facts(&f);
  if (rc != TB_OK) return rc;
  const int64_t items = T * ((D + kBlock - 1) / kBlock);
  int64_t blocks = (items + kEmbWarps - 1) / kEmbWarps;
  const int64_t cap = (int64_t)f.sms * 8;
  if (blocks > cap) blocks = cap;
  // block 1024 is fused; another block decodes the rows (exact in fp16: {-s, 0, s}) and then
  // runs the inverse transform in place, which computes the same as the fused kernel
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  embed_kernel<<<(int)blocks, kEmbWarps * 32, 0, s>>>(
      ids, T, w, reinterpret_cast<const __half*>(scales), reinterpret_cast<const __half*>(biases), V,
      D, signs, block == kBlock, reinterpret_cast<__half*>(out), dev_status);
  rc = check_launch();
  if (rc != TB_OK || block == 0 || block == kBlock) return rc;
  return launch_fwht(reinterpret_cast<const __half*>(out), reinterpret_cast<__half*>(out), signs, T, D,
                     block, 1, s);
}
