// Sign * normalised Sylvester-Walsh-Hadamard transform over blocks of 1024.
//
// [ARCH] kwkr.cn/news/564617, section "Hadamard 旋转把量化误差抹平的免费午餐": fwht is a
// fast Walsh-Hadamard transform with scale 1/sqrt(block); the forward path multiplies
// by the explicit signs first, the inverse path multiplies by them again at the end.
// [PACK] lpnh.cn/news/2438023, section "仿射 2-bit 格式与 Prism contract v1": block 1024,
// normalized-sylvester-walsh-hadamard, along the input's last dimension.
//
// One warp owns one 1024-element block: 32 values per lane, five butterfly stages
// in registers, a transpose through a padded shared-memory tile, five more stages
// in registers.  fp32 throughout, fp16 (round to nearest even) on the way out.
#include <cuda_runtime.h>

#include "tb_common.cuh"
#include "tb_host.h"

namespace tb {

constexpr int kFwhtWarps = 8;

// x (fp16) * signs for one block in layout B (element j*32 + lane)
TB_DEVI void load_signed_block_b(const __half* __restrict__ xb, const int8_t* __restrict__ sb,
                                 int lane, float (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    float f = __half2float(xb[j * 32 + lane]);
    if (sb && sb[j * 32 + lane] < 0) f = -f;
    v[j] = f;
  }
}

// Plain transform: y = (H/32)(s*x) or s*((H/32)x), row-major [M, K] -> [M, K].
__global__ void __launch_bounds__(kFwhtWarps * 32) fwht1024_kernel(const __half* x,
                                                                   __half* y,
                                                                   const int8_t* __restrict__ signs,
                                                                   int64_t M, int64_t K,
                                                                   int inverse) {
  __shared__ float scratch[kFwhtWarps][kWarpScratchFloats];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nblk = K / kBlock;
  const int64_t items = M * nblk;
  for (int64_t it = blockIdx.x * (int64_t)kFwhtWarps + warp; it < items;
       it += (int64_t)gridDim.x * kFwhtWarps) {
    const int64_t m = it / nblk, b = it % nblk;
    const int64_t base = m * K + b * kBlock;
    const int8_t* sb = signs ? signs + b * kBlock : nullptr;
    float v[32];
    load_signed_block_b(x + base, inverse ? nullptr : sb, lane, v);
    wht1024_b_to_a(v, scratch[warp], lane);  // now v[r] = element lane*32 + r
    if (inverse && sb) {
      const int4 s0 = *reinterpret_cast<const int4*>(sb + lane * 32);
      const int4 s1 = *reinterpret_cast<const int4*>(sb + lane * 32 + 16);
      const int8_t* sp0 = reinterpret_cast<const int8_t*>(&s0);
      const int8_t* sp1 = reinterpret_cast<const int8_t*>(&s1);
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        if (sp0[r] < 0) v[r] = -v[r];
        if (sp1[r] < 0) v[16 + r] = -v[16 + r];
      }
    }
    uint32_t packed[16];
#pragma unroll
    for (int r = 0; r < 16; ++r)
      packed[r] = pack_half2(v[2 * r] * kInvSqrtBlock, v[2 * r + 1] * kInvSqrtBlock);
    uint4* dst = reinterpret_cast<uint4*>(y + base + lane * 32);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
  }
}

// Operand producer of the tensor-core path: x' = (H/32)(s*x) (or x when rotate == 0),
// rounded to fp16 and written with the codes' pair order inside every 16 columns:
//   out[16c + 2p] = x'[16c + p],  out[16c + 2p + 1] = x'[16c + p + 8]   (p = 0..7)
// which is the order in which the GEMM decodes a packed word into half2 pairs.
__global__ void __launch_bounds__(kFwhtWarps * 32) rotate_pairorder_kernel(
    const __half* __restrict__ x, __half* __restrict__ out, const int8_t* __restrict__ signs,
    int64_t M, int64_t K, int rotate) {
  __shared__ float scratch[kFwhtWarps][kWarpScratchFloats];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nblk = (K + kBlock - 1) / kBlock;
  const int64_t items = M * nblk;
  for (int64_t it = blockIdx.x * (int64_t)kFwhtWarps + warp; it < items;
       it += (int64_t)gridDim.x * kFwhtWarps) {
    const int64_t m = it / nblk, b = it % nblk;
    const int64_t base = m * K + b * kBlock;
    float v[32];
    if (rotate) {
      load_signed_block_b(x + base, signs ? signs + b * kBlock : nullptr, lane, v);
      wht1024_b_to_a(v, scratch[warp], lane);
#pragma unroll
      for (int r = 0; r < 32; ++r) v[r] *= kInvSqrtBlock;
    } else {
      // no rotation: the last chunk of K may be shorter than 1024 (K % 128 == 0)
      if (b * kBlock + lane * 32 >= K) continue;
      const uint4* src = reinterpret_cast<const uint4*>(x + base + lane * 32);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 u = src[q];
        const __half* h = reinterpret_cast<const __half*>(&u);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[8 * q + e] = __half2float(h[e]);
      }
    }
    uint32_t packed[16];
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int p = 0; p < 8; ++p) packed[8 * c + p] = pack_half2(v[16 * c + p], v[16 * c + p + 8]);
    uint4* dst = reinterpret_cast<uint4*>(out + base + lane * 32);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
  }
}

int launch_rotate_pairorder(const __half* x, __half* out, const int8_t* signs, int64_t M,
                            int64_t K, int rotate, cudaStream_t s) {
  DeviceFacts f;
  int rc = device_facts(&f);
  if (rc != TB_OK) return rc;
  const int64_t items = M * ((K + kBlock - 1) / kBlock);
  int64_t blocks = (items + kFwhtWarps - 1) / kFwhtWarps;
  const int64_t cap = (int64_t)f.sms * 8;
  if (blocks > cap) blocks = cap;
  rotate_pairorder_kernel<<<(int)blocks, kFwhtWarps * 32, 0, s>>>(x, out, signs, M, K, rotate);
  return check_launch();
}

}  // namespace tb

extern "C" int tb_fwht(const uint16_t* x, uint16_t* y, const int8_t* signs, int64_t M, int64_t K,
                       int block, int inverse, void* stream) {
  using namespace tb;
  if (!x || !y) return TB_ERR_NULL;
  if (block != kBlock) return TB_ERR_UNSUPPORTED;
  if (M < 1 || K < kBlock || K % kBlock) return TB_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(y) || (signs && !aligned16(signs))) return TB_ERR_ALIGN;
  DeviceFacts f;
  int rc = device_facts(&f);
  if (rc != TB_OK) return rc;
  const int64_t items = M * (K / kBlock);
  int64_t blocks = (items + kFwhtWarps - 1) / kFwhtWarps;
  const int64_t cap = (int64_t)f.sms * 8;
  if (blocks > cap) blocks = cap;
  fwht1024_kernel<<<(int)blocks, kFwhtWarps * 32, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const __half*>(x), reinterpret_cast<__half*>(y), signs, M, K,
      inverse ? 1 : 0);
  return check_launch();
}
