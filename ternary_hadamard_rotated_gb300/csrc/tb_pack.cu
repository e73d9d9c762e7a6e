// Weight packer and unpacker of the W2-g128 affine container.
//
// [ARCH] kwkr.cn/news/564617, section "打包格式的工程MLX 2.25 bits 与 GGUF 的两种装箱":
// ternary codes are stored as {0,1,2}, "rearranged into uint32 words", with one
// fp16 scale and one fp16 bias = -scale per 128 weights; the codec carries an
// independent unpack() that checks the packing.  Word layout (a reading of that
// sentence): code i of a word at bits 2i..2i+1, least significant first.
#include <cuda_runtime.h>

#include "tb_common.cuh"
#include "tb_host.h"

namespace tb {

// 16 int8 codes -> one word.  Per byte q = (t + 1) mod 256; a code is valid when q <= 2.
__global__ void __launch_bounds__(256) pack_w2_kernel(const uint4* __restrict__ codes16,
                                                      uint32_t* __restrict__ w, int64_t n_words,
                                                      int32_t* __restrict__ dev_status) {
  bool bad = false;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_words;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 c = __ldg(codes16 + i);
    const uint32_t part[4] = {c.x, c.y, c.z, c.w};
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t q = __vadd4(part[j], 0x01010101u);  // bytewise t + 1, no carries
      bad |= __vcmpleu4(q, 0x02020202u) != 0xFFFFFFFFu;
      const uint32_t m = q & 0x03030303u;
      const uint32_t b = (m & 0x03u) | ((m >> 6) & 0x0Cu) | ((m >> 12) & 0x30u) | ((m >> 18) & 0xC0u);
      word |= b << (8 * j);
    }
    w[i] = word;
  }
  if (bad) set_status(dev_status, TB_DEV_BAD_CODE);
}

// biases = -scales: flip the fp16 sign bit (exact for every value)
__global__ void __launch_bounds__(256) negate_half_kernel(const uint16_t* __restrict__ s,
                                                          uint16_t* __restrict__ b, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    b[i] = s[i] ^ 0x8000u;
}

// one word -> 16 int8 codes t = q - 1
__global__ void __launch_bounds__(256) unpack_w2_kernel(const uint32_t* __restrict__ w,
                                                        uint4* __restrict__ codes16,
                                                        int64_t n_words) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_words;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t word = __ldg(w + i);
    uint32_t out[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t b = word >> (8 * j);  // codes 4j..4j+3 in the low byte
      const uint32_t q = (b & 3u) | ((b & 0x0Cu) << 6) | ((b & 0x30u) << 12) | ((b & 0xC0u) << 18);
      out[j] = __vsub4(q, 0x01010101u);
    }
    codes16[i] = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

static int grid_for(int64_t n, int threads) {
  DeviceFacts f;
  int sms = 148;
  if (device_facts(&f) == TB_OK) sms = f.sms;
  int64_t blocks = (n + threads - 1) / threads;
  const int64_t cap = (int64_t)sms * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}

}  // namespace tb

extern "C" int tb_pack_w2(const int8_t* codes, const uint16_t* scales, int64_t N, int64_t K,
                          uint32_t* w, uint16_t* biases, int32_t* dev_status, void* stream) {
  using namespace tb;
  if (!codes || !scales || !w || !biases) return TB_ERR_NULL;
  if (N < 1 || K < kGroup || K % kGroup) return TB_ERR_SHAPE;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(w) || !aligned16(biases))
    return TB_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t n_words = N * (K / kCodesPerWord);
  pack_w2_kernel<<<grid_for(n_words, 256), 256, 0, s>>>(reinterpret_cast<const uint4*>(codes), w,
                                                        n_words, dev_status);
  int rc = check_launch();
  if (rc != TB_OK) return rc;
  const int64_t n_groups = N * (K / kGroup);
  negate_half_kernel<<<grid_for(n_groups, 256), 256, 0, s>>>(scales, biases, n_groups);
  return check_launch();
}

extern "C" int tb_unpack_w2(const uint32_t* w, int64_t N, int64_t K, int8_t* codes, void* stream) {
  using namespace tb;
  if (!w || !codes) return TB_ERR_NULL;
  if (N < 1 || K < kCodesPerWord || K % kCodesPerWord) return TB_ERR_SHAPE;
  if (!aligned16(w) || !aligned16(codes)) return TB_ERR_ALIGN;
  const int64_t n_words = N * (K / kCodesPerWord);
  unpack_w2_kernel<<<grid_for(n_words, 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      w, reinterpret_cast<uint4*>(codes), n_words);
  return check_launch();
}
