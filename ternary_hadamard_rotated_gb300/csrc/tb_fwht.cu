// Sign * normalised Sylvester-Walsh-Hadamard transform over blocks of 1024.
//
// [ARCH] kwkr.cn/news/564617, section "Hadamard 旋转把量化误差抹平的免费午餐": fwht is a
// fast Walsh-Hadamard transform with scale 1/sqrt(block); the forward path multiplies
// by the explicit signs first, the inverse path multiplies by them again at the end.
// [PACK] lpnh.cn/news/2438023, section "仿射 2-bit 格式与 Prism contract v1": block 1024,
// normalized-sylvester-walsh-hadamard, along the input's last dimension.
//
// One warp owns one 1024-element block: 32 consecutive values per lane (16-byte loads and
// stores), five butterfly stages in registers, a transpose through a padded shared-memory
// tile, five more stages in registers and the transpose back.  fp32 throughout, fp16 (round to
// nearest even) on the way out.
#include <cuda_runtime.h>

#include "tb_common.cuh"
#include "tb_host.h"

namespace tb {

constexpr int kFwhtWarps = 8;
constexpr int kFwhtPerPass = 1;   // blocks a warp loads before transforming them (two measured slower)
constexpr int kFwhtMinCtas = 2;   // CTAs per SM the register allocation leaves room for

// Loads of one 1024-block for a warp in layout A (lane holds elements lane*32 .. lane*32 + 31):
// four 16-byte loads of x and two of the signs per lane.
struct BlockLoad {
  uint4 x[4];
  int4 s[2];
};
TB_DEVI void load_block_a(const __half* __restrict__ xb, const int8_t* __restrict__ sb, int lane,
                          BlockLoad& l) {
  const uint4* src = reinterpret_cast<const uint4*>(xb + lane * 32);
#pragma unroll
  for (int q = 0; q < 4; ++q) l.x[q] = __ldg(src + q);
  if (sb) {
    l.s[0] = __ldg(reinterpret_cast<const int4*>(sb + lane * 32));
    l.s[1] = __ldg(reinterpret_cast<const int4*>(sb + lane * 32 + 16));
  }
}
TB_DEVI void apply_signs_a(float (&v)[32], const int4 (&s)[2]) {
  const int8_t* sp = reinterpret_cast<const int8_t*>(s);
#pragma unroll
  for (int r = 0; r < 32; ++r)
    if (sp[r] < 0) v[r] = -v[r];
}
// (H/32)(s*x) (forward) or s*((H/32)x) (inverse) of one block, layout A in and out; the 32 x 33
// scratch of the warp carries the two transposes between the register stages.
TB_DEVI void transform_block_a(const BlockLoad& l, bool has_signs, bool inverse, float* scratch,
                               int lane, float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __half* h = reinterpret_cast<const __half*>(&l.x[q]);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[8 * q + e] = __half2float(h[e]);
  }
  if (has_signs && !inverse) apply_signs_a(v, l.s);
  wht1024_a_to_b(v, scratch, lane);  // register bits, transpose, lane bits: layout B
  transpose_b_to_a(v, scratch, lane);
#pragma unroll
  for (int r = 0; r < 32; ++r) v[r] *= kInvSqrtBlock;
  if (has_signs && inverse) apply_signs_a(v, l.s);
}

// Layout C of a block for the plain transform: lane L holds elements q*256 + 8L + i in
// v[8q + i] (q = 0..3, i = 0..7), so every 16-byte load or store instruction of the warp covers
// 512 contiguous bytes.  The register index spans element bits 0..2 and 8..9, the lane bits
// 3..7; the butterfly stages commute, so the same in-register stages and transposes as for
// layout A apply.
TB_DEVI void load_block_c(const __half* __restrict__ xb, const int8_t* __restrict__ sb, int lane,
                          BlockLoad& l) {
#pragma unroll
  for (int q = 0; q < 4; ++q) l.x[q] = __ldg(reinterpret_cast<const uint4*>(xb + q * 256 + lane * 8));
  if (sb) {
    const int2* s2 = reinterpret_cast<const int2*>(sb + lane * 8);
    const int2 a0 = __ldg(s2), a1 = __ldg(s2 + 32), a2 = __ldg(s2 + 64), a3 = __ldg(s2 + 96);
    l.s[0] = make_int4(a0.x, a0.y, a1.x, a1.y);
    l.s[1] = make_int4(a2.x, a2.y, a3.x, a3.y);
  }
}

// Plain transform: y = (H/32)(s*x) or s*((H/32)x), row-major [M, K] -> [M, K].  Each warp takes
// kFwhtPerPass blocks per pass (their loads in flight together).
__global__ void __launch_bounds__(kFwhtWarps * 32, kFwhtMinCtas) fwht1024_kernel(const __half* x,
                                                                   __half* y,
                                                                   const int8_t* __restrict__ signs,
                                                                   int64_t M, int64_t K,
                                                                   int inverse) {
  __shared__ float scratch[kFwhtWarps][kWarpScratchFloats];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nblk = K / kBlock;
  const int64_t items = M * nblk;
  const int64_t stride = (int64_t)gridDim.x * kFwhtWarps;
  for (int64_t it = blockIdx.x * (int64_t)kFwhtWarps + warp; it < items; it += kFwhtPerPass * stride) {
    BlockLoad l[kFwhtPerPass];
    int64_t base[kFwhtPerPass];
#pragma unroll
    for (int u = 0; u < kFwhtPerPass; ++u) {
      const int64_t iu = it + u * stride;
      if (iu >= items) break;
      const int64_t m = iu / nblk, b = iu % nblk;
      base[u] = m * K + b * kBlock;
      load_block_c(x + base[u], signs ? signs + b * kBlock : nullptr, lane, l[u]);
    }
#pragma unroll
    for (int u = 0; u < kFwhtPerPass; ++u) {
      if (it + u * stride >= items) break;
      float v[32];
      transform_block_a(l[u], signs != nullptr, inverse != 0, scratch[warp], lane, v);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(y + base[u] + q * 256 + lane * 8) =
            make_uint4(pack_half2(v[8 * q], v[8 * q + 1]), pack_half2(v[8 * q + 2], v[8 * q + 3]),
                       pack_half2(v[8 * q + 4], v[8 * q + 5]), pack_half2(v[8 * q + 6], v[8 * q + 7]));
    }
  }
}

// Operand producer of the tensor-core path: x' = (H/32)(s*x) (or x when rotate == 0),
// rounded to fp16 and written with the codes' pair order inside every 16 columns:
//   out[16c + 2p] = x'[16c + p],  out[16c + 2p + 1] = x'[16c + p + 8]   (p = 0..7)
// which is the order in which the GEMM decodes a packed word into half2 pairs.  Layout C (see
// above): a 16-column group lies in lanes 2m (columns p) and 2m + 1 (columns p + 8); one xor-1
// shuffle of four values gives each lane the 16 output bytes it stores.
__global__ void __launch_bounds__(kFwhtWarps * 32, kFwhtMinCtas) rotate_pairorder_kernel(
    const __half* __restrict__ x, __half* __restrict__ out, const int8_t* __restrict__ signs,
    int64_t M, int64_t K, int rotate) {
  __shared__ float scratch[kFwhtWarps][kWarpScratchFloats];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool odd = lane & 1;
  const int64_t nblk = (K + kBlock - 1) / kBlock;
  const int64_t items = M * nblk;
  const int64_t stride = (int64_t)gridDim.x * kFwhtWarps;
  for (int64_t it = blockIdx.x * (int64_t)kFwhtWarps + warp; it < items; it += stride) {
    const int64_t m = it / nblk, b = it % nblk;
    const int64_t base = m * K + b * kBlock;
    float v[32];
    bool live[4];  // this lane's columns q*256 + 8*lane .. + 7 lie inside K (always with rotate)
#pragma unroll
    for (int q = 0; q < 4; ++q) live[q] = rotate || b * kBlock + q * 256 + lane * 8 < K;
    if (rotate) {
      BlockLoad l;
      load_block_c(x + base, signs ? signs + b * kBlock : nullptr, lane, l);
      transform_block_a(l, signs != nullptr, false, scratch[warp], lane, v);
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 u = live[q] ? __ldg(reinterpret_cast<const uint4*>(x + base + q * 256 + lane * 8))
                                : make_uint4(0, 0, 0, 0);
        const __half* h = reinterpret_cast<const __half*>(&u);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[8 * q + e] = __half2float(h[e]);
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      // even lane keeps columns p = 0..3 and needs the odd lane's 0..3 (columns p + 8); the odd
      // lane keeps 4..7 and needs the even lane's 4..7
      float keep[4], give[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        keep[j] = odd ? v[8 * q + 4 + j] : v[8 * q + j];
        give[j] = odd ? v[8 * q + j] : v[8 * q + 4 + j];
      }
      const uint32_t g0 = pack_half2(give[0], give[1]), g1 = pack_half2(give[2], give[3]);
      const uint32_t r0 = __shfl_xor_sync(0xffffffffu, g0, 1), r1 = __shfl_xor_sync(0xffffffffu, g1, 1);
      const uint32_t k0 = pack_half2(keep[0], keep[1]), k1 = pack_half2(keep[2], keep[3]);
      // (first half, second half) of each output pair: (even's value, odd's value)
      const uint32_t f0 = odd ? r0 : k0, f1 = odd ? r1 : k1;  // columns p   (p = 4j' + 0..3)
      const uint32_t s0 = odd ? k0 : r0, s1 = odd ? k1 : r1;  // columns p + 8
      const uint4 o = make_uint4(__byte_perm(f0, s0, 0x5410), __byte_perm(f0, s0, 0x7632),
                                 __byte_perm(f1, s1, 0x5410), __byte_perm(f1, s1, 0x7632));
      if (live[q]) *reinterpret_cast<uint4*>(out + base + q * 256 + lane * 8) = o;
    }
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
