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
  // the consumer of x' (tensor-core GEMM or batched-decode GEMV, launched as a programmatic
  // dependent) may start its set-up and weight decoding now; it reads x' only after
  // griddepcontrol.wait, i.e. after this grid has completed
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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

// ---------------------------------------------------------------- blocks of 512, 2048, 4096
// The pack's loader accepts these block sizes too ([PACK] "仿射 2-bit 格式与 Prism contract v1").
// They reuse the warp transform of a 1024-chunk in layout C (register index = element bits
// 0..2 and 8..9, lane = bits 3..7):
//   512:  a warp transforms one 1024-chunk of a row without the stage of element bit 9 (register
//         bit 4), i.e. the two 512-blocks in it; a row that ends in the middle of a chunk leaves
//         its upper half unloaded and unstored;
//   2048, 4096: the G = 2 or 4 warps of a block each transform one chunk, write it to their
//         shared scratch, and the G-point stages across the chunks (element bits 10..11) run on
//         the values of equal (register, lane), which are equal element offsets in every chunk.
// Scale 1/sqrt(block) at the end, in fp32 (exact for 4096, rounded for 512 and 2048).

// the butterfly stages over the register bits set in MASK
template <int MASK>
TB_DEVI void butterfly32_mask(float (&v)[32]) {
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
    if (!(MASK & h)) continue;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = a + b;
        v[i + h] = a - b;
      }
    }
  }
}

// loads of one chunk in layout C with the lanes' q-quarters (elements q*256 + 8L .. + 7) live
// below `live_q`; dead quarters read as zero (and their signs as +1)
TB_DEVI void load_chunk_c(const __half* __restrict__ xb, const int8_t* __restrict__ sb, int lane,
                          int live_q, float (&v)[32], bool apply_signs) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u = make_uint4(0, 0, 0, 0);
    int2 sg = make_int2(0, 0);
    if (q < live_q) {
      u = __ldg(reinterpret_cast<const uint4*>(xb + q * 256 + lane * 8));
      if (apply_signs) sg = __ldg(reinterpret_cast<const int2*>(sb + q * 256 + lane * 8));
    }
    const __half* h = reinterpret_cast<const __half*>(&u);
    const int8_t* sp = reinterpret_cast<const int8_t*>(&sg);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float f = __half2float(h[e]);
      v[8 * q + e] = sp[e] < 0 ? -f : f;
    }
  }
}

// scale, the inverse path's signs, fp16 out, quarters below live_q
TB_DEVI void store_chunk_c(__half* yb, const int8_t* __restrict__ sb, int lane, int live_q,
                           float (&v)[32], float scale, bool apply_signs) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (q >= live_q) continue;
    int2 sg = make_int2(0, 0);
    if (apply_signs) sg = __ldg(reinterpret_cast<const int2*>(sb + q * 256 + lane * 8));
    const int8_t* sp = reinterpret_cast<const int8_t*>(&sg);
    float f[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = sp[e] < 0 ? -v[8 * q + e] * scale : v[8 * q + e] * scale;
    *reinterpret_cast<uint4*>(yb + q * 256 + lane * 8) =
        make_uint4(pack_half2(f[0], f[1]), pack_half2(f[2], f[3]), pack_half2(f[4], f[5]),
                   pack_half2(f[6], f[7]));
  }
}

__global__ void __launch_bounds__(kFwhtWarps * 32, kFwhtMinCtas) fwht512_kernel(
    const __half* x, __half* y, const int8_t* __restrict__ signs, int64_t M, int64_t K, int inverse,
    float scale) {
  __shared__ float scratch[kFwhtWarps][kWarpScratchFloats];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nchunk = (K + kBlock - 1) / kBlock;
  const int64_t items = M * nchunk;
  for (int64_t it = blockIdx.x * (int64_t)kFwhtWarps + warp; it < items;
       it += (int64_t)gridDim.x * kFwhtWarps) {
    const int64_t m = it / nchunk, c = it % nchunk;
    const int64_t base = m * K + c * kBlock;
    const int live_q = K - c * kBlock >= kBlock ? 4 : 2;  // K is a multiple of 512
    const int8_t* sb = signs ? signs + c * kBlock : nullptr;
    float v[32];
    load_chunk_c(x + base, sb, lane, live_q, v, sb && !inverse);
    butterfly32_mask<15>(v);  // element bits 0..2 and 8, not 9
    transpose_a_to_b(v, scratch[warp], lane);
    butterfly32(v);  // element bits 3..7
    transpose_b_to_a(v, scratch[warp], lane);
    store_chunk_c(y + base, sb, lane, live_q, v, scale, sb && inverse);
  }
}

// 2048: one warp holds a block's two chunks and runs the stage of element bit 10 in registers.
__global__ void __launch_bounds__(kFwhtWarps * 32, kFwhtMinCtas) fwht2048_kernel(
    const __half* x, __half* y, const int8_t* __restrict__ signs, int64_t M, int64_t K, int inverse,
    float scale) {
  constexpr int B = 2 * kBlock;
  __shared__ float scratch[kFwhtWarps][kWarpScratchFloats];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nb = K / B;
  const int64_t items = M * nb;
  for (int64_t bi = blockIdx.x * (int64_t)kFwhtWarps + warp; bi < items;
       bi += (int64_t)gridDim.x * kFwhtWarps) {
    const int64_t m = bi / nb, kb = bi % nb;
    const int64_t base = m * K + kb * B;
    const int8_t* sb = signs ? signs + kb * B : nullptr;
    float v[2][32];
#pragma unroll
    for (int g = 0; g < 2; ++g)
      load_chunk_c(x + base + g * kBlock, sb ? sb + g * kBlock : nullptr, lane, 4, v[g], sb && !inverse);
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      butterfly32(v[g]);  // element bits 0..2, 8, 9
      transpose_a_to_b(v[g], scratch[warp], lane);
      butterfly32(v[g]);  // element bits 3..7
      transpose_b_to_a(v[g], scratch[warp], lane);
    }
#pragma unroll
    for (int r = 0; r < 32; ++r) {  // element bit 10: equal (register, lane) is an equal offset
      const float a = v[0][r], b = v[1][r];
      v[0][r] = a + b;
      v[1][r] = a - b;
    }
#pragma unroll
    for (int g = 0; g < 2; ++g)
      store_chunk_c(y + base + g * kBlock, sb ? sb + g * kBlock : nullptr, lane, 4, v[g], scale,
                    sb && inverse);
  }
}

// 4096: a pair of warps per block, each holding two chunks (element bit 11 = which warp, bit 10 =
// which chunk of the warp's two); bit 10 in registers, bit 11 through the shared scratch with
// the partner warp on a named barrier of the pair.
constexpr int k4096Warps = 4;
__global__ void __launch_bounds__(k4096Warps * 32) fwht4096_kernel(
    const __half* x, __half* y, const int8_t* __restrict__ signs, int64_t M, int64_t K, int inverse,
    float scale) {
  constexpr int B = 4 * kBlock;
  __shared__ float scratch[k4096Warps][2][kWarpScratchFloats];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int half = warp & 1;      // element bit 11 of this warp's chunks
  const int bar = 1 + (warp >> 1);
  const int64_t nb = K / B;
  const int64_t items = M * nb;
  constexpr int kPairs = k4096Warps / 2;
  for (int64_t bi = blockIdx.x * (int64_t)kPairs + (warp >> 1); bi < items;
       bi += (int64_t)gridDim.x * kPairs) {
    const int64_t m = bi / nb, kb = bi % nb;
    const int64_t base = m * K + kb * B + half * 2 * kBlock;
    const int8_t* sb = signs ? signs + kb * B + half * 2 * kBlock : nullptr;
    float v[2][32];
#pragma unroll
    for (int g = 0; g < 2; ++g)
      load_chunk_c(x + base + g * kBlock, sb ? sb + g * kBlock : nullptr, lane, 4, v[g], sb && !inverse);
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      butterfly32(v[g]);  // element bits 0..2, 8, 9
      transpose_a_to_b(v[g], scratch[warp][0], lane);
      butterfly32(v[g]);  // element bits 3..7
      transpose_b_to_a(v[g], scratch[warp][0], lane);
    }
#pragma unroll
    for (int r = 0; r < 32; ++r) {  // element bit 10
      const float a = v[0][r], b = v[1][r];
      v[0][r] = a + b;
      v[1][r] = a - b;
    }
    // element bit 11: the partner warp holds the other half at equal (chunk, register, lane)
#pragma unroll
    for (int g = 0; g < 2; ++g)
#pragma unroll
      for (int r = 0; r < 32; ++r) scratch[warp][g][r * 33 + lane] = v[g][r];
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(64) : "memory");
#pragma unroll
    for (int g = 0; g < 2; ++g)
#pragma unroll
      for (int r = 0; r < 32; ++r) {
        const float o = scratch[warp ^ 1][g][r * 33 + lane];
        v[g][r] = half ? o - v[g][r] : v[g][r] + o;
      }
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(64) : "memory");  // before the scratch is reused
#pragma unroll
    for (int g = 0; g < 2; ++g)
      store_chunk_c(y + base + g * kBlock, sb ? sb + g * kBlock : nullptr, lane, 4, v[g], scale,
                    sb && inverse);
  }
}

// y = fwht(x) over blocks of `block` (512, 1024, 2048 or 4096); arguments already checked
int launch_fwht(const __half* x, __half* y, const int8_t* signs, int64_t M, int64_t K, int block,
                int inverse, cudaStream_t s) {
  DeviceFacts f;
  int rc = device_facts(&f);
  if (rc != TB_OK) return rc;
  if (block == kBlock) {
    const int64_t items = M * (K / kBlock);
    int64_t blocks = (items + kFwhtWarps - 1) / kFwhtWarps;
    const int64_t cap = (int64_t)f.sms * 8;
    if (blocks > cap) blocks = cap;
    fwht1024_kernel<<<(int)blocks, kFwhtWarps * 32, 0, s>>>(x, y, signs, M, K, inverse ? 1 : 0);
    return check_launch();
  }
  const float scale = (float)(1.0 / sqrt((double)block));
  const int inv = inverse ? 1 : 0;
  const int64_t cap = (int64_t)f.sms * 8;
  if (block == 512) {
    const int64_t items = M * ((K + kBlock - 1) / kBlock);
    int64_t blocks = (items + kFwhtWarps - 1) / kFwhtWarps;
    if (blocks > cap) blocks = cap;
    fwht512_kernel<<<(int)blocks, kFwhtWarps * 32, 0, s>>>(x, y, signs, M, K, inv, scale);
    return check_launch();
  }
  const int64_t items = M * (K / block);
  if (block == 2048) {
    int64_t blocks = (items + kFwhtWarps - 1) / kFwhtWarps;
    if (blocks > cap) blocks = cap;
    fwht2048_kernel<<<(int)blocks, kFwhtWarps * 32, 0, s>>>(x, y, signs, M, K, inv, scale);
    return check_launch();
  }
  if (block != 4096) return TB_ERR_UNSUPPORTED;
  int64_t blocks = (items + k4096Warps / 2 - 1) / (k4096Warps / 2);
  if (blocks > 2 * cap) blocks = 2 * cap;
  fwht4096_kernel<<<(int)blocks, k4096Warps * 32, 0, s>>>(x, y, signs, M, K, inv, scale);
  return check_launch();
}

}  // namespace tb

extern "C" int tb_fwht(const uint16_t* x, uint16_t* y, const int8_t* signs, int64_t M, int64_t K,
                       int block, int inverse, void* stream) {
  using namespace tb;
  if (!x || !y) return TB_ERR_NULL;
  if (!supported_block(block)) return TB_ERR_UNSUPPORTED;
  if (M < 1 || K < block || K % block) return TB_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(y) || (signs && !aligned16(signs))) return TB_ERR_ALIGN;
  return launch_fwht(reinterpret_cast<const __half*>(x), reinterpret_cast<__half*>(y), signs, M, K,
                     block, inverse, static_cast<cudaStream_t>(stream));
}
