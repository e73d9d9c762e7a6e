// Device building blocks of the TMA-streamed decode GEMV (W2-g128 codes x fp16 x'), shared by
// the per-call kernel (tb_gemv_tma.cu) and the chained persistent kernel (tb_chain.cu).
//
// [ARCH] kwkr.cn/news/564617, section "Hadamard 旋转把量化误差抹平的免费午餐": the layer is
// the rotated input (signs, then the block Hadamard transform) times the packed 2-bit codes
// with their fp16 scales and biases (group 128), consumed directly and never expanded to a
// dense matrix.
//
// Work unit: 128 output rows x 512 k (4 groups of 128) = one 16 KB TMA box of packed codes
// (128 rows x 128 B, 128-byte swizzle).  Arithmetic per group of 128 and token: LOP3 puts each
// 2-bit code into the mantissa of an fp16 1024.0 (1024 + sigma*q, exact; sigma = 4^j from the
// field's bit position j); those half2 are mma.sync A fragments, x'/sigma the B fragment.  The
// first MMA of a group starts from zero (no register moves for the start value) and the
// epilogue takes C = 1024*sum(x'/sigma) off, which leaves D - C = sum q*x':
//   y += s * (D - C) + b * S,   S = sum x' over the group.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "tb_common.cuh"

namespace tb {

constexpr int kUnitRows = 128;
constexpr int kUnitGroups = 4;                          // groups per unit (512 k)
constexpr int kSlotBytes = kUnitRows * 128;             // 16 KB box of packed codes
constexpr int kGroupsOfWarps = 3;                       // unit groups
constexpr int kWarpsPerUnit = 4;                        // 32 rows each
constexpr int kTmaConsumers = kGroupsOfWarps * kWarpsPerUnit;
constexpr int kMaxSlotsPerGroup = 2;  // a deeper ring measured slower: it takes the L1 that the scale and activation loads hit
constexpr int kPreIssue = 1;        // units per group issued before the activations are loaded (two measured
                                    // 1.8% slower on a 257-call decode step: the activation loads queue
                                    // behind the weights; none leaves the first weights late)
constexpr int kCutSlots = 4;        // shared sums of tiles cut by a group or CTA boundary
constexpr int kScaleStageBytes = 32 * kUnitGroups * 8;  // per warp: 32 rows x 4 groups of fp32 (s, b)
constexpr uint32_t kMagic1024 = 0x64006400u;

constexpr int kMaxMats = 4;  // matrices sharing one input in one launch

struct GemvTmaLayout {
  int codes, img, cs, sstage, accs, cnt, bars, total;
};

__host__ __device__ inline int rup(int v, int a) { return (v + a - 1) / a * a; }


template <int MT>
__host__ __device__ inline GemvTmaLayout gemv_tma_layout(int G, int dw, int slot = kSlotBytes) {
  GemvTmaLayout L;
  int off = 0;
  L.codes = off;  // 1024-aligned slots (the 128-byte swizzle repeats every 1024 bytes)
  off += kGroupsOfWarps * dw * slot;
  L.img = off;
  off += G * 256 * MT;
  L.cs = off;
  off += G * MT * 8;
  off = rup(off, 16);
  L.sstage = off;
  off += kTmaConsumers * kScaleStageBytes;
  L.accs = off;
  off += kCutSlots * kUnitRows * MT * 4;
  L.cnt = off;
  off += kCutSlots * 4;
  off = rup(off, 8);
  L.bars = off;
  off += (2 * kGroupsOfWarps * dw + 1) * 8;
  L.total = off + 1024;  // slack to align the base to 1024
  return L;
}

// stream-K unit range [lo, hi) of CTA c
__host__ __device__ inline void cta_range_of(int c, int grid, int n_tiles, int C, int& lo, int& hi) {
  const int64_t S = (int64_t)n_tiles * C;
  lo = (int)(S * c / grid);
  hi = (int)(S * (c + 1) / grid);
}

// owner of global unit s when S units are cut into grid ranges [S*i/grid, S*(i+1)/grid)
__host__ __device__ inline int stage_owner(int64_t s, int64_t S, int grid) {
  return (int)(((s + 1) * grid - 1) / S);
}

TB_DEVI void mma16816_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}


TB_DEVI void mma16816_zero(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                           uint32_t b0, uint32_t b1) {
  const float z = 0.f;
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
}

TB_DEVI void decode_word_sigma(uint32_t w, uint32_t (&P)[8]) {
  const uint32_t w6 = w >> 6;
  P[0] = lop3_and_or(w, 0x00030003u, kMagic1024);   // codes 0, 8   sigma 1
  P[1] = lop3_and_or(w, 0x000C000Cu, kMagic1024);   // codes 1, 9   sigma 4
  P[2] = lop3_and_or(w, 0x00300030u, kMagic1024);   // codes 2, 10  sigma 16
  P[3] = lop3_and_or(w, 0x00C000C0u, kMagic1024);   // codes 3, 11  sigma 64
  P[4] = lop3_and_or(w, 0x03000300u, kMagic1024);   // codes 4, 12  sigma 256
  P[5] = lop3_and_or(w6, 0x00300030u, kMagic1024);  // codes 5, 13  sigma 16
  P[6] = lop3_and_or(w6, 0x00C000C0u, kMagic1024);  // codes 6, 14  sigma 64
  P[7] = lop3_and_or(w6, 0x03000300u, kMagic1024);  // codes 7, 15  sigma 256
}

TB_DEVI float inv_sigma_p(int p) {
  return p == 0 ? 1.0f : p == 1 ? 0.25f : (p == 2 || p == 5) ? 0.0625f
       : (p == 3 || p == 6) ? 0.015625f : 0.00390625f;
}

TB_DEVI void tma2d(uint32_t dst, const CUtensorMap* tm, int x, int y, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// One group gi (0..3) of a unit for the warp's two 16-row blocks: decode, 2 x 8 mma (two
// independent accumulator chains sharing one B fragment), scale epilogue.
//   box:  the unit's code box; R0, R0 + 16: this lane's A rows of block 0 (block 1 = + 16)
//   imgt: B-fragment image entry of this lane; csa: (C, S) pairs [G][MT]
//   ss:   this warp's staged (scale, bias) pairs, fp32 [32 rows][4 groups]
template <int MT>
TB_DEVI void unit_group(uint32_t box, int R0, int t, int gi, int grp, uint32_t imgt, uint32_t ss,
                        int rA, uint32_t csa, int t0, int t1, float (&acc)[2][4]) {
  const int c = 2 * gi + (t >> 1);  // logical 16-byte chunk of the 128-byte row
  uint2 w[2][2];
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int R = R0 + 16 * j + 8 * h;  // (R & 7) == (rA & 7)
      w[j][h] = ld_shared_v2(box + R * 128 + ((c ^ (rA & 7)) << 4) + (t & 1) * 8);
    }
  const float2 cs0 = ld_shared_f2(csa + (grp * MT + t0) * 8);
  const float2 cs1 = MT > 1 ? ld_shared_f2(csa + (grp * MT + t1) * 8) : cs0;
  float d[2][4];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const uint4 i0 = ld_shared_v4(imgt + (grp * 4 + 2 * half) * MT * 64);
    const uint4 i1 = ld_shared_v4(imgt + (grp * 4 + 2 * half + 1) * MT * 64);
    uint32_t P[2][8], Q[2][8];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      decode_word_sigma(half ? w[j][0].y : w[j][0].x, P[j]);
      decode_word_sigma(half ? w[j][1].y : w[j][1].x, Q[j]);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (half == 0) mma16816_zero(d[j], P[j][0], Q[j][0], P[j][1], Q[j][1], i0.x, i0.y);
      else mma16816_acc(d[j], P[j][0], Q[j][0], P[j][1], Q[j][1], i0.x, i0.y);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) mma16816_acc(d[j], P[j][2], Q[j][2], P[j][3], Q[j][3], i0.z, i0.w);
#pragma unroll
    for (int j = 0; j < 2; ++j) mma16816_acc(d[j], P[j][4], Q[j][4], P[j][5], Q[j][5], i1.x, i1.y);
#pragma unroll
    for (int j = 0; j < 2; ++j) mma16816_acc(d[j], P[j][6], Q[j][6], P[j][7], Q[j][7], i1.z, i1.w);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int ra = 16 * j + rA, rb = ra + 8;  // rows within the warp's 32
    const float2 A = ld_shared_f2(ss + (ra * kUnitGroups + gi) * 8);  // (s, b) of row ra
    const float2 B = ld_shared_f2(ss + (rb * kUnitGroups + gi) * 8);
    acc[j][0] = fmaf(A.x, d[j][0] - cs0.x, fmaf(A.y, cs0.y, acc[j][0]));
    acc[j][2] = fmaf(B.x, d[j][2] - cs0.x, fmaf(B.y, cs0.y, acc[j][2]));
    if (MT > 1) {  // D columns 2t+1 hold a second token only when there is one
      acc[j][1] = fmaf(A.x, d[j][1] - cs1.x, fmaf(A.y, cs1.y, acc[j][1]));
      acc[j][3] = fmaf(B.x, d[j][3] - cs1.x, fmaf(B.y, cs1.y, acc[j][3]));
    }
  }
}

// the unit after (or before) (tile, chunk) in tile-major order
TB_DEVI void step_unit(int& tile, int& chunk, int C, bool back) {
  if (back) {
    if (--chunk < 0) {
      chunk = C - 1;
      --tile;
    }
  } else if (++chunk == C) {
    chunk = 0;
    ++tile;
  }
}

// The 1024-blocks of x that the units [lo, lo + nst) of one CTA read: [b1, e1) and [b2, e2)
// (the second interval is non-empty only when the range wraps past the end of a tile and
// the two pieces do not already cover every block; both are empty for an empty range).
TB_DEVI void blocks_needed(int lo, int nst, int C, int K, int& b1, int& e1, int& b2, int& e2) {
  b1 = 0;
  e1 = nst > 0 ? K / kBlock : 0;
  b2 = 0;
  e2 = 0;
  if (nst > 0 && nst < C) {
    constexpr int kChunksPerBlock = kBlock / (kUnitGroups * kGroup);
    const int clo = lo % C, cend = clo + nst;
    b1 = clo / kChunksPerBlock;
    if (cend <= C) {
      e1 = (cend - 1) / kChunksPerBlock + 1;
    } else {
      e2 = (cend - C - 1) / kChunksPerBlock + 1;
      if (e2 >= b1) {
        b1 = 0;
        e2 = 0;
      }
    }
  }
}

// Fused prologue (sign * FWHT-1024, x' rounded to fp16) of the blocks [b1, e1) u [b2, e2)
// of Mc tokens, written as the decode GEMV's operands:
//   img: B-fragment image of x'/sigma, fp16, [group][4 mma k-steps][MT tokens][32 lanes x 8 B]
//   cs:  per group and token (1024 * sum(x'/sigma), sum x')
// Warp `w` of `nw` takes items (token, block) w, w + nw, ...; the loads of two items are in
// flight together.  x is read through L2 (ld.global.cg): it may have been written by other
// SMs earlier in the same launch.  `scratch` is a 4 KB shared buffer of the warp for the
// transform's transposes.
template <int MT>
TB_DEVI void prologue_image(const __half* x, const int8_t* signs, int K, int Mc, int rotate,
                            int b1, int e1, int b2, int e2, int w, int nw, int lane,
                            __half* img, float2* cs, uint32_t scratch) {
  const int t = lane & 3;
  const int nblk = (e1 - b1) + (e2 - b2);
  auto block_of = [&](int bi) { return bi < e1 - b1 ? b1 + bi : b2 + (bi - (e1 - b1)); };
  auto load_block = [&](int it, uint4 (&xr)[4], uint4 (&sr)[2]) {
    const int tok = it / nblk, b = block_of(it - tok * nblk);
    if (tok < Mc) {
      const uint4* xs = reinterpret_cast<const uint4*>(x + (int64_t)tok * K + b * kBlock + lane * 32);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) xr[q4] = __ldcg(xs + q4);
    } else {
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) xr[q4] = make_uint4(0, 0, 0, 0);
    }
    if (signs) {
      const uint4* sp = reinterpret_cast<const uint4*>(signs + b * kBlock + lane * 32);
      sr[0] = __ldg(sp);
      sr[1] = __ldg(sp + 1);
    }
  };
  auto transform_block = [&](int it, const uint4 (&xr)[4], const uint4 (&sr)[2]) {
    const int tok = it / nblk, b = block_of(it - tok * nblk);
    float v[32];  // layout A: v[r] = element b*1024 + lane*32 + r
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const __half* h = reinterpret_cast<const __half*>(&xr[q4]);
#pragma unroll
      for (int e = 0; e < 8; ++e) v[8 * q4 + e] = __half2float(h[e]);
    }
    if (signs) {
      const int8_t* sg = reinterpret_cast<const int8_t*>(sr);
#pragma unroll
      for (int r = 0; r < 32; ++r)
        if (sg[r] < 0) v[r] = -v[r];
    }
    if (rotate) {
      wht1024_a_smem(v, scratch, lane);
#pragma unroll
      for (int r = 0; r < 32; ++r) v[r] *= kInvSqrtBlock;
    }
    const int grp = b * (kBlock / kGroup) + (lane >> 2);
#pragma unroll
    for (int r = 0; r < 32; ++r) v[r] = __half2float(__float2half_rn(v[r]));  // x' rounded to fp16
    float ssum = tree_sum32(v);
    ssum += __shfl_xor_sync(0xffffffffu, ssum, 1);
    ssum += __shfl_xor_sync(0xffffffffu, ssum, 2);
    float cpart[4];  // C as four partial sums (one per mma k-step) of the fp16 values x'/sigma
#pragma unroll
    for (int mp = 0; mp < 4; ++mp) {
      uint32_t pk[4];
      float c2[4];
#pragma unroll
      for (int e2_ = 0; e2_ < 4; ++e2_) {
        const int p = 4 * (mp & 1) + e2_;
        const int r = (mp >> 1) * 16 + p;
        const float is = inv_sigma_p(p);
        const __half lo_ = __float2half_rn(v[r] * is), hi_ = __float2half_rn(v[r + 8] * is);
        c2[e2_] = __half2float(lo_) + __half2float(hi_);
        pk[e2_] = (uint32_t)__half_as_ushort(lo_) | ((uint32_t)__half_as_ushort(hi_) << 16);
      }
      cpart[mp] = (c2[0] + c2[1]) + (c2[2] + c2[3]);
      *reinterpret_cast<uint4*>(img + ((size_t)(grp * 4 + mp) * MT + tok) * 32 + t * 8) =
          make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
    float csum = (cpart[0] + cpart[1]) + (cpart[2] + cpart[3]);
    csum += __shfl_xor_sync(0xffffffffu, csum, 1);
    csum += __shfl_xor_sync(0xffffffffu, csum, 2);
    if (t == 0) cs[grp * MT + tok] = make_float2(1024.f * csum, ssum);
  };
  const int items = MT * nblk;
  for (int it = w; it < items; it += 2 * nw) {
    const int it2 = it + nw;
    uint4 xa[4], sa[2], xb[4], sb[2];
    load_block(it, xa, sa);
    if (it2 < items) load_block(it2, xb, sb);
    transform_block(it, xa, sa);
    if (it2 < items) transform_block(it2, xb, sb);
  }
}
}  // namespace tb
