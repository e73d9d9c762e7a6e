// Decode path of the Packed layer, TMA-streamed: fused sign*FWHT prologue + W2-g128 GEMV.
//
// [ARCH] kwkr.cn/news/564617, section "Hadamard 旋转把量化误差抹平的免费午餐":
//   if self.block: x = fwht(x, block, signs); y = quantized_matmul(x, weight, scales,
//   biases, transpose=True, group_size=128, bits=2): the packed 2-bit words are consumed
//   directly and never expanded to fp16.
// [PACK] lpnh.cn/news/2438023, section "文本模型加载artifact.load_model 与 Packed 模块".
//
// Work unit: 128 output rows x 512 k (4 groups of 128) = one 16 KB TMA box of packed codes
// (128 rows x 128 B, 128-byte swizzle; rows past N are zero-filled).  Each SM can keep only
// a handful of TMA requests in flight, so requests are made large: 16 KB boxes stream at
// the HBM rate where 2-4 KB requests stall at a fraction of it.  Scales and biases (8 B
// per row per unit) are read by the consumer warps themselves, two units ahead, and staged
// through shared memory.
//
// Schedule (stream-K): the units of all 128-row tiles, tile-major, are cut into one
// contiguous, equal range per CTA (one persistent CTA per SM).  A producer warp keeps a
// ring of 16 KB slots in flight; 12 consumer warps form 3 unit groups of 4 warps; group u
// takes the CTA's units u, u + 3, ... and warp i of the group the rows 32i..32i+31 of the
// unit.  Every warp adds its 32-row partial sums into a per-tile shared accumulator; the
// warp that completes a tile's count in this CTA writes y, or, when the tile continues in a
// neighbouring CTA, adds the CTA's partial into the tile's fp32 sum in the workspace, and
// the last of the tile's CTAs converts that sum to y and returns sum and counter to zero.
//
// Arithmetic (per group of 128, per token): LOP3 puts each 2-bit code into the mantissa of
// an fp16 1024.0 (1024 + sigma*q, exact; sigma = 4^j from the field's bit position j);
// those half2 are mma.sync A fragments, x'/sigma the B fragment, and the accumulator
// starts at -1024*sum(x'/sigma) so the tensor core returns D = sum q*x' directly:
//   y += s * D + b * S,   S = sum x' over the group.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>
#include <unordered_map>

#include "tb_common.cuh"
#include "tb_host.h"

namespace tb {

constexpr int kUnitRows = 128;
constexpr int kUnitGroups = 4;                       // groups per unit (512 k)
constexpr int kBoxBytes = kUnitRows * 128;           // 16 KB
constexpr int kGroupsOfWarps = 3;                    // unit groups
constexpr int kWarpsPerUnit = 4;                     // 32 rows each
constexpr int kTmaConsumers = kGroupsOfWarps * kWarpsPerUnit;
constexpr int kTmaThreads = (kTmaConsumers + 1) * 32;
constexpr int kTmaFwhtWarps = kTmaConsumers;  // every consumer warp transforms blocks
constexpr int kMaxSlotsPerGroup = 5;
constexpr int kScaleStageBytes = 32 * kUnitGroups * 8;  // per warp: 32 rows x 4 groups of fp32 (s, b)
constexpr uint32_t kMagic1024 = 0x64006400u;

constexpr int kMaxMats = 4;  // matrices sharing one input in one launch

struct GemvTmaArgs {
  const __half* x;               // [Mc, K]
  const int8_t* signs;           // [K] or null
  const __half* scales[kMaxMats];  // [N_i, G]
  const __half* biases[kMaxMats];  // [N_i, G]
  __half* y[kMaxMats];           // [Mc, N_i]
  int N[kMaxMats];               // rows of matrix i
  int tile0[kMaxMats + 1];       // first 128-row tile of matrix i in the concatenated tile list
  int nmat;
  float* ws_partial;             // [kFixupCtas][128][MT] fp32 sums of shared tiles, or null (tile-aligned)
  int* ws_count;                 // [kFixupCtas]
  int Mc, K, G, C;               // C = units per tile = K / 512
  int rotate, dw, tslots;
  int n_tiles;                   // total 128-row tiles of all matrices
  int split;                     // 1: stream-K ranges; 0: ranges on tile boundaries
  int32_t* status;
};

struct CodeMaps {
  CUtensorMap m[kMaxMats];
};

// matrix of a global tile index
TB_DEVI int mat_of(const GemvTmaArgs& a, int tile) {
  int i = 0;
#pragma unroll
  for (int k = 1; k < kMaxMats; ++k) i += (k < a.nmat && tile >= a.tile0[k]);
  return i;
}

struct GemvTmaLayout {
  int codes, img, cs, scratch, sstage, accs, cnt, bars, total;
};

__host__ __device__ inline int rup(int v, int a) { return (v + a - 1) / a * a; }

template <int MT>
__host__ __device__ inline GemvTmaLayout gemv_tma_layout(int G, int dw, int tslots) {
  GemvTmaLayout L;
  int off = 0;
  L.codes = off;  // 1024-aligned boxes (the 128-byte swizzle repeats every 1024 bytes)
  off += kGroupsOfWarps * dw * kBoxBytes;
  L.img = off;
  off += G * 256 * MT;
  L.cs = off;
  off += G * MT * 8;
  off = rup(off, 16);
  // scale staging and tile accumulators (the prologue needs no scratch)
  L.scratch = off;
  const int fw = 0;
  L.sstage = off;
  L.accs = L.sstage + kTmaConsumers * kScaleStageBytes;
  L.cnt = L.accs + (tslots + 1) * kUnitRows * MT * 4;
  const int after = L.cnt + (tslots + 1) * 4;
  off = off + fw > after ? off + fw : after;
  off = rup(off, 8);
  L.bars = off;
  off += 2 * kGroupsOfWarps * dw * 8;
  L.total = off + 1024;  // slack to align the base to 1024
  return L;
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
  for (int j = 0; j < 2; ++j) {
    d[j][0] = -cs0.x;
    d[j][1] = -cs1.x;
    d[j][2] = -cs0.x;
    d[j][3] = -cs1.x;
  }
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
    for (int j = 0; j < 2; ++j) mma16816_acc(d[j], P[j][0], Q[j][0], P[j][1], Q[j][1], i0.x, i0.y);
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
    acc[j][0] = fmaf(A.x, d[j][0], fmaf(A.y, cs0.y, acc[j][0]));
    acc[j][2] = fmaf(B.x, d[j][2], fmaf(B.y, cs0.y, acc[j][2]));
    if (MT > 1) {  // D columns 2t+1 hold a second token only when there is one
      acc[j][1] = fmaf(A.x, d[j][1], fmaf(A.y, cs1.y, acc[j][1]));
      acc[j][3] = fmaf(B.x, d[j][3], fmaf(B.y, cs1.y, acc[j][3]));
    }
  }
}

template <int MT>
__global__ void __launch_bounds__(kTmaThreads, 1)
    w2_gemv_tma_kernel(const __grid_constant__ CodeMaps maps, const __grid_constant__ GemvTmaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // unit group u owns slots [u*DW, (u+1)*DW) and takes the CTA's units u, u + 3, ... in
  // order, so no wait is ever more than one phase ahead of its barrier
  const int DW = a.dw, TS = a.tslots, C = a.C, G = a.G, K = a.K;
  const GemvTmaLayout L = gemv_tma_layout<MT>(G, DW, TS);
  const uint32_t codes_u32 = smem_u32(smem + L.codes);
  __half* img = reinterpret_cast<__half*>(smem + L.img);
  float2* cs = reinterpret_cast<float2*>(smem + L.cs);    // [G][MT] = (1024 sum x'/sigma, sum x')
  float* accs = reinterpret_cast<float*>(smem + L.accs);  // [TS][128][MT]
  int* cnt = reinterpret_cast<int*>(smem + L.cnt);         // [TS]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kGroupsOfWarps * DW;
  __shared__ volatile int aborted;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // this CTA's unit range
  const int64_t S = (int64_t)a.n_tiles * C;
  int64_t lo, hi;
  if (a.split) {
    lo = S * blockIdx.x / gridDim.x;
    hi = S * (blockIdx.x + 1) / gridDim.x;
  } else {
    lo = (int64_t)C * ((int64_t)a.n_tiles * blockIdx.x / gridDim.x);
    hi = (int64_t)C * ((int64_t)a.n_tiles * (blockIdx.x + 1) / gridDim.x);
  }
  const int nst = (int)(hi - lo);
  const int64_t tile_lo = lo / C;
  // Order of this CTA's units: a partial tail tile first, then a partial head tile, then the
  // complete tiles in order, so the cross-CTA sums of the shared tiles overlap the rest of
  // the work.  The partial tail tile has its own accumulator slot (TS).
  const int64_t last_tile = (hi - 1) / C;
  const bool one_tile = tile_lo == last_tile;
  const int hp = (!one_tile && lo % C) ? (int)((tile_lo + 1) * C - lo) : 0;
  const int tp = (!one_tile && hi % C) ? (int)(hi - last_tile * C) : 0;
  auto unit_of = [&](int q) -> int64_t {
    if (q < tp) return last_tile * C + q;
    if (q < tp + hp) return lo + (q - tp);
    return lo + (q - tp);  // head and middle in order after the tail
  };
  auto slot_of = [&](int64_t tile) -> int {
    return (tp > 0 && tile == last_tile) ? TS : (int)((tile - tile_lo) % TS);
  };

  if (threadIdx.x == 0) {
    aborted = 0;
    for (int i = 0; i < kGroupsOfWarps * DW; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, kWarpsPerUnit);
    }
    fence_barrier_init();
  }
  __syncthreads();

  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (aborted) return;
    if (!mbar_wait(bar, parity)) {
      aborted = 1;
      set_status(a.status, TB_DEV_TIMEOUT);
    }
  };

  if (warp == kTmaConsumers) {
    // ---- producer: the packed codes never depend on the previous kernel ----
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      for (int q = 0; q < nst; ++q) {
        const int n = q / kGroupsOfWarps, j = n % DW, k = n / DW;
        const int slot = (q % kGroupsOfWarps) * DW + j;
        if (k > 0) wait(empty + slot, (k - 1) & 1);
        const int64_t s = unit_of(q);
        const int tile = (int)(s / C), chunk = (int)(s - (int64_t)tile * C);
        const int mi = mat_of(a, tile);
        mbar_arrive_expect_tx(full + slot, kBoxBytes);
        tma2d(codes_u32 + slot * kBoxBytes, &maps.m[mi], chunk * 32, (tile - a.tile0[mi]) * kUnitRows,
              full + slot, pol);
      }
      // leave no copy in flight: the last use of every slot has completed
      for (int q = nst - 1; q >= 0 && q >= nst - kGroupsOfWarps * DW; --q) {
        const int n = q / kGroupsOfWarps;
        wait(full + (q % kGroupsOfWarps) * DW + n % DW, (n / DW) & 1);
      }
    }
    __syncwarp();
    return;
  }

  // ---- consumers ----
  const int g = lane >> 2, t = lane & 3;
  const int ug = warp / kWarpsPerUnit, wi = warp % kWarpsPerUnit;
  // scale / bias prefetch for this warp's units (rows 32*wi + lane of the unit)
  auto load_sb = [&](int q, uint2& sv, uint2& bv) {
    sv = make_uint2(0, 0);
    bv = make_uint2(0, 0);
    if (q >= nst) return;
    const int64_t s = unit_of(q);
    const int tile = (int)(s / C), chunk = (int)(s - (int64_t)tile * C);
    const int mi = mat_of(a, tile);
    const int row = (tile - a.tile0[mi]) * kUnitRows + 32 * wi + lane;
    if (row < a.N[mi]) {
      const int64_t off = (int64_t)row * G + chunk * kUnitGroups;
      sv = __ldg(reinterpret_cast<const uint2*>(a.scales[mi] + off));
      bv = __ldg(reinterpret_cast<const uint2*>(a.biases[mi] + off));
    }
  };
  uint2 s0, b0, s1, b1;
  load_sb(ug, s0, b0);
  load_sb(ug + kGroupsOfWarps, s1, b1);

  asm volatile("griddepcontrol.wait;" ::: "memory");
  {
    // prologue: x' = fwht(signs * x) -> B-fragment image, (C, S) per group and token.
    // Every consumer warp takes blocks (token, 1024-slice) warp, warp + 12, ...; the loads of
    // two blocks are issued before either is transformed, so a warp waits once per pair.
    const int nchunk = K / kBlock;
    auto load_block = [&](int it, uint4 (&xr)[4], uint4 (&sr)[2]) {
      const int tok = it / nchunk, b = it - tok * nchunk;
      if (tok < a.Mc) {
        const uint4* xs = reinterpret_cast<const uint4*>(a.x + (int64_t)tok * K + b * kBlock + lane * 32);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) xr[q4] = __ldg(xs + q4);
      } else {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) xr[q4] = make_uint4(0, 0, 0, 0);
      }
      if (a.signs) {
        const uint4* sp = reinterpret_cast<const uint4*>(a.signs + b * kBlock + lane * 32);
        sr[0] = __ldg(sp);
        sr[1] = __ldg(sp + 1);
      }
    };
    auto transform_block = [&](int it, const uint4 (&xr)[4], const uint4 (&sr)[2]) {
      const int tok = it / nchunk, b = it - tok * nchunk;
      // layout A: v[r] = element b*1024 + lane*32 + r
      float v[32];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const __half* h = reinterpret_cast<const __half*>(&xr[q4]);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[8 * q4 + e] = __half2float(h[e]);
      }
      if (a.signs) {
        const int8_t* sg = reinterpret_cast<const int8_t*>(sr);
#pragma unroll
        for (int r = 0; r < 32; ++r)
          if (sg[r] < 0) v[r] = -v[r];
      }
      if (a.rotate) {
        wht1024_a_shfl(v, lane);  // all ten stages, layout A kept
#pragma unroll
        for (int r = 0; r < 32; ++r) v[r] *= kInvSqrtBlock;
      }
      const int grp = b * (kBlock / kGroup) + (lane >> 2);
      float ssum = 0.f, csum = 0.f;
#pragma unroll
      for (int r = 0; r < 32; ++r) {
        v[r] = __half2float(__float2half_rn(v[r]));  // x' rounded to fp16
        ssum += v[r];
      }
#pragma unroll
      for (int mp = 0; mp < 4; ++mp) {
        uint32_t pk[4];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          const int p = 4 * (mp & 1) + e2;
          const int r = (mp >> 1) * 16 + p;
          const float is = inv_sigma_p(p);
          const __half lo_ = __float2half_rn(v[r] * is), hi_ = __float2half_rn(v[r + 8] * is);
          csum += __half2float(lo_) + __half2float(hi_);
          pk[e2] = (uint32_t)__half_as_ushort(lo_) | ((uint32_t)__half_as_ushort(hi_) << 16);
        }
        *reinterpret_cast<uint4*>(img + ((size_t)(grp * 4 + mp) * MT + tok) * 32 + t * 8) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      ssum += __shfl_xor_sync(0xffffffffu, ssum, 1);
      ssum += __shfl_xor_sync(0xffffffffu, ssum, 2);
      csum += __shfl_xor_sync(0xffffffffu, csum, 1);
      csum += __shfl_xor_sync(0xffffffffu, csum, 2);
      if (t == 0) cs[grp * MT + tok] = make_float2(1024.f * csum, ssum);
    };
    const int items = MT * nchunk;
    for (int it = warp; it < items; it += 2 * kTmaFwhtWarps) {
      const int it2 = it + kTmaFwhtWarps;
      uint4 xa[4], sa[2], xb[4], sb2[2];
      load_block(it, xa, sa);
      if (it2 < items) load_block(it2, xb, sb2);
      transform_block(it, xa, sa);
      if (it2 < items) transform_block(it2, xb, sb2);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kTmaConsumers * 32) : "memory");
    // zero the tile accumulators
    for (int i = threadIdx.x; i < (TS + 1) * kUnitRows * MT; i += kTmaConsumers * 32) accs[i] = 0.f;
    for (int i = threadIdx.x; i <= TS; i += kTmaConsumers * 32) cnt[i] = 0;
    asm volatile("bar.sync 1, %0;" ::"n"(kTmaConsumers * 32) : "memory");
  }

  // mma row g <-> unit row 32*wi + 16*j + rA (and + 8): conflict-free swizzled reads
  const int rA = 2 * (g & 3) + (g >> 2);
  const int tokc = g < MT ? g : 0;
  const uint32_t imgt = smem_u32(img) + tokc * 64 + t * 16;
  const uint32_t csa = smem_u32(cs);
  const uint32_t ss = smem_u32(smem + L.sstage) + warp * kScaleStageBytes;
  const uint32_t accs_u32 = smem_u32(accs);
  const int t0 = min(2 * t, MT - 1), t1 = min(2 * t + 1, MT - 1);

  for (int q = ug, n = 0; q < nst; q += kGroupsOfWarps, ++n) {
    // stage this unit's scales and biases, prefetch the ones two units ahead
    {
      const uint32_t r = ss + lane * kUnitGroups * 8;
      const __half2 sh0 = *reinterpret_cast<const __half2*>(&s0.x), sh1 = *reinterpret_cast<const __half2*>(&s0.y);
      const __half2 bh0 = *reinterpret_cast<const __half2*>(&b0.x), bh1 = *reinterpret_cast<const __half2*>(&b0.y);
      const float2 sf0 = __half22float2(sh0), sf1 = __half22float2(sh1);
      const float2 bf0 = __half22float2(bh0), bf1 = __half22float2(bh1);
      asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(r), "f"(sf0.x), "f"(bf0.x), "f"(sf0.y), "f"(bf0.y) : "memory");
      asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(r + 16), "f"(sf1.x), "f"(bf1.x), "f"(sf1.y), "f"(bf1.y) : "memory");
      s0 = s1;
      b0 = b1;
      load_sb(q + 2 * kGroupsOfWarps, s1, b1);
      __syncwarp();
    }
    const int slot = ug * DW + n % DW;
    wait(full + slot, (n / DW) & 1);
    const int64_t s = unit_of(q);
    const int tile = (int)(s / C), chunk = (int)(s - (int64_t)tile * C);
    const uint32_t box = codes_u32 + slot * kBoxBytes;
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int gi = 0; gi < kUnitGroups; ++gi)
      unit_group<MT>(box, 32 * wi + rA, t, gi, chunk * kUnitGroups + gi, imgt, ss, rA, csa, t0, t1, acc);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + slot);

    // add this warp's 32 rows into the tile's shared accumulator
    const int ts = slot_of(tile);
    const uint32_t atu = accs_u32 + ts * kUnitRows * MT * 4;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int ra = 32 * wi + 16 * j + rA, rb = ra + 8;
      if (2 * t < MT) {
        red_shared_add(atu + (ra * MT + 2 * t) * 4, acc[j][0]);
        red_shared_add(atu + (rb * MT + 2 * t) * 4, acc[j][2]);
      }
      if (2 * t + 1 < MT) {
        red_shared_add(atu + (ra * MT + 2 * t + 1) * 4, acc[j][1]);
        red_shared_add(atu + (rb * MT + 2 * t + 1) * 4, acc[j][3]);
      }
    }
    const int64_t t_beg = (int64_t)tile * C, t_end = t_beg + C;
    const int64_t c_beg = t_beg > lo ? t_beg : lo, c_end = t_end < hi ? t_end : hi;
    const int need = (int)(c_end - c_beg) * kWarpsPerUnit;
    __syncwarp();
    int last = 0;
    if (lane == 0) {
      __threadfence_block();
      last = atomicAdd(cnt + ts, 1) == need - 1;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) continue;

    // this warp finishes the tile for this CTA
    __threadfence_block();
    float* at = accs + ts * kUnitRows * MT;
    const int mi = mat_of(a, tile);
    const int N = a.N[mi], row0 = (tile - a.tile0[mi]) * kUnitRows;
    __half* yo = a.y[mi];
    const bool complete = t_beg >= lo && t_end <= hi;
    // a tile shared with other CTAs is summed in the workspace slot of its first CTA
    const int first = complete ? 0 : stage_owner(t_beg, S, gridDim.x);
    float* wsum = a.ws_partial + (int64_t)first * kUnitRows * MT;
    for (int e = lane; e < kUnitRows * MT; e += 32) {
      const float u = at[e];
      at[e] = 0.f;
      const int r_ = e / MT, k_ = e - r_ * MT;
      if (complete) {
        if (row0 + r_ < N && k_ < a.Mc) yo[(int64_t)k_ * N + row0 + r_] = __float2half_rn(u);
      } else {
        atomicAdd(wsum + e, u);
      }
    }
    __syncwarp();
    if (lane == 0) cnt[ts] = 0;
    __threadfence_block();
    if (complete) continue;
    // the last of the tile's CTAs converts the sum, then returns the slot and counter to zero
    const int lastc = stage_owner(t_end - 1, S, gridDim.x);
    int fin = 0;
    if (lane == 0) {
      __threadfence();
      fin = atomicAdd(a.ws_count + first, 1) == lastc - first;
    }
    fin = __shfl_sync(0xffffffffu, fin, 0);
    if (!fin) continue;
    __threadfence();
    for (int e = lane; e < kUnitRows * MT; e += 32) {
      const float v = __ldcg(wsum + e);
      wsum[e] = 0.f;
      const int r_ = e / MT, k_ = e - r_ * MT;
      if (row0 + r_ < N && k_ < a.Mc) yo[(int64_t)k_ * N + row0 + r_] = __float2half_rn(v);
    }
    if (lane == 0) a.ws_count[first] = 0;
  }
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// tensor map of one packed matrix's codes, cached by (pointer, shape)
static int code_map(const uint32_t* w, int64_t N, int64_t K, CUtensorMap* out) {
  struct Key {
    const void* w;
    int64_t N, K;
    bool operator==(const Key& o) const { return w == o.w && N == o.N && K == o.K; }
  };
  struct Hash {
    size_t operator()(const Key& k) const {
      return std::hash<const void*>()(k.w) ^ std::hash<int64_t>()(k.N * 131 + k.K);
    }
  };
  static std::mutex mu;
  static std::unordered_map<Key, CUtensorMap, Hash> cache;
  const Key key{w, N, K};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *out = it->second;
      return TB_OK;
    }
  }
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return TB_ERR_CUDA;
  CUtensorMap m;
  const cuuint64_t dims[2] = {(cuuint64_t)(K / 16), (cuuint64_t)N};
  const cuuint64_t strides[1] = {(cuuint64_t)(K / 4)};
  const cuuint32_t box[2] = {32, (cuuint32_t)kUnitRows};
  const cuuint32_t es[2] = {1, 1};
  if (enc(&m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, (void*)w, dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return TB_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (cache.size() > 4096) cache.clear();
    cache[key] = m;
  }
  *out = m;
  return TB_OK;
}

// workspace of the split (stream-K) schedule: fp32 sums [kFixupCtas][128][8] of tiles shared
// by several CTAs (indexed by the tile's first CTA), then counters [kFixupCtas]; both must
// be zero before a call and are zero after it
constexpr int kFixupCtas = 256;
constexpr size_t kFixupPartialBytes = (size_t)kFixupCtas * kUnitRows * 8 * 4;
size_t gemv_fixup_bytes() { return kFixupPartialBytes + kFixupCtas * 4; }

template <int MT>
static int launch_tma_mt(GemvTmaArgs a, const CodeMaps& maps, int64_t M, int64_t K,
                         const DeviceFacts& f, cudaStream_t s) {
  // slots per unit group from what is left of shared memory
  int dw = kMaxSlotsPerGroup;
  auto ts_for = [&](int d) { return kGroupsOfWarps * d / a.C + 3; };
  while (dw >= 1 && gemv_tma_layout<MT>(a.G, dw, ts_for(dw)).total > f.smem_optin) --dw;
  if (dw < 1) return TB_ERR_SHAPE;
  a.dw = dw;
  a.tslots = ts_for(dw);
  const int bytes = gemv_tma_layout<MT>(a.G, dw, a.tslots).total;
  cudaError_t e = cudaFuncSetAttribute(w2_gemv_tma_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return TB_ERR_CUDA;
  }
  const int64_t S = (int64_t)a.n_tiles * a.C;
  int grid = f.sms;
  if (!a.split && a.n_tiles < grid) grid = a.n_tiles;
  if (S < grid) grid = (int)S;
  const __half* x0 = a.x;
  __half* y0[kMaxMats];
  for (int i = 0; i < a.nmat; ++i) y0[i] = a.y[i];
  for (int64_t m0 = 0; m0 < M; m0 += MT) {
    a.x = x0 + m0 * K;
    for (int i = 0; i < a.nmat; ++i) a.y[i] = y0[i] + m0 * a.N[i];
    a.Mc = (int)((M - m0) < MT ? (M - m0) : MT);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTmaThreads);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, w2_gemv_tma_kernel<MT>, maps, a);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      return TB_ERR_CUDA;
    }
  }
  return TB_OK;
}

// tokens per pass: the largest of 8, 4, 2, 1 (not above M rounded up) whose B image leaves
// room for two slots per unit group
static int tma_tokens_per_pass(int64_t M, int G, int C, int smem_optin) {
  int mt = M >= 5 ? 8 : M >= 3 ? 4 : M == 2 ? 2 : 1;
  auto fits = [&](int total) { return total <= smem_optin; };
  while (mt > 1) {
    const int ts = kGroupsOfWarps * 2 / C + 3;
    const bool ok = mt == 8 ? fits(gemv_tma_layout<8>(G, 2, ts).total)
                  : mt == 4 ? fits(gemv_tma_layout<4>(G, 2, ts).total)
                            : fits(gemv_tma_layout<2>(G, 2, ts).total);
    if (ok) break;
    mt >>= 1;
  }
  return mt;
}

// One launch for up to kMaxMats packed matrices that read the same x (their row tiles are
// concatenated; the rotated x' is computed once per CTA for all of them).
int launch_gemv_tma_multi(const __half* x, int64_t M, int64_t K, const int8_t* signs, int block,
                          int nmat, const uint32_t* const* w, const __half* const* scales,
                          const __half* const* biases, const int64_t* N, __half* const* y,
                          void* workspace, size_t ws_bytes, int32_t* status, cudaStream_t s) {
  DeviceFacts f;
  int rc = device_facts(&f);
  if (rc != TB_OK) return rc;
  if (nmat < 1 || nmat > kMaxMats) return TB_ERR_SHAPE;
  if (K > (1 << 22) || K % kBlock) return TB_ERR_SHAPE;
  GemvTmaArgs a = {};
  CodeMaps maps;
  int tiles = 0;
  for (int i = 0; i < nmat; ++i) {
    if (N[i] < 1 || N[i] > (1LL << 30)) return TB_ERR_SHAPE;
    rc = code_map(w[i], N[i], K, &maps.m[i]);
    if (rc != TB_OK) return rc;
    a.scales[i] = scales[i];
    a.biases[i] = biases[i];
    a.y[i] = y[i];
    a.N[i] = (int)N[i];
    a.tile0[i] = tiles;
    tiles += (int)((N[i] + kUnitRows - 1) / kUnitRows);
  }
  for (int i = nmat; i <= kMaxMats; ++i) a.tile0[i] = tiles;
  for (int i = nmat; i < kMaxMats; ++i) maps.m[i] = maps.m[0];
  a.nmat = nmat;
  a.x = x;
  a.signs = signs;
  const bool split = workspace && ws_bytes >= gemv_fixup_bytes() && f.sms <= kFixupCtas;
  a.ws_partial = split ? static_cast<float*>(workspace) : nullptr;
  a.ws_count = split ? reinterpret_cast<int*>(static_cast<char*>(workspace) + kFixupPartialBytes)
                     : nullptr;
  a.split = split ? 1 : 0;
  a.K = (int)K;
  a.G = (int)(K / kGroup);
  a.C = (int)(K / (kUnitGroups * kGroup));
  a.rotate = block != 0;
  a.n_tiles = tiles;
  a.status = status;
  const int mt = tma_tokens_per_pass(M, a.G, a.C, f.smem_optin);
  switch (mt) {
    case 8: return launch_tma_mt<8>(a, maps, M, K, f, s);
    case 4: return launch_tma_mt<4>(a, maps, M, K, f, s);
    case 2: return launch_tma_mt<2>(a, maps, M, K, f, s);
    default: return launch_tma_mt<1>(a, maps, M, K, f, s);
  }
}

int launch_gemv_tma(const __half* x, int64_t M, int64_t K, const int8_t* signs, int block,
                    const uint32_t* w, const __half* scales, const __half* biases, int64_t N,
                    __half* y, void* workspace, size_t ws_bytes, int32_t* status, cudaStream_t s) {
  return launch_gemv_tma_multi(x, M, K, signs, block, 1, &w, &scales, &biases, &N, &y, workspace,
                               ws_bytes, status, s);
}

}  // namespace tb
