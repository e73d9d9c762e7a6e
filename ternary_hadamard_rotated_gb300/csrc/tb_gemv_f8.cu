// Decode path of the Packed layer on the fifth-generation tensor cores (tcgen05): the W2-g128
// codes become e4m3 operands in tensor memory, the rotated activations three e4m3 terms in
// shared memory, and the multiply-adds run as tcgen05.mma with fp32 accumulators.
//
// [ARCH] kwkr.cn/news/564617, section "Hadamard 旋转把量化误差抹平的免费午餐": a folded module
// rotates its input by the signed block Hadamard transform (scale 1/sqrt(1024)) and multiplies it
// by the packed 2-bit, group-128 affine weights, which are never expanded to an fp16 matrix;
// section "打包格式的工程MLX 2.25 bits 与 GGUF 的两种装箱": codes {0,1,2} in uint32 words, one
// fp16 scale and one fp16 bias per 128 weights, a code decoding to s*q + b.
//
// Operands (M <= 2 tokens, one pass):
//  * A, tensor memory, 128 rows (= lanes) x 512 k per unit.  A packed word w (codes 0..15 at
//    bits 2i..2i+1) becomes four 32-bit columns, each four e4m3 bytes:
//      w & 0x03030303, w & 0x0C0C0C0C, (w >> 4) & 0x03030303, (w >> 4) & 0x0C0C0C0C.
//    A 2-bit field in bits 0-1 of a byte is the subnormal q * 2^-9; in bits 2-3 it is q * 2^-7
//    (q = 1 sets the top mantissa bit, q = 2 the lowest exponent bit, q = 3 both: 2^-7, 2^-6,
//    1.5 * 2^-6).  Both are linear in q and exact, so no offset or magic constant is needed:
//    one shift and four ANDs per 16 codes.  Byte b of column i of word j holds code 4b + i, so
//    the MMA's k order inside each 16 codes is the 4 x 4 transpose of the natural one.
//  * B, shared memory, K-major with the 128-byte swizzle, one 1 KB atom (8 rows x 128 k) per
//    group of 128 k: x' scaled by 2^(9-E) where the code sits in bits 0-1 and by 2^(7-E) where
//    it sits in bits 2-3 (E per group and token, so every value is below 256), split into three
//    e4m3 terms h + m/16 + l/256 that hold the fp16 value exactly (rows 3t, 3t+1, 3t+2 of
//    token t; the values below 2^-14 of the group's largest lose their last bits).
//  * D, tensor memory, fp32: 16 columns per group (N = 16, the MMA's smallest at M = 128).
//    sum_k q x' = 2^E (D[3t] + D[3t+1]/16 + D[3t+2]/256), then y += s * that + b * S with
//    S = sum x' over the group.  Rows 8..15 of B read the next atom: those D columns are unused.
//
// Roles (one CTA of ten warps per SM): warp 0 streams 16 KB boxes of packed codes (128 rows x
// 512 k) into a six-slot TMA ring; warps 2..9 form two decoder warpgroups, each walking a
// contiguous half of the CTA's stream-K unit range (the second one backwards, so that the tiles
// shared with both neighbouring CTAs are finished first).  Per group of 128 k a warpgroup loads
// its rows' 8 words per thread from the box, decodes them, stores 32 columns of A into one of six
// tensor-memory slots and signals an mbarrier; warp 1 issues the group's four MMAs into one of
// four accumulators and commits them to the slot's and the accumulator's mbarriers; the
// warpgroup reads the accumulator three groups later.  No step waits on a CTA-wide barrier.
#include <cuda.h>
#include <cuda_fp8.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <vector>

#include "tb_common.cuh"
#include "tb_gemv_core.cuh"
#include "tb_host.h"
#include "tb_tcgen05.cuh"

namespace tb {

int code_map(const uint32_t* w, int64_t N, int64_t K, CUtensorMap* out);
size_t gemv_fixup_bytes();

constexpr int kF8ConsumerWarps = 8;                     // two decoder warpgroups
constexpr int kF8Threads = (kF8ConsumerWarps + 2) * 32;  // + the producer and the MMA warp
constexpr int kF8Ring = 6;                              // 16 KB code boxes in flight per CTA
constexpr int kF8MaxBlocks = 6;                         // 1024-blocks of x' one CTA's image holds
constexpr int kF8RA = 6;                                // A slots (32 columns, one group) per warpgroup
constexpr int kF8RD = 4;                                // accumulators (16 columns) per warpgroup
constexpr int kF8Lag = 3;                               // groups between a group's MMAs and its epilogue
constexpr int kF8TmemCols = 512;                        // 2 warpgroups x (6 x 32 + 4 x 16)
constexpr int kF8CutSlots = 3;                          // tiles cut by the lo / mid / hi boundaries
constexpr int kF8PartStride = kUnitRows * 8;            // floats per workspace part slot
static_assert(kF8Lag < kUnitGroups && kF8Lag < kF8RD, "epilogue lag");
static_assert(2 * (32 * kF8RA + 16 * kF8RD) <= kF8TmemCols, "tensor memory");
// tcgen05 instruction descriptor: fp32 D, e4m3 A and B (both K-major), N = 16, M = 128
constexpr uint32_t kF8Idesc = (1u << 4) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

struct F8Args {
  const __half* x;                 // [Mc, K]
  const int8_t* signs;             // [K] or null
  const __half* scales[kMaxMats];  // [N_i, G]
  const __half* biases[kMaxMats];  // [N_i, G] or null (each bias -s)
  __half* y[kMaxMats];             // [Mc, N_i]
  int N[kMaxMats];
  int tile0[kMaxMats + 1];         // first 128-row tile of matrix i in the concatenated list
  int nmat;
  float* ws_partial;               // [grid][2][128 * 8] fp32 parts of tiles shared between CTAs
  int* ws_count;                   // [grid] contributions per shared tile (zero before and after)
  int Mc, K, G, C, rotate, n_tiles, split, nblk_max;
  int32_t* status;
};

struct F8Maps {
  CUtensorMap codes[kMaxMats];  // uint32 [N][K/16], box 32 x 128, 128-byte swizzle
};

struct F8Layout {
  int ring, img, cg, accs, cnt, bars, tslot, total;
};

template <int MT>
__host__ __device__ inline F8Layout f8_layout(int nblk) {
  F8Layout L;
  int off = 0;
  L.ring = off;  // 1024-aligned boxes (the swizzle pattern repeats every 1024 bytes)
  off += kF8Ring * kSlotBytes;
  L.img = off;  // one 1 KB atom per group of 128 k, plus the atom rows 8..15 of the last read
  off += (nblk * 8 + 1) * 1024;
  L.cg = off;  // per group and token: (S = sum x', 2^E)
  off += nblk * 8 * MT * 8;
  L.accs = off;
  off += kF8CutSlots * kUnitRows * MT * 4;
  L.cnt = off;
  off += 16;
  L.bars = off;
  off += (2 * kF8Ring + 4 * kF8RA + 4 * kF8RD) * 8;
  L.tslot = off;
  off += 16;
  L.total = off + 1024;  // slack to align the base to 1024
  return L;
}

// 1024-blocks of x that the units [lo, lo + nst) read: [b1, e1) and [b2, e2) (host and device)
__host__ __device__ inline void f8_blocks_needed(int lo, int nst, int C, int K, int& b1, int& e1, int& b2,
                                                 int& e2) {
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

// this CTA's unit range [lo, hi)
__host__ __device__ inline void f8_cta_range(int c, int grid, int n_tiles, int C, int split, int& lo, int& hi) {
  if (split) {
    const int64_t S = (int64_t)n_tiles * C;
    lo = (int)(S * c / grid);
    hi = (int)(S * (c + 1) / grid);
  } else {
    lo = C * (int)((int64_t)n_tiles * c / grid);
    hi = C * (int)((int64_t)n_tiles * (c + 1) / grid);
  }
}

TB_DEVI int f8_mat_of(const F8Args& a, int tile) {
  int i = 0;
#pragma unroll
  for (int k = 1; k < kMaxMats; ++k) i += (k < a.nmat && tile >= a.tile0[k]);
  return i;
}

// the eight decoder warps' named barrier (an immediate id: the kernel uses two barriers)
TB_DEVI void bar_consumers() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
TB_DEVI void f8_sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

TB_DEVI uint16_t to_e4m3x2(__half2 v) {
  __half2_raw r = static_cast<__half2_raw>(v);
  return (uint16_t)__nv_cvt_halfraw2_to_fp8x2(r, __NV_SATFINITE, __NV_E4M3);
}
TB_DEVI __half2 from_e4m3x2(uint16_t v) {
  return static_cast<__half2>(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3));
}

// One 16-byte chunk of a B row: e[0..15] as e4m3 pairs T[p] = (e[2p], e[2p+1]); byte 4i + b of
// the chunk is e[4b + i] (the A columns' k order).
TB_DEVI void store_b_chunk(uint32_t addr, const uint16_t (&T)[8]) {
  const uint32_t lo0 = (uint32_t)T[0] | ((uint32_t)T[2] << 16), hi0 = (uint32_t)T[4] | ((uint32_t)T[6] << 16);
  const uint32_t lo1 = (uint32_t)T[1] | ((uint32_t)T[3] << 16), hi1 = (uint32_t)T[5] | ((uint32_t)T[7] << 16);
  f8_sts128(addr, __byte_perm(lo0, hi0, 0x6420), __byte_perm(lo0, hi0, 0x7531), __byte_perm(lo1, hi1, 0x6420),
         __byte_perm(lo1, hi1, 0x7531));
}

template <int MT>
__global__ void __launch_bounds__(kF8Threads, 1)
    w2_gemv_f8_kernel(const __grid_constant__ F8Maps maps, const __grid_constant__ F8Args a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int C = a.C, K = a.K, G = a.G;
  const F8Layout L = f8_layout<MT>(a.nblk_max);
  const uint32_t ring = smem_u32(smem + L.ring);
  const uint32_t img = smem_u32(smem + L.img);
  float2* cg = reinterpret_cast<float2*>(smem + L.cg);
  float* accs = reinterpret_cast<float*>(smem + L.accs);  // [kF8CutSlots][128][MT]
  int* cnt = reinterpret_cast<int*>(smem + L.cnt);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kF8Ring;
  // per warpgroup: A slots written (afull) / read by the MMAs (aempty); accumulators written by
  // the MMAs (dfull) / read by the epilogue (dempty)
  uint64_t* afull = empty + kF8Ring;
  uint64_t* aempty = afull + 2 * kF8RA;
  uint64_t* dfull = aempty + 2 * kF8RA;
  uint64_t* dempty = dfull + 2 * kF8RD;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + L.tslot);
  __shared__ volatile int aborted;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int S = a.n_tiles * C;
  int lo, hi;
  f8_cta_range(blockIdx.x, gridDim.x, a.n_tiles, C, a.split, lo, hi);
  const int nst = hi - lo, mid = lo + nst / 2;
  const int cnt0 = mid - lo, cnt1 = hi - mid, mboth = cnt0 < cnt1 ? cnt0 : cnt1;
  int b1, e1, b2, e2;  // the 1024-blocks of x this CTA's units read
  f8_blocks_needed(lo, nst, C, K, b1, e1, b2, e2);
  const int nblk = (e1 - b1) + (e2 - b2);
  auto img_group = [&](int gglob) {  // image atom of global group gglob (128 k)
    const int blk = gglob >> 3;
    const int bpos = (blk >= b1 && blk < e1) ? blk - b1 : (e1 - b1) + (blk - b2);
    return bpos * 8 + (gglob & 7);
  };

  if (threadIdx.x == 0) {
    aborted = 0;
    for (int i = 0; i < kF8Ring; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, 4);  // the four warps of the warpgroup that owns the box
    }
    for (int i = 0; i < 2 * kF8RA; ++i) {
      mbar_init(afull + i, 4);  // one arrival per warp of the warpgroup
      mbar_init(aempty + i, 1);  // one commit
    }
    for (int i = 0; i < 2 * kF8RD; ++i) {
      mbar_init(dfull + i, 1);
      mbar_init(dempty + i, 4);
    }
    fence_barrier_init();
  }
  for (int i = threadIdx.x; i < kF8CutSlots * kUnitRows * MT; i += blockDim.x) accs[i] = 0.f;
  if (threadIdx.x < kF8CutSlots) cnt[threadIdx.x] = 0;
  if (warp == 1) tmem_alloc(tslot, kF8TmemCols);
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tmem = *tslot;

  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (aborted) return;
    if (!mbar_wait(bar, parity)) {
      aborted = 1;
      set_status(a.status, TB_DEV_TIMEOUT);
    }
  };

  if (warp == 0) {
    // ---- producer: boxes of both warpgroups interleaved (the weights never depend on the
    // previous kernel, so this streams before griddepcontrol.wait)
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const int total = cnt0 + cnt1;
      for (int f = 0; f < total; ++f) {
        int u, n;
        if (f < 2 * mboth) {
          u = f & 1;
          n = f >> 1;
        } else {
          u = cnt0 > cnt1 ? 0 : 1;
          n = f - mboth;
        }
        const int unit = u == 0 ? lo + n : hi - 1 - n;
        const int tile = unit / C, chunk = unit - tile * C;
        const int slot = f % kF8Ring, k = f / kF8Ring;
        if (k > 0) wait(empty + slot, (k - 1) & 1);
        const int mi = f8_mat_of(a, tile);
        const int row = (tile - a.tile0[mi]) * kUnitRows;
        mbar_arrive_expect_tx(full + slot, kSlotBytes);
        tma2d(ring + slot * kSlotBytes, &maps.codes[mi], chunk * 32, row, full + slot, pol);
      }
      // leave no copy in flight: wait (bounded, even after a timeout) for the last fill of each slot
      for (int f = total - 1; f >= 0 && f >= total - kF8Ring; --f)
        if (!mbar_wait(full + f % kF8Ring, (f / kF8Ring) & 1)) set_status(a.status, TB_DEV_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issuer: the two warpgroups' groups in lockstep, four MMAs per group of 128 k
    if (lane == 0) {
      const int n4[2] = {4 * cnt0, 4 * cnt1};
      const int nmax = n4[0] > n4[1] ? n4[0] : n4[1];
      for (int i = 0; i < nmax; ++i) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          if (i >= n4[u]) continue;
          const int sa = i % kF8RA, sd = i % kF8RD;
          wait(afull + u * kF8RA + sa, (i / kF8RA) & 1);
          if (i >= kF8RD) wait(dempty + u * kF8RD + sd, ((i / kF8RD) - 1) & 1);
          tmem_fence_after();
          const int n = i >> 2;
          const int unit = u == 0 ? lo + n : hi - 1 - n;
          const int chunk = unit % C;
          const uint32_t atom = img + (uint32_t)img_group(chunk * kUnitGroups + (i & 3)) * 1024u;
          const uint32_t tA = tmem + (uint32_t)(u * 256 + 32 * sa);
          const uint32_t tD = tmem + (uint32_t)(u * 256 + 32 * kF8RA + 16 * sd);
#pragma unroll
          for (int m = 0; m < 4; ++m)
            mma_f8f6f4_ts(tD, tA + (uint32_t)(8 * m), smem_desc_sw128(atom + 32u * m, 1024u), kF8Idesc, m > 0);
          mma_commit(aempty + u * kF8RA + sa);
          mma_commit(dfull + u * kF8RD + sd);
        }
      }
      // every MMA issued has completed before the columns are given back
#pragma unroll
      for (int u = 0; u < 2; ++u)
        if (n4[u] > 0 && !mbar_wait(dfull + u * kF8RD + (n4[u] - 1) % kF8RD, ((n4[u] - 1) / kF8RD) & 1))
          set_status(a.status, TB_DEV_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ---- decoders: warpgroup u; thread r of it = unit row r = tensor-memory lane r
    const int dw = warp - 2;
    const int u = dw >> 2, q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const uint32_t tAu = tmem + (uint32_t)(u * 256), tDu = tAu + 32 * kF8RA;
    const int glo = u == 0 ? lo : mid, ghi = u == 0 ? mid : hi;
    const int ncnt = ghi - glo;
    const bool back = u == 1;
    uint64_t* afu = afull + u * kF8RA;
    uint64_t* aeu = aempty + u * kF8RA;
    uint64_t* dfu = dfull + u * kF8RD;
    uint64_t* deu = dempty + u * kF8RD;

    // scale and bias words of unit n for this row (8 bytes each: the unit's four groups)
    auto load_sb = [&](int n, uint2& sv, uint2& bv) {
      sv = make_uint2(0, 0);
      bv = make_uint2(0, 0);
      if (n >= ncnt) return;
      const int unit = back ? ghi - 1 - n : glo + n;
      const int tile = unit / C, chunk = unit - tile * C;
      const int mi = f8_mat_of(a, tile);
      const int row = (tile - a.tile0[mi]) * kUnitRows + r;
      if (row >= a.N[mi]) return;
      const __half* sp = a.scales[mi] + (int64_t)row * G + chunk * kUnitGroups;
      sv = __ldg(reinterpret_cast<const uint2*>(sp));
      const __half* bp = a.biases[mi];
      // no biases given: each is the pack's -scale (the fp16 sign bit flipped), not read
      bv = bp ? __ldg(reinterpret_cast<const uint2*>(bp + (int64_t)row * G + chunk * kUnitGroups))
              : make_uint2(sv.x ^ 0x80008000u, sv.y ^ 0x80008000u);
    };
    // units n - 1, n, n + 1 at the top of iteration n
    uint2 sv0 = make_uint2(0, 0), bv0 = make_uint2(0, 0), sv1 = make_uint2(0, 0), bv1 = make_uint2(0, 0), sv2, bv2;
    load_sb(0, sv2, bv2);
    if (a.signs) {  // the signs never depend on the previous kernel: into L1 before the wait
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        const int it = dw + qq * kF8ConsumerWarps;
        if (it < 2 * nblk) {
          const int bi = it >> 1;
          const int b = bi < e1 - b1 ? b1 + bi : b2 + (bi - (e1 - b1));
          asm volatile("prefetch.global.L1 [%0];" ::"l"(a.signs + b * kBlock + (it & 1) * 512 + lane * 16));
        }
      }
    }

    asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---- prologue: x' = fwht(signs * x) rounded to fp16, as the B image and (S, 2^E) per group.
    // An item is one half of a (token, block) pair: outputs 0..511 of H1024 are H512 (x_lo + x_hi),
    // outputs 512..1023 are H512 (x_lo - x_hi); lane l holds elements 16 l .. 16 l + 15 of both
    // input halves and of its output half, i.e. chunk l % 8 of group 4 hh + l / 8 of the block.
    {
      const int items = 2 * MT * nblk;
      auto item_of = [&](int it, int& tok, int& bi, int& b, int& hh) {
        hh = it & 1;
        const int rest = it >> 1;
        tok = rest / nblk;
        bi = rest - tok * nblk;
        b = bi < e1 - b1 ? b1 + bi : b2 + (bi - (e1 - b1));
      };
      auto load_item = [&](int it, uint4 (&xr)[4], uint4 (&sr)[2]) {
        int tok, bi, b, hh;
        item_of(it, tok, bi, b, hh);
        if (tok < a.Mc) {
          const uint4* xs = reinterpret_cast<const uint4*>(a.x + (int64_t)tok * K + b * kBlock + lane * 16);
          xr[0] = __ldg(xs);
          xr[1] = __ldg(xs + 1);
          xr[2] = __ldg(xs + kBlock / 16);  // the same elements of the upper half
          xr[3] = __ldg(xs + kBlock / 16 + 1);
        } else {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) xr[q4] = make_uint4(0, 0, 0, 0);
        }
        if (a.signs) {
          const uint4* sp = reinterpret_cast<const uint4*>(a.signs + b * kBlock + lane * 16);
          sr[0] = __ldg(sp);
          sr[1] = __ldg(sp + kBlock / 32);
        }
      };
      auto do_item = [&](int it, const uint4 (&xr)[4], const uint4 (&sr)[2]) {
        int tok, bi, b, hh;
        item_of(it, tok, bi, b, hh);
        float v[16];
        {
          const __half* xl = reinterpret_cast<const __half*>(&xr[0]);
          const __half* xh = reinterpret_cast<const __half*>(&xr[2]);
          const int8_t* sl = reinterpret_cast<const int8_t*>(&sr[0]);
          const int8_t* sh = reinterpret_cast<const int8_t*>(&sr[1]);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float lo_ = __half2float(xl[e]), hi_ = __half2float(xh[e]);
            if (a.signs) {
              if (sl[e] < 0) lo_ = -lo_;
              if (sh[e] < 0) hi_ = -hi_;
            }
            v[e] = a.rotate ? (hh ? lo_ - hi_ : lo_ + hi_) : (hh ? hi_ : lo_);
          }
        }
        if (a.rotate) {
          wht512_a_shfl(v, lane);  // the other nine stages; lane l keeps elements 16 l ..
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] *= kInvSqrtBlock;
        }
        float ssum = 0.f, amax = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          v[e] = __half2float(__float2half_rn(v[e]));  // x' rounded to fp16
          ssum += v[e];
          amax = fmaxf(amax, fabsf(v[e]));
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {  // the eight lanes of one group of 128
          ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        }
        // E: 2^(E-2) <= amax < 2^(E-1), so x' * 2^(9-E) and x' * 2^(7-E) stay below 256
        const int E = amax > 0.f ? (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127 + 2 : 0;
        const float se = __uint_as_float((uint32_t)(127 + 9 - E) << 23);
        const float so = __uint_as_float((uint32_t)(127 + 7 - E) << 23);
        uint16_t th[8], tm[8], tl[8];
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const __half2 v2 = __floats2half2_rn(v[2 * p] * se, v[2 * p + 1] * so);  // exact (power of 2)
          th[p] = to_e4m3x2(v2);
          const __half2 r16 = __hmul2(__hsub2(v2, from_e4m3x2(th[p])), __float2half2_rn(16.f));
          tm[p] = to_e4m3x2(r16);
          const __half2 r256 = __hmul2(__hsub2(r16, from_e4m3x2(tm[p])), __float2half2_rn(16.f));
          tl[p] = to_e4m3x2(r256);
        }
        const int ig = bi * 8 + 4 * hh + (lane >> 3), j = lane & 7;
        const uint32_t atom = img + (uint32_t)ig * 1024u;
        const int row0 = 3 * tok;
        store_b_chunk(atom + (row0 + 0) * 128 + ((j ^ (row0 + 0)) << 4), th);
        store_b_chunk(atom + (row0 + 1) * 128 + ((j ^ (row0 + 1)) << 4), tm);
        store_b_chunk(atom + (row0 + 2) * 128 + ((j ^ (row0 + 2)) << 4), tl);
        if ((lane & 7) == 0) cg[ig * MT + tok] = make_float2(ssum, __uint_as_float((uint32_t)(127 + E) << 23));
      };
      for (int it = dw; it < items; it += 2 * kF8ConsumerWarps) {
        const int it2 = it + kF8ConsumerWarps;
        uint4 xa[4], sa[2], xb[4], sb2[2];
        load_item(it, xa, sa);
        if (it2 < items) load_item(it2, xb, sb2);
        do_item(it, xa, sa);
        if (it2 < items) do_item(it2, xb, sb2);
      }
      fence_proxy_async_smem();  // the image (generic writes) before the tensor core reads it
      bar_consumers();
    }

    // Add this thread's sums of tile T (all of the warpgroup's units of T) to wherever T is finished.
    float acc[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) acc[t] = 0.f;
    auto flush = [&](int T) {
      const int mi = f8_mat_of(a, T);
      const int N = a.N[mi], row0 = (T - a.tile0[mi]) * kUnitRows;
      __half* yo = a.y[mi];
      const int tb_ = T * C, te = tb_ + C;
      if (tb_ >= glo && te <= ghi) {  // the whole tile is this warpgroup's: this row is final
        if (row0 + r < N)
#pragma unroll
          for (int t = 0; t < MT; ++t)
            if (t < a.Mc) yo[(int64_t)t * N + row0 + r] = __float2half_rn(acc[t]);
        return;
      }
      // a tile cut by a boundary: its shared slot is the first boundary that falls in it
      const int b = (lo / C == T) ? 0 : (mid / C == T) ? 1 : 2;
      const int groups = (cnt0 > 0 && lo < te && mid > tb_) + (cnt1 > 0 && mid < te && hi > tb_);
      const uint32_t at_u32 = smem_u32(accs) + (uint32_t)(b * kUnitRows * MT) * 4u;
#pragma unroll
      for (int t = 0; t < MT; ++t) red_shared_add(at_u32 + (uint32_t)(r * MT + t) * 4u, acc[t]);
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        __threadfence_block();
        last = atomicAdd(cnt + b, 1) == groups * 4 - 1;
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (!last) return;
      __threadfence_block();  // this warp finishes the tile for this CTA
      float* at = accs + b * kUnitRows * MT;
      if (tb_ >= lo && te <= hi) {
        for (int e = lane; e < kUnitRows * MT; e += 32) {
          const int r_ = e / MT, k_ = e - r_ * MT;
          if (row0 + r_ < N && k_ < a.Mc) yo[(int64_t)k_ * N + row0 + r_] = __float2half_rn(at[e]);
        }
        return;
      }
      // shared with other CTAs: this CTA's part to its own workspace slot (0 for the tile of its
      // first unit, 1 for the tile of its last)
      float* mine = a.ws_partial + ((int64_t)blockIdx.x * 2 + (lo / C == T ? 0 : 1)) * kF8PartStride;
      for (int e = lane; e < kUnitRows * MT; e += 32) __stcg(mine + e, at[e]);
      __syncwarp();
      // the last of the tile's CTAs to count in adds the parts in CTA order (the result does not
      // depend on which CTA finishes last) and returns the counter to zero
      const int first = stage_owner(tb_, S, gridDim.x);
      const int lastc = stage_owner(te - 1, S, gridDim.x);
      int fin = 0;
      if (lane == 0) {
        fence_acq_rel_gpu();  // the warp's part before the count
        fin = atomicAdd(a.ws_count + first, 1) == lastc - first;
      }
      fin = __shfl_sync(0xffffffffu, fin, 0);
      if (!fin) return;
      fence_acq_rel_gpu();  // every contributor's part after the count
      int flo, fhi;
      f8_cta_range(first, gridDim.x, a.n_tiles, C, a.split, flo, fhi);
      const float* p0 = a.ws_partial + ((int64_t)first * 2 + (flo / C == T ? 0 : 1)) * kF8PartStride;
      for (int eb = 0; eb < kUnitRows * MT; eb += 128) {  // four elements per lane per pass
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        for (int c = first; c <= lastc; c += 4) {  // four contributors' loads in flight at once
          float l[4][4];
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const int cc = c + qq;
            const float* pc = cc == first ? p0 : a.ws_partial + (int64_t)cc * 2 * kF8PartStride;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int e = eb + lane + 32 * k;
              l[qq][k] = (cc <= lastc && e < kUnitRows * MT) ? __ldcg(pc + e) : 0.f;
            }
          }
#pragma unroll
          for (int qq = 0; qq < 4; ++qq)
#pragma unroll
            for (int k = 0; k < 4; ++k) v[k] += l[qq][k];
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int e = eb + lane + 32 * k;
          if (e >= kUnitRows * MT) continue;
          const int r_ = e / MT, k_ = e - r_ * MT;
          if (row0 + r_ < N && k_ < a.Mc) yo[(int64_t)k_ * N + row0 + r_] = __float2half_rn(v[k]);
        }
      }
      if (lane == 0) a.ws_count[first] = 0;
    };

    // Epilogue of group j of this warpgroup (group gg of a unit with chunk `chunk`): its
    // accumulator, then y += s * 2^E (D0 + D1/16 + D2/256) + b * S
    constexpr int kDc = MT == 1 ? 4 : 8;  // accumulator columns read
    auto epilogue = [&](int j, int chunk, int gg, uint2 sv, uint2 bv) {
      const int sd = j % kF8RD;
      wait(dfu + sd, (j / kF8RD) & 1);
      tmem_fence_after();
      float d[kDc];
      if constexpr (MT == 1) tmem_ld4(tDu + (uint32_t)(16 * sd) + lane_off, d);
      else tmem_ld8(tDu + (uint32_t)(16 * sd) + lane_off, d);
      tmem_wait_ld();
      tmem_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(deu + sd);
      const uint32_t sw = gg < 2 ? sv.x : sv.y, bw = gg < 2 ? bv.x : bv.y;
      const float s = __half2float(__ushort_as_half((unsigned short)((gg & 1) ? sw >> 16 : sw & 0xFFFFu)));
      const float bb = __half2float(__ushort_as_half((unsigned short)((gg & 1) ? bw >> 16 : bw & 0xFFFFu)));
      const float2* c2 = cg + img_group(chunk * kUnitGroups + gg) * MT;
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        const float2 cs = c2[t];
        const float dq = fmaf(d[3 * t + 2], 0.00390625f, fmaf(d[3 * t + 1], 0.0625f, d[3 * t])) * cs.y;
        acc[t] = fmaf(s, dq, fmaf(bb, cs.x, acc[t]));
      }
    };

    const int rsw = r & 7;
    int ptile = 0, pchunk = 0;  // unit n - 1
    for (int n = 0; n < ncnt; ++n) {
      const int unit = back ? ghi - 1 - n : glo + n;
      const int tile = unit / C, chunk = unit - tile * C;
      const int f = n < mboth ? 2 * n + u : mboth + n;
      const int slot = f % kF8Ring;
      sv0 = sv1;
      bv0 = bv1;
      sv1 = sv2;
      bv1 = bv2;
      load_sb(n + 1, sv2, bv2);
      wait(full + slot, (f / kF8Ring) & 1);
      const uint32_t box = ring + (uint32_t)slot * kSlotBytes + (uint32_t)r * 128u;
#pragma unroll
      for (int g = 0; g < kUnitGroups; ++g) {
        const int i = 4 * n + g;
        const uint4 wa = ld_shared_v4(box + ((uint32_t)((2 * g) ^ rsw) << 4));
        const uint4 wb = ld_shared_v4(box + ((uint32_t)((2 * g + 1) ^ rsw) << 4));
        uint32_t A[32];
        const uint32_t wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const uint32_t w4 = wv[jj] >> 4;
          A[4 * jj + 0] = wv[jj] & 0x03030303u;  // codes 0, 4, 8, 12:  q * 2^-9
          A[4 * jj + 1] = wv[jj] & 0x0C0C0C0Cu;  // codes 1, 5, 9, 13:  q * 2^-7
          A[4 * jj + 2] = w4 & 0x03030303u;      // codes 2, 6, 10, 14: q * 2^-9
          A[4 * jj + 3] = w4 & 0x0C0C0C0Cu;      // codes 3, 7, 11, 15: q * 2^-7
        }
        if (g == kUnitGroups - 1) {  // the box is read: the producer may refill it
          __syncwarp();
          if (lane == 0) mbar_arrive(empty + slot);
        }
        const int sa = i % kF8RA;
        if (i >= kF8RA) wait(aeu + sa, ((i / kF8RA) - 1) & 1);  // the MMAs that read it are done
        tmem_fence_after();
        tmem_st32(tAu + (uint32_t)(32 * sa) + lane_off, A);
        tmem_wait_st();
        tmem_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(afu + sa);
        // the epilogue runs kF8Lag groups behind: groups 1..3 of unit n - 1, then group 0 of n
        if (i >= kF8Lag) {
          if (g < kF8Lag) {
            epilogue(i - kF8Lag, pchunk, g + kUnitGroups - kF8Lag, sv0, bv0);
            if (g == kF8Lag - 1 && tile != ptile) {  // unit n - 1 is done and its tile ends there
              flush(ptile);
#pragma unroll
              for (int t = 0; t < MT; ++t) acc[t] = 0.f;
            }
          } else {
            epilogue(i - kF8Lag, chunk, g - kF8Lag, sv1, bv1);
          }
        }
      }
      ptile = tile;
      pchunk = chunk;
    }
    if (ncnt > 0) {  // the last kF8Lag groups
      const int i_end = 4 * ncnt;
      for (int j = i_end - kF8Lag; j < i_end; ++j) {
        if (j < 0) continue;
        const int gg = j & 3;
        epilogue(j, pchunk, gg, sv1, bv1);
      }
      flush(ptile);
    }
  }

  // every MMA of this CTA has completed (the issuer waited for its last commits) and every load
  // from tensor memory has returned: give the columns back
  tmem_fence_before();
  __syncthreads();
  if (warp == 1) {
    tmem_fence_after();
    tmem_dealloc(tmem, kF8TmemCols);
  }
}

// ------------------------------------------------------------------ host side
template <int MT>
static int launch_f8_mt(const F8Args& a, const F8Maps& maps, int grid, int smem_optin, cudaStream_t s) {
  // at least 116 KB, so that shared memory admits one CTA per SM (it takes all 512 tensor-memory
  // columns)
  int bytes = f8_layout<MT>(a.nblk_max).total;
  bytes = bytes < 116 * 1024 ? 116 * 1024 : bytes;
  if (bytes > smem_optin) return TB_ERR_UNSUPPORTED;
  cudaError_t e = cudaFuncSetAttribute(w2_gemv_f8_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(w2_gemv_f8_kernel<MT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return TB_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kF8Threads);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, w2_gemv_f8_kernel<MT>, maps, a);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return TB_ERR_CUDA;
  }
  return TB_OK;
}

// The tensor-memory decode GEMV for M <= 2 tokens over up to kMaxMats matrices that read the same
// x.  Returns TB_ERR_UNSUPPORTED (launching nothing) where it does not apply: more than 2 tokens,
// K not a multiple of 1024, more than 256 SMs, or a CTA whose units need more 1024-blocks of x'
// than its image holds; the caller then runs the warp-level GEMV.
int launch_gemv_f8_multi(const __half* x, int64_t M, int64_t K, const int8_t* signs, int block,
                         int nmat, const uint32_t* const* w, const __half* const* scales,
                         const __half* const* biases, const int64_t* N, __half* const* y,
                         void* workspace, size_t ws_bytes, int32_t* status, cudaStream_t s) {
  if (M < 1 || M > 2 || K < kBlock || K % kBlock || K > (1 << 22) || nmat < 1 || nmat > kMaxMats)
    return TB_ERR_UNSUPPORTED;
  if (block != 0 && block != kBlock) return TB_ERR_UNSUPPORTED;
  DeviceFacts f;
  int rc = device_facts(&f);
  if (rc != TB_OK) return rc;
  if (f.sms > 256) return TB_ERR_UNSUPPORTED;
  F8Args a = {};
  F8Maps maps;
  int64_t tiles = 0;
  for (int i = 0; i < nmat; ++i) {
    if (N[i] < 1 || N[i] > (1LL << 30)) return TB_ERR_SHAPE;
    a.scales[i] = scales[i];
    a.biases[i] = biases[i];
    a.y[i] = y[i];
    a.N[i] = (int)N[i];
    a.tile0[i] = (int)tiles;
    tiles += (N[i] + kUnitRows - 1) / kUnitRows;
  }
  const int C = (int)(K / (kUnitGroups * kGroup));
  if (tiles * C > (int64_t)INT32_MAX / 2) return TB_ERR_SHAPE;
  for (int i = nmat; i <= kMaxMats; ++i) a.tile0[i] = (int)tiles;
  const bool split = workspace && ws_bytes >= gemv_fixup_bytes();
  const int64_t S = tiles * C;
  int grid = f.sms;
  if (!split && tiles < grid) grid = (int)tiles;
  if (S < grid) grid = (int)S;
  // the most 1024-blocks of x' any CTA's units read
  int nblk_max = 1;
  for (int c = 0; c < grid; ++c) {
    int lo, hi, b1, e1, b2, e2;
    f8_cta_range(c, grid, (int)tiles, C, split ? 1 : 0, lo, hi);
    f8_blocks_needed(lo, hi - lo, C, (int)K, b1, e1, b2, e2);
    const int nb = (e1 - b1) + (e2 - b2);
    nblk_max = nb > nblk_max ? nb : nblk_max;
  }
  if (nblk_max > kF8MaxBlocks) return TB_ERR_UNSUPPORTED;
  for (int i = 0; i < nmat; ++i) {
    rc = code_map(w[i], N[i], K, &maps.codes[i]);
    if (rc != TB_OK) return rc;
  }
  for (int i = nmat; i < kMaxMats; ++i) maps.codes[i] = maps.codes[0];
  a.nmat = nmat;
  a.x = x;
  a.signs = block ? signs : nullptr;
  a.ws_count = split ? static_cast<int*>(workspace) : nullptr;
  a.ws_partial = split ? reinterpret_cast<float*>(static_cast<char*>(workspace) + 1024) : nullptr;
  a.Mc = (int)M;
  a.K = (int)K;
  a.G = (int)(K / kGroup);
  a.C = C;
  a.rotate = block != 0;
  a.n_tiles = (int)tiles;
  a.split = split ? 1 : 0;
  a.nblk_max = nblk_max;
  a.status = status;
  return M == 1 ? launch_f8_mt<1>(a, maps, grid, f.smem_optin, s) : launch_f8_mt<2>(a, maps, grid, f.smem_optin, s);
}

}  // namespace tb
