// Decode path of the Packed layer, TMA-streamed: fused sign*FWHT prologue + W2-g128 GEMV.
//
// [ARCH] kwkr.cn/news/564617, section "Hadamard 旋转把量化误差抹平的免费午餐":
//   a folded module rotates its input by the signed block Hadamard transform, then multiplies
//   it by the packed 2-bit, group-128 affine weights; the words are consumed as they are and
//   never expanded to an fp16 matrix.
// [PACK] lpnh.cn/news/2438023, section "文本模型加载artifact.load_model 与 Packed 模块".
//
// Work unit: 128 output rows x 512 k (4 groups of 128) = one 16 KB TMA box of packed codes
// (128 rows x 128 B, 128-byte swizzle; rows past N are zero-filled).  Each SM can keep only
// a handful of TMA requests in flight, so requests are made large: 16 KB boxes stream at
// the HBM rate where 2-4 KB requests stall at a fraction of it.  The scales and biases of the
// unit's rows come in the same ring slot, as TMA boxes of 8 groups (the unit's 4 and its
// neighbour's: a tensor copy's inner extent is at least 16 bytes), so the consumer warps issue
// no global loads of their own in the stream; each warp stages its rows' values as fp32
// pairs in shared memory.
//
// Schedule (stream-K): the units of all 128-row tiles, tile-major, are cut into one
// contiguous, equal range per CTA (one persistent CTA per SM), and each CTA's range into
// three contiguous sub-ranges, one per unit group of 4 consumer warps (warp i of a group owns
// rows 32i..32i+31 of every unit).  The first two groups walk their sub-range forwards, the
// last one backwards, so a tile shared with a neighbouring CTA is finished first.  A group
// keeps its partial sums in registers while it stays in one tile; a tile that lies wholly in
// the group's sub-range is written straight from registers; a tile cut by a group boundary is
// summed in shared memory, and one cut by a CTA boundary is summed in an fp32 workspace slot
// whose last contributor converts it to y and returns slot and counter to zero.  One producer
// warp per group keeps that group's ring of slots in flight (a group that is slow to release a
// slot holds back no other group's refill); before the activations are loaded each issues only
// one unit, so the loads of x are not queued behind megabytes of weight traffic.
//
// Arithmetic (per group of 128, per token): LOP3 puts each 2-bit code into the mantissa of
// an fp16 1024.0 (1024 + sigma*q, exact; sigma = 4^j from the field's bit position j);
// those half2 are mma.sync A fragments, x'/sigma the B fragment; the group's first MMA
// starts from zero and C = 1024*sum(x'/sigma) is taken off in the epilogue:
//   y += s * (D - C) + b * S,   S = sum x' over the group.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>
#include <unordered_map>

#include "tb_common.cuh"
#include "tb_gemv_core.cuh"
#include "tb_host.h"

namespace tb {

struct GemvTmaArgs {
  const __half* x;               // [Mc, K]
  const int8_t* signs;           // [K] or null
  const __half* scales[kMaxMats];  // [N_i, G]
  const __half* biases[kMaxMats];  // [N_i, G]
  __half* y[kMaxMats];           // [Mc, N_i]
  int N[kMaxMats];               // rows of matrix i
  int tile0[kMaxMats + 1];       // first 128-row tile of matrix i in the concatenated tile list
  int nmat;
  float* ws_partial;             // [kFixupCtas][2][128][MT] fp32 partial tiles, or null (tile-aligned)
  int* ws_count;                 // [kFixupCtas] contributions counted per shared tile
  int Mc, K, G, C;               // C = units per tile = K / 512
  int rotate, dw;
  int n_tiles;                   // total 128-row tiles of all matrices
  int split;                     // 1: stream-K ranges; 0: ranges on tile boundaries
  int32_t* status;
};

// ring slot: the unit's code box, then the scales and the biases of its 128 rows for the two
// chunks around it (boxes of 8 groups: the smallest inner extent a tensor copy takes)
constexpr int kGvSbBox = kUnitRows * 8 * 2;
constexpr int kGvSlot = kSlotBytes + 2 * kGvSbBox;

struct CodeMaps {
  CUtensorMap codes[kMaxMats];   // uint32 [N][K/16], box 32 x 128, 128-byte swizzle
  CUtensorMap sb[kMaxMats][2];   // fp16 scales, biases [N][G], box 8 x 128
};

// matrix of a global tile index
TB_DEVI int mat_of(const GemvTmaArgs& a, int tile) {
  int i = 0;
#pragma unroll
  for (int k = 1; k < kMaxMats; ++k) i += (k < a.nmat && tile >= a.tile0[k]);
  return i;
}

// Warp roles: warps 0..11 consume (three unit groups of four), warps 12..14 produce (one per
// group); warp 15 only completes the producers' warpgroup so that registers can move between
// the roles: the launch gives 128 per thread, the producer warpgroup drops to 40 and the
// consumers rise to 152 (12 x 32 x 152 + 4 x 32 x 40 = 63488 of the 65536 the block was
// launched with).
constexpr int kWsThreads = 16 * 32;
template <int MT>
__global__ void __launch_bounds__(kWsThreads, 1)
    w2_gemv_tma_kernel(const __grid_constant__ CodeMaps maps, const __grid_constant__ GemvTmaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int DW = a.dw, C = a.C, G = a.G, K = a.K;
  const GemvTmaLayout L = gemv_tma_layout<MT>(G, DW, kGvSlot);
  const uint32_t slots_u32 = smem_u32(smem + L.codes);
  __half* img = reinterpret_cast<__half*>(smem + L.img);
  float2* cs = reinterpret_cast<float2*>(smem + L.cs);    // [G][MT] = (1024 sum x'/sigma, sum x')
  float* accs = reinterpret_cast<float*>(smem + L.accs);  // [kCutSlots][128][MT]
  int* cnt = reinterpret_cast<int*>(smem + L.cnt);         // [kCutSlots]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kGroupsOfWarps * DW;
  uint64_t* xready = empty + kGroupsOfWarps * DW;
  __shared__ volatile int aborted;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // this CTA's unit range [lo, hi) and its cut into the groups' sub-ranges [bnd[u], bnd[u+1])
  const int S = a.n_tiles * C;
  int lo, hi;
  if (a.split) {
    lo = (int)((int64_t)S * blockIdx.x / gridDim.x);
    hi = (int)((int64_t)S * (blockIdx.x + 1) / gridDim.x);
  } else {
    lo = C * (int)((int64_t)a.n_tiles * blockIdx.x / gridDim.x);
    hi = C * (int)((int64_t)a.n_tiles * (blockIdx.x + 1) / gridDim.x);
  }
  const int nst = hi - lo;
  const int bnd1 = lo + nst / 3, bnd2 = lo + (2 * nst) / 3;

  if (threadIdx.x == 0) {
    aborted = 0;
    for (int i = 0; i < kGroupsOfWarps * DW; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, kWarpsPerUnit);
    }
    mbar_init(xready, kTmaConsumers);
    fence_barrier_init();
  }
  for (int i = threadIdx.x; i < kCutSlots * kUnitRows * MT; i += blockDim.x) accs[i] = 0.f;
  if (threadIdx.x < kCutSlots) cnt[threadIdx.x] = 0;
  __syncthreads();

  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (aborted) return;
    if (!mbar_wait(bar, parity)) {
      aborted = 1;
      set_status(a.status, TB_DEV_TIMEOUT);
    }
  };
  auto group_range = [&](int u, int& glo, int& ghi) {
    glo = u == 0 ? lo : u == 1 ? bnd1 : bnd2;
    ghi = u == 0 ? bnd1 : u == 1 ? bnd2 : hi;
  };

  if (warp >= kTmaConsumers) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 40;" ::: "memory");
    const int u = warp - kTmaConsumers;  // one producer warp per unit group
    if (u >= kGroupsOfWarps) return;
    // ---- producer of group u: the packed weights never depend on the previous kernel ----
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int glo, ghi;
      group_range(u, glo, ghi);
      const int cntu = ghi - glo;
      const bool back = u == kGroupsOfWarps - 1;
      const int first = back ? ghi - 1 : glo;
      int tl = first / C, ch = first - (first / C) * C;
      for (int n = 0, si = 0, k = 0; n < cntu; ++n) {  // si = n % DW, k = n / DW
        if (n == kPreIssue) wait(xready, 0);  // the activations have been read
        const int slot = u * DW + si;
        if (k > 0) wait(empty + slot, (k - 1) & 1);
        const int mi = mat_of(a, tl);
        const int row = (tl - a.tile0[mi]) * kUnitRows;
        const bool hb = a.biases[mi] != nullptr;
        mbar_arrive_expect_tx(full + slot, kSlotBytes + (hb ? 2 : 1) * kGvSbBox);
        const uint32_t dst = slots_u32 + slot * kGvSlot;
        tma2d(dst, &maps.codes[mi], ch * 32, row, full + slot, pol);
        tma2d(dst + kSlotBytes, &maps.sb[mi][0], 8 * (ch >> 1), row, full + slot, pol);
        if (hb) tma2d(dst + kSlotBytes + kGvSbBox, &maps.sb[mi][1], 8 * (ch >> 1), row, full + slot, pol);
        step_unit(tl, ch, C, back);
        if (++si == DW) {
          si = 0;
          ++k;
        }
      }
      // leave no copy in flight: wait (bounded, even after a timeout) for the last fill of
      // every slot of this group
      for (int n = cntu - 1; n >= 0 && n >= cntu - DW; --n)
        if (!mbar_wait(full + u * DW + n % DW, (n / DW) & 1)) set_status(a.status, TB_DEV_TIMEOUT);
    }
    __syncwarp();
    return;
  }

  // ---- consumers ----
  asm volatile("setmaxnreg.inc.sync.aligned.u32 152;" ::: "memory");
  const int g = lane >> 2, t = lane & 3;
  const int ug = warp / kWarpsPerUnit, wi = warp % kWarpsPerUnit;
  int glo, ghi;
  group_range(ug, glo, ghi);
  const bool back = ug == kGroupsOfWarps - 1;
  const int ncnt = ghi - glo;
  int tile = 0, chunk = 0;
  if (ncnt > 0) {
    const int first = back ? ghi - 1 : glo;
    tile = first / C;
    chunk = first - tile * C;
  }
  if (a.signs) {  // the signs never depend on the previous kernel: into L1 before the wait
    int pb1, pe1, pb2, pe2;
    blocks_needed(lo, nst, C, K, pb1, pe1, pb2, pe2);
    const int pnb = (pe1 - pb1) + (pe2 - pb2);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int it = warp + q * kTmaConsumers;
      if (it < a.Mc * pnb) {
        const int bi = it % pnb;
        const int b = bi < pe1 - pb1 ? pb1 + bi : pb2 + (bi - (pe1 - pb1));
        asm volatile("prefetch.global.L1 [%0];" ::"l"(a.signs + b * kBlock + lane * 32));
      }
    }
  }

  asm volatile("griddepcontrol.wait;" ::: "memory");
  {
    // prologue: x' = fwht(signs * x) -> B-fragment image, (C, S) per group and token, for the
    // 1024-blocks that this CTA's units read.  Every consumer warp takes items (token, block,
    // half) warp, warp + 12, ...; the loads of two items are issued before either is
    // transformed, so a warp waits once per pair.
    const int nb = K / kBlock;
    int b1 = 0, e1 = nb, b2 = 0, e2 = 0;  // the blocks needed: [b1, e1) and [b2, e2)
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
    const int nblk = (e1 - b1) + (e2 - b2);
    // An item is one half of a (token, block) pair: since H1024 = [[H512, H512], [H512, -H512]],
    // outputs 0..511 of the block are H512 (x_lo + x_hi) and outputs 512..1023 are
    // H512 (x_lo - x_hi), two independent 512-point transforms on two warps.  Lane l holds
    // elements 16 l .. 16 l + 15 of both input halves and of its output half.
    auto item_block = [&](int it, int& tok, int& b, int& hh) {
      hh = it & 1;
      const int rest = it >> 1;
      tok = rest / nblk;
      const int bi = rest - tok * nblk;
      b = bi < e1 - b1 ? b1 + bi : b2 + (bi - (e1 - b1));
    };
    auto load_block = [&](int it, uint4 (&xr)[4], uint4 (&sr)[2]) {
      int tok, b, hh;
      item_block(it, tok, b, hh);
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
    auto transform_block = [&](int it, const uint4 (&xr)[4], const uint4 (&sr)[2]) {
      int tok, b, hh;
      item_block(it, tok, b, hh);
      // v[e] = output element b*1024 + 512*hh + lane*16 + e
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
        wht512_a_shfl(v, lane);  // the other nine stages, layout kept
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] *= kInvSqrtBlock;
      }
      // group of 128 of this output: eight lanes (q = lane & 7) of 16 elements each
      const int grp = b * (kBlock / kGroup) + 4 * hh + (lane >> 3);
      const int q = lane & 7;
      float ssum = 0.f, csum = 0.f;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        v[e] = __half2float(__float2half_rn(v[e]));  // x' rounded to fp16
        ssum += v[e];
      }
      ssum += __shfl_xor_sync(0xffffffffu, ssum, 1);
      ssum += __shfl_xor_sync(0xffffffffu, ssum, 2);
      ssum += __shfl_xor_sync(0xffffffffu, ssum, 4);
      // B-fragment image: entry (grp, mp) holds, for each fragment lane t, group elements
      // 32 t + 16 (mp >> 1) + 4 (mp & 1) + {0..3} and the same + 8, divided by sigma of their
      // position; this lane's 16 elements are those of t = q >> 1 and mp = 2 (q & 1) + {0, 1}
#pragma unroll
      for (int m1 = 0; m1 < 2; ++m1) {
        const int mp = 2 * (q & 1) + m1;
        uint32_t pk[4];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          const int p = 4 * m1 + e2;
          const float is = inv_sigma_p(p);
          const __half lo_ = __float2half_rn(v[p] * is), hi_ = __float2half_rn(v[p + 8] * is);
          csum += __half2float(lo_) + __half2float(hi_);
          pk[e2] = (uint32_t)__half_as_ushort(lo_) | ((uint32_t)__half_as_ushort(hi_) << 16);
        }
        *reinterpret_cast<uint4*>(img + ((size_t)(grp * 4 + mp) * MT + tok) * 32 + (q >> 1) * 8) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      csum += __shfl_xor_sync(0xffffffffu, csum, 1);
      csum += __shfl_xor_sync(0xffffffffu, csum, 2);
      csum += __shfl_xor_sync(0xffffffffu, csum, 4);
      if (q == 0) cs[grp * MT + tok] = make_float2(1024.f * csum, ssum);
    };
    const int items = 2 * MT * nblk;
    bool told = false;
    for (int it = warp; it < items; it += 2 * kTmaConsumers) {
      const int it2 = it + kTmaConsumers;
      uint4 xa[4], sa[2], xb[4], sb2[2];
      load_block(it, xa, sa);
      if (it2 < items) load_block(it2, xb, sb2);
      transform_block(it, xa, sa);
      if (it2 < items) transform_block(it2, xb, sb2);
      if (!told) {  // this warp's first activations are in: the producer may stream on
        told = true;
        __syncwarp();
        if (lane == 0) mbar_arrive(xready);
      }
    }
    if (!told && lane == 0) mbar_arrive(xready);
    asm volatile("bar.sync 1, %0;" ::"n"(kTmaConsumers * 32) : "memory");
  }

  // mma row g <-> unit row 32*wi + 16*j + rA (and + 8): conflict-free swizzled reads
  const int rA = 2 * (g & 3) + (g >> 2);
  const int R0 = 32 * wi + rA;
  const int tokc = g < MT ? g : 0;
  const uint32_t imgt = smem_u32(img) + tokc * 64 + t * 16;
  const uint32_t csa = smem_u32(cs);
  const uint32_t accs_u32 = smem_u32(accs);
  const int t0 = min(2 * t, MT - 1), t1 = min(2 * t + 1, MT - 1);
  const uint32_t ss = smem_u32(smem + L.sstage) + warp * kScaleStageBytes;

  // Add this warp's sums of tile T (all of the group's units of T) to wherever T is finished.
  auto flush = [&](int T, float (&acc)[2][4]) {
    const int mi = mat_of(a, T);
    const int N = a.N[mi], row0 = (T - a.tile0[mi]) * kUnitRows;
    __half* yo = a.y[mi];
    const int tb = T * C, te = tb + C;
    if (tb >= glo && te <= ghi) {  // the whole tile is this group's: these 32 rows are final
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int ra = row0 + R0 + 16 * j, rb = ra + 8;
        if (2 * t < a.Mc) {
          if (ra < N) yo[(int64_t)(2 * t) * N + ra] = __float2half_rn(acc[j][0]);
          if (rb < N) yo[(int64_t)(2 * t) * N + rb] = __float2half_rn(acc[j][2]);
        }
        if (2 * t + 1 < a.Mc) {
          if (ra < N) yo[(int64_t)(2 * t + 1) * N + ra] = __float2half_rn(acc[j][1]);
          if (rb < N) yo[(int64_t)(2 * t + 1) * N + rb] = __float2half_rn(acc[j][3]);
        }
      }
      return;
    }
    // a tile cut by a boundary: its shared slot is the first boundary that falls in it
    const int b = (lo / C == T) ? 0 : (bnd1 / C == T) ? 1 : (bnd2 / C == T) ? 2 : 3;
    // contributions expected in this CTA: 4 warps of every group whose sub-range meets T
    int groups = 0;
#pragma unroll
    for (int u = 0; u < kGroupsOfWarps; ++u) {
      int ulo, uhi;
      group_range(u, ulo, uhi);
      groups += (ulo < uhi && ulo < te && uhi > tb);
    }
    const uint32_t atu = accs_u32 + b * kUnitRows * MT * 4;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int ra = R0 + 16 * j, rb = ra + 8;
      if (2 * t < MT) {
        red_shared_add(atu + (ra * MT + 2 * t) * 4, acc[j][0]);
        red_shared_add(atu + (rb * MT + 2 * t) * 4, acc[j][2]);
      }
      if (2 * t + 1 < MT) {
        red_shared_add(atu + (ra * MT + 2 * t + 1) * 4, acc[j][1]);
        red_shared_add(atu + (rb * MT + 2 * t + 1) * 4, acc[j][3]);
      }
    }
    __syncwarp();
    int last = 0;
    if (lane == 0) {
      __threadfence_block();
      last = atomicAdd(cnt + b, 1) == groups * kWarpsPerUnit - 1;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    // this warp finishes the tile for this CTA
    __threadfence_block();
    const float* at = accs + b * kUnitRows * MT;
    if (tb >= lo && te <= hi) {
      for (int e = lane; e < kUnitRows * MT; e += 32) {
        const int r_ = e / MT, k_ = e - r_ * MT;
        if (row0 + r_ < N && k_ < a.Mc) yo[(int64_t)k_ * N + row0 + r_] = __float2half_rn(at[e]);
      }
      return;
    }
    // shared with other CTAs: this CTA's part goes to its own workspace slot (plain stores:
    // float atomics into one shared slot wait far longer under the weight stream), slot 0
    // for the tile of its first unit, 1 for the tile of its last
    float* mine = a.ws_partial + ((int64_t)blockIdx.x * 2 + (lo / C == T ? 0 : 1)) * kUnitRows * MT;
    for (int e = lane; e < kUnitRows * MT; e += 32) __stcg(mine + e, at[e]);
    __syncwarp();
    // the last of the tile's CTAs to count in adds the parts in CTA order (the result does
    // not depend on which CTA finishes last) and returns the counter to zero
    const int first = stage_owner(tb, S, gridDim.x);
    const int lastc = stage_owner(te - 1, S, gridDim.x);
    int fin = 0;
    if (lane == 0) {
      fence_acq_rel_gpu();  // the warp's part before the count
      fin = atomicAdd(a.ws_count + first, 1) == lastc - first;
    }
    fin = __shfl_sync(0xffffffffu, fin, 0);
    if (!fin) return;
    fence_acq_rel_gpu();  // every contributor's part after the count
    // the tile starts inside CTA `first` (its slot 0 when the tile is also the tile of its
    // first unit, else 1); every later contributor starts inside the tile (slot 0)
    int flo, fhi;
    cta_range_of(first, gridDim.x, a.n_tiles, C, flo, fhi);
    const float* p0 = a.ws_partial + ((int64_t)first * 2 + (flo / C == T ? 0 : 1)) * kUnitRows * MT;
    for (int eb = 0; eb < kUnitRows * MT; eb += 128) {  // four elements per lane per pass
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      for (int c = first; c <= lastc; c += 4) {  // four contributors' loads in flight at once
        float l[4][4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int cc = c + q;
          const float* pc = cc == first ? p0 : a.ws_partial + (int64_t)cc * 2 * kUnitRows * MT;
#pragma unroll
          for (int k = 0; k < 4; ++k) l[q][k] = cc <= lastc ? __ldcg(pc + eb + lane + 32 * k) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int k = 0; k < 4; ++k) v[k] += l[q][k];
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = eb + lane + 32 * k;
        const int r_ = e / MT, k_ = e - r_ * MT;
        if (row0 + r_ < N && k_ < a.Mc) yo[(int64_t)k_ * N + row0 + r_] = __float2half_rn(v[k]);
      }
    }
    if (lane == 0) a.ws_count[first] = 0;
  };

  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  int si = 0;        // ring slot of the current unit within the group's DW slots: n % DW
  uint32_t ph = 0;   // its fill parity: (n / DW) & 1
  // unit n with its scales and biases in (sv, bv), which are then reloaded for unit n + 2
  auto body = [&](int n) {
    const int slot = ug * DW + si;
    wait(full + slot, ph);
    if (++si == DW) {
      si = 0;
      ph ^= 1;
    }
    const uint32_t box = slots_u32 + slot * kGvSlot;
    {  // this warp's 32 rows' (s, b) of the unit's four groups, from the slot, as fp32 pairs
      const uint32_t sp = box + kSlotBytes + (32 * wi + lane) * 16 + (chunk & 1) * 8;
      const uint2 sv = ld_shared_v2(sp);
      const uint2 bv = a.biases[mat_of(a, tile)] ? ld_shared_v2(sp + kGvSbBox)
                                                 : make_uint2(sv.x ^ 0x80008000u, sv.y ^ 0x80008000u);
      const uint32_t r = ss + lane * kUnitGroups * 8;
      const float2 sf0 = __half22float2(*reinterpret_cast<const __half2*>(&sv.x));
      const float2 sf1 = __half22float2(*reinterpret_cast<const __half2*>(&sv.y));
      const float2 bf0 = __half22float2(*reinterpret_cast<const __half2*>(&bv.x));
      const float2 bf1 = __half22float2(*reinterpret_cast<const __half2*>(&bv.y));
      asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(r), "f"(sf0.x), "f"(bf0.x), "f"(sf0.y), "f"(bf0.y) : "memory");
      asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(r + 16), "f"(sf1.x), "f"(bf1.x), "f"(sf1.y), "f"(bf1.y) : "memory");
      __syncwarp();
    }
#pragma unroll
    for (int gi = 0; gi < kUnitGroups; ++gi)
      unit_group<MT>(box, R0, t, gi, chunk * kUnitGroups + gi, imgt, ss, rA, csa, t0, t1, acc);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + slot);
    const int cur = tile;
    step_unit(tile, chunk, C, back);
    if (tile != cur || n == ncnt - 1) {
      flush(cur, acc);
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
    }
  };
  for (int n = 0; n < ncnt; ++n) body(n);
}

// ------------------------------------------------------------------ host side
// cuTensorMapEncodeTiled from the driver, resolved once through the runtime (the library does not
// link libcuda directly, so it loads on machines without a driver too); null if unavailable
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// tensor map of one packed matrix's codes (box 32 words x 128 rows, 128-byte swizzle), cached
// by (pointer, shape)
int code_map(const uint32_t* w, int64_t N, int64_t K, CUtensorMap* out) {
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
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
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

// workspace of the split (stream-K) schedule: counters [kFixupCtas] of tiles shared by
// several CTAs (indexed by the tile's first CTA; zero before a call and after it), then
// each CTA's fp32 parts [kFixupCtas][2][128][8] of the shared tiles it computes (scratch)
constexpr int kFixupCtas = 256;
constexpr size_t kFixupCounterBytes = 1024;
constexpr size_t kFixupPartialBytes = (size_t)kFixupCtas * 2 * kUnitRows * 8 * 4;
static_assert(kFixupCtas * 4 <= kFixupCounterBytes, "counters fit their region");
size_t gemv_fixup_bytes() { return kFixupCounterBytes + kFixupPartialBytes; }
size_t gemv_fixup_counter_bytes() { return kFixupCounterBytes; }

template <int MT>
static int launch_tma_mt(GemvTmaArgs a, const CodeMaps& maps, int64_t M, int64_t K,
                         const DeviceFacts& f, cudaStream_t s) {
  // slots per unit group from what is left of shared memory
  int dw = kMaxSlotsPerGroup;
  while (dw >= 1 && gemv_tma_layout<MT>(a.G, dw, kGvSlot).total > f.smem_optin) --dw;
  if (dw < 1) return TB_ERR_SHAPE;
  a.dw = dw;
  const int bytes = gemv_tma_layout<MT>(a.G, dw, kGvSlot).total;
  int rc = ensure_dynamic_smem(reinterpret_cast<const void*>(w2_gemv_tma_kernel<MT>), f.device, bytes);
  if (rc != TB_OK) return rc;
  cudaError_t e;
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
    cfg.blockDim = dim3(kWsThreads);
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
static int tma_tokens_per_pass(int64_t M, int G, int smem_optin) {
  int mt = M >= 5 ? 8 : M >= 3 ? 4 : M == 2 ? 2 : 1;
  auto fits = [&](int total) { return total <= smem_optin; };
  while (mt > 1) {
    const bool ok = mt == 8 ? fits(gemv_tma_layout<8>(G, 2, kGvSlot).total)
                  : mt == 4 ? fits(gemv_tma_layout<4>(G, 2, kGvSlot).total)
                            : fits(gemv_tma_layout<2>(G, 2, kGvSlot).total);
    if (ok) break;
    mt >>= 1;
  }
  return mt;
}

// tensor map of a [N, G] fp16 array of scales or biases (box 8 groups x 128 rows, no swizzle),
// cached by (pointer, shape)
int group_map(const __half* p, int64_t N, int64_t G, CUtensorMap* out) {
  struct Key {
    const void* p;
    int64_t N, G;
    bool operator==(const Key& o) const { return p == o.p && N == o.N && G == o.G; }
  };
  struct Hash {
    size_t operator()(const Key& k) const { return std::hash<const void*>()(k.p) ^ std::hash<int64_t>()(k.N * 131 + k.G); }
  };
  static std::mutex mu;
  static std::unordered_map<Key, CUtensorMap, Hash> cache;
  const Key key{p, N, G};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *out = it->second;
      return TB_OK;
    }
  }
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return TB_ERR_CUDA;
  CUtensorMap m;
  const cuuint64_t dims[2] = {(cuuint64_t)G, (cuuint64_t)N};
  const cuuint64_t strides[1] = {(cuuint64_t)G * 2};
  const cuuint32_t box[2] = {8, (cuuint32_t)kUnitRows};
  const cuuint32_t es[2] = {1, 1};
  if (enc(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(p), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return TB_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() > 4096) cache.clear();
  cache[key] = m;
  *out = m;
  return TB_OK;
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
  int64_t tiles = 0;
  for (int i = 0; i < nmat; ++i) {
    if (N[i] < 1 || N[i] > (1LL << 30)) return TB_ERR_SHAPE;
    rc = code_map(w[i], N[i], K, &maps.codes[i]);
    if (rc == TB_OK) rc = group_map(scales[i], N[i], K / kGroup, &maps.sb[i][0]);
    if (rc == TB_OK) rc = biases[i] ? group_map(biases[i], N[i], K / kGroup, &maps.sb[i][1]) : TB_OK;
    if (!biases[i]) maps.sb[i][1] = maps.sb[i][0];
    if (rc != TB_OK) return rc;
    a.scales[i] = scales[i];
    a.biases[i] = biases[i];
    a.y[i] = y[i];
    a.N[i] = (int)N[i];
    a.tile0[i] = (int)tiles;
    tiles += (N[i] + kUnitRows - 1) / kUnitRows;
  }
  // unit indices (tiles x K/512) are 32-bit in the kernel
  if (tiles * (K / (kUnitGroups * kGroup)) > (int64_t)INT32_MAX / 2) return TB_ERR_SHAPE;
  for (int i = nmat; i <= kMaxMats; ++i) a.tile0[i] = (int)tiles;
  for (int i = nmat; i < kMaxMats; ++i) {
    maps.codes[i] = maps.codes[0];
    maps.sb[i][0] = maps.sb[0][0];
    maps.sb[i][1] = maps.sb[0][1];
  }
  a.nmat = nmat;
  a.x = x;
  a.signs = signs;
  const bool split = workspace && ws_bytes >= gemv_fixup_bytes() && f.sms <= kFixupCtas;
  a.ws_count = split ? static_cast<int*>(workspace) : nullptr;
  a.ws_partial = split ? reinterpret_cast<float*>(static_cast<char*>(workspace) + kFixupCounterBytes)
                       : nullptr;
  a.split = split ? 1 : 0;
  a.K = (int)K;
  a.G = (int)(K / kGroup);
  a.C = (int)(K / (kUnitGroups * kGroup));
  a.rotate = block != 0;
  a.n_tiles = (int)tiles;
  a.status = status;
  const int mt = tma_tokens_per_pass(M, a.G, f.smem_optin);
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
