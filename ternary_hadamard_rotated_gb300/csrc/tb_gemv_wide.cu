// Batched decode (9 to 64 tokens) of the Packed layer on the fifth-generation tensor cores: the
// weights are the MMA's 128-row side, the tokens its N side, so no token tile is padded to 128.
//
// [ARCH] kwkr.cn/news/564617, section "Hadamard 旋转把量化误差抹平的免费午餐": the rotated input
// times the packed 2-bit, group-128 affine weights, never expanded in memory; section
// "打包格式的工程MLX 2.25 bits 与 GGUF 的两种装箱": a code decodes to s*q + b, exactly {-s, 0, s}
// in fp16 for the pack's b = -s.
//
// Per CTA (one per SM), in the GEMV's stream-K ranges of units (128 rows x 512 k):
//  * warp 0 streams the 16 KB boxes of packed codes, and warp 10, independently, per group of
//    128 k the two 64-k boxes of x' (fp16 [MT rows, 64 k] each, 128-byte swizzle; rows past M
//    read as zero), x' being the rotation kernel's output in the pair order of a decoded word
//    (pair p of 16 columns holds columns p and p + 8);
//  * warps 2..5 (groups 0 and 2 of a unit) and 6..9 (groups 1 and 3) decode a group's 128 codes
//    of their row into 64 fp16 pairs s*q + b and store them as 64 columns of a tensor-memory A
//    slot (six slots; a group's A slot and x' slot are released by one commit of its MMAs);
//  * warp 1 issues the group's eight tcgen05.mma (kind::f16, M = 128, N = MT, K = 16) into the
//    accumulator of the current tile segment (two accumulators of MT columns: a segment's is read
//    while the next one fills);
//  * at the end of a segment warps 2..5 read the accumulator: a whole tile is written to y, a
//    tile shared with other CTAs goes through the workspace, the last of them adding the parts in
//    CTA order.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "tb_common.cuh"
#include "tb_gemv_core.cuh"
#include "tb_host.h"
#include "tb_tcgen05.cuh"

namespace tb {

int code_map(const uint32_t* w, int64_t N, int64_t K, CUtensorMap* out);

constexpr int kWdThreads = 11 * 32;  // code producer, MMA issuer, two decoder warpgroups, x' producer
constexpr int kWdRing = 6;           // A slots (64 columns of fp16 pairs: one group of 128 k)
constexpr int kWdTmemCols = 512;
// 16 KB code boxes and x' slots (two 64-k boxes of MT rows: one group) in about 200 KB of shared
// memory; x' comes from L2 with a long latency, so its ring is as deep as the room allows
template <int MT> struct WideRings {
  static constexpr int kCode = MT <= 32 ? 6 : 4;
  static constexpr int kX = MT <= 16 ? 24 : MT <= 32 ? 12 : MT <= 48 ? 10 : 8;
};

TB_DEVI void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, int accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

TB_DEVI void tma2d_plain(uint32_t dst, const CUtensorMap* tm, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 32 consecutive fp32 columns of this thread's lane
TB_DEVI void tmem_ld32(uint32_t taddr, float (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]), "=f"(r[7]),
        "=f"(r[8]), "=f"(r[9]), "=f"(r[10]), "=f"(r[11]), "=f"(r[12]), "=f"(r[13]), "=f"(r[14]),
        "=f"(r[15]), "=f"(r[16]), "=f"(r[17]), "=f"(r[18]), "=f"(r[19]), "=f"(r[20]), "=f"(r[21]),
        "=f"(r[22]), "=f"(r[23]), "=f"(r[24]), "=f"(r[25]), "=f"(r[26]), "=f"(r[27]), "=f"(r[28]),
        "=f"(r[29]), "=f"(r[30]), "=f"(r[31])
      : "r"(taddr)
      : "memory");
}
TB_DEVI void tmem_ld16(uint32_t taddr, float (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]), "=f"(r[7]),
        "=f"(r[8]), "=f"(r[9]), "=f"(r[10]), "=f"(r[11]), "=f"(r[12]), "=f"(r[13]), "=f"(r[14]), "=f"(r[15])
      : "r"(taddr)
      : "memory");
}

struct WideArgs {
  const uint32_t* w;     // codes [N, K/16] (through the tensor map)
  const __half* scales;  // [N, G]
  const __half* biases;  // [N, G] or null (each bias -s)
  __half* y;             // [M, N]
  float* part;           // [grid][2][128][MT] fp32 parts of tiles shared between CTAs (scratch)
  int* count;            // [grid] contributions per shared tile, indexed by its first CTA
  int M, N, K, G, C, n_tiles;
  int32_t* status;
};

struct WideLayout {
  int code, xs, bars, tslot, total;
};

template <int MT>
__host__ __device__ constexpr WideLayout wide_layout() {
  WideLayout L{0, 0, 0, 0, 0};
  int off = 0;
  L.code = off;
  off += WideRings<MT>::kCode * kSlotBytes;
  L.xs = off;  // 1024-aligned: two boxes of MT rows x 128 bytes per slot
  off += WideRings<MT>::kX * 2 * MT * 128;
  L.bars = off;
  off += (2 * WideRings<MT>::kCode + 2 * WideRings<MT>::kX + 2 * kWdRing + 4) * 8;
  L.tslot = off;
  off += 16;
  L.total = off + 1024;
  return L;
}

// the CTA owning global unit s when S units are cut into grid equal ranges
TB_DEVI int wd_owner(int64_t s, int64_t S, int grid) { return (int)(((s + 1) * grid - 1) / S); }
TB_DEVI int wd_lo(int c, int64_t S, int grid) { return (int)(S * c / grid); }

template <int MT>
__global__ void __launch_bounds__(kWdThreads, 1)
    w2_gemv_wide_kernel(const __grid_constant__ CUtensorMap cmap, const __grid_constant__ CUtensorMap xmap,
                        const __grid_constant__ WideArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int C = a.C, G = a.G;
  constexpr WideLayout L = wide_layout<MT>();
  constexpr int kXSlot = 2 * MT * 128;
  constexpr int kWdCodeRing = WideRings<MT>::kCode, kWdXRing = WideRings<MT>::kX;
  const uint32_t code = smem_u32(smem + L.code);
  const uint32_t xs = smem_u32(smem + L.xs);
  uint64_t* cfull = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* cempty = cfull + kWdCodeRing;
  uint64_t* xfull = cempty + kWdCodeRing;
  uint64_t* xempty = xfull + kWdXRing;  // the MMAs that read the x' slot are done
  uint64_t* afull = xempty + kWdXRing;
  uint64_t* gdone = afull + kWdRing;  // the MMAs that read the A slot are done
  uint64_t* dfull = gdone + kWdRing;  // [2]: a segment's accumulator is complete
  uint64_t* dempty = dfull + 2;       // [2]: it has been read
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + L.tslot);
  __shared__ volatile int aborted;
  __shared__ int fin_s;  // this CTA is the last contributor of a shared tile

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int64_t S = (int64_t)a.n_tiles * C;
  const int lo = wd_lo(blockIdx.x, S, gridDim.x), hi = wd_lo(blockIdx.x + 1, S, gridDim.x);
  const int nunits = hi - lo;

  if (threadIdx.x == 0) {
    aborted = 0;
    for (int i = 0; i < kWdCodeRing; ++i) {
      mbar_init(cfull + i, 1);
      mbar_init(cempty + i, 8);  // every decoder warp reads every box
    }
    for (int i = 0; i < kWdXRing; ++i) {
      mbar_init(xfull + i, 1);
      mbar_init(xempty + i, 1);
    }
    for (int i = 0; i < kWdRing; ++i) {
      mbar_init(afull + i, 4);  // the four warps of the warpgroup that decodes the group
      mbar_init(gdone + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(dfull + i, 1);
      mbar_init(dempty + i, 4);
    }
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tslot, kWdTmemCols);
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tD0 = tmem + kWdRing * 64;  // accumulators after the A slots

  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (aborted) return;
    if (!mbar_wait(bar, parity)) {
      aborted = 1;
      set_status(a.status, TB_DEV_TIMEOUT);
    }
  };
  // a unit ends its tile segment in this CTA when it is the last of its tile or of the range
  auto seg_end = [&](int unit) { return unit + 1 == hi || (unit + 1) % C == 0; };

  if (warp == 0) {
    // ---- code producer: the packed weights never depend on the previous kernel
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      for (int n = 0; n < nunits; ++n) {
        const int unit = lo + n, tile = unit / C, chunk = unit - tile * C;
        const int slot = n % kWdCodeRing;
        if (n >= kWdCodeRing) wait(cempty + slot, ((n / kWdCodeRing) - 1) & 1);
        mbar_arrive_expect_tx(cfull + slot, kSlotBytes);
        tma2d(code + slot * kSlotBytes, &cmap, chunk * 32, tile * kUnitRows, cfull + slot, pol);
      }
      // leave no copy in flight
      for (int n = nunits - 1; n >= 0 && n >= nunits - kWdCodeRing; --n)
        if (!mbar_wait(cfull + n % kWdCodeRing, (n / kWdCodeRing) & 1)) set_status(a.status, TB_DEV_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 10) {
    // ---- x' producer: two boxes per group, each slot refilled once its MMAs are done
    if (lane == 0) {
      asm volatile("griddepcontrol.wait;" ::: "memory");  // x' is the previous kernel's output
      for (int n = 0; n < nunits; ++n) {
        const int chunk = (lo + n) % C;
#pragma unroll 1
        for (int g = 0; g < kUnitGroups; ++g) {
          const int i = 4 * n + g, slot = i % kWdXRing;
          if (i >= kWdXRing) wait(xempty + slot, ((i / kWdXRing) - 1) & 1);
          mbar_arrive_expect_tx(xfull + slot, kXSlot);
          const int k0 = chunk * 512 + g * 128;
          tma2d_plain(xs + slot * kXSlot, &xmap, k0, 0, xfull + slot);
          tma2d_plain(xs + slot * kXSlot + MT * 128, &xmap, k0 + 64, 0, xfull + slot);
        }
      }
      const int ni = 4 * nunits;
      for (int i = ni - 1; i >= 0 && i >= ni - kWdXRing; --i)
        if (!mbar_wait(xfull + i % kWdXRing, (i / kWdXRing) & 1)) set_status(a.status, TB_DEV_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issuer: eight MMAs per group into the current segment's accumulator
    if (lane == 0) {
      // kind::f16 instruction descriptor: fp16 A and B, fp32 D, both K-major, M = 128, N = MT
      constexpr uint32_t idesc = (1u << 4) | ((uint32_t)(MT >> 3) << 17) | ((128u >> 4) << 24);
      int seg = 0;
      bool seg_start = true;
      for (int n = 0; n < nunits; ++n) {
        const int unit = lo + n;
#pragma unroll 1
        for (int g = 0; g < kUnitGroups; ++g) {
          const int i = 4 * n + g;
          const int sl = i % kWdRing, sx = i % kWdXRing, sd = seg & 1;
          if (seg_start && g == 0 && seg >= 2) wait(dempty + sd, ((seg >> 1) - 1) & 1);
          wait(afull + sl, (i / kWdRing) & 1);
          wait(xfull + sx, (i / kWdXRing) & 1);
          tmem_fence_after();
          const uint32_t xb = xs + (uint32_t)(sx * kXSlot);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t baddr = xb + (uint32_t)((kk >> 2) * MT * 128 + (kk & 3) * 32);
            mma_f16_ts(tD0 + (uint32_t)(sd * MT), tmem + (uint32_t)(sl * 64 + 8 * kk),
                       smem_desc_sw128(baddr, 1024u), idesc, (seg_start && g == 0 && kk == 0) ? 0 : 1);
          }
          mma_commit(gdone + sl);
          mma_commit(xempty + sx);
          seg_start = false;
          if (g == kUnitGroups - 1 && seg_end(unit)) {
            mma_commit(dfull + sd);
            ++seg;
            seg_start = true;
          }
        }
      }
      // every MMA issued has completed before the columns are given back
      if (seg > 0 && !mbar_wait(dfull + ((seg - 1) & 1), ((seg - 1) >> 1) & 1)) set_status(a.status, TB_DEV_TIMEOUT);
    }
    __syncwarp();
  } else if (warp < 10) {
    // ---- decoders: warpgroup u decodes groups u and u + 2 of every unit; thread r = unit row r
    // = tensor-memory lane r.  Warpgroup 0 also finishes the tile segments.
    const int u = (warp - 2) >> 2, q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const int rsw = r & 7;

    // scales and biases of unit n for this row (the unit's four groups), as fp16 pairs
    auto load_sb = [&](int n, uint2& sv, uint2& bv) {
      sv = make_uint2(0, 0);
      bv = make_uint2(0, 0);
      if (n >= nunits) return;
      const int unit = lo + n, tile = unit / C, chunk = unit - tile * C;
      const int row = tile * kUnitRows + r;
      if (row >= a.N) return;
      sv = __ldg(reinterpret_cast<const uint2*>(a.scales + (int64_t)row * G + chunk * kUnitGroups));
      bv = a.biases ? __ldg(reinterpret_cast<const uint2*>(a.biases + (int64_t)row * G + chunk * kUnitGroups))
                    : make_uint2(sv.x ^ 0x80008000u, sv.y ^ 0x80008000u);
    };

    // Read a segment's accumulator (MT fp32 columns of this row) and finish it: y for a tile that
    // lies wholly in this CTA's range, else this CTA's part of a tile shared with others.
    auto finish_segment = [&](int seg, int tile, bool whole) {
      const int sd = seg & 1;
      wait(dfull + sd, (seg >> 1) & 1);
      tmem_fence_after();
      float v[MT];
      const uint32_t tD = tD0 + (uint32_t)(sd * MT) + lane_off;
      if constexpr (MT == 16) {
        tmem_ld16(tD, *reinterpret_cast<float(*)[16]>(&v[0]));
      } else if constexpr (MT == 32) {
        tmem_ld32(tD, *reinterpret_cast<float(*)[32]>(&v[0]));
      } else if constexpr (MT == 48) {
        tmem_ld32(tD, *reinterpret_cast<float(*)[32]>(&v[0]));
        tmem_ld16(tD + 32, *reinterpret_cast<float(*)[16]>(&v[32]));
      } else {
        tmem_ld32(tD, *reinterpret_cast<float(*)[32]>(&v[0]));
        tmem_ld32(tD + 32, *reinterpret_cast<float(*)[32]>(&v[32]));
      }
      tmem_wait_ld();
      tmem_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dempty + sd);
      const int row = tile * kUnitRows + r;
      if (whole) {
        if (row < a.N)
#pragma unroll
          for (int t = 0; t < MT; ++t)
            if (t < a.M) a.y[(int64_t)t * a.N + row] = __float2half_rn(v[t]);
        return;
      }
      // shared with other CTAs: this CTA's part to its own slot (0: the tile of its first unit)
      const int tb_ = tile * C, te = tb_ + C;
      float* mine = a.part + ((int64_t)blockIdx.x * 2 + (lo / C == tile ? 0 : 1)) * kUnitRows * MT;
#pragma unroll
      for (int t = 0; t < MT; ++t) __stcg(mine + t * kUnitRows + r, v[t]);
      // the four warps' parts, then one count per CTA: every writer fences its own stores (the
      // barrier orders them only within the CTA)
      fence_acq_rel_gpu();
      asm volatile("bar.sync 1, 128;" ::: "memory");
      const int first = wd_owner(tb_, S, gridDim.x), lastc = wd_owner(te - 1, S, gridDim.x);
      if (threadIdx.x == 64) {  // lane 0 of warp 2
        fin_s = atomicAdd(a.count + first, 1) == lastc - first;
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (!fin_s) return;
      fence_acq_rel_gpu();  // every contributor's part after the count
      const int flo = wd_lo(first, S, gridDim.x);
      float acc[MT];
#pragma unroll
      for (int t = 0; t < MT; ++t) acc[t] = 0.f;
      for (int c = first; c <= lastc; ++c) {  // the parts in CTA order: the same sum every call
        const int slot = c == first ? (flo / C == tile ? 0 : 1) : 0;
        const float* pc = a.part + ((int64_t)c * 2 + slot) * kUnitRows * MT;
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[t] += __ldcg(pc + t * kUnitRows + r);
      }
      if (row < a.N)
#pragma unroll
        for (int t = 0; t < MT; ++t)
          if (t < a.M) a.y[(int64_t)t * a.N + row] = __float2half_rn(acc[t]);
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (threadIdx.x == 64) a.count[first] = 0;
    };

    // scale / bias words of units n, n + 1, n + 2 (loaded two units ahead of their use)
    uint2 sv0, bv0, sv1, bv1, sv2, bv2;
    load_sb(0, sv1, bv1);
    load_sb(1, sv2, bv2);
    int seg = 0, pend_seg = -1, pend_tile = 0;
    bool pend_whole = false;
    for (int n = 0; n < nunits; ++n) {
      const int unit = lo + n, tile = unit / C;
      const int slot = n % kWdCodeRing;
      sv0 = sv1;
      bv0 = bv1;
      sv1 = sv2;
      bv1 = bv2;
      load_sb(n + 2, sv2, bv2);
      wait(cfull + slot, (n / kWdCodeRing) & 1);
      const uint32_t box = code + (uint32_t)slot * kSlotBytes + (uint32_t)r * 128u;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int g = u + 2 * h, i = 4 * n + g, sl = i % kWdRing;
        const uint4 wa = ld_shared_v4(box + ((uint32_t)((2 * g) ^ rsw) << 4));
        const uint4 wb = ld_shared_v4(box + ((uint32_t)((2 * g + 1) ^ rsw) << 4));
        if (h == 1) {  // this warp has read the box: its loads before the copy that refills it
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(cempty + slot);
        }
        const uint32_t sw = h ? sv0.y : sv0.x, bw = h ? bv0.y : bv0.x;  // groups u, u + 2
        const uint16_t sh = (uint16_t)(u ? sw >> 16 : sw & 0xFFFFu);
        const uint16_t bh = (uint16_t)(u ? bw >> 16 : bw & 0xFFFFu);
        const __half2 s2 = __halves2half2(__ushort_as_half(sh), __ushort_as_half(sh));
        const __half2 b2 = __halves2half2(__ushort_as_half(bh), __ushort_as_half(bh));
        const __half2 k1024 = __half2half2(__ushort_as_half(0x6400u));
        const uint32_t wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
        if (i >= kWdRing) wait(gdone + sl, ((i / kWdRing) - 1) & 1);  // its previous MMAs are done
        tmem_fence_after();
#pragma unroll
        for (int half = 0; half < 2; ++half) {  // 4 words = 64 codes = 32 columns per store
          uint32_t A[32];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const uint32_t w = wv[4 * half + jj];
#pragma unroll
            for (int p = 0; p < 8; ++p) {
              // pair p of the word: codes p and p + 8 as 1024 + q (exact), then s*q + b (one rounding)
              const uint32_t qv = lop3_and_or(w >> (2 * p), 0x00030003u, 0x64006400u);
              const __half2 qh = __hsub2(*reinterpret_cast<const __half2*>(&qv), k1024);
              const __half2 wh = __hfma2(qh, s2, b2);
              A[8 * jj + p] = *reinterpret_cast<const uint32_t*>(&wh);
            }
          }
          tmem_st32(tmem + (uint32_t)(sl * 64 + 32 * half) + lane_off, A);
        }
        tmem_wait_st();
        tmem_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(afull + sl);
        // the previous segment's accumulator, once this unit's first group is on its way
        if (u == 0 && h == 0 && pend_seg >= 0) {
          finish_segment(pend_seg, pend_tile, pend_whole);
          pend_seg = -1;
        }
      }
      if (seg_end(unit)) {
        pend_seg = seg;
        pend_tile = tile;
        const int first_unit = (unit / C) * C > lo ? (unit / C) * C : lo;
        pend_whole = first_unit == tile * C && unit == tile * C + C - 1;
        ++seg;
      }
    }
    if (u == 0 && pend_seg >= 0) finish_segment(pend_seg, pend_tile, pend_whole);
  }

  // every MMA has completed (the issuer waited for its last commit) and every load from tensor
  // memory has returned: give the columns back
  tmem_fence_before();
  __syncthreads();
  if (warp == 1) {
    tmem_fence_after();
    tmem_dealloc(tmem, kWdTmemCols);
  }
}

template <int MT>
static int launch_wide_mt(const CUtensorMap& cmap, const CUtensorMap& xmap, const WideArgs& a, int grid,
                          int smem_optin, int device, cudaStream_t s) {
  constexpr int bytes = wide_layout<MT>().total;
  if (bytes > smem_optin) return TB_ERR_UNSUPPORTED;
  const int rc = ensure_dynamic_smem(reinterpret_cast<const void*>(w2_gemv_wide_kernel<MT>), device, bytes);
  if (rc != TB_OK) return rc;
  cudaError_t e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kWdThreads);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, w2_gemv_wide_kernel<MT>, cmap, xmap, a);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return TB_ERR_CUDA;
  }
  return TB_OK;
}

// Bytes of fp32 parts the wide GEMV needs (slots of 128 rows x 64 tokens for up to 256 SMs).
size_t gemv_wide_part_bytes() { return (size_t)256 * 2 * kUnitRows * 64 * 4; }

// The batched-decode GEMV on x' already rotated into pair order (fp16 [M, K], xp), for 9 <= M
// <= 64 tokens in one pass.  `count` is 1 KB of zeroed counters (left zero), `part` scratch of
// gemv_wide_part_bytes().  TB_ERR_UNSUPPORTED where it does not apply.
int launch_gemv_wide(const __half* xp, int64_t M, int64_t K, const uint32_t* w, const __half* scales,
                     const __half* biases, int64_t N, __half* y, int* count, float* part, int32_t* status,
                     cudaStream_t s) {
  if (M < 1 || M > 64 || K < kBlock || K % kBlock || K > (1 << 22) || N < 1 || N > (1LL << 30))
    return TB_ERR_UNSUPPORTED;
  DeviceFacts f;
  int rc = device_facts(&f);
  if (rc != TB_OK) return rc;
  if (f.sms > 256) return TB_ERR_UNSUPPORTED;
  const int64_t tiles = (N + kUnitRows - 1) / kUnitRows;
  const int C = (int)(K / (kUnitGroups * kGroup));
  if (tiles * C > (int64_t)INT32_MAX / 2) return TB_ERR_SHAPE;
  const int MT = M <= 16 ? 16 : M <= 32 ? 32 : M <= 48 ? 48 : 64;
  CUtensorMap cmap, xmap;
  rc = code_map(w, N, K, &cmap);
  if (rc != TB_OK) return rc;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)MT};
    const cuuint32_t estr[2] = {1, 1};
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return TB_ERR_CUDA;
    if (encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(xp), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return TB_ERR_CUDA;
  }
  WideArgs a = {};
  a.w = w;
  a.scales = scales;
  a.biases = biases;
  a.y = y;
  a.part = part;
  a.count = count;
  a.M = (int)M;
  a.N = (int)N;
  a.K = (int)K;
  a.G = (int)(K / kGroup);
  a.C = C;
  a.n_tiles = (int)tiles;
  a.status = status;
  const int64_t S = tiles * C;
  const int grid = (int)(S < f.sms ? S : f.sms);
  switch (MT) {
    case 16: return launch_wide_mt<16>(cmap, xmap, a, grid, f.smem_optin, f.device, s);
    case 32: return launch_wide_mt<32>(cmap, xmap, a, grid, f.smem_optin, f.device, s);
    case 48: return launch_wide_mt<48>(cmap, xmap, a, grid, f.smem_optin, f.device, s);
    default: return launch_wide_mt<64>(cmap, xmap, a, grid, f.smem_optin, f.device, s);
  }
}

}  // namespace tb
