// Prefill path of the Packed layer: tcgen05 / TMEM tensor-core GEMM on packed W2-g128 weights.
//
// [ARCH] kwkr.cn/news/564617, section "Hadamard 旋转把量化误差抹平的免费午餐": the same
// Packed.__call__ (fwht on the activations, then quantized_matmul with group 128,
// 2 bits, transpose) at M = prompt length.  Ternary codes times an fp16 scale plus
// the fp16 bias -s give {-s, 0, s}, exact in fp16, so fp16 tensor-core operands lose
// nothing on the weight side.
//
// y[M, N] = x'[M, K] . W[N, K]^T with
//   A = x' (fp16, written by the rotate kernel into the workspace, TMA-loaded with the
//       128-byte swizzle), tile 128 tokens x 64 k;
//   B = W decoded in shared memory by 8 decoder warps straight from the packed words
//       (never materialised in global memory), tile 256 rows x 64 k, written in the
//       same K-major 128-byte-swizzled layout the UMMA descriptor reads;
//   D = fp32 accumulator, 128 x 256, in tensor memory (256 columns).
// Warp roles: warp 0 issues the TMA loads, warp 1 owns TMEM and issues tcgen05.mma
// (one thread), warps 2..9 decode B and afterwards drain TMEM to fp16 y.
// A 4-stage mbarrier ring couples the three roles; every wait is bounded.
#include <cuda.h>
#include <algorithm>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "tb_common.cuh"
#include "tb_host.h"

namespace tb {

constexpr int kTcBM = 128, kTcBK = 64;  // token subtile, k per stage
// 12 warps: 0 loads the activations, 1 issues the MMAs, 2-4, 6-8, 10-11 decode the weights and
// 4-11 drain the accumulator (two per tensor-memory lane quarter, which warp w may read as
// w % 4).  Warps 5 and 9 only drain, so the MMA warp shares its SM sub-partition (w % 4 == 1)
// with no decoder: its issue loop sets the k-block rate.
constexpr int kTcThreads = 384;
constexpr int kTcABytes = kTcBM * kTcBK * 2;  // 16 KB

// K-major operand in the 128-byte swizzle: 8-row core groups 1024 bytes apart.
TB_DEVI uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);  // start address
  d |= (uint64_t)1u << 16;                  // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024u >> 4) << 32;        // stride byte offset: next 8-row group
  d |= (uint64_t)1u << 46;                  // descriptor version (tcgen05)
  d |= (uint64_t)2u << 61;                  // 128-byte swizzle
  return d;
}


TB_DEVI void tma_load_2d(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// the same box into the shared memory of every CTA of the cluster in `mask` (same offset), each
// CTA's barrier at `bar`'s offset receiving the complete_tx of its copy
TB_DEVI void tma_load_2d_mc(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* bar, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar)), "h"(mask)
      : "memory");
}

TB_DEVI uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// every thread of every CTA of the cluster (release / acquire)
TB_DEVI void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

TB_DEVI void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
TB_DEVI void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

TB_DEVI void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}

TB_DEVI void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// one arrival on the barrier at `bar`'s offset in every CTA of `mask` once this thread's earlier
// tcgen05 operations are complete
TB_DEVI void tc_commit_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}

TB_DEVI void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

TB_DEVI void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// one packed word (codes k..k+15) -> 8 half2 (s*q_p + b, s*q_{p+8} + b), p = 0..7
TB_DEVI void decode_word_affine(uint32_t w, __half2 s2, __half2 b2, uint32_t (&o)[8]) {
  const __half2 k1024 = __half2half2(__ushort_as_half(0x6400u));
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const uint32_t v = lop3_and_or(w >> (2 * p), 0x00030003u, 0x64006400u);
    const __half2 q = __hsub2(*reinterpret_cast<const __half2*>(&v), k1024);  // exact {0,1,2,3}
    const __half2 r = __hfma2(q, s2, b2);
    o[p] = *reinterpret_cast<const uint32_t*>(&r);
  }
}

// NSUB M-subtiles of 128 tokens share every decoded B tile (NSUB = 2: 256 tokens per CTA,
// the decode cost per flop halves).  Stage s holds A[sub] (16 KB each), then B decoded
// (BN x 64 fp16).
template <int NSUB, int BN>
struct TcCfg {
  static constexpr int kBBytes = BN * kTcBK * 2;
  static constexpr int kStageBytes = NSUB * kTcABytes + kBBytes;
  // three 64 KB stages for two subtiles (two measured up to 15 % slower at long K, where the
  // activations come from HBM), 160 KB for one subtile: the rest of the SM memory stays L1,
  // which the decoders' word loads hit
  static constexpr int kStages = ((NSUB == 2 ? 192 : 160) * 1024) / kStageBytes;
  static constexpr int kEpiBytes = 8 * 32 * 64;  // per drain warp: 32 rows x 32 fp16 of y
  // packed words of one k-block (BN rows x 16 bytes) per slot, loaded by TMA four k-blocks ahead
  static constexpr int kWSlots = 4;
  static constexpr int kWBytes = BN * 16;
  static constexpr int kSmem = kStages * kStageBytes + 1024 + kEpiBytes + kWSlots * kWBytes + 1024;
  // stages, barriers, y staging, word ring, alignment
  static constexpr int kTmemCols = NSUB * BN;
  // kind::f16 instruction descriptor: fp16 A and B, fp32 D, both K-major, M = 128, N = BN
  static constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(kTcBM >> 4) << 24);
  static constexpr int kThreadsPerRow = 256 / BN;  // decoder threads per B row
};

// Stream-K schedule: the units (output tile, 64-k block) of all tiles, tile-major, are cut
// into one equal contiguous range per CTA (one persistent CTA per SM).  A CTA walks its range
// as segments (runs of k-blocks of one tile); a segment that covers its whole tile is written
// to y directly, one that covers part of it goes as fp32 to this CTA's workspace slot, and the
// last of the tile's CTAs to count in adds the parts in CTA order and writes y.  A grid of at
// most one CTA per tile splits a tile between two CTAs at most; a grid of q CTAs per tile
// splits every tile into q equal k-ranges; one CTA per tile splits nothing.
struct TcSkArgs {
  const uint32_t* w;     // [N, K/16]
  const __half* scales;  // [N, G]
  const __half* biases;  // [N, G]
  __half* y;             // [M, N]
  int M, N, K, G;
  int tiles_n, nkb;      // tile t = (t / tiles_n) token tile, (t % tiles_n) row tile
  int tiles_np;          // row tiles per token tile in steps of the cluster size (= tiles_n for one)
  int units;             // (token tiles * tiles_np) * nkb: the schedule's units are a cluster's
  float* part;           // [grid][2][BN/4][NSUB*128][4] fp32 parts of split tiles (scratch)
  int* count;            // [tiles] claims of split tiles, then at done_off [tiles] parts written
                         // (both zero before a call and after it)
  int done_off;
  int32_t* status;
};

TB_DEVI int sk_owner(int u, int units, int grid) { return (int)(((int64_t)(u + 1) * grid - 1) / units); }
TB_DEVI int sk_lo(int c, int units, int grid) { return (int)((int64_t)units * c / grid); }

// CS = 1: one CTA per schedule slot.  CS = 2 (two 128-token subtiles): a cluster of two CTAs
// takes one token tile and k-range on two neighbouring row tiles; each CTA loads one subtile of
// every activation stage and multicasts it to both, so each SM reads half the activation bytes,
// and a stage is refilled only when the MMAs of both CTAs have read it.
template <int NSUB, int BN, int CS>
__global__ void __launch_bounds__(kTcThreads, 1)
    w2_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                      const TcSkArgs a) {
  static_assert(CS == 1 || (CS == 2 && NSUB == 2), "a cluster pair shares two token subtiles");
  using Cfg = TcCfg<NSUB, BN>;
  constexpr int S = Cfg::kStages;
  constexpr int kPartFloats = NSUB * kTcBM * BN;
  // a part is stored as [BN / 4 column quads][NSUB * 128 rows][4]: the 32 threads of a warp hold
  // 32 consecutive rows, so each of their 16-byte stores and loads covers 512 contiguous bytes
  constexpr int kPartRows = NSUB * kTcBM;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * Cfg::kStageBytes);
  // full[s]: the stage's activations have landed (expect_tx by the producer) and its weights are
  // decoded (one arrival per decoder warp), so the MMA warp waits once per k-block
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* accum = bars + 2 * S;      // one phase per segment: its accumulator is complete
  uint64_t* tfree = bars + 2 * S + 1;  // one phase per segment: its accumulator has been read
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 2);
  // word ring: wfull[j % 4] when k-block j's packed words have landed, wempty when every decoder
  // warp has read them
  constexpr int kWS = Cfg::kWSlots;
  uint64_t* wfull = bars + 2 * S + 3;
  uint64_t* wempty = wfull + kWS;
  uint8_t* wring = smem + S * Cfg::kStageBytes + 1024 + Cfg::kEpiBytes;
  // the split-tile fixup of a CTA's last segment streams the other parts through the idle stage
  // ring: six 32 KB slots, filled by bulk copies (pfull) and released by the eight drain warps
  constexpr int kFixSlots = 6;
  constexpr bool kBulkFix = NSUB == 2 && BN == 256;
  static_assert(!kBulkFix || kFixSlots * 32 * 2 * kTcBM * 4 <= S * Cfg::kStageBytes, "fixup slots fit the ring");
  uint64_t* pfull = wempty + kWS;
  uint64_t* pempty = pfull + kFixSlots;
  __shared__ volatile int aborted;
  __shared__ int last_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int crank = CS > 1 ? (int)cluster_rank() : 0;  // row tile within the cluster's pair
  const int cid = (int)blockIdx.x / CS;                 // the schedule works in clusters
  const int nkb = a.nkb, units = a.units, grid = (int)gridDim.x / CS;
  const int lo = sk_lo(cid, units, grid), hi = sk_lo(cid + 1, units, grid);

  if (threadIdx.x == 0) {
    aborted = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(full + s, 1 + 8);
      mbar_init(empty + s, CS);  // the MMAs of every CTA that reads the stage
    }
    mbar_init(accum, 1);
    mbar_init(tfree, 8);  // lane 0 of each of the 8 drain warps
    for (int i = 0; i < kWS; ++i) {
      mbar_init(wfull + i, 1);
      mbar_init(wempty + i, 8);  // lane 0 of each decoder warp
    }
    for (int i = 0; i < kFixSlots; ++i) {
      mbar_init(pfull + i, 1);
      mbar_init(pempty + i, 8);  // lane 0 of each drain warp
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(Cfg::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CS > 1) cluster_sync();  // the peer's barriers exist before anything lands in them
  tc_fence_after();
  const uint32_t tmem_d = *tmem_slot;

  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity) || aborted) return;  // the common case costs one test
    if (!mbar_wait(bar, parity)) {
      aborted = 1;
      set_status(a.status, TB_DEV_TIMEOUT);
    }
  };
  // segment starting at unit u: the cluster's tile t (token tile t / tiles_np), k-blocks [k0, k1)
  auto segment = [&](int u, int& t, int& k0, int& k1) {
    t = u / nkb;
    k0 = u - t * nkb;
    k1 = min(nkb, k0 + (hi - u));
  };

  if (warp == 0) {
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
      // the packed words of the CTA's k-block j (unit lo + j): its row tile's 16 bytes per row
      const int nblk = hi - lo;
      auto issue_words = [&](int j) {
        const int u = lo + j, tt = u / nkb, kb = u - tt * nkb;
        const int nt = (tt % a.tiles_np) * CS + crank;
        const int sl = j % kWS;
        mbar_arrive_expect_tx(wfull + sl, Cfg::kWBytes);
        tma_load_2d(wring + sl * Cfg::kWBytes, &tmW, kb * 4, nt * BN, wfull + sl);
      };
      for (int j = 0; j < kWS && j < nblk; ++j) issue_words(j);  // the weights need no wait
      // x' is the previous kernel's output (programmatic launch): everything before this, and the
      // decoders' first stages, overlap that kernel's tail
      asm volatile("griddepcontrol.wait;" ::: "memory");
      int it = 0;
      for (int u = lo; u < hi;) {
        int t, k0, k1;
        segment(u, t, k0, k1);
        const int m0 = (t / a.tiles_np) * (NSUB * kTcBM);
        for (int kb = k0; kb < k1; ++kb, ++it) {
          const int s = it % S, ph = it / S;
          if (ph > 0) wait(empty + s, (ph - 1) & 1);
          mbar_arrive_expect_tx(full + s, NSUB * kTcABytes);
          if constexpr (CS == 1) {
#pragma unroll
            for (int sub = 0; sub < NSUB; ++sub)
              tma_load_2d(smem + s * Cfg::kStageBytes + sub * kTcABytes, &tmA, kb * kTcBK,
                          m0 + sub * kTcBM, full + s);
          } else {
            tma_load_2d_mc(smem + s * Cfg::kStageBytes + crank * kTcABytes, &tmA, kb * kTcBK,
                           m0 + crank * kTcBM, full + s, (uint16_t)((1u << CS) - 1u));
          }
          const int jw = it + kWS;  // the words four k-blocks ahead, once their slot is read
          if (jw < nblk) {
            wait(wempty + jw % kWS, (jw / kWS - 1) & 1);
            issue_words(jw);
          }
        }
        u += k1 - k0;
      }
      if constexpr (CS > 1) {
        // the peer's last commits into this CTA's barriers have landed before the cluster exits
        for (int s = 0; s < S && s < it; ++s) {
          const int last = it - 1 - ((it - 1 - s) % S);  // the last k-block that used stage s
          wait(empty + s, (last / S) & 1);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      int it = 0, seg = 0;
      for (int u = lo; u < hi; ++seg) {
        int t, k0, k1;
        segment(u, t, k0, k1);
        if (seg > 0) wait(tfree, (seg - 1) & 1);  // the previous segment's accumulator is read
        tc_fence_after();
        for (int kb = k0; kb < k1; ++kb, ++it) {
          const int s = it % S, ph = it / S;
          wait(full + s, ph & 1);
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * Cfg::kStageBytes);
          const uint64_t bd = umma_desc_sw128(sa + NSUB * kTcABytes);
#pragma unroll
          for (int k = 0; k < kTcBK / 16; ++k)
#pragma unroll
            for (int sub = 0; sub < NSUB; ++sub)
              tc_mma(tmem_d + sub * BN, umma_desc_sw128(sa + sub * kTcABytes) + 2 * k, bd + 2 * k,
                     Cfg::kIdesc, (kb != k0) || (k != 0));
          if constexpr (CS > 1) tc_commit_mc(empty + s, (uint16_t)((1u << CS) - 1u));
          else tc_commit(empty + s);
        }
        tc_commit(accum);
        u += k1 - k0;
      }
    }
    __syncwarp();
  } else {
    // ---- decoders: thread d owns (part of) row n0 + d % BN of the B tile ----
    const bool is_dec = warp != 5 && warp != 9;
    const bool is_epi = warp >= 4;
    const int dt = (warp - 2 - (warp > 5) - (warp > 9)) * 32 + lane;  // decoder thread 0..255
    constexpr int WPT = 4 / Cfg::kThreadsPerRow;  // packed words per thread per k-block
    const int d = dt % BN;
    const int wq = (dt / BN) * WPT;          // first word of this thread
    const int q = warp & 3;                 // TMEM lane quarter this warp may read
    const int part = (warp - 4) >> 2;       // which half of the columns / which subtile
    const int sub = NSUB == 2 ? part : 0;
    const int c0 = NSUB == 2 ? 0 : part * (BN / 2);
    const int lrow = sub * kTcBM + q * 32 + lane;  // token row within the tile
    const uint32_t epi = smem_u32(smem + S * Cfg::kStageBytes + 1024) + (uint32_t)(warp - 4) * 2048u;
    int it = 0, seg = 0;
    for (int u = lo; u < hi; ++seg) {
      int t, k0, k1;
      segment(u, t, k0, k1);
      const int nt = (t % a.tiles_np) * CS + crank;  // this CTA's row tile
      const bool has_tile = nt < a.tiles_n;           // false: the partner of an odd last row tile
      const int n0 = nt * BN, m0 = (t / a.tiles_np) * (NSUB * kTcBM);
      const int tile = (t / a.tiles_np) * a.tiles_n + nt;  // its count slot when split
      const int row = n0 + d;
      const bool valid = is_dec && row < a.N;  // the drain-only warps load nothing
      const __half* srow = a.scales + (int64_t)(valid ? row : 0) * a.G;
      // no biases given: each is the pack's -scale (the fp16 sign bit flipped), not read
      const bool has_b = a.biases != nullptr;
      const __half* brow = has_b ? a.biases + (int64_t)(valid ? row : 0) * a.G : nullptr;
      // scales and biases of eight groups (16 k-blocks) per load, the next eight loaded while
      // these are used: the loads go to HBM when the weights are read once
      const bool vec8 = (a.G % 8) == 0;
      auto load_sb8 = [&](int gb, uint4& sv, uint4& bv) {
        if (valid && vec8 && 8 * gb < a.G) {
          sv = __ldg(reinterpret_cast<const uint4*>(srow) + gb);
          bv = has_b ? __ldg(reinterpret_cast<const uint4*>(brow) + gb)
                     : make_uint4(sv.x ^ 0x80008000u, sv.y ^ 0x80008000u, sv.z ^ 0x80008000u,
                                  sv.w ^ 0x80008000u);
        } else {
          uint16_t hs[8], hb[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const bool in = valid && 8 * gb + e < a.G;
            hs[e] = in ? __half_as_ushort(srow[8 * gb + e]) : 0;
            hb[e] = !in ? 0 : has_b ? __half_as_ushort(brow[8 * gb + e]) : (uint16_t)(hs[e] ^ 0x8000u);
          }
          sv = make_uint4(hs[0] | (uint32_t)hs[1] << 16, hs[2] | (uint32_t)hs[3] << 16,
                          hs[4] | (uint32_t)hs[5] << 16, hs[6] | (uint32_t)hs[7] << 16);
          bv = make_uint4(hb[0] | (uint32_t)hb[1] << 16, hb[2] | (uint32_t)hb[3] << 16,
                          hb[4] | (uint32_t)hb[5] << 16, hb[6] | (uint32_t)hb[7] << 16);
        }
      };
      auto pick = [](const uint4& v, int g) {  // fp16 number g (0..7) of eight
        const uint32_t w2 = (g >> 2) ? ((g >> 1) & 1 ? v.w : v.z) : ((g >> 1) & 1 ? v.y : v.x);
        return __ushort_as_half((uint16_t)((g & 1) ? (w2 >> 16) : (w2 & 0xFFFFu)));
      };
      uint4 s_cur, b_cur, s_nxt, b_nxt;
      load_sb8(k0 >> 4, s_cur, b_cur);
      load_sb8((k0 >> 4) + 1, s_nxt, b_nxt);
      for (int kb = k0; kb < (is_dec ? k1 : k0); ++kb, ++it) {
        const int s = it % S, ph = it / S;
        // this row's packed words of the k-block from the word ring (rows past N are zeros)
        const int wsl = it % kWS;
        wait(wfull + wsl, (it / kWS) & 1);
        uint32_t wv[WPT];
        const uint32_t wa = smem_u32(wring + wsl * Cfg::kWBytes) + (uint32_t)(d * 16 + wq * 4);
        if constexpr (WPT == 4) {
          const uint4 v = ld_shared_v4(wa);
          wv[0] = v.x;
          wv[1] = v.y;
          wv[2] = v.z;
          wv[3] = v.w;
        } else {
          const uint2 v = ld_shared_v2(wa);
          wv[0] = v.x;
          wv[1] = v.y;
        }
        if (ph > 0) wait(empty + s, (ph - 1) & 1);
        const uint32_t stage = smem_u32(smem + s * Cfg::kStageBytes);
        const int g = (kb >> 1) & 7;
        const __half sv = pick(s_cur, g), bv = pick(b_cur, g);
        const uint32_t bt = stage + NSUB * kTcABytes + d * 128;
        const uint32_t sw = d & 7;
#pragma unroll
        for (int jj = 0; jj < WPT; ++jj) {
          const int j = wq + jj;  // word of the row's 64-k slice: 16-byte chunks 2j, 2j+1
          uint32_t o[8];
          decode_word_affine(wv[jj], __half2half2(sv), __half2half2(bv), o);  // a row past N gives 0
          sts128(bt + (((2 * j) ^ sw) << 4), o[0], o[1], o[2], o[3]);
          sts128(bt + (((2 * j + 1) ^ sw) << 4), o[4], o[5], o[6], o[7]);
        }
        // this thread's stores before the tensor core reads them, and its reads of the word slot
        // before the copy engine refills it (generic accesses, then async-proxy ones)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(full + s);
          mbar_arrive(wempty + wsl);
        }
        if ((kb & 15) == 15) {  // the next k-block starts a new block of eight groups
          s_cur = s_nxt;
          b_cur = b_nxt;
          load_sb8((kb >> 4) + 2, s_nxt, b_nxt);
        }
      }

      if (is_epi) {
        // ---- epilogue of the segment: TMEM -> fp16 y; a split tile goes through the parts ----
        wait(accum, seg & 1);
        tc_fence_after();
        const bool whole = k0 == 0 && k1 == nkb;
        constexpr int CW = NSUB == 2 ? BN : BN / 2;  // columns this thread drains
        // 32 accumulator columns (from c) of the warp's 32 token rows to fp16 y, staged through
        // the warp's 2 KB of shared memory so that four lanes write each row's 64 contiguous bytes
        // (16-byte slot s of row r sits at slot s ^ ((r >> 1) & 3): conflict-free both ways).
        // Warp-collective: every lane calls it.
        auto store_y = [&](int c, const float (&f)[32]) {
          const int n = n0 + c0 + c;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t h[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) h[e] = pack_half2(f[8 * v + 2 * e], f[8 * v + 2 * e + 1]);
            sts128(epi + (uint32_t)(lane * 4 + (v ^ ((lane >> 1) & 3))) * 16u, h[0], h[1], h[2], h[3]);
          }
          __syncwarp();
          const int tok0 = m0 + sub * kTcBM + q * 32;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = 8 * i + (lane >> 2), v = lane & 3;
            const int tk = tok0 + r, col = n + 8 * v;
            if (tk < a.M && col < a.N) {
              const uint4 o = ld_shared_v4(epi + (uint32_t)(r * 4 + (v ^ ((r >> 1) & 3))) * 16u);
              __half* dst = a.y + (int64_t)tk * a.N + col;
              if ((a.N % 8) == 0 && col + 8 <= a.N) {
                *reinterpret_cast<uint4*>(dst) = o;
              } else {
                const __half* hv = reinterpret_cast<const __half*>(&o);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  if (col + e < a.N) dst[e] = hv[e];
              }
            }
          }
          __syncwarp();
        };
        auto tmem_cols = [&](int c, float (&f)[32]) {
          uint32_t r[32];
          tc_ld32(tmem_d + ((uint32_t)(q * 32) << 16) + (uint32_t)(sub * BN + c0 + c), r);
#pragma unroll
          for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(r[e]);
        };
        if (!has_tile) {
          // the partner of an odd last row tile computed zeros: nothing to write
        } else if (whole) {
#pragma unroll 1
          for (int c = 0; c < CW; c += 32) {
            float f[32];
            tmem_cols(c, f);
            store_y(c, f);
          }
        } else {
          // A split tile: each contributor claims a turn as its accumulator completes.  The last
          // to claim adds the parts in CTA order (its own from tensor memory, never written out),
          // so the sum does not depend on the order of arrival, and writes y; the others write
          // their parts and count them done.  The last claimer waits only for CTAs that claimed
          // before it: those are running and have nothing left to do but write their parts.
          const int first = sk_owner(t * nkb, units, grid);
          const int lastc = sk_owner(t * nkb + nkb - 1, units, grid);
          int* done = a.count + a.done_off + tile;
          if (threadIdx.x == 128) last_flag = atomicAdd(a.count + tile, 1) == lastc - first;  // warp 4, lane 0
          asm volatile("bar.sync 2, 256;" ::: "memory");
          if (!last_flag) {
            float* mine = a.part + ((int64_t)blockIdx.x * 2 + (u == lo ? 0 : 1)) * kPartFloats;
#pragma unroll 1
            for (int c = 0; c < CW; c += 32) {
              float f[32];
              tmem_cols(c, f);
              float4* dst = reinterpret_cast<float4*>(mine) + (int64_t)((c0 + c) / 4) * kPartRows + lrow;
#pragma unroll
              for (int v = 0; v < 8; ++v)
                __stcg(dst + v * kPartRows, make_float4(f[4 * v], f[4 * v + 1], f[4 * v + 2], f[4 * v + 3]));
            }
            // every writer fences its own stores: the barrier orders them only within the CTA
            fence_acq_rel_gpu();
            asm volatile("bar.sync 2, 256;" ::: "memory");
            if (threadIdx.x == 128) atomicAdd(done, 1);
          } else {
            if (threadIdx.x == 128) {
              const uint64_t t0 = globaltimer_ns();
              while (ld_acquire_gpu(reinterpret_cast<const uint32_t*>(done)) != (uint32_t)(lastc - first)) {
                if (globaltimer_ns() - t0 > TB_WAIT_NS) {
                  aborted = 1;
                  set_status(a.status, TB_DEV_TIMEOUT);
                  break;
                }
              }
              a.count[tile] = 0;
              *done = 0;
            }
            asm volatile("bar.sync 2, 256;" ::: "memory");
          }
          if (last_flag) {
            fence_acq_rel_gpu();  // each reader's acquire of the counted parts
            const int me = cid;  // contributors are counted in clusters; cluster cc's CTA of this row tile
            if (kBulkFix && u + (k1 - k0) >= hi) {
              // Last segment: no stage is loaded again and every MMA is complete, so the ring
              // holds the other contributors' parts, 32 columns of one part per slot, in the order
              // they are added (chunk by chunk, contributors in CTA order).
              constexpr uint32_t kSlotBytes = 32u * kPartRows * 4u;
              const int nothers = lastc - first;
              const int ncopy = (CW / 32) * nothers;
              auto issue = [&](int j) {  // copy j: chunk j / nothers of the (j % nothers)-th other
                const int i = j % nothers, cc = first + i + (first + i >= me ? 1 : 0);
                const int slot = sk_lo(cc, units, grid) / nkb == t ? 0 : 1;
                const float* src = a.part + ((int64_t)(cc * CS + crank) * 2 + slot) * kPartFloats +
                                   (int64_t)((c0 + (j / nothers) * 32) / 4) * kPartRows * 4;
                const int sl = j % kFixSlots;
                mbar_arrive_expect_tx(pfull + sl, kSlotBytes);
                bulk_g2s(smem + sl * kSlotBytes, src, kSlotBytes, pfull + sl);
              };
              if (threadIdx.x == 128) {
                asm volatile("fence.proxy.async.global;" ::: "memory");  // parts read by the copy engine
                for (int j = 0; j < ncopy && j < kFixSlots; ++j) issue(j);
              }
              int j = 0;
#pragma unroll 1
              for (int c = 0; c < CW; c += 32) {
                float f[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) f[e] = 0.f;
                for (int cc = first; cc <= lastc; ++cc) {
                  if (cc == me) {
                    float m[32];
                    tmem_cols(c, m);
#pragma unroll
                    for (int e = 0; e < 32; ++e) f[e] += m[e];
                    continue;
                  }
                  const int sl = j % kFixSlots;
                  wait(pfull + sl, (j / kFixSlots) & 1);
                  const uint32_t src = smem_u32(smem + sl * kSlotBytes) + (uint32_t)lrow * 16u;
#pragma unroll
                  for (int v = 0; v < 8; ++v) {
                    const uint4 o = ld_shared_v4(src + (uint32_t)(v * kPartRows * 16));
                    f[4 * v] += __uint_as_float(o.x);
                    f[4 * v + 1] += __uint_as_float(o.y);
                    f[4 * v + 2] += __uint_as_float(o.z);
                    f[4 * v + 3] += __uint_as_float(o.w);
                  }
                  fence_proxy_async_smem();  // these loads before the copy that refills the slot
                  __syncwarp();
                  if (lane == 0) mbar_arrive(pempty + sl);
                  if (threadIdx.x == 128 && j + kFixSlots < ncopy) {
                    wait(pempty + sl, (j / kFixSlots) & 1);  // all eight warps have read the slot
                    issue(j + kFixSlots);
                  }
                  __syncwarp();  // converged again before the next tensor-memory load
                  ++j;
                }
                store_y(c, f);
              }
            } else {
              auto load_part = [&](int cc, int c, float4 (&o)[8]) {
                const int slot = sk_lo(cc, units, grid) / nkb == t ? 0 : 1;
                const float4* op = reinterpret_cast<const float4*>(
                                       a.part + ((int64_t)(cc * CS + crank) * 2 + slot) * kPartFloats) +
                                   (int64_t)((c0 + c) / 4) * kPartRows + lrow;
#pragma unroll
                for (int v = 0; v < 8; ++v) o[v] = __ldcg(op + v * kPartRows);
              };
              auto add_part = [](float (&f)[32], const float4 (&o)[8]) {
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                  f[4 * v] += o[v].x;
                  f[4 * v + 1] += o[v].y;
                  f[4 * v + 2] += o[v].z;
                  f[4 * v + 3] += o[v].w;
                }
              };
#pragma unroll 1
              for (int c = 0; c < CW; c += 32) {
                float f[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) f[e] = 0.f;
                // the parts in CTA order, its own from tensor memory (one part in flight: two measured
                // no faster and hold 30 more registers across the whole kernel)
                for (int cc = first; cc <= lastc; ++cc) {
                  if (cc == me) {
                    float m[32];
                    tmem_cols(c, m);
#pragma unroll
                    for (int e = 0; e < 32; ++e) f[e] += m[e];
                  } else {
                    float4 A[8];
                    load_part(cc, c, A);
                    add_part(f, A);
                  }
                }
                store_y(c, f);
              }
            }
          }
        }
        // the accumulator is read: the next segment's first mma may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tfree);
      }
      u += k1 - k0;
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (CS > 1) cluster_sync();  // nothing of the peer's still lands in this CTA
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_d),
                 "r"(Cfg::kTmemCols)
                 : "memory");
  }
}

int launch_rotate_pairorder(const __half* x, __half* out, const int8_t* signs, int64_t M,
                            int64_t K, int rotate, cudaStream_t s);

// Workspace of the tensor-core path (after the caller's fixup region):
//   x'      fp16 [M, K], rotated activations;
//   counts  int32 per output tile of the smallest tile shape (128 x 128), zero before a call
//           and after it;
//   parts   fp32 [SMs][2][256 x 256], the stream-K parts of split tiles (scratch).
static int64_t tc_sms_bound() {
  DeviceFacts f;
  return device_facts(&f) == TB_OK ? f.sms : 256;  // no device: the largest SM count supported
}
static size_t rup256(size_t v) { return (v + 255) / 256 * 256; }
static size_t tc_x_bytes(int64_t M, int64_t K) { return rup256((size_t)M * (size_t)K * 2); }
// two int32 counters per output tile of the smallest tile shape (claims, parts written)
static int64_t tc_count_tiles(int64_t M, int64_t N) { return ((M + kTcBM - 1) / kTcBM) * ((N + 127) / 128); }
static size_t tc_count_bytes(int64_t M, int64_t N) { return rup256((size_t)tc_count_tiles(M, N) * 2 * 4); }
static size_t tc_part_bytes() { return (size_t)tc_sms_bound() * 2 * (2 * kTcBM) * 256 * 4; }

size_t gemm_tc_x_bytes(int64_t M, int64_t K) { return tc_x_bytes(M, K); }

// offset of the parts region inside the tensor-core path's workspace (after x' and the counts)
size_t gemm_tc_part_offset(int64_t M, int64_t K, int64_t N) { return tc_x_bytes(M, K) + tc_count_bytes(M, N); }

size_t gemm_tc_workspace(int64_t M, int64_t K, int64_t N) {
  return tc_x_bytes(M, K) + tc_count_bytes(M, N) + tc_part_bytes();
}

template <int NS, int B, int CS>
static cudaError_t launch_tc(int grid, const CUtensorMap& tm, const CUtensorMap& tw, const TcSkArgs& a,
                             cudaStream_t s) {
  constexpr int smem = TcCfg<NS, B>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(w2_gemm_tc_kernel<NS, B, CS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see griddepcontrol.wait
  at[0].val.programmaticStreamSerializationAllowed = 1;
  at[1].id = cudaLaunchAttributeClusterDimension;
  at[1].val.clusterDim.x = CS;
  at[1].val.clusterDim.y = 1;
  at[1].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = CS > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, w2_gemm_tc_kernel<NS, B, CS>, tm, tw, a);
}

// How many two-CTA clusters of the 256 x 256 kernel can be resident at once on the current
// device (0: none, or the query failed: the pair schedule is not used).
static int64_t tc_resident_pairs() {
  static int cached[64];
  static bool known[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (known[dev]) return cached[dev];
  int n = 0;
  constexpr int smem = TcCfg<2, 256>::kSmem;
  if (cudaFuncSetAttribute(w2_gemm_tc_kernel<2, 256, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ==
      cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, w2_gemm_tc_kernel<2, 256, 2>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
  } else {
    (void)cudaGetLastError();
  }
  cached[dev] = n;
  known[dev] = true;
  return n;
}

// the GEMM alone, on x' already rotated into pair order in xp (fp16 [M, K]); `gws` is the
// workspace after x' (counts, then parts)
int launch_gemm_tc_rotated(const __half* xp, int64_t M, int64_t K, const uint32_t* w,
                           const __half* scales, const __half* biases, int64_t N, __half* y,
                           void* gws, int32_t* status, cudaStream_t s) {
  if (M > 0x7fffffffLL || N > 0x7fffffffLL || K > (1 << 24)) return TB_ERR_SHAPE;

  CUtensorMap tm;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kTcBK, (cuuint32_t)kTcBM};
  const cuuint32_t estr[2] = {1, 1};
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return TB_ERR_CUDA;
  CUresult cr = encode(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(xp), dims, strides,
                                       box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                       CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return TB_ERR_CUDA;

  // Tile shape and schedule.  Above 128 tokens: 256 x 256 tiles (two 128-token subtiles share
  // each decoded weight tile, which halves the decode work and the activation reads per flop
  // of smaller tiles; the per-k-block decode then hides behind the k-block's mma), taken by
  // clusters of two CTAs on neighbouring row tiles that share each activation stage (one
  // multicast load per CTA) when pairs can be resident; as stream-K over the resident slots
  // (CTAs or pairs) when every slot gets a tile, one slot per tile when the tiles fill most of
  // the slots, else every tile split into q <= 4 k-ranges.  Up to 128 tokens: 128 x 256 tiles the
  // same way, or 128 x 128 tiles when those keep more SMs busy (the cost of a k-block grows with
  // the tile's rows, so the count of SMs in use sets the time when tokens are few).
  DeviceFacts f;
  int rcf = device_facts(&f);
  if (rcf != TB_OK) return rcf;
  if (f.sms > 256) return TB_ERR_TOO_LARGE;
  const int64_t sms = f.sms;
  auto tiles = [&](int ns, int b) { return ((M + ns * kTcBM - 1) / (ns * kTcBM)) * ((N + b - 1) / b); };
  int nsub = 1, bn = 256, cs = 1;
  int64_t grid64 = 0;  // in schedule slots (clusters of cs CTAs); 0: one slot per tile
  const int64_t full = sms * 4 / 5;
  const int64_t nkb0 = K / kTcBK;  // a split never leaves a CTA without a k-block
  const int64_t tiles_n = (N + 255) / 256;
  if (M > kTcBM) {
    nsub = 2;
    const int64_t pairs = tiles_n >= 2 ? tc_resident_pairs() : 0;
    cs = pairs > 0 ? 2 : 1;
    const int64_t slots = cs == 2 ? pairs : sms;
    const int64_t T2 = ((M + 2 * kTcBM - 1) / (2 * kTcBM)) * ((tiles_n + cs - 1) / cs);
    if (T2 >= slots) grid64 = slots;  // stream-K, two slots per tile at most
    else if (T2 < slots * 4 / 5) grid64 = T2 * std::min<int64_t>(std::min<int64_t>(4, nkb0), slots / T2);
  } else if (tiles(1, 256) >= sms) { grid64 = sms; }
  else if (tiles(1, 256) >= full) {}
  else {  // few tiles: the tile width (256 or 128 rows, split into q <= 4 k-ranges, or one CTA
          // per tile when they fill most of the SMs) that keeps the most SMs busy, 256 on a tie
    const int64_t T256 = tiles(1, 256), T128 = tiles(1, 128);
    const int64_t g256 = T256 * std::min<int64_t>(std::min<int64_t>(4, nkb0), sms / T256);
    const int64_t g128 = T128 >= full ? std::min<int64_t>(T128, sms)
                                      : T128 * std::min<int64_t>(std::min<int64_t>(4, nkb0), sms / T128);
    if (g128 > g256) {
      bn = 128;
      grid64 = T128 >= sms ? sms : T128 >= full ? 0 : g128;
    } else {
      grid64 = g256;
    }
  }
  const int64_t tn = (N + bn - 1) / bn, tnp = (tn + cs - 1) / cs;
  const int64_t T = ((M + nsub * kTcBM - 1) / (nsub * kTcBM)) * tnp;  // schedule tiles
  const int64_t nkb = K / kTcBK;
  if (T * nkb > 0x7fffffffLL) return TB_ERR_SHAPE;
  const int grid = (int)((grid64 ? grid64 : T) * cs);
  TcSkArgs a;
  a.w = w;
  a.scales = scales;
  a.biases = biases;
  a.y = y;
  a.M = (int)M;
  a.N = (int)N;
  a.K = (int)K;
  a.G = (int)(K / kGroup);
  a.tiles_n = (int)tn;
  a.tiles_np = (int)tnp;
  a.nkb = (int)nkb;
  a.units = (int)(T * nkb);
  a.count = static_cast<int*>(gws);
  a.done_off = (int)tc_count_tiles(M, N);
  a.part = reinterpret_cast<float*>(static_cast<char*>(gws) + tc_count_bytes(M, N));
  a.status = status;
  // the packed words [N][K/16] as a 2-D tensor: one box = one k-block (4 words) of bn rows
  CUtensorMap tw;
  {
    const cuuint64_t wd[2] = {(cuuint64_t)(K / 16), (cuuint64_t)N};
    const cuuint64_t wst[1] = {(cuuint64_t)(K / 16) * 4};
    const cuuint32_t wbox[2] = {4, (cuuint32_t)bn};
    cr = encode(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(w), wd, wst, wbox, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return TB_ERR_CUDA;
  }
  cudaError_t e;
  if (nsub == 2 && cs == 2) e = launch_tc<2, 256, 2>(grid, tm, tw, a, s);
  else if (nsub == 2) e = launch_tc<2, 256, 1>(grid, tm, tw, a, s);
  else if (bn == 256) e = launch_tc<1, 256, 1>(grid, tm, tw, a, s);
  else e = launch_tc<1, 128, 1>(grid, tm, tw, a, s);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return TB_ERR_CUDA;
  }
  return check_launch();
}

int launch_gemm_tc(const __half* x, int64_t M, int64_t K, const int8_t* signs, int block,
                   const uint32_t* w, const __half* scales, const __half* biases, int64_t N,
                   __half* y, void* workspace, int32_t* status, cudaStream_t s) {
  if (M > 0x7fffffffLL || N > 0x7fffffffLL || K > (1 << 24)) return TB_ERR_SHAPE;
  __half* xp = static_cast<__half*>(workspace);
  int rc = launch_rotate_pairorder(x, xp, signs, M, K, block != 0, s);
  if (rc != TB_OK) return rc;
  return launch_gemm_tc_rotated(xp, M, K, w, scales, biases, N, y,
                                static_cast<char*>(workspace) + tc_x_bytes(M, K), status, s);
}

}  // namespace tb
