// Chained decode: a sequence of Packed linears (M <= 8 tokens) in one persistent launch.
//
// [ARCH] kwkr.cn/news/564617, section "Hadamard 旋转把量化误差抹平的免费午餐": every linear of
// the stack is the module's forward pass (rotate the input, then the W2-g128 matmul); a decode
// step runs them one after another, each reading what the ones before it wrote.  [PACK]
// lpnh.cn/news/2438023, section "文本模型加载artifact.load_model 与 Packed 模块": the modules
// and their packed tensors.
//
// Link i of the chain is what tb_packed_linear_multi does for one input x_i and up to four
// matrices that read it.  Link i + 1 may read the outputs of link i (or of any earlier link):
// the consumers of every CTA read x_{i+1} only after all CTAs have counted link i complete on
// a device-wide counter (release by each CTA after its outputs of link i are written, acquire
// before the prologue of link i + 1), which is the ordering a stream gives between launches.
//
// What the chain saves over one launch per link is the boundary between launches: the
// producer warp of each CTA streams the packed weights of link i + 1 into its ring while the
// consumers still finish link i, wait for the other CTAs and transform x_{i+1}; the weights
// never depend on the activations.  Per link the work is the same as in the per-call decode
// GEMV: the units (128 rows x 512 k, one 16 KB TMA box) of all row tiles of the link are cut
// into one equal contiguous range per CTA and each range into three sub-ranges, one per group
// of four consumer warps; tiles cut by a group boundary are summed in shared memory, tiles cut
// by a CTA boundary through per-CTA fp32 parts in the workspace, added in CTA order by the
// last contributor.
//
// The plan (tb_chain_plan) holds, in device memory written once by the host: a header, one
// CUtensorMap per matrix (the TMA descriptor of its codes, read by the copies straight from
// global memory) and one ChainLink per link.
#include <cstddef>
#include <cuda.h>
#include <cuda_runtime.h>
#include <string.h>

#include <vector>

#include "tb_common.cuh"
#include "tb_gemv_core.cuh"
#include "tb_host.h"

namespace tb {

int code_map(const uint32_t* w, int64_t N, int64_t K, CUtensorMap* out);
int group_map(const __half* p, int64_t N, int64_t G, CUtensorMap* out);

// ring slot: a unit's code box, then the scales and the biases of its 128 rows for its chunk and
// the neighbouring one (TMA boxes of 8 groups: a tensor copy's inner extent is at least 16 bytes)
constexpr int kChSbBox = kUnitRows * 8 * 2;
constexpr int kChSlot = kSlotBytes + 2 * kChSbBox;
constexpr int kChMapsPerMat = 3;  // codes, scales, biases (the scales' map again without biases)

constexpr uint32_t kChainMagic = 0x54424348u;  // "TBCH"
constexpr int kChainMaxCtas = 256;                // parts slots of the fixup region
constexpr int64_t kChainMaxTokens = 8;
constexpr int64_t kChainMaxK = 1 << 20;
// Units per unit group that the producer streams into a link before the consumers have
// loaded that link's activations: the loads of x wait behind the weight copies in flight.
constexpr int kChainPreIssue = 1;

struct ChainLink {
  const __half* x;                // [Mc, K]
  const int8_t* signs;            // [K] or null
  const __half* scales[kMaxMats];  // [N_i, G]
  const __half* biases[kMaxMats];
  __half* y[kMaxMats];            // [Mc, N_i]
  int N[kMaxMats];
  int tile0[kMaxMats + 1];        // first 128-row tile of matrix i in the link's tile list
  int nmat, K, G, C, rotate, n_tiles, map0, pad;
};

struct ChainHeader {
  uint32_t magic;
  int32_t n_links, M, max_K;
  int64_t maps_off, links_off, bytes;
  int64_t wait_ns;      // limit of each wait on the previous link, ns of %globaltimer (0: TB_WAIT_NS)
  int32_t extra_count;  // added to the count each link waits for (0; > 0 only to test the timeout)
  int32_t pad0;
  int64_t pad1;
};
static_assert(sizeof(ChainHeader) == 64, "header size");

// Workspace: [fixup counters, 1 KiB][link counter, CTA exit counter, 256 B]
//            [per-CTA fp32 parts of shared tiles: kChainMaxCtas x 2 x 128 rows x 8 tokens]
constexpr size_t kChainCounterBytes = 1024;
constexpr size_t kChainSyncBytes = 256;
constexpr size_t kChainPartBytes = (size_t)kChainMaxCtas * 2 * kUnitRows * 8 * 4;
size_t chain_workspace_bytes() { return kChainCounterBytes + kChainSyncBytes + kChainPartBytes; }

struct ChainRun {
  const CUtensorMap* maps;
  const ChainHeader* header;
  int n_links, Mc, max_K, dw;
  int preissue;        // units per group the producer issues into a link before its x is loaded
  int* ws_count;       // [kChainMaxCtas] contributions per shared tile (zero between links)
  uint32_t* sync;      // [0] links completed, summed over CTAs; [1] CTAs finished
  float* ws_partial;   // [kChainMaxCtas][2][128][MT]
  int32_t* status;
};

TB_DEVI int link_mat_of(const int (&tile0)[kMaxMats + 1], int nmat, int tile) {
  int i = 0;
#pragma unroll
  for (int k = 1; k < kMaxMats; ++k) i += (k < nmat && tile >= tile0[k]);
  return i;
}

// same, reading the link's tile table from the plan (used only when a tile starts or ends)
TB_DEVI int link_mat_of_g(const ChainLink* lk, int tile, int& tile0_of) {
  const int nmat = __ldg(&lk->nmat);
  int i = 0;
#pragma unroll
  for (int k = 1; k < kMaxMats; ++k) i += (k < nmat && tile >= __ldg(&lk->tile0[k]));
  tile0_of = __ldg(&lk->tile0[i]);
  return i;
}

// This CTA's unit range [lo, hi) of a link with n_tiles row tiles of C units each, and the
// group boundaries in it.  With at least one unit per CTA the units are cut into equal ranges
// (stream-K; no range is empty, so every CTA between the first and the last owner of a tile
// contributes to it); with fewer, every tile goes whole to one CTA and the other CTAs idle.
struct LinkRange {
  int lo, hi, bnd1, bnd2;
};
TB_DEVI LinkRange link_range(int n_tiles, int C) {
  LinkRange r;
  const int S = n_tiles * C;
  if (S >= (int)gridDim.x) {
    r.lo = (int)((int64_t)S * blockIdx.x / gridDim.x);
    r.hi = (int)((int64_t)S * (blockIdx.x + 1) / gridDim.x);
  } else {
    r.lo = C * (int)((int64_t)n_tiles * blockIdx.x / gridDim.x);
    r.hi = C * (int)((int64_t)n_tiles * (blockIdx.x + 1) / gridDim.x);
  }
  const int nst = r.hi - r.lo;
  r.bnd1 = r.lo + nst / 3;
  r.bnd2 = r.lo + (2 * nst) / 3;
  return r;
}
TB_DEVI void link_group_range(const LinkRange& r, int u, int& glo, int& ghi) {
  glo = u == 0 ? r.lo : u == 1 ? r.bnd1 : r.bnd2;
  ghi = u == 0 ? r.bnd1 : u == 1 ? r.bnd2 : r.hi;
}

// Warp roles: warps 0..11 consume (three unit groups of four), warp 12 produces; warps 13..15
// only complete the producer's warpgroup so that registers can move between the roles: the
// launch gives 128 per thread, the producer warpgroup drops to 56 and the consumers rise to 152
// (12 x 32 x 152 + 4 x 32 x 56 = 65536, the block's whole launch allocation).  At 128 registers
// for every warp the consumers spilled and a decode step took 6 % longer.
constexpr int kChainThreads = 16 * 32;
template <int MT>
__global__ void __launch_bounds__(kChainThreads, 1) w2_gemv_chain_kernel(const __grid_constant__ ChainRun a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int DW = a.dw;
  const GemvTmaLayout L = gemv_tma_layout<MT>(a.max_K / kGroup, DW, kChSlot);
  const uint32_t slots_u32 = smem_u32(smem + L.codes);
  __half* img = reinterpret_cast<__half*>(smem + L.img);
  float2* cs = reinterpret_cast<float2*>(smem + L.cs);
  float* accs = reinterpret_cast<float*>(smem + L.accs);  // [kCutSlots][128][MT]
  int* cnt = reinterpret_cast<int*>(smem + L.cnt);         // [kCutSlots]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + kGroupsOfWarps * DW;
  uint64_t* xready = empty + kGroupsOfWarps * DW;  // one phase per link: its x is loaded
  __shared__ volatile int aborted;

  // a plan that does not match the launch: every CTA returns before any wait
  const ChainHeader* hdr = a.header;
  if (hdr->magic != kChainMagic || hdr->n_links != a.n_links || hdr->M != a.Mc || hdr->max_K > a.max_K) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(a.status, TB_DEV_BAD_PLAN);
    return;
  }
  const ChainLink* links =
      reinterpret_cast<const ChainLink*>(reinterpret_cast<const uint8_t*>(hdr) + hdr->links_off);

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

  if (warp >= kTmaConsumers) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 56;" ::: "memory");
    if (warp != kTmaConsumers) return;
    // ---- producer: streams the codes of every link in order; never waits for a link's input
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int si[kGroupsOfWarps] = {0, 0, 0};  // ring position (fill index % DW) of each group
      int kf[kGroupsOfWarps] = {0, 0, 0};  // fills of that slot so far (fill index / DW)
      for (int li = 0; li < a.n_links; ++li) {
        const ChainLink* lk = links + li;
        const int C = lk->C, nmat = lk->nmat;
        int tile0[kMaxMats + 1];
#pragma unroll
        for (int k = 0; k <= kMaxMats; ++k) tile0[k] = lk->tile0[k];
        const CUtensorMap* maps = a.maps + kChMapsPerMat * lk->map0;
        const LinkRange r = link_range(lk->n_tiles, C);
        int tl[kGroupsOfWarps], ch[kGroupsOfWarps], cntu[kGroupsOfWarps];
        int maxcnt = 0;
#pragma unroll
        for (int u = 0; u < kGroupsOfWarps; ++u) {
          int glo, ghi;
          link_group_range(r, u, glo, ghi);
          cntu[u] = ghi - glo;
          const int first = u == kGroupsOfWarps - 1 ? ghi - 1 : glo;
          tl[u] = cntu[u] > 0 ? first / C : 0;
          ch[u] = cntu[u] > 0 ? first - tl[u] * C : 0;
          maxcnt = cntu[u] > maxcnt ? cntu[u] : maxcnt;
        }
        for (int n = 0; n < maxcnt; ++n) {
          if (n == a.preissue) wait(xready, li & 1);  // this link's x has been read
#pragma unroll
          for (int u = 0; u < kGroupsOfWarps; ++u) {
            if (n >= cntu[u]) continue;
            const int slot = u * DW + si[u];
            if (kf[u] > 0) wait(empty + slot, (kf[u] - 1) & 1);
            const int mi = link_mat_of(tile0, nmat, tl[u]);
            const int row = (tl[u] - tile0[mi]) * kUnitRows;
            const bool hb = lk->biases[mi] != nullptr;
            mbar_arrive_expect_tx(full + slot, kSlotBytes + (hb ? 2 : 1) * kChSbBox);
            const uint32_t dst = slots_u32 + slot * kChSlot;
            const CUtensorMap* mm = maps + kChMapsPerMat * mi;
            tma2d(dst, mm, ch[u] * 32, row, full + slot, pol);
            tma2d(dst + kSlotBytes, mm + 1, 8 * (ch[u] >> 1), row, full + slot, pol);
            if (hb) tma2d(dst + kSlotBytes + kChSbBox, mm + 2, 8 * (ch[u] >> 1), row, full + slot, pol);
            step_unit(tl[u], ch[u], C, u == kGroupsOfWarps - 1);
            if (++si[u] == DW) {
              si[u] = 0;
              ++kf[u];
            }
          }
        }
        // every phase of xready is waited for in order (a parity wait tells apart only the
        // current phase and the one before it)
        if (maxcnt <= a.preissue) wait(xready, li & 1);
      }
      // leave no copy in flight: wait (bounded, even after a timeout) for the last fill of
      // every slot that was filled
#pragma unroll
      for (int u = 0; u < kGroupsOfWarps; ++u) {
        const int total = kf[u] * DW + si[u];
        for (int n = total - 1; n >= 0 && n >= total - DW; --n)
          if (!mbar_wait(full + u * DW + n % DW, (n / DW) & 1)) set_status(a.status, TB_DEV_TIMEOUT);
      }
    }
    __syncwarp();
    return;
  }

  // ---- consumers ----
  asm volatile("setmaxnreg.inc.sync.aligned.u32 152;" ::: "memory");
  const int g = lane >> 2, t = lane & 3;
  const int ug = warp / kWarpsPerUnit, wi = warp % kWarpsPerUnit;
  const bool back = ug == kGroupsOfWarps - 1;
  const int rA = 2 * (g & 3) + (g >> 2);  // mma row g <-> unit row 32*wi + 16*j + rA (and + 8)
  const int R0 = 32 * wi + rA;
  const int tokc = g < MT ? g : 0;
  const uint32_t imgt = smem_u32(img) + tokc * 64 + t * 16;
  const uint32_t csa = smem_u32(cs);
  const uint32_t accs_u32 = smem_u32(accs);
  const int t0 = min(2 * t, MT - 1), t1 = min(2 * t + 1, MT - 1);
  const uint32_t ss = smem_u32(smem + L.sstage) + warp * kScaleStageBytes;
  const int Mc = a.Mc;
  int si = 0;       // ring slot of the group's next unit within its DW slots
  uint32_t ph = 0;  // its fill parity

  for (int li = 0; li < a.n_links; ++li) {
    const ChainLink* lk = links + li;
    const int C = lk->C, K = lk->K;
    const int S = lk->n_tiles * C;
    const LinkRange r = link_range(lk->n_tiles, C);
    // everything the prologue needs but x itself is read before the wait on the previous link
    const __half* lx = lk->x;
    const int8_t* lsg = lk->signs;
    const int lrot = lk->rotate;
    int b1, e1, b2, e2;
    blocks_needed(r.lo, r.hi - r.lo, C, K, b1, e1, b2, e2);
    if (lsg) {
      const int nblk = (e1 - b1) + (e2 - b2);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int it = warp + q * kTmaConsumers;
        if (it < Mc * nblk) {
          const int bi = it % nblk;
          const int b = bi < e1 - b1 ? b1 + bi : b2 + (bi - (e1 - b1));
          asm volatile("prefetch.global.L1 [%0];" ::"l"(lsg + b * kBlock + lane * 32));
        }
      }
    }
    int glo, ghi;
    link_group_range(r, ug, glo, ghi);
    const int ncnt = ghi - glo;
    int tile = 0, chunk = 0;
    if (ncnt > 0) {
      const int first = back ? ghi - 1 : glo;
      tile = first / C;
      chunk = first - tile * C;
    }

    // x of this link may be an output of the previous one: wait until every CTA has
    // counted that link complete
    if (li > 0) {
      if (threadIdx.x == 0 && !aborted) {
        const uint32_t target = (uint32_t)li * gridDim.x + (uint32_t)hdr->extra_count;
        const uint64_t limit = hdr->wait_ns > 0 ? (uint64_t)hdr->wait_ns : TB_WAIT_NS;
        if (ld_acquire_gpu(a.sync) < target) {
          const uint64_t t_0 = globaltimer_ns();
          while (ld_acquire_gpu(a.sync) < target) {
            if (globaltimer_ns() - t_0 > limit) {
              aborted = 1;
              set_status(a.status, TB_DEV_TIMEOUT);
              break;
            }
          }
        }
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kTmaConsumers * 32) : "memory");
    }
    {
      // scratch of the transform: the slot after the one that holds this group's first unit
      // of the link; the producer fills it only after every consumer warp has arrived on
      // xready for this link
      const uint32_t scratch = slots_u32 + (ug * DW + (si + 1 == DW ? 0 : si + 1)) * kChSlot + wi * 4096;
      prologue_image<MT>(lx, lsg, K, Mc, lrot, b1, e1, b2, e2, warp, kTmaConsumers, lane, img, cs, scratch);
    }
    fence_proxy_async_smem();  // the scratch's generic accesses before the copies that refill it
    __syncwarp();
    if (lane == 0) mbar_arrive(xready);  // the producer may stream on into this link
    asm volatile("bar.sync 1, %0;" ::"n"(kTmaConsumers * 32) : "memory");

    // Add this warp's sums of tile T (all of the group's units of T) to wherever T is finished.
    auto flush = [&](int T, float (&acc)[2][4]) {
      int t0m;
      const int mi = link_mat_of_g(lk, T, t0m);
      const int N = lk->N[mi], row0 = (T - t0m) * kUnitRows;
      __half* yo = lk->y[mi];
      const int tb = T * C, te = tb + C;
      if (tb >= glo && te <= ghi) {  // the whole tile is this group's: these 32 rows are final
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int ra = row0 + R0 + 16 * j, rb = ra + 8;
          if (2 * t < Mc) {
            if (ra < N) yo[(int64_t)(2 * t) * N + ra] = __float2half_rn(acc[j][0]);
            if (rb < N) yo[(int64_t)(2 * t) * N + rb] = __float2half_rn(acc[j][2]);
          }
          if (2 * t + 1 < Mc) {
            if (ra < N) yo[(int64_t)(2 * t + 1) * N + ra] = __float2half_rn(acc[j][1]);
            if (rb < N) yo[(int64_t)(2 * t + 1) * N + rb] = __float2half_rn(acc[j][3]);
          }
        }
        return;
      }
      // a tile cut by a boundary: its shared slot is the first boundary that falls in it
      const int b = (r.lo / C == T) ? 0 : (r.bnd1 / C == T) ? 1 : (r.bnd2 / C == T) ? 2 : 3;
      int groups = 0;  // contributions expected in this CTA: 4 warps of every group meeting T
#pragma unroll
      for (int u = 0; u < kGroupsOfWarps; ++u) {
        int ulo, uhi;
        link_group_range(r, u, ulo, uhi);
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
      // this warp finishes the tile for this CTA, and returns the slot to zero for the next link
      __threadfence_block();
      float* at = accs + b * kUnitRows * MT;
      if (lane == 0) cnt[b] = 0;
      if (tb >= r.lo && te <= r.hi) {
        for (int e = lane; e < kUnitRows * MT; e += 32) {
          const int r_ = e / MT, k_ = e - r_ * MT;
          if (row0 + r_ < N && k_ < Mc) yo[(int64_t)k_ * N + row0 + r_] = __float2half_rn(at[e]);
          at[e] = 0.f;
        }
        return;
      }
      // shared with other CTAs: this CTA's part to its own workspace slot (slot 0 for the tile
      // of its first unit, 1 for the tile of its last)
      float* mine = a.ws_partial + ((int64_t)blockIdx.x * 2 + (r.lo / C == T ? 0 : 1)) * kUnitRows * MT;
      for (int e = lane; e < kUnitRows * MT; e += 32) {
        __stcg(mine + e, at[e]);
        at[e] = 0.f;
      }
      __syncwarp();
      // the last of the tile's CTAs to count in adds the parts in CTA order and returns the
      // counter to zero
      const int first = stage_owner(tb, S, gridDim.x);
      const int lastc = stage_owner(te - 1, S, gridDim.x);
      int fin = 0;
      if (lane == 0) {
        fence_acq_rel_gpu();
        fin = atomicAdd(a.ws_count + first, 1) == lastc - first;
      }
      fin = __shfl_sync(0xffffffffu, fin, 0);
      if (!fin) return;
      fence_acq_rel_gpu();
      int flo, fhi;
      cta_range_of(first, gridDim.x, lk->n_tiles, C, flo, fhi);
      const float* p0 = a.ws_partial + ((int64_t)first * 2 + (flo / C == T ? 0 : 1)) * kUnitRows * MT;
      for (int eb = 0; eb < kUnitRows * MT; eb += 128) {
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        for (int c = first; c <= lastc; c += 4) {
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
          if (row0 + r_ < N && k_ < Mc) yo[(int64_t)k_ * N + row0 + r_] = __float2half_rn(v[k]);
        }
      }
      if (lane == 0) a.ws_count[first] = 0;
    };

    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    int hb_tile = -1;
    bool has_b = true;
    auto body = [&](int n) {
      const int slot = ug * DW + si;
      wait(full + slot, ph);
      if (++si == DW) {
        si = 0;
        ph ^= 1;
      }
      const uint32_t box = slots_u32 + slot * kChSlot;
      {  // this warp's 32 rows' (s, b) of the unit's four groups, from the slot, as fp32 pairs
        if (tile != hb_tile) {  // whether the tile's matrix has biases, looked up per tile
          hb_tile = tile;
          int t0m;
          has_b = lk->biases[link_mat_of_g(lk, tile, t0m)] != nullptr;
        }
        const uint32_t sp = box + kSlotBytes + (32 * wi + lane) * 16 + (chunk & 1) * 8;
        const uint2 sv = ld_shared_v2(sp);
        // no biases given: each is the pack's -scale (the fp16 sign bit flipped)
        const uint2 bv = has_b ? ld_shared_v2(sp + kChSbBox) : make_uint2(sv.x ^ 0x80008000u, sv.y ^ 0x80008000u);
        const uint32_t rr = ss + lane * kUnitGroups * 8;
        const float2 sf0 = __half22float2(*reinterpret_cast<const __half2*>(&sv.x));
        const float2 sf1 = __half22float2(*reinterpret_cast<const __half2*>(&sv.y));
        const float2 bf0 = __half22float2(*reinterpret_cast<const __half2*>(&bv.x));
        const float2 bf1 = __half22float2(*reinterpret_cast<const __half2*>(&bv.y));
        asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(rr), "f"(sf0.x), "f"(bf0.x), "f"(sf0.y), "f"(bf0.y) : "memory");
        asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(rr + 16), "f"(sf1.x), "f"(bf1.x), "f"(sf1.y), "f"(bf1.y) : "memory");
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

    // every output of this link from this CTA is written: count the link complete (a release
    // reduction: the CTA's writes, ordered before it by the barrier, become visible first; the
    // thread does not wait for a returned value)
    asm volatile("bar.sync 1, %0;" ::"n"(kTmaConsumers * 32) : "memory");
    if (threadIdx.x == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(a.sync) : "memory");
  }

  // the last CTA to finish returns both counters to zero for the next launch (every CTA has
  // passed its last wait on the link counter before it counts itself finished)
  if (threadIdx.x == 0) {
    fence_acq_rel_gpu();
    if (atomicAdd(a.sync + 1, 1u) == gridDim.x - 1) {
      atomicExch(a.sync, 0u);
      atomicExch(a.sync + 1, 0u);
    }
  }
}

// ------------------------------------------------------------------ host side
static size_t plan_bytes_for(int n_links, int n_maps) {
  return sizeof(ChainHeader) + 64 + (size_t)n_maps * kChMapsPerMat * sizeof(CUtensorMap) +
         (size_t)n_links * sizeof(ChainLink);
}

static int tokens_per_pass(int64_t M) { return M >= 5 ? 8 : M >= 3 ? 4 : M == 2 ? 2 : 1; }

template <int MT>
static int chain_slots(int max_K, int smem_optin) {
  int dw = kMaxSlotsPerGroup;
  while (dw >= 2 && gemv_tma_layout<MT>(max_K / kGroup, dw, kChSlot).total > smem_optin) --dw;
  return dw >= 2 ? dw : 0;
}

static int chain_slots_for(int mt, int max_K, int smem_optin) {
  switch (mt) {
    case 8: return chain_slots<8>(max_K, smem_optin);
    case 4: return chain_slots<4>(max_K, smem_optin);
    case 2: return chain_slots<2>(max_K, smem_optin);
    default: return chain_slots<1>(max_K, smem_optin);
  }
}

template <int MT>
static int launch_chain_mt(const ChainRun& a, int grid, cudaStream_t s) {
  const int bytes = gemv_tma_layout<MT>(a.max_K / kGroup, a.dw, kChSlot).total;
  cudaError_t e = cudaFuncSetAttribute(w2_gemv_chain_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return TB_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kChainThreads);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident at once: CTAs wait on each other
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, w2_gemv_chain_kernel<MT>, a);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return TB_ERR_CUDA;
  }
  return TB_OK;
}

}  // namespace tb

using namespace tb;

extern "C" size_t tb_chain_plan_size(int n_links) {
  if (n_links < 1) return 0;
  return plan_bytes_for(n_links, n_links * kMaxMats);
}

extern "C" size_t tb_chain_workspace_size(void) { return chain_workspace_bytes(); }

extern "C" int tb_chain_plan(const tb_chain_link* links, int n_links, int64_t M, void* plan,
                             size_t plan_bytes, void* stream) {
  if (!links || !plan) return TB_ERR_NULL;
  if (n_links < 1 || M < 1) return TB_ERR_SHAPE;
  if (M > kChainMaxTokens) return TB_ERR_TOO_LARGE;
  if (reinterpret_cast<uintptr_t>(plan) & 127u) return TB_ERR_ALIGN;
  int n_maps = 0;
  int64_t max_K = 0;
  for (int i = 0; i < n_links; ++i) {
    const tb_chain_link& l = links[i];
    if (l.block != 0 && l.block != kBlock) return TB_ERR_UNSUPPORTED;
    if (!l.x) return TB_ERR_NULL;
    if (l.n < 1 || l.n > kMaxMats) return TB_ERR_SHAPE;
    if (l.K < kBlock || l.K % kBlock || l.K > kChainMaxK) return TB_ERR_SHAPE;
    if (!aligned16(l.x) || (l.signs && !aligned16(l.signs))) return TB_ERR_ALIGN;
    int64_t tiles = 0;
    for (int j = 0; j < l.n; ++j) {
      if (!l.w[j] || !l.scales[j] || !l.y[j]) return TB_ERR_NULL;  // biases may be NULL
      if (l.N[j] < 1 || l.N[j] > (1LL << 30)) return TB_ERR_SHAPE;
      if (!aligned16(l.w[j]) || !aligned16(l.scales[j]) || !aligned16(l.y[j]) ||
          (l.biases[j] && !aligned16(l.biases[j])))
        return TB_ERR_ALIGN;
      tiles += (l.N[j] + kUnitRows - 1) / kUnitRows;
    }
    if (tiles * (l.K / (kUnitGroups * kGroup)) > (int64_t)INT32_MAX / 2) return TB_ERR_SHAPE;
    n_maps += l.n;
    max_K = l.K > max_K ? l.K : max_K;
  }
  const size_t need = plan_bytes_for(n_links, n_maps);
  if (plan_bytes < need) return TB_ERR_WORKSPACE;

  std::vector<uint8_t> host(need, 0);
  ChainHeader h = {};
  h.magic = kChainMagic;
  h.n_links = n_links;
  h.M = (int32_t)M;
  h.max_K = (int32_t)max_K;
  h.maps_off = 128;  // 128-byte aligned tensor maps (a TMA descriptor needs 64)
  h.links_off = h.maps_off + (int64_t)n_maps * kChMapsPerMat * sizeof(CUtensorMap);
  h.bytes = (int64_t)need;
  memcpy(host.data(), &h, sizeof(h));
  CUtensorMap* maps = reinterpret_cast<CUtensorMap*>(host.data() + h.maps_off);
  int map = 0;
  for (int i = 0; i < n_links; ++i) {
    const tb_chain_link& l = links[i];
    ChainLink d = {};
    d.x = reinterpret_cast<const __half*>(l.x);
    d.signs = l.block ? l.signs : nullptr;
    int64_t tiles = 0;
    for (int j = 0; j < kMaxMats; ++j) {
      if (j < l.n) {
        CUtensorMap* mm = &maps[kChMapsPerMat * (map + j)];
        int rc = code_map(l.w[j], l.N[j], l.K, mm);
        if (rc == TB_OK) rc = group_map(reinterpret_cast<const __half*>(l.scales[j]), l.N[j], l.K / kGroup, mm + 1);
        if (rc == TB_OK && l.biases[j])
          rc = group_map(reinterpret_cast<const __half*>(l.biases[j]), l.N[j], l.K / kGroup, mm + 2);
        if (!l.biases[j]) mm[2] = mm[1];
        if (rc != TB_OK) return rc;
        d.scales[j] = reinterpret_cast<const __half*>(l.scales[j]);
        d.biases[j] = reinterpret_cast<const __half*>(l.biases[j]);
        d.y[j] = reinterpret_cast<__half*>(l.y[j]);
        d.N[j] = (int)l.N[j];
        d.tile0[j] = (int)tiles;
        tiles += (l.N[j] + kUnitRows - 1) / kUnitRows;
      } else {
        d.tile0[j] = (int)tiles;
      }
    }
    d.tile0[kMaxMats] = (int)tiles;
    d.nmat = l.n;
    d.K = (int)l.K;
    d.G = (int)(l.K / kGroup);
    d.C = (int)(l.K / (kUnitGroups * kGroup));
    d.rotate = l.block != 0;
    d.n_tiles = (int)tiles;
    d.map0 = map;
    memcpy(host.data() + h.links_off + (size_t)i * sizeof(ChainLink), &d, sizeof(d));
    map += l.n;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(plan, host.data(), need, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);  // the host image is freed on return
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return TB_ERR_CUDA;
  }
  return TB_OK;
}

extern "C" int tb_chain_set_wait(void* plan, int64_t wait_ns, int32_t extra_count, void* stream) {
  if (!plan) return TB_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(plan) & 127u) return TB_ERR_ALIGN;
  if (wait_ns < 0 || extra_count < 0) return TB_ERR_VALUE;
  struct {
    int64_t wait_ns;
    int32_t extra_count;
  } f = {wait_ns, extra_count};
  static_assert(offsetof(ChainHeader, extra_count) == offsetof(ChainHeader, wait_ns) + 8, "header fields");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(static_cast<uint8_t*>(plan) + offsetof(ChainHeader, wait_ns), &f, 12,
                                  cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);  // `f` lives on this stack frame
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return TB_ERR_CUDA;
  }
  return TB_OK;
}

extern "C" int tb_chain_run(const void* plan, int n_links, int64_t M, int64_t max_K, void* workspace,
                            size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (!plan) return TB_ERR_NULL;
  if (n_links < 1 || M < 1 || max_K < kBlock || max_K % kBlock || max_K > kChainMaxK) return TB_ERR_SHAPE;
  if (M > kChainMaxTokens) return TB_ERR_TOO_LARGE;
  if (reinterpret_cast<uintptr_t>(plan) & 127u) return TB_ERR_ALIGN;
  if (!workspace || workspace_bytes < chain_workspace_bytes()) return TB_ERR_WORKSPACE;
  if (!aligned16(workspace)) return TB_ERR_ALIGN;
  DeviceFacts f;
  int rc = device_facts(&f);
  if (rc != TB_OK) return rc;
  if (f.sms > kChainMaxCtas) return TB_ERR_TOO_LARGE;
  const int mt = tokens_per_pass(M);
  const int dw = chain_slots_for(mt, (int)max_K, f.smem_optin);
  if (dw == 0) return TB_ERR_TOO_LARGE;
  const uint8_t* p = static_cast<const uint8_t*>(plan);
  ChainRun a = {};
  a.header = reinterpret_cast<const ChainHeader*>(p);
  a.maps = reinterpret_cast<const CUtensorMap*>(p + 128);  // the links follow the maps (header)
  a.n_links = n_links;
  a.Mc = (int)M;
  a.max_K = (int)max_K;
  a.dw = dw;
  a.preissue = kChainPreIssue;
  char* ws = static_cast<char*>(workspace);
  a.ws_count = reinterpret_cast<int*>(ws);
  a.sync = reinterpret_cast<uint32_t*>(ws + kChainCounterBytes);
  a.ws_partial = reinterpret_cast<float*>(ws + kChainCounterBytes + kChainSyncBytes);
  a.status = dev_status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (mt) {
    case 8: return launch_chain_mt<8>(a, f.sms, s);
    case 4: return launch_chain_mt<4>(a, f.sms, s);
    case 2: return launch_chain_mt<2>(a, f.sms, s);
    default: return launch_chain_mt<1>(a, f.sms, s);
  }
}
