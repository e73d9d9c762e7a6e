// Decode path of the Packed layer: fused sign*FWHT prologue + W2-g128 GEMV.
//
// [ARCH] kwkr.cn/news/564617, section "Hadamard 旋转把量化误差抹平的免费午餐":
//   a folded module first rotates its input (sign flip, then the normalised block Hadamard
//   transform) and then multiplies it by the 2-bit, group-128 affine weights, which stay
//   packed: they are consumed as words and never expanded to an fp16 matrix.
// [PACK] lpnh.cn/news/2438023, section "文本模型加载artifact.load_model 与 Packed 模块".
//
// Design (one GB300 SM = one persistent CTA of 8 warps):
//  * Output rows are cut into tiles of 16 (one mma.m16n8k16 A operand); CTA b takes
//    tiles b, b + grid, ...  The 8 warps split the K groups of every tile.
//  * Every warp streams its own share of each tile into a private ring of shared
//    memory stages with 1-D bulk copies (one copy per weight row, evict-first in L2),
//    so ~100 KB of packed words per SM are in flight while it computes.
//  * The tile's scales and biases arrive by two bulk copies into a double-buffered
//    slot (rows of a 16-row tile are contiguous in [N, K/128]).
//  * Decoding is two instructions per pair of weights and never rounds: LOP3 puts a
//    2-bit field into the mantissa of an fp16 1024.0, giving 1024 + sigma*q exactly
//    (sigma = 4^j for the field's bit position j); no shift or subtraction is needed.
//    Those half2 values are the A fragments of mma.sync.m16n8k16 (fp32 accumulate);
//    the B fragment is the rotated activation x' divided by sigma (exact in fp16).
//    Per group of 128:  D = sum (1024 + sigma q) x'/sigma = sum q x' + C,
//    C = 1024 * sum x'/sigma is a per-token constant, so
//    y += s * (D - C) + b * S,  S = sum x' over the group.
//  * x' = fwht(x) is computed once per CTA at the start (while the first weight stages
//    are already in flight) and stored in shared memory directly in B-fragment order.
//  * The k order inside an mma is a permutation of the group's k (codes p and p+8 of a
//    word share a half2); the B fragment image uses the same permutation.
// Tokens (M <= 8 per pass) are the mma's N = 8 columns.
#include <cuda_runtime.h>

#include "tb_common.cuh"
#include "tb_host.h"

namespace tb {

constexpr int kGemvWarps = 8;
constexpr int kGemvThreads = kGemvWarps * 32;
constexpr int kTileRows = 16;
constexpr int kStageGroups = 4;                                 // K groups per ring stage
constexpr int kStagePitch = kStageGroups * 32 + 32;             // bytes per row (== 32 mod 128)
constexpr int kStageBytes = kTileRows * kStagePitch;            // 2560
constexpr int kMaxScaleSlots = 8;                              // tiles of scales in flight
constexpr int kScaleSlotBytesPerGroup = 2 * kTileRows * 2;      // scale + bias of 16 rows
constexpr uint32_t kMagic = 0x64006400u;                        // half2(1024, 1024)

struct GemvArgs {
  const __half* x;       // [Mc, K] tokens of this pass
  const int8_t* signs;   // [K] or null
  const uint32_t* w;     // [N, K/16]
  const __half* scales;  // [N, G]
  const __half* biases;  // [N, G]
  __half* y;             // [Mc, N]
  int Mc;                // tokens in this pass (<= MT)
  int K, N, G;
  int rotate;            // 1: x' = fwht(x); 0: x' = x
  int ring;              // stages per warp ring
  int sslots;            // tiles of scales/biases in flight
  int32_t* status;
};

struct GemvLayout {
  int bars, img, cs, scl, scratch, ringb, total;
};

__host__ __device__ inline int round_up(int v, int a) { return (v + a - 1) / a * a; }

template <int MT>
__host__ __device__ inline GemvLayout gemv_layout(int G, int ring, int sslots) {
  GemvLayout L;
  int off = 0;
  L.bars = off;
  off += (kGemvWarps * ring + sslots) * 8;
  off = round_up(off, 128);
  L.img = off;
  off += G * 256 * MT;
  L.cs = off;
  off += G * MT * 8;
  off = round_up(off, 128);
  L.scl = off;
  off += sslots * 2 * kTileRows * G * 2;
  off = round_up(off, 128);
  L.scratch = off;
  const int fw = kGemvWarps * kWarpScratchFloats * 4;
  const int red = 2 * kGemvWarps * kTileRows * MT * 4;
  off += fw > red ? fw : red;
  off = round_up(off, 128);
  L.ringb = off;
  off += kGemvWarps * ring * kStageBytes;
  L.total = off;
  return L;
}

TB_DEVI void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                      uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16 codes of a word -> 8 half2 A-fragment values (1024 + sigma_p q_p, 1024 + sigma_p q_{p+8})
// sigma = 1, 4, 16, 64, 256, 16, 64, 256 for p = 0..7
TB_DEVI void decode_word(uint32_t w, uint32_t (&P)[8]) {
  const uint32_t w6 = w >> 6;
  P[0] = lop3_and_or(w, 0x00030003u, kMagic);
  P[1] = lop3_and_or(w, 0x000C000Cu, kMagic);
  P[2] = lop3_and_or(w, 0x00300030u, kMagic);
  P[3] = lop3_and_or(w, 0x00C000C0u, kMagic);
  P[4] = lop3_and_or(w, 0x03000300u, kMagic);
  P[5] = lop3_and_or(w6, 0x00300030u, kMagic);
  P[6] = lop3_and_or(w6, 0x00C000C0u, kMagic);
  P[7] = lop3_and_or(w6, 0x03000300u, kMagic);
}

TB_DEVI float inv_sigma(int p) {
  // 1/sigma_p for p = 0..7
  return p == 0 ? 1.0f : p == 1 ? 0.25f : (p == 2 || p == 5) ? 0.0625f
       : (p == 3 || p == 6) ? 0.015625f : 0.00390625f;
}

// One or two K groups of a 16-row tile: decode, 8 mma each (two independent chains when
// NG = 2), then the per-group scale epilogue into acc.
template <int MT, int NG>
TB_DEVI void gemv_groups(const uint8_t* rowg, int gi0, int grp0, const uint4* imgt, const __half* ss,
                         const __half* sb, int G, int g, const float2* cs, int t0, int t1,
                         float (&acc)[4]) {
  uint2 wa[NG], wb[NG];
#pragma unroll
  for (int n = 0; n < NG; ++n) {
    wa[n] = *reinterpret_cast<const uint2*>(rowg + (gi0 + n) * 32);
    wb[n] = *reinterpret_cast<const uint2*>(rowg + 8 * kStagePitch + (gi0 + n) * 32);
  }
  float d[NG][4];
#pragma unroll
  for (int n = 0; n < NG; ++n) d[n][0] = d[n][1] = d[n][2] = d[n][3] = 0.f;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t P[NG][8], Q[NG][8];
    uint4 i0[NG], i1[NG];
#pragma unroll
    for (int n = 0; n < NG; ++n) {
      decode_word(half ? wa[n].y : wa[n].x, P[n]);
      decode_word(half ? wb[n].y : wb[n].x, Q[n]);
      i0[n] = imgt[((grp0 + n) * 4 + 2 * half) * MT * 4];
      i1[n] = imgt[((grp0 + n) * 4 + 2 * half + 1) * MT * 4];
    }
#pragma unroll
    for (int n = 0; n < NG; ++n) mma16816(d[n], P[n][0], Q[n][0], P[n][1], Q[n][1], i0[n].x, i0[n].y);
#pragma unroll
    for (int n = 0; n < NG; ++n) mma16816(d[n], P[n][2], Q[n][2], P[n][3], Q[n][3], i0[n].z, i0[n].w);
#pragma unroll
    for (int n = 0; n < NG; ++n) mma16816(d[n], P[n][4], Q[n][4], P[n][5], Q[n][5], i1[n].x, i1[n].y);
#pragma unroll
    for (int n = 0; n < NG; ++n) mma16816(d[n], P[n][6], Q[n][6], P[n][7], Q[n][7], i1[n].z, i1[n].w);
  }
#pragma unroll
  for (int n = 0; n < NG; ++n) {
    const int grp = grp0 + n;
    // sb == nullptr: no biases given, each is the pack's -scale
    const float sA = __half2float(ss[g * G + grp]), bA = sb ? __half2float(sb[g * G + grp]) : -sA;
    const float sB = __half2float(ss[(g + 8) * G + grp]),
                bB = sb ? __half2float(sb[(g + 8) * G + grp]) : -sB;
    const float2 c0 = cs[grp * MT + t0], c1 = cs[grp * MT + t1];
    acc[0] += sA * (d[n][0] - c0.x) + bA * c0.y;
    acc[1] += sA * (d[n][1] - c1.x) + bA * c1.y;
    acc[2] += sB * (d[n][2] - c0.x) + bB * c0.y;
    acc[3] += sB * (d[n][3] - c1.x) + bB * c1.y;
  }
}

template <int MT>
__global__ void __launch_bounds__(kGemvThreads, 1) w2_gemv_kernel(const GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int K = a.K, N = a.N, G = a.G, D = a.ring, R = a.sslots;
  const GemvLayout L = gemv_layout<MT>(G, D, R);

  // the next kernel on the stream may start now; it waits for this grid before reading
  // anything this grid writes (programmatic dependent launch)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);  // [warp][D]
  uint64_t* sfull = full + kGemvWarps * D;                       // [R]
  __half* img = reinterpret_cast<__half*>(smem + L.img);
  float2* cs = reinterpret_cast<float2*>(smem + L.cs);           // [G][MT] = (C, S)
  __half* scl = reinterpret_cast<__half*>(smem + L.scl);         // [slot][s|b][16][G]
  float* scratch = reinterpret_cast<float*>(smem + L.scratch);
  uint8_t* ring = smem + L.ringb + warp * D * kStageBytes;
  __shared__ volatile int aborted;

  const int n_tiles = (N + kTileRows - 1) / kTileRows;
  const int nt = blockIdx.x < n_tiles ? (n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int g0 = (G * warp) / kGemvWarps, g1 = (G * (warp + 1)) / kGemvWarps;
  const int spt = (g1 - g0 + kStageGroups - 1) / kStageGroups;  // stages per tile for this warp
  const int total = nt * spt;
  const uint64_t pol = policy_evict_first();

  if (threadIdx.x == 0) {
    aborted = 0;
    for (int i = 0; i < kGemvWarps * D; ++i) mbar_init(full + i, 1);
    for (int i = 0; i < R; ++i) mbar_init(sfull + i, 1);
    fence_barrier_init();
  }
  __syncthreads();

  // ---- producers ------------------------------------------------------------
  auto issue_stage = [&](int i) {
    const int j = i / spt, c = i - j * spt;
    const int r0 = (blockIdx.x + j * gridDim.x) * kTileRows;
    const int ga = g0 + c * kStageGroups;
    const int gn = min(kStageGroups, g1 - ga);
    const int rows = min(kTileRows, N - r0);
    const int slot = i % D;
    if (lane == 0) mbar_arrive_expect_tx(full + warp * D + slot, (uint32_t)(rows * gn * 32));
    __syncwarp();
    if (lane < rows)
      bulk_g2s_hint(ring + slot * kStageBytes + lane * kStagePitch,
                    a.w + (int64_t)(r0 + lane) * (K / kCodesPerWord) + ga * 8, (uint32_t)(gn * 32),
                    full + warp * D + slot, pol);
  };
  // scales and biases of local tile j into slot j % R (warp 0 only)
  auto issue_scales = [&](int j) {
    const int r0 = (blockIdx.x + j * gridDim.x) * kTileRows;
    const int rows = min(kTileRows, N - r0);
    const int slot = j % R;
    __half* ds = scl + slot * 2 * kTileRows * G;
    __half* db = ds + kTileRows * G;
    const uint32_t bytes = (uint32_t)(rows * G * 2);
    if ((bytes & 15u) == 0) {
      if (lane == 0) {
        mbar_arrive_expect_tx(sfull + slot, a.biases ? 2 * bytes : bytes);
        bulk_g2s_hint(ds, a.scales + (int64_t)r0 * G, bytes, sfull + slot, pol);
        if (a.biases) bulk_g2s_hint(db, a.biases + (int64_t)r0 * G, bytes, sfull + slot, pol);
      }
    } else {  // ragged last tile: plain copies
      for (int e = lane; e < rows * G; e += 32) {
        ds[e] = a.scales[(int64_t)r0 * G + e];
        if (a.biases) db[e] = a.biases[(int64_t)r0 * G + e];
      }
      __threadfence_block();
      __syncwarp();
      if (lane == 0) mbar_arrive(sfull + slot);
    }
    __syncwarp();
  };

  // weights, scales and biases are never written by a kernel that lets this one start
  // early, so their prefetch may run ahead of the dependency wait
  for (int i = 0; i < min(D, total); ++i) issue_stage(i);
  if (warp == 0)
    for (int j = 0; j < min(R, nt); ++j) issue_scales(j);
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- prologue: x' = fwht(signs * x) -> B-fragment image, C and S per group ----
  {
    const int nchunk = (K + kBlock - 1) / kBlock;
    float* sw = scratch + warp * kWarpScratchFloats;
    for (int it = warp; it < MT * nchunk; it += kGemvWarps) {
      const int tok = it / nchunk, b = it - tok * nchunk;
      float v[32];
      const bool live = tok < a.Mc;
      if (a.rotate) {
        if (live) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            float f = __half2float(a.x[(int64_t)tok * K + b * kBlock + j * 32 + lane]);
            if (a.signs && a.signs[b * kBlock + j * 32 + lane] < 0) f = -f;
            v[j] = f;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0.f;
        }
        wht1024_b_to_a(v, sw, lane);
#pragma unroll
        for (int r = 0; r < 32; ++r) v[r] *= kInvSqrtBlock;
      } else {
        const bool in = live && (b * kBlock + lane * 32 < K);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 u = make_uint4(0, 0, 0, 0);
          if (in) u = *reinterpret_cast<const uint4*>(a.x + (int64_t)tok * K + b * kBlock + lane * 32 + 8 * q);
          const __half* h = reinterpret_cast<const __half*>(&u);
#pragma unroll
          for (int e = 0; e < 8; ++e) v[8 * q + e] = __half2float(h[e]);
        }
      }
      // v[r] = x' of element b*1024 + lane*32 + r: lane covers words 2t, 2t+1 of group grp
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
          const int p = 4 * (mp & 1) + e2;           // position pair of the word
          const int r = (mp >> 1) * 16 + p;          // lo element; hi element is r + 8
          const float is = inv_sigma(p);
          const __half lo = __float2half_rn(v[r] * is), hi = __float2half_rn(v[r + 8] * is);
          csum += __half2float(lo) + __half2float(hi);
          pk[e2] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
        }
        if (grp < G)
          *reinterpret_cast<uint4*>(img + ((size_t)(grp * 4 + mp) * MT + tok) * 32 + t * 8) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      ssum += __shfl_xor_sync(0xffffffffu, ssum, 1);
      ssum += __shfl_xor_sync(0xffffffffu, ssum, 2);
      csum += __shfl_xor_sync(0xffffffffu, csum, 1);
      csum += __shfl_xor_sync(0xffffffffu, csum, 2);
      if (t == 0 && grp < G) cs[grp * MT + tok] = make_float2(1024.f * csum, ssum);
    }
  }
  __syncthreads();

  // ---- main loop ------------------------------------------------------------
  // Lanes whose mma column g is not a live token read token 0's image: their D columns
  // are never used.
  const int tokc = g < MT ? g : 0;
  const uint4* imgt = reinterpret_cast<const uint4*>(img) + tokc * 4 + t;
  const int t0 = min(2 * t, MT - 1), t1 = min(2 * t + 1, MT - 1);
  float* red = scratch;  // [2][warp][16][MT]
  int i = 0;

  for (int j = 0; j < nt; ++j) {
    const int r0 = (blockIdx.x + j * gridDim.x) * kTileRows;
    const int sslot = j % R;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (spt > 0) {
      if (!aborted && !mbar_wait(sfull + sslot, (j / R) & 1)) {
        aborted = 1;
        set_status(a.status, TB_DEV_TIMEOUT);
      }
      const __half* ss = scl + sslot * 2 * kTileRows * G;
      const __half* sb = a.biases ? ss + kTileRows * G : nullptr;
      for (int c = 0; c < spt; ++c, ++i) {
        const int slot = i % D;
        if (!aborted && !mbar_wait(full + warp * D + slot, (i / D) & 1)) {
          aborted = 1;
          set_status(a.status, TB_DEV_TIMEOUT);
        }
        const int ga = g0 + c * kStageGroups;
        const int gn = min(kStageGroups, g1 - ga);
        const uint8_t* rowg = ring + slot * kStageBytes + g * kStagePitch + t * 8;
        int gi = 0;
        for (; gi + 2 <= gn; gi += 2)
          gemv_groups<MT, 2>(rowg, gi, ga + gi, imgt, ss, sb, G, g, cs, t0, t1, acc);
        if (gi < gn) gemv_groups<MT, 1>(rowg, gi, ga + gi, imgt, ss, sb, G, g, cs, t0, t1, acc);
        __syncwarp();
        if (i + D < total) {
          fence_proxy_async_smem();  // generic reads of this slot before the async refill
          issue_stage(i + D);
        }
      }
    }
    // cross-warp reduction of the tile
    float* rw = red + ((j & 1) * kGemvWarps + warp) * kTileRows * MT;
    if (2 * t < MT) {
      rw[g * MT + 2 * t] = acc[0];
      rw[(g + 8) * MT + 2 * t] = acc[2];
    }
    if (2 * t + 1 < MT) {
      rw[g * MT + 2 * t + 1] = acc[1];
      rw[(g + 8) * MT + 2 * t + 1] = acc[3];
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kGemvThreads) : "memory");
    if (warp == 0 && j + R < nt) issue_scales(j + R);
    if (threadIdx.x < kTileRows * MT) {
      const int row = threadIdx.x / MT, tok = threadIdx.x - row * MT;
      float sum = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < kGemvWarps; ++w2)
        sum += red[((j & 1) * kGemvWarps + w2) * kTileRows * MT + threadIdx.x];
      if (r0 + row < N && tok < a.Mc) a.y[(int64_t)tok * N + r0 + row] = __float2half_rn(sum);
    }
  }
}

// host side --------------------------------------------------------------------
// tiles of scales and biases kept in flight: enough to cover the DRAM latency of small
// tiles, at most 32 KB
static int gemv_scale_slots(int G) {
  int r = 32768 / (kScaleSlotBytesPerGroup * G);
  return r < 2 ? 2 : (r > kMaxScaleSlots ? kMaxScaleSlots : r);
}

template <int MT>
static int gemv_ring_for(int G, int smem_optin) {
  const int fixed = gemv_layout<MT>(G, 0, gemv_scale_slots(G)).total + kGemvWarps * 8 * 16;  // bars headroom
  const int per = kGemvWarps * kStageBytes;
  const int d = (smem_optin - fixed) / per;
  return d > 16 ? 16 : d;
}

template <int MT>
static int launch_gemv_mt(const GemvArgs& base, int64_t M, int64_t K, const DeviceFacts& f,
                          cudaStream_t s) {
  GemvArgs a = base;
  const int ring = gemv_ring_for<MT>(a.G, f.smem_optin);
  if (ring < 2) return TB_ERR_SHAPE;
  a.ring = ring;
  a.sslots = gemv_scale_slots(a.G);
  const int bytes = gemv_layout<MT>(a.G, ring, a.sslots).total;
  cudaError_t e = cudaFuncSetAttribute(w2_gemv_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       bytes);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return TB_ERR_CUDA;
  }
  const int n_tiles = (a.N + kTileRows - 1) / kTileRows;
  const int grid = n_tiles < f.sms ? n_tiles : f.sms;
  for (int64_t m0 = 0; m0 < M; m0 += MT) {
    a.x = base.x + m0 * K;
    a.y = base.y + m0 * a.N;
    a.Mc = (int)((M - m0) < MT ? (M - m0) : MT);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGemvThreads);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, w2_gemv_kernel<MT>, a);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      return TB_ERR_CUDA;
    }
  }
  return TB_OK;
}

// the largest token count per pass (1, 2, 4 or 8) whose B image leaves a ring of >= 3 stages
static int gemv_tokens_per_pass(int64_t M, int G, int smem_optin) {
  int mt = M >= 8 ? 8 : M >= 4 ? (M == 4 ? 4 : 8) : (M >= 2 ? (M == 2 ? 2 : 4) : 1);
  while (mt > 1) {
    int d = mt == 8 ? gemv_ring_for<8>(G, smem_optin)
          : mt == 4 ? gemv_ring_for<4>(G, smem_optin)
                    : gemv_ring_for<2>(G, smem_optin);
    if (d >= 3) break;
    mt >>= 1;
  }
  return mt;
}

int launch_gemv(const __half* x, int64_t M, int64_t K, const int8_t* signs, int block,
                const uint32_t* w, const __half* scales, const __half* biases, int64_t N,
                __half* y, int32_t* status, cudaStream_t s) {
  DeviceFacts f;
  int rc = device_facts(&f);
  if (rc != TB_OK) return rc;
  if (N > (int64_t)0x7fffffff - kTileRows || K > (1 << 24)) return TB_ERR_SHAPE;
  GemvArgs a;
  a.x = x;
  a.signs = signs;
  a.w = w;
  a.scales = scales;
  a.biases = biases;
  a.y = y;
  a.Mc = 0;
  a.K = (int)K;
  a.N = (int)N;
  a.G = (int)(K / kGroup);
  a.rotate = block != 0;
  a.ring = 0;
  a.sslots = 0;
  a.status = status;
  const int mt = gemv_tokens_per_pass(M, a.G, f.smem_optin);
  switch (mt) {
    case 8: return launch_gemv_mt<8>(a, M, K, f, s);
    case 4: return launch_gemv_mt<4>(a, M, K, f, s);
    case 2: return launch_gemv_mt<2>(a, M, K, f, s);
    default: return launch_gemv_mt<1>(a, M, K, f, s);
  }
}

}  // namespace tb
