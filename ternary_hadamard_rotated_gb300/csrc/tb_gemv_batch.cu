// Batched decode of the Packed layer (1 to 64 tokens per pass) on mma.sync: the decode GEMV's
// arithmetic with the tokens spread over several mma N tiles of 8, fed by a rotation pre-pass.
//
// [ARCH] kwkr.cn/news/564617, section "Hadamard 旋转把量化误差抹平的免费午餐": the layer is the
// rotated input (signs, then the normalised block Hadamard transform) times the packed 2-bit,
// group-128 affine weights, which are consumed directly and never expanded in memory.
//
// Two kernels:
//  * batch_image_kernel rotates x once (two warps per 1024-block and token, as in the decode
//    GEMV's prologue) and writes, per pass of MT tokens and per 512-k chunk, one contiguous
//    blob: the mma B-fragment image of x'/sigma (4 groups x 4 entries x MT tokens x 64 bytes)
//    followed by (C, S) = (1024 * sum(x'/sigma), sum(x')) per group and token, fp32.  Tokens
//    past M are zero.
//  * w2_gemv_batch_kernel<NT> (MT = 8 NT tokens): one CTA per SM walks a stream-K range of
//    units (128 rows x 512 k, tile-major).  A producer warp streams each unit's 16 KB box of
//    packed codes (TMA, 128-byte swizzle), the 128 rows' scales and biases of two chunks (TMA
//    boxes of 8 groups: the smallest the copy engine takes) and the chunk's blob (one bulk
//    copy) into one ring slot, so the consumers issue no global loads (a fence on their path
//    would wait for any still in flight); eight consumer warps of 16 rows each decode their
//    codes once per group (LOP3 into fp16 1024 + sigma*q) and run them against the NT token
//    tiles of the blob:
//      y[row, tok] += s * (D - C) + b * S   per group of 128,
//    D the group's mma sum starting from zero.  A tile that lies wholly in the CTA's range is
//    written from registers; a tile cut by a range boundary goes through the workspace (each
//    CTA's fp32 part in its own slot, a counter, the last contributor adding the parts in CTA
//    order, so repeated calls give the same bits).
//
// Workspace (batch region): counters [256] int (zero at rest, returned to zero by every call),
// parts [256][2][128][MT] fp32, blobs [passes][K/512][blob bytes].
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "tb_common.cuh"
#include "tb_gemv_core.cuh"
#include "tb_host.h"

namespace tb {

int code_map(const uint32_t* w, int64_t N, int64_t K, CUtensorMap* out);
int group_map(const __half* p, int64_t N, int64_t G, CUtensorMap* out);

constexpr int kBtConsumers = 8;                         // warps of 16 rows: one 128-row unit
constexpr int kBtThreads = (kBtConsumers + 1) * 32;     // and the producer warp
constexpr int kBtMaxCtas = 256;                         // part slots and counters per call
constexpr int kBtImgWarps = 8;                          // warps per block of the image kernel
constexpr size_t kBtCounterBytes = 1024;

// slot: codes [128 rows][128 B] (swizzled), scales and biases [128 rows][8 groups] fp16, blob
constexpr int kBtSbBox = kUnitRows * 8 * 2;        // one box of scales (or biases): 2 KB
constexpr int kBtScaleOff = kSlotBytes;
constexpr int kBtBiasOff = kSlotBytes + kBtSbBox;
constexpr int kBtBlobOff = kSlotBytes + 2 * kBtSbBox;
__host__ __device__ constexpr int bt_blob_bytes(int MT) { return 1024 * MT + 32 * MT; }
__host__ __device__ constexpr int bt_slot_bytes(int MT) {
  return (kBtBlobOff + bt_blob_bytes(MT) + 1023) / 1024 * 1024;  // codes stay 1024-aligned
}
// ring slots per token count: four up to 16 tokens (five or six measured the same), fewer as
// the blobs widen
__host__ __device__ constexpr int bt_slots(int MT) { return MT <= 16 ? 4 : MT <= 32 ? 3 : 2; }
__host__ __device__ constexpr int bt_smem_bytes(int MT) {
  return bt_slots(MT) * bt_slot_bytes(MT) + 2 * 4 * 8 + 1024;
}

struct BatchArgs {
  int has_bias;          // biases given (else each is -s)
  __half* y;             // [Mc, N] (this pass's tokens)
  const uint8_t* blob;   // [C][bt_blob_bytes(MT)] of this pass
  float* part;           // [kBtMaxCtas][2][128][MT]
  int* count;            // [kBtMaxCtas]
  int Mc, N, G, C, n_tiles;
  int32_t* status;
};

// ------------------------------------------------------------------ rotation into blobs
// Item = (token, 1024-block, half): H1024 = [[H512, H512], [H512, -H512]], so outputs 0..511 of
// a block are H512(x_lo + x_hi) and 512..1023 are H512(x_lo - x_hi); lane l holds elements
// 16 l .. 16 l + 15 of both input halves and of its output half.
template <int MT>
__global__ void __launch_bounds__(kBtImgWarps * 32) batch_image_kernel(
    const __half* __restrict__ x, const int8_t* __restrict__ signs, int M, int K, int rotate,
    int n_tok, uint8_t* __restrict__ blob) {
  // the GEMV (a programmatic dependent) may start streaming weights; it reads the blobs only
  // after griddepcontrol.wait, i.e. after this grid has completed
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int nblk = K / kBlock, C = K / (kUnitGroups * kGroup);
  const int it = blockIdx.x * kBtImgWarps + (threadIdx.x >> 5);
  if (it >= n_tok * nblk * 2) return;
  const int hh = it & 1, rest = it >> 1;
  const int tok = rest / nblk, b = rest - (rest / nblk) * nblk;
  float v[16];
  {
    uint4 xr[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                   make_uint4(0, 0, 0, 0)};
    if (tok < M) {
      const uint4* xs = reinterpret_cast<const uint4*>(x + (int64_t)tok * K + b * kBlock + lane * 16);
      xr[0] = __ldg(xs);
      xr[1] = __ldg(xs + 1);
      xr[2] = __ldg(xs + kBlock / 16);  // the same elements of the upper half
      xr[3] = __ldg(xs + kBlock / 16 + 1);
    }
    uint4 sr[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    if (signs) {
      const uint4* sp = reinterpret_cast<const uint4*>(signs + b * kBlock + lane * 16);
      sr[0] = __ldg(sp);
      sr[1] = __ldg(sp + kBlock / 32);
    }
    const __half* xl = reinterpret_cast<const __half*>(&xr[0]);
    const __half* xh = reinterpret_cast<const __half*>(&xr[2]);
    const int8_t* sl = reinterpret_cast<const int8_t*>(&sr[0]);
    const int8_t* sh = reinterpret_cast<const int8_t*>(&sr[1]);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      float lo_ = __half2float(xl[e]), hi_ = __half2float(xh[e]);
      if (signs) {
        if (sl[e] < 0) lo_ = -lo_;
        if (sh[e] < 0) hi_ = -hi_;
      }
      v[e] = rotate ? (hh ? lo_ - hi_ : lo_ + hi_) : (hh ? hi_ : lo_);
    }
  }
  if (rotate) {
    wht512_a_shfl(v, lane);
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] *= kInvSqrtBlock;
  }
  // group of 128 of this lane's outputs: chunk 2b + hh, group lane >> 3 in it, eight lanes of 16
  const int chunk = 2 * b + hh, gi = lane >> 3, q = lane & 7;
  const int pass = tok / MT, tl = tok - (tok / MT) * MT;
  uint8_t* base = blob + ((size_t)pass * C + chunk) * bt_blob_bytes(MT);
  float ssum = 0.f, csum = 0.f;
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    v[e] = __half2float(__float2half_rn(v[e]));  // x' rounded to fp16
    ssum += v[e];
  }
  // image entry (gi, mp) of token tl, fragment lane t: group elements 32 t + 16 (mp >> 1) +
  // 4 (mp & 1) + {0..3} and the same + 8, each divided by sigma of its position; this lane's
  // 16 elements are those of t = q >> 1 and mp = 2 (q & 1) + {0, 1}
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
    *reinterpret_cast<uint4*>(base + ((gi * 4 + mp) * MT + tl) * 64 + (q >> 1) * 16) =
        make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
    csum += __shfl_xor_sync(0xffffffffu, csum, o);
  }
  if (q == 0)
    *reinterpret_cast<float2*>(base + 1024 * MT + (gi * MT + tl) * 8) = make_float2(1024.f * csum, ssum);
}

// ------------------------------------------------------------------ the GEMV
// One group of 128 k of this warp's 16 rows: decode each row's two words per half once, run
// them against the NT token tiles, then y += s (D - C) + b S per token.
//   box: the unit's code box; R: this lane's A row (and R + 8) in the unit; img, csb: the blob
//   sb: the slot's scale box at this unit's group 0 (biases kBtSbBox further)
TB_DEVI float lds_half(uint32_t a) {
  unsigned short h;
  asm("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(a));
  return __half2float(__ushort_as_half(h));
}

template <int NT>
TB_DEVI void batch_group(uint32_t box, uint32_t img, uint32_t csb, int R, int rA, int g, int t, int gi,
                         uint32_t sb, bool has_bias, float (&acc)[NT][4]) {
  constexpr int MT = 8 * NT;
  const int c = 2 * gi + (t >> 1);  // logical 16-byte chunk of the 128-byte row
  const uint32_t wo = ((c ^ (rA & 7)) << 4) + (t & 1) * 8;
  const uint2 w0 = ld_shared_v2(box + R * 128 + wo);
  const uint2 w1 = ld_shared_v2(box + (R + 8) * 128 + wo);
  float d[NT][4];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t P[8], Q[8];
    decode_word_sigma(half ? w0.y : w0.x, P);
    decode_word_sigma(half ? w1.y : w1.x, Q);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const uint32_t e = img + ((gi * 4 + 2 * half) * MT + 8 * nt + g) * 64 + t * 16;
      const uint4 i0 = ld_shared_v4(e);
      const uint4 i1 = ld_shared_v4(e + MT * 64);
      if (half == 0)
        mma16816_zero(d[nt], P[0], Q[0], P[1], Q[1], i0.x, i0.y);
      else
        mma16816_acc(d[nt], P[0], Q[0], P[1], Q[1], i0.x, i0.y);
      mma16816_acc(d[nt], P[2], Q[2], P[3], Q[3], i0.z, i0.w);
      mma16816_acc(d[nt], P[4], Q[4], P[5], Q[5], i1.x, i1.y);
      mma16816_acc(d[nt], P[6], Q[6], P[7], Q[7], i1.z, i1.w);
    }
  }
  float2 A, B;  // (s, b) of rows R and R + 8
  A.x = lds_half(sb + R * 16 + gi * 2);
  B.x = lds_half(sb + (R + 8) * 16 + gi * 2);
  A.y = has_bias ? lds_half(sb + kBtSbBox + R * 16 + gi * 2) : -A.x;
  B.y = has_bias ? lds_half(sb + kBtSbBox + (R + 8) * 16 + gi * 2) : -B.x;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    // D columns 2t, 2t + 1 of tile nt: tokens 8 nt + 2t and the next; their (C, S) side by side
    const uint4 cu = ld_shared_v4(csb + (gi * MT + 8 * nt + 2 * t) * 8);
    const float C0 = __uint_as_float(cu.x), S0 = __uint_as_float(cu.y);
    const float C1 = __uint_as_float(cu.z), S1 = __uint_as_float(cu.w);
    acc[nt][0] = fmaf(A.x, d[nt][0] - C0, fmaf(A.y, S0, acc[nt][0]));
    acc[nt][1] = fmaf(A.x, d[nt][1] - C1, fmaf(A.y, S1, acc[nt][1]));
    acc[nt][2] = fmaf(B.x, d[nt][2] - C0, fmaf(B.y, S0, acc[nt][2]));
    acc[nt][3] = fmaf(B.x, d[nt][3] - C1, fmaf(B.y, S1, acc[nt][3]));
  }
}

// Warp roles: warps 0..7 consume (rows 16 w .. 16 w + 15 of every unit), warp 8 produces.
template <int NT>
__global__ void __launch_bounds__(kBtThreads, 1)
    w2_gemv_batch_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS,
                         const __grid_constant__ CUtensorMap tmB, const BatchArgs a) {
  constexpr int MT = 8 * NT;
  constexpr int SB = bt_slot_bytes(MT), DW = bt_slots(MT), BLOB = bt_blob_bytes(MT);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t ring = smem_u32(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + DW * SB);
  uint64_t* empty = full + DW;
  __shared__ volatile int aborted;
  __shared__ int fin;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = a.C;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int S = a.n_tiles * C;
  const int lo = (int)((int64_t)S * blockIdx.x / gridDim.x);
  const int hi = (int)((int64_t)S * (blockIdx.x + 1) / gridDim.x);
  const int cnt = hi - lo;
  if (threadIdx.x == 0) {
    aborted = 0;
    for (int i = 0; i < DW; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, kBtConsumers);
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

  if (warp == kBtConsumers) {
    // ---- producer: slot n % DW <- the codes, scales and biases of unit lo + n and the blob
    // of its chunk ----
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const uint32_t bytes = kBtBlobOff - (a.has_bias ? 0 : kBtSbBox) + BLOB;
      auto weights = [&](int slot, int tile, int ch) {
        const uint32_t d = ring + slot * SB;
        tma2d(d, &tmW, ch * 32, tile * kUnitRows, full + slot, pol);
        // the box of eight groups that holds this chunk's four (x a multiple of 8 elements)
        tma2d(d + kBtScaleOff, &tmS, 8 * (ch >> 1), tile * kUnitRows, full + slot, pol);
        if (a.has_bias) tma2d(d + kBtBiasOff, &tmB, 8 * (ch >> 1), tile * kUnitRows, full + slot, pol);
      };
      const int pro = cnt < DW ? cnt : DW;
      int tile = lo / C, ch = lo - (lo / C) * C;
      for (int n = 0; n < pro; ++n) {  // the weights do not depend on the previous kernel
        mbar_arrive_expect_tx(full + n, bytes);
        weights(n, tile, ch);
        step_unit(tile, ch, C, false);
      }
      asm volatile("griddepcontrol.wait;" ::: "memory");  // the blobs are the rotation's output
      tile = lo / C;
      ch = lo - (lo / C) * C;
      for (int n = 0; n < pro; ++n) {
        bulk_g2s(smem + n * SB + kBtBlobOff, a.blob + (size_t)ch * BLOB, BLOB, full + n);
        step_unit(tile, ch, C, false);
      }
      for (int n = pro; n < cnt; ++n) {
        const int slot = n % DW;
        wait(empty + slot, (n / DW - 1) & 1);
        mbar_arrive_expect_tx(full + slot, bytes);
        weights(slot, tile, ch);
        bulk_g2s(smem + slot * SB + kBtBlobOff, a.blob + (size_t)ch * BLOB, BLOB, full + slot);
        step_unit(tile, ch, C, false);
      }
      // leave no copy in flight: wait (bounded, even after a timeout) for the last fill of
      // every slot
      for (int n = cnt - 1; n >= 0 && n >= cnt - DW; --n)
        if (!mbar_wait(full + n % DW, (n / DW) & 1)) set_status(a.status, TB_DEV_TIMEOUT);
    }
    return;
  }

  // ---- consumers ----
  const int g = lane >> 2, t = lane & 3;
  const int rA = 2 * (g & 3) + (g >> 2);  // mma row g <-> unit row 16 warp + rA (and + 8)
  const int R = 16 * warp + rA;
  // y, the parts and the counters are written only after the previous kernel has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // Add the CTA's sums of tile T to y: directly when the whole tile is this CTA's, else through
  // the part slots, the last contributor adding them in CTA order.
  auto flush = [&](int T, float (&acc)[NT][4]) {
    const int row0 = T * kUnitRows;
    const int tb = T * C, te = tb + C;
    if (tb >= lo && te <= hi) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int m = 8 * nt + 2 * t;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int row = row0 + R + 8 * h;
          if (row < a.N) {
            if (m < a.Mc) a.y[(int64_t)m * a.N + row] = __float2half_rn(acc[nt][2 * h]);
            if (m + 1 < a.Mc) a.y[(int64_t)(m + 1) * a.N + row] = __float2half_rn(acc[nt][2 * h + 1]);
          }
        }
      }
      return;
    }
    float* mine = a.part + ((size_t)blockIdx.x * 2 + (lo / C == T ? 0 : 1)) * kUnitRows * MT;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int m = 8 * nt + 2 * t;
      __stcg(reinterpret_cast<float2*>(mine + R * MT + m), make_float2(acc[nt][0], acc[nt][1]));
      __stcg(reinterpret_cast<float2*>(mine + (R + 8) * MT + m), make_float2(acc[nt][2], acc[nt][3]));
    }
    fence_acq_rel_gpu();  // this thread's part before the count
    asm volatile("bar.sync 1, %0;" ::"n"(kBtConsumers * 32) : "memory");
    const int first = stage_owner(tb, S, gridDim.x), lastc = stage_owner(te - 1, S, gridDim.x);
    if (threadIdx.x == 0) fin = atomicAdd(a.count + first, 1) == lastc - first;
    asm volatile("bar.sync 1, %0;" ::"n"(kBtConsumers * 32) : "memory");
    if (!fin) return;
    fence_acq_rel_gpu();  // every contributor's part after the count
    // thread i adds the float4 runs i, i + 256, ... (NT of them) of every contributor's part, two
    // contributors' loads in flight at once, in CTA order
    auto part_of = [&](int cc) {
      const int clo = (int)((int64_t)S * cc / gridDim.x);
      return reinterpret_cast<const float4*>(a.part + ((size_t)cc * 2 + (clo / C == T ? 0 : 1)) * kUnitRows * MT);
    };
    float4 v[NT];
#pragma unroll
    for (int k = 0; k < NT; ++k) v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int cc = first; cc <= lastc; cc += 2) {
      const float4* p0 = part_of(cc);
      const float4* p1 = cc + 1 <= lastc ? part_of(cc + 1) : nullptr;
      float4 l0[NT], l1[NT];
#pragma unroll
      for (int k = 0; k < NT; ++k) {
        l0[k] = __ldcg(p0 + threadIdx.x + kBtConsumers * 32 * k);
        l1[k] = p1 ? __ldcg(p1 + threadIdx.x + kBtConsumers * 32 * k) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < NT; ++k) {
        v[k].x += l0[k].x; v[k].y += l0[k].y; v[k].z += l0[k].z; v[k].w += l0[k].w;
        v[k].x += l1[k].x; v[k].y += l1[k].y; v[k].z += l1[k].z; v[k].w += l1[k].w;
      }
    }
#pragma unroll
    for (int k = 0; k < NT; ++k) {
      const int e = 4 * (threadIdx.x + kBtConsumers * 32 * k);  // (row r, tokens m .. m + 3)
      const int r = e / MT, m = e - (e / MT) * MT;
      if (row0 + r < a.N) {
        __half* yo = a.y + (int64_t)m * a.N + row0 + r;
        if (m < a.Mc) yo[0] = __float2half_rn(v[k].x);
        if (m + 1 < a.Mc) yo[a.N] = __float2half_rn(v[k].y);
        if (m + 2 < a.Mc) yo[2 * (int64_t)a.N] = __float2half_rn(v[k].z);
        if (m + 3 < a.Mc) yo[3 * (int64_t)a.N] = __float2half_rn(v[k].w);
      }
    }
    if (threadIdx.x == 0) a.count[first] = 0;
  };

  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
  int tile = lo / C, chunk = lo - (lo / C) * C;
  auto body = [&](int n) {
    const int slot = n % DW;
    wait(full + slot, (n / DW) & 1);
    const uint32_t box = ring + slot * SB, img = box + kBtBlobOff, csb = img + 1024 * MT;
    const uint32_t sb = box + kBtScaleOff + (chunk & 1) * 8;
    if (NT <= 2) {  // the groups' MMA chains overlap; wider tiles have enough chains already
#pragma unroll
      for (int gi = 0; gi < kUnitGroups; ++gi)
        batch_group<NT>(box, img, csb, R, rA, g, t, gi, sb, a.has_bias != 0, acc);
    } else {
#pragma unroll 1
      for (int gi = 0; gi < kUnitGroups; ++gi)
        batch_group<NT>(box, img, csb, R, rA, g, t, gi, sb, a.has_bias != 0, acc);
    }
    fence_proxy_async_smem();  // this thread's reads of the slot before the copies that refill it
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + slot);
    const int cur = tile;
    step_unit(tile, chunk, C, false);
    if (tile != cur || n == cnt - 1) {
      flush(cur, acc);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
    }
  };
  for (int n = 0; n < cnt; ++n) body(n);
}

// ------------------------------------------------------------------ host side
static int bt_tiles_nt(int64_t M) { return M <= 8 ? 1 : M <= 16 ? 2 : M <= 32 ? 4 : 8; }

// bytes of the batch region: counters, parts, blobs (1 KB aligned pieces)
static size_t bt_part_bytes(int MT) { return (size_t)kBtMaxCtas * 2 * kUnitRows * MT * 4; }
static size_t bt_blob_total(int64_t M, int64_t K) {
  const int MT = 8 * bt_tiles_nt(M);
  const int64_t passes = (M + MT - 1) / MT;
  return ((size_t)passes * (size_t)(K / (kUnitGroups * kGroup)) * bt_blob_bytes(MT) + 1023) / 1024 * 1024;
}
size_t gemv_batch_bytes(int64_t M, int64_t K) {
  if (M < 1 || K < kBlock) return 0;
  return kBtCounterBytes + bt_part_bytes(8 * bt_tiles_nt(M)) + bt_blob_total(M, K);
}

// x' of M tokens (K a multiple of 1024) into the blobs of the batch region
int launch_batch_image(const __half* x, int64_t M, int64_t K, const int8_t* signs, int rotate,
                       void* region, cudaStream_t s) {
  if (M < 1 || K < kBlock || K % kBlock || K > (1 << 22) || M > (1 << 20)) return TB_ERR_UNSUPPORTED;
  const int NT = bt_tiles_nt(M), MT = 8 * NT;
  const int64_t n_tok = (M + MT - 1) / MT * MT;
  const int64_t items = n_tok * (K / kBlock) * 2;
  if (items > (int64_t)INT32_MAX / 2) return TB_ERR_SHAPE;
  uint8_t* blob = static_cast<uint8_t*>(region) + kBtCounterBytes + bt_part_bytes(MT);
  const int blocks = (int)((items + kBtImgWarps - 1) / kBtImgWarps);
  switch (NT) {
    case 1:
      batch_image_kernel<8><<<blocks, kBtImgWarps * 32, 0, s>>>(x, signs, (int)M, (int)K, rotate, (int)n_tok, blob);
      break;
    case 2:
      batch_image_kernel<16><<<blocks, kBtImgWarps * 32, 0, s>>>(x, signs, (int)M, (int)K, rotate, (int)n_tok, blob);
      break;
    case 4:
      batch_image_kernel<32><<<blocks, kBtImgWarps * 32, 0, s>>>(x, signs, (int)M, (int)K, rotate, (int)n_tok, blob);
      break;
    default:
      batch_image_kernel<64><<<blocks, kBtImgWarps * 32, 0, s>>>(x, signs, (int)M, (int)K, rotate, (int)n_tok, blob);
  }
  return check_launch();
}

template <int NT>
static int launch_batch_nt(const CUtensorMap& map, const CUtensorMap& smap, const CUtensorMap& bmap, BatchArgs a, const uint8_t* blob0, int64_t M, int grid,
                           int smem_optin, int device, cudaStream_t s) {
  constexpr int MT = 8 * NT;
  constexpr int bytes = bt_smem_bytes(MT);
  if (bytes > smem_optin) return TB_ERR_UNSUPPORTED;
  const int rc = ensure_dynamic_smem(reinterpret_cast<const void*>(w2_gemv_batch_kernel<NT>), device, bytes);
  if (rc != TB_OK) return rc;
  cudaError_t e;
  __half* y0 = a.y;
  for (int64_t m0 = 0; m0 < M; m0 += MT) {
    a.y = y0 + m0 * a.N;
    a.Mc = (int)(M - m0 < MT ? M - m0 : MT);
    a.blob = blob0 + (size_t)(m0 / MT) * a.C * bt_blob_bytes(MT);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kBtThreads);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, w2_gemv_batch_kernel<NT>, map, smap, bmap, a);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      return TB_ERR_CUDA;
    }
  }
  return TB_OK;
}

// The batched GEMV over blobs already written by launch_batch_image into the same region.
int launch_batch_gemv(int64_t M, int64_t K, const uint32_t* w, const __half* scales, const __half* biases,
                      int64_t N, __half* y, void* region, int32_t* status, cudaStream_t s) {
  if (M < 1 || K < kBlock || K % kBlock || K > (1 << 22) || N < 1 || N > (1LL << 30))
    return TB_ERR_UNSUPPORTED;
  DeviceFacts f;
  int rc = device_facts(&f);
  if (rc != TB_OK) return rc;
  if (f.sms > kBtMaxCtas) return TB_ERR_UNSUPPORTED;
  const int64_t tiles = (N + kUnitRows - 1) / kUnitRows;
  const int C = (int)(K / (kUnitGroups * kGroup));
  if (tiles * C > (int64_t)INT32_MAX / 2) return TB_ERR_SHAPE;
  CUtensorMap map, smap, bmap;
  rc = code_map(w, N, K, &map);
  if (rc == TB_OK) rc = group_map(scales, N, K / kGroup, &smap);
  if (rc == TB_OK) rc = biases ? group_map(biases, N, K / kGroup, &bmap) : (bmap = smap, TB_OK);
  if (rc != TB_OK) return rc;
  const int NT = bt_tiles_nt(M), MT = 8 * NT;
  uint8_t* base = static_cast<uint8_t*>(region);
  BatchArgs a = {};
  a.has_bias = biases != nullptr;
  a.y = y;
  a.part = reinterpret_cast<float*>(base + kBtCounterBytes);
  a.count = reinterpret_cast<int*>(base);
  a.N = (int)N;
  a.G = (int)(K / kGroup);
  a.C = C;
  a.n_tiles = (int)tiles;
  a.status = status;
  const uint8_t* blob0 = base + kBtCounterBytes + bt_part_bytes(MT);
  const int64_t S = tiles * C;
  const int grid = (int)(S < f.sms ? S : f.sms);
  switch (NT) {
    case 1: return launch_batch_nt<1>(map, smap, bmap, a, blob0, M, grid, f.smem_optin, f.device, s);
    case 2: return launch_batch_nt<2>(map, smap, bmap, a, blob0, M, grid, f.smem_optin, f.device, s);
    case 4: return launch_batch_nt<4>(map, smap, bmap, a, blob0, M, grid, f.smem_optin, f.device, s);
    default: return launch_batch_nt<8>(map, smap, bmap, a, blob0, M, grid, f.smem_optin, f.device, s);
  }
}

}  // namespace tb
