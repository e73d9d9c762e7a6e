// Packed linear read straight from the GGUF blocks of the ternary weights (no transcoding):
// y[M, N] = x'[M, K] . W[N, K]^T with W[n, k] = d_g * t (t in {-1, 0, 1}, one fp16 scale d_g per
// block of 128 weights), x' = the rotated activations.
//
// [ARCH] kwkr.cn/news/564617, section "打包格式的工程MLX 2.25 bits 与 GGUF 的两种装箱": the same
// trits and group scales packed as PQ2_0 (34 bytes per 128 weights, each trit in a 2-bit slot) or
// PTQ1_0 (28 bytes, five trits per byte, the densest form, at the price of extra arithmetic to
// decode).  The byte layout inside a block is the one tb_transcode_gguf reads: bytes 0-1 the fp16
// scale; PQ2_0 slot i at bits 2(i%4) of byte 2 + i/4 holding t + 1; PTQ1_0 byte 2 + j holding
// sum_i (t[5j+i] + 1) 3^i over the trits 5j .. 5j+4 below 128.
//
// Arithmetic: a code q = t + 1 in {0, 1, 2} is made an exact float by putting its field, left in
// place (bits 2f of a 16-bit word, or of a decoded PTQ1_0 byte), into the mantissa of 2^23 and
// subtracting 2^23: q * 4^f.  The activations are stored in shared memory multiplied by 4^-f for
// the position f their code has in its word, so q * 4^f * (x * 4^-f) = q * x with no extra
// instruction, and per block y += d * (sum q x - sum x).  Decoding runs on the CUDA cores: at one
// token a weight costs an and-or, an add and an FMA, while the block bytes stream from HBM.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "tb_common.cuh"
#include "tb_host.h"

namespace tb {

constexpr int kGgWarps = 16;    // warps per CTA (one CTA per SM)
constexpr int kGgStages = 4;    // staged block iterations per warp in flight (cp.async)
constexpr int kGgLanesPerRow = 8;
constexpr int kGgRowsPerWarp = 32 / kGgLanesPerRow;

template <int FMT>
struct GgFmt {
  static constexpr int kBytes = FMT == TB_FMT_PQ2_0 ? 34 : 28;      // bytes per block of 128
  static constexpr int kRowBytes = kGgLanesPerRow * kBytes;         // one iteration of one row
  static constexpr int kStageBytes = kGgRowsPerWarp * kRowBytes;    // 1088 or 896
  static constexpr int kChunks = kRowBytes / 16;                    // 16-byte copies per row
  static constexpr int kLutBytes = FMT == TB_FMT_PTQ1_0 ? 256 * 32 * 4 : 0;
};

// shared memory of one CTA: staging rings, the activation image, per-block sums, the table
template <int FMT, int MT>
__host__ __device__ constexpr int gg_smem_bytes(int G) {
  return kGgWarps * kGgStages * GgFmt<FMT>::kStageBytes + MT * G * 128 * 4 + MT * G * 4 +
         GgFmt<FMT>::kLutBytes;
}

TB_DEVI void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
TB_DEVI void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
TB_DEVI void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

TB_DEVI uint32_t ld_shared_u16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}

// the field of `word` under `mask` (a code left in place) as an exact float: field value
TB_DEVI float field_float(uint32_t word, uint32_t mask) {
  return __int_as_float(static_cast<int>((word & mask) | 0x4B000000u)) - 8388608.0f;
}

// One warp: rows 4 at a time (eight lanes per row), each lane one block of its row per iteration;
// x' [MT][K] fp16 (natural order), blocks [N][G] of FMT, y [MT][N] fp16.
template <int FMT, int MT>
__global__ void __launch_bounds__(kGgWarps * 32, 1)
    gguf_gemv_kernel(const uint8_t* __restrict__ blocks, const __half* __restrict__ xp, int64_t N, int K,
                     __half* __restrict__ y, int32_t* status) {
  using F = GgFmt<FMT>;
  const int G = K / 128;
  const int nb = G / kGgLanesPerRow;  // iterations per row group
  extern __shared__ __align__(16) uint8_t sm[];
  uint8_t* ring = sm;
  float* ximg = reinterpret_cast<float*>(sm + kGgWarps * kGgStages * F::kStageBytes);
  float* xsum = ximg + MT * G * 128;
  uint32_t* lut = reinterpret_cast<uint32_t*>(xsum + MT * G);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- prologue: the activation image, the per-block sums of x', the base-3 table ----
  // PQ2_0 image: float4 [t][m = 0..15][h = 0..1][g], positions 8m + 4h .. + 3 of block g, each
  // times 4^-(position % 8); PTQ1_0 image: float [t][p = 0..127][g], times 4^-(p % 5).  Consecutive
  // blocks are consecutive in shared memory, so the eight lanes of a row read without conflicts.
  for (int tg = warp; tg < MT * G; tg += kGgWarps) {
    const int t = tg / G, g = tg % G;
    const __half* src = xp + (int64_t)t * K + (int64_t)g * 128 + lane * 4;
    const uint2 raw = *reinterpret_cast<const uint2*>(src);
    const __half* h4 = reinterpret_cast<const __half*>(&raw);
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int p = lane * 4 + e;
      const float v = __half2float(h4[e]);
      s += v;
      if constexpr (FMT == TB_FMT_PQ2_0) {
        const float sc = __int_as_float((127 - 2 * (p % 8)) << 23);  // 4^-(p % 8)
        const int m = p / 8, h = (p % 8) / 4, k = p % 4;
        ximg[((((t * 16 + m) * 2 + h) * G + g) * 4) + k] = v * sc;
      } else {
        const float sc = __int_as_float((127 - 2 * (p % 5)) << 23);  // 4^-(p % 5)
        ximg[(t * 128 + p) * G + g] = v * sc;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) xsum[t * G + g] = s;
  }
  if constexpr (FMT == TB_FMT_PTQ1_0) {
    // byte value v -> its five base-3 digits (first trit least significant) at bits 2k; values
    // 243..255 are not five trits: all zero digits here, flagged where a block holds one
    for (int i = threadIdx.x; i < 256 * 32; i += blockDim.x) {
      const int v = i >> 5;
      uint32_t e = 0;
      if (v < 243) {
        int r = v;
#pragma unroll
        for (int k = 0; k < 5; ++k) {
          e |= (uint32_t)(r % 3) << (2 * k);
          r /= 3;
        }
      }
      lut[i] = e;  // [v][lane]: every lane reads its own bank
    }
  }
  __syncthreads();

  // ---- main loop ----
  const int r = lane / kGgLanesPerRow, l = lane % kGgLanesPerRow;
  const int64_t rgroups = (N + kGgRowsPerWarp - 1) / kGgRowsPerWarp;
  const int64_t wstride = (int64_t)gridDim.x * kGgWarps;
  const int64_t wid = (int64_t)blockIdx.x * kGgWarps + warp;
  const int64_t my_groups = wid < rgroups ? (rgroups - wid + wstride - 1) / wstride : 0;
  const int64_t items = my_groups * nb;
  const int64_t row_bytes = (int64_t)G * F::kBytes;
  const uint32_t ring_u32 = smem_u32(ring) + (uint32_t)warp * kGgStages * F::kStageBytes;

  auto issue = [&](int64_t i) {  // stage item i (row group, block iteration) into its ring slot
    if (i < items) {
      const int64_t rg = wid + (i / nb) * wstride;
      const int b = (int)(i % nb);
      const uint32_t dst = ring_u32 + (uint32_t)(i % kGgStages) * F::kStageBytes;
      for (int c = lane; c < kGgRowsPerWarp * F::kChunks; c += 32) {
        const int rr = c / F::kChunks, piece = c % F::kChunks;
        const int64_t row = rg * kGgRowsPerWarp + rr;
        if (row < N)
          cp_async16(dst + (uint32_t)(rr * F::kRowBytes + piece * 16),
                     blocks + row * row_bytes + (int64_t)b * F::kRowBytes + piece * 16);
      }
    }
    cp_async_commit();  // one group per item, empty past the end
  };
#pragma unroll
  for (int i = 0; i < kGgStages; ++i) issue(i);

  float ypart[MT];
#pragma unroll
  for (int t = 0; t < MT; ++t) ypart[t] = 0.f;
  bool bad = false;
  for (int64_t i = 0; i < items; ++i) {
    cp_async_wait<kGgStages - 1>();
    __syncwarp();  // the other lanes' copies of this stage are visible
    const int b = (int)(i % nb);
    const int g = b * kGgLanesPerRow + l;
    const int64_t row = (wid + (i / nb) * wstride) * kGgRowsPerWarp + r;  // past N: stale stage, not reported
    bool bi = false;
    const uint32_t blk = ring_u32 + (uint32_t)(i % kGgStages) * F::kStageBytes + (uint32_t)(r * F::kRowBytes + l * F::kBytes);
    const float d = __half2float(__ushort_as_half((uint16_t)ld_shared_u16(blk)));
    float acc[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) acc[t] = 0.f;
    if constexpr (FMT == TB_FMT_PQ2_0) {
#pragma unroll 4
      for (int m = 0; m < 16; ++m) {
        const uint32_t v = ld_shared_u16(blk + 2 + 2 * m);  // slots 8m .. 8m+7 at bits 2f
        bi |= ((v & (v >> 1) & 0x5555u) != 0);              // a slot holding 3 is not a trit
        float q[8];
#pragma unroll
        for (int f = 0; f < 8; ++f) q[f] = field_float(v, 3u << (2 * f));
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          const float4* xi = reinterpret_cast<const float4*>(ximg) + (((t * 16 + m) * 2) * G + g);
          const float4 a0 = xi[0], a1 = xi[G];
          acc[t] = fmaf(q[0], a0.x, acc[t]);
          acc[t] = fmaf(q[1], a0.y, acc[t]);
          acc[t] = fmaf(q[2], a0.z, acc[t]);
          acc[t] = fmaf(q[3], a0.w, acc[t]);
          acc[t] = fmaf(q[4], a1.x, acc[t]);
          acc[t] = fmaf(q[5], a1.y, acc[t]);
          acc[t] = fmaf(q[6], a1.z, acc[t]);
          acc[t] = fmaf(q[7], a1.w, acc[t]);
        }
      }
    } else {
      const uint32_t lut_lane = smem_u32(lut) + (uint32_t)lane * 4u;
#pragma unroll
      for (int m = 0; m < 13; ++m) {
        const uint32_t v = ld_shared_u16(blk + 2 + 2 * m);  // bytes 2m, 2m + 1 of the trits
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          const int j = 2 * m + hb;  // byte j: trits 5j .. 5j+4 (three below 128 in byte 25)
          const uint32_t byte = (v >> (8 * hb)) & 0xFFu;
          uint32_t e;
          asm volatile("ld.shared.u32 %0, [%1];" : "=r"(e) : "r"(lut_lane + byte * 128u));
          bi |= byte >= 243u;
          if (j == 25) bi |= (e >> 6) != 0;  // digits past trit 127 must be zero
          const int nk = j == 25 ? 3 : 5;
#pragma unroll
          for (int k = 0; k < 5; ++k) {
            if (k >= nk) break;
            const float q = field_float(e, 3u << (2 * k));
            const int p = 5 * j + k;
#pragma unroll
            for (int t = 0; t < MT; ++t) acc[t] = fmaf(q, ximg[(t * 128 + p) * G + g], acc[t]);
          }
        }
      }
    }
    bad |= bi && row < N;
#pragma unroll
    for (int t = 0; t < MT; ++t) ypart[t] = fmaf(d, acc[t] - xsum[t * G + g], ypart[t]);
    __syncwarp();  // every lane has read the stage before it is refilled
    issue(i + kGgStages);
    if (b == nb - 1) {  // the row group's last iteration: the eight lanes of each row add up
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        float s = ypart[t];
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        s += __shfl_xor_sync(0xffffffffu, s, 4);
        if (l == 0 && row < N) y[(int64_t)t * N + row] = __float2half_rn(s);
        ypart[t] = 0.f;
      }
    }
  }
  cp_async_wait<0>();
  if (bad && status) atomicOr(status, TB_DEV_BAD_CODE);
}

template <int FMT, int MT>
static int launch_gguf_pass(const uint8_t* blocks, const __half* xp, int64_t N, int K, __half* y,
                            int32_t* status, const DeviceFacts& f, cudaStream_t s) {
  const int smem = gg_smem_bytes<FMT, MT>(K / 128);
  // the kernel's shared-memory limit is raised once per device, to the device's opt-in maximum
  static int raised[64];
  if (f.device < 0 || f.device >= 64) return TB_ERR_CUDA;
  if (raised[f.device] != f.smem_optin) {
    cudaError_t e = cudaFuncSetAttribute(gguf_gemv_kernel<FMT, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         f.smem_optin);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      return TB_ERR_CUDA;
    }
    raised[f.device] = f.smem_optin;
  }
  const int64_t groups = (N + kGgRowsPerWarp - 1) / kGgRowsPerWarp;
  int64_t grid = (groups + kGgWarps - 1) / kGgWarps;
  if (grid > f.sms) grid = f.sms;
  gguf_gemv_kernel<FMT, MT><<<(int)grid, kGgWarps * 32, smem, s>>>(blocks, xp, N, K, y, status);
  return check_launch();
}

// tokens per pass: as many (1, 2 or 4) as the activation image leaves room for
template <int FMT>
static int gguf_tokens_per_pass(int K, int smem_optin) {
  const int G = K / 128;
  if (gg_smem_bytes<FMT, 4>(G) <= smem_optin) return 4;
  if (gg_smem_bytes<FMT, 2>(G) <= smem_optin) return 2;
  if (gg_smem_bytes<FMT, 1>(G) <= smem_optin) return 1;
  return 0;
}

template <int FMT>
static int launch_gguf(const uint8_t* blocks, const __half* xp, int64_t M, int64_t N, int K, __half* y,
                       int32_t* status, cudaStream_t s) {
  DeviceFacts f;
  int rc = device_facts(&f);
  if (rc != TB_OK) return rc;
  const int mt = gguf_tokens_per_pass<FMT>(K, f.smem_optin);
  if (mt == 0) return TB_ERR_TOO_LARGE;
  for (int64_t t0 = 0; t0 < M;) {
    const int64_t m = M - t0;
    const int w = (m >= 4 && mt >= 4) ? 4 : (m >= 2 && mt >= 2) ? 2 : 1;  // tokens in this pass
    const __half* xt = xp + t0 * K;
    __half* yt = y + t0 * N;
    rc = w == 4 ? launch_gguf_pass<FMT, 4>(blocks, xt, N, K, yt, status, f, s)
       : w == 2 ? launch_gguf_pass<FMT, 2>(blocks, xt, N, K, yt, status, f, s)
                : launch_gguf_pass<FMT, 1>(blocks, xt, N, K, yt, status, f, s);
    if (rc != TB_OK) return rc;
    t0 += w;
  }
  return TB_OK;
}

}  // namespace tb

extern "C" size_t tb_gguf_linear_workspace_size(int64_t M, int64_t K, int block) {
  if (M < 1 || K < 1 || block == 0) return 0;
  return (size_t)M * (size_t)K * 2;  // x' [M, K] fp16
}

extern "C" int tb_gguf_linear(const uint16_t* x, const int8_t* signs, int block, const uint8_t* blocks, int format,
                              int64_t M, int64_t K, int64_t N, uint16_t* y, void* workspace,
                              size_t workspace_bytes, int32_t* dev_status, void* stream) {
  using namespace tb;
  if (!x || !blocks || !y) return TB_ERR_NULL;
  if (format != TB_FMT_PQ2_0 && format != TB_FMT_PTQ1_0) return TB_ERR_UNSUPPORTED;
  if (block != 0 && !supported_block(block)) return TB_ERR_UNSUPPORTED;
  if (M < 1 || N < 1 || K < 1024 || K % 1024 || (block && K % block) || K > (1 << 24)) return TB_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(y) || !aligned16(blocks) || (signs && !aligned16(signs))) return TB_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const __half* xp = reinterpret_cast<const __half*>(x);
  if (block) {
    if (!workspace || workspace_bytes < tb_gguf_linear_workspace_size(M, K, block)) return TB_ERR_WORKSPACE;
    if (!aligned16(workspace)) return TB_ERR_ALIGN;
    __half* ws = static_cast<__half*>(workspace);
    const int rc = launch_fwht(xp, ws, signs, M, K, block, 0, s);
    if (rc != TB_OK) return rc;
    xp = ws;
  }
  __half* yh = reinterpret_cast<__half*>(y);
  return format == TB_FMT_PQ2_0 ? launch_gguf<TB_FMT_PQ2_0>(blocks, xp, M, N, (int)K, yh, dev_status, s)
                                : launch_gguf<TB_FMT_PTQ1_0>(blocks, xp, M, N, (int)K, yh, dev_status, s);
}
