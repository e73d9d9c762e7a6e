// Entry points of the non-embedding path: argument checks and the choice of kernel by token
// count: the streaming GEMV (M <= 2), the batched GEMV on mma.sync (3..32), the batched GEMV on
// tensor memory (33..64) and the tensor-core GEMM (prefill).
//
// [ARCH] kwkr.cn/news/564617, section "Hadamard 旋转把量化误差抹平的免费午餐":
//   the module's forward pass rotates the input (signs, then the normalised block Hadamard
//   transform) when the module is folded, and then multiplies the result by the transposed
//   2-bit, group-128 affine weight matrix with its scales and biases.
#include <cuda_runtime.h>

#include "tb_common.cuh"
#include "tb_host.h"

namespace tb {

int launch_gemv(const __half* x, int64_t M, int64_t K, const int8_t* signs, int block,
                const uint32_t* w, const __half* scales, const __half* biases, int64_t N,
                __half* y, int32_t* status, cudaStream_t s);
int launch_gemm_tc(const __half* x, int64_t M, int64_t K, const int8_t* signs, int block,
                   const uint32_t* w, const __half* scales, const __half* biases, int64_t N,
                   __half* y, void* workspace, int32_t* status, cudaStream_t s);
size_t gemm_tc_workspace(int64_t M, int64_t K, int64_t N);
size_t gemm_tc_x_bytes(int64_t M, int64_t K);
int launch_gemv_tma(const __half* x, int64_t M, int64_t K, const int8_t* signs, int block,
                    const uint32_t* w, const __half* scales, const __half* biases, int64_t N,
                    __half* y, void* workspace, size_t ws_bytes, int32_t* status, cudaStream_t s);
size_t gemv_fixup_bytes();
int launch_gemv_tma_multi(const __half* x, int64_t M, int64_t K, const int8_t* signs, int block,
                          int nmat, const uint32_t* const* w, const __half* const* scales,
                          const __half* const* biases, const int64_t* N, __half* const* y,
                          void* workspace, size_t ws_bytes, int32_t* status, cudaStream_t s);
int launch_rotate_pairorder(const __half* x, __half* out, const int8_t* signs, int64_t M,
                            int64_t K, int rotate, cudaStream_t s);
int launch_gemm_tc_rotated(const __half* xp, int64_t M, int64_t K, const uint32_t* w,
                           const __half* scales, const __half* biases, int64_t N, __half* y,
                           void* gws, int32_t* status, cudaStream_t s);
int launch_gemv_f8_multi(const __half* x, int64_t M, int64_t K, const int8_t* signs, int block,
                         int nmat, const uint32_t* const* w, const __half* const* scales,
                         const __half* const* biases, const int64_t* N, __half* const* y,
                         void* workspace, size_t ws_bytes, int32_t* status, cudaStream_t s);
int launch_gemv_wide(const __half* xp, int64_t M, int64_t K, const uint32_t* w, const __half* scales,
                     const __half* biases, int64_t N, __half* y, int* count, float* part, int32_t* status,
                     cudaStream_t s);
size_t gemv_wide_part_bytes();
size_t gemm_tc_part_offset(int64_t M, int64_t K, int64_t N);
size_t gemv_batch_bytes(int64_t M, int64_t K);
int launch_batch_image(const __half* x, int64_t M, int64_t K, const int8_t* signs, int rotate,
                       void* region, cudaStream_t s);
int launch_batch_gemv(int64_t M, int64_t K, const uint32_t* w, const __half* scales, const __half* biases,
                      int64_t N, __half* y, void* region, int32_t* status, cudaStream_t s);
constexpr int kMaxMulti = 4;

// Workspace layout: [fixup region of the GEMV split schedule (zero before the first call,
// left zero by every completed call)][the tensor-core path's x' in pair order, counters and
// parts][x' in natural order for a block other than 1024], 1 KB aligned.
static size_t fixup_region() { return (gemv_fixup_bytes() + 1023) / 1024 * 1024; }

// Blocks 512, 2048 and 4096 are not fused into the matmul kernels: x' = fwht(x) goes through
// the workspace first, then the matmul runs unrotated on it (the same x', rounded to fp16, that
// the fused kernels compute for block 1024).
static bool separate_block(int block) { return block != 0 && block != kBlock; }
static size_t natural_x_bytes(int64_t M, int64_t K) { return (size_t)((M * K * 2 + 1023) / 1024 * 1024); }

// AUTO's token-count bounds, from same-box timings of the four kernels on the 27B model's layer
// shapes (5120 -> 17408, 17408 -> 5120, 5120 -> 6144): the streaming GEMV up to kGemvMaxTokens
// (its fused prologue transforms every token's x in every CTA, which costs more per token than
// the batched GEMV's one rotation pass from three tokens on), the batched GEMV on mma.sync up to
// kBatchMaxTokens (above it, 40..64 tokens, its MMAs cost more than the tensor-memory kernel's),
// the tensor-memory one up to kWideMaxTokens, the tensor-core GEMM above
constexpr int64_t kGemvMaxTokens = 2;
constexpr int64_t kBatchMaxTokens = 32;
constexpr int64_t kWideMaxTokens = 64;

static int resolve_algo(int64_t M, int algo) {
  if (algo == TB_ALGO_AUTO)
    return M <= kGemvMaxTokens    ? TB_ALGO_GEMV
           : M <= kBatchMaxTokens ? TB_ALGO_GEMV_BATCH
           : M <= kWideMaxTokens  ? TB_ALGO_GEMV_WIDE
                                  : TB_ALGO_TC;
  return algo;
}
// the batched-decode GEMV uses the tensor-core path's workspace (x', then its parts region)
static bool uses_tc_workspace(int use) { return use == TB_ALGO_TC || use == TB_ALGO_GEMV_WIDE; }

// x' = fwht(x) in pair order into the workspace, then the batched-decode GEMV in passes of up to
// 64 tokens over it (K a multiple of 1024).
static int launch_wide_path(const __half* xh, int64_t M, int64_t K, const int8_t* sg, int block,
                            const uint32_t* w, const __half* sh, const __half* bh, int64_t N, __half* yh,
                            void* workspace, int32_t* dev_status, cudaStream_t s, bool rotate_x) {
  char* ws = static_cast<char*>(workspace);
  __half* xp = reinterpret_cast<__half*>(ws + fixup_region());
  if (rotate_x) {
    const int rc = launch_rotate_pairorder(xh, xp, sg, M, K, block != 0, s);
    if (rc != TB_OK) return rc;
  }
  int* count = reinterpret_cast<int*>(ws);
  float* part = reinterpret_cast<float*>(ws + fixup_region() + gemm_tc_part_offset(M, K, N));
  for (int64_t m0 = 0; m0 < M; m0 += kWideMaxTokens) {
    const int64_t mc = M - m0 < kWideMaxTokens ? M - m0 : kWideMaxTokens;
    const int rc = launch_gemv_wide(xp + m0 * K, mc, K, w, sh, bh, N, yh + m0 * N, count, part, dev_status, s);
    if (rc != TB_OK) return rc;
  }
  return TB_OK;
}

// The streaming GEMV (decode): the warp-level TMA kernel (K a multiple of 1024), else the
// row-streaming one; the tensor-memory kernel only when asked for (TB_ALGO_GEMV_TMEM: at one or
// two tokens it measured slower, its MMA issue rate being below the weights' arrival rate).
// `which` is TB_ALGO_GEMV, _GEMV_SYNC or _GEMV_TMEM.
static int launch_streaming_gemv(int which, const __half* x, int64_t M, int64_t K, const int8_t* sg,
                                 int block, int n, const uint32_t* const* w, const __half* const* sh,
                                 const __half* const* bh, const int64_t* N, __half* const* yh,
                                 void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                 cudaStream_t s) {
  if (which == TB_ALGO_GEMV_TMEM)
    return K % kBlock == 0 ? launch_gemv_f8_multi(x, M, K, sg, block, n, w, sh, bh, N, yh, workspace,
                                                  workspace_bytes, dev_status, s)
                           : TB_ERR_UNSUPPORTED;
  if (K % kBlock == 0)  // TMA-streamed GEMV; without a workspace its ranges stay on tile bounds
    return launch_gemv_tma_multi(x, M, K, sg, block, n, w, sh, bh, N, yh, workspace, workspace_bytes,
                                 dev_status, s);
  if (n != 1) return TB_ERR_SHAPE;
  return launch_gemv(x, M, K, sg, block, w[0], sh[0], bh[0], N[0], yh[0], dev_status, s);
}

static int check_linear_shape(int64_t M, int64_t K, int block, int64_t N) {
  if (block != 0 && !supported_block(block)) return TB_ERR_UNSUPPORTED;
  if (M < 1 || N < 1 || K < kGroup || K % kGroup) return TB_ERR_SHAPE;
  if (block && K % block) return TB_ERR_SHAPE;
  return TB_OK;
}

// bytes the matmul path itself needs after the GEMV's fixup region: the tensor-core path's x'
// and schedule state, or the batched GEMV's counters, parts and operand images
static size_t matmul_region(int64_t M, int64_t K, int64_t N, int use) {
  if (uses_tc_workspace(use)) return gemm_tc_workspace(M, K, N);
  if (use == TB_ALGO_GEMV_BATCH) return gemv_batch_bytes(M, K);
  return 0;
}

// bytes of workspace one call needs: the GEMV's fixup region, the matmul path's region, and x'
// in natural order for a block that is not fused
static size_t linear_workspace(int64_t M, int64_t K, int64_t N, int block, int use) {
  size_t b = fixup_region() + matmul_region(M, K, N, use);
  if (separate_block(block)) b += natural_x_bytes(M, K);
  return b;
}

// where x' in natural order goes: after everything the matmul path itself uses
static __half* natural_x(void* workspace, int64_t M, int64_t K, int64_t N, int use) {
  return reinterpret_cast<__half*>(static_cast<char*>(workspace) + fixup_region() +
                                   matmul_region(M, K, N, use));
}

// x' once into the batch region as the operand image, then the batched GEMV per matrix
static int launch_batch_path(const __half* xh, int64_t M, int64_t K, const int8_t* sg, int block, int n,
                             const uint32_t* const* w, const __half* const* sh, const __half* const* bh,
                             const int64_t* N, __half* const* yh, void* workspace, int32_t* dev_status,
                             cudaStream_t s) {
  void* region = static_cast<char*>(workspace) + fixup_region();
  int rc = launch_batch_image(xh, M, K, sg, block != 0, region, s);
  for (int i = 0; i < n && rc == TB_OK; ++i)
    rc = launch_batch_gemv(M, K, w[i], sh[i], bh[i], N[i], yh[i], region, dev_status, s);
  return rc;
}

}  // namespace tb

extern "C" size_t tb_packed_linear_algo_workspace_size(int64_t M, int64_t K, int64_t N, int block,
                                                       int algo) {
  using namespace tb;
  if (check_linear_shape(M, K, block, N) != TB_OK) return 0;
  return linear_workspace(M, K, N, block, resolve_algo(M, algo));
}

extern "C" size_t tb_packed_linear_workspace_size(int64_t M, int64_t K, int64_t N, int block) {
  return tb_packed_linear_algo_workspace_size(M, K, N, block, TB_ALGO_AUTO);
}

extern "C" int tb_packed_linear_algo(const uint16_t* x, int64_t M, int64_t K, const int8_t* signs,
                                     int block, const uint32_t* w, const uint16_t* scales,
                                     const uint16_t* biases, int64_t N, uint16_t* y,
                                     void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                     int algo, void* stream) {
  using namespace tb;
  if (!x || !w || !scales || !y) return TB_ERR_NULL;  // biases may be NULL: each is -scale
  int rc = check_linear_shape(M, K, block, N);
  if (rc != TB_OK) return rc;
  if (algo < TB_ALGO_AUTO || algo > TB_ALGO_GEMV_BATCH) return TB_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(w) || !aligned16(scales) || (biases && !aligned16(biases)) ||
      !aligned16(y) ||
      (signs && !aligned16(signs)) || (workspace && !aligned16(workspace)))
    return TB_ERR_ALIGN;
  const int use = resolve_algo(M, algo);
  const int8_t* sg = block ? signs : nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const __half* xh = reinterpret_cast<const __half*>(x);
  const __half* sh = reinterpret_cast<const __half*>(scales);
  const __half* bh = reinterpret_cast<const __half*>(biases);
  __half* yh = reinterpret_cast<__half*>(y);
  if (separate_block(block)) {  // x' = fwht(x) into the workspace, then the unrotated matmul
    if (!workspace || workspace_bytes < linear_workspace(M, K, N, block, use)) return TB_ERR_WORKSPACE;
    __half* xn = natural_x(workspace, M, K, N, use);
    int rc2 = launch_fwht(xh, xn, sg, M, K, block, 0, s);
    if (rc2 != TB_OK) return rc2;
    xh = xn;
    sg = nullptr;
    block = 0;
  }
  if (use == TB_ALGO_GEMV_BATCH) {
    if (K % kBlock) return TB_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < fixup_region() + gemv_batch_bytes(M, K)) return TB_ERR_WORKSPACE;
    return launch_batch_path(xh, M, K, sg, block, 1, &w, &sh, &bh, &N, &yh, workspace, dev_status, s);
  }
  if (use == TB_ALGO_GEMV_WIDE) {
    if (K % kBlock) return TB_ERR_UNSUPPORTED;
    const size_t need = fixup_region() + gemm_tc_workspace(M, K, N);
    if (!workspace || workspace_bytes < need) return TB_ERR_WORKSPACE;
    return launch_wide_path(xh, M, K, sg, block, w, sh, bh, N, yh, workspace, dev_status, s, true);
  }
  if (use == TB_ALGO_TC) {
    const size_t need = fixup_region() + gemm_tc_workspace(M, K, N);
    if (!workspace || workspace_bytes < need) return TB_ERR_WORKSPACE;
    return launch_gemm_tc(xh, M, K, sg, block, w, sh, bh, N, yh,
                          static_cast<char*>(workspace) + fixup_region(), dev_status, s);
  }
  return launch_streaming_gemv(use, xh, M, K, sg, block, 1, &w, &sh, &bh, &N, &yh, workspace,
                               workspace_bytes, dev_status, s);
}

extern "C" int tb_packed_linear(const uint16_t* x, int64_t M, int64_t K, const int8_t* signs,
                                int block, const uint32_t* w, const uint16_t* scales,
                                const uint16_t* biases, int64_t N, uint16_t* y, void* workspace,
                                size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return tb_packed_linear_algo(x, M, K, signs, block, w, scales, biases, N, y, workspace,
                               workspace_bytes, dev_status, TB_ALGO_AUTO, stream);
}

extern "C" int tb_packed_linear_multi(const uint16_t* x, int64_t M, int64_t K, const int8_t* signs,
                                      int block, int n, const uint32_t* const* w,
                                      const uint16_t* const* scales, const uint16_t* const* biases,
                                      const int64_t* N, uint16_t* const* y, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status, void* stream) {
  using namespace tb;
  if (!x || !w || !scales || !N || !y) return TB_ERR_NULL;  // biases (or an entry) may be NULL
  if (n < 1 || n > kMaxMulti) return TB_ERR_SHAPE;
  if (block != 0 && !supported_block(block)) return TB_ERR_UNSUPPORTED;
  if (M < 1 || K < kBlock || K % kBlock || (block && K % block)) return TB_ERR_SHAPE;
  if (!aligned16(x) || (signs && !aligned16(signs)) || (workspace && !aligned16(workspace)))
    return TB_ERR_ALIGN;
  const __half* sh[kMaxMulti];
  const __half* bh[kMaxMulti];
  __half* yh[kMaxMulti];
  for (int i = 0; i < n; ++i) {
    const uint16_t* bi = biases ? biases[i] : nullptr;
    if (!w[i] || !scales[i] || !y[i]) return TB_ERR_NULL;
    if (N[i] < 1) return TB_ERR_SHAPE;
    if (!aligned16(w[i]) || !aligned16(scales[i]) || !aligned16(y[i]) || (bi && !aligned16(bi)))
      return TB_ERR_ALIGN;
    sh[i] = reinterpret_cast<const __half*>(scales[i]);
    bh[i] = reinterpret_cast<const __half*>(bi);
    yh[i] = reinterpret_cast<__half*>(y[i]);
  }
  const int8_t* sg = block ? signs : nullptr;
  const __half* xh = reinterpret_cast<const __half*>(x);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (separate_block(block)) {  // x' once into the workspace, then the unrotated matrices
    int64_t maxN = 0;
    for (int i = 0; i < n; ++i) maxN = N[i] > maxN ? N[i] : maxN;
    const int use = resolve_algo(M, TB_ALGO_AUTO);
    if (!workspace || workspace_bytes < linear_workspace(M, K, maxN, block, use)) return TB_ERR_WORKSPACE;
    __half* xn = natural_x(workspace, M, K, maxN, use);
    int rc2 = launch_fwht(xh, xn, sg, M, K, block, 0, s);
    if (rc2 != TB_OK) return rc2;
    xh = xn;
    sg = nullptr;
    block = 0;
  }
  if (M <= kGemvMaxTokens)
    return launch_streaming_gemv(TB_ALGO_GEMV, xh, M, K, sg, block, n, w, sh, bh, N, yh, workspace,
                                 workspace_bytes, dev_status, s);
  if (M <= kBatchMaxTokens) {  // one rotation into the operand image, then one launch per matrix
    if (!workspace || workspace_bytes < fixup_region() + gemv_batch_bytes(M, K)) return TB_ERR_WORKSPACE;
    return launch_batch_path(xh, M, K, sg, block, n, w, sh, bh, N, yh, workspace, dev_status, s);
  }
  // prefill: one rotation of x into the workspace, then one GEMM per matrix
  int64_t maxN = 0;
  for (int i = 0; i < n; ++i) maxN = N[i] > maxN ? N[i] : maxN;
  const size_t need = fixup_region() + gemm_tc_workspace(M, K, maxN);
  if (!workspace || workspace_bytes < need) return TB_ERR_WORKSPACE;
  __half* xp = reinterpret_cast<__half*>(static_cast<char*>(workspace) + fixup_region());
  void* gws = static_cast<char*>(workspace) + fixup_region() + gemm_tc_x_bytes(M, K);
  int rc = launch_rotate_pairorder(xh, xp, sg, M, K, block != 0, s);
  for (int i = 0; i < n && rc == TB_OK; ++i)
    rc = M <= kWideMaxTokens
             ? launch_wide_path(xh, M, K, sg, block, w[i], sh[i], bh[i], N[i], yh[i], workspace, dev_status, s, false)
             : launch_gemm_tc_rotated(xp, M, K, w[i], sh[i], bh[i], N[i], yh[i], gws, dev_status, s);
  return rc;
}
