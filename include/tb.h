/*
 * tb.h — C ABI of the folded-Hadamard ternary "Packed" layer on one GB300 (sm_103a).
 *
 * The layer (restated from two pages about the Ternary-Bonsai-2-27B-mlx-2bit pack):
 *   [ARCH] "3.9GB 里藏了什么Bonsai 的混合注意力 推测解码 262K 上下文端侧架构逐层拆"
 *          (kwkr.cn/news/564617), sections "Hadamard 旋转把量化误差抹平的免费午餐" and
 *          "打包格式的工程MLX 2.25 bits 与 GGUF 的两种装箱";
 *   [PACK] PACK-RUNTIME.md walkthrough (lpnh.cn/news/2438023), sections
 *          "文本模型加载artifact.load_model 与 Packed 模块" and
 *          "仿射 2-bit 格式与 Prism contract v1".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All array arguments are DEVICE pointers owned by the caller; the library
 *    allocates no device memory and keeps no state between calls.
 *  - fp16 arrays are passed as uint16_t* holding IEEE binary16 bit patterns.
 *  - Every array is row-major and contiguous.  Device pointers must be 16-byte
 *    aligned (TB_ERR_ALIGN otherwise).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call is
 *    asynchronous on that stream; the return value reports argument validation
 *    and launch errors only.  Errors that depend on data (a bad code, an id out
 *    of range, a bounded wait that ran out) are OR-ed into the optional device
 *    word `dev_status` (TB_DEV_* bits), which the caller reads after a sync.
 *    Kernels never trap.
 *  - The layer refuses rather than guesses: a shape, block or group size it
 *    does not implement is an error, never a silent fallback.
 *  - Codes: ternary t in {-1,0,1} is stored as q = t + 1 in {0,1,2}; a uint32
 *    word holds 16 codes, code i of the word at bits 2i..2i+1 (least
 *    significant first); word j of a row holds the row's codes 16j..16j+15.
 *  - Group size 128 and 2 bits per code are fixed.  Per group: one fp16 scale s
 *    and one fp16 bias b (= -s in the pack); a code decodes to s*q + b.
 *  - Scale-only form: every call that takes `biases` also accepts NULL there.
 *    Each bias is then taken as the pack's -s (the fp16 sign bit of s flipped)
 *    and never read, so a code decodes to s*(q - 1) = s*t and the call reads
 *    1/64 byte less per weight.  For a pack written by tb_pack_w2 the result is
 *    bit-identical to passing its stored biases.  ([ARCH] "打包格式的工程": the
 *    stored bias is always -scale, so it adds bytes but no information.)
 *  - Hadamard block: 1024 (the pack's block_size) or 0 (= module not folded,
 *    no transform).  The transform is the normalised Sylvester-Walsh-Hadamard
 *    matrix in natural order, H[i][j] = (-1)^popcount(i&j), scaled by
 *    1/sqrt(1024) = 1/32, applied to consecutive 1024-element blocks of the
 *    last axis; the sign vector is indexed by the absolute position on that axis.
 */
#ifndef TB_H
#define TB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* return codes */
enum {
  TB_OK = 0,
  TB_ERR_NULL = -1,        /* a required pointer is NULL */
  TB_ERR_SHAPE = -2,       /* M, N, K, T, V or D out of range or not a multiple it must be */
  TB_ERR_UNSUPPORTED = -3, /* block not 0, 512, 1024, 2048 or 4096 (the chain and the
                              no-allocation GEMV: not 0 or 1024), or an algorithm not built */
  TB_ERR_VALUE = -4,       /* a host-checked value is invalid */
  TB_ERR_CUDA = -5,        /* a CUDA launch or query failed (see tb_last_cuda_error) */
  TB_ERR_ALIGN = -6,       /* a device pointer is not 16-byte aligned */
  TB_ERR_WORKSPACE = -7,   /* workspace NULL or smaller than the size query returned */
  TB_ERR_TOO_LARGE = -8    /* beyond a fixed limit: the no-allocation scratch, or the chain's M <= 8 and SM ring */
};

/* bits OR-ed into *dev_status by kernels */
#define TB_DEV_BAD_CODE 1  /* tb_pack_w2: a code outside {-1,0,1}; tb_transcode_gguf: a block
                              slot or digit that is not a trit */
#define TB_DEV_BAD_ID 2    /* tb_embed_lookup: an id outside [0, V) (its row is written as zeros) */
#define TB_DEV_TIMEOUT 4   /* a bounded wait inside a kernel gave up; outputs are not valid */
#define TB_DEV_BAD_PLAN 8  /* tb_chain_run: the plan does not match the launch (nothing computed) */

/* algorithm choice for tb_packed_linear_algo */
#define TB_ALGO_AUTO 0       /* the GEMV for M <= 2, the batched GEMV on mma.sync for 3..32
                                tokens, the batched-decode GEMV on tensor memory for 33..64, the
                                tensor-core GEMM above */
#define TB_ALGO_GEMV 1       /* fused sign*FWHT prologue + streaming W2 GEMV (the warp-level one);
                                any M (passes of 8 tokens) */
#define TB_ALGO_TC 2         /* FWHT kernel into the workspace + tcgen05/TMEM GEMM; any M */
#define TB_ALGO_GEMV_SYNC 3  /* the warp-level GEMV only (mma.sync on fp16 operands); any M */
#define TB_ALGO_GEMV_TMEM 4  /* the tensor-memory GEMV (tcgen05.mma on e4m3 operands, decoded
                                codes in tensor memory): M <= 2, K a multiple of 1024, block 0
                                or 1024, at most 6 1024-blocks of x per SM's share of the work;
                                TB_ERR_UNSUPPORTED where it does not apply.  Slower than the
                                warp-level GEMV at these token counts; never chosen by AUTO */
#define TB_ALGO_GEMV_WIDE 5  /* the batched-decode GEMV on tensor memory: the weights the MMA's
                                128-row side (decoded to fp16 s*q + b in tensor memory), the
                                tokens its N side; x' rotated into the workspace first, as for
                                TB_ALGO_TC (same workspace); M <= 64 (else passes of 64 tokens),
                                K a multiple of 1024 (TB_ERR_UNSUPPORTED otherwise) */
#define TB_ALGO_GEMV_BATCH 6 /* the batched-decode GEMV on mma.sync: x' rotated once into the
                                workspace as the mma's operand image (per 512-k chunk and pass of
                                8, 16, 32 or 64 tokens), then every unit of packed codes decoded
                                once and run against all tokens of the pass; any M (passes of 64
                                tokens above 32), K a multiple of 1024 (TB_ERR_UNSUPPORTED
                                otherwise); tb_packed_linear_algo_workspace_size gives its
                                workspace */

/* Human-readable text of a return code; never NULL. */
const char* tb_status_string(int status);

/* Text of the last CUDA error seen by this thread's calls (or ""). */
const char* tb_last_cuda_error(void);

/* Library version, major*10000 + minor*100 + patch. */
int tb_version(void);

/*
 * tb_pack_w2 — weight packer of the W2-g128 affine container.
 * [ARCH] "打包格式的工程": codes {0,1,2} rearranged into uint32 words; bias = -scale.
 *   codes   int8 [N, K], values in {-1,0,1}
 *   scales  fp16 [N, K/128]
 *   w       uint32 [N, K/16]   (out) packed codes, layout as above
 *   biases  fp16 [N, K/128]    (out) -scales (sign bit flipped; exact)
 *   dev_status optional int32: TB_DEV_BAD_CODE if a code is not -1, 0 or 1
 *              (that field is still written, as (t+1) & 3).
 * K must be a positive multiple of 128, N >= 1.
 */
int tb_pack_w2(const int8_t* codes, const uint16_t* scales, int64_t N, int64_t K,
               uint32_t* w, uint16_t* biases, int32_t* dev_status, void* stream);

/*
 * tb_unpack_w2 — inverse of the packer (verification support).
 * [ARCH] "打包格式的工程": the codec ships an independent unpack() to check the packing.
 *   w      uint32 [N, K/16];  codes int8 [N, K] (out) = q - 1 (a field q = 3 gives 2).
 * K must be a positive multiple of 16, N >= 1.
 */
int tb_unpack_w2(const uint32_t* w, int64_t N, int64_t K, int8_t* codes, void* stream);

/* GGUF block formats of the same trits (tb_transcode_gguf) */
#define TB_FMT_PQ2_0 1  /* 34 bytes per 128 weights: fp16 scale, 128 2-bit slots */
#define TB_FMT_PTQ1_0 2 /* 28 bytes per 128 weights: fp16 scale, 128 trits five per byte */

/*
 * tb_transcode_gguf — lossless transcoding of GGUF blocks into the W2-g128 container.
 * [ARCH] "打包格式的工程": PQ2_0 (34 bytes per 128 weights, each trit in a 2-bit slot) and
 * PTQ1_0 (28 bytes, dense trits) carry the same trits and group scales; the transcoder takes
 * the scale from the block header, sets the bias to its negation and rearranges the codes
 * into uint32 words.  The page gives the block sizes, not the byte layout inside a block;
 * the layout read here: bytes 0-1 the fp16 scale; PQ2_0: slot i at bits 2(i%4) of byte
 * 2 + i/4, slot value t + 1; PTQ1_0: byte 2 + j = sum_i (t[5j+i] + 1) * 3^i over the trits
 * 5j .. 5j+4 below 128 (first trit least significant; byte 27 holds trits 125..127).
 *   blocks  uint8, N * (K/128) blocks back to back, row by row (row n, group g at block
 *           n*K/128 + g); 2-byte aligned for PQ2_0, 4-byte aligned for PTQ1_0;
 *   format  TB_FMT_PQ2_0 or TB_FMT_PTQ1_0 (else TB_ERR_UNSUPPORTED);
 *   w       uint32 [N, K/16] (out), as tb_pack_w2 writes it; 16-byte aligned;
 *   scales  fp16 [N, K/128] (out); biases fp16 [N, K/128] (out, = -scales) or NULL.
 * K a positive multiple of 128, N >= 1.  dev_status optional: TB_DEV_BAD_CODE when a PQ2_0
 * slot holds 3, a PTQ1_0 byte is 243 or more, or a digit past trit 127 is not zero (the
 * outputs of such a block are then not valid).
 */
int tb_transcode_gguf(const uint8_t* blocks, int format, int64_t N, int64_t K, uint32_t* w,
                      uint16_t* scales, uint16_t* biases, int32_t* dev_status, void* stream);

/*
 * tb_gguf_linear — the packed layer read straight from GGUF blocks, no transcoding:
 *   y[M,N] = fwht(x)[M,K] . W[N,K]^T,  W[n, 128g + i] = d[n,g] * t[n, 128g + i],
 * the trits t and block scales d as the blocks hold them (the layout tb_transcode_gguf reads;
 * the scale-only form: a code q = t + 1 decodes to d * (q - 1)).  [ARCH] "打包格式的工程":
 * PQ2_0 and PTQ1_0 carry the same trits and scales as the 2.25-bit container; PTQ1_0 is the
 * densest of the three (1.75 bits per weight) and costs extra arithmetic to decode.
 *   x       fp16 [M, K];  signs, block: as tb_packed_linear (block 0: x used as it is);
 *   blocks  uint8, N * (K/128) blocks of `format` back to back, row by row; 16-byte aligned;
 *   format  TB_FMT_PQ2_0 or TB_FMT_PTQ1_0 (else TB_ERR_UNSUPPORTED);
 *   y       fp16 [M, N] (out);
 *   workspace  device scratch of at least tb_gguf_linear_workspace_size(M, K, block) bytes
 *           (x' [M, K] fp16; none needed for block 0), 16-byte aligned.
 * K a multiple of 1024 (TB_ERR_SHAPE otherwise), M, N >= 1.  dev_status optional:
 * TB_DEV_BAD_CODE when a PQ2_0 slot holds 3 (read as d * 2), a PTQ1_0 byte is 243 or more (read
 * as five trits of -1) or a PTQ1_0 digit past trit 127 is not zero (not read).  Tokens are taken
 * in passes of up to 4 (fewer when x' of 4 tokens does not fit in shared memory).
 */
/*
 * tb_encode_gguf — the other direction: the W2-g128 container (words and scales, the scale-only
 * reading: each bias taken as -scale, not read) written as GGUF blocks of `format`, in the layout
 * tb_transcode_gguf reads.  Lossless for codes 0..2; a code of 3 is not a trit: TB_DEV_BAD_CODE,
 * kept in its slot by PQ2_0, written as 2 by PTQ1_0.
 *   w       uint32 [N, K/16], 16-byte aligned;  scales fp16 [N, K/128];
 *   blocks  uint8 (out), N * (K/128) blocks; 2-byte aligned for PQ2_0, 4-byte for PTQ1_0.
 * K a positive multiple of 128, N >= 1.
 */
int tb_encode_gguf(const uint32_t* w, const uint16_t* scales, int64_t N, int64_t K, int format,
                   uint8_t* blocks, int32_t* dev_status, void* stream);

size_t tb_gguf_linear_workspace_size(int64_t M, int64_t K, int block);
int tb_gguf_linear(const uint16_t* x, const int8_t* signs, int block, const uint8_t* blocks, int format,
                   int64_t M, int64_t K, int64_t N, uint16_t* y, void* workspace, size_t workspace_bytes,
                   int32_t* dev_status, void* stream);

/*
 * tb_fwht — sign * normalised Walsh-Hadamard transform over blocks of `block` elements.
 * [ARCH] "Hadamard 旋转": fwht uses hadamard_transform with scale 1/sqrt(block);
 * forward multiplies by the signs first, the inverse multiplies by them again at the end.
 * [PACK] "仿射 2-bit 格式与 Prism contract v1": the pack uses block 1024; its loader also
 * accepts 512, 2048 and 4096.
 *   x  fp16 [M, K];  y fp16 [M, K] (out; y may equal x);
 *   signs int8 [K] of +-1, or NULL for all +1 (not checked on the device);
 *   forward (inverse = 0): y = (H/sqrt(block)) (signs * x) per block;
 *   inverse (inverse = 1): y = signs * ((H/sqrt(block)) x) per block.
 * Computed in fp32 (the scale 1/sqrt(block) rounded to fp32 for 512 and 2048, exact for
 * 1024 and 4096), rounded to fp16 (round to nearest even).  block: 512, 1024, 2048 or 4096
 * (else TB_ERR_UNSUPPORTED); K a positive multiple of block, M >= 1.
 */
int tb_fwht(const uint16_t* x, uint16_t* y, const int8_t* signs, int64_t M, int64_t K,
            int block, int inverse, void* stream);

/*
 * Bytes of workspace tb_packed_linear uses for these sizes.  Layout: a fixup region
 * (about 2 MB) for the decode GEMV's split schedule: counters of output tiles shared by
 * several SMs in its first 1024 bytes, then the SMs' fp32 parts of those tiles; then, for
 * the tensor-core path, the rotated activations x' (fp16 [M, K]) and the split schedule's
 * counters and parts; then, for a block other than 0 and 1024, x' in natural order (fp16
 * [M, K]).  The first 1024 bytes
 * must be zero before the first call that uses the workspace (zero-filling the whole
 * workspace will do); every completed call leaves them zero (a call that reported
 * TB_DEV_TIMEOUT may not: zero them again).  Calls sharing one workspace must be
 * ordered on one stream.
 */
size_t tb_packed_linear_workspace_size(int64_t M, int64_t K, int64_t N, int block);
size_t tb_packed_linear_algo_workspace_size(int64_t M, int64_t K, int64_t N, int block, int algo);

/*
 * tb_packed_linear — Packed.__call__ on the non-embedding path.
 * [ARCH] "Hadamard 旋转" (a folded module rotates its input, then multiplies it by the
 * transposed 2-bit, group-128 affine matrix)
 * and [PACK] "文本模型加载" (packed weights consumed directly, never expanded).
 *   y[m, n] = sum_k x'[m, k] * (s[n, k/128] * q[n, k] + b[n, k/128]),
 *   x' = fwht(x, block, signs) rounded to fp16 (x' = x when block = 0);
 *   x fp16 [M, K]; signs int8 [K] (+-1) or NULL (all +1; ignored when block = 0);
 *   w uint32 [N, K/16]; scales fp16 [N, K/128]; biases fp16 [N, K/128] or NULL
 *   (scale-only, b = -s); y fp16 [M, N] (out).
 * fp32 accumulation, fp16 output (round to nearest even).
 * block: 1024 (the pack's; the transform is fused into the matmul kernels), 0 (no transform),
 * or 512, 2048, 4096 (accepted by the pack's loader: x' = tb_fwht(x) into the workspace
 * first, then the matmul on it; the same x' rounded to fp16, one more launch).
 * K: positive multiple of 128 and of block.  M, N >= 1.
 * workspace: device memory of at least tb_packed_linear_workspace_size(...) bytes,
 * zero-filled before its first use (see above).  The GEMV path (M <= 8) with block 0 or 1024
 * also runs with workspace = NULL, then with output tiles never split between SMs (slower on
 * shapes whose row-tile count is not a multiple of the SM count).
 * dev_status optional (TB_DEV_TIMEOUT).
 */
int tb_packed_linear(const uint16_t* x, int64_t M, int64_t K, const int8_t* signs, int block,
                     const uint32_t* w, const uint16_t* scales, const uint16_t* biases, int64_t N,
                     uint16_t* y, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                     void* stream);

/* Same as tb_packed_linear with an explicit algorithm (TB_ALGO_*). */
int tb_packed_linear_algo(const uint16_t* x, int64_t M, int64_t K, const int8_t* signs, int block,
                          const uint32_t* w, const uint16_t* scales, const uint16_t* biases,
                          int64_t N, uint16_t* y, void* workspace, size_t workspace_bytes,
                          int32_t* dev_status, int algo, void* stream);

/*
 * tb_packed_linear_multi — tb_packed_linear for n (1..4) packed matrices that read the same
 * input x, as the q/k/v, gate/up and in_proj_qkv/in_proj_z modules of one layer do
 * ([ARCH] "Hadamard 旋转": the folded transform depends only on the input width, so the
 * modules that share x also share x' = fwht(x)).  x' is computed once per launch; matrix i
 * writes y[i] (fp16 [M, N[i]]).  w, scales, biases, N, y are HOST arrays of n entries holding
 * device pointers / row counts; biases (the array, or any entry) may be NULL (scale-only for
 * those matrices); K must be a positive multiple of 1024 (and of block); block as for
 * tb_packed_linear (512, 2048, 4096: x' computed once into the workspace).  Workspace as for
 * tb_packed_linear, sized with tb_packed_linear_workspace_size(M, K, max N, block).
 * The kernels are those AUTO picks for M: M <= 2, one decode GEMV launch for all matrices;
 * 3..32, one rotation into the operand image, then one batched GEMV launch per matrix; above,
 * one rotation, then one batched-decode GEMV (33..64) or tensor-core GEMM launch per matrix.
 */
int tb_packed_linear_multi(const uint16_t* x, int64_t M, int64_t K, const int8_t* signs, int block,
                           int n, const uint32_t* const* w, const uint16_t* const* scales,
                           const uint16_t* const* biases, const int64_t* N, uint16_t* const* y,
                           void* workspace, size_t workspace_bytes, int32_t* dev_status,
                           void* stream);

/*
 * Chained decode: a sequence of Packed linears (M <= 8 tokens) in one persistent launch.
 * [ARCH] "Hadamard 旋转": each linear is Packed.__call__ (fwht of its input, then the W2-g128
 * matmul); a decode step runs the model's linears one after another, every one reading what
 * an earlier one wrote.  [PACK] "文本模型加载": the modules and their packed tensors.
 *
 * Link i computes, for its input x and its n matrices (1..4, the modules that read the same
 * input), exactly what tb_packed_linear_multi computes.  The result of the whole chain equals
 * calling tb_packed_linear_multi once per link, in order, on one stream: link i reads x only
 * after every output of links 0..i-1 is complete, so x of a link may be (a slice of) any
 * earlier link's y.  The launch keeps one CTA per SM resident (a cooperative launch); while
 * the SMs wait for link i to complete, they already stream the packed weights of link i+1.
 */
typedef struct tb_chain_link {
  const uint16_t* x;          /* fp16 [M, K]; may be an output of an earlier link */
  const int8_t* signs;        /* int8 [K] (+-1) or NULL (all +1); ignored when block = 0 */
  int64_t K;                  /* positive multiple of 1024 (at most 2^20) */
  int32_t block;              /* 1024, or 0 = module not folded */
  int32_t n;                  /* matrices reading x: 1..4 */
  const uint32_t* w[4];       /* uint32 [N[i], K/16] packed codes */
  const uint16_t* scales[4];  /* fp16 [N[i], K/128] */
  const uint16_t* biases[4];  /* fp16 [N[i], K/128], or NULL (scale-only, b = -s) */
  int64_t N[4];               /* rows of matrix i, >= 1 */
  uint16_t* y[4];             /* fp16 [M, N[i]] (out) */
} tb_chain_link;

/* Bytes of device memory a plan of n_links links needs (an upper bound: 4 matrices per link). */
size_t tb_chain_plan_size(int n_links);

/*
 * tb_chain_plan — validate the links (same rules as tb_packed_linear_multi; M in 1..8) and
 * write the plan (link table + one TMA descriptor per matrix) to `plan`, device memory of at
 * least tb_chain_plan_size(n_links) bytes, 128-byte aligned, owned by the caller.  Copies the
 * plan on `stream` and waits for that copy (call it before any stream capture).  The plan
 * stays valid while every pointer in the links stays valid; it holds no other state.
 * Errors: TB_ERR_NULL, TB_ERR_SHAPE, TB_ERR_UNSUPPORTED, TB_ERR_ALIGN, TB_ERR_TOO_LARGE (M > 8),
 * TB_ERR_WORKSPACE (plan_bytes too small), TB_ERR_CUDA.
 */
int tb_chain_plan(const tb_chain_link* links, int n_links, int64_t M, void* plan,
                  size_t plan_bytes, void* stream);

/*
 * Bytes of workspace tb_chain_run uses (about 2 MB): counters in its first 1280 bytes, which
 * must be zero before the first run (zero-filling the whole workspace will do) and which every
 * completed run leaves zero (a run that reported TB_DEV_TIMEOUT may not: zero them again),
 * then per-SM fp32 parts of output tiles shared by several SMs (scratch).
 */
size_t tb_chain_workspace_size(void);

/*
 * tb_chain_set_wait — the bound of a plan's waits on the previous link.
 * Before its prologue, every CTA waits until all CTAs have counted the previous link complete;
 * that wait gives up after wait_ns nanoseconds (0 = the library default, 2 s), sets
 * TB_DEV_TIMEOUT and lets the run wind down (its outputs are then not valid; zero the
 * workspace's counters before the next run).  extra_count raises the count each link waits for
 * by that many, so that the wait cannot complete: it exists to test the timeout path without a
 * fault or a hang, and must be 0 for a run whose results are used.  Writes the two fields of the
 * plan on `stream` and waits for that copy.  Errors: TB_ERR_NULL, TB_ERR_ALIGN, TB_ERR_VALUE
 * (a negative value), TB_ERR_CUDA.  A new plan starts with wait_ns = 0 and extra_count = 0.
 */
int tb_chain_set_wait(void* plan, int64_t wait_ns, int32_t extra_count, void* stream);

/*
 * tb_chain_run — run a plan: one launch on `stream`, asynchronous.  n_links, M and max_K
 * (the largest K of the links) must be the values the plan was made with; a mismatch that
 * the device can see sets TB_DEV_BAD_PLAN and computes nothing.  Runs that share one
 * workspace must be ordered on one stream.  Errors: TB_ERR_NULL, TB_ERR_SHAPE, TB_ERR_ALIGN,
 * TB_ERR_WORKSPACE, TB_ERR_TOO_LARGE (more than 256 SMs, or M and max_K leave no room for
 * the weight ring in shared memory), TB_ERR_CUDA.  dev_status optional (TB_DEV_TIMEOUT,
 * TB_DEV_BAD_PLAN).
 */
int tb_chain_run(const void* plan, int n_links, int64_t M, int64_t max_K, void* workspace,
                 size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * tb_embed_lookup — Packed.__call__ on the embedding path.
 * [ARCH] "Hadamard 旋转" (the looked-up rows are dequantised, then inverse-transformed) and
 * [PACK] "文本模型加载" (mx.dequantize of the looked-up rows, then the inverse transform).
 *   out[t, :] = signs * ((H/32) e) per block,  e = s*q + b of row ids[t] of the table.
 *   ids int32 [T]; w uint32 [V, D/16]; scales fp16 [V, D/128]; biases the same or NULL
 *   (scale-only, b = -s);
 *   signs int8 [D] (+-1) or NULL (all +1); out fp16 [T, D] (out).
 * An id outside [0, V) writes a row of zeros and sets TB_DEV_BAD_ID in dev_status.
 * block 1024 (fused), 512, 2048 or 4096 (the rows decoded into out, then the inverse
 * tb_fwht in place: the same result, since the pack's rows {-s, 0, s} are exact in fp16;
 * rows of a general affine bias are rounded to fp16 before that transform), or 0; D a
 * multiple of 128 and of block; T >= 0 (T = 0 is a no-op).
 */
int tb_embed_lookup(const int32_t* ids, int64_t T, const uint32_t* w, const uint16_t* scales,
                    const uint16_t* biases, int64_t V, int64_t D, const int8_t* signs, int block,
                    uint16_t* out, int32_t* dev_status, void* stream);

/*
 * tb_packed_linear_gemv_noalloc — the decode GEMV of tb_packed_linear for callers that
 * cannot provide device memory.  (No counterpart on the pages: it exists for callers
 * that are not allowed to allocate, e.g. code running under CUDA graph capture, plugins
 * inside a host runtime that owns all device memory, or services with a fixed memory
 * budget after start-up.)
 * Same arguments and result as tb_packed_linear for M <= 8 tokens, without workspace.
 * The state of the GEMV's split schedule lives in a fixed array inside the library
 * (about 2 MiB on every GPU that loads it, held until the process exits).
 *   - It allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *   - Limits: M <= 8 and a GPU with at most 256 SMs, else TB_ERR_TOO_LARGE;
 *     K a positive multiple of 1024 (block 1024, or block 0 with such a K), else TB_ERR_SHAPE.
 *   - The first call on each device looks up the array's device address for that device
 *     (cudaGetSymbolAddress); make that first call before any stream capture.
 *   - Each call clears the array's counters on `stream` before using it (cudaMemsetAsync).  All calls
 *     share the one array: calls that can overlap on the GPU (different streams, or
 *     different host threads) race and give wrong results; order them on one stream.
 */
int tb_packed_linear_gemv_noalloc(const uint16_t* x, int64_t M, int64_t K, const int8_t* signs,
                                  int block, const uint32_t* w, const uint16_t* scales,
                                  const uint16_t* biases, int64_t N, uint16_t* y,
                                  int32_t* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TB_H */
