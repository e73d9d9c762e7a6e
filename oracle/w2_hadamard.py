"""Plain CPU oracle of the folded-Hadamard ternary ``Packed`` layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this module.  The
CUDA library never calls it and shares no code with it.

Everything here is float64 NumPy written for clarity, not speed.  Sources
(cited by page and section; the pages are Chinese-language articles about the
Ternary-Bonsai-2-27B-mlx-2bit weight pack):

[ARCH]  "3.9GB 里藏了什么：Bonsai 的混合注意力 + 推测解码 + 262K 上下文端侧架构逐层拆"
        (kwkr.cn/news/564617)
        - section "Hadamard 旋转：把量化误差抹平的免费午餐": the ``Packed.__call__``
          code (fwht on activations, then quantized_matmul with group_size 128,
          bits 2, transpose; embedding path: dequantize then inverse fwht), and
          the statement that fwht scales by 1/sqrt(block), multiplies by the
          signs first on the forward path and again at the end on the inverse
          path.
        - section "打包格式的工程：MLX 2.25 bits 与 GGUF 的两种装箱": the affine
          container, one fp16 scale and one fp16 bias = -scale per 128 weights,
          2-bit codes {0,1,2} decoding to {-s, 0, s}; codes rearranged into
          uint32 words.
[PACK]  "PACK-RUNTIME.md" walkthrough (lpnh.cn/news/2438023)
        - section "文本模型加载：artifact.load_model 与 Packed 模块": the two
          forward paths of ``Packed``; packed uint32 weights never expanded.
        - section "仿射 2-bit 格式与 Prism contract v1": block_size 1024,
          transform normalized-sylvester-walsh-hadamard, axis
          input-last-dimension, explicit +-1 sign vectors.

Readings of points the pages leave open (each one is listed with its reason
in the design notes):
  * bit order: code k of a row sits in word k // 16 at bits 2*(k % 16) and up
    (least significant first); rows are contiguous along K;
  * Hadamard order: natural Sylvester order, H[i, j] = (-1)**popcount(i & j);
  * blocks are consecutive slices of ``block`` elements starting at index 0 of
    the last axis; the sign index is the absolute position along that axis;
  * the decoder applies the affine formula to any 2-bit code (code 3 -> 3s+b);
  * nothing is rounded: the oracle keeps x' = fwht(x) in float64.
"""
from __future__ import annotations

import numpy as np

GROUP = 128          # weights per scale/bias group
BITS = 2             # bits per code
CODES_PER_WORD = 16  # 2-bit codes in one uint32 word


# ----------------------------------------------------------------------------
# Normalised Sylvester-Walsh-Hadamard transform with explicit signs
# ----------------------------------------------------------------------------
def fwht(x, block: int, signs=None, inverse: bool = False) -> np.ndarray:
    """Blockwise sign + normalised Walsh-Hadamard transform along the last axis.

    [ARCH] "Hadamard 旋转" (fwht built on hadamard_transform with scale
    1/sqrt(block); forward: signs first, inverse: signs again last) and [PACK]
    "仿射 2-bit 格式与 Prism contract v1" (normalized Sylvester transform on
    the input's last dimension, block 1024).

    forward:  x'[b] = (1/sqrt(block)) * H_block @ (signs[b] * x[b])
    inverse:  x[b]  = signs[b] * ((1/sqrt(block)) * H_block @ x'[b])

    H is applied by the in-place butterfly: for h = 1, 2, 4, ..., block/2 every
    pair (i, i + h) with bit h of i clear becomes (a + b, a - b).  That is the
    recursion H_2n = [[H_n, H_n], [H_n, -H_n]] written as a loop.
    ``block == 0`` means "module not folded": x is returned unchanged.
    """
    x = np.asarray(x, dtype=np.float64)
    if block == 0:
        return x.copy()
    K = x.shape[-1]
    if block < 1 or block & (block - 1):
        raise ValueError("block must be a power of two")
    if K % block:
        raise ValueError("last dimension must be a multiple of the block size")
    s = np.ones(K) if signs is None else np.asarray(signs, dtype=np.float64)
    if s.shape != (K,):
        raise ValueError("signs must have one entry per element of the last axis")

    lead = x.shape[:-1]
    v = x * s if not inverse else x.copy()
    v = v.reshape(lead + (K // block, block))
    h = 1
    while h < block:
        v = v.reshape(lead + (K // block, block // (2 * h), 2, h))
        a = v[..., 0, :]
        b = v[..., 1, :]
        v = np.stack([a + b, a - b], axis=-2)
        h *= 2
    v = v.reshape(lead + (K,)) / np.sqrt(block)
    if inverse:
        v = v * s
    return v


# ----------------------------------------------------------------------------
# W2-g128 affine container
# ----------------------------------------------------------------------------
def pack_w2(codes) -> np.ndarray:
    """Ternary codes t in {-1,0,1} [N, K] -> uint32 words [N, K/16].

    [ARCH] "打包格式的工程": codes are stored as {0,1,2} (q = t + 1) and
    rearranged into uint32 words.  Word j of a row holds q[16j + i] at bits
    2i..2i+1 (least significant first).
    """
    t = np.asarray(codes)
    if t.ndim != 2 or t.shape[1] % CODES_PER_WORD:
        raise ValueError("codes must be [N, K] with K a multiple of 16")
    if not np.isin(t, (-1, 0, 1)).all():
        raise ValueError("ternary codes must be -1, 0 or 1")
    N, K = t.shape
    q = (t.astype(np.int64) + 1).reshape(N, K // CODES_PER_WORD, CODES_PER_WORD)
    words = np.zeros((N, K // CODES_PER_WORD), dtype=np.int64)
    for i in range(CODES_PER_WORD):
        words |= q[:, :, i] << (BITS * i)
    return words.astype(np.uint32)


def unpack_w2(words, K: int) -> np.ndarray:
    """uint32 words [N, K/16] -> codes t = q - 1 (int8) [N, K]; q = 3 gives 2."""
    w = np.asarray(words, dtype=np.uint64)
    N = w.shape[0]
    if w.shape[1] * CODES_PER_WORD != K:
        raise ValueError("word count does not match K")
    shifts = (BITS * np.arange(CODES_PER_WORD)).astype(np.uint64)
    q = (w[:, :, None] >> shifts) & np.uint64(3)
    return (q.reshape(N, K).astype(np.int64) - 1).astype(np.int8)


def biases_for(scales) -> np.ndarray:
    """The container's bias: b = -s for every group ([ARCH] "打包格式的工程")."""
    return (-np.asarray(scales, dtype=np.float16)).astype(np.float16)


def decode_w2(words, scales, biases, K: int) -> np.ndarray:
    """Dequantise to float64: W[n, k] = s[n, k//128] * q[n, k] + b[n, k//128].

    [ARCH] "打包格式的工程": with b = -s the codes {0,1,2} give exactly
    {-s, 0, s}.  The formula is applied as written for any 2-bit code.

    ``biases=None`` is the scale-only reading of the same container: the bias of
    every group is the pack's -s, so the weight is the ternary value times its
    scale, W[n, k] = s[n, k//128] * t[n, k] with t = q - 1 (the bias carries no
    information of its own in that section).
    """
    t = unpack_w2(words, K).astype(np.float64)
    s = np.asarray(scales, dtype=np.float64)
    G = K // GROUP
    if K % GROUP or s.shape != (t.shape[0], G):
        raise ValueError("scales/biases must be [N, K/128]")
    s_full = np.repeat(s, GROUP, axis=1)
    if biases is None:
        return s_full * t
    b = np.asarray(biases, dtype=np.float64)
    if b.shape != s.shape:
        raise ValueError("scales/biases must be [N, K/128]")
    b_full = np.repeat(b, GROUP, axis=1)
    return s_full * (t + 1.0) + b_full


# ----------------------------------------------------------------------------
# Packed.__call__
# ----------------------------------------------------------------------------
def packed_linear(x, signs, block: int, words, scales, biases) -> np.ndarray:
    """Non-embedding path: y = fwht(x, block, signs) @ W^T, float64.

    [ARCH] "Hadamard 旋转" (a folded module rotates its input first, then
    multiplies by the transposed 2-bit, group-128 affine matrix) and
    [PACK] "文本模型加载" (non-embedding path).  x: [M, K]; words [N, K/16];
    scales, biases [N, K/128] (biases None: scale-only, b = -s); returns [M, N].
    """
    x = np.asarray(x, dtype=np.float64)
    K = x.shape[-1]
    xr = fwht(x, block, signs, inverse=False)
    W = decode_w2(words, scales, biases, K)
    return xr @ W.T


def rotated_input(x, signs, block: int) -> np.ndarray:
    """x' = fwht(x) in float64: the operand the matmul sees."""
    return fwht(np.asarray(x, dtype=np.float64), block, signs, inverse=False)


def abs_product_sum(x, signs, block: int, words, scales, biases) -> np.ndarray:
    """sum_k |x'_k * W[n, k]| for every output (the scale of the tolerance)."""
    xr = np.abs(rotated_input(x, signs, block))
    W = np.abs(decode_w2(words, scales, biases, np.asarray(x).shape[-1]))
    return xr @ W.T


def embed_lookup(ids, words, scales, biases, signs, block: int) -> np.ndarray:
    """Embedding path: dequantise the looked-up rows, then the inverse fwht.

    [ARCH] "Hadamard 旋转" (the embedding path ends with the inverse
    transform of the dequantised rows) and [PACK] "文本模型加载" (``mx.dequantize`` of the looked-up rows, then
    the inverse Hadamard transform).  ids: [T]; returns [T, D] float64.
    Raises on an id outside [0, V).
    """
    ids = np.asarray(ids, dtype=np.int64)
    words = np.asarray(words)
    V = words.shape[0]
    if ids.size and (ids.min() < 0 or ids.max() >= V):
        raise IndexError("token id out of range")
    D = words.shape[1] * CODES_PER_WORD
    b = None if biases is None else np.asarray(biases)[ids]
    rows = decode_w2(words[ids], np.asarray(scales)[ids], b, D)
    return fwht(rows, block, signs, inverse=True)
