"""Plain CPU oracle of the GGUF block formats of the same ternary weights, and of their
lossless transcoding into the W2-g128 container.

TEST INFRASTRUCTURE ONLY (see the package docstring): never used by the library.

Source: [ARCH] "3.9GB 里藏了什么" (kwkr.cn/news/564617), section "打包格式的工程MLX 2.25 bits
与 GGUF 的两种装箱": two GGUF packings of the same trits per 128 weights, PQ2_0 (34 bytes: each
trit in a 2-bit slot, cheap to decode) and PTQ1_0 (28 bytes: dense trits, extra arithmetic to
decode); the transcoder takes the scale from the block header, sets the bias to its negation,
and rearranges the codes into uint32 words, losslessly.

The pages give the block sizes but not the byte layout inside a block.  Readings (each the
plainest one the sizes allow):
  * both blocks start with the group's fp16 scale d (2 bytes, little-endian);
  * PQ2_0: the 32 remaining bytes hold the 128 slots, slot i in byte i // 4 at bits
    2 (i % 4) .. + 1 (least significant first), slot value q = t + 1 in {0, 1, 2} (the same
    mapping as the W2 container);
  * PTQ1_0: the 26 remaining bytes hold the trits five per byte (3^5 = 243 <= 256; 26 bytes
    are the fewest that hold 128 trits), byte j holds trits 5j .. 5j + 4 (those below 128) as
    the base-3 number sum_i (t_{5j+i} + 1) 3^i, the first trit the least significant digit;
  * the blocks of a row follow each other along K, rows one after another.
"""
from __future__ import annotations

import numpy as np

from .w2_hadamard import GROUP, biases_for, pack_w2

PQ2_0_BYTES = 34
PTQ1_0_BYTES = 28
TRITS_PER_BYTE = 5
PTQ1_0_TRIT_BYTES = 26


def _scale_bytes(d) -> np.ndarray:
    """fp16 scales [N, G] -> their little-endian bytes [N, G, 2]."""
    return np.ascontiguousarray(np.asarray(d, dtype=np.float16)).view(np.uint8).reshape(d.shape + (2,))


def _check_codes(t, K):
    t = np.asarray(t)
    if t.ndim != 2 or t.shape[1] != K or K % GROUP:
        raise ValueError("codes must be [N, K] with K a multiple of 128")
    if not np.isin(t, (-1, 0, 1)).all():
        raise ValueError("ternary codes must be -1, 0 or 1")
    return t.astype(np.int64)


def pq2_0_encode(t, d) -> np.ndarray:
    """Trits t [N, K] and fp16 scales d [N, K/128] -> PQ2_0 blocks, uint8 [N, K/128, 34]."""
    t = np.asarray(t)
    N, K = t.shape
    t = _check_codes(t, K)
    G = K // GROUP
    q = (t + 1).reshape(N, G, GROUP)
    out = np.zeros((N, G, PQ2_0_BYTES), dtype=np.uint8)
    out[:, :, 0:2] = _scale_bytes(np.asarray(d, dtype=np.float16).reshape(N, G))
    for i in range(GROUP):
        out[:, :, 2 + i // 4] |= (q[:, :, i] << (2 * (i % 4))).astype(np.uint8)
    return out


def pq2_0_decode(blocks, K: int):
    """PQ2_0 blocks uint8 [N, K/128, 34] -> (trits int8 [N, K], fp16 scales [N, K/128]).
    Raises on a slot value of 3 (not a trit)."""
    b = np.asarray(blocks, dtype=np.uint8)
    N, G = b.shape[0], K // GROUP
    if b.shape != (N, G, PQ2_0_BYTES):
        raise ValueError("PQ2_0 blocks must be [N, K/128, 34]")
    d = np.ascontiguousarray(b[:, :, 0:2]).view(np.float16).reshape(N, G)
    t = np.zeros((N, G, GROUP), dtype=np.int64)
    for i in range(GROUP):
        q = (b[:, :, 2 + i // 4].astype(np.int64) >> (2 * (i % 4))) & 3
        if (q == 3).any():
            raise ValueError("PQ2_0 slot value 3 is not a trit")
        t[:, :, i] = q - 1
    return t.reshape(N, K).astype(np.int8), d


def ptq1_0_encode(t, d) -> np.ndarray:
    """Trits t [N, K] and fp16 scales d [N, K/128] -> PTQ1_0 blocks, uint8 [N, K/128, 28]."""
    t = np.asarray(t)
    N, K = t.shape
    t = _check_codes(t, K)
    G = K // GROUP
    q = (t + 1).reshape(N, G, GROUP)
    out = np.zeros((N, G, PTQ1_0_BYTES), dtype=np.uint8)
    out[:, :, 0:2] = _scale_bytes(np.asarray(d, dtype=np.float16).reshape(N, G))
    for j in range(PTQ1_0_TRIT_BYTES):
        v = np.zeros((N, G), dtype=np.int64)
        for i in reversed(range(TRITS_PER_BYTE)):  # Horner: the first trit ends least significant
            k = TRITS_PER_BYTE * j + i
            v = 3 * v + (q[:, :, k] if k < GROUP else 0)
        out[:, :, 2 + j] = v.astype(np.uint8)
    return out


def ptq1_0_decode(blocks, K: int):
    """PTQ1_0 blocks uint8 [N, K/128, 28] -> (trits int8 [N, K], fp16 scales [N, K/128]).
    Raises on a byte that is not five base-3 digits (>= 243), or whose digits past trit 127 are
    not zero."""
    b = np.asarray(blocks, dtype=np.uint8)
    N, G = b.shape[0], K // GROUP
    if b.shape != (N, G, PTQ1_0_BYTES):
        raise ValueError("PTQ1_0 blocks must be [N, K/128, 28]")
    d = np.ascontiguousarray(b[:, :, 0:2]).view(np.float16).reshape(N, G)
    t = np.zeros((N, G, GROUP), dtype=np.int64)
    for j in range(PTQ1_0_TRIT_BYTES):
        v = b[:, :, 2 + j].astype(np.int64)
        if (v >= 3 ** TRITS_PER_BYTE).any():
            raise ValueError("PTQ1_0 byte above 242")
        for i in range(TRITS_PER_BYTE):
            k = TRITS_PER_BYTE * j + i
            digit = v % 3
            v = v // 3
            if k < GROUP:
                t[:, :, k] = digit - 1
            elif (digit != 0).any():
                raise ValueError("PTQ1_0 digit past trit 127 is not zero")
    return t.reshape(N, K).astype(np.int8), d


def transcode_to_w2(blocks, fmt: str, K: int):
    """GGUF blocks -> the W2-g128 container (words uint32 [N, K/16], scales, biases = -scales),
    losslessly: the decoded trits packed by pack_w2, the block scales as the group scales."""
    if fmt == "PQ2_0":
        t, d = pq2_0_decode(blocks, K)
    elif fmt == "PTQ1_0":
        t, d = ptq1_0_decode(blocks, K)
    else:
        raise ValueError("format must be PQ2_0 or PTQ1_0")
    return pack_w2(t), d, biases_for(d)
