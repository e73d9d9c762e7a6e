"""Seeded synthetic inputs for the folded-Hadamard ternary ``Packed`` layer.

This module is shared by the CPU oracle (``oracle/``), the tests and the bench.
It holds *no* arithmetic of the method itself (no transform, no packing, no
dequantisation): it only draws the random tensors the method consumes.

Two families of generators:

* small tensors (activations ``x``, sign vectors, token ids) come from NumPy's
  ``Generator(PCG64(seed))`` on the host;
* ternary codes and group scales come from a counter-based generator,
  SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014; mixing constants as in Vigna's reference
  ``splitmix64.c``), so that any row of a multi-GB weight matrix can be
  regenerated on its own.  ``tb_inputs/csrc/synth.cu`` implements the same
  definition on the device for the large decode-sweep workload, and
  ``device.py`` loads it.  Both sides use only integer operations and
  correctly rounded fp32 operations (no fused multiply-add), so they agree bit
  for bit.

Distributions (the workload the Bonsai-2 27B pages describe, restated):
  * x ~ N(0, 1) rounded to fp16;
  * ternary codes t in {-1, 0, +1} with p = (0.38, 0.24, 0.38);
  * scales s ~ U[0.005, 0.02] rounded to fp16 (one per 128 weights);
  * sign vectors: Rademacher +-1, one vector per width;
  * token ids uniform over the vocabulary.
"""
from __future__ import annotations

import numpy as np

MASK64 = np.uint64(0xFFFFFFFFFFFFFFFF)
GAMMA = np.uint64(0x9E3779B97F4A7C15)
MIX1 = np.uint64(0xBF58476D1CE4E5B9)
MIX2 = np.uint64(0x94D049BB133111EB)

# p(-1) = 0.38, p(0) = 0.24, p(+1) = 0.38 on a 24-bit uniform u:
#   t = -1 if u < T_NEG;  t = 0 if u < T_ZERO;  else t = +1
U24 = 1 << 24
T_NEG = 6375342        # floor(0.38 * 2**24)
T_ZERO = 10401874      # floor(0.62 * 2**24) + 1  -> 0.24 of the mass in [T_NEG, T_ZERO)

SCALE_LO = np.float32(0.005)
SCALE_SPAN = np.float32(0.015)

# stream ids so that codes and scales of one tensor never share counters
STREAM_CODES = 0
STREAM_SCALES = 1


def _mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function (the three xor-shift-multiply rounds)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * MIX1
        z = (z ^ (z >> np.uint64(27))) * MIX2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int) -> np.uint64:
    """Per-(seed, stream) starting state: the SplitMix64 output of the pair."""
    base = np.uint64((int(seed) * 2 + int(stream)) & 0xFFFFFFFFFFFFFFFF)
    with np.errstate(over="ignore"):
        return _mix64(np.array([base * GAMMA + GAMMA], dtype=np.uint64))[0]


def counter_hash(seed: int, stream: int, idx: np.ndarray) -> np.ndarray:
    """SplitMix64 value number ``idx`` of the sequence started at ``stream_key``.

    state_i = key + (idx + 1) * GAMMA  (mod 2**64);  value = mix64(state_i)
    """
    key = stream_key(seed, stream)
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = key + (idx + np.uint64(1)) * GAMMA
    return _mix64(z)


def ternary_codes(seed: int, n0: int, n1: int, K: int) -> np.ndarray:
    """Codes t in {-1,0,1} (int8) for rows [n0, n1) of an [N, K] matrix.

    Element (n, k) uses counter n*K + k, so a row does not depend on the rows
    around it.
    """
    rows = np.arange(n0, n1, dtype=np.uint64)[:, None]
    cols = np.arange(K, dtype=np.uint64)[None, :]
    u = counter_hash(seed, STREAM_CODES, rows * np.uint64(K) + cols) >> np.uint64(40)
    t = np.where(u < T_NEG, -1, np.where(u < T_ZERO, 0, 1)).astype(np.int8)
    return t


def group_scales(seed: int, n0: int, n1: int, G: int) -> np.ndarray:
    """fp16 scales ~ U[0.005, 0.02] for rows [n0, n1) of an [N, G] matrix.

    s = fp16( 0.005f + 0.015f * (u * 2**-24) ), every step a correctly rounded
    fp32 operation, u the top 24 bits of the counter hash of n*G + g.
    """
    rows = np.arange(n0, n1, dtype=np.uint64)[:, None]
    cols = np.arange(G, dtype=np.uint64)[None, :]
    u = counter_hash(seed, STREAM_SCALES, rows * np.uint64(G) + cols) >> np.uint64(40)
    f = u.astype(np.float32) * np.float32(1.0 / U24)
    f = SCALE_SPAN * f
    f = SCALE_LO + f
    return f.astype(np.float16)


def raw_words(seed: int, N: int, K: int) -> np.ndarray:
    """Uniformly random uint32 words [N, K/16]: every 2-bit field equally likely to hold
    0, 1, 2 or 3.  Inputs for the general affine container (a field of 3, which the
    packer never writes, included); no packing is done here, the bits are drawn as words."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.integers(0, 1 << 32, size=(N, K // 16), dtype=np.uint64).astype(np.uint32)


def free_biases(seed: int, N: int, G: int) -> np.ndarray:
    """fp16 biases ~ U[-0.03, 0.01] [N, G], drawn independently of any scale (so b != -s)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return (rng.random((N, G)) * 0.04 - 0.03).astype(np.float16)


def activations(seed: int, M: int, K: int) -> np.ndarray:
    """x ~ N(0,1) rounded to fp16, shape [M, K]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.standard_normal((M, K)).astype(np.float16)


def rademacher_signs(seed: int, K: int) -> np.ndarray:
    """Explicit +-1 sign vector (int8) of width K."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return np.where(rng.integers(0, 2, size=K) == 0, -1, 1).astype(np.int8)


def token_ids(seed: int, T: int, V: int) -> np.ndarray:
    """T token ids drawn uniformly from [0, V) (int32)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.integers(0, V, size=T).astype(np.int32)


# ----------------------------------------------------------------------------
# Workload shapes (Bonsai-2 27B text model: hidden 5120, 64 layers with a 3:1
# linear:full attention mix, MLP 17408, vocabulary 248320)
# ----------------------------------------------------------------------------
HIDDEN = 5120
MLP = 17408
VOCAB = 248320
N_LAYERS = 64
FULL_ATTN_EVERY = 4

TINY = dict(M=1, K=1024, N=256, seed=0)

# decode GEMV shapes at M = 1, (name, K, N)
LAYER_SHAPES = [
    ("gate_up", HIDDEN, MLP),
    ("down", MLP, HIDDEN),
    ("q_proj", HIDDEN, 6144),
    ("o_proj", 6144, HIDDEN),
    ("kv_proj", HIDDEN, 1024),
]


def sweep_layers():
    """The 401 packed linears of one decode step, in execution order.

    Returns a list of (name, K, N). Layers l with (l+1) % 4 == 0 are full
    attention (q, k, v, o); the others are linear attention (in_proj_qkv,
    in_proj_z, out_proj). Every layer has an MLP (gate, up, down); lm_head last.
    """
    out = []
    for l in range(N_LAYERS):
        if (l + 1) % FULL_ATTN_EVERY == 0:
            out += [("q_proj", HIDDEN, 6144), ("k_proj", HIDDEN, 1024),
                    ("v_proj", HIDDEN, 1024), ("o_proj", 6144, HIDDEN)]
        else:
            out += [("in_proj_qkv", HIDDEN, 10240), ("in_proj_z", HIDDEN, 6144),
                    ("out_proj", 6144, HIDDEN)]
        out += [("gate_proj", HIDDEN, MLP), ("up_proj", HIDDEN, MLP), ("down_proj", MLP, HIDDEN)]
    out.append(("lm_head", HIDDEN, VOCAB))
    return out


def sweep_weight_count() -> int:
    return sum(K * N for _, K, N in sweep_layers())


def packed_bytes(K: int, N: int) -> int:
    """Bytes of one W2-g128 affine matrix: 2-bit codes + fp16 scale + fp16 bias per 128."""
    return N * K // 4 + 2 * (N * (K // 128) * 2)


def config_seed(config: int, tensor: int) -> int:
    """Seed rule for the configs other than the tiny one: 1000*config + tensor."""
    return 1000 * config + tensor
