"""Shared helpers of the GPU parity tests: seeded layers on both sides, tolerances.

The CUDA side gets its weights from ``tb_pack_w2`` (codes drawn on the host, or
on the device by ``tb_inputs.device`` for the large tables); the oracle side
packs the same codes itself with ``oracle.pack_w2``.  Nothing the oracle uses
comes from the CUDA path.
"""
from __future__ import annotations

import numpy as np

import oracle
import tb_inputs as ti

# tolerance of the linear and GEMM outputs:
#   |y_gpu - y_ref| <= 2e-3 * sum_k |x'_k w_k| + 1e-5   (per element)
LIN_REL = 2e-3
LIN_ABS = 1e-5
# tolerance of transform outputs (FWHT, embedding): 1e-3 relative, with an absolute
# floor of 1e-6 * ||block||_2 for elements near zero (relative error is undefined there)
FWHT_REL = 1e-3


class HostLayer:
    """Codes/scales drawn on the host; oracle-side packing."""

    def __init__(self, seed: int, N: int, K: int, rows=None):
        self.N, self.K, self.G = N, K, K // 128
        r0, r1 = (0, N) if rows is None else rows
        self.codes = ti.ternary_codes(seed, r0, r1, K)
        self.scales = ti.group_scales(seed, r0, r1, self.G)
        self.biases = oracle.biases_for(self.scales)
        self.words = oracle.pack_w2(self.codes)


def device_layer(seed: int, N: int, K: int, from_host: HostLayer | None = None, chunk_rows=None):
    """Packed layer on the GPU: w (int32 view of uint32) [N, K/16], scales, biases fp16.

    Codes come from the host layer when given, else from the device generator in
    row chunks (bounded temporary memory).  Packing is tb_pack_w2 on the device.
    """
    import torch

    import ternary_hadamard_rotated_gb300 as tb
    from tb_inputs import device as tdev

    dev = torch.device("cuda")
    G = K // 128
    w = torch.empty((N, K // 16), dtype=torch.int32, device=dev)
    scales = torch.empty((N, G), dtype=torch.float16, device=dev)
    biases = torch.empty((N, G), dtype=torch.float16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    if from_host is not None:
        codes = torch.from_numpy(from_host.codes).to(dev)
        scales.copy_(torch.from_numpy(from_host.scales))
        tb.tb_pack_w2(codes, scales, w, biases, status)
    else:
        step = chunk_rows or max(1, (1 << 28) // K)
        tmp = torch.empty((min(step, N), K), dtype=torch.int8, device=dev)
        for r0 in range(0, N, step):
            n = min(step, N - r0)
            tdev.fill_codes(tmp[:n], seed, r0, K)
            tdev.fill_scales(scales[r0:r0 + n], seed, r0, G)
            tb.tb_pack_w2(tmp[:n], scales[r0:r0 + n], w[r0:r0 + n], biases[r0:r0 + n], status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return w, scales, biases


def linear_reference(x16, signs, block, layer: HostLayer, scale_only=False):
    """(y_ref, bound) in float64 for the rows held by the host layer (scale_only: the
    oracle's reading without biases, W = s * t)."""
    x = x16.astype(np.float64)
    b = None if scale_only else layer.biases
    y = oracle.packed_linear(x, signs, block, layer.words, layer.scales, b)
    bound = LIN_REL * oracle.abs_product_sum(x, signs, block, layer.words, layer.scales, b) + LIN_ABS
    return y, bound


def assert_linear_close(y_gpu, y_ref, bound, what=""):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first {idx.tolist()} "
                             f"gpu={y_gpu[tuple(idx[0])]} ref={y_ref[tuple(idx[0])]} "
                             f"bound={bound[tuple(idx[0])]}")
    rms = np.sqrt(np.mean(y_ref ** 2)) or 1.0
    return float(err.max() / rms), float(np.sqrt(np.mean(err ** 2)) / rms)


def assert_transform_close(out_gpu, ref, block=1024, what=""):
    out_gpu = np.asarray(out_gpu, dtype=np.float64)
    lead = ref.shape[:-1]
    K = ref.shape[-1]
    nb = max(1, K // block)
    norms = np.linalg.norm(ref.reshape(lead + (nb, -1)), axis=-1)
    floor = np.repeat(norms, K // nb, axis=-1).reshape(ref.shape) * 1e-6
    err = np.abs(out_gpu - ref)
    bad = ~(err <= FWHT_REL * np.abs(ref) + floor)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first {idx.tolist()}")


def compare_chain_runs(first, second, spec, ulps=8):
    """Two runs of one chain on the same inputs: a link whose input is bit-identical in both runs
    gives outputs within `ulps` fp16 ulps (+1e-6).  The only run-to-run freedom inside a link is
    the order of the shared-memory fp32 sums of tiles cut between unit groups.  A link whose input
    already differs is not compared: a last-place difference in its input moves every output by
    an amount set by the input's scale, not by that output's own ulp.  Each run is held to the
    oracle on its own inputs elsewhere.  `first` and `second` map buffer names to fp16 arrays;
    `spec` is [(input name, [(output name, K, N), ...]), ...].  Returns the links compared."""
    compared = []
    for src, mats in spec:
        if not np.array_equal(np.asarray(first[src]).view(np.uint16), np.asarray(second[src]).view(np.uint16)):
            continue
        for name, _, _ in mats:
            a = np.asarray(first[name]).astype(np.float64)
            b = np.asarray(second[name]).astype(np.float64)
            ulp = np.spacing(np.abs(a).astype(np.float16)).astype(np.float64)
            bad = ~(np.abs(a - b) <= ulps * ulp + 1e-6)
            if bad.any():
                raise AssertionError(f"{name}: {int(bad.sum())} outputs differ by more than {ulps} ulp "
                                     f"between two runs on the same input {src}")
        compared.append(src)
    return compared
