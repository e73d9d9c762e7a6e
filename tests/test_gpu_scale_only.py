"""GPU parity of the scale-only form: every entry point with biases = NULL.

The pack's bias is always -scale (the affine container of the Bonsai article), so a
caller may pass no biases; the kernels then take each bias as the scale with its fp16
sign bit flipped and read 1/64 byte less per weight.  Two checks per path:
  * the same result as the call with the pack's stored biases: the same arithmetic on the
    same values, so bit-identical where the path sums in a fixed order (tensor-core GEMM,
    the K % 1024 GEMV, the embedding) and within two fp16 units in the last place where
    the decode GEMV's shared-memory sums of a row tile cut between three warp groups may
    meet in another order;
  * within the linear (or transform) tolerance of the oracle's scale-only reading,
    W = s * t, computed without biases.
"""
import numpy as np
import pytest

import oracle
import tb_inputs as ti
from helpers import (HostLayer, assert_linear_close, assert_transform_close, device_layer,
                     linear_reference)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import ternary_hadamard_rotated_gb300 as tbm

    tbm.load()
    return tbm


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_same(y0, yb, exact):
    if exact:
        np.testing.assert_array_equal(y0.view(np.uint16), yb.view(np.uint16))
    else:
        ulp = np.spacing(np.abs(yb).astype(np.float16)).astype(np.float64)
        assert (np.abs(y0.astype(np.float64) - yb.astype(np.float64)) <= 2 * ulp).all()


def linear(tb, xd, sd, block, w, s, b, M, N, algo):
    K = xd.shape[1]
    ws = torch.zeros(tb.tb_packed_linear_workspace_size(M, K, N, block, algo), dtype=torch.uint8,
                     device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    tb.tb_packed_linear(xd, sd, block, w, s, b, y, ws, st, algo=algo)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return y.cpu().numpy()


# decode GEMV (TMA path, split schedule, ragged rows), the K % 1024 != 0 GEMV (block 0),
# the tensor-core GEMM (whole tiles, stream-K split tiles, a group count not a multiple of 8)
CASES = [
    (1, 5120, 6144, 1, 1024),
    (3, 2048, 300, 1, 1024),
    (8, 1024, 77, 1, 1024),
    (1, 1152, 40, 1, 0),
    (5, 1152, 33, 1, 0),
    (200, 2048, 300, 2, 1024),
    (300, 1024, 19500, 2, 1024),
    (100, 1152, 64, 2, 0),
]


@pytest.mark.parametrize("M,K,N,algo,block", CASES)
def test_linear_scale_only(tb, M, K, N, algo, block):
    x = ti.activations(500 + M, M, K)
    sg = ti.rademacher_signs(500, K) if block else None
    L = HostLayer(501 + N, N, K)
    w, s, b = device_layer(0, N, K, from_host=L)
    xd, sd = dev(x), (dev(sg) if sg is not None else None)
    y_b = linear(tb, xd, sd, block, w, s, b, M, N, algo)
    y_0 = linear(tb, xd, sd, block, w, s, None, M, N, algo)
    assert_same(y_0, y_b, exact=not (algo == 1 and K % 1024 == 0))
    ref, bound = linear_reference(x, sg, block, L, scale_only=True)
    assert_linear_close(y_0, ref, bound, f"scale-only {M}x{K}x{N} algo={algo}")


@pytest.mark.parametrize("M", [1, 3, 64])
def test_multi_scale_only_mixed(tb, M):
    # one matrix with its stored biases, two without: each as the same call with biases
    K, Ns = 2048, (300, 1000, 77)
    x = ti.activations(520 + M, M, K)
    sg = ti.rademacher_signs(520, K)
    layers = [HostLayer(521 + i, N, K) for i, N in enumerate(Ns)]
    mats = [device_layer(0, N, K, from_host=L) for N, L in zip(Ns, layers)]
    ws = torch.zeros(tb.tb_packed_linear_workspace_size(M, K, max(Ns), 1024), dtype=torch.uint8,
                     device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for sel in ([m for m in mats], [mats[0], (mats[1][0], mats[1][1], None), (mats[2][0], mats[2][1], None)]):
        ys = [torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda") for N in Ns]
        tb.tb_packed_linear_multi(dev(x), dev(sg), 1024, sel, ys, ws, st)
        outs.append([y.cpu().numpy() for y in ys])
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for i, L in enumerate(layers):
        assert_same(outs[1][i], outs[0][i], exact=M > 8)
        ref, bound = linear_reference(x, sg, 1024, L, scale_only=True)
        assert_linear_close(outs[1][i], ref, bound, f"multi scale-only M={M} N={L.N}")


@pytest.mark.parametrize("block", [1024, 0])
def test_embedding_scale_only(tb, block):
    V, D = 300, 2048
    L = HostLayer(530, V, D)
    w, s, b = device_layer(0, V, D, from_host=L)
    sg = ti.rademacher_signs(530, D)
    ids = ti.token_ids(531, 37, V)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for bb in (b, None):
        out = torch.full((len(ids), D), float("nan"), dtype=torch.float16, device="cuda")
        tb.tb_embed_lookup(dev(ids), w, s, bb, dev(sg) if block else None, block, out, st)
        outs.append(out)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o_b, o_0 = (o.cpu().numpy() for o in outs)
    np.testing.assert_array_equal(o_0.view(np.uint16), o_b.view(np.uint16))
    ref = oracle.embed_lookup(ids, L.words, L.scales, None, sg if block else None, block)
    if block:
        assert_transform_close(o_0, ref, what="embedding scale-only")
    else:
        np.testing.assert_array_equal(o_0.astype(np.float64), ref)  # {-s, 0, s}: exact


def test_chain_scale_only(tb):
    # every link's output against the oracle's scale-only reading of that link's input (the
    # links feed one another, so last-place differences of cut-tile sums propagate: no
    # comparison with the stored-bias run beyond that)
    from test_gpu_chain import SPEC, SmallChain

    M = 2
    c = SmallChain(tb, SPEC, M, seed=540)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    args0 = [(x, sg, blk, [(w, s, None) for w, s, _ in ms], ys) for x, sg, blk, ms, ys in c.args]
    tb.Chain(args0, M).run(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    c.check("chain scale-only", scale_only=True)
