"""The decode GEMV entry point that allocates nothing, against the regular one.

tb_packed_linear_gemv_noalloc serves callers that cannot allocate device memory (code
under CUDA graph capture, plugins inside a runtime that owns all device memory, services
with a fixed memory budget).  Its split-schedule state lives in a fixed array inside the
library; this test calls it twice in a row through the C ABI and checks both results
against tb_packed_linear's on the same inputs and against the float64 oracle, each within
the linear-path tolerance.  The file is named to run last, so a failure here leaves every
other result in place.
"""
import numpy as np
import pytest

import oracle
import tb_inputs as ti
from helpers import LIN_ABS, LIN_REL, HostLayer, device_layer

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import ternary_hadamard_rotated_gb300 as tbm

    tbm.load()
    return tbm


class _AffineLayer:
    """Random words (every 2-bit field 0..3) and biases drawn apart from the scales."""

    def __init__(self, seed, N, K):
        self.words = ti.raw_words(seed, N, K)
        self.scales = ti.group_scales(seed, 0, N, K // 128)
        self.biases = ti.free_biases(seed, N, K // 128)


@pytest.mark.parametrize("M,K,N,affine", [(1, 17408, 5120, False), (3, 5120, 1000, False),
                                          (1, 2048, 77, False), (2, 5120, 300, True)])
def test_noalloc_gemv_matches_regular_entry(tb, M, K, N, affine):
    x = ti.activations(90 + M, M, K)
    sg = ti.rademacher_signs(90, K)
    if affine:
        L = _AffineLayer(91, N, K)
        w = torch.from_numpy(L.words.view(np.int32)).cuda()
        s = torch.from_numpy(L.scales).cuda()
        b = torch.from_numpy(L.biases).cuda()
    else:
        L = HostLayer(90, N, K)
        w, s, b = device_layer(90, N, K, from_host=L)
    xd = torch.from_numpy(x).cuda()
    sd = torch.from_numpy(sg).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(tb.tb_packed_linear_workspace_size(M, K, N, 1024, tb.TB_ALGO_GEMV),
                     dtype=torch.uint8, device="cuda")
    y_reg = torch.empty((M, N), dtype=torch.float16, device="cuda")
    tb.tb_packed_linear(xd, sd, 1024, w, s, b, y_reg, ws, st, algo=tb.TB_ALGO_GEMV)
    outs = []
    for _ in range(2):  # two calls in a row share the one static array
        y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        tb.tb_packed_linear_gemv_noalloc(xd, sd, 1024, w, s, b, y, st)
        outs.append(y)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    xf = x.astype(np.float64)
    bound = LIN_REL * oracle.abs_product_sum(xf, sg, 1024, L.words, L.scales, L.biases) + LIN_ABS
    y_or = oracle.packed_linear(xf, sg, 1024, L.words, L.scales, L.biases)
    y_rg = y_reg.cpu().numpy().astype(np.float64)
    assert (np.abs(y_rg - y_or) <= bound).all()
    for y in outs:
        yn = y.cpu().numpy().astype(np.float64)
        for ref, what in ((y_rg, "regular entry"), (y_or, "oracle")):
            err = np.abs(yn - ref)
            assert (err <= bound).all(), (what, float(err.max()))


def test_noalloc_gemv_scale_only(tb):
    # biases = NULL: each bias is the pack's -scale; the result is the stored-bias one up to
    # the order in which shared-memory sums of cut tiles meet
    M, K, N = 2, 5120, 1000
    x = ti.activations(95, M, K)
    sg = ti.rademacher_signs(95, K)
    L = HostLayer(95, N, K)
    w, s, b = device_layer(95, N, K, from_host=L)
    xd = torch.from_numpy(x).cuda()
    sd = torch.from_numpy(sg).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for bb in (b, None):
        y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        tb.tb_packed_linear_gemv_noalloc(xd, sd, 1024, w, s, bb, y, st)
        outs.append(y.cpu().numpy())
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ulp = np.spacing(np.abs(outs[0]).astype(np.float16)).astype(np.float64)  # sum order of cut tiles
    assert (np.abs(outs[1].astype(np.float64) - outs[0].astype(np.float64)) <= 2 * ulp).all()
    ref = oracle.packed_linear(x.astype(np.float64), sg, 1024, L.words, L.scales, None)
    bound = LIN_REL * oracle.abs_product_sum(x.astype(np.float64), sg, 1024, L.words, L.scales,
                                             None) + LIN_ABS
    assert (np.abs(outs[1].astype(np.float64) - ref) <= bound).all()


def test_noalloc_gemv_refuses_too_many_tokens(tb):
    K, N, M = 1024, 16, 9
    x = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    w = torch.zeros((N, K // 16), dtype=torch.int32, device="cuda")
    s = torch.zeros((N, K // 128), dtype=torch.float16, device="cuda")
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    with pytest.raises(tb.TBError) as ei:
        tb.tb_packed_linear_gemv_noalloc(x, None, 1024, w, s, s, y)
    assert ei.value.status == tb.TB_ERR_TOO_LARGE
