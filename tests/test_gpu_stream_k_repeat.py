"""Tensor-core GEMM schedules whose CTAs walk several segments (stream-K), called repeatedly on
one workspace and compared with the float64 oracle on every element:
  |y_gpu - y_ref| <= 2e-3 * sum_k |x'_k w_k| + 1e-5

These are the schedules in which the decoders' word slots, the split-tile parts and their
counters are reused most: a slot refilled before its readers are done, a part read before it
is written or a counter not returned to zero shows up as a band of wrong rows in one tile, on
some calls only, so every call is checked in full.
  - single CTAs: 100 tokens (one 128-token subtile), 1024 -> 40000: 157 tiles of 256 rows,
    more than one per SM, cut into one equal range of k-blocks per SM;
  - CTA pairs: 2048 tokens (256-token tiles), 1024 -> 4864: 80 tiles of two row tiles each,
    shared by the resident pairs the same way.
"""
import numpy as np
import pytest

import tb_inputs as ti
from helpers import HostLayer, assert_linear_close, device_layer, linear_reference

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TC = 2


@pytest.fixture(scope="module")
def tb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import ternary_hadamard_rotated_gb300 as tbm

    tbm.load()
    return tbm


@pytest.mark.parametrize("M,K,N", [(100, 1024, 40000), (2048, 1024, 4864)])
def test_stream_k_repeated_calls_every_element(tb, M, K, N):
    seed = 960 + M % 7
    x = ti.activations(seed, M, K)
    sg = ti.rademacher_signs(seed, K)
    L = HostLayer(seed + 1, N, K)
    w, s, b = device_layer(seed + 1, N, K, from_host=L)
    ref, bound = linear_reference(x, sg, 1024, L)
    xd = torch.from_numpy(x).cuda()
    sd = torch.from_numpy(sg).cuda()
    ws = torch.zeros(tb.tb_packed_linear_workspace_size(M, K, N, 1024, TC), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(4):
        y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        tb.tb_packed_linear(xd, sd, 1024, w, s, b, y, ws, st, algo=TC)
        outs.append(y)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    first = outs[0].cpu().numpy()
    for i, y in enumerate(outs):
        yh = y.cpu().numpy()
        assert_linear_close(yh, ref, bound, f"call {i} M={M} {K}->{N}")
        # the parts of a split tile are added in CTA order: the same bits every call
        np.testing.assert_array_equal(yh.view(np.uint16), first.view(np.uint16))
