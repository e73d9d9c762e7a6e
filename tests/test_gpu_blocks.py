"""GPU parity at the Hadamard block sizes the pack's loader accepts besides 1024.

[PACK] "仿射 2-bit 格式与 Prism contract v1": the contract's block_size is 1024, and the loader
also takes 512, 2048 and 4096.  tb_fwht transforms any of them; tb_packed_linear(_multi) and
tb_embed_lookup run the transform as its own launch for these sizes (x' through the workspace,
or the decoded rows in place), then the unrotated kernels.  Every result against the oracle:
transforms within 1e-3 relative (floor 1e-6 of the block's norm), linear outputs within
2e-3 * sum_k |x'_k w_k| + 1e-5.  Group counts that leave the transform's last pass partly
empty (several blocks per CTA pass at 512 and 2048) are included.
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


@pytest.mark.parametrize("block", [512, 2048, 4096])
@pytest.mark.parametrize("M,nb", [(1, 1), (3, 3), (7, 2)])
@pytest.mark.parametrize("inverse", [False, True])
def test_fwht_other_blocks(tb, block, M, nb, inverse):
    K = nb * block
    x = ti.activations(600 + M, M, K)
    sg = ti.rademacher_signs(600 + block, K)
    y = torch.full((M, K), float("nan"), dtype=torch.float16, device="cuda")
    tb.tb_fwht(dev(x), y, dev(sg), block, inverse)
    ref = oracle.fwht(x.astype(np.float64), block, sg, inverse=inverse)
    assert_transform_close(y.cpu().numpy(), ref, block=block, what=f"fwht {block} M={M} inv={inverse}")
    # in place, without signs
    xd = dev(x)
    tb.tb_fwht(xd, xd, None, block, inverse)
    ref0 = oracle.fwht(x.astype(np.float64), block, None, inverse=inverse)
    assert_transform_close(xd.cpu().numpy(), ref0, block=block, what=f"fwht {block} in place")


@pytest.mark.parametrize("block,M,K,N,algo", [
    (512, 1, 1536, 77, 1),      # K not a multiple of 1024: the plain GEMV
    (512, 3, 5120, 300, 1),
    (2048, 1, 6144, 1000, 1),
    (4096, 2, 8192, 257, 1),
    (512, 200, 1536, 300, 2),
    (2048, 130, 4096, 520, 2),
    (4096, 64, 8192, 256, 2),
])
@pytest.mark.parametrize("scale_only", [False, True])
def test_linear_other_blocks(tb, block, M, K, N, algo, scale_only):
    x = ti.activations(610 + M, M, K)
    sg = ti.rademacher_signs(610 + block, K)
    L = HostLayer(611 + N, N, K)
    w, s, b = device_layer(0, N, K, from_host=L)
    nws = tb.tb_packed_linear_workspace_size(M, K, N, block, algo)
    assert nws >= M * K * 2
    ws = torch.zeros(nws, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    tb.tb_packed_linear(dev(x), dev(sg), block, w, s, None if scale_only else b, y, ws, st, algo=algo)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert int(ws[:1024].count_nonzero().item()) == 0
    ref, bound = linear_reference(x, sg, block, L, scale_only=scale_only)
    assert_linear_close(y.cpu().numpy(), ref, bound, f"block {block} {M}x{K}x{N} algo={algo}")


@pytest.mark.parametrize("M", [1, 16, 64])  # the decode GEMV, the batched GEMV, the tensor-memory one
def test_multi_other_block(tb, M):
    K, Ns, block = 4096, (300, 1000), 2048
    x = ti.activations(620 + M, M, K)
    sg = ti.rademacher_signs(620, K)
    layers = [HostLayer(621 + i, N, K) for i, N in enumerate(Ns)]
    mats = [device_layer(0, N, K, from_host=L) for N, L in zip(Ns, layers)]
    ys = [torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda") for N in Ns]
    ws = torch.zeros(tb.tb_packed_linear_workspace_size(M, K, max(Ns), block), dtype=torch.uint8,
                     device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tb_packed_linear_multi(dev(x), dev(sg), block, mats, ys, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for y, L in zip(ys, layers):
        ref, bound = linear_reference(x, sg, block, L)
        assert_linear_close(y.cpu().numpy(), ref, bound, f"multi block {block} M={M} N={L.N}")


@pytest.mark.parametrize("block", [512, 2048, 4096])
def test_embedding_other_blocks(tb, block):
    V, D = 300, 8192
    L = HostLayer(630, V, D)
    w, s, b = device_layer(0, V, D, from_host=L)
    sg = ti.rademacher_signs(630 + block, D)
    ids = np.concatenate([ti.token_ids(631, 20, V), np.array([V + 3], np.int32)])  # one bad id
    out = torch.full((len(ids), D), float("nan"), dtype=torch.float16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tb_embed_lookup(dev(ids), w, s, b, dev(sg), block, out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == tb.TB_DEV_BAD_ID
    o = out.cpu().numpy()
    assert (o[-1] == 0).all()
    ref = oracle.embed_lookup(ids[:-1], L.words, L.scales, L.biases, sg, block)
    assert_transform_close(o[:-1], ref, block=block, what=f"embedding block {block}")
