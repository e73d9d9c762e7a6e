"""GPU parity of the batched-decode GEMV (9..64 tokens per pass on tcgen05: the decoded weights the
MMA's 128-row side, the tokens its N side) against the float64 oracle:
  |y_gpu - y_ref| <= 2e-3 * sum_k |x'_k w_k| + 1e-5   per element
Token counts on both sides of every pass width (16, 32, 48, 64) and above 64 (passes), ragged row
tiles, split (stream-K) tiles and their reduction, scale-only and general affine packs, the multi
entry point, and the guard words around y and the workspace.
"""
import numpy as np
import pytest

import oracle
import tb_inputs as ti
from helpers import HostLayer, assert_linear_close, device_layer, linear_reference

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

WIDE = 5


@pytest.fixture(scope="module")
def tb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import ternary_hadamard_rotated_gb300 as tbm

    tbm.load()
    return tbm


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run(tb, x, sg, mats, N, algo=WIDE, repeat=1, block=1024):
    M, K = x.shape
    ws = torch.zeros(tb.tb_packed_linear_workspace_size(M, K, N, block, algo), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    w, s, b = mats
    outs = []
    for _ in range(repeat):
        y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        tb.tb_packed_linear(dev(x), None if sg is None else dev(sg), block, w, s, b, y, ws, st, algo=algo)
        outs.append(y)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert int(ws[:1024].count_nonzero().item()) == 0  # the shared tiles' counters are left zero
    return [o.cpu().numpy() for o in outs]


@pytest.mark.parametrize("M", [9, 15, 16, 17, 31, 32, 33, 40, 48, 49, 63, 64, 65, 100])
def test_wide_token_counts_ragged(tb, M):
    K, N = 2048, 300  # three row tiles, the last ragged; units split between CTAs
    x = ti.activations(900 + M, M, K)
    sg = ti.rademacher_signs(900, K)
    L = HostLayer(901, N, K)
    mats = device_layer(901, N, K, from_host=L)
    y1, y2 = run(tb, x, sg, mats, N, repeat=2)
    ref, bound = linear_reference(x, sg, 1024, L)
    mx, rms = assert_linear_close(y1, ref, bound, f"wide M={M}")
    assert rms < 2e-3, rms
    # the parts of a split tile are added in CTA order: the same bits every call
    np.testing.assert_array_equal(y1.view(np.uint16), y2.view(np.uint16))


@pytest.mark.parametrize("M", [16, 32, 64])
@pytest.mark.parametrize("K,N", [(5120, 17408), (17408, 5120), (5120, 1024)])
def test_wide_layer_shapes_sampled(tb, M, K, N):
    seed = ti.config_seed(5, M + K % 13)
    x = ti.activations(seed, M, K)
    sg = ti.rademacher_signs(seed, K)
    mats = device_layer(seed, N, K)
    (y,) = run(tb, x, sg, mats, N, algo=0)  # the automatic choice at these token counts
    rng = np.random.default_rng(seed)
    cols = np.sort(rng.choice(N, size=min(N, 200), replace=False))
    codes = np.concatenate([ti.ternary_codes(seed, c, c + 1, K) for c in cols])
    scales = np.concatenate([ti.group_scales(seed, c, c + 1, K // 128) for c in cols])
    words = oracle.pack_w2(codes)
    biases = oracle.biases_for(scales)
    xf = x.astype(np.float64)
    ref = oracle.packed_linear(xf, sg, 1024, words, scales, biases)
    bound = 2e-3 * oracle.abs_product_sum(xf, sg, 1024, words, scales, biases) + 1e-5
    mx, rms = assert_linear_close(y[:, cols], ref, bound, f"wide {M}x{K}->{N}")
    assert rms < 2e-3, rms


@pytest.mark.parametrize("M", [12, 64])
def test_wide_scale_only_block0_and_affine(tb, M):
    K, N = 3072, 200
    x = ti.activations(910 + M, M, K)
    sg = ti.rademacher_signs(910, K)
    L = HostLayer(911, N, K)
    w, s, b = device_layer(911, N, K, from_host=L)
    (y0,) = run(tb, x, sg, (w, s, None), N)
    ref0, bound0 = linear_reference(x, sg, 1024, L, scale_only=True)
    assert_linear_close(y0, ref0, bound0, "wide scale-only")
    (y1,) = run(tb, x, None, (w, s, b), N, block=0)
    ref1, bound1 = linear_reference(x, None, 0, L)
    assert_linear_close(y1, ref1, bound1, "wide block 0")
    words = ti.raw_words(912, N, K)
    sc = ti.group_scales(912, 0, N, K // 128)
    bi = ti.free_biases(912, N, K // 128)
    (y2,) = run(tb, x, sg, (dev(words.view(np.int32)), dev(sc), dev(bi)), N)
    xf = x.astype(np.float64)
    ref2 = oracle.packed_linear(xf, sg, 1024, words, sc, bi)
    bound2 = 2e-3 * oracle.abs_product_sum(xf, sg, 1024, words, sc, bi) + 1e-5
    assert_linear_close(y2, ref2, bound2, "wide general affine")


def test_wide_multi(tb):
    M, K, Ns = 24, 5120, (6144, 1024, 1024)
    x = ti.activations(920, M, K)
    sg = ti.rademacher_signs(920, K)
    layers = [HostLayer(921 + i, n, K) for i, n in enumerate(Ns)]
    mats = [device_layer(921 + i, n, K, from_host=L) for i, (n, L) in enumerate(zip(Ns, layers))]
    ys = [torch.full((M, n), float("nan"), dtype=torch.float16, device="cuda") for n in Ns]
    ws = torch.zeros(tb.tb_packed_linear_workspace_size(M, K, max(Ns), 1024), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tb_packed_linear_multi(dev(x), dev(sg), 1024, mats, ys, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for y, L in zip(ys, layers):
        ref, bound = linear_reference(x, sg, 1024, L)
        assert_linear_close(y.cpu().numpy(), ref, bound, f"wide multi N={L.N}")


def test_wide_guards_and_refusal(tb):
    M, K, N = 40, 2048, 77
    x = dev(ti.activations(930, M, K))
    w, s, b = device_layer(931, N, K, from_host=HostLayer(931, N, K))
    G = 4096
    y_raw = torch.full((2 * G + M * N * 2,), 0xA5, dtype=torch.uint8, device="cuda")
    y = y_raw[G:G + M * N * 2].view(torch.float16).view(M, N)
    nws = tb.tb_packed_linear_workspace_size(M, K, N, 1024, WIDE)
    ws_raw = torch.full((2 * G + nws,), 0xA5, dtype=torch.uint8, device="cuda")
    ws = ws_raw[G:G + nws]
    ws.zero_()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tb_packed_linear(x, dev(ti.rademacher_signs(930, K)), 1024, w, s, b, y, ws, st, algo=WIDE)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for raw, n in ((y_raw, M * N * 2), (ws_raw, nws)):
        assert bool((raw[:G] == 0xA5).all()) and bool((raw[G + n:] == 0xA5).all())
    # K not a multiple of 1024: the batched-decode GEMV refuses (block 0, K = 384)
    x2 = torch.zeros((M, 384), dtype=torch.float16, device="cuda")
    w2 = torch.zeros((N, 384 // 16), dtype=torch.int32, device="cuda")
    s2 = torch.zeros((N, 3), dtype=torch.float16, device="cuda")
    ws2 = torch.zeros(tb.tb_packed_linear_workspace_size(M, 384, N, 0, WIDE), dtype=torch.uint8, device="cuda")
    with pytest.raises(tb.TBError) as e:
        tb.tb_packed_linear(x2, None, 0, w2, s2, None, torch.empty((M, N), dtype=torch.float16, device="cuda"),
                            ws2, st, algo=WIDE)
    assert e.value.status == tb.TB_ERR_UNSUPPORTED
