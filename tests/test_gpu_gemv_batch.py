"""GPU parity of the batched-decode GEMV on mma.sync (TB_ALGO_GEMV_BATCH: x' rotated once into the
workspace as the operand image, each unit of packed codes decoded once for all tokens of a pass of
8, 16, 32 or 64) against the float64 oracle:
  |y_gpu - y_ref| <= 2e-3 * sum_k |x'_k w_k| + 1e-5   per element
Token counts on both sides of every pass width and above 64 (passes), ragged row tiles, split
(stream-K) tiles with two and with many contributors, repeated calls (the same bits: parts are added
in CTA order), scale-only, block 0, a block that is not fused, general affine packs (b != -s, fields
of 3), the layer shapes of the 27B model on sampled rows, guard words and the refusal of K not a
multiple of 1024.
"""
import numpy as np
import pytest

import oracle
import tb_inputs as ti
from helpers import HostLayer, assert_linear_close, device_layer, linear_reference

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

BATCH = 6


@pytest.fixture(scope="module")
def tb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import ternary_hadamard_rotated_gb300 as tbm

    tbm.load()
    return tbm


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run(tb, x, sg, mats, N, repeat=1, block=1024):
    M, K = x.shape
    ws = torch.zeros(tb.tb_packed_linear_workspace_size(M, K, N, block, BATCH), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    w, s, b = mats
    outs = []
    for _ in range(repeat):
        y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        tb.tb_packed_linear(dev(x), None if sg is None else dev(sg), block, w, s, b, y, ws, st, algo=BATCH)
        outs.append(y)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return [o.cpu().numpy() for o in outs]


@pytest.mark.parametrize("M", [1, 2, 3, 7, 8, 9, 15, 16, 17, 31, 32, 33, 48, 63, 64, 65, 130])
def test_batch_token_counts_ragged(tb, M):
    K, N = 2048, 300  # three row tiles, the last ragged; units split between CTAs
    x = ti.activations(1400 + M, M, K)
    sg = ti.rademacher_signs(1400, K)
    L = HostLayer(1401, N, K)
    mats = device_layer(1401, N, K, from_host=L)
    y1, y2, y3 = run(tb, x, sg, mats, N, repeat=3)
    ref, bound = linear_reference(x, sg, 1024, L)
    mx, rms = assert_linear_close(y1, ref, bound, f"batch M={M}")
    assert rms < 2e-3, rms
    # the parts of a split tile are added in CTA order, and every call leaves the counters at
    # zero for the next: the same bits every call
    np.testing.assert_array_equal(y1.view(np.uint16), y2.view(np.uint16))
    np.testing.assert_array_equal(y1.view(np.uint16), y3.view(np.uint16))


@pytest.mark.parametrize("M,K,N", [
    (16, 1024, 40000),  # 313 tiles of 2 units: many tiles cut between two CTAs
    (24, 8192, 512),    # 4 tiles of 16 units on 64 CTAs: every tile added from 16 parts
    (64, 1024, 130),    # 4 units in all: one per CTA, a ragged second tile
])
def test_batch_split_schedules_every_element(tb, M, K, N):
    seed = 1410 + K % 97
    x = ti.activations(seed, M, K)
    sg = ti.rademacher_signs(seed, K)
    L = HostLayer(seed + 1, N, K)
    mats = device_layer(seed + 1, N, K, from_host=L)
    y1, y2 = run(tb, x, sg, mats, N, repeat=2)
    ref, bound = linear_reference(x, sg, 1024, L)
    assert_linear_close(y1, ref, bound, f"batch split M={M} {K}->{N}")
    np.testing.assert_array_equal(y1.view(np.uint16), y2.view(np.uint16))


@pytest.mark.parametrize("M", [1, 8, 16, 32, 64])
@pytest.mark.parametrize("K,N", [(5120, 17408), (17408, 5120), (5120, 6144)])
def test_batch_layer_shapes_sampled(tb, M, K, N):
    seed = ti.config_seed(6, M + K % 13)
    x = ti.activations(seed, M, K)
    sg = ti.rademacher_signs(seed, K)
    mats = device_layer(seed, N, K)
    (y,) = run(tb, x, sg, mats, N)
    rng = np.random.default_rng(seed)
    cols = np.sort(rng.choice(N, size=min(N, 160), replace=False))
    codes = np.concatenate([ti.ternary_codes(seed, c, c + 1, K) for c in cols])
    scales = np.concatenate([ti.group_scales(seed, c, c + 1, K // 128) for c in cols])
    words = oracle.pack_w2(codes)
    biases = oracle.biases_for(scales)
    xf = x.astype(np.float64)
    ref = oracle.packed_linear(xf, sg, 1024, words, scales, biases)
    bound = 2e-3 * oracle.abs_product_sum(xf, sg, 1024, words, scales, biases) + 1e-5
    mx, rms = assert_linear_close(y[:, cols], ref, bound, f"batch {M}x{K}->{N}")
    assert rms < 2e-3, rms


@pytest.mark.parametrize("M", [5, 24, 64])
def test_batch_scale_only_block0_affine_and_unfused_block(tb, M):
    K, N = 4096, 200
    x = ti.activations(1420 + M, M, K)
    sg = ti.rademacher_signs(1420, K)
    L = HostLayer(1421, N, K)
    w, s, b = device_layer(1421, N, K, from_host=L)
    (y0,) = run(tb, x, sg, (w, s, None), N)
    ref0, bound0 = linear_reference(x, sg, 1024, L, scale_only=True)
    assert_linear_close(y0, ref0, bound0, "batch scale-only")
    (y1,) = run(tb, x, None, (w, s, b), N, block=0)
    ref1, bound1 = linear_reference(x, None, 0, L)
    assert_linear_close(y1, ref1, bound1, "batch block 0")
    (y3,) = run(tb, x, sg, (w, s, b), N, block=2048)
    ref3, bound3 = linear_reference(x, sg, 2048, L)
    assert_linear_close(y3, ref3, bound3, "batch block 2048")
    words = ti.raw_words(1422, N, K)
    sc = ti.group_scales(1422, 0, N, K // 128)
    bi = ti.free_biases(1422, N, K // 128)
    (y2,) = run(tb, x, sg, (dev(words.view(np.int32)), dev(sc), dev(bi)), N)
    xf = x.astype(np.float64)
    ref2 = oracle.packed_linear(xf, sg, 1024, words, sc, bi)
    bound2 = 2e-3 * oracle.abs_product_sum(xf, sg, 1024, words, sc, bi) + 1e-5
    assert_linear_close(y2, ref2, bound2, "batch general affine")


def test_batch_guards_and_refusal(tb):
    M, K, N = 40, 2048, 77
    x = dev(ti.activations(1430, M, K))
    w, s, b = device_layer(1431, N, K, from_host=HostLayer(1431, N, K))
    G = 4096
    y_raw = torch.full((2 * G + M * N * 2,), 0xA5, dtype=torch.uint8, device="cuda")
    y = y_raw[G:G + M * N * 2].view(torch.float16).view(M, N)
    nws = tb.tb_packed_linear_workspace_size(M, K, N, 1024, BATCH)
    ws_raw = torch.full((2 * G + nws,), 0xA5, dtype=torch.uint8, device="cuda")
    ws = ws_raw[G:G + nws]
    ws.zero_()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tb_packed_linear(x, dev(ti.rademacher_signs(1430, K)), 1024, w, s, b, y, ws, st, algo=BATCH)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for raw, n in ((y_raw, M * N * 2), (ws_raw, nws)):
        assert bool((raw[:G] == 0xA5).all()) and bool((raw[G + n:] == 0xA5).all())
    # K not a multiple of 1024: the batched GEMV refuses (block 0, K = 384)
    x2 = torch.zeros((M, 384), dtype=torch.float16, device="cuda")
    w2 = torch.zeros((N, 384 // 16), dtype=torch.int32, device="cuda")
    s2 = torch.zeros((N, 3), dtype=torch.float16, device="cuda")
    ws2 = torch.zeros(tb.tb_packed_linear_workspace_size(M, 384, N, 0, BATCH) + 1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(tb.TBError) as e:
        tb.tb_packed_linear(x2, None, 0, w2, s2, None, torch.empty((M, N), dtype=torch.float16, device="cuda"),
                            ws2, st, algo=BATCH)
    assert e.value.status == tb.TB_ERR_UNSUPPORTED
