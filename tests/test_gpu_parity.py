"""GPU parity: every entry point of libtb.so against the float64 CPU oracle.

Same seeded inputs on both sides; bit-exact for packing/unpacking, within the
stated tolerances for floating-point outputs:
  linear / GEMM:  |y_gpu - y_ref| <= 2e-3 * sum_k |x'_k w_k| + 1e-5   per element
  transforms:     |out - ref| <= 1e-3 |ref| + 1e-6 ||block||_2
Sizes span several tiles with ragged tails; the full workload shapes are covered
element by element where the oracle is fast enough, else on sampled rows.
"""
import functools

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
    from tb_inputs import device as tdev

    tbm.load()
    tdev._load()
    return tbm


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_linear(tb, x16, signs, block, w, s, b, N, algo=0, workspace="zeros", repeat=1):
    """One tb_packed_linear call (or `repeat` calls reusing one workspace)."""
    M, K = x16.shape
    xd = dev(x16)
    sd = dev(signs) if signs is not None else None
    nws = tb.tb_packed_linear_workspace_size(M, K, N, block, algo)
    ws = torch.zeros(nws, dtype=torch.uint8, device="cuda") if workspace == "zeros" else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(repeat):
        y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        tb.tb_packed_linear(xd, sd, block, w, s, b, y, ws, st, algo=algo)
        outs.append(y)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    if ws is not None:  # the counters of shared output tiles are left zero for the next call
        assert int(ws[:1024].count_nonzero().item()) == 0
        use = algo or (1 if M <= 2 else 6 if M <= 32 else 5 if M <= 64 else 2)  # AUTO's choice
        if use == 2:
            # tensor-core path: after the 2 MB fixup region and x' (rounded up to 256 bytes)
            # come the stream-K tile counters, left zero as well
            c0 = 2098176 + (M * K * 2 + 255) // 256 * 256
            nc = -(-M // 128) * -(-N // 128)
            assert int(ws[c0:c0 + 4 * nc].count_nonzero().item()) == 0
        if use == 6:  # the batched GEMV's counters open the region after the fixup region
            assert int(ws[2098176:2098176 + 1024].count_nonzero().item()) == 0
    if repeat > 1:
        return [o.cpu().numpy() for o in outs]
    return outs[0].cpu().numpy()


# ---------------------------------------------------------------- packing
def test_pack_unpack_bit_exact(tb):
    N, K = 300, 1152
    L = HostLayer(21, N, K)
    w, s, b = device_layer(21, N, K, from_host=L)
    np.testing.assert_array_equal(w.cpu().numpy().view(np.uint32), L.words)
    np.testing.assert_array_equal(b.cpu().numpy().view(np.uint16), L.biases.view(np.uint16))
    codes = torch.empty((N, K), dtype=torch.int8, device="cuda")
    tb.tb_unpack_w2(w, codes)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(codes.cpu().numpy(), L.codes)


def test_pack_flags_bad_codes(tb):
    t = ti.ternary_codes(3, 0, 4, 128)
    t[2, 77] = 2
    w = torch.empty((4, 8), dtype=torch.int32, device="cuda")
    s = dev(ti.group_scales(3, 0, 4, 1))
    b = torch.empty_like(s)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tb_pack_w2(dev(t), s, w, b, st)
    torch.cuda.synchronize()
    assert int(st.item()) == tb.TB_DEV_BAD_CODE


def test_device_generator_matches_host(tb):
    from tb_inputs import device as tdev

    K, G = 2048, 16
    c = torch.empty((5, K), dtype=torch.int8, device="cuda")
    s = torch.empty((5, G), dtype=torch.float16, device="cuda")
    tdev.fill_codes(c, 77, 1000, K)
    tdev.fill_scales(s, 77, 1000, G)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(c.cpu().numpy(), ti.ternary_codes(77, 1000, 1005, K))
    np.testing.assert_array_equal(s.cpu().numpy().view(np.uint16),
                                  ti.group_scales(77, 1000, 1005, G).view(np.uint16))


# ---------------------------------------------------------------- FWHT
@pytest.mark.parametrize("inverse", [False, True])
def test_fwht_matches_oracle(tb, inverse):
    M, K = 5, 5120
    x = ti.activations(31, M, K)
    sg = ti.rademacher_signs(31, K)
    y = torch.empty((M, K), dtype=torch.float16, device="cuda")
    tb.tb_fwht(dev(x), y, dev(sg), 1024, inverse)
    torch.cuda.synchronize()
    ref = oracle.fwht(x.astype(np.float64), 1024, sg, inverse=inverse)
    assert_transform_close(y.cpu().numpy(), ref, what="fwht")


def test_fwht_in_place_and_unsigned(tb):
    M, K = 3, 17408
    x = ti.activations(32, M, K)
    xd = dev(x)
    tb.tb_fwht(xd, xd, None, 1024, False)
    torch.cuda.synchronize()
    assert_transform_close(xd.cpu().numpy(), oracle.fwht(x.astype(np.float64), 1024), what="in place")


# ---------------------------------------------------------------- linear: decode path
def test_linear_tiny_config(tb):
    # M = 1, K = 1024 (one block), N = 256, seed 0
    M, K, N = 1, 1024, 256
    x = ti.activations(0, M, K)
    sg = ti.rademacher_signs(0, K)
    L = HostLayer(0, N, K)
    w, s, b = device_layer(0, N, K, from_host=L)
    y = run_linear(tb, x, sg, 1024, w, s, b, N)
    ref, bound = linear_reference(x, sg, 1024, L)
    mx, rms = assert_linear_close(y, ref, bound, "tiny")
    assert rms < 2e-3, rms


@pytest.mark.parametrize("K,N", [(5120, 17408), (17408, 5120), (5120, 6144), (6144, 5120),
                                 (5120, 1024)])
def test_linear_decode_layer_shapes(tb, K, N):
    # the 27B layer shapes at M = 1, every output checked
    seed = ti.config_seed(2, K % 1000 + N % 997)
    x = ti.activations(seed, 1, K)
    sg = ti.rademacher_signs(seed + 1, K)
    L = HostLayer(seed, N, K)
    w, s, b = device_layer(seed, N, K, from_host=L)
    y = run_linear(tb, x, sg, 1024, w, s, b, N)
    ref, bound = linear_reference(x, sg, 1024, L)
    mx, rms = assert_linear_close(y, ref, bound, f"{K}->{N}")
    assert rms < 2e-3, rms


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 11, 16])
@pytest.mark.parametrize("algo", [1, 2])
def test_linear_tokens_and_ragged_rows(tb, M, algo):
    K, N = 2048, 77   # 77 rows: 4 full row tiles + a ragged tail
    x = ti.activations(100 + M, M, K)
    sg = ti.rademacher_signs(100, K)
    L = HostLayer(100, N, K)
    w, s, b = device_layer(100, N, K, from_host=L)
    y = run_linear(tb, x, sg, 1024, w, s, b, N, algo=algo)
    ref, bound = linear_reference(x, sg, 1024, L)
    assert_linear_close(y, ref, bound, f"M={M} algo={algo}")


@pytest.mark.parametrize("K,N", [(2048, 77), (17408, 5120), (5120, 1024), (1024, 33)])
@pytest.mark.parametrize("M", [1, 3])
def test_gemv_split_schedule_and_reuse(tb, K, N, M):
    # stream-K ranges split row tiles between SMs; the same workspace serves two calls in a
    # row; without a workspace the ranges stay on tile boundaries and agree
    x = ti.activations(40 + M, M, K)
    sg = ti.rademacher_signs(40, K)
    L = HostLayer(40, N, K)
    w, s, b = device_layer(40, N, K, from_host=L)
    ref, bound = linear_reference(x, sg, 1024, L)
    y1, y2 = run_linear(tb, x, sg, 1024, w, s, b, N, algo=1, repeat=2)
    y3 = run_linear(tb, x, sg, 1024, w, s, b, N, algo=1, workspace=None)
    for y, what in ((y1, "split"), (y2, "split, second call"), (y3, "tile aligned")):
        assert_linear_close(y, ref, bound, f"{what} M={M} {K}->{N}")
    # stage partials of a tile meet in fp32 shared-memory atomics, whose order may change
    # between calls: the two calls agree to an fp16 unit in the last place or two
    ulp = np.spacing(np.abs(y1).astype(np.float16)).astype(np.float64)
    assert (np.abs(y1.astype(np.float64) - y2.astype(np.float64)) <= 2 * ulp).all()


@pytest.mark.parametrize("algo", [1, 2])
def test_linear_unrotated_odd_groups(tb, algo):
    # block = 0 (module not folded): K only needs to be a multiple of 128
    M, K, N = 3, 384, 50
    x = ti.activations(7, M, K)
    L = HostLayer(7, N, K)
    w, s, b = device_layer(7, N, K, from_host=L)
    y = run_linear(tb, x, None, 0, w, s, b, N, algo=algo)
    ref, bound = linear_reference(x, None, 0, L)
    assert_linear_close(y, ref, bound, "block 0")


@pytest.mark.parametrize("N", [1, 3, 16, 17])
def test_linear_tiny_output_counts(tb, N):
    M, K = 1, 1024
    x = ti.activations(8, M, K)
    sg = ti.rademacher_signs(8, K)
    L = HostLayer(8, N, K)
    w, s, b = device_layer(8, N, K, from_host=L)
    for algo in (1, 2):
        y = run_linear(tb, x, sg, 1024, w, s, b, N, algo=algo)
        ref, bound = linear_reference(x, sg, 1024, L)
        assert_linear_close(y, ref, bound, f"N={N} algo={algo}")


@pytest.mark.parametrize("M", [1, 3, 200])
@pytest.mark.parametrize("K,Ns", [(5120, (6144, 1024, 1024)), (2048, (300, 77)), (1024, (17,))])
def test_linear_multi_shared_input(tb, M, K, Ns):
    # several matrices reading the same x in one call (q/k/v, gate/up, qkv/z of one layer)
    x = ti.activations(60 + M, M, K)
    sg = ti.rademacher_signs(60, K)
    layers = [HostLayer(61 + i, N, K) for i, N in enumerate(Ns)]
    mats = [device_layer(61 + i, N, K, from_host=L) for i, (N, L) in enumerate(zip(Ns, layers))]
    ys = [torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda") for N in Ns]
    ws = torch.zeros(tb.tb_packed_linear_workspace_size(M, K, max(Ns), 1024), dtype=torch.uint8,
                     device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tb_packed_linear_multi(dev(x), dev(sg), 1024, mats, ys, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for y, L in zip(ys, layers):
        ref, bound = linear_reference(x, sg, 1024, L)
        assert_linear_close(y.cpu().numpy(), ref, bound, f"multi M={M} N={L.N}")


# ---------------------------------------------------------------- tensor-core path
@pytest.mark.parametrize("M,K,N", [(128, 1024, 256), (200, 2048, 300), (512, 1024, 520)])
def test_linear_tc_tiles(tb, M, K, N):
    x = ti.activations(M + N, M, K)
    sg = ti.rademacher_signs(5, K)
    L = HostLayer(M, N, K)
    w, s, b = device_layer(M, N, K, from_host=L)
    y = run_linear(tb, x, sg, 1024, w, s, b, N, algo=2)
    ref, bound = linear_reference(x, sg, 1024, L)
    mx, rms = assert_linear_close(y, ref, bound, f"tc {M}x{K}x{N}")
    assert rms < 2e-3, rms


@pytest.mark.parametrize("M,K,N", [(100, 2048, 20000), (300, 1024, 19500), (260, 2048, 40000), (40, 1024, 40000)])
def test_linear_tc_stream_k_split_tiles(tb, M, K, N):
    # at least one output tile per SM (128 x 128, 256 x 256 and 128 x 256 tiles): the stream-K
    # schedule cuts tiles between two CTAs and the second one adds the other's part; ragged
    # token and row tails; the same workspace serves two calls in a row (the tiles' counters
    # are left zero), and the two results are identical (two addends: the order in which the
    # CTAs count in does not change the sum)
    x = ti.activations(M + 7, M, K)
    sg = ti.rademacher_signs(9, K)
    L = HostLayer(M + N, N, K)
    w, s, b = device_layer(M + N, N, K, from_host=L)
    y1, y2 = run_linear(tb, x, sg, 1024, w, s, b, N, algo=2, repeat=2)
    ref, bound = linear_reference(x, sg, 1024, L)
    mx, rms = assert_linear_close(y1, ref, bound, f"stream-K {M}x{K}x{N}")
    assert rms < 2e-3, rms
    np.testing.assert_array_equal(y1.view(np.uint16), y2.view(np.uint16))


@pytest.mark.parametrize("M,K,N", [(3, 128, 40), (100, 128, 300), (200, 128, 64), (130, 256, 520)])
def test_linear_tc_short_k(tb, M, K, N):
    # fewer 64-k blocks than the k split would want: no CTA may be left without one (its
    # tile would never be finished), and the tile counters are left zero
    x = ti.activations(M + K, M, K)
    L = HostLayer(M + 3, N, K)
    w, s, b = device_layer(M + 3, N, K, from_host=L)
    y = run_linear(tb, x, None, 0, w, s, b, N, algo=2)
    ref, bound = linear_reference(x, None, 0, L)
    assert_linear_close(y, ref, bound, f"tc short k {M}x{K}x{N}")


@pytest.mark.parametrize("M,K,N", [(512, 5120, 17408), (512, 17408, 5120), (4096, 5120, 17408),
                                   (4096, 17408, 5120)])
def test_prefill_configs_sampled(tb, M, K, N):
    # full prefill shapes through the auto path; the oracle checks sampled rows x all outputs
    seed = ti.config_seed(4, M + K % 7)
    x = ti.activations(seed, M, K)
    sg = ti.rademacher_signs(seed, K)
    w, s, b = device_layer(seed, N, K)
    y = run_linear(tb, x, sg, 1024, w, s, b, N)
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(M, size=4, replace=False))
    cols = np.sort(rng.choice(N, size=384, replace=False))
    # oracle-side rows of the weight matrix, regenerated from the counter-based generator
    codes = np.concatenate([ti.ternary_codes(seed, c, c + 1, K) for c in cols])
    scales = np.concatenate([ti.group_scales(seed, c, c + 1, K // 128) for c in cols])
    words = oracle.pack_w2(codes)
    biases = oracle.biases_for(scales)
    xs = x[rows].astype(np.float64)
    ref = oracle.packed_linear(xs, sg, 1024, words, scales, biases)
    bound = 2e-3 * oracle.abs_product_sum(xs, sg, 1024, words, scales, biases) + 1e-5
    mx, rms = assert_linear_close(y[np.ix_(rows, cols)], ref, bound, f"prefill {M}x{K}x{N}")
    assert rms < 2e-3, rms


@functools.lru_cache(maxsize=1)
def _batched_host_layer():
    # every 37th row of the 5120 -> 17408 matrix, regenerated by the counter-based generator
    K, N = 5120, 17408
    cols = np.arange(0, N, 37)
    L = HostLayer(5005, 1, K)
    L.codes = np.concatenate([ti.ternary_codes(5005, c, c + 1, K) for c in cols])
    L.scales = np.concatenate([ti.group_scales(5005, c, c + 1, K // 128) for c in cols])
    L.biases = oracle.biases_for(L.scales)
    L.words = oracle.pack_w2(L.codes)
    return cols, L


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16, 32, 64])
def test_batched_decode_config(tb, M):
    K, N = 5120, 17408
    seed = ti.config_seed(5, M)
    x = ti.activations(seed, M, K)
    sg = ti.rademacher_signs(seed, K)
    w, s, b = device_layer(5005, N, K)
    y = run_linear(tb, x, sg, 1024, w, s, b, N)
    cols, L = _batched_host_layer()
    ref, bound = linear_reference(x, sg, 1024, L)
    assert_linear_close(y[:, cols], ref, bound, f"batched M={M}")


# ---------------------------------------------------------------- embedding
def test_embedding_config(tb):
    # packed table 248320 x 5120, 256 uniform ids, inverse FWHT with width-5120 signs
    V, D, T = 248320, 5120, 256
    seed = ti.config_seed(5, 99)
    w, s, b = device_layer(seed, V, D)
    sg = ti.rademacher_signs(seed, D)
    ids = ti.token_ids(seed, T, V)
    out = torch.empty((T, D), dtype=torch.float16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tb_embed_lookup(dev(ids), w, s, b, dev(sg), 1024, out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    uniq = np.unique(ids)
    codes = np.concatenate([ti.ternary_codes(seed, i, i + 1, D) for i in uniq])
    scales = np.concatenate([ti.group_scales(seed, i, i + 1, D // 128) for i in uniq])
    words = oracle.pack_w2(codes)
    pos = {v: j for j, v in enumerate(uniq)}
    ref = oracle.embed_lookup(np.array([pos[i] for i in ids]), words, scales,
                              oracle.biases_for(scales), sg, 1024)
    assert_transform_close(out.cpu().numpy(), ref, what="embedding")


def test_embedding_bad_ids_and_unrotated(tb):
    V, D = 40, 384
    L = HostLayer(12, V, D)
    w, s, b = device_layer(12, V, D, from_host=L)
    ids = np.array([0, 39, 40, -1, 7], np.int32)
    out = torch.full((5, D), 1.0, dtype=torch.float16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tb_embed_lookup(dev(ids), w, s, b, None, 0, out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == tb.TB_DEV_BAD_ID
    o = out.cpu().numpy().astype(np.float64)
    assert (o[2] == 0).all() and (o[3] == 0).all()
    good = [0, 1, 4]
    ref = oracle.embed_lookup(ids[good], L.words, L.scales, L.biases, None, 0)
    np.testing.assert_array_equal(o[good], ref)  # exact: {-s, 0, s} needs no rounding
