"""GPU parity of the tensor-memory decode GEMV (TB_ALGO_GEMV_TMEM: tcgen05.mma on e4m3 operands)
against the float64 oracle, and against the warp-level GEMV (TB_ALGO_GEMV_SYNC) on the same inputs.

The kernel carries x' (rounded to fp16) as three e4m3 terms per group of 128 with a per-group
power-of-two scale; the inputs here include activations whose magnitudes span many binades inside
one group, all-zero groups, and signs, so that the choice of the scale and the three-term split are
exercised, not only the synthetic N(0, 1) case.  Per element:
  |y_gpu - y_ref| <= 2e-3 * sum_k |x'_k w_k| + 1e-5
"""
import numpy as np
import pytest

import oracle
import tb_inputs as ti
from helpers import HostLayer, assert_linear_close, device_layer, linear_reference

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TMEM, SYNC = 4, 3


@pytest.fixture(scope="module")
def tb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import ternary_hadamard_rotated_gb300 as tbm

    tbm.load()
    return tbm


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def call(tb, x, sg, block, mats_or_one, Ns, algo, workspace=True, repeat=1):
    """tb_packed_linear (one matrix) or tb_packed_linear_multi; returns [repeat][matrix] arrays."""
    M, K = x.shape
    xd = dev(x)
    sd = dev(sg) if sg is not None else None
    ws = (torch.zeros(tb.tb_packed_linear_workspace_size(M, K, max(Ns), block, algo), dtype=torch.uint8,
                      device="cuda") if workspace else None)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(repeat):
        ys = [torch.full((M, n), float("nan"), dtype=torch.float16, device="cuda") for n in Ns]
        if len(Ns) == 1:
            w, s, b = mats_or_one[0]
            tb.tb_packed_linear(xd, sd, block, w, s, b, ys[0], ws, st, algo=algo)
        else:
            assert algo in (1, 0)
            tb.tb_packed_linear_multi(xd, sd, block, mats_or_one, ys, ws, st)
        outs.append(ys)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    if ws is not None:
        assert int(ws[:1024].count_nonzero().item()) == 0
    return [[y.cpu().numpy() for y in ys] for ys in outs]


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("K,N", [(1024, 256), (5120, 17408), (17408, 5120), (5120, 6144), (6144, 5120),
                                 (5120, 1024), (2048, 77), (3072, 1), (4096, 129)])
def test_tmem_gemv_against_oracle_and_warp_level(tb, M, K, N):
    seed = 800 + K % 97 + N % 89 + M
    x = ti.activations(seed, M, K)
    sg = ti.rademacher_signs(seed + 1, K)
    L = HostLayer(seed, N, K)
    mats = [device_layer(seed, N, K, from_host=L)]
    (y1,), (y2,) = call(tb, x, sg, 1024, mats, [N], TMEM, repeat=2)
    ((ys,),) = call(tb, x, sg, 1024, mats, [N], SYNC)
    ref, bound = linear_reference(x, sg, 1024, L)
    mx, rms = assert_linear_close(y1, ref, bound, f"tmem M={M} {K}->{N}")
    assert rms < 2e-3, rms
    assert_linear_close(y2, ref, bound, f"tmem second call M={M} {K}->{N}")
    assert_linear_close(ys, ref, bound, f"warp-level M={M} {K}->{N}")
    # the two calls differ at most by the order in which the two warpgroups' parts of a cut tile
    # meet in shared memory
    ulp = np.spacing(np.abs(y1).astype(np.float16)).astype(np.float64)
    assert (np.abs(y1.astype(np.float64) - y2.astype(np.float64)) <= 2 * ulp).all()


@pytest.mark.parametrize("M", [1, 2])
def test_tmem_gemv_wide_dynamic_range(tb, M):
    # activations spanning 2^-12 .. 2^12 inside every group, block 0 (x' = x, so the spread reaches
    # the operand unmixed), plus an all-zero block and a group holding a single non-zero value
    K, N = 4096, 300
    rng = np.random.default_rng(71)
    x = (rng.standard_normal((M, K)) * np.exp2(rng.integers(-12, 13, size=(M, K)))).astype(np.float16)
    x[:, 1024:2048] = 0
    x[:, 2048:2176] = 0
    x[:, 2100] = 3.0
    L = HostLayer(72, N, K)
    mats = [device_layer(72, N, K, from_host=L)]
    ((y,),) = call(tb, x, None, 0, mats, [N], TMEM)
    ref, bound = linear_reference(x, None, 0, L)
    assert_linear_close(y, ref, bound, f"tmem wide range M={M}")
    # the same activations rotated
    sg = ti.rademacher_signs(73, K)
    ((y,),) = call(tb, x, sg, 1024, mats, [N], TMEM)
    ref, bound = linear_reference(x, sg, 1024, L)
    assert_linear_close(y, ref, bound, f"tmem wide range rotated M={M}")


@pytest.mark.parametrize("M", [1, 2])
def test_tmem_gemv_zero_input(tb, M):
    K, N = 2048, 200
    x = np.zeros((M, K), np.float16)
    L = HostLayer(74, N, K)
    mats = [device_layer(74, N, K, from_host=L)]
    ((y,),) = call(tb, x, ti.rademacher_signs(74, K), 1024, mats, [N], TMEM)
    assert (y == 0).all()


@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("K,N", [(2048, 77), (6144, 5120), (5120, 20000)])
def test_tmem_gemv_without_workspace_and_scale_only(tb, M, K, N):
    # no workspace: ranges on tile boundaries; biases = NULL: each bias -s (W = s*t)
    x = ti.activations(75 + M, M, K)
    sg = ti.rademacher_signs(75, K)
    L = HostLayer(76, N, K)
    w, s, b = device_layer(76, N, K, from_host=L)
    ((y0,),) = call(tb, x, sg, 1024, [(w, s, b)], [N], TMEM, workspace=False)
    ((y1,),) = call(tb, x, sg, 1024, [(w, s, None)], [N], TMEM)
    ref, bound = linear_reference(x, sg, 1024, L)
    assert_linear_close(y0, ref, bound, "tmem tile-aligned")
    ref0, bound0 = linear_reference(x, sg, 1024, L, scale_only=True)
    assert_linear_close(y1, ref0, bound0, "tmem scale-only")


def test_tmem_gemv_general_affine(tb):
    # random words (fields 0..3) and biases apart from the scales
    M, K, N = 2, 5120, 1000
    x = ti.activations(85, M, K)
    sg = ti.rademacher_signs(85, K)
    words = ti.raw_words(86, N, K)
    sc = ti.group_scales(86, 0, N, K // 128)
    bi = ti.free_biases(86, N, K // 128)
    mats = [(dev(words.view(np.int32)), dev(sc), dev(bi))]
    ((y,),) = call(tb, x, sg, 1024, mats, [N], TMEM)
    xf = x.astype(np.float64)
    ref = oracle.packed_linear(xf, sg, 1024, words, sc, bi)
    bound = 2e-3 * oracle.abs_product_sum(xf, sg, 1024, words, sc, bi) + 1e-5
    assert_linear_close(y, ref, bound, "tmem general affine")


def test_tmem_gemv_refusals(tb):
    # more than two tokens, K not a multiple of 1024, or a block the kernel does not fuse: the
    # tensor-memory path alone refuses; TB_ALGO_GEMV falls back to the warp-level kernel
    K, N = 2048, 64
    w, s, b = device_layer(87, N, K, from_host=HostLayer(87, N, K))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for M, K_, block in ((3, 2048, 1024), (1, 384, 0)):
        x = torch.zeros((M, K_), dtype=torch.float16, device="cuda")
        y = torch.empty((M, N), dtype=torch.float16, device="cuda")
        ww = w if K_ == K else torch.zeros((N, K_ // 16), dtype=torch.int32, device="cuda")
        ss = s if K_ == K else torch.zeros((N, K_ // 128), dtype=torch.float16, device="cuda")
        with pytest.raises(tb.TBError) as e:
            tb.tb_packed_linear(x, None, block, ww, ss, None, y, None, st, algo=TMEM)
        assert e.value.status == tb.TB_ERR_UNSUPPORTED
        tb.tb_packed_linear(x, None, block, ww, ss, None, y, None, st, algo=1)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def test_tmem_gemv_image_limit_falls_back(tb):
    # without a workspace the ranges stay on tile boundaries, so a CTA of 17408 -> 5120 reads all
    # 17 blocks of x', more than its image holds: the tensor-memory path refuses; with a
    # workspace it runs
    M, K, N = 1, 17408, 5120
    x = ti.activations(88, M, K)
    sg = ti.rademacher_signs(88, K)
    L = HostLayer(88, N, K)
    w, s, b = device_layer(88, N, K, from_host=L)
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    with pytest.raises(tb.TBError) as e:
        tb.tb_packed_linear(dev(x), dev(sg), 1024, w, s, b, y, None, None, algo=TMEM)
    assert e.value.status == tb.TB_ERR_UNSUPPORTED
    ref, bound = linear_reference(x, sg, 1024, L)
    ((y1,),) = call(tb, x, sg, 1024, [(w, s, b)], [N], 1, workspace=False)
    ((y2,),) = call(tb, x, sg, 1024, [(w, s, b)], [N], TMEM)
    assert_linear_close(y1, ref, bound, "fallback")
    assert_linear_close(y2, ref, bound, "tmem with workspace")
