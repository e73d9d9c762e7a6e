"""GPU parity on the general affine container: stored biases that are not -s, and fields
holding 3 (which the packer never writes).

The pack's own biases are always -s, and tb_pack_w2 refuses codes outside {-1, 0, 1}, so every
other GPU test sees b = -s and q <= 2 only.  The header promises more: a code q decodes to
s*q + b for any stored bias and any 2-bit field.  Here the words are uniformly random uint32
(each field 0, 1, 2 or 3 with equal odds) and the biases are drawn independently of the scales;
both are uploaded as they are.  Each path is compared element by element with the float64
oracle on the same words, scales and biases:
  |y_gpu - y_ref| <= 2e-3 * sum_k |x'_k w_k| + 1e-5      (linear paths)
  |out - ref| <= 1e-3 |ref| + 1e-6 ||block||_2            (embedding)
"""
import numpy as np
import pytest

import oracle
import tb_inputs as ti
from helpers import assert_linear_close, assert_transform_close, linear_reference

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


class AffineLayer:
    """Random words (fields 0..3), scales from the counter generator, free biases (b != -s)."""

    def __init__(self, seed, N, K):
        self.N, self.K, self.G = N, K, K // 128
        self.words = ti.raw_words(seed, N, K)
        self.scales = ti.group_scales(seed, 0, N, self.G)
        self.biases = ti.free_biases(seed, N, self.G)

    def device(self):
        return dev(self.words.view(np.int32)), dev(self.scales), dev(self.biases)


def _call(tb, x, sg, block, L, algo, repeat=1):
    M, K = x.shape
    w, s, b = L.device()
    ws = torch.zeros(tb.tb_packed_linear_workspace_size(M, K, L.N, block, algo), dtype=torch.uint8,
                     device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(repeat):
        y = torch.full((M, L.N), float("nan"), dtype=torch.float16, device="cuda")
        tb.tb_packed_linear(dev(x), None if sg is None else dev(sg), block, w, s, b, y, ws, st, algo=algo)
        outs.append(y)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert int(ws[:1024].count_nonzero().item()) == 0
    return [o.cpu().numpy() for o in outs]


def test_affine_fields_cover_every_code():
    L = AffineLayer(1, 64, 2048)
    q = oracle.unpack_w2(L.words, L.K) + 1
    assert set(np.unique(q).tolist()) == {0, 1, 2, 3}
    assert (L.biases.astype(np.float64) != -L.scales.astype(np.float64)).all()


@pytest.mark.parametrize("M", [1, 3, 8])
@pytest.mark.parametrize("K,N", [(5120, 1000), (2048, 77), (17408, 300)])
def test_affine_decode_gemv(tb, M, K, N):
    x = ti.activations(500 + M, M, K)
    sg = ti.rademacher_signs(500, K)
    L = AffineLayer(501 + K % 7, N, K)
    y1, y2 = _call(tb, x, sg, 1024, L, tb.TB_ALGO_GEMV, repeat=2)
    ref, bound = linear_reference(x, sg, 1024, L)
    for y in (y1, y2):
        assert_linear_close(y, ref, bound, f"affine GEMV M={M} {K}->{N}")


def test_affine_gemv_k_not_multiple_of_1024(tb):
    # block 0 with K % 1024 != 0 runs the row-streaming GEMV
    M, K, N = 3, 384, 50
    x = ti.activations(510, M, K)
    L = AffineLayer(511, N, K)
    (y,) = _call(tb, x, None, 0, L, tb.TB_ALGO_GEMV)
    ref, bound = linear_reference(x, None, 0, L)
    assert_linear_close(y, ref, bound, "affine K % 1024 GEMV")


@pytest.mark.parametrize("M,K,N", [(128, 1024, 256), (200, 2048, 300), (100, 2048, 20000), (40, 1024, 40000)])
def test_affine_tensor_core_gemm(tb, M, K, N):
    # whole tiles, ragged tiles, and stream-K schedules that split tiles between CTAs;
    # the decoders round s*q + b to fp16 once (exact when b = -s), inside the tolerance
    x = ti.activations(520 + M, M, K)
    sg = ti.rademacher_signs(520, K)
    L = AffineLayer(521 + N % 11, N, K)
    y1, y2 = _call(tb, x, sg, 1024, L, tb.TB_ALGO_TC, repeat=2)
    ref, bound = linear_reference(x, sg, 1024, L)
    assert_linear_close(y1, ref, bound, f"affine TC {M}x{K}x{N}")
    np.testing.assert_array_equal(y1.view(np.uint16), y2.view(np.uint16))


@pytest.mark.parametrize("M", [1, 5, 130])
def test_affine_multi_mixed_with_pack_layers(tb, M):
    # one call over an affine matrix, a pack-written matrix passed without biases, and
    # another affine matrix
    K = 2048
    x = ti.activations(530 + M, M, K)
    sg = ti.rademacher_signs(530, K)
    A1, A2 = AffineLayer(531, 700, K), AffineLayer(532, 129, K)
    t = ti.ternary_codes(533, 0, 300, K)
    sc = ti.group_scales(533, 0, 300, K // 128)
    words = oracle.pack_w2(t)
    mats = [A1.device(), (dev(words.view(np.int32)), dev(sc), None), A2.device()]
    Ns = (700, 300, 129)
    ys = [torch.full((M, n), float("nan"), dtype=torch.float16, device="cuda") for n in Ns]
    ws = torch.zeros(tb.tb_packed_linear_workspace_size(M, K, 700, 1024), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tb_packed_linear_multi(dev(x), dev(sg), 1024, mats, ys, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    xf = x.astype(np.float64)
    for y, (wd, s_, b_, what) in zip(ys, ((A1.words, A1.scales, A1.biases, "affine 1"),
                                          (words, sc, None, "scale-only"),
                                          (A2.words, A2.scales, A2.biases, "affine 2"))):
        ref = oracle.packed_linear(xf, sg, 1024, wd, s_, b_)
        bound = 2e-3 * oracle.abs_product_sum(xf, sg, 1024, wd, s_, b_) + 1e-5
        assert_linear_close(y.cpu().numpy(), ref, bound, f"multi M={M} {what}")


@pytest.mark.parametrize("M", [1, 3])
def test_affine_chain(tb, M):
    # a three-link chain of affine matrices; every link checked on the input it read
    K0 = 2048
    x0 = ti.activations(540 + M, M, K0)
    sg = {K: ti.rademacher_signs(540 + K, K) for K in (2048, 3072)}
    La, Lb = AffineLayer(541, 3072, 2048), AffineLayer(542, 1000, 2048)
    Lh, Lo = AffineLayer(543, 2048, 3072), AffineLayer(544, 20000, 2048)
    bufs = {"x0": dev(x0)}
    for name, L in (("a", La), ("b", Lb), ("h", Lh), ("o", Lo)):
        bufs[name] = torch.full((M, L.N), float("nan"), dtype=torch.float16, device="cuda")
    links = [(bufs["x0"], dev(sg[2048]), 1024, [La.device(), Lb.device()], [bufs["a"], bufs["b"]]),
             (bufs["a"], dev(sg[3072]), 1024, [Lh.device()], [bufs["h"]]),
             (bufs["h"], dev(sg[2048]), 1024, [Lo.device()], [bufs["o"]])]
    chain = tb.Chain(links, M)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    chain.run(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = {k: v.cpu().numpy() for k, v in bufs.items()}
    for src, K, outs in (("x0", 2048, (("a", La), ("b", Lb))), ("a", 3072, (("h", Lh),)),
                         ("h", 2048, (("o", Lo),))):
        assert np.isfinite(got[src]).all()
        for name, L in outs:
            ref, bound = linear_reference(got[src], sg[K], 1024, L)
            assert_linear_close(got[name], ref, bound, f"affine chain M={M} {name}")
    assert int(chain.workspace[:1280].count_nonzero().item()) == 0


@pytest.mark.parametrize("block", [1024, 0])
def test_affine_embedding(tb, block):
    V, D, T = 300, 2048, 40
    L = AffineLayer(550, V, D)
    sg = ti.rademacher_signs(551, D)
    ids = ti.token_ids(552, T, V)
    w, s, b = L.device()
    out = torch.empty((T, D), dtype=torch.float16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tb_embed_lookup(dev(ids), w, s, b, dev(sg) if block else None, block, out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.embed_lookup(ids, L.words, L.scales, L.biases, sg if block else None, block)
    assert_transform_close(out.cpu().numpy(), ref, block=block or 1024, what=f"affine embedding {block}")
