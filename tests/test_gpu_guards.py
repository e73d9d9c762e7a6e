"""Guard words around every buffer an entry point writes: nothing is written outside it.

NaN-prefilled outputs catch elements a kernel forgets to write; this file catches the other
mistake, a write past the end (or before the start) of a ragged tail.  Each output, and each
workspace, sits between two runs of canary bytes; after the call (results checked elsewhere)
both runs must be unchanged, and inputs must be unchanged as a whole.  Shapes are chosen with
ragged row tiles, token counts that are not a multiple of the kernels' passes, K not a multiple
of 1024, and blocks other than 1024.
"""
import numpy as np
import pytest

import oracle
import tb_inputs as ti

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

GUARD = 4096  # bytes of canary on each side (keeps the data 16-byte aligned)
CANARY = 0xA5


@pytest.fixture(scope="module")
def tb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import ternary_hadamard_rotated_gb300 as tbm

    tbm.load()
    return tbm


class Guarded:
    """A tensor of `shape`/`dtype` between two canary runs of GUARD bytes."""

    def __init__(self, shape, dtype, fill=None):
        n = int(np.prod(shape)) if len(shape) else 1
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((GUARD + nbytes + GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + nbytes].view(dtype).view(shape)
        if fill is not None:
            self.t.copy_(fill if torch.is_tensor(fill) else torch.as_tensor(fill).to(self.t.device))
        self.nbytes = nbytes

    def check(self, what):
        torch.cuda.synchronize()
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.nbytes:]
        assert bool((head == CANARY).all()), f"{what}: write before the start"
        assert bool((tail == CANARY).all()), f"{what}: write past the end"


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def packed(seed, N, K):
    t = ti.ternary_codes(seed, 0, N, K)
    s = ti.group_scales(seed, 0, N, K // 128)
    return dev(oracle.pack_w2(t).view(np.int32)), dev(s), dev(oracle.biases_for(s))


@pytest.mark.parametrize("M,K,N,block,algo", [
    (1, 2048, 77, 1024, 1), (3, 5120, 1000, 1024, 1), (8, 1024, 33, 1024, 1),
    (3, 384, 50, 0, 1),                       # K % 1024 != 0: the row-streaming GEMV
    (130, 2048, 300, 1024, 2), (40, 1024, 20000, 1024, 2), (200, 2048, 77, 1024, 0),
    (2, 4096, 129, 2048, 0), (5, 2048, 65, 512, 0), (130, 4096, 200, 4096, 0),
])
def test_linear_guards(tb, M, K, N, block, algo):
    x = ti.activations(700 + M, M, K)
    sg = ti.rademacher_signs(700, K)
    w, s, b = packed(701, N, K)
    xin = dev(x)
    w0, s0, b0, x0 = w.clone(), s.clone(), b.clone(), xin.clone()
    y = Guarded((M, N), torch.float16)
    nws = tb.tb_packed_linear_workspace_size(M, K, N, block, algo)
    ws = Guarded((nws,), torch.uint8, fill=torch.zeros(nws, dtype=torch.uint8))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tb_packed_linear(xin, dev(sg) if block else None, block, w, s, b, y.t, ws.t, st, algo=algo)
    y.check("y")
    ws.check("workspace")
    assert int(st.item()) == 0
    for a_, b_, what in ((w, w0, "w"), (s, s0, "scales"), (b, b0, "biases"), (xin, x0, "x")):
        assert torch.equal(a_, b_), f"{what} changed"


@pytest.mark.parametrize("M", [1, 3, 140])
def test_multi_guards(tb, M):
    K, Ns = 2048, (300, 77, 1000)
    x = dev(ti.activations(710 + M, M, K))
    sg = dev(ti.rademacher_signs(710, K))
    mats = [packed(711 + i, n, K) for i, n in enumerate(Ns)]
    ys = [Guarded((M, n), torch.float16) for n in Ns]
    nws = tb.tb_packed_linear_workspace_size(M, K, max(Ns), 1024)
    ws = Guarded((nws,), torch.uint8, fill=torch.zeros(nws, dtype=torch.uint8))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tb_packed_linear_multi(x, sg, 1024, mats, [g.t for g in ys], ws.t, st)
    for i, g in enumerate(ys):
        g.check(f"y[{i}]")
    ws.check("workspace")
    assert int(st.item()) == 0


@pytest.mark.parametrize("M", [1, 3])
def test_chain_guards(tb, M):
    K = 2048
    x = dev(ti.activations(720 + M, M, K))
    sg = dev(ti.rademacher_signs(720, K))
    m1, m2, m3 = packed(721, 300, K), packed(722, 2048, K), packed(723, 77, K)
    y1, y2, y3 = Guarded((M, 300), torch.float16), Guarded((M, 2048), torch.float16), Guarded((M, 77), torch.float16)
    links = [(x, sg, 1024, [m1, m2], [y1.t, y2.t]), (y2.t, sg, 1024, [m3], [y3.t])]
    chain = tb.Chain(links, M)
    ws = Guarded((tb.tb_chain_workspace_size(),), torch.uint8,
                 fill=torch.zeros(tb.tb_chain_workspace_size(), dtype=torch.uint8))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tb_chain_run(chain.plan, chain.n, M, chain.max_K, ws.t, st)
    for g, what in ((y1, "y1"), (y2, "y2"), (y3, "y3"), (ws, "workspace")):
        g.check(what)
    assert int(st.item()) == 0


@pytest.mark.parametrize("block,T,D", [(1024, 37, 2048), (0, 5, 384), (512, 9, 1536), (4096, 3, 4096)])
def test_embedding_guards(tb, block, T, D):
    V = 211
    w, s, b = packed(730, V, D)
    ids = dev(ti.token_ids(731, T, V))
    out = Guarded((T, D), torch.float16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tb_embed_lookup(ids, w, s, b, dev(ti.rademacher_signs(732, D)) if block else None, block, out.t, st)
    out.check("out")
    assert int(st.item()) == 0


@pytest.mark.parametrize("block,M,K", [(1024, 3, 3072), (512, 5, 1536), (2048, 3, 6144), (4096, 2, 8192)])
def test_fwht_guards(tb, block, M, K):
    x = dev(ti.activations(740, M, K))
    y = Guarded((M, K), torch.float16)
    tb.tb_fwht(x, y.t, dev(ti.rademacher_signs(741, K)), block, False)
    y.check("fwht out")


def test_pack_unpack_transcode_guards(tb):
    N, K = 37, 384
    t = dev(ti.ternary_codes(750, 0, N, K))
    s = dev(ti.group_scales(750, 0, N, K // 128))
    w = Guarded((N, K // 16), torch.int32)
    b = Guarded((N, K // 128), torch.float16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tb_pack_w2(t, s, w.t, b.t, st)
    w.check("packed words")
    b.check("biases")
    codes = Guarded((N, K), torch.int8)
    tb.tb_unpack_w2(w.t, codes.t)
    codes.check("unpacked codes")
    for fmt, nbytes in ((tb.TB_FMT_PQ2_0, 34), (tb.TB_FMT_PTQ1_0, 28)):
        blocks = torch.zeros((N * (K // 128), nbytes), dtype=torch.uint8, device="cuda")
        blocks[:, 0:2] = s.reshape(-1).view(torch.uint8).view(-1, 2)
        blocks[:, 2:] = 0x55 if fmt == tb.TB_FMT_PQ2_0 else 121  # all-zero trits: valid in both
        blocks[:, -1] = 0x55 if fmt == tb.TB_FMT_PQ2_0 else 13
        w2 = Guarded((N, K // 16), torch.int32)
        s2 = Guarded((N, K // 128), torch.float16)
        b2 = Guarded((N, K // 128), torch.float16)
        tb.tb_transcode_gguf(blocks, fmt, N, K, w2.t, s2.t, b2.t, st)
        for g, what in ((w2, "words"), (s2, "scales"), (b2, "biases")):
            g.check(f"transcode {fmt} {what}")
    torch.cuda.synchronize()
    assert int(st.item()) == 0
