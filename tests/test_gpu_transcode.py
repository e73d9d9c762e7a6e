"""GPU parity of tb_transcode_gguf: GGUF PQ2_0 / PTQ1_0 blocks into the W2 container.

The blocks come from the oracle's encoders (the readings of the block layout); the library's
words, scales and biases must equal the oracle's transcoding bit for bit, and equal what
tb_pack_w2 writes for the same trits and scales.  Invalid slots and digits set
TB_DEV_BAD_CODE.
"""
import numpy as np
import pytest

import oracle
import tb_inputs as ti

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import ternary_hadamard_rotated_gb300 as tbm

    tbm.load()
    return tbm


FMTS = {"PQ2_0": (1, oracle.pq2_0_encode), "PTQ1_0": (2, oracle.ptq1_0_encode)}


def run(tb, blocks, fmt, N, K, with_biases=True):
    bd = torch.from_numpy(np.ascontiguousarray(blocks).reshape(-1)).cuda()
    w = torch.full((N, K // 16), -1, dtype=torch.int32, device="cuda")
    s = torch.full((N, K // 128), float("nan"), dtype=torch.float16, device="cuda")
    b = torch.full((N, K // 128), float("nan"), dtype=torch.float16, device="cuda") if with_biases else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tb_transcode_gguf(bd, FMTS[fmt][0], N, K, w, s, b, st)
    torch.cuda.synchronize()
    return w, s, b, int(st.item())


@pytest.mark.parametrize("fmt", ["PQ2_0", "PTQ1_0"])
@pytest.mark.parametrize("N,K", [(1, 128), (7, 384), (300, 5120), (4096, 5120)])
def test_transcode_matches_oracle(tb, fmt, N, K):
    t = ti.ternary_codes(700 + N, 0, N, K)
    d = ti.group_scales(700 + N, 0, N, K // 128)
    blocks = FMTS[fmt][1](t, d)
    w, s, b, st = run(tb, blocks, fmt, N, K)
    assert st == 0
    ww, ws, wb = oracle.transcode_to_w2(blocks, fmt, K)
    np.testing.assert_array_equal(w.cpu().numpy().view(np.uint32), ww)
    np.testing.assert_array_equal(s.cpu().numpy().view(np.uint16), ws.view(np.uint16))
    np.testing.assert_array_equal(b.cpu().numpy().view(np.uint16), wb.view(np.uint16))
    if N <= 300:  # the same words and biases as the packer writes for these trits and scales
        w2 = torch.empty_like(w)
        b2 = torch.empty_like(b)
        st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
        tb.tb_pack_w2(torch.from_numpy(t).cuda(), s, w2, b2, st2)
        torch.cuda.synchronize()
        assert int(st2.item()) == 0
        assert torch.equal(w2, w) and torch.equal(b2.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("fmt", ["PQ2_0", "PTQ1_0"])
def test_transcode_without_biases(tb, fmt):
    N, K = 5, 256
    t = ti.ternary_codes(710, 0, N, K)
    d = ti.group_scales(710, 0, N, K // 128)
    blocks = FMTS[fmt][1](t, d)
    w, s, _, st = run(tb, blocks, fmt, N, K, with_biases=False)
    assert st == 0
    ww, ws, _ = oracle.transcode_to_w2(blocks, fmt, K)
    np.testing.assert_array_equal(w.cpu().numpy().view(np.uint32), ww)


def test_transcode_flags_invalid_blocks(tb):
    N, K = 3, 256
    t = np.zeros((N, K), np.int8)
    d = np.ones((N, K // 128), np.float16)
    pq = oracle.pq2_0_encode(t, d)
    pq[1, 1, 9] = 0xC5  # one slot holds 3
    assert run(tb, pq, "PQ2_0", N, K)[3] == tb.TB_DEV_BAD_CODE
    pt = oracle.ptq1_0_encode(t, d)
    pt[2, 0, 4] = 250  # not five base-3 digits
    assert run(tb, pt, "PTQ1_0", N, K)[3] == tb.TB_DEV_BAD_CODE
    pt = oracle.ptq1_0_encode(t, d)
    pt[0, 1, 27] = 13 + 27  # a digit past trit 127
    assert run(tb, pt, "PTQ1_0", N, K)[3] == tb.TB_DEV_BAD_CODE
    # the valid blocks around them are transcoded all the same
    w, s, b, st = run(tb, oracle.ptq1_0_encode(t, d), "PTQ1_0", N, K)
    assert st == 0
