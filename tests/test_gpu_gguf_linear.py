"""GPU parity of the packed layer read straight from GGUF blocks (tb_gguf_linear) against the
float64 oracle: the blocks are written by the oracle's own encoders from seeded trits and
scales, and the reference is the oracle's transcoding of the same blocks into the W2-g128
container followed by its packed linear (the scale-only form, each bias -d).  Per element:
  |y_gpu - y_ref| <= 2e-3 * sum_k |x'_k w_k| + 1e-5
Both formats, blocks 0 / 512 / 1024, ragged row counts, 1..8 tokens (passes of up to four),
and the slot / digit values that are not trits (flagged in dev_status).
"""
import numpy as np
import pytest

import oracle
import tb_inputs as ti
from helpers import assert_linear_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

PQ2, PTQ1 = 1, 2


@pytest.fixture(scope="module")
def tb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import ternary_hadamard_rotated_gb300 as tbm

    tbm.load()
    return tbm


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def encode(fmt, seed, N, K):
    t = ti.ternary_codes(seed, 0, N, K)
    d = ti.group_scales(seed, 0, N, K // 128)
    blocks = oracle.pq2_0_encode(t, d) if fmt == PQ2 else oracle.ptq1_0_encode(t, d)
    return blocks


def reference(x, sg, block, blocks, fmt, K):
    words, scales, biases = oracle.transcode_to_w2(blocks, "PQ2_0" if fmt == PQ2 else "PTQ1_0", K)
    xf = x.astype(np.float64)
    ref = oracle.packed_linear(xf, sg, block, words, scales, biases)
    bound = 2e-3 * oracle.abs_product_sum(xf, sg, block, words, scales, biases) + 1e-5
    return ref, bound


def run(tb, x, sg, block, blocks, fmt, N, status=None):
    M, K = x.shape
    y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    wsz = tb.tb_gguf_linear_workspace_size(M, K, block)
    ws = torch.empty(max(wsz, 16), dtype=torch.uint8, device="cuda") if wsz else None
    st = status if status is not None else torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tb_gguf_linear(dev(x), None if sg is None else dev(sg), block, dev(blocks.reshape(-1)), fmt, y, ws, st)
    torch.cuda.synchronize()
    return y.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("fmt", [PQ2, PTQ1])
@pytest.mark.parametrize("M,K,N,block", [(1, 1024, 77, 1024), (1, 5120, 1000, 1024), (3, 2048, 300, 1024),
                                         (2, 17408, 256, 1024), (8, 1024, 129, 0), (5, 4096, 64, 512),
                                         (1, 6144, 515, 1024)])
def test_gguf_linear_against_oracle(tb, fmt, M, K, N, block):
    seed = 700 + fmt * 31 + K % 97 + N % 13 + M
    x = ti.activations(seed, M, K)
    sg = ti.rademacher_signs(seed, K) if block else None
    blocks = encode(fmt, seed, N, K)
    y, st = run(tb, x, sg, block, blocks, fmt, N)
    assert st == 0
    ref, bound = reference(x, sg, block, blocks, fmt, K)
    mx, rms = assert_linear_close(y, ref, bound, f"fmt {fmt} M={M} {K}->{N} block {block}")
    assert rms < 2e-3, rms


def test_gguf_linear_bad_codes_flagged(tb):
    K, N = 1024, 16
    x = ti.activations(705, 1, K)
    sg = ti.rademacher_signs(705, K)
    # PQ2_0: one slot of value 3 (read as d * 2)
    b2 = encode(PQ2, 706, N, K)
    b2[3, 2, 5] |= 0x0C  # slot 4*3 + 1 of block (3, 2) ... byte 5 bits 2-3 -> 3 wherever it was
    y, st = run(tb, x, sg, 1024, b2, PQ2, N)
    assert st & 1 and np.isfinite(y).all()
    # PTQ1_0: a byte above 242, and a digit past trit 127 in the last byte
    b1 = encode(PTQ1, 707, N, K)
    b1[1, 4, 10] = 250
    y, st = run(tb, x, sg, 1024, b1, PTQ1, N)
    assert st & 1 and np.isfinite(y).all()
    b1 = encode(PTQ1, 707, N, K)
    b1[2, 0, 27] = int(b1[2, 0, 27]) % 27 + 27  # digit 3 (trit 128) set to 1
    y, st = run(tb, x, sg, 1024, b1, PTQ1, N)
    assert st & 1
    # clean blocks leave the status untouched
    y, st = run(tb, x, sg, 1024, encode(PTQ1, 708, N, K), PTQ1, N)
    assert st == 0


@pytest.mark.parametrize("fmt", [PQ2, PTQ1])
@pytest.mark.parametrize("N,K", [(5, 128), (77, 1024), (300, 5120)])
def test_encode_gguf_bit_exact_and_round_trip(tb, fmt, N, K):
    seed = 740 + fmt + N
    t = ti.ternary_codes(seed, 0, N, K)
    d = ti.group_scales(seed, 0, N, K // 128)
    words = oracle.pack_w2(t)
    want = oracle.pq2_0_encode(t, d) if fmt == PQ2 else oracle.ptq1_0_encode(t, d)
    blocks = torch.zeros(want.size, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tb_encode_gguf(dev(words.view(np.int32)), dev(d), fmt, blocks, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    np.testing.assert_array_equal(blocks.cpu().numpy(), want.reshape(-1))
    # and back through the transcoder: the same words and scales
    w2 = torch.zeros((N, K // 16), dtype=torch.int32, device="cuda")
    s2 = torch.zeros((N, K // 128), dtype=torch.float16, device="cuda")
    tb.tb_transcode_gguf(blocks, fmt, N, K, w2, s2, None, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    np.testing.assert_array_equal(w2.cpu().numpy().view(np.uint32), words)
    np.testing.assert_array_equal(s2.cpu().numpy().view(np.uint16), d.view(np.uint16))


def test_encode_gguf_flags_code_3(tb):
    N, K = 4, 256
    words = ti.raw_words(745, N, K)  # fields 0..3
    d = ti.group_scales(745, 0, N, K // 128)
    for fmt in (PQ2, PTQ1):
        blocks = torch.zeros(N * (K // 128) * (34 if fmt == PQ2 else 28), dtype=torch.uint8, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        tb.tb_encode_gguf(dev(words.view(np.int32)), dev(d), fmt, blocks, st)
        torch.cuda.synchronize()
        assert int(st.item()) & 1
