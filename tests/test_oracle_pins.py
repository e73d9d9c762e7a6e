"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each test checks the oracle against the mathematics (explicit matrices built by
a different construction, closed forms, invariants), against hand-computed
fixtures under tests/golden/, or against brute force on tiny inputs written
independently of the oracle's code.  A plausible slip in the oracle (dropped
scale, wrong sign order, transposed index, sequency instead of natural order,
MSB-first packing, bias ignored) fails at least one of them.
"""
import itertools

import numpy as np
import pytest

import oracle
import tb_inputs as ti
from conftest import read_golden


# ----------------------------------------------------------------------------
# Sylvester-Walsh-Hadamard transform
# ----------------------------------------------------------------------------
def sylvester(n):
    """H_n by the recursion H_2n = [[H, H], [H, -H]], H_1 = [1]."""
    H = np.array([[1.0]])
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]])
    return H


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 64, 256, 1024])
def test_sylvester_builder_is_orthogonal(n):
    H = sylvester(n)
    assert np.array_equal(H @ H.T, n * np.eye(n))


def test_sylvester_natural_order_closed_form():
    # natural (Sylvester) order: H[i, j] = (-1) ** popcount(i & j)
    n = 128
    H = sylvester(n)
    for i, j in itertools.product(range(n), repeat=2):
        assert H[i, j] == (-1) ** bin(i & j).count("1")


@pytest.mark.parametrize("n", [1, 2, 4, 8, 32, 128, 512, 1024, 2048])
def test_fwht_equals_explicit_matrix(n):
    rng = np.random.default_rng(n)
    K = 3 * n
    x = rng.standard_normal((2, K))
    s = rng.choice([-1, 1], size=K)
    H = sylvester(n) / np.sqrt(n)
    want_f = np.concatenate([(H @ (s[b * n:(b + 1) * n] * x[:, b * n:(b + 1) * n]).T).T
                             for b in range(3)], axis=1)
    want_i = np.concatenate([s[b * n:(b + 1) * n] * (H @ x[:, b * n:(b + 1) * n].T).T
                             for b in range(3)], axis=1)
    np.testing.assert_allclose(oracle.fwht(x, n, s), want_f, rtol=0, atol=1e-12)
    np.testing.assert_allclose(oracle.fwht(x, n, s, inverse=True), want_i, rtol=0, atol=1e-12)


def test_fwht_worked_examples():
    rows = read_golden("fwht_worked.txt")
    it = iter(rows)
    r = next(it)
    assert r[0] == "block" and int(r[1]) == 4
    x = np.array(next(it)[1:], float)
    s = np.array(next(it)[1:], float)
    fwd = np.array(next(it)[1:], float)
    inv = np.array(next(it)[1:], float)
    np.testing.assert_array_equal(oracle.fwht(x, 4, s), fwd)
    np.testing.assert_array_equal(oracle.fwht(x, 4, s, inverse=True), inv)
    r = next(it)
    assert r[0] == "block" and int(r[1]) == 2
    x = np.array(next(it)[1:], float)
    s = np.array(next(it)[1:], float)
    fwd2 = np.array(next(it)[1:], float)
    np.testing.assert_allclose(oracle.fwht(x, 2, s) * np.sqrt(2), fwd2, atol=1e-15)


def test_fwht_closed_forms_block_1024():
    K = 1024
    delta = np.zeros(K)
    delta[0] = 1.0
    ones = np.ones(K)
    # H e_0 is the all-ones column; normalised by 1/32
    np.testing.assert_array_equal(oracle.fwht(delta, 1024), np.full(K, 1 / 32))
    # H 1 = 1024 e_0; normalised: 32 e_0
    want = np.zeros(K)
    want[0] = 32.0
    np.testing.assert_array_equal(oracle.fwht(ones, 1024), want)
    # a delta at j gives column j: (-1)^popcount(i & j) / 32
    j = 0b1011001101
    dj = np.zeros(K)
    dj[j] = 1.0
    col = np.array([(-1) ** bin(i & j).count("1") for i in range(K)]) / 32
    np.testing.assert_array_equal(oracle.fwht(dj, 1024), col)


@pytest.mark.parametrize("n", [512, 2048, 4096])
def test_fwht_closed_forms_other_blocks(n):
    # the pack's loader also accepts blocks 512, 2048 and 4096 (scale 1/sqrt(n): 1/(16 sqrt 2),
    # 1/(32 sqrt 2), 1/64)
    K = 2 * n
    delta = np.zeros(K)
    delta[n] = 1.0  # first element of the second block
    want = np.zeros(K)
    want[n:] = 1 / np.sqrt(n)
    np.testing.assert_allclose(oracle.fwht(delta, n), want, rtol=1e-15, atol=0)
    ones = np.ones(K)
    want = np.zeros(K)
    want[0] = want[n] = np.sqrt(n)
    np.testing.assert_allclose(oracle.fwht(ones, n), want, rtol=1e-15, atol=1e-12)
    j = (n // 2) | 5
    dj = np.zeros(n)
    dj[j] = 1.0
    col = np.array([(-1) ** bin(i & j).count("1") for i in range(n)]) / np.sqrt(n)
    np.testing.assert_allclose(oracle.fwht(dj, n), col, rtol=1e-15, atol=0)
    # signs on the inverse path come last: s * (H/sqrt n) x
    s_ = ti.rademacher_signs(n, K)
    x = np.random.default_rng(n).standard_normal(K)
    np.testing.assert_allclose(oracle.fwht(oracle.fwht(x, n, s_), n, s_, inverse=True), x, atol=1e-12)


def test_fwht_involution_parseval_and_signs():
    rng = np.random.default_rng(7)
    K = 5120
    x = rng.standard_normal((3, K))
    s = ti.rademacher_signs(3, K)
    xr = oracle.fwht(x, 1024, s)
    np.testing.assert_allclose(oracle.fwht(xr, 1024, s, inverse=True), x, atol=1e-12)
    # orthogonal per block: norms of every block are preserved
    nb = np.linalg.norm(x.reshape(3, 5, 1024), axis=-1)
    nr = np.linalg.norm(xr.reshape(3, 5, 1024), axis=-1)
    np.testing.assert_allclose(nr, nb, rtol=1e-12)
    # signs +1 reduces to the textbook transform
    np.testing.assert_allclose(oracle.fwht(x[:, :1024], 1024),
                               x[:, :1024] @ sylvester(1024).T / 32, atol=1e-12)
    # the forward and the inverse are different maps when signs are not all +1
    assert not np.allclose(oracle.fwht(x, 1024, s), oracle.fwht(x, 1024, s, inverse=True))


def test_fwht_block0_and_errors():
    x = np.arange(8.0)
    np.testing.assert_array_equal(oracle.fwht(x, 0), x)
    with pytest.raises(ValueError):
        oracle.fwht(np.zeros(1000), 1024)
    with pytest.raises(ValueError):
        oracle.fwht(np.zeros(12), 3)


# ----------------------------------------------------------------------------
# W2-g128 container
# ----------------------------------------------------------------------------
def test_pack_golden_words():
    for r in read_golden("pack_words.txt"):
        t = np.array([int(v) for v in r[:16]], dtype=np.int8)[None, :]
        want = int(r[16], 16)
        assert int(oracle.pack_w2(t)[0, 0]) == want, r
        np.testing.assert_array_equal(oracle.unpack_w2(np.array([[want]], np.uint32), 16), t)


def test_pack_unpack_round_trip_and_errors():
    t = ti.ternary_codes(11, 0, 37, 256)
    w = oracle.pack_w2(t)
    assert w.dtype == np.uint32 and w.shape == (37, 16)
    np.testing.assert_array_equal(oracle.unpack_w2(w, 256), t)
    bad = t.copy()
    bad[3, 17] = 2
    with pytest.raises(ValueError):
        oracle.pack_w2(bad)
    # code 3 is never packed but unpacks to t = 2 (q - 1)
    assert oracle.unpack_w2(np.array([[0xFFFFFFFF]], np.uint32), 16).tolist() == [[2] * 16]


def test_decode_worked_example():
    g = {r[0]: r[1:] for r in read_golden("decode_worked.txt")}
    s = np.array([[int(g["scale_bits"][0], 16)]], np.uint16).view(np.float16)
    b = np.array([[int(g["bias_bits"][0], 16)]], np.uint16).view(np.float16)
    assert b[0, 0] == -s[0, 0]
    np.testing.assert_array_equal(oracle.biases_for(s), b)
    words = np.full((1, 8), 0x55555555, np.uint32)
    words[0, 0] = int(g["word"][0], 16)
    W = oracle.decode_w2(words, s, b, 128)
    want = np.zeros(128)
    want[:16] = np.array(g["values_over_s"], float) * float(s[0, 0])
    np.testing.assert_array_equal(W[0], want)


def test_decode_value_set_and_counts():
    N, K = 9, 512
    t = ti.ternary_codes(2, 0, N, K)
    s = ti.group_scales(2, 0, N, K // 128)
    b = oracle.biases_for(s)
    W = oracle.decode_w2(oracle.pack_w2(t), s, b, K)
    S = np.repeat(s.astype(np.float64), 128, axis=1)
    assert np.array_equal(W == S, t == 1)
    assert np.array_equal(W == -S, t == -1)
    assert np.array_equal(W == 0, t == 0)
    for n in range(N):
        vals, counts = np.unique(np.sign(W[n]), return_counts=True)
        tv, tc = np.unique(t[n], return_counts=True)
        assert vals.tolist() == tv.tolist() and counts.tolist() == tc.tolist()


def test_decode_uses_bias_as_stored():
    # a general affine group (bias != -scale) must follow s*q + b literally
    words = np.array([[0x22550A46] * 8], np.uint32)
    s = np.array([[0.5]], np.float16)
    b = np.array([[0.25]], np.float16)
    q = np.array([2, 1, 0, 1, 2, 2, 0, 0, 1, 1, 1, 1, 2, 0, 2, 0] * 8, float)
    np.testing.assert_array_equal(oracle.decode_w2(words, s, b, 128)[0], 0.5 * q + 0.25)


def test_decode_scale_only_worked_example():
    # the scale-only reading (no bias read) of the worked group: the page's {-s, 0, s}
    g = {r[0]: r[1:] for r in read_golden("decode_worked.txt")}
    s = np.array([[int(g["scale_bits"][0], 16)]], np.uint16).view(np.float16)
    words = np.full((1, 8), 0x55555555, np.uint32)
    words[0, 0] = int(g["word"][0], 16)
    want = np.zeros(128)
    want[:16] = np.array(g["values_over_s"], float) * float(s[0, 0])
    np.testing.assert_array_equal(oracle.decode_w2(words, s, None, 128)[0], want)


def test_decode_scale_only_equals_the_packed_bias():
    # for every code the pack writes (and code 3, which it never writes), s*t is exactly
    # s*q + b with the pack's b = -s
    N, K = 7, 384
    t = ti.ternary_codes(4, 0, N, K)
    s = ti.group_scales(4, 0, N, K // 128)
    w = oracle.pack_w2(t)
    W0 = oracle.decode_w2(w, s, None, K)
    np.testing.assert_array_equal(W0, oracle.decode_w2(w, s, oracle.biases_for(s), K))
    np.testing.assert_array_equal(W0, t.astype(np.float64) * np.repeat(s.astype(np.float64), 128, axis=1))
    w3 = np.full((1, 8), 0xFFFFFFFF, np.uint32)
    s3 = np.array([[0.5]], np.float16)
    np.testing.assert_array_equal(oracle.decode_w2(w3, s3, None, 128), np.ones((1, 128)))
    np.testing.assert_array_equal(oracle.decode_w2(w3, s3, oracle.biases_for(s3), 128), np.ones((1, 128)))


# ----------------------------------------------------------------------------
# Packed.__call__: non-embedding and embedding paths
# ----------------------------------------------------------------------------
def _bits_of_word(word):
    """2-bit fields of a uint32 read off its binary string (least significant first)."""
    s = format(int(word), "032b")[::-1]
    return [int(s[2 * i]) + 2 * int(s[2 * i + 1]) for i in range(16)]


def test_packed_linear_brute_force():
    M, K, N, block = 2, 256, 3, 128
    rng = np.random.default_rng(5)
    x = rng.standard_normal((M, K)).astype(np.float16)
    signs = ti.rademacher_signs(9, K)
    t = ti.ternary_codes(4, 0, N, K)
    w = oracle.pack_w2(t)
    s = ti.group_scales(4, 0, N, K // 128)
    b = oracle.biases_for(s)
    H = sylvester(block)
    y = np.zeros((M, N))
    xr_all = []
    for m in range(M):
        xr = []
        xr_all.append(xr)
        for blk in range(K // block):
            seg = [float(x[m, blk * block + i]) * int(signs[blk * block + i]) for i in range(block)]
            for i in range(block):
                xr.append(sum(H[i, j] * seg[j] for j in range(block)) / np.sqrt(block))
        for n in range(N):
            acc = 0.0
            for k in range(K):
                q = _bits_of_word(w[n, k // 16])[k % 16]
                acc += xr[k] * (float(s[n, k // 128]) * q + float(b[n, k // 128]))
            y[m, n] = acc
    got = oracle.packed_linear(x, signs, block, w, s, b)
    np.testing.assert_allclose(got, y, rtol=1e-12, atol=1e-12)
    # scale-only (no biases read): the same sums with the ternary codes times their scale
    y0 = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            y0[m, n] = sum(xr_all[m][k] * float(s[n, k // 128]) * int(t[n, k]) for k in range(K))
    np.testing.assert_allclose(oracle.packed_linear(x, signs, block, w, s, None), y0, rtol=1e-12, atol=1e-12)


def test_abs_product_sum_brute_force():
    # the scale of every linear tolerance, sum_k |x'_k| * |s q + b|, by explicit loops on the
    # tiny configuration's block: x' from the Sylvester matrix (not the butterfly), each weight
    # read bit by bit off its word, a stored bias that is not -s and a field holding 3
    M, K, N, block = 2, 1024, 3, 1024
    x = ti.activations(0, M, K)
    signs = ti.rademacher_signs(0, K)
    w = ti.raw_words(17, N, K)
    w[0, 0] = 0xFFFFFFFF  # sixteen fields of 3
    s = ti.group_scales(17, 0, N, K // 128)
    b = ti.free_biases(17, N, K // 128)
    assert (b.astype(np.float64) != -s.astype(np.float64)).all()
    H = sylvester(block)
    want = np.zeros((M, N))
    want0 = np.zeros((M, N))
    xr = np.zeros((M, K))
    for m in range(M):
        seg = x[m].astype(np.float64) * signs
        xr[m] = (H @ seg) / 32.0
        for n in range(N):
            acc = acc0 = 0.0
            for k in range(K):
                q = _bits_of_word(w[n, k // 16])[k % 16]
                sc, bi = float(s[n, k // 128]), float(b[n, k // 128])
                acc += abs(xr[m, k]) * abs(sc * q + bi)
                acc0 += abs(xr[m, k]) * abs(sc * (q - 1))
            want[m, n] = acc
            want0[m, n] = acc0
    got = oracle.abs_product_sum(x, signs, block, w, s, b)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=0)
    np.testing.assert_allclose(oracle.abs_product_sum(x, signs, block, w, s, None), want0, rtol=1e-12)
    # the slips this pin exists for would each move the sum well away from the loops' value
    Wabs = np.abs(oracle.decode_w2(w, s, b, K))
    slips = {
        "|x| for |x'|": np.abs(x.astype(np.float64)) @ Wabs.T,
        "|s| dropped": np.abs(xr) @ np.abs(oracle.decode_w2(w, np.ones_like(s), b, K)).T,
        "bias dropped": np.abs(xr) @ np.abs(oracle.decode_w2(w, s, np.zeros_like(b), K)).T,
        "|x' w| summed signed": np.abs(xr @ oracle.decode_w2(w, s, b, K).T),
    }
    for what, v in slips.items():
        assert np.abs(v - want).max() > 1e-3 * np.abs(want).max(), what


def test_group_sum_identity():
    # y = sum_g s_g * sum_{k in g} q_k x'_k + b_g * sum_{k in g} x'_k
    M, K, N = 3, 2048, 17
    x = ti.activations(1, M, K)
    signs = ti.rademacher_signs(2, K)
    t = ti.ternary_codes(3, 0, N, K)
    w = oracle.pack_w2(t)
    s = ti.group_scales(3, 0, N, K // 128)
    b = oracle.biases_for(s)
    xr = oracle.rotated_input(x, signs, 1024).reshape(M, K // 128, 128)
    q = (t.astype(np.float64) + 1).reshape(N, K // 128, 128)
    y = (np.einsum("mgk,ngk->mng", xr, q) * s.astype(np.float64)[None]
         + xr.sum(-1)[:, None, :] * b.astype(np.float64)[None]).sum(-1)
    np.testing.assert_allclose(oracle.packed_linear(x, signs, 1024, w, s, b), y,
                               rtol=1e-12, atol=1e-12)


def test_fold_invariant_float_weights():
    # rotating the weights' input axis offline and the activations at run time
    # leaves the product unchanged: fwht(x) . fwht(w) = x . w (blockwise orthogonal)
    rng = np.random.default_rng(3)
    K, N = 3072, 5
    x = rng.standard_normal((2, K))
    W = rng.standard_normal((N, K))
    s = ti.rademacher_signs(4, K)
    lhs = oracle.fwht(x, 1024, s) @ oracle.fwht(W, 1024, s).T
    np.testing.assert_allclose(lhs, x @ W.T, rtol=1e-10, atol=1e-10)


def test_fold_invariant_links_linear_and_embedding():
    # For a stored (rotated) ternary matrix W', the linear path computes
    # x . (inverse-rotated W')^T, and the inverse-rotated rows are exactly what
    # the embedding path returns for those rows.
    K, N = 2048, 24
    x = ti.activations(8, 2, K)
    s_ = ti.rademacher_signs(8, K)
    t = ti.ternary_codes(8, 0, N, K)
    w = oracle.pack_w2(t)
    s = ti.group_scales(8, 0, N, K // 128)
    b = oracle.biases_for(s)
    E = oracle.embed_lookup(np.arange(N), w, s, b, s_, 1024)
    np.testing.assert_allclose(oracle.packed_linear(x, s_, 1024, w, s, b),
                               x.astype(np.float64) @ E.T, rtol=1e-10, atol=1e-12)


def test_embedding_forward_transform_recovers_row():
    V, D = 50, 2048
    t = ti.ternary_codes(6, 0, V, D)
    w = oracle.pack_w2(t)
    s = ti.group_scales(6, 0, V, D // 128)
    b = oracle.biases_for(s)
    sg = ti.rademacher_signs(6, D)
    ids = np.array([3, 0, 49, 3])
    out = oracle.embed_lookup(ids, w, s, b, sg, 1024)
    np.testing.assert_allclose(oracle.fwht(out, 1024, sg), oracle.decode_w2(w[ids], s[ids], b[ids], D),
                               atol=1e-12)
    with pytest.raises(IndexError):
        oracle.embed_lookup(np.array([50]), w, s, b, sg, 1024)


def test_block_zero_means_unrotated():
    K, N = 256, 4
    x = ti.activations(2, 1, K)
    t = ti.ternary_codes(2, 0, N, K)
    s = ti.group_scales(2, 0, N, 2)
    b = oracle.biases_for(s)
    w = oracle.pack_w2(t)
    W = oracle.decode_w2(w, s, b, K)
    np.testing.assert_allclose(oracle.packed_linear(x, None, 0, w, s, b),
                               x.astype(np.float64) @ W.T, rtol=1e-13)


# ----------------------------------------------------------------------------
# Seeded input generators (shared by the oracle side and the CUDA side)
# ----------------------------------------------------------------------------
def test_splitmix64_published_outputs():
    # splitmix64 started at state 0 yields 0xe220a8397b1dcdaf, 0x6e789e6aa1b965f4, ...
    z = ti._mix64(np.array([1, 2], dtype=np.uint64) * ti.GAMMA)
    assert [int(v) for v in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4]


def test_generators_distribution_and_row_independence():
    t = ti.ternary_codes(5, 0, 256, 4096)
    freq = [(t == v).mean() for v in (-1, 0, 1)]
    np.testing.assert_allclose(freq, [0.38, 0.24, 0.38], atol=0.005)
    np.testing.assert_array_equal(ti.ternary_codes(5, 100, 101, 4096), t[100:101])
    s = ti.group_scales(5, 0, 512, 40)
    assert s.dtype == np.float16 and s.min() >= np.float16(0.005) and s.max() <= np.float16(0.02)
    np.testing.assert_array_equal(ti.group_scales(5, 7, 9, 40), s[7:9])
    sg = ti.rademacher_signs(0, 5120)
    assert set(np.unique(sg).tolist()) == {-1, 1}
    assert len(ti.sweep_layers()) == 401
    assert ti.sweep_weight_count() == 25_095_045_120


# ----------------------------------------------------------------------------
# GGUF block formats (PQ2_0, PTQ1_0) and their transcoding into the W2 container
# ----------------------------------------------------------------------------
def _golden_blocks():
    out = []
    for r in read_golden("gguf_blocks.txt"):
        fmt, sbits, fill, nlead = r[0], int(r[1], 16), int(r[2]), int(r[3])
        lead = [int(v) for v in r[4:4 + nlead]]
        byts = np.array([int(v, 16) for v in r[4 + nlead:]], dtype=np.uint8)
        t = np.full((1, 128), fill, dtype=np.int8)
        t[0, :nlead] = lead
        d = np.array([[sbits]], np.uint16).view(np.float16)
        out.append((fmt, t, d, byts))
    return out


def test_gguf_blocks_golden():
    rows = _golden_blocks()
    assert len(rows) == 8
    for fmt, t, d, byts in rows:
        enc = oracle.pq2_0_encode if fmt == "PQ2_0" else oracle.ptq1_0_encode
        dec = oracle.pq2_0_decode if fmt == "PQ2_0" else oracle.ptq1_0_decode
        got = enc(t, d)
        assert got.shape == (1, 1, oracle.PQ2_0_BYTES if fmt == "PQ2_0" else oracle.PTQ1_0_BYTES)
        np.testing.assert_array_equal(got[0, 0], byts, err_msg=fmt)
        t2, d2 = dec(byts.reshape(1, 1, -1), 128)
        np.testing.assert_array_equal(t2, t)
        np.testing.assert_array_equal(d2.view(np.uint16), d.view(np.uint16))


def test_gguf_pq2_0_slots_are_the_w2_words():
    # with the same slot order, a PQ2_0 block's 32 code bytes are the little-endian bytes of
    # the group's eight W2 words (both put code i at bits 2 (i % 16) of its word)
    t = ti.ternary_codes(21, 0, 3, 384)
    d = ti.group_scales(21, 0, 3, 3)
    blocks = oracle.pq2_0_encode(t, d)
    words = oracle.pack_w2(t).reshape(3, 3, 8)
    np.testing.assert_array_equal(blocks[:, :, 2:], words.view(np.uint8).reshape(3, 3, 32))


@pytest.mark.parametrize("fmt", ["PQ2_0", "PTQ1_0"])
def test_gguf_round_trip_and_transcode(fmt):
    N, K = 5, 640
    t = ti.ternary_codes(22, 0, N, K)
    d = ti.group_scales(22, 0, N, K // 128)
    enc = oracle.pq2_0_encode if fmt == "PQ2_0" else oracle.ptq1_0_encode
    blocks = enc(t, d)
    w, s, b = oracle.transcode_to_w2(blocks, fmt, K)
    # lossless: the container holds exactly the trits and scales the blocks held
    np.testing.assert_array_equal(oracle.unpack_w2(w, K), t)
    np.testing.assert_array_equal(s.view(np.uint16), d.view(np.uint16))
    np.testing.assert_array_equal(b.view(np.uint16), (d.view(np.uint16) ^ 0x8000))
    W = oracle.decode_w2(w, s, b, K)
    np.testing.assert_array_equal(W, t * np.repeat(d.astype(np.float64), 128, axis=1))


def test_gguf_invalid_blocks_refused():
    t = np.zeros((1, 128), np.int8)
    d = np.ones((1, 1), np.float16)
    pq = oracle.pq2_0_encode(t, d)
    pq[0, 0, 7] = 0xFF  # slot value 3
    with pytest.raises(ValueError):
        oracle.pq2_0_decode(pq, 128)
    pt = oracle.ptq1_0_encode(t, d)
    pt[0, 0, 5] = 243  # not five base-3 digits
    with pytest.raises(ValueError):
        oracle.ptq1_0_decode(pt, 128)
    pt = oracle.ptq1_0_encode(t, d)
    pt[0, 0, 27] = 13 + 81  # a digit past trit 127
    with pytest.raises(ValueError):
        oracle.ptq1_0_decode(pt, 128)
    with pytest.raises(ValueError):
        oracle.transcode_to_w2(pq, "Q4_0", 128)
