"""GPU parity of the chained decode (tb_chain_plan / tb_chain_run) against the float64 oracle.

Each link's output is checked against the oracle applied to that link's input as the GPU
holds it after the run (the input of a link is an earlier link's fp16 output), so every link
is held to the per-element tolerance of the layer:
  |y_gpu - y_ref| <= 2e-3 * sum_k |x'_k w_k| + 1e-5
Intermediate buffers start as NaN: a link that read its input before the link producing it
had finished would carry NaN (or stale values that miss the oracle) into its output.
"""
import numpy as np
import pytest

import oracle
import tb_inputs as ti
from helpers import HostLayer, assert_linear_close, compare_chain_runs, device_layer, linear_reference

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


class SmallChain:
    """A chain over host-drawn layers: spec = [(input, [(name, K, N), ...]), ...] where input is
    'x0' or the name of an earlier output; all outputs start as NaN."""

    def __init__(self, tb, spec, M, seed):
        self.M = M
        K0 = spec[0][1][0][1]
        self.x0 = ti.activations(seed, M, K0)
        self.bufs = {"x0": dev(self.x0)}
        self.signs = {}
        self.host = {}
        self.args = []
        for li, (src, mats) in enumerate(spec):
            K = mats[0][1]
            if K not in self.signs:
                self.signs[K] = ti.rademacher_signs(seed + K, K)
            ms, ys = [], []
            for mi, (name, K_, N) in enumerate(mats):
                L = HostLayer(seed + 31 * li + mi, N, K_)
                self.host[name] = L
                ms.append(device_layer(0, N, K_, from_host=L))
                self.bufs[name] = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
                ys.append(self.bufs[name])
            self.args.append((self.bufs[src], dev(self.signs[K]), 1024, ms, ys))
        self.spec = spec

    def check(self, what="", scale_only=False):
        got = {k: v.cpu().numpy() for k, v in self.bufs.items()}
        for src, mats in self.spec:
            x = got[src]
            assert np.isfinite(x).all(), f"{what}: NaN in input {src}"
            K = mats[0][1]
            for name, _, _ in mats:
                ref, bound = linear_reference(x, self.signs[K], 1024, self.host[name], scale_only)
                assert_linear_close(got[name], ref, bound, f"{what} {name}")
        return got


# a stack-like chain on small shapes: several row tiles with ragged tails, every K on a
# 1024 boundary, shared-input links of 2 and 3 matrices, links with fewer units than SMs
SPEC = [
    ("x0", [("a_qkv", 2048, 1000), ("a_z", 2048, 3072)]),
    ("a_z", [("h1", 3072, 2048)]),
    ("h1", [("g1", 2048, 4096), ("u1", 2048, 4096)]),
    ("g1", [("h2", 4096, 2048)]),
    ("h2", [("q", 2048, 3072), ("k", 2048, 300), ("v", 2048, 130)]),
    ("q", [("h3", 3072, 1024)]),
    ("h3", [("tiny", 1024, 17)]),
    ("h3", [("head", 1024, 20000)]),
]


@pytest.mark.parametrize("M", [1, 2, 3, 8])
def test_chain_matches_oracle_link_by_link(tb, M):
    c = SmallChain(tb, SPEC, M, seed=400 + M)
    chain = tb.Chain(c.args, M)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    chain.run(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    c.check(f"chain M={M}")
    # every completed run leaves the workspace's counters at zero
    assert int(chain.workspace[:1280].count_nonzero().item()) == 0


def test_chain_twice_and_against_per_call(tb):
    M = 1
    c = SmallChain(tb, SPEC, M, seed=450)
    chain = tb.Chain(c.args, M)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    chain.run(st)
    first = {k: v.clone() for k, v in c.bufs.items()}
    for v in c.bufs.values():
        if v is not c.bufs["x0"]:
            v.fill_(float("nan"))
    chain.run(st)  # the second run on the same workspace
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    second = c.check("second run")
    # links whose input is bit-identical in both runs agree to a few ulps (shared-memory fp32 sums
    # of cut tiles may meet in another order); the links reading x0 always qualify
    compared = compare_chain_runs({k: v.cpu().numpy() for k, v in first.items()}, second, c.spec)
    assert "x0" in compared
    # the same links as one tb_packed_linear(_multi) call each agree with the chain
    for v in c.bufs.values():
        if v is not c.bufs["x0"]:
            v.fill_(float("nan"))
    ws = torch.zeros(tb.tb_packed_linear_workspace_size(M, 4096, 20000, 1024), dtype=torch.uint8,
                     device="cuda")
    for x, sg, block, mats, ys in c.args:
        tb.tb_packed_linear_multi(x, sg, block, mats, ys, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    c.check("per call")


def test_chain_plan_mismatch_computes_nothing(tb):
    M = 1
    spec = SPEC[:2]
    c = SmallChain(tb, spec, M, seed=470)
    chain = tb.Chain(c.args, M)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    # one link fewer than the plan holds: the kernel sees the mismatch and returns at once
    tb.tb_chain_run(chain.plan, chain.n - 1, M, chain.max_K, chain.workspace, st)
    torch.cuda.synchronize()
    assert int(st.item()) == tb.TB_DEV_BAD_PLAN
    assert torch.isnan(c.bufs["h1"]).all() and torch.isnan(c.bufs["a_z"]).all()
    st.zero_()
    chain.run(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    c.check("after a refused run")


def test_chain_host_refusals(tb):
    M = 1
    c = SmallChain(tb, SPEC[:1], M, seed=480)
    chain = tb.Chain(c.args, M)
    small_ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(tb.TBError) as e:
        tb.tb_chain_run(chain.plan, chain.n, M, chain.max_K, small_ws)
    assert e.value.status == tb.TB_ERR_WORKSPACE
    with pytest.raises(tb.TBError) as e:
        tb.tb_chain_run(chain.plan, chain.n, 9, chain.max_K, chain.workspace)
    assert e.value.status == tb.TB_ERR_TOO_LARGE
    x9 = torch.zeros((9, 2048), dtype=torch.float16, device="cuda")
    with pytest.raises(tb.TBError) as e:
        tb.Chain([(x9,) + tuple(c.args[0][1:])], 9)
    assert e.value.status == tb.TB_ERR_TOO_LARGE


@pytest.fixture(scope="module")
def stack(tb):
    """The bench's synthetic 64-layer stack (257 links, 7.06 GB of packed weights)."""
    import bench
    from tb_inputs import device as tdev

    return bench.Stack(tb, tdev, torch)


def check_stack_link(st, li, rng, what, rows_per_matrix=96):
    """Sampled rows of every matrix of link li against the oracle, on the input the link read
    (still in its buffer); the rows' codes and scales are regenerated on the host."""
    x, K, mats = st.links[li]
    xs = x.cpu().numpy()
    assert np.isfinite(xs).all(), f"{what}: non-finite input of link {li}"
    sg = st.signs[K].cpu().numpy()
    xf = xs.astype(np.float64)
    for name, p, layer, y in mats:
        rows = np.sort(rng.choice(p.N, size=min(p.N, rows_per_matrix), replace=False))
        seed = ti.config_seed(3, layer)
        codes = np.concatenate([ti.ternary_codes(seed, r, r + 1, K) for r in rows])
        scales = np.concatenate([ti.group_scales(seed, r, r + 1, K // 128) for r in rows])
        words = oracle.pack_w2(codes)
        biases = oracle.biases_for(scales)
        ref = oracle.packed_linear(xf, sg, 1024, words, scales, biases)
        bound = 2e-3 * oracle.abs_product_sum(xf, sg, 1024, words, scales, biases) + 1e-5
        got = y[:, : p.N].cpu().numpy()[:, rows]
        assert_linear_close(got, ref, bound, f"{what} link {li} {name}")


def test_decode_stack_calls_sampled(tb, stack):
    """The bench's timed path at full size: the 257 links as one tb_packed_linear(_multi) call
    each, in order.  Checked on sampled rows: the last in_proj_qkv + in_proj_z link (one call
    over 10240 + 6144 rows) right after it ran, then, after the rest of the step, lm_head
    (5120 -> 248320 in one call: 1940 row tiles, the longest split schedule) and the last
    down_proj."""
    import bench

    st = stack
    links = st.link_args()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(tb.tb_packed_linear_workspace_size(1, ti.MLP, ti.HIDDEN), dtype=torch.uint8,
                     device="cuda")
    for b in (st.h, st.qkv, st.z, st.q, st.k, st.v, st.gate, st.up, st.logits):
        b.fill_(float("nan"))
    j = max(i for i, (_, _, mats) in enumerate(st.links) if mats[0][0] == "in_proj_qkv")
    assert [m[0] for m in st.links[j][2]] == ["in_proj_qkv", "in_proj_z"]
    bench.run_calls(tb, links[: j + 1], ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rng = np.random.default_rng(5)
    check_stack_link(st, j, rng, "calls")
    bench.run_calls(tb, links[j + 1:], ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert bool(torch.isfinite(st.logits).all())
    n = len(st.links)
    assert st.links[n - 1][2][0][0] == "lm_head"
    for li in (n - 1, n - 2):
        check_stack_link(st, li, rng, "calls", rows_per_matrix=256 if li == n - 1 else 96)
    assert int(ws[:1024].count_nonzero().item()) == 0


def test_decode_stack_chain_sampled(tb, stack):
    """The bench's decode step at full size (257 links, 7.06 GB of weights, one chain launch):
    sampled rows of sampled links against the oracle, on the inputs those links read."""
    st = stack
    links = st.link_args()
    chain = tb.Chain(links, 1)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for b in (st.h, st.qkv, st.z, st.q, st.k, st.v, st.gate, st.up, st.logits):
        b.fill_(float("nan"))
    chain.run(status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert bool(torch.isfinite(st.logits).all())
    # lm_head (reads h, writes the logits) and the last down_proj (reads the gate output,
    # writes h): links whose input and output are both still in their buffers after the run
    rng = np.random.default_rng(3)
    for li in (len(st.links) - 1, len(st.links) - 2):
        check_stack_link(st, li, rng, "chain")
    assert int(chain.workspace[:1280].count_nonzero().item()) == 0


def test_chain_wait_timeout_winds_down(tb):
    """The bounded wait on the previous link: with the awaited count raised past what the CTAs
    can reach, every CTA gives up after the plan's limit (1 ms), the run reports TB_DEV_TIMEOUT
    and ends (no hang, no fault); the same plan with the count restored runs correctly."""
    import time

    M = 1
    spec = SPEC[:4]
    c = SmallChain(tb, spec, M, seed=490)
    chain = tb.Chain(c.args, M)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tb_chain_set_wait(chain.plan, 1_000_000, 1)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    chain.run(st)
    torch.cuda.synchronize()
    took = time.perf_counter() - t0
    assert int(st.item()) & tb.TB_DEV_TIMEOUT
    assert took < 10.0, took  # one 1 ms limit per CTA, far below the default 2 s per wait
    with pytest.raises(tb.TBError) as e:
        tb.tb_chain_set_wait(chain.plan, -1, 0)
    assert e.value.status == tb.TB_ERR_VALUE
    # after a timed-out run the workspace's counters are zeroed again, as the header asks
    chain.workspace.zero_()
    tb.tb_chain_set_wait(chain.plan, 0, 0)
    for v in c.bufs.values():
        if v is not c.bufs["x0"]:
            v.fill_(float("nan"))
    st.zero_()
    chain.run(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    c.check("after a timed-out run")
    assert int(chain.workspace[:1280].count_nonzero().item()) == 0
