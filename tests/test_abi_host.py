"""Host-side checks of the C ABI (no GPU needed).

The library loads, exports every entry point include/tb.h declares, and refuses
bad arguments before touching the device.  Argument validation returns before
any CUDA call, so these run on a machine without a GPU.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import ternary_hadamard_rotated_gb300 as tb
    from ternary_hadamard_rotated_gb300 import build as tbbuild

    if not os.path.exists(tb.LIB_PATH):
        tbbuild.build()
    return tb.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "tb.h"), encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tb_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_layer_entry_points():
    names = declared_functions()
    for required in ("tb_pack_w2", "tb_unpack_w2", "tb_fwht", "tb_packed_linear",
                     "tb_embed_lookup", "tb_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    import ternary_hadamard_rotated_gb300 as tb

    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in tb.EXPORTED, f"binding lacks {name}"


def test_status_strings(lib):
    for code in range(0, -8, -1):
        s = lib.tb_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.tb_status_string(42).decode() == "unknown status"
    assert lib.tb_version() >= 100


P = 0x1000  # a 16-byte aligned non-null placeholder; never dereferenced by these calls


def test_packed_linear_refuses_bad_arguments(lib):
    f = lib.tb_packed_linear
    ok = dict(x=P, M=1, K=1024, signs=P, block=1024, w=P, s=P, b=P, N=16, y=P)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["x"], a["M"], a["K"], a["signs"], a["block"], a["w"], a["s"], a["b"], a["N"],
                 a["y"], None, 0, None, None)

    assert call(x=None) == -1
    assert call(w=None) == -1
    assert call(y=None) == -1
    assert call(block=256) == -3          # 512, 1024, 2048, 4096 (and 0 = not folded) only
    assert call(block=8192) == -3
    assert call(block=2048) == -2         # K = 1024 is not a multiple of the block
    assert call(block=4096, K=2048) == -2
    assert call(block=2048, K=2048) == -7  # x' of an unfused block goes through the workspace
    assert call(K=1000) == -2             # not a multiple of 128
    assert call(K=1152) == -2             # a multiple of 128 but not of the 1024 block
    assert call(M=0) == -2
    assert call(N=0) == -2
    assert call(x=P + 2) == -6            # misaligned
    # biases may be NULL (scale-only: each bias is -scale); the other checks still apply
    assert call(b=None, K=1000) == -2
    assert call(b=None, x=None) == -1
    assert call(b=P + 2) == -6            # given biases must be aligned
    # algorithm choice
    g = lib.tb_packed_linear_algo
    assert g(P, 1, 1024, P, 1024, P, P, P, 16, P, None, 0, None, 7, None) == -3
    # the tensor-core path needs its workspace
    assert g(P, 300, 1024, P, 1024, P, P, P, 16, P, None, 0, None, 2, None) == -7
    assert g(P, 300, 1024, P, 1024, P, P, P, 16, P, P, 100, None, 2, None) == -7


def test_workspace_size_query(lib):
    ws = lib.tb_packed_linear_workspace_size
    fix = ws(1, 5120, 17408, 1024)                  # decode path: the fixup region only
    assert 1024 < fix <= 3 << 20 and fix % 1024 == 0
    assert ws(2, 5120, 17408, 1024) == fix

    # batched GEMV (3..32 tokens): 1 KB of counters, fp32 parts [256 CTAs][2][128][MT], then the
    # operand images: per pass of MT tokens and 512-k chunk, 1024 MT + 32 MT bytes (1 KB rounded)
    def batch(M, K):
        MT = 8 if M <= 8 else 16 if M <= 16 else 32 if M <= 32 else 64
        passes = -(-M // MT)
        return 1024 + 256 * 2 * 128 * MT * 4 + (passes * (K // 512) * 1056 * MT + 1023) // 1024 * 1024

    assert ws(8, 5120, 17408, 1024) == fix + batch(8, 5120)
    assert ws(3, 17408, 5120, 1024) == fix + batch(3, 17408)
    assert ws(32, 5120, 6144, 1024) == fix + batch(32, 5120)
    assert lib.tb_packed_linear_algo_workspace_size(100, 2048, 64, 1024, 6) == fix + batch(100, 2048)
    # a block that is not fused: x' in natural order (fp16 [M, K], 1 KB rounded) after the region
    assert ws(16, 4096, 1000, 2048) == fix + batch(16, 4096) + (16 * 4096 * 2 + 1023) // 1024 * 1024
    assert ws(16, 1000, 1000, 2048) == 0            # K not a multiple of the block
    # tensor-core path: x' (fp16 [M, K]), two int32 counters per 128 x 128 output tile (claims
    # of a split tile, parts written), then two fp32 256 x 256 parts per SM for the stream-K
    # schedule's split tiles (with no GPU visible the bound is 256 SMs), each region rounded up
    # to 256 bytes
    def up(v):
        return (v + 255) // 256 * 256

    def tc(M, K, N, sms):
        return up(M * K * 2) + up(-(-M // 128) * -(-N // 128) * 8) + sms * 2 * 256 * 256 * 4

    big = ws(512, 5120, 17408, 1024)
    sms = (big - fix - up(512 * 5120 * 2) - up(4 * 136 * 8)) // (2 * 256 * 256 * 4)
    assert 1 <= sms <= 256
    assert big == fix + tc(512, 5120, 17408, sms)
    assert ws(512, 1000, 17408, 1024) == 0          # invalid shape -> 0
    assert lib.tb_packed_linear_algo_workspace_size(4, 2048, 64, 1024, 2) == fix + tc(4, 2048, 64, sms)


def test_other_entry_points_refuse_bad_arguments(lib):
    assert lib.tb_pack_w2(None, P, 4, 128, P, P, None, None) == -1
    assert lib.tb_pack_w2(P, P, 4, 100, P, P, None, None) == -2
    assert lib.tb_pack_w2(P, P, 0, 128, P, P, None, None) == -2
    assert lib.tb_unpack_w2(P, 4, 20, P, None) == -2
    assert lib.tb_fwht(P, P, None, 2, 1024, 256, 0, None) == -3
    assert lib.tb_fwht(P, P, None, 2, 1024, 768, 0, None) == -3
    assert lib.tb_fwht(P, P, None, 2, 1536, 1024, 0, None) == -2
    assert lib.tb_fwht(P, P, None, 2, 2048, 4096, 0, None) == -2
    assert lib.tb_fwht(P, P, None, 2, 6144, 4096, 0, None) == -2
    assert lib.tb_fwht(P + 8, P, None, 2, 1024, 1024, 0, None) == -6
    e = lib.tb_embed_lookup
    assert e(P, 4, P, P, P, 100, 1000, None, 1024, P, None, None) == -2
    assert e(P, 4, P, P, P, 100, 1024, None, 4096, P, None, None) == -2   # D not a multiple of block
    assert e(P, 4, P, P, P, 100, 1024, None, 256, P, None, None) == -3
    assert e(P, 4, P, P, P, 0, 1024, None, 1024, P, None, None) == -2
    assert e(P, 0, P, P, P, 100, 1024, None, 1024, P, None, None) == 0   # T = 0: no-op
    assert e(None, 4, P, P, P, 100, 1024, None, 1024, P, None, None) == -1
    assert e(P, 4, P, P, None, 100, 1000, None, 1024, P, None, None) == -2   # biases NULL: allowed
    assert e(P, 4, P, P, P + 2, 100, 1024, None, 1024, P, None, None) == -6


def test_transcode_refuses_bad_arguments(lib):
    import ternary_hadamard_rotated_gb300 as tb

    f = lib.tb_transcode_gguf
    assert f(None, 1, 4, 128, P, P, P, None, None) == tb.TB_ERR_NULL
    assert f(P, 1, 4, 128, None, P, P, None, None) == tb.TB_ERR_NULL
    assert f(P, 3, 4, 128, P, P, P, None, None) == tb.TB_ERR_UNSUPPORTED
    assert f(P, 1, 0, 128, P, P, P, None, None) == tb.TB_ERR_SHAPE
    assert f(P, 2, 4, 100, P, P, P, None, None) == tb.TB_ERR_SHAPE
    assert f(P + 1, 1, 4, 128, P, P, P, None, None) == tb.TB_ERR_ALIGN   # PQ2_0: 2-byte blocks
    assert f(P + 2, 2, 4, 128, P, P, P, None, None) == tb.TB_ERR_ALIGN   # PTQ1_0: 4-byte blocks
    assert f(P, 1, 4, 128, P + 4, P, P, None, None) == tb.TB_ERR_ALIGN   # words 16-byte aligned


def test_multi_refuses_bad_arguments(lib):
    import ctypes

    arr = (ctypes.c_void_p * 5)(*([P] * 5))
    ns = (ctypes.c_int64 * 5)(*([16] * 5))
    f = lib.tb_packed_linear_multi
    assert f(P, 1, 1024, P, 1024, 5, arr, arr, arr, ns, arr, None, 0, None, None) == -2   # n > 4
    assert f(P, 1, 1024, P, 1024, 0, arr, arr, arr, ns, arr, None, 0, None, None) == -2   # n < 1
    assert f(P, 1, 1536, P, 1024, 2, arr, arr, arr, ns, arr, None, 0, None, None) == -2   # K % 1024
    assert f(P, 1, 1024, P, 256, 2, arr, arr, arr, ns, arr, None, 0, None, None) == -3
    assert f(P, 1, 1024, P, 2048, 2, arr, arr, arr, ns, arr, None, 0, None, None) == -2
    # a block other than 1024 needs the workspace for x' even on the decode path
    assert f(P, 1, 2048, P, 2048, 2, arr, arr, arr, ns, arr, None, 0, None, None) == -7
    assert f(None, 1, 1024, P, 1024, 2, arr, arr, arr, ns, arr, None, 0, None, None) == -1
    nul = (ctypes.c_void_p * 2)(P, None)
    assert f(P, 1, 1024, P, 1024, 2, nul, arr, arr, ns, arr, None, 0, None, None) == -1
    bad = (ctypes.c_int64 * 2)(16, 0)
    assert f(P, 1, 1024, P, 1024, 2, arr, arr, arr, bad, arr, None, 0, None, None) == -2
    # the prefill path of a multi call needs the x' workspace
    assert f(P, 64, 1024, P, 1024, 2, arr, arr, arr, ns, arr, None, 0, None, None) == -7


def test_chain_link_struct_matches_header():
    import ternary_hadamard_rotated_gb300 as tb

    # int64 K, two int32, five arrays of four 8-byte fields, two pointers: 192 bytes, no padding
    assert ctypes.sizeof(tb.ChainLink) == 192
    assert tb.ChainLink.K.offset == 16 and tb.ChainLink.w.offset == 32 and tb.ChainLink.y.offset == 160


def test_chain_refuses_bad_arguments(lib):
    import ternary_hadamard_rotated_gb300 as tb

    assert lib.tb_chain_plan_size(0) == 0
    assert lib.tb_chain_plan_size(3) >= 3 * (4 * 128 + 176)
    assert lib.tb_chain_workspace_size() >= 1280

    def link(**kw):
        lk = tb.ChainLink()
        lk.x, lk.signs, lk.K, lk.block, lk.n = P, P, 1024, 1024, 1
        lk.w[0], lk.scales[0], lk.biases[0], lk.N[0], lk.y[0] = P, P, P, 16, P
        for k, v in kw.items():
            setattr(lk, k, v)
        return lk

    def plan(lk, M=1, plan_ptr=0x10000, nbytes=1 << 20):
        arr = (tb.ChainLink * 1)(lk)
        return lib.tb_chain_plan(ctypes.cast(arr, ctypes.c_void_p), 1, M, plan_ptr, nbytes, None)

    assert lib.tb_chain_plan(None, 1, 1, 0x10000, 1 << 20, None) == tb.TB_ERR_NULL
    assert plan(link(), plan_ptr=0) == tb.TB_ERR_NULL
    assert plan(link(), M=0) == tb.TB_ERR_SHAPE
    assert plan(link(), M=9) == tb.TB_ERR_TOO_LARGE
    assert plan(link(), plan_ptr=0x10040) == tb.TB_ERR_ALIGN        # plan not 128-byte aligned
    assert plan(link(block=512)) == tb.TB_ERR_UNSUPPORTED
    assert plan(link(K=1536)) == tb.TB_ERR_SHAPE
    assert plan(link(n=0)) == tb.TB_ERR_SHAPE
    assert plan(link(n=5)) == tb.TB_ERR_SHAPE
    assert plan(link(x=None)) == tb.TB_ERR_NULL
    assert plan(link(x=P + 8)) == tb.TB_ERR_ALIGN
    assert plan(link(), nbytes=64) == tb.TB_ERR_WORKSPACE
    lk = link()
    lk.biases[0] = P + 8
    assert plan(lk) == tb.TB_ERR_ALIGN
    lk.biases[0] = None                                              # scale-only: allowed
    assert plan(lk, nbytes=64) == tb.TB_ERR_WORKSPACE
    r = lib.tb_chain_run
    assert r(None, 1, 1, 1024, P, 1 << 22, None, None) == tb.TB_ERR_NULL
    assert r(0x10000, 0, 1, 1024, P, 1 << 22, None, None) == tb.TB_ERR_SHAPE
    assert r(0x10000, 1, 9, 1024, P, 1 << 22, None, None) == tb.TB_ERR_TOO_LARGE
    assert r(0x10000, 1, 1, 1000, P, 1 << 22, None, None) == tb.TB_ERR_SHAPE
    assert r(0x10040, 1, 1, 1024, P, 1 << 22, None, None) == tb.TB_ERR_ALIGN
    assert r(0x10000, 1, 1, 1024, P, 1024, None, None) == tb.TB_ERR_WORKSPACE
    assert r(0x10000, 1, 1, 1024, None, 1 << 22, None, None) == tb.TB_ERR_WORKSPACE


def declared_prototypes():
    """name -> number of parameters, from the prototypes in include/tb.h."""
    src = open(os.path.join(ROOT, "include", "tb.h"), encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    out = {}
    for m in re.finditer(r"\b(tb_[a-z0-9_]+)\s*\(([^()]*)\)\s*;", src):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_signatures_match_the_header():
    import ternary_hadamard_rotated_gb300 as tb

    protos = declared_prototypes()
    assert set(protos) == set(declared_functions())
    for name, n in protos.items():
        assert name in tb._SIGNATURES, name
        assert len(tb._SIGNATURES[name][1]) == n, (name, n, len(tb._SIGNATURES[name][1]))


def test_gguf_linear_refuses_bad_arguments(lib):
    f = lib.tb_gguf_linear
    ws = lib.tb_gguf_linear_workspace_size
    assert ws(2, 4096, 1024) == 2 * 4096 * 2 and ws(2, 4096, 0) == 0
    # (x, signs, block, blocks, format, M, K, N, y, workspace, workspace_bytes, status, stream)
    assert f(None, None, 0, P, 1, 1, 1024, 8, P, None, 0, None, None) == -1       # x NULL
    assert f(P, None, 0, P, 3, 1, 1024, 8, P, None, 0, None, None) == -3          # format
    assert f(P, None, 768, P, 1, 1, 1536, 8, P, P, 1 << 20, None, None) == -3     # block
    assert f(P, None, 0, P, 1, 1, 1536, 8, P, None, 0, None, None) == -2          # K % 1024
    assert f(P, None, 0, P, 2, 0, 1024, 8, P, None, 0, None, None) == -2          # M
    assert f(P, None, 0, P + 2, 1, 1, 1024, 8, P, None, 0, None, None) == -6      # blocks alignment
    assert f(P, None, 1024, P, 1, 2, 2048, 8, P, P, 2 * 2048 * 2 - 16, None, None) == -7  # workspace
    assert f(P, None, 1024, P, 2, 2, 2048, 8, P, None, 0, None, None) == -7       # no workspace


def test_encode_gguf_refuses_bad_arguments(lib):
    f = lib.tb_encode_gguf
    # (w, scales, N, K, format, blocks, status, stream)
    assert f(None, P, 4, 1024, 1, P, None, None) == -1
    assert f(P, P, 4, 1024, 0, P, None, None) == -3
    assert f(P, P, 4, 100, 1, P, None, None) == -2
    assert f(P, P, 0, 1024, 2, P, None, None) == -2
    assert f(P, P, 4, 1024, 1, P + 1, None, None) == -6
    assert f(P, P, 4, 1024, 2, P + 2, None, None) == -6
    assert f(P + 4, P, 4, 1024, 1, P, None, None) == -6
