"""Python binding of the GB300 folded-Hadamard ternary ``Packed`` layer library.

Argument marshalling only: every step of the layer runs in the sm_103a kernels of
``libtb.so`` (C ABI declared in ``include/tb.h``).  Tensors are torch CUDA
tensors (torch provides device memory and streams); the calls are asynchronous
on the current torch stream unless a stream is given.  There is no CPU path:
if the library is not built, importing the calls raises.

Names follow the C ABI: ``tb_pack_w2``, ``tb_unpack_w2``, ``tb_fwht``,
``tb_packed_linear``, ``tb_packed_linear_multi``, ``tb_embed_lookup``, and the chained decode
``tb_chain_plan`` / ``tb_chain_run`` (``ChainLink`` mirrors ``tb_chain_link``).
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtb.so")

TB_OK = 0
TB_ERR_NULL = -1
TB_ERR_SHAPE = -2
TB_ERR_UNSUPPORTED = -3
TB_ERR_VALUE = -4
TB_ERR_CUDA = -5
TB_ERR_ALIGN = -6
TB_ERR_WORKSPACE = -7
TB_ERR_TOO_LARGE = -8

TB_DEV_BAD_CODE = 1
TB_DEV_BAD_ID = 2
TB_DEV_TIMEOUT = 4
TB_DEV_BAD_PLAN = 8

TB_ALGO_AUTO = 0
TB_ALGO_GEMV = 1
TB_ALGO_TC = 2
TB_ALGO_GEMV_SYNC = 3
TB_ALGO_GEMV_TMEM = 4
TB_ALGO_GEMV_WIDE = 5
TB_ALGO_GEMV_BATCH = 6

TB_FMT_PQ2_0 = 1
TB_FMT_PTQ1_0 = 2

_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int
_SZ = ctypes.c_size_t

_SIGNATURES = {
    "tb_status_string": (ctypes.c_char_p, [_INT]),
    "tb_last_cuda_error": (ctypes.c_char_p, []),
    "tb_version": (_INT, []),
    "tb_pack_w2": (_INT, [_P, _P, _I64, _I64, _P, _P, _P, _P]),
    "tb_unpack_w2": (_INT, [_P, _I64, _I64, _P, _P]),
    "tb_fwht": (_INT, [_P, _P, _P, _I64, _I64, _INT, _INT, _P]),
    "tb_packed_linear_workspace_size": (_SZ, [_I64, _I64, _I64, _INT]),
    "tb_packed_linear_algo_workspace_size": (_SZ, [_I64, _I64, _I64, _INT, _INT]),
    "tb_packed_linear": (_INT, [_P, _I64, _I64, _P, _INT, _P, _P, _P, _I64, _P, _P, _SZ, _P, _P]),
    "tb_packed_linear_algo": (_INT, [_P, _I64, _I64, _P, _INT, _P, _P, _P, _I64, _P, _P, _SZ, _P,
                                     _INT, _P]),
    "tb_embed_lookup": (_INT, [_P, _I64, _P, _P, _P, _I64, _I64, _P, _INT, _P, _P, _P]),
    "tb_packed_linear_gemv_noalloc": (_INT, [_P, _I64, _I64, _P, _INT, _P, _P, _P, _I64, _P, _P, _P]),
    "tb_packed_linear_multi": (_INT, [_P, _I64, _I64, _P, _INT, _INT, _P, _P, _P, _P, _P, _P, _SZ, _P,
                                      _P]),
    "tb_chain_plan_size": (_SZ, [_INT]),
    "tb_chain_workspace_size": (_SZ, []),
    "tb_chain_plan": (_INT, [_P, _INT, _I64, _P, _SZ, _P]),
    "tb_chain_set_wait": (_INT, [_P, _I64, ctypes.c_int32, _P]),
    "tb_chain_run": (_INT, [_P, _INT, _I64, _I64, _P, _SZ, _P, _P]),
    "tb_transcode_gguf": (_INT, [_P, _INT, _I64, _I64, _P, _P, _P, _P, _P]),
    "tb_gguf_linear_workspace_size": (ctypes.c_size_t, [_I64, _I64, _INT]),
    "tb_encode_gguf": (_INT, [_P, _P, _I64, _I64, _INT, _P, _P, _P]),
    "tb_gguf_linear": (_INT, [_P, _P, _INT, _P, _INT, _I64, _I64, _I64, _P, _P, ctypes.c_size_t, _P, _P]),
}

EXPORTED = tuple(_SIGNATURES)


class TBError(RuntimeError):
    def __init__(self, fn, status):
        lib = load()
        msg = lib.tb_status_string(status).decode()
        if status == TB_ERR_CUDA:
            msg += ": " + lib.tb_last_cuda_error().decode()
        super().__init__(f"{fn} failed ({status}): {msg}")
        self.status = status


def load(path: str = LIB_PATH):
    """Load libtb.so (built by build.py); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise ImportError(f"libtb.so not built at {path}; run ternary_hadamard_rotated_gb300.build")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, rc):
    if rc != TB_OK:
        raise TBError(fn, rc)


def tb_pack_w2(codes, scales, w, biases, dev_status=None, stream=None):
    """codes int8 [N,K], scales fp16 [N,K/128] -> w uint32 [N,K/16] (as int32), biases fp16."""
    N, K = codes.shape
    _check("tb_pack_w2", load().tb_pack_w2(_ptr(codes), _ptr(scales), N, K, _ptr(w), _ptr(biases),
                                           _ptr(dev_status), _stream(stream)))


def tb_transcode_gguf(blocks, fmt, N, K, w, scales, biases=None, dev_status=None, stream=None):
    """GGUF blocks (uint8, N * K/128 blocks of 34 (PQ2_0) or 28 (PTQ1_0) bytes) -> the W2
    container: w uint32 [N, K/16] (as int32), scales fp16 [N, K/128], biases = -scales (or None)."""
    _check("tb_transcode_gguf", load().tb_transcode_gguf(_ptr(blocks), fmt, N, K, _ptr(w), _ptr(scales),
                                                         _ptr(biases), _ptr(dev_status), _stream(stream)))


def tb_encode_gguf(w, scales, fmt, blocks, dev_status=None, stream=None):
    """W2 words [N, K/16] and scales [N, K/128] -> GGUF blocks of fmt (scale-only reading)."""
    N, G = scales.shape
    _check("tb_encode_gguf", load().tb_encode_gguf(_ptr(w), _ptr(scales), N, G * 128, fmt, _ptr(blocks),
                                                   _ptr(dev_status), _stream(stream)))


def tb_gguf_linear_workspace_size(M, K, block=1024):
    return int(load().tb_gguf_linear_workspace_size(M, K, block))


def tb_gguf_linear(x, signs, block, blocks, fmt, y, workspace=None, dev_status=None, stream=None):
    """y[M,N] = fwht(x)[M,K] . W^T with W read from GGUF blocks (TB_FMT_PQ2_0 / TB_FMT_PTQ1_0)."""
    M, K = x.shape
    N = y.shape[-1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("tb_gguf_linear", load().tb_gguf_linear(_ptr(x), _ptr(signs), block, _ptr(blocks), fmt, M, K, N,
                                                   _ptr(y), _ptr(workspace), ws_bytes, _ptr(dev_status),
                                                   _stream(stream)))


def tb_unpack_w2(w, codes, stream=None):
    N, K = codes.shape
    _check("tb_unpack_w2", load().tb_unpack_w2(_ptr(w), N, K, _ptr(codes), _stream(stream)))


def tb_fwht(x, y, signs=None, block=1024, inverse=False, stream=None):
    M, K = x.shape
    _check("tb_fwht", load().tb_fwht(_ptr(x), _ptr(y), _ptr(signs), M, K, block, int(bool(inverse)),
                                     _stream(stream)))


def tb_packed_linear_workspace_size(M, K, N, block=1024, algo=TB_ALGO_AUTO):
    return load().tb_packed_linear_algo_workspace_size(M, K, N, block, algo)


def tb_packed_linear(x, signs, block, w, scales, biases, y, workspace=None, dev_status=None,
                     algo=TB_ALGO_AUTO, stream=None):
    """y[M,N] = fwht(x)[M,K] . dequant(w)^T with the packed W2-g128 weights."""
    M, K = x.shape
    N = y.shape[-1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("tb_packed_linear",
           load().tb_packed_linear_algo(_ptr(x), M, K, _ptr(signs), block, _ptr(w), _ptr(scales),
                                        _ptr(biases), N, _ptr(y), _ptr(workspace), ws_bytes,
                                        _ptr(dev_status), algo, _stream(stream)))


def tb_packed_linear_multi(x, signs, block, mats, ys, workspace=None, dev_status=None, stream=None):
    """One call for several packed matrices reading the same x.

    mats: sequence of (w, scales, biases); ys: matching outputs [M, N_i].
    """
    M, K = x.shape
    n = len(mats)
    arr_p = ctypes.c_void_p * n
    w = arr_p(*[_ptr(m[0]) for m in mats])
    sc = arr_p(*[_ptr(m[1]) for m in mats])
    bi = arr_p(*[_ptr(m[2]) for m in mats])
    Ns = (ctypes.c_int64 * n)(*[int(y.shape[-1]) for y in ys])
    yp = arr_p(*[_ptr(y) for y in ys])
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("tb_packed_linear_multi",
           load().tb_packed_linear_multi(_ptr(x), M, K, _ptr(signs), block, n, w, sc, bi, Ns, yp,
                                         _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream)))


def tb_embed_lookup(ids, w, scales, biases, signs, block, out, dev_status=None, stream=None):
    T = ids.shape[0]
    V = w.shape[0]
    D = out.shape[-1]
    _check("tb_embed_lookup",
           load().tb_embed_lookup(_ptr(ids), T, _ptr(w), _ptr(scales), _ptr(biases), V, D,
                                  _ptr(signs), block, _ptr(out), _ptr(dev_status), _stream(stream)))


def tb_packed_linear_gemv_noalloc(x, signs, block, w, scales, biases, y, dev_status=None, stream=None):
    """Decode GEMV (M <= 8) without a workspace: its scratch is a fixed array in the library."""
    M, K = x.shape
    N = y.shape[-1]
    _check("tb_packed_linear_gemv_noalloc",
           load().tb_packed_linear_gemv_noalloc(_ptr(x), M, K, _ptr(signs), block, _ptr(w),
                                                _ptr(scales), _ptr(biases), N, _ptr(y),
                                                _ptr(dev_status), _stream(stream)))


class ChainLink(ctypes.Structure):
    """ctypes image of ``tb_chain_link`` (include/tb.h)."""

    _fields_ = [
        ("x", ctypes.c_void_p),
        ("signs", ctypes.c_void_p),
        ("K", ctypes.c_int64),
        ("block", ctypes.c_int32),
        ("n", ctypes.c_int32),
        ("w", ctypes.c_void_p * 4),
        ("scales", ctypes.c_void_p * 4),
        ("biases", ctypes.c_void_p * 4),
        ("N", ctypes.c_int64 * 4),
        ("y", ctypes.c_void_p * 4),
    ]


def chain_link(x, signs, block, mats, ys):
    """One link: input x [M, K] (a tensor or a view of an earlier link's output), up to four
    (w, scales, biases) matrices reading it and their outputs ys [M, N_i]."""
    n = len(mats)
    if not 1 <= n <= 4 or len(ys) != n:
        raise ValueError("a chain link holds 1..4 matrices with one output each")
    lk = ChainLink()
    lk.x = _ptr(x)
    lk.signs = _ptr(signs)
    lk.K = int(x.shape[-1])
    lk.block = int(block)
    lk.n = n
    for i, ((w, sc, bi), y) in enumerate(zip(mats, ys)):
        lk.w[i] = _ptr(w)
        lk.scales[i] = _ptr(sc)
        lk.biases[i] = _ptr(bi)
        lk.N[i] = int(y.shape[-1])
        lk.y[i] = _ptr(y)
    return lk


def tb_chain_plan_size(n_links):
    return load().tb_chain_plan_size(n_links)


def tb_chain_workspace_size():
    return load().tb_chain_workspace_size()


def tb_chain_plan(links, M, plan, stream=None):
    """Write the plan of ``links`` (ChainLink list) for M tokens into the device buffer ``plan``."""
    n = len(links)
    arr = (ChainLink * n)(*links)
    nbytes = plan.numel() * plan.element_size()
    _check("tb_chain_plan", load().tb_chain_plan(ctypes.cast(arr, ctypes.c_void_p), n, M, _ptr(plan), nbytes,
                                                 _stream(stream)))


def tb_chain_set_wait(plan, wait_ns, extra_count=0, stream=None):
    """Bound of the plan's waits on the previous link (ns, 0 = default); extra_count > 0 only to
    test the timeout path (the awaited count can then not be reached)."""
    _check("tb_chain_set_wait", load().tb_chain_set_wait(_ptr(plan), int(wait_ns), int(extra_count),
                                                         _stream(stream)))


def tb_chain_run(plan, n_links, M, max_K, workspace, dev_status=None, stream=None):
    """Run a plan made by tb_chain_plan: one persistent launch for all its links."""
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("tb_chain_run", load().tb_chain_run(_ptr(plan), n_links, M, max_K, _ptr(workspace), ws_bytes,
                                               _ptr(dev_status), _stream(stream)))


class Chain:
    """A planned chain of packed linears on the current device.

    ``links``: sequence of (x, signs, block, mats, ys) as for :func:`chain_link`.  Holds the
    device plan (made once, here) and a zeroed workspace; ``run()`` launches the whole chain.
    """

    def __init__(self, links, M, device=None):
        import torch

        dev = torch.device("cuda") if device is None else device
        self.links = [chain_link(*lk) for lk in links]
        self.n = len(self.links)
        self.M = int(M)
        self.max_K = max(int(lk.K) for lk in self.links)
        nbytes = tb_chain_plan_size(self.n)
        self.plan = torch.empty(nbytes + 128, dtype=torch.uint8, device=dev)
        off = (-self.plan.data_ptr()) % 128
        self.plan = self.plan[off: off + nbytes]
        self.workspace = torch.zeros(tb_chain_workspace_size(), dtype=torch.uint8, device=dev)
        tb_chain_plan(self.links, self.M, self.plan)

    def run(self, dev_status=None, stream=None):
        tb_chain_run(self.plan, self.n, self.M, self.max_K, self.workspace, dev_status, stream)
