"""Device-side fill of synthetic codes and scales (tb_inputs/csrc/synth.cu).

Used for workloads too large to draw on the host (the 25-billion-weight decode
sweep).  The values equal ``tb_inputs.ternary_codes`` / ``tb_inputs.group_scales``
for the same seed, row and column.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc", "synth.cu")
LIB = os.path.join(HERE, "libtbsynth.so")

_lib = None


def build(verbose: bool = False) -> str:
    nvcc = os.environ.get("NVCC", "nvcc")
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
           "-Xcompiler", "-fPIC", "-shared", SRC, "-o", LIB + ".tmp"]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {SRC}:\n{r.stdout}\n{r.stderr}")
    os.replace(LIB + ".tmp", LIB)
    return LIB


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise ImportError(f"{LIB} not built; call tb_inputs.device.build()")
        lib = ctypes.CDLL(LIB)
        for name in ("tbs_fill_codes", "tbs_fill_scales"):
            fn = getattr(lib, name)
            fn.restype = ctypes.c_int
            fn.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64,
                           ctypes.c_int64, ctypes.c_void_p]
        _lib = lib
    return _lib


def _stream(stream):
    import torch
    return (stream or torch.cuda.current_stream()).cuda_stream


def fill_codes(out, seed: int, row0: int, K: int, stream=None) -> None:
    """out: int8 CUDA tensor [nrows, K] <- codes of rows row0.. of the seeded matrix."""
    rc = _load().tbs_fill_codes(out.data_ptr(), seed, row0, out.shape[0], K, _stream(stream))
    if rc:
        raise RuntimeError(f"tbs_fill_codes failed ({rc})")


def fill_scales(out, seed: int, row0: int, G: int, stream=None) -> None:
    """out: fp16 CUDA tensor [nrows, G] <- scales of rows row0.. of the seeded matrix."""
    rc = _load().tbs_fill_scales(out.data_ptr(), seed, row0, out.shape[0], G, _stream(stream))
    if rc:
        raise RuntimeError(f"tbs_fill_scales failed ({rc})")
