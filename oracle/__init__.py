"""CPU oracle for NCHW conv2d and the per-channel NCHW broadcast.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline call it; the library never does.  The arithmetic lives in
``oracle.c`` (plain C, fp64, one output element at a time); this module only
compiles it with gcc and marshals numpy arrays through ctypes.

Sources followed (see oracle.c for the formulas):
  * conv2d: "Tuning High Performance Convolution on NVIDIA GPUs" (TVM v0.5
    autotvm tutorial), Step 1 -- topi.nn.conv2d_nchw with inlined zero padding.
  * broadcast: "[CINN] Add the TileBroadcastTactic for NCHW broadcast"
    (PaddlePaddle PR 70092), Introduction / Example -- [1,C,1,1] => [N,C,H,W].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

EPI_NONE, EPI_BIAS, EPI_BIAS_EXP, EPI_BIAS_RSQRT, EPI_BIAS_RECIP, EPI_BIAS_RELU = 0, 1, 2, 3, 4, 5
BC_COPY, BC_EXP, BC_RSQRT, BC_RECIP = 0, 1, 2, 3


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile oracle.c into a shared library (gcc, OpenMP).  Returns the path."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
           "-fno-fast-math", "-ffp-contract=off", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building first if needed) and return the ctypes handle."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    i, d, f, p = ctypes.c_int, ctypes.c_double, ctypes.c_float, ctypes.c_void_p
    lib.oracle_out_size.argtypes = [i, i, i, i]
    lib.oracle_out_size.restype = i
    lib.oracle_conv_flops.argtypes = [i] * 10
    lib.oracle_conv_flops.restype = d
    lib.oracle_conv2d_nchw.argtypes = [i] * 10 + [p, p, p, i, d, p, p, i]
    lib.oracle_conv2d_nchw.restype = i
    lib.oracle_conv2d_nchw_points.argtypes = [i] * 10 + [p, p, p, i, d, ctypes.c_long, p, p, p]
    lib.oracle_conv2d_nchw_points.restype = i
    lib.oracle_bcast_value.argtypes = [i, f, f]
    lib.oracle_bcast_value.restype = d
    lib.oracle_bcast_nchw.argtypes = [i, i, i, i, i, p, f, p]
    lib.oracle_bcast_nchw.restype = i
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = i
    return lib


def _f64(a) -> np.ndarray:
    """Exact widening of an fp16/bf16/fp32 array (numpy or torch) to fp64."""
    if hasattr(a, "detach"):  # torch tensor: bf16 has no numpy dtype
        import torch
        a = a.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def out_size(n: int, k: int, stride: int, pad: int, lib=None) -> int:
    return (lib or load()).oracle_out_size(n, k, stride, pad)


def conv_flops(N, CI, H, W, CO, KH, KW, stride, pad, groups=1, lib=None) -> float:
    return (lib or load()).oracle_conv_flops(N, CI, H, W, CO, KH, KW, stride, pad, groups)


def conv2d_nchw(data, kernel, stride=1, pad=0, groups=1, bias=None,
                epi=EPI_NONE, eps=1e-5, nthreads=1, lib=None):
    """Full conv.  data [N,CI,H,W], kernel [CO,CI/groups,KH,KW].
    Returns (out, absum), both float64 [N,CO,Ho,Wo]."""
    lib = lib or load()
    x, w = _f64(data), _f64(kernel)
    N, CI, H, W = x.shape
    CO, cig, KH, KW = w.shape
    if cig * groups != CI:
        raise ValueError("kernel input channels do not match CI/groups")
    Ho, Wo = lib.oracle_out_size(H, KH, stride, pad), lib.oracle_out_size(W, KW, stride, pad)
    if Ho <= 0 or Wo <= 0:
        raise ValueError("empty output")
    b = _f64(bias) if bias is not None else None
    out = np.empty((N, CO, Ho, Wo), np.float64)
    sabs = np.empty_like(out)
    rc = lib.oracle_conv2d_nchw(N, CI, H, W, CO, KH, KW, stride, pad, groups,
                                x.ctypes.data, w.ctypes.data,
                                b.ctypes.data if b is not None else None,
                                epi, eps, out.ctypes.data, sabs.ctypes.data, nthreads)
    if rc != 0:
        raise ValueError("oracle rejected the shape")
    return out, sabs


def conv2d_nchw_points(data, kernel, flat_idx, stride=1, pad=0, groups=1, bias=None,
                       epi=EPI_NONE, eps=1e-5, lib=None):
    """The definition at chosen flat output indices.  Returns (out, absum)."""
    lib = lib or load()
    x, w = _f64(data), _f64(kernel)
    N, CI, H, W = x.shape
    CO, _, KH, KW = w.shape
    idx = np.ascontiguousarray(np.asarray(flat_idx, dtype=np.int64))
    b = _f64(bias) if bias is not None else None
    out = np.empty(idx.shape, np.float64)
    sabs = np.empty_like(out)
    rc = lib.oracle_conv2d_nchw_points(N, CI, H, W, CO, KH, KW, stride, pad, groups,
                                       x.ctypes.data, w.ctypes.data,
                                       b.ctypes.data if b is not None else None,
                                       epi, eps, idx.size, idx.ctypes.data,
                                       out.ctypes.data, sabs.ctypes.data)
    if rc != 0:
        raise ValueError("oracle rejected the shape or an index")
    return out, sabs


def bcast_value(op: int, v: float, eps: float = 1e-5, lib=None) -> float:
    return (lib or load()).oracle_bcast_value(op, v, eps)


def bcast_nchw(N, C, H, W, op, var, eps=1e-5, lib=None):
    """out[n,c,h,w] = op(var[c]) as float64 [N,C,H,W]."""
    lib = lib or load()
    v = np.ascontiguousarray(np.asarray(var, dtype=np.float32))
    if v.shape != (C,):
        raise ValueError("var must have C elements")
    out = np.empty((N, C, H, W), np.float64)
    if lib.oracle_bcast_nchw(N, C, H, W, op, v.ctypes.data, eps, out.ctypes.data) != 0:
        raise ValueError("oracle rejected the shape or op")
    return out


def num_threads(lib=None) -> int:
    return (lib or load()).oracle_num_threads()
