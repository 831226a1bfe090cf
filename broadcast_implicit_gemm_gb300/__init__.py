"""Python binding of libbigemm.so: NCHW conv2d (tcgen05 implicit GEMM / SIMT)
and the per-channel NCHW broadcast on one GB300 GPU.

The functions named like the C ABI (``conv2d_nchw_plan``, ``conv2d_nchw_run``,
``bcast_nchw_run``, ...) only marshal arguments through ctypes: every step of
the computation runs in the library's CUDA kernels.  PyTorch supplies device
memory and the current stream.  There is no fallback: if the library is
missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import json
import os
import threading

__all__ = [
    "F32", "F16", "BF16", "EPI_NONE", "EPI_BIAS", "EPI_BIAS_EXP", "EPI_BIAS_RSQRT", "EPI_BIAS_RECIP", "EPI_BIAS_RELU",
    "BC_COPY", "BC_EXP", "BC_RSQRT", "BC_RECIP", "KIND_AUTO", "KIND_UMMA", "KIND_SIMT",
    "MODE_NHWC", "MODE_DIRECT", "MODE_HALO", "MODE_SUB", "MODE_STACK", "MODE_STRIDED",
    "MODE_IM2COL",
    "BigemmError", "Plan", "PlanOptions", "library_path", "load_library",
    "conv2d_nchw_plan", "conv2d_nchw_plan_ex", "conv2d_nchw_run", "conv2d_nchw_plan_destroy",
    "conv2d_nchw_plan_describe", "conv2d_nchw_run_noalloc", "bcast_nchw_run",
    "bcast_nchw_run_flat", "bcast_run",
    "bigemm_status_string", "bigemm_last_device_error", "bigemm_clear_device_error",
    "bigemm_set_wait_timeout_ns", "bigemm_debug_wait_timeout", "bigemm_profile_enable",
    "bigemm_profile_read", "bigemm_version", "conv2d", "bcast", "out_size",
]

F32, F16, BF16 = 0, 1, 2
EPI_NONE, EPI_BIAS, EPI_BIAS_EXP, EPI_BIAS_RSQRT, EPI_BIAS_RECIP, EPI_BIAS_RELU = 0, 1, 2, 3, 4, 5
BC_COPY, BC_EXP, BC_RSQRT, BC_RECIP = 0, 1, 2, 3
KIND_AUTO, KIND_UMMA, KIND_SIMT = 0, 1, 2
MODE_NHWC, MODE_DIRECT, MODE_HALO, MODE_SUB, MODE_STACK, MODE_STRIDED, MODE_IM2COL = 1, 2, 3, 4, 5, 6, 7
EPI_NAMES = {"none": EPI_NONE, "bias": EPI_BIAS, "bias_exp": EPI_BIAS_EXP,
             "bias_rsqrt": EPI_BIAS_RSQRT, "bias_recip": EPI_BIAS_RECIP, "bias_relu": EPI_BIAS_RELU}
DTYPE_CODES = {"f32": F32, "f16": F16, "bf16": BF16}

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


class BigemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {bigemm_status_string(status)} (status {status})")


class PlanOptions(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("tile_n", ctypes.c_int), ("split_k", ctypes.c_int),
                ("stages", ctypes.c_int), ("box_w", ctypes.c_int), ("box_h", ctypes.c_int),
                ("mode", ctypes.c_int), ("resident_b", ctypes.c_int), ("epi_warps", ctypes.c_int),
                ("cta_pair", ctypes.c_int)]


class KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int),
                ("total_ms", ctypes.c_double)]


def library_path() -> str:
    return os.environ.get("BIGEMM_LIB", os.path.join(_HERE, "libbigemm.so"))


def load_library():
    """Load libbigemm.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build the CUDA library first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        _declare(lib)
        _lib = lib
        return lib


def _declare(lib):
    i, u64, f, p, sz = ctypes.c_int, ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
    plan_args = [i] * 10 + [i, i, i, i]
    lib.conv2d_nchw_plan.argtypes = plan_args + [p, ctypes.POINTER(p)]
    lib.conv2d_nchw_plan_ex.argtypes = plan_args + [ctypes.POINTER(PlanOptions), p, ctypes.POINTER(p)]
    lib.conv2d_nchw_run.argtypes = [p, p, p, p, f, p, p]
    lib.conv2d_nchw_plan_destroy.argtypes = [p]
    lib.conv2d_nchw_plan_describe.argtypes = [p, ctypes.c_char_p, sz]
    lib.conv2d_nchw_run_noalloc.argtypes = [i] * 9 + [i, i, i, p, p, p, f, p, p, p]
    lib.bcast_nchw_run.argtypes = [i, i, i, i, i, p, f, p, i, p]
    lib.bcast_nchw_run_flat.argtypes = [i, i, i, i, i, p, f, p, i, p]
    lib.bcast_run.argtypes = [i, i, i, i, p, f, p, i, p]
    lib.bigemm_status_string.argtypes = [i]
    lib.bigemm_status_string.restype = ctypes.c_char_p
    lib.bigemm_last_device_error.argtypes = []
    lib.bigemm_clear_device_error.argtypes = []
    lib.bigemm_set_wait_timeout_ns.argtypes = [u64]
    lib.bigemm_debug_wait_timeout.argtypes = [u64, p]
    lib.bigemm_profile_enable.argtypes = [i]
    lib.bigemm_profile_read.argtypes = [ctypes.POINTER(KernelTime), i, ctypes.POINTER(i)]
    lib.bigemm_version.argtypes = []
    lib.bigemm_version.restype = ctypes.c_char_p
    for name in ("conv2d_nchw_plan", "conv2d_nchw_plan_ex", "conv2d_nchw_run",
                 "conv2d_nchw_run_noalloc",
                 "conv2d_nchw_plan_destroy", "conv2d_nchw_plan_describe", "bcast_nchw_run",
                 "bcast_nchw_run_flat", "bcast_run", "bigemm_last_device_error",
                 "bigemm_clear_device_error",
                 "bigemm_set_wait_timeout_ns", "bigemm_debug_wait_timeout",
                 "bigemm_profile_enable", "bigemm_profile_read"):
        getattr(lib, name).restype = i


def _check(status: int, where: str):
    if status != 0:
        raise BigemmError(status, where)


def _stream(stream):
    """A cudaStream_t value: an int, a torch.cuda.Stream, or None = torch's current stream."""
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


# --------------------------------------------------------------------- C ABI

def bigemm_status_string(status: int) -> str:
    return load_library().bigemm_status_string(status).decode()


def bigemm_version() -> str:
    return load_library().bigemm_version().decode()


class Plan:
    """Owns a bigemm_plan handle (and its device scratch) until closed."""

    def __init__(self, handle, shape):
        self._h = handle
        self.shape = shape

    @property
    def handle(self):
        if self._h is None:
            raise ValueError("plan already destroyed")
        return self._h

    def describe(self) -> dict:
        return json.loads(conv2d_nchw_plan_describe(self))

    def close(self):
        if self._h is not None:
            h, self._h = self._h, None
            _check(load_library().conv2d_nchw_plan_destroy(h), "conv2d_nchw_plan_destroy")

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def conv2d_nchw_plan(N, H, W, CO, CI, KH, KW, stride, padding, groups, in_dtype, out_dtype,
                     epi=EPI_NONE, search=0, stream=None) -> Plan:
    h = ctypes.c_void_p()
    _check(load_library().conv2d_nchw_plan(N, H, W, CO, CI, KH, KW, stride, padding, groups,
                                           in_dtype, out_dtype, epi, search, _stream(stream),
                                           ctypes.byref(h)), "conv2d_nchw_plan")
    return Plan(h.value, (N, H, W, CO, CI, KH, KW, stride, padding, groups))


def conv2d_nchw_plan_ex(N, H, W, CO, CI, KH, KW, stride, padding, groups, in_dtype, out_dtype,
                        epi=EPI_NONE, search=0, options: PlanOptions | dict | None = None,
                        stream=None) -> Plan:
    if isinstance(options, dict):
        options = PlanOptions(**options)
    h = ctypes.c_void_p()
    _check(load_library().conv2d_nchw_plan_ex(N, H, W, CO, CI, KH, KW, stride, padding, groups,
                                              in_dtype, out_dtype, epi, search,
                                              ctypes.byref(options) if options is not None else None,
                                              _stream(stream), ctypes.byref(h)),
           "conv2d_nchw_plan_ex")
    return Plan(h.value, (N, H, W, CO, CI, KH, KW, stride, padding, groups))


def conv2d_nchw_run(plan: Plan, data, kernel, bias, eps, out, stream=None):
    _check(load_library().conv2d_nchw_run(plan.handle, _ptr(data), _ptr(kernel), _ptr(bias),
                                          float(eps), _ptr(out), _stream(stream)),
           "conv2d_nchw_run")


def conv2d_nchw_plan_destroy(plan: Plan):
    plan.close()


def conv2d_nchw_plan_describe(plan: Plan) -> str:
    buf = ctypes.create_string_buffer(1 << 16)
    _check(load_library().conv2d_nchw_plan_describe(plan.handle, buf, len(buf)),
           "conv2d_nchw_plan_describe")
    return buf.value.decode()


def conv2d_nchw_run_noalloc(N, H, W, CO, CI, KH, KW, stride, padding, in_dtype, out_dtype, epi,
                            data, kernel, bias, eps, out, timeout_flag=None, stream=None):
    """The allocation-free convolution (no plan; scratch in the library's fixed
    device array).  For callers that cannot allocate device memory."""
    _check(load_library().conv2d_nchw_run_noalloc(N, H, W, CO, CI, KH, KW, stride, padding,
                                                  in_dtype, out_dtype, epi, _ptr(data),
                                                  _ptr(kernel), _ptr(bias), float(eps), _ptr(out),
                                                  _ptr(timeout_flag), _stream(stream)),
           "conv2d_nchw_run_noalloc")


def bcast_nchw_run(N, C, H, W, op, var, eps, out, out_dtype, stream=None):
    _check(load_library().bcast_nchw_run(N, C, H, W, op, _ptr(var), float(eps), _ptr(out),
                                         out_dtype, _stream(stream)), "bcast_nchw_run")


def bcast_nchw_run_flat(N, C, H, W, op, var, eps, out, out_dtype, stream=None):
    _check(load_library().bcast_nchw_run_flat(N, C, H, W, op, _ptr(var), float(eps), _ptr(out),
                                              out_dtype, _stream(stream)), "bcast_nchw_run_flat")


def bcast_run(B0, P, B1, op, var, eps, out, out_dtype, stream=None):
    """The general broadcast [1,P,1] => [B0,P,B1]: out[b0,p,b1] = op(var[p])."""
    _check(load_library().bcast_run(B0, P, B1, op, _ptr(var), float(eps), _ptr(out), out_dtype,
                                    _stream(stream)), "bcast_run")


def bigemm_last_device_error() -> int:
    return load_library().bigemm_last_device_error()


def bigemm_clear_device_error():
    _check(load_library().bigemm_clear_device_error(), "bigemm_clear_device_error")


def bigemm_set_wait_timeout_ns(ns: int):
    _check(load_library().bigemm_set_wait_timeout_ns(int(ns)), "bigemm_set_wait_timeout_ns")


def bigemm_debug_wait_timeout(ns: int, stream=None):
    _check(load_library().bigemm_debug_wait_timeout(int(ns), _stream(stream)),
           "bigemm_debug_wait_timeout")


def bigemm_profile_enable(on: bool):
    _check(load_library().bigemm_profile_enable(1 if on else 0), "bigemm_profile_enable")


def bigemm_profile_read() -> dict:
    """{kernel name: (launches, total_ms)} of the launches recorded since enable(True)."""
    arr = (KernelTime * 64)()
    n = ctypes.c_int()
    _check(load_library().bigemm_profile_read(arr, 64, ctypes.byref(n)), "bigemm_profile_read")
    return {arr[i].name.decode(): (arr[i].launches, arr[i].total_ms) for i in range(min(n.value, 64))}


# ------------------------------------------------------------ convenience

def out_size(n: int, k: int, stride: int, pad: int) -> int:
    """Output extent of one axis (the library validates the same rule)."""
    span = n + 2 * pad - k
    return -1 if span < 0 else span // stride + 1


_TORCH_CODES = None


def _dtype_code(t) -> int:
    global _TORCH_CODES
    if _TORCH_CODES is None:
        import torch
        _TORCH_CODES = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}
    return _TORCH_CODES[t]


_plans: dict = {}


def conv2d(x, w, stride=1, padding=0, groups=1, bias=None, epi=EPI_NONE, eps=1e-5,
           out_dtype=None, search=0, out=None, stream=None):
    """out = op(conv2d_nchw(x, w) + bias) with a cached plan per shape (torch tensors on CUDA)."""
    import torch
    N, CI, H, W = x.shape
    CO, _, KH, KW = w.shape
    odt = out_dtype if out_dtype is not None else x.dtype
    key = (N, H, W, CO, CI, KH, KW, stride, padding, groups, x.dtype, odt, epi, search,
           x.device.index)
    plan = _plans.get(key)
    if plan is None:
        plan = conv2d_nchw_plan(N, H, W, CO, CI, KH, KW, stride, padding, groups,
                                _dtype_code(x.dtype), _dtype_code(odt), epi, search, stream)
        _plans[key] = plan
    if out is None:
        Ho, Wo = out_size(H, KH, stride, padding), out_size(W, KW, stride, padding)
        out = torch.empty((N, CO, Ho, Wo), dtype=odt, device=x.device)
    conv2d_nchw_run(plan, x, w, bias, eps, out, stream)
    return out


def bcast(var, N, H, W, op=BC_EXP, eps=1e-5, out_dtype=None, out=None, stream=None):
    """out[n,c,h,w] = op(var[c]) for a CUDA fp32 tensor var of C elements."""
    import torch
    C = var.numel()
    odt = out_dtype or torch.float32
    if out is None:
        out = torch.empty((N, C, H, W), dtype=odt, device=var.device)
    bcast_nchw_run(N, C, H, W, op, var, eps, out, _dtype_code(odt), stream)
    return out
