"""ctypes binding for libattn.so -- argument marshalling only.

The names mirror the C ABI in ``include/attn.h``.  Nothing here computes any
part of the attention forward; if the shared library is missing the first call
raises ``AttnError`` (there is no fallback).
"""
from __future__ import annotations

import ctypes
import os
import threading

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_TIMEOUT = 4
ATTN_DTYPE_BF16 = 0
ATTN_DTYPE_F16 = 1

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libattn.so"

# Every symbol include/attn.h declares (checked by the CPU tests).
EXPORTED = ("attn_fwd", "attn_fwd_ex", "attn_fwd_splitkv", "attn_fwd_splitkv_workspace_size",
            "attn_fwd_splitkv_noalloc", "attn_status_str", "attn_last_device_status",
            "attn_check_device_status",
            "attn_kernel_launches", "attn_debug_wait_timeout", "attn_bwd", "attn_bwd_workspace_size",
            "attn_debug_unit_rates", "attn_debug_unit_schedule")

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status} ({_status_name(status)})")
        self.status = status


def _status_name(st: int) -> str:
    return {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED",
            3: "ATTN_ERR_CUDA", 4: "ATTN_ERR_TIMEOUT"}.get(st, "unknown")


def library_path() -> str:
    return os.environ.get("LIBATTN_PATH", os.path.join(_PKG, _LIB_NAME))


def load_library():
    """Load libattn.so (once); raises AttnError if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise AttnError(ATTN_ERR_CUDA, f"{path} is missing; run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, ctypes.c_float, P]
        lib.attn_fwd.restype = I
        lib.attn_fwd_ex.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, ctypes.c_float, I, P]
        lib.attn_fwd_ex.restype = I
        lib.attn_status_str.argtypes = [I]
        lib.attn_status_str.restype = ctypes.c_char_p
        lib.attn_check_device_status.argtypes = [P]
        lib.attn_check_device_status.restype = I
        lib.attn_last_device_status.argtypes = []
        lib.attn_last_device_status.restype = I
        lib.attn_kernel_launches.argtypes = []
        lib.attn_kernel_launches.restype = ctypes.c_ulonglong
        lib.attn_debug_wait_timeout.argtypes = [ctypes.c_uint, P]
        lib.attn_debug_wait_timeout.restype = I
        lib.attn_debug_unit_rates.argtypes = [ctypes.POINTER(ctypes.c_double), I, P]
        lib.attn_debug_unit_rates.restype = I
        IP = ctypes.POINTER(ctypes.c_int)
        lib.attn_debug_unit_schedule.argtypes = [I, I, I, I, I, I, I, I, IP, IP, I, IP]
        lib.attn_debug_unit_schedule.restype = I
        lib.attn_fwd_splitkv_workspace_size.argtypes = [I, I, I, I, I, I, I,
                                                        ctypes.POINTER(ctypes.c_size_t)]
        lib.attn_fwd_splitkv_workspace_size.restype = I
        lib.attn_fwd_splitkv.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, ctypes.c_float, P,
                                         ctypes.c_size_t, P]
        lib.attn_fwd_splitkv.restype = I
        lib.attn_fwd_splitkv_noalloc.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I,
                                                 ctypes.c_float, P]
        lib.attn_fwd_splitkv_noalloc.restype = I
        lib.attn_bwd_workspace_size.argtypes = [I, I, I, I, I, I, ctypes.POINTER(ctypes.c_size_t)]
        lib.attn_bwd_workspace_size.restype = I
        lib.attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, ctypes.c_float, I, P,
                                 ctypes.c_size_t, P]
        lib.attn_bwd.restype = I
        _lib = lib
        return lib


def exported_symbols():
    lib = load_library()
    return {name: getattr(lib, name, None) is not None for name in EXPORTED}


def attn_status_str(status: int) -> str:
    return load_library().attn_status_str(int(status)).decode()


def _stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def attn_fwd_ptr(q: int, k: int, v: int, o: int, lse: int, B: int, Sq: int, Skv: int, Hq: int,
                 Hkv: int, D: int, causal: int, scale: float, stream: int) -> int:
    """Raw-pointer call of the C entry point; returns the attn_status_t value."""
    return int(load_library().attn_fwd(q, k, v, o, lse, B, Sq, Skv, Hq, Hkv, D, causal,
                                       ctypes.c_float(scale), stream))


def attn_fwd_ex_ptr(q: int, k: int, v: int, o: int, lse: int, B: int, Sq: int, Skv: int, Hq: int,
                    Hkv: int, D: int, causal: int, scale: float, dtype: int, stream: int) -> int:
    """Raw-pointer call of attn_fwd_ex (dtype: ATTN_DTYPE_BF16 or ATTN_DTYPE_F16)."""
    return int(load_library().attn_fwd_ex(q, k, v, o, lse, B, Sq, Skv, Hq, Hkv, D, causal,
                                          ctypes.c_float(scale), dtype, stream))


def attn_fwd(q, k, v, o=None, lse=None, causal: int = 0, scale: float | None = None,
             stream=None, want_lse: bool = True):
    """O = softmax(scale * Q K^T [+ causal mask]) V and its fp32 log-sum-exp.

    q: bf16 or float16 CUDA tensor [B, Sq, Hq, D]; k, v: [B, Skv, Hkv, D], same
    dtype; all contiguous.
    o (optional): bf16 [B, Sq, Hq, D]; lse (optional): fp32 [B, Hq, Sq].
    causal: 0 none, 1 bottom-right aligned, 2 top-left aligned.  Returns (o, lse or None).
    Runs asynchronously on ``stream`` (default: torch's current stream).
    """
    import torch
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise AttnError(ATTN_ERR_INVALID_ARG, "q, k, v must be 4-d [B, S, H, D]")
    B, Sq, Hq, D = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise AttnError(ATTN_ERR_INVALID_ARG, "q must be bf16 or float16")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != q.dtype or not t.is_cuda or not t.is_contiguous():
            raise AttnError(ATTN_ERR_INVALID_ARG,
                            f"{name} must be a contiguous CUDA tensor of q's dtype")
    if tuple(v.shape) != tuple(k.shape) or k.shape[0] != B or k.shape[3] != D:
        raise AttnError(ATTN_ERR_INVALID_ARG, "k/v shapes do not match q")
    if o is None:
        o = torch.empty_like(q)
    if o.dtype != q.dtype:
        raise AttnError(ATTN_ERR_INVALID_ARG, "o must have q's dtype")
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / (D ** 0.5)
    dtype = ATTN_DTYPE_F16 if q.dtype == torch.float16 else ATTN_DTYPE_BF16
    st = attn_fwd_ex_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                         lse.data_ptr() if lse is not None else 0, B, Sq, Skv, Hq, Hkv, D,
                         int(causal), float(scale), dtype, _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd")
    return o, lse


def attn_fwd_splitkv_workspace_size(B: int, Sq: int, Skv: int, Hq: int, Hkv: int, D: int,
                                    causal: int) -> int:
    """Workspace bytes attn_fwd_splitkv needs on the current device (0: no split)."""
    n = ctypes.c_size_t(0)
    st = int(load_library().attn_fwd_splitkv_workspace_size(B, Sq, Skv, Hq, Hkv, D, causal,
                                                            ctypes.byref(n)))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_splitkv_workspace_size")
    return int(n.value)


def attn_fwd_splitkv_ptr(q: int, k: int, v: int, o: int, lse: int, B: int, Sq: int, Skv: int,
                         Hq: int, Hkv: int, D: int, causal: int, scale: float, workspace: int,
                         workspace_bytes: int, stream: int) -> int:
    """Raw-pointer call of attn_fwd_splitkv; returns the attn_status_t value."""
    return int(load_library().attn_fwd_splitkv(q, k, v, o, lse, B, Sq, Skv, Hq, Hkv, D, causal,
                                               ctypes.c_float(scale), workspace, workspace_bytes,
                                               stream))


def attn_fwd_splitkv(q, k, v, o=None, lse=None, causal: int = 0, scale: float | None = None,
                     workspace=None, stream=None, want_lse: bool = True):
    """attn_fwd with KV split across SMs.  `workspace`: a CUDA byte tensor of at
    least attn_fwd_splitkv_workspace_size(...) bytes, allocated here if None."""
    import torch
    B, Sq, Hq, D = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise AttnError(ATTN_ERR_INVALID_ARG, f"{name} must be a contiguous bf16 CUDA tensor")
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / (D ** 0.5)
    if workspace is None:
        n = attn_fwd_splitkv_workspace_size(B, Sq, Skv, Hq, Hkv, D, int(causal))
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)
    st = attn_fwd_splitkv_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              lse.data_ptr() if lse is not None else 0, B, Sq, Skv, Hq, Hkv, D,
                              int(causal), float(scale), workspace.data_ptr(), workspace.numel(),
                              _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_splitkv")
    return o, lse


def attn_fwd_splitkv_noalloc_ptr(q: int, k: int, v: int, o: int, lse: int, B: int, Sq: int,
                                 Skv: int, Hq: int, Hkv: int, D: int, causal: int, scale: float,
                                 stream: int) -> int:
    """Raw-pointer call of attn_fwd_splitkv_noalloc, the split-KV entry point for
    callers that cannot allocate device memory: its scratch is a static array
    inside libattn.  Returns the attn_status_t value."""
    return int(load_library().attn_fwd_splitkv_noalloc(q, k, v, o, lse, B, Sq, Skv, Hq, Hkv, D,
                                                       causal, ctypes.c_float(scale), stream))


def attn_bwd_workspace_size(B: int, Sq: int, Skv: int, Hq: int, Hkv: int, D: int) -> int:
    n = ctypes.c_size_t(0)
    st = load_library().attn_bwd_workspace_size(B, Sq, Skv, Hq, Hkv, D, ctypes.byref(n))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd_workspace_size")
    return int(n.value)


def attn_bwd_ptr(q: int, k: int, v: int, o: int, lse: int, do: int, dq: int, dk: int, dv: int,
                 B: int, Sq: int, Skv: int, Hq: int, Hkv: int, D: int, causal: int, scale: float,
                 dtype: int, workspace: int, workspace_bytes: int, stream: int) -> int:
    """Raw C-ABI call (device pointers as ints); returns the status code."""
    return load_library().attn_bwd(q, k, v, o, lse, do, dq, dk, dv, B, Sq, Skv, Hq, Hkv, D,
                                   int(causal), float(scale), int(dtype), workspace,
                                   int(workspace_bytes), stream)


def attn_bwd(q, k, v, o, lse, do, causal: int = 0, scale: float | None = None, dq=None, dk=None,
             dv=None, workspace=None, stream=None):
    """dq, dk, dv of sum(do * o) for o = attn_fwd(q, k, v, causal, scale); o and lse
    are that forward's outputs.  bf16 or float16 CUDA tensors (all the same type),
    lse fp32 [B, Hq, Sq].  Outputs and the workspace are allocated here if None."""
    import torch
    B, Sq, Hq, D = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise AttnError(ATTN_ERR_INVALID_ARG, "q must be bf16 or float16")
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        if t.dtype != q.dtype or not t.is_cuda or not t.is_contiguous():
            raise AttnError(ATTN_ERR_INVALID_ARG, f"{name} must be a contiguous CUDA tensor of q's dtype")
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous():
        raise AttnError(ATTN_ERR_INVALID_ARG, "lse must be a contiguous fp32 CUDA tensor")
    dtype = ATTN_DTYPE_F16 if q.dtype == torch.float16 else ATTN_DTYPE_BF16
    if scale is None:
        scale = 1.0 / (D ** 0.5)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(attn_bwd_workspace_size(B, Sq, Skv, Hq, Hkv, D), dtype=torch.uint8,
                                device=q.device)
    st = attn_bwd_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Sq, Skv, Hq,
                      Hkv, D, int(causal), float(scale), dtype, workspace.data_ptr(),
                      workspace.numel(), _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd")
    return dq, dk, dv


def attn_last_device_status() -> int:
    """Wait for all work on the current device, then return (and clear) the
    kernels' device status word."""
    return int(load_library().attn_last_device_status())


def attn_check_device_status(stream=None) -> int:
    """Synchronise ``stream`` and return (then clear) the kernels' device status word."""
    return int(load_library().attn_check_device_status(_stream_handle(stream)))


def attn_kernel_launches() -> int:
    """Number of kernels libattn has launched in this process."""
    return int(load_library().attn_kernel_launches())


def attn_debug_wait_timeout(poll_limit: int, stream=None) -> int:
    """Launch the bounded-wait self-test kernel (an mbarrier nothing arrives on)."""
    return int(load_library().attn_debug_wait_timeout(int(poll_limit), _stream_handle(stream)))


ATTN_UNIT_RATES = 8
UNIT_RATE_NAMES = ("mma_ss_n128", "mma_ts_n128", "mma_ss_n256", "mma_ss_n64", "mma_ts_n64",
                   "ex2_cycles_per_warp_instr", "ex2_per_cycle_per_sm", "sms")


def attn_debug_unit_rates(stream=None) -> dict:
    """Measured issue rates (diagnostic): SM clock cycles per tcgen05 MMA
    (M = 128, K = 16) for the operand sources and N the kernels use, cycles per
    warp-wide ex2 on one SM sub-partition, ex2 per cycle per SM, SMs measured."""
    out = (ctypes.c_double * ATTN_UNIT_RATES)()
    st = load_library().attn_debug_unit_rates(out, ATTN_UNIT_RATES, _stream_handle(stream))
    if st != ATTN_OK:
        raise AttnError(st, "attn_debug_unit_rates")
    return dict(zip(UNIT_RATE_NAMES, list(out)))


def attn_debug_unit_schedule(B: int, Sq: int, Skv: int, Hq: int, Hkv: int, D: int, causal: int, sms: int):
    """The forward's unit table for a shape on `sms` SMs (host only): (cta_begin,
    units) as lists, or None when the snake order is used instead."""
    grid_cap, cap = 257, 1 << 16
    cta_begin = (ctypes.c_int * grid_cap)()
    units = (ctypes.c_int * cap)()
    n = ctypes.c_int(-1)
    st = load_library().attn_debug_unit_schedule(int(B), int(Sq), int(Skv), int(Hq), int(Hkv), int(D), int(causal),
                                                 int(sms), cta_begin, units, cap, ctypes.byref(n))
    if st != ATTN_OK:
        raise AttnError(st, "attn_debug_unit_schedule")
    if n.value == 0:
        return None
    grid = min(sms, n.value)
    return list(cta_begin[:grid + 1]), list(units[:n.value])
