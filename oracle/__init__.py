"""fp64 CPU oracle for the attention forward pass -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The product
path (the CUDA library and its Python binding) never imports it and shares no
code with it.

Contents
  * ``attn_rows`` / ``attn_full`` -- the C oracle (``oracle.c``): textbook
    two-pass softmax(scale * Q K^T [+ mask]) V in fp64, natural-log LSE.
    Definition: the Pallas page (``attention_mgpu.py``), ``attention_reference``.
  * ``partial_triple`` / ``merge_triples`` -- un-normalised (m, l, o) of a row
    over a key range, and the merge rule of the kernbench page
    (``_gqa_attention_prefill_short.py``, ``_merge_running``).
  * ``attn_bwd`` / ``attn_bwd_dq_rows`` / ``attn_bwd_dkv_keys`` -- the C
    oracle's gradients dq, dk, dv of sum(dO * o) in fp64: the plain
    vector-Jacobian product of the definition (the Pallas page's
    ``_attention_bwd``), for every element or for sampled rows / keys; on
    request with delta_i = sum_d dO * o taken from a given 16-bit forward
    output, as that page's backward kernel takes it from its stored ``out``.
  * ``round_bf16`` -- exact round-to-nearest-even of fp64 values to bf16, the
    comparison value for the bf16 output.
  * ``twin`` (module ``oracle.twin``) -- an independent numpy fp64 restatement
    for tiny shapes, used to cross-check the C oracle by brute force.

Parity pins (tests/test_oracle_pins.py) tie every function here to something
other than itself: closed forms, library routines, invariants, brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` with gcc + OpenMP (no -ffast-math)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fno-fast-math", "-fopenmp", "-shared", "-fPIC", "-std=c11",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def configure(lib):
    """Declare the C signatures on a loaded oracle library."""
    P = ctypes.c_void_p
    L = ctypes.c_long
    lib.oracle_attn_rows.argtypes = [P, P, P, L, L, L, L, L, L, ctypes.c_int,
                                     ctypes.c_double, ctypes.c_int, L, P, P, P]
    lib.oracle_attn_rows.restype = ctypes.c_int
    lib.oracle_attn_fwd.argtypes = [P, P, P, L, L, L, L, L, L, ctypes.c_int,
                                    ctypes.c_double, ctypes.c_int, P, P]
    lib.oracle_attn_fwd.restype = ctypes.c_int
    lib.oracle_partial_triple.argtypes = [P, P, P, L, L, L, L, L, L, ctypes.c_int,
                                          ctypes.c_double, ctypes.c_int, L, L, L, L, L, P, P, P]
    lib.oracle_partial_triple.restype = ctypes.c_int
    lib.oracle_attn_bwd.argtypes = [P, P, P, P, P, L, L, L, L, L, L, ctypes.c_int,
                                    ctypes.c_double, ctypes.c_int, P, P, P]
    lib.oracle_attn_bwd.restype = ctypes.c_int
    lib.oracle_attn_bwd_dq_rows.argtypes = [P, P, P, P, P, L, L, L, L, L, L, ctypes.c_int,
                                            ctypes.c_double, ctypes.c_int, L, P, P]
    lib.oracle_attn_bwd_dq_rows.restype = ctypes.c_int
    lib.oracle_attn_bwd_dkv_keys.argtypes = [P, P, P, P, P, L, L, L, L, L, L, ctypes.c_int,
                                             ctypes.c_double, ctypes.c_int, L, P, P, P]
    lib.oracle_attn_bwd_dkv_keys.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = configure(ctypes.CDLL(build()))
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _check_inputs(q, k, v):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != np.uint16 or t.ndim != 4 or not t.flags.c_contiguous:
            raise ValueError(f"{name} must be a C-contiguous 4-d uint16 array of bf16 bits")
    B, Sq, Hq, D = q.shape
    Bk, Skv, Hkv, Dk = k.shape
    if v.shape != k.shape or Bk != B or Dk != D:
        raise ValueError("k and v must be [B, Skv, Hkv, D] with q's B and D")
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    return B, Sq, Skv, Hq, Hkv, D


def num_threads() -> int:
    """OpenMP threads the C oracle uses."""
    return int(_load().oracle_num_threads())


def attn_rows(q, k, v, rows, causal: int, scale: float, f16: bool = False):
    """fp64 o (len(rows) x D) and lse (len(rows)) for the listed (b, h, i) rows.
    causal: 0 none, 1 bottom-right (j <= i + Skv - Sq), 2 top-left (j <= i: the
    Pallas page's `attention_reference` mask, `q_idx >= kv_idx`, for any Sq, Skv).
    f16: the uint16 inputs are IEEE binary16 bit patterns instead of bf16."""
    B, Sq, Skv, Hq, Hkv, D = _check_inputs(q, k, v)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    o = np.zeros((rows.shape[0], D), dtype=np.float64)
    lse = np.zeros(rows.shape[0], dtype=np.float64)
    rc = _load().oracle_attn_rows(_ptr(q), _ptr(k), _ptr(v), B, Sq, Skv, Hq, Hkv, D,
                                  int(causal), float(scale), int(bool(f16)), rows.shape[0],
                                  _ptr(rows), _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_attn_rows rejected its arguments")
    return o, lse


def attn_full(q, k, v, causal: int, scale: float, f16: bool = False):
    """fp64 o [B,Sq,Hq,D] and lse [B,Hq,Sq] for every row (f16: binary16 inputs)."""
    B, Sq, Skv, Hq, Hkv, D = _check_inputs(q, k, v)
    o = np.zeros((B, Sq, Hq, D), dtype=np.float64)
    lse = np.zeros((B, Hq, Sq), dtype=np.float64)
    rc = _load().oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), B, Sq, Skv, Hq, Hkv, D,
                                 int(causal), float(scale), int(bool(f16)), _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_attn_fwd rejected its arguments")
    return o, lse


def partial_triple(q, k, v, causal: int, scale: float, b: int, h: int, i: int,
                   j_lo: int, j_hi: int, f16: bool = False):
    """Un-normalised (m, l, o) of row (b, h, i) over keys [j_lo, j_hi)."""
    B, Sq, Skv, Hq, Hkv, D = _check_inputs(q, k, v)
    m = np.zeros(1, dtype=np.float64)
    l = np.zeros(1, dtype=np.float64)
    o = np.zeros(D, dtype=np.float64)
    rc = _load().oracle_partial_triple(_ptr(q), _ptr(k), _ptr(v), B, Sq, Skv, Hq, Hkv, D,
                                       int(causal), float(scale), int(bool(f16)), b, h, i,
                                       j_lo, j_hi,
                                       _ptr(m), _ptr(l), _ptr(o))
    if rc != 0:
        raise ValueError("oracle_partial_triple rejected its arguments")
    return float(m[0]), float(l[0]), o


def _check_do(q, do):
    if do.dtype != np.uint16 or do.shape != q.shape or not do.flags.c_contiguous:
        raise ValueError("do must be a C-contiguous uint16 array shaped like q")


def _delta_arg(q, do, o, delta, f16):
    """The delta_i the C entry points are given: None (the exact sum_j p_ij dp_ij),
    an explicit fp64 [B, Hq, Sq] array, or sum_d do * o over a 16-bit forward
    output o in q's layout and format (the page's backward takes delta from its
    stored `out`)."""
    B, Sq, Hq, D = q.shape
    if o is not None:
        if delta is not None:
            raise ValueError("pass o or delta, not both")
        if o.dtype != np.uint16 or o.shape != q.shape:
            raise ValueError("o must be a uint16 array of 16-bit patterns with q's shape")
        w = f16_bits_to_f64 if f16 else bf16_bits_to_f64
        delta = np.einsum("bihd,bihd->bhi", w(do), w(o))
    if delta is None:
        return None
    delta = np.ascontiguousarray(np.asarray(delta, dtype=np.float64))
    if delta.shape != (B, Hq, Sq):
        raise ValueError("delta must be [B, Hq, Sq]")
    return delta


def attn_bwd(q, k, v, do, causal: int, scale: float, f16: bool = False, o=None, delta=None):
    """fp64 (dq [B,Sq,Hq,D], dk [B,Skv,Hkv,D], dv [B,Skv,Hkv,D]): the gradient of
    sum(do * o) with o the attention output; do has q's shape and 16-bit format.
    By default delta_i = sum_j p_ij dp_ij (exact).  o: a 16-bit forward output
    (q's layout and format) to take delta_i = sum_d do * o from, as a backward
    given the stored output does; delta: explicit fp64 [B, Hq, Sq] values."""
    B, Sq, Skv, Hq, Hkv, D = _check_inputs(q, k, v)
    _check_do(q, do)
    dl = _delta_arg(q, do, o, delta, f16)
    dq = np.zeros((B, Sq, Hq, D), dtype=np.float64)
    dk = np.zeros((B, Skv, Hkv, D), dtype=np.float64)
    dv = np.zeros((B, Skv, Hkv, D), dtype=np.float64)
    rc = _load().oracle_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do),
                                 None if dl is None else _ptr(dl), B, Sq, Skv, Hq, Hkv, D,
                                 int(causal), float(scale), int(bool(f16)), _ptr(dq), _ptr(dk),
                                 _ptr(dv))
    if rc != 0:
        raise ValueError("oracle_attn_bwd rejected its arguments")
    return dq, dk, dv


def attn_bwd_dq_rows(q, k, v, do, rows, causal: int, scale: float, f16: bool = False, o=None,
                     delta=None):
    """fp64 dq (len(rows) x D) of the listed (b, h, i) rows; o, delta as for attn_bwd."""
    B, Sq, Skv, Hq, Hkv, D = _check_inputs(q, k, v)
    _check_do(q, do)
    dl = _delta_arg(q, do, o, delta, f16)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    dq = np.zeros((rows.shape[0], D), dtype=np.float64)
    rc = _load().oracle_attn_bwd_dq_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(do),
                                         None if dl is None else _ptr(dl), B, Sq, Skv, Hq,
                                         Hkv, D, int(causal), float(scale), int(bool(f16)),
                                         rows.shape[0], _ptr(rows), _ptr(dq))
    if rc != 0:
        raise ValueError("oracle_attn_bwd_dq_rows rejected its arguments")
    return dq


def attn_bwd_dkv_keys(q, k, v, do, keys, causal: int, scale: float, f16: bool = False, o=None,
                      delta=None):
    """fp64 (dk, dv), each len(keys) x D, of the listed (b, g, j) keys (g: key/value
    head); o, delta as for attn_bwd."""
    B, Sq, Skv, Hq, Hkv, D = _check_inputs(q, k, v)
    _check_do(q, do)
    dl = _delta_arg(q, do, o, delta, f16)
    keys = np.ascontiguousarray(np.asarray(keys, dtype=np.int64).reshape(-1, 3))
    dk = np.zeros((keys.shape[0], D), dtype=np.float64)
    dv = np.zeros((keys.shape[0], D), dtype=np.float64)
    rc = _load().oracle_attn_bwd_dkv_keys(_ptr(q), _ptr(k), _ptr(v), _ptr(do),
                                          None if dl is None else _ptr(dl), B, Sq, Skv, Hq,
                                          Hkv, D, int(causal), float(scale), int(bool(f16)),
                                          keys.shape[0], _ptr(keys), _ptr(dk), _ptr(dv))
    if rc != 0:
        raise ValueError("oracle_attn_bwd_dkv_keys rejected its arguments")
    return dk, dv


def merge_triples(t1, t2):
    """Merge two un-normalised (m, l, o) triples over disjoint key sets.

    The kernbench page's ``_merge_running``: m = max(m1, m2),
    l = l1 e^(m1-m) + l2 e^(m2-m), o = o1 e^(m1-m) + o2 e^(m2-m).
    An empty triple (m = -inf, l = 0) is the identity.
    """
    m1, l1, o1 = t1
    m2, l2, o2 = t2
    if m1 == -np.inf:
        return m2, l2, np.array(o2, dtype=np.float64)
    if m2 == -np.inf:
        return m1, l1, np.array(o1, dtype=np.float64)
    m = max(m1, m2)
    a1 = np.exp(m1 - m)
    a2 = np.exp(m2 - m)
    return m, l1 * a1 + l2 * a2, np.asarray(o1) * a1 + np.asarray(o2) * a2


def finish_triple(t):
    """(normalised o, lse) of a merged triple; o = 0, lse = -inf when nothing is visible."""
    m, l, o = t
    if l <= 0.0:
        return np.zeros_like(np.asarray(o, dtype=np.float64)), -np.inf
    return np.asarray(o) / l, m + np.log(l)


def round_bf16(x) -> np.ndarray:
    """Exact round-to-nearest-even of fp64 values to bf16 (returned as fp64).

    bf16 keeps 8 significant bits and fp32's exponent range.  The value is
    split as x = f * 2^e with 0.5 <= |f| < 1; f * 2^8 is rounded half-to-even;
    below the smallest normal (2^-126) the grid is fixed at 2^-133.
    Overflow past bf16's largest finite value goes to +-inf.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, dtype=np.float64, copy=True)
    finite = np.isfinite(x) & (x != 0.0)
    xf = x[finite]
    f, e = np.frexp(xf)
    normal = e >= -125  # |x| >= 2^-126  <=>  e - 1 >= -126
    r = np.empty_like(xf)
    r[normal] = np.ldexp(np.rint(np.ldexp(f[normal], 8)), e[normal] - 8)
    r[~normal] = np.ldexp(np.rint(np.ldexp(xf[~normal], 133)), -133)
    max_bf16 = float.fromhex("0x1.fep127")
    r[np.abs(r) > max_bf16] = np.copysign(np.inf, r[np.abs(r) > max_bf16])
    out[finite] = r
    return out


def round_f16(x) -> np.ndarray:
    """Exact round-to-nearest-even of fp64 values to IEEE binary16 (returned as fp64).

    binary16 keeps 11 significant bits; normal numbers start at 2^-14, below
    that the grid is fixed at 2^-24; past 65504 (plus half a step) values go to
    +-inf.  Same splitting as round_bf16: x = f * 2^e, 0.5 <= |f| < 1, f * 2^11
    rounded half-to-even.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, dtype=np.float64, copy=True)
    finite = np.isfinite(x) & (x != 0.0)
    xf = x[finite]
    f, e = np.frexp(xf)
    normal = e >= -13  # |x| >= 2^-14  <=>  e - 1 >= -14
    r = np.empty_like(xf)
    r[normal] = np.ldexp(np.rint(np.ldexp(f[normal], 11)), e[normal] - 11)
    r[~normal] = np.ldexp(np.rint(np.ldexp(xf[~normal], 24)), -24)
    r[np.abs(r) > 65504.0] = np.copysign(np.inf, r[np.abs(r) > 65504.0])
    out[finite] = r
    return out


def f16_bits_to_f64(bits) -> np.ndarray:
    """Widen IEEE binary16 bit patterns (uint16) to fp64 exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where(b >> 15, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    frac = (b & 0x3FF).astype(np.float64)
    mag = np.where(e == 0, np.ldexp(frac, -24), np.ldexp(frac + 1024.0, e - 25))
    mag = np.where(e == 31, np.where(frac > 0, np.nan, np.inf), mag)
    return sign * mag


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to fp64 exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)
