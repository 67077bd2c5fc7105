"""CPU oracle for the decode linear layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library never does: it has no CPU
fallback, and this oracle shares no code with it.

The arithmetic of the linear layer lives in ``dl_oracle.c`` (plain C, IEEE
double, k ascending, explicit E4M3FN table); this module compiles it with the
host C compiler and marshals numpy arrays to it.  See the C file's header for
the definition and the passages of the pages each part follows.  The SwiGLU
epilogue (``silu``, ``swiglu``) is written here in float64 numpy on top of it.

Parity pins: e4m3 table (closed form, anchors, an independent decoder),
bf16 decode (all 65536 patterns), one-hot columns, scale = 1 blocks,
linearity, exact-rational brute force and the worked examples of
"Multi-GPU Inference and Serving at Scale" (Examples 2 and 3); SiLU closed
forms (sigma(ln 3) = 3/4), its odd-part identity and the gate/up pairing of
SwiGLU; see ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dl_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle_dl.so")
_lock = threading.Lock()
_lib = None

BF16 = 0
FP8_B128 = 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no fast-math) if it is missing or stale."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.dl_oracle_e4m3_table.argtypes = [ctypes.c_void_p]
            lib.dl_oracle_e4m3_table.restype = None
            lib.dl_oracle_bf16_values.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
            lib.dl_oracle_bf16_values.restype = None
            lib.dl_oracle_round_f32_to_bf16_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                                              ctypes.c_int64]
            lib.dl_oracle_round_f32_to_bf16_array.restype = None
            lib.dl_oracle_linear.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.dl_oracle_linear.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def e4m3_table() -> np.ndarray:
    """float64[256]: value of every E4M3FN code (NaN for 0x7F and 0xFF)."""
    out = np.empty(256, dtype=np.float64)
    _load().dl_oracle_e4m3_table(out.ctypes.data)
    return out


def bf16_values(bits) -> np.ndarray:
    """Exact float64 value of each bf16 bit pattern (uint16 array)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    _load().dl_oracle_bf16_values(b.ctypes.data, out.ctypes.data, b.size)
    return out


def round_to_bf16(values) -> np.ndarray:
    """binary32 -> bf16 bit patterns, round to nearest even (uint16 array)."""
    v = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().dl_oracle_round_f32_to_bf16_array(v.ctypes.data, out.ctypes.data, v.size)
    return out


def linear(dtype: int, x_bits, w, scales=None, bias_bits=None, *, rows=None,
           k_range=None, with_abs: bool = True, threads: int | None = None):
    """Reference y (float64 [M, n_rows]) and, optionally, A = sum_k |x w| (same shape).

    dtype   -- BF16 (w: uint16 bf16 bits [N, K]) or FP8_B128 (w: uint8 e4m3 codes
               [N, K], scales: float32 [ceil(N/128), ceil(K/128)]).
    x_bits  -- uint16 bf16 bits [M, K].
    bias_bits -- uint16 bf16 bits [N] or None (added once, after the sum).
    rows    -- optional int64 list of output rows n to compute (default: all).
    k_range -- optional (k_begin, k_end): sum only that slice of K (a partial).
    """
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    if x.ndim != 2:
        raise ValueError("x must be [M, K]")
    M, K = x.shape
    if dtype == BF16:
        wa = np.ascontiguousarray(w, dtype=np.uint16)
        sc = None
    elif dtype == FP8_B128:
        wa = np.ascontiguousarray(w, dtype=np.uint8)
        if scales is None:
            raise ValueError("FP8 needs scales")
        sc = np.ascontiguousarray(scales, dtype=np.float32)
    else:
        raise ValueError("dtype must be BF16 or FP8_B128")
    N = wa.shape[0]
    if wa.shape != (N, K):
        raise ValueError("w must be [N, K]")
    if sc is not None and sc.shape != ((N + 127) // 128, (K + 127) // 128):
        raise ValueError("scales must be [ceil(N/128), ceil(K/128)]")
    b = None if bias_bits is None else np.ascontiguousarray(bias_bits, dtype=np.uint16)
    if b is not None and b.shape != (N,):
        raise ValueError("bias must be [N]")
    r = None
    n_rows = N
    if rows is not None:
        r = np.ascontiguousarray(rows, dtype=np.int64)
        if r.size and (r.min() < 0 or r.max() >= N):
            raise ValueError("row index out of range")
        n_rows = r.size
    k0, k1 = (0, K) if k_range is None else k_range
    y = np.zeros((M, n_rows), dtype=np.float64)
    a = np.zeros((M, n_rows), dtype=np.float64) if with_abs else None
    rc = _load().dl_oracle_linear(dtype, M, N, K, x.ctypes.data, wa.ctypes.data, _ptr(sc),
                                  _ptr(b), int(k0), int(k1), _ptr(r), n_rows, y.ctypes.data,
                                  _ptr(a), threads or default_threads())
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return (y, a) if with_abs else y


def silu(g):
    """SiLU in float64: silu(g) = g * sigma(g) = g / (1 + e^-g).  e^-g overflows
    to inf for very negative g, which gives the correct limit -0."""
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def swiglu_rows(I: int):
    """Gate and up row indices of outputs 0..I-1 in the interleaved weight
    layout of the SwiGLU call: gate row 16 (j // 8) + j % 8, up row 8 further."""
    j = np.arange(I, dtype=np.int64)
    g = 16 * (j // 8) + j % 8
    return g, g + 8


def swiglu(dtype: int, x_bits, w, scales=None, bias_bits=None, *, outputs=None,
           threads: int | None = None):
    """SwiGLU reference for the interleaved gate_up weights w [N, K] (N % 16 == 0):
    y[m][j] = silu(g) * u, g and u the reference sums (+ bias) of the gate and up
    rows of output j ("Multi-GPU Inference and Serving at Scale", Example 3: the
    nonlinearity between the MLP's two matrices; SwiGLU being the variant real
    models use, in its usual SiLU-gated form).  Returns y, g, u, A_g, A_u as
    float64 [M, n_outputs] (A = sum_k |x w| of each row, the tolerance scale).
    outputs -- optional list of output columns j (default: all N / 2)."""
    N = np.asarray(w).shape[0]
    if N % 16:
        raise ValueError("SwiGLU weights need N % 16 == 0")
    gate, up = swiglu_rows(N // 2)
    if outputs is not None:
        sel = np.asarray(outputs, dtype=np.int64)
        gate, up = gate[sel], up[sel]
    g, ag = linear(dtype, x_bits, w, scales, bias_bits, rows=gate, threads=threads)
    u, au = linear(dtype, x_bits, w, scales, bias_bits, rows=up, threads=threads)
    return silu(g) * u, g, u, ag, au


def argmax_lowest(values):
    """Row-wise argmax of a [M, N] array: the lowest index n among the largest
    values, a NaN counting as larger than every number (the first NaN wins) and
    -0 equal to +0 -- greedy selection of the next token from the lm_head
    logits.  Per row: the first NaN if there is one, else the first index whose
    value equals the maximum (float64 comparisons, exact for fp32 inputs)."""
    v = np.asarray(values, dtype=np.float64)
    out = np.zeros(v.shape[0], dtype=np.int64)
    for m in range(v.shape[0]):
        nan = np.flatnonzero(np.isnan(v[m]))
        out[m] = nan[0] if nan.size else np.flatnonzero(v[m] == v[m].max())[0]
    return out
