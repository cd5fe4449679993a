"""CPU oracle for the fused-chain hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference leg
may import this package.  The product path (``epilogue_chains_gb300``) never imports it, and it
never imports the product path: the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, single thread, ``-O2 -ffp-contract=off``, so every
float expression rounds where it is written).  This module only compiles that file with gcc,
loads it with ctypes and marshals numpy arrays.  Each C function cites the passage of the pages it
follows; the -m "not gpu" tests pin every function against closed forms, printed values,
invariants and brute force on tiny inputs.

Parity status of each function:
  chain, affine_closed_form, rmsnorm, causal_softmax, causal_softmax_unfused, gemm_epilogue,
  gelu, add_rmsnorm, silu, silu_mul, attention: pinned (tests/test_oracle_pins.py).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-Wall"]

_lock = threading.Lock()
_lib = None

DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2}


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so with gcc (no-op when up to date)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P, I64, I32, F32, F64, U32 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                      ctypes.c_float, ctypes.c_double, ctypes.c_uint32)
        sig = {
            "orc_round_half": ([F64], F64), "orc_round_bf16": ([F64], F64),
            "orc_round_f32": ([F64], F64),
            "orc_half_bits": ([F64], ctypes.c_uint16), "orc_bf16_bits": ([F64], ctypes.c_uint16),
            "orc_half_value": ([ctypes.c_uint16], F64), "orc_bf16_value": ([ctypes.c_uint16], F64),
            "orc_chain": ([P, P, P, I32, P, P, I64, I32], None),
            "orc_affine_closed_form": ([P, P, I64, I32, F32, F32], None),
            "orc_rmsnorm": ([P, P, P, I64, I64, F64], None),
            "orc_causal_softmax": ([P, P, I64, I64, F64, I32], None),
            "orc_causal_softmax_unfused": ([P, P, I64, I64, F64, I32], None),
            "orc_gemm_epilogue": ([P, P, P, P, P, I64, I64, I64, U32, P, I64], None),
            "orc_gelu": ([F64], F64),
            "orc_add_rmsnorm": ([P, P, P, P, P, I64, I64, F64], None),
            "orc_silu": ([F64], F64),
            "orc_silu_mul": ([P, P, I64, P, I64, I64, I32, I32], None),
            "orc_attention": ([P, P, P, P, I64, I64, I64, F64, P, I64], None),
            "orc_version": ([], I32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- scalar conversions
def round_half(v: float) -> float:
    return _load().orc_round_half(float(v))


def round_bf16(v: float) -> float:
    return _load().orc_round_bf16(float(v))


def half_bits(v: float) -> int:
    return int(_load().orc_half_bits(float(v)))


def bf16_bits(v: float) -> int:
    return int(_load().orc_bf16_bits(float(v)))


def half_value(h: int) -> float:
    return _load().orc_half_value(int(h))


def bf16_value(h: int) -> float:
    return _load().orc_bf16_value(int(h))


def gelu(v: float) -> float:
    return _load().orc_gelu(float(v))


# ---------------------------------------------------------------- the hot-path oracles
def chain(relu, a, b, x: np.ndarray, dtype: str = "f32") -> np.ndarray:
    """Pointwise chain y = f_{K-1}(...f_0(x)), f_s(v) = ReLU?(fl32(fl32(a_s v) + b_s)).

    ``x`` is float32 for dtype "f32", else uint16 bit patterns of fp16/bf16."""
    relu = _c(relu, np.int32)
    a = _c(a, np.float32)
    b = _c(b, np.float32)
    K = int(a.size)
    assert relu.size == K and b.size == K
    x = _c(x, np.float32 if dtype == "f32" else np.uint16)
    y = np.empty_like(x)
    _load().orc_chain(_ptr(relu), _ptr(a), _ptr(b), K, _ptr(x), _ptr(y), x.size,
                      DTYPE_CODES[dtype])
    return y


def affine_closed_form(x: np.ndarray, K: int, A: float, B: float) -> np.ndarray:
    """Closed form A^K x + B (A^K - 1)/(A - 1) in double (A, B taken as fp32 constants)."""
    x = _c(x, np.float32)
    y = np.empty(x.shape, dtype=np.float64)
    _load().orc_affine_closed_form(_ptr(x), _ptr(y), x.size, int(K), float(A), float(B))
    return y


def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    x = _c(x, np.float32)
    w = _c(w, np.float32)
    rows, hidden = x.shape
    assert w.shape == (hidden,)
    y = np.empty_like(x)
    _load().orc_rmsnorm(_ptr(x), _ptr(w), _ptr(y), rows, hidden, float(eps))
    return y


def causal_softmax(s_bits: np.ndarray, scale: float, out: str = "bf16",
                   unfused: bool = False) -> np.ndarray:
    """s_bits: uint16 bf16 patterns [BH, S, S] (or [S, S]).  Returns uint16 bf16 patterns
    (out="bf16") or float32 (out="f32") of the same shape."""
    s_bits = _c(s_bits, np.uint16)
    shape = s_bits.shape
    S = shape[-1]
    assert shape[-2] == S
    BH = s_bits.size // (S * S)
    p = np.empty(shape, dtype=np.uint16 if out == "bf16" else np.float32)
    fn = _load().orc_causal_softmax_unfused if unfused else _load().orc_causal_softmax
    fn(_ptr(s_bits), _ptr(p), BH, S, float(scale), DTYPE_CODES[out])
    return p


def gemm_epilogue(A: np.ndarray, B: np.ndarray, bias: np.ndarray, R: np.ndarray,
                  cut_mask: int = 0, rows=None) -> np.ndarray:
    """A [M,K], B [K,N], bias [N], R [M,N] as uint16 fp16 patterns.  Returns uint16 fp16
    patterns of Y restricted to ``rows`` ([len(rows), N]) or all of Y ([M, N])."""
    A = _c(A, np.uint16)
    B = _c(B, np.uint16)
    bias = _c(bias, np.uint16)
    R = _c(R, np.uint16)
    M, K = A.shape
    K2, N = B.shape
    assert K == K2 and bias.shape == (N,) and R.shape == (M, N)
    if rows is None:
        Y = np.empty((M, N), dtype=np.uint16)
        _load().orc_gemm_epilogue(_ptr(A), _ptr(B), _ptr(bias), _ptr(R), _ptr(Y), M, N, K,
                                  int(cut_mask), None, 0)
    else:
        rows = _c(rows, np.int64)
        assert rows.min() >= 0 and rows.max() < M
        Y = np.empty((rows.size, N), dtype=np.uint16)
        _load().orc_gemm_epilogue(_ptr(A), _ptr(B), _ptr(bias), _ptr(R), _ptr(Y), M, N, K,
                                  int(cut_mask), _ptr(rows), rows.size)
    return Y


def add_rmsnorm(x: np.ndarray, r: np.ndarray, w: np.ndarray, eps: float):
    """Residual add + RMSNorm over rows: h = fl32(x + r); y = RMSNorm(h) * w.  Returns (h, y)."""
    x = _c(x, np.float32)
    r = _c(r, np.float32)
    w = _c(w, np.float32)
    rows, hidden = x.shape
    assert r.shape == x.shape and w.size == hidden
    h = np.empty_like(x)
    y = np.empty_like(x)
    _load().orc_add_rmsnorm(_ptr(x), _ptr(r), _ptr(w), _ptr(h), _ptr(y), rows, hidden, float(eps))
    return h, y


def silu(v: float) -> float:
    return _load().orc_silu(float(v))


def silu_mul(g: np.ndarray, u: np.ndarray, dtype: str = "bf16", unfused: bool = False) -> np.ndarray:
    """y = SiLU(g) * u element-wise over two [rows, cols] arrays (float32 for "f32", else uint16
    bit patterns of fp16/bf16).  Returns y [rows, cols] in the storage type."""
    edt = np.float32 if dtype == "f32" else np.uint16
    g = _c(g, edt)
    u = _c(u, edt)
    assert g.shape == u.shape and g.ndim == 2
    rows, cols = g.shape
    y = np.empty((rows, cols), dtype=edt)
    _load().orc_silu_mul(_ptr(g), _ptr(u), cols, _ptr(y), rows, cols, DTYPE_CODES[dtype],
                         1 if unfused else 0)
    return y


def silu_mul_merged(gu: np.ndarray, dtype: str = "bf16", unfused: bool = False) -> np.ndarray:
    """The same on one merged gate/up output [rows, 2 cols]: gate = gu[:, :cols], up =
    gu[:, cols:], both read with row stride 2 cols."""
    edt = np.float32 if dtype == "f32" else np.uint16
    gu = _c(gu, edt)
    rows, ld = gu.shape
    assert ld % 2 == 0
    cols = ld // 2
    flat = gu.reshape(-1)
    y = np.empty((rows, cols), dtype=edt)
    _load().orc_silu_mul(_ptr(flat), _ptr(flat[cols:]), ld, _ptr(y), rows, cols,
                         DTYPE_CODES[dtype], 1 if unfused else 0)
    return y


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, rows=None) -> np.ndarray:
    """Causal attention o = softmax(scale q k^T, j <= i) v per slice; q, k, v uint16 bf16 bit
    patterns [BH, S, D] (or [S, D]).  rows: optional query rows of every slice.  Returns uint16
    bf16 patterns [BH, S or len(rows), D]."""
    q = _c(q, np.uint16)
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    squeeze = q.ndim == 2
    if squeeze:
        q, k, v = q[None], k[None], v[None]
    BH, S, D = q.shape
    assert k.shape == q.shape and v.shape == q.shape
    if rows is None:
        o = np.empty((BH, S, D), np.uint16)
        _load().orc_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(o), BH, S, D, float(scale), None, 0)
    else:
        r = _c(rows, np.int64)
        assert r.ndim == 1 and (r.size == 0 or (r.min() >= 0 and r.max() < S))
        o = np.empty((BH, r.size, D), np.uint16)
        _load().orc_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(o), BH, S, D, float(scale), _ptr(r),
                              r.size)
    return o[0] if squeeze else o
