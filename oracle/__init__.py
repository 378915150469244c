"""Oracle for trellis-coded weight linear layers: a thin ctypes wrapper over
``trellis_oracle.c`` (plain C, fp64 sums, bit-by-bit window walk).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``trellis_coded_weight_gb300`` and its CUDA library) never imports it, and the
two share no code; only the seeded input generators feed both.

Every function below follows the pages' statement of the method; the C file's
header gives the passages.  Each function is pinned by the ``-m "not gpu"``
tests in ``tests/test_oracle_pins.py`` (worked examples under
``tests/golden/``, closed forms, invariants, library routines, brute force).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "trellis_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-Wall"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/_build/liboracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_P_U32 = ctypes.POINTER(ctypes.c_uint32)
_P_U16 = ctypes.POINTER(ctypes.c_uint16)
_P_I32 = ctypes.POINTER(ctypes.c_int32)
_P_I64 = ctypes.POINTER(ctypes.c_int64)
_P_F32 = ctypes.POINTER(ctypes.c_float)
_P_F64 = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.c_int64
_INT = ctypes.c_int


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            sig = {
                "or_geom_check": (_INT, [_INT, _INT, _INT, _I64, _I64]),
                "or_state": (ctypes.c_uint32, [_P_U32, _INT, _INT, _INT, _INT]),
                "or_code_y": (_INT, [ctypes.c_uint32]),
                "or_code_val": (ctypes.c_float, [_INT]),
                "or_lut": (None, [_INT, _P_I32, _P_F32]),
                "or_f16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
                "or_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
                "or_bf16_rne": (ctypes.c_uint16, [ctypes.c_float]),
                "or_bf16_rne_f64": (ctypes.c_uint16, [ctypes.c_double]),
                "or_decode_rows": (None, [_P_U32, _P_U16, _INT, _INT, _INT, _I64, _I64, _P_I64, _I64,
                                          _P_U32, _P_I32, _P_F32]),
                "or_expand_bf16": (None, [_P_U32, _P_U16, _INT, _INT, _INT, _I64, _I64, _P_I64, _I64, _P_U16]),
                "or_matvec_axis1": (None, [_P_U32, _P_U16, _P_U16, _INT, _INT, _INT, _INT, _I64, _I64,
                                           _P_I64, _I64, _P_F64, _P_F64]),
                "or_matvec_axis0": (None, [_P_U32, _P_U16, _P_U16, _INT, _INT, _INT, _INT, _I64, _I64,
                                           _P_I64, _I64, _P_F64, _P_F64]),
                "or_matvec_axis0_bf16w": (None, [_P_U32, _P_U16, _P_U16, _INT, _INT, _INT, _INT, _I64, _I64,
                                                 _P_I64, _I64, _P_F64, _P_F64]),
                "or_swiglu_bf16": (ctypes.c_uint16, [ctypes.c_uint16, ctypes.c_uint16]),
                "or_swiglu_bf16_many": (None, [_P_U16, _P_U16, _P_U16, _I64]),
                "or_gateup_sums": (None, [_P_U32, _P_U16, _P_U32, _P_U16, _P_U16, _INT, _INT, _INT, _INT,
                                          _I64, _I64, _P_I64, _I64, _P_F64, _P_F64, _P_F64, _P_F64]),
                "or_prefill": (None, [_P_U32, _P_U16, _P_U16, _INT, _INT, _INT, _INT, _I64, _I64,
                                      _P_I64, _I64, _P_F64, _P_F64]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _u32(a):
    return np.ascontiguousarray(a, dtype=np.uint32)


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


def _idx(idx, n):
    if idx is None:
        return np.arange(n, dtype=np.int64)
    return np.ascontiguousarray(np.asarray(idx, dtype=np.int64).reshape(-1))


def _geom(k, L, T, rows, cols):
    if _load().or_geom_check(k, L, T, rows, cols) != 0:
        raise ValueError(f"oracle: invalid geometry k={k} L={L} T={T} rows={rows} cols={cols}")


# ---------------------------------------------------------------- primitives

def geom_check(k, L, T, rows, cols) -> int:
    return int(_load().or_geom_check(k, L, T, rows, cols))


def state(block_words, T: int, k: int, L: int, t: int) -> int:
    """state_t of one packed block (its T*k/32 words)."""
    b = _u32(block_words)
    assert b.size == T * k // 32
    return int(_load().or_state(_ptr(b, ctypes.c_uint32), T, k, L, t))


def code_y(s: int) -> int:
    return int(_load().or_code_y(ctypes.c_uint32(s & 0xFFFFFFFF)))


def code_val(y: int) -> np.float32:
    return np.float32(_load().or_code_val(int(y)))


def lut(L: int):
    """(y, value) for every state s < 2^L."""
    n = 1 << L
    ys = np.empty(n, dtype=np.int32)
    vs = np.empty(n, dtype=np.float32)
    _load().or_lut(L, _ptr(ys, ctypes.c_int32), _ptr(vs, ctypes.c_float))
    return ys, vs


def f16_to_f32(h: int) -> np.float32:
    return np.float32(_load().or_f16_to_f32(int(h)))


def bf16_to_f32(b: int) -> np.float32:
    return np.float32(_load().or_bf16_to_f32(int(b)))


def bf16_rne(v: float) -> int:
    return int(_load().or_bf16_rne(float(np.float32(v))))


def bf16_rne_f64(v: float) -> int:
    return int(_load().or_bf16_rne_f64(float(v)))


def bf16_rne_f64_many(v) -> np.ndarray:
    f = _load().or_bf16_rne_f64
    a = np.asarray(v, dtype=np.float64).reshape(-1)
    return np.array([f(float(t)) for t in a], dtype=np.uint16).reshape(np.shape(v))


# ---------------------------------------------------------------- layers

def decode_rows(codes, scales, k, L, T, rows=None):
    """(states, y, fp32 matvec weights) of the selected stored rows: [n, cols] each."""
    codes, scales = _u32(codes), _u16(scales)
    R, cols = codes.shape[0], codes.shape[1] * 32 // k
    _geom(k, L, T, R, cols)
    idx = _idx(rows, R)
    st = np.empty((idx.size, cols), dtype=np.uint32)
    ys = np.empty((idx.size, cols), dtype=np.int32)
    ws = np.empty((idx.size, cols), dtype=np.float32)
    _load().or_decode_rows(_ptr(codes, ctypes.c_uint32), _ptr(scales, ctypes.c_uint16), k, L, T, R, cols,
                           _ptr(idx, ctypes.c_int64), idx.size, _ptr(st, ctypes.c_uint32),
                           _ptr(ys, ctypes.c_int32), _ptr(ws, ctypes.c_float))
    return st, ys, ws


def expand_bf16(codes, scales, k, L, T, rows=None) -> np.ndarray:
    """bf16 bits of the decoded stored matrix (selected rows): [n, cols]."""
    codes, scales = _u32(codes), _u16(scales)
    R, cols = codes.shape[0], codes.shape[1] * 32 // k
    _geom(k, L, T, R, cols)
    idx = _idx(rows, R)
    out = np.empty((idx.size, cols), dtype=np.uint16)
    _load().or_expand_bf16(_ptr(codes, ctypes.c_uint32), _ptr(scales, ctypes.c_uint16), k, L, T, R, cols,
                           _ptr(idx, ctypes.c_int64), idx.size, _ptr(out, ctypes.c_uint16))
    return out


def _mv(fn, codes, scales, x, k, L, T, idx_of, n_of):
    codes, scales, x = _u32(codes), _u16(scales), _u16(x)
    R, cols = codes.shape[0], codes.shape[1] * 32 // k
    _geom(k, L, T, R, cols)
    M = x.shape[0]
    idx = _idx(idx_of, n_of(R, cols))
    ref = np.empty((M, idx.size), dtype=np.float64)
    ab = np.empty((M, idx.size), dtype=np.float64)
    fn(_ptr(codes, ctypes.c_uint32), _ptr(scales, ctypes.c_uint16), _ptr(x, ctypes.c_uint16), M, k, L, T, R,
       cols, _ptr(idx, ctypes.c_int64), idx.size, _ptr(ref, ctypes.c_double), _ptr(ab, ctypes.c_double))
    return ref, ab


def matvec_axis1(codes, scales, x, k, L, T, rows=None):
    """(ref, absum) [M, n]: out[m, r] = sum_c w(r,c) x[m,c] in double."""
    assert np.shape(x)[1] == np.shape(codes)[1] * 32 // k
    return _mv(_load().or_matvec_axis1, codes, scales, x, k, L, T, rows, lambda R, C: R)


def matvec_axis0(codes, scales, x, k, L, T, cols=None):
    """(ref, absum) [M, n]: out[m, c] = sum_r w(r,c) x[m,r] in double (stored W^T)."""
    assert np.shape(x)[1] == np.shape(codes)[0]
    return _mv(_load().or_matvec_axis0, codes, scales, x, k, L, T, cols, lambda R, C: C)


def matvec_axis0_bf16w(codes, scales, x, k, L, T, cols=None):
    """Axis-0 matvec with bf16-rounded weights (the expand weights), in double."""
    assert np.shape(x)[1] == np.shape(codes)[0]
    return _mv(_load().or_matvec_axis0_bf16w, codes, scales, x, k, L, T, cols, lambda R, C: C)


def matvec_axis1_bf16w(codes, scales, x, k, L, T, rows=None):
    """Axis-1 matvec with bf16-rounded weights: the same sum as prefill()."""
    return prefill(codes, scales, x, k, L, T, rows)


def prefill(codes, scales, x, k, L, T, rows=None):
    """(ref, absum) [M, n]: out[m, r] = sum_c bf16 expand weight(r,c) x[m,c]."""
    assert np.shape(x)[1] == np.shape(codes)[1] * 32 // k
    return _mv(_load().or_prefill, codes, scales, x, k, L, T, rows, lambda R, C: R)


def gateup_sums(gcodes, gscales, ucodes, uscales, x, k, L, T, rows=None):
    """(gref, gabs, uref, uabs) [M, n] of the two axis-1 matvecs."""
    gcodes, ucodes = _u32(gcodes), _u32(ucodes)
    gscales, uscales, x = _u16(gscales), _u16(uscales), _u16(x)
    R, cols = gcodes.shape[0], gcodes.shape[1] * 32 // k
    _geom(k, L, T, R, cols)
    assert ucodes.shape == gcodes.shape and x.shape[1] == cols
    M = x.shape[0]
    idx = _idx(rows, R)
    outs = [np.empty((M, idx.size), dtype=np.float64) for _ in range(4)]
    _load().or_gateup_sums(_ptr(gcodes, ctypes.c_uint32), _ptr(gscales, ctypes.c_uint16),
                           _ptr(ucodes, ctypes.c_uint32), _ptr(uscales, ctypes.c_uint16),
                           _ptr(x, ctypes.c_uint16), M, k, L, T, R, cols, _ptr(idx, ctypes.c_int64), idx.size,
                           *[_ptr(o, ctypes.c_double) for o in outs])
    return tuple(outs)


def swiglu_bf16(g_bits, u_bits) -> np.ndarray:
    """The bf16 activation chain applied elementwise to bf16 gate/up bits."""
    g, u = _u16(g_bits), _u16(u_bits)
    assert g.shape == u.shape
    out = np.empty(g.shape, dtype=np.uint16)
    _load().or_swiglu_bf16_many(_ptr(g, ctypes.c_uint16), _ptr(u, ctypes.c_uint16), _ptr(out, ctypes.c_uint16),
                                g.size)
    return out
