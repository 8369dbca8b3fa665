"""ctypes wrapper around the C oracle (oracle/tffn_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference arm of ``bench.py``; never by the library under
``transformer_ffn_gb300/``.  Arrays are numpy: bf16 tensors travel as uint16
bit patterns, logits as float32, results come back as float64.
"""
import ctypes

import numpy as np

from . import build_oracle

ACT_NONE, ACT_RELU, ACT_GELU_TANH, ACT_SILU = 0, 1, 2, 3

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = build_oracle.build()
        L = ctypes.CDLL(path)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64p = ctypes.POINTER(ctypes.c_int64)
        i32p = ctypes.POINTER(ctypes.c_int32)
        f32p = ctypes.POINTER(ctypes.c_float)
        i64 = ctypes.c_int64
        L.tffn_oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.tffn_oracle_bf16_to_f64.restype = ctypes.c_double
        L.tffn_oracle_f64_to_bf16.argtypes = [ctypes.c_double]
        L.tffn_oracle_f64_to_bf16.restype = ctypes.c_uint16
        L.tffn_oracle_act.argtypes = [ctypes.c_int, ctypes.c_double]
        L.tffn_oracle_act.restype = ctypes.c_double
        L.tffn_oracle_ffn.argtypes = [u16p, u16p, u16p, u16p, u16p, ctypes.c_int,
                                      ctypes.c_int, i64, i64, i64, i64, i64p, i64,
                                      ctypes.c_int, f64p, u16p]
        L.tffn_oracle_ffn.restype = ctypes.c_int
        L.tffn_oracle_glu_ffn.argtypes = [u16p, u16p, u16p, u16p, ctypes.c_int, i64, i64, i64,
                                          i64, i64p, i64, ctypes.c_int, f64p, u16p]
        L.tffn_oracle_glu_ffn.restype = ctypes.c_int
        L.tffn_oracle_moe_route.argtypes = [f32p, i64, ctypes.c_int, ctypes.c_int,
                                            i32p, f64p]
        L.tffn_oracle_moe_route.restype = ctypes.c_int
        L.tffn_oracle_moe_permute.argtypes = [i32p, i64, ctypes.c_int, ctypes.c_int,
                                              i32p, i32p]
        L.tffn_oracle_moe_permute.restype = ctypes.c_int
        vpp = ctypes.POINTER(ctypes.c_void_p)
        L.tffn_oracle_moe_ffn.argtypes = [u16p, f32p, ctypes.c_int, vpp, vpp, vpp, vpp,
                                          i64, i64, i64, i64, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, i64p, i64, f64p]
        L.tffn_oracle_moe_ffn.restype = ctypes.c_int
        L.tffn_oracle_moe_glu_ffn.argtypes = [u16p, f32p, ctypes.c_int, vpp, vpp, vpp, i64, i64, i64, i64,
                                              ctypes.c_int, ctypes.c_int, i64p, i64, f64p]
        L.tffn_oracle_moe_glu_ffn.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 tensors are passed as uint16 bit patterns")
    return a


def bf16_to_f64(h: int) -> float:
    return lib().tffn_oracle_bf16_to_f64(int(h))


def f64_to_bf16(x: float) -> int:
    return lib().tffn_oracle_f64_to_bf16(float(x))


def act(kind: int, x: float) -> float:
    return lib().tffn_oracle_act(int(kind), float(x))


def ffn(X, W1, b1, W2, b2, act1, act2, rows=None, round_h=True, want_h=False):
    """Y (float64, len(rows) x P) of Y = act2(act1(X W1 + b1) W2 + b2)."""
    X, W1, W2 = _u16(X), _u16(W1), _u16(W2)
    b1 = None if b1 is None else _u16(b1)
    b2 = None if b2 is None else _u16(b2)
    M, N = X.shape
    N2, O = W1.shape
    O2, P = W2.shape
    assert N == N2 and O == O2
    if rows is None:
        r = None
        nrows = M
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = r.shape[0]
    Y = np.empty((nrows, P), dtype=np.float64)
    H = np.empty((nrows, O), dtype=np.uint16) if want_h else None
    rc = lib().tffn_oracle_ffn(_ptr(X, ctypes.c_uint16), _ptr(W1, ctypes.c_uint16),
                               _ptr(b1, ctypes.c_uint16), _ptr(W2, ctypes.c_uint16),
                               _ptr(b2, ctypes.c_uint16), int(act1), int(act2),
                               M, N, O, P, _ptr(r, ctypes.c_int64), nrows,
                               1 if round_h else 0, _ptr(Y, ctypes.c_double),
                               _ptr(H, ctypes.c_uint16))
    if rc != 0:
        raise RuntimeError(f"oracle ffn failed: {rc}")
    return (Y, H) if want_h else Y


def glu_ffn(X, W1, W3, W2, act=ACT_SILU, rows=None, round_h=True, want_h=False):
    """Y (float64, len(rows) x P) of the gated FFN Y = (act(X W1) * (X W3)) W2."""
    X, W1, W3, W2 = _u16(X), _u16(W1), _u16(W3), _u16(W2)
    M, N = X.shape
    N2, O = W1.shape
    O2, P = W2.shape
    assert N == N2 and O == O2 and W3.shape == W1.shape
    if rows is None:
        r = None
        nrows = M
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = r.shape[0]
    Y = np.empty((nrows, P), dtype=np.float64)
    H = np.empty((nrows, O), dtype=np.uint16) if want_h else None
    rc = lib().tffn_oracle_glu_ffn(_ptr(X, ctypes.c_uint16), _ptr(W1, ctypes.c_uint16),
                                   _ptr(W3, ctypes.c_uint16), _ptr(W2, ctypes.c_uint16), int(act),
                                   M, N, O, P, _ptr(r, ctypes.c_int64), nrows,
                                   1 if round_h else 0, _ptr(Y, ctypes.c_double),
                                   _ptr(H, ctypes.c_uint16))
    if rc != 0:
        raise RuntimeError(f"oracle glu_ffn failed: {rc}")
    return (Y, H) if want_h else Y


def moe_route(logits, k):
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    rc = lib().tffn_oracle_moe_route(_ptr(logits, ctypes.c_float), T, E, k,
                                     _ptr(idx, ctypes.c_int32), _ptr(w, ctypes.c_double))
    if rc != 0:
        raise RuntimeError(f"oracle moe_route failed: {rc}")
    return idx, w


def moe_permute(topk_idx, E):
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, k = topk_idx.shape
    perm = np.empty(T * k, dtype=np.int32)
    offs = np.empty(E + 1, dtype=np.int32)
    rc = lib().tffn_oracle_moe_permute(_ptr(topk_idx, ctypes.c_int32), T, E, k,
                                       _ptr(perm, ctypes.c_int32), _ptr(offs, ctypes.c_int32))
    if rc != 0:
        raise RuntimeError(f"oracle moe_permute failed: {rc}")
    return perm, offs


def moe_ffn(X, logits, top_k, W1s, b1s, W2s, b2s, act1, act2, tokens=None):
    """Y (float64, len(tokens) x P) of the routed, gate-weighted expert FFNs."""
    X = _u16(X)
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, N = X.shape
    E = len(W1s)
    W1s = [_u16(w) for w in W1s]
    W2s = [_u16(w) for w in W2s]
    b1s = None if b1s is None else [_u16(b) for b in b1s]
    b2s = None if b2s is None else [_u16(b) for b in b2s]
    O = W1s[0].shape[1]
    P = W2s[0].shape[1]

    def arr(lst):
        if lst is None:
            return None
        a = (ctypes.c_void_p * E)(*[x.ctypes.data for x in lst])
        return ctypes.cast(a, ctypes.POINTER(ctypes.c_void_p)), a

    a1, a2, a3, a4 = arr(W1s), arr(b1s), arr(W2s), arr(b2s)
    if tokens is None:
        tk, ntok = None, T
    else:
        tk = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
        ntok = tk.shape[0]
    Y = np.empty((ntok, P), dtype=np.float64)
    rc = lib().tffn_oracle_moe_ffn(_ptr(X, ctypes.c_uint16), _ptr(logits, ctypes.c_float),
                                   int(top_k), a1[0], a2[0] if a2 else None, a3[0],
                                   a4[0] if a4 else None, T, N, O, P, E, int(act1),
                                   int(act2), _ptr(tk, ctypes.c_int64), ntok,
                                   _ptr(Y, ctypes.c_double))
    if rc != 0:
        raise RuntimeError(f"oracle moe_ffn failed: {rc}")
    return Y


def moe_glu_ffn(X, logits, top_k, W1s, W3s, W2s, act=ACT_SILU, tokens=None):
    """Y (float64, len(tokens) x P) of the routed, gate-weighted gated experts."""
    X = _u16(X)
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, N = X.shape
    E = len(W1s)
    W1s = [_u16(w) for w in W1s]
    W3s = [_u16(w) for w in W3s]
    W2s = [_u16(w) for w in W2s]
    O = W1s[0].shape[1]
    P = W2s[0].shape[1]

    def arr(lst):
        a = (ctypes.c_void_p * E)(*[x.ctypes.data for x in lst])
        return ctypes.cast(a, ctypes.POINTER(ctypes.c_void_p)), a

    a1, a3, a2 = arr(W1s), arr(W3s), arr(W2s)
    if tokens is None:
        tk, ntok = None, T
    else:
        tk = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
        ntok = tk.shape[0]
    Y = np.empty((ntok, P), dtype=np.float64)
    rc = lib().tffn_oracle_moe_glu_ffn(_ptr(X, ctypes.c_uint16), _ptr(logits, ctypes.c_float), int(top_k),
                                       a1[0], a3[0], a2[0], T, N, O, P, E, int(act), _ptr(tk, ctypes.c_int64),
                                       ntok, _ptr(Y, ctypes.c_double))
    if rc != 0:
        raise RuntimeError(f"oracle moe_glu_ffn failed: {rc}")
    return Y
