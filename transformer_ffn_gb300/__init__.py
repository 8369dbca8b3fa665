"""GB300-native fused Transformer FFN and MoE-FFN.

Thin ctypes binding over the C ABI in include/tffn.h: it checks dtypes,
shapes and devices of torch tensors and passes their device pointers and the
current CUDA stream.  Every step of the computation runs in the library's CUDA
kernels; there is no fallback.  If the compiled library (libtffn.so, built by
``transformer_ffn_gb300.build``) is missing, every call raises.
"""
import ctypes
import os

import torch

__all__ = ["ffn_forward", "moe_ffn_forward", "load", "check", "set_option", "workspace_bytes",
           "set_workspace", "last_launch_count", "timing_begin", "timing_end", "TffnError",
           "ACT_NONE", "ACT_RELU", "ACT_GELU_TANH", "ACT_SILU", "ffn_glu_forward", "moe_glu_forward", "OPT_PATH", "OPT_WAIT_LIMIT_MS",
           "OPT_SKIP_FLAG", "OPT_GROUP_M", "OPT_MOE_ORDER", "OPT_MOE_COMBINE", "LIB_PATH"]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtffn.so")

ACT_NONE, ACT_RELU, ACT_GELU_TANH, ACT_SILU = 0, 1, 2, 3
_ACTS = {"none": ACT_NONE, None: ACT_NONE, "relu": ACT_RELU, "gelu_tanh": ACT_GELU_TANH,
         "gelu": ACT_GELU_TANH, "silu": ACT_SILU, "swish": ACT_SILU}
OPT_PATH, OPT_WAIT_LIMIT_MS, OPT_SKIP_FLAG, OPT_GROUP_M, OPT_MOE_ORDER, OPT_MOE_COMBINE = 1, 2, 3, 4, 5, 6

_lib = None


class TffnError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        msg = _lib.tffn_status_string(code).decode() if _lib else str(code)
        super().__init__(f"tffn error {code} ({msg}){': ' + what if what else ''}")


class _Routing(ctypes.Structure):
    _fields_ = [("topk_idx", ctypes.c_void_p), ("topk_w", ctypes.c_void_p),
                ("perm", ctypes.c_void_p), ("expert_offsets", ctypes.c_void_p)]


def load():
    """Load libtffn.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"the CUDA library {LIB_PATH} is missing; build it with "
                           "`python -m transformer_ffn_gb300.build` (no CPU fallback exists)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.ffn_forward.argtypes = [vp, vp, vp, vp, vp, i32, i32, i64, i64, i64, i64, vp, vp]
    L.ffn_glu_forward.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i64, vp, vp]
    L.ffn_glu_forward.restype = i32
    L.ffn_forward.restype = i32
    L.moe_ffn_forward.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, i64, i64, i64, i64, i32, i32, i32,
                                  ctypes.POINTER(_Routing), vp]
    L.moe_ffn_forward.restype = i32
    L.moe_glu_forward.argtypes = [vp, vp, i32, vp, vp, vp, vp, i64, i64, i64, i64, i32, i32,
                                  ctypes.POINTER(_Routing), vp]
    L.moe_glu_forward.restype = i32
    L.tffn_workspace_bytes.argtypes = [i64, i64, i64, i64, i32, i32]
    L.tffn_workspace_bytes.restype = ctypes.c_size_t
    L.tffn_set_workspace.argtypes = [vp, ctypes.c_size_t]
    L.tffn_set_workspace.restype = i32
    L.tffn_check.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
    L.tffn_check.restype = i32
    L.tffn_status_string.argtypes = [i32]
    L.tffn_status_string.restype = ctypes.c_char_p
    L.tffn_set_option.argtypes = [i32, i64]
    L.tffn_set_option.restype = i64
    L.tffn_last_launch_count.argtypes = []
    L.tffn_last_launch_count.restype = i32
    L.tffn_timing_begin.argtypes = []
    L.tffn_timing_begin.restype = i32
    L.tffn_timing_end.argtypes = [ctypes.POINTER(i32), ctypes.POINTER(ctypes.c_double)]
    L.tffn_timing_end.restype = i32
    L.tffn_timing_sample.argtypes = [i32]
    L.tffn_timing_sample.restype = i32
    L.tffn_debug_engine_task.argtypes = [i64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, i64,
                                         ctypes.POINTER(ctypes.c_int32)]
    L.tffn_debug_engine_task.restype = i64
    L.tffn_debug_tiles.argtypes = [ctypes.POINTER(ctypes.c_int32)]
    L.tffn_debug_tiles.restype = None
    L.tffn_debug_stream_plan.argtypes = [i32, i64, i64, i64, i64, i32, i32, ctypes.POINTER(ctypes.c_int64)]
    L.tffn_debug_stream_plan.restype = i32
    _lib = L
    return L


def _act(a):
    if isinstance(a, int):
        return a
    return _ACTS[a]


def _stream_ptr(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_bf16(name, t, shape_len, device):
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if t.dim() != shape_len:
        raise ValueError(f"{name} must have {shape_len} dimensions")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _raise(rc, what):
    if rc != 0:
        raise TffnError(rc, what)


def ffn_forward(X, W1, b1, W2, b2, act1="gelu_tanh", act2="none", out=None, stream=None):
    """Y = act2(act1(X @ W1 + b1) @ W2 + b2) in bf16 (b1, b2 may be None)."""
    L = load()
    dev = X.device
    _check_bf16("X", X, 2, dev)
    _check_bf16("W1", W1, 2, dev)
    _check_bf16("W2", W2, 2, dev)
    M, N = X.shape
    N2, O = W1.shape
    O2, P = W2.shape
    if N2 != N or O2 != O:
        raise ValueError("shape mismatch")
    if b1 is not None:
        _check_bf16("b1", b1, 1, dev)
        if b1.shape[0] != O:
            raise ValueError("b1 shape")
    if b2 is not None:
        _check_bf16("b2", b2, 1, dev)
        if b2.shape[0] != P:
            raise ValueError("b2 shape")
    Y = out if out is not None else torch.empty((M, P), dtype=torch.bfloat16, device=dev)
    _check_bf16("out", Y, 2, dev)
    rc = L.ffn_forward(_ptr(X), _ptr(W1), _ptr(b1), _ptr(W2), _ptr(b2), _act(act1), _act(act2),
                       M, N, O, P, _ptr(Y), _stream_ptr(stream))
    _raise(rc, "ffn_forward")
    return Y


def ffn_glu_forward(X, W1, W3, W2, act="silu", out=None, stream=None):
    """Gated FFN Y = (act(X @ W1) * (X @ W3)) @ W2 in bf16 (SwiGLU: act="silu")."""
    L = load()
    dev = X.device
    for name, t in (("X", X), ("W1", W1), ("W3", W3), ("W2", W2)):
        _check_bf16(name, t, 2, dev)
    M, N = X.shape
    N2, O = W1.shape
    O2, P = W2.shape
    if N2 != N or O2 != O or tuple(W3.shape) != (N, O):
        raise ValueError("shape mismatch")
    Y = out if out is not None else torch.empty((M, P), dtype=torch.bfloat16, device=dev)
    _check_bf16("out", Y, 2, dev)
    rc = L.ffn_glu_forward(_ptr(X), _ptr(W1), _ptr(W3), _ptr(W2), _act(act), M, N, O, P, _ptr(Y),
                           _stream_ptr(stream))
    _raise(rc, "ffn_glu_forward")
    return Y


def moe_ffn_forward(X, gate_logits, top_k, W1, b1, W2, b2, act1="gelu_tanh", act2="none",
                    out=None, routing=False, stream=None):
    """Top-k routed MoE FFN.  W1, b1, W2, b2 are lists of per-expert tensors
    (b1 / b2 may be None).  With routing=True also returns a dict with
    topk_idx [T,k] int32, topk_w [T,k] fp32, perm [T*k] int32 and
    expert_offsets [E+1] int32."""
    L = load()
    dev = X.device
    _check_bf16("X", X, 2, dev)
    T, N = X.shape
    E = len(W1)
    if len(W2) != E or (b1 is not None and len(b1) != E) or (b2 is not None and len(b2) != E):
        raise ValueError("expert lists differ in length")
    if gate_logits.dtype != torch.float32 or gate_logits.shape != (T, E) or not gate_logits.is_contiguous():
        raise ValueError("gate_logits must be contiguous float32 [T, E]")
    O = W1[0].shape[1]
    P = W2[0].shape[1]
    for e in range(E):
        _check_bf16(f"W1[{e}]", W1[e], 2, dev)
        _check_bf16(f"W2[{e}]", W2[e], 2, dev)
        if tuple(W1[e].shape) != (N, O) or tuple(W2[e].shape) != (O, P):
            raise ValueError("expert weight shape")
        if b1 is not None:
            _check_bf16(f"b1[{e}]", b1[e], 1, dev)
        if b2 is not None:
            _check_bf16(f"b2[{e}]", b2[e], 1, dev)
    arr = ctypes.c_void_p * E
    w1a = arr(*[t.data_ptr() for t in W1])
    w2a = arr(*[t.data_ptr() for t in W2])
    b1a = arr(*[t.data_ptr() for t in b1]) if b1 is not None else None
    b2a = arr(*[t.data_ptr() for t in b2]) if b2 is not None else None
    Y = out if out is not None else torch.empty((T, P), dtype=torch.bfloat16, device=dev)
    _check_bf16("out", Y, 2, dev)
    r = None
    rp = None
    if routing:
        r = {"topk_idx": torch.empty((T, top_k), dtype=torch.int32, device=dev),
             "topk_w": torch.empty((T, top_k), dtype=torch.float32, device=dev),
             "perm": torch.empty((T * top_k,), dtype=torch.int32, device=dev),
             "expert_offsets": torch.empty((E + 1,), dtype=torch.int32, device=dev)}
        rp = ctypes.pointer(_Routing(r["topk_idx"].data_ptr(), r["topk_w"].data_ptr(),
                                     r["perm"].data_ptr(), r["expert_offsets"].data_ptr()))
    rc = L.moe_ffn_forward(_ptr(X), _ptr(gate_logits), int(top_k),
                           ctypes.cast(w1a, ctypes.c_void_p),
                           ctypes.cast(b1a, ctypes.c_void_p) if b1a is not None else None,
                           ctypes.cast(w2a, ctypes.c_void_p),
                           ctypes.cast(b2a, ctypes.c_void_p) if b2a is not None else None,
                           _ptr(Y), T, N, O, P, E, _act(act1), _act(act2), rp, _stream_ptr(stream))
    _raise(rc, "moe_ffn_forward")
    return (Y, r) if routing else Y


def moe_glu_forward(X, gate_logits, top_k, W1, W3, W2, act="silu", out=None, routing=False, stream=None):
    """Top-k routed MoE with gated experts: expert e is (act(x W1[e]) * (x W3[e])) W2[e]
    (SwiGLU with act="silu").  W1, W3, W2 are lists of per-expert tensors;
    routing as moe_ffn_forward."""
    L = load()
    dev = X.device
    _check_bf16("X", X, 2, dev)
    T, N = X.shape
    E = len(W1)
    if len(W3) != E or len(W2) != E:
        raise ValueError("expert lists differ in length")
    if gate_logits.dtype != torch.float32 or gate_logits.shape != (T, E) or not gate_logits.is_contiguous():
        raise ValueError("gate_logits must be contiguous float32 [T, E]")
    O = W1[0].shape[1]
    P = W2[0].shape[1]
    for e in range(E):
        for name, t, shape in ((f"W1[{e}]", W1[e], (N, O)), (f"W3[{e}]", W3[e], (N, O)), (f"W2[{e}]", W2[e], (O, P))):
            _check_bf16(name, t, 2, dev)
            if tuple(t.shape) != shape:
                raise ValueError(f"{name} shape")
    arr = ctypes.c_void_p * E
    w1a = arr(*[t.data_ptr() for t in W1])
    w3a = arr(*[t.data_ptr() for t in W3])
    w2a = arr(*[t.data_ptr() for t in W2])
    Y = out if out is not None else torch.empty((T, P), dtype=torch.bfloat16, device=dev)
    _check_bf16("out", Y, 2, dev)
    r = None
    rp = None
    if routing:
        r = {"topk_idx": torch.empty((T, top_k), dtype=torch.int32, device=dev),
             "topk_w": torch.empty((T, top_k), dtype=torch.float32, device=dev),
             "perm": torch.empty((T * top_k,), dtype=torch.int32, device=dev),
             "expert_offsets": torch.empty((E + 1,), dtype=torch.int32, device=dev)}
        rp = ctypes.pointer(_Routing(r["topk_idx"].data_ptr(), r["topk_w"].data_ptr(),
                                     r["perm"].data_ptr(), r["expert_offsets"].data_ptr()))
    rc = L.moe_glu_forward(_ptr(X), _ptr(gate_logits), int(top_k), ctypes.cast(w1a, ctypes.c_void_p),
                           ctypes.cast(w3a, ctypes.c_void_p), ctypes.cast(w2a, ctypes.c_void_p), _ptr(Y), T, N, O, P,
                           E, _act(act), rp, _stream_ptr(stream))
    _raise(rc, "moe_glu_forward")
    return (Y, r) if routing else Y


def check(stream=None):
    """Synchronise the stream and raise TffnError if a kernel reported an error."""
    L = load()
    detail = (ctypes.c_int32 * 4)()
    rc = L.tffn_check(_stream_ptr(stream), detail)
    if rc != 0:
        raise TffnError(rc, f"device detail {list(detail)}")


def workspace_bytes(M, N, O, P, E=0, top_k=0):
    return int(load().tffn_workspace_bytes(M, N, O, P, E, top_k))


def set_workspace(t):
    """Use a caller-owned uint8 CUDA tensor as the workspace (None: library-owned)."""
    L = load()
    if t is None:
        _raise(L.tffn_set_workspace(None, 0), "set_workspace")
    else:
        _raise(L.tffn_set_workspace(ctypes.c_void_p(t.data_ptr()), t.numel() * t.element_size()),
               "set_workspace")


def set_option(option, value):
    return int(load().tffn_set_option(option, int(value)))


def last_launch_count():
    return int(load().tffn_last_launch_count())


def timing_begin(every=1):
    """Time the dominant kernel of the next forward calls: one launch of every
    `every` gets a CUDA event pair (the others run back to back)."""
    L = load()
    _raise(L.tffn_timing_sample(int(every)), "timing_sample")
    _raise(L.tffn_timing_begin(), "timing_begin")


def timing_end():
    """(number of timed dominant-kernel launches, their summed milliseconds)."""
    n = ctypes.c_int(0)
    ms = ctypes.c_double(0.0)
    _raise(load().tffn_timing_end(ctypes.byref(n), ctypes.byref(ms)), "timing_end")
    return n.value, ms.value


def debug_engine_task(m_blocks, n1, n2, group_m, ticket):
    out = (ctypes.c_int32 * 3)()
    total = load().tffn_debug_engine_task(m_blocks, n1, n2, group_m, ticket, out)
    return int(total), (out[0], out[1], out[2])


def debug_stream_plan(path, M, N, O, P, sms, glu=False):
    """The work plan of the weight stream `path` (2 or 6) as a dict (host only)."""
    out = (ctypes.c_int64 * 12)()
    _raise(load().tffn_debug_stream_plan(path, M, N, O, P, sms, 1 if glu else 0, out), "debug_stream_plan")
    keys = ("grid", "win", "nblk", "slices0", "slices1", "kch0", "kch1", "units0", "units1", "maxp0", "maxp1",
            "partial_bytes")
    return dict(zip(keys, list(out)))


def debug_tiles():
    out = (ctypes.c_int32 * 6)()
    load().tffn_debug_tiles(out)
    return {"BM": out[0], "BN": out[1], "BK": out[2], "stages": out[3], "decode_slice": out[4],
            "decode_kc": out[5]}
