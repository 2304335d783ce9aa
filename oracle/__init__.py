"""fp64 CPU oracle of the decode hot path (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package. The CUDA library and its Python binding never import it.

The arithmetic lives in ``oracle.c`` (plain C, fp64); this module compiles it with
gcc on first use and marshals numpy arrays in and out. Every function states the
passage of "Hyper Optimizing Kimi K3 in vLLM: Moving Fast and Responsibly" it follows
in the C source.
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
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_build/liboracle.so`` (gcc, OpenMP, strict IEEE)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # ORACLE_LIB_OVERRIDE lets the mutation test load a deliberately broken copy
        override = os.environ.get("ORACLE_LIB_OVERRIDE")
        if override:
            lib = ctypes.CDLL(override)
        else:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_from_double.restype = ctypes.c_uint16
        lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
        lib.oracle_bf16_decode_array.argtypes = [P, P, ctypes.c_int64]
        lib.oracle_bf16_encode_array.argtypes = [P, P, ctypes.c_int64]
        lib.oracle_num_threads.restype = I
        lib.oracle_linear.argtypes = [P, P, P, I, I, I, P, P]
        lib.oracle_route.argtypes = [P, I, I, I, P, P, P]
        lib.oracle_moe_front.argtypes = [P, P, I, I, I, I, I, P, P, P, P, P]
        lib.oracle_route_map.argtypes = [P, I, I, I, P, P, P, P, P, P]
        lib.oracle_silu.restype = ctypes.c_double
        lib.oracle_silu.argtypes = [ctypes.c_double]
        lib.oracle_expert_mlp.argtypes = [P, P, P, I, I, P, P]
        lib.oracle_combine.argtypes = [I, I, I, P, P, P, P, P]
        lib.oracle_moe_experts.argtypes = [P, P, P, P, P, I, P, P, I, I, I, I, P, P]
        _lib = lib
        return lib


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected raw bf16 bits as uint16, got {a.dtype}")
    return a


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a):
    return None if a is None else a.ctypes.data


def num_threads() -> int:
    return int(_load().oracle_num_threads())


# ------------------------------------------------------------------ bf16 ----

def bf16_to_f64(h) -> np.ndarray:
    h = _u16(h)
    out = np.empty(h.shape, dtype=np.float64)
    _load().oracle_bf16_decode_array(_ptr(h), _ptr(out), h.size)
    return out


def f64_to_bf16(v) -> np.ndarray:
    v = _f64(v)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_bf16_encode_array(_ptr(v), _ptr(out), v.size)
    return out


def silu(t: float) -> float:
    return float(_load().oracle_silu(float(t)))


# ---------------------------------------------------------------- linear ----

def linear(X, W, R=None):
    """y = X . W^T (+ R) in fp64; returns (y_exact fp64 [B,N], Y bf16 bits [B,N])."""
    X, W = _u16(X), _u16(W)
    B, K = X.shape
    N, K2 = W.shape
    assert K == K2
    if R is not None:
        R = _u16(R)
        assert R.shape == (B, N)
    y = np.empty((B, N), dtype=np.float64)
    Y = np.empty((B, N), dtype=np.uint16)
    _load().oracle_linear(_ptr(X), _ptr(W), _ptr(R), B, N, K, _ptr(y), _ptr(Y))
    return y, Y


# ---------------------------------------------------------------- router ----

def route(logits, topk: int):
    """softmax / top-k / renormalise; returns (idx int32 [B,k], w fp64 [B,k], probs fp64 [B,E])."""
    logits = _f64(logits)
    B, E = logits.shape
    idx = np.empty((B, topk), dtype=np.int32)
    w = np.empty((B, topk), dtype=np.float64)
    probs = np.empty((B, E), dtype=np.float64)
    _load().oracle_route(_ptr(logits), B, E, topk, _ptr(idx), _ptr(w), _ptr(probs))
    return idx, w, probs


def moe_front(X, Wcat, E: int, L: int, topk: int):
    """Router + latent as one product, then routing.

    Returns dict(logits fp64 [B,E], latent bf16 bits [B,L], idx int32 [B,k], w fp64 [B,k],
    probs fp64 [B,E]).
    """
    X, Wcat = _u16(X), _u16(Wcat)
    B, K = X.shape
    assert Wcat.shape == (E + L, K)
    logits = np.empty((B, E), dtype=np.float64)
    latent = np.empty((B, L), dtype=np.uint16)
    idx = np.empty((B, topk), dtype=np.int32)
    w = np.empty((B, topk), dtype=np.float64)
    probs = np.empty((B, E), dtype=np.float64)
    _load().oracle_moe_front(_ptr(X), _ptr(Wcat), B, K, E, L, topk, _ptr(logits),
                             _ptr(latent), _ptr(idx), _ptr(w), _ptr(probs))
    return dict(logits=logits, latent=latent, idx=idx, w=w, probs=probs)


def route_map(idx, E: int):
    """Counting-sort inverse of the routing; returns dict of int32 arrays and num_used."""
    idx = _i32(idx)
    B, topk = idx.shape
    P = B * topk
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    pairs = np.empty(P, dtype=np.int32)
    pos = np.empty(P, dtype=np.int32)
    used = np.zeros(E, dtype=np.int32)
    nu = np.zeros(1, dtype=np.int32)
    _load().oracle_route_map(_ptr(idx), B, topk, E, _ptr(counts), _ptr(offsets), _ptr(pairs),
                             _ptr(pos), _ptr(used), _ptr(nu))
    return dict(counts=counts, offsets=offsets, pairs=pairs, pos=pos,
                used=used[: int(nu[0])].copy(), num_used=int(nu[0]))


# --------------------------------------------------------------- experts ----

def expert_mlp(x, Wgu, Wd):
    """One SiLU-gated MLP for one token; returns (a bf16 bits [I], y fp64 [H])."""
    x, Wgu, Wd = _u16(x), _u16(Wgu), _u16(Wd)
    H = x.shape[-1]
    I = Wgu.shape[0] // 2
    assert Wgu.shape == (2 * I, H) and Wd.shape == (H, I)
    a = np.empty(I, dtype=np.uint16)
    y = np.empty(H, dtype=np.float64)
    _load().oracle_expert_mlp(_ptr(x), _ptr(Wgu), _ptr(Wd), H, I, _ptr(a), _ptr(y))
    return a, y


def combine(w, yp, s=None):
    """y[b] = sum_j w[b,j] yp[b,j] (+ s[b]); returns (y_exact fp64 [B,H], Y bf16 bits)."""
    w, yp = _f64(w), _f64(yp)
    B, topk, H = yp.shape
    assert w.shape == (B, topk)
    if s is not None:
        s = _f64(s)
        assert s.shape == (B, H)
    y = np.empty((B, H), dtype=np.float64)
    Y = np.empty((B, H), dtype=np.uint16)
    _load().oracle_combine(B, H, topk, _ptr(w), _ptr(yp), _ptr(s), _ptr(y), _ptr(Y))
    return y, Y


def moe_experts(X, idx, w, Wgu, Wd, Wgu_s=None, Wd_s=None):
    """Routed experts + shared expert with every weight on the host (small shapes)."""
    X, Wgu, Wd = _u16(X), _u16(Wgu), _u16(Wd)
    idx, w = _i32(idx), _f64(w)
    B, H = X.shape
    E, twoI, H2 = Wgu.shape
    I = twoI // 2
    topk = idx.shape[1]
    assert H2 == H and Wd.shape == (E, H, I)
    if Wgu_s is not None:
        Wgu_s, Wd_s = _u16(Wgu_s), _u16(Wd_s)
    y = np.empty((B, H), dtype=np.float64)
    Y = np.empty((B, H), dtype=np.uint16)
    _load().oracle_moe_experts(_ptr(X), _ptr(idx), _ptr(w), _ptr(Wgu), _ptr(Wd), E,
                               _ptr(Wgu_s), _ptr(Wd_s), B, H, I, topk, _ptr(y), _ptr(Y))
    return y, Y
