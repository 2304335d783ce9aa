"""Python binding of ``libsplit_switched_decode.so`` (GB300 small-batch decode hot path).

Thin ctypes marshalling over the C ABI in ``include/split_switched_decode.h``: the
functions below have the same names as the C entry points, take torch CUDA tensors,
pass their device pointers, sizes and the current CUDA stream, and raise ``DecError``
on a non-OK status. Every step of the computation runs in the library's CUDA kernels;
there is no Python or CPU fallback, and importing a function that needs the library
fails loudly when it has not been built.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

LIB_PATH = _build.LIB_PATH

DEC_OK = 0
DEC_ERR_INVALID_ARG = 1
DEC_ERR_UNSUPPORTED_SHAPE = 2
DEC_ERR_MISALIGNED = 3
DEC_ERR_WORKSPACE_TOO_SMALL = 4
DEC_ERR_CUDA = 5
DEC_ERR_TIMEOUT = 6

VARIANT_NONE = -1
VARIANT_TINY = 0
VARIANT_SPLITK = 1
VARIANT_SPLITK_TC = 2
VARIANT_FRONT_ONE_LAUNCH = 3
VARIANT_SPLITK_TC_PAIR = 4

# every symbol the public header declares
EXPORTS = [
    "dec_status_string", "dec_variant_name", "dec_last_variant", "dec_version",
    "dec_set_force_variant", "dec_set_fault_inject", "dec_set_wait_limit_ns",
    "dec_sync_status", "dec_debug_wait_timeout", "dec_gemv", "dec_splitk_workspace_bytes",
    "dec_splitk_gemm", "dec_linear_workspace_bytes", "dec_linear", "moe_route_map_ints",
    "moe_front_workspace_bytes", "moe_front", "moe_experts_workspace_bytes", "moe_experts",
    "moe_layer_workspace_bytes", "moe_layer",
    "l2_prefetch", "dec_sim_comm_wait", "dec_splitk_gemm_noalloc",
    "dec_pack_weight", "dec_gemv_packed", "dec_splitk_gemm_packed", "dec_linear_packed",
    "dec_pack_expert_weights", "moe_experts_packed", "moe_layer_packed",
    "dec_read_stream_bytes", "dec_read_stream",
]

_lib = None


class DecError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _load().dec_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")


def build(force: bool = False) -> str:
    """Compile the CUDA library in-tree (nvcc, sm_103a)."""
    global _lib
    path = _build.build(force=force)
    return path


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it first (python -m split_switched_decode_gb300.build)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, S, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint64
    sig = {
        "dec_status_string": (ctypes.c_char_p, [I]),
        "dec_variant_name": (ctypes.c_char_p, [I]),
        "dec_last_variant": (I, []),
        "dec_version": (I, []),
        "dec_set_force_variant": (I, [I]),
        "dec_set_fault_inject": (I, [I]),
        "dec_set_wait_limit_ns": (I, [U64]),
        "dec_sync_status": (I, [P]),
        "dec_debug_wait_timeout": (I, [U64, P]),
        "dec_gemv": (I, [P, P, P, P, I, I, I, P]),
        "dec_splitk_workspace_bytes": (S, [I, I, I, I]),
        "dec_splitk_gemm": (I, [P, P, P, P, I, I, I, I, I, P, S, P]),
        "dec_linear_workspace_bytes": (S, [I, I, I]),
        "dec_linear": (I, [P, P, P, P, I, I, I, P, S, P]),
        "dec_pack_weight": (I, [P, I, I, P, P]),
        "dec_gemv_packed": (I, [P, P, P, P, I, I, I, P]),
        "dec_splitk_gemm_packed": (I, [P, P, P, P, I, I, I, I, I, P, S, P]),
        "dec_linear_packed": (I, [P, P, P, P, I, I, I, P, S, P]),
        "moe_route_map_ints": (S, [I, I, I]),
        "moe_front_workspace_bytes": (S, [I, I, I, I]),
        "moe_front": (I, [P, P, I, I, I, I, I, P, P, P, P, P, P, S, P]),
        "moe_experts_workspace_bytes": (S, [I, I, I, I, I]),
        "moe_experts": (I, [P, P, P, P, P, P, I, P, P, I, I, I, I, P, P, S, P, P, I]),
        "moe_layer_workspace_bytes": (S, [I, I, I, I, I, I]),
        "moe_layer": (I, [P, P, I, I, I, P, P, P, P, I, I, I, P, P, P, P, P, P, S, P, P, I]),
        "dec_pack_expert_weights": (I, [P, P, I, I, I, P, P, P]),
        "dec_read_stream_bytes": (S, [S]),
        "dec_read_stream": (I, [P, S, P]),
        "moe_experts_packed": (I, [P, P, P, P, P, P, I, P, P, I, I, I, I, P, P, S, P, P, I]),
        "moe_layer_packed": (I, [P, P, I, I, I, P, P, P, P, I, I, I, P, P, P, P, P, P, S, P, P,
                                 I]),
        "l2_prefetch": (I, [P, S, I, P]),
        "dec_sim_comm_wait": (I, [U64, P]),
        "dec_splitk_gemm_noalloc": (I, [P, P, P, P, I, I, I, I, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def lib():
    """The loaded ctypes library (raises if it has not been built)."""
    return _load()


# --------------------------------------------------------------- marshalling ----

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, where: str):
    if status != DEC_OK:
        raise DecError(status, where)


def _bf16(t, name):
    import torch
    if t is None:
        return
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous bfloat16 CUDA tensor")


def workspace(nbytes: int, device=None):
    """A zero-filled uint8 CUDA buffer (16-byte aligned by the caching allocator)."""
    import torch
    return torch.zeros(max(int(nbytes), 16), dtype=torch.uint8, device=device or "cuda")


# ------------------------------------------------------------------- status ----

def dec_last_variant() -> int:
    return _load().dec_last_variant()


def dec_variant_name(v: int) -> str:
    return _load().dec_variant_name(v).decode()


def dec_set_force_variant(v: int):
    _check(_load().dec_set_force_variant(v), "dec_set_force_variant")


def dec_set_fault_inject(n: int):
    _check(_load().dec_set_fault_inject(n), "dec_set_fault_inject")


def dec_set_wait_limit_ns(ns: int):
    _check(_load().dec_set_wait_limit_ns(ns), "dec_set_wait_limit_ns")


def dec_sync_status(stream=None) -> int:
    return _load().dec_sync_status(_stream(stream))


def dec_debug_wait_timeout(limit_ns: int, stream=None):
    _check(_load().dec_debug_wait_timeout(limit_ns, _stream(stream)), "dec_debug_wait_timeout")


# --------------------------------------------------------------- projection ----

def dec_gemv(X, W, R, Y, stream=None):
    for t, n in ((X, "X"), (W, "W"), (R, "R"), (Y, "Y")):
        _bf16(t, n)
    B, K = X.shape
    N = W.shape[0]
    _check(_load().dec_gemv(_ptr(X), _ptr(W), _ptr(R), _ptr(Y), B, N, K, _stream(stream)),
           "dec_gemv")


def dec_splitk_workspace_bytes(B, N, K, split_k=0) -> int:
    return int(_load().dec_splitk_workspace_bytes(B, N, K, split_k))


def dec_splitk_gemm(X, W, R, Y, ws, split_k=0, use_tc=0, stream=None):
    for t, n in ((X, "X"), (W, "W"), (R, "R"), (Y, "Y")):
        _bf16(t, n)
    B, K = X.shape
    N = W.shape[0]
    _check(_load().dec_splitk_gemm(_ptr(X), _ptr(W), _ptr(R), _ptr(Y), B, N, K, split_k, use_tc,
                                   _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "dec_splitk_gemm")


def dec_splitk_gemm_noalloc(X, W, R, Y, use_tc=0, stream=None):
    """dec_splitk_gemm for callers that cannot allocate: the scratch is a fixed 16 MiB
    array inside the library; calls on one GPU must not overlap."""
    for t, n in ((X, "X"), (W, "W"), (R, "R"), (Y, "Y")):
        _bf16(t, n)
    B, K = X.shape
    N = W.shape[0]
    _check(_load().dec_splitk_gemm_noalloc(_ptr(X), _ptr(W), _ptr(R), _ptr(Y), B, N, K, use_tc,
                                           _stream(stream)), "dec_splitk_gemm_noalloc")


def dec_linear_workspace_bytes(B, N, K) -> int:
    return int(_load().dec_linear_workspace_bytes(B, N, K))


def dec_linear(X, W, R, Y, ws, stream=None):
    for t, n in ((X, "X"), (W, "W"), (R, "R"), (Y, "Y")):
        _bf16(t, n)
    B, K = X.shape
    N = W.shape[0]
    nb = 0 if ws is None else ws.numel() * ws.element_size()
    _check(_load().dec_linear(_ptr(X), _ptr(W), _ptr(R), _ptr(Y), B, N, K, _ptr(ws), nb,
                              _stream(stream)), "dec_linear")


def dec_pack_weight(W, Wp=None, stream=None):
    """The tile-packed copy of a row-major W [N,K] (N % 128 == 0, K % 64 == 0): a tensor
    of the same shape and dtype whose storage is 16 KB blocks of 128 rows x 64 k. Pass it
    to the *_packed projections only."""
    import torch
    _bf16(W, "W")
    N, K = W.shape
    if Wp is None:
        Wp = torch.empty_like(W)
    _bf16(Wp, "Wp")
    _check(_load().dec_pack_weight(_ptr(W), N, K, _ptr(Wp), _stream(stream)), "dec_pack_weight")
    return Wp


def dec_gemv_packed(X, Wp, R, Y, stream=None):
    for t, n in ((X, "X"), (Wp, "Wp"), (R, "R"), (Y, "Y")):
        _bf16(t, n)
    B, K = X.shape
    N = Wp.shape[0]
    _check(_load().dec_gemv_packed(_ptr(X), _ptr(Wp), _ptr(R), _ptr(Y), B, N, K,
                                   _stream(stream)), "dec_gemv_packed")


def dec_splitk_gemm_packed(X, Wp, R, Y, ws, split_k=0, use_tc=0, stream=None):
    for t, n in ((X, "X"), (Wp, "Wp"), (R, "R"), (Y, "Y")):
        _bf16(t, n)
    B, K = X.shape
    N = Wp.shape[0]
    _check(_load().dec_splitk_gemm_packed(_ptr(X), _ptr(Wp), _ptr(R), _ptr(Y), B, N, K, split_k,
                                          use_tc, _ptr(ws), ws.numel() * ws.element_size(),
                                          _stream(stream)), "dec_splitk_gemm_packed")


def dec_linear_packed(X, Wp, R, Y, ws, stream=None):
    for t, n in ((X, "X"), (Wp, "Wp"), (R, "R"), (Y, "Y")):
        _bf16(t, n)
    B, K = X.shape
    N = Wp.shape[0]
    nb = 0 if ws is None else ws.numel() * ws.element_size()
    _check(_load().dec_linear_packed(_ptr(X), _ptr(Wp), _ptr(R), _ptr(Y), B, N, K, _ptr(ws), nb,
                                     _stream(stream)), "dec_linear_packed")


# ---------------------------------------------------------------------- MoE ----

def moe_route_map_ints(B, E, topk) -> int:
    return int(_load().moe_route_map_ints(B, E, topk))


def moe_front_workspace_bytes(B, E, L, K) -> int:
    return int(_load().moe_front_workspace_bytes(B, E, L, K))


def moe_front(X, Wcat, E, L, topk, latent, topk_idx, topk_w, ws, probs=None, route_map=None,
              stream=None):
    _bf16(X, "X")
    _bf16(Wcat, "Wcat")
    _bf16(latent, "latent")
    B, K = X.shape
    _check(_load().moe_front(_ptr(X), _ptr(Wcat), B, K, E, L, topk, _ptr(latent),
                             _ptr(topk_idx), _ptr(topk_w), _ptr(probs), _ptr(route_map),
                             _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_front")


def moe_experts_workspace_bytes(B, E, topk, H, I) -> int:
    return int(_load().moe_experts_workspace_bytes(B, E, topk, H, I))


def moe_experts(X, topk_idx, topk_w, route_map, Wgu, Wd, Wgu_shared, Wd_shared, Y, ws,
                main_stream=None, side_stream=None, side_max_ctas=0, packed=False):
    """packed: Wgu/Wd (and the shared pair) from dec_pack_expert_weights."""
    for t, n in ((X, "X"), (Wgu, "Wgu"), (Wd, "Wd"), (Wgu_shared, "Wgu_shared"),
                 (Wd_shared, "Wd_shared"), (Y, "Y")):
        _bf16(t, n)
    B, H = X.shape
    E, twoI, _ = Wgu.shape
    I = twoI // 2
    topk = topk_idx.shape[1]
    ms = _stream(main_stream)
    ss = _stream(side_stream) if side_stream is not None else ms
    fn = _load().moe_experts_packed if packed else _load().moe_experts
    _check(fn(_ptr(X), _ptr(topk_idx), _ptr(topk_w), _ptr(route_map), _ptr(Wgu), _ptr(Wd), E,
              _ptr(Wgu_shared), _ptr(Wd_shared), B, H, I, topk, _ptr(Y), _ptr(ws),
              ws.numel() * ws.element_size(), ms, ss, side_max_ctas), "moe_experts")


def dec_pack_expert_weights(Wgu, Wd, stream=None):
    """Tile-packed copies of an expert bank: Wgu [E, 2I, H] (gate rows, then up rows) and
    Wd [E, H, I] -> tensors of the same shapes whose storage is 16 KB blocks (64 gate rows
    + the 64 matching up rows, resp. 128 down rows, x 64 k). For moe_*(packed=True)."""
    import torch
    _bf16(Wgu, "Wgu")
    _bf16(Wd, "Wd")
    E, twoI, H = Wgu.shape
    Wgu_p, Wd_p = torch.empty_like(Wgu), torch.empty_like(Wd)
    _check(_load().dec_pack_expert_weights(_ptr(Wgu), _ptr(Wd), E, H, twoI // 2, _ptr(Wgu_p),
                                           _ptr(Wd_p), _stream(stream)), "dec_pack_expert_weights")
    return Wgu_p, Wd_p


def l2_prefetch(t, nbytes=None, max_ctas=0, stream=None):
    n = t.numel() * t.element_size() if nbytes is None else int(nbytes)
    _check(_load().l2_prefetch(_ptr(t), n, max_ctas, _stream(stream)), "l2_prefetch")


def dec_read_stream(t, stream=None) -> int:
    """Stream tensor t's bytes through every SM (bulk copies into shared memory; nothing
    is written) -- a measurement helper. Returns the bytes the call reads."""
    n = t.numel() * t.element_size()
    _check(_load().dec_read_stream(_ptr(t), n, _stream(stream)), "dec_read_stream")
    return int(_load().dec_read_stream_bytes(n))


def dec_sim_comm_wait(ns: int, stream=None):
    """Keep `stream` busy for ns nanoseconds without memory traffic (a stand-in for a
    communication phase)."""
    _check(_load().dec_sim_comm_wait(int(ns), _stream(stream)), "dec_sim_comm_wait")



def moe_layer_workspace_bytes(B, E, L, H, I, topk) -> int:
    return int(_load().moe_layer_workspace_bytes(B, E, L, H, I, topk))


def moe_layer(X, Wcat, E, L, topk, Wgu, Wd, Wgu_shared, Wd_shared, latent, topk_idx, topk_w,
              Y, ws, route_map=None, stream=None, side_stream=None, side_max_ctas=0,
              packed=False):
    """moe_front + moe_experts with the shared expert overlapping the routing (packed:
    expert banks from dec_pack_expert_weights)."""
    for t, n in ((X, "X"), (Wcat, "Wcat"), (Wgu, "Wgu"), (Wd, "Wd"), (Wgu_shared, "Wgu_shared"),
                 (Wd_shared, "Wd_shared"), (latent, "latent"), (Y, "Y")):
        _bf16(t, n)
    B, H = X.shape
    I = Wgu.shape[1] // 2
    main = _stream(stream)
    side = _stream(side_stream) if side_stream is not None else main
    fn = _load().moe_layer_packed if packed else _load().moe_layer
    _check(fn(_ptr(X), _ptr(Wcat), E, L, topk, _ptr(Wgu), _ptr(Wd), _ptr(Wgu_shared),
              _ptr(Wd_shared), B, H, I, _ptr(latent), _ptr(topk_idx), _ptr(topk_w),
              _ptr(route_map), _ptr(Y), _ptr(ws), ws.numel() * ws.element_size(), main, side,
              side_max_ctas), "moe_layer")
