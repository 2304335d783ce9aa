"""The split-K projection for callers that cannot allocate device memory.

Such callers (a plugin inside a runtime that owns the GPU memory pool, a serving loop
whose memory is frozen after warm-up) get dec_splitk_gemm_noalloc, whose scratch is a
fixed array inside the library. These tests call it through the C ABI twice in a row
on the same array and check each result against the fp64 oracle within the parity
tolerance used everywhere else, and bit for bit against the workspace-taking
dec_splitk_gemm (same planning and kernels). Shapes whose scratch does not fit the
array, and row counts the entry point does not take, must be refused with the
documented status before anything is launched. The file is named to be collected last.
"""
import ctypes

import pytest

from gpu_common import assert_close, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    import split_switched_decode_gb300 as ssd
    ssd.build()
    oracle.build()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    return torch, ssd, oracle, dev


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(env, X, W, R, Y, use_tc):
    torch, ssd, oracle, dev = env
    B, K = X.shape
    N = W.shape[0]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return ssd.lib().dec_splitk_gemm_noalloc(_ptr(X), _ptr(W), _ptr(R), _ptr(Y), B, N, K,
                                             use_tc, stream)


@pytest.mark.parametrize("use_tc", [0, 1])
@pytest.mark.parametrize("B,N,K", [(5, 1000, 1000), (64, 8192, 7168), (3, 7168, 16384),
                                   (1, 300, 456)])
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(env, use_tc, B, N, K):
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    ws = ssd.workspace(ssd.dec_splitk_workspace_bytes(B, N, K, 0), dev)
    for call in range(2):  # the second call reuses the array the first one left behind
        X = inputs.activations(B, K, dev, 70 + call)
        W = inputs.weight(N, K, dev, 70 + call)
        R = inputs.residual(B, N, dev, 70 + call) if call == 1 else None
        Y_ws = torch.empty(B, N, dtype=torch.bfloat16, device=dev)
        Y = torch.empty(B, N, dtype=torch.bfloat16, device=dev)
        ssd.dec_splitk_gemm(X, W, R, Y_ws, ws, split_k=0, use_tc=use_tc)
        st = _noalloc(env, X, W, R, Y, use_tc)
        assert st == ssd.DEC_OK, ssd.lib().dec_status_string(st)
        torch.cuda.synchronize()
        assert ssd.dec_sync_status() == ssd.DEC_OK
        y_ref, _ = oracle.linear(inputs.bits(X), inputs.bits(W),
                                 None if R is None else inputs.bits(R))
        assert_close(to_f64(oracle, Y), y_ref,
                     f"no-alloc call {call} B={B} N={N} K={K} tc={use_tc}")
        assert torch.equal(Y, Y_ws), f"no-alloc call {call} differs from dec_splitk_gemm"


def test_noalloc_wide_rows_that_fit(env):
    """100 speculative-verification rows on tensor cores (two 64-column groups), ragged
    N and K, with a residual, twice in a row."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    B, N, K = 100, 520, 776
    for call in range(2):
        X = inputs.activations(B, K, dev, 80 + call)
        W = inputs.weight(N, K, dev, 80 + call)
        R = inputs.residual(B, N, dev, 80 + call)
        Y = torch.empty(B, N, dtype=torch.bfloat16, device=dev)
        st = _noalloc(env, X, W, R, Y, 1)
        assert st == ssd.DEC_OK, ssd.lib().dec_status_string(st)
        torch.cuda.synchronize()
        assert ssd.dec_sync_status() == ssd.DEC_OK
        y_ref, _ = oracle.linear(inputs.bits(X), inputs.bits(W), inputs.bits(R))
        assert_close(to_f64(oracle, Y), y_ref, f"no-alloc wide call {call}")


def test_noalloc_cta_pair_rows_equal_workspace_entry_point(env):
    """200 rows: like dec_splitk_gemm with split_k = 0, the no-alloc call runs on CTA-pair
    tiles (same kernel, same bits), and matches the oracle; the shape's split-K scratch
    (the size contract both entry points keep) fits in the 16 MiB array."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    B, N, K = 200, 264, 520
    X = inputs.activations(B, K, dev, 85)
    W = inputs.weight(N, K, dev, 85)
    R = inputs.residual(B, N, dev, 85)
    Y = torch.empty(B, N, dtype=torch.bfloat16, device=dev)
    assert _noalloc(env, X, W, R, Y, 1) == ssd.DEC_OK
    torch.cuda.synchronize()
    assert ssd.dec_last_variant() == ssd.VARIANT_SPLITK_TC_PAIR
    Y_ws = torch.empty_like(Y)
    ws = ssd.workspace(ssd.dec_splitk_workspace_bytes(B, N, K, 0), dev)
    ssd.dec_splitk_gemm(X, W, R, Y_ws, ws, split_k=0, use_tc=1)
    torch.cuda.synchronize()
    assert torch.equal(Y, Y_ws)
    y_ref, _ = oracle.linear(inputs.bits(X), inputs.bits(W), inputs.bits(R))
    assert_close(to_f64(oracle, Y), y_ref, "no-alloc CTA-pair rows")


@pytest.mark.parametrize("B,N,K,use_tc,status", [
    (256, 8192, 7168, 1, "DEC_ERR_WORKSPACE_TOO_SMALL"),  # ~34 MB of partial tiles
    (257, 512, 512, 1, "DEC_ERR_UNSUPPORTED_SHAPE"),       # more than one launch of rows
    (65, 512, 512, 0, "DEC_ERR_UNSUPPORTED_SHAPE"),        # wide rows need tensor cores
])
def test_noalloc_refusals(env, B, N, K, use_tc, status):
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    X = inputs.activations(B, K, dev, 90)
    W = inputs.weight(N, K, dev, 90)
    Y = torch.full((B, N), 3.0, dtype=torch.bfloat16, device=dev)
    assert _noalloc(env, X, W, None, Y, use_tc) == getattr(ssd, status)
    torch.cuda.synchronize()
    assert bool(torch.all(Y == 3.0)), "a refused call must not write its output"
    assert ssd.dec_sync_status() == ssd.DEC_OK
