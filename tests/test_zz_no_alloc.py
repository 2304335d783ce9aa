"""The split-K projection for callers that cannot allocate device memory.

Such callers (a plugin inside a runtime that owns the GPU memory pool, a serving loop
whose memory is frozen after warm-up) get dec_splitk_gemm_noalloc, whose scratch is a
fixed array inside the library. These tests call it through the C ABI twice in a row
and compare each result with the workspace-taking dec_splitk_gemm, within the parity
tolerance used everywhere else. The file is named to be collected last.
"""
import ctypes

import pytest

from gpu_common import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import split_switched_decode_gb300 as ssd
    ssd.build()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    return torch, ssd, dev


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("use_tc", [0, 1])
@pytest.mark.parametrize("B,N,K", [(5, 1000, 1000), (64, 8192, 7168), (3, 7168, 16384)])
def test_noalloc_matches_workspace_entry_point_twice(env, use_tc, B, N, K):
    torch, ssd, dev = env
    from split_switched_decode_gb300 import inputs
    lib = ssd.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ws = ssd.workspace(ssd.dec_splitk_workspace_bytes(B, N, K, 0), dev)
    for call in range(2):  # the second call reuses the array the first one left behind
        X = inputs.activations(B, K, dev, 70 + call)
        W = inputs.weight(N, K, dev, 70 + call)
        R = inputs.residual(B, N, dev, 70 + call) if call == 1 else None
        Y_ref = torch.empty(B, N, dtype=torch.bfloat16, device=dev)
        Y = torch.empty(B, N, dtype=torch.bfloat16, device=dev)
        ssd.dec_splitk_gemm(X, W, R, Y_ref, ws, split_k=0, use_tc=use_tc)
        st = lib.dec_splitk_gemm_noalloc(_ptr(X), _ptr(W), _ptr(R), _ptr(Y), B, N, K, use_tc,
                                         stream)
        assert st == ssd.DEC_OK, ssd.lib().dec_status_string(st)
        torch.cuda.synchronize()
        assert ssd.dec_sync_status() == ssd.DEC_OK
        assert_close(Y.double().cpu().numpy(), Y_ref.double().cpu().numpy(),
                     f"no-alloc call {call} B={B} N={N} K={K} tc={use_tc}")
