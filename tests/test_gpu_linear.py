"""GPU parity of the decode projection against the fp64 oracle, through the C ABI.

Covers the tiny-matrix kernel (B <= 2), the split-K kernel on CUDA cores (any B), the
batch-size switch of dec_linear, the fused residual, ragged N and K, the full-size
decode input projection (K=7168, N=8192, B=1..64) and the output-projection-like shape
(K=16384, N=7168 + residual), determinism, pins that hold exactly, forced variants,
host fault injection and the bounded-wait status path ("Hyper Optimizing Kimi K3 in
vLLM", Part 1 / 1 and / 2; Part 2 / 3: tests must exercise the changed path).
"""
import numpy as np
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
    ssd.dec_set_force_variant(ssd.VARIANT_NONE)
    return torch, ssd, oracle, dev


def _case(env, B, N, K, seed, residual=True):
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    X = inputs.activations(B, K, dev, seed)
    W = inputs.weight(N, K, dev, seed)
    R = inputs.residual(B, N, dev, seed) if residual else None
    Y = torch.empty(B, N, dtype=torch.bfloat16, device=dev)
    return X, W, R, Y


def _oracle_rows(env, X, W, R, rows=None):
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    if rows is None:
        y, _ = oracle.linear(inputs.bits(X), inputs.bits(W), None if R is None else inputs.bits(R))
        return y
    ri = torch.as_tensor(rows, device=W.device)
    Rs = None if R is None else inputs.bits(R[:, ri].contiguous())
    y, _ = oracle.linear(inputs.bits(X), inputs.bits(W[ri].contiguous()), Rs)
    return y


@pytest.mark.parametrize("B,N,K", [(1, 2048, 1024), (2, 2048, 1024), (1, 1000, 328),
                                   (2, 77, 8), (1, 8192, 7168), (2, 8192, 7168),
                                   (1, 3, 16392), (3, 2048, 1024), (4, 2048, 1024),
                                   (3, 77, 8), (4, 1000, 328), (3, 3, 16392),
                                   (4, 7168, 16384)])
@pytest.mark.parametrize("residual", [False, True])
def test_tiny_kernel_matches_oracle(env, B, N, K, residual):
    torch, ssd, oracle, dev = env
    X, W, R, Y = _case(env, B, N, K, 11, residual)
    ssd.dec_gemv(X, W, R, Y)
    torch.cuda.synchronize()
    assert ssd.dec_last_variant() == ssd.VARIANT_TINY
    assert_close(to_f64(oracle, Y), _oracle_rows(env, X, W, R), f"tiny B={B} N={N} K={K}")


@pytest.mark.parametrize("B,N,K", [(3, 300, 456), (5, 129, 64), (8, 1000, 1000),
                                   (17, 640, 2048), (33, 256, 520), (63, 130, 136),
                                   (64, 512, 1024), (1, 300, 456), (2, 128, 8), (16, 1, 64)])
@pytest.mark.parametrize("split_k", [0, 1, 3])
def test_splitk_cuda_core_matches_oracle(env, B, N, K, split_k):
    torch, ssd, oracle, dev = env
    KB = (K + 63) // 64
    if split_k > KB:
        pytest.skip("split larger than the k-blocks of a tile")
    X, W, R, Y = _case(env, B, N, K, 12, residual=(B % 2 == 1))
    ws = ssd.workspace(ssd.dec_splitk_workspace_bytes(B, N, K, split_k), dev)
    ssd.dec_splitk_gemm(X, W, R, Y, ws, split_k=split_k, use_tc=0)
    torch.cuda.synchronize()
    assert ssd.dec_last_variant() == ssd.VARIANT_SPLITK
    assert_close(to_f64(oracle, Y), _oracle_rows(env, X, W, R), f"splitk B={B} N={N} K={K} S={split_k}")
    assert ssd.dec_sync_status() == ssd.DEC_OK


@pytest.mark.parametrize("B", [1, 2, 4, 8, 16, 32, 64])
def test_decode_input_projection_full_size(env, B):
    """K=7168, N=8192 through the batch-size switch; every output row against the oracle."""
    torch, ssd, oracle, dev = env
    N, K = 8192, 7168
    X, W, _, Y = _case(env, B, N, K, 0, residual=False)
    ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
    ssd.dec_linear(X, W, None, Y, ws)
    torch.cuda.synchronize()
    if B == 1:
        assert ssd.dec_last_variant() == ssd.VARIANT_TINY
    elif B == 2:  # tiny, or tensor cores where the shape is on the two-halves schedule
        assert ssd.dec_last_variant() in (ssd.VARIANT_TINY, ssd.VARIANT_SPLITK_TC)
    else:
        assert ssd.dec_last_variant() in (ssd.VARIANT_SPLITK, ssd.VARIANT_SPLITK_TC)
    assert_close(to_f64(oracle, Y), _oracle_rows(env, X, W, None), f"input projection B={B}")


@pytest.mark.parametrize("B", [1, 2, 3, 4, 8, 16, 32, 64])
def test_output_projection_with_residual_full_size(env, B):
    """K=16384, N=7168 with the fused residual; every output row against the oracle."""
    torch, ssd, oracle, dev = env
    N, K = 7168, 16384
    X, W, R, Y = _case(env, B, N, K, 4, residual=True)
    ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
    ssd.dec_linear(X, W, R, Y, ws)
    torch.cuda.synchronize()
    assert_close(to_f64(oracle, Y), _oracle_rows(env, X, W, R), f"output projection B={B}")


def test_splitk_is_deterministic_and_split_independent(env):
    torch, ssd, oracle, dev = env
    B, N, K = 24, 1000, 3000
    X, W, R, Y = _case(env, B, N, K, 13)
    outs = {}
    for S in (0, 0, 2, 7):
        ws = ssd.workspace(ssd.dec_splitk_workspace_bytes(B, N, K, S), dev)
        ssd.dec_splitk_gemm(X, W, R, Y, ws, split_k=S)
        torch.cuda.synchronize()
        outs.setdefault(S, []).append(Y.clone())
    assert torch.equal(outs[0][0], outs[0][1])  # same split: bit-identical
    y_ref = _oracle_rows(env, X, W, R)
    for S, ys in outs.items():
        assert_close(to_f64(oracle, ys[0]), y_ref, f"S={S}")


def test_workspace_reusable_across_calls(env):
    """Arrival counters are reset by the kernel: back-to-back calls on one workspace."""
    torch, ssd, oracle, dev = env
    B, N, K = 9, 700, 904
    ws = ssd.workspace(ssd.dec_splitk_workspace_bytes(B, N, K, 0), dev)
    for seed in (21, 22, 23):
        X, W, R, Y = _case(env, B, N, K, seed)
        ssd.dec_splitk_gemm(X, W, R, Y, ws)
        torch.cuda.synchronize()
        assert_close(to_f64(oracle, Y), _oracle_rows(env, X, W, R), f"seed {seed}")
    counter_bytes = (((N + 127) // 128) * 4 + 255) // 256 * 256
    assert int(ws[-counter_bytes:].view(torch.int32).abs().sum()) == 0


@pytest.mark.parametrize("variant,B", [("tiny", 1), ("tiny", 2), ("tiny", 3), ("tiny", 4),
                                       ("splitk", 1), ("splitk", 2), ("splitk", 7)])
def test_exact_pins_on_gpu(env, variant, B):
    """One-hot rows give weight columns exactly; W=0 gives R exactly; small integers sum
    exactly in fp32 (|partial sums| < 2^24)."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    ssd.dec_set_force_variant(ssd.VARIANT_TINY if variant == "tiny" else ssd.VARIANT_SPLITK)
    try:
        N, K = 260, 520
        W = inputs.weight(N, K, dev, 5)
        X = torch.zeros(B, K, dtype=torch.bfloat16, device=dev)
        ks = [3, K - 1, 100, 257, 8, 9, 10][:B]
        for b, k in enumerate(ks):
            X[b, k] = 1.0
        Y = torch.empty(B, N, dtype=torch.bfloat16, device=dev)
        ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
        ssd.dec_linear(X, W, None, Y, ws)
        torch.cuda.synchronize()
        for b, k in enumerate(ks):
            assert torch.equal(Y[b], W[:, k])
        R = inputs.residual(B, N, dev, 5)
        ssd.dec_linear(X, torch.zeros_like(W), R, Y, ws)
        torch.cuda.synchronize()
        assert torch.equal(Y.float(), R.float())
        g = torch.Generator(device=dev).manual_seed(9)
        Xi = torch.randint(-4, 5, (B, K), device=dev, generator=g).to(torch.bfloat16)
        Wi = torch.randint(-4, 5, (N, K), device=dev, generator=g).to(torch.bfloat16)
        ssd.dec_linear(Xi, Wi, None, Y, ws)
        torch.cuda.synchronize()
        exact = (Xi.double() @ Wi.double().T)
        y_ref, Y_ref = oracle.linear(inputs.bits(Xi), inputs.bits(Wi))
        assert np.array_equal(y_ref, exact.cpu().numpy())
        assert np.array_equal(inputs.bits(Y), Y_ref)
    finally:
        ssd.dec_set_force_variant(ssd.VARIANT_NONE)


def test_forced_variants_and_switch(env):
    torch, ssd, oracle, dev = env
    N, K = 384, 512
    for B in (1, 2, 3, 64):
        X, W, R, Y = _case(env, B, N, K, 31)
        ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
        ssd.dec_linear(X, W, R, Y, ws)
        torch.cuda.synchronize()
        expect = ssd.VARIANT_TINY if B <= 2 else ssd.VARIANT_SPLITK
        assert ssd.dec_last_variant() in ((expect,) if B <= 2 else (ssd.VARIANT_SPLITK, ssd.VARIANT_SPLITK_TC))
        assert_close(to_f64(oracle, Y), _oracle_rows(env, X, W, R), f"switch B={B}")
    ssd.dec_set_force_variant(ssd.VARIANT_TINY)
    try:
        X, W, R, Y = _case(env, 5, N, K, 32)
        ws = ssd.workspace(ssd.dec_linear_workspace_bytes(5, N, K), dev)
        with pytest.raises(ssd.DecError) as ei:
            ssd.dec_linear(X, W, R, Y, ws)
        assert ei.value.status == ssd.DEC_ERR_UNSUPPORTED_SHAPE
    finally:
        ssd.dec_set_force_variant(ssd.VARIANT_NONE)


def test_workspace_too_small_is_rejected(env):
    torch, ssd, oracle, dev = env
    X, W, R, Y = _case(env, 8, 256, 256, 33)
    need = ssd.dec_splitk_workspace_bytes(8, 256, 256, 0)
    ws = ssd.workspace(need - 256, dev)
    with pytest.raises(ssd.DecError) as ei:
        ssd.dec_splitk_gemm(X, W, R, Y, ws)
    assert ei.value.status == ssd.DEC_ERR_WORKSPACE_TOO_SMALL


def test_host_fault_injection(env):
    torch, ssd, oracle, dev = env
    X, W, R, Y = _case(env, 1, 256, 256, 34)
    ssd.dec_set_fault_inject(1)
    with pytest.raises(ssd.DecError) as ei:
        ssd.dec_gemv(X, W, R, Y)
    assert ei.value.status == ssd.DEC_ERR_CUDA
    ssd.dec_gemv(X, W, R, Y)  # the next launch goes through
    torch.cuda.synchronize()
    assert_close(to_f64(oracle, Y), _oracle_rows(env, X, W, R), "after injected fault")


def test_bounded_wait_reports_timeout_and_context_survives(env):
    torch, ssd, oracle, dev = env
    assert ssd.dec_sync_status() == ssd.DEC_OK
    ssd.dec_debug_wait_timeout(20_000_000)  # 20 ms on a barrier nothing arrives at
    assert ssd.dec_sync_status() == ssd.DEC_ERR_TIMEOUT
    assert ssd.dec_sync_status() == ssd.DEC_OK  # the word is cleared by the read
    X, W, R, Y = _case(env, 4, 256, 256, 35)
    ws = ssd.workspace(ssd.dec_splitk_workspace_bytes(4, 256, 256, 0), dev)
    ssd.dec_splitk_gemm(X, W, R, Y, ws)
    torch.cuda.synchronize()
    assert_close(to_f64(oracle, Y), _oracle_rows(env, X, W, R), "after time-out")


@pytest.mark.parametrize("B,N,K,residual", [(32, 8192, 12288, False), (64, 7168, 16384, True),
                                            (17, 300, 12288, True), (64, 130, 16384, False)])
@pytest.mark.parametrize("tc", [0, 1])
def test_deferred_reduction_matches_oracle(env, monkeypatch, B, N, K, residual, tc):
    """Split-K with the reduction deferred to the finishing kernel (the large-batch path),
    forced on at every batch; bit-identical on repeat."""
    torch, ssd, oracle, dev = env
    monkeypatch.setenv("DEC_DEFER_MIN_B", "1")
    X, W, R, Y = _case(env, B, N, K, 14, residual=residual)
    ws = ssd.workspace(ssd.dec_splitk_workspace_bytes(B, N, K, 0), dev)
    ssd.dec_splitk_gemm(X, W, R, Y, ws, use_tc=tc)
    torch.cuda.synchronize()
    Y1 = Y.clone()
    ssd.dec_splitk_gemm(X, W, R, Y, ws, use_tc=tc)
    torch.cuda.synchronize()
    assert torch.equal(Y, Y1)
    rng = np.random.default_rng(B + N)
    rows = np.unique(np.concatenate([rng.choice(N, min(N, 256), replace=False), [0, N - 1]]))
    y_ref = _oracle_rows(env, X, W, R, rows)
    assert_close(to_f64(oracle, Y)[:, rows], y_ref, f"deferred B={B} N={N} K={K} tc={tc}")


@pytest.mark.parametrize("B,N,K", [(16, 1024, 512), (64, 2048, 1024), (5, 1000, 256)])
@pytest.mark.parametrize("shift_y,shift_r", [(0, 0), (1, 0), (0, 1)])
def test_output_alignment_paths(env, B, N, K, shift_y, shift_r):
    """Y and R one element off a 16-byte boundary take the per-element epilogue; aligned
    ones the 16-byte one. Both match the oracle and each other bit for bit."""
    torch, ssd, oracle, dev = env
    X, W, R, _ = _case(env, B, N, K, 17)
    Rb = torch.empty(B * N + 8, dtype=torch.bfloat16, device=dev)
    Rv = Rb[shift_r:shift_r + B * N].view(B, N)
    Rv.copy_(R)
    Yb = torch.empty(B * N + 8, dtype=torch.bfloat16, device=dev)
    Yv = Yb[shift_y:shift_y + B * N].view(B, N)
    ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
    ssd.dec_linear(X, W, Rv, Yv, ws)
    Y0 = torch.empty(B, N, dtype=torch.bfloat16, device=dev)
    ssd.dec_linear(X, W, R, Y0, ws)
    torch.cuda.synchronize()
    assert torch.equal(Yv, Y0)
    assert_close(to_f64(oracle, Y0), _oracle_rows(env, X, W, R), f"aligned B={B} N={N}")
