"""GPU parity of the tile-packed weight layout (dec_pack_weight and the *_packed
projections) through the C ABI: the packed tensor is exactly the layout its definition
gives (a reshape and permute of the row-major W); every packed split-K projection --
CUDA cores and tensor cores, the two-halves cluster schedule, the deferred reduction,
wide rows, the batch-size switch above the tiny kernel -- gives the same bits as its
row-major counterpart on the unpacked W, which the oracle checks in test_gpu_linear.py;
the packed tiny kernel (its own lane mapping and summation order) and the full-size
Kimi projections are compared with the fp64 oracle.
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


def _packed_reference(W):
    """The layout by its definition: block (n/128, k/64) of 128 rows x 64 k, blocks in
    (n/128, k/64) order, rows of 64 k inside."""
    N, K = W.shape
    return W.view(N // 128, 128, K // 64, 64).permute(0, 2, 1, 3).contiguous().view(N, K)


@pytest.mark.parametrize("N,K", [(128, 64), (256, 192), (384, 7168), (8192, 7168)])
def test_pack_weight_layout(env, N, K):
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    W = inputs.weight(N, K, dev, 21)
    Wp = ssd.dec_pack_weight(W)
    torch.cuda.synchronize()
    assert torch.equal(Wp, _packed_reference(W))
    # element (n, k) where the definition puts it
    points = [(0, 0), (127, 63), (128, 64), (N - 1, K - 1), (N // 2 + 3, K // 3 + 5)]
    for n, k in [(n, k) for n, k in points if n < N and k < K]:
        at = ((n // 128) * (K // 64) + k // 64) * 8192 + (n % 128) * 64 + k % 64
        assert Wp.view(-1)[at].item() == W[n, k].item()


def _run_both(env, fn_rm, fn_pk, B, N, K, residual, seed, **kw):
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    X = inputs.activations(B, K, dev, seed)
    W = inputs.weight(N, K, dev, seed)
    R = inputs.residual(B, N, dev, seed) if residual else None
    Wp = ssd.dec_pack_weight(W)
    Y0 = torch.full((B, N), float("nan"), dtype=torch.bfloat16, device=dev)
    Y1 = torch.full((B, N), float("nan"), dtype=torch.bfloat16, device=dev)
    fn_rm(X, W, R, Y0, **kw)
    v0 = ssd.dec_last_variant()
    fn_pk(X, Wp, R, Y1, **kw)
    v1 = ssd.dec_last_variant()
    torch.cuda.synchronize()
    assert ssd.dec_sync_status() == ssd.DEC_OK
    return X, W, R, Y0, Y1, (v0, v1)


@pytest.mark.parametrize("B", [1, 2, 3, 4])
@pytest.mark.parametrize("N,K,residual", [(128, 64, True), (256, 192, True), (384, 1088, False),
                                          (2048, 1024, True), (8192, 7168, False),
                                          (7168, 16384, True)])
def test_gemv_packed_matches_oracle(env, B, N, K, residual):
    """The packed tiny kernel (4 rows x 128 bytes per warp load) against the oracle on every
    output, ragged quads per CTA and k-pieces included; repeated calls give the same bits."""
    torch, ssd, oracle, dev = env
    X, W, R, Y0, Y1, v = _run_both(env, ssd.dec_gemv, ssd.dec_gemv_packed, B, N, K, residual, 22)
    assert v == (ssd.VARIANT_TINY, ssd.VARIANT_TINY)
    from split_switched_decode_gb300 import inputs
    y, _ = oracle.linear(inputs.bits(X), inputs.bits(W), None if R is None else inputs.bits(R))
    assert_close(to_f64(oracle, Y1), y, f"packed tiny B={B} N={N} K={K}")
    Y2 = torch.empty_like(Y1)
    ssd.dec_gemv_packed(X, ssd.dec_pack_weight(W), R, Y2)
    torch.cuda.synchronize()
    assert torch.equal(Y1, Y2)


@pytest.mark.parametrize("B", [1, 2, 3, 5, 16, 33, 64, 100, 300])
@pytest.mark.parametrize("N,K", [(256, 192), (384, 1024), (8192, 7168), (7168, 16384)])
@pytest.mark.parametrize("use_tc,split_k", [(1, 0), (0, 0), (1, 3)])
def test_splitk_packed_equals_row_major(env, B, N, K, use_tc, split_k):
    torch, ssd, oracle, dev = env
    if B > 64 and not use_tc:
        pytest.skip("wide rows run on tensor cores only")
    if split_k > K // 64:
        pytest.skip("more splits than k-blocks")
    if B > 64 and N * K > 8192 * 7168:
        pytest.skip("one wide full-size shape is enough")
    ws = ssd.workspace(ssd.dec_splitk_workspace_bytes(B, N, K, split_k), dev)
    X, W, R, Y0, Y1, v = _run_both(env, ssd.dec_splitk_gemm, ssd.dec_splitk_gemm_packed, B, N, K,
                                   True, 23, ws=ws, split_k=split_k, use_tc=use_tc)
    assert v[0] == v[1]
    assert torch.equal(Y0, Y1)


@pytest.mark.parametrize("B", [1, 2, 3, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("N,K,residual", [(8192, 7168, False), (7168, 16384, True),
                                          (2048, 1024, False)])
def test_linear_packed_equals_row_major(env, B, N, K, residual):
    torch, ssd, oracle, dev = env
    ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
    X, W, R, Y0, Y1, v = _run_both(env, ssd.dec_linear, ssd.dec_linear_packed, B, N, K,
                                   residual, 24, ws=ws)
    if K >= 12288:  # packed weights: split-K tiles from this K on, at every batch
        assert v[1] in (ssd.VARIANT_SPLITK, ssd.VARIANT_SPLITK_TC)
    else:
        assert v[0] == v[1]
    if v[0] != v[1] or v[1] == ssd.VARIANT_TINY:  # another kernel or summation order
        from split_switched_decode_gb300 import inputs
        y, _ = oracle.linear(inputs.bits(X), inputs.bits(W), None if R is None else inputs.bits(R))
        assert_close(to_f64(oracle, Y1), y, f"packed switch B={B} N={N} K={K}")
    else:
        assert torch.equal(Y0, Y1)


@pytest.mark.parametrize("B", [1, 2, 64])
@pytest.mark.parametrize("N,K,residual", [(8192, 7168, False), (7168, 16384, True)])
def test_linear_packed_full_size_matches_oracle(env, B, N, K, residual):
    """Every row of the packed full-size projection against the fp64 oracle."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    X = inputs.activations(B, K, dev, 25)
    W = inputs.weight(N, K, dev, 25)
    R = inputs.residual(B, N, dev, 25) if residual else None
    Wp = ssd.dec_pack_weight(W)
    Y = torch.empty(B, N, dtype=torch.bfloat16, device=dev)
    ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
    ssd.dec_linear_packed(X, Wp, R, Y, ws)
    torch.cuda.synchronize()
    y, _ = oracle.linear(inputs.bits(X), inputs.bits(W), None if R is None else inputs.bits(R))
    assert_close(to_f64(oracle, Y), y, f"packed B={B} N={N} K={K}")


def test_packed_chained_calls_are_deterministic(env):
    """Packed projections queued back to back (programmatic dependent launches, the next
    call's weight loads overlapping the previous call): bit-identical every time."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    N, K = 8192, 7168
    W = inputs.weight(N, K, dev, 26)
    Wp = ssd.dec_pack_weight(W)
    for B in (1, 4, 64):
        X = inputs.activations(B, K, dev, 26)
        ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
        outs = [torch.empty(B, N, dtype=torch.bfloat16, device=dev) for _ in range(8)]
        for Y in outs:
            ssd.dec_linear_packed(X, Wp, None, Y, ws)
        torch.cuda.synchronize()
        for Y in outs[1:]:
            assert torch.equal(outs[0], Y)
    assert ssd.dec_sync_status() == ssd.DEC_OK


@pytest.mark.parametrize("B", [1, 4, 64])
@pytest.mark.parametrize("N,K", [(8192, 7168), (7168, 16384)])
def test_packed_l2_prefetch_keeps_bits(env, monkeypatch, B, N, K):
    """The optional L2 prefetch of each worker's next k-blocks before its dependency wait
    (DEC_L2PF_KB; one 16 KB bulk prefetch per packed block) writes nothing: the same bits."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    X = inputs.activations(B, K, dev, 27)
    W = inputs.weight(N, K, dev, 27)
    Wp = ssd.dec_pack_weight(W)
    ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
    outs = []
    for kb in ("0", "24"):
        monkeypatch.setenv("DEC_L2PF_KB", kb)
        Y = torch.empty(B, N, dtype=torch.bfloat16, device=dev)
        ssd.dec_splitk_gemm_packed(X, Wp, None, Y, ws, split_k=0, use_tc=1)
        torch.cuda.synchronize()
        assert ssd.dec_sync_status() == ssd.DEC_OK
        outs.append(Y)
    assert torch.equal(outs[0], outs[1])
