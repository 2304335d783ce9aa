"""GPU parity of the wide tensor-core projection: 65..512 rows per call, the shape of
speculative-decoding verification (B sequences x (draft length + 1) tokens; "Hyper
Optimizing Kimi K3 in vLLM", Part 3: Performance Deep Dive, decode with DSpark), where
groups of 64 batch columns share each weight tile and are reduced separately (launches
of at most 256 rows), and from 129 rows the CTA-pair tiles (one launch up to 512 rows;
tests/test_gpu_pair_projection.py covers that kernel on its own)."""
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
    X = inputs.activations(B, K, dev, seed, "wide_x")
    W = inputs.weight(N, K, dev, seed, "wide_w")
    R = inputs.residual(B, N, dev, seed, "wide_r") if residual else None
    Y = torch.empty(B, N, dtype=torch.bfloat16, device=dev)
    return X, W, R, Y


def _ref(X, W, R, rows=None):
    import oracle
    from split_switched_decode_gb300 import inputs
    if rows is not None:
        W = W[rows]
        R = None if R is None else R[:, rows].contiguous()
    y, _ = oracle.linear(inputs.bits(X), inputs.bits(W.contiguous()),
                         None if R is None else inputs.bits(R))
    return y


@pytest.mark.parametrize("B,N,K", [(65, 256, 512), (72, 300, 456), (128, 1000, 1000),
                                   (129, 130, 136), (200, 640, 2048), (256, 512, 1024),
                                   (256, 77, 64), (96, 1, 64), (257, 256, 512),
                                   (300, 300, 456), (512, 512, 1024)])
@pytest.mark.parametrize("split_k", [0, 3])
def test_wide_projection_matches_oracle(env, B, N, K, split_k):
    torch, ssd, oracle, dev = env
    if split_k > (K + 63) // 64:
        pytest.skip("split larger than the k-blocks of a tile")
    X, W, R, Y = _case(env, B, N, K, 20, residual=(B % 2 == 1))
    ws = ssd.workspace(ssd.dec_splitk_workspace_bytes(B, N, K, split_k), dev)
    ssd.dec_splitk_gemm(X, W, R, Y, ws, split_k=split_k, use_tc=1)
    torch.cuda.synchronize()
    # from 129 rows the one-range-per-SM plan runs on CTA-pair tiles, one launch (two
    # k-halves: at least two k-blocks)
    pair = split_k == 0 and B > 128 and K > 64
    assert ssd.dec_last_variant() == (ssd.VARIANT_SPLITK_TC_PAIR if pair else ssd.VARIANT_SPLITK_TC)
    assert ssd.dec_sync_status() == ssd.DEC_OK
    Y1 = Y.clone()
    ssd.dec_splitk_gemm(X, W, R, Y, ws, split_k=split_k, use_tc=1)
    torch.cuda.synchronize()
    assert torch.equal(Y, Y1)
    assert_close(to_f64(oracle, Y), _ref(X, W, R), f"wide B={B} N={N} K={K} S={split_k}")


@pytest.mark.parametrize("B", [72, 128, 256, 512])
@pytest.mark.parametrize("which", ["input", "output"])
def test_wide_full_size_projections(env, B, which):
    """The decode input projection (7168 -> 8192) and the output projection
    (16384 -> 7168 + residual) at speculative-verification row counts through
    dec_linear; every row of Y checked on sampled output columns."""
    torch, ssd, oracle, dev = env
    N, K, res = (8192, 7168, False) if which == "input" else (7168, 16384, True)
    X, W, R, Y = _case(env, B, N, K, 21, residual=res)
    ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
    ssd.dec_linear(X, W, R, Y, ws)
    torch.cuda.synchronize()
    # CTA-pair tiles from 129 rows, and from 65 rows where their clusters (4 CTAs per 256
    # rows of W) cover >= 80 % of the SMs: the input projection's 128 CTAs, not the output
    # projection's 112
    pair = B > 128 or which == "input"
    assert ssd.dec_last_variant() == (ssd.VARIANT_SPLITK_TC_PAIR if pair else
                                      ssd.VARIANT_SPLITK_TC)
    rng = np.random.default_rng(B)
    rows = np.unique(np.concatenate([rng.choice(N, 96, replace=False), [0, 127, 128, N - 1]]))
    assert_close(to_f64(oracle, Y)[:, rows], _ref(X, W, R, rows), f"{which} B={B}")


def test_wide_rows_equal_narrow_calls(env):
    """Rows 0..63 of a 256-row call equal a 64-row call on those rows, bit for bit when
    both use the same split (the column groups are reduced independently)."""
    torch, ssd, oracle, dev = env
    B, N, K = 256, 1024, 2048
    X, W, R, Y = _case(env, B, N, K, 22)
    ws = ssd.workspace(ssd.dec_splitk_workspace_bytes(B, N, K, 4), dev)
    ssd.dec_splitk_gemm(X, W, R, Y, ws, split_k=4, use_tc=1)
    for g in range(4):
        Xg = X[64 * g:64 * g + 64].contiguous()
        Rg = R[64 * g:64 * g + 64].contiguous()
        Yg = torch.empty(64, N, dtype=torch.bfloat16, device=dev)
        wsg = ssd.workspace(ssd.dec_splitk_workspace_bytes(64, N, K, 4), dev)
        ssd.dec_splitk_gemm(Xg, W, Rg, Yg, wsg, split_k=4, use_tc=1)
        torch.cuda.synchronize()
        assert torch.equal(Yg, Y[64 * g:64 * g + 64]), f"column group {g}"


def test_wide_needs_tensor_cores(env):
    torch, ssd, oracle, dev = env
    B, N, K = 65, 128, 64
    X, W, R, Y = _case(env, B, N, K, 23)
    ws = ssd.workspace(ssd.dec_splitk_workspace_bytes(B, N, K, 0), dev)
    with pytest.raises(ssd.DecError):
        ssd.dec_splitk_gemm(X, W, R, Y, ws, use_tc=0)
    Xb = torch.zeros(513, K, dtype=torch.bfloat16, device=dev)
    Yb = torch.empty(513, N, dtype=torch.bfloat16, device=dev)
    with pytest.raises(ssd.DecError):
        ssd.dec_linear(Xb, W, None, Yb, ws)


@pytest.mark.parametrize("B,N,K", [(72, 300, 456), (256, 512, 1024), (160, 1000, 2048)])
def test_wide_last_arriver_reduction(env, monkeypatch, B, N, K):
    """Wide projections with the reduction in each tile's last arriver (DEC_WIDE_DEFER=0)
    instead of the finishing kernel: same results within tolerance, deterministic."""
    torch, ssd, oracle, dev = env
    monkeypatch.setenv("DEC_WIDE_PAIR_MMA", "0")  # the one-CTA tiles' reductions
    monkeypatch.setenv("DEC_WIDE_DEFER", "0")
    X, W, R, Y = _case(env, B, N, K, 24)
    ws = ssd.workspace(ssd.dec_splitk_workspace_bytes(B, N, K, 0), dev)
    ssd.dec_splitk_gemm(X, W, R, Y, ws, use_tc=1)
    torch.cuda.synchronize()
    Y1 = Y.clone()
    ssd.dec_splitk_gemm(X, W, R, Y, ws, use_tc=1)
    torch.cuda.synchronize()
    assert ssd.dec_sync_status() == ssd.DEC_OK
    assert torch.equal(Y, Y1)
    assert_close(to_f64(oracle, Y), _ref(X, W, R), f"wide last-arriver B={B} N={N} K={K}")


@pytest.mark.parametrize("B", [72, 128, 129, 200, 256, 300])
def test_wide_cluster_pair_matches_finishing_kernel(env, monkeypatch, B):
    """A wide projection whose tiles split into two k-halves (64 tiles: the two-halves
    schedule): the halves added inside 2-CTA clusters through distributed shared memory,
    column group by column group, give the same bits as the finishing kernel adding the
    same two partial tiles, and match the oracle."""
    torch, ssd, oracle, dev = env
    monkeypatch.setenv("DEC_WIDE_PAIR_MMA", "0")  # one-CTA tiles, launches of <= 256 rows
    N, K = 8192, 1024
    X, W, R, Y = _case(env, B, N, K, 26)
    ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
    ssd.dec_linear(X, W, R, Y, ws)
    torch.cuda.synchronize()
    assert ssd.dec_sync_status() == ssd.DEC_OK
    monkeypatch.setenv("DEC_PAIR_DSMEM_COLS", "0")
    Y0 = torch.empty_like(Y)
    ssd.dec_linear(X, W, R, Y0, ws)
    torch.cuda.synchronize()
    assert torch.equal(Y, Y0)
    rows = np.unique(np.concatenate([np.linspace(0, N - 1, 160).astype(int), [127, 128]]))
    assert_close(to_f64(oracle, Y)[:, rows], _ref(X, W, R, rows), f"wide pair B={B}")
