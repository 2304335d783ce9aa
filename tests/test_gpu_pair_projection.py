"""GPU parity of the CTA-pair tensor-core projection (65..512 rows in one launch): the
speculative-verification shape (sequences x (draft length + 1) tokens; "Hyper Optimizing
Kimi K3 in vLLM", Part 3: Performance Deep Dive, decode with DSpark) where two SMs share
each MMA of 256 weight rows and the two k-halves of every weight tile are added inside a
4-CTA cluster. Every case is compared with the fp64 oracle: ragged N and K, an odd number
of 128-row tiles (a half-empty last slice), the smallest k-range (two k-blocks), one MMA
of N = 128 or 256 or two of 256 per K step (up to 128 / 256 / 512 rows), residual or not,
vector and scalar stores."""
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


def _case(env, B, N, K, seed, residual):
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    X = inputs.activations(B, K, dev, seed, "pair_x")
    W = inputs.weight(N, K, dev, seed, "pair_w")
    R = inputs.residual(B, N, dev, seed, "pair_r") if residual else None
    Y = torch.full((B, N), float("nan"), dtype=torch.bfloat16, device=dev)
    return X, W, R, Y


def _ref(X, W, R, tokens=None):
    import oracle
    from split_switched_decode_gb300 import inputs
    if tokens is not None:
        X = X[tokens].contiguous()
        R = None if R is None else R[tokens].contiguous()
    y, _ = oracle.linear(inputs.bits(X), inputs.bits(W), None if R is None else inputs.bits(R))
    return y


@pytest.mark.parametrize("B,N,K,residual", [
    (129, 256, 128, True),     # smallest batch of the kernel, two k-blocks (one per half)
    (160, 384, 456, False),    # three tiles: the second slice's odd tile is empty
    (200, 1, 128, True),       # one output row
    (255, 300, 1000, True),    # ragged N (scalar stores), ragged last k-block
    (256, 640, 2048, False),   # one MMA per K step, full
    (257, 256, 512, True),     # two MMAs per K step, one column in the second
    (300, 130, 136, False),    # odd k-block count: halves of 1 and 2 blocks
    (384, 512, 1024, True),    # two MMAs of N = 192 per K step, full
    (385, 256, 512, False),    # two MMAs of N = 256, one column past 384
    (511, 1000, 520, False),
    (512, 256, 2048, True),    # two MMAs, full
])
def test_pair_projection_matches_oracle(env, B, N, K, residual):
    torch, ssd, oracle, dev = env
    X, W, R, Y = _case(env, B, N, K, 40, residual)
    ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
    ssd.dec_linear(X, W, R, Y, ws)
    torch.cuda.synchronize()
    assert ssd.dec_last_variant() == ssd.VARIANT_SPLITK_TC_PAIR
    assert ssd.dec_sync_status() == ssd.DEC_OK
    Y1 = Y.clone()
    ssd.dec_linear(X, W, R, Y, ws)
    torch.cuda.synchronize()
    assert torch.equal(Y, Y1), "repeated call changed bits"
    assert_close(to_f64(oracle, Y), _ref(X, W, R), f"pair B={B} N={N} K={K}")


@pytest.mark.parametrize("B,N,K,residual", [
    (65, 8192, 128, True),     # one MMA of N = 128 per K step, two k-blocks
    (100, 8064, 456, False),   # ragged K
    (128, 8100, 1000, True),   # ragged N: per-thread stores, a partly empty last tile
    (128, 8192, 2048, False),
])
def test_pair_projection_128_columns_matches_oracle(env, B, N, K, residual):
    """65..128 rows on CTA-pair tiles of N = 128 (each CTA stages 64 activation rows per
    k-block), taken where the clusters cover >= 80 % of the SMs (about 8192 rows of W)."""
    torch, ssd, oracle, dev = env
    X, W, R, Y = _case(env, B, N, K, 45, residual)
    ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
    ssd.dec_linear(X, W, R, Y, ws)
    torch.cuda.synchronize()
    assert ssd.dec_last_variant() == ssd.VARIANT_SPLITK_TC_PAIR
    assert ssd.dec_sync_status() == ssd.DEC_OK
    assert_close(to_f64(oracle, Y), _ref(X, W, R), f"pair128 B={B} N={N} K={K}")


def test_pair_tiles_below_129_rows_need_enough_clusters(env):
    """Below 129 rows a shape whose clusters would cover too few SMs stays on one-CTA
    tiles (the HBM-bound calls need the SMs more than the shared activation boxes)."""
    torch, ssd, oracle, dev = env
    B, N, K = 100, 1024, 1024
    X, W, R, Y = _case(env, B, N, K, 46, True)
    ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
    ssd.dec_linear(X, W, R, Y, ws)
    torch.cuda.synchronize()
    assert ssd.dec_last_variant() == ssd.VARIANT_SPLITK_TC
    assert_close(to_f64(oracle, Y), _ref(X, W, R), "one-CTA tiles B=100")


@pytest.mark.parametrize("B,which", [(512, "input"), (300, "output"), (136, "input")])
def test_pair_full_size_projection_every_row(env, B, which):
    """The decode input projection (7168 -> 8192) and the output projection (16384 ->
    7168 + residual) at verification row counts: every output row, on tokens that cover
    both CTAs of each pair MMA, both MMAs and both k-halves' column ranges."""
    torch, ssd, oracle, dev = env
    N, K, res = (8192, 7168, False) if which == "input" else (7168, 16384, True)
    X, W, R, Y = _case(env, B, N, K, 41, res)
    ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
    ssd.dec_linear(X, W, R, Y, ws)
    torch.cuda.synchronize()
    assert ssd.dec_last_variant() == ssd.VARIANT_SPLITK_TC_PAIR
    assert ssd.dec_sync_status() == ssd.DEC_OK
    cand = [0, 1, 127, 128, 129, 255, 256, 257, 383, 384, 511, B // 2, B - 1]
    tokens = sorted({t for t in cand if t < B})
    assert_close(to_f64(oracle, Y)[tokens], _ref(X, W, R, tokens), f"pair full {which} B={B}")


@pytest.mark.parametrize("B", [200, 300])
def test_pair_unaligned_output_rows_use_per_thread_stores(env, B):
    """Y and R views one element off a 16-byte boundary (N % 8 == 0): no TMA tiles for
    them, the per-thread stores instead; same values as the aligned call."""
    torch, ssd, oracle, dev = env
    N, K = 512, 1024
    X, W, R, Y = _case(env, B, N, K, 47, True)
    ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
    ssd.dec_linear(X, W, R, Y, ws)
    Ybuf = torch.full((B * N + 8,), float("nan"), dtype=torch.bfloat16, device=dev)
    Rbuf = torch.empty(B * N + 8, dtype=torch.bfloat16, device=dev)
    Yu = Ybuf[1:1 + B * N].view(B, N)
    Ru = Rbuf[1:1 + B * N].view(B, N)
    Ru.copy_(R)
    ssd.dec_linear(X, W, Ru, Yu, ws)
    torch.cuda.synchronize()
    assert ssd.dec_last_variant() == ssd.VARIANT_SPLITK_TC_PAIR
    assert ssd.dec_sync_status() == ssd.DEC_OK
    assert torch.equal(Yu, Y)
    assert_close(to_f64(oracle, Yu), _ref(X, W, R), f"pair unaligned B={B}")


def test_pair_packed_weights_equal_row_major(env):
    """Tile-packed W gives the same bits as row-major W (same boxes, same MMA order)."""
    torch, ssd, oracle, dev = env
    B, N, K = 400, 1024, 2048
    X, W, R, Y0 = _case(env, B, N, K, 42, True)
    Y1 = torch.empty_like(Y0)
    ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
    ssd.dec_linear(X, W, R, Y0, ws)
    ssd.dec_linear_packed(X, ssd.dec_pack_weight(W), R, Y1, ws)
    torch.cuda.synchronize()
    assert ssd.dec_last_variant() == ssd.VARIANT_SPLITK_TC_PAIR
    assert torch.equal(Y0, Y1)
    tokens = [0, 199, 200, 255, 256, 399]
    assert_close(to_f64(oracle, Y1)[tokens], _ref(X, W, R, tokens), "pair packed")


def test_pair_chained_calls_read_fresh_inputs(env):
    """Back-to-back calls on one stream (programmatic dependent launch: weights may be
    loaded before the previous kernel ends, activations only after): each call's output
    equals the same call made alone, also when one call's output is the next one's
    input."""
    torch, ssd, oracle, dev = env
    B, N, K = 320, 512, 512
    X, W, R, Y = _case(env, B, N, K, 43, True)
    W2 = W.clone()
    ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
    Ya = torch.empty_like(Y)
    Yb = torch.empty_like(Y)
    ssd.dec_linear(X, W, R, Ya, ws)
    ssd.dec_linear(Ya, W2, None, Yb, ws)  # N == K: the output feeds the next call
    torch.cuda.synchronize()
    Ya_alone = torch.empty_like(Y)
    ssd.dec_linear(X, W, R, Ya_alone, ws)
    torch.cuda.synchronize()
    Yb_alone = torch.empty_like(Y)
    ssd.dec_linear(Ya_alone, W2, None, Yb_alone, ws)
    torch.cuda.synchronize()
    assert torch.equal(Ya, Ya_alone)
    assert torch.equal(Yb, Yb_alone)
    assert_close(to_f64(oracle, Yb), _ref(Ya, W2, None), "pair chained")


@pytest.mark.parametrize("B", [200, 512])
def test_pair_and_one_cta_tiles_agree_with_oracle(env, monkeypatch, B):
    """The same call on CTA-pair tiles and on one-CTA tiles (DEC_WIDE_PAIR_MMA=0, launches
    of at most 256 rows): both within tolerance of the oracle; the summation order
    differs, so bits may differ."""
    torch, ssd, oracle, dev = env
    N, K = 1024, 3072
    X, W, R, Y = _case(env, B, N, K, 44, True)
    ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
    ssd.dec_linear(X, W, R, Y, ws)
    torch.cuda.synchronize()
    assert ssd.dec_last_variant() == ssd.VARIANT_SPLITK_TC_PAIR
    monkeypatch.setenv("DEC_WIDE_PAIR_MMA", "0")
    Y0 = torch.empty_like(Y)
    ssd.dec_linear(X, W, R, Y0, ws)
    torch.cuda.synchronize()
    assert ssd.dec_last_variant() == ssd.VARIANT_SPLITK_TC
    ref = _ref(X, W, R)
    assert_close(to_f64(oracle, Y), ref, f"pair B={B}")
    assert_close(to_f64(oracle, Y0), ref, f"one-CTA tiles B={B}")
