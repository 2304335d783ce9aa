"""GPU parity of the tcgen05 tensor-core split-K tiles (swap-AB: weight rows are the
MMA M = 128 dimension, batch columns the MMA N dimension, fp32 accumulator in tensor
memory) against the fp64 oracle, for the projection, the MoE front end and the expert
GEMVs ("Hyper Optimizing Kimi K3 in vLLM", Part 1 / 1 and / 3)."""
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


@pytest.fixture
def force_tc(env):
    torch, ssd, oracle, dev = env
    ssd.dec_set_force_variant(ssd.VARIANT_SPLITK_TC)
    yield
    ssd.dec_set_force_variant(ssd.VARIANT_NONE)


def _case(env, B, N, K, seed, residual=True):
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    X = inputs.activations(B, K, dev, seed)
    W = inputs.weight(N, K, dev, seed)
    R = inputs.residual(B, N, dev, seed) if residual else None
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


@pytest.mark.parametrize("B,N,K", [(16, 256, 128), (3, 300, 456), (5, 129, 64), (8, 1000, 1000),
                                   (17, 640, 2048), (33, 256, 520), (63, 130, 136),
                                   (64, 512, 1024), (1, 300, 456), (2, 128, 8), (16, 1, 64)])
@pytest.mark.parametrize("split_k", [0, 3])
def test_splitk_tensor_core_matches_oracle(env, B, N, K, split_k):
    torch, ssd, oracle, dev = env
    if split_k > (K + 63) // 64:
        pytest.skip("split larger than the k-blocks of a tile")
    X, W, R, Y = _case(env, B, N, K, 12, residual=(B % 2 == 1))
    ws = ssd.workspace(ssd.dec_splitk_workspace_bytes(B, N, K, split_k), dev)
    ssd.dec_splitk_gemm(X, W, R, Y, ws, split_k=split_k, use_tc=1)
    torch.cuda.synchronize()
    assert ssd.dec_last_variant() == ssd.VARIANT_SPLITK_TC
    assert ssd.dec_sync_status() == ssd.DEC_OK
    assert_close(to_f64(oracle, Y), _ref(X, W, R), f"tc B={B} N={N} K={K} S={split_k}")


@pytest.mark.parametrize("B", [4, 16, 32, 64])
def test_tensor_core_full_size_projections(env, force_tc, B):
    torch, ssd, oracle, dev = env
    rng = np.random.default_rng(B)
    for (N, K, res) in ((8192, 7168, False), (7168, 16384, True)):
        X, W, R, Y = _case(env, B, N, K, 0, residual=res)
        ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
        ssd.dec_linear(X, W, R, Y, ws)
        torch.cuda.synchronize()
        assert ssd.dec_last_variant() == ssd.VARIANT_SPLITK_TC
        rows = np.unique(np.concatenate([rng.choice(N, 256, replace=False), [0, N - 1]]))
        assert_close(to_f64(oracle, Y)[:, rows], _ref(X, W, R, torch.as_tensor(rows, device=dev)),
                     f"tc full B={B} N={N} K={K}")


def test_tensor_core_small_integers_exact(env, force_tc):
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    B, N, K = 40, 300, 1000
    g = torch.Generator(device=dev).manual_seed(9)
    Xi = torch.randint(-4, 5, (B, K), device=dev, generator=g).to(torch.bfloat16)
    Wi = torch.randint(-4, 5, (N, K), device=dev, generator=g).to(torch.bfloat16)
    Y = torch.empty(B, N, dtype=torch.bfloat16, device=dev)
    ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
    ssd.dec_linear(Xi, Wi, None, Y, ws)
    torch.cuda.synchronize()
    _, Y_ref = oracle.linear(inputs.bits(Xi), inputs.bits(Wi))
    assert np.array_equal(inputs.bits(Y), Y_ref)
    X = torch.zeros(B, K, dtype=torch.bfloat16, device=dev)
    X[np.arange(B), np.arange(B) * 7] = 1.0
    W = inputs.weight(N, K, dev, 5)
    ssd.dec_linear(X, W, None, Y, ws)
    torch.cuda.synchronize()
    for b in range(B):
        assert torch.equal(Y[b], W[:, 7 * b])


def test_tensor_core_deterministic(env):
    torch, ssd, oracle, dev = env
    B, N, K = 48, 1000, 3000
    X, W, R, Y = _case(env, B, N, K, 13)
    ws = ssd.workspace(ssd.dec_splitk_workspace_bytes(B, N, K, 0), dev)
    outs = []
    for _ in range(3):
        ssd.dec_splitk_gemm(X, W, R, Y, ws, use_tc=1)
        torch.cuda.synchronize()
        outs.append(Y.clone())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    assert_close(to_f64(oracle, outs[0]), _ref(X, W, R), "tc deterministic")


@pytest.mark.parametrize("B", [1, 8, 64])
def test_tensor_core_moe_front(env, force_tc, B):
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    E, L, K, k = 384, 512, 7168, 8
    X = inputs.activations(B, K, dev, 0, "front_x")
    Wc = inputs.weight(E + L, K, dev, 0, "front_w")
    lat = torch.empty(B, L, dtype=torch.bfloat16, device=dev)
    idx = torch.empty(B, k, dtype=torch.int32, device=dev)
    w = torch.empty(B, k, dtype=torch.float32, device=dev)
    rm = torch.empty(ssd.moe_route_map_ints(B, E, k), dtype=torch.int32, device=dev)
    ws = ssd.workspace(ssd.moe_front_workspace_bytes(B, E, L, K), dev)
    ssd.moe_front(X, Wc, E, L, k, lat, idx, w, ws, route_map=rm)
    torch.cuda.synchronize()
    # both front-end paths multiply on tensor cores (one launch, or product + finish)
    assert ssd.dec_last_variant() in (ssd.VARIANT_SPLITK_TC, ssd.VARIANT_FRONT_ONE_LAUNCH)
    ref = oracle.moe_front(inputs.bits(X), inputs.bits(Wc), E, L, k)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert_close(w.cpu().numpy(), ref["w"], "tc front weights")
    assert_close(to_f64(oracle, lat), oracle.bf16_to_f64(ref["latent"]), "tc front latent")
    m = oracle.route_map(ref["idx"], E)
    assert rm.cpu().numpy()[2 * E + 1 + 2 * B * k] == m["num_used"]


@pytest.mark.parametrize("B,k", [(1, 8), (17, 8), (64, 8), (64, 1)])
def test_tensor_core_experts(env, force_tc, B, k):
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    E, H, I = 16, 256, 128
    Wgu, Wd = inputs.expert_bank(E, H, I, dev, 4)
    Wgs, Wds = inputs.shared_expert(H, I, dev, 4)
    X = inputs.activations(B, H, dev, 4, "ex")
    rng = np.random.default_rng(40 + B)
    idx_np = np.stack([rng.choice(E, k, replace=False) for _ in range(B)]).astype(np.int32)
    w_np = (rng.random((B, k)) + 0.05).astype(np.float32)
    w_np /= w_np.sum(1, keepdims=True)
    Y = torch.empty(B, H, dtype=torch.bfloat16, device=dev)
    ws = ssd.workspace(ssd.moe_experts_workspace_bytes(B, E, k, H, I), dev)
    side = torch.cuda.Stream(device=dev)
    ssd.moe_experts(X, torch.from_numpy(idx_np).to(dev), torch.from_numpy(w_np).to(dev), None,
                    Wgu, Wd, Wgs, Wds, Y, ws, side_stream=side)
    torch.cuda.synchronize()
    assert ssd.dec_sync_status() == ssd.DEC_OK
    y_ref, _ = oracle.moe_experts(inputs.bits(X), idx_np, w_np.astype(np.float64),
                                  inputs.bits(Wgu), inputs.bits(Wd), inputs.bits(Wgs),
                                  inputs.bits(Wds))
    assert_close(to_f64(oracle, Y), y_ref, f"tc experts B={B} k={k}")


@pytest.mark.parametrize("B,N,K,split_k", [(64, 512, 1024, 7), (64, 384, 1024, 16),
                                           (33, 300, 2048, 11), (40, 256, 1024, 16),
                                           (8, 200, 1024, 16), (3, 130, 4096, 64)])
def test_many_contributor_tiles(env, B, N, K, split_k):
    """Tiles with many split-K contributors (up to 64), added by the last arriver in
    worker order; bit-identical on repeat."""
    torch, ssd, oracle, dev = env
    X, W, R, Y = _case(env, B, N, K, 16, residual=True)
    ws = ssd.workspace(ssd.dec_splitk_workspace_bytes(B, N, K, split_k), dev)
    ssd.dec_splitk_gemm(X, W, R, Y, ws, split_k=split_k, use_tc=1)
    torch.cuda.synchronize()
    Y1 = Y.clone()
    ssd.dec_splitk_gemm(X, W, R, Y, ws, split_k=split_k, use_tc=1)
    torch.cuda.synchronize()
    assert ssd.dec_sync_status() == ssd.DEC_OK
    assert torch.equal(Y, Y1)
    assert_close(to_f64(oracle, Y), _ref(X, W, R), f"tc B={B} N={N} K={K} S={split_k}")


@pytest.mark.parametrize("B,N,K", [(1, 200, 256), (2, 8192, 7168), (3, 300, 512),
                                   (16, 1000, 1024), (40, 130, 2048), (64, 8192, 7168),
                                   (64, 256, 128)])
def test_cluster_pair_reduction_matches_global_one(env, monkeypatch, B, N, K):
    """Tiles split into two k-halves (split_k = 2, even k-block count): the two halves
    added through distributed shared memory inside a 2-CTA cluster give the same bits as
    the last-arriver reduction through global memory (same order: first half + second),
    and match the oracle."""
    torch, ssd, oracle, dev = env
    monkeypatch.setenv("DEC_PAIR_DSMEM_COLS", "64")
    X, W, R, Y = _case(env, B, N, K, 25, residual=True)
    ws = ssd.workspace(ssd.dec_splitk_workspace_bytes(B, N, K, 2), dev)
    ssd.dec_splitk_gemm(X, W, R, Y, ws, split_k=2, use_tc=1)
    torch.cuda.synchronize()
    assert ssd.dec_sync_status() == ssd.DEC_OK
    monkeypatch.setenv("DEC_PAIR_DSMEM_COLS", "0")
    Y0 = torch.empty_like(Y)
    ssd.dec_splitk_gemm(X, W, R, Y0, ws, split_k=2, use_tc=1)
    torch.cuda.synchronize()
    assert torch.equal(Y, Y0)
    rows = np.unique(np.concatenate([np.linspace(0, N - 1, min(N, 200)).astype(int), [N - 1]]))
    assert_close(to_f64(oracle, Y)[:, rows], _ref(X, W, R, rows), f"pair B={B} N={N} K={K}")
