"""GPU parity of the MoE front end, the routed experts + shared expert, and the L2
prefetch ("Hyper Optimizing Kimi K3 in vLLM", Part 1 / 3 and / 4) against the fp64
oracle, through the C ABI. Expert indices must match bit for bit; floats within the
tolerance of gpu_common."""
import numpy as np
import pytest

from gpu_common import assert_close, to_f64, topk_gap

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


def _run_front(env, X, Wc, E, L, k, probs=True, route_map=True):
    torch, ssd, oracle, dev = env
    B = X.shape[0]
    lat = torch.empty(B, L, dtype=torch.bfloat16, device=dev) if L else None
    idx = torch.full((B, k), -1, dtype=torch.int32, device=dev)
    w = torch.empty(B, k, dtype=torch.float32, device=dev)
    pr = torch.empty(B, E, dtype=torch.float32, device=dev) if probs else None
    rm = torch.full((ssd.moe_route_map_ints(B, E, k),), -7, dtype=torch.int32, device=dev) if route_map else None
    ws = ssd.workspace(ssd.moe_front_workspace_bytes(B, E, L, X.shape[1]), dev)
    ssd.moe_front(X, Wc, E, L, k, lat, idx, w, ws, probs=pr, route_map=rm)
    torch.cuda.synchronize()
    return lat, idx, w, pr, rm


def _check_front(env, X, Wc, E, L, k, what):
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    lat, idx, w, pr, rm = _run_front(env, X, Wc, E, L, k)
    ref = oracle.moe_front(inputs.bits(X), inputs.bits(Wc), E, L, k)
    gi = idx.cpu().numpy()
    if not np.array_equal(gi, ref["idx"]):
        bad = np.where((gi != ref["idx"]).any(1))[0]
        gaps = [topk_gap(ref["logits"][b], k) for b in bad]
        raise AssertionError(f"{what}: top-k differs for tokens {bad.tolist()} "
                             f"(oracle near-tie gaps {gaps})")
    assert_close(w.cpu().numpy(), ref["w"], f"{what} weights")
    assert_close(pr.cpu().numpy(), ref["probs"], f"{what} probs")
    if L:
        assert_close(to_f64(oracle, lat), oracle.bf16_to_f64(ref["latent"]), f"{what} latent")
    m = oracle.route_map(ref["idx"], E)
    r = rm.cpu().numpy()
    B, P = X.shape[0], X.shape[0] * k
    assert np.array_equal(r[:E], m["counts"])
    assert np.array_equal(r[E:2 * E + 1], m["offsets"])
    assert np.array_equal(r[2 * E + 1:2 * E + 1 + P], m["pairs"])
    assert np.array_equal(r[2 * E + 1 + P:2 * E + 1 + 2 * P], m["pos"])
    assert r[2 * E + 1 + 2 * P] == m["num_used"]
    assert np.array_equal(r[2 * E + 2 + 2 * P:2 * E + 2 + 2 * P + m["num_used"]], m["used"])
    return ref


@pytest.mark.parametrize("B", [1, 8, 64])
def test_moe_front_full_size(env, B):
    """X[B,7168] x Wcat[384+512,7168], softmax over 384, top-8, renormalised."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    E, L, K, k = 384, 512, 7168, 8
    X = inputs.activations(B, K, dev, 0, "front_x")
    Wc = inputs.weight(E + L, K, dev, 0, "front_w")
    _check_front(env, X, Wc, E, L, k, f"front B={B}")


@pytest.mark.parametrize("B,E,L,K,k", [(1, 40, 24, 200, 3), (5, 130, 0, 456, 16),
                                       (33, 512, 8, 64, 1), (64, 16, 100, 1032, 16),
                                       (2, 1, 0, 8, 1), (64, 512, 0, 128, 16),
                                       (8, 512, 512, 136, 16)])
def test_moe_front_ragged_shapes(env, B, E, L, K, k):
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    X = inputs.activations(B, K, dev, 1, "fx")
    Wc = inputs.randn_bf16((E + L, K), 0.2, dev, 1, "fw", E, L, K)
    _check_front(env, X, Wc, E, L, k, f"front B={B} E={E} L={L} K={K} k={k}")


@pytest.mark.parametrize("B", [1, 2, 3, 7, 8, 9])
def test_moe_front_cluster_route_map_equals_counter_path(env, monkeypatch, B):
    """The two-launch front end (DEC_FRONT_FUSED=0: product kernel + finishing kernel):
    up to 8 tokens, the finishing kernel's router CTAs form one thread-block cluster
    and CTA 0 builds the route map from the ids the others put in its shared memory;
    DEC_FRONT_CLUSTER=0 builds it in the CTA that routes the last token instead. Every
    output is bit-identical, and both match the oracle (B = 9 takes the counter path
    either way)."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    monkeypatch.setenv("DEC_FRONT_FUSED", "0")
    E, L, K, k = 384, 512, 7168, 8
    X = inputs.activations(B, K, dev, 8, "cfx")
    Wc = inputs.weight(E + L, K, dev, 8, "cfw")
    ref = _check_front(env, X, Wc, E, L, k, f"front cluster B={B}")
    a = _run_front(env, X, Wc, E, L, k)
    monkeypatch.setenv("DEC_FRONT_CLUSTER", "0")
    c = _run_front(env, X, Wc, E, L, k)
    for x, y, name in zip(a, c, ["latent", "idx", "w", "probs", "route map"]):
        assert torch.equal(x, y), name
    assert ssd.dec_sync_status() == ssd.DEC_OK
    assert np.array_equal(c[1].cpu().numpy(), ref["idx"])


@pytest.mark.parametrize("B,E,L,K,k", [(1, 384, 512, 7168, 8), (2, 384, 512, 7168, 8),
                                       (3, 384, 512, 7168, 8), (4, 384, 512, 7168, 8),
                                       (5, 384, 512, 7168, 8), (8, 384, 512, 7168, 8),
                                       (17, 384, 512, 7168, 8), (33, 384, 512, 7168, 8),
                                       (64, 384, 512, 7168, 8), (64, 384, 512, 7168, 16),
                                       (5, 130, 0, 456, 16), (33, 512, 8, 64, 1),
                                       (64, 16, 100, 1032, 16), (2, 1, 0, 8, 1),
                                       # clusters of 4 and 8 CTAs: more than 4 tokens per CTA
                                       (17, 40, 24, 256, 4), (40, 100, 20, 512, 8),
                                       (64, 384, 512, 512, 8), (3, 40, 24, 256, 4)])
def test_moe_front_one_launch_and_two_launch_paths(env, monkeypatch, B, E, L, K, k):
    """The one-launch front end (clusters reduce the split-K partials on chip, arrival
    counters elect the routing CTAs) and the two-launch path both match the oracle: the
    same top-k ids and route map bit for bit, latent and weights within tolerance. The
    one-launch path repeated on the same workspace gives the same bits (fixed reduction
    order; its arrival counters are back at zero after each call). Without the full
    softmax the one-launch path routes by candidate filtering and ranking instead of k
    warp rounds: the same ids, weights and route map, bit for bit."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    X = inputs.activations(B, K, dev, 13, "pfx")
    Wc = inputs.randn_bf16((E + L, K), 0.02 if K > 1000 else 0.2, dev, 13, "pfw", E, L, K)
    monkeypatch.setenv("DEC_FRONT_FUSED", "1")
    _check_front(env, X, Wc, E, L, k, f"one-launch front B={B} E={E} L={L} K={K} k={k}")
    assert ssd.dec_last_variant() == ssd.VARIANT_FRONT_ONE_LAUNCH  # no silent fallback
    a = _run_front(env, X, Wc, E, L, k)
    b = _run_front(env, X, Wc, E, L, k)
    for x, y, name in zip(a, b, ["latent", "idx", "w", "probs", "route map"]):
        if x is not None:
            assert torch.equal(x, y), f"one-launch {name} not repeatable"
    f = _run_front(env, X, Wc, E, L, k, probs=False)
    for i, name in [(0, "latent"), (1, "idx"), (2, "w"), (4, "route map")]:
        if a[i] is not None:
            assert torch.equal(a[i], f[i]), f"filtered routing: {name} differs"
    monkeypatch.setenv("DEC_FRONT_FUSED", "0")
    _check_front(env, X, Wc, E, L, k, f"two-launch front B={B} E={E} L={L} K={K} k={k}")
    assert ssd.dec_last_variant() == ssd.VARIANT_SPLITK_TC
    c = _run_front(env, X, Wc, E, L, k)
    assert torch.equal(a[1], c[1]) and torch.equal(a[4], c[4]), "paths route differently"
    assert ssd.dec_sync_status() == ssd.DEC_OK


@pytest.mark.parametrize("B", [1, 9, 16, 17, 33, 64])
@pytest.mark.parametrize("stages", ["4", "2", "8"])
def test_moe_front_one_launch_chained_calls_are_deterministic(env, monkeypatch, B, stages):
    """24 one-launch front ends queued back to back on one stream (each may start loading
    weights while the previous one finishes) with several stage-ring depths: every call
    gives bit-identical outputs to the first, and the first matches the oracle."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    monkeypatch.setenv("DEC_FRONT_FUSED", "1")
    monkeypatch.setenv("DEC_FRONT_STAGES", stages)
    E, L, K, k = 384, 512, 7168, 8
    X = inputs.activations(B, K, dev, 14, "chx")
    Wc = inputs.weight(E + L, K, dev, 14, "chw")
    lat = torch.empty(B, L, dtype=torch.bfloat16, device=dev)
    ws = ssd.workspace(ssd.moe_front_workspace_bytes(B, E, L, K), dev)
    outs = []
    for _ in range(24):
        idx = torch.empty(B, k, dtype=torch.int32, device=dev)
        w = torch.empty(B, k, dtype=torch.float32, device=dev)
        # entries of used[] past num_used are left as they are: pre-fill them alike
        rm = torch.full((ssd.moe_route_map_ints(B, E, k),), -7, dtype=torch.int32, device=dev)
        lat_i = torch.empty_like(lat)
        ssd.moe_front(X, Wc, E, L, k, lat_i, idx, w, ws, route_map=rm)
        assert ssd.dec_last_variant() == ssd.VARIANT_FRONT_ONE_LAUNCH
        outs.append((lat_i, idx, w, rm))
    torch.cuda.synchronize()
    assert ssd.dec_sync_status() == ssd.DEC_OK
    for i, o in enumerate(outs[1:]):
        for x, y, name in zip(outs[0], o, ["latent", "idx", "w", "route map"]):
            assert torch.equal(x, y), f"call {i + 1}: {name} differs from the first call"
    ref = oracle.moe_front(inputs.bits(X), inputs.bits(Wc), E, L, k)
    assert np.array_equal(outs[0][1].cpu().numpy(), ref["idx"])
    assert_close(outs[0][2].cpu().numpy(), ref["w"], f"chained B={B} weights")


@pytest.mark.parametrize("B", [1, 4, 5, 8, 9, 17, 64])
def test_moe_front_single_and_grouped_routing_agree(env, monkeypatch, B):
    """The one-launch front end routes up to DEC_FRONT_SINGLE_B tokens in one CTA (a warp
    per token, several tokens per warp beyond 8) and larger batches per token group with a
    second counter electing the route-map builder. Forcing either way for every batch
    gives bit-identical outputs, with and without the full softmax, matching the oracle."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    monkeypatch.setenv("DEC_FRONT_FUSED", "1")
    E, L, K, k = 384, 512, 7168, 8
    X = inputs.activations(B, K, dev, 15, "sgx")
    Wc = inputs.weight(E + L, K, dev, 15, "sgw")
    ref = oracle.moe_front(inputs.bits(X), inputs.bits(Wc), E, L, k)
    m = oracle.route_map(ref["idx"], E)
    outs = {}
    for single in ["0", "8", "64"]:
        monkeypatch.setenv("DEC_FRONT_SINGLE_B", single)
        for probs in (False, True):
            outs[(single, probs)] = _run_front(env, X, Wc, E, L, k, probs=probs)
            assert ssd.dec_last_variant() == ssd.VARIANT_FRONT_ONE_LAUNCH
    assert ssd.dec_sync_status() == ssd.DEC_OK
    a = outs[("8", False)]
    assert np.array_equal(a[1].cpu().numpy(), ref["idx"])
    assert_close(a[2].cpu().numpy(), ref["w"], f"B={B} weights")
    P = B * k
    r = a[4].cpu().numpy()
    assert np.array_equal(r[:2 * E + 1 + 2 * P + 1],
                          np.concatenate([m["counts"], m["offsets"], m["pairs"], m["pos"],
                                          [m["num_used"]]]))
    for key, o in outs.items():
        for i, name in [(0, "latent"), (1, "idx"), (2, "w"), (4, "route map")]:
            assert torch.equal(a[i], o[i]), f"single_b={key[0]} probs={key[1]}: {name}"


def test_moe_front_filtered_routing_ties_and_many_candidates(env, monkeypatch):
    """Routing without the full softmax (candidates above a lower bound, exact ranks):
    (a) 32 copies of each of 4 router rows: the 32 copies of the largest logit are the
    candidates, the 8 lowest experts among them win, equal weights 1/8; (b) all router
    rows zero: 128 equal logits, more candidates than the ranking keeps, so the warp
    falls back to k rounds: experts 0..7, weights 1/8; (c) planted duplicate rows as in
    the softmax-path tie test. Every case matches the oracle bit for bit on the ids."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    monkeypatch.setenv("DEC_FRONT_FUSED", "1")
    B, E, L, K, k = 16, 128, 16, 512, 8
    X = inputs.activations(B, K, dev, 16, "ftx")
    Wc = inputs.weight(E + L, K, dev, 16, "ftw")
    base = [inputs.randn_bf16((K,), 0.5, dev, 16, f"fb{i}") for i in range(4)]
    Wa = Wc.clone()
    for r in range(E):  # one 128-row tile: copies accumulate in the same order
        Wa[r] = base[r % 4]
    for name, W in [("copies", Wa), ("zeros", None), ("pairs", None)]:
        if name == "zeros":
            W = Wc.clone()
            W[:E] = 0
        elif name == "pairs":
            W = Wc.clone()
            big = inputs.randn_bf16((K,), 0.5, dev, 16, "fbig")
            W[9] = big
            W[40] = big
            W[20] = -big
            W[33] = -big
        lat, idx, w, pr, rm = _run_front(env, X, W, E, L, k, probs=False)
        assert ssd.dec_last_variant() == ssd.VARIANT_FRONT_ONE_LAUNCH
        ref = oracle.moe_front(inputs.bits(X), inputs.bits(W), E, L, k)
        assert np.array_equal(idx.cpu().numpy(), ref["idx"]), name
        assert_close(w.cpu().numpy(), ref["w"], f"{name} weights")
        if name == "zeros":
            assert np.array_equal(idx.cpu().numpy(), np.tile(np.arange(k), (B, 1)))
            assert torch.all(w == 1.0 / k)
        if name == "copies":
            # the winning row group: 8 lowest of its 16 copies, equal weights
            for b in range(B):
                g = int(ref["idx"][b, 0]) % 4
                assert idx[b].tolist() == [g + 4 * i for i in range(k)], idx[b].tolist()
                assert torch.all(w[b] == 1.0 / k)
        m = oracle.route_map(ref["idx"], E)
        r = rm.cpu().numpy()
        assert np.array_equal(r[:E], m["counts"]) and np.array_equal(r[E:2 * E + 1], m["offsets"])
    assert ssd.dec_sync_status() == ssd.DEC_OK


def test_moe_front_ties_go_to_lower_index(env):
    """Duplicate router rows in one tile give bit-identical fp32 logits: lower index first.
    All-zero router rows give equal logits: experts 0..k-1, weights 1/k, probs 1/E."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    B, E, L, K, k = 16, 64, 16, 512, 4
    X = inputs.activations(B, K, dev, 2, "tx")
    Wc = inputs.weight(E + L, K, dev, 2, "tw")
    big = inputs.randn_bf16((K,), 0.5, dev, 2, "big")
    Wc[9] = big
    Wc[40] = big          # same tile (rows 0..127): identical accumulation order
    Wc[20] = -big
    Wc[33] = -big
    lat, idx, w, pr, rm = _run_front(env, X, Wc, E, L, k)
    ref = oracle.moe_front(inputs.bits(X), inputs.bits(Wc), E, L, k)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    tied = 0
    for b in range(B):
        top2 = sorted(ref["idx"][b, :2].tolist())
        if top2 in ([9, 40], [20, 33]):  # the planted pair leads this token: a real tie
            tied += 1
            assert idx[b, :2].tolist() == top2, idx[b].tolist()
            assert w[b, 0].item() == w[b, 1].item()
    assert tied >= B // 2
    Wz = Wc.clone()
    Wz[:E] = 0
    lat, idx, w, pr, rm = _run_front(env, X, Wz, E, L, k)
    assert np.array_equal(idx.cpu().numpy(), np.tile(np.arange(k), (B, 1)))
    assert torch.all(w == 1.0 / k) and torch.all(pr == 1.0 / E)


def test_moe_front_optional_outputs(env):
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    B, E, L, K, k = 3, 96, 32, 256, 6
    X = inputs.activations(B, K, dev, 3, "ox")
    Wc = inputs.weight(E + L, K, dev, 3, "ow")
    lat, idx, w, pr, rm = _run_front(env, X, Wc, E, L, k, probs=False, route_map=False)
    ref = oracle.moe_front(inputs.bits(X), inputs.bits(Wc), E, L, k)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    assert_close(w.cpu().numpy(), ref["w"], "weights without optional outputs")


# ------------------------------------------------------------------ experts ----

def _routing(B, E, k, seed):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(B)]).astype(np.int32)
    w = rng.random((B, k)).astype(np.float32) + 0.05
    w /= w.sum(1, keepdims=True)
    return idx, w.astype(np.float32)


def _run_experts(env, X, idx, w, Wgu, Wd, Wgs, Wds, rm=None, side=True, side_ctas=0, ws=None,
                 packed=False):
    torch, ssd, oracle, dev = env
    B, H = X.shape
    E, twoI, _ = Wgu.shape
    k = idx.shape[1]
    Y = torch.empty(B, H, dtype=torch.bfloat16, device=dev)
    if ws is None:
        ws = ssd.workspace(ssd.moe_experts_workspace_bytes(B, E, k, H, twoI // 2), dev)
    ss = torch.cuda.Stream(device=dev) if side else None
    ssd.moe_experts(X, idx, w, rm, Wgu, Wd, Wgs, Wds, Y, ws, side_stream=ss, side_max_ctas=side_ctas,
                    packed=packed)
    torch.cuda.synchronize()
    assert ssd.dec_sync_status() == ssd.DEC_OK
    return Y


@pytest.mark.parametrize("B,k", [(1, 8), (4, 2), (17, 8), (64, 8), (64, 1)])
@pytest.mark.parametrize("shared,side", [(True, True), (True, False), (False, False)])
def test_moe_experts_small_bank(env, B, k, shared, side):
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    E, H, I = 16, 256, 128
    Wgu, Wd = inputs.expert_bank(E, H, I, dev, 4)
    Wgs, Wds = inputs.shared_expert(H, I, dev, 4) if shared else (None, None)
    X = inputs.activations(B, H, dev, 4, "ex")
    idx_np, w_np = _routing(B, E, k, 40 + B)
    idx = torch.from_numpy(idx_np).to(dev)
    w = torch.from_numpy(w_np).to(dev)
    Y = _run_experts(env, X, idx, w, Wgu, Wd, Wgs, Wds, side=side)
    y_ref, _ = oracle.moe_experts(inputs.bits(X), idx_np, w_np.astype(np.float64),
                                  inputs.bits(Wgu), inputs.bits(Wd),
                                  None if Wgs is None else inputs.bits(Wgs),
                                  None if Wds is None else inputs.bits(Wds))
    assert_close(to_f64(oracle, Y), y_ref, f"experts B={B} k={k} shared={shared} side={side}")


def _packed_bank_reference(torch, Wgu, Wd):
    """Tile-packed banks by their definition: gate/up blocks of 64 gate rows then the 64
    matching up rows, down blocks of 128 rows, each block 64 k wide, blocks in (expert,
    tile, k-block) order."""
    E, twoI, H = Wgu.shape
    I = twoI // 2
    g = Wgu[:, :I].reshape(E, I // 64, 64, H)
    u = Wgu[:, I:].reshape(E, I // 64, 64, H)
    rows = torch.cat([g, u], dim=2).reshape(-1, 128, H // 64, 64)
    gu = rows.permute(0, 2, 1, 3).contiguous().view(E, twoI, H)
    d = Wd.reshape(-1, 128, I // 64, 64).permute(0, 2, 1, 3).contiguous().view(E, H, I)
    return gu, d


@pytest.mark.parametrize("E,H,I", [(3, 256, 128), (1, 384, 192), (2, 128, 64)])
def test_pack_expert_weights_layout(env, E, H, I):
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    Wgu, Wd = inputs.expert_bank(E, H, I, dev, 30)
    gu, d = ssd.dec_pack_expert_weights(Wgu, Wd)
    torch.cuda.synchronize()
    rgu, rd = _packed_bank_reference(torch, Wgu, Wd)
    assert torch.equal(gu, rgu) and torch.equal(d, rd)
    # one element of each by the block formula
    e, t, r, k = E - 1, I // 64 - 1, 70, H - 1  # an up row of the last tile
    blk = (e * (I // 64) + t) * (H // 64) + k // 64
    assert gu.view(-1)[blk * 8192 + r * 64 + k % 64].item() == Wgu[e, I + t * 64 + r - 64, k].item()


@pytest.mark.parametrize("B,k", [(1, 8), (4, 2), (17, 8), (64, 8), (64, 1)])
@pytest.mark.parametrize("shared,side,with_map", [(True, True, False), (True, False, True),
                                                  (False, False, False)])
def test_moe_experts_packed_equals_row_major(env, B, k, shared, side, with_map):
    """Packed expert banks run the same tiles in the same order: bit-identical outputs,
    with and without the shared expert, side stream and a given route map."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    E, H, I = 16, 256, 128
    Wgu, Wd = inputs.expert_bank(E, H, I, dev, 31)
    Wgs, Wds = inputs.shared_expert(H, I, dev, 31) if shared else (None, None)
    Pgu, Pd = ssd.dec_pack_expert_weights(Wgu, Wd)
    Pgs, Pds = ssd.dec_pack_expert_weights(Wgs[None], Wds[None]) if shared else (None, None)
    X = inputs.activations(B, H, dev, 31, "pex")
    idx_np, w_np = _routing(B, E, k, 50 + B)
    idx = torch.from_numpy(idx_np).to(dev)
    w = torch.from_numpy(w_np).to(dev)
    rm = _host_route_map(oracle, idx_np, E, dev) if with_map else None
    Y0 = _run_experts(env, X, idx, w, Wgu, Wd, Wgs, Wds, rm=rm, side=side)
    Y1 = _run_experts(env, X, idx, w, Pgu, Pd, None if Pgs is None else Pgs[0],
                      None if Pds is None else Pds[0], rm=rm, side=side, packed=True)
    assert torch.equal(Y0, Y1)


@pytest.mark.parametrize("B,E,k", [(64, 512, 16), (3, 1, 1), (64, 2, 2)])
def test_moe_experts_routing_extremes(env, B, E, k):
    """The largest routing the library takes (64 tokens x 16 slots over 512 experts:
    1024 (token, slot) entries, most experts with one or two tokens), a single expert
    with one slot, and two experts that every token uses."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    H, I = 128, 64
    Wgu, Wd = inputs.expert_bank(E, H, I, dev, 9, "extreme_bank")
    Wgs, Wds = inputs.shared_expert(H, I, dev, 9, "extreme_shared")
    X = inputs.activations(B, H, dev, 9, "extreme_x")
    idx_np, w_np = _routing(B, E, k, 90 + B + E)
    idx = torch.from_numpy(idx_np).to(dev)
    w = torch.from_numpy(w_np).to(dev)
    Y = _run_experts(env, X, idx, w, Wgu, Wd, Wgs, Wds, side=True)
    y_ref, _ = oracle.moe_experts(inputs.bits(X), idx_np, w_np.astype(np.float64),
                                  inputs.bits(Wgu), inputs.bits(Wd), inputs.bits(Wgs),
                                  inputs.bits(Wds))
    assert_close(to_f64(oracle, Y), y_ref, f"experts extremes B={B} E={E} k={k}")


def _host_route_map(oracle, idx_np, E, dev):
    """The route-map layout of the header, assembled from the oracle's counting sort."""
    import torch
    m = oracle.route_map(idx_np, E)
    B, k = idx_np.shape
    used = np.zeros(E, dtype=np.int32)
    used[:m["num_used"]] = m["used"]
    rm = np.concatenate([m["counts"], m["offsets"], m["pairs"], m["pos"],
                         np.array([m["num_used"]], dtype=np.int32), used]).astype(np.int32)
    return torch.from_numpy(rm).to(dev)


@pytest.mark.parametrize("B,k", [(1, 8), (5, 3), (17, 8), (64, 8), (64, 16)])
@pytest.mark.parametrize("shared,side", [(True, True), (True, False), (False, False)])
def test_fused_combine_equals_combine_launch(env, monkeypatch, B, k, shared, side):
    """With a route map, the combine can run inside the down launches' epilogues (the
    tile that completes a (token, 128-row block) adds it up, DEC_FUSED_COMBINE=1) or as
    its own launch: the same bits either way, both within tolerance of the oracle, and a
    second call on the same workspace (counters back at zero) gives the same bits."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    E, H, I = 24, 384, 128
    Wgu, Wd = inputs.expert_bank(E, H, I, dev, 12, "fc_bank")
    Wgs, Wds = inputs.shared_expert(H, I, dev, 12, "fc_shared") if shared else (None, None)
    X = inputs.activations(B, H, dev, 12, "fc_x")
    idx_np, w_np = _routing(B, E, k, 120 + B)
    idx = torch.from_numpy(idx_np).to(dev)
    w = torch.from_numpy(w_np).to(dev)
    rm = _host_route_map(oracle, idx_np, E, dev)
    ws = ssd.workspace(ssd.moe_experts_workspace_bytes(B, E, k, H, I), dev)
    # the fused combine keeps the shared expert on its own launches: compare like with like
    monkeypatch.setenv("DEC_SHARED_IN_ROUTED", "0")
    monkeypatch.setenv("DEC_FUSED_COMBINE", "1")
    Y1 = _run_experts(env, X, idx, w, Wgu, Wd, Wgs, Wds, rm=rm, side=side, ws=ws)
    Y1b = _run_experts(env, X, idx, w, Wgu, Wd, Wgs, Wds, rm=rm, side=side, ws=ws)
    monkeypatch.setenv("DEC_FUSED_COMBINE", "0")
    Y0 = _run_experts(env, X, idx, w, Wgu, Wd, Wgs, Wds, rm=rm, side=side)
    assert torch.equal(Y1, Y0)
    assert torch.equal(Y1, Y1b)
    y_ref, _ = oracle.moe_experts(inputs.bits(X), idx_np, w_np.astype(np.float64),
                                  inputs.bits(Wgu), inputs.bits(Wd),
                                  None if Wgs is None else inputs.bits(Wgs),
                                  None if Wds is None else inputs.bits(Wds))
    assert_close(to_f64(oracle, Y1), y_ref, f"fused combine B={B} k={k} shared={shared}")


def test_moe_experts_every_token_on_one_expert(env):
    """64 tokens on one expert: the widest grouped tile (4 activation boxes)."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    E, H, I, B = 6, 384, 192, 64
    Wgu, Wd = inputs.expert_bank(E, H, I, dev, 5)
    X = inputs.activations(B, H, dev, 5, "one")
    idx_np = np.tile(np.array([[3, 1]], np.int32), (B, 1))
    w_np = np.tile(np.array([[0.75, 0.25]], np.float32), (B, 1))
    Y = _run_experts(env, X, torch.from_numpy(idx_np).to(dev), torch.from_numpy(w_np).to(dev),
                     Wgu, Wd, None, None, side=False)
    y_ref, _ = oracle.moe_experts(inputs.bits(X), idx_np, w_np.astype(np.float64),
                                  inputs.bits(Wgu), inputs.bits(Wd))
    assert_close(to_f64(oracle, Y), y_ref, "one expert for all tokens")


def test_route_map_from_front_equals_rebuilt(env):
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    B, E, L, K, k, I = 12, 32, 0, 256, 4, 64
    X = inputs.activations(B, K, dev, 6, "rx")
    Wc = inputs.weight(E, K, dev, 6, "rw")
    _, idx, w, _, rm = _run_front(env, X, Wc, E, L, k)
    Wgu, Wd = inputs.expert_bank(E, K, I, dev, 6)
    Y1 = _run_experts(env, X, idx, w, Wgu, Wd, None, None, rm=rm, side=False)
    Y2 = _run_experts(env, X, idx, w, Wgu, Wd, None, None, rm=None, side=False)
    assert torch.equal(Y1, Y2)


def test_side_cta_cap_changes_schedule_not_result(env):
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    E, H, I, B, k = 8, 256, 128, 6, 2
    Wgu, Wd = inputs.expert_bank(E, H, I, dev, 7)
    Wgs, Wds = inputs.shared_expert(H, I, dev, 7)
    X = inputs.activations(B, H, dev, 7, "cap")
    idx_np, w_np = _routing(B, E, k, 7)
    idx, w = torch.from_numpy(idx_np).to(dev), torch.from_numpy(w_np).to(dev)
    y_ref, _ = oracle.moe_experts(inputs.bits(X), idx_np, w_np.astype(np.float64),
                                  inputs.bits(Wgu), inputs.bits(Wd), inputs.bits(Wgs),
                                  inputs.bits(Wds))
    for cap in (1, 3, 40):
        Y = _run_experts(env, X, idx, w, Wgu, Wd, Wgs, Wds, side=True, side_ctas=cap)
        assert_close(to_f64(oracle, Y), y_ref, f"side cap {cap}")


@pytest.fixture(scope="module")
def big_layer(env):
    """The synthetic MoE decode layer: 384 experts (gate/up 2x2048x7168, down 7168x2048)
    plus a shared expert of the same shape and the 384+512-row front end (~34 GB)."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    E, H, I, L = 384, 7168, 2048, 512
    Wgu, Wd = inputs.expert_bank(E, H, I, dev, 0, "bank")
    Wgs, Wds = inputs.shared_expert(H, I, dev, 0, "bank_shared")
    Wc = inputs.weight(E + L, H, dev, 0, "front_w")
    yield dict(Wgu=Wgu, Wd=Wd, Wgs=Wgs, Wds=Wds, Wc=Wc, E=E, H=H, I=I, L=L)
    del Wgu, Wd
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B,with_map", [(1, True), (1, False), (2, False), (4, False),
                                        (8, False), (16, False), (32, False), (64, True),
                                        (64, False)])
def test_moe_layer_full_size(env, big_layer, B, with_map):
    """Front end -> routed experts + shared expert (side stream) on the full-size layer,
    with the route map from the front end or built by the experts' gather launch, end
    to end against the oracle: the GPU's top-k ids must equal the oracle front end's on
    the same X bit for bit, and the reference layer output uses the oracle's own fp64
    routing weights. Up to 8 tokens (the first, the last and spread between) are checked
    with their experts copied to the host."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    g = big_layer
    E, H, I, L, k = g["E"], g["H"], g["I"], g["L"], 8
    X = inputs.activations(B, H, dev, 0, "layer_x")
    lat, idx, w, _, rm = _run_front(env, X, g["Wc"], E, L, k)
    Y = _run_experts(env, X, idx, w, g["Wgu"], g["Wd"], g["Wgs"], g["Wds"],
                     rm=rm if with_map else None, side=True)
    xb = inputs.bits(X)
    ref = oracle.moe_front(xb, inputs.bits(g["Wc"]), E, L, k)
    gi = idx.cpu().numpy()
    if not np.array_equal(gi, ref["idx"]):
        bad = np.where((gi != ref["idx"]).any(1))[0]
        gaps = [topk_gap(ref["logits"][b], k) for b in bad]
        raise AssertionError(f"layer B={B}: top-k differs from the oracle for tokens "
                             f"{bad.tolist()} (oracle near-tie gaps {gaps})")
    assert_close(w.cpu().numpy(), ref["w"], f"layer B={B} routing weights")
    assert_close(to_f64(oracle, lat), oracle.bf16_to_f64(ref["latent"]), f"layer B={B} latent")
    Yf = to_f64(oracle, Y)
    gs, ds = inputs.bits(g["Wgs"]), inputs.bits(g["Wds"])
    n_tok = min(B, 8)
    tokens = sorted({0, B - 1} | {(t * (B - 1)) // max(n_tok - 1, 1) for t in range(n_tok)})
    assert len(tokens) == n_tok
    y_ref = np.empty((len(tokens), H))
    for t, b in enumerate(tokens):
        yp = np.empty((1, k, H))
        for j in range(k):
            e = int(ref["idx"][b, j])
            _, yp[0, j] = oracle.expert_mlp(xb[b], inputs.bits(g["Wgu"][e]), inputs.bits(g["Wd"][e]))
        _, s = oracle.expert_mlp(xb[b], gs, ds)
        y_ref[t] = oracle.combine(ref["w"][b:b + 1], yp, s[None, :])[0][0]
    assert_close(Yf[tokens], y_ref, f"MoE layer B={B}")


@pytest.mark.parametrize("B", [1, 8, 64])
def test_moe_layer_packed_full_size_equals_row_major(env, big_layer, B):
    """The full-size layer on tile-packed expert banks (moe_layer_packed) against the
    row-major layer, which test_moe_layer_full_size checks against the oracle: the same
    top-k ids, route map, latent and output bits."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    g = big_layer
    if "Pgu" not in g:
        g["Pgu"], g["Pd"] = ssd.dec_pack_expert_weights(g["Wgu"], g["Wd"])
        ps, pd = ssd.dec_pack_expert_weights(g["Wgs"][None], g["Wds"][None])
        g["Pgs"], g["Pds"] = ps[0], pd[0]
    E, H, I, L, k = g["E"], g["H"], g["I"], g["L"], 8
    X = inputs.activations(B, H, dev, 32, "player_x")
    outs = []
    for packed in (False, True):
        lat = torch.empty(B, L, dtype=torch.bfloat16, device=dev)
        idx = torch.empty(B, k, dtype=torch.int32, device=dev)
        w = torch.empty(B, k, dtype=torch.float32, device=dev)
        rm = torch.full((ssd.moe_route_map_ints(B, E, k),), -7, dtype=torch.int32, device=dev)
        Y = torch.empty(B, H, dtype=torch.bfloat16, device=dev)
        ws = ssd.workspace(ssd.moe_layer_workspace_bytes(B, E, L, H, I, k), dev)
        Wgu, Wd, Wgs, Wds = ((g["Pgu"], g["Pd"], g["Pgs"], g["Pds"]) if packed else
                             (g["Wgu"], g["Wd"], g["Wgs"], g["Wds"]))
        ssd.moe_layer(X, g["Wc"], E, L, k, Wgu, Wd, Wgs, Wds, lat, idx, w, Y, ws, route_map=rm,
                      side_stream=torch.cuda.Stream(device=dev), packed=packed)
        torch.cuda.synchronize()
        assert ssd.dec_sync_status() == ssd.DEC_OK
        outs.append((lat, idx, w, rm, Y))
    for a, b, name in zip(outs[0], outs[1], ["latent", "idx", "w", "route map", "Y"]):
        assert torch.equal(a, b), name


def test_l2_prefetch_does_not_change_results(env):
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    B, N, K = 4, 2048, 2048
    X = inputs.activations(B, K, dev, 8)
    W = inputs.weight(N, K, dev, 8)
    Y1 = torch.empty(B, N, dtype=torch.bfloat16, device=dev)
    Y2 = torch.empty_like(Y1)
    ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
    ssd.dec_linear(X, W, None, Y1, ws)
    side = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(side):
        ssd.l2_prefetch(W, max_ctas=4, stream=side)
    ssd.l2_prefetch(W)  # also on the main stream, any byte count
    ssd.l2_prefetch(W, nbytes=W.numel() * 2 - 40)
    torch.cuda.synchronize()
    ssd.dec_linear(X, W, None, Y2, ws)
    torch.cuda.synchronize()
    assert torch.equal(Y1, Y2)


@pytest.mark.parametrize("B", [1, 16, 64])
def test_prefetch_during_communication_phase_keeps_results(env, B):
    """The output projection behind a simulated communication phase, with the second
    half of its weights prefetched into L2 on a side stream meanwhile: bit-identical
    output, and the phase ends on time."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    N, K = 7168, 4096
    X = inputs.activations(B, K, dev, 10)
    W = inputs.weight(N, K, dev, 10)
    R = inputs.residual(B, N, dev, 10)
    Y1 = torch.empty(B, N, dtype=torch.bfloat16, device=dev)
    Y2 = torch.empty_like(Y1)
    ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
    ssd.dec_sim_comm_wait(20_000)
    ssd.dec_linear(X, W, R, Y1, ws)
    side = torch.cuda.Stream(device=dev)
    main = torch.cuda.current_stream()
    fork, join = torch.cuda.Event(), torch.cuda.Event()
    fork.record(main)
    side.wait_event(fork)
    flat = W.view(-1)
    ssd.l2_prefetch(flat[flat.numel() // 2:], max_ctas=64, stream=side)
    join.record(side)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(main)
    ssd.dec_sim_comm_wait(2_000_000)
    b.record(main)
    main.wait_event(join)
    ssd.dec_linear(X, W, R, Y2, ws)
    torch.cuda.synchronize()
    assert ssd.dec_sync_status() == ssd.DEC_OK
    assert torch.equal(Y1, Y2)
    assert 1.9 <= a.elapsed_time(b) <= 50.0  # ms: the 2 ms phase ends on time


@pytest.mark.parametrize("B", [1, 8, 64])
def test_moe_experts_one_launch_equals_two_launches_full_size(env, big_layer, monkeypatch, B):
    """The full-size routed experts in one launch (down tiles waiting for their expert's
    gate/up tiles) and in two launches on whole tiles compute every tile in the same k
    order in one CTA: the same bits."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    g = big_layer
    E, H, I, L, k = g["E"], g["H"], g["I"], g["L"], 8
    X = inputs.activations(B, H, dev, 33, "one_launch_x")
    _, idx, w, _, rm = _run_front(env, X, g["Wc"], E, L, k)
    outs = []
    monkeypatch.setenv("DEC_SHARED_IN_ROUTED", "0")  # the shared expert on its own launches
    for one in ("1", "0"):
        monkeypatch.setenv("DEC_EXPERT_ONE_LAUNCH", one)
        monkeypatch.setenv("DEC_EXPERT_DYN_MIN_TILES", "0")
        outs.append(_run_experts(env, X, idx, w, g["Wgu"], g["Wd"], g["Wgs"], g["Wds"], rm=rm,
                                 side=True))
    assert torch.equal(outs[0], outs[1])


def test_invalid_routing_is_reported_not_faulted(env):
    """An out-of-range or repeated expert index passed without a route map is caught by
    the rebuild kernel: empty map, DEC_ERR_INVALID_ARG from dec_sync_status."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    E, H, I, B = 8, 256, 64, 3
    Wgu, Wd = inputs.expert_bank(E, H, I, dev, 9)
    X = inputs.activations(B, H, dev, 9, "bad")
    w = torch.full((B, 2), 0.5, dtype=torch.float32, device=dev)
    Y = torch.empty(B, H, dtype=torch.bfloat16, device=dev)
    ws = ssd.workspace(ssd.moe_experts_workspace_bytes(B, E, 2, H, I), dev)
    for bad in ([[0, 1], [2, 8], [3, 4]], [[0, 1], [5, 5], [3, 4]], [[-1, 1], [2, 3], [3, 4]]):
        idx = torch.tensor(bad, dtype=torch.int32, device=dev)
        ssd.moe_experts(X, idx, w, None, Wgu, Wd, None, None, Y, ws)
        assert ssd.dec_sync_status() == ssd.DEC_ERR_INVALID_ARG
    idx = torch.tensor([[0, 1], [2, 7], [3, 4]], dtype=torch.int32, device=dev)
    ssd.moe_experts(X, idx, w, None, Wgu, Wd, None, None, Y, ws)
    assert ssd.dec_sync_status() == ssd.DEC_OK
    y_ref, _ = oracle.moe_experts(inputs.bits(X), idx.cpu().numpy(), w.cpu().numpy().astype(np.float64),
                                  inputs.bits(Wgu), inputs.bits(Wd))
    assert_close(to_f64(oracle, Y), y_ref, "valid routing after invalid ones")


@pytest.mark.parametrize("B,k", [(1, 4), (5, 2), (17, 4), (64, 8)])
@pytest.mark.parametrize("side", [True, False])
def test_moe_layer_matches_oracle(env, B, k, side):
    """moe_layer (front end while the shared expert streams on the side stream, then
    the routed experts): routing bit-exact against the oracle, latent, weights and Y
    within tolerance, route map equal to the rebuilt one."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    E, L, H, I = 40, 24, 256, 128
    X = inputs.activations(B, H, dev, 11, "layer")
    Wc = inputs.weight(E + L, H, dev, 11, "layer_wc")
    Wgu, Wd = inputs.expert_bank(E, H, I, dev, 11, "layer_bank")
    Wgs, Wds = inputs.shared_expert(H, I, dev, 11, "layer_shared")
    lat = torch.empty(B, L, dtype=torch.bfloat16, device=dev)
    idx = torch.full((B, k), -1, dtype=torch.int32, device=dev)
    w = torch.empty(B, k, dtype=torch.float32, device=dev)
    rm = torch.full((ssd.moe_route_map_ints(B, E, k),), -7, dtype=torch.int32, device=dev)
    Y = torch.empty(B, H, dtype=torch.bfloat16, device=dev)
    ws = ssd.workspace(ssd.moe_layer_workspace_bytes(B, E, L, H, I, k), dev)
    ss = torch.cuda.Stream(device=dev) if side else None
    ssd.moe_layer(X, Wc, E, L, k, Wgu, Wd, Wgs, Wds, lat, idx, w, Y, ws, route_map=rm,
                  side_stream=ss)
    torch.cuda.synchronize()
    assert ssd.dec_sync_status() == ssd.DEC_OK
    ref = oracle.moe_front(inputs.bits(X), inputs.bits(Wc), E, L, k)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"]), "top-k differs from the oracle"
    assert_close(w.cpu().numpy().astype(np.float64), ref["w"], "routing weights")
    assert_close(to_f64(oracle, lat), oracle.bf16_to_f64(ref["latent"]), "latent")
    m = oracle.route_map(ref["idx"], E)
    r, P = rm.cpu().numpy(), B * k
    assert np.array_equal(r[:E], m["counts"])
    assert np.array_equal(r[E:2 * E + 1], m["offsets"])
    assert np.array_equal(r[2 * E + 1:2 * E + 1 + P], m["pairs"])
    assert np.array_equal(r[2 * E + 1 + P:2 * E + 1 + 2 * P], m["pos"])
    assert r[2 * E + 1 + 2 * P] == m["num_used"]
    y_ref, _ = oracle.moe_experts(inputs.bits(X), ref["idx"], ref["w"], inputs.bits(Wgu),
                                  inputs.bits(Wd), inputs.bits(Wgs), inputs.bits(Wds))
    assert_close(to_f64(oracle, Y), y_ref, f"moe_layer B={B}")
