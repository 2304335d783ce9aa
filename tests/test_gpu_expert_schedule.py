"""GPU parity of the schedules of the routed-expert launches, through the C ABI.

One launch (the default on tensor cores): every gate/up and down tile claimed at run
time from one counter, whole tiles only, each down tile loading its expert's A once that
expert's gate/up tiles have published it. Two launches with the whole-tile schedule: each
CTA streams a static share of the tiles, then claims the rest one at a time. Both
compute every tile over all of its k-blocks in one CTA, so they give the same bits as
each other whatever the claims, the static share, the number of CTAs (side-stream cap),
the layout of the banks or the route-map source. Checked here: agreement with the fp64
oracle; those equalities; the counters (cleared by the gather launch) starting from zero
on every call that reuses a workspace; the fused combine; an invalid routing reported,
not faulted.
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


SCHEDULES = {
    # gate/up and down in one launch (the default)
    "one_launch": {"DEC_EXPERT_ONE_LAUNCH": "1"},
    # two launches, whole tiles at every batch size (by default from 6.5 tiles per CTA)
    "two_launch_whole_tiles": {"DEC_EXPERT_ONE_LAUNCH": "0", "DEC_EXPERT_DYN_MIN_TILES": "0"},
}


@pytest.fixture(params=sorted(SCHEDULES))
def whole_tiles(request, monkeypatch):
    monkeypatch.delenv("DEC_EXPERT_DYN", raising=False)
    for k, v in SCHEDULES[request.param].items():
        monkeypatch.setenv(k, v)
    monkeypatch.schedule = request.param
    return monkeypatch


def _routing(B, E, k, seed):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(B)]).astype(np.int32)
    w = rng.random((B, k)).astype(np.float32) + 0.05
    w /= w.sum(1, keepdims=True)
    return idx, w.astype(np.float32)


def _host_route_map(oracle, idx_np, E, dev):
    import torch
    m = oracle.route_map(idx_np, E)
    used = np.zeros(E, dtype=np.int32)
    used[:m["num_used"]] = m["used"]
    rm = np.concatenate([m["counts"], m["offsets"], m["pairs"], m["pos"],
                         np.array([m["num_used"]], dtype=np.int32), used]).astype(np.int32)
    return torch.from_numpy(rm).to(dev)


def _run(env, X, idx, w, Wgu, Wd, Wgs, Wds, rm=None, side=True, side_ctas=0, ws=None,
         packed=False):
    torch, ssd, oracle, dev = env
    B, H = X.shape
    E, twoI, _ = Wgu.shape
    k = idx.shape[1]
    Y = torch.full((B, H), float("nan"), dtype=torch.bfloat16, device=dev)
    if ws is None:
        ws = ssd.workspace(ssd.moe_experts_workspace_bytes(B, E, k, H, twoI // 2), dev)
    ss = torch.cuda.Stream(device=dev) if side else None
    ssd.moe_experts(X, idx, w, rm, Wgu, Wd, Wgs, Wds, Y, ws, side_stream=ss,
                    side_max_ctas=side_ctas, packed=packed)
    torch.cuda.synchronize()
    assert ssd.dec_sync_status() == ssd.DEC_OK
    return Y


def _problem(env, B, E, H, I, k, seed, shared=True):
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    Wgu, Wd = inputs.expert_bank(E, H, I, dev, seed, "wt_bank")
    Wgs, Wds = inputs.shared_expert(H, I, dev, seed, "wt_shared") if shared else (None, None)
    X = inputs.activations(B, H, dev, seed, "wt_x")
    idx_np, w_np = _routing(B, E, k, 700 + seed + B)
    return dict(Wgu=Wgu, Wd=Wd, Wgs=Wgs, Wds=Wds, X=X, idx_np=idx_np, w_np=w_np,
                idx=torch.from_numpy(idx_np).to(dev), w=torch.from_numpy(w_np).to(dev))


def _oracle_y(env, pb):
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    y, _ = oracle.moe_experts(inputs.bits(pb["X"]), pb["idx_np"], pb["w_np"].astype(np.float64),
                              inputs.bits(pb["Wgu"]), inputs.bits(pb["Wd"]),
                              None if pb["Wgs"] is None else inputs.bits(pb["Wgs"]),
                              None if pb["Wds"] is None else inputs.bits(pb["Wds"]))
    return y


@pytest.mark.parametrize("B,k", [(1, 8), (4, 2), (17, 8), (64, 8), (64, 16)])
@pytest.mark.parametrize("shared,side,with_map", [(True, True, True), (True, False, False),
                                                  (False, False, True)])
def test_whole_tile_schedule_matches_oracle(env, whole_tiles, B, k, shared, side, with_map):
    torch, ssd, oracle, dev = env
    E, H, I = 24, 384, 256
    pb = _problem(env, B, E, H, I, k, 1, shared)
    rm = _host_route_map(oracle, pb["idx_np"], E, dev) if with_map else None
    Y = _run(env, pb["X"], pb["idx"], pb["w"], pb["Wgu"], pb["Wd"], pb["Wgs"], pb["Wds"], rm=rm,
             side=side)
    assert_close(to_f64(oracle, Y), _oracle_y(env, pb),
                 f"whole tiles B={B} k={k} shared={shared} side={side} map={with_map}")


@pytest.mark.parametrize("B,k", [(5, 3), (33, 8), (64, 8)])
def test_whole_tile_result_does_not_depend_on_the_schedule(env, whole_tiles, B, k):
    """One launch, and two launches with static shares from none (every tile claimed) to
    all, each with different CTA counts for the routed launches (side-stream caps): the
    same bits every time."""
    torch, ssd, oracle, dev = env
    E, H, I = 32, 256, 192
    pb = _problem(env, B, E, H, I, k, 2)
    rm = _host_route_map(oracle, pb["idx_np"], E, dev)
    whole_tiles.setenv("DEC_SHARED_IN_ROUTED", "0")  # routed schedules only; shared on its own
    outs = []
    for one in ("1", "0"):
        whole_tiles.setenv("DEC_EXPERT_ONE_LAUNCH", one)
        whole_tiles.setenv("DEC_EXPERT_DYN_MIN_TILES", "0")
        for share in (("230",) if one == "1" else ("1", "128", "230", "256")):
            whole_tiles.setenv("DEC_EXPERT_DYN", share)
            for cap in (0, 7, 60):
                outs.append(_run(env, pb["X"], pb["idx"], pb["w"], pb["Wgu"], pb["Wd"],
                                 pb["Wgs"], pb["Wds"], rm=rm, side=True, side_ctas=cap))
    for Y in outs[1:]:
        assert torch.equal(outs[0], Y)
    assert_close(to_f64(oracle, outs[0]), _oracle_y(env, pb), f"schedule-independent B={B}")


def test_whole_tile_claim_counters_restart_on_every_call(env, whole_tiles):
    """One workspace for a sequence of calls (route map given or rebuilt by the gather,
    different routings): each call's claim counters start from zero, so repeating a call
    repeats its bits, and a call after many others still matches the oracle."""
    torch, ssd, oracle, dev = env
    E, H, I, B, k = 20, 256, 128, 9, 4
    pa = _problem(env, B, E, H, I, k, 3)
    pb = _problem(env, B, E, H, I, k, 4)
    ws = ssd.workspace(ssd.moe_experts_workspace_bytes(B, E, k, H, I), dev)
    rma = _host_route_map(oracle, pa["idx_np"], E, dev)
    seq = []
    for pr, rm in ((pa, rma), (pb, None), (pa, None), (pb, None), (pa, rma)):
        seq.append(_run(env, pr["X"], pr["idx"], pr["w"], pr["Wgu"], pr["Wd"], pr["Wgs"],
                        pr["Wds"], rm=rm, side=True, ws=ws))
    assert torch.equal(seq[0], seq[2]) and torch.equal(seq[0], seq[4])
    assert torch.equal(seq[1], seq[3])
    assert_close(to_f64(oracle, seq[4]), _oracle_y(env, pa), "after a sequence of calls")
    assert_close(to_f64(oracle, seq[3]), _oracle_y(env, pb), "second routing")


def test_whole_tile_equals_packed_and_stream_k_within_tolerance(env, whole_tiles):
    """Tile-packed banks give the same bits as row-major ones under the whole-tile
    schedule; the stream-K schedule (another summation split) agrees within the oracle
    tolerance."""
    torch, ssd, oracle, dev = env
    E, H, I, B, k = 16, 384, 128, 40, 8
    pb = _problem(env, B, E, H, I, k, 5)
    Pgu, Pd = ssd.dec_pack_expert_weights(pb["Wgu"], pb["Wd"])
    Pgs, Pds = ssd.dec_pack_expert_weights(pb["Wgs"][None], pb["Wds"][None])
    Y0 = _run(env, pb["X"], pb["idx"], pb["w"], pb["Wgu"], pb["Wd"], pb["Wgs"], pb["Wds"])
    Y1 = _run(env, pb["X"], pb["idx"], pb["w"], Pgu, Pd, Pgs[0], Pds[0], packed=True)
    assert torch.equal(Y0, Y1)
    whole_tiles.setenv("DEC_EXPERT_ONE_LAUNCH", "0")
    whole_tiles.setenv("DEC_EXPERT_DYN", "0")
    Y2 = _run(env, pb["X"], pb["idx"], pb["w"], pb["Wgu"], pb["Wd"], pb["Wgs"], pb["Wds"])
    y = _oracle_y(env, pb)
    assert_close(to_f64(oracle, Y0), y, "whole tiles")
    assert_close(to_f64(oracle, Y2), y, "stream-K")


@pytest.mark.parametrize("B,k", [(5, 3), (64, 8)])
@pytest.mark.parametrize("shared", [True, False])
def test_whole_tile_fused_combine_equals_combine_launch(env, whole_tiles, B, k, shared):
    torch, ssd, oracle, dev = env
    E, H, I = 24, 384, 128
    pb = _problem(env, B, E, H, I, k, 6, shared)
    rm = _host_route_map(oracle, pb["idx_np"], E, dev)
    ws = ssd.workspace(ssd.moe_experts_workspace_bytes(B, E, k, H, I), dev)
    whole_tiles.setenv("DEC_SHARED_IN_ROUTED", "0")  # the fused combine keeps it on its own
    whole_tiles.setenv("DEC_FUSED_COMBINE", "1")
    Y1 = _run(env, pb["X"], pb["idx"], pb["w"], pb["Wgu"], pb["Wd"], pb["Wgs"], pb["Wds"], rm=rm,
              ws=ws)
    Y1b = _run(env, pb["X"], pb["idx"], pb["w"], pb["Wgu"], pb["Wd"], pb["Wgs"], pb["Wds"], rm=rm,
               ws=ws)
    whole_tiles.setenv("DEC_FUSED_COMBINE", "0")
    Y0 = _run(env, pb["X"], pb["idx"], pb["w"], pb["Wgu"], pb["Wd"], pb["Wgs"], pb["Wds"], rm=rm)
    assert torch.equal(Y1, Y0) and torch.equal(Y1, Y1b)
    assert_close(to_f64(oracle, Y1), _oracle_y(env, pb), f"fused combine B={B}")


def test_whole_tile_invalid_routing_is_reported_not_faulted(env, whole_tiles):
    """An invalid routing leaves an empty route map (no tile to claim): the calls end with
    DEC_ERR_INVALID_ARG, and a valid call on the same workspace afterwards is correct."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    E, H, I, B = 8, 256, 64, 3
    Wgu, Wd = inputs.expert_bank(E, H, I, dev, 9)
    X = inputs.activations(B, H, dev, 9, "bad")
    w = torch.full((B, 2), 0.5, dtype=torch.float32, device=dev)
    Y = torch.empty(B, H, dtype=torch.bfloat16, device=dev)
    ws = ssd.workspace(ssd.moe_experts_workspace_bytes(B, E, 2, H, I), dev)
    for bad in ([[0, 1], [2, 8], [3, 4]], [[0, 1], [5, 5], [3, 4]]):
        idx = torch.tensor(bad, dtype=torch.int32, device=dev)
        ssd.moe_experts(X, idx, w, None, Wgu, Wd, None, None, Y, ws)
        assert ssd.dec_sync_status() == ssd.DEC_ERR_INVALID_ARG
    idx_np = np.array([[0, 1], [2, 7], [3, 4]], dtype=np.int32)
    ssd.moe_experts(X, torch.from_numpy(idx_np).to(dev), w, None, Wgu, Wd, None, None, Y, ws)
    assert ssd.dec_sync_status() == ssd.DEC_OK
    y_ref, _ = oracle.moe_experts(inputs.bits(X), idx_np, w.cpu().numpy().astype(np.float64),
                                  inputs.bits(Wgu), inputs.bits(Wd))
    assert_close(to_f64(oracle, Y), y_ref, "valid routing after invalid ones")


@pytest.mark.parametrize("B,k", [(1, 8), (4, 2), (17, 8), (64, 8), (64, 1)])
@pytest.mark.parametrize("with_map,packed", [(True, False), (False, True)])
def test_shared_expert_inside_the_routed_launch(env, monkeypatch, B, k, with_map, packed):
    """The shared expert as one more group of the one-launch routed experts (the default):
    its gate/up and down tiles claimed with the routed ones, its activation rows appended
    to the gathered ones, its output read by the combine. Against the oracle, and within
    the same tolerance of the shared expert on its own launches (another summation split)."""
    torch, ssd, oracle, dev = env
    E, H, I = 24, 384, 256
    pb = _problem(env, B, E, H, I, k, 8)
    rm = _host_route_map(oracle, pb["idx_np"], E, dev) if with_map else None
    Wgu, Wd, Wgs, Wds = pb["Wgu"], pb["Wd"], pb["Wgs"], pb["Wds"]
    if packed:
        Wgu, Wd = ssd.dec_pack_expert_weights(Wgu, Wd)
        gs, ds = ssd.dec_pack_expert_weights(Wgs[None], Wds[None])
        Wgs, Wds = gs[0], ds[0]
    monkeypatch.setenv("DEC_EXPERT_ONE_LAUNCH", "1")
    monkeypatch.setenv("DEC_SHARED_IN_ROUTED", "1")
    Y1 = _run(env, pb["X"], pb["idx"], pb["w"], Wgu, Wd, Wgs, Wds, rm=rm, side=True,
              packed=packed)
    Y1b = _run(env, pb["X"], pb["idx"], pb["w"], Wgu, Wd, Wgs, Wds, rm=rm, side=False,
               packed=packed)
    assert torch.equal(Y1, Y1b)  # the side stream is not used: the same launches
    monkeypatch.setenv("DEC_SHARED_IN_ROUTED", "0")
    Y0 = _run(env, pb["X"], pb["idx"], pb["w"], Wgu, Wd, Wgs, Wds, rm=rm, side=True,
              packed=packed)
    y = _oracle_y(env, pb)
    assert_close(to_f64(oracle, Y1), y, f"shared in routed B={B} k={k}")
    assert_close(to_f64(oracle, Y0), y, f"shared on the side B={B} k={k}")


def test_shared_expert_inside_with_invalid_routing_is_reported(env, monkeypatch):
    """An invalid routing leaves an empty route map; with the shared expert inside the
    routed launch, that launch then holds the shared expert's tiles only. The call ends
    with DEC_ERR_INVALID_ARG and faults nothing; a valid call on the same workspace
    afterwards is correct."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    monkeypatch.setenv("DEC_EXPERT_ONE_LAUNCH", "1")
    monkeypatch.setenv("DEC_SHARED_IN_ROUTED", "1")
    E, H, I, B = 8, 256, 64, 3
    Wgu, Wd = inputs.expert_bank(E, H, I, dev, 10)
    Wgs, Wds = inputs.shared_expert(H, I, dev, 10)
    X = inputs.activations(B, H, dev, 10, "bad_shared")
    w = torch.full((B, 2), 0.5, dtype=torch.float32, device=dev)
    Y = torch.empty(B, H, dtype=torch.bfloat16, device=dev)
    ws = ssd.workspace(ssd.moe_experts_workspace_bytes(B, E, 2, H, I), dev)
    bad = torch.tensor([[0, 1], [2, 9], [3, 4]], dtype=torch.int32, device=dev)
    ssd.moe_experts(X, bad, w, None, Wgu, Wd, Wgs, Wds, Y, ws)
    assert ssd.dec_sync_status() == ssd.DEC_ERR_INVALID_ARG
    idx_np = np.array([[0, 1], [2, 7], [3, 4]], dtype=np.int32)
    ssd.moe_experts(X, torch.from_numpy(idx_np).to(dev), w, None, Wgu, Wd, Wgs, Wds, Y, ws)
    assert ssd.dec_sync_status() == ssd.DEC_OK
    y_ref, _ = oracle.moe_experts(inputs.bits(X), idx_np, w.cpu().numpy().astype(np.float64),
                                  inputs.bits(Wgu), inputs.bits(Wd), inputs.bits(Wgs),
                                  inputs.bits(Wds))
    assert_close(to_f64(oracle, Y), y_ref, "valid routing after an invalid one")
