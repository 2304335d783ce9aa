"""Ordering of dependent launches ("Hyper Optimizing Kimi K3 in vLLM", Part 2 / 3
"Validate correctness": an activation read moved ahead of a synchronisation wait
survives simple functional checks).

Kernels are launched with programmatic dependent launch: a kernel may start, and
stream its weights, while the previous kernel of the stream is still running; its
activation reads must wait. These tests chain projections whose inputs are the
previous call's outputs, back to back on one stream, into buffers that still hold
the previous round's values, so a read issued before the wait would see stale data
and miss the oracle.
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
    return torch, ssd, oracle, dev


VARIANTS = {"tiny": 0, "splitk": 1, "splitk_tc": 2}


@pytest.mark.parametrize("variant", ["tiny", "splitk", "splitk_tc"])
@pytest.mark.parametrize("B", [1, 2, 5, 64])
def test_chained_projections_read_fresh_activations(env, variant, B):
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    if variant == "tiny" and B > 2:
        pytest.skip("tiny kernel is for B <= 2")
    ssd.dec_set_force_variant(VARIANTS[variant])
    try:
        N = K = 2048
        depth = 6
        Ws = [inputs.weight(N, K, dev, 80 + i) for i in range(depth)]
        bufs = [torch.empty(B, K, dtype=torch.bfloat16, device=dev) for _ in range(depth + 1)]
        ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
        for rnd in range(3):
            bufs[0].copy_(inputs.activations(B, K, dev, 90 + rnd))
            for i in range(depth):
                ssd.dec_linear(bufs[i], Ws[i], None, bufs[i + 1], ws)
            torch.cuda.synchronize()
            for i in range(depth):
                y_ref, _ = oracle.linear(inputs.bits(bufs[i]), inputs.bits(Ws[i]))
                assert_close(to_f64(oracle, bufs[i + 1]), y_ref, f"{variant} B={B} round {rnd} link {i}")
    finally:
        ssd.dec_set_force_variant(-1)


def test_front_then_experts_reads_fresh_route_map(env):
    """moe_front writes the route map the grouped expert launch reads first."""
    torch, ssd, oracle, dev = env
    from split_switched_decode_gb300 import inputs
    B, E, L, K, k, I = 16, 32, 16, 512, 4, 128
    Wc = inputs.weight(E + L, K, dev, 95)
    Wgu, Wd = inputs.expert_bank(E, K, I, dev, 95)
    lat = torch.empty(B, L, dtype=torch.bfloat16, device=dev)
    idx = torch.empty(B, k, dtype=torch.int32, device=dev)
    w = torch.empty(B, k, dtype=torch.float32, device=dev)
    rm = torch.empty(ssd.moe_route_map_ints(B, E, k), dtype=torch.int32, device=dev)
    Y = torch.empty(B, K, dtype=torch.bfloat16, device=dev)
    wsf = ssd.workspace(ssd.moe_front_workspace_bytes(B, E, L, K), dev)
    wse = ssd.workspace(ssd.moe_experts_workspace_bytes(B, E, k, K, I), dev)
    for rnd in range(3):
        X = inputs.activations(B, K, dev, 96 + rnd)
        ssd.moe_front(X, Wc, E, L, k, lat, idx, w, wsf, route_map=rm)
        ssd.moe_experts(X, idx, w, rm, Wgu, Wd, None, None, Y, wse)
        torch.cuda.synchronize()
        ref = oracle.moe_front(inputs.bits(X), inputs.bits(Wc), E, L, k)
        assert np.array_equal(idx.cpu().numpy(), ref["idx"])
        y_ref, _ = oracle.moe_experts(inputs.bits(X), ref["idx"], w.cpu().numpy().astype(np.float64),
                                      inputs.bits(Wgu), inputs.bits(Wd))
        assert_close(to_f64(oracle, Y), y_ref, f"round {rnd}")
