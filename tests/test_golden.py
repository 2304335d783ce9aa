"""Golden fixtures (tests/golden/*.json, written by tests/golden/make_golden.py from the
oracle alone): the oracle must reproduce them (a change to its arithmetic shows up
here), each is pinned to exact rational arithmetic that shares nothing with the
oracle, and the CUDA path (through the C ABI) must match them on the GPU."""
import glob
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import exact_ref

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = sorted(glob.glob(os.path.join(HERE, "golden", "*.json")))


def _load(name):
    with open(os.path.join(HERE, "golden", name + ".json")) as f:
        return json.load(f)


def _u16(s, shape):
    a = np.array([int(s[i:i + 4], 16) for i in range(0, len(s), 4)], dtype=np.uint16)
    return a.reshape(shape)


def _linear_inputs(c):
    B, N, K = c["B"], c["N"], c["K"]
    X = _u16(c["inputs"]["X"], (B, K))
    W = _u16(c["inputs"]["W"], (N, K))
    R = None if c["inputs"]["R"] is None else _u16(c["inputs"]["R"], (B, N))
    return X, W, R


LINEAR = ["linear_tiny_residual", "linear_splitk_ragged", "linear_integer_exact"]


def test_every_fixture_names_its_source():
    assert len(GOLDEN) >= 4
    for p in GOLDEN:
        with open(p) as f:
            c = json.load(f)
        assert "Hyper Optimizing Kimi K3 in vLLM" in c["cite"], p
        assert "Part 1 /" in c["cite"], p


@pytest.mark.parametrize("name", LINEAR)
def test_oracle_reproduces_linear_fixture(oracle_mod, name):
    c = _load(name)
    X, W, R = _linear_inputs(c)
    y, Y = oracle_mod.linear(X, W, R)
    assert np.array_equal(Y, _u16(c["expected"]["Y"], Y.shape))
    assert np.array_equal(y.ravel(), np.array(c["expected"]["y"]))


@pytest.mark.parametrize("name", LINEAR)
def test_linear_fixture_equals_exact_rationals(name):
    """Every stored output equals the exactly computed sum rounded once to bf16, and the
    stored fp64 value is within the fp64 summation bound of the exact sum."""
    c = _load(name)
    X, W, R = _linear_inputs(c)
    B, N, K = c["B"], c["N"], c["K"]
    ex = exact_ref.linear_exact(X.tolist(), W.tolist(), None if R is None else R.tolist())
    Y = _u16(c["expected"]["Y"], (B, N))
    y = np.array(c["expected"]["y"]).reshape(B, N)
    for b in range(B):
        for n in range(N):
            assert Y[b, n] == exact_ref.fraction_to_bf16_bits(ex[b][n]), (b, n)
            mag = sum(abs(exact_ref.bf16_bits_to_fraction(X[b, k]) *
                          exact_ref.bf16_bits_to_fraction(W[n, k])) for k in range(K))
            if R is not None:
                mag += abs(exact_ref.bf16_bits_to_fraction(R[b, n]))
            assert abs(Fraction(y[b, n]) - ex[b][n]) <= (K + 1) * Fraction(1, 2 ** 52) * mag
    if c.get("exact"):
        assert all(Fraction(y[b, n]) == ex[b][n] for b in range(B) for n in range(N))


def _front_inputs(c):
    B, E, L, K = c["B"], c["E"], c["L"], c["K"]
    return _u16(c["inputs"]["X"], (B, K)), _u16(c["inputs"]["Wcat"], (E + L, K))


def test_oracle_reproduces_front_fixture(oracle_mod):
    c = _load("front_ties")
    X, Wc = _front_inputs(c)
    E, L, k = c["E"], c["L"], c["topk"]
    f = oracle_mod.moe_front(X, Wc, E, L, k)
    ex = c["expected"]
    assert np.array_equal(f["idx"].ravel(), np.array(ex["idx"]))
    assert np.array_equal(f["w"].ravel(), np.array(ex["w"]))
    assert np.array_equal(f["probs"].ravel(), np.array(ex["probs"]))
    assert np.array_equal(f["logits"].ravel(), np.array(ex["logits"]))
    assert np.array_equal(f["latent"], _u16(ex["latent"], f["latent"].shape))
    m = oracle_mod.route_map(f["idx"], E)
    for key in ("counts", "offsets", "pairs", "pos", "used"):
        assert m[key].tolist() == ex[key], key
    assert m["num_used"] == ex["num_used"]


def test_front_fixture_equals_exact_routing():
    """Top-k from exactly computed logits (compared in fp32, ties to the lower index),
    the planted duplicate router rows tie exactly, the latent is the exact sum rounded
    once, the weights are exp-ratios of the chosen logits, and the route map is the
    (expert, entry) sort of the routing."""
    import math
    c = _load("front_ties")
    X, Wc = _front_inputs(c)
    B, E, L, k = c["B"], c["E"], c["L"], c["topk"]
    ex = c["expected"]
    Z = exact_ref.linear_exact(X.tolist(), Wc.tolist())
    idx = np.array(ex["idx"]).reshape(B, k)
    w = np.array(ex["w"]).reshape(B, k)
    lat = _u16(ex["latent"], (B, L))
    for a, b2 in c["duplicate_rows"]:
        assert all(Z[b][a] == Z[b][b2] for b in range(B))
    for b in range(B):
        l32 = np.array([float(Z[b][e]) for e in range(E)], dtype=np.float32)
        order = np.lexsort((np.arange(E), -l32.astype(np.float64)))[:k]
        assert idx[b].tolist() == order.tolist(), b
        m = max(float(Z[b][e]) for e in range(E))
        ez = [math.exp(float(Z[b][e]) - m) for e in order]
        np.testing.assert_allclose(w[b], np.array(ez) / sum(ez), rtol=1e-12)
        for j in range(L):
            assert lat[b, j] == exact_ref.fraction_to_bf16_bits(Z[b][E + j])
    entries = sorted(((int(idx.ravel()[q]), q // k, q) for q in range(B * k)))
    assert ex["pairs"] == [q for _, _, q in entries]
    counts = np.bincount(idx.ravel(), minlength=E)
    assert ex["counts"] == counts.tolist()
    assert ex["offsets"] == [0] + np.cumsum(counts).tolist()
    assert ex["used"] == [e for e in range(E) if counts[e] > 0]
    pos = [0] * (B * k)
    for at, q in enumerate(ex["pairs"]):
        pos[q] = at
    assert ex["pos"] == pos


# ------------------------------------------------------------------- GPU ----

@pytest.fixture(scope="module")
def gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import split_switched_decode_gb300 as ssd
    ssd.build()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    ssd.dec_set_force_variant(ssd.VARIANT_NONE)
    return torch, ssd, dev


def _dev_bf16(torch, a, dev):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def _host_bits(t):
    import torch
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.gpu
@pytest.mark.parametrize("name", LINEAR)
@pytest.mark.parametrize("path", ["tiny", "splitk_cc", "splitk_tc", "switch"])
def test_gpu_matches_linear_fixture(gpu, name, path):
    from gpu_common import assert_close
    torch, ssd, dev = gpu
    c = _load(name)
    X, W, R = _linear_inputs(c)
    B, N, K = c["B"], c["N"], c["K"]
    if path == "tiny" and B > 4:
        pytest.skip("the tiny kernel takes at most 4 rows")
    Xd, Wd = _dev_bf16(torch, X, dev), _dev_bf16(torch, W, dev)
    Rd = None if R is None else _dev_bf16(torch, R, dev)
    Y = torch.empty(B, N, dtype=torch.bfloat16, device=dev)
    ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N, K), dev)
    if path == "tiny":
        ssd.dec_gemv(Xd, Wd, Rd, Y)
    elif path == "switch":
        ssd.dec_linear(Xd, Wd, Rd, Y, ws)
    else:
        ssd.dec_splitk_gemm(Xd, Wd, Rd, Y, ws, use_tc=1 if path == "splitk_tc" else 0)
    torch.cuda.synchronize()
    assert ssd.dec_sync_status() == ssd.DEC_OK
    Yg = _host_bits(Y)
    if c.get("exact"):
        assert np.array_equal(Yg, _u16(c["expected"]["Y"], (B, N)))
    else:
        import oracle
        assert_close(oracle.bf16_to_f64(Yg), np.array(c["expected"]["y"]).reshape(B, N),
                     f"{name} {path}")


@pytest.mark.gpu
def test_gpu_matches_front_fixture(gpu):
    from gpu_common import assert_close
    import oracle
    torch, ssd, dev = gpu
    c = _load("front_ties")
    X, Wc = _front_inputs(c)
    B, E, L, K, k = c["B"], c["E"], c["L"], c["K"], c["topk"]
    ex = c["expected"]
    lat = torch.empty(B, L, dtype=torch.bfloat16, device=dev)
    idx = torch.empty(B, k, dtype=torch.int32, device=dev)
    w = torch.empty(B, k, dtype=torch.float32, device=dev)
    pr = torch.empty(B, E, dtype=torch.float32, device=dev)
    rm = torch.full((ssd.moe_route_map_ints(B, E, k),), -7, dtype=torch.int32, device=dev)
    ws = ssd.workspace(ssd.moe_front_workspace_bytes(B, E, L, K), dev)
    ssd.moe_front(_dev_bf16(torch, X, dev), _dev_bf16(torch, Wc, dev), E, L, k, lat, idx, w, ws,
                  probs=pr, route_map=rm)
    torch.cuda.synchronize()
    assert ssd.dec_sync_status() == ssd.DEC_OK
    assert idx.cpu().numpy().ravel().tolist() == ex["idx"]
    assert_close(w.cpu().numpy().astype(np.float64), np.array(ex["w"]).reshape(B, k), "weights")
    assert_close(pr.cpu().numpy().astype(np.float64), np.array(ex["probs"]).reshape(B, E), "probs")
    assert_close(oracle.bf16_to_f64(_host_bits(lat)),
                 oracle.bf16_to_f64(_u16(ex["latent"], (B, L))), "latent")
    r, P = rm.cpu().numpy(), B * k
    assert r[:E].tolist() == ex["counts"]
    assert r[E:2 * E + 1].tolist() == ex["offsets"]
    assert r[2 * E + 1:2 * E + 1 + P].tolist() == ex["pairs"]
    assert r[2 * E + 1 + P:2 * E + 1 + 2 * P].tolist() == ex["pos"]
    assert r[2 * E + 1 + 2 * P] == ex["num_used"]
