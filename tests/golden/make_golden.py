"""Write the golden fixtures of this directory (test infrastructure).

The pages ("Hyper Optimizing Kimi K3 in vLLM: Moving Fast and Responsibly") print no
worked example and no kernel-level value, so every stored expected value here is
written by this script, which calls nothing but ``oracle/`` on small seeded inputs.
The fixtures freeze the oracle's results: a later change to its arithmetic shows up
in ``tests/test_golden.py`` (which also pins each fixture to exact rational
arithmetic independent of the oracle), and the GPU path is compared with them there.

Inputs are drawn with numpy's PCG64 from fixed seeds and rounded to bf16 by the
oracle's round-to-nearest-even; arrays of bf16 are stored as one string of 4-digit
hex patterns, floats as JSON numbers (exact round trip).

    python tests/golden/make_golden.py      # rewrites the *.json files here
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402

PAGE = "Hyper Optimizing Kimi K3 in vLLM: Moving Fast and Responsibly"


def hexs(a) -> str:
    return "".join(f"{int(v):04x}" for v in np.asarray(a, dtype=np.uint16).ravel())


def bf16(rng, shape, std):
    return oracle.f64_to_bf16(rng.standard_normal(shape) * std)


def linear_case(name, seed, B, N, K, residual, cite):
    rng = np.random.default_rng(seed)
    X = bf16(rng, (B, K), 1.0)
    W = bf16(rng, (N, K), 0.05)
    R = bf16(rng, (B, N), 1.0) if residual else None
    y, Y = oracle.linear(X, W, R)
    return dict(case=name, cite=cite, B=B, N=N, K=K,
                inputs=dict(X=hexs(X), W=hexs(W), R=None if R is None else hexs(R)),
                expected=dict(Y=hexs(Y), y=y.ravel().tolist()))


def front_case(name, seed, B, E, L, K, topk, dup, cite):
    rng = np.random.default_rng(seed)
    X = bf16(rng, (B, K), 1.0)
    Wc = bf16(rng, (E + L, K), 0.2)
    for a, b in dup:  # identical router rows: bit-identical logits, ties to the lower index
        Wc[b] = Wc[a]
    f = oracle.moe_front(X, Wc, E, L, topk)
    m = oracle.route_map(f["idx"], E)
    return dict(case=name, cite=cite, B=B, E=E, L=L, K=K, topk=topk, duplicate_rows=dup,
                inputs=dict(X=hexs(X), Wcat=hexs(Wc)),
                expected=dict(logits=f["logits"].ravel().tolist(), latent=hexs(f["latent"]),
                              idx=f["idx"].ravel().tolist(), w=f["w"].ravel().tolist(),
                              probs=f["probs"].ravel().tolist(),
                              counts=m["counts"].tolist(), offsets=m["offsets"].tolist(),
                              pairs=m["pairs"].tolist(), pos=m["pos"].tolist(),
                              used=m["used"].tolist(), num_used=m["num_used"]))


def linear_integer_case(name, seed, B, N, K, cite):
    """Integers in [-4, 4]: every partial sum is exact in fp32, so any summation order
    gives the same bf16 result and the GPU must match bit for bit."""
    rng = np.random.default_rng(seed)
    X = oracle.f64_to_bf16(rng.integers(-4, 5, (B, K)).astype(np.float64))
    W = oracle.f64_to_bf16(rng.integers(-4, 5, (N, K)).astype(np.float64))
    y, Y = oracle.linear(X, W)
    return dict(case=name, cite=cite, B=B, N=N, K=K, exact=True,
                inputs=dict(X=hexs(X), W=hexs(W), R=None),
                expected=dict(Y=hexs(Y), y=y.ravel().tolist()))


CASES = [
    linear_case("linear_tiny_residual", 101, 2, 9, 24, True,
                f'"{PAGE}", Part 1 / 1 "Tune shapes for the workload" (small-matrix kernel, '
                f'batch 1-2) and Part 1 / 2 "Overlap computation and communication" '
                f'(residual added before the single rounding)'),
    linear_case("linear_splitk_ragged", 102, 5, 130, 72, False,
                f'"{PAGE}", Part 1 / 1 "Tune shapes for the workload" (split-K kernels '
                f'for larger batches); two row tiles, a full and a ragged k-block'),
    front_case("front_ties", 103, 3, 20, 6, 72, 4, [[2, 11], [5, 6]],
               f'"{PAGE}", Part 1 / 3 "Improve MoE scheduling and overlap" (router and '
               f'latent projection in one product); routing read as softmax, top-k on '
               f'the logits with ties to the lower index, renormalised weights'),
    linear_integer_case("linear_integer_exact", 104, 3, 17, 48,
                        f'"{PAGE}", Part 1 / 1 "Tune shapes for the workload" (the '
                        f'projection itself; exact sums make the result order-free)'),
]


def main():
    oracle.build()
    for c in CASES:
        path = os.path.join(HERE, c["case"] + ".json")
        with open(path, "w") as f:
            json.dump(c, f, separators=(",", ":"))
            f.write("\n")
        print(path, os.path.getsize(path), "bytes")


if __name__ == "__main__":
    main()
