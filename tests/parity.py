"""Comparison rules between the CUDA path and the CPU oracle.

Floating-point outputs: relative L2 error <= 2e-3 and max |err| <= 1e-2 *
max |ref| per token (the target the method is held to).  Dequantized
weights, top-k ids, counts, offsets and permutations: bit-exact.

The top-k choice is an integer decided by floating point.  Both sides take
it on fp32 logits; the GPU's fp32 logits differ from the oracle's
correctly rounded ones by summation order (measured |diff| <= ~2.4e-6 on
these inputs).  So ids must be bit-exact on every token whose fp64 margin
z_(k) - z_(k+1) is at least TAU = 1e-5 and whose selected logits are
pairwise more than TAU apart; a token under TAU at the boundary must still
pick a valid selection (no unselected expert more than TAU above a selected
one), and its output is not compared (the experts may legitimately differ).
Two selected logits closer than TAU may come out in either order (the set,
and so the output, is the same): the order is then checked to be
descending up to TAU.
"""
from __future__ import annotations

import numpy as np

REL_L2 = 2e-3
MAX_REL = 1e-2
TAU = 1e-5


def rel_l2(got: np.ndarray, ref: np.ndarray) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    r = rel_l2(got, ref)
    m = float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-300))
    assert r <= REL_L2 and m <= MAX_REL, f"{what}: rel_l2={r:.3e} max_rel={m:.3e}"
    return r, m


def routing_ok(gpu_ids, oracle_ids, z64, margin, k):
    """True when the selection must equal the oracle's and does (the order
    may differ only between selected logits closer than TAU); False for a
    boundary near-tie, after checking that the GPU's choice is a valid one."""
    gpu_ids = np.asarray(gpu_ids)
    oracle_ids = np.asarray(oracle_ids)
    zs = np.asarray(z64)[gpu_ids]
    assert len(set(gpu_ids.tolist())) == k
    assert np.all(zs[:-1] >= zs[1:] - TAU), ("selection not in descending order", gpu_ids, zs)
    if margin >= TAU:
        assert set(gpu_ids.tolist()) == set(oracle_ids.tolist()), (gpu_ids, oracle_ids, margin)
        if not np.array_equal(gpu_ids, oracle_ids):  # only near-equal selected logits may swap
            for a, b in zip(gpu_ids, oracle_ids):
                if a != b:
                    assert abs(z64[a] - z64[b]) < TAU, (gpu_ids, oracle_ids)
        return True
    sel = set(gpu_ids.tolist())
    unsel = [e for e in range(len(z64)) if e not in sel]
    if unsel:
        assert min(z64[list(sel)]) >= max(z64[unsel]) - TAU
    return bool(set(gpu_ids.tolist()) == set(oracle_ids.tolist()))


def same_by_id(gpu_ids, gpu_w, oracle_ids, oracle_w, atol):
    """Weights compared per expert id (the order of near-equal logits may differ)."""
    g = dict(zip(np.asarray(gpu_ids).tolist(), np.asarray(gpu_w).tolist()))
    o = dict(zip(np.asarray(oracle_ids).tolist(), np.asarray(oracle_w).tolist()))
    assert g.keys() == o.keys()
    for e in g:
        assert abs(g[e] - o[e]) <= atol, (e, g[e], o[e])
