"""Write tests/golden/dedup_bias.json: the router-logit offset beta that makes
the 32 hot experts carry 60% of the renormalised top-k routing mass on the
small-batch dedup workload (512 steps x 4 tokens, Qwen3-30B-A3B layer shape).

Calls only the CPU oracle (routing) and the seeded input generators.
Run from the repository root:  python tests/golden/make_dedup_bias.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from quantized_moe_expert_gemv_gb300 import synth  # noqa: E402

TARGET = 0.60


def hot_share(beta, rw, xs, seed, k):
    bias = synth.dedup_router_bias(seed, beta)
    ids, w, _, _ = oracle.route_tokens(rw, xs, k, bias=bias)
    hot = np.isin(ids, synth.dedup_hot_set(seed))
    return float((w * hot).sum() / w.sum()), ids, hot


def main():
    wl = synth.WORKLOADS["dedup4"]
    shape, seed = wl["shape"], wl["seed"]
    rw = synth.make_router_w(shape, seed)
    xs = synth.make_tokens(shape, seed, wl["tokens_per_step"] * wl["n_steps"])
    lo, hi = 0.0, 8.0
    for _ in range(40):
        mid = np.float32(0.5 * (lo + hi))
        share, _, _ = hot_share(float(mid), rw, xs, seed, shape.top_k)
        if share < TARGET:
            lo = float(mid)
        else:
            hi = float(mid)
    beta = float(np.float32(hi))
    share, ids, hot = hot_share(beta, rw, xs, seed, shape.top_k)
    steps = ids.reshape(wl["n_steps"], wl["tokens_per_step"] * shape.top_k)
    unique = np.array([len(set(s.tolist())) for s in steps])
    out = {
        "beta": beta,
        "hot_mass_share": share,
        "hot_slot_share": float(hot.mean()),
        "mean_unique_experts_per_step": float(unique.mean()),
        "n_tokens": int(xs.shape[0]),
        "how": "bisection on beta (fp32) until the hot set's share of the renormalised top-k "
               "weight mass reaches 0.60; routing by the CPU oracle",
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "dedup_bias.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=2)
        f.write("\n")
    print(json.dumps(out, indent=2))


if __name__ == "__main__":
    main()
