"""Find the router-bias scale of the skewed 16-expert workload -- TEST INFRASTRUCTURE.

The skewed-routing workload (T = 32 x 2048 tokens, d = 4096, E = 16, top-2)
adds a router bias b_e = alpha * ln(z_e), z the Zipf(s = 1.1) distribution
over expert ranks, so that the 4 hottest experts receive about 60 % of the
top-2 selections.  alpha is found by bisection (40 steps) on the seeded
inputs, with the oracle's fp64 logits and its top-k rule, and written to
tests/golden/skewed16_zipf_bias.json, which the input generator reads.

    python oracle/calibrate_zipf_bias.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import moe_inputs  # noqa: E402
import oracle      # noqa: E402

TARGET, TOL = 0.60, 0.01


def main(seed: int = 0):
    w = moe_inputs.get("skewed16_bf16")
    inp = moe_inputs.make_inputs(w, seed, parts=("x", "W_r"))
    cfg = oracle.OracleConfig(T=w.T, d=w.d, f=1, E=w.E, k=w.k)
    base = oracle.router_logits(cfg, moe_inputs.as_f64(inp["x"], "bf16"),
                                moe_inputs.as_f64(inp["W_r"], "bf16"))

    def top4_share(alpha):
        b = moe_inputs.zipf_bias(w.E, alpha).astype(np.float64)
        counts = oracle.route(cfg, base + b[None, :])["counts"]
        return float(np.sort(counts)[::-1][:4].sum()) / (w.T * w.k)

    lo, hi = 0.0, 8.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if top4_share(mid) < TARGET:
            lo = mid
        else:
            hi = mid
    alpha = 0.5 * (lo + hi)
    share = top4_share(alpha)
    assert abs(share - TARGET) <= TOL, share
    out = {"alpha": alpha, "top4_share": share, "target": TARGET, "seed": seed,
           "zipf_s": 1.1, "bisection_steps": 40,
           "written_by": "oracle/calibrate_zipf_bias.py (oracle fp64 logits and top-k)",
           "recipe": "b_e = alpha * ln(z_e), z_e = e^-1.1 / sum_r r^-1.1 for expert rank e = 1..16 "
                     "(expert 0 hottest); x ~ N(0,1), W_r ~ N(0,0.02), both rounded to bf16"}
    with open(moe_inputs.ZIPF_BIAS_FILE, "w") as fh:
        json.dump(out, fh, indent=1)
        fh.write("\n")
    print(json.dumps(out))


if __name__ == "__main__":
    main()
