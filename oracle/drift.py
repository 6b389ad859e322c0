"""Quality figure of the multi-layer cached step (test infrastructure only).

With more than one layer the method reuses stale deeper-layer K/V by design
("LaCache: Exact Caching and Precision-Adaptive Inference for Diffusion Large
Language Models", limitations: reuse is exact only in the first layer), so the
cached step loop differs from the plain definition, a full forward of every
row at every step.  This module measures that difference on the same inputs:
step by step while the two trajectories hold the same tokens, the largest
change of the top-1 probability, the mean change of the entropy, and the
share of equal argmaxes; then whether the generated tokens agree at the end.
It is a report, not a parity gate: GPU parity is checked against the cached
algorithm.

    python -m oracle.drift mid_multi
"""
import sys

import numpy as np

from .run import run_dense, weights_f64


def drift(w, m, tok0, n_steps=None):
    """Per-step drift records of the cached loop against the recompute loop,
    the share of equal generated tokens at the end, and the first step whose
    tokens (after the step) differ between the two loops (None if none)."""
    W = weights_f64(w, m)
    cached = run_dense(w, W, tok0, n_steps=n_steps, mode="cached")
    plain = run_dense(w, W, tok0, n_steps=n_steps, mode="recompute")
    steps, first = [], None
    for a, r in zip(cached, plain):
        steps.append({
            "t": a["t"], "s": a["s"],
            "max_dp1": float(np.max(np.abs(a["p1"] - r["p1"]))),
            "mean_dent": float(np.mean(np.abs(a["ent"] - r["ent"]))),
            "argmax_agree": float(np.mean(a["argmax"] == r["argmax"])),
        })
        if first is None and not np.array_equal(a["tok"], r["tok"]):
            first = a["t"]
    tok_agree = float(np.mean(cached[-1]["tok"] == plain[-1]["tok"])) if cached else 1.0
    return steps, tok_agree, first


def main(argv):
    from workloads import configs as C
    from workloads import generate as G
    name = argv[1] if len(argv) > 1 else "mid_multi"
    w = C.get(name)
    m = G.model(w)
    tok0 = G.prompt_tokens(w)
    steps, tok_agree, first = drift(w, m, tok0)
    worst = max(steps, key=lambda r: r["max_dp1"])
    print(f"{name}: {len(steps)} steps, {w.n_layers} layers")
    print(f"  largest |p1 cached - p1 recompute|: {worst['max_dp1']:.3e} (step {worst['t']})")
    print(f"  mean |entropy difference| over steps: {np.mean([r['mean_dent'] for r in steps]):.3e}")
    print(f"  argmax agreement over steps: {np.mean([r['argmax_agree'] for r in steps]):.4f}")
    print(f"  generated tokens equal at the end: {tok_agree:.4f}; first step with different tokens: {first}")


if __name__ == "__main__":
    main(sys.argv)
