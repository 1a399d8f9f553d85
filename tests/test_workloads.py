"""The seeded benchmark workloads route as the measured numbers say (CPU): the
expert histograms that the decode, prefill and large layers produce through the
oracle's router.  A change to the input recipe (seeds, scales, the Zipf bias)
shows up here before it silently changes what the benchmark measures."""
from __future__ import annotations

import numpy as np
import pytest

import oracle as O
from mixture_experts_ffn_renorm_gb300 import workloads as W

# name -> (max, min, experts touched) of the rows per expert
EXPECTED = {
    "decode": (5, 0, 85),       # T=16, K=8 over 128 experts, uniform router
    "prefill": (7459, 7, 128),  # T=8192, K=8 over 128 experts, Zipf(1.1) logit bias
    "large": (99, 43, 256),     # T=2048, K=8 over 256 experts
}


@pytest.mark.parametrize("name", sorted(EXPECTED))
def test_workload_expert_histogram(name):
    cfg = {"decode": W.DECODE, "prefill": W.PREFILL, "large": W.LARGE}[name]
    d = W.layer_inputs(cfg, with_weights=False)
    ids, w, _, _ = O.route_topk(d["x"], d["w_router"], d.get("logit_bias"), T=cfg.T, H=cfg.H,
                                E=cfg.E, K=cfg.K)
    counts = np.bincount(ids.ravel(), minlength=cfg.E)
    assert counts.sum() == cfg.T * cfg.K
    assert (int(counts.max()), int(counts.min()), int((counts > 0).sum())) == EXPECTED[name]
    # every token's K experts are distinct, and the renormalised weights sum to one
    assert all(len(set(r)) == cfg.K for r in ids.tolist())
    assert np.allclose(w.astype(np.float64).sum(1), 1.0, atol=cfg.K * 2.0**-23)
