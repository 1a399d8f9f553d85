"""The oracle reproduces its stored tiny-layer result bit for bit on this host."""
import json
import os

import numpy as np

from tests.golden.gen_golden import tiny_layer_result

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_tiny_layer_golden():
    with open(os.path.join(HERE, "tiny_layer.json")) as f:
        stored = json.load(f)
    now = tiny_layer_result()
    assert now["inputs_sha256"] == stored["inputs_sha256"], "seeded inputs changed"
    assert now["topk_ids"] == stored["topk_ids"]
    assert now["topk_w_f32_hex"] == stored["topk_w_f32_hex"]
    assert now["out_bf16_hex"] == stored["out_bf16_hex"]
    # the routing weights of each token sum to one (renormalised softmax)
    w = np.array([[float.fromhex(v) for v in r] for r in stored["topk_w_f32_hex"]])
    assert np.allclose(w.sum(1), 1.0, atol=4e-7)
