"""The oracle reproduces its stored tiny-layer results (bf16 and keep-quant experts) bit for
bit on this host."""
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


def test_tiny_keep_quant_layer_golden():
    from tests.golden.gen_golden import tiny_layer_q_result

    with open(os.path.join(HERE, "tiny_layer_q.json")) as f:
        stored = json.load(f)
    now = tiny_layer_q_result()
    for fmt in ("q8_0", "q4_k"):
        assert now[fmt]["inputs_sha256"] == stored[fmt]["inputs_sha256"], "seeded inputs changed"
        assert now[fmt]["topk_ids"] == stored[fmt]["topk_ids"]
        assert now[fmt]["out_bf16_hex"] == stored[fmt]["out_bf16_hex"]
    # the two formats are different weights: their outputs differ
    assert stored["q8_0"]["out_bf16_hex"] != stored["q4_k"]["out_bf16_hex"]
