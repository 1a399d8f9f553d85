"""Write tests/golden/tiny_layer.json and tiny_layer_q.json from the CPU oracle alone.

The pages print no worked example for the MoE block, so the stored values
here are the oracle's own result on the tiny seeded layer (T=4, H=64, I=32,
E=8, top-2, shared expert I=32 with its sigmoid gate).  They pin the oracle
across hosts and compilers: an x86 and an Arm build must reproduce them bit
for bit.  tiny_layer_q.json holds the same kind of record for a small layer
with keep-quant expert weights (random valid GGUF Q8_0 and Q4_K blocks, T=4,
H=I=256, E=4, top-2, shared expert I=32).  Run:  python tests/golden/gen_golden.py
"""
import hashlib
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle as O  # noqa: E402
from mixture_experts_ffn_renorm_gb300 import workloads as W  # noqa: E402


def tiny_layer_result():
    cfg = W.TINY
    d = W.layer_inputs(cfg)
    out, ids, w = O.moe_layer_tokens(
        d["x"], d["w_router"], d["logit_bias"], d["w13"], d["w2"], d["w_shared_gate"],
        d["w13_shared"], d["w2_shared"], H=cfg.H, I=cfg.I, E=cfg.E, K=cfg.K,
        I_shared=cfg.I_shared, tokens=np.arange(cfg.T, dtype=np.int32))
    inputs_sha = hashlib.sha256(b"".join(
        np.ascontiguousarray(d[k]).tobytes() for k in
        ("x", "w_router", "w13", "w2", "w_shared_gate", "w13_shared", "w2_shared"))).hexdigest()
    return {
        "what": "oracle output of the tiny MoE layer (see gen_golden.py)",
        "config": cfg.name,
        "inputs_sha256": inputs_sha,
        "topk_ids": ids.tolist(),
        "topk_w_f32_hex": [[float(v).hex() for v in row] for row in w],
        "out_bf16_hex": [[f"{int(v):04x}" for v in row] for row in out],
    }


Q_TINY = W.LayerConfig("tiny_q_T4_H256_I256_E4_K2_shared32", T=4, H=256, I=256, E=4, K=2,
                       I_shared=32, seed=7)


def tiny_layer_q_result():
    cfg = Q_TINY
    res = {"what": "oracle output of the tiny keep-quant MoE layer (see gen_golden.py)",
           "config": cfg.name}
    d = W.layer_inputs(cfg, with_weights=False)
    for name, fmt in (("q8_0", O.Q8_0), ("q4_k", O.Q4_K)):
        q = W.layer_q_weights(cfg, name)
        out, ids, w = O.moe_layer_tokens_q(
            d["x"], d["w_router"], d["logit_bias"], q["w13q"], q["w2q"], fmt, d["w_shared_gate"],
            d["w13_shared"], d["w2_shared"], H=cfg.H, I=cfg.I, E=cfg.E, K=cfg.K,
            I_shared=cfg.I_shared, tokens=np.arange(cfg.T, dtype=np.int32))
        sha = hashlib.sha256(b"".join(
            np.ascontiguousarray(a).tobytes() for a in
            (d["x"], d["w_router"], q["w13q"], q["w2q"], d["w_shared_gate"], d["w13_shared"],
             d["w2_shared"]))).hexdigest()
        res[name] = {
            "inputs_sha256": sha,
            "topk_ids": ids.tolist(),
            "out_bf16_hex": [[f"{int(v):04x}" for v in row] for row in out],
        }
    return res


if __name__ == "__main__":
    for fname, fn in (("tiny_layer.json", tiny_layer_result),
                      ("tiny_layer_q.json", tiny_layer_q_result)):
        with open(os.path.join(HERE, fname), "w") as f:
            json.dump(fn(), f, indent=1)
        print("wrote", os.path.join(HERE, fname))
