"""Host-side logic around the keep-quant experts (CPU, no device calls): the
layer's argument checks, the benchmark's choice between the keep-quant kernels
and the bf16 expansion, and the layout of the seeded GGUF weight blocks."""
from __future__ import annotations

import argparse
import importlib.util
import os

import numpy as np
import pytest

from mixture_experts_ffn_renorm_gb300 import workloads as W
from mixture_experts_ffn_renorm_gb300.layer import MoeBlock

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_layer_refuses_bad_keep_quant_arguments_before_any_device_work():
    cfg = W.TINY
    d = {"w_router": None}
    with pytest.raises(ValueError, match="qweights"):
        MoeBlock(cfg.H, cfg.I, cfg.E, cfg.K, d, max_tokens=cfg.T, device="cpu", qweights="q5_k")
    with pytest.raises(ValueError, match="exclude"):
        MoeBlock(cfg.H, cfg.I, cfg.E, cfg.K, d, max_tokens=cfg.T, device="cpu", qweights="q4_k",
                 fp8_weights=True)
    with pytest.raises(ValueError, match="q_dequant"):
        MoeBlock(cfg.H, cfg.I, cfg.E, cfg.K, d, max_tokens=cfg.T, device="cpu", q_dequant=True)


def test_bench_expands_keep_quant_blocks_only_for_many_rows_per_expert():
    b = _bench()
    ns = lambda mode: argparse.Namespace(q_dequant=mode)  # noqa: E731
    # decode: 128 routed rows over 128 experts; prefill and large: 512 and 64 per expert
    assert not b.q_dequant_on(ns("auto"), W.DECODE)
    assert b.q_dequant_on(ns("auto"), W.PREFILL)
    assert b.q_dequant_on(ns("auto"), W.LARGE)
    assert b.q_dequant_on(ns("on"), W.DECODE)
    assert not b.q_dequant_on(ns("off"), W.PREFILL)
    # the format table of the benchmark matches the generator's
    for name, (fid, blk, nbytes) in b.Q_WEIGHTS.items():
        assert W.Q_FORMATS[name][:3] == (fid, blk, nbytes)


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
def test_seeded_blocks_layout_and_scales(fmt):
    fid, blk, nbytes, n16 = W.Q_FORMATS[fmt]
    G, R, K = 2, 3, 512
    w = W.q_weights(5, 99, G, R, K, fmt, 0.02)
    assert w.dtype == np.uint8 and w.shape == (G, R, (K // blk) * nbytes)
    blocks = w.reshape(-1, nbytes)
    scales = blocks[:, :2 * n16].copy().view(np.float16).astype(np.float64)
    assert np.all(scales > 0) and np.all(np.isfinite(scales))
    if fmt == "q8_0":
        assert np.all(np.abs(scales / (0.02 / 74.0) - 1.0) <= 0.21)
    else:
        d, dmin = scales[:, 0], scales[:, 1]
        assert np.all(np.abs(d / (0.02 / 240.0) - 1.0) <= 0.21)
        assert np.all(np.abs(dmin / (7.5 * d) - 1.0) <= 0.21)
    # the same seed and tag give the same bytes; another tag other bytes
    assert np.array_equal(w, W.q_weights(5, 99, G, R, K, fmt, 0.02))
    assert not np.array_equal(w, W.q_weights(5, 98, G, R, K, fmt, 0.02))
    with pytest.raises(ValueError):
        W.q_weights(5, 99, G, R, K + 16, fmt, 0.02)
