"""The benchmark's command-line contract on a host without a GPU: the reference
arm (the oracle on the host cores) prints one complete JSON line, on one rank
or on rank 0 of two; the product arm and the layer refuse to run without CUDA
instead of falling back to the CPU."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest
import torch

from mixture_experts_ffn_renorm_gb300 import workloads as W
from mixture_experts_ffn_renorm_gb300.layer import MoeBlock

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
needs_no_gpu = pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU behaviour")


def _bench(*args, timeout=300, torchrun=0):
    cmd = [sys.executable]
    if torchrun:
        s = socket.socket()
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
        s.close()
        cmd += ["-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={torchrun}",
                "--master-addr", "127.0.0.1", "--master-port", str(port)]
    cmd += [os.path.join(ROOT, "bench.py"), *args]
    return subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=timeout)


def _json_lines(out):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def _check_reference_line(d, weights, n_gpus):
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["n_gpus"] == n_gpus
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert (d["steps"], d["warmup"]) == (3, 3)
    assert d["value"] > 0 and d["ms_per_step"] > 0
    cfg = d["config"]
    assert cfg["workload"].startswith("tiny_T4_H64_I32_E8_K2") and cfg["weights"] == weights
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert "tokens per step" in cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


@pytest.mark.parametrize("weights", ["bf16", "q8_0"])
def test_reference_arm_prints_one_complete_line(weights):
    r = _bench("--impl", "reference", "--config", "tiny", "--weights", weights,
               "--steps", "3", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_reference_line(lines[0], weights, 1)


def test_reference_arm_under_torchrun_prints_on_rank_0_only():
    r = _bench("--impl", "reference", "--gpus", "2", "--config", "tiny", "--steps", "3",
               "--warmup", "3", torchrun=2)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_reference_line(lines[0], "bf16", 2)


@needs_no_gpu
def test_product_arm_fails_loudly_without_a_gpu():
    r = _bench("--config", "tiny", "--steps", "3", "--warmup", "3")
    assert r.returncode != 0
    assert _json_lines(r.stdout) == []


def test_layer_refuses_a_cpu_device():
    cfg = W.TINY
    with pytest.raises(ValueError, match="CUDA device"):
        MoeBlock(cfg.H, cfg.I, cfg.E, cfg.K, {"w_router": None}, max_tokens=cfg.T, device="cpu")


def test_layer_refuses_an_unknown_gather_mode():
    cfg = W.TINY
    with pytest.raises(ValueError, match="gather must be"):
        MoeBlock(cfg.H, cfg.I, cfg.E, cfg.K, {"w_router": None}, max_tokens=cfg.T, device="cuda",
                 gather="sometimes")
    # "auto" with staged rows is refused like gather=True
    with pytest.raises(ValueError, match="staged rows"):
        MoeBlock(cfg.H, cfg.I, cfg.E, cfg.K, {"w_router": None}, max_tokens=cfg.T, device="cuda",
                 gather="auto", staged=True)
