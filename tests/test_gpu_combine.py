"""GPU parity of moe_combine, moe_combine_gate and shared_expert_gate against
the CPU oracle: bit-exact in every dtype arm (vllm.cpp PR #509 review rework:
sequential K order, single store rounding, no contraction)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mixture_experts_ffn_renorm_gb300 as m
import oracle as O
from mixture_experts_ffn_renorm_gb300 import workloads as W

from .gpu_util import empty, launched_since, launches, to_dev, to_host

pytestmark = pytest.mark.gpu

F32, BF16 = m.F32, m.BF16


def _arr(rng, shape, dt, scale=1.0):
    a = (scale * rng.standard_normal(shape)).astype(np.float32)
    return W.to_bf16_bits(a) if dt == BF16 else a


def _out(T, H, dt):
    return empty((T, H), torch.float32 if dt == F32 else torch.bfloat16)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    m.lib()
    m.moe_device_status(clear=True)
    yield
    assert m.moe_device_status() == 0


ARMS = [(BF16, BF16, BF16), (F32, F32, F32), (BF16, F32, F32), (F32, BF16, BF16),
        (BF16, BF16, F32), (F32, F32, BF16)]


@pytest.mark.parametrize("eo_dt,sh_dt,out_dt", ARMS)
@pytest.mark.parametrize("T,K,H", [(1, 1, 8), (7, 3, 40), (33, 8, 264), (5, 20, 16), (3, 32, 8),
                                   (2, 64, 8)])
@pytest.mark.parametrize("rs", [1.0, 0.7])
def test_combine_bit_exact(eo_dt, sh_dt, out_dt, T, K, H, rs):
    rng = np.random.default_rng(T * 100 + K * 10 + H)
    eo = _arr(rng, (T, K, H), eo_dt)
    sh = _arr(rng, (T, H), sh_dt)
    w = rng.uniform(0, 1, (T, K)).astype(np.float32)
    for ww in (w, None):
        for shared in (sh, None):
            want = O.combine(eo, ww, shared, routed_scale=rs, T=T, K=K, H=H, out_dtype=out_dt)
            out = _out(T, H, out_dt)
            before = launches()
            m.moe_combine(to_dev(eo), eo_dt, None if ww is None else to_dev(ww),
                          None if shared is None else to_dev(shared), sh_dt, rs, T, K, H, out,
                          out_dt)
            assert launched_since(before, "combine") == 1
            assert np.array_equal(to_host(out), want)


@pytest.mark.parametrize("eo_dt,sd_dt,out_dt", ARMS)
@pytest.mark.parametrize("T,K,H", [(1, 1, 8), (9, 4, 72), (300, 8, 24)])
@pytest.mark.parametrize("rs", [1.0, 0.7])
def test_combine_gate_bit_exact(eo_dt, sd_dt, out_dt, T, K, H, rs):
    rng = np.random.default_rng(T + K + H)
    eo = _arr(rng, (T, K, H), eo_dt)
    sd = _arr(rng, (T, H), sd_dt)
    gl = rng.normal(0, 2, T).astype(np.float32)
    gl[0] = 0.0
    w = rng.uniform(0, 1, (T, K)).astype(np.float32)
    ws = empty((m.moe_gate_workspace_size(T),), torch.uint8)
    for ww in (w, None):
        want = O.combine_gate(eo, ww, sd, gl, routed_scale=rs, T=T, K=K, H=H, out_dtype=out_dt)
        for wsp in (None, ws):   # sigmoids inside the stream, or precomputed into the workspace
            out = _out(T, H, out_dt)
            before = launches()
            m.moe_combine_gate(to_dev(eo), eo_dt, None if ww is None else to_dev(ww), to_dev(sd),
                               sd_dt, to_dev(gl), rs, T, K, H, out, out_dt, wsp,
                               0 if wsp is None else wsp.numel())
            assert launched_since(before, "combine_gate") == 1
            assert np.array_equal(to_host(out), want)


@pytest.mark.parametrize("sd_dt", [F32, BF16])
@pytest.mark.parametrize("out_dt", [F32, BF16])
def test_shared_expert_gate_four_arms(sd_dt, out_dt):
    rng = np.random.default_rng(3)
    T, H = 257, 136
    sd = _arr(rng, (T, H), sd_dt)
    gl = rng.normal(0, 4, T).astype(np.float32)
    gl[:6] = [0.0, -0.0, 100.0, -100.0, 17.0, -89.0]
    want = O.shared_expert_gate(sd, gl, T=T, H=H, out_dtype=out_dt)
    ws = empty((m.moe_gate_workspace_size(T),), torch.uint8)
    for wsp in (None, ws):
        out = _out(T, H, out_dt)
        before = launches()
        m.shared_expert_gate(to_dev(sd), sd_dt, to_dev(gl), T, H, out, out_dt, wsp,
                             0 if wsp is None else wsp.numel())
        assert launched_since(before, "shared_gate") == 1
        assert np.array_equal(to_host(out), want)


def test_sigmoid_bit_exact_on_a_wide_sweep():
    # shared_expert_gate with sd = 1 (f32 out) returns sigma(gl) itself: the GPU's
    # binary32 exp and sigmoid against the oracle's on 2^22 random bit patterns
    # plus the edges of the range
    rng = np.random.default_rng(17)
    bits = rng.integers(0, 2**32, 1 << 22, dtype=np.uint64).astype(np.uint32)
    g = bits.view(np.float32)
    g = g[np.isfinite(g)]
    edges = np.array([0.0, -0.0, 88.72, -88.72, 89.0, -89.0, 103.9, -103.9, 104.0, -104.0,
                      16.6, 17.0, -16.6, np.inf, -np.inf, 1e-30, -1e-30], np.float32)
    g = np.concatenate([edges, g, rng.uniform(-110, 110, 1 << 20).astype(np.float32)])
    T, H = g.size, 8
    sd = np.ones((T, H), np.float32)
    want = O.shared_expert_gate(sd[:, :1].copy(), g, T=T, H=1, out_dtype=F32)[:, 0]
    ws = empty((m.moe_gate_workspace_size(T),), torch.uint8)
    for wsp in (None, ws):
        out = _out(T, H, F32)
        m.shared_expert_gate(to_dev(sd), F32, to_dev(g), T, H, out, F32, wsp,
                             0 if wsp is None else wsp.numel())
        got = to_host(out)[:, 0]
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_combine_gate_full_size_workload():
    # the combine/gate bandwidth workload: T=4096, K=8, H=2048, weights from the
    # renormalised softmax top-8 of N(0,1) logits over 128 experts
    cfg = W.COMBINE
    d = W.combine_inputs(cfg)
    T, K, H = cfg.T, cfg.K, cfg.H
    _, w, _, _ = O.route_topk(logits_in=d["logits"], T=T, H=1, E=cfg.E_logits, K=K)
    want = O.combine_gate(d["expert_out"], w, d["sd"], d["gl"], T=T, K=K, H=H, out_dtype=BF16)
    ws = empty((m.moe_gate_workspace_size(T),), torch.uint8)
    for wsp in (None, ws):
        out = _out(T, H, BF16)
        m.moe_combine_gate(to_dev(d["expert_out"]), BF16, to_dev(w), to_dev(d["sd"]), BF16,
                           to_dev(d["gl"]), 1.0, T, K, H, out, BF16, wsp,
                           0 if wsp is None else wsp.numel())
        assert np.array_equal(to_host(out), want)


def test_refusals_enqueue_nothing():
    T, K, H = 2, 2, 8
    eo = torch.zeros((T, K, H), dtype=torch.float16, device="cuda")
    out = _out(T, H, BF16)
    before = launches()
    with pytest.raises(m.MoeError) as ei:
        m.moe_combine(eo, m.F16, None, None, BF16, 1.0, T, K, H, out, BF16)
    assert ei.value.code == m.ERR_DTYPE and "f16" in str(ei.value)
    with pytest.raises(m.MoeError) as ei:
        m.shared_expert_gate(eo, m.F16, to_dev(np.zeros(T, np.float32)), T, H, out, BF16)
    assert ei.value.code == m.ERR_DTYPE
    small = empty((16,), torch.uint8)
    with pytest.raises(m.MoeError) as ei:
        m.shared_expert_gate(out, BF16, to_dev(np.zeros(T, np.float32)), 4096, H, out, BF16, small,
                             16)
    assert ei.value.code == m.ERR_WORKSPACE
    with pytest.raises(m.MoeError) as ei:
        m.moe_combine(out, BF16, None, None, BF16, 1.0, T, 0, H, out, BF16)
    assert ei.value.code == m.ERR_ARG
    with pytest.raises(m.MoeError) as ei:
        m.moe_combine(out, BF16, None, None, BF16, 1.0, T, K, 12, out, BF16)
    assert ei.value.code == m.ERR_ALIGN
    after = launches()
    assert after == before
    # T = 0 is a legal no-op
    assert m.moe_combine(out, BF16, None, None, BF16, 1.0, 0, K, H, out, BF16) == 0


def test_empty_batch_enqueues_nothing():
    # T = 0: every combine and gate op returns at once, with no launch
    d = empty((16,), torch.float32)
    before = launches()
    m.moe_combine(d, BF16, None, None, BF16, 1.0, 0, 8, 64, d, BF16)
    m.moe_combine_gate(d, BF16, None, d, BF16, d, 1.0, 0, 8, 64, d, BF16)
    m.shared_expert_gate(d, BF16, d, 0, 64, d, BF16)
    for k in ("combine", "combine_gate", "shared_gate", "gate_sigmoid"):
        assert launched_since(before, k) == 0, k
