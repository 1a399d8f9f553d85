"""The whole MoE expert block on the GPU against the CPU oracle.

Tiny layer: every output element.  Full-size workloads (decode T=16, prefill
T=8192 with Zipf-skewed load, large T=2048 with a shared expert), in the same
launch configuration the benchmark times: stage by stage, each stage fed the
GPU's own inputs so that it is checked on its own --
  router   logits within the dot-product bound on sampled tokens; ids and
           weights bit-exact given the GPU logits
  permute  bit-exact (all rows)
  gate/up  sampled rows, NMSE <= 1e-5 and max rel <= 2e-2
  down     sampled rows, same tolerance
  combine  sampled tokens, bit-exact given the GPU's expert outputs
and end to end on sampled tokens (oracle from the raw inputs), excluding the
few tokens whose top-k set sits on a near-tie the logit bound cannot decide.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mixture_experts_ffn_renorm_gb300 as m
import oracle as O
from mixture_experts_ffn_renorm_gb300 import workloads as W
from mixture_experts_ffn_renorm_gb300.layer import MoeBlock

from .gpu_util import (GEMM_MAXREL, GEMM_NMSE, assert_gemm_close, bf16_to_f64, launched_since,
                       launches, nmse_maxrel, to_dev, to_host)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    m.lib()
    m.moe_device_status(clear=True)
    yield
    assert m.moe_device_status() == 0


def _block(cfg, d):
    return MoeBlock(cfg.H, cfg.I, cfg.E, cfg.K, d, max_tokens=cfg.T, device="cuda",
                    I_shared=cfg.I_shared)


def _oracle_tokens(cfg, d, tokens):
    return O.moe_layer_tokens(d["x"], d["w_router"], d["logit_bias"], d["w13"], d["w2"],
                              d["w_shared_gate"], d["w13_shared"], d["w2_shared"], H=cfg.H,
                              I=cfg.I, E=cfg.E, K=cfg.K, I_shared=cfg.I_shared,
                              tokens=np.asarray(tokens, np.int32))


def test_tiny_layer_every_element():
    cfg = W.TINY
    d = W.layer_inputs(cfg)
    blk = _block(cfg, d)
    before = launches()
    out = to_host(blk.forward(to_dev(d["x"])))
    for k in ("route_logits", "route_topk", "permute_small", "combine_gate"):
        assert launched_since(before, k) == 1, k
    # the shared expert runs inside the routed GEMM launches
    assert launched_since(before, "gemm_gateup") == 1 and launched_since(before, "gemm_down") == 1
    want, ids, w = _oracle_tokens(cfg, d, range(cfg.T))
    assert np.array_equal(to_host(blk.topk_ids), ids)
    nmse, rel = nmse_maxrel(bf16_to_f64(out), bf16_to_f64(want))
    assert nmse <= GEMM_NMSE and rel <= GEMM_MAXREL, (nmse, rel)


def _stagewise(cfg, n_tok_sample, n_row_sample):
    d = W.layer_inputs(cfg)
    T, H, I, E, K = cfg.T, cfg.H, cfg.I, cfg.E, cfg.K
    P = T * K
    blk = _block(cfg, d)
    x_dev = to_dev(d["x"])
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    out = to_host(blk.forward(x_dev))
    torch.cuda.synchronize()
    ids = to_host(blk.topk_ids)
    wts = to_host(blk.topk_w)
    rng = np.random.default_rng(99)
    toks = np.unique(np.concatenate([[0, T - 1], rng.choice(T, min(T, n_tok_sample), replace=False)]))

    # router: logits (re-run with logits_out, otherwise the forward's own call, so
    # that it takes the same path) within the bound; ids/w exact from them
    ws = blk.workspace
    gl_rerun = torch.empty((T,), dtype=torch.float32, device="cuda") if cfg.I_shared else None
    m.moe_route_topk(x_dev, blk.w_router, blk.logit_bias,
                     blk.w_shared_gate if cfg.I_shared else None, None, T, H, E, K, 1, 0, 1,
                     blk.topk_ids, blk.topk_w, logits, gl_rerun, ws, ws.numel())
    lo = to_host(logits)
    want_ids, want_w, _, _ = O.route_topk(logits_in=lo, T=T, H=1, E=E, K=K)
    assert np.array_equal(ids, want_ids) and np.array_equal(wts.view(np.uint32), want_w.view(np.uint32))
    _, _, lo_ora, _ = O.route_topk(d["x"][toks], d["w_router"], d["logit_bias"], T=len(toks), H=H,
                                   E=E, K=K, want_logits=True)
    xf, wf = bf16_to_f64(d["x"][toks]), bf16_to_f64(d["w_router"])
    bound = (H + 2) * 2.0**-23 * (np.abs(xf) @ np.abs(wf).T + (0 if d["logit_bias"] is None else np.abs(d["logit_bias"])))
    assert np.all(np.abs(lo[toks].astype(np.float64) - lo_ora) <= 2 * bound)
    if cfg.I_shared:
        # the shared-gate logit gl[t] = x[t,:] . wsg, within the same dot-product bound
        _, _, _, gl_ora = O.route_topk(d["x"][toks], d["w_router"], d["logit_bias"],
                                       d["w_shared_gate"], T=len(toks), H=H, E=E, K=K)
        gl_gpu = to_host(blk.gate_logit)[toks].astype(np.float64)
        gbound = (H + 2) * 2.0**-23 * (np.abs(xf) @ np.abs(bf16_to_f64(d["w_shared_gate"])))
        assert np.all(np.abs(gl_gpu - gl_ora) <= 2 * gbound)

    # permute: bit-exact over all rows
    off, sp, p2r, _ = O.permute(ids, None, T=T, K=K, E=E)
    assert np.array_equal(to_host(blk.expert_offsets), off)
    assert np.array_equal(to_host(blk.sorted_pair)[:P], sp)
    assert np.array_equal(to_host(blk.pair_to_row)[:P], p2r)
    counts = np.diff(off)
    big = int(np.argmax(counts))
    small = int(np.argmin(np.where(counts > 0, counts, P + 1)))
    rows = np.unique(np.concatenate([
        [0, P - 1], rng.choice(P, min(P, n_row_sample), replace=False),
        off[1:-1][off[1:-1] < P],            # first row of every expert (tile starts)
        np.arange(off[big], off[big + 1]),   # every row of the largest expert
        np.arange(off[small], off[small + 1]),   # and of the smallest non-empty one
    ])).astype(np.int32)
    # gate/up on sampled rows, fed the same routed rows of x the GPU used
    act = to_host(blk.act)
    if blk.x_perm is not None:
        assert np.array_equal(to_host(blk.x_perm)[rows], d["x"][sp[rows] // K])
    want_act = O.gateup_silu(d["x"], d["w13"], off, P=P, H=H, I=I, G=E, rows=rows,
                             a_row_gather=(sp // K).astype(np.int32))
    assert_gemm_close(act[rows], want_act[rows], "gate/up rows")

    # down on sampled rows, fed the GPU's own act
    eo = to_host(blk.expert_out)
    want_eo = O.down(act, d["w2"], off, P=P, I=I, H=H, G=E, pair_weight=wts.ravel(),
                     row_to_pair=sp, rows=rows)
    assert_gemm_close(eo[sp[rows]], want_eo[sp[rows]], "down rows")

    # combine on sampled tokens: bit-exact given the GPU's expert outputs
    eo3 = eo.reshape(T, K, H)
    if cfg.I_shared:
        sd = to_host(blk.sd)
        gl = to_host(blk.gate_logit)
        want_out = O.combine_gate(np.ascontiguousarray(eo3[toks]), None,
                                  np.ascontiguousarray(sd[toks]), np.ascontiguousarray(gl[toks]),
                                  T=len(toks), K=K, H=H)
        # the shared expert's two GEMMs, fed the GPU's own x and act
        Is = cfg.I_shared
        one = np.array([0, T], np.int32)
        sact = to_host(blk.act_shared)
        want_sact = O.gateup_silu(d["x"], d["w13_shared"], one, P=T, H=H, I=Is, G=1, rows=toks)
        assert_gemm_close(sact[toks], want_sact[toks], "shared gate/up")
        want_sd = O.down(sact, d["w2_shared"], one, P=T, I=Is, H=H, G=1, rows=toks)
        assert_gemm_close(sd[toks], want_sd[toks], "shared down")
    else:
        want_out = O.combine(np.ascontiguousarray(eo3[toks]), None, T=len(toks), K=K, H=H)
    assert np.array_equal(out[toks], want_out)

    # end to end from the raw inputs on sampled tokens
    want_tok, ora_ids, _ = _oracle_tokens(cfg, d, toks)
    same = np.all(np.sort(ora_ids, 1) == np.sort(ids[toks], 1), axis=1)
    assert same.mean() >= 0.95, f"routing differs on {np.sum(~same)} of {len(toks)} tokens"
    # end to end the two sides round each of the K expert rows to bf16 independently
    # (one-ulp flips of 2^-8 relative), so elements are compared against the
    # output's rms as well as their own size
    g, r = bf16_to_f64(out[toks][same]), bf16_to_f64(want_tok[same])
    nmse, _ = nmse_maxrel(g, r)
    rms = float(np.sqrt(np.mean(r * r)))
    worst = float(np.max(np.abs(g - r) / np.maximum(np.abs(r), rms)))
    assert nmse <= GEMM_NMSE and worst <= GEMM_MAXREL, (nmse, worst)
    return blk


def test_decode_layer_stagewise():
    _stagewise(W.DECODE, 16, 128)


@pytest.mark.slow
def test_prefill_zipf_layer_stagewise():
    blk = _stagewise(W.PREFILL, 48, 160)
    counts = np.diff(to_host(blk.expert_offsets))
    assert counts.max() > 4 * counts.mean()      # the load really is skewed


@pytest.mark.slow
def test_large_shared_layer_stagewise():
    _stagewise(W.LARGE, 32, 96)


@pytest.mark.parametrize("cfg", [W.DECODE, W.PREFILL], ids=["decode", "prefill"])
def test_materialised_x_perm_path_matches_gather_path(cfg):
    # decode runs single-CTA tiles, prefill CTA-pair tiles (gatherer warps in
    # both CTAs, the odd CTA's copies relayed to the even CTA's barrier)
    d = W.layer_inputs(cfg)
    x = to_dev(d["x"])
    a = to_host(MoeBlock(cfg.H, cfg.I, cfg.E, cfg.K, d, max_tokens=cfg.T, device="cuda",
                         gather=True).forward(x))
    blk = MoeBlock(cfg.H, cfg.I, cfg.E, cfg.K, d, max_tokens=cfg.T, device="cuda", gather=False)
    b = to_host(blk.forward(x))
    assert np.array_equal(a, b)
    sp = to_host(blk.sorted_pair)
    assert np.array_equal(to_host(blk.x_perm), d["x"][sp // cfg.K])


@pytest.mark.parametrize("cfg", [W.DECODE, W.PREFILL], ids=["decode", "prefill"])
def test_staged_rows_match_the_x_perm_path(cfg):
    # staged=True: the gate/up call writes x_perm itself (on CTA pairs inside the
    # GEMM launch, behind per-chunk flags whose value the workspace carries from
    # call to call); eager calls and graph replays must give the x_perm path's bits
    d = W.layer_inputs(cfg)
    x = to_dev(d["x"])
    ref = MoeBlock(cfg.H, cfg.I, cfg.E, cfg.K, d, max_tokens=cfg.T, device="cuda")
    want = to_host(ref.forward(x))
    blk = MoeBlock(cfg.H, cfg.I, cfg.E, cfg.K, d, max_tokens=cfg.T, device="cuda", staged=True)
    for _ in range(2):
        assert np.array_equal(to_host(blk.forward(x)), want)
    assert np.array_equal(to_host(blk.x_perm), to_host(ref.x_perm))
    blk.capture(x)
    for _ in range(2):
        assert np.array_equal(to_host(blk.replay()), want)
    assert m.moe_device_status() == 0


@pytest.mark.parametrize("cfg", [W.TINY, W.DECODE], ids=["tiny", "decode"])
def test_host_batches_match_forward(cfg):
    # run_host_batches: pinned host batches of different sizes go up on one
    # stream, compute on the current one and come back on a third, with the
    # device buffers double-buffered; every output must be the bits forward()
    # gives for the same batch, and the tiny layer's must match the oracle
    d = W.layer_inputs(cfg)
    blk = _block(cfg, d)
    rng = np.random.default_rng(11)
    sizes = [cfg.T, max(1, cfg.T - 3), 1, cfg.T, max(1, cfg.T // 2)]
    xs = [W.to_bf16_bits(rng.standard_normal((n, cfg.H)).astype(np.float32)) for n in sizes]
    xs[0] = d["x"]
    x_hosts = [torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory() for a in xs]
    out_hosts = [torch.empty((n, cfg.H), dtype=torch.bfloat16).pin_memory() for n in sizes]
    blk.run_host_batches(x_hosts, out_hosts)
    torch.cuda.synchronize()
    for a, o in zip(xs, out_hosts):
        want = to_host(blk.forward(to_dev(a)))
        assert np.array_equal(o.view(torch.int16).numpy().view(np.uint16), want)
    if cfg is W.TINY:
        want, _, _ = _oracle_tokens(cfg, d, range(cfg.T))
        got = out_hosts[0].view(torch.int16).numpy().view(np.uint16)
        nmse, _ = nmse_maxrel(bf16_to_f64(got), bf16_to_f64(want))
        assert nmse <= GEMM_NMSE


@pytest.mark.parametrize("cfg,gathers", [(W.DECODE, True), (W.PREFILL, False), (W.LARGE, False)],
                         ids=["decode", "prefill", "large"])
def test_gather_auto_picks_by_rows_per_expert(cfg, gathers):
    # gather="auto": at most 16 routed rows per expert (decode) read x inside the
    # gate/up GEMM and the permute copies no rows; larger batches (and the fused
    # shared expert of the large layer) keep x_perm.  The bits are those of the
    # x_perm path either way.
    d = W.layer_inputs(cfg)
    x = to_dev(d["x"])
    want = to_host(_block(cfg, d).forward(x))
    blk = MoeBlock(cfg.H, cfg.I, cfg.E, cfg.K, d, max_tokens=cfg.T, device="cuda",
                   I_shared=cfg.I_shared, gather="auto")
    before = launches()
    got = to_host(blk.forward(x))
    assert launched_since(before, "permute_gather") == (0 if gathers else 1)
    assert np.array_equal(got, want)


def test_two_blocks_on_two_streams_at_once():
    # the library keeps no per-call state outside the caller's buffers: two
    # layers enqueued on two streams without ordering between them give the
    # bits each gives alone
    cfgs = [W.DECODE, W.PREFILL]
    ds = [W.layer_inputs(c) for c in cfgs]
    blks = [_block(c, d) for c, d in zip(cfgs, ds)]
    xs = [to_dev(d["x"]) for d in ds]
    alone = [to_host(b.forward(x)) for b, x in zip(blks, xs)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    outs = [None, None]
    for rep in range(3):
        for i in (1, 0):
            with torch.cuda.stream(streams[i]):
                outs[i] = blks[i].forward(xs[i], stream=streams[i].cuda_stream)
        torch.cuda.synchronize()
        for i in range(2):
            assert np.array_equal(to_host(outs[i]), alone[i]), (rep, cfgs[i].name)


@pytest.mark.parametrize("cfg", [W.DECODE, W.LARGE], ids=["decode", "large"])
def test_pdl_off_gives_the_same_bits(cfg):
    # programmatic dependent launch only lets a kernel start its set-up early;
    # every kernel waits for its predecessor before touching global memory, so
    # plain stream order must give the same bits
    d = W.layer_inputs(cfg)
    blk = _block(cfg, d)
    x = to_dev(d["x"])
    on = to_host(blk.forward(x))
    prev = m.moe_set_pdl(False)
    try:
        off = to_host(blk.forward(x))
    finally:
        m.moe_set_pdl(prev)
    assert np.array_equal(on, off)


@pytest.mark.slow
def test_gemm_tilings_agree_on_prefill():
    # single-CTA and CTA-pair tiles differ only in f32 accumulation order
    cfg = W.PREFILL
    d = W.layer_inputs(cfg)
    blk = _block(cfg, d)
    x = to_dev(d["x"])
    res = {}
    prev = m.moe_set_gemm_pairing(m.GEMM_AUTO)
    try:
        for mode in (m.GEMM_SINGLE, m.GEMM_PAIR):
            m.moe_set_gemm_pairing(mode)
            res[mode] = (to_host(blk.forward(x)).copy(), to_host(blk.act).copy())
    finally:
        m.moe_set_gemm_pairing(prev)
    assert m.moe_device_status() == 0
    (out_s, act_s), (out_p, act_p) = res[m.GEMM_SINGLE], res[m.GEMM_PAIR]
    assert nmse_maxrel(bf16_to_f64(act_p), bf16_to_f64(act_s))[0] <= 1e-6
    assert nmse_maxrel(bf16_to_f64(out_p), bf16_to_f64(out_s))[0] <= 1e-6
