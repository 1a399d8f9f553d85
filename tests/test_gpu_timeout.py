"""The bounded-wait path of the grouped GEMMs, made to run out on purpose
without a faulty kernel.

Issue #1590 "kSharedExpertGate is CPU-only" asks for failures that are named,
not left to hang.  Every pipeline wait inside the GEMM kernels has a limit,
which moe_set_wait_limit_ns shortens.  At 1 us a prefill-sized gate/up or down
launch cannot finish: with K = 2048 in both GEMMs, its epilogue waits about
15 us for the first accumulator (a suspended probe may overrun its 1 us hint,
so a wait of a few microseconds can still complete in time).  The launch must
still end, raise MOE_STATUS_TIMEOUT in the status
word, and leave the device usable: with the limit restored and the status
cleared, the next calls in the same process give the same bits as before, and
those match the oracle.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mixture_experts_ffn_renorm_gb300 as m
import oracle as O
from mixture_experts_ffn_renorm_gb300 import workloads as W

from .gpu_util import assert_gemm_close, empty, launched_since, launches, to_dev, to_host

pytestmark = pytest.mark.gpu

FULL_LIMIT_NS = 10**9


@pytest.fixture(autouse=True)
def _restore_limit():
    m.lib()
    m.moe_device_status(clear=True)
    yield
    m.moe_set_wait_limit_ns(FULL_LIMIT_NS)
    m.moe_device_status(clear=True)


def _problem():
    rng = np.random.default_rng(1590)
    G, H, I = 8, 2048, 2048
    sizes = rng.multinomial(8192, np.full(G, 1.0 / G))
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    P = int(off[-1])
    A = W.to_bf16_bits(rng.standard_normal((P, H)).astype(np.float32))
    W13 = W.to_bf16_bits((0.02 * rng.standard_normal((G, 2 * I, H))).astype(np.float32))
    W2 = W.to_bf16_bits((0.02 * rng.standard_normal((G, H, I))).astype(np.float32))
    wts = rng.uniform(0.05, 1.0, P).astype(np.float32)
    r2p = rng.permutation(P).astype(np.int32)
    return G, H, I, P, off, A, W13, W2, wts, r2p


@pytest.fixture(params=[m.GEMM_SINGLE, m.GEMM_PAIR], ids=["single", "pair"])
def tiling(request):
    prev = m.moe_set_gemm_pairing(request.param)
    yield request.param
    m.moe_set_gemm_pairing(prev)


def test_wait_limit_expiry_is_reported_and_the_device_stays_usable(tiling):
    G, H, I, P, off, A, W13, W2, wts, r2p = _problem()
    dA, dW13, dW2, doff = to_dev(A), to_dev(W13), to_dev(W2), to_dev(off)
    dwts, dr2p = to_dev(wts), to_dev(r2p)
    act = empty((P, I), torch.bfloat16)
    out = empty((P, H), torch.bfloat16)

    def run():
        m.moe_grouped_gemm_gateup_silu_bf16(dA, P, None, 1, dW13, doff, P, H, I, G, act)
        m.moe_grouped_gemm_down_bf16(act, dW2, doff, dwts, dr2p, P, I, H, G, out)
        torch.cuda.synchronize()
        return to_host(act), to_host(out)

    ref_act, ref_out = run()
    assert m.moe_device_status() == 0

    # gathered rows (identity gather: row r reads A row r) take the gatherer
    # warps' waits, and on CTA pairs the odd CTA's relay
    ident = to_dev(np.arange(P, dtype=np.int32))
    act_g = empty((P, I), torch.bfloat16)

    def gathered():
        return m.moe_grouped_gemm_gateup_silu_bf16(dA, P, ident, 1, dW13, doff, P, H, I, G, act_g)

    # staged rows (identity again): on CTA pairs the tiles also wait for the
    # chunks that stager warps of other CTAs write; the workspace carries the
    # flag value of the last launch across the timed-out call
    act_s = empty((P, I), torch.bfloat16)
    xp_s = empty((P, H), torch.bfloat16)
    ws_s = torch.zeros(m.moe_gateup_staged_workspace_size(P), dtype=torch.uint8, device="cuda")

    def staged():
        return m.moe_grouped_gemm_gateup_silu_bf16_staged(dA, P, ident, 1, xp_s, dW13, doff, P, H,
                                                          I, G, act_s, ws_s, ws_s.numel())

    # a 1 us limit: every launch gives up, reports it and ends
    m.moe_set_wait_limit_ns(1000)
    for call in ("gateup", "gateup_gather", "gateup_staged", "down"):
        before = launches()
        if call == "gateup":
            rc = m.moe_grouped_gemm_gateup_silu_bf16(dA, P, None, 1, dW13, doff, P, H, I, G, act)
        elif call == "gateup_gather":
            rc = gathered()
        elif call == "gateup_staged":
            rc = staged()
        else:
            rc = m.moe_grouped_gemm_down_bf16(act, dW2, doff, dwts, dr2p, P, I, H, G, out)
        assert rc == m.OK                       # the launch itself was accepted
        torch.cuda.synchronize()                # and the kernel ended
        assert launched_since(before, "gemm_" + call.split("_")[0]) == 1
        status = m.moe_device_status(clear=True)
        assert status & m.STATUS_TIMEOUT, f"{call}: status {status}"
        assert m.moe_device_status() == 0

    # limit restored: the same process computes the same bits again
    m.moe_set_wait_limit_ns(FULL_LIMIT_NS)
    got_act, got_out = run()
    assert gathered() == m.OK
    assert staged() == m.OK
    torch.cuda.synchronize()
    assert m.moe_device_status() == 0
    assert np.array_equal(got_act, ref_act)
    assert np.array_equal(to_host(act_g), ref_act)
    assert np.array_equal(to_host(act_s), ref_act)
    assert np.array_equal(to_host(xp_s), A)
    assert np.array_equal(got_out, ref_out)
    # and they are the oracle's, on sampled rows
    rows = np.unique(np.concatenate([off[:-1], np.random.default_rng(3).choice(P, 200, False),
                                     [P - 1]])).astype(np.int32)
    want_act = O.gateup_silu(A, W13, off, P=P, H=H, I=I, G=G, rows=rows)
    assert_gemm_close(got_act[rows], want_act[rows], "gate/up after a timeout")
    want_out = O.down(got_act, W2, off, P=P, I=I, H=H, G=G, pair_weight=wts, row_to_pair=r2p,
                      rows=rows)
    assert_gemm_close(got_out[r2p[rows]], want_out[r2p[rows]], "down after a timeout")


def test_wait_limit_expiry_on_decode_sized_gathered_tiles():
    # few rows per group (P <= 16 G): 32-row tiles whose rows one gatherer warp
    # copies from x; the 1 us limit makes every launch give up and report it,
    # and with the limit restored the gathered call gives the x_perm call's bits
    rng = np.random.default_rng(16)
    G, H, I = 128, 2048, 2048
    sizes = rng.choice([0, 1, 1, 2, 3], G)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    P = int(off[-1])
    K = 8
    T = (P + K - 1) // K + 1
    x = W.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    pair = rng.permutation(T * K)[:P].astype(np.int32)
    W13 = W.to_bf16_bits((0.02 * rng.standard_normal((G, 2 * I, H))).astype(np.float32))
    dx, dpair, dW13, doff = to_dev(x), to_dev(pair), to_dev(W13), to_dev(off)
    act = empty((P, I), torch.bfloat16)
    m.moe_set_wait_limit_ns(1000)
    before = launches()
    assert m.moe_grouped_gemm_gateup_silu_bf16(dx, T, dpair, K, dW13, doff, P, H, I, G, act) == m.OK
    torch.cuda.synchronize()
    assert launched_since(before, "gemm_gateup") == 1
    assert m.moe_device_status(clear=True) & m.STATUS_TIMEOUT
    m.moe_set_wait_limit_ns(FULL_LIMIT_NS)
    assert m.moe_grouped_gemm_gateup_silu_bf16(dx, T, dpair, K, dW13, doff, P, H, I, G, act) == m.OK
    ref = empty((P, I), torch.bfloat16)
    xp = to_dev(x[pair // K])
    assert m.moe_grouped_gemm_gateup_silu_bf16(xp, P, None, 1, dW13, doff, P, H, I, G, ref) == m.OK
    torch.cuda.synchronize()
    assert m.moe_device_status() == 0
    assert np.array_equal(to_host(act), to_host(ref))
    want = O.gateup_silu(x, W13, off, P=P, H=H, I=I, G=G, a_row_gather=(pair // K).astype(np.int32))
    assert_gemm_close(to_host(act), want, "gathered gate/up on 32-row tiles after a timeout")
