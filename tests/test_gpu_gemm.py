"""GPU parity of the grouped BF16 GEMMs (tcgen05) against the CPU oracle.

kMoeGroupedGemmBf16GateUpSilu and kMoeGroupedGemmBf16 (vllm.cpp issue #3094
"Row: BACKEND-ROCM-BF16-MOE"): stage-wise, the oracle consumes the same A, and
the outputs must have NMSE <= 1e-5 and max relative error <= 2e-2 against the
oracle's f32-accumulated bf16 result.  Shapes span several M, N and K tiles,
ragged tails in every dimension, empty and one-row groups."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mixture_experts_ffn_renorm_gb300 as m
import oracle as O
from mixture_experts_ffn_renorm_gb300 import workloads as W

from .gpu_util import assert_gemm_close, empty, launched_since, launches, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    m.lib()
    m.moe_device_status(clear=True)
    yield
    assert m.moe_device_status() == 0


@pytest.fixture(params=[m.GEMM_SINGLE, m.GEMM_MCAST, m.GEMM_PAIR, m.GEMM_SPLIT, m.GEMM_TALL],
                ids=["single", "mcast", "pair", "split", "tall"])
def pairing(request):
    """Every tiling of the grouped GEMMs: single CTAs (the default), A-multicast
    clusters, CTA pairs (2-SM, 256-row tiles), and whole 256-row blocks on CTA
    pairs with the rest on A-multicast clusters."""
    prev = m.moe_set_gemm_pairing(request.param)
    yield request.param
    m.moe_set_gemm_pairing(prev)


def _case(sizes, H, I, seed):
    rng = np.random.default_rng(seed)
    G = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    P = int(off[-1])
    A = W.to_bf16_bits(rng.standard_normal((P, H)).astype(np.float32))
    W13 = W.to_bf16_bits((0.02 * rng.standard_normal((G, 2 * I, H))).astype(np.float32))
    W2 = W.to_bf16_bits((0.02 * rng.standard_normal((G, H, I))).astype(np.float32))
    return off, P, G, A, W13, W2


SHAPES = [
    # group sizes, H, I  (I / 128 and H / 256 even or odd: multicast or its fallback)
    ([4], 64, 32),
    ([3, 200, 0, 77], 512, 256),
    ([600, 5, 256, 255, 513], 256, 256),
    ([0, 1, 130, 129, 40], 256, 192),
    ([300], 512, 128),
    ([1, 1, 1, 1, 1, 1, 1, 1], 2048, 768),
    ([257, 0, 0, 3], 136, 72),
    ([128, 128, 255, 1], 1024, 256),
    # few rows per expert (P <= 16 G): 32-row tiles, experts spanning several of them
    ([40, 0, 70, 1, 33] + [0] * 11, 256, 192),
    ([2, 1, 0, 3] * 16 + [97], 512, 128),
]


@pytest.mark.parametrize("sizes,H,I", SHAPES + [([300, 0, 520], 2048, 768)])
def test_gateup_silu(sizes, H, I, pairing):
    off, P, G, A, W13, _ = _case(sizes, H, I, sum(sizes) + H)
    want = O.gateup_silu(A, W13, off, P=P, H=H, I=I, G=G)
    act = empty((P, I), torch.bfloat16)
    act.fill_(0)
    before = launches()
    m.moe_grouped_gemm_gateup_silu_bf16(to_dev(A), P, None, 1, to_dev(W13), to_dev(off), P, H, I, G,
                                        act)
    assert launched_since(before, "gemm_gateup") == (2 if pairing == m.GEMM_SPLIT else 1)
    assert m.moe_device_status() == 0
    assert_gemm_close(to_host(act), want, "gate/up")


@pytest.mark.parametrize("sizes,H,I", SHAPES)
@pytest.mark.parametrize("K", [1, 3, 8])
def test_gateup_silu_gathered_rows(sizes, H, I, K):
    # product row r reads x[pair[r] // K]: the routed rows come straight from the
    # token matrix through TMA gather4 (no x_perm)
    off, P, G, _, W13, _ = _case(sizes, H, I, sum(sizes) + 7 * H + K)
    rng = np.random.default_rng(P + K)
    T = max(1, (P + K - 1) // K) + 3
    x = W.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    pair = rng.integers(0, T * K, P).astype(np.int32)
    want = O.gateup_silu(x, W13, off, P=P, H=H, I=I, G=G, a_row_gather=(pair // K).astype(np.int32))
    act = empty((P, I), torch.bfloat16)
    act.fill_(0)
    before = launches()
    m.moe_grouped_gemm_gateup_silu_bf16(to_dev(x), T, to_dev(pair), K, to_dev(W13), to_dev(off), P,
                                        H, I, G, act)
    assert launched_since(before, "gemm_gateup") == 1
    assert m.moe_device_status() == 0
    assert_gemm_close(to_host(act), want, "gathered gate/up")


@pytest.mark.parametrize("sizes,H,I", SHAPES + [([300, 0, 520], 2048, 768)])
def test_down_weight_scatter(sizes, H, I, pairing):
    off, P, G, _, _, W2 = _case(sizes, H, I, sum(sizes) + I)
    rng = np.random.default_rng(1)
    act = W.to_bf16_bits(rng.standard_normal((P, I)).astype(np.float32))
    wts = rng.uniform(0.05, 1.0, P).astype(np.float32)
    r2p = rng.permutation(P).astype(np.int32)
    for pw, rp in ((wts, r2p), (None, None), (wts, None)):
        want = O.down(act, W2, off, P=P, I=I, H=H, G=G, pair_weight=pw, row_to_pair=rp)
        out = empty((P, H), torch.bfloat16)
        out.fill_(0)
        before = launches()
        m.moe_grouped_gemm_down_bf16(to_dev(act), to_dev(W2), to_dev(off),
                                     None if pw is None else to_dev(pw),
                                     None if rp is None else to_dev(rp), P, I, H, G, out)
        assert launched_since(before, "gemm_down") == (2 if pairing == m.GEMM_SPLIT else 1)
        assert m.moe_device_status() == 0
        assert_gemm_close(to_host(out), want, "down")


FUSED = [
    # routed group sizes, H, I, shared rows Ts, shared I_s (ragged tiles on both sides)
    ([3, 200, 0, 77], 512, 256, 130, 192),
    ([600, 5, 256, 255, 513], 256, 256, 1, 64),
    ([1, 1, 1, 1, 1, 1, 1, 1], 2048, 768, 16, 256),
    ([0, 0], 256, 128, 300, 128),          # no routed rows: the shared GEMM alone
    ([40, 9], 256, 128, 0, 128),           # no shared rows: the routed GEMM alone
    ([4, 3], 64, 32, 4, 32),               # narrower than one tile everywhere
    ([257, 0, 0, 3], 136, 72, 70, 40),     # K and N not multiples of the tile
]


@pytest.mark.parametrize("sizes,H,I,Ts,Is", FUSED)
def test_fused_shared_expert_launch(sizes, H, I, Ts, Is):
    # the routed GEMM and the shared expert's GEMM in one launch: bit-identical
    # to the two separate launches (same tiles, same K order), and the shared
    # half within tolerance of the oracle
    off, P, G, A, W13, W2 = _case(sizes, H, I, sum(sizes) + Ts + Is)
    rng = np.random.default_rng(Ts + 3 * Is)
    xs = W.to_bf16_bits(rng.standard_normal((Ts, H)).astype(np.float32))
    w13s = W.to_bf16_bits((0.02 * rng.standard_normal((1, 2 * Is, H))).astype(np.float32))
    w2s = W.to_bf16_bits((0.02 * rng.standard_normal((1, H, Is))).astype(np.float32))
    wts = rng.uniform(0.05, 1.0, P).astype(np.float32)
    r2p = rng.permutation(P).astype(np.int32)
    dA, dW13, dW2, doff = to_dev(A), to_dev(W13), to_dev(W2), to_dev(off)
    dxs, dw13s, dw2s, dwts, dr2p = to_dev(xs), to_dev(w13s), to_dev(w2s), to_dev(wts), to_dev(r2p)

    def bufs(rows, cols):
        t = empty((rows, cols), torch.bfloat16)
        t.fill_(0)
        return t

    act_a, acts_a, out_a, sd_a = bufs(P, I), bufs(Ts, Is), bufs(P, H), bufs(Ts, H)
    m.moe_grouped_gemm_gateup_silu_bf16(dA, P, None, 1, dW13, doff, P, H, I, G, act_a)
    m.moe_grouped_gemm_gateup_silu_bf16(dxs, Ts, None, 1, dw13s, None, Ts, H, Is, 1, acts_a)
    m.moe_grouped_gemm_down_bf16(act_a, dW2, doff, dwts, dr2p, P, I, H, G, out_a)
    m.moe_grouped_gemm_down_bf16(acts_a, dw2s, None, None, None, Ts, Is, H, 1, sd_a)

    act_b, acts_b, out_b, sd_b = bufs(P, I), bufs(Ts, Is), bufs(P, H), bufs(Ts, H)
    before = launches()
    m.moe_grouped_gemm_gateup_silu_bf16_shared(dA, dW13, doff, P, H, I, G, act_b, dxs, Ts, dw13s,
                                               Is, acts_b)
    m.moe_grouped_gemm_down_bf16_shared(act_b, dW2, doff, dwts, dr2p, P, I, H, G, out_b, acts_b,
                                        Ts, dw2s, Is, sd_b)
    assert launched_since(before, "gemm_gateup") == 1
    assert launched_since(before, "gemm_down") == 1
    assert m.moe_device_status() == 0
    for a, b in ((act_a, act_b), (acts_a, acts_b), (out_a, out_b), (sd_a, sd_b)):
        assert np.array_equal(to_host(a), to_host(b))
    if Ts:
        one = np.array([0, Ts], np.int32)
        want_acts = O.gateup_silu(xs, w13s, one, P=Ts, H=H, I=Is, G=1)
        assert_gemm_close(to_host(acts_b), want_acts, "fused shared gate/up")
        want_sd = O.down(to_host(acts_b), w2s, one, P=Ts, I=Is, H=H, G=1)
        assert_gemm_close(to_host(sd_b), want_sd, "fused shared down")
    if P:
        want_act = O.gateup_silu(A, W13, off, P=P, H=H, I=I, G=G)
        assert_gemm_close(to_host(act_b), want_act, "fused routed gate/up")


def test_fused_shared_refusals():
    x = empty((4, 64), torch.bfloat16)
    before = launches()
    with pytest.raises(m.MoeError) as ei:   # I_shared not a multiple of 8
        m.moe_grouped_gemm_gateup_silu_bf16_shared(x, x, None, 4, 64, 64, 1, x, x, 4, x, 36, x)
    assert ei.value.code == m.ERR_ALIGN
    with pytest.raises(m.MoeError) as ei:   # shared rows without operands
        m.moe_grouped_gemm_down_bf16_shared(x, x, None, None, None, 4, 64, 64, 1, x, None, 4,
                                            None, 64, None)
    assert ei.value.code == m.ERR_ARG
    assert launches() == before


FP8_SHAPES = [
    # group sizes, H, I (few-row histograms take the 32-row tiles)
    ([3, 200, 0, 77], 512, 256),
    ([1, 1, 1, 1, 1, 1, 1, 1], 2048, 768),
    ([40, 0, 70, 1, 33] + [0] * 11, 256, 192),
    ([600, 5, 256, 255, 513], 256, 256),
    ([257, 0, 0, 3], 144, 80),
]


def _fp8_weights(rng, G, R, C):
    q = rng.integers(0, 256, (G, R, C), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x40                      # no NaN codes
    scale = rng.uniform(1e-4, 3e-3, (G, (R + 127) // 128, (C + 127) // 128)).astype(np.float32)
    return q, scale


@pytest.mark.parametrize("sizes,H,I", FP8_SHAPES)
def test_fp8_weight_gemms_against_the_oracle(sizes, H, I):
    # block-scaled FP8 weights: the GPU dequantises in shared memory exactly as
    # the oracle does (bf16(f32(code) * scale)), then the bf16 GEMM contract
    off, P, G, A, _, _ = _case(sizes, H, I, sum(sizes) + 3 * H + I)
    rng = np.random.default_rng(P + H)
    q13, s13 = _fp8_weights(rng, G, 2 * I, H)
    q2, s2 = _fp8_weights(rng, G, H, I)
    W13 = O.dequant_fp8_block(q13, s13, G=G, R=2 * I, C=H)
    W2 = O.dequant_fp8_block(q2, s2, G=G, R=H, C=I)
    want_act = O.gateup_silu(A, W13, off, P=P, H=H, I=I, G=G)
    act = empty((P, I), torch.bfloat16)
    act.fill_(0)
    before = launches()
    m.moe_grouped_gemm_gateup_silu_fp8w(to_dev(A), to_dev(q13), to_dev(s13), to_dev(off), P, H, I,
                                        G, act)
    assert launched_since(before, "gemm_gateup") == 1
    assert m.moe_device_status() == 0
    got_act = to_host(act)
    assert_gemm_close(got_act, want_act, "fp8 gate/up")
    wts = rng.uniform(0.05, 1.0, P).astype(np.float32)
    r2p = rng.permutation(P).astype(np.int32)
    want = O.down(got_act, W2, off, P=P, I=I, H=H, G=G, pair_weight=wts, row_to_pair=r2p)
    out = empty((P, H), torch.bfloat16)
    out.fill_(0)
    m.moe_grouped_gemm_down_fp8w(act, to_dev(q2), to_dev(s2), to_dev(off), to_dev(wts),
                                 to_dev(r2p), P, I, H, G, out)
    assert m.moe_device_status() == 0
    assert_gemm_close(to_host(out), want, "fp8 down")


def test_fp8_weights_equal_their_bf16_dequantisation_on_the_gpu():
    # the FP8 path against the bf16 path fed the oracle's dequantised weights:
    # same tiles, same K order, so the results are bit-identical
    sizes, H, I = [300, 0, 520, 7], 512, 256
    off, P, G, A, _, _ = _case(sizes, H, I, 77)
    rng = np.random.default_rng(78)
    q13, s13 = _fp8_weights(rng, G, 2 * I, H)
    W13 = O.dequant_fp8_block(q13, s13, G=G, R=2 * I, C=H)
    a, b = empty((P, I), torch.bfloat16), empty((P, I), torch.bfloat16)
    m.moe_grouped_gemm_gateup_silu_fp8w(to_dev(A), to_dev(q13), to_dev(s13), to_dev(off), P, H, I,
                                        G, a)
    m.moe_grouped_gemm_gateup_silu_bf16(to_dev(A), P, None, 1, to_dev(W13), to_dev(off), P, H, I,
                                        G, b)
    assert np.array_equal(to_host(a), to_host(b))


def test_fp8_refusals():
    x = empty((4, 64), torch.bfloat16)
    q = empty((1, 128, 64), torch.uint8)
    before = launches()
    with pytest.raises(m.MoeError) as ei:      # scales missing
        m.moe_grouped_gemm_gateup_silu_fp8w(x, q, None, None, 4, 64, 64, 1, x)
    assert ei.value.code == m.ERR_ARG
    with pytest.raises(m.MoeError) as ei:      # contraction length not a multiple of 16
        m.moe_grouped_gemm_down_fp8w(x, q, empty((1,), torch.float32), None, None, None, 4, 72,
                                     64, 1, x)
    assert ei.value.code == m.ERR_ALIGN
    assert launches() == before


def test_gateup_narrowing_is_visible_on_the_gpu(pairing):
    # g = u = 1 + 2^-9 exactly: narrowing before the activation gives
    # bf16(silu(1) * 1) = 0x3F3B; without it the result would be 0x3F3C
    H, I = 64, 32
    A = np.zeros((1, H), np.float32)
    A[0, 0], A[0, 1] = 1.0, 2.0**-9
    Wt = np.zeros((1, 2 * I, H), np.float32)
    Wt[0, :, 0] = 1.0
    Wt[0, :, 1] = 1.0
    act = empty((1, I), torch.bfloat16)
    m.moe_grouped_gemm_gateup_silu_bf16(to_dev(W.to_bf16_bits(A)), 1, None, 1,
                                        to_dev(W.to_bf16_bits(Wt)), to_dev(np.array([0, 1], np.int32)),
                                        1, H, I, 1, act)
    assert np.all(to_host(act) == 0x3F3B)


def test_single_group_without_offsets_and_rows_outside_groups(pairing):
    H, I, P = 128, 64, 200
    rng = np.random.default_rng(2)
    A = W.to_bf16_bits(rng.standard_normal((P, H)).astype(np.float32))
    W13 = W.to_bf16_bits((0.05 * rng.standard_normal((1, 2 * I, H))).astype(np.float32))
    act = empty((P, I), torch.bfloat16)
    m.moe_grouped_gemm_gateup_silu_bf16(to_dev(A), P, None, 1, to_dev(W13), None, P, H, I, 1, act)
    want = O.gateup_silu(A, W13, np.array([0, P], np.int32), P=P, H=H, I=I, G=1)
    assert_gemm_close(to_host(act), want, "single group")
    # rows past group_offsets[G] are not written
    off = np.array([0, 150], np.int32)
    act.fill_(0)
    m.moe_grouped_gemm_gateup_silu_bf16(to_dev(A), P, None, 1, to_dev(W13), to_dev(off), P, H, I, 1,
                                        act)
    h = to_host(act)
    assert np.all(h[150:] == 0)
    assert_gemm_close(h[:150], want[:150], "partial group")


def test_gemm_refusals_and_empty():
    act = empty((4, 64), torch.bfloat16)
    with pytest.raises(m.MoeError) as ei:
        m.moe_grouped_gemm_gateup_silu_bf16(act, 4, None, 1, act, None, 4, 64, 60, 1, act)
    assert ei.value.code == m.ERR_ALIGN
    with pytest.raises(m.MoeError) as ei:
        m.moe_grouped_gemm_gateup_silu_bf16(act, 4, None, 1, act, None, 4, 64, 32, 2, act)
    assert ei.value.code == m.ERR_ARG
    before = launches()
    assert m.moe_grouped_gemm_down_bf16(act, act, None, None, None, 0, 64, 64, 1, act) == 0
    assert launches() == before
