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

from .gpu_util import (assert_gemm_close, bf16_to_f64, empty, launched_since, launches, to_dev,
                       to_host)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    m.lib()
    m.moe_device_status(clear=True)
    yield
    assert m.moe_device_status() == 0


TILINGS = [m.GEMM_SINGLE, m.GEMM_PAIR]
TILING_IDS = ["single", "pair"]


@pytest.fixture(params=TILINGS, ids=TILING_IDS)
def tiling(request):
    """Every built tiling of the grouped GEMMs: single-CTA tiles with rows on the
    MMA's M side, and CTA-pair tiles with weight rows on M and up to 256 rows of
    a group on N (forced here for every shape, down to one-row groups)."""
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
    # group sizes, H, I
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
def test_gateup_silu(sizes, H, I, tiling):
    off, P, G, A, W13, _ = _case(sizes, H, I, sum(sizes) + H)
    want = O.gateup_silu(A, W13, off, P=P, H=H, I=I, G=G)
    act = empty((P, I), torch.bfloat16)
    act.fill_(0)
    before = launches()
    m.moe_grouped_gemm_gateup_silu_bf16(to_dev(A), P, None, 1, to_dev(W13), to_dev(off), P, H, I, G,
                                        act)
    assert launched_since(before, "gemm_gateup") == 1
    assert m.moe_device_status() == 0
    assert_gemm_close(to_host(act), want, "gate/up")


@pytest.mark.parametrize("sizes,H,I", SHAPES)
@pytest.mark.parametrize("K", [1, 3, 8])
def test_gateup_silu_gathered_rows(sizes, H, I, K, tiling):
    # product row r reads x[pair[r] // K]: the routed rows come straight from the
    # token matrix, copied by gatherer warps with cp.async (no x_perm); on CTA
    # pairs each CTA copies its half of a tile's tokens
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


@pytest.mark.parametrize("sizes,H,I", [([40, 0, 70, 1, 33] + [0] * 11, 256, 192),
                                       ([600, 5, 256, 255, 513], 256, 256)],
                         ids=["32-row tiles", "128-row tiles"])
def test_gateup_silu_gathered_rows_outside_x(sizes, H, I, tiling):
    # a gathered row whose source index lies outside [0, a_rows) reads zeros, on
    # the decode-sized 32-row tiles (one gatherer warp) and on 128-row tiles
    K = 4
    off, P, G, _, W13, _ = _case(sizes, H, I, 41 + H)
    rng = np.random.default_rng(P)
    T = (P + K - 1) // K + 1
    x = W.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    pair = rng.integers(0, T * K, P).astype(np.int32)
    pair[::13] = T * K + 3                            # row T: outside x
    pair[5::29] = -K                                  # row -1: outside x
    src = pair // K
    ok = (src >= 0) & (src < T)
    want = O.gateup_silu(np.concatenate([x, np.zeros((1, H), np.uint16)]), W13, off, P=P, H=H,
                         I=I, G=G, a_row_gather=np.where(ok, src, T).astype(np.int32))
    act = empty((P, I), torch.bfloat16)
    m.moe_grouped_gemm_gateup_silu_bf16(to_dev(x), T, to_dev(pair), K, to_dev(W13), to_dev(off), P,
                                        H, I, G, act)
    assert m.moe_device_status() == 0
    assert_gemm_close(to_host(act), want, "gathered gate/up, rows outside x")


@pytest.mark.parametrize("sizes,H,I", SHAPES + [([300, 0, 520], 2048, 768)])
def test_down_weight_scatter(sizes, H, I, tiling):
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
        assert launched_since(before, "gemm_down") == 1
        assert m.moe_device_status() == 0
        assert_gemm_close(to_host(out), want, "down")


@pytest.mark.parametrize("G", [513, 1024])
def test_most_groups_both_gemms(G, tiling):
    # more groups than a CTA-pair launch takes (512): the single-CTA schedule
    # tables at up to their 1024 groups, most groups empty or of one to three
    # rows (32-row tiles) -- gate/up and down against the oracle
    rng = np.random.default_rng(G)
    sizes = [int(v) for v in rng.choice([0, 0, 1, 2, 3, 40], G)]
    sizes[-1] = 70                                   # the last group spans three 32-row tiles
    H, I = 128, 64
    off, P, G_, A, W13, W2 = _case(sizes, H, I, G + 5)
    want = O.gateup_silu(A, W13, off, P=P, H=H, I=I, G=G_)
    act = empty((P, I), torch.bfloat16)
    m.moe_grouped_gemm_gateup_silu_bf16(to_dev(A), P, None, 1, to_dev(W13), to_dev(off), P, H, I,
                                        G_, act)
    assert m.moe_device_status() == 0
    assert_gemm_close(to_host(act), want, "gate/up, many groups")
    wts = rng.uniform(0.05, 1.0, P).astype(np.float32)
    r2p = rng.permutation(P).astype(np.int32)
    want_d = O.down(want, W2, off, P=P, I=I, H=H, G=G_, pair_weight=wts, row_to_pair=r2p)
    out = empty((P, H), torch.bfloat16)
    m.moe_grouped_gemm_down_bf16(to_dev(want), to_dev(W2), to_dev(off), to_dev(wts), to_dev(r2p), P,
                                 I, H, G_, out)
    assert m.moe_device_status() == 0
    assert_gemm_close(to_host(out), want_d, "down, many groups")


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


def test_gateup_narrowing_is_visible_on_the_gpu(tiling):
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


def test_single_group_without_offsets_and_rows_outside_groups(tiling):
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


def test_down_rounds_once_after_the_weight_on_the_gpu(tiling):
    # Issue #3094: the routing weight is applied before the down result is
    # stored, so the one bf16 rounding comes after the weight.  The dot product
    # y = 1 + 2^-8 + 2^-10 is exact in any summation order, so the tensor-core
    # result is fixed bit for bit: bf16(y * 0.75) = 0x3F41, where rounding y to
    # bf16 before the weight would give 0x3F42 (worked in the oracle's pin).
    I, H, P = 64, 256, 130
    act = np.zeros((P, I), np.float32)
    act[:, :3] = [1.0, 2.0**-8, 2.0**-10]
    w2 = np.zeros((2, H, I), np.float32)
    w2[:, :, :3] = 1.0
    off = np.array([0, 70, P], np.int32)
    r2p = np.random.default_rng(5).permutation(P).astype(np.int32)
    out = empty((P, H), torch.bfloat16)
    m.moe_grouped_gemm_down_bf16(to_dev(W.to_bf16_bits(act)), to_dev(W.to_bf16_bits(w2)),
                                 to_dev(off), to_dev(np.full(P, 0.75, np.float32)), to_dev(r2p),
                                 P, I, H, 2, out)
    assert m.moe_device_status() == 0
    assert np.all(to_host(out) == 0x3F41)
    m.moe_grouped_gemm_down_bf16(to_dev(W.to_bf16_bits(act)), to_dev(W.to_bf16_bits(w2)),
                                 to_dev(off), None, None, P, I, H, 2, out)
    assert np.all(to_host(out) == 0x3F81)     # no weight: bf16(y) = 1 + 1/128


def _zipf_sizes(G, total, s, seed):
    rng = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, G + 1) ** s
    sizes = rng.multinomial(total, p / p.sum())
    return [int(v) for v in rng.permutation(sizes)]


MULTI_ROUND = [
    # (group sizes, H, I): tiles outnumber the 152 SMs several times over, so every
    # persistent CTA walks several tiles and wraps its stage ring and both TMEM
    # accumulators many times
    (_zipf_sizes(64, 24000, 1.1, 3), 768, 384),        # 220 M-tiles x 3 N-tiles each GEMM
    ([1 + (g % 2) for g in range(128)], 2048, 768),     # decode-like: 32-row tiles, 1536 and 1024 tiles
]


@pytest.mark.parametrize("sizes,H,I", MULTI_ROUND, ids=["zipf24k", "decode128"])
def test_multi_round_schedule_every_row(sizes, H, I, tiling):
    off, P, G, A, W13, W2 = _case(sizes, H, I, 11 + H)
    act = empty((P, I), torch.bfloat16)
    m.moe_grouped_gemm_gateup_silu_bf16(to_dev(A), P, None, 1, to_dev(W13), to_dev(off), P, H, I,
                                        G, act)
    assert m.moe_device_status() == 0
    got_act = to_host(act)
    want_act = O.gateup_silu(A, W13, off, P=P, H=H, I=I, G=G)
    assert_gemm_close(got_act, want_act, "multi-round gate/up")
    # every row on its own too: a wrong tile leaves a row far off even when the
    # whole-matrix NMSE is small
    g, r = bf16_to_f64(got_act), bf16_to_f64(want_act)
    row_err = np.sum((g - r) ** 2, 1) / np.maximum(np.sum(r * r, 1), 1e-30)
    assert row_err.max() <= 1e-4, (int(row_err.argmax()), float(row_err.max()))
    rng = np.random.default_rng(P)
    wts = rng.uniform(0.05, 1.0, P).astype(np.float32)
    r2p = rng.permutation(P).astype(np.int32)
    out = empty((P, H), torch.bfloat16)
    m.moe_grouped_gemm_down_bf16(act, to_dev(W2), to_dev(off), to_dev(wts), to_dev(r2p), P, I, H,
                                 G, out)
    assert m.moe_device_status() == 0
    want = O.down(got_act, W2, off, P=P, I=I, H=H, G=G, pair_weight=wts, row_to_pair=r2p)
    got = to_host(out)
    assert_gemm_close(got, want, "multi-round down")
    g, r = bf16_to_f64(got), bf16_to_f64(want)
    row_err = np.sum((g - r) ** 2, 1) / np.maximum(np.sum(r * r, 1), 1e-30)
    assert row_err.max() <= 1e-4, (int(row_err.argmax()), float(row_err.max()))


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


def _staged_ws(P):
    # zero-filled once; later calls pass it unchanged
    return torch.zeros(max(1, m.moe_gateup_staged_workspace_size(P)), dtype=torch.uint8,
                       device="cuda")


def _staged(x, T, pair, K, W13, off, P, H, I, G, ws):
    xp = empty((P, H), torch.bfloat16)
    act = empty((P, I), torch.bfloat16)
    before = launches()
    m.moe_grouped_gemm_gateup_silu_bf16_staged(to_dev(x), T, to_dev(pair), K, xp, to_dev(W13),
                                               to_dev(off), P, H, I, G, act, ws, ws.numel())
    assert launched_since(before, "gemm_gateup") == 1
    assert m.moe_device_status() == 0
    return to_host(xp), to_host(act)


@pytest.mark.parametrize("sizes,H,I", SHAPES)
@pytest.mark.parametrize("K", [1, 8])
def test_gateup_silu_staged_rows(sizes, H, I, K, tiling):
    # x_perm is written by the call itself (on CTA pairs by stager warps of the
    # GEMM launch, ahead of the tiles that read it): it must hold x[pair // K],
    # and act must be the oracle's and bit-identical to the x_perm entry on it
    off, P, G, _, W13, _ = _case(sizes, H, I, sum(sizes) + 5 * H + K)
    rng = np.random.default_rng(P + 31 * K)
    T = max(1, (P + K - 1) // K) + 2
    x = W.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    pair = rng.integers(0, T * K, P).astype(np.int32)
    ws = _staged_ws(P)
    xp, act = _staged(x, T, pair, K, W13, off, P, H, I, G, ws)
    assert np.array_equal(xp, x[pair // K])
    want = O.gateup_silu(x, W13, off, P=P, H=H, I=I, G=G, a_row_gather=(pair // K).astype(np.int32))
    assert_gemm_close(act, want, "staged gate/up")
    ref = empty((P, I), torch.bfloat16)
    m.moe_grouped_gemm_gateup_silu_bf16(to_dev(xp), P, None, 1, to_dev(W13), to_dev(off), P, H, I,
                                        G, ref)
    assert np.array_equal(act, to_host(ref))


def test_staged_rows_repeated_calls_and_out_of_range_rows(tiling):
    # one workspace over several calls with new inputs each time: every call must
    # wait for its own chunks (the flags of earlier launches mean nothing to it);
    # source rows outside [0, T) are staged as zeros
    sizes, H, I = _zipf_sizes(16, 6000, 1.1, 7), 512, 256
    off, P, G, _, W13, _ = _case(sizes, H, I, 77)
    K, T = 8, 6000 // 8 + 1
    ws = _staged_ws(P)
    for call in range(3):
        rng = np.random.default_rng(100 + call)
        x = W.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
        pair = rng.integers(0, T * K, P).astype(np.int32)
        pair[::97] = T * K + 5                        # row T: outside x
        xp, act = _staged(x, T, pair, K, W13, off, P, H, I, G, ws)
        src = pair // K
        ok = src < T
        assert np.array_equal(xp[ok], x[src[ok]])
        assert not xp[~ok].any()
        want = O.gateup_silu(np.concatenate([x, np.zeros((1, H), np.uint16)]), W13, off, P=P, H=H,
                             I=I, G=G, a_row_gather=np.minimum(src, T).astype(np.int32))
        assert_gemm_close(act, want, f"staged gate/up, call {call}")


@pytest.mark.parametrize("sizes,H,I", MULTI_ROUND[:1], ids=["zipf24k"])
def test_staged_rows_multi_round_every_row(sizes, H, I, tiling):
    # several rounds of tiles per CTA, every row compared with the oracle
    off, P, G, A, W13, _ = _case(sizes, H, I, 13 + H)
    K = 8
    pair = np.random.default_rng(P).integers(0, P * K, P).astype(np.int32)
    src = pair // K                                   # rows of A, used as x (T = P)
    xp, act = _staged(A, P, pair, K, W13, off, P, H, I, G, _staged_ws(P))
    assert np.array_equal(xp, A[src])
    want = O.gateup_silu(A, W13, off, P=P, H=H, I=I, G=G, a_row_gather=src.astype(np.int32))
    assert_gemm_close(act, want, "staged multi-round gate/up")
    g, r = bf16_to_f64(act), bf16_to_f64(want)
    row_err = np.sum((g - r) ** 2, 1) / np.maximum(np.sum(r * r, 1), 1e-30)
    assert row_err.max() <= 1e-4, (int(row_err.argmax()), float(row_err.max()))
