"""Pins of the keep-quant half of the oracle (CPU only).

The keep-quant expert GEMM is kMatmulBTQuant / kMatmulBTQuantGrouped of
vllm.cpp PR #523 ("What changed"): the expert matmul runs on GGUF Q8_0 / Q4_K
weight blocks with activations quantized to 8-bit blocks and exact integer
block sums.  Each pin below checks the oracle against something other than
itself:
  - fp16 conversion against NumPy's IEEE float16 cast (a library routine);
  - the Q4_K scale/min unpacking and both dequantisers against blocks whose
    values were worked out by hand from the GGUF block layouts;
  - the integer-core dot product against the plain definition: dequantise
    weights and activations exactly, then a float64 dot product;
  - the activation quantizer against exact cases (integer-valued blocks,
    half-way ties, zero and non-finite blocks) and its error bound;
  - the fused epilogues and the whole keep-quant layer against compositions
    of separately pinned pieces.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle as O
from mixture_experts_ffn_renorm_gb300 import workloads as W

Q8_0, Q4_K = O.Q8_0, O.Q4_K
FMT = {"q8_0": Q8_0, "q4_k": Q4_K}


def _bf16(x):
    return W.to_bf16_bits(np.asarray(x, np.float32))


# ---------------------------------------------------------------- fp16


def test_f32_to_f16_matches_numpy_cast():
    rng = np.random.default_rng(5)
    parts = [
        rng.standard_normal(4000).astype(np.float32) * np.float32(1000.0),
        rng.standard_normal(4000).astype(np.float32) * np.float32(1e-5),   # fp16 subnormals
        rng.standard_normal(2000).astype(np.float32) * np.float32(1e-8),   # below half the smallest
        np.array([65504.0, 65519.0, 65520.0, 7e4, -7e4, 0.0, -0.0, np.inf, -np.inf,
                  2.0 ** -24, 2.0 ** -25, 1.5 * 2.0 ** -25, 2.0 ** -26, 2.0 ** -14,
                  (1 + 2 ** -11) * 1.0, (1 + 3 * 2 ** -11) * 1.0, 1e-45], np.float32),
    ]
    # exact ties at the fp16 spacing, both parities
    k = np.arange(1024, 2048, dtype=np.float32)
    parts.append((k + np.float32(0.5)) * np.float32(2.0 ** -10))
    x = np.concatenate(parts).astype(np.float32)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    got = O.f32_to_f16(x)
    assert np.array_equal(got, want)
    nan = O.f32_to_f16(np.array([np.nan], np.float32))[0]
    assert (nan & 0x7C00) == 0x7C00 and (nan & 0x3FF) != 0


def test_f16_to_f32_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = bits.view(np.float16).astype(np.float32)
    got = O.f16_to_f32(bits)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


# ---------------------------------------------------------------- Q4_K / Q8_0 layouts

# 12 packed scale bytes worked out by hand from the Q4_K layout: bytes 0-3 hold
# the scales of sub-blocks 0-3 in their low six bits (1, 2, 3, 4) and the top
# two bits of the scales of sub-blocks 4-7 (3, 2, 1, 0); bytes 4-7 the mins of
# sub-blocks 0-3 (5, 6, 7, 8) and the top bits of the mins 4-7 (0, 1, 2, 3);
# bytes 8-11 the low nibbles of scale (low half) and min (high half) 4-7.
SCALES12 = np.array([0b11000001, 0b10000010, 0b01000011, 0b00000100,
                     0b00000101, 0b01000110, 0b10000111, 0b11001000,
                     0x9A, 0xBC, 0xDE, 0xF0], np.uint8)
SC_M = [(1, 5), (2, 6), (3, 7), (4, 8),
        (0xA | 3 << 4, 0x9 | 0 << 4), (0xC | 2 << 4, 0xB | 1 << 4),
        (0xE | 1 << 4, 0xD | 2 << 4), (0x0 | 0 << 4, 0xF | 3 << 4)]


def test_q4k_scale_min_hand_values():
    assert SC_M[4:] == [(58, 9), (44, 27), (30, 45), (0, 63)]
    for j in range(8):
        assert O.q4k_scale_min(SCALES12, j) == SC_M[j], j


def _q4k_block():
    b = np.zeros(144, np.uint8)
    b[0:2] = np.array([0x00, 0x38], np.uint8)   # d = 0.5
    b[2:4] = np.array([0x00, 0x34], np.uint8)   # dmin = 0.25
    b[4:16] = SCALES12
    qs = b[16:]
    qs[0] = 0x73    # weight 0 (sub-block 0): 3; weight 32 (sub-block 1): 7
    qs[33] = 0x2F   # weight 65 (sub-block 2): 15; weight 97 (sub-block 3): 2
    qs[127] = 0x5A  # weight 223 (sub-block 6): 10; weight 255 (sub-block 7): 5
    return b


def test_q4k_dequant_hand_block():
    w = O.dequant_q(_q4k_block(), Q4_K, rows=1, K=256)[0]
    # w = d*sc_j*q - dmin*m_j, worked by hand
    assert w[0] == 0.5 * 1 * 3 - 0.25 * 5 == 0.25
    assert w[32] == 0.5 * 2 * 7 - 0.25 * 6 == 5.5
    assert w[65] == 0.5 * 3 * 15 - 0.25 * 7 == 20.75
    assert w[97] == 0.5 * 4 * 2 - 0.25 * 8 == 2.0
    assert w[223] == 0.5 * 30 * 10 - 0.25 * 45 == 138.75
    assert w[255] == 0.5 * 0 * 5 - 0.25 * 63 == -15.75
    # every other code is 0: the weight is -dmin * m_j of its sub-block
    for k in (1, 31, 33, 64, 96, 128, 200, 224, 254):
        assert w[k] == -0.25 * SC_M[k // 32][1], k


def test_q8_0_dequant_hand_block():
    b = np.zeros(34 * 2, np.uint8)
    b[0:2] = [0x00, 0x38]                 # d = 0.5
    b[2:6] = np.array([-128, -1, 0, 1], np.int8).view(np.uint8)
    b[33] = 127
    b[34:36] = [0x00, 0xC0]               # d = -2
    b[36] = 3
    w = O.dequant_q(b, Q8_0, rows=1, K=64)[0]
    assert list(w[:4]) == [-64.0, -0.5, 0.0, 0.5]
    assert w[31] == 63.5 and w[32] == -6.0
    assert np.all(w[4:31] == 0) and np.all(w[33:] == 0)


# ---------------------------------------------------------------- integer core


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
def test_keep_quant_dot_equals_dequantised_dot(fmt):
    """y = sum_k w[k] * (d_x * q_x[k]) computed from exact dequantised values."""
    f = FMT[fmt]
    blk = O.Q_BLOCK[f]
    G, N, K, P = 3, 5, 512, 9
    w = W.q_weights(3, 77, G, N, K, fmt, 0.02)
    rng = np.random.default_rng(8)
    aq = rng.integers(-127, 128, size=(P, K), dtype=np.int8)
    ad = (rng.uniform(0.5, 2.0, size=(P, K // blk)) * 1e-2).astype(np.float32)
    off = np.array([0, 4, 4, 9], np.int32)            # an empty middle group
    y, ya = O.gemm_q(aq, ad, w, f, off, P=P, K=K, N=N, G=G)
    wv = O.dequant_q(w, f, rows=G * N, K=K).reshape(G, N, K)
    av = aq.astype(np.float64) * np.repeat(ad.astype(np.float64), blk, axis=1)
    for r in range(P):
        g = int(np.searchsorted(off, r, side="right") - 1)
        ref = wv[g] @ av[r]
        assert np.all(np.abs(y[r] - ref) <= 1e-12 * ya[r] + 1e-300), (fmt, r)
        assert np.all(ya[r] >= np.abs(y[r]) * (1 - 1e-12))


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
def test_keep_quant_gather_reads_row_over_div(fmt):
    f = FMT[fmt]
    blk = O.Q_BLOCK[f]
    T, Kk, K, N = 4, 2, 256, 3
    P = T * Kk
    w = W.q_weights(4, 78, 2, N, K, fmt, 0.02)
    rng = np.random.default_rng(9)
    aq = rng.integers(-127, 128, size=(T, K), dtype=np.int8)
    ad = rng.uniform(0.01, 0.02, size=(T, K // blk)).astype(np.float32)
    sp = rng.permutation(P).astype(np.int32)
    off = np.array([0, 5, P], np.int32)
    y, _ = O.gemm_q(aq, ad, w, f, off, P=P, K=K, N=N, G=2, a_row_gather=sp, gather_div=Kk)
    y2, _ = O.gemm_q(np.ascontiguousarray(aq[sp // Kk]), np.ascontiguousarray(ad[sp // Kk]), w, f,
                     off, P=P, K=K, N=N, G=2)
    assert np.array_equal(y, y2)


# ---------------------------------------------------------------- activation quantizer


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
def test_quantizer_integer_block_is_exact(fmt):
    f = FMT[fmt]
    blk = O.Q_BLOCK[f]
    rng = np.random.default_rng(1)
    v = rng.integers(-126, 127, size=blk).astype(np.float32)
    v[blk // 3] = 127.0                                  # amax 127: d = 1, id = 1
    q, d = O.quantize_act_q8(_bf16(v)[None], f, R=1, K=blk)
    assert d[0, 0] == 1.0
    assert np.array_equal(q[0].astype(np.float32), v)


def test_quantizer_ties_round_away_from_zero():
    v = np.zeros(32, np.float32)
    v[0] = 127.0
    v[1:9] = [2.5, -2.5, 0.5, -0.5, 1.5, -1.5, 126.5, -126.5]
    q, d = O.quantize_act_q8(_bf16(v)[None], Q8_0, R=1, K=32)
    assert d[0, 0] == 1.0
    assert list(q[0, 1:9]) == [3, -3, 1, -1, 2, -2, 127, -127]


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
def test_quantizer_zero_and_nonfinite_blocks(fmt):
    f = FMT[fmt]
    blk = O.Q_BLOCK[f]
    x = np.zeros((3, blk), np.float32)
    x[1, 0], x[1, 1], x[1, 2] = np.inf, 1.0, -3.0
    x[2, 0], x[2, 1] = np.nan, 0.5
    x[2, 2] = -127.0 * 0.5
    q, d = O.quantize_act_q8(_bf16(x), f, R=3, K=blk)
    assert d[0, 0] == 0.0 and not q[0].any()             # all-zero block
    assert np.isinf(d[1, 0]) and not q[1].any()           # Inf: id = 0, every code 0
    assert d[2, 0] == 0.5                                 # amax 63.5: d = 0.5 exactly
    assert q[2, 0] == 0 and q[2, 1] == 1 and q[2, 2] == -127  # NaN -> 0, ignored by amax


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
def test_quantizer_error_bound_and_scales(fmt):
    f = FMT[fmt]
    blk = O.Q_BLOCK[f]
    R, K = 5, 1024
    rng = np.random.default_rng(2)
    x = rng.standard_normal((R, K)).astype(np.float32)
    x *= np.repeat(rng.uniform(0.01, 100.0, size=(R, K // blk)).astype(np.float32), blk, axis=1)
    xb = _bf16(x)
    xv = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    q, d = O.quantize_act_q8(xb, f, R=R, K=K)
    amax = np.abs(xv).reshape(R, K // blk, blk).max(axis=2)
    d_exact = amax / 127.0
    if f == Q8_0:   # the Q8_0 block stores d rounded to fp16
        assert np.array_equal(d, (amax / 127.0).astype(np.float32).astype(np.float16)
                              .astype(np.float32))
    else:
        assert np.all(np.abs(d - d_exact) <= d_exact * 2.0 ** -23)
    err = np.abs(xv - np.repeat(d_exact, blk, axis=1) * q)
    assert np.all(err <= np.repeat(d_exact, blk, axis=1) * (0.5 + 1e-5))
    qb = np.abs(q.astype(np.int32)).reshape(R, K // blk, blk)
    assert np.all(qb.max(axis=2) == 127) and np.all(qb <= 127)


# ---------------------------------------------------------------- epilogues and the layer


def _groups(P, G, seed):
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.integers(0, P + 1, size=G - 1))
    return np.concatenate([[0], cuts, [P]]).astype(np.int32)


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
def test_gateup_q_is_the_bf16_epilogue_on_gemm_q(fmt):
    f = FMT[fmt]
    G, H, I, T, Kk = 3, 256, 48, 5, 2
    P = T * Kk
    w13 = W.q_weights(5, 79, G, 2 * I, H, fmt, 0.02)
    x = W.normal_bf16(5, 80, (T, H), 1.0)
    aq, ad = O.quantize_act_q8(x, f, R=T, K=H)
    sp = np.random.default_rng(3).permutation(P).astype(np.int32)
    off = _groups(P, G, 4)
    act = O.gateup_silu_q(aq, ad, w13, f, off, P=P, H=H, I=I, G=G, a_row_gather=sp,
                          gather_div=Kk)
    y, _ = O.gemm_q(aq, ad, w13, f, off, P=P, K=H, N=2 * I, G=G, a_row_gather=sp, gather_div=Kk)
    g = O.f32_to_bf16(y[:, :I].astype(np.float32))
    u = O.f32_to_bf16(y[:, I:].astype(np.float32))
    gf = O.bf16_to_f32(g).astype(np.float32)
    uf = O.bf16_to_f32(u).astype(np.float32)
    ref = O.f32_to_bf16((gf / (np.float32(1) + np.exp(-gf))) * uf)
    diff = np.abs(act.astype(np.int32) - ref.astype(np.int32))
    assert diff.max() <= 1        # numpy's exp against the C library's: one bf16 step at most
    assert (diff == 0).mean() > 0.99


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
def test_down_q_is_weight_and_scatter_on_gemm_q(fmt):
    f = FMT[fmt]
    blk = O.Q_BLOCK[f]
    G, I, H, P = 2, 512, 40, 7
    w2 = W.q_weights(6, 81, G, H, I, fmt, 0.02)
    act = W.normal_bf16(6, 82, (P, I), 0.5)
    aq, ad = O.quantize_act_q8(act, f, R=P, K=I)
    assert ad.shape == (P, I // blk)
    off = np.array([0, 3, P], np.int32)
    r2p = np.random.default_rng(5).permutation(P).astype(np.int32)
    pw = np.random.default_rng(6).uniform(0.1, 1.0, size=P).astype(np.float32)
    out = O.down_q(aq, ad, w2, f, off, P=P, I=I, H=H, G=G, pair_weight=pw, row_to_pair=r2p)
    y, _ = O.gemm_q(aq, ad, w2, f, off, P=P, K=I, N=H, G=G)
    want = np.zeros_like(out)
    want[r2p] = O.f32_to_bf16(y.astype(np.float32) * pw[r2p][:, None])
    assert np.array_equal(out, want)


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
def test_layer_q_token_by_token_equals_batch_pieces(fmt):
    f = FMT[fmt]
    cfg = W.LayerConfig("q_tiny", T=6, H=256, I=256, E=4, K=2, I_shared=32, seed=3)
    d = W.layer_inputs(cfg)
    q = W.layer_q_weights(cfg, fmt)
    T, H, I, E, K = cfg.T, cfg.H, cfg.I, cfg.E, cfg.K
    out, ids, wts = O.moe_layer_tokens_q(d["x"], d["w_router"], d["logit_bias"], q["w13q"],
                                         q["w2q"], f, d["w_shared_gate"], d["w13_shared"],
                                         d["w2_shared"], H=H, I=I, E=E, K=K, I_shared=32,
                                         tokens=np.arange(T))
    # the same layer from the batch pieces
    r_ids, r_w, _, gl = O.route_topk(d["x"], d["w_router"], d["logit_bias"],
                                     d["w_shared_gate"], T=T, H=H, E=E, K=K)
    assert np.array_equal(r_ids, ids) and np.array_equal(r_w, wts)
    off, sp, _, _ = O.permute(r_ids, T=T, K=K, E=E)
    xq, xd = O.quantize_act_q8(d["x"], f, R=T, K=H)
    P = T * K
    act = O.gateup_silu_q(xq, xd, q["w13q"], f, off, P=P, H=H, I=I, G=E, a_row_gather=sp,
                          gather_div=K)
    aq, ad = O.quantize_act_q8(act, f, R=P, K=I)
    eo = O.down_q(aq, ad, q["w2q"], f, off, P=P, I=I, H=H, G=E, pair_weight=r_w.ravel(),
                  row_to_pair=sp)
    acts = O.gateup_silu(d["x"], d["w13_shared"], None, P=T, H=H, I=32, G=1)
    sd = O.down(acts, d["w2_shared"], None, P=T, I=32, H=H, G=1)
    ref = O.combine_gate(eo.reshape(T, K, H), None, sd, gl, T=T, K=K, H=H)
    assert np.array_equal(out, ref)


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
def test_dequant_bf16_is_the_exact_value_rounded(fmt):
    # Q8_0 and Q4_K values are formed exactly in f32 except for Q4_K's one
    # subtraction; the bf16 result must equal the round-to-nearest-even of the
    # exact value whenever that subtraction is exact, and be within one bf16
    # step of it always
    f = FMT[fmt]
    w = W.q_weights(9, 83, 1, 6, 1024, fmt, 0.02)
    exact = O.dequant_q(w, f, rows=6, K=1024)
    got = O.dequant_q_bf16(w, f, rows=6, K=1024)
    ref = O.f32_to_bf16(exact.astype(np.float32))      # exact -> f32 is exact here or one rounding
    if fmt == "q8_0":
        assert np.array_equal(got, ref)
    else:
        g = (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        step = np.abs(exact) * 2.0 ** -7 + 1e-30
        assert np.all(np.abs(g - exact) <= step)
        assert (got == ref).mean() > 0.999
    hand = O.dequant_q_bf16(_q4k_block(), Q4_K, rows=1, K=256)[0]
    hv = (hand.astype(np.uint32) << 16).view(np.float32)
    assert hv[0] == 0.25 and hv[32] == 5.5 and hv[255] == -15.75
    assert hv[223] == 139.0      # 138.75 rounds to 139: bf16 spacing is 1 in [128, 256)
