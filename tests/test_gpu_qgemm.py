"""GPU parity of the keep-quant expert GEMMs and the activation quantizer.

kMatmulBTQuant / kMatmulBTQuantGrouped of vllm.cpp PR #523 ("What changed"):
GGUF Q8_0 / Q4_K weight blocks, 8-bit activation blocks, exact integer block
sums.  The quantizer is bit-exact against the oracle.  The plain grouped op
(f32 out) is held to a rounding bound derived from its arithmetic: every block
sum is an exact integer, so the only error is f32 rounding of the block terms
and of their sum, at most 2^-18 times the sum of the terms' magnitudes (the
bound allows for 64 roundings of 2^-24 each; a wrong block, scale or index
errs by the size of the terms themselves).  The gate/up and down ops hold the
grouped-GEMM tolerance of the bf16 path (NMSE <= 1e-5, max relative error
<= 2e-2; the pages' own check is NMSE <= 5e-4).  The oracle consumes the
oracle's own quantized activations, never the GPU's."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mixture_experts_ffn_renorm_gb300 as m
import oracle as O
from mixture_experts_ffn_renorm_gb300 import workloads as W

from .gpu_util import assert_gemm_close, empty, launched_since, launches, to_dev, to_host

pytestmark = pytest.mark.gpu

FMTS = {"q8_0": (m.QFMT_Q8_0, O.Q8_0), "q4_k": (m.QFMT_Q4_K, O.Q4_K)}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    m.lib()
    m.moe_device_status(clear=True)
    yield
    assert m.moe_device_status() == 0


def _quant_dev(x_bits, fmt, R, K):
    gf, _ = FMTS[fmt]
    blk = O.Q_BLOCK[FMTS[fmt][1]]
    q = empty((max(R, 1), K), torch.int8)
    d = empty((max(R, 1), K // blk), torch.float32)
    m.moe_quantize_act_q8(to_dev(x_bits), R, K, gf, q, d)
    torch.cuda.synchronize()
    return q, d


# ---------------------------------------------------------------- quantizer


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
@pytest.mark.parametrize("R,K", [(1, 256), (7, 768), (300, 2048), (3, 4096)])
def test_quantizer_bit_exact(fmt, R, K):
    rng = np.random.default_rng(R * 7 + K)
    x = rng.standard_normal((R, K)).astype(np.float32)
    x *= np.exp(rng.uniform(-12, 12, size=(R, K // 32))).astype(np.float32).repeat(32, axis=1)
    x[0, :32] = 0.0                                    # an all-zero sub-block
    if K >= 512:
        x[0, 256:264] = [2.5, -2.5, 0.5, -0.5, 127.0, 126.5, -126.5, 1.5]  # ties
    xb = W.to_bf16_bits(x)
    if R > 1:
        xb[1, 5] = 0x7F80                              # +Inf
        xb[1, 40] = 0x7FC0                             # NaN
        xb[1, 300 % K] = 0x0001                        # bf16 subnormal
    q, d = _quant_dev(xb, fmt, R, K)
    q_ref, d_ref = O.quantize_act_q8(xb, FMTS[fmt][1], R=R, K=K)
    assert np.array_equal(to_host(q), q_ref)
    dh = to_host(d)
    assert np.array_equal(np.isnan(dh), np.isnan(d_ref))
    assert np.array_equal(dh.view(np.uint32)[~np.isnan(dh)], d_ref.view(np.uint32)[~np.isnan(d_ref)])


# ---------------------------------------------------------------- plain grouped op


def _mag_bound(w, fmt_o, aq, ad, rows_src, gidx, N, K):
    """sum_k |d_x a_k| (|positive part of w_k| + |min part of w_k|) per (row, col)."""
    blk = O.Q_BLOCK[fmt_o]
    G = w.shape[0]
    wp = w.copy()
    wm = w.copy()
    if fmt_o == O.Q4_K:
        bb = wp.reshape(-1, 144)
        bb[:, 2:4] = 0                                  # dmin = 0: d*sc*q
        bm = wm.reshape(-1, 144)
        bm[:, 0:2] = 0                                  # d = 0: -dmin*m
    A = np.abs(O.dequant_q(wp, fmt_o, rows=G * N, K=K)).reshape(G, N, K)
    B = (np.abs(O.dequant_q(wm, fmt_o, rows=G * N, K=K)).reshape(G, N, K)
         if fmt_o == O.Q4_K else 0.0)
    av = np.abs(aq[rows_src].astype(np.float64) * np.repeat(ad[rows_src].astype(np.float64), blk,
                                                              axis=1))
    out = np.zeros((len(rows_src), N))
    for i in range(len(rows_src)):
        out[i] = (A[gidx[i]] + (B[gidx[i]] if fmt_o == O.Q4_K else 0.0)) @ av[i]
    return out


PLAIN_CASES = [
    # group sizes, K, N
    ([4], 256, 64),
    ([3, 0, 9, 1, 17], 512, 70),
    ([8, 8, 16, 7], 2048, 33),
    ([1, 1, 1, 1, 1, 1], 4096, 5),
    ([130, 2], 768, 1),
    ([2, 1], 16384, 3),          # the longest rows: many K chunks, the largest shared-memory carve-up
]


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
@pytest.mark.parametrize("case", range(len(PLAIN_CASES)))
def test_plain_grouped_q_within_rounding_bound(fmt, case):
    sizes, K, N = PLAIN_CASES[case]
    gf, fo = FMTS[fmt]
    G = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    P = int(off[-1])
    w = W.q_weights(11 + case, 90, G, N, K, fmt, 0.02)
    x = W.normal_bf16(12 + case, 91, (P, K), 1.0)
    aq, ad = O.quantize_act_q8(x, fo, R=P, K=K)
    y_ref, _ = O.gemm_q(aq, ad, w, fo, off, P=P, K=K, N=N, G=G)
    out = torch.full((P, N), float("nan"), device="cuda:0")
    before = launches()
    m.moe_grouped_gemm_q(to_dev(aq), to_dev(ad), P, None, 1, to_dev(w), gf,
                         to_dev(off) if G > 1 else None, P, K, N, G, out)
    assert launched_since(before, "gemm_q") == 1
    got = to_host(out).astype(np.float64)
    gidx = np.searchsorted(off, np.arange(P), side="right") - 1
    bound = _mag_bound(w, fo, aq, ad, np.arange(P), gidx, N, K)
    err = np.abs(got - y_ref)
    assert np.all(err <= 2.0 ** -18 * bound + 1e-30), f"max err/bound {np.max(err / (bound + 1e-30)):.3e}"


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
def test_plain_grouped_q_gather_and_out_of_range(fmt):
    gf, fo = FMTS[fmt]
    T, Kk, K, N = 5, 3, 512, 40
    P = T * Kk
    off = np.array([0, 4, 4, 11, P], np.int32)
    G = 4
    w = W.q_weights(21, 92, G, N, K, fmt, 0.02)
    x = W.normal_bf16(22, 93, (T, K), 1.0)
    aq, ad = O.quantize_act_q8(x, fo, R=T, K=K)
    sp = np.random.default_rng(3).permutation(P).astype(np.int32)
    y_ref, _ = O.gemm_q(aq, ad, w, fo, off, P=P, K=K, N=N, G=G, a_row_gather=sp, gather_div=Kk)
    bad = sp.copy()
    bad[2] = -3                          # rows outside [0, a_rows) read zeros
    bad[9] = T * Kk + 7
    out = empty((P, N), torch.float32)
    m.moe_grouped_gemm_q(to_dev(aq), to_dev(ad), T, to_dev(bad), Kk, to_dev(w), gf, to_dev(off),
                         P, K, N, G, out)
    got = to_host(out).astype(np.float64)
    assert np.all(got[2] == 0) and np.all(got[9] == 0)
    keep = np.setdiff1d(np.arange(P), [2, 9])
    assert np.allclose(got[keep], y_ref[keep], rtol=1e-4, atol=1e-3 * np.abs(y_ref).max())


# ---------------------------------------------------------------- gate/up and down


GU_CASES = [
    # group sizes, H, I
    ([2, 0, 5], 256, 32),
    ([9, 1, 17, 8], 768, 96),
    ([1] * 12, 2048, 768),
]


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
@pytest.mark.parametrize("case", range(len(GU_CASES)))
def test_gateup_q_matches_oracle(fmt, case):
    sizes, H, I = GU_CASES[case]
    gf, fo = FMTS[fmt]
    G = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    P = int(off[-1])
    Kk = 2
    T = (P + Kk - 1) // Kk
    w13 = W.q_weights(31 + case, 94, G, 2 * I, H, fmt, 0.02)
    x = W.normal_bf16(32 + case, 95, (T, H), 1.0)
    sp = np.random.default_rng(case).permutation(T * Kk)[:P].astype(np.int32)
    aq, ad = O.quantize_act_q8(x, fo, R=T, K=H)
    ref = O.gateup_silu_q(aq, ad, w13, fo, off, P=P, H=H, I=I, G=G, a_row_gather=sp,
                          gather_div=Kk)
    act = empty((P, I), torch.bfloat16)
    before = launches()
    m.moe_grouped_gemm_gateup_silu_q(to_dev(aq), to_dev(ad), T, to_dev(sp), Kk, to_dev(w13), gf,
                                     to_dev(off), P, H, I, G, act)
    assert launched_since(before, "gemm_q_gateup") == 1
    assert_gemm_close(to_host(act), ref, f"gateup {fmt} case {case}")


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
@pytest.mark.parametrize("case", range(len(GU_CASES)))
def test_down_q_matches_oracle(fmt, case):
    sizes, H, I = GU_CASES[case]
    I, H = H, max(64, I)                      # contraction over I (a multiple of 256)
    gf, fo = FMTS[fmt]
    G = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    P = int(off[-1])
    w2 = W.q_weights(41 + case, 96, G, H, I, fmt, 0.02)
    act = W.normal_bf16(42 + case, 97, (P, I), 0.3)
    aq, ad = O.quantize_act_q8(act, fo, R=P, K=I)
    r2p = np.random.default_rng(case + 5).permutation(P).astype(np.int32)
    pw = np.random.default_rng(case + 6).uniform(0.05, 1.0, size=P).astype(np.float32)
    ref = O.down_q(aq, ad, w2, fo, off, P=P, I=I, H=H, G=G, pair_weight=pw, row_to_pair=r2p)
    out = empty((P, H), torch.bfloat16)
    before = launches()
    m.moe_grouped_gemm_down_q(to_dev(aq), to_dev(ad), to_dev(w2), gf, to_dev(off), to_dev(pw),
                              to_dev(r2p), P, I, H, G, out)
    assert launched_since(before, "gemm_q_down") == 1
    assert_gemm_close(to_host(out), ref, f"down {fmt} case {case}")


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
def test_down_q_rows_outside_groups_untouched(fmt):
    gf, fo = FMTS[fmt]
    P, I, H, G = 12, 256, 64, 2
    off = np.array([2, 5, 9], np.int32)        # rows 0-1 and 9-11 belong to no group
    w2 = W.q_weights(51, 98, G, H, I, fmt, 0.02)
    act = W.normal_bf16(52, 99, (P, I), 0.3)
    aq, ad = O.quantize_act_q8(act, fo, R=P, K=I)
    ref = O.down_q(aq, ad, w2, fo, off, P=P, I=I, H=H, G=G)
    out = torch.full((P, H), 7.0, dtype=torch.bfloat16, device="cuda:0")
    m.moe_grouped_gemm_down_q(to_dev(aq), to_dev(ad), to_dev(w2), gf, to_dev(off), None, None, P,
                              I, H, G, out)
    got = to_host(out)
    seven = to_host(torch.full((1,), 7.0, dtype=torch.bfloat16))[0]
    assert np.all(got[[0, 1, 9, 10, 11]] == seven)
    assert_gemm_close(got[2:9], ref[2:9], f"down {fmt} inner rows")


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
def test_decode_size_gemms_match_oracle(fmt):
    """The decode layer's shapes (T=16, K=8, E=128, H=2048, I=768) on its own routing."""
    gf, fo = FMTS[fmt]
    cfg = W.DECODE
    T, H, I, E, K = cfg.T, cfg.H, cfg.I, cfg.E, cfg.K
    d = W.layer_inputs(cfg, with_weights=False)
    q = W.layer_q_weights(cfg, fmt)
    ids, wts, _, _ = O.route_topk(d["x"], d["w_router"], d["logit_bias"], T=T, H=H, E=E, K=K)
    off, sp, _, _ = O.permute(ids, T=T, K=K, E=E)
    P = T * K
    xq, xd = O.quantize_act_q8(d["x"], fo, R=T, K=H)
    act_ref = O.gateup_silu_q(xq, xd, q["w13q"], fo, off, P=P, H=H, I=I, G=E, a_row_gather=sp,
                              gather_div=K)
    act = empty((P, I), torch.bfloat16)
    w13 = to_dev(q["w13q"])
    m.moe_grouped_gemm_gateup_silu_q(to_dev(xq), to_dev(xd), T, to_dev(sp), K, w13, gf,
                                     to_dev(off), P, H, I, E, act)
    assert_gemm_close(to_host(act), act_ref, f"decode gateup {fmt}")
    aq, ad = O.quantize_act_q8(act_ref, fo, R=P, K=I)
    eo_ref = O.down_q(aq, ad, q["w2q"], fo, off, P=P, I=I, H=H, G=E, pair_weight=wts.ravel(),
                      row_to_pair=sp)
    eo = empty((P, H), torch.bfloat16)
    m.moe_grouped_gemm_down_q(to_dev(aq), to_dev(ad), to_dev(q["w2q"]), gf, to_dev(off),
                              to_dev(wts.ravel()), to_dev(sp), P, I, H, E, eo)
    assert_gemm_close(to_host(eo), eo_ref, f"decode down {fmt}")


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k"])
@pytest.mark.parametrize("rows,K", [(1, 256), (37, 768), (300, 2048)])
def test_dequantize_to_bf16_bit_exact(fmt, rows, K):
    gf, fo = FMTS[fmt]
    w = W.q_weights(rows + K, 84, 1, rows, K, fmt, 0.02).reshape(rows, -1)
    ref = O.dequant_q_bf16(w, fo, rows=rows, K=K)
    out = empty((rows, K), torch.bfloat16)
    before = launches()
    m.moe_dequantize_q_bf16(to_dev(w), gf, rows, K, out)
    assert launched_since(before, "dequant_q") == 1
    assert np.array_equal(to_host(out), ref)
