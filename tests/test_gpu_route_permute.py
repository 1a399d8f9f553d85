"""GPU parity of moe_route_topk and moe_permute against the CPU oracle.

Router (vllm.cpp PR #509 "Honest gaps": ungrouped softmax only): given the
same f32 logits, ids and weights are bit-exact; the tensor-core logits are
checked against the dot-product error bound.  Permute: bit-exact."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mixture_experts_ffn_renorm_gb300 as m
import oracle as O
from mixture_experts_ffn_renorm_gb300 import workloads as W

from .gpu_util import bf16_to_f64, empty, launched_since, launches, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    m.lib()
    m.moe_device_status(clear=True)
    yield
    assert m.moe_device_status() == 0


def gpu_route(x, wr, bias, wsg, logits_in, T, H, E, K, renorm=1, want_logits=False):
    ids = empty((T, K), torch.int32)
    w = empty((T, K), torch.float32)
    lo = empty((T, E), torch.float32) if want_logits else None
    gl = empty((T,), torch.float32) if wsg is not None else None
    wsz = m.moe_route_topk_workspace_size(T, E, K)
    ws = empty((max(wsz, 16),), torch.uint8)
    m.moe_route_topk(None if x is None else to_dev(x), None if wr is None else to_dev(wr),
                     None if bias is None else to_dev(bias), None if wsg is None else to_dev(wsg),
                     None if logits_in is None else to_dev(logits_in), T, H, E, K, renorm, 0, 1,
                     ids, w, lo, gl, ws, wsz)
    return (to_host(ids), to_host(w), None if lo is None else to_host(lo),
            None if gl is None else to_host(gl))


@pytest.mark.parametrize("E,K", [(8, 2), (128, 8), (256, 8), (1000, 32), (5, 5), (64, 1),
                                 (96, 8), (200, 6)])
@pytest.mark.parametrize("renorm", [1, 0])
def test_topk_bit_exact_from_logits(E, K, renorm):
    rng = np.random.default_rng(E * 7 + K)
    T = 301
    logits = rng.standard_normal((T, E)).astype(np.float32)
    # ties, signed zeros, NaN and infinities in a few rows
    logits[0, :] = 0.5
    logits[1, ::2] = -0.0
    logits[1, 1::2] = 0.0
    logits[2, 0] = np.nan
    logits[3, E - 1] = np.inf
    logits[4, : E // 2] = -np.inf
    logits[5, :] = np.nan                     # every key equal: the K lowest ids
    logits[6, ::3] = np.nan
    logits[7, :] = logits[7, 0]               # one value repeated: ties all the way down
    logits[7, E - 1] = np.inf
    want_ids, want_w, _, _ = O.route_topk(logits_in=logits, T=T, H=1, E=E, K=K,
                                          renormalize=renorm)
    before = launches()
    ids, w, _, _ = gpu_route(None, None, None, None, logits, T, 8, E, K, renorm)
    assert launched_since(before, "route_topk") == 1
    assert np.array_equal(ids, want_ids)
    ok = ~np.isnan(want_w)
    assert np.array_equal(np.isnan(w), ~ok)
    assert np.array_equal(w[ok].view(np.uint32), want_w[ok].view(np.uint32))


@pytest.mark.parametrize("T,H,E,K", [(4, 64, 8, 2), (300, 256, 128, 8), (131, 512, 256, 8),
                                     (16, 2048, 128, 8), (2, 72, 40, 3)])
def test_router_gemm_logits_within_bound_and_selection_exact(T, H, E, K):
    rng = np.random.default_rng(T + H + E)
    x = W.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    wr = W.to_bf16_bits((0.02 * rng.standard_normal((E, H))).astype(np.float32))
    bias = (0.5 * rng.standard_normal(E)).astype(np.float32)
    wsg = W.to_bf16_bits((0.02 * rng.standard_normal(H)).astype(np.float32))
    before = launches()
    ids, w, lo, gl = gpu_route(x, wr, bias, wsg, None, T, H, E, K, want_logits=True)
    assert launched_since(before, "route_logits") == 1
    xf, wf = bf16_to_f64(x), bf16_to_f64(wr)
    exact = xf @ wf.T + bias
    # tensor-core f32 accumulation: allow 2^-23 per addition (truncating adders)
    bound = (H + 2) * 2.0**-23 * (np.abs(xf) @ np.abs(wf).T + np.abs(bias))
    assert np.all(np.abs(lo - exact) <= bound), float(np.max(np.abs(lo - exact) / bound))
    # selection and weights are bit-exact functions of the GPU's logits
    want_ids, want_w, _, _ = O.route_topk(logits_in=lo, T=T, H=1, E=E, K=K)
    assert np.array_equal(ids, want_ids)
    assert np.array_equal(w.view(np.uint32), want_w.view(np.uint32))
    gl_exact = xf @ bf16_to_f64(wsg)
    gl_bound = (H + 2) * 2.0**-23 * (np.abs(xf) @ np.abs(bf16_to_f64(wsg)))
    assert np.all(np.abs(gl - gl_exact) <= gl_bound)
    # without logits_out the logits go to the workspace and the ids are the same
    ids2, w2, _, _ = gpu_route(x, wr, bias, None, None, T, H, E, K)
    assert np.array_equal(ids2, ids) and np.array_equal(w2, w)


# batches above 64 tokens (smaller ones take the CUDA-core logits kernel) that
# make few tiles: the K split takes 16, 16, 2, 4, 16 and 5 ranges
@pytest.mark.parametrize("T,H,E", [(65, 2048, 128), (100, 4096, 256), (2048, 4096, 256),
                                   (96, 200, 96), (128, 1024, 32), (70, 320, 20)])
def test_router_k_split_matches_unsplit_within_bound(T, H, E):
    # with a workspace the logits GEMM splits K into ranges whose partial sums
    # the selection adds in range order (then the bias); without one it runs
    # whole.  Both logits are within the dot-product bound, and each side's ids
    # and weights are the exact functions of its own logits.
    K = 8
    rng = np.random.default_rng(T * 3 + H + E)
    x = W.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    wr = W.to_bf16_bits((0.02 * rng.standard_normal((E, H))).astype(np.float32))
    bias = (0.5 * rng.standard_normal(E)).astype(np.float32)
    xf, wf = bf16_to_f64(x), bf16_to_f64(wr)
    exact = xf @ wf.T + bias
    bound = (H + 2) * 2.0**-23 * (np.abs(xf) @ np.abs(wf).T + np.abs(bias))
    wsz = m.moe_route_topk_workspace_size(T, E, K)
    res = []
    for ws in (empty((max(wsz, 16),), torch.uint8), None):
        ids = empty((T, K), torch.int32)
        w = empty((T, K), torch.float32)
        lo = empty((T, E), torch.float32)
        m.moe_route_topk(to_dev(x), to_dev(wr), to_dev(bias), None, None, T, H, E, K, 1, 0, 1,
                         ids, w, lo, None, ws, 0 if ws is None else ws.numel())
        lo_h, ids_h, w_h = to_host(lo), to_host(ids), to_host(w)
        assert np.all(np.abs(lo_h - exact) <= bound), float(np.max(np.abs(lo_h - exact) / bound))
        want_ids, want_w, _, _ = O.route_topk(logits_in=lo_h, T=T, H=1, E=E, K=K)
        assert np.array_equal(ids_h, want_ids)
        assert np.array_equal(w_h.view(np.uint32), want_w.view(np.uint32))
        res.append(ids_h)
    # the two orders round differently; the chosen sets agree except on near-ties
    same = np.all(np.sort(res[0], 1) == np.sort(res[1], 1), axis=1)
    assert same.mean() >= 0.95


@pytest.mark.parametrize("T", [1, 5, 16, 33, 64])
@pytest.mark.parametrize("H,E,K", [(2048, 128, 8), (4096, 256, 8), (72, 40, 3), (2048, 1000, 32),
                                   (64, 8, 2), (200, 300, 6)])
@pytest.mark.parametrize("renorm", [1, 0])
def test_router_small_batch_logits_within_bound_and_selection_exact(T, H, E, K, renorm):
    # up to 64 tokens: one CUDA-core kernel forms the finished logits (fused
    # multiply-adds per lane in index order, a butterfly over the warp, then the
    # bias), with or without a workspace; the selection reads them once
    rng = np.random.default_rng(7 * T + H + E)
    x = W.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    wr = W.to_bf16_bits((0.02 * rng.standard_normal((E, H))).astype(np.float32))
    bias = (0.5 * rng.standard_normal(E)).astype(np.float32)
    xf, wf = bf16_to_f64(x), bf16_to_f64(wr)
    exact = xf @ wf.T + bias
    bound = (H + 2) * 2.0**-24 * (np.abs(xf) @ np.abs(wf).T + np.abs(bias))
    before = launches()
    ids, w, lo, _ = gpu_route(x, wr, bias, None, None, T, H, E, K, renorm, want_logits=True)
    assert launched_since(before, "route_logits") == 1
    assert np.all(np.abs(lo - exact) <= bound), float(np.max(np.abs(lo - exact) / bound))
    want_ids, want_w, _, _ = O.route_topk(logits_in=lo, T=T, H=1, E=E, K=K, renormalize=renorm)
    assert np.array_equal(ids, want_ids)
    assert np.array_equal(w.view(np.uint32), want_w.view(np.uint32))
    ids2, w2, _, _ = gpu_route(x, wr, bias, None, None, T, H, E, K, renorm)
    assert np.array_equal(ids2, ids) and np.array_equal(w2.view(np.uint32), w.view(np.uint32))


EX_CASES = [
    # E, K, scoring, n_group, topk_group, group_score, select bias
    (256, 8, 1, 8, 4, 1, True),      # DeepSeek-V3 shape
    (160, 6, 0, 8, 3, 0, False),     # DeepSeek-V2 shape
    (64, 4, 1, 4, 2, 1, False),
    (128, 8, 1, 1, 1, 0, True),      # sigmoid + bias, no groups
    (1024, 8, 1, 64, 8, 1, True),    # widest rows and most groups
    (12, 3, 0, 6, 2, 1, False),      # two experts per group
]


@pytest.mark.parametrize("E,K,scoring,n_group,topk_group,gscore,with_bias", EX_CASES)
@pytest.mark.parametrize("renorm", [1, 0])
def test_router_ex_bit_exact_from_logits(E, K, scoring, n_group, topk_group, gscore, with_bias,
                                         renorm):
    rng = np.random.default_rng(E + 13 * K + n_group)
    T = 133
    l = rng.standard_normal((T, E)).astype(np.float32)
    l[0, : E // 2] = l[0, E // 2:]      # ties between groups and between experts
    l[1, :] = 0.0
    l[2, 3] = np.nan
    bias = (0.1 * rng.standard_normal(E)).astype(np.float32) if with_bias else None
    want_ids, want_w = O.route_topk_ex(l, bias, T=T, E=E, K=K, renormalize=renorm,
                                       scoring=scoring, n_group=n_group, topk_group=topk_group,
                                       group_score=gscore)
    ids = empty((T, K), torch.int32)
    w = empty((T, K), torch.float32)
    before = launches()
    m.moe_route_topk_ex(None, None, None, None if bias is None else to_dev(bias), None, to_dev(l),
                        T, 8, E, K, renorm, scoring, n_group, topk_group, gscore, ids, w, None,
                        None, None, 0)
    assert launched_since(before, "route_topk") == 1
    assert np.array_equal(to_host(ids), want_ids)
    # a NaN logit makes a full-softmax row NaN (renormalize 0): positions must
    # agree; NaN payloads are not part of the contract
    got = to_host(w)
    ok = ~np.isnan(want_w)
    assert np.array_equal(np.isnan(got), ~ok)
    assert np.array_equal(got[ok].view(np.uint32), want_w[ok].view(np.uint32))


def test_router_ex_through_the_logits_gemm():
    # DeepSeek-V3-like routing of 16 and 300 tokens: logits from the CUDA-core
    # kernel (16 tokens) and from the tensor-core GEMM with its K split (300),
    # ids and weights exact given those logits
    E, K, H = 256, 8, 1024
    rng = np.random.default_rng(8)
    wr = W.to_bf16_bits((0.02 * rng.standard_normal((E, H))).astype(np.float32))
    bias = (0.05 * rng.standard_normal(E)).astype(np.float32)
    for T in (16, 300):
        x = W.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
        ids = empty((T, K), torch.int32)
        w = empty((T, K), torch.float32)
        lo = empty((T, E), torch.float32)
        wsz = m.moe_route_topk_workspace_size(T, E, K)
        ws = empty((max(wsz, 16),), torch.uint8)
        m.moe_route_topk_ex(to_dev(x), to_dev(wr), None, to_dev(bias), None, None, T, H, E, K, 1,
                            1, 8, 4, 1, ids, w, lo, None, ws, wsz)
        want_ids, want_w = O.route_topk_ex(to_host(lo), bias, T=T, E=E, K=K, scoring=1,
                                           n_group=8, topk_group=4, group_score=1)
        assert np.array_equal(to_host(ids), want_ids)
        assert np.array_equal(to_host(w).view(np.uint32), want_w.view(np.uint32))


def test_router_ex_refusals():
    T, E = 4, 16
    logits = to_dev(np.zeros((T, E), np.float32))
    ids = empty((T, 8), torch.int32)
    w = empty((T, 8), torch.float32)
    bias = to_dev(np.zeros(E, np.float32))
    before = launches()
    for args, code in (((2, 1, 1, 0, 2, None), m.ERR_UNSUPPORTED),     # scoring 2
                       ((0, 1, 1, 0, 2, bias), m.ERR_UNSUPPORTED),     # bias with softmax
                       ((1, 3, 1, 0, 2, None), m.ERR_ARG),             # 3 does not divide 16
                       ((1, 4, 5, 0, 2, None), m.ERR_ARG),             # topk_group > n_group
                       ((1, 16, 2, 1, 2, None), m.ERR_ARG),            # two-best of one expert
                       ((1, 8, 1, 0, 3, None), m.ERR_ARG)):            # K > eligible experts
        scoring, n_group, topk_group, gscore, k, b = args
        with pytest.raises(m.MoeError) as ei:
            m.moe_route_topk_ex(None, None, None, b, None, logits, T, 8, E, k, 1, scoring, n_group,
                                topk_group, gscore, ids, w, None, None, None, 0)
        assert ei.value.code == code
    assert launches() == before


def test_router_refusals():
    T, E, K = 4, 8, 2
    logits = np.zeros((T, E), np.float32)
    ids = empty((T, K), torch.int32)
    w = empty((T, K), torch.float32)
    for scoring, n_group, k, code in ((1, 1, K, m.ERR_UNSUPPORTED), (0, 2, K, m.ERR_UNSUPPORTED),
                                      (0, 1, 9, m.ERR_ARG), (0, 1, 0, m.ERR_ARG)):
        with pytest.raises(m.MoeError) as ei:
            m.moe_route_topk(None, None, None, None, to_dev(logits), T, 8, E, k, 1, scoring,
                             n_group, ids, w, None, None, None, 0)
        assert ei.value.code == code


def gpu_permute(ids, x, T, K, E, H):
    P = T * K
    off = empty((E + 1,), torch.int32)
    sp = empty((max(P, 1),), torch.int32)
    p2r = empty((max(P, 1),), torch.int32)
    xp = empty((max(P, 1), H), torch.bfloat16) if x is not None else None
    wsz = m.moe_permute_workspace_size(T, K, E)
    ws = empty((max(wsz, 16),), torch.uint8)
    m.moe_permute(to_dev(ids) if P else None, None if x is None else to_dev(x), T, K, E, H, off,
                  sp, p2r, xp, ws, wsz)
    return (to_host(off), to_host(sp)[:P], to_host(p2r)[:P],
            None if xp is None else to_host(xp)[:P])


def _ids(T, K, E, seed, skew=False):
    rng = np.random.default_rng(seed)
    if skew:
        p = 1.0 / np.arange(1, E + 1) ** 1.1
        p /= p.sum()
        return np.stack([rng.choice(E, K, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    return np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,K,E,H", [(4, 2, 8, 64), (16, 8, 128, 2048), (1000, 8, 128, 64),
                                     (2048, 8, 256, 128), (77, 3, 1000, 16), (1, 1, 1, 8),
                                     (8192, 8, 128, 8), (512, 8, 128, 64), (513, 8, 128, 64),
                                     (1365, 3, 1024, 8), (2048, 8, 256, 64), (2049, 8, 256, 8),
                                     (2048, 8, 512, 8),
                                     # the chunked scan: segments of several batches, one
                                     # thread per expert, an expert count not a power of two
                                     (65536, 8, 128, 8), (16384, 8, 1024, 8), (8192, 4, 300, 8)])
def test_permute_bit_exact(T, K, E, H):
    ids = _ids(T, K, E, T + E, skew=(T >= 1000))
    rng = np.random.default_rng(5)
    x = rng.integers(0, 65535, (T, H), dtype=np.uint16)
    want = O.permute(ids, x, T=T, K=K, E=E, H=H)
    before = launches()
    got = gpu_permute(ids, x, T, K, E, H)
    # up to 32 chunks of 512 pairs whose histograms fit in 48 KB: one block
    chunks = (T * K + 511) // 512
    small = chunks <= 32 and (chunks + 1) * E * 4 <= 48 * 1024
    assert launched_since(before, "permute_small") == (1 if small else 0)
    assert launched_since(before, "permute_place") == (0 if small else 1)
    for g, w_, name in zip(got, want, ("expert_offsets", "sorted_pair", "pair_to_row", "x_perm")):
        assert np.array_equal(g, w_), name


def test_permute_empty_batch_zeroes_offsets():
    off, _, _, _ = gpu_permute(np.zeros((0, 2), np.int32), None, 0, 2, 8, 8)
    assert np.array_equal(off, np.zeros(9, np.int32))


@pytest.mark.parametrize("T", [2, 3000, 30000])
def test_permute_flags_out_of_range_ids(T):
    # bad ids are flagged and skipped on the one-block and the chunked paths
    K, E = 2, 4
    ids = _ids(T, K, E, 11)
    ids[1, 1] = 9
    ids[T - 1, 0] = -1
    m.moe_device_status(clear=True)
    off, sp, p2r, _ = gpu_permute(ids, None, T, K, E, 8)
    assert m.moe_device_status(clear=True) & m.STATUS_BAD_ID
    counts = np.bincount(ids[(ids >= 0) & (ids < E)], minlength=E)
    assert np.array_equal(np.diff(off), counts) and off[E] == T * K - 2


def test_permute_workspace_needs_no_initialisation():
    # the workspace's histograms start as any bytes (here all 0xFF, then what
    # the previous call left): every call gives the same bits
    T, K, E, H = 8192, 8, 128, 8
    ids = _ids(T, K, E, 21, skew=True)
    want = O.permute(ids, None, T=T, K=K, E=E, H=H)
    P = T * K
    wsz = m.moe_permute_workspace_size(T, K, E)
    ws = torch.full((wsz,), 255, dtype=torch.uint8, device="cuda")
    d_ids = to_dev(ids)
    for _ in range(3):
        off = empty((E + 1,), torch.int32)
        sp, p2r = empty((P,), torch.int32), empty((P,), torch.int32)
        m.moe_permute(d_ids, None, T, K, E, H, off, sp, p2r, None, ws, wsz)
        for g, w_ in zip((off, sp, p2r), want[:3]):
            assert np.array_equal(to_host(g), w_)
    assert m.moe_device_status() == 0


@pytest.mark.slow
def test_permute_many_chunks():
    # 5.6 M pairs, 10938 chunks: more chunk blocks than the GPU holds at once,
    # and a scan of 10938 counts per expert in 32-chunk batches
    T, K, E = 700000, 8, 128
    rng = np.random.default_rng(3)
    ids = rng.integers(0, E, (T, K), dtype=np.int32)
    want = O.permute(ids, None, T=T, K=K, E=E, H=8)
    before = launches()
    got = gpu_permute(ids, None, T, K, E, 8)
    assert launched_since(before, "permute_scan") == 1 and launched_since(before, "permute_place") == 1
    for g, w_ in zip(got[:3], want[:3]):
        assert np.array_equal(g, w_)
