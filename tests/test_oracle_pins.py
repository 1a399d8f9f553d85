"""Pins of the CPU oracle to things other than itself.

Each test checks the oracle against what the pages or plain mathematics fix:
closed forms, exact constructions whose result is known by hand, invariants,
float64 / high-precision recomputation, library routines (a stable sort, a
float64 matmul, mpmath's exp) and brute force on tiny inputs.  They are chosen
so that a plausible slip in the oracle (a dropped rounding, a wrong index, a
transposed operand, a reordered sum, a fused multiply-add) fails one of them.

Passages the checks follow (vllm.cpp pages):
  * issue #3094 "Row: BACKEND-ROCM-BF16-MOE": the numeric contract -- BF16
    narrowing of gate and up ahead of the activation, routing weight applied to the down result
    is stored, reduction without applying the weights twice;
  * PR #509 "MoE combine/gate ops": out = sigmoid(gl) * sd, weighted top-k sum
    with optional shared term, the shared term rounded to bf16 first, sequential
    K order with one store rounding and no contraction (review rework item 2),
    routed_scale applied to the routed sum before the shared term;
  * PR #509 "Honest gaps": the covered router is ungrouped softmax.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle as O
from mixture_experts_ffn_renorm_gb300 import workloads as W

F32, BF16, F16 = O.F32, O.BF16, O.F16


# ------------------------------------------------------------------ helpers (independent)
def f64_to_nearest_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Nearest bf16 to each float64 value, ties to even, by brute force over the
    bf16 neighbours (no bit trick): the definition of RNE narrowing.  For the
    distance, infinity stands at 2^128, which is where RNE overflows to it."""
    v = np.asarray(v, np.float64).ravel()
    out = np.empty(v.size, np.uint16)
    for i, x in enumerate(v):
        if math.isnan(x):
            out[i] = 0x7FC0
            continue
        if math.isinf(x):
            out[i] = 0x7F80 if x > 0 else 0xFF80
            continue
        f = np.float32(np.clip(x, -3.4028234e38, 3.4028234e38))
        t = int(np.array([f], np.float32).view(np.uint32)[0]) >> 16
        best, bestd = None, None
        for c in (t - 1, t, t + 1):
            c &= 0xFFFF
            cv = float(np.array([c << 16], np.uint32).view(np.float32)[0])
            if math.isnan(cv):
                continue
            if math.isinf(cv):
                cv = math.copysign(2.0**128, cv)
            d = abs(cv - x)
            if bestd is None or d < bestd or (d == bestd and (c & 1) == 0):
                best, bestd = c, d
        out[i] = best
    return out


def bits_to_f32(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_bits(x):
    return np.asarray(x, np.float32).view(np.uint32)


# ------------------------------------------------------------------ bf16 narrowing
def test_bf16_rne_known_values():
    cases = {
        1.0: 0x3F80,
        1.0 + 2**-8: 0x3F80,               # exact tie -> even (down)
        1.0 + 2**-7 + 2**-8: 0x3F82,       # exact tie -> even (up)
        1.0 + 2**-8 + 2**-20: 0x3F81,      # just above the tie -> up
        -0.0: 0x8000,
        2.0**-149: 0x0000,                 # smallest f32 subnormal rounds to zero
        float(np.finfo(np.float32).max): 0x7F80,  # rounds up into infinity
        float("inf"): 0x7F80,
        float("-inf"): 0xFF80,
    }
    for v, want in cases.items():
        got = O.f32_to_bf16(np.array([v], np.float32))[0]
        assert got == want, (v, hex(got), hex(want))
    nan = O.f32_to_bf16(np.array([np.nan], np.float32))[0]
    assert (nan & 0x7F80) == 0x7F80 and (nan & 0x7F) != 0


def test_bf16_rne_matches_brute_force_nearest():
    rng = np.random.default_rng(123)
    bits = rng.integers(0, 2**32, 4000, dtype=np.uint64).astype(np.uint32)
    # force many exact ties and near-ties
    bits[:1000] = (bits[:1000] & 0xFFFF0000) | 0x8000
    bits[1000:1500] = (bits[1000:1500] & 0xFFFF0000) | 0x7FFF
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    got = O.f32_to_bf16(x)
    want = f64_to_nearest_bf16_bits(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_rne_matches_torch_cast():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    x = rng.integers(0, 2**32, 1 << 20, dtype=np.uint64).astype(np.uint32).view(np.float32)
    x = x[~np.isnan(x)]
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.f32_to_bf16(x), want)


# ------------------------------------------------------------------ exp / sigmoid
def _cr_f32_exp(x: float, mp) -> np.float32:
    """Correctly rounded binary32 exp(x) from a 60-digit evaluation."""
    y = mp.exp(mp.mpf(float(x)))
    f = np.float32(float(y))
    best, bestd = None, None
    for c in (np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))):
        if not np.isfinite(c):
            continue
        d = abs(mp.mpf(float(c)) - y)
        if bestd is None or d < bestd:
            best, bestd = c, d
    return np.float32(best)


def test_exp_is_correctly_rounded_on_a_sample():
    mpmath = pytest.importorskip("mpmath")
    mp = mpmath.mp
    mp.dps = 60
    rng = np.random.default_rng(5)
    xs = np.concatenate([
        rng.uniform(-87.0, 88.5, 6000).astype(np.float32),
        rng.uniform(-1.0, 1.0, 3000).astype(np.float32),
        rng.uniform(-103.0, -87.5, 500).astype(np.float32),   # subnormal results
        np.array([0.0, -0.0, 1.0, -1.0, 0.5, 88.0, -87.0, 1e-8, -1e-8], np.float32),
    ])
    got = O.exp_f32(xs)
    want = np.array([_cr_f32_exp(float(v), mp) for v in xs], np.float32)
    bad = np.nonzero(f32_bits(got) != f32_bits(want))[0]
    assert bad.size == 0, [(float(xs[i]), float(got[i]), float(want[i])) for i in bad[:5]]


def test_exp_special_values():
    xs = np.array([np.nan, np.inf, -np.inf, 89.5, 88.8, -104.5, -200.0, 0.0], np.float32)
    y = O.exp_f32(xs)
    assert np.isnan(y[0])
    assert y[1] == np.inf and y[2] == 0.0 and y[3] == np.inf and y[4] == np.inf
    assert y[5] == 0.0 and y[6] == 0.0 and y[7] == 1.0


def test_sigmoid_closed_forms():
    assert O.sigmoid_f32(0.0) == np.float32(0.5)
    assert O.sigmoid_f32(-0.0) == np.float32(0.5)
    # exp(-g) < 2^-24 makes 1 + exp(-g) round to 1: sigma is exactly one
    assert O.sigmoid_f32(17.0) == np.float32(1.0)
    assert O.sigmoid_f32(100.0) == np.float32(1.0)
    # exp(-g) overflows to +inf: sigma is +0
    assert O.sigmoid_f32(-89.0) == 0.0 and not np.signbit(O.sigmoid_f32(-89.0))
    assert np.isnan(O.sigmoid_f32(float("nan")))


def test_sigmoid_against_high_precision():
    mpmath = pytest.importorskip("mpmath")
    mp = mpmath.mp
    mp.dps = 40
    rng = np.random.default_rng(11)
    for g in rng.normal(0, 4, 2000).astype(np.float32):
        s = O.sigmoid_f32(float(g))
        exact = 1 / (1 + mp.exp(-mp.mpf(float(g))))
        # three roundings (exp, 1 + e, the division), each within 2^-24 relative
        assert abs(float(s) - float(exact)) <= 3.01 * 2.0**-24 * float(exact), (g, s, exact)
        # symmetry of the logistic function: sigma(-g) = 1 - sigma(g)
        s2 = O.sigmoid_f32(float(-g))
        assert abs((float(s) + float(s2)) - 1.0) <= 2 * 2**-24


# ------------------------------------------------------------------ router
def _tiny_router_case(T=37, H=96, E=16, seed=3):
    rng = np.random.default_rng(seed)
    x = W.to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    wr = W.to_bf16_bits((0.1 * rng.standard_normal((E, H))).astype(np.float32))
    b = (0.3 * rng.standard_normal(E)).astype(np.float32)
    return x, wr, b


def test_router_logits_within_dot_product_error_bound():
    T, H, E = 37, 96, 16
    x, wr, b = _tiny_router_case(T, H, E)
    _, _, l, _ = O.route_topk(x, wr, b, T=T, H=H, E=E, K=4, want_logits=True)
    xf, wf = bits_to_f32(x).astype(np.float64), bits_to_f32(wr).astype(np.float64)
    exact = xf @ wf.T + b.astype(np.float64)
    bound = (H + 1) * 2.0**-24 * (np.abs(xf) @ np.abs(wf).T + np.abs(b))
    assert np.all(np.abs(l.astype(np.float64) - exact) <= bound * 1.01)


@pytest.mark.parametrize("K", [1, 2, 4, 8])
def test_router_topk_matches_stable_sort_and_float64_softmax(K):
    T, H, E = 37, 96, 16
    x, wr, b = _tiny_router_case(T, H, E)
    ids, w, l, _ = O.route_topk(x, wr, b, T=T, H=H, E=E, K=K, want_logits=True)
    for t in range(T):
        order = np.lexsort((np.arange(E), -l[t].astype(np.float64)))  # desc logit, then low id
        assert np.array_equal(ids[t], order[:K])
        sel = l[t, order[:K]].astype(np.float64)
        p = np.exp(sel - sel.max())
        p /= p.sum()
        assert np.allclose(w[t], p, rtol=2e-6, atol=0)
        assert abs(float(np.sum(w[t].astype(np.float64))) - 1.0) <= K * 2.0**-23
    if K == 1:
        assert np.all(w == np.float32(1.0))


def test_router_without_renormalisation_is_full_softmax():
    T, H, E, K = 9, 64, 12, 3
    x, wr, b = _tiny_router_case(T, H, E)
    ids, w, l, _ = O.route_topk(x, wr, b, T=T, H=H, E=E, K=K, renormalize=0, want_logits=True)
    p = np.exp(l.astype(np.float64) - l.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    assert np.allclose(w, np.take_along_axis(p, ids, 1), rtol=2e-6)


def test_router_ties_go_to_lower_expert_and_nan_ranks_last():
    E, K = 8, 4
    logits = np.array([
        [1.0, 3.0, 3.0, 0.5, 3.0, -1.0, 0.0, 2.0],
        [0.0, -0.0, 0.0, -0.0, 0.0, -0.0, 0.0, -0.0],
        [np.nan, 1.0, -np.inf, 2.0, np.nan, 0.0, -5.0, 1.0],
    ], np.float32)
    ids, w, _, _ = O.route_topk(logits_in=logits, T=3, H=1, E=E, K=K)
    assert ids[0].tolist() == [1, 2, 4, 7]
    assert ids[1].tolist() == [0, 1, 2, 3]
    assert ids[2].tolist() == [3, 1, 7, 5]
    # equal logits give equal weights: exp(0)=1 each, 1/4 exactly
    assert np.all(w[1] == np.float32(0.25))


def test_router_refuses_grouped_and_sigmoid_scoring():
    logits = np.zeros((2, 8), np.float32)
    with pytest.raises(ValueError):
        O.route_topk(logits_in=logits, T=2, H=1, E=8, K=2, scoring=1)
    with pytest.raises(ValueError):
        O.route_topk(logits_in=logits, T=2, H=1, E=8, K=2, n_group=2)
    with pytest.raises(ValueError):
        O.route_topk(logits_in=logits, T=2, H=1, E=8, K=9)


# ------------------------------------------------------------------ router forms beyond
# the pages' ungrouped softmax (grouped, sigmoid, bias-corrected): pinned by a
# sort-based NumPy formulation and by the cases that reduce to the plain router
def _np_route_ex(l, bias, K, scoring, n_group, topk_group, gmode, renorm):
    """Sort-based restatement: group scores by np.sort, group and expert choice
    by np.lexsort (descending key, then lower index), NaN keys last."""
    T, E = l.shape
    ids = np.zeros((T, K), np.int32)
    w = np.zeros((T, K), np.float32)
    gs = E // n_group
    for t in range(T):
        if scoring == 1:
            sc = np.array([O.lib().oracle_sigmoid_f32(float(v)) for v in l[t]], np.float32)
        else:
            sc = l[t].copy()
        key = (sc + bias).astype(np.float32) if bias is not None else sc
        kk = np.where(np.isnan(key), -np.inf, key).astype(np.float64)
        nanr = np.isnan(key).astype(np.int64)
        g_score = []
        for g in range(n_group):
            blk = key[g * gs:(g + 1) * gs]
            order = np.lexsort((np.arange(gs), -np.where(np.isnan(blk), -np.inf, blk), np.isnan(blk)))
            top = blk[order]
            g_score.append(top[0] if gmode == 0 else np.float32(top[0] + top[1]))
        g_score = np.array(g_score, np.float32)
        gorder = np.lexsort((np.arange(n_group), -np.where(np.isnan(g_score), -np.inf, g_score),
                             np.isnan(g_score)))
        eligible = np.zeros(E, bool)
        for g in gorder[:topk_group]:
            eligible[g * gs:(g + 1) * gs] = True
        cand = np.nonzero(eligible)[0]
        order = np.lexsort((cand, -kk[cand], nanr[cand]))
        sel = cand[order[:K]]
        ids[t] = sel
        if scoring == 1:
            den = np.float32(0.0)
            for j in range(K):
                den = np.float32(den + sc[sel[j]])
            w[t] = [np.float32(sc[j] / den) if renorm else sc[j] for j in sel]
        else:
            m = sc[sel[0]]
            ex = [O.lib().oracle_exp_f32(float(np.float32(sc[j] - m))) for j in sel]
            den = np.float32(0.0)
            for e in ex:
                den = np.float32(den + np.float32(e))
            w[t] = [np.float32(np.float32(e) / den) for e in ex]
    return ids, w


@pytest.mark.parametrize("E,K,n_group,topk_group,gmode,scoring,with_bias", [
    (256, 8, 8, 4, 1, 1, True),     # DeepSeek-V3 shape: sigmoid, bias, sum-of-top-2 groups
    (160, 6, 8, 3, 0, 0, False),    # DeepSeek-V2 shape: softmax, max-of-group
    (64, 4, 4, 2, 1, 1, False),
    (64, 4, 16, 16, 0, 1, True),    # every group eligible: the plain top-k of the keys
    (8, 2, 8, 2, 0, 0, False),      # one expert per group
])
def test_router_ex_matches_sort_based_restatement(E, K, n_group, topk_group, gmode, scoring,
                                                  with_bias):
    rng = np.random.default_rng(E + K + n_group)
    T = 23
    l = rng.standard_normal((T, E)).astype(np.float32)
    l[0, : E // 2] = l[0, E // 2:]           # exact ties between groups and experts
    bias = (0.1 * rng.standard_normal(E)).astype(np.float32) if with_bias else None
    ids, w = O.route_topk_ex(l, bias, T=T, E=E, K=K, scoring=scoring, n_group=n_group,
                             topk_group=topk_group, group_score=gmode)
    want_ids, want_w = _np_route_ex(l, bias, K, scoring, n_group, topk_group, gmode, 1)
    assert np.array_equal(ids, want_ids)
    assert np.array_equal(w.view(np.uint32), want_w.view(np.uint32))
    # the chosen experts lie in at most topk_group groups
    assert np.all([len(set((r // (E // n_group)).tolist())) <= topk_group for r in ids])
    # renormalised weights sum to one within K roundings
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1.0) <= K * 2.0**-23)


def test_router_ex_reduces_to_the_plain_router():
    rng = np.random.default_rng(4)
    T, E, K = 31, 64, 6
    l = rng.standard_normal((T, E)).astype(np.float32)
    plain_ids, plain_w, _, _ = O.route_topk(logits_in=l, T=T, H=1, E=E, K=K)
    # softmax, one group
    ids, w = O.route_topk_ex(l, T=T, E=E, K=K)
    assert np.array_equal(ids, plain_ids) and np.array_equal(w, plain_w)
    # softmax, every group eligible
    ids, w = O.route_topk_ex(l, T=T, E=E, K=K, n_group=8, topk_group=8)
    assert np.array_equal(ids, plain_ids) and np.array_equal(w, plain_w)
    # sigmoid is monotone: without a bias it chooses what softmax chooses, and
    # its weights are the chosen sigmoids over their sum
    ids, w = O.route_topk_ex(l, T=T, E=E, K=K, scoring=1)
    assert np.array_equal(ids, plain_ids)
    s = 1.0 / (1.0 + np.exp(-np.take_along_axis(l, ids, 1).astype(np.float64)))
    assert np.allclose(w, s / s.sum(1, keepdims=True), rtol=1e-6, atol=0)


def test_router_ex_bias_steers_choice_not_weights():
    T, E, K = 3, 16, 2
    l = np.zeros((T, E), np.float32)
    l[:, 5] = 2.0
    bias = np.zeros(E, np.float32)
    bias[11] = 10.0                       # expert 11 is always chosen first ...
    ids, w = O.route_topk_ex(l, bias, T=T, E=E, K=K, scoring=1)
    assert np.all(ids[:, 0] == 11) and np.all(ids[:, 1] == 5)
    # ... but weighs by its own score sigmoid(0) = 0.5 exactly, not by the bias
    s5 = np.float32(1.0) / np.float32(1.0 + np.float32(math.exp(-2.0)))
    den = np.float32(np.float32(0.5) + s5)
    assert np.all(w[:, 0] == np.float32(np.float32(0.5) / den))
    ids, w = O.route_topk_ex(l, bias, T=T, E=E, K=K, scoring=1, renormalize=0)
    assert np.all(w[:, 0] == np.float32(0.5))


def test_router_ex_refusals():
    l = np.zeros((2, 16), np.float32)
    for kw in (dict(scoring=2), dict(n_group=3, topk_group=1), dict(n_group=4, topk_group=5),
               dict(n_group=16, topk_group=1, group_score=1), dict(n_group=8, topk_group=1, K=3)):
        k = kw.pop("K", 2)
        with pytest.raises(ValueError):
            O.route_topk_ex(l, T=2, E=16, K=k, **kw)
    with pytest.raises(ValueError):           # a selection bias only with sigmoid scores
        O.route_topk_ex(l, np.zeros(16, np.float32), T=2, E=16, K=2, scoring=0)


def test_shared_gate_logit_is_a_dot_product():
    T, H, E = 5, 64, 8
    x, wr, _ = _tiny_router_case(T, H, E)
    wsg = W.to_bf16_bits(np.linspace(-0.5, 0.5, H).astype(np.float32))
    _, _, _, gl = O.route_topk(x, wr, None, wsg, T=T, H=H, E=E, K=2)
    exact = bits_to_f32(x).astype(np.float64) @ bits_to_f32(wsg).astype(np.float64)
    assert np.allclose(gl, exact, rtol=0, atol=H * 2**-24 * 4)


# ------------------------------------------------------------------ permute
def _random_ids(T, K, E, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,K,E", [(1, 1, 1), (7, 2, 8), (64, 8, 128), (33, 4, 5), (0, 2, 8)])
def test_permute_is_the_stable_counting_sort(T, K, E):
    H = 16
    ids = _random_ids(T, K, E, T + K + E) if T else np.zeros((0, K), np.int32)
    rng = np.random.default_rng(1)
    x = rng.integers(0, 65535, (T, H), dtype=np.uint16)
    off, sp, p2r, xp = O.permute(ids, x, T=T, K=K, E=E, H=H)
    flat = ids.ravel()
    assert np.array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    assert np.array_equal(sp, np.argsort(flat, kind="stable"))
    assert np.array_equal(p2r[sp], np.arange(T * K))
    # every token appears exactly K times
    assert np.array_equal(np.bincount(sp // K, minlength=T), np.full(T, K))
    assert np.array_equal(xp, x[sp // K]) if T else True
    for e in range(E):
        seg = sp[off[e]:off[e + 1]]
        assert np.all(np.diff(seg) > 0) and np.all(flat[seg] == e)


def test_permute_rejects_out_of_range_ids():
    ids = np.array([[0, 9]], np.int32)
    with pytest.raises(ValueError):
        O.permute(ids, T=1, K=2, E=8)


# ------------------------------------------------------------------ grouped GEMMs
def _silu64(z):
    return z / (1.0 + np.exp(-z))


def _gateup_ref64(A, W13, I):
    """float64 evaluation of one expert, narrowing g and u to bf16 first."""
    a = bits_to_f32(A).astype(np.float64)
    w = bits_to_f32(W13).astype(np.float64)
    g = a @ w[:I].T
    u = a @ w[I:].T
    gb = bits_to_f32(f64_to_nearest_bf16_bits(g)).reshape(g.shape).astype(np.float64)
    ub = bits_to_f32(f64_to_nearest_bf16_bits(u)).reshape(u.shape).astype(np.float64)
    return _silu64(gb) * ub


def _nmse_maxrel(got, ref):
    got = got.astype(np.float64)
    ref = ref.astype(np.float64)
    nmse = float(np.sum((got - ref) ** 2) / max(np.sum(ref**2), 1e-300))
    floor = 0.1 * math.sqrt(float(np.mean(ref**2)))
    rel = float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), floor)))
    return nmse, rel


def test_gateup_narrows_gate_and_up_before_activation():
    # g = u = 1 + 2^-9 in f32 (exact); narrowing rounds both to 1.0, so the
    # result must be bf16(silu(1) * 1) = bf16(0.7310586) = 0x3F3B, while the
    # un-narrowed value silu(1.00195) * 1.00195 = 0.7343 rounds to 0x3F3C.
    H, I = 2, 1
    A = W.to_bf16_bits(np.array([[1.0, 2.0**-9]], np.float32))
    W13 = W.to_bf16_bits(np.array([[1.0, 1.0], [1.0, 1.0]], np.float32))[None]
    off = np.array([0, 1], np.int32)
    act = O.gateup_silu(A, W13, off, P=1, H=H, I=I, G=1)
    assert act[0, 0] == 0x3F3B
    mutant = O.gateup_silu(A, W13, off, P=1, H=H, I=I, G=1, narrow=0)
    assert mutant[0, 0] == 0x3F3C


def test_gateup_gate_half_then_up_half():
    # silu(g)*u is not symmetric in g and u: with g=2, u=-1 the result is
    # -silu(2) = -1.7616, with the halves swapped it would be silu(-1)*2 = -0.5379
    H, I = 1, 1
    A = W.to_bf16_bits(np.array([[1.0]], np.float32))
    W13 = W.to_bf16_bits(np.array([[2.0], [-1.0]], np.float32))[None]
    act = O.gateup_silu(A, W13, np.array([0, 1], np.int32), P=1, H=H, I=I, G=1)
    want = f64_to_nearest_bf16_bits(np.array([-_silu64(2.0)]))[0]
    assert act[0, 0] == want


def _grouped_case(P=45, H=64, I=24, G=5, seed=9):
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.integers(0, P + 1, G - 1))
    off = np.concatenate([[0], cuts, [P]]).astype(np.int32)
    A = W.to_bf16_bits(rng.standard_normal((P, H)).astype(np.float32))
    W13 = W.to_bf16_bits((0.1 * rng.standard_normal((G, 2 * I, H))).astype(np.float32))
    W2 = W.to_bf16_bits((0.1 * rng.standard_normal((G, H, I))).astype(np.float32))
    return off, A, W13, W2


def test_grouped_gateup_against_float64_per_group():
    P, H, I, G = 45, 64, 24, 5
    off, A, W13, _ = _grouped_case(P, H, I, G)
    act = O.gateup_silu(A, W13, off, P=P, H=H, I=I, G=G)
    ref = np.zeros((P, I))
    for g in range(G):
        ref[off[g]:off[g + 1]] = _gateup_ref64(A[off[g]:off[g + 1]], W13[g], I)
    nmse, rel = _nmse_maxrel(bits_to_f32(act), ref)
    assert nmse <= 1e-5 and rel <= 2e-2, (nmse, rel)


def test_grouped_gateup_row_gather_and_row_subset():
    P, H, I, G = 45, 64, 24, 5
    off, A, W13, _ = _grouped_case(P, H, I, G)
    full = O.gateup_silu(A, W13, off, P=P, H=H, I=I, G=G)
    rng = np.random.default_rng(2)
    perm = rng.permutation(P).astype(np.int32)
    src = A[perm]                      # row r of A is row perm^-1... gathered back below
    inv = np.argsort(perm).astype(np.int32)
    gathered = O.gateup_silu(src, W13, off, P=P, H=H, I=I, G=G, a_row_gather=inv)
    assert np.array_equal(gathered, full)
    rows = np.array([0, 7, 44, 20], np.int32)
    part = O.gateup_silu(A, W13, off, P=P, H=H, I=I, G=G, rows=rows)
    assert np.array_equal(part[rows], full[rows])


def test_grouped_down_against_float64_with_weight_and_scatter():
    P, H, I, G = 45, 64, 24, 5
    off, _, _, W2 = _grouped_case(P, H, I, G)
    rng = np.random.default_rng(4)
    act = W.to_bf16_bits(rng.standard_normal((P, I)).astype(np.float32))
    wts = rng.uniform(0.05, 1.0, P).astype(np.float32)
    r2p = rng.permutation(P).astype(np.int32)
    out = O.down(act, W2, off, P=P, I=I, H=H, G=G, pair_weight=wts, row_to_pair=r2p)
    a = bits_to_f32(act).astype(np.float64)
    ref = np.zeros((P, H))
    for g in range(G):
        rr = np.arange(off[g], off[g + 1])
        y = a[rr] @ bits_to_f32(W2[g]).astype(np.float64).T
        ref[r2p[rr]] = y * wts[r2p[rr], None]
    nmse, rel = _nmse_maxrel(bits_to_f32(out), ref)
    assert nmse <= 1e-5 and rel <= 2e-2, (nmse, rel)


def test_routing_weight_applied_exactly_once():
    # With power-of-two weights, scaling commutes with every rounding, so the
    # weight applied in the down projection (and the combine unweighted) must
    # give the same bits as the weight applied in the combine (down
    # unweighted).  A weight applied twice, or never, breaks the identity.
    T, K, H, I, E = 6, 2, 32, 16, 4
    rng = np.random.default_rng(8)
    ids = _random_ids(T, K, E, 8)
    off, sp, p2r, _ = O.permute(ids, T=T, K=K, E=E)
    act = W.to_bf16_bits(rng.standard_normal((T * K, I)).astype(np.float32))
    W2 = W.to_bf16_bits((0.2 * rng.standard_normal((E, H, I))).astype(np.float32))
    wts = (2.0 ** -rng.integers(1, 4, T * K)).astype(np.float32)
    a = O.down(act, W2, off, P=T * K, I=I, H=H, G=E, pair_weight=wts, row_to_pair=sp)
    b = O.down(act, W2, off, P=T * K, I=I, H=H, G=E, pair_weight=None, row_to_pair=sp)
    out_a = O.combine(a.reshape(T, K, H), None, T=T, K=K, H=H)
    out_b = O.combine(b.reshape(T, K, H), wts.reshape(T, K), T=T, K=K, H=H)
    assert np.array_equal(out_a, out_b)
    twice = O.combine(a.reshape(T, K, H), wts.reshape(T, K), T=T, K=K, H=H)
    assert not np.array_equal(twice, out_b)


def test_down_rounds_once_after_the_weight():
    # Issue #3094 (numeric contract): the routing weight is applied before the
    # down result is stored, so the store rounding comes after the weight:
    # out = bf16(y * w), one rounding.  Here y = 1 + 2^-8 + 2^-10 exactly (a dot
    # product of three exact terms) and w = 0.75, worked by hand:
    #   y * w = 0.753662109375 = 2^-1 * (1 + 64.9375 / 128)  -> bf16 0x3F41 (0.75390625)
    # A store-width rounding before the weight gives a different value:
    #   bf16(y) = 1 + 1/128;  (1 + 1/128) * 0.75 = 2^-1 * (1 + 65.5 / 128), a tie
    #   -> even 66 / 128  -> bf16 0x3F42 (0.7578125)
    I, H = 8, 16
    act = np.zeros((1, I), np.float32)
    act[0, :3] = [1.0, 2.0**-8, 2.0**-10]
    w2 = np.zeros((1, H, I), np.float32)
    w2[0, :, :3] = 1.0
    off = np.array([0, 1], np.int32)
    out = O.down(W.to_bf16_bits(act), W.to_bf16_bits(w2), off, P=1, I=I, H=H, G=1,
                 pair_weight=np.array([0.75], np.float32))
    assert np.all(out == 0x3F41)
    # the mutant that rounds y to bf16 before the weight gives 0x3F42 here
    y_bf16 = W.to_bf16_bits(np.array([1.0 + 2.0**-8 + 2.0**-10], np.float32))
    mutant = W.to_bf16_bits(O.bf16_to_f32(y_bf16) * np.float32(0.75))
    assert mutant[0] == 0x3F42 and not np.any(out == mutant[0])
    # and with no weight the one rounding is of y itself: 1 + 1/128
    plain = O.down(W.to_bf16_bits(act), W.to_bf16_bits(w2), off, P=1, I=I, H=H, G=1)
    assert np.all(plain == 0x3F81)


def test_sparse_path_equals_dense_evaluation_of_every_expert():
    cfg = W.TINY
    d = W.layer_inputs(cfg)
    T, H, I, E, K = cfg.T, cfg.H, cfg.I, cfg.E, cfg.K
    ids, wts, _, _ = O.route_topk(d["x"], d["w_router"], T=T, H=H, E=E, K=K)
    off, sp, p2r, xp = O.permute(ids, d["x"], T=T, K=K, E=E, H=H)
    act = O.gateup_silu(xp, d["w13"], off, P=T * K, H=H, I=I, G=E)
    eo = O.down(act, d["w2"], off, P=T * K, I=I, H=H, G=E, pair_weight=wts.ravel(),
                row_to_pair=sp)
    # dense: every expert on every token, then pick (t, ids[t, j])
    for e in range(E):
        one = np.array([0, T], np.int32)
        dense_act = O.gateup_silu(d["x"], d["w13"][e:e + 1], one, P=T, H=H, I=I, G=1)
        for t in range(T):
            for j in range(K):
                if ids[t, j] != e:
                    continue
                p = t * K + j
                assert np.array_equal(act[p2r[p]], dense_act[t])
                wrow = np.full(1, wts[t, j], np.float32)
                dense_out = O.down(dense_act[t:t + 1], d["w2"][e:e + 1], np.array([0, 1], np.int32),
                                   P=1, I=I, H=H, G=1, pair_weight=wrow)
                assert np.array_equal(eo[p], dense_out[0])


# ------------------------------------------------------------------ combine / gate
def _exact_case(T, K, H, seed):
    """bf16 values k/8 with |k| < 64: every partial sum is exact in f32."""
    rng = np.random.default_rng(seed)
    eo = (rng.integers(-63, 64, (T, K, H)) / 8.0).astype(np.float32)
    return eo


@pytest.mark.parametrize("out_dtype", [F32, BF16])
def test_combine_sums_the_right_rows(out_dtype):
    T, K, H = 5, 3, 40
    eo = _exact_case(T, K, H, 1)
    sh = (np.random.default_rng(2).integers(-63, 64, (T, H)) / 4.0).astype(np.float32)
    out = O.combine(W.to_bf16_bits(eo), None, W.to_bf16_bits(sh), T=T, K=K, H=H,
                    out_dtype=out_dtype)
    exact = eo.astype(np.float64).sum(1) + sh
    if out_dtype == F32:
        assert np.array_equal(out, exact.astype(np.float32))
    else:
        assert np.array_equal(out.ravel(), f64_to_nearest_bf16_bits(exact))


def test_combine_sums_in_sequential_k_order():
    big = 2.0**25  # 2^25 + 1 is not an f32: order decides whether the 1 survives
    eo1 = np.array([[[big], [-big], [1.0]]], np.float32)   # ((0+B)-B)+1 = 1
    eo2 = np.array([[[1.0], [big], [-big]]], np.float32)   # ((0+1)+B)-B = 0
    o1 = O.combine(eo1, None, T=1, K=3, H=1, out_dtype=F32)
    o2 = O.combine(eo2, None, T=1, K=3, H=1, out_dtype=F32)
    assert o1[0, 0] == 1.0 and o2[0, 0] == 0.0


def test_combine_does_not_fuse_multiply_add():
    # p = (1+2^-7)(1+2^-20) = 1 + 2^-7 + 2^-20 + 2^-27 rounds to drop 2^-27 when
    # multiplied on its own; the second term cancels the rounded first one
    # exactly, whereas a fused multiply-add would leave -2^-27.
    eo = np.array([[[1.0 + 2**-7], [-(1.0 + 2**-7)]]], np.float32)
    w = np.array([[1.0 + 2**-20, 1.0 + 2**-20]], np.float32)
    out = O.combine(W.to_bf16_bits(eo), w, T=1, K=2, H=1, out_dtype=F32)
    assert out[0, 0] == 0.0


def test_combine_routed_scale_before_shared_term_and_identity():
    eo = np.array([[[2.0]]], np.float32)
    sh = np.array([[1.0]], np.float32)
    out = O.combine(eo, None, sh, routed_scale=0.5, T=1, K=1, H=1, out_dtype=F32)
    assert out[0, 0] == 2.0           # 2*0.5 + 1, not (2+1)*0.5
    rng = np.random.default_rng(3)
    e = W.to_bf16_bits(rng.standard_normal((7, 1, 33)).astype(np.float32))
    same = O.combine(e, np.ones((7, 1), np.float32), T=7, K=1, H=33)
    assert np.array_equal(same, e[:, 0, :])
    half = O.combine(e, None, routed_scale=0.25, T=7, K=1, H=33, out_dtype=F32)
    assert np.array_equal(half, bits_to_f32(e[:, 0, :]) * np.float32(0.25))


def test_combine_refuses_f16():
    eo = np.zeros((1, 1, 4), np.float16)
    with pytest.raises(ValueError):
        O.combine(eo, None, T=1, K=1, H=4)


def test_shared_gate_closed_forms_all_arms():
    rng = np.random.default_rng(6)
    T, H = 4, 24
    sd32 = rng.standard_normal((T, H)).astype(np.float32)
    sdb = W.to_bf16_bits(sd32)
    gl = np.array([0.0, 100.0, -100.0, 0.0], np.float32)
    for sd, sdt in ((sd32, F32), (sdb, BF16)):
        sdf = sd if sdt == F32 else bits_to_f32(sd)
        o32 = O.shared_expert_gate(sd, gl, T=T, H=H, out_dtype=F32)
        assert np.array_equal(o32[0], sdf[0] * np.float32(0.5))     # sigma(0) = 1/2
        assert np.array_equal(o32[1], sdf[1])                      # sigma(100) = 1
        assert np.all(o32[2] == 0.0)                               # sigma(-100) = 0
        ob = O.shared_expert_gate(sd, gl, T=T, H=H, out_dtype=BF16)
        assert np.array_equal(ob[0], f64_to_nearest_bf16_bits(sdf[0].astype(np.float64) * 0.5))


def test_shared_gate_against_float64():
    mpmath = pytest.importorskip("mpmath")
    rng = np.random.default_rng(10)
    T, H = 16, 8
    sd = rng.standard_normal((T, H)).astype(np.float32)
    gl = rng.normal(0, 2, T).astype(np.float32)
    out = O.shared_expert_gate(sd, gl, T=T, H=H, out_dtype=F32)
    for t in range(T):
        s = float(1 / (1 + mpmath.exp(-mpmath.mpf(float(gl[t])))))
        ref = s * sd[t].astype(np.float64)
        assert np.all(np.abs(out[t] - ref) <= 2.0 * np.spacing(np.abs(ref).astype(np.float32)))


def test_combine_gate_double_rounds_the_shared_term():
    # sd = 1 + 2^-9 (f32), sigma = 1: the gated term is rounded to bf16 (1.0)
    # before it is added, so out = 2 + 1 = 3 exactly (and not 3 + 2^-9).
    eo = np.array([[[2.0]]], np.float32)
    sd = np.array([[1.0 + 2**-9]], np.float32)
    gl = np.array([100.0], np.float32)
    out = O.combine_gate(eo, None, sd, gl, T=1, K=1, H=1, out_dtype=F32)
    assert out[0, 0] == 3.0


@pytest.mark.parametrize("eo_dt,sd_dt,out_dt", [(BF16, BF16, BF16), (F32, F32, F32),
                                                 (BF16, F32, F32), (F32, BF16, BF16)])
@pytest.mark.parametrize("rs", [1.0, 0.7])
def test_combine_gate_equals_host_composite(eo_dt, sd_dt, out_dt, rs):
    # combine_gate == combine(shared = bf16(shared_expert_gate(sd, gl))), the
    # host composite the pages use as the fused op's check
    rng = np.random.default_rng(12)
    T, K, H = 9, 4, 40
    eo = rng.standard_normal((T, K, H)).astype(np.float32)
    sd = rng.standard_normal((T, H)).astype(np.float32)
    if eo_dt == BF16:
        eo = W.to_bf16_bits(eo)
    if sd_dt == BF16:
        sd = W.to_bf16_bits(sd)
    gl = rng.normal(0, 2, T).astype(np.float32)
    gl[0] = 0.0
    w = rng.uniform(0, 1, (T, K)).astype(np.float32)
    for ww in (w, None):
        fused = O.combine_gate(eo, ww, sd, gl, routed_scale=rs, T=T, K=K, H=H, out_dtype=out_dt)
        shared = O.shared_expert_gate(sd, gl, T=T, H=H, out_dtype=BF16)
        comp = O.combine(eo, ww, shared, routed_scale=rs, T=T, K=K, H=H, out_dtype=out_dt)
        assert np.array_equal(fused, comp)


# ------------------------------------------------------------------ whole layer
def test_token_path_equals_batch_path_on_tiny_layer():
    cfg = W.TINY
    d = W.layer_inputs(cfg)
    T, H, I, E, K, Is = cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, cfg.I_shared
    ids, wts, _, gl = O.route_topk(d["x"], d["w_router"], None, d["w_shared_gate"], T=T, H=H, E=E,
                                   K=K)
    off, sp, p2r, _ = O.permute(ids, T=T, K=K, E=E)
    act = O.gateup_silu(d["x"], d["w13"], off, P=T * K, H=H, I=I, G=E,
                        a_row_gather=(sp // K).astype(np.int32))
    eo = O.down(act, d["w2"], off, P=T * K, I=I, H=H, G=E, pair_weight=wts.ravel(), row_to_pair=sp)
    one = np.array([0, T], np.int32)
    sact = O.gateup_silu(d["x"], d["w13_shared"], one, P=T, H=H, I=Is, G=1)
    sd = O.down(sact, d["w2_shared"], one, P=T, I=Is, H=H, G=1)
    out = O.combine_gate(eo.reshape(T, K, H), None, sd, gl, T=T, K=K, H=H)
    tok_out, tok_ids, tok_w = O.moe_layer_tokens(
        d["x"], d["w_router"], None, d["w13"], d["w2"], d["w_shared_gate"], d["w13_shared"],
        d["w2_shared"], H=H, I=I, E=E, K=K, I_shared=Is, tokens=np.arange(T, dtype=np.int32))
    assert np.array_equal(tok_ids, ids) and np.array_equal(tok_w, wts)
    assert np.array_equal(tok_out, out)


def test_oracle_threads_do_not_change_bits():
    cfg = W.TINY
    d = W.layer_inputs(cfg)
    args = (d["x"], d["w_router"], None, d["w13"], d["w2"], d["w_shared_gate"], d["w13_shared"],
            d["w2_shared"])
    kw = dict(H=cfg.H, I=cfg.I, E=cfg.E, K=cfg.K, I_shared=cfg.I_shared,
              tokens=np.arange(cfg.T, dtype=np.int32))
    n = O.max_threads()
    O.set_threads(1)
    a = O.moe_layer_tokens(*args, **kw)[0]
    O.set_threads(n)
    b = O.moe_layer_tokens(*args, **kw)[0]
    assert np.array_equal(a, b)


# ------------------------------------------------------------------ block-scaled FP8 weights
def test_e4m3_decode_matches_torch_float8_on_every_code():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    got = O.e4m3_to_f32(codes)
    want = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok].view(np.uint32), want[ok].view(np.uint32))
    # hand values: smallest subnormal, smallest normal, one, largest finite, NaN
    assert got[0x01] == 2.0**-9 and got[0x08] == 2.0**-6 and got[0x38] == 1.0
    assert got[0x7E] == 448.0 and np.isnan(got[0x7F]) and np.isnan(got[0xFF])


def test_fp8_block_dequant_uses_each_block_scale_once():
    # code 0x38 is 1.0 everywhere; block (g, i, j) gets scale 2^(g + 2i - j), so
    # every weight is exactly that power of two in bf16 and the block map shows
    G, R, C = 2, 300, 200
    q = np.full((G, R, C), 0x38, np.uint8)
    rb, cb = (R + 127) // 128, (C + 127) // 128
    scale = np.zeros((G, rb, cb), np.float32)
    for g in range(G):
        for i in range(rb):
            for j in range(cb):
                scale[g, i, j] = 2.0 ** (g + 2 * i - j)
    w = bits_to_f32(O.dequant_fp8_block(q, scale, G=G, R=R, C=C))
    r = np.arange(R)[None, :, None] // 128
    c = np.arange(C)[None, None, :] // 128
    g = np.arange(G)[:, None, None]
    assert np.array_equal(w, (2.0 ** (g + 2 * r - c)).astype(np.float32))


def test_fp8_block_dequant_rounds_the_product_once_to_bf16():
    rng = np.random.default_rng(12)
    G, R, C = 1, 128, 128
    q = rng.integers(0, 256, (G, R, C), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x30                     # no NaN codes
    scale = np.array([[[0.013]]], np.float32)
    w = O.dequant_fp8_block(q, scale, G=G, R=R, C=C)
    prod = (O.e4m3_to_f32(q).astype(np.float32) * np.float32(0.013)).astype(np.float32)
    assert np.array_equal(w.ravel(), f64_to_nearest_bf16_bits(prod.astype(np.float64)))
