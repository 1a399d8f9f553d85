"""NumPy front end of the plain CPU oracle (``moe_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  It shares no
code with the GPU library and never imports it.

Arrays: bf16 tensors travel as ``numpy.uint16`` holding the bf16 bit
patterns; f32 as ``numpy.float32``; indices as ``numpy.int32``.  Every
function mirrors one entry point of the GPU C-ABI, with host arrays and
without stream or workspace.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import build as _build

F32, BF16, F16 = 0, 1, 2
OK, ERR_ARG, ERR_DTYPE, ERR_UNSUPPORTED = 0, -1, -2, -3

_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        path = _build.build()
        _lib = ctypes.CDLL(path)
        _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_F = ctypes.c_float


def _declare(L: ctypes.CDLL) -> None:
    sig = {
        "oracle_abi_version": ([], _I),
        "oracle_set_threads": ([_I], None),
        "oracle_max_threads": ([], _I),
        "oracle_bf16_to_f32": ([ctypes.c_uint16], _F),
        "oracle_f32_to_bf16": ([_F], ctypes.c_uint16),
        "oracle_f32_to_bf16_array": ([_P, _P, _I64], None),
        "oracle_exp_f32": ([_F], _F),
        "oracle_exp_f32_array": ([_P, _P, _I64], None),
        "oracle_sigmoid_f32": ([_F], _F),
        "oracle_sigmoid_f32_array": ([_P, _P, _I64], None),
        "oracle_route_topk": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P], _I),
        "oracle_route_topk_ex": ([_P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P], _I),
        "oracle_e4m3_to_f32": ([ctypes.c_uint8], _F),
        "oracle_dequant_fp8_block": ([_P, _P, _I, _I, _I, _P], _I),
        "oracle_permute": ([_P, _P, _I, _I, _I, _I, _P, _P, _P, _P], _I),
        "oracle_gateup_silu": ([_P, _P, _P, _P, _I, _I, _I, _I, _P, _I, _P, _I], _I),
        "oracle_down": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _I, _P], _I),
        "oracle_combine": ([_P, _I, _P, _P, _I, _F, _I, _I, _I, _P, _I], _I),
        "oracle_combine_gate": ([_P, _I, _P, _P, _I, _P, _F, _I, _I, _I, _P, _I], _I),
        "oracle_shared_expert_gate": ([_P, _I, _P, _I, _I, _P, _I], _I),
        "oracle_moe_layer_tokens": ([_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F,
                                     _P, _I, _P, _P, _P], _I),
        "oracle_f16_to_f32": ([ctypes.c_uint16], _F),
        "oracle_f32_to_f16": ([_F], ctypes.c_uint16),
        "oracle_q4k_scale_min": ([_P, _I, _P], _I),
        "oracle_dequant_q": ([_P, _I, _I64, _I, _P], _I),
        "oracle_dequant_q_bf16": ([_P, _I, _I64, _I, _P], _I),
        "oracle_quantize_act_q8": ([_P, _I64, _I, _I, _P, _P], _I),
        "oracle_gemm_q": ([_P, _P, _P, _I, _P, _I, _P, _I, _I, _I, _I, _P, _I, _P, _P], _I),
        "oracle_gateup_silu_q": ([_P, _P, _P, _I, _P, _I, _P, _I, _I, _I, _I, _P, _I, _P], _I),
        "oracle_down_q": ([_P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _I, _P, _I, _P], _I),
        "oracle_moe_layer_tokens_q": ([_P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _I, _I,
                                       _F, _P, _I, _P, _P, _P], _I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _dt(a) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float16:
        return F16
    raise TypeError(f"unsupported dtype {a.dtype}")


def _check(rc: int, what: str) -> None:
    if rc != OK:
        raise ValueError(f"oracle {what} refused its arguments (code {rc})")


def set_threads(n: int) -> None:
    lib().oracle_set_threads(int(n))


def max_threads() -> int:
    return int(lib().oracle_max_threads())


# ---------------------------------------------------------------- scalars
def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening: the bf16 bits become the upper half of an f32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_f32_to_bf16_array(_ptr(x), _ptr(out), x.size)
    return out


def exp_f32(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(x)
    lib().oracle_exp_f32_array(_ptr(x), _ptr(out), x.size)
    return out


def sigmoid_f32(g: float) -> np.float32:
    return np.float32(lib().oracle_sigmoid_f32(float(g)))


def sigmoid_f32_array(g: np.ndarray) -> np.ndarray:
    g = np.ascontiguousarray(g, np.float32)
    out = np.empty_like(g)
    lib().oracle_sigmoid_f32_array(_ptr(g), _ptr(out), g.size)
    return out


# ---------------------------------------------------------------- steps
def route_topk(x=None, w_router=None, logit_bias=None, w_shared_gate=None, logits_in=None, *,
               T, H, E, K, renormalize=1, scoring=0, n_group=1, want_logits=False):
    ids = np.zeros((T, K), np.int32)
    w = np.zeros((T, K), np.float32)
    logits = np.zeros((T, E), np.float32) if want_logits else None
    gl = np.zeros((T,), np.float32) if w_shared_gate is not None else None
    rc = lib().oracle_route_topk(_ptr(x), _ptr(w_router), _ptr(logit_bias), _ptr(w_shared_gate),
                                 _ptr(logits_in), T, H, E, K, renormalize, scoring, n_group,
                                 _ptr(ids), _ptr(w), _ptr(logits), _ptr(gl))
    _check(rc, "route_topk")
    return ids, w, logits, gl


def route_topk_ex(logits, select_bias=None, *, T, E, K, renormalize=1, scoring=0, n_group=1,
                  topk_group=1, group_score=0):
    """The grouped / sigmoid / bias-corrected router forms on given f32 logits [T, E]."""
    ids = np.zeros((T, K), np.int32)
    w = np.zeros((T, K), np.float32)
    rc = lib().oracle_route_topk_ex(_ptr(np.ascontiguousarray(logits, np.float32)),
                                    _ptr(select_bias), T, E, K, renormalize, scoring, n_group,
                                    topk_group, group_score, _ptr(ids), _ptr(w))
    _check(rc, "route_topk_ex")
    return ids, w


def e4m3_to_f32(codes):
    """f32 values of FP8 E4M3 codes (uint8 array)."""
    codes = np.ascontiguousarray(codes, np.uint8)
    return np.array([lib().oracle_e4m3_to_f32(int(c)) for c in codes.ravel()],
                    np.float32).reshape(codes.shape)


def dequant_fp8_block(q, scale, *, G, R, C):
    """bf16 bits [G, R, C] of block-scaled FP8 weights (scale [G, ceil(R/128), ceil(C/128)])."""
    w = np.zeros((G, R, C), np.uint16)
    rc = lib().oracle_dequant_fp8_block(_ptr(np.ascontiguousarray(q, np.uint8)),
                                        _ptr(np.ascontiguousarray(scale, np.float32)), G, R, C,
                                        _ptr(w))
    _check(rc, "dequant_fp8_block")
    return w


def permute(topk_ids, x=None, *, T, K, E, H=0):
    P = T * K
    off = np.zeros((E + 1,), np.int32)
    sp = np.zeros((P,), np.int32)
    p2r = np.zeros((P,), np.int32)
    xp = np.zeros((P, H), np.uint16) if x is not None else None
    rc = lib().oracle_permute(_ptr(np.ascontiguousarray(topk_ids, np.int32)), _ptr(x), T, K, E, H,
                              _ptr(off), _ptr(sp), _ptr(p2r), _ptr(xp))
    _check(rc, "permute")
    return off, sp, p2r, xp


def gateup_silu(a, w13, group_offsets, *, P, H, I, G, a_row_gather=None, rows=None, narrow=1,
                act=None):
    if act is None:
        act = np.zeros((P, I), np.uint16)
    r = None if rows is None else np.ascontiguousarray(rows, np.int32)
    rc = lib().oracle_gateup_silu(_ptr(a), _ptr(a_row_gather), _ptr(w13), _ptr(group_offsets),
                                  P, H, I, G, _ptr(r), 0 if r is None else r.size, _ptr(act),
                                  narrow)
    _check(rc, "gateup_silu")
    return act


def down(act, w2, group_offsets, *, P, I, H, G, pair_weight=None, row_to_pair=None, rows=None,
         out=None):
    if out is None:
        out = np.zeros((P, H), np.uint16)
    r = None if rows is None else np.ascontiguousarray(rows, np.int32)
    rc = lib().oracle_down(_ptr(act), _ptr(w2), _ptr(group_offsets), _ptr(pair_weight),
                           _ptr(row_to_pair), P, I, H, G, _ptr(r), 0 if r is None else r.size,
                           _ptr(out))
    _check(rc, "down")
    return out


def combine(expert_out, w=None, shared=None, *, routed_scale=1.0, T, K, H, out_dtype=BF16):
    out = np.zeros((T, H), np.float32 if out_dtype == F32 else np.uint16)
    rc = lib().oracle_combine(_ptr(expert_out), _dt(expert_out), _ptr(w), _ptr(shared),
                              _dt(shared) if shared is not None else BF16, routed_scale, T, K, H,
                              _ptr(out), out_dtype)
    _check(rc, "combine")
    return out


def combine_gate(expert_out, w, sd, gl, *, routed_scale=1.0, T, K, H, out_dtype=BF16):
    out = np.zeros((T, H), np.float32 if out_dtype == F32 else np.uint16)
    rc = lib().oracle_combine_gate(_ptr(expert_out), _dt(expert_out), _ptr(w), _ptr(sd), _dt(sd),
                                   _ptr(gl), routed_scale, T, K, H, _ptr(out), out_dtype)
    _check(rc, "combine_gate")
    return out


def shared_expert_gate(sd, gl, *, T, H, out_dtype=BF16):
    out = np.zeros((T, H), np.float32 if out_dtype == F32 else np.uint16)
    rc = lib().oracle_shared_expert_gate(_ptr(sd), _dt(sd), _ptr(gl), T, H, _ptr(out), out_dtype)
    _check(rc, "shared_expert_gate")
    return out


def moe_layer_tokens(x, w_router, logit_bias, w13, w2, w_shared_gate, w13_shared, w2_shared, *,
                     H, I, E, K, I_shared=0, routed_scale=1.0, tokens):
    tok = np.ascontiguousarray(tokens, np.int32)
    n = tok.size
    ids = np.zeros((n, K), np.int32)
    w = np.zeros((n, K), np.float32)
    out = np.zeros((n, H), np.uint16)
    rc = lib().oracle_moe_layer_tokens(_ptr(x), _ptr(w_router), _ptr(logit_bias), _ptr(w13),
                                       _ptr(w2), _ptr(w_shared_gate), _ptr(w13_shared),
                                       _ptr(w2_shared), H, I, E, K, I_shared, routed_scale,
                                       _ptr(tok), n, _ptr(ids), _ptr(w), _ptr(out))
    _check(rc, "moe_layer_tokens")
    return out, ids, w


# ---------------------------------------------------------------- keep-quant
Q8_0, Q4_K = 1, 2
Q_BLOCK = {Q8_0: 32, Q4_K: 256}          # weights per block
Q_BLOCK_BYTES = {Q8_0: 34, Q4_K: 144}    # bytes per block


def f16_to_f32(bits):
    """f32 values of fp16 bit patterns (uint16 array)."""
    bits = np.ascontiguousarray(bits, np.uint16)
    return np.array([lib().oracle_f16_to_f32(int(b)) for b in bits.ravel()],
                    np.float32).reshape(bits.shape)


def f32_to_f16(x):
    """fp16 bit patterns (round to nearest even) of f32 values."""
    x = np.ascontiguousarray(x, np.float32)
    return np.array([lib().oracle_f32_to_f16(float(v)) for v in x.ravel()],
                    np.uint16).reshape(x.shape)


def q4k_scale_min(scales12, j):
    """(scale, min) of Q4_K sub-block j from the 12 packed scale bytes."""
    out = np.zeros(2, np.int32)
    _check(lib().oracle_q4k_scale_min(_ptr(np.ascontiguousarray(scales12, np.uint8)), int(j),
                                      _ptr(out)), "q4k_scale_min")
    return int(out[0]), int(out[1])


def dequant_q(w, fmt, *, rows, K):
    """exact values (float64 [rows, K]) of `rows` weight rows stored in `fmt` blocks."""
    out = np.zeros((rows, K), np.float64)
    rc = lib().oracle_dequant_q(_ptr(np.ascontiguousarray(w, np.uint8)), fmt, rows, K, _ptr(out))
    _check(rc, "dequant_q")
    return out


def dequant_q_bf16(w, fmt, *, rows, K):
    """bf16 bits [rows, K] of keep-quant weight rows (value formed in f32, rounded once)."""
    out = np.zeros((rows, K), np.uint16)
    rc = lib().oracle_dequant_q_bf16(_ptr(np.ascontiguousarray(w, np.uint8)), fmt, rows, K,
                                     _ptr(out))
    _check(rc, "dequant_q_bf16")
    return out


def quantize_act_q8(x, fmt, *, R, K):
    """8-bit activation blocks of bf16 rows x [R, K]: (codes int8 [R, K], scales f32 [R, K/blk])."""
    q = np.zeros((R, K), np.int8)
    d = np.zeros((R, K // Q_BLOCK[fmt]), np.float32)
    rc = lib().oracle_quantize_act_q8(_ptr(np.ascontiguousarray(x, np.uint16)), R, K, fmt,
                                      _ptr(q), _ptr(d))
    _check(rc, "quantize_act_q8")
    return q, d


def gemm_q(aq, ad, w, fmt, group_offsets, *, P, K, N, G, a_row_gather=None, gather_div=1,
           rows=None):
    """plain grouped keep-quant matmul: (y float64 [P, N], yabs float64 [P, N])."""
    y = np.zeros((P, N), np.float64)
    ya = np.zeros((P, N), np.float64)
    r = None if rows is None else np.ascontiguousarray(rows, np.int32)
    rc = lib().oracle_gemm_q(_ptr(aq), _ptr(ad), _ptr(a_row_gather), gather_div, _ptr(w), fmt,
                             _ptr(group_offsets), P, K, N, G, _ptr(r), 0 if r is None else r.size,
                             _ptr(y), _ptr(ya))
    _check(rc, "gemm_q")
    return y, ya


def gateup_silu_q(aq, ad, w13, fmt, group_offsets, *, P, H, I, G, a_row_gather=None,
                  gather_div=1, rows=None):
    act = np.zeros((P, I), np.uint16)
    r = None if rows is None else np.ascontiguousarray(rows, np.int32)
    rc = lib().oracle_gateup_silu_q(_ptr(aq), _ptr(ad), _ptr(a_row_gather), gather_div, _ptr(w13),
                                    fmt, _ptr(group_offsets), P, H, I, G, _ptr(r),
                                    0 if r is None else r.size, _ptr(act))
    _check(rc, "gateup_silu_q")
    return act


def down_q(aq, ad, w2, fmt, group_offsets, *, P, I, H, G, pair_weight=None, row_to_pair=None,
           rows=None):
    out = np.zeros((P, H), np.uint16)
    r = None if rows is None else np.ascontiguousarray(rows, np.int32)
    rc = lib().oracle_down_q(_ptr(aq), _ptr(ad), _ptr(w2), fmt, _ptr(group_offsets),
                             _ptr(pair_weight), _ptr(row_to_pair), P, I, H, G, _ptr(r),
                             0 if r is None else r.size, _ptr(out))
    _check(rc, "down_q")
    return out


def moe_layer_tokens_q(x, w_router, logit_bias, w13q, w2q, fmt, w_shared_gate, w13_shared,
                       w2_shared, *, H, I, E, K, I_shared=0, routed_scale=1.0, tokens):
    tok = np.ascontiguousarray(tokens, np.int32)
    n = tok.size
    ids = np.zeros((n, K), np.int32)
    w = np.zeros((n, K), np.float32)
    out = np.zeros((n, H), np.uint16)
    rc = lib().oracle_moe_layer_tokens_q(_ptr(x), _ptr(w_router), _ptr(logit_bias), _ptr(w13q),
                                         _ptr(w2q), fmt, _ptr(w_shared_gate), _ptr(w13_shared),
                                         _ptr(w2_shared), H, I, E, K, I_shared, routed_scale,
                                         _ptr(tok), n, _ptr(ids), _ptr(w), _ptr(out))
    _check(rc, "moe_layer_tokens_q")
    return out, ids, w


def abi_version() -> int:
    return int(lib().oracle_abi_version())


__all__ = [n for n in dir() if not n.startswith("_")]
