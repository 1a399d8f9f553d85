"""Python binding of libmoe.so: the BF16 MoE expert block on one GB300.

Argument marshalling only.  Every function here has the name, argument order
and meaning of the C entry point declared in ``include/moe.h``; tensors are
passed as raw device pointers (``tensor.data_ptr()``), the stream defaults to
PyTorch's current stream, and a negative return code raises ``MoeError`` with
the library's message.  All compute runs in the library's CUDA kernels: there
is no fallback of any kind, and calling into a missing or unbuilt library
raises immediately.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe.so")

F32, BF16, F16 = 0, 1, 2
OK = 0
ERR_ARG, ERR_DTYPE, ERR_UNSUPPORTED, ERR_ALIGN, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = (
    -1, -2, -3, -4, -5, -6, -7)
STATUS_TIMEOUT, STATUS_BAD_ID = 1, 2
KID = {
    "route_logits": 0, "route_topk": 1, "permute_count": 2, "permute_scan": 3,
    "permute_place": 4, "permute_gather": 5, "gemm_gateup": 6, "gemm_down": 7, "combine": 8,
    "combine_gate": 9, "shared_gate": 10, "gate_sigmoid": 11, "permute_small": 12,
    "quant_act": 13, "gemm_q": 14, "gemm_q_gateup": 15, "gemm_q_down": 16, "dequant_q": 17,
    "exp_sigmoid": 18,
}
KID_COUNT = 20
QFMT_Q8_0, QFMT_Q4_K = 1, 2

EXPORTS = (
    "moe_last_error", "moe_abi_version", "moe_route_topk", "moe_route_topk_workspace_size",
    "moe_permute", "moe_permute_workspace_size", "moe_permute_noalloc",
    "moe_grouped_gemm_gateup_silu_bf16",
    "moe_grouped_gemm_down_bf16", "moe_grouped_gemm_workspace_size", "moe_combine",
    "moe_combine_gate", "shared_expert_gate", "moe_device_status", "moe_launch_counts",
    "moe_set_gemm_pairing", "moe_gate_workspace_size", "moe_set_pdl", "moe_set_wait_limit_ns",
    "moe_grouped_gemm_gateup_silu_bf16_shared", "moe_grouped_gemm_down_bf16_shared",
    "moe_route_topk_ex", "moe_grouped_gemm_gateup_silu_fp8w", "moe_grouped_gemm_down_fp8w",
    "moe_quantize_act_q8", "moe_grouped_gemm_q", "moe_grouped_gemm_gateup_silu_q",
    "moe_grouped_gemm_down_q", "moe_dequantize_q_bf16", "moe_exp_sigmoid_f32",
    "moe_grouped_gemm_gateup_silu_bf16_staged", "moe_gateup_staged_workspace_size",
)


class MoeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t

_SIGS = {
    "moe_last_error": ([], ctypes.c_char_p),
    "moe_abi_version": ([], _I),
    "moe_route_topk": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _SZ,
                        _P], _I),
    "moe_route_topk_workspace_size": ([_I, _I, _I], _SZ),
    "moe_route_topk_ex": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P,
                           _P, _P, _P, _SZ, _P], _I),
    "moe_permute": ([_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P], _I),
    "moe_permute_workspace_size": ([_I, _I, _I], _SZ),
    "moe_permute_noalloc": ([_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P], _I),
    "moe_grouped_gemm_gateup_silu_bf16": ([_P, _I, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P, _SZ,
                                           _P], _I),
    "moe_grouped_gemm_gateup_silu_bf16_staged": ([_P, _I, _P, _I, _P, _P, _P, _I, _I, _I, _I, _P,
                                                  _P, _SZ, _P], _I),
    "moe_gateup_staged_workspace_size": ([_I], _SZ),
    "moe_grouped_gemm_down_bf16": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _SZ, _P], _I),
    "moe_grouped_gemm_workspace_size": ([_I, _I, _I, _I], _SZ),
    "moe_grouped_gemm_gateup_silu_fp8w": ([_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _SZ, _P], _I),
    "moe_grouped_gemm_down_fp8w": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _SZ, _P],
                                   _I),
    "moe_grouped_gemm_gateup_silu_bf16_shared": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _I, _P,
                                                  _I, _P, _P, _SZ, _P], _I),
    "moe_grouped_gemm_down_bf16_shared": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _I, _P,
                                           _I, _P, _P, _SZ, _P], _I),
    "moe_quantize_act_q8": ([_P, _I, _I, _I, _P, _P, _P], _I),
    "moe_grouped_gemm_q": ([_P, _P, _I, _P, _I, _P, _I, _P, _I, _I, _I, _I, _P, _P], _I),
    "moe_grouped_gemm_gateup_silu_q": ([_P, _P, _I, _P, _I, _P, _I, _P, _I, _I, _I, _I, _P, _P],
                                       _I),
    "moe_grouped_gemm_down_q": ([_P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _I, _P, _P], _I),
    "moe_dequantize_q_bf16": ([_P, _I, ctypes.c_longlong, _I, _P, _P], _I),
    "moe_set_gemm_pairing": ([_I], _I),
    "moe_set_pdl": ([_I], _I),
    "moe_set_wait_limit_ns": ([ctypes.c_ulonglong], _I),
    "moe_combine": ([_P, _I, _P, _P, _I, _F, _I, _I, _I, _P, _I, _P], _I),
    "moe_combine_gate": ([_P, _I, _P, _P, _I, _P, _F, _I, _I, _I, _P, _I, _P, _SZ, _P], _I),
    "shared_expert_gate": ([_P, _I, _P, _I, _I, _P, _I, _P, _SZ, _P], _I),
    "moe_gate_workspace_size": ([_I], _SZ),
    "moe_device_status": ([ctypes.POINTER(_I), _I], _I),
    "moe_exp_sigmoid_f32": ([ctypes.c_uint32, ctypes.c_longlong, _P, _P, _P], _I),
    "moe_launch_counts": ([ctypes.POINTER(ctypes.c_ulonglong), _I], _I),
}


def lib() -> ctypes.CDLL:
    """The loaded libmoe.so.  Raises if it has not been built (see build.py)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"libmoe.so is not built at {LIB_PATH}; run "
                "`python -c 'import __graft_entry__ as g; g.build()'` first")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int) -> int:
    if rc < 0:
        raise MoeError(rc, lib().moe_last_error().decode(errors="replace"))
    return rc


def last_error() -> str:
    return lib().moe_last_error().decode(errors="replace")


def abi_version() -> int:
    return lib().moe_abi_version()


# ------------------------------------------------------------------ entry points
def moe_route_topk(x, w_router, logit_bias, w_shared_gate, logits_in, T, H, E, K, renormalize,
                   scoring, n_group, topk_ids, topk_w, logits_out, gate_logit_out, workspace,
                   ws_bytes, stream=None, check=True):
    rc = lib().moe_route_topk(_ptr(x), _ptr(w_router), _ptr(logit_bias), _ptr(w_shared_gate),
                              _ptr(logits_in), T, H, E, K, renormalize, scoring, n_group,
                              _ptr(topk_ids), _ptr(topk_w), _ptr(logits_out),
                              _ptr(gate_logit_out), _ptr(workspace), ws_bytes, _stream(stream))
    return _check(rc) if check else rc


def moe_route_topk_ex(x, w_router, logit_bias, select_bias, w_shared_gate, logits_in, T, H, E,
                      K, renormalize, scoring, n_group, topk_group, group_score, topk_ids, topk_w,
                      logits_out, gate_logit_out, workspace, ws_bytes, stream=None, check=True):
    """Grouped / sigmoid / bias-corrected router (see moe.h)."""
    rc = lib().moe_route_topk_ex(_ptr(x), _ptr(w_router), _ptr(logit_bias), _ptr(select_bias),
                                 _ptr(w_shared_gate), _ptr(logits_in), T, H, E, K, renormalize,
                                 scoring, n_group, topk_group, group_score, _ptr(topk_ids),
                                 _ptr(topk_w), _ptr(logits_out), _ptr(gate_logit_out),
                                 _ptr(workspace), ws_bytes, _stream(stream))
    return _check(rc) if check else rc


def moe_route_topk_workspace_size(T, E, K) -> int:
    return lib().moe_route_topk_workspace_size(T, E, K)


def moe_permute(topk_ids, x, T, K, E, H, expert_offsets, sorted_pair, pair_to_row, x_perm,
                workspace, ws_bytes, stream=None, check=True):
    rc = lib().moe_permute(_ptr(topk_ids), _ptr(x), T, K, E, H, _ptr(expert_offsets),
                           _ptr(sorted_pair), _ptr(pair_to_row), _ptr(x_perm), _ptr(workspace),
                           ws_bytes, _stream(stream))
    return _check(rc) if check else rc


def moe_permute_workspace_size(T, K, E) -> int:
    return lib().moe_permute_workspace_size(T, K, E)


PERMUTE_NOALLOC_MAX_SCRATCH = 1 << 20


def moe_permute_noalloc(topk_ids, x, T, K, E, H, expert_offsets, sorted_pair, pair_to_row, x_perm,
                        stream=None, check=True):
    """moe_permute without a workspace: for callers that cannot allocate device
    memory.  Uses the library's fixed 1 MiB scratch array (see include/moe.h)."""
    rc = lib().moe_permute_noalloc(_ptr(topk_ids), _ptr(x), T, K, E, H, _ptr(expert_offsets),
                                   _ptr(sorted_pair), _ptr(pair_to_row), _ptr(x_perm),
                                   _stream(stream))
    return _check(rc) if check else rc


def moe_gateup_staged_workspace_size(P) -> int:
    return lib().moe_gateup_staged_workspace_size(P)


def moe_grouped_gemm_gateup_silu_bf16_staged(x, T, sorted_pair, K, x_perm, w13, group_offsets, P,
                                             H, I, G, act, workspace, ws_bytes, stream=None,
                                             check=True):
    rc = lib().moe_grouped_gemm_gateup_silu_bf16_staged(
        _ptr(x), T, _ptr(sorted_pair), K, _ptr(x_perm), _ptr(w13), _ptr(group_offsets), P, H, I,
        G, _ptr(act), _ptr(workspace), ws_bytes, _stream(stream))
    return _check(rc) if check else rc


def moe_grouped_gemm_gateup_silu_bf16(a, a_rows, a_row_gather, gather_div, w13, group_offsets, P,
                                      H, I, G, act, workspace=None, ws_bytes=0, stream=None,
                                      check=True):
    rc = lib().moe_grouped_gemm_gateup_silu_bf16(_ptr(a), a_rows, _ptr(a_row_gather), gather_div,
                                                 _ptr(w13), _ptr(group_offsets), P, H, I, G,
                                                 _ptr(act), _ptr(workspace), ws_bytes,
                                                 _stream(stream))
    return _check(rc) if check else rc


def moe_grouped_gemm_down_bf16(act, w2, group_offsets, pair_weight, row_to_pair, P, I, H, G, out,
                               workspace=None, ws_bytes=0, stream=None, check=True):
    rc = lib().moe_grouped_gemm_down_bf16(_ptr(act), _ptr(w2), _ptr(group_offsets),
                                          _ptr(pair_weight), _ptr(row_to_pair), P, I, H, G,
                                          _ptr(out), _ptr(workspace), ws_bytes, _stream(stream))
    return _check(rc) if check else rc


def moe_grouped_gemm_gateup_silu_bf16_shared(a, w13, group_offsets, P, H, I, G, act, xs, Ts,
                                             w13s, Is, acts, workspace=None, ws_bytes=0,
                                             stream=None, check=True):
    """Routed gate/up over x_perm plus the shared expert's gate/up over xs, one launch."""
    rc = lib().moe_grouped_gemm_gateup_silu_bf16_shared(
        _ptr(a), _ptr(w13), _ptr(group_offsets), P, H, I, G, _ptr(act), _ptr(xs), Ts, _ptr(w13s),
        Is, _ptr(acts), _ptr(workspace), ws_bytes, _stream(stream))
    return _check(rc) if check else rc


def moe_grouped_gemm_down_bf16_shared(act, w2, group_offsets, pair_weight, row_to_pair, P, I, H,
                                      G, out, acts, Ts, w2s, Is, sd, workspace=None, ws_bytes=0,
                                      stream=None, check=True):
    """Routed down (weight, scatter) plus the shared expert's down into sd, one launch."""
    rc = lib().moe_grouped_gemm_down_bf16_shared(
        _ptr(act), _ptr(w2), _ptr(group_offsets), _ptr(pair_weight), _ptr(row_to_pair), P, I, H,
        G, _ptr(out), _ptr(acts), Ts, _ptr(w2s), Is, _ptr(sd), _ptr(workspace), ws_bytes,
        _stream(stream))
    return _check(rc) if check else rc


def moe_grouped_gemm_gateup_silu_fp8w(a, w13_e4m3, w13_scale, group_offsets, P, H, I, G, act,
                                      workspace=None, ws_bytes=0, stream=None, check=True):
    """Gate/up GEMM + SiLU-mul with block-scaled FP8 weights (see moe.h)."""
    rc = lib().moe_grouped_gemm_gateup_silu_fp8w(_ptr(a), _ptr(w13_e4m3), _ptr(w13_scale),
                                                 _ptr(group_offsets), P, H, I, G, _ptr(act),
                                                 _ptr(workspace), ws_bytes, _stream(stream))
    return _check(rc) if check else rc


def moe_grouped_gemm_down_fp8w(act, w2_e4m3, w2_scale, group_offsets, pair_weight, row_to_pair,
                               P, I, H, G, out, workspace=None, ws_bytes=0, stream=None,
                               check=True):
    """Down GEMM (routing weight, scatter) with block-scaled FP8 weights (see moe.h)."""
    rc = lib().moe_grouped_gemm_down_fp8w(_ptr(act), _ptr(w2_e4m3), _ptr(w2_scale),
                                          _ptr(group_offsets), _ptr(pair_weight),
                                          _ptr(row_to_pair), P, I, H, G, _ptr(out),
                                          _ptr(workspace), ws_bytes, _stream(stream))
    return _check(rc) if check else rc


def moe_quantize_act_q8(x, R, K, qfmt, codes, scales, stream=None, check=True):
    """8-bit activation blocks of bf16 rows (Q8_0 for qfmt Q8_0, Q8_K for Q4_K; see moe.h)."""
    rc = lib().moe_quantize_act_q8(_ptr(x), R, K, qfmt, _ptr(codes), _ptr(scales),
                                   _stream(stream))
    return _check(rc) if check else rc


def moe_grouped_gemm_q(a_codes, a_scales, a_rows, a_row_gather, gather_div, w, qfmt,
                       group_offsets, P, K, N, G, out, stream=None, check=True):
    """Plain grouped keep-quant matmul, f32 out (see moe.h)."""
    rc = lib().moe_grouped_gemm_q(_ptr(a_codes), _ptr(a_scales), a_rows, _ptr(a_row_gather),
                                  gather_div, _ptr(w), qfmt, _ptr(group_offsets), P, K, N, G,
                                  _ptr(out), _stream(stream))
    return _check(rc) if check else rc


def moe_grouped_gemm_gateup_silu_q(a_codes, a_scales, a_rows, a_row_gather, gather_div, w13,
                                   qfmt, group_offsets, P, H, I, G, act, stream=None,
                                   check=True):
    """Keep-quant gate/up GEMM + SiLU-mul (see moe.h)."""
    rc = lib().moe_grouped_gemm_gateup_silu_q(_ptr(a_codes), _ptr(a_scales), a_rows,
                                              _ptr(a_row_gather), gather_div, _ptr(w13), qfmt,
                                              _ptr(group_offsets), P, H, I, G, _ptr(act),
                                              _stream(stream))
    return _check(rc) if check else rc


def moe_grouped_gemm_down_q(a_codes, a_scales, w2, qfmt, group_offsets, pair_weight,
                            row_to_pair, P, I, H, G, out, stream=None, check=True):
    """Keep-quant down GEMM with the routing weight and the scatter (see moe.h)."""
    rc = lib().moe_grouped_gemm_down_q(_ptr(a_codes), _ptr(a_scales), _ptr(w2), qfmt,
                                       _ptr(group_offsets), _ptr(pair_weight), _ptr(row_to_pair),
                                       P, I, H, G, _ptr(out), _stream(stream))
    return _check(rc) if check else rc


def moe_dequantize_q_bf16(w, qfmt, rows, K, out, stream=None, check=True):
    """Keep-quant weight rows expanded to bf16 (see moe.h)."""
    rc = lib().moe_dequantize_q_bf16(_ptr(w), qfmt, rows, K, _ptr(out), _stream(stream))
    return _check(rc) if check else rc


def moe_grouped_gemm_workspace_size(P, H, I, G) -> int:
    return lib().moe_grouped_gemm_workspace_size(P, H, I, G)


GEMM_AUTO, GEMM_SINGLE, GEMM_PAIR = 0, 1, 2


def moe_set_gemm_pairing(mode: int) -> int:
    """Tiling of the grouped GEMMs (GEMM_AUTO / GEMM_SINGLE / GEMM_PAIR); returns the
    previous mode."""
    return _check(lib().moe_set_gemm_pairing(int(mode)))


def moe_set_wait_limit_ns(ns: int) -> int:
    """Limit of the GEMM pipeline waits in nanoseconds (1000 .. 10**9, default 10**9)."""
    return _check(lib().moe_set_wait_limit_ns(int(ns)))


def moe_set_pdl(enable: bool) -> bool:
    """Programmatic dependent launch on (default) or off for every kernel;
    returns the previous setting."""
    return bool(_check(lib().moe_set_pdl(1 if enable else 0)))


def moe_combine(expert_out, eo_dtype, w, shared, sh_dtype, routed_scale, T, K, H, out, out_dtype,
                stream=None, check=True):
    rc = lib().moe_combine(_ptr(expert_out), eo_dtype, _ptr(w), _ptr(shared), sh_dtype,
                           float(routed_scale), T, K, H, _ptr(out), out_dtype, _stream(stream))
    return _check(rc) if check else rc


def moe_combine_gate(expert_out, eo_dtype, w, sd, sd_dtype, gl, routed_scale, T, K, H, out,
                     out_dtype, workspace=None, ws_bytes=0, stream=None, check=True):
    rc = lib().moe_combine_gate(_ptr(expert_out), eo_dtype, _ptr(w), _ptr(sd), sd_dtype, _ptr(gl),
                                float(routed_scale), T, K, H, _ptr(out), out_dtype,
                                _ptr(workspace), ws_bytes, _stream(stream))
    return _check(rc) if check else rc


def shared_expert_gate(sd, sd_dtype, gl, T, H, out, out_dtype, workspace=None, ws_bytes=0,
                       stream=None, check=True):
    rc = lib().shared_expert_gate(_ptr(sd), sd_dtype, _ptr(gl), T, H, _ptr(out), out_dtype,
                                  _ptr(workspace), ws_bytes, _stream(stream))
    return _check(rc) if check else rc


def moe_gate_workspace_size(T) -> int:
    return lib().moe_gate_workspace_size(T)


def moe_device_status(clear: bool = False) -> int:
    v = _I(0)
    _check(lib().moe_device_status(ctypes.byref(v), 1 if clear else 0))
    return v.value


def moe_exp_sigmoid_f32(first_bits, n, exp_out, sigmoid_out, stream=None, check=True):
    """The library's binary32 exp and sigmoid on bit patterns first_bits .. + n - 1."""
    rc = lib().moe_exp_sigmoid_f32(int(first_bits) & 0xFFFFFFFF, int(n), _ptr(exp_out),
                                   _ptr(sigmoid_out), _stream(stream))
    return _check(rc) if check else rc


def moe_launch_counts() -> list[int]:
    buf = (ctypes.c_ulonglong * KID_COUNT)()
    n = _check(lib().moe_launch_counts(buf, KID_COUNT))
    return [int(buf[i]) for i in range(n)]
