"""The C-ABI library builds for sm_103a, loads without a GPU and exports every
entry point include/moe.h declares; argument checks that fail before any CUDA
call are exercised here (no compute without a GPU)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import mixture_experts_ffn_renorm_gb300 as m
from mixture_experts_ffn_renorm_gb300 import build as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            for mt in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                                  src, flags=re.M):
                names.add(mt.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return m.lib()


def test_every_declared_symbol_is_exported(lib):
    declared = _declared()
    assert {"moe_route_topk", "moe_permute", "moe_grouped_gemm_gateup_silu_bf16",
            "moe_grouped_gemm_down_bf16", "moe_combine", "moe_combine_gate",
            "shared_expert_gate", "moe_last_error"} <= declared
    raw = ctypes.CDLL(m.LIB_PATH)
    for name in sorted(declared):
        assert hasattr(raw, name), f"{name} declared in include/ but not exported"
    assert set(m.EXPORTS) <= declared


def test_abi_version_and_refusals_without_gpu(lib):
    assert m.abi_version() == 10
    # dtype refusals name the missing arm and return before touching the device
    rc = lib.moe_combine(None, m.F16, None, None, m.BF16, 1.0, 1, 1, 8, None, m.BF16, None)
    assert rc == m.ERR_DTYPE and "f16" in m.last_error()
    rc = lib.shared_expert_gate(None, m.BF16, None, 1, 8, None, 7, None, 0, None)
    assert rc == m.ERR_DTYPE
    rc = lib.moe_route_topk(None, None, None, None, None, 1, 8, 8, 2, 1, 1, 1, None, None, None,
                            None, None, 0, None)
    assert rc == m.ERR_UNSUPPORTED and "softmax" in m.last_error()
    rc = lib.moe_route_topk(None, None, None, None, None, 1, 8, 8, 2, 1, 0, 4, None, None, None,
                            None, None, 0, None)
    assert rc == m.ERR_UNSUPPORTED
    rc = lib.moe_permute(None, None, 1, 0, 8, 8, None, None, None, None, None, 0, None)
    assert rc == m.ERR_ARG
    rc = lib.moe_grouped_gemm_down_bf16(None, None, None, None, None, 4, 60, 64, 1, None, None, 0,
                                        None)
    assert rc == m.ERR_ALIGN
    # T = 0 is a legal no-op for the stream ops
    assert lib.moe_combine(None, m.BF16, None, None, m.BF16, 1.0, 0, 2, 8, None, m.BF16, None) == 0


def test_process_switches(lib):
    # launch-mode switches are host-side state: they return the previous value
    # and refuse values outside their range without touching the device
    prev = m.moe_set_pdl(False)
    assert prev is True                       # on by default
    assert m.moe_set_pdl(True) is False
    assert lib.moe_set_pdl(2) == m.ERR_ARG and "enable" in m.last_error()
    assert m.moe_set_gemm_pairing(m.GEMM_PAIR) == m.GEMM_AUTO     # the default
    assert m.moe_set_gemm_pairing(m.GEMM_SINGLE) == m.GEMM_PAIR
    assert m.moe_set_gemm_pairing(m.GEMM_AUTO) == m.GEMM_SINGLE
    assert lib.moe_set_gemm_pairing(7) == m.ERR_ARG
    # the tilings measured slower and removed are refused by name
    for mode in (3, 4):
        assert lib.moe_set_gemm_pairing(mode) == m.ERR_UNSUPPORTED
    # the pipeline wait limit: 1 us .. 1 s
    assert lib.moe_set_wait_limit_ns(999) == m.ERR_ARG and "outside" in m.last_error()
    assert lib.moe_set_wait_limit_ns(2 * 10**9) == m.ERR_ARG
    assert m.moe_set_wait_limit_ns(10**9) == m.OK


def test_workspace_queries(lib):
    assert m.moe_route_topk_workspace_size(8192, 128, 8) >= 8192 * 128 * 4
    assert m.moe_permute_workspace_size(8192, 8, 128) >= (65536 // 512) * 128 * 4
    assert m.moe_permute_workspace_size(0, 8, 128) == 0
    assert m.moe_grouped_gemm_workspace_size(65536, 2048, 768, 128) == 0


def test_newer_entry_points_refuse_without_touching_the_device(lib):
    # argument checks of the fused shared-expert GEMMs, the extended router and
    # the FP8-weight GEMMs all fail before any CUDA call
    import ctypes
    I, Z = ctypes.c_int, ctypes.c_size_t(0)
    # fused shared expert: I_shared not a multiple of 8
    rc = lib.moe_grouped_gemm_gateup_silu_bf16_shared(None, None, None, 0, 64, 64, 1, None, None,
                                                      4, None, 36, None, None, Z, None)
    assert rc == m.ERR_ALIGN and "I_shared" in m.last_error()
    # fused shared expert: shared rows without operands
    rc = lib.moe_grouped_gemm_down_bf16_shared(None, None, None, None, None, 0, 64, 64, 1, None,
                                               None, 4, None, 64, None, None, Z, None)
    assert rc == m.ERR_ARG
    # extended router: scoring 2, a bias with softmax, a group count that does not divide E
    rc = lib.moe_route_topk_ex(None, None, None, None, None, None, 1, 8, 16, 2, 1, 2, 1, 1, 0,
                               None, None, None, None, None, Z, None)
    assert rc == m.ERR_UNSUPPORTED and "scoring" in m.last_error()
    bias = (ctypes.c_float * 16)()
    rc = lib.moe_route_topk_ex(None, None, None, bias, None, None, 1, 8, 16, 2, 1, 0, 1, 1, 0,
                               None, None, None, None, None, Z, None)
    assert rc == m.ERR_UNSUPPORTED and "sigmoid" in m.last_error()
    rc = lib.moe_route_topk_ex(None, None, None, None, None, None, 1, 8, 16, 2, 1, 1, 3, 1, 0,
                               None, None, None, None, None, Z, None)
    assert rc == m.ERR_ARG and "n_group" in m.last_error()
    # plain router points at the extended entry for grouped routing
    rc = lib.moe_route_topk(None, None, None, None, None, 1, 8, 16, 2, 1, 0, 4, None, None, None,
                            None, None, Z, None)
    assert rc == m.ERR_UNSUPPORTED and "moe_route_topk_ex" in m.last_error()
    # FP8 weights: missing scales
    buf = (ctypes.c_uint8 * 4096)()
    addr = (ctypes.addressof(buf) + 15) & ~15
    rc = lib.moe_grouped_gemm_gateup_silu_fp8w(ctypes.c_void_p(addr), ctypes.c_void_p(addr), None,
                                               None, 4, 64, 64, 1, ctypes.c_void_p(addr), None, Z,
                                               None)
    assert rc == m.ERR_ARG and "scales" in m.last_error()


def test_keep_quant_entry_points_refuse_without_touching_the_device(lib):
    # the keep-quant quantizer and GEMMs check format, sizes and alignment first
    import ctypes
    buf = (ctypes.c_uint8 * 4096)()
    a = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)
    assert lib.moe_quantize_act_q8(a, 2, 64, 3, a, a, None) == m.ERR_ARG
    assert "qfmt" in m.last_error()
    assert lib.moe_quantize_act_q8(a, 2, 48, m.QFMT_Q8_0, a, a, None) == m.ERR_ALIGN
    assert lib.moe_quantize_act_q8(a, 2, 64, m.QFMT_Q4_K, a, a, None) == m.ERR_ALIGN
    assert lib.moe_quantize_act_q8(None, 0, 256, m.QFMT_Q4_K, None, None, None) == m.OK
    # K not a multiple of 256, G out of range, NULL offsets with G > 1
    rc = lib.moe_grouped_gemm_q(a, a, 4, None, 1, a, m.QFMT_Q8_0, None, 4, 96, 8, 1, a, None)
    assert rc == m.ERR_ALIGN and "256" in m.last_error()
    rc = lib.moe_grouped_gemm_q(a, a, 4, None, 1, a, m.QFMT_Q4_K, None, 4, 256, 8, 2, a, None)
    assert rc == m.ERR_ARG and "group_offsets" in m.last_error()
    rc = lib.moe_grouped_gemm_gateup_silu_q(a, a, 4, a, 0, a, m.QFMT_Q4_K, None, 4, 256, 8, 1, a,
                                            None)
    assert rc == m.ERR_ARG and "gather_div" in m.last_error()
    rc = lib.moe_grouped_gemm_down_q(a, a, a, 0, None, None, None, 4, 256, 8, 1, a, None)
    assert rc == m.ERR_ARG
    rc = lib.moe_grouped_gemm_down_q(a, a, a, m.QFMT_Q8_0, None, None, None, 4, 256, 8, 1025, a,
                                     None)
    assert rc == m.ERR_ARG
    # weights not 16-byte aligned
    b = ctypes.c_void_p(a.value + 4)
    rc = lib.moe_grouped_gemm_down_q(a, a, b, m.QFMT_Q8_0, None, None, None, 4, 256, 8, 1, a, None)
    assert rc == m.ERR_ALIGN
    # P = 0 is a no-op
    assert lib.moe_grouped_gemm_q(None, None, 0, None, 1, None, m.QFMT_Q8_0, None, 0, 256, 8, 1,
                                  None, None) == m.OK


def test_block_expansion_refuses_without_touching_the_device(lib):
    # the bf16 expansion of keep-quant blocks checks format, sizes and alignment first
    import ctypes
    buf = (ctypes.c_uint8 * 4096)()
    a = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)
    odd = ctypes.c_void_p(a.value + 1)        # 1-byte aligned
    two = ctypes.c_void_p(a.value + 2)        # 2-byte aligned, not 16
    assert lib.moe_dequantize_q_bf16(a, 3, 1, 256, a, None) == m.ERR_ARG
    assert "qfmt" in m.last_error()
    assert lib.moe_dequantize_q_bf16(a, m.QFMT_Q8_0, -1, 32, a, None) == m.ERR_ARG
    assert lib.moe_dequantize_q_bf16(a, m.QFMT_Q8_0, 1, 0, a, None) == m.ERR_ARG
    assert lib.moe_dequantize_q_bf16(a, m.QFMT_Q8_0, 1, 48, a, None) == m.ERR_ALIGN
    assert lib.moe_dequantize_q_bf16(a, m.QFMT_Q4_K, 1, 128, a, None) == m.ERR_ALIGN
    assert lib.moe_dequantize_q_bf16(None, m.QFMT_Q4_K, 1, 256, a, None) == m.ERR_ARG
    assert lib.moe_dequantize_q_bf16(a, m.QFMT_Q4_K, 1, 256, None, None) == m.ERR_ARG
    # Q4_K blocks and the output want 16-byte alignment; Q8_0 blocks only 2-byte
    assert lib.moe_dequantize_q_bf16(two, m.QFMT_Q4_K, 1, 256, a, None) == m.ERR_ALIGN
    assert lib.moe_dequantize_q_bf16(odd, m.QFMT_Q8_0, 1, 32, a, None) == m.ERR_ALIGN
    assert lib.moe_dequantize_q_bf16(a, m.QFMT_Q8_0, 1, 32, two, None) == m.ERR_ALIGN
    # no rows is a no-op, whatever the pointers
    assert lib.moe_dequantize_q_bf16(None, m.QFMT_Q8_0, 0, 32, None, None) == m.OK


def test_staged_gateup_checks_arguments_without_touching_the_device(lib):
    # the gate/up entry with staged rows: workspace size, then every refusal that
    # happens before a launch
    import ctypes
    buf = (ctypes.c_uint8 * 8192)()
    a = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)
    odd = ctypes.c_void_p(a.value + 2)
    # a 256-byte control block, then one flag per 16 rows padded to 256 bytes
    assert lib.moe_gateup_staged_workspace_size(0) == 0
    assert lib.moe_gateup_staged_workspace_size(1) == 512
    assert lib.moe_gateup_staged_workspace_size(16 * 64) == 512
    assert lib.moe_gateup_staged_workspace_size(16 * 64 + 1) == 768
    f = lib.moe_grouped_gemm_gateup_silu_bf16_staged
    # P = 0 is a no-op and needs no workspace
    assert f(a, 1, None, 1, None, a, None, 0, 64, 64, 1, a, None, 0, None) == m.OK
    assert f(a, 4, a, 0, a, a, None, 4, 64, 64, 1, a, a, 4096, None) == m.ERR_ARG   # K = 0
    assert "K=0" in m.last_error()
    assert f(a, 0, a, 1, a, a, None, 4, 64, 64, 1, a, a, 4096, None) == m.ERR_ARG   # T = 0
    assert f(a, 4, None, 1, a, a, None, 4, 64, 64, 1, a, a, 4096, None) == m.ERR_ARG
    assert f(a, 4, a, 1, None, a, None, 4, 64, 64, 1, a, a, 4096, None) == m.ERR_ARG
    assert f(a, 4, a, 1, odd, a, None, 4, 64, 64, 1, a, a, 4096, None) == m.ERR_ALIGN
    assert f(a, 4, a, 1, a, a, None, 4, 64, 64, 1, a, a, 256, None) == m.ERR_WORKSPACE
    assert f(a, 4, a, 1, a, a, None, 4, 64, 64, 1, a, None, 4096, None) == m.ERR_WORKSPACE
    assert f(a, 4, a, 1, a, a, None, 4, 64, 64, 2, a, a, 4096, None) == m.ERR_ARG   # G > 1, no offsets
