"""The GPU's binary32 exp and sigmoid against the oracle's on every one of the
2^32 binary32 bit patterns.

PR #509's rework makes the shared-expert gate bit-exact; the router weights
need the same exp.  Both sides define exp as the binary32 rounding of one fixed
double-precision evaluation.  The kernels take that value from a binary32
table-driven form wherever the form decides and from the double chain
elsewhere (moe_exp_sigmoid_f32 evaluates exactly what they call).  Every
finite input, both infinities and every NaN are compared, in 16 chunks of 2^28
patterns: bits equal for every input that is not NaN, NaN for NaN.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mixture_experts_ffn_renorm_gb300 as m
import oracle as O

from .gpu_util import empty, launched_since, launches, to_host

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

CHUNK = 1 << 28


def _compare(what, got, want, x):
    nan_in = np.isnan(x)
    g = got.view(np.uint32)
    w = want.view(np.uint32)
    bad = (g != w) & ~nan_in
    assert not bad.any(), (
        f"{what}: {int(bad.sum())} inputs differ, first at x = {float(x[bad][0])!r} "
        f"(gpu {hex(int(g[bad][0]))}, oracle {hex(int(w[bad][0]))})")
    assert np.all(np.isnan(got[nan_in])), f"{what}: a NaN input gave a number"


def test_exp_and_sigmoid_bit_exact_on_every_binary32_input():
    m.lib()
    e_dev = empty((CHUNK,), torch.float32)
    s_dev = empty((CHUNK,), torch.float32)
    before = launches()
    for c in range((1 << 32) // CHUNK):
        first = c * CHUNK
        m.moe_exp_sigmoid_f32(first, CHUNK, e_dev, s_dev)
        x = np.arange(first, first + CHUNK, dtype=np.uint32).view(np.float32)
        got_e, got_s = to_host(e_dev), to_host(s_dev)
        _compare("exp", got_e, O.exp_f32(x), x)
        _compare("sigmoid", got_s, O.sigmoid_f32_array(x), x)
    assert launched_since(before, "exp_sigmoid") == (1 << 32) // CHUNK
    assert m.moe_device_status() == 0


def test_exp_sigmoid_entry_point_refusals():
    m.lib()
    out = empty((4,), torch.float32)
    with pytest.raises(m.MoeError) as ei:
        m.moe_exp_sigmoid_f32(0, 4, None, None)
    assert ei.value.code == m.ERR_ARG
    with pytest.raises(m.MoeError) as ei:
        m.moe_exp_sigmoid_f32(0, -1, out, None)
    assert ei.value.code == m.ERR_ARG
    # the edges of the range wrap around modulo 2^32: 0xFFFFFFFF (a NaN), then +0
    m.moe_exp_sigmoid_f32(0xFFFFFFFF, 2, out, None)
    h = to_host(out)
    assert np.isnan(h[0]) and h[1] == 1.0
