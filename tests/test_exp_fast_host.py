"""The library's binary32 table-driven exp (exp_fast_f32 in csrc/moe_common.cuh),
compiled for the host, against the oracle's binary32 exp (CPU).  Wherever the
fast form decides, its bits equal the oracle's; it declines NaN, the inputs
outside [-86, 88] and those whose value lies within 2^-16 ulp of a rounding
midpoint.  Inputs: every 131st binary32 pattern of [-86, 88], the 13 inputs of
that range on which a version without the midpoint margin rounds the wrong way
(found by an exhaustive host run over all 2,237,399,042 of them), and special
values."""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "exp_fast_host.cu")
HDR = os.path.join(ROOT, "mixture_experts_ffn_renorm_gb300", "csrc", "moe_common.cuh")
LIB = os.path.join(ROOT, "_build", "libexp_fast_host.so")


# the inputs of [-86, 88] where the binary32 pair, taken without the margin, rounds
# differently from the defined exp (exhaustive host run)
NEAR_MIDPOINT = [
    "-0x1.03d5bep+0", "-0x1.7acc62p+3", "-0x1.c1c4b8p-10", "-0x1.d2259ap+3",
    "-0x1.e1dbe2p-8", "0x1.112856p+6", "0x1.5ffc5cp-6", "0x1.62b666p+1", "0x1.747de2p-15",
    "0x1.8d7cb6p-12", "0x1.c1141cp-7", "0x1.cb763ap-12", "0x1p-24"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return None


@pytest.fixture(scope="module")
def fast():
    cc = _nvcc()
    if cc is None:
        pytest.skip("nvcc not found")
    stale = not os.path.exists(LIB) or os.path.getmtime(LIB) < max(
        os.path.getmtime(SRC), os.path.getmtime(HDR))
    if stale:
        os.makedirs(os.path.dirname(LIB), exist_ok=True)
        subprocess.check_call([cc, "-O2", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                               "-Xcompiler", "-ffp-contract=off",
                               "-I", os.path.join(ROOT, "include"),
                               "-I", os.path.dirname(HDR), SRC, "-o", LIB])
    lib = ctypes.CDLL(LIB)
    fn = lib.exp_fast_host_batch
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_longlong]
    fn.restype = None

    def run(x):
        x = np.ascontiguousarray(x, dtype=np.float32)
        y = np.empty_like(x)
        ok = np.empty(x.shape, np.uint8)
        fn(x.ctypes.data, y.ctypes.data, ok.ctypes.data, x.size)
        return y, ok.astype(bool)

    return run


def _bits(lo, hi, step):
    return np.arange(lo, hi + 1, step, dtype=np.uint64).astype(np.uint32).view(np.float32)


def _same_where_decided(fast, x):
    y, ok = fast(x)
    want = O.exp_f32(x)
    assert np.array_equal(y[ok].view(np.uint32), want[ok].view(np.uint32))
    return ok


def test_fast_exp_equals_the_oracle_on_a_stride_of_the_range(fast):
    top = int(np.float32(88.0).view(np.uint32))
    bottom = int(np.float32(-86.0).view(np.uint32))
    decided = total = 0
    for lo, hi in ((0, top), (0x80000000, bottom)):
        for start in range(lo, hi + 1, 131 * 2**22):      # chunks of 2^22 inputs
            x = _bits(start, min(hi, start + 131 * 2**22 - 1), 131)
            ok = _same_where_decided(fast, x)
            decided += int(ok.sum())
            total += x.size
    assert total > 17_000_000
    assert decided >= total - total // 20_000             # declines about 7 in a million


def test_fast_exp_near_midpoints_and_special_values(fast):
    near = np.array([float.fromhex(v) for v in NEAR_MIDPOINT], np.float32)
    y, ok = fast(near)
    assert not ok.any()   # each lies within 2^-16 ulp of a midpoint: the fast form declines
    special = np.array([np.nan, np.inf, -np.inf, 88.5, -86.5, 1e30, -1e30], np.float32)
    y, ok = fast(special)
    assert not ok.any()
    exact = np.array([0.0, -0.0, 1e-30, -1e-30, 2.0**-149], np.float32)
    y, ok = fast(exact)
    assert ok.all() and np.all(y == 1.0)
    _same_where_decided(fast, np.array([-86.0, 88.0, 1.0, -1.0, 0.5, 10.0, -10.0], np.float32))
