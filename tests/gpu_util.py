"""Helpers shared by the GPU parity tests: host <-> device moves of bf16 bit
arrays and the comparison metrics the tests state."""
from __future__ import annotations

import math

import numpy as np
import torch

DEV = "cuda:0"


def to_dev(a: np.ndarray) -> torch.Tensor:
    """numpy array -> device tensor with the same bytes (uint16 bf16 bits -> bfloat16)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(DEV)
    return torch.from_numpy(a.copy()).to(DEV)


def to_host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def empty(shape, dtype) -> torch.Tensor:
    return torch.empty(shape, dtype=dtype, device=DEV)


def nmse_maxrel(got: np.ndarray, ref: np.ndarray) -> tuple[float, float]:
    """NMSE and max relative error with a floor of 0.1 * rms(ref) in the
    denominator (keeps near-zero reference elements from dividing by ~0)."""
    got = np.asarray(got, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    den = float(np.sum(ref * ref))
    nmse = float(np.sum((got - ref) ** 2) / den) if den > 0 else float(np.sum((got - ref) ** 2))
    floor = 0.1 * math.sqrt(den / max(ref.size, 1))
    rel = float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), max(floor, 1e-30))))
    return nmse, rel


# the grouped-GEMM tolerance: NMSE <= 1e-5 and max relative error <= 2e-2 against
# the oracle's f32-accumulated bf16 result
GEMM_NMSE = 1e-5
GEMM_MAXREL = 2e-2


def assert_gemm_close(got_bits: np.ndarray, ref_bits: np.ndarray, what: str = "") -> None:
    nmse, rel = nmse_maxrel(bf16_to_f64(got_bits), bf16_to_f64(ref_bits))
    assert nmse <= GEMM_NMSE and rel <= GEMM_MAXREL, f"{what}: NMSE {nmse:.3e}, max rel {rel:.3e}"


def launches():
    import mixture_experts_ffn_renorm_gb300 as m

    torch.cuda.synchronize()
    return m.moe_launch_counts()


def launched_since(before, kid_name: str) -> int:
    import mixture_experts_ffn_renorm_gb300 as m

    return launches()[m.KID[kid_name]] - before[m.KID[kid_name]]
