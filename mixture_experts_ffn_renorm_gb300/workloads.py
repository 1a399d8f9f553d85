"""Seeded synthetic inputs for the MoE expert block.

This module only draws random numbers and lays them out; it holds none of the
block's arithmetic (no routing, no softmax, no GEMM, no rounding rule of the
method).  Both the GPU path and the CPU oracle consume the arrays it returns,
which is the only thing the two sides share.

Layout conventions (row-major everywhere):
  x           bf16 [T, H]         tokens
  w_router    bf16 [E, H]         router weight
  logit_bias  f32  [E] or None    additive router-logit bias (skewed load)
  w13         bf16 [E, 2I, H]     per-expert gate rows 0..I-1, up rows I..2I-1
  w2          bf16 [E, H, I]      per-expert down projection
  w_shared_gate bf16 [H] or None  shared-expert sigmoid-gate weight
  w13_shared  bf16 [1, 2Is, H]    shared expert gate/up
  w2_shared   bf16 [1, H, Is]     shared expert down
bf16 arrays are numpy ``uint16`` holding bf16 bit patterns.

Recipe: every tensor is drawn from its own stream ``default_rng([seed, tag,
chunk])`` (PCG64 through a SeedSequence), in chunks of 2**22 values, as f32
standard normals scaled by the tensor's standard deviation and converted to
bf16 by PyTorch's CPU round-to-nearest-even cast.  Chunked streams make the
result independent of the number of threads that fill them.
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

CHUNK = 1 << 22

# stream tags: one per tensor, fixed forever so that inputs never change
TAG_X, TAG_WR, TAG_W13, TAG_W2, TAG_WSG, TAG_W13S, TAG_W2S, TAG_RANK = 1, 2, 3, 4, 5, 6, 7, 8
TAG_EO, TAG_LOGITS, TAG_SD, TAG_GL = 11, 12, 13, 14
TAG_X_RANK = 1000  # + rank: the tokens of data-parallel replica `rank`
TAG_W13Q, TAG_W2Q, TAG_W13S_Q = 21, 22, 23  # keep-quant expert weights (random valid blocks)

# keep-quant weight formats: (weights per block, bytes per block, bytes of
# fp16 scale fields at the block's start); the remaining bytes of a block
# (int8 codes, resp. packed 6-bit scales/mins and 4-bit codes) are free bits
# in which every pattern is a valid block
Q_FORMATS = {"q8_0": (1, 32, 34, 1), "q4_k": (2, 256, 144, 2)}  # name: (id, block, bytes, fp16s)


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    H: int
    I: int
    E: int
    K: int
    I_shared: int = 0          # 0: no shared expert
    zipf_s: float = 0.0        # >0: router logits biased towards a Zipf(s) expert load
    seed: int = 0

    @property
    def P(self) -> int:
        return self.T * self.K


@dataclasses.dataclass(frozen=True)
class CombineConfig:
    name: str
    T: int
    K: int
    H: int
    E_logits: int = 128
    gl_std: float = 2.0
    seed: int = 0


# The five workloads of the block.  The first is the tiny case the oracle
# finishes instantly; the combine-only one streams [T, K, H] expert outputs.
TINY = LayerConfig("tiny_T4_H64_I32_E8_K2_shared32", T=4, H=64, I=32, E=8, K=2, I_shared=32)
COMBINE = CombineConfig("combine_gate_T4096_K8_H2048", T=4096, K=8, H=2048)
DECODE = LayerConfig("decode_T16_H2048_I768_E128_K8", T=16, H=2048, I=768, E=128, K=8)
PREFILL = LayerConfig("prefill_zipf1.1_T8192_H2048_I768_E128_K8", T=8192, H=2048, I=768, E=128,
                      K=8, zipf_s=1.1)
LARGE = LayerConfig("large_shared_T2048_H4096_I1024_E256_K8_Is1024", T=2048, H=4096, I=1024,
                    E=256, K=8, I_shared=1024)

LAYER_CONFIGS = {c.name: c for c in (TINY, DECODE, PREFILL, LARGE)}


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def normal_f32(seed: int, tag: int, n: int, std: float) -> np.ndarray:
    """n f32 normals N(0, std^2) from the chunked stream (seed, tag)."""
    out = np.empty(n, np.float32)
    nchunks = (n + CHUNK - 1) // CHUNK

    def fill(c: int) -> None:
        lo = c * CHUNK
        hi = min(n, lo + CHUNK)
        rng = np.random.default_rng([seed, tag, c])
        rng.standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])
        if std != 1.0:
            out[lo:hi] *= np.float32(std)

    if nchunks <= 1:
        for c in range(nchunks):
            fill(c)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(nchunks)))
    return out


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """f32 -> bf16 bit patterns through PyTorch's CPU cast (round to nearest even)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def normal_bf16(seed: int, tag: int, shape, std: float) -> np.ndarray:
    """Same values as to_bf16_bits(normal_f32(...)), converted chunk by chunk."""
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    nchunks = (n + CHUNK - 1) // CHUNK

    def fill(c: int) -> None:
        lo = c * CHUNK
        hi = min(n, lo + CHUNK)
        tmp = np.empty(hi - lo, np.float32)
        np.random.default_rng([seed, tag, c]).standard_normal(hi - lo, dtype=np.float32, out=tmp)
        if std != 1.0:
            tmp *= np.float32(std)
        out[lo:hi] = to_bf16_bits(tmp)

    if nchunks <= 1:
        for c in range(nchunks):
            fill(c)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.reshape(shape)


def zipf_logit_bias(cfg: LayerConfig) -> np.ndarray | None:
    """Additive router-logit bias that skews top-1 load towards Zipf(s).

    Router logits x.Wr have standard deviation sigma = 0.02*sqrt(H).  Treating
    them as Gumbel noise of the same variance (scale beta = sigma*sqrt(6)/pi),
    adding beta*ln(p_e) makes expert e win with probability ~ p_e; with
    p_e ~ rank(e)^-s the bias is -s*beta*ln(rank(e)).  rank is a seeded
    permutation of 1..E, so the heavy experts are scattered over the ids.
    """
    if cfg.zipf_s <= 0.0:
        return None
    beta = 0.02 * math.sqrt(cfg.H) * math.sqrt(6.0) / math.pi
    rank = np.random.default_rng([cfg.seed, TAG_RANK]).permutation(cfg.E) + 1
    return (-cfg.zipf_s * beta * np.log(rank.astype(np.float64))).astype(np.float32)


def layer_inputs(cfg: LayerConfig, with_weights: bool = True) -> dict:
    """All inputs of one MoE layer as host arrays (see the module docstring)."""
    s, T, H, I, E = cfg.seed, cfg.T, cfg.H, cfg.I, cfg.E
    d = {
        "x": normal_bf16(s, TAG_X, (T, H), 1.0),
        "w_router": normal_bf16(s, TAG_WR, (E, H), 0.02),
        "logit_bias": zipf_logit_bias(cfg),
        "w_shared_gate": None,
        "w13_shared": None,
        "w2_shared": None,
    }
    if with_weights:
        d["w13"] = normal_bf16(s, TAG_W13, (E, 2 * I, H), 0.02)
        d["w2"] = normal_bf16(s, TAG_W2, (E, H, I), 0.02)
    if cfg.I_shared > 0:
        Is = cfg.I_shared
        d["w_shared_gate"] = normal_bf16(s, TAG_WSG, (H,), 0.02)
        d["w13_shared"] = normal_bf16(s, TAG_W13S, (1, 2 * Is, H), 0.02)
        d["w2_shared"] = normal_bf16(s, TAG_W2S, (1, H, Is), 0.02)
    return d


def quantize_fp8_block(w_bits: np.ndarray):
    """Block-scaled FP8 copy of bf16 weights [G, R, C] (input preparation for the
    FP8-weight workloads): per 128 x 128 block, scale = max|w| / 448 (1 for an
    all-zero block) and code = E4M3(w / scale), rounded to nearest even by
    torch's float8_e4m3fn cast.  Returns (codes uint8 [G, R, C], scales f32
    [G, ceil(R/128), ceil(C/128)])."""
    import torch

    G, R, C = w_bits.shape
    rb, cb = (R + 127) // 128, (C + 127) // 128
    w = torch.from_numpy(bf16_bits_to_f32(w_bits))
    pad = torch.zeros((G, rb * 128, cb * 128), dtype=torch.float32)
    pad[:, :R, :C] = w
    blocks = pad.view(G, rb, 128, cb, 128)
    amax = blocks.abs().amax(dim=(2, 4))
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (blocks / scale[:, :, None, :, None]).to(torch.float8_e4m3fn)
    codes = q.view(torch.uint8).view(G, rb * 128, cb * 128)[:, :R, :C].contiguous()
    return codes.numpy(), scale.numpy().astype(np.float32)


def q_weights(seed: int, tag: int, G: int, R: int, K: int, fmt: str, std: float) -> np.ndarray:
    """Random valid keep-quant weight blocks, uint8 [G, R, (K / block) * bytes].

    Each block's free bytes are uniform random bytes.  Its fp16 scale fields
    are drawn so that the weights have a standard deviation near `std`:
    Q8_0 d = std/74 * U(0.8, 1.2) (uniform int8 codes have sd ~74); Q4_K
    d = std/240 * U(0.8, 1.2) and dmin = 7.5 d * U(0.8, 1.2), which centres
    d*sc*q - dmin*m for uniform 6-bit sc, m and 4-bit q.  The stream is
    chunked by 2**20 blocks, (seed, tag, chunk), like the bf16 tensors.
    """
    _, blk, bb, n16 = Q_FORMATS[fmt]
    if K % blk:
        raise ValueError(f"K={K} is not a multiple of the {fmt} block ({blk})")
    nblk = G * R * (K // blk)
    out = np.empty((nblk, bb), np.uint8)
    step = 1 << 20

    def fill(c: int) -> None:
        lo, hi = c * step, min(nblk, (c + 1) * step)
        rng = np.random.default_rng([seed, tag, c])
        out[lo:hi] = rng.integers(0, 256, size=(hi - lo, bb), dtype=np.uint8)
        u = rng.uniform(0.8, 1.2, size=(hi - lo, 2))
        if fmt == "q8_0":
            d = (std / 74.0) * u[:, 0]
            scales = d[:, None]
        else:
            d = (std / 240.0) * u[:, 0]
            scales = np.stack([d, 7.5 * d * u[:, 1]], axis=1)
        out[lo:hi, :2 * n16] = scales.astype(np.float16).view(np.uint8).reshape(hi - lo, 2 * n16)

    n = (nblk + step - 1) // step
    if n <= 1:
        for c in range(n):
            fill(c)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(n)))
    return out.reshape(G, R, (K // blk) * bb)


def layer_q_weights(cfg: LayerConfig, fmt: str) -> dict:
    """Keep-quant expert weights of a layer: w13q [E, 2I, H/blk*bytes], w2q [E, H, I/blk*bytes]."""
    return {
        "w13q": q_weights(cfg.seed, TAG_W13Q, cfg.E, 2 * cfg.I, cfg.H, fmt, 0.02),
        "w2q": q_weights(cfg.seed, TAG_W2Q, cfg.E, cfg.H, cfg.I, fmt, 0.02),
    }


def rank_tokens(cfg: LayerConfig, rank: int) -> np.ndarray:
    """Tokens of data-parallel replica `rank` (rank 0 has the workload's own x)."""
    if rank == 0:
        return normal_bf16(cfg.seed, TAG_X, (cfg.T, cfg.H), 1.0)
    return normal_bf16(cfg.seed, TAG_X_RANK + rank, (cfg.T, cfg.H), 1.0)


def combine_inputs(cfg: CombineConfig) -> dict:
    """Inputs of the combine/gate workload.

    ``logits`` [T, E_logits] f32 ~ N(0,1) are router logits; the routing
    weights of the workload are their renormalised softmax top-K, which the
    caller computes with the router under test (or the oracle's router).
    """
    s, T, K, H = cfg.seed, cfg.T, cfg.K, cfg.H
    return {
        "expert_out": normal_bf16(s, TAG_EO, (T, K, H), 1.0),
        "logits": normal_f32(s, TAG_LOGITS, T * cfg.E_logits, 1.0).reshape(T, cfg.E_logits),
        "sd": normal_bf16(s, TAG_SD, (T, H), 1.0),
        "gl": normal_f32(s, TAG_GL, T, cfg.gl_std),
    }


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (a shift), for inspecting inputs."""
    return (np.ascontiguousarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)
