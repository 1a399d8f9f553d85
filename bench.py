"""Benchmark of the BF16 MoE expert block on GB300.

Default workload: the prefill MoE layer (T=8192 tokens, H=2048, I=768, E=128
experts, top-8 renormalised softmax router with Zipf(1.1)-skewed expert load,
no shared expert).  One step = one full forward of the block: router (logits
GEMM + top-k), permute, grouped gate/up GEMM + SiLU-mul, grouped down GEMM
with routing weight and scatter, combine.  Inputs are synthetic and seeded;
the weights (1.21 GB) exceed the 126 MB L2, so no step finds the previous
step's operands in cache.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config prefill|decode|large] [--no-cpu-baseline]

Under torchrun (N > 1) every rank runs its own replica on its own GPU (the
tokens of a batch are independent: weak scaling, no collective on the data
path); rank 0 prints one JSON line with value = all ranks' tokens / max time.
--impl reference times the CPU oracle (the plain sequential definition of the
block) on this host's cores over a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s on 1 GB300; grouped-GEMM TFLOP/s and combine GB/s vs peak"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def recorded_traffic(workload, weights="bf16"):
    """DRAM traffic of one gate/up GEMM launch on `workload` from the committed
    ncu summary, or None when it covers another workload or the kernel
    sources have changed since it was captured."""
    import hashlib

    if weights == "bf16":
        names = ("gemm_gateup_traffic.txt", "gemm_gateup_traffic_decode.txt",
                 "gemm_gateup_traffic_large.txt")
        srcs = ("moe_gemm.cu", "moe_gemm_pair.cu", "gemm_common.cuh", "sm100_ptx.cuh")
    elif weights in Q_WEIGHTS:
        names, srcs = (f"qgemm_gateup_{weights}_traffic.txt",), ("moe_qgemm.cu", "sm100_ptx.cuh")
    else:
        return None
    kv = {}
    for name in names:  # the record of this workload, if one is committed
        path = os.path.join(ROOT, "profiles", name)
        if not os.path.exists(path):
            continue
        rec = {}
        for ln in open(path):
            if "=" in ln and not ln.startswith("#"):
                k, v = ln.strip().split("=", 1)
                rec[k] = v
        if rec.get("workload") == workload:
            kv = rec
            break
    h = hashlib.sha256()
    for f in srcs:
        with open(os.path.join(ROOT, "mixture_experts_ffn_renorm_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    if kv.get("sources_sha256") != h.hexdigest() or kv.get("workload") != workload:
        return None
    return int(kv["dram_bytes_read"]) + int(kv["dram_bytes_write"])


# keep-quant weight formats: name -> (oracle format id, weights per block, bytes per block)
Q_WEIGHTS = {"q8_0": (1, 32, 34), "q4_k": (2, 256, 144)}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            out = {}
            for k in FALLBACK:
                v = d.get(k)
                if isinstance(v, dict):
                    v = v.get("value")
                out[k] = float(v) if v is not None else FALLBACK[k]
            return out, "measured"
        except Exception:
            pass
    return dict(FALLBACK), "fallback"


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled every 2 ms during the
    timed region, read through NVML (read-only queries); nvidia-smi is the
    fallback when NVML cannot be loaded."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device):
        self.device = device
        self.samples = []
        self.max_mhz = None
        self._stop = False
        self._thread = None
        self._nvml = None
        self._handle = None

    def _open_nvml(self):
        import ctypes

        import torch

        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        p = torch.cuda.get_device_properties(self.device)
        bus = f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0".encode()
        if nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
            cnt = ctypes.c_uint()
            if nv.nvmlDeviceGetCount_v2(ctypes.byref(cnt)) != 0 or cnt.value != 1:
                return False
            if nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)) != 0:
                return False
        mx = ctypes.c_uint()
        if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        self._nvml, self._handle = nv, h
        return True

    def _poll(self):
        import ctypes

        nv, h = self._nvml, self._handle
        mhz = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        get_r = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop:
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0 and \
                    get_r(h, ctypes.byref(rs)) == 0:
                self.samples.append((float(mhz.value), int(rs.value)))
            time.sleep(0.002)

    def __enter__(self):
        import threading

        try:
            ok = self._open_nvml()
        except OSError:
            ok = False
        if ok:
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
            while not self.samples and self._thread.is_alive():
                time.sleep(0.001)
        return self

    def __exit__(self, *exc):
        self._stop = True
        if self._thread is not None:
            self._thread.join(timeout=2)

    def summary(self):
        if not self.samples:
            return None
        reasons = set()
        for _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s for s, _ in self.samples),
                "sm_max_mhz": self.max_mhz, "samples": len(self.samples),
                "reasons": sorted(reasons), "source": "nvml"}


def dist_setup(args):
    from mixture_experts_ffn_renorm_gb300 import dp

    ws, rank, local = dp.world()
    if ws > 1:
        import torch.distributed as dist

        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    from mixture_experts_ffn_renorm_gb300 import dp

    dp.barrier(ws)


def max_over_ranks(v, ws, device):
    from mixture_experts_ffn_renorm_gb300 import dp

    return dp.max_over_ranks(v, ws, device)


def layer_config(name):
    from mixture_experts_ffn_renorm_gb300 import workloads as W

    return {"prefill": W.PREFILL, "decode": W.DECODE, "large": W.LARGE, "tiny": W.TINY}[name]


def config_dict(cfg, ws):
    return {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "I": cfg.I, "E": cfg.E, "K": cfg.K,
            "I_shared": cfg.I_shared, "zipf_s": cfg.zipf_s, "tokens_per_gpu": cfg.T,
            "global_batch": cfg.T * ws, "parallelism": f"dp{ws} (independent replicas)",
            "l2": "operands larger than L2 (weights 1.21 GB > 126 MB), no flush needed"
            if cfg.T >= 8192 else "L2 flushed between steps (256 MB write)"}


def combine_gate_workload(dev, iters=20):
    """The combine/gate bandwidth workload (T=4096, K=8, H=2048): weighted top-8
    sum of bf16 expert rows plus the sigmoid-gated shared term.  `iters`
    back-to-back launches between two CUDA events, alternating between two
    copies of the inputs (2 x 168 MB > L2), so no launch finds its operands in
    L2."""
    import torch

    import mixture_experts_ffn_renorm_gb300 as m
    from mixture_experts_ffn_renorm_gb300 import workloads as W

    cfg = W.COMBINE
    d = W.combine_inputs(cfg)
    T, K, H, E = cfg.T, cfg.K, cfg.H, cfg.E_logits

    def dev_bf16(a):
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(dev)

    eo, sd = dev_bf16(d["expert_out"]), dev_bf16(d["sd"])
    eo2, sd2 = eo.clone(), sd.clone()
    gl = torch.from_numpy(d["gl"]).to(dev)
    logits = torch.from_numpy(d["logits"]).to(dev)
    ids = torch.empty((T, K), dtype=torch.int32, device=dev)
    w = torch.empty((T, K), dtype=torch.float32, device=dev)
    m.moe_route_topk(None, None, None, None, logits, T, 8, E, K, 1, 0, 1, ids, w, None, None, None,
                     0)
    outs = [torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    ws = torch.empty((m.moe_gate_workspace_size(T),), dtype=torch.uint8, device=dev)
    sets = [(eo, sd, outs[0]), (eo2, sd2, outs[1])]

    def launch(i):
        e, s_, o = sets[i % 2]
        m.moe_combine_gate(e, m.BF16, w, s_, m.BF16, gl, 1.0, T, K, H, o, m.BF16, ws, ws.numel())

    for i in range(4):
        launch(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(iters):
        launch(i)
    e1.record()
    torch.cuda.synchronize()
    us = 1000.0 * e0.elapsed_time(e1) / iters
    nbytes = T * K * H * 2 + 2 * T * H * 2 + T * K * 4 + T * 4
    return {"workload": cfg.name, "us": us, "gbs": nbytes / us / 1e3, "bytes": nbytes}


def combine_arms(dev, iters=20):
    """Every dtype arm of the combine/gate and combine ops on the bandwidth
    workload's shape (T=4096, K=8, H=2048, weighted): microseconds and GB/s per
    call, back to back over two input copies (more than L2)."""
    import torch

    import mixture_experts_ffn_renorm_gb300 as m

    T, K, H = 4096, 8, 2048
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    tdt = {m.F32: torch.float32, m.BF16: torch.bfloat16}
    size = {m.F32: 4, m.BF16: 2}
    w = torch.rand((T, K), device=dev, generator=g)
    gl = torch.randn((T,), device=dev, generator=g)
    ws = torch.empty((m.moe_gate_workspace_size(T),), dtype=torch.uint8, device=dev)
    out = {}
    arms = [(m.BF16, m.BF16, m.BF16), (m.F32, m.F32, m.F32), (m.BF16, m.F32, m.F32),
            (m.F32, m.BF16, m.BF16), (m.BF16, m.BF16, m.F32), (m.F32, m.F32, m.BF16)]
    name = {m.F32: "f32", m.BF16: "bf16"}
    for eo_dt, sd_dt, o_dt in arms:
        sets = []
        for _ in range(2):
            eo = torch.randn((T, K, H), device=dev, generator=g).to(tdt[eo_dt])
            sd = torch.randn((T, H), device=dev, generator=g).to(tdt[sd_dt])
            o = torch.empty((T, H), dtype=tdt[o_dt], device=dev)
            sets.append((eo, sd, o))
        for op in ("combine_gate", "combine"):
            def call(i):
                eo, sd, o = sets[i % 2]
                if op == "combine_gate":
                    m.moe_combine_gate(eo, eo_dt, w, sd, sd_dt, gl, 1.0, T, K, H, o, o_dt, ws,
                                       ws.numel())
                else:
                    m.moe_combine(eo, eo_dt, w, sd, sd_dt, 1.0, T, K, H, o, o_dt)
            for i in range(4):
                call(i)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for i in range(iters):
                call(i)
            e1.record()
            torch.cuda.synchronize()
            us = 1000.0 * e0.elapsed_time(e1) / iters
            nbytes = T * K * H * size[eo_dt] + T * H * (size[sd_dt] + size[o_dt]) + T * K * 4
            if op == "combine_gate":
                nbytes += T * 4
            out[f"{op} eo={name[eo_dt]} sd={name[sd_dt]} out={name[o_dt]}"] = {
                "us": us, "gbs": nbytes / us / 1e3, "bytes": nbytes}
        del sets
    return out


def q_dequant_on(args, cfg):
    """Whether keep-quant weights are expanded to bf16 for this run (--q-dequant)."""
    mode = getattr(args, "q_dequant", "auto")
    return mode == "on" or (mode == "auto" and cfg.T * cfg.K > 16 * cfg.E)


def layer_oracle(O, cfg, d, tokens):
    """The oracle's whole block on `tokens`: keep-quant experts when `d` holds
    GGUF blocks (w13q / w2q, format d["qfmt"]), bf16 experts otherwise."""
    if "w13q" in d:
        return O.moe_layer_tokens_q(d["x"], d["w_router"], d["logit_bias"], d["w13q"], d["w2q"],
                                    Q_WEIGHTS[d["qfmt"]][0], d["w_shared_gate"], d["w13_shared"],
                                    d["w2_shared"], H=cfg.H, I=cfg.I, E=cfg.E, K=cfg.K,
                                    I_shared=cfg.I_shared, tokens=tokens)
    return O.moe_layer_tokens(d["x"], d["w_router"], d["logit_bias"], d["w13"], d["w2"],
                              d["w_shared_gate"], d["w13_shared"], d["w2_shared"], H=cfg.H,
                              I=cfg.I, E=cfg.E, K=cfg.K, I_shared=cfg.I_shared, tokens=tokens)


def oracle_tokens_per_s(cfg, d, seconds=10.0):
    """Time the CPU oracle on a bounded sample of the workload's tokens."""
    import oracle as O

    def run(tokens):
        t0 = time.perf_counter()
        layer_oracle(O, cfg, d, np.asarray(tokens, np.int32))
        return time.perf_counter() - t0

    cores = O.max_threads()
    t1 = run(np.arange(min(cores, cfg.T)))
    per_tok = t1 / min(cores, cfg.T)
    n = int(max(min(cores, cfg.T), min(cfg.T, seconds / max(per_tok, 1e-9))))
    dt = run(np.arange(n))
    return n / dt, cores, n, dt


def run_reference(args):
    ws, rank, _ = dist_setup(args)
    if rank != 0:
        return 0
    cfg = layer_config(args.config)
    from mixture_experts_ffn_renorm_gb300 import workloads as W
    from oracle import build as ob

    ob.build()
    weights = getattr(args, "weights", "bf16")
    d = W.layer_inputs(cfg, with_weights=weights not in Q_WEIGHTS)
    import oracle as O

    if weights in Q_WEIGHTS:  # the keep-quant layer on the same GGUF blocks
        d.update(W.layer_q_weights(cfg, weights))
        d["qfmt"] = weights
    if weights == "fp8":  # the layer on the dequantised FP8 weights
        for key, R, C in (("w13", 2 * cfg.I, cfg.H), ("w2", cfg.H, cfg.I)):
            q, sc = W.quantize_fp8_block(d[key])
            d[key] = O.dequant_fp8_block(q, sc, G=cfg.E, R=R, C=C)
    cores = O.max_threads()
    n = max(cores, 8) if cfg.T >= 64 else cfg.T
    tokens = np.arange(n, dtype=np.int32)
    for _ in range(args.warmup if args.warmup < 2 else 1):
        layer_oracle(O, cfg, d, tokens)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        layer_oracle(O, cfg, d, tokens)
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(config_dict(cfg, 1), weights=weights,
                       **({"q_dequant": q_dequant_on(args, cfg)} if weights in Q_WEIGHTS else {})),
        "cpu_baseline": {"kind": "oracle", "cores": cores, "value": value, "unit": "tokens/s",
                         "sample": f"{n} of {cfg.T} tokens per step, full block per token"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_combine_only(args):
    import torch

    import __graft_entry__ as ge

    ge.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pk, pk_src = peaks()
    cg = combine_gate_workload(dev, iters=args.steps)
    arms = combine_arms(dev, iters=args.steps)
    for v in arms.values():
        v["frac_hbm"] = v["gbs"] / pk["hbm_gbs"]
    line = {"metric": "combine/gate GB/s (bandwidth workload)", "value": cg["gbs"], "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": 3, "ms_per_step": cg["us"] / 1000.0,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": {"workload": cg["workload"]},
            "roofline": {"bound": "hbm", "achieved": cg["gbs"], "peak": pk["hbm_gbs"],
                         "unit": "GB/s", "frac": cg["gbs"] / pk["hbm_gbs"],
                         "peak_source": pk_src, "traffic": None},
            "components": {"dtype_arms": arms}}
    print(json.dumps(line), flush=True)
    return 0


def timed_steps(blk, x_dev, steps, flush):
    """Mean step time in ms over `steps` forwards on the current stream.  With a
    flush buffer, L2 is flushed before every step and the flush is left out of
    the time (events at each step's first and last stage); without, the steps
    run back to back with no event between their kernels, so each kernel may
    start under programmatic dependent launch while its predecessor drains."""
    import torch

    step_marks = []
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record()
    for _ in range(steps):
        if flush is not None:
            flush.zero_()
            marks = []
            blk.forward(x_dev, marks=marks, stages=False)
            step_marks.append(marks)
        else:
            blk.forward(x_dev)
    t_end.record()
    torch.cuda.synchronize()
    if flush is None:
        return t_start.elapsed_time(t_end) / steps
    return sum(mk[0][1].elapsed_time(mk[-1][1]) for mk in step_marks) / steps


def stage_breakdown(blk, x_dev, steps, flush):
    """The same steps with an event after every stage: mean ms per stage."""
    import torch

    stage_ms = {}
    for _ in range(steps):
        if flush is not None:
            flush.zero_()
        marks = []
        blk.forward(x_dev, marks=marks)
        for (_, a), (name, b) in zip(marks[:-1], marks[1:]):
            stage_ms.setdefault(name, []).append((a, b))
    torch.cuda.synchronize()
    return {k: sum(a.elapsed_time(b) for a, b in v) / len(v) for k, v in stage_ms.items()}


def gemm_account(cfg, counts, stage_avg, pk, fp8=False, qw=None, qd=False):
    """Algorithmic FLOPs and bytes of the two grouped GEMMs of one forward, their
    rates from the per-stage times, and which roof binds the gate/up GEMM."""
    P = cfg.T * cfg.K
    touched = int((counts > 0).sum())
    flop_gateup = 2.0 * P * cfg.H * 2 * cfg.I
    flop_down = 2.0 * P * cfg.I * cfg.H
    wb = 1 if fp8 else 2          # bytes per expert weight (FP8 adds one f32 per 128x128 block)
    sc = 4.0 / (128 * 128) if fp8 else 0.0
    a_in = 2.0                    # bytes per activation element read by a GEMM
    if qw and not qd:             # GGUF blocks; 8-bit activation codes plus one f32 per block
        _, qblk, qbytes = Q_WEIGHTS[qw]
        wb, sc, a_in = qbytes / qblk, 0.0, 1.0 + 4.0 / qblk
    bytes_gateup = touched * 2 * cfg.I * cfg.H * (wb + sc) + P * cfg.H * a_in + P * cfg.I * 2
    bytes_down = touched * cfg.H * cfg.I * (wb + sc) + P * cfg.I * a_in + P * cfg.H * 2 + P * 4
    if cfg.I_shared:              # the shared expert runs inside the same two launches
        flop_gateup += 2.0 * cfg.T * cfg.H * 2 * cfg.I_shared
        flop_down += 2.0 * cfg.T * cfg.I_shared * cfg.H
        bytes_gateup += 2 * cfg.I_shared * cfg.H * 2 + cfg.T * cfg.I_shared * 2
        bytes_down += cfg.H * cfg.I_shared * 2 + cfg.T * cfg.I_shared * 2 + cfg.T * cfg.H * 2
    t_gu = stage_avg["gemm_gateup"] / 1000.0
    t_dn = stage_avg["gemm_down"] / 1000.0
    qk = bool(qw) and not qd      # the keep-quant kernels run (CUDA cores, against HBM)
    tensor_bound = (not qk and flop_gateup / (pk["bf16_tflops"] * 1e12)
                    >= bytes_gateup / (pk["hbm_gbs"] * 1e9))
    return {
        "touched": touched, "flop_gateup": flop_gateup, "flop_down": flop_down,
        "bytes_gateup": bytes_gateup, "bytes_down": bytes_down, "t_gu": t_gu, "t_dn": t_dn,
        "qk": qk, "tensor_bound": tensor_bound,
        "gemm_gateup_tflops": flop_gateup / t_gu / 1e12,
        "gemm_gateup_gbs": bytes_gateup / t_gu / 1e9,
        "gemm_down_tflops": flop_down / t_dn / 1e12,
        "gemm_down_gbs": bytes_down / t_dn / 1e9,
    }


def extra_layer(name, dev, steps, warmup, pk):
    """One more full-size workload (decode or the large layer) timed like the
    headline one: step time with L2 flushed between steps, per-stage times,
    and each GEMM's rate against the roof that binds it."""
    import torch

    from mixture_experts_ffn_renorm_gb300 import workloads as W
    from mixture_experts_ffn_renorm_gb300.layer import MoeBlock

    cfg = layer_config(name)
    d = W.layer_inputs(cfg)
    blk = MoeBlock(cfg.H, cfg.I, cfg.E, cfg.K, d, max_tokens=cfg.T, device=dev,
                   I_shared=cfg.I_shared, gather="auto")
    x_dev = torch.from_numpy(d["x"].view(np.int16).copy()).view(torch.bfloat16).to(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        blk.forward(x_dev)
    torch.cuda.synchronize()
    step_ms = timed_steps(blk, x_dev, steps, flush)
    # the same steps back to back with no flush: each step's weights (decode: the
    # 85 touched experts' 802 MB) are larger than L2 on their own, as in the
    # headline prefill timing, and no step starts against L2 lines another
    # step left dirty
    step_b2b_ms = timed_steps(blk, x_dev, steps, None)
    stage_avg = stage_breakdown(blk, x_dev, steps, flush)
    counts = np.diff(blk.expert_offsets.cpu().numpy())
    g = gemm_account(cfg, counts, stage_avg, pk)
    out = {"workload": cfg.name, "step_us": 1000.0 * step_ms,
           "tokens_per_s": cfg.T / (step_ms / 1000.0),
           "step_us_back_to_back": 1000.0 * step_b2b_ms,
           "stages_us": {k: 1000.0 * v for k, v in stage_avg.items()},
           "touched_experts": g["touched"],
           "gemm_gateup_gbs": g["gemm_gateup_gbs"], "gemm_down_gbs": g["gemm_down_gbs"],
           "gemm_gateup_frac_hbm": g["gemm_gateup_gbs"] / pk["hbm_gbs"],
           "gemm_down_frac_hbm": g["gemm_down_gbs"] / pk["hbm_gbs"],
           "gemm_gateup_tflops": g["gemm_gateup_tflops"],
           "gemm_down_tflops": g["gemm_down_tflops"],
           "l2": "flushed between steps (256 MB write), flush not timed"}
    del blk, flush, x_dev, d
    torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch

    if args.config == "combine":
        return run_combine_only(args)
    ws, rank, local = dist_setup(args)
    import __graft_entry__ as ge

    if rank == 0 or ws == 1:
        ge.build()
    barrier(ws)
    import mixture_experts_ffn_renorm_gb300 as m
    from mixture_experts_ffn_renorm_gb300 import workloads as W
    from mixture_experts_ffn_renorm_gb300.layer import MoeBlock

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = layer_config(args.config)
    qw = args.weights if args.weights in Q_WEIGHTS else None
    d = W.layer_inputs(cfg, with_weights=qw is None)
    if qw:
        d.update(W.layer_q_weights(cfg, qw))
        d["qfmt"] = qw
    if rank > 0:  # each replica gets its own tokens of the global batch
        d["x"] = W.rank_tokens(cfg, rank)
    # keep-quant weights on prefill-sized batches: expanded to bf16 once and run on
    # the tensor cores (--q-dequant auto picks that above 16 rows per expert)
    qd = bool(qw) and q_dequant_on(args, cfg)
    fp8 = args.weights == "fp8"
    if fp8:
        d["w13_e4m3"], d["w13_scale"] = W.quantize_fp8_block(d["w13"])
        d["w2_e4m3"], d["w2_scale"] = W.quantize_fp8_block(d["w2"])
    # gather="auto": decode-sized calls read their routed rows of x inside the
    # gate/up GEMM; prefill-sized ones stream x_perm
    blk = MoeBlock(cfg.H, cfg.I, cfg.E, cfg.K, d, max_tokens=cfg.T, device=dev,
                   I_shared=cfg.I_shared, fp8_weights=fp8, qweights=qw, q_dequant=qd,
                   gather="auto")
    x_host = torch.from_numpy(d["x"].view(np.int16).copy()).view(torch.bfloat16).pin_memory()
    x_dev = x_host.to(dev)
    out_host = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory()
    flush = None
    if cfg.T < 8192:
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    for _ in range(args.warmup):
        blk.forward(x_dev)
    torch.cuda.synchronize()

    # ---------------- timed: device-resident inputs, whole steps (no events
    # between the kernels of a step, so each may start under programmatic
    # dependent launch while its predecessor drains)
    counts0 = m.moe_launch_counts()
    with ClockSampler(dev) as clk:
        barrier(ws)
        torch.cuda.synchronize()
        step_ms = timed_steps(blk, x_dev, args.steps, flush)
        barrier(ws)
    counts1 = m.moe_launch_counts()
    launches = sum(b - a for a, b in zip(counts0, counts1))
    ms = max_over_ranks(step_ms, ws, dev)
    from mixture_experts_ffn_renorm_gb300 import dp

    value = dp.aggregate_tokens_per_s(cfg.T, ws, ms)

    # ---------------- per-stage breakdown: the same steps with an event after
    # every stage (reported as components; not the headline)
    stage_avg = stage_breakdown(blk, x_dev, args.steps, flush)

    # ---------------- end to end through the public API with host buffers:
    # every step copies its tokens in from pinned host memory and its output
    # back out; MoeBlock.run_host_batches overlaps those copies with compute
    e2e_steps = max(3, args.steps)
    out_hosts = [out_host, torch.empty_like(out_host).pin_memory()]
    blk.run_host_batches([x_host] * 2, out_hosts)  # warm-up of the copy streams
    torch.cuda.synchronize()
    barrier(ws)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    blk.run_host_batches([x_host] * e2e_steps, [out_hosts[i % 2] for i in range(e2e_steps)])
    e1.record()
    torch.cuda.synchronize()
    barrier(ws)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, ws, dev)
    e2e_value = ws * cfg.T / (e2e_ms / 1000.0)

    # ---------------- roofline of the dominant kernel (the gate/up GEMM):
    # tensor-bound when its FLOPs take longer at peak than its bytes at HBM
    # peak (the prefill layer), HBM-bound otherwise (decode, the large layer)
    pk, pk_src = peaks()
    P = cfg.T * cfg.K
    counts = np.diff(blk.expert_offsets.cpu().numpy())
    ga = gemm_account(cfg, counts, stage_avg, pk, fp8=fp8, qw=qw, qd=qd)
    touched, qk, tensor_bound = ga["touched"], ga["qk"], ga["tensor_bound"]
    flop_gateup, flop_down = ga["flop_gateup"], ga["flop_down"]
    bytes_gateup, bytes_down = ga["bytes_gateup"], ga["bytes_down"]
    t_gu, t_dn = ga["t_gu"], ga["t_dn"]
    # which bf16 gate/up kernel runs: the library's default tiling takes CTA-pair
    # tiles for P >= 1024 rows averaging >= 32 per group, unless the shared expert
    # rides in the same launch (single-CTA tiles)
    pair = P >= 1024 and P >= 32 * cfg.E and not cfg.I_shared
    # at most 16 rows per group: 32-row, 128-wide tiles, the routed rows of x
    # gathered inside the launch (the layer is built with gather="auto")
    narrow = P <= 16 * cfg.E
    gathered = bool(qk) or (narrow and not cfg.I_shared and not fp8)
    kname = ("grouped_gemm_kernel<gateup, FP8 weights> (gate/up GEMM + SiLU-mul)" if fp8 else
             f"qgemm_kernel<{qw}, gateup> (keep-quant gate/up + SiLU-mul, dp4a)" if qk else
             "pair_gemm_kernel<gateup> (CTA-pair gate/up GEMM + SiLU-mul)" if pair else
             "grouped_gemm_kernel<128,gateup,gathered,32 rows> (gate/up GEMM + SiLU-mul)"
             if narrow and not cfg.I_shared else
             "grouped_gemm_kernel<256,gateup> (gate/up GEMM + SiLU-mul)")
    traffic_key = "bf16" if qd else args.weights
    if tensor_bound:
        achieved = flop_gateup / t_gu / 1e12
        roofline = {"kernel": kname, "bound": "tensor", "achieved": achieved,
                    "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": achieved / pk["bf16_tflops"],
                    "peak_source": f"{pk_src} bf16 dense (burst)",
                    "traffic": recorded_traffic(cfg.name, traffic_key),
                    "traffic_unit": "bytes per launch (ncu dram read + write)",
                    "algorithmic_flop_per_launch": flop_gateup}
    else:
        achieved = bytes_gateup / t_gu / 1e9
        roofline = {"kernel": kname, "bound": "hbm", "achieved": achieved,
                    "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                    "peak_source": f"{pk_src} HBM copy bandwidth",
                    "traffic": recorded_traffic(cfg.name, traffic_key),
                    "traffic_unit": "bytes per launch (ncu dram read + write)",
                    "algorithmic_bytes_per_launch": bytes_gateup,
                    "touched_experts": touched}
    comb_bytes = P * cfg.H * 2 + cfg.T * cfg.H * 2
    if cfg.I_shared:
        comb_bytes += cfg.T * cfg.H * 2 + cfg.T * 4
    components = {
        "ms": stage_avg,
        "gemm_gateup_tflops": flop_gateup / t_gu / 1e12,
        "gemm_gateup_gbs": bytes_gateup / t_gu / 1e9,
        "gemm_down_tflops": flop_down / t_dn / 1e12,
        "gemm_down_gbs": bytes_down / t_dn / 1e9,
        "gemm_down_frac": (flop_down / t_dn / 1e12 / pk["bf16_tflops"] if tensor_bound
                           else bytes_down / t_dn / 1e9 / pk["hbm_gbs"]),
        "combine_gbs": comb_bytes / (stage_avg["combine"] / 1000.0) / 1e9,
        "combine_frac_hbm": comb_bytes / (stage_avg["combine"] / 1000.0) / 1e9 / pk["hbm_gbs"],
        "route_gbs": (cfg.T * cfg.H * 2 + cfg.E * cfg.H * 2) / (stage_avg["route"] / 1000.0) / 1e9,
        # with gathered rows the permute writes no x_perm (indices only)
        "permute_gbs": ((0 if gathered else 2 * P * cfg.H * 2) + P * 16)
                       / (stage_avg["permute"] / 1000.0) / 1e9,
        "gateup_rows": "gathered from x" if gathered else "x_perm",
        "hbm_peak_gbs": pk["hbm_gbs"],
        "stages_sum_ms": sum(stage_avg.values()),
    }
    cg = combine_gate_workload(dev)
    cg["frac_hbm"] = cg["gbs"] / pk["hbm_gbs"]
    components["combine_gate_workload"] = cg
    components["expert_load"] = {"max": int(counts.max()), "mean": float(counts.mean()),
                                 "min": int(counts.min()), "touched": touched}
    if ws == 1 and args.config == "prefill" and args.weights == "bf16" and not args.no_extra_layers:
        # the other full-size workloads, timed the same way in the same run
        del blk
        torch.cuda.empty_cache()
        for name in ("decode", "large"):
            components[name] = extra_layer(name, dev, args.steps, min(args.warmup, 5), pk)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        do = d
        if fp8:  # the oracle runs the layer on the dequantised FP8 weights
            import oracle as O

            do = dict(d)
            do["w13"] = O.dequant_fp8_block(d["w13_e4m3"], d["w13_scale"], G=cfg.E,
                                            R=2 * cfg.I, C=cfg.H)
            do["w2"] = O.dequant_fp8_block(d["w2_e4m3"], d["w2_scale"], G=cfg.E, R=cfg.H,
                                           C=cfg.I)
        v, cores, n, dt = oracle_tokens_per_s(cfg, do, seconds=args.cpu_seconds)
        cpu = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{n} of {cfg.T} tokens, whole block per token, {dt:.1f} s"}
        import oracle as O

        O.set_threads(1)
        try:
            v1, _, n1, dt1 = oracle_tokens_per_s(cfg, do, seconds=args.cpu_seconds / 2)
        finally:
            O.set_threads(cores)
        cpu["one_core"] = {"value": v1, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                           "sample": f"{n1} of {cfg.T} tokens, whole block per token, "
                                     f"{dt1:.1f} s"}

    clocks = clk.summary()
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int8" if qk else "bf16",
            "data": "synthetic (seeded normal inputs and weights, "
                    + (f"Zipf({cfg.zipf_s})-skewed router bias" if cfg.zipf_s
                       else "unbiased router")
                    + ("; routed expert weights FP8 E4M3 with 128x128 block scales, "
                       "quantised from the same bf16 weights)" if fp8 else
                       f"; routed expert weights random valid GGUF {qw.upper()} blocks, "
                       + ("expanded to bf16 once on the device)" if qd else
                          "activations quantized to 8-bit blocks on the device)") if qw else ")"),
            "config": dict(config_dict(cfg, ws), weights=args.weights,
                           **({"q_dequant": qd} if qw else {})),
            "e2e": {"value": e2e_value, "unit": "tokens/s",
                    "h2d_bytes_per_step": int(cfg.T * cfg.H * 2),
                    "d2h_bytes_per_step": int(cfg.T * cfg.H * 2)},
            "gpu_launches": launches,
            "roofline": roofline,
            "components": components,
            "cpu_baseline": cpu,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="prefill",
                    choices=["prefill", "decode", "large", "tiny", "combine"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--q-dequant", default="auto", choices=["auto", "on", "off"],
                    help="keep-quant weights: expand to bf16 once and use the tensor-core GEMMs "
                         "(auto: above 16 routed rows per expert)")
    ap.add_argument("--weights", default="bf16", choices=["bf16", "fp8", "q8_0", "q4_k"],
                    help="routed expert weights: bf16, FP8 E4M3 with 128x128 block scales, or "
                         "keep-quant GGUF Q8_0 / Q4_K blocks")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-extra-layers", action="store_true",
                    help="prefill run: skip the decode and large workloads' components")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
