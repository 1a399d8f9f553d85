"""The MoE expert block as one object: buffers in HBM plus the sequence of
C-ABI calls that make up one forward pass.

    route -> permute -> gate/up GEMM + SiLU-mul -> down GEMM (weight, scatter)
          [-> shared expert gate/up + down]  -> combine (or combine-gate)

PyTorch only allocates device memory and provides the stream; every step is
one call into libmoe.so.  All buffers are allocated once for ``max_tokens``
and reused, no call allocates or synchronises, so a whole forward can be
captured into a CUDA graph and replayed (``capture``/``replay``).
"""
from __future__ import annotations

import torch

from . import (BF16, QFMT_Q4_K, QFMT_Q8_0, moe_combine, moe_combine_gate,
               moe_gate_workspace_size, moe_grouped_gemm_down_bf16,
               moe_grouped_gemm_down_bf16_shared, moe_grouped_gemm_down_fp8w,
               moe_grouped_gemm_down_q, moe_grouped_gemm_gateup_silu_bf16,
               moe_grouped_gemm_gateup_silu_bf16_shared, moe_grouped_gemm_gateup_silu_bf16_staged,
               moe_grouped_gemm_gateup_silu_fp8w, moe_gateup_staged_workspace_size,
               moe_grouped_gemm_gateup_silu_q, moe_dequantize_q_bf16, moe_permute,
               moe_permute_workspace_size, moe_quantize_act_q8, moe_route_topk,
               moe_route_topk_workspace_size)

# keep-quant weight formats: name -> (library format id, weights per activation block)
Q_WEIGHTS = {"q8_0": (QFMT_Q8_0, 32), "q4_k": (QFMT_Q4_K, 256)}


def _dev_bf16(a, device):
    """numpy uint16 bf16 bits (or a tensor) -> contiguous device bf16 tensor."""
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        return a.to(device).contiguous()
    t = torch.from_numpy(a.view("int16").copy()).view(torch.bfloat16)
    return t.to(device).contiguous()


class MoeBlock:
    """One MoE expert block with resident weights.

    weights: dict with ``w_router`` [E,H], ``w13`` [E,2I,H], ``w2`` [E,H,I] (bf16),
    optional ``logit_bias`` [E] f32, and for a shared expert ``w_shared_gate``
    [H], ``w13_shared`` [1,2Is,H], ``w2_shared`` [1,H,Is].
    fp8_weights=True: the routed experts' weights are block-scaled FP8 instead,
    ``w13_e4m3`` / ``w13_scale`` and ``w2_e4m3`` / ``w2_scale`` (codes uint8 of
    the same shapes, f32 scales per 128 x 128 block); the shared expert stays
    bf16 and runs in launches of its own.
    qweights="q8_0" | "q4_k": keep-quant routed experts, ``w13q`` [E, 2I, H/blk*bytes]
    and ``w2q`` [E, H, I/blk*bytes] GGUF blocks (uint8).  The token rows and the
    act rows are quantized to 8-bit blocks on the device, the gate/up GEMM reads
    the token rows through sorted_pair / K (no x_perm), and the shared expert
    stays bf16 in launches of its own.
    gather=True reads the routed rows of x inside the gate/up GEMM on every call;
    gather="auto" does so only on calls with at most 16 routed rows per expert
    on average (decode-sized; plain bf16 experts, no fused shared expert), where
    the 32-row tiles gather as fast as they read x_perm and the permute's row
    copy is saved, and materialises x_perm otherwise.
    q_dequant=True (with qweights): the GGUF blocks are expanded to bf16 once, on the
    device, when the block is built, and the layer runs the bf16 tensor-core path --
    the faster choice when the experts see many rows each (prefill-sized batches).
    """

    def __init__(self, H, I, E, K, weights, max_tokens, device="cuda", I_shared=0,
                 routed_scale=1.0, gather=False, fuse_shared=True, fp8_weights=False,
                 qweights=None, q_dequant=False, staged=False):
        self.H, self.I, self.E, self.K, self.Is = H, I, E, K, I_shared
        if qweights is not None:
            if qweights not in Q_WEIGHTS:
                raise ValueError(f"qweights must be one of {sorted(Q_WEIGHTS)}")
            if fp8_weights:
                raise ValueError("qweights and fp8_weights exclude each other")
            if not q_dequant:
                gather = True
        self.qfmt, qblk = Q_WEIGHTS[qweights] if qweights is not None else (0, 0)
        if q_dequant:
            if qweights is None:
                raise ValueError("q_dequant needs qweights")
            weights = self._dequantized(weights, H, I, E, self.qfmt, device)
            self.qfmt, qblk = 0, 0
        self.max_tokens = max_tokens
        # gather=True: the gate/up GEMM reads each routed row straight from x
        # (through sorted_pair / K); False: permute materialises x_perm and the
        # GEMM streams it with tiled TMA loads
        if gather not in (False, True, "auto"):
            raise ValueError(f"gather must be False, True or 'auto', not {gather!r}")
        self.gather = gather
        always = gather is True
        # fuse_shared: the shared expert's GEMMs run inside the routed GEMM
        # launches (one launch each for gate/up and down); False: own launches
        self.fp8 = fp8_weights
        self.fuse_shared = fuse_shared and not always and not fp8_weights and not self.qfmt
        if fp8_weights and always:
            raise ValueError("FP8 expert weights read x_perm rows (gather=False)")
        # staged=True: permute skips its row gather and the gate/up call writes
        # x_perm itself (on CTA pairs inside the GEMM launch); bf16 experts only
        self.staged = staged
        if staged and (gather is not False or fp8_weights or self.qfmt or
                       (I_shared > 0 and self.fuse_shared)):
            raise ValueError("staged rows need plain bf16 experts, gather=False and no fused "
                             "shared expert")
        self.routed_scale = float(routed_scale)
        self.device = torch.device(device)
        if self.device.type != "cuda":
            # every step runs in the library's CUDA kernels, which take device pointers
            raise ValueError(f"MoeBlock needs a CUDA device, not {self.device}; there is no CPU path")
        dv = self.device
        self.w_router = _dev_bf16(weights["w_router"], dv)
        if fp8_weights:
            def dev(a, dt):
                return torch.as_tensor(a).to(dtype=dt).to(dv).contiguous()
            self.w13_q = dev(weights["w13_e4m3"], torch.uint8)
            self.w13_s = dev(weights["w13_scale"], torch.float32)
            self.w2_q = dev(weights["w2_e4m3"], torch.uint8)
            self.w2_s = dev(weights["w2_scale"], torch.float32)
            self.w13 = self.w2 = None
        elif self.qfmt:
            self.w13_q = torch.as_tensor(weights["w13q"], dtype=torch.uint8).to(dv).contiguous()
            self.w2_q = torch.as_tensor(weights["w2q"], dtype=torch.uint8).to(dv).contiguous()
            self.w13 = self.w2 = None
        else:
            self.w13 = _dev_bf16(weights["w13"], dv)
            self.w2 = _dev_bf16(weights["w2"], dv)
        lb = weights.get("logit_bias")
        self.logit_bias = None if lb is None else torch.as_tensor(lb, dtype=torch.float32).to(dv)
        self.has_shared = I_shared > 0
        if self.has_shared:
            self.w_shared_gate = _dev_bf16(weights["w_shared_gate"], dv)
            self.w13_shared = _dev_bf16(weights["w13_shared"], dv)
            self.w2_shared = _dev_bf16(weights["w2_shared"], dv)
        T, P = max_tokens, max_tokens * K
        i32, f32, bf = torch.int32, torch.float32, torch.bfloat16
        self.topk_ids = torch.empty((T, K), dtype=i32, device=dv)
        self.topk_w = torch.empty((T, K), dtype=f32, device=dv)
        self.gate_logit = torch.empty((T,), dtype=f32, device=dv)
        self.expert_offsets = torch.empty((E + 1,), dtype=i32, device=dv)
        self.sorted_pair = torch.empty((P,), dtype=i32, device=dv)
        self.pair_to_row = torch.empty((P,), dtype=i32, device=dv)
        self.x_perm = None if always else torch.empty((P, H), dtype=bf, device=dv)
        # zero-filled once, then passed unchanged to every staged call
        self.ws_staged = (torch.zeros(max(16, moe_gateup_staged_workspace_size(P)),
                                      dtype=torch.uint8, device=dv) if staged else None)
        self.act = torch.empty((P, I), dtype=bf, device=dv)
        if self.qfmt:
            # 8-bit activation blocks of the token rows and of the act rows
            self.x_q = torch.empty((T, H), dtype=torch.int8, device=dv)
            self.x_s = torch.empty((T, H // qblk), dtype=f32, device=dv)
            self.act_q = torch.empty((P, I), dtype=torch.int8, device=dv)
            self.act_s = torch.empty((P, I // qblk), dtype=f32, device=dv)
        self.expert_out = torch.empty((P, H), dtype=bf, device=dv)
        self.out = torch.empty((T, H), dtype=bf, device=dv)
        if self.has_shared:
            self.act_shared = torch.empty((T, I_shared), dtype=bf, device=dv)
            self.sd = torch.empty((T, H), dtype=bf, device=dv)
        self.ws_route = moe_route_topk_workspace_size(T, E, K)
        self.ws_perm = moe_permute_workspace_size(T, K, E)
        self.ws_gate = moe_gate_workspace_size(T)
        self.workspace = torch.empty((max(self.ws_route, self.ws_perm, self.ws_gate, 256),),
                                     dtype=torch.uint8, device=dv)
        self.graph = None
        self.graph_x = None
        self._pipe = None

    # one forward over x [T, H] bf16 (device); returns a view of the output buffer.
    # marks: optional list; a CUDA event is recorded after each stage and
    # appended as (stage name, event), for per-kernel timing on the stream.
    # stages=False records only the first ("start") and the last event: an
    # event between two kernels keeps the second from starting early under
    # programmatic dependent launch, so whole-step timings leave them out.
    def forward(self, x, stream=None, marks=None, out=None, stages=True):
        T = x.shape[0]
        assert T <= self.max_tokens and x.dtype == torch.bfloat16 and x.is_contiguous()
        H, I, E, K = self.H, self.I, self.E, self.K
        P = T * K
        ws = self.workspace

        def mark(name, edge=False):
            if marks is not None and (stages or edge):
                ev = torch.cuda.Event(enable_timing=True)
                ev.record(torch.cuda.current_stream(self.device) if stream is None else stream)
                marks.append((name, ev))

        mark("start", edge=True)
        moe_route_topk(x, self.w_router, self.logit_bias,
                       self.w_shared_gate if self.has_shared else None, None, T, H, E, K, 1, 0, 1,
                       self.topk_ids, self.topk_w, None,
                       self.gate_logit if self.has_shared else None, ws, ws.numel(), stream)
        mark("route")
        fused = self.has_shared and self.fuse_shared
        gathered = self.gather is True or (
            self.gather == "auto" and P <= 16 * E and not fused and not self.staged
            and not self.fp8 and not self.qfmt)
        moe_permute(self.topk_ids, x, T, K, E, H, self.expert_offsets, self.sorted_pair,
                    self.pair_to_row, None if (self.staged or gathered) else self.x_perm, ws,
                    ws.numel(), stream)
        mark("permute")
        if self.qfmt:
            moe_quantize_act_q8(x, T, H, self.qfmt, self.x_q, self.x_s, stream)
            mark("quant_x")
            moe_grouped_gemm_gateup_silu_q(self.x_q, self.x_s, T, self.sorted_pair, K, self.w13_q,
                                           self.qfmt, self.expert_offsets, P, H, I, E, self.act,
                                           stream)
        elif self.fp8:
            moe_grouped_gemm_gateup_silu_fp8w(self.x_perm, self.w13_q, self.w13_s,
                                              self.expert_offsets, P, H, I, E, self.act, None, 0,
                                              stream)
        elif fused:
            moe_grouped_gemm_gateup_silu_bf16_shared(self.x_perm, self.w13, self.expert_offsets,
                                                     P, H, I, E, self.act, x, T, self.w13_shared,
                                                     self.Is, self.act_shared, None, 0, stream)
        elif self.staged:
            moe_grouped_gemm_gateup_silu_bf16_staged(x, T, self.sorted_pair, K, self.x_perm,
                                                     self.w13, self.expert_offsets, P, H, I, E,
                                                     self.act, self.ws_staged,
                                                     self.ws_staged.numel(), stream)
        elif gathered:
            moe_grouped_gemm_gateup_silu_bf16(x, T, self.sorted_pair, K, self.w13,
                                              self.expert_offsets, P, H, I, E, self.act, None, 0,
                                              stream)
        else:
            moe_grouped_gemm_gateup_silu_bf16(self.x_perm, P, None, 1, self.w13,
                                              self.expert_offsets, P, H, I, E, self.act, None, 0,
                                              stream)
        mark("gemm_gateup")
        if self.qfmt:
            moe_quantize_act_q8(self.act, P, I, self.qfmt, self.act_q, self.act_s, stream)
            mark("quant_act")
            moe_grouped_gemm_down_q(self.act_q, self.act_s, self.w2_q, self.qfmt,
                                    self.expert_offsets, self.topk_w, self.sorted_pair, P, I, H, E,
                                    self.expert_out, stream)
        elif self.fp8:
            moe_grouped_gemm_down_fp8w(self.act, self.w2_q, self.w2_s, self.expert_offsets,
                                       self.topk_w, self.sorted_pair, P, I, H, E, self.expert_out,
                                       None, 0, stream)
        elif fused:
            moe_grouped_gemm_down_bf16_shared(self.act, self.w2, self.expert_offsets, self.topk_w,
                                              self.sorted_pair, P, I, H, E, self.expert_out,
                                              self.act_shared, T, self.w2_shared, self.Is, self.sd,
                                              None, 0, stream)
        else:
            moe_grouped_gemm_down_bf16(self.act, self.w2, self.expert_offsets, self.topk_w,
                                       self.sorted_pair, P, I, H, E, self.expert_out, None, 0,
                                       stream)
        mark("gemm_down")
        out = self.out[:T] if out is None else out
        if self.has_shared:
            if not fused:
                moe_grouped_gemm_gateup_silu_bf16(x, T, None, 1, self.w13_shared, None, T, H,
                                                  self.Is, 1, self.act_shared, None, 0, stream)
                moe_grouped_gemm_down_bf16(self.act_shared, self.w2_shared, None, None, None, T,
                                           self.Is, H, 1, self.sd, None, 0, stream)
                mark("shared_expert")
            moe_combine_gate(self.expert_out, BF16, None, self.sd, BF16, self.gate_logit,
                             self.routed_scale, T, K, H, out, BF16, ws, ws.numel(), stream)
            mark("combine", edge=True)
            return out
        else:
            moe_combine(self.expert_out, BF16, None, None, BF16, self.routed_scale, T, K, H, out,
                        BF16, stream)
        mark("combine", edge=True)
        return out

    @staticmethod
    def _dequantized(weights, H, I, E, qfmt, device):
        """`weights` with w13 / w2 expanded from the GGUF blocks to bf16 on the device."""
        dv = torch.device(device)
        out = dict(weights)
        for key, qkey, rows, Kd in (("w13", "w13q", E * 2 * I, H), ("w2", "w2q", E * H, I)):
            q = torch.as_tensor(weights[qkey], dtype=torch.uint8).to(dv).contiguous()
            w = torch.empty((rows, Kd), dtype=torch.bfloat16, device=dv)
            moe_dequantize_q_bf16(q, qfmt, rows, Kd, w)
            out[key] = w.view(E, rows // E, Kd)
        torch.cuda.current_stream(dv).synchronize()
        return out

    # launches per forward (for the bench's gpu_launches claim)
    def capture(self, x_static):
        """Record one forward over the fixed input buffer ``x_static`` into a CUDA graph."""
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            self.forward(x_static)  # warm-up outside the graph: sets kernel attributes once
        torch.cuda.current_stream(self.device).wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.forward(x_static)
        self.graph, self.graph_x = g, x_static
        return g

    def replay(self):
        self.graph.replay()
        return self.out[: self.graph_x.shape[0]]

    def run_host_batches(self, x_hosts, out_hosts):
        """End to end over pinned host batches: out_hosts[i] <- block(x_hosts[i]).

        Batch i computes on the current stream while batch i+1 is copied in
        on an upload stream and batch i-1 is copied out on a download stream;
        device input and output buffers are double-buffered and every reuse
        waits on the event that frees it.  Returns when all work is enqueued;
        synchronise the current stream (or the device) before reading
        out_hosts.  Batches may have different token counts up to max_tokens.
        """
        dev = self.device
        H = self.H
        if self._pipe is None:
            mk = lambda: torch.empty((self.max_tokens, H), dtype=torch.bfloat16, device=dev)
            ev = lambda: torch.cuda.Event()
            self._pipe = {
                "up": torch.cuda.Stream(device=dev), "down": torch.cuda.Stream(device=dev),
                "x": [mk(), mk()], "o": [mk(), mk()],
                "h2d": [ev(), ev()], "fwd": [ev(), ev()], "d2h": [ev(), ev()],
            }
        pp = self._pipe
        cs = torch.cuda.current_stream(dev)
        up, down = pp["up"], pp["down"]
        n = len(x_hosts)
        up.wait_stream(cs)
        down.wait_stream(cs)

        def upload(i):
            b = i % 2
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(pp["fwd"][b])      # batch i-2 no longer reads x[b]
                T = x_hosts[i].shape[0]
                pp["x"][b][:T].copy_(x_hosts[i], non_blocking=True)
                pp["h2d"][b].record(up)

        if n:
            upload(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                upload(i + 1)
            T = x_hosts[i].shape[0]
            cs.wait_event(pp["h2d"][b])
            if i >= 2:
                cs.wait_event(pp["d2h"][b])          # batch i-2's output has left o[b]
            self.forward(pp["x"][b][:T], out=pp["o"][b][:T])
            pp["fwd"][b].record(cs)
            with torch.cuda.stream(down):
                down.wait_event(pp["fwd"][b])
                out_hosts[i].copy_(pp["o"][b][:T], non_blocking=True)
                pp["d2h"][b].record(down)
        cs.wait_stream(up)
        cs.wait_stream(down)
        return out_hosts
