"""One step of the hot path over a workload, through the C ABI.

A step is, for the linears of the workload:
  re-pin every weight scale, then quantise every weight (once per step, one
  multi-tensor call each);
then for every micro-batch j and linear i:
  activation scale -> quantise X -> int8 forward -> dX -> dW, with dW
  accumulated into the linear's gradient in micro-batch order (level 1 of the
  replayed reduction);
and finally, when the workload has R > 1 replicas, TreeFold of the flat
gradient buffer with the R - 1 other replicas' partials (level 3), and, for
workloads with an optimiser, the global gradient norm and a clipped AdamW
update of the (flat) weights, which the next step re-pins and quantises.

With S > 1 shards (the audit's full three-level replay), level 2 folds this
virtual rank's G with the S - 1 other shards' partials of the same replica as a
running sum in mesh order, before TreeFold.

The other shards' and replicas' partials are built once, outside any timed
region, as Q_s = G (+) noise_s and P_r = G_2 (+) noise_r (G_2 the level-2 sum,
or G without shards) -- the same construction as the small single-linear case
-- so that every step folds real-sized, gradient-like buffers.  All arithmetic happens in librepro.so; this
module only allocates device memory (torch) and enqueues calls.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import inputs
from . import repro as R


@dataclass
class HostInputs:
    W: list          # [i] -> np.float32 [N_i, K_i]
    X: list          # [i][j] -> np.float32 [M, K_i]
    dY: list         # [i][j] -> np.float32 [M, N_i]
    noise: list      # [r] -> np.float32 [sum N_i K_i]  (r = 1..R-1; index 0 unused)
    shard_noise: list = None   # [s] -> np.float32 [sum N_i K_i] (s = 1..S-1; index 0 unused)


def generate_host_inputs(wl: inputs.Workload) -> HostInputs:
    L = len(wl.linears)
    W = [inputs.weight(wl, i) for i in range(L)]
    X = [[inputs.activation(wl, i, j) for j in range(wl.microbatches)] for i in range(L)]
    dY = [[inputs.upstream_grad(wl, i, j) for j in range(wl.microbatches)] for i in range(L)]
    n_grad = sum(l.n_out * l.k_in for l in wl.linears)
    noise = [None] + [inputs.replica_noise(wl, r, n_grad) for r in range(1, max(wl.replicas, 1))]
    snoise = [None] + [inputs.shard_noise(wl, s, n_grad) for s in range(1, max(wl.shards, 1))]
    return HostInputs(W, X, dY, noise, snoise)


def grad_offsets(wl: inputs.Workload):
    offs, o = [], 0
    for l in wl.linears:
        offs.append(o)
        o += l.n_out * l.k_in
    return offs, o


class HotPathStep:
    """Device buffers for one workload and the calls of one step."""

    CLASSES = ("wscale_w", "quant_w", "wscale_x", "quant_x", "fwd", "bwd_dx", "bwd_dw",
               "accum", "treefold")

    def __init__(self, wl: inputs.Workload, host: HostInputs | None = None,
                 fused_accum: bool = True, device: str = "cuda", dw_stream: bool | None = None):
        self.wl = wl
        self.fused_accum = fused_accum
        self.host = host if host is not None else generate_host_inputs(wl)
        dev = torch.device(device)
        self.dev = dev
        L, J, M = len(wl.linears), wl.microbatches, wl.tokens
        h = self.host
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
        offs, n_grad = grad_offsets(wl)
        # weights as views of one flat buffer laid out like the flat gradient
        self.Wflat = torch.cat([t(h.W[i]).reshape(-1) for i in range(L)])
        self.W = [self.Wflat[o:o + l.n_out * l.k_in].view(l.n_out, l.k_in)
                  for o, l in zip(offs, wl.linears)]
        self.X = [[t(h.X[i][j]) for j in range(J)] for i in range(L)]
        self.dY = [[t(h.dY[i][j]) for j in range(J)] for i in range(L)]
        self.Wq = [torch.empty(w.shape, dtype=torch.int8, device=dev) for w in self.W]
        self.Xq = [torch.empty((M, l.k_in), dtype=torch.int8, device=dev) for l in wl.linears]
        self.s_w = torch.zeros(L, dtype=torch.float32, device=dev)
        self.s_x = torch.zeros(L, dtype=torch.float32, device=dev)
        self.Y = [torch.empty((M, l.n_out), dtype=torch.float32, device=dev) for l in wl.linears]
        self.dX = [torch.empty((M, l.k_in), dtype=torch.float32, device=dev) for l in wl.linears]
        self.n_grad = n_grad
        self.G = torch.empty(n_grad, dtype=torch.float32, device=dev)
        self.Gv = [self.G[o:o + l.n_out * l.k_in].view(l.n_out, l.k_in)
                   for o, l in zip(offs, wl.linears)]
        self.dW_tmp = None
        if not fused_accum and J > 1:
            self.dW_tmp = [torch.empty((l.n_out, l.k_in), dtype=torch.float32, device=dev)
                           for l in wl.linears]
        n_max = max(max(w.numel() for w in self.W), max(x.numel() for x in self.X[0]))
        n_max = max(n_max, *(x.numel() for i in range(L) for x in self.X[i]))
        self.ws_scale = torch.empty(max(R.repro_wscale_ws_bytes(n_max), 16), dtype=torch.uint8,
                                    device=dev)
        self.ws_wmulti = torch.empty(
            max(R.repro_wscale_multi_ws_bytes([w.numel() for w in self.W]), 16),
            dtype=torch.uint8, device=dev)
        need = max(R.repro_linear_bwd_ws_bytes(M, l.n_out, l.k_in) for l in wl.linears)
        self.ws_bwd = torch.empty(need, dtype=torch.uint8, device=dev) if need > 0 else None
        # dW on a second stream, concurrent with the forward and dX of the same
        # linear (its own workspace): each fills the other's part-empty last
        # waves.  By default only when a linear's backward is long enough for
        # that to matter (2^30 multiply-adds); launch-bound steps would only pay
        # for the extra events.
        if dw_stream is None:
            dw_stream = min(M * l.n_out * l.k_in for l in wl.linears) >= (1 << 30)
        self.s_dw = torch.cuda.Stream(device=dev) if dw_stream else None
        self.ws_bwd_dw = None
        if dw_stream and need > 0:
            self.ws_bwd_dw = torch.empty(need, dtype=torch.uint8, device=dev)
        need = max(R.repro_linear_fwd_ws_bytes(M, l.n_out, l.k_in) for l in wl.linears)
        self.ws_fwd = torch.empty(need, dtype=torch.uint8, device=dev) if need > 0 else None
        self.parts = None
        self.TF = None
        if wl.replicas > 1:
            self.TF = torch.empty(n_grad, dtype=torch.float32, device=dev)
        self.shard_parts = None
        self.G2 = None
        if wl.shards > 1:
            self.G2 = torch.empty(n_grad, dtype=torch.float32, device=dev)
        self.use_optimizer = wl.optimizer
        self.step_t = 0
        if wl.optimizer:
            self.m = torch.zeros(n_grad, dtype=torch.float32, device=dev)
            self.v = torch.zeros(n_grad, dtype=torch.float32, device=dev)
            self.sumsq = torch.zeros(1, dtype=torch.float32, device=dev)
            self.ws_sumsq = torch.empty(max(R.repro_sumsq_ws_bytes(n_grad), 16),
                                        dtype=torch.uint8, device=dev)
            # per-step state hash of (parameters, first moment, second moment)
            self.state = [self.Wflat, self.m, self.v]
            self.digest = torch.zeros(32, dtype=torch.uint8, device=dev)
            self.ws_hash = torch.empty(max(R.repro_state_hash_ws_bytes(self.state), 16),
                                       dtype=torch.uint8, device=dev)
        # the zero fills above ran on the current stream; steps may run on another
        torch.cuda.synchronize(dev)

    # ------------------------------------------------------------------ step

    def _ev(self, timers, cls, stream):
        if timers is None:
            return None
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        timers.setdefault(cls, []).append([e, None])
        return e

    def _end(self, timers, cls, stream):
        if timers is None:
            return
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        timers[cls][-1][1] = e

    def run(self, stream: torch.cuda.Stream, timers: dict | None = None,
            wait_events: list | None = None, done_events: list | None = None,
            fold_wait_events: list | None = None) -> None:
        """Enqueue one step on `stream` (and, with dw_stream, its dW calls on
        the step's second stream, joined back before the folds).  With
        `timers`, records a CUDA event pair around every call, grouped by call
        class, and for concurrent dX/dW the fork event with both end events
        under "bwd_pair".  `wait_events[j]`, if given, is waited on before
        micro-batch j's first use of its inputs.  `done_events`, if given (a
        list of J + 1 slots), receives in slot j the events after which
        micro-batch j's X and dY are no longer read, and in slot J those for
        the weights W (read only by the scale and quantise calls at the start
        of the step), so a producer can refill each input as soon as this step
        is done with it.  `fold_wait_events`, if given, are waited on before
        TreeFold rewrites its output (a reader of the previous step's result
        may still be copying it out)."""
        wl, s = self.wl, stream
        L, J = len(wl.linears), wl.microbatches
        s2 = self.s_dw
        dw_done = [None] * L
        sw = lambda i: self.s_w[i:i + 1]  # noqa: E731
        sx = lambda i: self.s_x[i:i + 1]  # noqa: E731
        if wait_events is not None and wait_events[0] is not None:
            s.wait_event(wait_events[0])
        # every weight's scale, then every weight's codes: one pass each
        self._ev(timers, "wscale_w", s)
        R.repro_wscale_multi(self.W, R.REPRO_SCALE_WEIGHT_MEANABS, self.s_w, ws=self.ws_wmulti,
                             stream=s)
        self._end(timers, "wscale_w", s)
        self._ev(timers, "quant_w", s)
        R.repro_quant_i8_multi(self.W, self.s_w, self.Wq, stream=s)
        self._end(timers, "quant_w", s)
        if done_events is not None:
            e = torch.cuda.Event()
            e.record(s)
            done_events[J] = [e]
        for j in range(J):
            if wait_events is not None and j > 0 and wait_events[j] is not None:
                s.wait_event(wait_events[j])
            for i in range(L):
                X, dY = self.X[i][j], self.dY[i][j]
                if dw_done[i] is not None:
                    s.wait_event(dw_done[i])   # Xq[i] and s_x[i] are rewritten next
                self._ev(timers, "wscale_x", s)
                R.repro_wscale(X, R.REPRO_SCALE_ACT_AMAX, sx(i), ws=self.ws_scale, stream=s)
                self._end(timers, "wscale_x", s)
                self._ev(timers, "quant_x", s)
                R.repro_quant_i8(X, sx(i), self.Xq[i], stream=s)
                self._end(timers, "quant_x", s)
                fork = None
                if s2 is not None:
                    fork = torch.cuda.Event(enable_timing=timers is not None)
                    fork.record(s)
                    s2.wait_event(fork)
                    self._dw(i, j, dY, sx(i), s2, timers)
                    dw_done[i] = torch.cuda.Event()
                    dw_done[i].record(s2)
                self._ev(timers, "fwd", s)
                R.repro_linear_fwd(self.Xq[i], self.Wq[i], sx(i), sw(i), self.Y[i],
                                   ws=self.ws_fwd, stream=s)
                self._end(timers, "fwd", s)
                self._ev(timers, "bwd_dx", s)
                R.repro_linear_bwd(dY, None, self.Wq[i], None, sw(i), dx=self.dX[i], dw=None,
                                   ws=self.ws_bwd, stream=s)
                self._end(timers, "bwd_dx", s)
                if s2 is None:
                    self._dw(i, j, dY, sx(i), s, timers)
                elif timers is not None:
                    timers.setdefault("bwd_pair", []).append(
                        [fork, timers["bwd_dx"][-1][1], timers["bwd_dw"][-1][1]])
            if done_events is not None:
                e = torch.cuda.Event()
                e.record(s)
                done_events[j] = [e] + ([dw_done[L - 1]] if s2 is not None else [])
        for d in dw_done:
            if d is not None:
                s.wait_event(d)   # join the dW stream before the folds
        level2 = self.G
        if self.G2 is not None and self.shard_parts is not None:
            self._ev(timers, "running_sum", s)
            R.repro_running_sum([self.G] + self.shard_parts, self.G2, stream=s)
            self._end(timers, "running_sum", s)
            level2 = self.G2
        if self.TF is not None and not getattr(self, "skip_treefold", False):
            for ev in fold_wait_events or ():
                s.wait_event(ev)
            if self.parts is None:
                raise RuntimeError("prepare_replicas() must run before a step with TreeFold")
            self._ev(timers, "treefold", s)
            R.repro_treefold([level2] + self.parts, self.TF, stream=s)
            self._end(timers, "treefold", s)
        if self.use_optimizer and not getattr(self, "skip_treefold", False):
            grad = self.result()
            self.step_t += 1
            self._ev(timers, "sumsq", s)
            R.repro_sumsq(grad, self.sumsq, ws=self.ws_sumsq, stream=s)
            self._end(timers, "sumsq", s)
            self._ev(timers, "adamw", s)
            R.repro_adamw_step(self.Wflat, self.m, self.v, grad, self.sumsq, self.step_t, stream=s)
            self._end(timers, "adamw", s)
            self._ev(timers, "state_hash", s)
            R.repro_state_hash(self.state, self.digest, ws=self.ws_hash, stream=s)
            self._end(timers, "state_hash", s)

    def capture(self, stream: torch.cuda.Stream) -> "torch.cuda.CUDAGraph":
        """Capture one step into a CUDA graph.  Every call only enqueues on the
        caller's stream, allocates nothing and never synchronises, so the whole
        step captures; replaying the graph repeats its launches with one host
        call.  Run `prepare()` (replicated workloads) and a warm-up step first.
        A step with AdamW cannot be captured: the step count t is a host
        argument of repro_adamw_step and would be frozen in the graph."""
        if self.use_optimizer:
            raise RuntimeError("a step with the optimizer cannot be captured: t is a host argument")
        if self.TF is not None and self.parts is None:
            raise RuntimeError("prepare_replicas() must run before capturing a step with TreeFold")
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            self.run(stream)
        return g

    def _dw(self, i: int, j: int, dY, sx, st, timers) -> None:
        """dW of linear i for micro-batch j on stream `st`: fused into G, or
        into a scratch buffer then accumulated (the first micro-batch is a copy)."""
        ws = self.ws_bwd_dw if st is self.s_dw else self.ws_bwd
        if j == 0 or self.fused_accum:
            self._ev(timers, "bwd_dw", st)
            R.repro_linear_bwd(dY, self.Xq[i], None, sx, None, dx=None, dw=self.Gv[i],
                               accumulate=j > 0, ws=ws, stream=st)
            self._end(timers, "bwd_dw", st)
        else:
            self._ev(timers, "bwd_dw", st)
            R.repro_linear_bwd(dY, self.Xq[i], None, sx, None, dx=None, dw=self.dW_tmp[i],
                               ws=ws, stream=st)
            self._end(timers, "bwd_dw", st)
            self._ev(timers, "accum", st)
            R.repro_grad_accum(self.Gv[i], self.dW_tmp[i], stream=st)
            self._end(timers, "accum", st)

    def prepare_replicas(self, stream: torch.cuda.Stream) -> None:
        """Q_s = G (+) shard_noise_s (s = 1..S-1), then G_2 = running sum, then
        P_r = G_2 (+) noise_r (r = 1..R-1), from the current G (untimed)."""
        base = self.G
        if self.G2 is not None:
            self.shard_parts = []
            for sh in range(1, self.wl.shards):
                q = self.G.clone()
                R.repro_grad_accum(q, torch.from_numpy(self.host.shard_noise[sh]).to(self.dev),
                                   stream=stream)
                self.shard_parts.append(q)
            R.repro_running_sum([self.G] + self.shard_parts, self.G2, stream=stream)
            base = self.G2
        if self.wl.replicas <= 1:
            return
        self.parts = []
        for r in range(1, self.wl.replicas):
            p = base.clone()
            R.repro_grad_accum(p, torch.from_numpy(self.host.noise[r]).to(self.dev), stream=stream)
            self.parts.append(p)

    def input_buffers(self) -> list:
        """The step's seeded inputs in a fixed order: the flat weights, then X
        and dY of every linear, micro-batch by micro-batch."""
        L, J = len(self.wl.linears), self.wl.microbatches
        return [self.Wflat] + [t for j in range(J) for i in range(L) for t in (self.X[i][j], self.dY[i][j])]

    def input_digest(self) -> str:
        """RFC 6962 Merkle Tree Hash (SHA-256 over 4 KB leaves) of
        input_buffers(), taken on the device by repro_state_hash, as hex: the
        record of which bytes a run computed on.  Synchronises the device."""
        d = torch.empty(32, dtype=torch.uint8, device=self.dev)
        R.repro_state_hash(self.input_buffers(), d)
        torch.cuda.synchronize(self.dev)
        return bytes(d.cpu().numpy()).hex()

    def result(self) -> torch.Tensor:
        """The step's result: the folded gradient (or the level-2 sum, or G)."""
        if self.TF is not None:
            return self.TF
        return self.G2 if self.G2 is not None else self.G

    def prepare(self, stream: torch.cuda.Stream) -> None:
        """One step without the folds that need the other ranks' partials, then
        build those partials (everything untimed)."""
        self.skip_treefold, shards = True, self.shard_parts
        self.shard_parts = None
        self.run(stream)
        self.skip_treefold, self.shard_parts = False, shards
        self.prepare_replicas(stream)

    def flops(self):
        """Algorithmic work of one step: int8 MACs (forward) and fp32
        multiplies+adds (backward), per call class."""
        wl = self.wl
        M, J = wl.tokens, wl.microbatches
        mac = sum(M * l.n_out * l.k_in for l in wl.linears) * J
        return {"fwd_int_ops": 2 * mac, "bwd_dx_fp32_ops": 2 * mac, "bwd_dw_fp32_ops": 2 * mac}

    def tokens(self) -> int:
        return self.wl.tokens * self.wl.microbatches
