"""Benchmark of the routed-MoE decode forward over int4-grouped experts on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl coli|reference]
                    [--workload glm_decode_b1|glm_decode_b8|olmoe_decode|glm_prefill|quant]

Default workload: GLM-like decode layers at batch 1 -- 8 MoE layers, hidden
6144, 256 routed experts of FFN width 2048 plus 1 shared expert, top-8,
int4-grouped g64 experts quantised from N(0, 0.02) bf16 (43.7 GB resident),
bf16 router.  One step = one token through all 8 layers (router, top-k, route
counts, batch union, gate/up + SwiGLU, down, combine, shared expert); each
layer takes its own fresh N(0,1) input.  The timed region is the median of
--repeats windows of K steps.

Prints one JSON line (rank 0).  With torchrun (N > 1) every rank runs an
independent replica on its own GPU (the decode path has no exchange step);
`value` sums the ranks' tokens over the slowest rank's time.
"""
import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "MoE decode tokens/s and int4 expert-weight GB/s vs GB300 HBM peak"

# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of
# each kernel from an ncu capture of the current kernel build, keyed by
# workload and kernel; absent (null in the line) until such a capture exists
# or once the kernel has changed since.  Batch 1: the per-layer launch is the
# same in a 1- or 2-layer capture as in the full stack.
NCU_TRAFFIC = {}

# Captures of earlier builds of kernels that have changed since (the decode
# kernels' routing code, and for batch 8 also the expert-record lookup of the
# tiered store; the quantiser's lane teams).  The line reports them beside a
# null traffic, labelled as such, not as the traffic.
NCU_TRAFFIC_EARLIER = {
    # the one-token layer kernel (one launch per layer; mean of two captured launches)
    "olmoe_decode": {"k_layer1": 28637184},
    # the one-token gate/up (with the first layer's router) and down kernels
    "glm_decode_b1": {"k_gateup": 132213120, "k_down": 64369792},
    # the several-token kernel k_gateup_multi; its experts per launch vary with
    # the routing
    "glm_decode_b8": {"k_gateup": 879500288 + 7344384},
    # one launch over 16 experts' matrices: 402.7 MB read, 55.8 MB written
    "quant16": {"k_quant_vec": 402740480 + 55846144},
}
EARLIER_NOTE = ("traffic is null: the kernel changed after its last ncu capture; "
                "traffic_earlier_build is that capture")


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1900.0)), "measured"
    return 6800.0, 1900.0, "fallback"


# ---------------------------------------------------------------------------
# clocks sampled during the timed region


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, interval_ms=50):
        self.gpu = gpu_index
        self.interval = interval_ms
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", str(self.interval)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [s.strip() for s in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self, t0, t1):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        win = [s for t, s in self.samples if t0 <= t <= t1]
        note = None
        if len(win) < 3:  # timed region shorter than a few sampling intervals
            mid = 0.5 * (t0 + t1)
            win = [s for t, s in sorted(self.samples, key=lambda ts: abs(ts[0] - mid))[:5]]
            note = "timed region shorter than 3 samples; nearest 5 samples used"

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(s[1]) for s in win if num(s[1]) is not None]
        mx = [num(s[2]) for s in win if num(s[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in win for i in range(4)
                          if len(s) > 5 + i and s[5 + i].lower().startswith("active")})
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(win)}
        if note:
            out["note"] = note
        return out


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(v, world, dev):
    if world == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# decode workloads


class DecodeWorkload:
    """A decode stack resident in HBM: weights, routers, per-step inputs."""

    def __init__(self, shape, steps_total, dev, seed=0, router="softmax"):
        import int4_expert_ffn_gb300 as pkg
        from int4_expert_ffn_gb300 import synth
        self.coli = pkg.binding
        self.synth = synth
        self.shape = shape
        self.dev = dev
        c = self.coli
        L, H, F, E, S, T = (shape.layers, shape.hidden, shape.ffn, shape.experts, shape.shared,
                            shape.tokens)
        self.eb = c.coli_expert_packed_bytes(H, F)
        self.es = c.coli_expert_scale_count(H, F)
        n = E + S
        self.packed = torch.empty(L * n * self.eb, dtype=torch.uint8, device=dev)
        self.scales = torch.empty(L * n * self.es, dtype=torch.float32, device=dev)
        wrs = []
        for l in range(L):
            p0, s0 = l * n * self.eb, l * n * self.es
            for e in range(n):
                for m in range(3):
                    w = synth.expert_matrix(shape, l, e, m, seed, device=dev)
                    rows, cols = w.shape
                    nb, ns = rows * cols // 2, rows * cols // 64
                    c.coli_quant_i4g(w, self.packed[p0:p0 + nb].view(rows, -1),
                                     self.scales[s0:s0 + ns].view(rows, -1))
                    p0 += nb
                    s0 += ns
            wrs.append(synth.router_weights(shape, l, seed, device=dev))
        self.router = torch.stack(wrs).contiguous()
        # chained: one input per step ([K, T, H]); else one per step and layer ([K, L, T, H])
        if shape.chained:
            self.x = torch.stack([synth.tokens(shape, seed, i, device=dev)
                                  for i in range(steps_total)]).contiguous()
            self.out = torch.empty((steps_total, T, H), dtype=torch.float32, device=dev)
        else:
            self.x = torch.stack([torch.stack([synth.tokens(shape, seed, i, device=dev, layer=l)
                                               for l in range(L)])
                                  for i in range(steps_total)]).contiguous()
            self.out = torch.empty((steps_total, L, T, H), dtype=torch.float32, device=dev)
        self.layer_bytes = n * self.eb
        self.layer_scales = n * self.es
        self.counts = torch.zeros((steps_total, L, E), dtype=torch.int32, device=dev)
        rdt = c.COLI_BF16 if shape.router_dtype == "bf16" else c.COLI_F32
        if router == "sigmoid":
            # the GLM router: per-layer selection biases; one descriptor per layer
            # call (unchained) or one for the stack ([L, E] biases)
            self.bias = torch.stack([synth.router_bias(shape, l, seed, device=dev)
                                     for l in range(L)]).contiguous()
            fn = c.COLI_ROUTER_SIGMOID_BIAS
            self.desc = c.MoEDesc(H, F, E, S, T, c.COLI_F32, rdt, fn, self.bias)
            self.layer_desc = [c.MoEDesc(H, F, E, S, T, c.COLI_F32, rdt, fn, self.bias[l])
                               for l in range(L)]
        else:
            self.desc = c.MoEDesc(H, F, E, S, T, c.COLI_F32, rdt)
            self.layer_desc = [self.desc] * L
        self.ws = c.new_workspace(self.desc, shape.top_k)
        torch.cuda.synchronize()

    def step(self, i, stream=None, x=None, out=None):
        """One decode step: the token(s) through every layer.  Chained stacks
        are one stack call; otherwise one layer call per layer."""
        c, sh = self.coli, self.shape
        x = self.x[i] if x is None else x
        out = self.out[i] if out is None else out
        if sh.chained:
            c.coli_moe_stack_forward(self.desc, sh.top_k, sh.layers, x, self.router,
                                     self.packed, self.scales, self.ws, x_out=out,
                                     route_counts=self.counts[i], stream=stream)
            return
        pb, sb = self.layer_bytes, self.layer_scales
        for l in range(sh.layers):
            c.coli_moe_forward(self.layer_desc[l], sh.top_k, x[l], self.router[l],
                               self.packed[l * pb:(l + 1) * pb], self.scales[l * sb:(l + 1) * sb],
                               self.ws, out=out[l], route_counts=self.counts[i, l], stream=stream)

    def fused(self):
        """One token at whole 1024-column chunks with the used experts at most
        512 KB per SM: one fused kernel per layer (the library's rule)."""
        sh = self.shape
        sms = torch.cuda.get_device_properties(self.dev).multi_processor_count
        per_sm = (sh.top_k + sh.shared) * (self.eb + 4 * self.es) / sms
        return (sh.tokens == 1 and sh.hidden % 1024 == 0 and sh.ffn % 1024 == 0
                and per_sm <= 512 * 1024)

    def gu_router(self):
        """One token on the GEMV kernels: the first layer of each call forms
        its router logits inside the gate/up kernel (no router launch)."""
        return self.shape.tokens == 1 and not self.fused()

    def kernels_per_step(self):
        # per 16-token pass: chained, the first layer's router partials, then
        # the layer kernel(s) of every layer; else the router partials and the
        # layer kernel(s) per layer
        sh = self.shape
        passes = (sh.tokens + 15) // 16
        # fused: one kernel; else gate/up and down (several tokens: gate/up,
        # the per-expert down GEMVs and the combine)
        per_layer = 1 if self.fused() else (2 if sh.tokens == 1 else 3)
        route = 0 if self.gu_router() else 1
        return passes * ((route + per_layer * sh.layers) if sh.chained
                         else (route + per_layer) * sh.layers)

    def io_bytes_per_step(self):
        """Host <-> device bytes of one step's input and output (f32)."""
        sh = self.shape
        n = sh.tokens * sh.hidden * 4
        return (n, n) if sh.chained else (sh.layers * n, sh.layers * n)

    def kernel_bytes(self, kernel, steps):
        """Algorithmic bytes of every launch of one kernel over the given steps.
        gate/up: gate and up nibbles + scales of the layer's distinct routed
        experts and its shared experts, x in, h out.  down: down nibbles +
        scales of the same experts, h in, residual in, output out, and the
        next layer's router weights (the routing that follows in its tail).
        The one-token layer kernel: every used expert's whole record, x in,
        output out, and the next layer's router weights."""
        c, sh = self.coli, self.shape
        T, H, F, E, S, k = sh.tokens, sh.hidden, sh.ffn, sh.experts, sh.shared, sh.top_k
        uniq = (self.counts[steps] > 0).sum(dim=2).cpu().numpy()          # [K, L]
        n_exp = uniq + S
        h_bytes = T * (k + S) * F * 4
        rb = sh.experts * sh.hidden * (2 if sh.router_dtype == "bf16" else 4)
        n_route = len(steps) * (1 if sh.chained else sh.layers)
        if kernel == c.COLI_KERNEL_GATEUP:
            # with the first layer's router inside: its router weights too
            per_exp = 2 * (F * H // 2 + 4 * F * H // 64)
            router = n_route * rb if self.gu_router() else 0
            return int((n_exp * per_exp).sum() + uniq.size * (T * H * 4 + h_bytes) + router)
        if kernel == c.COLI_KERNEL_DOWN:
            per_exp = H * F // 2 + 4 * H * F // 64
            next_router = rb * (sh.layers - 1) * len(steps) if sh.chained else 0
            return int((n_exp * per_exp).sum() + uniq.size * (h_bytes + 2 * T * H * 4)
                       + next_router)
        if kernel == c.COLI_KERNEL_LAYER:
            per_exp = self.eb + 4 * self.es
            next_router = rb * (sh.layers - 1) * len(steps) if sh.chained else 0
            return int((n_exp * per_exp).sum() + uniq.size * 2 * T * H * 4 + next_router)
        return int(n_route * (rb + T * H * 4))

    def algorithmic_bytes(self, steps):
        """Bytes the method must move for the given steps: packed nibbles and
        scales of every distinct expert each layer routed to, the shared
        experts, the router weights, x in and out."""
        sh = self.shape
        per_expert = self.eb + 4 * self.es
        cnt = self.counts[steps].cpu().numpy()             # [K, L, E]
        unique = (cnt > 0).sum()
        router_b = sh.experts * sh.hidden * (2 if sh.router_dtype == "bf16" else 4)
        per_step_fixed = sh.layers * (sh.shared * per_expert + router_b + 2 * sh.tokens * sh.hidden * 4)
        return int(unique * per_expert + len(steps) * per_step_fixed), int(unique)


class PrefillWorkload:
    """One batched (prefill) layer resident in HBM: experts, a skewed router and
    a fresh batch of tokens per step."""

    def __init__(self, shape, steps_total, dev, seed=0, fmt="i4g"):
        import int4_expert_ffn_gb300 as pkg
        from int4_expert_ffn_gb300 import synth
        self.coli = c = pkg.binding
        self.shape = shape
        H, F, E, S, T = shape.hidden, shape.ffn, shape.experts, shape.shared, shape.tokens
        self.fmt = {"i4g": c.COLI_FMT_I4G, "mxfp4": c.COLI_FMT_MXFP4, "fp8": c.COLI_FMT_FP8,
                    "i4row": c.COLI_FMT_I4ROW}[fmt]
        quant, sdt = {"i4g": (c.coli_quant_i4g, torch.float32),
                      "mxfp4": (c.coli_quant_mxfp4, torch.uint8),
                      "fp8": (c.coli_quant_fp8b128, torch.float32),
                      "i4row": (c.coli_quant_i4row, torch.float32)}[fmt]
        esz = torch.tensor([], dtype=sdt).element_size()
        self.eb = c.coli_fmt_expert_bytes(self.fmt, H, F)
        self.es = c.coli_fmt_expert_scale_bytes(self.fmt, H, F) // esz
        n = E + S
        self.packed = torch.empty(n * self.eb, dtype=torch.uint8, device=dev)
        self.scales = torch.empty(n * self.es, dtype=sdt, device=dev)
        p0 = s0 = 0
        for e in range(n):
            for m in range(3):
                w = synth.expert_matrix(shape, 0, e, m, seed, device=dev)
                rows, cols = w.shape
                nb = rows * c.lib.coli_fmt_row_bytes(self.fmt, cols)
                ns = rows * c.lib.coli_fmt_scale_bytes(self.fmt, cols) // esz
                quant(w, self.packed[p0:p0 + nb].view(rows, -1),
                      self.scales[s0:s0 + ns].view(rows, -1))
                p0 += nb
                s0 += ns
        self.router = synth.router_weights(shape, 0, seed, device=dev,
                                           row_std=synth.skewed_router_std(E, H))
        self.x = torch.stack([synth.tokens(shape, seed, i, device=dev)
                              for i in range(steps_total)]).contiguous()
        self.out = torch.empty((T, H), dtype=torch.float32, device=dev)
        self.counts = torch.zeros((steps_total, E), dtype=torch.int32, device=dev)
        self.desc = c.MoEDesc(H, F, E, S, T, c.COLI_BF16 if shape.x_dtype == "bf16" else c.COLI_F32,
                              c.COLI_BF16 if shape.router_dtype == "bf16" else c.COLI_F32,
                              weight_fmt=self.fmt)
        self.ws = c.new_workspace(self.desc, shape.top_k)
        torch.cuda.synchronize()

    def step(self, i, stream=None, x=None, out=None):
        self.coli.coli_moe_forward(self.desc, self.shape.top_k, self.x[i] if x is None else x,
                                   self.router, self.packed, self.scales, self.ws,
                                   out=self.out if out is None else out,
                                   route_counts=self.counts[i], stream=stream)

    def gemm_flops(self):
        """Algorithmic FLOPs of one call's expert GEMMs: (gate/up, down)."""
        sh = self.shape
        routes = sh.tokens * (sh.top_k + sh.shared)
        return 2 * routes * 2 * sh.hidden * sh.ffn, 2 * routes * sh.hidden * sh.ffn

    def flops_per_step(self):
        sh = self.shape
        gu, dn = self.gemm_flops()
        return gu + dn + 2 * sh.tokens * sh.experts * sh.hidden


def run_prefill(args, shape, dev, world):
    steps, warmup = args.steps, args.warmup
    wl = PrefillWorkload(shape, warmup + steps, dev, fmt=args.weight_fmt)
    c = wl.coli
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for i in range(warmup):
            wl.step(i, stream=stream)
    stream.synchronize()
    sampler = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                           else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[0]))
    sampler.start()
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(warmup, warmup + steps):
            wl.step(i, stream=stream)
        ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world)
    time.sleep(0.15)
    sampler.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    # the two grouped GEMMs, each bracketed by events in a separate pass
    kern = {}
    gu_f, dn_f = wl.gemm_flops()
    for name, kid, fl in (("k_pgemm_gateup", c.COLI_KERNEL_PREFILL_GATEUP, gu_f),
                          ("k_pgemm_down", c.COLI_KERNEL_PREFILL_DOWN, dn_f)):
        before = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        after = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for e in before + after:
            e.record(stream)
        stream.synchronize()
        c.coli_profile_events(kid, before, after)
        try:
            with torch.cuda.stream(stream):
                for i in range(warmup, warmup + steps):
                    wl.step(i, stream=stream)
        finally:
            got = c.coli_profile_events(kid, [], [])
        torch.cuda.synchronize()
        assert got == steps
        us = float(np.mean([b.elapsed_time(a) for b, a in zip(before, after)])) * 1e3
        kern[name] = {"launches": steps, "us_per_launch": us, "flops_per_launch": fl,
                      "tflops": fl / (us * 1e-6) / 1e12}
    # end to end: bf16 tokens from pinned host memory in, f32 output back
    host_x = wl.x.cpu().pin_memory()
    host_out = torch.empty((steps, shape.tokens, shape.hidden), dtype=torch.float32).pin_memory()
    dx = torch.empty_like(wl.x[0])
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(steps):
            dx.copy_(host_x[warmup + i], non_blocking=True)
            wl.step(warmup + i, stream=stream, x=dx)
            host_out[i].copy_(wl.out, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e = {"value": world * steps * shape.tokens / (e2e_ms / 1e3), "unit": "tokens/s",
           "h2d_bytes_per_step": shape.tokens * shape.hidden * 2,
           "d2h_bytes_per_step": shape.tokens * shape.hidden * 4}
    hot = wl.counts[warmup:].sum(0).cpu().numpy()
    top32 = float(np.sort(hot)[::-1][:32].sum() / max(1, hot.sum()))
    res = {"tokens_per_rank": steps * shape.tokens, "ms": ms, "clocks": sampler.summary(t0, t1),
           "kernels": kern, "e2e": e2e, "launches": steps * 9, "top32_share": top32,
           "flops_per_step": wl.flops_per_step()}
    return wl, res


def capture_graphs(wl, idxs, stream):
    graphs = []
    for i in idxs:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            wl.step(i, stream=stream)
        graphs.append(g)
    return graphs


def run_decode(args, shape, dev, world, rank):
    steps, warmup = args.steps, args.warmup
    wl = DecodeWorkload(shape, warmup + steps, dev, router=getattr(args, "router", "softmax"))
    stream = torch.cuda.Stream(device=dev)
    # eager warm-up (first launches, module load), then graphs of each step
    with torch.cuda.stream(stream):
        wl.step(0, stream=stream)
    stream.synchronize()
    graphs = capture_graphs(wl, range(warmup + steps), stream)
    wl.counts.zero_()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(warmup):
            graphs[i].replay()
        # soak: keep the GPU at its steady clock before timing (untimed)
        t_soak = time.time()
        while time.time() - t_soak < 0.3:
            for i in range(warmup):
                graphs[i].replay()
            stream.synchronize()
    sampler = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                           else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[0]))
    sampler.start()
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    windows = []
    t0 = time.time()
    for _ in range(args.repeats):
        # each window: exactly K steps, barrier and synchronize on both sides
        wl.counts.zero_()
        barrier(world)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for i in range(warmup, warmup + steps):
                graphs[i].replay()
            ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        windows.append(ev0.elapsed_time(ev1))
    t1 = time.time()
    time.sleep(0.15)
    sampler.stop()
    ms = statistics.median(windows)
    ms_max = max_over_ranks(ms, world, dev)
    tokens = steps * shape.tokens
    alg_bytes, n_unique = wl.algorithmic_bytes(list(range(warmup, warmup + steps)))
    res = {
        "tokens_per_rank": tokens,
        "ms": ms_max,
        "windows_ms": [round(w, 4) for w in windows],
        "alg_bytes": alg_bytes,
        "unique_experts": n_unique,
        "clocks": sampler.summary(t0, t1),
        "launches": steps * wl.kernels_per_step(),
    }
    del graphs
    c = wl.coli
    kset = ((("k_layer1", c.COLI_KERNEL_LAYER),) if wl.fused() else
            (("k_gateup", c.COLI_KERNEL_GATEUP), ("k_down", c.COLI_KERNEL_DOWN)))
    res["kernels"] = {name: kernel_timing(wl, args, stream, kid) for name, kid in kset}
    res["e2e"] = run_e2e(wl, args, dev, world, stream)
    return wl, res


def kernel_timing(wl, args, stream, kernel):
    """Average launch duration of one kernel of the layer forward over the same
    steps as the timed region: the steps' graphs are captured again with CUDA
    event pairs around every launch of `kernel` (recorded on the launch
    stream) and replayed once.  The bracketing events serialise that kernel
    behind its predecessor, so this replay is kept apart from the timed step
    region; its own step time is reported beside the result."""
    c = wl.coli
    sh = wl.shape
    steps, warmup = args.steps, args.warmup
    per_step = sh.layers if kernel != c.COLI_KERNEL_ROUTE else 1
    n = steps * per_step
    before = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    after = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in before + after:     # torch creates the CUDA event on first record
        e.record(stream)
    stream.synchronize()
    c.coli_profile_events(kernel, before, after)
    try:
        graphs = capture_graphs(wl, range(warmup, warmup + steps), stream)
    finally:
        got = c.coli_profile_events(kernel, [], [])
    assert got == n, "bracketed %d launches, expected %d" % (got, n)
    save = wl.counts.clone()
    wl.counts.zero_()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for g in graphs:
            g.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    durations = np.array([b.elapsed_time(a) for b, a in zip(before, after)]) * 1e3   # us
    counts_ok = torch.equal(wl.counts[warmup:warmup + steps], save[warmup:warmup + steps])
    wl.counts.copy_(save)
    del graphs
    alg = wl.kernel_bytes(kernel, list(range(warmup, warmup + steps)))
    return {"launches": n, "us_per_launch": float(durations.mean()),
            "us_median": float(np.median(durations)), "total_ms": float(durations.sum() / 1e3),
            "alg_bytes_per_launch": alg / n,
            "bracketed_ms_per_step": ev0.elapsed_time(ev1) / steps,
            "same_routes": bool(counts_ok)}


def run_e2e(wl, args, dev, world, stream):
    """Same metric through the public API with host buffers: each step copies its
    input from pinned host memory, runs the stack, and reads the output back."""
    sh = wl.shape
    steps, warmup = args.steps, args.warmup
    n = warmup + steps
    host_x = wl.x.cpu().pin_memory()
    host_out = torch.empty(tuple(wl.out.shape), dtype=torch.float32).pin_memory()
    dx = torch.empty(tuple(wl.x.shape[1:]), dtype=torch.float32, device=dev)
    dout = torch.empty(tuple(wl.out.shape[1:]), dtype=torch.float32, device=dev)
    graphs = []
    for i in range(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            dx.copy_(host_x[i], non_blocking=True)
            wl.step(i, stream=stream, x=dx, out=dout)
            host_out[i].copy_(dout, non_blocking=True)
        graphs.append(g)
    with torch.cuda.stream(stream):
        for i in range(warmup):
            graphs[i].replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(warmup, n):
            graphs[i].replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    assert torch.equal(host_out[warmup:n], wl.out[warmup:n].cpu()), "e2e output mismatch"
    bi, bo = wl.io_bytes_per_step()
    return {"value": world * steps * sh.tokens / (ms / 1e3), "unit": "tokens/s",
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo}


# ---------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample of the same workload


def cpu_model():
    """Name of the host CPU: lscpu's model name, else /proc/cpuinfo's (x86
    "model name", Arm "CPU implementer" / "CPU part")."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    info = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    info.setdefault(k.strip().lower(), v.strip())
    except OSError:
        return "unknown"
    if "model name" in info:
        return info["model name"]
    if "cpu part" in info:
        return "arm implementer %s part %s" % (info.get("cpu implementer", "?"), info["cpu part"])
    return "unknown"


def oracle_baseline(shape, dev, budget_s=24.0, seed=0):
    """Time the oracle (as it stands) on fresh tokens through layer 0 of the
    workload and scale to tokens/s of the whole step (every layer has the
    same shape and cost).  Two legs on the host cores: the single-threaded
    build, one token at a time, and the OpenMP build over nproc threads, one
    token per thread (each leg about budget_s / 2 of oracle time, at least one
    batch).  Expert quantisation by the oracle is set-up, not timed."""
    import oracle as orc
    from int4_expert_ffn_gb300 import synth
    H, F, E, S, k = shape.hidden, shape.ffn, shape.experts, shape.shared, shape.top_k
    nproc = os.cpu_count() or 1
    wr = synth.router_weights(shape, 0, seed, device=dev).double().cpu().numpy()
    eb = orc.expert_packed_bytes(H, F)
    es = orc.expert_scales(H, F)
    packed = np.zeros((E + S) * eb, np.uint8)
    scales = np.zeros((E + S) * es, np.float32)
    done = set()

    def materialise(experts):
        prev = orc.set_threads(nproc)
        try:
            for e in experts:
                if e in done:
                    continue
                ps, ss = [], []
                for m in range(3):
                    w = synth.expert_matrix(shape, 0, e, m, seed, device=dev).float().cpu().numpy()
                    p, s = orc.quant_i4g(w)
                    ps.append(p.reshape(-1))
                    ss.append(s.reshape(-1))
                packed[e * eb:(e + 1) * eb] = np.concatenate(ps)
                scales[e * es:(e + 1) * es] = np.concatenate(ss)
                done.add(e)
        finally:
            orc.set_threads(prev)

    materialise(range(E, E + S))
    per_step_calls = shape.layers * shape.tokens   # token-layers per step
    legs = {}
    next_tok = 10_000
    for name, threads, batch in (("single", 1, 1), ("nproc", nproc, nproc)):
        n_tok, spent = 0, 0.0
        while spent < budget_s / 2 and n_tok < 4 * batch + 64:
            x = torch.cat([synth.tokens(shape, seed, next_tok + i, device=dev)[:1]
                           for i in range(batch)]).double().cpu().numpy()
            next_tok += batch
            lg = orc.router_logits(x, wr)
            materialise(sorted({int(e) for row in lg for e in np.argsort(-row)[:k + 2]}))
            prev = orc.set_threads(threads)
            try:
                t = time.perf_counter()
                orc.moe_forward(x, wr, packed, scales, H, F, E, S, k)
                spent += time.perf_counter() - t
            finally:
                orc.set_threads(prev)
            n_tok += batch
        per_token_layer = spent / n_tok
        legs[name] = {
            "value": shape.tokens / (per_token_layer * per_step_calls), "cores": threads,
            "sample": "%d fresh tokens through layer 0 (%.1f s of oracle time, %s), scaled to "
                      "the %d layer calls of a step" % (
                          n_tok, spent, "single-threaded build" if threads == 1 else
                          "OpenMP build, %d threads, one token per thread" % threads,
                          per_step_calls)}
    best = legs["nproc"]
    return {"value": best["value"], "unit": "tokens/s", "cores": best["cores"], "kind": "oracle",
            "sample": best["sample"], "cpu_model": cpu_model(), "nproc": nproc,
            "single_thread": legs["single"]}


# ---------------------------------------------------------------------------


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="coli", choices=["coli", "reference"])
    ap.add_argument("--workload", default="glm_decode_b1",
                    choices=["olmoe_decode", "glm_decode_b1", "glm_decode_b8", "glm_prefill",
                             "quant", "glm_tiered"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--repeats", type=int, default=20,
                    help="decode workloads: timed windows of K steps (the line reports the "
                         "median window)")
    ap.add_argument("--layers", type=int, default=None,
                    help="override the stack depth (small profiling cases only)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the batch size (small profiling cases only)")
    ap.add_argument("--experts", type=int, default=None,
                    help="quant workload: experts converted per step (default 256; smaller for "
                         "profiling captures)")
    ap.add_argument("--weight-fmt", default="i4g", choices=["i4g", "mxfp4", "fp8", "i4row"],
                    help="glm_prefill: the expert weight container (int4-grouped g64, MXFP4, "
                         "fp8-e4m3-b128, int4-row)")
    ap.add_argument("--router", default="softmax", choices=["softmax", "sigmoid"],
                    help="decode workloads: softmax routing, or the GLM router (sigmoid "
                         "scores with a per-layer selection bias)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)

    from int4_expert_ffn_gb300 import synth
    if args.workload == "glm_tiered":
        from int4_expert_ffn_gb300 import build as b
        if rank == 0:
            b.build()
        emit_tiered(args, dev, world, rank)
        return
    if args.workload == "quant":
        from int4_expert_ffn_gb300 import build as b
        if rank == 0:
            b.build()
        emit_quant(args, dev, world, rank)
        return
    shape = synth.SHAPES[args.workload]
    if args.layers is not None or args.tokens is not None:
        import dataclasses
        shape = dataclasses.replace(shape, layers=args.layers or shape.layers,
                                    tokens=args.tokens or shape.tokens)
    config = {"workload": "%s: %d MoE layers, hidden %d, %d experts of FFN width %d, top-%d, "
                          "%d shared, batch %d, int4-grouped g64 f32 scales, %s router%s"
                          % (shape.name, shape.layers, shape.hidden, shape.experts, shape.ffn,
                             shape.top_k, shape.shared, shape.tokens, shape.router_dtype,
                             ", sigmoid scores + selection bias" if args.router == "sigmoid"
                             else ""),
              "layers": shape.layers, "hidden": shape.hidden, "experts": shape.experts,
              "ffn": shape.ffn, "top_k": shape.top_k, "shared": shape.shared,
              "batch": shape.tokens, "parallelism": "replicas" if world > 1 else "single",
              "inputs": ("a fresh batch of N(0,1) tokens each step" if shape.layers == 1 else
                         "layer 0 takes a fresh N(0,1) token each step; layer l>0 takes "
                         "x_l + MoE_l(x_l)" if shape.chained else
                         "every layer takes its own fresh N(0,1) input each step"),
              "l2": "inputs larger than L2: %.2f GB of experts resident, fresh routing each step",
              "timing": "median of %d windows of %d steps (CUDA events on the launch stream)"
                        % (args.repeats, args.steps)}

    if args.impl == "reference":
        if rank == 0:
            base = oracle_baseline(shape, dev)
            line = {"metric": METRIC, "value": base["value"], "unit": "tokens/s",
                    "impl": "reference", "n_gpus": args.gpus, "steps": args.steps,
                    "warmup": args.warmup, "higher_is_better": True, "dtype": "f64",
                    "data": "synthetic", "config": dict(config, l2="n/a (CPU)",
                                                        timing="oracle wall time on the host "
                                                               "cores (perf_counter)"),
                    "cpu_baseline": base,
                    "e2e": {"value": base["value"], "unit": "tokens/s",
                            "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
            print(json.dumps(line), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    from int4_expert_ffn_gb300 import build as b
    if rank == 0:
        b.build()
    barrier(world)
    if shape.name == "glm_prefill":
        emit_prefill(args, shape, dev, world, rank, config)
        return
    wl, res = run_decode(args, shape, dev, world, rank)
    resident = wl.packed.numel() + 4 * wl.scales.numel()
    config["l2"] = config["l2"] % (resident / 1e9)
    hbm_peak, _, peak_kind = read_peaks()
    sec = res["ms"] / 1e3
    value = world * res["tokens_per_rank"] / sec
    gbs = res["alg_bytes"] / sec / 1e9
    kern = res["kernels"]
    dom = max(kern, key=lambda n: kern[n]["total_ms"])
    kd = kern[dom]
    k_gbs = kd["alg_bytes_per_launch"] / (kd["us_per_launch"] * 1e-6) / 1e9
    traffic = NCU_TRAFFIC.get(args.workload, {}).get(dom)
    earlier = NCU_TRAFFIC_EARLIER.get(args.workload, {}).get(dom) if traffic is None else None
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms"] / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("int4 weights x 15-bit fixed-point activations (dp4a, exact int32 dot), "
                  "f32 scale and accumulate"),
        "data": "synthetic (seeded; weights N(0,0.02) bf16 quantised on the GPU)",
        "config": config,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": k_gbs, "peak": hbm_peak,
                     "unit": "GB/s", "frac": k_gbs / hbm_peak,
                     "peak_kind": "%s (hbm_gbs, burst copy)" % peak_kind,
                     "traffic": traffic,
                     **({"traffic_earlier_build": earlier, "traffic_note": EARLIER_NOTE}
                        if earlier is not None else {}),
                     "alg_bytes_per_launch": kd["alg_bytes_per_launch"],
                     "us_per_launch": kd["us_per_launch"]},
        "step_roofline": {"achieved": gbs, "unit": "GB/s", "frac": gbs / hbm_peak,
                          "alg_bytes_per_step": res["alg_bytes"] / args.steps},
        "kernels": kern,
        "clocks": res["clocks"],
        "e2e": res["e2e"],
        "gpu_launches": res["launches"],
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_baseline(shape, dev)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def emit_quant(args, dev, world, rank):
    """Quantiser workload: 256 experts x {gate, up [2048, 6144], down [6144, 2048]}
    bf16 N(0, 0.02) with 1% outliers x20, one call per matrix kind (all experts'
    rows stacked).  Bytes moved: bf16 in, nibbles and f32 scales out."""
    import int4_expert_ffn_gb300 as pkg
    from int4_expert_ffn_gb300 import synth
    c = pkg.binding
    E, F, H = args.experts or 256, 2048, 6144
    kinds = [(F, H), (F, H), (H, F)]
    mats = []
    for m, (rows, cols) in enumerate(kinds):
        w = torch.empty((E * rows, cols), dtype=torch.bfloat16, device=dev)
        for e in range(E):
            w[e * rows:(e + 1) * rows] = synth.matrix(rows, cols, 0.02, 0, 5, e, m, device=dev,
                                                      outliers=0.01)
        packed = torch.empty((E * rows, cols // 2), dtype=torch.uint8, device=dev)
        scales = torch.empty((E * rows, cols // 64), dtype=torch.float32, device=dev)
        mats.append((w, packed, scales))
    elems = sum(w.numel() for w, _, _ in mats)
    nbytes = sum(w.numel() * 2 + p.numel() + 4 * s.numel() for w, p, s in mats)
    stream = torch.cuda.Stream(device=dev)

    def step():
        for w, p, s in mats:
            c.coli_quant_i4g(w, p, s, stream=stream)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                           else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[0]))
    sampler.start()
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    sampler.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev) / args.steps
    hbm_peak, _, peak_kind = read_peaks()
    gbs = nbytes / (ms / 1e3) / 1e9
    line = {
        "metric": "int4-grouped quantiser throughput (elements/s; bytes moved vs HBM peak)",
        "value": world * elems / (ms / 1e3), "unit": "elements/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16 -> u8 + f32",
        "data": "synthetic (seeded bf16 N(0,0.02), 1% outliers x20)",
        "config": {"workload": "quantiser: %d experts x {gate, up [2048,6144], down [6144,2048]}" % E,
                   "elements": elems, "bytes_per_step": nbytes,
                   "l2": "inputs larger than L2 (%.1f GB)" % (nbytes / 1e9)},
        # a launch here covers E experts' matrices of the 16-expert capture's
        # shape, so a capture scales by E / 16
        "roofline": {"bound": "hbm", "kernel": "k_quant_vec", "achieved": gbs, "peak": hbm_peak,
                     "unit": "GB/s", "frac": gbs / hbm_peak, "peak_kind": peak_kind,
                     "traffic": None,
                     "traffic_earlier_build": NCU_TRAFFIC_EARLIER["quant16"]["k_quant_vec"] * E / 16,
                     "traffic_note": EARLIER_NOTE + " (a 16-expert capture, scaled by experts)"},
        "clocks": sampler.summary(t0, t1), "gpu_launches": 3 * args.steps,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def emit_tiered(args, dev, world, rank):
    """Tiered store workload: one GLM-like layer (hidden 6144, 256 routed
    experts of width 2048, top-8, 1 shared) whose full store (5.46 GB) sits in
    pinned host memory, with an HBM pool of 128 slots holding the shared expert
    and 127 routed experts at the start; batch 1 decode through the layer
    with the skewed router (32 experts take about half of the routes), one LFRU
    tick (and its uploads) after every call.  A step = one token's forward plus
    its policy tick; missing experts are read over the host link by the expert
    GEMVs themselves."""
    import int4_expert_ffn_gb300 as pkg
    from int4_expert_ffn_gb300 import synth
    c = pkg.binding
    shape = dataclasses.replace(synth.GLM_DECODE_B1, name="glm_tiered", layers=1)
    H, F, E, S, k = shape.hidden, shape.ffn, shape.experts, shape.shared, shape.top_k
    eb, es = c.coli_expert_packed_bytes(H, F), c.coli_expert_scale_count(H, F)
    rec = eb + 4 * es
    steps, warmup = args.steps, args.warmup
    packed = torch.empty((E + S) * eb, dtype=torch.uint8, device=dev)
    scales = torch.empty((E + S) * es, dtype=torch.float32, device=dev)
    p0 = s0 = 0
    for e in range(E + S):
        for m in range(3):
            w = synth.expert_matrix(shape, 0, e, m, 0, device=dev)
            rows, cols = w.shape
            nb, ns = rows * cols // 2, rows * cols // 64
            c.coli_quant_i4g(w, packed[p0:p0 + nb].view(rows, -1), scales[s0:s0 + ns].view(rows, -1))
            p0 += nb
            s0 += ns
    host_p = packed.cpu().pin_memory()
    host_s = scales.cpu().pin_memory()
    del packed, scales
    torch.cuda.empty_cache()
    wr = synth.router_weights(shape, 0, 0, device=dev, row_std=synth.skewed_router_std(E, H))
    xs = torch.stack([synth.tokens(shape, 0, i, device=dev) for i in range(warmup + steps)])
    desc = c.MoEDesc(H, F, E, S, 1, c.COLI_F32, c.COLI_BF16)
    n_slots = 128
    owners = [E] + list(range(1, 2 * (n_slots - 1), 2))     # the shared expert, odd-numbered routed
    ws = c.new_workspace(desc, k)
    stream = torch.cuda.Stream(device=dev)
    counts = torch.zeros((warmup + steps, E), dtype=torch.int32, device=dev)
    out = torch.empty((warmup + steps, 1, H), dtype=torch.float32, device=dev)

    def run(tier, i0, i1):
        for i in range(i0, i1):
            c.coli_moe_forward_tiered(desc, k, xs[i], wr, host_p, host_s, tier, ws, out=out[i],
                                      route_counts=counts[i], stream=stream)
            c.coli_tier_update(desc, counts[i], host_p, host_s, tier, stream=stream)

    # host-link reference: a pinned host -> HBM copy of 2 GB by the copy engine
    hbuf = torch.empty(2 << 30, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(2 << 30, dtype=torch.uint8, device=dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = 1e9
    for _ in range(3):
        with torch.cuda.stream(stream):
            ev0.record(stream)
            dbuf.copy_(hbuf, non_blocking=True)
            ev1.record(stream)
        torch.cuda.synchronize()
        best = min(best, ev0.elapsed_time(ev1))
    link_gbs = (2 << 30) / (best / 1e3) / 1e9
    del hbuf, dbuf
    # timed: warm-up steps, then K steps, from a fresh placement
    tier = c.Tier(desc, owners, max_uploads=8, device=dev)
    c.coli_tier_place(desc, host_p, host_s, tier, stream=stream)
    with torch.cuda.stream(stream):
        run(tier, 0, warmup)
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                           else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[0]))
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        run(tier, warmup, warmup + steps)
        ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world)
    time.sleep(0.15)
    sampler.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    # the same sequence again from the same placement, one step at a time, to
    # count what the timed steps read from host memory and uploaded (the
    # policy is deterministic: same inputs, same placements)
    tier2 = c.Tier(desc, owners, max_uploads=8, device=dev)
    c.coli_tier_place(desc, host_p, host_s, tier2, stream=stream)
    cnt2 = torch.zeros_like(counts)
    host_bytes = up_bytes = resident_used = used = 0
    for i in range(warmup + steps):
        slot_of = tier2.slot_of[:E].clone()
        with torch.cuda.stream(stream):
            c.coli_moe_forward_tiered(desc, k, xs[i], wr, host_p, host_s, tier2, ws,
                                      route_counts=cnt2[i], stream=stream)
            c.coli_tier_update(desc, cnt2[i], host_p, host_s, tier2, stream=stream)
        torch.cuda.synchronize()
        if i < warmup:
            continue
        u = (cnt2[i] > 0)
        miss = int((u & (slot_of < 0)).sum())
        used += int(u.sum())
        resident_used += int(u.sum()) - miss
        host_bytes += miss * rec
        up_bytes += int(tier2.uploads[0]) * rec
    assert torch.equal(cnt2[warmup:], counts[warmup:]), "the replay routed differently"
    sec = ms / 1e3
    hbm_peak, _, peak_kind = read_peaks()
    line = {
        "metric": "MoE decode tokens/s over a tiered expert store (HBM pool + pinned host memory)",
        "value": world * steps / sec, "unit": "tokens/s", "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": ms / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("int4 weights x 15-bit fixed-point activations (dp4a, exact int32 dot), "
                  "f32 scale and accumulate"),
        "data": "synthetic (seeded; weights N(0,0.02) bf16 quantised on the GPU)",
        "config": {"workload": "glm_tiered: 1 MoE layer, hidden 6144, 256 experts of FFN width "
                               "2048, top-8, 1 shared, batch 1; store of 257 experts (%.2f GB) "
                               "in pinned host memory, HBM pool of %d slots (the shared expert "
                               "and 127 routed at the start); skewed router; one LFRU tick and "
                               "its uploads after every call" % ((E + S) * rec / 1e9, n_slots),
                   "l2": "inputs larger than L2"},
        "host_link": {"read_gbs": host_bytes / sec / 1e9, "upload_gbs": up_bytes / sec / 1e9,
                      "peak_gbs": link_gbs,
                      "peak_kind": "measured: pinned host -> HBM copy of 2 GB by the copy engine",
                      "frac": (host_bytes + up_bytes) / sec / 1e9 / link_gbs,
                      "host_bytes_per_step": host_bytes / steps,
                      "upload_bytes_per_step": up_bytes / steps,
                      "resident_hit_rate": resident_used / max(1, used)},
        "roofline": {"bound": "hbm", "kernel": "whole step", "achieved": None, "peak": hbm_peak,
                     "unit": "GB/s", "frac": None, "peak_kind": peak_kind, "traffic": None,
                     "note": "the host link bounds this workload; see host_link"},
        "clocks": sampler.summary(t0, t1), "gpu_launches": steps * 5,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def emit_prefill(args, shape, dev, world, rank, config):
    """Bench line of the batched (prefill) layer: tokens/s, with the dominant
    grouped GEMM's tensor throughput as the roofline."""
    wl, res = run_prefill(args, shape, dev, world)
    _, tf_peak, peak_kind = read_peaks()
    sec = res["ms"] / 1e3
    kern = res["kernels"]
    dom = max(kern, key=lambda n: kern[n]["us_per_launch"])
    kd = kern[dom]
    fmt_name = {"i4g": "int4-grouped g64 f32 scales",
                "mxfp4": "MXFP4 (E2M1 codes, E8M0 scale per 32)",
                "fp8": "fp8-e4m3-b128 (E4M3 codes, f32 scale per 128)",
                "i4row": "int4-row (nibbles, one f32 scale per row)"}[args.weight_fmt]
    config = dict(config, l2="inputs larger than L2: %.2f GB of experts resident"
                  % ((wl.packed.nbytes + wl.scales.nbytes) / 1e9),
                  weight_fmt=args.weight_fmt,
                  timing="one window of %d steps (CUDA events on the launch stream)" % args.steps,
                  workload=config["workload"].replace("int4-grouped g64 f32 scales", fmt_name),
                  routing="skewed router: the 32 most-used experts took %.1f%% of routes"
                  % (100 * res["top32_share"]))
    line = {
        "metric": "MoE prefill tokens/s (batched grouped GEMMs on tcgen05, %s weights)"
                  % args.weight_fmt,
        "value": world * res["tokens_per_rank"] / sec, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms"] / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp16 operands, f32 accumulate",
        "data": "synthetic (seeded; weights N(0,0.02) bf16 quantised on the GPU; bf16 tokens)",
        "config": config,
        "roofline": {"bound": "tensor", "kernel": dom, "achieved": kd["tflops"], "peak": tf_peak,
                     "unit": "TFLOP/s", "frac": kd["tflops"] / tf_peak,
                     "peak_kind": "%s bf16 burst (fp16 has the same nominal dense rate)" % peak_kind,
                     "traffic": None, "flops_per_launch": kd["flops_per_launch"],
                     "us_per_launch": kd["us_per_launch"]},
        "step_tflops": res["flops_per_step"] * args.steps / sec / 1e12,
        "kernels": kern, "clocks": res["clocks"], "e2e": res["e2e"],
        "gpu_launches": res["launches"],
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
