#!/usr/bin/env python
"""Split-KV sparse-MLA decode benchmark: µs per call and HBM GB/s (fraction of the
measured HBM peak) across s_q x num_splits, on synthetic data shaped like the
FlashMLA PR #25 workload (h_q = 64, d_qk = 576, d_v = 512, topk = 128 + 512,
one bf16 latent KV cache of 131072 rows, FP8 e4m3 output with a per-tensor scale).

One "step" is one decode call through mla_sparse_decode: the split kernel plus
the combine, or the direct-epilogue kernel when the plan picks one split, with
inputs resident in HBM. The K timed steps are K consecutive calls rotating over
per-layer KV caches and query / index sets whose reads exceed L2 several times
(as the layers of a model do), replayed as CUDA graphs and bracketed by one pair
of CUDA events on the launching stream. The line also carries an s_q x
num_splits sweep (with the balanced schedule and bf16 partials where they
apply) and the dense FP8 GQA variant's sweep (the same partial / LSE protocol).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--s-q 96] [--impl ours|reference]

Prints one JSON line. --impl reference times the fp64 CPU oracle on the same
workload (a bounded sample per step) instead of the GPU library.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "split-KV sparse-MLA decode µs/call and HBM GB/s (% roofline) vs s_q x splits"
N_KV = 131072
TOPK = 640
H_Q, D_QK, D_V = 64, 576, 512
INV_SCALE = 64.0
SWEEP_SQ = (1, 6, 16, 96, 384)
SWEEP_S = (1, 2, 4, 8, 16)
# more tokens than SMs: the one-split grid with its last wave cut (planner) against
# the uncut grid (forced one split); 160 leaves 8 tokens in the last wave on 152
# SMs (cut into splits), 228 leaves 76 (two dim groups each)
TAIL_SQ = (160, 228)
BF16_PARTIALS_SQ, BF16_PARTIALS_S = 16, (8, 0)   # sweep points also run with bf16 partials
FLUSH_BYTES = 256 << 20


def workload_name(s_q: int) -> str:
    return (f"sparse-MLA decode, s_q={s_q}, h_q=64, d_qk=576 (512 latent + 64 RoPE), d_v=512, "
            f"bf16 KV cache {N_KV} rows ~N(0,1), topk={TOPK} (128 most recent + 512 uniform), "
            f"Q bf16 ~N(0,1), sm_scale 1/sqrt(576), no sink, FP8 e4m3 output (inv_scale {INV_SCALE:g})")


def algorithmic_bytes(s_q: int, S: int, part: str = "call", partial_bytes: int = 4) -> int:
    """Bytes the split method must move (gathered rows counted per token).

    per token: Q 64*576*2 + idx topk*4 + rows topk*1152 (+ FP8 output 64*512 + LSE 64*4 when
    the output is written); S > 1 adds the fp32 partial O + LSE, written by the split
    kernel and read by the combine: S*(64*512*4 + 64*4) each way.
    part: "call" (whole call), "split" (the split or direct kernel alone).
    partial_bytes: 4 for fp32 O partials, 2 for bf16 ones (the LSE partials stay fp32).
    """
    per_tok_in = H_Q * D_QK * 2 + TOPK * 4 + TOPK * D_QK * 2
    out = H_Q * D_V * 1 + H_Q * 4
    partial = S * (H_Q * D_V * partial_bytes + H_Q * 4)
    if S == 1:
        return s_q * (per_tok_in + out)
    if part == "split":
        return s_q * (per_tok_in + partial)
    return s_q * (per_tok_in + 2 * partial + out)


def balanced_schedule(s_q: int, nb: int, num_sms: int):
    """The balanced one-shot schedule of mla_sparse_decode, restated on the host:
    the s_q * nb 64-row blocks cut into P near-equal contiguous ranges (one CTA
    each, P the fewest reaching ceil(s_q * nb / num_sms) blocks per CTA).
    Returns (P, blocks per CTA, tokens cut by a range boundary, pieces of those)."""
    U = s_q * nb
    per = -(-U // num_sms)
    P = -(-U // per)
    base, rem = divmod(U, P)
    big = rem * (base + 1)
    cta = lambda u: u // (base + 1) if u < big else rem + (u - big) // base
    cut = pieces = 0
    for t in range(s_q):
        pa, pb = cta(t * nb), cta((t + 1) * nb - 1)
        if pa != pb:
            cut += 1
            pieces += pb - pa + 1
    return P, per, cut, pieces


def balanced_bytes(s_q: int, num_sms: int) -> int:
    """Algorithmic bytes of the balanced schedule: every token's Q, indices,
    gathered rows and FP8 output + LSE; each piece of a cut token adds an fp32
    partial (O + LSE), written by its piece and read by the combine."""
    per_tok_in = H_Q * D_QK * 2 + TOPK * 4 + TOPK * D_QK * 2
    out = H_Q * D_V * 1 + H_Q * 4
    partial = H_Q * D_V * 4 + H_Q * 4
    _, _, cut, pieces = balanced_schedule(s_q, -(-TOPK // 64), num_sms)
    return s_q * (per_tok_in + out) + 2 * pieces * partial


def point_bytes(s_q: int, splits_used: int, balanced: bool, num_sms: int) -> int:
    """Algorithmic bytes of one swept call, from the schedule the plan actually runs:
    the balanced schedule's, else the (token, split) grid's with the plan's split
    count (for the planner's point too, whose requested count is 0)."""
    return balanced_bytes(s_q, num_sms) if balanced else algorithmic_bytes(s_q, splits_used, "call")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ----------------------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms in the background."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        t0, t1 = (self.marks[0], self.marks[1]) if len(self.marks) >= 2 else (0, 1e30)
        rows = [l for (t, l) in self.lines if t0 - 0.05 <= t <= t1 + 0.05] or [l for _, l in self.lines]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------- GPU arm --

L2_FALLBACK = 129 * 1000 * 1000
MAX_LAYERS = 320


def unique_bytes(s_q: int) -> int:
    """Bytes one call reads at most (queries, indices, gathered rows), ignoring the rows
    that tokens share: the footprint a rotation of caches has to exceed."""
    return s_q * (H_Q * D_QK * 2 + TOPK * 4 + TOPK * D_QK * 2)


LAYERS_OVERRIDE = 0


def tail_shape(plan, s_q: int):
    """(first tail token, splits, dim groups) when the plan's one-split grid cuts its
    last wave (r tokens): into min(num_blocks, SMs // r) >= 3 splits (dim groups 0),
    else, when 2 r <= SMs, into two dim groups per token (splits 0); None otherwise."""
    W = plan.num_sms
    if plan.tail_ctas <= 0 or plan.num_splits != 1 or s_q <= W:
        return None
    C = min(plan.tail_ctas, W)
    r = s_q - (-(-s_q // W) - 1) * W
    st = min(plan.num_blocks, C // r)
    if st >= 3:
        return (s_q - r, st, 0)
    return (s_q - r, 0, 2) if 2 * r <= C else None


def layers_for(s_q: int, l2_bytes: int) -> int:
    """How many per-layer caches (and query/index sets) a timed run rotates through so
    that what one call reads has left L2 by the time the same layer comes round again:
    at least 3x L2 of other calls' reads, at least 4 layers, at most MAX_LAYERS (or the
    --layers count when given)."""
    if LAYERS_OVERRIDE > 0:
        return LAYERS_OVERRIDE
    return max(4, min(MAX_LAYERS, -(-3 * l2_bytes // unique_bytes(s_q))))


class Case:
    """Plan, per-layer inputs, outputs and CUDA graphs for one (s_q, S) point.

    A decode step runs once per model layer, each layer with its own KV cache, so the
    same layer's rows come round again only after every other layer's reads have
    passed through L2. The timed runs do the same: consecutive calls rotate over
    `layers` caches (views of one allocation) and per-layer queries / indices whose
    total exceeds L2 several times, back to back in one CUDA graph."""

    def __init__(self, b, torch, kv_all, qs, idxs, sm_scale, S, bf16_partials=False):
        self.b, self.torch = b, torch
        self.layers = len(qs)
        self.s_q = qs[0].shape[0]
        self.kv_all, self.qs, self.idxs, self.sm_scale = kv_all, qs, idxs, sm_scale
        dev = kv_all.device
        self.plan = b.mla_decode_plan(self.s_q, TOPK, force_splits=S) if S else b.mla_decode_plan(self.s_q, TOPK)
        if bf16_partials:
            b.mla_plan_set_partials_bf16(self.plan)
        self.S = self.plan.num_splits
        # the automatic plan's one-shot call runs the balanced schedule (one kernel)
        # when the planner enabled it and this s_q leaves >= 2 blocks per CTA
        per = -(-(self.s_q * self.plan.num_blocks) // max(self.plan.num_sms, 1))
        self.balanced = self.plan.balanced_ctas > 0 and per >= 2
        if self.balanced:
            self.P, self.per, self.cut, self.pieces = balanced_schedule(self.s_q, self.plan.num_blocks,
                                                                        self.plan.num_sms)
        # a one-split grid of more than one wave cuts its last wave's tokens into splits
        self.tail = tail_shape(self.plan, self.s_q)
        # calls on one stream run one after another, so the layers share one workspace
        self.ws = (torch.empty(self.plan.workspace_bytes, dtype=torch.uint8, device=dev)
                   if self.plan.workspace_bytes else None)
        if self.ws is not None:
            b.mla_workspace_init(self.plan, self.ws)
        self.out = torch.empty(self.s_q, H_Q, D_V, dtype=torch.uint8, device=dev)
        self.lse = torch.empty(self.s_q, H_Q, dtype=torch.float32, device=dev)
        self.stream = torch.cuda.Stream()
        self.g_call = self._capture(lambda: [self._call(l) for l in range(self.layers)])
        self.g_kernel = self._capture(lambda: [self._kernel(l) for l in range(self.layers)])
        self._single = {}

    def _call(self, l):
        self.b.mla_sparse_decode(self.plan, self.s_q, self.qs[l], self.kv_all[l], N_KV, self.idxs[l], self.sm_scale,
                                 None, "e4m3", INV_SCALE, self.out, self.lse, None, self.ws, stream=self.stream)

    def _kernel(self, l):
        # the balanced call (decode kernel + combine of the cut tokens) has no
        # entry point for its decode kernel alone: timed whole
        if self.balanced or self.S == 1:
            self._call(l)
        else:
            self.b.mla_sparse_decode_split(self.plan, self.s_q, self.qs[l], self.kv_all[l], N_KV, self.idxs[l],
                                           self.sm_scale, self.ws, stream=self.stream)

    def launches(self) -> int:
        """Kernels one call launches."""
        split_tail = self.tail is not None and self.tail[1] > 0
        return 1 if (self.S == 1 and not self.balanced and not split_tail) else 2

    def schedule(self) -> str:
        if self.balanced:
            return (f"balanced: {self.P} CTAs x <= {self.per} blocks of 64 rows; "
                    f"{self.cut} of {self.s_q} tokens cut into {self.pieces} pieces, folded by the combine")
        D = self.plan.dim_groups
        bf = ", bf16 partials" if self.plan.partial_bf16 else ""
        if self.tail is not None:
            first, st, dg = self.tail
            r = self.s_q - first
            if st:
                return (f"uniform: 1 split per token, {first} whole tokens + the last wave's {r} cut into {st} "
                        f"splits ({first + r * st} CTAs), the tail folded by the combine" + bf)
            return (f"uniform: 1 split per token, {first} whole tokens + the last wave's {r} on {dg} CTAs each "
                    f"(a share of the dims each; {first + r * dg} CTAs, no combine)")
        return f"uniform: {self.S} split(s) per token x {D} dim group(s), {self.s_q * self.S * D} CTAs" + bf

    def _capture(self, fn):
        torch = self.torch
        with torch.cuda.stream(self.stream):
            fn()                                  # eager once (warms the module, checks arguments)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            fn()
        torch.cuda.synchronize()
        return g

    def _single_graph(self, kind, l):
        key = (kind, l)
        if key not in self._single:
            self._single[key] = self._capture(lambda: (self._call if kind == "call" else self._kernel)(l))
        return self._single[key]

    def time(self, kind, steps, warmup):
        """Mean device time (µs) of `steps` consecutive calls (kind "call": the whole
        decode call; "kernel": the split / direct / balanced kernel alone), rotating
        over the layers, bracketed by one pair of CUDA events on the case's stream."""
        torch = self.torch
        graph = self.g_call if kind == "call" else self.g_kernel
        full, rest = divmod(steps, self.layers)
        singles = [self._single_graph(kind, l) for l in range(rest)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            for _ in range(max(1, -(-warmup // self.layers))):
                graph.replay()
            torch.cuda.synchronize()
            e0.record(self.stream)
            for _ in range(full):
                graph.replay()
            for g in singles:
                g.replay()
            e1.record(self.stream)
        torch.cuda.synchronize()
        return 1000.0 * e0.elapsed_time(e1) / steps

    def time_flushed(self, reps, flush):
        """Per-call time of single calls (layer 0) with L2 flushed before each, each call
        bracketed by its own pair of CUDA events (includes the event / graph-launch floor)."""
        torch = self.torch
        g = self._single_graph("call", 0)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        with torch.cuda.stream(self.stream):
            for _ in range(3):
                flush.zero_()
                g.replay()
            torch.cuda.synchronize()
            for e0, e1 in ev:
                flush.zero_()
                e0.record(self.stream)
                g.replay()
                e1.record(self.stream)
        torch.cuda.synchronize()
        return statistics.fmean(1000.0 * e0.elapsed_time(e1) for e0, e1 in ev)


DENSE_DESC = ("dense FP8 GQA split-KV SDPA decode: batch 8, 32 query / 8 KV heads, d=128, 1-16 query tokens per "
              "sequence, causal KV lengths uniform in [1024,16384], e4m3 Q/K/V ~N(0,1) with per-tensor descales, "
              "bf16 O, seed 0")


def dense_splits(skv, h_kv: int, S: int, num_sms: int):
    """Per-sequence split counts of the dense planner's adaptive rule (restated
    from sdpa_fp8_decode_plan): clamp(ceil(tiles / T), 1, S) with T the fewest
    tiles per split from ceil(sum tiles * h_kv / num_sms) up whose jobs fit
    num_sms CTAs."""
    tiles = [-(-int(k) // 128) for k in skv]
    longest = max([1] + tiles)
    jobs = lambda T: sum(min(S, max(1, -(-t // T))) for t in tiles) * h_kv
    T = max(1, -(-(sum(tiles) * h_kv) // num_sms))
    while T < longest and jobs(T) > num_sms:
        T += 1
    return [min(S, max(1, -(-t // T))) for t in tiles]


def dense_bytes(sq, skv, h_q: int, h_kv: int, d: int, S: int, splits=None) -> int:
    """Algorithmic bytes of one dense call: every sequence's K and V (e4m3, all KV
    heads), Q (e4m3), bf16 O and fp32 LSE; with splits, the fp32 partial O + LSE of
    every split a sequence uses, written by the split kernel and read by the
    combine (splits: per-sequence counts, else S for every sequence)."""
    total_q = int(sum(sq))
    kv = 2 * int(sum(skv)) * h_kv * d
    q = total_q * h_q * d
    out = total_q * h_q * (d * 2 + 4)
    if splits is None:
        splits = [S] * len(sq)
    partial = 0 if S == 1 else sum(2 * n * int(t) * h_q * (d + 1) * 4 for n, t in zip(splits, sq))
    return kv + q + out + partial


DENSE_LAYERS = 4


class DenseCase:
    """Plan, outputs and CUDA graphs for one dense split count; consecutive timed calls
    rotate over DENSE_LAYERS copies of the inputs (143 MB of K / V each), as the layers
    of a model would."""

    def __init__(self, b, torch, inp, S, layers=DENSE_LAYERS):
        self.b, self.torch, self.inp = b, torch, inp
        dev = torch.device("cuda")
        self.layers = layers
        self.sq = (inp.cu_seqlens_q[1:] - inp.cu_seqlens_q[:-1]).tolist()
        self.skv = (inp.cu_seqlens_kv[1:] - inp.cu_seqlens_kv[:-1]).tolist()
        self.total_q, self.total_kv = int(inp.cu_seqlens_q[-1]), int(inp.cu_seqlens_kv[-1])
        self.plan = b.sdpa_fp8_decode_plan(inp.batch, inp.h_q, inp.h_kv, inp.d, 16, self.total_q, max(self.skv),
                                           force_splits=S)
        self.S = self.plan.num_splits
        self.qkv = [(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)) for _ in range(layers)]
        self.cq, self.ck = inp.cu_seqlens_q.to(dev), inp.cu_seqlens_kv.to(dev)
        self.ds = [torch.tensor([x], dtype=torch.float32, device=dev)
                   for x in (inp.descale_q, inp.descale_k, inp.descale_v)]
        self.ws = (torch.empty(self.plan.workspace_bytes, dtype=torch.uint8, device=dev)
                   if self.plan.workspace_bytes else None)
        self.out = torch.empty(self.total_q, inp.h_q, inp.d, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(self.total_q, inp.h_q, dtype=torch.float32, device=dev)
        self.stream = torch.cuda.Stream()
        self.g_call = Case._capture(self, lambda: [self._call(l) for l in range(layers)])
        self.g_kernel = Case._capture(self, lambda: [self._kernel(l) for l in range(layers)])
        self._single = {}

    def _call(self, l):
        q, k, v = self.qkv[l]
        self.b.sdpa_fp8_decode(self.plan, self.total_q, self.total_kv, q, k, v, self.cq, self.ck,
                               self.ds[0], self.ds[1], self.ds[2], self.inp.sm_scale, "bf16", 1.0, self.out,
                               self.lse, None, self.ws, stream=self.stream)

    def _kernel(self, l):
        if self.S == 1:
            self._call(l)
        else:
            q, k, v = self.qkv[l]
            self.b.sdpa_fp8_decode_split(self.plan, self.total_q, self.total_kv, q, k, v, self.cq,
                                         self.ck, self.ds[0], self.ds[1], self.ds[2], self.inp.sm_scale, self.ws,
                                         stream=self.stream)

    def _capture(self, fn):
        return Case._capture(self, fn)

    def time(self, kind, steps, warmup):
        return Case.time(self, kind, steps, warmup)

    def _single_graph(self, kind, l):
        return Case._single_graph(self, kind, l)

    def bytes(self) -> int:
        splits = (dense_splits(self.skv, self.inp.h_kv, self.S, self.plan.num_sms) if self.plan.adaptive_splits
                  else None)
        return dense_bytes(self.sq, self.skv, self.inp.h_q, self.inp.h_kv, self.inp.d, self.S, splits)


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import split_kv_sparse_gb300 as b
    from split_kv_sparse_gb300 import workloads as wl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peak, peak_src = load_peaks()

    # inputs: one seeded 131072-row cache, replicated as the per-layer caches of the
    # timed rotation (views of one allocation), and per-layer queries / indices per s_q
    l2_bytes = int(getattr(torch.cuda.get_device_properties(local), "L2_cache_size", 0) or L2_FALLBACK)
    s_q_list = [args.s_q] + ([] if (args.no_sweep or args.no_mla_sweep)
                             else [s for s in SWEEP_SQ + TAIL_SQ if s != args.s_q])
    global LAYERS_OVERRIDE
    LAYERS_OVERRIDE = args.layers   # a fixed rotation (a small device footprint, e.g. for a profiler capture)
    n_layers_max = max(layers_for(s, l2_bytes) for s in s_q_list)
    base = wl.mla_inputs(1, N_KV, TOPK, seed=0)
    kv_all = torch.empty(n_layers_max, N_KV, D_QK, dtype=torch.bfloat16, device=dev)
    kv_all[0].copy_(base.kv.to(dev))
    kv_all[1:].copy_(kv_all[0].expand(n_layers_max - 1, N_KV, D_QK))
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def layer_inputs(s_q):
        R = layers_for(s_q, l2_bytes)
        qs, idxs = [], []
        for l in range(R):
            q, idx = wl.mla_queries(s_q, N_KV, TOPK, seed=1000 + s_q + 7919 * l)
            qs.append(q.to(dev))
            idxs.append(idx.to(dev))
        return qs, idxs

    main_qs, main_idxs = layer_inputs(args.s_q)
    case = Case(b, torch, kv_all, main_qs, main_idxs, base.sm_scale, 0)

    props = torch.cuda.get_device_properties(local)
    sampler = ClockSampler(getattr(props, "uuid", None) and f"GPU-{props.uuid}" or str(local))
    sampler.start()
    time.sleep(0.2)

    # ---- headline: K consecutive decode calls over the rotating layers -------------------
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.mark()
    t_wall0 = time.perf_counter()
    mean_call = case.time("call", args.steps, args.warmup)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall0
    sampler.mark()
    mean_kern = case.time("kernel", args.steps, max(3, args.warmup // 2))
    flushed = case.time_flushed(min(args.steps, 200), flush)
    if world > 1:
        dist.barrier()

    mean_call, mean_kern, flushed = max_over_ranks([mean_call, mean_kern, flushed], dev)

    kbytes = (balanced_bytes(args.s_q, case.plan.num_sms) if case.balanced
              else algorithmic_bytes(args.s_q, case.S, "split"))
    achieved = kbytes / (mean_kern * 1e-6) / 1e9

    # ---- end to end through the C ABI with host buffers ---------------------------------
    # mla_sparse_decode_host: per call the library copies that layer's queries and indices
    # in from pinned host memory, decodes, and copies the FP8 output and the LSE back, on
    # the case's stream; consecutive calls rotate over the layers
    q_h = [q.cpu().pin_memory() for q in main_qs]
    idx_h = [i.cpu().pin_memory() for i in main_idxs]
    out_h = torch.empty(case.out.shape, dtype=case.out.dtype).pin_memory()
    lse_h = torch.empty(case.lse.shape, dtype=case.lse.dtype).pin_memory()
    n_e2e = min(args.steps, 500)

    def host_call(l):
        b.mla_sparse_decode_host(case.plan, case.s_q, q_h[l], case.qs[l], case.kv_all[l], N_KV, idx_h[l],
                                 case.idxs[l], case.sm_scale, None, "e4m3", INV_SCALE, case.out, out_h, case.lse,
                                 lse_h, None, case.ws, stream=case.stream)
    with torch.cuda.stream(case.stream):
        for i in range(args.warmup):
            host_call(i % case.layers)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(case.stream)
        for i in range(n_e2e):
            host_call(i % case.layers)
        e1.record(case.stream)
    torch.cuda.synchronize()
    e2e_us = max_over_ranks([1000.0 * e0.elapsed_time(e1) / n_e2e], dev)[0]
    h2d = q_h[0].numel() * q_h[0].element_size() + idx_h[0].numel() * idx_h[0].element_size()
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()

    # ---- sweep: s_q x splits (and the planner's choice) -------------------------------
    sweep, dense_sweep = [], []
    if not args.no_sweep:
        for s_q in (() if args.no_mla_sweep else SWEEP_SQ):
            qs, idxs = (main_qs, main_idxs) if s_q == args.s_q else layer_inputs(s_q)
            # forced (token, split) grids, the planner's choice (S = 0) and the
            # balanced one-shot schedule where it applies (S = -1)
            for S in list(SWEEP_S) + [0, -1]:
                c = Case(b, torch, kv_all, qs, idxs, base.sm_scale, S)
                if S == -1 and not c.balanced:
                    del c
                    continue
                steps = max(args.sweep_steps, c.layers)
                us = c.time("call", steps, c.layers)
                ks = c.time("kernel", steps, c.layers)
                cb = point_bytes(s_q, c.S, c.balanced, c.plan.num_sms)
                sweep.append({"s_q": s_q, "num_splits": {0: "planner", -1: "balanced"}.get(S, S),
                              "planner": S == 0, "partials": "fp32", "layers": c.layers, "steps": steps,
                              "schedule": c.schedule(), "us_per_call": round(us, 2),
                              "split_kernel_us": round(ks, 2), "alg_bytes": cb,
                              "gb_s": round(cb / (us * 1e-6) / 1e9, 1),
                              "frac_of_peak": round(cb / (us * 1e-6) / 1e9 / peak, 4)})
                del c
            if s_q == BF16_PARTIALS_SQ:
                # the opt-in bf16 partials, where the partials outweigh the inputs
                for S in BF16_PARTIALS_S:
                    c = Case(b, torch, kv_all, qs, idxs, base.sm_scale, S, bf16_partials=True)
                    steps = max(args.sweep_steps, c.layers)
                    us = c.time("call", steps, c.layers)
                    ks = c.time("kernel", steps, c.layers)
                    cb = algorithmic_bytes(s_q, c.S, "call", partial_bytes=2)
                    sweep.append({"s_q": s_q, "num_splits": S if S else "planner", "planner": S == 0,
                                  "partials": "bf16", "layers": c.layers, "steps": steps,
                                  "schedule": c.schedule(), "us_per_call": round(us, 2),
                                  "split_kernel_us": round(ks, 2), "alg_bytes": cb,
                                  "gb_s": round(cb / (us * 1e-6) / 1e9, 1),
                                  "frac_of_peak": round(cb / (us * 1e-6) / 1e9 / peak, 4)})
                    del c
            del qs, idxs
        for s_q in (() if args.no_mla_sweep else TAIL_SQ):
            qs, idxs = layer_inputs(s_q)
            for S in (1, 0):
                c = Case(b, torch, kv_all, qs, idxs, base.sm_scale, S)
                steps = max(args.sweep_steps, c.layers)
                us = c.time("call", steps, c.layers)
                ks = c.time("kernel", steps, c.layers)
                cb = point_bytes(s_q, c.S, c.balanced, c.plan.num_sms)
                if c.tail is not None and c.tail[1] > 0:   # the split tail's partials, written and read back
                    r = s_q - c.tail[0]
                    cb += 2 * c.tail[1] * r * H_Q * (D_V + 1) * 4
                sweep.append({"s_q": s_q, "num_splits": "planner" if S == 0 else S, "planner": S == 0,
                              "partials": "fp32", "layers": c.layers, "steps": steps,
                              "schedule": c.schedule(), "us_per_call": round(us, 2),
                              "split_kernel_us": round(ks, 2), "alg_bytes": cb,
                              "gb_s": round(cb / (us * 1e-6) / 1e9, 1),
                              "frac_of_peak": round(cb / (us * 1e-6) / 1e9 / peak, 4)})
                del c
            del qs, idxs
        torch.cuda.synchronize()
        # the dense FP8 GQA variant (same partial / LSE protocol), forced split
        # counts and the planner's choice
        dinp = wl.sdpa_inputs(8, 32, 8, 128, seed=0)
        for S in (args.dense_splits if args.dense_splits is not None else list(SWEEP_S) + [0]):
            c = DenseCase(b, torch, dinp, S)
            steps = max(args.sweep_steps, c.layers)
            us = c.time("call", steps, c.layers)
            ks = c.time("kernel", steps, c.layers)
            cb = c.bytes()
            dense_sweep.append({"num_splits": S if S else "planner", "planner": S == 0, "splits_used": c.S,
                                "per_sequence_splits": (dense_splits(c.skv, 8, c.S, c.plan.num_sms)
                                                        if c.plan.adaptive_splits else None),
                                "us_per_call": round(us, 2), "split_kernel_us": round(ks, 2), "alg_bytes": cb,
                                "gb_s": round(cb / (us * 1e-6) / 1e9, 1),
                                "frac_of_peak": round(cb / (us * 1e-6) / 1e9 / peak, 4)})
            del c
        torch.cuda.synchronize()
    sampler.stop()
    clocks = sampler.summary()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.s_q, args.cpu_seconds)

    st, site = b.mla_get_status()
    if st != 0:
        raise RuntimeError(f"device status {st:#x} (wait site {site})")

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(mean_call, 3), "unit": "us/call", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(mean_call / 1000.0, 6),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": workload_name(args.s_q), "s_q": args.s_q, "schedule": case.schedule(),
                       "n_kv": N_KV, "topk": TOPK, "h_q": H_Q, "d_qk": D_QK, "d_v": D_V,
                       "output": "e4m3", "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                       "l2": (f"inputs larger than L2: consecutive calls rotate over {case.layers} per-layer "
                              f"KV caches ({N_KV} rows each) and query / index sets, "
                              f"{case.layers * unique_bytes(args.s_q) / 1e6:.0f} MB read per rotation against "
                              f"{l2_bytes / 1e6:.0f} MB of L2"),
                       "timing": ("the K steps as consecutive decode calls (CUDA graphs of one call per layer), "
                                  "one pair of CUDA events on the launching stream around all K; value = "
                                  "elapsed / K"),
                       "layers": case.layers,
                       "single_call_l2_flushed_us": round(flushed, 3),
                       "wall_s_timed_region": round(wall, 4)},
            "roofline": {"bound": "hbm", "kernel": ("mla_decode_kernel + combine (balanced schedule, whole call)"
                                                    if case.balanced
                                                    else "mla_decode_kernel (split pass)" if case.S > 1
                                                    else "mla_decode_kernel (direct epilogue)"),
                         "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4),
                         "traffic": known_traffic(args.s_q, "balanced" if case.balanced else case.S),
                         "alg_bytes_per_launch": kbytes, "kernel_us": round(mean_kern, 3),
                         "peak_source": f"{peak_src} hbm_gbs (MEASURED_PEAKS.json)" if peak_src == "measured"
                         else "fallback 6.8 TB/s"},
            "e2e": {"value": round(e2e_us, 3), "unit": "us/call", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "note": "mla_sparse_decode_host: H2D of Q and indices from pinned host memory, the decode, "
                            "D2H of FP8 O and LSE, in one C-ABI call per step, rotating over the layers; the "
                            "KV caches are resident decode state"},
            "gpu_launches": args.steps * case.launches(),
            "clocks": clocks,
            "cpu_baseline": cpu,
            "sweep": sweep,
            "dense_sweep": {"workload": DENSE_DESC, "points": dense_sweep} if dense_sweep else None,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def max_over_ranks(values, device=None):
    """Element-wise max of per-rank values across the process group (identity on one
    process): each rank runs an independent replica and the slowest one sets the number."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def known_traffic(s_q, S):
    """DRAM bytes per launch of the dominant kernel from an ncu capture of the current kernel
    source, or None when no capture matches it (the source hash keys the table)."""
    import hashlib
    src = os.path.join(ROOT, "split_kv_sparse_gb300", "csrc", "mla_decode.cu")
    try:
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    table = {   # (source hash, s_q, S) -> dram bytes per launch
        ("072ba5384f5884da", 96, 1): 55_474_176,
    }
    return table.get((h, s_q, S))


# ---------------------------------------------------------------------- CPU baseline --

def _cpu_worker(s_q: int, seconds: float, mode: str):
    """Runs in a child process with a fixed BLAS thread count: times the fp64 oracle."""
    import numpy as np

    import oracle.mla as om
    from split_kv_sparse_gb300 import workloads as wl

    base = wl.mla_inputs(1, N_KV, TOPK, seed=0)
    inp = wl.mla_inputs(s_q, N_KV, TOPK, seed=1000 + s_q) if s_q != 1 else base
    q = inp.q.double().numpy()
    kv = base.kv.double().numpy()
    idx = inp.idx.numpy()
    per_tok = []
    t_start = time.perf_counter()
    i = 0
    while True:
        t = i % s_q
        t0 = time.perf_counter()
        O, L = om.attention(q[t:t + 1], kv, idx[t:t + 1], inp.sm_scale, D_V)
        from oracle import codecs
        codecs.e4m3_encode(O * INV_SCALE)
        per_tok.append(time.perf_counter() - t0)
        i += 1
        if time.perf_counter() - t_start > seconds and i >= min(s_q, 4):
            break
    print(json.dumps({"per_token_s": per_tok, "tokens": i}))


def cpu_baseline(s_q: int, seconds: float, steps=None):
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(cores)
    env["CUDA_VISIBLE_DEVICES"] = ""
    p = subprocess.run([sys.executable, os.path.abspath(__file__), "--_cpu-worker", "--s-q", str(s_q),
                        "--cpu-seconds", str(seconds)], stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                       text=True, env=env, cwd=ROOT)
    if p.returncode != 0:
        return {"value": None, "unit": "us/call", "cores": cores, "kind": "oracle",
                "sample": f"failed: {p.stderr[-300:]}"}
    d = json.loads(p.stdout.strip().splitlines()[-1])
    per_tok = statistics.fmean(d["per_token_s"])
    return {"value": round(per_tok * s_q * 1e6, 1), "unit": "us/call", "cores": cores, "kind": "oracle",
            "sample": f"{d['tokens']} single-token oracle calls (fp64 numpy, BLAS threads = {cores}) of the "
                      f"s_q={s_q} workload, ~{seconds:g} s; per-call value = mean per-token time x {s_q}",
            "per_token_s": per_tok}


def run_reference(args):
    """The fp64 oracle as the reference arm, on this process's host cores (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    # each step is a bounded sample: one token of the workload, scaled to the call
    seconds = max(5.0, min(60.0, 0.05 * (args.steps + args.warmup)))
    cb = cpu_baseline(args.s_q, seconds)
    v = cb["value"]
    line = {"metric": METRIC, "value": v, "unit": "us/call", "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": (v / 1000.0) if v else None,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": workload_name(args.s_q), "s_q": args.s_q, "n_kv": N_KV, "topk": TOPK,
                       "h_q": H_Q, "d_qk": D_QK, "d_v": D_V, "output": "e4m3"},
            "cpu_baseline": cb,
            "e2e": {"value": v, "unit": "us/call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--s-q", type=int, default=96)
    ap.add_argument("--sweep-steps", type=int, default=50)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-mla-sweep", action="store_true", help="run only the dense part of the sweep")
    ap.add_argument("--dense-splits", type=int, nargs="*", default=None,
                    help="the dense sweep's split counts (0 = the planner's choice); default 1 2 4 8 16 0")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="per-layer caches the timed calls rotate over (0: enough to exceed L2 3x)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--_cpu-worker", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args._cpu_worker:
        _cpu_worker(args.s_q, args.cpu_seconds, "call")
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
