#!/usr/bin/env python
"""Benchmark of one Windowed-MTP speculative-decoding attention step on GB300.

A step is the whole hot path over one batch: d draft steps (each the fused
ring append + sink/window draft attention, then its split merge) and the
verification attention of T = d + 1 positions over the full bf16 KV cache
(+ merge), then a rollback of the d speculative ring entries so every timed
step sees the same state.  It runs as one CUDA graph; the L2 is flushed between
timed steps (a write and then a read of buffers twice its size, so the
flush's own write-back is not charged to the step).  Defaults: 10 warm-up
and 50 timed steps.

Default workload: 1M-token context, full-attention layer of a hybrid target
(GQA 8, head_dim 256, S=4, W=4096), draft depth 3.

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle
on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from speculative_decoding_attention_gb300 import inputs as wm_inputs  # noqa: E402
from speculative_decoding_attention_gb300 import workloads  # noqa: E402

METRIC = "decode-attn µs/step & HBM GB/s (% roofline): windowed draft vs full verify, 1M"
UNIT = "us/step"
FALLBACK_HBM_GBS = 6800.0
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "verify_traffic.json")
KERNEL_SOURCES = ("attn_tc.cuh", "tc.cuh", "ptx.cuh", "wm_internal.h")


def parse():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    ap.add_argument("--workload", default=workloads.BENCH_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--depth", type=int, default=None, help="draft depth d (verify T = d + 1)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline leg")
    ap.add_argument("--context", type=int, default=None,
                    help="shorter context, same recipe (small cases for profiler captures; not a bench line)")
    return ap.parse_args()


# ----------------------------------------------------------------- plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            return json.load(open(p))
        except ValueError:
            pass
    return {}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        path = os.path.join(ROOT, "speculative_decoding_attention_gb300", "csrc", name)
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, depth: int, context=None):
    """DRAM bytes per verify launch from the committed ncu summary, if it was
    taken on the current kernel source for this workload (at its own context);
    else None."""
    if context is not None:
        return None
    try:
        rec = json.load(open(PROFILE_TRAFFIC))
    except (OSError, ValueError):
        return None
    if rec.get("kernel_hash") != kernel_source_hash():
        return None
    entry = rec.get("workloads", {}).get(f"{workload}/d{depth}")
    return None if entry is None else entry.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms (200 ms if refused).

    The caller keeps the GPU busy with untimed steps while the sampler starts
    (``load_until_sampled``) and after the timed region, so every sample is
    taken under the step's load; ``mark`` brackets the timed region so that
    the summary also counts the samples taken inside it.
    """

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 20

    def __init__(self, device):
        try:
            self.gpu = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
        except Exception:  # older torch: fall back to the ordinal
            self.gpu = str(device.index or 0)
        self.proc = None
        self.path = None
        self.window = None

    def _start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.interval_ms)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        self.interval_ms = self.INTERVAL_MS
        self._start()
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def _count(self) -> int:
        try:
            with open(self.path) as f:
                return sum(1 for _ in f)
        except OSError:
            return 0

    def load_until_sampled(self, step, n: int, limit_s: float = 3.0):
        """Run ``step`` (untimed) until ``n`` more samples have been written."""
        if self.proc is None:
            return
        goal = self._count() + n
        t0 = time.time()
        while self._count() < goal and time.time() - t0 < limit_s:
            if self.proc.poll() is not None and self._count() == 0 and self.interval_ms < 200:
                self.interval_ms = 200  # this nvidia-smi refused the short interval
                self._start()
                if self.proc is None:
                    return
            step()
            torch.cuda.synchronize()

    def mark(self, t_begin: float, t_end: float):
        self.window = (t_begin, t_end)

    def summary(self) -> dict:
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        except OSError:
            pass
        finally:
            if self.path and os.path.exists(self.path):
                os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        def stamp(x):
            try:
                return datetime.datetime.strptime(x, "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i - 5] for r in rows for i in range(5, 9) if r[i].lower() == "active"})
        out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
               "reasons": reasons, "samples": len(rows), "interval_ms": self.interval_ms,
               "window": "every sample taken while step graphs run (untimed steps before and after "
                         "the timed region, and the timed steps)"}
        if self.window:
            lo, hi = self.window
            inside = [r for r in rows if (s := stamp(r[0])) is not None and lo <= s <= hi]
            out["samples_in_timed_region"] = len(inside)
            out["timed_region_s"] = round(hi - lo, 4)
        return out


# ----------------------------------------------------------------- GPU arm

class Step:
    """Device state of one workload and its captured step."""

    def __init__(self, w: workloads.Workload, depth: int, device, context: int | None = None):
        from speculative_decoding_attention_gb300 import wm

        self.wm, self.w, self.d, self.T, self.dev = wm, w, depth, depth + 1, device
        self.inp = wm_inputs.make_inputs(w, depth=depth, device=device, context=context)
        inp = self.inp
        self.kv = wm.KVCache(inp.k, inp.v, inp.seq_lens, inp.block_table)
        self.ring = wm.Ring.create(w.batch, w.n_kv_heads, w.head_dim, w.sink, w.window, device)
        self._build_ring()
        B, Hq, D = w.batch, w.n_q_heads, w.head_dim
        self.base_len = inp.seq_lens.clone()
        self.d_out = torch.empty((depth, B, Hq, D), dtype=torch.bfloat16, device=device)
        self.d_lse = torch.empty((depth, B, Hq), dtype=torch.float32, device=device)
        self.v_out = torch.empty_like(inp.q_verify)
        self.v_lse = torch.empty(inp.q_verify.shape[:3], dtype=torch.float32, device=device)
        self.d_splits = wm.plan_splits(wm.WM_OP_DRAFT_STEP, B, w.n_kv_heads, Hq, 1, D, w.slots)
        self.v_splits = wm.plan_splits(wm.WM_OP_VERIFY, B, w.n_kv_heads, Hq, self.T, D, self.kv.capacity)
        dws = wm.workspace_size(wm.WM_OP_DRAFT, B, w.n_kv_heads, Hq, 1, D, w.slots)
        vws = wm.workspace_size(wm.WM_OP_VERIFY, B, w.n_kv_heads, Hq, self.T, D, self.kv.capacity)
        self.d_ws = torch.empty(max(dws, 256), dtype=torch.uint8, device=device)
        self.s_ws = wm.step_workspace(self.ring, Hq)  # the fused step's own (zeroed) workspace
        self.v_ws = torch.empty(max(vws, 256), dtype=torch.uint8, device=device)
        self.graph = None
        self.ev = None

    def _build_ring(self):
        wm, w, inp = self.wm, self.w, self.inp
        tail = w.ring_appends
        if tail:
            lens = inp.seq_lens - tail
            wm.ring_fill(self.ring, wm.KVCache(inp.k, inp.v, lens, inp.block_table))
            for t in range(tail):
                kj, vj = inp.position_rows([n - tail + t for n in inp.seq_lens_host])
                wm.ring_append(self.ring, kj.contiguous(), vj.contiguous())
        else:
            wm.ring_fill(self.ring, self.kv)

    def launches_per_step(self, fused: bool = True) -> int:
        per_draft = 2 if fused else 2 + (1 if self.d_splits > 1 else 0)
        return self.d * per_draft + 1 + (1 if self.v_splits > 1 else 0) + 1

    def draft(self, j: int, fused: bool = True, q=None, k_new=None, v_new=None):
        """Draft step j: the fused step (append in the attention launch, then the merge), or ring
        append + draft attention (+ merge)."""
        wm, w, inp = self.wm, self.w, self.inp
        q = inp.q_draft[j] if q is None else q
        k_new = inp.k_new[j] if k_new is None else k_new
        v_new = inp.v_new[j] if v_new is None else v_new
        if fused:
            wm.draft_step(self.ring, k_new, v_new, q, w.scale, self.s_ws, out=self.d_out[j], lse=self.d_lse[j])
        else:
            wm.ring_append(self.ring, k_new, v_new)
            wm.draft_attn(self.ring, q, w.scale, out=self.d_out[j], lse=self.d_lse[j], workspace=self.d_ws)

    def run(self, ev=None, fused: bool = True):
        wm, w, inp = self.wm, self.w, self.inp
        if ev:
            ev[0].record()
        for j in range(self.d):
            self.draft(j, fused)
        if ev:
            ev[1].record()
        wm.verify_attn(self.kv, inp.q_verify, w.scale, out=self.v_out, lse=self.v_lse, workspace=self.v_ws)
        if ev:
            ev[2].record()
        wm.ring_rollback(self.ring, self.base_len)

    def capture(self, fused: bool = True, events: bool = True):
        """Capture one step in a CUDA graph; returns (graph, in-graph events or None).
        With ``events`` the graph also records events before the draft chain,
        between it and the verify, and after the verify."""
        self.run(fused=fused)  # eager once: kernel attributes, descriptors, first-touch
        torch.cuda.synchronize()
        ev = None
        if events:
            try:
                ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(3)]
            except TypeError:
                ev = None
        s = torch.cuda.Stream(device=self.dev)
        s.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            self.run(ev, fused=fused)
        torch.cuda.synchronize()
        self.graph, self.ev = graph, ev
        return graph, ev


class L2Flush:
    """Flush the L2 between timed steps: write a buffer of twice the L2, then
    read another one as large.  The read evicts the dirty lines the write left
    behind, so their write-back to HBM happens here rather than inside the
    next timed step (where it would be charged to the step's kernels)."""

    def __init__(self, device):
        import torch

        n = max(2 * torch.cuda.get_device_properties(device).L2_cache_size, 256 << 20)
        self.wbuf = torch.empty(n, dtype=torch.uint8, device=device)
        self.rbuf = torch.zeros(n // 8, dtype=torch.int64, device=device)
        self.sink = torch.empty((), dtype=torch.int64, device=device)

    def __call__(self):
        import torch

        self.wbuf.zero_()
        torch.sum(self.rbuf, dim=0, out=self.sink)


def gpu_arm(args, rank, world, local):
    from speculative_decoding_attention_gb300 import build as wm_build
    from speculative_decoding_attention_gb300 import wm

    if not os.path.exists(wm_build.LIB) or not wm_build.up_to_date():
        wm_build.build()
    wm.load()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    init_dist(world, "nccl")
    w = workloads.get(args.workload)
    depth = args.depth if args.depth is not None else (
        workloads.BENCH_DEPTH if args.workload == workloads.BENCH_WORKLOAD else w.max_depth)

    st = Step(w, depth, device, context=args.context)
    # The timed graph holds the step's kernels only; a second capture with
    # events between the draft chain and the verify gives the breakdown.
    st.capture(events=False)
    timed_graph = st.graph
    flush = L2Flush(device)

    for _ in range(max(3, args.warmup)):
        flush()
        st.graph.replay()
    torch.cuda.synchronize()
    if wm.get_device_error():
        raise RuntimeError("device error during warm-up")

    step_ms, draft_ms, verify_ms = [], [], []
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)

    def untimed_step():
        flush()
        st.graph.replay()

    with ClockSampler(device) as clk:
        clk.load_until_sampled(untimed_step, 3)
        barrier(world)
        torch.cuda.synchronize()
        t_begin = time.time()
        for _ in range(args.steps):
            flush()
            e0.record()
            timed_graph.replay()
            e1.record()
            e1.synchronize()
            step_ms.append(e0.elapsed_time(e1))
        torch.cuda.synchronize()
        t_end = time.time()
        barrier(world)
        clk.mark(t_begin, t_end)
        clk.load_until_sampled(untimed_step, 2)
    clocks = clk.summary()
    # Breakdown: the step captured with in-graph events, replayed the same way.
    st.capture(events=True)
    if st.ev:
        for i in range(max(3, args.warmup) + args.steps):
            flush()
            st.graph.replay()
            torch.cuda.synchronize()
            if i >= max(3, args.warmup):
                draft_ms.append(st.ev[0].elapsed_time(st.ev[1]))
                verify_ms.append(st.ev[1].elapsed_time(st.ev[2]))
    # The same step graph replayed without the flush: the ring stays in L2
    # from one step to the next (the verify streams its cache evict-first).
    warm_draft_ms = []
    if st.ev:
        for i in range(3 + max(3, args.steps // 2)):
            st.graph.replay()
            torch.cuda.synchronize()
            if i >= 3:
                warm_draft_ms.append(st.ev[0].elapsed_time(st.ev[1]))
    if not st.ev:  # no in-graph events: time the verify alone, same way
        for _ in range(args.steps):
            flush()
            e0.record()
            wm.verify_attn(st.kv, st.inp.q_verify, w.scale, out=st.v_out, lse=st.v_lse, workspace=st.v_ws)
            e1.record()
            e1.synchronize()
            verify_ms.append(e0.elapsed_time(e1))
    if wm.get_device_error():
        raise RuntimeError("device error during the timed steps")
    out_ok = bool(torch.isfinite(st.v_out.float()).all() and torch.isfinite(st.d_out.float()).all())
    native_ms, native_step_ms = native_draft_chain(st, flush, args)
    unfused_ms = unfused_draft_chain(st, flush, args)
    masw = masw_draft_chain(st, flush, args)

    us_step = max_over_ranks(1e3 * sum(step_ms) / len(step_ms), world, device)
    us_verify = 1e3 * sum(verify_ms) / len(verify_ms)
    us_draft = 1e3 * sum(draft_ms) / len(draft_ms) if draft_ms else None

    B, Hq, Hkv, D = w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim
    sum_n = sum(st.inp.seq_lens_host)
    verify_bytes = 2 * Hkv * D * 2 * sum_n + 2 * (B * st.T * Hq * D * 2) + B * st.T * Hq * 4
    draft_bytes = 2 * B * Hkv * w.slots * D * 2 + 2 * (B * Hq * D * 2) + B * Hq * 4
    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = peak or FALLBACK_HBM_GBS
    achieved = verify_bytes / (us_verify * 1e-6) / 1e9
    draft_gbs = draft_bytes * depth / (us_draft * 1e-6) / 1e9 if us_draft else None

    e2e = None if args.no_e2e else e2e_leg(st, args, world, device)
    cpu = None
    if not args.no_cpu and rank == 0:
        cpu = cpu_baseline(st, args)

    if rank != 0:
        return
    line = {
        "metric": METRIC,
        "value": round(us_step, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(us_step / 1e3, 5),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) K/V and queries in the workload's shapes; no dataset)",
        "config": {
            "workload": w.name,
            "batch": B, "context": (args.context if args.context else w.context) if not w.ragged else
            list(st.inp.seq_lens_host),
            "n_q_heads": Hq, "n_kv_heads": Hkv, "head_dim": D, "sink": w.sink, "window": w.window,
            "draft_depth": depth, "verify_positions": st.T, "kv_layout": "paged" if w.page_size else "contiguous",
            "draft_splits": st.d_splits, "verify_splits": st.v_splits,
            "draft_execution": "per draft step: one launch of ring append fused into the draft attention, "
                               "then the split merge (which commits the append)",
            "l2": "flushed between timed steps (write of a 2x L2 buffer, then a read of another 2x L2 buffer so "
                  "the flush's dirty lines are written back before the step); each step also reads the full "
                  "KV cache (> L2)",
            "execution": "one CUDA graph per step (kernels only; the draft / verify breakdown in detail comes from a second capture with events between them)", "parallelism": f"replicas x{world}",
        },
        "detail": {
            "step_us_median": round(1e3 * sorted(step_ms)[len(step_ms) // 2], 2),
            "verify_us": round(us_verify, 2),
            "verify_gbs": round(achieved, 1),
            "draft_chain_us": None if us_draft is None else round(us_draft, 2),
            "draft_us_per_step": None if us_draft is None else round(us_draft / depth, 2),
            "draft_gbs": None if draft_gbs is None else round(draft_gbs, 1),
            "draft_frac_of_hbm": None if draft_gbs is None else round(draft_gbs / peak, 4),
            "draft_kv_bytes_per_step": 2 * B * Hkv * w.slots * D * 2,
            "draft_l2": "L2 flushed before each step; draft steps 2..d re-read the ring (S+W slots) "
                        "mostly from L2, as a decode loop does",
            "draft_us_per_step_warm_l2": (round(1e3 * sum(warm_draft_ms) / len(warm_draft_ms) / depth, 2)
                                          if warm_draft_ms else None),
            "draft_warm_l2": "the same step graph replayed without the flush: the ring stays in L2 from step "
                             "to step (the verify reads its cache evict-first)",
            "unfused_draft_us_per_step": None if unfused_ms is None else round(1e3 * unfused_ms / depth, 2),
            "masw_draft": masw,
            "verify_kv_bytes": 2 * Hkv * D * 2 * sum_n,
            "outputs_finite": out_ok,
            "steps_per_s_all_ranks": round(world * 1e6 / us_step, 1),
            "native_draft_chain_us": round(1e3 * native_ms, 2),
            "native_draft_us_per_step": round(1e3 * native_ms / depth, 2),
            "native_step_us": round(1e3 * native_step_ms, 2),
            "native_over_windowed_step": round(1e3 * native_step_ms / us_step, 3),
        },
        "roofline": {
            "kernel": "attn_tc_kernel (tcgen05 verify, split-KV) + lse_merge",
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "peak_source": f"{peak_src} hbm_gbs",
            "traffic": profiled_traffic(w.name, depth, args.context),
        },
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": st.launches_per_step() * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def unfused_draft_chain(st: Step, flush, args):
    """The draft chain as three launches per draft step (ring append, draft
    attention, split merge): the whole step captured with in-graph events,
    the draft interval averaged.  None without in-graph events."""
    graph, ev = st.capture(fused=False)
    if not ev:
        return None
    ms = []
    for i in range(max(3, args.warmup) + max(3, args.steps // 2)):
        flush()
        graph.replay()
        torch.cuda.synchronize()
        if i >= max(3, args.warmup):
            ms.append(ev[0].elapsed_time(ev[1]))
    return sum(ms) / len(ms)


MASW_SLOT_INTERVAL = 256  # one memory slot per 256 tokens of history


def masw_draft_chain(st: Step, flush, args):
    """The draft chain with memory slots (memory-augmented sliding window): the
    fused step over sinks + window + one materialized slot per
    MASW_SLOT_INTERVAL tokens of each sequence's history (synthetic slot K/V),
    captured with in-graph events.  None without in-graph events."""
    wm, w, inp = st.wm, st.w, st.inp
    B, Hq, Hkv, D = w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim
    counts = [n // MASW_SLOT_INTERVAL for n in inp.seq_lens_host]
    cap = max(1, max(counts))
    gen = torch.Generator(device=st.dev).manual_seed(4242)
    mem = wm.Mem.create(B, Hkv, D, cap, st.dev)
    mem.k.copy_(torch.randn(mem.k.shape, generator=gen, device=st.dev).to(torch.bfloat16))
    mem.v.copy_(torch.randn(mem.v.shape, generator=gen, device=st.dev).to(torch.bfloat16))
    mem.count.copy_(torch.tensor(counts, dtype=torch.int64, device=st.dev))
    ws = wm.step_workspace(st.ring, Hq, mem=mem)

    def chain(ev=None):
        if ev:
            ev[0].record()
        for j in range(st.d):
            wm.draft_step(st.ring, inp.k_new[j], inp.v_new[j], inp.q_draft[j], w.scale, ws, out=st.d_out[j],
                          lse=st.d_lse[j], mem=mem)
        if ev:
            ev[1].record()
        wm.ring_rollback(st.ring, st.base_len)

    chain()
    torch.cuda.synchronize()
    try:
        ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
    except TypeError:
        return None
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device=st.dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        chain(ev)
    ms = []
    for i in range(max(3, args.warmup) + max(3, args.steps // 2)):
        flush()
        g.replay()
        torch.cuda.synchronize()
        if i >= max(3, args.warmup):
            ms.append(ev[0].elapsed_time(ev[1]))
    us = 1e3 * sum(ms) / len(ms) / st.d
    kv_bytes = 2 * Hkv * D * 2 * sum(w.slots + c for c in counts)
    return {"slot_interval": MASW_SLOT_INTERVAL, "slots": counts, "us_per_step": round(us, 2),
            "kv_bytes_per_step": kv_bytes, "gbs": round(kv_bytes / (us * 1e-6) / 1e9, 1)}


def native_draft_chain(st: Step, flush, args) -> tuple[float, float]:
    """The draft chain without windowing (the native MTP draft the pages compare
    against): each of the d draft steps attends over the whole cache, i.e. the
    verify kernel with one query position over positions 0..N_b+j.  Returns the
    mean milliseconds per chain and per native step (the chain followed by the
    verify), each graph-captured with the L2 flushed between replays."""
    wm, w, inp = st.wm, st.w, st.inp
    B, Hq, D = w.batch, w.n_q_heads, w.head_dim
    lens = [torch.tensor([n + j + 1 for n in inp.seq_lens_host], dtype=torch.int64, device=st.dev)
            for j in range(st.d)]
    kvs = [wm.KVCache(inp.k, inp.v, lens[j], inp.block_table) for j in range(st.d)]
    qs = [inp.q_draft[j].view(B, 1, Hq, D) for j in range(st.d)]
    out = torch.empty((B, 1, Hq, D), dtype=torch.bfloat16, device=st.dev)
    lse = torch.empty((B, 1, Hq), dtype=torch.float32, device=st.dev)
    need = wm.workspace_size(wm.WM_OP_VERIFY, B, w.n_kv_heads, Hq, 1, D, st.kv.capacity)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=st.dev)

    def chain():
        for j in range(st.d):
            wm.verify_attn(kvs[j], qs[j], w.scale, out=out, lse=lse, workspace=ws)

    def step():  # the native step: the draft chain, then the same verify as the windowed step
        chain()
        wm.verify_attn(st.kv, inp.q_verify, w.scale, out=st.v_out, lse=st.v_lse, workspace=st.v_ws)

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=st.dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=s):
            fn()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        ms = []
        for i in range(max(3, args.warmup) + max(3, args.steps // 2)):
            flush()
            e0.record()
            g.replay()
            e1.record()
            e1.synchronize()
            if i >= max(3, args.warmup):
                ms.append(e0.elapsed_time(e1))
        return sum(ms) / len(ms)

    return timed(chain), timed(step)


def _packed(specs, device, pinned: bool):
    """One byte buffer holding tensors of the given (name, shape, dtype), each
    at a 256-byte aligned offset; returns (buffer, {name: typed view})."""
    layout, off = {}, 0
    for name, shape, dtype in specs:
        off = (off + 255) & ~255
        n = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        layout[name] = (off, shape, dtype, n)
        off += n
    if pinned:
        buf = torch.empty(off, dtype=torch.uint8).pin_memory()
    else:
        buf = torch.empty(off, dtype=torch.uint8, device=device)
    return buf, {name: buf[o:o + n].view(dt).view(shape) for name, (o, shape, dt, n) in layout.items()}


def e2e_leg(st: Step, args, world, device) -> dict:
    """The same step through the public API with host buffers: every step copies
    its inputs from pinned host memory (draft queries, the appended draft K/V,
    verify queries, the verify tokens' own K/V into the cache) and reads every
    output back; eager calls, no graph.  Inputs travel in one packed host-to-
    device copy and outputs in one device-to-host copy per step."""
    wm, w, inp = st.wm, st.w, st.inp
    T = st.T
    srcs = {"q_draft": inp.q_draft, "k_new": inp.k_new, "v_new": inp.v_new, "q_verify": inp.q_verify}
    contiguous = inp.block_table is None
    if contiguous:
        tail = [slice(n - T, n) for n in inp.seq_lens_host]
        srcs["k_tail"] = torch.stack([inp.k[b, :, tail[b]] for b in range(w.batch)])
        srcs["v_tail"] = torch.stack([inp.v[b, :, tail[b]] for b in range(w.batch)])
    in_specs = [(k, tuple(t.shape), t.dtype) for k, t in srcs.items()]
    host_in_buf, host_in = _packed(in_specs, device, pinned=True)
    dev_in_buf, dev_in = _packed(in_specs, device, pinned=False)
    for k, t in srcs.items():
        host_in[k].copy_(t.cpu())
    out_specs = [("d_out", tuple(st.d_out.shape), st.d_out.dtype), ("d_lse", tuple(st.d_lse.shape), st.d_lse.dtype),
                 ("v_out", tuple(st.v_out.shape), st.v_out.dtype), ("v_lse", tuple(st.v_lse.shape), st.v_lse.dtype)]
    host_out_buf, host_out = _packed(out_specs, device, pinned=True)
    dev_out_buf, dev_out = _packed(out_specs, device, pinned=False)
    h2d = host_in_buf.numel()
    d2h = host_out_buf.numel()

    def one():
        dev_in_buf.copy_(host_in_buf, non_blocking=True)
        if contiguous:
            for b, n in enumerate(inp.seq_lens_host):
                inp.k[b, :, n - T:n].copy_(dev_in["k_tail"][b])
                inp.v[b, :, n - T:n].copy_(dev_in["v_tail"][b])
        for j in range(st.d):
            wm.draft_step(st.ring, dev_in["k_new"][j], dev_in["v_new"][j], dev_in["q_draft"][j], w.scale, st.s_ws,
                          out=dev_out["d_out"][j], lse=dev_out["d_lse"][j])
        wm.verify_attn(st.kv, dev_in["q_verify"], w.scale, out=dev_out["v_out"], lse=dev_out["v_lse"],
                       workspace=st.v_ws)
        wm.ring_rollback(st.ring, st.base_len)
        host_out_buf.copy_(dev_out_buf, non_blocking=True)

    for _ in range(max(3, args.warmup)):
        one()
    torch.cuda.synchronize()
    if not (torch.equal(host_out["v_out"], dev_out["v_out"].cpu()) and torch.equal(host_out["d_lse"], dev_out["d_lse"].cpu())):
        raise RuntimeError("e2e: the packed read-back does not match the device outputs")
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        one()
    e1.record()
    e1.synchronize()
    barrier(world)
    us = max_over_ranks(1e3 * e0.elapsed_time(e1) / args.steps, world, device)
    return {"value": round(us, 2), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "note": "eager C-ABI calls; KV cache resident; per-step inputs cross PCIe/C2C in one packed copy "
                    "from pinned host memory, outputs in one packed copy back"}


# ----------------------------------------------------------------- CPU oracle

def oracle_sample(w, depth, inp_host, rows_fraction):
    """One bounded sample of the step on the host: every draft row of the d
    draft steps, and an evenly spaced fraction of the verify rows.  Returns
    (seconds spent, seconds per whole step, description, seconds per draft
    step, seconds per whole verify)."""
    import oracle

    B, Hq, T = w.batch, w.n_q_heads, depth + 1
    hist = oracle.KV(inp_host["k"], inp_host["v"], inp_host["block_table"])
    t0 = time.perf_counter()
    for j in range(depth):
        pos = [n + j for n in inp_host["lens"]]
        oracle.draft(hist, inp_host["q_draft"][j], pos, w.sink, w.window, w.scale)
    t_draft = time.perf_counter() - t0
    total_rows = B * T * Hq
    n_rows = max(1, int(round(total_rows * rows_fraction)))
    rows = [int(round(i * total_rows / n_rows)) for i in range(n_rows)]
    t1 = time.perf_counter()
    oracle.verify(hist, inp_host["q_verify"], inp_host["lens"], w.scale, rows=rows)
    t_verify = time.perf_counter() - t1
    verify_s = t_verify * total_rows / n_rows
    per_step = t_draft + verify_s
    desc = (f"all {B * Hq} draft rows x {depth} draft steps + {n_rows}/{total_rows} verify rows "
            f"(scaled x{total_rows / n_rows:.2f}) of {w.name}")
    return t_draft + t_verify, per_step, desc, t_draft / max(1, depth), verify_s


def host_inputs(inp):
    return {"k": inp.k.cpu(), "v": inp.v.cpu(),
            "block_table": None if inp.block_table is None else inp.block_table.cpu(),
            "lens": list(inp.seq_lens_host), "q_draft": inp.q_draft.cpu(), "q_verify": inp.q_verify.cpu()}


def pick_fraction(w, depth, inp_host, budget_s):
    """Verify-row fraction whose oracle time is about ``budget_s`` seconds."""
    probe = 1.0 / (w.batch * (depth + 1) * w.n_q_heads)
    secs = oracle_sample(w, depth, inp_host, probe)[0]
    rows_per_s = 1.0 / max(secs, 1e-6)
    frac = min(1.0, budget_s * rows_per_s / (w.batch * (depth + 1) * w.n_q_heads))
    return max(probe, frac)


def cpu_baseline(st: Step, args, min_seconds: float = 10.0) -> dict:
    """The oracle timed on repeated bounded samples until about ``min_seconds``
    of CPU work have run; reported per whole step."""
    import oracle

    oracle.set_num_threads(len(os.sched_getaffinity(0)))  # every host core this process may use
    inp_host = host_inputs(st.inp)
    frac = pick_fraction(st.w, st.d, inp_host, budget_s=min_seconds / 2)
    total, per_steps, drafts, verifies, desc = 0.0, [], [], [], ""
    while total < min_seconds:
        secs, per_step, desc, draft_s, verify_s = oracle_sample(st.w, st.d, inp_host, frac)
        total += secs
        per_steps.append(per_step)
        drafts.append(draft_s)
        verifies.append(verify_s)
    n = len(per_steps)
    return {"value": round(1e6 * sum(per_steps) / n, 1), "unit": UNIT,
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} x ({desc})", "sample_seconds": round(total, 2),
            "draft_us_per_step": round(1e6 * sum(drafts) / n, 1), "verify_us": round(1e6 * sum(verifies) / n, 1)}


def reference_arm(args, rank, world, local):
    """The fp64 CPU oracle on the host cores, on the GPU arm's workload."""
    import oracle

    if world > 1:
        init_dist(world, "gloo")
        if rank != 0:
            barrier(world)
            return
    oracle.build()
    # The launcher may cap each rank at one OpenMP thread; only this rank
    # works, so it takes every host core it may run on.
    oracle.set_num_threads(len(os.sched_getaffinity(0)))
    w = workloads.get(args.workload)
    depth = args.depth if args.depth is not None else (
        workloads.BENCH_DEPTH if args.workload == workloads.BENCH_WORKLOAD else w.max_depth)
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = wm_inputs.make_inputs(w, depth=depth, device=gen_dev)
    inp_host = host_inputs(inp)
    del inp
    budget = max(2.0, 150.0 / max(1, args.steps + args.warmup))
    frac = pick_fraction(w, depth, inp_host, budget_s=budget)
    for _ in range(args.warmup):
        oracle_sample(w, depth, inp_host, frac)
    per_steps, drafts, verifies, secs_total, desc = [], [], [], 0.0, ""
    for _ in range(args.steps):
        secs, per_step, desc, draft_s, verify_s = oracle_sample(w, depth, inp_host, frac)
        per_steps.append(per_step)
        drafts.append(draft_s)
        verifies.append(verify_s)
        secs_total += secs
    us = 1e6 * sum(per_steps) / len(per_steps)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) K/V and queries in the workload's shapes; no dataset)",
        "config": {"workload": w.name, "draft_depth": depth, "verify_positions": depth + 1,
                   "parallelism": "host cores (OpenMP over rows)"},
        "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": desc, "draft_us_per_step": round(1e6 * sum(drafts) / len(drafts), 1),
                         "verify_us": round(1e6 * sum(verifies) / len(verifies), 1)},
        "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        barrier(world)


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.gpus != world and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    if args.impl == "reference":
        reference_arm(args, rank, world, local)
    else:
        gpu_arm(args, rank, world, local)
    if torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
