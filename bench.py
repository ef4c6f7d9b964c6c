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
on whole steps of the same workload instead.
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
KERNEL_SOURCES = ("attn_tc.cuh", "attn_tcp.cuh", "tc.cuh", "ptx.cuh", "wm_internal.h")


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
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other 1M-context configurations measured beside the headline")
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


# NVML clock sampler, run as its own process (no GIL shared with the timing
# loop): samples the SM clock, its maximum and the clock-event reasons every
# interval until terminated; one line per sample, CLOCK_MONOTONIC seconds
# first, so the parent can tell which samples fall inside its timed region.
_NVML_SAMPLER = r"""
import ctypes, sys, time
uuid, interval = sys.argv[1].encode(), float(sys.argv[2])
nv = ctypes.CDLL("libnvidia-ml.so.1")
if nv.nvmlInit_v2() != 0:
    sys.exit(3)
h = ctypes.c_void_p()
if nv.nvmlDeviceGetHandleByUUID(ctypes.c_char_p(uuid), ctypes.byref(h)) != 0:
    sys.exit(4)
reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or nv.nvmlDeviceGetCurrentClocksThrottleReasons
sm, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
out = sys.stdout
print("ready", flush=True)
while True:
    t = time.monotonic()
    ok = nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) == 0
    ok = ok and nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0
    ok = ok and reasons(h, ctypes.byref(rs)) == 0
    if ok:
        out.write(f"{t:.6f},{sm.value},{mx.value},{rs.value}\n")
        out.flush()
    time.sleep(interval)
"""

# clock-event reason bits (NVML) and the names the JSON line uses
_REASON_BITS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap"}


class ClockSampler:
    """SM clocks and throttle reasons while the step's graphs run.

    Preferred: NVML queried from a separate process every 0.5 ms, so that even
    a timed region of a few milliseconds holds several samples.  Fallback:
    ``nvidia-smi -lms 20``.  The caller keeps the GPU busy with untimed steps
    while the sampler starts (``load_until_sampled``) and after the timed
    region, so every sample is taken under the step's load; ``mark``
    brackets the timed region (``time.monotonic()`` seconds) so that the
    summary also counts the samples taken inside it.
    """

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 20
    NVML_INTERVAL_MS = 0.5

    def __init__(self, device):
        try:
            self.gpu = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
        except Exception:  # older torch: fall back to the ordinal
            self.gpu = str(device.index or 0)
        self.proc = None
        self.path = None
        self.window = None
        self.source = None
        self.interval_ms = self.INTERVAL_MS

    def _start_smi(self):
        self.source = "nvidia-smi"
        self.interval_ms = self.INTERVAL_MS
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.interval_ms)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def _start_nvml(self) -> bool:
        if not self.gpu.startswith("GPU-"):
            return False
        try:
            proc = subprocess.Popen([sys.executable, "-c", _NVML_SAMPLER, self.gpu, str(self.NVML_INTERVAL_MS / 1e3)],
                                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return False
        first = proc.stdout.readline()
        if first.strip() != "ready":
            proc.kill()
            proc.wait()
            return False
        self.proc, self.source, self.interval_ms = proc, "nvml", self.NVML_INTERVAL_MS
        self.rows = []
        import threading

        def drain():  # the reader thread only appends lines (no GPU work, no timing)
            for line in proc.stdout:
                self.rows.append(line)

        self.reader = threading.Thread(target=drain, daemon=True)
        self.reader.start()
        return True

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        if not self._start_nvml():
            self._start_smi()
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.source == "nvml":
            self.reader.join(timeout=5)
            with open(self.path, "w") as f:
                f.writelines(self.rows)

    def _count(self) -> int:
        if self.source == "nvml":
            return len(self.rows)
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
            if self.source == "nvidia-smi" and self.proc.poll() is not None and self._count() == 0 \
                    and self.interval_ms < 200:
                self.interval_ms = 200  # this nvidia-smi refused the short interval
                self.proc = None
                try:
                    self.proc = subprocess.Popen(
                        ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                         "--format=csv,noheader,nounits", "-lms", "200"], stdout=open(self.path, "w"),
                        stderr=subprocess.DEVNULL)
                except OSError:
                    return
            step()
            torch.cuda.synchronize()

    def mark(self, t_begin: float, t_end: float):
        """The timed region, in time.monotonic() seconds."""
        self.window = (t_begin, t_end)

    def _parse(self):
        """(monotonic time or None, sm MHz, max MHz, set of reason names) per sample."""
        out = []
        try:
            lines = open(self.path).read().splitlines()
        except OSError:
            return out
        finally:
            if self.path and os.path.exists(self.path):
                os.unlink(self.path)

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 4:  # nvml: t, sm, max, reason bits
                t, sm, mx, bits = num(parts[0]), num(parts[1]), num(parts[2]), int(num(parts[3]) or 0)
                out.append((t, sm, mx, {name for bit, name in _REASON_BITS.items() if bits & bit}))
            elif len(parts) >= 9:  # nvidia-smi csv: wall-clock stamp, mapped onto monotonic time
                try:
                    wall = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    t = wall - (time.time() - time.monotonic())
                except ValueError:
                    t = None
                names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
                out.append((t, num(parts[1]), num(parts[2]),
                            {names[i - 5] for i in range(5, 9) if parts[i].lower() == "active"}))
        return out

    def summary(self) -> dict:
        rows = self._parse()
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [r[1] for r in rows if r[1] is not None]
        mx = [r[2] for r in rows if r[2] is not None]
        reasons = sorted(set().union(*(r[3] for r in rows)))
        out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
               "reasons": reasons, "samples": len(rows), "interval_ms": self.interval_ms, "source": self.source,
               "window": "every sample taken while step graphs run (untimed steps before and after "
                         "the timed region, and the timed steps)"}
        if self.window:
            lo, hi = self.window
            inside = [r for r in rows if r[0] is not None and lo <= r[0] <= hi]
            out["samples_in_timed_region"] = len(inside)
            out["timed_region_s"] = round(hi - lo, 4)
            if inside:
                out["sm_mhz_timed_region"] = statistics.median(r[1] for r in inside if r[1] is not None)
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
        self.v_persistent = wm.verify_persistent(B, w.n_kv_heads, Hq, self.T, D, self.kv.capacity) > 0
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
        verify = 3 if self.v_persistent else 1 + (1 if self.v_splits > 1 else 0)  # (schedule,) attention, merge
        return self.d * per_draft + verify + 1

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

    def release(self):
        """Drop the graphs and device buffers of this workload."""
        self.graph = self.ev = None
        for name in ("inp", "kv", "ring", "base_len", "d_out", "d_lse", "v_out", "v_lse", "d_ws", "s_ws", "v_ws"):
            setattr(self, name, None)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()


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


def workload_config(w, depth: int, context, world: int) -> dict:
    """The workload a line reports on: the same keys in the GPU arm and the
    reference arm (how the GPU arm runs it goes under ``detail``)."""
    return {
        "workload": w.name, "batch": w.batch,
        "context": (context if context else w.context) if not w.ragged else f"U[{w.ragged[0]}, {w.ragged[1]}] seeded",
        "n_q_heads": w.n_q_heads, "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "sink": w.sink,
        "window": w.window, "draft_depth": depth, "verify_positions": depth + 1,
        "kv_layout": f"paged ({w.page_size}-token pages)" if w.page_size else "contiguous",
        "l2": "flushed between timed steps (write of a 2x L2 buffer, then a read of another 2x L2 buffer so the "
              "flush's dirty lines are written back before the step); each step also reads the full KV cache (> L2)",
        "parallelism": f"replicas x{world}",
    }


def verify_schedule(st: "Step") -> str:
    if st.v_persistent:
        return (f"persistent: {st.v_splits} CTAs, each an equal run of the batch's key tiles (schedule made on "
                "the device from the actual lengths), then the segment merge")
    return f"split plan: {st.v_splits} splits per (sequence, KV head)" + (", then the merge" if st.v_splits > 1 else "")


def step_bytes(st: "Step") -> tuple[int, int]:
    """Algorithmic HBM bytes of one verify launch and of one draft step."""
    w = st.w
    B, Hq, Hkv, D = w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim
    sum_n = sum(st.inp.seq_lens_host)
    verify_bytes = 2 * Hkv * D * 2 * sum_n + 2 * (B * st.T * Hq * D * 2) + B * st.T * Hq * 4
    draft_bytes = 2 * B * Hkv * w.slots * D * 2 + 2 * (B * Hq * D * 2) + B * Hq * 4
    return verify_bytes, draft_bytes


def time_graph(graph, flush, n_warm: int, n: int, ev=None):
    """Replay ``graph`` n_warm + n times with the L2 flushed before each replay;
    mean milliseconds of the last n replays, timed by CUDA events around the
    replay, or (``ev``) by the graph's own in-graph events (list of intervals)."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    ms = []
    for i in range(n_warm + n):
        flush()
        if ev is None:
            e0.record()
        graph.replay()
        if ev is None:
            e1.record()
            e1.synchronize()
        else:
            torch.cuda.synchronize()
        if i >= n_warm:
            ms.append(e0.elapsed_time(e1) if ev is None else [ev[k].elapsed_time(ev[k + 1]) for k in range(len(ev) - 1)])
    return ms


def graph_ms(st: "Step", fn, flush, args, n=None) -> float:
    """Mean milliseconds of ``fn`` captured as a graph of its own: the L2
    flushed before every replay (pass ``flush=lambda: None`` to keep it warm),
    CUDA events on the stream around the replay."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device=st.dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        fn()
    torch.cuda.synchronize()
    ms = time_graph(g, flush, max(3, args.warmup), n or args.steps)
    return sum(ms) / len(ms)


def parts(st: "Step", flush, args) -> dict:
    """The draft chain and the verify, each timed as a graph of its own, the
    way the step is (``graph_ms``).  Each graph ends with the ring rollback
    that resets the ring for the next replay, so a graph holding only that
    rollback is timed too and subtracted (it also carries the graph launch's
    own fixed cost); the other draft chains below are timed the same way.
    The draft graph is also replayed without the flush: the ring stays in L2
    from one replay to the next, as in a decode loop.  Milliseconds."""
    wm, w, inp = st.wm, st.w, st.inp

    def rollback():
        wm.ring_rollback(st.ring, st.base_len)

    def drafts():
        for j in range(st.d):
            st.draft(j)
        rollback()

    def verify():
        wm.verify_attn(st.kv, inp.q_verify, w.scale, out=st.v_out, lse=st.v_lse, workspace=st.v_ws)
        rollback()

    no_flush = lambda: None
    st.rollback_graph_ms = graph_ms(st, rollback, flush, args)
    d_graph, v_graph = graph_ms(st, drafts, flush, args), graph_ms(st, verify, flush, args)
    return {"draft_ms": d_graph - st.rollback_graph_ms, "verify_ms": v_graph - st.rollback_graph_ms,
            "draft_graph_ms": d_graph, "verify_graph_ms": v_graph,
            "draft_warm_ms": graph_ms(st, drafts, no_flush, args) - graph_ms(st, rollback, no_flush, args),
            "rollback_graph_ms": st.rollback_graph_ms}


def breakdown(st: "Step", flush, args) -> tuple[float, float]:
    """Mean draft-chain and verify milliseconds from a capture of the step with
    events between them (the events cost time themselves, so this graph is never
    the one the step time comes from)."""
    st.capture(events=True)
    if not st.ev:
        return None, None
    ms = time_graph(st.graph, flush, max(3, args.warmup), args.steps, ev=st.ev)
    return sum(m[0] for m in ms) / len(ms), sum(m[1] for m in ms) / len(ms)


def extra_1m_line(name: str, depth: int, device, flush, args, peak: float) -> dict:
    """Step, verify and draft of another 1M-context configuration, measured like
    the headline (graph of the step's kernels; L2 flushed between steps)."""
    w = workloads.get(name)
    st = Step(w, depth, device)
    st.capture(events=False)
    step_ms = time_graph(st.graph, flush, max(3, args.warmup), args.steps)
    pt = parts(st, flush, args)
    draft_ms, verify_ms = pt["draft_ms"], pt["verify_ms"]
    vb, db = step_bytes(st)
    out = {"step_us": round(1e3 * sum(step_ms) / len(step_ms), 2)}
    if verify_ms:
        vg = vb / (verify_ms * 1e-3) / 1e9
        dg = db * depth / (draft_ms * 1e-3) / 1e9
        out.update({"verify_us": round(1e3 * verify_ms, 2), "verify_gbs": round(vg, 1),
                    "verify_frac_of_hbm": round(vg / peak, 4),
                    "draft_us_per_step": round(1e3 * draft_ms / depth, 2), "draft_gbs": round(dg, 1),
                    "draft_frac_of_hbm": round(dg / peak, 4), "draft_kv_bytes_per_step": db,
                    "draft_splits": st.d_splits, "verify_splits": st.v_splits, "verify_schedule": verify_schedule(st),
                    "draft_us_per_step_cuda_cores": fma_draft_chain(st, flush, args)})
    st.release()
    return out


def launch_floors(w, device, flush, args) -> dict:
    """Measured floors of a dependent chain of draft-step launches, as graphs
    of d launches with the L2 flushed before each replay (per launch, us):
    ``empty_kernel``: a ring rollback that changes nothing (one tiny kernel);
    ``one_tile``: draft attention over a 64-slot ring (one 64-key tile per
    (sequence, KV head), one split: the attention kernel alone);
    ``one_tile_fused_step``: the fused draft step on that ring (attention, then
    the merge that commits the append: the two launches of every draft step)."""
    from speculative_decoding_attention_gb300 import wm

    B, Hq, Hkv, D = w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim
    d = 8
    gen = torch.Generator(device=device).manual_seed(77)
    ring = wm.Ring.create(B, Hkv, D, 0, 64, device)
    hist = torch.randn((B, Hkv, 64, D), generator=gen, device=device).to(torch.bfloat16)
    wm.ring_fill(ring, wm.KVCache(hist, hist, torch.full((B,), 64, dtype=torch.int64, device=device)))
    q = torch.randn((B, Hq, D), generator=gen, device=device).to(torch.bfloat16)
    kn = torch.randn((B, Hkv, D), generator=gen, device=device).to(torch.bfloat16)
    keep = torch.full((B,), 64, dtype=torch.int64, device=device)
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=device)
    ws = wm.step_workspace(ring, Hq, n_split=1)
    chains = {
        "empty_kernel": lambda: [wm.ring_rollback(ring, keep) for _ in range(d)],
        "one_tile": lambda: [wm.draft_attn(ring, q, w.scale, n_split=1, out=out, lse=lse) for _ in range(d)],
        "one_tile_fused_step": lambda: ([wm.draft_step(ring, kn, kn, q, w.scale, ws, n_split=1, out=out, lse=lse)
                                         for _ in range(d)], wm.ring_rollback(ring, keep)),
    }
    res = {}
    for name, fn in chains.items():
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=device)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=s):
            fn()
        ms = time_graph(g, flush, max(3, args.warmup), args.steps)
        res[name] = round(1e3 * sum(ms) / len(ms) / d, 2)
    res["note"] = (f"per launch (per draft step for the fused step), graphs of {d} dependent launches "
                   f"with the workload's batch {B}, KV heads {Hkv}, head_dim {D} and {Hq // Hkv} rows per KV head")
    return res


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

    step_ms = []
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)

    def untimed_step():
        flush()
        st.graph.replay()

    with ClockSampler(device) as clk:
        clk.load_until_sampled(untimed_step, 3)
        barrier(world)
        torch.cuda.synchronize()
        t_begin = time.monotonic()
        for _ in range(args.steps):
            flush()
            e0.record()
            timed_graph.replay()
            e1.record()
            e1.synchronize()
            step_ms.append(e0.elapsed_time(e1))
        torch.cuda.synchronize()
        t_end = time.monotonic()
        barrier(world)
        clk.mark(t_begin, t_end)
        clk.load_until_sampled(untimed_step, 2)
    clocks = clk.summary()
    pt = parts(st, flush, args)
    draft_ms, verify_ms = pt["draft_ms"], pt["verify_ms"]
    # Cross-check: the step captured with events between its draft chain and
    # its verify (the event nodes cost time themselves).
    ev_draft_ms, ev_verify_ms = breakdown(st, flush, args)
    if wm.get_device_error():
        raise RuntimeError("device error during the timed steps")
    out_ok = bool(torch.isfinite(st.v_out.float()).all() and torch.isfinite(st.d_out.float()).all())
    native_ms, native_step_ms = native_draft_chain(st, flush, args)
    unfused_ms = unfused_draft_chain(st, flush, args)
    masw = masw_draft_chain(st, flush, args)
    fma_us = fma_draft_chain(st, flush, args)

    us_step = max_over_ranks(1e3 * sum(step_ms) / len(step_ms), world, device)
    us_verify = 1e3 * verify_ms
    us_draft = 1e3 * draft_ms if draft_ms else None

    B, Hq, Hkv, D = w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim
    sum_n = sum(st.inp.seq_lens_host)
    verify_bytes, draft_bytes = step_bytes(st)
    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = peak or FALLBACK_HBM_GBS
    achieved = verify_bytes / (us_verify * 1e-6) / 1e9
    draft_gbs = draft_bytes * depth / (us_draft * 1e-6) / 1e9 if us_draft else None

    e2e = None if args.no_e2e else e2e_leg(st, args, world, device)
    floors = None if args.context else launch_floors(w, device, flush, args)
    # the other 1M-context configurations (the headline stays the default workload)
    others = {}
    if args.workload == workloads.BENCH_WORKLOAD and depth == workloads.BENCH_DEPTH and not args.context \
            and not args.no_extra:
        launches_before = st.launches_per_step()
        for name, dd in (("hybrid_1m_d256", 1), ("hybrid_1m_d256", 5), ("nope_1m_b2", 4)):
            others[f"{name}/d{dd}"] = extra_1m_line(name, dd, device, flush, args, peak)
        assert launches_before == st.launches_per_step()
    cpu = None
    if not args.no_cpu and rank == 0:
        cpu = cpu_baseline(st, args)

    if rank != 0:
        return
    config = workload_config(w, depth, args.context, world)
    if w.ragged:
        config["context_per_sequence"] = list(st.inp.seq_lens_host)
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
        "config": config,
        "detail": {
            "execution": "one CUDA graph per step holding the step's kernels only; the draft and verify figures "
                         "time the draft chain and the verify each as a graph of its own (L2 flushed before every "
                         "replay, events on the stream around it), each ending with the ring rollback, minus a "
                         "graph holding only that rollback",
            "draft_execution": "per draft step: one launch of ring append fused into the draft attention, "
                               "then the split merge (which commits the append)",
            "draft_splits": st.d_splits, "verify_splits": st.v_splits, "verify_schedule": verify_schedule(st),
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
            "draft_us_per_step_warm_l2": round(1e3 * pt["draft_warm_ms"] / depth, 2),
            "draft_warm_l2": "the draft chain's graph replayed without the flush: the ring stays in L2 from "
                             "replay to replay",
            "rollback_graph_us": round(1e3 * pt["rollback_graph_ms"], 2),
            "marginal_in_step": {"draft_us_per_step": round((us_step - 1e3 * pt["verify_graph_ms"]) / depth, 2),
                                 "verify_us": round(us_step - 1e3 * pt["draft_graph_ms"], 2),
                                 "note": "what each part adds to the whole step: the step minus the graph of the "
                                         "verify (with the rollback), and minus the graph of the draft chain (with "
                                         "the rollback)"},
            "in_graph_events": {"draft_us_per_step": None if ev_draft_ms is None else round(1e3 * ev_draft_ms / depth, 2),
                                "verify_us": None if ev_verify_ms is None else round(1e3 * ev_verify_ms, 2),
                                "note": "the same split from one capture of the whole step with events between its "
                                        "draft chain and its verify; the event nodes cost time themselves"},
            "draft_launch_floor_us": floors,
            "unfused_draft_us_per_step": None if unfused_ms is None else round(1e3 * unfused_ms / depth, 2),
            "draft_us_per_step_cuda_cores": fma_us,
            "draft_cuda_cores": "the same fused draft chain with the draft kernel's Q.K and P.V on the CUDA cores "
                                "(fp32 FMA, warp-shuffle softmax) instead of mma.sync, for comparison",
            "masw_draft": masw,
            "verify_kv_bytes": 2 * Hkv * D * 2 * sum_n,
            "outputs_finite": out_ok,
            "steps_per_s_all_ranks": round(world * 1e6 / us_step, 1),
            "native_draft_chain_us": round(1e3 * native_ms, 2),
            "native_draft_us_per_step": round(1e3 * native_ms / depth, 2),
            "native_step_us": round(1e3 * native_step_ms, 2),
            "native_over_windowed_step": round(1e3 * native_step_ms / us_step, 3),
            "other_1m_configs": others or None,
        },
        "roofline": {
            "kernel": ("verify_sched + attn_tcp_kernel (persistent tcgen05 verify) + seg_merge" if st.v_persistent
                       else "attn_tc_kernel (tcgen05 verify, split-KV) + lse_merge"),
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


def fma_draft_chain(st: Step, flush, args):
    """The fused draft chain with the draft kernel's products on the CUDA cores
    (fp32 FMA, warp-shuffle softmax) instead of mma.sync: the measurement behind
    the choice of tensor cores for the draft.  Mean us per draft step, timed as
    the draft chain of ``parts`` is."""
    wm, w, inp = st.wm, st.w, st.inp
    wm.set_draft_math(wm.WM_DRAFT_MATH_FMA)
    try:
        ws = wm.step_workspace(st.ring, w.n_q_heads)

        def chain():
            for j in range(st.d):
                wm.draft_step(st.ring, inp.k_new[j], inp.v_new[j], inp.q_draft[j], w.scale, ws, out=st.d_out[j],
                              lse=st.d_lse[j])
            wm.ring_rollback(st.ring, st.base_len)

        ms = graph_ms(st, chain, flush, args, n=max(3, args.steps // 2)) - st.rollback_graph_ms
    finally:
        wm.set_draft_math(wm.WM_DRAFT_MATH_MMA)
    return round(1e3 * ms / st.d, 2)


def unfused_draft_chain(st: Step, flush, args):
    """The draft chain as three launches per draft step (ring append, draft
    attention, split merge), timed as the draft chain of ``parts`` is.  Mean
    milliseconds per chain."""
    def chain():
        for j in range(st.d):
            st.draft(j, fused=False)
        st.wm.ring_rollback(st.ring, st.base_len)

    return graph_ms(st, chain, flush, args, n=max(3, args.steps // 2)) - st.rollback_graph_ms


MASW_SLOT_INTERVAL = 256  # one memory slot per 256 tokens of history


def masw_draft_chain(st: Step, flush, args):
    """The draft chain with memory slots (memory-augmented sliding window): the
    fused step over sinks + window + one materialized slot per
    MASW_SLOT_INTERVAL tokens of each sequence's history (synthetic slot K/V),
    timed as the draft chain of ``parts`` is."""
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

    def chain():
        for j in range(st.d):
            wm.draft_step(st.ring, inp.k_new[j], inp.v_new[j], inp.q_draft[j], w.scale, ws, out=st.d_out[j],
                          lse=st.d_lse[j], mem=mem)
        wm.ring_rollback(st.ring, st.base_len)

    us = 1e3 * (graph_ms(st, chain, flush, args, n=max(3, args.steps // 2)) - st.rollback_graph_ms) / st.d
    kv_bytes = 2 * Hkv * D * 2 * sum(w.slots + c for c in counts)
    return {"slot_interval": MASW_SLOT_INTERVAL, "slots": counts, "us_per_step": round(us, 2),
            "kv_bytes_per_step": kv_bytes, "gbs": round(kv_bytes / (us * 1e-6) / 1e9, 1)}


def native_draft_chain(st: Step, flush, args) -> tuple[float, float]:
    """The draft chain without windowing (the native MTP draft the pages compare
    against): each of the d draft steps attends over the whole cache, i.e. the
    verify kernel with one query position over positions 0..N_b+j.  Returns the
    mean milliseconds per chain and per native step (the chain followed by the
    verify and the rollback, like the windowed step), each graph-captured with
    the L2 flushed between replays."""
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
        wm.ring_rollback(st.ring, st.base_len)  # as in the windowed chain's graph (a no-op here)

    def step():  # the native step: the draft chain, then the same verify as the windowed step, then the rollback
        for j in range(st.d):
            wm.verify_attn(kvs[j], qs[j], w.scale, out=out, lse=lse, workspace=ws)
        wm.verify_attn(st.kv, inp.q_verify, w.scale, out=st.v_out, lse=st.v_lse, workspace=st.v_ws)
        wm.ring_rollback(st.ring, st.base_len)

    # the chain as the windowed chain is timed; the step as the windowed step is
    n = max(3, args.steps // 2)
    return graph_ms(st, chain, flush, args, n=n) - st.rollback_graph_ms, graph_ms(st, step, flush, args, n=n)


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

def oracle_step(w, depth, inp_host) -> tuple[float, float]:
    """One whole step on the host cores: every row of the d draft steps and
    every verify row, as the GPU computes them.  Returns (seconds of the draft
    steps, seconds of the verify)."""
    import oracle

    hist = oracle.KV(inp_host["k"], inp_host["v"], inp_host["block_table"])
    t0 = time.perf_counter()
    for j in range(depth):
        pos = [n + j for n in inp_host["lens"]]
        oracle.draft(hist, inp_host["q_draft"][j], pos, w.sink, w.window, w.scale)
    t1 = time.perf_counter()
    oracle.verify(hist, inp_host["q_verify"], inp_host["lens"], w.scale)
    return t1 - t0, time.perf_counter() - t1


def step_description(w, depth) -> str:
    return (f"whole steps: all {w.batch * w.n_q_heads} draft rows x {depth} draft steps + all "
            f"{w.batch * (depth + 1) * w.n_q_heads} verify rows of {w.name}")


def host_inputs(inp):
    return {"k": inp.k.cpu(), "v": inp.v.cpu(),
            "block_table": None if inp.block_table is None else inp.block_table.cpu(),
            "lens": list(inp.seq_lens_host), "q_draft": inp.q_draft.cpu(), "q_verify": inp.q_verify.cpu()}


def cpu_baseline(st: Step, args, min_seconds: float = 10.0) -> dict:
    """The oracle timed on whole steps of the workload (no sampling of rows,
    nothing scaled) until about ``min_seconds`` of CPU work have run."""
    import oracle

    oracle.set_num_threads(len(os.sched_getaffinity(0)))  # every host core this process may use
    inp_host = host_inputs(st.inp)
    oracle_step(st.w, st.d, inp_host)  # warm-up: page faults, thread pool
    drafts, verifies = [], []
    while sum(drafts) + sum(verifies) < min_seconds or not drafts:
        dr, ve = oracle_step(st.w, st.d, inp_host)
        drafts.append(dr)
        verifies.append(ve)
    n = len(drafts)
    per_step = (sum(drafts) + sum(verifies)) / n
    return {"value": round(1e6 * per_step, 1), "unit": UNIT,
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} {step_description(st.w, st.d)} (1 untimed)",
            "sample_seconds": round(sum(drafts) + sum(verifies), 2),
            "draft_us_per_step": round(1e6 * sum(drafts) / n / st.d, 1),
            "verify_us": round(1e6 * sum(verifies) / n, 1)}


def reference_arm(args, rank, world, local):
    """The fp64 CPU oracle on the host cores, on the GPU arm's workload: each
    warm-up and timed step is one whole step (every draft and verify row)."""
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
    inp = wm_inputs.make_inputs(w, depth=depth, device=gen_dev, context=args.context)
    inp_host = host_inputs(inp)
    lens = list(inp.seq_lens_host)
    del inp
    for _ in range(args.warmup):
        oracle_step(w, depth, inp_host)
    drafts, verifies = [], []
    for _ in range(args.steps):
        dr, ve = oracle_step(w, depth, inp_host)
        drafts.append(dr)
        verifies.append(ve)
    us = 1e6 * (sum(drafts) + sum(verifies)) / args.steps
    config = workload_config(w, depth, args.context, world)
    if w.ragged:
        config["context_per_sequence"] = lens
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) K/V and queries in the workload's shapes; no dataset)",
        "config": config,
        "detail": {"execution": "the fp64 oracle (plain C, OpenMP over rows) on the host cores, one whole step "
                                "per timed step"},
        "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"{args.steps} {step_description(w, depth)}",
                         "draft_us_per_step": round(1e6 * sum(drafts) / args.steps / depth, 1),
                         "verify_us": round(1e6 * sum(verifies) / args.steps, 1)},
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
