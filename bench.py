"""Benchmark of the paged-KV attention hot path on one GB300 (or N replicas).

A step is one decode step of a 32-layer Llama-3-8B-shaped model's attention:
for every layer, wf_reshape_and_cache writes the B new tokens' K/V into that
layer's pool and wf_paged_decode attends each sequence over its whole paged
context (H_q=32, H_kv=8, D=128, P=16, bf16, B=231 by default).  Every layer has
its own pool (~2.2 GB with the allocator's headroom), so each launch streams
from HBM, never from the 129 MB L2.

Printed (rank 0, one JSON line): sequences*layers/s, the decode call's roofline
against the measured HBM copy bandwidth, an end-to-end figure through host
buffers, the oracle's CPU time on a bounded sample, launch count and clocks.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--batch 118|231]
                    [--workload llama8b|gpt2|llama1b|mixed|cow] [--kv bf16|fp8]
                    [--impl wf|reference] [--no-graph]

Under torchrun each rank runs its own replica on its own GPU (no data-path
collective; sequences are independent) and the slowest rank's time counts.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_wf_gb300 import workloads as W  # noqa: E402

METRIC = "paged decode attention: sequences·layers/s and achieved HBM GB/s (% of ~8 TB/s)"
UNIT = "seq·layers/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------
# environment
# ---------------------------------------------------------------------------
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def max_over_ranks(pg, x: float, device: str = "cuda") -> float:
    """The largest of every rank's value (replicas are timed by their slowest rank);
    x itself without a process group."""
    if pg is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, units_per_rank: float, ms: float) -> float:
    """Whole-job throughput: every rank processes units_per_rank in ms (the slowest
    rank's time)."""
    return world * units_per_rank / (ms / 1e3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_digest(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "paged_kv_cache_wf_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key: str, workload: str):
    """Per-launch DRAM bytes from a committed ncu summary, if taken on this exact source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel_key)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("workload") != workload:
        return None
    if rec.get("source_sha") != source_digest(rec.get("sources", [])):
        return None
    return rec.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"wf_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[4:8]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# algorithmic bytes (what the method must move; no block padding)
# ---------------------------------------------------------------------------
def decode_bytes(lay, kv_bytes=None) -> int:
    g = lay.geom
    e = W.elt_size(g.dtype)
    ekv = e if kv_bytes is None else kv_bytes
    kv = int(2 * lay.seq_lens.astype(np.int64).sum() * g.H_kv * g.D * ekv)
    qo = 2 * lay.B * g.H_q * g.D * e
    tables = int(sum(-(-int(s) // g.P) for s in lay.seq_lens) * 4) + 4 * lay.B
    return kv + qo + tables


def scatter_bytes(T: int, g, kv_bytes=None) -> int:
    e = W.elt_size(g.dtype)
    ekv = e if kv_bytes is None else kv_bytes
    return 2 * T * g.H_kv * g.D * (e + ekv) + 8 * T


def prefill_flops(lay) -> float:
    g = lay.geom
    tot = 0
    for b in range(lay.B):
        c, n = int(lay.prefix_lens[b]), int(lay.q_lens[b])
        tot += n * c + n * (n + 1) // 2          # sum_{i<n} (c + i + 1)
    return 4.0 * g.H_q * g.D * tot


# ---------------------------------------------------------------------------
# the wf arm
# ---------------------------------------------------------------------------
class DecodeWorkload:
    """L layers of (scatter of B new tokens, paged decode), one pool per layer.

    kv="fp8": the pools hold e4m3 codes (one byte an element) of the same draws,
    with k_scale = v_scale = value_scale / 64; q, the new rows and the outputs stay
    bf16 and the scatter quantizes."""

    def __init__(self, lay, layers: int, seed: int, kv: str = "bf16"):
        import torch
        from paged_kv_cache_wf_gb300 import binding as wf
        self.torch, self.wf = torch, wf
        self.lib = wf.load()
        self.lay = lay
        g = lay.geom
        self.L = layers
        self.kv = kv
        self.k_scale = self.v_scale = 1.0
        if kv == "fp8":
            self.k_scale = self.v_scale = g.value_scale / 64.0
            self.pools = [self._fp8_pools(seed + 17 * l) for l in range(layers)]
        else:
            self.pools = [W.device_pools(lay, seed=seed + 17 * l) for l in range(layers)]
        self.vals = [W.device_step_values(lay, seed=seed + 17 * l + 5) for l in range(layers)]
        self.outs = [torch.empty_like(v[0]) for v in self.vals]
        self.bt = torch.from_numpy(lay.block_tables).cuda()
        self.sl = torch.from_numpy(lay.seq_lens).cuda()
        self.slots = torch.from_numpy(lay.new_slots()).cuda()
        self.desc = wf.pool_desc(self.pools[0][0], self.k_scale, self.v_scale)
        self.max_seq_len = lay.max_seq_len
        self.ws_bytes = wf.wf_paged_decode_workspace_size(lay.B, g.H_q, self.max_seq_len, self.desc)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.scale = 1.0 / math.sqrt(g.D)
        self.stream = torch.cuda.current_stream()
        self.sp = self.stream.cuda_stream
        # scatter, the grid that zeroes the work queue (fp8: and prepares q), the
        # split kernel, and the combine when any sequence has more than one split
        self.launches_per_layer = (3 if self.tensor_cores() else 2) + (
            1 if -(-self.max_seq_len // self.split_span()) > 1 else 0)

    def tensor_cores(self) -> bool:
        """Whether the library runs this decode on its tensor-core kernel."""
        g = self.lay.geom
        shape = g.H_kv == 8 and g.P % 16 == 0 and g.H_q // g.H_kv in (2, 4)
        return shape and (g.D == 128 if self.kv == "fp8" else g.D in (64, 128))

    def split_span(self) -> int:
        """Positions per decode work item: 256 on the tensor cores for fp8 pools and
        for bf16 at D=128, 128 for bf16 at D=64, 64 on the CUDA cores."""
        if not self.tensor_cores():
            return 64
        return 256 if self.kv == "fp8" or self.lay.geom.D == 128 else 128

    def _fp8_pools(self, seed):
        """e4m3 codes of the bf16 draws (torch's conversion after clamping to +-448;
        NaN slots stay NaN codes)."""
        torch = self.torch
        kb, vb = W.device_pools(self.lay, seed=seed)
        kp = (kb.float() / self.k_scale).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
        vp = (vb.float() / self.v_scale).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
        del kb, vb
        return kp, vp

    def kv_bytes(self) -> int:
        return 1 if self.kv == "fp8" else W.elt_size(self.lay.geom.dtype)

    def _scatter(self, l, k=None, v=None, slots=None):
        kp, vp = self.pools[l]
        kk = k if k is not None else self.vals[l][1]
        vv = v if v is not None else self.vals[l][2]
        ss = slots if slots is not None else self.slots
        rc = self.lib.wf_reshape_and_cache(kk.data_ptr(), vv.data_ptr(), kp.data_ptr(), vp.data_ptr(),
                                           ss.data_ptr(), int(ss.shape[0]), self.desc, self.status.data_ptr(),
                                           self.sp)
        assert rc == 0, rc

    def _decode(self, l, q=None, bt=None, sl=None, out=None):
        kp, vp = self.pools[l]
        qq = q if q is not None else self.vals[l][0]
        oo = out if out is not None else self.outs[l]
        bt = bt if bt is not None else self.bt
        sl = sl if sl is not None else self.sl
        rc = self.lib.wf_paged_decode(oo.data_ptr(), qq.data_ptr(), kp.data_ptr(), vp.data_ptr(), bt.data_ptr(),
                                      int(bt.shape[1]), sl.data_ptr(), self.lay.B, self.max_seq_len,
                                      self.lay.geom.H_q, self.scale, self.desc, self.ws.data_ptr(), self.ws_bytes,
                                      self.status.data_ptr(), self.sp)
        assert rc == 0, rc

    def step(self, events=None):
        for l in range(self.L):
            self._scatter(l)
            if events is not None:
                e0, e1 = events.pop()
                e0.record(self.stream)
                self._decode(l)
                e1.record(self.stream)
                self._ev_done.append((e0, e1))
            else:
                self._decode(l)

    def timed(self, steps: int, per_launch: bool = True):
        torch = self.torch
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps * self.L)] if per_launch else None
        self._ev_done = []
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]   # step boundaries
        marks[0].record(self.stream)
        for i in range(steps):
            self.step(ev)
            marks[i + 1].record(self.stream)
        marks[-1].synchronize()
        total_ms = marks[0].elapsed_time(marks[-1])
        self.step_ms = [marks[i].elapsed_time(marks[i + 1]) for i in range(steps)]
        launch_ms = [a.elapsed_time(b) for a, b in self._ev_done] if per_launch else []
        return total_ms, launch_ms


def spread(xs):
    """median, p10 and p90 of a list of timings (nearest-rank)."""
    ys = sorted(xs)
    if not ys:
        return None
    pick = lambda q: ys[min(len(ys) - 1, max(0, int(math.ceil(q * len(ys))) - 1))]
    return {"median": statistics.median(ys), "p10": pick(0.10), "p90": pick(0.90), "n": len(ys)}


def graph_timed(wl, steps: int) -> float:
    """The workload's step captured once as a CUDA graph (on a side stream, as
    torch requires) and replayed: ms per replayed step, CUDA events around
    `steps` replays after three warm-up replays."""
    torch = wl.torch
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(wl.stream)
    eager_sp = wl.sp
    with torch.cuda.stream(side):
        wl.sp = side.cuda_stream           # every call of the step goes to the capture stream
        try:
            with torch.cuda.graph(graph, stream=side):
                wl.step()
        finally:
            wl.sp = eager_sp
    wl.stream.wait_stream(side)
    with torch.cuda.stream(wl.stream):
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(wl.stream)
        for _ in range(steps):
            graph.replay()
        end.record(wl.stream)
        end.synchronize()
    return start.elapsed_time(end) / steps


class E2EDecode:
    """The same step through host buffers: per layer, q / k_new / v_new come from
    pinned host memory and the attention output goes back to pinned host memory;
    block tables, lengths and slots are uploaded once per step.  The copies run on a
    copy stream, as an engine would issue them: layer l + 1's inputs upload into the
    other of two device input sets while layer l computes, and layer l's output is
    read back as soon as its decode is done.  Every copy is inside the timed region."""

    def __init__(self, wl: DecodeWorkload):
        torch = wl.torch
        self.wl = wl
        self.h_vals = [tuple(t.cpu().pin_memory() for t in v) for v in wl.vals]
        self.h_out = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in wl.outs]
        self.h_bt = wl.bt.cpu().pin_memory()
        self.h_sl = wl.sl.cpu().pin_memory()
        self.h_slots = wl.slots.cpu().pin_memory()
        self.d_sets = [[torch.empty_like(t) for t in wl.vals[0]] for _ in range(2)]
        self.d_bt, self.d_sl, self.d_slots = (torch.empty_like(wl.bt), torch.empty_like(wl.sl),
                                              torch.empty_like(wl.slots))
        self.cs = torch.cuda.Stream()          # host <-> device copies
        nb = lambda t: t.numel() * t.element_size()
        self.h2d = (sum(nb(t) for v in self.h_vals for t in v) + nb(self.h_bt) + nb(self.h_sl)
                    + nb(self.h_slots))
        self.d2h = sum(nb(t) for t in self.h_out)

    def step(self, after):
        """One step; its copies start after event `after`.  Returns the event that
        marks the last output copied back.  On the copy stream, layer l + 1's upload
        is issued before layer l's read-back (which waits for layer l's decode), so it
        overlaps layer l's kernels."""
        torch, wl, cs, comp = self.wl.torch, self.wl, self.cs, self.wl.stream
        cs.wait_event(after)
        with torch.cuda.stream(cs):
            self.d_bt.copy_(self.h_bt, non_blocking=True)
            self.d_sl.copy_(self.h_sl, non_blocking=True)
            self.d_slots.copy_(self.h_slots, non_blocking=True)
        done = [None] * wl.L
        ready = [None] * wl.L

        def upload(l):
            if l >= 2:
                cs.wait_event(done[l - 2])       # the input set is free again
            q, k, v = self.d_sets[l & 1]
            hq, hk, hv = self.h_vals[l]
            with torch.cuda.stream(cs):
                q.copy_(hq, non_blocking=True)
                k.copy_(hk, non_blocking=True)
                v.copy_(hv, non_blocking=True)
            ready[l] = torch.cuda.Event()
            ready[l].record(cs)

        upload(0)
        for l in range(wl.L):
            if l + 1 < wl.L:
                upload(l + 1)
            q, k, v = self.d_sets[l & 1]
            comp.wait_event(ready[l])
            wl._scatter(l, k, v, self.d_slots)
            wl._decode(l, q, self.d_bt, self.d_sl, wl.outs[l])
            done[l] = torch.cuda.Event()
            done[l].record(comp)
            cs.wait_event(done[l])
            with torch.cuda.stream(cs):
                self.h_out[l].copy_(wl.outs[l], non_blocking=True)
        last = torch.cuda.Event()
        last.record(cs)
        return last

    def timed(self, steps: int):
        torch = self.wl.torch
        s = self.wl.stream
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(s)
        mark = start
        for _ in range(steps):
            mark = self.step(mark)
        s.wait_event(mark)
        end.record(s)
        end.synchronize()
        return start.elapsed_time(end)


class MixedWorkload:
    """L layers of a mixed continuous-batching step at Llama-3-8B shapes: one
    scatter of every new token (prefill and decode rows), the causal prefill of the
    prefill requests and the decode of the decode sequences, all on one pool per layer."""

    def __init__(self, pf, dc, layers: int, seed: int):
        import torch
        from paged_kv_cache_wf_gb300 import binding as wf
        self.torch, self.wf = torch, wf
        self.lib = wf.load()
        self.pf, self.dc = pf, dc
        g = pf.geom
        self.L = layers
        self.pools = [W.device_pools([pf, dc], seed=seed + 17 * l) for l in range(layers)]
        self.pvals = [W.device_step_values(pf, seed=seed + 17 * l + 5) for l in range(layers)]
        self.dvals = [W.device_step_values(dc, seed=seed + 17 * l + 9) for l in range(layers)]
        self.knew = [torch.cat([a[1], b[1]]) for a, b in zip(self.pvals, self.dvals)]
        self.vnew = [torch.cat([a[2], b[2]]) for a, b in zip(self.pvals, self.dvals)]
        self.pouts = [torch.empty_like(v[0]) for v in self.pvals]
        self.douts = [torch.empty_like(v[0]) for v in self.dvals]
        self.slots = torch.from_numpy(np.concatenate([pf.new_slots(), dc.new_slots()])).cuda()
        self.pbt = torch.from_numpy(pf.block_tables).cuda()
        self.psl = torch.from_numpy(pf.seq_lens).cuda()
        self.pcu = torch.from_numpy(pf.cu_q_lens).cuda()
        self.dbt = torch.from_numpy(dc.block_tables).cuda()
        self.dsl = torch.from_numpy(dc.seq_lens).cuda()
        self.desc = wf.pool_desc(self.pools[0][0])
        self.ws_bytes = wf.wf_paged_decode_workspace_size(dc.B, g.H_q, dc.max_seq_len, self.desc)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.scale = 1.0 / math.sqrt(g.D)
        self.stream = torch.cuda.current_stream()
        self.sp = self.stream.cuda_stream
        self.launches_per_layer = 1 + 1 + 3   # scatter, prefill, queue reset + decode + combine

    def layer(self, l, ev=None):
        kp, vp = self.pools[l]
        g = self.pf.geom
        rc = self.lib.wf_reshape_and_cache(self.knew[l].data_ptr(), self.vnew[l].data_ptr(), kp.data_ptr(),
                                           vp.data_ptr(), self.slots.data_ptr(), int(self.slots.shape[0]),
                                           self.desc, self.status.data_ptr(), self.sp)
        assert rc == 0, rc
        if ev is not None:
            ev[0].record(self.stream)
        q = self.pvals[l][0]
        rc = self.lib.wf_paged_prefill(self.pouts[l].data_ptr(), q.data_ptr(), kp.data_ptr(), vp.data_ptr(),
                                       self.pbt.data_ptr(), int(self.pbt.shape[1]), self.psl.data_ptr(),
                                       self.pcu.data_ptr(), self.pf.B, int(q.shape[0]), self.pf.max_q_len,
                                       self.pf.max_seq_len, g.H_q, self.scale, self.desc, self.status.data_ptr(),
                                       self.sp)
        assert rc == 0, rc
        if ev is not None:
            ev[1].record(self.stream)
        q = self.dvals[l][0]
        rc = self.lib.wf_paged_decode(self.douts[l].data_ptr(), q.data_ptr(), kp.data_ptr(), vp.data_ptr(),
                                      self.dbt.data_ptr(), int(self.dbt.shape[1]), self.dsl.data_ptr(), self.dc.B,
                                      self.dc.max_seq_len, g.H_q, self.scale, self.desc, self.ws.data_ptr(),
                                      self.ws_bytes, self.status.data_ptr(), self.sp)
        assert rc == 0, rc
        if ev is not None:
            ev[2].record(self.stream)

    def step(self, evs=None):
        for l in range(self.L):
            self.layer(l, evs.pop() if evs is not None else None)

    def step_one_call(self):
        """The step with each layer's prefill and decode in one wf_paged_prefill_decode
        call (one grid when the shapes allow it)."""
        g = self.pf.geom
        for l in range(self.L):
            kp, vp = self.pools[l]
            rc = self.lib.wf_reshape_and_cache(self.knew[l].data_ptr(), self.vnew[l].data_ptr(), kp.data_ptr(),
                                               vp.data_ptr(), self.slots.data_ptr(), int(self.slots.shape[0]),
                                               self.desc, self.status.data_ptr(), self.sp)
            assert rc == 0, rc
            pq, dq = self.pvals[l][0], self.dvals[l][0]
            rc = self.lib.wf_paged_prefill_decode(
                self.pouts[l].data_ptr(), pq.data_ptr(), self.pbt.data_ptr(), int(self.pbt.shape[1]),
                self.psl.data_ptr(), self.pcu.data_ptr(), self.pf.B, int(pq.shape[0]), self.pf.max_q_len,
                self.pf.max_seq_len, self.douts[l].data_ptr(), dq.data_ptr(), self.dbt.data_ptr(),
                int(self.dbt.shape[1]), self.dsl.data_ptr(), self.dc.B, self.dc.max_seq_len, kp.data_ptr(),
                vp.data_ptr(), g.H_q, self.scale, self.desc, self.ws.data_ptr(), self.ws_bytes,
                self.status.data_ptr(), self.sp)
            assert rc == 0, rc

    def timed_one_call(self, steps: int) -> float:
        torch = self.torch
        for _ in range(2):
            self.step_one_call()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        torch.cuda.synchronize()
        ev[0].record(self.stream)
        for _ in range(steps):
            self.step_one_call()
        ev[1].record(self.stream)
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[1])

    def step_two_streams(self, side):
        """The step with each layer's decode on a second stream beside its prefill
        (both read the pool after the layer's scatter and are independent), as an
        engine can issue them; the next layer starts after both."""
        torch, g = self.torch, self.pf.geom
        for l in range(self.L):
            kp, vp = self.pools[l]
            rc = self.lib.wf_reshape_and_cache(self.knew[l].data_ptr(), self.vnew[l].data_ptr(), kp.data_ptr(),
                                               vp.data_ptr(), self.slots.data_ptr(), int(self.slots.shape[0]),
                                               self.desc, self.status.data_ptr(), self.sp)
            assert rc == 0, rc
            side.wait_stream(self.stream)
            q = self.dvals[l][0]
            rc = self.lib.wf_paged_decode(self.douts[l].data_ptr(), q.data_ptr(), kp.data_ptr(), vp.data_ptr(),
                                          self.dbt.data_ptr(), int(self.dbt.shape[1]), self.dsl.data_ptr(), self.dc.B,
                                          self.dc.max_seq_len, g.H_q, self.scale, self.desc, self.ws.data_ptr(),
                                          self.ws_bytes, self.status.data_ptr(), side.cuda_stream)
            assert rc == 0, rc
            q = self.pvals[l][0]
            rc = self.lib.wf_paged_prefill(self.pouts[l].data_ptr(), q.data_ptr(), kp.data_ptr(), vp.data_ptr(),
                                           self.pbt.data_ptr(), int(self.pbt.shape[1]), self.psl.data_ptr(),
                                           self.pcu.data_ptr(), self.pf.B, int(q.shape[0]), self.pf.max_q_len,
                                           self.pf.max_seq_len, g.H_q, self.scale, self.desc, self.status.data_ptr(),
                                           self.sp)
            assert rc == 0, rc
            self.stream.wait_stream(side)

    def timed_two_streams(self, steps: int) -> float:
        torch = self.torch
        side = torch.cuda.Stream()
        for _ in range(2):
            self.step_two_streams(side)
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(self.stream)
        for _ in range(steps):
            self.step_two_streams(side)
        end.record(self.stream)
        end.synchronize()
        return start.elapsed_time(end)

    def timed(self, steps: int):
        torch = self.torch
        evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps * self.L)]
        used = list(evs)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(self.stream)
        for _ in range(steps):
            self.step(evs)
        end.record(self.stream)
        end.synchronize()
        pre = [a.elapsed_time(b) for a, b, _ in used]
        dec = [b.elapsed_time(c) for _, b, c in used]
        return start.elapsed_time(end), pre, dec


def run_cow(args, rank, world):
    """Secondary line: the copy-on-write block copy of prefix sharing at Llama-3-8B
    block size (32 KB a block and pool), 4096 pairs a call; 0.5 GB moved per call,
    larger than L2."""
    import torch
    from paged_kv_cache_wf_gb300 import binding as wf
    lib = wf.load()
    geom, pairs = W.cow_copy_workload(n_pairs=4096, seed=rank)
    shape = (geom.N, geom.P, geom.H_kv, geom.D)
    gen = torch.Generator(device="cuda").manual_seed(11 + rank)
    kp = torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16)
    vp = torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16)
    pr = torch.from_numpy(pairs).cuda()
    desc = wf.pool_desc(kp)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sp = torch.cuda.current_stream().cuda_stream
    block_bytes = geom.P * geom.H_kv * geom.D * 2
    moved = 2 * 2 * pairs.shape[0] * block_bytes          # K and V, read and written

    def call():
        rc = lib.wf_copy_blocks(kp.data_ptr(), vp.data_ptr(), pr.data_ptr(), int(pairs.shape[0]), desc,
                                status.data_ptr(), sp)
        assert rc == 0, rc

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    if wf.wf_device_status_fetch(status) != 0:
        raise SystemExit("device status flagged an error during warm-up")
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in evs:
        a.record()
        call()
        b.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    t = statistics.mean(a.elapsed_time(b) for a, b in evs) / 1e3
    peaks, src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    if rank == 0:
        print(json.dumps({
            "metric": "copy-on-write block copy (prefix sharing): blocks/s", "value": world * pairs.shape[0] / t,
            "unit": "blocks/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "cow_copy_llama8b_block", "pairs": int(pairs.shape[0]), "block_bytes": block_bytes,
                       "N": geom.N, "l2": "0.5 GB moved per call, larger than L2"},
            "roofline": {"kernel": "wf_copy_blocks", "bound": "hbm", "achieved": moved / t / 1e9, "peak": hbm,
                         "unit": "GB/s", "frac": moved / t / 1e9 / hbm, "peak_source": src,
                         "algorithmic_bytes_per_launch": moved, "avg_launch_us": t * 1e6, "traffic": None},
            "gpu_launches": args.steps, "clocks": clk}), flush=True)


def run_mixed(args, rank, world):
    """Secondary line: the mixed prefill + decode step (all three calls)."""
    import torch
    pf, dc = W.mixed_step(0)
    g = pf.geom
    L = args.layers if args.layers > 0 else g.L
    wl = MixedWorkload(pf, dc, L, seed=3000 + 7919 * rank)
    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize()
    if wl.wf.wf_device_status_fetch(wl.status) != 0:
        raise SystemExit("device status flagged an error during warm-up")
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    total_ms, pre_ms, dec_ms = wl.timed(args.steps)
    clk = clocks.stop()
    two_ms = wl.timed_two_streams(args.steps) / args.steps
    if wl.wf.wf_device_status_fetch(wl.status) != 0:
        raise SystemExit("device status flagged an error during the two-stream steps")
    one_ms = wl.timed_one_call(args.steps) / args.steps
    if wl.wf.wf_device_status_fetch(wl.status) != 0:
        raise SystemExit("device status flagged an error during the one-call steps")
    peaks, src = load_peaks()
    ms_step = total_ms / args.steps
    flops = prefill_flops(pf)
    pre_s = statistics.mean(pre_ms) / 1e3
    dec_s = statistics.mean(dec_ms) / 1e3
    dbytes = decode_bytes(dc)
    tok = int(pf.q_lens.sum()) + dc.B
    tflops = flops / pre_s / 1e12
    peak_t = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    line = {
        "metric": "mixed prefill+decode step: new tokens·layers/s", "value": world * tok * L / (ms_step / 1e3),
        "unit": "tokens·layers/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "mixed_llama8b", "prefill_requests": pf.B, "prefill_tokens": int(pf.q_lens.sum()),
                   "decode_sequences": dc.B, "layers": L, "model_layers": g.L, "H_q": g.H_q, "H_kv": g.H_kv,
                   "D": g.D, "P": g.P,
                   "l2": "inputs larger than L2: each layer has its own pools (%.2f GB), read once per step"
                         % (2 * g.N * g.P * g.H_kv * g.D * W.elt_size(g.dtype) / 1e9)},
        "roofline": {"kernel": "wf_paged_prefill", "bound": "tensor", "achieved": tflops, "peak": peak_t,
                     "unit": "TFLOP/s", "frac": tflops / peak_t, "peak_source": src,
                     "algorithmic_flops_per_launch": flops, "avg_launch_us": pre_s * 1e6,
                     "traffic": recorded_traffic("paged_prefill", "mixed_llama8b")},
        "decode_roofline": {"kernel": "wf_paged_decode", "bound": "hbm", "achieved": dbytes / dec_s / 1e9,
                            "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                            "frac": dbytes / dec_s / 1e9 / float(peaks["hbm_gbs"]),
                            "algorithmic_bytes_per_launch": dbytes, "avg_launch_us": dec_s * 1e6},
        "gpu_launches": args.steps * L * wl.launches_per_layer,
        "two_streams": {"value": world * tok * L / (two_ms / 1e3), "unit": "tokens·layers/s", "ms_per_step": two_ms,
                        "note": "each layer's decode on a second stream beside its prefill, timed separately "
                                "after the main run; the kernel rooflines above come from the sequential run"},
        "one_call": {"value": world * tok * L / (one_ms / 1e3), "unit": "tokens·layers/s", "ms_per_step": one_ms,
                     "fused": bool(wl.wf.wf_paged_prefill_decode_fused(wl.desc, g.H_q)),
                     "note": "each layer's prefill and decode in one wf_paged_prefill_decode call (one grid: "
                             "prefill CTAs first, then persistent decode CTAs that fill the SMs the prefill's "
                             "tail leaves idle), timed separately after the main run"},
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the oracle (reference arm and CPU baseline)
# ---------------------------------------------------------------------------
def oracle_sample_inputs(lay, seed: int, wl=None, kv: str = "bf16", kv_scales=(1.0, 1.0)):
    """Host inputs of one layer for the oracle: the blocks the batch uses and this
    step's new rows.  Taken from the device pools when a wf workload exists (the
    values the GPU sees), else drawn on the host."""
    g = lay.geom
    if wl is not None:
        torch = wl.torch
        kp, vp = wl.pools[0]
        q, kn, vn = wl.vals[0]
        nb = [-(-int(s) // g.P) for s in lay.seq_lens]
        used = np.unique(np.concatenate([lay.block_tables[b, :n] for b, n in enumerate(nb)]))
        remap = np.zeros(g.N, np.int32)
        remap[used] = np.arange(used.shape[0], dtype=np.int32)
        idx = torch.from_numpy(used.astype(np.int64)).cuda()
        bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
        codes = lambda t: t.cpu().numpy()
        pool_host = codes if wl.kv == "fp8" else bits
        # pool contents before this step's write: the new slots are NaN in both
        hk, hv = pool_host(kp.index_select(0, idx)), pool_host(vp.index_select(0, idx))
        bt = np.zeros_like(lay.block_tables)
        for b, n in enumerate(nb):
            bt[b, :n] = remap[lay.block_tables[b, :n]]
        sub = W.Layout(W.Geometry(g.H_q, g.H_kv, g.D, g.P, used.shape[0], g.dtype), lay.seq_lens, lay.q_lens,
                       bt, 0)
        return sub, hk, hv, bits(q), bits(kn), bits(vn)
    rng = np.random.default_rng(seed)
    vals = W.draw_layer_values(lay, rng)
    import oracle
    if kv == "fp8":
        hk = np.full((g.N, g.P, g.H_kv, g.D), 0x7F, np.uint8)     # e4m3 NaN code
        hv = hk.copy()
        oracle.reshape_and_cache_fp8(vals.k_prefix, vals.v_prefix, hk, hv, lay.prefix_slots(), *kv_scales)
    else:
        hk, hv = W.empty_pool(g), W.empty_pool(g)
        oracle.reshape_and_cache(vals.k_prefix, vals.v_prefix, hk, hv, lay.prefix_slots(), g.dtype)
    return lay, hk, hv, vals.q, vals.k_new, vals.v_new


def oracle_time(sub, hk, hv, q, kn, vn, min_seconds: float, max_reps: int, fp8_scales=None):
    """Time scatter + decode of one layer of the batch in the oracle, repeated
    (fp8_scales = (k_scale, v_scale): e4m3 code pools)."""
    import oracle
    g = sub.geom
    scale = 1.0 / math.sqrt(g.D)
    slots = sub.new_slots()
    threads = os.cpu_count() or 1
    reps, t0 = 0, time.perf_counter()
    while True:
        kp, vp = hk.copy(), hv.copy()
        if fp8_scales is not None:
            ks, vs = fp8_scales
            oracle.reshape_and_cache_fp8(kn, vn, kp, vp, slots, ks, vs)
            oracle.paged_decode_fp8(q, kp, vp, sub.block_tables, sub.seq_lens, scale, ks, vs, threads)
        else:
            oracle.reshape_and_cache(kn, vn, kp, vp, slots, g.dtype)
            oracle.paged_decode(q, kp, vp, sub.block_tables, sub.seq_lens, scale, g.dtype, threads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= max_reps:
            return reps, el, threads


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------
def make_layout(args):
    sfx = "_fp8kv" if args.kv == "fp8" else ""
    if args.workload == "llama8b":
        return W.llama8b_decode(args.batch, seed=0), f"llama8b_decode_B{args.batch}{sfx}"
    if args.workload == "gpt2":
        return W.gpt2_decode(0), f"gpt2_decode_B32{sfx}"
    if args.workload == "llama1b":
        return W.llama1b_decode(0), f"llama1b_decode_B64{sfx}"
    raise SystemExit(f"unknown workload {args.workload}")


def run_reference(args, rank, world):
    if rank != 0:
        return
    lay, wname = make_layout(args)
    g = lay.geom
    L = g.L
    fp8 = (g.value_scale / 64.0,) * 2 if args.kv == "fp8" else None
    sub, hk, hv, q, kn, vn = oracle_sample_inputs(lay, seed=0, kv=args.kv, kv_scales=fp8 or (1.0, 1.0))
    for _ in range(max(0, args.warmup)):
        oracle_time(sub, hk, hv, q, kn, vn, 0.0, 1, fp8)
    times = []
    for _ in range(args.steps):
        reps, el, threads = oracle_time(sub, hk, hv, q, kn, vn, 0.0, 1, fp8)
        times.append(el)
    per_layer = sum(times) / len(times)
    value = lay.B / per_layer
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_layer * L * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wname, "B": lay.B, "layers": L, "H_q": g.H_q, "H_kv": g.H_kv, "D": g.D,
                   "P": g.P, "kv_dtype": "fp8_e4m3" if fp8 else g.dtype},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"each timed step = one layer of the {wname} batch (all {lay.B} sequences, "
                                   f"scatter + decode) in the fp64 oracle; ms_per_step scales it to {L} layers"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--batch", type=int, default=231, choices=[118, 231])
    ap.add_argument("--workload", default="llama8b", choices=["llama8b", "gpt2", "llama1b", "mixed", "cow"])
    ap.add_argument("--impl", default="wf", choices=["wf", "reference"])
    ap.add_argument("--kv", default="bf16", choices=["bf16", "fp8"],
                    help="KV pool format of the decode workloads (fp8: e4m3 codes)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-graph", action="store_true",
                    help="skip timing the step captured as one CUDA graph (reported under 'graph')")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: run this many layers instead of the model's (recorded in config)")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    rank, world, local = dist_env()

    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    assert torch.cuda.is_available(), "bench.py needs a CUDA GPU"
    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    from paged_kv_cache_wf_gb300 import build
    if rank == 0 or world == 1:
        build.build()
    if pg is not None:
        pg.barrier()

    if args.workload in ("mixed", "cow"):
        (run_mixed if args.workload == "mixed" else run_cow)(args, rank, world)
        if pg is not None:
            pg.destroy_process_group()
        return
    lay, wname = make_layout(args)
    g = lay.geom
    L = args.layers if args.layers > 0 else g.L
    wl = DecodeWorkload(lay, L, seed=1000 + 7919 * rank, kv=args.kv)
    fp8 = (wl.k_scale, wl.v_scale) if args.kv == "fp8" else None
    # oracle inputs are copied before any kernel of ours has touched the pools
    oracle_in = None
    if rank == 0 and not args.no_cpu_baseline:
        oracle_in = oracle_sample_inputs(lay, 0, wl)
    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize()
    if wl.wf.wf_device_status_fetch(wl.status) != 0:
        raise SystemExit("device status flagged an error during warm-up")

    # ---- timed region ---------------------------------------------------------
    clocks = ClockSampler(torch.cuda.current_device())
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize()
    clocks.start()
    total_ms, launch_ms = wl.timed(args.steps, per_launch=True)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if wl.wf.wf_device_status_fetch(wl.status) != 0:
        raise SystemExit("device status flagged an error during the timed steps")
    total_ms = max_over_ranks(pg, total_ms)
    ms_per_step = total_ms / args.steps
    value = job_rate(world, lay.B * L, ms_per_step)

    # ---- roofline of the decode call (split + combine kernels) -------------------
    peaks, peak_src = load_peaks()
    kvb = wl.kv_bytes()
    dbytes = decode_bytes(lay, kvb)
    avg_launch_s = (sum(launch_ms) / len(launch_ms)) / 1e3
    achieved = dbytes / avg_launch_s / 1e9
    hbm = float(peaks["hbm_gbs"])
    step_bytes = L * (dbytes + scatter_bytes(lay.B, g, kvb))
    traffic = recorded_traffic("paged_decode_fp8" if fp8 else "paged_decode", wname)

    # ---- the same step as one replayed CUDA graph ---------------------------------------
    graph = None
    if not args.no_graph:
        g_ms = max_over_ranks(pg, graph_timed(wl, args.steps))
        if wl.wf.wf_device_status_fetch(wl.status) != 0:
            raise SystemExit("device status flagged an error during the graph replays")
        graph = {"value": job_rate(world, lay.B * L, g_ms), "unit": UNIT, "ms_per_step": g_ms,
                 "note": "the step (scatter + decode for every layer) captured once as a CUDA graph and replayed"}

    # ---- end to end through host buffers --------------------------------------------
    e2e = None
    if not args.no_e2e:
        ee = E2EDecode(wl)
        mark = torch.cuda.Event()
        mark.record(wl.stream)
        for _ in range(3):
            mark = ee.step(mark)
        torch.cuda.synchronize()
        if pg is not None:
            pg.barrier()
        e_ms = max_over_ranks(pg, ee.timed(args.steps) / args.steps)
        e2e = {"value": job_rate(world, lay.B * L, e_ms), "unit": UNIT, "ms_per_step": e_ms,
               "h2d_bytes_per_step": ee.h2d, "d2h_bytes_per_step": ee.d2h}
        del ee

    # ---- oracle on the host cores (rank 0 only) ------------------------------------------
    cpu = None
    if oracle_in is not None:
        sub, hk, hv, q, kn, vn = oracle_in
        oracle_time(sub, hk, hv, q, kn, vn, 0.0, 1, fp8)  # warm
        reps, el, threads = oracle_time(sub, hk, hv, q, kn, vn, args.cpu_seconds, 1000, fp8)
        cpu = {"value": lay.B * reps / el, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"layer 0 of the {wname} batch (all {lay.B} sequences: scatter + decode), "
                         f"repeated {reps}x in {el:.1f} s with {threads} threads"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": ("e4m3 (e4m3 x e4m3 MMA, fp32 accumulate)" if wl.tensor_cores()
                                                     else "f32 (e4m3 codes widened to fp32)") if fp8 else "bf16", "data": "synthetic",
            "config": {"workload": wname, "B": lay.B, "layers": L, "model_layers": g.L, "H_q": g.H_q,
                       "H_kv": g.H_kv, "D": g.D, "P": g.P, "N_blocks_per_layer": g.N,
                       "kv_dtype": "fp8_e4m3" if fp8 else g.dtype,
                       "context_tokens": int(lay.seq_lens.sum()), "max_seq_len": lay.max_seq_len,
                       "l2": "inputs larger than L2: each layer's pools (%.2f GB) are read once per step, "
                             "and the step reads %.2f GB of pools between two reads of one layer's"
                             % (2 * g.N * g.P * g.H_kv * g.D * kvb / 1e9, L * 2 * g.N * g.P * g.H_kv * g.D * kvb / 1e9),
                       "parallelism": f"replicas{world}"},
            "step_ms_spread": spread(wl.step_ms),
            "hbm_gbs_step": step_bytes / (ms_per_step / 1e3) / 1e9,
            "pct_of_nominal_8tbs_step": 100.0 * step_bytes / (ms_per_step / 1e3) / 1e9 / NOMINAL_HBM_GBS,
            "roofline": {"kernel": "wf_paged_decode (split + combine)", "bound": "hbm", "achieved": achieved,
                         "peak": hbm, "unit": "GB/s", "frac": achieved / hbm, "peak_source": peak_src,
                         "traffic": traffic, "algorithmic_bytes_per_launch": dbytes,
                         "avg_launch_us": avg_launch_s * 1e6,
                         "launch_us_spread": spread([x * 1e3 for x in launch_ms]),
                         "pct_of_nominal_8tbs": 100.0 * achieved / NOMINAL_HBM_GBS},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "graph": graph,
            "gpu_launches": args.steps * L * wl.launches_per_layer,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
