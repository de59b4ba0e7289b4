#!/usr/bin/env python
"""Paged decode attention benchmark: µs per batch and KV GB/s vs HBM peak.

One step = one pass of the whole hot path over one synthetic batch: plan on
the host (lengths -> split-KV work list -> H2D copy of the plan image), the
decode kernel, and the split-KV merge kernel (by default replayed as one CUDA
graph per workspace; ``--graph off`` launches them one by one).

By default (``--workload all``) the five workloads of
paged_kv_decode_plan_gb300.workloads are timed one after another with the
same steps and warm-up: the single request, the 64-request batch, the
256-request long tail, the cascade and, as the headline line, the
long-context batch (8 x 131072 tokens, Hq 64 / Hkv 8, P 64, bf16, >= 132
partial states per request + merge), the largest one that fits one GPU.  The
other four are reported under ``per_config`` in the same line.
``--workload NAME`` times one workload alone.  For the cascade workload a step
plans the suffix table (the shared prefix, which does not change between
decode steps, is planned once per workspace) and runs the shared-prefix
kernel, the suffix decode and the cascade merge (``--cascade fused``,
pkd_run_cascade's launches), or the prefix and suffix runs merged by
merge_states (``--cascade shared``), or the prefix listed in every request's
table (``--cascade per-request``).

Rank 0 prints one JSON line.  Under torchrun every rank runs the same batch
on its own GPU (weak scaling, no data-path collective); timing is the maximum
over ranks.  ``--impl reference`` times the fp64 CPU oracle instead, on the
headline workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("paged decode attention µs/batch and KV GB/s as fraction of "
          "GB300 HBM peak")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 129 * 1024 * 1024
GRAPH_COPIES_MAX_KV = 64 * 1024 * 1024
DESCRIPTIONS = {
    "single": "single-request decode: 1 x 512 tokens, Hq 32 / Hkv 8, D 128, P 16, fp16",
    "batch64": "batch 64 decode: lengths U[128,4096], Hq 32 / Hkv 8, D 128, P 16, fp16",
    "longtail": "batch 256 long-tail decode: lengths logN(ln 1024, 1) in [16, 32768], "
                "Hq 32 / Hkv 8, D 128, P 1, bf16",
    "cascade": "cascade: 128 x (8192 shared prefix stored once + U[64,1024] suffix), "
               "Hq 32 / Hkv 8, D 128, P 16, fp16",
    "longctx": "long-context decode: 8 x 131072 tokens, Hq 64 / Hkv 8, D 128, P 64, bf16, "
               ">=132 partitions per request",
}
# "all" (the default) times the four others first and the long-context batch,
# the largest configuration that fits one GPU, last, as the headline
ALL_ORDER = ["single", "batch64", "longtail", "cascade", "longctx"]
HEADLINE = "longctx"
KERNEL_SOURCES = ["paged_kv_decode_plan_gb300/csrc/decode.cu",
                  "paged_kv_decode_plan_gb300/csrc/ptx.cuh",
                  "paged_kv_decode_plan_gb300/csrc/kernel_common.cuh"]


# ----------------------------------------------------------------- ranks

class Ranks:
    """Rank bookkeeping; a single process when WORLD_SIZE is unset."""

    def __init__(self, backend=None):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.dist = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend or "nccl")
            self.dist = dist
        self.backend = backend or "nccl"

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def reduce_max(self, x: float) -> float:
        if self.dist is None:
            return x
        import torch
        dev = "cuda" if self.backend == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def reduce_sum(self, x: float) -> float:
        if self.dist is None:
            return x
        import torch
        dev = "cuda" if self.backend == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()


def aggregate(ranks: Ranks, per_rank_bytes: float, elapsed_s: float, steps: int):
    """Whole-job throughput: all ranks' bytes over the slowest rank's time."""
    total_bytes = ranks.reduce_sum(per_rank_bytes)
    slowest = ranks.reduce_max(elapsed_s)
    return {"value_gbs": total_bytes * steps / slowest / 1e9,
            "ms_per_step": slowest * 1e3 / steps, "slowest_s": slowest}


# ----------------------------------------------------------------- helpers

def load_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def load_tensor_peak():
    """Measured dense bf16 burst TFLOP/s (f16 has the same nominal rate)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback"


def kernel_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary, if the
    summary was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "decode_%s_ncu.txt" % workload)
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_hash():
        return None
    return float(m_bytes.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.uuid = uuid
        self.proc = None
        self.path = None
        self.window = [None, None]

    def mark(self, which: int):
        """Records the sample-file offset at the start (0) / end (1) of load."""
        time.sleep(0.15 if which else 0.0)
        self.window[which] = os.path.getsize(self.path)

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader",
                 "-lms", "100"], stdout=open(self.path, "w"),
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                f.seek(self.window[0] or 0)
                text = f.read((self.window[1] or 1 << 30) - (self.window[0] or 0))
            for line in text.splitlines():
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                if self.uuid and self.uuid not in parts[1]:
                    continue
                try:
                    rows.append((float(parts[2].split()[0]), float(parts[3].split()[0]),
                                 parts[6:10]))
                except ValueError:
                    continue
        finally:
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"],
                    "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows
                          for i, f in enumerate(flags) if f.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------- our arm

class Runner:
    """Device-resident batch plus workspaces; one `step()` = plan + run.

    Two workspaces per table alternate between steps (turns), each with its
    own queries, device page tables and outputs.  Two schedules for the
    copies of a step:

    * ``side``: pkd_plan copies each plan image on a side stream while the
      previous step still runs (end to end, the input copy joins it and the
      read-back runs on a third stream), so the copies overlap the
      neighbouring steps' kernels; the kernels of a turn are one CUDA graph
      (``--graph on``, after two eager steps) or separate launches.
    * ``graph``: the host plans into the turn's pinned staging buffer and
      replays one CUDA graph holding the plan-image copy (pkd_copy_plan: a
      kernel that reads the pinned image, its size from its header), the
      input copy and read-back (end to end) and the kernels: the fewest host
      calls per step, but the copies no longer overlap other steps' kernels.
    """

    def __init__(self, wl, device, kv_loader=0, cascade="fused", layout="nhd",
                 graph=False, cascade_split=True, copies="side"):
        import torch
        import paged_kv_decode_plan_gb300 as pkd
        self.torch = torch
        self.pkd = pkd
        self.wl = wl
        self.device = device
        # every workspace turn holds its queries and packed page tables in one
        # device buffer (one host-to-device copy per step end to end); each
        # output pair (out, lse) likewise sits in one buffer (one read-back)
        self.q_bytes = wl.q.numel() * wl.q.element_size()
        self.k = wl.k_pages.to(device)
        self.v = wl.v_pages.to(device)
        self.layout = pkd.LAYOUT_HND if layout == "hnd" else pkd.LAYOUT_NHD
        if layout == "hnd":  # same values, [pages][Hkv][P][D]
            self.k = self.k.transpose(1, 2).contiguous()
            self.v = self.v.transpose(1, 2).contiguous()
        # cascade: the shared prefix once through the shared-prefix kernel,
        # its chunk states folded into the suffix states by the cascade merge
        # ("fused"), or merged to prefix states first and combined with
        # merge_states ("shared"); or listed in every request's table
        # ("per-request")
        self.shared = wl.name == "cascade" and cascade in ("shared", "fused")
        self.fused = wl.name == "cascade" and cascade == "fused"
        if wl.name == "cascade" and not self.shared:
            self.tables = [wl.extra_tables["prefix"], wl.extra_tables["suffix"]]
        elif self.shared:
            self.tables = [wl.extra_tables["suffix"]]
        else:
            self.tables = [wl.table]
        packed_tables = [pack_table(t) for t in self.tables]
        self.in_offsets, in_bytes = _layout([self.q_bytes] + [pk.nbytes for pk in packed_tables])
        self.inbufs = [torch.empty(in_bytes, dtype=torch.uint8, device=device)
                       for _ in range(2)]
        self.qs = [buf[:self.q_bytes].view(wl.q.dtype).view(wl.q.shape) for buf in self.inbufs]
        for qd in self.qs:
            qd.copy_(wl.q)
        self.q = self.qs[0]
        self.prefix = None
        # fused cascade: the shared-prefix kernel (shared-memory / tensor bound)
        # and the suffix decode (copy bound) run side by side on disjoint SMs:
        # the prefix plan gets about 30% of the SMs in whole (head x row tile)
        # groups, the suffix plan the rest, and the suffix decode, launched as
        # a programmatic dependent, starts at once on the free SMs
        sms = torch.cuda.get_device_properties(device).multi_processor_count
        prefix_ctas = suffix_ctas = 0
        if self.fused and cascade_split:
            group = wl.num_qo_heads // wl.num_kv_heads
            base = wl.num_kv_heads * max(1, -(-wl.batch * group // 256))
            prefix_ctas = base * max(1, round(0.3 * sms / base))
            if prefix_ctas < sms:
                suffix_ctas = sms - prefix_ctas
            else:
                prefix_ctas = 0
        self.cascade_ctas = (prefix_ctas, suffix_ctas)
        if self.shared:
            pt = wl.extra_tables["prefix"]
            pages = pt.kv_indices[: pt.kv_indptr[1]].copy()
            prob = pkd.make_problem(batch=pt.batch, num_qo_heads=wl.num_qo_heads,
                                    num_kv_heads=wl.num_kv_heads, page_size=pt.page_size,
                                    dtype=wl.dtype, num_pages=wl.num_pages,
                                    num_ctas=prefix_ctas, kv_layout=self.layout)
            # the shared prefix does not change from one decode step to the
            # next (only the suffixes grow), so each workspace turn plans it
            # once and reuses the plan; the suffixes are planned every step
            self.prefix = dict(
                pages=pages, last=int(pt.kv_last_page_len[0]),
                ws=[pkd.PrefixWorkspace(prob, pages.size, device=device) for _ in range(2)],
                plans=[None, None], outs=[self._pair() for _ in range(2)])
        self.parts = []
        for n, t in enumerate(self.tables):
            prob = pkd.make_problem(batch=t.batch, num_qo_heads=wl.num_qo_heads,
                                    num_kv_heads=wl.num_kv_heads, page_size=t.page_size,
                                    dtype=wl.dtype, num_pages=wl.num_pages,
                                    min_chunks_per_request=wl.min_chunks_per_request,
                                    num_ctas=suffix_ctas if self.fused else 0,
                                    kv_loader=kv_loader, kv_layout=self.layout)
            ws = [pkd.Workspace(prob, device=device) for _ in range(2)]
            # the three page-table arrays packed together after the queries in
            # the turn's input buffer; the API gets views into it
            packed = packed_tables[n]
            n0, n1 = t.kv_indptr.size, t.kv_indices.size
            off = self.in_offsets[1 + n]
            packs = [buf[off:off + packed.nbytes].view(torch.int32) for buf in self.inbufs]
            for pk in packs:
                pk.copy_(torch.from_numpy(packed))
            devs = [(pk[:n0], pk[n0:n0 + n1], pk[n0 + n1:]) for pk in packs]
            outs = [self._pair() for _ in range(2)]
            self.parts.append(dict(table=t, ws=ws, devs=devs, packs=packs, outs=outs))
        self.finals = [self._pair() for _ in range(2)]
        # graph mode plans on the host (num_ctas must be explicit)
        for part in self.parts:
            part["problem"] = _explicit(part["ws"][0].problem, self)
        if self.prefix is not None:
            self.prefix["problem"] = _explicit(self.prefix["ws"][0].problem, self)
        self.copy_stream = torch.cuda.Stream(device)
        self.read_stream = torch.cuda.Stream(device)
        # per-turn events, created once and re-recorded every step
        self.ready_ev = [torch.cuda.Event(), torch.cuda.Event()]
        self.done_ev = [torch.cuda.Event(), torch.cuda.Event()]
        self.read_ev = [torch.cuda.Event(), torch.cuda.Event()]
        self.done = [None, None]
        self.read = [None, None]   # read-back of a turn's outputs (end to end)
        self.last_turn = 0
        self.turn = 0
        self.launches_per_step = 0
        self.use_graph = graph
        self.copies = copies if graph else "side"
        # kernels of a step besides those of _launch: the plan-image copies
        # (pkd_copy_plan) of the one-graph schedule
        self.extra_launches = (len(self.tables) + (1 if self.shared else 0)
                               if self.copies == "graph" else 0)
        self.eager_steps = 0
        self.graphs = {}
        # timing events inside a graph must be real event-record nodes
        # ("external"); without that option the timed pass runs eagerly
        try:
            self.timing_events = tuple(torch.cuda.Event(enable_timing=True, external=True)
                                       for _ in range(4))
        except TypeError:
            self.timing_events = None
        self.timings = []   # (decode_ms, prefix_ms) of timed graph steps

    def _pair(self):
        """(out, lse, buffer): one output pair as views into one device buffer."""
        torch = self.torch
        lse_bytes = self.q.shape[0] * self.q.shape[1] * 4
        offs, total = _layout([self.q_bytes, lse_bytes])
        buf = torch.empty(total, dtype=torch.uint8, device=self.device)
        out = buf[:self.q_bytes].view(self.q.dtype).view(self.q.shape)
        lse = buf[offs[1]:offs[1] + lse_bytes].view(torch.float32).view(self.q.shape[:2])
        return out, lse, buf

    def host_inputs(self):
        """A pinned copy of a turn's input buffer (queries, packed tables)."""
        return self.inbufs[0].cpu().pin_memory()

    def step(self, events=None, inputs=None, outputs=None):
        """One step on workspace turn i.  ``inputs`` (a pinned copy of the input
        buffer: queries and packed page tables) is copied in before the
        kernels; ``outputs`` (a pinned buffer the size of a result pair's)
        receives the step's (out, lse).  Graph mode (after two eager steps):
        the host plans into the turn's pinned staging buffer(s) and replays one
        graph holding the plan-image copies, the input copy (end to end), the
        kernels and the read-back (end to end)."""
        timed_in_graph = events is None or self.timing_events is not None
        graph = self.use_graph and self.eager_steps >= 2 and timed_in_graph
        if graph and self.copies == "graph":
            self._step_graph(events, inputs, outputs)
        else:
            self._step_side(events, inputs, outputs, graph)
            if not graph:
                self.eager_steps += 1

    def _plan_graph(self, i):
        """Host planning of turn i into its pinned staging buffer(s); the
        turn's graph copies them to the device."""
        for part in self.parts:
            t = part["table"]
            part["plan"], _ = self.pkd.plan_host(part["problem"], t.kv_indptr,
                                                 t.kv_last_page_len,
                                                 image=part["ws"][i].staging[0])
        if self.prefix is not None:
            pre = self.prefix
            if pre["plans"][i] is None:
                pre["plans"][i], _ = self.pkd.plan_shared_prefix_host(
                    pre["problem"], pre["pages"], pre["last"], image=pre["ws"][i].staging)
            pre["plan"] = pre["plans"][i]

    def _step_graph(self, events, inputs, outputs):
        torch = self.torch
        i = self.turn
        self.turn ^= 1
        self.last_turn = i
        # the turn's previous graph must have read its staging buffers
        if self.done[i] is not None:
            self.done[i].synchronize()
        self._plan_graph(i)
        key = (i, events is not None, inputs is not None)
        if key not in self.graphs:
            self._capture(i, events is not None, inputs, outputs)
        self.graphs[key].replay()
        done = self.done_ev[i]
        done.record(torch.cuda.current_stream())
        self.done[i] = done
        if events is not None:
            torch.cuda.synchronize()
            e = self.timing_events
            self.timings.append((e[0].elapsed_time(e[1]),
                                 e[2].elapsed_time(e[3]) if self.prefix else None))

    def _capture(self, i, timed, inputs, outputs):
        """The graph of turn i: plan-image copies from the turn's pinned
        staging (pkd_copy_plan, which reads each image's size when it runs,
        so any later plan of the capacity fits), [input copy], the kernels,
        [read-back]."""
        torch = self.torch
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            # the input copy (copy engine) first, then only kernels until the
            # read-back: one engine hand-off each way
            if inputs is not None:
                self.inbufs[i].copy_(inputs, non_blocking=True)
            # pkd_copy_plan: a kernel reads each pinned image (its current
            # size from its header) into the workspace
            for part in self.parts:
                ws = part["ws"][i]
                self.pkd.copy_plan(ws.staging[0], ws.int_ws)
            if self.prefix is not None:
                ws = self.prefix["ws"][i]
                self.pkd.copy_plan(ws.staging, ws.int_ws)
            self._launch(i, self.timing_events if timed else None)
            if outputs is not None:
                outputs.copy_(self.result_turn(i)[2], non_blocking=True)
        torch.cuda.synchronize()
        self.graphs[(i, timed, inputs is not None)] = g

    def _capture_kernels(self, i, timed):
        """Turn i's kernel launches as one graph (valid for every later plan
        of the workspace's capacity)."""
        torch = self.torch
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self._launch(i, self.timing_events if timed else None)
        torch.cuda.synchronize()
        self.graphs[(i, timed, "kernels")] = g

    def _step_side(self, events=None, inputs=None, outputs=None, graph=False):
        """Copies beside the kernels: plan (pkd_plan copies the image on the
        copy stream), input copy on the copy stream, the kernels on the main
        stream (one kernel-only graph per turn with ``graph``), read-back on
        its own stream."""
        torch = self.torch
        main = torch.cuda.current_stream()
        i = self.turn
        self.turn ^= 1
        self.last_turn = i
        if self.done[i] is not None:
            self.copy_stream.wait_event(self.done[i])
        if inputs is not None:
            # plain stream switches: the stream context manager costs several
            # microseconds of Python per use on this host
            torch.cuda.set_stream(self.copy_stream)
            self.inbufs[i].copy_(inputs, non_blocking=True)
            torch.cuda.set_stream(main)
        for part in self.parts:
            t = part["table"]
            part["plan"] = part["ws"][i].plan(t.kv_indptr, t.kv_last_page_len, None,
                                              stream=self.copy_stream)
        if self.prefix is not None:
            pre = self.prefix
            if pre["plans"][i] is None:
                pre["plans"][i] = pre["ws"][i].plan(pre["pages"], pre["last"],
                                                    stream=self.copy_stream)
            pre["plan"] = pre["plans"][i]
        ready = self.ready_ev[i]
        ready.record(self.copy_stream)
        main.wait_event(ready)
        if self.read[i] is not None:   # this turn's previous outputs were read back
            main.wait_event(self.read[i])
        if graph:
            key = (i, events is not None, "kernels")
            if key not in self.graphs:
                self._capture_kernels(i, events is not None)
            self.graphs[key].replay()
            if events is not None:
                torch.cuda.synchronize()
                e = self.timing_events
                self.timings.append((e[0].elapsed_time(e[1]),
                                     e[2].elapsed_time(e[3]) if self.prefix else None))
        else:
            self._launch(i, events)
        done = self.done_ev[i]
        done.record(main)
        self.done[i] = done
        if outputs is not None:
            res = self.result()
            self.read_stream.wait_event(done)
            torch.cuda.set_stream(self.read_stream)
            outputs.copy_(res[2], non_blocking=True)
            torch.cuda.set_stream(main)
            rd = self.read_ev[i]
            rd.record(self.read_stream)
            self.read[i] = rd

    def _launch(self, i, events=None):
        """The kernel launches of one step on the current stream."""
        torch = self.torch
        main = torch.cuda.current_stream()
        launches = 0
        if self.fused:
            pre, part = self.prefix, self.parts[0]
            ws, plan, final = part["ws"][i], part["plan"], self.finals[i]
            if events is None:
                # the single call a user makes (its decode overlaps the prefix
                # kernel's last CTAs); the timed pass below launches the same
                # kernels one by one with events between them
                self.pkd.run_cascade(plan, pre["plan"], self.qs[i], self.k, self.v,
                                     *part["devs"][i], ws, pre["ws"][i], self.wl.sm_scale,
                                     out=final[0], lse=final[1])
                self.launches_per_step = 3
                return
            if events is not None:
                events[2].record(main)
            pre["ws"][i].run_states(pre["plan"], self.qs[i], self.k, self.v,
                                    self.wl.sm_scale)
            if events is not None:
                events[3].record(main)
                events[0].record(main)
            ws.run(plan, self.qs[i], self.k, self.v, *part["devs"][i], self.wl.sm_scale,
                   phase="decode_states")
            if events is not None:
                events[1].record(main)
            self.pkd.run_cascade_merge(plan, pre["plan"], ws, pre["ws"][i], final[0],
                                       final[1])
            self.launches_per_step = 3
            return
        if self.prefix is not None:
            pre = self.prefix
            if events is not None:
                events[2].record(main)
            pre["ws"][i].run(pre["plan"], self.qs[i], self.k, self.v, self.wl.sm_scale,
                             out=pre["outs"][i][0], lse=pre["outs"][i][1])
            if events is not None:
                events[3].record(main)
            launches += 2
        for n, part in enumerate(self.parts):
            ws, plan = part["ws"][i], part["plan"]
            if events is not None and n == 0:
                events[0].record(main)
            ws.run(plan, self.qs[i], self.k, self.v, *part["devs"][i], self.wl.sm_scale,
                   out=part["outs"][i][0], lse=part["outs"][i][1], phase="decode")
            if events is not None and n == 0:
                events[1].record(main)
            ws.run(plan, self.qs[i], self.k, self.v, *part["devs"][i], self.wl.sm_scale,
                   out=part["outs"][i][0], lse=part["outs"][i][1], phase="merge")
            launches += 1 + (plan.num_split_requests > 0 or self.use_graph)
        if len(self.parts) == 2 or self.prefix is not None:
            a = (self.parts[0] if self.prefix is None else self.prefix)["outs"][i]
            b = self.parts[-1]["outs"][i]
            self.pkd.merge_states(a[0], a[1], b[0], b[1],
                                  v_out=self.finals[i][0], s_out=self.finals[i][1])
            launches += 1
        self.launches_per_step = launches

    def read_timings(self, events):
        """(decode ms list, prefix ms list or None) of the timed pass."""
        if self.timings:
            dec = [t[0] for t in self.timings]
            pre = [t[1] for t in self.timings] if self.prefix is not None else None
            return dec, pre
        dec = [e[0].elapsed_time(e[1]) for e in events]
        pre = [e[2].elapsed_time(e[3]) for e in events] if self.prefix is not None else None
        return dec, pre

    def result(self):
        """(out, lse, buffer) of the last step."""
        return self.result_turn(self.last_turn)

    def result_turn(self, i):
        """(out, lse, buffer) of workspace turn i."""
        if len(self.parts) == 2 or self.prefix is not None:
            return self.finals[i]
        return self.parts[0]["outs"][i]

    def status(self):
        words = [self.pkd.check_status(ws.int_ws) for p in self.parts for ws in p["ws"]]
        if self.prefix is not None:
            words += [self.pkd.check_status(ws.int_ws) for ws in self.prefix["ws"]]
        return max(words)

    def kv_bytes(self):
        """Algorithmic KV bytes per step (a shared prefix counted once)."""
        return workload_kv_bytes(self.wl)

    def total_bytes(self):
        """All algorithmic bytes a step moves: KV (shared prefix once), the
        queries read and outputs / lse written by every run, page indices, and
        the fp32 partial states written and read back by the merges."""
        wl = self.wl
        elem = wl.k_pages.element_size()
        rows = wl.batch * wl.num_qo_heads
        slot = 4 * (wl.num_qo_heads * wl.head_dim + (wl.num_qo_heads + 3) // 4 * 4)
        state = rows * (wl.head_dim * elem + 4)          # out + lse of one run
        total = self.kv_bytes()
        if self.fused:
            pre, part = self.prefix, self.parts[0]
            prefix_states = wl.batch * pre["plan"].chunks * slot
            total += 4 * int(pre["pages"].size) + 4 * int(part["table"].kv_indices.size)
            total += 2 * rows * wl.head_dim * elem          # q read by both kernels
            # suffix decode: every request's state fp32 (split requests' partial
            # slots, one slot per unsplit request), written and read by the merge
            plan = part["plan"]
            suffix_slots = plan.num_partials + wl.batch - plan.num_split_requests
            total += 2 * suffix_slots * slot
            total += 2 * prefix_states                       # prefix states out and in
            total += state                                   # merge: final out / lse
            return total
        for part in self.parts:
            total += 4 * int(part["table"].kv_indices.size)
            total += rows * wl.head_dim * elem + state + 2 * part["plan"].num_partials * slot
        if self.prefix is not None:
            pre = self.prefix
            total += 4 * int(pre["pages"].size)
            total += rows * wl.head_dim * elem + state
            total += 2 * wl.batch * pre["plan"].chunks * slot
        if len(self.parts) == 2 or self.prefix is not None:
            total += 3 * state                             # merge_states: two in, one out
        return total

    def decode_kv_bytes(self):
        """KV bytes the timed decode launch reads (first table)."""
        wl = self.wl
        per_token = 2 * wl.num_kv_heads * wl.head_dim * wl.k_pages.element_size()
        return int(self.tables[0].lengths().sum()) * per_token


def _layout(sizes, align=256):
    """(offsets, total) of byte ranges packed one after another, each start
    aligned to ``align`` bytes."""
    offs, off = [], 0
    for n in sizes:
        offs.append(off)
        off += (n + align - 1) // align * align
    return offs, off


def workload_kv_bytes(wl):
    """Algorithmic KV bytes of one pass over a workload (a shared prefix
    counted once)."""
    per_token = 2 * wl.num_kv_heads * wl.head_dim * wl.k_pages.element_size()
    if wl.name == "cascade":
        prefix = wl.extra_tables["prefix"]
        prefix_tokens = int(prefix.lengths()[0]) if prefix.batch else 0
        return (prefix_tokens + int(wl.extra_tables["suffix"].lengths().sum())) * per_token
    return int(wl.table.lengths().sum()) * per_token


def workload_config(wl):
    """The JSON line's config: the workload, its sizes and the L2 note."""
    kv = workload_kv_bytes(wl)
    return {"workload": DESCRIPTIONS[wl.name], "name": wl.name,
            "batch": wl.batch, "num_qo_heads": wl.num_qo_heads,
            "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
            "page_size": wl.page_size, "kv_bytes_per_step": kv,
            "l2": ("inputs larger than L2 (KV %.0f MB vs 129 MB), no flush" % (kv / 1e6))
            if kv > 2 * L2_BYTES else
            ("KV (%.1f MB) fits in L2: L2 flushed before every timed step; "
             "e2e and warm_us_per_batch warm" % (kv / 1e6)),
            "parallelism": "replicas (weak scaling, no collective)"}


def pack_table(t):
    """indptr, indices and last_page_len of a page table in one int32 array."""
    return np.concatenate([t.kv_indptr, t.kv_indices, t.kv_last_page_len]).astype(np.int32)


def make_workload(args, name=None):
    from paged_kv_decode_plan_gb300 import workloads
    name = name or (HEADLINE if args.workload == "all" else args.workload)
    if args.batch is None:
        return workloads.WORKLOADS[name]()
    if name not in ("longctx", "cascade"):
        raise SystemExit("--batch applies to the longctx and cascade workloads")
    return workloads.WORKLOADS[name](batch=args.batch)


def run_ours(args, ranks):
    """Every workload of ``args.workload`` ("all": the five), each timed
    with the same steps and warm-up; returns rank 0's JSON line.  With
    "all", the long-context batch is the headline and the other four go
    into ``per_config``."""
    import torch
    torch.cuda.set_device(ranks.local)
    device = torch.device("cuda", ranks.local)
    if args.workload == "append":
        ap = measure_append(args, device, cpu=ranks.rank == 0)
        return {"metric": "page append: K/V bytes read + written per second", "value":
                ap["bulk"]["value"], "unit": "GB/s", "n_gpus": ranks.world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(ap["bulk"]["us"] / 1e3, 5),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f16", "data": "synthetic (seeded N(0,1))",
                "config": {"workload": APPEND_DESCRIPTION, "name": "append"},
                **{k_: ap[k_] for k_ in ("bulk", "decode_step", "roofline", "gpu_launches")},
                **({"cpu_baseline": ap["cpu_baseline"]} if "cpu_baseline" in ap else {})}
    names = ALL_ORDER if args.workload == "all" else [args.workload]
    lines = {}
    for name in names:
        wl = make_workload(args, name)
        lines[name] = measure(args, ranks, device, wl,
                              cpu=(name == names[-1] or len(names) == 1))
        del wl
        torch.cuda.empty_cache()
    line = lines[names[-1]]
    if len(names) > 1:
        line["per_config"] = {n: config_summary(lines[n]) for n in names[:-1]}
        line["config"]["per_config"] = ("the other four workloads, each timed in this "
                                        "run with the same steps and warm-up")
        # the page append step (new tokens' K/V into their pages), beside the
        # decode path it feeds
        line["page_append"] = measure_append(args, device, cpu=ranks.rank == 0)
    return line


APPEND_DESCRIPTION = ("page append on the batch-64 page pool (Hkv 8, D 128, P 16, fp16): "
                      "every token of the 64 requests rewritten (bulk), and one new "
                      "token per request (a decode step's append)")


def measure_append(args, device, cpu=True):
    """The page-append step on the batch-64 page pool, HBM-bound (a copy):
    a bulk append that rewrites every token of every request (new K/V rows
    read, page slots written) timed over the run's steps, and a decode
    step's append (one token per request, at its last position), each launch
    between two events inside a replayed graph.  Sampled rows are checked against the new rows; the
    oracle (oracle/append_ref.py) is timed on a compact pool of the first
    requests."""
    import torch
    import paged_kv_decode_plan_gb300 as pkd
    from paged_kv_decode_plan_gb300 import workloads
    wl = workloads.batch64()
    t = wl.table
    hkv, d = wl.num_kv_heads, wl.head_dim
    row_bytes = hkv * d * 2
    lengths = t.lengths()
    k = wl.k_pages.to(device)
    v = wl.v_pages.to(device)
    tab = [torch.from_numpy(a).to(device) for a in (t.kv_indptr, t.kv_indices,
                                                    t.kv_last_page_len)]
    prob = pkd.make_problem(batch=t.batch, num_qo_heads=wl.num_qo_heads, num_kv_heads=hkv,
                            page_size=t.page_size, dtype=wl.dtype, num_pages=wl.num_pages)
    bi = np.repeat(np.arange(t.batch, dtype=np.int32), lengths)
    pos = np.concatenate([np.arange(n, dtype=np.int32) for n in lengths])
    n = int(bi.size)
    gen = torch.Generator(device=device).manual_seed(4242)
    kn = torch.randn(n, hkv, d, generator=gen, device=device).to(k.dtype)
    vn = torch.randn(n, hkv, d, generator=gen, device=device).to(k.dtype)
    bi_d, pos_d = torch.from_numpy(bi).to(device), torch.from_numpy(pos).to(device)
    status = torch.zeros(1, dtype=torch.int32, device=device)

    def bulk():
        pkd.append_kv(prob, kn, vn, bi_d, pos_d, k, v, *tab, status=status)

    for _ in range(args.warmup):
        bulk()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(args.steps):
        bulk()
    end.record()
    torch.cuda.synchronize()
    bulk_s = start.elapsed_time(end) / 1e3 / args.steps
    if int(status.item()) != 0:
        raise RuntimeError("append status word %d" % int(status.item()))
    # sampled rows: page kv_indices[indptr[b] + pos // P], slot pos % P
    rng = np.random.default_rng(7)
    for i in rng.choice(n, size=32, replace=False).tolist():
        b, p_ = int(bi[i]), int(pos[i])
        page = int(t.kv_indices[int(t.kv_indptr[b]) + p_ // t.page_size])
        slot = p_ % t.page_size
        if not (torch.equal(k[page, slot], kn[i]) and torch.equal(v[page, slot], vn[i])):
            raise RuntimeError("appended row differs from the new row")
    moved = 2 * n * row_bytes * 2       # K and V rows, read once and written once
    peak, peak_kind = load_peak()
    achieved = moved / bulk_s / 1e9

    # a decode step's append: one token per request, at its last position
    live = np.nonzero(lengths > 0)[0].astype(np.int32)
    bi1 = torch.from_numpy(live).to(device)
    pos1 = torch.from_numpy((lengths[live] - 1).astype(np.int32)).to(device)
    kn1, vn1 = kn[: live.size].contiguous(), vn[: live.size].contiguous()
    # replayed as a graph with its events inside (event-record nodes:
    # "external" events), so that the interval holds the device's work and
    # not the host's submission of an eager launch
    try:
        e0, e1 = (torch.cuda.Event(enable_timing=True, external=True) for _ in range(2))
        graph = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=torch.cuda.Stream(device)):
            e0.record()
            pkd.append_kv(prob, kn1, vn1, bi1, pos1, k, v, *tab, status=status)
            e1.record()
        step_timing = "events inside a replayed graph"
    except TypeError:
        e0, e1 = (torch.cuda.Event(enable_timing=True) for _ in range(2))
        graph = None
        step_timing = "events around an eager launch (host submission included)"
    step_ts = []
    for it in range(args.warmup + args.steps):
        if graph is not None:
            graph.replay()
        else:
            e0.record()
            pkd.append_kv(prob, kn1, vn1, bi1, pos1, k, v, *tab, status=status)
            e1.record()
        torch.cuda.synchronize()
        if it >= args.warmup:
            step_ts.append(e0.elapsed_time(e1) * 1e3)
    if int(status.item()) != 0:
        raise RuntimeError("append status word %d" % int(status.item()))
    out = {"workload": APPEND_DESCRIPTION,
           "bulk": {"tokens": n, "us": round(bulk_s * 1e6, 2),
                    "bytes_per_launch": moved, "value": round(achieved, 1), "unit": "GB/s"},
           "decode_step": {"tokens": int(live.size),
                           "us_median": round(statistics.median(step_ts), 2),
                           "timing": step_timing},
           "roofline": {"bound": "hbm", "kernel": "append_kernel",
                        "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind,
                        "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": None,
                        "algorithmic_bytes_per_launch": moved},
           # launches inside the two timed loops
           "gpu_launches": 2 * args.steps}
    if cpu:
        out["cpu_baseline"] = append_cpu_baseline(wl, lengths, row_bytes)
    del k, v, kn, vn
    return out


def append_cpu_baseline(wl, lengths, row_bytes, budget_s: float = 3.0):
    """The append oracle on a compact pool of the first requests: every
    token of each request rewritten, as the bulk measurement does."""
    import oracle.append_ref as append_ref
    from paged_kv_decode_plan_gb300 import workloads
    t = wl.table
    k_all, v_all = workloads.as_codes(wl.k_pages), workloads.as_codes(wl.v_pages)
    rng = np.random.default_rng(5)
    tokens = 0
    elapsed = 0.0
    reqs = 0
    for b in range(t.batch):
        if elapsed >= budget_s:
            break
        pages = t.kv_indices[t.kv_indptr[b]: t.kv_indptr[b + 1]]
        n = int(lengths[b])
        if n == 0:
            continue
        k_pool, v_pool = k_all[pages], v_all[pages]
        kn = rng.integers(0, 1 << 15, size=(n,) + k_pool.shape[2:], dtype=np.uint16)
        vn = rng.integers(0, 1 << 15, size=(n,) + v_pool.shape[2:], dtype=np.uint16)
        indptr = np.array([0, pages.size], np.int32)
        indices = np.arange(pages.size, dtype=np.int32)
        last = t.kv_last_page_len[b: b + 1]
        t0 = time.perf_counter()
        append_ref.append_kv(k_pool, v_pool, kn, vn, np.zeros(n, np.int32),
                             np.arange(n, dtype=np.int32), indptr, indices, last)
        elapsed += time.perf_counter() - t0
        tokens += n
        reqs += 1
    moved = 2 * tokens * row_bytes * 2
    return {"value": round(moved / elapsed / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle", "seconds": round(elapsed, 2),
            "sample": "%d whole requests of the batch-64 pool (%d tokens), each in a "
                      "compact pool of its own pages, plain Python loop" % (reqs, tokens)}


def config_summary(line):
    """The figures of one workload's line that per_config reports."""
    keys = ("us_per_batch", "value", "unit", "ms_per_step", "steps", "warmup",
            "decode_us", "prefix_us", "host_enqueue_us_per_step", "host_cpu_us_per_step",
            "total_gbs",
            "plan_host_us", "num_units", "num_split_requests", "launch", "copies",
            "warm_us_per_batch",
            "gpu_launches", "dtype", "clocks")
    out = {"workload": line["config"]["workload"],
           "kv_bytes_per_step": line["config"]["kv_bytes_per_step"],
           "l2": line["config"]["l2"]}
    out.update({k: line[k] for k in keys if k in line})
    peak_key = [k for k in line if k.startswith("hbm_frac_of_")][0]
    out["step_" + peak_key] = line[peak_key]
    r = line["roofline"]
    out["roofline"] = {"kernel": r["kernel"], "achieved": r["achieved"], "peak": r["peak"],
                       "frac": r["frac"], "traffic": r["traffic"]}
    out["e2e"] = {"us_per_batch": line["e2e"]["us_per_batch"],
                  "value": line["e2e"]["value"], "unit": line["e2e"]["unit"]}
    if line.get("cascade"):
        out["cascade"] = line["cascade"]
        out["cascade_ctas"] = line["cascade_ctas"]
    if line.get("prefix_roofline"):
        out["prefix_roofline"] = line["prefix_roofline"]
    return out


def prefix_roofline(runner, prefix_ms):
    """Tensor roofline of the shared-prefix kernel: 4 * B * Hq * L * D flops
    (Q K^T and P V) per launch over its mean launch time."""
    wl = runner.wl
    pt = wl.extra_tables["prefix"]
    n_pages = int(pt.kv_indptr[1])
    length = (n_pages - 1) * pt.page_size + int(pt.kv_last_page_len[0])
    flops = 4.0 * pt.batch * wl.num_qo_heads * length * wl.head_dim
    achieved = flops / (prefix_ms * 1e-3) / 1e12
    peak, kind = load_tensor_peak()
    ctas, _ = runner.cascade_ctas
    sms = runner.torch.cuda.get_device_properties(runner.device).multi_processor_count
    out = {"bound": "tensor", "kernel": "shared_prefix_kernel",
           "achieved": round(achieved, 1), "peak": peak,
           "peak_kind": kind + " bf16 burst (f16 has the same nominal rate)",
           "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
           "algorithmic_flops_per_launch": flops}
    if ctas:
        # the kernel runs on `ctas` SMs beside the suffix decode
        out["ctas"] = ctas
        out["frac_of_its_sms"] = round(achieved / (peak * ctas / sms), 4)
    return out


def measure(args, ranks, device, wl, cpu):
    """One workload: warm-up, pass 1 (whole steps), pass 2 (events around
    each decode launch), end to end through the API; its JSON line."""
    import torch
    copies = args.copies
    if copies == "auto":
        # a step that moves little KV is bound by launch and copy latency and
        # by host calls: one graph per step; a bandwidth-bound step hides its
        # copies behind the neighbouring steps' kernels
        copies = "graph" if workload_kv_bytes(wl) <= GRAPH_COPIES_MAX_KV else "side"
    runner = Runner(wl, device, kv_loader={"auto": 0, "tma": 1, "bulk": 2}[args.loader],
                    cascade=args.cascade, layout=args.layout, graph=args.graph == "on",
                    cascade_split=args.cascade_split == "on", copies=copies)
    stream = torch.cuda.current_stream()

    # host plan time (median of 20)
    part = runner.parts[0]
    problem = _explicit(part["ws"][0].problem, runner)
    plan_times = []
    for _ in range(20):
        t0 = time.perf_counter()
        runner.pkd.plan_host(problem, part["table"].kv_indptr,
                             part["table"].kv_last_page_len)
        plan_times.append(time.perf_counter() - t0)

    # first steps: eager, then (graph mode) capture and replay; the result
    # and the device status word are checked before anything is timed
    for _ in range(3):
        runner.step()
    if runner.use_graph:
        for _ in range(3):
            runner.step()
    torch.cuda.synchronize()
    status = runner.status()
    if status:
        raise RuntimeError("device status word %d after the first steps" % status)
    out, lse, _ = runner.result()
    if not bool(torch.isfinite(out).all()) or bool(torch.isnan(lse).any()):
        raise RuntimeError("non-finite output after the first steps")

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(device).uuid)
    except Exception:  # noqa: BLE001 - older torch
        uuid = None
    k = args.steps
    events = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4))
              for _ in range(k)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # a batch whose KV fits in L2 is timed cold: a write of twice L2's size
    # before every timed step, the steps timed one by one (the warm figure is
    # reported beside it); larger batches stream more than L2 every step
    small = runner.kv_bytes() <= 2 * L2_BYTES
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device) if small else None
    warm_s = None
    with ClockSampler(uuid) as clocks:
        # the W warm-up steps run right before the timed region (the clock
        # sampler's start-up pause would otherwise sit between them)
        clocks.mark(0)
        for _ in range(args.warmup):
            runner.step()
        # pass 1: the whole step, start and end events only
        ranks.barrier()
        torch.cuda.synchronize()
        if small:
            step_ev = [(torch.cuda.Event(enable_timing=True),
                        torch.cuda.Event(enable_timing=True)) for _ in range(k)]
            host_s = host_cpu_s = 0.0
            for i in range(k):
                flush_buf.fill_(i & 0xFF)
                step_ev[i][0].record(stream)
                h0, c0 = time.perf_counter(), time.thread_time()
                runner.step()
                host_s += time.perf_counter() - h0
                host_cpu_s += time.thread_time() - c0
                step_ev[i][1].record(stream)
            torch.cuda.synchronize()
            elapsed = sum(a.elapsed_time(b) for a, b in step_ev) / 1e3
            start.record(stream)
            for _ in range(k):
                runner.step()
            end.record(stream)
            torch.cuda.synchronize()
            warm_s = start.elapsed_time(end) / 1e3
        else:
            start.record(stream)
            h0, c0 = time.perf_counter(), time.thread_time()
            for _ in range(k):
                runner.step()
            host_s = time.perf_counter() - h0
            host_cpu_s = time.thread_time() - c0
            end.record(stream)
            torch.cuda.synchronize()
            elapsed = start.elapsed_time(end) / 1e3
        ranks.barrier()
        # pass 2: the same steps with events around every decode launch
        ranks.barrier()
        torch.cuda.synchronize()
        for i in range(k):
            if small:
                flush_buf.fill_(i & 0xFF)
            runner.step(events[i])
        torch.cuda.synchronize()
        ranks.barrier()
        # end to end through the public API with host buffers
        e2e = run_e2e(args, runner, device, ranks, elapsed / k)
        clocks.mark(1)
    decode_ms, prefix_ms = runner.read_timings(events)
    agg = aggregate(ranks, runner.kv_bytes(), elapsed, k)
    decode_mean_ms = ranks.reduce_max(statistics.fmean(decode_ms))

    peak, peak_kind = load_peak()
    achieved = runner.decode_kv_bytes() / (decode_mean_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(agg["value_gbs"], 2), "unit": "GB/s",
        "n_gpus": ranks.world, "steps": k, "warmup": args.warmup,
        "ms_per_step": round(agg["ms_per_step"], 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "accumulate": "f32",
        "data": "synthetic (seeded N(0,1), shapes of the workload)",
        "config": workload_config(wl),
        "us_per_batch": round(agg["ms_per_step"] * 1e3, 2),
        "total_bytes_per_step": runner.total_bytes(),
        "total_gbs": round(runner.total_bytes() * ranks.world / (agg["ms_per_step"] * 1e-3)
                           / 1e9, 2),
        "hbm_frac_of_%s" % peak_kind: round(agg["value_gbs"] / ranks.world / peak, 4),
        "decode_us": round(decode_mean_ms * 1e3, 2),
        # host time to enqueue one step in pass 1 (plan + copies + launches);
        # above us_per_batch the step is host-bound
        "host_enqueue_us_per_step": round(host_s / k * 1e6, 2),
        # CPU time of the enqueuing thread in the same loop (waits for the
        # device spin, so they count too); far below the wall time above,
        # the thread was descheduled
        "host_cpu_us_per_step": round(host_cpu_s / k * 1e6, 2),
        "plan_host_us": round(statistics.median(plan_times) * 1e6, 1),
        "num_units": runner.parts[0]["plan"].num_units,
        "num_split_requests": runner.parts[0]["plan"].num_split_requests,
        "kv_loader": args.loader,
        "kv_layout": args.layout,
        "cascade": (args.cascade if wl.name == "cascade" else None),
        "cascade_ctas": (list(runner.cascade_ctas) if runner.fused else None),
        "prefix_us": (round(statistics.fmean(prefix_ms) * 1e3, 2)
                      if prefix_ms else None),
        "prefix_roofline": (prefix_roofline(runner, statistics.fmean(prefix_ms))
                            if prefix_ms else None),
        "launch": ("graph" if runner.use_graph else "eager"),
        "copies": runner.copies,
        "timing": "W warm-up steps right before pass 1; pass 1 (value, ms_per_step): K "
                  + ("steps, each after an L2 flush (a %d MB write) and timed alone "
                     "between two events (warm_us_per_batch: the same K steps back "
                     "to back without flushes)" % (2 * L2_BYTES >> 20) if small else
                     "steps between two events")
                  + "; pass 2 (decode_us, roofline): the same K steps with events "
                  "around each decode launch" +
                  (" (inside the replayed graph, one step at a time)"
                   if runner.use_graph else ""),
        "warm_us_per_batch": (round(warm_s / k * 1e6, 2) if warm_s is not None else None),
        "roofline": {"bound": "hbm", "kernel": "decode_kernel",
                     "achieved": round(achieved, 2), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     # the committed captures ran the default launch (NHD pages,
                     # auto loader, full workload)
                     "traffic": (profiled_traffic(wl.name)
                                 if args.layout == "nhd" and args.loader == "auto"
                                 and args.batch is None else None),
                     "algorithmic_bytes_per_launch": runner.decode_kv_bytes()},
        "e2e": e2e,
        "gpu_launches": (runner.launches_per_step + runner.extra_launches) * k,
        "clocks": clocks.summary(),
    }
    if cpu and ranks.rank == 0 and ranks.world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_budget_s)
    del runner
    return line


def _explicit(problem, runner):
    import paged_kv_decode_plan_gb300 as pkd
    p = pkd.Problem.from_buffer_copy(problem)
    if p.num_ctas <= 0:
        import torch
        p.num_ctas = torch.cuda.get_device_properties(runner.device).multi_processor_count
    return p


def run_e2e(args, runner, device, ranks, step_s):
    """Same metric through the public API: every step copies its inputs
    (queries and page table) host-to-device from pinned memory, plans, runs,
    and copies out and lse device-to-host into one of two pinned buffers.
    Graph mode: the copies are nodes of the step's graph, before and after
    its kernels.  Eager mode: they run on their own streams and overlap the
    neighbouring steps' kernels (each turn's device buffers are reused only
    after their read-back completed).  The timed region ends with a
    synchronise after the last read-back."""
    import torch
    wl = runner.wl
    in_h = runner.host_inputs()
    res_bytes = runner.result()[2].numel()
    outs_h = [torch.empty(res_bytes, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
    h2d = in_h.numel()
    d2h = res_bytes
    if args.e2e_steps > 0:
        steps = args.e2e_steps
    else:
        # about 0.2 s of steps (at least K, at most 2000): host jitter on a
        # loop of a few hundred microseconds would otherwise dominate
        steps = int(min(2000, max(args.steps, 0.2 / max(step_s, 1e-6))))

    def one():
        # each workspace turn reads back into its own pinned buffer
        runner.step(inputs=in_h, outputs=outs_h[runner.turn])

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    image_bytes = sum(int(p["plan"].int_ws_bytes_used) for p in runner.parts)
    if runner.prefix is not None and runner.use_graph and runner.copies == "graph":
        # the step's graph copies the (unchanged) prefix image too
        image_bytes += int(runner.prefix["plan"].int_ws_bytes_used)

    ranks.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    # the last read-back holds the last step's device result
    if not torch.equal(outs_h[runner.last_turn], runner.result()[2].cpu()):
        raise RuntimeError("read-back differs from the device result")
    agg = aggregate(ranks, runner.kv_bytes(), elapsed, steps)
    return {"value": round(agg["value_gbs"], 2), "unit": "GB/s",
            "us_per_batch": round(agg["ms_per_step"] * 1e3, 2), "steps": steps,
            "h2d_bytes_per_step": h2d + image_bytes, "d2h_bytes_per_step": d2h}


# ----------------------------------------------------------------- oracle arm

def _oracle_rows_for(wl, first_req, n_req):
    hq = wl.num_qo_heads
    return np.arange(first_req * hq, (first_req + n_req) * hq, dtype=np.int64)


def cpu_baseline(wl, budget_s: float, kind="oracle"):
    """Times the fp64 oracle on whole requests of the workload (in batch order,
    wrapping around) until about budget_s of wall time has passed."""
    import oracle
    from paged_kv_decode_plan_gb300 import workloads
    codes = (workloads.as_codes(wl.q), workloads.as_codes(wl.k_pages),
             workloads.as_codes(wl.v_pages))
    t = wl.table
    lengths = t.lengths()
    per_token = 2 * wl.num_kv_heads * wl.head_dim * wl.k_pages.element_size()
    done_bytes = 0
    done_req = 0
    elapsed = 0.0
    b = 0
    while elapsed < budget_s and done_req < 64 * wl.batch:
        rows = _oracle_rows_for(wl, b, 1)
        t0 = time.perf_counter()
        oracle.decode(*codes, t.kv_indptr, t.kv_indices, t.kv_last_page_len,
                      dtype=wl.dtype, sm_scale=wl.sm_scale, rows=rows)
        elapsed += time.perf_counter() - t0
        done_bytes += int(lengths[b]) * per_token
        done_req += 1
        b = (b + 1) % wl.batch
    gbs = done_bytes / elapsed / 1e9 if elapsed > 0 else 0.0
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": kind, "seconds": round(elapsed, 2),
            "us_per_batch_equiv": round(elapsed / max(done_bytes, 1) *
                                        sum(int(x) for x in lengths) * per_token * 1e6, 1),
            "sample": "%d whole requests (all %d query heads each) of the %s workload, "
                      "fp64 page-table walk" % (done_req, wl.num_qo_heads, wl.name)}


def run_reference(args, ranks):
    """The oracle as it stands, on the host cores, same metric and config."""
    import oracle
    from paged_kv_decode_plan_gb300 import workloads
    if args.workload == "append":
        raise SystemExit("--impl reference times the decode oracle; the append "
                         "oracle's timing is the cpu_baseline of --workload append")
    oracle.build()
    wl = make_workload(args)
    codes = (workloads.as_codes(wl.q), workloads.as_codes(wl.k_pages),
             workloads.as_codes(wl.v_pages))
    t = wl.table
    lengths = t.lengths()
    per_token = 2 * wl.num_kv_heads * wl.head_dim * wl.k_pages.element_size()
    hq = wl.num_qo_heads
    # calibrate: rows per step so that warm-up + steps take about budget_s
    t0 = time.perf_counter()
    oracle.decode(*codes, t.kv_indptr, t.kv_indices, t.kv_last_page_len,
                  dtype=wl.dtype, sm_scale=wl.sm_scale, rows=np.arange(hq))
    per_req = max(time.perf_counter() - t0, 1e-4)
    per_step = args.reference_budget_s / max(1, args.steps + args.warmup)
    rows_per_step = int(max(1, min(wl.batch * hq, per_step / per_req * hq)))
    cursor = [0]

    def step():
        total = wl.batch * hq
        rows = (np.arange(rows_per_step, dtype=np.int64) + cursor[0]) % total
        cursor[0] = (cursor[0] + rows_per_step) % total
        oracle.decode(*codes, t.kv_indptr, t.kv_indices, t.kv_last_page_len,
                      dtype=wl.dtype, sm_scale=wl.sm_scale, rows=rows)
        return sum(int(lengths[r // hq]) for r in rows) * per_token / hq

    for _ in range(args.warmup):
        step()
    done = 0.0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        done += step()
    elapsed = time.perf_counter() - t0
    gbs = done / elapsed / 1e9
    sample = ("%d (request, query-head) rows per step of the %s workload, fp64 "
              "page-table walk" % (rows_per_step, wl.name))
    return {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(elapsed * 1e3 / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1), shapes of the workload)",
        "config": workload_config(wl),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s",
                         "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["all", "append"] + sorted(DESCRIPTIONS),
                    default="all",
                    help="all (default): every workload timed in one run, the "
                         "long-context batch as the headline line and the others "
                         "under per_config")
    ap.add_argument("--e2e-steps", type=int, default=0,
                    help="steps of the end-to-end loop (0: about 0.2 s of steps, "
                         "at least --steps, at most 2000)")
    ap.add_argument("--layout", choices=["nhd", "hnd"], default="nhd",
                    help="page tensor layout (the same values either way)")
    ap.add_argument("--cascade-split", choices=["on", "off"], default="on",
                    help="fused cascade: the prefix kernel and the suffix decode on "
                         "disjoint SMs (about 30%% / 70%%) instead of one after the other")
    ap.add_argument("--cascade", choices=["fused", "shared", "per-request"],
                    default="fused",
                    help="cascade workload: shared-prefix kernel states folded into "
                         "the suffix states by the cascade merge (fused), prefix "
                         "states merged first and combined by merge_states (shared), "
                         "or the prefix pages listed in every request's table")
    ap.add_argument("--batch", type=int, default=None,
                    help="smaller batch of the longctx / cascade workload (profiling)")
    ap.add_argument("--loader", choices=["auto", "tma", "bulk"], default="auto",
                    help="K/V loader of the decode kernel (auto: bulk rows)")
    ap.add_argument("--cpu-budget-s", type=float, default=10.0)
    ap.add_argument("--reference-budget-s", type=float, default=90.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", choices=["on", "off"], default="on",
                    help="replay each step's launches as a CUDA graph (planning "
                         "stays per step on the host)")
    ap.add_argument("--copies", choices=["auto", "side", "graph"], default="auto",
                    help="graph mode: the step's plan / input / output copies on "
                         "side streams beside the kernel graph (side), or inside "
                         "one graph per step (graph); auto: graph for steps of at "
                         "most 64 MiB of KV, side otherwise")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return 0
        line = run_reference(args, _single_rank())
        print(json.dumps(line), flush=True)
        return 0

    import paged_kv_decode_plan_gb300 as pkd
    pkd.load()   # the CUDA library must be built; there is no other path
    ranks = Ranks()
    try:
        line = run_ours(args, ranks)
        if ranks.rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        ranks.close()
    return 0


def _single_rank():
    r = Ranks.__new__(Ranks)
    r.world, r.rank, r.local, r.dist, r.backend = 1, 0, 0, None, "none"
    return r


if __name__ == "__main__":
    sys.exit(main())
