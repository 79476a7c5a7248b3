#!/usr/bin/env python
"""Throughput of the KV compressor on one GB300 (or N, one process each).

One step = one pass of the whole hot path over one batch of synthetic input:
  C128 ragged prefill, batch 1024 (896 requests extending by 4, 128 by
  U[128,16384], prefix U[0,65536]), head_dim 512, bf16 -> fp32 compact:
      plan_prefill -> compress_pool_prefill -> compress_write
  then C128 decode, batch 512 (seq_len U[1,32768], 25 % forced to page
  boundaries), head_dim 512, bf16 -> fp32:
      plan_decode -> compress_decode
Metric: compressed KV rows per second (prefill compress records + decode rows
on a page boundary), and the achieved HBM bandwidth of the dominant kernel
(the C128 prefill pool) against the measured GB300 copy bandwidth.

Inputs live in HBM when the timed region starts.  Before every step (outside
the timed region) the prefill state is restored from a pristine copy and L2
is flushed (a buffer of twice its size written, then another one read).  The
step is one CUDA graph whose kernels keep their programmatic launch edges,
timed with CUDA events around it; a second graph of the same kernels with
event-record nodes between them gives per-kernel times (the roofline's
kernel time), and each kernel's cost inside the step is also taken by
difference (the step graph against the same graph without that kernel, no
event node between kernels).  ``e2e`` repeats the step through the same
API with the step's inputs copied from pinned host memory and its outputs
copied back inside the timed region.  Beside the step, the same line carries
the C4 kernels on their own workloads (``kernels_c4``) and the
speculative-decoding verify steps (``kernels_mtp``), each kernel's cost inside
its step by difference and back to back.

``--config NAME`` times one workload alone (c4_prefill_small, c4_decode,
c128_decode, c4_prefill, c128_prefill, the speculative-decoding verify shapes
c4_prefill_mtp / c128_prefill_mtp, the C4 prefill over SWA-paged state
c4_prefill_paged, the norm + RoPE + store step on the
C128 rows, norm_rope_c128_prefill / norm_rope_c128_decode, the C4 decode with
its norm + RoPE + store in two launches and fused, c4_decode_norm_rope, and the C128
workloads through the online state, c128_online_prefill / c128_online_decode;
``all`` for each in turn) and prints one line per workload.  ``--impl reference`` times the CPU oracle on the
host cores over a bounded sample of the same step.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from compressed_kv_attention_compressplan_gb300 import workloads as wl  # noqa: E402

METRIC = "compressed KV rows/sec and achieved HBM GB/s (fraction of GB300 peak), 1 GPU"
UNIT = "rows/s"
STEP_WORKLOAD = ("c128_prefill B=1024 (896 x extend 4 + 128 x extend U[128,16384], prefix U[0,65536]) "
                 "+ c128_decode B=512 (seq_len U[1,32768], 25% on page boundaries); head_dim 512, bf16 in, "
                 "fp32 out")


# ----------------------------------------------------------------------------- helpers
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def profiled_traffic(num_c: int):
    """DRAM bytes of one c128_prefill pool launch, from the committed ncu summary:
    its per-record traffic times the records of this launch, reported only
    while the pool kernel's source is the one that was profiled (else None)."""
    import hashlib
    import re

    path = os.path.join(ROOT, "profiles", "c128_prefill_pool__c128_prefill_small.md")
    try:
        text = open(path).read()
        per = float(re.search(r"traffic_bytes_per_compress_record: ([0-9.]+)", text).group(1))
        want = re.search(r"source_sha256: ([0-9a-f]+)", text).group(1)
        h = hashlib.sha256()
        for f in ("pool_c128.cu", "common.cuh", "async_copy.cuh"):
            h.update(open(os.path.join(ROOT, "compressed_kv_attention_compressplan_gb300", "csrc", f), "rb").read())
        return per * num_c if h.hexdigest() == want else None
    except Exception:
        return None


def elem(dt: torch.dtype) -> int:
    return 2 if dt == torch.bfloat16 else 4


def prefill_events(ratio, sl, el):
    """Per compress event: (buffer_len, masked-entry count) in plan order, from
    the request lengths (closed forms of the per-request loops)."""
    R = ratio
    W = 8 if R == 4 else 128
    sl = np.asarray(sl, np.int64)
    el = np.asarray(el, np.int64)
    pl = sl - el
    nc = sl // R - pl // R
    b = np.repeat(np.arange(len(sl)), nc)
    k = np.arange(int(nc.sum())) - np.repeat(np.cumsum(nc) - nc, nc)
    p = (pl[b] // R + k + 1) * R - 1
    j = p - pl[b]
    bl = W - np.minimum(j + 1, W)
    first = np.where((R == 4) & (p == 3), 4, 0)
    first_w = (sl // R) * R - (4 if R == 4 else 0)
    nw = sl - np.maximum(pl, first_w)
    return bl, first, int(nc.sum()), int(nw.sum())


def algorithmic_bytes(w: wl.Workload) -> dict:
    """Bytes each kernel must move at minimum, each counted once."""
    hd, R, W = w.head_dim, w.ratio, w.window
    ein, eout = elem(w.in_dtype), elem(w.out_dtype)
    entry = 2 * hd * ein                      # one window entry: kv + score (C4: one half row)
    row = w.width * ein                       # one kv_score row
    ape = W * hd * ein
    B = w.batch
    if w.mode == "prefill":
        bl, first, nc, nw = prefill_events(R, w.seq_lens.numpy(), w.extend_lens.numpy())
        n_state = np.maximum(bl - first, 0)
        n_input = W - np.maximum(bl, first)
        out_rows = w.num_q_tokens if w.out_layout == wl.TOKEN else nc
        pool = int((n_state + n_input).sum()) * entry + out_rows * hd * eout + ape + 16 * nc
        write = nw * (2 * row + 8)
        plan = 24 * B + 16 * nc + 8 * nw + 16
        return {"plan": plan, "pool": pool, "write": write, "rows": nc, "num_c": nc, "num_w": nw,
                "total": plan + pool + write}
    sl = w.seq_lens.numpy()
    bnd = sl % R == 0
    first = np.where((R == 4) & (sl == 4), 4, 0)
    reads = int(((W - 1 - first) * bnd).sum()) * entry
    dec = B * (2 * row + hd * eout + 16) + reads + ape
    plan = B * (16 + 16)
    return {"plan": plan, "decode": dec, "rows": int(bnd.sum()), "total": plan + dec}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        # raw samples go to a scratch file; the JSON line carries their summary
        self.path = os.path.join(tempfile.gettempdir(), f"ckv_clocks_{os.getpid()}.csv")
        sel = str(device_index)
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            if uuid:
                sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            pass
        self.sel = sel

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.sel, f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            lines = f.readlines()
        try:
            os.remove(self.path)
        except OSError:
            pass
        for line in lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------- device runners
class PrefillRunner:
    """Device buffers + the three prefill segments of one workload."""

    def __init__(self, ckv, w: wl.Workload, dev, padded: bool = False):
        self.ckv, self.w, self.dev = ckv, w, dev
        self.kv = w.kv_score.to(dev)
        self.ape = w.ape.to(dev)
        self.rid, self.sl, self.el = w.rid.to(dev), w.seq_lens.to(dev), w.extend_lens.to(dev)
        self.state = w.state.to(dev)
        self.pristine = self.state.clone()
        nq = w.num_q_tokens
        # padded: fixed-shape plan buffers of num_q_tokens records, tails filled with
        # the invalid record (the shape a captured graph replays for any lengths)
        self.padded = padded
        self.cap_c = nq if padded else ckv.capacity_compress(w.ratio, w.batch, nq)
        self.cap_w = nq if padded else ckv.capacity_write(w.ratio, w.batch, nq)
        self.plan_c = torch.empty(max(self.cap_c, 1), 16, dtype=torch.uint8, device=dev)
        self.plan_w = torch.empty(max(self.cap_w, 1), 8, dtype=torch.uint8, device=dev)
        self.counts = torch.zeros(4, dtype=torch.int32, device=dev)
        self.status = ckv.new_status(dev)
        self.layout = ckv.OUT_TOKEN if w.out_layout == wl.TOKEN else ckv.OUT_COMPACT
        rows = nq if self.layout == ckv.OUT_TOKEN else self.cap_c
        self.out = torch.empty(max(rows, 1), w.head_dim, dtype=w.out_dtype, device=dev)
        # the planner's inputs, handed to the pool as prefetch hints (legacy state rows)
        self.hints = (self.rid, self.sl, self.el)

    def plan(self):
        c = self.ckv
        c.plan_prefill(self.w.ratio, self.rid, self.sl, self.el, self.w.num_q_tokens, self.cap_c, self.cap_w,
                       self.padded, self.plan_c[: self.cap_c], self.plan_w[: self.cap_w], self.counts, self.status)

    def pool(self):
        self.ckv.compress_pool_prefill(self.w.ratio, self.w.head_dim, self.state, self.kv, self.ape,
                                       self.plan_c[: self.cap_c], self.counts, self.layout, self.w.out_dtype,
                                       self.out, self.status, hints=self.hints)

    def write(self):
        self.ckv.compress_write(self.w.ratio, self.w.head_dim, self.state, self.kv, self.plan_w[: self.cap_w],
                                self.counts, self.status)

    def restore(self):
        self.state.copy_(self.pristine)

    def plan_fns(self, n: int):
        """n launches of the planner, each on its own copy of the lengths and of the plan buffers."""
        c, w = self.ckv, self.w
        fns = []
        for _ in range(n):
            rid, sl, el = self.rid.clone(), self.sl.clone(), self.el.clone()
            pc, pw, cnt = self.plan_c.clone(), self.plan_w.clone(), self.counts.clone()

            def fn(rid=rid, sl=sl, el=el, pc=pc, pw=pw, cnt=cnt):
                c.plan_prefill(w.ratio, rid, sl, el, w.num_q_tokens, self.cap_c, self.cap_w, self.padded,
                               pc[: self.cap_c], pw[: self.cap_w], cnt, self.status)
            fns.append(fn)
        return fns

    def steady_fns(self, n: int, which: str):
        """n launches of the pool or of the write, each on its own copy of the state, input, plan records
        and output (the plans are built once, before)."""
        self.plan()
        torch.cuda.synchronize()
        c, w = self.ckv, self.w
        fns = []
        for i in range(n):
            st = self.state if i == 0 else self.pristine.clone()
            kv, cnt, out = self.kv.clone(), self.counts.clone(), self.out.clone()
            pc, pw = self.plan_c[: self.cap_c].clone(), self.plan_w[: self.cap_w].clone()
            if which == "pool":
                def fn(st=st, kv=kv, pc=pc, cnt=cnt, out=out):
                    c.compress_pool_prefill(w.ratio, w.head_dim, st, kv, self.ape, pc, cnt, self.layout, w.out_dtype,
                                            out, self.status, hints=self.hints)
            else:
                def fn(st=st, kv=kv, pw=pw, cnt=cnt):
                    c.compress_write(w.ratio, w.head_dim, st, kv, pw, cnt, self.status)
            fns.append(fn)
        return fns


class PagedPrefillRunner(PrefillRunner):
    """A prefill over SWA-paged state: the paged planner translates positions through the token maps."""

    def __init__(self, ckv, w: wl.Workload, maps: wl.PagedMaps, dev):
        super().__init__(ckv, w, dev)
        self.maps = maps
        self.r2t = maps.req_to_token.to(dev)
        self.f2s = maps.full_to_state.to(dev)
        self.cap_w = ckv.capacity_write_paged(w.ratio, w.batch, w.num_q_tokens, maps.swa_page_size)
        self.plan_w = torch.empty(max(self.cap_w, 1), 8, dtype=torch.uint8, device=dev)
        self.hints = None  # the hints name legacy rows

    def plan(self):
        m = self.maps
        self.ckv.plan_prefill_paged(self.w.ratio, self.rid, self.r2t, self.f2s, m.swa_page_size, m.ring_size, self.sl,
                                    self.el, self.w.num_q_tokens, self.cap_c, self.cap_w, counts=self.counts,
                                    status=self.status, plan_c=self.plan_c[: self.cap_c],
                                    plan_w=self.plan_w[: self.cap_w])


class DecodeRunner:
    def __init__(self, ckv, w: wl.Workload, dev):
        self.ckv, self.w, self.dev = ckv, w, dev
        self.kv = w.kv_score.to(dev)
        self.ape = w.ape.to(dev)
        self.rid, self.sl = w.rid.to(dev), w.seq_lens.to(dev)
        self.state = w.state.to(dev)
        self.pristine = self.state.clone()
        self.plan_d = torch.empty(max(w.batch, 1), 16, dtype=torch.uint8, device=dev)
        # C128: the planner also lists the page-boundary rows, so the decode reads its share of windows directly
        self.order = ckv.new_decode_order(w.batch, dev) if w.ratio == 128 else None
        self.status = ckv.new_status(dev)
        self.out = torch.empty(max(w.batch, 1), w.head_dim, dtype=w.out_dtype, device=dev)

    def plan(self):
        self.ckv.plan_decode(self.w.ratio, self.rid, self.sl, self.plan_d[: self.w.batch], self.status,
                             order=self.order)

    def hints(self):
        """The planner's rid / seq_lens, from which the decode prefetches its windows."""
        return {"rid_hint": self.rid, "seq_lens_hint": self.sl}

    def decode(self):
        self.ckv.compress_decode(self.w.ratio, self.w.head_dim, self.state, self.kv, self.ape,
                                 self.plan_d[: self.w.batch], self.w.out_dtype, self.out[: self.w.batch],
                                 self.status, order=self.order, **self.hints())

    def restore(self):
        self.state.copy_(self.pristine)

    def steady_fns(self, n: int):
        """n launches of the decode kernel, each on its own copy of the state, input, plan and output."""
        self.plan()
        torch.cuda.synchronize()
        fns = []
        for i in range(n):
            st = self.state if i == 0 else self.pristine.clone()
            kv, pd, out = self.kv.clone(), self.plan_d[: self.w.batch].clone(), self.out[: self.w.batch].clone()
            order = None if self.order is None else self.order.clone()

            def fn(st=st, kv=kv, pd=pd, out=out, order=order):
                self.ckv.compress_decode(self.w.ratio, self.w.head_dim, st, kv, self.ape, pd, self.w.out_dtype, out,
                                         self.status, order=order, **self.hints())
            fns.append(fn)
        return fns


_cudart = None


class NormRopeRunner:
    """Device buffers of the norm + RoPE + store step over one set of compressed rows.  The plan it reads is
    built once, by the library's planner, before any timing."""

    def __init__(self, ckv, x: wl.NormRopeInputs, dev):
        self.ckv, self.x, self.dev = ckv, x, dev
        self.status = ckv.new_status(dev)
        self.rows = x.rows.to(dev)
        self.weight = x.weight.to(dev)
        self.freqs = x.freqs.to(dev)
        self.out_loc = x.out_loc.to(dev)
        self.cache = torch.zeros(x.cache_rows, x.head_dim, dtype=x.cache_dtype, device=dev)
        rid, sl = x.rid.to(dev), x.seq_lens.to(dev)
        if x.extend_lens is not None:
            nq = int(x.extend_lens.sum())
            self.plan_c, _, self.counts = ckv.plan_prefill(x.ratio, rid, sl, x.extend_lens.to(dev), nq,
                                                           status=self.status)
            torch.cuda.synchronize()
            self.records = int(self.counts[0])
            if self.records > self.rows.shape[0]:
                raise RuntimeError("fewer rows than compress records")
        else:
            self.plan_d = ckv.plan_decode(x.ratio, rid, sl, status=self.status)
            self.records = rid.numel()
        self.boundary = int((x.seq_lens % x.ratio == 0).sum()) if x.extend_lens is None else self.records

    def run(self):
        c, x = self.ckv, self.x
        if x.extend_lens is not None:
            c.norm_rope_store_prefill(x.ratio, self.rows, self.plan_c, self.counts, self.weight, x.eps, self.freqs,
                                      self.out_loc, self.cache, in_layout=c.OUT_COMPACT, status=self.status)
        else:
            c.norm_rope_store_decode(x.ratio, self.rows, self.plan_d, self.weight, x.eps, self.freqs, self.out_loc,
                                     self.cache, status=self.status)

    def restore(self):
        pass

    def steady_fns(self, n: int):
        """n launches, each on its own copy of the rows, plan and out_loc (table, weight and cache shared)."""
        c, x = self.ckv, self.x
        fns = []
        for i in range(n):
            rows, loc = self.rows.clone(), self.out_loc.clone()
            if x.extend_lens is not None:
                pc, cnt = self.plan_c.clone(), self.counts.clone()

                def fn(rows=rows, loc=loc, pc=pc, cnt=cnt):
                    c.norm_rope_store_prefill(x.ratio, rows, pc, cnt, self.weight, x.eps, self.freqs, loc,
                                              self.cache, in_layout=c.OUT_COMPACT, status=self.status)
            else:
                pd = self.plan_d.clone()

                def fn(rows=rows, loc=loc, pd=pd):
                    c.norm_rope_store_decode(x.ratio, rows, pd, self.weight, x.eps, self.freqs, loc, self.cache,
                                             status=self.status)
            fns.append(fn)
        return fns

    def algorithmic_bytes(self) -> int:
        """Rows read (decode: boundary rows only; the rest are zero), cache rows written, plan and out_loc
        entries, one table row per record and the weight."""
        x = self.x
        per_write = x.head_dim * elem(x.cache_dtype) + 16 + 8 + 4 * x.rope_dim
        return self.boundary * x.head_dim * 4 + self.records * per_write + x.head_dim * 4


class OnlineRunner:
    """A C128 step through the online state.  Setup (not timed): the library
    folds each request's earlier tokens of its current group into the state,
    which is then kept as the pristine copy restored before every step."""

    def __init__(self, ckv, x: wl.OnlineInputs, dev):
        self.ckv, self.x, self.dev = ckv, x, dev
        hd = x.head_dim
        self.status = ckv.new_status(dev)
        self.kv = x.kv_score.to(dev)
        self.ape = x.ape.to(dev)
        self.rid, self.sl = x.rid.to(dev), x.seq_lens.to(dev)
        self.el = x.extend_lens.to(dev) if x.extend_lens is not None else None
        batch = x.rid.numel()
        self.state = torch.zeros(batch, 3 * hd, dtype=torch.float32, device=dev)
        has = x.prefix_lens > 0
        if bool(has.any()):
            end = x.seq_lens - (x.extend_lens if x.extend_lens is not None else 1)
            rows = x.prefix_rows.to(dev)
            n = int(x.prefix_lens.sum())
            units, counts = ckv.plan_online_prefill(x.rid[has].to(dev), end[has].to(dev),
                                                    x.prefix_lens[has].to(dev), n, status=self.status)
            ckv.compress_online_prefill(hd, self.state, rows, self.ape, units, counts, ckv.OUT_TOKEN,
                                        status=self.status)
        self.pristine = self.state.clone()
        if x.mode == "prefill":
            nq = int(x.extend_lens.sum())
            self.cap_u = ckv.capacity_online_units(batch, nq)
            self.units = torch.empty(self.cap_u, 16, dtype=torch.uint8, device=dev)
            self.counts = torch.zeros(4, dtype=torch.int32, device=dev)
            self.cap_c = ckv.capacity_compress(128, batch, nq)
            self.out = torch.empty(self.cap_c, hd, dtype=x.out_dtype, device=dev)
            self.plan()
            torch.cuda.synchronize()
            self.num_c, self.num_units = int(self.counts[0]), int(self.counts[1])
            self.loads = int((x.prefix_lens > 0).sum())
        else:
            self.plan_d = torch.empty(batch, 16, dtype=torch.uint8, device=dev)
            self.out = torch.empty(batch, hd, dtype=x.out_dtype, device=dev)
            self.num_c = int((x.seq_lens % 128 == 0).sum())
        torch.cuda.synchronize()

    def plan(self):
        c, x = self.ckv, self.x
        if x.mode == "prefill":
            c.plan_online_prefill(self.rid, self.sl, self.el, self.kv.shape[0], 0, self.cap_u, units=self.units,
                                  counts=self.counts, status=self.status)
        else:
            c.plan_online_decode(self.rid, self.sl, 0, plan_d=self.plan_d, status=self.status)

    def compute(self):
        c, x = self.ckv, self.x
        if x.mode == "prefill":
            c.compress_online_prefill(x.head_dim, self.state, self.kv, self.ape, self.units, self.counts,
                                      c.OUT_COMPACT, out=self.out, status=self.status)
        else:
            c.compress_online_decode(x.head_dim, self.state, self.kv, self.ape, self.plan_d, out=self.out,
                                     status=self.status)

    def restore(self):
        self.state.copy_(self.pristine)

    def steady_fns(self, n: int):
        """Decode: n launches of the fold, each on its own copy of the state, input, plan and output."""
        c, x = self.ckv, self.x
        self.plan()
        torch.cuda.synchronize()
        fns = []
        for i in range(n):
            st = self.state if i == 0 else self.pristine.clone()
            kv, pd, out = self.kv.clone(), self.plan_d.clone(), self.out.clone()

            def fn(st=st, kv=kv, pd=pd, out=out):
                c.compress_online_decode(x.head_dim, st, kv, self.ape, pd, out=out, status=self.status)
            fns.append(fn)
        return fns

    def algorithmic_bytes(self) -> int:
        """Input rows, plan records, slots loaded and stored, the output and ape, each once."""
        x = self.x
        hd = x.head_dim
        slot = 3 * hd * 4
        batch = x.rid.numel()
        if x.mode == "prefill":
            return (self.kv.numel() * 2 + self.num_units * 16 + self.loads * slot + batch * slot +
                    self.num_c * hd * elem(x.out_dtype) + 128 * hd * 2)
        first = int(((x.seq_lens - 1) % 128 == 0).sum())
        return (batch * (2 * hd * 2 + 16 + hd * elem(x.out_dtype) + slot) + (batch - first) * slot + 128 * hd * 2)


def cudart():
    """The CUDA runtime library this process already loaded (through torch)."""
    global _cudart
    if _cudart is None:
        import ctypes

        path = None
        with open("/proc/self/maps") as f:
            for line in f:
                if "libcudart.so" in line:
                    path = line.split()[-1]
                    break
        lib = ctypes.CDLL(path) if path else ctypes.CDLL("libcudart.so")
        lib.cudaEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
        lib.cudaEventRecordWithFlags.restype = ctypes.c_int
        _cudart = lib
    return _cudart


class StepGraph:
    """One CUDA graph for a whole step.  With inner_events the segments are
    separated by event-record nodes, so per-kernel times are GPU timestamps of
    one graph execution; without, only the whole step is bracketed and the
    kernels overlap their launches through programmatic dependent launch."""

    def __init__(self, segments, inner_events: bool = True):
        if not inner_events:  # one timed segment: the kernels keep their programmatic launch edges
            fns = [fn for _, fn in segments]
            segments = [("step", lambda: [f() for f in fns])]
        self.names = [n for n, _ in segments]
        for _, fn in segments:  # eager warm-up outside capture (function attributes, modules)
            fn()
        self.evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(segments) + 1)]
        for e in self.evs:
            e.record()  # creates the underlying events
        torch.cuda.synchronize()
        lib = cudart()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            st = torch.cuda.current_stream().cuda_stream
            rc = lib.cudaEventRecordWithFlags(self.evs[0].cuda_event, st, 1)  # cudaEventRecordExternal
            for i, (_, fn) in enumerate(segments):
                fn()
                rc |= lib.cudaEventRecordWithFlags(self.evs[i + 1].cuda_event, st, 1)
        if rc != 0:
            raise RuntimeError("cudaEventRecordWithFlags failed during capture")

    def replay(self):
        self.graph.replay()

    def times_ms(self):
        return [self.evs[i].elapsed_time(self.evs[i + 1]) for i in range(len(self.names))]


class L2Flush:
    """Writes a buffer of twice the L2 size, then reads another one of the same
    size: the timed region that follows starts with an L2 that holds none of
    its inputs and no dirty lines (whose write-back would otherwise compete
    with the timed kernel's own traffic)."""

    def __init__(self, dev):
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        n = 2 * max(l2, 64 << 20)
        self.w = torch.empty(n, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(n // 4, dtype=torch.int32, device=dev)

    def zero_(self):
        self.w.zero_()
        self.r.max()


def l2_flush_buffer(dev):
    return L2Flush(dev)


def l2_bytes(dev) -> int:
    return torch.cuda.get_device_properties(dev).L2_cache_size


def copies_for(bytes_per_launch: int, dev, cap: int = 16) -> int:
    """Input copies needed so that the other copies' traffic between two uses of one copy exceeds twice the L2."""
    return int(min(cap, max(2, -(-2 * l2_bytes(dev) // max(bytes_per_launch, 1)) + 1)))


def steady_state_us(fns, reps: int = 10, samples: int = 5) -> float:
    """Mean device time of one launch when launches run back to back, each of
    `fns` on its own copy of the inputs (the copies together exceed the L2, so
    every launch reads its inputs from HBM): one CUDA graph of reps x len(fns)
    launches bracketed by two events; the median of `samples` replays."""
    for f in fns:
        f()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            for f in fns:
                f()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g.replay()
    ts = []
    for _ in range(samples):
        torch.cuda.synchronize()
        e0.record()
        g.replay()
        e1.record()
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts) * 1e3 / (reps * len(fns))


def same_bytes_floor(nbytes: int, dev, peak: float) -> dict:
    """What plain device copies achieve when they move the same number of bytes as one launch of a kernel
    (nbytes = read + write), back to back over buffers that together exceed the L2, timed like the kernel
    (steady_state_us): torch copy_ (the operation the measured HBM peak comes from) and an elementwise SM
    kernel (bitwise_not over int32).  For launches of a few tens of MB the fixed costs of a launch (start,
    first-byte latency, drain) are not amortised, so this is the practical ceiling for such a kernel."""
    half = max(nbytes // 2 // 16 * 16, 16)
    n = copies_for(nbytes, dev)
    bufs = [(torch.empty(half // 4, dtype=torch.int32, device=dev), torch.empty(half // 4, dtype=torch.int32,
                                                                                device=dev)) for _ in range(n)]
    for a_, _ in bufs:
        a_.fill_(1)
    copy_us = steady_state_us([lambda a_=a_, b_=b_: b_.copy_(a_) for a_, b_ in bufs])
    ew_us = steady_state_us([lambda a_=a_, b_=b_: torch.bitwise_not(a_, out=b_) for a_, b_ in bufs])
    best = min(copy_us, ew_us)
    del bufs
    return {"bytes": 2 * half, "copy_us": copy_us, "elementwise_us": ew_us,
            "frac_of_peak": 2 * half / (best * 1e-6) / 1e9 / peak}


def instep_by_difference(segments, flush, restore, reps: int) -> dict:
    """In-step cost of every kernel of a step, free of event nodes between kernels: the median device time
    of the whole step graph minus the median time of the same graph with that one kernel left out (the
    other kernels keep their programmatic launch edges).  The variants are replayed in turn, `reps` times
    each, every replay after a state restore and an L2 flush, with CUDA events around the graph only."""
    graphs = [("step", StepGraph(segments, inner_events=False))]
    for i, (name, _) in enumerate(segments):
        graphs.append((name, StepGraph([s for j, s in enumerate(segments) if j != i], inner_events=False)))
    times = {name: [] for name, _ in graphs}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for rep in range(reps + 2):
        for name, g in graphs:
            restore()
            flush.zero_()
            torch.cuda.synchronize()
            e0.record()
            g.replay()
            e1.record()
            e1.synchronize()
            if rep >= 2:  # two untimed rounds first
                times[name].append(e0.elapsed_time(e1) * 1e3)
    full = np.array(times["step"])
    out = {"step_us": float(np.median(full)), "reps": reps}
    for name, _ in segments:
        # replays of one round ran back to back: the median of the paired differences
        d = full - np.array(times[name])
        out[f"{name}_us"] = float(np.median(d))
        out[f"{name}_us_iqr"] = [float(np.percentile(d, 25)), float(np.percentile(d, 75))]
    out["sum_us"] = sum(out[f"{n}_us"] for n, _ in segments)
    return out


class nvtx_range:
    """An NVTX range around a phase of the benchmark (visible in a profiler's timeline; free otherwise)."""

    def __init__(self, name: str):
        self.name = name

    def __enter__(self):
        torch.cuda.nvtx.range_push(self.name)

    def __exit__(self, *exc):
        torch.cuda.nvtx.range_pop()
        return False


def run_graph(step: StepGraph, flush, restore, steps, warmup, ws, sampler=None):
    """Per-step segment times (ms) of `steps` timed replays after `warmup` untimed ones."""
    for _ in range(warmup):
        restore()
        flush.zero_()
        with nvtx_range("warmup step"):
            step.replay()
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    seg = []
    t0 = time.perf_counter()
    for _ in range(steps):
        with nvtx_range("restore + L2 flush"):
            restore()
            flush.zero_()
        with nvtx_range("timed step"):
            step.replay()
            torch.cuda.synchronize()
        seg.append(step.times_ms())
    wall = time.perf_counter() - t0
    barrier(ws)
    clocks = sampler.stop() if sampler else None
    return np.array(seg), wall, clocks


def c4_kernels(args, ckv, dev, seed: int, peak: float) -> dict:
    """The C4 kernels on their own workloads, reported beside the headline step (which is C128): the C4
    ragged prefill (plan -> pool -> write) and the C4 decode (plan -> decode), each step in one graph,
    per-kernel costs inside the step by difference, the pool's and the decode's fraction of the peak, the
    decode back to back against its same-bytes floor, and the decode with its norm + RoPE + store in two
    launches against the fused launch."""
    w4 = wl.c4_prefill(seed)
    w2 = wl.c4_decode(seed)
    pre = PrefillRunner(ckv, w4, dev)
    dec = DecodeRunner(ckv, w2, dev)
    flush = l2_flush_buffer(dev)
    b4, b2 = algorithmic_bytes(w4), algorithmic_bytes(w2)
    reps = max(200, 10 * args.steps)
    pre_seg = [("plan_prefill", pre.plan), ("pool_prefill", pre.pool), ("write", pre.write)]
    dec_seg = [("plan_decode", dec.plan), ("decode", dec.decode)]
    ip = instep_by_difference(pre_seg, flush, pre.restore, reps)
    idc = instep_by_difference(dec_seg, flush, dec.restore, reps)
    ev_p, _, _ = run_graph(StepGraph(pre_seg), flush, pre.restore, args.steps, args.warmup, 1)
    ev_d, _, _ = run_graph(StepGraph(dec_seg), flush, dec.restore, args.steps, args.warmup, 1)
    if int(pre.status[0]) or int(dec.status[0]):
        raise RuntimeError(f"device status set: c4 prefill {int(pre.status[0])} decode {int(dec.status[0])}")
    pool_ev_us = float(ev_p[:, 1].mean()) * 1e3
    out = {
        "c4_prefill": {"workload": "c4_prefill B=64, prefix U[0,4096], extend U[1,4096], hd 512, bf16 -> bf16 token",
                       "num_c": b4["num_c"], "bytes": {"pool": b4["pool"], "write": b4["write"], "plan": b4["plan"]},
                       "events_us": {n: float(ev_p[:, i].mean()) * 1e3 for i, (n, _) in enumerate(pre_seg)},
                       "pool_events_frac": b4["pool"] / (pool_ev_us * 1e-6) / 1e9 / peak,
                       "instep": ip,
                       "pool_instep_frac": (b4["pool"] / (ip["pool_prefill_us"] * 1e-6) / 1e9 / peak
                                            if ip["pool_prefill_us"] > 0 else None)},
        "c4_decode": {"workload": "c4_decode B=256, seq_len U[1,8192], hd 512, bf16 -> f32", "rows": b2["rows"],
                      "bytes": b2["decode"],
                      "events_us": {n: float(ev_d[:, i].mean()) * 1e3 for i, (n, _) in enumerate(dec_seg)},
                      "instep": idc,
                      "decode_instep_frac": (b2["decode"] / (idc["decode_us"] * 1e-6) / 1e9 / peak
                                             if idc["decode_us"] > 0 else None)},
    }
    if not args.no_back_to_back:
        n = copies_for(b2["decode"], dev)
        us = steady_state_us(dec.steady_fns(n))
        floor = same_bytes_floor(b2["decode"], dev, peak)
        best = min(floor["copy_us"], floor["elementwise_us"])
        out["c4_decode"].update({"back_to_back_us": us,
                                 "back_to_back_frac": b2["decode"] / (us * 1e-6) / 1e9 / peak,
                                 "same_bytes_floor": floor, "floor_ratio": us / best})
    # the decode with its norm + RoPE + store: two launches against the fused one
    out["c4_decode_norm_rope"] = decode_norm_measure(args, "c4_decode_norm_rope", seed, ckv, dev)
    del pre, dec
    torch.cuda.empty_cache()
    return out


def mtp_kernels(args, ckv, dev, seed: int, peak: float) -> dict:
    """The speculative-decoding verify steps (1024 requests x extend 4, fixed-shape plan buffers padded with
    the invalid record), reported beside the headline step: per-kernel costs inside each step by difference
    and the planner, the pool and the write back to back (the write also against its same-bytes floor)."""
    out = {}
    for name in ("c128_prefill_mtp", "c4_prefill_mtp"):
        w = wl.NAMED[name](seed)
        r = PrefillRunner(ckv, w, dev, padded=True)
        flush = l2_flush_buffer(dev)
        b = algorithmic_bytes(w)
        segs = [("plan_prefill", r.plan), ("pool_prefill", r.pool), ("write", r.write)]
        ins = instep_by_difference(segs, flush, r.restore, max(200, 10 * args.steps))
        if int(r.status[0]):
            raise RuntimeError(f"device status set: {name} {int(r.status[0])}")
        d = {"workload": f"{name}: 1024 requests x extend 4, prefix U[0,65536], hd 512, padded plans",
             "bytes": {"pool": b["pool"], "write": b["write"], "plan": b["plan"]}, "num_c": b["num_c"],
             "instep": ins}
        if not args.no_back_to_back:
            d["plan_back_to_back_us"] = steady_state_us(r.plan_fns(16))
            d["pool_back_to_back_us"] = steady_state_us(r.steady_fns(copies_for(b["pool"], dev), "pool"))
            us = steady_state_us(r.steady_fns(copies_for(b["write"], dev), "write"))
            floor = same_bytes_floor(b["write"], dev, peak)
            d.update({"write_back_to_back_us": us, "write_back_to_back_frac": b["write"] / (us * 1e-6) / 1e9 / peak,
                      "write_vs_floor": min(floor["copy_us"], floor["elementwise_us"]) / us})
        out[name] = d
        del r
        torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------------------- CPU baseline (oracle)
def oracle_step(o, w5, w3, frac5=1.0):
    """The oracle over (a sample of) the step: C128 prefill pool + write, then
    C128 decode.  Returns (rows, seconds)."""
    t0 = time.perf_counter()
    pc, pw, (nc, nw), _ = o.plan_prefill(128, w5.rid, w5.seq_lens, w5.extend_lens)
    k = max(1, int(round(nc * frac5)))
    st5 = wl.bits(w5.state).copy() if frac5 >= 1.0 else None
    if st5 is None:
        st5 = wl.bits(w5.state)  # read-only use below (the write step is skipped for a sample)
    o.compress_pool_prefill(128, 512, o.BF16, o.F32, st5, wl.bits(w5.kv_score), wl.bits(w5.ape), pc[:k], k,
                            w5.num_q_tokens, o.OUT_COMPACT)
    if frac5 >= 1.0:
        o.compress_write(128, 512, o.BF16, st5, wl.bits(w5.kv_score), pw, nw)
    st3 = wl.bits(w3.state).copy()
    pd = o.plan_decode(128, w3.rid, w3.seq_lens)
    o.compress_decode(128, 512, o.BF16, o.F32, st3, wl.bits(w3.kv_score), wl.bits(w3.ape), pd)
    rows = k + int((w3.seq_lens.numpy() % 128 == 0).sum())
    return rows, time.perf_counter() - t0


def oracle_step_threads(o, w5, w3, threads: int):
    """The same oracle step with its independent parts spread over `threads` host threads (the C oracle
    runs outside the GIL): the prefill's compress records in contiguous chunks, then its write records
    in chunks (each writes its own state rows, after every pool), then the decode rows in chunks.  The
    oracle itself is unchanged.  Returns (rows, seconds)."""
    from concurrent.futures import ThreadPoolExecutor

    def chunks(n):
        b = np.linspace(0, n, threads + 1).astype(np.int64)
        return [(int(b[i]), int(b[i + 1])) for i in range(threads) if b[i + 1] > b[i]]

    t0 = time.perf_counter()
    pc, pw, (nc, nw), _ = o.plan_prefill(128, w5.rid, w5.seq_lens, w5.extend_lens)
    st5 = wl.bits(w5.state).copy()
    in5, ape5 = wl.bits(w5.kv_score), wl.bits(w5.ape)
    st3 = wl.bits(w3.state).copy()
    in3, ape3 = wl.bits(w3.kv_score), wl.bits(w3.ape)
    pd = o.plan_decode(128, w3.rid, w3.seq_lens)
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda c: o.compress_pool_prefill(128, 512, o.BF16, o.F32, st5, in5, ape5, pc[c[0]:c[1]],
                                                      c[1] - c[0], w5.num_q_tokens, o.OUT_COMPACT), chunks(nc)))
        list(ex.map(lambda c: o.compress_write(128, 512, o.BF16, st5, in5, pw[c[0]:c[1]], c[1] - c[0]), chunks(nw)))
        list(ex.map(lambda c: o.compress_decode(128, 512, o.BF16, o.F32, st3, in3[c[0]:c[1]], ape3, pd[c[0]:c[1]]),
                    chunks(w3.batch)))
    rows = nc + int((w3.seq_lens.numpy() % 128 == 0).sum())
    return rows, time.perf_counter() - t0


def cores_used() -> dict:
    try:
        aff = len(os.sched_getaffinity(0))
    except Exception:
        aff = os.cpu_count()
    return {"host_cores": aff}


# ----------------------------------------------------------------------------- main modes
def bench_step(args, ws, rank, local):
    from compressed_kv_attention_compressplan_gb300 import build as B
    from compressed_kv_attention_compressplan_gb300 import ckv

    B.build()
    ckv.load_library()
    dev = torch.device("cuda", local)
    seed = args.seed + rank
    w5 = wl.c128_prefill(seed)
    w3 = wl.c128_decode(seed)
    pre = PrefillRunner(ckv, w5, dev)
    dec = DecodeRunner(ckv, w3, dev)
    flush = l2_flush_buffer(dev)

    def restore():
        pre.restore()
        dec.restore()

    segments = [("plan_prefill", pre.plan), ("pool_prefill", pre.pool), ("write", pre.write),
                ("plan_decode", dec.plan), ("decode", dec.decode)]
    step = StepGraph(segments, inner_events=False)
    timed = StepGraph(segments, inner_events=True)
    launches_per_step = 5
    sampler = ClockSampler(local)
    with nvtx_range("headline step"):
        step_ms, wall, clocks = run_graph(step, flush, restore, args.steps, args.warmup, ws, sampler)
    step_ms = step_ms[:, 0]
    # per-kernel breakdown (event nodes between the kernels; not part of the headline)
    with nvtx_range("per-kernel events"):
        seg_ms, _, _ = run_graph(timed, flush, restore, args.steps, args.warmup, ws)
    if int(pre.status[0]) or int(dec.status[0]):
        raise RuntimeError(f"device status set: prefill {int(pre.status[0])} decode {int(dec.status[0])}")
    b5 = algorithmic_bytes(w5)
    b3 = algorithmic_bytes(w3)
    nc = int(pre.counts[0])
    assert nc == b5["num_c"] and int(pre.counts[1]) == b5["num_w"], "plan counts differ from the closed forms"
    rows_per_step = b5["rows"] + b3["rows"]
    total_s = float(step_ms.sum()) / 1e3
    total_s = max_over_ranks(total_s, ws)
    rows_all = sum_over_ranks(rows_per_step * args.steps, ws)
    value = rows_all / total_s
    peak, peak_kind = peaks()
    pool_ms = float(seg_ms[:, 1].mean())
    pool_gbs = b5["pool"] / (pool_ms * 1e-3) / 1e9
    dec_ms = float(seg_ms[:, 4].mean())
    dec_gbs = b3["decode"] / (dec_ms * 1e-3) / 1e9
    step_bytes = b5["total"] + b3["total"]
    # every kernel's cost inside the timed step, by difference (no event nodes between the kernels)
    instep_reps = max(200, 10 * args.steps)
    with nvtx_range("in-step costs by difference"):
        instep = {} if args.no_instep else instep_by_difference(segments, flush, restore, reps=instep_reps)
    for key, nbytes in (("pool_prefill", b5["pool"]), ("write", b5["write"]), ("decode", b3["decode"])):
        if args.no_instep:
            break
        us = instep[f"{key}_us"]
        instep[f"{key}_instep_gbs"] = nbytes / (us * 1e-6) / 1e9 if us > 0 else None
        instep[f"{key}_instep_frac"] = instep[f"{key}_instep_gbs"] / peak if us > 0 else None
    instep["method"] = None if args.no_instep else ("median over rounds of (step time - time of the step without that kernel), each round "
                        f"replaying every variant once; {instep_reps} rounds, L2 flushed before every replay")
    # the decode kernel back to back over copies of its inputs that together exceed the L2 (a kernel of ~10 us
    # is not resolved by event nodes around it: they add the graph's node-to-node latency)
    back_to_back = {}
    torch.cuda.nvtx.range_push("back to back")
    if not args.no_back_to_back:
        n_dec = copies_for(b3["decode"], dev)
        us = steady_state_us(dec.steady_fns(n_dec))
        gbs = b3["decode"] / (us * 1e-6) / 1e9
        floor = same_bytes_floor(b3["decode"], dev, peak)
        back_to_back = {"decode_back_to_back_us": us, "decode_back_to_back_gbs": gbs,
                        "decode_back_to_back_frac": gbs / peak, "decode_back_to_back_copies": n_dec,
                        "decode_same_bytes_floor": floor,
                        "decode_vs_floor": min(floor["copy_us"], floor["elementwise_us"]) / us}
        # the prefill write back to back, with its own same-bytes floor
        n_w = copies_for(b5["write"], dev)
        us = steady_state_us(pre.steady_fns(n_w, "write"))
        gbs = b5["write"] / (us * 1e-6) / 1e9
        floor = same_bytes_floor(b5["write"], dev, peak)
        back_to_back.update({"write_back_to_back_us": us, "write_back_to_back_gbs": gbs,
                             "write_back_to_back_frac": gbs / peak, "write_same_bytes_floor": floor,
                             "write_vs_floor": min(floor["copy_us"], floor["elementwise_us"]) / us})
        pre.restore()
        torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()

    # ---- end to end: inputs from pinned host memory, outputs back, inside the timed region
    torch.cuda.nvtx.range_push("end to end")
    h_kv5 = w5.kv_score.pin_memory()
    h_len5 = [t.pin_memory() for t in (w5.rid, w5.seq_lens, w5.extend_lens)]
    h_kv3 = w3.kv_score.pin_memory()
    h_len3 = [t.pin_memory() for t in (w3.rid, w3.seq_lens)]
    h_out5 = torch.empty(nc, w5.head_dim, dtype=w5.out_dtype).pin_memory()
    h_out3 = torch.empty(w3.batch, w3.head_dim, dtype=w3.out_dtype).pin_memory()
    h2d = (h_kv5.numel() * elem(w5.in_dtype) + sum(t.numel() * 8 for t in h_len5) +
           h_kv3.numel() * elem(w3.in_dtype) + sum(t.numel() * 8 for t in h_len3))
    d2h = h_out5.numel() * elem(w5.out_dtype) + h_out3.numel() * elem(w3.out_dtype)
    # Pipelined over two sets of device buffers: the upload of step k + 1 (copy stream) overlaps step k
    # (compute stream), and step k's outputs go back on a third stream; a set is overwritten only after
    # its previous step ran and its outputs were read.  The prefill state is not restored inside this
    # loop (each step does the same work on it).
    pre2, dec2 = PrefillRunner(ckv, w5, dev), DecodeRunner(ckv, w3, dev)
    step2 = StepGraph([("plan_prefill", pre2.plan), ("pool_prefill", pre2.pool), ("write", pre2.write),
                       ("plan_decode", dec2.plan), ("decode", dec2.decode)], inner_events=False)
    sets = [(pre, dec, step), (pre2, dec2, step2)]
    main = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    done = [torch.cuda.Event(), torch.cuda.Event()]   # the set's step ran
    read = [torch.cuda.Event(), torch.cuda.Event()]   # the set's outputs were read back
    e2e_steps = max(2, min(args.steps, 10))

    def e2e_pass(n):
        for k in range(n):
            i = k % 2
            p, d, g = sets[i]
            with torch.cuda.stream(up):
                if k >= 2:
                    up.wait_event(done[i])
                    up.wait_event(read[i])
                p.kv.copy_(h_kv5, non_blocking=True)
                for dst, h in zip((p.rid, p.sl, p.el), h_len5):
                    dst.copy_(h, non_blocking=True)
                d.kv.copy_(h_kv3, non_blocking=True)
                for dst, h in zip((d.rid, d.sl), h_len3):
                    dst.copy_(h, non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(up)
            main.wait_event(ready)
            g.replay()
            done[i].record(main)
            with torch.cuda.stream(down):
                down.wait_event(done[i])
                h_out5.copy_(p.out[:nc], non_blocking=True)
                h_out3.copy_(d.out[: w3.batch], non_blocking=True)
                read[i].record(down)
        main.wait_stream(down)
        main.wait_stream(up)

    e2e_pass(2)  # warms the copy engines and both graphs
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    e2e_pass(e2e_steps)
    e1.record(main)
    torch.cuda.synchronize()
    e2e_s = e0.elapsed_time(e1) / 1e3
    # the host link's own rate on this machine: the step's input alone, one plain copy, three times
    link = []
    for _ in range(3):
        l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        l0.record(up)
        with torch.cuda.stream(up):
            pre.kv.copy_(h_kv5, non_blocking=True)
        l1.record(up)
        torch.cuda.synchronize()
        link.append(h_kv5.numel() * elem(w5.in_dtype) / (l0.elapsed_time(l1) * 1e-3) / 1e9)
    link_gbs = float(np.median(link))
    del pre2, dec2, step2
    torch.cuda.nvtx.range_pop()
    e2e_s = max_over_ranks(e2e_s, ws)
    e2e_value = sum_over_ranks(rows_per_step * e2e_steps, ws) / e2e_s

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": float(step_ms.mean()), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded CPU generator; shapes and length mixes of the serving regimes)",
        "config": {"workload": STEP_WORKLOAD, "global_batch": ws * (w5.batch + w3.batch),
                   "num_q_tokens": w5.num_q_tokens, "compress_rows_prefill": b5["rows"],
                   "compress_rows_decode": b3["rows"], "head_dim": 512, "in_dtype": "bf16", "out_dtype": "f32",
                   "parallelism": f"independent requests x{ws} (no collective)",
                   "l2": "flushed before every step (2x L2 written, then 2x L2 read), prefill state restored "
                         "outside the timing",
                   "algorithmic_bytes_per_step": step_bytes},
        "roofline": {"bound": "hbm", "kernel": "c128_persistent_kernel (prefill pool)", "achieved": pool_gbs, "peak": peak,
                     "unit": "GB/s", "frac": pool_gbs / peak, "peak_kind": f"{peak_kind} hbm_gbs",
                     "traffic": profiled_traffic(b5["num_c"]), "traffic_source": "profiles/c128_prefill_pool__c128_prefill_small.md "
                     "(ncu dram bytes per compress record x records)", "algorithmic_bytes": b5["pool"],
                     "avg_launch_ms": pool_ms},
        "kernels": {
            "plan_prefill_us": float(seg_ms[:, 0].mean()) * 1e3,
            "pool_prefill_us": pool_ms * 1e3, "pool_prefill_gbs": pool_gbs,
            "write_us": float(seg_ms[:, 2].mean()) * 1e3, "plan_decode_us": float(seg_ms[:, 3].mean()) * 1e3,
            "decode_us": dec_ms * 1e3, "decode_gbs": dec_gbs, "decode_frac": dec_gbs / peak,
            "event_node_note": "the *_us above are timed with event nodes between the kernels; instep has "
                               "the costs inside the timed step",
            "instep": instep,
            **back_to_back,
            "sum_of_kernel_segments_us": float(seg_ms.sum(1).mean()) * 1e3,
            "step_gbs": step_bytes / (float(step_ms.mean()) * 1e-3) / 1e9},
        "kernels_c4": None,
        "kernels_mtp": None,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "steps": e2e_steps, "pipelined": "two sets of device buffers: the upload of step k+1 overlaps "
                                              "step k, outputs read back on a third stream",
                "host_link_h2d_gbs": link_gbs,
                "link_bound_ms_per_step": h2d / (link_gbs * 1e9) * 1e3,
                "ms_per_step": e2e_s / e2e_steps * 1e3},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if not args.no_c4:
        with nvtx_range("C4 kernels"):
            line["kernels_c4"] = c4_kernels(args, ckv, dev, seed, peak)
    if not args.no_mtp:
        with nvtx_range("speculative-decoding verify steps"):
            line["kernels_mtp"] = mtp_kernels(args, ckv, dev, seed, peak)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle as o

        o.build()
        rows, secs = oracle_step(o, w5, w3, 1.0)
        line["cpu_baseline"] = {"value": rows / secs, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": "one whole step (all c128_prefill compress records + write, all "
                                          "c128_decode rows), single-threaded C, fp64 pool",
                                "seconds": secs, **cores_used()}
        n_thr = cores_used()["host_cores"] or 1
        rows_t, secs_t = oracle_step_threads(o, w5, w3, n_thr)
        line["cpu_baseline_threads"] = {"value": rows_t / secs_t, "unit": UNIT, "cores": n_thr, "kind": "oracle",
                                        "sample": "the same step, its compress records, write records and decode "
                                                  "rows split in contiguous chunks over one host thread per core",
                                        "seconds": secs_t}
    if rank == 0:
        print(json.dumps(line), flush=True)


def small_workload(name: str, seed: int) -> wl.Workload:
    """Scaled-down variants for profiler captures: same shapes and mixes, fewer
    long requests, inputs still larger than L2."""
    if name == "c128_prefill":
        return wl.c128_prefill(seed, num_long=16)
    if name == "c4_prefill":
        return wl.c4_prefill(seed, batch=16)
    return wl.NAMED[name](seed)


def bench_config(args, name, ws, rank, local):
    """One workload alone; prints one line (not the headline contract line)."""
    from compressed_kv_attention_compressplan_gb300 import build as B
    from compressed_kv_attention_compressplan_gb300 import ckv

    B.build()
    ckv.load_library()
    dev = torch.device("cuda", local)
    if name in wl.NORM_ROPE:
        return bench_norm_rope(args, name, ws, rank, ckv, dev)
    if name in wl.ONLINE:
        return bench_online(args, name, ws, rank, ckv, dev)
    if name in wl.DECODE_NORM:
        return bench_decode_norm(args, name, ws, rank, ckv, dev)
    maps = None
    if name in wl.PAGED:
        w, maps = wl.PAGED[name](args.seed + rank)
    else:
        w = small_workload(name, args.seed + rank) if args.small else wl.NAMED[name](args.seed + rank)
    flush = l2_flush_buffer(dev)
    b = algorithmic_bytes(w)
    if maps is not None:
        r = PagedPrefillRunner(ckv, w, maps, dev)
        segs = [("plan_prefill_paged", r.plan), ("pool_prefill", r.pool), ("write", r.write)]
        r.plan()
        torch.cuda.synchronize()
        nw = int(r.counts[1])  # the paged write set (page ends included), from the planner
        b["write"] = nw * (2 * w.width * elem(w.in_dtype) + 8)
        # + the extra write records, and the map reads (4 + 8 bytes) of every translated position
        b["plan"] += 8 * (nw - b["num_w"]) + 12 * (nw + 2 * b["num_c"])
        b["num_w"] = nw
        b["total"] = b["plan"] + b["pool"] + b["write"]
        main_i, main_key = 1, "pool"
    elif w.mode == "prefill":
        r = PrefillRunner(ckv, w, dev, padded=name.endswith("_mtp"))
        segs = [("plan_prefill", r.plan), ("pool_prefill", r.pool), ("write", r.write)]
        main_i, main_key = (1, "pool") if b["pool"] >= b["write"] else (2, "write")
    else:
        r = DecodeRunner(ckv, w, dev)
        segs = [("plan_decode", r.plan), ("decode", r.decode)]
        main_i, main_key = 1, "decode"
    step = StepGraph(segs)
    seg_ms, wall, _ = run_graph(step, flush, r.restore, args.steps, args.warmup, ws)
    whole = StepGraph(segs, inner_events=False)
    whole_ms, _, _ = run_graph(whole, flush, r.restore, args.steps, args.warmup, ws)
    instep = {} if args.no_instep else instep_by_difference(segs, flush, r.restore, reps=max(200, 10 * args.steps))
    if int(r.status[0]):
        raise RuntimeError(f"device status {int(r.status[0])}")
    peak, kind = peaks()
    step_ms = whole_ms[:, 0]
    main_ms = float(seg_ms[:, main_i].mean())
    gbs = b[main_key] / (main_ms * 1e-3) / 1e9
    steady = {}
    if w.mode == "prefill" and main_ms < 0.05 and not args.no_back_to_back:
        # a short main kernel (the speculative-decoding verify steps): event nodes around ~10 us of work add
        # the graph's node-to-node latency, so it is also timed back to back (back_to_back_* = the main
        # kernel, the one with more bytes; the other of pool and write under its own key)
        n = copies_for(b[main_key], dev)
        us = steady_state_us(r.steady_fns(n, main_key))
        sg = b[main_key] / (us * 1e-6) / 1e9
        floor = same_bytes_floor(b[main_key], dev, peak)
        steady = {"back_to_back_kernel": main_key, "back_to_back_us": us, "back_to_back_gbs": sg,
                  "back_to_back_frac": sg / peak, "back_to_back_copies": n, "same_bytes_floor": floor,
                  "vs_floor": min(floor["copy_us"], floor["elementwise_us"]) / us}
        other = "write" if main_key == "pool" else "pool"
        steady[f"{other}_back_to_back_us"] = steady_state_us(r.steady_fns(copies_for(b[other], dev), other))
    if w.mode == "prefill" and maps is None and not args.no_back_to_back:
        # the planner alone, back to back over copies of its inputs and outputs
        steady["plan_back_to_back_us"] = steady_state_us(r.plan_fns(16))
    if w.mode == "decode" and not args.no_back_to_back:
        n = copies_for(b["decode"], dev)
        us = steady_state_us(r.steady_fns(n))
        sg = b["decode"] / (us * 1e-6) / 1e9
        floor = same_bytes_floor(b["decode"], dev, peak)
        steady = {"back_to_back_us": us, "back_to_back_gbs": sg, "back_to_back_frac": sg / peak,
                  "back_to_back_copies": n, "same_bytes_floor": floor,
                  "vs_floor": min(floor["copy_us"], floor["elementwise_us"]) / us}
    line = {"workload": name, **w.describe(), "rows_per_step": b["rows"],
            "rows_per_s": b["rows"] / (float(step_ms.mean()) * 1e-3), "ms_per_step": float(step_ms.mean()),
            "requests_per_s": w.batch / (float(step_ms.mean()) * 1e-3),
            "step_gbs": b["total"] / (float(step_ms.mean()) * 1e-3) / 1e9,
            "segments_us": {n: float(seg_ms[:, i].mean()) * 1e3 for i, n in enumerate(step.names)},
            "segments_us_min": {n: float(seg_ms[:, i].min()) * 1e3 for i, n in enumerate(step.names)},
            "instep": instep,
            "main_kernel": step.names[main_i], "main_bytes": b[main_key], "main_gbs": gbs, "main_frac": gbs / peak,
            "peak_gbs": peak, "peak_kind": kind, "algorithmic_bytes": b, **steady}
    if rank == 0:
        print(json.dumps(line), flush=True)


def bench_norm_rope(args, name, ws, rank, ckv, dev):
    """The norm + RoPE + store step alone on one set of compressed rows; prints one line."""
    x = wl.NORM_ROPE[name](args.seed + rank)
    flush = l2_flush_buffer(dev)
    r = NormRopeRunner(ckv, x, dev)
    step = StepGraph([("norm_rope_store", r.run)])
    seg_ms, _, _ = run_graph(step, flush, r.restore, args.steps, args.warmup, ws)
    if int(r.status[0]):
        raise RuntimeError(f"device status {int(r.status[0])}")
    peak, kind = peaks()
    ms = float(seg_ms[:, 0].mean())
    b = r.algorithmic_bytes()
    gbs = b / (ms * 1e-3) / 1e9
    steady = {}
    if not args.no_back_to_back:
        n = copies_for(b, dev)
        us = steady_state_us(r.steady_fns(n))
        sg = b / (us * 1e-6) / 1e9
        floor = same_bytes_floor(b, dev, peak)
        steady = {"back_to_back_us": us, "back_to_back_gbs": sg, "back_to_back_frac": sg / peak,
                  "back_to_back_copies": n, "same_bytes_floor": floor,
                  "vs_floor": min(floor["copy_us"], floor["elementwise_us"]) / us}
    line = {"workload": name, "ratio": x.ratio, "head_dim": x.head_dim, "rope_dim": x.rope_dim,
            "records": r.records, "rows_read": r.boundary, "cache_dtype": str(x.cache_dtype).replace("torch.", ""),
            "rows_per_s": r.records / (ms * 1e-3), "us": ms * 1e3, "us_min": float(seg_ms[:, 0].min()) * 1e3,
            "main_kernel": "norm_rope_store_kernel", "main_bytes": b, "main_gbs": gbs, "main_frac": gbs / peak,
            "peak_gbs": peak, "peak_kind": kind, **steady}
    if rank == 0:
        print(json.dumps(line), flush=True)


def bench_decode_norm(args, name, ws, rank, ckv, dev):
    """The C4 decode followed by norm + RoPE + store, alone; prints one line."""
    line = decode_norm_measure(args, name, args.seed + rank, ckv, dev)
    if rank == 0:
        print(json.dumps(line), flush=True)


def decode_norm_measure(args, name, seed, ckv, dev) -> dict:
    """The C4 decode followed by norm + RoPE + store: two launches (the decode's fp32 rows, then the norm
    step over them) against the one fused launch; the planner before both.  Costs inside each step by
    difference, and each form back to back."""
    x = wl.DECODE_NORM[name](seed)
    w = x.w
    d = DecodeRunner(ckv, w, dev)
    weight, freqs, loc = x.weight.to(dev), x.freqs.to(dev), x.out_loc.to(dev)
    cache = torch.zeros(x.cache_rows, w.head_dim, dtype=x.cache_dtype, device=dev)
    flush = l2_flush_buffer(dev)

    def norm():
        ckv.norm_rope_store_decode(4, d.out[: w.batch], d.plan_d[: w.batch], weight, x.eps, freqs, loc, cache,
                                   status=d.status)

    def fused():
        ckv.compress_decode_norm_rope_store(w.head_dim, d.state, d.kv, d.ape, d.plan_d[: w.batch], weight, x.eps,
                                            freqs, loc, cache, status=d.status, **d.hints())

    reps = max(200, 10 * args.steps)
    two_seg = [("plan_decode", d.plan), ("decode", d.decode), ("norm_rope_store", norm)]
    one_seg = [("plan_decode", d.plan), ("decode_norm_rope_store", fused)]
    if args.no_instep:  # one pass of each step (profiler captures)
        for _, f in two_seg + one_seg:
            f()
        torch.cuda.synchronize()
        two = one = {}
    else:
        two = instep_by_difference(two_seg, flush, d.restore, reps)
        one = instep_by_difference(one_seg, flush, d.restore, reps)
    if int(d.status[0]):
        raise RuntimeError(f"device status {int(d.status[0])}")
    line = {"workload": name, "ratio": 4, "head_dim": w.head_dim, "batch": w.batch, "rope_dim": x.rope_dim,
            "cache_dtype": str(x.cache_dtype).replace("torch.", ""), "two_launches_instep": two,
            "fused_instep": one}
    if not args.no_back_to_back:
        d.plan()
        torch.cuda.synchronize()
        n = copies_for(algorithmic_bytes(w)["decode"], dev)
        two_fns, one_fns = [], []
        for i in range(n):
            st = d.state if i == 0 else d.pristine.clone()
            kv, pd, out, lc = d.kv.clone(), d.plan_d[: w.batch].clone(), d.out[: w.batch].clone(), loc.clone()

            def f2(st=st, kv=kv, pd=pd, out=out, lc=lc):
                ckv.compress_decode(4, w.head_dim, st, kv, d.ape, pd, w.out_dtype, out, d.status, **d.hints())
                ckv.norm_rope_store_decode(4, out, pd, weight, x.eps, freqs, lc, cache, status=d.status)

            def f1(st=st, kv=kv, pd=pd, lc=lc):
                ckv.compress_decode_norm_rope_store(w.head_dim, st, kv, d.ape, pd, weight, x.eps, freqs, lc, cache,
                                                    status=d.status, **d.hints())
            two_fns.append(f2)
            one_fns.append(f1)
        line.update({"two_launches_back_to_back_us": steady_state_us(two_fns),
                     "fused_back_to_back_us": steady_state_us(one_fns), "back_to_back_copies": n})
    del d
    torch.cuda.empty_cache()
    return line


def bench_online(args, name, ws, rank, ckv, dev):
    """A C128 step through the online state (plan + fold); prints one line."""
    if args.small and name == "c128_online_prefill":  # profiler captures: 16 long requests, still > L2
        x = wl.c128_online_prefill(args.seed + rank, num_long=16)
    else:
        x = wl.ONLINE[name](args.seed + rank)
    flush = l2_flush_buffer(dev)
    r = OnlineRunner(ckv, x, dev)
    kname = "online_prefill" if x.mode == "prefill" else "online_decode"
    step = StepGraph([("plan", r.plan), (kname, r.compute)])
    seg_ms, _, _ = run_graph(step, flush, r.restore, args.steps, args.warmup, ws)
    whole = StepGraph([("plan", r.plan), (kname, r.compute)], inner_events=False)
    whole_ms, _, _ = run_graph(whole, flush, r.restore, args.steps, args.warmup, ws)
    if int(r.status[0]):
        raise RuntimeError(f"device status {int(r.status[0])}")
    peak, kind = peaks()
    b = r.algorithmic_bytes()
    ms = float(seg_ms[:, 1].mean())
    gbs = b / (ms * 1e-3) / 1e9
    step_ms = float(whole_ms[:, 0].mean())
    steady = {}
    if x.mode == "decode" and not args.no_back_to_back:
        n = copies_for(b, dev)
        us = steady_state_us(r.steady_fns(n))
        sg = b / (us * 1e-6) / 1e9
        floor = same_bytes_floor(b, dev, peak)
        steady = {"back_to_back_us": us, "back_to_back_gbs": sg, "back_to_back_frac": sg / peak,
                  "back_to_back_copies": n, "same_bytes_floor": floor,
                  "vs_floor": min(floor["copy_us"], floor["elementwise_us"]) / us}
    line = {"workload": name, "mode": x.mode, "head_dim": x.head_dim, "batch": x.rid.numel(),
            "compress_rows": r.num_c, "rows_per_s": r.num_c / (step_ms * 1e-3), "ms_per_step": step_ms,
            "segments_us": {n: float(seg_ms[:, i].mean()) * 1e3 for i, n in enumerate(step.names)},
            "main_kernel": kname, "main_bytes": b, "main_gbs": gbs, "main_frac": gbs / peak, "peak_gbs": peak,
            "peak_kind": kind, **steady}
    if rank == 0:
        print(json.dumps(line), flush=True)


def bench_reference(args, ws, rank):
    """The oracle as it stands on the host cores, each step a bounded sample."""
    if rank != 0:
        return
    import oracle as o

    o.build()
    w5 = wl.c128_prefill(args.seed)
    w3 = wl.c128_decode(args.seed)
    frac = args.ref_fraction
    for _ in range(args.warmup):
        oracle_step(o, w5, w3, frac)
    rows_total, secs_total = 0, 0.0
    for _ in range(args.steps):
        rows, secs = oracle_step(o, w5, w3, frac)
        rows_total += rows
        secs_total += secs
    value = rows_total / secs_total
    sample = (f"each step: the first {frac:.4g} of the c128_prefill compress records (pool only) + all "
              f"c128_decode rows, single-threaded C oracle, fp64 pool")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": secs_total / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": STEP_WORKLOAD, "head_dim": 512, "in_dtype": "bf16", "out_dtype": "f32"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample,
                             **cores_used()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="step",
                    help="step (default) | all | " + " | ".join(list(wl.NAMED) + list(wl.PAGED) + list(wl.NORM_ROPE) +
                                                                 list(wl.ONLINE)))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--small", action="store_true", help="with --config: scaled-down workloads for profiling")
    ap.add_argument("--no-c4", action="store_true", help="skip the C4 kernels block of the step line")
    ap.add_argument("--no-mtp", action="store_true",
                    help="skip the speculative-decoding verify steps block of the step line")
    ap.add_argument("--no-instep", action="store_true",
                    help="skip the in-step costs by difference (200 rounds of every step variant), e.g. under ncu")
    ap.add_argument("--no-back-to-back", action="store_true",
                    help="skip the back-to-back timing of short kernels (keeps a profiler's launch list to the step)")
    ap.add_argument("--ref-fraction", type=float, default=0.125,
                    help="share of the prefill compress records the reference arm pools per step")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        bench_reference(args, ws, rank)
    elif args.config == "step":
        bench_step(args, ws, rank, local)
    else:
        names = (list(wl.NAMED) + list(wl.PAGED) + list(wl.NORM_ROPE) + list(wl.DECODE_NORM) + list(wl.ONLINE)
                 if args.config == "all"
                 else [args.config])
        for n in names:
            bench_config(args, n, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
