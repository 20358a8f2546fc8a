"""Benchmark of the PagedAttention hot path on GB300.

One step = one pass of the whole path over one batch: slot mapping of the step's
new tokens, their K/V scatter into the paged pool, and attention over the mixed
batch of chunked prefills and decodes.  Default workload: the continuous-batching
step with an 8192-token budget (8 chunked-prefill chunks of 512 queries after a
cached context uniform in [0, 3072], plus 4096 decodes with seq_lens uniform in
[256, 2048]; 32/8 heads, head_dim 128, bf16, block tables randomly permuted).
The line also carries the long-context decode KV-read bandwidth (32 requests x
32768 tokens, 64/8 heads).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload mixed|long|decode|prefix|tiny] [--no-e2e] [--no-cpu]

Inputs are drawn on the device and resident in HBM when timing starts; each step
reads ~19 GB of KV (far above the 129 MB L2), so no L2 flush is needed between
steps.  Times are CUDA events on the launching stream, max over ranks.  With
--gpus N > 1 (torchrun) every rank runs an independent replica (the path has no
exchange step) and ``value`` sums the ranks' tokens over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "decode KV-read GB/s (% of HBM peak); mixed-step tokens/sec at 1 GB300"


# DRAM traffic of the decode kernel per algorithmic byte, from one-pass ncu captures of one
# decode launch of each workload (dram__bytes_read.sum + dram__bytes_write.sum):
#   mixed step:      19.5000 GB + 36.4 MB for 19.409 GB of algorithmic bytes;
#   batched decode:  505.07 MB + 3.20 MB for 503.62 MB (decode-only: K/V loaded evict-first).
# A ratio is reported only for the workload it was measured on, and only while the
# profiled sources are unchanged.
NCU_TRAFFIC = {
    "sources": ("k_decode.cu", "ptx.cuh", "pkv_internal.cuh"),
    "sha256": "396f2627c969ab1d0cedb14ea90942fb0cd0198eab2d7ecb813eee4160b87c5a",
    "decode": {"mixed": (19.499962e9 + 36.431872e6) / 19409039536, "decode": (505.073408e6 + 3.199744e6) / 503617604},
}


def traffic_ratio(kernel: str, workload: str):
    import hashlib
    t = NCU_TRAFFIC.get(kernel, {})
    if workload not in t:
        return None
    h = hashlib.sha256()
    for f in NCU_TRAFFIC["sources"]:
        with open(os.path.join(ROOT, "paged_kv_cache_248_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return t[workload] if h.hexdigest() == NCU_TRAFFIC["sha256"] else None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------------------- work accounting

def algorithmic_bytes(w) -> dict:
    """Bytes an ideal implementation must move for one attention launch, split by
    request kind: K and V of every visible context token (unique physical tokens
    where requests share blocks), q and out, the block-table entries read."""
    eb = w.elem_bytes
    kv_tok = 2 * w.num_kv_heads * w.head_dim * eb
    q_tok = w.num_q_heads * w.head_dim * eb
    ql = w.q_lens
    dec = ql == 1
    pre = ql > 1
    L = w.seq_lens.astype(np.int64)
    bt_bytes = ((L + 15) // 16) * 4
    if w.name == "prefix":
        n_prefix = w.notes["prefix_blocks"] * 16
        dec_kv = (n_prefix + int((L - n_prefix).sum())) * kv_tok
    else:
        dec_kv = int(L[dec].sum()) * kv_tok
    pre_kv = int(L[pre].sum()) * kv_tok
    dec_io = int(dec.sum()) * 2 * q_tok + int(bt_bytes[dec].sum())
    pre_io = int(ql[pre].sum()) * 2 * q_tok + int(bt_bytes[pre].sum())
    return {"decode": dec_kv + dec_io, "decode_kv": dec_kv, "prefill": pre_kv + pre_io,
            "total": dec_kv + dec_io + pre_kv + pre_io}


def algorithmic_flops(w) -> dict:
    """4 * head_dim * Hq flops per (query, visible key) pair; causal pairs only."""
    ql = w.q_lens.astype(np.int64)
    L = w.seq_lens.astype(np.int64)
    per_pair = 4 * w.head_dim * w.num_q_heads
    dec = int(L[ql == 1].sum())
    pre = 0
    for n, l in zip(ql[ql > 1], L[ql > 1]):
        c = l - n
        pre += int(n * c + n * (n + 1) // 2)
    return {"decode": dec * per_pair, "prefill": pre * per_pair}


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- the step

class Step:
    """Device-resident inputs of one workload and the three C-ABI calls of a step."""

    def __init__(self, pkv, w, device, cascade: bool = True, fused: bool = True):
        self.pkv, self.w, self.fused = pkv, w, fused
        t = w.make_tensors(device)
        self.t = t
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)  # noqa: E731
        self.bt, self.sl, self.qsl = dev(w.block_tables), dev(w.seq_lens), dev(w.query_start_loc)
        self.slots = torch.empty(w.num_tokens, dtype=torch.int64, device=device)
        self.out = torch.empty_like(t["q"])
        self.cow = (dev(w.cow_src), dev(w.cow_dst)) if w.cow_src is not None else None
        # the shared prefix, when the workload has one, is handed over as a group hint
        self.groups = None
        if cascade and "shared_prefix_ids" in w.notes:
            pid = np.asarray(w.notes["shared_prefix_ids"], np.int32)
            self.groups = (dev(pid[None, :]), dev(np.array([pid.size], np.int32)),
                           dev(np.array([0, w.num_seqs], np.int32)), dev(np.arange(w.num_seqs, dtype=np.int32)))

    def attend(self, q, out):
        p, w, t = self.pkv, self.w, self.t
        if self.groups is not None:
            p.paged_attention_cascade(q, t["k_cache"], t["v_cache"], self.bt, self.sl, self.qsl, w.scale,
                                      w.max_query_len, w.max_seq_len, *self.groups, out=out)
        else:
            p.paged_attention(q, t["k_cache"], t["v_cache"], self.bt, self.sl, self.qsl, w.scale,
                              w.max_query_len, w.max_seq_len, out=out)

    def write_and_attend(self, q, k_new, v_new, out, cow=None):
        """The step's calls after its inputs are on the device: the copy-on-write pairs
        ``cow`` (src, dst) if any, slot mapping, scatter and attention -- all in one call
        when fused."""
        p, w, t = self.pkv, self.w, self.t
        if self.fused:
            p.paged_attention_step(q, k_new, v_new, t["k_cache"], t["v_cache"], self.bt, self.sl, self.qsl, w.scale,
                                   w.max_query_len, w.max_seq_len, prefix_groups=self.groups, out=out, cow=cow)
        else:
            if cow:
                p.pkv_copy_blocks(cow[0], cow[1], t["k_cache"], t["v_cache"])
            p.pkv_slot_mapping(self.bt, self.sl, self.qsl, w.num_tokens, out=self.slots)
            p.pkv_write(k_new, v_new, self.slots, t["k_cache"], t["v_cache"])
            self.attend(q, out)

    def run(self):
        t = self.t
        self.write_and_attend(t["q"], t["k_new"], t["v_new"], self.out, cow=self.cow)

    def attention_only(self):
        self.attend(self.t["q"], self.out)


class E2EStep:
    """The same step from pinned HOST buffers: H2D of the step's inputs (q, new K/V,
    block tables, lengths, copy-on-write pairs), the library calls, D2H of the
    attention output."""

    def __init__(self, step: Step):
        self.s = step
        t = step.t
        pin = lambda x: x.detach().to("cpu").pin_memory()  # noqa: E731
        self.h = {k: pin(t[k]) for k in ("q", "k_new", "v_new")}
        self.h_bt, self.h_sl, self.h_qsl = pin(step.bt), pin(step.sl), pin(step.qsl)
        self.h_cow = tuple(pin(x) for x in step.cow) if step.cow is not None else ()
        self.h_out = torch.empty(t["q"].shape, dtype=t["q"].dtype).pin_memory()
        self.d = {k: torch.empty_like(t[k]) for k in ("q", "k_new", "v_new")}
        self.h2d = sum(x.numel() * x.element_size() for x in list(self.h.values()) + [self.h_bt, self.h_sl,
                                                                                           self.h_qsl] +
                       list(self.h_cow))
        self.d2h = self.h_out.numel() * self.h_out.element_size()

    def run(self):
        s, p, w, t = self.s, self.s.pkv, self.s.w, self.s.t
        for k in self.d:
            self.d[k].copy_(self.h[k], non_blocking=True)
        s.bt.copy_(self.h_bt, non_blocking=True)
        s.sl.copy_(self.h_sl, non_blocking=True)
        s.qsl.copy_(self.h_qsl, non_blocking=True)
        if s.cow is not None:
            for dst, src in zip(s.cow, self.h_cow):
                dst.copy_(src, non_blocking=True)
        s.write_and_attend(self.d["q"], self.d["k_new"], self.d["v_new"], s.out, cow=s.cow)
        self.h_out.copy_(s.out, non_blocking=True)


class E2EPipelined:
    """The end-to-end step as a serving loop would run it: two device copies of the
    step's inputs, host-to-device copies of step i + 1 on a copy stream while step i
    computes, and each step's output read back on the copy stream once it is done.
    Every step still copies its own inputs in and its own output out inside the timed
    region; only their overlap with compute differs from E2EStep."""

    def __init__(self, step: Step):
        self.s = step
        self.ser = E2EStep(step)  # pinned host buffers and byte counts
        t = step.t
        self.sets = []
        for _ in range(2):
            d = {k: torch.empty_like(t[k]) for k in ("q", "k_new", "v_new")}
            d["bt"], d["sl"], d["qsl"] = (torch.empty_like(step.bt), torch.empty_like(step.sl),
                                          torch.empty_like(step.qsl))
            d["out"] = torch.empty_like(t["q"])
            d["cow"] = tuple(torch.empty_like(x) for x in step.cow) if step.cow is not None else ()
            self.sets.append(d)
        self.h_out = [torch.empty(t["q"].shape, dtype=t["q"].dtype).pin_memory() for _ in range(2)]
        self.copy = torch.cuda.Stream()
        self.h2d, self.d2h = self.ser.h2d, self.ser.d2h

    def _h2d(self, d):
        e = self.ser
        for k in ("q", "k_new", "v_new"):
            d[k].copy_(e.h[k], non_blocking=True)
        d["bt"].copy_(e.h_bt, non_blocking=True)
        d["sl"].copy_(e.h_sl, non_blocking=True)
        d["qsl"].copy_(e.h_qsl, non_blocking=True)
        for dst, src in zip(d["cow"], e.h_cow):
            dst.copy_(src, non_blocking=True)

    def _compute(self, d):
        s, p, w, t = self.s, self.s.pkv, self.s.w, self.s.t
        cow = d["cow"] if d["cow"] else None
        if s.fused:
            p.paged_attention_step(d["q"], d["k_new"], d["v_new"], t["k_cache"], t["v_cache"], d["bt"], d["sl"],
                                   d["qsl"], w.scale, w.max_query_len, w.max_seq_len, prefix_groups=s.groups,
                                   out=d["out"], cow=cow)
        else:
            if cow:
                p.pkv_copy_blocks(cow[0], cow[1], t["k_cache"], t["v_cache"])
            p.pkv_slot_mapping(d["bt"], d["sl"], d["qsl"], w.num_tokens, out=s.slots)
            p.pkv_write(d["k_new"], d["v_new"], s.slots, t["k_cache"], t["v_cache"])
            p.paged_attention(d["q"], t["k_cache"], t["v_cache"], d["bt"], d["sl"], d["qsl"], w.scale,
                              w.max_query_len, w.max_seq_len, out=d["out"])

    def time(self, steps: int, warmup: int) -> float:
        comp = torch.cuda.current_stream()
        for rep in range(2):  # one warm-up pass, then the timed one
            n = warmup if rep == 0 else steps
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(comp)
            h2d_done = [torch.cuda.Event(), torch.cuda.Event()]
            comp_done = [torch.cuda.Event(), torch.cuda.Event()]
            self.copy.wait_event(e0)
            with torch.cuda.stream(self.copy):
                self._h2d(self.sets[0])
                h2d_done[0].record(self.copy)
            for i in range(n):
                b = i & 1
                comp.wait_event(h2d_done[b])
                self._compute(self.sets[b])
                comp_done[b].record(comp)
                with torch.cuda.stream(self.copy):
                    if i + 1 < n:  # next step's inputs, once the step that last used that set is done
                        if i >= 1:
                            self.copy.wait_event(comp_done[b ^ 1])
                        self._h2d(self.sets[b ^ 1])
                        h2d_done[b ^ 1].record(self.copy)
                    self.copy.wait_event(comp_done[b])
                    self.h_out[b].copy_(self.sets[b]["out"], non_blocking=True)
            comp.wait_stream(self.copy)
            e1.record(comp)
            torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: every rank must call it (a collective when world > 1)."""
    if world <= 1:
        return ms
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's step time."""
    return tokens_per_rank * world / (ms_max / 1e3)


def timed(fn, steps, warmup, barrier=None):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    return e0.elapsed_time(e1) / steps


# ----------------------------------------------------------------------------- CPU oracle sample

def _to_bits(x):
    return (x.view(torch.int16) if x.dtype == torch.bfloat16 else x).cpu().numpy().copy()


def host_batch(w, t_gpu, seq_ids):
    """Requests ``seq_ids`` with only their blocks, copied to the host (block ids
    renumbered), as the oracle reads them: (k_cache, v_cache, q, k_new, v_new,
    block_tables, seq_lens, query_start_loc, copy-on-write pairs or None)."""
    seq_ids = np.asarray(seq_ids, np.int64)
    qsl = w.query_start_loc
    bt = w.block_tables[seq_ids]
    ids = [bt[bt >= 0]]
    if w.cow_src is not None:   # the sources of the requests' copy-on-write pairs too
        ids.append(w.cow_src[seq_ids])
    used = np.unique(np.concatenate(ids))
    remap = np.full(w.num_blocks, -1, np.int32)
    remap[used] = np.arange(len(used), dtype=np.int32)
    cow = None if w.cow_src is None else (remap[w.cow_src[seq_ids]], remap[w.cow_dst[seq_ids]])
    bt2 = np.where(bt >= 0, remap[np.maximum(bt, 0)], -1).astype(np.int32)
    idx = torch.from_numpy(used.astype(np.int64)).to(t_gpu["k_cache"].device)
    kc = _to_bits(t_gpu["k_cache"].index_select(0, idx))
    vc = _to_bits(t_gpu["v_cache"].index_select(0, idx))
    rows = np.concatenate([np.arange(qsl[i], qsl[i + 1]) for i in seq_ids]).astype(np.int64)
    ridx = torch.from_numpy(rows).to(t_gpu["q"].device)
    q, kn, vn = (_to_bits(t_gpu[k].index_select(0, ridx)) for k in ("q", "k_new", "v_new"))
    qsl2 = np.concatenate([[0], np.cumsum(w.q_lens[seq_ids])]).astype(np.int32)
    return kc, vc, q, kn, vn, bt2, w.seq_lens[seq_ids].copy(), qsl2, cow


def row_macs(w, rows=None) -> int:
    """Multiply-adds of attention for the given query rows (default all): 2 * head_dim *
    Hq per (row, visible key) pair."""
    qsl, L = w.query_start_loc, w.seq_lens.astype(np.int64)
    req = np.searchsorted(qsl, np.arange(w.num_tokens), side="right") - 1
    pos = L[req] - (qsl[req + 1] - np.arange(w.num_tokens))   # absolute position of each row
    vis = pos + 1
    if rows is not None:
        vis = vis[np.asarray(rows)]
    return int(vis.sum()) * 2 * w.head_dim * w.num_q_heads


def cpu_sample(w, t_gpu, target_s: float = 12.0, seed: int = 0):
    """Time the oracle (as it stands) on a bounded sample of the workload: a sub-batch
    of requests (all chunks, a subset of decodes) with sampled query rows; returns
    (tokens/s, description, threads)."""
    import oracle
    rng = np.random.default_rng(seed)
    ql = w.q_lens
    dec_ids = np.nonzero(ql == 1)[0]
    pre_ids = np.nonzero(ql > 1)[0]

    def build(n_dec, rows_per_chunk):
        pick_dec = rng.choice(dec_ids, size=min(n_dec, len(dec_ids)), replace=False) if len(dec_ids) else []
        seq_ids = np.concatenate([pre_ids, np.sort(pick_dec)]).astype(np.int64)
        kc, vc, q, kn, vn, bt2, L, qsl2, _ = host_batch(w, t_gpu, seq_ids)
        q_lens = ql[seq_ids]
        sel = []
        for j in range(len(seq_ids)):
            n = int(q_lens[j])
            if n == 1:
                sel.append(qsl2[j])
            else:
                k = min(n, rows_per_chunk)
                sel.extend(qsl2[j] + np.sort(rng.choice(n, size=k, replace=False)))
        sel = np.asarray(sel, np.int64)
        return kc, vc, q, kn, vn, bt2, L, qsl2, sel

    def run(args):
        kc, vc, q, kn, vn, bt2, L, qsl2, sel = args
        t0 = time.perf_counter()
        slots = oracle.slot_mapping(bt2, L, qsl2)
        oracle.write(kn, vn, slots, kc, vc)
        oracle.attention(q, kc, vc, bt2, L, qsl2, w.scale, rows=sel)
        return time.perf_counter() - t0, len(sel)

    n_dec0, rpc0 = 32, 4
    dt, n = run(build(n_dec0, rpc0))
    scale = max(1.0, target_s / max(dt, 1e-3))
    n_dec, rpc = int(n_dec0 * scale), int(rpc0 * scale)   # capped by the workload's own size
    args = build(n_dec, rpc)
    dt, n = run(args)
    n_pre_rows = int(sum(min(int(x), rpc) for x in w.q_lens[w.q_lens > 1]))
    desc = (f"oracle step (slot mapping + write + attention) on {n} query rows: "
            f"{n - n_pre_rows} decode requests and {n_pre_rows} sampled prefill rows of the "
            f"{w.name} workload; wall {dt:.2f} s")
    return n / dt, desc, oracle.max_threads(), dt


def cpu_one_core(w, t_gpu, max_rows: int | None = None, seed: int = 0) -> dict:
    """The oracle on ONE thread.  Small workloads: the whole step (copy-on-write where
    the workload has it, slot mapping, write, attention of every row).  Large ones
    (``max_rows`` set): the step over a random subset of rows, timed, then
    extrapolated to the whole step by multiply-adds, and labelled so."""
    import oracle
    seq_ids = np.arange(w.num_seqs)
    if max_rows is not None and w.num_tokens > max_rows:
        rng = np.random.default_rng(seed)
        rows = np.sort(rng.choice(w.num_tokens, size=max_rows, replace=False))
        req = np.unique(np.searchsorted(w.query_start_loc, rows, side="right") - 1)
        seq_ids = req
    kc, vc, q, kn, vn, bt2, L, qsl2, cow = host_batch(w, t_gpu, seq_ids)
    full_rows = np.concatenate([np.arange(w.query_start_loc[i], w.query_start_loc[i + 1]) for i in seq_ids])
    if max_rows is not None and w.num_tokens > max_rows:
        keep = np.isin(full_rows, rows)
        sel = np.nonzero(keep)[0].astype(np.int64)
        timed_macs = row_macs(w, full_rows[keep])
    else:
        sel = None
        timed_macs = row_macs(w)
    t0 = time.perf_counter()
    if cow is not None:   # the requests' copy-on-write pairs, renumbered into the host batch
        oracle.copy_blocks(cow[0], cow[1], kc, vc)
    slots = oracle.slot_mapping(bt2, L, qsl2)
    oracle.write(kn, vn, slots, kc, vc)
    oracle.attention(q, kc, vc, bt2, L, qsl2, w.scale, rows=sel, n_threads=1)
    dt = time.perf_counter() - t0
    total_macs = row_macs(w)
    est = dt * total_macs / timed_macs
    kv = algorithmic_bytes(w)["decode_kv"] + algorithmic_bytes(w)["prefill"]
    out = {"s_per_step": est, "tokens_per_s": w.num_tokens / est, "kv_gbs": kv / est / 1e9, "threads": 1}
    if sel is None:
        out["how"] = "whole step timed"
    else:
        out["how"] = (f"extrapolated: {len(sel)} of {w.num_tokens} query rows timed ({dt:.2f} s, "
                      f"{100.0 * timed_macs / total_macs:.2f} % of the multiply-adds), scaled by multiply-adds")
    return out


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mixed", choices=list(wl.NAMES))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-decode-line", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="leave out the tiny, decode and prefix lines and the one-core oracle times")
    ap.add_argument("--no-cascade", action="store_true",
                    help="attend a shared prefix per request instead of once per group")
    ap.add_argument("--unfused", action="store_true",
                    help="separate slot-mapping, write and attention calls instead of paged_attention_step")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    barrier = None
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        barrier = dist.barrier

    w = wl.make(args.workload)
    if args.impl == "reference":
        return reference_arm(args, w, rank, world)

    import paged_kv_cache_248_gb300 as pkv
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    pk = peaks()
    step = Step(pkv, w, device, cascade=not args.no_cascade, fused=not args.unfused)
    work_b = algorithmic_bytes(w)
    work_f = algorithmic_flops(w)

    # ---- timed region: K steps as a caller runs them (no launch events), then the same
    # K steps again with the library recording CUDA events around each of its launches
    # on the launching stream: the per-kernel times and the launch count come from that
    # second region, the step time from the first
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ms = timed(step.run, args.steps, 0, barrier)
        pkv.pkv_trace_enable(True)
        pkv.pkv_trace_read()
        ms_traced = timed(step.run, args.steps, 0, barrier)
        trace = pkv.pkv_trace_read()
        pkv.pkv_trace_enable(False)
    st = pkv.pkv_get_last_error()
    if st != 0:
        raise RuntimeError(f"device error during bench: {pkv.status_string(st)}")
    clocks = clk.summary()

    ms_max = max_over_ranks(ms, world, device)
    tokens = w.num_tokens * world
    value = job_throughput(w.num_tokens, world, ms_max)

    launches = sum(n for n, _ in trace.values())
    kernel_ms = {k: (n, t) for k, (n, t) in trace.items() if n}
    # dominant kernel of the step and its roofline
    dom = max(kernel_ms, key=lambda k: kernel_ms[k][1])
    n_dom, t_dom = kernel_ms[dom]
    if "cascade" in kernel_ms:
        # shared-prefix groups: the cascade kernel reads the prefix, the decode kernel each
        # member's own keys, the merge joins them; the roofline covers that whole pass
        parts = [k for k in ("cascade", "decode", "merge") if k in kernel_ms]
        dom = "+".join(parts)
        n_dom, t_dom = kernel_ms["decode"][0], sum(kernel_ms[k][1] for k in parts)
    per_launch_ms = t_dom / n_dom
    if dom == "prefill":
        # a launch of ~0.1 ms at full clock: the burst GEMM peak is its denominator; the
        # power-capped sustained peak is reported beside it
        flops = work_f["prefill"]
        ach = flops / (per_launch_ms / 1e3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": ach / pk["bf16_tflops"], "traffic": None,
                "frac_of_sustained": ach / pk["bf16_tflops_sustained"]}
    else:
        b = work_b["decode"] if dom.startswith(("decode", "cascade")) else work_b["total"]
        ach = b / (per_launch_ms / 1e3) / 1e9
        ratio = traffic_ratio(dom, w.name)
        roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": ach / pk["hbm_gbs"], "traffic": ratio * b if ratio else None,
                "algorithmic_bytes_per_launch": b}
    roof["peak_source"] = pk["source"]

    res = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded N(0,1), shapes of the workload)",
        "config": {"workload": f"{w.name}: {describe(w)}", "global_batch_tokens": tokens,
                   "l2": "no flush: each step reads %.1f GB of KV, far above the 129 MB L2" % (
                       work_b["total"] / 1e9),
                   "parallelism": "replicas only" if world > 1 else "single GPU"},
        "clocks": clocks, "roofline": roof, "gpu_launches": launches,
        "ms_per_step_with_launch_events": max_over_ranks(ms_traced, world, device),
        "kernels": {k: {"launches": n, "ms_total": t, "ms_per_launch": t / n} for k, (n, t) in kernel_ms.items()},
        "work": {"bytes": work_b, "flops": work_f},
    }

    # the same step captured once into a CUDA graph and replayed (one launch per step)
    try:
        gs = torch.cuda.Stream()
        gs.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(gs):
            step.run()
        gs.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            step.run()
        ms_graph = timed(graph.replay, args.steps, args.warmup, barrier)
        if pkv.pkv_get_last_error() != 0:
            raise RuntimeError("device error during graph replay")
        ms_graph = max_over_ranks(ms_graph, world, device)
        res["graph_replay"] = {"ms_per_step": ms_graph, "value": job_throughput(w.num_tokens, world, ms_graph),
                               "unit": "tokens/s"}
        del graph
    except RuntimeError as e:  # capture not possible here: report why, keep the eager numbers
        res["graph_replay"] = {"error": str(e)[:200]}

    if not args.no_e2e:
        e2e = E2EStep(step)
        ms_serial = timed(e2e.run, max(3, args.steps // 2), 3, barrier)
        pipe = E2EPipelined(step)
        if barrier:
            barrier()
        # the same K steps as the device-timed region: the pipeline's fill (the first
        # step's inputs) and drain (the last step's output) are counted once per K steps
        ms_e2e = pipe.time(max(3, args.steps), 3)
        if barrier:
            barrier()
        ms_e2e = max_over_ranks(ms_e2e, world, device)
        res["e2e"] = {"value": job_throughput(w.num_tokens, world, ms_e2e), "unit": "tokens/s",
                      "h2d_bytes_per_step": e2e.h2d, "d2h_bytes_per_step": e2e.d2h, "ms_per_step": ms_e2e,
                      "io": "inputs of step i + 1 copied on a second stream while step i computes; "
                            "fill and drain included, over the same steps as value",
                      "serial_ms_per_step": ms_serial}
        if pkv.pkv_get_last_error() != 0:
            raise RuntimeError("device error during e2e")
        del e2e

    if not args.no_decode_line and args.workload == "mixed":
        res["decode_kv_read"] = decode_line(pkv, device, pk, args)

    if not args.no_configs and args.workload == "mixed":
        res["configs"] = config_lines(pkv, device, pk, args)

    if not args.no_cpu and rank == 0 and world == 1:
        v, desc, cores, dt = cpu_sample(w, step.t)
        res["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc}
        if args.workload == "mixed" and not args.no_configs:
            res["cpu_baseline"]["one_core"] = one_core_lines(pkv, device, step)

    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def decode_line(pkv, device, pk, args) -> dict:
    """KV-read bandwidth of the long-context decode (32 x 32768, 64/8 heads): the
    paged_attention launch alone, K timed launches after warm-up."""
    w = wl.make("long")
    s = Step(pkv, w, device)
    s.run()
    ms = timed(s.attention_only, max(10, args.steps), args.warmup)
    pkv.pkv_trace_enable(True)   # per-kernel times from a second, traced pass
    pkv.pkv_trace_read()
    timed(s.attention_only, max(10, args.steps), 0)
    trace = pkv.pkv_trace_read()
    pkv.pkv_trace_enable(False)
    if pkv.pkv_get_last_error() != 0:
        raise RuntimeError("device error in decode line")
    b = algorithmic_bytes(w)
    kv = b["decode_kv"]
    gbs = kv / (ms / 1e3) / 1e9
    ker = {k: {"launches": n, "ms_per_launch": t / n} for k, (n, t) in trace.items() if n}
    dom = max(ker, key=lambda k: ker[k]["ms_per_launch"] * ker[k]["launches"])
    kgbs = b["decode"] / (ker[dom]["ms_per_launch"] / 1e3) / 1e9
    out = {"workload": f"long: {describe(w)}", "kv_bytes": kv, "ms_per_call": ms, "kv_gbs": gbs,
           "frac_of_hbm": gbs / pk["hbm_gbs"], "peak_gbs": pk["hbm_gbs"], "peak_source": pk["source"],
           "kernel": dom, "kernel_gbs": kgbs, "kernel_frac": kgbs / pk["hbm_gbs"], "kernels": ker}
    del s
    torch.cuda.empty_cache()
    return out


def flushed_time(fn, steps: int, warmup: int, flush: torch.Tensor) -> float:
    """Mean device time of ``fn`` over ``steps`` calls, each bracketed by CUDA events on
    the launching stream, with a write of ``flush`` (larger than L2) before every
    call and outside its events, so that no call finds the previous one's data in L2."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    evs = []
    for _ in range(steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    return float(np.mean([a.elapsed_time(b) for a, b in evs]))


def config_lines(pkv, device, pk, args) -> dict:
    """The three smaller named workloads, each one whole step as the default line runs
    it (copy-on-write where the workload has it, then paged_attention_step; the shared
    prefix as a group hint), L2 flushed before every timed step:
      tiny   -- microseconds per step (launch-latency bound);
      decode -- KV GB/s and the fraction of the HBM peak the step and its decode
                kernel reach;
      prefix -- logical KV GB/s (the shared prefix counted once per request, so it
                may exceed HBM), the fraction of the HBM peak on the unique bytes the
                step must move, and the copy-on-write kernel's GB/s."""
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)  # 256 MB > 129 MB L2
    steps = max(10, args.steps)
    out = {}
    for name in ("tiny", "decode", "prefix"):
        w = wl.make(name)
        s = Step(pkv, w, device)
        ms = flushed_time(s.run, steps, args.warmup, flush)
        # decode and prefix steps read more than L2 holds, so back-to-back steps are a valid
        # timing too (L2 then keeps a little of the previous step's data)
        ms_b2b = timed(s.run, steps, 0) if name != "tiny" else None
        pkv.pkv_trace_enable(True)   # per-kernel times from a second, traced pass
        pkv.pkv_trace_read()
        flushed_time(s.run, steps, 0, flush)
        trace = pkv.pkv_trace_read()
        pkv.pkv_trace_enable(False)
        if pkv.pkv_get_last_error() != 0:
            raise RuntimeError(f"device error in the {name} line")
        ker = {k: {"launches": n, "ms_per_launch": t / n} for k, (n, t) in trace.items() if n}
        b = algorithmic_bytes(w)
        kv_tok = 2 * w.num_kv_heads * w.head_dim * w.elem_bytes
        new_tok = w.num_tokens * 2 * kv_tok          # read the new rows, write them into their slots
        line = {"workload": f"{name}: {describe(w)}", "ms_per_step": ms, "steps": steps,
                "l2": "flushed (256 MB write) before every step", "kernels": ker}
        if ms_b2b is not None:
            line["ms_per_step_back_to_back"] = ms_b2b
        if name == "tiny":
            line["us_per_step"] = ms * 1e3
            line["bound"] = "launch latency"
        elif name == "decode":
            step_bytes = b["total"] + new_tok
            line.update({"kv_bytes": b["decode_kv"], "kv_gbs": b["decode_kv"] / (ms / 1e3) / 1e9,
                         "step_bytes": step_bytes, "step_frac_of_hbm": step_bytes / (ms / 1e3) / 1e9 / pk["hbm_gbs"],
                         "step_frac_of_hbm_back_to_back": step_bytes / (ms_b2b / 1e3) / 1e9 / pk["hbm_gbs"],
                         "roofline_ms": step_bytes / (pk["hbm_gbs"] * 1e9) * 1e3})
            if "decode" in ker:
                kms = ker["decode"]["ms_per_launch"]
                line["decode_kernel_frac_of_hbm"] = b["decode"] / (kms / 1e3) / 1e9 / pk["hbm_gbs"]
        else:
            logical = int(w.seq_lens.astype(np.int64).sum()) * kv_tok
            n_cow = int(w.cow_src.shape[0])
            blk = w.num_kv_heads * 16 * w.head_dim * w.elem_bytes
            cow_bytes = n_cow * 2 * 2 * blk          # read and write K and V of each pair
            step_bytes = b["total"] + new_tok + cow_bytes
            line.update({"logical_kv_bytes": logical, "logical_kv_gbs": logical / (ms / 1e3) / 1e9,
                         "unique_step_bytes": step_bytes,
                         "unique_frac_of_hbm": step_bytes / (ms / 1e3) / 1e9 / pk["hbm_gbs"],
                         "unique_frac_of_hbm_back_to_back": step_bytes / (ms_b2b / 1e3) / 1e9 / pk["hbm_gbs"],
                         "roofline_ms": step_bytes / (pk["hbm_gbs"] * 1e9) * 1e3})
            if "copy_blocks" in ker:
                cms = ker["copy_blocks"]["ms_per_launch"]
                line["cow"] = {"pairs": n_cow, "bytes": cow_bytes, "ms_per_launch": cms,
                               "gbs": cow_bytes / (cms / 1e3) / 1e9,
                               "frac_of_hbm": cow_bytes / (cms / 1e3) / 1e9 / pk["hbm_gbs"]}
        line["peak_gbs"], line["peak_source"] = pk["hbm_gbs"], pk["source"]
        out[name] = line
        del s
        torch.cuda.empty_cache()
    del flush
    return out


def one_core_lines(pkv, device, mixed_step) -> dict:
    """The oracle on one thread for every named workload (section "CPU oracle timing"
    of the measurement plan): whole steps for tiny, decode and prefix; a timed subset
    extrapolated by multiply-adds for mixed and long."""
    res = {}
    for name in ("tiny", "decode", "prefix", "long"):
        w = wl.make(name)
        t = w.make_tensors(device)
        res[name] = cpu_one_core(w, t, max_rows=4 if name == "long" else None)
        del t
        torch.cuda.empty_cache()
    res["mixed"] = cpu_one_core(mixed_step.w, mixed_step.t, max_rows=256)
    return res


def describe(w) -> str:
    return (f"{w.num_seqs} requests, {w.num_tokens} query tokens, max context {w.max_seq_len}, "
            f"{w.num_q_heads}/{w.num_kv_heads} heads, head_dim {w.head_dim}, {w.dtype}, pool {w.num_blocks} blocks")


def reference_arm(args, w, rank, world):
    """The oracle (CPU, fp64) timed as it stands on this host's cores: each step is a
    bounded sample of the same workload.  Rank 0 only."""
    if rank != 0:
        return
    import oracle
    torch.manual_seed(0)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = w.make_tensors(dev)
    rates, descs, dts = [], [], []
    for i in range(args.warmup + args.steps):
        v, desc, cores, dt = cpu_sample(w, t, target_s=4.0, seed=i)
        if i >= args.warmup:
            rates.append(v)
            dts.append(dt)
            descs.append(desc)
    value = float(np.mean(rates))
    res = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": float(np.mean(dts)) * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded N(0,1), shapes of the workload)",
           "config": {"workload": f"{w.name}: {describe(w)}", "parallelism": "host cores"},
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.max_threads(), "kind": "oracle",
                            "sample": descs[-1]},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res))


if __name__ == "__main__":
    main()
