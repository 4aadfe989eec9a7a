#!/usr/bin/env python3
"""Benchmark of one step of the paged INT8 KV-cache hot path on GB300.

A step is one pass of the whole path over one batch: kv_cache_append of the
step's new K/V rows (quantize + scatter), then split-KV paged attention and
its log-sum-exp combine. Inputs are seeded and synthetic (see
quantized_paged_kv_cache_gb300/workloads.py); the cache history is appended
once, untimed, before the timed region.

Prints one JSON line. `value` is algorithmic bytes per second (int8 K/V codes
+ fp32 group scales + bf16 Q + bf16 O of the attention, plus the append's bf16
reads and int8/fp32 writes) over all ranks; `us_per_call` is the step time.
`--impl reference` times the fp64 CPU oracle on the same workload instead.

Multi-GPU: every rank runs an independent replica (no data-path collective);
the step time is the max over ranks and `value` sums the ranks' bytes.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged INT8-KV decode attention: µs/call and KV GB/s as % of GB300 HBM peak"
L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="mix",
                    help="mix (default: the largest single-GPU configuration, 8 x 1,024-row append + C8 x T4 "
                         "attention at 131,072) | tiny | c1_decode | c8_verify | long_context | c8_decode | c1_rk8v4 "
                         "| c1_i8f16 | c8_i8f16 | mix_prefill | prefill_32k")
    ap.add_argument("--kernel", choices=["mma", "simt"], default="mma", help="attention kernel of our arm")
    ap.add_argument("--num-ctas", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--out", default=None, help="also append the JSON line to this file")
    ap.add_argument("--profile", action="store_true",
                    help="short run for a profiler: no load pre-roll, clock sampling, e2e or CPU baseline")
    return ap.parse_args()


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def _code_only(text: str) -> str:
    """C++ source without comments and blank lines (a comment edit does not
    change the kernel the counters were taken on)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def source_hash() -> str:
    """Hash of the code of the decode split kernels' and the prefill kernel's
    sources and the headers they include (the kernels whose ncu traffic
    profiles/ncu_traffic.json records), comments excluded."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "quantized_paged_kv_cache_gb300", "csrc")
    for fn in sorted(os.listdir(d)):
        if fn.startswith(("nk_decode", "nk_prefill")) or fn in ("nk_common.cuh", "nk_ptx.cuh"):
            with open(os.path.join(d, fn), encoding="utf-8") as f:
                h.update(fn.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, kernel: str):
    """dram read+write bytes per launch of the attention kernel from the committed
    ncu summary, only if it was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(f"{workload}/{kernel}")
    if not ent or ent.get("source_sha") != source_hash():
        return None
    return ent.get("traffic_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle samples over the load window around the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons), "window": "load window containing the timed region"}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def setup_gpu(w, device, replicas, num_ctas, kernel):
    import torch

    import quantized_paged_kv_cache_gb300 as nk
    from quantized_paged_kv_cache_gb300 import workloads as wl

    bt = wl.block_table(w).to(device)
    ctx = torch.tensor(w.ctx_lens, dtype=torch.int32, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    append = {"rk8v4": nk.rk8v4_append, "i8f16": nk.i8f16_append, "bf16": nk.bf16kv_append}.get(w.fmt, nk.kv_append)
    base = nk.KVPool.empty(w.num_pages, w.P, w.Hkv, w.D, device=device, fill=0, fmt=w.fmt)
    hist, _ = wl.history_and_step(w)
    for b in range(w.B):
        pos = 0
        while pos < hist[b]:
            n = min(16384, hist[b] - pos)
            k, v = wl.kv_rows(w, b, pos, n, device=device)
            append(base, bt[b:b + 1].contiguous(), torch.tensor([pos], dtype=torch.int32, device=device),
                   torch.tensor([0, n], dtype=torch.int32, device=device), k, v, status=status)
            pos += n
    pools = [base] + [nk.KVPool(base.storage.clone(), w.num_pages, w.P, w.Hkv, w.D, w.fmt)
                      for _ in range(replicas - 1)]
    starts, _ = wl.history_and_step(w)
    k, v, sp, cu = wl.append_batch(w, starts, [w.append_len] * w.B, device=device)
    # copies of the append's bf16 input, rotated step by step like the pool,
    # so that the append reads rows that are not in L2 (when they are large
    # enough for that to matter)
    in_bytes = 2 * k.numel() * k.element_size()
    n_in = 1 if in_bytes >= 2 * L2_BYTES or in_bytes < 2 ** 20 else min(16, int(-(-2 * L2_BYTES // in_bytes)) + 1)
    ks = [k] + [k.clone() for _ in range(n_in - 1)]
    vs = [v] + [v.clone() for _ in range(n_in - 1)]
    q = wl.queries(w, device=device)
    nct = num_ctas
    # the chunked prefill takes no workspace
    ws_bytes = 256 if is_prefill(w) else nk.decode_workspace_bytes(w.B, w.T, w.Hq, w.Hkv, w.D, nct)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
    out = torch.empty_like(q)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"history append flagged device status {int(status.item())}")
    return dict(bt=bt, ctx=ctx, status=status, pools=pools, k=k, v=v, ks=ks, vs=vs, n_in=n_in, sp=sp.to(device),
                cu=cu.to(device), q=q, ws=ws, out=out, nct=nct, kernel=kernel, append=append)


def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's time: with one replica per rank, the job's time."""
    if world <= 1:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_gbs(step_bytes: int, ms: float, world: int) -> float:
    """Whole-job throughput: every rank moves step_bytes per step."""
    return step_bytes * world / (ms * 1e-3) / 1e9


def is_prefill(w) -> bool:
    """A chunked-prefill workload (T beyond the decode / verify widths)."""
    return w.T > 16


def attention_call(args, w):
    """The attention entry point the run times: the tensor-core or CUDA-core
    kernel of an INT8 pool, the kernels of the other formats, or the chunked
    prefill (which takes no split count or workspace)."""
    import quantized_paged_kv_cache_gb300 as nk

    if is_prefill(w):
        def prefill(pool, q, bt, ctx, sm_scale, max_ctx, num_ctas=0, workspace=None, out=None, status=None,
                    stream=None):
            return nk.paged_prefill_attn(pool, q, bt, ctx, sm_scale, max_ctx, out=out, status=status, stream=stream)
        return prefill

    if w.fmt != "int8":
        return {"rk8v4": nk.rk8v4_decode_attn, "i8f16": nk.i8f16_decode_attn, "bf16": nk.bf16kv_decode_attn}[w.fmt]
    return nk.paged_decode_attn if args.kernel == "mma" else nk.paged_decode_attn_simt


def one_call_step(args, w) -> bool:
    """Whether a step runs as one nk_decode_step call (INT8 pool, tensor-core decode kernels)."""
    return w.fmt == "int8" and args.kernel == "mma" and not is_prefill(w)


def run_ours(args, w, rank, world, device):
    import torch

    import quantized_paged_kv_cache_gb300 as nk

    sizer = {"rk8v4": nk.rk8v4_pool_bytes, "i8f16": nk.i8f16_pool_bytes, "bf16": nk.bf16kv_pool_bytes}.get(
        w.fmt, nk.kv_pool_bytes)
    pool_bytes = sizer(w.num_pages, w.P, w.Hkv, w.D)
    replicas = 1 if pool_bytes >= 2 * L2_BYTES else int(-(-2 * L2_BYTES // pool_bytes)) + 1
    S = setup_gpu(w, device, replicas, args.num_ctas, args.kernel)
    dec = attention_call(args, w)
    stream = torch.cuda.current_stream()

    def step(i, what="step"):
        pool = S["pools"][i % replicas]
        k, v = S["ks"][i % S["n_in"]], S["vs"][i % S["n_in"]]
        if what == "step" and one_call_step(args, w):  # append + attention in one call
            nk.decode_step(pool, S["bt"], S["sp"], S["cu"], k, v, S["q"], S["ctx"], w.sm_scale, w.max_ctx,
                           num_ctas=S["nct"], workspace=S["ws"], out=S["out"], status=S["status"], stream=stream)
            return
        if what != "attn":
            S["append"](pool, S["bt"], S["sp"], S["cu"], k, v, status=S["status"], stream=stream)
        if what != "append":
            dec(pool, S["q"], S["bt"], S["ctx"], w.sm_scale, w.max_ctx, num_ctas=S["nct"], workspace=S["ws"],
                out=S["out"], status=S["status"], stream=stream)

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    # keep the GPU loaded ~0.5 s so the clock samples cover the timed region
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 and not args.profile else None
    t_end = time.perf_counter() + (0.0 if args.profile else 0.5)
    i = 0
    host_per_step = None
    while time.perf_counter() < t_end or host_per_step is None:
        t_enq = time.perf_counter()
        for _ in range(50):
            step(i)
            i += 1
        host_per_step = (time.perf_counter() - t_enq) / 50  # host enqueue cost of one step
        torch.cuda.synchronize()

    K = args.steps

    def timed(what):
        # K back-to-back calls (what: "step" = append + attention, the
        # headline; "attn" or "append" alone, for the per-call breakdown),
        # enqueued behind a spin kernel that outlasts their host-side enqueue,
        # so Python/launch overhead never leaves the GPU idle between them:
        # e0..e1 is GPU time. No event is recorded between kernels (an event
        # between two kernels of the stream adds a gap to every call).
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        torch.cuda._sleep(int(min(K * host_per_step * 1.5 + 2e-3, 2.0) * 2.2e9))
        e0.record(stream)
        for j in range(K):
            step(j, what)
        e1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        return e0.elapsed_time(e1)

    total_ms = timed("step")
    attn_ms = timed("attn") / K
    append_ms = timed("append") / K
    clocks = sampler.stop() if sampler else None
    if int(S["status"].item()) != 0:
        raise RuntimeError(f"device status {int(S['status'].item())} during the benchmark")

    ms = max_over_ranks(total_ms / K, world, device)
    step_bytes = w.attn_bytes() + w.append_bytes()

    e2e = None
    if not args.no_e2e and not args.profile:
        e2e = run_e2e(args, w, S, dec, replicas, step_bytes, world, device)

    return dict(ms=ms, attn_ms=attn_ms, append_ms=append_ms, clocks=clocks, step_bytes=step_bytes, replicas=replicas,
                pool_bytes=pool_bytes, e2e=e2e, nct=S["nct"], n_in=S["n_in"],
                in_bytes=2 * S["k"].numel() * S["k"].element_size())


def run_e2e(args, w, S, dec, replicas, step_bytes, world, device):
    """The same step through the public API from pinned host buffers: every
    step copies its inputs (new K/V rows, Q, positions, lengths) host->device,
    runs append + attention, and reads the output back device->host."""
    import torch

    import quantized_paged_kv_cache_gb300 as nk

    # The step's inputs (new K/V rows, Q, positions, lengths) sit back to back
    # in one pinned host buffer and go over in one copy into one device
    # buffer whose views are passed to the API.
    names = ("k", "v", "q", "sp", "cu", "ctx")
    offs, off = {}, 0
    for name in names:
        offs[name] = off
        off += (S[name].numel() * S[name].element_size() + 255) // 256 * 256
    h_buf = torch.empty(off, dtype=torch.uint8).pin_memory()
    d_buf = torch.empty(off, dtype=torch.uint8, device=device)

    def view(buf, name):
        t = S[name]
        n = t.numel() * t.element_size()
        return buf[offs[name]:offs[name] + n].view(t.dtype).view(t.shape)

    for name in names:
        view(h_buf, name).copy_(S[name].cpu())
    dev = {name: view(d_buf, name) for name in names}
    out_h = torch.empty(S["out"].shape, dtype=S["out"].dtype).pin_memory()
    stream = torch.cuda.current_stream()
    bi = h_buf.numel()  # the one host->device copy of a step (inputs + alignment padding)
    bo = out_h.numel() * out_h.element_size()
    via = "Python API: one pinned host->device copy, the step's calls, the output read back"
    if one_call_step(args, w):
        # the library's host-memory step: one C call copies the inputs in,
        # runs the step, copies the output and the status word out, and waits
        B, T, Hq = int(S["q"].shape[0]), int(S["q"].shape[1]), int(S["q"].shape[2])
        total = int(S["k"].shape[0])
        nbytes, offs = nk.step_host_layout(B, total, T, Hq, w.Hkv, w.D)
        h_in = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
        for name, o in zip(("k", "v", "q", "sp", "cu", "ctx"), offs):
            t = S[name]
            n = t.numel() * t.element_size()
            h_in[o:o + n].view(t.dtype).view(t.shape).copy_(t.cpu())
        staging = torch.empty(nbytes, dtype=torch.uint8, device=device)
        st_h = torch.zeros(1, dtype=torch.int32).pin_memory()
        bi, bo = nbytes, bo + 4
        via = "nk_decode_step_host: one C call per step (host->device copy, append + attention, output and status read back, stream wait)"

        def step(i):
            pool = S["pools"][i % replicas]
            nk.decode_step_host(pool, S["bt"], B, total, T, Hq, w.sm_scale, w.max_ctx, h_in, staging, S["out"],
                                out_h, num_ctas=S["nct"], workspace=S["ws"], status=S["status"], status_host=st_h,
                                stream=stream)

        return _time_e2e(args, step, step_bytes, world, device, bi, bo, via)

    def step(i):
        d_buf.copy_(h_buf, non_blocking=True)
        pool = S["pools"][i % replicas]
        if one_call_step(args, w):
            nk.decode_step(pool, S["bt"], dev["sp"], dev["cu"], dev["k"], dev["v"], dev["q"], dev["ctx"], w.sm_scale,
                           w.max_ctx, num_ctas=S["nct"], workspace=S["ws"], out=S["out"], status=S["status"],
                           stream=stream)
        else:
            S["append"](pool, S["bt"], dev["sp"], dev["cu"], dev["k"], dev["v"], status=S["status"], stream=stream)
            dec(pool, dev["q"], S["bt"], dev["ctx"], w.sm_scale, w.max_ctx, num_ctas=S["nct"], workspace=S["ws"],
                out=S["out"], status=S["status"], stream=stream)
        out_h.copy_(S["out"], non_blocking=True)
        stream.synchronize()

    return _time_e2e(args, step, step_bytes, world, device, bi, bo, via)


def _time_e2e(args, step, step_bytes, world, device, bi, bo, via):
    import torch

    for i in range(max(args.warmup, 3)):
        step(i)
    K = args.steps
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for j in range(K):
        step(j)
    el = max_over_ranks((time.perf_counter() - t0) * 1e3 / K, world, device)
    return {"value": round(job_gbs(step_bytes, el, world), 3), "unit": "GB/s",
            "ms_per_step": round(el, 5), "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "sync": "host waits for each step's output", "via": via}


# ---------------------------------------------------------------------------
# the oracle (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

class OracleStep:
    """The fp64 oracle on a bounded sample of the workload: the step's append
    of every new row, and the attention of `rows` query rows (all rows of the
    first kv-heads) over their full contexts."""

    def __init__(self, w, max_rows=None):
        import numpy as np
        import torch

        import oracle
        from quantized_paged_kv_cache_gb300 import workloads as wl

        self.w, self.oracle, self.np = w, oracle, np
        rk = w.fmt == "rk8v4"
        self.fmt = {"i8f16": "int8_f16", "bf16": "bf16"}.get(w.fmt)  # the oracle's other formats
        if self.fmt:
            f = self.fmt
            self.append = lambda *a: oracle.fmt_append(f, *a)
            self.attention = lambda *a: oracle.fmt_paged_attention(f, *a)
            self.attention_row = None  # rows are sampled as whole sequences
            self.pool = oracle.fmt_new_pool(f, w.num_pages, w.P, w.Hkv, w.D)
        else:
            self.append = oracle.rk_append if rk else oracle.kv_append
            self.attention = oracle.rk_paged_attention if rk else oracle.paged_attention
            self.attention_row = oracle.rk_attention_row if rk else oracle.attention_row
            self.pool = (oracle.rk_new_pool if rk else oracle.new_pool)(w.num_pages, w.P, w.Hkv, w.D)
        self.bt = wl.block_table(w)
        hist, _ = wl.history_and_step(w)
        for b in range(w.B):
            pos = 0
            while pos < hist[b]:
                n = min(16384, hist[b] - pos)
                k, v = wl.kv_rows(w, b, pos, n, device="cpu")
                self.append(self.pool, w.num_pages, w.P, w.Hkv, w.D, self.bt[b:b + 1], [pos], [0, n], k, v)
                pos += n
        starts, _ = wl.history_and_step(w)
        self.k, self.v, self.sp, self.cu = wl.append_batch(w, starts, [w.append_len] * w.B, device="cpu")
        self.q = wl.queries(w, device="cpu")
        all_rows = [(b, t, i) for b in range(w.B) for t in range(w.T) for i in range(w.Hq)]
        self.rows = all_rows if max_rows is None else all_rows[:max_rows]
        self.nseq = w.B
        if self.fmt and len(self.rows) < len(all_rows):
            # the other formats' oracle attends whole sequences: the first ones
            self.nseq = max(1, len(self.rows) // (w.T * w.Hq))
            self.rows = all_rows[:self.nseq * w.T * w.Hq]
        self.frac_rows = len(self.rows) / len(all_rows)
        self.threads = oracle.num_threads()
        # algorithmic bytes of this sample: the whole append, and the KV bytes
        # each sampled row's kv-head stream would read, pro rata per row
        self.bytes = w.append_bytes() + w.attn_bytes() * self.frac_rows
        del torch

    def __call__(self):
        w = self.w
        self.append(self.pool, w.num_pages, w.P, w.Hkv, w.D, self.bt, self.sp, self.cu, self.k, self.v)
        if self.frac_rows == 1.0:
            self.attention(self.pool, w.num_pages, w.P, w.Hkv, w.D, self.bt, w.ctx_lens, self.q, w.T, w.Hq,
                           w.sm_scale)
        elif self.fmt:
            n = self.nseq
            self.attention(self.pool, w.num_pages, w.P, w.Hkv, w.D, self.bt[:n].contiguous(), w.ctx_lens[:n],
                           self.q[:n].contiguous(), w.T, w.Hq, w.sm_scale)
        else:
            for (b, t, i) in self.rows:
                self.attention_row(self.pool, w.num_pages, w.P, w.Hkv, w.D, self.bt, w.ctx_lens, self.q, w.T,
                                   w.Hq, w.sm_scale, b, t, i)

    def sample_text(self):
        return (f"{len(self.rows)} of {self.w.B * self.w.T * self.w.Hq} query rows over their full contexts "
                f"+ the step's whole append ({self.w.append_rows()} rows); bytes counted pro rata")


def pick_rows(w, budget_s=2.0):
    """Rows for a bounded oracle step: roughly budget_s of single-row work per
    thread at ~2 ns per key-channel (fp64), never fewer than one kv-head group."""
    import oracle

    threads = max(1, oracle.num_threads())
    per_row = max(w.ctx_lens) * w.D * 2e-9
    rows = max(w.G, int(budget_s * threads / max(per_row, 1e-9)))
    total = w.B * w.T * w.Hq
    return None if rows >= total else rows


def cpu_baseline(w):
    st = OracleStep(w, pick_rows(w, budget_s=4.0))
    st()  # warm
    t0 = time.perf_counter()
    n = 0
    while True:
        st()
        n += 1
        if time.perf_counter() - t0 > 8.0 or n >= 3:
            break
    el = (time.perf_counter() - t0) / n
    return {"value": round(st.bytes / el / 1e9, 4), "unit": "GB/s", "cores": st.threads, "kind": "oracle",
            "sample": st.sample_text(), "s_per_step": round(el, 4)}


def run_reference(args, w):
    st = OracleStep(w, pick_rows(w, budget_s=0.5))
    for _ in range(max(args.warmup, 3)):
        st()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        st()
    el = (time.perf_counter() - t0) / args.steps
    val = st.bytes / el / 1e9
    cb = {"value": round(val, 4), "unit": "GB/s", "cores": st.threads, "kind": "oracle", "sample": st.sample_text()}
    return {"impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(w, "host"), "cpu_baseline": cb,
            "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def config_dict(w, l2):
    return {"workload": w.name, "kv_format": w.fmt, "B": w.B, "T": w.T, "q_heads": w.Hq, "kv_heads": w.Hkv,
            "head_dim": w.D, "page_size": w.P, "ctx_lens": w.ctx_lens if w.B <= 8 else f"{w.B} seqs", "append_rows": w.append_rows(),
            "l2": l2}


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    from quantized_paged_kv_cache_gb300 import workloads as wl

    w = wl.make(args.config)
    if args.impl == "reference":
        if rank == 0:
            line = json.dumps(run_reference(args, w))
            print(line, flush=True)
            if args.out:
                with open(args.out, "a") as f:
                    f.write(line + "\n")
        return 0

    import torch

    if world > 1:
        torch.distributed.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    r = run_ours(args, w, rank, world, device)
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0
    peaks, src = measured_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    attn_us = r["attn_ms"] * 1e3
    append_us = r["append_ms"] * 1e3
    achieved = w.attn_bytes() / (attn_us * 1e-6) / 1e9
    prefill = is_prefill(w)
    if prefill:  # compute-bound: the tensor roofline (fp16 mma.sync at the bf16 rate)
        tflops = w.attn_flops() / (attn_us * 1e-6) / 1e12
        tpeak = float(peaks.get("bf16_tflops", 1900.0))
    traffic = ncu_traffic(w.name, args.kernel)
    us = r["ms"] * 1e3
    gbs = job_gbs(r["step_bytes"], r["ms"], world)
    l2 = (f"rotating {r['replicas']} pool copies ({r['replicas'] * r['pool_bytes'] / 2**20:.0f} MiB) > 2x L2"
          if r["replicas"] > 1 else f"pool {r['pool_bytes'] / 2**20:.0f} MiB > 2x L2")
    if r["n_in"] > 1:
        l2 += (f"; append input rotated over {r['n_in']} copies "
               f"({r['n_in'] * r['in_bytes'] / 2**20:.0f} MiB) > 2x L2")
    out = {
        "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(r["ms"], 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": {"rk8v4": "i8 K / i4 V KV (fp16 scales), f16 MMA operands (rotated Q hi + lo), f32 accumulate",
                  "i8f16": "i8 KV (fp16 scales), f16 MMA operands, f32 accumulate",
                  "bf16": "bf16 KV, bf16 MMA operands, f32 accumulate"}.get(
                      w.fmt, "i8 KV, f16 MMA operands, f32 accumulate"),
        "data": "synthetic",
        "config": config_dict(w, l2),
        "us_per_call": round(us, 3), "attn_us_per_call": round(attn_us, 3),
        "append_us_per_call": round(append_us, 3),
        "breakdown": (("value/ms_per_step: K back-to-back steps (nk_decode_step: append + attention); attn/append "
                       "us and the roofline: K back-to-back calls of nk_paged_decode_attn / nk_kv_append alone, same "
                       "inputs and pool rotation") if one_call_step(args, w) else
                      ("value/ms_per_step: K back-to-back steps (append call + attention call); attn/append us and "
                       "the roofline: K back-to-back calls of each alone, same inputs and pool rotation")),
        "append_gbs": round(w.append_bytes() / (append_us * 1e-6) / 1e9, 2),
        "attn_gbs": round(achieved, 2),
        "pct_of_hbm_peak": round(100 * gbs / world / peak, 2),
        "kernel": args.kernel if w.fmt == "int8" else w.fmt, "num_ctas": r["nct"] or "default",
        "clocks": r["clocks"], "e2e": r["e2e"], "gpu_launches": (2 if is_prefill(w) else 3) * args.steps,
        "roofline": ({"bound": "tensor", "achieved": round(tflops, 2), "peak": tpeak, "unit": "TFLOP/s",
                      "frac": round(tflops / tpeak, 4), "traffic": None,
                      "kernel": "chunked-prefill kernel (one nk_paged_prefill_attn call, mma.sync)",
                      "peak_source": f"{src} bf16_tflops (burst)", "flops_per_launch": w.attn_flops()}
                     if prefill else
                     {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": ("paged_decode split kernel + combine (one nk_paged_decode_attn call)"
                                if w.fmt == "int8" else
                                f"{w.fmt} split kernel + combine (one nk_{'bf16kv' if w.fmt == 'bf16' else w.fmt}"
                                "_decode_attn call)"),
                     "peak_source": f"{src} hbm_gbs", "bytes_per_launch": w.attn_bytes()}),
    }
    if not args.no_cpu_baseline and world == 1 and not args.profile:
        out["cpu_baseline"] = cpu_baseline(w)
    line = json.dumps(out)
    print(line, flush=True)
    if args.out:
        with open(args.out, "a") as f:
            f.write(line + "\n")
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
