#!/usr/bin/env python3
"""Benchmark: NVFP4 paged decode on one or more GB300s (one process per GPU).

One step = the step's new K/V tokens quantised into their pages + paged NVFP4
attention + the split-KV merge, in one launch (nvfp4kv_decode_append_run;
--separate-append runs nvfp4kv_quantize_append and nvfp4kv_decode_run as two
launches instead) over the long-context decode
workload (B=4, Hq=32, Hkv=8, D=128, kv_len=32771, page_size 16).  The plan is
built once, outside the timed region (as serving builds it once per batch
step and reuses it for every layer); the end-to-end leg re-plans every step.

Prints one JSON line (rank 0).  ``--impl reference`` times the float64 CPU
oracle on the same workload instead (bounded samples per step).
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
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import nvfp4_paged_kv_nvfp4kv_gb300 as N  # noqa: E402
from nvfp4_paged_kv_nvfp4kv_gb300 import workloads as W  # noqa: E402

METRIC = "NVFP4 paged decode: µs/call, KV tokens/s, achieved HBM GB/s vs GB300 peak"
UNIT = "KV tokens/s"
FALLBACK_HBM_GBS = 6800.0
_CSRC = os.path.join(ROOT, "nvfp4_paged_kv_nvfp4kv_gb300", "csrc")
_COMMON = ("append_fused.cuh", "device_common.cuh", "epilogue.cuh", "internal.h", "quantize.cuh")
# per workload: the committed ncu summary of its dominant kernel and the
# sources that kernel is built from (the DRAM bytes are used only while the
# sources still hash to the value the summary was taken on)
TRAFFIC = {
    "long_context_decode": ("attend_dec_long_context_decode.json",
                            ("attend_dec.cu", "device_common.cuh", "epilogue.cuh", "internal.h",
                             "quantize.cuh")),
    "prefix_cache_extend": ("attend_tcgen05_prefix_cache_extend.json",
                            ("attend_tcgen05.cu",) + _COMMON),
}


def workload_desc(cfg: W.Workload) -> str:
    lens = ("kv_len=%d" % cfg.kv_len_lo if cfg.kv_len_lo == cfg.kv_len_hi
            else "kv_len~U[%d,%d]" % (cfg.kv_len_lo, cfg.kv_len_hi))
    return ("%s: B=%d qo_len=%d Hq=%d Hkv=%d Dqk=%d Dvo=%d %s page_size=16%s, NVFP4 K/V "
            "(e2m1 + E4M3 per 16)" % (cfg.name, cfg.batch, cfg.qo_len, cfg.num_qo_heads,
                                      cfg.num_kv_heads, cfg.head_dim_qk, cfg.head_dim_vo,
                                      lens, ", causal" if cfg.causal else ""))


def algorithmic_bytes(batch: W.Batch, fused_append: bool = False) -> int:
    """KV bytes at 0.5 B/element + scale bytes + Q + O + lse + page table;
    with the append fused in, also the new tokens' bf16 K/V read and their
    packed bytes + scales written."""
    c = batch.cfg
    packed = (c.head_dim_qk // 2 + c.head_dim_qk // 16 + c.head_dim_vo // 2 +
              c.head_dim_vo // 16)
    kv = sum(batch.kv_lens) * c.num_kv_heads * packed
    rows = int(batch.qo_indptr[-1])
    qo = rows * c.num_qo_heads * (2 * c.head_dim_qk + 2 * c.head_dim_vo + 4)
    pt = 4 * (int(batch.kv_indices.numel()) + 2 * c.batch + 1 + c.batch + 1)
    new = 0
    if fused_append:
        new = rows * c.num_kv_heads * (2 * (c.head_dim_qk + c.head_dim_vo) + packed)
    return kv + qo + pt + new


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_hash(sources) -> str:
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(_CSRC, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_per_launch(workload: str):
    """DRAM bytes per launch of the workload's dominant kernel from its
    committed ncu summary, if one exists for this workload and was taken on
    the current kernel source (else None)."""
    if workload not in TRAFFIC:
        return None
    fname, sources = TRAFFIC[workload]
    try:
        with open(os.path.join(ROOT, "profiles", fname)) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("workload") != workload or d.get("kernel_hash") != kernel_hash(sources):
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while a region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self._t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
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
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def init_dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_gpu(args, world, rank, local):
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = W.WORKLOADS[args.workload]
    batch = W.make_batch(cfg)
    lay = batch.cache_layout(args.layout)
    cache = N.PagedCache.allocate(lay, batch.k_global_scale, batch.v_global_scale,
                                  device=dev)
    i32 = lambda t: torch.as_tensor(t).to(torch.int32).to(dev)
    kv_indices, kv_indptr, last = i32(batch.kv_indices), i32(batch.kv_indptr), \
        i32(batch.last_page_len)
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    ts = batch.prefix
    for s in range(0, ts.k.shape[0], 1 << 16):
        N.nvfp4kv_quantize_append(cache, ts.k[s:s + (1 << 16)].to(dev),
                                  ts.v[s:s + (1 << 16)].to(dev),
                                  i32(ts.batch_idx[s:s + (1 << 16)]),
                                  i32(ts.positions[s:s + (1 << 16)]), kv_indices, kv_indptr,
                                  last, device_flags=flags)
    new_k, new_v = batch.new.k.to(dev), batch.new.v.to(dev)
    new_b, new_p = i32(batch.new.batch_idx), i32(batch.new.positions)
    q = batch.q.to(dev)
    c = cfg
    plan = N.nvfp4kv_decode_plan(batch.qo_indptr, batch.kv_indptr, batch.last_page_len,
                                 c.num_qo_heads, c.num_kv_heads, c.head_dim_qk, c.head_dim_vo,
                                 causal=c.causal, kernel=args.kernel, device=local,
                                 force_chunk_tokens=args.chunk_tokens)
    rows = int(batch.qo_indptr[-1])
    out = torch.empty((rows, c.num_qo_heads, c.head_dim_vo), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((rows, c.num_qo_heads), dtype=torch.float32, device=dev)
    flush = (torch.empty(512 << 20, dtype=torch.uint8, device=dev)
             if args.l2_flush != "none" else None)
    flush_r = (torch.zeros(512 << 20, dtype=torch.uint8, device=dev)
               if args.l2_flush == "write_read" else None)
    stream = torch.cuda.current_stream(dev)

    # the step's new tokens, row-aligned with the query rows
    order = torch.argsort(batch.new.batch_idx.long() * (1 << 30) +
                          batch.new.positions.long())
    row_k, row_v = batch.new.k[order].to(dev), batch.new.v[order].to(dev)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        if args.separate_append:
            N.nvfp4kv_quantize_append(cache, new_k, new_v, new_b, new_p, kv_indices,
                                      kv_indptr, last, device_flags=flags)
            if ev:
                ev[1].record(stream)
        if args.separate_append:
            N.nvfp4kv_decode_run(plan, q, cache, kv_indices, batch.sm_scale, out=out, lse=lse)
        else:  # one launch: append fused into the attention (and the merge)
            N.nvfp4kv_decode_append_run(plan, row_k, row_v, q, cache, kv_indices,
                                        batch.sm_scale, out=out, lse=lse)
        if ev:
            ev[2].record(stream)

    def pre_step():
        l2_flush()
        torch.cuda._sleep(200000)   # bounded spin: keep the GPU busy while the
        #                             host enqueues the step back to back

    def l2_flush():
        if flush is None:
            return
        flush.fill_(1)              # evict the cache (write > L2) between steps
        if flush_r is not None:     # then read > L2: the flush's dirty lines are
            flush_r.max()           # written back here, not inside the timed step

    for _ in range(args.warmup):
        pre_step()
        step()
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for k in range(args.steps):
            pre_step()
            step(evs[k])
        torch.cuda.synchronize()
    barrier(world)
    t_step = [e[0].elapsed_time(e[2]) for e in evs]
    if args.separate_append:
        t_append = [e[0].elapsed_time(e[1]) for e in evs]
        t_attend = [e[1].elapsed_time(e[2]) for e in evs]
    else:  # one launch: no event between append and attention
        t_append, t_attend = [0.0], t_step
    ms_step = statistics.mean(t_step)
    q = sorted(t_step)
    spread = {"median": statistics.median(q), "p10": q[len(q) // 10],
              "p90": q[(9 * len(q)) // 10], "min": q[0], "max": q[-1]}
    ms_step_max = max_over_ranks(ms_step, world)
    kv_tokens = sum(batch.kv_lens)
    value = kv_tokens * world / (ms_step_max * 1e-3)

    def run_e2e():
        # ---- end to end through the public API with host buffers -------------
        # Serving makes a plan once per change of the batch's page or query
        # counts: here one plan with live last-page lengths (plan option
        # device_last_page_len).  Every step copies its inputs (Q, the new tokens'
        # K/V, the requests' last page lengths) from one pinned host buffer, runs
        # the fused append + attention, and copies out and lse back.  The step's
        # three calls are captured once as a CUDA graph and replayed; the eager
        # figure issues them every step.
        def packed(tensors, device):
            offs, n = [], 0
            for t in tensors:
                offs.append(n)
                n += (t.numel() * t.element_size() + 255) // 256 * 256
            buf = torch.empty(n, dtype=torch.uint8, device=device,
                              pin_memory=(device == "cpu"))
            views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                     for o, t in zip(offs, tensors)]
            return buf, views
        src = [batch.q, batch.new.k[order].contiguous(), batch.new.v[order].contiguous(),
               batch.last_page_len.to(torch.int32).contiguous()]
        if args.separate_append:  # the two-launch step also needs request and position
            src += [batch.new.batch_idx[order].contiguous(), batch.new.positions[order].contiguous()]
        h_in, h_views = packed(src, "cpu")
        for hv, t in zip(h_views, src):
            hv.copy_(t)
        d_in, d_views = packed(src, dev)
        d_q, d_k, d_v, d_lpl = d_views[:4]
        d_b, d_p = (d_views[4], d_views[5]) if args.separate_append else (None, None)
        h_res, (h_out, h_lse) = packed([out, lse], "cpu")
        d_res, (e_out, e_lse) = packed([out, lse], dev)
        d_in.copy_(h_in)
        plan_e = N.nvfp4kv_decode_plan(batch.qo_indptr, batch.kv_indptr, batch.last_page_len,
                                       c.num_qo_heads, c.num_kv_heads, c.head_dim_qk,
                                       c.head_dim_vo, causal=c.causal, kernel=args.kernel,
                                       force_chunk_tokens=args.chunk_tokens, device=local,
                                       device_last_page_len=d_lpl)

        def e2e_step():
            d_in.copy_(h_in, non_blocking=True)
            if args.separate_append:
                N.nvfp4kv_quantize_append(cache, d_k, d_v, d_b, d_p, kv_indices, kv_indptr, d_lpl,
                                          device_flags=flags)
                N.nvfp4kv_decode_run(plan_e, d_q, cache, kv_indices, batch.sm_scale, out=e_out,
                                     lse=e_lse)
            else:
                N.nvfp4kv_decode_append_run(plan_e, d_k, d_v, d_q, cache, kv_indices,
                                            batch.sm_scale, out=e_out, lse=e_lse)
            h_res.copy_(d_res, non_blocking=True)

        e2e_step()  # eager first call (the library prepares the kernel once)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            e2e_step()
        torch.cuda.synchronize()
        e2e_steps = max(3, min(args.steps, 200))
        # bytes moved per step: the packed buffers, with their alignment padding
        h2d = h_in.numel()
        d2h = h_res.numel()

        def time_e2e(run):
            ts = []
            for k in range(e2e_steps + 3):
                l2_flush()
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                run()
                torch.cuda.synchronize()
                if k >= 3:
                    ts.append(time.perf_counter() - t0)
            return ts
        times = time_e2e(graph.replay)
        assert torch.equal(h_out.view(torch.int16), out.cpu().view(torch.int16))
        times_eager = time_e2e(e2e_step)
        assert torch.equal(h_out.view(torch.int16), out.cpu().view(torch.int16))
        e2e_s = max_over_ranks(statistics.mean(times), world)
        e2e_value = kv_tokens * world / e2e_s
        return {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3,
                "ms_per_step_median": statistics.median(times) * 1e3,
                "ms_per_step_eager": statistics.mean(times_eager) * 1e3,
                "how": "plan with live last-page lengths made once; per step: inputs "
                       "copied from one pinned host buffer, fused append + attention, out "
                       "and lse copied back; the three calls replayed as a CUDA graph "
                       "(ms_per_step_eager: issued eagerly)"}
    e2e = None if args.no_e2e else run_e2e()

    # ---- roofline of the attention kernel -------------------------------
    peak, peak_kind = measured_peak()
    alg = algorithmic_bytes(batch, fused_append=not args.separate_append)
    ms_attend = statistics.mean(t_attend)
    achieved = alg / (ms_attend * 1e-3) / 1e9
    traffic = traffic_per_launch(cfg.name)
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 operands (exact e2m1 x E4M3), f32 accumulate", "data": "synthetic",
        "config": {
            "workload": workload_desc(cfg), "layout": args.layout,
            "step": ("quantize_append + decode_run (two launches)" if args.separate_append else
                     "decode_append_run: new tokens quantised into their pages, attention and "
                     "split-KV merge in one launch") + "; plan built once",
            "l2": {"write_read": "flushed between steps: 512 MB write, then 512 MB read (no "
                                 "dirty lines of the flush are written back inside the "
                                 "timed step)",
                   "write": "flushed between steps (512 MB write)",
                   "none": "not flushed (profiler capture; not a timing)"}[args.l2_flush],
            "kernel": {1: "tensor-core mma.sync f16/f32acc",
                       2: "CUDA-core f32",
                       3: "tcgen05.mma f16/f32acc, K_hat in tensor memory",
                       4: "FP4 query and probabilities: row-maximum launch + mma.sync "
                          "attention launch, FP4 operands expanded exactly to f16"}[plan.info.kernel],
            "split_units": int(plan.info.num_units), "split": int(plan.info.split),
            "chunk_pages": int(plan.info.chunk_pages),
            "us_per_call": ms_step_max * 1e3,
            "us_per_call_spread": {k: v * 1e3 for k, v in spread.items()},
            "us_attend_incl_fused_merge": ms_attend * 1e3,
            "us_separate_append": (statistics.mean(t_append) * 1e3
                                   if args.separate_append else None),
            "algorithmic_bytes_per_call": alg,
            "hbm_gbs_step": alg / (ms_step_max * 1e-3) / 1e9,
            "parallelism": "replicas (one independent batch per GPU)",
        },
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": peak_kind},
        "e2e": e2e,
        "gpu_launches": args.steps * ((2 if args.separate_append else 1) +
                                      (1 if plan.info.kernel == 4 else 0)),
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(batch, args.layout,
                                              fp4qp=plan.info.kernel == 4)
    return result


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------

def run_op(args, local):
    """The library's standalone operations on the workload's sizes (not the
    benchmark's metric: one JSON line per op for their profiles).

    merge_states: the float32 partial states of the workload's split plan
    (random values; every (query row, head) merges the plan's number of
    splits) folded into bf16 out + lse.  dequantize: every page of the
    workload's cache (quantised from its K/V) to float32 K and V.  GB/s counts
    the bytes each op must read and write."""
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = W.WORKLOADS[args.workload]
    batch = W.make_batch(cfg)
    c = cfg
    g = torch.Generator().manual_seed(cfg.seed + 101)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(512 << 20, dtype=torch.uint8, device=dev)
    if args.op == "merge_states":
        plan = N.nvfp4kv_decode_plan(batch.qo_indptr, batch.kv_indptr, batch.last_page_len,
                                     c.num_qo_heads, c.num_kv_heads, c.head_dim_qk,
                                     c.head_dim_vo, causal=c.causal, device=local,
                                     allocate=False)
        splits = max(1, int(plan.info.max_units_per_request))
        E = int(batch.qo_indptr[-1]) * c.num_qo_heads
        P = E * splits
        po = torch.randn((P, c.head_dim_vo), generator=g).to(dev)
        pl = (torch.randn((P,), generator=g) * 4).to(dev)
        mi = (torch.arange(E + 1, dtype=torch.int32) * splits).to(dev)
        run = lambda: N.nvfp4kv_merge_states(po, pl, mi)
        nbytes = P * (c.head_dim_vo + 1) * 4 + (E + 1) * 4 + E * (c.head_dim_vo * 2 + 4)
        desc = "%d (row, head) entries x %d partial states, Dv=%d" % (E, splits, c.head_dim_vo)
    else:
        lay = batch.cache_layout(args.layout)
        cache = N.PagedCache.allocate(lay, batch.k_global_scale, batch.v_global_scale,
                                      device=dev)
        i32 = lambda t: torch.as_tensor(t).to(torch.int32).to(dev)
        kv_indices, kv_indptr, last = i32(batch.kv_indices), i32(batch.kv_indptr), \
            i32(batch.last_page_len)
        for ts in (batch.prefix, batch.new):
            for s0 in range(0, ts.k.shape[0], 1 << 16):
                N.nvfp4kv_quantize_append(cache, ts.k[s0:s0 + (1 << 16)].to(dev),
                                          ts.v[s0:s0 + (1 << 16)].to(dev),
                                          i32(ts.batch_idx[s0:s0 + (1 << 16)]),
                                          i32(ts.positions[s0:s0 + (1 << 16)]),
                                          kv_indices, kv_indptr, last)
        pages = kv_indices
        n = int(pages.numel())
        k_out = torch.empty((n, 16, c.num_kv_heads, c.head_dim_qk), dtype=torch.float32,
                            device=dev)
        v_out = torch.empty((n, 16, c.num_kv_heads, c.head_dim_vo), dtype=torch.float32,
                            device=dev)
        run = lambda: N.nvfp4kv_dequantize_paged(cache, pages, k_out=k_out, v_out=v_out)
        elts = n * 16 * c.num_kv_heads
        nbytes = (elts * (c.head_dim_qk + c.head_dim_vo) * (0.5 + 1 / 16 + 4) + n * 4)
        desc = "%d pages x 16 tokens x %d kv heads, Dqk=%d Dvo=%d" % (
            n, c.num_kv_heads, c.head_dim_qk, c.head_dim_vo)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    t = []
    for _ in range(args.steps):
        if args.l2_flush != "none":
            flush.fill_(1)
            flush_r.max()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run()
        b.record(stream)
        t.append((a, b))
    torch.cuda.synchronize()
    ms = statistics.mean(x.elapsed_time(y) for x, y in t)
    return {"op": args.op, "metric": "standalone %s: achieved GB/s" % args.op,
            "value": nbytes / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms,
            "steps": args.steps, "warmup": args.warmup, "bytes_per_step": nbytes,
            "config": {"workload": workload_desc(cfg), "op": desc,
                       "l2": "flushed between steps" if args.l2_flush != "none" else "not flushed"}}


def _oracle():
    sys.path.insert(0, os.path.join(ROOT, "oracle"))
    import oracle as O
    return O


def _oracle_prefix_cache(batch, requests, layout):
    O = _oracle()
    c = O.Cache(batch.cache_layout(layout), batch.k_global_scale, batch.v_global_scale)
    pt = O.PageTable.of(batch)
    req = torch.tensor(sorted(requests))
    for ts in (batch.prefix,):
        m = torch.isin(ts.batch_idx, req.to(ts.batch_idx.dtype))
        sub = W.TokenSet(ts.batch_idx[m], ts.positions[m], ts.k[m], ts.v[m])
        assert O.quantize_append(c, pt, sub) == 0
    return c, pt


def _oracle_units(O, cache, pt, batch, units, threads, chunk=None, fp4qp=False):
    """Oracle step on (request, kv head) units: append the requests' new
    tokens, then exact attention (or, with fp4qp, the FP4 query and
    probabilities method of kernel 4), the units spread over a thread pool
    (ctypes releases the GIL)."""
    import concurrent.futures as cf
    c = batch.cfg
    reqs = sorted({b for b, _ in units})
    m = torch.isin(batch.new.batch_idx, torch.tensor(reqs, dtype=batch.new.batch_idx.dtype))
    sub = W.TokenSet(batch.new.batch_idx[m], batch.new.positions[m], batch.new.k[m],
                     batch.new.v[m])
    assert O.quantize_append(cache, pt, sub) == 0
    rows = int(batch.qo_indptr[-1])
    import numpy as np
    out = np.full((rows, c.num_qo_heads, c.head_dim_vo), np.nan)
    lse = np.full((rows, c.num_qo_heads), np.nan)
    fn = O.attention_fp4qp if fp4qp else O.attention
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(lambda u: fn(cache, pt, batch.qo_indptr, batch.q, c.num_qo_heads,
                                 c.causal, batch.sm_scale, units=[u], out=out, lse=lse),
                    units))
    return out, lse


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model", "hardware")):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def _timed_passes(O, cache, pt, batch, units, threads, min_s, max_passes, fp4qp=False):
    passes, t0 = 0, time.perf_counter()
    while True:
        _oracle_units(O, cache, pt, batch, units, threads, fp4qp=fp4qp)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_s or passes >= max_passes:
            return passes, dt


def cpu_baseline(batch, layout, min_s: float = 10.0, max_passes: int = 100, fp4qp=False):
    """The oracle as it stands on the host cores: up to 4 requests of the
    workload, one (request, kv head) unit per thread on all cores (whole
    passes repeated for about ``min_s`` seconds, at most ``max_passes``), and
    the same oracle on one core over the first request's first kv head."""
    O = _oracle()
    c = batch.cfg
    cores = os.cpu_count() or 1
    requests = list(range(min(4, c.batch)))
    cache, pt = _oracle_prefix_cache(batch, requests, layout)
    units = [(b, h) for b in requests for h in range(c.num_kv_heads)]
    threads = min(len(units), cores)
    passes, dt = _timed_passes(O, cache, pt, batch, units, threads, min_s, max_passes, fp4qp)
    toks = sum(batch.kv_lens[b] for b in requests)
    p1, dt1 = _timed_passes(O, cache, pt, batch, [(0, 0)], 1, min_s / 3, max_passes, fp4qp)
    return {"value": toks * passes / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "cpu_count": cores, "cpu_model": cpu_model(),
            "value_1core": batch.kv_lens[0] / c.num_kv_heads * p1 / dt1,
            "sample": "requests %s of the workload (%d KV tokens x %d kv heads), append of "
                      "their new tokens + float64 %s, one (request, kv head) "
                      "unit per thread on %d threads, %d passes in %.1f s; value_1core: "
                      "request 0, kv head 0 on one thread, %d passes in %.1f s" % (
                          requests, toks, c.num_kv_heads,
                          "FP4 query and probabilities attention" if fp4qp else
                          "exact attention", threads, passes, dt, p1, dt1)}


def run_reference(args, world, rank):
    """The oracle timed on the host cores: each step appends the new tokens of
    a bounded sample of (request, kv head) units and runs exact attention for
    them, one unit per thread on all cores."""
    if rank != 0:
        return None
    O = _oracle()
    cfg = W.WORKLOADS[args.workload]
    batch = W.make_batch(cfg)
    cores = os.cpu_count() or 1
    requests = list(range(min(4, cfg.batch)))
    cache, pt = _oracle_prefix_cache(batch, requests, args.layout)
    all_units = [(b, h) for b in requests for h in range(cfg.num_kv_heads)]
    # Per-step sample: as many units as fit the time budget of the whole
    # --warmup + --steps run (NVFP4KV_REF_BUDGET_S, default 150 s), at least
    # one; if even one unit per step is slower, the run stops at the budget
    # and reports the steps it timed.
    budget = float(os.environ.get("NVFP4KV_REF_BUDGET_S", "150"))
    t0 = time.perf_counter()
    _oracle_units(O, cache, pt, batch, all_units[:1], 1, fp4qp=args.kernel == 4)
    unit_s = time.perf_counter() - t0
    per_step = budget / max(1, args.steps + args.warmup)
    n_units = max(1, min(len(all_units), int(per_step / max(unit_s, 1e-9) * cores)))
    units = all_units[:n_units]
    threads = min(n_units, cores)
    times = []
    start = time.perf_counter()
    for k in range(args.warmup + args.steps):
        t = time.perf_counter()
        _oracle_units(O, cache, pt, batch, units, threads, fp4qp=args.kernel == 4)
        if k >= args.warmup:
            times.append(time.perf_counter() - t)
        if len(times) >= 3 and time.perf_counter() - start > budget:
            break
    dt = statistics.mean(times)
    toks = sum(batch.kv_lens[b] for b, _ in units) / cfg.num_kv_heads
    value = toks / dt
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": len(times), "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_desc(cfg), "layout": args.layout,
                   "sample": "%d (request, kv head) units per step" % n_units},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "cpu_count": cores, "cpu_model": cpu_model(),
                         "sample": "%d (request, kv head) units of requests %s per step, one "
                                   "per thread: append of their new tokens + float64 %s" % (
                                       n_units, sorted({b for b, _ in units}),
                                       "FP4 query and probabilities attention"
                                       if args.kernel == 4 else "exact attention")},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long_context_decode", choices=list(W.WORKLOADS))
    ap.add_argument("--layout", default="HND", choices=["HND", "NHD"])
    ap.add_argument("--kernel", type=int, default=0,
                    help="0 auto, 1 tensor-core mma.sync, 2 CUDA-core, 3 tcgen05, "
                         "4 FP4 query and probabilities")
    ap.add_argument("--chunk-tokens", type=int, default=0,
                    help="split-KV chunk in tokens (multiple of 16); 0 = the planner's choice")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--l2-flush", default="write_read", choices=["write", "write_read", "none"],
                    help="between steps: write 512 MB and then read another 512 MB, so no "
                         "dirty line of the flush is written back inside the timed step "
                         "(default), or only write 512 MB; 'none' is for profiler "
                         "captures, which flush the cache themselves (not a timing mode)")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end leg (profiler captures)")
    ap.add_argument("--separate-append", action="store_true",
                    help="quantize_append and decode_run as two launches per step")
    ap.add_argument("--op", default="attention", choices=["attention", "merge_states", "dequantize"],
                    help="time one of the library's standalone operations on the workload's "
                         "sizes instead (for their profiles; not the benchmark's metric)")
    args = ap.parse_args()
    if args.kernel == 2:  # the CUDA-core comparison kernel has no fused append
        args.separate_append = True
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = init_dist()
    if args.op != "attention":
        res = run_op(args, local) if rank == 0 else None
    elif args.impl == "reference":
        res = run_reference(args, world, rank)
    else:
        res = run_gpu(args, world, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
