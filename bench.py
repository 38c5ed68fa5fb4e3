#!/usr/bin/env python
"""Benchmark of the MSA operator on GB300: prefill tokens/s with per-kernel roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl msa|reference] [--workload NAME]

A step is one full pass of the hot path over one batch of synthetic input resident in HBM:
index selection (score + max-pool + top-k) followed by the main branch (scheduling, KV-outer
attention, combine) on the 64/4-head, L = 32768 prefill workload, then one paged decode step of
the 64-sequence workload (reported under "decode").  Prints ONE JSON line (rank 0) with:
  value / roofline / kernel_rooflines  prefill tokens/s and each kernel against the measured peaks
  e2e                    the same step through the public API from pinned host buffers
  e4m3_index             the index kernels timed again with e4m3 index vectors (same selections)
  index_scores           the index kernels timed again exporting every block's pooled score
  cuda_graph             the small prefill pass eager against a CUDA-graph replay of the same calls
  cpu_baseline           the CPU oracle on a bounded sample, on this host's cores

The path has no exchange step, so N > 1 runs N independent replicas (one per GPU, weak scaling)
with a barrier and the max over ranks around the timed region.
``--impl reference`` times the CPU oracle (the only reference there is) on bounded samples.
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import synthetic  # noqa: E402
from block_sparse_long_msa_gb300 import accounting as acc  # noqa: E402

METRIC = "MSA prefill tokens/s and decode tokens/s at 1 GB300; % tensor/HBM roofline"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=60)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="msa", choices=["msa", "reference"])
    p.add_argument("--workload", default="prefill_L32K")
    p.add_argument("--decode-workload", default="decode_b64_16K_256K")
    p.add_argument("--decode-batch", type=int, default=0, help="override (profiling)")
    p.add_argument("--decode-nmax", type=int, default=0, help="override (profiling)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e4m3-index", action="store_true",
                   help="skip timing the e4m3 (FP8) index kernels beside the bf16 step")
    p.add_argument("--no-index-scores", action="store_true",
                   help="skip timing the index kernels with the block-score export")
    p.add_argument("--no-graph", action="store_true",
                   help="skip timing the small prefill pass as a CUDA-graph replay")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--L", type=int, default=0, help="override the workload length (profiling)")
    return p.parse_args()


def workload(args):
    w = synthetic.WORKLOADS[args.workload]
    if args.L:
        w = synthetic.Workload(**{**w.__dict__, "L": args.L, "name": f"{w.name}@L{args.L}"})
    return w


# ------------------------------------------------------------------------------------------
# distributed plumbing (replicas only: no collective touches the data path)
# ------------------------------------------------------------------------------------------
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl == "msa" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = [r for r in csv.reader(io.StringIO(self.out or "")) if len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clocks unavailable"],
                    "samples": 0}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if "Active" in v
                          and "Not" not in v})
        power = []
        for r in rows:
            try:
                power.append(float(r[3]))
            except ValueError:
                pass
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(power) if power else None}


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu capture
# of the named kernel (profiles/ has the capture summaries).  A figure is reported only while the
# kernel's sources still hash to the value recorded with it; otherwise the traffic is null.
CSRC = os.path.join(ROOT, "block_sparse_long_msa_gb300", "csrc")
KERNEL_SOURCES = {
    "attention": ["attn_prefill.cu", "common.cuh", "ptx.cuh"],
    "combine": ["attn_prefill.cu", "common.cuh", "ptx.cuh"],
    "index": ["index_prefill.cu", "common.cuh", "ptx.cuh"],
    "index_e4m3": ["index_prefill.cu", "common.cuh", "ptx.cuh"],
    "decode_scan": ["decode.cu", "common.cuh", "ptx.cuh"],
    "decode_scan_e4m3": ["decode.cu", "common.cuh", "ptx.cuh"],
}
NCU_TRAFFIC = {
    # prefill L=32768, 64/4 heads, k=16 (profiles/dram_prefill_L32K_decode_b64.md)
    "attention": {"bytes_per_launch": 9828836096, "workload": "prefill_L32K@32768",
                  "sources_sha256": "7d4d5adc609b717953302cb6c3fc4d49f754da7eae7cf3f27036282b37e8205c"},
    "combine": {"bytes_per_launch": 9194790912, "workload": "prefill_L32K@32768",
                "sources_sha256": "7d4d5adc609b717953302cb6c3fc4d49f754da7eae7cf3f27036282b37e8205c"},
    "index": {"bytes_per_launch": 41903616, "workload": "prefill_L32K@32768",
              "sources_sha256": "549e86cc1e19b86d0fd21c929853b80722a68fa8fe9701ae39a3cc23b5248ac2"},
    "index_e4m3": {"bytes_per_launch": 21011413, "workload": "prefill_L32K@32768",
                   "sources_sha256": "549e86cc1e19b86d0fd21c929853b80722a68fa8fe9701ae39a3cc23b5248ac2"},
    # decode, 64 sequences of 16K-256K tokens
    "decode_scan": {"bytes_per_launch": 2084700160,
                    "workload": "decode_b64_16K_256K@64x262144",
                    "sources_sha256": "994ce2153b759ea1038980cc54121fca1a7ce5a247759beee4807547bab49afc"},
    "decode_scan_e4m3": {"bytes_per_launch": 1044300331,
                         "workload": "decode_b64_16K_256K@64x262144",
                         "sources_sha256": "994ce2153b759ea1038980cc54121fca1a7ce5a247759beee4807547bab49afc"},
}


def sources_sha256(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(kernel: str, workload: str):
    """ncu DRAM bytes per launch, or None unless they were taken on this workload with the
    current kernel sources."""
    t = NCU_TRAFFIC.get(kernel)
    if not t or t["workload"] != workload or t["sources_sha256"] != sources_sha256(kernel):
        return None
    return t["bytes_per_launch"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ------------------------------------------------------------------------------------------
# algorithmic work of each kernel (bytes / FLOPs per launch)
# ------------------------------------------------------------------------------------------
def prefill_work(w, sel_counts=None):
    L, G, k, B, Hq, d, di = w.L, w.G, w.k, w.B, w.Hq, w.d, w.di
    nb = (L + B - 1) // B
    units = acc.units_prefill(L, G, B, k)
    hpg = Hq // G
    return {
        "index_flops": acc.index_flops_prefill(L, G, di, B),
        "attn_flops": acc.attn_flops_prefill(L, Hq, d, B, k),
        "units": units,
        # attention: gather the 16 query heads of every (token, group, block) unit, write its
        # fp16 partial O and (m, lse); K and V of every (group, block) once
        "attn_bytes": units * (hpg * d * 2 + hpg * d * 2 + hpg * 8) + G * nb * B * d * 2 * 2,
        # combine: read every partial and its (m, lse), the selection; write O and LSE
        "combine_bytes": units * (hpg * d * 2 + hpg * 8) + G * L * k * 4 + L * Hq * (d * 2 + 4),
    }


def decode_work(w, seq_lens, index_bytes=2):
    """Algorithmic bytes of one decode step: the scan reads every index key strictly before each
    query's page (plus the index queries); the attention reads K and V of the selected pages
    (the local page up to n) plus q and o.  index_bytes: bytes per index element (2 bf16, 1
    e4m3)."""
    lens = [int(n) for n in seq_lens]
    scan = acc.decode_index_bytes(lens, w.B, w.di, w.G) * index_bytes // 2
    attn = acc.decode_attn_bytes(lens, w.B, w.d, w.G, w.Hq, w.k)
    return {"scan_bytes": scan, "attn_bytes": attn}


# ------------------------------------------------------------------------------------------
# MSA arm
# ------------------------------------------------------------------------------------------
def run_msa(args, world, rank):
    import block_sparse_long_msa_gb300 as msa
    msa.lib()
    w = workload(args)
    assert w.kind == "prefill", "the bench step is the prefill pass"
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = synthetic.prefill_inputs(w, device=dev)
    cfg = msa.config(w.G, w.hpg, w.k, w.scale)
    L = w.L
    sel = torch.empty((w.G, L, w.k), dtype=torch.int32, device=dev)
    o = torch.empty((L, w.Hq, w.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.Hq, L), dtype=torch.float32, device=dev)
    ws_bytes = max(msa.msa_attn_prefill_workspace(cfg, L),
                   msa.msa_index_select_workspace(cfg, L, L))
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    nchunks = -(-L // msa.msa_prefill_chunk_tokens(cfg, L))
    launches_per_step = 1 + msa.msa_attn_prefill_launches(cfg, L)
    stream = torch.cuda.current_stream()

    def ev():
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)  # materialise the handle
        return e

    nmarks = 3 * nchunks + 1

    # ---- decode: one new token for each of the 64 sequences of the paged workload ----
    dw0 = synthetic.WORKLOADS[args.decode_workload]
    dinp = synthetic.decode_inputs(dw0, device=dev, batch=args.decode_batch or None,
                                   n_hi=args.decode_nmax or None)
    dw = dinp["workload"]
    dcfg = msa.config(dw.G, dw.hpg, dw.k, dw.scale)
    paged = msa.paged_kv(dinp["k_idx_pool"], dinp["k_pool"], dinp["v_pool"], dinp["page_table"],
                         dinp["seq_lens"])
    dsel = torch.empty((dw.G, dw.batch, dw.k), dtype=torch.int32, device=dev)
    do = torch.empty((dw.batch, dw.Hq, dw.d), dtype=torch.bfloat16, device=dev)
    dlse = torch.empty((dw.Hq, dw.batch), dtype=torch.float32, device=dev)
    dws = torch.zeros(max(msa.msa_index_select_workspace(dcfg, dw.batch, 0, paged),
                          msa.msa_attn_decode_workspace(dcfg, paged)), dtype=torch.uint8,
                      device=dev)
    dec_launches = 4

    def step(marks=None, start=None, dmarks=None):
        if start is not None:
            start.record(stream)
        msa.msa_index_select(cfg, inp["q_idx"], inp["k_idx"], sel=sel, ws=ws)
        msa.msa_attn_prefill(cfg, inp["q"], inp["k"], inp["v"], sel, o=o, lse=lse, ws=ws,
                             marks=marks)
        if dmarks is not None:
            dmarks[0].record(stream)
        msa.msa_index_select(dcfg, dinp["q_idx"], paged=paged, sel=dsel, ws=dws)
        if dmarks is not None:
            dmarks[1].record(stream)
        msa.msa_attn_decode(dcfg, dinp["q"], paged, dsel, o=do, lse=dlse, ws=dws)
        if dmarks is not None:
            dmarks[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = msa.msa_get_device_status(ws) or msa.msa_get_device_status(dws)
    if status != 0:
        raise RuntimeError(f"device status {status} after warm-up")

    starts = [ev() for _ in range(args.steps)]
    marks = [[ev() for _ in range(nmarks)] for _ in range(args.steps)]
    dmarks = [[ev() for _ in range(3)] for _ in range(args.steps)]
    t0, t1 = ev(), ev()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clocks:
        barrier(world)
        torch.cuda.synchronize()
        t0.record(stream)
        for s in range(args.steps):
            step(marks[s], starts[s], dmarks[s])
        t1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    total_ms = t0.elapsed_time(t1)
    total_ms = max_over_ranks(total_ms, world)

    phase = {"index": 0.0, "schedule": 0.0, "attention": 0.0, "combine": 0.0}
    for s in range(args.steps):
        m = marks[s]
        phase["index"] += starts[s].elapsed_time(m[0])
        for c in range(nchunks):
            phase["schedule"] += m[3 * c].elapsed_time(m[3 * c + 1])
            phase["attention"] += m[3 * c + 1].elapsed_time(m[3 * c + 2])
            phase["combine"] += m[3 * c + 2].elapsed_time(m[3 * c + 3])
    dec_sel_ms = sum(d[0].elapsed_time(d[1]) for d in dmarks) / args.steps
    dec_attn_ms = sum(d[1].elapsed_time(d[2]) for d in dmarks) / args.steps
    prefill_ms = sum(starts[s].elapsed_time(marks[s][-1]) for s in range(args.steps)) / args.steps
    dec_ms = dec_sel_ms + dec_attn_ms
    per_launch_ms = {"index": phase["index"] / args.steps,
                     "attention": phase["attention"] / (args.steps * nchunks),
                     "combine": phase["combine"] / (args.steps * nchunks)}

    work = prefill_work(w)
    peaks = load_peaks()
    tensor_peak = peaks["bf16_tflops"]
    roof = {
        "index": ("tensor", work["index_flops"] / (per_launch_ms["index"] * 1e-3) / 1e12,
                  tensor_peak, "TFLOP/s"),
        "attention": ("hbm", work["attn_bytes"] / nchunks / (per_launch_ms["attention"] * 1e-3)
                      / 1e9, peaks["hbm_gbs"], "GB/s"),
        "combine": ("hbm", work["combine_bytes"] / nchunks / (per_launch_ms["combine"] * 1e-3)
                    / 1e9, peaks["hbm_gbs"], "GB/s"),
    }
    dominant = max(("index", "attention", "combine"), key=lambda n: phase[n])
    bound, achieved, peak, unit = roof[dominant]
    traffic = measured_traffic(dominant, f"{w.name}@{L}")

    # ---------------- end-to-end through the public API from pinned host buffers ------------
    # Each step copies its inputs in from pinned host memory and its results out, through the
    # same public calls.  The prefill tensors are double-buffered on the device and the copies
    # run on their own streams, so step s+1's inputs arrive and step s-1's results leave while
    # step s computes; the decode step's small inputs and outputs travel on the compute stream.
    e2e_on = args.e2e_steps > 0
    pin = (lambda t: t.cpu().pin_memory()) if e2e_on else (lambda t: t[:0].cpu())
    names_in = ("q", "k", "v", "q_idx", "k_idx")
    host_in = {k: pin(inp[k]) for k in names_in}
    host_out = [pin(t) for t in (o, lse, sel)]
    nbuf = 2 if e2e_on else 1
    dev_in = [{k: torch.empty_like(inp[k]) if e2e_on else inp[k] for k in names_in}
              for _ in range(nbuf)]
    dev_out = [[torch.empty_like(t) if e2e_on else t for t in (o, lse, sel)] for _ in range(nbuf)]
    h2d = sum(inp[k].numel() * inp[k].element_size() for k in names_in)
    d2h = sum(t.numel() * t.element_size() for t in (o, lse, sel))

    dhost_in = {k: pin(dinp[k]) for k in ("q", "q_idx", "seq_lens", "page_table")}
    ddev_in = {k: dinp[k] for k in dhost_in}
    dhost_out = [pin(t) for t in (do, dlse, dsel)]
    h2d += sum(dinp[k].numel() * dinp[k].element_size() for k in dhost_in)
    d2h += sum(t.numel() * t.element_size() for t in (do, dlse, dsel))

    s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]      # inputs of buffer b landed
    ev_used = [torch.cuda.Event() for _ in range(nbuf)]    # compute done with buffer b
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]     # results of buffer b copied out

    def e2e_step(i):
        b = i % nbuf
        with torch.cuda.stream(s_h2d):
            if i >= nbuf:
                s_h2d.wait_event(ev_used[b])
            for k_, t in host_in.items():
                dev_in[b][k_].copy_(t, non_blocking=True)
            ev_in[b].record(s_h2d)
        stream.wait_event(ev_in[b])
        if i >= nbuf:
            stream.wait_event(ev_out[b])
        ob, lb, sb = dev_out[b]
        di = dev_in[b]
        msa.msa_index_select(cfg, di["q_idx"], di["k_idx"], sel=sb, ws=ws, stream=stream)
        msa.msa_attn_prefill(cfg, di["q"], di["k"], di["v"], sb, o=ob, lse=lb, ws=ws,
                             stream=stream)
        for k_, t in dhost_in.items():
            ddev_in[k_].copy_(t, non_blocking=True)
        msa.msa_index_select(dcfg, ddev_in["q_idx"], paged=paged, sel=dsel, ws=dws,
                             stream=stream)
        msa.msa_attn_decode(dcfg, ddev_in["q"], paged, dsel, o=do, lse=dlse, ws=dws,
                            stream=stream)
        for hd, t in zip(dhost_out, (do, dlse, dsel)):
            hd.copy_(t, non_blocking=True)
        ev_used[b].record(stream)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(ev_used[b])
            for hd, t in zip(host_out, dev_out[b]):
                hd.copy_(t, non_blocking=True)
            ev_out[b].record(s_d2h)

    e2e_ms = None
    if args.e2e_steps > 0:
        for i in range(2 * nbuf):
            e2e_step(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        e0.record(s_h2d)  # the first operation of the timed region
        for i in range(args.e2e_steps):
            e2e_step(i)
        s_d2h.wait_stream(stream)
        e1.record(s_d2h)  # after the last copy out, which follows everything else
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
        # the pipelined step computed the same selection as the resident-input step
        assert torch.equal(host_out[2], sel.cpu()), "end-to-end selection differs"
    status = msa.msa_get_device_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {status} after timed region")

    # ---- e4m3 index vectors (the FP8 indexer, tcgen05 kind::f8f6f4): the integer/8 index
    # inputs are exact in e4m3, so the selections must equal the bf16 ones; the two index
    # kernels are timed alone and the step throughputs recomputed with their times ----
    e4m3 = None
    if not args.no_e4m3_index:
        f8 = torch.float8_e4m3fn
        q8, k8 = inp["q_idx"].to(f8), inp["k_idx"].to(f8)
        dq8, dk8 = dinp["q_idx"].to(f8), dinp["k_idx_pool"].to(f8)
        cfg8 = msa.config(w.G, w.hpg, w.k, w.scale, index_dtype="e4m3")
        dcfg8 = msa.config(dw.G, dw.hpg, dw.k, dw.scale, index_dtype="e4m3")
        paged8 = msa.paged_kv(dk8, dinp["k_pool"], dinp["v_pool"], dinp["page_table"],
                              dinp["seq_lens"])
        sel8, dsel8 = torch.empty_like(sel), torch.empty_like(dsel)

        def timed(fn, n):
            for _ in range(max(3, args.warmup)):
                fn()
            a0, a1 = ev(), ev()
            torch.cuda.synchronize()
            a0.record(stream)
            for _ in range(n):
                fn()
            a1.record(stream)
            torch.cuda.synchronize()
            return a0.elapsed_time(a1) / n

        n8 = max(3, args.steps)
        idx8_ms = timed(lambda: msa.msa_index_select(cfg8, q8, k8, sel=sel8, ws=ws), n8)
        didx8_ms = timed(lambda: msa.msa_index_select(dcfg8, dq8, paged=paged8, sel=dsel8,
                                                      ws=dws), n8)
        msa.msa_index_select(cfg, inp["q_idx"], inp["k_idx"], sel=sel, ws=ws)
        msa.msa_index_select(dcfg, dinp["q_idx"], paged=paged, sel=dsel, ws=dws)
        torch.cuda.synchronize()
        assert torch.equal(sel8, sel) and torch.equal(dsel8, dsel), "e4m3 selection differs"
        idx16_ms = phase["index"] / args.steps
        pre8_ms = prefill_ms - idx16_ms + idx8_ms
        dec8_ms = dec_attn_ms + didx8_ms
        scan8_bytes = decode_work(dw, dinp["seq_lens"].tolist(), index_bytes=1)["scan_bytes"]
        e4m3 = {
            "note": "index vectors in e4m3 (exact for the integer/8 inputs: same selections, "
                    "asserted); the main branch is unchanged, so the step times below are the "
                    "measured bf16 steps with the e4m3 index kernels' measured times in place "
                    "of the bf16 ones",
            "prefill_index_ms": idx8_ms, "prefill_index_ms_bf16": idx16_ms,
            "prefill_index_tflops": work["index_flops"] / (idx8_ms * 1e-3) / 1e12,
            "prefill_index_frac_of_fp8_peak": work["index_flops"] / (idx8_ms * 1e-3) / 1e12
                                              / (2 * tensor_peak),
            "prefill_tokens_per_s": world * L / (pre8_ms * 1e-3),
            "decode_index_ms": didx8_ms, "decode_index_ms_bf16": dec_sel_ms,
            "decode_scan_gbs": scan8_bytes / (didx8_ms * 1e-3) / 1e9,
            "traffic": {"prefill_index": measured_traffic("index_e4m3", f"{w.name}@{L}"),
                        "decode_scan": measured_traffic("decode_scan_e4m3",
                                                        f"{dw.name}@{dw.batch}x{dw.n_hi}")},
            "decode_tokens_per_s": world * dw.batch / (dec8_ms * 1e-3),
            "gpu_launches": 3 * n8,
        }

    # ---- block-score export (the indexer's KL alignment input): the same index kernels also
    # write every block's pooled score, [G][L][nb] for prefill, [G][batch][max_pages] for decode;
    # timed alone, against the selection-only launch of the same kernels ----
    scores = None
    if not args.no_index_scores:
        def timed_alone(fn, n):
            for _ in range(max(3, args.warmup)):
                fn()
            a0, a1 = ev(), ev()
            torch.cuda.synchronize()
            a0.record(stream)
            for _ in range(n):
                fn()
            a1.record(stream)
            torch.cuda.synchronize()
            return a0.elapsed_time(a1) / n

        nsc = max(3, args.steps)
        nb = (L + w.B - 1) // w.B
        bs = torch.empty((w.G, L, nb), dtype=torch.float32, device=dev)
        dbs = torch.empty((dw.G, dw.batch, dinp["max_pages"]), dtype=torch.float32, device=dev)
        sel_s, dsel_s = torch.empty_like(sel), torch.empty_like(dsel)
        sc_ms = timed_alone(lambda: msa.msa_index_select_scores(
            cfg, inp["q_idx"], inp["k_idx"], sel=sel_s, block_scores=bs, ws=ws, stream=stream),
            nsc)
        plain_ms = timed_alone(lambda: msa.msa_index_select(
            cfg, inp["q_idx"], inp["k_idx"], sel=sel, ws=ws, stream=stream), nsc)
        dsc_ms = timed_alone(lambda: msa.msa_index_select_scores(
            dcfg, dinp["q_idx"], paged=paged, sel=dsel_s, block_scores=dbs, ws=dws,
            stream=stream), nsc)
        dplain_ms = timed_alone(lambda: msa.msa_index_select(
            dcfg, dinp["q_idx"], paged=paged, sel=dsel, ws=dws, stream=stream), nsc)
        assert torch.equal(sel_s, sel) and torch.equal(dsel_s, dsel), "score export selection"
        out_b, dout_b = bs.numel() * 4, dbs.numel() * 4
        scores = {
            "note": "msa_index_select_scores: the index kernels also write every block's pooled "
                    "score (+inf own block, -inf later blocks); each timed alone, back to back, "
                    "beside the selection-only launch of the same kernels",
            "prefill_ms": sc_ms, "prefill_ms_select_only": plain_ms,
            "prefill_output_bytes": out_b,
            "prefill_extra_gbs": out_b / max(sc_ms - plain_ms, 1e-6) / 1e6,
            "decode_ms": dsc_ms, "decode_ms_select_only": dplain_ms,
            "decode_output_bytes": dout_b,
            "gpu_launches": 2 * nsc + 4 * nsc,
        }
        del bs, dbs

    # ---- the L = 2,048 prefill pass (launch-bound: eight short kernels) eager and as a replay of
    # a CUDA graph captured from the same calls (the library enqueues only, so it captures) ----
    graph = None
    if not args.no_graph:
        tw = synthetic.WORKLOADS["tiny_L2048"]
        tinp = synthetic.prefill_inputs(tw, device=dev)
        tcfg = msa.config(tw.G, tw.hpg, tw.k, tw.scale)
        tws_i = torch.zeros(msa.msa_index_select_workspace(tcfg, tw.L, tw.L), dtype=torch.uint8,
                            device=dev)
        tws_a = torch.zeros(msa.msa_attn_prefill_workspace(tcfg, tw.L), dtype=torch.uint8,
                            device=dev)
        tsel = torch.empty((tw.G, tw.L, tw.k), dtype=torch.int32, device=dev)
        to = torch.empty_like(tinp["q"])
        tlse = torch.empty((tw.Hq, tw.L), dtype=torch.float32, device=dev)

        def tiny_pass():
            msa.msa_index_select(tcfg, tinp["q_idx"], tinp["k_idx"], sel=tsel, ws=tws_i)
            msa.msa_attn_prefill(tcfg, tinp["q"], tinp["k"], tinp["v"], tsel, o=to, lse=tlse,
                                 ws=tws_a)

        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(3):
                tiny_pass()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg):
            tiny_pass()
        ntiny = 50

        def timed_cur(fn):
            for _ in range(3):
                fn()
            a0, a1 = ev(), ev()
            torch.cuda.synchronize()
            a0.record()
            for _ in range(ntiny):
                fn()
            a1.record()
            torch.cuda.synchronize()
            return a0.elapsed_time(a1) / ntiny

        eager_ms = timed_cur(tiny_pass)
        graph_ms = timed_cur(cg.replay)
        graph = {
            "workload": tw.name, "L": tw.L,
            "note": "index select + main branch of the small workload, back to back (inputs of "
                    "8 MiB stay in L2); eager calls against a replay of a CUDA graph captured "
                    "from the same calls",
            "eager_ms": eager_ms, "graph_ms": graph_ms,
            "tokens_per_s_eager": tw.L / (eager_ms * 1e-3),
            "tokens_per_s_graph": tw.L / (graph_ms * 1e-3),
            "launches_per_pass": 1 + msa.msa_attn_prefill_launches(tcfg, tw.L),
        }
        del cg

    cpu_base = None
    dec_cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_base = cpu_baseline(w, {k: inp[k].cpu() for k in ("q", "k", "v", "q_idx", "k_idx")},
                                target_s=15.0)
        dec_cpu = decode_cpu_baseline(dw, dinp)

    ms_per_step = total_ms / args.steps
    prefill_ms = max_over_ranks(prefill_ms, world)
    dec_ms = max_over_ranks(dec_ms, world)
    value = world * L / (prefill_ms * 1e-3)
    dwork = decode_work(dw, dinp["seq_lens"].tolist())
    dec_scan_gbs = dwork["scan_bytes"] / (dec_sel_ms * 1e-3) / 1e9
    dec_attn_gbs = dwork["attn_bytes"] / (dec_attn_ms * 1e-3) / 1e9
    dec_step_gbs = (dwork["scan_bytes"] + dwork["attn_bytes"]) / (dec_ms * 1e-3) / 1e9
    decode = {
        "metric": "MSA paged decode tokens/s (one new token per sequence per step)",
        "value": world * dw.batch / (dec_ms * 1e-3), "unit": "tokens/s",
        "ms_per_step": dec_ms,
        "config": {"workload": dw.name, "batch": dw.batch, "n_min": dw.n_lo, "n_max": dw.n_hi,
                   "context_tokens": int(dinp["seq_lens"].sum().item()), "Hq": dw.Hq,
                   "G": dw.G, "k": dw.k, "pages": dinp["num_pages"]},
        "phases_ms_per_step": {"index_select": dec_sel_ms, "attention": dec_attn_ms},
        "roofline": {"bound": "hbm", "kernel": "index page scan (+ top-k merge)",
                     "achieved": dec_scan_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": dec_scan_gbs / peaks["hbm_gbs"],
                     "traffic": measured_traffic("decode_scan",
                                                 f"{dw.name}@{dw.batch}x{dw.n_hi}"),
                     "peak_source": peaks["source"]},
        "attention_roofline": {"bound": "hbm", "achieved": dec_attn_gbs, "peak": peaks["hbm_gbs"],
                               "unit": "GB/s", "frac": dec_attn_gbs / peaks["hbm_gbs"]},
        "step_hbm_frac": dec_step_gbs / peaks["hbm_gbs"],
        "algorithmic_bytes": dwork,
        "gpu_launches": dec_launches * args.steps,
        "cpu_baseline": None,
    }
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded SplitMix64; N(0,1) q/k/v, integer/8 index q/k)",
        "config": {"workload": w.name, "L": L, "Hq": w.Hq, "G": w.G, "d": w.d, "B": w.B,
                   "k": w.k, "parallelism": f"replicas x{world}",
                   "step": "prefill (index select + main branch over all L queries) + one paged "
                           "decode step of the 64-sequence workload; value = prefill tokens/s",
                   "l2": f"inputs larger than L2 (q {L * w.Hq * w.d * 2 / 2**20:.0f} MiB) and "
                         f"{work['units'] * w.hpg * (w.d * 2 + 8) / 2**30:.1f} GiB of partials "
                         f"per step"},
        "phases_ms_per_step": {k: v / args.steps for k, v in phase.items()},
        "prefill_ms_per_step": prefill_ms,
        "gpu_launches": (launches_per_step + dec_launches) * args.steps,
        "roofline": {"bound": bound, "kernel": dominant, "achieved": achieved, "peak": peak,
                     "unit": unit, "frac": achieved / peak, "traffic": traffic,
                     "peak_source": peaks["source"]},
        "kernel_rooflines": {n: {"bound": r[0], "achieved": r[1], "peak": r[2], "unit": r[3],
                                 "frac": r[1] / r[2], "ms_per_launch": per_launch_ms[n]}
                             for n, r in roof.items()},
        "tensor_frac_main_branch": work["attn_flops"] / ((phase["attention"] + phase["combine"]
                                                          + phase["schedule"]) / args.steps
                                                         * 1e-3) / 1e12 / tensor_peak,
        "e2e": None if e2e_ms is None else {
                "value": world * L * args.e2e_steps / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": "prefill tokens over the whole step (prefill + decode) with every step's "
                        "inputs copied from pinned host memory and its outputs copied back, on "
                        "copy streams of their own (device buffers doubled, so the copies of "
                        "neighbouring steps overlap the compute); the decode KV cache is "
                        "resident state"},
        "clocks": clocks.summary(),
        "cpu_baseline": cpu_base,
        "decode": decode,
    }
    line["decode"]["cpu_baseline"] = dec_cpu
    line["e4m3_index"] = e4m3
    line["index_scores"] = scores
    line["cuda_graph"] = graph
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------
# CPU oracle timing (the reference arm, and the cpu_baseline of the MSA arm)
# ------------------------------------------------------------------------------------------
def _oracle_rows(w, inp, rows):
    import oracle
    t = time.perf_counter()
    sel = oracle.select_prefill(inp["q_idx"], inp["k_idx"], w.B, w.k, rows=rows)
    oracle.attn_prefill(inp["q"], inp["k"], inp["v"], sel, w.B, w.k, w.scale, rows=rows)
    return time.perf_counter() - t


def _strided_rows(L, n, phase=0):
    import numpy as np
    n = max(1, min(L, n))
    return (np.arange(n, dtype=np.int64) * L // n + phase) % L


def cpu_baseline(w, inp, target_s=15.0):
    import oracle
    oracle.build()
    n = 64
    dt = _oracle_rows(w, inp, _strided_rows(w.L, n))
    n2 = int(min(w.L, max(n, n * target_s / max(dt, 1e-3))))
    rows = _strided_rows(w.L, n2, 1)
    dt2 = _oracle_rows(w, inp, rows)
    return {"value": len(rows) / dt2, "unit": "tokens/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{len(rows)} evenly strided query rows of the L={w.L} workload "
                      f"(index selection + attention for all {w.G} groups / {w.Hq} heads), "
                      f"{dt2:.1f} s"}


def decode_cpu_baseline(w, dinp, target_s=10.0):
    """Oracle decode of all the workload's sequences, repeated to about target_s of CPU work.

    The index-key pages of every sequence are copied to the host; after the oracle's selection
    only the selected K/V pages are (the full pools do not fit the host).  Copies are untimed.
    """
    import oracle
    oracle.build()
    pt = dinp["page_table"].cpu()
    seq = dinp["seq_lens"].cpu()
    used = sorted({int(p) for p in pt.flatten().tolist() if p >= 0})
    remap = torch.zeros((dinp["num_pages"],), dtype=torch.int32)
    remap[torch.tensor(used)] = torch.arange(len(used), dtype=torch.int32)
    kip = dinp["k_idx_pool"].index_select(0, torch.tensor(used, device=dinp["k_idx_pool"].device)).cpu()
    pt2 = torch.where(pt >= 0, remap[pt.clamp(min=0).long()], torch.zeros_like(pt))
    q, qi = dinp["q"].cpu(), dinp["q_idx"].cpu()
    t = time.perf_counter()
    sel = oracle.select_decode(qi, kip, pt2, seq, w.B, w.k)
    t_sel = time.perf_counter() - t
    # the selected pages only, renumbered
    chosen = sorted({int(pt2[s_, b_]) for g in range(w.G) for s_ in range(sel.shape[1])
                     for b_ in sel[g, s_] if b_ >= 0})
    remap2 = torch.zeros((len(used),), dtype=torch.int32)
    remap2[torch.tensor(chosen)] = torch.arange(len(chosen), dtype=torch.int32)
    orig = torch.tensor(used)[torch.tensor(chosen)].to(dinp["k_pool"].device)
    kp = dinp["k_pool"].index_select(0, orig).cpu()
    vp = dinp["v_pool"].index_select(0, orig).cpu()
    pt3 = remap2[pt2.long()]
    t = time.perf_counter()
    oracle.attn_decode(q, kp, vp, pt3, seq, sel, w.B, w.k, w.scale)
    t_attn = time.perf_counter() - t
    one = t_sel + t_attn
    reps = int(max(1, min(20, round(target_s / max(one, 1e-3)))))
    total = one
    for _ in range(reps - 1):
        t = time.perf_counter()
        oracle.select_decode(qi, kip, pt2, seq, w.B, w.k)
        oracle.attn_decode(q, kp, vp, pt3, seq, sel, w.B, w.k, w.scale)
        total += time.perf_counter() - t
    return {"value": w.batch * reps / total, "unit": "tokens/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"all {w.batch} sequences ({int(seq.sum())} context tokens: index scan over "
                      f"every page, attention over the selected pages) x {reps} repetitions, "
                      f"{total:.1f} s"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = workload(args)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = {k: v.cpu() for k, v in synthetic.prefill_inputs(w, device=dev).items()
           if isinstance(v, torch.Tensor)}
    budget_s = 150.0
    cal = _oracle_rows(w, inp, _strided_rows(w.L, 16))
    per_row = cal / 16
    rows_per_step = int(max(4, min(2048, budget_s / (args.steps + args.warmup) / per_row)))
    for s in range(args.warmup):
        _oracle_rows(w, inp, _strided_rows(w.L, rows_per_step, s + 1))
    total, n = 0.0, 0
    for s in range(args.steps):
        rows = _strided_rows(w.L, rows_per_step, args.warmup + s + 1)
        total += _oracle_rows(w, inp, rows)
        n += len(rows)
    value = n / total
    cb = {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
          "sample": f"{rows_per_step} evenly strided query rows per step of the L={w.L} "
                    "workload (index selection + attention, all groups and heads)"}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "L": w.L, "Hq": w.Hq, "G": w.G, "d": w.d, "B": w.B,
                   "k": w.k, "parallelism": "cpu oracle (rank 0 only)"},
        "impl": "reference", "cpu_baseline": cb,
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world, rank = dist_setup(args)
    if args.gpus != world and world > 1:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE {world}")
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_msa(args, world, rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
