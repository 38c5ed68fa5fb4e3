#!/usr/bin/env python
"""Benchmark of the MSA operator on GB300: prefill tokens/s with per-kernel roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl msa|reference] [--workload NAME]

A step is one full pass of the hot path over one batch of synthetic input resident in HBM:
index selection (score + max-pool + top-k) followed by the main branch (scheduling, KV-outer
attention, combine) on the 64/4-head, L = 1,048,576 prefill workload with hot key blocks, then
one paged decode step of the 64-sequence workload (reported under "decode").  Prints ONE JSON line
(rank 0) with:
  value / roofline / kernel_rooflines / main_branch  prefill tokens/s and each kernel against the
                                                     measured peaks
  e2e                  the same step through the public API from pinned host buffers
  prefill_workloads    the L = 32,768 and L = 131,072 (clustered) prefills, each timed the same way
                       with its own rooflines and CPU baseline (and, for 32K, the block-score
                       export timed beside the selection-only kernels)
  e4m3_index           the same step timed with e4m3 index vectors (same selections, asserted)
  cuda_graph           the small prefill pass eager against a CUDA-graph replay of the same calls
  cpu_baseline         the CPU oracle on a bounded sample, on this host's cores

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
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="msa", choices=["msa", "reference"])
    p.add_argument("--workload", default="prefill_L1M_hot")
    p.add_argument("--sub-workloads", default="prefill_L32K,prefill_L128K_clustered",
                   help="other prefill workloads timed after the headline one (comma list)")
    p.add_argument("--scores-workload", default="prefill_L32K",
                   help="the sub-workload on which the block-score export is timed")
    p.add_argument("--decode-workload", default="decode_b64_16K_256K")
    p.add_argument("--decode-batch", type=int, default=0, help="override (profiling)")
    p.add_argument("--decode-nmax", type=int, default=0, help="override (profiling)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e4m3-index", action="store_true",
                   help="skip the step with e4m3 (FP8) index vectors")
    p.add_argument("--e4m3-steps", type=int, default=8)
    p.add_argument("--no-index-scores", action="store_true",
                   help="skip timing the index kernels with the block-score export")
    p.add_argument("--no-graph", action="store_true",
                   help="skip timing the small prefill pass as a CUDA-graph replay")
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--cp-shards", type=int, default=4,
                   help="shards of the context-parallel decode index branch (0: skip)")
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
# of the named kernel on the named workload.  A figure is reported only while the
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
    # index kernel: L=1,048,576 hot blocks and L=32,768 (profile_case, second launch)
    "index": [{"bytes_per_launch": 19651720704, "workload": "prefill_L1M_hot@1048576",
               "sources_sha256": "d543ec92396d5af3486dfe63ef914722bf2b38e8e2b854aa29aaafaf2933c155"},
              {"bytes_per_launch": 41905920, "workload": "prefill_L32K@32768",
               "sources_sha256": "d543ec92396d5af3486dfe63ef914722bf2b38e8e2b854aa29aaafaf2933c155"}],
    "index_e4m3": [{"bytes_per_launch": 6326164224, "workload": "prefill_L1M_hot@1048576",
                    "sources_sha256": "d543ec92396d5af3486dfe63ef914722bf2b38e8e2b854aa29aaafaf2933c155"},
                   {"bytes_per_launch": 21001216, "workload": "prefill_L32K@32768",
                    "sources_sha256": "d543ec92396d5af3486dfe63ef914722bf2b38e8e2b854aa29aaafaf2933c155"}],
    # attention and combine per launch (one query chunk): L=32,768 (its one chunk); L=131,072
    # (second chunk); L=1,048,576 (8th of 16 chunks, a middle one)
    "attention": [{"bytes_per_launch": 9905374976, "workload": "prefill_L32K@32768",
                   "sources_sha256": "91d4a0294468ac4a7479d9901505ceeb2e709ad276433f41e0b9e4dac012cbdb"},
                  {"bytes_per_launch": 20752672768, "workload": "prefill_L128K_clustered@131072",
                   "sources_sha256": "91d4a0294468ac4a7479d9901505ceeb2e709ad276433f41e0b9e4dac012cbdb"},
                  {"bytes_per_launch": 33455269120, "workload": "prefill_L1M_hot@1048576",
                   "sources_sha256": "91d4a0294468ac4a7479d9901505ceeb2e709ad276433f41e0b9e4dac012cbdb"}],
    "combine": [{"bytes_per_launch": 9193360896, "workload": "prefill_L32K@32768",
                 "sources_sha256": "91d4a0294468ac4a7479d9901505ceeb2e709ad276433f41e0b9e4dac012cbdb"},
                {"bytes_per_launch": 18667236096, "workload": "prefill_L128K_clustered@131072",
                 "sources_sha256": "91d4a0294468ac4a7479d9901505ceeb2e709ad276433f41e0b9e4dac012cbdb"},
                {"bytes_per_launch": 18936193792, "workload": "prefill_L1M_hot@1048576",
                 "sources_sha256": "91d4a0294468ac4a7479d9901505ceeb2e709ad276433f41e0b9e4dac012cbdb"}],
    # decode, 64 sequences of 16K-256K tokens
    "decode_scan": [{"bytes_per_launch": 2088173056, "workload": "decode_b64_16K_256K@64x262144",
                     "sources_sha256": "0f603e9e75afd96b62e8e789f25800aae524b40c7454c08370937806f2b45de6"}],
    "decode_scan_e4m3": [{"bytes_per_launch": 1047312896, "workload": "decode_b64_16K_256K@64x262144",
                          "sources_sha256": "0f603e9e75afd96b62e8e789f25800aae524b40c7454c08370937806f2b45de6"}],
}
# Tensor-pipe activity from the same captures (sm__pipe_tensor_cycles_active, % of elapsed
# cycles: a fraction of the part's nominal tensor rate at the clock of the moment).
NCU_TENSOR_PIPE = {
    "index": [{"pct": 71.59, "workload": "prefill_L1M_hot@1048576",
               "sources_sha256": "d543ec92396d5af3486dfe63ef914722bf2b38e8e2b854aa29aaafaf2933c155"},
              {"pct": 58.15, "workload": "prefill_L32K@32768",
               "sources_sha256": "d543ec92396d5af3486dfe63ef914722bf2b38e8e2b854aa29aaafaf2933c155"}],
    "index_e4m3": [{"pct": 46.5, "workload": "prefill_L1M_hot@1048576",
                    "sources_sha256": "d543ec92396d5af3486dfe63ef914722bf2b38e8e2b854aa29aaafaf2933c155"},
                   {"pct": 31.96, "workload": "prefill_L32K@32768",
                    "sources_sha256": "d543ec92396d5af3486dfe63ef914722bf2b38e8e2b854aa29aaafaf2933c155"}],
    # attention: ncu --set full at L=8,192 (the 32K kernel at a capture-sized length)
    "attention": [{"pct": 42.12, "workload": "prefill_L32K@8192",
                   "sources_sha256": "91d4a0294468ac4a7479d9901505ceeb2e709ad276433f41e0b9e4dac012cbdb"}],
}


def code_text(src: str) -> str:
    """The code of a C++/CUDA source without its comments and blank space, so that a change to
    the comments alone does not count as a change of the kernel.  String and character literals
    are kept whole (a // inside one is not a comment)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    lines = (" ".join(line.split()) for line in "".join(out).split("\n"))
    return "\n".join(line for line in lines if line)


def sources_sha256(kernel: str) -> str:
    """Hash of the code (comments left out) of the sources a kernel is built from."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(CSRC, f), encoding="utf-8") as fh:
            h.update(code_text(fh.read()).encode())
    return h.hexdigest()


def measured_traffic(kernel: str, workload: str):
    """ncu DRAM bytes per launch, or None unless they were taken on this workload with the
    current kernel sources."""
    for t in NCU_TRAFFIC.get(kernel, []):
        if t["workload"] == workload and t["sources_sha256"] == sources_sha256(kernel):
            return t["bytes_per_launch"]
    return None


def measured_tensor_pipe(kernel: str, workload: str = None):
    """ncu tensor-pipe activity (% of elapsed cycles) with the workload it was taken on, for
    the current kernel sources: the given workload's if there is one, else any."""
    found = [t for t in NCU_TENSOR_PIPE.get(kernel, [])
             if t["sources_sha256"] == sources_sha256(kernel)]
    for t in found:
        if t["workload"] == workload:
            return {"pct_of_elapsed": t["pct"], "workload": t["workload"]}
    return {"pct_of_elapsed": found[0]["pct"], "workload": found[0]["workload"]} if found else None


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


def decode_work(w, seq_lens, index_bytes=2, kv_bytes=2):
    """Algorithmic bytes of one decode step: the scan reads every index key strictly before each
    query's page (plus the index queries); the attention reads K and V of the selected pages
    (the local page up to n) plus q and o.  index_bytes / kv_bytes: bytes per element of the
    index keys and of the K/V pools (2 bf16, 1 e4m3)."""
    lens = [int(n) for n in seq_lens]
    scan = acc.decode_index_bytes(lens, w.B, w.di, w.G) * index_bytes // 2
    attn = acc.decode_attn_bytes(lens, w.B, w.d, w.G, w.Hq, w.k, kv_bytes=kv_bytes)
    return {"scan_bytes": scan, "attn_bytes": attn}


# ------------------------------------------------------------------------------------------
# MSA arm
# ------------------------------------------------------------------------------------------
def _event(stream):
    e = torch.cuda.Event(enable_timing=True)
    e.record(stream)  # materialise the handle
    return e


class PrefillCase:
    """Device inputs, outputs and workspace of one prefill workload, and the calls of a pass."""

    def __init__(self, msa, w, dev, index_dtype="bf16"):
        self.msa, self.w = msa, w
        self.inp = synthetic.prefill_inputs(w, device=dev, index_dtype=index_dtype)
        self.cfg = msa.config(w.G, w.hpg, w.k, w.scale, index_dtype=index_dtype)
        L = w.L
        self.sel = torch.empty((w.G, L, w.k), dtype=torch.int32, device=dev)
        self.o = torch.empty((L, w.Hq, w.d), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((w.Hq, L), dtype=torch.float32, device=dev)
        self.ws = torch.zeros(max(msa.msa_attn_prefill_workspace(self.cfg, L),
                                  msa.msa_index_select_workspace(self.cfg, L, L)),
                              dtype=torch.uint8, device=dev)
        self.nchunks = -(-L // msa.msa_prefill_chunk_tokens(self.cfg, L))
        self.launches = 1 + msa.msa_attn_prefill_launches(self.cfg, L)

    def nmarks(self):
        return 3 * self.nchunks + 1

    def run(self, marks=None, start=None, stream=None, cfg_index=None, q_idx=None, k_idx=None):
        """Index selection, then the main branch.  cfg_index/q_idx/k_idx: another encoding of
        the same index vectors (the e4m3 indexer)."""
        if start is not None:
            start.record(stream)
        self.msa.msa_index_select(cfg_index or self.cfg,
                                  self.inp["q_idx"] if q_idx is None else q_idx,
                                  self.inp["k_idx"] if k_idx is None else k_idx, sel=self.sel,
                                  ws=self.ws, stream=stream)
        self.msa.msa_attn_prefill(self.cfg, self.inp["q"], self.inp["k"], self.inp["v"],
                                  self.sel, o=self.o, lse=self.lse, ws=self.ws, stream=stream,
                                  marks=marks)

    def phases(self, starts, marks):
        """Per-step milliseconds of each phase, from the events of run(marks, start)."""
        n = len(starts)
        ph = {"index": 0.0, "schedule": 0.0, "attention": 0.0, "combine": 0.0, "prefill": 0.0}
        for s in range(n):
            m = marks[s]
            ph["index"] += starts[s].elapsed_time(m[0])
            for c in range(self.nchunks):
                ph["schedule"] += m[3 * c].elapsed_time(m[3 * c + 1])
                ph["attention"] += m[3 * c + 1].elapsed_time(m[3 * c + 2])
                ph["combine"] += m[3 * c + 2].elapsed_time(m[3 * c + 3])
            ph["prefill"] += starts[s].elapsed_time(m[-1])
        return {k: v / n for k, v in ph.items()}


class DecodeCase:
    """The paged decode workload: one new token for each sequence."""

    def __init__(self, msa, dw0, dev, batch=None, n_hi=None, index_dtype="bf16"):
        self.msa = msa
        self.inp = synthetic.decode_inputs(dw0, device=dev, batch=batch, n_hi=n_hi,
                                           index_dtype=index_dtype)
        dw = self.w = self.inp["workload"]
        self.cfg = msa.config(dw.G, dw.hpg, dw.k, dw.scale, index_dtype=index_dtype)
        self.paged = msa.paged_kv(self.inp["k_idx_pool"], self.inp["k_pool"], self.inp["v_pool"],
                                  self.inp["page_table"], self.inp["seq_lens"])
        self.sel = torch.empty((dw.G, dw.batch, dw.k), dtype=torch.int32, device=dev)
        self.o = torch.empty((dw.batch, dw.Hq, dw.d), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((dw.Hq, dw.batch), dtype=torch.float32, device=dev)
        self.ws = torch.zeros(max(msa.msa_index_select_workspace(self.cfg, dw.batch, 0,
                                                                 self.paged),
                                  msa.msa_attn_decode_workspace(self.cfg, self.paged)),
                              dtype=torch.uint8, device=dev)
        self.launches = 4

    def with_encoding(self, cfg, k_idx_pool, k_pool, v_pool):
        self.cfg = cfg
        self.paged = self.msa.paged_kv(k_idx_pool, k_pool, v_pool, self.inp["page_table"],
                                       self.inp["seq_lens"])
        return self

    def run(self, marks=None, stream=None, q_idx=None):
        if marks is not None:
            marks[0].record(stream)
        self.msa.msa_index_select(self.cfg, self.inp["q_idx"] if q_idx is None else q_idx,
                                  paged=self.paged, sel=self.sel, ws=self.ws, stream=stream)
        if marks is not None:
            marks[1].record(stream)
        self.msa.msa_attn_decode(self.cfg, self.inp["q"], self.paged, self.sel, o=self.o,
                                 lse=self.lse, ws=self.ws, stream=stream)
        if marks is not None:
            marks[2].record(stream)


def check_status(msa, *wss):
    for ws in wss:
        st = msa.msa_get_device_status(ws)
        if st != 0:
            raise RuntimeError(f"device status {st}")


def prefill_report(w, ph, nchunks, peaks, index_kernel="index"):
    """Rooflines of one prefill pass from its per-step phase times (ms).

    The index kernel and the attention kernel are contractions: their achieved rate is their
    algorithmic FLOPs over their time, against the bf16 tensor peak (burst for passes of a few
    milliseconds, sustained for passes that run for tenths of a second and more, as the long
    step keeps the part at its power limit).  The attention's HBM rate of its algorithmic bytes
    is given beside it; the combine is a stream over the partials (HBM)."""
    work = prefill_work(w)
    long_pass = ph["prefill"] >= 50.0
    t_peak = peaks["bf16_tflops_sustained"] if long_pass else peaks["bf16_tflops"]
    t_kind = "sustained" if long_pass else "burst"
    main_ms = ph["schedule"] + ph["attention"] + ph["combine"]
    idx_tf = work["index_flops"] / (ph["index"] * 1e-3) / 1e12
    att_tf = work["attn_flops"] / (ph["attention"] * 1e-3) / 1e12
    att_gbs = work["attn_bytes"] / (ph["attention"] * 1e-3) / 1e9
    com_gbs = work["combine_bytes"] / (ph["combine"] * 1e-3) / 1e9
    main_tf = work["attn_flops"] / (main_ms * 1e-3) / 1e12

    def tensor(a):
        return {"bound": "tensor", "achieved": a, "peak": t_peak, "unit": "TFLOP/s",
                "frac": a / t_peak, "peak_kind": t_kind,
                "frac_of_burst": a / peaks["bf16_tflops"],
                "frac_of_sustained": a / peaks["bf16_tflops_sustained"]}

    wl = f"{w.name}@{w.L}"
    kernels = {
        "index": {**tensor(idx_tf), "ms_per_launch": ph["index"],
                  "algorithmic_flops": work["index_flops"],
                  "ncu_tensor_pipe": measured_tensor_pipe(index_kernel, wl)},
        "attention": {**tensor(att_tf), "ms_per_launch": ph["attention"] / nchunks,
                      "algorithmic_flops": work["attn_flops"],
                      "ncu_tensor_pipe": measured_tensor_pipe("attention", wl),
                      "ncu_traffic_per_launch": measured_traffic("attention", wl),
                      "hbm_gbs_of_algorithmic_bytes": att_gbs,
                      "hbm_frac": att_gbs / peaks["hbm_gbs"],
                      "algorithmic_bytes": work["attn_bytes"]},
        "combine": {"bound": "hbm", "achieved": com_gbs, "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": com_gbs / peaks["hbm_gbs"],
                    "ms_per_launch": ph["combine"] / nchunks,
                    "algorithmic_bytes": work["combine_bytes"],
                    "ncu_traffic_per_launch": measured_traffic("combine", wl)},
    }
    main = {**tensor(main_tf), "ms": main_ms,
            "note": "attention FLOPs over schedule + attention + combine time"}
    dominant = max(("index", "attention", "combine"), key=lambda n: ph[n])
    return work, kernels, main, dominant


def prefill_object(case, ph, peaks, world, steps, index_kernel="index"):
    w = case.w
    work, kernels, main, dominant = prefill_report(w, ph, case.nchunks, peaks, index_kernel)
    dk = kernels[dominant]
    traffic = measured_traffic(index_kernel if dominant == "index" else dominant,
                               f"{w.name}@{w.L}")
    roof = {"bound": dk["bound"], "kernel": dominant, "achieved": dk["achieved"],
            "peak": dk["peak"], "unit": dk["unit"], "frac": dk["frac"],
            "traffic": traffic,
            "peak_source": peaks["source"]}
    return {
        "workload": w.name, "L": w.L,
        "value": world * w.L / (ph["prefill"] * 1e-3), "unit": "tokens/s",
        "ms_per_pass": ph["prefill"],
        "phases_ms_per_pass": {k: ph[k] for k in ("index", "schedule", "attention", "combine")},
        "query_chunks": case.nchunks,
        "roofline": roof,
        "kernel_rooflines": kernels,
        "main_branch": main,
        "gpu_launches": case.launches * steps,
    }


def decode_object(dc, ph, peaks, world, steps, index_bytes=2, kv_bytes=2):
    dw = dc.w
    dwork = decode_work(dw, dc.inp["seq_lens"].tolist(), index_bytes=index_bytes,
                        kv_bytes=kv_bytes)
    sel_ms, att_ms = ph["index_select"], ph["attention"]
    step_ms = sel_ms + att_ms
    scan_gbs = dwork["scan_bytes"] / (sel_ms * 1e-3) / 1e9
    att_gbs = dwork["attn_bytes"] / (att_ms * 1e-3) / 1e9
    step_gbs = (dwork["scan_bytes"] + dwork["attn_bytes"]) / (step_ms * 1e-3) / 1e9
    scan_kernel = "decode_scan" if index_bytes == 2 else "decode_scan_e4m3"
    return {
        "metric": "MSA paged decode tokens/s (one new token per sequence per step)",
        "value": world * dw.batch / (step_ms * 1e-3), "unit": "tokens/s",
        "ms_per_step": step_ms,
        "config": {"workload": dw.name, "batch": dw.batch, "n_min": dw.n_lo, "n_max": dw.n_hi,
                   "context_tokens": int(dc.inp["seq_lens"].sum().item()), "Hq": dw.Hq,
                   "G": dw.G, "k": dw.k, "pages": dc.inp["num_pages"],
                   "index_dtype": "bf16" if index_bytes == 2 else "e4m3",
                   "kv_dtype": "bf16" if kv_bytes == 2 else "e4m3"},
        "phases_ms_per_step": {"index_select": sel_ms, "attention": att_ms},
        "roofline": {"bound": "hbm", "kernel": "index page scan (+ top-k merge)",
                     "achieved": scan_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": scan_gbs / peaks["hbm_gbs"],
                     "frac_vs_8TBs": scan_gbs / 8000.0,
                     "traffic": measured_traffic(scan_kernel,
                                                 f"{dw.name}@{dw.batch}x{dw.n_hi}"),
                     "peak_source": peaks["source"]},
        "attention_roofline": {"bound": "hbm", "achieved": att_gbs, "peak": peaks["hbm_gbs"],
                               "unit": "GB/s", "frac": att_gbs / peaks["hbm_gbs"],
                               "frac_vs_8TBs": att_gbs / 8000.0},
        "step_hbm_frac": step_gbs / peaks["hbm_gbs"],
        "step_hbm_frac_vs_8TBs": step_gbs / 8000.0,
        "hbm_frac_headline": "frac: against the measured copy bandwidth of this GPU; "
                             "frac_vs_8TBs: against a nominal 8 TB/s",
        "algorithmic_bytes": dwork,
        "gpu_launches": dc.launches * steps,
        "cpu_baseline": None,
    }


def time_prefill_decode(case, dc, steps, warmup, world, stream, clocks=False, **kw):
    """Warm-up, then `steps` timed steps of prefill (+ decode when dc is given).  Returns the
    total milliseconds (max over ranks), the prefill phases, the decode phases and the clock
    summary (when asked)."""
    def step(marks=None, start=None, dmarks=None):
        case.run(marks=marks, start=start, stream=stream, **kw)
        if dc is not None:
            dc.run(marks=dmarks, stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    check_status(case.msa, case.ws, *([dc.ws] if dc is not None else []))
    starts = [_event(stream) for _ in range(steps)]
    marks = [[_event(stream) for _ in range(case.nmarks())] for _ in range(steps)]
    dmarks = [[_event(stream) for _ in range(3)] for _ in range(steps)]
    t0, t1 = _event(stream), _event(stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device()) if clocks else None
    if sampler:
        sampler.__enter__()
    barrier(world)
    torch.cuda.synchronize()
    t0.record(stream)
    for s in range(steps):
        step(marks[s], starts[s], dmarks[s] if dc is not None else None)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    if sampler:
        sampler.__exit__(None, None, None)
    check_status(case.msa, case.ws, *([dc.ws] if dc is not None else []))
    total_ms = max_over_ranks(t0.elapsed_time(t1), world)
    ph = case.phases(starts, marks)
    ph = {k: max_over_ranks(v, world) for k, v in ph.items()}
    dph = None
    if dc is not None:
        dph = {"index_select": sum(d[0].elapsed_time(d[1]) for d in dmarks) / steps,
               "attention": sum(d[1].elapsed_time(d[2]) for d in dmarks) / steps}
        dph = {k: max_over_ranks(v, world) for k, v in dph.items()}
    return total_ms, ph, dph, (sampler.summary() if sampler else None)


def host_memory_available():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def e2e_leg(msa, case, dc, steps, world, stream):
    """The same step through the public API with every step's inputs copied in from pinned host
    memory and its results copied back (inside the timed region).  All tensors a step copies
    (prefill and decode) are double-buffered on the device, and every copy runs on one of two
    copy streams, so step s+1's inputs arrive and step s-1's results leave while step s
    computes, and no copy waits in a copy engine's queue in front of the compute stream.
    Returns (ms, h2d bytes, d2h bytes, clocks sampled over the timed steps)."""
    names_in = ("q", "k", "v", "q_idx", "k_idx")
    dnames = ("q", "q_idx", "seq_lens", "page_table")
    inp = case.inp
    outs = (case.o, case.lse, case.sel)
    douts = (dc.o, dc.lse, dc.sel)
    h2d = sum(inp[k].numel() * inp[k].element_size() for k in names_in)
    h2d += sum(dc.inp[k].numel() * dc.inp[k].element_size() for k in dnames)
    d2h = sum(t.numel() * t.element_size() for t in outs + douts)

    def pinned_copy(t):
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        return h

    host_in = {k: pinned_copy(inp[k]) for k in names_in}
    dhost_in = {k: pinned_copy(dc.inp[k]) for k in dnames}
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs + douts]
    dev_in = [{**{k: inp[k] for k in names_in}, **{"d_" + k: dc.inp[k] for k in dnames}},
              {**{k: torch.empty_like(inp[k]) for k in names_in},
               **{"d_" + k: torch.empty_like(dc.inp[k]) for k in dnames}}]
    dev_out = [list(outs + douts), [torch.empty_like(t) for t in outs + douts]]
    pagedb = [msa.paged_kv(dc.inp["k_idx_pool"], dc.inp["k_pool"], dc.inp["v_pool"],
                           dev_in[b]["d_page_table"], dev_in[b]["d_seq_lens"]) for b in range(2)]
    s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_used = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    cfg = case.cfg

    c_marks = []  # per timed step: compute start and end on the compute stream
    h_marks, d_marks = [], []  # per timed step: its copies in, its copies out

    def e2e_step(i, mark=False):
        b = i % 2
        with torch.cuda.stream(s_h2d):
            if i >= 2:
                s_h2d.wait_event(ev_used[b])
            if mark:
                h_marks.append((_event(s_h2d), _event(s_h2d)))
                h_marks[-1][0].record(s_h2d)
            for k_, t in dhost_in.items():
                dev_in[b]["d_" + k_].copy_(t, non_blocking=True)
            for k_, t in host_in.items():
                dev_in[b][k_].copy_(t, non_blocking=True)
            if mark:
                h_marks[-1][1].record(s_h2d)
            ev_in[b].record(s_h2d)
        stream.wait_event(ev_in[b])
        if i >= 2:
            stream.wait_event(ev_out[b])
        ob, lb, sb, dob, dlb, dsb = dev_out[b]
        di = dev_in[b]
        if mark:
            c_marks.append((_event(stream), _event(stream)))
            c_marks[-1][0].record(stream)
        msa.msa_index_select(cfg, di["q_idx"], di["k_idx"], sel=sb, ws=case.ws, stream=stream)
        msa.msa_attn_prefill(cfg, di["q"], di["k"], di["v"], sb, o=ob, lse=lb, ws=case.ws,
                             stream=stream)
        msa.msa_index_select(dc.cfg, di["d_q_idx"], paged=pagedb[b], sel=dsb, ws=dc.ws,
                             stream=stream)
        msa.msa_attn_decode(dc.cfg, di["d_q"], pagedb[b], dsb, o=dob, lse=dlb, ws=dc.ws,
                            stream=stream)
        if mark:
            c_marks[-1][1].record(stream)
        ev_used[b].record(stream)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(ev_used[b])
            if mark:
                d_marks.append((_event(s_d2h), _event(s_d2h)))
                d_marks[-1][0].record(s_d2h)
            for hd, t in zip(host_out, dev_out[b]):
                hd.copy_(t, non_blocking=True)
            if mark:
                d_marks[-1][1].record(s_d2h)
            ev_out[b].record(s_d2h)

    ref_sel, ref_dsel = case.sel.clone(), dc.sel.clone()  # the resident-input step's selections
    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.__enter__()
    barrier(world)
    torch.cuda.synchronize()
    e0.record(s_h2d)  # the first operation of the timed region
    for i in range(steps):
        e2e_step(i, mark=True)
    s_d2h.wait_stream(stream)
    e1.record(s_d2h)  # after the last copy out, which follows everything else
    torch.cuda.synchronize()
    sampler.__exit__(None, None, None)
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    compute_ms = [a.elapsed_time(b) for a, b in c_marks]
    starts = [e0.elapsed_time(a) for a, _ in c_marks]
    check_status(msa, case.ws, dc.ws)
    # the pipelined steps computed the same selections as the resident-input step
    assert torch.equal(host_out[2], ref_sel.cpu()), "end-to-end selection differs"
    assert torch.equal(host_out[5], ref_dsel.cpu()), "end-to-end decode selection differs"
    del host_in, host_out, dev_in, dev_out, dhost_in
    h2d_ms = [a.elapsed_time(b) for a, b in h_marks]
    d2h_ms = [a.elapsed_time(b) for a, b in d_marks]
    detail = {"clocks": sampler.summary(),
              "compute_ms_per_step": statistics.median(compute_ms),
              "h2d_ms_per_step": [round(x, 1) for x in h2d_ms],
              "d2h_ms_per_step": [round(x, 1) for x in d2h_ms],
              "first_compute_start_ms": starts[0],
              "compute_start_spacing_ms": statistics.median(
                  [b - a for a, b in zip(starts, starts[1:])]) if len(starts) > 1 else None}
    return ms, h2d, d2h, detail


def timed_alone(fn, n, warmup, stream):
    for _ in range(max(3, warmup)):
        fn()
    a0, a1 = _event(stream), _event(stream)
    torch.cuda.synchronize()
    a0.record(stream)
    for _ in range(n):
        fn()
    a1.record(stream)
    torch.cuda.synchronize()
    return a0.elapsed_time(a1) / n


def run_msa(args, world, rank):
    import block_sparse_long_msa_gb300 as msa
    msa.lib()
    peaks = load_peaks()
    w = workload(args)
    assert w.kind == "prefill", "the bench step is a prefill pass plus a decode step"
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    K, W = args.steps, args.warmup

    # ---------------- headline: prefill of the main workload + one decode step ----------------
    case = PrefillCase(msa, w, dev)
    dc = DecodeCase(msa, synthetic.WORKLOADS[args.decode_workload], dev,
                    batch=args.decode_batch or None, n_hi=args.decode_nmax or None)
    total_ms, ph, dph, clocks = time_prefill_decode(case, dc, K, W, world, stream, clocks=True)
    head = prefill_object(case, ph, peaks, world, K)
    decode = decode_object(dc, dph, peaks, world, K)

    # ---------------- end to end through the public API from pinned host buffers -------------
    e2e = None
    if args.e2e_steps > 0:
        need = 1.6 * sum(t.numel() * t.element_size()
                         for t in list(case.inp[k] for k in ("q", "k", "v", "q_idx", "k_idx"))
                         + [case.o, case.lse, case.sel])
        avail = host_memory_available()
        if avail and avail < need:
            e2e = {"value": None, "unit": "tokens/s",
                   "skipped": f"host memory available {avail / 2**30:.0f} GiB < "
                              f"{need / 2**30:.0f} GiB"}
        else:
            ms, h2d, d2h, e2e_detail = e2e_leg(msa, case, dc, args.e2e_steps, world, stream)
            e2e = {"value": world * w.L * args.e2e_steps / (ms * 1e-3), "unit": "tokens/s",
                   "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                   "steps": args.e2e_steps, "ms_per_step": ms / args.e2e_steps,
                   **e2e_detail,
                   "note": "prefill tokens over the whole step (prefill + decode) with every "
                           "step's inputs copied from pinned host memory and its outputs copied "
                           "back, on copy streams of their own (device buffers doubled, so the "
                           "copies of neighbouring steps overlap the compute); the decode KV "
                           "cache is resident state"}

    # ---- e4m3 index vectors (the FP8 indexer, tcgen05 kind::f8f6f4): a real e4m3 step, timed
    # like the headline one; the integer/8 inputs are exact in e4m3, so the selections must be
    # the bf16 ones ----
    e4m3 = None
    if not args.no_e4m3_index:
        f8 = torch.float8_e4m3fn
        ref_sel, ref_dsel = case.sel.clone(), dc.sel.clone()
        q8, k8 = case.inp["q_idx"].to(f8), case.inp["k_idx"].to(f8)
        cfg8 = msa.config(w.G, w.hpg, w.k, w.scale, index_dtype="e4m3")
        dw = dc.w
        dcfg_bf16, dpaged_bf16 = dc.cfg, dc.paged
        dk8 = dc.inp["k_idx_pool"].to(f8)
        dq8 = dc.inp["q_idx"].to(f8)
        kp8, vp8 = dc.inp["k_pool"].to(f8), dc.inp["v_pool"].to(f8)  # the FP8 K/V cache
        dc.with_encoding(msa.config(dw.G, dw.hpg, dw.k, dw.scale, index_dtype="e4m3"), dk8,
                         kp8, vp8)
        dq_bf16 = dc.inp["q_idx"]
        dc.inp["q_idx"] = dq8
        K8 = max(3, min(K, args.e4m3_steps))
        _, ph8, dph8, _ = time_prefill_decode(case, dc, K8, min(W, 3), world, stream,
                                              cfg_index=cfg8, q_idx=q8, k_idx=k8)
        torch.cuda.synchronize()
        assert torch.equal(case.sel, ref_sel) and torch.equal(dc.sel, ref_dsel), \
            "e4m3 selection differs"
        pre8 = prefill_object(case, ph8, peaks, world, K8, index_kernel="index_e4m3")
        fp8_peak = 2 * (peaks["bf16_tflops_sustained"] if ph8["prefill"] >= 50.0
                        else peaks["bf16_tflops"])
        idx_tf = pre8["kernel_rooflines"]["index"]["achieved"]
        e4m3 = {
            "note": "index vectors in e4m3 (exact for the integer/8 inputs: same selections, "
                    "asserted); steps timed as the headline step (index select + main branch, "
                    "then the decode step with every pool in e4m3: index keys, K and V)",
            "prefill_tokens_per_s": pre8["value"], "prefill_ms_per_pass": pre8["ms_per_pass"],
            "phases_ms_per_pass": pre8["phases_ms_per_pass"],
            "prefill_index_tflops": idx_tf,
            "prefill_index_frac_of_fp8_peak": idx_tf / fp8_peak,
            "fp8_peak_tflops": fp8_peak,
            "fp8_peak_note": "the measured bf16 peak x 2 (the nominal fp8:bf16 ratio)",
            "decode": decode_object(dc, dph8, peaks, world, K8, index_bytes=1, kv_bytes=1),
            "steps": K8,
            "gpu_launches": (case.launches + dc.launches) * K8,
        }
        e4m3["decode"].pop("cpu_baseline", None)
        dc.cfg, dc.paged = dcfg_bf16, dpaged_bf16
        dc.inp["q_idx"] = dq_bf16
        del q8, k8, dk8, dq8, kp8, vp8

    # ---- context-parallel index branch of the decode step, its R shards run one after another
    # on this GPU: per-shard candidate kernels and the merge (the all-gather between GPUs is
    # not measured here) ----
    cpi = None if args.cp_shards < 2 else cp_indexer_object(msa, dc, args.cp_shards, K, W,
                                                            stream)

    # ---------------- CPU oracle on a bounded sample of the headline workload ----------------
    cpu_base, dec_cpu = None, None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_base = cpu_baseline(w, case.inp, target_s=15.0)
        dec_cpu = decode_cpu_baseline(dc.w, dc.inp)
    decode["cpu_baseline"] = dec_cpu
    del case
    torch.cuda.empty_cache()

    # ---------------- the other prefill workloads, each timed the same way ----------------
    subs = []
    for name in [s for s in args.sub_workloads.split(",") if s]:
        sw = synthetic.WORKLOADS[name]
        sc = PrefillCase(msa, sw, dev)
        _, sph, _, _ = time_prefill_decode(sc, None, K, W, world, stream)
        obj = prefill_object(sc, sph, peaks, world, K)
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            obj["cpu_baseline"] = cpu_baseline(sw, sc.inp, target_s=8.0)
        if name == args.scores_workload and not args.no_index_scores:
            obj["index_scores"] = index_scores_object(msa, sc, dc, K, W, stream)
        subs.append(obj)
        del sc
        torch.cuda.empty_cache()

    graph = None if args.no_graph else cuda_graph_object(msa, dev)

    value = head["value"]
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": total_ms / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded SplitMix64; N(0,1) q/k/v, integer/8 index q/k)",
        "config": {"workload": w.name, "L": w.L, "Hq": w.Hq, "G": w.G, "d": w.d, "B": w.B,
                   "k": w.k, "parallelism": f"replicas x{world}",
                   "step": f"prefill of the {w.name} workload (index select + main branch over "
                           f"all L queries) + one paged decode step of the "
                           f"{dc.w.batch}-sequence workload; value = prefill tokens/s",
                   "l2": f"inputs larger than L2 (q {w.L * w.Hq * w.d * 2 / 2**20:.0f} MiB)"},
        "prefill_ms_per_step": head["ms_per_pass"],
        "phases_ms_per_step": head["phases_ms_per_pass"],
        "gpu_launches": (case_launches(msa, w) + dc.launches) * K,
        "roofline": head["roofline"],
        "kernel_rooflines": head["kernel_rooflines"],
        "main_branch": head["main_branch"],
        "tensor_frac_main_branch": head["main_branch"]["frac"],
        "e2e": e2e,
        "clocks": clocks,
        "cpu_baseline": cpu_base,
        "decode": decode,
        "prefill_workloads": subs,
        "e4m3_index": e4m3,
        "cp_indexer": cpi,
        "cuda_graph": graph,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def case_launches(msa, w):
    cfg = msa.config(w.G, w.hpg, w.k, w.scale)
    return 1 + msa.msa_attn_prefill_launches(cfg, w.L)


def cp_indexer_object(msa, dc, R, K, W, stream):
    from block_sparse_long_msa_gb300 import cp
    dw = dc.w
    bounds = cp.split_by_work(cp.decode_work(dc.inp["seq_lens"].tolist(), dc.inp["max_pages"]),
                              R)
    wdt = dw.k - 1
    dev = dc.sel.device
    cs = torch.empty((R, dw.G, dw.batch, wdt), dtype=torch.float32, device=dev)
    cb = torch.empty((R, dw.G, dw.batch, wdt), dtype=torch.int32, device=dev)
    sel = torch.empty_like(dc.sel)
    n = max(3, K)
    shard_ms = []
    for r, (b0, b1) in enumerate(bounds):
        shard_ms.append(timed_alone(lambda: msa.msa_index_candidates(
            dc.cfg, dc.inp["q_idx"], paged=dc.paged, block_begin=b0, block_end=b1,
            cand_score=cs[r], cand_block=cb[r], ws=dc.ws, stream=stream), n, W, stream))
    merge_ms = timed_alone(lambda: msa.msa_index_merge(dc.cfg, cs, cb, seq_lens=dc.inp["seq_lens"],
                                                       sel=sel, ws=dc.ws, stream=stream), n, W,
                           stream)
    single_ms = timed_alone(lambda: msa.msa_index_select(
        dc.cfg, dc.inp["q_idx"], paged=dc.paged, sel=dc.sel, ws=dc.ws, stream=stream), n, W,
        stream)
    check_status(msa, dc.ws)
    assert torch.equal(sel, dc.sel), "context-parallel selection differs"
    pages = [sum(max(0, min(b1, (int(x) - 1) // dw.B) - b0) for x in dc.inp["seq_lens"].tolist())
             for b0, b1 in bounds]
    return {
        "note": f"the decode step's index branch split into {R} shards of logical blocks with "
                "about equal pages (one per GPU in a context-parallel run), run one after "
                "another on this GPU, then merged; selection asserted equal to the single "
                "call.  The all-gather between GPUs is not measured (one GPU per box).",
        "shards": bounds, "pages_per_shard": pages,
        "shard_ms": shard_ms, "merge_ms": merge_ms, "single_call_ms": single_ms,
        "exchange_bytes_per_rank": dw.G * dw.batch * wdt * 8,
        "gpu_launches": (2 * R + 1 + 2) * n,
    }


def index_scores_object(msa, sc, dc, K, W, stream):
    """Block-score export (the indexer's KL alignment input): the same index kernels also write
    every block's pooled score, [G][L][nb] for prefill, [G][batch][max_pages] for decode; each
    timed alone, against the selection-only launch of the same kernels."""
    w, dw = sc.w, dc.w
    n = max(3, K)
    nb = (w.L + w.B - 1) // w.B
    dev = sc.sel.device
    bs = torch.empty((w.G, w.L, nb), dtype=torch.float32, device=dev)
    dbs = torch.empty((dw.G, dw.batch, dc.inp["max_pages"]), dtype=torch.float32, device=dev)
    sel_s, dsel_s = torch.empty_like(sc.sel), torch.empty_like(dc.sel)
    q, k = sc.inp["q_idx"], sc.inp["k_idx"]
    sc_ms = timed_alone(lambda: msa.msa_index_select_scores(
        sc.cfg, q, k, sel=sel_s, block_scores=bs, ws=sc.ws, stream=stream), n, W, stream)
    plain_ms = timed_alone(lambda: msa.msa_index_select(
        sc.cfg, q, k, sel=sc.sel, ws=sc.ws, stream=stream), n, W, stream)
    dsc_ms = timed_alone(lambda: msa.msa_index_select_scores(
        dc.cfg, dc.inp["q_idx"], paged=dc.paged, sel=dsel_s, block_scores=dbs, ws=dc.ws,
        stream=stream), n, W, stream)
    dplain_ms = timed_alone(lambda: msa.msa_index_select(
        dc.cfg, dc.inp["q_idx"], paged=dc.paged, sel=dc.sel, ws=dc.ws, stream=stream), n, W,
        stream)
    assert torch.equal(sel_s, sc.sel) and torch.equal(dsel_s, dc.sel), "score export selection"
    out_b, dout_b = bs.numel() * 4, dbs.numel() * 4
    return {
        "note": "msa_index_select_scores: the index kernels also write every block's pooled "
                "score (+inf own block, -inf later blocks); each timed alone, back to back, "
                "beside the selection-only launch of the same kernels",
        "prefill_ms": sc_ms, "prefill_ms_select_only": plain_ms,
        "prefill_output_bytes": out_b,
        "prefill_extra_gbs": out_b / max(sc_ms - plain_ms, 1e-6) / 1e6,
        "decode_ms": dsc_ms, "decode_ms_select_only": dplain_ms,
        "decode_output_bytes": dout_b,
        "gpu_launches": 2 * n + 4 * n,
    }


def cuda_graph_object(msa, dev):
    """The L = 2,048 prefill pass (launch-bound: eight short kernels) eager and as a replay of a
    CUDA graph captured from the same calls (the library enqueues only, so it captures)."""
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
    cur = torch.cuda.current_stream()
    eager_ms = timed_alone(tiny_pass, 50, 3, cur)
    graph_ms = timed_alone(cg.replay, 50, 3, cur)
    del cg
    return {
        "workload": tw.name, "L": tw.L,
        "note": "index select + main branch of the small workload, back to back (inputs of "
                "8 MiB stay in L2); eager calls against a replay of a CUDA graph captured "
                "from the same calls",
        "eager_ms": eager_ms, "graph_ms": graph_ms,
        "tokens_per_s_eager": tw.L / (eager_ms * 1e-3),
        "tokens_per_s_graph": tw.L / (graph_ms * 1e-3),
        "launches_per_pass": 1 + msa.msa_attn_prefill_launches(tcfg, tw.L),
    }


# ------------------------------------------------------------------------------------------
# CPU oracle timing (the reference arm, and the cpu_baseline of the MSA arm)
# ------------------------------------------------------------------------------------------
def _host_index_and_kv(inp):
    """k, v, q_idx, k_idx of a prefill workload on the host (q stays where it is: the oracle is
    given only the query rows it samples)."""
    return {k: inp[k].cpu() for k in ("k", "v", "q_idx", "k_idx")}


def _q_rows(w, inp, rows):
    """The sampled rows of q on the host: gathered from the device tensor when there is one,
    else generated directly (the generator is counter-based, so the rows are the same)."""
    if "q" in inp:
        idx = torch.from_numpy(rows).to(inp["q"].device)
        return inp["q"].index_select(0, idx).cpu()
    return synthetic.prefill_q_rows(w, rows)


def _oracle_rows(w, host, q_rows, rows):
    import oracle
    t = time.perf_counter()
    sel = oracle.select_prefill(host["q_idx"], host["k_idx"], w.B, w.k, rows=rows)
    oracle.attn_prefill(q_rows, host["k"], host["v"], sel, w.B, w.k, w.scale, rows=rows,
                        q_compact=True)
    return time.perf_counter() - t


def _strided_rows(L, n, phase=0):
    import numpy as np
    n = max(1, min(L, n))
    return (np.arange(n, dtype=np.int64) * L // n + phase) % L


def cpu_baseline(w, inp, target_s=15.0):
    """The oracle (index selection + attention, all groups and heads) on evenly strided query
    rows of the workload, about target_s of CPU work; copies to the host are untimed."""
    import oracle
    oracle.build()
    host = _host_index_and_kv(inp)
    n = 32
    rows = _strided_rows(w.L, n)
    dt = _oracle_rows(w, host, _q_rows(w, inp, rows), rows)
    n2 = int(min(w.L, max(n, n * target_s / max(dt, 1e-3))))
    rows = _strided_rows(w.L, n2, 1)
    dt2 = _oracle_rows(w, host, _q_rows(w, inp, rows), rows)
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
    # the index vectors and K/V of the whole workload; q only for the rows each step samples
    inp = synthetic.prefill_inputs(w, device=dev, without_q=True)
    host = _host_index_and_kv(inp)
    del inp
    budget_s = 150.0
    rows = _strided_rows(w.L, 8)
    cal = _oracle_rows(w, host, synthetic.prefill_q_rows(w, rows), rows)
    per_row = cal / 8
    rows_per_step = int(max(4, min(2048, budget_s / (args.steps + args.warmup) / per_row)))
    for s in range(args.warmup):
        rows = _strided_rows(w.L, rows_per_step, s + 1)
        _oracle_rows(w, host, synthetic.prefill_q_rows(w, rows), rows)
    total, n = 0.0, 0
    for s in range(args.steps):
        rows = _strided_rows(w.L, rows_per_step, args.warmup + s + 1)
        total += _oracle_rows(w, host, synthetic.prefill_q_rows(w, rows), rows)
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
