"""Run one part of the MSA path on one workload, with only the tensors it needs, for profilers.

  python -m block_sparse_long_msa_gb300.profile_case --workload prefill_L1M_hot --what index
  python -m block_sparse_long_msa_gb300.profile_case --workload prefill_L32K --what attn --L 8192
  python -m block_sparse_long_msa_gb300.profile_case --workload decode_b64_16K_256K --what decode

--what index   msa_index_select on the prefill workload (q_idx, k_idx and sel on the device)
--what attn    msa_attn_prefill (one index selection first, untimed; then the index vectors are
               freed): each repetition launches the scheduling kernels, the attention and the
               combine once per query chunk
--what decode  one decode step (index select + attention) of the paged workload
Each part runs `--reps` times back to back and the program checks the device status word, so a
profiler can skip the first repetitions and capture the last.
"""
from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main(argv=None):
    import torch

    import block_sparse_long_msa_gb300 as msa
    import synthetic

    p = argparse.ArgumentParser()
    p.add_argument("--workload", required=True)
    p.add_argument("--what", choices=["index", "attn", "decode"], required=True)
    p.add_argument("--L", type=int, default=0, help="override the prefill length")
    p.add_argument("--reps", type=int, default=2)
    p.add_argument("--index-dtype", default="bf16", choices=["bf16", "e4m3"])
    p.add_argument("--kv-dtype", default="bf16", choices=["bf16", "e4m3"])
    p.add_argument("--batch", type=int, default=0, help="decode: override the batch")
    p.add_argument("--nmax", type=int, default=0, help="decode: override the longest context")
    a = p.parse_args(argv)
    msa.lib()
    dev = torch.device("cuda")
    w = synthetic.WORKLOADS[a.workload]
    if a.L:
        w = synthetic.Workload(**{**w.__dict__, "L": a.L, "name": f"{w.name}@L{a.L}"})
    if a.what == "decode":
        inp = synthetic.decode_inputs(w, device=dev, batch=a.batch or None, n_hi=a.nmax or None,
                                      index_dtype=a.index_dtype)
        dw = inp["workload"]
        kp, vp = inp["k_pool"], inp["v_pool"]
        if a.kv_dtype == "e4m3":
            kp, vp = kp.to(torch.float8_e4m3fn), vp.to(torch.float8_e4m3fn)
        cfg = msa.config(dw.G, dw.hpg, dw.k, dw.scale, index_dtype=a.index_dtype)
        paged = msa.paged_kv(inp["k_idx_pool"], kp, vp, inp["page_table"], inp["seq_lens"])
        ws = torch.zeros(max(msa.msa_index_select_workspace(cfg, dw.batch, 0, paged),
                             msa.msa_attn_decode_workspace(cfg, paged)), dtype=torch.uint8,
                         device=dev)
        for _ in range(a.reps):
            sel = msa.msa_index_select(cfg, inp["q_idx"], paged=paged, ws=ws)
            msa.msa_attn_decode(cfg, inp["q"], paged, sel, ws=ws)
    else:
        cfg = msa.config(w.G, w.hpg, w.k, w.scale, index_dtype=a.index_dtype)
        idx = synthetic.prefill_inputs(w, device=dev, index_only=True, index_dtype=a.index_dtype)
        ws = torch.zeros(max(msa.msa_index_select_workspace(cfg, w.L, w.L),
                             msa.msa_attn_prefill_workspace(cfg, w.L) if a.what == "attn"
                             else 0), dtype=torch.uint8, device=dev)
        sel = torch.empty((w.G, w.L, w.k), dtype=torch.int32, device=dev)
        reps = a.reps if a.what == "index" else 1
        for _ in range(reps):
            msa.msa_index_select(cfg, idx["q_idx"], idx["k_idx"], sel=sel, ws=ws)
        if a.what == "attn":
            del idx
            kv = synthetic.prefill_inputs(w, device=dev)
            del kv["q_idx"], kv["k_idx"]
            for _ in range(a.reps):
                msa.msa_attn_prefill(cfg, kv["q"], kv["k"], kv["v"], sel, ws=ws)
    torch.cuda.synchronize()
    st = msa.msa_get_device_status(ws)
    if st != 0:
        raise SystemExit(f"device status {st}")
    print(f"profile_case {a.workload} {a.what} L={getattr(w, 'L', 0)} reps={a.reps}: ok")


if __name__ == "__main__":
    main()
