"""The library's calls can be captured in a CUDA graph and replayed.

Every call only enqueues work on the caller's stream: it allocates nothing, never synchronises
and reads no device memory on the host, so a prefill (index select + main branch) or a decode
step captured once replays with the results of the eager calls, bit for bit, and picks up new
inputs written into the captured buffers.
"""
import pytest
import torch

import synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    import block_sparse_long_msa_gb300 as m
    m.lib()
    return m


def _capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture, as torch asks
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("index_dtype", ["bf16", "e4m3"])
def test_prefill_graph_replay_matches_eager(msa, index_dtype):
    w = synthetic.WORKLOADS["tiny_L2048"]
    L = w.L
    inp = synthetic.prefill_inputs(w, device="cuda", index_dtype=index_dtype)
    cfg = msa.config(w.G, w.hpg, w.k, w.scale, index_dtype=index_dtype)
    ws_i = torch.zeros(msa.msa_index_select_workspace(cfg, L, L), dtype=torch.uint8, device="cuda")
    ws_a = torch.zeros(msa.msa_attn_prefill_workspace(cfg, L), dtype=torch.uint8, device="cuda")
    sel = torch.empty((w.G, L, w.k), dtype=torch.int32, device="cuda")
    o = torch.empty_like(inp["q"])
    lse = torch.empty((w.Hq, L), dtype=torch.float32, device="cuda")
    bufs = {k: inp[k].clone() for k in ("q", "k", "v", "q_idx", "k_idx")}

    def step():
        msa.msa_index_select(cfg, bufs["q_idx"], bufs["k_idx"], sel=sel, ws=ws_i)
        msa.msa_attn_prefill(cfg, bufs["q"], bufs["k"], bufs["v"], sel, o=o, lse=lse, ws=ws_a)

    g = _capture(step)
    for seed_shift in (0, 1):
        if seed_shift:  # new inputs in the captured buffers
            w2 = synthetic.Workload(**{**w.__dict__, "seed": w.seed + 17})
            inp = synthetic.prefill_inputs(w2, device="cuda", index_dtype=index_dtype)
            for k in bufs:
                bufs[k].copy_(inp[k])
        sel_e = msa.msa_index_select(cfg, inp["q_idx"], inp["k_idx"])
        o_e, lse_e = msa.msa_attn_prefill(cfg, inp["q"], inp["k"], inp["v"], sel_e)
        o.zero_()
        lse.zero_()
        sel.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(sel, sel_e)
        assert torch.equal(o, o_e) and torch.equal(lse, lse_e)
    assert msa.msa_get_device_status(ws_i) == 0 and msa.msa_get_device_status(ws_a) == 0


def test_decode_graph_replay_matches_eager(msa):
    w = synthetic.Workload("graph_dec", "decode", batch=6, G=4, Hq=64, k=16, seed=91)
    inp = synthetic.decode_inputs(w, device="cuda", batch=6, n_lo=100, n_hi=7000)
    w = inp["workload"]
    cfg = msa.config(w.G, w.hpg, w.k, w.scale)
    paged = msa.paged_kv(inp["k_idx_pool"], inp["k_pool"], inp["v_pool"], inp["page_table"],
                         inp["seq_lens"])
    ws = torch.zeros(max(msa.msa_index_select_workspace(cfg, w.batch, 0, paged),
                         msa.msa_attn_decode_workspace(cfg, paged)), dtype=torch.uint8,
                     device="cuda")
    q, q_idx = inp["q"].clone(), inp["q_idx"].clone()
    sel = torch.empty((w.G, w.batch, w.k), dtype=torch.int32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((w.Hq, w.batch), dtype=torch.float32, device="cuda")

    def step():
        msa.msa_index_select(cfg, q_idx, paged=paged, sel=sel, ws=ws)
        msa.msa_attn_decode(cfg, q, paged, sel, o=o, lse=lse, ws=ws)

    g = _capture(step)
    sel_e = msa.msa_index_select(cfg, inp["q_idx"], paged=paged)
    o_e, lse_e = msa.msa_attn_decode(cfg, inp["q"], paged, sel_e)
    o.zero_()
    sel.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(sel, sel_e) and torch.equal(o, o_e) and torch.equal(lse, lse_e)
    assert msa.msa_get_device_status(ws) == 0
