"""Device-side failure detection, driven from the host; no GPU fault is made.

Every wait inside the kernels is bounded by msa_config_t.wait_limit_ns.  A wait that runs out
records MSA_ERR_DEVICE_TIMEOUT in the caller's status word; the kernel then waits (with the fixed
2 s drain limit) for its own copies and MMAs in flight, frees its tensor memory and returns.  Ids
out of range are skipped before any load and recorded as MSA_ERR_DEVICE_BOUNDS: a block id past
the query's own block in a prefill selection, a page id past the pool in a page table, a
context length past the page table.

The timeouts are made by a 1 ns limit: every kernel waits for a copy or an MMA right after it
starts, which takes longer than that.  After each failed call the same context runs the normal
call, which must match the oracle: the aborted kernels left no tensor memory allocated and no
copy in flight.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = pytest.mark.gpu

from parity_bar import MAX_ABS, MEAN_ABS, o_bar
TIMEOUT, BOUNDS = 5, 6


@pytest.fixture(scope="module")
def msa():
    import block_sparse_long_msa_gb300 as m
    m.lib()
    return m


def _prefill_case(L=1100, seed=611):
    w = synthetic.Workload(**{**synthetic.WORKLOADS["prefill_L32K"].__dict__, "L": L,
                              "seed": seed})
    return w, synthetic.prefill_inputs(w, device="cpu")


def _close(got_o, got_lse, r_o, r_lse):
    err, lerr = np.abs(got_o - r_o), np.abs(got_lse - r_lse)
    assert (err <= o_bar(r_o)).all() and err.mean() <= MEAN_ABS, err.max()
    assert lerr.max() <= MAX_ABS and lerr.mean() <= MEAN_ABS, lerr.max()


def test_prefill_wait_limit_runs_out_and_the_context_stays_usable(msa):
    w, inp = _prefill_case()
    dev = torch.device("cuda")
    d = {k: v.to(dev) for k, v in inp.items() if isinstance(v, torch.Tensor)}
    cfg = msa.config(w.G, w.hpg, w.k, w.scale)
    short = msa.config(w.G, w.hpg, w.k, w.scale, wait_limit_ns=1)
    ws_i = torch.zeros(msa.msa_index_select_workspace(cfg, w.L, w.L), dtype=torch.uint8,
                       device=dev)
    ws_a = torch.zeros(msa.msa_attn_prefill_workspace(cfg, w.L), dtype=torch.uint8, device=dev)
    sel = msa.msa_index_select(cfg, d["q_idx"], d["k_idx"], ws=ws_i)
    assert msa.msa_get_device_status(ws_i) == 0
    # index branch with the 1 ns limit: the call returns, the status word says timeout
    scratch = torch.empty_like(sel)
    msa.msa_index_select(short, d["q_idx"], d["k_idx"], sel=scratch, ws=ws_i)
    assert msa.msa_get_device_status(ws_i) == TIMEOUT
    # main branch with the 1 ns limit
    o_bad = torch.empty_like(d["q"])
    msa.msa_attn_prefill(short, d["q"], d["k"], d["v"], sel, o=o_bad, ws=ws_a)
    assert msa.msa_get_device_status(ws_a) == TIMEOUT
    # the status is sticky until reset; then the normal calls run in the same context
    msa.msa_reset_device_status(ws_i)
    msa.msa_reset_device_status(ws_a)
    sel2 = msa.msa_index_select(cfg, d["q_idx"], d["k_idx"], ws=ws_i)
    o, lse = msa.msa_attn_prefill(cfg, d["q"], d["k"], d["v"], sel2, ws=ws_a)
    assert msa.msa_get_device_status(ws_i) == 0 and msa.msa_get_device_status(ws_a) == 0
    r_sel = oracle.select_prefill(inp["q_idx"], inp["k_idx"], w.B, w.k)
    np.testing.assert_array_equal(sel2.cpu().numpy(), r_sel)
    r_o, r_lse = oracle.attn_prefill(inp["q"], inp["k"], inp["v"], r_sel, w.B, w.k, w.scale)
    _close(o.float().cpu().numpy(), lse.cpu().numpy(), r_o, r_lse)


def test_prefill_block_id_past_the_query_block_is_skipped_and_flagged(msa):
    w, inp = _prefill_case(L=1300, seed=612)
    dev = torch.device("cuda")
    d = {k: v.to(dev) for k, v in inp.items() if isinstance(v, torch.Tensor)}
    cfg = msa.config(w.G, w.hpg, w.k, w.scale)
    r_sel = oracle.select_prefill(inp["q_idx"], inp["k_idx"], w.B, w.k)
    # query 700 (block 5) of group 2: its first non-local entry becomes block 9 (> 5, < nb)
    g, i = 2, 700
    bad = r_sel.copy()
    assert bad[g, i, 0] < 5
    bad[g, i, 0] = 9
    ws = torch.zeros(msa.msa_attn_prefill_workspace(cfg, w.L), dtype=torch.uint8, device=dev)
    o, lse = msa.msa_attn_prefill(cfg, d["q"], d["k"], d["v"], torch.from_numpy(bad).to(dev),
                                  ws=ws)
    assert msa.msa_get_device_status(ws) == BOUNDS
    got_o, got_lse = o.float().cpu().numpy(), lse.cpu().numpy()
    assert np.isfinite(got_o).all() and np.isfinite(got_lse).all()
    # the skipped id acts as padding: the oracle with -1 in its place gives every row
    skipped = r_sel.copy()
    skipped[g, i, 0] = -1
    r_o, r_lse = oracle.attn_prefill(inp["q"], inp["k"], inp["v"], skipped, w.B, w.k, w.scale)
    _close(got_o, got_lse, r_o, r_lse)
    # and every other row is the plain result
    rows = np.array([r for r in range(w.L) if r != i])
    p_o, p_lse = oracle.attn_prefill(inp["q"], inp["k"], inp["v"], r_sel[:, rows], w.B, w.k,
                                     w.scale, rows=rows)
    _close(got_o[rows], got_lse[:, rows], p_o, p_lse)


def _decode_case(seed=613, batch=6):
    w = synthetic.Workload(**{**synthetic.WORKLOADS["decode_b64_16K_256K"].__dict__,
                              "seed": seed})
    inp = synthetic.decode_inputs(w, device="cpu", batch=batch, n_lo=300, n_hi=5000)
    return inp["workload"], inp


def _decode_oracle(w, inp, seqs):
    """Oracle selection and attention for the listed sequences (pools indexed directly)."""
    sel = oracle.select_decode(inp["q_idx"], inp["k_idx_pool"], inp["page_table"],
                               inp["seq_lens"], w.B, w.k)
    o, lse = oracle.attn_decode(inp["q"], inp["k_pool"], inp["v_pool"], inp["page_table"],
                                inp["seq_lens"], sel, w.B, w.k, w.scale)
    return sel[:, seqs], o[seqs], lse[:, seqs]


def _gpu_decode(msa, w, d, cfg, ws):
    paged = msa.paged_kv(d["k_idx_pool"], d["k_pool"], d["v_pool"], d["page_table"],
                         d["seq_lens"])
    sel = msa.msa_index_select(cfg, d["q_idx"], paged=paged, ws=ws)
    o, lse = msa.msa_attn_decode(cfg, d["q"], paged, sel, ws=ws)
    return sel, o, lse


def test_decode_wait_limit_runs_out_and_the_context_stays_usable(msa):
    # 48 sequences: 3,072 (sequence, group, slot) units, about 20 per attention CTA, so the
    # producer of every CTA waits for its 3-stage ring to drain (with a few units per CTA the
    # ring never fills and no wait need last longer than a copy)
    w, inp = _decode_case(batch=48)
    dev = torch.device("cuda")
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    cfg = msa.config(w.G, w.hpg, w.k, w.scale)
    short = msa.config(w.G, w.hpg, w.k, w.scale, wait_limit_ns=1)
    paged = msa.paged_kv(d["k_idx_pool"], d["k_pool"], d["v_pool"], d["page_table"],
                         d["seq_lens"])
    ws = torch.zeros(max(msa.msa_index_select_workspace(cfg, w.batch, 0, paged),
                         msa.msa_attn_decode_workspace(cfg, paged)), dtype=torch.uint8,
                     device=dev)
    sel = msa.msa_index_select(cfg, d["q_idx"], paged=paged, ws=ws)
    assert msa.msa_get_device_status(ws) == 0
    msa.msa_index_select(short, d["q_idx"], paged=paged, sel=torch.empty_like(sel), ws=ws)
    assert msa.msa_get_device_status(ws) == TIMEOUT
    msa.msa_reset_device_status(ws)
    msa.msa_attn_decode(short, d["q"], paged, sel, ws=ws)
    assert msa.msa_get_device_status(ws) == TIMEOUT
    msa.msa_reset_device_status(ws)
    sel2, o, lse = _gpu_decode(msa, w, d, cfg, ws)
    assert msa.msa_get_device_status(ws) == 0
    seqs = np.arange(w.batch)
    r_sel, r_o, r_lse = _decode_oracle(w, inp, seqs)
    np.testing.assert_array_equal(sel2.cpu().numpy(), r_sel)
    _close(o.float().cpu().numpy(), lse.cpu().numpy(), r_o, r_lse)


def test_decode_page_id_past_the_pool_is_skipped_and_flagged(msa):
    w, inp = _decode_case(seed=614)
    dev = torch.device("cuda")
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    cfg = msa.config(w.G, w.hpg, w.k, w.scale)
    s_bad = int(np.argmax(inp["seq_lens"].numpy()))  # the longest sequence: block 0 is scanned
    assert int(inp["seq_lens"][s_bad]) > 2 * w.B
    pt_bad = d["page_table"].clone()
    pt_bad[s_bad, 0] = inp["num_pages"]  # one past the pool
    d_bad = {**d, "page_table": pt_bad}
    paged = msa.paged_kv(d["k_idx_pool"], d["k_pool"], d["v_pool"], pt_bad, d["seq_lens"])
    ws = torch.zeros(max(msa.msa_index_select_workspace(cfg, w.batch, 0, paged),
                         msa.msa_attn_decode_workspace(cfg, paged)), dtype=torch.uint8,
                     device=dev)
    # the scan reads a stand-in page for the bad entry; the attention skips that block if chosen
    sel, o, lse = _gpu_decode(msa, w, d_bad, cfg, ws)
    assert msa.msa_get_device_status(ws) == BOUNDS
    # a selection that includes the bad block: the attention alone must skip and flag it
    msa.msa_reset_device_status(ws)
    forced = sel.clone()
    forced[:, s_bad, 0] = 0
    forced[:, s_bad] = torch.sort(forced[:, s_bad], dim=-1).values
    msa.msa_attn_decode(cfg, d["q"], paged, forced, ws=ws)
    assert msa.msa_get_device_status(ws) == BOUNDS
    others = np.array([s for s in range(w.batch) if s != s_bad])
    r_sel, r_o, r_lse = _decode_oracle(w, inp, others)
    np.testing.assert_array_equal(sel.cpu().numpy()[:, others], r_sel)
    _close(o.float().cpu().numpy()[others], lse.cpu().numpy()[:, others], r_o, r_lse)
    assert np.isfinite(o.float().cpu().numpy()[s_bad]).all()


def test_decode_context_length_past_the_page_table_is_flagged(msa):
    w, inp = _decode_case(seed=615)
    dev = torch.device("cuda")
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    cfg = msa.config(w.G, w.hpg, w.k, w.scale)
    s_bad = 2
    lens_bad = d["seq_lens"].clone()
    lens_bad[s_bad] = inp["max_pages"] * w.B + 7
    d_bad = {**d, "seq_lens": lens_bad}
    paged = msa.paged_kv(d["k_idx_pool"], d["k_pool"], d["v_pool"], d["page_table"], lens_bad)
    ws = torch.zeros(max(msa.msa_index_select_workspace(cfg, w.batch, 0, paged),
                         msa.msa_attn_decode_workspace(cfg, paged)), dtype=torch.uint8,
                     device=dev)
    sel, o, lse = _gpu_decode(msa, w, d_bad, cfg, ws)
    assert msa.msa_get_device_status(ws) == BOUNDS
    assert (sel[:, s_bad] == -1).all()
    others = np.array([s for s in range(w.batch) if s != s_bad])
    r_sel, r_o, r_lse = _decode_oracle(w, inp, others)
    np.testing.assert_array_equal(sel.cpu().numpy()[:, others], r_sel)
    _close(o.float().cpu().numpy()[others], lse.cpu().numpy()[:, others], r_o, r_lse)
