"""GPU parity of the context-parallel index branch (msa_index_candidates + msa_index_merge).

On one GPU the R shards run one after another; their stacked candidates are what an all-gather
over R ranks would deliver.  Checks:
  * each shard's candidates equal the oracle's pooled scores of that shard's blocks, ranked by
    (score desc, block asc) and cut at k-1, bit for bit (ids and fp32 scores);
  * the merged selection equals the single-call selection (msa_index_select) and the oracle's,
    bit for bit, for prefill and paged decode, with bf16 and e4m3 index vectors, with uneven,
    empty and single shards.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from block_sparse_long_msa_gb300 import cp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    import block_sparse_long_msa_gb300 as m
    m.lib()
    return m


def _oracle_candidates(scores, bis, b0, b1, w):
    """Rank blocks [b0, min(b1, b_i)) of each row by (score desc, block asc) from the oracle's
    pooled scores [G][T][nb]; returns ids [G][T][w] (-1 padded) and scores (-inf padded)."""
    G, T, _ = scores.shape
    ids = np.full((G, T, w), -1, np.int64)
    sc = np.full((G, T, w), -np.inf)
    for g in range(G):
        for t in range(T):
            hi = min(b1, int(bis[t]))
            blocks = list(range(b0, hi))
            blocks.sort(key=lambda b: (-scores[g, t, b], b))
            for r, b in enumerate(blocks[:w]):
                ids[g, t, r] = b
                sc[g, t, r] = scores[g, t, b]
    return ids, sc


def _prefill_shards(msa, cfg, d, L, bounds):
    cs, cb = [], []
    for b0, b1 in bounds:
        lo, hi = b0 * 128, min(b1 * 128, L)
        k_shard = d["k_idx"][lo:max(hi, lo + 1)] if hi > lo else d["k_idx"][:1]
        s, b = msa.msa_index_candidates(cfg, d["q_idx"], k_shard, L=L, block_begin=b0,
                                        block_end=b1)
        cs.append(s)
        cb.append(b)
    return torch.stack(cs), torch.stack(cb)


@pytest.mark.parametrize("index_dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("L,G,k,bounds", [
    (3000, 4, 16, [(0, 7), (7, 15), (15, 24)]),
    (2100, 2, 6, [(0, 1), (1, 2), (2, 9), (9, 9), (9, 17)]),
    (1500, 3, 16, [(0, 12)]),
    (1000, 1, 1, [(0, 3), (3, 8)]),
])
def test_prefill_shards_merge_to_the_selection(msa, index_dtype, L, G, k, bounds):
    w = synthetic.Workload("cp", "prefill", L=L, Hq=16 * G, G=G, k=k, seed=300 + L + G + k)
    host = synthetic.prefill_inputs(w, index_only=True, index_dtype=index_dtype)
    d = {n: host[n].cuda() for n in ("q_idx", "k_idx")}
    cfg = msa.config(G, 16, k, index_dtype=index_dtype)
    all_s, all_b = _prefill_shards(msa, cfg, d, L, bounds)
    sel_cp, sc_cp = msa.msa_index_merge(cfg, all_s, all_b, want_score=True)
    sel, sc = msa.msa_index_select(cfg, d["q_idx"], d["k_idx"], want_score=True)
    torch.cuda.synchronize()
    assert torch.equal(sel_cp, sel)
    assert torch.equal(sc_cp, sc)
    r_sel = oracle.select_prefill(host["q_idx"], host["k_idx"], w.B, w.k)
    np.testing.assert_array_equal(sel_cp.cpu().numpy(), r_sel)
    if k > 1:
        scores = oracle.block_scores_prefill(host["q_idx"], host["k_idx"], w.B)
        bis = np.arange(L) // w.B
        for r, (b0, b1) in enumerate(bounds):
            ids, rsc = _oracle_candidates(scores, bis, b0, b1, k - 1)
            np.testing.assert_array_equal(all_b[r].cpu().numpy(), ids)
            np.testing.assert_array_equal(all_s[r].cpu().numpy().astype(np.float64), rsc)


def _decode_inputs(lens, seed, G=4, k=16, index_dtype="bf16"):
    w = synthetic.Workload("cpd", "decode", batch=len(lens), G=G, Hq=16 * G, k=k, seed=seed)
    B = w.B
    pages = [(n + B - 1) // B for n in lens]
    P = sum(pages) + 2
    perm = synthetic.permutation(seed, synthetic.STREAM_PAGES, P).to(torch.int32)
    pt = torch.full((len(lens), max(pages)), -1, dtype=torch.int32)
    off = 0
    for s, npg in enumerate(pages):
        pt[s, :npg] = perm[off:off + npg]
        off += npg
    inp = {"seq_lens": torch.tensor(lens, dtype=torch.int32), "page_table": pt,
           "q_idx": synthetic.as_index_dtype(
               synthetic.int8th(seed, synthetic.STREAM_QI, (len(lens), G, w.di)), index_dtype),
           "k_idx_pool": synthetic.as_index_dtype(
               synthetic.int8th(seed, synthetic.STREAM_KI, (P, B, w.di)), index_dtype)}
    return w, inp


def _decode_cp(msa, cfg, d, bounds):
    paged = msa.paged_kv(d["k_idx_pool"], None, None, d["page_table"], d["seq_lens"])
    cs, cb = [], []
    for b0, b1 in bounds:
        s, b = msa.msa_index_candidates(cfg, d["q_idx"], paged=paged, block_begin=b0,
                                        block_end=b1)
        cs.append(s)
        cb.append(b)
    all_s, all_b = torch.stack(cs), torch.stack(cb)
    merged = msa.msa_index_merge(cfg, all_s, all_b, seq_lens=d["seq_lens"], want_score=True)
    single = msa.msa_index_select(cfg, d["q_idx"], paged=paged, want_score=True)
    torch.cuda.synchronize()
    return merged, single, all_s, all_b


@pytest.mark.parametrize("index_dtype", ["bf16", "e4m3"])
def test_decode_page_shards_merge_to_the_selection(msa, index_dtype):
    lens = [300, 5000, 129, 2560, 128, 1, 4097, 3333]
    w, inp = _decode_inputs(lens, seed=401, index_dtype=index_dtype)
    d = {n: v.cuda() for n, v in inp.items()}
    cfg = msa.config(w.G, 16, w.k, index_dtype=index_dtype)
    maxp = inp["page_table"].shape[1]
    bounds = cp.split_by_work(cp.decode_work(lens, maxp), 4)
    assert bounds[0][0] == 0 and bounds[-1][1] == maxp
    (sel_cp, sc_cp), (sel, sc), all_s, all_b = _decode_cp(msa, cfg, d, bounds)
    assert torch.equal(sel_cp, sel) and torch.equal(sc_cp, sc)
    r_sel = oracle.select_decode(inp["q_idx"], inp["k_idx_pool"], inp["page_table"],
                                 inp["seq_lens"], w.B, w.k)
    np.testing.assert_array_equal(sel_cp.cpu().numpy(), r_sel)
    scores = oracle.block_scores_decode(inp["q_idx"], inp["k_idx_pool"], inp["page_table"],
                                        inp["seq_lens"], w.B)
    bis = (np.array(lens) - 1) // w.B
    for r, (b0, b1) in enumerate(bounds):
        ids, rsc = _oracle_candidates(scores, bis, b0, b1, w.k - 1)
        np.testing.assert_array_equal(all_b[r].cpu().numpy(), ids)
        np.testing.assert_array_equal(all_s[r].cpu().numpy().astype(np.float64), rsc)


def test_full_size_decode_workload_over_four_shards(msa):
    """The 64-sequence workload (16K-256K tokens) split over 4 shards of about equal pages, as
    the pages' 4-GPU context-parallel indexer decode would split it."""
    dw = synthetic.WORKLOADS["decode_b64_16K_256K"]
    inp = synthetic.decode_inputs(dw, device="cuda")
    w = inp["workload"]
    d = {n: inp[n] for n in ("q_idx", "k_idx_pool", "page_table", "seq_lens")}
    cfg = msa.config(w.G, 16, w.k)
    bounds = cp.split_by_work(cp.decode_work(inp["seq_lens"].tolist(), inp["max_pages"]), 4)
    (sel_cp, sc_cp), (sel, sc), _, _ = _decode_cp(msa, cfg, d, bounds)
    assert torch.equal(sel_cp, sel) and torch.equal(sc_cp, sc)


def test_merge_flags_a_candidate_past_the_query_block(msa):
    L, G, k = 700, 2, 4
    cfg = msa.config(G, 16, k)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    cand_b = torch.full((1, G, L, k - 1), -1, dtype=torch.int32, device="cuda")
    cand_s = torch.full((1, G, L, k - 1), float("-inf"), device="cuda")
    cand_b[0, 1, 300, 0] = 3  # query 300 is in block 2: block 3 is not before it
    cand_s[0, 1, 300, 0] = 1.0
    cand_b[0, 0, 600, 0] = 1
    cand_s[0, 0, 600, 0] = 2.0
    sel = msa.msa_index_merge(cfg, cand_s, cand_b, ws=ws)
    assert msa.msa_get_device_status(ws) == 6
    assert sel[1, 300].tolist() == [2, -1, -1, -1]
    assert sel[0, 600].tolist() == [1, 4, -1, -1]
    assert sel[0, 0].tolist() == [0, -1, -1, -1]
