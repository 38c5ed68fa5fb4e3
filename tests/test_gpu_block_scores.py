"""GPU parity of the exported block scores (msa_index_select_scores) against the CPU oracle.

The indexer's KL alignment ("MiniMax M3 算力省 20 倍", section 三 item 1) fits the indexer's block
scores to the main branch's attention, so the index kernels can also write every block's pooled
score: the block max of the raw dot products for blocks before the query's own, +inf for its own
block, -inf after it.  Index inputs sit on the integer/8 grid, so the comparison is bit-exact, and
the selection returned alongside must equal msa_index_select's.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    import block_sparse_long_msa_gb300 as m
    m.lib()
    return m


def _prefill(msa, w, q_idx, k_idx, rows=None):
    dt = "e4m3" if q_idx.dtype == torch.float8_e4m3fn else "bf16"
    cfg = msa.config(w.G, w.hpg, w.k, w.scale, index_dtype=dt)
    qd, kd = q_idx.cuda(), k_idx.cuda()
    sel, bs = msa.msa_index_select_scores(cfg, qd, kd)
    sel_plain = msa.msa_index_select(cfg, qd, kd)
    torch.cuda.synchronize()
    L = q_idx.shape[0]
    assert bs.shape == (w.G, L, (L + 127) // 128)
    assert torch.equal(sel, sel_plain)
    got = bs.cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[:, rows]
    ref = oracle.block_scores_prefill(q_idx, k_idx, w.B, rows=rows)
    bad = np.argwhere((got != ref).any(-1))
    assert bad.size == 0, f"{len(bad)} rows differ, first (g, row) {bad[:5].tolist()}"
    return got


def test_tiny_workload_all_rows(msa):
    w = synthetic.WORKLOADS["tiny_L2048"]
    inp = synthetic.prefill_inputs(w, index_only=True)
    _prefill(msa, w, inp["q_idx"], inp["k_idx"])


@pytest.mark.parametrize("L", [1, 127, 129, 1000, 2048 + 77])
def test_ragged_lengths_all_rows(msa, L):
    w = synthetic.WORKLOADS["prefill_L32K"]
    inp = synthetic.prefill_inputs(w, index_only=True, L=L)
    _prefill(msa, synthetic.Workload(**{**w.__dict__, "L": L}), inp["q_idx"], inp["k_idx"])


@pytest.mark.parametrize("G,k,L", [(1, 1, 700), (2, 8, 3000), (4, 2, 1500), (1, 16, 1900)])
def test_group_and_k_variants(msa, G, k, L):
    """G = 1 runs one group per CTA with both epilogue warpgroups sharing its rows."""
    w = synthetic.Workload("bs", "prefill", L=L, Hq=16 * G, G=G, k=k, seed=62 + G + k)
    inp = synthetic.prefill_inputs(w, index_only=True)
    _prefill(msa, w, inp["q_idx"], inp["k_idx"])


@pytest.mark.parametrize("index_dtype", ["bf16", "e4m3"])
def test_full_size_32k_sampled_rows(msa, index_dtype):
    w = synthetic.WORKLOADS["prefill_L32K"]
    inp = synthetic.prefill_inputs(w, index_only=True, index_dtype=index_dtype)
    nb = w.L // 128
    rows = np.array(sorted({0, 127, 128, w.L - 1} |
                           set(synthetic.uniform_int(4, 77, 60, 0, w.L - 1).tolist())), np.int64)
    got = _prefill(msa, w, inp["q_idx"], inp["k_idx"], rows=rows)
    assert got.shape == (w.G, len(rows), nb)


def _decode(msa, w, inp):
    dev = torch.device("cuda")
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    dt = "e4m3" if d["q_idx"].dtype == torch.float8_e4m3fn else "bf16"
    cfg = msa.config(w.G, w.hpg, w.k, w.scale, index_dtype=dt)
    paged = msa.paged_kv(d["k_idx_pool"], d["k_pool"], d["v_pool"], d["page_table"],
                         d["seq_lens"])
    ws = torch.zeros(msa.msa_index_select_workspace(cfg, w.batch, 0, paged), dtype=torch.uint8,
                     device=dev)
    sel, bs = msa.msa_index_select_scores(cfg, d["q_idx"], paged=paged, ws=ws)
    sel_plain = msa.msa_index_select(cfg, d["q_idx"], paged=paged, ws=ws)
    torch.cuda.synchronize()
    assert msa.msa_get_device_status(ws) == 0
    assert torch.equal(sel, sel_plain)
    ref = oracle.block_scores_decode(inp["q_idx"].cpu(), inp["k_idx_pool"].cpu(),
                                     inp["page_table"].cpu(), inp["seq_lens"].cpu(), w.B)
    np.testing.assert_array_equal(bs.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("index_dtype", ["bf16", "e4m3"])
def test_decode_ragged_batch(msa, index_dtype):
    w = synthetic.Workload("bs_dec", "decode", batch=9, G=4, Hq=64, k=16, seed=71)
    inp = synthetic.decode_inputs(w, batch=9, n_lo=1, n_hi=6000, index_dtype=index_dtype)
    _decode(msa, inp["workload"], inp)


@pytest.mark.parametrize("G,k", [(1, 4), (2, 8)])
def test_decode_group_and_k_variants(msa, G, k):
    w = synthetic.Workload("bs_dec", "decode", batch=5, G=G, Hq=16 * G, k=k, seed=80 + G)
    inp = synthetic.decode_inputs(w, batch=5, n_lo=100, n_hi=9000)
    _decode(msa, inp["workload"], inp)


def test_decode_full_size_workload(msa):
    w0 = synthetic.WORKLOADS["decode_b64_16K_256K"]
    inp = synthetic.decode_inputs(w0, device="cuda")
    _decode(msa, inp["workload"], inp)
