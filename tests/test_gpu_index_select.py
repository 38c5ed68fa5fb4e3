"""GPU parity of the index branch (msa_index_select, prefill) against the CPU oracle, with bf16
and with E4M3 index vectors (the FP8 indexer, tcgen05 kind::f8f6f4).

Selections must match bit-exactly, and so must the pooled scores: index inputs sit on the
integer/8 grid, so every fp32 tensor-core dot product is exact (see test_oracle_pins).
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


def _check(msa, w, q_idx, k_idx, rows=None):
    dt = "e4m3" if q_idx.dtype == torch.float8_e4m3fn else "bf16"
    cfg = msa.config(w.G, w.hpg, w.k, w.scale, index_dtype=dt)
    sel, score = msa.msa_index_select(cfg, q_idx.cuda(), k_idx.cuda(), want_score=True)
    torch.cuda.synchronize()
    ref_sel, ref_score = oracle.select_prefill(q_idx, k_idx, w.B, w.k, rows=rows, want_score=True)
    got_sel = sel.cpu().numpy()
    got_score = score.cpu().numpy().astype(np.float64)
    if rows is not None:
        got_sel, got_score = got_sel[:, rows], got_score[:, rows]
    bad = np.argwhere((got_sel != ref_sel).any(-1))
    assert bad.size == 0, f"{len(bad)} rows differ, first (g, row) {bad[:5].tolist()}: " \
                          f"gpu {got_sel[tuple(bad[0])]} oracle {ref_sel[tuple(bad[0])]}"
    np.testing.assert_array_equal(got_score, ref_score)
    return got_sel


def _stratified_rows(L, n, seed):
    nb = (L + 127) // 128
    fixed = [0, 1, 127, 128, 129, L - 1] + list(range(128 * (nb - 1), L))
    rnd = synthetic.uniform_int(seed, 77, n, 0, L - 1).tolist()
    return np.array(sorted(set(r for r in fixed + rnd if 0 <= r < L)), np.int64)


def test_tiny_workload_all_rows(msa):
    w = synthetic.WORKLOADS["tiny_L2048"]
    inp = synthetic.prefill_inputs(w, index_only=True)
    _check(msa, w, inp["q_idx"], inp["k_idx"])


@pytest.mark.parametrize("L", [1, 127, 128, 129, 1000, 2048 + 77])
def test_ragged_lengths_all_rows(msa, L):
    w = synthetic.WORKLOADS["prefill_L32K"]
    inp = synthetic.prefill_inputs(w, index_only=True, L=L)
    sel = _check(msa, synthetic.Workload(**{**w.__dict__, "L": L}), inp["q_idx"], inp["k_idx"])
    assert (sel[..., :].max(-1) == np.arange(L) // 128).all()  # local block is the largest id


@pytest.mark.parametrize("G,k,L", [(2, 8, 3000), (1, 1, 700), (4, 2, 1500), (2, 16, 640),
                                   (3, 6, 1700)])
def test_group_and_k_variants(msa, G, k, L):
    w = synthetic.Workload("v", "prefill", L=L, Hq=16 * G, G=G, k=k, seed=42 + G + k)
    inp = synthetic.prefill_inputs(w, index_only=True)
    _check(msa, w, inp["q_idx"], inp["k_idx"])


def test_ties_duplicate_blocks(msa):
    w = synthetic.Workload("ties", "prefill", L=2560, Hq=64, G=4, k=6, seed=5)
    inp = synthetic.prefill_inputs(w, index_only=True)
    k_idx = inp["k_idx"].clone()
    for b in (1, 3, 7, 11):  # copies of block 5: equal pooled scores for every query
        k_idx[b * 128:(b + 1) * 128] = k_idx[5 * 128:6 * 128]
    _check(msa, w, inp["q_idx"], k_idx)


def test_pm1_inputs_exact(msa):
    """All +-1 index inputs: scores are integers up to 128 in magnitude, many ties."""
    w = synthetic.Workload("pm1", "prefill", L=1536, Hq=64, G=4, k=16, seed=8)
    q = (synthetic.sign_vector(8, 4, 1536 * 4 * 128).view(1536, 4, 128)).to(torch.bfloat16)
    k = (synthetic.sign_vector(8, 5, 1536 * 128).view(1536, 128)).to(torch.bfloat16)
    _check(msa, w, q, k)


def test_full_size_32k_sampled_rows(msa):
    w = synthetic.WORKLOADS["prefill_L32K"]
    inp = synthetic.prefill_inputs(w, index_only=True)
    _check(msa, w, inp["q_idx"], inp["k_idx"], rows=_stratified_rows(w.L, 384, 1))


def test_full_size_128k_clustered_sampled_rows(msa):
    w = synthetic.WORKLOADS["prefill_L128K_clustered"]
    inp = synthetic.prefill_inputs(w, index_only=True)
    sel = _check(msa, w, inp["q_idx"], inp["k_idx"], rows=_stratified_rows(w.L, 160, 2))
    assert sel.shape[-1] == 16


# ---------------------------------- E4M3 index vectors ----------------------------------
def test_e4m3_tiny_workload_all_rows(msa):
    w = synthetic.WORKLOADS["tiny_L2048"]
    inp = synthetic.prefill_inputs(w, index_only=True, index_dtype="e4m3")
    _check(msa, w, inp["q_idx"], inp["k_idx"])


@pytest.mark.parametrize("L", [1, 129, 1000, 2048 + 77])
def test_e4m3_ragged_lengths_all_rows(msa, L):
    w = synthetic.WORKLOADS["prefill_L32K"]
    inp = synthetic.prefill_inputs(w, index_only=True, L=L, index_dtype="e4m3")
    _check(msa, synthetic.Workload(**{**w.__dict__, "L": L}), inp["q_idx"], inp["k_idx"])


@pytest.mark.parametrize("G,k,L", [(2, 8, 3000), (1, 1, 700), (1, 16, 1900), (3, 12, 1300)])
def test_e4m3_group_and_k_variants(msa, G, k, L):
    w = synthetic.Workload("v8", "prefill", L=L, Hq=16 * G, G=G, k=k, seed=52 + G + k)
    inp = synthetic.prefill_inputs(w, index_only=True, index_dtype="e4m3")
    _check(msa, w, inp["q_idx"], inp["k_idx"])


def test_e4m3_ties_duplicate_blocks(msa):
    w = synthetic.Workload("ties8", "prefill", L=2560, Hq=64, G=4, k=6, seed=5)
    inp = synthetic.prefill_inputs(w, index_only=True, index_dtype="e4m3")
    k_idx = inp["k_idx"].view(torch.uint8).clone()
    for b in (1, 3, 7, 11):
        k_idx[b * 128:(b + 1) * 128] = k_idx[5 * 128:6 * 128]
    _check(msa, w, inp["q_idx"], k_idx.view(torch.float8_e4m3fn))


def test_e4m3_full_size_32k_sampled_rows_and_equal_to_bf16(msa):
    """Sampled rows against the oracle; every row against the bf16 path on the same values."""
    w = synthetic.WORKLOADS["prefill_L32K"]
    inp = synthetic.prefill_inputs(w, index_only=True, index_dtype="e4m3")
    got = _check(msa, w, inp["q_idx"], inp["k_idx"], rows=_stratified_rows(w.L, 256, 3))
    ref = synthetic.prefill_inputs(w, index_only=True)
    cfg = msa.config(w.G, w.hpg, w.k, w.scale)
    cfg8 = msa.config(w.G, w.hpg, w.k, w.scale, index_dtype="e4m3")
    s16 = msa.msa_index_select(cfg, ref["q_idx"].cuda(), ref["k_idx"].cuda())
    s8 = msa.msa_index_select(cfg8, inp["q_idx"].cuda(), inp["k_idx"].cuda())
    assert torch.equal(s16, s8)
    assert got.shape[-1] == 16


def test_e4m3_dtype_mismatch_is_rejected(msa):
    w = synthetic.WORKLOADS["tiny_L2048"]
    inp = synthetic.prefill_inputs(w, index_only=True)
    cfg8 = msa.config(w.G, w.hpg, w.k, w.scale, index_dtype="e4m3")
    with pytest.raises(msa.MsaError):
        msa.msa_index_select(cfg8, inp["q_idx"].cuda(), inp["k_idx"].cuda())
