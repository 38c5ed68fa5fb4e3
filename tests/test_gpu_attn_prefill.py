"""GPU parity of the prefill main branch (msa_attn_prefill) against the CPU oracle.

Tolerance (stated for the operator): O within max-abs 1e-2 and mean-abs 1e-3 of the fp64 oracle,
LSE likewise.  The selection fed to the kernel is the GPU index branch's, which the index tests
show to be bit-identical to the oracle's; the oracle recomputes its own.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = pytest.mark.gpu

from parity_bar import MAX_ABS, MEAN_ABS, o_bar


@pytest.fixture(scope="module")
def msa():
    import block_sparse_long_msa_gb300 as m
    m.lib()
    return m


def run_gpu(msa, w, inp):
    cfg = msa.config(w.G, w.hpg, w.k, w.scale)
    dev = torch.device("cuda")
    d = {k: v.to(dev) for k, v in inp.items() if isinstance(v, torch.Tensor)}
    sel = msa.msa_index_select(cfg, d["q_idx"], d["k_idx"])
    ws = torch.zeros(msa.msa_attn_prefill_workspace(cfg, w.L), dtype=torch.uint8, device=dev)
    o, lse = msa.msa_attn_prefill(cfg, d["q"], d["k"], d["v"], sel, ws=ws)
    torch.cuda.synchronize()
    assert msa.msa_get_device_status(ws) == 0
    return sel.cpu().numpy(), o.float().cpu().numpy(), lse.cpu().numpy()


def compare(w, inp, sel, o, lse, rows=None):
    cpu = {k: v.cpu() for k, v in inp.items() if isinstance(v, torch.Tensor)}
    r_sel = oracle.select_prefill(cpu["q_idx"], cpu["k_idx"], w.B, w.k, rows=rows)
    r_o, r_lse = oracle.attn_prefill(cpu["q"], cpu["k"], cpu["v"], r_sel, w.B, w.k, w.scale,
                                     rows=rows)
    if rows is not None:
        sel, o, lse = sel[:, rows], o[rows], lse[:, rows]
    np.testing.assert_array_equal(sel, r_sel)
    err = np.abs(o - r_o)
    lerr = np.abs(lse - r_lse)
    msg = (f"O max {err.max():.3g} mean {err.mean():.3g}; LSE max {lerr.max():.3g} "
           f"mean {lerr.mean():.3g}")
    assert (err <= o_bar(r_o)).all() and err.mean() <= MEAN_ABS, msg
    assert lerr.max() <= MAX_ABS and lerr.mean() <= MEAN_ABS, msg
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    print(f"[parity {w.name} L={w.L}] {msg}")
    return err.max(), err.mean()


def _rows(L, n, seed):
    fixed = [0, 1, 127, 128, 129, 255, 256, L // 2, L - 129, L - 128, L - 2, L - 1]
    rnd = synthetic.uniform_int(seed, 78, n, 0, L - 1).tolist()
    return np.array(sorted(set(r for r in fixed + rnd if 0 <= r < L)), np.int64)


def test_tiny_workload_all_rows(msa):
    w = synthetic.WORKLOADS["tiny_L2048"]
    inp = synthetic.prefill_inputs(w)
    compare(w, inp, *run_gpu(msa, w, inp))


@pytest.mark.parametrize("L", [1, 129, 1000, 2048 + 77])
def test_ragged_lengths_all_rows(msa, L):
    w = synthetic.Workload(**{**synthetic.WORKLOADS["prefill_L32K"].__dict__, "L": L})
    inp = synthetic.prefill_inputs(w)
    compare(w, inp, *run_gpu(msa, w, inp))


@pytest.mark.parametrize("G,k,L", [(2, 8, 3000), (1, 1, 700), (4, 2, 1500), (3, 7, 1400)])
def test_group_and_k_variants(msa, G, k, L):
    w = synthetic.Workload("v", "prefill", L=L, Hq=16 * G, G=G, k=k, seed=77 + G * k)
    inp = synthetic.prefill_inputs(w)
    compare(w, inp, *run_gpu(msa, w, inp))


def test_full_budget_matches_sdpa_on_gpu(msa):
    """k*B >= L: every causal token is selected, so MSA is full causal GQA attention."""
    import torch.nn.functional as F
    w = synthetic.Workload("full", "prefill", L=1920, Hq=64, G=4, k=16, seed=3)
    inp = synthetic.prefill_inputs(w)
    _, o, lse = run_gpu(msa, w, inp)
    Q = inp["q"].cuda().float().permute(1, 0, 2)[None]
    K = inp["k"].cuda().float().permute(1, 0, 2)[None]
    V = inp["v"].cuda().float().permute(1, 0, 2)[None]
    ref = F.scaled_dot_product_attention(Q, K, V, is_causal=True, scale=w.scale,
                                         enable_gqa=True)[0].permute(1, 0, 2).cpu().numpy()
    err = np.abs(o - ref)
    assert (err <= o_bar(ref)).all() and err.mean() <= MEAN_ABS, (err.max(), err.mean())


def test_full_size_32k_sampled_rows(msa):
    w = synthetic.WORKLOADS["prefill_L32K"]
    inp = synthetic.prefill_inputs(w, device="cuda")
    compare(w, inp, *run_gpu(msa, w, inp), rows=_rows(w.L, 200, 4))


def test_full_size_128k_clustered_sampled_rows(msa):
    w = synthetic.WORKLOADS["prefill_L128K_clustered"]
    inp = synthetic.prefill_inputs(w, device="cuda")
    compare(w, inp, *run_gpu(msa, w, inp), rows=_rows(w.L, 96, 5))


def test_deterministic_repeat(msa):
    w = synthetic.Workload(**{**synthetic.WORKLOADS["prefill_L32K"].__dict__, "L": 4096})
    inp = synthetic.prefill_inputs(w)
    a = run_gpu(msa, w, inp)
    b = run_gpu(msa, w, inp)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_full_size_1m_hot_sampled_rows(msa):
    """L = 1,048,576 with hot key blocks 0-3 (about 90% of queries choose them): 16 query passes
    of the main branch, heavily skewed work lists; sampled rows against the oracle."""
    w = synthetic.WORKLOADS["prefill_L1M_hot"]
    inp = synthetic.prefill_inputs(w, device="cuda")
    cfg = msa.config(w.G, w.hpg, w.k, w.scale)
    sel = msa.msa_index_select(cfg, inp["q_idx"], inp["k_idx"])
    ws = torch.zeros(msa.msa_attn_prefill_workspace(cfg, w.L), dtype=torch.uint8, device="cuda")
    o, lse = msa.msa_attn_prefill(cfg, inp["q"], inp["k"], inp["v"], sel, ws=ws)
    torch.cuda.synchronize()
    assert msa.msa_get_device_status(ws) == 0
    # the skew the workload is built for: most queries past block 4 pick all of blocks 0..3
    late = sel[:, 4 * 128::997]
    hot = (late[..., :4] == torch.arange(4, device="cuda")).all(-1).float().mean().item()
    assert hot > 0.8, hot
    rows = _rows(w.L, 40, 6)
    ridx = torch.tensor(rows, device="cuda")
    g_sel = sel[:, ridx].cpu().numpy()
    g_o = o[ridx].float().cpu().numpy()
    g_lse = lse[:, ridx].cpu().numpy()
    r_sel = oracle.select_prefill(inp["q_idx"].cpu(), inp["k_idx"].cpu(), w.B, w.k, rows=rows)
    np.testing.assert_array_equal(g_sel, r_sel)
    r_o, r_lse = oracle.attn_prefill(inp["q"][ridx].cpu(), inp["k"].cpu(), inp["v"].cpu(), r_sel,
                                     w.B, w.k, w.scale, rows=rows, q_compact=True)
    err, lerr = np.abs(g_o - r_o), np.abs(g_lse - r_lse)
    msg = (f"O max {err.max():.3g} mean {err.mean():.3g}; LSE max {lerr.max():.3g} "
           f"mean {lerr.mean():.3g}; hot fraction {hot:.3f}")
    assert (err <= o_bar(r_o)).all() and err.mean() <= MEAN_ABS, msg
    assert lerr.max() <= MAX_ABS and lerr.mean() <= MEAN_ABS, msg
    print(f"[parity {w.name} L={w.L}] {msg}")


def test_maximum_length_sampled_rows(msa):
    """L = 1,572,864, the longest prefill the library takes: 24 query passes, and the schedule's
    token mask of 12,288 key blocks fills 192 KiB of shared memory.  The hot-block key bias of the
    1M workload; the selection and the main branch on sampled rows against the oracle, the last
    rows included."""
    w = synthetic.Workload(**{**synthetic.WORKLOADS["prefill_L1M_hot"].__dict__, "L": 1572864,
                              "name": "prefill_Lmax_hot", "seed": 1571})
    inp = synthetic.prefill_inputs(w, device="cuda")
    cfg = msa.config(w.G, w.hpg, w.k, w.scale)
    assert msa.msa_attn_prefill_launches(cfg, w.L) == 24 * 7
    sel = msa.msa_index_select(cfg, inp["q_idx"], inp["k_idx"])
    ws = torch.zeros(msa.msa_attn_prefill_workspace(cfg, w.L), dtype=torch.uint8, device="cuda")
    o, lse = msa.msa_attn_prefill(cfg, inp["q"], inp["k"], inp["v"], sel, ws=ws)
    torch.cuda.synchronize()
    assert msa.msa_get_device_status(ws) == 0
    rows = _rows(w.L, 20, 8)
    ridx = torch.tensor(rows, device="cuda")
    g_sel = sel[:, ridx].cpu().numpy()
    g_o = o[ridx].float().cpu().numpy()
    g_lse = lse[:, ridx].cpu().numpy()
    del o, lse, ws
    r_sel = oracle.select_prefill(inp["q_idx"].cpu(), inp["k_idx"].cpu(), w.B, w.k, rows=rows)
    np.testing.assert_array_equal(g_sel, r_sel)
    r_o, r_lse = oracle.attn_prefill(inp["q"][ridx].cpu(), inp["k"].cpu(), inp["v"].cpu(), r_sel,
                                     w.B, w.k, w.scale, rows=rows, q_compact=True)
    err, lerr = np.abs(g_o - r_o), np.abs(g_lse - r_lse)
    wide = np.abs(r_o) >= 4.0  # bf16 spacing 1/32 there: the output must round faithfully
    msg = (f"O max {err.max():.3g} (below |o| = 4: {err[~wide].max():.3g}; {int(wide.sum())} "
           f"elements at |o| >= 4) mean {err.mean():.3g}; LSE max {lerr.max():.3g} "
           f"mean {lerr.mean():.3g}")
    assert (err <= o_bar(r_o)).all() and err.mean() <= MEAN_ABS, msg
    assert lerr.max() <= MAX_ABS and lerr.mean() <= MEAN_ABS, msg
    print(f"[parity {w.name} L={w.L}] {msg}")


@pytest.mark.parametrize("L,k", [(700, 5), (1300, 12)])
def test_more_than_four_groups_with_the_oracle_selection(msa, L, k):
    """The main branch takes any number of GQA groups (the index branch stops at four): G = 8,
    128 query heads, fed the oracle's selection; every row against the oracle."""
    w = synthetic.Workload("g8", "prefill", L=L, Hq=128, G=8, k=k, seed=808 + L)
    inp = synthetic.prefill_inputs(w)
    r_sel = oracle.select_prefill(inp["q_idx"], inp["k_idx"], w.B, w.k)
    cfg = msa.config(w.G, w.hpg, w.k, w.scale)
    dev = torch.device("cuda")
    d = {name: t.to(dev) for name, t in inp.items() if isinstance(t, torch.Tensor)}
    with pytest.raises(msa.MsaError):  # the index branch refuses more than four groups
        msa.msa_index_select(cfg, d["q_idx"], d["k_idx"])
    ws = torch.zeros(msa.msa_attn_prefill_workspace(cfg, w.L), dtype=torch.uint8, device=dev)
    o, lse = msa.msa_attn_prefill(cfg, d["q"], d["k"], d["v"], torch.from_numpy(r_sel).to(dev),
                                  ws=ws)
    torch.cuda.synchronize()
    assert msa.msa_get_device_status(ws) == 0
    r_o, r_lse = oracle.attn_prefill(inp["q"], inp["k"], inp["v"], r_sel, w.B, w.k, w.scale)
    got_o, got_lse = o.float().cpu().numpy(), lse.cpu().numpy()
    err, lerr = np.abs(got_o - r_o), np.abs(got_lse - r_lse)
    msg = f"O max {err.max():.3g} mean {err.mean():.3g}; LSE max {lerr.max():.3g}"
    assert (err <= o_bar(r_o)).all() and err.mean() <= MEAN_ABS, msg
    assert lerr.max() <= MAX_ABS and lerr.mean() <= MEAN_ABS, msg
    print(f"[parity G=8 L={L} k={k}] {msg}")


def _random_shapes(n, seed):
    """n seeded (L, G, k) draws: L in [130, 2600] (ragged tails), G in {1, 2, 4}, k in [1, 16]."""
    Ls = synthetic.uniform_int(seed, 81, n, 130, 2600).tolist()
    Gs = synthetic.uniform_int(seed, 82, n, 0, 2).tolist()
    ks = synthetic.uniform_int(seed, 83, n, 1, 16).tolist()
    return [(L, (1, 2, 4)[g], k) for L, g, k in zip(Ls, Gs, ks)]


@pytest.mark.parametrize("L,G,k", _random_shapes(6, 2024))
@pytest.mark.parametrize("index_dtype", ["bf16", "e4m3"])
def test_random_shapes_all_rows(msa, L, G, k, index_dtype):
    """Seeded random shapes, every row: selection bit-exact and O / LSE within tolerance, with
    bf16 and with e4m3 index vectors (the same integer/8 values)."""
    w = synthetic.Workload("rand", "prefill", L=L, Hq=16 * G, G=G, k=k, seed=L * 7 + G * 3 + k)
    inp = synthetic.prefill_inputs(w, index_dtype=index_dtype)
    cfg = msa.config(w.G, w.hpg, w.k, w.scale, index_dtype=index_dtype)
    dev = torch.device("cuda")
    d = {k_: v.to(dev) for k_, v in inp.items() if isinstance(v, torch.Tensor)}
    sel = msa.msa_index_select(cfg, d["q_idx"], d["k_idx"])
    ws = torch.zeros(msa.msa_attn_prefill_workspace(cfg, w.L), dtype=torch.uint8, device=dev)
    o, lse = msa.msa_attn_prefill(cfg, d["q"], d["k"], d["v"], sel, ws=ws)
    torch.cuda.synchronize()
    assert msa.msa_get_device_status(ws) == 0
    compare(w, inp, sel.cpu().numpy(), o.float().cpu().numpy(), lse.cpu().numpy())
