"""GPU parity of paged decode (msa_index_select with a page table, msa_attn_decode) against the
CPU oracle: selections and pooled scores bit-exact, O / LSE within max-abs 1e-2 and mean-abs
1e-3; plus decode of the token at n-1 equals the last row of a prefill of the same n tokens."""
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


def gpu_decode(msa, w, inp):
    dev = torch.device("cuda")
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    dt = "e4m3" if d["q_idx"].dtype == torch.float8_e4m3fn else "bf16"
    cfg = msa.config(w.G, w.hpg, w.k, w.scale, index_dtype=dt)
    paged = msa.paged_kv(d["k_idx_pool"], d["k_pool"], d["v_pool"], d["page_table"],
                         d["seq_lens"])
    ws = torch.zeros(max(msa.msa_index_select_workspace(cfg, w.batch, 0, paged),
                         msa.msa_attn_decode_workspace(cfg, paged)), dtype=torch.uint8,
                     device=dev)
    sel, score = msa.msa_index_select(cfg, d["q_idx"], paged=paged, want_score=True, ws=ws)
    o, lse = msa.msa_attn_decode(cfg, d["q"], paged, sel, ws=ws)
    torch.cuda.synchronize()
    assert msa.msa_get_device_status(ws) == 0
    return sel.cpu().numpy(), score.cpu().numpy(), o.float().cpu().numpy(), lse.cpu().numpy()


def oracle_decode(w, inp):
    """Oracle selection from the index keys, then oracle attention on a compacted copy of the
    selected pages (gathered on whatever device holds the pools; no arithmetic of the method)."""
    pt = inp["page_table"].cpu()
    seq = inp["seq_lens"].cpu()
    sel, score = oracle.select_decode(inp["q_idx"].cpu(), inp["k_idx_pool"].cpu(), pt, seq, w.B,
                                      w.k, want_score=True)
    used = sorted({int(pt[s, b]) for g in range(w.G) for s in range(sel.shape[1])
                   for b in sel[g, s] if b >= 0})
    remap = {p: i for i, p in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.long, device=inp["k_pool"].device)
    kp = inp["k_pool"].index_select(0, idx).cpu()
    vp = inp["v_pool"].index_select(0, idx).cpu()
    pt2 = torch.full_like(pt, 0)
    for s in range(pt.shape[0]):
        for b in range(pt.shape[1]):
            p = int(pt[s, b])
            pt2[s, b] = remap.get(p, 0)
    o, lse = oracle.attn_decode(inp["q"].cpu(), kp, vp, pt2, seq, sel, w.B, w.k, w.scale)
    return sel, score, o, lse


def check(w, inp, got):
    sel, score, o, lse = got
    r_sel, r_score, r_o, r_lse = oracle_decode(w, inp)
    np.testing.assert_array_equal(sel, r_sel)
    np.testing.assert_array_equal(score.astype(np.float64), r_score)
    err, lerr = np.abs(o - r_o), np.abs(lse - r_lse)
    msg = (f"O max {err.max():.3g} mean {err.mean():.3g}; LSE max {lerr.max():.3g} "
           f"mean {lerr.mean():.3g}")
    assert (err <= o_bar(r_o)).all() and err.mean() <= MEAN_ABS, msg
    assert lerr.max() <= MAX_ABS and lerr.mean() <= MEAN_ABS, msg
    print(f"[decode parity {w.name} batch={w.batch}] {msg}")


def _custom(lens, seed, G=4, k=16, device="cpu"):
    w = synthetic.Workload("decode_custom", "decode", batch=len(lens), G=G, Hq=16 * G, k=k,
                           seed=seed)
    base = synthetic.decode_inputs(w, device=device, batch=len(lens), n_lo=1, n_hi=1)
    # rebuild with the exact lengths: same generator streams, explicit lengths
    B = w.B
    pages = [(n + B - 1) // B for n in lens]
    P = sum(pages) + 3
    maxp = max(pages)
    perm = synthetic.permutation(seed, synthetic.STREAM_PAGES, P, device).to(torch.int32)
    pt = torch.full((len(lens), maxp), -1, dtype=torch.int32, device=device)
    off = 0
    for s, npg in enumerate(pages):
        pt[s, :npg] = perm[off:off + npg]
        off += npg
    inp = {
        "seq_lens": torch.tensor(lens, dtype=torch.int32, device=device),
        "page_table": pt,
        "q": base["q"], "q_idx": base["q_idx"],
        "k_idx_pool": synthetic.int8th(seed, synthetic.STREAM_KI, (P, B, w.di), device),
        "k_pool": synthetic.normal_bf16(seed, synthetic.STREAM_K, (P, G, B, w.d), device),
        "v_pool": synthetic.normal_bf16(seed, synthetic.STREAM_V, (P, G, B, w.d), device),
    }
    return w, inp


def test_ragged_lengths(msa):
    w, inp = _custom([1, 127, 128, 129, 1000, 3000, 2049], seed=11)
    check(w, inp, gpu_decode(msa, w, inp))


@pytest.mark.parametrize("G,k", [(1, 4), (2, 8), (4, 1), (3, 16)])
def test_group_and_k_variants(msa, G, k):
    w, inp = _custom([300, 5000, 129, 2560], seed=20 + G + k, G=G, k=k)
    check(w, inp, gpu_decode(msa, w, inp))


def test_more_than_four_groups_with_the_oracle_selection(msa):
    """Decode attention takes any number of GQA groups (the index branch stops at four): G = 8,
    128 query heads, fed the oracle's selection; every sequence against the oracle."""
    w, inp = _custom([1, 129, 700, 3000, 5000], seed=31, G=8, k=6)
    r_sel, _, r_o, r_lse = oracle_decode(w, inp)
    dev = torch.device("cuda")
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    cfg = msa.config(w.G, w.hpg, w.k, w.scale)
    paged = msa.paged_kv(d["k_idx_pool"], d["k_pool"], d["v_pool"], d["page_table"],
                         d["seq_lens"])
    ws = torch.zeros(msa.msa_attn_decode_workspace(cfg, paged), dtype=torch.uint8, device=dev)
    with pytest.raises(msa.MsaError):  # the index branch refuses more than four groups
        msa.msa_index_select(cfg, d["q_idx"], paged=paged, ws=ws)
    o, lse = msa.msa_attn_decode(cfg, d["q"], paged, torch.from_numpy(r_sel).to(dev), ws=ws)
    torch.cuda.synchronize()
    assert msa.msa_get_device_status(ws) == 0
    got_o, got_lse = o.float().cpu().numpy(), lse.cpu().numpy()
    err, lerr = np.abs(got_o - r_o), np.abs(got_lse - r_lse)
    assert (err <= o_bar(r_o)).all() and err.mean() <= MEAN_ABS, err.max()
    assert lerr.max() <= MAX_ABS and lerr.mean() <= MEAN_ABS, lerr.max()


def test_mid_size_batch(msa):
    w, inp = _custom([16384, 20000, 40000, 65536, 17000, 33333, 50001, 16385], seed=12)
    check(w, inp, gpu_decode(msa, w, inp))


def test_full_size_decode_workload(msa):
    w0 = synthetic.WORKLOADS["decode_b64_16K_256K"]
    inp = synthetic.decode_inputs(w0, device="cuda")
    w = inp["workload"]
    check(w, inp, gpu_decode(msa, w, inp))


def test_decode_equals_last_prefill_row(msa):
    """The token at n-1 decoded from a paged copy of a prefill's cache equals the prefill's
    last row (selection exactly, output within tolerance)."""
    n = 3000
    pw = synthetic.Workload(**{**synthetic.WORKLOADS["prefill_L32K"].__dict__, "L": n})
    inp = synthetic.prefill_inputs(pw, device="cuda")
    cfg = msa.config(pw.G, pw.hpg, pw.k, pw.scale)
    sel_p = msa.msa_index_select(cfg, inp["q_idx"], inp["k_idx"])
    o_p, lse_p = msa.msa_attn_prefill(cfg, inp["q"], inp["k"], inp["v"], sel_p)
    B, G = pw.B, pw.G
    npg = (n + B - 1) // B
    perm = synthetic.permutation(5, 10, npg + 2, "cuda")
    pt = perm[:npg].to(torch.int32)[None]
    P = npg + 2
    pad = npg * B - n
    kidx = torch.zeros(P, B, pw.di, dtype=torch.bfloat16, device="cuda")
    kp = torch.zeros(P, G, B, pw.d, dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    kidx[pt[0].long()] = torch.nn.functional.pad(inp["k_idx"], (0, 0, 0, pad)).view(npg, B, -1)
    kp[pt[0].long()] = torch.nn.functional.pad(inp["k"], (0, 0, 0, 0, 0, pad)) \
        .view(npg, B, G, -1).permute(0, 2, 1, 3)
    vp[pt[0].long()] = torch.nn.functional.pad(inp["v"], (0, 0, 0, 0, 0, pad)) \
        .view(npg, B, G, -1).permute(0, 2, 1, 3)
    seq = torch.tensor([n], dtype=torch.int32, device="cuda")
    paged = msa.paged_kv(kidx, kp, vp, pt.contiguous(), seq)
    sel_d = msa.msa_index_select(cfg, inp["q_idx"][n - 1:n].contiguous(), paged=paged)
    o_d, lse_d = msa.msa_attn_decode(cfg, inp["q"][n - 1:n].contiguous(), paged, sel_d)
    torch.cuda.synchronize()
    assert torch.equal(sel_d[:, 0], sel_p[:, n - 1])
    ref = o_p[n - 1].float().cpu().numpy()
    err = np.abs(o_d[0].float().cpu().numpy() - ref)
    assert (err <= o_bar(ref)).all(), err.max()  # two bf16 roundings of nearly the same value
    assert (lse_d[:, 0] - lse_p[:, n - 1]).abs().max().item() <= 1e-4


# ---------------------------------- E4M3 index vectors ----------------------------------
def _e4m3(inp):
    return {**inp, "q_idx": synthetic.as_index_dtype(inp["q_idx"], "e4m3"),
            "k_idx_pool": synthetic.as_index_dtype(inp["k_idx_pool"], "e4m3")}


def test_e4m3_ragged_lengths(msa):
    w, inp = _custom([1, 127, 128, 129, 1000, 3000, 2049], seed=13)
    inp = _e4m3(inp)
    check(w, inp, gpu_decode(msa, w, inp))


@pytest.mark.parametrize("G,k", [(1, 4), (2, 16)])
def test_e4m3_group_and_k_variants(msa, G, k):
    w, inp = _custom([300, 5000, 129, 2560], seed=30 + G + k, G=G, k=k)
    inp = _e4m3(inp)
    check(w, inp, gpu_decode(msa, w, inp))


def test_e4m3_full_size_decode_workload_equals_bf16(msa):
    """The 64-sequence workload with an E4M3 index-key pool: parity with the oracle, and the
    same selection as the bf16 pool holding the same values."""
    w0 = synthetic.WORKLOADS["decode_b64_16K_256K"]
    inp = synthetic.decode_inputs(w0, device="cuda", index_dtype="e4m3")
    w = inp["workload"]
    got = gpu_decode(msa, w, inp)
    check(w, inp, got)
    ref = synthetic.decode_inputs(w0, device="cuda")
    assert np.array_equal(gpu_decode(msa, w, ref)[0], got[0])


# ------------------------------------ E4M3 K/V cache ------------------------------------
def _e4m3_kv(inp):
    """The same pools stored as e4m3 (each value rounded to the nearest e4m3 value by torch's
    cast: an encoding of the input, no arithmetic of the method).  The oracle decodes the
    codes exactly, so the parity bar is the one of the bf16 cache."""
    return {**inp, "k_pool": inp["k_pool"].to(torch.float8_e4m3fn),
            "v_pool": inp["v_pool"].to(torch.float8_e4m3fn)}


def test_e4m3_kv_ragged_lengths(msa):
    w, inp = _custom([1, 127, 128, 129, 1000, 3000, 2049], seed=14)
    inp = _e4m3_kv(inp)
    check(w, inp, gpu_decode(msa, w, inp))


@pytest.mark.parametrize("G,k", [(1, 4), (2, 8), (3, 16), (4, 1)])
def test_e4m3_kv_group_and_k_variants(msa, G, k):
    w, inp = _custom([300, 5000, 129, 2560], seed=40 + G + k, G=G, k=k)
    inp = _e4m3_kv(inp)
    check(w, inp, gpu_decode(msa, w, inp))


def test_e4m3_kv_and_index_full_size_decode_workload(msa):
    """The 64-sequence workload with every pool in e4m3 (index keys, K, V): selection equal to
    the bf16-index one, O and LSE within the tolerance of the oracle on the e4m3 values."""
    w0 = synthetic.WORKLOADS["decode_b64_16K_256K"]
    inp = synthetic.decode_inputs(w0, device="cuda", index_dtype="e4m3")
    inp = _e4m3_kv(inp)
    w = inp["workload"]
    got = gpu_decode(msa, w, inp)
    check(w, inp, got)


def test_e4m3_kv_pools_must_share_a_dtype(msa):
    w, inp = _custom([300, 700], seed=15)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    with pytest.raises(msa.MsaError):
        msa.paged_kv(d["k_idx_pool"], d["k_pool"].to(torch.float8_e4m3fn), d["v_pool"],
                     d["page_table"], d["seq_lens"])
