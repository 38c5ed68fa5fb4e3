"""Pins for the CPU oracle, against things other than the oracle itself.

* hand-worked examples (tests/golden/msa_handworked.txt), derived from the definition on the page
  "MiniMax M3 算力省 20 倍" section 二 / 三 item 4;
* brute force on tiny inputs: a dense L x L numpy formulation with a full Python sort;
* the invariant that with k*B >= L every causal token is selected, so MSA equals full causal GQA
  attention (torch SDPA in fp64, a library routine);
* k = 1 reduces to block-local causal attention (SDPA with a block-diagonal causal mask);
* equal block scores rank the lower block id first; permuting tokens inside a selected
  non-local block changes nothing; a decode at position n-1 equals the last prefill row;
* the exported block scores (section 三 item 1) equal a dense numpy max-pool under the causal
  mask, and ranking them reproduces the selection.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "msa_handworked.txt")


def _bf(a) -> torch.Tensor:
    t = torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    assert torch.equal(t.float(), torch.as_tensor(np.asarray(a, dtype=np.float32))), "not bf16-exact"
    return t


def _parse_golden():
    cases, cur = {}, None
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, val = line.partition(":")
        key, val = key.strip(), val.strip()
        if key == "case":
            cur = cases.setdefault(val, {})
        elif key == "end":
            cur = None
        else:
            rows = [[float(x) for x in r.split()] for r in val.split("|")]
            if len(rows) > 1:
                cur[key] = rows
            else:
                cur[key] = rows[0][0] if len(rows[0]) == 1 and key not in ("lse_row0", "lse_row1") \
                    else rows[0]
    return cases


# ----------------------------------------------------------------------------------------------
# SplitMix64: published first outputs of the generator seeded with 0 (state += gamma, then mix).
# ----------------------------------------------------------------------------------------------
def test_splitmix64_published_sequence():
    expect = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    gamma = 0x9E3779B97F4A7C15
    for n, e in enumerate(expect):
        assert synthetic.splitmix64_int((n * gamma) & ((1 << 64) - 1)) == e
    x = torch.tensor([(n * gamma) % (1 << 64) for n in range(3)], dtype=torch.float64)
    xs = torch.tensor([synthetic._s64(n * gamma) for n in range(3)], dtype=torch.int64)
    got = [int(v) % (1 << 64) for v in synthetic.splitmix64(xs).tolist()]
    assert got == expect and x.numel() == 3


def test_generator_ranges_and_determinism():
    a = synthetic.int8th(7, 4, (1000,))
    assert torch.equal(a, synthetic.int8th(7, 4, (1000,)))
    v = (a.float() * 8)
    assert v.min() >= -8 and v.max() <= 8 and torch.equal(v, v.round())
    assert len(torch.unique(v)) == 17
    n = synthetic.normal_bf16(7, 1, (200000,)).double()
    assert abs(n.mean()) < 0.02 and abs(n.std() - 1) < 0.02
    p = synthetic.permutation(3, 10, 1000)
    assert torch.equal(torch.sort(p).values, torch.arange(1000))


def test_query_rows_generated_alone_equal_the_full_tensor():
    w = synthetic.Workload(**{**synthetic.WORKLOADS["prefill_L32K"].__dict__, "L": 700})
    full = synthetic.prefill_inputs(w)
    rows = np.array([0, 1, 255, 256, 511, 699], np.int64)
    assert torch.equal(synthetic.prefill_q_rows(w, rows), full["q"][torch.from_numpy(rows)])
    rest = synthetic.prefill_inputs(w, without_q=True)
    assert "q" not in rest and all(torch.equal(rest[k], full[k])
                                   for k in ("k", "v", "q_idx", "k_idx"))


# ----------------------------------------------------------------------------------------------
# Hand-worked fixtures
# ----------------------------------------------------------------------------------------------
def test_golden_uniform_case():
    c = _parse_golden()["uniform"]
    L, B, k, G, Hq, di, d = (int(c[x]) for x in ("L", "B", "k", "G", "Hq", "di", "d"))
    k_idx = _bf(c["k_idx"])
    q_idx = torch.zeros(L, G, di, dtype=torch.bfloat16)
    q_idx[:, 0, :] = _bf(c["q_idx_group0"])
    q_idx[:, 1, :] = _bf(c["q_idx_group1"])
    sel = oracle.select_prefill(q_idx, k_idx, B, k)
    assert sel.tolist()[0] == [[int(x) for x in r] for r in c["sel_group0"]]
    assert sel.tolist()[1] == [[int(x) for x in r] for r in c["sel_group1"]]
    bs = oracle.block_scores_prefill(q_idx, k_idx, B)
    assert bs.tolist()[0] == c["bs_group0"] and bs.tolist()[1] == c["bs_group1"]
    q = torch.zeros(L, Hq, d, dtype=torch.bfloat16)
    kk = torch.zeros(L, G, d, dtype=torch.bfloat16)
    vv = torch.zeros(L, G, d, dtype=torch.bfloat16)
    for j in range(L):
        for g in range(G):
            vv[j, g] = _bf([j, g + 1])
    o, lse = oracle.attn_prefill(q, kk, vv, sel, B, k, float(c["scale"]))
    for h in range(Hq):
        np.testing.assert_allclose(o[:, h, 0], c[f"o0_head{h}"], rtol=0, atol=1e-12)
        np.testing.assert_allclose(o[:, h, 1], h + 1, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[h], np.log(c[f"tsize_head{h}"]), rtol=0, atol=1e-12)


def test_golden_weighted_case():
    c = _parse_golden()["weighted"]
    q = _bf([[[1, 0]], [[1, 0]]])
    kk = _bf([[[0, 0]], [[2, 0]]])
    vv = _bf([[[1, 0]], [[0, 1]]])
    sel = np.array([[[0], [0]]], np.int32)
    o, lse = oracle.attn_prefill(q, kk, vv, sel, 2, 1, 0.5)
    np.testing.assert_allclose(o[0, 0], c["o_row0"], atol=1e-14)
    np.testing.assert_allclose(o[1, 0], c["o_row1"], atol=1e-14)
    np.testing.assert_allclose(lse[0], [c["lse_row0"][0], c["lse_row1"][0]], atol=1e-14)


# ----------------------------------------------------------------------------------------------
# Brute force on tiny inputs
# ----------------------------------------------------------------------------------------------
def brute_select(qi: np.ndarray, ki: np.ndarray, B: int, k: int) -> np.ndarray:
    L, G, _ = qi.shape
    s = np.einsum("igd,jd->gij", qi, ki)
    sel = np.full((G, L, k), -1, np.int32)
    for g in range(G):
        for i in range(L):
            bi = i // B
            ranked = sorted((-s[g, i, b * B:(b + 1) * B].max(), b) for b in range(bi))
            chosen = sorted([b for _, b in ranked[:k - 1]] + [bi])
            sel[g, i, :len(chosen)] = chosen
    return sel


def brute_attn(q, kk, vv, sel, B, scale):
    from scipy.special import logsumexp
    L, Hq, d = q.shape
    G = kk.shape[1]
    hpg = Hq // G
    o = np.zeros((L, Hq, d))
    lse = np.zeros((Hq, L))
    j = np.arange(L)
    for h in range(Hq):
        g = h // hpg
        z = scale * q[:, h, :] @ kk[:, g, :].T
        mask = np.zeros((L, L), bool)
        for i in range(L):
            blocks = [b for b in sel[g, i] if b >= 0]
            mask[i] = np.isin(j // B, blocks) & (j <= i)
        z = np.where(mask, z, -np.inf)
        lse[h] = logsumexp(z, axis=1)
        p = np.exp(z - lse[h][:, None])
        o[:, h, :] = p @ vv[:, g, :]
    return o, lse


@pytest.mark.parametrize("L,B,G,k,seed", [(1, 4, 1, 2, 0), (17, 4, 2, 3, 1), (64, 8, 3, 2, 2),
                                          (50, 4, 1, 5, 3), (40, 8, 2, 1, 4), (96, 4, 4, 4, 5)])
def test_selection_matches_bruteforce(L, B, G, k, seed):
    di = 8
    qi = synthetic.int8th(seed, 4, (L, G, di))
    ki = synthetic.int8th(seed, 5, (L, di))
    sel, score = oracle.select_prefill(qi, ki, B, k, want_score=True)
    ref = brute_select(qi.double().numpy(), ki.double().numpy(), B, k)
    np.testing.assert_array_equal(sel, ref)
    # scores of selected non-local blocks are the block max of raw dot products
    s = np.einsum("igd,jd->gij", qi.double().numpy(), ki.double().numpy())
    for g in range(G):
        for i in range(L):
            for r in range(k):
                b = sel[g, i, r]
                if b < 0:
                    assert score[g, i, r] == -np.inf
                elif b == i // B:
                    assert score[g, i, r] == np.inf
                else:
                    assert score[g, i, r] == s[g, i, b * B:(b + 1) * B].max()


@pytest.mark.parametrize("L,B,G,seed", [(1, 4, 1, 0), (17, 4, 2, 1), (64, 8, 3, 2), (50, 4, 1, 3),
                                       (96, 4, 4, 5)])
def test_block_scores_match_dense_pooling(L, B, G, seed):
    """Exported block scores against a dense numpy formulation: the L x L score matrix padded to
    whole blocks with -inf, reshaped and reduced by max, then the causal mask (+inf on the
    diagonal block, -inf above it)."""
    di = 8
    qi = synthetic.int8th(seed, 4, (L, G, di))
    ki = synthetic.int8th(seed, 5, (L, di))
    bs = oracle.block_scores_prefill(qi, ki, B)
    nb = (L + B - 1) // B
    s = np.full((G, L, nb * B), -np.inf)
    s[:, :, :L] = np.einsum("igd,jd->gij", qi.double().numpy(), ki.double().numpy())
    pooled = s.reshape(G, L, nb, B).max(axis=3)
    own = (np.arange(L) // B)[:, None]
    blk = np.arange(nb)[None, :]
    ref = np.where(blk < own, pooled, np.where(blk == own, np.inf, -np.inf))
    np.testing.assert_array_equal(bs, np.broadcast_to(ref, bs.shape))
    rows = np.array([0, L - 1, L // 2], np.int64)
    np.testing.assert_array_equal(oracle.block_scores_prefill(qi, ki, B, rows=rows), bs[:, rows])


@pytest.mark.parametrize("L,B,G,k,seed", [(17, 4, 2, 3, 1), (64, 8, 3, 2, 2), (96, 4, 4, 4, 5)])
def test_block_scores_rank_to_the_selection(L, B, G, k, seed):
    """The selection is the local block plus the k-1 best exported scores below it (ties to the
    lower id, a stable sort on the negated score), and the selection's scores are gathered from
    the exported row."""
    di = 8
    qi = synthetic.int8th(seed, 4, (L, G, di))
    ki = synthetic.int8th(seed, 5, (L, di))
    sel, score = oracle.select_prefill(qi, ki, B, k, want_score=True)
    bs = oracle.block_scores_prefill(qi, ki, B)
    for g in range(G):
        for i in range(L):
            bi = i // B
            order = np.argsort(-bs[g, i, :bi], kind="stable")[:k - 1]
            want = sorted(order.tolist() + [bi])
            assert sel[g, i].tolist() == want + [-1] * (k - len(want))
            for r in range(len(want)):
                assert score[g, i, r] == bs[g, i, sel[g, i, r]]


@pytest.mark.parametrize("L,B,Hq,G,k,seed", [(33, 4, 4, 2, 3, 0), (64, 8, 6, 3, 2, 1),
                                             (29, 4, 2, 1, 4, 2)])
def test_attention_matches_dense_masked(L, B, Hq, G, k, seed):
    d, di = 16, 8
    q = synthetic.normal_bf16(seed, 1, (L, Hq, d))
    kk = synthetic.normal_bf16(seed, 2, (L, G, d))
    vv = synthetic.normal_bf16(seed, 3, (L, G, d))
    sel = oracle.select_prefill(synthetic.int8th(seed, 4, (L, G, di)),
                                synthetic.int8th(seed, 5, (L, di)), B, k)
    scale = 1 / math.sqrt(d)
    o, lse = oracle.attn_prefill(q, kk, vv, sel, B, k, scale)
    ro, rl = brute_attn(q.double().numpy(), kk.double().numpy(), vv.double().numpy(), sel, B,
                        scale)
    np.testing.assert_allclose(o, ro, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, rl, rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------------------------
# Invariants against library routines
# ----------------------------------------------------------------------------------------------
def _sdpa(q, kk, vv, scale, mask=None):
    import torch.nn.functional as F
    Q = q.double().permute(1, 0, 2)[None]
    K = kk.double().permute(1, 0, 2)[None]
    V = vv.double().permute(1, 0, 2)[None]
    if mask is None:
        out = F.scaled_dot_product_attention(Q, K, V, is_causal=True, scale=scale, enable_gqa=True)
    else:
        out = F.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale, enable_gqa=True)
    return out[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("L,B,Hq,G,k", [(128, 16, 8, 2, 8), (100, 8, 4, 4, 13), (256, 32, 4, 1, 8)])
def test_full_budget_equals_causal_gqa(L, B, Hq, G, k):
    assert k * B >= L
    d, di = 32, 16
    q = synthetic.normal_bf16(11, 1, (L, Hq, d))
    kk = synthetic.normal_bf16(11, 2, (L, G, d))
    vv = synthetic.normal_bf16(11, 3, (L, G, d))
    sel = oracle.select_prefill(synthetic.int8th(11, 4, (L, G, di)),
                                synthetic.int8th(11, 5, (L, di)), B, k)
    scale = 1 / math.sqrt(d)
    o, lse = oracle.attn_prefill(q, kk, vv, sel, B, k, scale)
    np.testing.assert_allclose(o, _sdpa(q, kk, vv, scale), rtol=0, atol=1e-12)
    # lse against torch.logsumexp of the causally masked logits
    hpg = Hq // G
    for h in range(Hq):
        z = scale * q[:, h].double() @ kk[:, h // hpg].double().T
        z = z.masked_fill(torch.triu(torch.ones(L, L, dtype=torch.bool), 1), -math.inf)
        np.testing.assert_allclose(lse[h], torch.logsumexp(z, 1).numpy(), rtol=0, atol=1e-12)


def test_k1_is_block_local_causal():
    L, B, Hq, G, d, di = 70, 8, 4, 2, 16, 8
    q = synthetic.normal_bf16(5, 1, (L, Hq, d))
    kk = synthetic.normal_bf16(5, 2, (L, G, d))
    vv = synthetic.normal_bf16(5, 3, (L, G, d))
    sel = oracle.select_prefill(synthetic.int8th(5, 4, (L, G, di)),
                                synthetic.int8th(5, 5, (L, di)), B, 1)
    assert (sel[..., 0] == np.arange(L) // B).all()
    scale = 0.3
    o, _ = oracle.attn_prefill(q, kk, vv, sel, B, 1, scale)
    i = torch.arange(L)
    mask = (i[None, :] <= i[:, None]) & (i[None, :] // B == i[:, None] // B)
    np.testing.assert_allclose(o, _sdpa(q, kk, vv, scale, mask), rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------------------------
# Tie rule, permutation invariance, decode/prefill consistency
# ----------------------------------------------------------------------------------------------
def test_tie_prefers_lower_block():
    L, B, G, di, k = 48, 8, 1, 8, 3  # blocks 0..5, query block 5 -> candidates 0..4, 2 slots
    qi = synthetic.int8th(9, 4, (L, G, di))
    ki = synthetic.int8th(9, 5, (L, di)).clone()
    # make blocks 1 and 3 exact copies of block 4: equal pooled scores for every query
    for b in (1, 3):
        ki[b * B:(b + 1) * B] = ki[4 * B:5 * B]
    sel, score = oracle.select_prefill(qi, ki, B, k, want_score=True)
    for i in range(5 * B, L):
        sc = {b: s for b, s in zip(sel[0, i], score[0, i]) if 0 <= b < 5}
        chosen = sorted(sc)
        # whenever the tied group is partly chosen, the lower ids win
        tied = [b for b in (1, 3, 4) if b in chosen]
        if 0 < len(tied) < 3:
            assert tied == [1, 3, 4][:len(tied)], (i, sel[0, i])


def test_permutation_inside_nonlocal_block_is_invariant():
    L, B, Hq, G, d, di, k = 64, 8, 4, 2, 16, 8, 3
    q = synthetic.normal_bf16(21, 1, (L, Hq, d))
    kk = synthetic.normal_bf16(21, 2, (L, G, d))
    vv = synthetic.normal_bf16(21, 3, (L, G, d))
    qi = synthetic.int8th(21, 4, (L, G, di))
    ki = synthetic.int8th(21, 5, (L, di))
    sel = oracle.select_prefill(qi, ki, B, k)
    o, lse = oracle.attn_prefill(q, kk, vv, sel, B, k, 0.25)
    perm = torch.arange(L)
    perm[2 * B:3 * B] = 2 * B + synthetic.permutation(21, 99, B)
    sel2 = oracle.select_prefill(qi, ki[perm], B, k)
    np.testing.assert_array_equal(sel, sel2)
    o2, lse2 = oracle.attn_prefill(q, kk[perm], vv[perm], sel2, B, k, 0.25)
    rows = np.arange(3 * B, L)  # queries for which block 2 is wholly in the past
    np.testing.assert_allclose(o2[rows], o[rows], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2[:, rows], lse[:, rows], rtol=0, atol=1e-12)


def test_decode_equals_last_prefill_row():
    B, G, Hq, d, di, k = 8, 2, 4, 16, 8, 3
    lens = [1, 8, 9, 30, 57]
    maxp = max((n + B - 1) // B for n in lens)
    P = sum((n + B - 1) // B for n in lens) + 2
    perm = synthetic.permutation(4, 10, P)
    pools = {
        "k_idx_pool": synthetic.int8th(4, 5, (P, B, di)),
        "k_pool": synthetic.normal_bf16(4, 2, (P, G, B, d)),
        "v_pool": synthetic.normal_bf16(4, 3, (P, G, B, d)),
    }
    pt = torch.full((len(lens), maxp), -1, dtype=torch.int32)
    off = 0
    for s, n in enumerate(lens):
        npg = (n + B - 1) // B
        pt[s, :npg] = perm[off:off + npg].to(torch.int32)
        off += npg
    q_dec = synthetic.normal_bf16(4, 1, (len(lens), Hq, d))
    qi_dec = synthetic.int8th(4, 4, (len(lens), G, di))
    seq = torch.tensor(lens, dtype=torch.int32)
    sel_d, sc_d = oracle.select_decode(qi_dec, pools["k_idx_pool"], pt, seq, B, k, want_score=True)
    bs_d = oracle.block_scores_decode(qi_dec, pools["k_idx_pool"], pt, seq, B)
    o_d, lse_d = oracle.attn_decode(q_dec, pools["k_pool"], pools["v_pool"], pt, seq, sel_d, B, k,
                                    0.25)
    for s, n in enumerate(lens):
        pages = pt[s, :(n + B - 1) // B].long()
        ki = pools["k_idx_pool"][pages].reshape(-1, di)[:n]
        kk = pools["k_pool"][pages].permute(0, 2, 1, 3).reshape(-1, G, d)[:n]
        vv = pools["v_pool"][pages].permute(0, 2, 1, 3).reshape(-1, G, d)[:n]
        qi = torch.zeros(n, G, di, dtype=torch.bfloat16)
        qi[n - 1] = qi_dec[s]
        q = torch.zeros(n, Hq, d, dtype=torch.bfloat16)
        q[n - 1] = q_dec[s]
        rows = np.array([n - 1])
        sel_p, sc_p = oracle.select_prefill(qi, ki, B, k, rows=rows, want_score=True)
        np.testing.assert_array_equal(sel_p[:, 0], sel_d[:, s])
        np.testing.assert_array_equal(sc_p[:, 0], sc_d[:, s])
        bs_p = oracle.block_scores_prefill(qi, ki, B, rows=rows)
        npg = (n + B - 1) // B
        np.testing.assert_array_equal(bs_p[:, 0], bs_d[:, s, :npg])
        assert (bs_d[:, s, npg:] == -np.inf).all()
        o_p, lse_p = oracle.attn_prefill(q, kk, vv, sel_p, B, k, 0.25, rows=rows)
        np.testing.assert_allclose(o_p[0], o_d[s], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse_p[:, 0], lse_d[:, s], rtol=0, atol=1e-13)


def test_index_scores_exact_in_fp32():
    """Integer/8 index inputs: every partial dot product is a multiple of 1/64 below 2**8 in
    magnitude, so fp32 accumulation in any order equals the fp64 value.  This is what makes a
    bit-exact selection comparison against fp32 tensor-core accumulation legitimate."""
    qi = synthetic.int8th(3, 4, (64, 128)).double()
    ki = synthetic.int8th(3, 5, (256, 128)).double()
    exact = qi @ ki.T
    f32_fwd = torch.zeros(64, 256, dtype=torch.float32)
    f32_rev = torch.zeros(64, 256, dtype=torch.float32)
    for dd in range(128):
        f32_fwd += (qi[:, dd:dd + 1] * ki[:, dd][None]).float()
        f32_rev += (qi[:, 127 - dd:128 - dd] * ki[:, 127 - dd][None]).float()
    assert torch.equal(f32_fwd.double(), exact) and torch.equal(f32_rev.double(), exact)
    ones = torch.ones(128, dtype=torch.float64)
    assert float(ones @ ones) == 128.0


def test_compact_query_rows_match_full():
    L, B, Hq, G, d, di, k = 80, 8, 4, 2, 16, 8, 3
    q = synthetic.normal_bf16(31, 1, (L, Hq, d))
    kk = synthetic.normal_bf16(31, 2, (L, G, d))
    vv = synthetic.normal_bf16(31, 3, (L, G, d))
    rows = np.array([0, 7, 8, 40, 79])
    sel = oracle.select_prefill(synthetic.int8th(31, 4, (L, G, di)),
                                synthetic.int8th(31, 5, (L, di)), B, k, rows=rows)
    o1, l1 = oracle.attn_prefill(q, kk, vv, sel, B, k, 0.3, rows=rows)
    o2, l2 = oracle.attn_prefill(q[torch.tensor(rows)], kk, vv, sel, B, k, 0.3, rows=rows,
                                 q_compact=True)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


# ------------------------------------------------------------------------------------------
# E4M3 index vectors (the FP8 indexer): the oracle decodes the codes itself
# ------------------------------------------------------------------------------------------
def test_e4m3_decoder_matches_library_and_definition():
    """Every code against torch's float8_e4m3fn conversion (a library routine), plus values the
    format definition fixes: 1.0, -1.0, the largest normal 448, the smallest normal 2^-6, the
    smallest subnormal 2^-9, and the NaN code."""
    v = oracle.e4m3_values()
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    nan = np.isnan(v)
    assert np.array_equal(nan, np.isnan(lib))
    assert np.array_equal(v[~nan], lib[~nan].astype(np.float64))
    assert (v[0x38], v[0xB8], v[0x7E], v[0x08], v[0x01]) == (1.0, -1.0, 448.0, 2.0 ** -6, 2.0 ** -9)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]


def test_integer_eighths_are_exact_in_e4m3():
    """The index inputs (integers in [-8, 8] over 8) lose nothing in E4M3: the FP8 indexer
    scores them exactly as the bf16 one does."""
    x = torch.arange(-8, 9, dtype=torch.float32) / 8
    codes = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_values()[codes], x.numpy().astype(np.float64))


@pytest.mark.parametrize("L,G,k,seed", [(700, 2, 4, 3), (1300, 4, 16, 4)])
def test_e4m3_selection_equals_bf16_selection(L, G, k, seed):
    w = synthetic.Workload("e4", "prefill", L=L, Hq=16 * G, G=G, k=k, seed=seed)
    a = synthetic.prefill_inputs(w, index_only=True)
    b = synthetic.prefill_inputs(w, index_only=True, index_dtype="e4m3")
    assert b["q_idx"].dtype == torch.float8_e4m3fn
    sa, ca = oracle.select_prefill(a["q_idx"], a["k_idx"], w.B, k, want_score=True)
    sb, cb = oracle.select_prefill(b["q_idx"], b["k_idx"], w.B, k, want_score=True)
    assert np.array_equal(sa, sb) and np.array_equal(ca, cb)
    rows = np.array([0, w.B - 1, w.B, L // 2, L - 1], np.int64)
    assert np.array_equal(oracle.block_scores_prefill(a["q_idx"], a["k_idx"], w.B, rows=rows),
                          oracle.block_scores_prefill(b["q_idx"], b["k_idx"], w.B, rows=rows))
