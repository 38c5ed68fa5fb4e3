"""The checked build (libmsa_debug.so, loaded when MSA_DEBUG_CHECKS is set), on the GPU.

Its kernels check the indices they derive before each access, and with MSA_DEBUG_CHECKS set it
validates the caller's selections, sequence lengths and page tables before the kernels run.  The
checks stand in for a memory checker: on valid inputs no check may fire and every output must be
bit-identical to the release build's; on malformed inputs made on the host (none of which can
address memory out of range: the release kernels skip or tolerate them) the first failed check
must be recorded with its site and row.

The checked build runs in a child process (the library is chosen when it is first loaded), which
saves its outputs; this process runs the release build on the same seeded inputs and compares.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BOUNDS = 6


def _prefill_case():
    w = synthetic.Workload(**{**synthetic.WORKLOADS["prefill_L32K"].__dict__, "L": 2125,
                              "seed": 631})
    return w, synthetic.prefill_inputs(w, device="cuda")


def _decode_case():
    w = synthetic.Workload(**{**synthetic.WORKLOADS["decode_b64_16K_256K"].__dict__,
                              "seed": 632})
    inp = synthetic.decode_inputs(w, device="cuda", batch=12, n_lo=200, n_hi=6000)
    return inp["workload"], inp


def _valid_outputs(msa):
    """Every call of the path on valid inputs; returns the outputs and the status words."""
    out, status = {}, []
    w, d = _prefill_case()
    cfg = msa.config(w.G, w.hpg, w.k, w.scale)
    ws = torch.zeros(max(msa.msa_index_select_workspace(cfg, w.L, w.L),
                         msa.msa_attn_prefill_workspace(cfg, w.L)), dtype=torch.uint8,
                     device="cuda")
    out["sel"] = msa.msa_index_select(cfg, d["q_idx"], d["k_idx"], ws=ws)
    out["o"], out["lse"] = msa.msa_attn_prefill(cfg, d["q"], d["k"], d["v"], out["sel"], ws=ws)
    # context-parallel index branch: two shards of the key blocks, then the merge
    nb = (w.L + w.B - 1) // w.B
    cand = [msa.msa_index_candidates(cfg, d["q_idx"], d["k_idx"][b0 * w.B:min(b1 * w.B, w.L)],
                                     L=w.L, block_begin=b0, block_end=b1, ws=ws)
            for b0, b1 in ((0, nb // 2), (nb // 2, nb))]
    out["sel_cp"] = msa.msa_index_merge(cfg, torch.stack([c[0] for c in cand]),
                                        torch.stack([c[1] for c in cand]), ws=ws)
    status.append(msa.msa_get_device_status(ws))
    wd, dd = _decode_case()
    cfgd = msa.config(wd.G, wd.hpg, wd.k, wd.scale)
    paged = msa.paged_kv(dd["k_idx_pool"], dd["k_pool"], dd["v_pool"], dd["page_table"],
                         dd["seq_lens"])
    wsd = torch.zeros(max(msa.msa_index_select_workspace(cfgd, wd.batch, 0, paged),
                          msa.msa_attn_decode_workspace(cfgd, paged)), dtype=torch.uint8,
                      device="cuda")
    out["dsel"] = msa.msa_index_select(cfgd, dd["q_idx"], paged=paged, ws=wsd)
    out["do"], out["dlse"] = msa.msa_attn_decode(cfgd, dd["q"], paged, out["dsel"], ws=wsd)
    status.append(msa.msa_get_device_status(wsd))
    return {k: v.cpu() for k, v in out.items()}, status


def _malformed(msa, sel_p):
    """Host-made malformed inputs, one per call, each on a freshly reset workspace; returns
    (status, record) per case."""
    res = {}
    w, d = _prefill_case()
    cfg = msa.config(w.G, w.hpg, w.k, w.scale)
    ws = torch.zeros(msa.msa_attn_prefill_workspace(cfg, w.L), dtype=torch.uint8, device="cuda")

    def prefill(name, sel):
        msa.msa_reset_device_status(ws)
        msa.msa_attn_prefill(cfg, d["q"], d["k"], d["v"], sel, ws=ws)
        res[name] = (msa.msa_get_device_status(ws), msa.debug_record(ws))

    # group 1, query 1000 (block 7): two ids swapped, so the row is not ascending
    bad = sel_p.clone()
    row = bad[1, 1000]
    assert row[0] >= 0 and row[1] >= 0
    row[0], row[1] = row[1].clone(), row[0].clone()
    prefill("order", bad)
    # group 0, query 900 (block 7): its own block replaced by padding
    bad = sel_p.clone()
    n = int((bad[0, 900] >= 0).sum())
    assert int(bad[0, 900, n - 1]) == 900 // w.B
    bad[0, 900, n - 1] = -1
    prefill("local", bad)
    # group 3, query 5 (block 0): an id past the query's block
    bad = sel_p.clone()
    assert int(bad[3, 5, 0]) == 0 and int(bad[3, 5, 1]) == -1
    bad[3, 5, 0] = 2
    prefill("range", bad)

    wd, dd = _decode_case()
    cfgd = msa.config(wd.G, wd.hpg, wd.k, wd.scale)

    def decode(name, page_table, seq_lens):
        paged = msa.paged_kv(dd["k_idx_pool"], dd["k_pool"], dd["v_pool"], page_table, seq_lens)
        wsd = torch.zeros(max(msa.msa_index_select_workspace(cfgd, wd.batch, 0, paged),
                              msa.msa_attn_decode_workspace(cfgd, paged)), dtype=torch.uint8,
                          device="cuda")
        msa.msa_index_select(cfgd, dd["q_idx"], paged=paged, ws=wsd)
        res[name] = (msa.msa_get_device_status(wsd), msa.debug_record(wsd))

    pt = dd["page_table"].clone()
    pt[4, 0] = dd["num_pages"]  # one past the pool
    decode("page", pt, dd["seq_lens"])
    lens = dd["seq_lens"].clone()
    lens[7] = 0
    decode("seq_len", dd["page_table"], lens)
    return res


def _child(out_path):
    import block_sparse_long_msa_gb300 as msa
    assert msa.msa_debug_checks() == 3, msa.msa_debug_checks()
    assert os.path.basename(msa.lib()._name) == "libmsa_debug.so"
    out, status = _valid_outputs(msa)
    res = _malformed(msa, out["sel"].cuda())
    torch.save({"out": out, "status": status, "malformed": res}, out_path)


@pytest.fixture(scope="module")
def checked(tmp_path_factory):
    path = str(tmp_path_factory.mktemp("checked") / "out.pt")
    env = {**os.environ, "MSA_DEBUG_CHECKS": "1", "PYTHONPATH": ROOT}
    r = subprocess.run([sys.executable, os.path.abspath(__file__), path], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    return torch.load(path)


@pytest.fixture(scope="module")
def msa():
    import block_sparse_long_msa_gb300 as m
    assert m.msa_debug_checks() == 0, "the release build is expected in this process"
    return m


def test_checked_build_is_bit_identical_on_valid_inputs(checked, msa):
    assert checked["status"] == [0, 0]
    out, status = _valid_outputs(msa)
    assert status == [0, 0]
    for name, t in out.items():
        assert torch.equal(t, checked["out"][name]), name
    # and the selection is the oracle's (the release path's parity, through the checked build)
    w, d = _prefill_case()
    r_sel = oracle.select_prefill(d["q_idx"].cpu(), d["k_idx"].cpu(), w.B, w.k)
    np.testing.assert_array_equal(checked["out"]["sel"].numpy(), r_sel)
    np.testing.assert_array_equal(checked["out"]["sel_cp"].numpy(), r_sel)


def test_checked_build_records_each_malformed_input(checked):
    m = checked["malformed"]
    L = 2125
    assert m["order"] == (BOUNDS, {"site": "sel_order", "value": 1, "bound": 16,
                                   "row": 1 * L + 1000}), m["order"]
    st, rec = m["local"]
    assert st == BOUNDS and rec["site"] == "sel_local" and rec["row"] == 900, m["local"]
    assert rec["bound"] == 900 // 128 + 1
    assert m["range"] == (BOUNDS, {"site": "sel_range", "value": 2, "bound": 1,
                                   "row": 3 * L + 5}), m["range"]
    st, rec = m["page"]
    assert st == BOUNDS and rec["site"] == "page_id" and rec["row"] == 4, m["page"]
    assert rec["value"] == rec["bound"]
    _, inp = _decode_case()
    assert m["seq_len"] == (BOUNDS, {"site": "seq_len", "value": 0,
                                     "bound": inp["max_pages"] * 128 + 1, "row": 7}), m["seq_len"]


def test_release_build_tolerates_what_only_the_checked_build_rejects(msa):
    # an unsorted row addresses nothing out of range: the release kernels take the union of its
    # blocks, flag nothing, and give the sorted row's result
    w, d = _prefill_case()
    cfg = msa.config(w.G, w.hpg, w.k, w.scale)
    ws = torch.zeros(max(msa.msa_index_select_workspace(cfg, w.L, w.L),
                         msa.msa_attn_prefill_workspace(cfg, w.L)), dtype=torch.uint8,
                     device="cuda")
    sel = msa.msa_index_select(cfg, d["q_idx"], d["k_idx"], ws=ws)
    o, lse = msa.msa_attn_prefill(cfg, d["q"], d["k"], d["v"], sel, ws=ws)
    bad = sel.clone()
    row = bad[1, 1000]
    row[0], row[1] = row[1].clone(), row[0].clone()
    o2, lse2 = msa.msa_attn_prefill(cfg, d["q"], d["k"], d["v"], bad, ws=ws)
    assert msa.msa_get_device_status(ws) == 0
    assert msa.debug_record(ws) is None
    others = torch.ones(w.L, dtype=torch.bool)
    others[1000] = False
    assert torch.equal(o2[others], o[others])
    assert (o2[1000].float() - o[1000].float()).abs().max() <= 1e-2


if __name__ == "__main__":
    _child(sys.argv[1])
