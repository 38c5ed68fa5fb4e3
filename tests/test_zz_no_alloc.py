"""msa_attn_prefill_noalloc, the entry point for callers that cannot allocate device memory
(they are handed only inputs and outputs), must give the result of msa_attn_prefill with a
caller workspace.  Both run the same deterministic kernels, and every (token, group, block)
partial and the fixed-order combine depend only on that token's rows, so the outputs must be
bit-identical even though the no-allocation entry point works in passes of 128 queries.  A set of
rows is also checked against the oracle.  It is called through the C ABI twice in a row: the
second call reuses the library's static scratch that the first one left behind.

This file sorts last so that a run stopping at the first failure has run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = pytest.mark.gpu

from parity_bar import MAX_ABS, MEAN_ABS, o_bar  # the bar of the other parity tests


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_workspace_entry_point_twice():
    import block_sparse_long_msa_gb300 as msa
    lib = msa.lib()
    fn = lib.msa_attn_prefill_noalloc
    fn.argtypes = [ctypes.POINTER(msa.MsaConfig)] + [ctypes.c_void_p] * 3 + [ctypes.c_int64] + \
        [ctypes.c_void_p] * 5
    fn.restype = ctypes.c_int
    base = synthetic.WORKLOADS["prefill_L32K"]
    # several 128-query passes per call, a ragged tail, and two different inputs in a row
    for call, (L, seed) in enumerate([(1100, 501), (777, 502)]):
        w = synthetic.Workload(**{**base.__dict__, "L": L, "seed": seed})
        host = synthetic.prefill_inputs(w, device="cpu")
        inp = {k: v.cuda() for k, v in host.items() if isinstance(v, torch.Tensor)}
        cfg = msa.config(w.G, w.hpg, w.k, w.scale)
        sel = msa.msa_index_select(cfg, inp["q_idx"], inp["k_idx"])
        o_ref, lse_ref = msa.msa_attn_prefill(cfg, inp["q"], inp["k"], inp["v"], sel)
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        rc = fn(ctypes.byref(cfg), _p(inp["q"]), _p(inp["k"]), _p(inp["v"]), L, _p(sel), _p(o),
                _p(lse), _p(status), stream)
        assert rc == msa.MSA_OK, msa.status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
        assert torch.equal(o, o_ref), f"call {call}: O differs from the workspace entry point"
        assert torch.equal(lse, lse_ref), f"call {call}: LSE differs"
        # and a set of rows against the oracle, at the tolerance of the other prefill tests
        rows = np.array(sorted({0, 1, 127, 128, 129, L // 2, L - 129, L - 2, L - 1}), np.int64)
        r_sel = oracle.select_prefill(host["q_idx"], host["k_idx"], w.B, w.k, rows=rows)
        np.testing.assert_array_equal(sel.cpu().numpy()[:, rows], r_sel)
        r_o, r_lse = oracle.attn_prefill(host["q"], host["k"], host["v"], r_sel, w.B, w.k,
                                         w.scale, rows=rows)
        err = np.abs(o.float().cpu().numpy()[rows] - r_o)
        lerr = np.abs(lse.cpu().numpy()[:, rows] - r_lse)
        assert (err <= o_bar(r_o)).all() and err.mean() <= MEAN_ABS, (call, err.max())
        assert lerr.max() <= MAX_ABS and lerr.mean() <= MEAN_ABS, (call, lerr.max())


def test_noalloc_rejects_oversized_problem():
    import block_sparse_long_msa_gb300 as msa
    lib = msa.lib()
    fn = lib.msa_attn_prefill_noalloc
    fn.argtypes = [ctypes.POINTER(msa.MsaConfig)] + [ctypes.c_void_p] * 3 + [ctypes.c_int64] + \
        [ctypes.c_void_p] * 5
    fn.restype = ctypes.c_int
    cfg = msa.config(4, 16, 16)
    x = torch.zeros(64, dtype=torch.int32, device="cuda")  # never read: rejected on the host
    rc = fn(ctypes.byref(cfg), _p(x), _p(x), _p(x), 2 * 1536 * 1024, _p(x), _p(x), _p(x), None,
            None)
    assert rc == msa.MSA_ERR_UNSUPPORTED
