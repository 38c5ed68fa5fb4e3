"""The C-ABI library builds, loads and exports every entry point include/msa.h declares; host
argument checks answer without touching a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from block_sparse_long_msa_gb300 import build
    build.build()
    import block_sparse_long_msa_gb300 as msa
    return msa.lib()


def _declared():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(msa_\w+)\s*\(", txt, re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    import block_sparse_long_msa_gb300 as msa
    declared = _declared()
    assert len(declared) >= 9
    # the release build and the checked build export the same calls
    for path in (lib._name, msa.DEBUG_LIB_PATH):
        out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True,
                             text=True, check=True).stdout
        exported = set(re.findall(r"\bT\s+(msa_\w+)", out))
        missing = [n for n in declared if n not in exported]
        assert not missing, (path, missing)
        assert set(msa.EXPORTS) <= exported


def test_checked_build_describes_itself_without_a_gpu(lib):
    import block_sparse_long_msa_gb300 as msa
    assert lib.msa_debug_checks() == 0
    rec = msa.MsaDebugRecord()
    assert lib.msa_get_debug_record(None, ctypes.byref(rec), None) == msa.MSA_ERR_INVALID_ARG
    dbg = ctypes.CDLL(msa.DEBUG_LIB_PATH)
    dbg.msa_debug_checks.restype = ctypes.c_int32
    # bit 0: the checked build; bit 1 follows MSA_DEBUG_CHECKS in this process's environment
    assert dbg.msa_debug_checks() & 1 == 1
    assert (dbg.msa_debug_checks() >> 1) == int(msa.checked_build_requested())


def test_status_strings(lib):
    import block_sparse_long_msa_gb300 as msa
    for s in range(7):
        assert msa.status_string(s)
    assert msa.status_string(0) == "ok"


def test_host_argument_checks(lib):
    import block_sparse_long_msa_gb300 as msa
    cfg = msa.config(4, 16, 16)
    # config errors return before any CUDA work
    bad = msa.config(4, 16, 17)
    assert lib.msa_index_select(ctypes.byref(bad), None, None, 0, None, None, None, None, 0,
                                None) == msa.MSA_ERR_UNSUPPORTED
    bad = msa.config(4, 16, 0)
    assert lib.msa_index_select(ctypes.byref(bad), None, None, 0, None, None, None, None, 0,
                                None) == msa.MSA_ERR_INVALID_ARG
    bad = msa.config(4, 16, 16, head_dim=64)
    assert lib.msa_attn_prefill(ctypes.byref(bad), None, None, None, 0, None, None, None, None,
                                0, None) == msa.MSA_ERR_UNSUPPORTED
    # null pointers
    assert lib.msa_index_select(ctypes.byref(cfg), None, None, 16, None, None, None, None, 0,
                                None) == msa.MSA_ERR_INVALID_ARG
    # misaligned pointer (never dereferenced: the check happens first)
    assert lib.msa_index_select(ctypes.byref(cfg), ctypes.c_void_p(0x1002),
                                ctypes.c_void_p(0x2000), 16, None, ctypes.c_void_p(0x3000), None,
                                ctypes.c_void_p(0x4000), 1 << 20, None) == msa.MSA_ERR_INVALID_ARG
    # more than four groups: refused on the host (pointers never dereferenced)
    g5 = msa.config(5, 16, 16)
    assert lib.msa_index_select(ctypes.byref(g5), ctypes.c_void_p(0x1000),
                                ctypes.c_void_p(0x2000), 16, None, ctypes.c_void_p(0x3000), None,
                                ctypes.c_void_p(0x4000), 1 << 20, None) == msa.MSA_ERR_UNSUPPORTED
    # a paged cache with an unknown K/V storage type is refused before any work
    pk = msa.MsaPagedKV(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 1, 1, 1, 7)
    assert lib.msa_attn_decode(ctypes.byref(cfg), ctypes.c_void_p(0x6000), ctypes.byref(pk),
                               ctypes.c_void_p(0x7000), ctypes.c_void_p(0x8000),
                               ctypes.c_void_p(0x9000), ctypes.c_void_p(0xa000), 1 << 20,
                               None) == msa.MSA_ERR_INVALID_ARG
    # workspace queries are pure host arithmetic
    assert msa.msa_index_select_workspace(cfg, 32768, 32768) >= msa.WS_HEADER_BYTES
    assert lib.msa_index_select_workspace(ctypes.byref(bad), 1, 1, None) == 0


def test_prefill_length_limit_is_checked_on_the_host(lib):
    """The main branch supports L up to 1,572,864 tokens (the schedule keeps a 16-byte token mask
    per key block in shared memory); one token more is refused before any GPU work, with
    aligned stand-in pointers that are never dereferenced."""
    import block_sparse_long_msa_gb300 as msa
    cfg = msa.config(4, 16, 16)
    L_MAX = 1572864
    P = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(8)]

    def call(L):
        return lib.msa_attn_prefill(ctypes.byref(cfg), P[0], P[1], P[2], L, P[3], P[4], P[5],
                                    P[6], 1 << 62, None)

    assert call(L_MAX + 1) == msa.MSA_ERR_UNSUPPORTED
    assert msa.msa_attn_prefill_launches(cfg, L_MAX) == 24 * 7  # 24 passes of 65,536 queries
    assert msa.msa_attn_prefill_launches(cfg, L_MAX + 1) == 0
    assert msa.msa_attn_prefill_workspace(cfg, L_MAX) > 0


def test_launch_count_and_index_dtype_config(lib):
    """The prefill launch count is host arithmetic (seven kernels per 65,536-token chunk); an
    index_dtype other than bf16 (0) or e4m3 (1) is an invalid config."""
    import block_sparse_long_msa_gb300 as msa
    cfg = msa.config(4, 16, 16)
    assert msa.msa_prefill_chunk_tokens(cfg, 32768) == 32768
    assert msa.msa_attn_prefill_launches(cfg, 32768) == 7
    assert msa.msa_attn_prefill_launches(cfg, 131072) == 14
    assert msa.msa_attn_prefill_launches(cfg, 1 << 20) == 7 * 16
    assert msa.msa_attn_prefill_launches(cfg, 0) == 0
    assert msa.msa_attn_prefill_launches(msa.config(4, 16, 16, index_dtype="e4m3"), 2048) == 7
    bad = msa.config(4, 16, 16)
    bad.index_dtype = 2
    assert msa.msa_attn_prefill_launches(bad, 2048) == 0
    assert lib.msa_index_select(ctypes.byref(bad), None, None, 0, None, None, None, None, 0,
                                None) == msa.MSA_ERR_INVALID_ARG


def test_empty_inputs_return_before_any_gpu_work(lib):
    """L = 0 (prefill) and batch = 0 (decode) are valid calls that enqueue nothing."""
    import block_sparse_long_msa_gb300 as msa
    cfg = msa.config(4, 16, 16)
    p = ctypes.c_void_p(0x10000)  # 16-byte aligned, never dereferenced
    ws = msa.msa_attn_prefill_workspace(cfg, 0)
    assert lib.msa_attn_prefill(ctypes.byref(cfg), p, p, p, 0, p, p, p, p, ws, None) == msa.MSA_OK
    assert lib.msa_index_select(ctypes.byref(cfg), p, p, 0, None, p, None, p,
                                msa.msa_index_select_workspace(cfg, 0, 0), None) == msa.MSA_OK
    wsi = msa.msa_index_select_workspace(cfg, 0, 0)
    assert lib.msa_index_select_scores(ctypes.byref(cfg), p, p, 0, None, p, None, p, p, wsi,
                                       None) == msa.MSA_OK
    # the score export requires its output
    assert lib.msa_index_select_scores(ctypes.byref(cfg), p, p, 0, None, p, None, None, p, wsi,
                                       None) == msa.MSA_ERR_INVALID_ARG
    paged = msa.MsaPagedKV(0x10000, 0x10000, 0x10000, 0x10000, 0x10000, 0, 1, 1, 0)
    wsd = msa.msa_attn_decode_workspace(cfg, paged)
    assert lib.msa_attn_decode(ctypes.byref(cfg), p, ctypes.byref(paged), p, p, p, p, wsd,
                               None) == msa.MSA_OK
    assert lib.msa_index_select(ctypes.byref(cfg), p, None, 0, ctypes.byref(paged), p, None, p,
                                msa.msa_index_select_workspace(cfg, 0, 0, paged), None) == msa.MSA_OK


def test_block_scores_output_is_checked_before_any_call():
    """The binding rejects a block_scores buffer of the wrong shape or type before it reaches the
    library (no device work is enqueued)."""
    import torch
    import block_sparse_long_msa_gb300 as msa
    cfg = msa.config(4, 16, 16)
    q_idx = torch.zeros(300, 4, 128, dtype=torch.bfloat16)
    k_idx = torch.zeros(300, 128, dtype=torch.bfloat16)
    for bad in (torch.zeros(4, 300, 2), torch.zeros(4, 300, 3, dtype=torch.float64)):
        with pytest.raises(msa.MsaError):
            msa.msa_index_select_scores(cfg, q_idx, k_idx, block_scores=bad)
