"""MiniMax Sparse Attention (MSA) for GB300: Python binding of libmsa (include/msa.h).

Argument marshalling only: every step of the operator runs in the CUDA kernels of libmsa.so.
torch supplies device memory (outputs, workspace) and the current stream.  If the library has
not been built, every call raises; there is no CPU fallback.

With the environment variable MSA_DEBUG_CHECKS set (to anything but "" or "0") when the library
is first loaded, the checked build libmsa_debug.so is loaded instead: the same calls, with
bounds checks in the kernels and validation of the caller's index tensors (include/msa.h,
"Checked build"); debug_record() reads its record of the first failed check.
"""
from __future__ import annotations

import ctypes
import math
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmsa.so")
DEBUG_LIB_PATH = os.path.join(_HERE, "_build", "libmsa_debug.so")

MSA_OK, MSA_ERR_INVALID_ARG, MSA_ERR_UNSUPPORTED, MSA_ERR_WORKSPACE = 0, 1, 2, 3
MSA_ERR_CUDA, MSA_ERR_DEVICE_TIMEOUT, MSA_ERR_DEVICE_BOUNDS = 4, 5, 6
WS_HEADER_BYTES = 256

EXPORTS = ("msa_index_select_workspace", "msa_index_select", "msa_index_select_scores",
           "msa_index_candidates", "msa_index_merge",
           "msa_attn_prefill_workspace",
           "msa_attn_prefill", "msa_attn_prefill_marked", "msa_prefill_chunk_tokens",
           "msa_attn_prefill_launches",
           "msa_attn_decode_workspace", "msa_attn_decode",
           "msa_get_device_status", "msa_reset_device_status", "msa_status_string",
           "msa_debug_checks", "msa_get_debug_record")

# msa_debug_site_t
DEBUG_SITES = {0: "none", 1: "sel_range", 2: "sel_order", 3: "sel_local", 4: "seq_len",
               5: "page_id", 16: "sched_list", 17: "sched_item", 18: "attn_item",
               19: "attn_token", 20: "combine_pos", 21: "decode_page", 22: "index_row"}


class MsaConfig(ctypes.Structure):
    _fields_ = [("num_groups", ctypes.c_int32), ("heads_per_group", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("index_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float), ("index_dtype", ctypes.c_int32),
                ("wait_limit_ns", ctypes.c_int64)]


class MsaPagedKV(ctypes.Structure):
    _fields_ = [("k_idx_pool", ctypes.c_void_p), ("k_pool", ctypes.c_void_p),
                ("v_pool", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
                ("seq_lens", ctypes.c_void_p), ("batch", ctypes.c_int32),
                ("max_pages", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32)]


class MsaDebugRecord(ctypes.Structure):
    _fields_ = [("site", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("value", ctypes.c_int64), ("bound", ctypes.c_int64), ("row", ctypes.c_int64)]


class MsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lib = None


def checked_build_requested() -> bool:
    v = os.environ.get("MSA_DEBUG_CHECKS", "")
    return v not in ("", "0")


def lib() -> ctypes.CDLL:
    """The loaded libmsa.so (libmsa_debug.so when MSA_DEBUG_CHECKS is set); raises if it has not
    been built (no fallback exists)."""
    global _lib
    if _lib is None:
        path = DEBUG_LIB_PATH if checked_build_requested() else LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"{os.path.basename(path)} is not built ({path}); run "
                               "`python -m block_sparse_long_msa_gb300.build`")
        L = ctypes.CDLL(path)
        P, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
        cfgp, pagedp = ctypes.POINTER(MsaConfig), ctypes.POINTER(MsaPagedKV)
        L.msa_index_select_workspace.argtypes = [cfgp, i64, i64, pagedp]
        L.msa_index_select_workspace.restype = sz
        L.msa_index_select.argtypes = [cfgp, P, P, i64, pagedp, P, P, P, sz, P]
        L.msa_index_select_scores.argtypes = [cfgp, P, P, i64, pagedp, P, P, P, P, sz, P]
        L.msa_index_candidates.argtypes = [cfgp, P, P, i64, pagedp, ctypes.c_int32,
                                           ctypes.c_int32, P, P, P, sz, P]
        L.msa_index_merge.argtypes = [cfgp, ctypes.c_int32, P, P, i64, P, P, P, P, sz, P]
        L.msa_attn_prefill_workspace.argtypes = [cfgp, i64]
        L.msa_attn_prefill_workspace.restype = sz
        L.msa_attn_prefill.argtypes = [cfgp, P, P, P, i64, P, P, P, P, sz, P]
        L.msa_attn_prefill_marked.argtypes = [cfgp, P, P, P, i64, P, P, P, P, sz, P, P,
                                              ctypes.c_int32]
        L.msa_prefill_chunk_tokens.argtypes = [cfgp, i64]
        L.msa_prefill_chunk_tokens.restype = i64
        L.msa_attn_prefill_launches.argtypes = [cfgp, i64]
        L.msa_attn_prefill_launches.restype = ctypes.c_int32
        L.msa_attn_decode_workspace.argtypes = [cfgp, pagedp]
        L.msa_attn_decode_workspace.restype = sz
        L.msa_attn_decode.argtypes = [cfgp, P, pagedp, P, P, P, P, sz, P]
        L.msa_get_device_status.argtypes = [P, P]
        L.msa_reset_device_status.argtypes = [P, P]
        L.msa_status_string.argtypes = [ctypes.c_int]
        L.msa_status_string.restype = ctypes.c_char_p
        L.msa_debug_checks.argtypes = []
        L.msa_debug_checks.restype = ctypes.c_int32
        L.msa_get_debug_record.argtypes = [P, ctypes.POINTER(MsaDebugRecord), P]
        for name in ("msa_index_select", "msa_index_select_scores", "msa_index_candidates",
                     "msa_index_merge", "msa_attn_prefill",
                     "msa_attn_prefill_marked",
                     "msa_attn_decode",
                     "msa_get_device_status", "msa_reset_device_status",
                     "msa_get_debug_record"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().msa_status_string(status).decode()
    except RuntimeError:
        return f"status {status}"


INDEX_DTYPES = {"bf16": 0, "e4m3": 1}  # msa_index_dtype_t


def config(num_groups: int, heads_per_group: int, topk: int, softmax_scale: float | None = None,
           head_dim: int = 128, index_dim: int = 128, block_size: int = 128,
           wait_limit_ns: int = 0, index_dtype: str = "bf16") -> MsaConfig:
    """index_dtype: element type of q_idx, k_idx and the paged k_idx_pool, "bf16" or "e4m3"
    (torch.float8_e4m3fn tensors)."""
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(head_dim)
    return MsaConfig(num_groups, heads_per_group, head_dim, index_dim, block_size, topk,
                     softmax_scale, INDEX_DTYPES[index_dtype], wait_limit_ns)


def _index_dtype_ok(cfg: MsaConfig, *tensors):
    import torch
    want = torch.float8_e4m3fn if cfg.index_dtype == INDEX_DTYPES["e4m3"] else torch.bfloat16
    for t in tensors:
        if t is not None and t.dtype != want:
            raise MsaError(MSA_ERR_INVALID_ARG, f"index vectors must be {want}, got {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(st: int, where: str):
    if st != MSA_OK:
        raise MsaError(st, where)


# Workspaces of the calls made without one: one per (device, stream), grown as needed.  Calls on
# one stream run in order, so they may share it; its status word is cleared before each reuse.
_ws_cache: dict = {}


def _workspace(nbytes: int, device, ws, stream=None):
    import torch
    if ws is None:
        s = torch.cuda.current_stream(device) if stream is None else stream
        key = (str(device), s.cuda_stream)
        ws = _ws_cache.get(key)
        if ws is None or ws.numel() < nbytes:
            with torch.cuda.stream(s):  # allocated (and zeroed) in the order of the stream it serves
                ws = torch.zeros(max(nbytes, WS_HEADER_BYTES), dtype=torch.uint8, device=device)
            _ws_cache[key] = ws
        else:
            _check(lib().msa_reset_device_status(_ptr(ws), ctypes.c_void_p(s.cuda_stream)),
                   "msa_reset_device_status")
    if ws.numel() * ws.element_size() < nbytes:
        raise MsaError(MSA_ERR_WORKSPACE, "workspace")
    return ws


KV_DTYPES = {"bf16": 0, "e4m3": 1}  # msa_kv_dtype_t


def paged_kv(k_idx_pool, k_pool, v_pool, page_table, seq_lens) -> MsaPagedKV:
    """The paged cache; K/V pools of torch.bfloat16 or torch.float8_e4m3fn (both the same)."""
    import torch
    batch, max_pages = page_table.shape
    kv = 0
    if k_pool is not None:
        if v_pool is not None and v_pool.dtype != k_pool.dtype:
            raise MsaError(MSA_ERR_INVALID_ARG, "k_pool and v_pool must have the same dtype")
        if k_pool.dtype == torch.float8_e4m3fn:
            kv = KV_DTYPES["e4m3"]
        elif k_pool.dtype != torch.bfloat16:
            raise MsaError(MSA_ERR_INVALID_ARG, f"K/V pools must be bf16 or e4m3, got {k_pool.dtype}")
    return MsaPagedKV(k_idx_pool.data_ptr(), k_pool.data_ptr() if k_pool is not None else None,
                      v_pool.data_ptr() if v_pool is not None else None, page_table.data_ptr(),
                      seq_lens.data_ptr(), batch, max_pages, k_idx_pool.shape[0], kv)


def msa_index_select_workspace(cfg: MsaConfig, num_queries: int, num_keys: int,
                               paged: MsaPagedKV | None = None) -> int:
    return int(lib().msa_index_select_workspace(ctypes.byref(cfg), num_queries, num_keys,
                                                ctypes.byref(paged) if paged else None))


def msa_index_select(cfg: MsaConfig, q_idx, k_idx=None, paged: MsaPagedKV | None = None,
                     sel=None, sel_score=None, want_score: bool = False, ws=None, stream=None):
    """Index branch.  Returns sel int32 [G][T][k] (and sel_score fp32 if asked)."""
    import torch
    _index_dtype_ok(cfg, q_idx, k_idx)
    T = q_idx.shape[0]
    L = 0 if paged is not None else k_idx.shape[0]
    G, k = cfg.num_groups, cfg.topk
    if sel is None:
        sel = torch.empty((G, T, k), dtype=torch.int32, device=q_idx.device)
    if want_score and sel_score is None:
        sel_score = torch.empty((G, T, k), dtype=torch.float32, device=q_idx.device)
    ws = _workspace(msa_index_select_workspace(cfg, T, L, paged), q_idx.device, ws, stream)
    st = lib().msa_index_select(ctypes.byref(cfg), _ptr(q_idx), _ptr(k_idx), L,
                                ctypes.byref(paged) if paged is not None else None, _ptr(sel),
                                _ptr(sel_score), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "msa_index_select")
    return (sel, sel_score) if want_score else sel


def msa_index_select_scores(cfg: MsaConfig, q_idx, k_idx=None, paged: MsaPagedKV | None = None,
                            sel=None, block_scores=None, ws=None, stream=None):
    """Index branch plus every block's pooled score.  Returns (sel int32 [G][T][k],
    block_scores fp32 [G][T][nb]); nb = ceil(L/128) for prefill, max_pages for decode.
    Entries: the pooled score for blocks before the query's own, +inf for its own, -inf after."""
    import torch
    _index_dtype_ok(cfg, q_idx, k_idx)
    T = q_idx.shape[0]
    L = 0 if paged is not None else k_idx.shape[0]
    G, k = cfg.num_groups, cfg.topk
    nb = paged.max_pages if paged is not None else (L + cfg.block_size - 1) // cfg.block_size
    if sel is None:
        sel = torch.empty((G, T, k), dtype=torch.int32, device=q_idx.device)
    if block_scores is None:
        block_scores = torch.empty((G, T, nb), dtype=torch.float32, device=q_idx.device)
    elif (block_scores.dtype != torch.float32 or tuple(block_scores.shape) != (G, T, nb)
          or not block_scores.is_contiguous()):
        raise MsaError(MSA_ERR_INVALID_ARG, f"block_scores must be contiguous fp32 {(G, T, nb)}")
    ws = _workspace(msa_index_select_workspace(cfg, T, L, paged), q_idx.device, ws, stream)
    st = lib().msa_index_select_scores(ctypes.byref(cfg), _ptr(q_idx), _ptr(k_idx), L,
                                       ctypes.byref(paged) if paged is not None else None,
                                       _ptr(sel), None, _ptr(block_scores), _ptr(ws), ws.numel(),
                                       _stream(stream))
    _check(st, "msa_index_select_scores")
    return sel, block_scores


def msa_index_candidates(cfg: MsaConfig, q_idx, k_idx=None, L: int | None = None,
                         paged: MsaPagedKV | None = None, block_begin: int = 0,
                         block_end: int = 1 << 30, cand_score=None, cand_block=None, ws=None,
                         stream=None):
    """One shard of the context-parallel index branch: the top-(k-1) (score, block) candidates
    of key blocks [block_begin, block_end), in rank order, fp32 / int32 [G][T][k-1].

    Prefill: q_idx [L][G][di] holds every query, k_idx only the shard's keys (positions
    block_begin*128 .. ), L the whole length (default q_idx.shape[0]).  Decode: pass `paged`."""
    import torch
    _index_dtype_ok(cfg, q_idx, k_idx)
    T = q_idx.shape[0]
    if paged is None and L is None:
        L = T
    Lc = 0 if paged is not None else L
    G, w = cfg.num_groups, max(cfg.topk - 1, 0)
    if cand_score is None:
        cand_score = torch.empty((G, T, w), dtype=torch.float32, device=q_idx.device)
    if cand_block is None:
        cand_block = torch.empty((G, T, w), dtype=torch.int32, device=q_idx.device)
    ws = _workspace(msa_index_select_workspace(cfg, T, Lc, paged), q_idx.device, ws, stream)
    st = lib().msa_index_candidates(ctypes.byref(cfg), _ptr(q_idx), _ptr(k_idx), Lc,
                                    ctypes.byref(paged) if paged is not None else None,
                                    block_begin, block_end, _ptr(cand_score), _ptr(cand_block),
                                    _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "msa_index_candidates")
    return cand_score, cand_block


def msa_index_merge(cfg: MsaConfig, cand_score, cand_block, seq_lens=None, sel=None,
                    sel_score=None, want_score: bool = False, ws=None, stream=None):
    """Selection [G][T][k] from the stacked candidates [R][G][T][k-1] of R disjoint shards.
    seq_lens: decode context lengths [T] (None for prefill: query t at position t)."""
    import torch
    R, G, T, _ = cand_block.shape
    if sel is None:
        sel = torch.empty((G, T, cfg.topk), dtype=torch.int32, device=cand_block.device)
    if want_score and sel_score is None:
        sel_score = torch.empty((G, T, cfg.topk), dtype=torch.float32, device=cand_block.device)
    ws = _workspace(WS_HEADER_BYTES, cand_block.device, ws, stream)
    st = lib().msa_index_merge(ctypes.byref(cfg), R, _ptr(cand_score), _ptr(cand_block), T,
                               _ptr(seq_lens), _ptr(sel), _ptr(sel_score), _ptr(ws), ws.numel(),
                               _stream(stream))
    _check(st, "msa_index_merge")
    return (sel, sel_score) if want_score else sel


def msa_attn_prefill_workspace(cfg: MsaConfig, L: int) -> int:
    return int(lib().msa_attn_prefill_workspace(ctypes.byref(cfg), L))


def msa_prefill_chunk_tokens(cfg: MsaConfig, L: int) -> int:
    return int(lib().msa_prefill_chunk_tokens(ctypes.byref(cfg), L))


def msa_attn_prefill_launches(cfg: MsaConfig, L: int) -> int:
    return int(lib().msa_attn_prefill_launches(ctypes.byref(cfg), L))


def msa_attn_prefill(cfg: MsaConfig, q, k, v, sel, o=None, lse=None, ws=None, stream=None,
                     marks=None):
    """Main branch, prefill.  Returns o bf16 [L][Hq][d] and lse fp32 [Hq][L].

    marks: optional list of recorded torch.cuda.Event(enable_timing=True); see
    msa_attn_prefill_marked in include/msa.h for where each is recorded.
    """
    import torch
    L, Hq, d = q.shape
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, L), dtype=torch.float32, device=q.device)
    ws = _workspace(msa_attn_prefill_workspace(cfg, L), q.device, ws, stream)
    if marks:
        arr = (ctypes.c_void_p * len(marks))(*[m.cuda_event for m in marks])
        st = lib().msa_attn_prefill_marked(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), L,
                                           _ptr(sel), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(),
                                           _stream(stream), arr, len(marks))
    else:
        st = lib().msa_attn_prefill(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), L, _ptr(sel),
                                    _ptr(o), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "msa_attn_prefill")
    return o, lse


def msa_attn_decode_workspace(cfg: MsaConfig, paged: MsaPagedKV) -> int:
    return int(lib().msa_attn_decode_workspace(ctypes.byref(cfg), ctypes.byref(paged)))


def msa_attn_decode(cfg: MsaConfig, q, paged: MsaPagedKV, sel, o=None, lse=None, ws=None,
                    stream=None):
    """Main branch, paged decode.  Returns o bf16 [batch][Hq][d] and lse fp32 [Hq][batch]."""
    import torch
    batch, Hq, d = q.shape
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, batch), dtype=torch.float32, device=q.device)
    ws = _workspace(msa_attn_decode_workspace(cfg, paged), q.device, ws, stream)
    st = lib().msa_attn_decode(ctypes.byref(cfg), _ptr(q), ctypes.byref(paged), _ptr(sel),
                               _ptr(o), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "msa_attn_decode")
    return o, lse


def msa_get_device_status(ws, stream=None) -> int:
    return int(lib().msa_get_device_status(_ptr(ws), _stream(stream)))


def msa_reset_device_status(ws, stream=None) -> None:
    _check(lib().msa_reset_device_status(_ptr(ws), _stream(stream)), "msa_reset_device_status")


def msa_debug_checks() -> int:
    """0 for the release build; bit 0: the checked build; bit 1: input validation is on."""
    return int(lib().msa_debug_checks())


def debug_record(ws, stream=None) -> dict | None:
    """The checked build's record of the first failed check in ws ({"site", "value", "bound",
    "row"}; site "none" if no check failed); None for the release build."""
    rec = MsaDebugRecord()
    st = int(lib().msa_get_debug_record(_ptr(ws), ctypes.byref(rec), _stream(stream)))
    if st == MSA_ERR_UNSUPPORTED:
        return None
    _check(st, "msa_get_debug_record")
    return {"site": DEBUG_SITES.get(rec.site, str(rec.site)), "value": rec.value,
            "bound": rec.bound, "row": rec.row}
