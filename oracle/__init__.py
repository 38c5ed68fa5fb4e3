"""MSA oracle (TEST INFRASTRUCTURE ONLY).

Python face of ``msa_oracle.c``: a plain CPU, fp64-accumulation restatement of MiniMax Sparse
Attention ("MiniMax M3 算力省 20 倍", section 二 Index Branch / Main Branch, section 三 item 4 local
block, section 三 item 1 for the block scores exported to the indexer's KL alignment).  Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` use
it.  It shares no code with the CUDA path and never imports it.

Inputs are bf16 torch tensors on the CPU (or uint16 numpy arrays of bf16 bits; index vectors may
also be E4M3 tensors, decoded here from the format's definition); outputs are numpy.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp64, OpenMP, no fast-math) and return the library path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.oracle_select_prefill.argtypes = [P, P, i64, i32, i32, i32, i32, P, i64, P, P]
        lib.oracle_attn_prefill.argtypes = [P, P, P, i64, i32, i32, i32, i32, i32, f64, P, P, i64,
                                            P, P, i32]
        lib.oracle_select_decode.argtypes = [P, P, P, i64, P, i64, i32, i32, i32, i32, P, P]
        lib.oracle_attn_decode.argtypes = [P, P, P, P, i64, P, i64, i32, i32, i32, i32, i32, f64,
                                           P, P, P]
        lib.oracle_block_scores_prefill.argtypes = [P, P, i64, i32, i32, i32, P, i64, P]
        lib.oracle_block_scores_decode.argtypes = [P, P, P, i64, P, i64, i32, i32, i32, P]
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def e4m3_values() -> np.ndarray:
    """Value of every 8-bit E4M3 code (the OCP 8-bit float: sign, 4 exponent bits with bias 7,
    3 mantissa bits; exponent field 0 is subnormal, m * 2^-9; code S.1111.111 is NaN; no
    infinities), float64 [256], decoded from that definition."""
    v = np.empty(256, np.float64)
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            v[c] = np.nan
            continue
        mag = m * 2.0 ** -9 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
        v[c] = -mag if s else mag
    return v


def _e4m3_to_bf16_bits(codes: np.ndarray) -> np.ndarray:
    """Every E4M3 value has at most 4 significant bits and an exponent within bf16's range, so
    it is exactly a bf16 value: the top half of its fp32 pattern."""
    f32 = e4m3_values()[codes].astype(np.float32)
    u = f32.view(np.uint32)
    finite = np.isfinite(f32)
    assert not (u[finite] & 0xFFFF).any()
    out = (u >> 16).astype(np.uint16)
    out[~finite] = 0x7FC0
    return out


def _bits(x) -> np.ndarray:
    """bf16 (or E4M3, widened exactly to bf16) tensor/array -> contiguous uint16 numpy array of
    bf16 bits."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    if x.dtype == torch.float8_e4m3fn:
        codes = x.detach().cpu().contiguous().view(torch.uint8).numpy()
        return np.ascontiguousarray(_e4m3_to_bf16_bits(codes))
    assert x.dtype == torch.bfloat16, x.dtype
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy()
                                .view(np.uint16))


def _i32(x) -> np.ndarray:
    if not isinstance(x, np.ndarray):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x.astype(np.int32, copy=False))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def select_prefill(q_idx, k_idx, B: int, k: int, rows=None, want_score: bool = False):
    """Index branch for prefill.  q_idx [L][G][di], k_idx [L][di].

    Returns sel int32 [G][nrows][k] (ascending ids, -1 padded) and, if asked, the pooled scores
    float64 [G][nrows][k] (local block +inf, padding -inf).
    """
    qi, ki = _bits(q_idx), _bits(k_idx)
    L, G, di = qi.shape
    assert ki.shape == (L, di)
    rows = np.arange(L, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    sel = np.empty((G, len(rows), k), np.int32)
    score = np.empty((G, len(rows), k), np.float64) if want_score else None
    _load().oracle_select_prefill(_ptr(qi), _ptr(ki), L, G, di, B, k, _ptr(rows), len(rows),
                                  _ptr(sel), _ptr(score) if want_score else None)
    return (sel, score) if want_score else sel


def block_scores_prefill(q_idx, k_idx, B: int, rows=None):
    """Every block's pooled index score, float64 [G][nrows][ceil(L/B)]: the block max of the raw
    dot products for blocks before the query's own, +inf for its own, -inf after it."""
    qi, ki = _bits(q_idx), _bits(k_idx)
    L, G, di = qi.shape
    assert ki.shape == (L, di)
    rows = np.arange(L, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    out = np.empty((G, len(rows), (L + B - 1) // B), np.float64)
    _load().oracle_block_scores_prefill(_ptr(qi), _ptr(ki), L, G, di, B, _ptr(rows), len(rows),
                                        _ptr(out))
    return out


def block_scores_decode(q_idx, k_idx_pool, page_table, seq_lens, B: int):
    """Paged decode: float64 [G][batch][max_pages], same entries as block_scores_prefill."""
    qi, kp = _bits(q_idx), _bits(k_idx_pool)
    pt, sl = _i32(page_table), _i32(seq_lens)
    batch, G, di = qi.shape
    out = np.empty((G, batch, pt.shape[1]), np.float64)
    _load().oracle_block_scores_decode(_ptr(qi), _ptr(kp), _ptr(pt), pt.shape[1], _ptr(sl), batch,
                                       G, di, B, _ptr(out))
    return out


def attn_prefill(q, kk, vv, sel, B: int, k: int, scale: float, rows=None, q_compact=False):
    """Main branch for prefill.  q [L][Hq][d] (or [nrows][Hq][d] holding just `rows` when
    q_compact), kk/vv [L][G][d], sel [G][nrows][k] for `rows`.

    Returns o float64 [nrows][Hq][d] and lse float64 [Hq][nrows] (natural log).
    """
    qb, kb, vb = _bits(q), _bits(kk), _bits(vv)
    L, G, d = kb.shape
    Hq = qb.shape[1]
    rows = np.arange(L, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    if q_compact:
        assert qb.shape[0] == len(rows)
    else:
        assert qb.shape[0] == L
    s = _i32(sel)
    assert s.shape == (G, len(rows), k), (s.shape, G, len(rows), k)
    o = np.empty((len(rows), Hq, d), np.float64)
    lse = np.empty((Hq, len(rows)), np.float64)
    _load().oracle_attn_prefill(_ptr(qb), _ptr(kb), _ptr(vb), L, Hq, G, d, B, k, float(scale),
                                _ptr(s), _ptr(rows), len(rows), _ptr(o), _ptr(lse),
                                1 if q_compact else 0)
    return o, lse


def select_decode(q_idx, k_idx_pool, page_table, seq_lens, B: int, k: int,
                  want_score: bool = False):
    """Index branch for paged decode.  q_idx [batch][G][di], k_idx_pool [P][B][di]."""
    qi, kp = _bits(q_idx), _bits(k_idx_pool)
    pt, sl = _i32(page_table), _i32(seq_lens)
    batch, G, di = qi.shape
    sel = np.empty((G, batch, k), np.int32)
    score = np.empty((G, batch, k), np.float64) if want_score else None
    _load().oracle_select_decode(_ptr(qi), _ptr(kp), _ptr(pt), pt.shape[1], _ptr(sl), batch, G,
                                 di, B, k, _ptr(sel), _ptr(score) if want_score else None)
    return (sel, score) if want_score else sel


def attn_decode(q, k_pool, v_pool, page_table, seq_lens, sel, B: int, k: int, scale: float):
    """Main branch for paged decode.  q [batch][Hq][d], pools [P][G][B][d], sel [G][batch][k].

    Returns o float64 [batch][Hq][d], lse float64 [Hq][batch].
    """
    qb, kp, vp = _bits(q), _bits(k_pool), _bits(v_pool)
    pt, sl, s = _i32(page_table), _i32(seq_lens), _i32(sel)
    batch, Hq, d = qb.shape
    G = kp.shape[1]
    o = np.empty((batch, Hq, d), np.float64)
    lse = np.empty((Hq, batch), np.float64)
    _load().oracle_attn_decode(_ptr(qb), _ptr(kp), _ptr(vp), _ptr(pt), pt.shape[1], _ptr(sl),
                               batch, Hq, G, d, B, k, float(scale), _ptr(s), _ptr(o), _ptr(lse))
    return o, lse
