"""Seeded synthetic inputs for the MSA operator (shared by the oracle tests and the CUDA path).

This module draws numbers and lays them out; it holds none of the operator's arithmetic
(no scores, no pooling, no selection, no softmax).  Every draw comes from one counter-based
generator, SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014; the finaliser constants as published by Vigna), evaluated on a counter made of
(seed, stream id, element index).  The arithmetic is done on torch int64 tensors, whose
multiplication wraps modulo 2**64 on CPU and GPU alike, so the same call gives the same bits on
either device.

Distributions (the workloads of "MiniMax M3 算力省 20 倍", section 二 and 四, and the configs
built on them):
  * index queries/keys: integers uniform in [-8, 8] divided by 8, stored as bf16 (exact);
  * Q, K, V: N(0, 1) by Box-Muller in float64, rounded to bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

_M64 = (1 << 64) - 1


def _s64(c: int) -> int:
    c &= _M64
    return c - (1 << 64) if c >= (1 << 63) else c


_GAMMA = _s64(0x9E3779B97F4A7C15)
_MIX1 = _s64(0xBF58476D1CE4E5B9)
_MIX2 = _s64(0x94D049BB133111EB)


def _lsr(x: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of an int64 tensor viewed as uint64."""
    return (x >> s) & ((1 << (64 - s)) - 1)


def splitmix64(x: torch.Tensor) -> torch.Tensor:
    """SplitMix64 output function applied to the state x + gamma (int64 tensor, wrapping)."""
    z = x + _GAMMA
    z = (z ^ _lsr(z, 30)) * _MIX1
    z = (z ^ _lsr(z, 27)) * _MIX2
    return z ^ _lsr(z, 31)


def splitmix64_int(x: int) -> int:
    """Python-int version of :func:`splitmix64` (used for keys and by the self-test)."""
    z = (x + 0x9E3779B97F4A7C15) & _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: int) -> int:
    return splitmix64_int(splitmix64_int(seed) ^ (stream * 0xD1B54A32D192ED03 & _M64))


_CHUNK = 1 << 25


def hashes(seed: int, stream: int, start: int, n: int, device="cpu") -> torch.Tensor:
    """64-bit hashes of elements start..start+n-1 of one stream (int64 tensor)."""
    key = _s64(stream_key(seed, stream))
    idx = torch.arange(start, start + n, dtype=torch.int64, device=device)
    return splitmix64(idx * _GAMMA + key)


def hashes_at(seed: int, stream: int, idx: torch.Tensor) -> torch.Tensor:
    """64-bit hashes of the listed element indices of one stream (int64 tensor, any shape)."""
    key = _s64(stream_key(seed, stream))
    return splitmix64(idx.to(torch.int64) * _GAMMA + key)


def _fill(out_flat: torch.Tensor, seed: int, stream: int, fn) -> None:
    n = out_flat.numel()
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        out_flat[s:e] = fn(hashes(seed, stream, s, e - s, out_flat.device))


def _u32_hi(h):
    return _lsr(h, 32)


def _u32_lo(h):
    return h & 0xFFFFFFFF


def _int_pm8(h: torch.Tensor) -> torch.Tensor:
    """Integer uniform in [-8, 8] from the high 32 bits (multiply-shift range reduction)."""
    return ((_u32_hi(h) * 17) >> 32) - 8


def int8th(seed: int, stream: int, shape, device="cpu") -> torch.Tensor:
    """bf16 tensor of integers uniform in [-8, 8] divided by 8."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    _fill(out.view(-1), seed, stream, lambda h: _int_pm8(h).to(torch.float32) / 8.0)
    return out


def int_pm8(seed: int, stream: int, shape, device="cpu") -> torch.Tensor:
    """int64 tensor of integers uniform in [-8, 8] (before the division by 8)."""
    out = torch.empty(shape, dtype=torch.int64, device=device)
    _fill(out.view(-1), seed, stream, _int_pm8)
    return out


def _box_muller(h: torch.Tensor) -> torch.Tensor:
    u1 = (_u32_hi(h).to(torch.float64) + 1.0) * (1.0 / 4294967296.0)  # (0, 1]
    u2 = _u32_lo(h).to(torch.float64) * (1.0 / 4294967296.0)          # [0, 1)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def normal_bf16(seed: int, stream: int, shape, device="cpu") -> torch.Tensor:
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    _fill(out.view(-1), seed, stream, _box_muller)
    return out


def uniform01(seed: int, stream: int, n: int, device="cpu") -> torch.Tensor:
    """float64 uniforms in [0, 1)."""
    return _u32_hi(hashes(seed, stream, 0, n, device)).to(torch.float64) * (1.0 / 4294967296.0)


def uniform_int(seed: int, stream: int, n: int, lo: int, hi: int, device="cpu") -> torch.Tensor:
    """int64 uniforms in [lo, hi] inclusive (multiply-shift on the high 32 bits)."""
    span = hi - lo + 1
    assert 0 < span < (1 << 31)
    return ((_u32_hi(hashes(seed, stream, 0, n, device)) * span) >> 32) + lo


def permutation(seed: int, stream: int, n: int, device="cpu") -> torch.Tensor:
    """A random permutation of 0..n-1 (stable argsort of n hashes)."""
    h = hashes(seed, stream, 0, n, device)
    return torch.sort(h, stable=True).indices


def sign_vector(seed: int, stream: int, n: int, device="cpu") -> torch.Tensor:
    """int64 vector of +-1."""
    return (_lsr(hashes(seed, stream, 0, n, device), 63) * 2 - 1)


# --------------------------------------------------------------------------------------------
# Workload configurations.  Shapes follow the 109B research model described on "MiniMax M3 算力省
# 20 倍" (64 query heads, 4 KV heads, section 三), the deployment budget B = 128, k = 16 (section
# 二) and the contexts measured there (up to 1M, section 四).
# --------------------------------------------------------------------------------------------

STREAM_Q, STREAM_K, STREAM_V, STREAM_QI, STREAM_KI = 1, 2, 3, 4, 5
STREAM_PLANT_SIGN, STREAM_PLANT_BLOCKS, STREAM_HOT_COIN = 6, 7, 8
STREAM_SEQLEN, STREAM_PAGES = 9, 10


@dataclass
class Workload:
    name: str
    kind: str              # "prefill" or "decode"
    L: int = 0             # prefill tokens
    Hq: int = 64
    G: int = 4
    d: int = 128
    di: int = 128
    B: int = 128
    k: int = 16
    planted: str = "none"  # "none", "clustered", "hot"
    batch: int = 0         # decode sequences
    n_lo: int = 0
    n_hi: int = 0
    seed: int = 1000
    extra: dict = field(default_factory=dict)

    @property
    def hpg(self) -> int:
        return self.Hq // self.G

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


WORKLOADS = {
    "tiny_L2048": Workload("tiny_L2048", "prefill", L=2048, Hq=16, G=1, k=4, seed=1000),
    "prefill_L32K": Workload("prefill_L32K", "prefill", L=32768, seed=1001),
    "prefill_L128K_clustered": Workload("prefill_L128K_clustered", "prefill", L=131072,
                                        planted="clustered", seed=1002),
    "decode_b64_16K_256K": Workload("decode_b64_16K_256K", "decode", batch=64, n_lo=16384,
                                    n_hi=262144, seed=1003),
    "prefill_L1M_hot": Workload("prefill_L1M_hot", "prefill", L=1 << 20, planted="hot",
                                seed=1004),
}


def _planted_index(w: Workload, q_int: torch.Tensor, k_int: torch.Tensor, device) -> None:
    """Bias index queries/keys along a planted sign direction (in place, integer domain)."""
    nb = (w.L + w.B - 1) // w.B
    if w.planted == "clustered":
        # per group a sign vector; 32 distinct random key blocks per group, disjoint across groups
        perm = permutation(w.seed, STREAM_PLANT_BLOCKS, nb, device)
        for g in range(w.G):
            s = sign_vector(w.seed, STREAM_PLANT_SIGN * 64 + g, w.di, device)
            q_int[:, g, :] = torch.clamp(q_int[:, g, :] + 4 * s, -8, 8)
            for b in perm[32 * g:32 * (g + 1)].tolist():
                lo, hi = b * w.B, min(w.L, (b + 1) * w.B)
                k_int[lo:hi, :] = torch.clamp(k_int[lo:hi, :] + 4 * s, -8, 8)
    elif w.planted == "hot":
        # one shared direction; key blocks 0..3 carry it, each (i, g) query carries it w.p. 0.9
        s = sign_vector(w.seed, STREAM_PLANT_SIGN * 64, w.di, device)
        hi = min(w.L, 4 * w.B)
        k_int[:hi, :] = torch.clamp(k_int[:hi, :] + 4 * s, -8, 8)
        coin = uniform01(w.seed, STREAM_HOT_COIN, w.L * w.G, device).view(w.L, w.G) < 0.9
        for g in range(w.G):
            rows = coin[:, g]
            q_int[rows, g, :] = torch.clamp(q_int[rows, g, :] + 4 * s, -8, 8)


def as_index_dtype(t: torch.Tensor, index_dtype: str) -> torch.Tensor:
    """Index vectors in the requested storage type: "bf16", or "e4m3" (torch.float8_e4m3fn).
    The integer/8 values in [-1, 1] are exact in both, so this is a change of encoding only."""
    return t if index_dtype == "bf16" else t.to(torch.float8_e4m3fn)


def prefill_inputs(w: Workload, device="cpu", L: int | None = None,
                   index_only: bool = False, index_dtype: str = "bf16",
                   without_q: bool = False) -> dict:
    """q [L][Hq][d], k/v [L][G][d] bf16; q_idx [L][G][di], k_idx [L][di] in index_dtype.
    without_q leaves q out (prefill_q_rows gives any of its rows)."""
    assert w.kind == "prefill"
    if L is not None:
        w = Workload(**{**w.__dict__, "L": L})
    L = w.L
    out = {}
    if not index_only:
        if not without_q:
            out["q"] = normal_bf16(w.seed, STREAM_Q, (L, w.Hq, w.d), device)
        out["k"] = normal_bf16(w.seed, STREAM_K, (L, w.G, w.d), device)
        out["v"] = normal_bf16(w.seed, STREAM_V, (L, w.G, w.d), device)
    if w.planted == "none":
        out["q_idx"] = int8th(w.seed, STREAM_QI, (L, w.G, w.di), device)
        out["k_idx"] = int8th(w.seed, STREAM_KI, (L, w.di), device)
    else:
        q_int = int_pm8(w.seed, STREAM_QI, (L, w.G, w.di), device)
        k_int = int_pm8(w.seed, STREAM_KI, (L, w.di), device)
        _planted_index(w, q_int, k_int, device)
        out["q_idx"] = (q_int.to(torch.float32) / 8.0).to(torch.bfloat16)
        out["k_idx"] = (k_int.to(torch.float32) / 8.0).to(torch.bfloat16)
    out["q_idx"] = as_index_dtype(out["q_idx"], index_dtype)
    out["k_idx"] = as_index_dtype(out["k_idx"], index_dtype)
    out["workload"] = w
    return out


def prefill_q_rows(w: Workload, rows, device="cpu") -> torch.Tensor:
    """Rows `rows` of the workload's q, [len(rows)][Hq][d] bf16, equal to
    prefill_inputs(w)["q"][rows] without generating the rest (the generator is counter-based)."""
    rows = torch.as_tensor(rows, dtype=torch.int64, device=device)
    row = w.Hq * w.d
    idx = rows[:, None] * row + torch.arange(row, dtype=torch.int64, device=device)[None, :]
    return _box_muller(hashes_at(w.seed, STREAM_Q, idx)).to(torch.bfloat16).view(
        len(rows), w.Hq, w.d)


def decode_inputs(w: Workload, device="cpu", batch: int | None = None,
                  n_lo: int | None = None, n_hi: int | None = None, spare_pages: int = 3,
                  index_dtype: str = "bf16") -> dict:
    """Paged decode inputs.

    seq_lens int32 [batch] (context length n, the new token's K/V/index key already written at
    position n-1); page_table int32 [batch][max_pages], a random permutation of a shared pool;
    pools: k_idx_pool [P][B][di], k_pool / v_pool [P][G][B][d] (head-major inside a page);
    q [batch][Hq][d], q_idx [batch][G][di] (index vectors in index_dtype).
    """
    assert w.kind == "decode"
    batch = w.batch if batch is None else batch
    n_lo = w.n_lo if n_lo is None else n_lo
    n_hi = w.n_hi if n_hi is None else n_hi
    seq_lens = uniform_int(w.seed, STREAM_SEQLEN, batch, n_lo, n_hi, device)
    pages_per = (seq_lens + w.B - 1) // w.B
    max_pages = int(pages_per.max().item())
    used = int(pages_per.sum().item())
    P = used + spare_pages
    perm = permutation(w.seed, STREAM_PAGES, P, device).to(torch.int32)
    page_table = torch.full((batch, max_pages), -1, dtype=torch.int32, device=device)
    off = 0
    for s, npg in enumerate(pages_per.tolist()):
        page_table[s, :npg] = perm[off:off + npg]
        off += npg
    return {
        "seq_lens": seq_lens.to(torch.int32),
        "page_table": page_table,
        "num_pages": P,
        "max_pages": max_pages,
        "q": normal_bf16(w.seed, STREAM_Q, (batch, w.Hq, w.d), device),
        "q_idx": as_index_dtype(int8th(w.seed, STREAM_QI, (batch, w.G, w.di), device),
                                index_dtype),
        "k_idx_pool": as_index_dtype(int8th(w.seed, STREAM_KI, (P, w.B, w.di), device),
                                     index_dtype),
        "k_pool": normal_bf16(w.seed, STREAM_K, (P, w.G, w.B, w.d), device),
        "v_pool": normal_bf16(w.seed, STREAM_V, (P, w.G, w.B, w.d), device),
        "workload": Workload(**{**w.__dict__, "batch": batch, "n_lo": n_lo, "n_hi": n_hi}),
    }
