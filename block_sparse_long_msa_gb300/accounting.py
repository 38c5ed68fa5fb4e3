"""Algorithmic work of the MSA operator: FLOPs and compulsory bytes per call.

Counts follow the definition ("MiniMax M3 算力省 20 倍", section 二): the index branch scores every
key of every block strictly before the query's own block (the local block is forced, so it is
never scored), the main branch attends to the tokens of the selected blocks, causal inside the
local block.  A multiply-add counts as 2 FLOPs; padded tile work is never counted.
"""
from __future__ import annotations


def _sum_floor_div(L: int, B: int) -> int:
    """sum over i in [0, L) of floor(i / B)."""
    full = L // B
    rem = L - full * B
    return B * full * (full - 1) // 2 + rem * full


def index_flops_prefill(L: int, G: int, di: int, B: int) -> int:
    """Raw index scores q_idx . k_idx for every (query, group, earlier-block key)."""
    return 2 * di * G * B * _sum_floor_div(L, B)


def attended_tokens_prefill(L: int, B: int, k: int) -> int:
    """sum over queries of |T(i)|: (k-1 earlier blocks when they exist) * B + causal local part."""
    total = 0
    nb = (L + B - 1) // B
    for b in range(nb):
        lo, hi = b * B, min(L, (b + 1) * B)
        n = hi - lo
        total += n * min(k - 1, b) * B + n * (n + 1) // 2
    return total


def attn_flops_prefill(L: int, Hq: int, d: int, B: int, k: int) -> int:
    """QK^T and PV for every (query, head, attended token): 4d FLOPs each."""
    return 4 * d * Hq * attended_tokens_prefill(L, B, k)


def units_prefill(L: int, G: int, B: int, k: int) -> int:
    """(token, group, selected block) units of the KV-outer main branch."""
    nb = (L + B - 1) // B
    return G * sum((min(L, (b + 1) * B) - b * B) * (min(k - 1, b) + 1) for b in range(nb))


def decode_index_bytes(seq_lens, B: int, di: int, G: int) -> int:
    """Index keys of every block strictly before each query's block, plus the index queries."""
    return sum(((n - 1) // B) * B * di * 2 for n in seq_lens) + len(seq_lens) * G * di * 2


def decode_attn_bytes(seq_lens, B: int, d: int, G: int, Hq: int, k: int,
                      kv_bytes: int = 2) -> int:
    """K and V of the selected blocks (whole pages, the local one up to n; kv_bytes per element),
    plus q and o (bf16)."""
    total = 0
    for n in seq_lens:
        bi = (n - 1) // B
        blocks = min(k - 1, bi)
        toks = blocks * B + (n - bi * B)
        total += toks * G * d * kv_bytes * 2
    return total + len(seq_lens) * Hq * d * 2 * 2


def dense_gqa_flops_per_token(pos: int, Hq: int, d: int) -> int:
    return Hq * (pos + 1) * 4 * d


def msa_flops_per_token(pos: int, Hq: int, G: int, d: int, di: int, B: int, k: int) -> int:
    """Main branch at the full k*B budget plus the index scores over the causal window."""
    return Hq * min(k * B, pos + 1) * 4 * d + G * pos * 2 * di
