"""Context-parallel index branch over several ranks (one GPU each).

The pages describe the indexer's decode running context-parallel over 4 GB300 at 512K context
("MiniMax M3.1 Flash 开放权重与部署要点", section 权重能下载之后，为什么还要先看 vLLM).  Here the key
blocks are split into one contiguous shard per rank; each rank holds the index keys of its shard,
scores them against every query and keeps its top-(k-1) (msa_index_candidates); one all-gather
brings every rank the (score, block) candidates of all shards, (k-1) x 8 bytes per (query, group),
and msa_index_merge ranks them into the selection, identical to the single-GPU one.

This module is plumbing around two library calls: shard bounds (host arithmetic), the
all-gather (torch.distributed, NCCL between GPUs or gloo on the CPU) and the call sequence.
"""
from __future__ import annotations

B = 128


def split_by_work(work, world: int) -> list[tuple[int, int]]:
    """Contiguous block ranges [b0, b1), one per rank, with about equal total work.

    work[b] is the work of block b (for instance the number of queries that rank it).  Ranges
    cover [0, len(work)) without overlap; a rank may get an empty range."""
    nb = len(work)
    total = float(sum(work))
    bounds, b0, acc = [], 0, 0.0
    for r in range(world):
        if r == world - 1:
            b1 = nb
        else:
            goal = total * (r + 1) / world
            b1 = b0
            while b1 < nb and acc + work[b1] <= goal:
                acc += work[b1]
                b1 += 1
        bounds.append((b0, b1))
        b0 = b1
    return bounds


def prefill_work(L: int) -> list[int]:
    """Queries that rank each key block in a prefill of L tokens (those of later blocks)."""
    nb = (L + B - 1) // B
    return [max(0, L - (b + 1) * B) for b in range(nb)]


def decode_work(seq_lens, max_pages: int) -> list[int]:
    """Sequences that rank each logical block in one decode step (host list of lengths)."""
    work = [0] * max_pages
    for n in seq_lens:
        before = min((int(n) - 1) // B, max_pages) if n > 0 else 0
        for b in range(before):
            work[b] += 1
    return work


def all_gather_candidates(cand_score, cand_block, group=None):
    """Stack every rank's candidates, [G][T][k-1] each, into [world][G][T][k-1] (rank order =
    shard order)."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    scores = [torch.empty_like(cand_score) for _ in range(world)]
    blocks = [torch.empty_like(cand_block) for _ in range(world)]
    dist.all_gather(scores, cand_score.contiguous(), group=group)
    dist.all_gather(blocks, cand_block.contiguous(), group=group)
    return torch.stack(scores), torch.stack(blocks)


def index_select_context_parallel(cfg, q_idx, bounds, k_idx_shard=None, L=None, paged=None,
                                  seq_lens=None, group=None, ws=None, stream=None):
    """The selection [G][T][k] through this rank's shard bounds[rank] and one all-gather.

    Prefill: k_idx_shard holds the index keys of this rank's shard (positions
    bounds[rank][0]*128 ..), L the whole length.  Decode: paged (its page table is read only for
    the shard's blocks) and seq_lens, the device tensor of context lengths."""
    import torch.distributed as dist

    import block_sparse_long_msa_gb300 as msa
    rank = dist.get_rank(group)
    b0, b1 = bounds[rank]
    cs, cb = msa.msa_index_candidates(cfg, q_idx, k_idx_shard, L=L, paged=paged, block_begin=b0,
                                      block_end=b1, ws=ws, stream=stream)
    all_s, all_b = all_gather_candidates(cs, cb, group)
    return msa.msa_index_merge(cfg, all_s, all_b, seq_lens=seq_lens, ws=ws, stream=stream)
