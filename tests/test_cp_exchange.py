"""Host side of the context-parallel index branch, on the CPU.

Two gloo ranks (127.0.0.1) each hold the candidates of their own shard of the key blocks and
exchange them with block_sparse_long_msa_gb300.cp.all_gather_candidates, the call the GPU ranks
make over NCCL.  The candidates here come from the oracle's pooled block scores (each rank ranks
its own blocks), and the gathered stack, merged by ranking the union, must give the oracle's
selection: this checks that the exchange keeps the shards apart and in rank order.  The kernels'
own candidates and merge are checked on the GPU (test_gpu_cp_indexer.py).
"""
import os
import socket

import numpy as np
import torch
import torch.multiprocessing as mp

import oracle
import synthetic
from block_sparse_long_msa_gb300 import cp

L, G, K = 1400, 2, 6


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _shard_candidates(scores, b0, b1, w):
    """The shard's top-w blocks per row, in rank order, from pooled scores [G][L][nb]."""
    Gs, T, _ = scores.shape
    ids = np.full((Gs, T, w), -1, np.int32)
    sc = np.full((Gs, T, w), -np.inf, np.float32)
    for g in range(Gs):
        for t in range(T):
            blocks = sorted(range(b0, min(b1, t // 128)), key=lambda b: (-scores[g, t, b], b))
            for r, b in enumerate(blocks[:w]):
                ids[g, t, r] = b
                sc[g, t, r] = scores[g, t, b]
    return sc, ids


def _merge(all_s, all_b, k):
    """Rank the union of the shards' candidates; local block added; ascending, -1 padded."""
    R, Gs, T, w = all_b.shape
    sel = np.full((Gs, T, k), -1, np.int32)
    for g in range(Gs):
        for t in range(T):
            c = [(float(all_s[r, g, t, j]), int(all_b[r, g, t, j]))
                 for r in range(R) for j in range(w) if all_b[r, g, t, j] >= 0]
            c.sort(key=lambda x: (-x[0], x[1]))
            bi = t // 128
            ids = sorted([b for _, b in c[:min(k - 1, bi)]] + [bi])
            sel[g, t, :len(ids)] = ids
    return sel


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = synthetic.Workload("cpx", "prefill", L=L, Hq=16 * G, G=G, k=K, seed=77)
    inp = synthetic.prefill_inputs(w, index_only=True)
    scores = oracle.block_scores_prefill(inp["q_idx"], inp["k_idx"], w.B)
    bounds = cp.split_by_work(cp.prefill_work(L), world)
    b0, b1 = bounds[rank]
    sc, ids = _shard_candidates(scores, b0, b1, K - 1)
    all_s, all_b = cp.all_gather_candidates(torch.from_numpy(sc), torch.from_numpy(ids))
    ok = all_s.shape == (world, G, L, K - 1) and all_b.dtype == torch.int32
    # every rank holds every shard, in rank order
    for r, (c0, c1) in enumerate(bounds):
        blk = all_b[r].numpy()
        real = blk[blk >= 0]
        ok = ok and bool(((real >= c0) & (real < c1)).all())
    sel = _merge(all_s.numpy(), all_b.numpy(), K)
    ref = oracle.select_prefill(inp["q_idx"], inp["k_idx"], w.B, w.k)
    out.put((rank, bool(ok), bool(np.array_equal(sel, ref))))
    dist.destroy_process_group()


def test_two_gloo_ranks_exchange_candidates_into_the_selection():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(out.get(timeout=5) for _ in range(2))
    assert got == [(0, True, True), (1, True, True)], got


def test_split_by_work_covers_every_block_once_and_balances():
    for work in (cp.prefill_work(1 << 20), cp.decode_work([300, 5000, 129, 2560, 262144], 2048),
                 [0] * 10, [5], []):
        for world in (1, 2, 3, 4, 8):
            b = cp.split_by_work(work, world)
            assert len(b) == world and b[0][0] == 0 and b[-1][1] == len(work)
            assert all(b[i][1] == b[i + 1][0] and b[i][0] <= b[i][1] for i in range(world - 1))
            if work and max(work) > 0:
                tot = sum(work)
                shares = [sum(work[x:y]) for x, y in b]
                # each range ends at the first block that would pass its quantile
                assert max(shares) <= tot / world + max(work) * world
    w = cp.decode_work([1, 128, 129, 300], 3)
    assert w == [2, 1, 0]
    assert cp.prefill_work(300) == [172, 44, 0]
