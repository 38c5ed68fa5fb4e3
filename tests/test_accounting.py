"""FLOP accounting pinned to the one number the pages derive analytically: the 28.4x per-token
attention-FLOP reduction of MSA over GQA at 1M context ("MiniMax M3 算力省 20 倍", section 四;
also the DEVUP article on MiniMax-M3), for 64 query / 4 KV heads (section 三), head and index
dim 128, B = 128, k = 16 (section 二)."""
from block_sparse_long_msa_gb300 import accounting as acc


def test_per_token_reduction_at_1m_is_28_4():
    L = 1 << 20
    pos = L // 2 - 1
    dense = acc.dense_gqa_flops_per_token(pos, 64, 128)
    msa = acc.msa_flops_per_token(pos, 64, 4, 128, 128, 128, 16)
    assert round(dense / msa, 1) == 28.4


def test_prefill_counts_small_cases_by_enumeration():
    for L, B, k, G, di in [(1, 4, 2, 1, 8), (10, 4, 2, 2, 8), (37, 8, 3, 3, 4), (64, 16, 16, 1, 2)]:
        idx = sum(2 * di * G * (i // B) * B for i in range(L))
        assert acc.index_flops_prefill(L, G, di, B) == idx
        tok = sum(min(k - 1, i // B) * B + (i % B + 1) for i in range(L))
        assert acc.attended_tokens_prefill(L, B, k) == tok
        units = G * sum(min(k - 1, i // B) + 1 for i in range(L))
        assert acc.units_prefill(L, G, B, k) == units
