"""Host logic of the decoder-stack helper: the module-selection rule, fed the
stack's synthetic damage scores, puts compensators on exactly the seeded
blocks at the requested rank (Technical Summary 2.1 B; no GPU needed)."""
import numpy as np

from quantized_gemm_error_gb300.stack import BLOCK_LINEARS, memory_bytes, rank_cost_bytes, select_blocks


def test_select_blocks_marks_the_seeded_blocks_at_rank_64():
    mask, ranks = select_blocks(32, 4, 64, seed=0)
    assert mask.sum() == 4
    hot = np.random.default_rng(0).choice(32, size=4, replace=False)
    assert sorted(np.flatnonzero(mask).tolist()) == sorted(hot.tolist())
    assert set(ranks[mask == 1].tolist()) == {64} and not ranks[mask == 0].any()


def test_rank_cost_of_a_block():
    # A row (K) and a B column (N), bf16, summed over q, k, v, o, gate, up, down
    assert sum(rank_cost_bytes(K, N) for _, K, N in BLOCK_LINEARS) == 2 * (4 * 8192 + 3 * 15104)


def test_memory_of_the_stack():
    # 32 blocks of int4 codes + fp16 per-channel scales; rank-64 A, B, w_g on 4 blocks
    _, ranks = select_blocks(32, 4, 64, seed=0)
    m = memory_bytes(ranks)
    per_block_w = (4 * 4096 * 4096 + 3 * 4096 * 11008) // 2 + 2 * (5 * 4096 + 2 * 11008)
    per_block_c = 2 * (64 * (4 * 8192 + 3 * 15104) + 6 * 4096 + 11008)
    assert m["weight_bytes"] == 32 * per_block_w == 3_240_722_432
    assert m["compensator_bytes"] == 4 * per_block_c == 40_261_632
    assert abs(m["overhead"] - 0.012424) < 1e-6
