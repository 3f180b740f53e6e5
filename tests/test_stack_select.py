"""Host logic of the decoder-stack helper: the module-selection rule, fed the
stack's synthetic damage scores, puts compensators on exactly the seeded
blocks at the requested rank (Technical Summary 2.1 B; no GPU needed)."""
import numpy as np

from quantized_gemm_error_gb300.stack import BLOCK_LINEARS, rank_cost_bytes, select_blocks


def test_select_blocks_marks_the_seeded_blocks_at_rank_64():
    mask, ranks = select_blocks(32, 4, 64, seed=0)
    assert mask.sum() == 4
    hot = np.random.default_rng(0).choice(32, size=4, replace=False)
    assert sorted(np.flatnonzero(mask).tolist()) == sorted(hot.tolist())
    assert set(ranks[mask == 1].tolist()) == {64} and not ranks[mask == 0].any()


def test_rank_cost_of_a_block():
    # A row (K) and a B column (N), bf16, summed over q, k, v, o, gate, up, down
    assert sum(rank_cost_bytes(K, N) for _, K, N in BLOCK_LINEARS) == 2 * (4 * 8192 + 3 * 15104)
