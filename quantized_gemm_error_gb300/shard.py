"""Column-parallel split of a W4 layer over ranks, one GPU each.

Every output row n of the layer (a column of y) needs only row n of the codes,
scales, zero points and factor B, plus A, w_g and the tokens, which every rank
holds in full: y[:, n] = dequant(Wq[n]) x + alpha g(x) B[n] (A x).  Rank k
keeps the rows [n0, n1) of its range and computes y[:, n0:n1] with no exchange
between ranks; a consumer that wants all of y gathers the slices.  Ranges are
whole 64-row blocks (the library's shape rule for N), as even as the block
count allows.  Shards are views of the full layer's tensors (no copies).
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Tuple

from .spear import W4Layer

ROW_BLOCK = 64


def column_ranges(N: int, world: int, block: int = ROW_BLOCK) -> List[Tuple[int, int]]:
    """[(n0, n1)] per rank: contiguous, covering [0, N), multiples of `block`,
    sizes differing by at most one block; ranks past the block count get an
    empty range (n0 == n1)."""
    if N % block or N <= 0:
        raise ValueError(f"N={N} must be a positive multiple of {block}")
    if world < 1:
        raise ValueError("world must be >= 1")
    nb = N // block
    out = []
    for k in range(world):
        b0, b1 = nb * k // world, nb * (k + 1) // world
        out.append((b0 * block, b1 * block))
    return out


def column_shard(layer: W4Layer, rank: int, world: int) -> Optional[W4Layer]:
    """The rows of `layer` that rank `rank` of `world` owns, as a layer of its
    own (None for an empty range)."""
    n0, n1 = column_ranges(layer.N, world)[rank]
    if n0 == n1:
        return None
    rows = slice(n0, n1)
    return dataclasses.replace(
        layer, N=n1 - n0, qweight=layer.qweight[rows], scales=layer.scales[rows],
        zeros=None if layer.zeros is None else layer.zeros[rows],
        B=None if layer.B is None else layer.B[rows])


__all__ = ["ROW_BLOCK", "column_ranges", "column_shard"]
