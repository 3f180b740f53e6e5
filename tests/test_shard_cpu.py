"""Column-parallel split of a layer (quantized_gemm_error_gb300/shard.py) on CPU.

The shards are views of a layer packed by the oracle; the oracle's output for
each shard, concatenated over ranks, must equal its output for the whole layer
element for element (every output row depends only on its own row of codes,
scales, zero points and B).  The two-rank test runs the same split as gloo
ranks and gathers the slices on rank 0."""
import json
import multiprocessing as mp
import os
import socket
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from quantized_gemm_error_gb300.inputs import make_layer, make_tokens  # noqa: E402
from quantized_gemm_error_gb300.shard import column_ranges, column_shard  # noqa: E402
from quantized_gemm_error_gb300.spear import W4Layer  # noqa: E402


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def _packed_layer(N, K, G, sym, r, seed):
    """(W4Layer of CPU tensors, tokens) from the seeded recipe, packed by the oracle."""
    lay, rng = make_layer(N, K, r, seed=seed)
    q, s, z = oracle.quantize_pack(lay.W, G, sym)
    L = W4Layer(N, K, G, sym, torch.from_numpy(q), torch.from_numpy(s.view(np.int16)).view(torch.float16),
                None if z is None else torch.from_numpy(z), r, _bf16(lay.A) if r else None,
                _bf16(lay.B) if r else None, _bf16(lay.w_g) if r else None, lay.b_g, lay.alpha, r > 0)
    return L, make_tokens(rng, 5, K, outlier_frac=0.01)


def _oracle_dict(L):
    u16 = lambda t: None if t is None else t.view(torch.int16).numpy().view(np.uint16)
    return dict(N=L.N, K=L.K, G=L.group_size, sym=L.symmetric, qweight=L.qweight.numpy(),
                scales=u16(L.scales), zeros=None if L.zeros is None else L.zeros.numpy(), r=L.rank,
                A=u16(L.A), B=u16(L.B), w_g=u16(L.w_g), b_g=L.b_g, alpha=L.alpha, comp_enabled=int(L.comp_enabled))


@pytest.mark.parametrize("N,world", [(64, 1), (320, 2), (320, 3), (128, 4), (4096, 8)])
def test_column_ranges_cover_the_rows_in_blocks(N, world):
    rg = column_ranges(N, world)
    assert len(rg) == world
    assert rg[0][0] == 0 and rg[-1][1] == N
    for (a0, a1), (b0, b1) in zip(rg, rg[1:]):
        assert a1 == b0
    sizes = [n1 - n0 for n0, n1 in rg]
    assert all(n % 64 == 0 and n >= 0 for n in sizes)
    assert max(sizes) - min(sizes) <= 64


def test_column_ranges_reject_bad_shapes():
    with pytest.raises(ValueError):
        column_ranges(100, 2)
    with pytest.raises(ValueError):
        column_ranges(128, 0)


@pytest.mark.parametrize("N,K,G,sym,r,world", [
    (320, 256, 128, False, 16, 2),      # group scales, zero points, rank 16
    (320, 256, 256, True, 32, 3),       # per-channel symmetric, rank 32
    (192, 512, 128, False, 0, 2),       # plain W4
    (128, 256, 128, False, 16, 4),      # more ranks than 64-row blocks: two empty shards
])
def test_shards_concatenate_to_the_whole_layer(N, K, G, sym, r, world):
    L, x = _packed_layer(N, K, G, sym, r, seed=60 + N + r)
    full = oracle.linear(_oracle_dict(L), x)
    parts = []
    for k in range(world):
        S = column_shard(L, k, world)
        n0, n1 = column_ranges(N, world)[k]
        if S is None:
            assert n0 == n1
            continue
        assert S.N == n1 - n0 and S.qweight.data_ptr() == L.qweight[n0].data_ptr()   # a view
        parts.append(oracle.linear(_oracle_dict(S), x))
    assert np.array_equal(np.concatenate(parts, axis=1), full)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_path: str):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "MASTER_ADDR": "127.0.0.1",
                       "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    L, x = _packed_layer(320, 256, 128, False, 16, seed=77)       # the same seeded layer on every rank
    S = column_shard(L, rank, world)
    y = oracle.linear(_oracle_dict(S), x)
    got = [None] * world
    dist.all_gather_object(got, y)
    ok = None
    if rank == 0:
        ok = bool(np.array_equal(np.concatenate(got, axis=1), oracle.linear(_oracle_dict(L), x)))
    dist.barrier()
    dist.destroy_process_group()
    with open(f"{out_path}.{rank}", "w") as f:
        json.dump({"rank": rank, "cols": int(y.shape[1]), "ok": ok}, f)


@pytest.mark.timeout(120)
def test_two_gloo_ranks_gather_the_column_shards(tmp_path):
    ctx = mp.get_context("spawn")
    port = _free_port()
    out = str(tmp_path / "rank")
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0, f"rank exited with {p.exitcode}"
    res = [json.load(open(f"{out}.{r}")) for r in range(2)]
    assert res[0] == {"rank": 0, "cols": 128, "ok": True}
    assert res[1] == {"rank": 1, "cols": 192, "ok": None}
