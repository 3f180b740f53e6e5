"""Latency tables for SLO-constrained chunk selection (Technical Summary 2.2 C).

`measure_curves` times every layer kind of a model (shape, format,
compensator rank or none, gate form) at a set of token counts on both paths:
CUDA-graph replays of the library's own calls over several distinct layers of
that kind, so the weights stream from HBM as they do in a real step.
`choose_chunk` hands the per-layer curves to spear_chunk_select, which returns
the largest prefill chunk whose predicted mixed step meets an inter-token
latency target; a model with more compensated layers has slower curves and
gets a smaller chunk.
"""
from __future__ import annotations

from typing import Dict, List, Sequence, Tuple

import torch

from . import spear

Curve = Tuple[List[int], List[float]]


def layer_kind(L: spear.W4Layer) -> tuple:
    r = L.rank if (L.comp_enabled and L.rank > 0) else 0
    h = int(L.gate_w1.shape[0]) if (r and L.gate_w1 is not None) else 0
    return (L.K, L.N, L.group_size, bool(L.symmetric), r, h)


def _time_calls(calls, stream, reps: int) -> float:
    """Microseconds per pass of `calls` (a list of closures issuing library
    calls on `stream`), from one CUDA graph replayed `reps` times."""
    torch.cuda.synchronize()                # buffers were made on the default stream
    with torch.cuda.stream(stream):
        for c in calls:
            c()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for c in calls:
            c()
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / reps


def measure_curves(layers: Sequence[spear.W4Layer], prefill_M: Sequence[int], decode_M: Sequence[int],
                   device, per_kind: int = 8, reps: int = 10) -> Dict[tuple, Tuple[Curve, Curve]]:
    """{kind: (prefill curve, decode curve)}; each point is the mean time of one
    call over up to `per_kind` distinct layers of the kind (token buffers are
    random bf16; latency does not depend on the values)."""
    by_kind: Dict[tuple, List[spear.W4Layer]] = {}
    for L in layers:
        by_kind.setdefault(layer_kind(L), []).append(L)
    stream = torch.cuda.Stream(device)
    out = {}
    for kind, Ls in by_kind.items():
        Ls = Ls[:per_kind]
        K, N = kind[0], kind[1]
        pre_us, dec_us = [], []
        for M in prefill_M:
            x = torch.randn(M, K, device=device).to(torch.bfloat16)
            y = torch.empty(M, N, dtype=torch.bfloat16, device=device)
            ws = spear.new_workspace(max(spear.spear_prefill_workspace_bytes(L, M) for L in Ls), device, zero=False)
            calls = [lambda L=L: spear.spear_linear_prefill(L, x, y=y, workspace=ws, stream=stream) for L in Ls]
            pre_us.append(_time_calls(calls, stream, reps) / len(Ls))
        for M in decode_M:
            x = torch.randn(M, K, device=device).to(torch.bfloat16)
            y = torch.empty(M, N, dtype=torch.bfloat16, device=device)
            ws = spear.new_workspace(max(spear.spear_decode_workspace_bytes(L, M) for L in Ls), device)
            calls = [lambda L=L: spear.spear_linear_decode(L, x, y=y, workspace=ws, stream=stream) for L in Ls]
            dec_us.append(_time_calls(calls, stream, reps) / len(Ls))
        out[kind] = ((list(prefill_M), pre_us), (list(decode_M), dec_us))
    return out


def choose_chunk(layers: Sequence[spear.W4Layer], table: Dict[tuple, Tuple[Curve, Curve]], decode_tokens: int,
                 choices: Sequence[int], itl_target_us: float) -> Tuple[int, float]:
    """(chunk, predicted step microseconds) from spear_chunk_select over the
    model's layers, each with the curves of its kind."""
    pre = [table[layer_kind(L)][0] for L in layers]
    dec = [table[layer_kind(L)][1] for L in layers]
    return spear.spear_chunk_select(pre, dec, decode_tokens, list(choices), itl_target_us)


__all__ = ["layer_kind", "measure_curves", "choose_chunk"]
