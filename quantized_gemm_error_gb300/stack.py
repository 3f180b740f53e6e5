"""A Llama-7B-shaped decoder-block stack of W4 layers, some with compensators,
stepped as CUDA graphs.

Each block has seven linears: q, k, v, o (4096 x 4096), gate, up
(4096 -> 11008) and down (11008 -> 4096), int4 per-output-channel symmetric.
The module-selection rule (spear_layer_select_mask, Technical Summary 2.1 B)
picks which blocks carry a compensator and its rank; the other blocks are
plain W4 layers (rank 0).  One mixed step of chunked prefill is the seven
linears of every block on the step's tokens, a prefill chunk and the decode
tokens concatenated (prefill path); the decode tokens alone go through the
decode path.  Each path is captured once as a CUDA graph and replayed.

Block inputs are fixed buffers: the step measures the linears, the part the
pages accelerate; attention and the nonlinearities between them are not part
of the layer and are left out (random-init weights make their values
meaningless anyway).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List

import numpy as np
import torch

from . import spear
from .inputs import f32_to_bf16_bits, make_layer

# (name, K, N) of one block's linears
BLOCK_LINEARS = [("q", 4096, 4096), ("k", 4096, 4096), ("v", 4096, 4096), ("o", 4096, 4096),
                 ("gate", 4096, 11008), ("up", 4096, 11008), ("down", 11008, 4096)]


def rank_cost_bytes(K: int, N: int) -> int:
    """Bytes one unit of compensator rank costs a K -> N linear: a row of A
    (K bf16) and a column of B (N bf16)."""
    return 2 * (K + N)


def memory_bytes(ranks) -> dict:
    """Device bytes of the stack's packed weights (int4 codes and per-channel
    fp16 scales; symmetric, so no zero points) and of its compensators (A, B
    and w_g in bf16), from the shapes; ranks[b] is block b's rank (0: none)."""
    w = c = 0
    for r in ranks:
        r = int(r)
        for _, K, N in BLOCK_LINEARS:
            w += N * K // 2 + N * 2
            if r:
                c += 2 * (r * K + N * r + K)
    return {"weight_bytes": w, "compensator_bytes": c, "overhead": c / w}


def select_blocks(nblocks: int, nmasked: int, rank: int, seed: int = 0):
    """Module selection over blocks with synthetic damage scores: `nmasked`
    seeded blocks carry equal damage and the rest almost none, so the
    entropy rule selects those blocks; the budget buys `rank` on each.
    Returns (mask [nblocks] uint8, ranks [nblocks] int32)."""
    rng = np.random.default_rng(seed)
    hot = rng.choice(nblocks, size=nmasked, replace=False)
    damage = np.full(nblocks, 1e-9, np.float32)
    damage[hot] = 1.0
    cost = np.full(nblocks, float(sum(rank_cost_bytes(K, N) for _, K, N in BLOCK_LINEARS)), np.float32)
    budget = float(rank) * float(cost[0]) * nmasked
    return spear.spear_layer_select_mask(damage, cost, budget, 16, rank)


@dataclass
class StackLayer:
    block: int
    name: str
    K: int
    N: int
    layer: spear.W4Layer


def _bf16_dev(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def build_stack(ranks, device, seed: int = 0, recipe: str = "device") -> List[StackLayer]:
    """Packs every linear of the stack.  ranks[b] is block b's compensator rank
    (0: plain W4).  recipe "numpy" draws each layer with inputs.make_layer (the
    oracle's inputs, for parity); "device" draws the same distributions with a
    seeded torch generator on the GPU (for the full 32-block stack, where host
    draws of 26 GB of fp32 weights would dominate)."""
    layers = []
    gen = torch.Generator(device=device)
    for b, r in enumerate(ranks):
        r = int(r)
        for i, (name, K, N) in enumerate(BLOCK_LINEARS):
            lseed = seed + 1000 * b + i
            if recipe == "numpy":
                lay, _ = make_layer(N, K, r, seed=lseed)
                W = torch.from_numpy(lay.W).to(device)
                A = _bf16_dev(lay.A, device) if r else None
                B = _bf16_dev(lay.B, device) if r else None
                wg = _bf16_dev(lay.w_g, device) if r else None
                b_g, alpha = lay.b_g, lay.alpha
            else:
                gen.manual_seed(lseed)
                W = torch.randn(N, K, generator=gen, device=device) * 0.02
                A = (torch.randn(r, K, generator=gen, device=device) * 0.01).to(torch.bfloat16) if r else None
                B = (torch.randn(N, r, generator=gen, device=device) * 0.01).to(torch.bfloat16) if r else None
                wg = (torch.randn(K, generator=gen, device=device) * 0.05).to(torch.bfloat16) if r else None
                b_g, alpha = 0.0, 1.0
            q, s, z = spear.spear_pack_w4(W, K, True)          # per-output-channel symmetric
            del W
            layers.append(StackLayer(b, name, K, N, spear.W4Layer(N, K, K, True, q, s, z, r, A, B, wg, b_g,
                                                                  alpha, r > 0)))
    return layers


class StackStep:
    """Fixed token buffers, one output buffer per linear and path, shared
    workspaces, and one CUDA graph per path."""

    def __init__(self, layers: List[StackLayer], M_prefill: int, M_decode: int, device, seed: int = 0):
        self.layers, self.Mp, self.Md, self.device = layers, M_prefill, M_decode, device
        rng = np.random.default_rng(seed)
        widths = sorted({sl.K for sl in layers})
        # host bf16 bits of the token buffers (the oracle's inputs) and their device copies
        self.xp_bits = {K: f32_to_bf16_bits(rng.standard_normal((M_prefill, K), dtype=np.float32)) for K in widths}
        self.xd_bits = {K: f32_to_bf16_bits(rng.standard_normal((M_decode, K), dtype=np.float32)) for K in widths}
        self.xp = {K: _bf16_dev(v, device) for K, v in self.xp_bits.items()}
        self.xd = {K: _bf16_dev(v, device) for K, v in self.xd_bits.items()}
        self.yp = [torch.empty(M_prefill, sl.N, dtype=torch.bfloat16, device=device) for sl in layers]
        self.yd = [torch.empty(M_decode, sl.N, dtype=torch.bfloat16, device=device) for sl in layers]
        self.ws_p = spear.new_workspace(max(spear.spear_prefill_workspace_bytes(sl.layer, M_prefill)
                                            for sl in layers), device, zero=False)
        self.ws_d = spear.new_workspace(max(spear.spear_decode_workspace_bytes(sl.layer, M_decode)
                                            for sl in layers), device)
        self.stream = torch.cuda.Stream(device)
        self.aux = torch.cuda.Stream(device)
        self.graphs = {}

    def prefill_pass(self):
        for sl, y in zip(self.layers, self.yp):
            spear.spear_linear_prefill(sl.layer, self.xp[sl.K], y=y, workspace=self.ws_p, stream=self.stream,
                                       stream_aux=self.aux)

    def decode_pass(self):
        for sl, y in zip(self.layers, self.yd):
            spear.spear_linear_decode(sl.layer, self.xd[sl.K], y=y, workspace=self.ws_d, stream=self.stream)

    def capture(self):
        torch.cuda.synchronize(self.device)
        with torch.cuda.stream(self.stream):
            self.prefill_pass()                 # plans, tensor maps and function attributes settle eagerly
            self.decode_pass()
        torch.cuda.synchronize(self.device)
        for name, fn in (("prefill", self.prefill_pass), ("decode", self.decode_pass)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                fn()
            self.graphs[name] = g
        torch.cuda.synchronize(self.device)

    def replay(self, name: str):
        # a graph replays on the current stream: make it the step's own
        with torch.cuda.stream(self.stream):
            self.graphs[name].replay()

    def prefill_flops(self) -> float:
        f = 0.0
        for sl in self.layers:
            r = sl.layer.rank if sl.layer.comp_enabled else 0
            f += 2.0 * self.Mp * sl.N * sl.K + (2.0 * self.Mp * r * (sl.K + sl.N) + 2.0 * self.Mp * sl.K if r else 0.0)
        return f

    def decode_bytes(self) -> float:
        b = 0.0
        for sl in self.layers:
            K, N, r = sl.K, sl.N, (sl.layer.rank if sl.layer.comp_enabled else 0)
            b += N * K / 2 + N * 2 + (r + 1) * K * 2 * (r > 0) + N * r * 2 + self.Md * K * 2 + self.Md * N * 2
        return b


__all__ = ["BLOCK_LINEARS", "rank_cost_bytes", "memory_bytes", "select_blocks", "build_stack", "StackLayer", "StackStep"]
