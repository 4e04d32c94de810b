"""Seeded synthetic workloads for the headwise-chunked causal GQA attention layer.

This module holds the workload table and the seeded input generators, and
nothing else: none of the layer's arithmetic lives here.  Both the CUDA path
(through its tests and ``bench.py``) and the float64 oracle draw their inputs
from here, so the two sides see the same numbers without sharing any code.

The geometries are the attention layers the Untied Ulysses pages train
(Llama 3B / Llama3-8B / Qwen3-32B, "Results" of the memeeeeeex.com article and
the talk transcript on liquidgold.cc).  The pages use trained weights and real
data; here random values of the stated distributions stand in for them:
x ~ N(0, 1), each weight ~ N(0, 1/fan_in), the upstream gradient ~ N(0, 1),
all rounded to bf16.  Draw order: x, Wq, Wk, Wv, Wo, dOut (and, for the
qk-norm geometry, the two norm gains, which default to ones).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    S: int
    hidden: int
    Hq: int
    Hkv: int
    d: int
    chunk_heads: tuple
    rope_theta: float
    qk_norm: bool = False
    norm_eps: float = 1e-6
    passes: tuple = ("fwd",)
    sampled: bool = False          # oracle checks sampled rows only at this size

    @property
    def group(self) -> int:
        return self.Hq // self.Hkv

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    w.name: w
    for w in [
        # tiny causal GQA layer, one KV group per chunk
        Workload("tiny-s2048", S=2048, hidden=256, Hq=4, Hkv=2, d=64,
                 chunk_heads=(2,), rope_theta=1e4, passes=("fwd", "bwd")),
        # Llama-3.2-3B attention geometry, full layer on one GPU, 64K tokens
        Workload("llama3.2-3b-s65536", S=65536, hidden=3072, Hq=24, Hkv=8,
                 d=128, chunk_heads=(3, 6, 24), rope_theta=5e5,
                 passes=("fwd",), sampled=True),
        # Llama-3-8B, one rank of an 8-way Ulysses split: 4 of 32 q heads,
        # 1 of 8 kv heads, full 1M-token sequence
        Workload("llama3-8b-rank-s1m", S=1 << 20, hidden=4096, Hq=4, Hkv=1,
                 d=128, chunk_heads=(1, 2, 4), rope_theta=5e5,
                 passes=("fwd", "bwd"), sampled=True),
        # the same rank shard at 5M tokens
        Workload("llama3-8b-rank-s5m", S=5 * (1 << 20), hidden=4096, Hq=4,
                 Hkv=1, d=128, chunk_heads=(1,), rope_theta=5e5,
                 passes=("fwd",), sampled=True),
        # Qwen3-32B, one rank of an 8-way split: 8 of 64 q heads, 1 of 8 kv
        # heads, per-head RMSNorm on q and k before RoPE
        Workload("qwen3-32b-rank-s1m", S=1 << 20, hidden=5120, Hq=8, Hkv=1,
                 d=128, chunk_heads=(1, 2, 4, 8), rope_theta=1e6,
                 qk_norm=True, norm_eps=1e-6, passes=("fwd", "bwd"),
                 sampled=True),
    ]
}

WORKLOAD_ORDER = list(WORKLOADS)


_BLOCK = 1 << 28  # elements drawn per call for large tensors


def _randn(shape, std, gen, device):
    n = 1
    for s in shape:
        n *= s
    if n <= _BLOCK:
        t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        return t.to(torch.bfloat16)
    # large tensors (million-token x): drawn in row blocks so that no full
    # float32 copy exists; the values are a fixed function of the seed
    out = torch.empty(shape, device=device, dtype=torch.bfloat16)
    flat = out.view(-1)
    for lo in range(0, n, _BLOCK):
        hi = min(n, lo + _BLOCK)
        t = torch.randn(hi - lo, generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        flat[lo:hi] = t.to(torch.bfloat16)
    return out


def make_inputs(w: Workload, seed: int = 0, device: str = "cpu",
                with_grad: bool = False, norm_gains: str = "ones"):
    """Draw the layer's inputs for workload ``w``.

    Returns a dict of bf16 tensors on ``device``:
      x [S, hidden], Wq [Hq*d, hidden], Wk/Wv [Hkv*d, hidden],
      Wo [hidden, Hq*d] (nn.Linear layout: [out_features, in_features]),
      dout [S, hidden] when ``with_grad``;
    plus float32 norm gains q_gamma/k_gamma [d] for qk-norm workloads
    (ones, or N(1, 0.1) when ``norm_gains == "random"``).
    The generator lives on ``device`` (torch's Philox on CUDA, mt19937 on
    CPU), so the same seed gives different numbers on the two devices; each
    test states which device drew its inputs.
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    S, h, d = w.S, w.hidden, w.d
    out = {
        "x": _randn((S, h), 1.0, gen, device),
        "Wq": _randn((w.Hq * d, h), h ** -0.5, gen, device),
        "Wk": _randn((w.Hkv * d, h), h ** -0.5, gen, device),
        "Wv": _randn((w.Hkv * d, h), h ** -0.5, gen, device),
        "Wo": _randn((h, w.Hq * d), (w.Hq * d) ** -0.5, gen, device),
    }
    if with_grad:
        out["dout"] = _randn((S, h), 1.0, gen, device)
    if w.qk_norm:
        if norm_gains == "random":
            g = torch.randn((2, d), generator=gen, device=device) * 0.1 + 1.0
            out["q_gamma"], out["k_gamma"] = g[0].contiguous(), g[1].contiguous()
        else:
            out["q_gamma"] = torch.ones(d, device=device)
            out["k_gamma"] = torch.ones(d, device=device)
    return out


@dataclasses.dataclass(frozen=True)
class MlpWorkload:
    """The decoder layer's SwiGLU MLP over S tokens, computed in tiles of
    tile_rows tokens (the sequence-tiled MLP of the pages' memory stack)."""
    name: str
    S: int
    hidden: int
    ffn: int
    tile_rows: int

    def with_(self, **kw) -> "MlpWorkload":
        return dataclasses.replace(self, **kw)


MLP_WORKLOADS = {
    w.name: w
    for w in [
        # Llama-3-8B's MLP (hidden 4096, ffn 14336) on one rank of an 8-way
        # Ulysses split of 1M tokens: the MLP is sequence-sharded, so a rank
        # holds S/8 = 131072 tokens; tiles of 8192 tokens
        MlpWorkload("llama3-8b-mlp-rank-s1m", S=1 << 17, hidden=4096, ffn=14336,
                    tile_rows=8192),
    ]
}


def make_mlp_inputs(w: MlpWorkload, seed: int = 0, device: str = "cpu",
                    with_grad: bool = False):
    """Draw the MLP's inputs: x [S, hidden] ~ N(0, 1); Wg, Wu [ffn, hidden]
    ~ N(0, 1/hidden); Wd [hidden, ffn] ~ N(0, 1/ffn); dy [S, hidden] ~ N(0, 1)
    when ``with_grad``; all bf16, drawn in that order."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    out = {
        "x": _randn((w.S, w.hidden), 1.0, gen, device),
        "Wg": _randn((w.ffn, w.hidden), w.hidden ** -0.5, gen, device),
        "Wu": _randn((w.ffn, w.hidden), w.hidden ** -0.5, gen, device),
        "Wd": _randn((w.hidden, w.ffn), w.ffn ** -0.5, gen, device),
    }
    if with_grad:
        out["dy"] = _randn((w.S, w.hidden), 1.0, gen, device)
    return out


@dataclasses.dataclass(frozen=True)
class LossWorkload:
    """The last layer's cross-entropy loss over a vocabulary of ``vocab`` words
    for S tokens, computed in tiles of tile_rows tokens."""
    name: str
    S: int
    hidden: int
    vocab: int
    tile_rows: int

    def with_(self, **kw) -> "LossWorkload":
        return dataclasses.replace(self, **kw)


LOSS_WORKLOADS = {
    w.name: w
    for w in [
        # Llama-3-8B's output projection (hidden 4096, vocabulary 128256) on
        # one rank's 131072 tokens (1M over an 8-way split); tiles of 4096
        LossWorkload("llama3-8b-loss-rank-s1m", S=1 << 17, hidden=4096, vocab=128256,
                     tile_rows=4096),
    ]
}


def make_loss_inputs(w: LossWorkload, seed: int = 0, device: str = "cpu"):
    """Draw the loss's inputs: h [S, hidden] ~ N(0, 1), W [vocab, hidden]
    ~ N(0, 1/hidden) (bf16), and targets [S] int32 uniform over the
    vocabulary, in that order."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    out = {
        "h": _randn((w.S, w.hidden), 1.0, gen, device),
        "W": _randn((w.vocab, w.hidden), w.hidden ** -0.5, gen, device),
    }
    out["targets"] = torch.randint(0, w.vocab, (w.S,), generator=gen, device=device,
                                   dtype=torch.int32)
    return out


def sample_rows(S: int, n: int = 256, seed: int = 0, tile: int = 128):
    """Seeded sorted query rows: always 0, 1, tile-1, tile, S/2, S-1 and tile
    edges, the rest uniform; the same rows serve every head."""
    fixed = {0, 1, tile - 1, tile, tile + 1, S // 2, S - 1, S - 2,
             S - tile, S - tile - 1, 2 * tile - 1, 2 * tile}
    fixed = {r for r in fixed if 0 <= r < S}
    g = torch.Generator().manual_seed(seed)
    need = max(0, min(n, S) - len(fixed))
    rest = set()
    while len(rest) < need:
        cand = torch.randint(0, S, (need * 2,), generator=g).tolist()
        for c in cand:
            if c not in fixed:
                rest.add(c)
            if len(rest) >= need:
                break
    return sorted(fixed | rest)[: max(n, len(fixed))]
