"""Seeded synthetic inputs for the verify step (shared by tests, bench and smoke).

This module only draws inputs: logits with the shapes and value distributions of
the workloads below, draft tokens, accept uniforms r and per-sequence sampling
keys.  It holds none of the verify step's arithmetic.  The draft tokens stand
in for a draft model's sampler: they are drawn from softmax(draft / T) with
``torch.multinomial`` (T > 0) or taken as the draft argmax (T = 0).

Workloads (stand-ins for the pages' evaluation sets, which are not used):
  tiny    B=1,  gamma=4, V=1000,    fp32: z ~ N(0, 2^2); d = z + N(0, 0.5^2)
  spd     B=64, gamma=1, V=151936,  bf16: z ~ N(0, 3^2) with 20 peak ids per
          target row raised by +8; d = z + N(0, 1^2)
  eagle   B=32, gamma in {7, 15}, V=128256, bf16: z ~ N(0, 2.5^2);
          d = 0.8 z + N(0, 1.5^2)
  fanout  draft [8, 5, 128256] fp32 ~ N(0, 2^2); exclude[b,k] drawn from
          softmax(d[b,k]) for k < 4, -1 at k = 4; F = round(8 * 0.8^(k/1.5))
  sweep   the spd distributions at gamma=4, V=151936, fp32 / bf16,
          B in {1, 8, 64, 128, 256}
Any chain workload can also draw the draft row of the bonus position
(``bonus_draft``), which the speculation-cache fan-out ranks, and can draw its
draft tokens from the top_k / top_p restricted draft distribution (the
filtered verify's input).
All draws are fp32 from seeded ``torch.Generator`` s on the requested device,
then cast to the workload dtype; V is the last, contiguous axis.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

SEEDS = dict(tiny=(100, 101, 0, 1), spd=(200, 201, 0, 1), eagle=(300, 301, 2, 3), sweep=(200, 201, 0, 1))
PEAK_SEED = 202
FANOUT_SEEDS = (400, 4)
TREE_SEEDS = (500, 501, 5, 6)
# Draft-tree shapes: children per node, level by level.  "k21": the 21-node
# tree (root, 4, 8, 8) of tree-style verification; "w4": width-4 tree drafting
# (root with 4 children, each continued by a chain of 3); "b63": a binary
# tree of depth 5 (63 nodes, near the node limit).
TREE_SHAPES = {"k21": [4, 2, 1], "w4": [4, 1, 1, 1], "path4": [1, 1, 1, 1], "b63": [2, 2, 2, 2, 2]}
BONUS_SEED_OFFSET = 7919  # seed of the bonus-position draft row = draft seed + this


@dataclass
class ChainInputs:
    name: str
    target: torch.Tensor          # [B, gamma+1, V]
    draft: torch.Tensor           # [B, gamma, V]
    tokens: torch.Tensor          # [B, gamma] int32
    r: torch.Tensor               # [B, gamma] fp32 in (0, 1]
    keys: torch.Tensor            # [B] int64 holding uint64 bit patterns
    temperature: float
    meta: dict = field(default_factory=dict)
    draft_bonus: torch.Tensor | None = None  # [B, 1, V] draft logits at position gamma (fan-out input)

    @property
    def B(self):
        return self.target.shape[0]

    @property
    def gamma(self):
        return self.target.shape[1] - 1

    @property
    def V(self):
        return self.target.shape[2]


@dataclass
class FanoutInputs:
    name: str
    draft: torch.Tensor           # [B, K+1, V]
    exclude: torch.Tensor         # [B, K+1] int32, -1 = none
    fanout: list                  # K+1 ints


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _draft_tokens(d: torch.Tensor, temperature: float, seed: int, device, top_k=None, top_p=1.0) -> torch.Tensor:
    """The draft model's sampler: softmax(d / T), optionally restricted to the
    top_k logits and the top_p nucleus of those (torch.topk order)."""
    B, g, V = d.shape
    if g == 0:
        return torch.zeros(B, 0, dtype=torch.int32, device=device)
    flat = d.float().reshape(B * g, V)
    if temperature == 0:
        return flat.argmax(dim=1).to(torch.int32).reshape(B, g)
    if top_k is None:
        probs = torch.softmax(flat / temperature, dim=1)
        return torch.multinomial(probs, 1, generator=_gen(device, seed)).to(torch.int32).reshape(B, g)
    vals, ids = torch.topk(flat, min(top_k, V), dim=1)
    probs = torch.softmax(vals / temperature, dim=1)
    if top_p < 1.0:
        before = torch.cumsum(probs, dim=1) - probs
        probs = torch.where(before < top_p, probs, torch.zeros_like(probs))
    pick = torch.multinomial(probs, 1, generator=_gen(device, seed))
    return ids.gather(1, pick).to(torch.int32).reshape(B, g)


def _uniforms_and_keys(B, g, seed, device):
    gen = _gen(device, seed)
    r = 1.0 - torch.rand(B, g, generator=gen, device=device, dtype=torch.float32)
    keys = torch.randint(-(2 ** 63), 2 ** 63 - 1, (B,), generator=gen, device=device, dtype=torch.int64)
    return r, keys


def chain_from_params(name, B, gamma, V, dtype, temperature, z_std, d_scale, d_std, peaks, seeds,
                      device="cpu", bonus_draft=False, top_k=None, top_p=1.0) -> ChainInputs:
    """Generic generator: z ~ N(0, z_std^2) [B, gamma+1, V] (+8 on `peaks` ids
    per target row), d = d_scale * z[:, :gamma] + N(0, d_std^2).  With
    `bonus_draft` also the draft row of position gamma, d_scale * z[:, gamma]
    + N(0, d_std^2), from its own seed (the other draws are unchanged)."""
    s_z, s_d, s_tok, s_u = seeds
    z = torch.randn(B, gamma + 1, V, generator=_gen(device, s_z), device=device) * z_std
    if peaks:
        score = torch.rand(B, gamma + 1, V, generator=_gen(device, PEAK_SEED), device=device)
        idx = score.topk(peaks, dim=2).indices
        z.scatter_add_(2, idx, torch.full(idx.shape, 8.0, device=device))
        del score, idx
    d = torch.randn(B, gamma, V, generator=_gen(device, s_d), device=device) * d_std
    d.add_(z[:, :gamma], alpha=d_scale)
    draft_bonus = None
    if bonus_draft:
        db = torch.randn(B, 1, V, generator=_gen(device, s_d + BONUS_SEED_OFFSET), device=device) * d_std
        db.add_(z[:, gamma:], alpha=d_scale)
        draft_bonus = db.to(dtype)
        del db
    target = z.to(dtype)
    del z
    draft = d.to(dtype)
    del d
    tokens = _draft_tokens(draft, temperature, s_tok, device, top_k, top_p)
    r, keys = _uniforms_and_keys(B, gamma, s_u, device)
    meta = dict(B=B, gamma=gamma, V=V, dtype=str(dtype).replace("torch.", ""), T=float(temperature))
    if top_k is not None:
        meta.update(top_k=top_k, top_p=top_p)
    return ChainInputs(name, target, draft, tokens, r, keys, float(temperature), meta, draft_bonus)


def tiny(device="cpu", temperature=1.0, bonus_draft=False, top_k=None, top_p=1.0) -> ChainInputs:
    return chain_from_params("tiny", 1, 4, 1000, torch.float32, temperature, 2.0, 1.0, 0.5, 0,
                             SEEDS["tiny"], device, bonus_draft, top_k, top_p)


def spd(device="cpu", temperature=1.0, B=64, bonus_draft=False, top_k=None, top_p=1.0) -> ChainInputs:
    return chain_from_params("spd", B, 1, 151936, torch.bfloat16, temperature, 3.0, 1.0, 1.0, 20,
                             SEEDS["spd"], device, bonus_draft, top_k, top_p)


def eagle(gamma=7, device="cpu", temperature=1.0, B=32, bonus_draft=False, top_k=None, top_p=1.0) -> ChainInputs:
    return chain_from_params(f"eagle_g{gamma}", B, gamma, 128256, torch.bfloat16, temperature, 2.5, 0.8,
                             1.5, 0, SEEDS["eagle"], device, bonus_draft, top_k, top_p)


def sweep(B=64, dtype=torch.float32, device="cpu", temperature=1.0, V=151936, gamma=4,
          bonus_draft=False, top_k=None, top_p=1.0) -> ChainInputs:
    return chain_from_params(f"sweep_B{B}_{str(dtype).replace('torch.', '')}", B, gamma, V, dtype,
                             temperature, 3.0, 1.0, 1.0, 20, SEEDS["sweep"], device, bonus_draft, top_k, top_p)


def cache_fanout_inputs(w: ChainInputs):
    """Fan-out inputs of the speculation cache for a chain workload drawn with
    `bonus_draft`: draft rows of positions 0..gamma [B, gamma+1, V] and the
    token to skip at each, the verified draft token (k < gamma) or none (-1,
    position gamma)."""
    if w.draft_bonus is None:
        raise ValueError("workload drawn without bonus_draft")
    d = torch.cat([w.draft, w.draft_bonus], dim=1)
    ex = torch.cat([w.tokens, torch.full((w.B, 1), -1, dtype=torch.int32, device=w.tokens.device)], dim=1)
    return d, ex


def fanout(device="cpu", B=8, K=4, V=128256, fanout_sizes=(8, 7, 6, 5, 4)) -> FanoutInputs:
    s_d, s_x = FANOUT_SEEDS
    d = torch.randn(B, K + 1, V, generator=_gen(device, s_d), device=device) * 2.0
    ex = torch.full((B, K + 1), -1, dtype=torch.int32, device=device)
    if K > 0:
        probs = torch.softmax(d[:, :K].reshape(B * K, V), dim=1)
        ex[:, :K] = torch.multinomial(probs, 1, generator=_gen(device, s_x)).to(torch.int32).reshape(B, K)
    return FanoutInputs("fanout", d, ex, list(fanout_sizes))


def saguaro_tokens(w: ChainInputs, cache_ids: torch.Tensor, fanout, C: float, seed: int = 9) -> torch.Tensor:
    """The draft's Saguaro sampler (input generation): at position i draw from
    softmax(draft_i / T) with the probability of position i's listed
    candidates (cache_ids [B, sum F], k-major) divided by C."""
    B, g, V = w.draft.shape
    logits = w.draft.float() / w.temperature
    offs = [0]
    for f in fanout:
        offs.append(offs[-1] + int(f))
    for i in range(g):
        ids = cache_ids[:, offs[i]:offs[i + 1]].long()
        ok = (ids >= 0) & (ids < V)
        pen = torch.zeros(B, V, device=logits.device)
        pen.scatter_(1, ids.clamp(0, V - 1), torch.where(ok, -math.log(C), 0.0).float())
        logits[:, i] += pen
    probs = torch.softmax(logits.reshape(B * g, V), dim=1)
    gen = _gen(w.draft.device, seed)
    return torch.multinomial(probs, 1, generator=gen).to(torch.int32).reshape(B, g)


@dataclass
class TreeInputs:
    name: str
    target: torch.Tensor   # [B, N, V]: p at node v
    draft: torch.Tensor    # [B, N, V]: q at node v (its children are drawn from it)
    parent: torch.Tensor   # [B, N] int32, -1 at the root
    tokens: torch.Tensor   # [B, N] int32, token of node v (0 at the root)
    r: torch.Tensor        # [B, N] fp32 in (0, 1]
    keys: torch.Tensor     # [B] int64
    temperature: float

    @property
    def B(self):
        return self.target.shape[0]

    @property
    def N(self):
        return self.target.shape[1]

    @property
    def V(self):
        return self.target.shape[2]


def tree_parents(shape) -> list:
    """Parents of a tree built level by level: every node of a level gets
    shape[level] children; nodes are numbered breadth first."""
    parent, level = [-1], [0]
    for width in shape:
        nxt = []
        for u in level:
            for _ in range(width):
                parent.append(u)
                nxt.append(len(parent) - 1)
        level = nxt
    return parent


def tree(B=64, shape="k21", V=151936, dtype=torch.bfloat16, temperature=1.0, device="cpu", z_std=3.0, d_std=1.0,
         peaks=20) -> TreeInputs:
    """Draft trees on the spd distributions: z ~ N(0, z_std^2) per node (+8
    on `peaks` ids), d = z + N(0, d_std^2); at T > 0 the children of u are
    drawn i.i.d. from softmax(d_u / T), at T = 0 they are the top draft ids
    of u in rank order (distinct)."""
    par = tree_parents(TREE_SHAPES[shape])
    N = len(par)
    s_z, s_d, s_tok, s_u = TREE_SEEDS
    z = torch.randn(B, N, V, generator=_gen(device, s_z), device=device) * z_std
    if peaks:
        score = torch.rand(B, N, V, generator=_gen(device, PEAK_SEED), device=device)
        idx = score.topk(peaks, dim=2).indices
        z.scatter_add_(2, idx, torch.full(idx.shape, 8.0, device=device))
        del score, idx
    d = torch.randn(B, N, V, generator=_gen(device, s_d), device=device) * d_std
    d.add_(z)
    target, draft = z.to(dtype), d.to(dtype)
    del z, d
    tok = torch.zeros(B, N, dtype=torch.int32, device=device)
    gen = _gen(device, s_tok)
    kids = {}
    for v in range(1, N):
        kids.setdefault(par[v], []).append(v)
    for u, cs in kids.items():
        du = draft[:, u].float()
        if temperature == 0:
            top = du.topk(len(cs), dim=1).indices
            for j, c in enumerate(cs):
                tok[:, c] = top[:, j].to(torch.int32)
        else:
            probs = torch.softmax(du / temperature, dim=1)
            pick = torch.multinomial(probs, len(cs), replacement=True, generator=gen)
            for j, c in enumerate(cs):
                tok[:, c] = pick[:, j].to(torch.int32)
    g2 = _gen(device, s_u)
    r = 1.0 - torch.rand(B, N, generator=g2, device=device, dtype=torch.float32)
    keys = torch.randint(-(2 ** 63), 2 ** 63 - 1, (B,), generator=g2, device=device, dtype=torch.int64)
    parent = torch.tensor(par, dtype=torch.int32, device=device).repeat(B, 1)
    return TreeInputs(f"tree_{shape}", target, draft, parent, tok, r, keys, float(temperature))
