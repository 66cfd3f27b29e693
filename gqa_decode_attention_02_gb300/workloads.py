"""Seeded synthetic inputs for paged GQA decode / verify attention.

This module is shared by the tests, the bench and the CPU oracle's callers.  It
holds no arithmetic of the method itself (no scores, softmax, argmax or slot
arithmetic beyond laying out the block pool): it draws random numbers, lays out
a paged block pool and fills unused cache slots with NaN sentinels, so that any
read of a slot outside a sequence's context poisons the result.

Value recipe: every element is drawn as fp32 N(0,1) from a torch.Generator seeded
per workload and rounded (round-to-nearest-even) to the workload dtype.  Unused
cache slots hold NaN; unused block-table entries hold INT32_MAX.

Inputs of stochastic acceptance (speculative sampling) are probability rows
drawn from Dirichlet distributions: the target's rows q ~ Dir(alpha) (alpha < 1
gives the peaked rows of a language model), the draft's rows a mixture of q and
an independent Dirichlet row, so that drafts and target mostly agree; each draft
id is drawn from its draft row, and the acceptance uniforms are U[0,1) doubles.

The five named workloads follow the shapes of the pages' own running examples:
the 24-layer, 14-query-head, 2-KV-head, H=64 fp16 model measured on page "جعل
inference رخيصًا: KV cache وbatching والتكميم", a Llama-style N=32/K=8/H=128
bf16 geometry, and a 4-draft speculative-verify batch (page "Болжау арқылы Sonar
модельдерін жылдамдату").
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

INT32_MAX = 2**31 - 1
BLOCK_SIZE = 16

_TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    T: int
    N: int
    K: int
    H: int
    dtype: str  # "f16" | "bf16"
    layers: int
    block_size: int
    num_blocks: int
    max_blocks: int
    context_lens: torch.Tensor  # int32 [B]
    block_tables: torch.Tensor  # int32 [B, max_blocks]
    q: list  # per layer [B,T,N,H]
    k_cache: list  # per layer [NB,bs,K,H]
    v_cache: list
    k_new: list  # per layer [B,T,K,H] (the T tokens the append writes)
    v_new: list
    appended: bool  # True: the caches do NOT yet hold the T new tokens (NaN there)
    logits: Optional[torch.Tensor] = None  # fp32 [B,T,V] (verify workloads)
    draft: Optional[torch.Tensor] = None  # int32 [B,T-1]
    draft_k: Optional[np.ndarray] = None  # planted accepted-prefix length (tree: node) per b
    desc: str = ""
    windows: tuple = ()  # per layer: local-attention window, 0 = global (all 0 if empty)
    tree: tuple = ()  # draft tree over the T new tokens: parent of each (-1: the prefix)

    def window(self, layer: int) -> int:
        return self.windows[layer] if self.windows else 0

    def tree_mask(self) -> Optional[np.ndarray]:
        """uint64 [B,T] mask rows of the draft tree (bit j of row t: new token
        t's ancestor j), the same tree for every sequence; None without a tree."""
        if not self.tree:
            return None
        rows = np.zeros(self.T, np.uint64)
        for t, a in enumerate(self.tree):
            while a >= 0:
                rows[t] |= np.uint64(1) << np.uint64(a)
                a = self.tree[a]
        return np.tile(rows, (self.B, 1))

    def parents(self) -> Optional[np.ndarray]:
        """int32 [B,T] parent of each new token in the draft tree (-1 for the
        root), the same tree for every sequence; None without a tree."""
        if not self.tree:
            return None
        return np.tile(np.asarray(self.tree, np.int32), (self.B, 1))

    @property
    def G(self) -> int:
        return self.N // self.K

    @property
    def torch_dtype(self):
        return _TORCH_DT[self.dtype]


def _randn_into(out: torch.Tensor, gen: torch.Generator, chunk_elems: int = 1 << 26):
    """Fill `out` (fp16/bf16, any device) with N(0,1) rounded to its dtype,
    drawing fp32 in chunks so big caches never need an fp32 copy."""
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        flat[s:e] = torch.randn(e - s, generator=gen, dtype=torch.float32,
                                device=out.device).to(out.dtype)


def context_lengths(kind: str, B: int, rng: np.random.Generator, *args) -> np.ndarray:
    """Context-length mixes of the workloads (tokens held per sequence, including
    the new ones).  fixed(c); uniform(lo, hi) inclusive; lognormal(median, sigma,
    lo, hi): ln c ~ N(ln median, sigma^2), rounded to nearest, clipped."""
    if kind == "fixed":
        return np.full(B, int(args[0]), np.int64)
    if kind == "uniform":
        lo, hi = args
        return rng.integers(lo, hi + 1, size=B)
    if kind == "lognormal":
        median, sigma, lo, hi = args
        x = np.rint(np.exp(rng.normal(math.log(median), sigma, size=B)))
        return np.clip(x, lo, hi).astype(np.int64)
    raise ValueError(kind)


def build(name: str, B: int, T: int, N: int, K: int, H: int, dtype: str,
          ctx: np.ndarray, *, seed: int, layers: int = 1, shuffle: bool = True,
          append: bool = True, spare_blocks: int = 1, block_size: int = BLOCK_SIZE,
          max_blocks: Optional[int] = None, device="cpu", vocab: int = 0,
          desc: str = "", windows: tuple = (), tree: tuple = ()) -> Workload:
    """Lay out a paged block pool for the given context lengths and fill it.

    Physical blocks: sum_b ceil(ctx_b / bs) in use plus `spare_blocks` never
    referenced; ids are a random permutation of the pool when `shuffle`, else
    0,1,2,... in sequence order.  When `append` is set, the T newest positions
    of each sequence are left as NaN in the cache (the append fills them)."""
    assert N % K == 0
    gen = torch.Generator(device=device).manual_seed(seed)
    rng = np.random.default_rng(seed)
    ctx = np.asarray(ctx, np.int64)
    nblk = (ctx + block_size - 1) // block_size
    used = int(nblk.sum())
    NB = used + spare_blocks
    if max_blocks is None:
        max_blocks = max(1, int(nblk.max()) if B else 1)
    ids = rng.permutation(NB) if shuffle else np.arange(NB)
    tables = np.full((B, max_blocks), INT32_MAX, np.int64)
    off = 0
    for b in range(B):
        tables[b, : nblk[b]] = ids[off: off + nblk[b]]
        off += nblk[b]
    tdt = _TORCH_DT[dtype]
    nan_slots = []  # (block, row) pairs that must hold NaN
    for b in range(B):
        first_nan = ctx[b] - T if append else ctx[b]
        first_nan = max(first_nan, 0)
        for pos in range(first_nan, nblk[b] * block_size):
            nan_slots.append((tables[b, pos // block_size], pos % block_size))
    spare = ids[used:]

    qs, kcs, vcs, kns, vns = [], [], [], [], []
    for _ in range(layers):
        q = torch.empty((B, T, N, H), dtype=tdt, device=device)
        kc = torch.empty((NB, block_size, K, H), dtype=tdt, device=device)
        vc = torch.empty_like(kc)
        kn = torch.empty((B, T, K, H), dtype=tdt, device=device)
        vn = torch.empty_like(kn)
        for t_ in (q, kc, vc, kn, vn):
            _randn_into(t_, gen)
        if nan_slots:
            sl = torch.as_tensor(np.array(nan_slots, np.int64), device=device)
            kc[sl[:, 0], sl[:, 1]] = float("nan")
            vc[sl[:, 0], sl[:, 1]] = float("nan")
        if len(spare):
            sp = torch.as_tensor(spare, device=device)
            kc[sp] = float("nan")
            vc[sp] = float("nan")
        qs.append(q)
        kcs.append(kc)
        vcs.append(vc)
        kns.append(kn)
        vns.append(vn)

    w = Workload(name=name, B=B, T=T, N=N, K=K, H=H, dtype=dtype, layers=layers,
                 block_size=block_size, num_blocks=NB, max_blocks=max_blocks,
                 context_lens=torch.as_tensor(ctx.astype(np.int32), device=device),
                 block_tables=torch.as_tensor(tables.astype(np.int32), device=device),
                 q=qs, k_cache=kcs, v_cache=vcs, k_new=kns, v_new=vns,
                 appended=append, desc=desc, windows=tuple(windows), tree=tuple(tree))
    if vocab:
        logits = torch.randn((B, T, vocab), generator=gen, dtype=torch.float32,
                             device=device)
        # Drafts: the first k_b positions carry the target's choice by construction
        # (a planted logit of 10.0, far above any N(0,1) draw of this size), the
        # rest are uniform random ids.  The oracle, not this recipe, decides the
        # accepted length.  With a draft tree, k_b is a node and its branch is
        # planted the same way.
        kb = rng.integers(0, T, size=B)  # k uniform in 0..T-1
        draft = rng.integers(0, vocab, size=(B, max(T - 1, 0)))
        li = logits.cpu() if device != "cpu" else logits
        for b in range(B):
            if tree:
                # a draft tree: node kb[b]'s branch carries the target's choice
                # at every edge (the logit of the child's token planted at its
                # parent's row); draft[b, c-1] is node c's token
                c = int(kb[b])
                while c > 0:
                    li[b, tree[c], int(draft[b, c - 1])] = 10.0
                    c = tree[c]
            else:
                for t in range(int(kb[b])):
                    li[b, t, int(draft[b, t])] = 10.0
        if device != "cpu":
            logits.copy_(li)
        w.logits = logits
        w.draft = torch.as_tensor(draft.astype(np.int32), device=device)
        w.draft_k = kb
    return w


# The five workloads: (description, builder kwargs, context-length recipe, seed)
SPECS = {
    "cfg1": dict(
        desc="single layer, B=1, T=1, N=14, K=2, H=64, fp16, context 295, "
             "contiguous block table",
        B=1, T=1, N=14, K=2, H=64, dtype="f16", layers=1, shuffle=False,
        append=False, ctx=("fixed", 295), seed=101),
    "cfg2": dict(
        desc="24 layers back-to-back, B=64, T=1, N=14, K=2, H=64, fp16, context "
             "U[16,1024], block tables a random permutation of a shared pool",
        B=64, T=1, N=14, K=2, H=64, dtype="f16", layers=24, shuffle=True,
        append=True, ctx=("uniform", 16, 1024), seed=102),
    "cfg3": dict(
        desc="single layer, B=32, T=1, N=32, K=8, H=128, bf16, context 8192 "
             "(8191 cached + 1 appended), shuffled blocks",
        B=32, T=1, N=32, K=8, H=128, dtype="bf16", layers=1, shuffle=True,
        append=True, ctx=("fixed", 8192), seed=103),
    "cfg4": dict(
        desc="ragged batch, B=256, T=1, N=32, K=8, H=128, bf16, context "
             "log-normal (median 2048, sigma 1.0) clipped to [1,32768], shuffled, "
             "append 1 then decode",
        B=256, T=1, N=32, K=8, H=128, dtype="bf16", layers=1, shuffle=True,
        append=True, ctx=("lognormal", 2048, 1.0, 1, 32768), seed=104),
    "cfg5": dict(
        desc="speculative verify, B=16, T=5, N=64, K=8, H=128, bf16, context "
             "U[512,4096], causal among the 5 new tokens; greedy acceptance over "
             "fp32 logits [16,5,32000]",
        B=16, T=5, N=64, K=8, H=128, dtype="bf16", layers=1, shuffle=True,
        append=True, ctx=("uniform", 512, 4096), seed=105, vocab=32000),
    # Not one of the five: local attention in a hybrid-layer schedule (one
    # global layer in every six, the rest local), on the long-context geometry.
    "hybrid": dict(
        desc="hybrid local/global layers: 6 layers, layers 0-4 local attention with a "
             "1024-token window, layer 5 global; B=32, T=1, N=32, K=8, H=128, bf16, "
             "context 8192 (8191 cached + 1 appended), shuffled blocks",
        B=32, T=1, N=32, K=8, H=128, dtype="bf16", layers=6, shuffle=True,
        append=True, ctx=("fixed", 8192), seed=106, windows=(1024,) * 5 + (0,)),
    # Not one of the five: tree verification of a 26-node draft tree (a root,
    # then 3, 6, 8 and 8 candidates per level) on the verify geometry, then
    # greedy acceptance over the tree and compaction of the kept branch.
    "tree": dict(
        desc="tree verify, B=16, T=26 (draft tree: 1 root, 3, 6, 8, 8 nodes per level), "
             "N=64, K=8, H=128, bf16, context U[512,4096], custom mask among the new tokens; "
             "greedy acceptance over the tree (fp32 logits [16,26,32000]) and compaction "
             "of the kept branch's cache rows",
        B=16, T=26, N=64, K=8, H=128, dtype="bf16", layers=1, shuffle=True,
        append=True, ctx=("uniform", 512, 4096), seed=107, vocab=32000,
        tree=(-1, 0, 0, 0, 1, 1, 2, 2, 3, 3) + tuple(4 + i // 2 for i in range(8))
        + tuple(10 + i for i in range(8))),
}


def make(name: str, *, device="cpu", seed: Optional[int] = None,
         B: Optional[int] = None, layers: Optional[int] = None,
         append: Optional[bool] = None) -> Workload:
    """One of the five named workloads (optionally with fewer sequences or
    layers, for the oracle's bounded samples)."""
    s = dict(SPECS[name])
    seed = s.pop("seed") if seed is None else seed
    s.pop("seed", None)
    kind, *args = s.pop("ctx")
    desc = s.pop("desc")
    if B is not None:
        s["B"] = B
    if layers is not None:
        s["layers"] = layers
    if append is not None:
        s["append"] = append
    rng = np.random.default_rng(seed + 7919)
    ctx = context_lengths(kind, s["B"], rng, *args)
    return build(name, ctx=ctx, seed=seed, device=device, desc=desc, **s)


@dataclasses.dataclass
class SamplingInputs:
    q: torch.Tensor         # fp32 [B,T,V] target probabilities
    p: torch.Tensor         # fp32 [B,T-1,V] draft probabilities
    draft: torch.Tensor     # int32 [B,T-1], draft[b,t] drawn from p[b,t]
    uniforms: torch.Tensor  # fp64 [B,T] in [0,1)


def sampling_inputs(B: int, T: int, V: int, seed: int, device="cpu", alpha: float = 0.1,
                    mix: float = 0.7) -> SamplingInputs:
    """Seeded inputs for stochastic acceptance: q ~ Dir(alpha) per row, p =
    mix * q + (1 - mix) * Dir(alpha) per row, both rounded to fp32; drafts
    drawn from p (in fp64); uniforms U[0,1)."""
    rng = np.random.default_rng(seed)
    q64 = rng.dirichlet(np.full(V, alpha), size=(B, T))
    d64 = rng.dirichlet(np.full(V, alpha), size=(B, max(T - 1, 0)))
    p64 = mix * q64[:, : T - 1] + (1.0 - mix) * d64
    draft = np.zeros((B, max(T - 1, 0)), np.int32)
    for b in range(B):
        for t in range(T - 1):
            c = np.cumsum(p64[b, t])
            draft[b, t] = min(int(np.searchsorted(c, rng.random() * c[-1], side="right")),
                              V - 1)
    u = rng.random((B, T))
    return SamplingInputs(
        q=torch.as_tensor(q64.astype(np.float32), device=device),
        p=torch.as_tensor(p64.astype(np.float32).reshape(B, max(T - 1, 0), V), device=device),
        draft=torch.as_tensor(draft, device=device),
        uniforms=torch.as_tensor(u, dtype=torch.float64, device=device))
