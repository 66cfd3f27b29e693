"""Small helpers shared by the tests (no library or oracle arithmetic)."""
from __future__ import annotations

import numpy as np
import torch

from gqa_decode_attention_02_gb300 import workloads


def small(B=3, T=1, N=8, K=2, H=64, dtype="f16", ctx=(5, 17, 40), seed=0, append=False,
          shuffle=True, spare=2, max_blocks=None, layers=1, vocab=0):
    ctx = np.asarray(ctx, np.int64)
    assert len(ctx) == B
    return workloads.build("test", B=B, T=T, N=N, K=K, H=H, dtype=dtype, ctx=ctx, seed=seed,
                           layers=layers, shuffle=shuffle, append=append, spare_blocks=spare,
                           max_blocks=max_blocks, vocab=vocab)


def slot(w, b, pos):
    """(physical block, row) of logical position pos of sequence b."""
    return int(w.block_tables[b, pos // w.block_size]), pos % w.block_size


def unpage(w, b, n_tokens, layer=0):
    """Contiguous K, V [n_tokens, K, H] float64 of sequence b (test-side gather)."""
    kc, vc = w.k_cache[layer], w.v_cache[layer]
    ks, vs = [], []
    for pos in range(n_tokens):
        blk, r = slot(w, b, pos)
        ks.append(kc[blk, r].double())
        vs.append(vc[blk, r].double())
    return torch.stack(ks).numpy(), torch.stack(vs).numpy()


def set_token(w, b, pos, k=None, v=None, layer=0):
    blk, r = slot(w, b, pos)
    if k is not None:
        w.k_cache[layer][blk, r] = torch.as_tensor(k, dtype=w.torch_dtype)
    if v is not None:
        w.v_cache[layer][blk, r] = torch.as_tensor(v, dtype=w.torch_dtype)


def to(w, device):
    """Copy of a workload's tensors on `device` (same object type)."""
    import copy

    w2 = copy.copy(w)
    w2.context_lens = w.context_lens.to(device)
    w2.block_tables = w.block_tables.to(device)
    for name in ("q", "k_cache", "v_cache", "k_new", "v_new"):
        setattr(w2, name, [t.to(device) for t in getattr(w, name)])
    if w.logits is not None:
        w2.logits = w.logits.to(device)
        w2.draft = w.draft.to(device)
    return w2


def ulp(ref: np.ndarray, dtype: str) -> np.ndarray:
    """One unit in the last place of |ref| in the output dtype.  The parity bar
    is max(tol, one ulp): where the dtype's spacing is wider than the tolerance
    (bf16 from |x| = 2, fp16 from 4) a result whose arithmetic is within the
    tolerance can still round to the far neighbour of the exact value, so
    there the bar is a faithfully rounded output."""
    mant = 10 if dtype == "f16" else 7
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -14 if dtype == "f16" else -126)
    return np.exp2(e - mant)


TOL = {"f16": 2e-3, "bf16": 1e-2}


def assert_close(gpu: np.ndarray, ref: np.ndarray, dtype: str, what=""):
    """|gpu - ref| <= max(tol, one ulp of ref in the output dtype)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.isfinite(ref).all(), f"{what}: oracle produced non-finite values"
    bad_nan = ~np.isfinite(gpu)
    assert not bad_nan.any(), f"{what}: {bad_nan.sum()} non-finite GPU outputs"
    err = np.abs(gpu - ref)
    lim = np.maximum(TOL[dtype], ulp(ref, dtype))
    worst = float(err.max()) if err.size else 0.0
    assert (err <= lim).all(), (
        f"{what}: max |err| {worst:.3g} > tol {TOL[dtype]} at "
        f"{np.unravel_index(int(np.argmax(err - lim)), err.shape)}")
    return worst


def planted_tree_inputs(B, T, V, parents, rng, p_match=0.6):
    """Random logits and drafts where an edge agrees with the target with
    probability p_match (the parent's planted choice is reused as the child's
    token).  Returns logits [B,T,V] float32 and draft [B,T-1] int32."""
    lg = rng.normal(size=(B, T, V)).astype(np.float32)
    choice = rng.integers(0, V, size=(B, T))
    for b in range(B):
        for i in range(T):
            lg[b, i, choice[b, i]] = 10.0
    draft = rng.integers(0, V, size=(B, max(T - 1, 0))).astype(np.int32)
    for b in range(B):
        for c in range(1, T):
            if rng.random() < p_match:
                draft[b, c - 1] = choice[b, parents[b, c]]
    return lg, draft


def random_parents(B, T, rng, chain_bias=0.0):
    """int32 [B,T] random draft trees in topological order (parents[0] = -1,
    parents[i] < i); chain_bias: chance that a node continues the chain."""
    par = np.zeros((B, T), np.int32)
    par[:, 0] = -1
    for b in range(B):
        for i in range(1, T):
            par[b, i] = i - 1 if rng.random() < chain_bias else rng.integers(0, i)
    return par
