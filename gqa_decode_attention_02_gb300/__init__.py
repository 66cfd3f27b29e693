"""Paged grouped-query decode attention for GB300 (sm_103a).

Python face of the C ABI in include/gqa_decode.h: same operation names, torch
tensors in, argument marshalling only.  All computation runs in the library's
CUDA kernels; calling any op without the built library raises.

    kv_append(k_new, v_new, k_cache, v_cache, block_tables, context_lens)
    decode_attention(q, k_cache, v_cache, block_tables, context_lens) -> out
    verify_attention(q, k_cache, v_cache, block_tables, context_lens) -> out
    append_decode_attention(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens)
    append_verify_attention(...)  (kv_append fused into the attention launch)
    (every attention call takes window=W > 0 for local attention)
    kv_append_quant / decode_attention_quant / verify_attention_quant: the same
    over a one-byte (int8 or e4m3) cache with per-row fp32 scales
    accept_prefix(target_logits, draft_ids, context_lens=None) -> (accepted, next)
    accept_sampled(target_probs, draft_probs, draft_ids, uniforms,
                   context_lens=None) -> (accepted, next)
    accept_tree(target_logits, draft_ids, parents, context_lens=None)
        -> (accepted, next, path); then kv_compact(k_cache, v_cache, block_tables,
        context_lens, path, accepted) moves the accepted branch's cached rows
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import GqaError, Shape, Status, status_string  # noqa: F401

__all__ = ["kv_append", "kv_append_quant", "decode_attention", "verify_attention",
           "decode_attention_quant", "verify_attention_quant", "append_decode_attention_quant",
           "append_verify_attention_quant", "append_decode_attention",
           "append_verify_attention", "accept_prefix", "accept_sampled", "accept_tree",
           "kv_compact",
           "attention_workspace_size", "reset_workspaces", "GqaError", "Status", "Shape"]


def reset_workspaces():
    """Drop the workspaces the binding caches per (device, stream); see
    _lib.reset_workspaces."""
    _lib.reset_workspaces()


def _status_arg(status):
    if status is None:
        return None
    _lib._need(status, "status", torch.int32)
    return _lib._ptr(status)


def kv_append(k_new, v_new, k_cache, v_cache, block_tables, context_lens, *, status=None,
              stream=None, pdl=False):
    """gqa_kv_append: k_new/v_new [B,T,K,H] -> caches [NB,16,K,H] at positions
    context_lens[b]-T+t.  Asynchronous on `stream` (default: current).
    pdl: launch with programmatic dependent launch (GQA_FLAG_PDL)."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _lib._need(t, n, ndim=4)
    _lib._need(block_tables, "block_tables", torch.int32, 2)
    _lib._need(context_lens, "context_lens", torch.int32, 1)
    shape = _lib.make_shape(k_new, k_cache, block_tables, None, heads_dim=3,
                            flags=_lib.FLAG_PDL if pdl else 0)
    rc = _lib.lib().gqa_kv_append(ctypes.byref(shape), _lib._ptr(k_new), _lib._ptr(v_new),
                                  _lib._ptr(k_cache), _lib._ptr(v_cache),
                                  _lib._ptr(block_tables), _lib._ptr(context_lens),
                                  _status_arg(status), _lib._stream(stream))
    _lib._check("gqa_kv_append", rc)


_BYTE_DTYPES = (torch.uint8, torch.int8, torch.float8_e4m3fn)


def _need_quant_cache(cache, scale, name):
    if not isinstance(cache, torch.Tensor) or cache.dtype not in _BYTE_DTYPES:
        raise ValueError(f"{name} must be a one-byte tensor (uint8 / int8 / float8_e4m3fn)")
    _lib._need(cache, name, ndim=4)
    _lib._need(scale, name + " scale", torch.float32, 3)
    NB, bs, K, _ = cache.shape
    if tuple(scale.shape) != (NB, K, bs):
        raise ValueError(f"{name} scale must be [{NB},{K},{bs}], got {tuple(scale.shape)}")


def kv_append_quant(k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_tables,
                    context_lens, *, kv="int8", status=None, stream=None, pdl=False):
    """gqa_kv_append_quant: quantize k_new / v_new [B,T,K,H] (fp16 / bf16) row
    by row into one-byte caches [NB,16,K,H] and their scales fp32 [NB,K,16]."""
    _lib._need(k_new, "k_new", ndim=4)
    _lib._need(v_new, "v_new", k_new.dtype, 4)
    _need_quant_cache(k_cache, k_scale, "k_cache")
    _need_quant_cache(v_cache, v_scale, "v_cache")
    _lib._need(block_tables, "block_tables", torch.int32, 2)
    _lib._need(context_lens, "context_lens", torch.int32, 1)
    shape = _lib.make_shape(k_new, k_cache, block_tables, None, heads_dim=3,
                            flags=_lib.FLAG_PDL if pdl else 0, kv=kv)
    rc = _lib.lib().gqa_kv_append_quant(ctypes.byref(shape), _lib._ptr(k_new),
                                        _lib._ptr(v_new), _lib._ptr(k_cache),
                                        _lib._ptr(v_cache), _lib._ptr(k_scale),
                                        _lib._ptr(v_scale), _lib._ptr(block_tables),
                                        _lib._ptr(context_lens), _status_arg(status),
                                        _lib._stream(stream))
    _lib._check("gqa_kv_append_quant", rc)


def attention_engine(q, k_cache, block_tables, window=0, engine="auto") -> str:
    """Which kernel serves an attention call of this shape: "warp" (the
    persistent mma.sync kernel), "direct" (mma.sync, one CTA per sequence and
    KV head) or "tmem" (tcgen05 with tensor-memory accumulators);
    gqa_attention_engine.  Host logic only, for a call without a tree mask (a
    tree mask rules "direct" out)."""
    if engine not in _lib.ENGINES:
        raise ValueError(f"engine must be one of {sorted(_lib.ENGINES)}, got {engine!r}")
    shape = _lib.make_shape(q, k_cache, block_tables, None, window=window,
                            flags=_lib.ENGINES[engine])
    e = _lib.lib().gqa_attention_engine(ctypes.byref(shape))
    if e == 0:
        raise _lib.GqaError("gqa_attention_engine", _lib.Status.ERR_SHAPE)
    return _lib.ENGINE_NAMES[e]


def attention_workspace_size(q, k_cache, block_tables, scale=None, window=0) -> int:
    """Workspace bytes of one attention call (a window never needs more than
    full attention of the same shape)."""
    return _lib.workspace_size(_lib.make_shape(q, k_cache, block_tables, scale, window=window))


def _attention(fn_name, q, k_cache, v_cache, block_tables, context_lens, out, scale,
               workspace, status, stream, pdl, early_kv, k_new=None, v_new=None, window=0,
               tree_mask=None, engine="auto"):
    _lib._need(q, "q", ndim=4)
    if engine not in _lib.ENGINES:
        raise ValueError(f"engine must be one of {sorted(_lib.ENGINES)}, got {engine!r}")
    if tree_mask is not None:
        _lib._need(tree_mask, "tree_mask", torch.int64, 2)  # uint64 bits, held as int64
        if tuple(tree_mask.shape) != tuple(q.shape[:2]):
            raise ValueError(f"tree_mask must be [B,T] = {tuple(q.shape[:2])}")
        fn_name = fn_name.replace("verify_attention", "tree_verify_attention")
    if k_new is not None:
        _lib._need(k_new, "k_new", q.dtype, 4)
        _lib._need(v_new, "v_new", q.dtype, 4)
    _lib._need(k_cache, "k_cache", q.dtype, 4)
    _lib._need(v_cache, "v_cache", q.dtype, 4)
    _lib._need(block_tables, "block_tables", torch.int32, 2)
    _lib._need(context_lens, "context_lens", torch.int32, 1)
    flags = ((_lib.FLAG_PDL if pdl else 0) | (_lib.FLAG_EARLY_KV if early_kv else 0)
             | _lib.ENGINES[engine])
    shape = _lib.make_shape(q, k_cache, block_tables, scale, flags=flags, window=window)
    if out is None:
        out = torch.empty_like(q)
    else:
        _lib._need(out, "out", q.dtype, 4)
    nbytes = _lib.workspace_size(shape)
    if workspace is None:
        workspace = _lib.get_workspace(nbytes, q.device, stream)
    else:
        _lib._need(workspace, "workspace", torch.uint8)
    L = _lib.lib()
    new = () if k_new is None else (_lib._ptr(k_new), _lib._ptr(v_new))
    mask = () if tree_mask is None else (_lib._ptr(tree_mask),)
    rc = getattr(L, fn_name)(ctypes.byref(shape), _lib._ptr(q), *new, _lib._ptr(k_cache),
                             _lib._ptr(v_cache), _lib._ptr(block_tables),
                             _lib._ptr(context_lens), *mask, _lib._ptr(out),
                             _lib._ptr(workspace), workspace.numel(), _status_arg(status),
                             _lib._stream(stream))
    _lib._check(fn_name, rc)
    return out


def decode_attention(q, k_cache, v_cache, block_tables, context_lens, *, out=None, scale=None,
                     workspace=None, status=None, stream=None, pdl=False, early_kv=False,
                     window=0, engine="auto"):
    """gqa_decode_attention (T == 1).  q [B,1,N,H] -> out [B,1,N,H].
    pdl / early_kv select GQA_FLAG_PDL / GQA_FLAG_EARLY_KV (see the C header);
    window > 0 is local attention over each query's last `window` positions;
    engine "warp" / "direct" / "tmem" forces the persistent mma.sync, the
    direct mma.sync or the tcgen05 kernel ("auto": by shape; GQA_FLAG_WARP_MMA
    / GQA_FLAG_DIRECT / GQA_FLAG_TENSOR_MEMORY)."""
    return _attention("gqa_decode_attention", q, k_cache, v_cache, block_tables, context_lens,
                      out, scale, workspace, status, stream, pdl, early_kv, window=window,
                      engine=engine)


def verify_attention(q, k_cache, v_cache, block_tables, context_lens, *, out=None, scale=None,
                     workspace=None, status=None, stream=None, pdl=False, early_kv=False,
                     window=0, tree_mask=None, engine="auto"):
    """gqa_verify_attention (T >= 1, causal among the T new tokens), or with
    tree_mask (int64 [B,T] holding the uint64 mask rows)
    gqa_tree_verify_attention."""
    return _attention("gqa_verify_attention", q, k_cache, v_cache, block_tables, context_lens,
                      out, scale, workspace, status, stream, pdl, early_kv, window=window,
                      tree_mask=tree_mask, engine=engine)


def append_decode_attention(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, *,
                            out=None, scale=None, workspace=None, status=None, stream=None,
                            pdl=False, early_kv=False, window=0, engine="auto"):
    """gqa_append_decode_attention: kv_append + decode_attention in one launch
    (T == 1).  Writes k_new/v_new into the caches and returns out."""
    return _attention("gqa_append_decode_attention", q, k_cache, v_cache, block_tables,
                      context_lens, out, scale, workspace, status, stream, pdl, early_kv,
                      k_new=k_new, v_new=v_new, window=window, engine=engine)


def append_verify_attention(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, *,
                            out=None, scale=None, workspace=None, status=None, stream=None,
                            pdl=False, early_kv=False, window=0, tree_mask=None,
                            engine="auto"):
    """gqa_append_verify_attention: kv_append + verify_attention in one launch
    (gqa_append_tree_verify_attention with tree_mask; with the tensor-memory
    kernel the append is a launch of its own just before)."""
    return _attention("gqa_append_verify_attention", q, k_cache, v_cache, block_tables,
                      context_lens, out, scale, workspace, status, stream, pdl, early_kv,
                      k_new=k_new, v_new=v_new, window=window, tree_mask=tree_mask,
                      engine=engine)


def _attention_quant(fn_name, q, k_cache, v_cache, k_scale, v_scale, block_tables,
                     context_lens, out, scale, workspace, status, stream, pdl, early_kv, kv,
                     window=0, tree_mask=None):
    _lib._need(q, "q", ndim=4)
    if tree_mask is not None:
        _lib._need(tree_mask, "tree_mask", torch.int64, 2)  # uint64 bits, held as int64
        if tuple(tree_mask.shape) != tuple(q.shape[:2]):
            raise ValueError(f"tree_mask must be [B,T] = {tuple(q.shape[:2])}")
        fn_name = "gqa_tree_verify_attention_quant"
    _need_quant_cache(k_cache, k_scale, "k_cache")
    _need_quant_cache(v_cache, v_scale, "v_cache")
    _lib._need(block_tables, "block_tables", torch.int32, 2)
    _lib._need(context_lens, "context_lens", torch.int32, 1)
    flags = (_lib.FLAG_PDL if pdl else 0) | (_lib.FLAG_EARLY_KV if early_kv else 0)
    shape = _lib.make_shape(q, k_cache, block_tables, scale, flags=flags, window=window, kv=kv)
    if out is None:
        out = torch.empty_like(q)
    else:
        _lib._need(out, "out", q.dtype, 4)
    nbytes = _lib.workspace_size(shape)
    if workspace is None:
        workspace = _lib.get_workspace(nbytes, q.device, stream)
    else:
        _lib._need(workspace, "workspace", torch.uint8)
    mask = () if tree_mask is None else (_lib._ptr(tree_mask),)
    rc = getattr(_lib.lib(), fn_name)(ctypes.byref(shape), _lib._ptr(q), _lib._ptr(k_cache),
                                      _lib._ptr(v_cache), _lib._ptr(k_scale),
                                      _lib._ptr(v_scale), _lib._ptr(block_tables),
                                      _lib._ptr(context_lens), *mask, _lib._ptr(out),
                                      _lib._ptr(workspace), workspace.numel(),
                                      _status_arg(status), _lib._stream(stream))
    _lib._check(fn_name, rc)
    return out


def decode_attention_quant(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                           *, kv="int8", out=None, scale=None, workspace=None, status=None,
                           stream=None, pdl=False, early_kv=False, window=0):
    """gqa_decode_attention_quant over a one-byte cache (kv = "int8" / "e4m3");
    window > 0 is local attention as in decode_attention."""
    return _attention_quant("gqa_decode_attention_quant", q, k_cache, v_cache, k_scale, v_scale,
                            block_tables, context_lens, out, scale, workspace, status, stream,
                            pdl, early_kv, kv, window)


def verify_attention_quant(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                           *, kv="int8", out=None, scale=None, workspace=None, status=None,
                           stream=None, pdl=False, early_kv=False, window=0, tree_mask=None):
    """gqa_verify_attention_quant over a one-byte cache (kv = "int8" / "e4m3");
    window > 0 is local attention and tree_mask (int64 [B,T] holding the uint64
    mask rows) tree verification, as in verify_attention
    (gqa_tree_verify_attention_quant)."""
    return _attention_quant("gqa_verify_attention_quant", q, k_cache, v_cache, k_scale, v_scale,
                            block_tables, context_lens, out, scale, workspace, status, stream,
                            pdl, early_kv, kv, window, tree_mask)


def _append_attention_quant(fn_name, q, k_new, v_new, k_cache, v_cache, k_scale, v_scale,
                            block_tables, context_lens, out, scale, workspace, status, stream,
                            pdl, early_kv, kv, window):
    _lib._need(q, "q", ndim=4)
    _lib._need(k_new, "k_new", q.dtype, 4)
    _lib._need(v_new, "v_new", q.dtype, 4)
    _need_quant_cache(k_cache, k_scale, "k_cache")
    _need_quant_cache(v_cache, v_scale, "v_cache")
    _lib._need(block_tables, "block_tables", torch.int32, 2)
    _lib._need(context_lens, "context_lens", torch.int32, 1)
    flags = (_lib.FLAG_PDL if pdl else 0) | (_lib.FLAG_EARLY_KV if early_kv else 0)
    shape = _lib.make_shape(q, k_cache, block_tables, scale, flags=flags, window=window, kv=kv)
    if out is None:
        out = torch.empty_like(q)
    else:
        _lib._need(out, "out", q.dtype, 4)
    nbytes = _lib.workspace_size(shape)
    if workspace is None:
        workspace = _lib.get_workspace(nbytes, q.device, stream)
    else:
        _lib._need(workspace, "workspace", torch.uint8)
    P = _lib._ptr
    rc = getattr(_lib.lib(), fn_name)(ctypes.byref(shape), P(q), P(k_new), P(v_new),
                                      P(k_cache), P(v_cache), P(k_scale), P(v_scale),
                                      P(block_tables), P(context_lens), P(out), P(workspace),
                                      workspace.numel(), _status_arg(status),
                                      _lib._stream(stream))
    _lib._check(fn_name, rc)
    return out


def append_decode_attention_quant(q, k_new, v_new, k_cache, v_cache, k_scale, v_scale,
                                  block_tables, context_lens, *, kv="int8", out=None,
                                  scale=None, workspace=None, status=None, stream=None,
                                  pdl=False, early_kv=False, window=0):
    """gqa_append_decode_attention_quant: kv_append_quant of the new token and
    decode attention over the one-byte cache in one call (two launches; the
    caches and their scales are written)."""
    return _append_attention_quant("gqa_append_decode_attention_quant", q, k_new, v_new,
                                   k_cache, v_cache, k_scale, v_scale, block_tables,
                                   context_lens, out, scale, workspace, status, stream, pdl,
                                   early_kv, kv, window)


def append_verify_attention_quant(q, k_new, v_new, k_cache, v_cache, k_scale, v_scale,
                                  block_tables, context_lens, *, kv="int8", out=None,
                                  scale=None, workspace=None, status=None, stream=None,
                                  pdl=False, early_kv=False, window=0):
    """gqa_append_verify_attention_quant: the T new tokens appended to the
    one-byte cache and verify attention over it, in one call (two launches)."""
    return _append_attention_quant("gqa_append_verify_attention_quant", q, k_new, v_new,
                                   k_cache, v_cache, k_scale, v_scale, block_tables,
                                   context_lens, out, scale, workspace, status, stream, pdl,
                                   early_kv, kv, window)


def accept_prefix(target_logits, draft_ids, context_lens=None, *, accepted=None,
                  next_token=None, status=None, stream=None, workspace=None, cluster=False):
    """gqa_accept_prefix.  target_logits fp32 [B,T,V], draft_ids int32 [B,T-1].
    Returns (accepted [B], next_token [B]); updates context_lens in place if given.
    workspace: uint8 device tensor of at least gqa_accept_workspace_size(B, T)
    bytes (default: one cached per stream); cluster=True passes no workspace
    (one thread-block cluster per sequence)."""
    _lib._need(target_logits, "target_logits", torch.float32, 3)
    B, T, V = target_logits.shape
    if T > 1:
        _lib._need(draft_ids, "draft_ids", torch.int32, 2)
    if context_lens is not None:
        _lib._need(context_lens, "context_lens", torch.int32, 1)
    dev = target_logits.device
    if accepted is None:
        accepted = torch.empty(B, dtype=torch.int32, device=dev)
    if next_token is None:
        next_token = torch.empty(B, dtype=torch.int32, device=dev)
    L = _lib.lib()
    if cluster:
        workspace = None
    elif workspace is None:
        workspace = _lib.get_workspace(L.gqa_accept_workspace_size(B, T), dev, stream,
                                       kind="accept")
    else:
        _lib._need(workspace, "workspace", torch.uint8)
    rc = L.gqa_accept_prefix(B, T, V, _lib._ptr(target_logits),
                             _lib._ptr(draft_ids) if T > 1 else None,
                             _lib._ptr(accepted), _lib._ptr(next_token),
                             _lib._ptr(context_lens), _lib._ptr(workspace),
                             0 if workspace is None else workspace.numel(),
                             _status_arg(status), _lib._stream(stream))
    _lib._check("gqa_accept_prefix", rc)
    return accepted, next_token


def accept_tree(target_logits, draft_ids, parents, context_lens=None, *, accepted=None,
                next_token=None, path=None, status=None, stream=None, workspace=None,
                cluster=False):
    """gqa_accept_tree: greedy acceptance over a draft tree.  target_logits fp32
    [B,T,V] (row i: the target's prediction after node i's branch), draft_ids
    int32 [B,T-1] (node i's token at column i-1), parents int32 [B,T] (-1 for
    the root, then an index below the node's own).  Returns (accepted [B],
    next_token [B], path [B,T-1]: the accepted branch's nodes by depth, then
    -1); updates context_lens in place if given.  workspace / cluster as in
    accept_prefix."""
    _lib._need(target_logits, "target_logits", torch.float32, 3)
    B, T, V = target_logits.shape
    _lib._need(parents, "parents", torch.int32, 2)
    if tuple(parents.shape) != (B, T):
        raise ValueError(f"parents must be [{B},{T}], got {tuple(parents.shape)}")
    if T > 1:
        _lib._need(draft_ids, "draft_ids", torch.int32, 2)
        if tuple(draft_ids.shape) != (B, T - 1):
            raise ValueError(f"draft_ids must be [{B},{T - 1}], got {tuple(draft_ids.shape)}")
    if context_lens is not None:
        _lib._need(context_lens, "context_lens", torch.int32, 1)
    dev = target_logits.device
    if accepted is None:
        accepted = torch.empty(B, dtype=torch.int32, device=dev)
    if next_token is None:
        next_token = torch.empty(B, dtype=torch.int32, device=dev)
    if path is None:
        path = torch.empty((B, max(T - 1, 0)), dtype=torch.int32, device=dev)
    else:
        _lib._need(path, "path", torch.int32, 2)
        if tuple(path.shape) != (B, max(T - 1, 0)):
            raise ValueError(f"path must be [{B},{max(T - 1, 0)}], got {tuple(path.shape)}")
    L = _lib.lib()
    if cluster:
        workspace = None
    elif workspace is None:
        workspace = _lib.get_workspace(L.gqa_accept_workspace_size(B, T), dev, stream,
                                       kind="accept")
    else:
        _lib._need(workspace, "workspace", torch.uint8)
    rc = L.gqa_accept_tree(B, T, V, _lib._ptr(target_logits),
                           _lib._ptr(draft_ids) if T > 1 else None, _lib._ptr(parents),
                           _lib._ptr(accepted), _lib._ptr(next_token),
                           _lib._ptr(path) if T > 1 else None, _lib._ptr(context_lens),
                           _lib._ptr(workspace), 0 if workspace is None else workspace.numel(),
                           _status_arg(status), _lib._stream(stream))
    _lib._check("gqa_accept_tree", rc)
    return accepted, next_token, path


def kv_compact(k_cache, v_cache, block_tables, context_lens, path, accepted, *, k_scale=None,
               v_scale=None, kv="same", status=None, stream=None, pdl=False):
    """gqa_kv_compact: after accept_tree, position base+j (j = 1..a, base =
    context_lens[b] - 1 - a, context_lens as accept_tree left them) takes the
    cached K and V rows of node path[b][j-1].  Caches [NB,16,K,H] in q's dtype
    (kv="same"), or one-byte caches with their scales fp32 [NB,K,16]
    (kv="int8" / "e4m3").  The tree size T is path.shape[1] + 1."""
    if kv == "same":
        _lib._need(k_cache, "k_cache", ndim=4)
        _lib._need(v_cache, "v_cache", k_cache.dtype, 4)
        if k_cache.dtype not in _lib._DTYPES:
            raise ValueError(f"k_cache dtype {k_cache.dtype} unsupported (fp16 / bf16)")
        dtype = _lib._DTYPES[k_cache.dtype]
    else:
        _need_quant_cache(k_cache, k_scale, "k_cache")
        _need_quant_cache(v_cache, v_scale, "v_cache")
        dtype = 0
    _lib._need(block_tables, "block_tables", torch.int32, 2)
    _lib._need(context_lens, "context_lens", torch.int32, 1)
    _lib._need(path, "path", torch.int32, 2)
    _lib._need(accepted, "accepted", torch.int32, 1)
    NB, bs, K, H = k_cache.shape
    B = block_tables.shape[0]
    if tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache and v_cache must have the same shape")
    if context_lens.shape[0] != B or accepted.shape[0] != B or path.shape[0] != B:
        raise ValueError(f"context_lens, accepted and path must have {B} rows")
    shape = _lib.Shape(B=B, T=path.shape[1] + 1, N=K, K=K, H=H, block_size=bs, num_blocks=NB,
                       max_blocks_per_seq=block_tables.shape[1], dtype=dtype, scale=0.0,
                       flags=_lib.FLAG_PDL if pdl else 0, window=0,
                       kv_dtype=_lib.KV_DTYPES[kv])
    rc = _lib.lib().gqa_kv_compact(ctypes.byref(shape), _lib._ptr(k_cache), _lib._ptr(v_cache),
                                   _lib._ptr(k_scale), _lib._ptr(v_scale),
                                   _lib._ptr(block_tables), _lib._ptr(context_lens),
                                   _lib._ptr(path), _lib._ptr(accepted), _status_arg(status),
                                   _lib._stream(stream))
    _lib._check("gqa_kv_compact", rc)


def accept_sampled(target_probs, draft_probs, draft_ids, uniforms, context_lens=None, *,
                   accepted=None, next_token=None, status=None, stream=None):
    """gqa_accept_sampled.  target_probs fp32 [B,T,V], draft_probs fp32
    [B,T-1,V], draft_ids int32 [B,T-1], uniforms fp64 [B,T] in [0,1).
    Returns (accepted [B], next_token [B]); updates context_lens in place if given."""
    _lib._need(target_probs, "target_probs", torch.float32, 3)
    B, T, V = target_probs.shape
    _lib._need(uniforms, "uniforms", torch.float64, 2)
    if tuple(uniforms.shape) != (B, T):
        raise ValueError(f"uniforms must be [{B},{T}], got {tuple(uniforms.shape)}")
    if T > 1:
        _lib._need(draft_probs, "draft_probs", torch.float32, 3)
        _lib._need(draft_ids, "draft_ids", torch.int32, 2)
        if tuple(draft_probs.shape) != (B, T - 1, V) or tuple(draft_ids.shape) != (B, T - 1):
            raise ValueError("draft_probs must be [B,T-1,V] and draft_ids [B,T-1]")
    if context_lens is not None:
        _lib._need(context_lens, "context_lens", torch.int32, 1)
    dev = target_probs.device
    if accepted is None:
        accepted = torch.empty(B, dtype=torch.int32, device=dev)
    if next_token is None:
        next_token = torch.empty(B, dtype=torch.int32, device=dev)
    rc = _lib.lib().gqa_accept_sampled(B, T, V, _lib._ptr(target_probs),
                                       _lib._ptr(draft_probs) if T > 1 else None,
                                       _lib._ptr(draft_ids) if T > 1 else None,
                                       _lib._ptr(uniforms), _lib._ptr(accepted),
                                       _lib._ptr(next_token), _lib._ptr(context_lens),
                                       _status_arg(status), _lib._stream(stream))
    _lib._check("gqa_accept_sampled", rc)
    return accepted, next_token
