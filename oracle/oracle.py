"""ctypes front end of oracle.c (fp64 CPU oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).  Arrays are numpy; 16-bit
elements travel as their raw uint16 bit patterns, so the C side widens them to
double itself.  `dtype` is "f16" or "bf16".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_DT = {"f16": 0, "bf16": 1}


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (OpenMP when the compiler has it)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c99", "-shared", "-fPIC", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _get():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i = ctypes.c_int
            lib.oracle_f16_to_f64.restype = ctypes.c_double
            lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f64.restype = ctypes.c_double
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_kv_append.restype = i
            lib.oracle_kv_append.argtypes = [i] * 7 + [P] * 7
            lib.oracle_attention.restype = i
            lib.oracle_attention.argtypes = ([i] * 9 + [ctypes.c_double, i, P, i] + [P] * 8
                                             + [i, P, P, i])
            lib.oracle_quantize_row.restype = None
            lib.oracle_quantize_row.argtypes = [P, i, i, i, P, P]
            lib.oracle_kv_append_quant.restype = i
            lib.oracle_kv_append_quant.argtypes = [i] * 9 + [P] * 8 + [P]
            lib.oracle_quantize_rows.restype = None
            lib.oracle_quantize_rows.argtypes = [P, i, i, i, i, P, P]
            lib.oracle_e4m3_to_f64.restype = ctypes.c_double
            lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
            lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
            lib.oracle_accept_prefix.restype = None
            lib.oracle_accept_prefix.argtypes = [i, i, i, P, P, P, P, P]
            lib.oracle_accept_sampled.restype = None
            lib.oracle_accept_sampled.argtypes = [i, i, i] + [P] * 8
            lib.oracle_accept_tree.restype = None
            lib.oracle_accept_tree.argtypes = [i, i, i] + [P] * 8
            lib.oracle_kv_compact.restype = i
            lib.oracle_kv_compact.argtypes = [i] * 8 + [P] * 9
            lib.oracle_argmax.restype = i
            lib.oracle_argmax.argtypes = [P, i]
            lib.oracle_num_threads.restype = i
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _bits(a) -> np.ndarray:
    """Raw 16-bit patterns of an fp16/bf16 array (numpy uint16 or float16, or a
    torch CPU tensor)."""
    if hasattr(a, "detach"):  # torch tensor
        import torch

        t = a.detach().cpu().contiguous()
        if t.dtype in (torch.float16, torch.bfloat16):
            t = t.view(torch.int16)
        return t.numpy().view(np.uint16)
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    assert a.dtype in (np.uint16, np.int16), a.dtype
    return a.view(np.uint16)


def _i32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def f16_to_f64(bits: int) -> float:
    return _get().oracle_f16_to_f64(int(bits))


def bf16_to_f64(bits: int) -> float:
    return _get().oracle_bf16_to_f64(int(bits))


def num_threads() -> int:
    return _get().oracle_num_threads()


def kv_append(k_new, v_new, k_cache, v_cache, block_tables, context_lens):
    """Writes k_new/v_new [B,T,K,H] into copies of the caches [NB,bs,K,H].
    Returns (k_cache', v_cache', seq_err[B]) as uint16 bit arrays."""
    kn, vn = _bits(k_new), _bits(v_new)
    kc, vc = _bits(k_cache).copy(), _bits(v_cache).copy()
    bt, cl = _i32(block_tables), _i32(context_lens)
    B, T, K, H = kn.shape
    NB, bs = kc.shape[0], kc.shape[1]
    err = np.zeros(B, np.int32)
    _get().oracle_kv_append(B, T, K, H, bs, NB, bt.shape[1], _p(kn), _p(vn), _p(kc),
                            _p(vc), _p(bt), _p(cl), _p(err))
    return kc, vc, err


KV_KINDS = {"int8": 1, "e4m3": 2}


def attention(q, k_cache, v_cache, block_tables, context_lens, dtype, scale=0.0,
              b_list=None, nthreads=0, window=0, tree_mask=None, kv=None, k_scale=None,
              v_scale=None):
    """fp64 paged GQA attention.  q [B,T,N,H]; caches [NB,bs,K,H]; window > 0
    limits query position i to positions i-window+1 .. i; tree_mask [B,T]
    (uint64) lets new token t see new token j < t only if bit j is set.
    kv = "int8" / "e4m3": the caches hold one-byte codes (uint8 [NB,bs,K,H]) and
    k_scale / v_scale fp32 [NB,K,bs] their row scales.
    Returns (out [nb,T,N,H] float64, seq_err [nb]) for the listed sequences."""
    qb = _bits(q)
    if kv is None:
        kc, vc = _bits(k_cache), _bits(v_cache)
        ks = vs = None
    else:
        kc = np.ascontiguousarray(_u8(k_cache))
        vc = np.ascontiguousarray(_u8(v_cache))
        ks = np.ascontiguousarray(_f32(k_scale))
        vs = np.ascontiguousarray(_f32(v_scale))
    bt, cl = _i32(block_tables), _i32(context_lens)
    B, T, N, H = qb.shape
    NB, bs, K, H2 = kc.shape
    assert H2 == H
    bl = None if b_list is None else _i32(b_list)
    nb = B if bl is None else len(bl)
    out = np.zeros((nb, T, N, H), np.float64)
    err = np.zeros(max(nb, 1), np.int32)
    tm = None
    if tree_mask is not None:
        tm = np.ascontiguousarray(np.asarray(tree_mask).astype(np.uint64)).reshape(B, T)
    rc = _get().oracle_attention(B, T, N, K, H, bs, NB, bt.shape[1], _DT[dtype],
                                 float(scale), int(window), _p(tm),
                                 0 if kv is None else KV_KINDS[kv], _p(ks), _p(vs), _p(qb),
                                 _p(kc), _p(vc), _p(bt), _p(cl),
                                 _p(bl), nb, _p(out), _p(err), int(nthreads))
    if rc < 0:
        raise ValueError("oracle_attention: N must be a multiple of K, window >= 0, and a "
                         "tree mask needs window == 0 and T <= 64")
    return out, err[:nb]


def accept_prefix(logits, draft, context_lens=None):
    """Greedy acceptance.  logits [B,T,V] float32, draft [B,T-1] int32.
    Returns (accepted [B], next_token [B], context_lens' or None)."""
    if hasattr(logits, "detach"):
        logits = logits.detach().cpu().numpy()
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    B, T, V = lg.shape
    dr = _i32(draft).reshape(B, max(T - 1, 0))
    acc = np.zeros(B, np.int32)
    nxt = np.zeros(B, np.int32)
    cl = None if context_lens is None else _i32(context_lens).copy()
    _get().oracle_accept_prefix(B, T, V, _p(lg), _p(dr), _p(acc), _p(nxt), _p(cl))
    return acc, nxt, cl


def _u8(a):
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.asarray(a).view(np.uint8) if np.asarray(a).dtype == np.int8 else np.asarray(
        a, dtype=np.uint8)


def _f32(a):
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.asarray(a, dtype=np.float32)


def quantize_row(x, dtype, kv):
    """One-byte codes (uint8) and the fp32 scale of one fp16/bf16 row."""
    xb = np.ascontiguousarray(_bits(x)).reshape(-1)
    codes = np.zeros(xb.size, np.uint8)
    sc = np.zeros(1, np.float32)
    _get().oracle_quantize_row(_p(xb), xb.size, _DT[dtype], KV_KINDS[kv], _p(codes), _p(sc))
    return codes, float(sc[0])


def quantize_cache(cache, dtype, kv):
    """Quantize every row of a cache [NB,bs,K,H] (fp16/bf16): codes uint8
    [NB,bs,K,H] and scales fp32 [NB,K,bs]."""
    cb = _bits(cache)
    NB, bs, K, H = cb.shape
    flat = np.ascontiguousarray(cb.reshape(-1, H))
    codes = np.zeros(flat.shape, np.uint8)
    scales = np.zeros(flat.shape[0], np.float32)
    _get().oracle_quantize_rows(_p(flat), flat.shape[0], H, _DT[dtype], KV_KINDS[kv],
                                _p(codes), _p(scales))
    return (codes.reshape(NB, bs, K, H),
            np.ascontiguousarray(scales.reshape(NB, bs, K).transpose(0, 2, 1)))


def e4m3_to_f64(code: int) -> float:
    return _get().oracle_e4m3_to_f64(int(code))


def e4m3_from_float(x: float) -> int:
    return int(_get().oracle_e4m3_from_float(float(x)))


def kv_append_quant(k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_tables,
                    context_lens, dtype, kv):
    """Quantized append into copies of the one-byte caches uint8 [NB,bs,K,H] and
    their scales fp32 [NB,K,bs].  Returns (k_cache', v_cache', k_scale',
    v_scale', seq_err)."""
    kn, vn = _bits(k_new), _bits(v_new)
    kc, vc = _u8(k_cache).copy(), _u8(v_cache).copy()
    ks, vs = _f32(k_scale).copy(), _f32(v_scale).copy()
    bt, cl = _i32(block_tables), _i32(context_lens)
    B, T, K, H = kn.shape
    NB, bs = kc.shape[0], kc.shape[1]
    err = np.zeros(max(B, 1), np.int32)
    _get().oracle_kv_append_quant(B, T, K, H, bs, NB, bt.shape[1], _DT[dtype], KV_KINDS[kv],
                                  _p(kn), _p(vn), _p(kc), _p(vc), _p(ks), _p(vs), _p(bt),
                                  _p(cl), _p(err))
    return kc, vc, ks, vs, err[:B]


def accept_sampled(q, p, draft, u, context_lens=None):
    """Speculative sampling (stochastic acceptance).  q [B,T,V] float32 target
    probabilities, p [B,T-1,V] float32 draft probabilities, draft [B,T-1]
    int32, u [B,T] float64 uniforms in [0,1).  Returns (accepted [B],
    next_token [B], context_lens' or None, seq_err [B])."""
    qa = np.ascontiguousarray(q, dtype=np.float32)
    B, T, V = qa.shape
    if not 1 <= T <= 64:
        raise ValueError("accept_sampled: T must be in [1, 64]")
    pa = np.ascontiguousarray(p, dtype=np.float32).reshape(B, T - 1, V)
    dr = _i32(draft).reshape(B, T - 1)
    ua = np.ascontiguousarray(u, dtype=np.float64).reshape(B, T)
    acc = np.zeros(B, np.int32)
    nxt = np.zeros(B, np.int32)
    err = np.zeros(max(B, 1), np.int32)
    cl = None if context_lens is None else _i32(context_lens).copy()
    _get().oracle_accept_sampled(B, T, V, _p(qa), _p(pa), _p(dr), _p(ua), _p(acc), _p(nxt),
                                 _p(cl), _p(err))
    return acc, nxt, cl, err[:B]


def accept_tree(logits, draft, parents, context_lens=None):
    """Greedy acceptance over a draft tree.  logits [B,T,V] float32 (row i: the
    target's prediction after the root-to-node-i path), draft [B,T-1] int32
    (node i's token at column i-1), parents [B,T] int32 (-1 for node 0, then a
    parent index below the node's own).  Returns (accepted [B], next_token [B],
    path [B,T-1] (accepted nodes by depth, then -1), context_lens' or None,
    seq_err [B])."""
    if hasattr(logits, "detach"):
        logits = logits.detach().cpu().numpy()
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    B, T, V = lg.shape
    if not 1 <= T <= 64:
        raise ValueError("accept_tree: T must be in [1, 64]")
    dr = np.ascontiguousarray(_i32(draft).reshape(B, T - 1))
    par = np.ascontiguousarray(_i32(parents).reshape(B, T))
    acc = np.zeros(B, np.int32)
    nxt = np.zeros(B, np.int32)
    path = np.full((B, max(T - 1, 0)), -1, np.int32)
    err = np.zeros(max(B, 1), np.int32)
    cl = None if context_lens is None else _i32(context_lens).copy()
    _get().oracle_accept_tree(B, T, V, _p(lg), _p(dr), _p(par), _p(acc), _p(nxt), _p(path),
                              _p(cl), _p(err))
    return acc, nxt, path, cl, err[:B]


def kv_compact(k_cache, v_cache, block_tables, context_lens, path, accepted, T,
               k_scale=None, v_scale=None):
    """Cache compaction after tree acceptance, on copies: position base+j
    (j = 1..a, base = context_lens[b] - 1 - a) takes the rows of node
    path[b][j-1].  Caches [NB,bs,K,H] of 16-bit elements (numpy uint16/float16
    or torch fp16/bf16) or one-byte codes (uint8/int8, with k_scale / v_scale
    fp32 [NB,K,bs]).  Returns (k_cache', v_cache', k_scale', v_scale', seq_err)."""
    one_byte = k_scale is not None
    if one_byte:
        kc, vc = _u8(k_cache).copy(), _u8(v_cache).copy()
        ks, vs = _f32(k_scale).copy(), _f32(v_scale).copy()
        raw_k, raw_v = kc, vc
    else:
        kc, vc = _bits(k_cache).copy(), _bits(v_cache).copy()
        ks = vs = None
        raw_k, raw_v = kc.view(np.uint8), vc.view(np.uint8)
    NB, bs, K, H = kc.shape
    bt, cl = _i32(block_tables), _i32(context_lens)
    B = bt.shape[0]
    pt = np.ascontiguousarray(_i32(path).reshape(B, max(T - 1, 0)))
    ac = _i32(accepted).reshape(B)
    err = np.zeros(max(B, 1), np.int32)
    rc = _get().oracle_kv_compact(B, T, K, H, bs, NB, bt.shape[1], 1 if one_byte else 2,
                                  _p(raw_k), _p(raw_v), _p(ks), _p(vs), _p(bt), _p(cl), _p(pt),
                                  _p(ac), _p(err))
    if rc != 0:
        raise MemoryError("oracle_kv_compact")
    return kc, vc, ks, vs, err[:B]


def argmax(row) -> int:
    r = np.ascontiguousarray(row, dtype=np.float32)
    return _get().oracle_argmax(_p(r), r.shape[0])
