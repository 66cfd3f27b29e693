"""Closed-form byte / flop accounting for the decode path, from the pages'
formulas.  The bench uses `attention_algorithmic_bytes` as the numerator of its
roofline figure; the model-level calculators reproduce the pages' worked tables
(and are pinned to them in tests/golden/page_figures.json).
"""
from __future__ import annotations

import math
from typing import Iterable

import numpy as np


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    """Page "جعل inference رخيصًا: KV cache وbatching والتكميم", KV-cache section:
    each layer keeps one key and one value vector per KV head per token,
    2 * L * K * H * bytes."""
    return 2 * layers * kv_heads * head_dim * elem_bytes


def paged_kv_bytes(tokens: int, layers: int, kv_heads: int, head_dim: int, elem_bytes: int,
                   block_size: int = 16) -> int:
    """Bytes a paged cache reserves for `tokens` tokens: whole blocks (CS336
    lecture 10 §"PagedAttention": internal fragmentation is at most one block)."""
    blocks = -(-tokens // block_size)
    return blocks * block_size * kv_bytes_per_token(layers, kv_heads, head_dim, elem_bytes)


def transformer_params(V: int, D: int, F: int, L: int, N: int, K: int, H: int) -> int:
    """CS336 lecture 10 §"Пропускная способность и задержка": embedding +
    unembedding, 3 MLP matrices and the Q/O and K/V projections per layer."""
    return 2 * V * D + D * F * 3 * L + (2 * D * N * H + 2 * D * K * H) * L


def decode_step_model(B: int, S: int, V: int, D: int, F: int, L: int, N: int, K: int, H: int,
                      bandwidth: float, elem_bytes: int = 2):
    """Same section: memory = B * kv_cache_size + parameter bytes; every decode
    step reads all of it, so latency = memory / bandwidth and throughput =
    B / latency.  Returns (memory bytes, latency s, tokens/s)."""
    params = transformer_params(V, D, F, L, N, K, H) * elem_bytes
    kv = S * (K * H) * L * 2 * elem_bytes
    memory = B * kv + params
    latency = memory / bandwidth
    return memory, latency, B / latency


def accelerator_intensity(flops_per_s: float, bytes_per_s: float) -> float:
    """CS336 lecture 10 §"Напоминание: арифметическая интенсивность"."""
    return flops_per_s / bytes_per_s


def decode_attention_intensity(S: int, T: int = 1) -> float:
    """CS336 lecture 10 §"Арифметическая интенсивность инференса": attention
    FLOPs 4BSTD over bytes 4BSD + 4BTD -> ST / (S + T); S/(S+1) for decode."""
    return S * T / (S + T)


def score_matrix_bytes(n: int, cached: bool, elem_bytes: int = 4) -> int:
    """KV-cache section of the "جعل inference رخيصًا" page: recomputation builds
    the full n x n score matrix per step, the cached step a 1 x n row."""
    return (n if cached else n * n) * elem_bytes


def attention_algorithmic_bytes(ctx_lens: Iterable[int], T: int, N: int, K: int, H: int,
                                elem_bytes: int, block_size: int = 16, window: int = 0,
                                kv_elem_bytes: int = 0, row_scale_bytes: int = 0) -> int:
    """Bytes one decode/verify attention launch must move at minimum: every
    visible cached key and value once, q in and out back, the block ids in use
    and the context lengths.  With a window W > 0 the visible positions of a
    sequence are ctx - T - W + 1 .. ctx - 1 (clipped at 0): min(ctx, W + T - 1)
    tokens, in the blocks from the one holding the first of them.  A one-byte
    cache: kv_elem_bytes = 1 and row_scale_bytes = 4 (the fp32 scale of each
    cached key / value row)."""
    ctx = np.asarray(list(ctx_lens), np.int64)
    B = ctx.size
    first = np.maximum(0, ctx - T - window + 1) if window > 0 else np.zeros_like(ctx)
    kv = int((ctx - first).sum()) * 2 * K * (H * (kv_elem_bytes or elem_bytes) + row_scale_bytes)
    qo = 2 * B * T * N * H * elem_bytes
    ids = 4 * int(((ctx + block_size - 1) // block_size - first // block_size).sum())
    return kv + qo + ids + 4 * B


def attention_flops(ctx_lens: Iterable[int], T: int, N: int, H: int, window: int = 0) -> int:
    """4 * (visible tokens) * T * N * H (QK^T and PV; an upper bound when T > 1)."""
    ctx = np.asarray(list(ctx_lens), np.int64)
    if window > 0:
        ctx = np.minimum(ctx, window + T - 1)
    return 4 * int(ctx.sum()) * T * N * H


def kv_append_bytes(B: int, T: int, K: int, H: int, elem_bytes: int) -> int:
    """Read k_new/v_new, write them into the cache, plus B lengths and B*T ids."""
    return 2 * 2 * B * T * K * H * elem_bytes + 4 * B + 4 * B * T


def kv_append_quant_bytes(B: int, T: int, K: int, H: int, elem_bytes: int) -> int:
    """Read k_new / v_new, write one-byte codes and a 4-byte scale per row."""
    return 2 * B * T * K * (H * elem_bytes + H + 4) + 4 * B + 4 * B * T


def accept_bytes(B: int, T: int, V: int) -> int:
    """Read the fp32 logits and drafts, write accepted / next token / lengths."""
    return B * T * V * 4 + B * max(T - 1, 0) * 4 + 3 * 4 * B


def accept_tree_bytes(B: int, T: int, V: int) -> int:
    """Tree acceptance: read the fp32 logits, drafts and parent entries;
    write accepted / next token / the branch and read-write the lengths."""
    return B * T * V * 4 + B * max(T - 1, 0) * 4 + B * T * 4 + 4 * B * (T - 1 + 4)


def kv_compact_bytes(accepted, K: int, H: int, elem_bytes: int = 2, T: int = 1,
                     scale_bytes: int = 0) -> int:
    """Compaction after tree acceptance: every kept node's K and V rows (and a
    one-byte row's scale) read and written once, plus the branch, the count
    and the length per sequence."""
    rows = int(sum(int(a) for a in accepted))
    return rows * 2 * 2 * K * (H * elem_bytes + scale_bytes) + len(accepted) * 4 * (T - 1 + 2)


def accept_sampled_bytes(accepted, T: int, V: int) -> int:
    """Bytes stochastic acceptance must move, given the accepted counts: per
    sequence the T fp64 uniforms and T-1 draft ids, q(x) and p(x) of every draft
    test reached (min(a+1, T-1) of them), the row(s) of the final draw (q and p
    after a rejection, q alone after a full run), and accepted / next token /
    length (read and written)."""
    tot = 0
    for a in accepted:
        a = int(a)
        tests = min(a + 1, T - 1)
        rows = 2 if a < T - 1 else 1
        tot += 8 * T + 4 * (T - 1) + 8 * tests + rows * V * 4 + 4 * 4
    return tot


def spec_expected_tokens(alpha: float, gamma: int) -> float:
    """Expected tokens kept per verify pass with per-token acceptance alpha and
    gamma drafts (geometric run plus the target's own token).  The formula is
    missing from the extracted "جعل inference رخيصًا" page; this is the reading
    that reproduces its printed 1.4 tokens at 30 % acceptance."""
    if alpha == 1.0:
        return gamma + 1.0
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def spec_speedup(alpha: float, gamma: int, c: float) -> float:
    """Net speedup: expected tokens over the pass cost in target-model units,
    gamma draft steps of relative cost c plus one target pass."""
    return spec_expected_tokens(alpha, gamma) / (gamma * c + 1.0)


def round_half_up(x: float, nd: int = 0) -> float:
    q = 10 ** nd
    return math.floor(x * q + 0.5) / q
