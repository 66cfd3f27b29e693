"""Pins for the fp64 oracle: closed forms, invariants, the pages' cache ==
recompute equality, library routines on special cases and brute force.  Each
test is chosen so that a plausible slip in the oracle (dropped scale, wrong
sign, wrong head or slot index, wrong causal bound, bad widening) fails it."""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import set_token, slot, small, unpage

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---- element widening --------------------------------------------------------
def test_f16_widening_matches_numpy_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()


def test_bf16_widening_matches_torch_all_patterns():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).double().numpy()
    got = np.array([oracle.bf16_to_f64(int(b) & 0xFFFF) for b in bits.numpy()])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()


def test_widening_known_values():
    assert oracle.f16_to_f64(0x3C00) == 1.0
    assert oracle.f16_to_f64(0xC000) == -2.0
    assert oracle.f16_to_f64(0x0001) == 2.0 ** -24
    assert oracle.f16_to_f64(0x7BFF) == 65504.0
    assert math.isinf(oracle.f16_to_f64(0x7C00))
    assert oracle.bf16_to_f64(0x3F80) == 1.0
    assert oracle.bf16_to_f64(0xC040) == -3.0


# ---- attention: closed forms -------------------------------------------------
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_single_token_context_returns_its_v_row(dtype):
    w = small(B=2, T=1, N=6, K=3, H=64, dtype=dtype, ctx=(1, 1), seed=1)
    out, err = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                                w.context_lens, dtype)
    assert (err == 0).all()
    for b in range(2):
        blk, r = slot(w, b, 0)
        for n in range(6):
            np.testing.assert_array_equal(out[b, 0, n], w.v_cache[0][blk, r, n // 2].double())


@pytest.mark.parametrize("N,K", [(8, 2), (6, 6), (7, 1)])
def test_constant_v_per_kv_head_returns_that_constant(N, K):
    # V of KV head k is the constant k+1 at every position: head n must return
    # exactly (n // G) + 1 whatever q and the keys are.
    ctx = (3, 20, 33)
    w = small(B=3, T=1, N=N, K=K, H=64, ctx=ctx, seed=2)
    for b, c in enumerate(ctx):
        for pos in range(c):
            v = torch.arange(1, K + 1, dtype=torch.float64)[:, None].expand(K, 64)
            set_token(w, b, pos, v=v)
    out, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                              w.context_lens, "f16")
    G = N // K
    for n in range(N):
        np.testing.assert_allclose(out[:, 0, n, :], (n // G) + 1, rtol=0, atol=1e-12)


@pytest.mark.parametrize("T", [1, 3, 5])
def test_equal_keys_average_the_visible_rows(T):
    # All keys equal -> uniform weights over the visible positions.  With
    # v_j = j, query token t must return (ctx - T + t) / 2: this pins the
    # block-table slot arithmetic, the context-length reading and the causal
    # bound among the T new tokens (NaN sentinels sit in every unused slot).
    ctx = (T, 16 + T, 37, 64)
    w = small(B=4, T=T, N=4, K=2, H=64, ctx=ctx, seed=3)
    key = torch.randn(2, 64, generator=torch.Generator().manual_seed(9))
    for b, c in enumerate(ctx):
        for pos in range(c):
            set_token(w, b, pos, k=key, v=torch.full((2, 64), float(pos)))
    out, err = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                                w.context_lens, "f16")
    assert (err == 0).all()
    for b, c in enumerate(ctx):
        for t in range(T):
            np.testing.assert_allclose(out[b, t], (c - T + t) / 2.0, rtol=1e-12, atol=1e-12)


def test_two_tokens_weights_three_to_one():
    # s_1 - s_2 = scale * <q, k_1 - k_2> = ln 3  ->  weights 3/4 and 1/4.
    w = small(B=1, T=1, N=1, K=1, H=64, ctx=(2,), seed=4)
    q = torch.zeros(64)
    q[0] = 1.0
    w.q[0][0, 0, 0] = q
    k1 = torch.zeros(64)
    k1[0] = 1.0
    set_token(w, 0, 0, k=k1[None], v=torch.full((1, 64), 4.0))
    set_token(w, 0, 1, k=torch.zeros(1, 64), v=torch.full((1, 64), 8.0))
    out, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                              w.context_lens, "f16", scale=math.log(3.0))
    np.testing.assert_allclose(out[0, 0, 0], 0.75 * 4.0 + 0.25 * 8.0, rtol=1e-14)


def test_default_scale_is_inverse_sqrt_head_size():
    # H = 64 -> scale 1/8; q[0] = 8, k_1[0] = 1, k_2 = 0: s_1 - s_2 = 1.
    w = small(B=1, T=1, N=1, K=1, H=64, ctx=(2,), seed=5)
    q = torch.zeros(64)
    q[0] = 8.0
    w.q[0][0, 0, 0] = q
    k1 = torch.zeros(64)
    k1[0] = 1.0
    set_token(w, 0, 0, k=k1[None], v=torch.full((1, 64), 1.0))
    set_token(w, 0, 1, k=torch.zeros(1, 64), v=torch.full((1, 64), 0.0))
    out, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                              w.context_lens, "f16")
    e = math.e
    np.testing.assert_allclose(out[0, 0, 0], e / (1 + e), rtol=1e-14)


# ---- attention: the pages' cache == recompute equality -------------------------
@pytest.mark.parametrize("dtype,H,T", [("f16", 64, 1), ("bf16", 128, 1), ("bf16", 64, 4)])
def test_paged_cache_equals_full_causal_recompute(dtype, H, T):
    ctx = (T, 19, 50)
    w = small(B=3, T=T, N=6, K=2, H=H, dtype=dtype, ctx=ctx, seed=6)
    out, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                              w.context_lens, dtype)
    gen = torch.Generator().manual_seed(11)
    for b, c in enumerate(ctx):
        kk, vv = unpage(w, b, c)
        q_all = torch.randn(c, 6, H, generator=gen).to(w.torch_dtype).double().numpy()
        q_all[c - T:] = w.q[0][b].double().numpy()  # the new tokens' queries
        full = oracle.causal_attention_full(q_all, kk, vv, 1.0 / math.sqrt(H))
        np.testing.assert_allclose(out[b], full[c - T:], rtol=0, atol=1e-12)


# ---- attention: invariants ---------------------------------------------------
def test_block_permutation_leaves_output_bit_identical():
    ctx = (30, 47)
    w = small(B=2, T=1, N=4, K=2, H=64, ctx=ctx, seed=7, spare=3)
    ref, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                              w.context_lens, "f16")
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(3))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(w.num_blocks)
    kc = w.k_cache[0][perm]  # new block i holds old block perm[i]
    vc = w.v_cache[0][perm]
    tables = w.block_tables.clone()
    used = tables != 2**31 - 1
    tables[used] = inv[tables[used].long()].int()
    out, _ = oracle.attention(w.q[0], kc, vc, tables, w.context_lens, "f16")
    np.testing.assert_array_equal(out, ref)


def test_adding_a_multiple_of_q_to_every_key_changes_nothing():
    # Every score moves by the same amount, softmax is shift-invariant.  Small
    # dyadic values keep k + q exact in fp16.
    ctx = (21,)
    w = small(B=1, T=1, N=1, K=1, H=64, ctx=ctx, seed=8)
    g = torch.Generator().manual_seed(5)
    q = torch.randint(-4, 5, (64,), generator=g).double() / 4
    w.q[0][0, 0, 0] = q
    keys = [torch.randint(-4, 5, (1, 64), generator=g).double() / 4 for _ in range(21)]
    for pos in range(21):
        set_token(w, 0, pos, k=keys[pos])
    ref, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                              w.context_lens, "f16")
    for pos in range(21):
        set_token(w, 0, pos, k=keys[pos] + 0.5 * q[None])
    out, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                              w.context_lens, "f16")
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("N,K", [(6, 1), (6, 6), (8, 4)])
def test_each_head_equals_a_single_head_problem(N, K):
    # MQA (K = 1), MHA (K = N) and GQA: head n equals the same problem posed
    # with one query head and KV head n // G alone.
    ctx = (9, 33)
    w = small(B=2, T=1, N=N, K=K, H=64, ctx=ctx, seed=9)
    out, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                              w.context_lens, "f16")
    G = N // K
    for n in range(N):
        kh = n // G
        o1, _ = oracle.attention(w.q[0][:, :, n:n + 1].contiguous(),
                                 w.k_cache[0][:, :, kh:kh + 1].contiguous(),
                                 w.v_cache[0][:, :, kh:kh + 1].contiguous(),
                                 w.block_tables, w.context_lens, "f16")
        np.testing.assert_array_equal(out[:, :, n:n + 1], o1)


def test_subset_listing_matches_full_run():
    w = small(B=4, T=2, N=4, K=2, H=64, ctx=(2, 17, 33, 5), seed=10)
    full, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                               w.context_lens, "f16")
    sub, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                              w.context_lens, "f16", b_list=[3, 1])
    np.testing.assert_array_equal(sub, full[[3, 1]])


def test_bad_context_and_bad_block_give_zeros_and_codes():
    w = small(B=3, T=2, N=4, K=2, H=64, ctx=(1, 20, 20), seed=11)
    tables = w.block_tables.clone()
    tables[2, 1] = w.num_blocks + 5  # second block of sequence 2 is bogus
    out, err = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], tables, w.context_lens,
                                "f16")
    assert list(err) == [7, 0, 8]
    assert (out[0] == 0).all() and (out[2] == 0).all()
    assert np.isfinite(out[1]).all() and (out[1] != 0).any()


# ---- append ------------------------------------------------------------------
def test_kv_append_hand_example():
    # ctx = 17 with T = 2: the new tokens land at positions 15 and 16, i.e.
    # block table[0] row 15 and block table[1] row 0.
    w = small(B=1, T=2, N=2, K=1, H=64, ctx=(17,), seed=12, append=True, shuffle=True)
    kc, vc, err = oracle.kv_append(w.k_new[0], w.v_new[0], w.k_cache[0], w.v_cache[0],
                                   w.block_tables, w.context_lens)
    assert err[0] == 0
    b0, b1 = int(w.block_tables[0, 0]), int(w.block_tables[0, 1])
    kn = w.k_new[0].view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(kc[b0, 15], kn[0, 0])
    np.testing.assert_array_equal(kc[b1, 0], kn[0, 1])


def test_kv_append_round_trip_and_untouched_slots():
    ctx = (1, 16, 17, 40)
    w = small(B=4, T=1, N=4, K=2, H=128, dtype="bf16", ctx=ctx, seed=13, append=True)
    before_k = w.k_cache[0].view(torch.int16).numpy().view(np.uint16).copy()
    kc, vc, err = oracle.kv_append(w.k_new[0], w.v_new[0], w.k_cache[0], w.v_cache[0],
                                   w.block_tables, w.context_lens)
    assert (err == 0).all()
    changed = np.zeros(before_k.shape[:2], bool)
    kn = w.k_new[0].view(torch.int16).numpy().view(np.uint16)
    for b, c in enumerate(ctx):
        blk, r = slot(w, b, c - 1)
        np.testing.assert_array_equal(kc[blk, r], kn[b, 0])
        changed[blk, r] = True
    np.testing.assert_array_equal(kc[~changed], before_k[~changed])


def test_kv_append_errors_skip_the_sequence():
    w = small(B=2, T=3, N=2, K=1, H=64, ctx=(2, 10), seed=14, append=True)
    kc, vc, err = oracle.kv_append(w.k_new[0], w.v_new[0], w.k_cache[0], w.v_cache[0],
                                   w.block_tables, w.context_lens)
    assert list(err) == [7, 0]


# ---- acceptance ----------------------------------------------------------------
def test_argmax_matches_numpy_with_ties_and_nans():
    rng = np.random.default_rng(0)
    for trial in range(300):
        V = int(rng.integers(1, 50))
        x = rng.integers(-3, 4, size=V).astype(np.float32)  # many ties
        if trial % 3 == 0:
            x[rng.integers(0, V, size=2)] = np.nan
        if trial % 5 == 0:
            x[rng.integers(0, V)] = -0.0
        assert oracle.argmax(x) == int(np.argmax(x)), x


def test_accept_prefix_hand_cases():
    V = 6
    T = 4
    lg = np.zeros((5, T, V), np.float32)
    # argmax per position (rows listed per sequence)
    picks = [[1, 2, 3, 4], [1, 2, 3, 4], [0, 5, 5, 5], [2, 2, 2, 2], [3, 3, 3, 3]]
    for b in range(5):
        for t in range(T):
            lg[b, t, picks[b][t]] = 1.0
    lg[3, 1, 4] = 1.0  # tie at position 1 of seq 3: index 2 still wins
    lg[4, 0, 5] = np.nan  # NaN at position 0 of seq 4 wins the argmax
    draft = np.array([[1, 2, 3], [1, 9, 3], [5, 5, 5], [2, 2, 2], [5, 3, 3]], np.int32)
    ctx = np.array([10, 10, 10, 10, 10], np.int32)
    acc, nxt, ctx2 = oracle.accept_prefix(lg, draft, ctx)
    assert list(acc) == [3, 1, 0, 3, 3]
    assert list(nxt) == [4, 2, 0, 2, 3]
    assert list(ctx2) == [10, 8, 7, 10, 10]


def test_accept_prefix_single_token_and_planted_drafts():
    w = small(B=6, T=5, N=2, K=1, H=64, ctx=(8,) * 6, seed=15, vocab=1000)
    acc, nxt, _ = oracle.accept_prefix(w.logits, w.draft)
    assert (acc >= w.draft_k).all()  # planted prefix always accepted
    lg = w.logits.numpy()
    for b in range(6):
        assert nxt[b] == int(np.argmax(lg[b, acc[b]]))
    one, nxt1, _ = oracle.accept_prefix(w.logits[:, :1].contiguous(),
                                        np.zeros((6, 0), np.int32))
    assert (one == 0).all()
    assert list(nxt1) == [int(np.argmax(lg[b, 0])) for b in range(6)]


# ---- local (sliding-window) attention ------------------------------------------
@pytest.mark.parametrize("T", [1, 3])
@pytest.mark.parametrize("W", [1, 5, 16, 23])
def test_window_equal_keys_average_the_window(T, W):
    # Equal keys -> uniform weights over the visible band; v_j = j makes query
    # token t (position last = ctx - T + t) return the mean of
    # max(0, last - W + 1) .. last.  Pins both ends of the band.
    ctx = (T, 16 + T, 37, 64)
    w = small(B=4, T=T, N=4, K=2, H=64, ctx=ctx, seed=31)
    key = torch.randn(2, 64, generator=torch.Generator().manual_seed(9))
    for b, c in enumerate(ctx):
        for pos in range(c):
            set_token(w, b, pos, k=key, v=torch.full((2, 64), float(pos)))
    out, err = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                                w.context_lens, "f16", window=W)
    assert (err == 0).all()
    for b, c in enumerate(ctx):
        for t in range(T):
            last = c - T + t
            first = max(0, last - W + 1)
            np.testing.assert_allclose(out[b, t], (first + last) / 2.0, rtol=1e-12, atol=1e-12)


def test_window_of_one_returns_the_own_v_row():
    ctx = (9, 40)
    w = small(B=2, T=3, N=4, K=2, H=64, ctx=ctx, seed=32)
    out, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                              w.context_lens, "f16", window=1)
    for b, c in enumerate(ctx):
        for t in range(3):
            blk, r = slot(w, b, c - 3 + t)
            for n in range(4):
                np.testing.assert_array_equal(out[b, t, n], w.v_cache[0][blk, r, n // 2].double())


def test_window_wider_than_context_is_full_attention():
    ctx = (5, 17, 40)
    w = small(B=3, T=2, N=4, K=2, H=64, ctx=ctx, seed=33)
    full, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                               w.context_lens, "f16")
    win, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                              w.context_lens, "f16", window=41)
    np.testing.assert_array_equal(win, full)


@pytest.mark.parametrize("W,T", [(7, 1), (16, 2), (33, 4)])
def test_window_paged_equals_banded_recompute(W, T):
    ctx = (T, 30, 77)
    w = small(B=3, T=T, N=6, K=2, H=64, dtype="bf16", ctx=ctx, seed=34)
    out, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                              w.context_lens, "bf16", window=W)
    gen = torch.Generator().manual_seed(12)
    for b, c in enumerate(ctx):
        kk, vv = unpage(w, b, c)
        q_all = torch.randn(c, 6, 64, generator=gen).to(w.torch_dtype).double().numpy()
        q_all[c - T:] = w.q[0][b].double().numpy()
        full = oracle.causal_attention_full(q_all, kk, vv, 1.0 / 8.0, window=W)
        np.testing.assert_allclose(out[b], full[c - T:], rtol=0, atol=1e-12)


def test_tokens_outside_the_window_do_not_matter_and_freed_blocks_are_not_read():
    # Poison every position below the first window (NaN K and V) and free the
    # blocks that hold no visible position (INT32_MAX in the table): the output
    # stays finite and equal.  A band one token too wide would read a NaN.
    T, W = 2, 20
    ctx = (50, 64, 21)
    w = small(B=3, T=T, N=4, K=2, H=64, ctx=ctx, seed=35)
    ref, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                              w.context_lens, "f16", window=W)
    nan = torch.full((2, 64), float("nan"))
    tables = w.block_tables.clone()
    for b, c in enumerate(ctx):
        first = max(0, c - T - W + 1)
        for pos in range(first):
            set_token(w, b, pos, k=nan, v=nan)
        tables[b, : first // 16] = 2**31 - 1
    out, err = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], tables, w.context_lens,
                                "f16", window=W)
    assert (err == 0).all()
    np.testing.assert_array_equal(out, ref)
    # the first visible position does matter
    b, c = 0, ctx[0]
    set_token(w, b, c - T - W + 1, v=nan)
    out2, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], tables, w.context_lens,
                               "f16", window=W)
    assert np.isnan(out2[0, 0]).all() and np.isfinite(out2[0, 1]).all()


def test_window_block_check_covers_the_earliest_query_of_the_run():
    # T = 3, W = 20, ctx = 36: query 0 sees positions 14..33, query 2 sees
    # 16..35.  Block 0 holds position 14 and 15, so a bad id there is an error;
    # with ctx = 38 no query sees block 0 and the same bad id is never read.
    T, W = 3, 20
    w = small(B=2, T=T, N=4, K=2, H=64, ctx=(36, 38), seed=36)
    tables = w.block_tables.clone()
    tables[:, 0] = -1
    out, err = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], tables, w.context_lens,
                                "f16", window=W)
    assert err.tolist() == [8, 0]
    assert (out[0] == 0).all() and np.isfinite(out[1]).all()


# ---- tree verification (custom mask among the new tokens) -------------------------
def tree_masks(parents):
    """uint64 mask rows of a tree given as parent indices (-1: child of the
    prefix), nodes in topological order: bit j of row t set for every ancestor."""
    T = len(parents)
    m = np.zeros(T, np.uint64)
    for t in range(T):
        a = parents[t]
        while a >= 0:
            m[t] |= np.uint64(1) << np.uint64(a)
            a = parents[a]
    return m


TREE = [-1, 0, 0, 1, 1, 2, 3, -1]  # two roots, depth 4


def test_tree_chain_mask_equals_verify():
    T = 6
    ctx = (T, 30, 77)
    w = small(B=3, T=T, N=4, K=2, H=64, ctx=ctx, seed=41)
    chain = np.array([(1 << t) - 1 for t in range(T)], np.uint64)
    ref, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                              w.context_lens, "f16")
    got, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                              w.context_lens, "f16", tree_mask=np.tile(chain, (3, 1)))
    np.testing.assert_array_equal(got, ref)


def test_tree_equal_keys_average_prefix_and_ancestors():
    T = len(TREE)
    ctx = (T, 21, 50)
    w = small(B=3, T=T, N=4, K=2, H=64, ctx=ctx, seed=42)
    key = torch.randn(2, 64, generator=torch.Generator().manual_seed(9))
    for b, c in enumerate(ctx):
        for pos in range(c):
            set_token(w, b, pos, k=key, v=torch.full((2, 64), float(pos)))
    m = tree_masks(TREE)
    out, err = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                                w.context_lens, "f16", tree_mask=np.tile(m, (3, 1)))
    assert (err == 0).all()
    for b, c in enumerate(ctx):
        P = c - T
        for t in range(T):
            vis = list(range(P)) + [P + j for j in range(T) if j == t or (int(m[t]) >> j) & 1]
            np.testing.assert_allclose(out[b, t], np.mean(vis), rtol=1e-12, atol=1e-12)


def test_tree_rows_equal_causal_attention_down_their_path():
    """EAGLE's tree attention is causal attention of the prefix followed by the
    node's root-to-node path: recompute each path as a linear sequence."""
    T = len(TREE)
    ctx = (T + 3, 40, 100)
    w = small(B=3, T=T, N=6, K=2, H=64, dtype="bf16", ctx=ctx, seed=43)
    m = tree_masks(TREE)
    out, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                              w.context_lens, "bf16", tree_mask=np.tile(m, (3, 1)))
    for b, c in enumerate(ctx):
        P = c - T
        kk, vv = unpage(w, b, c)
        qn = w.q[0][b].double().numpy()  # [T, N, H]
        for t in range(T):
            path = [j for j in range(T) if (int(m[t]) >> j) & 1] + [t]
            seq = list(range(P)) + [P + j for j in path]
            q_all = np.zeros((len(seq), 6, 64))
            q_all[-1] = qn[t]
            full = oracle.causal_attention_full(q_all, kk[seq], vv[seq], 1.0 / 8.0)
            np.testing.assert_allclose(out[b, t], full[-1], rtol=0, atol=1e-12)


def test_tree_bits_at_or_after_the_row_are_ignored():
    T = len(TREE)
    w = small(B=2, T=T, N=4, K=2, H=64, ctx=(T, 60), seed=44)
    m = tree_masks(TREE)
    junk = m | np.array([~np.uint64(0) << np.uint64(t) for t in range(T)], np.uint64)
    a, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables, w.context_lens,
                            "f16", tree_mask=np.tile(m, (2, 1)))
    b_, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables, w.context_lens,
                             "f16", tree_mask=np.tile(junk, (2, 1)))
    np.testing.assert_array_equal(a, b_)
