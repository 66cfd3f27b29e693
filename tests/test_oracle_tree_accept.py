"""Pins of the oracle's greedy acceptance over a draft tree and of the cache
compaction that follows it, against what the pages and independent
formulations fix, not against the oracle itself.

"Болжау арқылы Sonar модельдерін жылдамдату", §"EAGLE": the draft explores a
tree of candidates, the target scores every node in one pass under a custom
attention mask (each node sees its ancestors), and the longest candidate
sequence the target agrees with is kept, plus one token from the target.
§"Спекулятивті кодтан шығару" is the chain case of the same rule.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import planted_tree_inputs as planted, random_parents, slot, small


def one_hot_logits(g, T, V):
    """logits [1,T,V] whose argmax at node i is g[i]."""
    lg = np.random.default_rng(0).normal(size=(1, T, V)).astype(np.float32)
    for i, v in g.items():
        lg[0, i, v] = 10.0
    return lg


# A hand-made tree (V = 8): root 0; its children 1, 2, 3 carry tokens 5, 3, 7;
# node 1's children 4, 5 carry 2, 6; node 3's child 6 carries 1; node 6's
# child 7 carries 4.  The target predicts 7 after the root, 1 after node 3 and
# 0 after node 6: node 3 (7 == 7) and node 6 (1 == 1) are kept, node 7 (4 != 0)
# is not.  Two accepted drafts, then the target's own 0.
HAND_PARENTS = [-1, 0, 0, 0, 1, 1, 3, 6]
HAND_TOKENS = [5, 3, 7, 2, 6, 1, 4]  # of nodes 1..7
HAND_G = {0: 7, 1: 2, 2: 0, 3: 1, 4: 0, 5: 0, 6: 0, 7: 3}


def test_hand_tree():
    lg = one_hot_logits(HAND_G, 8, 8)
    acc, nxt, path, ctx, err = oracle.accept_tree(
        lg, np.array([HAND_TOKENS], np.int32), np.array([HAND_PARENTS], np.int32),
        np.array([100], np.int32))
    assert acc[0] == 2 and nxt[0] == 0 and err[0] == 0
    assert list(path[0]) == [3, 6, -1, -1, -1, -1, -1]
    assert ctx[0] == 100 - (8 - 1 - 2)


def test_hand_tree_root_mismatch_keeps_only_the_target_token():
    g = dict(HAND_G)
    g[0] = 4  # no child of the root carries 4
    acc, nxt, path, _, err = oracle.accept_tree(
        one_hot_logits(g, 8, 8), np.array([HAND_TOKENS], np.int32),
        np.array([HAND_PARENTS], np.int32))
    assert acc[0] == 0 and nxt[0] == 4 and (path[0] == -1).all() and err[0] == 0


def test_deeper_branch_wins_and_equal_depth_goes_to_the_lower_index():
    # root's children 1 and 2 both carry the target's token 3 (duplicate
    # siblings); only node 2 has an accepted child (node 3, token 5 after g_2 = 5)
    par = np.array([[-1, 0, 0, 2, 1]], np.int32)
    tok = np.array([[3, 3, 5, 6]], np.int32)
    g = {0: 3, 1: 1, 2: 5, 3: 0, 4: 2}
    acc, nxt, path, _, _ = oracle.accept_tree(one_hot_logits(g, 5, 8), tok, par)
    assert acc[0] == 2 and list(path[0][:2]) == [2, 3] and nxt[0] == 0
    # same, but node 3's token no longer matches: nodes 1 and 2 tie at depth 1
    # and the lower index (1) is kept; the next token is the target's after it
    tok2 = np.array([[3, 3, 4, 6]], np.int32)
    acc, nxt, path, _, _ = oracle.accept_tree(one_hot_logits(g, 5, 8), tok2, par)
    assert acc[0] == 1 and path[0][0] == 1 and nxt[0] == 1


@pytest.mark.parametrize("T", [1, 2, 5, 16, 64])
def test_chain_tree_is_prefix_acceptance(T):
    """parents[i] = i - 1: exactly the pinned chain rule, for every output."""
    rng = np.random.default_rng(T)
    B, V = 24, 37
    par = np.tile(np.arange(-1, T - 1, dtype=np.int32), (B, 1))
    lg, draft = planted(B, T, V, par, rng, p_match=0.85)
    ctx = rng.integers(T, 500, size=B).astype(np.int32)
    acc, nxt, path, ctx2, err = oracle.accept_tree(lg, draft, par, ctx)
    a0, n0, c0 = oracle.accept_prefix(lg, draft, ctx)
    assert (err == 0).all()
    np.testing.assert_array_equal(acc, a0)
    np.testing.assert_array_equal(nxt, n0)
    np.testing.assert_array_equal(ctx2, c0)
    for b in range(B):  # the accepted chain nodes are 1..a
        assert list(path[b]) == list(range(1, acc[b] + 1)) + [-1] * (T - 1 - acc[b])


def greedy_walk(lg, draft, par):
    """Independent formulation: the greedy target emits its choice after the
    current node; every child carrying that token is followed (depth first);
    the deepest node reached wins, the lowest index among equals.  Returns
    (a, path, next)."""
    T = par.shape[0]
    children = [[] for _ in range(T)]
    for c in range(1, T):
        children[par[c]].append(c)

    def best_from(node, depth):
        g = int(np.argmax(lg[node]))  # numpy's first-max rule (rows here hold no NaN)
        best = (depth, node, [])
        for c in children[node]:
            if draft[c - 1] == g:
                d, n, p = best_from(c, depth + 1)
                if d > best[0] or (d == best[0] and n < best[1]):
                    best = (d, n, [c] + p)
        return best

    d, n, p = best_from(0, 0)
    return d, p, int(np.argmax(lg[n]))


@pytest.mark.parametrize("seed", range(6))
def test_matches_an_independent_greedy_walk(seed):
    rng = np.random.default_rng(100 + seed)
    B, T, V = 40, [3, 8, 12, 26, 40, 64][seed], 5  # a small V makes duplicate siblings common
    par = random_parents(B, T, rng, chain_bias=0.3)
    lg, draft = planted(B, T, V, par, rng, p_match=0.7)
    acc, nxt, path, _, err = oracle.accept_tree(lg, draft, par)
    assert (err == 0).all()
    for b in range(B):
        a, p, n = greedy_walk(lg[b], draft[b], par[b])
        assert acc[b] == a and nxt[b] == n, b
        assert list(path[b][:a]) == p and (path[b][a:] == -1).all(), b


def test_malformed_tree_rejects_the_broken_branch_and_reports_it():
    # node 2's parent entry points at itself: node 2 and its child 3 can never
    # be kept; node 1's branch is decided as usual
    par = np.array([[-1, 0, 2, 2, 1]], np.int32)
    tok = np.array([[4, 4, 1, 2]], np.int32)
    g = {0: 4, 1: 2, 2: 1, 3: 0, 4: 0}
    acc, nxt, path, _, err = oracle.accept_tree(one_hot_logits(g, 5, 8), tok, par)
    assert err[0] == 11
    assert acc[0] == 2 and list(path[0][:2]) == [1, 4] and nxt[0] == 0
    # a root entry other than -1 is reported, the rest decided as usual
    par2 = np.array([[0, 0, 0, 2, 1]], np.int32)
    acc, _, _, _, err = oracle.accept_tree(one_hot_logits(g, 5, 8), tok, par2)
    assert err[0] == 11 and acc[0] == 2


def test_context_underflow_is_left_unchanged():
    par = np.array([[-1, 0, 0]], np.int32)
    acc, _, _, ctx, err = oracle.accept_tree(one_hot_logits({0: 1, 1: 1, 2: 1}, 3, 4),
                                             np.array([[0, 2]], np.int32), par,
                                             np.array([1], np.int32))
    assert acc[0] == 0 and ctx[0] == 1 and err[0] == 7


# ---- cache compaction --------------------------------------------------------


def compact_case(dtype="f16", seed=0, T=8, ctx_after=(40, 17, 9), acc=(3, 0, 2),
                 paths=((2, 5, 7), (), (4, 6))):
    B = len(ctx_after)
    # the caches as appended: T tree nodes at base .. base+T-1, base = ctx - 1 - a
    ctx_before = [c - 1 - a + T for c, a in zip(ctx_after, acc)]
    w = small(B=B, T=T, N=8, K=2, H=64, dtype=dtype, ctx=tuple(ctx_before), seed=seed,
              max_blocks=8)
    path = np.full((B, T - 1), -1, np.int32)
    for b, p in enumerate(paths):
        path[b, :len(p)] = p
    return w, np.asarray(ctx_after, np.int32), np.asarray(acc, np.int32), path


def test_compaction_moves_the_accepted_rows_and_nothing_else():
    w, ctx, acc, path = compact_case()
    kc, vc, _, _, err = oracle.kv_compact(w.k_cache[0], w.v_cache[0], w.block_tables, ctx, path,
                                          acc, w.T)
    assert (err == 0).all()
    k0 = w.k_cache[0].view(torch.int16).numpy().view(np.uint16)
    v0 = w.v_cache[0].view(torch.int16).numpy().view(np.uint16)
    expect_k, expect_v = k0.copy(), v0.copy()
    for b in range(w.B):
        base = int(ctx[b]) - 1 - int(acc[b])
        for j in range(int(acc[b])):  # test-side restatement, written per row
            sb, sr = slot(w, b, base + int(path[b, j]))
            db, dr = slot(w, b, base + 1 + j)
            expect_k[db, dr] = k0[sb, sr]
            expect_v[db, dr] = v0[sb, sr]
    np.testing.assert_array_equal(kc, expect_k)
    np.testing.assert_array_equal(vc, expect_v)
    # the identity path (a chain) changes no byte
    ident = np.full_like(path, -1)
    for b in range(w.B):
        ident[b, :acc[b]] = np.arange(1, acc[b] + 1)
    kc2, vc2, _, _, _ = oracle.kv_compact(w.k_cache[0], w.v_cache[0], w.block_tables, ctx,
                                          ident, acc, w.T)
    np.testing.assert_array_equal(kc2, k0)
    np.testing.assert_array_equal(vc2, v0)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_tree_node_attention_equals_decode_after_compaction(dtype):
    """The point of compaction: node m's tree-masked verify output (it sees the
    prefix and its own ancestors) equals plain decode attention of node m's
    query over the compacted cache with the new length."""
    T = 8
    trees = [np.array(HAND_PARENTS, np.int32),            # kept path 0-3-6
             np.array([-1, 0, 0, 1, 2, 4, 3, 6], np.int32),  # kept path 0-2-4-5
             np.array(HAND_PARENTS, np.int32)]            # kept path 0-2
    w, ctx, acc, path = compact_case(dtype=dtype, seed=3, ctx_after=(40, 23, 9), acc=(2, 3, 1),
                                     paths=((3, 6), (2, 4, 5), (2,)))
    masks = np.zeros((w.B, T), np.uint64)
    for b in range(w.B):
        for t in range(T):
            a = t
            while a >= 0:
                masks[b, t] |= np.uint64(1) << np.uint64(a)
                a = trees[b][a]
    out_tree, err = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                                     w.context_lens, dtype, tree_mask=masks)
    assert (err == 0).all()
    kc, vc, _, _, cerr = oracle.kv_compact(w.k_cache[0], w.v_cache[0], w.block_tables, ctx, path,
                                           acc, T)
    assert (cerr == 0).all()
    tdt = w.torch_dtype
    kct = torch.from_numpy(kc.view(np.int16)).view(tdt)
    vct = torch.from_numpy(vc.view(np.int16)).view(tdt)
    for b in range(w.B):
        m = int(path[b, acc[b] - 1])
        one, e1 = oracle.attention(w.q[0][b:b + 1, m:m + 1], kct, vct, w.block_tables[b:b + 1],
                                   ctx[b:b + 1], dtype)
        assert e1[0] == 0
        np.testing.assert_allclose(one[0, 0], out_tree[b, m], rtol=0, atol=1e-12)


@pytest.mark.parametrize("kv", ["int8", "e4m3"])
def test_compaction_moves_one_byte_rows_with_their_scales(kv):
    w, ctx, acc, path = compact_case(dtype="bf16", seed=5)
    codes_k, sk = oracle.quantize_cache(w.k_cache[0], "bf16", kv)
    codes_v, sv = oracle.quantize_cache(w.v_cache[0], "bf16", kv)
    kc, vc, ks, vs, err = oracle.kv_compact(codes_k, codes_v, w.block_tables, ctx, path, acc, w.T,
                                            k_scale=sk, v_scale=sv)
    assert (err == 0).all()
    for b in range(w.B):
        base = int(ctx[b]) - 1 - int(acc[b])
        for j in range(int(acc[b])):
            sb, sr = slot(w, b, base + int(path[b, j]))
            db, dr = slot(w, b, base + 1 + j)
            np.testing.assert_array_equal(kc[db, dr], codes_k[sb, sr])
            np.testing.assert_array_equal(vc[db, dr], codes_v[sb, sr])
            np.testing.assert_array_equal(ks[db, :, dr], sk[sb, :, sr])
            np.testing.assert_array_equal(vs[db, :, dr], sv[sb, :, sr])


def test_compaction_checks_leave_the_sequence_untouched():
    w, ctx, acc, path = compact_case()
    bad_path = path.copy()
    bad_path[0, :3] = (5, 2, 7)            # not increasing
    bad_ctx = ctx.copy()
    bad_ctx[1] = 0                         # base = -1
    bt = w.block_tables.clone()
    base2 = int(ctx[2]) - 1 - int(acc[2])
    bt[2, (base2 + 3) // w.block_size] = w.num_blocks + 5  # a node's block id out of range
    kc, vc, _, _, err = oracle.kv_compact(w.k_cache[0], w.v_cache[0], bt, bad_ctx, bad_path,
                                          acc, w.T)
    assert list(err) == [11, 7, 8]
    np.testing.assert_array_equal(kc, w.k_cache[0].view(torch.int16).numpy().view(np.uint16))
    np.testing.assert_array_equal(vc, w.v_cache[0].view(torch.int16).numpy().view(np.uint16))
    # accepted outside [0, T-1]
    _, _, _, _, err = oracle.kv_compact(w.k_cache[0], w.v_cache[0], w.block_tables, ctx, path,
                                        np.array([8, 0, 2], np.int32), w.T)
    assert list(err) == [11, 0, 0]


def test_tree_workload_keeps_at_least_its_planted_branch():
    """The tree workload's recipe plants one branch per sequence whose every
    edge carries the target's choice; the kept branch is at least that deep,
    and a kept branch's edges all agree with the target (checked edge by edge
    with numpy's first-max argmax; the rows hold no NaN)."""
    from gqa_decode_attention_02_gb300 import workloads

    w = workloads.make("tree", B=6)
    par = w.parents()
    acc, nxt, path, _, err = oracle.accept_tree(w.logits, w.draft, par)
    assert (err == 0).all()
    lg = w.logits.numpy()
    dr = w.draft.numpy()
    for b in range(w.B):
        depth, node = 0, int(w.draft_k[b])
        while node > 0:
            depth, node = depth + 1, int(par[b, node])
        assert acc[b] >= depth
        prev = 0
        for j in range(acc[b]):
            c = int(path[b, j])
            assert par[b, c] == prev and dr[b, c - 1] == int(np.argmax(lg[b, prev]))
            prev = c
        assert nxt[b] == int(np.argmax(lg[b, prev]))
