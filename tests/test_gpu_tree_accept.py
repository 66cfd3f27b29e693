"""GPU greedy acceptance over a draft tree and the cache compaction after it,
bit-exact against the oracle (integers and raw cache bytes): random trees up
to 64 nodes, duplicate sibling tokens, ties, NaN, malformed trees, both accept
kernels (many blocks per sequence meeting in a workspace, and one thread-block
cluster per sequence), caches in q's dtype and one-byte caches with their
scales, and a whole tree step (fused append + tree verify, acceptance,
compaction, next decode) chained with programmatic dependent launch and
replayed from a CUDA graph."""
import numpy as np
import pytest
import torch

import gqa_decode_attention_02_gb300 as gq
import oracle
from gqa_decode_attention_02_gb300 import workloads
from helpers import assert_close, planted_tree_inputs, random_parents, small, to

pytestmark = pytest.mark.gpu

KERNELS = [False, True]  # cluster=False: the workspace kernel; True: one cluster per sequence


def run_tree(lg, draft, par, ctx, dev, cluster=False):
    lg_d = torch.as_tensor(lg).to(dev).contiguous()
    dr_d = torch.as_tensor(draft, dtype=torch.int32).to(dev).contiguous()
    par_d = torch.as_tensor(par, dtype=torch.int32).to(dev).contiguous()
    ctx_d = None if ctx is None else torch.as_tensor(ctx, dtype=torch.int32).to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    acc, nxt, path = gq.accept_tree(lg_d, dr_d, par_d, ctx_d, cluster=cluster, status=st)
    torch.cuda.synchronize()
    return (acc.cpu().numpy(), nxt.cpu().numpy(), path.cpu().numpy(),
            None if ctx_d is None else ctx_d.cpu().numpy(), int(st.item()))


def check_same(got, want):
    ga, gn, gp, gc, _ = got
    ra, rn, rp, rc, _ = want
    np.testing.assert_array_equal(ga, ra)
    np.testing.assert_array_equal(gn, rn)
    np.testing.assert_array_equal(gp, rp)
    if rc is not None:
        np.testing.assert_array_equal(gc, rc)


@pytest.mark.parametrize("cluster", KERNELS)
@pytest.mark.parametrize("B,T,V", [(16, 26, 32000), (3, 1, 7), (4, 8, 50257), (2, 64, 999),
                                   (300, 5, 100), (64, 12, 5), (500, 26, 4096)])
def test_tree_accept_matches_oracle(gpu, B, T, V, cluster):
    rng = np.random.default_rng(B * 131 + T)
    par = random_parents(B, T, rng, chain_bias=0.3)
    lg, draft = planted_tree_inputs(B, T, V, par, rng, p_match=0.7)
    ctx = rng.integers(T, 5000, size=B).astype(np.int32)
    want = oracle.accept_tree(lg, draft, par, ctx)
    assert (want[4] == 0).all()
    got = run_tree(lg, draft, par, ctx, gpu, cluster)
    assert got[4] == 0
    check_same(got, want)


@pytest.mark.parametrize("cluster", KERNELS)
def test_chain_parents_give_prefix_acceptance_bit_for_bit(gpu, cluster):
    rng = np.random.default_rng(5)
    B, T, V = 40, 6, 32000
    par = np.tile(np.arange(-1, T - 1, dtype=np.int32), (B, 1))
    lg, draft = planted_tree_inputs(B, T, V, par, rng, p_match=0.8)
    ctx = rng.integers(T, 900, size=B).astype(np.int32)
    ga, gn, gp, gc, st = run_tree(lg, draft, par, ctx, gpu, cluster)
    lg_d, dr_d = torch.as_tensor(lg).to(gpu), torch.as_tensor(draft).to(gpu)
    ctx_d = torch.as_tensor(ctx).to(gpu)
    pa, pn = gq.accept_prefix(lg_d, dr_d, ctx_d, cluster=cluster)
    torch.cuda.synchronize()
    assert st == 0
    np.testing.assert_array_equal(ga, pa.cpu().numpy())
    np.testing.assert_array_equal(gn, pn.cpu().numpy())
    np.testing.assert_array_equal(gc, ctx_d.cpu().numpy())
    for b in range(B):
        assert list(gp[b]) == list(range(1, ga[b] + 1)) + [-1] * (T - 1 - ga[b])


@pytest.mark.parametrize("cluster", KERNELS)
def test_ties_nan_and_duplicate_siblings(gpu, cluster):
    rng = np.random.default_rng(11)
    B, T, V = 64, 20, 6
    par = random_parents(B, T, rng)
    lg = rng.integers(-2, 3, size=(B, T, V)).astype(np.float32)  # heavy ties
    lg[::3, :, 4] = np.nan
    lg[1::4, :, :] = 0.0
    lg[1::4, :, 2] = -0.0
    draft = rng.integers(0, V, size=(B, T - 1)).astype(np.int32)  # V = 6: equal siblings
    for b in range(0, B, 2):  # many edges agree with the target
        for c in range(1, T):
            draft[b, c - 1] = oracle.argmax(lg[b, par[b, c]])
    want = oracle.accept_tree(lg, draft, par)
    got = run_tree(lg, draft, par, None, gpu, cluster)
    check_same(got, want)
    assert (want[0] > 0).sum() > B // 4  # the case exercises kept branches


@pytest.mark.parametrize("cluster", KERNELS)
def test_malformed_trees_and_context_underflow_are_reported(gpu, cluster):
    rng = np.random.default_rng(2)
    B, T, V = 8, 9, 50
    par = random_parents(B, T, rng)
    par[1, 4] = 4    # a node as its own parent
    par[2, 0] = 0    # a root entry other than -1
    par[3, 7] = 12   # a parent after the node
    lg, draft = planted_tree_inputs(B, T, V, par.clip(0, T - 1), rng, p_match=0.9)
    ctx = np.full(B, 100, np.int32)
    want = oracle.accept_tree(lg, draft, par, ctx)
    assert list(want[4][1:4]) == [11, 11, 11]
    got = run_tree(lg, draft, par, ctx, gpu, cluster)
    check_same(got, want)
    assert got[4] == 11
    # a length that would drop below zero stays as it is
    ctx2 = np.array([1] + [100] * (B - 1), np.int32)
    par_ok = random_parents(B, T, rng)
    lg2 = np.zeros((B, T, V), np.float32)  # argmax 0 everywhere
    draft2 = np.full((B, T - 1), 3, np.int32)  # nothing kept: a = 0 drops T-1 = 8
    got = run_tree(lg2, draft2, par_ok, ctx2, gpu, cluster)
    assert got[4] == 7 and got[3][0] == 1 and (got[3][1:] == 100 - (T - 1)).all()


def compaction_inputs(dtype, H, seed, T=12, B=7):
    """A batch whose T tree nodes sit at the end of each context, a random tree
    per sequence and the oracle's acceptance on planted logits."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(T, 200, size=B)
    ctx[0] = T  # the prefix is empty: base = 0
    w = small(B=B, T=T, N=4, K=2, H=H, dtype=dtype, ctx=tuple(int(c) for c in ctx), seed=seed)
    par = random_parents(B, T, rng, chain_bias=0.4)
    lg, draft = planted_tree_inputs(B, T, 11, par, rng, p_match=0.8)
    acc, nxt, path, ctx_after, err = oracle.accept_tree(lg, draft, par, w.context_lens)
    assert (err == 0).all() and acc.max() >= 2
    return w, acc, path, ctx_after


def bits(t):
    t = t.cpu()
    return t.view(torch.int16).numpy() if t.element_size() == 2 else t.numpy()


@pytest.mark.parametrize("dtype,H", [("f16", 64), ("bf16", 128)])
def test_compaction_matches_oracle_byte_for_byte(gpu, dtype, H):
    w, acc, path, ctx_after = compaction_inputs(dtype, H, seed=H)
    kc, vc, _, _, err = oracle.kv_compact(w.k_cache[0], w.v_cache[0], w.block_tables, ctx_after,
                                          path, acc, w.T)
    assert (err == 0).all()
    wd = to(w, gpu)
    st = torch.zeros(1, dtype=torch.int32, device=gpu)
    gq.kv_compact(wd.k_cache[0], wd.v_cache[0], wd.block_tables,
                  torch.as_tensor(ctx_after).to(gpu), torch.as_tensor(path).to(gpu),
                  torch.as_tensor(acc).to(gpu), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    np.testing.assert_array_equal(bits(wd.k_cache[0]).view(np.uint16), kc)
    np.testing.assert_array_equal(bits(wd.v_cache[0]).view(np.uint16), vc)


@pytest.mark.parametrize("kv", ["int8", "e4m3"])
def test_compaction_of_one_byte_caches_moves_the_scales(gpu, kv):
    w, acc, path, ctx_after = compaction_inputs("bf16", 128, seed=3)
    ck, sk = oracle.quantize_cache(w.k_cache[0], "bf16", kv)
    cv, sv = oracle.quantize_cache(w.v_cache[0], "bf16", kv)
    kc, vc, ks, vs, err = oracle.kv_compact(ck, cv, w.block_tables, ctx_after, path, acc, w.T,
                                            k_scale=sk, v_scale=sv)
    assert (err == 0).all()
    d = {n: torch.as_tensor(a).to(gpu) for n, a in
         (("ck", ck), ("cv", cv), ("sk", sk), ("sv", sv))}
    st = torch.zeros(1, dtype=torch.int32, device=gpu)
    gq.kv_compact(d["ck"], d["cv"], w.block_tables.to(gpu), torch.as_tensor(ctx_after).to(gpu),
                  torch.as_tensor(path).to(gpu), torch.as_tensor(acc).to(gpu),
                  k_scale=d["sk"], v_scale=d["sv"], kv=kv, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for name, want in (("ck", kc), ("cv", vc), ("sk", ks), ("sv", vs)):
        np.testing.assert_array_equal(d[name].cpu().numpy(), want)


def test_compaction_errors_leave_their_sequences_untouched(gpu):
    w, acc, path, ctx_after = compaction_inputs("f16", 64, seed=9)
    path = path.copy()
    ctx_after = ctx_after.copy()
    acc = acc.copy()
    bt = w.block_tables.clone()
    i2 = int(np.argmax(acc >= 2))
    path[i2, :2] = path[i2, 1], path[i2, 0]  # not increasing
    j = (i2 + 1) % w.B
    ctx_after[j] = acc[j]                     # base = -1
    k = (i2 + 2) % w.B
    base_k = int(ctx_after[k]) - 1 - int(acc[k])
    bt[k, (base_k + w.T - 1) // 16] = -5      # a tree node's block id out of range
    kc, vc, _, _, err = oracle.kv_compact(w.k_cache[0], w.v_cache[0], bt, ctx_after, path, acc,
                                          w.T)
    assert err[i2] == 11 and err[j] == 7 and err[k] == 8
    wd = to(w, gpu)
    st = torch.zeros(1, dtype=torch.int32, device=gpu)
    gq.kv_compact(wd.k_cache[0], wd.v_cache[0], bt.to(gpu), torch.as_tensor(ctx_after).to(gpu),
                  torch.as_tensor(path).to(gpu), torch.as_tensor(acc).to(gpu), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) in (7, 8, 11)
    np.testing.assert_array_equal(bits(wd.k_cache[0]).view(np.uint16), kc)
    np.testing.assert_array_equal(bits(wd.v_cache[0]).view(np.uint16), vc)


def test_tree_step_end_to_end_with_pdl_and_a_graph(gpu):
    """Fused append + tree verify, acceptance over the tree, compaction, then
    decode of the kept node's query over the compacted cache: caches and
    integers bit-exact with the oracle's chain of the same steps, attention
    within the parity bar, and the kept node's decode equal to its tree-verify
    row; the same step chained with PDL and replayed from a CUDA graph gives
    the same bits."""
    spec = workloads.SPECS["tree"]
    T = len(spec["tree"])
    rng = np.random.default_rng(17)
    ctx = rng.integers(40, 600, size=6)
    w = workloads.build("tree-small", B=6, T=T, N=16, K=2, H=128, dtype="bf16", ctx=ctx,
                        seed=17, append=True, vocab=1000, tree=spec["tree"])
    par = w.parents()
    mask = torch.from_numpy(w.tree_mask().view(np.int64).copy())
    # the oracle's chain of the same steps
    kc, vc, _ = oracle.kv_append(w.k_new[0], w.v_new[0], w.k_cache[0], w.v_cache[0],
                                 w.block_tables, w.context_lens)
    tdt = w.torch_dtype
    kct = torch.from_numpy(kc.view(np.int16)).view(tdt)
    vct = torch.from_numpy(vc.view(np.int16)).view(tdt)
    ref_tree, err = oracle.attention(w.q[0], kct, vct, w.block_tables, w.context_lens, "bf16",
                                     tree_mask=w.tree_mask())
    assert (err == 0).all()
    ra, rn, rp, rc, rerr = oracle.accept_tree(w.logits, w.draft, par, w.context_lens)
    assert (rerr == 0).all() and ra.max() >= 2
    kc2, vc2, _, _, cerr = oracle.kv_compact(kc, vc, w.block_tables, rc, rp, ra, T)
    assert (cerr == 0).all()

    def step(wd, ctx_d, outs, pdl):
        out_tree = gq.append_verify_attention(wd.q[0], wd.k_new[0], wd.v_new[0], wd.k_cache[0],
                                              wd.v_cache[0], wd.block_tables, ctx_d,
                                              tree_mask=mask_d, out=outs["tree"], pdl=pdl)
        gq.accept_tree(logits_d, draft_d, par_d, ctx_d, accepted=outs["acc"],
                       next_token=outs["nxt"], path=outs["path"])
        gq.kv_compact(wd.k_cache[0], wd.v_cache[0], wd.block_tables, ctx_d, outs["path"],
                      outs["acc"], pdl=pdl)
        return out_tree

    logits_d = w.logits.to(gpu)
    draft_d = w.draft.to(gpu)
    par_d = torch.as_tensor(par).to(gpu)
    mask_d = mask.to(gpu)

    def fresh():
        wd = to(w, gpu)
        outs = {"tree": torch.empty_like(wd.q[0]),
                "acc": torch.empty(w.B, dtype=torch.int32, device=gpu),
                "nxt": torch.empty(w.B, dtype=torch.int32, device=gpu),
                "path": torch.empty((w.B, T - 1), dtype=torch.int32, device=gpu)}
        return wd, wd.context_lens.clone(), outs

    wd, ctx_d, outs = fresh()
    step(wd, ctx_d, outs, pdl=False)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(outs["acc"].cpu().numpy(), ra)
    np.testing.assert_array_equal(outs["nxt"].cpu().numpy(), rn)
    np.testing.assert_array_equal(outs["path"].cpu().numpy(), rp)
    np.testing.assert_array_equal(ctx_d.cpu().numpy(), rc)
    np.testing.assert_array_equal(bits(wd.k_cache[0]).view(np.uint16), kc2)
    np.testing.assert_array_equal(bits(wd.v_cache[0]).view(np.uint16), vc2)
    assert_close(outs["tree"].float().cpu().double().numpy(), ref_tree, "bf16", "tree verify")
    # decode of each sequence's kept node over the compacted cache
    m = np.array([rp[b, ra[b] - 1] if ra[b] else 0 for b in range(w.B)])
    q1 = torch.stack([w.q[0][b, m[b]] for b in range(w.B)])[:, None].contiguous()
    dec = gq.decode_attention(q1.to(gpu), wd.k_cache[0], wd.v_cache[0], wd.block_tables, ctx_d)
    torch.cuda.synchronize()
    ref_dec, _ = oracle.attention(q1, torch.from_numpy(kc2.view(np.int16)).view(tdt),
                                  torch.from_numpy(vc2.view(np.int16)).view(tdt),
                                  w.block_tables, rc, "bf16")
    assert_close(dec.float().cpu().double().numpy(), ref_dec, "bf16", "decode after compaction")
    for b in range(w.B):  # the same keys in the same order as node m's tree row
        np.testing.assert_allclose(ref_dec[b, 0], ref_tree[b, m[b]], rtol=0, atol=1e-12)
    plain = [t.cpu() for t in (outs["tree"], outs["acc"], outs["path"], ctx_d,
                               wd.k_cache[0], wd.v_cache[0])]
    # chained with PDL, eagerly and from a CUDA graph
    for graph in (False, True):
        wd, ctx_d, outs = fresh()
        if graph:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):  # warm-up on copies (plans, workspaces)
                wd2, ctx2, outs2 = fresh()
                step(wd2, ctx2, outs2, pdl=True)
            torch.cuda.current_stream().wait_stream(s)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(wd, ctx_d, outs, pdl=True)
            g.replay()
        else:
            step(wd, ctx_d, outs, pdl=True)
        torch.cuda.synchronize()
        got = [t.cpu() for t in (outs["tree"], outs["acc"], outs["path"], ctx_d,
                                 wd.k_cache[0], wd.v_cache[0])]
        for a, b in zip(got, plain):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), graph
