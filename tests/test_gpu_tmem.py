"""GPU parity of the tensor-memory (tcgen05) attention kernel against the fp64
oracle: decode, verify and tree verify forced onto it, over ragged contexts,
row counts below, at and above one 128-row tile, both 16-bit dtypes, device
errors, the fused append, and the by-shape choice between the two kernels."""
import numpy as np
import pytest
import torch

import gqa_decode_attention_02_gb300 as gq
import oracle
from helpers import assert_close, set_token, small, to
from test_gpu_attention import as_i64, random_trees, tree_mask_rows

pytestmark = pytest.mark.gpu


def run(w, dev, engine="tmem", tree=None, status=None, pdl=False):
    wd = to(w, dev)
    kw = dict(status=status, engine=engine, pdl=pdl)
    if tree is not None:
        kw["tree_mask"] = as_i64(tree).to(dev)
    fn = gq.decode_attention if (w.T == 1 and tree is None) else gq.verify_attention
    out = fn(wd.q[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables, wd.context_lens, **kw)
    torch.cuda.synchronize()
    return out


def ref_of(w, tree=None):
    out, err = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                                w.context_lens, w.dtype, tree_mask=tree)
    return out, err


def as_np(out):
    return out.float().cpu().double().numpy()


CTX = (1, 2, 15, 16, 17, 63, 64, 65, 300, 4097)


@pytest.mark.parametrize("H", [128, 64])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("N,K", [(8, 8), (32, 8), (64, 8), (8, 1), (128, 1), (129, 1),
                                 (256, 2)])
def test_tmem_decode_matches_oracle(gpu, dtype, N, K, H):
    w = small(B=len(CTX), T=1, N=N, K=K, H=H, dtype=dtype, ctx=CTX, seed=3 * N + K + H)
    ref, err = ref_of(w)
    assert (err == 0).all()
    assert_close(as_np(run(w, gpu)), ref, dtype, f"tmem decode N={N} K={K} H={H}")


@pytest.mark.parametrize("H", [128, 64])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("T,N,K", [(2, 8, 2), (5, 64, 8), (8, 64, 8), (26, 64, 8),
                                   (64, 4, 4), (3, 16, 1), (17, 16, 2), (64, 8, 2), (5, 56, 8)])
def test_tmem_verify_matches_oracle(gpu, dtype, T, N, K, H):
    ctx = tuple(max(c, T) for c in (T, T + 1, 16, 17, 64, 65, 300, 2049))
    w = small(B=len(ctx), T=T, N=N, K=K, H=H, dtype=dtype, ctx=ctx, seed=T * 10 + N + K + H)
    ref, err = ref_of(w)
    assert (err == 0).all()
    assert_close(as_np(run(w, gpu)), ref, dtype, f"tmem verify T={T} N={N} K={K} H={H}")


@pytest.mark.parametrize("T,N,K,dtype,H", [(6, 64, 8, "bf16", 128), (26, 64, 8, "bf16", 128),
                                           (64, 2, 1, "f16", 128), (33, 8, 2, "bf16", 128),
                                           (4, 16, 2, "f16", 128), (6, 56, 8, "bf16", 64),
                                           (26, 64, 8, "f16", 64)])
def test_tmem_tree_matches_oracle(gpu, T, N, K, dtype, H):
    ctx = (T, T + 1, 16 + T, 300, 1029, 4100)
    w = small(B=len(ctx), T=T, N=N, K=K, H=H, dtype=dtype, ctx=ctx, seed=11 * T + N + H)
    m = random_trees(len(ctx), T, seed=T + 1)
    ref, err = ref_of(w, tree=m)
    assert (err == 0).all()
    assert_close(as_np(run(w, gpu, tree=m)), ref, dtype, f"tmem tree T={T} N={N} K={K}")


@pytest.mark.parametrize("first_new", [15, 16, 63, 64, 1023])
def test_tmem_tree_first_new_token_at_a_stage_edge(gpu, first_new):
    T = 4
    ctx = (first_new + T,) * 3
    w = small(B=3, T=T, N=64, K=2, H=128, dtype="f16", ctx=ctx, seed=first_new)
    m = np.zeros((3, T), np.uint64)
    m[1] = tree_mask_rows([-1, -1, 1, 2])
    m[2] = tree_mask_rows([-1, 0, 0, 0])
    ref, _ = ref_of(w, tree=m)
    assert_close(as_np(run(w, gpu, tree=m)), ref, "f16", f"tmem tree edge {first_new}")


def test_tmem_chain_mask_is_bit_identical_to_verify(gpu):
    T = 8
    ctx = (T, 40, 700, 3000)
    w = small(B=len(ctx), T=T, N=64, K=8, H=128, dtype="bf16", ctx=ctx, seed=61)
    chain = np.tile(np.array([(1 << t) - 1 for t in range(T)], np.uint64), (len(ctx), 1))
    junk = chain | np.tile(np.array([~np.uint64(0) << np.uint64(t) for t in range(T)],
                                    np.uint64), (len(ctx), 1))
    plain = run(w, gpu)
    assert torch.equal(plain, run(w, gpu, tree=chain))
    assert torch.equal(plain, run(w, gpu, tree=junk))


def test_tmem_scores_that_need_rescaling(gpu):
    """Large scores whose maximum moves late in the context: the running
    maximum is raised (and O rescaled in tensor memory) in later stages."""
    ctx = (70, 700, 3000)
    w = small(B=len(ctx), T=4, N=64, K=8, H=128, dtype="bf16", ctx=ctx, seed=62)
    w.q[0] *= 6
    H = 128
    for b, c in enumerate(ctx):
        for pos in (c // 3, c // 2, c - 9, c - 5):  # keys aligned with some queries
            k = (w.q[0][b, 0, 8 * (pos % 8)].double() * (0.2 + pos / c)).numpy()
            set_token(w, b, pos, k=k[:H])
    ref, err = ref_of(w)
    assert (err == 0).all()
    assert_close(as_np(run(w, gpu)), ref, "bf16", "tmem rescale")


def test_tmem_device_errors_zero_the_sequence_and_set_status(gpu):
    w = small(B=4, T=2, N=64, K=2, H=128, dtype="bf16", ctx=(1, 40, 200, 200), seed=63)
    w.block_tables[2, 9] = w.num_blocks + 3  # bad id inside sequence 2's context
    w.block_tables[3, 0] = -1
    ref, err = ref_of(w)
    assert list(err) == [7, 0, 8, 8]
    st = torch.zeros(1, dtype=torch.int32, device=gpu)
    got = as_np(run(w, gpu, status=st))
    assert int(st.item()) in (7, 8)
    assert (got[0] == 0).all() and (got[2] == 0).all() and (got[3] == 0).all()
    assert_close(got[1], ref[1], "bf16", "healthy sequence next to bad ones")


def test_tmem_poisoned_slots_past_the_context_are_not_read(gpu):
    """Cache rows past each context (in the last block and the stage's other
    blocks) hold NaN: the output stays finite and equal to the oracle's."""
    ctx = (17, 65, 130)
    w = small(B=3, T=3, N=64, K=8, H=128, dtype="bf16", ctx=ctx, seed=64)
    nan = np.full(128 * 8, np.nan).reshape(8, 128)
    for b, c in enumerate(ctx):
        for pos in range(c, (c + 15) // 16 * 16):
            blk = int(w.block_tables[b, pos // 16])
            w.k_cache[0][blk, pos % 16] = torch.from_numpy(nan).to(w.torch_dtype)
            w.v_cache[0][blk, pos % 16] = torch.from_numpy(nan).to(w.torch_dtype)
    ref, err = ref_of(w)
    assert (err == 0).all()
    assert_close(as_np(run(w, gpu)), ref, "bf16", "tmem poisoned tail")


@pytest.mark.parametrize("H", [128, 64])
@pytest.mark.parametrize("tree", [False, True])
def test_tmem_fused_append_matches_oracle(gpu, tree, H):
    T = 8
    ctx = (T, 70, 333, 2000)
    w = small(B=len(ctx), T=T, N=64, K=8, H=H, dtype="bf16", ctx=ctx, seed=65 + H, append=True)
    m = random_trees(len(ctx), T, seed=3) if tree else None
    kc, vc, _ = oracle.kv_append(w.k_new[0], w.v_new[0], w.k_cache[0], w.v_cache[0],
                                 w.block_tables, w.context_lens)
    kt = torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16)
    vt = torch.from_numpy(vc.view(np.int16)).view(torch.bfloat16)
    ref, err = oracle.attention(w.q[0], kt, vt, w.block_tables, w.context_lens, "bf16",
                                tree_mask=m)
    assert (err == 0).all()
    wd = to(w, gpu)
    kw = {} if m is None else {"tree_mask": as_i64(m).to(gpu)}
    out = gq.append_verify_attention(wd.q[0], wd.k_new[0], wd.v_new[0], wd.k_cache[0],
                                     wd.v_cache[0], wd.block_tables, wd.context_lens,
                                     engine="tmem", pdl=True, **kw)
    torch.cuda.synchronize()
    assert_close(as_np(out), ref, "bf16", "tmem fused append")
    np.testing.assert_array_equal(wd.k_cache[0].cpu().view(torch.int16).numpy().view(np.uint16),
                                  kc)
    np.testing.assert_array_equal(wd.v_cache[0].cpu().view(torch.int16).numpy().view(np.uint16),
                                  vc)


@pytest.mark.parametrize("tree", [False, True])
def test_tmem_early_kv_after_append_is_bit_identical(gpu, tree):
    """The fused append with PDL and early KV streaming (older positions read
    while the append kernel may still run), eager and replayed from a CUDA
    graph, equals the plain append followed by plain attention bit for bit."""
    T = 5
    ctx = (T, 17, 300, 2049, 4096)
    w = small(B=len(ctx), T=T, N=64, K=8, H=128, dtype="bf16", ctx=ctx, seed=67, append=True)
    m = random_trees(len(ctx), T, seed=5) if tree else None
    kw = {} if m is None else {"tree_mask": as_i64(m).to(gpu)}
    wp = to(w, gpu)
    gq.kv_append(wp.k_new[0], wp.v_new[0], wp.k_cache[0], wp.v_cache[0], wp.block_tables,
                 wp.context_lens)
    plain = gq.verify_attention(wp.q[0], wp.k_cache[0], wp.v_cache[0], wp.block_tables,
                                wp.context_lens, engine="tmem", **kw)
    for use_graph in (False, True):
        we = to(w, gpu)
        args = (we.q[0], we.k_new[0], we.v_new[0], we.k_cache[0], we.v_cache[0],
                we.block_tables, we.context_lens)
        out = torch.empty_like(we.q[0])
        if not use_graph:
            gq.append_verify_attention(*args, out=out, engine="tmem", pdl=True, early_kv=True,
                                       **kw)
        else:
            gq.append_verify_attention(*args, out=out, engine="tmem", **kw)  # outside capture
            torch.cuda.synchronize()
            we = to(w, gpu)  # fresh caches: the graph appends again
            args = (we.q[0], we.k_new[0], we.v_new[0], we.k_cache[0], we.v_cache[0],
                    we.block_tables, we.context_lens)
            g = torch.cuda.CUDAGraph()
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                with torch.cuda.graph(g, stream=st):
                    gq.append_verify_attention(*args, out=out, engine="tmem", pdl=True,
                                               early_kv=True, **kw)
            out.zero_()
            g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, plain), use_graph
        # bit patterns: unused cache slots hold NaN sentinels
        for a, b in ((we.k_cache[0], wp.k_cache[0]), (we.v_cache[0], wp.v_cache[0])):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), use_graph


def test_engine_choice_by_shape(gpu):
    """auto = tensor memory from 32 rows per KV head, a warp-level kernel
    below: bit-identical to the forced engine in each case."""
    for T, N, K in ((1, 32, 8), (3, 64, 8), (4, 64, 8), (5, 64, 8), (1, 64, 1), (26, 64, 8)):
        ctx = tuple(max(c, T) for c in (1, 100, 2000))
        w = small(B=3, T=T, N=N, K=K, H=128, dtype="bf16", ctx=ctx, seed=T + N)
        auto = run(w, gpu, engine="auto")
        pick = gq.attention_engine(w.q[0], w.k_cache[0], w.block_tables)
        assert (pick == "tmem") == (T * (N // K) >= 32), (T, N, K, pick)
        assert torch.equal(auto, run(w, gpu, engine=pick)), (T, N, K)


def test_tmem_pdl_and_graph_match_plain(gpu):
    T = 5
    ctx = (T, 800, 3000)
    w = small(B=3, T=T, N=64, K=8, H=128, dtype="bf16", ctx=ctx, seed=66)
    plain = run(w, gpu)
    assert torch.equal(plain, run(w, gpu, pdl=True))
    wd = to(w, gpu)
    out = torch.empty_like(wd.q[0])
    args = (wd.q[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables, wd.context_lens)
    gq.verify_attention(*args, out=out, engine="tmem")  # first call outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            gq.verify_attention(*args, out=out, engine="tmem", pdl=True)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, plain)


def test_tmem_empty_batch_and_unknown_engine(gpu):
    w = small(B=1, T=1, N=8, K=2, H=128, dtype="bf16", ctx=(5,), seed=67)
    wd = to(w, gpu)
    q0 = wd.q[0][:0]
    out = gq.decode_attention(q0, wd.k_cache[0], wd.v_cache[0], wd.block_tables[:0],
                              wd.context_lens[:0], engine="tmem")
    assert out.shape[0] == 0
    with pytest.raises(ValueError):
        run(w, gpu, engine="both")


@pytest.mark.parametrize("H", [128, 64])
def test_tmem_long_sequences_split_across_many_ctas(gpu, H):
    """Segments far longer than one CTA's share: pieces on many CTAs merged
    with log-sum-exp weights, next to short whole segments; a second call on
    the same workspace is bit-identical and leaves the flags at zero."""
    ctx = (30000, 5, 17000, 64, 1)
    w = small(B=len(ctx), T=1, N=32, K=8, H=H, dtype="bf16", ctx=ctx, seed=69 + H)
    ref, err = ref_of(w)
    assert (err == 0).all()
    wd = to(w, gpu)
    args = (wd.q[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables, wd.context_lens)
    nbytes = gq.attention_workspace_size(wd.q[0], wd.k_cache[0], wd.block_tables)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=gpu)
    a = gq.decode_attention(*args, workspace=ws, engine="tmem")
    b = gq.decode_attention(*args, workspace=ws, engine="tmem")
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert int(ws[: 256 * 1024].view(torch.int32).abs().sum().item()) == 0
    assert_close(as_np(a), ref, "bf16", "tmem split pieces")


def test_tmem_bad_block_in_a_split_segment(gpu):
    ctx = (20000, 300, 20000)
    w = small(B=3, T=2, N=64, K=8, H=128, dtype="bf16", ctx=ctx, seed=70)
    w.block_tables[2, 700] = -5
    ref, err = ref_of(w)
    assert list(err) == [0, 0, 8]
    st = torch.zeros(1, dtype=torch.int32, device=gpu)
    got = as_np(run(w, gpu, status=st))
    assert int(st.item()) == 8
    assert (got[2] == 0).all()
    assert_close(got[:2], ref[:2], "bf16", "healthy sequences next to a split bad one")


# ---- local attention on the tensor-memory kernel ---------------------------------
@pytest.mark.parametrize("T,N,K,H", [(5, 64, 8, 128), (1, 64, 1, 128), (26, 64, 8, 128),
                                     (5, 56, 8, 64)])
@pytest.mark.parametrize("W", [1, 15, 16, 17, 100, 1024])
def test_tmem_window_matches_oracle(gpu, T, N, K, H, W):
    ctx = tuple(max(c, T) for c in (1, 2, 15, 16, 17, 31, 295, 1029, 4097))
    w = small(B=len(ctx), T=T, N=N, K=K, H=H, dtype="bf16", ctx=ctx, seed=W + T + N + H)
    ref, err = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                                w.context_lens, "bf16", window=W)
    assert (err == 0).all()
    wd = to(w, gpu)
    fn = gq.decode_attention if T == 1 else gq.verify_attention
    st = torch.zeros(1, dtype=torch.int32, device=gpu)
    out = fn(wd.q[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables, wd.context_lens,
             window=W, engine="tmem", status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_close(out.float().cpu().double().numpy(), ref, "bf16", f"tmem window {W} T={T}")
    # the warp-level kernel on the same call: the same function
    warp = fn(wd.q[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables, wd.context_lens,
              window=W, engine="warp")
    torch.cuda.synchronize()
    assert_close(out.float().cpu().double().numpy(), warp.float().cpu().double().numpy(),
                 "bf16", "tmem vs warp, window")


def test_tmem_window_ignores_poisoned_rows_and_freed_blocks(gpu):
    """NaN in every position below the earliest window (keys and values) and
    INT32_MAX in the table entries of blocks no query sees: the same result as
    the clean cache, no error, on the tensor-memory kernel."""
    T, W = 5, 40
    ctx = (T, 45, 64, 300, 1000)
    w = small(B=len(ctx), T=T, N=64, K=8, H=128, dtype="bf16", ctx=ctx, seed=177)
    ref, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                              w.context_lens, "bf16", window=W)
    tables = w.block_tables.clone()
    for b, c in enumerate(ctx):
        first = max(0, c - T - W + 1)
        for pos in range(first):
            set_token(w, b, pos, k=torch.full((8, 128), float("nan")),
                      v=torch.full((8, 128), float("nan")))
        tables[b, : first // 16] = 2**31 - 1
    wd = to(w, gpu)
    st = torch.zeros(1, dtype=torch.int32, device=gpu)
    out = gq.verify_attention(wd.q[0], wd.k_cache[0], wd.v_cache[0], tables.to(gpu),
                              wd.context_lens, window=W, engine="tmem", status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = out.float().cpu().double().numpy()
    assert np.isfinite(got).all()
    assert_close(got, ref, "bf16", "tmem, poisoned window")


def test_tmem_window_fused_append_pdl_early_matches_oracle(gpu):
    """The append and windowed verify in one call, plain and with PDL and early
    KV reads: the oracle's result, and the same bits either way."""
    T, W = 5, 100
    ctx = (T, 17, 300, 2000, 64)
    w = small(B=len(ctx), T=T, N=64, K=8, H=128, dtype="bf16", ctx=ctx, seed=41, append=True)
    kc, vc, err = oracle.kv_append(w.k_new[0], w.v_new[0], w.k_cache[0], w.v_cache[0],
                                   w.block_tables, w.context_lens)
    assert (err == 0).all()
    ref, _ = oracle.attention(w.q[0], torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16),
                              torch.from_numpy(vc.view(np.int16)).view(torch.bfloat16),
                              w.block_tables, w.context_lens, "bf16", window=W)
    outs = []
    for flags in (dict(), dict(pdl=True, early_kv=True)):
        wd = to(w, gpu)
        out = gq.append_verify_attention(wd.q[0], wd.k_new[0], wd.v_new[0], wd.k_cache[0],
                                         wd.v_cache[0], wd.block_tables, wd.context_lens,
                                         window=W, engine="tmem", **flags)
        torch.cuda.synchronize()
        assert_close(out.float().cpu().double().numpy(), ref, "bf16", f"fused window {flags}")
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
