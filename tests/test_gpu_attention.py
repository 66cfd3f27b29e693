"""GPU parity of kv_append, decode_attention and verify_attention against the
fp64 oracle, element by element, at sizes the oracle finishes in seconds that
still span many 16-token tiles, several split pieces and ragged tails."""
import numpy as np
import pytest
import torch

import gqa_decode_attention_02_gb300 as gq
import oracle
from helpers import assert_close, set_token, small, to

pytestmark = pytest.mark.gpu


def run_attention(w, dev, fn=None, status=None):
    wd = to(w, dev)
    fn = fn or (gq.decode_attention if w.T == 1 else gq.verify_attention)
    out = fn(wd.q[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables, wd.context_lens,
             status=status)
    torch.cuda.synchronize()
    return out.float().cpu().double().numpy()


def oracle_out(w):
    out, err = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                                w.context_lens, w.dtype)
    return out, err


CTX_MIX = (1, 2, 15, 16, 17, 31, 295, 4097)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("H", [64, 128])
@pytest.mark.parametrize("N,K", [(1, 1), (8, 8), (14, 2), (32, 8), (64, 8), (8, 1)])
def test_decode_matches_oracle(gpu, dtype, H, N, K):
    w = small(B=len(CTX_MIX), T=1, N=N, K=K, H=H, dtype=dtype, ctx=CTX_MIX,
              seed=H + 7 * N + 131 * K + (dtype == "bf16"))
    ref, err = oracle_out(w)
    assert (err == 0).all()
    got = run_attention(w, gpu)
    assert_close(got, ref, dtype, f"decode {dtype} H={H} N={N} K={K}")


@pytest.mark.parametrize("T,N,K", [(2, 8, 2), (5, 64, 8), (3, 16, 1), (4, 12, 4), (6, 8, 1)])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_verify_matches_oracle(gpu, T, N, K, dtype):
    ctx = (T, T + 1, 16, 17, 33, 300, 1029)
    w = small(B=len(ctx), T=T, N=N, K=K, H=128, dtype=dtype, ctx=ctx, seed=T * 100 + N)
    ref, err = oracle_out(w)
    assert (err == 0).all()
    got = run_attention(w, gpu)
    assert_close(got, ref, dtype, f"verify T={T} N={N} K={K}")


def test_decode_entry_point_rejects_t_above_one(gpu):
    w = small(B=2, T=2, N=8, K=2, H=64, ctx=(4, 9), seed=1)
    with pytest.raises(gq.GqaError):
        run_attention(w, gpu, fn=gq.decode_attention)


@pytest.mark.parametrize("dtype,H", [("f16", 64), ("bf16", 128)])
def test_kv_append_bit_exact(gpu, dtype, H):
    ctx = (1, 3, 16, 17, 31, 32, 33, 500)
    for T in (1, 3):
        ctx_t = tuple(max(c, T) for c in ctx)  # at least the T new tokens
        w = small(B=len(ctx), T=T, N=8, K=4, H=H, dtype=dtype, ctx=ctx_t, seed=T, append=True)
        kc, vc, err = oracle.kv_append(w.k_new[0], w.v_new[0], w.k_cache[0], w.v_cache[0],
                                       w.block_tables, w.context_lens)
        assert (err == 0).all()
        wd = to(w, gpu)
        gq.kv_append(wd.k_new[0], wd.v_new[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables,
                     wd.context_lens)
        torch.cuda.synchronize()
        gk = wd.k_cache[0].cpu().view(torch.int16).numpy().view(np.uint16)
        gv = wd.v_cache[0].cpu().view(torch.int16).numpy().view(np.uint16)
        np.testing.assert_array_equal(gk, kc)  # every byte, sentinels included
        np.testing.assert_array_equal(gv, vc)


def test_append_then_attend_equals_oracle(gpu):
    w = small(B=5, T=3, N=32, K=8, H=128, dtype="bf16", ctx=(3, 16, 17, 250, 1000),
              seed=21, append=True)
    kc, vc, _ = oracle.kv_append(w.k_new[0], w.v_new[0], w.k_cache[0], w.v_cache[0],
                                 w.block_tables, w.context_lens)
    kc_t = torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16)
    vc_t = torch.from_numpy(vc.view(np.int16)).view(torch.bfloat16)
    ref, _ = oracle.attention(w.q[0], kc_t, vc_t, w.block_tables, w.context_lens, "bf16")
    wd = to(w, gpu)
    gq.kv_append(wd.k_new[0], wd.v_new[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables,
                 wd.context_lens)
    out = gq.verify_attention(wd.q[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables,
                              wd.context_lens)
    torch.cuda.synchronize()
    assert_close(out.float().cpu().double().numpy(), ref, "bf16", "append+verify")


def test_shared_prefix_blocks(gpu):
    # copy-on-write prefix sharing: several tables point at the same blocks.
    w = small(B=4, T=1, N=8, K=2, H=64, ctx=(64, 64, 64, 64), seed=5)
    w.block_tables[1, :2] = w.block_tables[0, :2]
    w.block_tables[2, :3] = w.block_tables[0, :3]
    w.block_tables[3, :] = w.block_tables[0, :]
    ref, _ = oracle_out(w)
    got = run_attention(w, gpu)
    assert_close(got, ref, "f16", "shared blocks")


def test_block_permutation_and_repeat_are_bit_identical(gpu):
    w = small(B=6, T=1, N=32, K=8, H=128, dtype="bf16", ctx=(5, 700, 1500, 33, 16, 2000),
              seed=6, spare=4)
    a = run_attention(w, gpu)
    b = run_attention(w, gpu)
    np.testing.assert_array_equal(a, b)  # deterministic merge order
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(1))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(w.num_blocks)
    w.k_cache[0] = w.k_cache[0][perm].contiguous()
    w.v_cache[0] = w.v_cache[0][perm].contiguous()
    used = w.block_tables != 2**31 - 1
    w.block_tables[used] = inv[w.block_tables[used].long()].int()
    c = run_attention(w, gpu)
    np.testing.assert_array_equal(a, c)


def test_device_errors_zero_the_sequence_and_set_status(gpu):
    w = small(B=4, T=2, N=8, K=2, H=64, ctx=(1, 40, 40, 40), seed=7)
    w.block_tables[2, 1] = w.num_blocks + 3  # bad id inside sequence 2's context
    w.block_tables[3, 0] = -1                # bad id in sequence 3
    ref, err = oracle_out(w)
    assert list(err) == [7, 0, 8, 8]
    st = torch.zeros(1, dtype=torch.int32, device=gpu)
    got = run_attention(w, gpu, status=st)
    assert int(st.item()) in (7, 8)
    assert (got[0] == 0).all() and (got[2] == 0).all() and (got[3] == 0).all()
    assert_close(got[1], ref[1], "f16", "healthy sequence next to bad ones")


def test_workspace_flags_return_to_zero(gpu):
    w = small(B=3, T=1, N=32, K=8, H=128, dtype="bf16", ctx=(3000, 5000, 40), seed=8)
    wd = to(w, gpu)
    n = gq.attention_workspace_size(wd.q[0], wd.k_cache[0], wd.block_tables)
    ws = torch.zeros(n, dtype=torch.uint8, device=gpu)
    for _ in range(3):
        gq.decode_attention(wd.q[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables,
                            wd.context_lens, workspace=ws)
    torch.cuda.synchronize()
    flags = ws[: 65536 * 4].view(torch.int32)  # the fixed publication-flag region
    assert int(flags.abs().sum().item()) == 0


def test_workspace_shared_by_shapes_of_different_sizes(gpu):
    # one buffer, a small-batch call (leaves partial results behind) and then
    # a large-batch call: the second must still find its flags at zero.
    cases = [small(B=B, T=1, N=8, K=2, H=64, ctx=ctx, seed=seed) for B, ctx, seed in
             ((2, (3000, 2500), 1), (40, tuple(range(700, 700 + 40 * 37, 37)), 2))]
    ws = None
    for w in cases:
        wd = to(w, gpu)
        if ws is None:
            n = max(gq.attention_workspace_size(c.q[0].to(gpu), c.k_cache[0].to(gpu),
                                                c.block_tables.to(gpu)) for c in cases)
            ws = torch.zeros(n, dtype=torch.uint8, device=gpu)
        out = gq.decode_attention(wd.q[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables,
                                  wd.context_lens, workspace=ws)
        torch.cuda.synchronize()
        ref, _ = oracle_out(w)
        assert_close(out.cpu().double().numpy(), ref, "f16", f"B={w.B}")


def test_empty_batch(gpu):
    q = torch.empty(0, 1, 8, 64, dtype=torch.float16, device=gpu)
    kc = torch.zeros(4, 16, 2, 64, dtype=torch.float16, device=gpu)
    bt = torch.zeros(0, 2, dtype=torch.int32, device=gpu)
    cl = torch.zeros(0, dtype=torch.int32, device=gpu)
    out = gq.decode_attention(q, kc, kc, bt, cl)
    assert out.shape == (0, 1, 8, 64)


def test_long_single_sequence_many_pieces(gpu):
    # one sequence, 32k tokens: the whole grid splits one segment per KV head.
    w = small(B=1, T=1, N=8, K=1, H=128, dtype="bf16", ctx=(32768,), seed=9)
    ref, _ = oracle_out(w)
    got = run_attention(w, gpu)
    assert_close(got, ref, "bf16", "32k context")


@pytest.mark.parametrize("T", [1, 5])
def test_pdl_and_early_kv_launches_match_plain_ones(gpu, T):
    # The same append + attention sequence over three layers, launched plainly
    # and with programmatic dependent launch / early KV reads, eagerly and from
    # a CUDA graph: identical bits.
    ctx = (T, 17, 300, 2000, 64)
    layers = 3
    w = small(B=5, T=T, N=32, K=8, H=128, dtype="bf16", ctx=ctx, seed=40 + T, append=True,
              layers=layers)
    fn = gq.decode_attention if T == 1 else gq.verify_attention

    def run(flags, graph):
        wd = to(w, gpu)
        outs = [torch.empty_like(q) for q in wd.q]
        ws = torch.zeros(gq.attention_workspace_size(wd.q[0], wd.k_cache[0], wd.block_tables),
                         dtype=torch.uint8, device=gpu)

        def step():
            for l in range(layers):
                gq.kv_append(wd.k_new[l], wd.v_new[l], wd.k_cache[l], wd.v_cache[l],
                             wd.block_tables, wd.context_lens, pdl=flags["pdl"])
                fn(wd.q[l], wd.k_cache[l], wd.v_cache[l], wd.block_tables, wd.context_lens,
                   out=outs[l], workspace=ws, **flags)

        if graph:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                step()  # warm-up (plans)
            torch.cuda.current_stream().wait_stream(s)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step()
            g.replay()
        else:
            step()
        torch.cuda.synchronize()
        return [o.cpu() for o in outs]

    ref = run(dict(pdl=False, early_kv=False), graph=False)
    for flags in (dict(pdl=True, early_kv=False), dict(pdl=True, early_kv=True)):
        for graph in (False, True):
            got = run(flags, graph)
            for l in range(layers):
                assert torch.equal(got[l].view(torch.int16), ref[l].view(torch.int16)), (
                    flags, graph, l)
    # and the plain result matches the oracle
    kc, vc, _ = oracle.kv_append(w.k_new[0], w.v_new[0], w.k_cache[0], w.v_cache[0],
                                 w.block_tables, w.context_lens)
    kc = torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16)
    vc = torch.from_numpy(vc.view(np.int16)).view(torch.bfloat16)
    o, _ = oracle.attention(w.q[0], kc, vc, w.block_tables, w.context_lens, "bf16")
    assert_close(ref[0].double().numpy(), o, "bf16", "layer 0")


def test_many_tiny_sequences_with_gaps(gpu):
    # 20000 one-block sequences (so each CTA range spans dozens of sequences and
    # the look-ahead windows of lengths and block ids roll over), some of them
    # empty (skipped, zeroed, reported).
    rng = np.random.default_rng(11)
    B = 20000
    ctx = rng.integers(1, 17, size=B)
    ctx[rng.choice(B, size=200, replace=False)] = 0
    w = small(B=B, T=1, N=2, K=1, H=64, ctx=np.maximum(ctx, 1), seed=12)
    w.context_lens[torch.as_tensor(ctx == 0)] = 0
    ref, err = oracle_out(w)
    assert (err[ctx == 0] == 7).all() and (err[ctx > 0] == 0).all()
    st = torch.zeros(1, dtype=torch.int32, device=gpu)
    got = run_attention(w, gpu, status=st)
    assert int(st.item()) == 7
    assert (got[ctx == 0] == 0).all()
    assert_close(got[ctx > 0], ref[ctx > 0], "f16", "tiny sequences")


@pytest.mark.parametrize("T,N,K,H,dtype,ctx", [
    (1, 32, 8, 128, "bf16", (1, 2, 16, 17, 33, 300, 4097)),
    (1, 14, 2, 64, "f16", (1, 15, 16, 17, 295, 1024)),
    (5, 64, 8, 128, "bf16", (5, 6, 16, 19, 20, 33, 512, 4096)),  # new tokens straddle blocks
    (3, 16, 1, 64, "f16", (3, 17, 18, 100)),
])
def test_fused_append_equals_append_then_attention(gpu, T, N, K, H, dtype, ctx):
    w = small(B=len(ctx), T=T, N=N, K=K, H=H, dtype=dtype, ctx=ctx, seed=T * 7 + H, append=True)
    # oracle: append, then attention
    kc, vc, err = oracle.kv_append(w.k_new[0], w.v_new[0], w.k_cache[0], w.v_cache[0],
                                   w.block_tables, w.context_lens)
    assert (err == 0).all()
    tdt = w.torch_dtype
    ref, _ = oracle.attention(w.q[0], torch.from_numpy(kc.view(np.int16)).view(tdt),
                              torch.from_numpy(vc.view(np.int16)).view(tdt), w.block_tables,
                              w.context_lens, dtype)
    # GPU: unfused pair, then the fused call on a fresh copy of the caches
    a = to(w, gpu)
    gq.kv_append(a.k_new[0], a.v_new[0], a.k_cache[0], a.v_cache[0], a.block_tables,
                 a.context_lens)
    fn = gq.decode_attention if T == 1 else gq.verify_attention
    out_pair = fn(a.q[0], a.k_cache[0], a.v_cache[0], a.block_tables, a.context_lens)
    b = to(w, gpu)
    ffn = gq.append_decode_attention if T == 1 else gq.append_verify_attention
    st = torch.zeros(1, dtype=torch.int32, device=gpu)
    out_fused = ffn(b.q[0], b.k_new[0], b.v_new[0], b.k_cache[0], b.v_cache[0], b.block_tables,
                    b.context_lens, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for mine, theirs in ((b.k_cache[0], kc), (b.v_cache[0], vc)):  # every cache byte
        np.testing.assert_array_equal(mine.cpu().view(torch.int16).numpy().view(np.uint16),
                                      theirs)
    assert torch.equal(out_fused.view(torch.int16), out_pair.view(torch.int16))
    assert_close(out_fused.float().cpu().double().numpy(), ref, dtype, "fused append")


@pytest.mark.parametrize("T", [1, 5])
def test_fused_append_pdl_early_graph_matches_plain(gpu, T):
    ctx = (T, 17, 300, 2000, 64)
    layers = 3
    w = small(B=5, T=T, N=32, K=8, H=128, dtype="bf16", ctx=ctx, seed=50 + T, append=True,
              layers=layers)
    ffn = gq.append_decode_attention if T == 1 else gq.append_verify_attention

    def run(flags, graph):
        wd = to(w, gpu)
        outs = [torch.empty_like(q) for q in wd.q]
        ws = torch.zeros(gq.attention_workspace_size(wd.q[0], wd.k_cache[0], wd.block_tables),
                         dtype=torch.uint8, device=gpu)

        def step():
            for l in range(layers):
                ffn(wd.q[l], wd.k_new[l], wd.v_new[l], wd.k_cache[l], wd.v_cache[l],
                    wd.block_tables, wd.context_lens, out=outs[l], workspace=ws, **flags)

        if graph:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                step()
            torch.cuda.current_stream().wait_stream(s)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step()
            g.replay()
        else:
            step()
        torch.cuda.synchronize()
        return [o.cpu() for o in outs], [c.cpu() for c in wd.k_cache]

    ref, ref_k = run(dict(pdl=False, early_kv=False), graph=False)
    for flags in (dict(pdl=True, early_kv=False), dict(pdl=True, early_kv=True)):
        for graph in (False, True):
            got, got_k = run(flags, graph)
            for l in range(layers):
                assert torch.equal(got[l].view(torch.int16), ref[l].view(torch.int16))
                assert torch.equal(got_k[l].view(torch.int16), ref_k[l].view(torch.int16))


# ---- local (sliding-window) attention --------------------------------------------
def oracle_window(w, W, tables=None):
    return oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0],
                            w.block_tables if tables is None else tables, w.context_lens,
                            w.dtype, window=W)


@pytest.mark.parametrize("T,N,K,H,dtype", [(1, 32, 8, 128, "bf16"), (1, 14, 2, 64, "f16"),
                                           (5, 64, 8, 128, "bf16"), (3, 16, 1, 64, "f16")])
@pytest.mark.parametrize("W", [1, 15, 16, 17, 100, 1024])
def test_window_matches_oracle(gpu, T, N, K, H, dtype, W):
    ctx = tuple(max(c, T) for c in (1, 2, 15, 16, 17, 31, 295, 1029, 4097))
    w = small(B=len(ctx), T=T, N=N, K=K, H=H, dtype=dtype, ctx=ctx, seed=W + 13 * T + N)
    ref, err = oracle_window(w, W)
    assert (err == 0).all()
    wd = to(w, gpu)
    fn = gq.decode_attention if T == 1 else gq.verify_attention
    out = fn(wd.q[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables, wd.context_lens, window=W)
    torch.cuda.synchronize()
    assert_close(out.float().cpu().double().numpy(), ref, dtype, f"window {W} T={T}")


@pytest.mark.parametrize("T", [1, 4])
def test_window_ignores_poisoned_and_freed_blocks(gpu, T):
    """NaN in every position below the earliest window and INT32_MAX in the
    table entries of blocks no query sees: same result, no error."""
    W = 40
    ctx = (T, 45, 64, 300, 1000)
    w = small(B=len(ctx), T=T, N=8, K=2, H=128, dtype="bf16", ctx=ctx, seed=77 + T)
    ref, _ = oracle_window(w, W)
    tables = w.block_tables.clone()
    for b, c in enumerate(ctx):
        first = max(0, c - T - W + 1)
        for pos in range(first):
            set_token(w, b, pos, k=torch.full((2, 128), float("nan")),
                      v=torch.full((2, 128), float("nan")))
        tables[b, : first // 16] = 2**31 - 1
    ref2, err = oracle_window(w, W, tables)
    assert (err == 0).all()
    np.testing.assert_array_equal(ref2, ref)
    wd = to(w, gpu)
    st = torch.zeros(1, dtype=torch.int32, device=gpu)
    fn = gq.decode_attention if T == 1 else gq.verify_attention
    out = fn(wd.q[0], wd.k_cache[0], wd.v_cache[0], tables.to(gpu), wd.context_lens, window=W,
             status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = out.float().cpu().double().numpy()
    assert np.isfinite(got).all()
    assert_close(got, ref, "bf16", "poisoned window")


def test_window_bad_block_inside_window_is_reported(gpu):
    T, W = 3, 20
    w = small(B=2, T=T, N=4, K=2, H=64, ctx=(36, 38), seed=36)
    tables = w.block_tables.clone()
    tables[:, 0] = -1  # seen by query 0 of sequence 0 only
    ref, err = oracle_window(w, W, tables)
    assert err.tolist() == [8, 0]
    wd = to(w, gpu)
    st = torch.zeros(1, dtype=torch.int32, device=gpu)
    out = gq.verify_attention(wd.q[0], wd.k_cache[0], wd.v_cache[0], tables.to(gpu),
                              wd.context_lens, window=W, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 8
    got = out.float().cpu().double().numpy()
    assert (got[0] == 0).all()
    assert_close(got[1:], ref[1:], "f16", "bad block in window")


@pytest.mark.parametrize("T", [1, 5])
def test_window_fused_append_matches_oracle(gpu, T):
    W = 64
    ctx = (T, 70, 333, 2000)
    w = small(B=len(ctx), T=T, N=64 if T == 5 else 32, K=8, H=128, dtype="bf16", ctx=ctx,
              seed=91 + T, append=True)
    kc, vc, _ = oracle.kv_append(w.k_new[0], w.v_new[0], w.k_cache[0], w.v_cache[0],
                                 w.block_tables, w.context_lens)
    kt = torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16)
    vt = torch.from_numpy(vc.view(np.int16)).view(torch.bfloat16)
    ref, err = oracle.attention(w.q[0], kt, vt, w.block_tables, w.context_lens, "bf16",
                                window=W)
    assert (err == 0).all()
    wd = to(w, gpu)
    fn = gq.append_decode_attention if T == 1 else gq.append_verify_attention
    out = fn(wd.q[0], wd.k_new[0], wd.v_new[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables,
             wd.context_lens, window=W)
    torch.cuda.synchronize()
    assert_close(out.float().cpu().double().numpy(), ref, "bf16", f"fused window T={T}")
    np.testing.assert_array_equal(wd.k_cache[0].cpu().view(torch.int16).numpy().view(np.uint16),
                                  kc)


def test_window_of_int_max_is_full_attention(gpu):
    w = small(B=3, T=2, N=8, K=2, H=64, dtype="f16", ctx=(2, 40, 1000), seed=5)
    ref, _ = oracle_out(w)
    wd = to(w, gpu)
    out = gq.verify_attention(wd.q[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables,
                              wd.context_lens, window=2**31 - 1)
    torch.cuda.synchronize()
    assert_close(out.float().cpu().double().numpy(), ref, "f16", "window INT_MAX")


# ---- tree verification ---------------------------------------------------------------
def tree_mask_rows(parents):
    T = len(parents)
    m = np.zeros(T, np.uint64)
    for t in range(T):
        a = parents[t]
        while a >= 0:
            m[t] |= np.uint64(1) << np.uint64(a)
            a = parents[a]
    return m


def random_trees(B, T, seed):
    """Per sequence a random tree in topological order (parent < child, -1 =
    child of the prefix)."""
    rng = np.random.default_rng(seed)
    rows = []
    for _ in range(B):
        parents = [-1] + [int(rng.integers(-1, t)) for t in range(1, T)]
        rows.append(tree_mask_rows(parents))
    return np.stack(rows)


def as_i64(mask):
    return torch.from_numpy(mask.view(np.int64).copy())


@pytest.mark.parametrize("T,N,K,H,dtype", [(6, 64, 8, 128, "bf16"), (5, 16, 2, 64, "f16"),
                                           (4, 14, 2, 64, "f16"), (2, 8, 8, 128, "bf16")])
def test_tree_verify_matches_oracle(gpu, T, N, K, H, dtype):
    ctx = (T, T + 1, 16, 17, 33, 300, 1029, 4100)
    w = small(B=len(ctx), T=T, N=N, K=K, H=H, dtype=dtype, ctx=ctx, seed=7 * T + N)
    m = random_trees(len(ctx), T, seed=T)
    ref, err = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                                w.context_lens, dtype, tree_mask=m)
    assert (err == 0).all()
    wd = to(w, gpu)
    out = gq.verify_attention(wd.q[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables,
                              wd.context_lens, tree_mask=as_i64(m).to(gpu))
    torch.cuda.synchronize()
    assert_close(out.float().cpu().double().numpy(), ref, dtype, f"tree T={T} N={N} K={K}")


def test_tree_chain_mask_is_bit_identical_to_verify(gpu):
    T = 5
    ctx = (T, 40, 700, 3000)
    w = small(B=len(ctx), T=T, N=64, K=8, H=128, dtype="bf16", ctx=ctx, seed=51)
    chain = np.tile(np.array([(1 << t) - 1 for t in range(T)], np.uint64), (len(ctx), 1))
    junk = chain | np.tile(np.array([~np.uint64(0) << np.uint64(t) for t in range(T)],
                                    np.uint64), (len(ctx), 1))
    wd = to(w, gpu)
    args = (wd.q[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables, wd.context_lens)
    plain = gq.verify_attention(*args)
    tree = gq.verify_attention(*args, tree_mask=as_i64(chain).to(gpu))
    tree_junk = gq.verify_attention(*args, tree_mask=as_i64(junk).to(gpu))
    torch.cuda.synchronize()
    assert torch.equal(plain, tree)
    assert torch.equal(plain, tree_junk)  # bits at or after the row are ignored


def test_tree_fused_append_matches_oracle(gpu):
    T = 6
    ctx = (T, 70, 333, 2000)
    w = small(B=len(ctx), T=T, N=64, K=8, H=128, dtype="bf16", ctx=ctx, seed=52, append=True)
    m = random_trees(len(ctx), T, seed=9)
    kc, vc, _ = oracle.kv_append(w.k_new[0], w.v_new[0], w.k_cache[0], w.v_cache[0],
                                 w.block_tables, w.context_lens)
    kt = torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16)
    vt = torch.from_numpy(vc.view(np.int16)).view(torch.bfloat16)
    ref, err = oracle.attention(w.q[0], kt, vt, w.block_tables, w.context_lens, "bf16",
                                tree_mask=m)
    assert (err == 0).all()
    wd = to(w, gpu)
    out = gq.append_verify_attention(wd.q[0], wd.k_new[0], wd.v_new[0], wd.k_cache[0],
                                     wd.v_cache[0], wd.block_tables, wd.context_lens,
                                     tree_mask=as_i64(m).to(gpu))
    torch.cuda.synchronize()
    assert_close(out.float().cpu().double().numpy(), ref, "bf16", "fused tree")
    np.testing.assert_array_equal(wd.v_cache[0].cpu().view(torch.int16).numpy().view(np.uint16),
                                  vc)


def test_tree_mask_with_window_is_rejected(gpu):
    w = small(B=2, T=3, N=8, K=2, H=64, ctx=(5, 40), seed=53)
    wd = to(w, gpu)
    m = as_i64(random_trees(2, 3, 1)).to(gpu)
    with pytest.raises(gq.GqaError):
        gq.verify_attention(wd.q[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables,
                            wd.context_lens, tree_mask=m, window=16)


@pytest.mark.parametrize("first_new", [15, 16, 31, 1023])
def test_tree_first_new_token_at_a_tile_edge(gpu, first_new):
    """Rows that do not descend from new token 0 must not see it, also when
    it is the last position of a tile."""
    T = 4
    ctx = (first_new + T,) * 3
    w = small(B=3, T=T, N=16, K=2, H=64, dtype="f16", ctx=ctx, seed=first_new)
    m = np.zeros((3, T), np.uint64)  # every node a root: prefix + itself only
    m[1] = tree_mask_rows([-1, -1, 1, 2])
    m[2] = tree_mask_rows([-1, 0, 0, 0])
    ref, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                              w.context_lens, "f16", tree_mask=m)
    wd = to(w, gpu)
    out = gq.verify_attention(wd.q[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables,
                              wd.context_lens, tree_mask=as_i64(m).to(gpu))
    torch.cuda.synchronize()
    assert_close(out.float().cpu().double().numpy(), ref, "f16", f"tree edge {first_new}")


# ---- more than 48 query rows per KV head: row chunks ---------------------------------
@pytest.mark.parametrize("N,K,H,dtype", [(64, 1, 128, "bf16"), (56, 1, 64, "f16"),
                                         (128, 2, 128, "bf16"), (49, 1, 64, "f16")])
def test_decode_many_query_heads_per_kv_head(gpu, N, K, H, dtype):
    ctx = (1, 15, 16, 17, 300, 2049)
    w = small(B=len(ctx), T=1, N=N, K=K, H=H, dtype=dtype, ctx=ctx, seed=N + K)
    ref, err = oracle_out(w)
    assert (err == 0).all()
    assert_close(run_attention(w, gpu), ref, dtype, f"decode G={N // K}")


@pytest.mark.parametrize("T,N,K", [(8, 64, 8), (26, 64, 8), (64, 4, 4), (7, 56, 8)])
def test_verify_more_than_48_rows(gpu, T, N, K):
    ctx = (T, T + 3, 100, 1500)
    w = small(B=len(ctx), T=T, N=N, K=K, H=128, dtype="bf16", ctx=ctx, seed=T * N)
    ref, err = oracle_out(w)
    assert (err == 0).all()
    assert_close(run_attention(w, gpu), ref, "bf16", f"verify T={T} G={N // K}")


def test_tree_verify_26_node_tree(gpu):
    """An EAGLE-sized tree (26 nodes: a root, then 3, 6, 8, 8 nodes per level)
    with 8 query heads per KV head: 208 rows in five chunks."""
    parents = [-1, 0, 0, 0, 1, 1, 2, 2, 3, 3] + [4 + i // 2 for i in range(8)] + \
              [10 + i for i in range(8)]
    T = len(parents)
    assert T == 26
    ctx = (T, 40, 1000, 3000)
    w = small(B=len(ctx), T=T, N=64, K=8, H=128, dtype="bf16", ctx=ctx, seed=26)
    m = np.tile(tree_mask_rows(parents), (len(ctx), 1))
    ref, err = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                                w.context_lens, "bf16", tree_mask=m)
    assert (err == 0).all()
    wd = to(w, gpu)
    out = gq.verify_attention(wd.q[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables,
                              wd.context_lens, tree_mask=as_i64(m).to(gpu))
    torch.cuda.synchronize()
    assert_close(out.float().cpu().double().numpy(), ref, "bf16", "26-node tree")


def test_fused_append_with_row_chunks_writes_the_cache_once(gpu):
    T = 8
    ctx = (T, 70, 900)
    w = small(B=len(ctx), T=T, N=64, K=8, H=128, dtype="bf16", ctx=ctx, seed=88, append=True)
    kc, vc, _ = oracle.kv_append(w.k_new[0], w.v_new[0], w.k_cache[0], w.v_cache[0],
                                 w.block_tables, w.context_lens)
    kt = torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16)
    vt = torch.from_numpy(vc.view(np.int16)).view(torch.bfloat16)
    ref, _ = oracle.attention(w.q[0], kt, vt, w.block_tables, w.context_lens, "bf16")
    wd = to(w, gpu)
    out = gq.append_verify_attention(wd.q[0], wd.k_new[0], wd.v_new[0], wd.k_cache[0],
                                     wd.v_cache[0], wd.block_tables, wd.context_lens)
    torch.cuda.synchronize()
    assert_close(out.float().cpu().double().numpy(), ref, "bf16", "fused, 64 rows")
    np.testing.assert_array_equal(wd.k_cache[0].cpu().view(torch.int16).numpy().view(np.uint16),
                                  kc)
    np.testing.assert_array_equal(wd.v_cache[0].cpu().view(torch.int16).numpy().view(np.uint16),
                                  vc)
