"""The direct warp-level kernel (one CTA per sequence and KV head, every warp
loading its own cache blocks, no split of a context over CTAs) against the fp64
oracle, and against the persistent warp-level kernel on the same inputs: plain
and fused-append calls, contexts from one token to several rounds of stages per
warp, invalid lengths and block ids, programmatic dependent launch and graphs."""
import numpy as np
import pytest
import torch

import gqa_decode_attention_02_gb300 as gq
import oracle
from helpers import TOL, assert_close, small, to, ulp

pytestmark = pytest.mark.gpu

# one token, tile edges, a ragged tail, several stages per warp (H = 64: 8 warps
# of 4-tile stages, so 1029 tokens = 65 blocks = 17 stages take three rounds)
CTX = (1, 2, 15, 16, 17, 31, 64, 65, 295, 1029)


def attend(w, dev, engine, status=None, fused=False):
    wd = to(w, dev)
    if fused:
        fn = gq.append_decode_attention if w.T == 1 else gq.append_verify_attention
        out = fn(wd.q[0], wd.k_new[0], wd.v_new[0], wd.k_cache[0], wd.v_cache[0],
                 wd.block_tables, wd.context_lens, status=status, engine=engine)
    else:
        fn = gq.decode_attention if w.T == 1 else gq.verify_attention
        out = fn(wd.q[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables, wd.context_lens,
                 status=status, engine=engine)
    torch.cuda.synchronize()
    return out, wd


def close_to_each_other(a, b, dtype):
    a = a.float().cpu().double().numpy()
    b = b.float().cpu().double().numpy()
    assert np.isfinite(a).all()
    lim = np.maximum(TOL[dtype], ulp(b, dtype))
    assert (np.abs(a - b) <= lim).all(), float(np.abs(a - b).max())


@pytest.mark.parametrize("T,N,K,H,dtype", [
    (1, 14, 2, 64, "f16"),     # 7 rows per KV head (the single-layer fp16 shape)
    (1, 32, 8, 128, "bf16"),   # 4 rows
    (1, 8, 1, 64, "bf16"),     # 8 rows
    (1, 8, 8, 128, "f16"),     # 1 row
    (2, 32, 8, 128, "bf16"),   # 2 tokens x 4 rows
    (4, 8, 4, 64, "f16"),      # 4 tokens x 2 rows
])
def test_direct_matches_oracle(gpu, T, N, K, H, dtype):
    ctx = tuple(max(c, T) for c in CTX)
    w = small(B=len(ctx), T=T, N=N, K=K, H=H, dtype=dtype, ctx=ctx, seed=3 * T + N + H)
    ref, err = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                                w.context_lens, dtype)
    assert (err == 0).all()
    st = torch.zeros(1, dtype=torch.int32, device=gpu)
    out, _ = attend(w, gpu, "direct", status=st)
    assert int(st.item()) == 0
    assert_close(out.float().cpu().double().numpy(), ref, dtype, f"direct T={T} N={N} K={K}")
    # the persistent kernel on the same inputs: the same function
    close_to_each_other(out, attend(w, gpu, "warp")[0], dtype)


def test_small_calls_pick_the_direct_kernel_by_default(gpu):
    """A single short sequence (the single-layer fp16 shape) and a 64-sequence
    batch of contexts up to 1024: auto is the direct kernel, bit for bit."""
    for B, ctx in ((1, (295,)), (64, tuple(16 + 15 * i for i in range(64)))):
        w = small(B=B, T=1, N=14, K=2, H=64, dtype="f16", ctx=ctx, seed=B)
        assert gq.attention_engine(w.q[0], w.k_cache[0], w.block_tables) == "direct"
        auto, _ = attend(w, gpu, "auto")
        assert torch.equal(auto.view(torch.int16), attend(w, gpu, "direct")[0].view(torch.int16))


@pytest.mark.parametrize("T,N,K,H,dtype", [(1, 14, 2, 64, "f16"), (1, 32, 8, 128, "bf16"),
                                           (2, 16, 4, 128, "bf16")])
def test_direct_fused_append_writes_the_cache_and_matches_oracle(gpu, T, N, K, H, dtype):
    # 65 and 129 with T = 2: the new positions straddle two stages, so two
    # different warps patch and write them
    ctx = tuple(max(c, T) for c in (1, 16, 17, 32, 33, 65, 129, 300, 1024))
    w = small(B=len(ctx), T=T, N=N, K=K, H=H, dtype=dtype, ctx=ctx, seed=T + 11 * K,
              append=True)
    kc, vc, err = oracle.kv_append(w.k_new[0], w.v_new[0], w.k_cache[0], w.v_cache[0],
                                   w.block_tables, w.context_lens)
    assert (err == 0).all()
    tdt = w.torch_dtype
    ref, _ = oracle.attention(w.q[0], torch.from_numpy(kc.view(np.int16)).view(tdt),
                              torch.from_numpy(vc.view(np.int16)).view(tdt), w.block_tables,
                              w.context_lens, dtype)
    st = torch.zeros(1, dtype=torch.int32, device=gpu)
    out, wd = attend(w, gpu, "direct", status=st, fused=True)
    assert int(st.item()) == 0
    for mine, theirs in ((wd.k_cache[0], kc), (wd.v_cache[0], vc)):  # every cache byte
        np.testing.assert_array_equal(mine.cpu().view(torch.int16).numpy().view(np.uint16),
                                      theirs)
    assert_close(out.float().cpu().double().numpy(), ref, dtype, "direct fused append")
    # the unfused pair on the direct kernel gives the same bits
    a = to(w, gpu)
    gq.kv_append(a.k_new[0], a.v_new[0], a.k_cache[0], a.v_cache[0], a.block_tables,
                 a.context_lens)
    fn = gq.decode_attention if T == 1 else gq.verify_attention
    pair = fn(a.q[0], a.k_cache[0], a.v_cache[0], a.block_tables, a.context_lens,
              engine="direct")
    torch.cuda.synchronize()
    assert torch.equal(pair.view(torch.int16), out.view(torch.int16))


def test_direct_device_errors_zero_the_rows_and_set_status(gpu):
    w = small(B=4, T=2, N=8, K=2, H=64, ctx=(1, 40, 40, 40), seed=7)
    w.block_tables[2, 1] = w.num_blocks + 3  # bad id inside sequence 2's context
    w.block_tables[3, 0] = -1                # bad id in sequence 3
    ref, err = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                                w.context_lens, w.dtype)
    assert list(err) == [7, 0, 8, 8]
    st = torch.zeros(1, dtype=torch.int32, device=gpu)
    out, _ = attend(w, gpu, "direct", status=st)
    got = out.float().cpu().double().numpy()
    assert int(st.item()) in (7, 8)
    assert (got[0] == 0).all() and (got[2] == 0).all() and (got[3] == 0).all()
    assert_close(got[1], ref[1], "f16", "healthy sequence next to bad ones")


def test_direct_long_context_is_still_exact(gpu):
    """Forced onto a context far beyond its default range (many rounds of
    stages per warp): still the oracle's result."""
    w = small(B=2, T=1, N=8, K=2, H=128, dtype="bf16", ctx=(9000, 3), seed=5)
    ref, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                              w.context_lens, "bf16")
    out, _ = attend(w, gpu, "direct")
    assert_close(out.float().cpu().double().numpy(), ref, "bf16", "direct, 9000 tokens")


def test_direct_empty_batch_and_rejected_shapes(gpu):
    w = small(B=1, T=1, N=8, K=2, H=64, ctx=(5,), seed=1)
    wd = to(w, gpu)
    empty = gq.decode_attention(wd.q[0][:0], wd.k_cache[0], wd.v_cache[0], wd.block_tables[:0],
                                wd.context_lens[:0], engine="direct")
    assert empty.shape[0] == 0
    with pytest.raises(gq.GqaError):  # a window: not served by the direct kernel
        gq.decode_attention(wd.q[0], wd.k_cache[0], wd.v_cache[0], wd.block_tables,
                            wd.context_lens, window=4, engine="direct")
    v = small(B=1, T=3, N=8, K=2, H=64, ctx=(5,), seed=2)  # 12 rows per KV head
    vd = to(v, gpu)
    with pytest.raises(gq.GqaError):
        gq.verify_attention(vd.q[0], vd.k_cache[0], vd.v_cache[0], vd.block_tables,
                            vd.context_lens, engine="direct")


def test_direct_pdl_early_kv_and_graph_match_plain(gpu):
    """Append + attention over three layers, plain and with programmatic
    dependent launch / early KV reads, eagerly and from a CUDA graph."""
    layers = 3
    ctx = (1, 17, 300, 1000, 64)
    w = small(B=5, T=1, N=14, K=2, H=64, dtype="f16", ctx=ctx, seed=41, append=True,
              layers=layers)

    def run(flags, graph, fused):
        wd = to(w, gpu)
        outs = [torch.empty_like(q) for q in wd.q]

        def step():
            for l in range(layers):
                if fused:
                    gq.append_decode_attention(wd.q[l], wd.k_new[l], wd.v_new[l], wd.k_cache[l],
                                               wd.v_cache[l], wd.block_tables, wd.context_lens,
                                               out=outs[l], engine="direct", **flags)
                else:
                    gq.kv_append(wd.k_new[l], wd.v_new[l], wd.k_cache[l], wd.v_cache[l],
                                 wd.block_tables, wd.context_lens, pdl=flags["pdl"])
                    gq.decode_attention(wd.q[l], wd.k_cache[l], wd.v_cache[l], wd.block_tables,
                                        wd.context_lens, out=outs[l], engine="direct", **flags)

        if graph:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                step()  # warm-up (plans, attributes)
            torch.cuda.current_stream().wait_stream(s)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step()
            g.replay()
        else:
            step()
        torch.cuda.synchronize()
        return [o.cpu() for o in outs]

    ref = run(dict(pdl=False, early_kv=False), False, False)
    for fused in (False, True):
        for flags in (dict(pdl=True, early_kv=False), dict(pdl=True, early_kv=True)):
            for graph in (False, True):
                got = run(flags, graph, fused)
                for l in range(layers):
                    assert torch.equal(got[l].view(torch.int16), ref[l].view(torch.int16)), (
                        fused, flags, graph, l)
    kc, vc, _ = oracle.kv_append(w.k_new[0], w.v_new[0], w.k_cache[0], w.v_cache[0],
                                 w.block_tables, w.context_lens)
    kc = torch.from_numpy(kc.view(np.int16)).view(torch.float16)
    vc = torch.from_numpy(vc.view(np.int16)).view(torch.float16)
    o, _ = oracle.attention(w.q[0], kc, vc, w.block_tables, w.context_lens, "f16")
    assert_close(ref[0].double().numpy(), o, "f16", "layer 0")
