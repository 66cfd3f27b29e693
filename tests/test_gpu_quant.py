"""GPU one-byte KV cache: the quantized append bit-exact against the oracle
(codes and scales), and attention over the quantized cache against the
oracle's attention over the same codes and scales."""
import numpy as np
import pytest
import torch

import gqa_decode_attention_02_gb300 as gq
import oracle
from helpers import assert_close, small, to

pytestmark = pytest.mark.gpu


def empty_quant(w, dev, fill=0):
    NB, bs, K, H = w.k_cache[0].shape
    kc = torch.full((NB, bs, K, H), fill, dtype=torch.uint8, device=dev)
    vc = torch.full_like(kc, fill)
    ks = torch.full((NB, K, bs), -1.0, dtype=torch.float32, device=dev)
    vs = torch.full_like(ks, -1.0)
    return kc, vc, ks, vs


@pytest.mark.parametrize("kv", ["int8", "e4m3"])
@pytest.mark.parametrize("dtype,H", [("bf16", 128), ("f16", 128), ("bf16", 64), ("f16", 64)])
@pytest.mark.parametrize("T", [1, 3])
def test_quant_append_bit_exact(gpu, kv, dtype, H, T):
    ctx = tuple(max(c, T) for c in (1, 3, 16, 17, 31, 32, 33, 500))
    w = small(B=len(ctx), T=T, N=8, K=4, H=H, dtype=dtype, ctx=ctx, seed=T + H, append=True)
    # rows with exact ties: scale 1 (max |x| = qmax), halves / e4m3 midpoints
    qmax = 127.0 if kv == "int8" else 448.0
    ties = [2.5, -2.5, 3.5, 0.5, -0.5, 17.0, 19.0, 0.01953125, 100.0, -1.5]
    row = torch.zeros(H)
    row[0] = qmax
    row[1:1 + len(ties)] = torch.tensor(ties)
    w.k_new[0][0, 0, 0] = row.to(w.torch_dtype)
    w.v_new[0][-1, T - 1, 3] = (-row).to(w.torch_dtype)
    w.k_new[0][1, 0, 1] = 0.0  # a row of zeros
    kc0, vc0, ks0, vs0 = empty_quant(w, "cpu", fill=0x5A)
    rk, rv, rks, rvs, err = oracle.kv_append_quant(w.k_new[0], w.v_new[0], kc0, vc0, ks0, vs0,
                                                   w.block_tables, w.context_lens, dtype, kv)
    assert (err == 0).all()
    wd = to(w, gpu)
    kc, vc, ks, vs = empty_quant(w, gpu, fill=0x5A)
    gq.kv_append_quant(wd.k_new[0], wd.v_new[0], kc, vc, ks, vs, wd.block_tables,
                       wd.context_lens, kv=kv)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(kc.cpu().numpy(), rk)
    np.testing.assert_array_equal(vc.cpu().numpy(), rv)
    np.testing.assert_array_equal(ks.cpu().numpy().view(np.uint32), rks.view(np.uint32))
    np.testing.assert_array_equal(vs.cpu().numpy().view(np.uint32), rvs.view(np.uint32))


def test_quant_append_reports_bad_context(gpu):
    w = small(B=2, T=2, N=8, K=2, H=128, dtype="bf16", ctx=(5, 40), seed=3, append=True)
    wd = to(w, gpu)
    wd.context_lens[0] = 1  # < T
    kc, vc, ks, vs = empty_quant(w, gpu)
    st = torch.zeros(1, dtype=torch.int32, device=gpu)
    gq.kv_append_quant(wd.k_new[0], wd.v_new[0], kc, vc, ks, vs, wd.block_tables,
                       wd.context_lens, kv="int8", status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 7


def quant_inputs(w, kv):
    kc, ks = oracle.quantize_cache(w.k_cache[0], w.dtype, kv)
    vc, vs = oracle.quantize_cache(w.v_cache[0], w.dtype, kv)
    return kc, vc, ks, vs


def run_quant(w, kv, kc, vc, ks, vs, dev, status=None, window=0, tables=None):
    wd = to(w, dev)
    fn = gq.decode_attention_quant if w.T == 1 else gq.verify_attention_quant
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    bt = wd.block_tables if tables is None else t(tables)
    out = fn(wd.q[0], t(kc), t(vc), t(ks), t(vs), bt, wd.context_lens, kv=kv,
             status=status, window=window)
    torch.cuda.synchronize()
    return out.float().cpu().double().numpy()


@pytest.mark.parametrize("kv", ["int8", "e4m3"])
@pytest.mark.parametrize("T,N,K,dtype", [(1, 32, 8, "bf16"), (1, 8, 8, "f16"), (1, 64, 8, "bf16"),
                                         (5, 64, 8, "bf16"), (3, 16, 2, "f16"), (2, 8, 1, "bf16")])
def test_quant_attention_matches_oracle(gpu, kv, T, N, K, dtype):
    ctx = tuple(max(c, T) for c in (1, 2, 15, 16, 17, 31, 295, 1029, 4097))
    w = small(B=len(ctx), T=T, N=N, K=K, H=128, dtype=dtype, ctx=ctx, seed=N + T + K)
    kc, vc, ks, vs = quant_inputs(w, kv)
    ref, err = oracle.attention(w.q[0], kc, vc, w.block_tables, w.context_lens, dtype, kv=kv,
                                k_scale=ks, v_scale=vs)
    assert (err == 0).all()
    got = run_quant(w, kv, kc, vc, ks, vs, gpu)
    from helpers import assert_close
    assert_close(got, ref, dtype, f"{kv} T={T} N={N} K={K}")


@pytest.mark.parametrize("kv", ["int8", "e4m3"])
def test_quant_append_then_attention(gpu, kv):
    """The decode step on a one-byte cache: the GPU's own quantized append of
    the new token, then attention, against the oracle doing both."""
    T = 1
    ctx = (1, 17, 300, 2000)
    w = small(B=len(ctx), T=T, N=32, K=8, H=128, dtype="bf16", ctx=ctx, seed=71, append=True)
    kc, vc, ks, vs = quant_inputs(w, kv)  # the cached part (new slots hold NaN -> zeros)
    rk, rv, rks, rvs, err = oracle.kv_append_quant(w.k_new[0], w.v_new[0], kc, vc, ks, vs,
                                                   w.block_tables, w.context_lens, "bf16", kv)
    assert (err == 0).all()
    ref, _ = oracle.attention(w.q[0], rk, rv, w.block_tables, w.context_lens, "bf16", kv=kv,
                              k_scale=rks, v_scale=rvs)
    wd = to(w, gpu)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(gpu)  # noqa: E731
    dkc, dvc, dks, dvs = t(kc), t(vc), t(ks), t(vs)
    gq.kv_append_quant(wd.k_new[0], wd.v_new[0], dkc, dvc, dks, dvs, wd.block_tables,
                       wd.context_lens, kv=kv, pdl=True)
    out = gq.decode_attention_quant(wd.q[0], dkc, dvc, dks, dvs, wd.block_tables,
                                    wd.context_lens, kv=kv, pdl=True)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(dkc.cpu().numpy(), rk)
    from helpers import assert_close
    assert_close(out.float().cpu().double().numpy(), ref, "bf16", f"{kv} append+attend")


def test_quant_attention_bad_block_and_shapes(gpu):
    w = small(B=2, T=1, N=8, K=2, H=128, dtype="bf16", ctx=(5, 40), seed=72)
    kc, vc, ks, vs = quant_inputs(w, "int8")
    w.block_tables[1, 1] = 10**6
    st = torch.zeros(1, dtype=torch.int32, device=gpu)
    got = run_quant(w, "int8", kc, vc, ks, vs, gpu, status=st)
    assert int(st.item()) == 8 and (got[1] == 0).all()
    # H = 64 has no one-byte attention kernel
    w64 = small(B=1, T=1, N=8, K=2, H=64, dtype="bf16", ctx=(5,), seed=73)
    kc, vc, ks, vs = quant_inputs(w64, "int8")
    with pytest.raises(gq.GqaError):
        run_quant(w64, "int8", kc, vc, ks, vs, gpu)


# ---- local attention and row chunks over a one-byte cache ---------------------------
@pytest.mark.parametrize("kv", ["int8", "e4m3"])
@pytest.mark.parametrize("T,N,K,dtype", [(1, 32, 8, "bf16"), (5, 64, 8, "bf16"), (3, 16, 2, "f16")])
@pytest.mark.parametrize("W", [1, 15, 17, 100, 1024])
def test_quant_window_matches_oracle(gpu, kv, T, N, K, dtype, W):
    ctx = tuple(max(c, T) for c in (1, 2, 15, 16, 17, 31, 295, 1029, 4097))
    w = small(B=len(ctx), T=T, N=N, K=K, H=128, dtype=dtype, ctx=ctx, seed=W + 7 * T + N)
    kc, vc, ks, vs = quant_inputs(w, kv)
    ref, err = oracle.attention(w.q[0], kc, vc, w.block_tables, w.context_lens, dtype,
                                window=W, kv=kv, k_scale=ks, v_scale=vs)
    assert (err == 0).all()
    got = run_quant(w, kv, kc, vc, ks, vs, gpu, window=W)
    assert_close(got, ref, dtype, f"{kv} window {W} T={T}")


@pytest.mark.parametrize("kv", ["int8", "e4m3"])
@pytest.mark.parametrize("T", [1, 4])
def test_quant_window_ignores_poisoned_rows_and_freed_blocks(gpu, kv, T):
    """Below the earliest window: codes of every value (e4m3 NaN codes too),
    NaN row scales, and INT32_MAX table entries for whole blocks.  Same
    result as the clean cache, no error."""
    W = 40
    ctx = (T, 45, 64, 300, 1000)
    w = small(B=len(ctx), T=T, N=8, K=2, H=128, dtype="bf16", ctx=ctx, seed=177 + T)
    kc, vc, ks, vs = quant_inputs(w, kv)
    ref, _ = oracle.attention(w.q[0], kc, vc, w.block_tables, w.context_lens, "bf16",
                              window=W, kv=kv, k_scale=ks, v_scale=vs)
    kc, vc, ks, vs = kc.copy(), vc.copy(), ks.copy(), vs.copy()
    tables = w.block_tables.numpy().copy()
    rng = np.random.default_rng(T)
    for b, c in enumerate(ctx):
        first = max(0, c - T - W + 1)
        for pos in range(first):
            blk, row = tables[b, pos // 16], pos % 16
            kc[blk, row] = rng.integers(0, 256, size=kc[blk, row].shape)
            vc[blk, row] = 0x7F  # the e4m3 NaN code; an ordinary code for int8
            ks[blk, :, row] = np.nan
            vs[blk, :, row] = np.nan
        tables[b, : first // 16] = 2**31 - 1
    ref2, err = oracle.attention(w.q[0], kc, vc, tables, w.context_lens, "bf16", window=W,
                                 kv=kv, k_scale=ks, v_scale=vs)
    assert (err == 0).all()
    np.testing.assert_array_equal(ref2, ref)
    st = torch.zeros(1, dtype=torch.int32, device=gpu)
    got = run_quant(w, kv, kc, vc, ks, vs, gpu, status=st, window=W, tables=tables)
    assert int(st.item()) == 0
    assert np.isfinite(got).all()
    assert_close(got, ref, "bf16", f"{kv} poisoned window")


@pytest.mark.parametrize("kv", ["int8", "e4m3"])
@pytest.mark.parametrize("T,N,K,W", [(4, 64, 4, 0), (7, 64, 8, 0), (5, 64, 2, 0), (4, 64, 4, 33)])
def test_quant_row_chunks_match_oracle(gpu, kv, T, N, K, W):
    """More than 48 query rows per KV head (T * N / K = 64, 56, 160): row
    chunks, each reading the KV head's blocks; with and without a window."""
    ctx = tuple(max(c, T) for c in (1, 16, 17, 300, 2049))
    w = small(B=len(ctx), T=T, N=N, K=K, H=128, dtype="bf16", ctx=ctx, seed=T * N + K + W)
    kc, vc, ks, vs = quant_inputs(w, kv)
    ref, err = oracle.attention(w.q[0], kc, vc, w.block_tables, w.context_lens, "bf16",
                                window=W, kv=kv, k_scale=ks, v_scale=vs)
    assert (err == 0).all()
    got = run_quant(w, kv, kc, vc, ks, vs, gpu, window=W)
    assert_close(got, ref, "bf16", f"{kv} chunks T={T} N={N} K={K} W={W}")


# ---- the append fused into the one-byte attention call --------------------------------
@pytest.mark.parametrize("kv", ["int8", "e4m3"])
@pytest.mark.parametrize("T,N,K,dtype,W", [(1, 32, 8, "bf16", 0), (1, 8, 2, "f16", 0),
                                           (5, 64, 8, "bf16", 0), (3, 16, 2, "bf16", 40),
                                           (4, 64, 4, "bf16", 0)])
def test_fused_quant_append_matches_oracle_and_the_pair(gpu, kv, T, N, K, dtype, W):
    """One call (the append launch, then the attention launch): the new rows
    quantized (codes and scales bit-exact with the oracle's append), attention
    over them within tolerance of the oracle, and the same bits as the two
    calls made separately.  Covers a window and row chunks (64 query rows per
    KV head), with and without programmatic dependent launch."""
    ctx = tuple(max(c, T) for c in (1, 16, 17, 33, 300, 2049))
    w = small(B=len(ctx), T=T, N=N, K=K, H=128, dtype=dtype, ctx=ctx, seed=T * N + K + W,
              append=True)
    kc, vc, ks, vs = quant_inputs(w, kv)  # the cached part (new slots hold NaN -> zeros)
    rk, rv, rks, rvs, err = oracle.kv_append_quant(w.k_new[0], w.v_new[0], kc, vc, ks, vs,
                                                   w.block_tables, w.context_lens, dtype, kv)
    assert (err == 0).all()
    ref, err = oracle.attention(w.q[0], rk, rv, w.block_tables, w.context_lens, dtype,
                                window=W, kv=kv, k_scale=rks, v_scale=rvs)
    assert (err == 0).all()
    wd = to(w, gpu)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(gpu)  # noqa: E731
    fused = gq.append_decode_attention_quant if T == 1 else gq.append_verify_attention_quant
    outs = []
    for flags in (dict(), dict(pdl=True, early_kv=True)):
        dkc, dvc, dks, dvs = t(kc), t(vc), t(ks), t(vs)
        st = torch.zeros(1, dtype=torch.int32, device=gpu)
        out = fused(wd.q[0], wd.k_new[0], wd.v_new[0], dkc, dvc, dks, dvs, wd.block_tables,
                    wd.context_lens, kv=kv, status=st, window=W, **flags)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        np.testing.assert_array_equal(dkc.cpu().numpy(), rk)
        np.testing.assert_array_equal(dvc.cpu().numpy(), rv)
        np.testing.assert_array_equal(dks.cpu().numpy().view(np.uint32), rks.view(np.uint32))
        np.testing.assert_array_equal(dvs.cpu().numpy().view(np.uint32), rvs.view(np.uint32))
        assert_close(out.float().cpu().double().numpy(), ref, dtype, f"fused {kv} T={T} W={W}")
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    # the separate append, then attention: the same bits
    dkc, dvc, dks, dvs = t(kc), t(vc), t(ks), t(vs)
    gq.kv_append_quant(wd.k_new[0], wd.v_new[0], dkc, dvc, dks, dvs, wd.block_tables,
                       wd.context_lens, kv=kv)
    attn = gq.decode_attention_quant if T == 1 else gq.verify_attention_quant
    pair = attn(wd.q[0], dkc, dvc, dks, dvs, wd.block_tables, wd.context_lens, kv=kv, window=W)
    torch.cuda.synchronize()
    assert torch.equal(pair.view(torch.int16), outs[0].view(torch.int16))


# ---- tree verification over a one-byte cache ---------------------------------------
@pytest.mark.parametrize("kv", ["int8", "e4m3"])
@pytest.mark.parametrize("T,N,K", [(6, 64, 8), (26, 64, 8), (4, 16, 2)])
def test_quant_tree_verify_matches_oracle(gpu, kv, T, N, K):
    """Draft trees (random ancestor masks, 24-208 query rows per KV head, row
    chunks included) over one-byte codes, against the oracle over the same
    codes and scales; the chain mask gives verify_attention_quant's bits."""
    from test_gpu_attention import as_i64, random_trees

    ctx = (T, T + 1, 16 + T, 300, 1029)
    w = small(B=len(ctx), T=T, N=N, K=K, H=128, dtype="bf16", ctx=ctx, seed=11 * T + N)
    kc, vc, ks, vs = quant_inputs(w, kv)
    m = random_trees(len(ctx), T, seed=T + 2)
    ref, err = oracle.attention(w.q[0], kc, vc, w.block_tables, w.context_lens, "bf16",
                                tree_mask=m, kv=kv, k_scale=ks, v_scale=vs)
    assert (err == 0).all()
    wd = to(w, gpu)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(gpu)  # noqa: E731
    dkc, dvc, dks, dvs = t(kc), t(vc), t(ks), t(vs)
    st = torch.zeros(1, dtype=torch.int32, device=gpu)
    out = gq.verify_attention_quant(wd.q[0], dkc, dvc, dks, dvs, wd.block_tables,
                                    wd.context_lens, kv=kv, status=st,
                                    tree_mask=as_i64(m).to(gpu))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_close(out.float().cpu().double().numpy(), ref, "bf16", f"{kv} tree T={T}")
    # the chain mask (every earlier new token) is plain causal verification
    chain = np.array([[(1 << t) - 1 for t in range(T)]] * len(ctx), dtype=np.uint64)
    a = gq.verify_attention_quant(wd.q[0], dkc, dvc, dks, dvs, wd.block_tables,
                                  wd.context_lens, kv=kv, tree_mask=as_i64(chain).to(gpu))
    b = gq.verify_attention_quant(wd.q[0], dkc, dvc, dks, dvs, wd.block_tables,
                                  wd.context_lens, kv=kv)
    torch.cuda.synchronize()
    ref_c, _ = oracle.attention(w.q[0], kc, vc, w.block_tables, w.context_lens, "bf16",
                                kv=kv, k_scale=ks, v_scale=vs)
    assert_close(a.float().cpu().double().numpy(), ref_c, "bf16", f"{kv} chain mask")
    assert_close(b.float().cpu().double().numpy(), ref_c, "bf16", f"{kv} verify")
