"""Parity at the named workloads' full sizes, through the same calls the
bench times (kv_append then decode/verify attention; accept_prefix).  Where the
oracle would take too long on the whole batch, it checks a seeded sample of
sequences that always includes the shortest and the longest."""
import numpy as np
import pytest
import torch

import gqa_decode_attention_02_gb300 as gq
import oracle
from gqa_decode_attention_02_gb300 import workloads
from helpers import assert_close

pytestmark = pytest.mark.gpu


def sample_sequences(ctx: np.ndarray, n: int, seed: int) -> np.ndarray:
    if len(ctx) <= n:
        return np.arange(len(ctx))
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(len(ctx), size=n - 2, replace=False).tolist())
    pick.add(int(np.argmin(ctx)))
    pick.add(int(np.argmax(ctx)))
    return np.array(sorted(pick), np.int32)


def check_workload(name, dev, sample=None, layers=None, fused=False):
    w = workloads.make(name, layers=layers)
    ctx = w.context_lens.numpy()
    bl = sample_sequences(ctx, sample, 1) if sample else np.arange(w.B, dtype=np.int32)
    worst = 0.0
    for layer in range(w.layers):
        kc, vc = w.k_cache[layer], w.v_cache[layer]
        if w.appended:
            okc, ovc, err = oracle.kv_append(w.k_new[layer], w.v_new[layer], kc, vc,
                                             w.block_tables, w.context_lens)
            assert (err == 0).all()
            okc = torch.from_numpy(okc.view(np.int16)).view(w.torch_dtype)
            ovc = torch.from_numpy(ovc.view(np.int16)).view(w.torch_dtype)
        else:
            okc, ovc = kc, vc
        win = w.window(layer)
        tm = w.tree_mask()
        extra = {} if tm is None else {
            "tree_mask": torch.from_numpy(tm.view(np.int64)).to(dev)}
        ref, err = oracle.attention(w.q[layer], okc, ovc, w.block_tables, w.context_lens,
                                    w.dtype, b_list=bl, window=win, tree_mask=tm)
        assert (err == 0).all()
        kd, vd = kc.to(dev), vc.to(dev)
        bt, cl = w.block_tables.to(dev), w.context_lens.to(dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        out = None
        if w.appended and fused:  # the append inside the attention launch (the bench's call)
            ffn = gq.append_decode_attention if w.T == 1 else gq.append_verify_attention
            out = ffn(w.q[layer].to(dev), w.k_new[layer].to(dev), w.v_new[layer].to(dev), kd, vd,
                      bt, cl, status=st, pdl=True, early_kv=True, window=win, **extra)
        elif w.appended:
            gq.kv_append(w.k_new[layer].to(dev), w.v_new[layer].to(dev), kd, vd, bt, cl,
                         status=st)
        if w.appended:
            # the append itself, bit for bit, on the blocks of the checked sequences
            tb = w.block_tables[torch.as_tensor(bl).long()]
            blocks = torch.unique(tb[tb != workloads.INT32_MAX]).long()
            np.testing.assert_array_equal(kd[blocks.to(dev)].cpu().view(torch.int16).numpy(),
                                          okc[blocks].view(torch.int16).numpy())
            np.testing.assert_array_equal(vd[blocks.to(dev)].cpu().view(torch.int16).numpy(),
                                          ovc[blocks].view(torch.int16).numpy())
        if out is None:
            fn = gq.decode_attention if w.T == 1 else gq.verify_attention
            out = fn(w.q[layer].to(dev), kd, vd, bt, cl, status=st, window=win, **extra)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        got = out.cpu()[torch.as_tensor(bl).long()].double().numpy()
        worst = max(worst, assert_close(got, ref, w.dtype, f"{name} layer {layer}"))
        del kd, vd
    return w, worst


def test_cfg1_single_layer_fp16(gpu):
    check_workload("cfg1", gpu)


def test_cfg2_24_layers(gpu):
    check_workload("cfg2", gpu)


def test_cfg3_fixed_8192(gpu):
    check_workload("cfg3", gpu, sample=12)


def test_cfg4_ragged_lognormal(gpu):
    w, _ = check_workload("cfg4", gpu, sample=24)
    assert w.context_lens.max() <= 32768 and w.context_lens.min() >= 1


def test_cfg5_verify_and_accept(gpu):
    w, _ = check_workload("cfg5", gpu)
    ctx = w.context_lens.numpy().copy()
    ra, rn, rc = oracle.accept_prefix(w.logits, w.draft, ctx)
    cl = w.context_lens.to(gpu)
    acc, nxt = gq.accept_prefix(w.logits.to(gpu), w.draft.to(gpu), cl)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(acc.cpu().numpy(), ra)
    np.testing.assert_array_equal(nxt.cpu().numpy(), rn)
    np.testing.assert_array_equal(cl.cpu().numpy(), rc)
    assert (ra >= w.draft_k).all()


@pytest.mark.parametrize("name,sample", [("cfg2", None), ("cfg3", 8), ("cfg4", 16), ("cfg5", None)])
def test_fused_append_at_full_size(gpu, name, sample):
    check_workload(name, gpu, sample=sample, fused=True)


@pytest.mark.parametrize("fused", [False, True])
def test_hybrid_local_global_layers(gpu, fused):
    """Six layers, five of local attention (1024-token window) and one global,
    on the long-context geometry, through the bench's calls."""
    w, _ = check_workload("hybrid", gpu, sample=8, fused=fused)
    assert w.windows == (1024,) * 5 + (0,)


@pytest.mark.parametrize("fused", [False, True])
def test_tree_verify_workload(gpu, fused):
    """The 26-node draft tree on the verify geometry (208 query rows per KV
    head, five row chunks), through the bench's calls."""
    w, _ = check_workload("tree", gpu, fused=fused)
    assert w.T == 26 and len(w.tree) == 26


@pytest.mark.parametrize("name,kv,sample", [("cfg4", "int8", 16), ("cfg3", "e4m3", 6),
                                            ("cfg5", "int8", None)])
def test_one_byte_cache_at_full_size(gpu, name, kv, sample):
    """The named workloads with a one-byte cache: the cached part quantized by
    the oracle, the new tokens appended by the library's quantized append
    (bit-exact on the checked sequences' blocks), then attention, against the
    oracle on a seeded sample of sequences."""
    w = workloads.make(name)
    ctx = w.context_lens.numpy()
    bl = sample_sequences(ctx, sample, 2) if sample else np.arange(w.B, dtype=np.int32)
    kc, ks = oracle.quantize_cache(w.k_cache[0], w.dtype, kv)
    vc, vs = oracle.quantize_cache(w.v_cache[0], w.dtype, kv)
    rk, rv, rks, rvs, err = oracle.kv_append_quant(w.k_new[0], w.v_new[0], kc, vc, ks, vs,
                                                   w.block_tables, w.context_lens, w.dtype, kv)
    assert (err == 0).all()
    ref, err = oracle.attention(w.q[0], rk, rv, w.block_tables, w.context_lens, w.dtype,
                                b_list=bl, kv=kv, k_scale=rks, v_scale=rvs)
    assert (err == 0).all()
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(gpu)  # noqa: E731
    dkc, dvc, dks, dvs = t(kc), t(vc), t(ks), t(vs)
    del kc, vc
    bt, cl = w.block_tables.to(gpu), w.context_lens.to(gpu)
    st = torch.zeros(1, dtype=torch.int32, device=gpu)
    gq.kv_append_quant(w.k_new[0].to(gpu), w.v_new[0].to(gpu), dkc, dvc, dks, dvs, bt, cl, kv=kv,
                       status=st, pdl=True)
    fn = gq.decode_attention_quant if w.T == 1 else gq.verify_attention_quant
    out = fn(w.q[0].to(gpu), dkc, dvc, dks, dvs, bt, cl, kv=kv, status=st, pdl=True,
             early_kv=True)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    tb = w.block_tables[torch.as_tensor(bl).long()]
    blocks = torch.unique(tb[tb != workloads.INT32_MAX]).long()
    np.testing.assert_array_equal(dkc[blocks.to(gpu)].cpu().numpy(), rk[blocks.numpy()])
    np.testing.assert_array_equal(dvs[blocks.to(gpu)].cpu().numpy(), rvs[blocks.numpy()])
    got = out.cpu()[torch.as_tensor(bl).long()].double().numpy()
    assert_close(got, ref, w.dtype, f"{name} {kv} cache")
