"""Pins of the oracle's one-byte KV cache (int8 and e4m3 codes with a per-row
fp32 scale) against the pages' rule, the e4m3 format definition, a library
implementation of e4m3 (torch.float8_e4m3fn) and an independent recompute.

"جعل inference رخيصًا: KV cache وbatching والتكميم", quantization section:
symmetric absolute-maximum quantization (qmax = 2^(bits-1) - 1, scale =
max|W| / qmax, codes round(W / scale) clamped to [-qmax-1, qmax], W_hat =
codes * scale).  "CS336, лекции 10 и 12", §"Квантование": fp8 (e4m3) and int8.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import small, unpage

E4M3_MAX = 448.0


# ---- e4m3 codes ----------------------------------------------------------------------
def test_e4m3_decode_matches_torch_for_all_codes():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_to_f64(c) for c in range(256)])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert set(np.flatnonzero(np.isnan(got))) == {0x7F, 0xFF}
    np.testing.assert_array_equal(got[~both_nan], ref[~both_nan])


def test_e4m3_landmarks_and_order():
    # the format's own landmarks: 1.0, the largest finite 448, the smallest
    # normal 2^-6 and subnormal 2^-9; codes 0x00..0x7e strictly increasing
    assert oracle.e4m3_to_f64(0x38) == 1.0
    assert oracle.e4m3_to_f64(0x7E) == E4M3_MAX
    assert oracle.e4m3_to_f64(0x08) == 2.0 ** -6
    assert oracle.e4m3_to_f64(0x01) == 2.0 ** -9
    vals = [oracle.e4m3_to_f64(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(vals, vals[1:]))
    for c in range(0x7F):  # encode(decode(c)) == c, and the sign bit mirrors
        assert oracle.e4m3_from_float(vals[c]) == c
        if c:
            assert oracle.e4m3_from_float(-vals[c]) == c | 0x80


def test_e4m3_encode_matches_torch_in_range():
    """Round to nearest, ties to even, against torch.float8_e4m3fn on every
    representable value, every midpoint between neighbours, and a dense sweep
    (|x| < 464, where torch does not produce NaN)."""
    vals = np.array([oracle.e4m3_to_f64(c) for c in range(0x7F)])
    mids = (vals[:-1] + vals[1:]) / 2
    rng = np.random.default_rng(0)
    sweep = np.exp(rng.uniform(math.log(1e-4), math.log(463.0), 20000))
    xs = np.concatenate([vals, mids, sweep, np.nextafter(mids, 0), np.nextafter(mids, 1e9)])
    xs = np.concatenate([xs, -xs]).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_from_float(float(x)) for x in xs], np.uint8)
    np.testing.assert_array_equal(got, ref)


def test_e4m3_saturates_instead_of_overflowing():
    for x in (464.0, 500.0, 1e30, float("inf")):
        assert oracle.e4m3_from_float(x) == 0x7E
        assert oracle.e4m3_from_float(-x) == 0xFE


# ---- the row quantizer ----------------------------------------------------------------
def rows(dtype, n=64, H=128, seed=0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, H, generator=g) * torch.exp(torch.randn(n, 1, generator=g) * 2)
    return x.to(torch.bfloat16 if dtype == "bf16" else torch.float16)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_int8_absmax_rule(dtype):
    x = rows(dtype)
    for r in range(x.shape[0]):
        codes, sc = oracle.quantize_row(x[r], dtype, "int8")
        xr = x[r].double().numpy()
        c = codes.view(np.int8).astype(np.float64)
        amax = np.abs(xr).max()
        assert sc == pytest.approx(amax / 127, rel=1e-6)
        # the largest element maps to +-127, every code lies in [-127, 127]
        i = int(np.argmax(np.abs(xr)))
        assert abs(c[i]) == 127 and np.sign(c[i]) == np.sign(xr[i])
        assert np.abs(c).max() <= 127
        # reconstruction within half a step
        assert np.all(np.abs(xr - c * sc) <= sc * (0.5 + 1e-5))


@pytest.mark.parametrize("kv", ["int8", "e4m3"])
def test_quantizer_sign_symmetry_and_power_of_two_scaling(kv):
    x = rows("bf16", n=16, seed=1)
    for r in range(x.shape[0]):
        c1, s1 = oracle.quantize_row(x[r], "bf16", kv)
        c2, s2 = oracle.quantize_row(-x[r], "bf16", kv)
        c3, s3 = oracle.quantize_row(x[r] * 4, "bf16", kv)
        if kv == "int8":
            np.testing.assert_array_equal(c2.view(np.int8), -c1.view(np.int8))
        else:
            np.testing.assert_array_equal(c2 ^ 0x80, c1)
        assert s2 == s1
        np.testing.assert_array_equal(c3, c1)
        assert s3 == 4 * s1


def test_e4m3_rule_relative_error():
    x = rows("bf16", seed=2)
    for r in range(x.shape[0]):
        codes, sc = oracle.quantize_row(x[r], "bf16", "e4m3")
        xr = x[r].double().numpy()
        assert sc == pytest.approx(np.abs(xr).max() / E4M3_MAX, rel=1e-6)
        deq = np.array([oracle.e4m3_to_f64(c) for c in codes]) * sc
        i = int(np.argmax(np.abs(xr)))
        assert codes[i] & 0x7F == 0x7E  # the largest element maps to +-448
        # three mantissa bits: half a step is 2^-4 of the value in the normal
        # range; below it (|x/scale| < 2^-6) an absolute 2^-10 of a scale unit
        err = np.abs(xr - deq)
        assert np.all(err <= np.maximum(np.abs(xr) * 2.0 ** -4, sc * 2.0 ** -10) * (1 + 1e-6))


@pytest.mark.parametrize("kv", ["int8", "e4m3"])
def test_zero_row(kv):
    codes, sc = oracle.quantize_row(torch.zeros(128, dtype=torch.bfloat16), "bf16", kv)
    assert sc == 0.0 and (codes == 0).all()


@pytest.mark.parametrize("kv", ["int8", "e4m3"])
def test_nan_element_leaves_the_rest_of_the_row_as_if_it_were_zero(kv):
    """A NaN element (outside the contract: the pages quantize finite values)
    does not enter max|x| -- the row's scale and every other code are those of
    the same row with that element at zero -- and gets code 0 for int8 and
    e4m3's NaN code 0x7f, the code torch.float8_e4m3fn gives a NaN."""
    x = torch.randn(128, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    x[17] = float("nan")
    zeroed = x.clone()
    zeroed[17] = 0.0
    codes, sc = oracle.quantize_row(x, "bf16", kv)
    codes0, sc0 = oracle.quantize_row(zeroed, "bf16", kv)
    assert sc == sc0 and sc > 0
    keep = np.arange(128) != 17
    np.testing.assert_array_equal(codes[keep], codes0[keep])
    if kv == "int8":
        assert codes[17] == 0
    else:
        want = torch.tensor([float("nan")]).to(torch.float8_e4m3fn).view(torch.uint8).item()
        assert codes[17] == want == 0x7F


# ---- quantized append and attention --------------------------------------------------
def empty_quant_cache(w):
    NB, bs, K, H = w.k_cache[0].shape
    kc = np.zeros((NB, bs, K, H), np.uint8)
    vc = np.zeros_like(kc)
    ks = np.zeros((NB, K, bs), np.float32)
    vs = np.zeros_like(ks)
    return kc, vc, ks, vs


def fill_quant_cache(w, kv):
    """Quantize every cached (non-new) position of layer 0 through the oracle's
    own append, one position at a time: returns the one-byte caches."""
    kc, vc, ks, vs = empty_quant_cache(w)
    ctx = w.context_lens.numpy()
    T = w.T
    for b, c in enumerate(ctx):
        kk, vv = unpage(w, b, int(c))
        for pos in range(int(c) - (T if w.appended else 0)):
            one = torch.tensor([pos + 1], dtype=torch.int32)
            kn = torch.from_numpy(kk[pos][None, None]).to(w.torch_dtype)
            vn = torch.from_numpy(vv[pos][None, None]).to(w.torch_dtype)
            kc, vc, ks, vs, err = oracle.kv_append_quant(kn, vn, kc, vc, ks, vs,
                                                         w.block_tables[b:b + 1], one,
                                                         w.dtype, kv)
            assert err[0] == 0
    return kc, vc, ks, vs


@pytest.mark.parametrize("kv", ["int8", "e4m3"])
def test_quant_append_writes_each_row_and_nothing_else(kv):
    T = 3
    w = small(B=3, T=T, N=8, K=2, H=128, dtype="bf16", ctx=(3, 20, 47), seed=61, append=True)
    kc, vc, ks, vs = empty_quant_cache(w)
    kc[:] = 0xA5
    ks[:] = -1.0
    kc2, vc2, ks2, vs2, err = oracle.kv_append_quant(w.k_new[0], w.v_new[0], kc, vc, ks, vs,
                                                     w.block_tables, w.context_lens, "bf16", kv)
    assert (err == 0).all()
    touched = np.zeros(kc.shape[:3], bool)
    for b, c in enumerate((3, 20, 47)):
        for t in range(T):
            pos = c - T + t
            blk, r = int(w.block_tables[b, pos // 16]), pos % 16
            for k in range(2):
                codes, sc = oracle.quantize_row(w.k_new[0][b, t, k], "bf16", kv)
                np.testing.assert_array_equal(kc2[blk, r, k], codes)
                assert ks2[blk, k, r] == np.float32(sc)
                codes, sc = oracle.quantize_row(w.v_new[0][b, t, k], "bf16", kv)
                np.testing.assert_array_equal(vc2[blk, r, k], codes)
                assert vs2[blk, k, r] == np.float32(sc)
                touched[blk, r, k] = True
    assert (kc2[~touched] == 0xA5).all()
    assert (ks2.transpose(0, 2, 1)[~touched] == -1.0).all()


@pytest.mark.parametrize("kv", ["int8", "e4m3"])
@pytest.mark.parametrize("T", [1, 3])
def test_quant_attention_equals_recompute_on_dequantized_cache(kv, T):
    """The paged attention over one-byte codes times their row scales equals
    causal attention recomputed (numpy, fp64) over the dequantized K and V."""
    ctx = (T, 30, 77)
    w = small(B=3, T=T, N=8, K=2, H=128, dtype="bf16", ctx=ctx, seed=62 + T)
    kc, vc, ks, vs = fill_quant_cache(w, kv)
    out, err = oracle.attention(w.q[0], kc, vc, w.block_tables, w.context_lens, "bf16",
                                kv=kv, k_scale=ks, v_scale=vs)
    assert (err == 0).all()
    dec = (lambda c: c.view(np.int8).astype(np.float64)) if kv == "int8" else (
        lambda c: np.vectorize(oracle.e4m3_to_f64)(c))
    gen = torch.Generator().manual_seed(5)
    for b, c in enumerate(ctx):
        kd = np.zeros((c, 2, 128))
        vd = np.zeros((c, 2, 128))
        for pos in range(c):
            blk, r = int(w.block_tables[b, pos // 16]), pos % 16
            for k in range(2):
                kd[pos, k] = dec(kc[blk, r, k]) * ks[blk, k, r]
                vd[pos, k] = dec(vc[blk, r, k]) * vs[blk, k, r]
        q_all = torch.randn(c, 8, 128, generator=gen).double().numpy()
        q_all[c - T:] = w.q[0][b].double().numpy()
        full = oracle.causal_attention_full(q_all, kd, vd, 1.0 / math.sqrt(128))
        np.testing.assert_allclose(out[b], full[c - T:], rtol=0, atol=1e-12)


@pytest.mark.parametrize("kv,tol", [("int8", 0.02), ("e4m3", 0.08)])
def test_quant_attention_stays_near_the_unquantized_one(kv, tol):
    ctx = (40, 300)
    w = small(B=2, T=1, N=8, K=2, H=128, dtype="bf16", ctx=ctx, seed=63)
    kc, vc, ks, vs = fill_quant_cache(w, kv)
    ref, _ = oracle.attention(w.q[0], w.k_cache[0], w.v_cache[0], w.block_tables,
                              w.context_lens, "bf16")
    got, _ = oracle.attention(w.q[0], kc, vc, w.block_tables, w.context_lens, "bf16",
                              kv=kv, k_scale=ks, v_scale=vs)
    assert np.abs(got - ref).max() < tol
