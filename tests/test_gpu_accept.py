"""GPU accept_prefix: bit-exact against the oracle (integers), ties, NaN, -0;
both kernels (many blocks per sequence meeting in a workspace, and one
thread-block cluster per sequence without one)."""
import numpy as np
import pytest
import torch

import gqa_decode_attention_02_gb300 as gq
import oracle
from helpers import small

pytestmark = pytest.mark.gpu


KERNELS = [False, True]  # cluster=False: the workspace kernel; True: one cluster per sequence


def run(lg, draft, ctx, dev, cluster=False, workspace=None):
    lg_d = torch.as_tensor(lg).to(dev).contiguous()
    dr_d = torch.as_tensor(draft, dtype=torch.int32).to(dev).contiguous()
    ctx_d = None if ctx is None else torch.as_tensor(ctx, dtype=torch.int32).to(dev)
    acc, nxt = gq.accept_prefix(lg_d, dr_d, ctx_d, cluster=cluster, workspace=workspace)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), nxt.cpu().numpy(), None if ctx_d is None else ctx_d.cpu().numpy()


@pytest.mark.parametrize("cluster", KERNELS)
@pytest.mark.parametrize("B,T,V", [(16, 5, 32000), (3, 1, 7), (4, 8, 50257), (2, 64, 999),
                                   (300, 2, 100), (1, 5, 3), (1000, 5, 4096)])
def test_accept_matches_oracle(gpu, B, T, V, cluster):
    w = small(B=B, T=T, N=1, K=1, H=64, ctx=(70,) * B, seed=B + T, vocab=V)
    ctx = np.full(B, 70, np.int32)
    ra, rn, rc = oracle.accept_prefix(w.logits, w.draft, ctx)
    ga, gn, gc = run(w.logits, w.draft, ctx, gpu, cluster)
    np.testing.assert_array_equal(ga, ra)
    np.testing.assert_array_equal(gn, rn)
    np.testing.assert_array_equal(gc, rc)


@pytest.mark.parametrize("cluster", KERNELS)
def test_accept_ties_nan_negative_zero(gpu, cluster):
    rng = np.random.default_rng(3)
    B, T, V = 64, 4, 37
    lg = rng.integers(-2, 3, size=(B, T, V)).astype(np.float32)  # heavy ties
    lg[::3, :, 5] = np.nan
    lg[1::4, :, :] = 0.0
    lg[1::4, :, 7] = -0.0
    lg[2::5] = -np.inf
    draft = rng.integers(0, V, size=(B, T - 1)).astype(np.int32)
    for b in range(0, B, 2):  # make some drafts right
        for t in range(T - 1):
            draft[b, t] = oracle.argmax(lg[b, t])
    ra, rn, _ = oracle.accept_prefix(lg, draft)
    ga, gn, _ = run(lg, draft, None, gpu, cluster)
    np.testing.assert_array_equal(ga, ra)
    np.testing.assert_array_equal(gn, rn)


@pytest.mark.parametrize("cluster", KERNELS)
def test_context_length_update_underflow_is_reported(gpu, cluster):
    lg = np.zeros((2, 3, 4), np.float32)
    draft = np.full((2, 2), 3, np.int32)  # argmax is 0 everywhere -> reject all
    ctx = torch.tensor([5, 1], dtype=torch.int32, device=gpu)
    st = torch.zeros(1, dtype=torch.int32, device=gpu)
    gq.accept_prefix(torch.as_tensor(lg).to(gpu), torch.as_tensor(draft).to(gpu), ctx,
                     status=st, cluster=cluster)
    torch.cuda.synchronize()
    assert ctx.cpu().tolist() == [3, 1]
    assert int(st.item()) == 7


@pytest.mark.parametrize("cluster", KERNELS)
@pytest.mark.parametrize("V", [32768, 32001])  # 16-byte loads; scalar loads
def test_accept_ties_across_cluster_slices(gpu, V, cluster):
    """Equal maxima and NaNs in several blocks' column slices: the smallest
    index still wins, over more rows than one pass holds."""
    rng = np.random.default_rng(V)
    B, T = 6, 13
    lg = rng.integers(-3, 2, size=(B, T, V)).astype(np.float32)  # max 1, ties everywhere
    lg[0, :, V - 5] = np.nan  # a NaN only in the last slice
    lg[1, :, ::4097] = np.nan  # NaNs in every slice: the first one wins
    lg[2, :, :] = -0.0
    lg[2, :, V // 2] = 0.0  # +0 ties with -0: index 0 wins
    lg[3, :, V - 1] = 2.0  # a unique maximum at the very end
    draft = np.zeros((B, T - 1), np.int32)
    for b in range(B):
        for t in range(T - 1):
            draft[b, t] = oracle.argmax(lg[b, t]) if (b + t) % 5 else 1
    ra, rn, _ = oracle.accept_prefix(lg, draft)
    ga, gn, _ = run(lg, draft, None, gpu, cluster)
    np.testing.assert_array_equal(ga, ra)
    np.testing.assert_array_equal(gn, rn)


def test_workspace_returns_to_zero_and_is_reused_across_sizes(gpu):
    """One caller workspace over calls of different sizes: every call leaves it
    zero-filled, and each result matches the oracle."""
    from gqa_decode_attention_02_gb300 import _lib

    need = _lib.lib().gqa_accept_workspace_size(512, 8)
    ws = torch.zeros(need, dtype=torch.uint8, device=gpu)
    for i, (B, T, V) in enumerate([(512, 8, 1000), (16, 5, 32000), (7, 3, 33), (512, 1, 64)]):
        w = small(B=B, T=T, N=1, K=1, H=64, ctx=(70,) * B, seed=100 + i, vocab=V)
        ra, rn, _ = oracle.accept_prefix(w.logits, w.draft)
        ga, gn, _ = run(w.logits, w.draft, None, gpu, workspace=ws)
        np.testing.assert_array_equal(ga, ra)
        np.testing.assert_array_equal(gn, rn)
        assert int(ws.count_nonzero().item()) == 0


def test_many_sequences_beyond_the_cluster_grid(gpu):
    """B > 65535 sequences: only the workspace kernel takes them."""
    rng = np.random.default_rng(11)
    B, T, V = 70000, 2, 8
    lg = rng.standard_normal((B, T, V)).astype(np.float32)
    draft = rng.integers(0, V, size=(B, T - 1)).astype(np.int32)
    ra, rn, _ = oracle.accept_prefix(lg, draft)
    ga, gn, _ = run(lg, draft, None, gpu)
    np.testing.assert_array_equal(ga, ra)
    np.testing.assert_array_equal(gn, rn)
    with pytest.raises(gq.GqaError):
        run(lg, draft, None, gpu, cluster=True)
