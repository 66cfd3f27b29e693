"""GPU stochastic acceptance (speculative sampling): bit-exact against the
oracle on the same seeded inputs and uniforms (accepted counts and drawn
tokens are integers; both sides take every decision in the same arithmetic)."""
import numpy as np
import pytest
import torch

import gqa_decode_attention_02_gb300 as gq
import oracle
from gqa_decode_attention_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def run(q, p, draft, u, ctx, dev, status=None):
    t = lambda a, dt: torch.as_tensor(np.ascontiguousarray(a), dtype=dt).to(dev)  # noqa: E731
    ctx_d = None if ctx is None else t(ctx, torch.int32)
    acc, nxt = gq.accept_sampled(t(q, torch.float32), t(p, torch.float32),
                                 t(draft, torch.int32), t(u, torch.float64), ctx_d,
                                 status=status)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), nxt.cpu().numpy(), None if ctx_d is None else ctx_d.cpu().numpy()


def check(q, p, draft, u, ctx, dev, expect_status=0):
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ra, rn, rc, err = oracle.accept_sampled(q, p, draft, u, ctx)
    ga, gn, gc = run(q, p, draft, u, ctx, dev, status=st)
    np.testing.assert_array_equal(ga, ra)
    np.testing.assert_array_equal(gn, rn)
    if ctx is not None:
        np.testing.assert_array_equal(gc, rc)
    assert int(st.item()) == expect_status
    if expect_status == 0:
        assert not err.any()
    return ra


@pytest.mark.parametrize("B,T,V,seed", [
    (16, 5, 32000, 205),   # the speculative-verify batch: 16-byte loads
    (16, 5, 32001, 206),   # ragged vocabulary: scalar loads
    (64, 2, 50257, 207),
    (3, 1, 7, 208),        # no drafts: a plain draw from q
    (2, 64, 999, 209),     # longest run
    (300, 3, 100, 210),    # many sequences, segments shorter than a chunk
    (5, 4, 1, 211),        # one-token vocabulary
])
def test_sampled_matches_oracle(gpu, B, T, V, seed):
    s = W.sampling_inputs(B, T, V, seed)
    ctx = np.full(B, 5000, np.int32)
    check(s.q.numpy(), s.p.numpy(), s.draft.numpy(), s.uniforms.numpy(), ctx, gpu)


def test_every_accepted_count_occurs(gpu):
    """Uniforms pushed to 0 keep a draft, pushed towards 1 reject it: plant a
    rejection at every position 0..T-1 (T-1 = all kept)."""
    B, T, V = 40, 5, 4096
    s = W.sampling_inputs(B, T, V, 212)
    q, p, d, u = s.q.numpy(), s.p.numpy(), s.draft.numpy(), s.uniforms.numpy().copy()
    want = np.arange(B) % T
    for b in range(B):
        u[b, : T - 1] = 0.0
        for t in range(T - 1):  # u = 0 keeps draft t iff q(x) > 0
            q[b, t, d[b, t]] = max(q[b, t, d[b, t]], 1e-6)
        if want[b] < T - 1:
            u[b, want[b]] = np.nextafter(1.0, 0)
            x = d[b, want[b]]
            q[b, want[b], x] = 0.5 * p[b, want[b], x]  # q/p = 1/2 < u: rejected
    acc = check(q, p, d, u, None, gpu)
    np.testing.assert_array_equal(acc, want)


def test_unaligned_rows_take_scalar_loads(gpu):
    """The same inputs at a 4-byte offset (rows no longer 16-byte aligned) give
    the same integers."""
    B, T, V = 8, 3, 4096
    s = W.sampling_inputs(B, T, V, 213)
    qa, pa = s.q.to(gpu), s.p.to(gpu)
    qbig = torch.empty(qa.numel() + 1, dtype=torch.float32, device=gpu)
    pbig = torch.empty(pa.numel() + 1, dtype=torch.float32, device=gpu)
    qbig[1:].copy_(qa.flatten())
    pbig[1:].copy_(pa.flatten())
    qv, pv = qbig[1:].view(B, T, V), pbig[1:].view(B, T - 1, V)
    assert qv.data_ptr() % 16 != 0
    d, u = s.draft.to(gpu), s.uniforms.to(gpu)
    a1, n1 = gq.accept_sampled(qa, pa, d, u)
    a2, n2 = gq.accept_sampled(qv, pv, d, u)
    ra, rn, _, _ = oracle.accept_sampled(s.q.numpy(), s.p.numpy(), s.draft.numpy(),
                                         s.uniforms.numpy())
    for a, n in ((a1, n1), (a2, n2)):
        np.testing.assert_array_equal(a.cpu().numpy(), ra)
        np.testing.assert_array_equal(n.cpu().numpy(), rn)


def test_hundred_thousand_draws_on_gpu(gpu):
    """The page's 100 000-draw exercise run through the kernel: the integers
    equal the oracle's, and the emitted law is q."""
    rng = np.random.default_rng(214)
    V, T, n = 5, 2, 100_000
    q = rng.dirichlet(np.ones(V), size=T).astype(np.float32)
    p = rng.dirichlet(np.ones(V), size=T - 1).astype(np.float32)
    c = np.cumsum(p[0].astype(np.float64))
    draft = np.minimum(np.searchsorted(c, rng.random(n) * c[-1], side="right"), V - 1)
    draft = draft.astype(np.int32)[:, None]
    u = rng.random((n, T))
    qt = np.broadcast_to(q, (n, T, V)).copy()
    pt = np.broadcast_to(p, (n, T - 1, V)).copy()
    check(qt, pt, draft, u, None, gpu)
    acc, nxt, _ = run(qt, pt, draft, u, None, gpu)
    first = np.where(acc == 1, draft[:, 0], nxt)
    freq = np.bincount(first, minlength=V) / n
    assert np.all(np.abs(freq - q[0]) < 5 * np.sqrt(q[0] * (1 - q[0]) / n))


def test_vanishing_residual_falls_back_to_target(gpu):
    q = np.array([[[0.5, 0.5], [0.5, 0.5]]], np.float32)
    p = np.array([[[1.0, 0.5]]], np.float32)
    check(q, p, np.array([[0]], np.int32), np.array([[0.7, 0.6]]), None, gpu)


def test_invalid_probability_is_flagged(gpu):
    s = W.sampling_inputs(4, 3, 256, 215)
    q = s.q.numpy().copy()
    q[2, :, 17] = np.nan  # in every row of sequence 2
    check(q, s.p.numpy(), s.draft.numpy(), s.uniforms.numpy(), None, gpu, expect_status=10)


def test_unreached_invalid_entry_is_not_flagged(gpu):
    """A NaN at a draft position after the first rejection is never read by
    the method, so it raises no error (the kernel tests every draft at once)."""
    B, T, V = 2, 4, 64
    s = W.sampling_inputs(B, T, V, 216)
    q, p, d, u = s.q.numpy().copy(), s.p.numpy().copy(), s.draft.numpy(), s.uniforms.numpy()
    u = u.copy()
    u[:, 0] = np.nextafter(1.0, 0)
    q[np.arange(B), 0, d[:, 0]] = 0.0  # draft 0 rejected for sure
    q[np.arange(B), 2, d[:, 2]] = np.nan  # test 2 never reached
    acc = check(q, p, d, u, None, gpu)
    np.testing.assert_array_equal(acc, 0)


def test_bad_uniform_is_flagged(gpu):
    s = W.sampling_inputs(3, 2, 64, 217)
    u = s.uniforms.numpy().copy()
    u[1, 1] = 1.5
    check(s.q.numpy(), s.p.numpy(), s.draft.numpy(), u, None, gpu, expect_status=10)


def test_context_update_underflow_is_reported(gpu):
    B, T, V = 2, 3, 2
    q = np.zeros((B, T, V), np.float32)
    q[:, :, 1] = 1
    p = np.zeros((B, T - 1, V), np.float32)
    p[:, :, 0] = 1
    check(q, p, np.zeros((B, T - 1), np.int32), np.zeros((B, T)), np.array([9, 1], np.int32),
          gpu, expect_status=7)


def test_empty_batch_and_bad_shapes(gpu):
    q = torch.zeros((0, 3, 10), dtype=torch.float32, device=gpu)
    p = torch.zeros((0, 2, 10), dtype=torch.float32, device=gpu)
    d = torch.zeros((0, 2), dtype=torch.int32, device=gpu)
    u = torch.zeros((0, 3), dtype=torch.float64, device=gpu)
    a, n = gq.accept_sampled(q, p, d, u)
    assert a.numel() == 0 and n.numel() == 0
    q = torch.zeros((1, 65, 10), dtype=torch.float32, device=gpu)
    p = torch.zeros((1, 64, 10), dtype=torch.float32, device=gpu)
    d = torch.zeros((1, 64), dtype=torch.int32, device=gpu)
    u = torch.zeros((1, 65), dtype=torch.float64, device=gpu)
    with pytest.raises(gq.GqaError):
        gq.accept_sampled(q, p, d, u)
