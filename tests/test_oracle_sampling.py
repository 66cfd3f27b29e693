"""Pins of the oracle's stochastic acceptance (speculative sampling) against
what the pages and the mathematics fix, not against itself.

"CS336, лекции 10 и 12: инференс и оценка моделей", §"Спекулятивное
сэмплирование": modified rejection sampling with proposal p (draft) and target
q; a draft token is kept with probability min(1, q/p), a rejection is replaced
by a draw from max(q - p, 0), and the emitted token is an exact sample of q
(the two-token proof, its numeric check, and the exercise that checks a
5-token vocabulary by drawing 100 000 times).
"""
import json
import pathlib

import numpy as np
import pytest

import oracle

GOLDEN = pathlib.Path(__file__).parent / "golden"


def tile(a, n):
    a = np.asarray(a)
    return np.broadcast_to(a, (n,) + a.shape).copy()


def run_one_draft(q0, q1, p0, x, u_acc, u_draw):
    """T = 2 (one draft) for many uniforms at once: returns (accepted, token)."""
    n = len(u_acc)
    V = len(q0)
    q = tile(np.stack([q0, q1]).astype(np.float32), n)
    p = tile(np.asarray(p0, np.float32)[None], n)
    d = np.full((n, 1), x, np.int32)
    u = np.stack([u_acc, u_draw], axis=1)
    acc, nxt, _, err = oracle.accept_sampled(q, p, d, u)
    assert not err.any()
    assert q.shape == (n, 2, V)
    return acc, nxt


def accept_threshold(q0, p0, x):
    """The u at which draft x switches from kept to rejected (bisection; the
    decision is monotone in u)."""
    lo, hi = 0.0, 1.0
    q1 = np.full(len(q0), 1.0 / len(q0))
    acc, _ = run_one_draft(q0, q1, p0, x, np.array([0.0, np.nextafter(1.0, 0)]),
                           np.array([0.5, 0.5]))
    if acc[1] == 1:
        return 1.0
    if acc[0] == 0:
        return 0.0
    for _ in range(60):
        mid = 0.5 * (lo + hi)
        a, _ = run_one_draft(q0, q1, p0, x, np.array([mid]), np.array([0.5]))
        lo, hi = (mid, hi) if a[0] == 1 else (lo, mid)
    return lo


def draw_law(q0, p0, x, M=200_000):
    """Law of the token drawn after draft x is rejected, over a uniform grid of
    M points in [0, 1)."""
    V = len(q0)
    q1 = np.full(V, 1.0 / V)
    ug = (np.arange(M) + 0.5) / M
    acc, tok = run_one_draft(q0, q1, p0, x, np.full(M, np.nextafter(1.0, 0)), ug)
    assert not acc.any()
    return np.bincount(tok, minlength=V) / M


def test_page_two_token_example():
    """The page's numeric check: q = [0.6, 0.4], p = [0.9, 0.1].  A is kept with
    probability 2/3 (contribution 0.6), B always (0.1), a rejected A is always
    replaced by B (0.3), so the emitted law is exactly q."""
    g = json.loads((GOLDEN / "speculative_sampling_example.json").read_text())
    q, p = np.array(g["q_target"]), np.array(g["p_draft"])
    a_A = accept_threshold(q, p, 0)
    a_B = accept_threshold(q, p, 1)
    # exact for the fp32 inputs; the page's decimals to fp32 resolution
    q32, p32 = q.astype(np.float32).astype(np.float64), p.astype(np.float32).astype(np.float64)
    assert a_A == pytest.approx(q32[0] / p32[0], abs=1e-12)
    assert a_A == pytest.approx(g["accept_prob_A"], abs=1e-6)
    assert a_B == g["accept_prob_B"]
    assert p[0] * a_A == pytest.approx(g["contribution_accepted_A"], abs=1e-6)
    assert p[1] * a_B == pytest.approx(g["contribution_accepted_B"], abs=1e-12)
    assert p[0] * (1 - a_A) == pytest.approx(g["contribution_rejected_A_replaced_by_B"],
                                             abs=1e-6)
    res = draw_law(q, p, 0, M=10_000)
    np.testing.assert_array_equal(res, g["residual"])
    emitted = p[0] * (a_A * np.array([1, 0]) + (1 - a_A) * res) + p[1] * np.array([0, 1])
    np.testing.assert_allclose(emitted, g["emitted"], atol=1e-6)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_exact_emitted_law_five_tokens(seed):
    """The proof, numerically and without sampling noise: for each draft x the
    keep probability equals min(1, q(x)/p(x)) and the replacement law equals the
    normalised residual, so sum_x p(x)[keep(x) 1{v=x} + (1-keep(x)) res_x(v)]
    equals q(v)."""
    rng = np.random.default_rng(seed)
    V = 5
    q = rng.dirichlet(np.ones(V)).astype(np.float32).astype(np.float64)
    p = rng.dirichlet(np.ones(V)).astype(np.float32).astype(np.float64)
    resid = np.maximum(q - p, 0)
    resid /= resid.sum()
    emitted = np.zeros(V)
    for x in range(V):
        keep = accept_threshold(q, p, x)
        assert keep == pytest.approx(min(1.0, q[x] / p[x]), abs=1e-12)  # q, p fp32-exact
        emitted[x] += p[x] * keep
        if keep < 1:
            law = draw_law(q, p, x)
            np.testing.assert_allclose(law, resid, atol=2e-5)
            emitted += p[x] * (1 - keep) * law
    np.testing.assert_allclose(emitted, q, atol=3e-5)


def test_hundred_thousand_draws_match_target():
    """The page's exercise: a 5-token vocabulary, 100 000 draws of the full
    draft-then-verify step (drafts drawn from p), emitted law == q.  Three
    drafts: every emitted position i follows q_i."""
    rng = np.random.default_rng(7)
    V, T, n = 5, 4, 100_000
    q = rng.dirichlet(np.ones(V), size=T).astype(np.float32)
    p = rng.dirichlet(np.ones(V), size=T - 1).astype(np.float32)
    cp = np.cumsum(p.astype(np.float64), axis=1)
    cp[:, -1] = 1.0
    draft = np.stack([np.searchsorted(cp[t], rng.random(n), side="right")
                      for t in range(T - 1)], axis=1).astype(np.int32)
    u = rng.random((n, T))
    acc, nxt, _, err = oracle.accept_sampled(tile(q, n), tile(p, n), draft, u)
    assert not err.any()
    for i in range(T):
        # position i is emitted when at least i drafts were kept
        sel = acc >= i
        tok = np.where(acc[sel] > i, draft[sel][:, min(i, T - 2)], nxt[sel])
        m = int(sel.sum())
        freq = np.bincount(tok, minlength=V) / m
        sigma = np.sqrt(q[i] * (1 - q[i]) / m)
        assert np.all(np.abs(freq - q[i]) < 5 * sigma + 1e-9), (i, freq, q[i])


def test_inverse_cdf_boundaries_exact():
    """Weights that are multiples of 2^-40 are drawn with no rounding at all:
    q = [1/4, 1/4, 1/2] switches token exactly at u = 1/4 and u = 1/2."""
    q0 = np.array([0.25, 0.25, 0.5])
    u = np.array([0.0, np.nextafter(0.25, 0), 0.25, np.nextafter(0.5, 0), 0.5,
                  np.nextafter(1.0, 0)])
    n = len(u)
    acc, tok, _, err = oracle.accept_sampled(tile(q0[None].astype(np.float32), n),
                                             np.zeros((n, 0, 3), np.float32),
                                             np.zeros((n, 0), np.int32), u[:, None])
    assert not err.any() and not acc.any()
    np.testing.assert_array_equal(tok, [0, 0, 1, 1, 2, 2])


def test_zero_probability_token_never_drawn():
    q0 = np.array([0.0, 0.3, 0.0, 0.7, 0.0], np.float32)
    M = 50_000
    u = ((np.arange(M) + 0.5) / M)[:, None]
    _, tok, _, err = oracle.accept_sampled(tile(q0[None], M), np.zeros((M, 0, 5), np.float32),
                                           np.zeros((M, 0), np.int32), u)
    assert not err.any()
    assert set(np.unique(tok)) == {1, 3}
    assert (tok == 1).mean() == pytest.approx(0.3, abs=1e-4)


def test_draft_equal_target_keeps_everything():
    """p == q: u * p(x) < q(x) for every u in [0, 1), so every draft is kept
    and the final token is drawn from q_{T-1}."""
    rng = np.random.default_rng(3)
    B, T, V = 64, 5, 11
    q = rng.dirichlet(np.ones(V), size=(B, T)).astype(np.float32)
    draft = rng.integers(0, V, size=(B, T - 1)).astype(np.int32)
    q[np.arange(B)[:, None], np.arange(T - 1)[None], draft] += 0.01  # p(x) > 0
    u = rng.random((B, T))
    u[:, :-1] = np.nextafter(1.0, 0)
    acc, nxt, _, err = oracle.accept_sampled(q, q[:, :-1], draft, u)
    assert not err.any()
    assert (acc == T - 1).all()
    # the bonus token alone, as a T = 1 call with the same uniform
    _, nb, _, _ = oracle.accept_sampled(q[:, -1:], np.zeros((B, 0, V), np.float32),
                                        np.zeros((B, 0), np.int32), u[:, -1:])
    np.testing.assert_array_equal(nxt, nb)


def test_disjoint_one_hots_reject_and_take_target():
    B, T, V = 8, 3, 6
    q = np.zeros((B, T, V), np.float32)
    p = np.zeros((B, T - 1, V), np.float32)
    y = np.arange(B) % V
    x = (y + 1) % V
    q[:, :, :] = 0
    q[np.arange(B), 0, y] = 1
    q[:, 1:, 0] = 1
    p[np.arange(B), 0, x] = 1
    p[:, 1, 0] = 1
    draft = np.stack([x, np.zeros(B, int)], axis=1).astype(np.int32)
    acc, nxt, _, err = oracle.accept_sampled(q, p, draft, np.zeros((B, T)))
    assert not err.any()
    np.testing.assert_array_equal(acc, 0)
    np.testing.assert_array_equal(nxt, y)


def test_greedy_limit_matches_greedy_acceptance():
    """One-hot target and draft distributions (the temperature-0 limit) make
    the sampler deterministic: it must then agree with greedy longest-prefix
    acceptance on the logits whose argmax the one-hots mark."""
    rng = np.random.default_rng(11)
    B, T, V = 200, 5, 40
    logits = rng.normal(size=(B, T, V)).astype(np.float32)
    g = logits.argmax(-1)
    draft = np.where(rng.random((B, T - 1)) < 0.7, g[:, :-1],
                     rng.integers(0, V, size=(B, T - 1))).astype(np.int32)
    q = np.zeros((B, T, V), np.float32)
    np.put_along_axis(q, g[..., None], 1.0, axis=-1)
    p = np.zeros((B, T - 1, V), np.float32)
    np.put_along_axis(p, draft[..., None].astype(np.int64), 1.0, axis=-1)
    ctx = np.full(B, 100, np.int32)
    acc, nxt, cl, err = oracle.accept_sampled(q, p, draft, rng.random((B, T)), ctx)
    ga, gn, gc = oracle.accept_prefix(logits, draft, ctx)
    assert not err.any()
    np.testing.assert_array_equal(acc, ga)
    np.testing.assert_array_equal(nxt, gn)
    np.testing.assert_array_equal(cl, gc)


def test_vanishing_residual_falls_back_to_target():
    """A rejected draft whose residual has no weight (only possible when p is
    not normalised or rounding makes q <= p everywhere) draws from q."""
    q = np.array([[[0.5, 0.5], [0.5, 0.5]]], np.float32)
    p = np.array([[[1.0, 0.5]]], np.float32)
    acc, nxt, _, err = oracle.accept_sampled(q, p, [[0]], [[0.7, 0.6]])
    assert acc[0] == 0 and nxt[0] == 1 and err[0] == 0


def test_invalid_inputs_flagged():
    q = np.full((4, 2, 3), 1 / 3, np.float32)
    p = np.full((4, 1, 3), 1 / 3, np.float32)
    q[0, 0, 1] = np.nan           # read by the draft test
    q[1, 1, 2] = -0.5             # read by the bonus draw
    u = np.full((4, 2), 0.5)
    u[2, 0] = 1.0                 # not in [0, 1)
    draft = np.array([[1], [0], [0], [7]], np.int32)  # 7: out of range -> rejected
    acc, nxt, _, err = oracle.accept_sampled(q, p, draft, u)
    np.testing.assert_array_equal(err, [10, 10, 10, 0])
    assert acc[3] == 0 and acc[2] == 1  # u taken as 0 keeps the draft


def test_context_update_and_underflow():
    q = np.zeros((2, 3, 2), np.float32)
    q[:, :, 1] = 1
    p = np.zeros((2, 2, 2), np.float32)
    p[:, :, 0] = 1
    ctx = np.array([9, 1], np.int32)
    acc, nxt, cl, err = oracle.accept_sampled(q, p, np.zeros((2, 2), np.int32),
                                              np.zeros((2, 3)), ctx)
    np.testing.assert_array_equal(acc, [0, 0])
    np.testing.assert_array_equal(nxt, [1, 1])
    np.testing.assert_array_equal(cl, [7, 1])
    np.testing.assert_array_equal(err, [0, 7])
