"""Pins for the oracle's verifier and the closed forms of one round."""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from oracle import theory

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                rows.append([float(x) for x in line.split()])
    return rows


# ------------------------------------------------------------- closed forms
def test_expected_tokens_table_gamma4():
    """The explainer's table: alpha -> tokens per round at gamma = 4."""
    for alpha, printed in _read_golden("expected_tokens_gamma4.txt"):
        e = theory.expected_tokens_equal_alpha(alpha, 4)
        assert round(e, 1) == printed
        # the product form with equal alphas is the same number
        assert abs(theory.expected_tokens([alpha] * 4) - e) < 1e-12


def test_expected_tokens_limits():
    assert theory.expected_tokens([Fraction(0)] * 5) == 1
    assert theory.expected_tokens([Fraction(1)] * 5) == 6
    assert theory.expected_tokens_equal_alpha(1, 5) == 6


def test_acceptance_rate_bounds_by_kept_mass():
    """SlimSpec article section 四: a drafter whose distribution is zero off a
    kept vocabulary has alpha at most the target's mass on that vocabulary."""
    rng = np.random.default_rng(0)
    p = rng.dirichlet(np.ones(50))
    keep = rng.random(50) < 0.5
    q = np.where(keep, rng.dirichlet(np.ones(50)), 0.0)
    q /= q.sum()
    assert theory.acceptance_rate(p, q) <= p[keep].sum() + 1e-15
    assert abs(theory.acceptance_rate(p, p) - 1.0) < 1e-12


# --------------------------------------------------------------- greedy ----
def test_greedy_worked_examples():
    for gamma, lead, emitted, accepted in _read_golden("greedy_rounds.txt"):
        gamma, lead = int(gamma), int(lead)
        V = 10
        target = np.zeros((gamma + 1, V))
        a = [(3 * j + 1) % V for j in range(gamma + 1)]
        for j in range(gamma + 1):
            target[j, a[j]] = 5.0
        x = [a[j] if j < lead else (a[j] + 1) % V for j in range(gamma)]
        toks, n = oracle.verify_greedy(target, x)
        assert n == accepted and len(toks) == emitted


def test_greedy_invariant_every_token_is_target_argmax():
    v = synth.verify_logits(7, B=6, gamma=5, V=300, kind="normal")
    rng = np.random.default_rng(1)
    for b in range(6):
        t = v["target"][b]
        a = np.argmax(t, axis=1)
        # drafts that agree with the target on a random prefix
        x = a[:5].copy()
        cut = rng.integers(0, 6)
        if cut < 5:
            x[cut] = (x[cut] + 1) % 300
        toks, n = oracle.verify_greedy(t, x)
        assert n == min(cut, 5)
        assert len(toks) == n + 1
        assert all(toks[j] == a[j] for j in range(len(toks)))


def test_greedy_ties_go_to_the_lowest_index():
    """Rows of small integers (many exact ties at the maximum): the target's
    choice at every position is numpy's argmax, which returns the first
    occurrence, so a draft token equal to a later tied maximum is rejected."""
    rng = np.random.default_rng(11)
    gamma, V = 4, 12
    for _ in range(50):
        t = rng.integers(0, 4, (gamma + 1, V)).astype(np.float64)
        a = np.argmax(t, axis=1)
        # the drafter picks the last tied maximum at a random position
        cut = int(rng.integers(0, gamma))
        x = a[:gamma].copy()
        ties = np.nonzero(t[cut] == t[cut].max())[0]
        x[cut] = ties[-1]
        toks, n = oracle.verify_greedy(t, x)
        want_n = cut if ties[-1] != a[cut] else (
            next((j for j in range(cut + 1, gamma) if x[j] != a[j]), gamma))
        assert n == want_n
        assert toks[-1] == a[n]


# ------------------------------------------------------------- sampling ----
def _rand_dist(rng, V, zero_some=False):
    w = [Fraction(int(x)) for x in rng.integers(1, 9, V)]
    if zero_some:
        w[int(rng.integers(0, V))] = Fraction(0)
    s = sum(w)
    return [x / s for x in w]


@pytest.mark.parametrize("V,gamma,seed", [(3, 2, 0), (4, 2, 1), (3, 3, 2), (4, 1, 3)])
def test_exhaustive_output_distribution_equals_target(V, gamma, seed):
    """Explainer "为什么答案不会变": accept + residual resampling reproduces p
    exactly.  Every emitted token, conditioned on the tokens before it in the
    same round, is distributed as the target row at its position; acceptance
    at position j happens with probability sum_x min(p_j, q_j); the expected
    number of tokens is sum_j prod_{i<j} alpha_i."""
    rng = np.random.default_rng(seed)
    p = [_rand_dist(rng, V) for _ in range(gamma + 1)]
    q = [_rand_dist(rng, V, zero_some=(j == 0)) for j in range(gamma)]
    dist = theory.enumerate_round(p, q)
    assert sum(dist.values()) == 1

    # marginal of the i-th emitted token given the previous ones
    for i in range(gamma + 1):
        joint = {}
        for (toks, n), pr in dist.items():
            if len(toks) > i:
                joint.setdefault(toks[:i], {}).setdefault(toks[i], Fraction(0))
                joint[toks[:i]][toks[i]] += pr
        for prefix, cond in joint.items():
            tot = sum(cond.values())
            for v in range(V):
                assert cond.get(v, Fraction(0)) / tot == p[i][v]

    alphas = [theory.acceptance_rate(p[j], q[j]) for j in range(gamma)]
    reach = Fraction(1)
    for j in range(gamma):
        p_ge = sum(pr for (toks, n), pr in dist.items() if n >= j)
        p_gt = sum(pr for (toks, n), pr in dist.items() if n > j)
        assert p_ge == reach
        assert p_gt == reach * alphas[j]
        reach *= alphas[j]
    mean = sum(pr * len(toks) for (toks, n), pr in dist.items())
    assert mean == theory.expected_tokens(alphas)


def test_all_zero_residual_falls_back_to_target():
    p = [np.array([0.1, 0.2]), np.array([0.5, 0.5])]
    q = [np.array([0.5, 0.5])]
    toks, n = oracle.verify_decide(p, q, [0], [0.5, 0.9])
    assert n == 0
    assert toks == [oracle.inverse_cdf(p[0], 0.9)] == [1]


def test_monte_carlo_acceptance_matches_alpha():
    """Float path: acceptance frequency of verify_sampling at position 0 over
    draws x ~ q, u ~ U(0,1) matches sum_x min(p, q) within 4 sigma."""
    v = synth.verify_logits(9, B=1, gamma=1, V=64, kind="normal", draft_sigma=1.0)
    T = 1.0
    p = oracle.softmax_t(v["target"][0, 0], T)
    q = oracle.softmax_t(v["draft"][0, 0], T)
    alpha = theory.acceptance_rate(p, q)
    rng = np.random.default_rng(10)
    N = 20000
    acc = 0
    for _ in range(N):
        x = oracle.inverse_cdf(q, rng.random())
        _, n = oracle.verify_sampling(v["target"][0], v["draft"][0], [x],
                                      [rng.random(), rng.random()], T)
        acc += n
    sd = np.sqrt(alpha * (1 - alpha) / N)
    assert abs(acc / N - alpha) < 4 * sd


def test_batch_padding_and_counts():
    v = synth.verify_logits(11, B=4, gamma=3, V=50, kind="zipf")
    x = np.argmax(v["draft"], axis=2)
    out, n = oracle.verify_batch(v["target"], v["draft"], x, v["u_verify"], 0.8)
    for b in range(4):
        assert np.all(out[b, : n[b] + 1] >= 0)
        assert np.all(out[b, n[b] + 1:] == -1)


# ----------------------------------------------- draft side from the head
def test_lowrank_verify_reads_draft_rows_through_w_up():
    """z rows that are unit vectors pick columns of W_up: the draft rows the
    low-rank form sees are exactly those columns, so it must agree with the
    plain verifier on those rows (a transposed or mis-indexed W_up fails)."""
    rng = np.random.default_rng(21)
    B, g, V, r, T = 5, 3, 40, 8, 0.8
    target = rng.standard_normal((B, g + 1, V))
    w_up = rng.standard_normal((V, r))
    cols = rng.integers(0, r, (B, g))
    z = np.zeros((B, g, r))
    for b in range(B):
        for j in range(g):
            z[b, j, cols[b, j]] = 1.0
    draft = np.stack([[w_up[:, cols[b, j]] for j in range(g)] for b in range(B)])
    x = rng.integers(0, V, (B, g))
    u = synth.uniforms(rng, (B, g + 1))
    got = oracle.verify_lowrank_batch(target, z, w_up, x, u, T)
    want = oracle.verify_batch(target, draft, x, u, T)
    np.testing.assert_array_equal(got[0], want[0])
    np.testing.assert_array_equal(got[1], want[1])
    # scaling z scales the draft logits: at T the same as z / 2 at T / 2
    got2 = oracle.verify_lowrank_batch(target * 0.5, z * 0.5, w_up, x, u, T * 0.5)
    np.testing.assert_array_equal(got2[0], want[0])


def test_lowrank_verify_draft_distribution_from_z():
    """With W_up = I (r = V) and z = log q, the draft distributions the
    low-rank form builds are q itself, at any temperature T applied to
    z = T log q; its outcomes then match the plain verifier on log q rows."""
    rng = np.random.default_rng(5)
    B, g, V = 4, 2, 6
    q = rng.dirichlet(np.ones(V), size=(B, g))
    target = rng.standard_normal((B, g + 1, V))
    x = rng.integers(0, V, (B, g))
    u = synth.uniforms(rng, (B, g + 1))
    w_up = np.eye(V)
    for T in (0.5, 1.0, 2.0):
        z = T * np.log(q)
        for b in range(B):
            for j in range(g):
                qb = oracle.softmax_t(oracle.up_projection(z[b, j][None, :], w_up)[0], T)
                np.testing.assert_allclose(qb, q[b, j], rtol=1e-12)
        got = oracle.verify_lowrank_batch(target, z, w_up, x, u, T)
        want = oracle.verify_batch(target, z, x, u, T)
        np.testing.assert_array_equal(got[0], want[0])
        np.testing.assert_array_equal(got[1], want[1])
