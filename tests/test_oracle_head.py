"""Pins for the oracle's bf16 rounding, low-rank head and row reduction.

Each check compares the oracle with something other than itself: exact
rational brute force, a library routine, a closed form or an invariant.
"""
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import synth


# ---------------------------------------------------------------- bf16 ------
def test_bf16_ties_to_even():
    u = 2.0 ** -7            # bf16 spacing just above 1.0
    x = np.array([1 + u / 2, 1 + 3 * u / 2, -(1 + u / 2), 1 + u / 2 + 2.0 ** -40,
                  1.0, 2.0 ** -126, 0.0])
    want = np.array([1.0, 1 + 2 * u, -1.0, 1 + u, 1.0, 2.0 ** -126, 0.0])
    np.testing.assert_array_equal(oracle.round_to_bf16(x), want)


def test_bf16_matches_torch_on_fp32_inputs():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-30, 30, 100000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.round_to_bf16(x.astype(np.float64)), ref)


def test_bf16_single_rounding_from_f64():
    # 1 + 2**-8 + 2**-30 is above the midpoint; a detour through fp32 would
    # first drop the 2**-30 and then tie to even (1.0).
    x = 1 + 2.0 ** -8 + 2.0 ** -30
    assert oracle.round_to_bf16(np.array([x]))[0] == 1 + 2.0 ** -7


def test_synth_bf16_matches_torch():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(50000).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(synth.round_f32_to_bf16(x), ref)


# ---------------------------------------------------------------- head ------
def _frac_matmul_t(a, b):
    """a (m, k) times b (n, k) transposed, in exact rationals."""
    return [[sum(Fraction(a[i][t]) * Fraction(b[j][t]) for t in range(len(a[i])))
             for j in range(len(b))] for i in range(len(a))]


def test_head_brute_force_exact():
    """Two-step projection against exact rational triple loops (tiny shapes)."""
    rng = np.random.default_rng(2)
    M, d, r, V = 2, 5, 3, 7
    h = rng.integers(-4, 5, (M, d)) / 4.0
    wd = rng.integers(-4, 5, (r, d)) / 8.0
    wu = rng.integers(-4, 5, (V, r)) / 16.0
    z = _frac_matmul_t(h.tolist(), wd.tolist())
    logits = _frac_matmul_t(z, wu.tolist())
    got = oracle.slimspec_head(h, wd, wu, "f32", 0.0)
    np.testing.assert_array_equal(got["z"], np.array(z, dtype=np.float64))
    np.testing.assert_array_equal(got["logits"], np.array(logits, dtype=np.float64))


def test_head_bf16_intermediate_rounding_exact():
    """z lands exactly on bf16 midpoints: the oracle must round them to even."""
    u = 2.0 ** -7
    h = np.array([[1.0, u / 2]])               # z_j = w_j0 + (u/2) w_j1
    wd = np.array([[1.0, 1.0], [1.0 + u, 1.0], [1.0, 3.0]])
    got = oracle.down_projection(h, wd, "bf16")
    # 1 + u/2 -> 1 (even); 1 + u + u/2 -> 1 + 2u (even); 1 + 3u/2 -> 1 + 2u
    np.testing.assert_array_equal(got, [[1.0, 1 + 2 * u, 1 + 2 * u]])


def test_low_rank_equals_dense():
    """Low-rank = dense: with W = W_up W_down, the unrounded low-rank head
    equals the dense head h W^T (fp64, relative 1e-12)."""
    inp = synth.head_inputs(3, M=3, d=96, r=16, V=777, dtype="f32")
    lr = oracle.slimspec_head(inp["hidden"], inp["w_down"], inp["w_up"], "f32", 0.0)
    W = inp["w_up"].astype(np.float64) @ inp["w_down"].astype(np.float64)
    dense = oracle.dense_head(inp["hidden"], W, 0.0)
    scale = np.max(np.abs(dense["logits"]))
    assert np.max(np.abs(lr["logits"] - dense["logits"])) <= 1e-12 * scale
    np.testing.assert_array_equal(lr["tokens"], dense["tokens"])


def test_identity_down_projection_is_plain_head():
    """Special case r = d, W_down = I: logits reduce to h W_up^T, which the
    dense head computes independently."""
    inp = synth.head_inputs(4, M=2, d=32, r=32, V=300, dtype="f32")
    I = np.eye(32)
    lr = oracle.slimspec_head(inp["hidden"], I, inp["w_up"], "f32", 0.0)
    dn = oracle.dense_head(inp["hidden"], inp["w_up"], 0.0)
    np.testing.assert_array_equal(lr["logits"], dn["logits"])


# ------------------------------------------------------------ reduction -----
def test_greedy_lowest_index_tie():
    l = np.array([0.5, 2.0, -1.0, 2.0, 2.0])
    assert oracle.row_reduce(l, 0.0)["token"] == 1
    l2 = np.random.default_rng(5).standard_normal(1000)
    assert oracle.row_reduce(l2, 0.0)["token"] == int(np.argmax(l2))


@pytest.mark.parametrize("T", [0.7, 1.0, 2.5])
def test_lse_logprob_match_scipy(T):
    l = np.random.default_rng(6).standard_normal(5000) * 3
    res = oracle.row_reduce(l, T, 0.37)
    assert abs(res["lse"] - scipy.special.logsumexp(l / T)) < 1e-10
    assert abs(res["logprob"] - scipy.special.log_softmax(l / T)[res["token"]]) < 1e-10
    assert res["max"] == l.max()


def test_inverse_cdf_exact_boundaries():
    w = [Fraction(1, 8), Fraction(0), Fraction(3, 8), Fraction(1, 4), Fraction(1, 4)]
    W = sum(w)
    cum = np.cumsum(np.array(w, dtype=object))
    for v in range(len(w)):
        lo = cum[v] - w[v]
        if w[v] > 0:
            assert oracle.inverse_cdf(np.array(w, dtype=object), (lo + cum[v]) / 2 / W) == v
            # a uniform exactly on a left boundary belongs to that token
            assert oracle.inverse_cdf(np.array(w, dtype=object), lo / W) == v
    # u * W equal to the last partial sum (impossible for u < 1) falls back to
    # the last positive weight
    assert oracle.inverse_cdf(np.array(w + [Fraction(0)], dtype=object), Fraction(1)) == 4


def test_inverse_cdf_frequencies_on_a_grid():
    """A uniform grid of N points reproduces softmax frequencies to 1/N."""
    l = np.array([0.3, -1.2, 2.0, 0.0, 1.1, -0.4])
    T = 0.8
    N = 20000
    counts = np.zeros(len(l))
    for i in range(N):
        counts[oracle.row_reduce(l, T, (i + 0.5) / N)["token"]] += 1
    np.testing.assert_allclose(counts / N, scipy.special.softmax(l / T), atol=1.0 / N + 1e-12)


def test_sampling_tends_to_argmax_as_t_to_zero():
    l = np.array([0.1, 3.0, 1.0, 2.9, -2.0])
    for u in np.linspace(0, 0.999, 50):
        assert oracle.row_reduce(l, 1e-3, u)["token"] == 1


# ----------------------------------------------------- static trimmed head ---
def test_trimmed_head_keeping_everything_is_the_dense_head():
    """Every row kept in vocabulary order: the dense head itself."""
    rng = np.random.default_rng(3)
    M, d, V = 4, 16, 50
    h = rng.standard_normal((M, d))
    W = rng.standard_normal((V, d))
    u = rng.random(M)
    for T in (0.0, 0.7):
        got = oracle.trimmed_head(h, W, np.arange(V), T, u if T > 0 else None)
        want = oracle.dense_head(h, W, T, u if T > 0 else None)
        np.testing.assert_array_equal(got["tokens"], want["tokens"])
        np.testing.assert_allclose(got["lse"], want["lse"], rtol=1e-14)


def test_trimmed_head_brute_force_over_the_kept_set():
    """Small integer heads: the greedy token is, by exhaustive search over the
    kept ids in kept order, the first kept id with the largest score; the
    sampled token's cumulative weights straddle u (exact fractions); tokens
    outside the kept set never appear, even when they hold the full head's
    maximum."""
    rng = np.random.default_rng(8)
    M, d, V = 6, 5, 30
    h = rng.integers(-3, 4, (M, d)).astype(np.float64)
    W = rng.integers(-3, 4, (V, d)).astype(np.float64)
    full = h @ W.T
    kept = np.array(sorted(rng.choice(V, 12, replace=False)))
    # for some rows the full head's best id is a dropped one
    assert any(int(np.argmax(full[m])) not in set(kept.tolist()) for m in range(M))
    got = oracle.trimmed_head(h, W[kept], kept, 0.0)
    for m in range(M):
        best_v, best_s = None, None
        for i, v in enumerate(kept):
            s = sum(int(h[m, k]) * int(W[v, k]) for k in range(d))
            if best_s is None or s > best_s:
                best_v, best_s = int(v), s
        assert got["tokens"][m] == best_v
        assert got["tokens"][m] in set(kept.tolist())
    # sampling at T = 1 with rational weights 2^(score) on the kept set
    u = np.array([Fraction(k, 7) for k in range(M)], dtype=object)
    got = oracle.trimmed_head(h, W[kept], kept, 1.0, [float(x) for x in u])
    for m in range(M):
        s = [sum(int(h[m, k]) * int(W[v, k]) for k in range(d)) for v in kept]
        mx = max(s)
        w = [np.exp(si - mx) for si in s]
        cum = np.cumsum(w) / np.sum(w)
        i = int(np.nonzero(kept == got["tokens"][m])[0][0])
        lo = cum[i - 1] if i > 0 else 0.0
        assert lo - 1e-12 <= float(u[m]) < cum[i] + 1e-12


def test_trimmed_head_kept_order_decides_ties():
    """Two kept rows with equal scores: the one earlier in the kept order wins,
    whatever their vocabulary ids."""
    h = np.array([[1.0, 0.0]])
    W = np.array([[2.0, 0.0], [2.0, 0.0], [1.0, 0.0]])   # kept rows, in kept order
    got = oracle.trimmed_head(h, W, np.array([40, 7, 3]), 0.0)
    assert got["tokens"][0] == 40
    got = oracle.trimmed_head(h, W[[1, 0, 2]], np.array([7, 40, 3]), 0.0)
    assert got["tokens"][0] == 7
