"""Comparison rules between the CUDA path and the CPU oracle.

The GPU accumulates in fp32, the oracle in fp64, so a decision taken from
floating point can legitimately differ when the inputs sit on a decision
boundary.  The rules (token ids are otherwise bit-exact):

* greedy: the GPU token must equal the oracle's lowest-index argmax, unless
  the oracle's top two logits lie within ``eps`` of each other; then it must be
  one of the tokens within ``eps`` of the maximum ("tie").
* inverse-CDF draw with uniform u over weights w: with C the oracle's
  normalised ascending partial sums, the GPU token v must satisfy
  C(v-1) - 1e-5 <= u < C(v) + 1e-5; it is "exact" when it equals the oracle's
  token and "boundary" otherwise.
* accept test u * q(x) < p(x): a differing decision is allowed only when
  |u - p(x)/q(x)| < 1e-5.
"""
from __future__ import annotations

import numpy as np

import oracle

WINDOW = 1e-5


def greedy_verdict(tok: int, logits_row, eps: float):
    l = np.asarray(logits_row, np.float64)
    m = l.max()
    ref = int(np.nonzero(l == m)[0][0])
    if tok == ref:
        return "exact"
    if 0 <= tok < l.size and l[tok] >= m - eps:
        return "tie"
    return None


def cdf_verdict(tok: int, weights, u: float, ref_tok: int | None = None):
    w = np.asarray(weights, np.float64)
    if not 0 <= tok < w.size:
        return None
    C = np.cumsum(w) / w.sum()
    lo = C[tok - 1] if tok > 0 else 0.0
    hi = C[tok]
    if not (lo - WINDOW <= u < hi + WINDOW):
        return None
    if ref_tok is None:
        ref_tok = oracle.inverse_cdf(w, u)
    return "exact" if tok == ref_tok else "boundary"


def softmax_weights(logits_row, T: float):
    l = np.asarray(logits_row, np.float64)
    return np.exp((l - l.max()) / T)


def check_head_tokens(tokens, logits, T, u, eps_greedy):
    """Returns counts {'exact','tie','boundary'}; raises on an invalid token."""
    counts = {"exact": 0, "tie": 0, "boundary": 0}
    for m, tok in enumerate(tokens):
        if T == 0:
            v = greedy_verdict(int(tok), logits[m], eps_greedy)
        else:
            v = cdf_verdict(int(tok), softmax_weights(logits[m], T), float(u[m]))
        assert v is not None, f"row {m}: token {tok} is not a valid draw"
        counts[v] += 1
    return counts


def check_verify_sampling(toks, n, target_rows, draft_rows, x, u, T):
    """Validity of one sequence's sampling verification outcome from the GPU.

    Returns 'exact' or 'boundary'; raises AssertionError if invalid."""
    gamma = len(x)
    ref_toks, ref_n = oracle.verify_sampling(target_rows, draft_rows, x, u, T)
    p = [oracle.softmax_t(target_rows[j], T) for j in range(gamma + 1)]
    q = [oracle.softmax_t(draft_rows[j], T) for j in range(gamma)]
    boundary = False
    # accept decisions up to the GPU's stopping point
    for j in range(min(n + 1, gamma)):
        xj = int(x[j])
        acc_ref = u[j] * q[j][xj] < p[j][xj]
        acc_gpu = j < n
        if acc_ref != acc_gpu:
            assert abs(u[j] - p[j][xj] / q[j][xj]) < WINDOW, f"accept decision at {j} differs"
            boundary = True
    assert list(toks[:n]) == [int(v) for v in x[:n]]
    # the final draw, from the distribution the GPU's n implies
    if n < gamma:
        w = np.maximum(p[n] - q[n], 0.0)
        if not np.any(w > 0):
            w = p[n]
    else:
        w = p[gamma]
    v = cdf_verdict(int(toks[n]), w, float(u[gamma]))
    assert v is not None, f"final token {toks[n]} invalid"
    if boundary or v == "boundary" or n != ref_n or list(toks[: n + 1]) != list(ref_toks):
        return "boundary"
    return "exact"
