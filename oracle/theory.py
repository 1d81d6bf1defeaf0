"""Closed forms and exact enumeration for one speculative round.

Test infrastructure only (see the package docstring).

* SlimSpec article, section 四: the acceptance rate of a drafted token is the
  sum over the vocabulary of min(target probability, draft probability).
* Explainer, section "这笔账划不划算，看一个数": with acceptance rate alpha at
  every position and gamma drafted tokens, the expected number of tokens a
  round yields has a closed form (Leviathan et al.); the article tabulates it
  at gamma = 4.
* Explainer, section "为什么答案不会变": accept + residual resampling yields
  exactly the target distribution.  ``enumerate_round`` computes the exact
  outcome distribution of ``verify_decide`` so that tests can check this.
"""
from __future__ import annotations

from fractions import Fraction
from itertools import product

import numpy as np

from .verify import verify_decide


def acceptance_rate(p, q):
    """alpha = sum_x min(p(x), q(x)) (section 四)."""
    return sum(min(a, b) for a, b in zip(p, q))


def expected_tokens_equal_alpha(alpha, gamma: int):
    """(1 - alpha**(gamma+1)) / (1 - alpha): expected tokens per round when
    every position has acceptance rate alpha; gamma + 1 when alpha == 1."""
    if alpha == 1:
        return gamma + 1
    return (1 - alpha ** (gamma + 1)) / (1 - alpha)


def expected_tokens(alphas):
    """sum_{j=0}^{gamma} prod_{i<j} alpha_i: position j is reached only when all
    earlier drafted tokens were kept, and each round yields one more token than
    it keeps."""
    total, run = 0, 1
    for a in alphas:
        total += run
        run *= a
    return total + run


def _cdf_breaks(w):
    w = list(w)
    tot = sum(w)
    if tot == 0:
        return []
    out, c = [], 0
    for x in w[:-1]:
        c += x
        out.append(c / tot)
    return out


def enumerate_round(p_rows, q_rows):
    """Exact outcome distribution of one round driven by ``verify_decide``.

    p_rows: gamma+1 target distributions, q_rows: gamma draft distributions,
    as lists of Fractions.  Drafted tokens x_j ~ q_j independently.  For every
    x, each uniform's unit interval is cut at the points where a decision of
    verify_decide can change: u_j (j < gamma) at min(1, p_j(x_j)/q_j(x_j)),
    u_gamma at every cumulative breakpoint of every distribution the final
    draw might use.  verify_decide is evaluated once per cell, at its midpoint,
    and the cell's volume times P(x) is added to that outcome.

    Returns {(tokens tuple, n): probability}.
    """
    gamma = len(q_rows)
    V = len(p_rows[0])
    P = [np.array(r, dtype=object) for r in p_rows]
    Q = [np.array(r, dtype=object) for r in q_rows]
    finals = []
    for j in range(gamma):
        diff = [a - b for a, b in zip(p_rows[j], q_rows[j])]
        res = [d if d > 0 else Fraction(0) for d in diff]
        finals.append(res if any(x > 0 for x in res) else list(p_rows[j]))
    finals.append(list(p_rows[gamma]))
    breaks = set()
    for f in finals:
        breaks.update(_cdf_breaks(f))
    last = [Fraction(0)] + sorted(b for b in breaks if 0 < b < 1) + [Fraction(1)]
    last_cells = [((a + b) / 2, b - a) for a, b in zip(last[:-1], last[1:]) if b > a]

    dist = {}
    for x in product(range(V), repeat=gamma):
        px = Fraction(1)
        for j in range(gamma):
            px *= q_rows[j][x[j]]
        if px == 0:
            continue
        per_u = []
        for j in range(gamma):
            qx, pxj = q_rows[j][x[j]], p_rows[j][x[j]]
            t = min(Fraction(1), pxj / qx)
            cells = [(t / 2, t)]
            if t < 1:
                cells.append(((t + 1) / 2, 1 - t))
            per_u.append(cells)
        for combo in product(*per_u):
            w = px
            us = []
            for mid, vol in combo:
                w *= vol
                us.append(mid)
            for mid, vol in last_cells:
                toks, n = verify_decide(P, Q, list(x), us + [mid])
                key = (tuple(toks), n)
                dist[key] = dist.get(key, Fraction(0)) + w * vol
    return dist
