"""Oracle for the SlimSpec low-rank head and its per-row reduction.

Test infrastructure only (see the package docstring).

SlimSpec article, section 三: the dense head (a V x d matrix, O(V*d)) is
replaced by two factors: W_down takes the d-dimensional hidden state to an
r-dimensional summary and W_up takes that summary to V scores, cost
O(r*d + V*r); every one of the V vocabulary entries keeps its score.
"""
from __future__ import annotations

import numpy as np

from .bf16 import round_to_bf16


def down_projection(hidden, w_down, dtype: str) -> np.ndarray:
    """z = h @ W_down.T in float64 (SlimSpec article, section 三, first factor).

    hidden (M, d) and w_down (r, d) hold exact input values.  For bf16
    workloads z is then rounded to the nearest bf16 (reading: a bf16 model's
    intermediate activation is bf16); for fp32 workloads it is left unrounded.
    """
    z = np.asarray(hidden, np.float64) @ np.asarray(w_down, np.float64).T
    if dtype == "bf16":
        z = round_to_bf16(z)
    elif dtype != "f32":
        raise ValueError(dtype)
    return z


def up_projection(z, w_up) -> np.ndarray:
    """logits = z @ W_up.T over the full vocabulary (section 三, second factor)."""
    return np.asarray(z, np.float64) @ np.asarray(w_up, np.float64).T


def dense_logits(hidden, w) -> np.ndarray:
    """logits = h @ W.T for a full V x d head (section 三, the O(V*d) baseline)."""
    return np.asarray(hidden, np.float64) @ np.asarray(w, np.float64).T


def inverse_cdf(weights, u):
    """Smallest index v with  sum_{v' <= v} w_v'  >  u * sum_v w_v.

    Weights are non-negative and are summed in ascending index order.  If
    rounding leaves no such index (u * W at or above the last partial sum), the
    last index with a positive weight is returned.  Works on float64 arrays and
    on object arrays of fractions.Fraction alike.
    """
    w = np.asarray(weights)
    cum = np.cumsum(w)
    target = u * cum[-1]
    hits = np.nonzero(cum > target)[0]
    if hits.size:
        return int(hits[0])
    positive = np.nonzero(w > 0)[0]
    return int(positive[-1])


def row_reduce(logits_row, temperature: float, u=None) -> dict:
    """Reduce one row of logits to a token and its softmax statistics.

    * greedy (temperature == 0): the token is the lowest index attaining the
      maximum; lse is reported as the maximum and logprob as 0.
    * sampling (temperature > 0): w_v = exp((l_v - m) / T) with m the row
      maximum, W = sum_v w_v; the token is inverse_cdf(w, u);
      lse = m / T + log W = log sum_v exp(l_v / T) and
      logprob = (l_token - m) / T - log W.

    The drafter samples at temperature 0 or 1 in the SlimSpec article's
    experiments (section 六); any T > 0 is accepted here.
    """
    l = np.asarray(logits_row, np.float64)
    m = float(np.max(l))
    if temperature == 0.0:
        token = int(np.nonzero(l == m)[0][0])
        return {"token": token, "max": m, "lse": m, "logprob": 0.0}
    T = float(temperature)
    w = np.exp((l - m) / T)
    W = float(np.sum(w))
    token = inverse_cdf(w, float(u))
    logW = float(np.log(W))
    return {"token": token, "max": m, "lse": m / T + logW,
            "logprob": (float(l[token]) - m) / T - logW}


def _reduce_rows(logits, temperature, u) -> dict:
    rows = [row_reduce(logits[i], temperature, None if u is None else u[i])
            for i in range(logits.shape[0])]
    return {
        "tokens": np.array([r["token"] for r in rows], np.int64),
        "max": np.array([r["max"] for r in rows]),
        "lse": np.array([r["lse"] for r in rows]),
        "logprob": np.array([r["logprob"] for r in rows]),
        "logits": logits,
    }


def slimspec_head(hidden, w_down, w_up, dtype: str, temperature: float,
                  u=None) -> dict:
    """Full low-rank head: z, logits over all V, then the per-row reduction."""
    z = down_projection(hidden, w_down, dtype)
    logits = up_projection(z, w_up)
    out = _reduce_rows(logits, temperature, u)
    out["z"] = z
    return out


def dense_head(hidden, w, temperature: float, u=None) -> dict:
    """The dense V x d head followed by the same reduction (comparison path)."""
    return _reduce_rows(dense_logits(hidden, w), temperature, u)


def trimmed_head(hidden, w_kept, kept_ids, temperature: float, u=None) -> dict:
    """Static vocabulary trimming (SlimSpec article, section 二: FR-Spec and
    VocabTrim keep a fixed subset of the vocabulary and score only it): the
    dense head over the kept rows w_kept (V' x d, the head rows of the kept
    ids, in the kept order), the row reduction over those V' scores, and the
    chosen kept row mapped back to its vocabulary id through kept_ids.  Ties
    and the inverse-CDF order follow the kept order (ascending kept_ids make
    that ascending vocabulary id).  Tokens outside the kept set are never
    drafted.
    """
    out = _reduce_rows(dense_logits(hidden, w_kept), temperature, u)
    out["kept_index"] = out["tokens"].copy()
    out["tokens"] = np.asarray(kept_ids, np.int64)[out["tokens"]]
    return out
