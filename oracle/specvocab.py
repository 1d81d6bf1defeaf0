"""Oracle for the SpecVocab-style dynamic-vocabulary head.

Test infrastructure only (see the package docstring).

SpecVocab write-up, sections 2.2.1-2.2.3: a small router first scores the whole
vocabulary at reduced width (h' = W_down h with d' = d/16, s = W_vocab h'), the
k = 2048 best-scoring ids are kept (k_t = topk(s, k)), and exact logits are
computed for those ids only (z' = U[k_t] h, q = softmax(z')).
"""
from __future__ import annotations

import numpy as np

from .bf16 import round_to_bf16
from .head import row_reduce


def approx_scores(hidden, w_down, w_vocab, dtype: str = "bf16"):
    """h' = W_down h (rounded to bf16 for bf16 workloads) and s = W_vocab h'.

    Section 2.2.1.  hidden (M, d), w_down (d', d), w_vocab (V, d').  Returns
    (h_prime (M, d'), scores (M, V)) in float64.
    """
    hp = np.asarray(hidden, np.float64) @ np.asarray(w_down, np.float64).T
    if dtype == "bf16":
        hp = round_to_bf16(hp)
    s = hp @ np.asarray(w_vocab, np.float64).T
    return hp, s


def topk_lowest_index(scores_row, k: int) -> np.ndarray:
    """The k highest-scoring ids of one row, ties broken toward the lowest id.

    Section 2.2.2 picks k_t = topk(s, k); the articles do not say how ties are
    broken, and the oracle breaks them toward the lower id.  The ids are
    returned in ascending id order (the order the exact stage and its
    inverse-CDF walk them in).
    """
    s = np.asarray(scores_row, np.float64)
    V = s.shape[0]
    if not 0 < k <= V:
        raise ValueError("k out of range")
    ids = np.arange(V)
    # lexsort: last key is primary -> by descending score, then ascending id
    order = np.lexsort((ids, -s))
    return np.sort(order[:k])


def specvocab_head(hidden, w_down, w_vocab, u_full, k: int, temperature: float,
                   u=None, dtype: str = "bf16") -> dict:
    """Router scores, top-k, exact logits over the candidates, then a draw.

    Section 2.2.3: U' = U[k_t, :], z' = U' h, q = softmax(z').  The draw over the
    k candidates follows the same rule as the full head (row_reduce): greedy
    picks the lowest-index maximum, sampling walks the candidates in ascending
    id order with one uniform.
    """
    hidden = np.asarray(hidden, np.float64)
    hp, s = approx_scores(hidden, w_down, w_vocab, dtype)
    M = hidden.shape[0]
    cand = np.zeros((M, k), np.int64)
    zc = np.zeros((M, k))
    q = np.zeros((M, k))
    tokens = np.zeros(M, np.int64)
    for i in range(M):
        cand[i] = topk_lowest_index(s[i], k)
        zc[i] = np.asarray(u_full[cand[i]], np.float64) @ hidden[i]
        red = row_reduce(zc[i], temperature, None if u is None else u[i])
        tokens[i] = cand[i][red["token"]]
        if temperature > 0:
            w = np.exp((zc[i] - red["max"]) / temperature)
            q[i] = w / w.sum()
        else:
            q[i] = (np.arange(k) == red["token"]).astype(np.float64)
    return {"h_prime": hp, "scores": s, "candidates": cand, "cand_logits": zc,
            "q": q, "tokens": tokens}
