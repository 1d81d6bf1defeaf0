"""Oracle for the verification step of speculative decoding.

Test infrastructure only (see the package docstring).

Explainer, sections "小模型起草，大模型批改" and "为什么答案不会变": the target's
gamma+1 next-token judgements are compared with the gamma drafted tokens from
left to right.  Greedy: a drafted token stays while it equals the target's
choice; the first mismatch is replaced by the target's token and the rest is
dropped; if all gamma match, the target's judgement at position gamma is added.
Sampling: drafted token x is kept with probability min(1, p(x)/q(x)); at the
first rejection a token is drawn from the positive part of p - q,
renormalised; SpecTr-GBV article (第三步) and the explainer: when every drafted
token is kept, one more token is drawn from the target at the next position.
"""
from __future__ import annotations

import numpy as np

from .head import inverse_cdf, up_projection


def softmax_t(logits_row, temperature: float) -> np.ndarray:
    """softmax(l / T) in float64 (T > 0)."""
    l = np.asarray(logits_row, np.float64)
    w = np.exp((l - np.max(l)) / float(temperature))
    return w / np.sum(w)


def verify_greedy(target_rows, draft_tokens):
    """Greedy verification of one sequence.

    target_rows (gamma+1, V); draft_tokens (gamma,).  a_j is the lowest-index
    argmax of target row j.  n = the first j with x_j != a_j, else gamma.
    Emitted tokens: x_0 .. x_{n-1}, a_n.  Returns (tokens, n).
    """
    t = np.asarray(target_rows, np.float64)
    gamma = len(draft_tokens)
    a = [int(np.nonzero(t[j] == np.max(t[j]))[0][0]) for j in range(gamma + 1)]
    n = gamma
    for j in range(gamma):
        if int(draft_tokens[j]) != a[j]:
            n = j
            break
    return [int(x) for x in draft_tokens[:n]] + [a[n]], n


def verify_decide(p_rows, q_rows, draft_tokens, u):
    """The accept / reject / resample decisions for one sequence.

    p_rows: gamma+1 target distributions; q_rows: gamma draft distributions
    (any numeric type with +, -, * and comparisons, e.g. float64 arrays or
    object arrays of Fractions).  u: gamma+1 uniforms in [0, 1).
    Position j < gamma keeps x_j iff u_j * q_j(x_j) < p_j(x_j), which is
    "u_j < min(1, p/q)" without a division.  At the first rejection n the
    token is inverse_cdf(max(0, p_n - q_n), u_gamma); if that residual is all
    zero, inverse_cdf(p_n, u_gamma).  If all gamma are kept the bonus token is
    inverse_cdf(p_gamma, u_gamma).  Returns (tokens, n).
    """
    gamma = len(draft_tokens)
    for j in range(gamma):
        x = int(draft_tokens[j])
        if not (u[j] * q_rows[j][x] < p_rows[j][x]):
            p = np.asarray(p_rows[j])
            q = np.asarray(q_rows[j])
            diff = p - q
            resid = np.where(diff > 0, diff, diff * 0)
            if not np.any(resid > 0):
                resid = p
            tok = inverse_cdf(resid, u[gamma])
            return [int(v) for v in draft_tokens[:j]] + [tok], j
    tok = inverse_cdf(np.asarray(p_rows[gamma]), u[gamma])
    return [int(v) for v in draft_tokens] + [tok], gamma


def verify_sampling(target_rows, draft_rows, draft_tokens, u, temperature):
    """Sampling verification of one sequence from logits: p = softmax(target/T),
    q = softmax(draft/T), then verify_decide."""
    gamma = len(draft_tokens)
    p = [softmax_t(target_rows[j], temperature) for j in range(gamma + 1)]
    q = [softmax_t(draft_rows[j], temperature) for j in range(gamma)]
    return verify_decide(p, q, draft_tokens, u)


def verify_batch(target, draft, draft_tokens, u, temperature: float):
    """Batched form.  target (B, gamma+1, V); draft (B, gamma, V) or None when
    temperature == 0; draft_tokens (B, gamma); u (B, gamma+1) or None.

    Returns out_tokens (B, gamma+1) int64 padded with -1 after the n+1 emitted
    tokens, and num_accepted (B,).
    """
    B, g1, _ = target.shape
    out = np.full((B, g1), -1, np.int64)
    nacc = np.zeros(B, np.int64)
    for b in range(B):
        if temperature == 0.0:
            toks, n = verify_greedy(target[b], draft_tokens[b])
        else:
            toks, n = verify_sampling(target[b], draft[b], draft_tokens[b], u[b],
                                      temperature)
        out[b, :len(toks)] = toks
        nacc[b] = n
    return out, nacc


def verify_lowrank_batch(target, z, w_up, draft_tokens, u, temperature: float):
    """Sampling verification when the draft distributions come from the
    low-rank drafter head itself (SlimSpec article, section 三: the drafter's
    scores are z W_up^T over the full vocabulary; explainer, section
    "为什么答案不会变": the accept test and the residual need q at each
    position).  z (B, gamma, r) holds the drafter's intermediate rows (the
    bf16-rounded values the head multiplied), w_up (V, r).  The draft rows are
    q_j = softmax(z_j W_up^T / T); everything else is verify_batch.
    """
    B, g, _ = z.shape
    draft = np.stack([up_projection(z[b], w_up) for b in range(B)])
    return verify_batch(target, draft, draft_tokens, u, temperature)
