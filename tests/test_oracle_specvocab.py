"""Pins for the oracle's SpecVocab path (router scores, top-k, exact stage)."""
import numpy as np
import scipy.special

import oracle
import synth


def test_topk_matches_stable_argsort_with_ties():
    rng = np.random.default_rng(0)
    s = rng.integers(0, 40, 5000).astype(np.float64)   # many exact ties
    for k in (1, 7, 100, 2048, 5000):
        want = np.sort(np.argsort(-s, kind="stable")[:k])
        np.testing.assert_array_equal(oracle.topk_lowest_index(s, k), want)


def test_topk_definition_brute_force():
    """Every kept id scores >= every dropped id; among ids tied with the
    threshold, the kept ones are the lowest."""
    rng = np.random.default_rng(1)
    for trial in range(50):
        V = int(rng.integers(2, 40))
        k = int(rng.integers(1, V + 1))
        s = rng.integers(0, 5, V).astype(np.float64)
        kept = set(oracle.topk_lowest_index(s, k).tolist())
        assert len(kept) == k
        dropped = [v for v in range(V) if v not in kept]
        if dropped:
            assert min(s[v] for v in kept) >= max(s[v] for v in dropped)
            thr = min(s[v] for v in kept)
            tied_kept = [v for v in kept if s[v] == thr]
            tied_dropped = [v for v in dropped if s[v] == thr]
            if tied_dropped:
                assert max(tied_kept) < min(tied_dropped)


def test_full_candidate_set_is_dense_softmax():
    """With k = V the exact stage is the dense head: q = softmax(U h / T)."""
    inp = synth.specvocab_inputs(2, M=2, d=64, d_prime=8, V=200)
    T = 0.9
    u = np.array([0.25, 0.75])
    out = oracle.specvocab_head(inp["hidden"], inp["w_down"], inp["w_vocab"],
                                inp["u_full"], 200, T, u)
    dense = inp["hidden"].astype(np.float64) @ inp["u_full"].astype(np.float64).T
    for i in range(2):
        np.testing.assert_array_equal(out["candidates"][i], np.arange(200))
        np.testing.assert_allclose(out["q"][i], scipy.special.softmax(dense[i] / T), rtol=1e-12)
        assert out["tokens"][i] == oracle.row_reduce(dense[i], T, u[i])["token"]


def test_router_scores_brute_force():
    """s = W_vocab h' with h' = bf16(W_down h): exact rationals on small ints."""
    from fractions import Fraction
    rng = np.random.default_rng(3)
    h = rng.integers(-3, 4, (1, 6)) / 2.0
    wd = rng.integers(-3, 4, (2, 6)) / 4.0
    wv = rng.integers(-3, 4, (5, 2)) / 8.0
    hp, s = oracle.approx_scores(h, wd, wv, "f32")
    for j in range(2):
        assert hp[0, j] == float(sum(Fraction(h[0, t]) * Fraction(wd[j, t]) for t in range(6)))
    for v in range(5):
        assert s[0, v] == float(sum(Fraction(hp[0, j]) * Fraction(wv[v, j]) for j in range(2)))


def test_router_hprime_is_rounded_to_bf16():
    """Hand-worked: h = (1, 1), W_down = (1, 2^-9) makes the exact h' = 1 + 2^-9,
    a quarter of the bf16 spacing above 1 (2^-7), so bf16 h' is exactly 1 and
    the score through W_vocab = 3 is 3; the fp32 workload keeps 3 + 3 * 2^-9."""
    h = np.array([[1.0, 1.0]])
    wd = np.array([[1.0, 2.0 ** -9]])
    wv = np.array([[3.0]])
    hp, s = oracle.approx_scores(h, wd, wv, "bf16")
    assert hp[0, 0] == 1.0 and s[0, 0] == 3.0
    hp, s = oracle.approx_scores(h, wd, wv, "f32")
    assert hp[0, 0] == 1.0 + 2.0 ** -9 and s[0, 0] == 3.0 + 3.0 * 2.0 ** -9


def test_greedy_specvocab_token_is_candidate_argmax():
    inp = synth.specvocab_inputs(4, M=3, d=128, d_prime=8, V=1000)
    out = oracle.specvocab_head(inp["hidden"], inp["w_down"], inp["w_vocab"],
                                inp["u_full"], 64, 0.0)
    for i in range(3):
        c = out["candidates"][i]
        assert out["tokens"][i] == c[int(np.argmax(out["cand_logits"][i]))]
        assert np.all(np.diff(c) > 0)
