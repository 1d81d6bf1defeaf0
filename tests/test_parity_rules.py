"""The GPU-versus-oracle comparison rules (tests/parity.py) reject wrong
results: each rule is run on the oracle's own answer, on an answer inside its
stated tolerance, and on a wrong one, on the CPU."""
import numpy as np
import pytest

import oracle
import synth
from parity import (WINDOW, cdf_verdict, check_head_tokens, check_verify_sampling,
                    greedy_verdict, softmax_weights)


def test_greedy_verdict():
    row = np.array([0.0, 3.0, 3.0 - 1e-4, 1.0, 3.0])
    assert greedy_verdict(1, row, 1e-3) == "exact"      # lowest index of the maximum
    assert greedy_verdict(4, row, 1e-3) == "tie"        # the same maximum, later index
    assert greedy_verdict(2, row, 1e-3) == "tie"        # within eps of the maximum
    assert greedy_verdict(2, row, 1e-5) is None         # outside a tighter eps
    assert greedy_verdict(3, row, 1e-3) is None
    assert greedy_verdict(5, row, 1e-3) is None         # out of range


def test_cdf_verdict():
    w = np.array([1.0, 2.0, 0.0, 1.0])                  # C = 0.25, 0.75, 0.75, 1.0
    assert cdf_verdict(1, w, 0.5) == "exact"
    assert cdf_verdict(0, w, 0.5) is None
    assert cdf_verdict(3, w, 0.5) is None
    assert cdf_verdict(4, w, 0.5) is None               # out of range
    # u just below a boundary: the neighbour across it is allowed, as "boundary"
    assert cdf_verdict(1, w, 0.25 - WINDOW / 2) == "boundary"
    assert cdf_verdict(1, w, 0.25 - 2 * WINDOW) is None


def test_check_head_tokens_rejects_a_wrong_draw():
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((6, 50))
    u = synth.uniforms(rng, (6,))
    toks = np.array([oracle.row_reduce(logits[m], 1.0, u[m])["token"] for m in range(6)])
    assert check_head_tokens(toks, logits, 1.0, u, 1e-3)["exact"] == 6
    bad = toks.copy()
    w = softmax_weights(logits[2], 1.0)
    C = np.cumsum(w) / w.sum()
    # a token whose CDF interval is far from u[2]
    far = int(np.argmax(np.abs((C - w / w.sum() / 2) - u[2])))
    bad[2] = far
    with pytest.raises(AssertionError):
        check_head_tokens(bad, logits, 1.0, u, 1e-3)
    greedy = np.argmax(logits, axis=1)
    assert check_head_tokens(greedy, logits, 0.0, None, 1e-3)["exact"] == 6
    with pytest.raises(AssertionError):
        check_head_tokens((greedy + 1) % 50, logits, 0.0, None, 1e-3)


def test_check_verify_sampling_rejects_wrong_outcomes():
    v = synth.verify_logits(9, B=8, gamma=4, V=64, kind="normal", draft_sigma=0.5)
    T = 1.0
    checked = 0
    for b in range(8):
        x = np.array([oracle.row_reduce(v["draft"][b, j], T, v["u_draft"][b, j])["token"]
                      for j in range(4)])
        toks, n = oracle.verify_sampling(v["target"][b], v["draft"][b], x, v["u_verify"][b], T)
        full = np.full(5, -1)
        full[:n + 1] = toks
        assert check_verify_sampling(full, n, v["target"][b], v["draft"][b], x,
                                     v["u_verify"][b], T) == "exact"
        # one more accepted token than the oracle's, where the test clearly rejects
        if n < 4:
            p = oracle.softmax_t(v["target"][b, n], T)
            q = oracle.softmax_t(v["draft"][b, n], T)
            if abs(v["u_verify"][b, n] - p[x[n]] / q[x[n]]) > 10 * WINDOW:
                wrong = full.copy()
                wrong[n] = x[n]
                with pytest.raises(AssertionError):
                    check_verify_sampling(wrong, n + 1, v["target"][b], v["draft"][b], x,
                                          v["u_verify"][b], T)
                checked += 1
        # a final token outside its CDF interval
        wrong = full.copy()
        wrong[n] = -5
        with pytest.raises(AssertionError):
            check_verify_sampling(wrong, n, v["target"][b], v["draft"][b], x,
                                  v["u_verify"][b], T)
    assert checked > 0
