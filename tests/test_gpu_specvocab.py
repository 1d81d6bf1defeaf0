"""GPU parity of the SpecVocab head and its top-k stage against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
import speculative_decoding_drafter_slimspec_gb300 as ss
from parity import cdf_verdict, greedy_verdict
from gpu_util import device, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("k", [1, 100, 2048, 20000])
def test_topk_ties_bit_exact(k):
    """Integer-valued scores (thousands of exact ties, -0.0 next to +0.0): the
    kept set and its ascending order are bit-exact."""
    rng = np.random.default_rng(k)
    M, V = 6, 20000
    s = rng.integers(-50, 50, (M, V)).astype(np.float32)
    s[0, ::7] = -0.0
    s[1] = 0.0
    got = ss.ss_topk_rows(to_dev(s, "f32"), k)
    torch.cuda.synchronize()
    g = got.cpu().numpy()
    for m in range(M):
        np.testing.assert_array_equal(g[m], oracle.topk_lowest_index(s[m], k))


def test_topk_continuous_scores():
    rng = np.random.default_rng(1)
    M, V, k = 4, 151936, 2048
    s = rng.standard_normal((M, V)).astype(np.float32)
    g = ss.ss_topk_rows(to_dev(s, "f32"), k).cpu().numpy()
    for m in range(M):
        np.testing.assert_array_equal(g[m], oracle.topk_lowest_index(s[m], k))


@pytest.mark.parametrize("M", [1, 32, 40])
def test_topk_cluster_shapes(M):
    """Rows split over clusters of 8, 4 and 2 CTAs (the cluster size follows
    the row count); candidates of every CTA meet in one ordered buffer."""
    rng = np.random.default_rng(100 + M)
    V, k = 151936, 2048
    s = rng.standard_normal((M, V)).astype(np.float32)
    s[:, ::1000] += 3.0   # a spread of large scores across every CTA's range
    g = ss.ss_topk_rows(to_dev(s, "f32"), k).cpu().numpy()
    for m in range(M):
        np.testing.assert_array_equal(g[m], oracle.topk_lowest_index(s[m], k))


def test_topk_skewed_rows_fall_back():
    """The largest scores packed into the first ids of a row (one warp's
    region overflows), at the end of a row, and a row of exact ties: the
    whole-row selection gives the same ids."""
    rng = np.random.default_rng(7)
    M, V, k = 3, 151936, 2048
    s = rng.standard_normal((M, V)).astype(np.float32)
    s[0, :3000] += 10.0
    s[1, -2500:] += 10.0
    s[2] = 1.0
    g = ss.ss_topk_rows(to_dev(s, "f32"), k).cpu().numpy()
    for m in range(M):
        np.testing.assert_array_equal(g[m], oracle.topk_lowest_index(s[m], k))


def _run(seed, M, d, dp, V, k, T):
    """One SpecVocab call against the oracle, stage by stage: the router's
    scores element-wise; the candidate set (ids may swap only inside the
    rounding band of the k-th score); the exact stage's logits z' = U[K] h
    element-wise on every candidate id both sides kept; q over the
    candidates relative to its own size (T > 0) or one-hot at a valid argmax
    (T = 0); the drawn token by the parity rules."""
    inp = synth.specvocab_inputs(seed, M=M, d=d, d_prime=dp, V=V)
    u = synth.uniforms(np.random.default_rng(seed + 1), (M,))
    t = {kk: to_dev(vv, "bf16") for kk, vv in inp.items()}
    out = ss.specvocab_head_forward(t["hidden"], t["w_down"], t["w_vocab"], t["u_full"], k, T,
                                    to_dev(u, "f32") if T > 0 else None, want_prob=True,
                                    want_logits=True, want_scores=True)
    torch.cuda.synchronize()
    assert ss.ss_get_device_error() == ss.SS_OK
    ref = oracle.specvocab_head(inp["hidden"], inp["w_down"], inp["w_vocab"], inp["u_full"],
                                k, T, u if T > 0 else None)
    g = {kk: vv.cpu().numpy() for kk, vv in out.items()}
    assert np.max(np.abs(g["scores"] - ref["scores"])) <= 2e-2
    same_rows = 0
    for m in range(M):
        gid, oid = g["topk_idx"][m], ref["candidates"][m]
        assert np.all(np.diff(gid) > 0)
        # exact logits of every id both sides kept, element by element
        shared, gi, oi = np.intersect1d(gid, oid, assume_unique=True, return_indices=True)
        assert shared.size >= k - 8
        assert np.max(np.abs(g["topk_logits"][m][gi] - ref["cand_logits"][m][oi])) <= 2e-2
        if shared.size != k:
            # only ids whose router score is within the rounding band of the
            # k-th score may swap in or out
            sk = np.sort(ref["scores"][m])[::-1][k - 1]
            band = 1e-3 * (1 + abs(sk))
            for vid in np.setxor1d(gid, oid):
                assert abs(ref["scores"][m][vid] - sk) <= band
            continue
        same_rows += 1
        # q over the candidates and the token
        j = int(np.searchsorted(oid, g["tokens"][m]))
        assert oid[j] == g["tokens"][m]
        if T == 0:
            assert greedy_verdict(j, ref["cand_logits"][m], 2e-3) is not None
            np.testing.assert_array_equal(g["topk_prob"][m], np.arange(k) == j)
        else:
            q = ref["q"][m]
            assert np.all(np.abs(g["topk_prob"][m] - q) <= 2e-2 * q + 1e-7)
            w = np.exp((ref["cand_logits"][m] - ref["cand_logits"][m].max()) / T)
            assert cdf_verdict(j, w, float(u[m])) is not None
    assert same_rows >= M - 1
    return same_rows


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_specvocab_small(T):
    _run(21, M=4, d=512, dp=32, V=5000, k=256, T=T)


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_specvocab_qwen8b_shape(T):
    p = synth.PRESETS["specvocab8b"]
    _run(p.seed, M=p.M, d=p.d, dp=p.d_prime, V=p.V, k=p.k, T=T)
