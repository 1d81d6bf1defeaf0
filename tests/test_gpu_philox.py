"""The library's Philox4x32-10 stream on the GPU against the oracle's, and
every sampling call with (seed, offset) in place of caller uniforms.

Both sides implement the generator on their own (CUDA in the library, numpy
integers in oracle/philox.py, pinned there by the published known-answer
vectors); here their outputs must agree bit for bit, and a sampling call
given no uniforms must draw exactly the oracle's uniforms at its (row, slot)
counters: the same outcome as the call given those uniforms explicitly, and a
valid draw by the rules of tests/parity.py against the oracle.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
import speculative_decoding_drafter_slimspec_gb300 as ss
from parity import cdf_verdict, check_head_tokens, check_verify_sampling
from gpu_util import device, to_dev

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _words_to_dev(w):
    """uint32 words -> an int32 device tensor with the same bit patterns."""
    return torch.from_numpy(np.asarray(w, np.uint32).view(np.int32).copy()).to(device())


def _dev_words(t):
    return t.cpu().numpy().view(np.uint32).astype(np.uint64)


def test_known_answers_on_device():
    rows = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        rows.append([int(t, 16) for t in line.split()])
    blocks = np.array([r[:6] for r in rows], np.uint64)
    got = _dev_words(ss.ss_philox4x32_10(_words_to_dev(blocks)))
    np.testing.assert_array_equal(got, np.array([r[6:] for r in rows], np.uint64))


def test_random_blocks_bit_exact():
    rng = np.random.default_rng(1)
    blocks = rng.integers(0, 2 ** 32, (100_000, 6), dtype=np.uint64)
    got = _dev_words(ss.ss_philox4x32_10(_words_to_dev(blocks)))
    np.testing.assert_array_equal(got, oracle.philox4x32_10(blocks[:, :4], blocks[:, 4:]))


@pytest.mark.parametrize("seed,offset", [(2024, 5), (2 ** 64 - 1, 2 ** 63 + 12345),
                                         (0x9E3779B97F4A7C15, 2 ** 32)])
def test_uniforms_match_oracle_on_a_million_counters(seed, offset):
    got = ss.ss_philox_uniforms(seed, offset, 1000, 1000).cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(got, oracle.philox_uniforms(seed, offset, 1000, 1000))


# -------------------------------------------------------------- the heads ---
HEADS = [
    # seed, M, d, r, V, dtype, T       path
    (11, 1, 256, 32, 4096, "f32", 1.0),   # the oracle-scale workload, CUDA-core stream
    (13, 9, 128, 128, 3001, "f32", 0.7),  # two m-tiles of the stream
    (16, 8, 1024, 512, 4133, "bf16", 1.0),  # tensor cores, ragged last tile
    (21, 130, 256, 128, 1100, "bf16", 1.0),  # two M tiles of z: rows past 128
]


@pytest.mark.parametrize("case", HEADS, ids=lambda c: f"M{c[1]}-r{c[3]}-V{c[4]}-{c[5]}")
def test_head_draws_from_seed_and_offset(case):
    s, M, d, r, V, dtype, T = case
    inp = synth.head_inputs(s, M=M, d=d, r=r, V=V, dtype=dtype)
    t = {k: to_dev(v, dtype) for k, v in inp.items()}
    seed, offset = 1000 + s, 7 * s
    a = ss.slimspec_head_forward(t["hidden"], t["w_down"], t["w_up"], T, None, seed=seed,
                                 offset=offset)
    u_dev = ss.ss_philox_uniforms(seed, offset, M, 1).reshape(M).contiguous()
    b = ss.slimspec_head_forward(t["hidden"], t["w_down"], t["w_up"], T, u_dev)
    torch.cuda.synchronize()
    assert ss.ss_get_device_error() == ss.SS_OK
    for k in a:
        assert torch.equal(a[k], b[k]), k
    u = oracle.philox_uniforms(seed, offset, M, 1)[:, 0]
    ref = oracle.slimspec_head(inp["hidden"], inp["w_down"], inp["w_up"], dtype, T, u)
    counts = check_head_tokens(a["tokens"].cpu().numpy(), ref["logits"], T, u, 0.0)
    assert counts["exact"] >= M - 1


def test_head_gptoss20b_shape_seed_offset():
    p = synth.PRESETS["gptoss20b"]
    inp = synth.head_inputs(p.seed, M=p.M, d=p.d, r=p.r, V=p.V, dtype=p.dtype)
    t = {k: to_dev(v, "bf16") for k, v in inp.items()}
    o = ss.slimspec_head_forward(t["hidden"], t["w_down"], t["w_up"], p.temperature, None,
                                 seed=77, offset=3)
    torch.cuda.synchronize()
    u = oracle.philox_uniforms(77, 3, p.M, 1)[:, 0]
    ref = oracle.slimspec_head(inp["hidden"], inp["w_down"], inp["w_up"], "bf16",
                               p.temperature, u)
    counts = check_head_tokens(o["tokens"].cpu().numpy(), ref["logits"], p.temperature, u, 0.0)
    assert counts["exact"] >= p.M - 1
    np.testing.assert_allclose(o["lse"].cpu().numpy(), ref["lse"], atol=2e-2, rtol=0)


def test_offset_advances_the_stream():
    """Two calls that differ only in offset draw different uniforms: on a flat
    distribution over 3000 ids almost every row's token changes."""
    M, d, r, V = 64, 64, 32, 3000
    dev = device()
    h = torch.zeros(M, d, dtype=torch.bfloat16, device=dev)
    wd = torch.zeros(r, d, dtype=torch.bfloat16, device=dev)
    wu = torch.zeros(V, r, dtype=torch.bfloat16, device=dev)
    a = ss.slimspec_head_forward(h, wd, wu, 1.0, None, seed=5, offset=0)["tokens"]
    b = ss.slimspec_head_forward(h, wd, wu, 1.0, None, seed=5, offset=1)["tokens"]
    c = ss.slimspec_head_forward(h, wd, wu, 1.0, None, seed=5, offset=0)["tokens"]
    torch.cuda.synchronize()
    assert torch.equal(a, c)
    assert int((a != b).sum()) >= M - 2
    want = np.floor(oracle.philox_uniforms(5, 1, M, 1)[:, 0] * V)
    assert np.all(np.abs(b.cpu().numpy() - want) <= 1)


def test_trimmed_head_seed_offset():
    rng = np.random.default_rng(8)
    M, d, V, Vk, T = 8, 512, 20000, 3001, 1.0
    h = synth.normal(rng, (M, d), 1.0, "bf16")
    W = synth.normal(rng, (V, d), 1.0 / np.sqrt(d), "bf16")
    kept = np.sort(rng.choice(V, Vk, replace=False)).astype(np.int32)
    o = ss.trimmed_head_forward(to_dev(h, "bf16"), to_dev(W[kept], "bf16"), to_dev(kept, "i32"),
                                T, None, seed=11, offset=12)
    torch.cuda.synchronize()
    u = oracle.philox_uniforms(11, 12, M, 1)[:, 0]
    ref = oracle.trimmed_head(h, W[kept], kept, T, u)
    pos = {int(v): i for i, v in enumerate(kept)}
    got = o["tokens"].cpu().numpy()
    for m in range(M):
        w = np.exp((ref["logits"][m] - ref["logits"][m].max()) / T)
        assert cdf_verdict(pos[int(got[m])], w, float(u[m])) is not None
    assert np.sum(got == ref["tokens"]) >= M - 1


def test_specvocab_seed_offset():
    M, d, dp, V, k, T = 4, 512, 32, 5000, 256, 1.0
    inp = synth.specvocab_inputs(21, M=M, d=d, d_prime=dp, V=V)
    t = {kk: to_dev(vv, "bf16") for kk, vv in inp.items()}
    o = ss.specvocab_head_forward(t["hidden"], t["w_down"], t["w_vocab"], t["u_full"], k, T,
                                  None, seed=3, offset=9)
    torch.cuda.synchronize()
    assert ss.ss_get_device_error() == ss.SS_OK
    u = oracle.philox_uniforms(3, 9, M, 1)[:, 0]
    ref = oracle.specvocab_head(inp["hidden"], inp["w_down"], inp["w_vocab"], inp["u_full"],
                                k, T, u)
    got = o["tokens"].cpu().numpy()
    for m in range(M):
        j = int(np.searchsorted(ref["candidates"][m], got[m]))
        assert ref["candidates"][m][j] == got[m]
        w = np.exp((ref["cand_logits"][m] - ref["cand_logits"][m].max()) / T)
        assert cdf_verdict(j, w, float(u[m])) is not None
    assert np.sum(got == ref["tokens"]) >= M - 1


# --------------------------------------------------------------- verifier ---
@pytest.mark.parametrize("B,g,V,T", [(64, 4, 4096, 1.0), (16, 6, 201088, 0.7)])
def test_verify_seed_offset(B, g, V, T):
    """Accept test j of sequence b draws (row b, slot j), the final draw
    (row b, slot gamma): the oracle, given those uniforms, must agree."""
    v = synth.verify_logits(600 + B, B=B, gamma=g, V=V, kind="zipf" if V > 10000 else "normal")
    x = np.zeros((B, g), np.int32)
    for b in range(B):
        for j in range(g):
            x[b, j] = oracle.row_reduce(v["draft"][b, j], T, v["u_draft"][b, j])["token"]
    seed, offset = 123456789, 42
    tgt, dr, xd = to_dev(v["target"], "f32"), to_dev(v["draft"], "f32"), to_dev(x, "i32")
    a = ss.spec_verify(tgt, dr, xd, T, None, seed=seed, offset=offset)
    u_dev = ss.ss_philox_uniforms(seed, offset, B, g + 1)
    b_ = ss.spec_verify(tgt, dr, xd, T, u_dev)
    torch.cuda.synchronize()
    assert ss.ss_get_device_error() == ss.SS_OK
    assert torch.equal(a["tokens"], b_["tokens"])
    assert torch.equal(a["num_accepted"], b_["num_accepted"])
    u = oracle.philox_uniforms(seed, offset, B, g + 1)
    toks, nacc = a["tokens"].cpu().numpy(), a["num_accepted"].cpu().numpy()
    exact = 0
    for b in range(B):
        n = int(nacc[b])
        assert np.all(toks[b, n + 1:] == -1)
        verdict = check_verify_sampling(toks[b], n, v["target"][b], v["draft"][b], x[b], u[b], T)
        exact += verdict == "exact"
    assert exact >= 0.8 * B


def test_verify_lowrank_seed_offset():
    rng = np.random.default_rng(17)
    B, g, V, r, T = 40, 4, 20000, 128, 1.0   # 40 sequences: the residual-mode epilogue
    z = synth.normal(rng, (g, B, r), 1.0, "bf16")
    w_up = synth.normal(rng, (V, r), 1.0 / np.sqrt(r), "bf16")
    draft = np.einsum("jbr,vr->bjv", z.astype(np.float64), w_up.astype(np.float64))
    target = np.empty((B, g + 1, V), np.float32)
    target[:, :g] = draft + 0.5 * rng.standard_normal((B, g, V))
    target[:, g] = 2.0 * rng.standard_normal((B, V))
    x = np.zeros((B, g), np.int32)
    lp = np.zeros((g, B), np.float32)
    ls = np.zeros((g, B), np.float32)
    ud = synth.uniforms(rng, (B, g))
    for b in range(B):
        for j in range(g):
            rr = oracle.row_reduce(draft[b, j], T, ud[b, j])
            x[b, j], lp[j, b], ls[j, b] = rr["token"], rr["logprob"], rr["lse"]
    args = (to_dev(target, "f32"), to_dev(z.reshape(g * B, r), "bf16"), to_dev(w_up, "bf16"),
            to_dev(lp.reshape(-1), "f32"), to_dev(ls.reshape(-1), "f32"),
            to_dev(np.ascontiguousarray(x.T).reshape(-1), "i32"), T)
    a = ss.spec_verify_lowrank(*args, None, seed=99, offset=100)
    b_ = ss.spec_verify_lowrank(*args, ss.ss_philox_uniforms(99, 100, B, g + 1))
    torch.cuda.synchronize()
    assert ss.ss_get_device_error() == ss.SS_OK
    assert torch.equal(a["tokens"], b_["tokens"])
    assert torch.equal(a["num_accepted"], b_["num_accepted"])
    u = oracle.philox_uniforms(99, 100, B, g + 1)
    toks, nacc = a["tokens"].cpu().numpy(), a["num_accepted"].cpu().numpy()
    exact = 0
    for b in range(B):
        n = int(nacc[b])
        exact += check_verify_sampling(toks[b], n, target[b], draft[b], x[b], u[b], T) == "exact"
    assert exact >= B - 2
