"""GPU parity of spec_verify against the CPU oracle (greedy and sampling).

Logit rows are fp32 inputs shared bit-for-bit by both sides, so argmax
decisions are exact; sampling decisions follow tests/parity.py.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import speculative_decoding_drafter_slimspec_gb300 as ss
from parity import check_verify_sampling
from gpu_util import device, to_dev

pytestmark = pytest.mark.gpu


def _drafts(v, T):
    """Drafted tokens from the draft rows: argmax (T = 0) or an inverse-CDF
    draw with the drafter's own uniforms (the oracle's row_reduce)."""
    B, g, V = v["draft"].shape
    x = np.zeros((B, g), np.int32)
    for b in range(B):
        for j in range(g):
            r = oracle.row_reduce(v["draft"][b, j], T, v["u_draft"][b, j] if T > 0 else None)
            x[b, j] = r["token"]
    return x


def run_verify(v, x, T):
    tgt = to_dev(v["target"], "f32")
    dr = to_dev(v["draft"], "f32") if T > 0 else None
    u = to_dev(v["u_verify"], "f32") if T > 0 else None
    o = ss.spec_verify(tgt, dr, to_dev(x, "i32"), T, u)
    torch.cuda.synchronize()
    assert ss.ss_get_device_error() == ss.SS_OK
    return o["tokens"].cpu().numpy(), o["num_accepted"].cpu().numpy()


def check(v, x, T, toks, nacc):
    B = x.shape[0]
    if T == 0:
        ref_t, ref_n = oracle.verify_batch(v["target"], None, x, None, 0.0)
        np.testing.assert_array_equal(nacc, ref_n)
        np.testing.assert_array_equal(toks, ref_t)
        return {"exact": B, "boundary": 0}
    counts = {"exact": 0, "boundary": 0}
    for b in range(B):
        n = int(nacc[b])
        assert 0 <= n <= x.shape[1]
        assert np.all(toks[b, n + 1:] == -1)
        verdict = check_verify_sampling(toks[b], n, v["target"][b], v["draft"][b], x[b],
                                        v["u_verify"][b], T)
        counts[verdict] += 1
    return counts


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_verify_tiny(T):
    p = synth.PRESETS["tiny"]
    v = synth.verify_logits(p.seed, B=64, gamma=p.gamma, V=p.V, kind="normal", draft_sigma=1.0)
    x = _drafts(v, T)
    toks, n = run_verify(v, x, T)
    c = check(v, x, T, toks, n)
    assert c["exact"] >= 0.9 * 64


@pytest.mark.parametrize("V", [1, 3, 1001, 4097])
@pytest.mark.parametrize("T", [0.0, 0.5])
def test_verify_ragged_vocab(V, T):
    """V not a multiple of 4 (scalar path), V = 1, one element past a chunk."""
    v = synth.verify_logits(40 + V, B=7, gamma=3, V=V, kind="normal")
    x = _drafts(v, T)
    toks, n = run_verify(v, x, T)
    check(v, x, T, toks, n)


def test_verify_tiny_vocab_many_sequences():
    """V = 4, gamma = 2 with 4096 random (draft, uniform) combinations: every
    outcome matches the oracle's decision procedure."""
    rng = np.random.default_rng(9)
    B, g, V, T = 4096, 2, 4, 1.0
    base_t = rng.standard_normal((g + 1, V)).astype(np.float32)
    base_d = rng.standard_normal((g, V)).astype(np.float32)
    v = {"target": np.ascontiguousarray(np.broadcast_to(base_t, (B, g + 1, V))),
         "draft": np.ascontiguousarray(np.broadcast_to(base_d, (B, g, V))),
         "u_verify": synth.uniforms(rng, (B, g + 1))}
    x = rng.integers(0, V, (B, g)).astype(np.int32)
    toks, n = run_verify(v, x, T)
    c = check(v, x, T, toks, n)
    assert c["exact"] >= B - 5
    # empirical acceptance at position 0 against sum_x min(p, q) under x ~ uniform
    p0 = oracle.softmax_t(base_t[0], T)
    q0 = oracle.softmax_t(base_d[0], T)
    acc = np.mean([min(1.0, p0[xx] / q0[xx]) for xx in x[:, 0]])
    assert abs(np.mean(n > 0) - acc) < 4 * np.sqrt(acc * (1 - acc) / B) + 1e-3


def _tied_rows(seed, B, g, V):
    """Integer-valued target rows whose maximum (8) is held by several ids of
    every row, spread over the row's 2048-float chunks; draft rows = target +
    small integers.  Returns (target, draft, lowest tied id per row)."""
    rng = np.random.default_rng(seed)
    target = rng.integers(-20, 5, (B, g + 1, V)).astype(np.float32)
    low = np.zeros((B, g + 1), np.int64)
    tied = {}
    for b in range(B):
        for j in range(g + 1):
            ids = np.sort(rng.choice(V, 2 + (b + j) % 5, replace=False))
            target[b, j, ids] = 8.0
            low[b, j] = ids[0]
            tied[b, j] = ids
    draft = (target[:, :g] + rng.integers(-2, 3, (B, g, V))).astype(np.float32)
    return target, draft, low, tied


@pytest.mark.parametrize("V", [5003, 131072])
def test_verify_greedy_exact_ties_lowest_index(V):
    """Several ids share each target row's maximum: the target's choice is
    the lowest of them.  A draft at the lowest tied id is kept, one at a
    higher tied id is rejected and replaced by the lowest; bit-exact with the
    oracle (the larger V also runs the position-0 split)."""
    B, g = 24, 4
    target, draft, low, tied = _tied_rows(31 + V, B, g, V)
    x = low[:, :g].astype(np.int32).copy()
    for b in range(B):
        if b % 3 == 1:
            x[b, 2] = tied[b, 2][-1]           # a higher tied id at position 2
        elif b % 3 == 2:
            x[b, 0] = tied[b, 0][1]            # the second-lowest tied id at position 0
    v = {"target": target, "draft": draft}
    toks, n = run_verify(v, x, 0.0)
    check(v, x, 0.0, toks, n)
    assert np.all(n[0::3] == g) and np.all(n[1::3] == 2) and np.all(n[2::3] == 0)
    np.testing.assert_array_equal(toks[0::3, g], low[0::3, g])
    np.testing.assert_array_equal(toks[1::3, 2], low[1::3, 2])
    np.testing.assert_array_equal(toks[2::3, 0], low[2::3, 0])


@pytest.mark.parametrize("T", [1.0, 0.5])
def test_verify_sampling_on_tied_integer_rows(T):
    """Sampling on rows of exact ties (integer logits): every accept decision,
    residual and bonus draw meets the parity rules."""
    B, g, V = 32, 4, 5003
    target, draft, low, tied = _tied_rows(77, B, g, V)
    rng = np.random.default_rng(78)
    v = {"target": target, "draft": draft, "u_draft": synth.uniforms(rng, (B, g)),
         "u_verify": synth.uniforms(rng, (B, g + 1))}
    x = _drafts(v, T)
    toks, n = run_verify(v, x, T)
    c = check(v, x, T, toks, n)
    assert c["exact"] >= B - 2


def test_verify_bad_token_reports_device_error():
    v = synth.verify_logits(5, B=2, gamma=3, V=500, kind="normal")
    x = np.array([[1, 2, 3], [4, 600, 5]], np.int32)   # 600 >= V
    o = ss.spec_verify(to_dev(v["target"], "f32"), None, to_dev(x, "i32"), 0.0)
    assert ss.ss_get_device_error() == ss.SS_ERR_DEVICE_INDEX
    assert int(o["num_accepted"][1]) <= 1
    assert ss.ss_get_device_error() == ss.SS_OK      # cleared by the read


def test_verify_split_greedy():
    """Rows above the split size: position 0 is decided between two row
    passes.  Half the sequences keep their position-0 token (so their later
    rows are read), half reject it (so theirs are not)."""
    B, g, V = 32, 4, 131072
    assert B * (g + 1) * V * 4 >= 64 * 2 ** 20
    v = synth.verify_logits(77, B=B, gamma=g, V=V, kind="zipf")
    x = _drafts(v, 0.0)
    a0 = np.argmax(v["target"][:, 0], axis=1)
    x[::2, 0] = a0[::2]                              # kept at position 0
    x[1::2, 0] = (a0[1::2] + 1) % V                  # rejected at position 0
    x[::4, 1:] = np.argmax(v["target"][::4, 1:g], axis=2)  # and some keep everything
    toks, n = run_verify(v, x, 0.0)
    check(v, x, 0.0, toks, n)
    assert np.all(n[1::2] == 0) and np.all(n[::4] == g)


@pytest.mark.parametrize("T", [0.7, 1.5])
def test_verify_split_sampling(T):
    """Sampling above the split size, with drafts close to the target (most
    sequences keep position 0) and far from it (most do not)."""
    B, g, V = 16, 3, 262144
    assert B * (2 * g + 1) * V * 4 >= 64 * 2 ** 20
    v = synth.verify_logits(78, B=B, gamma=g, V=V, kind="zipf", draft_sigma=0.3)
    far = synth.verify_logits(79, B=B, gamma=g, V=V, kind="zipf", draft_sigma=3.0)
    v["draft"][B // 2:] = far["draft"][B // 2:]
    x = _drafts(v, T)
    toks, n = run_verify(v, x, T)
    c = check(v, x, T, toks, n)
    print("split sampling", T, c, n.tolist())
    assert c["exact"] >= 0.8 * B


# ------------------------------------------------ full workload shapes -----
def test_verify_llama8b_shape_greedy():
    p = synth.PRESETS["llama8b"]
    v = synth.verify_logits(p.seed, B=p.B, gamma=p.gamma, V=p.V, kind="zipf")
    x = _drafts(v, 0.0)
    toks, n = run_verify(v, x, 0.0)
    check(v, x, 0.0, toks, n)


def test_verify_gptoss20b_shape_sampling():
    p = synth.PRESETS["gptoss20b"]
    v = synth.verify_logits(p.seed, B=p.B, gamma=p.gamma, V=p.V, kind="zipf",
                            draft_sigma=p.draft_sigma)
    x = _drafts(v, p.temperature)
    toks, n = run_verify(v, x, p.temperature)
    c = check(v, x, p.temperature, toks, n)
    print("gptoss20b verify", c)
    assert c["exact"] >= 0.8 * p.B


@pytest.mark.parametrize("sigma", [0.5, 1.0, 2.0])
def test_verify_qwen30b_shape_sampling(sigma):
    p = synth.PRESETS["qwen30b"]
    v = synth.verify_logits(p.seed + int(sigma * 10), B=p.B, gamma=p.gamma, V=p.V, kind="zipf",
                            draft_sigma=sigma)
    x = _drafts(v, p.temperature)
    toks, n = run_verify(v, x, p.temperature)
    c = check(v, x, p.temperature, toks, n)
    print("qwen30b verify sigma", sigma, c)
    # every outcome is valid (checked above); tokens drawn from the long tail,
    # where neighbouring ids hold ~1e-7 of the mass each, may legitimately sit
    # on the other side of an fp32-vs-fp64 rounding boundary
    assert c["exact"] >= 0.8 * p.B


# ------------------------------------------ draft side from the low-rank head
def _lowrank_case(seed, B, g, V, r, T, sigma):
    """z rows (position-major, g x B) and W_up with bf16 values, draft logits
    z W_up^T, target = draft + N(0, sigma^2) at the drafted positions, tokens
    drawn from q, and the head-side log q(x) and LSE (oracle values in fp32)."""
    rng = np.random.default_rng(seed)
    z = synth.normal(rng, (g, B, r), 1.0, "bf16")
    w_up = synth.normal(rng, (V, r), 1.0 / np.sqrt(r), "bf16")
    draft_pm = np.einsum("jbr,vr->jbv", z.astype(np.float64), w_up.astype(np.float64))
    draft = np.ascontiguousarray(draft_pm.transpose(1, 0, 2))           # (B, g, V)
    target = np.empty((B, g + 1, V), np.float32)
    target[:, :g] = draft + sigma * rng.standard_normal((B, g, V))
    target[:, g] = 2.0 * rng.standard_normal((B, V))
    u_draft = synth.uniforms(rng, (B, g))
    x = np.zeros((B, g), np.int32)
    logprob = np.zeros((g, B), np.float32)
    lse = np.zeros((g, B), np.float32)
    for b in range(B):
        for j in range(g):
            rr = oracle.row_reduce(draft[b, j], T, u_draft[b, j])
            x[b, j] = rr["token"]
            logprob[j, b] = rr["logprob"]
            lse[j, b] = rr["lse"]
    u = synth.uniforms(rng, (B, g + 1))
    z_seq = np.ascontiguousarray(z.transpose(1, 0, 2))                  # (B, g, r)
    return dict(z=z, z_seq=z_seq, w_up=w_up, draft=draft, target=target, x=x, logprob=logprob,
                lse=lse, u=u)


def _run_lowrank(c, T, position_major=True):
    g, B, r = c["z"].shape
    if position_major:
        z, lp, ls = c["z"].reshape(g * B, r), c["logprob"].reshape(-1), c["lse"].reshape(-1)
        x = np.ascontiguousarray(c["x"].T).reshape(-1)
    else:
        z = c["z_seq"].reshape(B * g, r)
        lp = np.ascontiguousarray(c["logprob"].T).reshape(-1)
        ls = np.ascontiguousarray(c["lse"].T).reshape(-1)
        x = c["x"].reshape(-1)
    o = ss.spec_verify_lowrank(to_dev(c["target"], "f32"), to_dev(z, "bf16"),
                               to_dev(c["w_up"], "bf16"), to_dev(lp, "f32"), to_dev(ls, "f32"),
                               to_dev(x, "i32"), T, to_dev(c["u"], "f32"),
                               position_major=position_major)
    torch.cuda.synchronize()
    assert ss.ss_get_device_error() == ss.SS_OK
    return o["tokens"].cpu().numpy(), o["num_accepted"].cpu().numpy()


def _check_lowrank(c, T, toks, nacc):
    ref_t, ref_n = oracle.verify_lowrank_batch(c["target"], c["z_seq"], c["w_up"], c["x"], c["u"], T)
    B = c["x"].shape[0]
    counts = {"exact": 0, "boundary": 0}
    for b in range(B):
        n = int(nacc[b])
        assert 0 <= n <= c["x"].shape[1]
        assert np.all(toks[b, n + 1:] == -1)
        verdict = check_verify_sampling(toks[b], n, c["target"][b], c["draft"][b], c["x"][b],
                                        c["u"][b], T)
        counts[verdict] += 1
    same = int(np.sum(np.all(toks == ref_t, axis=1)))
    return counts, same


@pytest.mark.parametrize("V,r,T,sigma,B", [(1000, 64, 1.0, 0.3, 16), (1001, 40, 0.7, 1.0, 48),
                                           (50000, 256, 1.0, 0.5, 48), (20000, 360, 0.7, 2.0, 16),
                                           (20000, 360, 0.7, 2.0, 48), (4097, 512, 1.3, 0.5, 33)])
def test_verify_lowrank_matches_oracle(V, r, T, sigma, B):
    """Draft side from z rows and W_up (ragged vocabularies, r not a multiple
    of 64, close and far drafts; below 32 sequences the recomputed rows are
    written out, from 32 on they are reduced in the tensor-core epilogue):
    every outcome is one the oracle's decision procedure allows, and almost
    all are the oracle's own."""
    g = 4
    c = _lowrank_case(V + r, B, g, V, r, T, sigma)
    toks, n = _run_lowrank(c, T)
    counts, same = _check_lowrank(c, T, toks, n)
    print("lowrank", V, r, T, sigma, counts, "identical rows", same, "accepted", n.tolist())
    assert counts["exact"] >= B - 2 and same >= B - 2


def test_verify_lowrank_sequence_major_rows():
    """z, log q and LSE given sequence-major (B x gamma rows) give the same
    outcome as position-major."""
    c = _lowrank_case(9, 8, 3, 5000, 128, 1.0, 0.5)
    a = _run_lowrank(c, 1.0, position_major=True)
    b = _run_lowrank(c, 1.0, position_major=False)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_verify_lowrank_split_path():
    """Target rows above the split size (position 0 decided between two row
    passes) with the low-rank draft side."""
    B, g, V, r, T = 32, 4, 131072, 128, 1.0
    assert B * (g + 1) * V * 4 >= 64 * 2 ** 20
    c = _lowrank_case(31, B, g, V, r, T, 0.3)
    toks, n = _run_lowrank(c, T)
    counts, same = _check_lowrank(c, T, toks, n)
    print("lowrank split", counts, "identical rows", same, "accepted", n.tolist())
    assert counts["exact"] >= B - 2


def test_verify_lowrank_after_head_calls():
    """A whole sampling round on the GPU: gamma low-rank head calls produce
    tokens, log q(x), LSE and z; the verifier consumes them as they are.
    Outcomes are checked against the oracle fed the head's own z rows."""
    B, g, d, r, V, T = 8, 3, 512, 128, 20000, 1.0
    rng = np.random.default_rng(44)
    inp = synth.head_inputs(44, M=B, d=d, r=r, V=V, dtype="bf16")
    w_down, w_up = inp["w_down"], inp["w_up"]
    hs = [synth.normal(rng, (B, d), 1.0, "bf16") for _ in range(g)]
    u_head = synth.uniforms(rng, (g, B))
    zs, lps, lses, toks = [], [], [], []
    for j in range(g):
        o = ss.slimspec_head_forward(to_dev(hs[j], "bf16"), to_dev(w_down, "bf16"),
                                     to_dev(w_up, "bf16"), T, to_dev(u_head[j], "f32"),
                                     want_stats=True, want_z=True)
        zs.append(o["z"]); lps.append(o["logprob"]); lses.append(o["lse"]); toks.append(o["tokens"])
    torch.cuda.synchronize()
    z = torch.cat(zs).contiguous()                       # (g*B, r) position-major
    lp = torch.cat(lps).contiguous()
    ls = torch.cat(lses).contiguous()
    x = torch.cat(toks).contiguous()                     # (g*B,) position-major
    z_seq = z.float().cpu().numpy().reshape(g, B, r).transpose(1, 0, 2).copy()
    draft = np.einsum("bjr,vr->bjv", z_seq.astype(np.float64), w_up.astype(np.float64))
    target = np.empty((B, g + 1, V), np.float32)
    target[:, :g] = draft + 0.5 * rng.standard_normal((B, g, V))
    target[:, g] = rng.standard_normal((B, V))
    u = synth.uniforms(rng, (B, g + 1))
    o = ss.spec_verify_lowrank(to_dev(target, "f32"), z, to_dev(w_up, "bf16"), lp, ls, x, T,
                               to_dev(u, "f32"))
    torch.cuda.synchronize()
    assert ss.ss_get_device_error() == ss.SS_OK
    got_t, got_n = o["tokens"].cpu().numpy(), o["num_accepted"].cpu().numpy()
    xn = x.cpu().numpy().reshape(g, B).T.copy()
    for b in range(B):
        n = int(got_n[b])
        assert np.all(got_t[b, :n] == xn[b, :n])
        verdict = check_verify_sampling(got_t[b], n, target[b], draft[b], xn[b], u[b], T)
        assert verdict is not None


def _run_both(v, x, T, seed=5):
    """The split and the lazy schedule on the same inputs (Philox draws at the
    same seed and offset)."""
    tgt = to_dev(v["target"], "f32")
    dr = to_dev(v["draft"], "f32") if T > 0 else None
    xd = to_dev(x, "i32")
    a = ss.spec_verify(tgt, dr, xd, T, seed=seed, offset=3)
    b = ss.spec_verify(tgt, dr, xd, T, seed=seed, offset=3, lazy=True)
    torch.cuda.synchronize()
    assert ss.ss_get_device_error() == ss.SS_OK
    return ({k: t.cpu().numpy() for k, t in a.items()},
            {k: t.cpu().numpy() for k, t in b.items()})


@pytest.mark.parametrize("T", [0.0, 1.0])
@pytest.mark.parametrize("B,g,V", [(7, 3, 1001), (64, 4, 4097), (16, 6, 40000), (4, 32, 2048)])
def test_verify_lazy_equals_split(B, g, V, T):
    """The lazy schedule (rows read position by position, only for the
    sequences still kept) gives the split schedule's results bit for bit:
    its decisions take the same partials of the same rows."""
    v = synth.verify_logits(300 + V + g, B=B, gamma=g, V=V, kind="zipf", draft_sigma=0.5)
    x = _drafts(v, T)
    if T == 0.0:
        a0 = np.argmax(v["target"][:, :g], axis=2)
        x[::3] = a0[::3]                      # some sequences keep every position
        x[1::3, 0] = (a0[1::3, 0] + 1) % V    # some reject position 0
    a, b = _run_both(v, x, T)
    np.testing.assert_array_equal(b["num_accepted"], a["num_accepted"])
    np.testing.assert_array_equal(b["tokens"], a["tokens"])
    if T == 0.0:
        assert np.all(a["num_accepted"][::3] == g)
        assert np.all(a["num_accepted"][1::3] == 0)


@pytest.mark.parametrize("T", [0.0, 0.7])
def test_verify_lazy_matches_oracle(T):
    """The lazy schedule against the oracle above the split size, with
    sequences rejected at every position."""
    B, g, V = 24, 5, 65536
    v = synth.verify_logits(91, B=B, gamma=g, V=V, kind="zipf", draft_sigma=0.4)
    x = _drafts(v, T)
    if T == 0.0:
        a = np.argmax(v["target"][:, :g], axis=2)
        for b in range(B):                    # sequence b keeps exactly min(b % (g+1), g) tokens
            keep = b % (g + 1)
            x[b, :keep] = a[b, :keep]
            if keep < g:
                x[b, keep] = (a[b, keep] + 1) % V
    tgt = to_dev(v["target"], "f32")
    dr = to_dev(v["draft"], "f32") if T > 0 else None
    u = to_dev(v["u_verify"], "f32") if T > 0 else None
    o = ss.spec_verify(tgt, dr, to_dev(x, "i32"), T, u, lazy=True)
    torch.cuda.synchronize()
    assert ss.ss_get_device_error() == ss.SS_OK
    toks, n = o["tokens"].cpu().numpy(), o["num_accepted"].cpu().numpy()
    c = check(v, x, T, toks, n)
    if T == 0.0:
        np.testing.assert_array_equal(n, [b % (g + 1) for b in range(B)])
    else:
        assert c["exact"] >= 0.8 * B
