"""GPU parity of the SlimSpec low-rank head against the CPU oracle.

Sizes span several vocabulary tiles with a ragged last tile, several m-tiles,
the fp32 and bf16 paths and every row-width geometry; the full workload
shapes run in the same launch configuration the benchmark times.
Tolerances: logits / statistics 2e-2 absolute for bf16 weights, 1e-5 for the
fp32 workload; tokens by the rules in tests/parity.py.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import speculative_decoding_drafter_slimspec_gb300 as ss
from parity import cdf_verdict, check_head_tokens, greedy_verdict
from gpu_util import device, to_dev

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}
EPS_GREEDY = {"f32": 1e-5, "bf16": 2e-3}


def _z_check(z_gpu, hidden, w_down, dtype):
    ref = oracle.down_projection(hidden, w_down, dtype)
    if dtype == "f32":
        scale = np.maximum(1.0, np.abs(ref))
        assert np.max(np.abs(z_gpu - ref) / scale) < 1e-5
        return 0
    # bf16: equal to the oracle's rounding unless the unrounded value sits
    # within fp32 accumulation error of a rounding midpoint (then one ulp off).
    # The error of a d-term fp32 dot product is at most gamma_d * sum |h_i w_i|
    # with gamma_d = d u / (1 - d u), u = 2^-24 (the standard bound for
    # recursive summation), so that is the distance allowed.
    raw = oracle.down_projection(hidden, w_down, "f32")
    diff = z_gpu != ref
    if np.any(diff):
        ulp = np.abs(ref[diff]) * 2.0 ** -7
        assert np.all(np.abs(z_gpu[diff] - ref[diff]) <= ulp * 1.01)
        d = hidden.shape[1]
        gamma = d * 2.0 ** -24 / (1 - d * 2.0 ** -24)
        abs_sum = np.abs(hidden.astype(np.float64)) @ np.abs(w_down.astype(np.float64)).T
        mid_dist = np.abs(raw[diff] - (z_gpu[diff] + ref[diff]) / 2)
        assert np.all(mid_dist <= gamma * abs_sum[diff] + 1e-30)
    return int(diff.sum())


def run_case(seed, M, d, r, V, dtype, T, logits=True):
    inp = synth.head_inputs(seed, M=M, d=d, r=r, V=V, dtype=dtype)
    u = synth.uniforms(np.random.default_rng(seed + 1), (M,))
    dev = device()
    t = {k: to_dev(v, dtype) for k, v in inp.items()}
    out = ss.slimspec_head_forward(t["hidden"], t["w_down"], t["w_up"], T,
                                   to_dev(u, "f32") if T > 0 else None,
                                   want_z=True, want_logits=logits)
    torch.cuda.synchronize()
    assert ss.ss_get_device_error() == ss.SS_OK
    ref = oracle.slimspec_head(inp["hidden"], inp["w_down"], inp["w_up"], dtype, T,
                               u if T > 0 else None)
    g = {k: v.float().cpu().numpy() if v.dtype != torch.int32 else v.cpu().numpy()
         for k, v in out.items()}
    flips = _z_check(g["z"].astype(np.float64), inp["hidden"], inp["w_down"], dtype)
    tol = TOL[dtype]
    if logits:
        assert np.max(np.abs(g["logits"] - ref["logits"])) <= tol
    counts = check_head_tokens(g["tokens"], ref["logits"], T, u, EPS_GREEDY[dtype])
    np.testing.assert_allclose(g["row_max"], ref["max"], atol=tol, rtol=0)
    np.testing.assert_allclose(g["lse"], ref["lse"], atol=tol, rtol=0)
    # logprob of the token the GPU chose, from the oracle's logits
    lt = ref["logits"][np.arange(M), g["tokens"]]
    if T > 0:
        ref_lp = (lt - ref["max"]) / T - (ref["lse"] - ref["max"] / T)
    else:
        ref_lp = np.zeros(M)
    np.testing.assert_allclose(g["logprob"], ref_lp, atol=tol, rtol=0)
    return counts, flips


SMALL = [
    # seed, M, d, r, V, dtype          geometry exercised
    (11, 1, 256, 32, 4096, "f32"),    # the oracle-scale workload (LPR=8)
    (12, 3, 64, 64, 999, "f32"),      # LPR=32, CPL=1, ragged tail
    (13, 9, 128, 128, 3001, "f32"),   # CPL=2, two m-tiles of 8
    (14, 1, 256, 64, 1000, "bf16"),   # CPL=1 with idle lanes
    (15, 5, 720, 360, 2000, "bf16"),  # r=360: 45 chunks, CPL=2 tail
    (16, 8, 1024, 512, 4133, "bf16"), # CPL=2, MT=8
    (17, 16, 512, 512, 2050, "bf16"), # two m-tiles
    (18, 4, 1024, 1024, 1500, "bf16"),# CPL=4, MT=4
    (19, 2, 64, 32, 1, "bf16"),       # V = 1
    (20, 3, 64, 32, 31, "bf16"),      # V smaller than one tile
    (21, 130, 256, 128, 1100, "bf16"),# two 128-row tiles of z, the second with 2 rows
    (22, 40, 512, 200, 777, "bf16"),  # 5 swizzle atoms of z, last K block 8 wide
    (23, 8, 512, 512, 4096, "bf16"),  # wide stages: 4-D boxes of 4 K blocks, 32 tiles
    (24, 3, 256, 256, 1000, "bf16"),  # wide stages, last tile 104 rows (groups past V read 0)
]


@pytest.mark.parametrize("T", [0.0, 0.7, 1.0])
@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"M{c[1]}-r{c[3]}-V{c[4]}-{c[5]}")
def test_head_small(case, T):
    seed, M, d, r, V, dtype = case
    run_case(seed, M, d, r, V, dtype, T)


def test_head_empty_batch():
    dev = device()
    h = torch.zeros(0, 64, dtype=torch.bfloat16, device=dev)
    out = ss.slimspec_head_forward(h, torch.zeros(32, 64, dtype=torch.bfloat16, device=dev),
                                   torch.zeros(100, 32, dtype=torch.bfloat16, device=dev))
    torch.cuda.synchronize()
    assert out["tokens"].numel() == 0


def test_head_deterministic():
    inp = synth.head_inputs(5, M=8, d=512, r=512, V=20000, dtype="bf16")
    t = {k: to_dev(v, "bf16") for k, v in inp.items()}
    u = to_dev(synth.uniforms(np.random.default_rng(2), (8,)), "f32")
    a = ss.slimspec_head_forward(t["hidden"], t["w_down"], t["w_up"], 1.0, u)
    b = ss.slimspec_head_forward(t["hidden"], t["w_down"], t["w_up"], 1.0, u)
    torch.cuda.synchronize()
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_head_sampling_tie_of_equal_logits():
    """All logits equal: inverse CDF over a flat distribution picks
    floor(u * V) (up to boundary rounding); greedy picks index 0."""
    M, d, r, V = 4, 64, 32, 3000
    dev = device()
    h = torch.zeros(M, d, dtype=torch.bfloat16, device=dev)
    wd = torch.zeros(r, d, dtype=torch.bfloat16, device=dev)
    wu = torch.zeros(V, r, dtype=torch.bfloat16, device=dev)
    u = np.array([0.0, 0.25, 0.5, 0.999], np.float32)
    g = ss.slimspec_head_forward(h, wd, wu, 0.0)
    s = ss.slimspec_head_forward(h, wd, wu, 1.0, to_dev(u, "f32"))
    torch.cuda.synchronize()
    assert g["tokens"].tolist() == [0] * M
    got = s["tokens"].cpu().numpy()
    assert np.all(np.abs(got - np.floor(u * V)) <= 1)


@pytest.mark.parametrize("V", [4133, 128256])
def test_head_greedy_ties_across_tiles(V):
    """Integer logits with the row maximum held by ids in different
    vocabulary tiles (so different CTAs): the lowest such id wins.  h = e_0
    and W_down's column 0 = e_0 make z = e_0 and logits = W_up[:, 0]."""
    M, d, r = 4, 64, 64
    rng = np.random.default_rng(V)
    h = np.zeros((M, d), np.float32)
    h[:, 0] = 1.0
    wd = np.zeros((r, d), np.float32)
    wd[0, 0] = 1.0
    wu = np.zeros((V, r), np.float32)
    wu[:, 0] = rng.integers(-30, 5, V)
    ties = np.sort(rng.choice(np.arange(200, V), 5, replace=False))
    wu[ties, 0] = 9.0
    got = ss.slimspec_head_forward(to_dev(h, "bf16"), to_dev(wd, "bf16"), to_dev(wu, "bf16"),
                                   0.0)
    torch.cuda.synchronize()
    assert got["tokens"].cpu().tolist() == [int(ties[0])] * M
    assert np.all(got["row_max"].cpu().numpy() == 9.0)
    # sampling on the same integer rows: the draw meets the CDF-window rule
    u = synth.uniforms(np.random.default_rng(1), (M,))
    s = ss.slimspec_head_forward(to_dev(h, "bf16"), to_dev(wd, "bf16"), to_dev(wu, "bf16"), 1.0,
                                 to_dev(u, "f32"))
    torch.cuda.synchronize()
    logits = np.broadcast_to(wu[:, 0].astype(np.float64), (M, V))
    check_head_tokens(s["tokens"].cpu().numpy(), logits, 1.0, u, 0.0)


# ------------------------------------------------ full workload shapes -----
@pytest.mark.parametrize("M", [1, 4, 8])
def test_head_llama8b_shape_greedy(M):
    p = synth.PRESETS["llama8b"]
    counts, _ = run_case(p.seed + M, M, p.d, p.r, p.V, p.dtype, 0.0, logits=False)
    assert counts["exact"] + counts["tie"] == M


def test_head_gptoss20b_shape_sampling():
    p = synth.PRESETS["gptoss20b"]
    run_case(p.seed, p.M, p.d, p.r, p.V, p.dtype, p.temperature, logits=False)


def test_head_qwen30b_shape_sampled_rows():
    """M = 256 rows (64 sequences x gamma 4); the oracle checks 24 sampled rows."""
    p = synth.PRESETS["qwen30b"]
    inp = synth.head_inputs(p.seed, M=p.M, d=p.d, r=p.r, V=p.V, dtype=p.dtype)
    u = synth.uniforms(np.random.default_rng(p.seed + 1), (p.M,))
    t = {k: to_dev(v, "bf16") for k, v in inp.items()}
    out = ss.slimspec_head_forward(t["hidden"], t["w_down"], t["w_up"], p.temperature,
                                   to_dev(u, "f32"))
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, 1, 7, 8, 127, 128, 255],
                                     np.random.default_rng(3).integers(0, p.M, 17)]))
    ref = oracle.slimspec_head(inp["hidden"][rows], inp["w_down"], inp["w_up"], "bf16",
                               p.temperature, u[rows])
    toks = out["tokens"].cpu().numpy()[rows]
    check_head_tokens(toks, ref["logits"], p.temperature, u[rows], EPS_GREEDY["bf16"])
    np.testing.assert_allclose(out["lse"].cpu().numpy()[rows], ref["lse"], atol=2e-2, rtol=0)


# ------------------------------------------ many rows: tensor-core z = h W^T --
@pytest.mark.parametrize("seed,M,d,r,V", [
    (31, 200, 2056, 136, 5000),    # ragged K block, ragged second N tile, two M tiles
    (32, 64, 4096, 512, 3000),     # the smallest batch on this path
    (33, 256, 2048, 256, 8192),    # the Qwen-shaped batch
])
@pytest.mark.parametrize("T", [0.0, 1.0])
def test_head_many_rows_split_k_down_projection(seed, M, d, r, V, T):
    """From 64 rows of h the down-projection is a split-K tensor-core GEMM
    (fp32 slices summed in order, then rounded): z within one rounding of
    the oracle's, tokens and statistics as for every head."""
    counts, flips = run_case(seed, M, d, r, V, "bf16", T, logits=True)
    assert counts["exact"] >= M - 2


# -------------------------------------------- sampling finish, run sizes ---
# The sampling finish keeps each warp's run of sub-tile partials in registers,
# in arrays of 8, 16 or 24 per lane chosen by ceil(n_sub / 256), n_sub =
# 2 * ceil(V / 128): these vocabularies give runs of 1, 10 and 19.
@pytest.mark.parametrize("V", [2000, 150000, 300000])
@pytest.mark.parametrize("T", [0.7, 1.0])
def test_head_sampling_finish_run_sizes(V, T):
    run_case(40 + V % 97, 3, 128, 64, V, "bf16", T, logits=False)


# ------------------------------------------------- position-adaptive rank ---
@pytest.mark.parametrize("r", [384, 640, 768, 896, 1024, 2048])
@pytest.mark.parametrize("T", [0.0, 1.0])
def test_head_rank_per_position(r, T):
    """A different rank per drafted position means one head call per rank;
    every rank from r = d/8 up to r = d/2 (K blocks past 512, where the
    finish recomputes a sub-tile over several groups of chunks) runs on the
    tensor cores and matches the oracle."""
    counts, flips = run_case(200 + r, 8, 4096, r, 9000, "bf16", T, logits=True)
    assert counts["exact"] >= 7


# ----------------------------------------------------- static trimmed head ---
def _trimmed_case(seed, M, d, V, Vk, sorted_ids=True):
    rng = np.random.default_rng(seed)
    h = synth.normal(rng, (M, d), 1.0, "bf16")
    W = synth.normal(rng, (V, d), 1.0 / np.sqrt(d), "bf16")
    kept = rng.choice(V, Vk, replace=False)
    if sorted_ids:
        kept = np.sort(kept)
    return h, W[kept], kept.astype(np.int32)


@pytest.mark.parametrize("M,d,V,Vk,T,sorted_ids", [
    (1, 4096, 128256, 32768, 0.0, True),      # FR-Spec-sized: 32K of Llama's 128K ids
    (8, 4096, 128256, 32768, 1.0, True),
    (16, 4096, 50000, 20000, 0.7, True),      # h at the shared-memory limit
    (3, 512, 20000, 1001, 1.0, False),        # ragged kept count, unsorted ids
    (5, 2880, 201088, 16384, 0.0, False),     # d not a multiple of 64
])
def test_trimmed_head_matches_oracle(M, d, V, Vk, T, sorted_ids):
    h, Wk, kept = _trimmed_case(M + d + Vk, M, d, V, Vk, sorted_ids)
    u = synth.uniforms(np.random.default_rng(5), (M,))
    o = ss.trimmed_head_forward(to_dev(h, "bf16"), to_dev(Wk, "bf16"), to_dev(kept, "i32"), T,
                                to_dev(u, "f32") if T > 0 else None)
    torch.cuda.synchronize()
    assert ss.ss_get_device_error() == ss.SS_OK
    ref = oracle.trimmed_head(h, Wk, kept, T, u if T > 0 else None)
    got = o["tokens"].cpu().numpy()
    assert set(got.tolist()) <= set(kept.tolist())
    pos = {int(v): i for i, v in enumerate(kept)}
    for m in range(M):
        j = pos[int(got[m])]
        if T == 0:
            assert greedy_verdict(j, ref["logits"][m], 2e-3) is not None
        else:
            w = np.exp((ref["logits"][m] - ref["logits"][m].max()) / T)
            assert cdf_verdict(j, w, float(u[m])) is not None
    assert np.sum(got == ref["tokens"]) >= M - 1
    # the statistics over the kept set, at the bf16 tolerance
    np.testing.assert_allclose(o["row_max"].cpu().numpy(), ref["max"], atol=2e-2, rtol=0)
    np.testing.assert_allclose(o["lse"].cpu().numpy(), ref["lse"], atol=2e-2, rtol=0)
    kept_index = np.array([pos[int(v)] for v in got])
    lt = ref["logits"][np.arange(M), kept_index]
    ref_lp = (lt - ref["max"]) / T - (ref["lse"] - ref["max"] / T) if T > 0 else np.zeros(M)
    np.testing.assert_allclose(o["logprob"].cpu().numpy(), ref_lp, atol=2e-2, rtol=0)
