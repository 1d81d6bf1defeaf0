"""Whole rounds captured once in a CUDA graph and replayed on fresh inputs.

Every library call is asynchronous, never allocates and never synchronises,
so a round (host-to-device copies of its inputs, the drafting calls on one
stream, the verifier's rows copied on a second stream, the verifier) can be
captured once and replayed.  Each replay here gets new inputs through the same
pinned host buffers; its outputs are checked against the oracle, and must be
bit-identical to the same calls issued one by one (the kernels are
deterministic, so a counter or a workspace word that a replay failed to reset
shows up as a difference).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import speculative_decoding_drafter_slimspec_gb300 as ss
from parity import check_head_tokens, check_verify_sampling
from gpu_util import device

pytestmark = pytest.mark.gpu


class _Round:
    """Static buffers of one round and its step as a sequence of calls."""

    def __init__(self, B, g, d, r, V, T, lowrank):
        dev = device()
        self.B, self.g, self.T, self.lowrank = B, g, T, lowrank
        self.h_host = torch.empty(g, B, d, dtype=torch.bfloat16).pin_memory()
        self.uh_host = torch.empty(g, B, dtype=torch.float32).pin_memory()
        self.t_host = torch.empty(B, g + 1, V, dtype=torch.float32).pin_memory()
        self.uv_host = torch.empty(B, g + 1, dtype=torch.float32).pin_memory()
        self.h = torch.empty(g, B, d, dtype=torch.bfloat16, device=dev)
        self.uh = torch.empty(g, B, dtype=torch.float32, device=dev)
        self.t = torch.empty(B, g + 1, V, dtype=torch.float32, device=dev)
        self.uv = torch.empty(B, g + 1, dtype=torch.float32, device=dev)
        n = g * B   # the head calls' rows, position-major
        self.lr = {"tokens": torch.empty(n, dtype=torch.int32, device=dev),
                   "z": torch.empty(n, r, dtype=torch.bfloat16, device=dev),
                   "logprob": torch.empty(n, dtype=torch.float32, device=dev),
                   "lse": torch.empty(n, dtype=torch.float32, device=dev),
                   "row_max": torch.empty(n, dtype=torch.float32, device=dev)}
        self.x = torch.empty(B, g, dtype=torch.int32, device=dev)
        self.head_ws = torch.empty(ss.slimspec_head_workspace_size(B, d, r, V, ss.SS_BF16),
                                   dtype=torch.uint8, device=dev)
        vws = (ss.spec_verify_lowrank_workspace_size(B, g, V, r) if lowrank
               else ss.spec_verify_workspace_size(B, g, V, T))
        self.ver_ws = torch.empty(max(256, vws), dtype=torch.uint8, device=dev)
        self.out = {"tokens": torch.empty(B, g + 1, dtype=torch.int32, device=dev),
                    "num_accepted": torch.empty(B, dtype=torch.int32, device=dev)}
        self.copy_stream = torch.cuda.Stream(device=dev)
        self.started = torch.cuda.Event()
        self.copied = torch.cuda.Event()

    def step(self, w_down, w_up):
        s = torch.cuda.current_stream()
        self.h.copy_(self.h_host, non_blocking=True)
        self.uh.copy_(self.uh_host, non_blocking=True)
        self.started.record(s)
        self.copy_stream.wait_event(self.started)
        with torch.cuda.stream(self.copy_stream):
            self.t.copy_(self.t_host, non_blocking=True)
            self.uv.copy_(self.uv_host, non_blocking=True)
            self.copied.record(self.copy_stream)
        B, T = self.B, self.T
        for j in range(self.g):
            o = {k: v[j * B:(j + 1) * B] for k, v in self.lr.items()}
            ss.slimspec_head_forward(self.h[j], w_down, w_up, T, self.uh[j] if T > 0 else None,
                                     want_stats=True, want_z=True, workspace=self.head_ws,
                                     out=o)
        s.wait_event(self.copied)
        if self.lowrank:
            ss.spec_verify_lowrank(self.t, self.lr["z"], w_up, self.lr["logprob"],
                                   self.lr["lse"], self.lr["tokens"], T, self.uv,
                                   position_major=True, workspace=self.ver_ws, out=self.out)
        else:
            self.x.copy_(self.lr["tokens"].view(self.g, B).t())
            ss.spec_verify(self.t, None, self.x, T, None, workspace=self.ver_ws, out=self.out)

    def results(self):
        return {"head_tokens": self.lr["tokens"].cpu().numpy().reshape(self.g, self.B),
                "z": self.lr["z"].float().cpu().numpy(),
                "tokens": self.out["tokens"].cpu().numpy(),
                "num_accepted": self.out["num_accepted"].cpu().numpy()}


def _inputs(seed, B, g, d, w_down, w_up):
    """Hidden rows, uniforms, and target rows close to the drafter's own
    logits (so that accept chains of every length occur)."""
    rng = np.random.default_rng(seed)
    hs = [synth.normal(rng, (B, d), 1.0, "bf16") for _ in range(g)]
    logits = [oracle.slimspec_head(h, w_down, w_up, "bf16", 0.0)["logits"] for h in hs]
    V = w_up.shape[0]
    target = np.empty((B, g + 1, V), np.float32)
    for j in range(g):
        target[:, j] = logits[j] + 0.05 * rng.standard_normal((B, V))
    target[:, g] = rng.standard_normal((B, V))
    return {"hidden": hs, "logits": logits, "target": target,
            "u_head": synth.uniforms(rng, (g, B)), "u_verify": synth.uniforms(rng, (B, g + 1))}


def _load(rnd, inp):
    rnd.h_host.copy_(torch.from_numpy(np.stack(inp["hidden"])).to(torch.bfloat16))
    rnd.uh_host.copy_(torch.from_numpy(inp["u_head"]))
    rnd.t_host.copy_(torch.from_numpy(inp["target"]))
    rnd.uv_host.copy_(torch.from_numpy(inp["u_verify"]))


def _run_rounds(T, lowrank, seeds):
    B, g, d, r, V = 8, 3, 512, 128, 20000
    dev = device()
    wi = synth.head_inputs(90, M=B, d=d, r=r, V=V, dtype="bf16")
    w_down = torch.from_numpy(wi["w_down"]).to(torch.bfloat16).to(dev)
    w_up = torch.from_numpy(wi["w_up"]).to(torch.bfloat16).to(dev)
    rnd = _Round(B, g, d, r, V, T, lowrank)
    s = torch.cuda.Stream(device=dev)
    inputs = [_inputs(sd, B, g, d, wi["w_down"], wi["w_up"]) for sd in seeds]
    # the calls one by one on the stream (this also sets kernel attributes
    # before the capture)
    eager = []
    for inp in inputs:
        _load(rnd, inp)
        with torch.cuda.stream(s):
            rnd.step(w_down, w_up)
        s.synchronize()
        assert ss.ss_get_device_error() == ss.SS_OK
        eager.append(rnd.results())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s, capture_error_mode="thread_local"):
        rnd.step(w_down, w_up)
    replayed = []
    for inp in inputs:
        _load(rnd, inp)
        with torch.cuda.stream(s):
            graph.replay()
        s.synchronize()
        assert ss.ss_get_device_error() == ss.SS_OK
        replayed.append(rnd.results())
    return wi, inputs, eager, replayed


def _same(a, b):
    for k in a:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


def test_greedy_round_replayed_as_graph():
    wi, inputs, eager, replayed = _run_rounds(0.0, False, seeds=[1, 2, 3])
    accepted = 0
    for inp, e, got in zip(inputs, eager, replayed):
        _same(e, got)
        for j, tok in enumerate(got["head_tokens"]):
            check_head_tokens(tok, inp["logits"][j], 0.0, None, 2e-3)
        x = got["head_tokens"].T.copy()
        ref_t, ref_n = oracle.verify_batch(inp["target"], None, x, None, 0.0)
        np.testing.assert_array_equal(got["num_accepted"], ref_n)
        np.testing.assert_array_equal(got["tokens"], ref_t)
        accepted += int(got["num_accepted"].sum())
    assert accepted > 0


def test_sampling_lowrank_round_replayed_as_graph():
    T = 1.0
    wi, inputs, eager, replayed = _run_rounds(T, True, seeds=[4, 5])
    w_up = wi["w_up"].astype(np.float64)
    for inp, e, got in zip(inputs, eager, replayed):
        _same(e, got)
        g, B = got["head_tokens"].shape
        for j, tok in enumerate(got["head_tokens"]):
            check_head_tokens(tok, inp["logits"][j], T, inp["u_head"][j], 2e-3)
        # the draft side is the GPU's own z rows through W_up
        z_seq = got["z"].reshape(g, B, -1).transpose(1, 0, 2).astype(np.float64)
        draft = np.einsum("bjr,vr->bjv", z_seq, w_up)
        x = got["head_tokens"].T.copy()
        for b in range(B):
            n = int(got["num_accepted"][b])
            assert np.all(got["tokens"][b, :n] == x[b, :n])
            assert check_verify_sampling(got["tokens"][b], n, inp["target"][b], draft[b], x[b],
                                         inp["u_verify"][b], T) is not None


def test_specvocab_head_replayed_as_graph():
    """The SpecVocab head (router, cluster top-k, gather, exact stage) replayed
    on new hidden rows gives the eager call's outputs bit for bit; the eager
    call is checked against the oracle in test_gpu_specvocab."""
    M, d, dp, V, k, T = 8, 512, 32, 20000, 256, 1.0
    dev = device()
    inp = synth.specvocab_inputs(31, M=M, d=d, d_prime=dp, V=V)
    t = {kk: torch.from_numpy(vv).to(torch.bfloat16).to(dev) for kk, vv in inp.items()}
    rng = np.random.default_rng(32)
    hs = [synth.normal(rng, (M, d), 1.0, "bf16") for _ in range(3)]
    us = [synth.uniforms(rng, (M,)) for _ in range(3)]
    h = torch.empty(M, d, dtype=torch.bfloat16, device=dev)
    u = torch.empty(M, dtype=torch.float32, device=dev)
    ws = torch.empty(ss.specvocab_head_workspace_size(M, d, dp, V, k), dtype=torch.uint8,
                     device=dev)
    out = {"tokens": torch.empty(M, dtype=torch.int32, device=dev),
           "topk_idx": torch.empty(M, k, dtype=torch.int32, device=dev),
           "topk_prob": torch.empty(M, k, dtype=torch.float32, device=dev)}
    s = torch.cuda.Stream(device=dev)

    def call():
        ss.specvocab_head_forward(h, t["w_down"], t["w_vocab"], t["u_full"], k, T, u,
                                  want_prob=True, workspace=ws, out=out)

    def load(i):
        h.copy_(torch.from_numpy(hs[i]).to(torch.bfloat16))
        u.copy_(torch.from_numpy(us[i]))

    eager = []
    for i in range(3):
        load(i)
        with torch.cuda.stream(s):
            call()
        s.synchronize()
        eager.append({kk: vv.cpu().numpy() for kk, vv in out.items()})
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s, capture_error_mode="thread_local"):
        call()
    for i in range(3):
        load(i)
        with torch.cuda.stream(s):
            graph.replay()
        s.synchronize()
        assert ss.ss_get_device_error() == ss.SS_OK
        _same(eager[i], {kk: vv.cpu().numpy() for kk, vv in out.items()})
    # the three inputs really differ
    assert not np.array_equal(eager[0]["topk_idx"], eager[1]["topk_idx"])
