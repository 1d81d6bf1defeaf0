"""The low-rank head entry point that needs no caller workspace.

Callers that cannot allocate device memory -- a runtime that fixes its device
memory at start-up, plugin code without a device allocator, a loop that cannot
afford cudaMalloc's possible synchronisation -- call
slimspec_head_forward_noalloc, whose scratch is a fixed array inside the
library.  These tests call it through the C ABI and check that it returns what
slimspec_head_forward returns with a caller workspace, call after call, and
that a request too large for the fixed scratch is refused.  This file is
collected last so that a run stopping at its first failure has already run the
other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
import speculative_decoding_drafter_slimspec_gb300 as ss
from gpu_util import device, to_dev

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _noalloc(t, T, u, dtype=None, seed=0, offset=0):
    """Direct C-ABI call of slimspec_head_forward_noalloc (dtype code from the
    tensors unless given)."""
    M, d = t["hidden"].shape
    r = t["w_down"].shape[0]
    V = t["w_up"].shape[0]
    dev = t["hidden"].device
    if dtype is None:
        dtype = ss.SS_BF16 if t["hidden"].dtype == torch.bfloat16 else ss.SS_F32
    out = {"tokens": torch.full((M,), -7, dtype=torch.int32, device=dev),
           "logprob": torch.empty(M, dtype=torch.float32, device=dev),
           "row_max": torch.empty(M, dtype=torch.float32, device=dev),
           "lse": torch.empty(M, dtype=torch.float32, device=dev),
           "z": torch.empty(M, r, dtype=t["hidden"].dtype, device=dev)}
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = ss.lib().slimspec_head_forward_noalloc(
        _p(t["hidden"]), _p(t["w_down"]), _p(t["w_up"]), M, d, r, V, dtype, float(T), seed,
        offset, _p(u), _p(out["tokens"]), _p(out["logprob"]), _p(out["row_max"]),
        _p(out["lse"]), _p(out["z"]), None, stream)
    return st, out


CALLS = [
    # (seed, M, d, r, V, T): Llama-shaped greedy, GPT-OSS-shaped sampling, then
    # the first inputs again (the scratch still holds the previous call's data)
    (31, 8, 4096, 512, 128256, 0.0),
    (32, 16, 2880, 360, 201088, 0.7),
    (31, 8, 4096, 512, 128256, 0.0),
]


def test_noalloc_matches_workspace_entry_point_call_after_call():
    device()
    for seed, M, d, r, V, T in CALLS:
        inp = synth.head_inputs(seed, M=M, d=d, r=r, V=V, dtype="bf16")
        t = {k: to_dev(v, "bf16") for k, v in inp.items()}
        u = to_dev(synth.uniforms(np.random.default_rng(seed), (M,)), "f32") if T > 0 else None
        ref = ss.slimspec_head_forward(t["hidden"], t["w_down"], t["w_up"], T, u, want_z=True)
        st, got = _noalloc(t, T, u)
        assert st == ss.SS_OK, ss.lib().ss_status_string(st)
        torch.cuda.synchronize()
        assert ss.ss_get_device_error() == ss.SS_OK
        assert torch.equal(got["tokens"], ref["tokens"])
        assert torch.equal(got["z"], ref["z"])
        for k in ("logprob", "row_max", "lse"):
            assert torch.max(torch.abs(got[k] - ref[k])).item() <= 2e-2, k


def test_noalloc_fp32_head_and_philox_draws():
    """The fp32 head (the CUDA-core stream, whose scratch size follows the
    SM count) at the oracle-scale shape, sampling with uniforms and with the
    Philox stream, twice in a row: the same bits as the workspace call."""
    device()
    inp = synth.head_inputs(11, M=1, d=256, r=32, V=4096, dtype="f32")
    t = {k: to_dev(v, "f32") for k, v in inp.items()}
    u = to_dev(synth.uniforms(np.random.default_rng(3), (1,)), "f32")
    for _ in range(2):
        for uu, seed, offset in ((u, 0, 0), (None, 17, 4)):
            ref = ss.slimspec_head_forward(t["hidden"], t["w_down"], t["w_up"], 1.0, uu,
                                           seed=seed, offset=offset, want_z=True)
            st, got = _noalloc(t, 1.0, uu, seed=seed, offset=offset)
            assert st == ss.SS_OK, ss.lib().ss_status_string(st)
            torch.cuda.synchronize()
            assert ss.ss_get_device_error() == ss.SS_OK
            for k in ("tokens", "z", "logprob", "row_max", "lse"):
                assert torch.equal(got[k], ref[k]), k


def test_noalloc_rejects_an_invalid_dtype_without_writing():
    dev = device()
    t = {"hidden": torch.zeros(2, 64, dtype=torch.bfloat16, device=dev),
         "w_down": torch.zeros(32, 64, dtype=torch.bfloat16, device=dev),
         "w_up": torch.zeros(100, 32, dtype=torch.bfloat16, device=dev)}
    st, got = _noalloc(t, 0.0, None, dtype=7)
    assert st == ss.SS_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(got["tokens"] == -7)


def test_noalloc_refuses_requests_beyond_its_scratch():
    """256 rows at the Qwen3-30B shape need more than the fixed 4 MiB."""
    dev = device()
    M, d, r, V = 256, 2048, 256, 151936
    assert ss.slimspec_head_workspace_size(M, d, r, V, ss.SS_BF16) > (4 << 20)
    t = {"hidden": torch.zeros(M, d, dtype=torch.bfloat16, device=dev),
         "w_down": torch.zeros(r, d, dtype=torch.bfloat16, device=dev),
         "w_up": torch.zeros(V, r, dtype=torch.bfloat16, device=dev)}
    st, got = _noalloc(t, 0.0, None)
    assert st == ss.SS_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(got["tokens"] == -7)   # nothing was written
