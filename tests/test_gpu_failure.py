"""Failure detection on the GPU without a fault: a bounded wait runs out.

The library's test switch makes the tensor-core up-projection's MMA issuer
wait on a barrier that nothing arrives on.  With the pipeline wait limit
lowered to 2 ms, the stalled call gives up: every role of the kernel records
SS_ERR_TIMEOUT, lets the copies it issued land, frees its tensor memory and
returns.  The context stays usable: with the switch off and the limit back
at 1 s, the next calls on the same workspace match the oracle.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import synth
import speculative_decoding_drafter_slimspec_gb300 as ss
from parity import check_head_tokens
from gpu_util import device, to_dev

pytestmark = pytest.mark.gpu


def _check_head(out, inp, T, u):
    ref = oracle.slimspec_head(inp["hidden"], inp["w_down"], inp["w_up"], "bf16", T, u)
    check_head_tokens(out["tokens"].cpu().numpy(), ref["logits"], T, u, 2e-3)
    np.testing.assert_allclose(out["lse"].cpu().numpy(), ref["lse"], atol=2e-2, rtol=0)


@pytest.mark.parametrize("r,V", [(64, 5000), (512, 20000)])
def test_stalled_head_times_out_and_the_next_call_is_correct(r, V):
    dev = device()
    M, d = 4, 512
    inp = synth.head_inputs(70 + r, M=M, d=d, r=r, V=V, dtype="bf16")
    t = {k: to_dev(v, "bf16") for k, v in inp.items()}
    ws = torch.zeros(ss.slimspec_head_workspace_size(M, d, r, V, ss.SS_BF16), dtype=torch.uint8,
                     device=dev)
    u = synth.uniforms(np.random.default_rng(r), (M,))
    ud = to_dev(u, "f32")
    assert ss.ss_get_device_error() == ss.SS_OK
    try:
        ss.ss_set_wait_limit_ns(2_000_000)
        ss.ss_set_stall_test(True)
        t0 = time.perf_counter()
        ss.slimspec_head_forward(t["hidden"], t["w_down"], t["w_up"], 0.0, workspace=ws)
        assert ss.ss_get_device_error() == ss.SS_ERR_TIMEOUT
        assert time.perf_counter() - t0 < 0.9   # gave up at the short limit, not at 1 s
    finally:
        ss.ss_set_stall_test(False)
        ss.ss_set_wait_limit_ns(10 ** 9)
    assert ss.ss_get_device_error() == ss.SS_OK  # the read cleared it
    for T in (0.0, 1.0):
        out = ss.slimspec_head_forward(t["hidden"], t["w_down"], t["w_up"], T,
                                       ud if T > 0 else None, workspace=ws)
        torch.cuda.synchronize()
        assert ss.ss_get_device_error() == ss.SS_OK
        _check_head(out, inp, T, u)
