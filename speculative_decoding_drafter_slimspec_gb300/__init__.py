"""GB300 (sm_103a) drafter head and speculative verifier.

A thin ctypes binding over ``libslimspec.so`` (C ABI in ``include/slimspec.h``).
Every step of the computation runs in the library's CUDA kernels; this module
only checks tensors, allocates outputs and workspace with PyTorch and passes
raw device pointers plus the current CUDA stream.  There is no CPU path: if
the library is missing or a tensor is not on a CUDA device, the call raises.

Public calls (same names as the C ABI):
    slimspec_head_forward   SlimSpec low-rank head + per-row reduction
    specvocab_head_forward  SpecVocab-style dynamic-vocabulary head
    ss_topk_rows            the top-k stage on its own
    spec_verify             greedy / sampling verification
    spec_verify_lowrank     sampling verification with the draft side from the head
    trimmed_head_forward    dense head over a kept subset of the vocabulary
    ss_philox_uniforms      the Philox4x32-10 uniforms a sampling call draws
    ss_philox4x32_10        raw Philox4x32-10 blocks
    ss_get_device_error     device error word (synchronises the stream)

Sampling calls draw their uniforms from the library's Philox4x32-10 stream at
(seed, offset) unless ``uniforms`` is given (a hook for exact tests).
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

__all__ = [
    "SS_OK", "SS_ERR_INVALID_ARG", "SS_ERR_UNSUPPORTED", "SS_ERR_WORKSPACE",
    "SS_ERR_CUDA", "SS_ERR_TIMEOUT", "SS_ERR_DEVICE_INDEX", "SlimspecError",
    "lib", "lib_path", "header_functions", "slimspec_head_forward",
    "specvocab_head_forward", "ss_topk_rows", "spec_verify", "spec_verify_lazy", "spec_verify_lowrank",
    "ss_get_device_error", "slimspec_head_workspace_size", "specvocab_head_workspace_size",
    "spec_verify_workspace_size", "spec_verify_lowrank_workspace_size", "ss_topk_workspace_size",
    "trimmed_head_forward", "trimmed_head_workspace_size", "ss_philox_uniforms",
    "ss_philox4x32_10", "ss_set_wait_limit_ns", "ss_set_stall_test",
]

SS_OK, SS_ERR_INVALID_ARG, SS_ERR_UNSUPPORTED, SS_ERR_WORKSPACE = 0, 1, 2, 3
SS_ERR_CUDA, SS_ERR_TIMEOUT, SS_ERR_DEVICE_INDEX = 4, 5, 6
SS_F32, SS_BF16 = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_HEADER = os.path.join(os.path.dirname(_HERE), "include", "slimspec.h")
_LIB = None

_vp, _i, _f, _sz, _u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_uint64
_SIGS = {
    "ss_status_string": (ctypes.c_char_p, [_i]),
    "ss_version": (_i, []),
    "ss_get_device_error": (_i, [_vp]),
    "slimspec_head_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
    "ss_philox_uniforms": (_i, [_u64, _u64, _i, _i, _vp, _vp]),
    "ss_philox4x32_10": (_i, [_vp, _i, _vp, _vp]),
    "slimspec_head_forward": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _u64, _u64, _vp, _vp,
                                   _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "slimspec_head_forward_noalloc": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _u64, _u64,
                                           _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "specvocab_head_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
    "specvocab_head_forward": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _u64, _u64, _vp,
                                    _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "ss_topk_workspace_size": (_sz, [_i, _i, _i]),
    "ss_topk_rows": (_i, [_vp, _i, _i, _i, _vp, _vp, _sz, _vp]),
    "spec_verify_workspace_size": (_sz, [_i, _i, _i, _f]),
    "spec_verify": (_i, [_vp, _vp, _vp, _i, _i, _i, _f, _u64, _u64, _vp, _vp, _vp, _vp, _sz,
                         _vp]),
    "spec_verify_lazy": (_i, [_vp, _vp, _vp, _i, _i, _i, _f, _u64, _u64, _vp, _vp, _vp, _vp, _sz,
                         _vp]),
    "spec_verify_lowrank_workspace_size": (_sz, [_i, _i, _i, _i]),
    "trimmed_head_workspace_size": (_sz, [_i, _i, _i]),
    "trimmed_head_forward": (_i, [_vp, _vp, _vp, _i, _i, _i, _f, _u64, _u64, _vp, _vp, _vp,
                                  _vp, _vp, _vp, _sz, _vp]),
    "spec_verify_lowrank": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _vp, _i, _i, _i, _f, _u64,
                                 _u64, _vp, _vp, _vp, _vp, _sz, _vp]),
    "ss_launch_count": (ctypes.c_longlong, []),
    "ss_profile_start": (_i, []),
    "ss_profile_stop": (_i, []),
    "ss_profile_read": (_i, [_vp, _vp, _i, _i]),
    "ss_profile_kind_name": (ctypes.c_char_p, [_i]),
    "ss_set_wait_limit_ns": (_i, [_u64]),
    "ss_set_stall_test": (_i, [_i]),
}


class SlimspecError(RuntimeError):
    """A non-zero ss_status returned by the library."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {lib().ss_status_string(status).decode()}")


def lib_path() -> str:
    return os.path.join(_HERE, "libslimspec.so")


def header_functions() -> list:
    """Names of the functions declared in include/slimspec.h."""
    src = open(_HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(?:int|size_t|long long|const char\*)\s+(\w+)\s*\(", src)))


def lib() -> ctypes.CDLL:
    """Loads libslimspec.so (built by ``_build.build()``); raises if absent."""
    global _LIB
    if _LIB is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(
                "libslimspec.so is not built; run "
                "`python -c 'import __graft_entry__ as g; g.build()'` first")
        l = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = l
    return _LIB


# ------------------------------------------------------------------ helpers --
def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SS_BF16
    if t.dtype == torch.float32:
        return SS_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int, where: str):
    if status != SS_OK:
        raise SlimspecError(status, where)


def _workspace(nbytes: int, device, workspace):
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small")
        return workspace
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def slimspec_head_workspace_size(M, d, r, V, dtype_code) -> int:
    return int(lib().slimspec_head_workspace_size(M, d, r, V, dtype_code))


def specvocab_head_workspace_size(M, d, d_prime, V, k) -> int:
    return int(lib().specvocab_head_workspace_size(M, d, d_prime, V, k))


def spec_verify_workspace_size(B, gamma, V, temperature) -> int:
    return int(lib().spec_verify_workspace_size(B, gamma, V, float(temperature)))


def spec_verify_lowrank_workspace_size(B, gamma, V, r) -> int:
    return int(lib().spec_verify_lowrank_workspace_size(B, gamma, V, r))


def trimmed_head_workspace_size(M, d, V_kept) -> int:
    return int(lib().trimmed_head_workspace_size(M, d, V_kept))


def ss_topk_workspace_size(M, V, k) -> int:
    return int(lib().ss_topk_workspace_size(M, V, k))


# -------------------------------------------------------------- entry points --
def slimspec_head_forward(hidden, w_down, w_up, temperature=0.0, uniforms=None, *, seed=0,
                          offset=0, want_stats=True, want_z=False, want_logits=False,
                          workspace=None, out=None, stream=None) -> dict:
    """Low-rank head h -> h W_down^T -> . W_up^T fused with the row reduction.

    hidden (M, d), w_down (r, d), w_up (V, r): same dtype (bf16 or fp32), CUDA.
    Sampling (temperature > 0) draws row m's uniform from Philox4x32-10 at
    (seed, offset, row m, slot 0), or takes uniforms[m] when given.
    Returns a dict with 'tokens' (M int32) and, as requested, 'logprob',
    'row_max', 'lse' (M float32), 'z' (M, r) and 'logits' (M, V float32).
    ``out`` may supply preallocated output tensors under the same keys.
    """
    M, d = hidden.shape
    r, d2 = w_down.shape
    V, r2 = w_up.shape
    if d2 != d or r2 != r or w_down.dtype != hidden.dtype or w_up.dtype != hidden.dtype:
        raise ValueError("shape or dtype mismatch")
    code = _dtype_code(hidden)
    dev = hidden.device
    o = dict(out or {})
    if "tokens" not in o:
        o["tokens"] = torch.empty(M, dtype=torch.int32, device=dev)
    if want_stats:
        for k in ("logprob", "row_max", "lse"):
            if k not in o:
                o[k] = torch.empty(M, dtype=torch.float32, device=dev)
    if want_z:
        if "z" not in o:
            o["z"] = torch.empty(M, r, dtype=hidden.dtype, device=dev)
    if want_logits:
        if "logits" not in o:
            o["logits"] = torch.empty(M, V, dtype=torch.float32, device=dev)
    nbytes = slimspec_head_workspace_size(M, d, r, V, code)
    ws = _workspace(nbytes, dev, workspace)
    st = lib().slimspec_head_forward(
        _ptr(hidden), _ptr(w_down), _ptr(w_up), M, d, r, V, code, float(temperature), int(seed),
        int(offset), _ptr(uniforms), _ptr(o["tokens"]), _ptr(o.get("logprob")),
        _ptr(o.get("row_max")),
        _ptr(o.get("lse")), _ptr(o.get("z")), _ptr(o.get("logits")), _ptr(ws), ws.numel(),
        _stream(stream))
    _check(st, "slimspec_head_forward")
    return o


def specvocab_head_forward(hidden, w_down, w_vocab, u_full, k, temperature=0.0, uniforms=None,
                           *, seed=0, offset=0, want_topk=True, want_prob=False,
                           want_logits=False, want_scores=False, workspace=None, out=None,
                           stream=None) -> dict:
    """SpecVocab head: router scores, top-k, exact candidate logits, draw (bf16).

    Returns 'tokens' and, as requested, 'topk_idx' (M, k) ascending ids,
    'topk_prob' (M, k) q over them, 'topk_logits' (M, k) their exact logits and
    'scores' (M, V) the router's approximate scores."""
    M, d = hidden.shape
    dp, d2 = w_down.shape
    V, dp2 = w_vocab.shape
    V2, d3 = u_full.shape
    if d2 != d or dp2 != dp or V2 != V or d3 != d:
        raise ValueError("shape mismatch")
    dev = hidden.device
    o = dict(out or {})
    if "tokens" not in o:
        o["tokens"] = torch.empty(M, dtype=torch.int32, device=dev)
    if want_topk:
        if "topk_idx" not in o:
            o["topk_idx"] = torch.empty(M, k, dtype=torch.int32, device=dev)
    if want_prob:
        if "topk_prob" not in o:
            o["topk_prob"] = torch.empty(M, k, dtype=torch.float32, device=dev)
    if want_logits:
        if "topk_logits" not in o:
            o["topk_logits"] = torch.empty(M, k, dtype=torch.float32, device=dev)
    if want_scores:
        if "scores" not in o:
            o["scores"] = torch.empty(M, V, dtype=torch.float32, device=dev)
    nbytes = specvocab_head_workspace_size(M, d, dp, V, k)
    ws = _workspace(nbytes, dev, workspace)
    st = lib().specvocab_head_forward(
        _ptr(hidden), _ptr(w_down), _ptr(w_vocab), _ptr(u_full), M, d, dp, V, k,
        float(temperature), int(seed), int(offset), _ptr(uniforms), _ptr(o["tokens"]),
        _ptr(o.get("topk_idx")), _ptr(o.get("topk_prob")), _ptr(o.get("topk_logits")),
        _ptr(o.get("scores")), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "specvocab_head_forward")
    return o


def ss_topk_rows(scores, k, *, out=None, stream=None):
    """Top-k ids (ascending, ties to the lowest id) of each row of fp32 scores."""
    M, V = scores.shape
    o = out if out is not None else torch.empty(M, k, dtype=torch.int32, device=scores.device)
    nbytes = ss_topk_workspace_size(M, V, k)
    ws = _workspace(nbytes, scores.device, None)
    st = lib().ss_topk_rows(_ptr(scores), M, V, k, _ptr(o), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "ss_topk_rows")
    return o


def spec_verify(target_logits, draft_logits, draft_tokens, temperature=0.0, uniforms=None, *,
                seed=0, offset=0, lazy=False, workspace=None, out=None, stream=None) -> dict:
    """Verification of B sequences: target (B, g+1, V), draft (B, g, V) fp32,
    draft_tokens (B, g) int32.  Sampling draws u[b, j] from Philox4x32-10 at
    (seed, offset, row b, slot j), or takes uniforms (B, g+1) fp32 when given.
    lazy=True reads the rows position by position, only for the sequences
    still kept (spec_verify_lazy); the results are the same."""
    B, g1, V = target_logits.shape
    gamma = g1 - 1
    dev = target_logits.device
    o = dict(out or {})
    if "tokens" not in o:
        o["tokens"] = torch.empty(B, g1, dtype=torch.int32, device=dev)
    if "num_accepted" not in o:
        o["num_accepted"] = torch.empty(B, dtype=torch.int32, device=dev)
    nbytes = spec_verify_workspace_size(B, gamma, V, temperature)
    ws = _workspace(nbytes, dev, workspace)
    fn = lib().spec_verify_lazy if lazy else lib().spec_verify
    st = fn(
        _ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens), B, gamma, V,
        float(temperature), int(seed), int(offset), _ptr(uniforms), _ptr(o["tokens"]),
        _ptr(o["num_accepted"]), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "spec_verify_lazy" if lazy else "spec_verify")
    return o


def spec_verify_lowrank(target_logits, z, w_up, draft_logprob, draft_lse, draft_tokens,
                        temperature, uniforms=None, *, seed=0, offset=0, position_major=True,
                        workspace=None, out=None, stream=None) -> dict:
    """Sampling verification of B sequences with the draft side from the
    low-rank head: target (B, g+1, V) fp32; z (g*B, r) bf16 in position-major
    order (row j*B + b: g head calls of B rows), or (B*g, r) sequence-major
    with position_major=False; draft_logprob, draft_lse fp32 in the same
    order; w_up (V, r) bf16; draft_tokens int32 in the same order;
    uniforms (B, g+1), or None for the Philox stream at (seed, offset)."""
    B, g1, V = target_logits.shape
    gamma = g1 - 1
    r = z.shape[-1]
    dev = target_logits.device
    ss, sp = (1, B) if position_major else (gamma, 1)
    o = dict(out or {})
    if "tokens" not in o:
        o["tokens"] = torch.empty(B, g1, dtype=torch.int32, device=dev)
    if "num_accepted" not in o:
        o["num_accepted"] = torch.empty(B, dtype=torch.int32, device=dev)
    nbytes = spec_verify_lowrank_workspace_size(B, gamma, V, r)
    ws = _workspace(nbytes, dev, workspace)
    st = lib().spec_verify_lowrank(
        _ptr(target_logits), _ptr(z), _ptr(w_up), _ptr(draft_logprob), _ptr(draft_lse), ss, sp,
        r, _ptr(draft_tokens), B, gamma, V, float(temperature), int(seed), int(offset),
        _ptr(uniforms),
        _ptr(o["tokens"]), _ptr(o["num_accepted"]), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "spec_verify_lowrank")
    return o


def trimmed_head_forward(hidden, w_kept, kept_ids, temperature=0.0, uniforms=None, *,
                         seed=0, offset=0, want_stats=True, workspace=None, out=None,
                         stream=None) -> dict:
    """Dense head over the kept vocabulary rows w_kept (V_kept, d) bf16 with
    their ids kept_ids (V_kept,) int32; hidden (M, d) bf16.  Returns 'tokens'
    (vocabulary ids) and, with want_stats, 'logprob', 'row_max', 'lse' over
    the kept set."""
    M, d = hidden.shape
    Vk = w_kept.shape[0]
    dev = hidden.device
    o = dict(out or {})
    if "tokens" not in o:
        o["tokens"] = torch.empty(M, dtype=torch.int32, device=dev)
    if want_stats:
        for k in ("logprob", "row_max", "lse"):
            if k not in o:
                o[k] = torch.empty(M, dtype=torch.float32, device=dev)
    nbytes = trimmed_head_workspace_size(M, d, Vk)
    ws = _workspace(nbytes, dev, workspace)
    st = lib().trimmed_head_forward(
        _ptr(hidden), _ptr(w_kept), _ptr(kept_ids), M, d, Vk, float(temperature), int(seed),
        int(offset), _ptr(uniforms),
        _ptr(o["tokens"]), _ptr(o.get("logprob")), _ptr(o.get("row_max")), _ptr(o.get("lse")),
        _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "trimmed_head_forward")
    return o


def ss_philox_uniforms(seed, offset, rows, slots, *, device=None, stream=None):
    """The (rows, slots) float32 uniforms a sampling call draws at (seed,
    offset) when given no uniforms of its own, computed on the device."""
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    o = torch.empty(rows, slots, dtype=torch.float32, device=dev)
    _check(lib().ss_philox_uniforms(int(seed), int(offset), rows, slots, _ptr(o),
                                    _stream(stream)), "ss_philox_uniforms")
    return o


def ss_philox4x32_10(blocks, *, stream=None):
    """Raw Philox4x32-10: blocks (n, 6) int32/uint32 words (counter c0..c3, key
    k0, k1) on a CUDA device -> (n, 4) output words as int32 (bit patterns)."""
    n = blocks.shape[0]
    if blocks.dim() != 2 or blocks.shape[1] != 6 or blocks.element_size() != 4:
        raise ValueError("blocks must be (n, 6) 32-bit words")
    o = torch.empty(n, 4, dtype=torch.int32, device=blocks.device)
    _check(lib().ss_philox4x32_10(_ptr(blocks), n, _ptr(o), _stream(stream)), "ss_philox4x32_10")
    return o


N_KERNEL_KINDS = 14


def launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(lib().ss_launch_count())


def profile_start():
    _check(lib().ss_profile_start(), "ss_profile_start")


def profile_stop():
    _check(lib().ss_profile_stop(), "ss_profile_stop")


def profile_read(keep: bool = False) -> dict:
    """{kernel name: (timed launches, summed ms)} of the recorded launches;
    the records are dropped unless ``keep``."""
    n = N_KERNEL_KINDS
    launches = (ctypes.c_int * n)()
    ms = (ctypes.c_double * n)()
    _check(lib().ss_profile_read(ctypes.cast(launches, ctypes.c_void_p),
                                 ctypes.cast(ms, ctypes.c_void_p), n, 1 if keep else 0),
           "ss_profile_read")
    return {lib().ss_profile_kind_name(k).decode(): (launches[k], ms[k])
            for k in range(n) if launches[k]}


def ss_set_wait_limit_ns(limit_ns: int):
    """Limit of the kernels' pipeline waits on the current device (default 1 s)."""
    _check(lib().ss_set_wait_limit_ns(int(limit_ns)), "ss_set_wait_limit_ns")


def ss_set_stall_test(on: bool):
    """Test switch: the tensor-core up-projection waits on a barrier nothing
    arrives on, so its calls time out (SS_ERR_TIMEOUT) instead of running."""
    _check(lib().ss_set_stall_test(1 if on else 0), "ss_set_stall_test")


def ss_get_device_error(stream=None) -> int:
    """Synchronises the stream, then reads and clears the device error word."""
    return int(lib().ss_get_device_error(_stream(stream)))
