"""The C ABI without a GPU: the library builds and loads, exports every symbol
the header declares, sizes workspaces, and rejects bad arguments on the host
before launching anything (fake device pointers are never dereferenced here:
each call below fails validation first)."""
import ctypes
import math

import pytest

import __graft_entry__
import speculative_decoding_drafter_slimspec_gb300 as ss


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return ss.lib()


FAKE = ctypes.c_void_p(1 << 20)      # 16-byte aligned, never dereferenced
MISAL = ctypes.c_void_p((1 << 20) + 8)
MISAL4 = ctypes.c_void_p((1 << 20) + 2)  # not even 4-byte aligned
NULL = None


def test_every_declared_symbol_is_exported(lib):
    names = ss.header_functions()
    assert set(names) == set(ss._SIGS)
    for n in names:
        assert hasattr(lib, n), n
    assert lib.ss_version() == 200


def test_status_strings(lib):
    for s in range(7):
        assert lib.ss_status_string(s).decode().startswith("SS_")
    assert lib.ss_status_string(99) == b"unknown status"


def test_workspace_sizes(lib):
    w = lib.slimspec_head_workspace_size(8, 4096, 512, 128256, ss.SS_BF16)
    # z (8 x 512 bf16) + three partial arrays of at least 8 x ceil(128256/64)
    # (one partial per 64-row vocabulary sub-tile or finer)
    assert w >= 8 * 512 * 2 + 3 * 8 * 2004 * 4
    assert lib.slimspec_head_workspace_size(-1, 4096, 512, 128256, ss.SS_BF16) == 0
    assert lib.slimspec_head_workspace_size(8, 4096, 2048, 128256, ss.SS_BF16) > 0   # tensor cores
    assert lib.slimspec_head_workspace_size(8, 8192, 8192, 128256, ss.SS_BF16) == 0  # r too wide
    assert lib.spec_verify_workspace_size(16, 6, 201088, ctypes.c_float(0.7)) > 0
    assert lib.spec_verify_workspace_size(16, 0, 201088, ctypes.c_float(0.7)) == 0
    assert lib.specvocab_head_workspace_size(32, 4096, 256, 151936, 2048) >= 32 * 151936 * 4
    assert lib.specvocab_head_workspace_size(32, 4096, 256, 151936, 0) == 0


def _head(lib, **kw):
    a = dict(hidden=FAKE, w_down=FAKE, w_up=FAKE, M=2, d=64, r=32, V=100, dtype=ss.SS_BF16,
             T=0.0, seed=0, offset=0, u=NULL, tok=FAKE, lp=NULL, mx=NULL, lse=NULL, z=NULL,
             logits=NULL, ws=FAKE, wsb=1 << 20, stream=NULL)
    a.update(kw)
    return lib.slimspec_head_forward(a["hidden"], a["w_down"], a["w_up"], a["M"], a["d"], a["r"],
                                     a["V"], a["dtype"], a["T"], a["seed"], a["offset"], a["u"],
                                     a["tok"], a["lp"], a["mx"], a["lse"], a["z"], a["logits"],
                                     a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("dtype,r,M,ok", [
    ("bf16", 1024, 300, True), ("bf16", 1032, 300, False),  # r <= 1024 at any M
    ("bf16", 2048, 40, True), ("bf16", 2048, 41, False),    # beyond: z must fit in smem
    ("bf16", 4096, 16, True), ("bf16", 4096, 17, False), ("bf16", 4104, 1, False),
    ("f32", 256, 8, True), ("f32", 260, 8, False), ("f32", 512, 8, False),
])
def test_head_supported_shapes(dtype, r, M, ok):
    """The shape limits the header states, through the workspace query (0 =
    unsupported) on the host."""
    code = ss.SS_BF16 if dtype == "bf16" else ss.SS_F32
    assert (ss.slimspec_head_workspace_size(M, 64, r, 128256, code) > 0) == ok


@pytest.mark.parametrize("call,ok", [
    (lambda: ss.specvocab_head_workspace_size(4, 4096, 1024, 5000, 2048), True),
    (lambda: ss.specvocab_head_workspace_size(4, 4096, 1032, 5000, 2048), False),  # d' <= 1024
    (lambda: ss.specvocab_head_workspace_size(4, 4104, 256, 5000, 2048), False),   # d <= 4096
    (lambda: ss.specvocab_head_workspace_size(4, 4096, 256, 5000, 4096), True),
    (lambda: ss.specvocab_head_workspace_size(4, 4096, 256, 5000, 4097), False),   # k <= 4096
    (lambda: ss.specvocab_head_workspace_size(4, 4096, 256, 3000, 3001), False),   # k <= V
    (lambda: ss.trimmed_head_workspace_size(16, 4096, 32768), True),
    (lambda: ss.trimmed_head_workspace_size(17, 4096, 32768), False),  # h must fit beside W
    (lambda: ss.trimmed_head_workspace_size(8, 4104, 32768), False),   # d <= 4096
    (lambda: ss.spec_verify_workspace_size(8, 32, 1000, 1.0), True),
    (lambda: ss.spec_verify_workspace_size(8, 33, 1000, 1.0), False),  # gamma <= 32
    (lambda: ss.spec_verify_lowrank_workspace_size(8, 32, 1000, 64), True),
    (lambda: ss.spec_verify_lowrank_workspace_size(8, 33, 1000, 64), False),
])
def test_other_supported_shapes(call, ok):
    """The limits the header states for the other entry points, through their
    workspace queries (0 = unsupported) on the host."""
    assert (call() > 0) == ok


def test_head_argument_errors(lib):
    E = ss.SS_ERR_INVALID_ARG
    assert _head(lib, M=-1) == E
    assert _head(lib, d=60) == E                     # d % 8
    assert _head(lib, r=20) == E                     # r % 8 for bf16
    assert _head(lib, dtype=7) == E
    assert _head(lib, T=float("nan")) == E
    assert _head(lib, T=-0.5) == E
    assert _head(lib, T=math.inf) == E
    assert _head(lib, hidden=NULL) == E
    assert _head(lib, tok=NULL) == E
    assert _head(lib, w_up=MISAL) == E
    assert _head(lib, T=1.0, u=MISAL4) == E          # uniforms, when given, 4-byte aligned
    assert _head(lib, r=8192) == ss.SS_ERR_UNSUPPORTED
    assert _head(lib, ws=NULL) == ss.SS_ERR_WORKSPACE
    assert _head(lib, wsb=16) == ss.SS_ERR_WORKSPACE
    assert _head(lib, ws=MISAL) == ss.SS_ERR_WORKSPACE
    assert _head(lib, M=0) == ss.SS_OK               # empty batch: nothing to do


@pytest.mark.parametrize("entry", ["spec_verify", "spec_verify_lazy"])
def test_verify_argument_errors(lib, entry):
    fn = getattr(lib, entry)

    def call(B=2, g=3, V=100, T=0.0, tgt=FAKE, dr=NULL, tok=FAKE, u=NULL, ot=FAKE, on=FAKE,
             ws=FAKE, wsb=1 << 20):
        return fn(tgt, dr, tok, B, g, V, T, 0, 0, u, ot, on, ws, wsb, NULL)
    E = ss.SS_ERR_INVALID_ARG
    assert call(B=-1) == E
    assert call(g=0) == E
    assert call(g=33) == E
    assert call(V=0) == E
    assert call(T=float("nan")) == E
    assert call(tgt=NULL) == E
    assert call(T=0.7) == E                          # sampling needs draft logits
    assert call(T=0.7, dr=FAKE, u=MISAL4) == E        # uniforms, when given, aligned
    assert call(tgt=MISAL) == E
    assert call(wsb=8) == ss.SS_ERR_WORKSPACE
    assert call(B=0) == ss.SS_OK


def test_verify_lowrank_argument_errors(lib):
    def call(B=2, g=3, V=104, r=64, T=1.0, ss_=1, sp=2, tgt=FAKE, z=FAKE, w=FAKE, lp=FAKE,
             lse=FAKE, tok=FAKE, u=FAKE, ws=FAKE, wsb=1 << 24):
        return lib.spec_verify_lowrank(tgt, z, w, lp, lse, ss_, sp, r, tok, B, g, V, T, 0, 0, u,
                                       FAKE, FAKE, ws, wsb, NULL)
    E = ss.SS_ERR_INVALID_ARG
    assert call(T=0.0) == E                          # sampling only
    assert call(T=float("inf")) == E
    assert call(B=-1) == E
    assert call(g=0) == E
    assert call(g=33) == E
    assert call(r=0) == E
    assert call(ss_=-1) == E
    assert call(z=NULL) == E
    assert call(lse=NULL) == E
    assert call(u=MISAL4) == E
    assert call(z=MISAL) == E
    assert call(w=MISAL) == E
    assert call(r=12) == ss.SS_ERR_UNSUPPORTED        # r % 8 != 0: no recompute kernel
    assert call(r=520) == ss.SS_ERR_UNSUPPORTED       # r > 512
    assert call(B=300) == ss.SS_ERR_UNSUPPORTED       # B > 256
    assert call(wsb=8) == ss.SS_ERR_WORKSPACE
    assert call(B=0) == ss.SS_OK
    assert lib.spec_verify_lowrank_workspace_size(16, 6, 201088, 360) > \
        lib.spec_verify_lowrank_workspace_size(16, 6, 201088, 8)


def test_trimmed_head_argument_errors(lib):
    def call(M=2, d=64, Vk=100, T=0.0, h=FAKE, w=FAKE, ids=FAKE, u=NULL, ws=FAKE, wsb=1 << 24):
        return lib.trimmed_head_forward(h, w, ids, M, d, Vk, T, 0, 0, u, FAKE, NULL, NULL, NULL,
                                        ws, wsb, NULL)
    E = ss.SS_ERR_INVALID_ARG
    assert call(M=-1) == E
    assert call(d=12) == E
    assert call(Vk=0) == E
    assert call(ids=NULL) == E
    assert call(T=1.0, u=MISAL4) == E                # uniforms, when given, aligned
    assert call(h=MISAL) == E
    assert call(d=8192) == ss.SS_ERR_UNSUPPORTED     # beyond the tensor-core plan
    assert call(M=64, d=4096) == ss.SS_ERR_UNSUPPORTED  # h does not fit beside the stages
    assert call(wsb=8) == ss.SS_ERR_WORKSPACE
    assert call(M=0) == ss.SS_OK
    assert lib.trimmed_head_workspace_size(8, 4096, 32768) > 0


def test_specvocab_and_topk_argument_errors(lib):
    def sv(M=2, d=64, dp=16, V=100, k=10, T=0.0, u=NULL, lg=NULL, ws=FAKE, wsb=1 << 24):
        return lib.specvocab_head_forward(FAKE, FAKE, FAKE, FAKE, M, d, dp, V, k, T, 0, 0, u,
                                          FAKE, NULL, NULL, lg, NULL, ws, wsb, NULL)
    assert sv(k=0) == ss.SS_ERR_INVALID_ARG
    assert sv(k=101) == ss.SS_ERR_INVALID_ARG
    assert sv(dp=12) == ss.SS_ERR_INVALID_ARG
    assert sv(d=8192) == ss.SS_ERR_UNSUPPORTED
    assert sv(T=1.0, u=MISAL4) == ss.SS_ERR_INVALID_ARG  # misaligned uniforms
    assert sv(lg=MISAL4) == ss.SS_ERR_INVALID_ARG  # misaligned logits
    assert sv(wsb=1) == ss.SS_ERR_WORKSPACE
    assert sv(M=0) == ss.SS_OK
    assert lib.ss_topk_rows(FAKE, 2, 100, 0, FAKE, NULL, 0, NULL) == ss.SS_ERR_INVALID_ARG
    assert lib.ss_topk_rows(FAKE, 2, 100, 101, FAKE, NULL, 0, NULL) == ss.SS_ERR_INVALID_ARG
    assert lib.ss_topk_rows(NULL, 2, 100, 5, FAKE, NULL, 0, NULL) == ss.SS_ERR_INVALID_ARG
    assert lib.ss_topk_rows(FAKE, 0, 100, 5, FAKE, NULL, 0, NULL) == ss.SS_OK


def test_philox_argument_errors(lib):
    E = ss.SS_ERR_INVALID_ARG
    assert lib.ss_philox_uniforms(1, 2, -1, 4, FAKE, NULL) == E
    assert lib.ss_philox_uniforms(1, 2, 4, -1, FAKE, NULL) == E
    assert lib.ss_philox_uniforms(1, 2, 4, 4, NULL, NULL) == E
    assert lib.ss_philox_uniforms(1, 2, 4, 4, MISAL4, NULL) == E
    assert lib.ss_philox_uniforms(1, 2, 1 << 16, 1 << 15, FAKE, NULL) == ss.SS_ERR_UNSUPPORTED
    assert lib.ss_philox_uniforms(2 ** 64 - 1, 2 ** 64 - 1, 0, 7, NULL, NULL) == ss.SS_OK
    assert lib.ss_philox4x32_10(FAKE, -1, FAKE, NULL) == E
    assert lib.ss_philox4x32_10(NULL, 3, FAKE, NULL) == E
    assert lib.ss_philox4x32_10(FAKE, 3, NULL, NULL) == E
    assert lib.ss_philox4x32_10(NULL, 0, NULL, NULL) == ss.SS_OK


def test_wait_limit_range(lib):
    assert lib.ss_set_wait_limit_ns(10 ** 10 + 1) == ss.SS_ERR_INVALID_ARG
    assert lib.ss_set_wait_limit_ns(2 ** 64 - 1) == ss.SS_ERR_INVALID_ARG


def test_python_binding_refuses_cpu_tensors(lib):
    import torch
    h = torch.zeros(2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        ss.slimspec_head_forward(h, torch.zeros(32, 64, dtype=torch.bfloat16),
                                 torch.zeros(100, 32, dtype=torch.bfloat16))


def test_missing_library_fails_loudly(lib, monkeypatch):
    """No CPU fallback: with the shared library absent every call raises."""
    import torch
    monkeypatch.setattr(ss, "_LIB", None)
    monkeypatch.setattr(ss, "lib_path", lambda: "/nonexistent/libslimspec.so")
    with pytest.raises(RuntimeError, match="not built"):
        ss.lib()
    with pytest.raises(RuntimeError):
        ss.slimspec_head_workspace_size(2, 64, 32, 100, ss.SS_BF16)
    h = torch.zeros(2, 64, dtype=torch.bfloat16)
    with pytest.raises((RuntimeError, ValueError)):
        ss.slimspec_head_forward(h, torch.zeros(32, 64, dtype=torch.bfloat16),
                                 torch.zeros(100, 32, dtype=torch.bfloat16))
