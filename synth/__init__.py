"""Seeded synthetic inputs for the drafter head and the verifier.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no projection, no reduction, no sampling, no acceptance
rule).  Both the CUDA path (through the tests and the benchmark) and the CPU
oracle read their inputs from here, so that the two see identical values.

Conventions
-----------
* Every bf16 tensor is returned as a float32 array whose values are exactly
  representable in bf16 (fp32 values rounded to nearest-even on the 16-bit
  boundary).  float32 is a lossless carrier for bf16 values; ``bf16_bits`` gives
  the 16-bit pattern a device upload needs.
* Weights are iid N(0, 1/fan_in); hidden states are iid N(0, 1).
* Uniforms are float32 multiples of 2**-24 in [0, 1) (24 random bits), so they
  are exact in every precision either side computes in.
* Zipf-like logit rows: -1.1 * ln(rank) over a fresh random permutation of the
  ranks 1..V for every row, plus N(0, 0.5**2) noise.  They stand in for real LM
  output distributions on the chat/code/math benchmarks the articles measure
  on; no benchmark item or trained weight is used or reproduced.

The named presets at the bottom carry the five workload shapes.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "round_f32_to_bf16", "bf16_bits", "normal", "uniforms", "head_inputs",
    "specvocab_inputs", "logit_rows", "verify_logits", "Preset", "PRESETS",
]


# ----------------------------------------------------------------------------
# bf16 carrier helpers (input quantisation only)
# ----------------------------------------------------------------------------
def round_f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 value (ties to even); float32 out."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    bits = ((bits + 0x7FFF + lsb) >> 16) << 16
    return bits.astype(np.uint32).view(np.float32)


def bf16_bits(x_bf16_valued_f32: np.ndarray) -> np.ndarray:
    """16-bit patterns of float32 arrays that already hold bf16 values."""
    x = np.ascontiguousarray(x_bf16_valued_f32, dtype=np.float32)
    bits = x.view(np.uint32)
    if np.any(bits & 0xFFFF):
        raise ValueError("array holds values that are not bf16")
    return (bits >> 16).astype(np.uint16)


# ----------------------------------------------------------------------------
# primitive draws
# ----------------------------------------------------------------------------
def normal(rng: np.random.Generator, shape, std: float, dtype: str) -> np.ndarray:
    """iid N(0, std**2) as float32, rounded to bf16 values when dtype == 'bf16'."""
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if dtype == "bf16":
        return round_f32_to_bf16(x)
    if dtype == "f32":
        return x
    raise ValueError(dtype)


def uniforms(rng: np.random.Generator, shape) -> np.ndarray:
    """float32 uniforms in [0, 1) on the 2**-24 grid."""
    bits = rng.integers(0, 1 << 24, size=shape, dtype=np.int64)
    return (bits.astype(np.float64) * 2.0 ** -24).astype(np.float32)


# ----------------------------------------------------------------------------
# drafter heads
# ----------------------------------------------------------------------------
def head_inputs(seed: int, M: int, d: int, r: int, V: int, dtype: str) -> dict:
    """Hidden states and the two low-rank factors of the drafter head.

    hidden (M, d), w_down (r, d), w_up (V, r); all N(0, 1/fan_in) except hidden.
    """
    rng = np.random.default_rng(seed)
    w_down = normal(rng, (r, d), 1.0 / np.sqrt(d), dtype)
    w_up = normal(rng, (V, r), 1.0 / np.sqrt(r), dtype)
    hidden = normal(rng, (M, d), 1.0, dtype)
    return {"hidden": hidden, "w_down": w_down, "w_up": w_up}


def dense_head_inputs(seed: int, M: int, d: int, V: int, dtype: str) -> dict:
    """Hidden states and a full V x d head, N(0, 1/d)."""
    rng = np.random.default_rng(seed)
    w = normal(rng, (V, d), 1.0 / np.sqrt(d), dtype)
    hidden = normal(rng, (M, d), 1.0, dtype)
    return {"hidden": hidden, "w": w}


def specvocab_inputs(seed: int, M: int, d: int, d_prime: int, V: int,
                     dtype: str = "bf16") -> dict:
    """Router factors W_down (d', d), W_vocab (V, d'), full head U (V, d), hidden."""
    rng = np.random.default_rng(seed)
    w_down = normal(rng, (d_prime, d), 1.0 / np.sqrt(d), dtype)
    w_vocab = normal(rng, (V, d_prime), 1.0 / np.sqrt(d_prime), dtype)
    u_full = normal(rng, (V, d), 1.0 / np.sqrt(d), dtype)
    hidden = normal(rng, (M, d), 1.0, dtype)
    return {"hidden": hidden, "w_down": w_down, "w_vocab": w_vocab, "u_full": u_full}


# ----------------------------------------------------------------------------
# verifier logits
# ----------------------------------------------------------------------------
def logit_rows(rng: np.random.Generator, n_rows: int, V: int, kind: str,
               sigma: float = 2.0) -> np.ndarray:
    """n_rows x V float32 target logits.

    kind='normal': iid N(0, sigma**2).
    kind='zipf'  : -1.1*ln(rank) over a per-row random permutation + N(0, 0.25).
    """
    if kind == "normal":
        return normal(rng, (n_rows, V), sigma, "f32")
    if kind != "zipf":
        raise ValueError(kind)
    out = np.empty((n_rows, V), dtype=np.float32)
    base = (-1.1 * np.log(np.arange(1, V + 1, dtype=np.float64))).astype(np.float32)
    for i in range(n_rows):
        perm = rng.permutation(V)
        out[i] = base[perm]
    out += normal(rng, (n_rows, V), 0.5, "f32")
    return out


def verify_logits(seed: int, B: int, gamma: int, V: int, kind: str,
                  draft_sigma: float = 1.0, target_sigma: float = 2.0) -> dict:
    """Target rows (B, gamma+1, V), draft rows (B, gamma, V) and uniforms.

    draft = target[:, :gamma] + N(0, draft_sigma**2).  ``u_draft`` (B, gamma) are
    the uniforms a drafter would use to pick its tokens; ``u_verify``
    (B, gamma+1) are the verifier's: one accept test per drafted position and
    one for the residual / bonus draw.
    """
    rng = np.random.default_rng(seed)
    target = logit_rows(rng, B * (gamma + 1), V, kind, target_sigma)
    target = target.reshape(B, gamma + 1, V)
    noise = normal(rng, (B, gamma, V), draft_sigma, "f32")
    draft = (target[:, :gamma, :] + noise).astype(np.float32)
    return {
        "target": np.ascontiguousarray(target),
        "draft": np.ascontiguousarray(draft),
        "u_draft": uniforms(rng, (B, gamma)),
        "u_verify": uniforms(rng, (B, gamma + 1)),
    }


# ----------------------------------------------------------------------------
# workload presets (shapes of the five configurations)
# ----------------------------------------------------------------------------
@dataclass(frozen=True)
class Preset:
    name: str
    d: int
    r: int
    V: int
    dtype: str
    M: int
    gamma: int
    B: int
    temperature: float
    logits: str = "zipf"
    draft_sigma: float = 1.0
    d_prime: int = 0
    k: int = 0
    seed: int = 0
    extra: dict = field(default_factory=dict)


PRESETS = {
    # oracle-scale case: fp32, d=256, r=32, V=4096, one row, gamma=4
    "tiny": Preset("tiny", d=256, r=32, V=4096, dtype="f32", M=1, gamma=4, B=1,
                   temperature=1.0, logits="normal", draft_sigma=1.0, seed=101),
    # Llama-3.1-8B shaped head, greedy gamma=6 chain, M in {1,4,8}
    "llama8b": Preset("llama8b", d=4096, r=512, V=128256, dtype="bf16", M=8,
                      gamma=6, B=8, temperature=0.0, logits="zipf", seed=202,
                      extra={"M_list": (1, 4, 8)}),
    # GPT-OSS-20B shaped: 16 rows, T=0.7, residual resample and bonus
    "gptoss20b": Preset("gptoss20b", d=2880, r=360, V=201088, dtype="bf16", M=16,
                        gamma=6, B=16, temperature=0.7, logits="zipf", seed=303),
    # Qwen3-30B-A3B shaped: 64 sequences x gamma=4 = 256 draft rows, T=1
    "qwen30b": Preset("qwen30b", d=2048, r=256, V=151936, dtype="bf16", M=256,
                      gamma=4, B=64, temperature=1.0, logits="zipf", seed=404,
                      extra={"draft_sigmas": (0.5, 1.0, 2.0)}),
    # SpecVocab dynamic vocabulary at the Qwen3-8B shape
    "specvocab8b": Preset("specvocab8b", d=4096, r=0, V=151936, dtype="bf16",
                          M=32, gamma=6, B=32, temperature=1.0, d_prime=256,
                          k=2048, seed=505),
}
