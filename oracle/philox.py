"""Oracle for the counter-based uniforms the sampling calls draw.

Test infrastructure only (see the package docstring).

The Explainer's section "为什么答案不会变" needs one uniform per accept test
and one per final draw; the SlimSpec head and the SpecVocab head need one per
drafted row.  When the caller does not pass its own uniforms, both sides of
this project draw them from one published counter-based generator, each side
with its own code:

Philox4x32-10 -- J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw,
"Parallel Random Numbers: As Easy as 1, 2, 3", SC'11, section 4 (the Philox
S-box).  Written here from that definition, not from any library's source:

* state: four 32-bit counter words (c0, c1, c2, c3) and two key words
  (k0, k1);
* one round: multiply c0 by M0 and c2 by M1 as full 64-bit products, then
      c0' = hi(M1*c2) ^ c1 ^ k0      c1' = lo(M1*c2)
      c2' = hi(M0*c0) ^ c3 ^ k1      c3' = lo(M0*c0)
* the key of round i+1 is the key of round i plus the Weyl constants
  (W0, W1) modulo 2^32 (the first round uses the key as given);
* ten rounds.

Multipliers and Weyl constants are the paper's for N = 4, W = 32:
M0 = 0xD2511F53, M1 = 0xCD9E8D57, W0 = 0x9E3779B9 (golden ratio), W1 = 0xBB67AE85
(sqrt(3) - 1).

Draw layout (this project's choice; the articles name no generator):
    key     = (seed mod 2^32, seed >> 32)
    counter = (row, slot, offset mod 2^32, offset >> 32)
    u       = (first output word >> 8) * 2^-24        in [0, 1), exact in fp32
Rows and slots: a head call's row m uses (row m, slot 0); a verification's
sequence b uses (row b, slot j) for its accept test at drafted position j and
(row b, slot gamma) for its final draw -- the same (row, slot) that index a
caller-supplied uniforms array of shape (rows, slots).  Callers advance
`offset` between calls so that no two calls share a counter.
"""
from __future__ import annotations

import numpy as np

PHILOX_M4x32 = (0xD2511F53, 0xCD9E8D57)
PHILOX_W32 = (0x9E3779B9, 0xBB67AE85)
ROUNDS = 10
_MASK32 = 0xFFFFFFFF


def philox_block(counter, key, mult=PHILOX_M4x32, weyl=PHILOX_W32, bits: int = 32,
                 rounds: int = ROUNDS):
    """One Philox4xW block of plain Python integers (any word width W).

    counter: four words, key: two words, each < 2**bits.  Returns the four
    output words.  With the default arguments this is Philox4x32-10; other
    widths take their own multipliers and Weyl constants.
    """
    mask = (1 << bits) - 1
    c0, c1, c2, c3 = (int(v) & mask for v in counter)
    k0, k1 = (int(v) & mask for v in key)
    for i in range(rounds):
        if i > 0:  # the key schedule: a Weyl sequence, bumped between rounds
            k0 = (k0 + weyl[0]) & mask
            k1 = (k1 + weyl[1]) & mask
        p0 = mult[0] * c0
        p1 = mult[1] * c2
        c0, c1, c2, c3 = ((p1 >> bits) ^ c1 ^ k0, p1 & mask, (p0 >> bits) ^ c3 ^ k1, p0 & mask)
    return c0, c1, c2, c3


def philox4x32_10(counters, keys) -> np.ndarray:
    """Philox4x32-10 over arrays: counters (..., 4), keys (..., 2) of values
    below 2**32 (broadcast against each other).  Returns (..., 4) uint64 words.

    The same rounds as philox_block, with numpy uint64 arithmetic: a product of
    two 32-bit words is exact below 2**64."""
    ctr = np.asarray(counters, dtype=np.uint64)
    key = np.asarray(keys, dtype=np.uint64)
    shape = np.broadcast_shapes(ctr.shape[:-1], key.shape[:-1])
    ctr = np.broadcast_to(ctr, shape + (4,))
    key = np.broadcast_to(key, shape + (2,))
    m32 = np.uint64(_MASK32)
    s32 = np.uint64(32)
    c0, c1, c2, c3 = (ctr[..., i].copy() for i in range(4))
    k0, k1 = key[..., 0].copy(), key[..., 1].copy()
    mul0, mul1 = np.uint64(PHILOX_M4x32[0]), np.uint64(PHILOX_M4x32[1])
    for i in range(ROUNDS):
        if i > 0:
            k0 = (k0 + np.uint64(PHILOX_W32[0])) & m32
            k1 = (k1 + np.uint64(PHILOX_W32[1])) & m32
        p0 = mul0 * c0
        p1 = mul1 * c2
        c0, c1, c2, c3 = ((p1 >> s32) ^ c1 ^ k0, p1 & m32, (p0 >> s32) ^ c3 ^ k1, p0 & m32)
    return np.stack([c0, c1, c2, c3], axis=-1)


def draw_counter_key(seed: int, offset: int, row, slot):
    """The (counter, key) words of draw (row, slot) of call (seed, offset)."""
    seed, offset = int(seed), int(offset)
    if not (0 <= seed < 1 << 64 and 0 <= offset < 1 << 64):
        raise ValueError("seed and offset are 64-bit unsigned")
    row = np.asarray(row, dtype=np.uint64)
    slot = np.asarray(slot, dtype=np.uint64)
    row, slot = np.broadcast_arrays(row, slot)
    ctr = np.stack([row, slot, np.full_like(row, offset & _MASK32),
                    np.full_like(row, offset >> 32)], axis=-1)
    key = np.array([seed & _MASK32, seed >> 32], dtype=np.uint64)
    return ctr, key


def uniform_at(seed: int, offset: int, row: int, slot: int) -> float:
    """One draw, u(seed, offset, row, slot), through the plain-integer block."""
    seed, offset = int(seed), int(offset)
    if not (0 <= seed < 1 << 64 and 0 <= offset < 1 << 64):
        raise ValueError("seed and offset are 64-bit unsigned")
    x0 = philox_block((row, slot, offset & _MASK32, offset >> 32),
                      (seed & _MASK32, seed >> 32))[0]
    return (x0 >> 8) * 2.0 ** -24


def uniforms(seed: int, offset: int, rows: int, slots: int) -> np.ndarray:
    """The (rows, slots) uniforms of one call: u[row, slot] in [0, 1), float64
    (every value a multiple of 2**-24, so exact in fp32 as well)."""
    r, s = np.meshgrid(np.arange(rows, dtype=np.uint64), np.arange(slots, dtype=np.uint64),
                       indexing="ij")
    ctr, key = draw_counter_key(seed, offset, r, s)
    x0 = philox4x32_10(ctr, key)[..., 0]
    return (x0 >> np.uint64(8)).astype(np.float64) * 2.0 ** -24
