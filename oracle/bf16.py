"""Round-to-nearest-even onto the bf16 grid, from float64.

bf16 keeps 8 significant bits (1 implicit + 7 stored) and float32's exponent
range.  The rounding is done in one step from the float64 value, never through
float32, so that it is a single correct rounding.

Test infrastructure only (see the package docstring).
"""
import numpy as np

_BF16_SIG_BITS = 8          # significant bits including the implicit one
_BF16_MIN_EXP = -125        # frexp exponent of the smallest normal (2**-126)
_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def round_to_bf16(x) -> np.ndarray:
    """Nearest bf16 value of each float64 element, ties to the even significand.

    x = f * 2**e with f in [0.5, 1); the bf16 spacing at x is 2**(e - 8) for
    normal numbers and 2**(-133) in the subnormal range.  Dividing by the
    spacing gives an exact float64 number whose nearest-even integer (np.rint)
    is the rounded significand.  Values beyond the largest finite bf16 become
    +-inf, as IEEE rounding does.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e, _BF16_MIN_EXP)
    spacing = np.ldexp(1.0, e - _BF16_SIG_BITS)
    y = np.rint(x / spacing) * spacing
    # overflow: anything whose rounded magnitude exceeds the largest bf16
    y = np.where(np.abs(y) > _BF16_MAX, np.copysign(np.inf, x), y)
    return y
