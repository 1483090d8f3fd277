"""bfloat16 rounding for the oracle (test infrastructure only).

bfloat16 is the IEEE-754 binary32 layout cut to its top 16 bits: 1 sign bit,
8 exponent bits (bias 127), 7 stored fraction bits.  A finite float64 x is
rounded here straight to the nearest bfloat16 value, ties to the even
significand, with gradual underflow below 2**-126 (quantum 2**-133) and
overflow to infinity, then encoded as 16 bits.  Rounding straight from fp64
avoids the double rounding of an fp64 -> fp32 -> bf16 chain.
"""

import numpy as np

_MIN_EXP = -133  # quantum of the subnormal range: 2**-126 * 2**-7


def round_to_bf16(x):
    """Round float64 values to the nearest bfloat16 value (ties to even).

    Returns float64 values that are exactly representable in bfloat16.
    NaN and +-inf pass through unchanged.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    fin = np.isfinite(x) & (x != 0.0)
    xf = x[fin]
    _, e = np.frexp(xf)                       # xf = f * 2**e, 0.5 <= |f| < 1
    q_exp = np.maximum(e - 8, _MIN_EXP)       # 8 significant bits
    q = np.ldexp(1.0, q_exp)
    r = np.rint(xf / q) * q                   # np.rint rounds half to even
    r[np.abs(r) >= np.ldexp(1.0, 128)] = np.inf * np.sign(r[np.abs(r) >= np.ldexp(1.0, 128)])
    out[fin] = r
    return out


def bf16_bits(x):
    """Encode float64 values as bfloat16 bit patterns (uint16), rounding RNE."""
    r = round_to_bf16(x)
    with np.errstate(over="ignore"):
        f32 = r.astype(np.float32)            # exact: r is bf16-representable
    bits = (f32.view(np.uint32) >> 16).astype(np.uint16)
    nan = np.isnan(r)
    bits[nan] = 0x7FC0
    return bits


def bits_to_f64(bits):
    """Decode bfloat16 bit patterns (uint16) to float64, exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def ordered(bits):
    """Map bf16 bit patterns to integers that are monotone in the value.

    +0 and -0 both map to 0, so the distance between adjacent representable
    values is 1 across the whole line.
    """
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def ulp_distance(bits_a, bits_b):
    """Number of bfloat16 steps between two bit patterns (absolute)."""
    return np.abs(ordered(bits_a) - ordered(bits_b))
