"""bfloat16 rounding for the oracle (test infrastructure only).

bfloat16 keeps the float32 exponent (8 bits) and 7 explicit fraction bits, so a
finite value in [2**E, 2**(E+1)) lies on a grid of spacing 2**(E-7), and below
the smallest normal 2**-126 the grid spacing stays 2**-133.  Rounding is IEEE
round-to-nearest, ties to the even grid point, applied once to the exact value
(float64 in, no intermediate float32 rounding).  Values at or above the largest
finite bfloat16 plus half a spacing overflow to infinity.

Every activation on the boundary path is stored in bf16 ("第 7 课：序列并行 SP",
"具体演示与数值推演": BF16, 2 bytes per element).
"""
import numpy as np

BF16_MAX = float.fromhex("0x1.fep127")   # (2 - 2**-7) * 2**127
_SUBNORMAL_EXP = -133                    # spacing below 2**-126


def bf16_round(x):
    """Round each value of ``x`` to the nearest bfloat16 (ties to even).

    Returns float32 (every bfloat16 is exactly representable in float32).
    """
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    finite = np.isfinite(ax)
    safe = np.where(finite, ax, 0.0)
    _, e = np.frexp(safe)                 # safe = m * 2**e with 0.5 <= m < 1
    grid_exp = np.maximum((e - 1) - 7, _SUBNORMAL_EXP)
    steps = np.rint(np.ldexp(safe, -grid_exp))   # rint: ties go to even
    mag = np.ldexp(steps, grid_exp)
    mag = np.where(mag > BF16_MAX, np.inf, mag)
    mag = np.where(finite, mag, ax)       # inf stays inf, nan stays nan
    return np.copysign(mag, x).astype(np.float32)


def bits_to_f32(bits):
    """bfloat16 bit patterns (uint16 / int16) -> float32 values."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32)
    return (b << np.uint32(16)).view(np.float32)


def f32_to_bits(values):
    """float32 values that are exact bfloat16 numbers -> uint16 bit patterns."""
    v = np.ascontiguousarray(np.asarray(values, dtype=np.float32))
    u = v.view(np.uint32)
    if np.any(u & np.uint32(0xFFFF)):
        raise ValueError("value is not an exact bfloat16 number")
    return (u >> np.uint32(16)).astype(np.uint16)


def order_key(bits):
    """Map bf16 bit patterns to integers that are monotone in the value.

    Adjacent bfloat16 numbers differ by 1 in this key and +0 / -0 share a key,
    so ``|key(a) - key(b)|`` counts units in the last place between a and b.
    """
    b = np.asarray(bits).astype(np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)
