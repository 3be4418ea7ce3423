"""Round-to-nearest-even conversion of fp64 values to bfloat16 (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

bfloat16 keeps 8 significant bits (1 implicit + 7 stored) and the float32
exponent range.  The packed computation rounds RoPE-rotated Q and K to bf16
before attention, so the oracle applies the same single rounding to its fp64
values.  The rounding is done directly from fp64 (no intermediate float32, so
no double rounding): ``frexp`` gives x = m * 2**e with 0.5 <= |m| < 1, and
``rint`` (ties to even) rounds m * 2**8 to an integer.
"""
import numpy as np


def round_to_bf16(x):
    """Return fp64 array whose values are ``x`` rounded to bfloat16 (RNE).

    Subnormal bfloat16 values (|x| < 2**-126) and overflow are not reached by
    the N(0,1)-scale data the oracle sees; ``rint`` still rounds them to a
    multiple of the local spacing, which is what RNE does for normals.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 256.0), e - 8)


def bf16_bits(x):
    """uint16 bit patterns of bf16 values held exactly in fp64 ``x``."""
    f32 = np.asarray(x, dtype=np.float32)
    return (f32.view(np.uint32) >> 16).astype(np.uint16)


def from_bf16_bits(bits):
    """fp64 values of uint16 bfloat16 bit patterns."""
    u32 = np.asarray(bits, dtype=np.uint32) << 16
    return u32.view(np.float32).astype(np.float64)
