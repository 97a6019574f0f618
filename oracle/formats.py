"""Number formats, written from their definitions.  TEST INFRASTRUCTURE ONLY.

Storage is always raw bits (``uint16`` for fp16/bf16, ``uint8`` for e4m3 and
E8M0) so the oracle decodes inputs itself instead of trusting anyone's cast.

Pins (tests/test_oracle_formats.py): every decoder against torch/numpy over
all codes; every rounding encoder against a brute-force nearest-value search
over the complete table of the target format, ties to even.
"""
import numpy as np

# ---------------------------------------------------------------- fp16 -------

def f16_bits_to_f64(bits):
    """IEEE binary16 bits -> float64 (exact)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def f64_to_f16_bits(x):
    """float64 -> IEEE binary16 bits, round to nearest, ties to even.

    numpy converts double to half in one correctly rounded step (no detour
    through float32, so no double rounding)."""
    with np.errstate(over="ignore"):       # overflow to +-inf is the rule
        return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


# ---------------------------------------------------------------- bf16 -------

def bf16_bits_to_f64(bits):
    """bfloat16 bits (the top half of a binary32) -> float64 (exact)."""
    wide = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):    # NaN codes stay NaN
        return wide.view(np.float32).astype(np.float64)


def _round_to_binary(x, mant_bits, emin, emax):
    """Round float64 ``x`` to a binary format with ``mant_bits`` stored
    mantissa bits, minimum normal exponent ``emin`` and maximum exponent
    ``emax``, nearest/ties-to-even, overflow to +-inf.  Returns float64."""
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    fin = np.isfinite(x) & (x != 0)
    xf = x[fin]
    _, e2 = np.frexp(xf)                    # |x| in [2**(e2-1), 2**e2)
    exp = np.maximum(e2 - 1, emin)          # subnormals share the emin spacing
    ulp = np.ldexp(1.0, exp - mant_bits)
    q = np.round(xf / ulp) * ulp            # np.round is ties-to-even; x/ulp is exact
    big = np.ldexp(1.0, emax + 1)
    q = np.where(np.abs(q) >= big, np.copysign(np.inf, xf), q)
    out[fin] = q
    return out


def f64_to_bf16_bits(x):
    """float64 -> bfloat16 bits, round to nearest, ties to even, in one step
    (8 significant bits, exponent range of binary32)."""
    q = _round_to_binary(x, mant_bits=7, emin=-126, emax=127)
    return (q.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def f64_to_f32(x):
    """float64 -> float32, round to nearest even (numpy's cast is correctly
    rounded)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32)


# ---------------------------------------------------------------- e4m3 -------

def decode_e4m3(codes):
    """float8 e4m3 ("fn" variant) -> float64.

    Layout S EEEE MMM, exponent bias 7.  E == 0 is subnormal (M/8 * 2**-6);
    otherwise (1 + M/8) * 2**(E-7).  S.1111.111 is NaN; there is no infinity,
    so the largest finite magnitude is 1.75 * 2**8 = 448."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0,
                   (m / 8.0) * 2.0 ** -6,
                   (1.0 + m / 8.0) * np.ldexp(1.0, (e - 7).astype(np.int64)))
    val = sign * val
    return np.where((e == 0xF) & (m == 0x7), np.nan, val)


def decode_e8m0(codes):
    """E8M0 scale (an unsigned 8-bit biased exponent, bias 127) -> float64:
    2**(s-127); the code 255 is NaN."""
    s = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    return np.where(s == 255, np.nan, np.ldexp(1.0, s - 127))
