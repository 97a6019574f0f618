"""Pins for oracle.formats: every decoder against an independent decode of the
whole code table, every rounding encoder against brute-force nearest search
over the whole table of the target format (ties to the code with an even last
mantissa bit)."""
import numpy as np
import pytest
import torch

from oracle import formats


def _all16():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


def _decode_binary16_by_fields(bits):
    """IEEE binary16 from its fields: 1 sign, 5 exponent (bias 15), 10 mantissa."""
    out = []
    for b in bits.tolist():
        s = -1.0 if b & 0x8000 else 1.0
        e = (b >> 10) & 0x1F
        m = b & 0x3FF
        if e == 0:
            out.append(s * m * 2.0 ** -24)
        elif e == 0x1F:
            out.append(s * np.inf if m == 0 else np.nan)
        else:
            out.append(s * (1 + m / 1024.0) * 2.0 ** (e - 15))
    return np.array(out)


def test_f16_decode_all_codes():
    bits = _all16()
    got = formats.f16_bits_to_f64(bits)
    want = _decode_binary16_by_fields(bits)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


def test_bf16_decode_all_codes_vs_torch():
    bits = _all16()
    got = formats.bf16_bits_to_f64(bits)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


def _nearest_even_bruteforce(x, table_vals, table_bits, inf_value):
    """Round each x to the nearest entry of a finite table (positive and
    negative), ties to the entry with an even low bit; |x| beyond the largest
    entry rounds against a pseudo entry 'inf_value' (IEEE overflow rule)."""
    vals = np.concatenate([table_vals, [inf_value, -inf_value]])
    bits = np.concatenate([table_bits, [0, 0]]).astype(np.int64)   # inf codes end in 0
    order = np.argsort(vals, kind="stable")
    vals, bits = vals[order], bits[order]
    out = np.empty_like(x)
    for i, v in enumerate(x):
        j = np.searchsorted(vals, v)
        cands = [k for k in (j - 1, j) if 0 <= k < len(vals)]
        d = [abs(vals[k] - v) for k in cands]
        best = min(d)
        tied = [k for k, dd in zip(cands, d) if dd == best]
        if len(tied) > 1:
            tied = [k for k in tied if bits[k] % 2 == 0] or tied
        r = vals[tied[0]]
        out[i] = np.inf * np.sign(r) if abs(r) == inf_value else r
    return out


def _table(decode):
    bits = _all16()
    vals = decode(bits)
    fin = np.isfinite(vals)
    vals, bits = vals[fin], bits[fin]
    # drop -0 duplicate of +0 so ties are not split between them
    keep = ~((vals == 0) & (bits != 0))
    return vals[keep], bits[keep]


def _probe_values(table_vals, rng):
    pos = np.unique(table_vals[table_vals > 0])
    mids = (pos[:-1] + pos[1:]) / 2                       # exact ties
    pick = rng.choice(len(mids), 3000, replace=False)
    near = mids[pick] * (1 + rng.uniform(-1e-6, 1e-6, size=3000))
    rnd = rng.standard_normal(3000) * rng.choice([1e-6, 1e-3, 1, 1e3, 1e5], 3000)
    x = np.concatenate([mids[pick], near, rnd, -mids[pick[:500]], [0.0, 1.0, -2.5]])
    return x


def test_f64_to_f16_matches_bruteforce():
    rng = np.random.default_rng(1)
    vals, bits = _table(formats.f16_bits_to_f64)
    x = _probe_values(vals, rng)
    x = np.concatenate([x, [65504.0, 65519.99, 65520.0, 70000.0, 2.0 ** -25, 2.0 ** -26, 3 * 2.0 ** -26]])
    got = formats.f16_bits_to_f64(formats.f64_to_f16_bits(x))
    want = _nearest_even_bruteforce(x, vals, bits, inf_value=65536.0)
    assert np.array_equal(got, want)


def test_f64_to_bf16_matches_bruteforce():
    rng = np.random.default_rng(2)
    vals, bits = _table(formats.bf16_bits_to_f64)
    x = _probe_values(vals, rng)
    big = float(vals.max())
    x = np.concatenate([x, [big, big * (1 + 2.0 ** -9), 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -134, 1e-45]])
    got = formats.bf16_bits_to_f64(formats.f64_to_bf16_bits(x))
    want = _nearest_even_bruteforce(x, vals, bits, inf_value=2.0 ** 128)
    assert np.array_equal(got, want)


def test_f64_to_bf16_matches_torch_on_float32_inputs():
    # for inputs that are exact float32 values torch's float->bfloat16 cast is RNE
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000)).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = formats.f64_to_bf16_bits(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_e4m3_decode_all_codes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = formats.decode_e4m3(codes)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x38, 1.0), (0x7E, 448.0), (0xFE, -448.0), (0x01, 2.0 ** -9),
    (0x08, 2.0 ** -6), (0x07, 7 * 2.0 ** -9), (0x40, 2.0), (0x3C, 1.5)])
def test_e4m3_known_values(code, value):
    assert formats.decode_e4m3(np.array([code], np.uint8))[0] == value


def test_e4m3_nan_codes():
    v = formats.decode_e4m3(np.array([0x7F, 0xFF], np.uint8))
    assert np.isnan(v).all()


def test_e8m0():
    v = formats.decode_e8m0(np.array([127, 128, 126, 0, 254, 255], np.uint8))
    assert v[0] == 1.0 and v[1] == 2.0 and v[2] == 0.5
    assert v[3] == 2.0 ** -127 and v[4] == 2.0 ** 127 and np.isnan(v[5])


def _decode_binary32_by_fields(bits):
    """IEEE binary32 from its fields: 1 sign, 8 exponent (bias 127), 23
    mantissa; float64 holds every binary32 value exactly."""
    b = np.asarray(bits, dtype=np.uint64)
    s = np.where(b >> 31, -1.0, 1.0)
    e = ((b >> 23) & 0xFF).astype(np.int64)
    m = (b & 0x7FFFFF).astype(np.float64)
    val = np.where(e == 0, m * 2.0 ** -149, (1.0 + m / 2.0 ** 23) * np.ldexp(1.0, (e - 127).clip(-126, 127)))
    val = np.where(e == 0xFF, np.where(m == 0, np.inf, np.nan), val)
    return s * val


def _f32_nearest_even_check(x, got_bits):
    """The defining property of round-to-nearest-even into binary32, checked
    on each x against the two binary32 codes next to the result (bit pattern
    +-1 of the same sign; zero's neighbours are the smallest subnormals):
    the result is no farther from x than either neighbour, a tie goes to the
    even code, and a result of +-inf means |x| reached the overflow bound
    2**128 - 2**103 (halfway between the largest finite value and 2**128)."""
    bad = []
    for xi, gb in zip(x.tolist(), got_bits.tolist()):
        y = float(_decode_binary32_by_fields(np.array([gb]))[0])
        if np.isinf(y):
            if not (abs(xi) >= 2.0 ** 128 - 2.0 ** 103 and np.sign(y) == np.sign(xi)):
                bad.append(xi)
            continue
        mag = gb & 0x7FFFFFFF
        sign = gb & 0x80000000
        neigh = []
        for dm in (-1, 1):
            nm = mag + dm
            if nm < 0:
                neigh.append((0x80000000 ^ sign) | 1)       # across zero: the other sign's smallest subnormal
            elif nm <= 0x7F7FFFFF:
                neigh.append(sign | nm)
        d = abs(y - xi)
        for nb in neigh:
            v = float(_decode_binary32_by_fields(np.array([nb]))[0])
            dn = abs(v - xi)
            if dn < d or (dn == d and v != y and (gb & 1) and not (nb & 1)):
                bad.append(xi)
                break
    return bad


def test_f64_to_f32_matches_nearest_even_neighbour_search():
    rng = np.random.default_rng(4)
    # random doubles over many binades (their low 29 bits are what rounding drops)
    rnd = rng.standard_normal(4000) * 10.0 ** rng.integers(-40, 38, 4000)
    # exact ties: the midpoint of two adjacent binary32 values, both parities
    lo_bits = rng.integers(0x00800000, 0x7F7FFFFF, 3000).astype(np.uint64)
    lo = _decode_binary32_by_fields(lo_bits)
    hi = _decode_binary32_by_fields(lo_bits + 1)
    mids = (lo + hi) / 2                                   # exact in float64
    near = mids * (1 + rng.uniform(-1e-12, 1e-12, 3000))
    edges = [2.0 ** -149, 2.0 ** -150, 3 * 2.0 ** -150, 5 * 2.0 ** -151, 2.0 ** -126, 2.0 ** -126 - 2.0 ** -150,
             float(np.finfo(np.float32).max), 2.0 ** 128 - 2.0 ** 104, 2.0 ** 128 - 2.0 ** 103,
             2.0 ** 128 - 2.0 ** 103 - 2.0 ** 70, 1e39, 0.0, 1.0, -1.0 - 2.0 ** -24, 1.0 + 2.0 ** -24,
             1.0 + 3 * 2.0 ** -24]
    x = np.concatenate([rnd, mids, -mids[:500], near, edges, [-e for e in edges]])
    with np.errstate(over="ignore"):
        got = formats.f64_to_f32(x)
    assert got.dtype == np.float32
    assert _f32_nearest_even_check(x, got.view(np.uint32)) == []


def test_f32_neighbour_check_catches_a_planted_truncation():
    """Truncation toward zero (a plausible mistake in an f32 encoder) must
    fail the nearest-even check above."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal(2000) * 10.0 ** rng.integers(-20, 20, 2000)
    trunc = x.astype(np.float32)
    up = np.abs(trunc.astype(np.float64)) > np.abs(x)
    trunc[up] = np.nextafter(trunc[up], np.float32(0))
    assert len(_f32_nearest_even_check(x, trunc.view(np.uint32))) > 100


def test_binary32_field_decoder_known_values():
    known = {0x3F800000: 1.0, 0xC0000000: -2.0, 0x00000001: 2.0 ** -149, 0x00800000: 2.0 ** -126,
             0x7F7FFFFF: (2 - 2.0 ** -23) * 2.0 ** 127, 0x7F800000: np.inf, 0x00000000: 0.0, 0x3EAAAAAB: None}
    for b, v in known.items():
        got = float(_decode_binary32_by_fields(np.array([b]))[0])
        if v is None:
            assert abs(got - 1 / 3) < 2.0 ** -25
        else:
            assert got == v
