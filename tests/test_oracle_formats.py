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
