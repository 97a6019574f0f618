"""Helpers shared by the GPU parity tests: moving raw numpy storage to the
device, reading results back, and the acceptance checks."""
import numpy as np
import torch

import block_swizzled_tile_gb300 as bst
from oracle import formats

# Acceptance: fp16/bf16 outputs need relative Frobenius error <= 1e-3 and
# per-element |err| <= 1e-2 * (|ref| + 1); MXFP8 and dequantised outputs need
# relative Frobenius error <= 2e-3.  The swizzle map and int32 accumulators
# must match bit for bit.
FRO_F16 = 1e-3
ELEM_F16 = 1e-2
FRO_MX = 2e-3


def dev(arr, canary=0):
    """numpy raw storage -> a CUDA tensor holding the same bytes.  With
    ``canary`` > 0 the tensor is a view into a larger buffer padded on both
    sides with ``canary`` bytes of 0xA5 (see ``canary_intact``)."""
    a = np.ascontiguousarray(arr)
    raw = torch.from_numpy(a.view(np.uint8).reshape(-1).copy())
    if canary:
        pad = torch.full((canary,), 0xA5, dtype=torch.uint8)
        buf = torch.cat([pad, raw, pad]).cuda()
        return buf, buf[canary:canary + raw.numel()]
    return raw.cuda()


def empty_bytes(nbytes, canary=0, fill=0x5A):
    """Device buffer of nbytes (filled with ``fill``) plus canary padding."""
    buf = torch.full((nbytes + 2 * canary,), fill, dtype=torch.uint8, device="cuda")
    if canary:
        buf[:canary] = 0xA5
        buf[canary + nbytes:] = 0xA5
    return buf, buf[canary:canary + nbytes]


def canary_intact(buf, canary):
    head = buf[:canary]
    tail = buf[buf.numel() - canary:]
    return bool((head == 0xA5).all().item()) and bool((tail == 0xA5).all().item())


def host(t, dtype):
    """CUDA byte tensor -> numpy array of ``dtype``."""
    return t.cpu().numpy().view(dtype)


def decode_out(raw, out_dtype):
    if out_dtype == "f16":
        return formats.f16_bits_to_f64(raw.view(np.uint16))
    if out_dtype == "bf16":
        return formats.bf16_bits_to_f64(raw.view(np.uint16))
    return raw.view(np.float32).astype(np.float64)


def rel_fro(got, ref):
    den = np.linalg.norm(ref)
    num = np.linalg.norm(got - ref)
    return num / den if den > 0 else num


def assert_close_f16(got, ref, fro=FRO_F16, elem=ELEM_F16):
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), "non-finite output"
    e = rel_fro(got, ref)
    bad = np.abs(got - ref) > elem * (np.abs(ref) + 1)
    assert e <= fro, "relative Frobenius error %.3g > %.3g" % (e, fro)
    assert not bad.any(), "%d elements beyond %.0e*(|ref|+1), first at %s" % (
        bad.sum(), elem, np.argwhere(bad)[0])


def assert_close_fro(got, ref, fro):
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), "non-finite output"
    e = rel_fro(got, ref)
    assert e <= fro, "relative Frobenius error %.3g > %.3g" % (e, fro)


def assert_special_equal(got, ref, fro):
    """NaN positions, and infinity positions with their signs, equal the
    reference's; the finite rest is within the relative Frobenius bound."""
    assert got.shape == ref.shape
    nan_r, inf_r = np.isnan(ref), np.isinf(ref)
    assert np.array_equal(np.isnan(got), nan_r), "NaN positions differ"
    assert np.array_equal(np.isinf(got), inf_r), "infinity positions differ"
    assert np.array_equal(got[inf_r], ref[inf_r]), "infinity signs differ"
    ok = ~(nan_r | inf_r)
    assert_close_fro(got[ok], ref[ok], fro)


DT = {"f16": bst.F16, "bf16": bst.BF16, "f32": bst.F32}
OUT_BYTES = {"f16": 2, "bf16": 2, "f32": 4}
