"""Pins of the oracle's E4M3FN codec, per-tensor scale and pack (no GPU).

The E4M3FN format (1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
subnormal step 2^-9, largest finite 448 = 0x7E, NaN = S.1111.111, no
infinities) is fixed by its definition; the decode table is checked against
torch's own float8_e4m3fn conversion (a library routine), and the encoder
against the format's grid and against torch's conversion inside the finite
range.  The quantisation rule is scale = amax/448 and
q = satfinite_rne(x/scale) (FlyDSL PR #860: per-tensor fp8 pack; the
saturating RNE reading is the one the fp8 conv reference needs to be exact).
"""
import numpy as np
import pytest
import torch

import oracle


def _torch_e4m3_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_decode_table_matches_torch_for_all_codes():
    got = oracle.e4m3_decode_table()
    ref = _torch_e4m3_decode_all()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}
    assert np.array_equal(got[~nan], ref[~nan])
    # signs of zero
    assert np.signbit(got[0x80]) and not np.signbit(got[0x00])


def test_decode_closed_forms():
    assert oracle.e4m3_to_f64(0x7E) == 448.0
    assert oracle.e4m3_to_f64(0x01) == 2.0 ** -9          # smallest subnormal
    assert oracle.e4m3_to_f64(0x07) == 7 * 2.0 ** -9      # largest subnormal
    assert oracle.e4m3_to_f64(0x08) == 2.0 ** -6          # smallest normal
    assert oracle.e4m3_to_f64(0x38) == 1.0
    assert oracle.e4m3_to_f64(0xB8) == -1.0
    assert oracle.e4m3_to_f64(0x3C) == 1.5
    assert oracle.e4m3_to_f64(0x77) == 240.0


def test_encode_roundtrips_every_finite_code():
    tab = oracle.e4m3_decode_table()
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.f32_to_e4m3(float(np.float32(tab[c]))) == c


def test_encode_midpoints_go_to_even_code():
    tab = oracle.e4m3_decode_table()
    for c in range(0x00, 0x7E):
        mid = (tab[c] + tab[c + 1]) / 2.0   # exactly representable in binary32
        assert float(np.float32(mid)) == mid
        even = c if c % 2 == 0 else c + 1
        assert oracle.f32_to_e4m3(mid) == even, hex(c)
        assert oracle.f32_to_e4m3(-mid) == 0x80 | even
        # just off the midpoint goes to the nearer neighbour
        below = np.nextafter(np.float32(mid), np.float32(0))
        above = np.nextafter(np.float32(mid), np.float32(1000))
        assert oracle.f32_to_e4m3(float(below)) == c
        assert oracle.f32_to_e4m3(float(above)) == c + 1


def test_encode_saturates_and_keeps_signs():
    assert oracle.f32_to_e4m3(448.0 * (1 + 2 ** -5)) == 0x7E
    for v in (449.0, 463.99, 464.0, 480.0, 1000.0, 3.0e38, float("inf")):
        assert oracle.f32_to_e4m3(v) == 0x7E
        assert oracle.f32_to_e4m3(-v) == 0xFE
    assert oracle.f32_to_e4m3(2.0 ** -10) == 0x00      # tie between 0 and 2^-9 -> even (0)
    assert oracle.f32_to_e4m3(3 * 2.0 ** -10) == 0x02  # tie between 1 and 2 (x 2^-9) -> 2
    assert oracle.f32_to_e4m3(-(2.0 ** -11)) == 0x80   # rounds to -0
    assert oracle.f32_to_e4m3(-0.0) == 0x80
    assert oracle.f32_to_e4m3(0.0) == 0x00


def _all_bf16_as_f32():
    bits = np.arange(65536, dtype=np.uint32) << 16
    return bits.view(np.float32)


@pytest.mark.parametrize("scale", [1.0, 0.0078125, 3.0 / 448.0, 0.37])
def test_encode_matches_torch_inside_finite_range(scale):
    vals = _all_bf16_as_f32()
    finite = np.isfinite(vals)
    with np.errstate(over="ignore"):    # large values over a small scale: inf, dropped below
        q = (vals[finite] / np.float32(scale)).astype(np.float32)
    keep = np.abs(q) < 464.0            # torch's cast is non-saturating beyond this
    q = q[keep]
    ref = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    lib = oracle._load()
    got = np.fromiter((lib.oracle_f32_to_e4m3(float(v)) for v in q), dtype=np.uint8, count=q.size)
    assert np.array_equal(got, ref)


def test_scale_and_quantize_rule():
    xb = torch.tensor([0.5, -3.25, 2.0, 0.0, 1e-3], dtype=torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    amax = oracle.amax_bf16(bits)
    assert amax == 3.25
    scale = oracle.fp8_scale(amax)
    assert scale == float(np.float32(3.25) / np.float32(448.0))
    q = oracle.quantize_e4m3(bits, scale)
    assert q[1] == 0xFE               # the amax element lands on -448
    assert q[3] == 0x00
    tab = oracle.e4m3_decode_table()
    # dequantised values are within half a code step of the scaled input
    for v, c in zip(xb.float().numpy(), q):
        qv = np.float32(v) / np.float32(scale)
        assert abs(tab[c] - qv) <= 0.5 * max(2.0 ** -9, 2.0 ** (np.floor(np.log2(abs(qv) + 1e-30)) - 3)) + 1e-12
    assert oracle.fp8_scale(0.0) == 1.0


def test_pack_bf16_is_transpose():
    x = torch.randn((2, 5, 3, 4, 6)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    out = oracle.pack_ncdhw_to_ndhwc_bf16(bits)
    assert np.array_equal(out, np.transpose(bits, (0, 2, 3, 4, 1)))


def test_pack_fp8_is_transpose_of_quantized():
    x = (torch.randn((2, 7, 3, 4, 5)) * 3).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    out, scale = oracle.pack_ncdhw_to_ndhwc_fp8(bits)
    amax = float(x.abs().max())
    assert scale == float(np.float32(amax) / np.float32(448.0))
    q = oracle.quantize_e4m3(bits, scale)
    assert np.array_equal(out, np.transpose(q, (0, 2, 3, 4, 1)))
    assert (out & 0x7F).max() == 0x7E      # the amax element maps to 448
    # all-zero input: scale 1, every code 0
    zeros = np.zeros((1, 2, 1, 1, 3), dtype=np.uint16)
    out0, s0 = oracle.pack_ncdhw_to_ndhwc_fp8(zeros)
    assert s0 == 1.0 and not out0.any()


def test_fp8_conv_reference_uses_decoded_values():
    """The fp8-cast conv reference: conv of decoded e4m3 values times both
    scales (FlyDSL PR #860, fp8 test description)."""
    rng = np.random.default_rng(11)
    qx = rng.integers(0, 256, size=(1, 3, 4, 4, 16), dtype=np.uint8)
    qw = rng.integers(0, 256, size=(8, 1, 3, 3, 16), dtype=np.uint8)
    qx[(qx & 0x7F) == 0x7F] = 0x11   # no NaN codes
    qw[(qw & 0x7F) == 0x7F] = 0x22
    tab = oracle.e4m3_decode_table()
    got = oracle.conv3d(qx, qw, pad=(0, 1, 1), scale_x=0.25, scale_w=0.125)
    ref = oracle.conv3d(tab[qx], tab[qw], pad=(0, 1, 1)) * (0.25 * 0.125)
    np.testing.assert_allclose(got, ref, rtol=1e-15, atol=0)
