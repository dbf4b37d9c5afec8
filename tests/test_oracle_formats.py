"""Pins for the oracle's exact code decoding and e4m3 rounding (CPU only).

The oracle decodes stored fp16 / bf16 / e4m3 codes from the format definitions; here
every code is compared with independent library conversions (numpy float16, torch
bfloat16 and float8_e4m3fn), and the e4m3 encoder with torch's round-to-nearest-even.
"""
import numpy as np
import pytest
import torch

from oracle import formats


def _same(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    nan = np.isnan(a)
    assert np.array_equal(nan, np.isnan(b))
    assert np.array_equal(a[~nan], b[~nan])
    # signed zeros must agree too
    assert np.array_equal(np.signbit(a[~nan]), np.signbit(b[~nan]))


def test_f16_all_codes_match_numpy():
    codes = np.arange(1 << 16, dtype=np.uint16)
    _same(formats.to_f64(codes, "f16"), codes.view(np.float16).astype(np.float64))


def test_bf16_all_codes_match_torch():
    codes = torch.arange(1 << 16, dtype=torch.int32).to(torch.int16)
    ref = codes.view(torch.bfloat16).to(torch.float64).numpy()
    _same(formats.to_f64(codes.numpy().view(np.uint16), "bf16"), ref)


def test_e4m3_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    _same(formats.to_f64(codes.numpy(), "e4m3"), ref)


def test_e4m3_special_values():
    t = formats.e4m3_table()
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0          # largest finite
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])          # S.1111.111 is NaN
    assert t[0x01] == 2.0 ** -9                             # smallest subnormal
    assert t[0x08] == 2.0 ** -6                             # smallest normal
    assert t[0x38] == 1.0


def test_e4m3_encoder_matches_torch_rne():
    g = torch.Generator().manual_seed(7)
    x = torch.cat([torch.randn(4000, generator=g) * 4, torch.randn(1000, generator=g) * 200,
                   torch.randn(1000, generator=g) * 1e-2])
    # exact midpoints between neighbouring codes exercise the ties-to-even rule
    t = formats.e4m3_table()
    pos = np.array([t[c] for c in range(0x7F)])
    mids = torch.tensor((pos[:-1] + pos[1:]) / 2.0, dtype=torch.float32)
    x = torch.cat([x, mids, -mids]).clamp(-448, 448)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = formats.encode_e4m3(x.to(torch.float64).numpy())
    assert np.array_equal(got, ref)


def test_e4m3_encoder_saturates():
    got = formats.encode_e4m3(np.array([500.0, -1e9, 449.0, np.inf, -np.inf]))
    assert list(got) == [0x7E, 0xFE, 0x7E, 0x7E, 0xFE]
    assert formats.encode_e4m3(np.array([np.nan]))[0] == 0x7F
