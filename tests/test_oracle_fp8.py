"""Pins of the oracle's 8-bit (E4M3) cache storage: the decoding table, the
rounding rule and the scaled storage, against a library implementation of
the same format (torch.float8_e4m3fn) and against values worked by hand.  A
wrong exponent bias, a truncating encoder or ties away from even would fail
one of them."""
import numpy as np
import pytest
import torch

from oracle import fp8


def _torch_decode(codes):
    t = torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def _torch_encode(x):
    t = torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_decode_table_matches_library():
    codes = np.arange(256, dtype=np.uint8)
    ours, lib = fp8.e4m3_decode(codes), _torch_decode(codes)
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    ok = ~np.isnan(ours)
    assert np.array_equal(ours[ok], lib[ok])
    assert np.isnan(ours).sum() == 2  # 0x7F and 0xFF


def test_decode_by_hand():
    # 0x38: exponent 7, mantissa 0 -> 1.0; 0x7E -> 1.75 * 2^8; 0x01 -> 2^-9; 0x08 -> 2^-6
    assert fp8.e4m3_decode([0x38, 0x7E, 0x01, 0x08, 0xB8, 0x00, 0x80]).tolist()[:5] == \
        [1.0, 448.0, 2.0 ** -9, 2.0 ** -6, -1.0]
    z = fp8.e4m3_decode([0x00, 0x80])
    assert z[0] == 0 and z[1] == 0 and np.signbit(z[1])


def test_encode_matches_library_below_saturation():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 30, rng.uniform(-447, 447, 20000),
                        rng.standard_normal(5000) * 1e-2]).astype(np.float32)
    assert np.array_equal(fp8.e4m3_encode(x), _torch_encode(x))


def test_encode_by_hand():
    e = fp8.e4m3_encode
    assert e(1.0) == 0x38 and e(-1.0) == 0xB8
    assert e(448.0) == 0x7E and e(1e9) == 0x7E and e(-1e9) == 0xFE  # saturation
    assert e(np.inf) == 0x7E and e(np.nan) == 0x7F
    assert e(2.0 ** -9) == 0x01
    assert e(2.0 ** -10) == 0x00           # halfway between 0 and 2^-9: even code 0
    assert e(1.5 * 2.0 ** -9) == 0x02      # halfway between codes 1 and 2: even code 2
    assert e(1.0625) == 0x38               # halfway between 1.0 and 1.125: mantissa 0
    assert e(1.1875) == 0x3A               # halfway between 1.125 and 1.25: mantissa 2
    assert e(1.0625 + 1e-9) == 0x39        # just above halfway rounds up
    assert e(-0.0) == 0x80


def test_round_trip_of_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    assert np.array_equal(fp8.e4m3_encode(fp8.e4m3_decode(codes)), codes)


def test_scaled_storage():
    s = 2.0 ** -6
    x = np.array([0.5, -3.0, 7.0, 1e3])
    codes = fp8.quantize(x, s)
    back = fp8.dequantize(codes, s)
    assert back[0] == 0.5 and back[1] == -3.0 and back[2] == 7.0  # exactly representable
    assert back[3] == 448.0 * s                                   # saturated


def test_mutations_fail(monkeypatch):
    # a wrong bias and a truncating encoder disagree with the pins above
    wrong = lambda c: np.asarray(fp8.e4m3_decode(c)) * 2.0
    assert not np.array_equal(wrong(np.arange(0x7F, dtype=np.uint8)),
                              _torch_decode(np.arange(0x7F, dtype=np.uint8)))
    x = np.float64(1.1875)
    trunc = np.searchsorted(fp8._POS, x, side="right") - 1
    assert trunc != fp8.e4m3_encode(x)
