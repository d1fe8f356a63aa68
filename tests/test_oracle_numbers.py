"""Pins of the oracle's number formats: E4M3 (OCP FP8) and bf16 conversions.

The oracle's codecs are written from the format definitions; here they are
checked against closed forms of the format and against torch's own casts
(library routines independent of the oracle)."""
import numpy as np
import pytest
import torch

import oracle

ALL = np.arange(256, dtype=np.uint8)


def torch_e4m3_values(codes):
    return torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decode_matches_torch_for_all_codes():
    ours = oracle.e4m3_decode(ALL)
    ref = torch_e4m3_values(ALL)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_closed_forms():
    d = oracle.e4m3_decode
    assert d(np.array([0x7E], np.uint8))[0] == 448.0            # largest finite
    assert d(np.array([0x01], np.uint8))[0] == 2.0 ** -9        # smallest subnormal
    assert d(np.array([0x08], np.uint8))[0] == 2.0 ** -6        # smallest normal
    assert d(np.array([0x38], np.uint8))[0] == 1.0              # exponent field = bias 7
    assert d(np.array([0xB8], np.uint8))[0] == -1.0
    assert d(np.array([0x07], np.uint8))[0] == 7 * 2.0 ** -9    # largest subnormal
    finite = ~np.isnan(oracle.e4m3_decode(ALL))
    assert finite.sum() == 254
    pos = oracle.e4m3_decode(ALL[:0x7F])
    assert np.all(np.diff(pos) > 0)                             # codes 0..126 increase


def test_e4m3_encode_roundtrips_every_finite_code():
    vals = oracle.e4m3_decode(ALL)
    finite = ~np.isnan(vals)
    codes = oracle.e4m3_encode(vals[finite].astype(np.float32))
    assert np.array_equal(codes, ALL[finite])


def test_e4m3_encode_ties_to_even_at_every_midpoint():
    pos = oracle.e4m3_decode(ALL[:0x7F])          # 0 .. 448, increasing
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (pos[:-1] + pos[1:]) / 2)  # exact in fp32
    got = oracle.e4m3_encode(mids)
    lo_code = ALL[:0x7E]
    expect = np.where(lo_code % 2 == 0, lo_code, lo_code + 1)   # the even mantissa wins
    assert np.array_equal(got, expect)
    # one fp32 ulp either side of each midpoint rounds to the nearer neighbour
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(-np.inf))
    assert np.array_equal(oracle.e4m3_encode(up), lo_code + 1)
    assert np.array_equal(oracle.e4m3_encode(dn), lo_code)
    assert np.array_equal(oracle.e4m3_encode(-up), (lo_code + 1) | 0x80)


def test_e4m3_encode_matches_torch_on_random_in_range_values():
    rng = np.random.default_rng(7)
    v = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * np.float32(3.0),
        (rng.uniform(-448, 448, 50000)).astype(np.float32),
        (rng.standard_normal(50000) * 2.0 ** -8).astype(np.float32),   # subnormal range
    ])
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(v), ref)


def test_e4m3_encode_saturates():
    v = np.array([448.0, 460.0, 464.0, 500.0, 1e9, np.inf, -np.inf, -1e9], np.float32)
    assert list(oracle.e4m3_encode(v)) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


def test_bf16_rne_matches_torch_including_ties():
    rng = np.random.default_rng(3)
    v = rng.standard_normal(100000).astype(np.float32)
    ties = ((rng.integers(0, 2**15, 2000).astype(np.uint32) << 16) | 0x8000).view(np.float32)
    v = np.concatenate([v, ties[np.isfinite(ties)]])
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_rne(v), ref)


def test_bf16_trunc_rounds_toward_zero_within_one_ulp():
    rng = np.random.default_rng(4)
    v = rng.standard_normal(50000).astype(np.float32)
    hi = oracle.bf16_value(oracle.bf16_trunc(v))
    v64 = v.astype(np.float64)
    assert np.all(np.abs(hi) <= np.abs(v64))
    assert np.all(np.sign(hi) == np.sign(v64))
    # dropped part is below one bf16 ulp: |v - hi| < 2^-7 |v|
    assert np.all(np.abs(v64 - hi) < 2.0 ** -7 * np.abs(v64))


def test_quant_group_rule():
    rng = np.random.default_rng(5)
    v = rng.standard_normal(128).astype(np.float32) * np.float32(3.7)
    q, s = oracle.quant_group(v)
    amax = np.float32(np.abs(v).max())
    assert s == np.float32(amax / np.float32(448.0))
    # the largest magnitude lands on +-448
    i = int(np.argmax(np.abs(v)))
    assert q[i] & 0x7F == 0x7E
    # codes equal torch's cast of v/s computed in fp32
    ref = torch.from_numpy(v / np.float32(s)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)
    deq = oracle.e4m3_decode(q) * s
    normal = np.abs(v / s) >= 2.0 ** -6
    assert np.all(np.abs(deq - v)[normal] <= 2.0 ** -4 * np.abs(v)[normal] + 1e-12)
    assert np.all(np.abs(deq - v)[~normal] <= 2.0 ** -10 * s + 1e-12)


def test_quant_group_zero_and_x_rows():
    q, s = oracle.quant_group(np.zeros(128, np.float32))
    assert s == 1.0 and not q.any()
    x = torch.randn(3, 256, generator=torch.Generator().manual_seed(1)).bfloat16()
    bits = x.view(torch.int16).numpy().view(np.uint16)
    xq, xs = oracle.quant_x(bits)
    xf = x.float().numpy()
    for t in range(3):
        for g in range(2):
            q, s = oracle.quant_group(xf[t, g * 128:(g + 1) * 128])
            assert xs[t, g] == np.float32(s)
            assert np.array_equal(xq[t, g * 128:(g + 1) * 128], q)
