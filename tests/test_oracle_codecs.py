"""Pins for oracle/codecs.py: number formats checked against torch's own
casts (an independent library), the OCP MX format tables, hand-enumerated tie
cases and exhaustive code round trips."""
import math

import numpy as np
import pytest
import torch

from oracle import codecs


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = codecs.e4m3_decode(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    # hand values: max normal 448 = 1.75 * 2^8 (0x7E), min normal 2^-6, min subnormal 2^-9
    assert ours[0x7E] == 448.0 and ours[0x08] == 2.0 ** -6 and ours[0x01] == 2.0 ** -9
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF])


def test_e4m3_round_matches_torch_in_range():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 100, 20000),
                        rng.uniform(-448, 448, 20000), rng.normal(0, 1e-2, 20000)])
    v = v.astype(np.float32).astype(np.float64)
    v = v[np.abs(v) <= 448.0]          # torch's cast is non-saturating beyond 448
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(codecs.round_e4m3(v), ref)


def test_e4m3_ties_to_even_and_saturation():
    vals = codecs.e4m3_decode(np.arange(0x00, 0x7F, dtype=np.uint8))   # 0 .. 448
    for c in range(0x7E):
        lo, hi = vals[c], vals[c + 1]
        mid = 0.5 * (lo + hi)
        expect = lo if c % 2 == 0 else hi          # the even code wins a tie
        assert codecs.round_e4m3(mid) == expect, (c, lo, hi)
        assert codecs.round_e4m3(-mid) == -expect
    for big in (448.0 + 1e-9, 449.0, 464.0, 480.0, 1e6, 1e30):
        assert codecs.round_e4m3(big) == 448.0 and codecs.round_e4m3(-big) == -448.0


def test_e4m3_encode_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = codecs.e4m3_decode(codes)
    assert np.array_equal(codecs.e4m3_encode(vals), codes)
    with pytest.raises(ValueError):
        codecs.e4m3_encode(np.array([1.0 + 2.0 ** -5]))


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.normal(0, 1, 50000), rng.normal(0, 1e30, 1000),
                        rng.normal(0, 1e-39, 1000), rng.normal(0, 1e-3, 50000)])
    v32 = v.astype(np.float32)
    ref = torch.from_numpy(v32).to(torch.bfloat16).double().numpy()
    assert np.array_equal(codecs.round_bf16(v32.astype(np.float64)), ref)


def test_bf16_round_hand_cases():
    assert codecs.round_bf16(1 + 2.0 ** -8) == 1.0                 # tie -> even
    assert codecs.round_bf16(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6   # tie -> even
    assert codecs.round_bf16(1 + 2.0 ** -8 + 2.0 ** -40) == 1 + 2.0 ** -7   # above tie
    assert codecs.round_bf16(2.0 ** -133) == 2.0 ** -133           # min subnormal
    assert codecs.round_bf16(codecs.BF16_MAX) == codecs.BF16_MAX
    assert np.isinf(codecs.round_bf16(3.4e38 * 1.01))


def test_round_fp32_is_ieee():
    rng = np.random.default_rng(2)
    a = rng.normal(0, 1, 1000).astype(np.float32)
    b = rng.normal(0, 1, 1000).astype(np.float32)
    # fp32 division of fp32 operands, correctly rounded, equals torch fp32 division
    q = codecs.round_fp32(a.astype(np.float64) / b.astype(np.float64))
    ref = (torch.from_numpy(a) / torch.from_numpy(b)).double().numpy()
    assert np.array_equal(q, ref)


def test_e2m1_table_from_ocp_mx_spec():
    # OCP Microscaling Formats v1.0, FP4 E2M1 table: 0, 0.5, 1, 1.5, 2, 3, 4, 6
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    ours = codecs.e2m1_decode(np.arange(16))
    assert list(ours[:8]) == table
    assert list(ours[8:]) == [-t for t in table]


def test_e8m0_matches_torch():
    codes = np.arange(255, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e8m0fnu).double().numpy()
    assert np.array_equal(codecs.e8m0_decode(codes), ref)


def test_unpack_fp4_nibble_order():
    assert list(codecs.unpack_fp4(np.array([0x21, 0xF0], dtype=np.uint8), 4)) == [1, 2, 0, 15]


def test_ceil_pow2():
    for s in [1.0, 2.0, 0.25, 3.0, 0.3, 1e-10, 5e5, float(np.float32(1e-10) / 448)]:
        expect = 2.0 ** math.ceil(math.log2(s))
        assert codecs.ceil_pow2(s) == expect, s
