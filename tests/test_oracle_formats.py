"""Pins of the oracle's element formats and of the seeded input generator,
against published definitions and library routines (no GPU)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import golden


def test_philox_known_answers():
    for row in golden("philox4x32_10_kat.txt"):
        v = [int(t, 16) for t in row]
        out = synth.philox(v[0:4], v[4:6])
        assert [int(x) for x in out] == v[6:10]


def test_unit_normal_moments_and_support():
    z = synth.normal_f32((1 << 20,), 0, synth.tag(synth.KIND_STREAM, 3, 1))
    assert abs(z.mean()) < 5e-3
    assert abs(z.std() - 1.0) < 5e-3
    # Irwin-Hall(8): support within sqrt(1.5) * 4
    assert np.abs(z).max() <= 4.0 * 1.2247449 + 1e-6
    # distinct tags give independent streams
    z2 = synth.normal_f32((1 << 20,), 0, synth.tag(synth.KIND_STREAM, 3, 2))
    assert abs(np.corrcoef(z, z2)[0, 1]) < 5e-3


def test_normal_scaling_is_two_roundings():
    z = synth.normal_f32((4096,), 7, 99)
    v = synth.normal_f32((4096,), 7, 99, 1.0, 0.1)
    ref = (np.float32(0.1) * z).astype(np.float32) + np.float32(1.0)
    assert np.array_equal(v, ref.astype(np.float32))


def test_bf16_generator_matches_torch_rounding():
    v = synth.normal_f32((1 << 16,), 3, 5, 0.0, 1.0)
    b = synth.normal_bf16((1 << 16,), 3, 5, 0.0, 1.0)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.uint16).numpy()
    assert np.array_equal(b, ref)


def test_e2m1_decode_golden():
    for kind, code, val in golden("e2m1.txt"):
        if kind != "decode":
            continue
        got = oracle.e2m1_decode(int(code, 16))
        assert got == float(val) and np.signbit(got) == np.signbit(float(val)), (code, got)


def test_e2m1_encode_golden():
    for kind, val, code in golden("e2m1.txt"):
        if kind != "encode":
            continue
        assert oracle.e2m1_encode(float(val)) == int(code, 16), (val, code)


def test_e2m1_encode_is_nearest_even_on_a_dense_grid():
    table = {c: float(v) for k, c, v in golden("e2m1.txt") if k == "decode" for c in [int(c, 16)]}
    mags = [table[c] for c in range(8)]
    for a in np.linspace(0.0, 6.0, 6001):
        a = float(np.float32(a))
        d = [abs(a - m) for m in mags]
        best = min(d)
        cands = [c for c in range(8) if d[c] == best]
        want = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
        assert oracle.e2m1_encode(a) == want, a
        assert oracle.e2m1_encode(-a) == want | 8, a


def test_e4m3_decode_matches_torch_and_golden():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = np.array([oracle.e4m3_decode(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))
    for kind, code, val in golden("e4m3.txt"):
        if kind == "decode":
            assert oracle.e4m3_decode(int(code, 16)) == float(val)


def test_e4m3_encode_matches_torch_in_range_and_saturates():
    rs = np.random.RandomState(0)
    v = np.concatenate([rs.uniform(-447.9, 447.9, 100000), rs.uniform(-1, 1, 100000) * 0.05,
                        rs.uniform(-1, 1, 50000) * 2e-3]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(x)) for x in v], dtype=np.uint8)
    assert np.array_equal(got, ref)
    for kind, val, code in golden("e4m3.txt"):
        if kind == "encode":
            assert oracle.e4m3_encode(float(val)) == int(code, 16), val
            assert oracle.e4m3_encode(-float(val)) == int(code, 16) | 0x80, val


def test_bf16_rounding_matches_torch_on_fp32_values():
    rs = np.random.RandomState(1)
    v = (rs.standard_normal(20000) * 10.0 ** rs.uniform(-6, 6, 20000)).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.uint16).numpy()
    got = np.array([oracle.bf16_from_double(float(x)) for x in v], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_rounds_once_from_fp64():
    # 1 + 2^-8 is the midpoint between 1 and 1 + 2^-7; a hair above it must round up
    # even though rounding to fp32 first would land on the midpoint and go to even.
    above = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert oracle.bf16_from_double(above) == 0x3F81
    assert oracle.bf16_from_double(1.0 + 2.0 ** -8) == 0x3F80
    assert oracle.bf16_to_f64(np.array([0x3F81]))[0] == 1.0 + 2.0 ** -7
