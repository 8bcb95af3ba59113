"""Pins of the oracle's NVFP4 quantizer (no GPU): worked special cases, scale
invariance, brute-force nearest codes and scales, and the error bound."""
import numpy as np

import oracle
from helpers import golden

E2M1 = np.array([float(v) for k, c, v in golden("e2m1.txt") if k == "decode"])


def _nibbles(codes):
    lo = codes & 15
    hi = codes >> 4
    return np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)


def test_equal_block_at_tensor_max_gives_six_and_448():
    v = np.full((2, 32), 0.75, np.float32)
    v[1, 16:] = -0.75
    codes, sf, sg, amax = oracle.nvfp4_quantize(v)
    assert amax == np.float32(0.75)
    assert sg == np.float32(0.75) / np.float32(2688.0)
    assert np.all(sf == 0x7E)                    # 448
    n = _nibbles(codes)
    assert np.all(n[0] == 7) and np.all(n[1, :16] == 7) and np.all(n[1, 16:] == 15)


def test_zero_tensor_and_zero_block():
    codes, sf, sg, amax = oracle.nvfp4_quantize(np.zeros((3, 48), np.float32))
    assert sg == 0 and amax == 0 and not codes.any() and not sf.any()
    v = np.zeros((1, 32), np.float32)
    v[0, 16:] = np.linspace(-1, 1, 16)
    codes, sf, sg, _ = oracle.nvfp4_quantize(v)
    assert sf[0, 0] == 0 and not _nibbles(codes)[0, :16].any()


def test_power_of_two_scale_invariance():
    rs = np.random.RandomState(2)
    v = (rs.standard_normal((16, 128)) * 0.02).astype(np.float32)
    c0, s0, g0, _ = oracle.nvfp4_quantize(v)
    for m in (-7, -1, 3, 9):
        c1, s1, g1, _ = oracle.nvfp4_quantize((v * np.float32(2.0 ** m)).astype(np.float32))
        assert np.array_equal(c0, c1) and np.array_equal(s0, s1)
        assert g1 == np.float32(g0 * np.float32(2.0 ** m))


def test_low_nibble_holds_the_even_element():
    v = np.zeros((1, 16), np.float32)
    v[0, 0] = 6.0   # code 7
    v[0, 1] = -3.0  # code 0xd
    codes, sf, sg, _ = oracle.nvfp4_quantize(v)
    assert codes[0, 0] == 0x7 | (0xD << 4)


def test_codes_and_scales_are_nearest_by_brute_force():
    rs = np.random.RandomState(3)
    v = (rs.standard_normal((64, 256)) * rs.uniform(0.01, 3.0, (64, 1))).astype(np.float32)
    codes, sf, sg, amax = oracle.nvfp4_quantize(v)
    assert amax == np.abs(v).max()
    e4m3_vals = np.array([oracle.e4m3_decode(c) for c in range(127)])
    n = _nibbles(codes)
    ties = 0
    for r in range(v.shape[0]):
        for b in range(v.shape[1] // 16):
            blk = v[r, 16 * b:16 * b + 16].astype(np.float64)
            target = float(np.float32(np.float32(np.abs(blk).max() / np.float32(6.0)) / sg))
            dist = np.abs(e4m3_vals - min(target, 448.0))
            best = np.flatnonzero(dist == dist.min())
            assert sf[r, b] in best
            d = float(np.float32(oracle.e4m3_decode(int(sf[r, b])) * sg))
            for i in range(16):
                err = np.abs(np.abs(blk[i]) / d - E2M1[:8]) if d > 0 else None
                c = n[r, 16 * b + i]
                cand = np.flatnonzero(err == err.min())
                if len(cand) > 1:
                    ties += 1
                assert (c & 7) in cand, (r, b, i)
                if blk[i] != 0 and (c & 7) != 0:
                    assert (c >> 3) == (blk[i] < 0)
    assert ties < 5


def test_dequantization_error_bound():
    rs = np.random.RandomState(4)
    v = (rs.standard_normal((32, 512)) * 0.02).astype(np.float32)
    codes, sf, sg, _ = oracle.nvfp4_quantize(v)
    vh = oracle.nvfp4_dequantize(codes, sf, sg, 32, 512)
    d = np.repeat(np.array([[oracle.e4m3_decode(int(s)) for s in row] for row in sf]), 16, axis=1) * sg
    # half the widest gap of the e2m1 grid (4 -> 6) is one unit of the block scale
    assert np.all(np.abs(v - vh) <= d * (1.0 + 1e-6))
    # relative rms error of NVFP4 on Gaussian data is a few percent, never tens of percent
    rel = np.sqrt(np.mean((v - vh) ** 2) / np.mean(v.astype(np.float64) ** 2))
    assert 0.02 < rel < 0.15


def test_dequantize_matches_format_tables():
    rs = np.random.RandomState(5)
    codes = rs.randint(0, 256, (4, 16), dtype=np.uint8)
    sf = rs.randint(0, 127, (4, 2), dtype=np.uint8)
    sg = np.float32(0.37)
    got = oracle.nvfp4_dequantize(codes, sf, sg, 4, 32)
    e4 = {int(c, 16): float(v) for k, c, v in golden("e4m3.txt") if k == "decode"}
    for r in range(4):
        for c in range(32):
            code = (codes[r, c // 2] >> (4 * (c % 2))) & 15
            scale = oracle.e4m3_decode(int(sf[r, c // 16]))
            if int(sf[r, c // 16]) in e4:
                assert scale == e4[int(sf[r, c // 16])]
            assert got[r, c] == E2M1[code] * scale * float(sg)
