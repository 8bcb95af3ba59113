"""Pins of the oracle's draft context-KV projection (no GPU).

The projection (the DSpark page, _project_muse_context_kv and
precompute_and_store_context_kv) normalises the context rows with
hidden_norm, then with each layer's pre_qkv_proj_norm, multiplies by each
layer's stacked K/V rows, normalises every key head in fp32 without a weight,
rotates the keys by their positions and writes keys and values into the
cache at the given slots.  The pins: closed forms of the norms on constant
rows, scale invariance without eps, library matmuls over exact sums, one-hot
key heads whose rotation is a named cosine and sine, pair norms and relative
positions preserved by the rotation, and a brute-force cache scatter.
"""
import math

import numpy as np

import oracle


def _bf16_bits(a):
    import torch
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.uint16).numpy()


def _f64(bits):
    return oracle.bf16_to_f64(np.asarray(bits, np.uint16))


def _bits_of(v):
    return np.array([oracle.bf16_from_double(float(t)) for t in np.ravel(v)],
                    np.uint16).reshape(np.shape(v))


def _kv_rows(rs, L, n, KVH, D, scale=1.0):
    return _bf16_bits(rs.standard_normal((L, n, 2 * KVH * D)) * scale)


# ------------------------------------------------------------------ norms


def test_constant_rows_closed_form():
    """ctx = c with w_hidden = 1 gives a constant fc = bf16(sign(c) / sqrt(1 + eps/c^2));
    each layer's input is then bf16(sign(f) / sqrt(1 + eps/f^2) * w_pre[l])."""
    H, L, eps = 64, 3, 1e-6
    rs = np.random.RandomState(0)
    w_pre = (1.0 + 0.1 * rs.standard_normal((L, H))).astype(np.float32)
    for c in (1e-3, -2.5, 0.75):
        ctx = _bf16_bits(np.full((1, H), c))
        cb = _f64(ctx[0, :1])[0]
        fc, u = np.zeros((1, H), np.uint16), np.zeros((L, 1, H), np.uint16)
        oracle.lib().oracle_ctx_norms(1, H, L, eps, oracle._p(ctx), oracle._p(np.ones(H, np.float32)),
                                      oracle._p(w_pre), oracle._p(fc), oracle._p(u), None, None)
        f_want = _bits_of(np.full(H, np.sign(cb) / math.sqrt(1.0 + eps / cb ** 2)))
        assert np.array_equal(fc[0], f_want)
        f = _f64(f_want[:1])[0]
        for l in range(L):
            want = np.sign(f) / math.sqrt(1.0 + eps / f ** 2) * w_pre[l].astype(np.float64)
            assert np.array_equal(u[l, 0], _bits_of(want))


def test_norms_are_scale_free_without_eps():
    rs = np.random.RandomState(1)
    n, H, L, KVH, D = 3, 128, 2, 2, 32
    ctx = _bf16_bits(rs.standard_normal((n, H)))
    w_h = (1.0 + 0.1 * rs.standard_normal(H)).astype(np.float32)
    w_pre = (1.0 + 0.1 * rs.standard_normal((L, H))).astype(np.float32)
    w_kv = _bf16_bits(rs.standard_normal((L, 2 * KVH * D, H)) / 8)
    pos = np.arange(n)
    a = oracle.context_kv(ctx, pos, w_h, w_pre, w_kv, KVH, D, 0.0, 1e-6, 10000.0)
    b = oracle.context_kv(_bf16_bits(_f64(ctx) * 2.0 ** -7), pos, w_h, w_pre, w_kv, KVH, D, 0.0,
                          1e-6, 10000.0)
    for key in ("fc", "u", "kv", "k", "v"):
        assert np.array_equal(a[key], b[key]), key


def test_projection_is_a_library_matmul_per_layer():
    """kv[l] = u[l] . W_kv[l]^T with every fp64 sum exact, rounded once to bf16."""
    rs = np.random.RandomState(2)
    n, H, L, KVH, D = 4, 64, 3, 2, 16
    ctx = _bf16_bits(rs.standard_normal((n, H)))
    w_pre = (1.0 + 0.1 * rs.standard_normal((L, H))).astype(np.float32)
    w_kv = _bf16_bits(rs.standard_normal((L, 2 * KVH * D, H)) / 8)
    o = oracle.context_kv(ctx, np.zeros(n), np.ones(H, np.float32), w_pre, w_kv, KVH, D, 1e-6, 1e-6, 0.0)
    for l in range(L):
        assert np.array_equal(o["kv"][l], _bits_of(_f64(o["u"][l]) @ _f64(w_kv[l]).T))


# ------------------------------------------------------------- keys and values


def test_key_norm_of_constant_heads_and_values_pass_through():
    """A constant key head c normalises to bf16(sign(c) / sqrt(1 + qk_eps/c^2)) with no
    weight; position 0 (or theta = 0) leaves it unrotated; values are copied."""
    L, n, KVH, D, qk_eps = 2, 3, 2, 16, 1e-6
    rs = np.random.RandomState(3)
    kv = _kv_rows(rs, L, n, KVH, D)
    cs = rs.choice([1e-3, -0.5, 3.0], size=(L, n, KVH))
    for l in range(L):
        for r in range(n):
            for h in range(KVH):
                kv[l, r, h * D:(h + 1) * D] = _bf16_bits(np.full(D, cs[l, r, h]))
    for theta, pos in ((10000.0, np.zeros(n)), (0.0, np.arange(n) * 7)):
        k, v, _ = oracle.k_norm_rope(kv, pos, KVH, D, qk_eps, theta)
        for l in range(L):
            for r in range(n):
                for h in range(KVH):
                    c = _f64(kv[l, r, h * D:h * D + 1])[0]
                    want = np.sign(c) / math.sqrt(1.0 + qk_eps / c ** 2)
                    assert np.all(k[l, r, h] == _bits_of(want)), (l, r, h)
        assert np.array_equal(v.reshape(L, n, -1), kv[:, :, KVH * D:])


def test_one_hot_key_rotates_into_its_partner_dimension():
    """A key head with only dimension j set rotates into j and j + D/2 by the angle
    pos * theta^(-2j/D): (x cos, x sin); one with only j + D/2 set gives (-x sin, x cos).
    The normalised value x is bf16 before the rotation."""
    D, theta, qk_eps = 32, 500.0, 1e-6
    positions = np.array([0, 1, 3, 17, 250, 4095, 12345, 77777], np.int64)
    n = len(positions)
    for j in (0, 1, 5, D // 2 - 1):
        for lo in (True, False):
            dim = j if lo else j + D // 2
            kv = np.zeros((1, n, 2 * D), np.uint16)
            kv[0, :, dim] = _bf16_bits(np.full(n, 1.7))
            k, _, ke = oracle.k_norm_rope(kv, positions, 1, D, qk_eps, theta)
            x = _f64(_bits_of([1.7 / math.sqrt(1.7 ** 2 / D + qk_eps)]))[0]
            for r, p in enumerate(positions):
                ang = p * theta ** (-2.0 * j / D)
                a, b = (x * math.cos(ang), x * math.sin(ang)) if lo else (-x * math.sin(ang), x * math.cos(ang))
                got = k[0, r, 0]
                assert np.array_equal(_f64(got[[j, j + D // 2]]), _f64(_bits_of([a, b]))), (j, lo, p)
                others = np.delete(np.arange(D), [j, j + D // 2])
                assert not _f64(got[others]).any()          # zeros of either sign
                np.testing.assert_allclose(ke[0, r, 0, [j, j + D // 2]], [a, b], rtol=1e-12, atol=1e-12)


def test_rotation_keeps_pair_norms_and_depends_on_relative_position():
    """Before its rounding the rotation keeps every (j, j + D/2) pair's norm, and the
    dot product of two rotated keys depends only on their position difference."""
    D, KVH, theta = 64, 2, 10000.0
    rs = np.random.RandomState(4)
    kv = _kv_rows(rs, 1, 2, KVH, D)
    kv[0, 1] = kv[0, 0]
    _, _, base = oracle.k_norm_rope(kv, np.array([0, 0]), KVH, D, 1e-6, 0.0)
    dots = []
    for p0 in (0, 9, 1000):
        _, _, ke = oracle.k_norm_rope(kv, np.array([p0, p0 + 5]), KVH, D, 1e-6, theta)
        h = D // 2
        np.testing.assert_allclose(ke[0, 0, :, :h] ** 2 + ke[0, 0, :, h:] ** 2,
                                   base[0, 0, :, :h] ** 2 + base[0, 0, :, h:] ** 2, rtol=1e-12)
        dots.append(np.sum(ke[0, 0] * ke[0, 1], axis=-1))
    np.testing.assert_allclose(dots[1], dots[0], rtol=1e-10)
    np.testing.assert_allclose(dots[2], dots[0], rtol=1e-10)


def test_cache_scatter_by_brute_force():
    """Per-layer and shared slot maps; negative slots write nothing."""
    rs = np.random.RandomState(5)
    L, n, KVH, D, n_slots = 2, 5, 2, 8, 11
    k = rs.randint(0, 1 << 16, (L, n, KVH, D)).astype(np.uint16)
    v = rs.randint(0, 1 << 16, (L, n, KVH, D)).astype(np.uint16)
    kc0 = rs.randint(0, 1 << 16, (L, n_slots, KVH, D)).astype(np.uint16)
    vc0 = rs.randint(0, 1 << 16, (L, n_slots, KVH, D)).astype(np.uint16)
    shared = np.array([3, -1, 0, 10, 7], np.int64)
    per_layer = np.array([[2, 4, -1, 9, 0], [-1, -1, 5, 6, 1]], np.int64)
    for slots in (shared, per_layer):
        kc, vc = oracle.kv_cache_write(k, v, slots, n_slots, kc0, vc0)
        wk, wv = kc0.copy(), vc0.copy()
        for l in range(L):
            for r in range(n):
                s = slots[r] if slots.ndim == 1 else slots[l, r]
                if s >= 0:
                    wk[l, s], wv[l, s] = k[l, r], v[l, r]
        assert np.array_equal(kc, wk) and np.array_equal(vc, wv)


def test_key_tolerance_covers_one_step_projection_differences():
    """The end-to-end key tolerance of the GPU tests, 3 * 2^-7 of the pair's norm,
    holds when projection outputs move by one bf16 step (the staged GEMM check's
    allowance): the key norm carries the step, the casts before the rotation may
    round apart, the rotation keeps the difference's length and the final casts
    may add one more step.  Two steps (2^-6) do not suffice.  The differences are
    a fifth of the outputs here, far more than the staged check lets through, and
    still few enough that the head's RMS barely moves (a step in every output of
    a head, in opposite directions, could move it by up to one more step)."""
    rs = np.random.RandomState(6)
    L, n, KVH, D = 2, 64, 8, 128
    kv = _kv_rows(rs, L, n, KVH, D)
    pos = rs.randint(0, 32768, n)
    k0, _, _ = oracle.k_norm_rope(kv, pos, KVH, D, 1e-6, 10000.0)
    a = _f64(k0)
    h = D // 2
    pair = np.sqrt(a[..., :h] ** 2 + a[..., h:] ** 2)
    pair = np.concatenate([pair, pair], axis=-1)
    worst = 0.0
    for _ in range(20):
        kv1 = kv.copy()
        m = rs.rand(*kv.shape) < 0.2
        step = rs.choice([-1, 1], kv.shape)
        kv1[m] = (kv1[m].astype(np.int64) + step[m]).astype(np.uint16)
        k1, _, _ = oracle.k_norm_rope(kv1, pos, KVH, D, 1e-6, 10000.0)
        worst = max(worst, float(np.max(np.abs(_f64(k1) - a) / pair)))
    assert worst <= 3 * 2.0 ** -7
    assert worst > 2.0 ** -6
