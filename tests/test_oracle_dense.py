"""Pins of the oracle's dense draft layer (no GPU).

The layer (the DSpark page, MuseSparkDSparkDecoderLayer.forward) adds the
normalised attention output to the fp32 stream, normalises the stream cast to
bf16 as the MLP input, runs the gated bf16 MLP and adds its normalised output.
Each pin fixes one part by something other than the oracle itself: closed
forms of the norms on constant rows, the bf16 cast before the input norm on a
two-valued row, library matmuls where every fp64 sum is exact, single-entry
weights that make each MLP output one named product, and scale invariance
without eps.
"""
import numpy as np

import oracle
from helpers import silu


def _bf16_bits(a):
    import torch
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.uint16).numpy()


def _f64(bits):
    return oracle.bf16_to_f64(np.asarray(bits, np.uint16))


def _bits_of(v):
    return np.array([oracle.bf16_from_double(float(t)) for t in np.ravel(v)],
                    np.uint16).reshape(np.shape(v))


def _case(rows, H, I, seed, w_scale=2.0 ** -3):
    """Random operands whose products and sums are exact in fp64: bf16 values of
    a few binades, H and I small, so any summation order gives the same sum."""
    rs = np.random.RandomState(seed)
    attn = _bf16_bits(rs.standard_normal((rows, H)))
    stream = rs.standard_normal((rows, H)).astype(np.float32)
    w13 = _bf16_bits(rs.standard_normal((2 * I, H)) * w_scale)
    w2 = _bf16_bits(rs.standard_normal((H, I)) * w_scale)
    norms = [(1.0 + 0.1 * rs.standard_normal(H)).astype(np.float32) for _ in range(3)]
    return attn, stream, w13, w2, norms


def _run(attn, stream, w13, w2, norms, eps=1e-6):
    return oracle.dense_layer(attn, stream, norms[0], norms[1], w13, w2, norms[2], eps)


def test_zero_attention_and_zero_down_leave_the_stream_unchanged():
    attn, stream, w13, w2, norms = _case(3, 64, 32, 0)
    o = _run(np.zeros_like(attn), stream, w13, np.zeros_like(w2), norms)
    assert np.array_equal(o["stream"], stream)
    assert not o["f"].any()


def test_post_attention_norm_of_constant_rows_closed_form():
    """attn = c: rmsnorm gives sign(c) / sqrt(1 + eps/c^2); c = 1e-3 makes the
    eps term as large as the mean square.  A zero down projection leaves s1."""
    H, I, eps = 64, 16, 1e-6
    _, _, w13, w2, norms = _case(1, H, I, 1)
    for c in (1e-3, -0.75, 5.0):
        attn = _bf16_bits(np.full((1, H), c))
        cb = _f64(attn[0, :1])[0]
        o = _run(attn, np.zeros((1, H), np.float32), w13, np.zeros_like(w2), norms, eps)
        want = np.sign(cb) / np.sqrt(1.0 + eps / cb ** 2) * norms[0].astype(np.float64)
        assert np.array_equal(o["stream"][0], want.astype(np.float32))


def test_mlp_input_normalises_the_stream_cast_to_bf16():
    """A stream row of 1 + 2^-8 (exactly halfway between bf16 neighbours, rounds
    to even 1) and 3: the cast row has mean square 5, so the MLP input is
    bf16(v / sqrt(5 + eps) * w_pre) with v = 1 or 3.  Normalising the fp32 row
    instead changes the mean square by about 2^-9 and flips many roundings."""
    H, I, eps = 256, 16, 1e-6
    _, _, w13, w2, norms = _case(1, H, I, 2)
    row = np.concatenate([np.full(H // 2, 1.0 + 2.0 ** -8), np.full(H // 2, 3.0)])
    o = _run(np.zeros((1, H), np.uint16), row[None].astype(np.float32), w13, w2, norms, eps)
    v = np.concatenate([np.ones(H // 2), np.full(H // 2, 3.0)])
    want = v / np.sqrt(5.0 + eps) * norms[1].astype(np.float64)
    assert np.array_equal(o["x"][0], _bits_of(want))


def test_projections_are_library_matmuls_over_exact_sums():
    """gate/up = W13 x and f = W2 a with every product and sum exact in fp64,
    so numpy's matmul gives the same sums; each rounded once to bf16."""
    rows, H, I = 3, 64, 48
    attn, stream, w13, w2, norms = _case(rows, H, I, 3)
    o = _run(attn, stream, w13, w2, norms)
    gu = _f64(o["x"]) @ _f64(w13).T
    assert np.array_equal(o["gu"], _bits_of(gu))
    f = _f64(o["a"]) @ _f64(w2).T
    assert np.array_equal(o["f"], _bits_of(f))


def test_single_entry_weights_name_each_product():
    """Gate row j reads x[c_j], up row j reads 2 * x[d_j], down row i reads a[j_i]:
    g_j = x[c_j], u_j = 2 x[d_j], a_j = bf16(silu(g_j) u_j), f_i = a[j_i] / 4.
    Gate rows come first in w13, then up rows; w2 is [hidden][inter]."""
    H, I = 64, 8
    attn, stream, _, _, norms = _case(2, H, I, 4)
    rs = np.random.RandomState(5)
    c, d = rs.choice(H, I, replace=False), rs.choice(H, I, replace=False)
    w13 = np.zeros((2 * I, H), np.float32)
    w13[np.arange(I), c] = 1.0
    w13[I + np.arange(I), d] = 2.0
    ji = rs.randint(0, I, H)
    w2 = np.zeros((H, I), np.float32)
    w2[np.arange(H), ji] = 0.25
    o = _run(attn, stream, _bf16_bits(w13), _bf16_bits(w2), norms)
    x = _f64(o["x"])
    g, u = x[:, c], 2.0 * x[:, d]
    assert np.array_equal(o["gu"], _bits_of(np.concatenate([g, u], axis=1)))
    a_bits = _bits_of(silu(g) * u)
    assert np.array_equal(o["a"], a_bits)
    assert np.array_equal(o["f"], _bits_of(_f64(a_bits)[:, ji] * 0.25))


def test_output_norm_of_a_constant_down_projection():
    """All-equal f = v per row: the output branch is sign(v) / sqrt(1 + eps/v^2)
    times w_post_ffn, added to s1 in fp32 (read back from a run with zero W2)."""
    H, I, eps = 64, 8, 1e-6
    attn, stream, _, _, norms = _case(1, H, I, 6)
    w13 = np.zeros((2 * I, H), np.float32)
    w13[:, 0] = 1.0                     # g = u = x[0] for every j
    w2 = np.zeros((H, I), np.float32)
    w2[:, 0] = 1.0                      # f_i = a_0 for every i
    o = _run(attn, stream, _bf16_bits(w13), _bf16_bits(w2), norms, eps)
    s1 = _run(attn, stream, _bf16_bits(w13), np.zeros((H, I), np.uint16), norms, eps)["stream"]
    v = _f64(o["f"][0, :1])[0]
    assert v != 0.0 and np.all(o["f"][0] == o["f"][0, 0])
    want = s1[0].astype(np.float64) + np.sign(v) / np.sqrt(1.0 + eps / v ** 2) * norms[2].astype(np.float64)
    assert np.array_equal(o["stream"][0], want.astype(np.float32))


def test_scale_free_without_eps():
    """Without eps, scaling the attention output or the down weights by a power of
    two changes no result after the norms: every rounding scales exactly."""
    attn, stream, w13, w2, norms = _case(2, 64, 32, 7)
    base = _run(attn, stream, w13, w2, norms, eps=0.0)
    big_attn = _bf16_bits(_f64(attn) * 2.0 ** 6)
    small_w2 = _bf16_bits(_f64(w2) * 2.0 ** -4)
    o = _run(big_attn, stream, w13, small_w2, norms, eps=0.0)
    assert np.array_equal(o["stream"], base["stream"]) and np.array_equal(o["x"], base["x"])
    assert np.array_equal(_f64(o["f"]), _f64(base["f"]) * 2.0 ** -4)
