"""The synthetic input recipe (no GPU): each generator draws the distribution,
shape and structure the workloads state, and independent tensors draw
independent values.

Shapes are the workloads' own; moments are checked to a few standard errors
of the sample.
"""
import numpy as np
import pytest

import synth


def _f64(bits):
    import torch
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).double().numpy()


def _moments_ok(v, mu, sigma, z=6.0):
    v = np.asarray(v, np.float64).ravel()
    n = v.size
    assert abs(v.mean() - mu) <= z * sigma / np.sqrt(n), (v.mean(), mu)
    assert abs(v.std() - sigma) <= z * sigma / np.sqrt(2 * n) + 0.004 * sigma, (v.std(), sigma)


def test_step_inputs_are_unit_normals_and_variants_differ():
    w = synth.WORKLOADS["serving"]
    stream, branch = synth.step_inputs(w, 0)
    assert stream.shape == (8, 7168) and stream.dtype == np.float32
    assert branch.shape == (8, 7168) and branch.dtype == np.uint16
    _moments_ok(stream, 0.0, 1.0)
    _moments_ok(_f64(branch), 0.0, 1.0)
    s1, b1 = synth.step_inputs(w, 1)
    assert not np.array_equal(s1, stream) and not np.array_equal(b1, branch)


def test_norm_router_and_expert_distributions():
    w = synth.WORKLOADS["serving"]
    for wt in synth.norm_weights(w, 0) + synth.final_norm_weights(w):
        _moments_ok(wt, 1.0, 0.1)
    _moments_ok(_f64(synth.router_weights(w, 0)), 0.0, 1.0 / 16.0)    # N(0, 1/256): variance
    t = synth.WORKLOADS["tiny"]
    g, u, d = (synth.expert_raw(t, 0, 3, k) for k in ("gate", "up", "down"))
    assert g.shape == (128, 256) and u.shape == (128, 256) and d.shape == (256, 128)
    for x in (g, u, d):
        _moments_ok(x, 0.0, 0.02)
    assert not np.array_equal(g, u)
    assert not np.array_equal(synth.expert_raw(t, 0, 3, "gate"), synth.expert_raw(t, 0, 4, "gate"))
    assert not np.array_equal(synth.expert_raw(t, 0, 3, "gate"), synth.expert_raw(t, 1, 3, "gate"))


def test_zipf_bias_is_a_permuted_power_law():
    w = synth.WORKLOADS["sweep"]
    b = synth.router_bias(w, 0)
    E = w.n_experts
    want = (2.0 * np.arange(1, E + 1, dtype=np.float64) ** -1.1).astype(np.float32)
    assert np.array_equal(np.sort(b)[::-1], want)
    assert b.max() == np.float32(2.0) and len(set(b.tolist())) == E
    assert not np.array_equal(b, want)                           # permuted, not sorted
    assert synth.router_bias(synth.WORKLOADS["serving"], 0) is None
    assert not np.array_equal(synth.router_bias(w, 1), b)


def test_dense_draft_weights():
    w = synth.DENSE_WORKLOADS["draft_dense_small"]
    w13, w2 = synth.dense_weights(w, 0)
    assert w13.shape == (2 * w.inter, w.hidden) and w2.shape == (w.hidden, w.inter)
    _moments_ok(_f64(w13), 0.0, 0.02)
    _moments_ok(_f64(w2), 0.0, 0.02)
    for wt in synth.dense_norm_weights(w, 0):
        _moments_ok(wt, 1.0, 0.1)


@pytest.mark.parametrize("name", ["draft_ctx_kv", "draft_ctx_kv_small"])
def test_context_kv_inputs(name):
    w = synth.CTXKV_WORKLOADS[name]
    for variant in range(4):
        ctx, pos, slots = synth.ctxkv_inputs(w, variant)
        assert ctx.shape == (w.n_ctx, w.hidden)
        assert np.array_equal(np.diff(pos), np.ones(w.n_ctx - 1)) and 0 <= pos[0]
        assert pos[-1] < w.max_position
        assert len(set(slots.tolist())) == w.n_ctx and slots.min() >= 0 and slots.max() < w.n_slots
    _moments_ok(_f64(synth.ctxkv_inputs(w.with_ctx(64), 0)[0]), 0.0, 1.0)
    wh, wp = synth.ctxkv_norm_weights(w)
    assert wp.shape == (w.n_layers, w.hidden)
    _moments_ok(wh, 1.0, 0.1)
    _moments_ok(wp, 1.0, 0.1)
    assert not np.array_equal(wp[0], wp[1])
    if name.endswith("small"):
        wkv = synth.ctxkv_weights(w)
        assert wkv.shape == (w.n_layers, 2 * w.n_kv_heads * w.head_dim, w.hidden)
        _moments_ok(_f64(wkv), 0.0, 0.02)
