"""Pins of the oracle's layer step (no GPU): closed forms of the dual norm,
library softmax and brute-force top-k for the routing, pooler invariants, and
the reduction of the routed experts to a dense gated MLP."""
import itertools

import numpy as np
import pytest
from scipy.special import softmax

import oracle
import synth
from helpers import oracle_weights, silu

TINY = synth.WORKLOADS["tiny"]


def _bf16_bits(a):
    import torch
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.uint16).numpy()


# ---------------------------------------------------------------- boundary


def test_zero_branch_leaves_stream_unchanged():
    s, _ = synth.step_inputs(TINY)
    w_post, w_pre = synth.norm_weights(TINY, 0)
    s2, x, xe = oracle.boundary(np.zeros_like(s, np.float64), s, w_post, w_pre, 1e-6)
    assert np.array_equal(s2, s)


def test_constant_rows_closed_form():
    H, eps = 64, 1e-6
    rs = np.random.RandomState(0)
    w_post = (1 + 0.1 * rs.standard_normal(H)).astype(np.float32)
    w_pre = (1 + 0.1 * rs.standard_normal(H)).astype(np.float32)
    c, sval = -0.7, 0.0
    branch = np.full((1, H), c)
    stream = np.full((1, H), sval, np.float32)
    s2, x, xe = oracle.boundary(branch, stream, w_post, w_pre, eps)
    # rmsnorm of a constant row c is sign(c) / sqrt(1 + eps / c^2)
    want_s = (np.sign(c) / np.sqrt(1 + eps / c ** 2) * w_post.astype(np.float64)).astype(np.float32)
    assert np.array_equal(s2[0], want_s)
    ms = np.mean(s2[0].astype(np.float64) ** 2)
    want_x = s2[0].astype(np.float64) / np.sqrt(ms + eps) * w_pre
    np.testing.assert_allclose(xe[0], want_x, rtol=1e-14)
    assert np.array_equal(x[0], [oracle.bf16_from_double(v) for v in want_x])


def test_norm_is_scale_free_without_eps():
    rs = np.random.RandomState(1)
    b = rs.standard_normal((3, 128))
    s = rs.standard_normal((3, 128)).astype(np.float32)
    w = np.ones(128, np.float32)
    s1, x1, _ = oracle.boundary(b, s, w, w, 0.0)
    s2, x2, _ = oracle.boundary(b * 2.0 ** 5, s, w, w, 0.0)
    assert np.array_equal(s1, s2) and np.array_equal(x1, x2)
    # the MoE input has unit rms before the weight and the bf16 rounding
    _, _, xe = oracle.boundary(b, s, w, w, 0.0)
    np.testing.assert_allclose(np.mean(xe ** 2, axis=1), 1.0, rtol=1e-12)


# ------------------------------------------------------------------ routing


def _route_case(rows, H, E, k, seed, bias=False):
    rs = np.random.RandomState(seed)
    x = _bf16_bits(rs.standard_normal((rows, H)))
    wr = _bf16_bits(rs.standard_normal((E, H)) / 16)
    b = rs.uniform(0, 2, E).astype(np.float32) if bias else None
    return x, wr, b


@pytest.mark.parametrize("bias", [False, True])
def test_k_equals_E_is_the_full_softmax(bias):
    rows, H, E = 5, 96, 6
    x, wr, b = _route_case(rows, H, E, E, 1, bias)
    r = oracle.route(x, wr, b, E)
    logits = oracle.bf16_to_f64(x) @ oracle.bf16_to_f64(wr).T
    if b is not None:
        logits = logits + b.astype(np.float64)
    p = softmax(logits, axis=1)
    np.testing.assert_allclose(r["logits"], logits, rtol=1e-12, atol=1e-12)
    for i in range(rows):
        order = sorted(range(E), key=lambda e: (-p[i, e], e))
        assert list(r["ids"][i]) == order
        np.testing.assert_allclose(r["gates"][i], p[i, order], rtol=1e-12)
        assert r["flags"][i] == 0


@pytest.mark.parametrize("k", [1, 2, 3])
def test_topk_brute_force_subsets(k):
    rows, H, E = 16, 64, 7
    x, wr, b = _route_case(rows, H, E, k, 2)
    r = oracle.route(x, wr, b, k)
    p = r["probs"]
    for i in range(rows):
        best = max(itertools.combinations(range(E), k), key=lambda S: sum(p[i, list(S)]))
        assert set(r["ids"][i]) == set(best)
        assert np.all(np.diff(p[i, r["ids"][i]]) <= 0)          # slots by descending p
        assert abs(r["gates"][i].sum() - 1.0) < 1e-12
        sp = np.sort(p[i])[::-1]
        assert r["gap"][i] == pytest.approx(sp[k - 1] - sp[k], abs=1e-15)


def test_ties_go_to_the_lower_expert_and_are_flagged():
    rows, H, E, k = 2, 32, 5, 2
    x, wr, _ = _route_case(rows, H, E, k, 3)
    wr[3] = wr[1]          # experts 1 and 3 always tie
    wr[4] = wr[0]
    r = oracle.route(x, wr, None, k)
    for i in range(rows):
        ids = list(r["ids"][i])
        if 1 in ids or 3 in ids:
            assert not (3 in ids and 1 not in ids)
        if 0 in ids or 4 in ids:
            assert not (4 in ids and 0 not in ids)
    # make the tie sit exactly at the k/k+1 boundary
    wr2 = np.zeros((3, H), np.uint16)
    wr2[0] = x[0]                           # logit |x|^2 > 0 = the other two
    r = oracle.route(x[:1], wr2, None, 2)   # experts 1 and 2 tie for the second slot
    assert list(r["ids"][0])[1] == 1 and r["flags"][0] == 1 and r["gap"][0] == 0.0


def _bf16_f64(bits):
    import torch
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).double().numpy()


def test_front_stream_is_the_embedding_exactly():
    rs = np.random.RandomState(3)
    emb = _bf16_bits(rs.standard_normal((5, 96)) * 3.0)
    w = (1.0 + 0.1 * rs.standard_normal(96)).astype(np.float32)
    stream, out, _ = oracle.front(emb, w, 1e-6)
    np.testing.assert_array_equal(stream.astype(np.float64), _bf16_f64(emb))


def test_front_constant_rows_closed_form():
    """A row of constant c: rms = |c|, so out = bf16(sign(c) * w / sqrt(1 + eps/c^2));
    c = 1e-3 makes eps/c^2 = 1 (the eps term matters)."""
    H, eps = 64, 1e-6
    rs = np.random.RandomState(4)
    w = (1.0 + 0.1 * rs.standard_normal(H)).astype(np.float32)
    cs = [1e-3, -2.5, 7.0]
    emb = _bf16_bits(np.array([[c] * H for c in cs]))
    _, out, exact = oracle.front(emb, w, eps)
    for i in range(len(cs)):
        c = _bf16_f64(emb[i, :1])[0]
        want = np.sign(c) * w.astype(np.float64) / np.sqrt(1.0 + eps / (c * c))
        np.testing.assert_allclose(exact[i], want, rtol=1e-12)
        np.testing.assert_array_equal(out[i], _bf16_bits(want.astype(np.float32)))


def test_front_is_scale_free_without_eps():
    """Doubling the input (exact in bf16) leaves the normalised output bit
    for bit unchanged when eps = 0."""
    rs = np.random.RandomState(5)
    emb = _bf16_bits(rs.standard_normal((4, 128)))
    emb2 = _bf16_bits(_bf16_f64(emb) * 2.0)
    w = (1.0 + 0.1 * rs.standard_normal(128)).astype(np.float32)
    s1, out1, _ = oracle.front(emb, w, 0.0)
    s2, out2, _ = oracle.front(emb2, w, 0.0)
    np.testing.assert_array_equal(s2, 2.0 * s1)
    np.testing.assert_array_equal(out1, out2)


def test_near_tie_flag_is_the_gap_below_1e6():
    """With x = 0 the logits are the biases exactly; experts 0 and 1 lead,
    the rest are negligible.  The k-th/(k+1)-th probability gap is then the
    closed-form softmax gap, and the row is flagged exactly when it is below
    1e-6 (gaps of about 1e-5, 2e-6 and 5e-7)."""
    E, k, H = 4, 1, 16
    x = np.zeros((3, H), np.uint16)                  # bf16 +0
    wr = np.zeros((E, H), np.uint16)
    for delta, flagged in ((2e-5, 0), (4e-6, 0), (1e-6, 1)):
        bias = np.array([0.0, -delta, -40.0, -40.0], np.float32)
        r = oracle.route(x[:1], wr, bias, k)
        lg = bias.astype(np.float64)
        p = np.exp(lg - lg.max())
        p /= p.sum()
        assert list(r["ids"][0]) == [0]
        assert r["gap"][0] == pytest.approx(p[0] - p[1], rel=1e-9)
        assert int(r["flags"][0]) == flagged, (delta, r["gap"][0])


# ------------------------------------------------------------------- pooler


@pytest.mark.parametrize("rows,E,k", [(13, 9, 3), (2, 9, 2)])
def test_pooler_invariants(rows, E, k):
    """Counts, offsets and pair order by brute force; the second shape leaves
    most experts idle, so the active list must skip them."""
    rs = np.random.RandomState(4)
    ids = np.array([rs.choice(E, k, replace=False) for _ in range(rows)], np.int32)
    pl = oracle.pool(ids, E)
    assert pl["count"].sum() == rows * k
    assert np.array_equal(pl["offset"], np.concatenate([[0], np.cumsum(pl["count"])]))
    assert sorted(pl["pair_order"]) == list(range(rows * k))
    flat = ids.reshape(-1)
    exp_of = flat[pl["pair_order"]]
    assert np.all(np.diff(exp_of) >= 0)
    for e in range(E):
        seg = pl["pair_order"][pl["offset"][e]:pl["offset"][e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg // k) > 0)
    assert list(pl["active"]) == [e for e in range(E) if pl["count"][e] > 0]


# ------------------------------------------------------------------ experts


def _dense_moe_output(wts, e, xq, rows_of_e):
    """Dense gated MLP of expert e on the dequantized MoE input rows; h is one
    NVFP4 tensor over exactly the given rows (as the routed step quantizes it)."""
    H, I = wts.H, wts.I
    w13 = oracle.nvfp4_dequantize(wts.w13[e][:I], wts.w13_sf[e][:I], wts.gscale[e, 0], I, H)
    w13u = oracle.nvfp4_dequantize(wts.w13[e][I:], wts.w13_sf[e][I:], wts.gscale[e, 1], I, H)
    w2 = oracle.nvfp4_dequantize(wts.w2[e], wts.w2_sf[e], wts.gscale[e, 2], H, I)
    xr = xq[rows_of_e]
    h = (silu(xr @ w13.T) * (xr @ w13u.T)).astype(np.float32)
    hc, hs, hg, _ = oracle.nvfp4_quantize(h)
    hh = oracle.nvfp4_dequantize(hc, hs, hg, len(rows_of_e), I)
    return hh @ w2.T


def _layer_case(w, layer=0):
    wts = oracle_weights(w, layer)
    stream, branch = synth.step_inputs(w)
    return wts, stream, oracle.bf16_to_f64(branch)


def test_single_expert_with_gate_one_is_a_dense_gated_mlp():
    w = synth.Workload("one", rows=6, hidden=64, n_experts=1, top_k=1, inter=48)
    wts, stream, branch = _layer_case(w)
    out = oracle.layer_step(wts, 1, w.eps, branch, stream)
    assert np.all(out["gates"] == 1.0) and np.all(out["ids"] == 0)
    xq = oracle.nvfp4_dequantize(out["x_codes"], out["x_sf"], out["x_sg"], w.rows, w.hidden)
    dense = _dense_moe_output(wts, 0, xq, np.arange(w.rows))
    # o is stored in fp32: one rounding (half an ulp, 2^-24 relative) apart
    np.testing.assert_allclose(out["o"], dense, rtol=2.0 ** -23, atol=1e-12 * np.abs(dense).max())


def test_every_expert_selected_matches_gated_dense_sum():
    w = synth.Workload("two", rows=5, hidden=96, n_experts=2, top_k=2, inter=32)
    wts, stream, branch = _layer_case(w)
    out = oracle.layer_step(wts, 2, w.eps, branch, stream)
    xq = oracle.nvfp4_dequantize(out["x_codes"], out["x_sf"], out["x_sg"], w.rows, w.hidden)
    dense = {e: _dense_moe_output(wts, e, xq, np.arange(w.rows)) for e in range(2)}
    y = oracle.gather(out["gates"], out["o"], 2)
    want = np.zeros_like(y)
    for r in range(w.rows):
        for s in range(2):
            want[r] += out["gates"][r, s] * dense[out["ids"][r, s]][r]
    # each o term carries one fp32 rounding; the two gated terms may cancel
    np.testing.assert_allclose(y, want, rtol=2.0 ** -22, atol=2.0 ** -23 * np.abs(out["o"]).max())


def test_row_permutation_permutes_outputs():
    wts, stream, branch = _layer_case(TINY)
    a = oracle.layer_step(wts, TINY.top_k, TINY.eps, branch, stream)
    perm = np.random.RandomState(5).permutation(TINY.rows)
    b = oracle.layer_step(wts, TINY.top_k, TINY.eps, branch[perm], stream[perm])
    assert np.array_equal(a["stream"][perm], b["stream"])
    assert np.array_equal(a["ids"][perm], b["ids"])
    np.testing.assert_array_equal(a["gates"][perm], b["gates"])
    k = TINY.top_k
    pairs = (perm[:, None] * k + np.arange(k)).reshape(-1)
    np.testing.assert_array_equal(a["o"][pairs], b["o"])
    ya = oracle.gather(a["gates"], a["o"], k)
    yb = oracle.gather(b["gates"], b["o"], k)
    np.testing.assert_array_equal(ya[perm], yb)


def test_zero_experts_give_zero_output_and_unchanged_next_stream():
    wts, stream, branch = _layer_case(TINY)
    for e in wts.w2:
        wts.w2[e][:] = 0
    wts._struct = None
    out = oracle.layer_step(wts, TINY.top_k, TINY.eps, branch, stream)
    assert not out["o"].any()
    y = oracle.gather(out["gates"], out["o"], TINY.top_k)
    w_post, w_fin = synth.final_norm_weights(TINY)
    s2, _, _ = oracle.boundary(y, out["stream"], w_post, w_fin, TINY.eps)
    assert np.array_equal(s2, out["stream"])


def test_forced_ids_reproduce_own_choice_and_renormalise():
    wts, stream, branch = _layer_case(TINY)
    a = oracle.layer_step(wts, TINY.top_k, TINY.eps, branch, stream)
    b = oracle.layer_step(wts, TINY.top_k, TINY.eps, branch, stream, forced_ids=a["ids"])
    np.testing.assert_array_equal(a["o"], b["o"])
    rev = a["ids"][:, ::-1].copy()
    c = oracle.layer_step(wts, TINY.top_k, TINY.eps, branch, stream, forced_ids=rev)
    np.testing.assert_allclose(c["gates"], a["gates"][:, ::-1], rtol=1e-15)


def test_tiny_layer_statistics():
    wts, stream, branch = _layer_case(TINY)
    out = oracle.layer_step(wts, TINY.top_k, TINY.eps, branch, stream)
    assert np.allclose(out["gates"].sum(1), 1.0, atol=1e-12)
    assert out["n_active"] == len(set(out["ids"].reshape(-1)))
    assert np.all(np.isfinite(out["o"])) and np.abs(out["o"]).max() > 0
    # every pair's h tensor scale is that expert's amax / 2688
    for e in out["active"]:
        assert out["h_sg"][e] == np.float32(out["h_amax"][e] / np.float32(2688.0))


def test_chained_layers_amplify_a_one_ulp_input_change():
    """Why a chained step is checked layer by layer from the GPU's own state
    at each layer's entry, not end to end from the step's inputs (R32): the
    chain is ill-conditioned.  The oracle run twice over the same eight
    chained layers (H 1024, 16 experts, top-8, I 256), the second time from a
    stream one fp32 ulp up and with the first run's expert ids forced, agrees
    with itself after the first layer to about 1e-6 of the stream's rms, yet
    ends far more than the end-to-end tolerance (2e-3 * rms) apart after the
    eighth: each NVFP4 quantization -- a code, a block scale, and above all a
    per-expert tensor scale of h -- turns a sub-ulp difference into a whole
    quantization step, and the next boundary's rmsnorm(y) carries it into the
    stream at full size.  An fp32 evaluation differs from the fp64 oracle by
    at least one ulp, so the tolerance can hold per layer, not over the
    chain."""
    w = synth.Workload("chain8_small", rows=8, hidden=1024, n_experts=16, top_k=8, inter=256,
                       n_layers=8)
    ows = [oracle_weights(w, l) for l in range(w.n_layers)]
    s0, b0 = synth.step_inputs(w, 0)

    def run(s, forced=None):
        br, outs = oracle.bf16_to_f64(b0), []
        for l in range(w.n_layers):
            o = oracle.layer_step(ows[l], w.top_k, w.eps, br, s,
                                  forced_ids=None if forced is None else forced[l])
            outs.append(o)
            s, br = o["stream"], oracle.gather(o["gates"], o["o"], w.top_k)
        return outs

    a = run(s0)
    b = run(np.nextafter(s0, np.float32(np.inf)).astype(np.float32), [o["ids"] for o in a])

    def rel(l):
        sa = a[l]["stream"].astype(np.float64)
        return np.max(np.abs(sa - b[l]["stream"])) / np.sqrt(np.mean(sa ** 2))

    assert rel(0) < 1e-5
    assert rel(w.n_layers - 1) > 10 * 2e-3
    # the growth passes through a changed h tensor scale on the way
    assert any(not np.array_equal(a[l]["h_sg"], b[l]["h_sg"]) for l in range(w.n_layers))


def test_moe_step_is_layer_step_after_its_boundary():
    """The MoE part alone, from the boundary's bf16 output, reproduces every
    intermediate of the whole layer bit for bit (the same arithmetic)."""
    w = synth.Workload("moe_part", rows=6, hidden=512, n_experts=12, top_k=3, inter=256)
    ow = oracle_weights(w, 0)
    s0, b0 = synth.step_inputs(w, 0)
    full = oracle.layer_step(ow, w.top_k, w.eps, oracle.bf16_to_f64(b0), s0)
    part = oracle.moe_step(ow, w.top_k, full["x"])
    for name in ("ids", "gates", "flags", "x_codes", "x_sf", "x_sg", "count", "offset", "pair_order",
                 "active", "h", "h_codes", "h_sf", "h_sg", "o"):
        assert np.array_equal(np.asarray(full[name]), np.asarray(part[name])), name
    forced = np.roll(full["ids"], 1, axis=1)
    a = oracle.layer_step(ow, w.top_k, w.eps, oracle.bf16_to_f64(b0), s0, forced_ids=forced)
    b = oracle.moe_step(ow, w.top_k, a["x"], forced_ids=forced)
    assert np.array_equal(a["gates"], b["gates"]) and np.array_equal(a["o"], b["o"])


def test_one_ulp_moe_input_change_moves_the_experts_past_the_tolerance():
    """Why a layer's end-to-end check continues from the GPU's MoE input where
    the oracle's differs from it at a bf16 rounding midpoint (R34): one
    element of x moved by one bf16 ulp -- the size of such a difference --
    flips its NVFP4 code when it sits at a code boundary, and that moves the
    layer's expert outputs by far more than the end-to-end tolerance
    (2e-3 * rms): h changes, its per-expert NVFP4 tensor is re-quantized, and
    whole quantization steps follow."""
    w = synth.Workload("moe_ulp", rows=4, hidden=1024, n_experts=8, top_k=2, inter=256)
    ow = oracle_weights(w, 0)
    s0, b0 = synth.step_inputs(w, 0)
    a = oracle.layer_step(ow, w.top_k, w.eps, oracle.bf16_to_f64(b0), s0)
    rms = np.sqrt(np.mean(a["o"].astype(np.float64) ** 2))
    worst, flips = 0.0, 0
    for r in range(w.rows):
        for col in range(0, w.hidden, 3):
            x = a["x"].copy()
            x[r, col] = np.uint16(x[r, col] + 1)  # one bf16 ulp (away from zero)
            b = oracle.moe_step(ow, w.top_k, x, forced_ids=a["ids"])
            if np.array_equal(a["x_codes"], b["x_codes"]) and np.array_equal(a["x_sf"], b["x_sf"]):
                continue                           # most such changes leave every code alone
            flips += 1
            worst = max(worst, float(np.max(np.abs(a["o"].astype(np.float64) - b["o"]))) / rms)
        if flips >= 6:
            break
    assert flips >= 3
    assert worst > 5 * 2e-3
