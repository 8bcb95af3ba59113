"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle.

Staged checks feed each oracle stage the GPU's own output of the stage before
(the ids, the MoE input's codes, h), so every integer decision is compared bit
for bit and every floating-point stage against a tight tolerance; the
end-to-end checks run the oracle independently and apply the workload's
stream tolerance max|err| <= 2e-3 * rms(stream).  Rows whose k-th/(k+1)-th
router-probability gap is below 1e-6 are flagged and excluded from id checks.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import (bf16_near_tie, check_gpu_weights, dev_array, expert_subproblem, gpu_layer_weights,
                     oracle_weights, read_debug)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

STREAM_TOL = 2e-3          # end-to-end: max|err| <= STREAM_TOL * rms(stream)
STAGE_TOL = 1e-4           # staged floats: max|err| <= STAGE_TOL * rms(reference)


def _rms(a):
    return float(np.sqrt(np.mean(np.asarray(a, np.float64) ** 2)))


def _close(got, ref, tol, what):
    err = float(np.max(np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64)))) if np.size(ref) else 0.0
    bound = tol * max(_rms(ref), 1e-30)
    assert err <= bound, f"{what}: max|err| {err:.3e} > {bound:.3e}"
    return err


def _bf16_f32(bits):
    return oracle.bf16_to_f64(bits).astype(np.float32)


def _sgpu():
    import synth.gpu as sgpu
    return sgpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import speculative_decode_routed_gb300 as moe
    moe.lib()
    yield


# ----------------------------------------------------------------- pieces


@pytest.mark.parametrize("shape,scale", [((1, 16), 1.0), ((3, 48), 1e-3), ((64, 256), 0.02),
                                         ((7, 7168), 3.0), ((128, 2048), 1e4)])
def test_quantizer_bit_exact(shape, scale):
    import speculative_decode_routed_gb300 as moe
    rs = np.random.RandomState(sum(shape))
    v = (rs.standard_normal(shape) * scale).astype(np.float32)
    v[0, :16] = 0.0                                     # a zero block
    if shape[1] >= 32:
        v[-1, 16:32] = np.float32(scale) * np.array([6, 5, 3.5, 2.5, 1.75, 1.25, 0.75, 0.25] * 2)
    codes, sf, sg, amax = oracle.nvfp4_quantize(v)
    tv = torch.from_numpy(v).cuda()
    tc = torch.empty(shape[0], shape[1] // 2, dtype=torch.uint8, device="cuda")
    ts = torch.empty(shape[0], shape[1] // 16, dtype=torch.uint8, device="cuda")
    tg = torch.empty(1, device="cuda")
    ta = torch.empty(1, device="cuda")
    moe.moe_nvfp4_quantize(tv, tc, ts, tg, ta)
    torch.cuda.synchronize()
    assert ta.item() == amax and tg.item() == sg
    assert np.array_equal(ts.cpu().numpy(), sf)
    assert np.array_equal(tc.cpu().numpy(), codes)


def test_quantizer_zero_tensor():
    import speculative_decode_routed_gb300 as moe
    tv = torch.zeros(4, 64, device="cuda")
    tc = torch.full((4, 32), 0xAB, dtype=torch.uint8, device="cuda")
    ts = torch.full((4, 4), 0xAB, dtype=torch.uint8, device="cuda")
    tg = torch.full((1,), 7.0, device="cuda")
    ta = torch.full((1,), 7.0, device="cuda")
    moe.moe_nvfp4_quantize(tv, tc, ts, tg, ta)
    torch.cuda.synchronize()
    assert tg.item() == 0.0 and ta.item() == 0.0
    assert not tc.any().item() and not ts.any().item()


def test_device_generator_bit_exact():
    for tg, (mu, sd), n in ((synth.tag(synth.KIND_GATE, 2, 17), (0.0, 0.02), 100003),
                            (synth.tag(synth.KIND_W_PRE, 0), (1.0, 0.1), 4096)):
        t = torch.empty(n, device="cuda")
        synth.dev_normal_f32(t, 0, tg, mu, sd)
        assert np.array_equal(t.cpu().numpy(), synth.normal_f32((n,), 0, tg, mu, sd))
    b = torch.empty(5000, dtype=torch.bfloat16, device="cuda")
    synth.dev_normal_bf16(b, 3, 9)
    assert np.array_equal(b.view(torch.uint16).cpu().numpy(), synth.normal_bf16((5000,), 3, 9))


# -------------------------------------------------------- staged layer check


def check_stages(w, d, ow, experts, br, s_in, s_out, rows):
    """Every stage of one layer the GPU ran, each against the oracle's stage on
    the GPU's own input to it.  d: the layer's debug arrays (read_debug); ow:
    oracle.LayerWeights holding at least `experts` ("all": every active one);
    br: the branch (fp64) the layer's boundary added; s_in / s_out: the stream
    before and after the layer."""
    k, E, I = w.top_k, w.n_experts, w.inter
    # A: dual-norm boundary
    s_ref, x_ref, xe = oracle.boundary(br, s_in, ow.w_post, ow.w_pre, w.eps)
    _close(s_out, s_ref, 1e-5, "stream after the boundary")
    diff = d["x"] != x_ref
    assert not np.any(diff & ~bf16_near_tie(xe)), "MoE input differs away from bf16 near-ties"
    assert np.mean(diff) < 1e-3

    # B: router, routing, pooler, activation quantization (from the GPU's x)
    r = oracle.route(d["x"], ow.router_w, ow.router_bias, k)
    ok_rows = r["flags"] == 0
    assert np.array_equal(d["ids"][ok_rows], r["ids"][ok_rows]), "expert ids"
    np.testing.assert_allclose(d["gates"][ok_rows], r["gates"][ok_rows], atol=1e-5)
    np.testing.assert_allclose(d["gates"].sum(1), 1.0, atol=1e-6)
    _close(d["logits"], r["logits"], 1e-5, "router logits")
    pl = oracle.pool(d["ids"], E)
    for key in ("count", "offset", "pair_order"):
        assert np.array_equal(d[key], pl[key]), key
    assert d["n_active"] == pl["n_active"] and np.array_equal(d["active"], pl["active"])
    xc, xs, xg, _ = oracle.nvfp4_quantize(_bf16_f32(d["x"]))
    assert d["x_sg"] == xg and np.array_equal(d["x_sf"], xs) and np.array_equal(d["x_codes"], xc)

    # C-E: experts, per expert, on the GPU's own stage inputs
    active = list(d["active"]) if experts == "all" else [e for e in experts if d["count"][e] > 0]
    for e in active:
        p0, p1 = d["offset"][e], d["offset"][e + 1]
        pairs = d["pair_order"][p0:p1]
        n = p1 - p0
        sub = expert_subproblem(ow, e)
        zi, off, order = np.zeros((n, 1), np.int32), np.array([0, n], np.int32), np.arange(n, dtype=np.int32)
        rws = pairs // k
        h_ref = oracle.gate_up(sub, 1, d["x_codes"][rws], d["x_sf"][rws], d["x_sg"], zi, off, order)
        _close(d["h"][p0:p1], h_ref, STAGE_TOL, f"h of expert {e}")
        hq = oracle.h_quant(1, I, off, d["h"][p0:p1])
        assert d["h_sg"][e] == hq["h_sg"][0], f"h scale of expert {e}"
        assert np.array_equal(d["h_sf"][p0:p1], hq["h_sf"]), f"h block scales of expert {e}"
        assert np.array_equal(d["h_codes"][p0:p1], hq["h_codes"]), f"h codes of expert {e}"
        o_ref = oracle.down(sub, 1, zi, off, order, d["h_codes"][p0:p1], d["h_sf"][p0:p1],
                            np.array([d["h_sg"][e]], np.float32))
        _close(d["o"][pairs], o_ref, STAGE_TOL, f"o of expert {e}")


def staged_layer(w, dec, ow, layer, rows, branch, stream, experts="all", prev=None):
    """Run one layer on the GPU and check every stage.  branch: bf16 CUDA tensor,
    or None (chained: the previous layer's unpooled output, from `prev`).
    `ow` is oracle.LayerWeights, or a function of the GPU's debug data that
    returns (LayerWeights, experts to check) -- for sampling at full size."""
    k = w.top_k
    s_in = stream.cpu().numpy().copy()
    dec.layer(layer, rows, branch, stream)
    torch.cuda.synchronize()
    dec.check()
    d = read_debug(dec, rows)
    if callable(ow):
        ow, experts = ow(d)
    if branch is not None:
        br = oracle.bf16_to_f64(branch.view(torch.uint16).cpu().numpy())
    else:
        br = oracle.gather(prev["gates"].astype(np.float64), prev["o"], k)
    d["stream"] = stream.cpu().numpy().copy()
    check_stages(w, d, ow, experts, br, s_in, d["stream"], rows)
    return d


def _final_check(w, dec, d, rows, stream):
    wpf, wf = synth.final_norm_weights(w)
    out = torch.empty(rows, w.hidden, dtype=torch.bfloat16, device="cuda")
    s_in = stream.cpu().numpy().copy()
    dec.final(rows, stream, out)
    torch.cuda.synchronize()
    y = oracle.gather(d["gates"].astype(np.float64), d["o"], w.top_k)
    s_ref, out_ref, oe = oracle.boundary(y, s_in, wpf, wf, w.eps)
    _close(stream.cpu().numpy(), s_ref, 1e-5, "stream after the final boundary")
    got = out.view(torch.uint16).cpu().numpy()
    assert not np.any((got != out_ref) & ~bf16_near_tie(oe)), "final output away from near-ties"
    assert np.mean(got != out_ref) < 1e-3


def _check_weights(dec, ow, layer, experts):
    check_gpu_weights(dec, ow, layer, experts)


# ---------------------------------------------------------------- end to end


def run_step_layerwise(w, dec, rows, branch, stream, out, keep_debug=()):
    """The step as moe_decode_step launches it -- every layer, then the final
    boundary, the same kernels in the same order -- one layer call at a time,
    keeping each layer's routing, MoE input, gates, unpooled outputs and the
    stream around it (and the whole debug view of the layers in keep_debug)."""
    k, H = w.top_k, w.hidden
    per = []
    for l in range(w.n_layers):
        s_in = stream.cpu().numpy().copy()
        dec.layer(l, rows, branch if l == 0 else None, stream)
        torch.cuda.synchronize()
        if l in keep_debug:
            d = read_debug(dec, rows)
        else:
            v = dec.debug()
            d = dict(ids=dev_array(v.ids, (rows, k), np.int32), x=dev_array(v.x, (rows, H), np.uint16),
                     gates=dev_array(v.gates, (rows, k), np.float32),
                     o=dev_array(v.o, (rows * k, H), np.float32),
                     n_active=int(dev_array(v.n_active, (1,), np.int32)[0]))
            d["active"] = dev_array(v.active, (w.n_experts,), np.int32)[: d["n_active"]]
        d["stream_in"], d["stream"] = s_in, stream.cpu().numpy().copy()
        per.append(d)
    s_final_in = stream.cpu().numpy().copy()
    dec.final(rows, stream, out)
    torch.cuda.synchronize()
    dec.check()
    return per, s_final_in


def final_output_band(s_got, s_ref, wf, eps):
    """Per element of the final output, how far its unrounded value may move
    given the measured stream error: out = s * w / sqrt(mean(s^2) + eps), so a
    stream error of at most E in the row moves out_h by at most
    |w_h| * inv * E * (1 + |s_h| * inv^2 * rms) to first order (the norm's own
    change is at most E * rms / rms^2).  Doubled for the second-order terms."""
    s_ref = np.asarray(s_ref, np.float64)
    E = np.max(np.abs(np.asarray(s_got, np.float64) - s_ref), axis=1, keepdims=True)
    ms = np.mean(s_ref ** 2, axis=1, keepdims=True)
    inv = 1.0 / np.sqrt(ms + eps)
    return 2.0 * np.abs(np.asarray(wf, np.float64))[None, :] * inv * E * (1.0 + np.abs(s_ref) * inv ** 2 * np.sqrt(ms))


def check_final_output(got, out_ref, exact, band, what="final output"):
    """bf16 output bits against the oracle's: equal except where the oracle's
    unrounded value lies within R19's band plus `band` (an array, or None) of
    a rounding midpoint; there the GPU's value may have rounded the other
    way, so it lies within half its own quantum plus that band of the
    oracle's unrounded value."""
    x = np.asarray(exact, np.float64)
    tol = 1e-5 * np.abs(x) + 1e-5 * np.sqrt(np.mean(x ** 2))
    if band is not None:
        tol = tol + band
    diff = got != out_ref
    off = diff & ~bf16_near_tie(x, band=band)
    assert not np.any(off), f"{what}: {int(off.sum())} elements differ away from rounding midpoints"
    g = oracle.bf16_to_f64(got)
    a = np.maximum(np.abs(g), np.abs(x))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    half_q = np.exp2(np.maximum(e, -126) - 8)
    far = diff & (np.abs(g - x) > half_q + tol)
    assert not np.any(far), f"{what}: {int(far.sum())} elements round beyond the band"


def end_to_end(w, dec, rows, variant=0, sample_layers=None, n_sample=1, stage_layers=(), chain_report=None):
    """One whole step on the GPU (every layer and the final boundary) against
    the oracle, over every active expert, with the experts' NVFP4 weights as
    the GPU packed them (a sample per layer checked bit for bit against the
    oracle's own packing).  Each layer is recomputed by the oracle as a whole
    -- boundary, router, routing, pooler, both quantizations, the experts,
    the gather into the next boundary -- from the GPU's state at that
    layer's entry (its stream and branch), with the GPU's expert ids (R14);
    a single-layer workload is therefore checked end to end from the step's
    inputs.  Asserts:
      - at every layer, the oracle's routing of the GPU's MoE input gives the
        GPU's ids on every unflagged row (bit for bit);
      - the oracle's own routing of its own MoE input agrees with the GPU's
        ids on every unflagged row whose input is bitwise the GPU's;
      - after each layer, the stream at the next boundary (the next layer's,
        or the final) within STREAM_TOL * rms(stream), and the next bf16
        output (the next MoE input, or the final output) equal except at
        rounding midpoints, the band derived from that stream error;
      - the layers in stage_layers pass every staged check on a sample.
    Over several layers the stream is not compared from the step's inputs
    alone: the chain is ill-conditioned (R32), a one-ulp change of its input
    grows past the tolerance within a few layers in the oracle itself.  Within
    a layer, where the oracle's MoE input differs from the GPU's at a bf16
    midpoint, the MoE part runs from the GPU's input (R34).  With
    chain_report (a list), the oracle is also run freely from the step's
    inputs (the GPU's ids forced) and its per-layer divergence is appended.
    Returns the per-layer report."""
    k = w.top_k
    wr = w.with_rows(rows) if rows != w.rows else w
    stream, branch = _sgpu().step_tensors(wr, variant)
    out = torch.empty_like(branch)
    per, s_final_in = run_step_layerwise(w, dec, rows, branch, stream, out, keep_debug=stage_layers)
    s_host, b_host = synth.step_inputs(wr, variant)
    s_gpu = stream.cpu().numpy()
    out_gpu = out.view(torch.uint16).cpu().numpy()
    wpf, wf = synth.final_norm_weights(w)
    sample_layers = range(w.n_layers) if sample_layers is None else sample_layers
    report = []
    free_s, free_br = s_host, oracle.bf16_to_f64(b_host)
    for l in range(w.n_layers):
        g = per[l]
        # the GPU's branch into layer l: the step's, or its gather of layer l - 1
        br = oracle.bf16_to_f64(b_host) if l == 0 else \
            oracle.gather(per[l - 1]["gates"].astype(np.float64), per[l - 1]["o"], k)
        ow = gpu_layer_weights(dec, w, l, g["active"])
        if l in sample_layers:
            hot = sorted(set(int(e) for e in g["active"][:: max(1, len(g["active"]) // n_sample)][:n_sample]))
            check_gpu_weights(dec, oracle_weights(w, l, experts=hot), l, hot)
        if l in stage_layers:
            d = per[l]
            picks = sorted(set([int(max(d["active"], key=lambda e: d["count"][e]))]
                               + [int(e) for e in d["active"][:1]]))
            check_gpu_weights(dec, oracle_weights(w, l, experts=picks), l, picks)
            check_stages(w, d, ow, picks, br, d["stream_in"], d["stream"], rows)
        # the oracle's routing on the GPU's own MoE input: the GPU's ids (staged, bit for bit)
        rg = oracle.route(g["x"], ow.router_w, ow.router_bias, k)
        okg = rg["flags"] == 0
        assert np.array_equal(rg["ids"][okg], g["ids"][okg]), f"layer {l}: ids on the GPU's input"
        # the whole layer from the GPU's entry state, then the next boundary
        o = oracle.layer_step(ow, k, w.eps, br, g["stream_in"], forced_ids=g["ids"])
        own = oracle.route(o["x"], ow.router_w, ow.router_bias, k)
        same_x = np.all(o["x"] == g["x"], axis=1)
        agree = np.all(own["ids"] == g["ids"], axis=1)
        flagged = own["flags"] != 0
        assert np.all(agree | flagged | ~same_x), f"layer {l}: ids differ on an unflagged row"
        # where the oracle's MoE input differs from the GPU's (at a bf16
        # rounding midpoint: the previous boundary's check bounds that), the
        # MoE part continues from the GPU's input: one ulp at an NVFP4 code
        # boundary moves the experts' outputs by whole quantization steps (R34)
        moe = o if np.all(same_x) else oracle.moe_step(ow, k, g["x"], forced_ids=g["ids"])
        y = oracle.gather(moe["gates"], moe["o"], k)
        last = l == w.n_layers - 1
        nxt_w = (wpf, wf) if last else synth.norm_weights(w, l + 1)
        s_ref, b_ref, b_exact = oracle.boundary(y, o["stream"], nxt_w[0], nxt_w[1], w.eps)
        s_got = s_gpu if last else per[l + 1]["stream"]
        b_got = out_gpu if last else per[l + 1]["x"]
        err = float(np.max(np.abs(s_got.astype(np.float64) - s_ref)))
        bound = STREAM_TOL * _rms(s_ref)
        assert err <= bound, f"layer {l}: stream at the next boundary max|err| {err:.3e} > {bound:.3e}"
        check_final_output(b_got, b_ref, b_exact, final_output_band(s_got, s_ref, nxt_w[1], w.eps),
                           "final output" if last else f"layer {l + 1}'s MoE input")
        report.append(dict(layer=l, rows=rows, agree=int(agree.sum()), flagged=int(flagged.sum()),
                           x_differs=int((~same_x).sum()), n_active=len(g["active"]),
                           err_over_rms=err / _rms(s_ref)))
        if chain_report is not None and w.n_layers > 1:
            of = oracle.layer_step(ow, k, w.eps, free_br, free_s, forced_ids=g["ids"])
            free_s, free_br = of["stream"], oracle.gather(of["gates"], of["o"], k)
            gs = per[l]["stream"].astype(np.float64)
            chain_report.append(float(np.max(np.abs(gs - free_s)) / _rms(free_s)))
    # the final boundary staged: the oracle's on the GPU's last gather and stream
    y = oracle.gather(per[-1]["gates"].astype(np.float64), per[-1]["o"], k)
    fs_ref, fo_ref, fe = oracle.boundary(y, s_final_in, wpf, wf, w.eps)
    _close(s_gpu, fs_ref, 1e-5, "stream after the final boundary (staged)")
    check_final_output(out_gpu, fo_ref, fe, None, "final output (staged)")
    print(f"{w.name} b={rows}: per layer "
          + "; ".join(f"L{r['layer']}: max|err|/rms {r['err_over_rms']:.2e}, {r['agree']}/{rows} ids agree, "
                      f"{r['flagged']} flagged, {r['x_differs']} inputs differ, {r['n_active']} experts"
                      for r in report)
          + ("" if not chain_report else "; free-running chain max|err|/rms per layer: "
             + " ".join(f"{x:.1e}" for x in chain_report)))
    return report, stream, out


LAYOUTS = {"row_major": 0, "tiled": 1, "tiled_copy": 2}   # moe_decode_dims.code_layout


@pytest.mark.parametrize("layout", sorted(LAYOUTS))
def test_tiny_layer_staged(layout):
    """Every stage of one tiny layer, with the expert codes read in each
    layout: row-major in place, the caller's tiles in place, the handle's
    tiled copy."""
    w = synth.WORKLOADS["tiny"]
    sgpu = _sgpu()
    dec = sgpu.build(w, layout=LAYOUTS[layout])
    ow = oracle_weights(w, 0)
    _check_weights(dec, ow, 0, range(w.n_experts))
    stream, branch = sgpu.step_tensors(w)
    d = staged_layer(w, dec, ow, 0, w.rows, branch, stream)
    _final_check(w, dec, d, w.rows, stream)
    dec.close()


def _oracle_step(w, variant=0, experts_needed=None):
    stream, branch = synth.step_inputs(w, variant)
    s = stream
    br = oracle.bf16_to_f64(branch)
    outs = []
    for l in range(w.n_layers):
        ow = oracle_weights(w, l)
        o = oracle.layer_step(ow, w.top_k, w.eps, br, s)
        outs.append(o)
        s = o["stream"]
        br = oracle.gather(o["gates"], o["o"], w.top_k)
    wpf, wf = synth.final_norm_weights(w)
    s, out, oe = oracle.boundary(br, s, wpf, wf, w.eps)
    return s, out, oe, outs


def test_tiny_step_end_to_end_graph_and_host():
    import speculative_decode_routed_gb300 as moe
    w = synth.WORKLOADS["tiny"]
    sgpu = _sgpu()
    dec = sgpu.build(w)
    s_ref, out_ref, oe, outs = _oracle_step(w)
    # eager
    stream, branch = sgpu.step_tensors(w)
    out = torch.empty_like(branch)
    dec.step(w.rows, branch, stream, out)
    torch.cuda.synchronize()
    dec.check()
    ids = dev_array(dec.debug().ids, (w.rows, w.top_k), np.int32)
    ok = outs[-1]["flags"] == 0
    assert np.array_equal(ids[ok], outs[-1]["ids"][ok])
    eager_stream, eager_out = stream.cpu().numpy(), out.view(torch.uint16).cpu().numpy()
    err = np.abs(eager_stream - s_ref).max()
    assert err <= STREAM_TOL * _rms(s_ref), f"end-to-end stream max|err| {err:.3e}"
    check_final_output(eager_out, out_ref, oe,
                       final_output_band(eager_stream, s_ref, synth.final_norm_weights(w)[1], w.eps))
    # graph replay is bitwise the eager result, twice in a row
    for _ in range(2):
        stream2, branch2 = sgpu.step_tensors(w)
        out2 = torch.empty_like(branch2)
        dec.step_graph(w.rows, branch2, stream2, out2)
        torch.cuda.synchronize()
        assert np.array_equal(stream2.cpu().numpy(), eager_stream)
        assert np.array_equal(out2.view(torch.uint16).cpu().numpy(), eager_out)
    # host-buffer path
    s_h, b_h = synth.step_inputs(w)
    sh = torch.from_numpy(s_h).pin_memory()
    bh = torch.from_numpy(b_h).view(torch.bfloat16).pin_memory()
    oh = torch.empty_like(bh).pin_memory()
    for _ in range(2):                      # captured on the first call, replayed on the second
        sh.copy_(torch.from_numpy(s_h))
        dec.step_host(w.rows, bh, sh, oh)
        assert np.array_equal(sh.numpy(), eager_stream)
        assert np.array_equal(oh.view(torch.uint16).numpy(), eager_out)
    # pageable host buffers take the separate copies
    sp = torch.from_numpy(s_h.copy())
    op = torch.empty_like(oh, device="cpu")
    dec.step_host(w.rows, torch.from_numpy(b_h.copy()).view(torch.bfloat16), sp, op)
    assert np.array_equal(sp.numpy(), eager_stream)
    assert np.array_equal(op.view(torch.uint16).numpy(), eager_out)
    # per layer: boundary, router and the experts (tensor cores; beyond 8
    # rows the routing kernel, beyond 32 the pooler gather), or the CUDA-core
    # build's gate/up and down; plus the final boundary
    assert moe.moe_decode_step_kernel_count(dec.handle) in (3 * w.n_layers + 1, 4 * w.n_layers + 1,
                                                          5 * w.n_layers + 1)
    dec.close()


def test_repeated_replays_bitwise():
    """Many graph replays of one input give the eager result bit for bit with
    no device-side error.  The shape makes the gate/up kernel's stage ring
    (5 stages) not a multiple of its K-phase groups (2), with tens of stage
    fills per CTA, so a stage-barrier phase mix-up between the groups would
    show as a timeout or a changed result."""
    w = synth.Workload("replay", rows=8, hidden=4096, n_experts=64, top_k=8, inter=1024)
    sgpu = _sgpu()
    dec = sgpu.build(w)
    stream, branch = sgpu.step_tensors(w)
    s0 = stream.clone()
    out = torch.empty_like(branch)
    dec.step(w.rows, branch, stream, out)
    torch.cuda.synchronize()
    dec.check()
    ref_s, ref_o = stream.clone(), out.clone()
    bad = 0
    for _ in range(400):
        stream.copy_(s0)
        dec.step_graph(w.rows, branch, stream, out)
        bad += int(not torch.equal(stream, ref_s)) + int(not torch.equal(out, ref_o))
    torch.cuda.synchronize()
    dec.check()
    assert bad == 0, f"{bad} replays differ from the eager result"
    dec.close()


def test_bounded_wait_gives_up_and_the_handle_recovers():
    """The experts kernel's give-up path, with no fault: with a 1 ms wait
    limit, a layer whose completed experts are never published to the down
    phase makes every down item's wait run out.  The call returns within the
    limit's order (the default 2 s would not have given up yet), the latched
    code reads as a wait timeout and is cleared by reading it, and the next
    steps -- eager and graph, under the short limit and the default -- give
    the reference result bit for bit."""
    import time

    import speculative_decode_routed_gb300 as moe
    w = synth.WORKLOADS["tiny"]
    sgpu = _sgpu()
    dec = sgpu.build(w)
    stream, branch = sgpu.step_tensors(w)
    s0 = stream.clone()
    out = torch.empty_like(branch)
    dec.step(w.rows, branch, stream, out)
    torch.cuda.synchronize()
    dec.check()
    ref_s, ref_o = stream.clone(), out.clone()
    dec.set_wait_limit(1_000_000)
    s1 = s0.clone()
    t0 = time.perf_counter()
    dec.selftest_wait_timeout(w.rows, branch, s1)
    rc = dec.last_error()
    elapsed = time.perf_counter() - t0
    assert rc == moe.MOE_EDEVICE, f"expected a latched wait timeout, got {rc}"
    assert b"error 1 " in moe.lib().moe_decode_error_message()
    assert elapsed < 1.0, f"the self-test took {elapsed:.3f} s"
    assert dec.last_error() == moe.MOE_OK
    for limit in (1_000_000, 2_000_000_000):
        dec.set_wait_limit(limit)
        for call in (dec.step, dec.step_graph):
            stream.copy_(s0)
            out.zero_()
            call(w.rows, branch, stream, out)
            torch.cuda.synchronize()
            dec.check()
            assert torch.equal(stream, ref_s) and torch.equal(out, ref_o)
    with pytest.raises(moe.MoeError):
        dec.set_wait_limit(10)
    dec.close()


def test_workspace_guards_catch_a_stray_write():
    """A write past the end of a workspace region lands in the guard after it,
    and the next error check reports the region by name (then the guard is
    rewritten, so a later check is clean).  The write is made here, by the
    host, into the guard that follows the MoE input x: every region is
    followed by a 256-byte guard, and x holds max_rows * H bf16 values."""
    import speculative_decode_routed_gb300 as moe
    from helpers import _CudaArray
    w = synth.WORKLOADS["tiny"]
    sgpu = _sgpu()
    dec = sgpu.build(w)
    stream, branch = sgpu.step_tensors(w)
    out = torch.empty_like(branch)
    dec.step(w.rows, branch, stream, out)
    torch.cuda.synchronize()
    dec.check()                                     # every guard intact after a step
    x_bytes = dec.dims.max_rows * dec.dims.hidden * 2
    guard = dec.debug().x + (x_bytes + 255) // 256 * 256
    torch.as_tensor(_CudaArray(guard, (4,), "|u1"), device="cuda").fill_(0x77)
    torch.cuda.synchronize()
    with pytest.raises(moe.MoeError) as err:
        dec.check()
    assert err.value.code == moe.MOE_EDEVICE and "region 'x'" in str(err.value)
    dec.check()
    dec.step(w.rows, branch, stream, out)
    dec.check()
    dec.close()


def test_loaded_library_variant():
    """The library the tests run against: the bounds-check variant when the
    environment asks for it (the bounds-check run of this file), else the
    default build."""
    import os

    import speculative_decode_routed_gb300 as moe
    info = moe.lib().moe_decode_build_info()
    want = 1 if os.environ.get("MOE_DECODE_EXPECT_BOUNDS") == "1" else 0
    assert info & 1 == want


def test_tile_codes_matches_the_layout():
    """moe_tile_codes against the layout its header states (untiled on the
    host), the bytes of a partial last K-block zero."""
    import speculative_decode_routed_gb300 as moe
    from helpers import untile_codes
    g = torch.Generator(device="cuda").manual_seed(5)
    for rows, rb in ((256, 3584), (384, 192), (128, 64), (256, 1024)):
        src = torch.randint(0, 256, (rows, rb), dtype=torch.uint8, device="cuda", generator=g)
        dst = torch.full((moe.moe_tiled_code_bytes(rows, rb),), 0xEE, dtype=torch.uint8, device="cuda")
        moe.moe_tile_codes(src, dst)
        torch.cuda.synchronize()
        t = dst.cpu().numpy()
        assert np.array_equal(untile_codes(t, rows, rb), src.cpu().numpy())
        kb = -(-rb // 128)
        tail = t.reshape(rows // 128, kb, 128, 128)[:, -1, :, rb - (kb - 1) * 128:]
        assert not tail.any(), "bytes beyond the row in the last K-block must be zero"


def test_graph_cache_evicts_and_recaptures():
    """More distinct (branch, stream, out) buffer sets than the step-graph cache
    keeps (32): every call gives the eager result bit for bit, including the
    first sets again once their graphs were evicted and are captured anew."""
    w = synth.WORKLOADS["tiny"]
    sgpu = _sgpu()
    dec = sgpu.build(w)
    stream, branch = sgpu.step_tensors(w)
    s0 = stream.clone()
    out = torch.empty_like(branch)
    dec.step(w.rows, branch, stream, out)
    torch.cuda.synchronize()
    dec.check()
    ref_s, ref_o = stream.clone(), out.clone()
    sets = [(branch.clone(), s0.clone(), torch.empty_like(out)) for _ in range(40)]
    for b, s, o in sets + sets[:3]:
        s.copy_(s0)
        dec.step_graph(w.rows, b, s, o)
        torch.cuda.synchronize()
        assert torch.equal(s, ref_s) and torch.equal(o, ref_o)
    dec.check()
    dec.close()


@pytest.mark.parametrize("H", [256, 7168])
def test_front_and_aux_copies(H):
    """The first layer's front against the oracle (stream bit-exact, the
    attention input exact away from bf16 near-ties), its aux copy, and the
    final boundary's aux copy of the stream."""
    w = synth.Workload(f"front{H}", rows=8, hidden=H, n_experts=8, top_k=2, inter=128)
    sgpu = _sgpu()
    dec = sgpu.build(w)
    emb_bits, wn = synth.front_inputs(w)
    emb = torch.from_numpy(emb_bits.view(np.int16)).view(torch.bfloat16).cuda()
    stream = torch.empty(w.rows, H, dtype=torch.float32, device="cuda")
    attn = torch.empty(w.rows, H, dtype=torch.bfloat16, device="cuda")
    aux = torch.full_like(stream, float("nan"))
    dec.front(w.rows, emb, torch.from_numpy(wn).cuda(), stream, attn, aux)
    torch.cuda.synchronize()
    dec.check()
    s_ref, out_ref, exact = oracle.front(emb_bits, wn, w.eps)
    assert np.array_equal(stream.cpu().numpy(), s_ref)
    assert torch.equal(aux, stream)
    got = attn.view(torch.uint16).cpu().numpy()
    assert not np.any((got != out_ref) & ~bf16_near_tie(exact)), "attention input away from near-ties"
    assert np.mean(got != out_ref) < 1e-3
    # a layer on that stream, then the final boundary with its aux copy
    _, branch = sgpu.step_tensors(w)
    dec.layer(0, w.rows, branch, stream)
    out = torch.empty_like(attn)
    aux2 = torch.full_like(stream, float("nan"))
    dec.final(w.rows, stream, out, aux2)
    torch.cuda.synchronize()
    dec.check()
    assert torch.equal(aux2, stream)
    dec.close()


ODD_SHAPES = [
    # (rows, H, E, k, I): a ragged H (cluster of 1, 12 chunks/row), a single
    # expert, k == E, a row count with many rows per expert (> 8: the
    # multi-group path, 16 router row blocks), one row
    (5, 384, 6, 3, 384),
    (3, 128, 1, 1, 128),
    (3, 1024, 16, 16, 256),
    (128, 256, 8, 2, 128),
    (1, 512, 32, 4, 640),
    # two experts for 128 rows: ~64 pairs each, so every expert's work is
    # split into several 32-pair parts whose h is quantized as one tensor
    (128, 256, 2, 1, 256),
]


@pytest.mark.parametrize("rows,H,E,k,I", ODD_SHAPES)
def test_odd_shapes_staged(rows, H, E, k, I):
    _odd_shape(rows, H, E, k, I, LAYOUTS["tiled"])


@pytest.mark.parametrize("rows,H,E,k,I", [ODD_SHAPES[0], ODD_SHAPES[4], ODD_SHAPES[5]])
def test_odd_shapes_row_major_codes(rows, H, E, k, I):
    """The row-major weight maps (read in place) on a ragged H and I (a last
    K-block half filled) and on experts split into several 32-pair parts."""
    _odd_shape(rows, H, E, k, I, LAYOUTS["row_major"])


def _odd_shape(rows, H, E, k, I, layout):
    w = synth.Workload(f"odd{H}", rows=rows, hidden=H, n_experts=E, top_k=k, inter=I)
    sgpu = _sgpu()
    dec = sgpu.build(w, layout=layout)
    ow = oracle_weights(w, 0)
    stream, branch = sgpu.step_tensors(w)
    d = staged_layer(w, dec, ow, 0, rows, branch, stream)
    _final_check(w, dec, d, rows, stream)
    dec.close()


def test_zero_branch_keeps_stream_and_rows_below_max():
    w = synth.WORKLOADS["tiny"]
    sgpu = _sgpu()
    dec = sgpu.build(w, max_rows=16)
    ow = oracle_weights(w, 0)
    stream, branch = sgpu.step_tensors(w)
    s0 = stream.cpu().numpy().copy()
    zero = torch.zeros_like(branch)
    dec.layer(0, w.rows, zero, stream)
    torch.cuda.synchronize()
    assert np.array_equal(stream.cpu().numpy(), s0)
    # fewer rows than max_rows
    stream, branch = sgpu.step_tensors(w)
    staged_layer(w, dec, ow, 0, 3, branch[:3], stream[:3].clone())
    dec.close()


# ------------------------------------------------------------- full sizes


def _sample_experts(d, n_extra=2, seed=0):
    """The expert with the most pairs plus a few seeded picks among the active."""
    act = list(d["active"])
    hot = int(max(act, key=lambda e: d["count"][e]))
    rs = np.random.RandomState(seed)
    pick = [int(e) for e in rs.choice(act, size=min(n_extra, len(act)), replace=False)]
    return sorted(set([hot] + pick))


def _staged_full(w, dec, layer, rows, branch, stream, n_extra=2, prev=None):
    """Staged check at full size: routing / pooler / act quant for every row,
    experts on a sample (weights quantized by the oracle only for those)."""
    def pick(d):
        sample = _sample_experts(d, n_extra, seed=layer)
        ow = oracle_weights(w, layer, experts=sample)
        _check_weights(dec, ow, layer, sample)
        return ow, sample
    return staged_layer(w, dec, pick, layer, rows, branch, stream, prev=prev)


def _graph_equals_eager(w, dec, rows, variant=1):
    """The library's captured step replays bit for bit what the eager step computes."""
    sgpu = _sgpu()
    wr = w.with_rows(rows) if rows != w.rows else w
    s1, b1 = sgpu.step_tensors(wr, variant=variant)
    o1 = torch.empty_like(b1)
    dec.step(rows, b1, s1, o1)
    s2, b2 = sgpu.step_tensors(wr, variant=variant)
    o2 = torch.empty_like(b2)
    dec.step_graph(rows, b2, s2, o2)
    torch.cuda.synchronize()
    dec.check()
    assert torch.equal(s1, s2) and torch.equal(o1, o2), "graph replay differs from the eager step"


@pytest.mark.slow
@pytest.mark.parametrize("layout", ["tiled", "row_major"])
def test_serving_end_to_end(layout):
    """One layer at serving width (H 7168, 256 experts, top-8, I 2048, b 8), the
    bench's configuration and launch path: every active expert end to end
    against the oracle, the layer's stages on a sample, the final boundary,
    and the graph replay against the eager step."""
    w = synth.WORKLOADS["serving"]
    dec = _sgpu().build(w, layout=LAYOUTS[layout])
    end_to_end(w, dec, w.rows, stage_layers=(0,))
    _graph_equals_eager(w, dec, w.rows)
    dec.close()


@pytest.mark.slow
def test_chained_layers_end_to_end():
    """Eight chained layers (H 5120, 128 experts, top-8, I 1536): every layer
    end to end against the oracle from the GPU's state at its entry (R32),
    every layer's stages on a sample (the chained gather included), the
    final boundary, and the graph."""
    w = synth.WORKLOADS["chained8"]
    dec = _sgpu().build(w)
    end_to_end(w, dec, w.rows, stage_layers=tuple(range(w.n_layers)), chain_report=[])
    _graph_equals_eager(w, dec, w.rows)
    dec.close()


@pytest.mark.slow
@pytest.mark.parametrize("rows", synth.SWEEP_ROWS)
def test_batch_skew_sweep_end_to_end(rows):
    """H 7168, 256 experts, top-8, I 2048 with a Zipf(1.1) logit bias, b in
    {1, 8, 32, 64, 128}: end to end over every active expert, the stages on a
    sample (the hottest expert included)."""
    w = synth.WORKLOADS["sweep"].with_rows(rows)
    dec = _sgpu().build(w)
    end_to_end(w, dec, rows, stage_layers=(0,))
    dec.close()


@pytest.mark.slow
def test_stack16_end_to_end():
    """The 16-layer stack at serving widths (about 101.5 GB of NVFP4 weights,
    generated on the device), b 8, the codes held once in tiles: every layer
    end to end against the oracle from the GPU's state at its entry (R32),
    three layers' stages on a sample, the final boundary, and the graph
    replay against the eager step."""
    import speculative_decode_routed_gb300 as moe
    w = synth.WORKLOADS["stack16"]
    dec = _sgpu().build(w)
    H, I, E = w.hidden, w.inter, w.n_experts
    codes = E * (2 * I * H // 2 + H * I // 2)
    # the handle holds only the scale atoms (1/8 of the code bytes), no copy of the codes
    assert moe.moe_decode_weight_copy_bytes(dec.handle) <= w.n_layers * codes // 8 + (1 << 20)
    end_to_end(w, dec, w.rows, sample_layers=(0, 8, 15), stage_layers=(0, 8, 15), chain_report=[])
    _graph_equals_eager(w, dec, w.rows)
    dec.close()
