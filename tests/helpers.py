"""Test helpers: workload weights for the oracle (host) from the seeded
generators.  Turning raw weights into NVFP4 here uses the oracle's own
quantizer; the GPU side quantizes the same raw values with its own kernel."""
import numpy as np

import oracle
import synth


def golden(name):
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", name)
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def quantize_expert(w, layer, e):
    """(w13 codes [2I, H/2], w13 sf [2I, H/16], w2 codes [H, I/2], w2 sf [H, I/16], gscale[3])."""
    cg, sg_, g_sg, _ = oracle.nvfp4_quantize(synth.expert_raw(w, layer, e, "gate"))
    cu, su, u_sg, _ = oracle.nvfp4_quantize(synth.expert_raw(w, layer, e, "up"))
    cd, sd, d_sg, _ = oracle.nvfp4_quantize(synth.expert_raw(w, layer, e, "down"))
    return (np.vstack([cg, cu]), np.vstack([sg_, su]), cd, sd,
            np.array([g_sg, u_sg, d_sg], np.float32))


def oracle_weights(w, layer, experts=None):
    """oracle.LayerWeights of one layer; only `experts` (default: all) get tensors."""
    E = w.n_experts
    experts = range(E) if experts is None else sorted(set(int(e) for e in experts))
    w_post, w_pre = synth.norm_weights(w, layer)
    w13, w13_sf, w2, w2_sf = {}, {}, {}, {}
    gscale = np.zeros((E, 3), np.float32)
    for e in experts:
        w13[e], w13_sf[e], w2[e], w2_sf[e], gscale[e] = quantize_expert(w, layer, e)
    return oracle.LayerWeights(E, w.hidden, w.inter, w_post, w_pre, synth.router_weights(w, layer),
                               synth.router_bias(w, layer), w13, w13_sf, w2, w2_sf, gscale)


def silu(z):
    return z / (1.0 + np.exp(-z))


# --------------------------------------------------------------- GPU side


class _CudaArray:
    """Zero-copy view of raw device memory for torch.as_tensor."""

    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (int(ptr), False), "version": 3, "strides": None}


def dev_array(ptr, shape, dtype):
    """Copy `shape` elements of numpy `dtype` at device address `ptr` to the host."""
    import torch
    dt = np.dtype(dtype)
    t = torch.as_tensor(_CudaArray(ptr, shape, dt.str), device="cuda")
    return t.cpu().numpy().copy()


def read_debug(dec, rows):
    """The workspace intermediates of the last layer run, as numpy arrays."""
    v = dec.debug()
    d = dec.dims
    H, E, k, I = d.hidden, d.n_experts, d.top_k, d.inter
    n = rows * k
    out = dict(
        x=dev_array(v.x, (rows, H), np.uint16),
        x_codes=dev_array(v.x_codes, (rows, H // 2), np.uint8),
        x_sf=dev_array(v.x_sf, (rows, H // 16), np.uint8),
        x_sg=dev_array(v.x_sg, (1,), np.float32)[0],
        logits=dev_array(v.logits, (rows, E), np.float32),
        ids=dev_array(v.ids, (rows, k), np.int32),
        gates=dev_array(v.gates, (rows, k), np.float32),
        flags=dev_array(v.flags, (rows,), np.uint8),
        count=dev_array(v.count, (E,), np.int32),
        offset=dev_array(v.offset, (E + 1,), np.int32),
        pair_order=dev_array(v.pair_order, (n,), np.int32),
        pos_of_pair=dev_array(v.pos_of_pair, (n,), np.int32),
        n_active=int(dev_array(v.n_active, (1,), np.int32)[0]),
        h=dev_array(v.h, (n, I), np.float32),
        h_sg=dev_array(v.h_sg, (E,), np.float32),
        h_codes=dev_array(v.h_codes, (n, I // 2), np.uint8),
        h_sf=dev_array(v.h_sf, (n, I // 16), np.uint8),
        o=dev_array(v.o, (n, H), np.float32),
    )
    out["active"] = dev_array(v.active, (E,), np.int32)[: out["n_active"]]
    return out


def bf16_near_tie(exact, rel=1e-5, abs_frac=1e-5, band=None):
    """True where the fp64 value sits within rel * |value| + abs_frac * rms(values)
    (+ band, an array of further absolute allowances, if given) of a bf16
    rounding midpoint, so an fp32 evaluation may round it the other way.  The
    absolute term covers values left small by cancellation, whose fp32
    relative error is large although their absolute error is not."""
    x = np.asarray(exact, np.float64)
    a = np.abs(x)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    q = np.exp2(np.maximum(e, -126) - 7)        # bf16 quantum in this binade
    frac = a / q - np.floor(a / q)
    tol = rel * a + abs_frac * np.sqrt(np.mean(x ** 2))
    if band is not None:
        tol = tol + np.asarray(band, np.float64)
    return np.abs(frac - 0.5) * q <= tol


def bits_match(got, ref, exact, what, slack=0, exclude=None):
    """Assert that the bf16 bit patterns `got` equal `ref` except at rounding
    midpoints of `exact` (bf16_near_tie) or where `exclude` is set, and at
    most max(2, slack) further elements, each one bf16 step away."""
    off = (got != ref) & ~bf16_near_tie(exact)
    if exclude is not None:
        off &= ~exclude
    n_off = int(off.sum())
    if n_off:
        steps = np.abs(got.astype(np.int32) - ref.astype(np.int32))[off]
        assert n_off <= max(2, slack) and steps.max() <= 1, \
            f"{what}: {n_off} of {got.size} elements differ away from rounding midpoints " \
            f"(max {steps.max()} steps)"


def expert_subproblem(ow, e):
    """A one-expert oracle.LayerWeights holding expert e of `ow` as expert 0."""
    import oracle
    g = np.zeros((1, 3), np.float32)
    g[0] = ow.gscale[e]
    return oracle.LayerWeights(1, ow.H, ow.I, ow.w_post, ow.w_pre, ow.router_w[:1], None,
                               {0: ow.w13[e]}, {0: ow.w13_sf[e]}, {0: ow.w2[e]},
                               {0: ow.w2_sf[e]}, g)


# ------------------------------------------------- expert codes in 16 KB tiles


def untile_codes(tiles, rows, row_bytes):
    """Row-major codes [rows, row_bytes] from their tiles, the layout
    moe_tile_codes writes: [rows / 128][ceil(row_bytes / 128)][128 rows][128 B],
    row tile outermost, zero beyond row_bytes."""
    kb = -(-row_bytes // 128)
    t = np.asarray(tiles, np.uint8).reshape(rows // 128, kb, 128, 128)
    return np.ascontiguousarray(t.transpose(0, 2, 1, 3).reshape(rows, kb * 128)[:, :row_bytes])


def tiled_expert_bytes(rows_per_expert, row_bytes):
    """Bytes of one expert's tiles (they are contiguous, expert after expert)."""
    return rows_per_expert // 128 * (-(-row_bytes // 128)) * 16384


def gpu_expert(dec, layer, e):
    """(w13 codes [2I, H/2], w13 sf [2I, H/16], w2 codes [H, I/2], w2 sf [H, I/16],
    gscale [3]) of expert e as the handle holds them on the device, copied back
    (the codes untiled when the caller holds them in tiles)."""
    import speculative_decode_routed_gb300 as moe
    t, d = dec.layers[layer], dec.dims
    H, I = d.hidden, d.inter
    if d.code_layout == moe.MOE_CODES_TILED:
        n13, n2 = tiled_expert_bytes(2 * I, H // 2), tiled_expert_bytes(H, I // 2)
        w13 = untile_codes(t.w13[e * n13:(e + 1) * n13].cpu().numpy(), 2 * I, H // 2)
        w2 = untile_codes(t.w2[e * n2:(e + 1) * n2].cpu().numpy(), H, I // 2)
    else:
        w13, w2 = t.w13[e].cpu().numpy(), t.w2[e].cpu().numpy()
    return (w13, t.w13_sf[e].cpu().numpy(), w2, t.w2_sf[e].cpu().numpy(),
            t.w_gscale[e].cpu().numpy())


def gpu_layer_weights(dec, w, layer, experts):
    """oracle.LayerWeights of one layer: norms and router from the host
    generators, the NVFP4 experts `experts` as the GPU packed them (copied
    back).  The weights are inputs of the step; a sample of experts is checked
    bit for bit against the oracle's own packing (check_gpu_weights) before
    these are trusted."""
    E = w.n_experts
    w13, w13_sf, w2, w2_sf = {}, {}, {}, {}
    gscale = np.zeros((E, 3), np.float32)
    for e in sorted(set(int(x) for x in experts)):
        w13[e], w13_sf[e], w2[e], w2_sf[e], gscale[e] = gpu_expert(dec, layer, e)
    w_post, w_pre = synth.norm_weights(w, layer)
    return oracle.LayerWeights(E, w.hidden, w.inter, w_post, w_pre, synth.router_weights(w, layer),
                               synth.router_bias(w, layer), w13, w13_sf, w2, w2_sf, gscale)


def check_gpu_weights(dec, ow, layer, experts):
    """The GPU's NVFP4 packing of `experts` equals the oracle's own (ow), bit for bit."""
    for e in experts:
        g13, g13s, g2, g2s, gg = gpu_expert(dec, layer, e)
        assert np.array_equal(g13, ow.w13[e]), f"w13 codes of expert {e}"
        assert np.array_equal(g13s, ow.w13_sf[e]), f"w13 scales of expert {e}"
        assert np.array_equal(g2, ow.w2[e]), f"w2 codes of expert {e}"
        assert np.array_equal(g2s, ow.w2_sf[e]), f"w2 scales of expert {e}"
        assert np.array_equal(gg, ow.gscale[e]), f"tensor scales of expert {e}"
