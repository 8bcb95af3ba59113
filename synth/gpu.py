"""Device twin of the workload recipes in ``synth``: the same raw values,
generated where they live (HBM) by the device Philox generator and packed into
NVFP4 by the library's own quantizer entry point (``moe_nvfp4_quantize``).
Small tensors (norm weights, router, step inputs) come from the host
generator and are copied over.  Used by the GPU tests and the bench."""
from __future__ import annotations

import numpy as np

import synth


def _t(a, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def _bf16(bits, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits)).view(torch.bfloat16).to(device)


def layer_tensors(w: synth.Workload, layer: int, device="cuda", experts=None, layout=0,
                  scratch=None):
    """speculative_decode_routed_gb300.LayerTensors of one layer.  Experts not in
    `experts` (default: all) are left zero-filled.  layout: the handle's
    code_layout; with MOE_CODES_TILED the codes are quantized row-major into
    `scratch` (a dict of reusable buffers, or None) and tiled into w13 / w2,
    so only the tiled copy stays resident."""
    import torch

    import speculative_decode_routed_gb300 as moe

    E, H, I = w.n_experts, w.hidden, w.inter
    w_post, w_pre = synth.norm_weights(w, layer)
    bias = synth.router_bias(w, layer)
    tiled = layout == moe.MOE_CODES_TILED

    def codes(shape, key):
        if not tiled:
            return torch.zeros(*shape, dtype=torch.uint8, device=device)
        buf = None if scratch is None else scratch.get(key)
        if buf is None or tuple(buf.shape) != tuple(shape):
            buf = torch.zeros(*shape, dtype=torch.uint8, device=device)
            if scratch is not None:
                scratch[key] = buf
        elif experts is not None:
            buf.zero_()
        return buf

    t = moe.LayerTensors(
        w_post=_t(w_post, device), w_pre=_t(w_pre, device),
        router_w=_bf16(synth.router_weights(w, layer), device),
        router_bias=None if bias is None else _t(bias, device),
        w13=codes((E, 2 * I, H // 2), "w13"),
        w13_sf=torch.zeros(E, 2 * I, H // 16, dtype=torch.uint8, device=device),
        w2=codes((E, H, I // 2), "w2"),
        w2_sf=torch.zeros(E, H, I // 16, dtype=torch.uint8, device=device),
        w_gscale=torch.zeros(E, 3, dtype=torch.float32, device=device))
    raw = torch.empty(H * I, dtype=torch.float32, device=device)
    amax = torch.empty(1, dtype=torch.float32, device=device)
    for e in (range(E) if experts is None else experts):
        for which, col in (("gate", 0), ("up", 1), ("down", 2)):
            shape = (H, I) if which == "down" else (I, H)
            r = raw.view(*shape)
            synth.dev_expert_raw(r, w, layer, e, which)
            if which == "down":
                c, sf = t.w2[e], t.w2_sf[e]
            else:
                rows = slice(0, I) if which == "gate" else slice(I, 2 * I)
                c, sf = t.w13[e, rows], t.w13_sf[e, rows]
            moe.moe_nvfp4_quantize(r, c, sf, t.w_gscale[e, col:col + 1], amax)
    if tiled:
        for name, rows, rb in (("w13", E * 2 * I, H // 2), ("w2", E * H, I // 2)):
            dst = torch.empty(moe.moe_tiled_code_bytes(rows, rb), dtype=torch.uint8, device=device)
            moe.moe_tile_codes(getattr(t, name).view(rows, rb), dst)
            setattr(t, name, dst)
        torch.cuda.synchronize(device)  # the row-major scratch may be reused at once
    return t


def final_tensors(w: synth.Workload, device="cuda"):
    a, b = synth.final_norm_weights(w)
    return _t(a, device), _t(b, device)


def step_tensors(w: synth.Workload, variant: int = 0, device="cuda"):
    """(stream fp32 [b, H], branch bf16 [b, H]) on the device."""
    s, b = synth.step_inputs(w, variant)
    return _t(s, device), _bf16(b, device)


def build(w: synth.Workload, device="cuda", max_rows=None, layout=None):
    """A MoEDecode handle over freshly generated device weights for every layer.
    layout: the handle's code_layout (default MOE_CODES_TILED: the caller holds
    the codes in tiles, the one copy the handle reads)."""
    import speculative_decode_routed_gb300 as moe

    layout = moe.MOE_CODES_TILED if layout is None else layout
    scratch = {}
    layers = [layer_tensors(w, l, device, layout=layout, scratch=scratch) for l in range(w.n_layers)]
    scratch.clear()
    wpf, wf = final_tensors(w, device)
    return moe.MoEDecode(w.hidden, w.n_experts, w.top_k, w.inter, max_rows or w.rows, layers,
                         wpf, wf, eps=w.eps, code_layout=layout)
