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


def layer_tensors(w: synth.Workload, layer: int, device="cuda", experts=None):
    """speculative_decode_routed_gb300.LayerTensors of one layer.  Experts not in
    `experts` (default: all) are left zero-filled."""
    import torch

    import speculative_decode_routed_gb300 as moe

    E, H, I = w.n_experts, w.hidden, w.inter
    w_post, w_pre = synth.norm_weights(w, layer)
    bias = synth.router_bias(w, layer)
    t = moe.LayerTensors(
        w_post=_t(w_post, device), w_pre=_t(w_pre, device),
        router_w=_bf16(synth.router_weights(w, layer), device),
        router_bias=None if bias is None else _t(bias, device),
        w13=torch.zeros(E, 2 * I, H // 2, dtype=torch.uint8, device=device),
        w13_sf=torch.zeros(E, 2 * I, H // 16, dtype=torch.uint8, device=device),
        w2=torch.zeros(E, H, I // 2, dtype=torch.uint8, device=device),
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
                codes, sf = t.w2[e], t.w2_sf[e]
            else:
                rows = slice(0, I) if which == "gate" else slice(I, 2 * I)
                codes, sf = t.w13[e, rows], t.w13_sf[e, rows]
            moe.moe_nvfp4_quantize(r, codes, sf, t.w_gscale[e, col:col + 1], amax)
    return t


def final_tensors(w: synth.Workload, device="cuda"):
    a, b = synth.final_norm_weights(w)
    return _t(a, device), _t(b, device)


def step_tensors(w: synth.Workload, variant: int = 0, device="cuda"):
    """(stream fp32 [b, H], branch bf16 [b, H]) on the device."""
    s, b = synth.step_inputs(w, variant)
    return _t(s, device), _bf16(b, device)


def build(w: synth.Workload, device="cuda", max_rows=None):
    """A MoEDecode handle over freshly generated device weights for every layer."""
    import speculative_decode_routed_gb300 as moe

    layers = [layer_tensors(w, l, device) for l in range(w.n_layers)]
    wpf, wf = final_tensors(w, device)
    return moe.MoEDecode(w.hidden, w.n_experts, w.top_k, w.inter, max_rows or w.rows, layers,
                         wpf, wf, eps=w.eps)
