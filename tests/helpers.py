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
