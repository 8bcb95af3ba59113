"""CPU oracle of the routed NVFP4 MoE decode layer-step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The GPU
library never loads it and shares no source with it.

This is a thin ctypes binding over ``oracle.c`` (plain C, fp64 accumulation);
every function cites, in the C source, the passage it follows.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(_HERE, "liboracle.so")

_i32, _i64, _f32, _f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double
_u8, _u16, _vp = ctypes.c_uint8, ctypes.c_uint16, ctypes.c_void_p


class _LayerWeights(ctypes.Structure):
    _fields_ = [("w_post", _vp), ("w_pre", _vp), ("router_w", _vp), ("router_bias", _vp),
                ("w13", _vp), ("w13_sf", _vp), ("w2", _vp), ("w2_sf", _vp), ("gscale", _vp)]


class _LayerOut(ctypes.Structure):
    _fields_ = [(n, _vp) for n in (
        "x", "x_exact", "x_codes", "x_sf", "x_sg", "x_amax",
        "probs", "ids", "gates", "flags", "gap",
        "count", "offset", "pair_order", "active", "n_active",
        "h", "h_codes", "h_sf", "h_sg", "h_amax", "o")]


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} missing: run __graft_entry__.build() first")
        L = ctypes.CDLL(LIB)
        sig = {
            "oracle_e2m1_decode": (_f64, [_u8]),
            "oracle_e2m1_encode": (_u8, [_f32]),
            "oracle_e4m3_decode": (_f64, [_u8]),
            "oracle_e4m3_encode": (_u8, [_f32]),
            "oracle_bf16_from_double": (_u16, [_f64]),
            "oracle_bf16_decode": (_f64, [_u16]),
            "oracle_nvfp4_quantize": (None, [_vp, _i64, _i64, _vp, _vp, _vp, _vp]),
            "oracle_nvfp4_dequantize": (None, [_vp, _vp, _f32, _i64, _i64, _vp]),
            "oracle_boundary": (None, [ctypes.c_int, ctypes.c_int, _f64, _vp, _vp, _vp, _vp, _vp, _vp]),
            "oracle_front": (None, [ctypes.c_int, ctypes.c_int, _f64, _vp, _vp, _vp, _vp, _vp]),
            "oracle_dense_layer": (None, [ctypes.c_int, ctypes.c_int, ctypes.c_int, _f64] + [_vp] * 12),
            "oracle_bf16_linear": (None, [ctypes.c_int] * 3 + [_vp] * 4),
            "oracle_silu_mul": (None, [ctypes.c_int, ctypes.c_int, _vp, _vp, _vp]),
            "oracle_ctx_norms": (None, [ctypes.c_int] * 3 + [_f64] + [_vp] * 7),
            "oracle_layer_norms": (None, [ctypes.c_int] * 3 + [_f64] + [_vp] * 4),
            "oracle_k_norm_rope": (None, [ctypes.c_int] * 4 + [_f64, _f64] + [_vp] * 6),
            "oracle_kv_cache_write": (None, [ctypes.c_int] * 4 + [_vp, ctypes.c_int, _i64] + [_vp] * 4),
            "oracle_route": (None, [ctypes.c_int] * 4 + [_vp] * 9),
            "oracle_pool": (None, [ctypes.c_int] * 3 + [_vp] * 6),
            "oracle_gate_up": (ctypes.c_int, [ctypes.c_int] * 5 + [_vp, _vp, _vp, _f32, _vp, _vp, _vp, _vp]),
            "oracle_h_quant": (None, [ctypes.c_int, ctypes.c_int] + [_vp] * 6),
            "oracle_down": (ctypes.c_int, [ctypes.c_int] * 5 + [_vp] * 8),
            "oracle_gather": (None, [ctypes.c_int] * 3 + [_vp] * 3),
            "oracle_layer_step": (ctypes.c_int, [ctypes.c_int] * 5 + [_f64, _vp, _vp, _vp, _vp, _vp]),
            "oracle_moe_step": (ctypes.c_int, [ctypes.c_int] * 5 + [_vp, _vp, _vp]),
            "oracle_num_threads": (ctypes.c_int, []),
            "oracle_set_num_threads": (None, [ctypes.c_int]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ formats


def e2m1_decode(code: int) -> float:
    return lib().oracle_e2m1_decode(code)


def e2m1_encode(v: float) -> int:
    return lib().oracle_e2m1_encode(v)


def e4m3_decode(code: int) -> float:
    return lib().oracle_e4m3_decode(code)


def e4m3_encode(v: float) -> int:
    return lib().oracle_e4m3_encode(v)


def bf16_from_double(v: float) -> int:
    return lib().oracle_bf16_from_double(v)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- quantizer


def nvfp4_quantize(v: np.ndarray):
    """One fp32 tensor [rows, cols] -> (codes [rows, cols/2] u8, sf [rows, cols/16] u8, sg, amax)."""
    v = _c(v, np.float32)
    rows, cols = v.shape
    assert cols % 16 == 0
    codes = np.zeros((rows, cols // 2), np.uint8)
    sf = np.zeros((rows, cols // 16), np.uint8)
    sg = np.zeros(1, np.float32)
    amax = np.zeros(1, np.float32)
    lib().oracle_nvfp4_quantize(_p(v), rows, cols, _p(codes), _p(sf), _p(sg), _p(amax))
    return codes, sf, np.float32(sg[0]), np.float32(amax[0])


def nvfp4_dequantize(codes, sf, sg, rows, cols) -> np.ndarray:
    codes, sf = _c(codes, np.uint8), _c(sf, np.uint8)
    out = np.zeros((rows, cols), np.float64)
    lib().oracle_nvfp4_dequantize(_p(codes), _p(sf), float(sg), rows, cols, _p(out))
    return out


# ------------------------------------------------------------------- stages


def boundary(branch, stream, w_post, w_pre, eps):
    """-> (stream' fp32, x bf16 bits, x before rounding fp64)."""
    branch = _c(branch, np.float64)
    s = np.array(stream, dtype=np.float32, copy=True, order="C")
    rows, H = s.shape
    x = np.zeros((rows, H), np.uint16)
    xe = np.zeros((rows, H), np.float64)
    lib().oracle_boundary(rows, H, eps, _p(branch), _p(s), _p(_c(w_post, np.float32)),
                          _p(_c(w_pre, np.float32)), _p(x), _p(xe))
    return s, x, xe


def front(embedded, w, eps):
    """The first layer's front: embedded bf16 bits [rows, H] -> (stream fp32,
    out bf16 bits, out before rounding fp64)."""
    embedded = _c(embedded, np.uint16)
    rows, H = embedded.shape
    w = _c(w, np.float32)
    stream = np.zeros((rows, H), np.float32)
    out = np.zeros((rows, H), np.uint16)
    exact = np.zeros((rows, H))
    lib().oracle_front(rows, H, eps, _p(embedded), _p(w), _p(stream), _p(out), _p(exact))
    return stream, out, exact


def dense_layer(attn_out, stream, w_post_attn, w_pre_ffn, w13, w2, w_post_ffn, eps):
    """One dense draft layer's MLP block -> dict(stream, x, gu, a, f, x_exact):
    bf16 bits for the intermediates, fp64 for x before its rounding."""
    attn_out = _c(attn_out, np.uint16)
    rows, H = attn_out.shape
    w13, w2 = _c(w13, np.uint16), _c(w2, np.uint16)
    I = w2.shape[1]
    s = np.array(stream, dtype=np.float32, copy=True, order="C")
    out = dict(stream=s, x=np.zeros((rows, H), np.uint16), gu=np.zeros((rows, 2 * I), np.uint16),
               a=np.zeros((rows, I), np.uint16), f=np.zeros((rows, H), np.uint16),
               x_exact=np.zeros((rows, H), np.float64))
    lib().oracle_dense_layer(rows, H, I, eps, _p(attn_out), _p(s), _p(_c(w_post_attn, np.float32)),
                             _p(_c(w_pre_ffn, np.float32)), _p(w13), _p(w2),
                             _p(_c(w_post_ffn, np.float32)), _p(out["x"]), _p(out["gu"]),
                             _p(out["a"]), _p(out["f"]), _p(out["x_exact"]))
    return out


def bf16_linear(a, b):
    """(bf16 bits of a . b^T, its fp64 value before rounding) for bf16-bit
    operands a [M, K] and b [N, K]."""
    a, b = _c(a, np.uint16), _c(b, np.uint16)
    M, K = a.shape
    N = b.shape[0]
    out, exact = np.zeros((M, N), np.uint16), np.zeros((M, N), np.float64)
    lib().oracle_bf16_linear(M, N, K, _p(a), _p(b), _p(out), _p(exact))
    return out, exact


def silu_mul(gu):
    """(bf16 bits of silu(gate) * up, its fp64 value) from bf16 bits gu [rows, 2I]."""
    gu = _c(gu, np.uint16)
    rows, I = gu.shape[0], gu.shape[1] // 2
    out, exact = np.zeros((rows, I), np.uint16), np.zeros((rows, I), np.float64)
    lib().oracle_silu_mul(rows, I, _p(gu), _p(out), _p(exact))
    return out, exact


def context_kv(ctx, positions, w_hidden, w_pre, w_kv, n_kv_heads, head_dim, eps, qk_eps, theta):
    """The draft's context-KV projection -> dict(fc, u, fc_exact, u_exact, kv, k, v, k_exact).
    ctx bf16 bits [n, H]; w_pre fp32 [L, H]; w_kv bf16 bits [L, 2*KVH*D, H]
    (K rows, then V rows); k and v bf16 bits [L, n, KVH, D]."""
    ctx = _c(ctx, np.uint16)
    n, H = ctx.shape
    w_pre = _c(w_pre, np.float32)
    L = w_pre.shape[0]
    KD = n_kv_heads * head_dim
    w_kv = _c(w_kv, np.uint16).reshape(L, 2 * KD, H)
    pos = _c(positions, np.int64)
    out = dict(fc=np.zeros((n, H), np.uint16), u=np.zeros((L, n, H), np.uint16),
               fc_exact=np.zeros((n, H), np.float64), u_exact=np.zeros((L, n, H), np.float64),
               kv=np.zeros((L, n, 2 * KD), np.uint16),
               k=np.zeros((L, n, n_kv_heads, head_dim), np.uint16),
               v=np.zeros((L, n, n_kv_heads, head_dim), np.uint16),
               k_exact=np.zeros((L, n, n_kv_heads, head_dim), np.float64))
    lib().oracle_ctx_norms(n, H, L, eps, _p(ctx), _p(_c(w_hidden, np.float32)), _p(w_pre),
                           _p(out["fc"]), _p(out["u"]), _p(out["fc_exact"]), _p(out["u_exact"]))
    for l in range(L):
        out["kv"][l] = bf16_linear(out["u"][l], w_kv[l])[0]
    lib().oracle_k_norm_rope(L, n, n_kv_heads, head_dim, qk_eps, theta, _p(pos), _p(out["kv"]),
                             _p(out["k"]), _p(out["v"]), _p(out["k_exact"]), None)
    return out


def layer_norms(fc, w_pre, eps):
    """(u bf16 bits [L, n, H], u before rounding) from bf16 bits fc [n, H] (the
    GPU's own, staged): each layer's pre_qkv_proj_norm."""
    fc, w_pre = _c(fc, np.uint16), _c(w_pre, np.float32)
    n, H = fc.shape
    L = w_pre.shape[0]
    u, ue = np.zeros((L, n, H), np.uint16), np.zeros((L, n, H), np.float64)
    lib().oracle_layer_norms(n, H, L, eps, _p(fc), _p(w_pre), _p(u), _p(ue))
    return u, ue


def k_norm_rope(kv, positions, n_kv_heads, head_dim, qk_eps, theta, with_norm=False):
    """(k, v, k_exact[, kn_exact]) from bf16 bits kv [L, n, 2*KVH*D] (the GPU's
    own, staged); kn_exact: the normalised keys before their bf16 cast."""
    kv = _c(kv, np.uint16)
    L, n = kv.shape[:2]
    shape = (L, n, n_kv_heads, head_dim)
    k, v, ke = np.zeros(shape, np.uint16), np.zeros(shape, np.uint16), np.zeros(shape, np.float64)
    kne = np.zeros(shape, np.float64)
    lib().oracle_k_norm_rope(L, n, n_kv_heads, head_dim, qk_eps, theta, _p(_c(positions, np.int64)),
                             _p(kv), _p(k), _p(v), _p(ke), _p(kne))
    return (k, v, ke, kne) if with_norm else (k, v, ke)


def kv_cache_write(k, v, slots, n_slots, k_cache, v_cache):
    """Scatters k, v [L, n, KVH, D] into copies of the caches [L, n_slots, KVH, D]
    by slots ([n] for every layer, or [L, n]); -> (k_cache, v_cache)."""
    k, v = _c(k, np.uint16), _c(v, np.uint16)
    L, n, KVH, D = k.shape
    slots = _c(slots, np.int64)
    stride = 0 if slots.ndim == 1 else slots.shape[1]
    kc = np.array(k_cache, dtype=np.uint16, copy=True, order="C")
    vc = np.array(v_cache, dtype=np.uint16, copy=True, order="C")
    lib().oracle_kv_cache_write(L, n, KVH, D, _p(slots), stride, n_slots, _p(k), _p(v), _p(kc), _p(vc))
    return kc, vc


def route(x, router_w, bias, k):
    x, router_w = _c(x, np.uint16), _c(router_w, np.uint16)
    rows, H = x.shape
    E = router_w.shape[0]
    out = dict(logits=np.zeros((rows, E)), probs=np.zeros((rows, E)),
               ids=np.zeros((rows, k), np.int32), gates=np.zeros((rows, k)),
               flags=np.zeros(rows, np.uint8), gap=np.zeros(rows))
    b = None if bias is None else _c(bias, np.float32)
    lib().oracle_route(rows, H, E, k, _p(x), _p(router_w), _p(b), _p(out["logits"]),
                       _p(out["probs"]), _p(out["ids"]), _p(out["gates"]), _p(out["flags"]),
                       _p(out["gap"]))
    return out


def pool(ids, E):
    ids = _c(ids, np.int32)
    rows, k = ids.shape
    out = dict(count=np.zeros(E, np.int32), offset=np.zeros(E + 1, np.int32),
               pair_order=np.zeros(rows * k, np.int32), active=np.zeros(E, np.int32),
               n_active=np.zeros(1, np.int32))
    lib().oracle_pool(rows, E, k, _p(ids), _p(out["count"]), _p(out["offset"]),
                      _p(out["pair_order"]), _p(out["active"]), _p(out["n_active"]))
    out["n_active"] = int(out["n_active"][0])
    out["active"] = out["active"][: out["n_active"]]
    return out


class LayerWeights:
    """One layer's weights for the oracle.  Expert tensors are given per expert
    (dicts expert -> array); experts that are not given must not be routed to."""

    def __init__(self, E, H, I, w_post, w_pre, router_w, router_bias, w13, w13_sf, w2, w2_sf,
                 gscale):
        self.E, self.H, self.I = E, H, I
        self.w_post = _c(w_post, np.float32)
        self.w_pre = _c(w_pre, np.float32)
        self.router_w = _c(router_w, np.uint16)
        self.router_bias = None if router_bias is None else _c(router_bias, np.float32)
        self.w13 = {e: _c(a, np.uint8) for e, a in w13.items()}
        self.w13_sf = {e: _c(a, np.uint8) for e, a in w13_sf.items()}
        self.w2 = {e: _c(a, np.uint8) for e, a in w2.items()}
        self.w2_sf = {e: _c(a, np.uint8) for e, a in w2_sf.items()}
        self.gscale = _c(gscale, np.float32).reshape(E, 3)
        self._struct = None

    def struct(self):
        if self._struct is None:
            E = self.E

            def table(d):
                t = (ctypes.c_void_p * E)()
                for e, a in d.items():
                    t[e] = a.ctypes.data
                return t

            self._tables = [table(self.w13), table(self.w13_sf), table(self.w2), table(self.w2_sf)]
            s = _LayerWeights()
            s.w_post, s.w_pre = _p(self.w_post), _p(self.w_pre)
            s.router_w, s.router_bias = _p(self.router_w), _p(self.router_bias)
            s.w13, s.w13_sf, s.w2, s.w2_sf = [ctypes.cast(t, _vp) for t in self._tables]
            s.gscale = _p(self.gscale)
            self._struct = s
        return self._struct


def gate_up(w: LayerWeights, k, x_codes, x_sf, x_sg, ids, offset, pair_order):
    rows = ids.shape[0]
    h = np.zeros((rows * k, w.I), np.float32)
    rc = lib().oracle_gate_up(rows, w.H, w.E, k, w.I, ctypes.byref(w.struct()),
                              _p(_c(x_codes, np.uint8)), _p(_c(x_sf, np.uint8)), float(x_sg),
                              _p(_c(ids, np.int32)), _p(_c(offset, np.int32)),
                              _p(_c(pair_order, np.int32)), _p(h))
    if rc:
        raise ValueError("oracle_gate_up: an active expert's weights were not given")
    return h


def h_quant(E, I, offset, h):
    n = h.shape[0]
    out = dict(h_codes=np.zeros((n, I // 2), np.uint8), h_sf=np.zeros((n, I // 16), np.uint8),
               h_sg=np.zeros(E, np.float32), h_amax=np.zeros(E, np.float32))
    lib().oracle_h_quant(E, I, _p(_c(offset, np.int32)), _p(_c(h, np.float32)),
                         _p(out["h_codes"]), _p(out["h_sf"]), _p(out["h_sg"]), _p(out["h_amax"]))
    return out


def down(w: LayerWeights, k, ids, offset, pair_order, h_codes, h_sf, h_sg):
    rows = ids.shape[0]
    o = np.zeros((rows * k, w.H), np.float32)
    rc = lib().oracle_down(rows, w.H, w.E, k, w.I, ctypes.byref(w.struct()),
                           _p(_c(ids, np.int32)), _p(_c(offset, np.int32)),
                           _p(_c(pair_order, np.int32)), _p(_c(h_codes, np.uint8)),
                           _p(_c(h_sf, np.uint8)), _p(_c(h_sg, np.float32)), _p(o))
    if rc:
        raise ValueError("oracle_down: an active expert's weights were not given")
    return o


def gather(gates, o, k):
    gates = _c(gates, np.float64)
    rows = gates.shape[0]
    H = o.shape[1]
    y = np.zeros((rows, H), np.float64)
    lib().oracle_gather(rows, H, k, _p(gates), _p(_c(o, np.float32)), _p(y))
    return y


def _layer_outputs(rows, H, E, k, I):
    n = rows * k
    return dict(
        x=np.zeros((rows, H), np.uint16), x_exact=np.zeros((rows, H)),
        x_codes=np.zeros((rows, H // 2), np.uint8), x_sf=np.zeros((rows, H // 16), np.uint8),
        x_sg=np.zeros(1, np.float32), x_amax=np.zeros(1, np.float32),
        probs=np.zeros((rows, E)), ids=np.zeros((rows, k), np.int32), gates=np.zeros((rows, k)),
        flags=np.zeros(rows, np.uint8), gap=np.zeros(rows),
        count=np.zeros(E, np.int32), offset=np.zeros(E + 1, np.int32),
        pair_order=np.zeros(n, np.int32), active=np.zeros(E, np.int32),
        n_active=np.zeros(1, np.int32),
        h=np.zeros((n, I), np.float32), h_codes=np.zeros((n, I // 2), np.uint8),
        h_sf=np.zeros((n, I // 16), np.uint8), h_sg=np.zeros(E, np.float32),
        h_amax=np.zeros(E, np.float32), o=np.zeros((n, H), np.float32))


def _finish(o):
    o["x_sg"] = np.float32(o["x_sg"][0])
    o["x_amax"] = np.float32(o["x_amax"][0])
    o["n_active"] = int(o["n_active"][0])
    o["active"] = o["active"][: o["n_active"]]
    return o


def layer_step(w: LayerWeights, k, eps, branch, stream, forced_ids=None):
    """One layer: boundary, routing, pooler, NVFP4 experts.  Returns a dict with
    the new fp32 stream and every intermediate."""
    branch = _c(branch, np.float64)
    s = np.array(stream, dtype=np.float32, copy=True, order="C")
    rows, H = s.shape
    o = _layer_outputs(rows, H, w.E, k, w.I)
    st = _LayerOut(**{name: _p(a) for name, a in o.items()})
    fi = None if forced_ids is None else _c(forced_ids, np.int32)
    rc = lib().oracle_layer_step(rows, H, w.E, k, w.I, eps, ctypes.byref(w.struct()), _p(branch),
                                 _p(s), _p(fi), ctypes.byref(st))
    if rc:
        raise ValueError("oracle_layer_step: an active expert's weights were not given")
    o["stream"] = s
    return _finish(o)


def moe_step(w: LayerWeights, k, x, forced_ids=None):
    """A layer's MoE part alone from its bf16 MoE input x (uint16 [rows, H]):
    routing (forced_ids as in layer_step), pooler, the input's NVFP4
    quantization and the experts.  The same arithmetic as layer_step after its
    boundary."""
    x = _c(x, np.uint16)
    rows, H = x.shape
    o = _layer_outputs(rows, H, w.E, k, w.I)
    o["x"][...] = x
    st = _LayerOut(**{name: _p(a) for name, a in o.items()})
    fi = None if forced_ids is None else _c(forced_ids, np.int32)
    rc = lib().oracle_moe_step(rows, H, w.E, k, w.I, ctypes.byref(w.struct()), _p(fi), ctypes.byref(st))
    if rc:
        raise ValueError("oracle_moe_step: an active expert's weights were not given")
    return _finish(o)


def num_threads() -> int:
    return lib().oracle_num_threads()


def set_num_threads(n: int) -> None:
    """Host threads of the oracle's parallel loops (timing only; results do not change)."""
    lib().oracle_set_num_threads(int(n))
