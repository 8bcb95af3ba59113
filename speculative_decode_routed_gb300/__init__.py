"""GB300 (sm_103a) routed NVFP4 mixture-of-experts decode layer-step.

A thin ctypes binding over ``libmoe_decode.so`` (see ``include/moe_decode.h``
for the contract of every entry point).  The functions below keep the C
names and only marshal arguments: device pointers come from torch tensors'
``data_ptr()``, the CUDA stream from ``torch.cuda.current_stream()``.  Every
step of the computation runs in the library's kernels; there is no other
code path, and loading fails loudly if the library was not built.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

_HERE = os.path.dirname(os.path.abspath(__file__))
# MOE_DECODE_LIB may name another build of the library (the bounds-check
# variant, libmoe_decode_bounds.so, beside this file)
LIB_PATH = os.environ.get("MOE_DECODE_LIB") or os.path.join(_HERE, "libmoe_decode.so")

MOE_OK, MOE_EINVAL, MOE_EUNSUPPORTED, MOE_ECUDA, MOE_ENOMEM, MOE_EDEVICE = 0, -1, -2, -3, -4, -5
# moe_decode_dims.code_layout
MOE_CODES_ROW_MAJOR, MOE_CODES_TILED, MOE_CODES_TILED_COPY = 0, 1, 2

# Every symbol include/moe_decode.h declares.
EXPORTS = (
    "moe_decode_create", "moe_decode_layer", "moe_decode_final", "moe_decode_front", "moe_decode_step",
    "moe_decode_step_graph", "moe_decode_step_host", "moe_decode_layer_profile", "moe_decode_debug",
    "moe_decode_last_error", "moe_decode_workspace_bytes", "moe_decode_weight_copy_bytes",
    "moe_decode_step_kernel_count", "moe_tiled_code_bytes", "moe_tile_codes",
    "moe_decode_set_wait_limit", "moe_decode_selftest_wait_timeout", "moe_decode_build_info",
    "moe_decode_destroy", "moe_decode_strerror", "moe_decode_error_message",
    "moe_nvfp4_quantize", "moe_nvfp4_quantize_noalloc",
    "moe_dense_create", "moe_dense_layer", "moe_dense_layer_profile", "moe_dense_debug",
    "moe_dense_layer_host", "moe_dense_kernel_count", "moe_dense_last_error", "moe_dense_destroy",
    "moe_ctxkv_create", "moe_ctxkv_project", "moe_ctxkv_project_host", "moe_ctxkv_profile", "moe_ctxkv_debug",
    "moe_ctxkv_last_error", "moe_ctxkv_kernel_count", "moe_ctxkv_destroy",
)


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = _lib().moe_decode_error_message().decode()
        super().__init__(f"{where}: {_lib().moe_decode_strerror(code).decode()} ({code}): {msg}")


class Dims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("n_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("inter", ctypes.c_int), ("max_rows", ctypes.c_int), ("n_layers", ctypes.c_int),
                ("eps", ctypes.c_float), ("code_layout", ctypes.c_int)]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "w_post", "w_pre", "router_w", "router_bias", "w13", "w13_sf", "w2", "w2_sf", "w_gscale")]


class DenseDims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("inter", ctypes.c_int), ("max_rows", ctypes.c_int),
                ("eps", ctypes.c_float)]


class DenseWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("w_post_attn", "w_pre_ffn", "w13", "w2", "w_post_ffn")]


class DenseDebugView(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("x", "gu", "a", "f")]


class CtxKvDims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("n_layers", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("max_ctx", ctypes.c_int), ("max_position", ctypes.c_int),
                ("eps", ctypes.c_float), ("qk_eps", ctypes.c_float), ("rope_theta", ctypes.c_double)]


class CtxKvWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("w_hidden", "w_pre", "w_kv")]


class CtxKvDebugView(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("fc", "u", "kv", "k", "v")]


class DebugView(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "x", "x_codes", "x_sf", "x_sg", "logits", "ids", "gates", "flags", "count", "offset",
        "pair_order", "pos_of_pair", "active", "n_active", "h", "h_sg", "h_codes", "h_sf", "o")]


_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        sig = {
            "moe_decode_create": (i32, [ctypes.POINTER(Dims), ctypes.POINTER(LayerWeights), vp, vp,
                                        ctypes.POINTER(vp)]),
            "moe_decode_layer": (i32, [vp, i32, i32, vp, vp, vp]),
            "moe_decode_final": (i32, [vp, i32, vp, vp, vp, vp]),
            "moe_decode_front": (i32, [vp, i32, vp, vp, vp, vp, vp, vp]),
            "moe_decode_step": (i32, [vp, i32, vp, vp, vp, vp]),
            "moe_decode_step_graph": (i32, [vp, i32, vp, vp, vp, vp]),
            "moe_decode_step_host": (i32, [vp, i32, vp, vp, vp, vp]),
            "moe_decode_layer_profile": (i32, [vp, i32, i32, vp, vp, vp, vp]),
            "moe_decode_debug": (i32, [vp, ctypes.POINTER(DebugView)]),
            "moe_decode_last_error": (i32, [vp]),
            "moe_decode_workspace_bytes": (ctypes.c_size_t, [vp]),
            "moe_decode_weight_copy_bytes": (ctypes.c_size_t, [vp]),
            "moe_tiled_code_bytes": (i64, [i64, i64]),
            "moe_tile_codes": (i32, [vp, i64, i64, vp, vp]),
            "moe_decode_set_wait_limit": (i32, [vp, ctypes.c_uint64]),
            "moe_decode_build_info": (i32, []),
            "moe_decode_selftest_wait_timeout": (i32, [vp, i32, vp, vp, vp]),
            "moe_decode_step_kernel_count": (i32, [vp]),
            "moe_decode_destroy": (None, [vp]),
            "moe_decode_strerror": (ctypes.c_char_p, [i32]),
            "moe_decode_error_message": (ctypes.c_char_p, []),
            "moe_nvfp4_quantize": (i32, [vp, i64, i64, vp, vp, vp, vp, vp]),
            "moe_nvfp4_quantize_noalloc": (i32, [vp, i64, i64, vp, vp, vp, vp]),
            "moe_dense_create": (i32, [ctypes.POINTER(DenseDims), ctypes.POINTER(DenseWeights),
                                       ctypes.POINTER(vp)]),
            "moe_dense_layer": (i32, [vp, i32, vp, vp, vp]),
            "moe_dense_layer_profile": (i32, [vp, i32, vp, vp, vp, vp]),
            "moe_dense_debug": (i32, [vp, ctypes.POINTER(DenseDebugView)]),
            "moe_dense_layer_host": (i32, [vp, i32, vp, vp, vp]),
            "moe_dense_kernel_count": (i32, [vp, i32]),
            "moe_dense_last_error": (i32, [vp]),
            "moe_dense_destroy": (None, [vp]),
            "moe_ctxkv_create": (i32, [ctypes.POINTER(CtxKvDims), ctypes.POINTER(CtxKvWeights),
                                       ctypes.POINTER(vp)]),
            "moe_ctxkv_project": (i32, [vp, i32, vp, vp, vp, i32, vp, vp, i64, vp, vp, vp]),
            "moe_ctxkv_project_host": (i32, [vp, i32, vp, vp, vp, i32, vp, vp, i64, vp, vp, vp]),
            "moe_ctxkv_profile": (i32, [vp, i32, vp, vp, vp, i32, vp, vp, i64, vp, vp]),
            "moe_ctxkv_debug": (i32, [vp, ctypes.POINTER(CtxKvDebugView)]),
            "moe_ctxkv_last_error": (i32, [vp]),
            "moe_ctxkv_kernel_count": (i32, [vp, i32]),
            "moe_ctxkv_destroy": (None, [vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def lib():
    """The loaded library (raises ImportError if it was not built)."""
    return _lib()


def _check(rc: int, where: str):
    if rc != MOE_OK:
        raise MoeError(rc, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


# ------------------------------------------------------------------ C names


def moe_decode_create(dims: Dims, layers, w_post_final, w_final) -> ctypes.c_void_p:
    arr = (LayerWeights * len(layers))(*layers)
    h = ctypes.c_void_p()
    _check(_lib().moe_decode_create(ctypes.byref(dims), arr, _ptr(w_post_final), _ptr(w_final),
                                    ctypes.byref(h)), "moe_decode_create")
    return h


def moe_decode_layer(h, layer, rows, branch, stream_buf, stream=None):
    _check(_lib().moe_decode_layer(h, layer, rows, _ptr(branch), _ptr(stream_buf),
                                   _stream(stream)), "moe_decode_layer")


def moe_decode_final(h, rows, stream_buf, out, aux=None, stream=None):
    _check(_lib().moe_decode_final(h, rows, _ptr(stream_buf), _ptr(out), _ptr(aux), _stream(stream)),
           "moe_decode_final")


def moe_decode_front(h, rows, embedded, w_norm, stream_buf, attn_input, aux=None, stream=None):
    _check(_lib().moe_decode_front(h, rows, _ptr(embedded), _ptr(w_norm), _ptr(stream_buf),
                                   _ptr(attn_input), _ptr(aux), _stream(stream)), "moe_decode_front")


def moe_decode_step(h, rows, branch, stream_buf, out, stream=None):
    _check(_lib().moe_decode_step(h, rows, _ptr(branch), _ptr(stream_buf), _ptr(out),
                                  _stream(stream)), "moe_decode_step")


def moe_decode_step_graph(h, rows, branch, stream_buf, out, stream=None):
    _check(_lib().moe_decode_step_graph(h, rows, _ptr(branch), _ptr(stream_buf), _ptr(out),
                                        _stream(stream)), "moe_decode_step_graph")


def moe_decode_step_host(h, rows, branch_host, stream_host, out_host, stream=None):
    """Host (CPU) tensors, ideally pinned; stream_host is updated in place."""
    _check(_lib().moe_decode_step_host(h, rows, _ptr(branch_host), _ptr(stream_host),
                                       _ptr(out_host), _stream(stream)), "moe_decode_step_host")


def moe_decode_layer_profile(h, layer, rows, branch, stream_buf, stream=None):
    """-> [boundary, router, pool, gate/up, down] kernel durations in ms."""
    ms = (ctypes.c_float * 5)()
    _check(_lib().moe_decode_layer_profile(h, layer, rows, _ptr(branch), _ptr(stream_buf),
                                           _stream(stream), ms), "moe_decode_layer_profile")
    return list(ms)


def moe_decode_debug(h) -> DebugView:
    v = DebugView()
    _check(_lib().moe_decode_debug(h, ctypes.byref(v)), "moe_decode_debug")
    return v


def moe_decode_last_error(h) -> int:
    return _lib().moe_decode_last_error(h)


def moe_decode_workspace_bytes(h) -> int:
    return _lib().moe_decode_workspace_bytes(h)


def moe_decode_weight_copy_bytes(h) -> int:
    return _lib().moe_decode_weight_copy_bytes(h)


def moe_tiled_code_bytes(rows, row_bytes) -> int:
    n = _lib().moe_tiled_code_bytes(rows, row_bytes)
    _check(min(n, 0), "moe_tiled_code_bytes")
    return n


def moe_tile_codes(src, dst, stream=None):
    """src u8 CUDA tensor [rows, row_bytes] (row-major codes) -> dst u8 CUDA
    tensor of moe_tiled_code_bytes(rows, row_bytes) bytes (the 16 KB tiles)."""
    rows, row_bytes = src.shape
    _check(_lib().moe_tile_codes(_ptr(src), rows, row_bytes, _ptr(dst), _stream(stream)),
           "moe_tile_codes")


def moe_decode_step_kernel_count(h) -> int:
    return _lib().moe_decode_step_kernel_count(h)


def moe_decode_destroy(h):
    _lib().moe_decode_destroy(h)


def moe_nvfp4_quantize(v, codes, sf, sg, amax, stream=None):
    """v fp32 [rows, cols] -> codes u8 [rows, cols/2], sf u8 [rows, cols/16], sg / amax fp32 [1]
    (all CUDA tensors)."""
    rows, cols = v.shape
    _check(_lib().moe_nvfp4_quantize(_ptr(v), rows, cols, _ptr(codes), _ptr(sf), _ptr(sg),
                                     _ptr(amax), _stream(stream)), "moe_nvfp4_quantize")


def moe_nvfp4_quantize_noalloc(v, codes, sf, sg, stream=None):
    """As moe_nvfp4_quantize, for callers that cannot allocate device memory:
    the max |v| reduction uses a fixed scratch array inside the library
    (at most 2**30 elements; calls that overlap on the GPU race on it)."""
    rows, cols = v.shape
    _check(_lib().moe_nvfp4_quantize_noalloc(_ptr(v), rows, cols, _ptr(codes), _ptr(sf), _ptr(sg),
                                             _stream(stream)), "moe_nvfp4_quantize_noalloc")


# --------------------------------------------------------- torch convenience


@dataclass
class LayerTensors:
    """One layer's device tensors (kept alive by the handle)."""
    w_post: object
    w_pre: object
    router_w: object          # bf16 [E, H]
    router_bias: object       # fp32 [E] or None
    w13: object               # u8 [E, 2I, H/2], or its 16 KB tiles (MOE_CODES_TILED)
    w13_sf: object            # u8 [E, 2I, H/16]
    w2: object                # u8 [E, H, I/2], or its 16 KB tiles (MOE_CODES_TILED)
    w2_sf: object             # u8 [E, H, I/16]
    w_gscale: object          # fp32 [E, 3]

    def struct(self) -> LayerWeights:
        return LayerWeights(*[None if t is None else t.data_ptr() for t in (
            self.w_post, self.w_pre, self.router_w, self.router_bias, self.w13, self.w13_sf,
            self.w2, self.w2_sf, self.w_gscale)])


class MoEDecode:
    """Owns a handle over caller-owned device weights (torch tensors)."""

    def __init__(self, hidden, n_experts, top_k, inter, max_rows, layers, w_post_final=None,
                 w_final=None, eps=1e-6, code_layout=MOE_CODES_ROW_MAJOR):
        self.dims = Dims(hidden, n_experts, top_k, inter, max_rows, len(layers), eps, code_layout)
        self.layers = list(layers)
        self.w_post_final, self.w_final = w_post_final, w_final
        self.handle = moe_decode_create(self.dims, [l.struct() for l in self.layers],
                                        w_post_final, w_final)

    def layer(self, layer, rows, branch, stream_buf, stream=None):
        moe_decode_layer(self.handle, layer, rows, branch, stream_buf, stream)

    def final(self, rows, stream_buf, out, aux=None, stream=None):
        moe_decode_final(self.handle, rows, stream_buf, out, aux, stream)

    def front(self, rows, embedded, w_norm, stream_buf, attn_input, aux=None, stream=None):
        moe_decode_front(self.handle, rows, embedded, w_norm, stream_buf, attn_input, aux, stream)

    def step(self, rows, branch, stream_buf, out, stream=None):
        moe_decode_step(self.handle, rows, branch, stream_buf, out, stream)

    def step_graph(self, rows, branch, stream_buf, out, stream=None):
        moe_decode_step_graph(self.handle, rows, branch, stream_buf, out, stream)

    def step_host(self, rows, branch_host, stream_host, out_host, stream=None):
        moe_decode_step_host(self.handle, rows, branch_host, stream_host, out_host, stream)

    def layer_profile(self, layer, rows, branch, stream_buf, stream=None):
        return moe_decode_layer_profile(self.handle, layer, rows, branch, stream_buf, stream)

    def debug(self) -> DebugView:
        return moe_decode_debug(self.handle)

    def set_wait_limit(self, limit_ns):
        _check(_lib().moe_decode_set_wait_limit(self.handle, int(limit_ns)), "moe_decode_set_wait_limit")

    def selftest_wait_timeout(self, rows, branch, stream_buf, stream=None):
        _check(_lib().moe_decode_selftest_wait_timeout(self.handle, rows, _ptr(branch), _ptr(stream_buf),
                                                       _stream(stream)), "moe_decode_selftest_wait_timeout")

    def last_error(self) -> int:
        return moe_decode_last_error(self.handle)

    def check(self):
        rc = self.last_error()
        if rc != MOE_OK:
            raise MoeError(rc, "device")

    def close(self):
        if self.handle:
            moe_decode_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------------- dense draft layer


class DenseLayer:
    """One dense draft layer's MLP block (moe_dense_*) over caller-owned
    device tensors: w_post_attn, w_pre_ffn, w_post_ffn fp32 [H]; w13 bf16
    [2I, H] (gate rows, then up rows); w2 bf16 [H, I]."""

    def __init__(self, hidden, inter, max_rows, w_post_attn, w_pre_ffn, w13, w2, w_post_ffn,
                 eps=1e-6):
        dims = DenseDims(hidden, inter, max_rows, eps)
        self._keep = (w_post_attn, w_pre_ffn, w13, w2, w_post_ffn)
        wts = DenseWeights(*[t.data_ptr() for t in self._keep])
        out = ctypes.c_void_p()
        _check(_lib().moe_dense_create(ctypes.byref(dims), ctypes.byref(wts), ctypes.byref(out)),
               "moe_dense_create")
        self.handle = out

    def layer(self, rows, attn_out, stream_buf, stream=None):
        _check(_lib().moe_dense_layer(self.handle, rows, _ptr(attn_out), _ptr(stream_buf),
                                      _stream(stream)), "moe_dense_layer")

    def layer_host(self, rows, attn_host, stream_host, stream=None):
        """The layer on host tensors (page-locked for the fastest path)."""
        _check(_lib().moe_dense_layer_host(self.handle, rows, _ptr(attn_host), _ptr(stream_host),
                                           _stream(stream)), "moe_dense_layer_host")

    def layer_profile(self, rows, attn_out, stream_buf, stream=None):
        ms = (ctypes.c_float * 5)()
        _check(_lib().moe_dense_layer_profile(self.handle, rows, _ptr(attn_out), _ptr(stream_buf),
                                              _stream(stream), ms), "moe_dense_layer_profile")
        return list(ms)

    def kernel_count(self, rows):
        n = _lib().moe_dense_kernel_count(self.handle, rows)
        _check(min(n, 0), "moe_dense_kernel_count")
        return n

    def debug(self) -> DenseDebugView:
        v = DenseDebugView()
        _check(_lib().moe_dense_debug(self.handle, ctypes.byref(v)), "moe_dense_debug")
        return v

    def check(self):
        _check(_lib().moe_dense_last_error(self.handle), "moe_dense_last_error")

    def close(self):
        if self.handle:
            _lib().moe_dense_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class ContextKV:
    """The draft's context-KV projection (moe_ctxkv_*) over caller-owned device
    tensors: w_hidden fp32 [H]; w_pre fp32 [L, H]; w_kv bf16 [L, 2*KVH*D, H]
    (each layer's K rows, then V rows)."""

    def __init__(self, hidden, n_layers, n_kv_heads, head_dim, max_ctx, w_hidden, w_pre, w_kv,
                 eps=1e-6, qk_eps=1e-6, rope_theta=10000.0, max_position=0):
        dims = CtxKvDims(hidden, n_layers, n_kv_heads, head_dim, max_ctx, max_position, eps, qk_eps,
                         rope_theta)
        self.dims = dims
        self._keep = (w_hidden, w_pre, w_kv)
        wts = CtxKvWeights(*[t.data_ptr() for t in self._keep])
        out = ctypes.c_void_p()
        _check(_lib().moe_ctxkv_create(ctypes.byref(dims), ctypes.byref(wts), ctypes.byref(out)),
               "moe_ctxkv_create")
        self.handle = out

    @staticmethod
    def _slot_args(slots, k_cache, v_cache):
        if slots is None:
            return None, 0, None, None, 0
        stride = 0 if slots.dim() == 1 else slots.shape[1]
        return _ptr(slots), stride, _ptr(k_cache), _ptr(v_cache), k_cache.shape[1]

    def project(self, n_ctx, context, positions, slots=None, k_cache=None, v_cache=None,
                k_out=None, v_out=None, stream=None):
        sp, stride, kc, vc, n_slots = self._slot_args(slots, k_cache, v_cache)
        _check(_lib().moe_ctxkv_project(self.handle, n_ctx, _ptr(context), _ptr(positions), sp, stride,
                                        kc, vc, n_slots, _ptr(k_out), _ptr(v_out), _stream(stream)),
               "moe_ctxkv_project")

    def project_host(self, n_ctx, context, positions, k_out, v_out, slots=None, k_cache=None, v_cache=None,
                     stream=None):
        """The projection with host tensors for the context, positions, slots and
        outputs (page-locked for the fastest path); the caches are device tensors."""
        sp, stride, kc, vc, n_slots = self._slot_args(slots, k_cache, v_cache)
        _check(_lib().moe_ctxkv_project_host(self.handle, n_ctx, _ptr(context), _ptr(positions), sp, stride,
                                             kc, vc, n_slots, _ptr(k_out), _ptr(v_out), _stream(stream)),
               "moe_ctxkv_project_host")

    def profile(self, n_ctx, context, positions, slots=None, k_cache=None, v_cache=None, stream=None):
        sp, stride, kc, vc, n_slots = self._slot_args(slots, k_cache, v_cache)
        ms = (ctypes.c_float * 3)()
        _check(_lib().moe_ctxkv_profile(self.handle, n_ctx, _ptr(context), _ptr(positions), sp, stride,
                                        kc, vc, n_slots, _stream(stream), ms), "moe_ctxkv_profile")
        return list(ms)

    def kernel_count(self, n_ctx):
        n = _lib().moe_ctxkv_kernel_count(self.handle, n_ctx)
        _check(min(n, 0), "moe_ctxkv_kernel_count")
        return n

    def debug(self) -> CtxKvDebugView:
        v = CtxKvDebugView()
        _check(_lib().moe_ctxkv_debug(self.handle, ctypes.byref(v)), "moe_ctxkv_debug")
        return v

    def check(self):
        _check(_lib().moe_ctxkv_last_error(self.handle), "moe_ctxkv_last_error")

    def close(self):
        if self.handle:
            _lib().moe_ctxkv_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
