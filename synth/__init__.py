"""Seeded synthetic inputs shared by the CPU oracle's tests and the GPU path.

This module holds no arithmetic of the MoE decode step: it maps a
(seed, tag, element index) triple to a pseudo-random value with Philox4x32-10
(Salmon et al., SC'11) and an Irwin-Hall(8) approximately-normal deviate, on
the host (``synth_host.c``) and, independently, on the device
(``synth_dev.cu``).  Both produce the same bits; a GPU test checks that.

It also holds the workload recipes: the shapes and value distributions of the
synthetic configurations (a tiny correctness layer, one serving-width layer,
eight chained layers, a batch/skew sweep and a 16-layer stack).  Expert
weights are produced here as raw fp32 normals only; turning them into NVFP4
is the method's arithmetic and is done by the oracle (host) or by the
library's quantizer (device), each on its own.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(_HERE, "libsynth_host.so")
DEV_LIB = os.path.join(_HERE, "libsynth_dev.so")

# Tensor kinds, the low byte of a Philox key tag.
KIND_STREAM = 1
KIND_BRANCH = 2
KIND_W_POST = 3
KIND_W_PRE = 4
KIND_ROUTER = 5
KIND_GATE = 6
KIND_UP = 7
KIND_DOWN = 8
KIND_W_POST_FINAL = 9
KIND_W_FINAL = 10
KIND_ZIPF_PERM = 11
KIND_EMBED = 12
KIND_W_FRONT = 13
KIND_DENSE_W13 = 14
KIND_DENSE_W2 = 15
KIND_W_POST_FFN = 16
KIND_CTX = 17
KIND_W_HIDDEN = 18
KIND_W_PRE_QKV = 19
KIND_W_KV = 20
KIND_CTX_PLACE = 21


def tag(kind: int, layer: int = 0, index: int = 0) -> int:
    """Philox key word 1 for tensor `kind` of `layer` (and expert / variant `index`)."""
    if not (0 <= kind < 256 and 0 <= layer < 256 and 0 <= index < 65536):
        raise ValueError("tag field out of range")
    return kind | (layer << 8) | (index << 16)


_host = None
_dev = None


def _load_host():
    global _host
    if _host is None:
        if not os.path.exists(HOST_LIB):
            raise RuntimeError(f"{HOST_LIB} missing: run __graft_entry__.build() first")
        lib = ctypes.CDLL(HOST_LIB)
        u32, u64, f32 = ctypes.c_uint32, ctypes.c_uint64, ctypes.c_float
        vp = ctypes.c_void_p
        lib.synth_philox4x32_10.argtypes = [vp, vp, vp]
        lib.synth_philox4x32_10.restype = None
        lib.synth_unit_normal.argtypes = [u32, u32, u64]
        lib.synth_unit_normal.restype = f32
        lib.synth_normal.argtypes = [u32, u32, u64, f32, f32]
        lib.synth_normal.restype = f32
        lib.synth_f32_to_bf16.argtypes = [f32]
        lib.synth_f32_to_bf16.restype = ctypes.c_uint16
        lib.synth_normal_f32.argtypes = [vp, u64, u32, u32, f32, f32]
        lib.synth_normal_f32.restype = None
        lib.synth_normal_bf16.argtypes = [vp, u64, u32, u32, f32, f32]
        lib.synth_normal_bf16.restype = None
        lib.synth_philox_words.argtypes = [vp, u64, u32, u32]
        lib.synth_philox_words.restype = None
        _host = lib
    return _host


def _load_dev():
    global _dev
    if _dev is None:
        if not os.path.exists(DEV_LIB):
            raise RuntimeError(f"{DEV_LIB} missing: run __graft_entry__.build() first")
        lib = ctypes.CDLL(DEV_LIB)
        u32, u64, f32, vp = ctypes.c_uint32, ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p
        for name in ("synth_dev_normal_f32", "synth_dev_normal_bf16"):
            fn = getattr(lib, name)
            fn.argtypes = [vp, u64, u32, u32, f32, f32, vp]
            fn.restype = ctypes.c_int
        _dev = lib
    return _dev


# ----------------------------------------------------------------------------- host


def philox(ctr, key) -> np.ndarray:
    c = np.asarray(ctr, dtype=np.uint32)
    k = np.asarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    _load_host().synth_philox4x32_10(c.ctypes.data, k.ctypes.data, out.ctypes.data)
    return out


def philox_words(n_blocks: int, seed: int, tg: int) -> np.ndarray:
    out = np.empty((n_blocks, 4), dtype=np.uint32)
    _load_host().synth_philox_words(out.ctypes.data, n_blocks, seed, tg)
    return out


def normal_f32(shape, seed: int, tg: int, mu: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _load_host().synth_normal_f32(out.ctypes.data, out.size, seed, tg, mu, sigma)
    return out


def normal_bf16(shape, seed: int, tg: int, mu: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    """bf16 bit patterns (uint16)."""
    out = np.empty(shape, dtype=np.uint16)
    _load_host().synth_normal_bf16(out.ctypes.data, out.size, seed, tg, mu, sigma)
    return out


# ----------------------------------------------------------------------------- device


def dev_normal_f32(t, seed: int, tg: int, mu: float = 0.0, sigma: float = 1.0, stream=None):
    """Fill the contiguous fp32 CUDA tensor `t` in place."""
    import torch

    assert t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()
    s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    rc = _load_dev().synth_dev_normal_f32(t.data_ptr(), t.numel(), seed, tg, mu, sigma, s)
    if rc != 0:
        raise RuntimeError(f"synth_dev_normal_f32 failed: cuda error {rc}")
    return t


def dev_normal_bf16(t, seed: int, tg: int, mu: float = 0.0, sigma: float = 1.0, stream=None):
    import torch

    assert t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()
    s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    rc = _load_dev().synth_dev_normal_bf16(t.data_ptr(), t.numel(), seed, tg, mu, sigma, s)
    if rc != 0:
        raise RuntimeError(f"synth_dev_normal_bf16 failed: cuda error {rc}")
    return t


# ----------------------------------------------------------------------------- workloads


@dataclass(frozen=True)
class Workload:
    """Shapes and value distributions of one synthetic configuration."""

    name: str
    rows: int            # b: rows of the step (1 + 7 speculative tokens = 8)
    hidden: int          # H
    n_experts: int       # E
    top_k: int           # k
    inter: int           # I: expert intermediate width
    n_layers: int = 1
    zipf_bias: bool = False
    eps: float = 1e-6
    seed: int = 0
    # value distributions (mean, std) of the raw fp32 inputs
    stream_dist: tuple = (0.0, 1.0)
    branch_dist: tuple = (0.0, 1.0)
    norm_dist: tuple = (1.0, 0.1)
    router_dist: tuple = (0.0, 1.0 / 16.0)   # N(0, 1/256): variance 1/256
    expert_dist: tuple = (0.0, 0.02)
    notes: str = field(default="", compare=False)

    def with_rows(self, rows: int) -> "Workload":
        d = dict(self.__dict__)
        d["rows"] = rows
        return Workload(**d)


WORKLOADS = {
    "tiny": Workload("tiny", rows=8, hidden=256, n_experts=8, top_k=2, inter=128),
    "serving": Workload("serving", rows=8, hidden=7168, n_experts=256, top_k=8, inter=2048),
    "chained8": Workload("chained8", rows=8, hidden=5120, n_experts=128, top_k=8, inter=1536,
                         n_layers=8),
    "sweep": Workload("sweep", rows=8, hidden=7168, n_experts=256, top_k=8, inter=2048,
                      zipf_bias=True),
    "stack16": Workload("stack16", rows=8, hidden=7168, n_experts=256, top_k=8, inter=2048,
                        n_layers=16),
    # serving widths with 64 experts (~1.6 GB of weights): small enough for
    # multi-pass profiler captures, still far larger than L2
    "serving_e64": Workload("serving_e64", rows=8, hidden=7168, n_experts=64, top_k=8,
                            inter=2048),
}
SWEEP_ROWS = (1, 8, 32, 64, 128)

# Dense draft layers (no experts: n_experts and top_k are 0).  The pages give
# no draft widths; hidden follows the target and the MLP is four times as wide,
# so one layer's bf16 weights (1.23 GB) dwarf the L2.
DENSE_WORKLOADS = {
    "draft_dense": Workload("draft_dense", rows=8, hidden=7168, n_experts=0, top_k=0,
                            inter=28672),
    "draft_dense_small": Workload("draft_dense_small", rows=8, hidden=256, n_experts=0, top_k=0,
                                  inter=384),
}


def step_inputs(w: Workload, variant: int = 0):
    """(stream fp32 [b,H], branch bf16-bits [b,H]) of one step; `variant` selects
    an independent draw (the bench cycles through several)."""
    b, h = w.rows, w.hidden
    stream = normal_f32((b, h), w.seed, tag(KIND_STREAM, 0, variant), *w.stream_dist)
    branch = normal_bf16((b, h), w.seed, tag(KIND_BRANCH, 0, variant), *w.branch_dist)
    return stream, branch


def norm_weights(w: Workload, layer: int):
    """(w_post, w_pre) fp32 [H] of one layer: 1 + 0.1 N(0,1)."""
    h = w.hidden
    return (normal_f32((h,), w.seed, tag(KIND_W_POST, layer), *w.norm_dist),
            normal_f32((h,), w.seed, tag(KIND_W_PRE, layer), *w.norm_dist))


def final_norm_weights(w: Workload):
    h = w.hidden
    return (normal_f32((h,), w.seed, tag(KIND_W_POST_FINAL), *w.norm_dist),
            normal_f32((h,), w.seed, tag(KIND_W_FINAL), *w.norm_dist))


def front_inputs(w: Workload, variant: int = 0):
    """The first layer's front: (embedded tokens bf16 bits [b, H] ~ N(0, 1),
    its input norm weight fp32 [H] = 1 + 0.1 N(0, 1))."""
    emb = normal_bf16((w.rows, w.hidden), w.seed, tag(KIND_EMBED, 0, variant), *w.branch_dist)
    wn = normal_f32((w.hidden,), w.seed, tag(KIND_W_FRONT), *w.norm_dist)
    return emb, wn


def router_weights(w: Workload, layer: int) -> np.ndarray:
    """bf16 bits [E, H]."""
    return normal_bf16((w.n_experts, w.hidden), w.seed, tag(KIND_ROUTER, layer), *w.router_dist)


def router_bias(w: Workload, layer: int):
    """fp32 [E] additive logit bias, or None.  A seeded permutation ranks the
    experts 1..E; the bias is 2.0 * rank^-1.1 (Zipf, s = 1.1, hottest +2.0)."""
    if not w.zipf_bias:
        return None
    words = philox_words(w.n_experts, w.seed, tag(KIND_ZIPF_PERM, layer))[:, 0]
    order = np.argsort(words, kind="stable")        # order[r] = expert of rank r+1
    rank = np.empty(w.n_experts, dtype=np.float64)
    rank[order] = np.arange(1, w.n_experts + 1, dtype=np.float64)
    return (2.0 * rank ** -1.1).astype(np.float32)


def expert_raw(w: Workload, layer: int, expert: int, which: str) -> np.ndarray:
    """Raw fp32 weights of one projection of one expert, K-major:
    gate/up [I, H], down [H, I]."""
    kind = {"gate": KIND_GATE, "up": KIND_UP, "down": KIND_DOWN}[which]
    shape = (w.hidden, w.inter) if which == "down" else (w.inter, w.hidden)
    return normal_f32(shape, w.seed, tag(kind, layer, expert), *w.expert_dist)


def dev_expert_raw(out, w: Workload, layer: int, expert: int, which: str, stream=None):
    """Device twin of expert_raw, into the fp32 CUDA tensor `out`."""
    kind = {"gate": KIND_GATE, "up": KIND_UP, "down": KIND_DOWN}[which]
    return dev_normal_f32(out, w.seed, tag(kind, layer, expert), *w.expert_dist, stream=stream)


# ----------------------------------------------------------------------------- dense draft layer


def dense_norm_weights(w: Workload, layer: int):
    """(w_post_attn, w_pre_ffn, w_post_ffn) fp32 [H] of one dense layer, each
    1 + 0.1 N(0, 1); the first two are the routed layers' (w_post, w_pre)."""
    post_attn, pre_ffn = norm_weights(w, layer)
    post_ffn = normal_f32((w.hidden,), w.seed, tag(KIND_W_POST_FFN, layer), *w.norm_dist)
    return post_attn, pre_ffn, post_ffn


def dense_weights(w: Workload, layer: int):
    """(w13 bf16 bits [2I, H]: gate rows then up rows, w2 bf16 bits [H, I]),
    every entry N(0, 0.02)."""
    w13 = normal_bf16((2 * w.inter, w.hidden), w.seed, tag(KIND_DENSE_W13, layer), *w.expert_dist)
    w2 = normal_bf16((w.hidden, w.inter), w.seed, tag(KIND_DENSE_W2, layer), *w.expert_dist)
    return w13, w2


def dev_dense_weights(w13, w2, w: Workload, layer: int, stream=None):
    """Device twin of dense_weights, into bf16 CUDA tensors [2I, H] and [H, I]."""
    dev_normal_bf16(w13, w.seed, tag(KIND_DENSE_W13, layer), *w.expert_dist, stream=stream)
    dev_normal_bf16(w2, w.seed, tag(KIND_DENSE_W2, layer), *w.expert_dist, stream=stream)
    return w13, w2


# ----------------------------------------------------------------------------- draft context-KV


@dataclass(frozen=True)
class CtxKvWorkload:
    """Shapes and value distributions of one context-KV projection."""

    name: str
    n_ctx: int           # context rows per call
    hidden: int          # H
    n_layers: int        # L: draft layers
    n_kv_heads: int      # KVH
    head_dim: int        # D
    rope_theta: float = 10000.0
    max_position: int = 32768
    n_slots: int = 4096  # cache slots per layer (256 blocks of 16)
    eps: float = 1e-6
    qk_eps: float = 1e-6
    seed: int = 0
    ctx_dist: tuple = (0.0, 1.0)
    norm_dist: tuple = (1.0, 0.1)
    weight_dist: tuple = (0.0, 0.02)

    def with_ctx(self, n_ctx: int) -> "CtxKvWorkload":
        d = dict(self.__dict__)
        d["n_ctx"] = n_ctx
        return CtxKvWorkload(**d)


# The pages give no draft geometry: hidden follows the target, eight KV heads
# of 128, four draft layers (117 MB of K/V weights: under L2, so the bench
# writes a buffer larger than L2 between timed steps).
CTXKV_WORKLOADS = {
    "draft_ctx_kv": CtxKvWorkload("draft_ctx_kv", n_ctx=8, hidden=7168, n_layers=4, n_kv_heads=8,
                                  head_dim=128),
    "draft_ctx_kv_small": CtxKvWorkload("draft_ctx_kv_small", n_ctx=8, hidden=256, n_layers=2,
                                        n_kv_heads=2, head_dim=64, max_position=4096, n_slots=64),
}


def ctxkv_inputs(w: CtxKvWorkload, variant: int = 0):
    """(context bf16 bits [n, H] ~ N(0, 1), positions int64 [n], slots int64 [n]).
    The positions are consecutive from a seeded start; the slots are n distinct
    seeded slots of the n_slots."""
    ctx = normal_bf16((w.n_ctx, w.hidden), w.seed, tag(KIND_CTX, 0, variant), *w.ctx_dist)
    words = philox_words(max(w.n_slots, 1), w.seed, tag(KIND_CTX_PLACE, 0, variant))
    start = int(words[0, 1]) % max(w.max_position - w.n_ctx, 1)
    positions = np.arange(start, start + w.n_ctx, dtype=np.int64)
    slots = np.argsort(words[:, 0], kind="stable")[: w.n_ctx].astype(np.int64)
    return ctx, positions, slots


def ctxkv_norm_weights(w: CtxKvWorkload):
    """(w_hidden fp32 [H], w_pre fp32 [L, H]), each 1 + 0.1 N(0, 1)."""
    wh = normal_f32((w.hidden,), w.seed, tag(KIND_W_HIDDEN), *w.norm_dist)
    wp = np.stack([normal_f32((w.hidden,), w.seed, tag(KIND_W_PRE_QKV, l), *w.norm_dist)
                   for l in range(w.n_layers)])
    return wh, wp


def ctxkv_weights(w: CtxKvWorkload) -> np.ndarray:
    """bf16 bits [L, 2*KVH*D, H]: each layer's K rows, then V rows, N(0, 0.02)."""
    rows = 2 * w.n_kv_heads * w.head_dim
    return np.stack([normal_bf16((rows, w.hidden), w.seed, tag(KIND_W_KV, l), *w.weight_dist)
                     for l in range(w.n_layers)])


def dev_ctxkv_weights(out, w: CtxKvWorkload, stream=None):
    """Device twin of ctxkv_weights, into the bf16 CUDA tensor [L, 2*KVH*D, H]."""
    for l in range(w.n_layers):
        dev_normal_bf16(out[l], w.seed, tag(KIND_W_KV, l), *w.weight_dist, stream=stream)
    return out
