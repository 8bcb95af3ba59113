"""GPU parity of the draft context-KV projection (moe_ctxkv_*), through the C
ABI, against the CPU oracle.

Staged checks feed each oracle piece the GPU's own output of the stage before
(u into each layer's projection, kv into the key norm and rotation, the keys
and values into the cache scatter): projections and keys bit for bit except
at bf16 rounding midpoints, values and caches bit for bit.  End to end the
oracle runs on its own; a rounding taken the other way upstream may move a
projection output by one bf16 step (up to 2^-7 of it), which the key norm
carries into the normalised key; the two casts before the rotation may then
round apart by another step, the rotation keeps the pair's difference vector's
length, and the two final casts may add a third: a key may differ by up to
3 * 2^-7 of its pair's norm, and a value by 2^-7 of itself.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import bf16_near_tie, bits_match, dev_array

torch = pytest.importorskip("torch")

# end-to-end key tolerance, relative to the pair's norm (three bf16 steps)
KEY_TOL = 3 * 2.0 ** -7
pytestmark = pytest.mark.gpu

SMALL = synth.CTXKV_WORKLOADS["draft_ctx_kv_small"]
FULL = synth.CTXKV_WORKLOADS["draft_ctx_kv"]
GEMM_SLACK = 1e-3          # projections: share of outputs one step off away from midpoints


def _shape(w, **kw):
    d = dict(w.__dict__)
    d.update(kw)
    return synth.CtxKvWorkload(**d)


def _bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


_bits_match = bits_match     # equal bf16 bits away from rounding midpoints


class _Case:
    def __init__(self, w, max_ctx):
        import speculative_decode_routed_gb300 as moe
        self.w = w
        L, H, KD = w.n_layers, w.hidden, w.n_kv_heads * w.head_dim
        self.wkv = torch.empty(L, 2 * KD, H, dtype=torch.bfloat16, device="cuda")
        synth.dev_ctxkv_weights(self.wkv, w)
        self.wh, self.wp = synth.ctxkv_norm_weights(w)
        self.wkv_h = synth.ctxkv_weights(w)
        self.wh_t, self.wp_t = torch.from_numpy(self.wh).cuda(), torch.from_numpy(self.wp).cuda()
        self.op = moe.ContextKV(H, L, w.n_kv_heads, w.head_dim, max_ctx, self.wh_t, self.wp_t, self.wkv,
                                eps=w.eps, qk_eps=w.qk_eps, rope_theta=w.rope_theta,
                                max_position=w.max_position)

    def caches(self, seed):
        w = self.w
        rs = np.random.RandomState(seed)
        shape = (w.n_layers, w.n_slots, w.n_kv_heads, w.head_dim)
        return rs.randint(0, 1 << 16, shape).astype(np.uint16), rs.randint(0, 1 << 16, shape).astype(np.uint16)

    def run(self, n, variant=0, slots=None, positions=None):
        """-> (inputs, GPU outputs); slots None: the workload's shared map."""
        w = self.w.with_ctx(n)
        ctx, pos, shared = synth.ctxkv_inputs(w, variant)
        if positions is not None:
            pos = positions
        slots = shared if slots is None else slots
        kc0, vc0 = self.caches(variant)
        kc, vc = _bf16_dev(kc0), _bf16_dev(vc0)
        self.op.project(n, _bf16_dev(ctx), torch.from_numpy(pos).cuda(), torch.from_numpy(slots).cuda(), kc, vc)
        torch.cuda.synchronize()
        self.op.check()
        v = self.op.debug()
        L, H, KVH, D = w.n_layers, w.hidden, w.n_kv_heads, w.head_dim
        got = dict(fc=dev_array(v.fc, (n, H), np.uint16), u=dev_array(v.u, (L, n, H), np.uint16),
                   kv=dev_array(v.kv, (L, n, 2 * KVH * D), np.uint16),
                   k=dev_array(v.k, (L, n, KVH, D), np.uint16), v=dev_array(v.v, (L, n, KVH, D), np.uint16),
                   k_cache=kc.view(torch.int16).cpu().numpy().view(np.uint16),
                   v_cache=vc.view(torch.int16).cpu().numpy().view(np.uint16))
        return (ctx, pos, slots, kc0, vc0), got

    def close(self):
        self.op.close()


def _check(case, n, variant=0, slots=None, positions=None):
    w = case.w
    (ctx, pos, slots, kc0, vc0), got = case.run(n, variant, slots, positions)
    KVH, D = w.n_kv_heads, w.head_dim
    ref = oracle.context_kv(ctx, pos, case.wh, case.wp, case.wkv_h, KVH, D, w.eps, w.qk_eps, w.rope_theta)
    _bits_match(got["fc"], ref["fc"], ref["fc_exact"], "fc")
    u, u_ex = oracle.layer_norms(got["fc"], case.wp, w.eps)
    _bits_match(got["u"], u, u_ex, "u")
    for l in range(w.n_layers):
        kv, kv_ex = oracle.bf16_linear(got["u"][l], case.wkv_h[l])
        _bits_match(got["kv"][l], kv, kv_ex, f"kv of layer {l}", slack=GEMM_SLACK * kv.size)
    k, v, k_ex, kn_ex = oracle.k_norm_rope(got["kv"], pos, KVH, D, w.qk_eps, w.rope_theta, with_norm=True)
    # a normalised key at a midpoint may be cast the other way before the
    # rotation, which then moves both outputs of its pair
    tie = bf16_near_tie(kn_ex)
    h = D // 2
    pair_tie = np.concatenate([tie[..., :h] | tie[..., h:]] * 2, axis=-1)
    _bits_match(got["k"], k, k_ex, "keys", exclude=pair_tie)
    assert np.array_equal(got["v"], v), "values"
    kc, vc = oracle.kv_cache_write(got["k"], got["v"], slots, w.n_slots, kc0, vc0)
    assert np.array_equal(got["k_cache"], kc), "key cache"
    assert np.array_equal(got["v_cache"], vc), "value cache"
    # end to end
    dk = np.abs(oracle.bf16_to_f64(got["k"]) - oracle.bf16_to_f64(ref["k"]))
    rk = oracle.bf16_to_f64(ref["k"])
    pair = np.sqrt(rk[..., :h] ** 2 + rk[..., h:] ** 2)
    pair = np.concatenate([pair, pair], axis=-1)
    assert np.all(dk <= KEY_TOL * pair), f"keys: max excess {np.max(dk - KEY_TOL * pair):.3e}"
    rv = oracle.bf16_to_f64(ref["v"])
    dv = np.abs(oracle.bf16_to_f64(got["v"]) - rv)
    rms_v = float(np.sqrt(np.mean(rv ** 2)))
    assert np.all(dv <= 2.0 ** -7 * np.abs(rv) + 1e-3 * rms_v), "values end to end"


def test_small_shared_slots():
    case = _Case(SMALL, max_ctx=64)
    try:
        _check(case, 8)
        _check(case, 1, variant=1)
        assert case.op.kernel_count(37) == 3   # norms, tensor-core projection, keys
    finally:
        case.close()


def test_ragged_rows_with_per_layer_slots_and_skipped_rows():
    case = _Case(SMALL, max_ctx=64)
    try:
        n = 37
        rs = np.random.RandomState(11)
        slots = np.stack([rs.permutation(SMALL.n_slots)[:n] for _ in range(SMALL.n_layers)]).astype(np.int64)
        slots[0, ::5] = -1
        slots[1, 3] = -7
        _check(case, n, variant=2, slots=slots)
    finally:
        case.close()


@pytest.mark.parametrize("kw,n", [
    (dict(hidden=1032, n_layers=3, n_kv_heads=3, head_dim=128, rope_theta=500000.0,
          max_position=1 << 17, n_slots=40), 5),
    (dict(hidden=512, n_layers=1, n_kv_heads=1, head_dim=256, rope_theta=0.0, n_slots=16), 2),
    (dict(hidden=384, n_layers=2, n_kv_heads=4, head_dim=64, n_slots=300), 256),
    # one 64-wide head over hidden 4096: the streamed projection in 32 K-splits,
    # summed by the key kernel in four groups of eight
    (dict(hidden=4096, n_layers=1, n_kv_heads=1, head_dim=64, n_slots=64), 8),
    (dict(hidden=4096, n_layers=1, n_kv_heads=1, head_dim=64, n_slots=64), 3),
])
def test_other_geometries(kw, n):
    w = _shape(SMALL, **kw)
    case = _Case(w, max_ctx=n)
    try:
        pos = None
        if w.rope_theta > 0:             # the last rows of the rotary table
            pos = np.arange(w.max_position - n, w.max_position, dtype=np.int64)
        _check(case, n, positions=pos)
    finally:
        case.close()


@pytest.mark.parametrize("n", [8, 128])
def test_full_width(n):
    """Hidden 7168, four layers of eight 128-wide KV heads: the configuration the
    bench times (8 rows) and a longer context (128 rows)."""
    case = _Case(FULL, max_ctx=n)
    try:
        _check(case, n)
    finally:
        case.close()


def test_out_of_range_position_and_slot_latch_errors():
    import speculative_decode_routed_gb300 as moe
    case = _Case(SMALL, max_ctx=8)
    try:
        ctx, pos, slots = synth.ctxkv_inputs(SMALL, 0)
        kc0, vc0 = case.caches(0)
        kc, vc = _bf16_dev(kc0), _bf16_dev(vc0)
        bad = pos.copy()
        bad[3] = SMALL.max_position               # one past the table
        case.op.project(8, _bf16_dev(ctx), torch.from_numpy(bad).cuda(), torch.from_numpy(slots).cuda(), kc, vc)
        with pytest.raises(moe.MoeError, match="position"):
            case.op.check()
        case.op.check()                           # cleared
        bad_slots = slots.copy()
        bad_slots[5] = SMALL.n_slots
        case.op.project(8, _bf16_dev(ctx), torch.from_numpy(pos).cuda(), torch.from_numpy(bad_slots).cuda(),
                        kc, vc)
        with pytest.raises(moe.MoeError, match="slot"):
            case.op.check()
        with pytest.raises(moe.MoeError):
            case.op.project(9, _bf16_dev(ctx), torch.from_numpy(pos).cuda())
        # three kernels, all the library's own: norms, the streamed (up to 8
        # rows) or tensor-core projection, and the key kernel
        assert case.op.kernel_count(8) == 3
    finally:
        case.close()


def test_graph_replays_bitwise():
    case = _Case(SMALL, max_ctx=8)
    try:
        ctx, pos, slots = synth.ctxkv_inputs(SMALL, 3)
        c_t, p_t, s_t = _bf16_dev(ctx), torch.from_numpy(pos).cuda(), torch.from_numpy(slots).cuda()
        kc0, vc0 = case.caches(3)
        kc_e, vc_e = _bf16_dev(kc0), _bf16_dev(vc0)
        case.op.project(8, c_t, p_t, s_t, kc_e, vc_e)
        kc_g, vc_g = _bf16_dev(kc0), _bf16_dev(vc0)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            case.op.project(8, c_t, p_t, s_t, kc_g.clone(), vc_g.clone())
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            case.op.project(8, c_t, p_t, s_t, kc_g, vc_g)
        for _ in range(2):
            kc_g.copy_(_bf16_dev(kc0))
            vc_g.copy_(_bf16_dev(vc0))
            g.replay()
            torch.cuda.synchronize()
            # the caches start as random bits, NaNs included: compare the bits
            assert torch.equal(kc_g.view(torch.int16), kc_e.view(torch.int16))
            assert torch.equal(vc_g.view(torch.int16), vc_e.view(torch.int16))
        case.op.check()
    finally:
        case.close()


def test_host_buffers_match_the_device_call():
    """moe_ctxkv_project_host: page-locked buffers (read and written by the
    kernels) and pageable ones (copied) give the device call's keys, values and
    caches bit for bit."""
    case = _Case(SMALL, max_ctx=8)
    try:
        w = SMALL
        L, KVH, D = w.n_layers, w.n_kv_heads, w.head_dim
        ctx, pos, slots = synth.ctxkv_inputs(w, 5)
        kc0, vc0 = case.caches(5)
        kc, vc = _bf16_dev(kc0), _bf16_dev(vc0)
        k_dev = torch.empty(L, 8, KVH, D, dtype=torch.bfloat16, device="cuda")
        v_dev = torch.empty_like(k_dev)
        case.op.project(8, _bf16_dev(ctx), torch.from_numpy(pos).cuda(), torch.from_numpy(slots).cuda(), kc, vc,
                        k_out=k_dev, v_out=v_dev)
        torch.cuda.synchronize()
        want = [t.view(torch.int16).cpu().numpy() for t in (k_dev, v_dev, kc, vc)]
        for pinned in (True, False):
            c_h = torch.from_numpy(ctx.view(np.int16).copy()).view(torch.bfloat16)
            p_h, s_h = torch.from_numpy(pos.copy()), torch.from_numpy(slots.copy())
            k_h = torch.empty(L, 8, KVH, D, dtype=torch.bfloat16)
            v_h = torch.empty_like(k_h)
            if pinned:
                c_h, p_h, s_h, k_h, v_h = (t.pin_memory() for t in (c_h, p_h, s_h, k_h, v_h))
            kc2, vc2 = _bf16_dev(kc0), _bf16_dev(vc0)
            case.op.project_host(8, c_h, p_h, k_h, v_h, slots=s_h, k_cache=kc2, v_cache=vc2)
            got = [k_h.view(torch.int16).numpy(), v_h.view(torch.int16).numpy(),
                   kc2.view(torch.int16).cpu().numpy(), vc2.view(torch.int16).cpu().numpy()]
            for g_, w_, what in zip(got, want, ("keys", "values", "key cache", "value cache")):
                assert np.array_equal(g_, w_), f"{what} differ ({'page-locked' if pinned else 'pageable'})"
        case.op.check()
    finally:
        case.close()
