"""GPU parity of the dense draft layer (moe_dense_*), through the C ABI, against
the CPU oracle.

Staged checks feed each oracle piece the GPU's own output of the stage before
(x into the gate/up projection, gu into SiLU * mul, a into the down
projection, f into the output norm), so every bf16 rounding is compared bit
for bit except where the exact value sits at a bf16 rounding midpoint (fp32
accumulation may round those either way).  The end-to-end check runs the
oracle independently: each stream element within 2e-3 * rms(stream) plus one
bf16 step of the output branch there (the layer's f is bf16, so one rounding
taken the other way upstream may move an f element by a step).
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import bits_match, dev_array

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

STREAM_TOL = 2e-3          # end-to-end: max|err| <= STREAM_TOL * rms(stream)
STAGE_TOL = 1e-4           # staged output norm: max|err| <= STAGE_TOL * rms(stream)
BF16_STEP = 2.0 ** -7      # largest relative step between neighbouring bf16 values
GEMM_SLACK = 1e-3          # projections: share of outputs one step off away from midpoints

SMALL = synth.DENSE_WORKLOADS["draft_dense_small"]
FULL = synth.DENSE_WORKLOADS["draft_dense"]


def _rms(a):
    return float(np.sqrt(np.mean(np.asarray(a, np.float64) ** 2)))


def _shape(w, hidden, inter):
    d = dict(w.__dict__)
    d.update(hidden=hidden, inter=inter)
    return synth.Workload(**d)


def _bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


class _Case:
    """One dense layer on the device and the same weights on the host."""

    def __init__(self, w, max_rows, layer=0):
        import speculative_decode_routed_gb300 as moe
        H, I = w.hidden, w.inter
        self.w = w
        self.w13 = torch.empty(2 * I, H, dtype=torch.bfloat16, device="cuda")
        self.w2 = torch.empty(H, I, dtype=torch.bfloat16, device="cuda")
        synth.dev_dense_weights(self.w13, self.w2, w, layer)
        self.norms_h = synth.dense_norm_weights(w, layer)
        self.norms = [torch.from_numpy(n).cuda() for n in self.norms_h]
        self.w13_h, self.w2_h = synth.dense_weights(w, layer)
        self.layer = moe.DenseLayer(H, I, max_rows, self.norms[0], self.norms[1], self.w13,
                                    self.w2, self.norms[2], eps=w.eps)

    def run(self, rows, variant=0):
        """-> (inputs, GPU outputs) of one layer call on `rows` rows."""
        H, I = self.w.hidden, self.w.inter
        stream, attn = synth.step_inputs(self.w.with_rows(rows), variant)
        s_t = torch.from_numpy(stream).cuda()
        a_t = _bf16_dev(attn)
        self.layer.layer(rows, a_t, s_t)
        torch.cuda.synchronize()
        v = self.layer.debug()
        got = dict(stream=s_t.cpu().numpy(), x=dev_array(v.x, (rows, H), np.uint16),
                   gu=dev_array(v.gu, (rows, 2 * I), np.uint16),
                   a=dev_array(v.a, (rows, I), np.uint16), f=dev_array(v.f, (rows, H), np.uint16))
        return (stream, attn), got

    def close(self):
        self.layer.close()


_bits_match = bits_match     # equal bf16 bits away from rounding midpoints


def _check(case, rows, variant=0):
    w = case.w
    (stream, attn), got = case.run(rows, variant)
    na, npre, npost = case.norms_h
    ref = oracle.dense_layer(attn, stream, na, npre, case.w13_h, case.w2_h, npost, w.eps)
    # x: the stream after the attention branch is fp32 on both sides but may
    # differ in its last bit; where that bit moves bf16(s1) across a midpoint
    # one element of x moves by one step
    _bits_match(got["x"], ref["x"], ref["x_exact"], "x", slack=got["x"].size // 10000)
    # the projections: the tensor-core kernel's fp32 summation (the MMA's
    # internal accumulation order is unspecified) strays past the 1e-5 midpoint band now and then
    # at K in the thousands; those results are one bf16 step away, and rare
    gu, gu_ex = oracle.bf16_linear(got["x"], case.w13_h)
    _bits_match(got["gu"], gu, gu_ex, "gate/up", slack=GEMM_SLACK * gu.size)
    a, a_ex = oracle.silu_mul(got["gu"])
    _bits_match(got["a"], a, a_ex, "silu * up")
    f, f_ex = oracle.bf16_linear(got["a"], case.w2_h)
    _bits_match(got["f"], f, f_ex, "down", slack=GEMM_SLACK * f.size)
    s1, _, _ = oracle.boundary(oracle.bf16_to_f64(attn), stream, na, npre, w.eps)
    s2, _, _ = oracle.boundary(oracle.bf16_to_f64(got["f"]), s1, npost, npost, w.eps)
    rms = _rms(ref["stream"])
    err_stage = float(np.max(np.abs(got["stream"].astype(np.float64) - s2)))
    assert err_stage <= STAGE_TOL * rms, f"output norm: {err_stage:.3e} > {STAGE_TOL * rms:.3e}"
    # end to end: f is bf16, so a rounding that fp32 accumulation takes the
    # other way anywhere upstream can move an f element by one bf16 step (at
    # most 2^-7 of it), which the output norm carries into the stream
    err = np.abs(got["stream"].astype(np.float64) - ref["stream"])
    branch = np.abs(ref["stream"].astype(np.float64) - s1)
    bound = BF16_STEP * branch + STREAM_TOL * rms
    worst = int(np.argmax(err - bound))
    assert np.all(err <= bound), \
        f"stream: err {err.flat[worst]:.3e} > {bound.flat[worst]:.3e} at {np.unravel_index(worst, err.shape)}"
    return float(err.max()) / rms


# (256, 384) and (256, 4096) take the streamed projections (the latter's down
# projection in 16 K-splits, summed by the boundary in two groups of eight);
# the others the tensor-core projection kernel
@pytest.mark.parametrize("hidden,inter,rows", [(256, 384, 8), (256, 384, 1), (256, 4096, 8),
                                               (256, 4096, 5), (1152, 520, 3),
                                               (1152, 520, 33), (384, 136, 128),
                                               (4224, 136, 2)])
def test_dense_layer_matches_oracle(hidden, inter, rows):
    case = _Case(_shape(SMALL, hidden, inter), max_rows=max(rows, 8))
    try:
        _check(case, rows)
        _check(case, rows, variant=1)
    finally:
        case.close()


def test_dense_layer_full_width():
    """The 7168 x 28672 layer at 8 rows, the configuration the bench times."""
    case = _Case(FULL, max_rows=8)
    try:
        _check(case, 8)
    finally:
        case.close()


@pytest.mark.parametrize("hidden,inter", [(1152, 520), (256, 384)])
def test_dense_layer_graph_replays_bitwise(hidden, inter):
    """A captured layer replays to the eager result bit for bit (the library
    tensor-core path and the streamed path, both with programmatic dependent
    launches)."""
    case = _Case(_shape(SMALL, hidden, inter), max_rows=8)
    try:
        stream, attn = synth.step_inputs(case.w.with_rows(8), 2)
        a_t = _bf16_dev(attn)
        s_eager = torch.from_numpy(stream).cuda()
        case.layer.layer(8, a_t, s_eager)
        s_graph = torch.from_numpy(stream).cuda()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):          # a first call outside capture
            case.layer.layer(8, a_t, s_graph.clone())
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            case.layer.layer(8, a_t, s_graph)
        for _ in range(2):
            s_graph.copy_(torch.from_numpy(stream))
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(s_graph, s_eager)
    finally:
        case.close()


def test_dense_layer_profile_and_row_limits():
    import speculative_decode_routed_gb300 as moe
    case = _Case(SMALL, max_rows=8)
    try:
        stream, attn = synth.step_inputs(SMALL, 0)
        s_t, a_t = torch.from_numpy(stream).cuda(), _bf16_dev(attn)
        ms = case.layer.layer_profile(8, a_t, s_t)
        assert len(ms) == 5 and all(t > 0.0 for t in ms)
        # four kernels, all the library's own, streamed (up to 8 rows) or not
        assert case.layer.kernel_count(8) == 4
        for rows in (0, 9):
            with pytest.raises(moe.MoeError):
                case.layer.layer(rows, a_t, s_t)
    finally:
        case.close()


@pytest.mark.parametrize("hidden,inter", [(256, 384), (1152, 520)])
def test_dense_layer_host_buffers_match_the_device_call(hidden, inter):
    """moe_dense_layer_host: page-locked buffers (read and written by the
    kernels, twice: captured, then replayed) and pageable ones (copied) give
    the device call's stream bit for bit."""
    case = _Case(_shape(SMALL, hidden, inter), max_rows=8)
    try:
        stream, attn = synth.step_inputs(case.w.with_rows(8), 4)
        s_dev = torch.from_numpy(stream).cuda()
        case.layer.layer(8, _bf16_dev(attn), s_dev)
        want = s_dev.cpu().numpy()
        a_pin = torch.from_numpy(attn.view(np.int16)).view(torch.bfloat16).pin_memory()
        s_pin = torch.from_numpy(stream).pin_memory()
        for _ in range(2):
            s_pin.copy_(torch.from_numpy(stream))
            case.layer.layer_host(8, a_pin, s_pin)
            assert np.array_equal(s_pin.numpy(), want)
        s_page = torch.from_numpy(stream.copy())
        case.layer.layer_host(8, torch.from_numpy(attn.view(np.int16).copy()).view(torch.bfloat16), s_page)
        assert np.array_equal(s_page.numpy(), want)
    finally:
        case.close()
