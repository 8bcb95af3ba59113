"""The quantizer entry point that allocates no device memory.

It serves callers that cannot call cudaMalloc: code that runs inside another
runtime which hands it only its input and output buffers, or a loop that
cannot afford an allocation's device synchronization.  Its scratch is a fixed
array inside the library that every call shares.  These checks go through the
C ABI and compare it, bit for bit like the other quantizer tests, with
moe_nvfp4_quantize on two calls in a row.  The second tensor has a much smaller
max |v| than the first, so anything the first call left in the shared scratch
and the second failed to clear would change its tensor scale.

The file is named to be collected last: a run that stops at the first failure
has then run every other test already.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _with_existing(moe, v):
    rows, cols = v.shape
    codes = torch.empty(rows, cols // 2, dtype=torch.uint8, device=v.device)
    sf = torch.empty(rows, cols // 16, dtype=torch.uint8, device=v.device)
    sg = torch.empty(1, dtype=torch.float32, device=v.device)
    amax = torch.empty(1, dtype=torch.float32, device=v.device)
    moe.moe_nvfp4_quantize(v, codes, sf, sg, amax)
    return codes, sf, sg


def _with_noalloc(moe, v):
    rows, cols = v.shape
    codes = torch.full((rows, cols // 2), 0xAB, dtype=torch.uint8, device=v.device)
    sf = torch.full((rows, cols // 16), 0xCD, dtype=torch.uint8, device=v.device)
    sg = torch.full((1,), -1.0, dtype=torch.float32, device=v.device)
    moe.moe_nvfp4_quantize_noalloc(v, codes, sf, sg)
    return codes, sf, sg


def test_noalloc_quantizer_matches_existing_on_two_calls_in_a_row():
    import speculative_decode_routed_gb300 as moe
    rs = np.random.RandomState(7)
    # 1000 x 7168: 110 chunks of 65536 elements, the last one ragged
    v1 = torch.from_numpy((rs.standard_normal((1000, 7168)) * 5.0).astype(np.float32)).cuda()
    # 37 x 2048: two chunks; max |v| about 5000x below the first tensor's
    v2 = torch.from_numpy((rs.standard_normal((37, 2048)) * 1e-3).astype(np.float32)).cuda()
    v2[3, :16] = 0.0                                     # a zero block
    for v in (v1, v2):
        got = _with_noalloc(moe, v)
        ref = _with_existing(moe, v)
        torch.cuda.synchronize()
        for g, r, what in zip(got, ref, ("codes", "block scales", "tensor scale")):
            assert torch.equal(g, r), f"{what} differ from moe_nvfp4_quantize for shape {tuple(v.shape)}"


def test_noalloc_quantizer_rejects_tensors_beyond_its_scratch():
    import speculative_decode_routed_gb300 as moe
    v = torch.zeros(1, 16, dtype=torch.float32, device="cuda")
    codes = torch.zeros(1, 8, dtype=torch.uint8, device="cuda")
    sf = torch.zeros(1, 1, dtype=torch.uint8, device="cuda")
    sg = torch.zeros(1, dtype=torch.float32, device="cuda")
    lib = moe.lib()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    # 2^30 + 16 elements: one past the limit; rejected before any launch
    rc = lib.moe_nvfp4_quantize_noalloc(p(v), (1 << 26) + 1, 16, p(codes), p(sf), p(sg), None)
    assert rc == moe.MOE_EUNSUPPORTED
    assert b"2^30" in lib.moe_decode_error_message()
    # an empty tensor is accepted: it writes a zero tensor scale
    sg.fill_(-1.0)
    torch.cuda.synchronize()
    rc = lib.moe_nvfp4_quantize_noalloc(p(v), 0, 16, p(codes), p(sf), p(sg), None)
    assert rc == moe.MOE_OK
    torch.cuda.synchronize()
    assert float(sg.item()) == 0.0


def test_noalloc_quantizer_many_chunks_ragged_tail():
    """More chunks than the last CTA's threads (300 full chunks of 65536 and a
    ragged 16-element tail): the final reduction's strided loop takes several
    partials per thread.  Bit for bit with moe_nvfp4_quantize, twice in a row."""
    import speculative_decode_routed_gb300 as moe
    n = 300 * 65536 + 16
    g = torch.Generator(device="cuda").manual_seed(11)
    v = torch.randn(n // 16, 16, generator=g, device="cuda") * 3.0
    v[-1, 5] = 77.0          # the tensor's max |v| sits in the ragged last chunk
    for _ in range(2):
        got = _with_noalloc(moe, v)
        ref = _with_existing(moe, v)
        torch.cuda.synchronize()
        for a, b, what in zip(got, ref, ("codes", "block scales", "tensor scale")):
            assert torch.equal(a, b), f"{what} differ from moe_nvfp4_quantize"
    assert float(got[2].item()) == np.float32(77.0) / np.float32(2688.0)


def test_noalloc_quantizer_rejects_misaligned_pointers():
    """v off its 16-byte alignment, codes off 8 and sg off 4 are each rejected
    before any launch with MOE_EINVAL."""
    import speculative_decode_routed_gb300 as moe
    v = torch.zeros(2, 64, dtype=torch.float32, device="cuda")
    codes = torch.zeros(2 * 32 + 8, dtype=torch.uint8, device="cuda")
    sf = torch.zeros(2 * 4, dtype=torch.uint8, device="cuda")
    sg = torch.zeros(4, dtype=torch.float32, device="cuda")
    lib = moe.lib()
    vp = ctypes.c_void_p
    base = (vp(v.data_ptr()), vp(codes.data_ptr()), vp(sf.data_ptr()), vp(sg.data_ptr()))
    for i, shift in ((0, 4), (1, 4), (3, 2)):
        args = list(base)
        args[i] = vp(args[i].value + shift)
        rc = lib.moe_nvfp4_quantize_noalloc(args[0], 1, 16, args[1], args[2], args[3], None)
        assert rc == moe.MOE_EINVAL, f"pointer {i} off by {shift} bytes: rc {rc}"
        assert b"aligned" in lib.moe_decode_error_message()
    rc = lib.moe_nvfp4_quantize_noalloc(*base[:1], 1, 16, *base[1:], None)
    assert rc == moe.MOE_OK
    torch.cuda.synchronize()
