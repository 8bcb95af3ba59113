"""The C ABI library without a GPU: it loads, exports every symbol the public
header declares, and rejects invalid arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

import speculative_decode_routed_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "moe_decode.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_header_symbols_are_exported():
    lib = moe.lib()
    names = _declared()
    assert "moe_decode_create" in names and "moe_nvfp4_quantize" in names
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(moe.EXPORTS) == names


def _dims(**kw):
    d = dict(hidden=256, n_experts=8, top_k=2, inter=128, max_rows=8, n_layers=1, eps=1e-6,
             code_layout=0)
    d.update(kw)
    return moe.Dims(**d)


def _fake_layer(align=256):
    # non-null, aligned fake addresses: validation runs before any CUDA call
    base = 1 << 20
    return moe.LayerWeights(*(base + i * align for i in range(3)), None,
                           *(base + (4 + i) * align for i in range(5)))


def _create(dims, layers):
    h = ctypes.c_void_p()
    arr = (moe.LayerWeights * len(layers))(*layers)
    rc = moe.lib().moe_decode_create(ctypes.byref(dims), arr, None, None, ctypes.byref(h))
    return rc, moe.lib().moe_decode_error_message().decode()


@pytest.mark.parametrize("kw", [dict(hidden=200), dict(hidden=16384), dict(inter=100),
                                dict(n_experts=0), dict(n_experts=2000), dict(top_k=0),
                                dict(top_k=9), dict(top_k=17, n_experts=32), dict(max_rows=0),
                                dict(max_rows=129), dict(n_layers=0)])
def test_unsupported_shapes(kw):
    rc, msg = _create(_dims(**kw), [_fake_layer()])
    assert rc == moe.MOE_EUNSUPPORTED, (kw, rc, msg)
    assert msg


def test_null_and_misaligned_pointers():
    lay = _fake_layer()
    lay.w13 = None
    rc, msg = _create(_dims(), [lay])
    assert rc == moe.MOE_EINVAL and "NULL" in msg
    lay = _fake_layer()
    lay.w2 = lay.w2 + 4
    rc, msg = _create(_dims(), [lay])
    assert rc == moe.MOE_EINVAL and "aligned" in msg
    rc = moe.lib().moe_decode_create(None, None, None, None, None)
    assert rc == moe.MOE_EINVAL


def test_code_layout_is_validated():
    rc, msg = _create(_dims(code_layout=3), [_fake_layer()])
    assert rc == moe.MOE_EINVAL and "code_layout" in msg
    rc, msg = _create(_dims(code_layout=-1), [_fake_layer()])
    assert rc == moe.MOE_EINVAL and "code_layout" in msg


def test_tiled_code_sizes_and_argument_checks():
    """moe_tiled_code_bytes follows the header's layout (whole 16 KB tiles, a
    partial last K-block padded) and rejects shapes it cannot tile; the tiling
    call rejects bad pointers before any launch."""
    L = moe.lib()
    assert L.moe_tiled_code_bytes(256 * 4096, 3584) == 256 * 4096 * 3584      # H 7168: whole tiles
    assert L.moe_tiled_code_bytes(128, 192) == 2 * 16384                      # H 384: one and a half
    assert L.moe_tiled_code_bytes(384, 16) == 3 * 16384
    for rows, rb in ((100, 64), (0, 64), (128, 8), (128, 0), (-128, 64), (1 << 40, 1 << 20)):
        assert L.moe_tiled_code_bytes(rows, rb) == moe.MOE_EINVAL, (rows, rb)
    base = 1 << 20
    assert L.moe_tile_codes(None, 128, 64, base, None) == moe.MOE_EINVAL
    assert L.moe_tile_codes(base, 128, 64, None, None) == moe.MOE_EINVAL
    assert L.moe_tile_codes(base + 8, 128, 64, base << 4, None) == moe.MOE_EINVAL
    assert L.moe_tile_codes(base, 128, 64, base + 4096, None) == moe.MOE_EINVAL   # overlapping
    assert b"overlap" in L.moe_decode_error_message()
    assert L.moe_tile_codes(base, 100, 64, base << 4, None) == moe.MOE_EINVAL
    assert L.moe_decode_weight_copy_bytes(None) == 0


def test_calls_on_a_null_handle_fail_cleanly():
    L = moe.lib()
    assert L.moe_decode_layer(None, 0, 1, None, None, None) == moe.MOE_EINVAL
    assert L.moe_decode_step(None, 1, None, None, None, None) == moe.MOE_EINVAL
    assert L.moe_decode_final(None, 1, None, None, None, None) == moe.MOE_EINVAL
    assert L.moe_decode_front(None, 1, None, None, None, None, None, None) == moe.MOE_EINVAL
    assert L.moe_decode_last_error(None) == moe.MOE_EINVAL
    assert L.moe_decode_workspace_bytes(None) == 0
    L.moe_decode_destroy(None)
    assert L.moe_decode_strerror(moe.MOE_EDEVICE).decode() == "device-side check failed"
    assert L.moe_nvfp4_quantize(None, 1, 16, None, None, None, None, None) == moe.MOE_EINVAL
    assert L.moe_nvfp4_quantize(1 << 20, 1, 17, 1 << 20, 1 << 20, 1 << 20, 1 << 20, None) == moe.MOE_EINVAL


def _dense_create(hidden=256, inter=128, max_rows=8, eps=1e-6, null=None, shift=None):
    dims = moe.DenseDims(hidden, inter, max_rows, eps)
    ptrs = [(1 << 20) + i * 256 for i in range(5)]
    if null is not None:
        ptrs[null] = None
    if shift is not None:
        ptrs[shift] += 4
    w = moe.DenseWeights(*ptrs)
    h = ctypes.c_void_p()
    rc = moe.lib().moe_dense_create(ctypes.byref(dims), ctypes.byref(w), ctypes.byref(h))
    return rc, moe.lib().moe_decode_error_message().decode()


@pytest.mark.parametrize("kw", [dict(hidden=200), dict(hidden=16512), dict(hidden=0),
                                dict(inter=100), dict(inter=0), dict(max_rows=0),
                                dict(max_rows=129)])
def test_dense_unsupported_shapes(kw):
    rc, msg = _dense_create(**kw)
    assert rc == moe.MOE_EUNSUPPORTED, (kw, rc, msg)
    assert msg


def test_dense_invalid_arguments():
    for i in range(5):
        rc, msg = _dense_create(null=i)
        assert rc == moe.MOE_EINVAL and "NULL" in msg
        rc, msg = _dense_create(shift=i)
        assert rc == moe.MOE_EINVAL and "aligned" in msg
    rc, msg = _dense_create(eps=0.0)
    assert rc == moe.MOE_EINVAL and "eps" in msg
    L = moe.lib()
    assert L.moe_dense_create(None, None, None) == moe.MOE_EINVAL
    assert L.moe_dense_layer(None, 1, None, None, None) == moe.MOE_EINVAL
    ms = (ctypes.c_float * 5)()
    assert L.moe_dense_layer_profile(None, 1, None, None, None, ms) == moe.MOE_EINVAL
    assert L.moe_dense_debug(None, None) == moe.MOE_EINVAL
    assert L.moe_dense_kernel_count(None, 1) == moe.MOE_EINVAL
    assert L.moe_dense_layer_host(None, 1, None, None, None) == moe.MOE_EINVAL
    L.moe_dense_destroy(None)


def _ctxkv_create(null=None, shift=None, **kw):
    d = dict(hidden=256, n_layers=2, n_kv_heads=2, head_dim=64, max_ctx=8, max_position=64,
             eps=1e-6, qk_eps=1e-6, rope_theta=10000.0)
    d.update(kw)
    dims = moe.CtxKvDims(**d)
    ptrs = [(1 << 20) + i * 256 for i in range(3)]
    if null is not None:
        ptrs[null] = None
    if shift is not None:
        ptrs[shift] += 8
    h = ctypes.c_void_p()
    rc = moe.lib().moe_ctxkv_create(ctypes.byref(dims), ctypes.byref(moe.CtxKvWeights(*ptrs)),
                                    ctypes.byref(h))
    return rc, moe.lib().moe_decode_error_message().decode()


@pytest.mark.parametrize("kw", [dict(hidden=100), dict(hidden=8200), dict(n_layers=0),
                                dict(n_layers=257), dict(head_dim=96), dict(n_kv_heads=0),
                                dict(n_kv_heads=129, head_dim=256), dict(max_ctx=0),
                                dict(max_ctx=65537), dict(max_position=0),
                                dict(max_position=(1 << 20) + 1),
                                dict(n_layers=256, max_ctx=65536, n_kv_heads=8)])
def test_ctxkv_unsupported_shapes(kw):
    rc, msg = _ctxkv_create(**kw)
    assert rc == moe.MOE_EUNSUPPORTED, (kw, rc, msg)
    assert msg


def test_ctxkv_invalid_arguments():
    for i in range(3):
        rc, msg = _ctxkv_create(null=i)
        assert rc == moe.MOE_EINVAL and "NULL" in msg
        rc, msg = _ctxkv_create(shift=i)
        assert rc == moe.MOE_EINVAL and "aligned" in msg
    for kw in (dict(eps=0.0), dict(qk_eps=-1.0), dict(rope_theta=-1.0)):
        rc, msg = _ctxkv_create(**kw)
        assert rc == moe.MOE_EINVAL, kw
    L = moe.lib()
    assert L.moe_ctxkv_create(None, None, None) == moe.MOE_EINVAL
    assert L.moe_ctxkv_project(None, 1, None, None, None, 0, None, None, 0, None, None, None) == moe.MOE_EINVAL
    ms = (ctypes.c_float * 3)()
    assert L.moe_ctxkv_profile(None, 1, None, None, None, 0, None, None, 0, None, ms) == moe.MOE_EINVAL
    assert L.moe_ctxkv_debug(None, None) == moe.MOE_EINVAL
    assert L.moe_ctxkv_last_error(None) == moe.MOE_EINVAL
    assert L.moe_ctxkv_kernel_count(None, 1) == moe.MOE_EINVAL
    assert L.moe_ctxkv_project_host(None, 1, None, None, None, 0, None, None, 0, None, None, None) == moe.MOE_EINVAL
    L.moe_ctxkv_destroy(None)


def test_cuda_core_expert_variant_compiles_cleanly(tmp_path):
    """The CUDA-core expert path, kept for measurement against the tensor-core
    path, still compiles (the -DMOE_EXPERT_FMA switch lives in capi.cu) with
    no warnings, as the default build does."""
    import shutil
    import subprocess
    nvcc = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc")
                                    else None)
    if nvcc is None:
        pytest.skip("nvcc not available")
    from speculative_decode_routed_gb300 import _build
    for extra in ((), ("-DMOE_EXPERT_FMA",)):
        (obj, argv), = [c for c in _build.compile_commands(nvcc, extra) if c[0].endswith("capi.o")]
        argv = [str(tmp_path / "capi.o") if a == obj else a for a in argv]
        r = subprocess.run(argv, capture_output=True, text=True, timeout=300)
        assert r.returncode == 0, r.stderr[-2000:]
        assert "warning" not in (r.stdout + r.stderr).lower(), (extra, r.stderr[-2000:])


def test_weight_streaming_split_choice(tmp_path):
    """gemv_splits (the split-K choice of the weight-streaming projection), run
    as host code: no split when K is not a multiple of 128 or R of 32; else a
    split count that divides K into 128-column steps, whose busiest-SM bytes
    are within 3 % of the best choice keeping 8 warps busy on every SM, and
    the fewest such splits."""
    import shutil
    import subprocess
    nvcc = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc")
                                    else None)
    if nvcc is None:
        pytest.skip("nvcc not available")
    csrc = os.path.join(os.path.dirname(moe.__file__), "csrc")
    cases = [(4, 2048, 7168, 152), (1, 7168, 28672, 152), (1, 4096, 1024, 152), (2, 512, 4096, 152),
             (4, 2048, 7168, 148), (1, 256, 384, 152), (1, 7168, 7000, 152), (1, 7000, 7168, 152),
             (8, 32, 128, 4)]
    src = tmp_path / "splits.cu"
    src.write_text('#include <cstdio>\n#include "gemv.cuh"\nint main() {\n' + "".join(
        f'  std::printf("%d\\n", moe::gemv_splits({L}, {R}, {K}, {n}));\n' for L, R, K, n in cases)
        + "  return 0;\n}\n")
    exe = tmp_path / "splits"
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-I", csrc,
                        str(src), "-o", str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True,
                                          timeout=60).stdout.split()]
    for (L, R, K, n), s in zip(cases, got):
        if K % 128 or R % 32:
            assert s == 0
            continue
        valid = [c for c in range(1, 33) if K % (128 * c) == 0]
        cost = {c: -(-(L * (R // 32) * c) // n) * (K // c) for c in valid}
        busy = [c for c in valid if L * (R // 32) * c >= 8 * n] or valid
        best = min(cost[c] for c in busy)
        assert s in busy and cost[s] * 100 <= best * 103, (L, R, K, n, s)
        assert all(cost[c] * 100 > best * 103 for c in busy if c < s), (L, R, K, n, s)
    assert got[0] == 7   # the context-KV projection: 4 layers of 2048 rows, K 7168


def test_header_is_plain_c_and_a_c_program_links(tmp_path):
    """include/moe_decode.h compiles as strict C11 (no C++ in the ABI), and a C
    program links against the library and gets a validation error back from
    moe_decode_create before any CUDA call."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    libdir = os.path.dirname(moe.LIB_PATH)
    src = tmp_path / "c_abi.c"
    src.write_text('#include "moe_decode.h"\n#include <stdio.h>\n'
                   "int main(void) {\n  moe_decode_dims d = {0};\n  moe_decode_t* h = NULL;\n"
                   "  int rc = moe_decode_create(&d, NULL, NULL, NULL, &h);\n"
                   '  printf("%d %s\\n", rc, moe_decode_strerror(rc));\n  return !(rc < 0 && h == NULL);\n}\n')
    exe = tmp_path / "c_abi"
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-I", os.path.join(root, "include"), str(src), "-L", libdir, "-lmoe_decode",
                        f"-Wl,-rpath,{libdir}", "-o", str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.split()[0] == str(moe.MOE_EINVAL)


def test_build_info_names_each_variant():
    """The default library is the tensor-core build without bounds checks; the
    bounds-check variant that build() makes beside it says so."""
    from speculative_decode_routed_gb300 import _build as pb
    assert moe.lib().moe_decode_build_info() == 0
    b = ctypes.CDLL(pb.LIB_BOUNDS)
    b.moe_decode_build_info.restype = ctypes.c_int
    assert b.moe_decode_build_info() == 1
