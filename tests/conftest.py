import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: large sampled parity cases")


def _ensure_cpu_libs():
    """Build the CPU oracle and the host input generator if they are missing or
    older than their sources (plain gcc, a second or two)."""
    from oracle import _build as ob
    from synth import _build as sb

    for cmd in ob.commands() + sb.commands()[:1]:
        out = cmd[cmd.index("-o") + 1]
        srcs = [a for a in cmd if a.endswith(".c")]
        stale = not os.path.exists(out) or any(
            os.path.getmtime(s) > os.path.getmtime(out) for s in srcs)
        if stale:
            subprocess.check_call(cmd)


_ensure_cpu_libs()


def _ensure_cuda_lib():
    """Build the CUDA library (nvcc cross-compiles without a GPU) if it is
    missing or older than its sources, so the C-ABI host tests do not depend
    on an earlier build() of this checkout."""
    import shutil

    from speculative_decode_routed_gb300 import _build as pb
    srcs = [os.path.join(pb.CSRC, f) for f in os.listdir(pb.CSRC)]
    srcs.append(os.path.join(ROOT, "include", "moe_decode.h"))
    if all(os.path.exists(lib) and all(os.path.getmtime(s) <= os.path.getmtime(lib) for s in srcs)
           for lib in (pb.LIB, pb.LIB_BOUNDS)):
        return
    if shutil.which("nvcc") is None:
        return  # the tests that load the library then fail loudly
    import __graft_entry__
    try:
        __graft_entry__.build()
    except Exception as e:  # noqa: BLE001 -- the oracle's tests still run
        print(f"conftest: building the CUDA library failed: {e}")


_ensure_cuda_lib()


def has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if has_gpu():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)
