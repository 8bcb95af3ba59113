"""The CUDA path and the oracle share no code, and the product has no CPU path.

Static checks on the sources (no GPU): the package's Python never imports the
oracle or the tests' helpers; the CUDA sources and the public header include
nothing from the oracle, and the oracle includes nothing from them; the
seeded-input generators import neither side; bench.py reaches the oracle only
inside its CPU-baseline functions; and the binding raises ImportError, rather
than computing anything, when the library was not built.
"""
import ast
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "speculative_decode_routed_gb300")


def _files(top, exts):
    out = []
    for d, _, names in os.walk(top):
        if "__pycache__" in d or os.sep + "_build" in d:
            continue
        out += [os.path.join(d, n) for n in names if n.endswith(exts)]
    return sorted(out)


def _imported_modules(path):
    tree = ast.parse(open(path).read(), path)
    mods = set()
    for n in ast.walk(tree):
        if isinstance(n, ast.Import):
            mods |= {a.name.split(".")[0] for a in n.names}
        elif isinstance(n, ast.ImportFrom) and n.module and n.level == 0:
            mods.add(n.module.split(".")[0])
    return mods


def _includes(path):
    return re.findall(r'^\s*#\s*include\s*[<"]([^">]+)[">]', open(path).read(), re.M)


def test_package_python_imports_neither_the_oracle_nor_the_tests():
    files = _files(PKG, (".py",))
    assert files
    for f in files:
        bad = _imported_modules(f) & {"oracle", "helpers", "tests", "synth"}
        assert not bad, (f, bad)


def test_cuda_sources_and_oracle_include_nothing_of_each_other():
    cuda = _files(os.path.join(PKG, "csrc"), (".cu", ".cuh", ".h")) + _files(os.path.join(ROOT, "include"), (".h",))
    assert len(cuda) >= 10
    for f in cuda:
        for inc in _includes(f):
            assert "oracle" not in inc, (f, inc)
    oracle_src = _files(os.path.join(ROOT, "oracle"), (".c", ".h"))
    assert oracle_src
    for f in oracle_src:
        for inc in _includes(f):
            assert inc == "oracle.h" or "/" not in inc and not inc.endswith((".cuh", ".cu")), (f, inc)
            assert "moe_decode" not in inc and "csrc" not in inc, (f, inc)
    # the generators' C sources use system headers only
    gen = _files(os.path.join(ROOT, "synth"), (".c", ".cu", ".h"))
    assert gen
    for f in gen:
        for inc in _includes(f):
            assert "/" not in inc and inc.split(".")[0] in {"stdint", "stddef", "cstdint", "cuda_runtime",
                                                          "cuda_bf16", "math", "cmath", "string"}, (f, inc)


def test_oracle_and_input_generators_import_neither_side():
    for f in _files(os.path.join(ROOT, "oracle"), (".py",)):
        bad = _imported_modules(f) & {"speculative_decode_routed_gb300", "synth", "torch"}
        assert not bad, (f, bad)
    # the generators themselves serve both sides; synth/gpu.py only wraps their
    # output in the binding's structs for the GPU side
    for f in _files(os.path.join(ROOT, "synth"), (".py",)):
        banned = {"oracle", "helpers"}
        if os.path.basename(f) != "gpu.py":
            banned.add("speculative_decode_routed_gb300")
        bad = _imported_modules(f) & banned
        assert not bad, (f, bad)


def test_bench_reaches_the_oracle_only_in_its_cpu_baselines():
    path = os.path.join(ROOT, "bench.py")
    tree = ast.parse(open(path).read(), path)
    for n in tree.body:
        if isinstance(n, (ast.Import, ast.ImportFrom)):
            mods = {a.name for a in n.names} | {getattr(n, "module", None) or ""}
            assert not mods & {"oracle", "helpers"}, n.lineno
    seen = []
    for fn in ast.walk(tree):
        if not isinstance(fn, ast.FunctionDef):
            continue
        for n in ast.walk(fn):
            if isinstance(n, (ast.Import, ast.ImportFrom)):
                mods = {a.name for a in n.names} | {getattr(n, "module", None) or ""}
                if mods & {"oracle", "helpers"}:
                    seen.append(fn.name)
                    assert fn.name.endswith(("cpu_baseline", "cpu_baseline_modules")), (fn.name, n.lineno)
    assert seen


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    import speculative_decode_routed_gb300 as moe
    monkeypatch.setattr(moe, "_LIB", None)
    monkeypatch.setattr(moe, "LIB_PATH", str(tmp_path / "libmoe_decode.so"))
    with pytest.raises(ImportError):
        moe.lib()


def test_profile_summaries_name_their_commands():
    """Every ncu summary under profiles/ is short text that gives the command
    that made it: ncu with --clock-control none, running committed files only."""
    pdir = os.path.join(ROOT, "profiles")
    names = sorted(os.listdir(pdir))
    assert names
    for n in names:
        assert n.endswith((".md", ".txt")), n
        text = open(os.path.join(pdir, n)).read()
        assert len(text) < 16000, n
        assert "ncu " in text and "--clock-control none" in text, n
        assert "_work/" not in text and "/root/" not in text, n
