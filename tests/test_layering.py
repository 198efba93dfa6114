"""Layering of the repository, checked on the source text (no GPU needed).

- The oracle and the CUDA path share no code: the oracle's C source includes
  only the C library, the CUDA sources include nothing of the oracle, and
  neither Python side imports the other. The seeded input generators
  (``workloads``) hold no arithmetic of the method and serve both.
- The product path never reaches the oracle: the package does not import it,
  and ``bench.py`` imports it only inside its CPU-baseline and reference legs.
- There is no CPU fallback: a missing CUDA library makes the first call raise.
"""
import ast
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "diffusion_transformer_joint_gb300")
C_LIBRARY = {"math.h", "pthread.h", "stdint.h", "stdlib.h", "string.h", "stddef.h", "stdio.h"}
BENCH_CPU_LEGS = {"cpu_baseline", "proj_cpu_baseline", "_oracle_sample", "cpu_report",
                  "run_reference"}


def _files(top, exts):
    for d, _, names in os.walk(top):
        if "_build" in d or "__pycache__" in d:
            continue
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def _includes(path):
    return re.findall(r'^\s*#\s*include\s*[<"]([^>"]+)[>"]', open(path).read(), flags=re.M)


def _imports(path):
    """(top-level module, enclosing function or None) for every import in a file."""
    found = []

    def walk(node, fn):
        for ch in ast.iter_child_nodes(node):
            inner = ch.name if isinstance(ch, (ast.FunctionDef, ast.AsyncFunctionDef)) else fn
            if isinstance(ch, ast.Import):
                found.extend((a.name.split(".")[0], fn) for a in ch.names)
            elif isinstance(ch, ast.ImportFrom) and ch.level == 0 and ch.module:
                found.append((ch.module.split(".")[0], fn))
            walk(ch, inner)

    walk(ast.parse(open(path).read()), None)
    return found


def test_oracle_c_source_includes_only_the_c_library():
    srcs = list(_files(os.path.join(ROOT, "oracle"), (".c", ".h")))
    assert srcs
    for path in srcs:
        assert set(_includes(path)) <= C_LIBRARY, path


def test_cuda_sources_include_nothing_of_the_oracle():
    srcs = list(_files(PKG, (".cu", ".cuh", ".h", ".cpp"))) + list(
        _files(os.path.join(ROOT, "include"), (".h",)))
    assert srcs
    for path in srcs:
        for inc in _includes(path):
            assert "oracle" not in inc, (path, inc)
        assert "liboracle" not in open(path).read(), path


def test_oracle_package_imports_nothing_of_the_product():
    for path in _files(os.path.join(ROOT, "oracle"), (".py",)):
        mods = {m for m, _ in _imports(path)}
        assert not mods & {"diffusion_transformer_joint_gb300", "bench", "binding"}, path


def test_product_package_never_imports_the_oracle():
    for path in _files(PKG, (".py",)):
        assert "oracle" not in {m for m, _ in _imports(path)}, path
        assert "liboracle" not in open(path).read(), path


def test_bench_reaches_the_oracle_only_in_its_cpu_legs():
    uses = [fn for m, fn in _imports(os.path.join(ROOT, "bench.py")) if m == "oracle"]
    assert uses, "the CPU baseline needs the oracle"
    assert None not in uses, "a module-level import would load the oracle on every run"
    assert set(uses) <= BENCH_CPU_LEGS, set(uses) - BENCH_CPU_LEGS


def test_missing_cuda_library_fails_loudly():
    env = dict(os.environ, FLUX_ATTN_LIB=os.path.join(ROOT, "_no_such_dir", "libflux_attn.so"))
    res = subprocess.run(
        [sys.executable, "-c", "from diffusion_transformer_joint_gb300 import binding; "
                               "binding.load()"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=120)
    assert res.returncode != 0
    assert "CUDA library not built" in res.stderr
