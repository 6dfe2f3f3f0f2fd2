"""The oracle and the CUDA path stay independent, and the product path has
no fallback: static checks of the sources, plus an import of the binding
without its library.  CPU only."""
from __future__ import annotations

import os
import re
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "query_conditioned_kv_gb300")


def _sources(folder, exts):
    for base, _, files in os.walk(folder):
        if "_build" in base or "__pycache__" in base:
            continue
        for f in files:
            if f.endswith(exts):
                yield os.path.join(base, f)


def test_product_sources_never_reference_the_oracle():
    pat = re.compile(r"\boracle\b|liboracle|orc_[a-z]")
    for path in [*_sources(PKG, (".py", ".cu", ".cuh", ".h")),
                 *_sources(os.path.join(ROOT, "include"), (".h",))]:
        with open(path) as f:
            hits = [ln for ln in f if pat.search(ln)]
        assert not hits, (path, hits[:3])


def test_oracle_includes_only_the_c_library():
    with open(os.path.join(ROOT, "oracle", "oracle.c")) as f:
        inc = re.findall(r'^\s*#\s*include\s*[<"]([^>"]+)[>"]', f.read(), re.M)
    assert set(inc) <= {"math.h", "stdint.h", "stdlib.h", "string.h"}, inc
    for name in ("__init__.py", "build.py"):
        with open(os.path.join(ROOT, "oracle", name)) as f:
            text = f.read()
        assert "query_conditioned_kv_gb300" not in text and "kvc_" not in text, name


def test_benchmark_loads_the_oracle_only_in_its_cpu_legs():
    with open(os.path.join(ROOT, "bench.py")) as f:
        src = f.read()
    top = [ln for ln in src.splitlines() if re.match(r"(import|from)\s+oracle\b", ln)]
    assert not top  # no module-level import: only inside the CPU-baseline functions
    # and those functions run only in the CPU-baseline legs (never in a timed region)
    for fn in ("_oracle_event", "_oracle_slotmap"):
        callers = [m.start() for m in re.finditer(rf"(?<!def ){fn}\(", src)]
        for pos in callers:
            caller = re.findall(r"^def (\w+)", src[:pos], re.M)
            assert not caller or caller[-1] in (fn, "cpu_baseline", "run_reference",
                                                 "config_event", "slot_map_event"), caller[-1:]
    for m in re.finditer(r"^\s+(?:import|from)\s+oracle\b", src, re.M):
        fn = re.findall(r"^def (\w+)", src[:m.start()], re.M)[-1]
        assert fn in ("_oracle_event", "_oracle_slotmap"), fn


def test_binding_without_its_library_fails_loudly(tmp_path):
    dst = tmp_path / "query_conditioned_kv_gb300"
    dst.mkdir()
    shutil.copyfile(os.path.join(PKG, "__init__.py"), dst / "__init__.py")
    p = subprocess.run([sys.executable, "-c", "import query_conditioned_kv_gb300"],
                       cwd=tmp_path, capture_output=True, text=True, timeout=120)
    assert p.returncode != 0
    assert "ImportError" in p.stderr and "no fallback" in p.stderr.replace("\n", " ")
