"""The C ABI used from a plain C program (tests/c/host_abi.c) compiled with
the system C compiler against include/pa.h and linked to libpa.so: the host
entry points (allocator, step planner, partition chooser, work order) behave
as from Python.  No GPU needed."""
import os
import shutil
import subprocess

import pytest

from paged_kv_cache_283_gb300 import pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_host_entry_points_from_c(tmp_path):
    cc = shutil.which("cc") or shutil.which("gcc")
    if cc is None:
        pytest.skip("no C compiler")
    if not os.path.exists(pa.LIB_PATH):
        from paged_kv_cache_283_gb300 import build
        build.build()
    libdir = os.path.dirname(pa.LIB_PATH)
    exe = str(tmp_path / "host_abi")
    subprocess.run([cc, "-std=c99", "-O1", "-o", exe, os.path.join(ROOT, "tests", "c", "host_abi.c"),
                    "-I", os.path.join(ROOT, "include"), "-L", libdir, "-lpa",
                    "-Wl,-rpath," + libdir], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok"
