"""The boundary is a plain C ABI: a C program built against include/sa_api.h and linked to
libsa.so calls the host-only entry points and the argument checks (no GPU needed)."""
import os
import shutil
import subprocess

import pytest

import content_adaptive_sparse_gb300 as sa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_client_links_and_runs(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = sa.build_library()
    exe = tmp_path / "abi_smoke"
    subprocess.run([cc, "-std=c99", "-O1", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c", "abi_smoke.c"), "-o", str(exe),
                    "-L", os.path.dirname(lib), "-lsa", "-Wl,-rpath," + os.path.dirname(lib)],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    assert "c abi ok" in out.stdout
