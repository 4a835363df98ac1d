"""The public header compiles as C99 and a C program linked against libpa
calls the host entry points (no Python between them, no GPU)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libdir():
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_167_gb300 import build
    return os.path.dirname(build.LIBRARY)


def test_host_calls_from_c(tmp_path, libdir):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from paged_kv_cache_167_gb300 import build
    cuda_inc = os.path.join(build._cuda_home(), "include")
    exe = tmp_path / "abi_from_c"
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
                    os.path.join(ROOT, "tests", "c", "abi_from_c.c"), "-o", str(exe), "-L", libdir, "-lpa",
                    "-Wl,-rpath," + libdir], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout + out.stderr
