"""The C ABI from plain C: tests/c_abi_consumer.c is compiled with gcc against include/psk.h,
linked to the in-tree libpsk.so and run (size queries and argument checks only, no launch)."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plain_c_consumer():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from page_sparse_kv_gb300.build import build
    lib = build()
    libdir = os.path.dirname(lib)
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "consumer")
        r = subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                            os.path.join(ROOT, "tests", "c_abi_consumer.c"), "-L", libdir, "-lpsk",
                            f"-Wl,-rpath,{libdir}", "-o", exe], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
        r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
        assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
        assert r.stdout.startswith("version 100;")
