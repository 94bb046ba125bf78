"""The C ABI from a plain C program (no Python binding, no torch): it is
compiled against include/ddl.h, linked with libddl.so, and run; it checks an
all-reduce of integer-valued inputs against their exact sums itself."""
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_allreduce_from_plain_c(tmp_path):
    import __graft_entry__
    __graft_entry__.build()
    libdir = os.path.join(ROOT, "gradient_all_reduce_ddl_gb300")
    exe = str(tmp_path / "allreduce_from_c")
    subprocess.check_call(["nvcc", "-O2", "-x", "c", os.path.join(ROOT, "tests", "c_abi", "allreduce_from_c.c"),
                           "-I", os.path.join(ROOT, "include"), "-L", libdir, "-lddl",
                           "-Xlinker", "-rpath", "-Xlinker", libdir, "-o", exe])
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.strip() == "ok"
