"""include/mla.h is a C header: a strict C99 program includes it, links
libmla.so and calls the host-only paths (version, status strings, argument
checks) from C, without a GPU."""

import os
import shutil
import subprocess

import pytest

from mla_latent_kv_71_b300 import mla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_header_compiles_as_c99_and_links(tmp_path):
    mla.library()  # builds libmla.so in-tree if it is missing or stale
    lib_dir = os.path.dirname(mla.LIB_PATH)
    exe = str(tmp_path / "c_abi_check")
    cmd = ["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_abi_check.c"),
           "-L", lib_dir, "-lmla", f"-Wl,-rpath,{lib_dir}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
