"""The boundary from plain C: include/pagedattn.h compiles as strict C99 with
warnings as errors, a C program binds every declared entry point to a function
pointer of its declared type, links against libpagedattn and runs the calls
that return before any CUDA call. CPU only."""
import glob
import os
import re
import shutil
import subprocess

import pytest

from paged_kv_cache_255_gb300 import build

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_c_program_links_and_runs(pa_lib, tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    exe = tmp_path / "abi_from_c"
    lib_dir = os.path.dirname(build.LIB_PATH)
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), os.path.join(HERE, "abi_from_c.c"),
                    "-o", str(exe), "-L", lib_dir, "-lpagedattn", "-Wl,-rpath," + lib_dir],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "ok 0"


def test_c_program_names_every_declared_entry_point():
    declared = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        with open(h) as fh:
            declared |= set(re.findall(r"PA_API\s+[\w\s\*]+?\b(pa_\w+)\s*\(", fh.read()))
    with open(os.path.join(HERE, "abi_from_c.c")) as fh:
        bound = set(re.findall(r"=\s*(pa_\w+);", fh.read()))
    assert declared and declared == bound, sorted(declared ^ bound)
