"""NVTX ranges around the C ABI's entry points. A small NVTX tool
(tests/nvtx_recorder.c, built here with gcc) records the domain events that
libpagedattn emits; every entry point called must open exactly one range named
after itself in the domain "libpagedattn" and close it, also when it returns an
error. CPU only: every call below returns before any CUDA call (empty work, or
an argument rejected on the host)."""
import os
import shutil
import subprocess
import sys
import textwrap

import pytest

from paged_kv_cache_255_gb300 import build

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

# (entry point, call with ctypes arguments that return before any CUDA call)
CALLS = [
    ("pa_store_kvcache", "L.pa_store_kvcache(16, 16, 16, 16, 16, 0, 8, 128, 16, 10, None)"),
    ("pa_store_kvcache_layout",
     "L.pa_store_kvcache_layout(16, 16, 16, 16, 16, 0, 8, 128, 16, 10, 1, None)"),
    ("pa_decode", "L.pa_decode(16, 16, 16, 16, 4, 16, 0.1, 16, 0, 16, 8, 128, 16, 10, 16, 1 << 20, None)"),
    ("pa_decode_splitk",
     "L.pa_decode_splitk(16, 16, 16, 16, 4, 16, 0.1, 16, 0, 16, 8, 128, 16, 10, 16, 1 << 20, 3, None)"),
    ("pa_decode_layout",
     "L.pa_decode_layout(16, 16, 16, 16, 4, 16, 0.1, 16, 0, 16, 8, 128, 16, 10, 1, 16, 1 << 20, 0, None)"),
    ("pa_decode_multi",
     "L.pa_decode_multi(16, 16, 16, 16, 4, 16, 2, 0.1, 16, 0, 16, 8, 128, 16, 10, 16, 1 << 20, None)"),
    ("pa_decode_multi_layout",
     "L.pa_decode_multi_layout(16, 16, 16, 16, 4, 16, 2, 0.1, 16, 0, 16, 8, 128, 16, 10, 1, 16, 1 << 20, None)"),
    ("pa_prefill",
     "L.pa_prefill(16, 16, 16, 16, 4, 16, 16, 8, 0.1, 16, 0, 0, 16, 8, 128, 16, 10, None)"),
    ("pa_prefill_layout",
     "L.pa_prefill_layout(16, 16, 16, 16, 4, 16, 16, 8, 0.1, 16, 0, 0, 16, 8, 128, 16, 10, 1, None)"),
    ("pa_decode_step",
     "L.pa_decode_step(16, 16, 16, 0, 16, 16, 16, 16, 4, 16, 0.1, 16, 0, 16, 8, 128, 16, 10, 0, 16, 1 << 20, None)"),
    ("pa_take_device_error", "L.pa_take_device_error(None, None)"),
    # an argument error: the range still closes
    ("pa_decode", "L.pa_decode(16, 16, 16, 16, 4, 16, 0.1, 16, 2, 16, 8, 64, 16, 10, 16, 1 << 20, None)"),
]

EXPECTED_STATUS = [0] * 10 + [1, 2]     # PA_ERR_INVALID_ARG (null code), PA_ERR_UNSUPPORTED (head_dim)


def _cuda_include():
    nvcc = build._nvcc()
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "include")


@pytest.fixture(scope="module")
def recorder(tmp_path_factory, pa_lib):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    inc = _cuda_include()
    if not os.path.exists(os.path.join(inc, "nvtx3", "nvToolsExt.h")):
        pytest.skip("NVTX3 headers not found")
    out = tmp_path_factory.mktemp("nvtx") / "libnvtx_recorder.so"
    subprocess.run([gcc, "-shared", "-fPIC", "-O1", "-I", inc, "-o", str(out),
                    os.path.join(HERE, "nvtx_recorder.c")], check=True)
    return str(out)


def test_every_entry_point_opens_and_closes_its_range(recorder, tmp_path):
    log = tmp_path / "events.txt"
    script = textwrap.dedent("""
        import sys
        sys.path.insert(0, %r)
        from paged_kv_cache_255_gb300 import pagedattn as pa
        L = pa.lib()
        print(",".join(str(s) for s in [%s]))
    """) % (ROOT, ", ".join(c for _, c in CALLS))
    env = dict(os.environ, NVTX_INJECTION64_PATH=recorder, NVTX_RECORD_PATH=str(log),
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", script], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    assert [int(x) for x in r.stdout.strip().split(",")] == EXPECTED_STATUS
    events = [ln.split(" ", 2) for ln in log.read_text().splitlines()]
    ours = [e for e in events if len(e) > 1 and e[1] == "libpagedattn"]
    assert ours[0] == ["create", "libpagedattn"]
    assert sum(1 for e in ours if e[0] == "create") == 1
    want = []
    for name, _ in CALLS:
        want += [["push", "libpagedattn", name], ["pop", "libpagedattn"]]
    assert ours[1:] == want
