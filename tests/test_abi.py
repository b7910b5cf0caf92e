"""The C ABI: the shared library loads, exports every entry point that
include/*.h declares, and rejects bad arguments on the host before any CUDA
call. CPU only: none of these calls reaches a kernel."""
import ctypes
import glob
import os
import re

import pytest

from paged_kv_cache_255_gb300 import pagedattn as pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_entry_points():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        with open(h) as fh:
            text = fh.read()
        names += re.findall(r"PA_API\s+[\w\s\*]+?\b(pa_\w+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(pa_lib):
    names = declared_entry_points()
    assert "pa_decode" in names and "pa_store_kvcache" in names
    for n in names:
        assert hasattr(pa_lib, n), f"{n} declared but not exported"
        assert n in pa.SIGNATURES, f"{n} has no binding"


def test_status_strings(pa_lib):
    assert pa.status_string(pa.PA_OK) == "PA_OK"
    assert pa.status_string(pa.PA_ERR_WORKSPACE) == "PA_ERR_WORKSPACE"
    assert pa.status_string(99) == "PA_ERR_UNKNOWN"


NULL = None


def _decode(pa_lib, **over):
    a = dict(q=16, k=16, v=16, bt=16, mb=4, cl=16, scale=0.1, out=16, S=2, Hq=16, Hkv=8, D=128,
             bs=16, NB=10, ws=16, wsb=1 << 20, stream=None)
    a.update(over)
    return pa_lib.pa_decode(a["q"], a["k"], a["v"], a["bt"], a["mb"], a["cl"], a["scale"],
                            a["out"], a["S"], a["Hq"], a["Hkv"], a["D"], a["bs"], a["NB"],
                            a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("over,want", [
    (dict(D=64), pa.PA_ERR_UNSUPPORTED),
    (dict(bs=24), pa.PA_ERR_UNSUPPORTED),
    (dict(bs=8), pa.PA_ERR_UNSUPPORTED),
    (dict(bs=512), pa.PA_ERR_UNSUPPORTED),
    (dict(Hq=12, Hkv=8), pa.PA_ERR_INVALID_ARG),
    (dict(Hq=8 * 64, Hkv=8), pa.PA_ERR_UNSUPPORTED),
    (dict(S=-1), pa.PA_ERR_INVALID_ARG),
    (dict(q=NULL), pa.PA_ERR_INVALID_ARG),
    (dict(cl=NULL), pa.PA_ERR_INVALID_ARG),
    (dict(out=18), pa.PA_ERR_INVALID_ARG),          # misaligned
    (dict(k=8), pa.PA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), pa.PA_ERR_INVALID_ARG),
    (dict(mb=0), pa.PA_ERR_INVALID_ARG),
    (dict(S=0, q=NULL, out=NULL), pa.PA_OK),        # empty batch: nothing to do
])
def test_decode_host_checks(pa_lib, over, want):
    assert _decode(pa_lib, **over) == want


def test_splitk_rejects_negative_partitions(pa_lib):
    st = pa_lib.pa_decode_splitk(16, 16, 16, 16, 4, 16, 0.1, 16, 2, 16, 8, 128, 16, 10, 16, 1 << 20,
                                 -1, None)
    assert st == pa.PA_ERR_INVALID_ARG


@pytest.mark.parametrize("over,want", [
    (dict(D=96), pa.PA_ERR_UNSUPPORTED),
    (dict(bs=48), pa.PA_ERR_UNSUPPORTED),
    (dict(N=-3), pa.PA_ERR_INVALID_ARG),
    (dict(k=NULL), pa.PA_ERR_INVALID_ARG),
    (dict(kc=24), pa.PA_ERR_INVALID_ARG),
    (dict(N=0, k=NULL, v=NULL, sm=NULL), pa.PA_OK),
])
def test_store_host_checks(pa_lib, over, want):
    a = dict(k=16, v=16, kc=16, vc=16, sm=16, N=4, Hkv=8, D=128, bs=16, NB=10)
    a.update(over)
    st = pa_lib.pa_store_kvcache(a["k"], a["v"], a["kc"], a["vc"], a["sm"], a["N"], a["Hkv"],
                                 a["D"], a["bs"], a["NB"], None)
    assert st == want


def test_workspace_size_rejects_bad_heads(pa_lib):
    assert pa_lib.pa_decode_workspace_size(12, 8, 128, 0) == 0
    assert pa_lib.pa_decode_workspace_size(16, 8, 64, 0) == 0
    assert pa_lib.pa_decode_workspace_size(16, 8, 128, -2) == 0


def test_binding_refuses_cpu_tensors(pa_lib):
    import torch
    q = torch.zeros(2, 16, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pa.decode(q, q, q, torch.zeros(2, 1, dtype=torch.int32), torch.zeros(2, dtype=torch.int32),
                  0.1)
