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
    (dict(NB=1 << 27), pa.PA_ERR_UNSUPPORTED),      # 2^31 token rows: past 32-bit coordinates
    (dict(NB=1 << 26, Hq=32, Hkv=32), pa.PA_ERR_UNSUPPORTED),  # 2^31 (block, head) rows
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


# One-call decode step: the store's checks, then the decode's, all before any
# launch (with no device visible, a launch attempt would return PA_ERR_CUDA).
@pytest.mark.parametrize("over,want", [
    (dict(N=-1), pa.PA_ERR_INVALID_ARG),
    (dict(k=NULL), pa.PA_ERR_INVALID_ARG),
    (dict(D=64), pa.PA_ERR_UNSUPPORTED),
    (dict(layout=3), pa.PA_ERR_INVALID_ARG),
    (dict(Hq=12), pa.PA_ERR_INVALID_ARG),            # the store is valid, nothing is launched
    (dict(q=NULL), pa.PA_ERR_INVALID_ARG),
    (dict(cl=24), pa.PA_ERR_INVALID_ARG),           # misaligned is only checked for 16-byte tensors
    (dict(out=18), pa.PA_ERR_INVALID_ARG),
    (dict(N=0, S=0, k=NULL, q=NULL), pa.PA_OK),     # nothing to store, no sequence
])
def test_decode_step_host_checks(pa_lib, over, want):
    a = dict(k=16, v=16, sm=16, N=4, q=16, kc=16, vc=16, bt=16, mb=4, cl=16, scale=0.1, out=16,
             S=2, Hq=16, Hkv=8, D=128, bs=16, NB=10, layout=0, ws=16, wsb=1 << 20)
    a.update(over)
    if a["cl"] == 24:       # lengths have no alignment rule: use a null instead
        a["cl"] = NULL
    st = pa_lib.pa_decode_step(a["k"], a["v"], a["sm"], a["N"], a["q"], a["kc"], a["vc"], a["bt"],
                               a["mb"], a["cl"], a["scale"], a["out"], a["S"], a["Hq"], a["Hkv"],
                               a["D"], a["bs"], a["NB"], a["layout"], a["ws"], a["wsb"], None)
    assert st == want


def test_workspace_size_rejects_bad_heads(pa_lib):
    assert pa_lib.pa_decode_workspace_size(12, 8, 128, 0) == 0
    assert pa_lib.pa_decode_workspace_size(16, 8, 64, 0) == 0
    assert pa_lib.pa_decode_workspace_size(16, 8, 128, -2) == 0


# Prefill: every case is rejected (or has no work) before any CUDA call.
@pytest.mark.parametrize("over,want", [
    (dict(D=64), pa.PA_ERR_UNSUPPORTED),
    (dict(bs=24), pa.PA_ERR_UNSUPPORTED),
    (dict(Hq=12, Hkv=8), pa.PA_ERR_INVALID_ARG),
    (dict(Hq=8 * 32, Hkv=8), pa.PA_ERR_UNSUPPORTED),     # group above 16
    (dict(S=-1), pa.PA_ERR_INVALID_ARG),
    (dict(T=-1), pa.PA_ERR_INVALID_ARG),
    (dict(mql=-1), pa.PA_ERR_INVALID_ARG),
    (dict(mb=-1), pa.PA_ERR_INVALID_ARG),
    (dict(NB=-1), pa.PA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), pa.PA_ERR_INVALID_ARG),
    (dict(q=NULL), pa.PA_ERR_INVALID_ARG),
    (dict(qsl=NULL), pa.PA_ERR_INVALID_ARG),
    (dict(bt=NULL), pa.PA_ERR_INVALID_ARG),
    (dict(out=24), pa.PA_ERR_INVALID_ARG),               # misaligned
    (dict(v=40), pa.PA_ERR_INVALID_ARG),
    (dict(mb=0), pa.PA_ERR_INVALID_ARG),
    (dict(NB=0), pa.PA_ERR_INVALID_ARG),
    (dict(S=70000), pa.PA_ERR_UNSUPPORTED),              # grid limit
    (dict(Hq=70000 * 2, Hkv=70000), pa.PA_ERR_UNSUPPORTED),
    (dict(S=0, q=NULL, out=NULL, qsl=NULL), pa.PA_OK),   # empty batch
    (dict(T=0, q=NULL, out=NULL), pa.PA_OK),             # no query rows
    (dict(NB=1 << 27), pa.PA_ERR_UNSUPPORTED),           # pool rows past 32-bit coordinates
    (dict(NB=1 << 26, Hq=32, Hkv=32), pa.PA_ERR_UNSUPPORTED),
])
def test_prefill_host_checks(pa_lib, over, want):
    a = dict(q=16, k=16, v=16, bt=16, mb=4, cl=16, qsl=16, mql=8, scale=0.1, out=16, S=2, T=20,
             Hq=16, Hkv=8, D=128, bs=16, NB=10)
    a.update(over)
    args = (a["q"], a["k"], a["v"], a["bt"], a["mb"], a["cl"], a["qsl"], a["mql"], a["scale"],
            a["out"], a["S"], a["T"], a["Hq"], a["Hkv"], a["D"], a["bs"], a["NB"])
    assert pa_lib.pa_prefill(*args, None) == want
    assert pa_lib.pa_prefill_layout(*args, 1, None) == want


def test_prefill_layout_argument_is_checked(pa_lib):
    args = (16, 16, 16, 16, 4, 16, 16, 8, 0.1, 16, 2, 20, 16, 8, 128, 16, 10)
    assert pa_lib.pa_prefill_layout(*args, 2, None) == pa.PA_ERR_INVALID_ARG
    assert pa_lib.pa_prefill_layout(*args, -1, None) == pa.PA_ERR_INVALID_ARG


# Multi-token decode: q_len new tokens per sequence; (query token, head)
# columns of one KV head are at most 16.
@pytest.mark.parametrize("over,want", [
    (dict(Q=0), pa.PA_ERR_INVALID_ARG),
    (dict(Q=17), pa.PA_ERR_UNSUPPORTED),
    (dict(Q=9), pa.PA_ERR_UNSUPPORTED),                  # 2 heads x 9 tokens = 18 columns
    (dict(Q=4, Hq=40, Hkv=8), pa.PA_ERR_UNSUPPORTED),    # group 5 x 4 tokens pads past 16
    (dict(D=256), pa.PA_ERR_UNSUPPORTED),
    (dict(Hq=10, Hkv=4), pa.PA_ERR_INVALID_ARG),
    (dict(S=-2), pa.PA_ERR_INVALID_ARG),
    (dict(q=NULL), pa.PA_ERR_INVALID_ARG),
    (dict(out=8), pa.PA_ERR_INVALID_ARG),
    (dict(S=0, q=NULL, out=NULL), pa.PA_OK),
])
def test_decode_multi_host_checks(pa_lib, over, want):
    a = dict(q=16, k=16, v=16, bt=16, mb=4, cl=16, Q=4, scale=0.1, out=16, S=2, Hq=16, Hkv=8,
             D=128, bs=16, NB=10, ws=16, wsb=1 << 20)
    a.update(over)
    args = (a["q"], a["k"], a["v"], a["bt"], a["mb"], a["cl"], a["Q"], a["scale"], a["out"],
            a["S"], a["Hq"], a["Hkv"], a["D"], a["bs"], a["NB"])
    assert pa_lib.pa_decode_multi(*args, a["ws"], a["wsb"], None) == want
    assert pa_lib.pa_decode_multi_layout(*args, 1, a["ws"], a["wsb"], None) == want


def test_layout_arguments_are_checked(pa_lib):
    dec = (16, 16, 16, 16, 4, 16, 0.1, 16, 2, 16, 8, 128, 16, 10)
    assert pa_lib.pa_decode_layout(*dec, 3, 16, 1 << 20, 0, None) == pa.PA_ERR_INVALID_ARG
    assert pa_lib.pa_decode_layout(*dec, 0, 16, 1 << 20, -1, None) == pa.PA_ERR_INVALID_ARG
    multi = (16, 16, 16, 16, 4, 16, 2, 0.1, 16, 2, 16, 8, 128, 16, 10)
    assert pa_lib.pa_decode_multi_layout(*multi, 7, 16, 1 << 20, None) == pa.PA_ERR_INVALID_ARG
    st = (16, 16, 16, 16, 16, 4, 8, 128, 16, 10)
    assert pa_lib.pa_store_kvcache_layout(*st, 2, None) == pa.PA_ERR_INVALID_ARG


def test_multi_workspace_size_rejects_bad_shapes(pa_lib):
    assert pa_lib.pa_decode_multi_workspace_size(0, 16, 8, 128) == 0
    assert pa_lib.pa_decode_multi_workspace_size(17, 16, 8, 128) == 0
    assert pa_lib.pa_decode_multi_workspace_size(9, 16, 8, 128) == 0
    assert pa_lib.pa_decode_multi_workspace_size(2, 12, 8, 128) == 0
    assert pa_lib.pa_decode_multi_workspace_size(2, 16, 8, 64) == 0


def test_binding_refuses_cpu_tensors(pa_lib):
    import torch
    q = torch.zeros(2, 16, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pa.decode(q, q, q, torch.zeros(2, 1, dtype=torch.int32), torch.zeros(2, dtype=torch.int32),
                  0.1)
