"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Such a caller cannot hand pa_decode a workspace (it may not call cudaMalloc
on its path, or device memory belongs to a framework that only passes in
inputs and outputs), so this entry point keeps its scratch in a static
device array inside the library. The test calls it through the C ABI twice
in a row, on two decode steps with the same head configuration and different
length mixes (partial results a first call left in the shared array would
show up in the second), and checks each output bit for bit against
pa_decode's on the same inputs and element by element against the fp64
oracle; a head configuration too big for the static scratch must be refused.

Kept in its own file, collected last, so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

import oracle
from paged_kv_cache_255_gb300 import inputs
from paged_kv_cache_255_gb300 import pagedattn as pa

import gpu_util as gu

pytestmark = pytest.mark.gpu
NOALLOC_SCRATCH_BYTES = 16 << 20      # PA_NOALLOC_SCRATCH_BYTES in include/pagedattn.h


def _noalloc(lib, d, wl):
    s = wl.spec
    out = torch.full_like(d["q"], float("nan"))
    st = lib.pa_decode_noalloc(
        d["q"].data_ptr(), d["k_cache"].data_ptr(), d["v_cache"].data_ptr(),
        d["block_tables"].data_ptr(), d["block_tables"].shape[1], d["context_lens"].data_ptr(),
        ctypes.c_float(wl.scale), out.data_ptr(), wl.num_seqs, s.num_q_heads, s.num_kv_heads,
        s.head_dim, s.block_size, wl.num_blocks,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, out


def test_noalloc_matches_decode_and_oracle_on_two_calls(pa_lib):
    # both steps have 32 query / 8 KV heads; the second mixes one long
    # sequence (cut into many split-K pieces) with short ones
    steps = [inputs.scaled(inputs.SPECS["large_batch"], num_seqs=24, ctx_div=4),
             inputs.scaled(inputs.SPECS["long_context"], num_seqs=16, ctx_div=8)]
    heads = {(s.num_q_heads, s.num_kv_heads) for s in steps}
    assert len(heads) == 1
    O = oracle.get()
    for i, spec in enumerate(steps):
        wl = inputs.generate(spec, seed=40 + i, device="cuda")
        host_k, host_v = wl.k_cache.cpu(), wl.v_cache.cpu()
        d = gu.device_inputs(wl)
        if wl.slot_mapping.shape[0]:
            pa.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slot_mapping"])
        want = pa.decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                         d["context_lens"], wl.scale)
        st, got = _noalloc(pa_lib, d, wl)
        torch.cuda.synchronize()
        assert st == pa.PA_OK, pa.status_string(st)
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), \
            f"noalloc call {i + 1} differs from pa_decode"
        kc, vc = O.store_kvcache(wl.k_new.cpu(), wl.v_new.cpu(), host_k, host_v, wl.slot_mapping)
        ref = O.decode(wl.q.cpu(), kc, vc, wl.block_tables, wl.context_lens, wl.scale)
        gu.assert_close(got, ref, f"noalloc call {i + 1} against the oracle")


def test_noalloc_refuses_scratch_beyond_limit(pa_lib):
    # a group of 16 query heads per KV head needs more scratch than the array
    need = pa.decode_workspace_size(32, 2)
    if need <= NOALLOC_SCRATCH_BYTES:
        pytest.skip("this device's scratch need fits the static array")
    spec = inputs.Spec("g16", ((3, 10, 100),), 32, 2, 16)
    wl = inputs.generate(spec, seed=3, device="cuda")
    d = gu.device_inputs(wl)
    st, out = _noalloc(pa_lib, d, wl)
    torch.cuda.synchronize()
    assert st == pa.PA_ERR_WORKSPACE
    assert torch.isnan(out.float()).all(), "a refused call must launch nothing"
