"""A decode step captured into a CUDA graph gives the same bits as the eager
calls, before and after its input buffers are updated in place."""
import pytest
import torch

import oracle
from paged_kv_cache_255_gb300 import inputs
from paged_kv_cache_255_gb300 import pagedattn as pa

import gpu_util as gu
import pins

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(pa_lib):
    return pa_lib


def _eager(d, wl):
    kc, vc = d["k_cache"].clone(), d["v_cache"].clone()
    pa.store_kvcache(d["k_new"], d["v_new"], kc, vc, d["slot_mapping"])
    out = pa.decode(d["q"], kc, vc, d["block_tables"], d["context_lens"], wl.scale)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("name", ["tiny", "large_batch"])
def test_graph_replay_matches_eager(name):
    spec = inputs.SPECS[name] if name == "tiny" else inputs.scaled(inputs.SPECS[name], num_seqs=24,
                                                                     ctx_div=4)
    wl = inputs.generate(spec, seed=21)
    d = gu.device_inputs(wl)
    want = _eager(d, wl)
    g = pa.DecodeStepGraph(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                           d["context_lens"], wl.scale, k_new=d["k_new"], v_new=d["v_new"],
                           slot_mapping=d["slot_mapping"])
    for _ in range(3):
        got = g.replay()
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    # new query and new rows, written into the graph's buffers in place
    wl2 = inputs.generate(spec, seed=22)
    d["q"].copy_(wl2.q.to(d["q"].device))
    d["k_new"].copy_(wl2.k_new.to(d["q"].device))
    d["v_new"].copy_(wl2.v_new.to(d["q"].device))
    got = g.replay()
    torch.cuda.synchronize()
    ref, _, _ = pins.run_step(oracle.get(), dataclasses_replace(wl, q=wl2.q, k_new=wl2.k_new,
                                                                 v_new=wl2.v_new))
    gu.assert_close(got, ref, f"{name} after in-place update")


def dataclasses_replace(wl, **kw):
    import dataclasses
    return dataclasses.replace(wl, **kw)


def test_graph_with_host_buffers():
    wl = inputs.generate(inputs.SPECS["tiny"], seed=23)
    d = gu.device_inputs(wl)
    want = _eager(d, wl)
    # pack q into a pinned staging buffer; the graph copies it in and the output out
    nbytes = d["q"].numel() * 2
    h_stage = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h_stage.copy_(wl.q.contiguous().view(-1).view(torch.uint8))
    d_stage = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    q_view = d_stage.view(torch.bfloat16).view(d["q"].shape)
    h_out = torch.empty(d["q"].shape, dtype=torch.bfloat16, pin_memory=True)
    g = pa.DecodeStepGraph(q_view, d["k_cache"], d["v_cache"], d["block_tables"],
                           d["context_lens"], wl.scale, k_new=d["k_new"], v_new=d["v_new"],
                           slot_mapping=d["slot_mapping"], host_stage=h_stage,
                           device_stage=d_stage, host_out=h_out)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(h_out.view(torch.int16), want.cpu().view(torch.int16))
