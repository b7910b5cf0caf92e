"""pa_decode_step (the store of a step's new rows, then decode, in one call)
through the C ABI: bit-identical to pa_store_kvcache followed by pa_decode on
the same inputs, the pool bit-exact against the oracle's store, and the
output against the oracle, on every decode shape (last-token stores, random
slots with -1 padding, an empty store) and both pool layouts."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_255_gb300 import inputs
from paged_kv_cache_255_gb300 import pagedattn as pa

import gpu_util as gu
import pins

pytestmark = pytest.mark.gpu
SP = inputs.SPECS

CASES = {
    "tiny": SP["tiny"],
    "qwen3_small": inputs.scaled(SP["qwen3_0_6b"], num_seqs=12),
    "large_small": inputs.scaled(SP["large_batch"], num_seqs=16, ctx_div=4),
    "long_small": inputs.scaled(SP["long_context"], num_seqs=16, ctx_div=16),
    "prefix_small": inputs.scaled(SP["prefix_shared"], num_seqs=8, ctx_div=8),
    "no_store": inputs.scaled(SP["qwen3_0_6b"], num_seqs=10, store_mode="none"),
}


@pytest.fixture(scope="module", autouse=True)
def _lib(pa_lib):
    return pa_lib


@pytest.mark.parametrize("name", sorted(CASES))
def test_step_matches_two_calls_and_oracle(name):
    wl = inputs.generate(CASES[name], seed=21)
    ref, kc, vc = pins.run_step(oracle.get(), wl)
    a = gu.device_inputs(wl)
    got = pa.decode_step(a["k_new"], a["v_new"], a["slot_mapping"], a["q"], a["k_cache"],
                         a["v_cache"], a["block_tables"], a["context_lens"], wl.scale)
    b = gu.device_inputs(wl)
    if wl.slot_mapping.shape[0]:
        pa.store_kvcache(b["k_new"], b["v_new"], b["k_cache"], b["v_cache"], b["slot_mapping"])
    want = pa.decode(b["q"], b["k_cache"], b["v_cache"], b["block_tables"], b["context_lens"],
                     wl.scale)
    torch.cuda.synchronize()
    assert pa.take_device_error() == 0
    assert torch.equal(got.view(torch.int16), want.view(torch.int16)), name
    kc, vc = oracle._bits(kc), oracle._bits(vc)     # the pools after the oracle's store
    assert np.array_equal(gu.host_bits(a["k_cache"]), kc) and np.array_equal(gu.host_bits(a["v_cache"]), vc)
    gu.assert_close(got, ref, name)


def test_step_on_head_major_pool():
    wl = inputs.generate(CASES["large_small"], seed=22)
    ref, _, _ = pins.run_step(oracle.get(), wl)
    a = gu.device_inputs(wl)
    kc = a["k_cache"].permute(0, 2, 1, 3).contiguous()
    vc = a["v_cache"].permute(0, 2, 1, 3).contiguous()
    got = pa.decode_step(a["k_new"], a["v_new"], a["slot_mapping"], a["q"], kc, vc,
                         a["block_tables"], a["context_lens"], wl.scale, head_major=True)
    torch.cuda.synchronize()
    gu.assert_close(got, ref, "head-major step")


def test_steps_back_to_back_read_each_others_rows():
    # two steps in a row on one pool: the second step's decode must see the
    # row the first step stored (and its own), with its lengths one longer
    spec = inputs.scaled(SP["qwen3_0_6b"], num_seqs=8)
    wl = inputs.generate(spec, seed=23)
    O = oracle.get()
    kc, vc = O.store_kvcache(wl.k_new, wl.v_new, wl.k_cache, wl.v_cache, wl.slot_mapping)
    a = gu.device_inputs(wl)
    pa.decode_step(a["k_new"], a["v_new"], a["slot_mapping"], a["q"], a["k_cache"], a["v_cache"],
                   a["block_tables"], a["context_lens"], wl.scale)
    # step 2: one more token per sequence where the block has room
    bs = spec.block_size
    L2 = wl.context_lens.astype(np.int64) + 1
    ok = (L2 + bs - 1) // bs <= (wl.context_lens.astype(np.int64) + bs - 1) // bs
    L2 = np.where(ok, L2, wl.context_lens).astype(np.int32)
    slots = np.array([int(wl.block_tables[s, (L2[s] - 1) // bs]) * bs + (L2[s] - 1) % bs if ok[s]
                      else -1 for s in range(wl.num_seqs)], dtype=np.int64)
    g = torch.Generator().manual_seed(5)
    k2 = torch.randn(wl.k_new.shape, generator=g).to(torch.bfloat16)
    v2 = torch.randn(wl.v_new.shape, generator=g).to(torch.bfloat16)
    q2 = torch.randn(wl.q.shape, generator=g).to(torch.bfloat16)
    kc2, vc2 = O.store_kvcache(k2, v2, kc, vc, slots)
    ref = O.decode(q2, kc2, vc2, wl.block_tables, L2, wl.scale)
    got = pa.decode_step(k2.cuda(), v2.cuda(), torch.from_numpy(slots).cuda(), q2.cuda(),
                         a["k_cache"], a["v_cache"], a["block_tables"],
                         torch.from_numpy(L2).cuda(), wl.scale)
    torch.cuda.synchronize()
    assert np.array_equal(gu.host_bits(a["k_cache"]), kc2)
    gu.assert_close(got, ref, "second step")
