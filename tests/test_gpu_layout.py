"""Head-major pool [NB, Hkv, bs, D]: the store is bit-exact against the
oracle, and decode matches the oracle and, with a fixed partition count, the
token-major decode of the same values bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_255_gb300 import inputs
from paged_kv_cache_255_gb300 import pagedattn as pa

import gpu_util as gu

pytestmark = pytest.mark.gpu
SP = inputs.SPECS
CASES = {
    "tiny": SP["tiny"],
    "large_small": inputs.scaled(SP["large_batch"], num_seqs=16, ctx_div=4),
    "prefix_small": inputs.scaled(SP["prefix_shared"], num_seqs=8, ctx_div=8),
    "bs256": inputs.scaled(SP["qwen3_0_6b_bs256"], num_seqs=8),
    "g16_bs32": inputs.Spec("g16", ((5, 1, 500),), 32, 2, 32),
}


@pytest.fixture(scope="module", autouse=True)
def _lib(pa_lib):
    return pa_lib


def hm(t):
    return t.permute(0, 2, 1, 3).contiguous()


@pytest.mark.parametrize("name", sorted(CASES))
def test_head_major_store_and_decode(name):
    wl = inputs.generate(CASES[name], seed=61)
    O = oracle.get()
    hk_ref, hv_ref = O.store_kvcache_head_major(wl.k_new, wl.v_new, hm(wl.k_cache),
                                                hm(wl.v_cache), wl.slot_mapping)
    ref = O.decode_head_major(wl.q, hk_ref, hv_ref, wl.block_tables, wl.context_lens, wl.scale)
    d = gu.device_inputs(wl)
    hk, hv = hm(d["k_cache"]), hm(d["v_cache"])
    pa.store_kvcache(d["k_new"], d["v_new"], hk, hv, d["slot_mapping"], head_major=True)
    torch.cuda.synchronize()
    assert np.array_equal(gu.host_bits(hk), hk_ref) and np.array_equal(gu.host_bits(hv), hv_ref)
    out = pa.decode(d["q"], hk, hv, d["block_tables"], d["context_lens"], wl.scale,
                    head_major=True)
    torch.cuda.synchronize()
    gu.assert_close(out, ref, name)
    # same values in the token-major pool, same fixed partition count: same bits
    pa.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slot_mapping"])
    a = pa.decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                  wl.scale, num_partitions=97)
    b = pa.decode(d["q"], hk, hv, d["block_tables"], d["context_lens"], wl.scale,
                  num_partitions=97, head_major=True)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_layout_argument_is_checked(pa_lib):
    assert pa_lib.pa_store_kvcache_layout(16, 16, 16, 16, 16, 4, 8, 128, 16, 10, 7, None) == \
        pa.PA_ERR_INVALID_ARG


@pytest.mark.parametrize("name,Q", [("tiny", 3), ("large_small", 4), ("bs256", 8)])
def test_head_major_multi_token_decode(name, Q):
    """pa_decode_multi_layout on a head-major pool: against the oracle, and bit
    for bit against the token-major pool holding the same values."""
    wl = inputs.generate(CASES[name], seed=63)
    O = oracle.get()
    q = torch.randn((wl.num_seqs, Q, wl.spec.num_q_heads, wl.spec.head_dim),
                    generator=torch.Generator().manual_seed(64)).to(torch.bfloat16)
    kc, vc = O.store_kvcache(wl.k_new, wl.v_new, wl.k_cache, wl.v_cache, wl.slot_mapping)
    ref = O.decode_multi(q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
    d = gu.device_inputs(wl)
    pa.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slot_mapping"])
    hk, hv = hm(d["k_cache"]), hm(d["v_cache"])
    qd = q.cuda()
    a = pa.decode_multi(qd, d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                        wl.scale)
    b = pa.decode_multi(qd, hk, hv, d["block_tables"], d["context_lens"], wl.scale,
                        head_major=True)
    torch.cuda.synchronize()
    gu.assert_close(b, ref, f"{name} Q={Q} head-major")
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_multi_layout_argument_is_checked(pa_lib):
    st = pa_lib.pa_decode_multi_layout(None, None, None, None, 1, None, 2, 1.0, None, 1, 16, 8,
                                       128, 16, 4, 7, None, 0, None)
    assert st == 1    # PA_ERR_INVALID_ARG
