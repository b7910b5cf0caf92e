"""Multi-token decode (speculative verification) through the C ABI against
the fp64 oracle: query token i of Q attends to keys t <= L - Q + i."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_255_gb300 import inputs
from paged_kv_cache_255_gb300 import pagedattn as pa

import gpu_util as gu

pytestmark = pytest.mark.gpu
SP = inputs.SPECS

CASES = [
    ("tiny", SP["tiny"], 3),                                                    # g 2, 6 columns
    ("qwen3_small", inputs.scaled(SP["qwen3_0_6b"], num_seqs=10), 4),         # g 2, 8 columns
    ("large_small", inputs.scaled(SP["large_batch"], num_seqs=12, ctx_div=4), 4),  # g 4, 16
    ("long_small", inputs.scaled(SP["long_context"], num_seqs=16, ctx_div=16), 2),
    ("g8", inputs.scaled(SP["prefix_shared"], num_seqs=6, ctx_div=8), 2),     # g 8, 16 columns
    ("mha_q16", inputs.Spec("mha", ((4, 20, 300),), 8, 8, 16), 16),           # g 1, 16 columns
    ("g3_bs64", inputs.Spec("g3", ((5, 1, 400),), 24, 8, 64), 5),             # g 3, 15 columns
    ("bs256", inputs.scaled(SP["qwen3_0_6b_bs256"], num_seqs=6), 8),          # g 2, 16 columns
]


@pytest.fixture(scope="module", autouse=True)
def _lib(pa_lib):
    return pa_lib


def _multi_q(wl, Q, seed):
    g = torch.Generator().manual_seed(seed)
    S, Hq, D = wl.q.shape
    return torch.randn((S, Q, Hq, D), generator=g).to(torch.bfloat16)


def _run(wl, q, context_lens=None):
    O = oracle.get()
    cl = wl.context_lens if context_lens is None else context_lens
    kc, vc = wl.k_cache, wl.v_cache
    if wl.slot_mapping.shape[0]:
        kc, vc = O.store_kvcache(wl.k_new, wl.v_new, kc, vc, wl.slot_mapping)
    ref = O.decode_multi(q, kc, vc, wl.block_tables, cl, wl.scale)
    d = gu.device_inputs(wl)
    if wl.slot_mapping.shape[0]:
        pa.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slot_mapping"])
    out = pa.decode_multi(q.cuda(), d["k_cache"], d["v_cache"], d["block_tables"],
                          torch.from_numpy(np.asarray(cl, np.int32)).cuda(), wl.scale)
    torch.cuda.synchronize()
    return out, ref, d


@pytest.mark.parametrize("name,spec,Q", CASES, ids=[c[0] for c in CASES])
def test_multi_matches_oracle(name, spec, Q):
    wl = inputs.generate(spec, seed=41)
    q = _multi_q(wl, Q, 42)
    out, ref, _ = _run(wl, q)
    gu.assert_close(out, ref, f"{name} Q={Q}")


def test_single_query_token_equals_decode():
    wl = inputs.generate(inputs.scaled(SP["large_batch"], num_seqs=12, ctx_div=4), seed=43)
    q = wl.q[:, None]                                      # [S, 1, Hq, D]
    out, _, d = _run(wl, q)
    want = pa.decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                     wl.scale)
    torch.cuda.synchronize()
    assert torch.equal(out[:, 0].view(torch.int16), want.view(torch.int16))


def test_sequences_shorter_than_the_query_block():
    lens = [0, 1, 2, 3, 5, 16, 17, 40]
    spec = inputs.Spec("short", ((len(lens), 1, 1),), 16, 4, 16)
    wl = inputs.generate(spec, seed=44, context_lens=lens)
    Q = 4
    q = _multi_q(wl, Q, 45)
    out, ref, _ = _run(wl, q)
    gu.assert_close(out, ref, "short sequences")
    # query tokens before the sequence start see nothing
    assert torch.count_nonzero(out[0]) == 0
    assert torch.count_nonzero(out[1, :3]) == 0 and torch.count_nonzero(out[2, :2]) == 0


def test_multi_rejects_too_many_columns(pa_lib):
    # 4 heads per KV head x 5 query tokens = 20 columns > 16
    assert pa_lib.pa_decode_multi_workspace_size(5, 32, 8, 128) == 0
