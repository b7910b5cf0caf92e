"""Seeded random decode steps through the C ABI against the fp64 oracle.

Each case draws the group size, the KV heads, the block size, the pool mode,
a length mix with zero-length sequences and lengths on and next to block
edges, the number of query tokens per sequence, the pool layout, and (for
single-token steps) a forced partition count. The store is checked bit for
bit and every output element against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_255_gb300 import inputs
from paged_kv_cache_255_gb300 import pagedattn as pa

import gpu_util as gu

pytestmark = pytest.mark.gpu
N_CASES = 16


@pytest.fixture(scope="module", autouse=True)
def _lib(pa_lib):
    return pa_lib


def _draw(case):
    rng = np.random.default_rng(9000 + case)
    g = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
    hkv = int(rng.choice([1, 2, 4, 8]))
    bs = int(rng.choice([16, 32, 64, 128, 256]))
    q_len = int(rng.choice([1, 1, 1, 2, 4]))
    while g * q_len > 16:
        q_len //= 2
    S = int(rng.integers(1, 24))
    lens = []
    for _ in range(S):
        kind = rng.random()
        if kind < 0.1:
            lens.append(0)
        elif kind < 0.35:
            lens.append(max(0, int(rng.integers(1, 6)) * bs + int(rng.integers(-1, 2))))
        else:
            lens.append(int(rng.integers(1, 1500)))
    spec = inputs.Spec(f"rand{case}", ((S, 1, 1),), g * hkv, hkv, bs,
                       pool_mode=str(rng.choice(["permute", "fragmented"])), pool_factor=1.3)
    head_major = bool(rng.integers(0, 2))
    parts = int(rng.choice([0, 0, 1, 3, 17, 300])) if q_len == 1 else 0
    return spec, np.asarray(lens, np.int32), q_len, head_major, parts


def _hm(t):
    return t.permute(0, 2, 1, 3).contiguous()


@pytest.mark.parametrize("case", range(N_CASES))
def test_random_decode_step(case):
    spec, lens, q_len, head_major, parts = _draw(case)
    wl = inputs.generate(spec, seed=case, context_lens=lens)
    O = oracle.get()
    d = gu.device_inputs(wl)
    what = (f"case {case}: g {spec.num_q_heads // spec.num_kv_heads}, Hkv {spec.num_kv_heads}, "
            f"bs {spec.block_size}, S {len(lens)}, q_len {q_len}, head_major {head_major}, "
            f"parts {parts}")
    if q_len > 1:
        q = torch.randn((len(lens), q_len, spec.num_q_heads, spec.head_dim),
                        generator=torch.Generator().manual_seed(case)).to(torch.bfloat16)
        kc, vc = O.store_kvcache(wl.k_new, wl.v_new, wl.k_cache, wl.v_cache, wl.slot_mapping)
        ref = O.decode_multi(q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
        pa.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slot_mapping"])
        torch.cuda.synchronize()
        assert np.array_equal(gu.host_bits(d["k_cache"]), kc), what
        assert np.array_equal(gu.host_bits(d["v_cache"]), vc), what
        kd, vd = (_hm(d["k_cache"]), _hm(d["v_cache"])) if head_major else (d["k_cache"], d["v_cache"])
        out = pa.decode_multi(q.cuda(), kd, vd, d["block_tables"], d["context_lens"], wl.scale,
                              head_major=head_major)
        torch.cuda.synchronize()
    elif head_major:
        hk_ref, hv_ref = O.store_kvcache_head_major(wl.k_new, wl.v_new, _hm(wl.k_cache),
                                                    _hm(wl.v_cache), wl.slot_mapping)
        ref = O.decode_head_major(wl.q, hk_ref, hv_ref, wl.block_tables, wl.context_lens,
                                  wl.scale)
        hk, hv = _hm(d["k_cache"]), _hm(d["v_cache"])
        pa.store_kvcache(d["k_new"], d["v_new"], hk, hv, d["slot_mapping"], head_major=True)
        out = pa.decode(d["q"], hk, hv, d["block_tables"], d["context_lens"], wl.scale,
                        num_partitions=parts, head_major=True)
        torch.cuda.synchronize()
        assert np.array_equal(gu.host_bits(hk), hk_ref), what
        assert np.array_equal(gu.host_bits(hv), hv_ref), what
    else:
        kc, vc = O.store_kvcache(wl.k_new, wl.v_new, wl.k_cache, wl.v_cache, wl.slot_mapping)
        ref = O.decode(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
        out, gkc, gvc = gu.gpu_step(wl, num_partitions=parts, d=d)
        assert np.array_equal(gu.host_bits(gkc), kc), what
        assert np.array_equal(gu.host_bits(gvc), vc), what
    gu.assert_close(out, ref, what)


def test_many_short_sequences():
    """3000 sequences of 0..40 tokens: the share planning scans the lengths in
    several chunks, and warps cross many small units."""
    lens = np.random.default_rng(77).integers(0, 41, 3000).astype(np.int32)
    spec = inputs.Spec("many", ((3000, 1, 1),), 32, 8, 16, pool_factor=1.2)
    wl = inputs.generate(spec, seed=3, context_lens=lens)
    O = oracle.get()
    kc, vc = O.store_kvcache(wl.k_new, wl.v_new, wl.k_cache, wl.v_cache, wl.slot_mapping)
    ref = O.decode(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
    out, gkc, gvc = gu.gpu_step(wl)
    assert np.array_equal(gu.host_bits(gkc), kc) and np.array_equal(gu.host_bits(gvc), vc)
    gu.assert_close(out, ref, "3000 short sequences")


def test_sequence_count_past_16_bits():
    """70,000 sequences of 0..40 tokens (2 q heads / 1 KV head, bs 16): more
    sequences than a 16-bit index holds; the share planning scans the lengths
    in about 550 chunks per CTA, and every output and the pool after the
    store are checked."""
    spec = inputs.Spec("many_seqs", ((70000, 0, 40),), 2, 1, 16)
    wl = inputs.generate(spec, seed=9)
    O = oracle.get()
    kc, vc = O.store_kvcache(wl.k_new, wl.v_new, wl.k_cache, wl.v_cache, wl.slot_mapping)
    ref = O.decode(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
    out, gkc, gvc = gu.gpu_step(wl)
    assert np.array_equal(gu.host_bits(gkc), kc) and np.array_equal(gu.host_bits(gvc), vc)
    gu.assert_close(out, ref, "70,000 sequences")
