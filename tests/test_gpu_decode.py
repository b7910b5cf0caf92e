"""GPU parity: the CUDA path (called through the C ABI) against the fp64 oracle.

Small cases are compared element by element; the full-size decode steps are
run in the launch configuration the benchmark times and compared on sampled
(sequence, head) outputs that the oracle computes one by one, plus
properties that hold at any size. The store is bit-exact everywhere.
"""
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

SMALL = {
    "tiny": SP["tiny"],
    "qwen3_small": inputs.scaled(SP["qwen3_0_6b"], num_seqs=12),
    "qwen3_bs256_small": inputs.scaled(SP["qwen3_0_6b_bs256"], num_seqs=12),
    "large_small": inputs.scaled(SP["large_batch"], num_seqs=16, ctx_div=4),
    "long_small": inputs.scaled(SP["long_context"], num_seqs=16, ctx_div=16),
    "prefix_small": inputs.scaled(SP["prefix_shared"], num_seqs=8, ctx_div=8),
    "mha": inputs.Spec("mha", ((5, 1, 200),), 8, 8, 16),
    "g8_bs32": inputs.Spec("g8_bs32", ((6, 1, 400),), 64, 8, 32),
    "one_kv_head": inputs.Spec("one_kv_head", ((3, 30, 500),), 4, 1, 64),
    "g3": inputs.Spec("g3", ((5, 1, 300),), 24, 8, 16),
    "g5_bs128": inputs.Spec("g5_bs128", ((4, 100, 900),), 40, 8, 128),
    "g12": inputs.Spec("g12", ((4, 1, 333),), 48, 4, 16),
    "g16": inputs.Spec("g16", ((6, 1, 700),), 32, 2, 32),
}
# tile computations: tensor cores (default) and CUDA cores (group <= 8)
KERNELS = ["mma", "simt"]


@pytest.fixture(params=KERNELS)
def kernel(request, monkeypatch):
    gu.decode_kernel(request.param)
    return request.param


@pytest.fixture(scope="module", autouse=True)
def _lib(pa_lib):
    return pa_lib


@pytest.mark.parametrize("name", sorted(SMALL))
def test_decode_matches_oracle(name, kernel):
    wl = inputs.generate(SMALL[name], seed=1)
    ref, kc, vc = pins.run_step(oracle.get(), wl)
    out, gkc, gvc = gu.gpu_step(wl)
    assert np.array_equal(gu.host_bits(gkc), kc) and np.array_equal(gu.host_bits(gvc), vc)
    gu.assert_close(out, ref, name)


@pytest.mark.parametrize("name", ["tiny", "large_small", "long_small", "prefix_small"])
@pytest.mark.parametrize("parts", [1, 2, 7, 64, 5000])
def test_forced_partitions(name, parts, kernel):
    wl = inputs.generate(SMALL[name], seed=2)
    ref, _, _ = pins.run_step(oracle.get(), wl)
    out, _, _ = gu.gpu_step(wl, num_partitions=parts)
    gu.assert_close(out, ref, f"{name} P={parts}")


@pytest.mark.parametrize("bs", [16, 64, 256])
def test_edge_lengths(bs, kernel):
    lens = [0, 1, 2, 15, 16, 17, 31, 32, 33, 255, 256, 257, 0, 1000]
    spec = inputs.Spec("edges", ((len(lens), 1, 1),), 16, 4, bs)
    wl = inputs.generate(spec, seed=3, context_lens=lens)
    ref, _, _ = pins.run_step(oracle.get(), wl)
    for parts in (0, 3):
        out, _, _ = gu.gpu_step(wl, num_partitions=parts)
        gu.assert_close(out, ref, f"edges bs={bs} P={parts}")
        assert torch.count_nonzero(out[0]) == 0 and torch.count_nonzero(out[12]) == 0


def test_store_skips_padding_bit_exact():
    wl = inputs.generate(SP["prefix_shared"], seed=4)
    kc, vc = oracle.store_kvcache(wl.k_new, wl.v_new, wl.k_cache, wl.v_cache, wl.slot_mapping)
    d = gu.device_inputs(wl)
    pa.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slot_mapping"])
    torch.cuda.synchronize()
    assert np.array_equal(gu.host_bits(d["k_cache"]), kc)
    assert np.array_equal(gu.host_bits(d["v_cache"]), vc)


def test_single_token_returns_v_row_exactly(kernel):
    spec = inputs.Spec("one", ((7, 1, 1),), 32, 8, 16)
    wl = inputs.generate(spec, seed=5)
    out, _, _ = gu.gpu_step(wl)
    v = wl.v_new.to(out.device)                      # the stored row is the only token
    want = v.repeat_interleave(4, dim=1)
    assert torch.equal(out.view(torch.int16), want.view(torch.int16))


def test_unit_values_give_exact_one(kernel):
    spec = inputs.scaled(SP["large_batch"], num_seqs=8, ctx_div=4)
    wl = inputs.generate(spec, seed=6, keep_content=True)
    wl = pins._with_values(wl, v_fill=1.0)
    out, _, _ = gu.gpu_step(wl)
    assert torch.equal(out, torch.ones_like(out))


def test_renumbering_and_private_prefix_are_bit_identical(kernel):
    spec = inputs.scaled(SP["prefix_shared"], num_seqs=6, ctx_div=8, store_mode="none",
                         store_rows=0, pad_rows=0)
    wl = inputs.generate(spec, seed=7)
    a, _, _ = gu.gpu_step(wl)
    b, _, _ = gu.gpu_step(pins._renumber(wl, seed=8))
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # private copies of the shared prefix blocks
    pb, S = spec.prefix_blocks, wl.num_seqs
    kc = torch.cat([wl.k_cache, wl.k_cache[torch.from_numpy(wl.block_tables[:, :pb].reshape(-1)).long()]])
    vc = torch.cat([wl.v_cache, wl.v_cache[torch.from_numpy(wl.block_tables[:, :pb].reshape(-1)).long()]])
    bt = wl.block_tables.copy()
    bt[:, :pb] = wl.num_blocks + np.arange(S * pb).reshape(S, pb)
    import dataclasses
    wl2 = dataclasses.replace(wl, k_cache=kc, v_cache=vc, block_tables=bt,
                              num_blocks=int(kc.shape[0]))
    c, _, _ = gu.gpu_step(wl2)
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


FULL = ["qwen3_0_6b", "qwen3_0_6b_bs256", "large_batch", "long_context", "prefix_shared"]


def _sample_pairs(wl, n, seed):
    """Every query head of the 8 longest sequences (on long_context these are
    the units the split-K path cuts into the most pieces), the first and last
    output, and random (sequence, head) pairs up to n more."""
    rng = np.random.Generator(np.random.PCG64(seed))
    S, Hq = wl.num_seqs, wl.spec.num_q_heads
    longest = np.argsort(-wl.context_lens, kind="stable")[:8]
    pairs = [(int(s), h) for s in longest for h in range(Hq)]
    pairs += [(0, 0), (S - 1, Hq - 1)]
    for _ in range(n):
        pairs.append((int(rng.integers(S)), int(rng.integers(Hq))))
    return np.array(pairs, dtype=np.int32)


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name):
    wl = inputs.generate(SP[name], seed=0, device="cuda")
    host_k, host_v = wl.k_cache.cpu(), wl.v_cache.cpu()        # pre-store pools for the oracle
    out, gkc, gvc = gu.gpu_step(wl)                              # default launch, as benchmarked
    O = oracle.get()
    if wl.slot_mapping.shape[0]:
        kc, vc = O.store_kvcache(wl.k_new.cpu(), wl.v_new.cpu(), host_k, host_v, wl.slot_mapping)
        assert np.array_equal(gu.host_bits(gkc), kc) and np.array_equal(gu.host_bits(gvc), vc)
    else:
        kc, vc = host_k, host_v
    pairs = _sample_pairs(wl, 40, seed=1)
    ref = O.decode_pairs(wl.q.cpu(), kc, vc, wl.block_tables, wl.context_lens, wl.scale, pairs)
    got = out[torch.from_numpy(pairs[:, 0]).long(), torch.from_numpy(pairs[:, 1]).long()]
    gu.assert_close(got, ref, name)
    # any size: finite, and a convex combination of N(0,1) rows stays small
    assert torch.isfinite(out).all()
    assert out.float().abs().max().item() < 6.0


def test_full_size_step_on_head_major_pool():
    """The headline step on a head-major pool, as the benchmark runs it: one
    pa_decode_step call; every head of the 8 longest sequences and 40 more
    sampled outputs against the oracle, the pool bit-exact after the store."""
    wl = inputs.generate(SP["long_context"], seed=0, device="cuda")
    host_k, host_v = wl.k_cache.cpu(), wl.v_cache.cpu()
    kc = wl.k_cache.permute(0, 2, 1, 3).contiguous()
    vc = wl.v_cache.permute(0, 2, 1, 3).contiguous()
    del wl.k_cache, wl.v_cache
    out = pa.decode_step(wl.k_new, wl.v_new, torch.from_numpy(wl.slot_mapping).cuda(), wl.q, kc,
                         vc, torch.from_numpy(wl.block_tables).cuda(),
                         torch.from_numpy(wl.context_lens).cuda(), wl.scale, head_major=True)
    torch.cuda.synchronize()
    assert pa.take_device_error() == 0
    O = oracle.get()
    rk, rv = O.store_kvcache(wl.k_new.cpu(), wl.v_new.cpu(), host_k, host_v, wl.slot_mapping)
    got_k = gu.host_bits(kc.permute(0, 2, 1, 3).contiguous())
    assert np.array_equal(got_k, rk)
    pairs = _sample_pairs(wl, 40, seed=2)
    ref = O.decode_pairs(wl.q.cpu(), rk, rv, wl.block_tables, wl.context_lens, wl.scale, pairs)
    got = out[torch.from_numpy(pairs[:, 0]).long(), torch.from_numpy(pairs[:, 1]).long()]
    gu.assert_close(got, ref, "long_context head-major")


def test_full_size_multi_token_decode():
    """The qwen3-shaped step with 4 new query tokens per sequence, as the
    benchmark runs it (the step's store, then pa_decode_multi): every output
    against the oracle."""
    wl = inputs.generate(SP["qwen3_0_6b"], seed=0, device="cuda")
    host_k, host_v = wl.k_cache.cpu(), wl.v_cache.cpu()
    g = torch.Generator().manual_seed(11)
    S, Hq, D = wl.q.shape
    q = torch.randn((S, 4, Hq, D), generator=g).to(torch.bfloat16)
    d = gu.device_inputs(wl)
    pa.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slot_mapping"])
    out = pa.decode_multi(q.cuda(), d["k_cache"], d["v_cache"], d["block_tables"],
                          d["context_lens"], wl.scale)
    torch.cuda.synchronize()
    assert pa.take_device_error() == 0
    O = oracle.get()
    rk, rv = O.store_kvcache(wl.k_new.cpu(), wl.v_new.cpu(), host_k, host_v, wl.slot_mapping)
    ref = O.decode_multi(q, rk, rv, wl.block_tables, wl.context_lens, wl.scale)
    gu.assert_close(out, ref, "qwen3 Q=4")


@pytest.mark.parametrize("scale", [0.0, -0.08838834764831845, 1.0])
def test_decode_scales(scale, kernel):
    """Scale edge cases on both tile computations: zero (every weight equal,
    the output the mean of the V rows), negative (the softmax of the negated
    scores: the running minimum of the raw scores leads), and 1.0, eleven
    times the usual 1/sqrt(128) (sharp weights and large running-max jumps
    between tiles); store then decode against the oracle."""
    wl = inputs.generate(SMALL["large_small"], seed=5)
    O = oracle.get()
    kc, vc = O.store_kvcache(wl.k_new, wl.v_new, wl.k_cache, wl.v_cache, wl.slot_mapping)
    ref = O.decode(wl.q, kc, vc, wl.block_tables, wl.context_lens, scale)
    d = gu.device_inputs(wl)
    pa.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slot_mapping"])
    out = pa.decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                    scale)
    torch.cuda.synchronize()
    assert pa.take_device_error() == 0
    gu.assert_close(out, ref, f"scale {scale}")


def test_million_token_sequence():
    """A maximum-length step: one sequence of 2^20 tokens among three short
    ones (32 q / 8 KV heads, bs 16; a block-table row of 65,536 entries), in
    the benchmark's launch configuration. Each long (sequence, KV head) is cut
    into about 230 split-K pieces that the combine merges in many batches;
    the store is checked bit for bit and every output row against the oracle."""
    spec = inputs.Spec("million", ((1, 1 << 20, 1 << 20), (3, 1, 2000)), 32, 8, 16)
    wl = inputs.generate(spec, seed=3, device="cuda")
    host_k, host_v = wl.k_cache.cpu(), wl.v_cache.cpu()
    out, gkc, gvc = gu.gpu_step(wl)
    O = oracle.get()
    kc, vc = O.store_kvcache(wl.k_new.cpu(), wl.v_new.cpu(), host_k, host_v, wl.slot_mapping)
    assert np.array_equal(gu.host_bits(gkc), kc) and np.array_equal(gu.host_bits(gvc), vc)
    del gkc, gvc, host_k, host_v
    S, Hq = wl.q.shape[0], wl.q.shape[1]
    pairs = np.array([(s, h) for s in range(S) for h in range(Hq)], dtype=np.int32)
    ref = O.decode_pairs(wl.q.cpu(), kc, vc, wl.block_tables, wl.context_lens, wl.scale, pairs)
    got = out[torch.from_numpy(pairs[:, 0]).long(), torch.from_numpy(pairs[:, 1]).long()]
    gu.assert_close(got, ref, "2^20-token sequence")
