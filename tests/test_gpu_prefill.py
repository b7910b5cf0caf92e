"""Paged prefill through the C ABI against the fp64 oracle: each sequence's
chunk of new rows is stored through its slot mapping, then row i of a chunk of
n in a sequence of L attends to keys t <= L - n + i."""
import time

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_255_gb300 import inputs
from paged_kv_cache_255_gb300 import pagedattn as pa

import gpu_util as gu

pytestmark = pytest.mark.gpu
PS = inputs.PREFILL_SPECS


def _spec(name, Hq, Hkv, bs):
    return inputs.Spec(name, ((1, 1, 1),), Hq, Hkv, bs, store_mode="none")


_MANY = [int(x) for x in np.random.default_rng(5).integers(1, 41, 300)]
# the largest batch whose CTAs start longest-first (256 sequences are ranked in
# shared memory; some chunks and one context empty); many_short (300) is past it
_rng = np.random.default_rng(6)
_CTX256 = [int(x) for x in _rng.integers(0, 300, 256)]
_CHK256 = [0 if i % 17 == 3 else int(min(c, x))
           for i, (c, x) in enumerate(zip(_CTX256, _rng.integers(1, 140, 256)))]
_CTX256[20] = _CHK256[20] = 0

# (id, spec, chunk, context_lens, chunk_lens)
CASES = [
    ("g4_mixed", _spec("a", 8, 2, 16), None, [37, 200, 16, 129, 5], [37, 64, 1, 100, 5]),
    ("g1_bs32", _spec("b", 8, 8, 32), None, [1, 70, 130, 64], [1, 70, 3, 64]),
    ("g2_prompts", inputs.scaled(PS["qwen3_0_6b_prompts"][0], num_seqs=6, ctx_div=4), None,
     None, None),
    ("g4_chunked", inputs.scaled(PS["chunked_8b"][0], num_seqs=4, ctx_div=16), 100, None, None),
    ("g8_bs64", _spec("c", 64, 8, 64), None, [300, 77, 129], [150, 77, 65]),
    ("g16_bs256", _spec("d", 32, 2, 256), None, [520, 33, 1000], [520, 10, 257]),
    ("g3_pad4", _spec("e", 24, 8, 16), None, [90, 17, 256], [45, 17, 200]),
    ("g5_pad8", _spec("f", 40, 8, 128), None, [400, 9], [131, 9]),
    ("empty_chunks", _spec("g", 16, 8, 16), None, [0, 5, 16, 64, 65, 3],
     [0, 0, 16, 1, 65, 3]),
    # many short whole prompts: 300 sequences of 1..40 tokens (one CTA row per sequence)
    ("many_short", _spec("h", 16, 4, 16), None, _MANY, _MANY),
    ("ranked_256", _spec("p", 16, 4, 16), None, _CTX256, _CHK256),
    # one KV head with a group that pads up: the padded group is taller than q's heads
    ("g3_one_kv", _spec("i", 3, 1, 16), None, [150, 40], [150, 17]),
    ("g6_one_kv", _spec("j", 6, 1, 32), None, [90, 260], [90, 65]),
]


@pytest.fixture(scope="module", autouse=True)
def _lib(pa_lib):
    return pa_lib


def _device(pb):
    wl = pb.wl
    return dict(
        q=pb.q.cuda(), k_new=pb.k_new.cuda(), v_new=pb.v_new.cuda(),
        slot_mapping=torch.from_numpy(pb.slot_mapping).cuda(),
        k_cache=wl.k_cache.cuda(), v_cache=wl.v_cache.cuda(),
        block_tables=torch.from_numpy(wl.block_tables).cuda(),
        context_lens=torch.from_numpy(wl.context_lens).cuda(),
        qsl=torch.from_numpy(pb.query_start_loc).cuda())


def _gpu_step(pb, d, max_query_len=None):
    """Store the chunk rows, then prefill (the engine's prompt step)."""
    if pb.slot_mapping.shape[0]:
        pa.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slot_mapping"])
    out = pa.prefill(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                     d["qsl"], pb.wl.scale, max_query_len=max_query_len)
    torch.cuda.synchronize()
    return out


def _oracle_caches(pb):
    O = oracle.get()
    kc, vc = pb.wl.k_cache, pb.wl.v_cache
    if pb.slot_mapping.shape[0]:
        kc, vc = O.store_kvcache(pb.k_new, pb.v_new, kc, vc, pb.slot_mapping)
    return kc, vc


@pytest.fixture(autouse=True)
def _no_device_error():
    assert pa.take_device_error() == 0
    yield
    assert pa.take_device_error() == 0, "a prefill launch recorded a device-side error"


# tc: tcgen05 with TMEM accumulators (the default); mma: the mma.sync kernel
KERNELS = ["tc", "mma"]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("name,spec,chunk,lens,chunks", CASES, ids=[c[0] for c in CASES])
def test_prefill_matches_oracle(name, spec, chunk, lens, chunks, kernel, monkeypatch):
    gu.prefill_kernel(kernel)
    pb = inputs.prefill_batch(spec, seed=61, chunk=chunk, context_lens=lens, chunk_lens=chunks)
    kc, vc = _oracle_caches(pb)
    ref = oracle.get().prefill(pb.q, kc, vc, pb.wl.block_tables, pb.wl.context_lens,
                               pb.query_start_loc, pb.wl.scale)
    d = _device(pb)
    out = _gpu_step(pb, d)
    gu.assert_close(out, ref, f"{name} ({kernel})")
    # the store half of the step is byte-exact
    assert np.array_equal(gu.host_bits(d["k_cache"]), np.asarray(kc))
    assert np.array_equal(gu.host_bits(d["v_cache"]), np.asarray(vc))


@pytest.mark.parametrize("kernel", KERNELS)
def test_small_max_query_len_hint_still_correct(kernel, monkeypatch):
    """The hint only sizes the grid: a CTA walks further query tiles itself."""
    gu.prefill_kernel(kernel)
    spec = _spec("h", 16, 8, 16)
    pb = inputs.prefill_batch(spec, seed=62, context_lens=[700, 300], chunk_lens=[650, 300])
    d = _device(pb)
    want = _gpu_step(pb, d)
    got = pa.prefill(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                     d["qsl"], pb.wl.scale, max_query_len=8)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_equal_chunks_match_multi_token_decode():
    """With Q new rows in every sequence, prefill and multi-token decode compute
    the same attention; both stay within tolerance of the oracle."""
    spec = _spec("i", 32, 8, 16)
    Q, lens = 4, [40, 90, 17, 33, 300]
    pb = inputs.prefill_batch(spec, seed=63, context_lens=lens, chunk_lens=[Q] * len(lens))
    d = _device(pb)
    out = _gpu_step(pb, d)
    multi = pa.decode_multi(d["q"].view(len(lens), Q, 32, 128), d["k_cache"], d["v_cache"],
                            d["block_tables"], d["context_lens"], pb.wl.scale)
    torch.cuda.synchronize()
    kc, vc = _oracle_caches(pb)
    ref = oracle.get().prefill(pb.q, kc, vc, pb.wl.block_tables, pb.wl.context_lens,
                               pb.query_start_loc, pb.wl.scale)
    gu.assert_close(out, ref, "prefill")
    gu.assert_close(multi.reshape(out.shape), ref, "decode_multi")


def _sampled_rows_ref(pb, kc, vc, rows):
    """Oracle output of chosen rows: row i of a chunk of n in a sequence of L
    is a one-row chunk of a sequence cut to its first L - n + i + 1 tokens."""
    qsl = pb.query_start_loc
    seq = np.searchsorted(qsl, rows, side="right") - 1
    n = qsl[seq + 1] - qsl[seq]
    i = rows - qsl[seq]
    L = pb.wl.context_lens[seq].astype(np.int64)
    cut = (L - n + i + 1).astype(np.int32)
    one = np.arange(len(rows) + 1, dtype=np.int32)
    return oracle.get().prefill(pb.q[torch.from_numpy(rows)], kc, vc,
                                pb.wl.block_tables[seq], cut, one, pb.wl.scale)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("scale", [-0.3, 0.0])
def test_negative_and_zero_scale(kernel, scale, monkeypatch):
    """A negative scale flips which score is the max; scale 0 is uniform
    attention over the visible keys (masked keys still get nothing)."""
    gu.prefill_kernel(kernel)
    spec = _spec("k", 16, 8, 16)
    pb = inputs.prefill_batch(spec, seed=66, context_lens=[150, 40, 300],
                              chunk_lens=[100, 40, 260])
    kc, vc = _oracle_caches(pb)
    ref = oracle.get().prefill(pb.q, kc, vc, pb.wl.block_tables, pb.wl.context_lens,
                               pb.query_start_loc, scale)
    d = _device(pb)
    pa.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slot_mapping"])
    out = pa.prefill(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                     d["qsl"], scale)
    torch.cuda.synchronize()
    gu.assert_close(out, ref, f"scale {scale} ({kernel})")


@pytest.mark.parametrize("name", sorted(PS))
def test_full_size_sampled_rows(name):
    """The benchmarked prefill steps at full size, in the benchmark's launch
    configuration; the oracle checks a sample of rows one by one (the first and
    last rows of the first 16 chunks and 32 random rows)."""
    spec, chunk = PS[name]
    pb = inputs.prefill_batch(spec, seed=0, chunk=chunk)
    d = _device(pb)
    out = _gpu_step(pb, d, max_query_len=pb.max_query_len)
    qsl = pb.query_start_loc
    rng = np.random.Generator(np.random.PCG64(64))
    firsts = qsl[:-1][np.diff(qsl) > 0]
    lasts = qsl[1:][np.diff(qsl) > 0] - 1
    rows = np.unique(np.concatenate([firsts[:16], lasts[:16],
                                     rng.integers(0, qsl[-1], size=32)])).astype(np.int64)
    kc = d["k_cache"].cpu()
    vc = d["v_cache"].cpu()
    ref = _sampled_rows_ref(pb, kc, vc, rows)
    gu.assert_close(out[torch.from_numpy(rows).cuda()], ref, name)
    assert torch.isfinite(out.float()).all()


def test_long_chunk_over_long_context():
    """A maximum-size prefill: one sequence of 131,072 tokens takes a chunk of
    its last 16,384 (32 q / 8 KV heads, so 256 pairs of query tiles per KV
    head, each reading up to 1024 key tiles), beside a 300-token whole prompt;
    the persistent CTAs walk thousands of items. The oracle checks sampled rows
    one by one: the first and last rows of both chunks and 20 random ones."""
    pb = inputs.prefill_batch(_spec("long_chunk", 32, 8, 16), seed=17,
                              context_lens=[131072, 300], chunk_lens=[16384, 300])
    d = _device(pb)
    out = _gpu_step(pb, d, max_query_len=pb.max_query_len)
    qsl = pb.query_start_loc
    rng = np.random.Generator(np.random.PCG64(71))
    rows = np.unique(np.concatenate([qsl[:-1], qsl[1:] - 1,
                                     rng.integers(0, qsl[-1], size=20)])).astype(np.int64)
    ref = _sampled_rows_ref(pb, d["k_cache"].cpu(), d["v_cache"].cpu(), rows)
    gu.assert_close(out[torch.from_numpy(rows).cuda()], ref, "16k-row chunk over 128k tokens")
    assert torch.isfinite(out.float()).all()


def test_launches_on_two_streams_at_once():
    """Persistent CTAs take over only CTAs of their own grid: two prefill
    launches running at the same time on two streams, each grid several times
    the SM count, both match the oracle. The batches differ in group size and
    length mix, so a cell handed across grids would be detected."""
    specs = [(_spec("two_a", 32, 8, 16), [3000, 900, 2200, 64, 1500, 4000], [600, 900, 128, 64, 1, 700]),
             (_spec("two_b", 16, 8, 32), [700, 1800, 300, 2500, 90], [700, 400, 300, 513, 90])]
    jobs = []
    for i, (spec, lens, chunks) in enumerate(specs):
        pb = inputs.prefill_batch(spec, seed=90 + i, context_lens=lens, chunk_lens=chunks)
        kc, vc = _oracle_caches(pb)
        ref = oracle.get().prefill(pb.q, kc, vc, pb.wl.block_tables, pb.wl.context_lens,
                                   pb.query_start_loc, pb.wl.scale)
        d = _device(pb)
        if pb.slot_mapping.shape[0]:
            pa.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slot_mapping"])
        jobs.append((pb, d, ref))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in jobs]
    outs = []
    for (pb, d, _), st in zip(jobs, streams):
        with torch.cuda.stream(st):
            outs.append(pa.prefill(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                   d["context_lens"], d["qsl"], pb.wl.scale))
    torch.cuda.synchronize()
    for (pb, _, ref), out in zip(jobs, outs):
        gu.assert_close(out, ref, pb.wl.spec.name)


def test_rejects_bad_shapes():
    spec = _spec("j", 16, 8, 16)
    pb = inputs.prefill_batch(spec, seed=65, context_lens=[20], chunk_lens=[20])
    d = _device(pb)
    with pytest.raises(ValueError):
        pa.prefill(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                   d["qsl"][:1], pb.wl.scale)
    with pytest.raises(pa.PagedAttnError):      # 12 query heads over 8 KV heads
        pa.prefill(d["q"][:, :12].contiguous(), d["k_cache"], d["v_cache"],
                   d["block_tables"], d["context_lens"], d["qsl"], pb.wl.scale)


def _random_case(rng):
    """A seeded random prefill step: group size, block size, lengths and chunk
    pattern drawn over the supported range."""
    Hkv = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.choice([1, 2, 3, 4, 6, 8, 16]))
    bs = int(rng.choice([16, 32, 64, 128, 256]))
    S = int(rng.integers(1, 6))
    lens, chunks = [], []
    for _ in range(S):
        L = int(rng.integers(0, 700))
        kind = rng.integers(0, 4)
        n = L if kind == 0 else (0 if kind == 1 or L == 0 else int(rng.integers(1, L + 1)))
        lens.append(L)
        chunks.append(n)
    return _spec("r", g * Hkv, Hkv, bs), lens, chunks


@pytest.mark.parametrize("case", range(12))
def test_random_prefill_steps(case, monkeypatch):
    """Twelve seeded random steps, tcgen05 kernel, element-wise against the
    oracle (and the mma.sync kernel on the same inputs)."""
    rng = np.random.Generator(np.random.PCG64(1000 + case))
    spec, lens, chunks = _random_case(rng)
    pb = inputs.prefill_batch(spec, seed=2000 + case, context_lens=lens, chunk_lens=chunks)
    kc, vc = _oracle_caches(pb)
    ref = oracle.get().prefill(pb.q, kc, vc, pb.wl.block_tables, pb.wl.context_lens,
                               pb.query_start_loc, pb.wl.scale)
    for kernel in KERNELS:
        gu.prefill_kernel(kernel)
        d = _device(pb)
        out = _gpu_step(pb, d)
        gu.assert_close(out, ref, f"random case {case} ({kernel}): g {spec.num_q_heads // spec.num_kv_heads} "
                                  f"Hkv {spec.num_kv_heads} bs {spec.block_size} lens {lens} chunks {chunks}")


LAYOUT_CASES = [
    ("g4_mixed", _spec("a", 8, 2, 16), [37, 200, 16, 129, 5], [37, 64, 1, 100, 5]),
    ("g2_bs64", _spec("l", 16, 8, 64), [300, 77, 600], [150, 77, 333]),
    ("g8_bs256", _spec("m", 64, 8, 256), [520, 33], [520, 10]),
]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("name,spec,lens,chunks", LAYOUT_CASES, ids=[c[0] for c in LAYOUT_CASES])
def test_head_major_pool(name, spec, lens, chunks, kernel, monkeypatch):
    """The step on a head-major pool [NB, Hkv, bs, D] (store and prefill both
    head-major) matches the oracle, and the prefill gives the same bits as on
    the token-major pool holding the same values."""
    gu.prefill_kernel(kernel)
    pb = inputs.prefill_batch(spec, seed=67, context_lens=lens, chunk_lens=chunks)
    kc, vc = _oracle_caches(pb)
    ref = oracle.get().prefill(pb.q, kc, vc, pb.wl.block_tables, pb.wl.context_lens,
                               pb.query_start_loc, pb.wl.scale)
    d = _device(pb)
    k_hm = d["k_cache"].permute(0, 2, 1, 3).contiguous()
    v_hm = d["v_cache"].permute(0, 2, 1, 3).contiguous()
    pa.store_kvcache(d["k_new"], d["v_new"], k_hm, v_hm, d["slot_mapping"], head_major=True)
    out_hm = pa.prefill(d["q"], k_hm, v_hm, d["block_tables"], d["context_lens"], d["qsl"],
                        pb.wl.scale, head_major=True)
    out_tm = _gpu_step(pb, d)
    torch.cuda.synchronize()
    gu.assert_close(out_hm, ref, f"{name} head-major ({kernel})")
    assert torch.equal(out_hm.view(torch.int16), out_tm.view(torch.int16))
    assert torch.equal(k_hm.permute(0, 2, 1, 3).view(torch.int16), d["k_cache"].view(torch.int16))


def test_bounded_wait_runs_out_and_reports():
    """The tcgen05 kernel's waits are bounded: with the test hook holding back
    one barrier arrival, the launch returns after about 2 s with code 2 instead
    of hanging, and the context stays usable (the next launch is correct)."""
    spec = _spec("t", 2, 1, 16)
    pb = inputs.prefill_batch(spec, seed=68, context_lens=[100], chunk_lens=[100])
    d = _device(pb)
    pa.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slot_mapping"])
    torch.cuda.synchronize()
    pa.debug_prefill_fault(1)
    try:
        t0 = time.time()
        pa.prefill(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                   d["qsl"], pb.wl.scale)
        torch.cuda.synchronize()
        dt = time.time() - t0
    finally:
        pa.debug_prefill_fault(0)
    assert pa.take_device_error() == 2
    assert 1.0 < dt < 60.0, dt
    kc, vc = _oracle_caches(pb)
    ref = oracle.get().prefill(pb.q, kc, vc, pb.wl.block_tables, pb.wl.context_lens,
                               pb.query_start_loc, pb.wl.scale)
    out = pa.prefill(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                     d["qsl"], pb.wl.scale)
    torch.cuda.synchronize()
    gu.assert_close(out, ref, "after a timed-out launch")
