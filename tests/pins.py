"""Checks that tie the fp64 oracle to something other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with what the pages and the mathematics fix:

* a library routine: torch's fp64 scaled_dot_product_attention (with its
  grouped-query mode) over each sequence's contiguous K/V, which the input
  generator assembles from whole blocks without any per-token addressing;
  numpy's fancy-index assignment for the store;
* closed forms: one token (output = its V row exactly), all-zero keys
  (output = mean of the V rows), all-one values (output = 1), a hand-worked
  three-token case (softmax of 0, 1, 2), a dominant key (output ~ its V row);
* invariants the pages fix: renumbering physical blocks, sharing prefix
  blocks vs private copies, the block size, and NaN in every block no
  sequence owns (the null block among them) leave the output unchanged.

The same functions run against copies of the oracle with planted mistakes
(test_oracle_mutants.py) to show that each mistake fails at least one pin.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch
import torch.nn.functional as F

from paged_kv_cache_255_gb300 import inputs

BF16 = torch.bfloat16


def run_step(O, wl, threads=0):
    """Oracle store (if the step has one) then decode; returns (out, kc, vc)."""
    kc, vc = wl.k_cache, wl.v_cache
    if wl.slot_mapping.shape[0]:
        kc, vc = O.store_kvcache(wl.k_new, wl.v_new, kc, vc, wl.slot_mapping)
    out = O.decode(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale, threads=threads)
    return out, kc, vc


def sdpa_reference(wl):
    """Per-sequence fp64 SDPA over the generator's contiguous K/V (after the store)."""
    s = wl.spec
    outs = np.zeros((wl.num_seqs, s.num_q_heads, s.head_dim))
    for i in range(wl.num_seqs):
        L = int(wl.context_lens[i])
        if L == 0:
            continue
        k, v = wl.logical_kv(i)
        q = wl.q[i].cpu().double()[None, :, None, :]          # [1, Hq, 1, D]
        kk = k.double().permute(1, 0, 2)[None]                 # [1, Hkv, L, D]
        vv = v.double().permute(1, 0, 2)[None]
        o = F.scaled_dot_product_attention(q, kk, vv, scale=wl.scale, enable_gqa=True)
        outs[i] = o[0, :, 0, :].numpy()
    return outs


def _small_specs():
    S = inputs.SPECS
    return [
        S["tiny"],
        inputs.scaled(S["large_batch"], num_seqs=6, ctx_div=16, name="large_small"),
        inputs.scaled(S["prefix_shared"], num_seqs=5, ctx_div=16, name="prefix_small",
                      store_mode="none", store_rows=0, pad_rows=0),
        inputs.scaled(S["qwen3_0_6b_bs256"], num_seqs=4, ctx_div=1, name="bs256_small"),
        inputs.Spec("mha", ((3, 1, 70),), 4, 4, 16),              # g = 1
        inputs.Spec("g16", ((2, 20, 90),), 16, 1, 32),            # one KV head
    ]


def pin_sdpa(O, seed=0):
    for spec in _small_specs():
        wl = inputs.generate(spec, seed=seed, keep_content=True)
        out, _, _ = run_step(O, wl)
        ref = sdpa_reference(wl)
        err = np.abs(out - ref).max()
        assert err <= 1e-10, f"{spec.name}: oracle vs fp64 SDPA max err {err}"


def pin_single_token(O):
    spec = inputs.Spec("one", ((5, 1, 1),), 8, 2, 16)
    wl = inputs.generate(spec, seed=3, keep_content=True)
    out, _, _ = run_step(O, wl)
    g = spec.num_q_heads // spec.num_kv_heads
    for i in range(wl.num_seqs):
        _, v = wl.logical_kv(i)
        for h in range(spec.num_q_heads):
            want = v[0, h // g].double().numpy()
            assert np.array_equal(out[i, h], want), f"L=1 seq {i} head {h}"


def _with_values(wl, k_fill=None, v_fill=None):
    """Copy of ``wl`` whose K (V) rows are all ``k_fill`` (``v_fill``), NaN
    rows left NaN."""
    kc, vc, kn, vn = wl.k_cache.clone(), wl.v_cache.clone(), wl.k_new.clone(), wl.v_new.clone()
    if k_fill is not None:
        kc[~torch.isnan(kc)] = k_fill
        kn.fill_(k_fill)
    if v_fill is not None:
        vc[~torch.isnan(vc)] = v_fill
        vn.fill_(v_fill)
    ck = wl.content_k.clone() if k_fill is None else torch.full_like(wl.content_k, k_fill)
    cv = wl.content_v.clone() if v_fill is None else torch.full_like(wl.content_v, v_fill)
    return dataclasses.replace(wl, k_cache=kc, v_cache=vc, k_new=kn, v_new=vn,
                               content_k=ck, content_v=cv)


def pin_zero_keys(O):
    wl = inputs.generate(inputs.SPECS["tiny"], seed=5, keep_content=True)
    wl = _with_values(wl, k_fill=0.0)
    out, _, _ = run_step(O, wl)
    g = wl.spec.num_q_heads // wl.spec.num_kv_heads
    for i in range(wl.num_seqs):
        _, v = wl.logical_kv(i)
        mean = v.double().numpy().mean(axis=0)               # [Hkv, D]
        for h in range(wl.spec.num_q_heads):
            err = np.abs(out[i, h] - mean[h // g]).max()
            assert err <= 1e-12, f"K=0 seq {i} head {h}: {err}"


def pin_unit_values(O):
    spec = inputs.scaled(inputs.SPECS["large_batch"], num_seqs=4, ctx_div=8, name="ones")
    wl = inputs.generate(spec, seed=6, keep_content=True)
    wl = _with_values(wl, v_fill=1.0)
    out, _, _ = run_step(O, wl)
    assert np.abs(out - 1.0).max() <= 1e-13


def pin_three_tokens(O):
    """softmax(0, 1, 2) by hand: one head, D = 2, block size 2, scale 1/2,
    three tokens in physical blocks 3 then 1 (blocks 0 and 2 hold NaN)."""
    nan = float("nan")
    D, bs, NB = 2, 2, 4
    kc = torch.full((NB, bs, 1, D), nan)
    vc = torch.full((NB, bs, 1, D), nan)
    # logical token t has key (2t, 0): with q = (1, 0) and scale 1/2 its score is t
    kc[3, 0, 0] = torch.tensor([0.0, 0.0]); vc[3, 0, 0] = torch.tensor([1.0, 0.0])
    kc[3, 1, 0] = torch.tensor([2.0, 0.0]); vc[3, 1, 0] = torch.tensor([0.0, 1.0])
    kc[1, 0, 0] = torch.tensor([4.0, 0.0]); vc[1, 0, 0] = torch.tensor([0.0, 0.0])
    q = torch.tensor([[[1.0, 0.0]]])
    bt = np.array([[3, 1]], dtype=np.int32)
    out = O.decode(q.to(BF16), kc.to(BF16), vc.to(BF16), bt, np.array([3], np.int32), 0.5)
    z = 1.0 + math.e + math.e ** 2
    want = np.array([1.0 / z, math.e / z])      # weights of tokens 0 and 1
    assert np.abs(out[0, 0] - want).max() <= 1e-15, (out, want)


def pin_dominant_key(O):
    wl = inputs.generate(inputs.SPECS["tiny"], seed=7, keep_content=True)
    q = wl.q.clone()
    g = wl.spec.num_q_heads // wl.spec.num_kv_heads
    targets = []
    for i in range(wl.num_seqs):
        k, _ = wl.logical_kv(i)
        j = int(wl.context_lens[i]) // 2
        targets.append(j)
        for h in range(wl.spec.num_q_heads):
            q[i, h] = (k[j, h // g].float() * 4.0).to(BF16)   # |q.k_j| dominates every other score
    wl = dataclasses.replace(wl, q=q)
    out, _, _ = run_step(O, wl)
    for i in range(wl.num_seqs):
        _, v = wl.logical_kv(i)
        for h in range(wl.spec.num_q_heads):
            want = v[targets[i], h // g].double().numpy()
            assert np.abs(out[i, h] - want).max() <= 1e-6, f"dominant key seq {i} head {h}"


def _renumber(wl, seed):
    """Move every owned block to a new physical id and rewrite the tables."""
    rng = np.random.Generator(np.random.PCG64(seed))
    NB = wl.num_blocks
    perm = np.zeros(NB, dtype=np.int64)          # perm[old] = new; 0 stays 0
    perm[1:] = 1 + rng.permutation(NB - 1)
    kc = torch.empty_like(wl.k_cache)
    vc = torch.empty_like(wl.v_cache)
    kc[torch.from_numpy(perm)] = wl.k_cache
    vc[torch.from_numpy(perm)] = wl.v_cache
    bt = perm[wl.block_tables].astype(np.int32)
    sm = wl.slot_mapping.copy()
    bs = wl.spec.block_size
    ok = sm >= 0
    sm[ok] = perm[sm[ok] // bs] * bs + sm[ok] % bs
    return dataclasses.replace(wl, k_cache=kc, v_cache=vc, block_tables=bt, slot_mapping=sm)


def pin_renumbering(O):
    for spec in (inputs.SPECS["tiny"],
                 inputs.scaled(inputs.SPECS["prefix_shared"], num_seqs=4, ctx_div=16,
                               name="prefix_small")):
        wl = inputs.generate(spec, seed=11)
        a, _, _ = run_step(O, wl)
        b, _, _ = run_step(O, _renumber(wl, seed=12))
        assert np.array_equal(a, b), f"{spec.name}: renumbering changed the output"


def pin_prefix_private(O):
    spec = inputs.scaled(inputs.SPECS["prefix_shared"], num_seqs=4, ctx_div=16,
                         name="prefix_small", store_mode="none", store_rows=0, pad_rows=0)
    wl = inputs.generate(spec, seed=13)
    shared, _, _ = run_step(O, wl)
    # give every sequence private copies of the prefix blocks
    pb = spec.prefix_blocks
    S = wl.num_seqs
    NB2 = wl.num_blocks + S * pb
    kc = torch.full((NB2,) + tuple(wl.k_cache.shape[1:]), float("nan"), dtype=BF16)
    vc = torch.full_like(kc, float("nan"))
    kc[:wl.num_blocks] = wl.k_cache
    vc[:wl.num_blocks] = wl.v_cache
    bt = wl.block_tables.copy()
    nxt = wl.num_blocks
    for i in range(S):
        for j in range(pb):
            kc[nxt] = wl.k_cache[bt[i, j]]
            vc[nxt] = wl.v_cache[bt[i, j]]
            bt[i, j] = nxt
            nxt += 1
    private = O.decode(wl.q, kc, vc, bt, wl.context_lens, wl.scale)
    assert np.array_equal(shared, private), "private prefix copies changed the output"


def pin_block_size(O):
    """The same logical K/V in 16-token and 256-token blocks."""
    a_spec = inputs.Spec("bs16", ((4, 100, 700),), 16, 8, 16)
    wa = inputs.generate(a_spec, seed=21, keep_content=True)
    outs = []
    for bs in (16, 256):
        S = wa.num_seqs
        L = wa.context_lens
        nbs = [-(-int(x) // bs) for x in L]
        NB = 1 + sum(nbs)
        shape = (NB, bs) + tuple(wa.k_cache.shape[2:])
        kc = torch.full(shape, float("nan"), dtype=BF16)
        vc = torch.full(shape, float("nan"), dtype=BF16)
        bt = np.zeros((S, max(nbs)), np.int32)
        nxt = NB - 1          # fill from the top down so ids differ from the 16-token pool
        for i in range(S):
            k, v = wa.logical_kv(i)
            for j in range(nbs[i]):
                rows = k[j * bs:(j + 1) * bs]
                kc[nxt, :rows.shape[0]] = rows
                vc[nxt, :rows.shape[0]] = v[j * bs:(j + 1) * bs]
                bt[i, j] = nxt
                nxt -= 1
        outs.append(O.decode(wa.q, kc, vc, bt, L, wa.scale))
    assert np.abs(outs[0] - outs[1]).max() <= 1e-13, "block size changed the output"


def pin_nan_free(O):
    for spec in (inputs.SPECS["tiny"],
                 inputs.scaled(inputs.SPECS["large_batch"], num_seqs=8, ctx_div=8, name="lb")):
        wl = inputs.generate(spec, seed=17)
        assert torch.isnan(wl.k_cache[0].float()).all(), "null block must be poisoned"
        out, _, _ = run_step(O, wl)
        assert np.isfinite(out).all(), f"{spec.name}: output touched a poisoned row"


def pin_store(O):
    for spec in (inputs.SPECS["tiny"],
                 inputs.scaled(inputs.SPECS["prefix_shared"], num_seqs=8, ctx_div=4,
                               name="ps_store")):
        wl = inputs.generate(spec, seed=19)
        kc, vc = O.store_kvcache(wl.k_new, wl.v_new, wl.k_cache, wl.v_cache, wl.slot_mapping)
        NB, bs, Hkv, D = wl.k_cache.shape
        sm = wl.slot_mapping
        ok = sm >= 0
        for new, cache, got in ((wl.k_new, wl.k_cache, kc), (wl.v_new, wl.v_cache, vc)):
            want = cache.view(torch.int16).numpy().view(np.uint16).reshape(NB * bs, Hkv * D).copy()
            src = new.view(torch.int16).numpy().view(np.uint16).reshape(-1, Hkv * D)
            want[sm[ok]] = src[ok]                       # numpy scatter, -1 rows dropped
            assert np.array_equal(got.reshape(NB * bs, Hkv * D), want), f"{spec.name}: store"


def _multi_workload(spec, seed, Q):
    """A decode step with Q new query tokens per sequence (q: [S, Q, Hq, D])."""
    wl = inputs.generate(spec, seed=seed, keep_content=True)
    g = torch.Generator().manual_seed(seed)
    S, Hq, D = wl.q.shape
    q = torch.randn((S, Q, Hq, D), generator=g).to(BF16)
    return wl, q


def pin_multi_sdpa(O):
    """Q new tokens per sequence against torch's fp64 SDPA with an explicit
    causal mask: token i sees keys t <= L - Q + i."""
    for spec, Q in ((inputs.SPECS["tiny"], 3),
                    (inputs.scaled(inputs.SPECS["large_batch"], num_seqs=5, ctx_div=16), 4),
                    (inputs.Spec("mq", ((4, 1, 40),), 8, 2, 16), 2)):
        wl, q = _multi_workload(spec, 31, Q)
        kc, vc = wl.k_cache, wl.v_cache
        if wl.slot_mapping.shape[0]:
            kc, vc = O.store_kvcache(wl.k_new, wl.v_new, kc, vc, wl.slot_mapping)
        out = O.decode_multi(q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
        for i in range(wl.num_seqs):
            L = int(wl.context_lens[i])
            if L == 0:
                assert np.all(out[i] == 0)
                continue
            k, v = wl.logical_kv(i)
            qq = q[i].double().permute(1, 0, 2)[None]          # [1, Hq, Q, D]
            kk = k.double().permute(1, 0, 2)[None]
            vv = v.double().permute(1, 0, 2)[None]
            pos = torch.arange(L)[None, :]
            lim = (L - Q + torch.arange(Q))[:, None]
            mask = pos <= lim                                  # [Q, L]
            ref = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=wl.scale,
                                                 enable_gqa=True)[0].permute(1, 0, 2).numpy()
            seen = (lim[:, 0] >= 0).numpy()
            err = np.abs(out[i][seen] - np.nan_to_num(ref[seen])).max() if seen.any() else 0.0
            assert err <= 1e-10, f"{spec.name}: multi-token vs SDPA max err {err}"
            assert np.all(out[i][~seen] == 0)


def pin_multi_prefix(O):
    """Query token i of Q equals a single-token decode of the same query row
    over the sequence cut to its first L - Q + i + 1 tokens."""
    spec = inputs.scaled(inputs.SPECS["qwen3_0_6b"], num_seqs=4, ctx_div=8)
    Q = 3
    wl, q = _multi_workload(spec, 32, Q)
    kc, vc = O.store_kvcache(wl.k_new, wl.v_new, wl.k_cache, wl.v_cache, wl.slot_mapping)
    out = O.decode_multi(q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
    for i in range(Q):
        cut = np.maximum(wl.context_lens - Q + i + 1, 0).astype(np.int32)
        single = O.decode(q[:, i].contiguous(), kc, vc, wl.block_tables, cut, wl.scale)
        assert np.array_equal(out[:, i], single), f"query token {i}"


def _head_major(pool):
    return pool.permute(0, 2, 1, 3).contiguous()


def pin_head_major(O):
    """The head-major pool [NB, Hkv, bs, D] is the token-major one with two
    axes swapped: its store and decode give the same values, bit for bit."""
    for spec in (inputs.SPECS["tiny"],
                 inputs.scaled(inputs.SPECS["prefix_shared"], num_seqs=6, ctx_div=8, name="ps")):
        wl = inputs.generate(spec, seed=51)
        kc, vc = O.store_kvcache(wl.k_new, wl.v_new, wl.k_cache, wl.v_cache, wl.slot_mapping)
        hk, hv = O.store_kvcache_head_major(wl.k_new, wl.v_new, _head_major(wl.k_cache),
                                            _head_major(wl.v_cache), wl.slot_mapping)
        assert np.array_equal(hk, np.ascontiguousarray(kc.transpose(0, 2, 1, 3))), "head-major store"
        assert np.array_equal(hv, np.ascontiguousarray(vc.transpose(0, 2, 1, 3))), "head-major store"
        a = O.decode(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale)
        b = O.decode_head_major(wl.q, hk, hv, wl.block_tables, wl.context_lens, wl.scale)
        assert np.array_equal(a, b), "head-major decode"


def _prefill_case(seed, lens, chunks, Hq=8, Hkv=2, bs=16):
    """A pool holding len(lens) sequences and a packed query block of
    chunks[s] <= lens[s] new tokens per sequence."""
    spec = inputs.Spec("pf", ((len(lens), 1, 1),), Hq, Hkv, bs, store_mode="none")
    wl = inputs.generate(spec, seed=seed, keep_content=True, context_lens=lens)
    qsl = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((int(qsl[-1]), Hq, 128), generator=g).to(BF16)
    return wl, q, qsl


def pin_prefill_sdpa(O):
    """Prefill rows against torch's fp64 SDPA with an explicit causal mask."""
    lens, chunks = [37, 200, 16, 129, 5], [37, 64, 1, 100, 5]
    wl, q, qsl = _prefill_case(71, lens, chunks)
    out = O.prefill(q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, qsl, wl.scale)
    for s in range(len(lens)):
        L, n = lens[s], chunks[s]
        k, v = wl.logical_kv(s, after_store=False)
        qq = q[qsl[s]:qsl[s + 1]].double().permute(1, 0, 2)[None]      # [1, Hq, n, D]
        kk = k.double().permute(1, 0, 2)[None]
        vv = v.double().permute(1, 0, 2)[None]
        mask = torch.arange(L)[None, :] <= (L - n + torch.arange(n))[:, None]
        ref = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=wl.scale,
                                             enable_gqa=True)[0].permute(1, 0, 2).numpy()
        err = np.abs(out[qsl[s]:qsl[s + 1]] - ref).max()
        assert err <= 1e-10, f"prefill seq {s}: max err {err}"


def pin_prefill_is_multi_token(O):
    """With the same number Q of new tokens in every sequence, prefill is the
    multi-token decode of the same rows."""
    lens, Q = [40, 90, 17, 33], 4
    wl, q, qsl = _prefill_case(72, lens, [Q] * len(lens))
    a = O.prefill(q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, qsl, wl.scale)
    b = O.decode_multi(q.view(len(lens), Q, *q.shape[1:]), wl.k_cache, wl.v_cache,
                       wl.block_tables, wl.context_lens, wl.scale)
    assert np.array_equal(a, b.reshape(a.shape))


def pin_pairs_sdpa(O):
    """decode_pairs (the sampled outputs the full-size GPU checks use) on a
    shuffled list of (sequence, head) pairs with repeats: each output is that
    row of fp64 SDPA over the sequence's contiguous K/V."""
    spec = inputs.scaled(inputs.SPECS["large_batch"], num_seqs=6, ctx_div=16, name="pairs_small")
    wl = inputs.generate(spec, seed=4, keep_content=True)
    _, kc, vc = run_step(O, wl)
    ref = sdpa_reference(wl)
    rng = np.random.Generator(np.random.PCG64(8))
    S, Hq = wl.num_seqs, spec.num_q_heads
    pairs = np.stack([rng.integers(0, S, 40), rng.integers(0, Hq, 40)], axis=1).astype(np.int32)
    got = O.decode_pairs(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale, pairs)
    err = np.abs(got - ref[pairs[:, 0], pairs[:, 1]]).max()
    assert err <= 1e-10, f"decode_pairs vs fp64 SDPA max err {err}"


ALL_PINS = [pin_sdpa, pin_single_token, pin_zero_keys, pin_unit_values, pin_three_tokens,
            pin_dominant_key, pin_renumbering, pin_prefix_private, pin_block_size,
            pin_nan_free, pin_store, pin_multi_sdpa, pin_multi_prefix, pin_head_major,
            pin_prefill_sdpa, pin_prefill_is_multi_token, pin_pairs_sdpa]
