"""Structure of the synthetic decode steps (no values drawn for the big ones)."""
import numpy as np
import pytest
import torch

from paged_kv_cache_255_gb300 import inputs


def _live_entries(wl):
    bs = wl.spec.block_size
    for i, L in enumerate(wl.context_lens):
        for j in range(-(-int(L) // bs)):
            yield i, j, int(wl.block_tables[i, j])


@pytest.mark.parametrize("name", sorted(inputs.SPECS))
def test_structure(name):
    spec = inputs.SPECS[name]
    wl = inputs.generate(spec, seed=0, values=False)
    assert wl.num_seqs == spec.num_seqs
    lo = min(g[1] for g in spec.ctx_groups)
    hi = max(g[2] for g in spec.ctx_groups)
    assert wl.context_lens.min() >= lo and wl.context_lens.max() <= hi
    ids = np.array([b for _, _, b in _live_entries(wl)])
    # the null block is never handed out, every id is inside the pool
    assert ids.min() >= 1 and ids.max() < wl.num_blocks
    if spec.pool_mode != "prefix_shared":
        assert len(np.unique(ids)) == len(ids), "private blocks must not repeat"
    sm = wl.slot_mapping
    ok = sm[sm >= 0]
    assert len(np.unique(ok)) == len(ok), "store slots must be distinct"
    assert ok.max(initial=0) < wl.num_blocks * spec.block_size


def test_fragmented_pool_uses_odd_blocks():
    wl = inputs.generate(inputs.SPECS["large_batch"], values=False)
    ids = np.array([b for _, _, b in _live_entries(wl)])
    assert np.all(ids % 2 == 1)
    assert wl.num_blocks == 2 * len(ids) + 1


def test_prefix_shared_tables():
    spec = inputs.SPECS["prefix_shared"]
    wl = inputs.generate(spec, values=False)
    bt = wl.block_tables
    assert np.all(wl.context_lens == 2304)
    assert np.all(bt[:, :128] == bt[0, :128]), "every sequence shares the 128 prefix blocks"
    uniq = bt[:, 128:144].reshape(-1)
    assert len(np.unique(uniq)) == uniq.size and not np.isin(uniq, bt[0, :128]).any()
    sm = wl.slot_mapping
    assert sm.shape == (4096,) and int((sm == -1).sum()) == 410
    blocks = sm[sm >= 0] // spec.block_size
    assert np.isin(blocks, uniq).all(), "stores only go to unique blocks"


def test_tiny_pool_and_poison():
    wl = inputs.generate(inputs.SPECS["tiny"], seed=0)
    assert wl.num_blocks == 128
    assert torch.isnan(wl.k_cache[0].float()).all() and torch.isnan(wl.v_cache[0].float()).all()
    free = np.setdiff1d(np.arange(1, 128), wl.owned_blocks)
    assert torch.isnan(wl.k_cache[torch.from_numpy(free)].float()).all()
    # the row each last-token store writes is poisoned until the store runs
    flat = wl.k_cache.view(-1, 8, 128)
    assert torch.isnan(flat[torch.from_numpy(wl.slot_mapping)].float()).all()


def test_seed_determinism():
    a = inputs.generate(inputs.SPECS["tiny"], seed=9)
    b = inputs.generate(inputs.SPECS["tiny"], seed=9)
    assert np.array_equal(a.block_tables, b.block_tables)
    assert torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))
    assert torch.equal(a.k_cache.view(torch.int16), b.k_cache.view(torch.int16))
