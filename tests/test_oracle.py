"""The fp64 oracle against its pins (library routines, closed forms, and the
invariants the pages fix), plus its own argument checks. CPU only."""
import numpy as np
import pytest

import oracle
from paged_kv_cache_255_gb300 import inputs

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.get())


def test_threads_do_not_change_results():
    wl = inputs.generate(inputs.scaled(inputs.SPECS["large_batch"], num_seqs=8, ctx_div=8), seed=2)
    a, _, _ = pins.run_step(oracle.get(), wl, threads=1)
    b, _, _ = pins.run_step(oracle.get(), wl, threads=0)
    assert np.array_equal(a, b)


def test_pairs_match_full():
    wl = inputs.generate(inputs.SPECS["tiny"], seed=4)
    O = oracle.get()
    out, kc, vc = pins.run_step(O, wl)
    pairs = np.array([[0, 0], [3, 15], [2, 7], [1, 8]], dtype=np.int32)
    got = O.decode_pairs(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale, pairs)
    assert np.array_equal(got, out[pairs[:, 0], pairs[:, 1]])


def test_zero_length_is_zero():
    spec = inputs.Spec("z", ((3, 5, 40),), 8, 4, 16)
    wl = inputs.generate(spec, seed=1, context_lens=[0, 17, 0])
    out, _, _ = pins.run_step(oracle.get(), wl)
    assert np.all(out[0] == 0) and np.all(out[2] == 0) and np.isfinite(out[1]).all()


def test_rejects_bad_indices():
    wl = inputs.generate(inputs.SPECS["tiny"], seed=0)
    O = oracle.get()
    bad = wl.slot_mapping.copy()
    bad[0] = wl.num_blocks * wl.spec.block_size
    with pytest.raises(oracle.OracleError):
        O.store_kvcache(wl.k_new, wl.v_new, wl.k_cache, wl.v_cache, bad)
    bt = wl.block_tables.copy()
    bt[0, 0] = wl.num_blocks
    with pytest.raises(oracle.OracleError):
        O.decode(wl.q, wl.k_cache, wl.v_cache, bt, wl.context_lens, wl.scale)
