"""Out-of-range indices on the device, through the C ABI. The kernels must
neither fault nor read outside the pool: a store slot outside the pool is
skipped, and a block-table entry outside the pool reads as zero rows. Each
case is reported by pa_take_device_error (codes 3 and 4), and the outputs
match the oracle run on the defined behaviour (the bad row left out, or the
entry pointed at an all-zero block)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_255_gb300 import inputs
from paged_kv_cache_255_gb300 import pagedattn as pa

import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(pa_lib):
    return pa_lib


@pytest.fixture(autouse=True)
def _clean_error_record():
    pa.take_device_error()
    yield
    assert pa.take_device_error() == 0, "a test left a device error behind"


def _with_zero_block(t):
    """The pool with one all-zero block appended (its id is the old block count)."""
    return torch.cat([t, torch.zeros_like(t[:1])])


def test_store_skips_out_of_range_slots_and_reports():
    wl = inputs.generate(inputs.SPECS["tiny"], seed=5)
    d = gu.device_inputs(wl)
    # padding alone (-1) is not an error
    pad = np.full_like(wl.slot_mapping, -1)
    pa.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], torch.from_numpy(pad).cuda())
    torch.cuda.synchronize()
    assert pa.take_device_error() == 0
    sm = wl.slot_mapping.copy()
    sm[0] = wl.num_blocks * wl.spec.block_size + 7      # past the pool
    sm[1] = -3                                            # negative, not padding
    pa.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], torch.from_numpy(sm).cuda())
    torch.cuda.synchronize()
    assert pa.take_device_error() == 3
    ref_sm = sm.copy()
    ref_sm[:2] = -1
    kc, vc = oracle.get().store_kvcache(wl.k_new, wl.v_new, wl.k_cache, wl.v_cache, ref_sm)
    assert np.array_equal(gu.host_bits(d["k_cache"]), kc)
    assert np.array_equal(gu.host_bits(d["v_cache"]), vc)


def _decode_case(seed):
    spec = inputs.Spec("bad_block", ((6, 40, 300),), 16, 8, 16, store_mode="none")
    wl = inputs.generate(spec, seed=seed)
    bs = spec.block_size
    nb = (wl.context_lens.astype(np.int64) + bs - 1) // bs
    s = int(np.argmax(nb >= 3))
    assert nb[s] >= 3
    return wl, s, nb


@pytest.mark.parametrize("kernel", ["mma", "simt"])
def test_decode_reads_out_of_range_block_as_zeros_and_reports(kernel, monkeypatch):
    gu.decode_kernel(kernel)
    wl, s, nb = _decode_case(9)
    bt = wl.block_tables.copy()
    bt[s, 1] = wl.num_blocks + 11                        # a live entry, outside the pool
    bt_ref = bt.copy()
    bt_ref[s, 1] = wl.num_blocks                         # the appended zero block
    ref = oracle.get().decode(wl.q, _with_zero_block(wl.k_cache), _with_zero_block(wl.v_cache),
                              bt_ref, wl.context_lens, wl.scale)
    d = gu.device_inputs(wl)
    out = pa.decode(d["q"], d["k_cache"], d["v_cache"], torch.from_numpy(bt).cuda(),
                    d["context_lens"], wl.scale)
    torch.cuda.synchronize()
    assert pa.take_device_error() == 4
    gu.assert_close(out, ref, f"bad block ({kernel})")


def test_decode_never_reads_entries_past_the_last_block():
    wl, _, nb = _decode_case(10)
    bt = wl.block_tables.copy()
    for s in range(bt.shape[0]):
        bt[s, nb[s]:] = wl.num_blocks + 1000 + s         # padding entries far outside the pool
    d = gu.device_inputs(wl)
    a = pa.decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                  wl.scale, num_partitions=13)
    b = pa.decode(d["q"], d["k_cache"], d["v_cache"], torch.from_numpy(bt).cuda(),
                  d["context_lens"], wl.scale, num_partitions=13)
    torch.cuda.synchronize()
    assert pa.take_device_error() == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("kernel", ["mma", "simt"])
def test_decode_clamps_lengths_to_the_table(kernel):
    """A length below zero or past what its block-table row can hold is
    clamped to [0, max_blocks_per_seq * block_size], as the header states: a
    negative length gives a zero output, and a sequence whose row is full,
    given 1000 tokens more than the row holds, reads exactly its row. Nothing
    is recorded (clamping is defined behaviour, not an error)."""
    gu.decode_kernel(kernel)
    spec = inputs.Spec("clamp", ((4, 1, 1),), 16, 8, 16, store_mode="none")
    wl = inputs.generate(spec, seed=21, context_lens=[320, 100, 37, 250])
    cap = wl.block_tables.shape[1] * spec.block_size
    assert cap == 320                                    # sequence 0 fills its row
    ref = oracle.get().decode(wl.q, wl.k_cache, wl.v_cache, wl.block_tables,
                              np.array([320, 0, 37, 250], np.int32), wl.scale)
    d = gu.device_inputs(wl)
    cl = torch.tensor([cap + 1000, -5, 37, 250], dtype=torch.int32, device="cuda")
    out = pa.decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], cl, wl.scale)
    torch.cuda.synchronize()
    assert pa.take_device_error() == 0
    gu.assert_close(out, ref, f"clamped lengths ({kernel})")
    assert torch.count_nonzero(out[1]).item() == 0


@pytest.mark.parametrize("kernel", ["tc", "mma"])
def test_prefill_reads_out_of_range_block_as_zeros_and_reports(kernel, monkeypatch):
    gu.prefill_kernel(kernel)
    spec = inputs.Spec("bad_pf", ((1, 1, 1),), 16, 8, 16, store_mode="none")
    pb = inputs.prefill_batch(spec, seed=3, context_lens=[300, 90], chunk_lens=[100, 90])
    O = oracle.get()
    kc, vc = O.store_kvcache(pb.k_new, pb.v_new, pb.wl.k_cache, pb.wl.v_cache, pb.slot_mapping)
    bt = pb.wl.block_tables.copy()
    bt[0, 2] = pb.wl.num_blocks + 5                      # a context block of sequence 0
    bt_ref = bt.copy()
    bt_ref[0, 2] = pb.wl.num_blocks
    zero = np.zeros_like(kc[:1])
    ref = O.prefill(pb.q, np.concatenate([kc, zero]), np.concatenate([vc, zero]), bt_ref,
                    pb.wl.context_lens, pb.query_start_loc, pb.wl.scale)
    kd, vd = pb.wl.k_cache.cuda(), pb.wl.v_cache.cuda()
    pa.store_kvcache(pb.k_new.cuda(), pb.v_new.cuda(), kd, vd,
                     torch.from_numpy(pb.slot_mapping).cuda())
    out = pa.prefill(pb.q.cuda(), kd, vd, torch.from_numpy(bt).cuda(),
                     torch.from_numpy(pb.wl.context_lens).cuda(),
                     torch.from_numpy(pb.query_start_loc).cuda(), pb.wl.scale)
    torch.cuda.synchronize()
    assert pa.take_device_error() == 4
    gu.assert_close(out, ref, f"prefill bad block ({kernel})")
