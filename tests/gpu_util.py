"""Helpers for the GPU parity tests: run a synthetic decode step through the
C ABI (via the ctypes binding) and compare it with the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

from paged_kv_cache_255_gb300 import pagedattn as pa

# bf16 output vs fp64 oracle: |gpu - ref| <= ATOL + RTOL * |ref|, element-wise
ATOL = 2e-2
RTOL = 2e-2


def device_inputs(wl, dev="cuda"):
    """Device copies of a workload (caches cloned: the store writes them)."""
    d = dict(
        q=wl.q.to(dev).contiguous(),
        k_cache=wl.k_cache.to(dev).clone(),
        v_cache=wl.v_cache.to(dev).clone(),
        k_new=wl.k_new.to(dev).contiguous(),
        v_new=wl.v_new.to(dev).contiguous(),
        slot_mapping=torch.from_numpy(wl.slot_mapping).to(dev),
        block_tables=torch.from_numpy(wl.block_tables).to(dev),
        context_lens=torch.from_numpy(wl.context_lens).to(dev),
    )
    return d


def gpu_step(wl, num_partitions=0, d=None):
    """Store (if any) then decode on the GPU; returns (out, k_cache, v_cache)."""
    if d is None:
        d = device_inputs(wl)
    if wl.slot_mapping.shape[0]:
        pa.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slot_mapping"])
    out = pa.decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                    wl.scale, num_partitions=num_partitions)
    torch.cuda.synchronize()
    return out, d["k_cache"], d["v_cache"]


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_close(gpu_out: torch.Tensor, ref: np.ndarray, what: str = ""):
    got = gpu_out.detach().float().cpu().double().numpy()
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; first at "
                             f"{tuple(idx)}: gpu {got[tuple(idx)]} ref {ref[tuple(idx)]}; "
                             f"max err {err.max()}")
    return float(err.max())
