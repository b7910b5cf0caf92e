"""Host-side choices of bench.py that decide what its numbers mean (no GPU):
which decode steps run back to back (inputs larger than L2) and which get the
L2 flush before each step, and the config note that says so."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from paged_kv_cache_255_gb300 import inputs  # noqa: E402


class _Step:
    """Stands in for a generated workload: only its byte counts matter here."""

    def __init__(self, unique, logical=None):
        self._u, self._l = unique, unique if logical is None else logical

    def unique_kv_bytes(self):
        return self._u

    def kv_bytes(self):
        return self._l


def test_back_to_back_from_eight_times_the_l2():
    edge = bench.LARGE_INPUT_FACTOR * bench.L2_BYTES
    assert bench.large_inputs(_Step(edge))
    assert not bench.large_inputs(_Step(edge - 1))
    assert bench.l2_note(_Step(edge - 1)) == bench.L2_FLUSHED
    assert bench.l2_note(_Step(edge)).startswith("not flushed: inputs larger than L2")


def test_shared_prefix_counts_once():
    # the prefix-shared step reads 1.2 GB logically but only 143 MB of distinct
    # rows: L2 serves the prefix, so it must be flushed, not run back to back
    step = _Step(unique=142_606_336, logical=1_207_959_552)
    assert not bench.large_inputs(step)
    assert bench.l2_note(step) == bench.L2_FLUSHED


def test_small_generated_step_is_flushed():
    # the tiny step (2.8 MB of K/V) through the generator and the config
    wl = inputs.generate(inputs.SPECS["tiny"], seed=0, device="cpu")
    assert not bench.large_inputs(wl)
    assert bench.workload_config(wl)["l2"] == bench.L2_FLUSHED
    # the flush buffer stays larger than twice the L2 it replaces
    assert bench.L2_FLUSH_BYTES > 2 * bench.L2_BYTES
