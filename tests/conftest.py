import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    import torch
    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def pa_lib():
    """libpagedattn built in-tree (nvcc cross-compiles without a GPU) and loaded."""
    from paged_kv_cache_255_gb300 import build, pagedattn
    build.build()
    return pagedattn.lib()


@pytest.fixture(autouse=True)
def _product_kernels_after_each_test():
    """Tests that select a comparison kernel (pa_debug_kernel_variant) leave
    the product kernels selected for the next test."""
    yield
    from paged_kv_cache_255_gb300 import pagedattn
    if pagedattn._lib is not None:
        pagedattn.debug_kernel_variant(0)
