"""libpagedattn: paged KV-cache store and single-token decode attention for GB300.

The compute lives in CUDA kernels behind the C ABI of ``include/pagedattn.h``;
``pagedattn`` binds it for torch tensors. ``inputs`` draws seeded synthetic
decode steps. Importing the package does not load the shared library; the
first call does, and raises if it has not been built (``build.build()``).
"""
from .pagedattn import (  # noqa: F401
    PagedAttnError,
    decode,
    decode_workspace_size,
    lib,
    status_string,
    store_kvcache,
    workspace_for,
)
