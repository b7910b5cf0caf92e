"""Python binding of libpagedattn (ctypes): argument marshalling only.

Every function here checks tensor devices, dtypes and shapes, then calls the
C ABI declared in ``include/pagedattn.h`` with raw device pointers and the
current torch CUDA stream. All computation happens in the library's CUDA
kernels; there is no fallback. If the shared library has not been built, the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA = range(5)

# every entry point include/pagedattn.h declares, with its ctypes signature
_P, _I32, _I64, _F32, _SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                             ctypes.c_size_t)
SIGNATURES = {
    "pa_status_string": ([_I32], ctypes.c_char_p),
    "pa_store_kvcache": ([_P, _P, _P, _P, _P, _I64, _I32, _I32, _I32, _I64, _P], _I32),
    "pa_decode_workspace_size": ([_I32, _I32, _I32, _I32], _SZ),
    "pa_decode": ([_P, _P, _P, _P, _I32, _P, _F32, _P, _I32, _I32, _I32, _I32, _I32, _I64,
                   _P, _SZ, _P], _I32),
    "pa_decode_splitk": ([_P, _P, _P, _P, _I32, _P, _F32, _P, _I32, _I32, _I32, _I32, _I32,
                          _I64, _P, _SZ, _I32, _P], _I32),
    "pa_decode_noalloc": ([_P, _P, _P, _P, _I32, _P, _F32, _P, _I32, _I32, _I32, _I32, _I32,
                           _I64, _P], _I32),
    "pa_decode_multi_workspace_size": ([_I32, _I32, _I32, _I32], _SZ),
    "pa_prefill": ([_P, _P, _P, _P, _I32, _P, _P, _I32, _F32, _P, _I32, _I32, _I32, _I32, _I32,
                    _I32, _I64, _P], _I32),
    "pa_take_device_error": ([_P, _P], _I32),
    "pa_debug_prefill_fault": ([_I32], _I32),
    "pa_debug_kernel_variant": ([_I32], _I32),
    "pa_prefill_layout": ([_P, _P, _P, _P, _I32, _P, _P, _I32, _F32, _P, _I32, _I32, _I32, _I32,
                           _I32, _I32, _I64, _I32, _P], _I32),
    "pa_store_kvcache_layout": ([_P, _P, _P, _P, _P, _I64, _I32, _I32, _I32, _I64, _I32, _P],
                                _I32),
    "pa_decode_layout": ([_P, _P, _P, _P, _I32, _P, _F32, _P, _I32, _I32, _I32, _I32, _I32, _I64,
                          _I32, _P, _SZ, _I32, _P], _I32),
    "pa_decode_multi": ([_P, _P, _P, _P, _I32, _P, _I32, _F32, _P, _I32, _I32, _I32, _I32, _I32,
                         _I64, _P, _SZ, _P], _I32),
    "pa_decode_step": ([_P, _P, _P, _I64, _P, _P, _P, _P, _I32, _P, _F32, _P, _I32, _I32, _I32,
                        _I32, _I32, _I64, _I32, _P, _SZ, _P], _I32),
    "pa_decode_multi_layout": ([_P, _P, _P, _P, _I32, _P, _I32, _F32, _P, _I32, _I32, _I32, _I32,
                                _I32, _I64, _I32, _P, _SZ, _P], _I32),
}

_lock = threading.Lock()
_lib = None
_workspaces = {}


class PagedAttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")


def library_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded libpagedattn; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libpagedattn is not built ({path} missing): run "
                    "paged_kv_cache_255_gb300.build.build() first")
            handle = ctypes.CDLL(path)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.argtypes = args
                fn.restype = res
            _lib = handle
    return _lib


def status_string(status: int) -> str:
    return lib().pa_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != PA_OK:
        raise PagedAttnError(fn, status)


def _stream_ptr(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream)


def _cuda(t: torch.Tensor, name: str, dtype, device=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def store_kvcache(k, v, k_cache, v_cache, slot_mapping, stream=None, head_major=False):
    """Write row i of k/v to cache slot slot_mapping[i] (-1 rows skipped).

    k, v: bf16 [N, Hkv, D]; k_cache, v_cache: bf16 [NB, bs, Hkv, D], or
    [NB, Hkv, bs, D] with ``head_major``; slot_mapping: int64 [N]. Runs on the
    current stream (or ``stream``).
    """
    dev = k_cache.device
    for t, n, dt in ((k, "k", torch.bfloat16), (v, "v", torch.bfloat16),
                     (k_cache, "k_cache", torch.bfloat16), (v_cache, "v_cache", torch.bfloat16),
                     (slot_mapping, "slot_mapping", torch.int64)):
        _cuda(t, n, dt, dev)
    if head_major:
        NB, Hkv, bs, D = k_cache.shape
    else:
        NB, bs, Hkv, D = k_cache.shape
    N = slot_mapping.shape[0]
    if v_cache.shape != k_cache.shape or k.shape != (N, Hkv, D) or v.shape != (N, Hkv, D):
        raise ValueError("shape mismatch between k, v, caches and slot_mapping")
    with torch.cuda.device(dev):
        st = lib().pa_store_kvcache_layout(k.data_ptr(), v.data_ptr(), k_cache.data_ptr(),
                                           v_cache.data_ptr(), slot_mapping.data_ptr(), N, Hkv,
                                           D, bs, NB, 1 if head_major else 0,
                                           _stream_ptr(stream, dev))
    _check("pa_store_kvcache", st)


def decode_step(k_new, v_new, slot_mapping, q, k_cache, v_cache, block_tables, context_lens,
                scale, out=None, workspace=None, stream=None, head_major=False):
    """One decode step through pa_decode_step: store the step's new K/V rows
    (``k_new``, ``v_new`` bf16 [N, Hkv, D] at ``slot_mapping`` int64 [N]),
    then single-token decode over the updated cache; returns ``out``. Same
    results as store_kvcache followed by decode; the decode plans its work
    split while the store runs."""
    dev = q.device
    for t, n, dt in ((k_new, "k_new", torch.bfloat16), (v_new, "v_new", torch.bfloat16),
                     (slot_mapping, "slot_mapping", torch.int64), (q, "q", torch.bfloat16),
                     (k_cache, "k_cache", torch.bfloat16), (v_cache, "v_cache", torch.bfloat16),
                     (block_tables, "block_tables", torch.int32),
                     (context_lens, "context_lens", torch.int32)):
        _cuda(t, n, dt, dev)
    S, Hq, D = q.shape
    if head_major:
        NB, Hkv, bs, D2 = k_cache.shape
    else:
        NB, bs, Hkv, D2 = k_cache.shape
    N = slot_mapping.shape[0]
    if v_cache.shape != k_cache.shape or D2 != D or block_tables.dim() != 2 \
            or block_tables.shape[0] != S or context_lens.shape != (S,) \
            or k_new.shape != (N, Hkv, D) or v_new.shape != (N, Hkv, D):
        raise ValueError("shape mismatch between the step's tensors")
    if out is None:
        out = torch.empty_like(q)
    else:
        _cuda(out, "out", torch.bfloat16, dev)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    if workspace is None:
        workspace = workspace_for(Hq, Hkv, D, 0, dev)
    else:
        _cuda(workspace, "workspace", workspace.dtype, dev)
    with torch.cuda.device(dev):
        st = lib().pa_decode_step(k_new.data_ptr(), v_new.data_ptr(), slot_mapping.data_ptr(), N,
                                  q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                  block_tables.data_ptr(), block_tables.shape[1],
                                  context_lens.data_ptr(), float(scale), out.data_ptr(), S, Hq,
                                  Hkv, D, bs, NB, 1 if head_major else 0, workspace.data_ptr(),
                                  workspace.numel() * workspace.element_size(),
                                  _stream_ptr(stream, dev))
    _check("pa_decode_step", st)
    return out


def decode_workspace_size(num_q_heads: int, num_kv_heads: int, head_dim: int = 128,
                          num_partitions: int = 0, device=None) -> int:
    """Workspace bytes pa_decode needs on ``device`` (default: current)."""
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        n = lib().pa_decode_workspace_size(num_q_heads, num_kv_heads, head_dim, num_partitions)
    if n == 0:
        raise ValueError("unsupported head configuration")
    return int(n)


def workspace_for(num_q_heads, num_kv_heads, head_dim=128, num_partitions=0, device=None):
    """A cached uint8 workspace tensor big enough for these heads on ``device``."""
    device = torch.device(device if device is not None else f"cuda:{torch.cuda.current_device()}")
    n = decode_workspace_size(num_q_heads, num_kv_heads, head_dim, num_partitions, device)
    key = (device, n)
    ws = _workspaces.get(key)
    if ws is None:
        ws = torch.empty(n, dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def decode(q, k_cache, v_cache, block_tables, context_lens, scale, out=None, workspace=None,
           num_partitions: int = 0, stream=None, head_major=False):
    """Single-token paged decode attention; returns ``out`` (bf16 [S, Hq, D]).

    q: bf16 [S, Hq, D]; caches: bf16 [NB, bs, Hkv, D] ([NB, Hkv, bs, D] with
    ``head_major``); block_tables: int32 [S, max_blocks]; context_lens: int32
    [S]. ``num_partitions`` > 0 forces the split-K share count
    (pa_decode_splitk).
    """
    dev = q.device
    for t, n, dt in ((q, "q", torch.bfloat16), (k_cache, "k_cache", torch.bfloat16),
                     (v_cache, "v_cache", torch.bfloat16), (block_tables, "block_tables", torch.int32),
                     (context_lens, "context_lens", torch.int32)):
        _cuda(t, n, dt, dev)
    S, Hq, D = q.shape
    if head_major:
        NB, Hkv, bs, D2 = k_cache.shape
    else:
        NB, bs, Hkv, D2 = k_cache.shape
    if v_cache.shape != k_cache.shape or D2 != D or block_tables.dim() != 2 \
            or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("shape mismatch between q, caches, block_tables and context_lens")
    if out is None:
        out = torch.empty_like(q)
    else:
        _cuda(out, "out", torch.bfloat16, dev)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    if workspace is None:
        workspace = workspace_for(Hq, Hkv, D, num_partitions, dev)
    else:
        _cuda(workspace, "workspace", workspace.dtype, dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    args = (q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
            block_tables.shape[1], context_lens.data_ptr(), float(scale), out.data_ptr(), S, Hq,
            Hkv, D, bs, NB, workspace.data_ptr(), ws_bytes)
    with torch.cuda.device(dev):
        if head_major:
            st = lib().pa_decode_layout(*args[:14], 1, *args[14:], int(num_partitions),
                                        _stream_ptr(stream, dev))
        elif num_partitions:
            st = lib().pa_decode_splitk(*args, int(num_partitions), _stream_ptr(stream, dev))
        else:
            st = lib().pa_decode(*args, _stream_ptr(stream, dev))
    _check("pa_decode", st)
    return out


def decode_multi(q, k_cache, v_cache, block_tables, context_lens, scale, out=None,
                 workspace=None, stream=None, head_major=False):
    """Decode of Q new tokens per sequence (speculative verification): q is
    bf16 [S, Q, Hq, D]; query token i attends to keys t <= L - Q + i, with
    L = context_lens[s] counting all Q new tokens. The pool is
    [NB, bs, Hkv, D], or [NB, Hkv, bs, D] with head_major=True. Returns out
    [S, Q, Hq, D]."""
    dev = q.device
    for t, n, dt in ((q, "q", torch.bfloat16), (k_cache, "k_cache", torch.bfloat16),
                     (v_cache, "v_cache", torch.bfloat16), (block_tables, "block_tables", torch.int32),
                     (context_lens, "context_lens", torch.int32)):
        _cuda(t, n, dt, dev)
    S, Q, Hq, D = q.shape
    if head_major:
        NB, Hkv, bs, D2 = k_cache.shape
    else:
        NB, bs, Hkv, D2 = k_cache.shape
    if v_cache.shape != k_cache.shape or D2 != D or block_tables.dim() != 2 \
            or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("shape mismatch between q, caches, block_tables and context_lens")
    if out is None:
        out = torch.empty_like(q)
    else:
        _cuda(out, "out", torch.bfloat16, dev)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    if workspace is None:
        with torch.cuda.device(dev):
            n = lib().pa_decode_multi_workspace_size(Q, Hq, Hkv, D)
        if n == 0:
            raise ValueError("unsupported query-token / head configuration")
        key = (dev, "multi", n)
        workspace = _workspaces.get(key)
        if workspace is None:
            workspace = torch.zeros(n, dtype=torch.uint8, device=dev)
            _workspaces[key] = workspace
    else:
        _cuda(workspace, "workspace", workspace.dtype, dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(dev):
        st = lib().pa_decode_multi_layout(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                          block_tables.data_ptr(), block_tables.shape[1],
                                          context_lens.data_ptr(), Q, float(scale),
                                          out.data_ptr(), S, Hq, Hkv, D, bs, NB,
                                          1 if head_major else 0,
                                          workspace.data_ptr(), ws_bytes, _stream_ptr(stream, dev))
    _check("pa_decode_multi_layout", st)
    return out


def prefill(q, k_cache, v_cache, block_tables, context_lens, query_start_loc, scale,
            max_query_len=None, out=None, stream=None, head_major=False):
    """Paged prefill: q is bf16 [total_q, Hq, D], rows packed per sequence by
    query_start_loc (int32 [S + 1]); row i of sequence s sits at position
    context_lens[s] - n_s + i and attends causally to the sequence's cached
    tokens. The pool is [NB, bs, Hkv, D], or [NB, Hkv, bs, D] with
    head_major=True. Returns out [total_q, Hq, D]."""
    dev = q.device
    for t, n, dt in ((q, "q", torch.bfloat16), (k_cache, "k_cache", torch.bfloat16),
                     (v_cache, "v_cache", torch.bfloat16), (block_tables, "block_tables", torch.int32),
                     (context_lens, "context_lens", torch.int32),
                     (query_start_loc, "query_start_loc", torch.int32)):
        _cuda(t, n, dt, dev)
    T, Hq, D = q.shape
    if head_major:
        NB, Hkv, bs, D2 = k_cache.shape
    else:
        NB, bs, Hkv, D2 = k_cache.shape
    S = context_lens.shape[0]
    if v_cache.shape != k_cache.shape or D2 != D or block_tables.dim() != 2 \
            or block_tables.shape[0] != S or query_start_loc.shape != (S + 1,):
        raise ValueError("shape mismatch between q, caches, block_tables and query_start_loc")
    if max_query_len is None:
        max_query_len = int((query_start_loc[1:] - query_start_loc[:-1]).max().item()) if S else 0
    if out is None:
        out = torch.empty_like(q)
    else:
        _cuda(out, "out", torch.bfloat16, dev)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    with torch.cuda.device(dev):
        st = lib().pa_prefill_layout(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                     block_tables.data_ptr(), block_tables.shape[1],
                                     context_lens.data_ptr(), query_start_loc.data_ptr(),
                                     int(max_query_len), float(scale), out.data_ptr(), S, T, Hq,
                                     Hkv, D, bs, NB, 1 if head_major else 0,
                                     _stream_ptr(stream, dev))
    _check("pa_prefill_layout", st)
    return out


def take_device_error(stream=None, device=None) -> int:
    """Synchronize the stream and return (and clear) the first device-side
    error code a prefill launch recorded: 0 none, 1 shared memory misaligned,
    2 a tensor-core wait ran out."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    code = ctypes.c_int32(0)
    with torch.cuda.device(dev):
        st = lib().pa_take_device_error(ctypes.addressof(code), _stream_ptr(stream, dev))
    _check("pa_take_device_error", st)
    return int(code.value)


def debug_prefill_fault(mode: int) -> None:
    """Test hook (off by default): mode 1 makes later prefill launches hold back
    one barrier arrival so that a bounded wait runs out and code 2 is recorded;
    mode 0 turns it off."""
    _check("pa_debug_prefill_fault", lib().pa_debug_prefill_fault(int(mode)))


VARIANT_DECODE_SIMT, VARIANT_PREFILL_MMA = 1, 2


def debug_kernel_variant(flags: int) -> None:
    """Test hook (off by default): run the comparison kernels kept for tests
    (VARIANT_DECODE_SIMT: CUDA-core decode tiles; VARIANT_PREFILL_MMA: the
    mma.sync prefill kernel) instead of the product kernels; 0 restores them."""
    _check("pa_debug_kernel_variant", lib().pa_debug_kernel_variant(int(flags)))


class DecodeStepGraph:
    """One decode step (store of the new K/V rows, then decode, through
    pa_decode_step) captured into a CUDA graph and replayed with one launch
    per step.

    The tensors passed in are the graph's fixed buffers: update their contents
    in place (q, k_new, v_new, slot_mapping, block_tables, context_lens) and
    call replay(); the result lands in ``out``. With ``host_stage`` (a pinned
    uint8 tensor) and ``device_stage`` (a device uint8 tensor of the same size
    whose slices back the input tensors), the host-to-device copy of the step's
    inputs is captured too, and with ``host_out`` (pinned) the read-back of
    ``out``: one replay is then the whole step from host buffers to host
    buffers. The decode is the automatic-partition pa_decode; its workspace is
    allocated once here, before capture.
    """

    def __init__(self, q, k_cache, v_cache, block_tables, context_lens, scale, k_new=None,
                 v_new=None, slot_mapping=None, out=None, host_stage=None, device_stage=None,
                 host_out=None, head_major=False):
        dev = q.device
        S, Hq, D = q.shape
        Hkv = k_cache.shape[1] if head_major else k_cache.shape[2]
        self.out = out if out is not None else torch.empty_like(q)
        self.workspace = workspace_for(Hq, Hkv, D, 0, dev)
        has_store = slot_mapping is not None and slot_mapping.shape[0] > 0

        def body():
            if host_stage is not None:
                device_stage.copy_(host_stage, non_blocking=True)
            if has_store:
                decode_step(k_new, v_new, slot_mapping, q, k_cache, v_cache, block_tables,
                            context_lens, scale, out=self.out, workspace=self.workspace,
                            head_major=head_major)
            else:
                decode(q, k_cache, v_cache, block_tables, context_lens, scale, out=self.out,
                       workspace=self.workspace, head_major=head_major)
            if host_out is not None:
                host_out.copy_(self.out, non_blocking=True)

        # one eager run first: library set-up calls happen outside the capture
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            body()
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize(dev)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            body()

    def replay(self):
        self.graph.replay()
        return self.out
