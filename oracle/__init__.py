"""Python access to the fp64 CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use this module; the library does not. The
oracle shares no code with the CUDA path.

``build()`` compiles ``oracle.c`` with gcc (OpenMP on) into
``oracle/_build/liboracle.so``; the functions below compile it on first use
when the shared object is missing.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_ARG, ERR_RANGE = 0, 1, 2


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` and return its path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    fresh = (os.path.exists(_LIB_PATH)
             and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall", "-Wextra",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bits(x) -> np.ndarray:
    """Host, contiguous uint16 view of a bf16 tensor (or pass a uint16 array)."""
    if isinstance(x, torch.Tensor):
        assert x.dtype == torch.bfloat16, x.dtype
        x = x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    x = np.ascontiguousarray(x)
    assert x.dtype == np.uint16, x.dtype
    return x


def _arr(x, dtype) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x), dtype=dtype)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """The oracle's entry points, bound to one compiled copy of ``oracle.c``."""

    def __init__(self, lib):
        p = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_store_kvcache.argtypes = [p, p, p, p, p, i64, i32, i32, i32, i64]
        lib.oracle_store_kvcache.restype = i32
        lib.oracle_decode.argtypes = [p, p, p, p, i32, p, dbl, p, i32, i32, i32, i32, i32,
                                      i64, i32]
        lib.oracle_decode.restype = i32
        lib.oracle_decode_pairs.argtypes = [p, p, p, p, i32, p, dbl, p, i64, p, i32, i32, i32,
                                            i32, i32, i64, i32]
        lib.oracle_decode_pairs.restype = i32
        lib.oracle_decode_multi.argtypes = [p, p, p, p, i32, p, i32, dbl, p, i32, i32, i32, i32,
                                            i32, i64, i32]
        lib.oracle_decode_multi.restype = i32
        lib.oracle_store_kvcache_layout.argtypes = [p, p, p, p, p, i64, i32, i32, i32, i64, i32]
        lib.oracle_store_kvcache_layout.restype = i32
        lib.oracle_decode_layout.argtypes = [p, p, p, p, i32, p, dbl, p, i32, i32, i32, i32, i32,
                                             i64, i32, i32]
        lib.oracle_decode_layout.restype = i32
        lib.oracle_prefill.argtypes = [p, p, p, p, i32, p, p, dbl, p, i32, i32, i32, i32, i32,
                                       i32, i64, i32]
        lib.oracle_prefill.restype = i32
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = i32
        self.lib = lib

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def store_kvcache(self, k, v, k_cache, v_cache, slot_mapping):
        """Return new (k_cache, v_cache) uint16 arrays after the store.

        ``k``/``v``: bf16 [N, Hkv, D]; caches: bf16 [NB, bs, Hkv, D];
        ``slot_mapping``: int64 [N] (-1 = skip). Inputs are not modified.
        """
        kb, vb = _bits(k), _bits(v)
        kc, vc = _bits(k_cache).copy(), _bits(v_cache).copy()
        sm = _arr(slot_mapping, np.int64)
        NB, bs, Hkv, D = kc.shape
        N = sm.shape[0]
        assert kb.shape == (N, Hkv, D) and vb.shape == (N, Hkv, D)
        rc = self.lib.oracle_store_kvcache(_ptr(kb), _ptr(vb), _ptr(kc), _ptr(vc), _ptr(sm), N,
                                           Hkv, D, bs, NB)
        if rc != OK:
            raise OracleError(f"oracle_store_kvcache returned {rc}")
        return kc, vc

    def store_kvcache_into(self, k, v, k_cache_bits, v_cache_bits, slot_mapping):
        """The store, writing into the given uint16 cache arrays in place."""
        kb, vb = _bits(k), _bits(v)
        sm = _arr(slot_mapping, np.int64)
        kc, vc = k_cache_bits, v_cache_bits
        assert kc.dtype == np.uint16 and vc.dtype == np.uint16
        assert kc.flags.c_contiguous and vc.flags.c_contiguous and kc.shape == vc.shape
        NB, bs, Hkv, D = kc.shape
        rc = self.lib.oracle_store_kvcache(_ptr(kb), _ptr(vb), _ptr(kc), _ptr(vc), _ptr(sm),
                                           sm.shape[0], Hkv, D, bs, NB)
        if rc != OK:
            raise OracleError(f"oracle_store_kvcache returned {rc}")

    def decode(self, q, k_cache, v_cache, block_tables, context_lens, scale, threads: int = 0):
        """fp64 [S, Hq, D] attention output over the paged cache."""
        qb, kc, vc = _bits(q), _bits(k_cache), _bits(v_cache)
        bt = _arr(block_tables, np.int32)
        cl = _arr(context_lens, np.int32)
        S, Hq, D = qb.shape
        NB, bs, Hkv, D2 = kc.shape
        assert D == D2 and vc.shape == kc.shape and cl.shape == (S,)
        if bt.ndim != 2 or bt.shape[0] != S:
            raise ValueError("block_tables must be [num_seqs, max_blocks_per_seq]")
        out = np.zeros((S, Hq, D), dtype=np.float64)
        rc = self.lib.oracle_decode(_ptr(qb), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1],
                                    _ptr(cl), float(scale), _ptr(out), S, Hq, Hkv, D, bs, NB,
                                    int(threads))
        if rc != OK:
            raise OracleError(f"oracle_decode returned {rc}")
        return out

    def decode_pairs(self, q, k_cache, v_cache, block_tables, context_lens, scale, pairs,
                     threads: int = 0):
        """fp64 [P, D] outputs for the given (sequence, query head) pairs."""
        qb, kc, vc = _bits(q), _bits(k_cache), _bits(v_cache)
        bt = _arr(block_tables, np.int32)
        cl = _arr(context_lens, np.int32)
        pr = _arr(pairs, np.int32).reshape(-1, 2)
        S, Hq, D = qb.shape
        NB, bs, Hkv, _ = kc.shape
        out = np.zeros((pr.shape[0], D), dtype=np.float64)
        rc = self.lib.oracle_decode_pairs(_ptr(qb), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1],
                                          _ptr(cl), float(scale), _ptr(pr), pr.shape[0],
                                          _ptr(out), S, Hq, Hkv, D, bs, NB, int(threads))
        if rc != OK:
            raise OracleError(f"oracle_decode_pairs returned {rc}")
        return out


    def store_kvcache_head_major(self, k, v, k_cache, v_cache, slot_mapping):
        """The store into a head-major pool [NB, Hkv, bs, D]; returns new
        (k_cache, v_cache) uint16 arrays."""
        kb, vb = _bits(k), _bits(v)
        kc, vc = _bits(k_cache).copy(), _bits(v_cache).copy()
        sm = _arr(slot_mapping, np.int64)
        NB, Hkv, bs, D = kc.shape
        rc = self.lib.oracle_store_kvcache_layout(_ptr(kb), _ptr(vb), _ptr(kc), _ptr(vc),
                                                  _ptr(sm), sm.shape[0], Hkv, D, bs, NB, 1)
        if rc != OK:
            raise OracleError(f"oracle_store_kvcache_layout returned {rc}")
        return kc, vc

    def decode_head_major(self, q, k_cache, v_cache, block_tables, context_lens, scale,
                          threads: int = 0):
        """fp64 [S, Hq, D] decode over a head-major pool [NB, Hkv, bs, D]."""
        qb, kc, vc = _bits(q), _bits(k_cache), _bits(v_cache)
        bt = _arr(block_tables, np.int32)
        cl = _arr(context_lens, np.int32)
        S, Hq, D = qb.shape
        NB, Hkv, bs, _ = kc.shape
        out = np.zeros((S, Hq, D), dtype=np.float64)
        rc = self.lib.oracle_decode_layout(_ptr(qb), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1],
                                           _ptr(cl), float(scale), _ptr(out), S, Hq, Hkv, D, bs,
                                           NB, 1, int(threads))
        if rc != OK:
            raise OracleError(f"oracle_decode_layout returned {rc}")
        return out

    def prefill(self, q, k_cache, v_cache, block_tables, context_lens, query_start_loc, scale,
                threads: int = 0):
        """fp64 [total_q, Hq, D] prefill outputs; rows of q ([total_q, Hq, D]) are
        packed per sequence by query_start_loc ([S + 1])."""
        qb, kc, vc = _bits(q), _bits(k_cache), _bits(v_cache)
        bt = _arr(block_tables, np.int32)
        cl = _arr(context_lens, np.int32)
        qsl = _arr(query_start_loc, np.int32)
        T, Hq, D = qb.shape
        NB, bs, Hkv, _ = kc.shape
        S = cl.shape[0]
        out = np.zeros((T, Hq, D), dtype=np.float64)
        rc = self.lib.oracle_prefill(_ptr(qb), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1],
                                     _ptr(cl), _ptr(qsl), float(scale), _ptr(out), S, T, Hq, Hkv,
                                     D, bs, NB, int(threads))
        if rc != OK:
            raise OracleError(f"oracle_prefill returned {rc}")
        return out

    def decode_multi(self, q, k_cache, v_cache, block_tables, context_lens, scale,
                     threads: int = 0):
        """fp64 [S, Q, Hq, D] outputs for Q new tokens per sequence (q is
        [S, Q, Hq, D]); token i attends to keys t <= L - Q + i."""
        qb, kc, vc = _bits(q), _bits(k_cache), _bits(v_cache)
        bt = _arr(block_tables, np.int32)
        cl = _arr(context_lens, np.int32)
        S, Q, Hq, D = qb.shape
        NB, bs, Hkv, _ = kc.shape
        out = np.zeros((S, Q, Hq, D), dtype=np.float64)
        rc = self.lib.oracle_decode_multi(_ptr(qb), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1],
                                          _ptr(cl), Q, float(scale), _ptr(out), S, Hq, Hkv, D,
                                          bs, NB, int(threads))
        if rc != OK:
            raise OracleError(f"oracle_decode_multi returned {rc}")
        return out


def compile_variant(src: str, out_path: str) -> "Oracle":
    """Compile another copy of the oracle source (the tests plant mistakes in
    copies to check that the pins catch them) and bind it."""
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-I", _HERE,
           "-o", out_path, src, "-lm"]
    subprocess.run(cmd, check=True)
    return Oracle(ctypes.CDLL(out_path))


def get() -> Oracle:
    """The oracle built from ``oracle.c`` (compiled on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(ctypes.CDLL(build()))
    return _lib


def num_threads() -> int:
    return get().num_threads()


def store_kvcache(*a, **kw):
    return get().store_kvcache(*a, **kw)


def decode(*a, **kw):
    return get().decode(*a, **kw)


def decode_pairs(*a, **kw):
    return get().decode_pairs(*a, **kw)


def decode_multi(*a, **kw):
    return get().decode_multi(*a, **kw)


def prefill(*a, **kw):
    return get().prefill(*a, **kw)
