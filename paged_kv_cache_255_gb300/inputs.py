"""Seeded synthetic inputs for paged decode attention.

This module only builds inputs: sequence lengths, block tables drawn from a
block pool, slot mappings and bf16 values. It holds none of the attention
arithmetic, and neither the CUDA path nor the oracle lives here; both the
tests and the benchmark draw their inputs from it.

Structure follows the pages:
  * a sequence's ``block_table`` maps its logical blocks to physical blocks of
    one pool ("Building a minimal vLLM implementation", sequence.py, the
    ``block_table`` field);
  * blocks hold a fixed number of tokens (same page, config.py,
    ``kvcache_block_size``);
  * the pool reserves block 0 as a null block that is never handed out
    ("Implementation Details", PagedAttention -- BlockPool);
  * prefix caching lets several sequences point at the same physical block
    (same section, the block-hash map and ``--enable-prefix-caching``).

Pool layout: ``[num_blocks, block_size, num_kv_heads, head_dim]`` bf16, so
that cache slot ``block_id * block_size + offset`` names one contiguous
``num_kv_heads * head_dim`` row.

Values are N(0, 1) drawn in fp32 and rounded to bf16 (round to nearest even,
done by torch's dtype conversion). Every pool row that no live sequence owns
(the null block, free blocks, the unused tail of each sequence's last block,
and the row that the step's store is about to write) is filled with NaN, so
that any read of it shows up as a NaN in the output.

Structure (lengths, tables, slots) always comes from numpy's PCG64 seeded
with ``seed``. Values come from the same numpy stream on the CPU, or from a
torch CUDA generator seeded with ``seed`` when ``device`` is a CUDA device
(the big workloads would take tens of seconds to draw on the host).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

HEAD_DIM = 128


@dataclasses.dataclass
class Spec:
    """Shape of one synthetic decode step."""

    name: str
    # (count, lo, hi): ``count`` sequences with context length uniform in [lo, hi]
    ctx_groups: tuple
    num_q_heads: int
    num_kv_heads: int
    block_size: int
    head_dim: int = HEAD_DIM
    # "permute": tables are a random permutation of blocks 1..NB-1 (NB set by
    #            pool_factor, or an explicit num_blocks);
    # "fragmented": every other block id (the odd ones, in order) goes to a
    #            sequence, the even ones stay free;
    # "prefix_shared": every sequence starts with the same prefix_blocks
    #            physical blocks, then owns unique_blocks blocks of its own.
    pool_mode: str = "permute"
    pool_factor: float = 1.0
    num_blocks: Optional[int] = None
    prefix_blocks: int = 0
    unique_blocks: int = 0
    # "last_token": one new row per sequence, written at position L_s - 1
    #               (the token this decode step attends with);
    # "random_slots": store_rows distinct slots drawn from the sequences'
    #               unique (non-prefix) blocks, pad_rows of them set to -1;
    # "none": no store in this step.
    store_mode: str = "last_token"
    store_rows: int = 0
    pad_rows: int = 0

    @property
    def num_seqs(self) -> int:
        return sum(c for c, _, _ in self.ctx_groups)


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


# The five decode steps the benchmark and the parity tests are built around.
SPECS = {
    # 4 sequences, 16 q / 8 KV heads, pool of 128 blocks with block 0 null.
    "tiny": Spec("tiny", ((4, 1, 300),), 16, 8, 16, num_blocks=128),
    # 60 sequences shaped like a Qwen3-0.6B decode batch (16 q / 8 KV heads).
    "qwen3_0_6b": Spec("qwen3_0_6b", ((60, 64, 1024),), 16, 8, 16, pool_factor=1.2),
    "qwen3_0_6b_bs256": Spec("qwen3_0_6b_bs256", ((60, 64, 1024),), 16, 8, 256,
                             pool_factor=1.2),
    # 256 sequences shaped like a Qwen3-8B decode batch (32 q / 8 KV heads),
    # in a fragmented pool.
    "large_batch": Spec("large_batch", ((256, 512, 4096),), 32, 8, 16,
                        pool_mode="fragmented"),
    # 8 very long sequences among 120 short ones.
    "long_context": Spec("long_context", ((8, 32768, 131072), (120, 128, 512)), 32, 8, 16),
    # 128 sequences sharing a 2048-token prefix, then 256 tokens each of their
    # own; 64 q / 8 KV heads; a separate 4096-row store with 10% padding.
    "prefix_shared": Spec("prefix_shared", ((128, 2304, 2304),), 64, 8, 16,
                          pool_mode="prefix_shared", prefix_blocks=128,
                          unique_blocks=16, store_mode="random_slots",
                          store_rows=4096, pad_rows=410),
}


def scaled(spec: Spec, num_seqs: Optional[int] = None, ctx_div: int = 1,
           name: Optional[str] = None, **over) -> Spec:
    """A smaller copy of ``spec``: fewer sequences and/or shorter contexts.

    Group counts are scaled in proportion (each group keeps at least one
    sequence); context bounds are divided by ``ctx_div``; prefix-shared pools
    scale their prefix and unique block counts the same way.
    """
    groups = list(spec.ctx_groups)
    if num_seqs is not None:
        total = spec.num_seqs
        groups = [(max(1, round(c * num_seqs / total)), lo, hi) for c, lo, hi in groups]
    groups = tuple((c, max(1, lo // ctx_div), max(1, hi // ctx_div)) for c, lo, hi in groups)
    fields = dict(ctx_groups=groups, name=name or f"{spec.name}_small")
    if spec.pool_mode == "prefix_shared":
        pb = max(1, spec.prefix_blocks // ctx_div)
        ub = max(1, spec.unique_blocks // ctx_div)
        L = (pb + ub) * spec.block_size
        fields["ctx_groups"] = tuple((c, L, L) for c, _, _ in groups)
        fields["prefix_blocks"] = pb
        fields["unique_blocks"] = ub
    if spec.store_mode == "random_slots":
        n_seq = sum(c for c, _, _ in fields["ctx_groups"])
        cap = n_seq * fields.get("unique_blocks", spec.unique_blocks) * spec.block_size
        rows = min(spec.store_rows, cap)
        fields["store_rows"] = rows
        fields["pad_rows"] = round(rows * spec.pad_rows / spec.store_rows)
    fields.update(over)
    return dataclasses.replace(spec, **fields)


@dataclasses.dataclass
class Workload:
    spec: Spec
    seed: int
    # structure (numpy, host)
    context_lens: np.ndarray      # int32 [S]
    block_tables: np.ndarray      # int32 [S, max_blocks_per_seq], padding = 0
    slot_mapping: np.ndarray      # int64 [N], -1 = skip
    num_blocks: int
    owned_blocks: np.ndarray      # sorted int array: physical blocks some sequence uses
    # values (torch bf16, on ``device``)
    q: torch.Tensor               # [S, Hq, D]
    k_new: torch.Tensor           # [N, Hkv, D]
    v_new: torch.Tensor           # [N, Hkv, D]
    k_cache: torch.Tensor         # [NB, bs, Hkv, D]
    v_cache: torch.Tensor         # [NB, bs, Hkv, D]
    # bookkeeping for the brute-force check: the distinct block contents in
    # draw order, and for each (sequence, logical block) which of them it is
    content_index: np.ndarray     # int64 [S, max_blocks_per_seq], -1 = padding
    content_k: Optional[torch.Tensor] = None   # [n_content, bs, Hkv, D]
    content_v: Optional[torch.Tensor] = None

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.context_lens.size else 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.spec.head_dim)

    def kv_bytes(self) -> int:
        """Logical K+V bytes one decode reads: every context token, K and V."""
        s = self.spec
        return int(self.context_lens.astype(np.int64).sum()) * s.num_kv_heads * s.head_dim * 2 * 2

    def unique_kv_bytes(self) -> int:
        """K+V bytes of the distinct physical rows the decode reads."""
        s = self.spec
        rows = set()
        for i in range(self.num_seqs):
            L = int(self.context_lens[i])
            for j in range(_cdiv(L, s.block_size)):
                n = min(s.block_size, L - j * s.block_size)
                rows.add((int(self.block_tables[i, j]), n))
        per_block = {}
        for b, n in rows:
            per_block[b] = max(per_block.get(b, 0), n)
        return sum(per_block.values()) * s.num_kv_heads * s.head_dim * 2 * 2

    def logical_kv(self, s_idx: int, after_store: bool = True):
        """Contiguous K, V of sequence ``s_idx`` as [L, Hkv, D] tensors.

        Built by concatenating the sequence's block contents in table order
        (whole blocks, from the generator's own record of what it placed
        where) and, for a last-token store, putting the stored row at L-1.
        Only for workloads generated with ``keep_content=True``.
        """
        assert self.content_k is not None, "generate with keep_content=True"
        L = int(self.context_lens[s_idx])
        s = self.spec
        idx = [int(c) for c in self.content_index[s_idx, :_cdiv(L, s.block_size)]]
        if not idx:
            shape = (0, s.num_kv_heads, s.head_dim)
            return (torch.empty(shape, dtype=torch.bfloat16),
                    torch.empty(shape, dtype=torch.bfloat16))
        k = torch.cat([self.content_k[c] for c in idx], 0)[:L].clone()
        v = torch.cat([self.content_v[c] for c in idx], 0)[:L].clone()
        if after_store and s.store_mode == "last_token":
            k[L - 1] = self.k_new[s_idx].cpu()
            v[L - 1] = self.v_new[s_idx].cpu()
        assert s.store_mode != "random_slots" or not after_store, \
            "random-slot stores have no per-sequence logical view"
        return k, v


def _normal_bf16(rng: np.random.Generator, tgen, shape, device) -> torch.Tensor:
    if tgen is None:
        x = rng.standard_normal(size=shape, dtype=np.float32)
        return torch.from_numpy(x).to(torch.bfloat16)
    x = torch.randn(shape, generator=tgen, device=device, dtype=torch.float32)
    return x.to(torch.bfloat16)


def generate(spec: Spec, seed: int = 0, device="cpu", keep_content: bool = False,
             context_lens=None, values: bool = True) -> Workload:
    """Draw one decode step for ``spec``.

    ``context_lens`` overrides the drawn lengths (edge-case tests);
    ``values=False`` draws the structure only (all tensors None).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    bs, Hkv, D = spec.block_size, spec.num_kv_heads, spec.head_dim
    device = torch.device(device)

    # -- lengths
    if context_lens is None:
        parts = [rng.integers(lo, hi + 1, size=c) for c, lo, hi in spec.ctx_groups]
        ctx = np.concatenate(parts).astype(np.int32) if parts else np.zeros(0, np.int32)
    else:
        ctx = np.asarray(context_lens, dtype=np.int32)
    S = int(ctx.shape[0])
    nb = [(_cdiv(int(L), bs)) for L in ctx]
    max_nb = max(1, max(nb) if nb else 1)

    # -- tables: content_index[s, j] names the distinct block content that
    # logical block j of sequence s holds; phys[c] is where content c lives.
    content_index = np.full((S, max_nb), -1, dtype=np.int64)
    if spec.pool_mode == "prefix_shared":
        pb, ub = spec.prefix_blocks, spec.unique_blocks
        n_content = pb + S * ub
        for i in range(S):
            assert nb[i] <= pb + ub
            content_index[i, :nb[i]] = [j if j < pb else pb + i * ub + (j - pb)
                                        for j in range(nb[i])]
        NB = spec.num_blocks or (n_content + 1)
        phys = 1 + rng.permutation(NB - 1)[:n_content]
    else:
        n_content = int(sum(nb))
        c = 0
        for i in range(S):
            content_index[i, :nb[i]] = np.arange(c, c + nb[i])
            c += nb[i]
        if spec.pool_mode == "fragmented":
            NB = spec.num_blocks or (2 * n_content + 1)
            phys = 1 + 2 * np.arange(n_content)          # odd ids, in order
        else:
            NB = spec.num_blocks or (math.ceil(spec.pool_factor * n_content) + 1)
            phys = 1 + rng.permutation(NB - 1)[:n_content]
    assert NB - 1 >= n_content, "pool too small"
    phys = np.asarray(phys, dtype=np.int64)
    block_tables = np.zeros((S, max_nb), dtype=np.int32)
    for i in range(S):
        block_tables[i, :nb[i]] = phys[content_index[i, :nb[i]]]

    # -- store batch
    if spec.store_mode == "last_token":
        rows = []
        for i in range(S):
            L = int(ctx[i])
            if L == 0:
                rows.append(-1)
                continue
            pos = L - 1
            rows.append(int(block_tables[i, pos // bs]) * bs + pos % bs)
        slot_mapping = np.asarray(rows, dtype=np.int64)
    elif spec.store_mode == "random_slots":
        pb, ub = spec.prefix_blocks, spec.unique_blocks
        uniq_phys = phys[pb:pb + S * ub]
        cand = (uniq_phys[:, None] * bs + np.arange(bs)[None, :]).reshape(-1)
        pick = rng.choice(cand.shape[0], size=spec.store_rows, replace=False)
        slot_mapping = cand[pick].astype(np.int64)
        pad = rng.permutation(spec.store_rows)[:spec.pad_rows]
        slot_mapping[pad] = -1
    else:
        slot_mapping = np.zeros(0, dtype=np.int64)
    N = int(slot_mapping.shape[0])

    if not values:
        return Workload(spec=spec, seed=seed, context_lens=ctx, block_tables=block_tables,
                        slot_mapping=slot_mapping, num_blocks=int(NB),
                        owned_blocks=np.unique(phys), q=None, k_new=None, v_new=None,
                        k_cache=None, v_cache=None, content_index=content_index)

    # -- values
    tgen = None
    if device.type == "cuda":
        tgen = torch.Generator(device=device)
        tgen.manual_seed(seed)
    Hq = spec.num_q_heads
    q = _normal_bf16(rng, tgen, (S, Hq, D), device)
    k_new = _normal_bf16(rng, tgen, (N, Hkv, D), device)
    v_new = _normal_bf16(rng, tgen, (N, Hkv, D), device)
    ck = _normal_bf16(rng, tgen, (n_content, bs, Hkv, D), device)
    cv = _normal_bf16(rng, tgen, (n_content, bs, Hkv, D), device)

    nan = torch.tensor(float("nan"), dtype=torch.bfloat16)
    k_cache = torch.full((NB, bs, Hkv, D), nan.item(), dtype=torch.bfloat16, device=device)
    v_cache = torch.full((NB, bs, Hkv, D), nan.item(), dtype=torch.bfloat16, device=device)
    pidx = torch.from_numpy(phys).to(device)
    k_cache[pidx] = ck
    v_cache[pidx] = cv
    # poison the unused tail of each last block, and each row a last-token
    # store is about to write
    for i in range(S):
        L = int(ctx[i])
        if L == 0:
            continue
        last = int(block_tables[i, nb[i] - 1])
        used = L - (nb[i] - 1) * bs
        if used < bs and spec.pool_mode != "prefix_shared":
            k_cache[last, used:] = nan
            v_cache[last, used:] = nan
    if spec.store_mode == "last_token":
        flat_k = k_cache.view(NB * bs, Hkv, D)
        flat_v = v_cache.view(NB * bs, Hkv, D)
        valid = torch.from_numpy(slot_mapping[slot_mapping >= 0]).to(device)
        flat_k[valid] = nan
        flat_v[valid] = nan

    wl = Workload(spec=spec, seed=seed, context_lens=ctx, block_tables=block_tables,
                  slot_mapping=slot_mapping, num_blocks=int(NB),
                  owned_blocks=np.unique(phys), q=q, k_new=k_new, v_new=v_new,
                  k_cache=k_cache, v_cache=v_cache, content_index=content_index)
    if keep_content:
        wl.content_k = ck.cpu()
        wl.content_v = cv.cpu()
    return wl


# -- prefill batches ---------------------------------------------------------
#
# A prefill step takes a chunk of n_s new tokens per sequence (n_s <= L_s, the
# last n_s positions of the sequence): their K/V rows are stored through a
# slot mapping, then every chunk row attends causally to the sequence's first
# L_s - n_s + i + 1 tokens. The pool holds the earlier L_s - n_s tokens; the
# rows the store is about to write hold NaN until it does.

# name -> (pool spec, chunk): chunk None means the whole prompt (n_s = L_s),
# an int c means n_s = min(c, L_s).
PREFILL_SPECS = {
    # 60 batched prompts of 64..1024 tokens, Qwen3-0.6B attention shape
    # (16 q / 8 KV heads): the prompt phase of the 60-prompt decode batch.
    "qwen3_0_6b_prompts": (Spec("qwen3_0_6b_prompts", ((60, 64, 1024),), 16, 8, 16,
                                pool_factor=1.2, store_mode="none"), None),
    # chunked prefill: 32 sequences with 2k..8k tokens of context each take a
    # 512-token chunk, Qwen3-8B attention shape (32 q / 8 KV heads).
    "chunked_8b": (Spec("chunked_8b", ((32, 2048, 8192),), 32, 8, 16,
                        store_mode="none"), 512),
}


@dataclasses.dataclass
class PrefillBatch:
    wl: Workload                  # pool, tables and lengths (L_s counts the chunk)
    query_start_loc: np.ndarray   # int32 [S + 1]
    q: torch.Tensor               # bf16 [T, Hq, D]
    k_new: torch.Tensor           # bf16 [T, Hkv, D], the chunk rows' K
    v_new: torch.Tensor           # bf16 [T, Hkv, D]
    slot_mapping: np.ndarray      # int64 [T], where each chunk row is stored

    @property
    def chunk_lens(self) -> np.ndarray:
        return np.diff(self.query_start_loc)

    @property
    def max_query_len(self) -> int:
        return int(self.chunk_lens.max()) if self.chunk_lens.size else 0

    def causal_pairs(self) -> int:
        """(row, key) pairs one query head attends over: row i of a chunk of n
        in a sequence of L sees L - n + i + 1 keys."""
        L = self.wl.context_lens.astype(np.int64)
        n = self.chunk_lens.astype(np.int64)
        return int((n * (L - n) + n * (n + 1) // 2).sum())


def prefill_batch(spec: Spec, seed: int = 0, chunk=None, context_lens=None,
                  chunk_lens=None, keep_content: bool = False) -> PrefillBatch:
    """Draw one prefill step over a pool drawn by ``generate`` (store_mode
    "none"). ``chunk_lens`` (one per sequence, each <= L_s) overrides
    ``chunk``."""
    assert spec.store_mode == "none"
    wl = generate(spec, seed=seed, context_lens=context_lens, keep_content=keep_content)
    L = wl.context_lens.astype(np.int64)
    if chunk_lens is not None:
        n = np.asarray(chunk_lens, dtype=np.int64)
    elif chunk is None:
        n = L.copy()
    else:
        n = np.minimum(L, int(chunk))
    assert n.shape == L.shape and (n >= 0).all() and (n <= L).all()
    qsl = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    bs = spec.block_size
    slots = []
    for s in range(wl.num_seqs):
        pos = np.arange(L[s] - n[s], L[s])
        slots.append(wl.block_tables[s, pos // bs].astype(np.int64) * bs + pos % bs)
    slot_mapping = np.concatenate(slots) if slots else np.zeros(0, np.int64)
    T = int(qsl[-1])
    rng = np.random.Generator(np.random.PCG64(seed + 1_000_003))
    Hq, Hkv, D = spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    q = _normal_bf16(rng, None, (T, Hq, D), "cpu")
    k_new = _normal_bf16(rng, None, (T, Hkv, D), "cpu")
    v_new = _normal_bf16(rng, None, (T, Hkv, D), "cpu")
    NB = wl.num_blocks
    nan = float("nan")
    idx = torch.from_numpy(slot_mapping)
    wl.k_cache.view(NB * bs, Hkv, D)[idx] = nan
    wl.v_cache.view(NB * bs, Hkv, D)[idx] = nan
    return PrefillBatch(wl=wl, query_start_loc=qsl, q=q, k_new=k_new, v_new=v_new,
                        slot_mapping=slot_mapping)
