"""Seeded synthetic inputs for paged decode attention.

This module is shared by the tests, the benchmark and the oracle-side checks.
It holds NO arithmetic of the method itself: no attention, no slot formula,
no block-manager state machine. It only draws lengths, permutations and
random tensor contents, and lays sequences onto a shuffled pool in the
plainest possible way (sequence b's logical blocks take the next ids of a
seeded permutation, in order).

Shapes follow the model geometry the pages quote: a Llama-3.1-8B-class layer
(32 query heads, 8 KV heads, head dim 128, bf16; "How Paged Attention and
Continuous Batching Actually Work", §The problem) and a Llama-3-70B-class
layer (64/8 heads, head dim 128; "PagedAttention" glossary, §The
fragmentation problem). Block size is 16 ("How Paged Attention ...",
§Paged attention: virtual memory for the KV cache) unless a recipe is asked
for 8 or 32, the other typical sizes ("Paged Attention as a Memory Manager",
§PagedAttention).

Every random draw is seeded: numpy ``default_rng(seed)`` for lengths,
permutations and structure; a torch generator for tensor contents
(N(0, 1) in fp32, rounded to bf16).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

BLOCK_SIZE = 16


@dataclasses.dataclass
class Recipe:
    """Everything needed to build one synthetic decode workload."""

    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    # context length of every sequence before this step's append
    lens0: np.ndarray
    # number of tokens appended per sequence in the step (0 or 1)
    append: int
    # total physical blocks in the pool
    num_blocks: int
    # order in which the pool hands out physical block ids (a permutation)
    free_order: np.ndarray
    # shared-prefix structure (config 5 only); None elsewhere
    shared_prefix_tokens: int = 0
    diverge_seqs: Optional[np.ndarray] = None
    diverge_cut: Optional[np.ndarray] = None
    seed: int = 0

    @property
    def gqa_group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


def _blocks_for(n_tokens: np.ndarray, bs: int) -> np.ndarray:
    return (np.asarray(n_tokens, dtype=np.int64) + bs - 1) // bs


def _pool_size(need_blocks: int, factor: float = 1.25) -> int:
    return int(math.ceil(factor * need_blocks))


def tiny(seed: int = 1) -> Recipe:
    """4 sequences, lengths {1,5,17,33}, 4 q heads / 1 KV head, d=64, 16 blocks."""
    rng = np.random.default_rng(seed)
    lens = np.array([1, 5, 17, 33], dtype=np.int64)
    return Recipe("tiny", 4, 4, 1, 64, BLOCK_SIZE, lens, 1, 16,
                  rng.permutation(16).astype(np.int32), seed=seed)


def _bs_suffix(block_size: int) -> str:
    return "" if block_size == BLOCK_SIZE else f"_bs{block_size}"


def llama8b_layer(seed: int = 2, batch: int = 64, block_size: int = BLOCK_SIZE) -> Recipe:
    """Llama-3.1-8B-class layer: B=64, 32/8 heads, d=128, L~U[128,2048]."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(128, 2048, size=batch, endpoint=True).astype(np.int64)
    need = int(_blocks_for(lens + 1, block_size).sum())
    nb = _pool_size(need)
    return Recipe("llama8b_b64" + _bs_suffix(block_size), batch, 32, 8, 128, block_size, lens, 1,
                  nb, rng.permutation(nb).astype(np.int32), seed=seed)


def llama8b_high_concurrency(seed: int = 3, batch: int = 256) -> Recipe:
    """B=256, 32/8 heads, d=128, L0 ~ lognormal(median 800, sigma 1), clipped [16, 4096]."""
    rng = np.random.default_rng(seed)
    lens = np.rint(np.exp(rng.normal(math.log(800.0), 1.0, size=batch)))
    lens = np.clip(lens, 16, 4096).astype(np.int64)
    need = int(_blocks_for(lens + 1, BLOCK_SIZE).sum())
    nb = _pool_size(need)
    return Recipe("llama8b_b256_lognormal", batch, 32, 8, 128, BLOCK_SIZE, lens, 1, nb,
                  rng.permutation(nb).astype(np.int32), seed=seed)


def llama70b_long(seed: int = 4, batch: int = 8, block_size: int = BLOCK_SIZE) -> Recipe:
    """Llama-3-70B-class long context: 64/8 heads, d=128, L ~ U[8192, 32768]."""
    rng = np.random.default_rng(seed * 100 + batch)
    lens = rng.integers(8192, 32768, size=batch, endpoint=True).astype(np.int64)
    need = int(_blocks_for(lens + 1, block_size).sum())
    nb = _pool_size(need)
    return Recipe(f"llama70b_long_b{batch}" + _bs_suffix(block_size), batch, 64, 8, 128,
                  block_size, lens, 1, nb, rng.permutation(nb).astype(np.int32), seed=seed)


def shared_prefix(seed: int = 5, batch: int = 512, prefix_tokens: int = 1024,
                  n_diverge: int = 32) -> Recipe:
    """512 sequences over one 1024-token shared prefix; 32 of them diverge.

    The non-diverging sequences hold the whole prefix plus a private suffix of
    U[16, 512] tokens. A diverging sequence holds only the first
    ``prefix_tokens - r`` prefix tokens, r ~ U[1, 15], so its next token
    lands inside the last shared block.
    """
    rng = np.random.default_rng(seed)
    suffix = rng.integers(16, 512, size=batch, endpoint=True).astype(np.int64)
    div = np.sort(rng.choice(batch - 1, size=n_diverge, replace=False) + 1).astype(np.int64)
    cut = rng.integers(1, 15, size=n_diverge, endpoint=True).astype(np.int64)
    lens = prefix_tokens + suffix
    lens[div] = prefix_tokens - cut
    shared_blocks = prefix_tokens // BLOCK_SIZE
    private = 0
    for b in range(batch):
        if b in set(div.tolist()):
            private += 1  # copy-on-write target
        else:
            private += int(_blocks_for(lens[b] + 1, BLOCK_SIZE)) - shared_blocks
    nb = _pool_size(shared_blocks + private)
    return Recipe("shared_prefix_cow", batch, 32, 8, 128, BLOCK_SIZE, lens, 1, nb,
                  rng.permutation(nb).astype(np.int32), shared_prefix_tokens=prefix_tokens,
                  diverge_seqs=div, diverge_cut=cut, seed=seed)


def subset(r: Recipe, seqs, seed: int = 99) -> Recipe:
    """The sequences ``seqs`` of a recipe without sharing, laid on a pool of
    their own (1.25x their need, a seeded permutation): the same lengths and
    geometry as in the full workload at a fraction of its memory. Used for
    bounded host-side samples."""
    if r.diverge_seqs is not None:
        raise ValueError("subset() takes recipes without a shared prefix")
    lens = np.asarray(r.lens0, dtype=np.int64)[np.asarray(seqs, dtype=np.int64)]
    need = int(_blocks_for(lens + r.append, r.block_size).sum())
    nb = _pool_size(need)
    rng = np.random.default_rng(seed)
    return Recipe(r.name + f"_sample{len(lens)}", len(lens), r.num_q_heads, r.num_kv_heads,
                  r.head_dim, r.block_size, lens, r.append, nb,
                  rng.permutation(nb).astype(np.int32), seed=r.seed)


def all_recipes() -> List[Recipe]:
    return [tiny(), llama8b_layer(), llama8b_high_concurrency(), llama70b_long(batch=8),
            llama70b_long(batch=32), shared_prefix()]


def sequential_tables(lens: np.ndarray, free_order: np.ndarray, bs: int,
                      max_blocks: Optional[int] = None) -> np.ndarray:
    """Lay each sequence's logical blocks onto the next ids of ``free_order``.

    Returns int32 [B][max_blocks], unused entries -1. This is the simple
    placement used for workloads with no sharing; it is input layout, not
    the block manager.
    """
    nblk = _blocks_for(lens, bs)
    mb = int(nblk.max()) if max_blocks is None else max_blocks
    tables = np.full((len(lens), mb), -1, dtype=np.int32)
    pos = 0
    for b, n in enumerate(nblk.tolist()):
        tables[b, :n] = free_order[pos:pos + n]
        pos += n
    if pos > len(free_order):
        raise ValueError("pool too small for the requested lengths")
    return tables


def bf16_normal(shape, seed: int, device: str = "cpu"):
    """N(0,1) drawn in fp32 with a seeded torch generator, rounded to bf16."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def fill_padding_nan(cache, tables: np.ndarray, lens: np.ndarray, bs: int) -> None:
    """Write NaN into the slots past the end of each sequence's last block.

    Only blocks that are some sequence's last (partial) block and that no
    other sequence covers further are touched. Proves that masked slots are
    never read into a result.
    """
    import torch

    nb = cache.shape[0]
    fill = np.zeros(nb, dtype=np.int64)
    for b in range(len(lens)):
        L = int(lens[b])
        nblk = (L + bs - 1) // bs
        for j in range(nblk):
            blk = int(tables[b, j])
            fill[blk] = max(fill[blk], min(bs, L - j * bs))
    partial = np.nonzero((fill > 0) & (fill < bs))[0]
    for blk in partial.tolist():
        cache[blk, :, int(fill[blk]):, :] = float("nan")
    _ = torch  # cache is a torch tensor; indexing above is torch's


def lengths_after_append(r: Recipe) -> np.ndarray:
    return r.lens0 + r.append


# --------------------------------------------------------------------------
# Driving a pool through a recipe. The pool object does all block-manager
# arithmetic; these helpers only issue the recipe's operations in order, so
# the product pool and the oracle's model each produce their own tables.
# Both expose seq_create / seq_fork / append_tokens / append_slot / table.
# --------------------------------------------------------------------------

def drive_prefill(pool, r: Recipe) -> List[int]:
    """Create every sequence of the recipe with its pre-step length."""
    if r.diverge_seqs is None:
        seqs = []
        for b in range(r.num_seqs):
            s = pool.seq_create()
            pool.append_tokens(s, int(r.lens0[b]))
            seqs.append(s)
        return seqs
    div = set(int(x) for x in r.diverge_seqs)
    root = pool.seq_create()
    pool.append_tokens(root, r.shared_prefix_tokens)
    seqs = [root]
    for b in range(1, r.num_seqs):
        n = int(r.lens0[b]) if b in div else r.shared_prefix_tokens
        seqs.append(pool.seq_fork(root, n))
    for b in range(r.num_seqs):
        if b not in div:
            pool.append_tokens(seqs[b], int(r.lens0[b]) - r.shared_prefix_tokens)
    return seqs


def drive_step_append(pool, seqs: List[int], r: Recipe):
    """Reserve this step's slot for every sequence (``r.append`` tokens each).

    Returns (slot_mapping int64 [B * append], cow_pairs int32 [P][2]).
    """
    slots, cows = [], []
    for s in seqs:
        for _ in range(r.append):
            slot, cow = pool.append_slot(s)
            slots.append(slot)
            if cow is not None:
                cows.append(cow)
    return (np.asarray(slots, dtype=np.int64),
            np.asarray(cows, dtype=np.int32).reshape(-1, 2))


def tables_of(pool, seqs: List[int], max_blocks: Optional[int] = None) -> np.ndarray:
    rows = [pool.table(s) for s in seqs]
    mb = max(len(t) for t in rows) if max_blocks is None else max_blocks
    out = np.full((len(seqs), mb), -1, dtype=np.int32)
    for i, t in enumerate(rows):
        out[i, :len(t)] = t
    return out


def step_tensors(r: Recipe, device: str = "cpu", seed_offset: int = 0):
    """Random tensor contents of one step: q, k_new, v_new, k_cache, v_cache (bf16)."""
    import torch

    s = r.seed * 1000 + seed_offset
    B, Hq, Hkv, D, BS = r.num_seqs, r.num_q_heads, r.num_kv_heads, r.head_dim, r.block_size
    q = bf16_normal((B, Hq, D), s + 1, device)
    k_new = bf16_normal((B * r.append, Hkv, D), s + 2, device)
    v_new = bf16_normal((B * r.append, Hkv, D), s + 3, device)
    k_cache = torch.empty((r.num_blocks, Hkv, BS, D), dtype=torch.bfloat16, device=device)
    v_cache = torch.empty_like(k_cache)
    chunk = max(1, (1 << 26) // (Hkv * BS * D))  # ~64M elements per draw
    for i, c in enumerate((k_cache, v_cache)):
        for j, start in enumerate(range(0, r.num_blocks, chunk)):
            stop = min(r.num_blocks, start + chunk)
            c[start:stop] = bf16_normal((stop - start, Hkv, BS, D), s + 10 + 7919 * i + 31 * j, device)
    return q, k_new, v_new, k_cache, v_cache
