"""Oracle for paged decode attention: plain, slow, obviously correct, float64.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package. It shares no code with
the CUDA library and never imports it.

Contents
--------
* ``paged_decode`` -- the C oracle (``pa_oracle.c``): reassemble each
  sequence's K/V through its block table, then textbook softmax attention in
  float64 (sources: "Paged Attention as a Memory Manager", §How the Kernel
  Executes Paged Attention; "PagedAttention and continuous batching",
  §Attention kernel modification).
* ``paged_decode_numpy`` -- an independent numpy twin of the same definition.
* ``brute_force_decode`` -- pure-Python loops over a contiguous K/V, tiny
  inputs only.
* ``partition_decode`` / ``merge_partitions`` -- the split-K model: each
  partition of ``P`` tokens yields (m, l, acc) and a log-sum-exp merge
  recombines them. The pages do not describe split-K; this is the plain
  reading of a flash-decoding partition.
* ``reshape_and_cache`` / ``copy_blocks`` -- byte copies through the slot
  formula ("How Paged Attention and Continuous Batching Actually Work",
  §Paged attention: virtual memory for the KV cache; §One step, end to end)
  and of whole blocks ("Paged Attention as a Memory Manager", §Prefix
  Caching and Copy-on-Write).
* ``PoolModel`` -- the block manager as the pages describe it: a free list
  with O(1) pop/push, per-sequence block tables, reference counts, a fresh
  block when a token crosses a block boundary, copy-on-write when the
  target block is shared.

Parity status: every function here is pinned by ``tests/test_oracle.py``
against the pages' worked example, brute force, closed-form invariants or a
library routine (torch SDPA in float64); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import itertools
import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        p = ctypes.c_void_p
        i32 = ctypes.c_int32
        i64 = ctypes.c_int64
        lib.oracle_paged_decode.argtypes = [p, p, p, p, i32, p, i32, i32, i32, i32, i32, i32,
                                            ctypes.c_double, p, i64, p, p]
        lib.oracle_paged_decode.restype = ctypes.c_int
        lib.oracle_reshape_and_cache.argtypes = [p, p, p, p, p, i32, i32, i32, i32, i32]
        lib.oracle_reshape_and_cache.restype = ctypes.c_int
        lib.oracle_copy_blocks.argtypes = [p, p, p, i32, i32, i32, i32, i32]
        lib.oracle_copy_blocks.restype = ctypes.c_int
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        lib.oracle_set_num_threads.restype = None
        u8 = ctypes.c_uint8
        lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_from_float.restype = u8
        lib.oracle_e4m3_to_double.argtypes = [u8]
        lib.oracle_e4m3_to_double.restype = ctypes.c_double
        lib.oracle_reshape_and_cache_fp8.argtypes = [p, p, p, p, p, p, p, i32, i32, i32, i32, i32]
        lib.oracle_reshape_and_cache_fp8.restype = ctypes.c_int
        lib.oracle_paged_decode_fp8.argtypes = [p, p, p, p, p, p, i32, p, i32, i32, i32, i32,
                                                i32, i32, ctypes.c_double, p, i64, p, p]
        lib.oracle_paged_decode_fp8.restype = ctypes.c_int
        lib.oracle_paged_decode_multi.argtypes = [p, p, p, p, i32, p, i32, i32, i32, i32, i32,
                                                  i32, i32, ctypes.c_double, p]
        lib.oracle_paged_decode_multi.restype = ctypes.c_int
        lib.oracle_paged_decode_multi_fp8.argtypes = [p, p, p, p, p, p, i32, p, i32, i32, i32,
                                                      i32, i32, i32, i32, ctypes.c_double, p]
        lib.oracle_paged_decode_multi_fp8.restype = ctypes.c_int
        _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Host threads the C oracle's loops use from now on (timing only; every
    unit is computed by one thread, so results do not depend on it)."""
    _load().oracle_set_num_threads(int(n))


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def bf16_bits(x) -> np.ndarray:
    """Accept a numpy uint16/int16 array or a CPU torch bf16 tensor; return uint16 bits."""
    if hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        import torch

        return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(x)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bits as uint16, got {a.dtype}")
    return a


def bf16_to_f64(bits) -> np.ndarray:
    """Exact widening: a bf16 bit pattern is the top half of an IEEE float32."""
    b = bf16_bits(bits)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# decode attention
# --------------------------------------------------------------------------

def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale: Optional[float] = None,
                 units: Optional[Sequence[Tuple[int, int]]] = None, return_lse: bool = False):
    """C oracle. Shapes: q [B][Hq][d], caches [NB][Hkv][BS][d] (bf16 bits),
    block_tables int32 [B][max_blocks], context_lens int32 [B].

    Returns float64 [B][Hq][d], or [n_units][d] when ``units`` is given.
    """
    lib = _load()
    q = bf16_bits(q)
    kc = bf16_bits(k_cache)
    vc = bf16_bits(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, Hq, D = q.shape
    NB, Hkv, BS, D2 = kc.shape
    if D2 != D or vc.shape != kc.shape:
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if units is None:
        u = None
        n = B * Hq
        out = np.empty((B, Hq, D), dtype=np.float64)
    else:
        u = np.ascontiguousarray(np.asarray(units, dtype=np.int32).reshape(-1, 2))
        n = u.shape[0]
        out = np.empty((n, D), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    rc = lib.oracle_paged_decode(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(cl),
                                 B, Hq, Hkv, D, BS, NB, float(scale),
                                 None if u is None else _ptr(u), n, _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_paged_decode failed with code {rc}")
    if return_lse:
        return out, (lse.reshape(B, Hq) if units is None else lse)
    return out


def paged_decode_multi(q, k_cache, v_cache, block_tables, context_lens,
                       scale: Optional[float] = None) -> np.ndarray:
    """Decode of several new tokens per sequence, causal among them (C oracle).
    q [B][query_len][Hq][d] bf16; the last query_len of each sequence's
    context_lens[b] tokens are the queries. Returns float64 [B][query_len][Hq][d]."""
    lib = _load()
    qb = bf16_bits(q)
    kc, vc = bf16_bits(k_cache), bf16_bits(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, QL, Hq, D = qb.shape
    NB, Hkv, BS, D2 = kc.shape
    if D2 != D or vc.shape != kc.shape:
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.empty((B, QL, Hq, D), dtype=np.float64)
    rc = lib.oracle_paged_decode_multi(_ptr(qb), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1],
                                       _ptr(cl), B, QL, Hq, Hkv, D, BS, NB, float(scale), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_paged_decode_multi failed with code {rc}")
    return out


def gather_contiguous(cache_f64: np.ndarray, table_row: np.ndarray, L: int, kv_head: int) -> np.ndarray:
    """Rows 0..L-1 of one sequence's K (or V) for one KV head, in logical order."""
    BS = cache_f64.shape[2]
    t = np.arange(L)
    blk = table_row[t // BS]
    return cache_f64[blk, kv_head, t % BS, :]


def paged_decode_numpy(q, k_cache, v_cache, block_tables, context_lens,
                       scale: Optional[float] = None) -> np.ndarray:
    """Independent numpy twin of ``paged_decode`` (float64)."""
    qd = bf16_to_f64(q)
    kd = bf16_to_f64(k_cache)
    vd = bf16_to_f64(v_cache)
    B, Hq, D = qd.shape
    Hkv = kd.shape[1]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.empty((B, Hq, D), dtype=np.float64)
    for b in range(B):
        L = int(context_lens[b])
        for g in range(Hkv):
            K = gather_contiguous(kd, block_tables[b], L, g)
            V = gather_contiguous(vd, block_tables[b], L, g)
            for h in range(g * G, (g + 1) * G):
                s = (K @ qd[b, h]) * scale
                w = np.exp(s - s.max())
                w /= w.sum()
                out[b, h] = w @ V
    return out


def brute_force_decode(q_rows: List[List[float]], K: List[List[float]], V: List[List[float]],
                       scale: float) -> List[List[float]]:
    """Pure-Python loops over contiguous K/V for one KV head: tiny inputs only.

    q_rows: the query heads that share this KV head; K, V: L rows of d floats.
    """
    out = []
    for qv in q_rows:
        scores = [scale * math.fsum(a * b for a, b in zip(qv, k)) for k in K]
        m = max(scores)
        e = [math.exp(s - m) for s in scores]
        z = math.fsum(e)
        out.append([math.fsum(e[t] / z * V[t][c] for t in range(len(K))) for c in range(len(qv))])
    return out


def partition_decode(q_f64: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float,
                     partition_tokens: int):
    """Split-K model for one (sequence, query head): per partition of
    ``partition_tokens`` consecutive tokens, return (m_p, l_p, acc_p) with
    m_p = max score, l_p = sum exp(s - m_p), acc_p = sum exp(s - m_p) v."""
    L = K.shape[0]
    parts = []
    for start in range(0, L, partition_tokens):
        s = (K[start:start + partition_tokens] @ q_f64) * scale
        m = s.max()
        e = np.exp(s - m)
        parts.append((m, e.sum(), e @ V[start:start + partition_tokens]))
    return parts


def merge_partitions(parts) -> np.ndarray:
    """Log-sum-exp merge: M = max m_p; out = sum e^(m_p-M) acc_p / sum e^(m_p-M) l_p."""
    M = max(p[0] for p in parts)
    num = sum(math.exp(p[0] - M) * p[2] for p in parts)
    den = sum(math.exp(p[0] - M) * p[1] for p in parts)
    return num / den


# --------------------------------------------------------------------------
# cache writes
# --------------------------------------------------------------------------

def reshape_and_cache(k_new, v_new, k_cache, v_cache, slot_mapping) -> Tuple[np.ndarray, np.ndarray]:
    """C oracle byte copy. Returns new (k_cache, v_cache) bit arrays (inputs untouched)."""
    lib = _load()
    kn = bf16_bits(k_new)
    vn = bf16_bits(v_new)
    kc = bf16_bits(k_cache).copy()
    vc = bf16_bits(v_cache).copy()
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    NB, Hkv, BS, D = kc.shape
    rc = lib.oracle_reshape_and_cache(_ptr(kn), _ptr(vn), _ptr(kc), _ptr(vc), _ptr(sm),
                                      sm.shape[0], Hkv, D, BS, NB)
    if rc != 0:
        raise ValueError(f"oracle_reshape_and_cache failed with code {rc}")
    return kc, vc


def copy_blocks(k_cache, v_cache, pairs) -> Tuple[np.ndarray, np.ndarray]:
    """C oracle block copy. Returns new (k_cache, v_cache) bit arrays."""
    lib = _load()
    kc = bf16_bits(k_cache).copy()
    vc = bf16_bits(v_cache).copy()
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    NB, Hkv, BS, D = kc.shape
    rc = lib.oracle_copy_blocks(_ptr(kc), _ptr(vc), _ptr(pr), pr.shape[0], Hkv, D, BS, NB)
    if rc != 0:
        raise ValueError(f"oracle_copy_blocks failed with code {rc}")
    return kc, vc


# --------------------------------------------------------------------------
# 8-bit (FP8 E4M3) KV cache: K [block][head][offset][d], V [block][head][d][offset]
# --------------------------------------------------------------------------

def e4m3_to_f64(codes) -> np.ndarray:
    """Exact value of E4M3 codes (NaN for the two NaN codes)."""
    lib = _load()
    table = np.array([lib.oracle_e4m3_to_double(c) for c in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8)]


def e4m3_from_f32(x) -> np.ndarray:
    """float32 -> E4M3 codes, round to nearest even, saturating (element by element)."""
    lib = _load()
    a = np.asarray(x, dtype=np.float32)
    return np.array([lib.oracle_e4m3_from_float(float(v)) for v in a.reshape(-1)],
                    dtype=np.uint8).reshape(a.shape)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def reshape_and_cache_fp8(k_new, v_new, k_cache, v_cache, slot_mapping, k_scale, v_scale
                          ) -> Tuple[np.ndarray, np.ndarray]:
    """Quantising KV write into an E4M3 cache. Returns new (k_cache, v_cache) uint8 arrays."""
    lib = _load()
    kn, vn = bf16_bits(k_new), bf16_bits(v_new)
    kc = np.ascontiguousarray(k_cache, dtype=np.uint8).copy()
    vc = np.ascontiguousarray(v_cache, dtype=np.uint8).copy()
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    ks, vs = _f32(k_scale), _f32(v_scale)
    NB, Hkv, BS, D = kc.shape
    rc = lib.oracle_reshape_and_cache_fp8(_ptr(kn), _ptr(vn), _ptr(kc), _ptr(vc), _ptr(sm),
                                          _ptr(ks), _ptr(vs), sm.shape[0], Hkv, D, BS, NB)
    if rc != 0:
        raise ValueError(f"oracle_reshape_and_cache_fp8 failed with code {rc}")
    return kc, vc


def paged_decode_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                     scale: Optional[float] = None, units=None):
    """Decode over an E4M3 cache: K/V dequantised exactly (code value x head scale)."""
    lib = _load()
    qb = bf16_bits(q)
    kc = np.ascontiguousarray(k_cache, dtype=np.uint8)
    vc = np.ascontiguousarray(v_cache, dtype=np.uint8)
    ks, vs = _f32(k_scale), _f32(v_scale)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, Hq, D = qb.shape
    NB, Hkv, BS, D2 = kc.shape
    if D2 != D or vc.size != kc.size:  # V^T tiles: [NB][Hkv][D][BS], the same bytes
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if units is None:
        u, n = None, B * Hq
        out = np.empty((B, Hq, D), dtype=np.float64)
    else:
        u = np.ascontiguousarray(np.asarray(units, dtype=np.int32).reshape(-1, 2))
        n = u.shape[0]
        out = np.empty((n, D), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    rc = lib.oracle_paged_decode_fp8(_ptr(qb), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), _ptr(bt),
                                     bt.shape[1], _ptr(cl), B, Hq, Hkv, D, BS, NB, float(scale),
                                     None if u is None else _ptr(u), n, _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_paged_decode_fp8 failed with code {rc}")
    return out


def paged_decode_multi_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                           scale: Optional[float] = None) -> np.ndarray:
    """paged_decode_multi over an E4M3 cache (dequantised exactly, code value x
    head scale). q [B][query_len][Hq][d] bf16; returns float64 of that shape."""
    lib = _load()
    qb = bf16_bits(q)
    kc = np.ascontiguousarray(k_cache, dtype=np.uint8)
    vc = np.ascontiguousarray(v_cache, dtype=np.uint8)
    ks, vs = _f32(k_scale), _f32(v_scale)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, QL, Hq, D = qb.shape
    NB, Hkv, BS, D2 = kc.shape
    if D2 != D or vc.size != kc.size:
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.empty((B, QL, Hq, D), dtype=np.float64)
    rc = lib.oracle_paged_decode_multi_fp8(_ptr(qb), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs),
                                           _ptr(bt), bt.shape[1], _ptr(cl), B, QL, Hq, Hkv, D, BS,
                                           NB, float(scale), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_paged_decode_multi_fp8 failed with code {rc}")
    return out


def copy_blocks_fp8(k_cache, v_cache, pairs) -> Tuple[np.ndarray, np.ndarray]:
    """Block copy of an E4M3 cache (a byte copy of whole blocks, as for bf16)."""
    kc = np.ascontiguousarray(k_cache, dtype=np.uint8)
    vc = np.ascontiguousarray(v_cache, dtype=np.uint8)
    NB, Hkv, BS, D = kc.shape
    k2, v2 = copy_blocks(kc.view(np.uint16), vc.view(np.uint16), pairs)
    return k2.view(np.uint8).reshape(kc.shape), v2.view(np.uint8).reshape(vc.shape)


# --------------------------------------------------------------------------
# block manager reference model
# --------------------------------------------------------------------------

class PoolError(Exception):
    pass


class PoolOOM(PoolError):
    pass


class PoolModel:
    """Reference model of the block manager.

    * Free list: a stack. ``free_order[0]`` is handed out first; a block whose
      reference count drops to zero is pushed on top and is handed out next
      (pop and push are O(1): "How Paged Attention and Continuous Batching
      Actually Work", §Paged attention).
    * Block table: entry i is the physical block backing logical tokens
      [BS*i, BS*i + BS - 1] (PagedAttention architecture page, §The
      architecture: every piece explained).
    * Append: a fresh block is taken when the sequence length is a multiple
      of BS before the append (every 16th token grabs a fresh block, same
      section). If the target block is shared (refcount > 1) the append first
      does copy-on-write: allocate, record (src, dst) for the data copy,
      decrement the old block's refcount, patch this one table entry ("Paged
      Attention as a Memory Manager", §Prefix Caching and Copy-on-Write).
    * Fork: the child points at the parent's first ceil(n/BS) blocks, each
      refcount + 1 ("How Paged Attention ...", §Paged attention -- sharing).
    * Free: the sequence's blocks are released in logical order.
    * Any failing operation leaves the state unchanged.
    * Prefix cache ("How Paged Attention ...", FAQ on prefix caching;
      PagedAttention architecture page, §The architecture and §End-to-end
      flow): a prompt's full blocks are matched in order against the cache
      by their whole token prefix (the exact form of a chained block hash);
      the leading run of matches is shared (refcount + 1), the rest of the
      prompt gets fresh blocks and its full ones enter the cache. A cached
      block freed to refcount 0 stays cached and is handed out only when no
      never-cached block is free, least recently freed first, leaving the
      cache then. A cached block is immutable: an append into it copies it.
    """

    def __init__(self, num_blocks: int, block_size: int, free_order: Optional[Sequence[int]] = None):
        if num_blocks < 1 or block_size < 1:
            raise PoolError("bad pool size")
        order = list(range(num_blocks)) if free_order is None else [int(x) for x in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise PoolError("free_order must be a permutation")
        self.block_size = block_size
        self.num_blocks = num_blocks
        self.free: List[int] = list(reversed(order))  # top of stack = end of list
        self.ref = [0] * num_blocks
        self.tables: Dict[int, List[int]] = {}
        self.lens: Dict[int, int] = {}
        self._next_seq = 0
        self.prefix_of: Dict[int, tuple] = {}   # cached block -> its whole token prefix
        self.block_of: Dict[tuple, int] = {}    # token prefix -> cached block
        self.evictable: List[int] = []          # cached, refcount 0, least recently freed first
        self.lookups = 0
        self.hits = 0

    # ---- blocks
    def alloc(self) -> int:
        if self.free:
            blk = self.free.pop()
        elif self.evictable:
            blk = self.evictable.pop(0)
            del self.block_of[self.prefix_of.pop(blk)]
        else:
            raise PoolOOM("pool exhausted")
        self.ref[blk] = 1
        return blk

    def incref(self, blk: int) -> None:
        self._check_live(blk)
        self.ref[blk] += 1

    def decref(self, blk: int) -> None:
        self._check_live(blk)
        self.ref[blk] -= 1
        if self.ref[blk] == 0:
            if blk in self.prefix_of:
                self.evictable.append(blk)
            else:
                self.free.append(blk)

    def _check_live(self, blk: int) -> None:
        if not (0 <= blk < self.num_blocks):
            raise PoolError("block id out of range")
        if self.ref[blk] <= 0:
            raise PoolError("block is not allocated")

    def stats(self) -> Dict[str, int]:
        used = sum(1 for r in self.ref if r > 0)
        return {"free": len(self.free) + len(self.evictable), "used": used,
                "shared": sum(1 for r in self.ref if r > 1),
                "max_refcount": max(self.ref) if self.ref else 0}

    # ---- sequences
    def seq_create(self) -> int:
        s = self._next_seq
        self._next_seq += 1
        self.tables[s] = []
        self.lens[s] = 0
        return s

    def seq_free(self, s: int) -> None:
        for blk in self.tables.pop(s):
            self.decref(blk)
        del self.lens[s]

    def seq_fork(self, parent: int, num_tokens: int) -> int:
        if not (0 <= num_tokens <= self.lens[parent]):
            raise PoolError("fork length out of range")
        n = -(-num_tokens // self.block_size)
        child = self.seq_create()
        self.tables[child] = list(self.tables[parent][:n])
        self.lens[child] = num_tokens
        for blk in self.tables[child]:
            self.ref[blk] += 1
        return child

    def slot_of(self, s: int, pos: int) -> int:
        """The indexing formula: table[pos // BS] * BS + pos % BS."""
        return self.tables[s][pos // self.block_size] * self.block_size + pos % self.block_size

    def append_slot(self, s: int) -> Tuple[int, Optional[Tuple[int, int]]]:
        """Reserve the slot for the next token. Returns (slot, cow_pair or None)."""
        pos = self.lens[s]
        j = pos // self.block_size
        cow = None
        if pos % self.block_size == 0:
            self.tables[s].append(self.alloc())
        else:
            src = self.tables[s][j]
            if self.ref[src] > 1 or src in self.prefix_of:  # shared, or cached (immutable)
                dst = self.alloc()
                self.decref(src)
                self.tables[s][j] = dst
                cow = (src, dst)
        self.lens[s] = pos + 1
        return self.slot_of(s, pos), cow

    def append_tokens(self, s: int, n: int):
        slots, cows = [], []
        for _ in range(n):
            slot, cow = self.append_slot(s)
            slots.append(slot)
            if cow:
                cows.append(cow)
        return slots, cows

    def create_prompt(self, tokens: Sequence[int]):
        """New sequence holding a prompt. Returns (seq, cached_tokens, slots)."""
        bs = self.block_size
        tokens = [int(t) for t in tokens]
        n = len(tokens)
        nfull, nblocks = n // bs, -(-n // bs)
        matched = []
        for i in range(nfull):
            blk = self.block_of.get(tuple(tokens[:(i + 1) * bs]))
            if blk is None:
                break
            matched.append(blk)
        revive = sum(1 for b in matched if self.ref[b] == 0)
        if nblocks - len(matched) > len(self.free) + len(self.evictable) - revive:
            raise PoolOOM("pool exhausted")
        for b in matched:
            if self.ref[b] == 0:
                self.evictable.remove(b)
            self.ref[b] += 1
        s = self.seq_create()
        table = list(matched)
        for i in range(len(matched), nblocks):
            blk = self.alloc()
            table.append(blk)
            prefix = tuple(tokens[:(i + 1) * bs])
            if i < nfull and prefix not in self.block_of:
                self.block_of[prefix] = blk
                self.prefix_of[blk] = prefix
        self.tables[s] = table
        self.lens[s] = n
        self.lookups += nfull
        self.hits += len(matched)
        return s, len(matched) * bs, [self.slot_of(s, t) for t in range(n)]

    def prefix_stats(self) -> Dict[str, int]:
        return {"cached_blocks": len(self.prefix_of), "evictable_blocks": len(self.evictable),
                "lookups": self.lookups, "hits": self.hits}

    def table(self, s: int) -> List[int]:
        return list(self.tables[s])

    def length(self, s: int) -> int:
        return self.lens[s]


def blocks_needed(num_tokens: int, block_size: int) -> int:
    """ceil(t / BS) ("How Paged Attention ...", §Paged attention)."""
    return -(-num_tokens // block_size)


def all_pairs(B: int, Hq: int):
    return list(itertools.product(range(B), range(Hq)))
