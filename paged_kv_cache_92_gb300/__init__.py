"""Python binding of libpagedkv.so: paged KV-cache decode attention on GB300.

Argument marshalling only. Every step of the data path runs in the CUDA
kernels of ``libpagedkv.so`` (see ``include/pagedkv.h``); torch supplies
device memory and streams. There is no CPU fallback: if the library has not
been built, every call raises.

Names follow the C ABI: ``pa_decode``, ``pa_decode_workspace_size``,
``pa_reshape_and_cache``, ``pa_copy_blocks``, ``pa_device_errors`` and the
``pa_pool_*`` / ``pa_seq_*`` block-pool calls (wrapped by ``Pool``).
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import List, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedkv.so")

PA_OK = 0
STATUS_NAMES = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_OOM",
                4: "PA_ERR_REFCOUNT", 5: "PA_ERR_BOUNDS", 6: "PA_ERR_CUDA"}
DEVERR_TABLE_ENTRY = 0x1
DEVERR_CONTEXT_LEN = 0x2
DEVERR_SLOT = 0x4
DEVERR_COPY_PAIR = 0x8
DEVERR_TIMEOUT = 0x10
DEVERR_APPEND_SLOT = 0x20

KV_BF16 = 0
KV_FP8_E4M3 = 1

EXPORTED_SYMBOLS = [
    "pa_status_string", "pa_last_error", "pa_version", "pa_device_errors",
    "pa_decode_workspace_size", "pa_decode", "pa_decode_noalloc", "pa_append_decode",
    "pa_step_host_layout", "pa_step_host_workspace_size", "pa_step_host",
    "pa_reshape_and_cache", "pa_reshape_and_cache_fp8", "pa_copy_blocks_fp8",
    "pa_copy_blocks",
    "pa_pool_create", "pa_pool_destroy", "pa_pool_alloc", "pa_pool_incref", "pa_pool_decref",
    "pa_pool_refcount", "pa_pool_stats", "pa_seq_create", "pa_seq_free", "pa_seq_fork",
    "pa_seq_append_slot", "pa_seq_append_tokens", "pa_seq_length", "pa_seq_table",
    "pa_pool_export", "pa_seq_create_prompt", "pa_pool_prefix_stats",
]


class PagedKVError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {detail}")


class PoolOOM(PagedKVError):
    pass


class DecodeParams(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("out", ctypes.c_void_p),
        ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("block_tables", ctypes.c_void_p), ("context_lens", ctypes.c_void_p),
        ("max_blocks_per_seq", ctypes.c_int32), ("num_seqs", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32), ("max_context_len", ctypes.c_int32),
        ("scale", ctypes.c_float), ("partition_tokens", ctypes.c_int32),
        ("variant", ctypes.c_int32), ("overlap_prologue", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32), ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("query_len", ctypes.c_int32), ("wait_timeout_us", ctypes.c_int32),
    ]


DECODE_TENSOR_CORE = 0
DECODE_CUDA_CORE = 1


class AppendParams(ctypes.Structure):
    _fields_ = [
        ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
        ("slot_mapping", ctypes.c_void_p),
        ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
    ]


class StepLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in
                ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens",
                 "cow_pairs", "total")]


class StepHostParams(ctypes.Structure):
    _fields_ = [
        ("host_in", ctypes.c_void_p), ("host_out", ctypes.c_void_p),
        ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("num_seqs", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32), ("max_context_len", ctypes.c_int32),
        ("num_cow_pairs", ctypes.c_int32), ("scale", ctypes.c_float), ("variant", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32), ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("query_len", ctypes.c_int32),
    ]


class PrefixStats(ctypes.Structure):
    _fields_ = [("cached_blocks", ctypes.c_int32), ("evictable_blocks", ctypes.c_int32),
                ("lookups", ctypes.c_int64), ("hits", ctypes.c_int64)]


class PoolStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("num_blocks", "block_size", "free_blocks", "used_blocks", "shared_blocks",
                 "max_refcount", "live_seqs")]


_lib = None


def load():
    """Load libpagedkv.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: run paged_kv_cache_92_gb300.build.build() "
                          "(or __graft_entry__.build()) first; there is no fallback path")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    P = ctypes.POINTER
    sigs = {
        "pa_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "pa_last_error": ([], ctypes.c_char_p),
        "pa_version": ([], i32),
        "pa_device_errors": ([vp, P(ctypes.c_uint32)], ctypes.c_int),
        "pa_decode_workspace_size": ([P(DecodeParams)], sz),
        "pa_decode": ([P(DecodeParams), vp, sz, vp], ctypes.c_int),
        "pa_decode_noalloc": ([P(DecodeParams), vp], ctypes.c_int),
        "pa_append_decode": ([P(DecodeParams), P(AppendParams), vp, sz, vp], ctypes.c_int),
        "pa_step_host_layout": ([P(StepHostParams), P(StepLayout)], ctypes.c_int),
        "pa_step_host_workspace_size": ([P(StepHostParams)], sz),
        "pa_step_host": ([P(StepHostParams), vp, sz, vp], ctypes.c_int),
        "pa_reshape_and_cache": ([vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp], ctypes.c_int),
        "pa_copy_blocks": ([vp, vp, vp, i32, i32, i32, i32, i32, vp], ctypes.c_int),
        "pa_reshape_and_cache_fp8": ([vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp],
                                     ctypes.c_int),
        "pa_copy_blocks_fp8": ([vp, vp, vp, i32, i32, i32, i32, i32, vp], ctypes.c_int),
        "pa_pool_create": ([i32, i32, vp, P(vp)], ctypes.c_int),
        "pa_pool_destroy": ([vp], None),
        "pa_pool_alloc": ([vp, P(i32)], ctypes.c_int),
        "pa_pool_incref": ([vp, i32], ctypes.c_int),
        "pa_pool_decref": ([vp, i32], ctypes.c_int),
        "pa_pool_refcount": ([vp, i32], i32),
        "pa_pool_stats": ([vp, P(PoolStats)], ctypes.c_int),
        "pa_seq_create": ([vp, P(i32)], ctypes.c_int),
        "pa_seq_free": ([vp, i32], ctypes.c_int),
        "pa_seq_fork": ([vp, i32, i32, P(i32)], ctypes.c_int),
        "pa_seq_append_slot": ([vp, i32, P(i64), P(i32), P(i32)], ctypes.c_int),
        "pa_seq_append_tokens": ([vp, i32, i32, vp, vp, P(i32)], ctypes.c_int),
        "pa_seq_length": ([vp, i32, P(i32)], ctypes.c_int),
        "pa_seq_table": ([vp, i32, vp, i32, P(i32)], ctypes.c_int),
        "pa_pool_export": ([vp, vp, i32, i32, vp, vp], ctypes.c_int),
        "pa_seq_create_prompt": ([vp, vp, i32, P(i32), P(i32), vp], ctypes.c_int),
        "pa_pool_prefix_stats": ([vp, P(PrefixStats)], ctypes.c_int),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _check(status: int, where: str) -> None:
    if status != PA_OK:
        detail = load().pa_last_error().decode(errors="replace")
        cls = PoolOOM if status == 3 else PagedKVError
        raise cls(status, where, detail)


# --------------------------------------------------------------------------
# device calls (torch tensors in, marshalled to raw pointers)
# --------------------------------------------------------------------------

def _dev_ptr(t, dtype, name: str) -> int:
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def make_decode_params(q, out, k_cache, v_cache, block_tables, context_lens,
                       max_context_len: int, scale: Optional[float] = None,
                       partition_tokens: int = 0, variant: int = DECODE_TENSOR_CORE,
                       overlap_prologue: bool = False, k_scale=None,
                       v_scale=None, wait_timeout_us: int = 0) -> DecodeParams:
    """Marshal a pa_decode call. q and out are bf16 [B][Hq][D] (one new token
    per sequence) or [B][Q][Hq][D] (Q new tokens per sequence, causal among
    them). bf16 caches [NB][Hkv][BS][D]; uint8 caches are the 8-bit E4M3 cache
    (K [NB][Hkv][BS][D], V^T in 16-key sub-tiles [NB][Hkv][BS/16][D][16]) and
    need k_scale / v_scale, float32 CUDA tensors [Hkv]."""
    import torch

    if q.dim() == 4:
        B, QL, Hq, D = q.shape
    else:
        (B, Hq, D), QL = q.shape, 0
    fp8 = k_cache.dtype == torch.uint8
    NB, Hkv, BS, D2 = k_cache.shape
    v_ok = tuple(v_cache.shape) in fp8_v_shapes(NB, Hkv, BS, D2) if fp8 else \
        tuple(v_cache.shape) == tuple(k_cache.shape)
    if D2 != D or not v_ok or tuple(out.shape) != tuple(q.shape):
        raise ValueError("shape mismatch between q / out / k_cache / v_cache")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or tuple(context_lens.shape) != (B,):
        raise ValueError("block_tables must be [num_seqs][max_blocks], context_lens [num_seqs]")
    p = DecodeParams()
    p.q = _dev_ptr(q, torch.bfloat16, "q")
    p.out = _dev_ptr(out, torch.bfloat16, "out")
    cache_dtype = torch.uint8 if fp8 else torch.bfloat16
    p.k_cache = _dev_ptr(k_cache, cache_dtype, "k_cache")
    p.v_cache = _dev_ptr(v_cache, cache_dtype, "v_cache")
    if fp8:
        if k_scale is None or v_scale is None:
            raise ValueError("the 8-bit cache needs k_scale and v_scale")
        p.kv_dtype = KV_FP8_E4M3
        p.k_scale = _dev_ptr(k_scale, torch.float32, "k_scale")
        p.v_scale = _dev_ptr(v_scale, torch.float32, "v_scale")
    p.block_tables = _dev_ptr(block_tables, torch.int32, "block_tables")
    p.context_lens = _dev_ptr(context_lens, torch.int32, "context_lens")
    p.max_blocks_per_seq = block_tables.shape[1]
    p.num_seqs, p.num_q_heads, p.num_kv_heads = B, Hq, Hkv
    p.head_dim, p.block_size, p.num_blocks = D, BS, NB
    p.max_context_len = int(max_context_len)
    p.scale = float(1.0 / math.sqrt(D) if scale is None else scale)
    p.partition_tokens = int(partition_tokens)
    p.variant = int(variant)
    p.overlap_prologue = int(bool(overlap_prologue))
    p.query_len = int(QL)
    p.wait_timeout_us = int(wait_timeout_us)
    return p


def pa_decode_workspace_size(params: DecodeParams) -> int:
    return int(load().pa_decode_workspace_size(ctypes.byref(params)))


def pa_decode(q, k_cache, v_cache, block_tables, context_lens, max_context_len: int,
              scale: Optional[float] = None, partition_tokens: int = 0, out=None,
              workspace=None, stream=None, variant: int = DECODE_TENSOR_CORE,
              overlap_prologue: bool = False, k_scale=None, v_scale=None,
              wait_timeout_us: int = 0):
    """Paged decode attention; returns ``out`` (bf16, the shape of ``q``:
    [B][Hq][d], or [B][Q][Hq][d] for Q new tokens per sequence).

    ``workspace`` is a uint8 CUDA tensor of at least
    ``pa_decode_workspace_size`` bytes; allocated here when omitted.
    """
    import torch

    lib = load()
    if out is None:
        out = torch.empty_like(q)
    p = make_decode_params(q, out, k_cache, v_cache, block_tables, context_lens,
                           max_context_len, scale, partition_tokens, variant, overlap_prologue,
                           k_scale, v_scale, wait_timeout_us)
    need = int(lib.pa_decode_workspace_size(ctypes.byref(p)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _dev_ptr(workspace, torch.uint8, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() if workspace is not None else 0
    _check(lib.pa_decode(ctypes.byref(p), ws_ptr, ws_bytes, _stream_handle(stream)), "pa_decode")
    return out


def make_append_params(k_new, v_new, slot_mapping, k_cache, v_cache) -> AppendParams:
    import torch

    T, Hkv, D = k_new.shape  # T = num_seqs * (new tokens per sequence)
    if tuple(v_new.shape) != (T, Hkv, D) or tuple(slot_mapping.shape) != (T,) \
            or tuple(k_cache.shape[1:2]) != (Hkv,) or k_cache.shape[3] != D:
        raise ValueError("k_new/v_new must be [num_seqs * Q][num_kv_heads][head_dim] matching "
                         "the cache, slot_mapping [num_seqs * Q]")
    a = AppendParams()
    a.k_new = _dev_ptr(k_new, torch.bfloat16, "k_new")
    a.v_new = _dev_ptr(v_new, torch.bfloat16, "v_new")
    a.slot_mapping = _dev_ptr(slot_mapping, torch.int64, "slot_mapping")
    cache_dtype = torch.uint8 if k_cache.dtype == torch.uint8 else torch.bfloat16
    a.k_cache = _dev_ptr(k_cache, cache_dtype, "k_cache")
    a.v_cache = _dev_ptr(v_cache, cache_dtype, "v_cache")
    return a


def pa_append_decode(q, k_cache, v_cache, block_tables, context_lens, max_context_len: int,
                     k_new, v_new, slot_mapping, scale: Optional[float] = None,
                     partition_tokens: int = 0, out=None, workspace=None, stream=None,
                     variant: int = DECODE_TENSOR_CORE, overlap_prologue: bool = False,
                     k_scale=None, v_scale=None):
    """One decode step in one launch: write token b's K/V (``k_new[b]``,
    ``v_new[b]``) at ``slot_mapping[b]`` -- which must be the slot of token
    ``context_lens[b] - 1`` of sequence b -- then paged decode attention over
    the updated caches. Same result as ``pa_reshape_and_cache`` followed by
    ``pa_decode``; returns ``out``. With q [B][Q][Hq][d], row b*Q + i of
    ``k_new``/``v_new``/``slot_mapping`` is token ``context_lens[b] - Q + i``.
    For the 8-bit cache (uint8 caches, with ``k_scale``/``v_scale``) the write
    is the quantising one of ``pa_reshape_and_cache_fp8``."""
    import torch

    lib = load()
    if out is None:
        out = torch.empty_like(q)
    p = make_decode_params(q, out, k_cache, v_cache, block_tables, context_lens,
                           max_context_len, scale, partition_tokens, variant, overlap_prologue,
                           k_scale, v_scale)
    a = make_append_params(k_new, v_new, slot_mapping, k_cache, v_cache)
    need = int(lib.pa_decode_workspace_size(ctypes.byref(p)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _dev_ptr(workspace, torch.uint8, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() if workspace is not None else 0
    _check(lib.pa_append_decode(ctypes.byref(p), ctypes.byref(a), ws_ptr, ws_bytes,
                                _stream_handle(stream)), "pa_append_decode")
    return out


def make_step_host_params(k_cache, v_cache, num_seqs: int, num_q_heads: int,
                          max_blocks_per_seq: int, max_context_len: int, num_cow_pairs: int = 0,
                          scale: Optional[float] = None,
                          variant: int = DECODE_TENSOR_CORE, k_scale=None,
                          v_scale=None, query_len: int = 0) -> StepHostParams:
    """Shape half of a host-driven step; host_in / host_out are set by the caller
    (or by ``pa_step_host``). uint8 caches are the 8-bit (E4M3) cache and need
    ``k_scale`` / ``v_scale`` (float32 CUDA tensors [num_kv_heads]). With
    ``query_len`` Q > 1 every sequence brings Q new tokens (the layouts of
    ``pa_append_decode``)."""
    import torch

    NB, Hkv, BS, D = k_cache.shape
    p = StepHostParams()
    fp8 = k_cache.dtype == torch.uint8
    cache_dtype = torch.uint8 if fp8 else torch.bfloat16
    p.k_cache = _dev_ptr(k_cache, cache_dtype, "k_cache")
    p.v_cache = _dev_ptr(v_cache, cache_dtype, "v_cache")
    if fp8:
        if k_scale is None or v_scale is None:
            raise ValueError("the 8-bit cache needs k_scale and v_scale")
        p.kv_dtype = KV_FP8_E4M3
        p.k_scale = _dev_ptr(k_scale, torch.float32, "k_scale")
        p.v_scale = _dev_ptr(v_scale, torch.float32, "v_scale")
    p.num_seqs, p.num_q_heads, p.num_kv_heads, p.head_dim = num_seqs, num_q_heads, Hkv, D
    p.block_size, p.num_blocks = BS, NB
    p.max_blocks_per_seq, p.max_context_len = max_blocks_per_seq, int(max_context_len)
    p.num_cow_pairs = num_cow_pairs
    p.scale = float(1.0 / math.sqrt(D) if scale is None else scale)
    p.variant = int(variant)
    p.query_len = int(query_len)
    return p


def pa_step_host_layout(params: StepHostParams) -> StepLayout:
    out = StepLayout()
    _check(load().pa_step_host_layout(ctypes.byref(params), ctypes.byref(out)),
           "pa_step_host_layout")
    return out


def pa_step_host_workspace_size(params: StepHostParams) -> int:
    return int(load().pa_step_host_workspace_size(ctypes.byref(params)))


def pack_step_inputs(params: StepHostParams, q, k_new, v_new, slot_mapping, block_tables,
                     context_lens, cow_pairs=None, pin: bool = True):
    """Marshal one step's host inputs into the packed buffer of ``pa_step_host``
    (a uint8 CPU tensor; pinned unless ``pin`` is False)."""
    import torch

    L = pa_step_host_layout(params)
    buf = torch.zeros(int(L.total), dtype=torch.uint8, pin_memory=pin)
    parts = [(L.q, q, torch.bfloat16), (L.k_new, k_new, torch.bfloat16),
             (L.v_new, v_new, torch.bfloat16), (L.slot_mapping, slot_mapping, torch.int64),
             (L.block_tables, block_tables, torch.int32), (L.context_lens, context_lens, torch.int32)]
    if params.num_cow_pairs:
        parts.append((L.cow_pairs, cow_pairs, torch.int32))
    for off, t, dt in parts:
        t = torch.as_tensor(t).to("cpu", dt).contiguous().view(torch.uint8).reshape(-1)
        buf[int(off):int(off) + t.numel()] = t
    return buf


def pa_step_host(params: StepHostParams, host_in, host_out, workspace, stream=None) -> None:
    """One whole step from host memory (see the C header): ``host_in`` is a
    uint8 CPU tensor packed by ``pa_step_host_layout`` (pinned for speed),
    ``host_out`` a bf16 CPU tensor [num_seqs][num_q_heads][head_dim] (with Q new
    tokens per sequence [num_seqs][Q][num_q_heads][head_dim]),
    ``workspace`` a uint8 CUDA tensor. Returns when host_out holds the result."""
    import torch

    if host_in.device.type != "cpu" or host_out.device.type != "cpu":
        raise ValueError("host_in and host_out must be host (CPU) tensors")
    if not host_in.is_contiguous() or not host_out.is_contiguous():
        raise ValueError("host_in and host_out must be contiguous")
    if host_out.dtype != torch.bfloat16 or host_in.dtype != torch.uint8:
        raise ValueError("host_in must be uint8, host_out bf16")
    params.host_in = host_in.data_ptr()
    params.host_out = host_out.data_ptr()
    ws = _dev_ptr(workspace, torch.uint8, "workspace")
    _check(load().pa_step_host(ctypes.byref(params), ws, workspace.numel(),
                               _stream_handle(stream)), "pa_step_host")


def pa_decode_noalloc(q, k_cache, v_cache, block_tables, context_lens, max_context_len: int,
                      scale: Optional[float] = None, partition_tokens: int = 0, out=None,
                      stream=None, variant: int = DECODE_TENSOR_CORE):
    """Same decode as ``pa_decode`` without any workspace: for callers that
    cannot allocate device memory at decode time (all free HBM already handed
    to the KV pool, or no room for cudaMalloc's synchronisation in the serving
    loop). The split-K partials live in a fixed 16 MiB device array inside the
    library; larger needs are rejected. ``out`` must be given by such callers;
    when omitted it is allocated here for convenience. Calls that overlap on
    the GPU share that array and race."""
    import torch

    lib = load()
    if out is None:
        out = torch.empty_like(q)
    p = make_decode_params(q, out, k_cache, v_cache, block_tables, context_lens,
                           max_context_len, scale, partition_tokens, variant)
    _check(lib.pa_decode_noalloc(ctypes.byref(p), _stream_handle(stream)), "pa_decode_noalloc")
    return out


def pa_reshape_and_cache(k_new, v_new, k_cache, v_cache, slot_mapping, stream=None) -> None:
    import torch

    T, Hkv, D = k_new.shape
    NB, Hkv2, BS, D2 = k_cache.shape
    if (Hkv2, D2) != (Hkv, D) or tuple(v_new.shape) != tuple(k_new.shape) \
            or tuple(v_cache.shape) != tuple(k_cache.shape) or tuple(slot_mapping.shape) != (T,):
        raise ValueError("shape mismatch in pa_reshape_and_cache")
    lib = load()
    _check(lib.pa_reshape_and_cache(
        _dev_ptr(k_new, torch.bfloat16, "k_new"), _dev_ptr(v_new, torch.bfloat16, "v_new"),
        _dev_ptr(k_cache, torch.bfloat16, "k_cache"), _dev_ptr(v_cache, torch.bfloat16, "v_cache"),
        _dev_ptr(slot_mapping, torch.int64, "slot_mapping"), T, Hkv, D, BS, NB,
        _stream_handle(stream)), "pa_reshape_and_cache")


def pa_copy_blocks(k_cache, v_cache, pairs, stream=None) -> None:
    import torch

    NB, Hkv, BS, D = k_cache.shape
    if pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs must be int32 [n][2]")
    lib = load()
    _check(lib.pa_copy_blocks(
        _dev_ptr(k_cache, torch.bfloat16, "k_cache"), _dev_ptr(v_cache, torch.bfloat16, "v_cache"),
        _dev_ptr(pairs, torch.int32, "pairs"), pairs.shape[0], Hkv, D, BS, NB,
        _stream_handle(stream)), "pa_copy_blocks")


def fp8_v_shapes(NB: int, Hkv: int, BS: int, D: int):
    """Shapes accepted for the 8-bit V^T cache: [NB][Hkv][BS/W][D][W] (sub-tiles
    of W = min(BS, 16) keys), and up to block size 16 also [NB][Hkv][D][W]."""
    W = min(BS, 16)
    shapes = [(NB, Hkv, BS // W, D, W)]
    if BS <= 16:
        shapes.append((NB, Hkv, D, W))
    return shapes


def pa_reshape_and_cache_fp8(k_new, v_new, k_cache, v_cache, slot_mapping, k_scale, v_scale,
                             stream=None) -> None:
    """KV write into the 8-bit cache (uint8 K [NB][Hkv][BS][D], V^T in sub-tiles
    of W = min(BS, 16) keys, [NB][Hkv][BS/W][D][W])."""
    import torch

    T, Hkv, D = k_new.shape
    NB, Hkv2, BS, D2 = k_cache.shape
    if (Hkv2, D2) != (Hkv, D) or tuple(v_new.shape) != tuple(k_new.shape) \
            or tuple(v_cache.shape) not in fp8_v_shapes(NB, Hkv, BS, D) \
            or tuple(slot_mapping.shape) != (T,):
        raise ValueError("shape mismatch in pa_reshape_and_cache_fp8")
    lib = load()
    _check(lib.pa_reshape_and_cache_fp8(
        _dev_ptr(k_new, torch.bfloat16, "k_new"), _dev_ptr(v_new, torch.bfloat16, "v_new"),
        _dev_ptr(k_cache, torch.uint8, "k_cache"), _dev_ptr(v_cache, torch.uint8, "v_cache"),
        _dev_ptr(slot_mapping, torch.int64, "slot_mapping"),
        _dev_ptr(k_scale, torch.float32, "k_scale"), _dev_ptr(v_scale, torch.float32, "v_scale"),
        T, Hkv, D, BS, NB, _stream_handle(stream)), "pa_reshape_and_cache_fp8")


def pa_copy_blocks_fp8(k_cache, v_cache, pairs, stream=None) -> None:
    import torch

    NB, Hkv, BS, D = k_cache.shape
    if pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs must be int32 [n][2]")
    lib = load()
    _check(lib.pa_copy_blocks_fp8(
        _dev_ptr(k_cache, torch.uint8, "k_cache"), _dev_ptr(v_cache, torch.uint8, "v_cache"),
        _dev_ptr(pairs, torch.int32, "pairs"), pairs.shape[0], Hkv, D, BS, NB,
        _stream_handle(stream)), "pa_copy_blocks_fp8")


def pa_device_errors(stream=None) -> int:
    flags = ctypes.c_uint32(0)
    _check(load().pa_device_errors(_stream_handle(stream), ctypes.byref(flags)), "pa_device_errors")
    return int(flags.value)


# --------------------------------------------------------------------------
# host block pool
# --------------------------------------------------------------------------

class Pool:
    """Host block pool (``pa_pool_*`` / ``pa_seq_*``). Free list is a stack seeded
    from ``free_order`` (first element handed out first)."""

    def __init__(self, num_blocks: int, block_size: int = 16,
                 free_order: Optional[Sequence[int]] = None):
        self._lib = load()
        self._h = ctypes.c_void_p()
        order = None
        if free_order is not None:
            order = np.ascontiguousarray(np.asarray(free_order, dtype=np.int32))
        _check(self._lib.pa_pool_create(num_blocks, block_size,
                                        None if order is None else order.ctypes.data,
                                        ctypes.byref(self._h)), "pa_pool_create")
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self) -> None:
        if self._h:
            self._lib.pa_pool_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def alloc(self) -> int:
        b = ctypes.c_int32()
        _check(self._lib.pa_pool_alloc(self._h, ctypes.byref(b)), "pa_pool_alloc")
        return b.value

    def incref(self, blk: int) -> None:
        _check(self._lib.pa_pool_incref(self._h, blk), "pa_pool_incref")

    def decref(self, blk: int) -> None:
        _check(self._lib.pa_pool_decref(self._h, blk), "pa_pool_decref")

    def refcount(self, blk: int) -> int:
        return int(self._lib.pa_pool_refcount(self._h, blk))

    def stats(self) -> dict:
        st = PoolStats()
        _check(self._lib.pa_pool_stats(self._h, ctypes.byref(st)), "pa_pool_stats")
        return {n: getattr(st, n) for n, _ in PoolStats._fields_}

    def seq_create(self) -> int:
        s = ctypes.c_int32()
        _check(self._lib.pa_seq_create(self._h, ctypes.byref(s)), "pa_seq_create")
        return s.value

    def seq_free(self, seq: int) -> None:
        _check(self._lib.pa_seq_free(self._h, seq), "pa_seq_free")

    def seq_fork(self, parent: int, num_tokens: int) -> int:
        c = ctypes.c_int32()
        _check(self._lib.pa_seq_fork(self._h, parent, num_tokens, ctypes.byref(c)), "pa_seq_fork")
        return c.value

    def append_slot(self, seq: int) -> Tuple[int, Optional[Tuple[int, int]]]:
        slot = ctypes.c_int64()
        pair = (ctypes.c_int32 * 2)()
        has = ctypes.c_int32()
        _check(self._lib.pa_seq_append_slot(self._h, seq, ctypes.byref(slot), pair,
                                            ctypes.byref(has)), "pa_seq_append_slot")
        return slot.value, ((pair[0], pair[1]) if has.value else None)

    def append_tokens(self, seq: int, n: int, want_slots: bool = True):
        slots = np.empty(max(n, 1), dtype=np.int64)
        pairs = np.empty((max(n, 1), 2), dtype=np.int32)
        ncow = ctypes.c_int32()
        _check(self._lib.pa_seq_append_tokens(
            self._h, seq, n, slots.ctypes.data if want_slots else None, pairs.ctypes.data,
            ctypes.byref(ncow)), "pa_seq_append_tokens")
        return (slots[:n].tolist() if want_slots else None,
                [tuple(int(x) for x in r) for r in pairs[:ncow.value]])

    def length(self, seq: int) -> int:
        n = ctypes.c_int32()
        _check(self._lib.pa_seq_length(self._h, seq, ctypes.byref(n)), "pa_seq_length")
        return n.value

    def table(self, seq: int) -> List[int]:
        n = ctypes.c_int32()
        _check(self._lib.pa_seq_table(self._h, seq, None, 0, ctypes.byref(n)), "pa_seq_table")
        buf = np.empty(max(n.value, 1), dtype=np.int32)
        _check(self._lib.pa_seq_table(self._h, seq, buf.ctypes.data, buf.shape[0],
                                      ctypes.byref(n)), "pa_seq_table")
        return buf[:n.value].tolist()

    def export(self, seqs: Sequence[int], max_blocks: int):
        s = np.ascontiguousarray(np.asarray(seqs, dtype=np.int32))
        tables = np.empty((len(s), max_blocks), dtype=np.int32)
        lens = np.empty(len(s), dtype=np.int32)
        _check(self._lib.pa_pool_export(self._h, s.ctypes.data, len(s), max_blocks,
                                        tables.ctypes.data, lens.ctypes.data), "pa_pool_export")
        return tables, lens

    def create_prompt(self, tokens: Sequence[int]):
        """New sequence holding a prompt, its leading full blocks mapped from the
        prefix cache. Returns (seq, cached_tokens, slots)."""
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        seq, cached = ctypes.c_int32(), ctypes.c_int32()
        slots = np.empty(max(len(t), 1), dtype=np.int64)
        _check(self._lib.pa_seq_create_prompt(self._h, t.ctypes.data if len(t) else None, len(t),
                                              ctypes.byref(seq), ctypes.byref(cached),
                                              slots.ctypes.data), "pa_seq_create_prompt")
        return seq.value, cached.value, slots[:len(t)].tolist()

    def prefix_stats(self) -> dict:
        st = PrefixStats()
        _check(self._lib.pa_pool_prefix_stats(self._h, ctypes.byref(st)), "pa_pool_prefix_stats")
        return {"cached_blocks": st.cached_blocks, "evictable_blocks": st.evictable_blocks,
                "lookups": st.lookups, "hits": st.hits}
