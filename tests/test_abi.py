"""CPU checks of the C ABI: the library loads, exports every symbol that
include/pagedkv.h declares, and rejects bad host-side arguments before any
launch (no GPU is touched by these calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_92_gb300 import build

    build.build()
    import paged_kv_cache_92_gb300 as pk

    pk.load()
    return pk


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_header_declares_the_expected_calls(pk):
    declared = _declared_functions()
    assert set(declared) == set(pk.EXPORTED_SYMBOLS)
    for name in ("pa_decode", "pa_reshape_and_cache", "pa_copy_blocks", "pa_pool_create",
                 "pa_seq_append_slot"):
        assert name in declared


def test_library_exports_every_declared_symbol(pk):
    lib = ctypes.CDLL(pk.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert pk.load().pa_version() == 1


def test_status_strings(pk):
    lib = pk.load()
    for code, name in pk.STATUS_NAMES.items():
        assert lib.pa_status_string(code).decode() == name


def _params(pk, **kw):
    p = pk.DecodeParams()
    base = dict(max_blocks_per_seq=4, num_seqs=2, num_q_heads=8, num_kv_heads=2, head_dim=128,
                block_size=16, num_blocks=8, max_context_len=64, scale=0.088, partition_tokens=0)
    base.update(kw)
    for k, v in base.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), 2),
    (dict(block_size=64), 2),
    (dict(block_size=32), 1),  # block size 32: tensor-core kernel, valid shapes, NULL pointers
    (dict(block_size=8), 1),
    (dict(block_size=32, head_dim=64), 1),  # block sizes 8 and 32 at head_dim 64: bf16
    # the 8-bit cache at block size 8 and head_dim 64: the CUDA-core kernel (NULL pointers)
    (dict(block_size=8, head_dim=64, kv_dtype=1), 1),
    (dict(kv_dtype=1, variant=1), 1),
    (dict(kv_dtype=1, head_dim=64), 1),
    (dict(kv_dtype=1, variant=1, block_size=32), 1),
    (dict(block_size=8, variant=1), 1),  # block sizes 8 and 32 on the CUDA-core kernel too
    (dict(block_size=8, query_len=4), 1),  # block size 8: column groups of 8 per KV head
    (dict(block_size=8, kv_dtype=1), 1),
    (dict(num_q_heads=12, num_kv_heads=1), 2),
    (dict(num_q_heads=6, num_kv_heads=4), 1),
    (dict(max_context_len=0), 1),
    (dict(partition_tokens=24), 1),
    (dict(partition_tokens=8192), 1),
    (dict(scale=0.0), 1),
    (dict(num_seqs=70000), 1),
    (dict(variant=2), 1),
    (dict(num_blocks=1 << 24, num_kv_heads=8), 1),  # cache rows past 2^31
    (dict(query_len=-1), 1),
    (dict(query_len=2000), 1),
    (dict(query_len=3, num_q_heads=16, num_kv_heads=2), 1),  # two column groups (G 8)
    (dict(query_len=2, variant=1), 1),  # several new tokens on the CUDA-core kernel too
    (dict(query_len=1024, num_seqs=70, variant=1), 2),  # ... up to 65535 (sequence, token) rows
    (dict(query_len=4, num_q_heads=64, num_kv_heads=8, kv_dtype=1), 1),  # groups of one token
    # more virtual sequences (sequences x column groups) than the tensor-core
    # plan holds: the CUDA-core kernel takes them (40 x 1024 rows) ...
    (dict(query_len=1024, num_seqs=40, num_q_heads=64, num_kv_heads=8), 1),
    # ... and no more than 65535 rows
    (dict(query_len=1024, num_seqs=70, num_q_heads=64, num_kv_heads=8), 2),
    (dict(query_len=4), 1),  # valid shapes (G 4, 16 columns per KV head), NULL pointers
    (dict(), 1),  # valid shapes, NULL pointers
])
def test_decode_rejects_bad_arguments_on_the_host(pk, kw, status):
    lib = pk.load()
    p = _params(pk, **kw)
    assert lib.pa_decode(ctypes.byref(p), None, 0, None) == status
    assert lib.pa_last_error()


def _ru(x):
    return (x + 255) // 256 * 256


def _groups(Hq, Hkv, QL, cols_total=128, cols_head=16):
    """Tokens per column group and groups: G x (tokens rounded up to a power
    of two) <= cols_head columns per KV head and Hkv x that <= cols_total."""
    if QL <= 1:
        return 1, 1
    G = Hq // Hkv
    cols = min(cols_head, cols_total // Hkv)
    cap = cols // G
    qg = QL if QL <= cap else cap
    return qg, -(-QL // qg)


def _expected_ws(B, Hq, D, parts, grid, Hkv=None, QL=1, variant=0):
    """The workspace of the kernel that will run. Tensor-core kernel (variant
    0): the stream-K plan and the partials per (sequence + CTA) and query
    column, Hkv * G * (QL rounded up to a power of two) columns; with QL > 1
    the bf16 queries are also staged in column order, [B][N][D] with N the
    columns padded to 16/32/64/128. CUDA-core kernel (variant 1): the
    per-partition partials of every (sequence, new token) row, when a
    sequence can split."""
    if variant == 1:
        simt = 0
        if parts > 1:
            rows = B * QL * Hq * parts
            simt = 2 * _ru(rows * 4) + _ru(rows * D * 4)
        return 256 + simt
    qg, ng = _groups(Hq, Hkv or 2, QL)
    V = B * ng  # virtual sequences
    qlp = 1
    while qlp < qg:
        qlp *= 2
    cols = Hq * qlp
    rows = (V + grid) * cols
    tc = _ru((V + 2) * 4) + 2 * _ru(rows * 4) + _ru(rows * D * 4)
    if QL > 1:
        n_pad = next(n for n in (16, 32, 64, 128) if cols <= n)
        tc += _ru(V * n_pad * D * 2)
    return 256 + tc


def test_decode_workspace_size(pk):
    """Header + the workspace of the kernel the parameters select: the
    tensor-core plan + per-(sequence, SM) partials, or the CUDA-core
    per-partition partials. Without a GPU the SM count used for sizing is
    256."""
    lib = pk.load()
    got = lib.pa_decode_workspace_size(ctypes.byref(_params(pk)))
    assert got == _expected_ws(2, 8, 128, 1, 256)
    p = _params(pk, max_context_len=2048, max_blocks_per_seq=128)
    assert lib.pa_decode_workspace_size(ctypes.byref(p)) == _expected_ws(2, 8, 128, 4, 256)
    p = _params(pk, num_seqs=64, num_q_heads=32, num_kv_heads=8, max_context_len=32768,
                max_blocks_per_seq=2048)
    assert lib.pa_decode_workspace_size(ctypes.byref(p)) == _expected_ws(64, 32, 128, 64, 256)
    assert lib.pa_decode_workspace_size(ctypes.byref(_params(pk, head_dim=96))) == 0
    # the CUDA-core variant sizes its own partials only
    for mx, parts in ((64, 1), (2048, 4), (32768, 64)):
        p = _params(pk, num_seqs=64, num_q_heads=32, num_kv_heads=8, max_context_len=mx,
                    max_blocks_per_seq=2048, variant=1)
        assert lib.pa_decode_workspace_size(ctypes.byref(p)) == _expected_ws(64, 32, 128, parts,
                                                                             256, variant=1)
    # the 70B-class batch of 32 (64/8 heads, contexts up to 32768): only the
    # tensor-core kernel's partials, far below the CUDA-core kernel's
    # 32 x 64 x 64 partitions x 130 floats
    p = _params(pk, num_seqs=32, num_q_heads=64, num_kv_heads=8, max_context_len=32769,
                max_blocks_per_seq=2049)
    tc = lib.pa_decode_workspace_size(ctypes.byref(p))
    assert tc == _expected_ws(32, 64, 128, 65, 256)
    assert tc < 12 * 1024 * 1024
    p.variant = 1
    assert lib.pa_decode_workspace_size(ctypes.byref(p)) == _expected_ws(32, 64, 128, 65, 256,
                                                                         variant=1)
    # a shape the tensor-core kernel does not take runs on the CUDA-core one,
    # whatever the variant says, and is sized for it
    p = _params(pk, num_q_heads=16, num_kv_heads=16, max_context_len=2048,
                max_blocks_per_seq=128)
    assert lib.pa_decode_workspace_size(ctypes.byref(p)) == _expected_ws(2, 16, 128, 4, 256,
                                                                         variant=1)
    # several new tokens per sequence
    for ql in (2, 3, 4):
        p = _params(pk, query_len=ql)
        assert lib.pa_decode_workspace_size(ctypes.byref(p)) == _expected_ws(2, 8, 128, 1, 256,
                                                                             QL=ql)
    p = _params(pk, num_seqs=64, num_q_heads=32, num_kv_heads=8, max_context_len=2048,
                max_blocks_per_seq=128, query_len=2)
    assert lib.pa_decode_workspace_size(ctypes.byref(p)) == _expected_ws(64, 32, 128, 4, 256,
                                                                         Hkv=8, QL=2)
    # more new tokens than one column group holds: the query-major kernel, its
    # keys unsplit for contexts under 4 chunks (the header only) ...
    for ql in (8, 9, 64):
        p = _params(pk, query_len=ql)
        assert lib.pa_decode_workspace_size(ctypes.byref(p)) == 256
    # ... and split over up to 16 CTAs for small batches: 8 sequences x 4 head
    # pairs = 32 units, 8 splits; partials (m, l) then O rows per (row, split)
    p = _params(pk, num_seqs=8, num_q_heads=32, num_kv_heads=8, max_context_len=2048,
                max_blocks_per_seq=128, query_len=16)
    rows = 8 * 16 * 32 * 8
    assert lib.pa_decode_workspace_size(ctypes.byref(p)) == 256 + rows * 2 * 4 + rows * 128 * 4
    # 64 sequences x 4 head pairs = 256 units: no split, the header only
    p.num_seqs = 64
    assert lib.pa_decode_workspace_size(ctypes.byref(p)) == 256
    p.query_len = 4  # one column group but 16 rows per KV head: query-major as well
    assert lib.pa_decode_workspace_size(ctypes.byref(p)) == 256
    p.query_len = 3  # 12 rows per KV head in one column group: the column-layout decode
    assert lib.pa_decode_workspace_size(ctypes.byref(p)) == _expected_ws(64, 32, 128, 4, 256,
                                                                         Hkv=8, QL=3)
    # several new tokens on the CUDA-core kernel: partials per (sequence, token)
    for ql in (2, 7):
        p = _params(pk, query_len=ql, max_context_len=2048, max_blocks_per_seq=128, variant=1)
        assert lib.pa_decode_workspace_size(ctypes.byref(p)) == _expected_ws(2, 8, 128, 4, 256,
                                                                             QL=ql, variant=1)


def _query_major_plan(B, Hq, Hkv, QL, mx, bs=16, variant=0, kv_dtype=0, D=128):
    """Whether the many-token kernel takes a shape, and its key splits.

    Restated from the kernel's launch rules: a KV head has QL x G query rows,
    tiled by 128; a work item holds two KV heads when their rows fit 64 and
    the head count is even, else one. The kernel takes bf16 head_dim 128 at
    block size 16 or 32, G in {1, 2, 4, 8}, several new tokens, and either
    more tokens than one column group of the column-layout decode holds
    (16 columns per KV head, at most 128 over all KV heads, G per token) or
    at least 16 rows per KV head with 128 (sequence, KV head, tile) units.
    Small batches split each item's keys to reach 256 items, every split
    at least 4 chunks of 64 / heads-per-item keys, at most 16 splits."""
    G = Hq // Hkv
    rows = QL * G
    tiles = -(-rows // 128)
    per_head = min(16, 128 // Hkv)
    group_tokens = per_head // G if per_head >= G else 0
    groups = -(-QL // group_tokens) if group_tokens else 0
    takes = (variant == 0 and kv_dtype == 0 and D == 128 and bs in (16, 32) and QL > 1
             and G in (1, 2, 4, 8)
             and (groups > 1 or (rows >= 16 and B * Hkv * tiles >= 128)))
    if not takes:
        return False, 0
    pair = 2 if rows <= 64 and Hkv % 2 == 0 else 1
    items = B * (Hkv // pair) * tiles
    if items >= 256:
        return True, 1
    chunk = 64 // pair
    splits = min(-(-256 // items), -(-mx // chunk) // 4, 16)
    return True, max(splits, 1)


def test_query_major_routing_and_key_splits_over_a_spread_of_shapes(pk):
    """The workspace the library asks for follows the many-token kernel's
    routing and split rules: the header alone when its keys are unsplit, the
    (m, l) pairs and the O rows of every (row, split) when they are split,
    and the column-layout decode's workspace when the kernel does not take
    the shape. Checked over batch sizes, head layouts (odd KV head counts
    among them), new-token counts, block sizes and context lengths."""
    lib = pk.load()
    seen = {"unsplit": 0, "split": 0, "column": 0, "max_splits": 0, "rejected": 0}
    heads = ((8, 2), (32, 8), (64, 8), (16, 8), (8, 8), (24, 3), (6, 6), (8, 1), (16, 16),
             (32, 16))
    for B in (1, 2, 3, 8, 17, 64, 300):
        for Hq, Hkv in heads:
            for QL in (2, 3, 4, 5, 8, 16, 33, 64, 128, 256, 1024):
                for bs in (16, 32):
                    for mx in (40, 300, 2048, 32769):
                        nb = -(-mx // bs)
                        p = _params(pk, num_seqs=B, num_q_heads=Hq, num_kv_heads=Hkv,
                                    query_len=QL, block_size=bs, max_context_len=mx,
                                    max_blocks_per_seq=nb, num_blocks=B * nb)
                        got = lib.pa_decode_workspace_size(ctypes.byref(p))
                        if got == 0:
                            # rejected: more than 65,535 new tokens in the step on a shape
                            # the column-layout decode does not take (a limit of the
                            # CUDA-core kernel's grid that the checks apply there)
                            assert B * QL > 65535, (B, Hq, Hkv, QL, bs, mx)
                            seen["rejected"] += 1
                            continue
                        qm, ns = _query_major_plan(B, Hq, Hkv, QL, mx, bs)
                        if qm:
                            want = 256
                            if ns > 1:
                                rows = B * QL * Hq * ns
                                want += _ru(rows * 2 * 4) + _ru(rows * 128 * 4)
                            seen["split" if ns > 1 else "unsplit"] += 1
                            seen["max_splits"] = max(seen["max_splits"], ns)
                            assert got == want, (B, Hq, Hkv, QL, bs, mx, ns)
                        elif bs == 16 and Hkv in (2, 8) and Hq // Hkv in (2, 4, 8):
                            # the column-layout tensor-core decode
                            want = _expected_ws(B, Hq, 128, 1, 256, Hkv=Hkv, QL=QL)
                            seen["column"] += 1
                            assert got == want, (B, Hq, Hkv, QL, bs, mx)
                        else:
                            assert got > 0
    # every branch of the rules is reached, splits up to the cap of 16
    assert min(seen["unsplit"], seen["split"], seen["column"]) > 20 and seen["rejected"] > 0
    assert seen["max_splits"] == 16
    # the CUDA-core variant and the 8-bit cache never take the many-token kernel
    for kw in (dict(variant=1), dict(kv_dtype=1)):
        p = _params(pk, num_seqs=8, num_q_heads=32, num_kv_heads=8, query_len=64,
                    max_context_len=2048, max_blocks_per_seq=128, **kw)
        qm, _ = _query_major_plan(8, 32, 8, 64, 2048, **kw)
        assert not qm
        assert lib.pa_decode_workspace_size(ctypes.byref(p)) > 256


def test_cache_ops_reject_bad_arguments_on_the_host(pk):
    lib = pk.load()
    assert lib.pa_reshape_and_cache(None, None, None, None, None, 4, 8, 128, 64, 10, None) == 2
    assert lib.pa_reshape_and_cache(None, None, None, None, None, 4, 8, 128, 12, 10, None) == 2
    for bs in (8, 16, 32):
        assert lib.pa_reshape_and_cache(None, None, None, None, None, 4, 8, 128, bs, 10, None) == 1
        assert lib.pa_copy_blocks(None, None, None, 2, 8, 128, bs, 10, None) == 1
    assert lib.pa_copy_blocks(None, None, None, 2, 8, 128, 4, 10, None) == 2
    for bs in (8, 16, 32):  # the 8-bit cache at every block size (NULL pointers)
        assert lib.pa_reshape_and_cache_fp8(None, None, None, None, None, None, None, 4, 8, 128,
                                            bs, 10, None) == 1
        assert lib.pa_copy_blocks_fp8(None, None, None, 2, 8, 128, bs, 10, None) == 1
    assert lib.pa_reshape_and_cache_fp8(None, None, None, None, None, None, None, 4, 8, 128, 12,
                                        10, None) == 2
    assert lib.pa_copy_blocks_fp8(None, None, None, 2, 8, 128, 4, 10, None) == 2
    assert lib.pa_reshape_and_cache(None, None, None, None, None, 0, 8, 128, 16, 10, None) == 0
    assert lib.pa_copy_blocks(None, None, None, 2, 8, 128, 16, 10, None) == 1
    assert lib.pa_copy_blocks(None, None, None, 0, 8, 128, 16, 10, None) == 0
    assert lib.pa_copy_blocks(None, None, None, 70000, 8, 128, 16, 10, None) == 1


def test_append_decode_rejects_bad_arguments_on_the_host(pk):
    """pa_append_decode validates its append arguments before any launch (no
    pointer is dereferenced on the host)."""
    lib = pk.load()
    p = _params(pk)
    fake = 1 << 20  # 16-byte aligned, never dereferenced by the host checks
    p.q = p.out = p.k_cache = p.v_cache = fake
    p.block_tables = p.context_lens = fake
    assert lib.pa_append_decode(ctypes.byref(p), None, None, 0, None) == 1
    a = pk.AppendParams()
    assert lib.pa_append_decode(ctypes.byref(p), ctypes.byref(a), None, 0, None) == 1  # NULLs
    a.k_new = a.v_new = a.slot_mapping = fake
    a.k_cache, a.v_cache = fake + 256, fake  # not the decode's cache
    assert lib.pa_append_decode(ctypes.byref(p), ctypes.byref(a), None, 0, None) == 1
    assert b"decode's caches" in lib.pa_last_error()
    a.k_cache = fake
    a.k_new = fake + 8  # misaligned
    assert lib.pa_append_decode(ctypes.byref(p), ctypes.byref(a), None, 0, None) == 1
    a.k_new = fake
    assert lib.pa_append_decode(ctypes.byref(p), ctypes.byref(a), None, 0, None) == 1  # no workspace
    assert b"workspace" in lib.pa_last_error()
    p.head_dim = 96
    assert lib.pa_append_decode(ctypes.byref(p), ctypes.byref(a), None, 0, None) == 2


def test_step_host_layout_and_workspace(pk):
    """The packed-input layout of pa_step_host: sections in header order, each
    256-byte aligned and exactly large enough; the workspace holds the staged
    input, the staged output and a decode workspace."""
    lib = pk.load()
    p = pk.StepHostParams()
    p.num_seqs, p.num_q_heads, p.num_kv_heads, p.head_dim = 3, 8, 2, 128
    p.block_size, p.num_blocks, p.max_blocks_per_seq, p.max_context_len = 16, 10, 5, 80
    p.num_cow_pairs, p.scale = 2, 0.088
    L = pk.StepLayout()
    assert lib.pa_step_host_layout(ctypes.byref(p), ctypes.byref(L)) == 0
    sizes = [3 * 8 * 128 * 2, 3 * 2 * 128 * 2, 3 * 2 * 128 * 2, 3 * 8, 3 * 5 * 4, 3 * 4, 2 * 8]
    offs = [L.q, L.k_new, L.v_new, L.slot_mapping, L.block_tables, L.context_lens, L.cow_pairs]
    assert offs[0] == 0
    for i in range(len(offs)):
        assert offs[i] % 256 == 0
        end = offs[i + 1] if i + 1 < len(offs) else L.total
        assert end == _ru(offs[i] + sizes[i])
    dec = _params(pk, num_seqs=3, num_q_heads=8, num_kv_heads=2, max_blocks_per_seq=5,
                  max_context_len=80, num_blocks=10)
    want = _ru(L.total + 3 * 8 * 128 * 2) + lib.pa_decode_workspace_size(ctypes.byref(dec))
    assert lib.pa_step_host_workspace_size(ctypes.byref(p)) == want
    assert lib.pa_step_host(ctypes.byref(p), None, 0, None) == 1  # NULL buffers
    p.num_cow_pairs = 70000
    assert lib.pa_step_host_layout(ctypes.byref(p), ctypes.byref(L)) == 1
    assert lib.pa_step_host_workspace_size(ctypes.byref(p)) == 0


def test_step_host_layout_with_new_tokens_and_cache_type(pk):
    """With query_len Q the q, k_new, v_new and slot sections hold Q rows per
    sequence and the staged output Q times the rows; kv_dtype and query_len
    outside their ranges are rejected."""
    lib = pk.load()
    p = pk.StepHostParams()
    p.num_seqs, p.num_q_heads, p.num_kv_heads, p.head_dim = 3, 8, 2, 128
    p.block_size, p.num_blocks, p.max_blocks_per_seq, p.max_context_len = 16, 10, 5, 80
    p.scale, p.query_len = 0.088, 4
    L = pk.StepLayout()
    assert lib.pa_step_host_layout(ctypes.byref(p), ctypes.byref(L)) == 0
    sizes = [3 * 4 * 8 * 128 * 2, 3 * 4 * 2 * 128 * 2, 3 * 4 * 2 * 128 * 2, 3 * 4 * 8, 3 * 5 * 4,
             3 * 4, 0]
    offs = [L.q, L.k_new, L.v_new, L.slot_mapping, L.block_tables, L.context_lens, L.cow_pairs]
    for i in range(len(offs)):
        assert offs[i] % 256 == 0
        end = offs[i + 1] if i + 1 < len(offs) else L.total
        assert end == _ru(offs[i] + sizes[i])
    dec = _params(pk, num_seqs=3, num_q_heads=8, num_kv_heads=2, max_blocks_per_seq=5,
                  max_context_len=80, num_blocks=10)
    dec.query_len = 4
    want = _ru(L.total + 3 * 4 * 8 * 128 * 2) + lib.pa_decode_workspace_size(ctypes.byref(dec))
    assert lib.pa_step_host_workspace_size(ctypes.byref(p)) == want
    for field, bad in (("query_len", -1), ("query_len", 1025), ("kv_dtype", 7)):
        q = pk.StepHostParams.from_buffer_copy(p)
        setattr(q, field, bad)
        assert lib.pa_step_host_layout(ctypes.byref(q), ctypes.byref(L)) == 1  # PA_ERR_INVALID_ARG
        assert lib.pa_step_host_workspace_size(ctypes.byref(q)) == 0
