"""GPU parity of the decode of several new tokens per sequence (query_len Q > 1).

The new tokens are the last Q of each sequence's context_lens[b] and already
in the cache; query token i attends to the first L - Q + i + 1 tokens (causal
among the new tokens). The float64 oracle computes every (sequence, token,
head) row; the bar is the decode's: max-abs <= 2e-2, mean-abs <= 2e-3, and
bit-exact caches for the fused KV write. Padding slots hold NaN, so a masked
slot that leaks into a result fails the finiteness check.
"""
import numpy as np
import pytest

import oracle
import workloads
from tests import harness

pytestmark = pytest.mark.gpu

DEVERR_CONTEXT_LEN = 0x2
DEVERR_APPEND_SLOT = 0x20


@pytest.fixture(scope="module")
def pk():
    import torch

    from paged_kv_cache_92_gb300 import build

    build.build()
    import paged_kv_cache_92_gb300 as pk

    pk.load()
    assert torch.cuda.is_available()
    return pk


def _sm_count():
    import torch

    return torch.cuda.get_device_properties(0).multi_processor_count


def _case(lens, QL, Hq, Hkv, D, seed, extra_blocks=3):
    """Random tables over a shuffled pool, N(0,1) bf16 cache with NaN in the
    padding slots, q [B][QL][Hq][D]."""
    import torch

    lens = np.asarray(lens, dtype=np.int64)
    need = int(((lens + 15) // 16).sum())
    NB = need + extra_blocks
    order = np.random.default_rng(seed).permutation(NB).astype(np.int32)
    tables = workloads.sequential_tables(lens, order, 16)
    q = workloads.bf16_normal((len(lens), QL, Hq, D), seed + 1, "cuda")
    kc = workloads.bf16_normal((NB, Hkv, 16, D), seed + 2, "cuda")
    vc = workloads.bf16_normal((NB, Hkv, 16, D), seed + 3, "cuda")
    workloads.fill_padding_nan(kc, tables, lens, 16)
    workloads.fill_padding_nan(vc, tables, lens, 16)
    return q, kc, vc, tables, lens.astype(np.int32), torch


def _decode(pk, q, kc, vc, tables, lens, torch, **kw):
    out = pk.pa_decode(q, kc, vc, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                       max_context_len=int(lens.max()), **kw)
    torch.cuda.synchronize()
    return out


def _check(pk, q, kc, vc, tables, lens, torch, **kw):
    out = _decode(pk, q, kc, vc, tables, lens, torch, **kw)
    want = oracle.paged_decode_multi(q.cpu(), kc.cpu(), vc.cpu(), tables, lens)
    stats = harness.assert_close(harness.bf16_tensor_to_f64(out), want)
    assert pk.pa_device_errors() == 0
    return stats


# (G, Hkv, Q): every columns-per-KV-head width (G x Q rounded up to a power
# of two: 2 .. 16), padded widths N = 16 .. 128, Q not a power of two
SHAPES = [(1, 8, 2), (1, 1, 16), (1, 8, 16), (2, 4, 4), (2, 2, 8), (4, 8, 2), (4, 8, 3),
          (4, 8, 4), (4, 1, 4), (8, 8, 2), (8, 1, 2), (8, 4, 2)]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G,Hkv,QL", SHAPES)
def test_multi_edge_lengths(pk, D, G, Hkv, QL):
    """Lengths from exactly Q (every key is a new token) through block
    boundaries inside the new tokens to several thousand (split over CTAs)."""
    lens = sorted({QL, QL + 1, 15, 16, 17, 18, 31, 33, 100, 511, 513, 1025, 4098})
    lens = [L for L in lens if L >= QL]
    _check(pk, *_case(lens, QL, G * Hkv, Hkv, D, seed=G * 100 + Hkv * 10 + QL + D))


@pytest.mark.parametrize("QL", [2, 3, 4, 16])
def test_multi_piece_with_masked_columns_merges(pk, QL):
    """One sequence of SM count + 1 (or + 2, odd) blocks: the split gives two
    blocks to each CTA, so its last block is a piece of its own. With the
    sequence ending 2 tokens into that block, the first Q - 2 query tokens see
    nothing of it: their partials there are (max -inf, sum 0) and the merge
    must drop them."""
    nb = _sm_count() + 1
    if nb % 2 == 0:
        nb += 1
    L = (nb - 1) * 16 + 2
    G, Hkv = (1, 8) if QL == 16 else (4, 8)
    _check(pk, *_case([L, 40], QL, G * Hkv, Hkv, 128, seed=70 + QL))


def test_multi_llama8b_layer(pk):
    """64 sequences, 32/8 heads, lengths U[128, 2048], 4 new tokens each (N = 128)."""
    r = workloads.llama8b_layer()
    _check(pk, *_case(r.lens0 + 4, 4, 32, 8, 128, seed=81))


def test_multi_llama70b_long(pk):
    """8 sequences, 64/8 heads, lengths U[8192, 32768], 2 new tokens each."""
    r = workloads.llama70b_long(batch=8)
    _check(pk, *_case(r.lens0 + 2, 2, 64, 8, 128, seed=82))


def test_one_token_as_4d_is_bit_identical(pk):
    """q [B][1][Hq][D] is the single-token decode."""
    q, kc, vc, tables, lens, torch = _case([1, 17, 300, 2049], 1, 32, 8, 128, seed=83)
    a = _decode(pk, q, kc, vc, tables, lens, torch)
    b = _decode(pk, q[:, 0].contiguous(), kc, vc, tables, lens, torch)
    assert torch.equal(a[:, 0].view(torch.int16), b.view(torch.int16))


def test_multi_rows_equal_single_token_decodes(pk):
    """Token i of Q equals the single-token decode of a sequence that ends at
    it: the causal limit is the only difference between the rows."""
    QL = 4
    q, kc, vc, tables, lens, torch = _case([37, 64, 700], QL, 32, 8, 128, seed=84)
    multi = harness.bf16_tensor_to_f64(_decode(pk, q, kc, vc, tables, lens, torch))
    for i in range(QL):
        li = (lens - QL + i + 1).astype(np.int32)
        one = _decode(pk, q[:, i].contiguous(), kc, vc, tables, li, torch)
        d = np.abs(multi[:, i] - harness.bf16_tensor_to_f64(one))
        assert d.max() <= 2e-2 and d.mean() <= 2e-3


def test_multi_short_sequences_are_flagged_and_zero(pk):
    """0 < L < Q cannot hold the new tokens: zero rows and PA_DEVERR_CONTEXT_LEN;
    L = 0 gives zero rows; the other sequences are unaffected."""
    QL = 4
    q, kc, vc, tables, lens, torch = _case([40, 2, 0, 50], QL, 16, 4, 128, seed=85)
    out = torch.full_like(q, 7.0)
    pk.pa_decode(q, kc, vc, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                 max_context_len=50, out=out)
    torch.cuda.synchronize()
    assert pk.pa_device_errors() & DEVERR_CONTEXT_LEN
    got = harness.bf16_tensor_to_f64(out)
    assert not got[1].any() and not got[2].any()
    keep = [0, 3]
    want = oracle.paged_decode_multi(q.cpu()[keep], kc.cpu(), vc.cpu(), tables[keep], lens[keep])
    harness.assert_close(got[keep], want)


def test_multi_placement_invariance_bit_exact(pk):
    import torch

    q, kc, vc, tables, lens, _ = _case([300, 47, 900], 3, 16, 4, 128, seed=86)
    NB = kc.shape[0]
    perm = np.random.default_rng(9).permutation(NB)
    kcb, vcb = torch.empty_like(kc), torch.empty_like(vc)
    kcb[torch.from_numpy(perm).cuda()] = kc
    vcb[torch.from_numpy(perm).cuda()] = vc
    tables_b = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    a = _decode(pk, q, kc, vc, tables, lens, torch)
    b = _decode(pk, q, kcb, vcb, tables_b, lens, torch)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ---------------------------------------------------------------- query-major kernel
#
# When the column-group decode would need several groups and the batch gives
# at least 128 (sequence, KV head, 128-row tile) CTAs, the new tokens run on
# the query-major tensor-core kernel: each CTA streams one KV head's blocks
# once for up to 128 query rows (tokens x G heads).

QM_LENS = [64, 65, 63, 129, 200, 511, 513, 1025, 2049, 100, 300, 700, 90, 1500, 127, 128]


def _qm_lens(QL, B=16):
    lens = [max(L, QL) for L in QM_LENS]
    lens[0], lens[1] = QL, QL + 1  # every key a new token; one older key
    return (lens * ((B + len(lens) - 1) // len(lens)))[:B]


@pytest.mark.parametrize("G,Hkv,QL,B", [
    # at most 32 rows (tokens x G) per KV head: two heads per work item, half filled
    (4, 8, 8, 16), (8, 8, 4, 16), (1, 8, 20, 16), (2, 8, 12, 16), (4, 8, 5, 16), (8, 8, 3, 16),
    # 16 rows, within one column group: query-major from 16 rows per head
    (4, 8, 4, 16), (2, 8, 8, 16), (8, 8, 2, 16),
    # at most 64 rows: two heads per item
    (4, 8, 16, 16), (1, 8, 33, 16), (2, 8, 24, 16), (4, 8, 12, 16), (8, 8, 6, 16),
    # one head per item; one, two and three 128-row tiles
    (2, 8, 64, 16), (4, 8, 64, 16), (8, 4, 16, 32), (8, 8, 40, 16),
    # an odd number of KV heads: one head per item, few rows
    (2, 3, 16, 48), (8, 1, 6, 128)])
def test_query_major_against_the_oracle(pk, G, Hkv, QL, B):
    """Lengths from Q (every key a new token) across chunk and block boundaries
    to 2049; two KV heads per work item or one, partly filled tiles and
    several tiles per head."""
    q, kc, vc, tables, lens, torch = _case(_qm_lens(QL, B), QL, G * Hkv, Hkv, 128,
                                           seed=700 + G * 10 + QL)
    _check(pk, q, kc, vc, tables, lens, torch)


@pytest.mark.parametrize("G,Hkv,QL,lens", [
    (8, 8, 8, [4100, 2900]),               # 70B-class heads: 8 units, 16 splits
    (4, 8, 16, [3000, 16, 700, 2049]),     # every key new; splits with no keys
    (2, 3, 64, [1500, 2600]),              # one head per item (odd head count), two tiles
    (1, 8, 40, [64, 5000, 333]),
])
def test_query_major_split_keys(pk, G, Hkv, QL, lens):
    """Small batches: each item's keys split over CTAs, fp32 partials merged
    by log-sum-exp weights; splits past a short sequence's keys (or past a
    row's causal limit) contribute nothing."""
    q, kc, vc, tables, lens, torch = _case(lens, QL, G * Hkv, Hkv, 128, seed=740 + QL + G)
    _check(pk, q, kc, vc, tables, lens, torch)


@pytest.mark.parametrize("G,Hkv,QL,B", [(4, 8, 64, 16), (8, 4, 32, 40), (1, 8, 256, 16),
                                        (4, 3, 64, 48), (2, 8, 128, 40)])
def test_query_major_two_tiles_per_item(pk, G, Hkv, QL, B):
    """One KV head per item with an even number of 128-row tiles per head:
    items of two tiles sharing each load of the keys (eight softmax warps),
    several items per CTA."""
    q, kc, vc, tables, lens, torch = _case(_qm_lens(QL, B), QL, G * Hkv, Hkv, 128,
                                           seed=770 + G + QL)
    _check(pk, q, kc, vc, tables, lens, torch)


def test_query_major_two_tiles_short_and_empty_sequences(pk):
    QL = 64
    lens = _qm_lens(QL, 32)
    lens[3], lens[5], lens[7] = 0, 40, 0  # empty, and too short for the new tokens
    q, kc, vc, tables, lens, torch = _case(lens, QL, 32, 8, 128, seed=790)
    out = torch.full_like(q, 7.0)
    pk.pa_decode(q, kc, vc, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                 max_context_len=int(lens.max()), out=out)
    torch.cuda.synchronize()
    assert pk.pa_device_errors() & DEVERR_CONTEXT_LEN
    got = harness.bf16_tensor_to_f64(out)
    for b in (3, 5, 7):
        assert not got[b].any()
    keep = [b for b in range(len(lens)) if b not in (3, 5, 7)]
    want = oracle.paged_decode_multi(q.cpu()[keep], kc.cpu(), vc.cpu(), tables[keep], lens[keep])
    harness.assert_close(got[keep], want)


def _split_plan(lens, QL, G, Hkv, grid, BS=16):
    """Which key-split plan the query-major kernel takes, restated from its
    scheduling rule (test-side, so that a case can state what it exercises).

    With fewer than 256 (sequence, head group, tile) units and a split bound
    `cap` > 1 (the workspace's partials per row), the uniform plan splits
    every unit `cap` ways and deals the items in a snake over `grid` CTAs;
    the one-wave plan cuts each (sequence, tile) into ceil(n / T) <= cap
    pieces, T the smallest piece length (in 64-column chunks) that leaves
    every CTA at most one item. The kernel takes the one-wave plan when its
    largest piece, plus 2 chunks per item, is below the uniform plan's
    busiest CTA (each item also counted 2 chunks more)."""
    lens = [int(x) for x in lens]
    B, mx = len(lens), max(lens)
    rows = QL * G
    tiles = -(-rows // 128)
    hb = 2 if rows <= 64 and Hkv % 2 == 0 else 1
    NB, QT, hgc = 64 // (BS * hb), (128 // hb) // G, Hkv // hb
    units = B * hgc * tiles
    if units >= 256:
        return "unsplit"
    cap = max(1, min(-(-256 // units), -(-mx // (64 // hb)) // 4, 16))
    if cap == 1:
        return "unsplit"
    n_rt = []  # chunks of each (sequence by decreasing length, tile)
    for b in sorted(range(B), key=lambda v: (-lens[v], v)):
        for t in range(tiles):
            L = 0 if 0 < lens[b] < QL else lens[b]
            keys = L - QL + min(QL, (t + 1) * QT) if L > 0 else 0
            n_rt.append(-(-(-(-keys // BS)) // NB))
    load = [0] * grid
    per_seq = hgc * tiles * cap
    for x in range(B * per_seq):
        rem = x % per_seq
        sp, n = rem % cap, n_rt[x // per_seq * tiles + rem // cap % tiles]
        size = (sp + 1) * n // cap - sp * n // cap
        p, pos = divmod(x, grid)
        if size:
            load[grid - 1 - pos if p & 1 else pos] += size + 2
    pieces = lambda n, T: min(cap, -(-n // T)) if n > 0 else 1
    count = lambda T: sum(hgc * pieces(n, T) for n in n_rt)
    if max(n_rt) == 0 or count(max(n_rt)) > grid:
        return "uniform"
    T = next(T for T in range(1, max(n_rt) + 1) if count(T) <= grid)
    wave = max(-(-n // pieces(n, T)) for n in n_rt) + 2
    return "wave" if wave < max(load) else "uniform"


@pytest.mark.parametrize("G,Hkv,QL,lens,plan", [
    (8, 8, 8, [4000, 3900, 3000, 2200, 1700, 1600, 1100, 1000], "wave"),  # 70B-class heads
    (8, 8, 8, [4100, 2000, 3500, 900], "wave"),                          # up to 16 splits
    (4, 3, 48, [2500, 900, 1800], "wave"),         # one head per item, two tiles per head
    (4, 8, 16, [2600, 2400, 900, 1500, 300, 2000, 1100, 700], "wave"),
    (4, 8, 8, [1048, 1232, 159, 1236, 771, 835, 992, 520] * 4, "uniform"),  # 2 splits at most
    (8, 8, 8, [4100, 2900], "uniform"),
])
def test_query_major_split_plans(pk, G, Hkv, QL, lens, plan):
    """Split keys under both plans: every unit split the workspace's number
    of ways, or one wave of pieces of at most T chunks, where a row may have
    fewer splits than the workspace holds and its last split marks the rest
    empty. The workspace is filled with 0x7f bytes first (partials of m =
    3.4e38), so a slot left unmarked would swamp the merge."""
    import torch

    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert _split_plan(lens, QL, G, Hkv, 152) == plan
    q, kc, vc, tables, lens, torch = _case(lens, QL, G * Hkv, Hkv, 128, seed=860 + QL + G)
    p = pk.make_decode_params(q, torch.empty_like(q), kc, vc, torch.from_numpy(tables).cuda(),
                              torch.from_numpy(lens).cuda(), max_context_len=int(lens.max()))
    ws = torch.full((pk.pa_decode_workspace_size(p),), 0x7F, dtype=torch.uint8, device="cuda")
    _check(pk, q, kc, vc, tables, lens, torch, workspace=ws)


def test_query_major_one_wave_with_an_empty_sequence(pk):
    """An empty sequence in a one-wave plan: one item with no keys, whose
    partials (and the row's unused slots) are empty, so its rows come out
    zero; the other rows match the oracle."""
    import torch

    lens = [3000, 0, 2500, 1200, 800, 2000]
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert _split_plan(lens, 8, 8, 8, 152) == "wave"
    q, kc, vc, tables, lens, torch = _case(lens, 8, 64, 8, 128, seed=880)
    p = pk.make_decode_params(q, torch.empty_like(q), kc, vc, torch.from_numpy(tables).cuda(),
                              torch.from_numpy(lens).cuda(), max_context_len=int(lens.max()))
    ws = torch.full((pk.pa_decode_workspace_size(p),), 0x7F, dtype=torch.uint8, device="cuda")
    out = _decode(pk, q, kc, vc, tables, lens, torch, workspace=ws)
    assert pk.pa_device_errors() == 0
    got = harness.bf16_tensor_to_f64(out)
    assert not got[1].any()
    keep = [0, 2, 3, 4, 5]
    want = oracle.paged_decode_multi(q.cpu()[keep], kc.cpu(), vc.cpu(), tables[keep], lens[keep])
    harness.assert_close(got[keep], want)


@pytest.mark.parametrize("seed", range(24))
def test_query_major_random_shapes(pk, seed):
    """Seeded random shapes across the query-major space: G, the KV head
    count (odd included), Q, the batch (split keys or not) and lengths from Q
    up, some on block and chunk boundaries; the oracle's work is kept small."""
    rng = np.random.default_rng(900 + seed)
    G = int(rng.choice([1, 2, 4, 8]))
    Hkv = int(rng.choice([1, 2, 3, 4, 8]))
    QL = int(rng.integers(3, 81))
    B = int(rng.integers(1, 41))
    budget = 1e8  # query rows x keys
    lmax = max(QL + 1, min(4000, int(budget / (B * QL * G * Hkv))))
    lens = rng.integers(QL, lmax + 1, size=B)
    edges = [QL, QL + 1, 16 * ((QL + 15) // 16), 64 * ((QL + 63) // 64) + 1]
    for k in range(min(B, len(edges))):
        lens[k] = min(edges[k], lmax)
    q, kc, vc, tables, lens, torch = _case(lens, QL, G * Hkv, Hkv, 128, seed=950 + seed)
    _check(pk, q, kc, vc, tables, lens, torch)


@pytest.mark.parametrize("G,Hkv,QL,B", [(4, 8, 8, 400), (4, 8, 64, 24), (2, 8, 24, 200)])
def test_query_major_many_items_per_cta(pk, G, Hkv, QL, B):
    """More work items than SMs: each persistent CTA takes several in turn
    (a snake over the items by length; unranked beyond 256 sequences), the
    next item's loads overlapping the current one's end. Short lengths keep
    the oracle quick."""
    lens = np.random.default_rng(730 + QL).integers(QL, QL + 300, size=B)
    lens[:3] = [QL, QL + 1, QL + 15]
    q, kc, vc, tables, lens, torch = _case(lens, QL, G * Hkv, Hkv, 128, seed=731 + QL)
    _check(pk, q, kc, vc, tables, lens, torch)


def test_query_major_short_and_empty_sequences(pk):
    QL = 8
    lens = _qm_lens(QL)
    lens[3], lens[5], lens[7] = 0, 5, 0  # empty, and too short for the new tokens
    q, kc, vc, tables, lens, torch = _case(lens, QL, 32, 8, 128, seed=720)
    out = torch.full_like(q, 7.0)
    pk.pa_decode(q, kc, vc, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                 max_context_len=int(lens.max()), out=out)
    torch.cuda.synchronize()
    assert pk.pa_device_errors() & DEVERR_CONTEXT_LEN
    got = harness.bf16_tensor_to_f64(out)
    for b in (3, 5, 7):
        assert not got[b].any()
    keep = [b for b in range(len(lens)) if b not in (3, 5, 7)]
    want = oracle.paged_decode_multi(q.cpu()[keep], kc.cpu(), vc.cpu(), tables[keep], lens[keep])
    harness.assert_close(got[keep], want)


def test_query_major_placement_invariance_bit_exact(pk):
    import torch

    q, kc, vc, tables, lens, _ = _case(_qm_lens(16), 16, 32, 8, 128, seed=721)
    NB = kc.shape[0]
    perm = np.random.default_rng(29).permutation(NB)
    kcb, vcb = torch.empty_like(kc), torch.empty_like(vc)
    kcb[torch.from_numpy(perm).cuda()] = kc
    vcb[torch.from_numpy(perm).cuda()] = vc
    tables_b = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    a = _decode(pk, q, kc, vc, tables, lens, torch)
    b = _decode(pk, q, kcb, vcb, tables_b, lens, torch)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("QL,lens,G", [
    (16, None, 4),                          # 16 sequences: two heads per item, 4 splits
    (64, [3000, 64, 500, 65], 4),           # one head per item, two tiles, 5 splits
    (8, [900] * 40 + [2049] * 24, 8),       # 256 items, no split
])
def test_query_major_fused_append(pk, QL, lens, G):
    """pa_append_decode on this path: the KV write inside the kernel (each item
    writes the new tokens among its keys before it loads them; the new slots
    hold NaN before the step, so a read before the write shows), then the
    query-major decode; caches bit-exact, rows against the oracle."""
    lens = _qm_lens(QL) if lens is None else lens
    q, kc, vc, tables, lens, slots, kn, vn, torch = _append_case(lens, QL, 8 * G, 8,
                                                                 seed=722 + QL)
    kc2, vc2 = kc.clone(), vc.clone()
    out = pk.pa_append_decode(q, kc2, vc2, torch.from_numpy(tables).cuda(),
                              torch.from_numpy(lens).cuda(), int(lens.max()), kn, vn,
                              torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    assert pk.pa_device_errors() == 0
    ko, vo = oracle.reshape_and_cache(kn.cpu(), vn.cpu(), oracle.bf16_bits(kc.cpu()),
                                      oracle.bf16_bits(vc.cpu()), slots)
    assert np.array_equal(oracle.bf16_bits(kc2.cpu()), ko)
    assert np.array_equal(oracle.bf16_bits(vc2.cpu()), vo)
    want = oracle.paged_decode_multi(q.cpu(), ko, vo, tables, lens)
    harness.assert_close(harness.bf16_tensor_to_f64(out), want)


def test_query_major_fused_append_slot_rules(pk):
    """A slot that is not its token's is not written (PA_DEVERR_APPEND_SLOT); a
    negative slot writes nothing; the other tokens are written, split items
    included."""
    QL = 16
    q, kc, vc, tables, lens, slots, kn, vn, torch = _append_case([40, 70, 300, 2049], QL, 32, 8,
                                                                 seed=760)
    bad = slots.copy()
    bad[1] = slots[1] + 1 if slots[1] % 16 != 15 else slots[1] - 1  # wrong offset
    bad[20] = -1
    bad[60] = slots[62]  # another token's slot
    kc2, vc2 = kc.clone(), vc.clone()
    pk.pa_append_decode(q, kc2, vc2, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                        int(lens.max()), kn, vn, torch.from_numpy(bad).cuda())
    torch.cuda.synchronize()
    assert pk.pa_device_errors() & DEVERR_APPEND_SLOT
    written = [t for t in range(len(slots)) if t not in (1, 20, 60)]
    ko, vo = oracle.reshape_and_cache(kn.cpu()[written], vn.cpu()[written],
                                      oracle.bf16_bits(kc.cpu()), oracle.bf16_bits(vc.cpu()),
                                      slots[written])
    assert np.array_equal(oracle.bf16_bits(kc2.cpu()), ko)
    assert np.array_equal(oracle.bf16_bits(vc2.cpu()), vo)


def test_query_major_llama8b_layer(pk):
    """The bench's 8B layer with 16 new tokens per sequence (the query-major path)."""
    r = workloads.llama8b_layer()
    _check(pk, *_case(r.lens0 + 16, 16, 32, 8, 128, seed=723))


# ---------------------------------------------------------------- CUDA-core kernel
#
# The CUDA-core variant decodes each (sequence, new token) row on its own:
# row (b, i) streams the first L - Q + i + 1 keys, split into 512-token
# partitions and merged like a one-token decode.

CUDA_CORE_SHAPES = [(1, 8, 2), (4, 8, 3), (8, 8, 2), (4, 2, 8), (2, 4, 17)]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G,Hkv,QL", CUDA_CORE_SHAPES)
def test_multi_cuda_core_edge_lengths(pk, D, G, Hkv, QL):
    """Lengths from exactly Q through block and partition boundaries (511 ..
    514 put the rows of one sequence on both sides of 512) to five partitions."""
    lens = sorted({QL, QL + 1, 15, 16, 17, 33, 511, 512, 513, 514, 1025, 2100})
    lens = [L for L in lens if L >= QL]
    _check(pk, *_case(lens, QL, G * Hkv, Hkv, D, seed=500 + G * 100 + Hkv * 10 + QL + D),
           variant=pk.DECODE_CUDA_CORE)


def test_multi_cuda_core_rows_are_single_token_decodes_bit_exact(pk):
    """Row (b, i) is bit for bit the one-token CUDA-core decode of query row
    (b, i) over a sequence that ends at its token."""
    QL = 5
    q, kc, vc, tables, lens, torch = _case([37, 64, 515, 1030], QL, 32, 8, 128, seed=510)
    multi = _decode(pk, q, kc, vc, tables, lens, torch, variant=pk.DECODE_CUDA_CORE)
    for i in range(QL):
        li = (lens - QL + i + 1).astype(np.int32)
        one = _decode(pk, q[:, i].contiguous(), kc, vc, tables, li, torch,
                      variant=pk.DECODE_CUDA_CORE)
        assert torch.equal(multi[:, i].contiguous().view(torch.int16), one.view(torch.int16))


def test_multi_cuda_core_short_sequences_are_flagged_and_zero(pk):
    QL = 4
    q, kc, vc, tables, lens, torch = _case([40, 2, 0, 600], QL, 16, 4, 128, seed=511)
    out = torch.full_like(q, 7.0)
    pk.pa_decode(q, kc, vc, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                 max_context_len=600, out=out, variant=pk.DECODE_CUDA_CORE)
    torch.cuda.synchronize()
    assert pk.pa_device_errors() & DEVERR_CONTEXT_LEN
    got = harness.bf16_tensor_to_f64(out)
    assert not got[1].any() and not got[2].any()
    keep = [0, 3]
    want = oracle.paged_decode_multi(q.cpu()[keep], kc.cpu(), vc.cpu(), tables[keep], lens[keep])
    harness.assert_close(got[keep], want)


def test_multi_cuda_core_llama70b_rows(pk):
    """64/8 heads, two new tokens, contexts of several partitions."""
    q, kc, vc, tables, lens, torch = _case([3000, 4097, 130], 2, 64, 8, 128, seed=512)
    _check(pk, q, kc, vc, tables, lens, torch, variant=pk.DECODE_CUDA_CORE)


def test_multi_cuda_core_matches_tensor_core(pk):
    """Both kernels compute the same function: within the bf16 tolerance of
    each other on the same inputs."""
    q, kc, vc, tables, lens, torch = _case([100, 513, 2000], 3, 32, 8, 128, seed=513)
    a = harness.bf16_tensor_to_f64(_decode(pk, q, kc, vc, tables, lens, torch))
    b = harness.bf16_tensor_to_f64(_decode(pk, q, kc, vc, tables, lens, torch,
                                           variant=pk.DECODE_CUDA_CORE))
    d = np.abs(a - b)
    assert d.max() <= 2e-2 and d.mean() <= 2e-3


# ---------------------------------------------------------------- column groups
#
# A column group holds G x (its tokens, rounded up to a power of two) <= 16
# columns per KV head and at most 128 in all (64 for the 8-bit cache). More
# new tokens are split into groups of that many, each decoded as a virtual
# sequence that streams the keys its last token sees: (G, Hkv, Q) below have
# 2 to 16 groups, a last group shorter than the others, and Q = 64.

GROUP_SHAPES = [(4, 8, 8), (4, 8, 16), (4, 8, 5), (8, 8, 3), (8, 8, 8), (8, 2, 3), (2, 8, 64),
                (4, 1, 64), (1, 8, 33)]


@pytest.mark.parametrize("G,Hkv,QL", GROUP_SHAPES)
def test_multi_column_groups(pk, G, Hkv, QL):
    lens = sorted({QL, QL + 1, 15, 16, 17, 33, 100, 513, 1025, 3000})
    lens = [L for L in lens if L >= QL]
    _check(pk, *_case(lens, QL, G * Hkv, Hkv, 128, seed=300 + G * 100 + Hkv * 10 + QL))


def test_multi_column_groups_head_dim_64(pk):
    lens = [8, 9, 16, 17, 100, 700, 2049]
    _check(pk, *_case(lens, 8, 32, 8, 64, seed=331))


def test_multi_column_groups_llama8b_layer(pk):
    """The 64-sequence 8B layer with 16 new tokens per sequence (chunked-prefill
    slices): 4 column groups of 4 tokens, 256 virtual sequences."""
    r = workloads.llama8b_layer()
    _check(pk, *_case(r.lens0 + 16, 16, 32, 8, 128, seed=332))


def test_multi_column_groups_llama70b_long(pk):
    """Three 70B-class sequences (64/8 heads, 8k-33k tokens) with 8 new tokens:
    4 column groups of 2, each streaming up to 33k tokens over many CTAs."""
    r = workloads.llama70b_long(batch=8)
    _check(pk, *_case(r.lens0[:3] + 8, 8, 64, 8, 128, seed=333))


def test_multi_column_groups_placement_invariance_bit_exact(pk):
    import torch

    q, kc, vc, tables, lens, _ = _case([300, 47, 900, 8], 8, 32, 8, 128, seed=334)
    NB = kc.shape[0]
    perm = np.random.default_rng(19).permutation(NB)
    kcb, vcb = torch.empty_like(kc), torch.empty_like(vc)
    kcb[torch.from_numpy(perm).cuda()] = kc
    vcb[torch.from_numpy(perm).cuda()] = vc
    tables_b = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    a = _decode(pk, q, kc, vc, tables, lens, torch)
    b = _decode(pk, q, kcb, vcb, tables_b, lens, torch)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("QL", [8, 13])
def test_multi_column_groups_fused_append(pk, QL):
    """Every group writes the new tokens its own stream reads before it reads
    their blocks (the same bytes where groups overlap): caches bit-exact, and
    the rows against the oracle."""
    nb = _sm_count() + 1
    long_len = nb * 16 + 5
    lens = [long_len, 17, 33, 16 + QL, 500, QL]
    q, kc, vc, tables, lens, slots, kn, vn, torch = _append_case(lens, QL, 32, 8, seed=340 + QL)
    kc2, vc2 = kc.clone(), vc.clone()
    out = pk.pa_append_decode(q, kc2, vc2, torch.from_numpy(tables).cuda(),
                              torch.from_numpy(lens).cuda(), int(lens.max()), kn, vn,
                              torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    assert pk.pa_device_errors() == 0
    ko, vo = oracle.reshape_and_cache(kn.cpu(), vn.cpu(), oracle.bf16_bits(kc.cpu()),
                                      oracle.bf16_bits(vc.cpu()), slots)
    assert np.array_equal(oracle.bf16_bits(kc2.cpu()), ko)
    assert np.array_equal(oracle.bf16_bits(vc2.cpu()), vo)
    want = oracle.paged_decode_multi(q.cpu(), ko, vo, tables, lens)
    harness.assert_close(harness.bf16_tensor_to_f64(out), want)


def test_multi_column_groups_short_sequences_are_flagged_and_zero(pk):
    QL = 8
    q, kc, vc, tables, lens, torch = _case([40, 5, 0, 50], QL, 32, 8, 128, seed=345)
    out = torch.full_like(q, 7.0)
    pk.pa_decode(q, kc, vc, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                 max_context_len=50, out=out)
    torch.cuda.synchronize()
    assert pk.pa_device_errors() & DEVERR_CONTEXT_LEN
    got = harness.bf16_tensor_to_f64(out)
    assert not got[1].any() and not got[2].any()
    keep = [0, 3]
    want = oracle.paged_decode_multi(q.cpu()[keep], kc.cpu(), vc.cpu(), tables[keep], lens[keep])
    harness.assert_close(got[keep], want)


# ---------------------------------------------------------------- fused KV write


def _append_case(lens, QL, Hq, Hkv, seed):
    """The new tokens' slots hold NaN before the step; k_new/v_new rows
    b*QL + i are written at token L - QL + i."""
    q, kc, vc, tables, lens, torch = _case(lens, QL, Hq, Hkv, 128, seed)
    slots = []
    for b, L in enumerate(lens):
        for i in range(QL):
            pos = int(L) - QL + i
            slots.append(int(tables[b, pos // 16]) * 16 + pos % 16)
    slots = np.array(slots, dtype=np.int64)
    for s in slots.tolist():
        kc[s // 16, :, s % 16] = float("nan")
        vc[s // 16, :, s % 16] = float("nan")
    T = len(slots)
    kn = workloads.bf16_normal((T, Hkv, 128), seed + 11, "cuda")
    vn = workloads.bf16_normal((T, Hkv, 128), seed + 12, "cuda")
    return q, kc, vc, tables, lens, slots, kn, vn, torch


@pytest.mark.parametrize("QL", [2, 4])
def test_multi_fused_append_matches_oracle(pk, QL):
    """The new tokens straddle block boundaries, and in the long sequence the
    two blocks holding them go to different CTAs."""
    nb = _sm_count() + 1
    if nb % 2 == 0:
        nb += 1
    long_len = (nb - 1) * 16 + 2
    lens = [long_len, 17, 33, 16 + QL, 500]
    q, kc, vc, tables, lens, slots, kn, vn, torch = _append_case(lens, QL, 32, 8, seed=90 + QL)
    kc2, vc2 = kc.clone(), vc.clone()
    out = pk.pa_append_decode(q, kc2, vc2, torch.from_numpy(tables).cuda(),
                              torch.from_numpy(lens).cuda(), int(lens.max()), kn, vn,
                              torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    assert pk.pa_device_errors() == 0
    ko, vo = oracle.reshape_and_cache(kn.cpu(), vn.cpu(), oracle.bf16_bits(kc.cpu()),
                                      oracle.bf16_bits(vc.cpu()), slots)
    assert np.array_equal(oracle.bf16_bits(kc2.cpu()), ko)
    assert np.array_equal(oracle.bf16_bits(vc2.cpu()), vo)
    want = oracle.paged_decode_multi(q.cpu(), ko, vo, tables, lens)
    harness.assert_close(harness.bf16_tensor_to_f64(out), want)


@pytest.mark.parametrize("QL", [2, 5])
def test_multi_cuda_core_fused_append_matches_oracle(pk, QL):
    """On the CUDA-core kernel the step's write runs first (same slot rule,
    token L - Q + i), then the decode."""
    lens = [600, 17, 33, 16 + QL, 1500]
    q, kc, vc, tables, lens, slots, kn, vn, torch = _append_case(lens, QL, 32, 8, seed=520 + QL)
    kc2, vc2 = kc.clone(), vc.clone()
    out = pk.pa_append_decode(q, kc2, vc2, torch.from_numpy(tables).cuda(),
                              torch.from_numpy(lens).cuda(), int(lens.max()), kn, vn,
                              torch.from_numpy(slots).cuda(), variant=pk.DECODE_CUDA_CORE)
    torch.cuda.synchronize()
    assert pk.pa_device_errors() == 0
    ko, vo = oracle.reshape_and_cache(kn.cpu(), vn.cpu(), oracle.bf16_bits(kc.cpu()),
                                      oracle.bf16_bits(vc.cpu()), slots)
    assert np.array_equal(oracle.bf16_bits(kc2.cpu()), ko)
    assert np.array_equal(oracle.bf16_bits(vc2.cpu()), vo)
    want = oracle.paged_decode_multi(q.cpu(), ko, vo, tables, lens)
    harness.assert_close(harness.bf16_tensor_to_f64(out), want)


def test_multi_cuda_core_fused_append_slot_rules(pk):
    QL = 3
    q, kc, vc, tables, lens, slots, kn, vn, torch = _append_case([40, 70], QL, 16, 4, seed=530)
    bad = slots.copy()
    bad[1] = slots[1] + 1 if slots[1] % 16 != 15 else slots[1] - 1  # wrong offset
    bad[4] = -1
    kc2, vc2 = kc.clone(), vc.clone()
    pk.pa_append_decode(q, kc2, vc2, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                        int(lens.max()), kn, vn, torch.from_numpy(bad).cuda(),
                        variant=pk.DECODE_CUDA_CORE)
    torch.cuda.synchronize()
    assert pk.pa_device_errors() & DEVERR_APPEND_SLOT
    written = [t for t in range(len(slots)) if t not in (1, 4)]
    ko, vo = oracle.reshape_and_cache(kn.cpu()[written], vn.cpu()[written],
                                      oracle.bf16_bits(kc.cpu()), oracle.bf16_bits(vc.cpu()),
                                      slots[written])
    assert np.array_equal(oracle.bf16_bits(kc2.cpu()), ko)
    assert np.array_equal(oracle.bf16_bits(vc2.cpu()), vo)


def test_multi_fused_append_slot_rules(pk):
    """A slot that is not its token's is not written (PA_DEVERR_APPEND_SLOT); a
    negative slot writes nothing; the other tokens are written."""
    QL = 3
    q, kc, vc, tables, lens, slots, kn, vn, torch = _append_case([40, 70], QL, 16, 4, seed=95)
    bad = slots.copy()
    bad[1] = slots[1] + 1 if slots[1] % 16 != 15 else slots[1] - 1  # wrong offset
    bad[4] = -1
    kc2, vc2 = kc.clone(), vc.clone()
    pk.pa_append_decode(q, kc2, vc2, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                        int(lens.max()), kn, vn, torch.from_numpy(bad).cuda())
    torch.cuda.synchronize()
    assert pk.pa_device_errors() & DEVERR_APPEND_SLOT
    written = [t for t in range(len(slots)) if t not in (1, 4)]
    ko, vo = oracle.reshape_and_cache(kn.cpu()[written], vn.cpu()[written],
                                      oracle.bf16_bits(kc.cpu()), oracle.bf16_bits(vc.cpu()),
                                      slots[written])
    assert np.array_equal(oracle.bf16_bits(kc2.cpu()), ko)
    assert np.array_equal(oracle.bf16_bits(vc2.cpu()), vo)


@pytest.mark.parametrize("QL,pinned", [(2, True), (4, True), (3, False)])
def test_multi_step_host_matches_device_step(pk, QL, pinned):
    """pa_step_host with query_len Q (q, k_new, v_new, slots and the output
    carrying Q rows per sequence) gives pa_append_decode's output and caches
    bit for bit, with pinned and pageable buffers."""
    lens = [QL, 17, 33, 16 + QL, 500, 2049]
    q, kc, vc, tables, lens, slots, kn, vn, torch = _append_case(lens, QL, 32, 8, seed=120 + QL)
    kd, vd = kc.clone(), vc.clone()
    want = pk.pa_append_decode(q, kd, vd, torch.from_numpy(tables).cuda(),
                               torch.from_numpy(lens).cuda(), int(lens.max()), kn, vn,
                               torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    kh, vh = kc.clone(), vc.clone()
    B, _, Hq, D = q.shape
    p = pk.make_step_host_params(kh, vh, B, Hq, tables.shape[1], int(lens.max()), query_len=QL)
    host_in = pk.pack_step_inputs(p, q.cpu(), kn.cpu(), vn.cpu(), slots, tables, lens, pin=pinned)
    host_out = torch.empty((B, QL, Hq, D), dtype=torch.bfloat16)
    if pinned:
        host_out = host_out.pin_memory()
    ws = torch.empty(pk.pa_step_host_workspace_size(p), dtype=torch.uint8, device="cuda")
    pk.pa_step_host(p, host_in, host_out, ws)
    assert pk.pa_device_errors() == 0
    assert torch.equal(host_out.view(torch.int16), want.cpu().view(torch.int16))
    assert torch.equal(kh.view(torch.int16), kd.view(torch.int16))
    assert torch.equal(vh.view(torch.int16), vd.view(torch.int16))
    ko, vo = oracle.reshape_and_cache(kn.cpu(), vn.cpu(), oracle.bf16_bits(kc.cpu()),
                                      oracle.bf16_bits(vc.cpu()), slots)
    harness.assert_close(harness.bf16_tensor_to_f64(host_out),
                         oracle.paged_decode_multi(q.cpu(), ko, vo, tables, lens))


def test_multi_cuda_core_step_host_matches_device_step(pk):
    """The same on the CUDA-core kernel (its write kernel, then the decode)."""
    QL = 3
    lens = [QL, 17, 33, 16 + QL, 600]
    q, kc, vc, tables, lens, slots, kn, vn, torch = _append_case(lens, QL, 32, 8, seed=540)
    kd, vd = kc.clone(), vc.clone()
    want = pk.pa_append_decode(q, kd, vd, torch.from_numpy(tables).cuda(),
                               torch.from_numpy(lens).cuda(), int(lens.max()), kn, vn,
                               torch.from_numpy(slots).cuda(), variant=pk.DECODE_CUDA_CORE)
    torch.cuda.synchronize()
    kh, vh = kc.clone(), vc.clone()
    B, _, Hq, D = q.shape
    p = pk.make_step_host_params(kh, vh, B, Hq, tables.shape[1], int(lens.max()), query_len=QL,
                                 variant=pk.DECODE_CUDA_CORE)
    host_in = pk.pack_step_inputs(p, q.cpu(), kn.cpu(), vn.cpu(), slots, tables, lens, pin=True)
    host_out = torch.empty((B, QL, Hq, D), dtype=torch.bfloat16).pin_memory()
    ws = torch.empty(pk.pa_step_host_workspace_size(p), dtype=torch.uint8, device="cuda")
    pk.pa_step_host(p, host_in, host_out, ws)
    assert pk.pa_device_errors() == 0
    assert torch.equal(host_out.view(torch.int16), want.cpu().view(torch.int16))
    assert torch.equal(kh.view(torch.int16), kd.view(torch.int16))
    assert torch.equal(vh.view(torch.int16), vd.view(torch.int16))


# ---------------------------------------------------------------- 8-bit cache


def _fp8_multi_case(pk, lens, QL, Hq, Hkv, seed):
    import torch

    D = 128
    lens = np.asarray(lens, dtype=np.int64)
    need = int(((lens + 15) // 16).sum())
    NB = need + 3
    order = np.random.default_rng(seed).permutation(NB).astype(np.int32)
    tables = workloads.sequential_tables(lens, order, 16)
    q = workloads.bf16_normal((len(lens), QL, Hq, D), seed + 1, "cuda")
    kn = workloads.bf16_normal((NB * 16, Hkv, D), seed + 2, "cuda")
    vn = workloads.bf16_normal((NB * 16, Hkv, D), seed + 3, "cuda")
    rng = np.random.default_rng(seed + 4)
    ks = torch.from_numpy((0.05 * np.exp(rng.uniform(-0.5, 0.5, Hkv))).astype(np.float32)).cuda()
    vs = torch.from_numpy((0.03 * np.exp(rng.uniform(-0.5, 0.5, Hkv))).astype(np.float32)).cuda()
    k8 = torch.zeros((NB, Hkv, 16, D), dtype=torch.uint8, device="cuda")
    v8 = torch.zeros((NB, Hkv, D, 16), dtype=torch.uint8, device="cuda")
    pk.pa_reshape_and_cache_fp8(kn, vn, k8, v8, torch.arange(NB * 16, device="cuda"), ks, vs)
    for b, L in enumerate(lens):
        if L % 16:
            blk = int(tables[b, (L - 1) // 16])
            k8[blk, :, L % 16:, :] = 0x7F  # E4M3 NaN
            v8[blk, :, :, L % 16:] = 0x7F
    torch.cuda.synchronize()
    return q, k8, v8, ks, vs, tables, lens.astype(np.int32), torch


@pytest.mark.parametrize("G,Hkv,QL", [(4, 8, 2), (1, 8, 4), (2, 4, 4), (4, 4, 4), (8, 2, 2),
                                      (4, 1, 3)])
def test_multi_fp8_edge_lengths(pk, G, Hkv, QL):
    lens = [L for L in (QL, 15, 16, 17, 18, 100, 513, 1025, 4098) if L >= QL]
    q, k8, v8, ks, vs, tables, lens, torch = _fp8_multi_case(pk, lens, QL, G * Hkv, Hkv,
                                                             seed=G * 10 + Hkv + QL)
    out = pk.pa_decode(q, k8, v8, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                       max_context_len=int(lens.max()), k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    want = oracle.paged_decode_multi_fp8(q.cpu(), k8.cpu().numpy(), v8.cpu().numpy(),
                                         ks.cpu().numpy(), vs.cpu().numpy(), tables, lens)
    harness.assert_close(harness.bf16_tensor_to_f64(out), want)
    assert pk.pa_device_errors() == 0


@pytest.mark.parametrize("G,Hkv,QL", [(8, 8, 4), (4, 8, 8), (4, 8, 5), (2, 2, 16)])
def test_multi_fp8_column_groups(pk, G, Hkv, QL):
    """The 8-bit cache allows 64 columns: 8 query heads per KV head take one
    token per group, four take two."""
    lens = [L for L in (QL, 15, 16, 17, 100, 513, 2049) if L >= QL]
    q, k8, v8, ks, vs, tables, lens, torch = _fp8_multi_case(pk, lens, QL, G * Hkv, Hkv,
                                                             seed=350 + G * 10 + QL)
    out = pk.pa_decode(q, k8, v8, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                       max_context_len=int(lens.max()), k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    want = oracle.paged_decode_multi_fp8(q.cpu(), k8.cpu().numpy(), v8.cpu().numpy(),
                                         ks.cpu().numpy(), vs.cpu().numpy(), tables, lens)
    harness.assert_close(harness.bf16_tensor_to_f64(out), want)
    assert pk.pa_device_errors() == 0


def test_multi_fp8_llama8b_layer(pk):
    """64 sequences, 32/8 heads, U[128, 2048], 2 new tokens (64 columns)."""
    r = workloads.llama8b_layer()
    q, k8, v8, ks, vs, tables, lens, torch = _fp8_multi_case(pk, r.lens0 + 2, 2, 32, 8, seed=96)
    out = pk.pa_decode(q, k8, v8, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                       max_context_len=int(lens.max()), k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    want = oracle.paged_decode_multi_fp8(q.cpu(), k8.cpu().numpy(), v8.cpu().numpy(),
                                         ks.cpu().numpy(), vs.cpu().numpy(), tables, lens)
    harness.assert_close(harness.bf16_tensor_to_f64(out), want)
    assert pk.pa_device_errors() == 0
