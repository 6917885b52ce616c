"""The C++ block pool against the oracle's block-manager model.

Both follow the same stated policy (LIFO free list seeded from a given
order, a fresh block at each block boundary, copy-on-write into shared
blocks, state unchanged on failure), so their block tables, slots,
copy-on-write pairs, refcounts and stats must agree exactly on any sequence
of operations. Also: the pages' allocator arithmetic and the shared-prefix
workload's refcounts.
"""
import json
import os

import numpy as np
import pytest

import oracle
import workloads


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_92_gb300 import build

    build.build()
    import paged_kv_cache_92_gb300 as pk

    return pk


def _snapshot(pool, model, seqs):
    for s in seqs:
        assert pool.table(s) == model.table(s)
        assert pool.length(s) == model.length(s)
    for b in range(model.num_blocks):
        assert pool.refcount(b) == model.ref[b]
    st = pool.stats()
    ms = model.stats()
    assert (st["free_blocks"], st["used_blocks"], st["shared_blocks"], st["max_refcount"]) == \
        (ms["free"], ms["used"], ms["shared"], ms["max_refcount"])


@pytest.mark.parametrize("seed", range(6))
def test_random_operation_sequences_match_model(pk, seed):
    rng = np.random.default_rng(seed)
    NB, BS = 48, 4
    order = rng.permutation(NB)
    pool = pk.Pool(NB, BS, free_order=order)
    model = oracle.PoolModel(NB, BS, free_order=order)
    live = []
    for step in range(400):
        op = rng.choice(["create", "append", "append_n", "fork", "free"],
                        p=[0.1, 0.45, 0.15, 0.15, 0.15])
        if op == "create" or not live:
            a, b = pool.seq_create(), model.seq_create()
            assert a == b
            live.append(a)
        elif op == "append":
            s = int(rng.choice(live))
            try:
                want = model.append_slot(s)
            except oracle.PoolOOM:
                with pytest.raises(pk.PoolOOM):
                    pool.append_slot(s)
            else:
                assert pool.append_slot(s) == want
        elif op == "append_n":
            s = int(rng.choice(live))
            n = int(rng.integers(0, 9))
            before = (list(model.free), list(model.ref), model.table(s), model.length(s))
            try:
                want = model.append_tokens(s, n)
            except oracle.PoolOOM:
                # the model stopped part-way; the C pool is all-or-nothing
                model.free, model.ref = before[0], before[1]
                model.tables[s], model.lens[s] = before[2], before[3]
                with pytest.raises(pk.PoolOOM):
                    pool.append_tokens(s, n)
            else:
                assert pool.append_tokens(s, n) == (want[0], want[1])
        elif op == "fork":
            s = int(rng.choice(live))
            n = int(rng.integers(0, model.length(s) + 1))
            c1, c2 = pool.seq_fork(s, n), model.seq_fork(s, n)
            assert c1 == c2
            live.append(c1)
        else:
            s = int(rng.choice(live))
            pool.seq_free(s)
            model.seq_free(s)
            live.remove(s)
        _snapshot(pool, model, live)


def test_worked_example_through_the_pool(pk, golden_dir):
    gold = json.load(open(os.path.join(golden_dir, "worked_block_table.json")))
    table = gold["block_table"]
    order = table + [b for b in range(16) if b not in table]
    pool = pk.Pool(16, gold["block_size"], free_order=order)
    s = pool.seq_create()
    slots, cows = pool.append_tokens(s, gold["num_tokens"])
    assert pool.table(s) == table and slots == gold["slots"] and cows == []


def test_allocator_arithmetic(pk, golden_dir):
    gold = json.load(open(os.path.join(golden_dir, "allocator_arithmetic.json")))
    for case in gold["cases"]:
        pool = pk.Pool(400, 16)
        s = pool.seq_create()
        pool.append_tokens(s, case["tokens"], want_slots=False)
        assert len(pool.table(s)) == case["blocks"]
    share = gold["prefix_share"]
    pool = pk.Pool(200, 16)
    pre = pool.seq_create()
    pool.append_tokens(pre, share["shared_blocks"] * 16, want_slots=False)
    used = pool.stats()["used_blocks"]
    req = pool.seq_fork(pre, share["shared_blocks"] * 16)
    pool.append_tokens(req, share["prompt_tokens"] - share["shared_blocks"] * 16, want_slots=False)
    assert len(pool.table(req)) == 75
    assert pool.stats()["used_blocks"] - used == share["new_blocks"]


def test_error_codes(pk):
    pool = pk.Pool(2, 16)
    with pytest.raises(pk.PagedKVError) as e:
        pool.decref(0)
    assert e.value.status == 4  # PA_ERR_REFCOUNT
    with pytest.raises(pk.PagedKVError) as e:
        pool.incref(5)
    assert e.value.status == 5  # PA_ERR_BOUNDS
    assert pool.refcount(9) == -1
    s = pool.seq_create()
    pool.append_tokens(s, 32, want_slots=False)
    with pytest.raises(pk.PoolOOM):
        pool.append_slot(s)
    assert pool.length(s) == 32 and pool.stats()["free_blocks"] == 0
    with pytest.raises(pk.PagedKVError):
        pk.Pool(4, 16, free_order=[0, 1, 1, 2])
    with pytest.raises(pk.PagedKVError):
        pool.seq_fork(s, 33)
    pool.seq_free(s)
    with pytest.raises(pk.PagedKVError):
        pool.seq_free(s)
    assert pool.stats()["free_blocks"] == 2


def test_shared_prefix_workload_refcounts(pk):
    """Shared-prefix layout: 512 sequences on 64 shared blocks, 32 copy-on-writes."""
    r = workloads.shared_prefix()
    pool = pk.Pool(r.num_blocks, 16, free_order=r.free_order)
    model = oracle.PoolModel(r.num_blocks, 16, free_order=r.free_order)
    div = set(r.diverge_seqs.tolist())
    for P in (pool, model):
        root = P.seq_create()
        if isinstance(P, oracle.PoolModel):
            P.append_tokens(root, r.shared_prefix_tokens)
        else:
            P.append_tokens(root, r.shared_prefix_tokens, want_slots=False)
        seqs = [root]
        for b in range(1, r.num_seqs):
            n = int(r.lens0[b]) if b in div else r.shared_prefix_tokens
            seqs.append(P.seq_fork(root, n))
        for b in range(r.num_seqs):
            if b not in div:
                P.append_tokens(seqs[b], int(r.lens0[b]) - r.shared_prefix_tokens)
    shared = model.table(0)[:64]
    assert all(model.ref[x] == 512 for x in shared)
    assert all(pool.refcount(x) == 512 for x in shared)
    cows_pool, cows_model = [], []
    for b in range(r.num_seqs):
        sp, cp = pool.append_slot(b)
        sm, cm = model.append_slot(b)
        assert (sp, cp) == (sm, cm)
        if cp:
            cows_pool.append(cp)
    assert len(cows_pool) == 32
    assert all(src == shared[63] for src, _ in cows_pool)
    assert pool.refcount(shared[63]) == 480
    assert all(pool.refcount(x) == 512 for x in shared[:63])
