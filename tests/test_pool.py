"""The C++ block pool against the oracle's block-manager model.

Both follow the same stated policy (LIFO free list seeded from a given
order, a fresh block at each block boundary, copy-on-write into shared
blocks, state unchanged on failure), so their block tables, slots,
copy-on-write pairs, refcounts and stats must agree exactly on any sequence
of operations. Also: the pages' allocator arithmetic and the shared-prefix
workload's refcounts.
"""
import copy
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
    assert pool.prefix_stats() == model.prefix_stats()


@pytest.mark.parametrize("seed", range(6))
def test_random_operation_sequences_match_model(pk, seed):
    rng = np.random.default_rng(seed)
    NB, BS = 48, 4
    order = rng.permutation(NB)
    pool = pk.Pool(NB, BS, free_order=order)
    model = oracle.PoolModel(NB, BS, free_order=order)
    live = []
    # prompts share prefixes with a few base texts, so the prefix cache hits
    bases = [rng.integers(0, 50, size=40) for _ in range(3)]
    for step in range(400):
        op = rng.choice(["create", "prompt", "append", "append_n", "fork", "free"],
                        p=[0.06, 0.1, 0.4, 0.14, 0.15, 0.15])
        if op == "prompt":
            base = bases[int(rng.integers(0, 3))]
            toks = np.concatenate([base[:int(rng.integers(0, 41))],
                                   rng.integers(0, 50, size=int(rng.integers(0, 11)))])
            try:
                want = model.create_prompt(toks)
            except oracle.PoolOOM:
                with pytest.raises(pk.PoolOOM):
                    pool.create_prompt(toks)
            else:
                assert pool.create_prompt(toks) == want
                live.append(want[0])
        elif op == "create" or not live:
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
            before = copy.deepcopy(model.__dict__)
            try:
                want = model.append_tokens(s, n)
            except oracle.PoolOOM:
                # the model stopped part-way; the C pool is all-or-nothing
                model.__dict__.update(before)
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


def test_prefix_cache_worked_trace(pk, golden_dir):
    """The pages' end-to-end trace: a 1,200-token prompt whose first 900 tokens
    are a preamble already seen maps 56 cached blocks (896 tokens, the block
    granularity) and takes 19 fresh ones, 75 in all; the preamble stays warm
    after the first request ends."""
    share = json.load(open(os.path.join(golden_dir, "allocator_arithmetic.json")))["prefix_share"]
    rng = np.random.default_rng(3)
    preamble = rng.integers(0, 32000, size=900)
    first = np.concatenate([preamble, rng.integers(0, 32000, size=300)])
    second = np.concatenate([preamble, rng.integers(0, 32000, size=300)])
    for P in (pk.Pool(300, 16), oracle.PoolModel(300, 16)):
        a, cached_a, _ = P.create_prompt(first)
        assert cached_a == 0
        P.seq_free(a)  # the request completes; its blocks stay cached
        used0 = P.stats()["used"] if isinstance(P, oracle.PoolModel) else P.stats()["used_blocks"]
        b, cached_b, slots = P.create_prompt(second)
        assert cached_b == share["shared_blocks"] * 16 == 896
        assert len(P.table(b)) == share["prompt_tokens"] // 16 == 75
        used1 = P.stats()["used"] if isinstance(P, oracle.PoolModel) else P.stats()["used_blocks"]
        assert used1 - used0 == 75 and len(slots) == 1200
        st = P.prefix_stats()
        assert st["hits"] == 56 and st["lookups"] == 150


def test_prefix_cache_eviction_order_and_immutability(pk):
    """Never-cached free blocks go first, then the least recently freed cached
    block (which leaves the cache); an append into a cached block copies it
    even when no one else holds it."""
    for P in (pk.Pool(6, 4), oracle.PoolModel(6, 4)):
        s1, _, _ = P.create_prompt([1, 2, 3, 4, 5, 6, 7, 8])   # 2 cached blocks
        s2, _, _ = P.create_prompt([9, 9, 9, 9])               # 1 cached block
        t1, t2 = P.table(s1), P.table(s2)
        P.seq_free(s1)
        P.seq_free(s2)  # evictable, oldest first: t1[0], t1[1], t2[0]
        assert P.prefix_stats()["evictable_blocks"] == 3
        fresh = [P.alloc() for _ in range(3)]  # the never-cached blocks
        assert not set(fresh) & set(t1 + t2)
        assert P.alloc() == t1[0]               # then the oldest cached block
        assert P.prefix_stats()["cached_blocks"] == 2
        # a prompt matching the second cached prefix revives it (no allocation)
        s3, cached, _ = P.create_prompt([9, 9, 9, 9, 1])
        assert cached == 4 and P.table(s3)[0] == t2[0]
        # fork a partial view of the cached block, drop the owner, append:
        # the cached block is copied, not written
        for b in fresh + [t1[0]]:
            P.decref(b)
        c = P.seq_fork(s3, 2)
        P.seq_free(s3)
        slot, cow = P.append_slot(c)
        assert cow is not None and cow[0] == t2[0]
