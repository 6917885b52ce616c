"""Pins for the oracle: it is checked against things other than itself.

* the pages' worked block-table example (tests/golden/worked_block_table.json)
* brute force (pure-Python loops) and an independent numpy twin on tiny inputs
* a library routine: torch scaled_dot_product_attention in float64
* closed-form invariants: weights sum to 1, L=1 returns v_0, equal keys give
  the mean of V, a dominant score selects its value row, output unchanged
  under any physical placement, GQA equals MHA with repeated KV heads, the
  split-K log-sum-exp merge equals the unsplit result
* masking: NaN in padding slots never reaches a result
* mutation checks: plausible mistakes planted in a copy of the numpy twin
  (dropped scale, wrong GQA map, wrong in-block offset, off-by-one mask) are
  each rejected by at least one of the pins above.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import PoolModel


def _bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def _random_case(seed, B=3, Hq=4, Hkv=2, D=8, BS=4, lens=(1, 3, 9), NB=None):
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int32)
    nblk = (lens + BS - 1) // BS
    need = int(nblk.sum())
    NB = NB or need + 3
    perm = rng.permutation(NB).astype(np.int32)
    mb = int(nblk.max())
    tables = np.full((B, mb), -1, dtype=np.int32)
    pos = 0
    for b in range(B):
        tables[b, :nblk[b]] = perm[pos:pos + nblk[b]]
        pos += nblk[b]
    q = _bf16((B, Hq, D), seed + 1)
    kc = _bf16((NB, Hkv, BS, D), seed + 2)
    vc = _bf16((NB, Hkv, BS, D), seed + 3)
    return q, kc, vc, tables, lens


def _sdpa_unpaged(q, K, V, scale=None):
    """torch SDPA, float64, KV heads repeated to the query heads."""
    Hq = q.shape[0]
    G = Hq // K.shape[0]
    Kr = K.repeat_interleave(G, dim=0)  # [Hq, L, D]
    Vr = V.repeat_interleave(G, dim=0)
    out = torch.nn.functional.scaled_dot_product_attention(
        q[:, None, :], Kr, Vr, scale=scale)  # [Hq, 1, D]
    return out[:, 0, :]


# ---------------------------------------------------------------- worked example

def test_worked_example_slots(golden_dir):
    gold = json.load(open(os.path.join(golden_dir, "worked_block_table.json")))
    BS = gold["block_size"]
    table = gold["block_table"]
    others = [b for b in range(16) if b not in table]
    pool = PoolModel(16, BS, free_order=table + others)
    s = pool.seq_create()
    slots, cows = pool.append_tokens(s, gold["num_tokens"])
    assert pool.table(s) == table
    assert slots == gold["slots"]
    assert cows == []


def test_worked_example_gather_equals_unpaged(golden_dir):
    gold = json.load(open(os.path.join(golden_dir, "worked_block_table.json")))
    BS, n = gold["block_size"], gold["num_tokens"]
    NB, Hkv, D = 12, 1, 4
    Kt = _bf16((n, D), 11)  # token t's key, in logical order
    Vt = _bf16((n, D), 12)
    kc = torch.full((NB, Hkv, BS, D), float("nan"), dtype=torch.bfloat16)
    vc = kc.clone()
    for t, slot in enumerate(gold["slots"]):
        kc[slot // BS, 0, slot % BS] = Kt[t]
        vc[slot // BS, 0, slot % BS] = Vt[t]
    q = _bf16((1, 2, D), 13)
    tables = np.array([gold["block_table"]], dtype=np.int32)
    lens = np.array([n], dtype=np.int32)
    got = oracle.paged_decode(q, kc, vc, tables, lens)
    ref = _sdpa_unpaged(q[0].double(), Kt.double()[None], Vt.double()[None]).numpy()
    np.testing.assert_allclose(got[0], ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- brute force / twin / library

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_oracle_matches_brute_force(seed):
    q, kc, vc, tables, lens = _random_case(seed)
    got = oracle.paged_decode(q, kc, vc, tables, lens)
    twin = oracle.paged_decode_numpy(q, kc, vc, tables, lens)
    np.testing.assert_allclose(got, twin, rtol=0, atol=1e-12)
    qd, kd, vd = (oracle.bf16_to_f64(x) for x in (q, kc, vc))
    B, Hq, D = qd.shape
    Hkv, BS = kd.shape[1], kd.shape[2]
    G = Hq // Hkv
    for b in range(B):
        for g in range(Hkv):
            # contiguous K/V assembled by walking the table with plain loops
            K, V = [], []
            for t in range(int(lens[b])):
                blk = int(tables[b][t // BS])
                K.append(list(kd[blk, g, t % BS]))
                V.append(list(vd[blk, g, t % BS]))
            ref = oracle.brute_force_decode([list(qd[b, h]) for h in range(g * G, g * G + G)],
                                            K, V, 1.0 / math.sqrt(D))
            np.testing.assert_allclose(got[b, g * G:(g + 1) * G], np.array(ref), rtol=0, atol=1e-12)


def test_identity_table_equals_library_sdpa():
    B, Hq, Hkv, D, BS = 2, 8, 2, 16, 4
    lens = np.array([13, 7], dtype=np.int32)
    mb = 4
    tables = np.arange(B * mb, dtype=np.int32).reshape(B, mb)
    q = _bf16((B, Hq, D), 21)
    kc = _bf16((B * mb, Hkv, BS, D), 22)
    vc = _bf16((B * mb, Hkv, BS, D), 23)
    got = oracle.paged_decode(q, kc, vc, tables, lens)
    for b in range(B):
        L = int(lens[b])
        K = kc[b * mb:(b + 1) * mb].double().permute(1, 0, 2, 3).reshape(Hkv, mb * BS, D)[:, :L]
        V = vc[b * mb:(b + 1) * mb].double().permute(1, 0, 2, 3).reshape(Hkv, mb * BS, D)[:, :L]
        ref = _sdpa_unpaged(q[b].double(), K, V).numpy()
        np.testing.assert_allclose(got[b], ref, rtol=0, atol=1e-12)


def test_units_subset_matches_full():
    q, kc, vc, tables, lens = _random_case(5)
    full = oracle.paged_decode(q, kc, vc, tables, lens)
    units = [(2, 3), (0, 1), (1, 0)]
    sub = oracle.paged_decode(q, kc, vc, tables, lens, units=units)
    for i, (b, h) in enumerate(units):
        assert np.array_equal(sub[i], full[b, h])


# ---------------------------------------------------------------- invariants

def test_permutation_invariance_is_exact():
    q, kc, vc, tables, lens = _random_case(7, lens=(5, 16, 17))
    base = oracle.paged_decode(q, kc, vc, tables, lens)
    NB = kc.shape[0]
    perm = np.random.default_rng(99).permutation(NB)
    kc2 = torch.empty_like(kc)
    vc2 = torch.empty_like(vc)
    kc2[torch.from_numpy(perm)] = kc
    vc2[torch.from_numpy(perm)] = vc
    t2 = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    moved = oracle.paged_decode(q, kc2, vc2, t2, lens)
    assert np.array_equal(base, moved)


def test_gqa_equals_mha_with_repeated_kv_heads():
    q, kc, vc, tables, lens = _random_case(8, Hq=8, Hkv=2)
    gqa = oracle.paged_decode(q, kc, vc, tables, lens)
    mha = oracle.paged_decode(q, kc.repeat_interleave(4, dim=1), vc.repeat_interleave(4, dim=1),
                              tables, lens)
    assert np.array_equal(gqa, mha)


def test_length_one_returns_v0_exactly():
    q, kc, vc, tables, lens = _random_case(9, lens=(1, 1, 1))
    got = oracle.paged_decode(q, kc, vc, tables, lens)
    vd = oracle.bf16_to_f64(vc)
    G = q.shape[1] // kc.shape[1]
    for b in range(3):
        for h in range(q.shape[1]):
            assert np.array_equal(got[b, h], vd[tables[b, 0], h // G, 0])


def test_weights_sum_to_one():
    q, kc, vc, tables, lens = _random_case(10, lens=(3, 40, 77), BS=8)
    ones = torch.ones_like(vc)
    got = oracle.paged_decode(q * 4, kc, ones, tables, lens)
    np.testing.assert_allclose(got, 1.0, rtol=0, atol=1e-12)


def test_equal_keys_give_mean_of_v():
    q, kc, vc, tables, lens = _random_case(11, lens=(6, 21, 2))
    kc_const = torch.zeros_like(kc) + kc[0, 0, 0]
    got = oracle.paged_decode(q, kc_const, vc, tables, lens)
    vd = oracle.bf16_to_f64(vc)
    G = q.shape[1] // kc.shape[1]
    for b in range(3):
        for h in range(q.shape[1]):
            V = oracle.gather_contiguous(vd, tables[b], int(lens[b]), h // G)
            np.testing.assert_allclose(got[b, h], V.mean(axis=0), rtol=0, atol=1e-12)


def test_dominant_score_selects_its_value_row():
    B, Hq, Hkv, D, BS = 1, 1, 1, 8, 4
    L = 10
    tables = np.array([[2, 0, 1]], dtype=np.int32)
    kc = torch.zeros((3, Hkv, BS, D), dtype=torch.bfloat16)
    vc = _bf16((3, Hkv, BS, D), 31)
    q = torch.zeros((B, Hq, D), dtype=torch.bfloat16)
    q[0, 0, 0] = 64.0
    t_star = 6  # logical token 6 -> table[1] = block 0, offset 2
    kc[0, 0, 2, 0] = 64.0  # score = 64*64/sqrt(8) ~ 1448 above every other
    got = oracle.paged_decode(q, kc, vc, tables, np.array([L], dtype=np.int32))
    want = oracle.bf16_to_f64(vc)[0, 0, 2]
    assert t_star // BS == 1
    np.testing.assert_allclose(got[0, 0], want, rtol=0, atol=1e-300)


def test_padding_slots_never_read():
    q, kc, vc, tables, lens = _random_case(12, lens=(3, 6, 11), BS=4)
    base = oracle.paged_decode(q, kc, vc, tables, lens)
    kc2, vc2 = kc.clone(), vc.clone()
    for b in range(3):
        L = int(lens[b])
        last = tables[b, (L - 1) // 4]
        kc2[last, :, L % 4 or 4:] = float("nan")
        vc2[last, :, L % 4 or 4:] = float("nan")
    # unused blocks too
    used = set(tables[tables >= 0].tolist())
    for blk in range(kc.shape[0]):
        if blk not in used:
            kc2[blk] = float("nan")
            vc2[blk] = float("nan")
    got = oracle.paged_decode(q, kc2, vc2, tables, lens)
    assert np.isfinite(got).all()
    assert np.array_equal(base, got)


@pytest.mark.parametrize("P", [4, 8, 12, 16, 64])
def test_split_merge_identity(P):
    q, kc, vc, tables, lens = _random_case(13, lens=(1, 16, 33), BS=4)
    full = oracle.paged_decode(q, kc, vc, tables, lens)
    qd, kd, vd = (oracle.bf16_to_f64(x) for x in (q, kc, vc))
    G = qd.shape[1] // kd.shape[1]
    for b in range(3):
        for h in range(qd.shape[1]):
            K = oracle.gather_contiguous(kd, tables[b], int(lens[b]), h // G)
            V = oracle.gather_contiguous(vd, tables[b], int(lens[b]), h // G)
            parts = oracle.partition_decode(qd[b, h], K, V, 1 / math.sqrt(qd.shape[2]), P)
            assert len(parts) == -(-int(lens[b]) // P)
            np.testing.assert_allclose(oracle.merge_partitions(parts), full[b, h], rtol=0, atol=1e-12)


def test_scale_argument_is_used():
    q, kc, vc, tables, lens = _random_case(14)
    a = oracle.paged_decode(q, kc, vc, tables, lens)
    b = oracle.paged_decode(q, kc, vc, tables, lens, scale=1.0 / math.sqrt(q.shape[2]))
    c = oracle.paged_decode(q, kc, vc, tables, lens, scale=1.0)
    assert np.array_equal(a, b)
    assert not np.allclose(a[1:], c[1:])


def test_bad_table_entry_is_an_error():
    q, kc, vc, tables, lens = _random_case(15)
    bad = tables.copy()
    bad[2, 0] = kc.shape[0]  # out of range
    with pytest.raises(ValueError):
        oracle.paged_decode(q, kc, vc, bad, lens)


# ---------------------------------------------------------------- mutation checks

def _twin_mutant(kind):
    """A copy of the numpy twin with one plausible mistake planted in it."""
    def run(q, k_cache, v_cache, block_tables, context_lens):
        qd, kd, vd = (oracle.bf16_to_f64(x) for x in (q, k_cache, v_cache))
        B, Hq, D = qd.shape
        Hkv, BS = kd.shape[1], kd.shape[2]
        G = Hq // Hkv
        scale = 1.0 if kind == "no_scale" else 1 / math.sqrt(D)
        out = np.empty((B, Hq, D))
        for b in range(B):
            L = int(context_lens[b]) - (1 if kind == "mask_off_by_one" and context_lens[b] > 1 else 0)
            for h in range(Hq):
                g = h % Hkv if kind == "gqa_modulo" else h // G
                t = np.arange(L)
                off = (t + 1) % BS if kind == "offset" else t % BS
                blk = block_tables[b][t // BS]
                K, V = kd[blk, g, off], vd[blk, g, off]
                s = K @ qd[b, h] * scale
                w = np.exp(s - s.max())
                out[b, h] = (w / w.sum()) @ V
        return out
    return run


def _brute_force_pin(q, kc, vc, tables, lens):
    """The brute-force pin: each sequence's K/V assembled by walking its table
    with plain loops, then the pure-Python triple loop."""
    qd, kd, vd = (oracle.bf16_to_f64(x) for x in (q, kc, vc))
    B, Hq, D = qd.shape
    Hkv, BS = kd.shape[1], kd.shape[2]
    G = Hq // Hkv
    out = np.empty((B, Hq, D))
    for b in range(B):
        for g in range(Hkv):
            K, V = [], []
            for t in range(int(lens[b])):
                blk = int(tables[b][t // BS])
                K.append(list(kd[blk, g, t % BS]))
                V.append(list(vd[blk, g, t % BS]))
            out[b, g * G:(g + 1) * G] = np.array(oracle.brute_force_decode(
                [list(qd[b, h]) for h in range(g * G, g * G + G)], K, V, 1.0 / math.sqrt(D)))
    return out


def _identity_case(seed):
    """An identity-table case for the library pin (torch SDPA in float64)."""
    B, Hq, Hkv, D, BS, mb = 2, 4, 2, 8, 4, 4
    lens = np.array([13, 7], dtype=np.int32)
    tables = np.arange(B * mb, dtype=np.int32).reshape(B, mb)
    q = _bf16((B, Hq, D), seed + 1)
    kc = _bf16((B * mb, Hkv, BS, D), seed + 2)
    vc = _bf16((B * mb, Hkv, BS, D), seed + 3)
    return q, kc, vc, tables, lens


def _sdpa_pin(q, kc, vc, tables, lens):
    B, Hq, D = q.shape
    Hkv, BS = kc.shape[1], kc.shape[2]
    mb = tables.shape[1]
    out = np.empty((B, Hq, D))
    for b in range(B):
        L = int(lens[b])
        K = kc[b * mb:(b + 1) * mb].double().permute(1, 0, 2, 3).reshape(Hkv, mb * BS, D)[:, :L]
        V = vc[b * mb:(b + 1) * mb].double().permute(1, 0, 2, 3).reshape(Hkv, mb * BS, D)[:, :L]
        out[b] = _sdpa_unpaged(q[b].double(), K, V).numpy()
    return out


def _rejected_by_a_pin(impl):
    """True when ``impl`` disagrees with the brute-force pin on a shuffled
    table or with the library pin on an identity table."""
    q, kc, vc, tables, lens = _random_case(16, Hq=4, Hkv=2, lens=(5, 9, 13))
    bf = np.abs(impl(q, kc, vc, tables, lens) - _brute_force_pin(q, kc, vc, tables, lens)).max()
    q, kc, vc, tables, lens = _identity_case(17)
    lib = np.abs(impl(q, kc, vc, tables, lens) - _sdpa_pin(q, kc, vc, tables, lens)).max()
    return bf > 1e-3 or lib > 1e-3


def test_pins_accept_the_unmutated_twin():
    """Control for the mutation test: the unmutated twin passes both pins."""
    assert not _rejected_by_a_pin(oracle.paged_decode_numpy)
    assert not _rejected_by_a_pin(_twin_mutant("none"))


@pytest.mark.parametrize("kind", ["no_scale", "gqa_modulo", "offset", "mask_off_by_one"])
def test_pins_reject_planted_mistakes(kind):
    """Each planted mistake is caught by the brute-force or the library pin
    themselves (not by a comparison with the oracle)."""
    assert _rejected_by_a_pin(_twin_mutant(kind))


# ---------------------------------------------------------------- cache writes

def test_reshape_and_cache_matches_indexing_definition():
    NB, Hkv, BS, D, T = 6, 2, 4, 8, 5
    kc = _bf16((NB, Hkv, BS, D), 41)
    vc = _bf16((NB, Hkv, BS, D), 42)
    kn = _bf16((T, Hkv, D), 43)
    vn = _bf16((T, Hkv, D), 44)
    slots = np.array([5, -1, 0, 23, 14], dtype=np.int64)
    k2, v2 = oracle.reshape_and_cache(kn, vn, kc, vc, slots)
    ke = oracle.bf16_bits(kc).copy()
    ve = oracle.bf16_bits(vc).copy()
    for t, s in enumerate(slots):
        if s >= 0:
            ke[s // BS, :, s % BS, :] = oracle.bf16_bits(kn)[t]
            ve[s // BS, :, s % BS, :] = oracle.bf16_bits(vn)[t]
    assert np.array_equal(k2, ke) and np.array_equal(v2, ve)
    # untouched slots keep their bits
    touched = {(s // BS, s % BS) for s in slots if s >= 0}
    kb = oracle.bf16_bits(kc)
    for blk in range(NB):
        for off in range(BS):
            if (blk, off) not in touched:
                assert np.array_equal(k2[blk, :, off], kb[blk, :, off])


def test_reshape_and_cache_then_decode_reads_the_new_token(golden_dir):
    gold = json.load(open(os.path.join(golden_dir, "worked_block_table.json")))
    BS = gold["block_size"]
    NB, Hkv, D = 12, 1, 4
    kc = torch.full((NB, Hkv, BS, D), float("nan"), dtype=torch.bfloat16)
    vc = kc.clone()
    kn = _bf16((5, Hkv, D), 51)
    vn = _bf16((5, Hkv, D), 52)
    k2, v2 = oracle.reshape_and_cache(kn, vn, kc, vc, np.array(gold["slots"], dtype=np.int64))
    q = _bf16((1, 1, D), 53)
    got = oracle.paged_decode(q, k2, v2, np.array([gold["block_table"]], np.int32),
                              np.array([5], np.int32))
    ref = _sdpa_unpaged(q[0].double(), kn.double().permute(1, 0, 2), vn.double().permute(1, 0, 2))
    np.testing.assert_allclose(got[0], ref.numpy(), rtol=0, atol=1e-12)


def test_reshape_and_cache_rejects_out_of_range_slot():
    kc = _bf16((2, 1, 4, 8), 61)
    with pytest.raises(ValueError):
        oracle.reshape_and_cache(_bf16((1, 1, 8), 62), _bf16((1, 1, 8), 63), kc, kc,
                                 np.array([8], dtype=np.int64))


def test_copy_blocks_matches_definition():
    NB, Hkv, BS, D = 8, 2, 4, 8
    kc = _bf16((NB, Hkv, BS, D), 71)
    vc = _bf16((NB, Hkv, BS, D), 72)
    pairs = np.array([[1, 5], [3, 6], [0, 7]], dtype=np.int32)
    k2, v2 = oracle.copy_blocks(kc, vc, pairs)
    kb, vb = oracle.bf16_bits(kc), oracle.bf16_bits(vc)
    for blk in range(NB):
        src = {5: 1, 6: 3, 7: 0}.get(blk, blk)
        assert np.array_equal(k2[blk], kb[src]) and np.array_equal(v2[blk], vb[src])


# ---------------------------------------------------------------- block manager model

def test_allocator_arithmetic(golden_dir):
    gold = json.load(open(os.path.join(golden_dir, "allocator_arithmetic.json")))
    BS = gold["block_size"]
    for case in gold["cases"]:
        n = case["tokens"]
        pool = PoolModel(400, BS)
        s = pool.seq_create()
        pool.append_tokens(s, n)
        assert len(pool.table(s)) == case["blocks"] == oracle.blocks_needed(n, BS)
        wasted = case["blocks"] * BS - n
        assert wasted <= gold["max_waste_slots"]["value"]
        if "wasted_slots" in case:
            assert wasted == case["wasted_slots"]
            assert abs(wasted / n - case["fragmentation_vs_length"]) < 1e-12
        if "utilisation_pct_rounded" in case:
            assert round(100 * n / (case["blocks"] * BS)) == case["utilisation_pct_rounded"]
    for n in range(1, 400):
        assert 0 <= oracle.blocks_needed(n, BS) * BS - n <= gold["max_waste_slots"]["value"]


def test_prefix_share_counts(golden_dir):
    gold = json.load(open(os.path.join(golden_dir, "allocator_arithmetic.json")))["prefix_share"]
    pool = PoolModel(200, 16)
    pre = pool.seq_create()
    pool.append_tokens(pre, gold["shared_blocks"] * 16)  # the resident preamble blocks
    used_before = pool.stats()["used"]
    req = pool.seq_fork(pre, gold["shared_blocks"] * 16)
    pool.append_tokens(req, gold["prompt_tokens"] - gold["shared_blocks"] * 16)
    assert len(pool.table(req)) == 75
    assert pool.stats()["used"] - used_before == gold["new_blocks"]
    assert pool.table(req)[:56] == pool.table(pre)
    assert all(pool.ref[b] == 2 for b in pool.table(pre))


def test_new_block_exactly_when_crossing_a_boundary():
    pool = PoolModel(100, 16)
    s = pool.seq_create()
    pool.append_tokens(s, 1200)
    assert len(pool.table(s)) == 75
    pool.append_slot(s)  # token index 1200, the 1,201st token
    assert len(pool.table(s)) == 76
    pool.append_tokens(s, 15)
    assert len(pool.table(s)) == 76
    pool.append_slot(s)
    assert len(pool.table(s)) == 77


def test_copy_on_write_state_machine():
    pool = PoolModel(10, 4, free_order=list(range(10)))
    a = pool.seq_create()
    pool.append_tokens(a, 6)  # blocks 0, 1 (block 1 partial: 2 of 4)
    b = pool.seq_fork(a, 6)
    assert pool.ref[0] == 2 and pool.ref[1] == 2
    slot, cow = pool.append_slot(b)  # writes into shared partial block 1 -> CoW
    assert cow == (1, 2)
    assert pool.table(b) == [0, 2] and pool.table(a) == [0, 1]
    assert pool.ref[1] == 1 and pool.ref[2] == 1 and pool.ref[0] == 2
    assert slot == 2 * 4 + 2
    slot_a, cow_a = pool.append_slot(a)  # a's block 1 is now private: no CoW
    assert cow_a is None and slot_a == 1 * 4 + 2
    pool.seq_free(b)
    assert pool.ref[0] == 1 and pool.ref[2] == 0
    assert pool.alloc() == 2  # freed block handed out next (LIFO free list)


def test_oom_leaves_state_unchanged():
    pool = PoolModel(2, 4)
    s = pool.seq_create()
    pool.append_tokens(s, 8)
    snap = (list(pool.free), list(pool.ref), pool.table(s), pool.length(s))
    with pytest.raises(oracle.PoolOOM):
        pool.append_slot(s)
    assert snap == (list(pool.free), list(pool.ref), pool.table(s), pool.length(s))
    t = pool.seq_fork(s, 7)
    snap = (list(pool.free), list(pool.ref), pool.table(t), pool.length(t))
    with pytest.raises(oracle.PoolOOM):
        pool.append_slot(t)  # CoW needs a block; none left
    assert snap == (list(pool.free), list(pool.ref), pool.table(t), pool.length(t))


def test_double_free_and_bad_ids():
    pool = PoolModel(4, 4)
    blk = pool.alloc()
    pool.decref(blk)
    with pytest.raises(oracle.PoolError):
        pool.decref(blk)
    with pytest.raises(oracle.PoolError):
        pool.incref(7)


# ---------------------------------------------------------------- 8-bit (E4M3) KV cache
# The pages only say that 8-bit KV quantisation halves the bytes per block
# ("PagedAttention" glossary page, §What paging costs); the format pinned here
# is the library's reading: OCP FP8 E4M3 with per-KV-head scales.

E4M3 = getattr(torch, "float8_e4m3fn", None)
needs_torch_fp8 = pytest.mark.skipif(E4M3 is None, reason="torch without float8_e4m3fn")


def test_e4m3_decode_landmarks():
    """Values the E4M3 definition fixes: zero, the smallest subnormal and normal,
    one, the largest finite value, exactly two NaN codes, sign symmetry, and a
    strictly increasing positive range."""
    t = oracle.e4m3_to_f64(np.arange(256))
    assert t[0x00] == 0.0 and np.signbit(t[0x80])
    assert t[0x01] == 2.0 ** -9 and t[0x07] == 7 * 2.0 ** -9
    assert t[0x08] == 2.0 ** -6 and t[0x38] == 1.0 and t[0x7E] == 448.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF]) and np.isnan(t).sum() == 2
    assert np.all(np.diff(t[:0x7F]) > 0)
    assert np.array_equal(t[0x80:0xFF], -t[0x00:0x7F])
    # eight evenly spaced values per binade above the subnormals
    for e in range(-6, 9):
        vals = t[(e + 7) * 8:(e + 7) * 8 + (8 if e < 8 else 7)]  # the last code is NaN
        assert np.allclose(np.diff(vals), 2.0 ** (e - 3)) and vals[0] == 2.0 ** e


@needs_torch_fp8
def test_e4m3_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    want = codes.view(E4M3).to(torch.float64).numpy()
    got = oracle.e4m3_to_f64(np.arange(256))
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all()


@needs_torch_fp8
def test_e4m3_encoder_matches_torch_in_range_and_saturates():
    """Round to nearest even, compared with torch's float32 -> float8_e4m3fn cast
    on random values, exact ties and subnormals (|x| < 448, where the two agree
    by definition); beyond 448 the encoder saturates (torch does not)."""
    rng = np.random.default_rng(11)
    grid = oracle.e4m3_to_f64(np.arange(0x7F))
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)  # exact ties (representable)
    x = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * 30,
        (rng.standard_normal(2000) * 2.0 ** -8).astype(np.float32),
        mids, -mids, np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(0)),
        grid[:0x7F].astype(np.float32),
    ])
    x = x[np.abs(x) < 448]
    want = torch.from_numpy(x).to(E4M3).view(torch.uint8).numpy()
    got = oracle.e4m3_from_f32(x)
    assert np.array_equal(got, want)
    sat = oracle.e4m3_from_f32(np.array([448.0, 463.9, 464.0, 1e6, np.inf, -500.0, -np.inf],
                                        dtype=np.float32))
    assert list(sat) == [0x7E] * 5 + [0xFE] * 2
    assert oracle.e4m3_from_f32(np.array([np.nan], dtype=np.float32))[0] == 0x7F


def _fp8_case(seed, B=3, Hq=8, Hkv=2, D=16, BS=4, lens=(1, 6, 11), scales=(0.5, 2.0)):
    q, kc, vc, tables, lens = _random_case(seed, B=B, Hq=Hq, Hkv=Hkv, D=D, BS=BS, lens=lens)
    ks = np.array([scales[0] * (h + 1) for h in range(Hkv)], dtype=np.float32)
    vs = np.array([scales[1] / (h + 1) for h in range(Hkv)], dtype=np.float32)
    # fill the whole pool through the quantising write, one slot per token
    NB = kc.shape[0]
    slots = np.arange(NB * BS, dtype=np.int64)
    kn = _bf16((NB * BS, Hkv, D), seed + 7)
    vn = _bf16((NB * BS, Hkv, D), seed + 8)
    k8, v8 = oracle.reshape_and_cache_fp8(kn, vn, np.zeros((NB, Hkv, BS, D), np.uint8),
                                          np.zeros((NB, Hkv, BS, D), np.uint8), slots, ks, vs)
    return q, k8, v8, ks, vs, tables, lens, kn, vn


@needs_torch_fp8
def test_fp8_write_quantises_per_head_and_transposes_v():
    """code = E4M3(float32(x) / scale[h]) (torch's cast, in range here); K rows
    at (block, head, offset), V stored as column `offset` of the (block, head)
    tile [d][offset]; negative slots write nothing."""
    q, k8, v8, ks, vs, tables, lens, kn, vn = _fp8_case(21)
    NB, Hkv, BS, D = k8.shape
    kx = torch.from_numpy(oracle.bf16_to_f64(kn).astype(np.float32)) / torch.from_numpy(ks)[:, None]
    vx = torch.from_numpy(oracle.bf16_to_f64(vn).astype(np.float32)) / torch.from_numpy(vs)[:, None]
    kcode = kx.to(E4M3).view(torch.uint8).numpy()  # [slot][h][d]
    vcode = vx.to(E4M3).view(torch.uint8).numpy()
    for slot in (0, 5, NB * BS - 1):
        blk, off = divmod(slot, BS)
        for h in range(Hkv):
            assert np.array_equal(k8[blk, h, off, :], kcode[slot, h])
            assert np.array_equal(v8.reshape(NB, Hkv, D, BS)[blk, h, :, off], vcode[slot, h])
    k2, v2 = oracle.reshape_and_cache_fp8(kn[:2], vn[:2], k8, v8, np.array([-1, -7]), ks, vs)
    assert np.array_equal(k2, k8) and np.array_equal(v2, v8)


def test_fp8_decode_equals_bf16_oracle_on_the_dequantised_cache():
    """With power-of-two scales every dequantised value (code value x scale) is
    exactly a bf16 value, so the 8-bit decode must equal the bf16 oracle run
    on a bf16 cache holding those values (V transposed back)."""
    q, k8, v8, ks, vs, tables, lens, _, _ = _fp8_case(22, scales=(0.25, 4.0))
    ks = np.array([0.25, 0.5], dtype=np.float32)
    vs = np.array([4.0, 2.0], dtype=np.float32)
    NB, Hkv, BS, D = k8.shape
    kd = oracle.e4m3_to_f64(k8) * ks[None, :, None, None]
    vd = (oracle.e4m3_to_f64(v8).reshape(NB, Hkv, D, BS) * vs[None, :, None, None]).transpose(0, 1, 3, 2)
    kb = torch.from_numpy(np.ascontiguousarray(kd)).to(torch.bfloat16)
    vb = torch.from_numpy(np.ascontiguousarray(vd)).to(torch.bfloat16)
    assert np.array_equal(oracle.bf16_to_f64(kb), kd) and np.array_equal(oracle.bf16_to_f64(vb), vd)
    want = oracle.paged_decode(q, kb, vb, tables, lens)
    got = oracle.paged_decode_fp8(q, k8, v8, ks, vs, tables, lens)
    assert np.abs(got - want).max() < 1e-12


def test_fp8_decode_scales_act_as_the_definition_says():
    """k_scale multiplies every score of its head (so doubling it equals
    doubling the softmax scale for those heads' queries) and v_scale scales
    the output linearly."""
    q, k8, v8, ks, vs, tables, lens, _, _ = _fp8_case(23)
    base = oracle.paged_decode_fp8(q, k8, v8, ks, vs, tables, lens)
    two_k = oracle.paged_decode_fp8(q, k8, v8, ks * 2, vs, tables, lens)
    D = q.shape[2]
    twice_scale = oracle.paged_decode_fp8(q, k8, v8, ks, vs, tables, lens, scale=2 / math.sqrt(D))
    assert np.abs(two_k - twice_scale).max() < 1e-12
    assert np.abs(two_k - base).max() > 1e-3
    three_v = oracle.paged_decode_fp8(q, k8, v8, ks, vs * 3, tables, lens)
    assert np.abs(three_v - 3 * base).max() < 1e-12


def test_fp8_copy_blocks_is_a_byte_copy():
    _, k8, v8, *_ = _fp8_case(24)
    k2, v2 = oracle.copy_blocks_fp8(k8, v8, [[1, 4], [2, 0]])
    assert np.array_equal(k2[4], k8[1]) and np.array_equal(v2[0], v8[2])
    assert np.array_equal(k2[3], k8[3])


# ---------------------------------------------------------------- several new tokens per sequence

def _multi_case(seed, lens, QL, Hq=4, Hkv=2, D=8, BS=4):
    q1, kc, vc, tables, lens = _random_case(seed, B=len(lens), Hq=Hq, Hkv=Hkv, D=D, BS=BS,
                                            lens=lens)
    q = _bf16((len(lens), QL, Hq, D), seed + 7)
    return q, kc, vc, tables, lens


def test_multi_query_equals_library_sdpa_with_explicit_causal_mask():
    """Identity tables, so the cache is contiguous: query i of a sequence of L
    tokens attends to keys 0 .. L - QL + i (the new tokens are the last QL),
    written as a boolean mask handed to torch SDPA in float64."""
    B, QL, Hq, Hkv, D, BS = 2, 5, 8, 2, 16, 4
    lens = np.array([13, 5], dtype=np.int32)
    mb = 4
    tables = np.arange(B * mb, dtype=np.int32).reshape(B, mb)
    q = _bf16((B, QL, Hq, D), 31)
    kc = _bf16((B * mb, Hkv, BS, D), 32)
    vc = _bf16((B * mb, Hkv, BS, D), 33)
    got = oracle.paged_decode_multi(q, kc, vc, tables, lens)
    G = Hq // Hkv
    for b in range(B):
        L = int(lens[b])
        K = kc[b * mb:(b + 1) * mb].double().permute(1, 0, 2, 3).reshape(Hkv, mb * BS, D)[:, :L]
        V = vc[b * mb:(b + 1) * mb].double().permute(1, 0, 2, 3).reshape(Hkv, mb * BS, D)[:, :L]
        allowed = torch.arange(L)[None, :] <= (L - QL + torch.arange(QL))[:, None]  # [QL, L]
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[b].double().permute(1, 0, 2),  # [Hq, QL, D]
            K.repeat_interleave(G, dim=0), V.repeat_interleave(G, dim=0), attn_mask=allowed)
        np.testing.assert_allclose(got[b], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("QL", [1, 2, 7])
def test_multi_query_rows_equal_single_token_decodes_at_their_lengths(QL):
    """Row i of a sequence of L tokens is the single-token decode of a sequence
    of L - QL + i + 1 tokens over the same table; with QL = 1 the two calls
    coincide."""
    lens = (7, 9, 16, 30)
    q, kc, vc, tables, lens = _multi_case(41 + QL, lens, QL)
    got = oracle.paged_decode_multi(q, kc, vc, tables, lens)
    for i in range(QL):
        want = oracle.paged_decode(q[:, i], kc, vc, tables, lens - QL + i + 1)
        np.testing.assert_array_equal(got[:, i], want)


def test_multi_query_brute_force_and_bad_lengths():
    q, kc, vc, tables, lens = _multi_case(50, (3, 6), QL=3, Hq=2, Hkv=1, D=4, BS=2)
    got = oracle.paged_decode_multi(q, kc, vc, tables, lens)
    qd, kd, vd = (oracle.bf16_to_f64(x) for x in (q, kc, vc))
    for b in range(2):
        L = int(lens[b])
        K = [list(kd[tables[b][t // 2], 0, t % 2]) for t in range(L)]
        V = [list(vd[tables[b][t // 2], 0, t % 2]) for t in range(L)]
        for i in range(3):
            n = L - 3 + i + 1
            ref = oracle.brute_force_decode([list(qd[b, i, h]) for h in range(2)], K[:n], V[:n],
                                            0.5)
            np.testing.assert_allclose(got[b, i], np.array(ref), rtol=0, atol=1e-12)
    with pytest.raises(ValueError):
        oracle.paged_decode_multi(q, kc, vc, tables, np.array([2, 6], dtype=np.int32))


def test_multi_query_fp8_equals_bf16_multi_on_the_dequantised_cache():
    """As for one token: with power-of-two scales the dequantised cache is
    exactly bf16, so the 8-bit multi-token decode equals the (pinned) bf16
    multi-token decode over it."""
    _, k8, v8, _, _, tables, lens, _, _ = _fp8_case(23, lens=(4, 6, 11), scales=(0.25, 4.0))
    ks = np.array([0.25, 0.5], dtype=np.float32)
    vs = np.array([4.0, 2.0], dtype=np.float32)
    NB, Hkv, BS, D = k8.shape
    kd = oracle.e4m3_to_f64(k8) * ks[None, :, None, None]
    vd = (oracle.e4m3_to_f64(v8).reshape(NB, Hkv, D, BS) * vs[None, :, None, None]).transpose(0, 1, 3, 2)
    kb = torch.from_numpy(np.ascontiguousarray(kd)).to(torch.bfloat16)
    vb = torch.from_numpy(np.ascontiguousarray(vd)).to(torch.bfloat16)
    q = _bf16((3, 4, 8, D), 24)
    want = oracle.paged_decode_multi(q, kb, vb, tables, lens)
    got = oracle.paged_decode_multi_fp8(q, k8, v8, ks, vs, tables, lens)
    assert np.abs(got - want).max() < 1e-12
    # one new token: the single-token 8-bit decode
    one = oracle.paged_decode_multi_fp8(q[:, :1], k8, v8, ks, vs, tables, lens)
    np.testing.assert_array_equal(one[:, 0], oracle.paged_decode_fp8(q[:, 0], k8, v8, ks, vs,
                                                                      tables, lens))


@needs_torch_fp8
def test_fp8_write_at_block_size_32_uses_16_key_subtiles():
    """Block size 32: V of slot offset `off` sits in sub-tile off // 16 of its
    (block, head) tile, row d, column off % 16 -- checked by plain numpy
    reshapes against torch's cast -- and the decode over that cache equals the
    bf16 oracle on the exactly dequantised cache (power-of-two scales)."""
    BS, Hkv, D, NB = 32, 2, 16, 4
    ks = np.array([0.25, 0.5], dtype=np.float32)
    vs = np.array([4.0, 2.0], dtype=np.float32)
    slots = np.arange(NB * BS, dtype=np.int64)
    kn = _bf16((NB * BS, Hkv, D), 61)
    vn = _bf16((NB * BS, Hkv, D), 62)
    k8, v8 = oracle.reshape_and_cache_fp8(kn, vn, np.zeros((NB, Hkv, BS, D), np.uint8),
                                          np.zeros((NB, Hkv, BS, D), np.uint8), slots, ks, vs)
    vx = torch.from_numpy(oracle.bf16_to_f64(vn).astype(np.float32)) / torch.from_numpy(vs)[:, None]
    vcode = vx.to(E4M3).view(torch.uint8).numpy()  # [slot][h][d]
    tiles = v8.reshape(NB, Hkv, BS // 16, D, 16)
    for slot in (0, 15, 16, 31, 77, NB * BS - 1):
        blk, off = divmod(slot, BS)
        for h in range(Hkv):
            assert np.array_equal(tiles[blk, h, off // 16, :, off % 16], vcode[slot, h])
    kd = oracle.e4m3_to_f64(k8) * ks[None, :, None, None]
    vd = np.ascontiguousarray((oracle.e4m3_to_f64(v8).reshape(NB, Hkv, BS // 16, D, 16)
                               * vs[None, :, None, None, None]).transpose(0, 1, 2, 4, 3)
                              .reshape(NB, Hkv, BS, D))
    kb = torch.from_numpy(np.ascontiguousarray(kd)).to(torch.bfloat16)
    vb = torch.from_numpy(vd).to(torch.bfloat16)
    tables = np.array([[2, 0], [3, 1]], dtype=np.int32)
    lens = np.array([40, 64], dtype=np.int32)
    q = _bf16((2, 4, D), 63)
    want = oracle.paged_decode(q, kb, vb, tables, lens)
    got = oracle.paged_decode_fp8(q, k8, v8, ks, vs, tables, lens)
    assert np.abs(got - want).max() < 1e-12
