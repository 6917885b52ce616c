"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Bit-exact: KV write through the slot mapping and the copy-on-write block
copy (whole caches compared). Decode attention: max-abs <= 2e-2 and
mean-abs <= 2e-3 (bf16 inputs, fp32 accumulation). Padding slots hold NaN
in every case, so a masked slot that leaks into a result fails the
finiteness check.
"""
import math

import numpy as np
import pytest

import oracle
import workloads
from tests import harness

pytestmark = pytest.mark.gpu

VARIANTS = pytest.mark.parametrize("variant", [0, 1], ids=["tensor_core", "cuda_core"])


@pytest.fixture(scope="module")
def pk():
    import torch

    from paged_kv_cache_92_gb300 import build

    build.build()
    import paged_kv_cache_92_gb300 as pk

    pk.load()
    assert torch.cuda.is_available()
    return pk


def _check_errors(pk):
    assert pk.pa_device_errors() == 0


# ---------------------------------------------------------------- the five workloads

@VARIANTS
def test_tiny_workload_full(pk, variant):
    """4 sequences {1,5,17,33}, 4/1 heads, d=64: decode, append, decode again."""
    import torch

    r = workloads.tiny()
    case = harness.build_case(r)
    # decode before the append, over the pre-step lengths
    kc, vc = case.k_cache, case.v_cache
    out0 = pk.pa_decode(case.q, kc, vc, torch.from_numpy(case.tables0).cuda(),
                        torch.from_numpy(case.lens0).cuda(), max_context_len=33, variant=variant)
    ref0 = oracle.paged_decode(case.q.cpu(), kc.cpu(), vc.cpu(), case.tables0, case.lens0)
    harness.assert_close(harness.bf16_tensor_to_f64(out0), ref0)
    # the step: append one token per sequence (no boundary crossed), decode over {2,6,18,34}
    assert case.cows.shape[0] == 0
    assert list(case.lens) == [2, 6, 18, 34]
    out, kg, vg = harness.run_step_gpu(case, variant=variant)
    ref, ko, vo = harness.run_step_oracle(case)
    assert np.array_equal(oracle.bf16_bits(kg.cpu()), ko)
    assert np.array_equal(oracle.bf16_bits(vg.cpu()), vo)
    harness.assert_close(harness.bf16_tensor_to_f64(out), ref)
    _check_errors(pk)


@VARIANTS
def test_llama8b_layer_full(pk, variant):
    case = harness.build_case(workloads.llama8b_layer())
    out, kg, vg = harness.run_step_gpu(case, variant=variant)
    ref, ko, vo = harness.run_step_oracle(case)
    assert np.array_equal(oracle.bf16_bits(kg.cpu()), ko)
    assert np.array_equal(oracle.bf16_bits(vg.cpu()), vo)
    harness.assert_close(harness.bf16_tensor_to_f64(out), ref)
    _check_errors(pk)


@VARIANTS
def test_llama8b_high_concurrency_full(pk, variant):
    r = workloads.llama8b_high_concurrency()
    case = harness.build_case(r)
    # new blocks were allocated exactly for the sequences sitting on a boundary
    grew = (case.tables >= 0).sum(1) - (case.tables0 >= 0).sum(1)
    assert np.array_equal(grew, (r.lens0 % 16 == 0).astype(int))
    out, kg, vg = harness.run_step_gpu(case, variant=variant)
    ref, ko, vo = harness.run_step_oracle(case)
    assert np.array_equal(oracle.bf16_bits(kg.cpu()), ko)
    assert np.array_equal(oracle.bf16_bits(vg.cpu()), vo)
    harness.assert_close(harness.bf16_tensor_to_f64(out), ref)
    _check_errors(pk)


@VARIANTS
@pytest.mark.parametrize("batch", [8, 32])
def test_llama70b_long_context(pk, batch, variant):
    """64/8 heads, L ~ U[8192, 32768]: split-K over 512-token partitions + merge."""
    r = workloads.llama70b_long(batch=batch)
    case = harness.build_case(r)
    out, kg, vg = harness.run_step_gpu(case, variant=variant)
    # every (sequence, query head) row: 512 / 2048 rows of 8k-32k tokens
    ref, ko, vo = harness.run_step_oracle(case)
    assert np.array_equal(oracle.bf16_bits(kg.cpu()), ko)
    assert np.array_equal(oracle.bf16_bits(vg.cpu()), vo)
    harness.assert_close(harness.bf16_tensor_to_f64(out), ref)
    _check_errors(pk)


@VARIANTS
def test_shared_prefix_copy_on_write(pk, variant):
    r = workloads.shared_prefix()
    case = harness.build_case(r)
    assert case.cows.shape == (32, 2)
    assert len(set(case.cows[:, 0].tolist())) == 1  # all copies come from the last shared block
    out, kg, vg = harness.run_step_gpu(case, variant=variant)
    ref, ko, vo = harness.run_step_oracle(case)
    assert np.array_equal(oracle.bf16_bits(kg.cpu()), ko)
    assert np.array_equal(oracle.bf16_bits(vg.cpu()), vo)
    harness.assert_close(harness.bf16_tensor_to_f64(out), ref)
    _check_errors(pk)


# ---------------------------------------------------------------- edge cases

def _direct_case(lens, Hq, Hkv, D, seed, extra_blocks=3, reverse=False, identity=False):
    import torch

    lens = np.asarray(lens, dtype=np.int64)
    need = int(((lens + 15) // 16).sum())
    NB = need + extra_blocks
    rng = np.random.default_rng(seed)
    if identity:
        order = np.arange(NB, dtype=np.int32)
    elif reverse:
        order = np.arange(NB, dtype=np.int32)[::-1].copy()
    else:
        order = rng.permutation(NB).astype(np.int32)
    tables = workloads.sequential_tables(lens, order, 16)
    q = workloads.bf16_normal((len(lens), Hq, D), seed + 1, "cuda")
    kc = workloads.bf16_normal((NB, Hkv, 16, D), seed + 2, "cuda")
    vc = workloads.bf16_normal((NB, Hkv, 16, D), seed + 3, "cuda")
    workloads.fill_padding_nan(kc, tables, lens, 16)
    workloads.fill_padding_nan(vc, tables, lens, 16)
    return q, kc, vc, tables, lens.astype(np.int32), torch


@VARIANTS
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("partition", [0, 16, 80, 4096])
def test_edge_lengths(pk, D, G, partition, variant):
    lens = [1, 15, 16, 17, 511, 512, 513, 1024, 1025, 4097]
    Hkv = 2
    q, kc, vc, tables, lens, torch = _direct_case(lens, G * Hkv, Hkv, D, seed=D * 10 + G)
    out = pk.pa_decode(q, kc, vc, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                       max_context_len=int(lens.max()), partition_tokens=partition,
                       variant=variant)
    torch.cuda.synchronize()
    ref = oracle.paged_decode(q.cpu(), kc.cpu(), vc.cpu(), tables, lens)
    harness.assert_close(harness.bf16_tensor_to_f64(out), ref)
    _check_errors(pk)


@VARIANTS
@pytest.mark.parametrize("partition", [0, 16])
def test_length_one_returns_v0_bit_exact(pk, partition, variant):
    q, kc, vc, tables, lens, torch = _direct_case([1] * 6, 8, 2, 128, seed=5)
    out = pk.pa_decode(q, kc, vc, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                       max_context_len=1, partition_tokens=partition, variant=variant)
    torch.cuda.synchronize()
    vh = vc.cpu()
    for b in range(6):
        for h in range(8):
            assert torch.equal(out[b, h].cpu(), vh[tables[b, 0], h // 4, 0])


@VARIANTS
def test_physical_placement_does_not_change_a_bit(pk, variant):
    lens = [37, 300, 1, 900, 16, 513]
    outs = []
    for kind in ("random", "reverse", "identity"):
        q, kc, vc, tables, lens_a, torch = _direct_case(
            lens, 32, 8, 128, seed=77, extra_blocks=0,
            reverse=(kind == "reverse"), identity=(kind == "identity"))
        # same logical contents under every placement: rebuild the caches from logical order
        base_q, base_kc, base_vc, base_tables, _, _ = _direct_case(lens, 32, 8, 128, seed=77,
                                                                    extra_blocks=0)
        kc2 = torch.empty_like(base_kc)
        vc2 = torch.empty_like(base_vc)
        kc2[torch.from_numpy(tables[tables >= 0]).long().cuda()] = \
            base_kc[torch.from_numpy(base_tables[base_tables >= 0]).long().cuda()]
        vc2[torch.from_numpy(tables[tables >= 0]).long().cuda()] = \
            base_vc[torch.from_numpy(base_tables[base_tables >= 0]).long().cuda()]
        out = pk.pa_decode(base_q, kc2, vc2, torch.from_numpy(tables).cuda(),
                           torch.from_numpy(lens_a).cuda(), max_context_len=900, variant=variant)
        outs.append(out.cpu())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


@VARIANTS
def test_split_and_unsplit_agree(pk, variant):
    q, kc, vc, tables, lens, torch = _direct_case([700, 2049, 3000], 32, 8, 128, seed=9)
    bt, cl = torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda()
    a = pk.pa_decode(q, kc, vc, bt, cl, max_context_len=3000, partition_tokens=4096,
                     variant=variant)
    b = pk.pa_decode(q, kc, vc, bt, cl, max_context_len=3000, partition_tokens=128,
                     variant=variant)
    torch.cuda.synchronize()
    ref = oracle.paged_decode(q.cpu(), kc.cpu(), vc.cpu(), tables, lens)
    harness.assert_close(harness.bf16_tensor_to_f64(a), ref)
    harness.assert_close(harness.bf16_tensor_to_f64(b), ref)


@VARIANTS
def test_zero_length_rows_are_zero(pk, variant):
    q, kc, vc, tables, lens, torch = _direct_case([5, 20, 3], 8, 2, 128, seed=11)
    lens2 = lens.copy()
    lens2[1] = 0
    out = torch.full_like(q, 7.0)
    pk.pa_decode(q, kc, vc, torch.from_numpy(tables).cuda(), torch.from_numpy(lens2).cuda(),
                 max_context_len=20, out=out, variant=variant)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out[1]).item() == 0
    ref = oracle.paged_decode(q.cpu(), kc.cpu(), vc.cpu(), tables, lens)
    got = harness.bf16_tensor_to_f64(out)
    harness.assert_close(got[[0, 2]], ref[[0, 2]])


def test_empty_batch_and_empty_writes(pk):
    import torch

    q = torch.empty((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((4, 2, 16, 128), dtype=torch.bfloat16, device="cuda")
    out = pk.pa_decode(q, kc, kc, torch.empty((0, 1), dtype=torch.int32, device="cuda"),
                       torch.empty((0,), dtype=torch.int32, device="cuda"), max_context_len=1)
    assert out.shape == (0, 8, 128)
    pk.pa_reshape_and_cache(torch.empty((0, 2, 128), dtype=torch.bfloat16, device="cuda"),
                            torch.empty((0, 2, 128), dtype=torch.bfloat16, device="cuda"), kc, kc,
                            torch.empty((0,), dtype=torch.int64, device="cuda"))
    pk.pa_copy_blocks(kc, kc, torch.empty((0, 2), dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    _check_errors(pk)


def test_reshape_and_cache_skips_negative_slots_bit_exact(pk):
    import torch

    NB, Hkv, D = 12, 8, 128
    kc = workloads.bf16_normal((NB, Hkv, 16, D), 1, "cuda")
    vc = workloads.bf16_normal((NB, Hkv, 16, D), 2, "cuda")
    kn = workloads.bf16_normal((7, Hkv, D), 3, "cuda")
    vn = workloads.bf16_normal((7, Hkv, D), 4, "cuda")
    slots = np.array([0, -1, 191, 17, -5, 100, 16], dtype=np.int64)
    k2, v2 = kc.clone(), vc.clone()
    pk.pa_reshape_and_cache(kn, vn, k2, v2, torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    ko, vo = oracle.reshape_and_cache(kn.cpu(), vn.cpu(), kc.cpu(), vc.cpu(), slots)
    assert np.array_equal(oracle.bf16_bits(k2.cpu()), ko)
    assert np.array_equal(oracle.bf16_bits(v2.cpu()), vo)


def test_copy_blocks_bit_exact_and_untouched_blocks(pk):
    import torch

    NB, Hkv, D = 20, 8, 128
    kc = workloads.bf16_normal((NB, Hkv, 16, D), 5, "cuda")
    vc = workloads.bf16_normal((NB, Hkv, 16, D), 6, "cuda")
    pairs = np.array([[3, 11], [3, 12], [0, 19], [7, 2]], dtype=np.int32)
    k2, v2 = kc.clone(), vc.clone()
    pk.pa_copy_blocks(k2, v2, torch.from_numpy(pairs).cuda())
    torch.cuda.synchronize()
    ko, vo = oracle.copy_blocks(kc.cpu(), vc.cpu(), pairs)
    assert np.array_equal(oracle.bf16_bits(k2.cpu()), ko)
    assert np.array_equal(oracle.bf16_bits(v2.cpu()), vo)


# ---------------------------------------------------------------- device-side range checks

@VARIANTS
def test_bad_device_values_set_error_bits_without_faulting(pk, variant):
    import torch

    q, kc, vc, tables, lens, _ = _direct_case([40, 7], 8, 2, 128, seed=13)
    assert pk.pa_device_errors() == 0
    bad = tables.copy()
    bad[0, 1] = kc.shape[0] + 1000  # past the pool
    pk.pa_decode(q, kc, vc, torch.from_numpy(bad).cuda(), torch.from_numpy(lens).cuda(),
                 max_context_len=40, variant=variant)
    assert pk.pa_device_errors() & pk.DEVERR_TABLE_ENTRY
    long = lens.copy()
    long[1] = 41  # above the host-promised maximum
    pk.pa_decode(q, kc, vc, torch.from_numpy(tables).cuda(), torch.from_numpy(long).cuda(),
                 max_context_len=40, variant=variant)
    assert pk.pa_device_errors() & pk.DEVERR_CONTEXT_LEN
    kn = workloads.bf16_normal((1, 2, 128), 1, "cuda")
    pk.pa_reshape_and_cache(kn, kn, kc.clone(), vc.clone(),
                            torch.tensor([kc.shape[0] * 16], dtype=torch.int64, device="cuda"))
    assert pk.pa_device_errors() & pk.DEVERR_SLOT
    pk.pa_copy_blocks(kc.clone(), vc.clone(),
                      torch.tensor([[0, kc.shape[0]]], dtype=torch.int32, device="cuda"))
    assert pk.pa_device_errors() & pk.DEVERR_COPY_PAIR
    # the context is still healthy
    out = pk.pa_decode(q, kc, vc, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                       max_context_len=40, variant=variant)
    torch.cuda.synchronize()
    ref = oracle.paged_decode(q.cpu(), kc.cpu(), vc.cpu(), tables, lens)
    harness.assert_close(harness.bf16_tensor_to_f64(out), ref)
    assert pk.pa_device_errors() == 0


@pytest.mark.parametrize("query_len", [1, 3, 8])
def test_wait_budget_exit_reports_timeout_and_leaves_the_context_usable(pk, query_len):
    """The tensor-core kernels' bounded waits, made to run out: with a budget
    of 1 us per barrier wait (far below a chunk's turnaround) a well-formed
    launch gives up in every CTA that holds more chunks than its ring. The
    launch must end, report PA_DEVERR_TIMEOUT, and leave the context usable:
    the next launch with the default budget, on the same buffers, matches the
    oracle (every copy in flight had landed and the tensor memory was freed).
    One new token and three (12 query rows per KV head) run on the decode
    kernel, eight on the query-major kernel."""
    import torch

    rng = np.random.default_rng(31)
    lens = rng.integers(128, 2048, size=64)
    q, kc, vc, tables, lens, _ = _direct_case(lens, 32, 8, 128, seed=29)
    if query_len > 1:
        q = workloads.bf16_normal((len(lens), query_len, 32, 128), 33, "cuda")
    bt, cl = torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda()
    mx = int(lens.max())
    assert pk.pa_device_errors() == 0
    ws = torch.empty(1 << 26, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    for _ in range(2):
        pk.pa_decode(q, kc, vc, bt, cl, max_context_len=mx, out=out, workspace=ws,
                     wait_timeout_us=1)
        assert pk.pa_device_errors() & pk.DEVERR_TIMEOUT
    out = pk.pa_decode(q, kc, vc, bt, cl, max_context_len=mx, out=out, workspace=ws)
    torch.cuda.synchronize()
    if query_len == 1:
        ref = oracle.paged_decode(q.cpu(), kc.cpu(), vc.cpu(), tables, lens)
    else:
        ref = oracle.paged_decode_multi(q.cpu(), kc.cpu(), vc.cpu(), tables, lens)
    harness.assert_close(harness.bf16_tensor_to_f64(out), ref)
    assert pk.pa_device_errors() == 0


@VARIANTS
def test_scale_is_applied(pk, variant):
    q, kc, vc, tables, lens, torch = _direct_case([33, 70], 8, 2, 64, seed=17)
    out = pk.pa_decode(q, kc, vc, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                       max_context_len=70, scale=0.3, variant=variant)
    torch.cuda.synchronize()
    ref = oracle.paged_decode(q.cpu(), kc.cpu(), vc.cpu(), tables, lens, scale=0.3)
    harness.assert_close(harness.bf16_tensor_to_f64(out), ref)
    assert not math.isclose(0.3, 1 / 8)


def test_batch_beyond_the_tensor_core_plan_runs_and_matches(pk):
    """More sequences than the tensor-core kernel plans in shared memory: the
    call still succeeds (CUDA-core kernel) and matches the oracle."""
    import torch

    rng = np.random.default_rng(21)
    lens = rng.integers(1, 40, size=2100)
    q, kc, vc, tables, lens, _ = _direct_case(lens, 8, 2, 64, seed=23)
    out = pk.pa_decode(q, kc, vc, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                       max_context_len=int(lens.max()), partition_tokens=16, variant=0)
    torch.cuda.synchronize()
    units = harness.sample_units(len(lens), 8, 300, seed=5)
    ref = oracle.paged_decode(q.cpu(), kc.cpu(), vc.cpu(), tables, lens, units=units)
    got = harness.bf16_tensor_to_f64(out)
    harness.assert_close(np.stack([got[b, h] for b, h in units]), ref)
    _check_errors(pk)


# ---------------------------------------------------------------- overlapped set-up

def test_overlapped_prologue_is_bit_identical_to_stream_order(pk):
    """overlap_prologue lets the decode plan its work while the KV write is
    still running (programmatic dependent launch). It must read the cache only
    after the write: the new token of every sequence is in the result, and the
    output equals the plain stream-ordered launch bit for bit, step after step."""
    import torch

    case = harness.build_case(workloads.llama8b_layer(), "cuda")
    want, _, _ = harness.run_step_gpu(case)
    for _ in range(3):
        got, _, _ = harness.run_step_gpu(case, overlap_prologue=True)
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    units = harness.sample_units(case.q.shape[0], case.q.shape[1], 64, seed=3)
    ref, _, _ = harness.run_step_oracle(case, units=units)
    g = harness.bf16_tensor_to_f64(want)
    harness.assert_close(np.stack([g[b, h] for b, h in units]), ref)
    _check_errors(pk)


def test_overlapped_decodes_back_to_back_keep_their_partials(pk):
    """Two overlapped decodes in a row on one workspace (two layers of a
    step): the second must not write its plan or partials before the first
    one's merge has read them."""
    import torch

    case = harness.build_case(workloads.llama8b_layer(), "cuda")
    tables = torch.from_numpy(case.tables).cuda()
    lens = torch.from_numpy(case.lens).cuda()
    q2 = workloads.bf16_normal(tuple(case.q.shape), 99, "cuda")
    mx = int(case.lens.max())
    p = pk.make_decode_params(case.q, torch.empty_like(case.q), case.k_cache, case.v_cache,
                              tables, lens, max_context_len=mx, overlap_prologue=True)
    ws = torch.empty(pk.pa_decode_workspace_size(p), dtype=torch.uint8, device="cuda")
    plain = [pk.pa_decode(q, case.k_cache, case.v_cache, tables, lens, max_context_len=mx,
                          workspace=ws) for q in (case.q, q2)]
    for _ in range(3):
        got = [pk.pa_decode(q, case.k_cache, case.v_cache, tables, lens, max_context_len=mx,
                            workspace=ws, overlap_prologue=True) for q in (case.q, q2)]
        torch.cuda.synchronize()
        for a, b in zip(got, plain):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    _check_errors(pk)


# ---------------------------------------------------------------- fused KV append

FUSED_CASES = {
    "tiny": workloads.tiny,
    "llama8b_layer": workloads.llama8b_layer,
    "llama8b_high_concurrency": workloads.llama8b_high_concurrency,
    "llama70b_long_b8": lambda: workloads.llama70b_long(batch=8),
    "shared_prefix": workloads.shared_prefix,
}


@VARIANTS
@pytest.mark.parametrize("name", list(FUSED_CASES))
def test_fused_append_decode_matches_oracle_and_separate_launches(pk, name, variant):
    """pa_append_decode (KV write inside the decode) against the oracle's KV
    write + decode, and bit for bit against pa_reshape_and_cache + pa_decode."""
    import torch

    case = harness.build_case(FUSED_CASES[name]())
    got, kg, vg = harness.run_step_gpu(case, variant=variant, fused_append=True,
                                       overlap_prologue=True)
    ko, vo = harness.oracle_caches(case)
    assert np.array_equal(oracle.bf16_bits(kg.cpu()), ko)
    assert np.array_equal(oracle.bf16_bits(vg.cpu()), vo)
    B, Hq = case.q.shape[0], case.q.shape[1]
    units = harness.sample_units(B, Hq, min(B * Hq, 96), seed=7,
                                 must=[(int(np.argmax(case.lens)), Hq - 1)])
    ref = oracle.paged_decode(case.q.cpu(), ko, vo, case.tables, case.lens, units=units)
    g = harness.bf16_tensor_to_f64(got)
    harness.assert_close(np.stack([g[b, h] for b, h in units]), ref)
    want, _, _ = harness.run_step_gpu(case, variant=variant)
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    _check_errors(pk)


@VARIANTS
def test_fused_append_slot_rules(pk, variant):
    """Sequence 0 appends at its last token's slot (written); sequence 1 has a
    negative slot (nothing written); sequence 2 names a slot that is not its
    last token's (error bit, nothing written); sequence 3 is empty (nothing
    written, zero output)."""
    import torch

    lens = np.array([41, 8, 17, 0])
    q, kc, vc, tables, lens, _ = _direct_case(lens, 8, 2, 128, seed=31)
    last = [(int(tables[b, (lens[b] - 1) // 16]) * 16 + (lens[b] - 1) % 16) if lens[b] else -1
            for b in range(4)]
    spare = (kc.shape[0] - 1) * 16  # a slot of an unused block
    slots = np.array([last[0], -1, last[2] + 1, spare], dtype=np.int64)
    kn = workloads.bf16_normal((4, 2, 128), 41, "cuda")
    vn = workloads.bf16_normal((4, 2, 128), 42, "cuda")
    k2, v2 = kc.clone(), vc.clone()
    out = pk.pa_append_decode(q, k2, v2, torch.from_numpy(tables).cuda(),
                              torch.from_numpy(lens).cuda(), int(lens.max()), kn, vn,
                              torch.from_numpy(slots).cuda(), variant=variant)
    torch.cuda.synchronize()
    assert pk.pa_device_errors() == pk.DEVERR_APPEND_SLOT
    only0 = np.array([last[0], -1, -1, -1], dtype=np.int64)
    ko, vo = oracle.reshape_and_cache(kn.cpu(), vn.cpu(), oracle.bf16_bits(kc.cpu()),
                                      oracle.bf16_bits(vc.cpu()), only0)
    assert np.array_equal(oracle.bf16_bits(k2.cpu()), ko)
    assert np.array_equal(oracle.bf16_bits(v2.cpu()), vo)
    units = [(b, h) for b in range(3) for h in range(8)]  # the oracle has no empty sequence
    ref = oracle.paged_decode(q.cpu(), ko, vo, tables, lens, units=units)
    got = harness.bf16_tensor_to_f64(out)
    harness.assert_close(got[:3].reshape(24, -1), ref)
    assert not got[3].any()


# ---------------------------------------------------------------- host-driven step

@VARIANTS
@pytest.mark.parametrize("name", ["tiny", "llama8b_layer", "shared_prefix"])
def test_step_host_matches_device_step(pk, name, variant):
    """pa_step_host (packed host inputs in, host output back, one call) gives
    the device-side step's output and caches bit for bit; the caches also
    match the oracle's copy-on-write + KV write."""
    import torch

    case = harness.build_case(FUSED_CASES[name]())
    want, kw, vw = harness.run_step_gpu(case, variant=variant, fused_append=True)
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    B, Hq, D = case.q.shape
    p = pk.make_step_host_params(kc, vc, B, Hq, case.tables.shape[1], int(case.lens.max()),
                                 num_cow_pairs=len(case.cows), variant=variant)
    host_in = pk.pack_step_inputs(p, case.q.cpu(), case.k_new.cpu(), case.v_new.cpu(), case.slots,
                                  case.tables, case.lens, case.cows if len(case.cows) else None)
    host_out = torch.empty((B, Hq, D), dtype=torch.bfloat16).pin_memory()
    ws = torch.empty(pk.pa_step_host_workspace_size(p), dtype=torch.uint8, device="cuda")
    pk.pa_step_host(p, host_in, host_out, ws)
    assert torch.equal(host_out.view(torch.int16), want.cpu().view(torch.int16))
    assert torch.equal(kc.view(torch.int16), kw.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), vw.view(torch.int16))
    ko, vo = harness.oracle_caches(case)
    assert np.array_equal(oracle.bf16_bits(kc.cpu()), ko)
    assert np.array_equal(oracle.bf16_bits(vc.cpu()), vo)
    _check_errors(pk)


@pytest.mark.parametrize("pinned_in,pinned_out", [(False, False), (True, False), (False, True)])
def test_step_host_pageable_buffers(pk, pinned_in, pinned_out):
    """Pinned buffers are read and written by the kernels themselves; pageable
    ones take the DMA copies. Every mix gives the device-side step's output
    and caches bit for bit."""
    import torch

    case = harness.build_case(FUSED_CASES["shared_prefix"]())
    want, kw, vw = harness.run_step_gpu(case, variant=0, fused_append=True)
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    B, Hq, D = case.q.shape
    p = pk.make_step_host_params(kc, vc, B, Hq, case.tables.shape[1], int(case.lens.max()),
                                 num_cow_pairs=len(case.cows))
    host_in = pk.pack_step_inputs(p, case.q.cpu(), case.k_new.cpu(), case.v_new.cpu(), case.slots,
                                  case.tables, case.lens, case.cows if len(case.cows) else None,
                                  pin=pinned_in)
    host_out = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16)
    if pinned_out:
        host_out = host_out.pin_memory()
    assert host_in.is_pinned() == pinned_in and host_out.is_pinned() == pinned_out
    ws = torch.empty(pk.pa_step_host_workspace_size(p), dtype=torch.uint8, device="cuda")
    for _ in range(2):  # the second call reuses the workspace
        pk.pa_step_host(p, host_in, host_out, ws)
        assert torch.equal(host_out.view(torch.int16), want.cpu().view(torch.int16))
        kc.copy_(case.k_cache)
        vc.copy_(case.v_cache)
    pk.pa_step_host(p, host_in, host_out, ws)
    assert torch.equal(kc.view(torch.int16), kw.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), vw.view(torch.int16))
    _check_errors(pk)
