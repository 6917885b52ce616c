"""pa_decode_noalloc: the decode for callers that cannot allocate device memory.

Such callers are, for example, engines that gave all free HBM to their KV
block pool at start-up (nothing is left for a workspace) or serving loops that
cannot take cudaMalloc's implicit synchronisation. The entry point keeps its
split-K partials in a fixed array inside the library. These tests call it
through the C ABI and check it against pa_decode, which uses a caller-provided
workspace, on two calls in a row: the second call finds the first call's
partials still in the shared array and must not be affected by them.
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads
from tests import harness

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_92_gb300 import build

    build.build()
    import paged_kv_cache_92_gb300 as pk

    pk.load()
    return pk


def _inputs(seed, lens, Hq=32, Hkv=8, D=128):
    import torch

    lens = np.asarray(lens, dtype=np.int64)
    need = int(((lens + 15) // 16).sum())
    order = np.random.default_rng(seed).permutation(need + 5).astype(np.int32)
    tables = workloads.sequential_tables(lens, order, 16)
    q = workloads.bf16_normal((len(lens), Hq, D), seed + 1, "cuda")
    kc = workloads.bf16_normal((need + 5, Hkv, 16, D), seed + 2, "cuda")
    vc = workloads.bf16_normal((need + 5, Hkv, 16, D), seed + 3, "cuda")
    workloads.fill_padding_nan(kc, tables, lens, 16)
    workloads.fill_padding_nan(vc, tables, lens, 16)
    return (q, kc, vc, torch.from_numpy(tables).cuda(),
            torch.from_numpy(lens.astype(np.int32)).cuda(), int(lens.max()), tables, lens)


def test_noalloc_matches_workspace_decode_on_two_calls_in_a_row(pk):
    import torch

    # two different batches, both long enough to split into 512-token partitions
    cases = [_inputs(3, [1900, 37, 2049, 700, 1, 1536]),
             _inputs(4, [513, 1200, 16, 2000])]
    for q, kc, vc, bt, cl, mx, tables, lens in cases:
        ref_out = pk.pa_decode(q, kc, vc, bt, cl, max_context_len=mx)
        p = pk.make_decode_params(q, torch.empty_like(q), kc, vc, bt, cl, max_context_len=mx)
        assert pk.pa_decode_workspace_size(p) > 256  # split-K partials beyond the counter header
        out = torch.empty_like(q)
        p = pk.make_decode_params(q, out, kc, vc, bt, cl, max_context_len=mx)
        stream = torch.cuda.current_stream().cuda_stream or None
        status = pk.load().pa_decode_noalloc(ctypes.byref(p), stream)  # the C ABI call itself
        assert status == 0, pk.load().pa_last_error()
        torch.cuda.synchronize()
        harness.assert_close(harness.bf16_tensor_to_f64(out), harness.bf16_tensor_to_f64(ref_out))
        want = oracle.paged_decode(q.cpu(), kc.cpu(), vc.cpu(), tables, lens.astype(np.int32))
        harness.assert_close(harness.bf16_tensor_to_f64(out), want)
    assert pk.pa_device_errors() == 0


def _noalloc_call(pk, q, kc, vc, bt, cl, mx, variant=0):
    """pa_decode_noalloc through the C ABI; returns the output tensor."""
    import torch

    out = torch.empty_like(q)
    p = pk.make_decode_params(q, out, kc, vc, bt, cl, max_context_len=mx, variant=variant)
    stream = torch.cuda.current_stream().cuda_stream or None
    status = pk.load().pa_decode_noalloc(ctypes.byref(p), stream)
    assert status == 0, pk.load().pa_last_error()
    torch.cuda.synchronize()
    return out


def test_noalloc_cuda_core_variant_on_two_calls_in_a_row(pk):
    """The CUDA-core kernel keeps its per-partition partials in the same
    array when a sequence spans several 512-token partitions."""
    cases = [_inputs(5, [1900, 37, 2049, 700, 1, 1536]),
             _inputs(6, [513, 1200, 16, 2000, 1100])]
    for q, kc, vc, bt, cl, mx, tables, lens in cases:
        assert mx > 512  # several partitions
        ref_out = pk.pa_decode(q, kc, vc, bt, cl, max_context_len=mx, variant=1)
        out = _noalloc_call(pk, q, kc, vc, bt, cl, mx, variant=1)
        harness.assert_close(harness.bf16_tensor_to_f64(out), harness.bf16_tensor_to_f64(ref_out))
        want = oracle.paged_decode(q.cpu(), kc.cpu(), vc.cpu(), tables, lens.astype(np.int32))
        harness.assert_close(harness.bf16_tensor_to_f64(out), want)
    assert pk.pa_device_errors() == 0


@pytest.mark.parametrize("recipe", ["llama70b_long_b8", "shared_prefix_cow_b512"])
def test_noalloc_full_workloads_against_the_oracle(pk, recipe):
    """Whole steps of the 70B-class batch of 8 (long contexts, split over
    CTAs) and of the shared-prefix batch with its copy-on-write appends: the
    block copies and the KV write, then the decode through pa_decode_noalloc,
    whose tensor-core partials fit the fixed array."""
    import torch

    r = (workloads.llama70b_long(batch=8) if recipe == "llama70b_long_b8"
         else workloads.shared_prefix())
    case = harness.build_case(r)
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    if len(case.cows):
        pk.pa_copy_blocks(kc, vc, torch.from_numpy(case.cows).cuda())
    pk.pa_reshape_and_cache(case.k_new, case.v_new, kc, vc, torch.from_numpy(case.slots).cuda())
    bt = torch.from_numpy(case.tables).cuda()
    cl = torch.from_numpy(case.lens).cuda()
    mx = int(case.lens.max())
    p = pk.make_decode_params(case.q, torch.empty_like(case.q), kc, vc, bt, cl, max_context_len=mx)
    assert pk.pa_decode_workspace_size(p) <= 16 << 20
    ref, _, _ = harness.run_step_oracle(case)
    for _ in range(2):
        out = _noalloc_call(pk, case.q, kc, vc, bt, cl, mx)
        harness.assert_close(harness.bf16_tensor_to_f64(out), ref)
    assert pk.pa_device_errors() == 0


def test_noalloc_rejects_shapes_beyond_its_fixed_scratch(pk):
    import torch

    # 1024 seqs x 64 q heads x 64 partitions x (128 + 2) x 4 B is far above 16 MiB
    p = pk.DecodeParams()
    q = torch.empty((1024, 64, 128), dtype=torch.bfloat16, device="cuda")
    p.q = p.out = p.k_cache = p.v_cache = q.data_ptr()
    bt = torch.zeros((1024, 2048), dtype=torch.int32, device="cuda")
    p.block_tables = p.context_lens = bt.data_ptr()
    p.max_blocks_per_seq, p.num_seqs, p.num_q_heads, p.num_kv_heads = 2048, 1024, 64, 8
    p.head_dim, p.block_size, p.num_blocks, p.max_context_len = 128, 16, 8, 32768
    p.scale, p.partition_tokens = 0.088, 512
    assert pk.load().pa_decode_noalloc(ctypes.byref(p), None) == 1  # PA_ERR_INVALID_ARG
    assert b"PA_NOALLOC_SCRATCH_BYTES" in pk.load().pa_last_error()
