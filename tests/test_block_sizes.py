"""GPU parity at block sizes 8 and 32 ("Paged Attention as a Memory Manager",
§PagedAttention: the block size is a compile-time constant, typically 8, 16
or 32).

The same bars as at block size 16: bit-exact caches after the KV write and
the copy-on-write copy; decode within max-abs 2e-2 / mean-abs 2e-3 of the
float64 oracle; NaN in every padding slot.
"""
import numpy as np
import pytest

import oracle
import workloads
from tests import harness

pytestmark = pytest.mark.gpu

BLOCK_SIZES = pytest.mark.parametrize("bs", [8, 32])


@pytest.fixture(scope="module")
def pk():
    import torch

    from paged_kv_cache_92_gb300 import build

    build.build()
    import paged_kv_cache_92_gb300 as pk

    pk.load()
    assert torch.cuda.is_available()
    return pk


def _case(lens, Hq, Hkv, bs, seed, QL=0, D=128, extra_blocks=3):
    import torch

    lens = np.asarray(lens, dtype=np.int64)
    need = int(((lens + bs - 1) // bs).sum())
    NB = need + extra_blocks
    order = np.random.default_rng(seed).permutation(NB).astype(np.int32)
    tables = workloads.sequential_tables(lens, order, bs)
    qshape = (len(lens), QL, Hq, D) if QL else (len(lens), Hq, D)
    q = workloads.bf16_normal(qshape, seed + 1, "cuda")
    kc = workloads.bf16_normal((NB, Hkv, bs, D), seed + 2, "cuda")
    vc = workloads.bf16_normal((NB, Hkv, bs, D), seed + 3, "cuda")
    workloads.fill_padding_nan(kc, tables, lens, bs)
    workloads.fill_padding_nan(vc, tables, lens, bs)
    return q, kc, vc, tables, lens.astype(np.int32), torch


def _decode(pk, q, kc, vc, tables, lens, torch, **kw):
    out = pk.pa_decode(q, kc, vc, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                       max_context_len=int(lens.max()), **kw)
    torch.cuda.synchronize()
    return out


# ---------------------------------------------------------------- whole steps through the pool


@BLOCK_SIZES
@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
def test_llama8b_layer_step(pk, bs, fused):
    """The pool lays out the 64-sequence layer at this block size; one step
    (KV write + decode) against the oracle's own pool model and decode."""
    case = harness.build_case(workloads.llama8b_layer(block_size=bs))
    out, kg, vg = harness.run_step_gpu(case, fused_append=fused)
    ref, ko, vo = harness.run_step_oracle(case)
    assert np.array_equal(oracle.bf16_bits(kg.cpu()), ko)
    assert np.array_equal(oracle.bf16_bits(vg.cpu()), vo)
    harness.assert_close(harness.bf16_tensor_to_f64(out), ref)
    assert pk.pa_device_errors() == 0


@BLOCK_SIZES
def test_llama70b_long_step(pk, bs):
    case = harness.build_case(workloads.llama70b_long(batch=8, block_size=bs))
    out, kg, vg = harness.run_step_gpu(case, fused_append=True)
    units = harness.sample_units(8, 64, 96, seed=5)
    ref, ko, vo = harness.run_step_oracle(case, units=units)
    assert np.array_equal(oracle.bf16_bits(kg.cpu()), ko)
    got = harness.bf16_tensor_to_f64(out)
    harness.assert_close(np.stack([got[b, h] for b, h in units]), ref)
    assert pk.pa_device_errors() == 0


# ---------------------------------------------------------------- decode edge cases


@BLOCK_SIZES
@pytest.mark.parametrize("G,Hkv", [(1, 8), (2, 4), (4, 8), (8, 8), (4, 1), (8, 2), (1, 1)])
def test_edge_lengths(pk, bs, G, Hkv):
    """Lengths at and around every block boundary of both sizes, and long
    enough to split over CTAs."""
    lens = [1, 7, 8, 9, 15, 16, 17, 31, 32, 33, 100, 511, 513, 1025, 4097]
    q, kc, vc, tables, lens, torch = _case(lens, G * Hkv, Hkv, bs, seed=bs * 10 + G * 3 + Hkv)
    out = _decode(pk, q, kc, vc, tables, lens, torch)
    ref = oracle.paged_decode(q.cpu(), kc.cpu(), vc.cpu(), tables, lens)
    harness.assert_close(harness.bf16_tensor_to_f64(out), ref)
    assert pk.pa_device_errors() == 0


@BLOCK_SIZES
def test_split_and_placement(pk, bs):
    """One long sequence beside short ones (stream-K pieces across CTAs), and
    the same logical cache under another physical placement gives the same
    bits."""
    import torch

    q, kc, vc, tables, lens, _ = _case([9000, 3, 47, 700], 32, 8, bs, seed=90 + bs)
    a = _decode(pk, q, kc, vc, tables, lens, torch)
    ref = oracle.paged_decode(q.cpu(), kc.cpu(), vc.cpu(), tables, lens)
    harness.assert_close(harness.bf16_tensor_to_f64(a), ref)
    NB = kc.shape[0]
    perm = np.random.default_rng(3).permutation(NB)
    kcb, vcb = torch.empty_like(kc), torch.empty_like(vc)
    kcb[torch.from_numpy(perm).cuda()] = kc
    vcb[torch.from_numpy(perm).cuda()] = vc
    tables_b = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    b = _decode(pk, q, kcb, vcb, tables_b, lens, torch)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("bs,G,Hkv,QL", [(8, 4, 8, 2), (8, 1, 8, 8), (8, 2, 2, 4), (32, 4, 8, 4),
                                         (32, 8, 8, 2), (32, 1, 1, 16), (32, 4, 1, 3),
                                         # column groups: 8 columns per KV head at block
                                         # size 8, 16 at 32
                                         (8, 4, 8, 8), (8, 8, 2, 3), (32, 4, 8, 16),
                                         (32, 8, 8, 5)])
def test_multi_token(pk, bs, G, Hkv, QL):
    lens = [L for L in (QL, 9, 16, 17, 31, 33, 34, 100, 513, 2049) if L >= QL]
    q, kc, vc, tables, lens, torch = _case(lens, G * Hkv, Hkv, bs, seed=bs + G * 7 + QL, QL=QL)
    out = _decode(pk, q, kc, vc, tables, lens, torch)
    ref = oracle.paged_decode_multi(q.cpu(), kc.cpu(), vc.cpu(), tables, lens)
    harness.assert_close(harness.bf16_tensor_to_f64(out), ref)
    assert pk.pa_device_errors() == 0


@pytest.mark.parametrize("G,Hkv,QL,lens", [
    (4, 8, 8, [5000, 40, 33, 700] * 4),    # two heads per item (one 32-key block a chunk)
    (4, 8, 64, [3000, 64, 65, 1023]),      # one head per item (two blocks a chunk), two tiles
    (8, 8, 8, [4100, 2900]),               # keys split over CTAs
    (2, 3, 16, [1500, 16, 2600]),          # odd KV head count
    (4, 8, 16, [900, 31, 32, 33] * 16),    # 256 items, no split
    (4, 8, 64, [700, 64, 65, 1023] * 8),   # two tiles per item, sharing each load
])
def test_query_major_block_size_32(pk, G, Hkv, QL, lens):
    """The query-major kernel at block size 32: boxes of HB heads x 32 keys,
    lengths across 32-key block and chunk boundaries, every key new at L = Q."""
    q, kc, vc, tables, lens, torch = _case(lens, G * Hkv, Hkv, 32, seed=180 + G + QL, QL=QL)
    out = _decode(pk, q, kc, vc, tables, lens, torch)
    ref = oracle.paged_decode_multi(q.cpu(), kc.cpu(), vc.cpu(), tables, lens)
    harness.assert_close(harness.bf16_tensor_to_f64(out), ref)
    assert pk.pa_device_errors() == 0


@BLOCK_SIZES
def test_copy_blocks_bit_exact(pk, bs):
    import torch

    rng = np.random.default_rng(bs)
    k0 = workloads.bf16_normal((12, 8, bs, 128), 5, "cuda")
    v0 = workloads.bf16_normal((12, 8, bs, 128), 6, "cuda")
    kc, vc = k0.clone(), v0.clone()
    pairs = np.array([[1, 7], [3, 2], [11, 0]], dtype=np.int32)
    pk.pa_copy_blocks(kc, vc, torch.from_numpy(pairs).cuda())
    torch.cuda.synchronize()
    ko, vo = oracle.copy_blocks(oracle.bf16_bits(k0.cpu()), oracle.bf16_bits(v0.cpu()), pairs)
    assert np.array_equal(oracle.bf16_bits(kc.cpu()), ko)
    assert np.array_equal(oracle.bf16_bits(vc.cpu()), vo)
    _ = rng


@BLOCK_SIZES
@pytest.mark.parametrize("G,Hkv,QL", [(4, 8, 1), (8, 1, 1), (1, 4, 1), (4, 2, 3), (4, 8, 8)])
def test_head_dim_64(pk, bs, G, Hkv, QL):
    """head_dim 64 at block sizes 8 and 32: lengths around both block sizes,
    one sequence split over CTAs, several new tokens (column groups at 8)."""
    nb = 2 * int(__import__("torch").cuda.get_device_properties(0).multi_processor_count) + 3
    lens = [L for L in (QL, 7, 8, 9, 31, 32, 33, 100, 513, nb * bs + 1) if L >= QL]
    q, kc, vc, tables, lens, torch = _case(lens, G * Hkv, Hkv, bs, seed=bs * 7 + G + QL, D=64,
                                           QL=QL if QL > 1 else 0)
    out = _decode(pk, q, kc, vc, tables, lens, torch)
    if QL > 1:
        ref = oracle.paged_decode_multi(q.cpu(), kc.cpu(), vc.cpu(), tables, lens)
    else:
        ref = oracle.paged_decode(q.cpu(), kc.cpu(), vc.cpu(), tables, lens)
    harness.assert_close(harness.bf16_tensor_to_f64(out), ref)
    assert pk.pa_device_errors() == 0


# ---------------------------------------------------------------- the CUDA-core kernel


@BLOCK_SIZES
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G,Hkv", [(1, 8), (4, 8), (8, 8), (4, 3)])
def test_cuda_core_edge_lengths(pk, bs, D, G, Hkv):
    """Block and partition boundaries on the CUDA-core kernel (4 KV heads
    with G 4 is a shape only it takes)."""
    lens = [1, bs - 1, bs, bs + 1, 100, 511, 512, 513, 1025, 1600]
    q, kc, vc, tables, lens, torch = _case(lens, G * Hkv, Hkv, bs, seed=900 + bs + G + Hkv + D, D=D)
    out = _decode(pk, q, kc, vc, tables, lens, torch, variant=pk.DECODE_CUDA_CORE)
    harness.assert_close(harness.bf16_tensor_to_f64(out),
                         oracle.paged_decode(q.cpu(), kc.cpu(), vc.cpu(), tables, lens))
    assert pk.pa_device_errors() == 0


@BLOCK_SIZES
@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
def test_cuda_core_llama8b_layer_step(pk, bs, fused):
    case = harness.build_case(workloads.llama8b_layer(block_size=bs))
    out, kg, vg = harness.run_step_gpu(case, variant=1, fused_append=fused)
    ref, ko, vo = harness.run_step_oracle(case)
    assert np.array_equal(oracle.bf16_bits(kg.cpu()), ko)
    assert np.array_equal(oracle.bf16_bits(vg.cpu()), vo)
    harness.assert_close(harness.bf16_tensor_to_f64(out), ref)
    assert pk.pa_device_errors() == 0


@BLOCK_SIZES
def test_cuda_core_multi_token(pk, bs):
    QL = 3
    lens = [QL, bs + 1, 2 * bs + 2, 600]
    q, kc, vc, tables, lens, torch = _case(lens, 32, 8, bs, seed=910 + bs, QL=QL)
    out = _decode(pk, q, kc, vc, tables, lens, torch, variant=pk.DECODE_CUDA_CORE)
    harness.assert_close(harness.bf16_tensor_to_f64(out),
                         oracle.paged_decode_multi(q.cpu(), kc.cpu(), vc.cpu(), tables, lens))


def test_cuda_core_partitions_must_be_whole_blocks(pk):
    import torch

    q, kc, vc, tables, lens, _ = _case([40], 8, 2, 32, seed=8)
    with pytest.raises(pk.PagedKVError):
        _decode(pk, q, kc, vc, tables, lens, torch, variant=pk.DECODE_CUDA_CORE,
                partition_tokens=48)


# ---------------------------------------------------------------- the 8-bit cache at block size 32


def _fp8_case(pk, lens, Hq, Hkv, seed, QL=0, BS=32, D=128):
    """The 8-bit cache at block size BS (V^T in sub-tiles of W = min(BS, 16)
    keys), every slot written through pa_reshape_and_cache_fp8, E4M3 NaN in
    every padding slot."""
    import torch

    lens = np.asarray(lens, dtype=np.int64)
    need = int(((lens + BS - 1) // BS).sum())
    NB = need + 3
    order = np.random.default_rng(seed).permutation(NB).astype(np.int32)
    tables = workloads.sequential_tables(lens, order, BS)
    qshape = (len(lens), QL, Hq, D) if QL else (len(lens), Hq, D)
    q = workloads.bf16_normal(qshape, seed + 1, "cuda")
    kn = workloads.bf16_normal((NB * BS, Hkv, D), seed + 2, "cuda")
    vn = workloads.bf16_normal((NB * BS, Hkv, D), seed + 3, "cuda")
    rng = np.random.default_rng(seed + 4)
    ks = torch.from_numpy((0.05 * np.exp(rng.uniform(-0.5, 0.5, Hkv))).astype(np.float32)).cuda()
    vs = torch.from_numpy((0.03 * np.exp(rng.uniform(-0.5, 0.5, Hkv))).astype(np.float32)).cuda()
    W = min(BS, 16)
    k8 = torch.zeros((NB, Hkv, BS, D), dtype=torch.uint8, device="cuda")
    v8 = torch.zeros((NB, Hkv, BS // W, D, W), dtype=torch.uint8, device="cuda")
    pk.pa_reshape_and_cache_fp8(kn, vn, k8, v8, torch.arange(NB * BS, device="cuda"), ks, vs)
    for b, L in enumerate(lens):
        if L % BS:
            blk, off = int(tables[b, (L - 1) // BS]), int(L % BS)
            k8[blk, :, off:, :] = 0x7F  # E4M3 NaN in the padding slots
            for o in range(off, BS):
                v8[blk, :, o // W, :, o % W] = 0x7F
    torch.cuda.synchronize()
    return q, k8, v8, ks, vs, tables, lens.astype(np.int32), kn, vn, torch


def test_fp8_write_bit_exact_at_block_size_32(pk):
    import torch

    Hkv, D, NB, BS = 4, 128, 6, 32
    rng = np.random.default_rng(11)
    T = 70
    kn = torch.from_numpy(rng.standard_normal((T, Hkv, D)) * 30).to(torch.bfloat16)
    vn = torch.from_numpy(rng.standard_normal((T, Hkv, D)) * 30).to(torch.bfloat16)
    ks = np.array([1.0, 0.5, 2.0, 0.37], dtype=np.float32)
    vs = np.array([1.0, 3.0, 0.25, 1.7], dtype=np.float32)
    slots = rng.permutation(NB * BS)[:T].astype(np.int64)
    slots[[4, 40]] = -1
    k0 = rng.integers(0, 256, size=(NB, Hkv, BS, D), dtype=np.uint8)
    v0 = rng.integers(0, 256, size=(NB, Hkv, BS // 16, D, 16), dtype=np.uint8)
    kc, vc = torch.from_numpy(k0).cuda(), torch.from_numpy(v0).cuda()
    pk.pa_reshape_and_cache_fp8(kn.cuda(), vn.cuda(), kc, vc, torch.from_numpy(slots).cuda(),
                                torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda())
    torch.cuda.synchronize()
    ko, vo = oracle.reshape_and_cache_fp8(kn, vn, k0, v0.reshape(NB, Hkv, BS, D), slots, ks, vs)
    assert np.array_equal(kc.cpu().numpy(), ko)
    assert np.array_equal(vc.cpu().numpy().reshape(NB, Hkv, BS, D), vo)
    assert pk.pa_device_errors() == 0


@pytest.mark.parametrize("G,Hkv", [(4, 8), (8, 8), (1, 4), (4, 2), (8, 1)])
def test_fp8_decode_at_block_size_32(pk, G, Hkv):
    lens = [1, 15, 16, 17, 31, 32, 33, 100, 513, 1025, 4097]
    q, k8, v8, ks, vs, tables, lens, _, _, torch = _fp8_case(pk, lens, G * Hkv, Hkv,
                                                              seed=40 + G + Hkv)
    out = _decode(pk, q, k8, v8, tables, lens, torch, k_scale=ks, v_scale=vs)
    NB = k8.shape[0]
    want = oracle.paged_decode_fp8(q.cpu(), k8.cpu().numpy(), v8.cpu().numpy().reshape(NB, Hkv, 32, 128),
                                   ks.cpu().numpy(), vs.cpu().numpy(), tables, lens)
    harness.assert_close(harness.bf16_tensor_to_f64(out), want)
    assert pk.pa_device_errors() == 0


def test_fp8_multi_token_at_block_size_32(pk):
    QL = 2
    lens = [2, 17, 31, 32, 33, 600, 2049]
    q, k8, v8, ks, vs, tables, lens, _, _, torch = _fp8_case(pk, lens, 32, 8, seed=77, QL=QL)
    out = _decode(pk, q, k8, v8, tables, lens, torch, k_scale=ks, v_scale=vs)
    NB = k8.shape[0]
    want = oracle.paged_decode_multi_fp8(q.cpu(), k8.cpu().numpy(),
                                         v8.cpu().numpy().reshape(NB, 8, 32, 128),
                                         ks.cpu().numpy(), vs.cpu().numpy(), tables, lens)
    harness.assert_close(harness.bf16_tensor_to_f64(out), want)
    assert pk.pa_device_errors() == 0


@pytest.mark.parametrize("G,Hkv", [(4, 8), (1, 4), (8, 2)])
def test_fp8_decode_at_block_size_32_cuda_core(pk, G, Hkv):
    lens = [1, 31, 32, 33, 513, 1025]
    q, k8, v8, ks, vs, tables, lens, _, _, torch = _fp8_case(pk, lens, G * Hkv, Hkv,
                                                              seed=140 + G + Hkv)
    out = _decode(pk, q, k8, v8, tables, lens, torch, k_scale=ks, v_scale=vs,
                  variant=pk.DECODE_CUDA_CORE)
    NB = k8.shape[0]
    want = oracle.paged_decode_fp8(q.cpu(), k8.cpu().numpy(), v8.cpu().numpy().reshape(NB, Hkv, 32, 128),
                                   ks.cpu().numpy(), vs.cpu().numpy(), tables, lens)
    harness.assert_close(harness.bf16_tensor_to_f64(out), want)
    assert pk.pa_device_errors() == 0


# ---------------------------------------------------------------- the 8-bit cache at block size 8
#
# V^T is stored in sub-tiles of 8 keys, [NB][Hkv][D][8] per (block, head); the
# tensor-core kernel's operand layout needs 16-key rows, so this cache decodes
# on the CUDA-core kernel whatever the variant says.


def test_fp8_write_bit_exact_at_block_size_8(pk):
    import torch

    Hkv, D, NB, BS = 4, 128, 10, 8
    rng = np.random.default_rng(12)
    T = 60
    kn = torch.from_numpy(rng.standard_normal((T, Hkv, D)) * 30).to(torch.bfloat16)
    vn = torch.from_numpy(rng.standard_normal((T, Hkv, D)) * 30).to(torch.bfloat16)
    ks = np.array([1.0, 0.5, 2.0, 0.37], dtype=np.float32)
    vs = np.array([1.0, 3.0, 0.25, 1.7], dtype=np.float32)
    slots = rng.permutation(NB * BS)[:T].astype(np.int64)
    slots[[3, 30]] = -1
    k0 = rng.integers(0, 256, size=(NB, Hkv, BS, D), dtype=np.uint8)
    v0 = rng.integers(0, 256, size=(NB, Hkv, D, BS), dtype=np.uint8)
    kc, vc = torch.from_numpy(k0).cuda(), torch.from_numpy(v0).cuda()
    pk.pa_reshape_and_cache_fp8(kn.cuda(), vn.cuda(), kc, vc, torch.from_numpy(slots).cuda(),
                                torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda())
    torch.cuda.synchronize()
    ko, vo = oracle.reshape_and_cache_fp8(kn, vn, k0, v0.reshape(NB, Hkv, BS, D), slots, ks, vs)
    assert np.array_equal(kc.cpu().numpy(), ko)
    assert np.array_equal(vc.cpu().numpy().reshape(NB, Hkv, BS, D), vo)
    assert pk.pa_device_errors() == 0


@pytest.mark.parametrize("variant", [0, 1])
@pytest.mark.parametrize("D,G,Hkv", [(128, 4, 8), (128, 8, 8), (64, 1, 4), (128, 2, 1)])
def test_fp8_decode_at_block_size_8(pk, variant, D, G, Hkv):
    lens = [1, 7, 8, 9, 100, 511, 512, 513, 1025]
    q, k8, v8, ks, vs, tables, lens, _, _, torch = _fp8_case(pk, lens, G * Hkv, Hkv,
                                                              seed=150 + G + Hkv + D, BS=8, D=D)
    out = _decode(pk, q, k8, v8, tables, lens, torch, k_scale=ks, v_scale=vs, variant=variant)
    NB = k8.shape[0]
    want = oracle.paged_decode_fp8(q.cpu(), k8.cpu().numpy(), v8.cpu().numpy().reshape(NB, Hkv, 8, D),
                                   ks.cpu().numpy(), vs.cpu().numpy(), tables, lens)
    harness.assert_close(harness.bf16_tensor_to_f64(out), want)
    assert pk.pa_device_errors() == 0


def test_fp8_multi_token_at_block_size_8(pk):
    QL = 3
    lens = [3, 9, 17, 600]
    q, k8, v8, ks, vs, tables, lens, _, _, torch = _fp8_case(pk, lens, 32, 8, seed=160, QL=QL, BS=8)
    out = _decode(pk, q, k8, v8, tables, lens, torch, k_scale=ks, v_scale=vs)
    NB = k8.shape[0]
    want = oracle.paged_decode_multi_fp8(q.cpu(), k8.cpu().numpy(),
                                         v8.cpu().numpy().reshape(NB, 8, 8, 128),
                                         ks.cpu().numpy(), vs.cpu().numpy(), tables, lens)
    harness.assert_close(harness.bf16_tensor_to_f64(out), want)
    assert pk.pa_device_errors() == 0


def test_fp8_fused_append_at_block_size_8(pk):
    """The step's write (the preparation launch's write, same slot rule), then
    the decode: caches bit-exact against the oracle's write, rows against its
    decode."""
    import torch

    lens = [1, 8, 9, 300, 1025]
    q, k8, v8, ks, vs, tables, lens, _, _, _ = _fp8_case(pk, lens, 32, 8, seed=170, BS=8)
    NB, BS, Hkv, D = k8.shape[0], 8, 8, 128
    slots = np.array([int(tables[b, (L - 1) // BS]) * BS + (L - 1) % BS for b, L in enumerate(lens)],
                     dtype=np.int64)
    kn = workloads.bf16_normal((len(lens), Hkv, D), 171, "cuda")
    vn = workloads.bf16_normal((len(lens), Hkv, D), 172, "cuda")
    k0, v0 = k8.cpu().numpy(), v8.cpu().numpy().reshape(NB, Hkv, BS, D)
    out = pk.pa_append_decode(q, k8, v8, torch.from_numpy(tables).cuda(),
                              torch.from_numpy(lens).cuda(), int(lens.max()), kn, vn,
                              torch.from_numpy(slots).cuda(), k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pk.pa_device_errors() == 0
    ko, vo = oracle.reshape_and_cache_fp8(kn.cpu(), vn.cpu(), k0, v0, slots, ks.cpu().numpy(),
                                          vs.cpu().numpy())
    assert np.array_equal(k8.cpu().numpy(), ko)
    assert np.array_equal(v8.cpu().numpy().reshape(NB, Hkv, BS, D), vo)
    want = oracle.paged_decode_fp8(q.cpu(), ko, vo, ks.cpu().numpy(), vs.cpu().numpy(), tables,
                                   lens)
    harness.assert_close(harness.bf16_tensor_to_f64(out), want)
