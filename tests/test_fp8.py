"""GPU parity of the 8-bit (E4M3) KV cache against the float64 oracle.

Bit-exact: the quantising KV write (whole caches compared, including exact
rounding ties and saturation) and the block copy. Decode: max-abs <= 2e-2 and
mean-abs <= 2e-3 against the exact attention over the dequantised cache (the
oracle decodes every code exactly and multiplies by its head's scale in
float64). Padding slots hold E4M3 NaN codes, so a masked slot that leaks into
a result fails the finiteness check.
"""
import numpy as np
import pytest

import oracle
import workloads
from tests import harness

pytestmark = pytest.mark.gpu

NAN8 = 0x7F


@pytest.fixture(scope="module")
def pk():
    import torch

    from paged_kv_cache_92_gb300 import build

    build.build()
    import paged_kv_cache_92_gb300 as pk

    pk.load()
    assert torch.cuda.is_available()
    return pk


def _scales(Hkv, seed, base):
    rng = np.random.default_rng(seed)
    return (base * np.exp(rng.uniform(-0.5, 0.5, size=Hkv))).astype(np.float32)


def _fp8_case(pk, lens, Hq, Hkv, seed, extra_blocks=3, D=128, QL=1):
    """Random tables; every slot of the pool written through
    pa_reshape_and_cache_fp8 (bf16 N(0,1) rows, per-head scales); padding
    slots of each sequence's last block then set to the NaN code."""
    import torch

    lens = np.asarray(lens, dtype=np.int64)
    need = int(((lens + 15) // 16).sum())
    NB = need + extra_blocks
    order = np.random.default_rng(seed).permutation(NB).astype(np.int32)
    tables = workloads.sequential_tables(lens, order, 16)
    q = workloads.bf16_normal((len(lens), QL, Hq, D) if QL > 1 else (len(lens), Hq, D), seed + 1,
                              "cuda")
    kn = workloads.bf16_normal((NB * 16, Hkv, D), seed + 2, "cuda")
    vn = workloads.bf16_normal((NB * 16, Hkv, D), seed + 3, "cuda")
    ks = torch.from_numpy(_scales(Hkv, seed + 4, 0.05)).cuda()
    vs = torch.from_numpy(_scales(Hkv, seed + 5, 0.03)).cuda()
    k8 = torch.zeros((NB, Hkv, 16, D), dtype=torch.uint8, device="cuda")
    v8 = torch.zeros((NB, Hkv, D, 16), dtype=torch.uint8, device="cuda")
    slots = torch.arange(NB * 16, dtype=torch.int64, device="cuda")
    pk.pa_reshape_and_cache_fp8(kn, vn, k8, v8, slots, ks, vs)
    for b, L in enumerate(lens):
        if L % 16:
            blk = int(tables[b, (L - 1) // 16])
            k8[blk, :, L % 16:, :] = NAN8
            v8[blk, :, :, L % 16:] = NAN8
    torch.cuda.synchronize()
    return q, k8, v8, ks, vs, tables, lens.astype(np.int32)


def _decode_and_check(pk, case, units=None, **kw):
    import torch

    q, k8, v8, ks, vs, tables, lens = case
    out = pk.pa_decode(q, k8, v8, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                       max_context_len=int(lens.max()), k_scale=ks, v_scale=vs, **kw)
    torch.cuda.synchronize()
    got = harness.bf16_tensor_to_f64(out)
    want = oracle.paged_decode_fp8(q.cpu(), k8.cpu().numpy(), v8.cpu().numpy(), ks.cpu().numpy(),
                                   vs.cpu().numpy(), tables, lens, units=units)
    if units is not None:
        got = np.stack([got[b, h] for b, h in units])
    stats = harness.assert_close(got, want)
    assert pk.pa_device_errors() == 0
    return stats


# ---------------------------------------------------------------- the write


def test_fp8_write_bit_exact_with_ties_and_saturation(pk):
    """Whole caches against the oracle's quantising write. The rows include
    every exact midpoint between neighbouring E4M3 values (round to nearest
    even decides them), values past 448 (saturation), zeros and negative
    slots."""
    import torch

    Hkv, D, NB = 4, 128, 12
    rng = np.random.default_rng(5)
    grid = oracle.e4m3_to_f64(np.arange(0x7F))
    mids = (grid[1:] + grid[:-1]) / 2  # exact in bf16 (at most 5 significant bits)
    special = np.concatenate([mids, -mids, [0.0, -0.0, 448.0, 460.0, 470.0, 1000.0, -3e4]])
    T = 40
    kn = rng.standard_normal((T, Hkv, D)) * 40
    vn = rng.standard_normal((T, Hkv, D)) * 40
    flat = kn.reshape(-1)
    flat[: len(special)] = special
    vflat = vn.reshape(-1)
    vflat[-len(special):] = special[::-1]
    kn_t = torch.from_numpy(kn).to(torch.bfloat16)
    vn_t = torch.from_numpy(vn).to(torch.bfloat16)
    ks = np.array([1.0, 0.5, 2.0, 0.37], dtype=np.float32)  # 1.0: the ties stay exact ties
    vs = np.array([1.0, 3.0, 0.25, 1.7], dtype=np.float32)
    slots = rng.permutation(NB * 16)[:T].astype(np.int64)
    slots[[3, 17]] = -1
    k0 = rng.integers(0, 256, size=(NB, Hkv, 16, D), dtype=np.uint8)
    v0 = rng.integers(0, 256, size=(NB, Hkv, D, 16), dtype=np.uint8)
    kc, vc = torch.from_numpy(k0).cuda(), torch.from_numpy(v0).cuda()
    pk.pa_reshape_and_cache_fp8(kn_t.cuda(), vn_t.cuda(), kc, vc, torch.from_numpy(slots).cuda(),
                                torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda())
    torch.cuda.synchronize()
    ko, vo = oracle.reshape_and_cache_fp8(kn_t, vn_t, k0, v0, slots, ks, vs)
    assert np.array_equal(kc.cpu().numpy(), ko)
    assert np.array_equal(vc.cpu().numpy(), vo)
    assert pk.pa_device_errors() == 0


def test_fp8_copy_blocks_bit_exact(pk):
    import torch

    rng = np.random.default_rng(6)
    k0 = rng.integers(0, 256, size=(10, 8, 16, 128), dtype=np.uint8)
    v0 = rng.integers(0, 256, size=(10, 8, 128, 16), dtype=np.uint8)
    kc, vc = torch.from_numpy(k0).cuda(), torch.from_numpy(v0).cuda()
    pairs = np.array([[1, 7], [3, 2], [9, 0]], dtype=np.int32)
    pk.pa_copy_blocks_fp8(kc, vc, torch.from_numpy(pairs).cuda())
    torch.cuda.synchronize()
    ko, vo = oracle.copy_blocks_fp8(k0, v0, pairs)
    assert np.array_equal(kc.cpu().numpy(), ko) and np.array_equal(vc.cpu().numpy(), vo)


# ---------------------------------------------------------------- the decode


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("Hkv", [1, 4, 8])
def test_fp8_decode_edge_lengths(pk, G, Hkv):
    lens = [1, 15, 16, 17, 100, 511, 513, 1025]
    case = _fp8_case(pk, lens, Hq=G * Hkv, Hkv=Hkv, seed=40 + G + Hkv)
    _decode_and_check(pk, case)


def test_fp8_decode_llama8b_layer_shape(pk):
    """64 sequences, 32/8 heads, lengths U[128, 2048]: the bench's shape."""
    r = workloads.llama8b_layer()
    case = _fp8_case(pk, r.lens0 + 1, Hq=32, Hkv=8, seed=51)
    units = harness.sample_units(64, 32, 256, seed=2)
    _decode_and_check(pk, case, units=units)


def test_fp8_decode_llama70b_shape(pk):
    """8 sequences, 64/8 heads, lengths U[8192, 32768]: sequences spread over
    many CTAs, merged by the split-K merge."""
    r = workloads.llama70b_long(batch=8)
    case = _fp8_case(pk, r.lens0 + 1, Hq=64, Hkv=8, seed=52)
    units = harness.sample_units(8, 64, 96, seed=3)
    _decode_and_check(pk, case, units=units)


def test_fp8_decode_zero_length_rows_are_zero(pk):
    import torch

    case = _fp8_case(pk, [40, 0, 3, 0], Hq=8, Hkv=2, seed=53)
    q, k8, v8, ks, vs, tables, lens = case
    out = torch.full_like(q, 7.0)
    pk.pa_decode(q, k8, v8, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                 max_context_len=40, k_scale=ks, v_scale=vs, out=out)
    torch.cuda.synchronize()
    got = harness.bf16_tensor_to_f64(out)
    assert not got[1].any() and not got[3].any()
    want = oracle.paged_decode_fp8(q.cpu(), k8.cpu().numpy(), v8.cpu().numpy(), ks.cpu().numpy(),
                                   vs.cpu().numpy(), tables, lens,
                                   units=[(b, h) for b in (0, 2) for h in range(8)])
    harness.assert_close(np.concatenate([got[0], got[2]]), want)


def test_fp8_decode_placement_invariance_bit_exact(pk):
    """The same logical cache under two physical placements gives the same bits."""
    import torch

    lens = [300, 47, 900]
    a = _fp8_case(pk, lens, Hq=16, Hkv=4, seed=54)
    q, k8, v8, ks, vs, tables, lens_a = a
    NB = k8.shape[0]
    perm = np.random.default_rng(9).permutation(NB)
    inv = np.argsort(perm)
    k8b, v8b = torch.empty_like(k8), torch.empty_like(v8)
    k8b[torch.from_numpy(perm).cuda()] = k8
    v8b[torch.from_numpy(perm).cuda()] = v8
    tables_b = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    assert (inv[perm] == np.arange(NB)).all()
    outs = []
    for kc, vc, tb in ((k8, v8, tables), (k8b, v8b, tables_b)):
        outs.append(pk.pa_decode(q, kc, vc, torch.from_numpy(tb).cuda(),
                                 torch.from_numpy(lens_a).cuda(), max_context_len=900,
                                 k_scale=ks, v_scale=vs))
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


# ---------------------------------------------------------------- the CUDA-core kernel
#
# The CUDA-core variant dequantises the codes in fp32: K rows with the head's
# scale folded into the query, V from each V^T tile transposed in shared
# memory, the V scale on the weighted sum. Same oracle, same bar.


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G,Hkv", [(1, 8), (4, 8), (8, 8), (2, 1), (4, 4), (8, 2)])
def test_fp8_cuda_core_edge_lengths(pk, D, G, Hkv):
    lens = [1, 15, 16, 17, 100, 511, 512, 513, 1025, 1600]
    case = _fp8_case(pk, lens, Hq=G * Hkv, Hkv=Hkv, seed=600 + G * 10 + Hkv + D, D=D)
    _decode_and_check(pk, case, variant=pk.DECODE_CUDA_CORE)


def test_fp8_cuda_core_matches_tensor_core(pk):
    import torch

    case = _fp8_case(pk, [40, 700, 2049], Hq=32, Hkv=8, seed=610)
    q, k8, v8, ks, vs, tables, lens = case
    outs = [harness.bf16_tensor_to_f64(
        pk.pa_decode(q, k8, v8, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                     max_context_len=2049, k_scale=ks, v_scale=vs, variant=v))
        for v in (pk.DECODE_TENSOR_CORE, pk.DECODE_CUDA_CORE)]
    d = np.abs(outs[0] - outs[1])
    assert d.max() <= 2e-2 and d.mean() <= 2e-3


def test_fp8_cuda_core_zero_length_rows_are_zero(pk):
    import torch

    case = _fp8_case(pk, [40, 0, 3, 0, 600], Hq=8, Hkv=2, seed=611)
    q, k8, v8, ks, vs, tables, lens = case
    out = torch.full_like(q, 7.0)
    pk.pa_decode(q, k8, v8, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                 max_context_len=600, k_scale=ks, v_scale=vs, out=out,
                 variant=pk.DECODE_CUDA_CORE)
    torch.cuda.synchronize()
    got = harness.bf16_tensor_to_f64(out)
    assert not got[1].any() and not got[3].any()
    keep = [0, 2, 4]
    want = oracle.paged_decode_fp8(q.cpu(), k8.cpu().numpy(), v8.cpu().numpy(), ks.cpu().numpy(),
                                   vs.cpu().numpy(), tables, lens,
                                   units=[(b, h) for b in keep for h in range(8)])
    harness.assert_close(np.concatenate([got[b] for b in keep]), want)


def test_fp8_cuda_core_placement_invariance_bit_exact(pk):
    import torch

    q, k8, v8, ks, vs, tables, lens = _fp8_case(pk, [300, 47, 900], Hq=16, Hkv=4, seed=612)
    NB = k8.shape[0]
    perm = np.random.default_rng(19).permutation(NB)
    k8b, v8b = torch.empty_like(k8), torch.empty_like(v8)
    k8b[torch.from_numpy(perm).cuda()] = k8
    v8b[torch.from_numpy(perm).cuda()] = v8
    tables_b = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    outs = [pk.pa_decode(q, kc, vc, torch.from_numpy(tb).cuda(), torch.from_numpy(lens).cuda(),
                         max_context_len=900, k_scale=ks, v_scale=vs, variant=pk.DECODE_CUDA_CORE)
            for kc, vc, tb in ((k8, v8, tables), (k8b, v8b, tables_b))]
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_fp8_cuda_core_several_new_tokens(pk):
    import torch

    QL = 3
    q, k8, v8, ks, vs, tables, lens = _fp8_case(pk, [QL, 17, 513, 1100], Hq=32, Hkv=8, seed=613,
                                                QL=QL)
    out = pk.pa_decode(q, k8, v8, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                       max_context_len=1100, k_scale=ks, v_scale=vs, variant=pk.DECODE_CUDA_CORE)
    torch.cuda.synchronize()
    assert pk.pa_device_errors() == 0
    want = oracle.paged_decode_multi_fp8(q.cpu(), k8.cpu().numpy(), v8.cpu().numpy(),
                                         ks.cpu().numpy(), vs.cpu().numpy(), tables, lens)
    harness.assert_close(harness.bf16_tensor_to_f64(out), want)


# ---------------------------------------------------------------- the write fused into the decode


def _fused_fp8(pk, lens, Hq, Hkv, seed, QL=1, bad=None, bs=16, variant=0):
    """pa_append_decode on the 8-bit cache: the new tokens' (the last QL of each
    sequence) slots are overwritten with the quantised rows of k_new/v_new, as
    pa_reshape_and_cache_fp8 would, before the decode reads them."""
    import torch

    D = 128
    lens = np.asarray(lens, dtype=np.int64)
    NB = int(((lens + bs - 1) // bs).sum()) + 3
    order = np.random.default_rng(seed).permutation(NB).astype(np.int32)
    tables = workloads.sequential_tables(lens, order, bs)
    q = workloads.bf16_normal((len(lens), QL, Hq, D) if QL > 1 else (len(lens), Hq, D), seed + 1,
                              "cuda")
    ks = torch.from_numpy(_scales(Hkv, seed + 4, 0.05)).cuda()
    vs = torch.from_numpy(_scales(Hkv, seed + 5, 0.03)).cuda()
    # the pool before the step: every slot holds the oracle's codes of bf16
    # N(0,1) rows; the padding slots of each last block hold the NaN code
    k0, v0 = oracle.reshape_and_cache_fp8(
        workloads.bf16_normal((NB * bs, Hkv, D), seed + 6, "cpu"),
        workloads.bf16_normal((NB * bs, Hkv, D), seed + 7, "cpu"),
        np.zeros((NB, Hkv, bs, D), np.uint8), np.zeros((NB, Hkv, bs, D), np.uint8),
        np.arange(NB * bs, dtype=np.int64), ks.cpu().numpy(), vs.cpu().numpy())
    v0 = v0.reshape(NB, Hkv, bs // 16, D, 16)
    for b, L in enumerate(lens):
        if L % bs:
            blk = int(tables[b, (L - 1) // bs])
            k0[blk, :, L % bs:, :] = NAN8
            for o in range(int(L % bs), bs):
                v0[blk, :, o // 16, :, o % 16] = NAN8
    slots = []
    for b, L in enumerate(lens):
        for i in range(QL):
            pos = int(L) - QL + i
            slots.append(int(tables[b, pos // bs]) * bs + pos % bs)
    slots = np.array(slots, dtype=np.int64)
    if bad is not None:
        slots = bad(slots)
    T = len(slots)
    kn = workloads.bf16_normal((T, Hkv, D), seed + 2, "cuda")
    vn = workloads.bf16_normal((T, Hkv, D), seed + 3, "cuda")
    k8, v8 = torch.from_numpy(k0).cuda(), torch.from_numpy(v0).cuda()
    out = pk.pa_append_decode(q, k8, v8, torch.from_numpy(tables).cuda(),
                              torch.from_numpy(lens.astype(np.int32)).cuda(), int(lens.max()),
                              kn, vn, torch.from_numpy(slots).cuda(), k_scale=ks, v_scale=vs,
                              variant=variant)
    torch.cuda.synchronize()
    return dict(q=q, k0=k0, v0=v0, k8=k8, v8=v8, kn=kn, vn=vn, ks=ks, vs=vs, slots=slots,
                tables=tables, lens=lens.astype(np.int32), out=out, NB=NB, Hkv=Hkv, bs=bs)


@pytest.mark.parametrize("bs,QL,variant", [(16, 1, 0), (16, 2, 0), (32, 1, 0), (32, 2, 0),
                                           (16, 1, 1), (16, 3, 1)])
def test_fp8_fused_append_matches_the_quantising_write_and_oracle(pk, bs, QL, variant):
    """variant 1: the CUDA-core kernel (the preparation launch's write, then the decode)."""
    lens = [QL, 15, 16, 17, 33, 100, 513, 2049]
    c = _fused_fp8(pk, lens, 32, 8, seed=60 + bs + QL + 7 * variant, QL=QL, bs=bs,
                   variant=variant)
    assert pk.pa_device_errors() == 0
    NB, Hkv, D = c["NB"], c["Hkv"], 128
    ks, vs = c["ks"].cpu().numpy(), c["vs"].cpu().numpy()
    ko, vo = oracle.reshape_and_cache_fp8(c["kn"].cpu(), c["vn"].cpu(), c["k0"],
                                          c["v0"].reshape(NB, Hkv, bs, D), c["slots"], ks, vs)
    assert np.array_equal(c["k8"].cpu().numpy(), ko)
    assert np.array_equal(c["v8"].cpu().numpy().reshape(NB, Hkv, bs, D), vo)
    if QL > 1:
        want = oracle.paged_decode_multi_fp8(c["q"].cpu(), ko, vo, ks, vs, c["tables"], c["lens"])
    else:
        want = oracle.paged_decode_fp8(c["q"].cpu(), ko, vo, ks, vs, c["tables"], c["lens"])
    harness.assert_close(harness.bf16_tensor_to_f64(c["out"]), want)


@pytest.mark.parametrize("variant", [0, 1])
def test_fp8_fused_append_slot_rules(pk, variant):
    """A slot that is not its token's is not written (PA_DEVERR_APPEND_SLOT); a
    negative slot writes nothing."""
    def bad(s):
        s = s.copy()
        s[1] = s[1] + 1 if s[1] % 16 != 15 else s[1] - 1
        s[2] = -1
        return s

    c = _fused_fp8(pk, [40, 70, 33], 16, 4, seed=71, bad=bad, variant=variant)
    assert pk.pa_device_errors() & 0x20
    NB, Hkv, D = c["NB"], c["Hkv"], 128
    keep = [0]
    ko, vo = oracle.reshape_and_cache_fp8(c["kn"].cpu()[keep], c["vn"].cpu()[keep], c["k0"],
                                          c["v0"].reshape(NB, Hkv, 16, D), c["slots"][keep],
                                          c["ks"].cpu().numpy(), c["vs"].cpu().numpy())
    assert np.array_equal(c["k8"].cpu().numpy(), ko)
    assert np.array_equal(c["v8"].cpu().numpy().reshape(NB, Hkv, 16, D), vo)


@pytest.mark.parametrize("scale_set", [0, 1, 2])
def test_fp8_fused_write_every_bf16_value(pk, scale_set):
    """The fused write divides by the head's scale with a reciprocal and one
    correction step; its codes must equal the oracle's for every bf16 bit
    pattern (zeros, subnormals, infinities and NaNs included), for power-of-two
    and other scales. 64 sequences append one token each with 8 KV heads of
    128 values: 65,536 K and 65,536 V values per call."""
    import torch

    B, Hkv, D, bs = 64, 8, 128, 16
    rng = np.random.default_rng(90 + scale_set)
    lens = rng.integers(1, 100, size=B).astype(np.int64)
    NB = int(((lens + bs - 1) // bs).sum()) + 2
    order = rng.permutation(NB).astype(np.int32)
    tables = workloads.sequential_tables(lens, order, bs)
    slots = np.array([int(tables[b, (L - 1) // bs]) * bs + (L - 1) % bs
                      for b, L in enumerate(lens)], dtype=np.int64)
    bits = np.arange(65536, dtype=np.uint16)
    kn = torch.from_numpy(bits.view(np.int16).reshape(B, Hkv, D).copy()).view(torch.bfloat16)
    vn = torch.from_numpy(rng.permutation(bits).view(np.int16).reshape(B, Hkv, D).copy()
                          ).view(torch.bfloat16)
    if scale_set == 0:
        ks = np.array([1.0, 0.5, 0.25, 2.0, 0.0625, 4.0, 0.125, 1.0], np.float32)
        vs = np.array([0.75, 3.0, 0.1, 0.3, 7.0, 0.01, 1.5, 0.2], np.float32)
    else:
        ks = (np.exp(rng.uniform(-6, 4, size=Hkv))).astype(np.float32)
        vs = (np.exp(rng.uniform(-6, 4, size=Hkv))).astype(np.float32)
    k0 = rng.integers(0, 0x7F, size=(NB, Hkv, bs, D), dtype=np.uint8)
    v0 = rng.integers(0, 0x7F, size=(NB, Hkv, bs, D), dtype=np.uint8)
    k8 = torch.from_numpy(k0).cuda()
    v8 = torch.from_numpy(v0.reshape(NB, Hkv, bs // 16, D, 16)).cuda()  # V^T sub-tiles
    q = workloads.bf16_normal((B, 32, D), 93, "cuda")
    pk.pa_append_decode(q, k8, v8, torch.from_numpy(tables).cuda(),
                        torch.from_numpy(lens.astype(np.int32)).cuda(), int(lens.max()),
                        kn.cuda(), vn.cuda(), torch.from_numpy(slots).cuda(),
                        k_scale=torch.from_numpy(ks).cuda(), v_scale=torch.from_numpy(vs).cuda())
    torch.cuda.synchronize()
    assert pk.pa_device_errors() == 0
    ko, vo = oracle.reshape_and_cache_fp8(kn, vn, k0, v0, slots, ks, vs)
    assert np.array_equal(k8.cpu().numpy(), ko)
    assert np.array_equal(v8.cpu().numpy().reshape(NB, Hkv, bs, D), vo)


@pytest.mark.parametrize("pinned", [True, False])
def test_fp8_step_host_matches_device_step(pk, pinned):
    """pa_step_host on the 8-bit cache (one copy-on-write pair, then the
    quantising KV write and the decode) gives the device-side step's output
    and caches bit for bit: pa_copy_blocks_fp8, then pa_append_decode."""
    import torch

    Hq, Hkv, D, bs = 32, 8, 128, 16
    lens = np.array([1, 17, 64, 300, 1025], dtype=np.int64)
    NB = int(((lens + bs - 1) // bs).sum()) + 4
    order = np.random.default_rng(95).permutation(NB).astype(np.int32)
    tables = workloads.sequential_tables(lens, order, bs)
    slots = np.array([int(tables[b, (L - 1) // bs]) * bs + (L - 1) % bs
                      for b, L in enumerate(lens)], dtype=np.int64)
    used = set(int(x) for x in tables.ravel() if x >= 0)
    spare = [b for b in range(NB) if b not in used]
    cows = np.array([[int(tables[3, 2]), spare[0]]], dtype=np.int32)  # a full block of seq 3
    B = len(lens)
    ks = torch.from_numpy(_scales(Hkv, 96, 0.05)).cuda()
    vs = torch.from_numpy(_scales(Hkv, 97, 0.03)).cuda()
    k0, v0 = oracle.reshape_and_cache_fp8(
        workloads.bf16_normal((NB * bs, Hkv, D), 98, "cpu"),
        workloads.bf16_normal((NB * bs, Hkv, D), 99, "cpu"),
        np.zeros((NB, Hkv, bs, D), np.uint8), np.zeros((NB, Hkv, bs, D), np.uint8),
        np.arange(NB * bs, dtype=np.int64), ks.cpu().numpy(), vs.cpu().numpy())
    q = workloads.bf16_normal((B, Hq, D), 100, "cuda")
    kn = workloads.bf16_normal((B, Hkv, D), 101, "cuda")
    vn = workloads.bf16_normal((B, Hkv, D), 102, "cuda")
    t_d = torch.from_numpy(tables).cuda()
    l_d = torch.from_numpy(lens.astype(np.int32)).cuda()

    def fresh():
        return (torch.from_numpy(k0).cuda(),
                torch.from_numpy(v0.reshape(NB, Hkv, bs // 16, D, 16)).cuda())

    kd, vd = fresh()
    pk.pa_copy_blocks_fp8(kd, vd, torch.from_numpy(cows).cuda())
    want = pk.pa_append_decode(q, kd, vd, t_d, l_d, int(lens.max()), kn, vn,
                               torch.from_numpy(slots).cuda(), k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()

    kh, vh = fresh()
    p = pk.make_step_host_params(kh, vh, B, Hq, tables.shape[1], int(lens.max()),
                                 num_cow_pairs=len(cows), k_scale=ks, v_scale=vs)
    host_in = pk.pack_step_inputs(p, q.cpu(), kn.cpu(), vn.cpu(), slots, tables,
                                  lens.astype(np.int32), cows, pin=pinned)
    host_out = torch.empty((B, Hq, D), dtype=torch.bfloat16)
    if pinned:
        host_out = host_out.pin_memory()
    ws = torch.empty(pk.pa_step_host_workspace_size(p), dtype=torch.uint8, device="cuda")
    pk.pa_step_host(p, host_in, host_out, ws)
    assert pk.pa_device_errors() == 0
    assert torch.equal(host_out.view(torch.int16), want.cpu().view(torch.int16))
    assert torch.equal(kh, kd) and torch.equal(vh, vd)
    # and the caches are the oracle's copy + quantising write
    ko, vo = oracle.copy_blocks_fp8(k0, v0, cows.tolist())
    ko, vo = oracle.reshape_and_cache_fp8(kn.cpu(), vn.cpu(), ko, vo, slots, ks.cpu().numpy(),
                                          vs.cpu().numpy())
    assert np.array_equal(kh.cpu().numpy(), ko)
    assert np.array_equal(vh.cpu().numpy().reshape(NB, Hkv, bs, D), vo)


def test_fp8_step_host_with_several_new_tokens(pk):
    """pa_step_host on the 8-bit cache with query_len 2: output and caches bit
    for bit against pa_append_decode on the same inputs."""
    import torch

    QL = 2
    c = _fused_fp8(pk, [QL, 17, 40, 300, 1025], 32, 8, seed=130, QL=QL)
    NB, Hkv, D, bs = c["NB"], c["Hkv"], 128, c["bs"]
    B = len(c["lens"])
    kh = torch.from_numpy(c["k0"]).cuda()
    vh = torch.from_numpy(c["v0"]).cuda()
    p = pk.make_step_host_params(kh, vh, B, 32, c["tables"].shape[1], int(c["lens"].max()),
                                 k_scale=c["ks"], v_scale=c["vs"], query_len=QL)
    host_in = pk.pack_step_inputs(p, c["q"].cpu(), c["kn"].cpu(), c["vn"].cpu(), c["slots"],
                                  c["tables"], c["lens"])
    host_out = torch.empty((B, QL, 32, D), dtype=torch.bfloat16).pin_memory()
    ws = torch.empty(pk.pa_step_host_workspace_size(p), dtype=torch.uint8, device="cuda")
    pk.pa_step_host(p, host_in, host_out, ws)
    assert pk.pa_device_errors() == 0
    assert torch.equal(host_out.view(torch.int16), c["out"].cpu().view(torch.int16))
    assert torch.equal(kh, c["k8"]) and torch.equal(vh, c["v8"])


def test_fp8_wait_budget_exit_reports_timeout_and_leaves_the_context_usable(pk):
    """The 8-bit decode with a 1 us budget per barrier wait: the launch gives
    up, reports PA_DEVERR_TIMEOUT and winds down; the next launch with the
    default budget matches the oracle."""
    import torch

    rng = np.random.default_rng(41)
    case = _fp8_case(pk, rng.integers(128, 2048, size=64), 32, 8, seed=43)
    q, k8, v8, ks, vs, tables, lens = case
    assert pk.pa_device_errors() == 0
    for _ in range(2):
        pk.pa_decode(q, k8, v8, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(),
                     max_context_len=int(lens.max()), k_scale=ks, v_scale=vs, wait_timeout_us=1)
        assert pk.pa_device_errors() & pk.DEVERR_TIMEOUT
    _decode_and_check(pk, case)
    assert pk.pa_device_errors() == 0
