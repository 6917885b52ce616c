"""Builds one decode step both ways from a seeded recipe.

Product side: the C++ pool lays out the cache, the CUDA kernels run the step
(copy-on-write copies, KV write, decode). Oracle side: the block-manager
model lays out its own tables, the C oracle does the same step on the host.
The two layouts are asserted identical (integer work, bit-exact) before any
arithmetic is compared.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

import oracle
import workloads

ATOL_MAX = 2e-2   # max-abs error bound for bf16 inputs with fp32 accumulation
ATOL_MEAN = 2e-3  # mean-abs error bound


@dataclasses.dataclass
class Case:
    recipe: workloads.Recipe
    tables0: np.ndarray      # before the step's append
    tables: np.ndarray       # after
    lens0: np.ndarray
    lens: np.ndarray
    slots: np.ndarray        # int64 [T]
    cows: np.ndarray         # int32 [P][2]
    q: object                # torch bf16 on device
    k_new: object
    v_new: object
    k_cache: object          # state before the step (NaN in padding slots)
    v_cache: object


def build_case(r: workloads.Recipe, device: str = "cuda") -> Case:
    import paged_kv_cache_92_gb300 as pk

    pool = pk.Pool(r.num_blocks, r.block_size, free_order=r.free_order)
    model = oracle.PoolModel(r.num_blocks, r.block_size, free_order=r.free_order)
    sp = workloads.drive_prefill(pool, r)
    sm = workloads.drive_prefill(model, r)
    t0p, t0m = workloads.tables_of(pool, sp), workloads.tables_of(model, sm)
    assert np.array_equal(t0p, t0m), "product pool and model disagree on the prefill layout"
    slp, cwp = workloads.drive_step_append(pool, sp, r)
    slm, cwm = workloads.drive_step_append(model, sm, r)
    assert np.array_equal(slp, slm) and np.array_equal(cwp, cwm), "step slots / CoW pairs differ"
    tp, tm = workloads.tables_of(pool, sp), workloads.tables_of(model, sm)
    assert np.array_equal(tp, tm)
    q, kn, vn, kc, vc = workloads.step_tensors(r, device)
    workloads.fill_padding_nan(kc, t0m, r.lens0, r.block_size)
    workloads.fill_padding_nan(vc, t0m, r.lens0, r.block_size)
    pool.close()
    return Case(r, t0m, tm, r.lens0.astype(np.int32), (r.lens0 + r.append).astype(np.int32),
                slm, cwm, q, kn, vn, kc, vc)


def run_step_gpu(case: Case, partition_tokens: int = 0, variant: int = 0,
                 overlap_prologue: bool = False, fused_append: bool = False):
    """The hot path on the GPU: copy_blocks -> reshape_and_cache -> decode
    (or copy_blocks -> pa_append_decode, the KV write fused into the decode)."""
    import torch

    import paged_kv_cache_92_gb300 as pk

    dev = case.q.device
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    # tables and lengths are uploaded before the first kernel of the step, as
    # overlap_prologue requires
    tables = torch.from_numpy(case.tables).to(dev)
    lens = torch.from_numpy(case.lens).to(dev)
    if len(case.cows):
        pk.pa_copy_blocks(kc, vc, torch.from_numpy(case.cows).to(dev))
    slots = torch.from_numpy(case.slots).to(dev)
    if fused_append:
        out = pk.pa_append_decode(case.q, kc, vc, tables, lens, int(case.lens.max()),
                                  case.k_new, case.v_new, slots,
                                  partition_tokens=partition_tokens, variant=variant,
                                  overlap_prologue=overlap_prologue)
    else:
        pk.pa_reshape_and_cache(case.k_new, case.v_new, kc, vc, slots)
        out = pk.pa_decode(case.q, kc, vc, tables, lens, max_context_len=int(case.lens.max()),
                           partition_tokens=partition_tokens, variant=variant,
                           overlap_prologue=overlap_prologue)
    torch.cuda.synchronize()
    return out, kc, vc


def oracle_caches(case: Case):
    """The oracle's caches after the step's copy-on-write and KV write (bits)."""
    kc = oracle.bf16_bits(case.k_cache.cpu())
    vc = oracle.bf16_bits(case.v_cache.cpu())
    if len(case.cows):
        kc, vc = oracle.copy_blocks(kc, vc, case.cows)
    return oracle.reshape_and_cache(case.k_new.cpu(), case.v_new.cpu(), kc, vc, case.slots)


def run_step_oracle(case: Case, units=None):
    """Oracle side of the same step. Returns (out float64, k_cache bits, v_cache bits)."""
    kc = oracle.bf16_bits(case.k_cache.cpu())
    vc = oracle.bf16_bits(case.v_cache.cpu())
    if len(case.cows):
        kc, vc = oracle.copy_blocks(kc, vc, case.cows)
    kc, vc = oracle.reshape_and_cache(case.k_new.cpu(), case.v_new.cpu(), kc, vc, case.slots)
    out = oracle.paged_decode(case.q.cpu(), kc, vc, case.tables, case.lens, units=units)
    return out, kc, vc


def bf16_tensor_to_f64(t) -> np.ndarray:
    return oracle.bf16_to_f64(t.cpu())


def assert_close(got: np.ndarray, want: np.ndarray, atol_max: float = ATOL_MAX,
                 atol_mean: float = ATOL_MEAN) -> dict:
    assert got.shape == want.shape
    assert np.isfinite(got).all(), "non-finite values in the GPU output"
    err = np.abs(got - want)
    stats = {"max_abs": float(err.max()), "mean_abs": float(err.mean())}
    assert stats["max_abs"] <= atol_max, stats
    assert stats["mean_abs"] <= atol_mean, stats
    return stats


def sample_units(B: int, Hq: int, n: int, seed: int = 0, must: Optional[list] = None):
    rng = np.random.default_rng(seed)
    units = {(int(b), int(h)) for b, h in zip(rng.integers(0, B, n), rng.integers(0, Hq, n))}
    for u in must or []:
        units.add(u)
    return sorted(units)
