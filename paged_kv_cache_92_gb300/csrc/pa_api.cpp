// C ABI entry points of libpagedkv.so: host-side argument validation, launch
// policy (split-K partition count, workspace carve-up) and status reporting.
// Every check here runs before anything is launched.
#include <cuda_runtime_api.h>

#include <cstdint>
#include <cstdio>
#include <cstring>

#include "pa_internal.h"
#include "pa_query_major.h"

namespace pa {

namespace {
thread_local char g_msg[512] = "";

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int resolve_partition_tokens(const pa_decode_params* p) {
  return p->partition_tokens == 0 ? kDefaultPartitionTokens : p->partition_tokens;
}

// Full host validation of decode params. Returns PA_OK or an error (message set).
pa_status check_decode(const pa_decode_params* p, bool need_pointers) {
  if (!p) return set_error(PA_ERR_INVALID_ARG, "pa_decode: params is NULL");
  if (p->num_seqs < 0 || p->num_seqs > 65535)
    return set_error(PA_ERR_INVALID_ARG, "pa_decode: num_seqs must be in [0, 65535]");
  if (p->num_q_heads < 1 || p->num_kv_heads < 1 || p->num_q_heads % p->num_kv_heads != 0)
    return set_error(PA_ERR_INVALID_ARG,
                     "pa_decode: num_q_heads must be a positive multiple of num_kv_heads");
  if (p->num_kv_heads > 65535)
    return set_error(PA_ERR_INVALID_ARG, "pa_decode: num_kv_heads must be <= 65535");
  if (!block_size_ok(p->block_size))
    return set_error(PA_ERR_UNSUPPORTED, "pa_decode: block_size must be 8, 16 or 32");
  if (p->head_dim != 64 && p->head_dim != 128)
    return set_error(PA_ERR_UNSUPPORTED, "pa_decode: head_dim must be 64 or 128");
  const int g = p->num_q_heads / p->num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8)
    return set_error(PA_ERR_UNSUPPORTED, "pa_decode: query heads per KV head must be 1, 2, 4 or 8");
  if (p->num_blocks < 1) return set_error(PA_ERR_INVALID_ARG, "pa_decode: num_blocks < 1");
  if (p->max_blocks_per_seq < 1)
    return set_error(PA_ERR_INVALID_ARG, "pa_decode: max_blocks_per_seq < 1");
  if (p->max_context_len < 1)
    return set_error(PA_ERR_INVALID_ARG, "pa_decode: max_context_len < 1");
  if (int64_t(p->max_blocks_per_seq) * p->block_size > INT32_MAX)
    return set_error(PA_ERR_INVALID_ARG, "pa_decode: max_blocks_per_seq too large");
  const int pt = resolve_partition_tokens(p);
  if (pt < kBlockSize || pt > kMaxPartitionTokens || pt % kBlockSize != 0)
    return set_error(PA_ERR_INVALID_ARG,
                     "pa_decode: partition_tokens must be 0 or a multiple of 16 in [16, 4096]");
  if (p->variant != PA_DECODE_TENSOR_CORE && p->variant != PA_DECODE_CUDA_CORE)
    return set_error(PA_ERR_INVALID_ARG, "pa_decode: variant must be 0 (tensor core) or 1 (CUDA core)");
  if (int64_t(p->num_blocks) * p->num_kv_heads * p->block_size >= (int64_t(1) << 31) - 16 ||
      int64_t(p->num_seqs) * p->num_q_heads >= (int64_t(1) << 31) - 16)
    return set_error(PA_ERR_INVALID_ARG, "pa_decode: cache or query rows exceed 2^31");
  if (!(p->scale > 0.0f) || p->scale != p->scale)
    return set_error(PA_ERR_INVALID_ARG, "pa_decode: scale must be a positive finite number");
  if (p->kv_dtype != PA_KV_BF16 && p->kv_dtype != PA_KV_FP8_E4M3)
    return set_error(PA_ERR_INVALID_ARG, "pa_decode: kv_dtype must be PA_KV_BF16 or PA_KV_FP8_E4M3");
  if (p->query_len < 0 || p->query_len > 1024)
    return set_error(PA_ERR_INVALID_ARG, "pa_decode: query_len must be in [0, 1024]");
  if (p->wait_timeout_us < 0)
    return set_error(PA_ERR_INVALID_ARG, "pa_decode: wait_timeout_us must be >= 0");
  if (int64_t(p->num_seqs) * query_len_of(p) * p->num_q_heads >= (int64_t(1) << 31) - 16)
    return set_error(PA_ERR_INVALID_ARG, "pa_decode: query rows exceed 2^31");
  // the CUDA-core kernel's partitions are whole blocks
  if (!decode_uses_tc(p) && pt % p->block_size != 0)
    return set_error(PA_ERR_INVALID_ARG,
                     "pa_decode: on the CUDA-core kernel partition_tokens must be a multiple of "
                     "block_size");
  // the CUDA-core kernel runs one CTA row per (sequence, new token) in grid z
  if (!decode_uses_tc(p) && int64_t(p->num_seqs) * query_len_of(p) > 65535)
    return set_error(PA_ERR_UNSUPPORTED,
                     "pa_decode: on the CUDA-core kernel num_seqs * query_len must be <= 65535 "
                     "(the tensor-core kernel takes num_kv_heads 1/2/4/8 and num_seqs * "
                     "(query_len split into column groups) <= 16384)");
  if (p->kv_dtype == PA_KV_FP8_E4M3) {
    if (need_pointers && p->num_seqs > 0 &&
        (!p->k_scale || !p->v_scale || (reinterpret_cast<uintptr_t>(p->k_scale) & 3u) ||
         (reinterpret_cast<uintptr_t>(p->v_scale) & 3u)))
      return set_error(PA_ERR_INVALID_ARG,
                       "pa_decode: the 8-bit cache needs k_scale and v_scale (float arrays)");
  }
  if (need_pointers && p->num_seqs > 0) {
    if (!p->q || !p->out || !p->k_cache || !p->v_cache || !p->block_tables || !p->context_lens)
      return set_error(PA_ERR_INVALID_ARG, "pa_decode: a required pointer is NULL");
    if (!aligned16(p->q) || !aligned16(p->out) || !aligned16(p->k_cache) ||
        !aligned16(p->v_cache))
      return set_error(PA_ERR_INVALID_ARG,
                       "pa_decode: q, out, k_cache and v_cache must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(p->block_tables) & 3u) ||
        (reinterpret_cast<uintptr_t>(p->context_lens) & 3u))
      return set_error(PA_ERR_INVALID_ARG, "pa_decode: int32 arrays must be 4-byte aligned");
  }
  return PA_OK;
}

int num_partitions_for(const pa_decode_params* p) {
  const int pt = resolve_partition_tokens(p);
  int64_t cap = int64_t(p->max_blocks_per_seq) * p->block_size;
  int64_t mx = p->max_context_len < cap ? p->max_context_len : cap;
  return int((mx + pt - 1) / pt);
}
}  // namespace

pa_status set_error(pa_status s, const char* msg) {
  if (s != PA_OK) std::snprintf(g_msg, sizeof(g_msg), "%s", msg);
  return s;
}

pa_status set_cuda_error(const char* where, int err) {
  std::snprintf(g_msg, sizeof(g_msg), "%s: %s", where,
                cudaGetErrorString(static_cast<cudaError_t>(err)));
  return PA_ERR_CUDA;
}

bool decode_uses_tc(const pa_decode_params* p) {
  return p->variant == PA_DECODE_TENSOR_CORE && tc_supports(p);
}

WorkspaceLayout decode_workspace_layout(const pa_decode_params* p, int num_partitions,
                                        int grid) {
  WorkspaceLayout w{};
  const size_t H = kWorkspaceHeaderBytes;
  if (use_query_major(p)) {
    // the header, and with split keys the partials (m, l pairs, then O rows)
    w.total = H;
    const int ns = query_major_splits(p);
    if (ns > 1) {
      const size_t rows = size_t(p->num_seqs) * query_len_of(p) * p->num_q_heads * ns;
      w.tc_m = H;
      w.tc_acc = w.tc_m + round_up(rows * 2 * sizeof(float), 256);
      w.total = w.tc_acc + round_up(rows * p->head_dim * sizeof(float), 256);
    }
    return w;
  }
  if (!decode_uses_tc(p)) {
    // CUDA-core kernel: per-partition partials (only when a sequence can split)
    w.total = H;
    if (num_partitions > 1) {
      const size_t rows =
          size_t(p->num_seqs) * query_len_of(p) * p->num_q_heads * num_partitions;
      w.simt_m = H;
      w.simt_l = w.simt_m + round_up(rows * sizeof(float), 256);
      w.simt_acc = w.simt_l + round_up(rows * sizeof(float), 256);
      w.total = w.simt_acc + round_up(rows * p->head_dim * sizeof(float), 256);
    }
    return w;
  }
  // tensor-core kernel: stream-K plan, then one partial per (sequence, CTA)
  // segment and query column (= query head for one token per sequence). With
  // no device to query, the grid is taken as 256 CTAs (an upper bound).
  // (one virtual sequence per sequence and column group of its new tokens)
  const size_t V = size_t(tc_virtual_seqs(p));
  const size_t segs = V + size_t(grid > 0 ? grid : 256);
  const size_t rows = segs * size_t(tc_cols(p));
  w.tc_plan = H;
  w.tc_m = w.tc_plan + round_up((V + 2) * sizeof(int), 256);
  w.tc_l = w.tc_m + round_up(rows * sizeof(float), 256);
  w.tc_acc = w.tc_l + round_up(rows * sizeof(float), 256);
  size_t tc_end = w.tc_acc + round_up(rows * p->head_dim * sizeof(float), 256);
  const size_t n_pad = size_t(tc_n_pad(tc_cols(p)));
  if (p->kv_dtype == PA_KV_FP8_E4M3) {  // split queries [B][2N][D] bytes and [B][N] floats
    w.tc_q8 = tc_end;
    w.tc_qa = w.tc_q8 + round_up(V * 2 * n_pad * p->head_dim, 256);
    tc_end = w.tc_qa + round_up(V * n_pad * sizeof(float), 256);
  } else if (query_len_of(p) > 1) {  // queries in column order, bf16 [V][N][D]
    w.tc_qp = tc_end;
    tc_end = w.tc_qp + round_up(V * n_pad * p->head_dim * 2, 256);
  }
  w.total = tc_end;
  return w;
}

// Launch the selected decode kernel and its merge.
static pa_status run_decode(const pa_decode_params* p, unsigned char* ws,
                            const WorkspaceLayout& w, int np, int grid, pa_stream_t stream,
                            const char* who, const pa_append_params* append = nullptr) {
  DecodeLaunch L;
  L.p = p;
  L.append = append;
  L.partition_tokens = resolve_partition_tokens(p);
  L.num_partitions = np;
  L.grid = grid;
  char where[96];
  int e = 0;
  if (use_query_major(p)) {
    if (append) {  // the step's write first, with the fused path's slot rule
      AppendCheck chk;
      chk.block_tables = p->block_tables;
      chk.context_lens = p->context_lens;
      chk.max_blocks_per_seq = p->max_blocks_per_seq;
      chk.cap = p->max_blocks_per_seq * p->block_size < p->max_context_len
                    ? p->max_blocks_per_seq * p->block_size : p->max_context_len;
      chk.q_len = query_len_of(p);
      e = launch_reshape_and_cache(append->k_new, append->v_new, append->k_cache,
                                   append->v_cache, append->slot_mapping,
                                   p->num_seqs * query_len_of(p), p->num_kv_heads, p->head_dim,
                                   p->block_size, p->num_blocks, stream, chk);
    }
    // the decode's set-up overlaps the write (which changes neither tables nor
    // lengths), or the previous kernel when the caller allows it
    const bool split = query_major_splits(p) > 1;
    if (!e)
      e = launch_query_major_tc(p, stream, split ? reinterpret_cast<float*>(ws + w.tc_m) : nullptr,
                                split ? reinterpret_cast<float*>(ws + w.tc_acc) : nullptr,
                                append != nullptr || p->overlap_prologue != 0);
  } else if (decode_uses_tc(p)) {
    if (grid <= 0)
      return set_cuda_error("the SM count of the current device", int(cudaErrorNoDevice));
    L.plan = reinterpret_cast<int*>(ws + w.tc_plan);
    L.q8 = p->kv_dtype == PA_KV_FP8_E4M3 ? ws + w.tc_q8 : nullptr;
    L.q_inv_alpha =
        p->kv_dtype == PA_KV_FP8_E4M3 ? reinterpret_cast<float*>(ws + w.tc_qa) : nullptr;
    L.qp = p->kv_dtype == PA_KV_BF16 && query_len_of(p) > 1 ? ws + w.tc_qp : nullptr;
    L.part_m = reinterpret_cast<float*>(ws + w.tc_m);
    L.part_l = reinterpret_cast<float*>(ws + w.tc_l);
    L.part_acc = reinterpret_cast<float*>(ws + w.tc_acc);
    e = launch_decode_tc(L, stream);
  } else {
    if (append && p->kv_dtype == PA_KV_FP8_E4M3) {
      // the quantising write with the fused path's slot rule, then the decode
      e = launch_quantize_q(nullptr, nullptr, nullptr, query_map(p), p, append, stream);
    } else if (append) {  // the same effect in two launches
      AppendCheck chk;
      chk.block_tables = p->block_tables;
      chk.context_lens = p->context_lens;
      chk.max_blocks_per_seq = p->max_blocks_per_seq;
      chk.cap = p->max_blocks_per_seq * p->block_size < p->max_context_len
                    ? p->max_blocks_per_seq * p->block_size : p->max_context_len;
      chk.q_len = query_len_of(p);
      e = launch_reshape_and_cache(append->k_new, append->v_new, append->k_cache,
                                   append->v_cache, append->slot_mapping,
                                   p->num_seqs * query_len_of(p), p->num_kv_heads, p->head_dim,
                                   p->block_size, p->num_blocks, stream, chk);
    }
    if (e) {
      std::snprintf(where, sizeof(where), "%s: launch", who);
      return set_cuda_error(where, e);
    }
    L.plan = nullptr;
    L.part_m = np > 1 ? reinterpret_cast<float*>(ws + w.simt_m) : nullptr;
    L.part_l = np > 1 ? reinterpret_cast<float*>(ws + w.simt_l) : nullptr;
    L.part_acc = np > 1 ? reinterpret_cast<float*>(ws + w.simt_acc) : nullptr;
    e = launch_decode(L, stream);
    if (!e) e = launch_merge(L, stream);
  }
  if (e) {
    std::snprintf(where, sizeof(where), "%s: launch", who);
    return set_cuda_error(where, e);
  }
  return PA_OK;
}

// ---- host-driven step: packed input layout and the decode params over it

// The device address of host memory `p` when kernels can reach it (memory
// pinned through CUDA, mapped under unified addressing) and it is `align`-byte
// aligned there; nullptr otherwise (pageable memory, or an address CUDA does
// not know). Clears the error that the query leaves for unknown addresses.
static const void* device_view(const void* p, size_t align) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr) return nullptr;
  if (reinterpret_cast<uintptr_t>(at.devicePointer) % align != 0) return nullptr;
  return at.devicePointer;
}

static pa_status check_step(const pa_step_host_params* p) {
  if (!p) return set_error(PA_ERR_INVALID_ARG, "pa_step_host: params is NULL");
  if (p->num_seqs < 0 || p->num_q_heads < 1 || p->num_kv_heads < 1 || p->head_dim < 1 ||
      p->max_blocks_per_seq < 1)
    return set_error(PA_ERR_INVALID_ARG, "pa_step_host: counts must be positive");
  if (p->num_cow_pairs < 0 || p->num_cow_pairs > 65535)
    return set_error(PA_ERR_INVALID_ARG, "pa_step_host: num_cow_pairs must be in [0, 65535]");
  if (p->kv_dtype != PA_KV_BF16 && p->kv_dtype != PA_KV_FP8_E4M3)
    return set_error(PA_ERR_INVALID_ARG, "pa_step_host: kv_dtype must be PA_KV_BF16 or PA_KV_FP8_E4M3");
  if (p->query_len < 0 || p->query_len > 1024)
    return set_error(PA_ERR_INVALID_ARG, "pa_step_host: query_len must be in [0, 1024]");
  return PA_OK;
}

static void step_layout(const pa_step_host_params* p, pa_step_layout* L) {
  const size_t B = size_t(p->num_seqs), D = size_t(p->head_dim);
  const size_t Q = p->query_len > 1 ? size_t(p->query_len) : 1;  // new tokens per sequence
  size_t off = 0;
  auto put = [&](uint64_t& field, size_t bytes) {
    field = off;
    off = round_up(off + bytes, 256);
  };
  put(L->q, B * Q * p->num_q_heads * D * 2);
  put(L->k_new, B * Q * p->num_kv_heads * D * 2);
  put(L->v_new, B * Q * p->num_kv_heads * D * 2);
  put(L->slot_mapping, B * Q * sizeof(int64_t));
  put(L->block_tables, B * size_t(p->max_blocks_per_seq) * sizeof(int32_t));
  put(L->context_lens, B * sizeof(int32_t));
  put(L->cow_pairs, size_t(p->num_cow_pairs) * 2 * sizeof(int32_t));
  L->total = off;
}

// Workspace of a host-driven step: staged input, staged output, decode workspace.
struct StepSpace {
  pa_step_layout in;
  size_t out_off, dec_off, total;
};

static void step_decode_params(const pa_step_host_params* p, unsigned char* ws,
                               const StepSpace& sp, pa_decode_params* d) {
  std::memset(d, 0, sizeof(*d));
  d->q = ws ? ws + sp.in.q : nullptr;
  d->out = ws ? ws + sp.out_off : nullptr;
  d->k_cache = p->k_cache;
  d->v_cache = p->v_cache;
  d->block_tables = ws ? reinterpret_cast<const int32_t*>(ws + sp.in.block_tables) : nullptr;
  d->context_lens = ws ? reinterpret_cast<const int32_t*>(ws + sp.in.context_lens) : nullptr;
  d->max_blocks_per_seq = p->max_blocks_per_seq;
  d->num_seqs = p->num_seqs;
  d->num_q_heads = p->num_q_heads;
  d->num_kv_heads = p->num_kv_heads;
  d->head_dim = p->head_dim;
  d->block_size = p->block_size;
  d->num_blocks = p->num_blocks;
  d->max_context_len = p->max_context_len;
  d->scale = p->scale;
  d->partition_tokens = 0;
  d->variant = p->variant;
  d->overlap_prologue = 0;
  d->kv_dtype = p->kv_dtype;
  d->k_scale = p->k_scale;
  d->v_scale = p->v_scale;
  d->query_len = p->query_len;
}

static StepSpace step_space(const pa_step_host_params* p, const pa_decode_params& d, int np,
                            int grid) {
  StepSpace sp;
  step_layout(p, &sp.in);
  sp.out_off = sp.in.total;
  const size_t out_bytes = size_t(p->num_seqs) * (p->query_len > 1 ? p->query_len : 1) *
                           p->num_q_heads * p->head_dim * 2;
  sp.dec_off = round_up(sp.out_off + out_bytes, 256);
  sp.total = sp.dec_off + decode_workspace_layout(&d, np, grid).total;
  return sp;
}

}  // namespace pa

extern "C" {

const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_OOM: return "PA_ERR_OOM";
    case PA_ERR_REFCOUNT: return "PA_ERR_REFCOUNT";
    case PA_ERR_BOUNDS: return "PA_ERR_BOUNDS";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
  }
  return "PA_ERR_UNKNOWN";
}

const char* pa_last_error(void) { return pa::g_msg; }

int32_t pa_version(void) { return 1; }

pa_status pa_device_errors(pa_stream_t stream, uint32_t* flags) {
  if (!flags) return pa::set_error(PA_ERR_INVALID_ARG, "pa_device_errors: flags is NULL");
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return pa::set_cuda_error("pa_device_errors: stream sync", int(e));
  uint32_t a = 0, b = 0, c = 0, d = 0, qm = 0;
  int r = pa::read_and_clear_decode_errors(&a);
  if (r == 0) r = pa::read_and_clear_decode_tc_errors(&c);
  if (r == 0) r = pa::read_and_clear_cache_errors(&b);
  if (r == 0) r = pa::read_and_clear_fp8_errors(&d);
  if (r == 0) r = pa::read_and_clear_query_major_errors(&qm);
  if (r != 0) return pa::set_cuda_error("pa_device_errors: read", r);
  *flags = a | b | c | d | qm;
  return PA_OK;
}

size_t pa_decode_workspace_size(const pa_decode_params* p) {
  if (pa::check_decode(p, false) != PA_OK) return 0;
  return pa::decode_workspace_layout(p, pa::num_partitions_for(p), pa::tc_grid()).total;
}

pa_status pa_decode(const pa_decode_params* p, void* workspace, size_t workspace_bytes,
                    pa_stream_t stream) {
  pa_status st = pa::check_decode(p, true);
  if (st != PA_OK) return st;
  if (p->num_seqs == 0) return PA_OK;
  const int np = pa::num_partitions_for(p);
  const int grid = pa::tc_grid();
  const pa::WorkspaceLayout w = pa::decode_workspace_layout(p, np, grid);
  if (!workspace || workspace_bytes < w.total)
    return pa::set_error(PA_ERR_INVALID_ARG,
                         "pa_decode: workspace smaller than pa_decode_workspace_size()");
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return pa::set_error(PA_ERR_INVALID_ARG, "pa_decode: workspace must be 256-byte aligned");
  return pa::run_decode(p, static_cast<unsigned char*>(workspace), w, np, grid, stream,
                        "pa_decode");
}

pa_status pa_decode_noalloc(const pa_decode_params* p, pa_stream_t stream) {
  pa_status st = pa::check_decode(p, true);
  if (st != PA_OK) return st;
  if (p->num_seqs == 0) return PA_OK;
  const int np = pa::num_partitions_for(p);
  const int grid = pa::tc_grid();
  const pa::WorkspaceLayout w = pa::decode_workspace_layout(p, np, grid);
  if (w.total > pa::kNoAllocScratchBytes)
    return pa::set_error(PA_ERR_INVALID_ARG,
                         pa::decode_uses_tc(p)
                             ? "pa_decode_noalloc: these shapes need more split-K scratch than the "
                               "library's fixed PA_NOALLOC_SCRATCH_BYTES (the tensor-core kernel's "
                               "partials grow with num_seqs + SM count times the query columns); "
                               "use pa_decode with a workspace"
                             : "pa_decode_noalloc: these shapes need more split-K scratch than the "
                               "library's fixed PA_NOALLOC_SCRATCH_BYTES; use pa_decode with a "
                               "workspace or a larger partition_tokens");
  void* scratch = nullptr;
  const int e = pa::decode_scratch_address(&scratch);
  if (e != 0) return pa::set_cuda_error("pa_decode_noalloc: scratch lookup", e);
  // Nothing in the array needs to start at zero: every call writes its plan
  // and partials before reading them.
  return pa::run_decode(p, static_cast<unsigned char*>(scratch), w, np, grid, stream,
                        "pa_decode_noalloc");
}

pa_status pa_append_decode(const pa_decode_params* p, const pa_append_params* a,
                           void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  pa_status st = pa::check_decode(p, true);
  if (st != PA_OK) return st;
  if (!a) return pa::set_error(PA_ERR_INVALID_ARG, "pa_append_decode: append params are NULL");
  if (p->num_seqs == 0) return PA_OK;
  if (!a->k_new || !a->v_new || !a->slot_mapping || !a->k_cache || !a->v_cache)
    return pa::set_error(PA_ERR_INVALID_ARG, "pa_append_decode: a required pointer is NULL");
  if (a->k_cache != p->k_cache || a->v_cache != p->v_cache)
    return pa::set_error(PA_ERR_INVALID_ARG,
                         "pa_append_decode: append k_cache/v_cache must be the decode's caches");
  if (!pa::aligned16(a->k_new) || !pa::aligned16(a->v_new) ||
      (reinterpret_cast<uintptr_t>(a->slot_mapping) & 7u))
    return pa::set_error(PA_ERR_INVALID_ARG, "pa_append_decode: misaligned pointer");
  const int np = pa::num_partitions_for(p);
  const int grid = pa::tc_grid();
  const pa::WorkspaceLayout w = pa::decode_workspace_layout(p, np, grid);
  if (!workspace || workspace_bytes < w.total)
    return pa::set_error(PA_ERR_INVALID_ARG,
                         "pa_append_decode: workspace smaller than pa_decode_workspace_size()");
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return pa::set_error(PA_ERR_INVALID_ARG, "pa_append_decode: workspace must be 256-byte aligned");
  return pa::run_decode(p, static_cast<unsigned char*>(workspace), w, np, grid, stream,
                        "pa_append_decode", a);
}

pa_status pa_step_host_layout(const pa_step_host_params* p, pa_step_layout* out) {
  pa_status st = pa::check_step(p);
  if (st != PA_OK) return st;
  if (!out) return pa::set_error(PA_ERR_INVALID_ARG, "pa_step_host_layout: out is NULL");
  pa::step_layout(p, out);
  return PA_OK;
}

size_t pa_step_host_workspace_size(const pa_step_host_params* p) {
  if (pa::check_step(p) != PA_OK) return 0;
  pa_decode_params d;
  pa::step_decode_params(p, nullptr, pa::StepSpace{}, &d);
  if (pa::check_decode(&d, false) != PA_OK) return 0;
  return pa::step_space(p, d, pa::num_partitions_for(&d), pa::tc_grid()).total;
}

pa_status pa_step_host(const pa_step_host_params* p, void* workspace, size_t workspace_bytes,
                       pa_stream_t stream) {
  pa_status st = pa::check_step(p);
  if (st != PA_OK) return st;
  if (!p->host_in || !p->host_out || !p->k_cache || !p->v_cache)
    return pa::set_error(PA_ERR_INVALID_ARG, "pa_step_host: a required pointer is NULL");
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return pa::set_error(PA_ERR_INVALID_ARG, "pa_step_host: workspace must be 256-byte aligned");
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  pa_decode_params d;
  pa::step_decode_params(p, nullptr, pa::StepSpace{}, &d);
  st = pa::check_decode(&d, false);
  if (st != PA_OK) return st;
  const int np = pa::num_partitions_for(&d);
  const int grid = pa::tc_grid();
  const pa::StepSpace sp = pa::step_space(p, d, np, grid);
  if (workspace_bytes < sp.total)
    return pa::set_error(PA_ERR_INVALID_ARG,
                         "pa_step_host: workspace smaller than pa_step_host_workspace_size()");
  if (p->num_seqs == 0 && p->num_cow_pairs == 0) return PA_OK;
  pa::step_decode_params(p, ws, sp, &d);
  st = pa::check_decode(&d, true);
  if (st != PA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // Pinned host buffers are addressable from kernels (over NVLink-C2C on a
  // Grace-Blackwell part): a kernel then stages the inputs, and the decode
  // writes the output rows straight into host_out. Other host memory goes
  // through DMA copies.
  const void* in_dev = pa::device_view(p->host_in, 16);
  void* out_dev = const_cast<void*>(pa::device_view(p->host_out, 16));
  cudaError_t e = cudaSuccess;
  if (in_dev) {
    const int r = pa::launch_stage_in(in_dev, ws, sp.in.total, stream);
    if (r != 0) return pa::set_cuda_error("pa_step_host: input staging launch", r);
  } else {
    e = cudaMemcpyAsync(ws, p->host_in, sp.in.total, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return pa::set_cuda_error("pa_step_host: input copy", int(e));
  }
  if (p->num_cow_pairs > 0) {
    // the 8-bit cache's blocks are the bytes of a bf16 block of half the head_dim
    const int r = pa::launch_copy_blocks(p->k_cache, p->v_cache,
                                         reinterpret_cast<const int32_t*>(ws + sp.in.cow_pairs),
                                         p->num_cow_pairs, p->num_kv_heads,
                                         p->kv_dtype == PA_KV_FP8_E4M3 ? p->head_dim / 2
                                                                       : p->head_dim,
                                         p->block_size, p->num_blocks, stream);
    if (r != 0) return pa::set_cuda_error("pa_step_host: copy_blocks launch", r);
  }
  if (p->num_seqs > 0) {
    pa_append_params a;
    a.k_new = ws + sp.in.k_new;
    a.v_new = ws + sp.in.v_new;
    a.slot_mapping = reinterpret_cast<const int64_t*>(ws + sp.in.slot_mapping);
    a.k_cache = p->k_cache;
    a.v_cache = p->v_cache;
    const pa::WorkspaceLayout w = pa::decode_workspace_layout(&d, np, grid);
    if (out_dev) d.out = out_dev;
    if (in_dev && d.variant == PA_DECODE_TENSOR_CORE && pa::tc_supports(&d)) {
      // The lengths and tables in host_in are final before this call, so the
      // tensor-core decode reads them there and plans its work while the
      // staging kernel still runs (programmatic dependent launch); it reads
      // everything else from the staged copy after that kernel completes.
      const unsigned char* hin = static_cast<const unsigned char*>(in_dev);
      d.block_tables = reinterpret_cast<const int32_t*>(hin + sp.in.block_tables);
      d.context_lens = reinterpret_cast<const int32_t*>(hin + sp.in.context_lens);
      d.overlap_prologue = 1;
    }
    st = pa::run_decode(&d, ws + sp.dec_off, w, np, grid, stream, "pa_step_host", &a);
    if (st != PA_OK) return st;
    if (!out_dev) {
      e = cudaMemcpyAsync(p->host_out, ws + sp.out_off,
                          size_t(p->num_seqs) * (p->query_len > 1 ? p->query_len : 1) *
                              p->num_q_heads * p->head_dim * 2,
                          cudaMemcpyDeviceToHost, s);
      if (e != cudaSuccess) return pa::set_cuda_error("pa_step_host: output copy", int(e));
    }
  }
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return pa::set_cuda_error("pa_step_host: synchronize", int(e));
  return PA_OK;
}

pa_status pa_reshape_and_cache(const void* k_new, const void* v_new, void* k_cache,
                               void* v_cache, const int64_t* slot_mapping, int32_t num_tokens,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               int32_t num_blocks, pa_stream_t stream) {
  if (num_tokens < 0 || num_kv_heads < 1 || num_blocks < 1)
    return pa::set_error(PA_ERR_INVALID_ARG,
                         "pa_reshape_and_cache: num_tokens >= 0, num_kv_heads >= 1, num_blocks >= 1");
  if (!pa::block_size_ok(block_size))
    return pa::set_error(PA_ERR_UNSUPPORTED, "pa_reshape_and_cache: block_size must be 8, 16 or 32");
  if (head_dim < 8 || head_dim % 8 != 0 || head_dim > 1024)
    return pa::set_error(PA_ERR_UNSUPPORTED,
                         "pa_reshape_and_cache: head_dim must be a multiple of 8 in [8, 1024]");
  if (num_tokens == 0) return PA_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping)
    return pa::set_error(PA_ERR_INVALID_ARG, "pa_reshape_and_cache: a required pointer is NULL");
  if (!pa::aligned16(k_new) || !pa::aligned16(v_new) || !pa::aligned16(k_cache) ||
      !pa::aligned16(v_cache) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return pa::set_error(PA_ERR_INVALID_ARG, "pa_reshape_and_cache: misaligned pointer");
  // one thread per 16-byte chunk, 256 per CTA: keep the grid within gridDim.x
  if (int64_t(num_tokens) * num_kv_heads * (head_dim / 8) > (int64_t(1) << 38))
    return pa::set_error(PA_ERR_INVALID_ARG, "pa_reshape_and_cache: too many tokens");
  const int e = pa::launch_reshape_and_cache(k_new, v_new, k_cache, v_cache, slot_mapping,
                                             num_tokens, num_kv_heads, head_dim, block_size,
                                             num_blocks, stream);
  if (e != 0) return pa::set_cuda_error("pa_reshape_and_cache: launch", e);
  return PA_OK;
}

pa_status pa_reshape_and_cache_fp8(const void* k_new, const void* v_new, void* k_cache,
                                   void* v_cache, const int64_t* slot_mapping,
                                   const float* k_scale, const float* v_scale,
                                   int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t block_size, int32_t num_blocks, pa_stream_t stream) {
  if (num_tokens < 0 || num_kv_heads < 1 || num_blocks < 1)
    return pa::set_error(PA_ERR_INVALID_ARG,
                         "pa_reshape_and_cache_fp8: num_tokens >= 0, num_kv_heads >= 1, "
                         "num_blocks >= 1");
  if (!pa::block_size_ok(block_size))
    return pa::set_error(PA_ERR_UNSUPPORTED, "pa_reshape_and_cache_fp8: block_size 8, 16 or 32");
  if (head_dim < 8 || head_dim % 8 != 0 || head_dim > 1024)
    return pa::set_error(PA_ERR_UNSUPPORTED,
                         "pa_reshape_and_cache_fp8: head_dim must be a multiple of 8 in [8, 1024]");
  if (num_tokens == 0) return PA_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping || !k_scale || !v_scale)
    return pa::set_error(PA_ERR_INVALID_ARG, "pa_reshape_and_cache_fp8: a required pointer is NULL");
  if (!pa::aligned16(k_new) || !pa::aligned16(v_new) || !pa::aligned16(k_cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) ||
      (reinterpret_cast<uintptr_t>(k_scale) & 3u) || (reinterpret_cast<uintptr_t>(v_scale) & 3u))
    return pa::set_error(PA_ERR_INVALID_ARG, "pa_reshape_and_cache_fp8: misaligned pointer");
  if (int64_t(num_tokens) * num_kv_heads * (head_dim / 8) > (int64_t(1) << 38))
    return pa::set_error(PA_ERR_INVALID_ARG, "pa_reshape_and_cache_fp8: too many tokens");
  const int e = pa::launch_reshape_and_cache_fp8(k_new, v_new, k_cache, v_cache, slot_mapping,
                                                 k_scale, v_scale, num_tokens, num_kv_heads,
                                                 head_dim, block_size, num_blocks, stream);
  if (e != 0) return pa::set_cuda_error("pa_reshape_and_cache_fp8: launch", e);
  return PA_OK;
}

pa_status pa_copy_blocks_fp8(void* k_cache, void* v_cache, const int32_t* pairs,
                             int32_t num_pairs, int32_t num_kv_heads, int32_t head_dim,
                             int32_t block_size, int32_t num_blocks, pa_stream_t stream) {
  if (head_dim % 16 != 0)
    return pa::set_error(PA_ERR_UNSUPPORTED, "pa_copy_blocks_fp8: head_dim must be a multiple of 16");
  if (!pa::block_size_ok(block_size))
    return pa::set_error(PA_ERR_UNSUPPORTED, "pa_copy_blocks_fp8: block_size 8, 16 or 32");
  // one byte per element: the same bytes as a bf16 block of head_dim / 2
  return pa_copy_blocks(k_cache, v_cache, pairs, num_pairs, num_kv_heads, head_dim / 2, block_size,
                        num_blocks, stream);
}

pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int32_t num_pairs,
                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                         int32_t num_blocks, pa_stream_t stream) {
  if (num_pairs < 0 || num_pairs > 65535 || num_kv_heads < 1 || num_blocks < 1)
    return pa::set_error(PA_ERR_INVALID_ARG,
                         "pa_copy_blocks: num_pairs in [0, 65535], num_kv_heads >= 1, num_blocks >= 1");
  if (!pa::block_size_ok(block_size))
    return pa::set_error(PA_ERR_UNSUPPORTED, "pa_copy_blocks: block_size must be 8, 16 or 32");
  if (head_dim < 8 || head_dim % 8 != 0 || head_dim > 1024)
    return pa::set_error(PA_ERR_UNSUPPORTED,
                         "pa_copy_blocks: head_dim must be a multiple of 8 in [8, 1024]");
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !pairs)
    return pa::set_error(PA_ERR_INVALID_ARG, "pa_copy_blocks: a required pointer is NULL");
  if (!pa::aligned16(k_cache) || !pa::aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(pairs) & 3u))
    return pa::set_error(PA_ERR_INVALID_ARG, "pa_copy_blocks: misaligned pointer");
  const int e = pa::launch_copy_blocks(k_cache, v_cache, pairs, num_pairs, num_kv_heads, head_dim,
                                       block_size, num_blocks, stream);
  if (e != 0) return pa::set_cuda_error("pa_copy_blocks: launch", e);
  return PA_OK;
}

}  // extern "C"
