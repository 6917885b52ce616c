/*
 * pagedkv.h -- C ABI of libpagedkv.so: paged KV-cache decode attention for
 * GB300 (sm_103a), its companion cache kernels, and a host-side block pool.
 *
 * Sources for what each call computes:
 *  [P1] "How Paged Attention and Continuous Batching Actually Work"
 *       (netraruntime.com): §Paged attention: virtual memory for the KV cache
 *       (16-token blocks, free list, block table, the indexing rule: divide
 *       for the logical block, look up the physical block, multiply out, add
 *       the offset); §One step, end to end (write KV through the slot
 *       mapping, allocate_slots).
 *  [P2] "Paged Attention as a Memory Manager" (praveentn.live): §How the
 *       Kernel Executes Paged Attention (score_i = q.k_i / sqrt(d_k), the
 *       per-block loop: read the table entry, load the block, dot products,
 *       mask padding, running max and sum, weighted sum of V); §Prefix
 *       Caching and Copy-on-Write (refcounts; allocate, copy, decrement,
 *       update the table).
 *  [P3] PagedAttention architecture walk-through (aicassindra.com):
 *       §The architecture: every piece explained (entry i of the block table
 *       backs tokens [16i, 16i+15]; every 16th token takes a fresh block;
 *       a write to a shared block triggers copy-on-write).
 *  [P4] "PagedAttention and continuous batching" (ai-knowledge-tree):
 *       §Block table example; §Attention kernel modification (K/V loaded
 *       block by block through the table, running softmax across blocks).
 *
 * Data layout (the pages fix none; this library's choice):
 *   k_cache, v_cache  bf16 [num_blocks][num_kv_heads][block_size][head_dim]
 *                     (one (block, KV head) tile is block_size*head_dim*2
 *                     contiguous bytes: 4 KiB at block 16, head dim 128)
 *   q, out            bf16 [num_seqs][num_q_heads][head_dim]
 *   block_tables      int32 [num_seqs][max_blocks_per_seq]; entry j of row b
 *                     is the physical block of logical tokens
 *                     [j*block_size, (j+1)*block_size); entries past
 *                     ceil(len/block_size) are never read
 *   context_lens      int32 [num_seqs], the number of cached tokens of each
 *                     sequence including the one written this step
 *   slot_mapping      int64 [num_tokens]; slot = block*block_size + offset
 *   GQA               query head h reads KV head h / (num_q_heads/num_kv_heads)
 *
 * Conventions for every device call:
 *  - All array pointers are caller-owned DEVICE memory, 16-byte aligned,
 *    dense (no strides). The library never allocates device memory and never
 *    synchronises the stream (except pa_device_errors).
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and runs asynchronously.
 *  - Arguments are validated on the host before anything is launched; a
 *    failing check returns PA_ERR_INVALID_ARG or PA_ERR_UNSUPPORTED and
 *    launches nothing. A launch failure returns PA_ERR_CUDA.
 *  - Values that live only on the device (table entries, lengths, slots) are
 *    checked inside the kernels: an out-of-range value is never dereferenced
 *    (the access is clamped or skipped), a sticky device error bit is set,
 *    and the affected output is unspecified. pa_device_errors() reads the
 *    bits. No kernel faults or hangs on bad device-side values.
 *  - pa_last_error() returns a thread-local message for the last failing
 *    call on that thread.
 *
 * Supported shapes: block_size 8, 16 or 32 ("Paged Attention as a Memory
 * Manager", §PagedAttention: a compile-time constant, typically 8, 16 or 32);
 * head_dim 64 or 128; num_q_heads / num_kv_heads in {1, 2, 4, 8}. Both decode
 * kernels take every block size (the tensor-core kernel's 8-bit cache: head_dim
 * 128 and block size 16 or 32; the 8-bit cache at block size 8 decodes on the
 * CUDA-core kernel). Anything else returns PA_ERR_UNSUPPORTED.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pa_stream_t; /* same type as cudaStream_t */

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,  /* a host-checkable argument is wrong */
  PA_ERR_UNSUPPORTED = 2,  /* valid, but a shape this build does not implement */
  PA_ERR_OOM = 3,          /* block pool exhausted; pool state unchanged */
  PA_ERR_REFCOUNT = 4,     /* refcount underflow / block not allocated */
  PA_ERR_BOUNDS = 5,       /* an id or index out of range */
  PA_ERR_CUDA = 6          /* a CUDA runtime call or launch failed */
} pa_status;

/* Device error bits reported by pa_device_errors(). */
#define PA_DEVERR_TABLE_ENTRY 0x1u   /* block table entry outside [0, num_blocks) */
#define PA_DEVERR_CONTEXT_LEN 0x2u   /* context_len > max_context_len or > table capacity */
#define PA_DEVERR_SLOT 0x4u          /* slot_mapping entry >= num_blocks*block_size */
#define PA_DEVERR_COPY_PAIR 0x8u     /* copy_blocks pair outside [0, num_blocks) */
#define PA_DEVERR_TIMEOUT 0x10u      /* an mbarrier wait hit its iteration limit */
#define PA_DEVERR_APPEND_SLOT 0x20u  /* pa_append_decode: a slot_mapping entry is not the slot
                                        of its token (context_lens[b]-1 for one new token per
                                        sequence); that token is not written */

const char* pa_status_string(pa_status s);
const char* pa_last_error(void);
int32_t pa_version(void);

/* Sticky device error bits accumulated by every kernel of this library on the
 * current device since the last call. Synchronises `stream`, returns the bits
 * in *flags and clears them. */
pa_status pa_device_errors(pa_stream_t stream, uint32_t* flags);

/* ------------------------------------------------------------------------
 * pa_decode -- paged decode attention [P2 §How the Kernel Executes Paged
 * Attention; P4 §Attention kernel modification].
 *
 * For every sequence b and query head h (KV head g = h / G):
 *   K_b, V_b = rows t = 0..L_b-1 of the cache, row t read from physical block
 *              block_tables[b][t / block_size] at offset t % block_size [P1]
 *   s_t      = scale * (q[b][h] . K_b[t])
 *   out[b][h]= sum_t softmax(s)_t * V_b[t]                (bf16, round to nearest even)
 * computed with fp32 accumulation and a running (online) softmax. Sequences
 * longer than `partition_tokens` are split into partitions of that many
 * tokens; each partition yields (max, sum, weighted sum) and a second kernel
 * merges them by log-sum-exp (flash-decoding split; not on the pages).
 * Rows with L_b <= 0 are written as zeros.
 * ---------------------------------------------------------------------- */
typedef struct {
  const void* q;               /* bf16 [num_seqs][num_q_heads][head_dim] */
  void* out;                   /* bf16 [num_seqs][num_q_heads][head_dim] */
  const void* k_cache;         /* bf16 [num_blocks][num_kv_heads][block_size][head_dim] */
  const void* v_cache;         /* same layout as k_cache */
  const int32_t* block_tables; /* int32 [num_seqs][max_blocks_per_seq] */
  const int32_t* context_lens; /* int32 [num_seqs] */
  int32_t max_blocks_per_seq;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t block_size;
  int32_t num_blocks;
  int32_t max_context_len;     /* host-known upper bound of every context_lens[b] (>= 1) */
  float scale;                 /* softmax scale, normally 1/sqrt(head_dim) */
  int32_t partition_tokens;    /* split-K partition length; 0 = 512; else a multiple of 16 in
                                  [16, 4096], and on the CUDA-core kernel of block_size too */
  int32_t variant;             /* PA_DECODE_TENSOR_CORE (default) or PA_DECODE_CUDA_CORE */
  int32_t overlap_prologue;    /* nonzero: context_lens and block_tables were final before the
                                  previous kernel on `stream` began (e.g. uploaded once per step),
                                  so the tensor-core kernel may read them -- and plan its work --
                                  while that kernel still runs (programmatic dependent launch).
                                  q, the caches and every output are read or written only after
                                  the previous kernel has completed; before that the kernel only
                                  prefetches its first cache blocks into L2, which cannot change
                                  any result even if that kernel writes them. 0 = plain stream
                                  order. */
  int32_t kv_dtype;            /* PA_KV_BF16 (0, default) or PA_KV_FP8_E4M3 (1) */
  const float* k_scale;        /* PA_KV_FP8_E4M3 only: device float [num_kv_heads], the
                                  dequantisation scale of each KV head's K (value = code * scale) */
  const float* v_scale;        /* the same for V */
  int32_t query_len;           /* new tokens per sequence: 0 or 1 = one (the layouts above).
                                  Q > 1 ("How Paged Attention and Continuous Batching Actually
                                  Work", §Continuous batching: several scheduled tokens of one
                                  request, as in a chunked prefill): q and out are
                                  [num_seqs][Q][num_q_heads][head_dim], the new tokens are the
                                  last Q of each sequence's context_lens[b] (already in the cache),
                                  and query token i attends to the first context_lens[b] - Q + i + 1
                                  of them (causal among the new tokens). On the tensor-core
                                  variant with the bf16 cache, head_dim 128, block size 16 or 32
                                  and G in {1, 2, 4, 8}, a query-major kernel takes the new tokens
                                  when they are more than one column group holds (below), or
                                  when Q * G >= 16 and num_seqs * num_kv_heads * ceil(Q * G /
                                  128) >= 128: the query rows of one or two KV heads share each
                                  load of their keys; batches with fewer than 256 such units
                                  split each unit's keys over CTAs and merge the partials
                                  (workspace: pa_decode_workspace_size). Otherwise the
                                  tensor-core kernel's MMAs take the query tokens in column
                                  groups: G * Qp <= 16 columns per KV head (8 at block size 8,
                                  Qp = the group's tokens rounded up to a power of two) and
                                  num_kv_heads * G * Qp <= 128 (64 for the 8-bit cache); a
                                  sequence with more new tokens is decoded as several groups,
                                  each streaming the keys its last token sees, with num_seqs *
                                  groups <= 16384. Shapes beyond that (or with num_kv_heads
                                  other than 1, 2, 4 and 8), and the CUDA-core variant, need
                                  num_seqs * Q <= 65535 (else PA_ERR_UNSUPPORTED), also where
                                  the query-major kernel takes them; off that kernel they decode
                                  each (sequence, token) on its own. A sequence
                                  with 0 < context_lens[b] < Q gets zero rows and
                                  PA_DEVERR_CONTEXT_LEN. */
  int32_t wait_timeout_us;     /* tensor-core kernel: the longest one of its barrier waits may
                                  take, in microseconds; 0 = 2 s. A wait that runs out sets
                                  PA_DEVERR_TIMEOUT, and every CTA that saw it stops, lets the
                                  copies it has in flight land, frees its tensor memory and
                                  exits: the outputs are then unspecified, the context stays
                                  usable. A budget far below a launch's normal waits makes a
                                  well-formed launch run out (what the tests do to exercise that
                                  exit). Must be >= 0. */
} pa_decode_params;

/* Decode kernel variants; both compute the same function. The tensor-core
 * kernel handles num_kv_heads in {1, 2, 4, 8}, num_q_heads <= 64 and up to
 * 16384 sequences per call; other shapes run on the CUDA-core kernel
 * whatever `variant` says. */
/* Cache element types. PA_KV_FP8_E4M3 -- the 8-bit KV cache ("PagedAttention"
 * glossary page, §What paging costs: 8-bit KV quantisation halves the bytes per
 * block; the format is this library's reading): OCP E4M3 codes (uint8) with one
 * dequantisation scale per KV head for K and for V.
 *   k_cache  uint8 [num_blocks][num_kv_heads][block_size][head_dim]
 *   v_cache  uint8 [num_blocks][num_kv_heads][block_size/W][head_dim][W],
 *            W = min(block_size, 16) (V^T of each (block, head) tile in
 *            sub-tiles of W keys)
 * Written by pa_reshape_and_cache_fp8, copied by pa_copy_blocks_fp8. The decode
 * computes on the tensor cores (variant PA_DECODE_TENSOR_CORE, head_dim 128 and
 * the rest of the tensor-core shape rules) with the queries and the softmax
 * weights each split into two E4M3 terms, or on CUDA cores (variant
 * PA_DECODE_CUDA_CORE and shapes the tensor-core kernel does not take: head_dim
 * 64, block size 8) with the codes dequantised in fp32; either result is
 * within the bf16 tolerance of the exact decode over the dequantised cache.
 * Other shapes return PA_ERR_UNSUPPORTED. */
#define PA_KV_BF16 0
#define PA_KV_FP8_E4M3 1

#define PA_DECODE_TENSOR_CORE 0 /* tcgen05 MMAs, TMEM accumulators, tensor-map TMA ring */
#define PA_DECODE_CUDA_CORE 1   /* fp32 FMAs on CUDA cores, 1-D bulk-copy rings */

/* Bytes of device workspace pa_decode needs for these parameters on the
 * current device: a 256-byte header, then what the kernel these parameters
 * select needs -- the tensor-core kernel's work plan and per-(sequence + SM)
 * partials of every query column (variant PA_DECODE_TENSOR_CORE on a shape it
 * handles), else the CUDA-core kernel's per-partition partials (none when no
 * sequence can split). Returns 0 for invalid params. */
size_t pa_decode_workspace_size(const pa_decode_params* p);

/* Enqueue the decode. `workspace` is caller-owned device memory of at least
 * pa_decode_workspace_size(p) bytes, 256-byte aligned. Every call writes what
 * it later reads there, so its contents on entry do not matter; two calls in
 * flight at once must not share it. */
pa_status pa_decode(const pa_decode_params* p, void* workspace, size_t workspace_bytes,
                    pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_decode_noalloc -- the same decode as pa_decode, for callers that cannot
 * allocate device memory at decode time. The pages have no counterpart: it
 * exists because an engine that hands all free HBM to its KV block pool at
 * start-up has nothing left for a workspace, and a serving loop cannot take
 * cudaMalloc's implicit device synchronisation.
 *
 * The split-K partials go to a fixed device array inside the library
 * (PA_NOALLOC_SCRATCH_BYTES, held on every GPU that loads the library until
 * the process exits). Nothing is allocated or freed by the call.
 *  - Shapes whose workspace (pa_decode_workspace_size, which sizes the
 *    kernel the parameters select) exceeds that are rejected with
 *    PA_ERR_INVALID_ARG.
 *  - The first call in each CUDA context looks up the array's device address
 *    with that context's device current; make that first call before any
 *    stream capture. A device reset (cudaDeviceReset) or another context on
 *    the same device is a new context, and its first call looks the address
 *    up again.
 *  - Every call on a device shares the one array and leaves its partials in
 *    it. Calls whose kernels overlap on the GPU (different streams, no
 *    ordering between them) race on it and give unspecified results.
 * ---------------------------------------------------------------------- */
#define PA_NOALLOC_SCRATCH_BYTES (16u << 20) /* 16 MiB */
pa_status pa_decode_noalloc(const pa_decode_params* p, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_reshape_and_cache -- write each new token's K/V row into its slot
 * [P1 §One step, end to end: "gather and write KV through the slot-mapping
 * formula"; P3 §The architecture: the forward pass appends the new token's
 * K/V into the right physical block].
 *   for t in [0, num_tokens): slot = slot_mapping[t]; if slot < 0: skip
 *     k_cache[slot / block_size][h][slot % block_size][:] = k_new[t][h][:]  (every KV head h)
 *     v_cache[...]                                         = v_new[t][h][:]
 * Bit-exact copies. k_new/v_new: bf16 [num_tokens][num_kv_heads][head_dim].
 * Two tokens with the same slot race (unspecified which one lands).
 * ---------------------------------------------------------------------- */
pa_status pa_reshape_and_cache(const void* k_new, const void* v_new, void* k_cache,
                               void* v_cache, const int64_t* slot_mapping, int32_t num_tokens,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               int32_t num_blocks, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_append_decode -- one decode step's KV write and attention in one
 * launch: the effect of
 *   pa_reshape_and_cache(a->k_new, a->v_new, k_cache, v_cache,
 *                        a->slot_mapping, num_seqs, ...)
 *   pa_decode(p, ...)
 * [P1 §One step, end to end: the forward pass writes the new token's KV
 * through the slot mapping, then attention reads the paged cache].
 * Token b is sequence b's new token: k_new/v_new are bf16
 * [num_seqs][num_kv_heads][head_dim], slot_mapping is int64 [num_seqs], and
 * p->context_lens already counts the new token. The write of sequence b is
 * done by the part of the decode that reads b's last block, just before that
 * block is loaded, so
 *  - slot_mapping[b] must be the slot of token context_lens[b]-1 of b, i.e.
 *    block_tables[b][(L-1)/16]*16 + (L-1)%16. Any other non-negative value
 *    sets PA_DEVERR_APPEND_SLOT and is not written; a negative value writes
 *    nothing (padding); sequences of length 0 write nothing.
 *  - the written block must not be read by another sequence of the batch,
 *    which copy-on-write guarantees (a shared block is copied before a write).
 *  - with query_len Q > 1 every sequence brings Q new tokens (rows b*Q + i of
 *    k_new/v_new/slot_mapping, token L-Q+i); each is written by the part of
 *    the decode that reads its block, with the same slot rule.
 * a->k_cache / a->v_cache must equal p->k_cache / p->v_cache (the caches are
 * written through these). With the 8-bit cache (p->kv_dtype PA_KV_FP8_E4M3)
 * the write is that of pa_reshape_and_cache_fp8 with p->k_scale / p->v_scale
 * (bit-identical codes). Same workspace as pa_decode. The CUDA-core variant
 * and shapes the tensor-core kernel does not cover run the KV-write kernel
 * and then the decode, with the same result.
 * ---------------------------------------------------------------------- */
typedef struct {
  const void* k_new;            /* bf16 [num_seqs * Q][num_kv_heads][head_dim], 16-byte aligned
                                   (Q = the decode's query_len, at least 1); row b * Q + i is
                                   token context_lens[b] - Q + i of sequence b */
  const void* v_new;            /* same */
  const int64_t* slot_mapping;  /* int64 [num_seqs * Q], the slots of those tokens */
  void* k_cache;                /* == p->k_cache, written */
  void* v_cache;                /* == p->v_cache, written */
} pa_append_params;
pa_status pa_append_decode(const pa_decode_params* p, const pa_append_params* a, void* workspace,
                           size_t workspace_bytes, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_step_host -- one whole decode step driven from host memory, for a host
 * that builds each step's batch (the scheduler of [P1 §One step, end to
 * end]) and reads the result back: copy-on-write copies, the KV write of
 * one new token per sequence and paged decode attention, with the inputs
 * taken from one packed host buffer and the output returned to host memory.
 *
 * The call enqueues on `stream`
 *   1. the staging of the packed inputs into the workspace,
 *   2. pa_copy_blocks (pa_copy_blocks_fp8 for the 8-bit cache; if
 *      num_cow_pairs > 0), then pa_append_decode on the staged inputs and the
 *      device-resident caches (bf16, or 8-bit with kv_dtype and the scales),
 *   3. the return of the output to host_out,
 * and synchronises the stream before it returns (the output is in host_out).
 * Pinned host memory (page-locked through CUDA, hence mapped under unified
 * addressing) that is 16-byte aligned is read and written by the kernels
 * themselves over the host link (NVLink-C2C on a Grace-Blackwell part): a
 * staging kernel copies host_in into the workspace, the tensor-core decode
 * reads the lengths and tables in host_in to plan its work while that kernel
 * runs, and the decode writes its output rows straight into host_out. Any
 * other host memory goes through one DMA copy each way (cudaMemcpyAsync).
 * The bytes moved are the same. host_in must not change until the call
 * returns.
 *
 * Packed input (host memory; pinned memory lets the copy run at full speed):
 * sections at the byte offsets pa_step_host_layout reports, each 256-byte
 * aligned, in this order:
 *   q             bf16  [num_seqs][num_q_heads][head_dim]     (x Q: see query_len)
 *   k_new, v_new  bf16  [num_seqs][num_kv_heads][head_dim]    (x Q)
 *   slot_mapping  int64 [num_seqs]          (x Q; rules of pa_append_decode)
 *   block_tables  int32 [num_seqs][max_blocks_per_seq]
 *   context_lens  int32 [num_seqs]          (counting the new token)
 *   cow_pairs     int32 [num_cow_pairs][2]  (rules of pa_copy_blocks)
 * host_out: bf16 [num_seqs][num_q_heads][head_dim], host memory.
 * The workspace (device memory, 256-byte aligned, at least
 * pa_step_host_workspace_size bytes) holds the staged inputs, the staged
 * output and the decode workspace; nothing in it needs initialising.
 * Errors: host-checkable arguments as pa_decode (no copy is issued);
 * PA_ERR_CUDA when a copy, a launch or the synchronisation fails.
 * ---------------------------------------------------------------------- */
typedef struct {
  uint64_t q, k_new, v_new, slot_mapping, block_tables, context_lens, cow_pairs;
  uint64_t total;  /* bytes of the whole packed input */
} pa_step_layout;

typedef struct {
  const void* host_in;        /* packed inputs (see above) */
  void* host_out;             /* bf16 [num_seqs][num_q_heads][head_dim] */
  void* k_cache;              /* device caches, layout of pa_decode; written */
  void* v_cache;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t block_size;
  int32_t num_blocks;
  int32_t max_blocks_per_seq;
  int32_t max_context_len;    /* host-known upper bound of every context length */
  int32_t num_cow_pairs;
  float scale;
  int32_t variant;            /* PA_DECODE_TENSOR_CORE or PA_DECODE_CUDA_CORE */
  int32_t kv_dtype;           /* PA_KV_BF16 (0) or PA_KV_FP8_E4M3: the caches as in pa_decode;
                                 the 8-bit cache takes the tensor-core variant, the quantising
                                 KV write and pa_copy_blocks_fp8 */
  const float* k_scale;       /* PA_KV_FP8_E4M3 only: device float [num_kv_heads], as in
                                 pa_decode_params */
  const float* v_scale;
  int32_t query_len;          /* new tokens per sequence, Q (0 or 1 = one): q and host_out hold
                                 [num_seqs][Q][num_q_heads][head_dim], k_new / v_new
                                 [num_seqs * Q][num_kv_heads][head_dim], slot_mapping
                                 [num_seqs * Q]; row b * Q + i is token context_lens[b] - Q + i
                                 (as in pa_append_decode) */
} pa_step_host_params;

pa_status pa_step_host_layout(const pa_step_host_params* p, pa_step_layout* out);
size_t pa_step_host_workspace_size(const pa_step_host_params* p); /* 0 if p is invalid */
pa_status pa_step_host(const pa_step_host_params* p, void* workspace, size_t workspace_bytes,
                       pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_reshape_and_cache_fp8 -- the KV write into an 8-bit (PA_KV_FP8_E4M3)
 * cache: for token t and KV head h,
 *   code = E4M3(float32(x) / scale[h])   (round to nearest even; finite values
 *                                         beyond +-448 saturate)
 * K codes go to row (slot / block_size, h, slot % block_size); the V code of
 * offset o = slot % block_size, element d, to byte d*16 + o%16 of sub-tile
 * o/16 of the (block, h) tile. k_scale, v_scale: device float
 * [num_kv_heads]. Otherwise as pa_reshape_and_cache (negative slots skipped,
 * out-of-range slots set PA_DEVERR_SLOT). head_dim a multiple of 8; block_size
 * 16 or 32.
 * ---------------------------------------------------------------------- */
pa_status pa_reshape_and_cache_fp8(const void* k_new, const void* v_new, void* k_cache,
                                   void* v_cache, const int64_t* slot_mapping,
                                   const float* k_scale, const float* v_scale,
                                   int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t block_size, int32_t num_blocks, pa_stream_t stream);

/* pa_copy_blocks for an 8-bit cache: the same whole-block copy of both caches
 * (block_size * head_dim bytes per KV head); block_size 16 or 32. */
pa_status pa_copy_blocks_fp8(void* k_cache, void* v_cache, const int32_t* pairs,
                             int32_t num_pairs, int32_t num_kv_heads, int32_t head_dim,
                             int32_t block_size, int32_t num_blocks, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * pa_copy_blocks -- the data half of copy-on-write [P2 §Prefix Caching and
 * Copy-on-Write: "allocates a fresh physical block, copies the existing
 * content"]. For each pair i: block pairs[i][1] of both caches becomes a
 * bit-exact copy of block pairs[i][0] (all KV heads, all slots).
 * pairs: int32 [num_pairs][2] (src, dst), device memory. Destinations must
 * be pairwise distinct and disjoint from the sources (what the pool's
 * copy-on-write produces); overlapping pairs give unspecified contents.
 * ---------------------------------------------------------------------- */
pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int32_t num_pairs,
                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                         int32_t num_blocks, pa_stream_t stream);

/* ------------------------------------------------------------------------
 * Host block pool [P1 §Paged attention; P2 §Prefix Caching and Copy-on-Write;
 * P3 §The architecture]. All memory here is host memory owned by the pool.
 * Not thread-safe: one pool per thread, or external locking.
 *
 * Free list: a stack. free_order[0] (or block 0 when free_order is NULL) is
 * handed out first; a block whose refcount drops to zero is pushed on top
 * and handed out next (blocks of the prefix cache, below, excepted). Every
 * failing call leaves the pool unchanged. free_blocks in the stats counts
 * every block that can be handed out, evictable cached blocks included.
 * ---------------------------------------------------------------------- */
typedef struct pa_pool pa_pool;

typedef struct {
  int32_t num_blocks;
  int32_t block_size;
  int32_t free_blocks;
  int32_t used_blocks;   /* refcount >= 1 */
  int32_t shared_blocks; /* refcount >= 2 */
  int32_t max_refcount;
  int32_t live_seqs;
} pa_pool_stats_t;

/* free_order: host int32 [num_blocks], a permutation of 0..num_blocks-1, or NULL. */
pa_status pa_pool_create(int32_t num_blocks, int32_t block_size, const int32_t* free_order,
                         pa_pool** out);
void pa_pool_destroy(pa_pool* pool);
/* Pop one block (refcount 1). PA_ERR_OOM when empty. */
pa_status pa_pool_alloc(pa_pool* pool, int32_t* block);
pa_status pa_pool_incref(pa_pool* pool, int32_t block);
/* Refcount - 1; pushed back on the free list at 0. PA_ERR_REFCOUNT if not allocated. */
pa_status pa_pool_decref(pa_pool* pool, int32_t block);
/* Refcount of `block` (0 = free), or -1 for an out-of-range id. */
int32_t pa_pool_refcount(const pa_pool* pool, int32_t block);
pa_status pa_pool_stats(const pa_pool* pool, pa_pool_stats_t* stats);

/* Sequences: each owns a block table and a length. */
pa_status pa_seq_create(pa_pool* pool, int32_t* seq);
/* Release every block of the sequence (in logical order) and retire the id. */
pa_status pa_seq_free(pa_pool* pool, int32_t seq);
/* New sequence sharing the parent's first ceil(num_tokens/block_size) blocks
 * (each refcount + 1), length num_tokens <= parent length. */
pa_status pa_seq_fork(pa_pool* pool, int32_t parent, int32_t num_tokens, int32_t* child);
/* Reserve the slot of the sequence's next token (allocate_slots for one
 * token). If the length is a multiple of block_size a fresh block is
 * appended to the table. Otherwise, if the target block is shared
 * (refcount > 1), copy-on-write: a fresh block replaces it in this table, the
 * old block's refcount drops by one, and (src, dst) is returned in cow_pair
 * with *has_cow = 1 -- the caller must run pa_copy_blocks on that pair before
 * writing the token. *slot = table[len / bs] * bs + len % bs. */
pa_status pa_seq_append_slot(pa_pool* pool, int32_t seq, int64_t* slot, int32_t cow_pair[2],
                             int32_t* has_cow);
/* Append n tokens; slots (nullable, [n]) and cow_pairs (nullable, [n][2])
 * receive the results, *num_cow (nullable) the number of pairs. All or
 * nothing: on PA_ERR_OOM the pool is unchanged. */
pa_status pa_seq_append_tokens(pa_pool* pool, int32_t seq, int32_t n, int64_t* slots,
                               int32_t* cow_pairs, int32_t* num_cow);
pa_status pa_seq_length(const pa_pool* pool, int32_t seq, int32_t* length);
/* Copy the sequence's table into out[0..cap); *n_blocks = its block count. */
pa_status pa_seq_table(const pa_pool* pool, int32_t seq, int32_t* out, int32_t cap,
                       int32_t* n_blocks);
/* Pack the tables and lengths of seqs[0..n) into host arrays
 * tables[n][max_blocks] (unused entries -1) and lens[n], ready to upload. */
pa_status pa_pool_export(const pa_pool* pool, const int32_t* seqs, int32_t n, int32_t max_blocks,
                         int32_t* tables, int32_t* lens);

/* ------------------------------------------------------------------------
 * Prefix cache [P1 FAQ "Where does prefix caching fit?": blocks are
 * content-hashed and a new request whose prompt hashes to resident blocks
 * points at them; P3 §The architecture: the prefix cache hashes each full
 * block's token ids chained with its prefix hash, a match maps the existing
 * physical block with a bumped refcount and skips its prefill; §End-to-end
 * flow: on completion the shared blocks' refcounts tick down and the
 * preamble stays warm in the cache for the next request].
 *
 * pa_seq_create_prompt creates a sequence holding a prompt of num_tokens
 * token ids (host int32). Its full blocks are looked up in order by the chain
 * key (previous block's key, this block's block_size token ids); the leading
 * run of matches is mapped (refcount + 1) and the rest of the prompt gets
 * fresh blocks, whose full ones are entered in the cache. Matching stops at
 * the first miss. A key match is confirmed on the stored token ids, so a
 * hash collision never maps the wrong block.
 *  *cached_tokens = block_size * (matched blocks): their K/V is already in
 *   the cache; the caller writes only tokens [*cached_tokens, num_tokens).
 *  slots (nullable, [num_tokens]): every token's slot.
 * A block whose refcount drops to zero while it is in the cache stays in it
 * (evictable): pa_pool_alloc and appends hand out never-cached free blocks
 * first and then the least recently freed cached block, which leaves the
 * cache at that moment. A cached block is never written in place: an append
 * into it copies it first (copy-on-write), whatever its refcount. All or
 * nothing: on PA_ERR_OOM the pool is unchanged. Without this call the pool
 * behaves exactly as described above.
 * ---------------------------------------------------------------------- */
pa_status pa_seq_create_prompt(pa_pool* pool, const int32_t* tokens, int32_t num_tokens,
                               int32_t* seq, int32_t* cached_tokens, int64_t* slots);

typedef struct {
  int32_t cached_blocks;     /* blocks in the cache (in use or evictable) */
  int32_t evictable_blocks;  /* cached blocks with refcount 0 (counted as free) */
  int64_t lookups;           /* full prompt blocks looked up */
  int64_t hits;              /* of which mapped from the cache */
} pa_prefix_stats_t;
pa_status pa_pool_prefix_stats(const pa_pool* pool, pa_prefix_stats_t* stats);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
