// Paged decode attention on the 5th-generation tensor cores (sm_103a): the
// kernels and their host-side launch templates. Each including translation
// unit instantiates a share of the instances (pa_decode_tc.cu: bf16 head_dim
// 128 and the shared entry points; pa_decode_tc_d64.cu: bf16 head_dim 64;
// pa_decode_tc_fp8.cu: the 8-bit cache; pa_decode_tc_bs8.cu,
// pa_decode_tc_bs32.cu, pa_decode_tc_bs32_fp8.cu: block sizes 8 and 32), so
// they compile in parallel. Each has its own device error word.
//
// Same result as the CUDA-core kernel ("Paged Attention as a Memory
// Manager", §How the Kernel Executes Paged Attention; "PagedAttention and
// continuous batching", §Attention kernel modification): per (sequence,
// query head), softmax(scale * q.K^T) V over the cached tokens, K/V gathered
// block by block through the block table, a running softmax carried across
// blocks, padding slots of the last block masked.
//
// Data movement. A chunk is one paged block with ALL its KV heads: in the
// [block][kv head][16][d] cache that is 16*Hkv contiguous rows, so K and V
// each arrive as two 128-byte-swizzled tensor-map TMA boxes of 16*Hkv rows
// (16 KiB at Hkv = 8). For Hkv < 8 a chunk takes 8/Hkv blocks so that it
// always has 128 rows: row = (block u, KV head h, key). Large boxes matter:
// one issuing thread per SM keeps HBM busy with 16 KiB boxes, not with the
// 2 KiB a (block, head) tile would give.
//
// Math. The chunk is the M=128 side of two tcgen05 MMAs whose N side is the
// sequence's query columns (padded to 16, 32, 64 or 128):
//   S^T[128 rows][N] = Kchunk . Q^T                 (fp32 in TMEM)
//   O^T[d][N]       += V^Tchunk . P^T                (V read MN-major)
// Columns are grouped by KV head: head g owns GE consecutive columns. With
// one new token per sequence a column is a query head (GE = G, GQA: query
// head n reads KV head n / G). With Q new tokens ("How Paged Attention and
// Continuous Batching Actually Work", §Continuous batching: several scheduled
// tokens of one request) column g*GE + i*G + j is query token i of head
// g*G + j, GE = G * Q rounded up to a power of two, and it sees the keys up to
// its own token (causal among the new tokens). Row r only uses the columns of
// its own KV head, and P^T is block-diagonal (zero unless the column's head
// is r's), so the second MMA sums each column over its own KV head's keys
// only. The unused products are free: the tensor pipe runs at a few percent
// here. Softmax runs on CUDA cores, one thread per row. P^T's layout depends
// on the columns: K-major up to 32 (and at 64 with block size 8), per-head
// [16 keys][16 columns] tiles at 64 (the value product then runs per head and
// P^T takes 4 KiB, which leaves room for a third ring slot), MN-major like V
// at 128. The 8-bit cache splits queries and P into two E4M3 terms each
// (kind::f8f6f4), its queries split by a preparation launch.
//
// Scheduling (stream-K). The blocks of all sequences form one stream,
// measured in cost: a sequence costs its units plus a start charge of a few
// chunks (start_chunks); CTA c takes the c-th contiguous share of the cost.
// Before its dependency wait each CTA prefetches its first blocks into L2,
// so their DRAM latency overlaps the previous launch. A (sequence, CTA) segment that
// holds a whole sequence writes the bf16 output directly; otherwise it writes
// fp32 (max, sum, weighted sum) partials to slot (sequence + CTA), unique
// along the stream, and the merge kernel combines them by log-sum-exp.
//
// Roles: warp 4 produces (TMA into a ring of ST chunk slots; block-table
// windows and the next sequence's length prefetched into registers); warp 5
// issues the MMAs; warps 0-3 run the softmax. S is triple-buffered in TMEM, so
// the scores of chunks c+1 and c+2 and the value product of chunk c run on
// the tensor core while the CUDA cores do chunk c's softmax. O^T accumulates
// in TMEM relative to a per-column reference maximum that is raised (and O^T
// rescaled in place) only when a score exceeds it by more than 2^8. Every
// mbarrier wait is bounded; a wait that runs out sets PA_DEVERR_TIMEOUT and
// the CTA winds down through its named barriers, drains, frees TMEM and exits.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__device__ unsigned int g_tc_errors;

constexpr int ROWS = 128;      // rows of a chunk = MMA M
constexpr int NCONS = 4;       // softmax (consumer) warps 0-3
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int NTHREADS = 6 * 32;
constexpr int kCons = NCONS * 32;
// A chunk's rows come in groups of GB = min(block size, 16) keys of one KV
// head. Its "units" (the stream-K grain) are blocks, or for block size 32 the
// 16-token halves of a block, each with all its KV heads.
template <int BS>
struct Units {
  static constexpr int GB = BS < 16 ? BS : 16;  // rows of one (unit, KV head) group, tokens per unit
  static constexpr int VS = BS / GB;            // units per block (1, or 2 at block size 32)
  static constexpr int GROUPS = ROWS / GB;      // groups per chunk
};
// P^T per 16-key step (bf16, head_dim 128, 64 query columns, a KV head owning
// >= 8 of them, 16 tokens per unit): a 16-key step of the chunk is one (unit,
// KV head), and P is block-diagonal, so the value product runs per step over
// the 16 columns that hold the step's head, from a [16 columns][16 keys] tile
// whose other columns are zero. P takes 4 KiB instead of 16 KiB, which makes
// room for a third 64 KiB ring slot. (At 128 columns it frees no slot, and
// its narrower P stores made the step slower.)
template <int D, int GE, int N, bool F8, int BS>
constexpr bool kDiagP = !F8 && D == 128 && GE >= 8 && N == 64 && Units<BS>::GB == 16;
// P^T MN-major at 128 columns (bf16, head_dim 128, 16 columns per KV head,
// 16 tokens per unit): stored like V -- two 64-column halves of [128 keys]
// [128 bytes], 128B-swizzled -- so that each softmax thread (one key) writes
// its head's 16 columns as two 16-byte stores instead of 16 scattered 2-byte
// ones, and the value product reads P^T as an MN-major B operand.
template <int D, int GE, int N, bool F8, int BS>
constexpr bool kMnP = !F8 && D == 128 && GE == 16 && N == 128 && Units<BS>::GB == 16;
constexpr int kF8Tile = 16;  // keys of one 8-bit V^T sub-tile
// The stream-K plan's cost of a sequence start, in chunks: what an extra
// segment in a CTA costs (its epilogue, its queries, the pipeline
// turn-over), in units of chunk time. Chosen by measurement on GB300 (steps
// in us for the costs given):
//   bf16, one new token, 64-sequence 8B layer: 56.6 / 55.9 / 56.2 (1 / 2 / 3)
//   bf16, two new tokens, same layer: 65.7 / 62.1 / 62.2 (1 / 2 / 3); 60.9 at 4,
//     but the 70B-class batch of 8 is 124.4 at 2 and 124.8 at 3 or 4
//   bf16, four new tokens (128 columns: 32 KiB of queries, one query buffer,
//     64 KiB of partials per split segment), same layer: 94.5 / 88.2 / 87.1
//     (1 / 2 / 3), 85.1 / 81.1 / 82.6 (4 / 6 / 8); 256 sequences:
//     309.8 / 316.7 / 301.5 / 296.6 (3 / 4 / 6 / 8)
//   8-bit (chunks take half as long), same layer: 42.1 / 41.0 / 41.0
//     (1 / 2 / 3), and 256 sequences: 134.7 / 133.7 / 132.2 (4: 132.0, but
//     slower at 64 sequences)
__host__ __device__ constexpr int start_chunks(bool f8, int q_len) {
  return q_len >= 4 ? 6 : f8 ? 3 : 2;
}
constexpr int kMaxDynSmem = 232448;
constexpr float kLog2e = 1.4426950408889634f;
// The softmax reference maximum moves only when a score exceeds it by more
// than this (log2 units, a factor of 256); values of P stay <= 256.
constexpr float kRescaleLog2 = 8.0f;
// Most query columns one KV head owns (G times the new tokens per sequence,
// rounded up to a power of two).
constexpr int kMaxGE = 16;

enum : int { F_FIRST = 1, F_LAST = 2, F_WHOLE = 4, F_END = 8 };

struct __align__(16) ChunkMeta {
  int b;      // virtual sequence (its partial slot is b + blockIdx.x when it spans several CTAs)
  int orow0;  // its first output row: (sequence * query_len + first token of its group) * Hq
  int flags;
  int tok0;   // first token of the chunk
  int L;      // keys the virtual sequence streams (context length, clamped, less the
              // new tokens after its group's last)
  int nblk;   // blocks of the chunk holding cache data (the others read as zeros)
  int qslot;
  int qlen;   // query tokens of its group
};

// F8: the 8-bit (E4M3) cache. K rows are D bytes (one 128-byte atom at
// D = 128); V^T comes as one [D][16 keys] tile per (block, KV head), side by
// side; Q and P are each split into an E4M3 hi and lo term.
template <int D, int N, bool F8 = false, bool DIAG = false>
struct TcCfg {
  static_assert(!DIAG || (!F8 && D == 128 && N == 64), "per-head P tiles");
  static constexpr int HALVES = F8 ? 1 : D / 64;   // 128-byte swizzle atoms per K row
  static constexpr int HALF_BYTES = ROWS * 128;    // [128 rows][64 bf16] or [128 rows][128 e4m3]
  static constexpr int K_BYTES = HALVES * HALF_BYTES;
  static constexpr int VT_TILE = D * kF8Tile;     // F8: one [D][16] V^T sub-tile, bytes
  static constexpr int V_BYTES = F8 ? (ROWS / kF8Tile) * VT_TILE : K_BYTES;
  static constexpr int SLOT_BYTES = K_BYTES + V_BYTES;  // K then V
  static constexpr int QH_BYTES = N * 128;         // [N rows][64 bf16] or [N rows][128 e4m3]
  static constexpr int Q_BYTES = F8 ? 2 * QH_BYTES : HALVES * QH_BYTES;  // F8: hi, lo
  static constexpr int PH_BYTES = N * 128;         // P^T [N rows][64 keys] or [N rows][128 keys]
  // bf16: 128 keys; F8: hi and lo; DIAG: 8 steps of [16 columns][16 keys]
  static constexpr int P_BYTES = DIAG ? (ROWS / 16) * 512 : 2 * PH_BYTES;
  // P buffers. One: a second buffer would let the softmax write P(c) while
  // the value product of c-1 still reads P, but it costs a ring slot, and on
  // GB300 neither cache type ran faster with it (the softmax spends ~180
  // cycles of its ~1400-2400 per chunk waiting for that product).
  static constexpr int PB = 1;
  static constexpr int MISC_BYTES = 4096;
  // Q buffers: two let the next segment's queries load while the current
  // segment runs. One is kept when a second would cost a ring slot (at
  // N = 128, and at N = 64 with per-head P tiles: three slots instead of two).
  static constexpr int ST_CAP = F8 ? 6 : 4;
  static constexpr int FIT_Q2 =
      (kMaxDynSmem - 1024 - 2 * Q_BYTES - PB * P_BYTES - MISC_BYTES) / SLOT_BYTES;
  static constexpr int FIT_Q1 =
      (kMaxDynSmem - 1024 - Q_BYTES - PB * P_BYTES - MISC_BYTES) / SLOT_BYTES;
  static constexpr int QB =
      FIT_Q2 >= 2 && (FIT_Q2 >= ST_CAP || FIT_Q2 >= FIT_Q1) ? 2 : 1;
  static constexpr int ST_FIT =
      (kMaxDynSmem - 1024 - QB * Q_BYTES - PB * P_BYTES - MISC_BYTES) / SLOT_BYTES;
  static constexpr int ST = ST_FIT > ST_CAP ? ST_CAP : ST_FIT;
  static_assert(!F8 || D == 128, "the 8-bit cache is built for head_dim 128");
  static_assert(ST >= 2, "at least a double-buffered ring");
  // the stream-K plan's prefix pre[0 .. B] is built in the still-empty ring
  static_assert(size_t(ST) * SLOT_BYTES >= (size_t(kTcMaxSeqs) + 1) * sizeof(int),
                "the ring holds the plan of the largest batch");
  static constexpr int OFF_RING = 0;
  static constexpr int OFF_Q = ST * SLOT_BYTES;
  static constexpr int OFF_P = OFF_Q + QB * Q_BYTES;
  static constexpr int OFF_MISC = OFF_P + PB * P_BYTES;
  // full[ST] empty[ST] qempty[2] s[3] o[2] p[2] drain
  static constexpr int NBARS = 2 * ST + 10;
  static constexpr int OFF_BARS = OFF_MISC;
  static constexpr int OFF_META = OFF_BARS + (NBARS * 8 + 15) / 16 * 16;
  // red, red2: [groups][128 / groups] (8 groups of 16 columns, or 16 of 8)
  static constexpr int OFF_RED = OFF_META + ST * int(sizeof(ChunkMeta));
  static constexpr int OFF_RED2 = OFF_RED + 128 * 4;
  static constexpr int OFF_ALPHA = OFF_RED2 + 128 * 4;                       // [128] by column
  static constexpr int OFF_LS = OFF_ALPHA + 128 * 4;                         // [128]
  static constexpr int OFF_MS = OFF_LS + 128 * 4;                            // [128]
  static constexpr int OFF_WORDS = OFF_MS + 128 * 4;
  static constexpr int OFF_QALPHA = OFF_WORDS + 64;       // F8: [2 q slots][64] 1/alpha
  static constexpr int OFF_KVSCALE = OFF_QALPHA + 2 * 64 * 4;  // F8: k_scale[8], v_scale[8]
  static constexpr int OFF_COLROW = OFF_KVSCALE + 64;  // [128] output row of each column
  static constexpr int SMEM = OFF_COLROW + 128 * 4 + 1024;  // + alignment slack
  static_assert(OFF_COLROW + 128 * 4 <= OFF_MISC + MISC_BYTES, "misc area");
  static_assert(N <= 128 && (!F8 || N <= 64), "columns");
  static_assert(SMEM <= kMaxDynSmem, "shared memory budget");
  // MMA width: the query heads, twice over for the 8-bit cache (the hi and lo
  // terms of Q and of P side by side, one MMA for both)
  static constexpr int NS = F8 ? 2 * N : N;
  static constexpr int TMEM_COLS = 4 * NS;  // S triple buffer [0, 3NS), O at [3NS, 4NS)
  static constexpr int kSBufs = 3;
  static constexpr uint32_t IDESC_S =
      F8 ? dev::idesc_e4m3_f32(ROWS, NS) : dev::idesc_bf16_f32(ROWS, N, false, false);
  static constexpr uint32_t IDESC_PV =
      F8 ? dev::idesc_e4m3_f32(ROWS, NS) : dev::idesc_bf16_f32(ROWS, N, true, false);
  static constexpr uint32_t IDESC_PV16 = dev::idesc_bf16_f32(ROWS, 16, true, true);  // DIAG
  static constexpr uint32_t IDESC_PV_MN = dev::idesc_bf16_f32(ROWS, N, true, true);  // MN-major P^T
  static constexpr uint32_t CHUNK_TX = SLOT_BYTES;
  static constexpr uint32_t Q_TX = Q_BYTES + (F8 ? N * 4 : 0);  // F8: + 1/alpha per column
};

struct TcParams {
  const int32_t* block_tables;
  const int32_t* context_lens;
  __nv_bfloat16* out;
  float* part_m;    // [segments][Hq]
  float* part_l;    // [segments][Hq]
  float* part_acc;  // [segments][Hq][D]
  int* ws_plan;     // [0] = blocks per CTA, [1 .. B+1] = block prefix of the sequences
  // fused KV append (null k_new: none): token b goes to slot_mapping[b]
  const uint4* k_new;
  const uint4* v_new;
  const int64_t* slot_mapping;
  uint4* k_cache_w;
  uint4* v_cache_w;
  // 8-bit cache: per-KV-head dequantisation scales, and per (sequence, query
  // head) 1/alpha of the split queries ([B][N] floats)
  const float* k_scale;
  const float* v_scale;
  const float* q_inv_alpha;
  // the caches as plain pointers: L2 prefetch of the first blocks
  const unsigned char* k_base;
  const unsigned char* v_base;
  int max_blocks_per_seq, num_kv_heads, num_q_heads, num_blocks, cap, oob_row;
  // virtual sequences: num_seqs = sequences x n_groups; virtual sequence v is
  // column group v % n_groups (q_len tokens of the q_total new ones) of
  // sequence v / n_groups
  int num_seqs, n_groups, q_total;
  int oob_row_v;   // 8-bit cache: first V^T tile past the tensor map
  // (oob_row: the first K/V row past the tensor map -- or, for block size 32,
  // the first (block, head) tile past it)
  int q_rows;      // rows of one sequence's queries in the Q tensor map
  // Column layout: KV head g owns columns [g*GE, (g+1)*GE); column g*GE + r is
  // query token r >> g_log2 (of the column group) of query head g*G + (r & (G-1)),
  // unused when that token index is >= q_len. num_cols = num_kv_heads * GE.
  int num_cols, q_len, g_log2;
  float scale_log2;
  uint64_t wait_ns;  // budget of one barrier wait (2 s unless the caller set another)
};

// Context length of sequence b as the kernel uses it: clamped to the table
// capacity, and 0 (an empty sequence) when it cannot hold the new tokens.
__device__ __forceinline__ int real_len_of(const TcParams& P, int raw) {
  const int L = min(raw, P.cap);
  return L >= P.q_total ? L : 0;
}
// Query tokens of virtual sequence v's column group.
__device__ __forceinline__ int group_tokens(const TcParams& P, int v) {
  const int g = v % P.n_groups;
  return min(P.q_len, P.q_total - g * P.q_len);
}
// Keys virtual sequence v streams: those its group's last token sees (raw:
// the sequence's context_lens entry).
__device__ __forceinline__ int seq_len_of(const TcParams& P, int v, int raw) {
  const int L = real_len_of(P, raw);
  if (L == 0) return 0;
  const int g = v % P.n_groups;
  return L - P.q_total + g * P.q_len + group_tokens(P, v);
}
__device__ __forceinline__ int seq_len(const TcParams& P, int v) {
  return seq_len_of(P, v, P.context_lens[v / P.n_groups]);
}

// Output row of column n within its group's [q_len][Hq] rows, or -1 if the
// column is unused (with one token per sequence: n itself, for n < Hq).
__device__ __forceinline__ int column_row(const TcParams& P, int n, int ge) {
  const int g = n / ge, r = n - g * ge;
  const int i = r >> P.g_log2;
  if (n >= P.num_cols || i >= P.q_len) return -1;
  return i * P.num_q_heads + (g << P.g_log2) + (r & ((1 << P.g_log2) - 1));
}

// Byte offset of P^T[n][key] in the K-major, 128B-swizzled B-operand layout
// (two 64-key atoms of [N rows][128 B]).
template <int N>
__device__ __forceinline__ uint32_t p_offset(int n, int key) {
  const int half = key >> 6, kin = key & 63;
  const int r = n & 7, grp = n >> 3;
  return uint32_t(half * (N * 128) + grp * 1024 + r * 128 + (((kin >> 3) ^ r) << 4) +
                  (kin & 7) * 2);
}

// Byte offset of the E4M3 P^T[n][key] in the K-major, 128B-swizzled B-operand
// layout [N rows][128 keys] (one atom per row).
__device__ __forceinline__ uint32_t p8_offset(int n, int key) {
  const int r = n & 7, grp = n >> 3;
  return uint32_t(grp * 1024 + r * 128 + (((key >> 4) ^ r) << 4) + (key & 15));
}

// Byte offset of the 8 columns [8 cg, 8 cg + 8) of key t in the per-head P^T
// tile of 16-key step kk (columns within the step's 16-column window): the
// B operand MN-major without swizzle, core matrices of 8 keys x 16 bytes (8
// columns), the next 8 keys 128 bytes on, the next 8 columns 256 bytes on.
// A thread (one key) writes its 8 columns as one 16-byte store.
__device__ __forceinline__ uint32_t pdiag_offset(int kk, int cg, int t) {
  return uint32_t(kk * 512 + cg * 256 + (t >> 3) * 128 + (t & 7) * 16);
}

// S^T = Kchunk . Q^T for one chunk (single thread). bf16: D/16 MMAs of K = 16.
// E4M3: D/32 MMAs of K = 32, each over both query terms at once.
template <int D, int N, bool F8>
__device__ __forceinline__ void issue_scores(uint32_t tmem_col, const unsigned char* kv,
                                             const unsigned char* q) {
  using C = TcCfg<D, N, F8>;
  const uint32_t kb = dev::smem_addr(kv);
  const uint32_t qb = dev::smem_addr(q);
  if constexpr (F8) {
    // B = the 2N query rows (hi terms, then lo terms): score columns [0, N)
    // from hi, [N, 2N) from lo, added by the softmax
#pragma unroll
    for (int kk = 0; kk < D / 32; ++kk)
      dev::mma_e4m3(tmem_col, dev::smem_desc(kb + kk * 32, 16, 1024, dev::kSwizzle128B),
                    dev::smem_desc(qb + kk * 32, 16, 1024, dev::kSwizzle128B), C::IDESC_S, kk > 0);
  } else {
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t hf = kk >> 2, off = uint32_t(kk & 3) * 32;
      dev::mma_bf16(tmem_col,
                    dev::smem_desc(kb + hf * C::HALF_BYTES + off, 16, 1024, dev::kSwizzle128B),
                    dev::smem_desc(qb + hf * C::QH_BYTES + off, 16, 1024, dev::kSwizzle128B),
                    C::IDESC_S, kk > 0);
    }
  }
}

// ---------------------------------------------------------------------------
// MMA warp (one thread): per chunk, S^T = K.Q^T into S[chunk & 1] as soon as
// the chunk has landed, and O^T = V^T.P^T once the softmax warps have written
// P for it. Scores run one chunk ahead of the value product.
// ---------------------------------------------------------------------------
template <int D, int GE, int N, bool F8, bool DIAG, bool MNP>
__device__ __forceinline__ void mma_loop(unsigned char* ring, unsigned char* qbuf,
                                         unsigned char* pbuf, uint64_t* full, uint64_t* empty,
                                         uint64_t* qempty, uint64_t* bar_s, uint64_t* bar_o,
                                         uint64_t* bar_p, uint64_t* drain, const ChunkMeta* meta,
                                         uint32_t tmem, volatile int* abort_flag, int H,
                                         uint64_t wait_ns) {
  using C = TcCfg<D, N, F8, DIAG>;
  // D = 64: the second 64-row half of M re-reads the first (LBO 0); those
  // TMEM lanes are never read back.
  const uint32_t lbo = C::HALVES == 2 ? uint32_t(C::HALF_BYTES) : 0u;
  const uint32_t pbs = dev::smem_addr(pbuf);
  // Event loop: issue whichever is ready first -- the scores of the next
  // ring position once its data has landed (at most one position ahead of
  // the value products), or the value product of position c once the softmax
  // warps have written its P. Every ring position before the end sentinel
  // is a real chunk, so position = chunk index.
  int c = 0;           // position whose value product is next
  int s_pos = 0;       // next position to issue scores for
  int end_pos = -1;    // position of the end sentinel, once seen
  bool ok = true;
  uint64_t t_progress = dev::global_timer_ns();
  // Idle polls up to 64 columns spin (the wall clock is read every 256 of
  // them, which bounds the wait): the scores of a landed chunk are issued
  // sooner, steps 0.7-1.6 % shorter on GB300. At 128 columns the softmax warp
  // sharing this warp's sub-partition has more to issue, and a sleep between
  // polls measured faster.
  constexpr bool kSpin = N <= 64;
  uint32_t idle = 0;
  for (;;) {
    bool progress = false;
    // value product first: it frees a ring slot for the producer
    if (c < s_pos && c != end_pos &&
        dev::mbar_test(&bar_p[c % C::PB], uint32_t(c / C::PB) & 1u)) {
      const uint32_t pbc = pbs + uint32_t(c % C::PB) * C::P_BYTES;  // this chunk's P
      const int sl = c % C::ST;
      // O accumulates over a segment's chunks; its first chunk starts afresh
      const int fl = meta[sl].flags, qsl = meta[sl].qslot;  // read before the slot is freed
      const bool fresh = (fl & F_FIRST) != 0;
      dev::tc_fence_after();
      const uint32_t vb = dev::smem_addr(ring + size_t(sl) * C::SLOT_BYTES + C::K_BYTES);
      if constexpr (F8) {
        // V^T K-major without swizzle: 8-row x 16-byte core matrices, the
        // next 8 rows of d 128 B on (SBO), the next 16 keys one [D][16]
        // tile on (LBO); 32 keys per MMA. B = the 2N rows of P (hi terms,
        // then lo terms): O columns [0, N) from hi, [N, 2N) from lo.
#pragma unroll
        for (int kk = 0; kk < ROWS / 32; ++kk)
          dev::mma_e4m3(tmem + C::kSBufs * C::NS,
                        dev::smem_desc(vb + kk * 2 * C::VT_TILE, C::VT_TILE, 128,
                                       dev::kSwizzleNone),
                        dev::smem_desc(pbc + kk * 32, 16, 1024, dev::kSwizzle128B), C::IDESC_PV,
                        kk > 0 || !fresh);
      } else if constexpr (DIAG) {
        // step kk = (unit kk / H, KV head kk % H): O^T columns of the 16-wide
        // window holding that head's columns. With 8 columns per head a
        // window holds two heads; the first step of the pair in a chunk
        // starts it afresh in a segment's first chunk, the second (zero
        // P^T for the first head's columns) adds on.
#pragma unroll
        for (int kk = 0; kk < ROWS / 16; ++kk) {
          const int h = kk % H;
          const bool first = kk < H && (GE >= 16 || (h & 1) == 0);
          dev::mma_bf16(tmem + C::kSBufs * C::NS + uint32_t((h * GE) & ~15),
                        dev::smem_desc(vb + kk * 2048, lbo, 1024, dev::kSwizzle128B),
                        // MN-major, no swizzle: next 8 keys (K) 128 B on, next 8
                        // columns (N) 256 B on
                        dev::smem_desc(pbc + kk * 512, 128, 256, dev::kSwizzleNone),
                        C::IDESC_PV16, !(fresh && first));
        }
      } else if constexpr (MNP) {
        // P^T MN-major, laid out like V: the next 8 keys 1024 B on (SBO), the
        // second 64-column half 16 KiB on (LBO)
#pragma unroll
        for (int kk = 0; kk < ROWS / 16; ++kk) {
          dev::mma_bf16(tmem + C::kSBufs * C::NS,
                        dev::smem_desc(vb + kk * 2048, lbo, 1024, dev::kSwizzle128B),
                        dev::smem_desc(pbc + kk * 2048, 16384, 1024, dev::kSwizzle128B),
                        C::IDESC_PV_MN, kk > 0 || !fresh);
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < ROWS / 16; ++kk) {
          dev::mma_bf16(tmem + C::kSBufs * C::NS,
                        dev::smem_desc(vb + kk * 2048, lbo, 1024, dev::kSwizzle128B),
                        dev::smem_desc(pbc + (kk >> 2) * C::PH_BYTES + (kk & 3) * 32, 16, 1024,
                                       dev::kSwizzle128B),
                        C::IDESC_PV, kk > 0 || !fresh);
        }
      }
      dev::mma_commit(&bar_o[c % C::PB]);
      dev::mma_commit(&empty[sl]);
      // 8-bit cache: the softmax reads the segment's 1/alpha until it has
      // written this chunk's P, so the query slot is released only here
      if constexpr (F8) {
        if (fl & F_LAST) dev::mma_commit(&qempty[qsl]);
      }
      ++c;
      progress = true;
    }
    // scores of the next positions as soon as their data has landed, up to
    // two positions ahead of the value products (S is triple-buffered)
    if (end_pos < 0 && s_pos <= c + 2 &&
        dev::mbar_test(&full[s_pos % C::ST], uint32_t(s_pos / C::ST) & 1u)) {
      const int sl = s_pos % C::ST;
      const ChunkMeta mn = meta[sl];
      if (mn.flags & F_END) {
        end_pos = s_pos;
      } else {
        const int sb = s_pos % C::kSBufs;
        dev::tc_fence_after();
        issue_scores<D, N, F8>(tmem + sb * C::NS, ring + size_t(sl) * C::SLOT_BYTES,
                               qbuf + mn.qslot * C::Q_BYTES);
        dev::mma_commit(&bar_s[sb]);
        if constexpr (!F8) {
          if (mn.flags & F_LAST) dev::mma_commit(&qempty[mn.qslot]);
        }
      }
      ++s_pos;
      progress = true;
    }
    if (c == end_pos) break;
    if (progress) {
      idle = 0;
      if constexpr (!kSpin) t_progress = dev::global_timer_ns();
      continue;
    }
    if constexpr (kSpin) {
      if ((++idle & 255u) != 0u) continue;
      if (*abort_flag) break;
      const uint64_t now = dev::global_timer_ns();
      if (idle == 256u) {
        t_progress = now;  // the idle stretch began about now
      } else if (now - t_progress > wait_ns) {
        ok = false;
        break;
      }
    } else {
      if (*abort_flag) break;
      if (dev::global_timer_ns() - t_progress > wait_ns) {
        ok = false;
        break;
      }
      __nanosleep(20);
    }
  }
  if (!ok) {
    atomicOr(&g_tc_errors, PA_DEVERR_TIMEOUT);
    *abort_flag = 1;
  }
  // every MMA this thread issued completes before TMEM can be released
  dev::mma_commit(drain);
  (void)dev::mbar_wait(drain, 0);
}

// ---------------------------------------------------------------------------
// Softmax warps 0-3: thread = row of the chunk (scores), = head dimension
// (output). Chunk r: read S, running max (half-warp + shared-memory exchange
// across the chunk's groups of the same KV head), fold chunk r-1's O^T into
// the accumulators, write P and signal the MMA warp.
// ---------------------------------------------------------------------------
template <int D, int GE, int N, bool F8, int BS>
struct Softmax {
  using C = TcCfg<D, N, F8, kDiagP<D, GE, N, F8, BS>>;
  static constexpr int GB = Units<BS>::GB;          // rows of one (unit, KV head) group
  static constexpr int GROUPS = Units<BS>::GROUPS;  // groups per chunk
  static constexpr int WG = 32 / GB;                // groups per warp (2, or 4 at GB 8)
  static constexpr int KRED = 128 / GROUPS;         // columns per group in red, red2
  static_assert(GE <= KRED, "columns per KV head");
  // score columns a warp reads: the GE columns of each of its groups' heads
  static constexpr int LDC = WG * GE <= 8 ? 8 : WG * GE;
  // O^T columns per TMEM round trip (the 8-bit epilogue holds a second,
  // lo-term block beside them)
  static constexpr int CW = N <= (F8 ? 32 : 64) ? N : 32;

  __device__ __forceinline__ static void run(const TcParams& P, unsigned char* ring,
                                             unsigned char* pbuf, uint64_t* full,
                                             uint64_t* bar_s, uint64_t* bar_o, uint64_t* bar_p,
                                             const ChunkMeta* meta, float* red, float* red2,
                                             float* alpha_s, float* l_s, float* m_s,
                                             const float* qalpha, const float* kvscale,
                                             const int* colrow, uint32_t tmem,
                                             volatile int* abort_flag, int* consumed_out) {
    const int ctid = threadIdx.x;
    const int cw = ctid >> 5, lane = ctid & 31;
    const int H = P.num_kv_heads;
    const int NC = P.num_cols;
    const int U = GROUPS / H;  // units per chunk
    const int grp = ctid / GB;  // (unit u, KV head h) group of this row
    const int u = grp / H, h = grp - (grp / H) * H;
    const int key = ctid % GB;
    // The warp's groups hold min(H, WG) consecutive heads from h0 (all H of
    // them, repeated, when H < WG); this lane's head is the slice-th of them.
    const int HW = H < WG ? H : WG;
    const int h0 = (WG * cw) % H;
    const int col0 = h0 * GE;
    const int slice = (lane / GB) % HW;
    const uint32_t t_lane = uint32_t(cw * 32) << 16;
    const uint32_t tO = tmem + t_lane + C::kSBufs * C::NS;  // F8: + N for the lo terms

    // Reference maximum per query column (log2 domain) and this row's share of
    // the softmax sum relative to it. O^T accumulates in TMEM relative to the
    // same reference; the reference is raised (and O^T, l rescaled) only when
    // a score exceeds it by more than kRescaleLog2, and only then is the
    // chunk's maximum over its keys taken.
    float m_ref[GE], l_part[GE];
    // 8-bit cache: the segment's score factor per column, kept in registers
    // up to 4 columns per KV head (more spilled)
    constexpr bool kHoistF = F8 && GE <= 4;
    float fq[kHoistF ? GE : 1];
#pragma unroll
    for (int j = 0; j < GE; ++j) {
      m_ref[j] = -INFINITY;
      l_part[j] = 0.0f;
      if constexpr (kHoistF) fq[j] = 0.0f;
    }
    int c = 0;  // ring position = chunk index
    bool ok = true;
    int pv_done = -1;  // highest chunk whose value product is known to be complete
    // wait for chunk k's value product (k > pv_done)
    auto wait_pv = [&](int k) {
      ok = __all_sync(0xffffffffu, dev::mbar_wait(&bar_o[k % C::PB], uint32_t(k / C::PB) & 1u,
                                                   P.wait_ns, abort_flag)) &&
           ok;
      pv_done = k;
    };

    for (;;) {
      const int slot = c % C::ST;
      ok = __all_sync(0xffffffffu, dev::mbar_wait(&full[slot], uint32_t(c / C::ST) & 1u, P.wait_ns,
                                                 abort_flag)) &&
           ok;
      const ChunkMeta m = meta[slot];
      // every exit below is taken by all 128 threads together (named barriers follow)
      if (!dev::named_barrier_and(1, kCons, ok && *abort_flag == 0)) {
        ok = false;
        break;
      }
      if (m.flags & F_END) break;
      const int buf = c % C::kSBufs;
      const bool first = (m.flags & F_FIRST) != 0;

      // ---- scores of this chunk -> registers
      ok = __all_sync(0xffffffffu, dev::mbar_wait(&bar_s[buf], uint32_t(c / C::kSBufs) & 1u,
                                                 P.wait_ns, abort_flag)) &&
           ok;
      dev::tc_fence_after();
      float s[LDC];
      const uint32_t tS = tmem + t_lane + buf * C::NS + col0;
      if constexpr (LDC == 8) {
        dev::tmem_ld8(tS, s);
      } else {
        dev::tmem_ld_cols<LDC>(tS, s);
      }
      if constexpr (F8) {  // + the scores of the lo query terms
        float s2[LDC];
        if constexpr (LDC == 8) {
          dev::tmem_ld8(tS + N, s2);
        } else {
          dev::tmem_ld_cols<LDC>(tS + N, s2);
        }
#pragma unroll
        for (int i = 0; i < LDC; ++i) s[i] += s2[i];
      }

      // ---- scaled scores; row = (block u, head h, key)
      const int t = m.tok0 + u * GB + key;
      const bool row_in = u < m.nblk;           // the row holds cache data
      const bool valid = row_in && t < m.L;     // a token of the sequence
      // Causal limit: column j holds query token i = j >> g_log2 of the
      // group, whose last token (qlen - 1) sees the keys t < L; token i sees
      // t < L - qlen + 1 + i; columns with i >= qlen are unused.
      const int t_rel = t - (m.L - m.qlen + 1);
      float x[GE];
      bool need = false;
#pragma unroll
      for (int j = 0; j < GE; ++j) {
        float sj;
        if constexpr (WG == 2) {
          sj = slice ? s[GE + j] : s[j];
        } else {
          sj = slice == 0 ? s[j] : slice == 1 ? s[GE + j] : slice == 2 ? s[2 * GE + j] : s[3 * GE + j];
        }
        float f = P.scale_log2;
        if constexpr (F8) {  // the head's K scale and the query term's 1/alpha
          if constexpr (kHoistF) {  // taken once per segment
            if (first) fq[j] = f * kvscale[h] * qalpha[m.qslot * 64 + h * GE + j];
            f = fq[j];
          } else {
            f *= kvscale[h] * qalpha[m.qslot * 64 + h * GE + j];
          }
        }
        const int i = j >> P.g_log2;
        x[j] = row_in && t_rel < i && i < m.qlen ? sj * f : -INFINITY;
        need |= x[j] > m_ref[j] + kRescaleLog2;
      }

      // ---- raise the reference where a score exceeds it by more than
      // kRescaleLog2: to the chunk maximum of that column over its KV head's
      // rows (half-warp, then shared memory across the chunk's groups)
      if (dev::named_barrier_or(1, kCons, need)) {
        float cm[GE];
#pragma unroll
        for (int j = 0; j < GE; ++j) {
          float v = x[j];
#pragma unroll
          for (int o = GB / 2; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
          cm[j] = v;
        }
        if (U > 1) {  // the head's rows span several groups of the chunk
          if (key == 0) {
#pragma unroll
            for (int j = 0; j < GE; ++j) red[grp * KRED + j] = cm[j];
          }
          dev::named_barrier(1, kCons);
#pragma unroll
          for (int j = 0; j < GE; ++j) {
            float v = -INFINITY;
            for (int uu = 0; uu < U; ++uu) v = fmaxf(v, red[(uu * H + h) * KRED + j]);
            cm[j] = v;
          }
        }
#pragma unroll
        for (int j = 0; j < GE; ++j) {
          const float nr = cm[j] > m_ref[j] + kRescaleLog2 ? cm[j] : m_ref[j];
          // 1 where unchanged (also for a column that has seen no key yet)
          const float f = nr == m_ref[j] ? 1.0f : dev::fast_exp2(m_ref[j] - nr);
          l_part[j] *= f;
          m_ref[j] = nr;
          if (u == 0 && key == 0) alpha_s[h * GE + j] = f;
        }
        if (!first) {
          // chunk c-1's value product must be in O^T before it is scaled
          if (pv_done < c - 1) wait_pv(c - 1);
          dev::named_barrier(1, kCons);  // every factor is written
          dev::tc_fence_after();
#pragma unroll
          for (int part = 0; part < (F8 ? 2 : 1); ++part) {  // F8: hi and lo columns
#pragma unroll
            for (int cg = 0; cg < N; cg += CW) {
              float o[CW];
              dev::tmem_ld_cols<CW>(tO + part * N + cg, o);
#pragma unroll
              for (int n = 0; n < CW; ++n) o[n] *= alpha_s[cg + n];
              dev::tmem_st_cols<CW>(tO + part * N + cg, o);
            }
          }
        }
      }
      // the value product that last read this P buffer (chunk c - PB) must be done
      if (c - C::PB >= 0 && pv_done < c - C::PB) wait_pv(c - C::PB);
      unsigned char* pcur = pbuf + (c % C::PB) * C::P_BYTES;

      float pd[GE];  // per-head P tiles and 8-bit P: this row's P, stored after the loop
#pragma unroll
      for (int j = 0; j < GE; ++j) {
        // a masked score gives 0 (m_ref may still be -inf for its column)
        const float p = x[j] == -INFINITY ? 0.0f : dev::fast_exp2(x[j] - m_ref[j]);
        if constexpr (F8) {
          pd[j] = p;  // split below, two columns per conversion
        } else if constexpr (kDiagP<D, GE, N, F8, BS> || kMnP<D, GE, N, F8, BS>) {
          l_part[j] += p;
          pd[j] = p;  // stored below, 8 columns per 16-byte store
        } else {
          l_part[j] += p;
          *reinterpret_cast<__nv_bfloat16*>(pcur + p_offset<N>(h * GE + j, ctid)) =
              __float2bfloat16_rn(p);
        }
      }
      if constexpr (F8) {
        // P as two E4M3 terms, hi = E4M3(p) and lo = E4M3(p - hi); the sum
        // uses exactly what the MMA multiplies. Columns go in pairs through
        // the paired conversions (the same codes as one at a time).
#pragma unroll
        for (int j = 0; j < GE; j += 2) {
          if (j + 1 < GE) {
            const uint32_t h2 = dev::to_e4m3x2(pd[j], pd[j + 1]);
            const float2 hf = dev::from_e4m3x2(h2);
            const uint32_t l2 = dev::to_e4m3x2(pd[j] - hf.x, pd[j + 1] - hf.y);
            const float2 lf = dev::from_e4m3x2(l2);
            l_part[j] += hf.x + lf.x;
            l_part[j + 1] += hf.y + lf.y;
            const uint32_t o0 = p8_offset(h * GE + j, ctid), o1 = p8_offset(h * GE + j + 1, ctid);
            pcur[o0] = uint8_t(h2);
            pcur[o1] = uint8_t(h2 >> 8);
            pcur[C::PH_BYTES + o0] = uint8_t(l2);
            pcur[C::PH_BYTES + o1] = uint8_t(l2 >> 8);
          } else {
            const uint8_t ph = dev::to_e4m3(pd[j]);
            const float phf = dev::from_e4m3(ph);
            const uint8_t pl = dev::to_e4m3(pd[j] - phf);
            l_part[j] += phf + dev::from_e4m3(pl);
            const uint32_t o = p8_offset(h * GE + j, ctid);
            pcur[o] = ph;
            pcur[C::PH_BYTES + o] = pl;
          }
        }
      }
      if constexpr (kMnP<D, GE, N, F8, BS>) {
        // columns [16 h, 16 h + 16): 16-byte chunks 2 (h % 4) and 2 (h % 4) + 1
        // of key ctid's 128-byte row in half h / 4, each at its chunk index
        // XOR (ctid % 8) (the 128B swizzle)
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 v2 = __floats2bfloat162_rn(pd[8 * g + 2 * i], pd[8 * g + 2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&v2);
          }
          const int chunk = 2 * (h & 3) + g;
          *reinterpret_cast<uint4*>(pcur + (h >> 2) * 16384 + ctid * 128 +
                                    ((chunk ^ (ctid & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      if constexpr (kDiagP<D, GE, N, F8, BS>) {
        // columns [h GE, h GE + GE) are 8-column groups ((h GE) & 15) / 8 + g
        // of the step's window
#pragma unroll
        for (int g = 0; g < GE / 8; ++g) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 v2 = __floats2bfloat162_rn(pd[8 * g + 2 * i], pd[8 * g + 2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&v2);
          }
          *reinterpret_cast<uint4*>(pcur + pdiag_offset(ctid >> 4, ((h * GE) & 15) / 8 + g,
                                                        ctid & 15)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      // A row past the sequence inside a loaded block (the sequence's last,
      // partial block) may hold anything, NaN included: clear its V row so
      // 0 * V = 0.
      if (!valid && row_in) {
        unsigned char* kv = ring + size_t(slot) * C::SLOT_BYTES;
        if constexpr (F8) {  // row r is column r % 16 of [D][16] V^T sub-tile r / 16
          unsigned char* tile = kv + C::K_BYTES + (ctid / kF8Tile) * C::VT_TILE + ctid % kF8Tile;
#pragma unroll 16
          for (int d = 0; d < D; ++d) tile[d * kF8Tile] = 0;
        } else {
#pragma unroll
          for (int hf = 0; hf < C::HALVES; ++hf) {
            uint4* row =
                reinterpret_cast<uint4*>(kv + C::K_BYTES + hf * C::HALF_BYTES + ctid * 128);
#pragma unroll
            for (int i = 0; i < 8; ++i) row[i] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
      dev::fence_async_smem();
      dev::tc_fence_before();
      dev::mbar_arrive(&bar_p[c % C::PB]);  // P(c) written; S(c) read; O^T rescaled

      if (m.flags & F_LAST) {
        // per query column: softmax denominator over all rows of its KV head
#pragma unroll
        for (int j = 0; j < GE; ++j) {
          float v = l_part[j];
#pragma unroll
          for (int o2 = GB / 2; o2 >= 1; o2 >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o2);
          if (key == 0) red2[grp * KRED + j] = v;
        }
        dev::named_barrier(1, kCons);
        if (u == 0 && key == 0) {
#pragma unroll
          for (int j = 0; j < GE; ++j) {
            float l = 0.0f;
            for (int uu = 0; uu < U; ++uu) l += red2[(uu * H + h) * KRED + j];
            l_s[h * GE + j] = l;
            m_s[h * GE + j] = m_ref[j];
          }
        }
        wait_pv(c);
        dev::tc_fence_after();
        // O^T columns [cg, cg + CW) of this thread's lane (row d = ctid)
        auto load_o = [&](int cg, float (&o)[CW]) {
          dev::tmem_ld_cols<CW>(tO + cg, o);
          if constexpr (F8) {  // hi + lo terms, times the V scale of each column's KV head
#pragma unroll
            for (int c16 = 0; c16 < CW; c16 += 16) {
              float o2[16];
              dev::tmem_ld_cols<16>(tO + N + cg + c16, o2);
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int n = cg + c16 + i;
                o[c16 + i] = (o[c16 + i] + o2[i]) * kvscale[8 + (n < NC ? n / GE : 0)];
              }
            }
          }
        };
        float o[CW];
        load_o(0, o);
        dev::named_barrier(1, kCons);  // l_s, m_s written
        __nv_bfloat16* o_row = P.out + size_t(m.orow0) * D + (ctid < D ? ctid : 0);
        const int seg = m.b + int(blockIdx.x);  // partial slot
        const int row_end = m.qlen * P.num_q_heads;  // rows of the group's tokens
        float* a_row = P.part_acc + size_t(seg) * NC * D + (ctid < D ? ctid : 0);
#pragma unroll
        for (int cg = 0; cg < N; cg += CW) {
          if (cg > 0) load_o(cg, o);
          if (ctid < D) {
            if (m.flags & F_WHOLE) {
#pragma unroll
              for (int i = 0; i < CW; ++i) {
                const int r = colrow[cg + i];
                if (r >= 0 && r < row_end)
                  o_row[size_t(r) * D] = __float2bfloat16_rn(o[i] * __frcp_rn(l_s[cg + i]));
              }
            } else {
#pragma unroll
              for (int i = 0; i < CW; ++i)
                if (cg + i < NC) a_row[size_t(cg + i) * D] = o[i];
            }
          }
        }
        if (!(m.flags & F_WHOLE) && ctid < NC) {
          P.part_m[size_t(seg) * NC + ctid] = m_s[ctid];
          P.part_l[size_t(seg) * NC + ctid] = l_s[ctid];
        }
        dev::tc_fence_before();
#pragma unroll
        for (int j = 0; j < GE; ++j) {
          m_ref[j] = -INFINITY;
          l_part[j] = 0.0f;
        }
      }
      ++c;
    }
    if (!ok && ctid == 0) {
      atomicOr(&g_tc_errors, PA_DEVERR_TIMEOUT);
      *abort_flag = 1;
    }
    if (ctid == 0) *consumed_out = c;
  }
};

template <int D, int GE, int N, bool F8, int BS>
__global__ void __launch_bounds__(NTHREADS, 1)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ CUtensorMap tm_q, const TcParams P) {
  using C = TcCfg<D, N, F8, kDiagP<D, GE, N, F8, BS>>;
  static_assert(!F8 || BS >= 16, "the 8-bit V^T sub-tiles hold 16 keys");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* ring = smem + C::OFF_RING;
  unsigned char* qbuf = smem + C::OFF_Q;
  unsigned char* pbuf = smem + C::OFF_P;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::ST;
  uint64_t* qempty = bars + 2 * C::ST;
  uint64_t* bar_s = bars + 2 * C::ST + 2;  // [3] scores ready
  uint64_t* bar_o = bar_s + 3;              // [2] value product ready (by P buffer)
  uint64_t* bar_p = bar_o + 2;              // [2] P written by all 128 softmax threads
  uint64_t* drain = bar_p + 2;
  ChunkMeta* meta = reinterpret_cast<ChunkMeta*>(smem + C::OFF_META);
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
  float* red2 = reinterpret_cast<float*>(smem + C::OFF_RED2);
  float* alpha_s = reinterpret_cast<float*>(smem + C::OFF_ALPHA);
  float* l_s = reinterpret_cast<float*>(smem + C::OFF_LS);
  float* m_s = reinterpret_cast<float*>(smem + C::OFF_MS);
  int* words = reinterpret_cast<int*>(smem + C::OFF_WORDS);
  float* qalpha = reinterpret_cast<float*>(smem + C::OFF_QALPHA);    // F8
  float* kvscale = reinterpret_cast<float*>(smem + C::OFF_KVSCALE);  // F8
  int* colrow = reinterpret_cast<int*>(smem + C::OFF_COLROW);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&words[0]);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&words[1]);
  int* consumed = &words[2];
  int* issued = &words[3];

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int B = P.num_seqs;
  const int H = P.num_kv_heads;
  constexpr int UT = Units<BS>::GB;  // tokens per unit (the stream-K grain)
  constexpr int VS = Units<BS>::VS;  // units per block

  if (tid == 0) {
    for (int i = 0; i < C::ST; ++i) {
      dev::mbar_init(&full[i], 1);
      dev::mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) dev::mbar_init(&qempty[i], 1);
    for (int i = 0; i < 3; ++i) dev::mbar_init(&bar_s[i], 1);
    for (int i = 0; i < 2; ++i) {
      dev::mbar_init(&bar_o[i], 1);
      dev::mbar_init(&bar_p[i], kCons);
    }
    dev::mbar_init(drain, 1);
    *abort_flag = 0;
    *consumed = 0;
    *issued = 0;
    dev::fence_barrier_init();
  }
  // P^T is block-diagonal: the entries off the diagonal stay zero for good.
  for (int i = tid; i < C::PB * C::P_BYTES / 16; i += NTHREADS)
    reinterpret_cast<uint4*>(pbuf)[i] = make_uint4(0u, 0u, 0u, 0u);

  // ---- stream-K plan (uses the still-empty ring as scratch). The stream is
  // measured in cost: a sequence costs its units plus SC for its start (the
  // epilogue, the new queries and the pipeline turn-over of an extra segment
  // take about one chunk's time), so CTAs that hold several sequence starts
  // get fewer units. pre = exclusive prefix of the costs; CTA c takes the
  // cost range [c R, (c+1) R).
  const int SC = start_chunks(F8, P.q_len) * (Units<BS>::GROUPS / H);  // a sequence start's cost
  // (P.q_len: the tokens of a column group)
  int* pre = reinterpret_cast<int*>(ring);
  {
    const int seg = (B + NTHREADS - 1) / NTHREADS;
    const int b0 = min(B, tid * seg), b1 = min(B, b0 + seg);
    int local = 0;
    for (int b = b0; b < b1; ++b) {
      if (blockIdx.x == 0 && b % P.n_groups == 0) {
        const int L0 = P.context_lens[b / P.n_groups];
        if (L0 > P.cap || (L0 > 0 && L0 < P.q_total)) atomicOr(&g_tc_errors, PA_DEVERR_CONTEXT_LEN);
      }
      const int n = (seq_len(P, b) + UT - 1) / UT;
      local += n > 0 ? n + SC : 0;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) reinterpret_cast<int*>(red)[warp] = incl;
    __syncthreads();
    int run = incl - local;
    for (int w = 0; w < warp; ++w) run += reinterpret_cast<int*>(red)[w];
    for (int b = b0; b < b1; ++b) {
      pre[b] = run;
      const int n = (seq_len(P, b) + UT - 1) / UT;
      run += n > 0 ? n + SC : 0;
    }
    if (tid == NTHREADS - 1) pre[B] = run;
  }
  __syncthreads();
  const int total = pre[B];
  const int R = total > 0 ? (total + int(gridDim.x) - 1) / int(gridDim.x) : 1;
  const int u0 = min(total, int(blockIdx.x) * R);  // this CTA's cost range [u0, u1)
  const int u1 = min(total, u0 + R);
  int b_start = 0;
  if (u0 < u1) {
    int lo = 0, hi = B;  // largest b with pre[b] <= u0: the sequence holding position u0
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pre[mid] <= u0) lo = mid; else hi = mid;
    }
    b_start = lo;
  }
  const int cpos_start = u0 < u1 ? pre[b_start] : 0;  // cost position of b_start's start
  const int off_start = max(0, u0 - cpos_start - SC);  // its first unit in the range
  for (int i = tid; i < 128; i += NTHREADS) {
    alpha_s[i] = 1.0f;  // padded columns stay 1
    colrow[i] = column_row(P, i, GE);
  }

  if (warp == 0) dev::tmem_alloc(tmem_slot, C::TMEM_COLS);
  // Everything above read only context_lens (and shared memory). When this
  // kernel overlaps the previous one, that is all it may touch before
  // waiting; the producer also fetches its first block-table window first.
  int win0 = -1, len0 = 0;
  if (warp == kProducerWarp && u0 < u1) {
    const int j = (off_start + lane) / VS;  // the block of unit off_start + lane
    win0 = j < P.max_blocks_per_seq
               ? P.block_tables[size_t(b_start / P.n_groups) * P.max_blocks_per_seq + j] : -1;
    len0 = seq_len(P, b_start);
    // Pull the first blocks into L2 now, so that their copies after the
    // wait find them there: the kernel runs as a dependent of the previous
    // launch, and their DRAM latency overlaps its end (a prefetch cannot go
    // stale: every later write to these lines goes through L2). One lane per
    // block; a block's K, and its V (V^T), for all KV heads is one
    // contiguous range. The 8-bit decode follows the query-split launch and
    // takes the first ring's worth (64-sequence 8B layer: 41.5 -> 38.8 us
    // per step); bf16 follows the short merge of the previous step, and
    // takes one chunk's worth (55.6 -> 54.7 us; a whole ring made it slower,
    // 54.9 -> 55.7 us, as the copies after the wait queued behind it).
    const int n_pf = min((F8 ? C::ST : 1) * (Units<BS>::GROUPS / H),
                         (len0 + UT - 1) / UT - off_start);
    if (lane < n_pf && win0 >= 0 && win0 < P.num_blocks &&
        (lane == 0 || ((off_start + lane) % VS) == 0)) {
      const uint32_t blk_bytes = uint32_t(H * BS * D * (F8 ? 1 : 2));
      dev::prefetch_l2(P.k_base + size_t(win0) * blk_bytes, blk_bytes);
      dev::prefetch_l2(P.v_base + size_t(win0) * blk_bytes, blk_bytes);
    }
    if (lane == 0) {  // the tensor maps are kernel parameters: fetch them now too
      dev::prefetch_tmap(&tm_k);
      dev::prefetch_tmap(&tm_v);
      dev::prefetch_tmap(&tm_q);
    }
  }
  // The set-up ends here, before the dependency wait: the ring's plan
  // (generic-proxy writes) is ordered before the copies into it, the TMEM
  // address and the barriers are visible to every role. Nothing after the
  // wait stops the whole CTA, so the producer issues its first copies at once.
  dev::fence_async_smem();
  dev::tc_fence_before();
  __syncthreads();
  dev::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  dev::griddep_wait();
  if (blockIdx.x == 0) {  // the stream-K plan, for the merge kernel
    for (int i = tid; i <= B; i += NTHREADS) P.ws_plan[1 + i] = pre[i];
    if (tid == 0) P.ws_plan[0] = R;  // (the merge also takes SC)
    dev::fence_async_smem();
    __syncthreads();  // (CTA 0 only) the plan is read before the ring fills
  }
  if constexpr (F8) {
    // per-KV-head scales: k_scale in [0, 8), v_scale in [8, 16). Only the
    // softmax warps read them, after their first named barrier, which these
    // threads (softmax warp 0) reach after storing them.
    if (tid < 16) kvscale[tid] = (tid & 7) < H ? (tid < 8 ? P.k_scale : P.v_scale)[tid & 7] : 1.0f;
  }

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = dev::l2_evict_first_policy();
    const int U = Units<BS>::GROUPS / H;  // units per chunk
    const int grows = UT * H;              // rows of one unit (all KV heads)
    int chunk_seq = 0, seg_seq = 0;
    bool ok = true;
    // block-table window: lane j holds the entry of the block of unit first_unit + j
    auto load_window = [&](int v, int first_unit) {  // (v: virtual sequence)
      const int j = (first_unit + lane) / VS;
      return (v < B && j < P.max_blocks_per_seq)
                 ? P.block_tables[size_t(v / P.n_groups) * P.max_blocks_per_seq + j] : -1;
    };
    // The same window in two halves: window_raw loads it with the row and
    // entry clamped into the table (no condition on the loaded value, so the
    // warp does not stall on the load until the window is used), and
    // window_of applies the bounds when it is used. A sequence's next
    // windows and the next sequence's length are loaded this way at a
    // segment's start and taken at its chunk 32 or its end: a load whose
    // result is tested at once held up the first copies of a CTA by ~0.8 us.
    auto window_raw = [&](int v, int first_unit) {
      const int j = min((first_unit + lane) / VS, P.max_blocks_per_seq - 1);
      return P.block_tables[size_t(min(v, B - 1) / P.n_groups) * P.max_blocks_per_seq + j];
    };
    auto window_of = [&](int v, int first_unit, int raw) {
      return (v < B && (first_unit + lane) / VS < P.max_blocks_per_seq) ? raw : -1;
    };
    // Fused KV append: sequence b's new tokens (its last q_total, tokens
    // L-q_total .. L-1; row b*q_total + i of k_new/v_new/slot_mapping) are
    // written just before the copy of the chunk that reads their unit is
    // issued (so the chunks before it stream meanwhile). With several column
    // groups every group writes the new tokens its own stream reads (the same
    // bytes; each write precedes that group's own copy). A token's slot, table
    // entry and K/V rows are loaded together (one memory round trip) -- for
    // one new token per sequence already at the start of the piece -- then
    // checked and stored; a proxy fence makes the generic-proxy stores
    // visible to the TMA (async proxy) that follows.
    constexpr int CPR = D / 8;   // 16-byte chunks of one K or V row of one head
    constexpr int kRowMax = 4;   // chunks per lane of one token's rows (H <= 8, D <= 128)
    static_assert(8 * CPR <= 32 * kRowMax, "append row per lane");
    struct NewRow {
      int64_t slot;
      int e, pos;
      uint4 k[kRowMax], v[kRowMax];
    };
    const int n_row = H * CPR;
    auto load_row = [&](int b, int pos, int i, NewRow& r) {  // (b: a sequence)
      const size_t tok = size_t(b) * P.q_total + i;
      r.pos = pos;
      r.slot = P.slot_mapping[tok];
      r.e = P.block_tables[size_t(b) * P.max_blocks_per_seq + pos / BS];
#pragma unroll
      for (int j = 0; j < kRowMax; ++j) {
        const int k = lane + 32 * j;
        if (k < n_row) {
          r.k[j] = P.k_new[tok * n_row + k];
          r.v[j] = P.v_new[tok * n_row + k];
        }
      }
    };
    auto store_row = [&](const NewRow& r) {
      if (r.slot < 0) return;  // padding token
      if (r.slot >= int64_t(P.num_blocks) * BS) {
        if (lane == 0) atomicOr(&g_tc_errors, PA_DEVERR_SLOT);
        return;
      }
      if (r.e < 0 || r.e >= P.num_blocks || r.slot != int64_t(r.e) * BS + r.pos % BS) {
        if (lane == 0) atomicOr(&g_tc_errors, PA_DEVERR_APPEND_SLOT);
        return;
      }
#pragma unroll
      for (int j = 0; j < kRowMax; ++j) {
        const int k = lane + 32 * j;
        if (k < n_row) {
          const int hh = k / CPR, ch = k - (k / CPR) * CPR;
          const int off = r.pos % BS;
          const size_t dst = ((size_t(r.e) * H + hh) * BS + off) * CPR + ch;
          P.k_cache_w[dst] = r.k[j];
          P.v_cache_w[dst] = r.v[j];
        }
      }
    };
    NewRow pre_row;          // one new token per sequence: loaded at the piece start
    bool have_pre = false;
    // the new tokens of sequence b (context length L) that fall in units
    // [unit0, unit1) of a stream of its first L_stream tokens
    auto append_tokens = [&](int b, int L, int L_stream, int unit0, int unit1) {
      for (int i = 0; i < P.q_total; ++i) {
        const int pos = L - P.q_total + i;
        if (pos >= L_stream) break;
        if (pos < unit0 * UT || pos >= unit1 * UT) continue;
        if (have_pre && pre_row.pos == pos) {
          store_row(pre_row);
          have_pre = false;
        } else {
          NewRow r;
          load_row(b, pos, i, r);
          store_row(r);
        }
      }
      // each lane fences its own stores, then the warp syncs, so the copies
      // the issuing lanes start next see every lane's stores
      dev::fence_async_global();
      __syncwarp();
    };
    int b = b_start, off = off_start;
    int cpos = cpos_start;  // cost position of sequence b's start
    int win = win0;
    int L_cur = len0;
    while (ok && u0 < u1 && b < B) {
      if (*abort_flag) break;
      const int nb = L_cur > 0 ? (L_cur + UT - 1) / UT : 0;  // units
      if (nb == 0) {  // empty sequence: nothing of it in the stream
        ++b;
        off = 0;
        win = load_window(b, 0);
        L_cur = b < B ? seq_len(P, b) : 0;
        continue;
      }
      const int uend = min(nb, u1 - cpos - SC);  // b's units before the range's end
      if (uend <= off) break;                    // nothing of b (or after it) in range
      const int seg_nb = uend - off;
      const bool whole = off == 0 && seg_nb == nb;
      const int b_real = b / P.n_groups;
      // the sequence's context length (clamped), from what its group streams
      const int L_real = L_cur + P.q_total - (b - b_real * P.n_groups) * P.q_len - group_tokens(P, b);
      const int new_unit0 = (L_real - P.q_total) / UT;  // first unit holding a new token
      if constexpr (!F8) {  // (the 8-bit cache is written by the query-split launch)
        if (P.k_new != nullptr && P.q_total == 1 && off + seg_nb > new_unit0) {
          load_row(b_real, L_cur - 1, 0, pre_row);  // consumed at the chunk of its unit
          have_pre = true;
        }
      }
      // prefetched for later: the next sequence's length and first window,
      // this segment's second window
      const int L_nxt_raw = P.context_lens[min(b + 1, B - 1) / P.n_groups];
      const int win_nxt_seq_raw = window_raw(b + 1, 0);
      int win_nxt_raw = window_raw(b, off + 32);
      const int qs = seg_seq % C::QB;
      const int nch = (seg_nb + U - 1) / U;
      for (int c = 0; c < nch; ++c) {
        const int jb = c * U;  // first unit of the chunk within the segment
        if (jb > 0 && (jb & 31) == 0) {
          win = window_of(b, off + jb, win_nxt_raw);
          win_nxt_raw = window_raw(b, off + jb + 32);
        }
        if constexpr (!F8) {  // this chunk holds a unit of the new tokens
          const int nu = min(U, seg_nb - jb);
          if (P.k_new != nullptr && off + jb + nu > new_unit0)
            append_tokens(b_real, L_real, L_cur, off + jb, off + jb + nu);
        }
        const int slot = chunk_seq % C::ST;
        const uint32_t ph = uint32_t(chunk_seq / C::ST) & 1u;
        if (lane == 0) {
          ok = dev::mbar_wait_sleep(&empty[slot], ph ^ 1u, 64, P.wait_ns, abort_flag);
          if (ok) {
            ChunkMeta m;
            m.b = b;
            m.orow0 = (b_real * P.q_total + (b - b_real * P.n_groups) * P.q_len) * P.num_q_heads;
            m.qlen = group_tokens(P, b);
            m.flags = (c == 0 ? F_FIRST : 0) | (c == nch - 1 ? F_LAST : 0) | (whole ? F_WHOLE : 0);
            m.tok0 = (off + jb) * UT;
            m.L = L_cur;
            m.nblk = min(U, seg_nb - jb);
            m.qslot = qs;
            meta[slot] = m;
            dev::mbar_arrive_expect_tx(&full[slot], C::CHUNK_TX + (c == 0 ? C::Q_TX : 0u));
          }
        }
        ok = __shfl_sync(0xffffffffu, int(ok), 0) != 0;
        if (!ok) break;
        // lanes 0..U-1: one unit (all KV heads) each; lane 31 the queries
        const int e = __shfl_sync(0xffffffffu, win, (jb & 31) + (lane % U));
        unsigned char* kdst = ring + size_t(slot) * C::SLOT_BYTES;
        // A unit's coordinates: its block's rows (block size <= 16), or for
        // block size 32 its half (keys 16*half ..) of the block's H tiles.
        // Units past the segment, and bad table entries, read the zero fill
        // past the end of the tensor.
        int crd = P.oob_row, crd_v = P.oob_row_v, half = 0;
        if (lane < U && jb + lane < seg_nb) {
          if (e >= 0 && e < P.num_blocks) {
            crd = VS == 1 ? e * grows : e * H;
            crd_v = e * H;  // 8-bit V^T: the block's first tile
            half = (off + jb + lane) & (VS - 1);
          } else {
            atomicOr(&g_tc_errors, PA_DEVERR_TABLE_ENTRY);
          }
        }
        if constexpr (F8) {
          // K rows, and the unit's H V^T sub-tiles as one box
          if (lane < U) {
            if constexpr (VS == 1) {
              dev::tma_load_2d(kdst + lane * grows * 128, &tm_k, 0, crd, &full[slot], pol);
              dev::tma_load_3d(kdst + C::K_BYTES + lane * H * C::VT_TILE, &tm_v, 0, 0, crd_v,
                               &full[slot], pol);
            } else {
              dev::tma_load_3d(kdst + lane * grows * 128, &tm_k, 0, half * UT, crd, &full[slot],
                               pol);
              dev::tma_load_4d(kdst + C::K_BYTES + lane * H * C::VT_TILE, &tm_v, 0, 0, half,
                               crd_v, &full[slot], pol);
            }
          }
        } else {
          if (lane < U) {
#pragma unroll
            for (int hf = 0; hf < C::HALVES; ++hf) {
              unsigned char* d = kdst + hf * C::HALF_BYTES + lane * grows * 128;
              if constexpr (VS == 1) {
                dev::tma_load_2d(d, &tm_k, hf * 64, crd, &full[slot], pol);
                dev::tma_load_2d(d + C::K_BYTES, &tm_v, hf * 64, crd, &full[slot], pol);
              } else {
                dev::tma_load_3d(d, &tm_k, hf * 64, half * UT, crd, &full[slot], pol);
                dev::tma_load_3d(d + C::K_BYTES, &tm_v, hf * 64, half * UT, crd, &full[slot], pol);
              }
            }
          }
        }
        if (c == 0) {
          // The segment's queries, into query buffer qs once its previous
          // segment has read it. Only this copy waits for that: the chunk's
          // K/V copies above are already on their way, so with one query
          // buffer a segment's first data no longer waits behind the previous
          // segment's last score product.
          bool qok = true;
          if (lane == 31) {
            qok = dev::mbar_wait_sleep(&qempty[qs], (uint32_t(seg_seq / C::QB) & 1u) ^ 1u, 64,
                                       P.wait_ns, abort_flag);
            if (!qok) {
              // the chunk's barrier was told to expect the queries too: take
              // their bytes off it, so that its phase completes when the K/V
              // copies already issued have landed
              *abort_flag = 1;
              dev::mbar_complete_tx(&full[slot], C::Q_TX);
            } else {
              if constexpr (F8) {
                dev::tma_load_2d(qbuf + qs * C::Q_BYTES, &tm_q, 0, b * P.q_rows, &full[slot],
                                 pol);
                dev::bulk_load(qalpha + qs * 64, P.q_inv_alpha + size_t(b) * N, N * 4,
                               &full[slot], pol);
              } else {
#pragma unroll
                for (int hf = 0; hf < C::HALVES; ++hf)
                  dev::tma_load_2d(qbuf + qs * C::Q_BYTES + hf * C::QH_BYTES, &tm_q, hf * 64,
                                   b * P.q_rows, &full[slot], pol);
              }
            }
          }
          if (__shfl_sync(0xffffffffu, int(qok), 31) == 0) ok = false;
        }
        // counted as issued even when its queries were not: its K/V copies
        // are in flight, and the wind-down waits for them
        ++chunk_seq;
        if (lane == 0) *issued = chunk_seq;
        if (!ok) break;
      }
      ++seg_seq;
      if (uend < nb) break;  // the range ends inside b
      cpos += nb + SC;
      win = window_of(b + 1, 0, win_nxt_seq_raw);
      L_cur = b + 1 < B ? seq_len_of(P, b + 1, L_nxt_raw) : 0;
      ++b;
      off = 0;
    }
    // end of work: a sentinel chunk tells the consumers to stop. After an
    // abort there is none: every other role gives up its waits on the flag,
    // and an extra arrival on a barrier whose copies are still in flight
    // would be undefined.
    if (lane == 0) {
      if (!ok) {
        atomicOr(&g_tc_errors, PA_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      if (!*abort_flag) {
        const int slot = chunk_seq % C::ST;
        const uint32_t ph = uint32_t(chunk_seq / C::ST) & 1u;
        if (dev::mbar_wait(&empty[slot], ph ^ 1u, P.wait_ns, abort_flag)) {
          ChunkMeta m{};
          m.flags = F_END;
          meta[slot] = m;
          dev::mbar_arrive(&full[slot]);
        } else if (!*abort_flag) {
          atomicOr(&g_tc_errors, PA_DEVERR_TIMEOUT);
          *abort_flag = 1;
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0)
      mma_loop<D, GE, N, F8, kDiagP<D, GE, N, F8, BS>, kMnP<D, GE, N, F8, BS>>(
          ring, qbuf, pbuf, full, empty, qempty, bar_s, bar_o, bar_p, drain, meta, tmem,
          abort_flag, H, P.wait_ns);
  } else {
    // ------------------------------------------------------------ softmax
    Softmax<D, GE, N, F8, BS>::run(P, ring, pbuf, full, bar_s, bar_o, bar_p, meta, red, red2,
                              alpha_s, l_s, m_s, qalpha, kvscale, colrow, tmem, abort_flag,
                              consumed);
  }

  __syncthreads();
  if (*abort_flag && tid == 0) {
    // Wind down after a stalled wait: every bulk copy issued but not consumed
    // lands (each wait bounded by the full 2 s budget, whatever the caller's,
    // and deaf to the flag) before shared memory is released. (The MMA warp
    // has already waited for its own MMAs.)
    for (int c = *consumed; c < *issued; ++c)
      (void)dev::mbar_wait(&full[c % C::ST], uint32_t(c / C::ST) & 1u);
  }
  dev::tc_fence_before();
  __syncthreads();
  // The merge kernel (a programmatic dependent) can do nothing before this
  // grid ends: let it launch as the CTAs finish, not earlier, so its waiting
  // CTAs never share an SM with a running decode CTA.
  if (tid == 0) dev::griddep_launch_dependents();
  if (warp == 0) {
    dev::tc_fence_after();
    dev::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Log-sum-exp merge of the partials of sequences that span several CTAs, and
// zero rows for empty sequences. One warp per (sequence, column). The
// lanes read the pieces' (max, sum) pairs side by side while the rows of the
// first kPrefetch pieces are already in flight, so a typical merge costs one
// memory round trip.
template <int VPL>
struct Row {
  float v[VPL];
  __device__ void load(const float* src) {
    if constexpr (VPL == 4) {
      const float4 t = *reinterpret_cast<const float4*>(src);
      v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else {
      const float2 t = *reinterpret_cast<const float2*>(src);
      v[0] = t.x; v[1] = t.y;
    }
  }
  __device__ void madd_into(float* acc, float w) const {
#pragma unroll
    for (int j = 0; j < VPL; ++j) acc[j] = fmaf(w, v[j], acc[j]);
  }
};

struct MergeCols {
  int num_q_heads, num_cols, group_cols, g_log2;
  int q_group, q_total, n_groups;  // tokens per column group, new tokens, groups
  int seg_cost;  // the decode plan's cost of a sequence start (units)
};

template <int D>
__global__ void __launch_bounds__(128)
    merge_segments_kernel(__nv_bfloat16* __restrict__ out, const float* __restrict__ part_m,
                          const float* __restrict__ part_l, const float* __restrict__ part_acc,
                          const int* __restrict__ ws_plan, const MergeCols mc) {
  constexpr int VPL = D / 32;
  constexpr int kPrefetch = 16;
  // The next kernel on the stream may start its own set-up now (it waits
  // for this grid before it touches memory this grid writes).
  dev::griddep_launch_dependents();
  dev::griddep_wait();  // launched as a programmatic dependent of the decode
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * 4 + warp;  // column (the decode kernel's layout)
  const int b = blockIdx.y;             // virtual sequence
  if (n >= mc.num_cols) return;
  const int g = n / mc.group_cols, r = n - g * mc.group_cols;
  const int qi = r >> mc.g_log2;  // query token of the column within its group
  const int seq = b / mc.n_groups, tok = (b - seq * mc.n_groups) * mc.q_group + qi;
  if (qi >= mc.q_group || tok >= mc.q_total) return;  // unused column
  const int R = ws_plan[0];
  const int pre0 = ws_plan[1 + b], pre1 = ws_plan[2 + b];
  const size_t orow = (size_t(seq) * mc.q_total + tok) * mc.num_q_heads + (g << mc.g_log2) +
                      (r & ((1 << mc.g_log2) - 1));
  __nv_bfloat16* o = out + orow * D + lane * VPL;
  if (pre1 <= pre0) {  // empty sequence
#pragma unroll
    for (int j = 0; j < VPL; ++j) o[j] = __float2bfloat16_rn(0.0f);
    return;
  }
  // the sequence's units occupy cost positions [pre0 + seg_cost, pre1)
  const int c0 = (pre0 + mc.seg_cost) / R, c1 = (pre1 - 1) / R;
  if (c0 == c1) return;  // written whole by the decode kernel
  const int nseg = c1 - c0 + 1;
  // piece k of the sequence sits in partial slot (b + c0 + k)
  const size_t slot0 = size_t(b + c0) * mc.num_cols + n;
  const size_t stride = size_t(mc.num_cols);
  const float* src0 = part_acc + slot0 * D + lane * VPL;
  Row<VPL> pf[kPrefetch];
#pragma unroll
  for (int k = 0; k < kPrefetch; ++k)
    if (k < nseg) pf[k].load(src0 + size_t(k) * stride * D);
  float m_first = -INFINITY, l_first = 0.0f;  // this lane's piece among the first 32
  if (lane < nseg) {
    m_first = part_m[slot0 + lane * stride];
    l_first = part_l[slot0 + lane * stride];
  }
  float M = m_first;
  for (int k = 32 + lane; k < nseg; k += 32) M = fmaxf(M, part_m[slot0 + k * stride]);
#pragma unroll
  for (int o2 = 16; o2 >= 1; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
  float acc[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) acc[j] = 0.0f;
  float den = 0.0f;
  for (int base = 0; base < nseg; base += 32) {
    float w = 0.0f;
    if (base + lane < nseg) {
      const float mk = base == 0 ? m_first : part_m[slot0 + (base + lane) * stride];
      const float lk = base == 0 ? l_first : part_l[slot0 + (base + lane) * stride];
      w = dev::fast_exp2(mk - M);
      den = fmaf(w, lk, den);
    }
    const int cnt = min(32, nseg - base);
    int k0 = 0;
    if (base == 0) {
#pragma unroll
      for (int k = 0; k < kPrefetch; ++k) {
        const float wk = __shfl_sync(0xffffffffu, w, k);
        if (k < cnt) pf[k].madd_into(acc, wk);
      }
      k0 = kPrefetch;
    }
    for (int k = k0; k < cnt; k += 8) {
      Row<VPL> r[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (k + j < cnt) r[j].load(src0 + size_t(base + k + j) * stride * D);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float wj = __shfl_sync(0xffffffffu, w, (k + j) & 31);
        if (k + j < cnt) r[j].madd_into(acc, wj);
      }
    }
  }
#pragma unroll
  for (int o2 = 16; o2 >= 1; o2 >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o2);
  const float inv = __frcp_rn(den);
#pragma unroll
  for (int j = 0; j < VPL; ++j) o[j] = __float2bfloat16_rn(acc[j] * inv);
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
int g_sm_count[64] = {};

int encode_fn(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::call_once(g_encode_once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  *fn = g_encode;
  return g_encode ? 0 : int(cudaErrorNotSupported);
}

// A tiled tensor map of `rank` dimensions (innermost first): dims, byte
// strides of dimensions 1.., box; out-of-range elements read as zero.
int make_map_nd(CUtensorMap* m, CUtensorMapDataType type, int rank, const void* base,
                const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                CUtensorMapSwizzle swizzle) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  if (encode_fn(&enc)) return int(cudaErrorNotSupported);
  cuuint32_t estride[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(m, type, cuuint32_t(rank), const_cast<void*>(base), dims, strides, box,
                   estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : int(cudaErrorInvalidValue);
}

// 2-D bf16 tensor [rows][cols], box box_rows x 64 cols, 128B swizzle.
int make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  return make_map_nd(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

// 2-D byte tensor [rows][cols], box box_rows x box_cols, the given swizzle.
int make_map_u8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {box_cols, box_rows};
  return make_map_nd(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, swizzle);
}

// Block size 32: the K or V cache ([tiles][32 keys][D], one tile per (block,
// KV head)) as a 3-D tensor; box = 16 keys of `heads` consecutive tiles
// (box_cols of the row), 128B swizzle. elem: 2 (bf16) or 1 (E4M3) bytes.
int make_map_halves(CUtensorMap* m, const void* base, uint64_t tiles, uint64_t d, int elem,
                    uint32_t box_cols, uint32_t heads) {
  const cuuint64_t dims[3] = {d, 32, tiles};
  const cuuint64_t strides[2] = {d * elem, 32 * d * elem};
  const cuuint32_t box[3] = {box_cols, uint32_t(kF8Tile), heads};
  return make_map_nd(m, elem == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                     3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// The 8-bit V^T cache: per (block, KV head) tile, BS/16 sub-tiles of
// [D rows][16 bytes], each sub-tile D * 16 contiguous bytes. The map reads a
// sub-tile as rows of 256 bytes rather than D rows of 16 bytes: the same
// bytes land at the same shared-memory offsets (both boxes are contiguous
// row-major copies), with a sixteenth of the rows for the copy engine to walk
// and whole 32-byte sectors per row. Block size 16: a 3-D tensor
// [tiles][D/16][256], box = `heads` whole tiles. Block size 32: a 4-D tensor
// [tiles][2][D/16][256], box = one sub-tile of `heads` tiles. The kernel's
// coordinates are (0, 0, tile) and (0, 0, sub-tile, tile) either way. No
// swizzle.
int make_map_vt(CUtensorMap* m, const void* base, uint64_t tiles, uint64_t d, uint32_t heads,
                int block_size) {
  constexpr uint64_t kRow = 256;                  // bytes of one box row
  const uint64_t sub = d * kF8Tile;               // bytes of one sub-tile
  const uint64_t rows = sub / kRow;               // box rows of one sub-tile
  if (sub % kRow != 0) return int(cudaErrorInvalidValue);
  if (block_size == 16) {
    const cuuint64_t dims[3] = {kRow, rows, tiles};
    const cuuint64_t strides[2] = {kRow, sub};
    const cuuint32_t box[3] = {uint32_t(kRow), uint32_t(rows), heads};
    return make_map_nd(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  const cuuint64_t dims[4] = {kRow, rows, 2, tiles};
  const cuuint64_t strides[3] = {kRow, sub, 2 * sub};
  const cuuint32_t box[4] = {uint32_t(kRow), uint32_t(rows), 1, heads};
  return make_map_nd(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, base, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <int D, int GE, int N, bool F8, int BS>
int launch_tc_t(const DecodeLaunch& Lc, cudaStream_t stream) {
  using C = TcCfg<D, N, F8, kDiagP<D, GE, N, F8, BS>>;
  constexpr int VS = Units<BS>::VS;
  const pa_decode_params* p = Lc.p;
  const QueryMap qm = query_map(p);
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(paged_decode_tc_kernel<D, GE, N, F8, BS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return int(e);
    configured = true;
  }
  const int H = p->num_kv_heads;
  CUtensorMap tk, tv, tq;
  const uint64_t cache_rows = uint64_t(p->num_blocks) * H * BS;
  const uint64_t tiles = uint64_t(p->num_blocks) * H;
  int r = 0;
  if constexpr (F8) {
    // K rows of D bytes; V^T [D][16] sub-tiles per (block, head), copied as
    // 256-byte rows; the split queries, 2N rows of D bytes per sequence
    if constexpr (VS == 1) {
      r = make_map_u8(&tk, p->k_cache, cache_rows, D, D, uint32_t(BS * H),
                      CU_TENSOR_MAP_SWIZZLE_128B);
    } else {
      r = make_map_halves(&tk, p->k_cache, tiles, D, 1, D, uint32_t(H));
    }
    if (!r) r = make_map_vt(&tv, p->v_cache, tiles, D, uint32_t(H), BS);
    if (!r)
      r = make_map_u8(&tq, Lc.q8, uint64_t(qm.num_seqs) * 2 * N, D, D, uint32_t(2 * N),
                      CU_TENSOR_MAP_SWIZZLE_128B);
    if (!r) r = launch_quantize_q(p->q, Lc.q8, Lc.q_inv_alpha, qm, p, Lc.append, stream);
  } else {
    if constexpr (VS == 1) {
      r = make_map(&tk, p->k_cache, cache_rows, D, uint32_t(BS * H));
      if (!r) r = make_map(&tv, p->v_cache, cache_rows, D, uint32_t(BS * H));
    } else {
      r = make_map_halves(&tk, p->k_cache, tiles, D, 2, 64, uint32_t(H));
      if (!r) r = make_map_halves(&tv, p->v_cache, tiles, D, 2, 64, uint32_t(H));
    }
    if (qm.query_len == 1) {
      // the rows of q are already in column order (column = query head); a
      // box of N rows may run into the next sequence's rows, never used
      if (!r) r = make_map(&tq, p->q, uint64_t(p->num_seqs) * p->num_q_heads, D, uint32_t(N));
    } else {
      if (!r) r = make_map(&tq, Lc.qp, uint64_t(qm.num_seqs) * N, D, uint32_t(N));
      if (!r) r = launch_permute_q(p->q, Lc.qp, qm, stream);
    }
  }
  if (r) return r;
  TcParams P;
  P.block_tables = p->block_tables;
  P.context_lens = p->context_lens;
  P.out = static_cast<__nv_bfloat16*>(p->out);
  P.part_m = Lc.part_m;
  P.part_l = Lc.part_l;
  P.part_acc = Lc.part_acc;
  P.ws_plan = Lc.plan;
  // the 8-bit cache's new tokens were written by the query-split launch
  const pa_append_params* a = F8 ? nullptr : Lc.append;
  P.k_new = a ? static_cast<const uint4*>(a->k_new) : nullptr;
  P.v_new = a ? static_cast<const uint4*>(a->v_new) : nullptr;
  P.slot_mapping = a ? a->slot_mapping : nullptr;
  P.k_cache_w = a ? static_cast<uint4*>(a->k_cache) : nullptr;
  P.v_cache_w = a ? static_cast<uint4*>(a->v_cache) : nullptr;
  P.k_scale = p->k_scale;
  P.v_scale = p->v_scale;
  P.q_inv_alpha = Lc.q_inv_alpha;
  P.k_base = static_cast<const unsigned char*>(p->k_cache);
  P.v_base = static_cast<const unsigned char*>(p->v_cache);
  P.oob_row_v = int(tiles);  // first V^T tile past the cache
  P.q_rows = F8 ? 2 * N : (qm.query_len == 1 ? p->num_q_heads : N);
  P.num_cols = qm.num_cols;
  P.q_len = qm.q_group;
  P.q_total = qm.query_len;
  P.n_groups = qm.n_groups;
  P.g_log2 = qm.g_log2;
  P.max_blocks_per_seq = p->max_blocks_per_seq;
  P.num_seqs = qm.num_seqs;  // virtual sequences
  P.num_kv_heads = H;
  P.num_q_heads = p->num_q_heads;
  P.num_blocks = p->num_blocks;
  P.cap = min(p->max_blocks_per_seq * BS, p->max_context_len);
  P.oob_row = VS == 1 ? int(cache_rows) : int(tiles);
  P.scale_log2 = p->scale * kLog2e;
  P.wait_ns = p->wait_timeout_us > 0 ? uint64_t(p->wait_timeout_us) * 1000u : dev::kWaitNsLimit;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(Lc.grid);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // overlap the set-up with the previous kernel only when the caller says
  // context_lens and block_tables were final before that kernel began
  attr[0].val.programmaticStreamSerializationAllowed = p->overlap_prologue ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, paged_decode_tc_kernel<D, GE, N, F8, BS>, tk, tv, tq, P);
  if (e != cudaSuccess) return int(e);
  // the merge launches while the decode drains and waits for it on the device
  cudaLaunchConfig_t mcfg = {};
  mcfg.gridDim = dim3((qm.num_cols + 3) / 4, qm.num_seqs);
  mcfg.blockDim = dim3(128);
  mcfg.stream = stream;
  mcfg.attrs = attr;
  mcfg.numAttrs = 1;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  MergeCols mc;
  mc.num_q_heads = p->num_q_heads;
  mc.num_cols = qm.num_cols;
  mc.group_cols = qm.group_cols;
  mc.g_log2 = qm.g_log2;
  mc.q_group = qm.q_group;
  mc.q_total = qm.query_len;
  mc.n_groups = qm.n_groups;
  mc.seg_cost = start_chunks(F8, qm.q_group) * (Units<BS>::GROUPS / H);
  e = cudaLaunchKernelEx(&mcfg, merge_segments_kernel<D>, P.out,
                         static_cast<const float*>(P.part_m), static_cast<const float*>(P.part_l),
                         static_cast<const float*>(P.part_acc),
                         static_cast<const int*>(P.ws_plan), mc);
  return int(e);
}

// Instances by (columns per KV head GE, padded columns N). Block size 8 takes
// GE <= 8 (its groups of 8 rows leave 8 reduction columns per group).
template <int D, bool F8, int BS>
int dispatch_tc(const DecodeLaunch& Lc, cudaStream_t s) {
  const int GE = tc_group_cols(Lc.p);
  const int N = tc_n_pad(tc_cols(Lc.p));
  switch (GE * 1000 + N) {
    case 1016: return launch_tc_t<D, 1, 16, F8, BS>(Lc, s);
    case 2016: return launch_tc_t<D, 2, 16, F8, BS>(Lc, s);
    case 4016: return launch_tc_t<D, 4, 16, F8, BS>(Lc, s);
    case 4032: return launch_tc_t<D, 4, 32, F8, BS>(Lc, s);
    case 8016: return launch_tc_t<D, 8, 16, F8, BS>(Lc, s);
    case 8032: return launch_tc_t<D, 8, 32, F8, BS>(Lc, s);
    case 8064: return launch_tc_t<D, 8, 64, F8, BS>(Lc, s);
    default: break;
  }
  if constexpr (BS >= 16) {
    switch (GE * 1000 + N) {
      case 16016: return launch_tc_t<D, 16, 16, F8, BS>(Lc, s);
      case 16032: return launch_tc_t<D, 16, 32, F8, BS>(Lc, s);
      case 16064: return launch_tc_t<D, 16, 64, F8, BS>(Lc, s);
      case 16128:
        if constexpr (!F8) return launch_tc_t<D, 16, 128, F8, BS>(Lc, s);
        return int(cudaErrorInvalidValue);
      default: break;
    }
  }
  return int(cudaErrorInvalidValue);
}

// Device error word of the including translation unit, read and cleared.
inline int read_and_clear_tc_error_word(uint32_t* flags) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_tc_errors, sizeof(v));
  if (e != cudaSuccess) return int(e);
  e = cudaMemcpyToSymbol(g_tc_errors, &zero, sizeof(zero));
  *flags = v;
  return int(e);
}

}  // namespace
}  // namespace pa
