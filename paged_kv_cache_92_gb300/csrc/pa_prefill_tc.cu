// Several new tokens per sequence on the tensor cores, query-major ("How Paged
// Attention and Continuous Batching Actually Work", §Continuous batching: the
// scheduled tokens of one request, as in a chunked prefill). A unit of work (an
// item) is (sequence, group of HB KV heads, tile of query rows, split of the
// keys); it streams its share of those heads' blocks once for all its rows. A
// row is new token i of query head (kv head)*G + g and sees the sequence's
// first L - Q + i + 1 keys. With several splits (small batches) each item
// leaves fp32 partials (running maximum, sum, unnormalised O row) and a merge
// kernel combines a row's splits, as in a split-K decode. After the step's KV
// write the kernel launches as a programmatic dependent: its set-up overlaps
// the write, and every thread waits for it before touching the cache.
//
// The column-group decode (pa_decode_tc.cuh) puts the keys on the MMAs' M side
// and streams them once per group of new tokens; with many new tokens each
// group re-reads the keys. Here the queries are on the M side:
//   S[128 rows][64 columns]  = Q . K^T     (A = Q, B = K chunk, both K-major)
//   O[128 rows][128 d]      += P . V       (A = P from TMEM; B = V, MN-major)
// S and P are double-buffered in TMEM; P (bf16, two to a 32-bit column) feeds
// the value product from there, in columns of its own so that the scores of
// the next chunks need not wait for the value product that reads it. A thread
// owns a row: its softmax (running maximum, sum, the conditional rescale of
// its O row) needs no other thread.
//
// Persistent: one CTA per SM takes the items of its rank in a snake over the
// items sorted by sequence length (longest first, every second pass reversed).
// The producer, MMA and softmax warps each walk that list and keep their own
// counters, so the loads of the next item overlap the end of the current one:
// two Q buffers in shared memory, two O accumulators in TMEM, and one K/V
// ring whose chunk and barrier phases run on across items.
//
// Layout of an item's 128 rows (TMEM lanes): HB heads x RPH rows, row r0 of a
// head being token tile*QT + r0/G, query head g = r0 % G. A chunk's 64 columns
// are NB = 64/(BS*HB) blocks x HB heads x BS keys (BS the block size, 16 or
// 32): one 2-D tensor-map box [HB*BS rows][64 d] per block and 64-d half (the
// HB heads of a block are adjacent in the cache), so every TMA request moves
// 4 KiB or more with HB = 2 or BS = 32 (the TMA unit spends a fixed time per
// request: streaming 2 KiB requests tops out well below 4 KiB ones). A row's
// scores against the other heads' keys are computed and ignored: its P is
// zero there.
#include "pa_decode_tc.cuh"
#include "pa_query_major.h"

namespace pa {
namespace {

constexpr int QM_D = 128;
constexpr int QM_KC = 64;         // columns per chunk
constexpr int QM_ROWS = 128;      // query rows per item (MMA M)
constexpr int QM_ST = 5;          // ring slots
constexpr int QM_THREADS = 192;   // softmax warps 0-3, producer 4, MMA 5
constexpr int QM_HALF_Q = QM_ROWS * 128;     // one 64-d half of Q: [128 rows][128 B]
constexpr int QM_Q_BYTES = 2 * QM_HALF_Q;
constexpr int QM_HALF_KV = QM_KC * 128;      // one 64-d half of a K or V chunk: [64 rows][128 B]
constexpr int QM_KV_BYTES = 2 * QM_HALF_KV;  // K (or V) of a chunk
constexpr int QM_SLOT = 2 * QM_KV_BYTES;     // K halves, then V halves
constexpr int QM_OFF_Q = 0;                  // two Q buffers
constexpr int QM_OFF_RING = QM_OFF_Q + 2 * QM_Q_BYTES;
constexpr int QM_OFF_BARS = QM_OFF_RING + QM_ST * QM_SLOT;
// full[ST], empty[ST], qfull[2], qempty[2], s[2], p[2], o[2], oempty[2], drain
constexpr int QM_NBARS = 2 * QM_ST + 13;
constexpr int QM_OFF_WORDS = QM_OFF_BARS + QM_NBARS * 8;
constexpr int QM_OFF_ORDER = QM_OFF_WORDS + 64;      // sequence of each length rank (<= 256)
constexpr int QM_OFF_PLAN = QM_OFF_ORDER + 1024;     // first item of each (rank, tile) (< 256)
constexpr int QM_SMEM = QM_OFF_PLAN + 512 + 1024;    // + alignment slack
static_assert(QM_SMEM <= kMaxDynSmem, "shared memory budget");
constexpr int QM_MAX_RANKED = 256;
// CTAs of a split launch at most: the split plans stage 512 ints and one int
// per CTA in the still-empty ring
constexpr int QM_MAX_SPLIT_GRID = 4096;
static_assert(QM_ST * QM_SLOT >= (512 + QM_MAX_SPLIT_GRID) * int(sizeof(int)), "plan scratch");
// TMEM: S[2] at [0, 128), O[2] at [128, 384), P[2] at [384, 448)
constexpr uint32_t QM_TMEM_COLS = 512;
constexpr uint32_t QM_TMEM_P = 384;
constexpr uint32_t QM_IDESC_S = dev::idesc_bf16_f32(QM_ROWS, QM_KC, false, false);
constexpr uint32_t QM_IDESC_PV = dev::idesc_bf16_f32(QM_ROWS, QM_D, false, true);

// tcgen05.mma with A in TMEM (M rows in lanes; a K = 16 step is 8 columns,
// two bf16 of a row per 32-bit column, the lower-indexed in the low half).
__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(uint32_t(accumulate))
      : "memory");
}

struct QmParams {
  const int32_t* block_tables;
  const int32_t* context_lens;
  __nv_bfloat16* out;
  int num_seqs, num_kv_heads, num_q_heads, q_len, tiles, head_groups, splits, num_items,
      max_blocks_per_seq, num_blocks, cap, oob_row;
  float* part_ml;  // splits > 1: [B*Q*Hq rows][splits][m, l]
  float* part_o;   // splits > 1: [B*Q*Hq rows][splits][128]
  float scale_log2;
  uint64_t wait_ns;
};

// One item as every role sees it.
struct QmItem {
  int b, hg0, tile;  // sequence, first KV head, tile of new tokens
  int split, c0;     // split of the keys, its first chunk
  int ns;            // splits of this (sequence, head group, tile)
  int L;             // length after the rules (0: an empty sequence)
  int keys;          // keys the item's last row sees
  int nblk, n;       // blocks of those keys, chunks of this split
  bool bad_len;      // the length broke a rule (reported once per sequence)
};

template <int G, int HB, bool SPLIT, int BS>
__global__ void __launch_bounds__(QM_THREADS, 1)
    query_major_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_q, const QmParams P) {
  constexpr int RPH = QM_ROWS / HB;  // rows per head
  constexpr int QT = RPH / G;        // new tokens per tile
  constexpr int BR = BS * HB;        // rows of one block's box (HB heads x BS keys)
  constexpr int NB = QM_KC / BR;     // blocks per chunk
  constexpr int NC = BS * NB;        // scores of a chunk per thread (its head's keys)
  static_assert(QT >= 1 && NB >= 1 && BS % 16 == 0, "tile shape");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* qbuf = smem + QM_OFF_Q;
  unsigned char* ring = smem + QM_OFF_RING;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + QM_OFF_BARS);
  uint64_t* full = bars;
  uint64_t* empty = bars + QM_ST;
  uint64_t* qfull = bars + 2 * QM_ST;  // [2] Q of the item landed in buffer k
  uint64_t* qempty = qfull + 2;        // [2] the last scores reading Q buffer k completed
  uint64_t* bar_s = qempty + 2;        // [2] scores of chunk c (global count) in S[c % 2]
  uint64_t* bar_p = bar_s + 2;         // [2] P of chunk c written (P[c % 2]), S[c % 2] read
  uint64_t* bar_o = bar_p + 2;         // [2] value product of chunk c done
  uint64_t* oempty = bar_o + 2;        // [2] O accumulator k read out by the softmax warps
  uint64_t* drain = oempty + 2;
  int* words = reinterpret_cast<int*>(smem + QM_OFF_WORDS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&words[0]);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&words[1]);
  int* issued = &words[2];     // K/V chunks requested
  int* consumed = &words[3];   // K/V chunks whose value product was issued
  int* q_issued = &words[4];   // Q loads requested
  int* q_waited = &words[5];   // Q loads seen landed
  int* order = reinterpret_cast<int*>(smem + QM_OFF_ORDER);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Q = P.q_len;
  const bool ranked = P.num_seqs <= QM_MAX_RANKED;

  // ------------------------------------------------------------ set-up
  if (ranked) {
    // Sequences by decreasing length (ties by index): the lengths are staged
    // in the ring (before any copy lands there), then order[rank] = sequence.
    int* lens_s = reinterpret_cast<int*>(ring);
    for (int v = tid; v < P.num_seqs; v += QM_THREADS) lens_s[v] = P.context_lens[v];
    __syncthreads();
    for (int v = tid; v < P.num_seqs; v += QM_THREADS) {
      const int Lv = lens_s[v];
      int above = 0;
      for (int u = 0; u < P.num_seqs; ++u) {
        const int Lu = lens_s[u];
        above += Lu > Lv || (Lu == Lv && u < v);
      }
      order[above] = v;
    }
    dev::fence_async_smem();  // the staged lengths before the ring's first copy
  }

  // The keys an item of sequence length L and tile `tile` covers: the length
  // rules (at most the tables' capacity; a sequence shorter than its new
  // tokens is empty) and the keys its tile's last new token sees. Returns
  // the chunks of all its splits.
  auto span_of = [&](int L, int tile, QmItem& it) {
    it.bad_len = L > P.cap;
    if (L > P.cap) L = P.cap;
    if (L > 0 && L < Q) {  // no room for the new tokens: an empty sequence
      it.bad_len = true;
      L = 0;
    }
    it.L = L;
    const int i_last = min(Q, (tile + 1) * QT) - 1;  // the item's last new token
    const int keys = L > 0 ? L - Q + i_last + 1 : 0;  // what its last row sees
    it.keys = keys;
    it.nblk = (keys + BS - 1) / BS;
    return (it.nblk + NB - 1) / NB;
  };

  // Split keys (fewer than 256 (sequence, head group, tile) units; the
  // workspace holds P.splits partials per row). Two plans within that bound:
  // every unit split P.splits ways and dealt in the snake, or one wave: each
  // (sequence, tile) cut into pieces of at most T chunks, T the smallest that
  // leaves every CTA at most one item. Every CTA computes both from the
  // lengths and takes the one whose busiest CTA has fewer chunks (an item
  // counted kItemChunks more for its start and its partials).
  int* plan_wave = &words[6];   // the one-wave plan is in use
  int* plan_t = &words[7];      // its T
  int* plan_items = &words[8];  // items of the plan in use
  uint16_t* plan_off = reinterpret_cast<uint16_t*>(smem + QM_OFF_PLAN);
  auto wave_splits = [&](int n, int T) { return n > 0 ? min(P.splits, (n + T - 1) / T) : 1; };
  if (SPLIT && tid == 0) {  // the uniform plan unless the comparison below picks the other
    *plan_wave = 0;
    *plan_items = P.num_items;
  }
  if (SPLIT && ranked) {  // (fewer than 256 units: at most 255 sequences, all ranked)
    constexpr int kItemChunks = 2;
    int* scratch = reinterpret_cast<int*>(ring);  // the staged lengths at [0, 256)
    int* n_rt = scratch + 256;                     // chunks of each (rank, tile)
    int* per_cta = scratch + 512;                  // the uniform plan's chunks per CTA
    const int tiles = P.tiles, RT = P.num_seqs * tiles, cap = P.splits, hgc = P.head_groups;
    const int grid = int(gridDim.x);
    auto warp_max = [](int v) {
      for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
      return v;
    };
    __syncthreads();  // order[] complete
    for (int rt = tid; rt < RT; rt += QM_THREADS) {
      QmItem tmp;
      n_rt[rt] = span_of(scratch[order[rt / tiles]], rt % tiles, tmp);
    }
    for (int c = tid; c < grid; c += QM_THREADS) per_cta[c] = 0;
    __syncthreads();
    // uniform: item x is (rank, head group, tile, split), split fastest
    const int per_seq = hgc * tiles * cap;
    for (int x = tid; x < P.num_items; x += QM_THREADS) {
      const int rem = x % per_seq, sp = rem % cap;
      const int n = n_rt[x / per_seq * tiles + rem / cap % tiles];
      const int sz = (sp + 1) * n / cap - sp * n / cap;
      const int pass = x / grid, pos = x % grid;
      if (sz > 0) atomicAdd(&per_cta[(pass & 1) ? grid - 1 - pos : pos], sz + kItemChunks);
    }
    __syncthreads();
    if (warp == 0) {  // the uniform plan's busiest CTA
      int mx = 0;
      for (int c = lane; c < grid; c += 32) mx = max(mx, per_cta[c]);
      mx = warp_max(mx);
      if (lane == 0) words[9] = mx;
    } else if (warp == 1) {  // one wave: T by bisection (the item count falls as T grows)
      auto count = [&](int T) {
        int c = 0;
        for (int rt = lane; rt < RT; rt += 32) c += hgc * wave_splits(n_rt[rt], T);
        for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
        return c;
      };
      int nmax = 0;
      for (int rt = lane; rt < RT; rt += 32) nmax = max(nmax, n_rt[rt]);
      nmax = warp_max(nmax);
      int cost = 0x7fffffff, T = 1;
      if (nmax > 0 && count(nmax) <= grid) {
        int lo = 1, hi = nmax;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (count(mid) <= grid) {
            hi = mid;
          } else {
            lo = mid + 1;
          }
        }
        T = lo;
        int big = 0;  // the largest piece
        for (int rt = lane; rt < RT; rt += 32) {
          const int n = n_rt[rt], ns = wave_splits(n, T);
          big = max(big, (n + ns - 1) / ns);
        }
        cost = warp_max(big) + kItemChunks;
      }
      if (lane == 0) {
        words[10] = cost;
        *plan_t = T;
      }
    }
    __syncthreads();
    const bool wave = words[10] < words[9];
    if (warp == 0 && wave) {  // the first item of each (rank, tile), in rank order
      const int T = *plan_t, per = (RT + 31) / 32, r0 = lane * per;
      int local = 0;
      for (int i = 0; i < per; ++i)
        if (r0 + i < RT) local += hgc * wave_splits(n_rt[r0 + i], T);
      int incl = local;
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int base = incl - local;
      for (int i = 0; i < per; ++i) {
        if (r0 + i < RT) {
          plan_off[r0 + i] = uint16_t(base);
          base += hgc * wave_splits(n_rt[r0 + i], T);
        }
      }
      if (lane == 31) *plan_items = incl;
    }
    if (tid == 0) {
      *plan_wave = wave ? 1 : 0;
      if (!wave) *plan_items = P.num_items;
    }
    dev::fence_async_smem();  // the scratch before the ring's first copy
  }
  if (tid == 0) {
    for (int s = 0; s < QM_ST; ++s) {
      dev::mbar_init(&full[s], 1);
      dev::mbar_init(&empty[s], 1);
    }
    for (int k = 0; k < 2; ++k) {
      dev::mbar_init(&qfull[k], 1);
      dev::mbar_init(&qempty[k], 1);
      dev::mbar_init(&bar_s[k], 1);
      dev::mbar_init(&bar_p[k], 128);
      dev::mbar_init(&bar_o[k], 1);
      dev::mbar_init(&oempty[k], 128);
    }
    dev::mbar_init(drain, 1);
    *abort_flag = 0;
    *issued = 0;
    *consumed = 0;
    *q_issued = 0;
    *q_waited = 0;
    dev::fence_barrier_init();
  }
  if (warp == 0) dev::tmem_alloc(tmem_slot, QM_TMEM_COLS);
  dev::tc_fence_before();
  __syncthreads();
  dev::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // The items of this CTA: pass j takes item j*grid + k (j even) or
  // j*grid + grid - 1 - k (j odd).
  const int grid = int(gridDim.x), k = int(blockIdx.x);
  auto item_index = [&](int j) { return j * grid + ((j & 1) ? grid - 1 - k : k); };
  auto item_of = [&](int j) {
    QmItem it;
    const int x = item_index(j);
    const bool wave = SPLIT && *plan_wave != 0;
    int hg = 0, sp = 0, ns = SPLIT ? P.splits : 1, rem = 0;
    if (wave) {  // (rank, tile), then head group, then split
      int lo = 0, hi = P.num_seqs * P.tiles - 1;  // the last (rank, tile) starting at or before x
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (int(plan_off[mid]) <= x) {
          lo = mid;
        } else {
          hi = mid - 1;
        }
      }
      it.b = order[lo / P.tiles];
      it.tile = lo % P.tiles;
      rem = x - int(plan_off[lo]);
    } else {  // rank, then head group, then tile, then split
      const int per_seq = P.head_groups * P.tiles * ns;
      const int rank = x / per_seq;
      rem = x % per_seq;
      it.b = ranked ? order[rank] : rank;
      hg = rem / (P.tiles * ns);
      it.tile = rem / ns % P.tiles;
      sp = rem % ns;
    }
    const int n_all = span_of(P.context_lens[it.b], it.tile, it);  // chunks of all the splits
    if (wave) {
      ns = wave_splits(n_all, *plan_t);
      hg = rem / ns;
      sp = rem % ns;
    }
    it.hg0 = hg * HB;
    it.split = sp;
    it.ns = ns;
    it.c0 = SPLIT ? sp * n_all / ns : 0;
    it.n = SPLIT ? (sp + 1) * n_all / ns - it.c0 : n_all;
    return it;
  };
  auto has_item = [&](int j) { return item_index(j) < (SPLIT ? *plan_items : P.num_items); };

  // Launched as a programmatic dependent (after the step's KV write, which
  // changes neither the tables, the lengths nor q): nothing above touched the
  // cache or the outputs, and the producer requests the first item's Q
  // before the dependency wait.
  int q_first = -1;  // producer lane 0: the item whose Q is already requested
  if (warp == 4 && lane == 0) {
    for (int j = 0; has_item(j); ++j) {
      const QmItem it = item_of(j);
      if (it.n == 0) continue;
      const uint64_t pol = dev::l2_evict_first_policy();
      dev::mbar_arrive_expect_tx(&qfull[0], QM_Q_BYTES);
      for (int h2 = 0; h2 < 2; ++h2)
        for (int h = 0; h < HB; ++h)
          dev::tma_load_4d(qbuf + h2 * QM_HALF_Q + h * RPH * 128, &tm_q, h2 * 64,
                           (it.hg0 + h) * G, it.tile * QT, it.b, &qfull[0], pol);
      *q_issued = 1;
      q_first = j;
      break;
    }
  }
  dev::griddep_wait();

  if (warp == 4) {
    // ---------------------------------------------------------- producer
    const uint64_t pol = dev::l2_evict_first_policy();
    if (lane == 0) {
      dev::prefetch_tmap(&tm_k);
      dev::prefetch_tmap(&tm_v);
      dev::prefetch_tmap(&tm_q);
    }
    // lane l < 4*NB issues one request of a chunk: block u = l/4, K or V,
    // one 64-d half (the TMA unit takes requests from several lanes at once)
    const int u = (lane >> 2) % NB, hf = (lane >> 1) & 1, kv = lane & 1;
    int gc = 0, qi = 0;
    bool ok = true;
    for (int j = 0; ok && has_item(j); ++j) {
      const QmItem it = item_of(j);
      if (it.n == 0) continue;
      const int nblk = it.nblk;
      if (lane == 0 && j != q_first) {
        // Q of this item into buffer qi % 2 once the scores of the item that
        // used it last have completed
        const int qb = qi & 1;
        ok = dev::mbar_wait_sleep(&qempty[qb], (uint32_t(qi >> 1) & 1u) ^ 1u, 64, P.wait_ns,
                                  abort_flag);
        if (ok) {
          dev::mbar_arrive_expect_tx(&qfull[qb], QM_Q_BYTES);
          for (int h2 = 0; h2 < 2; ++h2)
            for (int h = 0; h < HB; ++h)
              dev::tma_load_4d(qbuf + qb * QM_Q_BYTES + h2 * QM_HALF_Q + h * RPH * 128, &tm_q,
                               h2 * 64, (it.hg0 + h) * G, it.tile * QT, it.b, &qfull[qb], pol);
          *q_issued = qi + 1;
        }
      }
      ok = __shfl_sync(0xffffffffu, int(ok), 0) != 0;
      if (!ok) break;
      const int32_t* trow = P.block_tables + size_t(it.b) * P.max_blocks_per_seq;
      // lane l holds the table entry of block w0 + l
      auto window = [&](int w0) {
        const int jj = w0 + lane;
        return (jj < P.max_blocks_per_seq && jj < nblk) ? trow[jj] : -1;
      };
      int w0 = it.c0 * NB;  // the split's first block
      int win = window(w0);
      for (int c = 0; c < it.n; ++c, ++gc) {
        if ((it.c0 + c) * NB >= w0 + 32) {
          w0 += 32;
          win = window(w0);
        }
        const int slot = gc % QM_ST;
        if (lane == 0) {
          ok = dev::mbar_wait_sleep(&empty[slot], (uint32_t(gc / QM_ST) & 1u) ^ 1u, 64, P.wait_ns,
                                    abort_flag);
          if (ok) dev::mbar_arrive_expect_tx(&full[slot], QM_SLOT);
        }
        ok = __shfl_sync(0xffffffffu, int(ok), 0) != 0;
        if (!ok) break;
        const int jb = (it.c0 + c) * NB + u;
        const int e = __shfl_sync(0xffffffffu, win, jb - w0);
        if (lane < 4 * NB) {
          int row = P.oob_row;  // past the sequence (or a bad entry): zero fill
          if (jb < nblk) {
            if (e >= 0 && e < P.num_blocks) {
              row = (e * P.num_kv_heads + it.hg0) * BS;
            } else if (kv == 0 && hf == 0) {
              atomicOr(&g_tc_errors, PA_DEVERR_TABLE_ENTRY);
            }
          }
          unsigned char* dst =
              ring + size_t(slot) * QM_SLOT + kv * QM_KV_BYTES + hf * QM_HALF_KV + u * BR * 128;
          dev::tma_load_2d(dst, kv ? &tm_v : &tm_k, hf * 64, row, &full[slot], pol);
        }
        if (lane == 0) *issued = gc + 1;
      }
      ++qi;
    }
    if (!ok && lane == 0) {
      atomicOr(&g_tc_errors, PA_DEVERR_TIMEOUT);
      *abort_flag = 1;
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------- MMA issue
    if (lane == 0) {
      // Two cursors over the items: the scores (S) run up to two chunks ahead
      // of the value products (PV), across item boundaries.
      int js = 0, cs = 0, gs = 0, qs = 0;  // S: item, chunk in item, global chunk, Q uses
      int jv = 0, cv = 0, gv = 0, qv = 0;  // PV: the same, qv = O uses
      QmItem its{}, itv{};
      auto seek = [&](int& j, int& c, QmItem& it) {  // the next item with chunks
        while (has_item(j)) {
          it = item_of(j);
          if (c < it.n) return true;
          ++j;
          c = 0;
        }
        return false;
      };
      bool s_more = seek(js, cs, its), v_more = seek(jv, cv, itv);
      bool ok = true;
      uint64_t t_idle = 0;
      uint32_t idle = 0;
      const uint32_t idle_mask = P.wait_ns < dev::kShortWaitNs ? 0u : 255u;
      while (ok && v_more) {
        bool progress = false;
        // the value product of chunk gv once its P is written (and, on an
        // item's first chunk, once its O accumulator has been read out); it
        // goes before the next scores when both are ready, so that its ring
        // slot frees without waiting for them (an MMA issue blocks while the
        // pipe is busy)
        if (gv < gs && dev::mbar_test(&bar_p[gv & 1], uint32_t(gv >> 1) & 1u) &&
            (cv > 0 || dev::mbar_test(&oempty[qv & 1], (uint32_t(qv >> 1) & 1u) ^ 1u))) {
          dev::tc_fence_after();
          const uint32_t vb = dev::smem_addr(ring + size_t(gv % QM_ST) * QM_SLOT + QM_KV_BYTES);
          const uint32_t od = tmem + 2 * QM_KC + uint32_t(qv & 1) * QM_D;
#pragma unroll
          for (int kk = 0; kk < QM_KC / 16; ++kk)
            mma_bf16_tmem_a(od, tmem + QM_TMEM_P + uint32_t(gv & 1) * 32 + uint32_t(kk * 8),
                            // V MN-major: next 8 rows 1024 B on (SBO), second 64-d
                            // half one half on (LBO)
                            dev::smem_desc(vb + kk * 2048, QM_HALF_KV, 1024, dev::kSwizzle128B),
                            QM_IDESC_PV, cv > 0 || kk > 0);
          dev::mma_commit(&bar_o[gv & 1]);
          dev::mma_commit(&empty[gv % QM_ST]);
          *consumed = gv + 1;
          ++gv;
          if (++cv == itv.n) {
            ++qv;
            ++jv;
            cv = 0;
            v_more = seek(jv, cv, itv);
          }
          progress = true;
        }
        // the scores of chunk gs: it has landed, its Q is in, and the softmax
        // of chunk gs - 2 has read S[gs % 2] (its value product is issued)
        if (s_more && gs <= gv + 1 &&
            (cs > 0 || dev::mbar_test(&qfull[qs & 1], uint32_t(qs >> 1) & 1u)) &&
            dev::mbar_test(&full[gs % QM_ST], uint32_t(gs / QM_ST) & 1u)) {
          if (cs == 0) *q_waited = qs + 1;
          const uint32_t qb = dev::smem_addr(qbuf + (qs & 1) * QM_Q_BYTES);
          const uint32_t kb = dev::smem_addr(ring + size_t(gs % QM_ST) * QM_SLOT);
          dev::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < QM_D / 16; ++kk) {
            const uint32_t h2 = kk >> 2, off = uint32_t(kk & 3) * 32;
            dev::mma_bf16(tmem + uint32_t(gs & 1) * QM_KC,
                          dev::smem_desc(qb + h2 * QM_HALF_Q + off, 16, 1024, dev::kSwizzle128B),
                          dev::smem_desc(kb + h2 * QM_HALF_KV + off, 16, 1024, dev::kSwizzle128B),
                          QM_IDESC_S, kk > 0);
          }
          dev::mma_commit(&bar_s[gs & 1]);
          ++gs;
          if (++cs == its.n) {  // the item's last scores: its Q buffer frees when they complete
            dev::mma_commit(&qempty[qs & 1]);
            ++qs;
            ++js;
            cs = 0;
            s_more = seek(js, cs, its);
          }
          progress = true;
        }
        if (progress) {
          idle = 0;
          continue;
        }
        // bounded idle: the wall clock is read every 256 polls (every poll
        // under a budget short enough to run out in a test)
        if ((++idle & idle_mask) != 0u) continue;
        if (*abort_flag) {
          ok = false;
          break;
        }
        const uint64_t now = dev::global_timer_ns();
        if (idle == idle_mask + 1u) {
          t_idle = now;
        } else if (now - t_idle > P.wait_ns) {
          ok = false;
        }
      }
      if (!ok) {
        atomicOr(&g_tc_errors, PA_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      dev::mma_commit(drain);
      (void)dev::mbar_wait(drain, 0);
    }
  } else {
    // ---------------------------------------------------------- softmax
    const int r = tid;  // TMEM lane
    const int h = r / RPH, r0 = r % RPH;  // head of the group, row of the head
    const uint32_t t_lane = uint32_t(warp * 32) << 16;
    const float sl2 = P.scale_log2;
    int pv_done = -1, gc = 0, qi = 0;
    bool ok = true;
    // value product of chunk kc done (it completes bar_o[kc % 2], phase kc / 2)
    auto wait_pv = [&](int kc) {
      ok = __all_sync(0xffffffffu, dev::mbar_wait(&bar_o[kc & 1], uint32_t(kc >> 1) & 1u,
                                                  P.wait_ns, abort_flag)) &&
           ok;
      pv_done = kc;
    };
    for (int j = 0; ok && has_item(j); ++j) {
      const QmItem it = item_of(j);
      const int i = it.tile * QT + r0 / G;
      const bool valid = i < Q && it.hg0 + h < P.num_kv_heads;
      __nv_bfloat16* orow =
          P.out +
          ((size_t(it.b) * Q + (valid ? i : 0)) * P.num_q_heads + (it.hg0 + h) * G + r0 % G) *
              QM_D;
      if (r == 0 && it.bad_len && it.tile == 0 && it.hg0 == 0 && it.split == 0)
        atomicOr(&g_tc_errors, PA_DEVERR_CONTEXT_LEN);
      // this row's partials (with several splits)
      const size_t prow =
          SPLIT ? ((size_t(it.b) * Q + (valid ? i : 0)) * P.num_q_heads + (it.hg0 + h) * G +
                   r0 % G) * P.splits + it.split
                : 0;
      // a plan with fewer splits than the workspace holds: the last split
      // marks the row's remaining partials empty (the merge skips m = -inf)
      if (SPLIT && valid && it.split == it.ns - 1)
        for (int s2 = it.ns; s2 < P.splits; ++s2)
          P.part_ml[(prow - it.split + s2) * 2] = -INFINITY;
      if (it.n == 0) {  // no keys in this split (or an empty sequence)
        if (valid) {
          if (!SPLIT) {  // zero rows
#pragma unroll
            for (int cg = 0; cg < QM_D; cg += 8)
              *reinterpret_cast<uint4*>(orow + cg) = make_uint4(0u, 0u, 0u, 0u);
          } else {  // an empty partial: weight 2^-inf = 0 in the merge
            P.part_ml[prow * 2] = -INFINITY;
            P.part_ml[prow * 2 + 1] = 0.0f;
#pragma unroll
            for (int cg = 0; cg < QM_D; cg += 4)
              *reinterpret_cast<float4*>(P.part_o + prow * QM_D + cg) =
                  make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        continue;
      }
      const int L = it.L;
      const int L_row = valid ? L - Q + i + 1 : 0;
      const uint32_t o_col = 2 * QM_KC + uint32_t(qi & 1) * QM_D;
      float m_ref = -INFINITY, l = 0.0f;
      for (int c = 0; c < it.n; ++c) {
        const int g = gc + c;
        ok = __all_sync(0xffffffffu, dev::mbar_wait(&bar_s[g & 1], uint32_t(g >> 1) & 1u,
                                                    P.wait_ns, abort_flag));
        if (!ok) break;
        dev::tc_fence_after();
        // this thread's scores: block u of the chunk, BS columns at u*BR + h*BS
        float s[NC];
        {
          uint32_t raw[NC];
#pragma unroll
          for (int t = 0; t < NC / 16; ++t)  // 16 columns at a time
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, "
                "%10, %11, %12, %13, %14, %15}, [%16];"
                : "=r"(raw[16 * t + 0]), "=r"(raw[16 * t + 1]), "=r"(raw[16 * t + 2]),
                  "=r"(raw[16 * t + 3]), "=r"(raw[16 * t + 4]), "=r"(raw[16 * t + 5]),
                  "=r"(raw[16 * t + 6]), "=r"(raw[16 * t + 7]), "=r"(raw[16 * t + 8]),
                  "=r"(raw[16 * t + 9]), "=r"(raw[16 * t + 10]), "=r"(raw[16 * t + 11]),
                  "=r"(raw[16 * t + 12]), "=r"(raw[16 * t + 13]), "=r"(raw[16 * t + 14]),
                  "=r"(raw[16 * t + 15])
                : "r"(tmem + t_lane + uint32_t(g & 1) * QM_KC +
                      uint32_t(t / (BS / 16) * BR + h * BS + t % (BS / 16) * 16)));
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
          for (int kx = 0; kx < NC; ++kx) s[kx] = __uint_as_float(raw[kx]);
        }
        const int key0 = (it.c0 + c) * NB * BS;  // key of s[0]; s[kx] is key key0 + kx
        if (!__all_sync(0xffffffffu, key0 + NC <= L_row)) {
#pragma unroll
          for (int kx = 0; kx < NC; ++kx) s[kx] = key0 + kx < L_row ? s[kx] : -INFINITY;
        }
        // maximum of the raw scores (the scale is positive), four chains
        float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
        for (int kx = 4; kx < NC; ++kx) mx[kx & 3] = fmaxf(mx[kx & 3], s[kx]);
        const float cm = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
        // the reference moves only when a score exceeds it by more than 2^8
        const bool need = cm > m_ref + kRescaleLog2;
        if (__any_sync(0xffffffffu, need)) {
          const float nr = need ? cm : m_ref;
          const float f = nr == m_ref || m_ref == -INFINITY ? 1.0f : dev::fast_exp2(m_ref - nr);
          if (c > 0) {
            if (pv_done < g - 1) wait_pv(g - 1);
            if (!ok) break;
            dev::tc_fence_after();
#pragma unroll
            for (int cg = 0; cg < QM_D; cg += 32) {
              float o[32];
              dev::tmem_ld_cols<32>(tmem + t_lane + o_col + cg, o);
#pragma unroll
              for (int kx = 0; kx < 32; ++kx) o[kx] *= f;
              dev::tmem_st_cols<32>(tmem + t_lane + o_col + cg, o);
            }
          }
          l *= f;
          m_ref = nr;
        }
        // p = 2^(s * scale - m): masked scores give 2^-inf = 0; with no
        // reference yet every score is masked and the offset is moot
        const float nm = m_ref == -INFINITY ? 0.0f : -m_ref;
        uint32_t pw[NC / 2];
        float la = 0.0f, lb = 0.0f;
#pragma unroll
        for (int kx = 0; kx < NC; kx += 2) {
          const float p0 = dev::fast_exp2(fmaf(s[kx], sl2, nm));
          const float p1 = dev::fast_exp2(fmaf(s[kx + 1], sl2, nm));
          la += p0;
          lb += p1;
          const __nv_bfloat162 v2 = __floats2bfloat162_rn(p0, p1);
          pw[kx / 2] = *reinterpret_cast<const uint32_t*>(&v2);
        }
        l += la + lb;
        if ((it.c0 + c + 1) * NB * BS > it.keys) {
          // no row of the item sees the keys from it.keys on; past the
          // sequence, in its last block, they may hold anything (NaN
          // included). Clear their V rows so that 0 * V = 0. Thread r clears
          // row x = r % 64 of half r / 64: block x / BR, key x % BS.
          const int x = r % QM_KC, h2 = r / QM_KC;
          if (((it.c0 + c) * NB + x / BR) * BS + x % BS >= it.keys) {
            uint4* vrow = reinterpret_cast<uint4*>(ring + size_t(g % QM_ST) * QM_SLOT +
                                                   QM_KV_BYTES + h2 * QM_HALF_KV + x * 128);
#pragma unroll
            for (int kx = 0; kx < 8; ++kx) vrow[kx] = make_uint4(0u, 0u, 0u, 0u);
          }
          dev::fence_async_smem();  // before the value product reads the ring
        }
        // P[g % 2]: column m holds chunk columns 2m, 2m+1; block u's BS
        // columns of this head are P columns (u*BR + h*BS)/2 + [0, BS/2),
        // the rest zero. The value product of chunk g - 2 read this buffer last.
        if (g >= 2 && pv_done < g - 2) wait_pv(g - 2);
        if (!ok) break;
        {
          float pp[QM_KC / 2];
#pragma unroll
          for (int m = 0; m < QM_KC / 2; ++m) {
            const int u = 2 * m / BR, hh = 2 * m % BR / BS;  // block and head of P column m
            pp[m] = hh == h ? __uint_as_float(pw[u * BS / 2 + m % (BS / 2)]) : 0.0f;
          }
          dev::tmem_st_cols<QM_KC / 2>(tmem + t_lane + QM_TMEM_P + uint32_t(g & 1) * 32, pp);
        }
        dev::tc_fence_before();
        dev::mbar_arrive(&bar_p[g & 1]);
      }
      if (!ok) break;
      gc += it.n;
      wait_pv(gc - 1);
      if (!ok) break;
      dev::tc_fence_after();
      const float inv = l > 0.0f ? __frcp_rn(l) : 0.0f;
      if (SPLIT && valid) {
        P.part_ml[prow * 2] = m_ref;
        P.part_ml[prow * 2 + 1] = l;
      }
#pragma unroll
      for (int cg = 0; cg < QM_D; cg += 32) {
        float o[32];
        dev::tmem_ld_cols<32>(tmem + t_lane + o_col + cg, o);
        if (SPLIT) {  // the unnormalised row, relative to 2^m_ref
          if (valid)
#pragma unroll
            for (int kx = 0; kx < 32; kx += 4)
              *reinterpret_cast<float4*>(P.part_o + prow * QM_D + cg + kx) =
                  make_float4(o[kx], o[kx + 1], o[kx + 2], o[kx + 3]);
        } else if (valid) {
#pragma unroll
          for (int kx = 0; kx < 32; kx += 8) {
            uint32_t w[4];
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2) {
              const __nv_bfloat162 v2 =
                  __floats2bfloat162_rn(o[kx + 2 * q2] * inv, o[kx + 2 * q2 + 1] * inv);
              w[q2] = *reinterpret_cast<const uint32_t*>(&v2);
            }
            *reinterpret_cast<uint4*>(orow + cg + kx) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      // this O accumulator may take the item after next
      dev::tc_fence_before();
      dev::mbar_arrive(&oempty[qi & 1]);
      ++qi;
    }
    if (!ok && lane == 0) {
      atomicOr(&g_tc_errors, PA_DEVERR_TIMEOUT);
      *abort_flag = 1;
    }
  }

  __syncthreads();
  if (*abort_flag && tid == 0) {
    // every copy issued but not consumed lands before shared memory is released
    for (int c = *consumed; c < *issued; ++c)
      (void)dev::mbar_wait(&full[c % QM_ST], uint32_t(c / QM_ST) & 1u);
    for (int c = *q_waited; c < *q_issued; ++c)
      (void)dev::mbar_wait(&qfull[c & 1], uint32_t(c >> 1) & 1u);
  }
  dev::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    dev::tc_fence_after();
    dev::tmem_dealloc(tmem, QM_TMEM_COLS);
  }
}

// ------------------------------------------------------------ two tiles per item
// With one KV head per item and an even number of 128-row tiles per head
// (many rows, large batches), an item takes two tiles of a head: each chunk of
// keys is loaded once and serves both tiles' scores and value products, which
// halves the TMA requests. Eight softmax warps (two per TMEM lane quarter: warp
// w serves tile w / 4, lanes 32 * (w % 4) ..); TMEM holds S[tile][2] with P
// over the first 32 columns of its S buffer, and O[tile] (512 columns), so the
// scores of chunk g wait for the value product of chunk g - 2 of the same tile
// and an item's first value product for its tile's previous read-out. Q of
// both tiles (64 KiB) is one buffer, loaded once the previous item's scores
// have completed.
constexpr int QD_THREADS = 320;  // softmax warps 0-7, producer 8, MMA 9
constexpr int QD_OFF_Q = 0;
constexpr int QD_OFF_RING = QD_OFF_Q + 2 * QM_Q_BYTES;
constexpr int QD_OFF_BARS = QD_OFF_RING + QM_ST * QM_SLOT;
// full[ST], empty[ST], qfull, qempty, s[2][2], p[2][2], o[2][2], oempty[2], drain
constexpr int QD_NBARS = 2 * QM_ST + 17;
constexpr int QD_OFF_WORDS = QD_OFF_BARS + QD_NBARS * 8;
constexpr int QD_OFF_ORDER = QD_OFF_WORDS + 64;
constexpr int QD_SMEM = QD_OFF_ORDER + 1024 + 1024;  // + alignment slack
static_assert(QD_SMEM <= kMaxDynSmem, "shared memory budget");
constexpr uint32_t QD_TMEM_O = 256;  // S[t][b] at t*128 + b*64, O[t] at 256 + t*128

template <int G, int BS>
__global__ void __launch_bounds__(QD_THREADS, 1)
    query_major_dual_kernel(const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v,
                            const __grid_constant__ CUtensorMap tm_q, const QmParams P) {
  constexpr int QT = QM_ROWS / G;  // new tokens per tile
  constexpr int NB = QM_KC / BS;   // blocks per chunk
  constexpr int NC = QM_KC;        // scores of a chunk per thread
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* qbuf = smem + QD_OFF_Q;  // tile t at t * QM_Q_BYTES
  unsigned char* ring = smem + QD_OFF_RING;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + QD_OFF_BARS);
  uint64_t* full = bars;
  uint64_t* empty = bars + QM_ST;
  uint64_t* qfull = bars + 2 * QM_ST;  // both tiles' Q landed
  uint64_t* qempty = qfull + 1;        // the previous item's scores completed
  uint64_t* bar_s = qempty + 1;        // [t * 2 + c % 2] scores of chunk c, tile t
  uint64_t* bar_p = bar_s + 4;         // [t * 2 + c % 2] P of chunk c, tile t, written
  uint64_t* bar_o = bar_p + 4;         // [t * 2 + c % 2] value product of chunk c, tile t
  uint64_t* oempty = bar_o + 4;        // [t] tile t's O read out
  uint64_t* drain = oempty + 2;
  int* words = reinterpret_cast<int*>(smem + QD_OFF_WORDS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&words[0]);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&words[1]);
  int* issued = &words[2];    // K/V chunks requested
  int* consumed = &words[3];  // K/V chunks whose two value products were issued
  int* q_issued = &words[4];  // Q loads requested
  int* q_waited = &words[5];  // Q loads seen landed
  int* order = reinterpret_cast<int*>(smem + QD_OFF_ORDER);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Q = P.q_len;
  const bool ranked = P.num_seqs <= QM_MAX_RANKED;
  const int pairs = P.tiles / 2;

  if (ranked) {  // sequences by decreasing length, as in query_major_kernel
    int* lens_s = reinterpret_cast<int*>(ring);
    for (int v = tid; v < P.num_seqs; v += QD_THREADS) lens_s[v] = P.context_lens[v];
    __syncthreads();
    for (int v = tid; v < P.num_seqs; v += QD_THREADS) {
      const int Lv = lens_s[v];
      int above = 0;
      for (int u = 0; u < P.num_seqs; ++u) {
        const int Lu = lens_s[u];
        above += Lu > Lv || (Lu == Lv && u < v);
      }
      order[above] = v;
    }
    dev::fence_async_smem();
  }
  if (tid == 0) {
    for (int s = 0; s < QM_ST; ++s) {
      dev::mbar_init(&full[s], 1);
      dev::mbar_init(&empty[s], 1);
    }
    dev::mbar_init(qfull, 1);
    dev::mbar_init(qempty, 1);
    for (int k = 0; k < 4; ++k) {
      dev::mbar_init(&bar_s[k], 1);
      dev::mbar_init(&bar_p[k], 128);
      dev::mbar_init(&bar_o[k], 1);
    }
    dev::mbar_init(&oempty[0], 128);
    dev::mbar_init(&oempty[1], 128);
    dev::mbar_init(drain, 1);
    *abort_flag = 0;
    *issued = 0;
    *consumed = 0;
    *q_issued = 0;
    *q_waited = 0;
    dev::fence_barrier_init();
  }
  if (warp == 0) dev::tmem_alloc(tmem_slot, QM_TMEM_COLS);
  dev::tc_fence_before();
  __syncthreads();
  dev::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int grid = int(gridDim.x), k = int(blockIdx.x);
  auto item_index = [&](int j) { return j * grid + ((j & 1) ? grid - 1 - k : k); };
  auto item_of = [&](int j) {  // tile = the pair's first tile
    QmItem it;
    const int x = item_index(j);
    const int per_seq = P.num_kv_heads * pairs;
    const int rank = x / per_seq, rem = x % per_seq;
    it.b = ranked ? order[rank] : rank;
    it.hg0 = rem / pairs;
    it.tile = rem % pairs * 2;
    it.split = 0;
    it.c0 = 0;
    int L = P.context_lens[it.b];
    it.bad_len = L > P.cap;
    if (L > P.cap) L = P.cap;
    if (L > 0 && L < Q) {
      it.bad_len = true;
      L = 0;
    }
    it.L = L;
    const int i_last = min(Q, (it.tile + 2) * QT) - 1;  // the second tile's last new token
    const int keys = L > 0 ? L - Q + i_last + 1 : 0;
    it.keys = keys;
    it.nblk = (keys + BS - 1) / BS;
    it.n = (it.nblk + NB - 1) / NB;
    return it;
  };
  auto has_item = [&](int j) { return item_index(j) < P.num_items; };
  auto load_q = [&](const QmItem& it, uint64_t pol) {  // both tiles, by one thread
    dev::mbar_arrive_expect_tx(qfull, 2 * QM_Q_BYTES);
    for (int t = 0; t < 2; ++t)
      for (int h2 = 0; h2 < 2; ++h2)
        dev::tma_load_4d(qbuf + t * QM_Q_BYTES + h2 * QM_HALF_Q, &tm_q, h2 * 64, it.hg0 * G,
                         (it.tile + t) * QT, it.b, qfull, pol);
  };

  int q_first = -1;  // producer lane 0: the item whose Q is already requested
  if (warp == 8 && lane == 0) {
    for (int j = 0; has_item(j); ++j) {
      const QmItem it = item_of(j);
      if (it.n == 0) continue;
      load_q(it, dev::l2_evict_first_policy());
      *q_issued = 1;
      q_first = j;
      break;
    }
  }
  dev::griddep_wait();

  if (warp == 8) {
    // ---------------------------------------------------------- producer
    const uint64_t pol = dev::l2_evict_first_policy();
    if (lane == 0) {
      dev::prefetch_tmap(&tm_k);
      dev::prefetch_tmap(&tm_v);
    }
    const int u = (lane >> 2) % NB, hf = (lane >> 1) & 1, kv = lane & 1;
    int gc = 0, qi = 0;
    bool ok = true;
    for (int j = 0; ok && has_item(j); ++j) {
      const QmItem it = item_of(j);
      if (it.n == 0) continue;
      if (lane == 0 && j != q_first) {
        // the single Q buffer, once the previous item's scores have completed
        ok = dev::mbar_wait_sleep(qempty, uint32_t(qi - 1) & 1u, 64, P.wait_ns, abort_flag);
        if (ok) {
          load_q(it, pol);
          *q_issued = qi + 1;
        }
      }
      ok = __shfl_sync(0xffffffffu, int(ok), 0) != 0;
      if (!ok) break;
      const int32_t* trow = P.block_tables + size_t(it.b) * P.max_blocks_per_seq;
      auto window = [&](int w0) {
        const int jj = w0 + lane;
        return (jj < P.max_blocks_per_seq && jj < it.nblk) ? trow[jj] : -1;
      };
      int w0 = 0;
      int win = window(0);
      for (int c = 0; c < it.n; ++c, ++gc) {
        if (c * NB >= w0 + 32) {
          w0 += 32;
          win = window(w0);
        }
        const int slot = gc % QM_ST;
        if (lane == 0) {
          ok = dev::mbar_wait_sleep(&empty[slot], (uint32_t(gc / QM_ST) & 1u) ^ 1u, 64, P.wait_ns,
                                    abort_flag);
          if (ok) dev::mbar_arrive_expect_tx(&full[slot], QM_SLOT);
        }
        ok = __shfl_sync(0xffffffffu, int(ok), 0) != 0;
        if (!ok) break;
        const int jb = c * NB + u;
        const int e = __shfl_sync(0xffffffffu, win, jb - w0);
        if (lane < 4 * NB) {
          int row = P.oob_row;
          if (jb < it.nblk) {
            if (e >= 0 && e < P.num_blocks) {
              row = (e * P.num_kv_heads + it.hg0) * BS;
            } else if (kv == 0 && hf == 0) {
              atomicOr(&g_tc_errors, PA_DEVERR_TABLE_ENTRY);
            }
          }
          unsigned char* dst =
              ring + size_t(slot) * QM_SLOT + kv * QM_KV_BYTES + hf * QM_HALF_KV + u * BS * 128;
          dev::tma_load_2d(dst, kv ? &tm_v : &tm_k, hf * 64, row, &full[slot], pol);
        }
        if (lane == 0) *issued = gc + 1;
      }
      ++qi;
    }
    if (!ok && lane == 0) {
      atomicOr(&g_tc_errors, PA_DEVERR_TIMEOUT);
      *abort_flag = 1;
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------- MMA issue
    if (lane == 0) {
      // One S cursor (both tiles' scores together) and one PV cursor per tile.
      int js = 0, cs = 0, gs = 0, qs = 0;
      int jv[2] = {0, 0}, cv[2] = {0, 0}, gv[2] = {0, 0}, qv[2] = {0, 0};
      QmItem its{}, itv[2] = {};
      auto seek = [&](int& j, int& c, QmItem& it) {
        while (has_item(j)) {
          it = item_of(j);
          if (c < it.n) return true;
          ++j;
          c = 0;
        }
        return false;
      };
      bool s_more = seek(js, cs, its);
      bool v_more[2] = {seek(jv[0], cv[0], itv[0]), seek(jv[1], cv[1], itv[1])};
      bool ok = true;
      uint64_t t_idle = 0;
      uint32_t idle = 0;
      const uint32_t idle_mask = P.wait_ns < dev::kShortWaitNs ? 0u : 255u;
      auto pv_done = [&](int t, int c) {  // value product of chunk c, tile t, completed
        return c < 0 || dev::mbar_test(&bar_o[t * 2 + (c & 1)], uint32_t(c >> 1) & 1u);
      };
      while (ok && (v_more[0] || v_more[1])) {
        bool progress = false;
        // the value product of chunk gv[t] of tile t once its P is written
        // (and, on an item's first chunk, once tile t's O has been read out);
        // a ring slot frees when both tiles' value products of its chunk are in.
        // They go before the next scores when both are ready (an MMA issue
        // blocks while the pipe is busy).
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int g = gv[t];
          if (v_more[t] && g < gs &&
              dev::mbar_test(&bar_p[t * 2 + (g & 1)], uint32_t(g >> 1) & 1u) &&
              (cv[t] > 0 || qv[t] == 0 ||
               dev::mbar_test(&oempty[t], uint32_t(qv[t] - 1) & 1u))) {
            dev::tc_fence_after();
            const uint32_t vb = dev::smem_addr(ring + size_t(g % QM_ST) * QM_SLOT + QM_KV_BYTES);
#pragma unroll
            for (int kk = 0; kk < QM_KC / 16; ++kk)
              mma_bf16_tmem_a(tmem + QD_TMEM_O + uint32_t(t * QM_D),
                              tmem + uint32_t(t * 128 + (g & 1) * QM_KC + kk * 8),
                              dev::smem_desc(vb + kk * 2048, QM_HALF_KV, 1024, dev::kSwizzle128B),
                              QM_IDESC_PV, cv[t] > 0 || kk > 0);
            dev::mma_commit(&bar_o[t * 2 + (g & 1)]);
            ++gv[t];
            if (gv[1 - t] > g) {  // the other tile's value product of chunk g is in too
              dev::mma_commit(&empty[g % QM_ST]);
              *consumed = g + 1;
            }
            if (++cv[t] == itv[t].n) {
              ++qv[t];
              ++jv[t];
              cv[t] = 0;
              v_more[t] = seek(jv[t], cv[t], itv[t]);
            }
            progress = true;
          }
        }
        // scores of chunk gs for both tiles: it has landed, the item's Q is in,
        // and each tile's value product of chunk gs - 2 (which read P from
        // the same S buffer) has completed
        if (s_more && gs <= min(gv[0], gv[1]) + 1 && pv_done(0, gs - 2) && pv_done(1, gs - 2) &&
            (cs > 0 || dev::mbar_test(qfull, uint32_t(qs) & 1u)) &&
            dev::mbar_test(&full[gs % QM_ST], uint32_t(gs / QM_ST) & 1u)) {
          if (cs == 0) *q_waited = qs + 1;
          const uint32_t kb = dev::smem_addr(ring + size_t(gs % QM_ST) * QM_SLOT);
          dev::tc_fence_after();
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const uint32_t qb = dev::smem_addr(qbuf + t * QM_Q_BYTES);
#pragma unroll
            for (int kk = 0; kk < QM_D / 16; ++kk) {
              const uint32_t h2 = kk >> 2, off = uint32_t(kk & 3) * 32;
              dev::mma_bf16(tmem + uint32_t(t * 128 + (gs & 1) * QM_KC),
                            dev::smem_desc(qb + h2 * QM_HALF_Q + off, 16, 1024, dev::kSwizzle128B),
                            dev::smem_desc(kb + h2 * QM_HALF_KV + off, 16, 1024,
                                           dev::kSwizzle128B),
                            QM_IDESC_S, kk > 0);
            }
            dev::mma_commit(&bar_s[t * 2 + (gs & 1)]);
          }
          ++gs;
          if (++cs == its.n) {  // the item's last scores: the Q buffer frees when they complete
            dev::mma_commit(qempty);
            ++qs;
            ++js;
            cs = 0;
            s_more = seek(js, cs, its);
          }
          progress = true;
        }
        if (progress) {
          idle = 0;
          continue;
        }
        if ((++idle & idle_mask) != 0u) continue;
        if (*abort_flag) {
          ok = false;
          break;
        }
        const uint64_t now = dev::global_timer_ns();
        if (idle == idle_mask + 1u) {
          t_idle = now;
        } else if (now - t_idle > P.wait_ns) {
          ok = false;
        }
      }
      if (!ok) {
        atomicOr(&g_tc_errors, PA_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      dev::mma_commit(drain);
      (void)dev::mbar_wait(drain, 0);
    }
  } else {
    // ---------------------------------------------------------- softmax
    const int t = warp >> 2;                // tile of the item
    const int r = (warp & 3) * 32 + lane;   // TMEM lane = row of the tile
    const uint32_t t_lane = uint32_t((warp & 3) * 32) << 16;
    const uint32_t s_col = uint32_t(t * 128), o_col = QD_TMEM_O + uint32_t(t * QM_D);
    const float sl2 = P.scale_log2;
    int pv_done = -1, gc = 0;
    bool ok = true;
    auto wait_pv = [&](int kc) {  // value product of chunk kc, tile t
      ok = __all_sync(0xffffffffu, dev::mbar_wait(&bar_o[t * 2 + (kc & 1)], uint32_t(kc >> 1) & 1u,
                                                  P.wait_ns, abort_flag)) &&
           ok;
      pv_done = kc;
    };
    for (int j = 0; ok && has_item(j); ++j) {
      const QmItem it = item_of(j);
      const int i = (it.tile + t) * QT + r / G;
      const bool valid = i < Q;
      __nv_bfloat16* orow =
          P.out + ((size_t(it.b) * Q + (valid ? i : 0)) * P.num_q_heads + it.hg0 * G + r % G) * QM_D;
      if (r == 0 && t == 0 && it.bad_len && it.tile == 0 && it.hg0 == 0)
        atomicOr(&g_tc_errors, PA_DEVERR_CONTEXT_LEN);
      if (it.n == 0) {  // an empty sequence: zero rows
        if (valid)
#pragma unroll
          for (int cg = 0; cg < QM_D; cg += 8)
            *reinterpret_cast<uint4*>(orow + cg) = make_uint4(0u, 0u, 0u, 0u);
        continue;
      }
      const int L = it.L;
      const int L_row = valid ? L - Q + i + 1 : 0;
      float m_ref = -INFINITY, l = 0.0f;
      for (int c = 0; c < it.n; ++c) {
        const int g = gc + c;
        ok = __all_sync(0xffffffffu, dev::mbar_wait(&bar_s[t * 2 + (g & 1)], uint32_t(g >> 1) & 1u,
                                                    P.wait_ns, abort_flag));
        if (!ok) break;
        dev::tc_fence_after();
        float s[NC];
        dev::tmem_ld_cols<NC>(tmem + t_lane + s_col + uint32_t((g & 1) * QM_KC), s);
        const int key0 = c * QM_KC;  // key of s[0]
        if (!__all_sync(0xffffffffu, key0 + NC <= L_row)) {
#pragma unroll
          for (int kx = 0; kx < NC; ++kx) s[kx] = key0 + kx < L_row ? s[kx] : -INFINITY;
        }
        float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
        for (int kx = 4; kx < NC; ++kx) mx[kx & 3] = fmaxf(mx[kx & 3], s[kx]);
        const float cm = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
        const bool need = cm > m_ref + kRescaleLog2;
        if (__any_sync(0xffffffffu, need)) {
          const float nr = need ? cm : m_ref;
          const float f = nr == m_ref || m_ref == -INFINITY ? 1.0f : dev::fast_exp2(m_ref - nr);
          if (c > 0) {
            if (pv_done < g - 1) wait_pv(g - 1);
            if (!ok) break;
            dev::tc_fence_after();
#pragma unroll
            for (int cg = 0; cg < QM_D; cg += 32) {
              float o[32];
              dev::tmem_ld_cols<32>(tmem + t_lane + o_col + cg, o);
#pragma unroll
              for (int kx = 0; kx < 32; ++kx) o[kx] *= f;
              dev::tmem_st_cols<32>(tmem + t_lane + o_col + cg, o);
            }
          }
          l *= f;
          m_ref = nr;
        }
        const float nm = m_ref == -INFINITY ? 0.0f : -m_ref;
        float pp[NC / 2];
        float la = 0.0f, lb = 0.0f;
#pragma unroll
        for (int kx = 0; kx < NC; kx += 2) {
          const float p0 = dev::fast_exp2(fmaf(s[kx], sl2, nm));
          const float p1 = dev::fast_exp2(fmaf(s[kx + 1], sl2, nm));
          la += p0;
          lb += p1;
          const __nv_bfloat162 v2 = __floats2bfloat162_rn(p0, p1);
          pp[kx / 2] = __uint_as_float(*reinterpret_cast<const uint32_t*>(&v2));
        }
        l += la + lb;
        if ((c + 1) * QM_KC > it.keys) {
          // no row of the item sees the keys from it.keys on (past the
          // sequence they may hold NaN): clear their V rows, both tiles'
          // threads alike, before either value product reads them
          const int x = r % QM_KC, h2 = r / QM_KC;
          if (c * QM_KC + x >= it.keys) {
            uint4* vrow = reinterpret_cast<uint4*>(ring + size_t(g % QM_ST) * QM_SLOT +
                                                   QM_KV_BYTES + h2 * QM_HALF_KV + x * 128);
#pragma unroll
            for (int kx = 0; kx < 8; ++kx) vrow[kx] = make_uint4(0u, 0u, 0u, 0u);
          }
          dev::fence_async_smem();
        }
        // P over the first 32 columns of S[t][g % 2] (the scores are in
        // registers); the value product of chunk g - 2, which read this
        // buffer's last P, completed before S(g) was issued
        dev::tmem_st_cols<NC / 2>(tmem + t_lane + s_col + uint32_t((g & 1) * QM_KC), pp);
        dev::tc_fence_before();
        dev::mbar_arrive(&bar_p[t * 2 + (g & 1)]);
      }
      if (!ok) break;
      gc += it.n;
      wait_pv(gc - 1);
      if (!ok) break;
      dev::tc_fence_after();
      const float inv = l > 0.0f ? __frcp_rn(l) : 0.0f;
#pragma unroll
      for (int cg = 0; cg < QM_D; cg += 32) {
        float o[32];
        dev::tmem_ld_cols<32>(tmem + t_lane + o_col + cg, o);
        if (valid) {
#pragma unroll
          for (int kx = 0; kx < 32; kx += 8) {
            uint32_t w[4];
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2) {
              const __nv_bfloat162 v2 =
                  __floats2bfloat162_rn(o[kx + 2 * q2] * inv, o[kx + 2 * q2 + 1] * inv);
              w[q2] = *reinterpret_cast<const uint32_t*>(&v2);
            }
            *reinterpret_cast<uint4*>(orow + cg + kx) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      // tile t's O may take the next item
      dev::tc_fence_before();
      dev::mbar_arrive(&oempty[t]);
    }
    if (!ok && lane == 0) {
      atomicOr(&g_tc_errors, PA_DEVERR_TIMEOUT);
      *abort_flag = 1;
    }
  }

  __syncthreads();
  if (*abort_flag && tid == 0) {
    for (int c = *consumed; c < *issued; ++c)
      (void)dev::mbar_wait(&full[c % QM_ST], uint32_t(c / QM_ST) & 1u);
    for (int c = *q_waited; c < *q_issued; ++c) (void)dev::mbar_wait(qfull, uint32_t(c) & 1u);
  }
  dev::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    dev::tc_fence_after();
    dev::tmem_dealloc(tmem, QM_TMEM_COLS);
  }
}

// One warp per output row: the splits' partials weighted by 2^(m_s - M)
// (M the largest reference; a split that saw no key has m = -inf), the sum
// divided by the weighted sums.
__global__ void __launch_bounds__(128)
    query_major_merge_kernel(const float* __restrict__ part_ml, const float* __restrict__ part_o,
                             __nv_bfloat16* __restrict__ out, int rows, int splits) {
  const int row = int(blockIdx.x) * 4 + int(threadIdx.x >> 5), lane = int(threadIdx.x & 31);
  if (row >= rows) return;
  const float* ml = part_ml + size_t(row) * splits * 2;
  float M = -INFINITY;
  for (int sp = 0; sp < splits; ++sp) M = fmaxf(M, ml[sp * 2]);
  float acc[4] = {0.f, 0.f, 0.f, 0.f}, lsum = 0.0f;
  if (M != -INFINITY) {
    for (int sp = 0; sp < splits; ++sp) {
      const float m = ml[sp * 2];
      if (m == -INFINITY) continue;
      const float wgt = dev::fast_exp2(m - M);
      lsum += wgt * ml[sp * 2 + 1];
      const float4 o =
          *reinterpret_cast<const float4*>(part_o + (size_t(row) * splits + sp) * QM_D + lane * 4);
      acc[0] += wgt * o.x;
      acc[1] += wgt * o.y;
      acc[2] += wgt * o.z;
      acc[3] += wgt * o.w;
    }
  }
  const float inv = lsum > 0.0f ? __frcp_rn(lsum) : 0.0f;
  const __nv_bfloat162 a = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
  const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
  uint2 w;
  w.x = *reinterpret_cast<const uint32_t*>(&a);
  w.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(out + size_t(row) * QM_D + lane * 4) = w;
}

template <int G, int HB, bool SPLIT, int BS>
int launch_qm_t(const pa_decode_params* p, cudaStream_t stream, float* part_ml, float* part_o,
                bool dependent) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(query_major_kernel<G, HB, SPLIT, BS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, QM_SMEM);
    if (e != cudaSuccess) return int(e);
    configured = true;
  }
  const int H = p->num_kv_heads, Q = query_len_of(p);
  const uint64_t cache_rows = uint64_t(p->num_blocks) * H * BS;
  CUtensorMap tk, tv, tq;
  // K, V [rows][128 d]: a box of HB heads x BS keys of one block, one 64-d half
  int r = make_map(&tk, p->k_cache, cache_rows, QM_D, uint32_t(BS * HB));
  if (!r) r = make_map(&tv, p->v_cache, cache_rows, QM_D, uint32_t(BS * HB));
  if (!r) {
    // q [B][Q][Hq][128]: box (64 d, G heads, QT tokens, 1 sequence)
    const cuuint64_t dims[4] = {uint64_t(QM_D), uint64_t(p->num_q_heads), uint64_t(Q),
                                uint64_t(p->num_seqs)};
    const cuuint64_t strides[3] = {uint64_t(QM_D) * 2, uint64_t(p->num_q_heads) * QM_D * 2,
                                   uint64_t(Q) * p->num_q_heads * QM_D * 2};
    const cuuint32_t box[4] = {64, uint32_t(G), uint32_t(QM_ROWS / (HB * G)), 1};
    r = make_map_nd(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p->q, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (r) return r;
  QmParams P;
  P.block_tables = p->block_tables;
  P.context_lens = p->context_lens;
  P.out = static_cast<__nv_bfloat16*>(p->out);
  P.num_seqs = p->num_seqs;
  P.num_kv_heads = H;
  P.num_q_heads = p->num_q_heads;
  P.q_len = Q;
  P.tiles = query_major_tiles(p);
  P.head_groups = H / HB;
  P.splits = query_major_splits(p);
  if ((P.splits > 1) != SPLIT || (SPLIT && (!part_ml || !part_o)))
    return int(cudaErrorInvalidValue);
  P.part_ml = part_ml;
  P.part_o = part_o;
  P.num_items = p->num_seqs * P.head_groups * P.tiles * P.splits;
  P.max_blocks_per_seq = p->max_blocks_per_seq;
  P.num_blocks = p->num_blocks;
  P.cap = std::min(p->max_blocks_per_seq * BS, p->max_context_len);
  P.oob_row = int(cache_rows);
  P.scale_log2 = p->scale * kLog2e;
  P.wait_ns = p->wait_timeout_us > 0 ? uint64_t(p->wait_timeout_us) * 1000u : dev::kWaitNsLimit;
  const int sms = tc_grid();
  if (sms <= 0) return int(cudaErrorInvalidDevice);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = dependent ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  // split launches take every SM: the one-wave plan may cut more items
  cfg.gridDim =
      dim3(unsigned(SPLIT ? std::min(sms, QM_MAX_SPLIT_GRID) : std::min(P.num_items, sms)));
  cfg.blockDim = dim3(QM_THREADS);
  cfg.dynamicSmemBytes = QM_SMEM;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int e = int(cudaLaunchKernelEx(&cfg, query_major_kernel<G, HB, SPLIT, BS>, tk, tv, tq, P));
  if (e || P.splits == 1) return e;
  const int rows = p->num_seqs * Q * p->num_q_heads;
  query_major_merge_kernel<<<unsigned((rows + 3) / 4), 128, 0, stream>>>(
      part_ml, part_o, P.out, rows, P.splits);
  return int(cudaGetLastError());
}

template <int G, int BS>
int launch_qd_t(const pa_decode_params* p, cudaStream_t stream, bool dependent) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(query_major_dual_kernel<G, BS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, QD_SMEM);
    if (e != cudaSuccess) return int(e);
    configured = true;
  }
  const int H = p->num_kv_heads, Q = query_len_of(p);
  const uint64_t cache_rows = uint64_t(p->num_blocks) * H * BS;
  CUtensorMap tk, tv, tq;
  int r = make_map(&tk, p->k_cache, cache_rows, QM_D, uint32_t(BS));
  if (!r) r = make_map(&tv, p->v_cache, cache_rows, QM_D, uint32_t(BS));
  if (!r) {
    const cuuint64_t dims[4] = {uint64_t(QM_D), uint64_t(p->num_q_heads), uint64_t(Q),
                                uint64_t(p->num_seqs)};
    const cuuint64_t strides[3] = {uint64_t(QM_D) * 2, uint64_t(p->num_q_heads) * QM_D * 2,
                                   uint64_t(Q) * p->num_q_heads * QM_D * 2};
    const cuuint32_t box[4] = {64, uint32_t(G), uint32_t(QM_ROWS / G), 1};
    r = make_map_nd(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p->q, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (r) return r;
  QmParams P;
  P.block_tables = p->block_tables;
  P.context_lens = p->context_lens;
  P.out = static_cast<__nv_bfloat16*>(p->out);
  P.num_seqs = p->num_seqs;
  P.num_kv_heads = H;
  P.num_q_heads = p->num_q_heads;
  P.q_len = Q;
  P.tiles = query_major_tiles(p);
  P.head_groups = H;
  P.splits = 1;
  P.part_ml = nullptr;
  P.part_o = nullptr;
  P.num_items = p->num_seqs * H * (P.tiles / 2);
  P.max_blocks_per_seq = p->max_blocks_per_seq;
  P.num_blocks = p->num_blocks;
  P.cap = std::min(p->max_blocks_per_seq * BS, p->max_context_len);
  P.oob_row = int(cache_rows);
  P.scale_log2 = p->scale * kLog2e;
  P.wait_ns = p->wait_timeout_us > 0 ? uint64_t(p->wait_timeout_us) * 1000u : dev::kWaitNsLimit;
  const int sms = tc_grid();
  if (sms <= 0) return int(cudaErrorInvalidDevice);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = dependent ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(std::min(P.num_items, sms)));
  cfg.blockDim = dim3(QD_THREADS);
  cfg.dynamicSmemBytes = QD_SMEM;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return int(cudaLaunchKernelEx(&cfg, query_major_dual_kernel<G, BS>, tk, tv, tq, P));
}

template <int G, int BS>
int launch_qm_b(const pa_decode_params* p, cudaStream_t stream, float* ml, float* o, bool a) {
  const bool split = query_major_splits(p) > 1;
  if (query_major_heads(p) == 2)
    return split ? launch_qm_t<G, 2, true, BS>(p, stream, ml, o, a)
                 : launch_qm_t<G, 2, false, BS>(p, stream, ml, o, a);
  if (split) return launch_qm_t<G, 1, true, BS>(p, stream, ml, o, a);
  // one head per item: an even number of tiles per head goes two tiles at a time
  if (query_major_tiles(p) % 2 == 0) return launch_qd_t<G, BS>(p, stream, a);
  return launch_qm_t<G, 1, false, BS>(p, stream, ml, o, a);
}
template <int G>
int launch_qm_g(const pa_decode_params* p, cudaStream_t stream, float* ml, float* o, bool a) {
  return p->block_size == 32 ? launch_qm_b<G, 32>(p, stream, ml, o, a)
                             : launch_qm_b<G, 16>(p, stream, ml, o, a);
}

}  // namespace

int launch_query_major_tc(const pa_decode_params* p, void* stream, float* part_ml,
                          float* part_o, bool dependent) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (p->num_q_heads / p->num_kv_heads) {
    case 1: return launch_qm_g<1>(p, s, part_ml, part_o, dependent);
    case 2: return launch_qm_g<2>(p, s, part_ml, part_o, dependent);
    case 4: return launch_qm_g<4>(p, s, part_ml, part_o, dependent);
    case 8: return launch_qm_g<8>(p, s, part_ml, part_o, dependent);
    default: return int(cudaErrorInvalidValue);
  }
}

int read_and_clear_query_major_errors(uint32_t* flags) {
  return read_and_clear_tc_error_word(flags);
}

}  // namespace pa
