// Several new tokens per sequence on the tensor cores, query-major: one CTA per
// (sequence, group of HB KV heads, tile of query rows) streams those heads'
// blocks once for all their rows ("How Paged Attention and Continuous Batching
// Actually Work", §Continuous batching: the scheduled tokens of one request,
// as in a chunked prefill). A row is new token i of query head (kv head)*G + g
// and sees the sequence's first L - Q + i + 1 keys.
//
// The column-group decode (pa_decode_tc.cuh) puts the keys on the MMAs' M side
// and streams them once per group of new tokens; with many new tokens each
// group re-reads the keys. Here the queries are on the M side:
//   S[128 rows][64 columns]  = Q . K^T     (A = Q, B = K chunk, both K-major)
//   O[128 rows][128 d]      += P . V       (A = P from TMEM; B = V, MN-major)
// with S double-buffered and O in TMEM (256 columns). P (bf16, two to a
// 32-bit column) overwrites the first 32 columns of its chunk's S buffer and
// feeds the value product from there, so shared memory holds Q and the K/V
// ring only. A thread owns a row: its softmax (running maximum, sum, the
// conditional rescale of its O row) needs no other thread.
//
// Layout of a tile's 128 rows (TMEM lanes): R copies x HB heads x RPH rows,
// row r0 of a head being token tile*QT + r0/G, query head g = r0 % G.
//  * A chunk's 64 columns are NB = 4/HB blocks x HB heads x 16 keys: one
//    2-D tensor-map box [HB*16 rows][64 d] per block and 64-d half (the HB
//    heads of a block are adjacent in the cache), so with HB = 2 every TMA
//    request moves 4 KiB (the TMA unit's fixed cost per request caps 2 KiB
//    requests well below the HBM rate). A row's scores against the other
//    heads' keys are computed and ignored: its P row is zero there.
//  * With at most 32 (or 64) rows per head-group the rows are held R = 2 (or
//    4) times over; copy q takes blocks [q*NB/R, (q+1)*NB/R) of each chunk with
//    its own running maximum and sum, so each thread exponentiates 16 or 32
//    scores a chunk and the softmax spreads over the four SM sub-partitions.
//    The copies of a row are merged once, at the end, as split-K partials are.
//    A row's P is zero outside its own keys.
#include "pa_decode_tc.cuh"
#include "pa_query_major.h"

namespace pa {
namespace {

constexpr int QM_D = 128;
constexpr int QM_KC = 64;         // columns per chunk
constexpr int QM_ROWS = 128;      // query rows per tile (MMA M)
constexpr int QM_ST = 6;          // ring slots
constexpr int QM_THREADS = 192;   // softmax warps 0-3, producer 4, MMA 5
constexpr int QM_HALF_Q = QM_ROWS * 128;     // one 64-d half of Q: [128 rows][128 B]
constexpr int QM_Q_BYTES = 2 * QM_HALF_Q;
constexpr int QM_HALF_KV = QM_KC * 128;      // one 64-d half of a K or V chunk: [64 rows][128 B]
constexpr int QM_KV_BYTES = 2 * QM_HALF_KV;  // K (or V) of a chunk
constexpr int QM_SLOT = 2 * QM_KV_BYTES;     // K halves, then V halves
constexpr int QM_OFF_Q = 0;
constexpr int QM_OFF_RING = QM_OFF_Q + QM_Q_BYTES;
constexpr int QM_OFF_BARS = QM_OFF_RING + QM_ST * QM_SLOT;
constexpr int QM_NBARS = 2 * QM_ST + 8;  // full, empty, qfull, s[2], p[2], o[2], drain
constexpr int QM_OFF_WORDS = QM_OFF_BARS + QM_NBARS * 8;
constexpr int QM_OFF_LENS = QM_OFF_WORDS + 64;      // up to 256 sequence lengths
constexpr int QM_SMEM = QM_OFF_LENS + 1024 + 1024;  // + alignment slack
static_assert(QM_SMEM <= kMaxDynSmem, "shared memory budget");
constexpr uint32_t QM_TMEM_COLS = 256;  // S[2] (P in each's first 32) at [0, 128), O at [128, 256)
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
  int num_seqs, num_kv_heads, num_q_heads, q_len, tiles, head_groups, max_blocks_per_seq,
      num_blocks, cap, oob_row;
  float scale_log2;
  uint64_t wait_ns;
};

template <int G, int R, int HB>
__global__ void __launch_bounds__(QM_THREADS, 1)
    query_major_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_q, const QmParams P) {
  constexpr int RW = QM_ROWS / R;   // rows per copy
  constexpr int RPH = RW / HB;      // rows per head
  constexpr int QT = RPH / G;       // new tokens per tile
  constexpr int NB = 4 / HB;        // blocks per chunk
  constexpr int BR = 16 * HB;       // rows of one block's box (HB heads x 16 keys)
  constexpr int TB = NB / R;        // blocks of a chunk per copy
  constexpr int NC = 16 * TB;       // scores of a chunk per thread
  static_assert(QT >= 1 && RPH >= 32 && TB >= 1, "tile shape");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* qbuf = smem + QM_OFF_Q;
  unsigned char* ring = smem + QM_OFF_RING;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + QM_OFF_BARS);
  uint64_t* full = bars;
  uint64_t* empty = bars + QM_ST;
  uint64_t* qfull = bars + 2 * QM_ST;
  uint64_t* bar_s = qfull + 1;  // [2] scores of chunk c in S[c % 2]
  uint64_t* bar_p = bar_s + 2;  // [2] P of chunk c written over S[c % 2]
  uint64_t* bar_o = bar_p + 2;  // [2] value product of chunk c (which read S[c % 2]'s P) done
  uint64_t* drain = bar_o + 2;
  int* words = reinterpret_cast<int*>(smem + QM_OFF_WORDS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&words[0]);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&words[1]);
  int* issued = &words[2];
  int* consumed = &words[3];
  int* found = &words[4];  // the sequence of this CTA's rank (below)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = int(blockIdx.x) % P.tiles;
  const int hg0 = (int(blockIdx.x) / P.tiles) % P.head_groups * HB;  // first KV head
  const int rank = int(blockIdx.x) / (P.tiles * P.head_groups);
  const int Q = P.q_len;
  // Longest sequences first (the CTAs start in index order, so the last wave
  // holds the shortest work): up to 256 sequences every CTA ranks the lengths
  // and takes the sequence of its rank (ties by index).
  int b = rank, L;
  if (P.num_seqs <= 256) {
    // the lengths staged in shared memory, one load each
    int* lens_s = reinterpret_cast<int*>(smem + QM_OFF_LENS);
    for (int v = tid; v < P.num_seqs; v += QM_THREADS) lens_s[v] = P.context_lens[v];
    if (tid == 0) *found = rank;
    __syncthreads();
    for (int v = tid; v < P.num_seqs; v += QM_THREADS) {
      const int Lv = lens_s[v];
      int above = 0;
      for (int u = 0; u < P.num_seqs; ++u) {
        const int Lu = lens_s[u];
        above += Lu > Lv || (Lu == Lv && u < v);
      }
      if (above == rank) *found = v;
    }
    __syncthreads();
    b = *found;
    L = lens_s[b];
  } else {
    L = P.context_lens[b];
  }
  const bool report = tid == 0 && tile == 0 && hg0 == 0;
  if (L > P.cap) {
    if (report) atomicOr(&g_tc_errors, PA_DEVERR_CONTEXT_LEN);
    L = P.cap;
  }
  if (L > 0 && L < Q) {  // no room for the new tokens: an empty sequence
    if (report) atomicOr(&g_tc_errors, PA_DEVERR_CONTEXT_LEN);
    L = 0;
  }
  const int i_last = min(Q, (tile + 1) * QT) - 1;  // the tile's last new token
  if (L <= 0) {  // zero rows
    for (int e = tid; e < HB * RPH * (QM_D / 8); e += QM_THREADS) {
      const int x = e / (QM_D / 8), ch = e % (QM_D / 8);
      const int h = x / RPH, r0 = x % RPH, i = tile * QT + r0 / G;
      if (i < Q && hg0 + h < P.num_kv_heads) {
        const size_t row = (size_t(b) * Q + i) * P.num_q_heads + (hg0 + h) * G + r0 % G;
        reinterpret_cast<uint4*>(P.out + row * QM_D)[ch] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    return;
  }
  const int keys = L - Q + i_last + 1;  // what the tile's last row sees
  const int nblk = (keys + 15) / 16;
  const int n = (nblk + NB - 1) / NB;

  if (tid == 0) {
    for (int s = 0; s < QM_ST; ++s) {
      dev::mbar_init(&full[s], 1);
      dev::mbar_init(&empty[s], 1);
    }
    dev::mbar_init(qfull, 1);
    for (int k = 0; k < 2; ++k) {
      dev::mbar_init(&bar_s[k], 1);
      dev::mbar_init(&bar_p[k], 128);
      dev::mbar_init(&bar_o[k], 1);
    }
    dev::mbar_init(drain, 1);
    *abort_flag = 0;
    *issued = 0;
    *consumed = 0;
    dev::fence_barrier_init();
  }
  if (warp == 0) dev::tmem_alloc(tmem_slot, QM_TMEM_COLS);
  dev::tc_fence_before();
  __syncthreads();
  dev::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ---------------------------------------------------------- producer
    const uint64_t pol = dev::l2_evict_first_policy();
    if (lane == 0) {
      dev::prefetch_tmap(&tm_k);
      dev::prefetch_tmap(&tm_v);
      dev::mbar_arrive_expect_tx(qfull, QM_Q_BYTES);
      // rows [q*RW + h*RPH, +RPH) of each half: head hg0 + h, QT tokens
      for (int hf = 0; hf < 2; ++hf)
        for (int q = 0; q < R; ++q)
          for (int h = 0; h < HB; ++h)
            dev::tma_load_4d(qbuf + hf * QM_HALF_Q + (q * RW + h * RPH) * 128, &tm_q, hf * 64,
                             (hg0 + h) * G, tile * QT, b, qfull, pol);
    }
    const int32_t* trow = P.block_tables + size_t(b) * P.max_blocks_per_seq;
    // lane l holds the table entry of block w0 + l
    auto window = [&](int w0) {
      const int j = w0 + lane;
      return (j < P.max_blocks_per_seq && j < nblk) ? trow[j] : -1;
    };
    int w0 = 0;
    int win = window(0);
    bool ok = true;
    // lane l < 4*NB issues one request of the chunk: block u = l/4, K or V,
    // one 64-d half (the TMA unit takes requests from several lanes at once)
    const int u = (lane >> 2) % NB, hf = (lane >> 1) & 1, kv = lane & 1;
    for (int c = 0; c < n && ok; ++c) {
      if (c * NB >= w0 + 32) {
        w0 += 32;
        win = window(w0);
      }
      const int slot = c % QM_ST;
      if (lane == 0) {
        ok = dev::mbar_wait_sleep(&empty[slot], (uint32_t(c / QM_ST) & 1u) ^ 1u, 64, P.wait_ns,
                                  abort_flag);
        if (ok) dev::mbar_arrive_expect_tx(&full[slot], QM_SLOT);
      }
      ok = __shfl_sync(0xffffffffu, int(ok), 0) != 0;
      if (!ok) break;
      const int j = c * NB + u;
      const int e = __shfl_sync(0xffffffffu, win, j - w0);
      if (lane < 4 * NB) {
        int row = P.oob_row;  // past the sequence (or a bad entry): zero fill
        if (j < nblk) {
          if (e >= 0 && e < P.num_blocks) {
            row = (e * P.num_kv_heads + hg0) * 16;
          } else if (kv == 0 && hf == 0) {
            atomicOr(&g_tc_errors, PA_DEVERR_TABLE_ENTRY);
          }
        }
        unsigned char* dst =
            ring + size_t(slot) * QM_SLOT + kv * QM_KV_BYTES + hf * QM_HALF_KV + u * BR * 128;
        dev::tma_load_2d(dst, kv ? &tm_v : &tm_k, hf * 64, row, &full[slot], pol);
      }
      if (lane == 0) *issued = c + 1;
    }
    if (!ok && lane == 0) {
      atomicOr(&g_tc_errors, PA_DEVERR_TIMEOUT);
      *abort_flag = 1;
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------- MMA issue
    if (lane == 0) {
      const uint32_t qb = dev::smem_addr(qbuf);
      bool ok = dev::mbar_wait(qfull, 0, P.wait_ns, abort_flag);
      auto issue_s = [&](int c) {
        const uint32_t kb = dev::smem_addr(ring + size_t(c % QM_ST) * QM_SLOT);
        dev::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < QM_D / 16; ++kk) {
          const uint32_t hf = kk >> 2, off = uint32_t(kk & 3) * 32;
          dev::mma_bf16(tmem + uint32_t(c & 1) * QM_KC,
                        dev::smem_desc(qb + hf * QM_HALF_Q + off, 16, 1024, dev::kSwizzle128B),
                        dev::smem_desc(kb + hf * QM_HALF_KV + off, 16, 1024, dev::kSwizzle128B),
                        QM_IDESC_S, kk > 0);
        }
        dev::mma_commit(&bar_s[c & 1]);
      };
      // Event loop: the scores of chunk s once it has landed and the value
      // product of chunk s - 2 (which read P from the same S buffer) has
      // completed, and the value product of chunk v once the softmax has
      // written its P -- whichever is ready first, so that neither waits
      // behind the other.
      int s_next = 0, v_next = 0;
      uint64_t t_idle = 0;
      uint32_t idle = 0;
      while (ok && v_next < n) {
        bool progress = false;
        if (s_next < n && s_next <= v_next + 1 &&
            (s_next < 2 || dev::mbar_test(&bar_o[s_next & 1], uint32_t((s_next - 2) >> 1) & 1u)) &&
            dev::mbar_test(&full[s_next % QM_ST], uint32_t(s_next / QM_ST) & 1u)) {
          issue_s(s_next);
          ++s_next;
          progress = true;
        }
        if (v_next < s_next &&
            dev::mbar_test(&bar_p[v_next & 1], uint32_t(v_next >> 1) & 1u)) {
          const int c = v_next;
          dev::tc_fence_after();
          const uint32_t vb = dev::smem_addr(ring + size_t(c % QM_ST) * QM_SLOT + QM_KV_BYTES);
#pragma unroll
          for (int kk = 0; kk < QM_KC / 16; ++kk)
            mma_bf16_tmem_a(tmem + 2 * QM_KC, tmem + uint32_t(c & 1) * QM_KC + uint32_t(kk * 8),
                            // V MN-major: next 8 rows 1024 B on (SBO), second 64-d
                            // half one half on (LBO)
                            dev::smem_desc(vb + kk * 2048, QM_HALF_KV, 1024, dev::kSwizzle128B),
                            QM_IDESC_PV, c > 0 || kk > 0);
          dev::mma_commit(&bar_o[c & 1]);
          dev::mma_commit(&empty[c % QM_ST]);
          *consumed = c + 1;
          ++v_next;
          progress = true;
        }
        if (progress) {
          idle = 0;
          continue;
        }
        // bounded idle: the wall clock is read every 256 polls
        if ((++idle & 255u) != 0u) continue;
        if (*abort_flag) {
          ok = false;
          break;
        }
        const uint64_t now = dev::global_timer_ns();
        if (idle == 256u) {
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
    const int q = r / RW, h = (r % RW) / RPH, r0 = r % RPH;  // copy, head, row of the head
    const int i = tile * QT + r0 / G;
    const bool valid = i < Q && hg0 + h < P.num_kv_heads;
    const int L_row = valid ? L - Q + i + 1 : 0;
    const uint32_t t_lane = uint32_t(warp * 32) << 16;
    const float sl2 = P.scale_log2;
    float m_ref = -INFINITY, l = 0.0f;
    int pv_done = -1;
    bool ok = true;
    // value product of chunk k done (it completes bar_o[k % 2], phase k / 2)
    auto wait_pv = [&](int k) {
      ok = __all_sync(0xffffffffu, dev::mbar_wait(&bar_o[k & 1], uint32_t(k >> 1) & 1u,
                                                  P.wait_ns, abort_flag)) &&
           ok;
      pv_done = k;
    };
    for (int c = 0; c < n && ok; ++c) {
      ok = __all_sync(0xffffffffu, dev::mbar_wait(&bar_s[c & 1], uint32_t(c >> 1) & 1u,
                                                  P.wait_ns, abort_flag));
      if (!ok) break;
      dev::tc_fence_after();
      // this thread's scores: blocks u = q*TB + t of the chunk, 16 columns each
      // at u*BR + h*16 (contiguous when HB = 1)
      float s[NC];
      {
        uint32_t raw[NC];
#pragma unroll
        for (int t = 0; t < TB; ++t)
          asm volatile(
              "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, "
              "%10, %11, %12, %13, %14, %15}, [%16];"
              : "=r"(raw[16 * t + 0]), "=r"(raw[16 * t + 1]), "=r"(raw[16 * t + 2]),
                "=r"(raw[16 * t + 3]), "=r"(raw[16 * t + 4]), "=r"(raw[16 * t + 5]),
                "=r"(raw[16 * t + 6]), "=r"(raw[16 * t + 7]), "=r"(raw[16 * t + 8]),
                "=r"(raw[16 * t + 9]), "=r"(raw[16 * t + 10]), "=r"(raw[16 * t + 11]),
                "=r"(raw[16 * t + 12]), "=r"(raw[16 * t + 13]), "=r"(raw[16 * t + 14]),
                "=r"(raw[16 * t + 15])
              : "r"(tmem + t_lane + uint32_t(c & 1) * QM_KC +
                    uint32_t((q * TB + t) * BR + h * 16)));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int k = 0; k < NC; ++k) s[k] = __uint_as_float(raw[k]);
      }
      const int key0 = (c * NB + q * TB) * 16;  // key of s[0]; s[k] is key key0 + k
      if (!__all_sync(0xffffffffu, key0 + NC <= L_row)) {
#pragma unroll
        for (int k = 0; k < NC; ++k) s[k] = key0 + k < L_row ? s[k] : -INFINITY;
      }
      // maximum of the raw scores (the scale is positive), four chains
      float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
      for (int k = 4; k < NC; ++k) mx[k & 3] = fmaxf(mx[k & 3], s[k]);
      const float cm = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
      // the reference moves only when a score exceeds it by more than 2^8
      const bool need = cm > m_ref + kRescaleLog2;
      if (__any_sync(0xffffffffu, need)) {
        const float nr = need ? cm : m_ref;
        const float f = nr == m_ref || m_ref == -INFINITY ? 1.0f : dev::fast_exp2(m_ref - nr);
        if (c > 0) {
          if (pv_done < c - 1) wait_pv(c - 1);
          if (!ok) break;
          dev::tc_fence_after();
#pragma unroll
          for (int cg = 0; cg < QM_D; cg += 32) {
            float o[32];
            dev::tmem_ld_cols<32>(tmem + t_lane + 2 * QM_KC + cg, o);
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] *= f;
            dev::tmem_st_cols<32>(tmem + t_lane + 2 * QM_KC + cg, o);
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
      for (int k = 0; k < NC; k += 2) {
        const float p0 = dev::fast_exp2(fmaf(s[k], sl2, nm));
        const float p1 = dev::fast_exp2(fmaf(s[k + 1], sl2, nm));
        la += p0;
        lb += p1;
        const __nv_bfloat162 v2 = __floats2bfloat162_rn(p0, p1);
        pw[k / 2] = *reinterpret_cast<const uint32_t*>(&v2);
      }
      l += la + lb;
      if ((c + 1) * NB * 16 > L) {
        // keys past the sequence in its last block may hold anything (NaN
        // included): clear their V rows so that 0 * V = 0. Thread r clears
        // row x = r % 64 of half r / 64: block x / BR, key x % 16.
        const int x = r % QM_KC, hf = r / QM_KC;
        if ((c * NB + x / BR) * 16 + x % 16 >= L) {
          uint4* vrow = reinterpret_cast<uint4*>(ring + size_t(c % QM_ST) * QM_SLOT +
                                                 QM_KV_BYTES + hf * QM_HALF_KV + x * 128);
#pragma unroll
          for (int k = 0; k < 8; ++k) vrow[k] = make_uint4(0u, 0u, 0u, 0u);
        }
        dev::fence_async_smem();  // before the value product reads the ring
      }
      // P over the first 32 columns of this chunk's S buffer (its scores are
      // in registers): column j holds columns 2j, 2j+1 of the chunk; block u's
      // 16 columns of this head are P columns (u*BR + h*16)/2 + [0, 8), the
      // rest zero. The value product of chunk c - 2, which read this buffer's
      // last P, completed before S(c) was issued.
      {
        float pp[QM_KC / 2];
#pragma unroll
        for (int k = 0; k < QM_KC / 2; ++k) {
          const int u = 2 * k / BR, hh = 2 * k % BR / 16;  // block and head of P column k
          pp[k] = u / TB == q && hh == h ? __uint_as_float(pw[8 * (u % TB) + k % 8]) : 0.0f;
        }
        dev::tmem_st_cols<QM_KC / 2>(tmem + t_lane + uint32_t(c & 1) * QM_KC, pp);
      }
      dev::tc_fence_before();
      dev::mbar_arrive(&bar_p[c & 1]);
    }
    if (ok && n > 0) wait_pv(n - 1);
    __nv_bfloat16* orow =
        P.out + ((size_t(b) * Q + (valid ? i : 0)) * P.num_q_heads + (hg0 + h) * G + r0 % G) * QM_D;
    if (R == 1) {
      if (ok) {
        dev::tc_fence_after();
        const float inv = l > 0.0f ? __frcp_rn(l) : 0.0f;
#pragma unroll
        for (int cg = 0; cg < QM_D; cg += 32) {
          float o[32];
          dev::tmem_ld_cols<32>(tmem + t_lane + 2 * QM_KC + cg, o);
          if (valid) {
#pragma unroll
            for (int k = 0; k < 32; k += 8) {
              uint32_t w[4];
#pragma unroll
              for (int q2 = 0; q2 < 4; ++q2) {
                const __nv_bfloat162 v2 =
                    __floats2bfloat162_rn(o[k + 2 * q2] * inv, o[k + 2 * q2 + 1] * inv);
                w[q2] = *reinterpret_cast<const uint32_t*>(&v2);
              }
              *reinterpret_cast<uint4*>(orow + cg + k) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      } else if (lane == 0) {
        atomicOr(&g_tc_errors, PA_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
    } else {
      // Merge the R copies of each row (every value product has completed,
      // so the ring is free): each thread leaves its raw O row, reference and
      // sum in shared memory; then copy q of a row writes output columns
      // [q*128/R, (q+1)*128/R), each the sum over copies of 2^(m_c - M) O_c,
      // divided by the sum of 2^(m_c - M) l_c (M the largest reference).
      // 16-byte chunk j of TMEM lane x sits at chunk (j + x) % 32 of its 512 bytes.
      if (!ok && lane == 0) {
        atomicOr(&g_tc_errors, PA_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      // a uniform decision: the softmax warps all finished, or none merges
      if (dev::named_barrier_and(1, 128, ok)) {
        float* mbuf = reinterpret_cast<float*>(ring + QM_ROWS * 512);
        float* lbuf = mbuf + QM_ROWS;
        dev::tc_fence_after();
        unsigned char* orow_s = ring + r * 512;
#pragma unroll
        for (int cg = 0; cg < QM_D; cg += 32) {
          float o[32];
          dev::tmem_ld_cols<32>(tmem + t_lane + 2 * QM_KC + cg, o);
#pragma unroll
          for (int k = 0; k < 32; k += 4)
            *reinterpret_cast<float4*>(orow_s + ((((cg + k) / 4 + r) & 31) << 4)) =
                make_float4(o[k], o[k + 1], o[k + 2], o[k + 3]);
        }
        mbuf[r] = m_ref;
        lbuf[r] = l;
        dev::named_barrier(1, 128);
        const int rr = r % RW;  // the row within a copy
        float M = -INFINITY;
#pragma unroll
        for (int qq = 0; qq < R; ++qq) M = fmaxf(M, mbuf[qq * RW + rr]);
        float fq[R], lt = 0.0f;
#pragma unroll
        for (int qq = 0; qq < R; ++qq) {
          const float mq = mbuf[qq * RW + rr];
          fq[qq] = mq == -INFINITY ? 0.0f : dev::fast_exp2(mq - M);
          lt += fq[qq] * lbuf[qq * RW + rr];
        }
        const float inv = lt > 0.0f ? __frcp_rn(lt) : 0.0f;
        if (valid) {
          constexpr int OC = QM_D / R;  // output columns of this thread
#pragma unroll
          for (int k = 0; k < OC; k += 8) {
            const int col = q * OC + k;
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int qq = 0; qq < R; ++qq) {
              const int x = qq * RW + rr;
              const unsigned char* src = ring + x * 512;
              const float4 a0 = *reinterpret_cast<const float4*>(src + (((col / 4 + x) & 31) << 4));
              const float4 a1 =
                  *reinterpret_cast<const float4*>(src + (((col / 4 + 1 + x) & 31) << 4));
              acc[0] += fq[qq] * a0.x;
              acc[1] += fq[qq] * a0.y;
              acc[2] += fq[qq] * a0.z;
              acc[3] += fq[qq] * a0.w;
              acc[4] += fq[qq] * a1.x;
              acc[5] += fq[qq] * a1.y;
              acc[6] += fq[qq] * a1.z;
              acc[7] += fq[qq] * a1.w;
            }
            uint32_t w[4];
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2) {
              const __nv_bfloat162 v2 =
                  __floats2bfloat162_rn(acc[2 * q2] * inv, acc[2 * q2 + 1] * inv);
              w[q2] = *reinterpret_cast<const uint32_t*>(&v2);
            }
            *reinterpret_cast<uint4*>(orow + col) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
  }

  __syncthreads();
  if (*abort_flag && tid == 0) {
    // every copy issued but not consumed lands before shared memory is released
    for (int c = *consumed; c < *issued; ++c)
      (void)dev::mbar_wait(&full[c % QM_ST], uint32_t(c / QM_ST) & 1u);
  }
  dev::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    dev::tc_fence_after();
    dev::tmem_dealloc(tmem, QM_TMEM_COLS);
  }
}

template <int G, int R, int HB>
int launch_qm_t(const pa_decode_params* p, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(query_major_kernel<G, R, HB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, QM_SMEM);
    if (e != cudaSuccess) return int(e);
    configured = true;
  }
  const int H = p->num_kv_heads, Q = query_len_of(p);
  const uint64_t cache_rows = uint64_t(p->num_blocks) * H * 16;
  CUtensorMap tk, tv, tq;
  // K, V [rows][128 d]: a box of HB heads x 16 keys of one block, one 64-d half
  int r = make_map(&tk, p->k_cache, cache_rows, QM_D, uint32_t(16 * HB));
  if (!r) r = make_map(&tv, p->v_cache, cache_rows, QM_D, uint32_t(16 * HB));
  if (!r) {
    // q [B][Q][Hq][128]: box (64 d, G heads, QT tokens, 1 sequence)
    const cuuint64_t dims[4] = {uint64_t(QM_D), uint64_t(p->num_q_heads), uint64_t(Q),
                                uint64_t(p->num_seqs)};
    const cuuint64_t strides[3] = {uint64_t(QM_D) * 2, uint64_t(p->num_q_heads) * QM_D * 2,
                                   uint64_t(Q) * p->num_q_heads * QM_D * 2};
    const cuuint32_t box[4] = {64, uint32_t(G), uint32_t(QM_ROWS / (R * HB * G)), 1};
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
  P.max_blocks_per_seq = p->max_blocks_per_seq;
  P.num_blocks = p->num_blocks;
  P.cap = std::min(p->max_blocks_per_seq * 16, p->max_context_len);
  P.oob_row = int(cache_rows);
  P.scale_log2 = p->scale * kLog2e;
  P.wait_ns = p->wait_timeout_us > 0 ? uint64_t(p->wait_timeout_us) * 1000u : dev::kWaitNsLimit;
  const dim3 grid(unsigned(p->num_seqs) * unsigned(P.head_groups) * unsigned(P.tiles));
  query_major_kernel<G, R, HB><<<grid, QM_THREADS, QM_SMEM, stream>>>(tk, tv, tq, P);
  return int(cudaGetLastError());
}

template <int G>
int launch_qm_g(const pa_decode_params* p, cudaStream_t stream) {
  const int R = query_major_copies(p), HB = query_major_heads(p);
  if (HB == 2) return R == 2 ? launch_qm_t<G, 2, 2>(p, stream) : launch_qm_t<G, 1, 2>(p, stream);
  return R == 4 ? launch_qm_t<G, 4, 1>(p, stream)
                : (R == 2 ? launch_qm_t<G, 2, 1>(p, stream) : launch_qm_t<G, 1, 1>(p, stream));
}

}  // namespace

int launch_query_major_tc(const pa_decode_params* p, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (p->num_q_heads / p->num_kv_heads) {
    case 1: return launch_qm_g<1>(p, s);
    case 2: return launch_qm_g<2>(p, s);
    case 4: return launch_qm_g<4>(p, s);
    case 8: return launch_qm_g<8>(p, s);
    default: return int(cudaErrorInvalidValue);
  }
}

int read_and_clear_query_major_errors(uint32_t* flags) {
  return read_and_clear_tc_error_word(flags);
}

}  // namespace pa
