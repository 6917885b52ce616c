// Paged decode attention on the 5th-generation tensor cores (sm_103a).
//
// Same result as the CUDA-core kernel ("Paged Attention as a Memory
// Manager", §How the Kernel Executes Paged Attention; "PagedAttention and
// continuous batching", §Attention kernel modification): per (sequence,
// query head), softmax(scale * q.K^T) V over the cached tokens, K/V gathered
// block by block through the block table, a running softmax across blocks,
// padding slots of the last block masked.
//
// Why tensor cores: with the query heads of one KV group packed, the score
// step is a small dense contraction [keys x d] x [d x G] and the value step
// [d x keys] x [keys x G]. Done in fp32 on CUDA cores they cost ~1000
// instructions per 8 KiB (block, KV head) tile, which left the CUDA-core
// kernel issue-bound at ~57 % of HBM bandwidth. On tcgen05 the same tile is
// two MMA instructions.
//
// Structure (one persistent CTA per SM, 5 warps):
//  * Warp 4 -- producer. Takes work items (sequence, KV head, partition)
//    from a global counter, reads the partition's block-table slice once
//    (range-checked), and streams K and V in chunks of 8 blocks = 128 keys
//    into a 3-stage shared-memory ring with tensor-map TMA (128-byte
//    swizzle; blocks past the item are loaded from an out-of-range row and
//    arrive as zeros). The item's query rows come with its first chunk.
//  * Warps 0-3 -- consumers, one thread per key of the chunk:
//      S^T[128 keys][16] = K[128][d] . Q^T  (tcgen05.mma, M=128, N=16, fp32 in TMEM)
//      running max / sum per head, P = exp2(S*scale*log2e - m) as bf16 in smem
//      O^T[d][16]      = V^T[d][128] . P^T   (tcgen05.mma, V read MN-major)
//      acc[h] = acc[h] * alpha[h] + O^T[dim][h]   (thread = head dimension)
//    The G real heads of the KV group use columns 0..G-1; the padded columns
//    are never read back.
//  * Results: one partition -> bf16 output; several -> fp32 partials merged
//    by the log-sum-exp merge kernel.
//
// Every mbarrier wait is bounded; a wait that runs out sets PA_DEVERR_TIMEOUT
// and the CTA winds down (uniformly, through its named barriers), drains its
// outstanding copies and MMAs with bounded waits, frees TMEM and exits.
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

constexpr int BS = kBlockSize;
constexpr int CHB = 8;         // blocks per chunk
constexpr int CHK = CHB * BS;  // keys per chunk = MMA M
constexpr int NQ = 16;         // MMA N: query heads of a KV group, padded
constexpr int NCONS = 4;       // consumer warps
constexpr int NTHREADS = (NCONS + 1) * 32;
constexpr int kCons = NCONS * 32;
constexpr int TMEM_COLS = 32;  // S^T in columns 0..15, O^T in 16..31
constexpr int MAX_ITEM_BLOCKS = kMaxPartitionTokens / BS;
constexpr float kLog2e = 1.4426950408889634f;

enum : int { F_FIRST = 1, F_LAST = 2, F_SPLIT = 4, F_ZERO = 8, F_END = 16 };

struct __align__(16) ChunkMeta {
  int b, g, p, flags;
  int tok0;     // first token of the chunk
  int tok_end;  // one past the item's last token
  int nblk;     // blocks of the chunk that hold cache data
  int qslot;
};

template <int D>
struct TcCfg {
  static constexpr int HALVES = D / 64;               // 128-byte swizzle atoms per row
  static constexpr int HALF_BYTES = CHK * 128;        // [128 rows][64 bf16]
  static constexpr int K_BYTES = HALVES * HALF_BYTES;
  static constexpr int SLOT_BYTES = 2 * K_BYTES;      // K then V
  static constexpr int ST = (D == 128) ? 3 : 5;
  static constexpr int QH_BYTES = NQ * 128;           // [16 rows][64 bf16]
  static constexpr int Q_BYTES = HALVES * QH_BYTES;
  static constexpr int P_BYTES = 2 * NQ * 128;        // P^T [16][128 keys]: 2 atoms of 64 keys
  static constexpr int BOX_BYTES = BS * 128;          // one TMA box: 16 rows x 64 bf16
  static constexpr uint32_t CHUNK_TX = CHB * 2 * HALVES * BOX_BYTES;
  static constexpr uint32_t Q_TX = HALVES * QH_BYTES;
  static constexpr int OFF_RING = 0;
  static constexpr int OFF_Q = OFF_RING + ST * SLOT_BYTES;
  static constexpr int OFF_P = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_BARS = OFF_P + P_BYTES;
  static constexpr int NBARS = 2 * ST + 5;  // full[ST] empty[ST] qempty[2] s o drain
  static constexpr int OFF_META = (OFF_BARS + NBARS * 8 + 15) / 16 * 16;
  static constexpr int OFF_TAB = OFF_META + ST * int(sizeof(ChunkMeta));
  static constexpr int OFF_RED = OFF_TAB + MAX_ITEM_BLOCKS * 4;
  static constexpr int OFF_RED2 = OFF_RED + NCONS * NQ * 4;
  static constexpr int OFF_MISC = OFF_RED2 + NCONS * NQ * 4;
  static constexpr int SMEM = OFF_MISC + 32 + 1024;  // + alignment slack
  static constexpr uint32_t IDESC_S = dev::idesc_bf16_f32(CHK, NQ, false, false);
  static constexpr uint32_t IDESC_PV = dev::idesc_bf16_f32(128, NQ, true, false);
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

struct TcParams {
  const int32_t* block_tables;
  const int32_t* context_lens;
  __nv_bfloat16* out;
  float* part_m;
  float* part_l;
  float* part_acc;
  unsigned int* counters;
  int max_blocks_per_seq, num_seqs, num_kv_heads, num_q_heads, group, num_blocks;
  int max_context_len, partition_tokens, num_partitions, total_items, oob_row;
  float scale_log2;
};

// Byte offset of P^T[h][key] in the K-major, 128B-swizzled B-operand layout.
__device__ __forceinline__ uint32_t p_offset(int h, int key) {
  const int half = key >> 6, kin = key & 63;
  const int r = h & 7, grp = h >> 3;
  return uint32_t(half * 2048 + grp * 1024 + r * 128 + (((kin >> 3) ^ r) << 4) + (kin & 7) * 2);
}

template <int D, int G>
__device__ __forceinline__ void consumer_loop(const TcParams& P, unsigned char* ring,
                                              unsigned char* qbuf, unsigned char* pbuf,
                                              uint64_t* full, uint64_t* empty, uint64_t* qempty,
                                              uint64_t* bar_s, uint64_t* bar_o,
                                              const ChunkMeta* meta, float* red, float* red2,
                                              uint32_t tmem, volatile int* abort_flag,
                                              int* consumed_out) {
  using C = TcCfg<D>;
  const int ctid = threadIdx.x;  // 0..127: key of the chunk, and head dimension
  const int cw = ctid >> 5, lane = ctid & 31;
  const uint32_t t_lane = uint32_t(cw * 32) << 16;
  const uint32_t tS = tmem + t_lane, tO = tmem + t_lane + 16;
  float m_run[G], l_part[G], acc[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m_run[h] = -INFINITY;
    l_part[h] = 0.0f;
    acc[h] = 0.0f;
  }
  int chunk_seq = 0;
  int mma_chunks = 0;
  bool carry_ok = true;
  for (;;) {
    const int slot = chunk_seq % C::ST;
    const uint32_t ph = uint32_t(chunk_seq / C::ST) & 1u;
    bool ok = __all_sync(0xffffffffu, dev::mbar_wait(&full[slot], ph));
    const ChunkMeta m = meta[slot];
    if (!dev::named_barrier_and(1, kCons, ok && carry_ok && *abort_flag == 0)) {
      if (ctid == 0) {
        atomicOr(&g_tc_errors, PA_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      break;
    }
    if (m.flags & F_END) break;
    if (m.flags & F_ZERO) {
      if (ctid < D) {
#pragma unroll
        for (int h = 0; h < G; ++h)
          P.out[(size_t(m.b) * P.num_q_heads + m.g * G + h) * D + ctid] = __float2bfloat16_rn(0.f);
      }
      if (ctid == 0) dev::mbar_arrive(&empty[slot]);
      ++chunk_seq;
      continue;
    }
    unsigned char* kv = ring + size_t(slot) * C::SLOT_BYTES;

    // ---- S^T = K . Q^T  (one thread issues; fp32 result in TMEM columns 0..15)
    if (ctid == 0) {
      dev::tc_fence_after();
      const uint32_t kb = dev::smem_addr(kv);
      const uint32_t qb = dev::smem_addr(qbuf + m.qslot * C::Q_BYTES);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t hf = kk >> 2, off = uint32_t(kk & 3) * 32;
        dev::mma_bf16(tmem, dev::smem_desc(kb + hf * C::HALF_BYTES + off, 16, 1024, dev::kSwizzle128B),
                      dev::smem_desc(qb + hf * C::QH_BYTES + off, 16, 1024, dev::kSwizzle128B),
                      C::IDESC_S, kk > 0);
      }
      dev::mma_commit(bar_s);
      if (m.flags & F_LAST) dev::mma_commit(&qempty[m.qslot]);
    }
    ok = __all_sync(0xffffffffu, dev::mbar_wait(bar_s, uint32_t(mma_chunks) & 1u));
    dev::tc_fence_after();
    float s[16];
    dev::tmem_ld16(tS, s);

    // ---- running softmax over this chunk (thread = key)
    const int t = m.tok0 + ctid;
    const bool valid = t < m.tok_end;
    float x[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      x[h] = valid ? s[h] * P.scale_log2 : -INFINITY;
      float v = x[h];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
      if (lane == 0) red[cw * NQ + h] = v;
    }
    ok = dev::named_barrier_and(1, kCons, ok);
    float alpha[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float cmax = red[h];
#pragma unroll
      for (int w = 1; w < NCONS; ++w) cmax = fmaxf(cmax, red[w * NQ + h]);
      const float m_new = fmaxf(m_run[h], cmax);
      alpha[h] = dev::fast_exp2(m_run[h] - m_new);
      m_run[h] = m_new;
      const float p = dev::fast_exp2(x[h] - m_new);
      l_part[h] = fmaf(l_part[h], alpha[h], p);
      *reinterpret_cast<__nv_bfloat16*>(pbuf + p_offset(h, ctid)) = __float2bfloat16_rn(p);
    }
    // A masked key inside a block that was loaded (the sequence's last,
    // partial block) may hold anything, NaN included: clear its V row so that
    // 0 * V stays 0 in the MMA.
    if (!valid && (ctid >> 4) < m.nblk) {
#pragma unroll
      for (int hf = 0; hf < C::HALVES; ++hf) {
        uint4* row = reinterpret_cast<uint4*>(kv + C::K_BYTES + hf * C::HALF_BYTES + ctid * 128);
#pragma unroll
        for (int i = 0; i < 8; ++i) row[i] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    dev::fence_async_smem();
    dev::tc_fence_before();
    ok = dev::named_barrier_and(1, kCons, ok);

    // ---- O^T = V^T . P^T  (V read MN-major; fresh accumulation each chunk)
    if (ctid == 0) {
      dev::tc_fence_after();
      const uint32_t vb = dev::smem_addr(kv + C::K_BYTES);
      const uint32_t pb = dev::smem_addr(pbuf);
      // D = 64: the second 64-row half of M re-reads the first (LBO 0); its
      // TMEM lanes are never read back.
      const uint32_t lbo = C::HALVES == 2 ? uint32_t(C::HALF_BYTES) : 0u;
#pragma unroll
      for (int kk = 0; kk < CHK / 16; ++kk) {
        dev::mma_bf16(tmem + 16, dev::smem_desc(vb + kk * 2048, lbo, 1024, dev::kSwizzle128B),
                      dev::smem_desc(pb + (kk >> 2) * C::QH_BYTES + (kk & 3) * 32, 16, 1024,
                                     dev::kSwizzle128B),
                      C::IDESC_PV, kk > 0);
      }
      dev::mma_commit(bar_o);
      dev::mma_commit(&empty[slot]);
    }
    ok = __all_sync(0xffffffffu, dev::mbar_wait(bar_o, uint32_t(mma_chunks) & 1u)) && ok;
    dev::tc_fence_after();
    float o[16];
    dev::tmem_ld16(tO, o);
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = fmaf(acc[h], alpha[h], o[h]);
    dev::tc_fence_before();
    ++mma_chunks;
    ++chunk_seq;

    if (m.flags & F_LAST) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float v = l_part[h];
#pragma unroll
        for (int o2 = 16; o2 >= 1; o2 >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o2);
        if (lane == 0) red2[cw * NQ + h] = v;
      }
      ok = dev::named_barrier_and(1, kCons, ok);
      if (ctid < D) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float l = red2[h];
#pragma unroll
          for (int w = 1; w < NCONS; ++w) l += red2[w * NQ + h];
          const size_t row = size_t(m.b) * P.num_q_heads + m.g * G + h;
          if (!(m.flags & F_SPLIT)) {
            P.out[row * D + ctid] = __float2bfloat16_rn(acc[h] * __frcp_rn(l));
          } else {
            const size_t prow = row * P.num_partitions + m.p;
            P.part_acc[prow * D + ctid] = acc[h];
            if (ctid == 0) {
              P.part_m[prow] = m_run[h];
              P.part_l[prow] = l;
            }
          }
        }
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        m_run[h] = -INFINITY;
        l_part[h] = 0.0f;
        acc[h] = 0.0f;
      }
    }
    carry_ok = ok;
  }
  if (ctid == 0) *consumed_out = chunk_seq;
}

template <int D, int G>
__global__ void __launch_bounds__(NTHREADS, 1)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ CUtensorMap tm_q, const TcParams P) {
  using C = TcCfg<D>;
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
  uint64_t* bar_s = bars + 2 * C::ST + 2;
  uint64_t* bar_o = bar_s + 1;
  uint64_t* drain = bar_s + 2;
  ChunkMeta* meta = reinterpret_cast<ChunkMeta*>(smem + C::OFF_META);
  int32_t* tab = reinterpret_cast<int32_t*>(smem + C::OFF_TAB);
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
  float* red2 = reinterpret_cast<float*>(smem + C::OFF_RED2);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  int* consumed = reinterpret_cast<int*>(smem + C::OFF_MISC + 8);
  int* issued = reinterpret_cast<int*>(smem + C::OFF_MISC + 12);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < C::ST; ++i) {
      dev::mbar_init(&full[i], 1);
      dev::mbar_init(&empty[i], 1);
    }
    dev::mbar_init(&qempty[0], 1);
    dev::mbar_init(&qempty[1], 1);
    dev::mbar_init(bar_s, 1);
    dev::mbar_init(bar_o, 1);
    dev::mbar_init(drain, 1);
    *abort_flag = 0;
    *consumed = 0;
    *issued = 0;
    dev::fence_barrier_init();
  }
  for (int i = tid; i < C::P_BYTES / 16; i += NTHREADS)
    reinterpret_cast<uint4*>(pbuf)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (warp == 0) dev::tmem_alloc(tmem_slot, TMEM_COLS);
  dev::fence_async_smem();
  dev::tc_fence_before();
  __syncthreads();
  dev::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == NCONS) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      dev::prefetch_tmap(&tm_k);
      dev::prefetch_tmap(&tm_v);
      dev::prefetch_tmap(&tm_q);
    }
    const uint64_t pol = dev::l2_evict_first_policy();
    const int PT = P.partition_tokens;
    const int bh = P.num_seqs * P.num_kv_heads;
    int chunk_seq = 0, item_seq = 0;
    bool ok = true;
    while (ok) {
      if (*abort_flag) break;
      int w = 0;
      if (lane == 0) w = int(atomicAdd(P.counters, 1u));
      w = __shfl_sync(0xffffffffu, w, 0);
      if (w >= P.total_items) break;
      const int p = w / bh;
      const int rem = w - p * bh;
      const int b = rem / P.num_kv_heads;
      const int g = rem - b * P.num_kv_heads;
      int L = P.context_lens[b];
      const int cap = min(P.max_blocks_per_seq * BS, P.max_context_len);
      if (L > cap) {
        if (lane == 0 && p == 0 && g == 0) atomicOr(&g_tc_errors, PA_DEVERR_CONTEXT_LEN);
        L = cap;
      }
      if (L <= 0) {
        if (p != 0) continue;
        const int slot = chunk_seq % C::ST;
        const uint32_t ph = uint32_t(chunk_seq / C::ST) & 1u;
        if (lane == 0) {
          ok = dev::mbar_wait(&empty[slot], ph ^ 1u);
          ChunkMeta m{};
          m.b = b;
          m.g = g;
          m.p = 0;
          m.flags = F_ZERO;
          meta[slot] = m;
          dev::mbar_arrive(&full[slot]);
        }
        ok = __shfl_sync(0xffffffffu, int(ok), 0) != 0;
        ++chunk_seq;
        continue;
      }
      const int np = (L + PT - 1) / PT;
      if (p >= np) continue;
      const int tok0 = p * PT;
      const int tok1 = min(L, tok0 + PT);
      const int nblk = (tok1 - tok0 + BS - 1) / BS;
      const int lb0 = tok0 / BS;
      __syncwarp();
      const int32_t* trow = P.block_tables + size_t(b) * P.max_blocks_per_seq + lb0;
      for (int j = lane; j < nblk; j += 32) {
        const int32_t e = trow[j];
        int row = P.oob_row;
        if (e < 0 || e >= P.num_blocks) {
          atomicOr(&g_tc_errors, PA_DEVERR_TABLE_ENTRY);
        } else {
          row = (e * P.num_kv_heads + g) * BS;
        }
        tab[j] = row;
      }
      __syncwarp();
      const int qs = item_seq & 1;
      const int nch = (nblk + CHB - 1) / CHB;
      for (int c = 0; c < nch; ++c) {
        const int slot = chunk_seq % C::ST;
        const uint32_t ph = uint32_t(chunk_seq / C::ST) & 1u;
        if (lane == 0) {
          ok = dev::mbar_wait(&empty[slot], ph ^ 1u);
          if (ok && c == 0) ok = dev::mbar_wait(&qempty[qs], (uint32_t(item_seq >> 1) & 1u) ^ 1u);
          if (ok) {
            ChunkMeta m;
            m.b = b;
            m.g = g;
            m.p = p;
            m.flags = (c == 0 ? F_FIRST : 0) | (c == nch - 1 ? F_LAST : 0) | (L > PT ? F_SPLIT : 0);
            m.tok0 = tok0 + c * CHK;
            m.tok_end = tok1;
            m.nblk = min(CHB, nblk - c * CHB);
            m.qslot = qs;
            meta[slot] = m;
            dev::mbar_arrive_expect_tx(&full[slot], C::CHUNK_TX + (c == 0 ? C::Q_TX : 0u));
          }
        }
        ok = __shfl_sync(0xffffffffu, int(ok), 0) != 0;
        if (!ok) break;
        unsigned char* kdst = ring + size_t(slot) * C::SLOT_BYTES;
        if (lane < CHB) {
          const int j = c * CHB + lane;
          const int row = j < nblk ? tab[j] : P.oob_row;
#pragma unroll
          for (int hf = 0; hf < C::HALVES; ++hf) {
            unsigned char* d = kdst + hf * C::HALF_BYTES + lane * C::BOX_BYTES;
            dev::tma_load_2d(d, &tm_k, hf * 64, row, &full[slot], pol);
            dev::tma_load_2d(d + C::K_BYTES, &tm_v, hf * 64, row, &full[slot], pol);
          }
        } else if (lane == CHB && c == 0) {
          const int qrow = b * P.num_q_heads + g * P.group;
#pragma unroll
          for (int hf = 0; hf < C::HALVES; ++hf)
            dev::tma_load_2d(qbuf + qs * C::Q_BYTES + hf * C::QH_BYTES, &tm_q, hf * 64, qrow,
                             &full[slot], pol);
        }
        ++chunk_seq;
        if (lane == 0) *issued = chunk_seq;
      }
      ++item_seq;
    }
    // end of work: a sentinel chunk tells the consumers to stop
    if (lane == 0) {
      const int slot = chunk_seq % C::ST;
      const uint32_t ph = uint32_t(chunk_seq / C::ST) & 1u;
      const bool ok2 = dev::mbar_wait(&empty[slot], ph ^ 1u);
      ChunkMeta m{};
      m.flags = F_END;
      meta[slot] = m;
      dev::mbar_arrive(&full[slot]);
      if (!ok || !ok2) {
        atomicOr(&g_tc_errors, PA_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    consumer_loop<D, G>(P, ring, qbuf, pbuf, full, empty, qempty, bar_s, bar_o, meta, red, red2,
                        tmem, abort_flag, consumed);
  }

  __syncthreads();
  if (*abort_flag && tid == 0) {
    // Wind down after a stalled wait: let every MMA issued so far finish and
    // every bulk copy issued but not consumed land (each wait bounded)
    // before TMEM and shared memory are released.
    dev::mma_commit(drain);
    (void)dev::mbar_wait(drain, 0);
    for (int c = *consumed; c < *issued; ++c)
      (void)dev::mbar_wait(&full[c % C::ST], uint32_t(c / C::ST) & 1u);
  }
  dev::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    dev::tc_fence_after();
    dev::tmem_dealloc(tmem, TMEM_COLS);
  }
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

// 2-D bf16 tensor [rows][cols] (row pitch cols*2 bytes), box 16 rows x 64 cols, 128B swizzle,
// out-of-range elements read as zero.
int make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  if (encode_fn(&enc)) return int(cudaErrorNotSupported);
  cuuint64_t gdim[2] = {cols, rows};
  cuuint64_t gstride[1] = {cols * 2};
  cuuint32_t box[2] = {64, 16};
  cuuint32_t estride[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride,
                   box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : int(cudaErrorInvalidValue);
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!g_sm_count[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

template <int D, int G>
int launch_tc_t(const DecodeLaunch& Lc, cudaStream_t stream) {
  using C = TcCfg<D>;
  const pa_decode_params* p = Lc.p;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(paged_decode_tc_kernel<D, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return int(e);
    configured = true;
  }
  CUtensorMap tk, tv, tq;
  const uint64_t cache_rows = uint64_t(p->num_blocks) * p->num_kv_heads * BS;
  int r = make_map(&tk, p->k_cache, cache_rows, D);
  if (!r) r = make_map(&tv, p->v_cache, cache_rows, D);
  if (!r) r = make_map(&tq, p->q, uint64_t(p->num_seqs) * p->num_q_heads, D);
  if (r) return r;
  TcParams P;
  P.block_tables = p->block_tables;
  P.context_lens = p->context_lens;
  P.out = static_cast<__nv_bfloat16*>(p->out);
  P.part_m = Lc.part_m;
  P.part_l = Lc.part_l;
  P.part_acc = Lc.part_acc;
  P.counters = Lc.counters;
  P.max_blocks_per_seq = p->max_blocks_per_seq;
  P.num_seqs = p->num_seqs;
  P.num_kv_heads = p->num_kv_heads;
  P.num_q_heads = p->num_q_heads;
  P.group = G;
  P.num_blocks = p->num_blocks;
  P.max_context_len = p->max_context_len;
  P.partition_tokens = Lc.partition_tokens;
  P.num_partitions = Lc.num_partitions;
  P.total_items = Lc.num_partitions * p->num_seqs * p->num_kv_heads;
  P.oob_row = int(cache_rows);
  P.scale_log2 = p->scale * kLog2e;
  int sms = sm_count();
  if (sms <= 0) return int(cudaErrorInvalidDevice);
  const int grid = P.total_items < sms ? P.total_items : sms;
  paged_decode_tc_kernel<D, G><<<grid, NTHREADS, C::SMEM, stream>>>(tk, tv, tq, P);
  return int(cudaGetLastError());
}

template <int D>
int dispatch_tc(const DecodeLaunch& Lc, cudaStream_t s) {
  switch (Lc.p->num_q_heads / Lc.p->num_kv_heads) {
    case 1: return launch_tc_t<D, 1>(Lc, s);
    case 2: return launch_tc_t<D, 2>(Lc, s);
    case 4: return launch_tc_t<D, 4>(Lc, s);
    case 8: return launch_tc_t<D, 8>(Lc, s);
    default: return int(cudaErrorInvalidValue);
  }
}

}  // namespace

int launch_decode_tc(const DecodeLaunch& Lc, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (Lc.p->head_dim) {
    case 64: return dispatch_tc<64>(Lc, s);
    case 128: return dispatch_tc<128>(Lc, s);
    default: return int(cudaErrorInvalidValue);
  }
}

int read_and_clear_decode_tc_errors(uint32_t* flags) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_tc_errors, sizeof(v));
  if (e != cudaSuccess) return int(e);
  e = cudaMemcpyToSymbol(g_tc_errors, &zero, sizeof(zero));
  *flags = v;
  return int(e);
}

}  // namespace pa
