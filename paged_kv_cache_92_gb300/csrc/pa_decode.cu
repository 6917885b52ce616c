// Paged decode attention for sm_103a.
//
// What it computes ("Paged Attention as a Memory Manager", §How the Kernel
// Executes Paged Attention; "PagedAttention and continuous batching",
// §Attention kernel modification): for each sequence b and query head h,
// softmax(scale * q.K^T) V over the sequence's cached tokens, with K/V read
// block by block through the block table and a running softmax carried
// across blocks. Tokens past the context length inside the last block are
// masked. With Q new tokens per sequence ("How Paged Attention and
// Continuous Batching Actually Work", §Continuous batching) row (b, i) of q
// is token L - Q + i of its sequence and sees its first L - Q + i + 1 tokens;
// each (sequence, token) is decoded as a sequence of its own (grid z).
//
// GB300 design (the pages' thread-group layout targets older GPUs and is not
// followed):
//  * One CTA per (partition of up to `partition_tokens` tokens, KV head,
//    sequence). The CTA packs all G = Hq/Hkv query heads of the KV group, so
//    every K/V byte leaves HBM once.
//  * The partition's block-table slice is read once into shared memory and
//    broadcast; each entry is range-checked there.
//  * Each of the 4 warps owns every 4th block of the partition and runs its
//    own ring of ST stages: lane 0 issues 1-D bulk async copies (TMA, no
//    tensor map) of the 4 KiB K tile and the 4 KiB V tile of a (block, KV
//    head) into shared memory, completion tracked by an mbarrier with a
//    bounded wait. No CTA-wide barrier inside the block loop.
//  * Math on CUDA cores in fp32: a warp covers TPI tokens per step, LPT lanes
//    per token, each lane a DPL-dim slice read with 16-byte conflict-free
//    shared loads. Per-head partial dot products are reduce-scattered across
//    the LPT lanes with shuffles; the running max / sum / rescale use exp2
//    with log2(e) folded into the query.
//  * The 4 warps' (max, sum, acc) are merged through shared memory. One
//    partition: normalised bf16 output. Several: fp32 partials to the
//    workspace, combined by the merge kernel (log-sum-exp).
//  * The reduction order depends only on logical token positions, so results
//    are bit-identical under any physical block placement.
//  * The 8-bit (E4M3) cache ("PagedAttention" glossary page, §What paging
//    costs): K rows are read as 8-byte chunks of codes, dequantised on the
//    fly with the head's K scale folded into the query; each (block, head)
//    V^T tile ([D][16] codes) is transposed in shared memory into V rows,
//    which the value loop reads like K, and the head's V scale multiplies the
//    weighted sum before the normalisation.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__device__ unsigned int g_decode_errors;

constexpr int NWARPS = 4;
constexpr int NTHREADS = NWARPS * 32;
constexpr float kLog2e = 1.4426950408889634f;

template <int D, int G, bool F8, int BS>
struct Cfg {
  // dims per lane: keep the per-lane query registers (DPL * G) at 64.
  static constexpr int DPL = (D >= 128 && G <= 4) ? 16 : 8;
  static constexpr int LPT = D / DPL;    // lanes per token
  static constexpr int TPI = 32 / LPT;   // tokens per warp step
  static constexpr int NIT = BS / TPI;   // warp steps per block
  static constexpr int CHUNKS = DPL / 8; // 8-element chunks per lane per row
  static constexpr int EB = F8 ? 1 : 2;  // bytes per cache element
  static constexpr int HSTRIDE = LPT / G;  // lanes between heads after the reduce-scatter
  static constexpr int TILE = BS * D * EB;  // bytes of one (block, KV head) tile
  static constexpr int ST = (D >= 128) ? 3 : 4;  // ring stages per warp
  // 8-bit: each warp's V rows, transposed from the V^T tile of its block
  // (sub-tiles of W keys)
  static constexpr int VROWS = F8 ? BS * D : 0;
  static constexpr int W = BS < 16 ? BS : 16;
  static_assert(G <= LPT, "each head needs a lane after the reduce-scatter");
  static_assert(BS % TPI == 0, "tokens per step must divide the block");
};

template <int D, int G, bool F8, int BS>
constexpr size_t decode_smem_bytes(int partition_tokens) {
  using C = Cfg<D, G, F8, BS>;
  size_t tiles = size_t(NWARPS) * (C::ST * 2 * C::TILE + C::VROWS);
  size_t merge = size_t(NWARPS) * G * (D + 2) * sizeof(float);
  if (merge > tiles) tiles = merge;
  return tiles + size_t(NWARPS) * C::ST * sizeof(uint64_t) +
         size_t(partition_tokens / BS) * sizeof(int32_t);
}

// 8 consecutive elements of a row in shared memory as floats: bf16 (16 bytes)
// or E4M3 codes (8 bytes).
template <bool F8>
__device__ __forceinline__ void load_row8(const unsigned char* p, float (&f)[8]) {
  if constexpr (F8) {
    const uint2 raw = *reinterpret_cast<const uint2*>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = dev::from_e4m3x2(((i < 2 ? raw.x : raw.y) >> (16 * (i & 1))) & 0xffffu);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  } else {
    dev::unpack8(*reinterpret_cast<const uint4*>(p), f);
  }
}

// Sum G values over the LPT lanes of a token group, scattering heads: on
// return v[0] holds the full sum for head (dl / HSTRIDE), dl = lane % LPT.
template <int G, int LPT>
__device__ __forceinline__ float reduce_scatter(float (&v)[G], int lane) {
  int n = G;
#pragma unroll
  for (int m = LPT / 2; m >= 1; m >>= 1) {
    if (n > 1) {
      const bool upper = (lane & m) != 0;
#pragma unroll
      for (int i = 0; i < G / 2; ++i) {
        if (i < n / 2) {
          const float send = upper ? v[i] : v[i + n / 2];
          const float keep = upper ? v[i + n / 2] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
      }
      n >>= 1;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], m);
    }
  }
  return v[0];
}

template <int D, int G, bool F8, int BS>
__global__ void __launch_bounds__(NTHREADS)
    paged_decode_kernel(const __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ out,
                        const unsigned char* __restrict__ k_cache,
                        const unsigned char* __restrict__ v_cache,
                        const float* __restrict__ k_scale, const float* __restrict__ v_scale,
                        const int32_t* __restrict__ block_tables,
                        const int32_t* __restrict__ context_lens, int max_blocks_per_seq,
                        int num_kv_heads, int num_blocks, int max_context_len, float scale_log2,
                        int partition_tokens, int num_partitions, float* __restrict__ part_m,
                        float* __restrict__ part_l, float* __restrict__ part_acc, int q_len) {
  using C = Cfg<D, G, F8, BS>;
  constexpr int ST = C::ST;
  const int part = blockIdx.x;
  const int g = blockIdx.y;
  const int z = blockIdx.z;  // row of q / out: sequence b, its new token qi
  const int b = z / q_len, qi = z - (z / q_len) * q_len;
  const int num_q_heads = num_kv_heads * G;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  int L = context_lens[b];
  const int cap = min(max_blocks_per_seq * BS, max_context_len);
  const bool report = tid == 0 && part == 0 && g == 0 && qi == 0;
  if (L > cap) {
    if (report) atomicOr(&g_decode_errors, PA_DEVERR_CONTEXT_LEN);
    L = cap;
  }
  if (L > 0 && L < q_len) {  // no room for the new tokens: an empty sequence
    if (report) atomicOr(&g_decode_errors, PA_DEVERR_CONTEXT_LEN);
    L = 0;
  }
  if (L > 0) L = L - q_len + qi + 1;  // the keys token qi sees
  if (L <= 0) {
    if (part == 0) {
      for (int i = tid; i < G * D; i += NTHREADS)
        out[(size_t(z) * num_q_heads + g * G) * D + i] = __float2bfloat16_rn(0.0f);
    }
    return;
  }
  const int tok0 = part * partition_tokens;
  if (tok0 >= L) return;
  const int tok1 = min(L, tok0 + partition_tokens);
  const int lblk0 = tok0 / BS;
  const int nblk = (tok1 - tok0 + BS - 1) / BS;
  const bool split = L > partition_tokens;

  extern __shared__ __align__(128) unsigned char smem[];
  size_t tiles_bytes = size_t(NWARPS) * (ST * 2 * C::TILE + C::VROWS);
  {
    const size_t merge = size_t(NWARPS) * G * (D + 2) * sizeof(float);
    if (merge > tiles_bytes) tiles_bytes = merge;
  }
  unsigned char* tiles = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + tiles_bytes);
  int32_t* table = reinterpret_cast<int32_t*>(bars + NWARPS * ST);

  // Block-table slice of this partition: read once, range-checked, broadcast.
  const int32_t* trow = block_tables + size_t(b) * max_blocks_per_seq + lblk0;
  for (int i = tid; i < nblk; i += NTHREADS) {
    int32_t e = trow[i];
    if (e < 0 || e >= num_blocks) {
      atomicOr(&g_decode_errors, PA_DEVERR_TABLE_ENTRY);
      e = 0;
    }
    table[i] = e;
  }
  uint64_t* my_bars = bars + warp * ST;
  if (lane == 0) {
    for (int s = 0; s < ST; ++s) dev::mbar_init(&my_bars[s], 1);
    dev::fence_barrier_init();
  }
  __syncthreads();

  const int n_my = nblk > warp ? (nblk - warp + NWARPS - 1) / NWARPS : 0;
  unsigned char* my_tiles = tiles + size_t(warp) * (ST * 2 * C::TILE + C::VROWS);
  unsigned char* my_vrows = my_tiles + ST * 2 * C::TILE;  // 8-bit: [BS][D] codes
  const size_t head_tile_bytes = size_t(C::TILE);
  const uint64_t policy = dev::l2_evict_first_policy();

  auto issue = [&](int i) {
    const int s = i % ST;
    const int32_t blk = table[warp + NWARPS * i];
    const size_t off = (size_t(blk) * num_kv_heads + g) * head_tile_bytes;
    dev::mbar_arrive_expect_tx(&my_bars[s], 2 * C::TILE);
    dev::bulk_load(my_tiles + size_t(s) * 2 * C::TILE, k_cache + off, C::TILE, &my_bars[s], policy);
    dev::bulk_load(my_tiles + size_t(s) * 2 * C::TILE + C::TILE, v_cache + off, C::TILE,
                   &my_bars[s], policy);
  };
  if (lane == 0) {
    for (int i = 0; i < ST && i < n_my; ++i) issue(i);
  }

  // Query slice of this lane, prescaled by scale*log2(e) (and, 8-bit, the
  // head's K scale): qf[h][k*8+e].
  const int dl = lane % C::LPT;
  const int tg = lane / C::LPT;
  const float qscale = F8 ? scale_log2 * k_scale[g] : scale_log2;
  float qf[G][C::DPL];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const uint4* qrow =
        reinterpret_cast<const uint4*>(q + (size_t(z) * num_q_heads + g * G + h) * D);
#pragma unroll
    for (int k = 0; k < C::CHUNKS; ++k) {
      float f[8];
      dev::unpack8(qrow[dl + C::LPT * k], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) qf[h][k * 8 + e] = f[e] * qscale;
    }
  }

  float acc[G][C::DPL];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int j = 0; j < C::DPL; ++j) acc[h][j] = 0.0f;
  float m_run = -INFINITY;  // running max of this lane's head (log2 domain)
  float l_part = 0.0f;      // running sum over this lane's tokens, same head
  int stalled_at = -1;  // block index whose wait ran out, if any

  for (int i = 0; i < n_my; ++i) {
    const int s = i % ST;
    // Warp-uniform outcome: if any lane's bounded wait ran out, all stop.
    if (!__all_sync(0xffffffffu, dev::mbar_wait(&my_bars[s], (i / ST) & 1))) {
      stalled_at = i;
      break;
    }
    const unsigned char* kt = my_tiles + size_t(s) * 2 * C::TILE;
    const unsigned char* vt = kt + C::TILE;
    if constexpr (F8) {
      // V^T sub-tiles [D][W keys] -> V rows [BS keys][D]: lane l takes V^T
      // rows RPL*l .. RPL*l + RPL-1 of each sub-tile and stores, per key,
      // their RPL codes together.
      constexpr int RPL = D / 32;
      constexpr int W = C::W;
#pragma unroll
      for (int sub = 0; sub < BS / W; ++sub) {
        uint32_t r[RPL][W / 4];
#pragma unroll
        for (int j = 0; j < RPL; ++j) {
          const unsigned char* src = vt + (sub * D + RPL * lane + j) * W;
          if constexpr (W == 16) {
            const uint4 x = *reinterpret_cast<const uint4*>(src);
            r[j][0] = x.x; r[j][1] = x.y; r[j][2] = x.z; r[j][3] = x.w;
          } else {
            const uint2 x = *reinterpret_cast<const uint2*>(src);
            r[j][0] = x.x; r[j][1] = x.y;
          }
        }
#pragma unroll
        for (int t = 0; t < W; ++t) {
          uint32_t w = 0;
#pragma unroll
          for (int j = 0; j < RPL; ++j) w |= ((r[j][t >> 2] >> ((t & 3) * 8)) & 0xffu) << (8 * j);
          unsigned char* dst = my_vrows + (sub * W + t) * D + RPL * lane;
          if constexpr (RPL == 4) {
            *reinterpret_cast<uint32_t*>(dst) = w;
          } else {
            *reinterpret_cast<uint16_t*>(dst) = uint16_t(w);
          }
        }
      }
      __syncwarp();
    }
    const unsigned char* vrows = F8 ? my_vrows : vt;
    const int t_base = (lblk0 + warp + NWARPS * i) * BS;
    const bool partial = t_base + BS > L;

    float sc[C::NIT];
#pragma unroll
    for (int it = 0; it < C::NIT; ++it) {
      const int t = it * C::TPI + tg;
      float part_dot[G];
#pragma unroll
      for (int h = 0; h < G; ++h) part_dot[h] = 0.0f;
#pragma unroll
      for (int k = 0; k < C::CHUNKS; ++k) {
        float f[8];
        load_row8<F8>(kt + (size_t(t) * D + (dl + C::LPT * k) * 8) * C::EB, f);
#pragma unroll
        for (int e = 0; e < 8; ++e)
#pragma unroll
          for (int h = 0; h < G; ++h) part_dot[h] = fmaf(qf[h][k * 8 + e], f[e], part_dot[h]);
      }
      const float sv = reduce_scatter<G, C::LPT>(part_dot, lane);
      sc[it] = (partial && t_base + t >= L) ? -INFINITY : sv;
    }
    float bmax = sc[0];
#pragma unroll
    for (int it = 1; it < C::NIT; ++it) bmax = fmaxf(bmax, sc[it]);
#pragma unroll
    for (int m = C::LPT; m < 32; m <<= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, m));
    const float m_new = fmaxf(m_run, bmax);
    if (__any_sync(0xffffffffu, m_new > m_run)) {
      const float alpha = dev::fast_exp2(m_run - m_new);
      l_part *= alpha;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float ah = __shfl_sync(0xffffffffu, alpha, h * C::HSTRIDE);
#pragma unroll
        for (int j = 0; j < C::DPL; ++j) acc[h][j] *= ah;
      }
      m_run = m_new;
    }
#pragma unroll
    for (int it = 0; it < C::NIT; ++it) {
      const int t = it * C::TPI + tg;
      const float p = dev::fast_exp2(sc[it] - m_run);
      l_part += p;
      float ph[G];
#pragma unroll
      for (int h = 0; h < G; ++h) ph[h] = __shfl_sync(0xffffffffu, p, tg * C::LPT + h * C::HSTRIDE);
      const bool masked = partial && t_base + t >= L;
#pragma unroll
      for (int k = 0; k < C::CHUNKS; ++k) {
        float f[8];
        load_row8<F8>(vrows + (size_t(t) * D + (dl + C::LPT * k) * 8) * C::EB, f);
        if (masked) {
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = 0.0f;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e)
#pragma unroll
          for (int h = 0; h < G; ++h) acc[h][k * 8 + e] = fmaf(ph[h], f[e], acc[h][k * 8 + e]);
      }
    }
    __syncwarp();
    if (lane == 0 && i + ST < n_my) issue(i + ST);
  }

  if (stalled_at >= 0) {
    // Record the stall, then wait (bounded) for this warp's copies still in
    // flight -- blocks stalled_at .. stalled_at+ST-1 -- so that no bulk copy
    // lands in shared memory after the CTA has exited. The output of this
    // CTA is unspecified.
    if (lane == 0) atomicOr(&g_decode_errors, PA_DEVERR_TIMEOUT);
    for (int j = stalled_at; j < n_my && j < stalled_at + ST; ++j)
      (void)dev::mbar_wait(&my_bars[j % ST], (j / ST) & 1);
  }

  // Totals over the token groups of the warp (lanes that share dl).
#pragma unroll
  for (int m = C::LPT; m < 32; m <<= 1) {
    l_part += __shfl_xor_sync(0xffffffffu, l_part, m);
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int j = 0; j < C::DPL; ++j) acc[h][j] += __shfl_xor_sync(0xffffffffu, acc[h][j], m);
  }

  // Merge the 4 warps through shared memory (reusing the tile ring).
  __syncthreads();
  float* sm_acc = reinterpret_cast<float*>(tiles);  // [NWARPS][G][D]
  float* sm_m = sm_acc + NWARPS * G * D;            // [NWARPS][G]
  float* sm_l = sm_m + NWARPS * G;                  // [NWARPS][G]
  if (tg == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int k = 0; k < C::CHUNKS; ++k) {
        float4* dst =
            reinterpret_cast<float4*>(sm_acc + (warp * G + h) * D + (dl + C::LPT * k) * 8);
        dst[0] = make_float4(acc[h][k * 8 + 0], acc[h][k * 8 + 1], acc[h][k * 8 + 2],
                             acc[h][k * 8 + 3]);
        dst[1] = make_float4(acc[h][k * 8 + 4], acc[h][k * 8 + 5], acc[h][k * 8 + 6],
                             acc[h][k * 8 + 7]);
      }
    if (dl % C::HSTRIDE == 0) {
      sm_m[warp * G + dl / C::HSTRIDE] = m_run;
      sm_l[warp * G + dl / C::HSTRIDE] = l_part;
    }
  }
  __syncthreads();

  for (int idx = tid; idx < G * D; idx += NTHREADS) {
    const int h = idx / D;
    const int d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NWARPS; ++w) M = fmaxf(M, sm_m[w * G + h]);
    float num = 0.0f, den = 0.0f;
#pragma unroll
    for (int w = 0; w < NWARPS; ++w) {
      const float wt = dev::fast_exp2(sm_m[w * G + h] - M);
      num = fmaf(wt, sm_acc[(w * G + h) * D + d], num);
      den = fmaf(wt, sm_l[w * G + h], den);
    }
    if constexpr (F8) num *= v_scale[g];  // the head's V dequantisation scale
    const size_t row = size_t(z) * num_q_heads + g * G + h;
    if (!split) {
      out[row * D + d] = __float2bfloat16_rn(num * __frcp_rn(den));
    } else {
      const size_t prow = row * num_partitions + part;
      part_acc[prow * D + d] = num;
      if (d == 0) {
        part_m[prow] = M;
        part_l[prow] = den;
      }
    }
  }
}

// Log-sum-exp merge of split-K partials: one warp per (row of q, query head),
// a row being a sequence's new token.
template <int D>
__global__ void __launch_bounds__(128)
    merge_partitions_kernel(__nv_bfloat16* __restrict__ out, const float* __restrict__ part_m,
                            const float* __restrict__ part_l, const float* __restrict__ part_acc,
                            const int32_t* __restrict__ context_lens, int num_q_heads,
                            int max_blocks_per_seq, int max_context_len, int partition_tokens,
                            int num_partitions, int q_len, int block_size) {
  constexpr int VPL = D / 32;  // values per lane
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.x * 4 + warp;
  const int z = blockIdx.y;
  const int b = z / q_len, qi = z - (z / q_len) * q_len;
  if (h >= num_q_heads) return;
  int L = context_lens[b];
  L = min(L, min(max_blocks_per_seq * block_size, max_context_len));
  if (L < q_len) return;  // empty: zero rows written by the decode kernel
  L = L - q_len + qi + 1;
  if (L <= partition_tokens) return;  // written directly by the decode kernel
  const int np = (L + partition_tokens - 1) / partition_tokens;
  const size_t row = (size_t(z) * num_q_heads + h) * num_partitions;
  float M = -INFINITY;
  for (int p = lane; p < np; p += 32) M = fmaxf(M, part_m[row + p]);
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
  float acc[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) acc[j] = 0.0f;
  float den = 0.0f;
  for (int p = 0; p < np; ++p) {
    const float wt = dev::fast_exp2(part_m[row + p] - M);
    den = fmaf(wt, part_l[row + p], den);
    const float* src = part_acc + (row + p) * D + lane * VPL;
    if constexpr (VPL == 4) {
      const float4 v = *reinterpret_cast<const float4*>(src);
      acc[0] = fmaf(wt, v.x, acc[0]);
      acc[1] = fmaf(wt, v.y, acc[1]);
      acc[2] = fmaf(wt, v.z, acc[2]);
      acc[3] = fmaf(wt, v.w, acc[3]);
    } else {
#pragma unroll
      for (int j = 0; j < VPL; ++j) acc[j] = fmaf(wt, src[j], acc[j]);
    }
  }
  const float inv = __frcp_rn(den);
  __nv_bfloat16* o = out + (size_t(z) * num_q_heads + h) * D + lane * VPL;
#pragma unroll
  for (int j = 0; j < VPL; ++j) o[j] = __float2bfloat16_rn(acc[j] * inv);
}

template <int D, int G, bool F8, int BS>
int launch_decode_t(const DecodeLaunch& Lc, cudaStream_t stream) {
  const pa_decode_params* p = Lc.p;
  const size_t smem = decode_smem_bytes<D, G, F8, BS>(Lc.partition_tokens);
  static size_t configured = 0;
  if (configured < smem) {
    cudaError_t e = cudaFuncSetAttribute(paged_decode_kernel<D, G, F8, BS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return int(e);
    configured = smem;
  }
  const int q_len = query_len_of(p);
  dim3 grid(Lc.num_partitions, p->num_kv_heads, p->num_seqs * q_len);
  const float scale_log2 = p->scale * kLog2e;
  paged_decode_kernel<D, G, F8, BS><<<grid, NTHREADS, smem, stream>>>(
      static_cast<const __nv_bfloat16*>(p->q), static_cast<__nv_bfloat16*>(p->out),
      static_cast<const unsigned char*>(p->k_cache), static_cast<const unsigned char*>(p->v_cache),
      p->k_scale, p->v_scale, p->block_tables, p->context_lens, p->max_blocks_per_seq, p->num_kv_heads, p->num_blocks,
      p->max_context_len, scale_log2, Lc.partition_tokens, Lc.num_partitions, Lc.part_m, Lc.part_l,
      Lc.part_acc, q_len);
  return int(cudaGetLastError());
}

template <int D>
int launch_merge_t(const DecodeLaunch& Lc, cudaStream_t stream) {
  const pa_decode_params* p = Lc.p;
  const int q_len = query_len_of(p);
  dim3 mgrid((p->num_q_heads + 3) / 4, p->num_seqs * q_len);
  merge_partitions_kernel<D><<<mgrid, 128, 0, stream>>>(
      static_cast<__nv_bfloat16*>(p->out), Lc.part_m, Lc.part_l, Lc.part_acc, p->context_lens,
      p->num_q_heads, p->max_blocks_per_seq, p->max_context_len, Lc.partition_tokens,
      Lc.num_partitions, q_len, p->block_size);
  return int(cudaGetLastError());
}

template <int D, bool F8, int BS>
int dispatch_group(const DecodeLaunch& Lc, cudaStream_t s) {
  switch (Lc.p->num_q_heads / Lc.p->num_kv_heads) {
    case 1: return launch_decode_t<D, 1, F8, BS>(Lc, s);
    case 2: return launch_decode_t<D, 2, F8, BS>(Lc, s);
    case 4: return launch_decode_t<D, 4, F8, BS>(Lc, s);
    case 8: return launch_decode_t<D, 8, F8, BS>(Lc, s);
    default: return int(cudaErrorInvalidValue);
  }
}

template <int D, bool F8>
int dispatch_block(const DecodeLaunch& Lc, cudaStream_t s) {
  switch (Lc.p->block_size) {
    case 8: return dispatch_group<D, F8, 8>(Lc, s);
    case 16: return dispatch_group<D, F8, 16>(Lc, s);
    case 32: return dispatch_group<D, F8, 32>(Lc, s);
    default: return int(cudaErrorInvalidValue);
  }
}

}  // namespace

int launch_decode(const DecodeLaunch& Lc, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool f8 = Lc.p->kv_dtype == PA_KV_FP8_E4M3;
  switch (Lc.p->head_dim) {
    case 64: return f8 ? dispatch_block<64, true>(Lc, s) : dispatch_block<64, false>(Lc, s);
    case 128: return f8 ? dispatch_block<128, true>(Lc, s) : dispatch_block<128, false>(Lc, s);
    default: return int(cudaErrorInvalidValue);
  }
}

// ---------------------------------------------------------------------------
// Decode without any caller-provided workspace.
//
// Some callers cannot allocate device memory when they decode: an engine that
// carved all free HBM into its KV block pool at start-up has nothing left to
// hand out, and a serving loop that must not stall cannot afford cudaMalloc's
// implicit synchronisation. For them the split-K partials live in this
// file-scope device array instead of a workspace. Every GPU that loads the
// library holds the array until the process exits.
//
// Host code cannot pass the array's name to a kernel (on the host it is only
// a stand-in, not a device address), so its device address is looked up with
// cudaGetSymbolAddress, with the device current, on the first call made in
// each CUDA context, and cached under the context's process-unique ID
// (cuCtxGetId). A device reset, or a driver-API context other than the
// primary one, is a new context: the address is looked up again there
// instead of reusing one that may no longer be valid.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
struct ScratchEntry {
  unsigned long long ctx_id;  // 0: not looked up yet
  void* addr;
};
ScratchEntry g_scratch[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
std::once_flag g_ctx_fn_once;
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// The process-unique ID of the calling thread's current context, 0 if there is none.
unsigned long long current_context_id() {
  std::call_once(g_ctx_fn_once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  if (!g_ctx_get_current || !g_ctx_get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}
}  // namespace

int decode_scratch_address(void** addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return int(e);
  if (dev < 0 || dev >= kMaxDevices) return int(cudaErrorInvalidDevice);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  const unsigned long long id = current_context_id();
  if (id == 0 || g_scratch[dev].ctx_id != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);  // makes the device's context current
    if (e != cudaSuccess) return int(e);
    // the context the lookup ran in (it may have just been created)
    g_scratch[dev].ctx_id = current_context_id();
    g_scratch[dev].addr = p;
  }
  *addr = g_scratch[dev].addr;
  return int(cudaSuccess);
}

int launch_merge(const DecodeLaunch& Lc, void* stream) {
  if (Lc.num_partitions <= 1) return int(cudaSuccess);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (Lc.p->head_dim) {
    case 64: return launch_merge_t<64>(Lc, s);
    case 128: return launch_merge_t<128>(Lc, s);
    default: return int(cudaErrorInvalidValue);
  }
}

int read_and_clear_decode_errors(uint32_t* flags) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_decode_errors, sizeof(v));
  if (e != cudaSuccess) return int(e);
  e = cudaMemcpyToSymbol(g_decode_errors, &zero, sizeof(zero));
  *flags = v;
  return int(e);
}

}  // namespace pa
