// Paged MLA decode on sm_103a tensor cores: a persistent kernel of CTA pairs
// (thread-block clusters of 2) with TMA page gathers, tcgen05 MMAs and
// tensor-memory (TMEM) accumulators.
//
// What it computes (problem statement of the FlashInfer page
// "prims_ts_batch_decode_with_kv_cache_mla"): for the 128 query rows
// (token x head) of one work item and the KV rows [kv_begin, kv_end) of its
// request, gathered page by page through block_tables,
//   S = Q K^T (576 dims),  P = softmax(bmm1 * S) under the bottom-right causal
//   (or dense) mask,  O = P V (V = first 512 dims of the same rows),
// streaming the KV range in 64-row tiles with an online (running-max) softmax.
//
// GB300 mapping.  A 128 x 512 fp32 accumulator fills a whole SM's TMEM and a
// 128 x 576 bf16 query tile nearly half its shared memory, so one work item
// is shared by the two CTAs of a cluster:
//  * the QK contraction is split along its 576 dims: CTA r holds 64-dim
//    chunks 4r .. 4r+4 of Q and of every KV tile and contracts 288 of the 576
//    dims (18 MMA K-steps of 16) into a partial S (M = 128 query rows,
//    N = 64 KV rows, fp32 in TMEM);
//  * the partial scores are exchanged through distributed shared memory, so
//    both CTAs hold the full S and run identical (bitwise equal) softmaxes;
//  * CTA r accumulates O^T for V dims [256 r, 256 r + 256) (its local chunks
//    0..3): O^T = V^T P^T with M = 128 V dims, N = 128 query rows, K = 64
//    KV rows -- two 128 x 128 fp32 TMEM blocks.
// Warp roles (384 threads): warp 0 TMA producer, warp 1 MMA issuer (and TMEM
// owner), warps 4-7 softmax (thread = query row = TMEM lane), warps 8-11
// O correction and epilogue (thread = V dim = TMEM lane).  The running max
// is only raised (and O^T rescaled) when it grows by more than 2^8, so most
// tiles need no correction pass.  Every wait is bounded; a timeout sets an
// error bit in the workspace status word and the kernel unwinds.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "mla_common.cuh"
#include "sm100_ptx.cuh"

namespace mla {

namespace {

using namespace ptx;

constexpr int kRows = 128;        // query rows per work item
constexpr int kTile = kKvTile;    // 64 KV rows per tile
constexpr int kLocalChunks = 5;   // 64-dim chunks each CTA holds (4r .. 4r+4)
constexpr int kQkSteps = 18;      // 16-wide K steps of the QK contraction per CTA
constexpr int kThreads = 384;
constexpr uint32_t kWaitLimit = 1u << 26;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// shared-memory layout (bytes from a 1024-aligned base)
constexpr uint32_t kChunkQ = kRows * 128;   // one 64-dim chunk of Q: 128 rows x 128 B
constexpr uint32_t kChunkKV = kTile * 128;  // one 64-dim chunk of a KV tile
constexpr uint32_t kStageBytes = kLocalChunks * kChunkKV;
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_KV = OFF_Q + kLocalChunks * kChunkQ;
constexpr uint32_t OFF_P = OFF_KV + 2 * kStageBytes;
constexpr uint32_t OFF_X = OFF_P + kRows * 128;
constexpr uint32_t OFF_MISC = OFF_X + kRows * kTile * 4;
constexpr uint32_t OFF_BARS = OFF_MISC;
constexpr uint32_t OFF_FAC = OFF_MISC + 512;          // float[2][128]
constexpr uint32_t OFF_STAT_M = OFF_FAC + 1024;       // float[2][128]
constexpr uint32_t OFF_STAT_L = OFF_STAT_M + 1024;    // float[2][128]
constexpr uint32_t OFF_FLAG = OFF_STAT_L + 1024;      // int[2] tile ids needing correction
constexpr uint32_t OFF_TMEM = OFF_FLAG + 16;
constexpr uint32_t OFF_ABORT = OFF_TMEM + 16;
constexpr uint32_t kSmemUsed = OFF_ABORT + 16;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;     // + alignment slack

// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_O = 0;    // two 128-column O^T blocks
constexpr uint32_t TM_S = 256;  // two 64-column S buffers

enum Bar {
  Q_FULL, Q_FREE, KV_FULL0, KV_FULL1, KV_EMPTY0, KV_EMPTY1, S_FULL0, S_FULL1, S_FREE0, S_FREE1,
  P_FULL, P_FREE, PV_DONE, CORR_REQ, CORR_DONE, X_FULL, X_FREE, STATS_READY, STATS_FREE, NUM_BARS
};

struct Ctx {
  unsigned char* sm;
  uint64_t* bars;
  volatile int* abort;
  int* status;
};

__device__ __forceinline__ bool wait_bar(const Ctx& c, int bar, uint32_t parity) {
  uint64_t* b = &c.bars[bar];
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    if (mbar_try_wait(b, parity)) return true;
    if ((i & 1023) == 1023 && *c.abort) return false;
  }
  *c.abort = 1;
  atomicOr(c.status, 32);
  return false;
}

__device__ __forceinline__ bool wait_bar_cluster(const Ctx& c, int bar, uint32_t parity) {
  uint64_t* b = &c.bars[bar];
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    if (mbar_try_wait_acq_cluster(b, parity)) return true;
    if ((i & 1023) == 1023 && *c.abort) return false;
  }
  *c.abort = 1;
  atomicOr(c.status, 32);
  return false;
}

__device__ __forceinline__ int n_tiles_of(const WorkItem& it) {
  return (it.kv_end - it.kv_begin + kTile - 1) / kTile;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
decode_sm103_kernel(const Problem p, const Layout lay, char* __restrict__ ws,
                    const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_kv) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int worker = (int)cluster_id_x();
  int* hdr = reinterpret_cast<int*>(ws);
  const WorkItem* items = reinterpret_cast<const WorkItem*>(ws + lay.items);
  const int* worker_begin = reinterpret_cast<const int*>(ws + lay.worker_ranges);
  float* part_o = reinterpret_cast<float*>(ws + lay.part_o);
  float* part_lse = reinterpret_cast<float*>(ws + lay.part_lse);

  Ctx c;
  c.sm = sm;
  c.bars = reinterpret_cast<uint64_t*>(sm + OFF_BARS);
  c.abort = reinterpret_cast<volatile int*>(sm + OFF_ABORT);
  c.status = &hdr[kHdrStatus];
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_TMEM);
  float* fac = reinterpret_cast<float*>(sm + OFF_FAC);
  float* stat_m = reinterpret_cast<float*>(sm + OFF_STAT_M);
  float* stat_l = reinterpret_cast<float*>(sm + OFF_STAT_L);
  volatile int* flag = reinterpret_cast<volatile int*>(sm + OFF_FLAG);

  if (tid == 0) {
    const uint32_t counts[NUM_BARS] = {1, 1, 1, 1, 1, 1, 1, 1, 128, 128,
                                       128, 1, 1, 128, 128, 128, 128, 128, 128};
    for (int i = 0; i < NUM_BARS; ++i) mbar_init(&c.bars[i], counts[i]);
    *c.abort = 0;
    flag[0] = -1;
    flag[1] = -1;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before any remote arrive
  const uint32_t tmem = *tmem_slot;
  const int item_begin = worker_begin[worker], item_end = worker_begin[worker + 1];
  const int H = p.num_heads;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_kv);
      uint32_t g = 0;
      int n_item = 0;
      const int ps = p.page_size;
      for (int idx = item_begin; idx < item_end; ++idx) {
        const WorkItem it = items[idx];
        const int nt = n_tiles_of(it);
        if (nt <= 0) continue;
        if (!wait_bar(c, Q_FREE, (n_item & 1) ^ 1)) goto done_producer;
        ++n_item;
        {
          mbar_arrive_expect_tx(&c.bars[Q_FULL], kLocalChunks * kChunkQ);
          const int qrow = it.q_start * H + it.g * kRows;
          for (int lc = 0; lc < kLocalChunks; ++lc)
            tma_load_2d(sm + OFF_Q + lc * kChunkQ, &tm_q, 64 * (4 * (int)rank + lc), qrow,
                        &c.bars[Q_FULL]);
        }
        for (int t = 0; t < nt; ++t, ++g) {
          const int s = g & 1;
          if (!wait_bar(c, KV_EMPTY0 + s, ((g >> 1) & 1) ^ 1)) goto done_producer;
          const int j0 = it.kv_begin + t * kTile;
          int pages[2];
          uint32_t bytes = 0;
          const int npg = kTile / ps;
          for (int pg = 0; pg < npg; ++pg) {
            const int jr = j0 + pg * ps;
            pages[pg] = -1;
            if (jr >= it.kv_end) continue;
            const int page = p.block_tables[(size_t)it.b * p.max_pages + jr / ps];
            if (page < 0 || (long long)page >= p.num_pages) {
              atomicOr(c.status, 16);
              continue;
            }
            pages[pg] = page;
            bytes += kLocalChunks * ps * 128;
          }
          mbar_arrive_expect_tx(&c.bars[KV_FULL0 + s], bytes);
          unsigned char* stage = sm + OFF_KV + s * kStageBytes;
          for (int pg = 0; pg < npg; ++pg) {
            if (pages[pg] < 0) continue;
            for (int lc = 0; lc < kLocalChunks; ++lc)
              tma_load_2d(stage + lc * kChunkKV + pg * ps * 128, &tm_kv, 64 * (4 * (int)rank + lc),
                          pages[pg] * ps, &c.bars[KV_FULL0 + s]);
          }
        }
      }
    done_producer:;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_f16(128, 64, false, false);
      constexpr uint32_t idesc_pv = idesc_f16(128, 128, true, false);
      const uint32_t q_base = smem_u32(sm + OFF_Q);
      const uint32_t kv_base = smem_u32(sm + OFF_KV);
      const uint32_t p_base = smem_u32(sm + OFF_P);
      uint32_t g = 0;
      int n_item = 0;
      bool ok = true;
      auto issue_qk = [&](uint32_t gq) -> bool {
        const int s = gq & 1;
        if (!wait_bar(c, KV_FULL0 + s, (gq >> 1) & 1)) return false;
        if (!wait_bar(c, S_FREE0 + s, ((gq >> 1) & 1) ^ 1)) return false;
        tc_fence_after();
        const uint32_t d = tmem + TM_S + 64 * s;
        for (int k = 0; k < kQkSteps; ++k) {
          const int gk = kQkSteps * (int)rank + k;  // global K step 0..35
          const int lc = gk / 4 - 4 * (int)rank;
          const int ks = gk % 4;
          const uint64_t a = smem_desc(q_base + lc * kChunkQ + ks * 32, 16, 1024, kSwizzle128B);
          const uint64_t b = smem_desc(kv_base + s * kStageBytes + lc * kChunkKV + ks * 32, 16,
                                       1024, kSwizzle128B);
          mma_bf16_ss(d, a, b, idesc_qk, k > 0 ? 1u : 0u);
        }
        mma_commit(&c.bars[S_FULL0 + s]);
        return true;
      };
      for (int idx = item_begin; idx < item_end && ok; ++idx) {
        const WorkItem it = items[idx];
        const int nt = n_tiles_of(it);
        if (nt <= 0) continue;
        if (!wait_bar(c, Q_FULL, n_item & 1)) break;
        ++n_item;
        tc_fence_after();
        if (!issue_qk(g)) break;
        for (int t = 0; t < nt; ++t, ++g) {
          if (t + 1 < nt) {
            if (!issue_qk(g + 1)) { ok = false; break; }
          } else {
            mma_commit(&c.bars[Q_FREE]);
          }
          if (!wait_bar(c, P_FULL, g & 1) || !wait_bar(c, CORR_DONE, g & 1)) { ok = false; break; }
          tc_fence_after();
          const int s = g & 1;
          for (int bb = 0; bb < 2; ++bb) {
            for (int ks = 0; ks < kTile / 16; ++ks) {
              const uint64_t a = smem_desc(kv_base + s * kStageBytes + (2 * bb) * kChunkKV +
                                               ks * 16 * 128,
                                           8192, 1024, kSwizzle128B);
              const uint64_t b = smem_desc(p_base + ks * 32, 16, 1024, kSwizzle128B);
              mma_bf16_ss(tmem + TM_O + 128 * bb, a, b, idesc_pv, (t == 0 && ks == 0) ? 0u : 1u);
            }
          }
          mma_commit(&c.bars[KV_EMPTY0 + s]);
          mma_commit(&c.bars[P_FREE]);
          mma_commit(&c.bars[PV_DONE]);
        }
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ softmax
    const int r = tid - 128;  // query row within the item == TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const float scale = p.bmm1_scale * kLog2e;
    const uint32_t x_local = smem_u32(sm + OFF_X + r * 256);
    const uint32_t x_peer = map_to_rank(x_local, peer);
    const uint32_t xfull_peer = map_to_rank(smem_u32(&c.bars[X_FULL]), peer);
    const uint32_t xfree_peer = map_to_rank(smem_u32(&c.bars[X_FREE]), peer);
    uint32_t g = 0;
    int n_item = 0;
    for (int idx = item_begin; idx < item_end; ++idx) {
      const WorkItem it = items[idx];
      const int nt = n_tiles_of(it);
      if (nt <= 0) continue;
      const int rows_total = it.q_len * H;
      const int row0 = it.g * kRows;
      const bool row_ok = r < rows_total - row0;
      const int qi = (row0 + r) / H;
      const int last = p.causal ? it.seq_len - it.q_len + qi : it.seq_len - 1;
      float m_ref = -INFINITY, l_sum = 0.f;
      for (int t = 0; t < nt; ++t, ++g) {
        const int s = g & 1;
        float sv[kTile];
        if (!wait_bar(c, S_FULL0 + s, (g >> 1) & 1)) goto done_softmax;
        tc_fence_after();
#pragma unroll
        for (int q4 = 0; q4 < kTile / 16; ++q4) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(tmem + lane_base + TM_S + 64 * s + 16 * q4, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) sv[16 * q4 + j] = __uint_as_float(v[j]);
        }
        tc_fence_before();
        mbar_arrive(&c.bars[S_FREE0 + s]);
        // exchange partial scores with the peer CTA
        if (!wait_bar(c, X_FREE, (g & 1) ^ 1)) goto done_softmax;
#pragma unroll
        for (int k = 0; k < 16; ++k)
          st_cluster_v4(x_peer + (uint32_t)((k ^ (r & 7)) << 4),
                        make_float4(sv[4 * k], sv[4 * k + 1], sv[4 * k + 2], sv[4 * k + 3]));
        mbar_arrive_cluster(xfull_peer);
        if (!wait_bar_cluster(c, X_FULL, g & 1)) goto done_softmax;
        {
          const float4* xs = reinterpret_cast<const float4*>(sm + OFF_X + r * 256);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float4 v = xs[k ^ (r & 7)];
            sv[4 * k] += v.x;
            sv[4 * k + 1] += v.y;
            sv[4 * k + 2] += v.z;
            sv[4 * k + 3] += v.w;
          }
        }
        mbar_arrive_cluster(xfree_peer);
        // mask, scale, online softmax
        const int j0 = it.kv_begin + t * kTile;
        float tmax = -INFINITY;
#pragma unroll
        for (int j = 0; j < kTile; ++j) {
          const int col = j0 + j;
          const bool ok = row_ok && col <= last && col < it.kv_end;
          sv[j] = ok ? sv[j] * scale : -INFINITY;
          tmax = fmaxf(tmax, sv[j]);
        }
        const float m_new = fmaxf(m_ref, tmax);
        bool need = false;
        float f = 1.f;
        if (t == 0) {
          m_ref = m_new;
        } else if (m_new > m_ref + kRescaleThreshold) {
          f = exp2f(m_ref - m_new);  // m_ref = -inf gives 0
          need = true;
          l_sum *= f;
          m_ref = m_new;
        }
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        float rs = 0.f;
#pragma unroll
        for (int j = 0; j < kTile; ++j) {
          sv[j] = exp2f(sv[j] - m_use);
          rs += sv[j];
        }
        l_sum += rs;
        // zero V rows past the end of the KV range in the last tile
        const int valid = it.kv_end - j0;
        if (valid < kTile) {
          unsigned char* stage = sm + OFF_KV + s * kStageBytes;
          const int nz = (kTile - valid) * 4 * 8;  // 16-byte units over 4 chunks
          for (int e = r; e < nz; e += 128) {
            const int row = valid + e / 32, ch = (e / 8) % 4, u = e % 8;
            *reinterpret_cast<uint4*>(stage + ch * kChunkKV + row * 128 + u * 16) =
                make_uint4(0, 0, 0, 0);
          }
        }
        // P (bf16) into the PV B-operand tile: row r, 128-byte swizzled
        if (!wait_bar(c, P_FREE, (g & 1) ^ 1)) goto done_softmax;
        {
          unsigned char* prow = sm + OFF_P + r * 128;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            uint4 w;
            w.x = pack_bf16(sv[8 * k + 0], sv[8 * k + 1]);
            w.y = pack_bf16(sv[8 * k + 2], sv[8 * k + 3]);
            w.z = pack_bf16(sv[8 * k + 4], sv[8 * k + 5]);
            w.w = pack_bf16(sv[8 * k + 6], sv[8 * k + 7]);
            *reinterpret_cast<uint4*>(prow + ((k ^ (r & 7)) << 4)) = w;
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&c.bars[P_FULL]);
        fac[(g & 1) * kRows + r] = f;
        if (__any_sync(0xffffffffu, need) && lane == 0) flag[g & 1] = (int)g;
        mbar_arrive(&c.bars[CORR_REQ]);
      }
      // final row statistics for the epilogue, LSE from CTA 0
      if (!wait_bar(c, STATS_FREE, (n_item & 1) ^ 1)) goto done_softmax;
      stat_m[(n_item & 1) * kRows + r] = m_ref;
      stat_l[(n_item & 1) * kRows + r] = l_sum;
      mbar_arrive(&c.bars[STATS_READY]);
      if (rank == 0 && row_ok) {
        const float lse = l_sum > 0.f ? (m_ref + log2f(l_sum)) * kLn2 : -INFINITY;
        const size_t grow = (size_t)it.q_start * H + row0 + r;
        if (it.slot < 0) {
          if (p.return_lse) p.lse[grow] = lse;
        } else {
          part_lse[(size_t)it.slot * kRows + r] = lse;
        }
      }
      ++n_item;
    }
  done_softmax:;
  } else if (warp >= 8) {
    // ------------------------------------------------------------ correction + epilogue
    const int v = tid - 256;  // V dim within each 128-wide O^T block == TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    uint32_t g = 0;
    int n_item = 0;
    for (int idx = item_begin; idx < item_end; ++idx) {
      const WorkItem it = items[idx];
      const int nt = n_tiles_of(it);
      if (nt <= 0) continue;
      for (int t = 0; t < nt; ++t, ++g) {
        if (!wait_bar(c, CORR_REQ, g & 1)) goto done_epi;
        if (t > 0 && flag[g & 1] == (int)g) {
          if (!wait_bar(c, PV_DONE, (g - 1) & 1)) goto done_epi;
          tc_fence_after();
          const float* f = fac + (g & 1) * kRows;
          for (int bb = 0; bb < 2; ++bb) {
#pragma unroll 1
            for (int q16 = 0; q16 < kRows / 16; ++q16) {
              uint32_t x[16];
              const uint32_t addr = tmem + lane_base + TM_O + 128 * bb + 16 * q16;
              tmem_ld_32x32b_x16(addr, x);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j)
                x[j] = __float_as_uint(__uint_as_float(x[j]) * f[16 * q16 + j]);
              tmem_st_32x32b_x16(addr, x);
            }
          }
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(&c.bars[CORR_DONE]);
      }
      if (!wait_bar(c, STATS_READY, n_item & 1)) goto done_epi;
      if (!wait_bar(c, PV_DONE, (g - 1) & 1)) goto done_epi;
      tc_fence_after();
      {
        const int rows_total = it.q_len * H;
        const int row0 = it.g * kRows;
        const int n_rows = min(kRows, rows_total - row0);
        const float* lrow = stat_l + (n_item & 1) * kRows;
        const size_t grow0 = (size_t)it.q_start * H + row0;
        for (int bb = 0; bb < 2; ++bb) {
          const int vd = 256 * (int)rank + 128 * bb + v;  // output V dim
#pragma unroll 1
          for (int q16 = 0; q16 < kRows / 16; ++q16) {
            uint32_t x[16];
            tmem_ld_32x32b_x16(tmem + lane_base + TM_O + 128 * bb + 16 * q16, x);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int q = 16 * q16 + j;
              if (q >= n_rows) break;
              const float l = lrow[q];
              const float inv = l > 0.f ? 1.f / l : 0.f;
              const float o = __uint_as_float(x[j]) * inv;
              if (it.slot < 0) {
                reinterpret_cast<__nv_bfloat16*>(p.out)[(grow0 + q) * kVDim + vd] =
                    __float2bfloat16_rn(o * p.bmm2_scale);
              } else {
                part_o[((size_t)it.slot * kRows + q) * kVDim + vd] = o;
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&c.bars[STATS_FREE]);
      ++n_item;
    }
  done_epi:;
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer no longer touches this CTA's shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side

namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, int elem_bytes, const void* base,
               uint64_t inner, uint64_t rows, uint32_t box_inner, uint32_t box_rows) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * elem_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t decode_sm103_setup(int sm_count, int* n_pairs) {
  cudaError_t e = cudaFuncSetAttribute(decode_sm103_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sm_count / 2), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, decode_sm103_kernel, &cfg);
  if (e != cudaSuccess) return e;
  if (clusters <= 0) return cudaErrorInvalidConfiguration;
  *n_pairs = std::min(clusters, sm_count / 2);
  return cudaSuccess;
}

cudaError_t launch_decode_sm103(const Problem& p, const Layout& lay, void* ws,
                                cudaStream_t stream) {
  CUtensorMap tm_q, tm_kv;
  const uint64_t q_rows = std::max<uint64_t>(1, (uint64_t)p.total_q * p.num_heads);
  if (!encode_2d(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.query, kQkDim, q_rows, 64, kRows))
    return cudaErrorInvalidValue;
  if (!encode_2d(&tm_kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.kv_cache, kQkDim,
                 (uint64_t)p.num_pages * p.page_size, 64, p.page_size))
    return cudaErrorInvalidValue;
  decode_sm103_kernel<<<lay.n_ctas, kThreads, kSmemBytes, stream>>>(p, lay, static_cast<char*>(ws),
                                                                     tm_q, tm_kv);
  return cudaGetLastError();
}

}  // namespace mla
