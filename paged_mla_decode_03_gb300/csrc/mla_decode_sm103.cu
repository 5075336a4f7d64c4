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
// 128 x 576 bf16 query tile needs 144 KB of shared memory, so one work item
// is shared by the two CTAs of a cluster:
//  * the QK contraction is split along its 576 dims: CTA r holds latent dims
//    [256 r, 256 r + 256) and RoPE dims [512 + 32 r, 512 + 32 r + 32) of Q
//    and of every KV tile (18 MMA K-steps of 16) and forms a partial
//    S_r (M = 128 query rows, N = 64 KV rows, fp32 in TMEM);
//  * the softmax is split by rows: CTA r owns query rows [64 r, 64 r + 64).
//    Its "sender" warps push the partial scores of the peer's rows into the
//    peer's shared memory with st.async (completing the peer's mbarrier
//    transaction count); its softmax warps add the peer's partial for their
//    own rows, normalise, write bf16 P rows and per-row rescale factors, and
//    a bulk DSMEM copy hands those to the peer, so both CTAs hold all 128
//    rows of P;
//  * CTA r accumulates O^T for V dims [256 r, 256 r + 256), i.e. its latent
//    chunks: O^T = V^T P^T with M = 128 V dims, N = 128 query rows, K = 64
//    KV rows -- two 128 x 128 fp32 TMEM blocks.
// Warp roles (448 threads): warp 0 TMA producer (3-stage KV ring), warp 1
// MMA issuer and TMEM owner, warps 2-9 scores (two threads per row; the
// warps on the peer's rows send, the warps on this CTA's rows run the
// softmax), warps 10-13 O correction and epilogue (thread = V dim = TMEM
// lane).  With an e4m3 cache two more warps (14-15) widen each staged e4m3
// tile to bf16 in shared memory (exact; the k_scale lives in bmm1/bmm2), and
// the bf16 ring is 2 deep.  A warp reaches TMEM lanes 32 (w mod 4) .. + 31, so each group of
// four consecutive warps covers all 128 lanes.
// The running max is only raised, and O^T rescaled, when it grows by more
// than 2^8.  Every wait is bounded; a timeout sets an error bit in the
// workspace status word and the kernel unwinds.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "mla_common.cuh"
#include "sm100_ptx.cuh"

namespace mla {

namespace {

using namespace ptx;

constexpr int kRows = 128;        // query rows per work item
constexpr int kHalfRows = 64;     // rows whose softmax each CTA owns
constexpr int kTile = kKvTile;    // 64 KV rows per tile
constexpr int kLatChunks = 4;     // 64-dim latent chunks per CTA (= its V dims)
// bf16 KV: a 3-deep ring of bf16 tiles.  e4m3 KV: a 2-deep ring of bf16
// tiles fed by a 2-deep ring of e4m3 staging tiles (converted in smem).
template <bool kFp8> struct Cfg {
  static constexpr int kStages = kFp8 ? 2 : 3;
  static constexpr int kThreads = kFp8 ? 512 : 448;  // + 2 converter warps
};
constexpr int kConvThreads = 64;
constexpr uint32_t kWaitLimit = 1u << 26;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// shared-memory layout (bytes from a 1024-aligned base)
constexpr uint32_t kChunkQ = kRows * 128;   // 64-dim chunk of Q, 128B-swizzled rows
constexpr uint32_t kRopeQ = kRows * 64;     // 32-dim RoPE half of Q, 64B-swizzled rows
constexpr uint32_t kChunkKV = kTile * 128;  // 64-dim chunk of a KV tile
constexpr uint32_t kRopeKV = kTile * 64;    // 32-dim RoPE half of a KV tile
constexpr uint32_t kStageBytes = kLatChunks * kChunkKV + kRopeKV;  // 36 KB
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_QROPE = OFF_Q + kLatChunks * kChunkQ;
constexpr uint32_t OFF_KV = OFF_QROPE + kRopeQ;
constexpr uint32_t kStgBytes = kLatChunks * kTile * 64 + kTile * 32;  // e4m3 tile, 18 KB
constexpr uint32_t OFF_STG = OFF_KV + 2 * kStageBytes;                // e4m3 staging (fp8 only)
constexpr uint32_t OFF_P = OFF_KV + 3 * kStageBytes;
static_assert(OFF_STG + 2 * kStgBytes == OFF_P, "e4m3 staging fills the third bf16 stage");
constexpr uint32_t OFF_X = OFF_P + kRows * 128;        // peer's partial scores of my rows
constexpr uint32_t OFF_BARS = OFF_X + kHalfRows * kTile * 4;
constexpr uint32_t kSliceBytes = 144;                  // per warp: fac[16], l[16], flag[4]
constexpr uint32_t kPartBytes = 4 * kSliceBytes;       // per rank: four warp slices
constexpr uint32_t OFF_FAC = OFF_BARS + 512;           // [2 tile parities][2 ranks] parts
constexpr uint32_t OFF_TMEM = OFF_FAC + 4 * kPartBytes;
constexpr uint32_t OFF_ABORT = OFF_TMEM + 16;
constexpr uint32_t kSmemUsed = OFF_ABORT + 16;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;     // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(OFF_KV % 1024 == 0 && kStageBytes % 1024 == 0 && OFF_P % 1024 == 0, "alignment");

// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_O = 0;    // two 128-column O^T blocks
constexpr uint32_t TM_S = 256;  // two 64-column S buffers

enum Bar {
  Q_FULL, Q_FREE, KV_FULL0, KV_FULL1, KV_FULL2, KV_EMPTY0, KV_EMPTY1, KV_EMPTY2,
  S_FULL0, S_FULL1, S_FREE0, S_FREE1, P_FULL, P_FREE, O_STABLE, CORR_DONE, CE_FREE, O_FINAL,
  EPI_DONE, X_FULL, PEER_X_FREE, PEER_P_FREE, STG_FULL0, STG_FULL1, STG_EMPTY0, STG_EMPTY1,
  NUM_BARS
};

// True if any of the eight 16-row groups (2 CTAs x 4 warps) asked for an O^T
// rescale at global tile g.
__device__ __forceinline__ bool rescale_requested(unsigned char* sm, uint32_t g);

struct Ctx {
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

// Pointer into the per-tile factor block: parity b, rank part k.
__device__ __forceinline__ unsigned char* fac_part(unsigned char* sm, int b, int k) {
  return sm + OFF_FAC + (2 * b + k) * kPartBytes;
}

__device__ __forceinline__ bool rescale_requested(unsigned char* sm, uint32_t g) {
  bool r = false;
#pragma unroll
  for (int k = 0; k < 8; ++k)
    r |= reinterpret_cast<volatile int*>(fac_part(sm, g & 1, k >> 2) + (k & 3) * kSliceBytes +
                                         128)[0] == (int)g;
  return r;
}

// Factor-block entry of query row q (0..127) for tile parity b: fac at +0,
// running sum l at +64 bytes.
__device__ __forceinline__ float* fac_of_row(unsigned char* sm, int b, int q) {
  return reinterpret_cast<float*>(fac_part(sm, b, q >> 6) + ((q >> 4) & 3) * kSliceBytes) +
         (q & 15);
}

}  // namespace

template <bool kFp8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg<kFp8>::kThreads, 1)
decode_sm103_kernel(const Problem p, const Layout lay, char* __restrict__ ws,
                    const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_q_rope,
                    const __grid_constant__ CUtensorMap tm_kv,
                    const __grid_constant__ CUtensorMap tm_kv_rope) {
  constexpr int kStages = Cfg<kFp8>::kStages;
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
  c.bars = reinterpret_cast<uint64_t*>(sm + OFF_BARS);
  c.abort = reinterpret_cast<volatile int*>(sm + OFF_ABORT);
  c.status = &hdr[kHdrStatus];
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_TMEM);

  if (tid == 0) {
    uint32_t counts[NUM_BARS];
    for (int i = 0; i < NUM_BARS; ++i) counts[i] = 1;
    counts[S_FREE0] = counts[S_FREE1] = 256;
    counts[P_FULL] = counts[PEER_X_FREE] = 2 * kHalfRows;
    counts[CORR_DONE] = counts[CE_FREE] = counts[EPI_DONE] = 128;
    if (kFp8) {
      for (int i = 0; i < kStages; ++i) counts[KV_FULL0 + i] = kConvThreads;
      counts[STG_EMPTY0] = counts[STG_EMPTY1] = kConvThreads;
    }
    for (int i = 0; i < NUM_BARS; ++i) mbar_init(&c.bars[i], counts[i]);
    *c.abort = 0;
    for (int b = 0; b < 2; ++b)
      for (int k = 0; k < 2; ++k)
        for (int w = 0; w < 4; ++w)
          reinterpret_cast<int*>(fac_part(sm, b, k) + w * kSliceBytes + 128)[0] = -1;
    fence_mbar_init();
    // the first tile's peer scores may arrive as soon as the cluster is up
    mbar_arrive_expect_tx(&c.bars[X_FULL], kHalfRows * kTile * 4);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before any remote access
  const uint32_t tmem = *tmem_slot;
  const int item_begin = worker_begin[worker], item_end = worker_begin[worker + 1];
  const int H = p.num_heads;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_q_rope);
      tma_prefetch_desc(&tm_kv);
      tma_prefetch_desc(&tm_kv_rope);
      uint32_t g = 0;
      int n_item = 0;
      const int ps = p.page_size;
      const int npg = kTile / ps;
      for (int idx = item_begin; idx < item_end; ++idx) {
        const WorkItem it = items[idx];
        const int nt = n_tiles_of(it);
        if (nt <= 0) continue;
        const int* bt = p.block_tables + (size_t)it.b * p.max_pages;
        // page ids of the first tile (later tiles are read one tile ahead)
        int pages[2] = {-1, -1};
        for (int pg = 0; pg < npg; ++pg) {
          const int jr = it.kv_begin + pg * ps;
          if (jr < it.kv_end) pages[pg] = bt[jr / ps];
        }
        if (!wait_bar(c, Q_FREE, (n_item & 1) ^ 1)) goto done_producer;
        ++n_item;
        {
          mbar_arrive_expect_tx(&c.bars[Q_FULL], kLatChunks * kChunkQ + kRopeQ);
          const int qrow = it.q_start * H + it.g * kRows;
          for (int lc = 0; lc < kLatChunks; ++lc)
            tma_load_2d(sm + OFF_Q + lc * kChunkQ, &tm_q, 256 * (int)rank + 64 * lc, qrow,
                        &c.bars[Q_FULL]);
          tma_load_2d(sm + OFF_QROPE, &tm_q_rope, 512 + 32 * (int)rank, qrow, &c.bars[Q_FULL]);
        }
        for (int t = 0; t < nt; ++t, ++g) {
          // bf16: load straight into the bf16 ring; e4m3: into the staging ring
          const int s = kFp8 ? (int)(g & 1) : (int)(g % kStages);
          const uint32_t use = kFp8 ? (g >> 1) : g / kStages;
          // read the next tile's page ids while this tile's slot drains
          int next[2] = {-1, -1};
          if (t + 1 < nt)
            for (int pg = 0; pg < npg; ++pg) {
              const int jr = it.kv_begin + (t + 1) * kTile + pg * ps;
              if (jr < it.kv_end) next[pg] = bt[jr / ps];
            }
          if (!wait_bar(c, kFp8 ? STG_EMPTY0 + s : KV_EMPTY0 + s, (use & 1) ^ 1)) goto done_producer;
          const int j0 = it.kv_begin + t * kTile;
          uint32_t bytes = 0;
          for (int pg = 0; pg < npg; ++pg) {
            if (j0 + pg * ps >= it.kv_end) {
              pages[pg] = -1;
              continue;
            }
            if (pages[pg] < 0 || (long long)pages[pg] >= p.num_pages) {
              atomicOr(c.status, 16);
              pages[pg] = -1;
              continue;
            }
            bytes += ps * (kLatChunks * 64 + 32) * (kFp8 ? 1 : 2);
          }
          uint64_t* full = &c.bars[kFp8 ? STG_FULL0 + s : KV_FULL0 + s];
          mbar_arrive_expect_tx(full, bytes);
          for (int pg = 0; pg < npg; ++pg) {
            if (pages[pg] < 0) continue;
            const int y = pages[pg] * ps;
            if (kFp8) {
              unsigned char* stg = sm + OFF_STG + s * kStgBytes;
              for (int lc = 0; lc < kLatChunks; ++lc)
                tma_load_2d(stg + lc * kTile * 64 + pg * ps * 64, &tm_kv, 256 * (int)rank + 64 * lc,
                            y, full);
              tma_load_2d(stg + kLatChunks * kTile * 64 + pg * ps * 32, &tm_kv_rope,
                          512 + 32 * (int)rank, y, full);
            } else {
              unsigned char* stage = sm + OFF_KV + s * kStageBytes;
              for (int lc = 0; lc < kLatChunks; ++lc)
                tma_load_2d(stage + lc * kChunkKV + pg * ps * 128, &tm_kv,
                            256 * (int)rank + 64 * lc, y, full);
              tma_load_2d(stage + kLatChunks * kChunkKV + pg * ps * 64, &tm_kv_rope,
                          512 + 32 * (int)rank, y, full);
            }
          }
          pages[0] = next[0];
          pages[1] = next[1];
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
      const uint32_t qr_base = smem_u32(sm + OFF_QROPE);
      const uint32_t kv_base = smem_u32(sm + OFF_KV);
      const uint32_t p_base = smem_u32(sm + OFF_P);
      uint32_t g = 0, n_rescale = 0;
      int n_item = 0;
      bool ok = true;
      auto issue_qk = [&](uint32_t gq) -> bool {
        const int s = gq % kStages;
        const int sb = gq & 1;
        if (!wait_bar(c, KV_FULL0 + s, (gq / kStages) & 1)) return false;
        if (!wait_bar(c, S_FREE0 + sb, ((gq >> 1) & 1) ^ 1)) return false;
        tc_fence_after();
        const uint32_t d = tmem + TM_S + 64 * sb;
        const uint32_t stage = kv_base + s * kStageBytes;
        for (int k = 0; k < 4 * kLatChunks; ++k) {
          const int lc = k >> 2, ks = k & 3;
          const uint64_t a = smem_desc(q_base + lc * kChunkQ + ks * 32, 16, 1024, kSwizzle128B);
          const uint64_t b = smem_desc(stage + lc * kChunkKV + ks * 32, 16, 1024, kSwizzle128B);
          mma_bf16_ss(d, a, b, idesc_qk, k > 0 ? 1u : 0u);
        }
        for (int ks = 0; ks < 2; ++ks) {
          const uint64_t a = smem_desc(qr_base + ks * 32, 16, 512, kSwizzle64B);
          const uint64_t b = smem_desc(stage + kLatChunks * kChunkKV + ks * 32, 16, 512,
                                       kSwizzle64B);
          mma_bf16_ss(d, a, b, idesc_qk, 1u);
        }
        mma_commit(&c.bars[S_FULL0 + sb]);
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
          if (!wait_bar(c, P_FULL, g & 1)) { ok = false; break; }
          if (t > 0 && rescale_requested(sm, g)) {
            // let the correction warps rescale O^T once the previous PV is done
            mma_commit(&c.bars[O_STABLE]);
            if (!wait_bar(c, CORR_DONE, n_rescale & 1)) { ok = false; break; }
            ++n_rescale;
          }
          if (t == 0 && n_item > 1) {
            // O^T of the previous item must have been read out before it is overwritten
            if (!wait_bar(c, EPI_DONE, (n_item - 2) & 1)) { ok = false; break; }
          }
          tc_fence_after();
          const int s = g % kStages;
          const uint32_t stage = kv_base + s * kStageBytes;
          for (int bb = 0; bb < 2; ++bb) {
            for (int ks = 0; ks < kTile / 16; ++ks) {
              const uint64_t a = smem_desc(stage + (2 * bb) * kChunkKV + ks * 16 * 128, 8192, 1024,
                                           kSwizzle128B);
              const uint64_t b = smem_desc(p_base + ks * 32, 16, 1024, kSwizzle128B);
              mma_bf16_ss(tmem + TM_O + 128 * bb, a, b, idesc_pv, (t == 0 && ks == 0) ? 0u : 1u);
            }
          }
          mma_commit(&c.bars[KV_EMPTY0 + s]);
          mma_commit(&c.bars[P_FREE]);
          if (t + 1 == nt) mma_commit(&c.bars[O_FINAL]);
        }
      }
    }
  } else if (warp >= 2 && warp < 10) {
    // ------------------------------------------------------------ scores
    // Warp w reads TMEM lanes 32 (w mod 4) + 16 grp + 0..15 (grp = 0 for
    // warps 2-5, 1 for warps 6-9) with two threads per row: thread t handles
    // row (t mod 16) of its 16 and columns [32 h, 32 h + 32), h = t / 16.
    const int sp = warp & 3, grp = (warp - 2) >> 2;
    const int half = lane >> 4;
    const int q = 32 * sp + 16 * grp + (lane & 15);  // query row == TMEM lane
    const bool mine = (q >> 6) == (int)rank;
    const uint32_t lane_addr = (uint32_t)(32 * sp + 16 * grp) << 16;
    uint32_t g = 0;
    if (!mine) {
      // sender: my half of the partial scores of a peer row -> peer's X buffer
      const int pr = q & 63;  // row index inside the peer's buffer
      const uint32_t x_peer = map_to_rank(smem_u32(sm + OFF_X + pr * 256), peer);
      const uint32_t xfull_peer = map_to_rank(smem_u32(&c.bars[X_FULL]), peer);
      for (int idx = item_begin; idx < item_end; ++idx) {
        const WorkItem it = items[idx];
        const int nt = n_tiles_of(it);
        if (nt <= 0) continue;
        for (int t = 0; t < nt; ++t, ++g) {
          const int sb = g & 1;
          if (!wait_bar(c, S_FULL0 + sb, (g >> 1) & 1)) goto done_scores;
          tc_fence_after();
          uint32_t v[32];
          tmem_ld_16x32bx2_x32(tmem + lane_addr + TM_S + 64 * sb, v);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(&c.bars[S_FREE0 + sb]);
          if (!wait_bar_cluster(c, PEER_X_FREE, (g & 1) ^ 1)) goto done_scores;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int chunk = 8 * half + k;
            st_async_v4(x_peer + (uint32_t)((chunk ^ (pr & 7)) << 4),
                        make_float4(__uint_as_float(v[4 * k]), __uint_as_float(v[4 * k + 1]),
                                    __uint_as_float(v[4 * k + 2]), __uint_as_float(v[4 * k + 3])),
                        xfull_peer);
          }
        }
      }
    } else {
      // softmax of my 64 rows: 4 warps x 16 rows x 2 threads per row.  Each
      // tile ends with its hand-off: bf16 P rows and rescale factors are
      // written locally and copied to the peer, then P_FULL is signalled.
      const int mr = q & 63;                  // my row index (0..63)
      const int wslice = mr >> 4;             // this warp's 16-row slice (0..3)
      const bool leader = mr == 0 && half == 0;
      const float scale = p.bmm1_scale * kLog2e;
      const uint32_t pfree_peer = map_to_rank(smem_u32(&c.bars[PEER_P_FREE]), peer);
      const uint32_t xfree_peer = map_to_rank(smem_u32(&c.bars[PEER_X_FREE]), peer);
      const uint32_t pfull_peer = map_to_rank(smem_u32(&c.bars[P_FULL]), peer);
      const uint32_t p_rows_off = OFF_P + (uint32_t)(32 * sp + 16 * grp) * 128;
      const uint32_t p_peer = map_to_rank(smem_u32(sm + p_rows_off), peer);
      const float4* xs = reinterpret_cast<const float4*>(sm + OFF_X + mr * 256);
      // state of the tile whose hand-off is pending
      float pv[32];
      float pf = 1.f, pl = 0.f, plse = 0.f;
      bool pneed = false, pending = false, plse_valid = false, copy_pending = false;
      int pslot = 0;
      size_t plse_idx = 0;
      uint32_t pg = 0;
      // hand-off of tile `pg`: P rows, factor slice, copies to the peer, P_FULL
      auto handoff = [&]() -> bool {
        if (!wait_bar(c, P_FREE, (pg & 1) ^ 1)) return false;
        if (!wait_bar(c, CE_FREE, (pg & 1) ^ 1)) return false;
        if (copy_pending) {  // the previous copy has finished reading my P rows
          if (lane == 0) bulk_wait_read0();
          __syncwarp();
          copy_pending = false;
        }
        if (leader) {
          // expect the peer's P rows and factor slices, then let the peer send them
          mbar_expect_tx(&c.bars[P_FULL], kHalfRows * 128 + kPartBytes);
          mbar_arrive_cluster_relaxed(pfree_peer);
        }
        unsigned char* prow = sm + OFF_P + q * 128;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint4 w;
          w.x = pack_bf16(pv[8 * k + 0], pv[8 * k + 1]);
          w.y = pack_bf16(pv[8 * k + 2], pv[8 * k + 3]);
          w.z = pack_bf16(pv[8 * k + 4], pv[8 * k + 5]);
          w.w = pack_bf16(pv[8 * k + 6], pv[8 * k + 7]);
          *reinterpret_cast<uint4*>(prow + (((4 * half + k) ^ (q & 7)) << 4)) = w;
        }
        unsigned char* slice = fac_part(sm, pg & 1, rank) + wslice * kSliceBytes;
        if (half == 0) {
          reinterpret_cast<float*>(slice)[lane] = pf;
          reinterpret_cast<float*>(slice + 64)[lane] = pl;
        }
        const bool any = __any_sync(0xffffffffu, pneed);
        if (lane == 0 && any) reinterpret_cast<volatile int*>(slice + 128)[0] = (int)pg;
        fence_proxy_async_smem();
        __syncwarp();
        bool ok = true;
        if (lane == 0) {
          ok = wait_bar_cluster(c, PEER_P_FREE, pg & 1);
          if (ok) {
            bulk_copy_to_peer(p_peer, sm + p_rows_off, 16 * 128, pfull_peer);
            bulk_copy_to_peer(map_to_rank(smem_u32(slice), peer), slice, kSliceBytes, pfull_peer);
            bulk_commit();
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) return false;
        copy_pending = true;
        mbar_arrive(&c.bars[P_FULL]);
        if (plse_valid) {
          if (pslot < 0) {
            if (p.return_lse) p.lse[plse_idx] = plse;
          } else {
            part_lse[plse_idx] = plse;
          }
        }
        pending = false;
        return true;
      };
      for (int idx = item_begin; idx < item_end; ++idx) {
        const WorkItem it = items[idx];
        const int nt = n_tiles_of(it);
        if (nt <= 0) continue;
        const int rows_total = it.q_len * H;
        const int row0 = it.g * kRows;
        const bool row_ok = q < rows_total - row0;
        const int qi = (row0 + q) / H;
        const int last = p.causal ? it.seq_len - it.q_len + qi : it.seq_len - 1;
        // tiles ending at or before `clean_end` need no mask for any valid row
        const int first_qi = row0 / H;
        const int clean_end =
            min(it.kv_end, p.causal ? it.seq_len - it.q_len + first_qi + 1 : it.seq_len);
        float m_ref = -INFINITY, l_half = 0.f;  // l_half: this thread's columns only
        for (int t = 0; t < nt; ++t, ++g) {
          const int sb = g & 1;
          float sv[32];
          if (!wait_bar(c, S_FULL0 + sb, (g >> 1) & 1)) goto done_scores;
          tc_fence_after();
          {
            uint32_t v[32];
            tmem_ld_16x32bx2_x32(tmem + lane_addr + TM_S + 64 * sb, v);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) sv[j] = __uint_as_float(v[j]);
          }
          tc_fence_before();
          mbar_arrive(&c.bars[S_FREE0 + sb]);
          // add the peer's partial for my half row, then release it to the peer
          if (!wait_bar(c, X_FULL, g & 1)) goto done_scores;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float4 x = xs[(8 * half + k) ^ (mr & 7)];
            sv[4 * k] += x.x;
            sv[4 * k + 1] += x.y;
            sv[4 * k + 2] += x.z;
            sv[4 * k + 3] += x.w;
          }
          if (leader) mbar_arrive_expect_tx(&c.bars[X_FULL], kHalfRows * kTile * 4);  // next tile
          mbar_arrive_cluster_relaxed(xfree_peer);
          // mask, online softmax (scale folded into the exponent)
          const int j0 = it.kv_begin + t * kTile;
          const int c0 = j0 + 32 * half;  // KV index of sv[0]
          float f = 1.f;
          bool need = false;
          float tmax = -INFINITY;
          if (row_ok) {
            if (j0 + kTile <= clean_end) {
#pragma unroll
              for (int j = 0; j < 32; ++j) tmax = fmaxf(tmax, sv[j]);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const int col = c0 + j;
                sv[j] = (col <= last && col < it.kv_end) ? sv[j] : -INFINITY;
                tmax = fmaxf(tmax, sv[j]);
              }
            }
          }
          // both threads of a row live in the same warp (lanes t and t + 16)
          tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
          if (row_ok) {
            const float m_new = fmaxf(m_ref, tmax * scale);
            if (t == 0) {
              m_ref = m_new;
            } else if (m_new > m_ref + kRescaleThreshold) {
              f = ex2(m_ref - m_new);  // m_ref = -inf gives 0
              need = true;
              l_half *= f;
              m_ref = m_new;
            }
            const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
            float rs = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              sv[j] = ex2(fmaf(sv[j], scale, -m_use));
              rs += sv[j];
            }
            l_half += rs;
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) sv[j] = 0.f;
          }
          const float l_row = l_half + __shfl_xor_sync(0xffffffffu, l_half, 16);
          // zero V rows past the end of the KV range (last tile of the item)
          const int valid = it.kv_end - j0;
          if (valid < kTile) {
            unsigned char* stage = sm + OFF_KV + (g % kStages) * kStageBytes;
            const int nz = (kTile - valid) * kLatChunks * 8;  // 16-byte units
            for (int e = 2 * mr + half; e < nz; e += 2 * kHalfRows) {
              const int row = valid + e / 32, ch = (e / 8) % 4, u = e % 8;
              *reinterpret_cast<uint4*>(stage + ch * kChunkKV + row * 128 + u * 16) =
                  make_uint4(0, 0, 0, 0);
            }
          }
          // hand-off of this tile
#pragma unroll
          for (int j = 0; j < 32; ++j) pv[j] = sv[j];
          pf = f;
          pl = l_row;
          pneed = need;
          pg = g;
          pending = true;
          plse_valid = (t + 1 == nt) && row_ok && half == 0;
          if (plse_valid) {
            plse = l_row > 0.f ? (m_ref + log2f(l_row)) * kLn2 : -INFINITY;
            pslot = it.slot;
            const size_t grow = (size_t)it.q_start * H + row0 + q;
            plse_idx = it.slot < 0 ? grow : (size_t)it.slot * kRows + q;
          }
          if (!handoff()) goto done_scores;
        }
      }
      if (copy_pending && lane == 0) bulk_wait_read0();
    }
  done_scores:;
  } else if (warp >= 10 && warp < 14) {
    // ------------------------------------------------------------ correction + epilogue
    const int v = 32 * (warp & 3) + lane;  // V dim within each 128-wide O^T block == TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    uint32_t g = 0, n_rescale = 0;
    int n_item = 0;
    for (int idx = item_begin; idx < item_end; ++idx) {
      const WorkItem it = items[idx];
      const int nt = n_tiles_of(it);
      if (nt <= 0) continue;
      for (int t = 0; t < nt; ++t, ++g) {
        if (!wait_bar(c, P_FULL, g & 1)) goto done_epi;
        if (t > 0 && rescale_requested(sm, g)) {
          if (!wait_bar(c, O_STABLE, n_rescale & 1)) goto done_epi;
          ++n_rescale;
          tc_fence_after();
          for (int bb = 0; bb < 2; ++bb) {
#pragma unroll 1
            for (int q16 = 0; q16 < kRows / 16; ++q16) {
              const float* f = fac_of_row(sm, g & 1, 16 * q16);
              uint32_t x[16];
              const uint32_t addr = tmem + lane_base + TM_O + 128 * bb + 16 * q16;
              tmem_ld_32x32b_x16(addr, x);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j) x[j] = __float_as_uint(__uint_as_float(x[j]) * f[j]);
              tmem_st_32x32b_x16(addr, x);
            }
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&c.bars[CORR_DONE]);
        }
        mbar_arrive(&c.bars[CE_FREE]);
      }
      // epilogue: O = O^T(transposed) / l, from the last tile's factor block
      if (!wait_bar(c, O_FINAL, n_item & 1)) goto done_epi;
      tc_fence_after();
      {
        const int rows_total = it.q_len * H;
        const int row0 = it.g * kRows;
        const int n_rows = min(kRows, rows_total - row0);
        const size_t grow0 = (size_t)it.q_start * H + row0;
        const int lb = (g - 1) & 1;
        for (int bb = 0; bb < 2; ++bb) {
          const int vd = 256 * (int)rank + 128 * bb + v;  // output V dim
#pragma unroll 1
          for (int q16 = 0; q16 < kRows / 16; ++q16) {
            if (16 * q16 >= n_rows) break;
            const float* lrow = fac_of_row(sm, lb, 16 * q16) + 16;
            uint32_t x[16];
            tmem_ld_32x32b_x16(tmem + lane_base + TM_O + 128 * bb + 16 * q16, x);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int qq = 16 * q16 + j;
              if (qq >= n_rows) break;
              const float l = lrow[j];
              const float inv = l > 0.f ? 1.f / l : 0.f;
              const float o = __uint_as_float(x[j]) * inv;
              if (it.slot < 0) {
                reinterpret_cast<__nv_bfloat16*>(p.out)[(grow0 + qq) * kVDim + vd] =
                    __float2bfloat16_rn(o * p.bmm2_scale);
              } else {
                part_o[((size_t)it.slot * kRows + qq) * kVDim + vd] = o;
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&c.bars[EPI_DONE]);
      ++n_item;
    }
  done_epi:;
  } else if (kFp8 && warp >= 14) {
    // ------------------------------------------------------------ e4m3 -> bf16
    // Thread r converts KV row r of each tile from the staging ring (row-major
    // bytes) into the bf16 ring in the swizzled layouts the MMAs read.
    const int r = tid - 14 * 32;
    uint32_t g = 0;
    for (int idx = item_begin; idx < item_end; ++idx) {
      const WorkItem it = items[idx];
      const int nt = n_tiles_of(it);
      if (nt <= 0) continue;
      for (int t = 0; t < nt; ++t, ++g) {
        const int s = g & 1;  // staging slot == bf16 slot (both 2 deep)
        if (!wait_bar(c, STG_FULL0 + s, (g >> 1) & 1)) goto done_conv;
        if (!wait_bar(c, KV_EMPTY0 + s, ((g >> 1) & 1) ^ 1)) goto done_conv;
        const unsigned char* src = sm + OFF_STG + s * kStgBytes;
        unsigned char* dst = sm + OFF_KV + s * kStageBytes;
#pragma unroll
        for (int lc = 0; lc < kLatChunks; ++lc) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // 16 e4m3 values -> 2 x 16-byte bf16 units
            const uint4 b = *reinterpret_cast<const uint4*>(src + lc * kTile * 64 + r * 64 + 16 * k);
            const uint32_t w[4] = {b.x, b.y, b.z, b.w};
            uint32_t o[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              o[2 * e] = e4m3x2_to_bf16x2(w[e] & 0xFFFFu);
              o[2 * e + 1] = e4m3x2_to_bf16x2(w[e] >> 16);
            }
            const int u0 = 2 * k, u1 = 2 * k + 1;  // 16-byte units of the 128-byte row
            *reinterpret_cast<uint4*>(dst + lc * kChunkKV + r * 128 + ((u0 ^ (r & 7)) << 4)) =
                make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(dst + lc * kChunkKV + r * 128 + ((u1 ^ (r & 7)) << 4)) =
                make_uint4(o[4], o[5], o[6], o[7]);
          }
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {  // RoPE half: 32 values -> four 16-byte units (64B swizzle)
          const uint4 b = *reinterpret_cast<const uint4*>(src + kLatChunks * kTile * 64 + r * 32 + 16 * k);
          const uint32_t w[4] = {b.x, b.y, b.z, b.w};
          uint32_t o[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            o[2 * e] = e4m3x2_to_bf16x2(w[e] & 0xFFFFu);
            o[2 * e + 1] = e4m3x2_to_bf16x2(w[e] >> 16);
          }
          const int sw = (r >> 1) & 3;
          const int u0 = 2 * k, u1 = 2 * k + 1;
          *reinterpret_cast<uint4*>(dst + kLatChunks * kChunkKV + r * 64 + ((u0 ^ sw) << 4)) =
              make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(dst + kLatChunks * kChunkKV + r * 64 + ((u1 ^ sw) << 4)) =
              make_uint4(o[4], o[5], o[6], o[7]);
        }
        fence_proxy_async_smem();
        mbar_arrive(&c.bars[KV_FULL0 + s]);
        mbar_arrive(&c.bars[STG_EMPTY0 + s]);
      }
    }
  done_conv:;
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

bool encode_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes,
               uint64_t rows, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kQkDim, rows};
  cuuint64_t strides[1] = {(cuuint64_t)kQkDim * elem_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kFp8>
cudaError_t setup_one(int sm_count, int* n_pairs) {
  auto kernel = decode_sm103_kernel<kFp8>;
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sm_count / 2), 1, 1);
  cfg.blockDim = dim3(Cfg<kFp8>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
  if (e != cudaSuccess) return e;
  if (clusters <= 0) return cudaErrorInvalidConfiguration;
  *n_pairs = std::min(clusters, sm_count / 2);
  return cudaSuccess;
}

}  // namespace

cudaError_t decode_sm103_setup(int kv_dtype, int sm_count, int* n_pairs) {
  return kv_dtype == 1 ? setup_one<true>(sm_count, n_pairs) : setup_one<false>(sm_count, n_pairs);
}

cudaError_t launch_decode_sm103(const Problem& p, const Layout& lay, void* ws,
                                cudaStream_t stream) {
  CUtensorMap tm_q, tm_q_rope, tm_kv, tm_kv_rope;
  const uint64_t q_rows = std::max<uint64_t>(1, (uint64_t)p.total_q * p.num_heads);
  const uint64_t kv_rows = (uint64_t)p.num_pages * p.page_size;
  if (!encode_2d(&tm_q, p.query, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, q_rows, 64, kRows,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tm_q_rope, p.query, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, q_rows, 32, kRows,
                 CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  const bool fp8 = p.kv_dtype == 1;
  if (fp8) {
    // e4m3 bytes land row-major in the staging ring; the converter swizzles
    if (!encode_2d(&tm_kv, p.kv_cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kv_rows, 64,
                   p.page_size, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&tm_kv_rope, p.kv_cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kv_rows, 32,
                   p.page_size, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
    decode_sm103_kernel<true><<<lay.n_ctas, Cfg<true>::kThreads, kSmemBytes, stream>>>(
        p, lay, static_cast<char*>(ws), tm_q, tm_q_rope, tm_kv, tm_kv_rope);
  } else {
    if (!encode_2d(&tm_kv, p.kv_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kv_rows, 64,
                   p.page_size, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tm_kv_rope, p.kv_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kv_rows, 32,
                   p.page_size, CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
    decode_sm103_kernel<false><<<lay.n_ctas, Cfg<false>::kThreads, kSmemBytes, stream>>>(
        p, lay, static_cast<char*>(ws), tm_q, tm_q_rope, tm_kv, tm_kv_rope);
  }
  return cudaGetLastError();
}

}  // namespace mla
