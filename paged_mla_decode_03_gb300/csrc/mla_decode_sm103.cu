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
// 128 x 576 bf16 query tile needs 144 KB, so one work item is shared by the
// two CTAs of a cluster, split along the head dims:
//  * CTA r holds latent dims [256 r, 256 r + 256) and RoPE dims
//    [512 + 32 r, 512 + 32 r + 32) of Q and of every KV tile.  Its Q latent
//    dims live in TMEM (A operand of 16 ts MMAs), its Q RoPE dims in shared
//    memory (2 ss MMAs); QK yields a partial S_r (M = 128 query rows,
//    N = 64 KV rows, fp32 in TMEM);
//  * each query row (TMEM lane l) has an owner CTA, (l / 16) mod 2.  The
//    owner runs that row's softmax: the other CTA pushes its partial scores of
//    the row (fp32, exactly as the MMA produced them) into the owner's shared
//    memory with st.async, the owner adds them to its own and forms P (bf16),
//    which it writes into the P tile of both CTAs (its own with st.shared, the
//    peer's with st.async), together with the row's rescale factor;
//  * O = P V with P from shared memory: M = 128 query rows, N = 256 (CTA r's
//    V dims, read MN-major from its latent chunks), K = 64 KV rows, into a
//    128 x 256 fp32 TMEM accumulator.  The PV commit is multicast to both CTAs,
//    so each of the two P tiles (one per tile parity) is rewritten only after
//    both CTAs' PV read it.
// Warp roles (448 threads, 704 with e4m3): warp 0 TMA producer (4-stage KV
// ring), warp 1 MMA issuer and TMEM owner (QK runs up to two tiles ahead of
// PV), warps 2-9 softmax of the 64 owned rows in two groups of four that take
// alternate KV tiles (group G the tiles of global parity G), so that two
// tiles' softmax latencies overlap; in a group, warp w covers the 16 owned
// lanes 32 (w mod 4) + 16 r .. + 15 of its TMEM subpartition, two threads per
// row (32 KV columns each, the 16x32bx2 access shape), so a row's maximum
// needs one shuffle.  Only the running-max reference passes from tile to
// tile between the groups; each group keeps its own row-sum partial, and the
// group of an item's last tile merges the two.  Warps 10-13 are the
// partial-score senders (the peer-owned lanes), O correction, epilogue and
// the Q latent load into TMEM (thread = query row = TMEM lane).
// An e4m3 cache runs by default on FP8 MMAs (kind::f8f6f4, a separate
// instantiation): the e4m3 tiles go from the TMA straight into an 8-deep ring
// in the operand layouts, the query enters as e4m3 (a bf16 row as two parts
// under a power-of-two scale per CTA half, split before this kernel by
// mla_qsplit.cu; the scores are brought back by it before the halves are
// added), and so does P (two parts).  Widening on request: eight more warps
// (14-21) widen each staged e4m3 tile to bf16 in shared memory (exact; the
// k_scale lives in bmm1/bmm2), and the bf16 ring is 3 deep beside a 2-deep
// e4m3 staging ring.
// Under sparse top-k selection (a separate instantiation, two warps more) a
// work item is one token's H query rows and its KV tiles are 64 entries of
// the token's position list: warp 0 and the two extra warps gather the listed
// rows (gather_producer) instead of warp 0 issuing page copies.
// The running max is only raised, and O rescaled, when it grows by more than
// 2^8.  Every wait is bounded; a timeout sets an error bit in the workspace
// status word and the kernel unwinds.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>

#include "mla_common.cuh"
#include "sm100_ptx.cuh"

namespace mla {

namespace {

using namespace ptx;

constexpr int kRows = 128;        // query rows per work item
constexpr int kOwnRows = 64;      // rows whose softmax this CTA runs
constexpr int kTile = kKvTile;    // 64 KV rows per tile
constexpr int kLatChunks = 4;     // 64-dim latent chunks per CTA (= its V dims)
constexpr int kSoftmaxWarps = 8;  // two groups of four
constexpr int kGroupWarps = 4;
constexpr int kCeWarps = 4;       // senders / correction / epilogue
constexpr int kConvThreads = 256;  // four per KV row of a tile
constexpr uint32_t kWaitLimit = 1u << 26;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// shared-memory layout (bytes from a 1024-aligned base): fixed regions first,
// then the KV ring
constexpr uint32_t kRopeQ = kRows * 64;     // 32-dim RoPE half of Q, 64B-swizzled rows
constexpr uint32_t kChunkKV = kTile * 128;  // 64-dim chunk of a KV tile
constexpr uint32_t kRopeKV = kTile * 64;    // 32-dim RoPE half of a KV tile
constexpr uint32_t kStageBytes = kLatChunks * kChunkKV + kRopeKV;  // 36 KB
constexpr uint32_t kPBytes = kRows * 128;   // P: 128 rows x 64 KV rows bf16, 128B-swizzled
constexpr uint32_t kStgBytes = kLatChunks * kTile * 64 + kTile * 32;  // e4m3 tile, 18 KB
// e4m3 tiles read by FP8 MMAs: two 128-dim latent chunks (128B-swizzled rows)
// and the 32 RoPE dims (32B-swizzled rows)
constexpr uint32_t kChunk8 = kTile * 128;
constexpr uint32_t kRope8 = kTile * 32;
constexpr uint32_t kStage8Bytes = 2 * kChunk8 + kRope8;  // 18 KB
constexpr uint32_t kPart8 = kRows * 64;  // one e4m3 part of a P tile (64B-swizzled rows)
// peer's partial scores of the owned rows: [64 rows][64] fp32 per tile parity
// (16-byte units of a row XOR-swizzled by the row index)
constexpr uint32_t kXRowBytes = kTile * 4;
constexpr uint32_t kXBytes = kOwnRows * kXRowBytes;
constexpr uint32_t OFF_QROPE = 0;
constexpr uint32_t OFF_P = OFF_QROPE + kRopeQ;   // P tiles of tile parity 0 and 1
constexpr uint32_t OFF_X = OFF_P + 2 * kPBytes;  // peer scores of tile parity 0 and 1
constexpr uint32_t OFF_BARS = OFF_X + 2 * kXBytes;
constexpr uint32_t OFF_FAC = OFF_BARS + 512;        // float fac[2][128]: rescale factor per row
constexpr uint32_t OFF_LROW = OFF_FAC + 2 * kRows * 4;  // float l[128]: row sums, last tile
constexpr uint32_t OFF_FLAG = OFF_LROW + kRows * 4;     // int flag[2][16]: own + peer warps
constexpr uint32_t OFF_MREF = OFF_FLAG + 2 * 16 * 4;    // float [2][128]: running max by tile parity
constexpr uint32_t OFF_LX = OFF_MREF + 2 * kRows * 4;   // float [2][2][128]: group (l, m) per slot
constexpr uint32_t OFF_TMEM = OFF_LX + 4 * kRows * 4;
constexpr uint32_t OFF_ABORT = OFF_TMEM + 16;
// uint64 [8][3]: usable rows of a sparse tile, by g mod 8 and gather warp
constexpr uint32_t OFF_VMASK = OFF_ABORT + 16;
constexpr int kGatherWarps = 3;  // sparse top-k: warps that gather KV rows
// float [2][128]: per-row query scale 2^-k of the FP8 path, by item parity
constexpr uint32_t OFF_QSCALE = OFF_VMASK + 8 * kGatherWarps * 8;
// float [128]: an item's final running max of the owned rows (log2 units),
// beside lrow, for the epilogue's split-chunk LSE
constexpr uint32_t OFF_MROW = OFF_QSCALE + 2 * kRows * 4;
constexpr uint32_t OFF_KV = (OFF_MROW + kRows * 4 + 1023) / 1024 * 1024;

// bf16 cache: a 4-stage ring.  e4m3 cache widened to bf16 (kFp8): 3 bf16
// stages and a 2-deep e4m3 staging ring in the fourth stage's space.  e4m3
// cache on FP8 MMAs (kF8): an 8-stage ring of e4m3 tiles.  Sparse top-k: two
// more warps (the last two) gather rows beside warp 0.
template <bool kFp8, bool kSparse = false, bool kF8 = false> struct Cfg {
  static_assert(!(kF8 && (kFp8 || kSparse)), "FP8 MMAs: dense e4m3 cache only");
  static constexpr int kStages = kF8 ? 8 : (kFp8 ? 3 : 4);
  static constexpr uint32_t kStage = kF8 ? kStage8Bytes : kStageBytes;  // bytes of a stage
  static constexpr int kThreads =
      (kFp8 ? 704 : 448) + (kSparse ? 32 * (kGatherWarps - 1) : 0);  // + 8 converter warps
  static constexpr int kFirstExtraGatherWarp = kThreads / 32 - (kGatherWarps - 1);
  static constexpr uint32_t OFF_STG = OFF_KV + kStages * kStage;  // e4m3 staging
  static constexpr uint32_t kRingEnd = OFF_STG + (kFp8 ? 2 * kStgBytes : 0);
  static constexpr uint32_t kSmemBytes = kRingEnd + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(OFF_STG % 1024 == 0, "alignment");
};
static_assert(OFF_KV % 1024 == 0 && kStageBytes % 1024 == 0 && OFF_P % 1024 == 0 &&
                  kPBytes % 1024 == 0 && OFF_FLAG % 16 == 0 && OFF_X % 16 == 0 &&
                  2 * kStgBytes == kStageBytes && OFF_VMASK % 8 == 0 &&
                  kStage8Bytes % 1024 == 0 && 2 * kPart8 == kPBytes && OFF_QSCALE % 16 == 0,
              "alignment");
// bytes the peer pushes into this CTA's P tile per KV tile (P rows, factors,
// the group's four flags), plus the row sums on an item's last tile
constexpr uint32_t kPeerPBytes = kOwnRows * 128 + kOwnRows * 4 + kGroupWarps * 4;
constexpr uint32_t kPeerLBytes = kOwnRows * 4;

// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_O = 0;    // O: 128 rows x 256 V dims (fp32)
constexpr uint32_t TM_S = 256;  // two 64-column S buffers (fp32)
constexpr uint32_t TM_Q = 384;  // Q latent: 128 rows x 256 dims (bf16 pairs)

enum Bar {
  Q_FULL, Q_FREE, QT_FULL,
  KV_FULL0, KV_EMPTY0 = KV_FULL0 + 8,  // 8 each: one per ring stage
  S_FULL0 = KV_EMPTY0 + 8, S_FULL1,
  S_FREE0, S_FREE1,
  X_FULL0, X_FULL1, PEER_X_FREE0, PEER_X_FREE1,
  P_FULL0, P_FULL1, P_FREE0, P_FREE1,
  MREF0,                       // 8: [tile parity][subpartition], running max published
  LX0 = MREF0 + 8,             // 8: [slot][subpartition], a group's (l, m) published
  LROW_FREE = LX0 + 8,
  O_STABLE, CORR_DONE, O_FINAL, EPI_DONE,
  STG_FULL0, STG_FULL1, STG_EMPTY0, STG_EMPTY1,
  MMA_DRAIN,                   // the issuer's last commit: every MMA it issued has completed
  QS_FULL0, QS_FULL1,          // FP8 path: the item's query row scales written, by item parity
  NUM_BARS
};
static_assert(NUM_BARS * 8 <= 512, "barrier area");

struct Ctx {
  uint64_t* bars;
  volatile int* abort;
  uint32_t peer_abort;  // the peer CTA's abort word (shared::cluster address)
  int* status;
};

// A wait that ran out: flag the status word and make both CTAs of the pair
// unwind (each waits for its own copies and MMAs in flight before leaving).
__device__ __forceinline__ void give_up(const Ctx& c) {
  *c.abort = 1;
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(c.peer_abort), "r"(1) : "memory");
  atomicOr(c.status, kStatusTimeout);
}

__device__ __forceinline__ bool wait_bar(const Ctx& c, int bar, uint32_t parity) {
  uint64_t* b = &c.bars[bar];
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    if (mbar_try_wait(b, parity)) return true;
    if ((i & 1023) == 1023 && *c.abort) return false;
  }
  give_up(c);
  return false;
}

__device__ __forceinline__ bool wait_bar_cluster(const Ctx& c, int bar, uint32_t parity) {
  uint64_t* b = &c.bars[bar];
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    if (mbar_try_wait_acq_cluster(b, parity)) return true;
    if ((i & 1023) == 1023 && *c.abort) return false;
  }
  give_up(c);
  return false;
}

// Bounded wait that ignores the abort word: used on the way out, for the
// completion of this CTA's own asynchronous copies and MMAs.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return;
}

__device__ __forceinline__ int n_tiles_of(const WorkItem& it) {
  return (it.kv_end - it.kv_begin + kTile - 1) / kTile;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// True if any softmax warp of either CTA asked for an O rescale at global tile g.
__device__ __forceinline__ bool rescale_requested(const unsigned char* sm, uint32_t g) {
  const unsigned char* f = sm + OFF_FLAG + 64 * (g & 1);
  bool r = false;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint4 v = ld_volatile_shared_v4(f + 16 * k);
    r |= (v.x == g) | (v.y == g) | (v.z == g) | (v.w == g);
  }
  return r;
}

}  // namespace

// Row `q` of a work item's e4m3 query, for the CTA of cluster rank `rank`:
// its latent dims [256 rank, 256 rank + 256) widened exactly to bf16 pairs
// into the TMEM columns at `tmem_q` (lane already in the address), where they
// are the A operand of the ts QK MMAs, and its RoPE dims [512 + 32 rank, +32)
// widened into the 64B-swizzled smem tile at `q_rope` (a bf16 query's RoPE
// half comes by TMA).  Rows past the query tensor are zero.  Called once per
// item and kept out of line, away from the per-tile loop of the calling warps.
__device__ __noinline__ void load_q_row_e4m3(const Problem& p, long long qrow, bool in, int q,
                                             uint32_t rank, uint32_t tmem_q,
                                             unsigned char* q_rope) {
  const uint4* src = reinterpret_cast<const uint4*>(
      reinterpret_cast<const unsigned char*>(p.query) + (in ? qrow : 0) * kQkDim);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t w[64];
#pragma unroll
    for (int u = 0; u < 8; ++u) {  // 16 codes -> 8 bf16 pairs
      const uint4 x = in ? __ldg(src + 16 * (int)rank + 8 * half + u) : make_uint4(0, 0, 0, 0);
      const uint32_t c4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        w[8 * u + 2 * e] = e4m3x2_to_bf16x2(c4[e] & 0xFFFFu);
        w[8 * u + 2 * e + 1] = e4m3x2_to_bf16x2(c4[e] >> 16);
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      tmem_st_32x32b_x16(tmem_q + 64 * half + 16 * j,
                         *reinterpret_cast<const uint32_t(*)[16]>(w + 16 * j));
  }
  const int sw = (q >> 1) & 3;
#pragma unroll
  for (int k = 0; k < 2; ++k) {  // RoPE dims 512 + 32 r + [16 k, 16 k + 16)
    const uint4 x = in ? __ldg(src + 32 + 2 * (int)rank + k) : make_uint4(0, 0, 0, 0);
    const uint32_t c4[4] = {x.x, x.y, x.z, x.w};
    uint32_t o[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      o[2 * e] = e4m3x2_to_bf16x2(c4[e] & 0xFFFFu);
      o[2 * e + 1] = e4m3x2_to_bf16x2(c4[e] >> 16);
    }
    *reinterpret_cast<uint4*>(q_rope + q * 64 + (((2 * k) ^ sw) << 4)) =
        make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(q_rope + q * 64 + (((2 * k + 1) ^ sw) << 4)) =
        make_uint4(o[4], o[5], o[6], o[7]);
  }
  fence_proxy_async_smem();  // read by the RoPE MMAs
}

// Row `q` of a work item's query for the FP8 MMAs, for the CTA of cluster rank
// `rank`: its latent dims [256 rank, 256 rank + 256) as e4m3 codes into the
// TMEM columns at `tmem_q` (four codes a column, in dim order; A operand of the
// ts QK MMAs) and its RoPE dims [512 + 32 rank, +32) into the 32B-swizzled
// smem tile at `q_rope`.  An e4m3 query is copied as it is (one part).  A
// bf16 query comes split (mla_qsplit.cu; records at q_split_offset) into hi
// codes, copied to columns [0, 64) and the first 4 KB of `q_rope`, and lo
// codes, to [64, 128) and the second 4 KB, with the factor 2^-k that the
// row's partial scores need.
// Returns that factor (1 for an e4m3 query).  Rows past the query tensor are
// zero (factor 1).  Called once per item, kept out of line.
__device__ __noinline__ float load_q_row_fp8_mma(const Problem& p, const uint4* split,
                                                 long long qrow, bool in, int q, uint32_t rank,
                                                 uint32_t tmem_q, unsigned char* q_rope) {
  const int sw = (q >> 2) & 1;  // 32B swizzle: 16-byte unit u of row q sits at u ^ sw
  if (p.q_fp8) {
    const uint4* src = reinterpret_cast<const uint4*>(
        reinterpret_cast<const unsigned char*>(p.query) + (in ? qrow : 0) * kQkDim);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint32_t w[32];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint4 x = in ? __ldg(src + 16 * (int)rank + 8 * half + u) : make_uint4(0, 0, 0, 0);
        w[4 * u] = x.x;
        w[4 * u + 1] = x.y;
        w[4 * u + 2] = x.z;
        w[4 * u + 3] = x.w;
      }
      tmem_st_32x32b_x16(tmem_q + 32 * half, *reinterpret_cast<const uint32_t(*)[16]>(w));
      tmem_st_32x32b_x16(tmem_q + 32 * half + 16, *reinterpret_cast<const uint32_t(*)[16]>(w + 16));
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint4 x = in ? __ldg(src + 32 + 2 * (int)rank + u) : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(q_rope + q * 32 + ((u ^ sw) << 4)) = x;
    }
    fence_proxy_async_smem();  // read by the RoPE MMA
    return 1.f;
  }
  // this (row, half)'s units: latent hi [0, 16), latent lo [16, 32), RoPE hi
  // [32, 34), RoPE lo [34, 36); one part per round of 18 loads
  const uint4* src = split + ((in ? qrow : 0) * 2 + rank) * kQSplitUnits;
#pragma unroll 1
  for (int part = 0; part < 2; ++part) {
    uint4 x[18];
#pragma unroll
    for (int u = 0; u < 16; ++u) x[u] = in ? __ldg(src + 16 * part + u) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < 2; ++u) x[16 + u] = in ? __ldg(src + 32 + 2 * part + u) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      tmem_st_32x32b_x16(tmem_q + 64 * part + 16 * j,
                         *reinterpret_cast<const uint32_t(*)[16]>(&x[4 * j]));
#pragma unroll
    for (int u = 0; u < 2; ++u)
      *reinterpret_cast<uint4*>(q_rope + part * (kRopeQ / 2) + q * 32 + ((u ^ sw) << 4)) = x[16 + u];
  }
  fence_proxy_async_smem();  // read by the RoPE MMAs
  return in ? __ldg(reinterpret_cast<const float*>(src + 36)) : 1.f;
}

// Producer of a sparse top-k decode: kGatherWarps warps (role 0 = warp 0,
// which also loads each item's query RoPE tile, and the last warps of the
// block) fill the ring together.  A tile is 64 entries of the item's token
// list, in 16 groups of four; role r takes the groups q = r, r + 3, ...  Its
// lane e resolves the e-th entry of those groups (the list entry, then its
// block-table page) into a cache row; an entry outside [0, L) (-1 padding, a
// position past the request) or with a page id out of range (which also sets
// kStatusPage) becomes the first row past the cache, which the copy fills
// with zeros, and its bit in the role's word of the tile's usable-row mask
// (shared memory, slot g mod 8) is clear, so the softmax masks its score.
// The rows come by TMA four-row gathers from maps with one-row boxes, so each
// row lands where, and swizzled as, a page copy would put it: per row group
// one gather per 64-dim latent chunk and one for the RoPE dims, into the bf16
// ring (e4m3: into the staging ring the converter warps widen).  A tile's full
// barrier waits for one arrival per role (role 0's also expects the tile's
// bytes), so it completes once every row has landed.  Issue from one warp
// is the limit (about 3 us a tile), hence several warps.  The index loads run
// ahead so that their latency stays off the tile period: during tile t the
// list entries of tile t + 3 and the page-table entries of tile t + 2 are
// loaded, and tile t + 1's rows are formed from loads issued a tile earlier.
template <bool kFp8>
__device__ __noinline__ void gather_producer(int role, const Ctx& c, const Problem& p,
                                             const WorkItem* items, int item_begin,
                                             int item_end, unsigned char* sm, uint32_t rank,
                                             int R, const CUtensorMap* tm_q_rope,
                                             const CUtensorMap* tm_kv,
                                             const CUtensorMap* tm_kv_rope) {
  using C = Cfg<kFp8, true>;
  constexpr int kStages = C::kStages;
  constexpr int kGroups = kTile / 4;
  const int lane = threadIdx.x & 31;
  const int H = p.num_heads, ps = p.page_size;
  const int past_end = (int)(p.num_pages * ps);  // first row past the cache: zero-filled
  const int n_groups = (kGroups - role + kGatherWarps - 1) / kGatherWarps;
  // the tile row this lane resolves (-1: none)
  const int my_row = lane < 4 * n_groups ? 4 * (role + kGatherWarps * (lane >> 2)) + (lane & 3) : -1;
  unsigned long long* vmask = reinterpret_cast<unsigned long long*>(sm + OFF_VMASK);
  if (lane == 0) {
    if (role == 0) tma_prefetch_desc(tm_q_rope);
    tma_prefetch_desc(tm_kv);
    tma_prefetch_desc(tm_kv_rope);
  }
  uint32_t g = 0;
  int n_item = 0;
  for (int idx = item_begin; idx < item_end; ++idx) {
    const WorkItem it = items[idx];
    const int nt = n_tiles_of(it);
    if (nt <= 0) continue;
    const int* list = p.sparse_idx + (size_t)(it.q_start + it.g) * (size_t)p.sparse_k;
    const int* bt = p.block_tables + (size_t)it.b * p.max_pages;
    // list entry of this lane's row of tile t (-1 past the item's range)
    auto load_list = [&](int t) -> int {
      const int n = it.kv_begin + t * kTile + my_row;
      return (my_row >= 0 && t < nt && n < it.kv_end) ? __ldg(list + n) : -1;
    };
    // its page-table entry (-1 for an unused entry)
    auto load_page = [&](int j) -> int {
      return (j >= 0 && j < it.seq_len) ? __ldg(bt + j / ps) : -1;
    };
    // its cache row, and this role's word of the usable-row mask
    auto finish = [&](int j, int pg, int& row, unsigned long long& word) {
      bool on = j >= 0 && j < it.seq_len;
      if (on && (pg < 0 || (long long)pg >= p.num_pages)) {
        atomicOr(c.status, kStatusPage);
        on = false;
      }
      row = on ? pg * ps + j % ps : past_end;
      const uint32_t lo = __reduce_or_sync(0xffffffffu, on && my_row < 32 ? 1u << my_row : 0u);
      const uint32_t hi =
          __reduce_or_sync(0xffffffffu, on && my_row >= 32 ? 1u << (my_row - 32) : 0u);
      word = ((unsigned long long)hi << 32) | lo;
    };
    // j1, j2: list entries of tiles t + 1, t + 2; pg1: page entry of tile t + 1
    const int j0 = load_list(0);
    int j1 = load_list(1), j2 = load_list(2);
    int pg1 = load_page(j1);
    int row;
    unsigned long long word;
    finish(j0, load_page(j0), row, word);
    if (role == 0) {
      const bool q_ok = lane == 0 ? wait_bar(c, Q_FREE, (n_item & 1) ^ 1) : false;
      if (!__shfl_sync(0xffffffffu, q_ok, 0)) goto out;
      if (lane == 0) {
        if (p.q_fp8) {
          mbar_arrive(&c.bars[Q_FULL]);  // the RoPE half is widened into smem with the latent part
        } else {
          mbar_arrive_expect_tx(&c.bars[Q_FULL], kRopeQ);
          tma_load_2d(sm + OFF_QROPE, tm_q_rope, 512 + 32 * (int)rank, it.q_start * H + it.g * R,
                      &c.bars[Q_FULL]);
        }
      }
    }
    ++n_item;
    for (int t = 0; t < nt; ++t, ++g) {
      const int s = kFp8 ? (int)(g & 1) : (int)(g % kStages);
      const uint32_t use = kFp8 ? (g >> 1) : g / kStages;
      const bool ok =
          lane == 0 ? wait_bar(c, kFp8 ? STG_EMPTY0 + s : KV_EMPTY0 + s, (use & 1) ^ 1) : false;
      if (!__shfl_sync(0xffffffffu, ok, 0)) goto out;
      // index loads of later tiles, in flight during this tile's gathers
      const int j3 = load_list(t + 3);
      const int pg2 = load_page(j2);
      uint64_t* full = &c.bars[kFp8 ? STG_FULL0 + s : KV_FULL0 + s];
      if (lane == 0) {
        vmask[kGatherWarps * (g & 7) + role] = word;
        if (role == 0)
          mbar_arrive_expect_tx(full, kFp8 ? kStgBytes : kStageBytes);
        else
          mbar_arrive(full);
      }
      // lane l < n_groups: row group q = role + 3 l, rows 4q .. 4q + 3
      int y[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) y[i] = __shfl_sync(0xffffffffu, row, (4 * lane + i) & 31);
      if (lane < n_groups) {
        const int q = role + kGatherWarps * lane;
#pragma unroll
        for (int part = 0; part <= kLatChunks; ++part) {
          if (kFp8) {
            unsigned char* stg = sm + C::OFF_STG + s * kStgBytes;
            if (part < kLatChunks)
              tma_gather4(stg + part * kTile * 64 + 4 * q * 64, tm_kv,
                          256 * (int)rank + 64 * part, y[0], y[1], y[2], y[3], full);
            else
              tma_gather4(stg + kLatChunks * kTile * 64 + 4 * q * 32, tm_kv_rope,
                          512 + 32 * (int)rank, y[0], y[1], y[2], y[3], full);
          } else {
            unsigned char* stage = sm + OFF_KV + s * kStageBytes;
            if (part < kLatChunks)
              tma_gather4(stage + part * kChunkKV + 4 * q * 128, tm_kv,
                          256 * (int)rank + 64 * part, y[0], y[1], y[2], y[3], full);
            else
              tma_gather4(stage + kLatChunks * kChunkKV + 4 * q * 64, tm_kv_rope,
                          512 + 32 * (int)rank, y[0], y[1], y[2], y[3], full);
          }
        }
      }
      finish(j1, pg1, row, word);
      j1 = j2;
      j2 = j3;
      pg1 = pg2;
    }
  }
out:
  // however the loop ended, no copy issued here may still be landing in shared
  // memory when the CTA leaves: wait for the last tiles of the ring and the
  // last query load (phases already complete pass at once)
  if (lane == 0) {
    const uint32_t depth = kFp8 ? 2u : (uint32_t)kStages;
    for (uint32_t d = 0; d < depth && d < g; ++d) {
      const uint32_t gi = g - 1 - d;
      const int s = kFp8 ? (int)(gi & 1) : (int)(gi % kStages);
      const uint32_t use = kFp8 ? (gi >> 1) : gi / kStages;
      drain_wait(&c.bars[kFp8 ? STG_FULL0 + s : KV_FULL0 + s], use & 1);
    }
    if (role == 0 && n_item > 0) drain_wait(&c.bars[Q_FULL], (uint32_t)(n_item - 1) & 1);
  }
}

template <bool kFp8, bool kSparse, bool kF8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg<kFp8, kSparse, kF8>::kThreads, 1)
decode_sm103_kernel(const Problem p, const Layout lay, char* __restrict__ ws,
                    const __grid_constant__ CUtensorMap tm_q_rope,
                    const __grid_constant__ CUtensorMap tm_kv,
                    const __grid_constant__ CUtensorMap tm_kv_rope) {
  using C = Cfg<kFp8, kSparse, kF8>;
  constexpr int kStages = C::kStages;
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
  uint4* part_o = reinterpret_cast<uint4*>(ws + lay.part_o);  // see part_unit
  float* part_lse = reinterpret_cast<float*>(ws + lay.part_lse);
  int* comb_done = reinterpret_cast<int*>(ws + lay.comb_done);

  Ctx c;
  c.bars = reinterpret_cast<uint64_t*>(sm + OFF_BARS);
  c.abort = reinterpret_cast<volatile int*>(sm + OFF_ABORT);
  c.peer_abort = map_to_rank(smem_u32(sm + OFF_ABORT), peer);
  c.status = &hdr[kHdrStatus];
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_TMEM);
  float* fac = reinterpret_cast<float*>(sm + OFF_FAC);
  float* lrow = reinterpret_cast<float*>(sm + OFF_LROW);
  float* mrow = reinterpret_cast<float*>(sm + OFF_MROW);
  volatile int* flags = reinterpret_cast<volatile int*>(sm + OFF_FLAG);

  if (tid == 0) {
    uint32_t counts[NUM_BARS];
    for (int i = 0; i < NUM_BARS; ++i) counts[i] = 1;
    // thread groups arrive once per warp (lane 0, after __syncwarp); a tile
    // of parity G is handled by softmax group G (four warps)
    counts[S_FREE0] = counts[S_FREE1] = kGroupWarps + kCeWarps;
    counts[PEER_X_FREE0] = counts[PEER_X_FREE1] = kGroupWarps;    // the peer's group
    counts[P_FULL0] = counts[P_FULL1] = kGroupWarps;              // + the peer's bytes
    counts[P_FREE0] = counts[P_FREE1] = 2;                        // both CTAs' PV
    counts[LROW_FREE] = 2 * kCeWarps;                             // both CTAs' epilogues
    counts[CORR_DONE] = counts[EPI_DONE] = counts[QT_FULL] = kCeWarps;
    counts[QS_FULL0] = counts[QS_FULL1] = kCeWarps;
    if (kFp8) {
      for (int i = 0; i < kStages; ++i) counts[KV_FULL0 + i] = kConvThreads / 32;
      counts[STG_EMPTY0] = counts[STG_EMPTY1] = kConvThreads / 32;
    }
    if (kSparse) {  // one arrival per gather warp on the ring the rows land in
      if (kFp8)
        counts[STG_FULL0] = counts[STG_FULL1] = kGatherWarps;
      else
        for (int i = 0; i < kStages; ++i) counts[KV_FULL0 + i] = kGatherWarps;
    }
    for (int i = 0; i < NUM_BARS; ++i) mbar_init(&c.bars[i], counts[i]);
    *c.abort = 0;
    for (int k = 0; k < 32; ++k) flags[k] = -1;
    fence_mbar_init();
    // the first two tiles' peer scores may arrive as soon as the cluster is up
    mbar_arrive_expect_tx(&c.bars[X_FULL0], kXBytes);
    mbar_arrive_expect_tx(&c.bars[X_FULL1], kXBytes);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before any remote access
  // the work list comes from the partition kernel; the combine kernel may be
  // scheduled as soon as SMs free up (it waits on the per-entry counters that
  // the epilogues bump, so every CTA here is resident before it can spin)
  pdl_wait();
  pdl_launch_dependents();
  const uint32_t tmem = *tmem_slot;
  const int item_begin = worker_begin[worker], item_end = worker_begin[worker + 1];
  const int H = p.num_heads;
  const int R = lay.rows_per_group;  // query rows of a work item: 128, or H (sparse top-k)

  if (kSparse && (warp == 0 || warp >= C::kFirstExtraGatherWarp)) {
    gather_producer<kFp8>(warp == 0 ? 0 : 1 + warp - C::kFirstExtraGatherWarp, c, p, items,
                          item_begin, item_end, sm, rank, R, &tm_q_rope, &tm_kv, &tm_kv_rope);
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // Lane 0 waits for ring slots and issues the copies.  The whole warp
    // fetches the item's page ids in batches of 32 (one per lane), one batch
    // ahead, so no page-table read latency sits between two tiles' copies.
    if (lane == 0) {
      tma_prefetch_desc(&tm_q_rope);
      tma_prefetch_desc(&tm_kv);
      tma_prefetch_desc(&tm_kv_rope);
    }
    uint32_t g = 0;
    int n_item = 0;
    const int ps = p.page_size;
    const int npg = kTile / ps;  // 1 or 2 pages per tile
    for (int idx = item_begin; idx < item_end; ++idx) {
      const WorkItem it = items[idx];
      const int nt = n_tiles_of(it);
      if (nt <= 0) continue;
      // page slot i of the item = block-table entry first + i (tiles start on
      // a page boundary); only the pages the item's rows touch are read
      const int* bt = p.block_tables + (size_t)it.b * p.max_pages + it.kv_begin / ps;
      const int n_pages = (it.kv_end - it.kv_begin + ps - 1) / ps;
      int cur = lane < n_pages ? bt[lane] : -1;
      int nxt = 32 + lane < n_pages ? bt[32 + lane] : -1;
      const bool q_ok = lane == 0 ? wait_bar(c, Q_FREE, (n_item & 1) ^ 1) : false;
      if (!__shfl_sync(0xffffffffu, q_ok, 0)) goto done_producer;
      ++n_item;
      if (lane == 0) {
        if (p.q_fp8 || kF8) {
          // the RoPE half is written into smem with the latent part (widened,
          // or split into e4m3 parts)
          mbar_arrive(&c.bars[Q_FULL]);
        } else {
          mbar_arrive_expect_tx(&c.bars[Q_FULL], kRopeQ);
          tma_load_2d(sm + OFF_QROPE, &tm_q_rope, 512 + 32 * (int)rank,
                      it.q_start * H + it.g * R, &c.bars[Q_FULL]);
        }
      }
      for (int t = 0; t < nt; ++t, ++g) {
        const int slot0 = t * npg;  // never straddles a batch: npg divides 32
        if (slot0 > 0 && (slot0 & 31) == 0) {
          cur = nxt;
          const int i = slot0 + 32 + lane;
          nxt = i < n_pages ? bt[i] : -1;
        }
        int pages[2];
        pages[0] = __shfl_sync(0xffffffffu, cur, slot0 & 31);
        pages[1] = __shfl_sync(0xffffffffu, cur, (slot0 + 1) & 31);
        // bf16: load straight into the bf16 ring; e4m3: into the staging ring
        const int s = kFp8 ? (int)(g & 1) : (int)(g % kStages);
        const uint32_t use = kFp8 ? (g >> 1) : g / kStages;
        const bool ok =
            lane == 0 ? wait_bar(c, kFp8 ? STG_EMPTY0 + s : KV_EMPTY0 + s, (use & 1) ^ 1) : false;
        if (!__shfl_sync(0xffffffffu, ok, 0)) goto done_producer;
        if (lane == 0) {
          const int j0 = it.kv_begin + t * kTile;
          uint32_t bytes = 0;
          for (int pg = 0; pg < npg; ++pg) {
            if (j0 + pg * ps >= it.kv_end) {
              pages[pg] = -1;
              continue;
            }
            if (pages[pg] < 0 || (long long)pages[pg] >= p.num_pages) {
              atomicOr(c.status, kStatusPage);
              pages[pg] = -1;
              continue;
            }
            bytes += ps * (kLatChunks * 64 + 32) * (kFp8 || kF8 ? 1 : 2);
          }
          uint64_t* full = &c.bars[kFp8 ? STG_FULL0 + s : KV_FULL0 + s];
          mbar_arrive_expect_tx(full, bytes);
          for (int pg = 0; pg < npg; ++pg) {
            if (pages[pg] < 0) continue;
            const int y = pages[pg] * ps;
            if (kF8) {
              // e4m3 rows straight into the ring, in the layouts the FP8 MMAs read
              unsigned char* stage = sm + OFF_KV + s * C::kStage;
              for (int lc = 0; lc < 2; ++lc)
                tma_load_2d(stage + lc * kChunk8 + pg * ps * 128, &tm_kv, 256 * (int)rank + 128 * lc,
                            y, full);
              tma_load_2d(stage + 2 * kChunk8 + pg * ps * 32, &tm_kv_rope, 512 + 32 * (int)rank, y,
                          full);
            } else if (kFp8) {
              unsigned char* stg = sm + C::OFF_STG + s * kStgBytes;
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
        }
      }
    }
  done_producer:
    // however the loop ended, no copy issued here may still be landing in
    // shared memory when the CTA leaves: wait for the last ones (the tiles of
    // the ring and the last query load; phases already complete pass at once)
    if (lane == 0) {
      const uint32_t depth = kFp8 ? 2u : (uint32_t)kStages;
      for (uint32_t k = 0; k < depth && k < g; ++k) {
        const uint32_t gi = g - 1 - k;
        const int s = kFp8 ? (int)(gi & 1) : (int)(gi % kStages);
        const uint32_t use = kFp8 ? (gi >> 1) : gi / kStages;
        drain_wait(&c.bars[kFp8 ? STG_FULL0 + s : KV_FULL0 + s], use & 1);
      }
      if (n_item > 0) drain_wait(&c.bars[Q_FULL], (uint32_t)(n_item - 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Within an item QK(g) is issued as soon as its KV tile and S buffer are
    // ready (up to two tiles ahead of PV), PV(g) as soon as P(g) is complete.
    if (lane == 0) {
      constexpr uint32_t idesc_qk = kF8 ? idesc_e4m3(128, 64, false, false)
                                        : idesc_f16(128, 64, false, false);
      constexpr uint32_t idesc_pv = kF8 ? idesc_e4m3(128, 256, false, true)
                                        : idesc_f16(128, 256, false, true);
      // FP8 path: a bf16 query is two e4m3 parts (hi, lo), an e4m3 query one
      const int q_parts = p.q_fp8 ? 1 : 2;
      const uint32_t qr_base = smem_u32(sm + OFF_QROPE);
      const uint32_t kv_base = smem_u32(sm + OFF_KV);
      const uint32_t p_base = smem_u32(sm + OFF_P);
      uint32_t g0 = 0, n_rescale = 0;
      int n_item = 0;
      for (int idx = item_begin; idx < item_end; ++idx) {
        const WorkItem it = items[idx];
        const int nt = n_tiles_of(it);
        if (nt <= 0) continue;
        if (!wait_bar(c, Q_FULL, n_item & 1) || !wait_bar(c, QT_FULL, n_item & 1)) goto done_mma;
        ++n_item;
        tc_fence_after();
        int qk = 0, pv = 0, pv_state = 0;
        uint32_t idle = 0;
        while (pv < nt) {
          bool progressed = false;
          // PV first: it frees a KV stage (and the next load) as early as possible
          if (pv < qk) {
            // PV(pv): wait (without blocking QK issue) for P, for an O rescale
            // if one was asked for, and for the previous item's epilogue.
            const uint32_t gp = g0 + pv;
            const int pb = gp & 1;
            if (pv_state == 0 && mbar_test_wait(&c.bars[P_FULL0 + pb], (gp >> 1) & 1)) {
              if (pv > 0 && rescale_requested(sm, gp)) {
                mma_commit(&c.bars[O_STABLE]);  // the correction warps start after PV(pv - 1)
                pv_state = 1;
              } else {
                pv_state = 2;
              }
              progressed = true;
            }
            if (pv_state == 1 && mbar_test_wait(&c.bars[CORR_DONE], n_rescale & 1)) {
              ++n_rescale;
              pv_state = 2;
              progressed = true;
            }
            if (pv_state == 2 &&
                (pv != 0 || n_item <= 1 || mbar_test_wait(&c.bars[EPI_DONE], (n_item - 2) & 1))) {
              tc_fence_after();
              // the peer's P rows arrived through st.async (generic proxy); order
              // them before this thread's MMA reads (async proxy)
              fence_proxy_async_smem();
              const int s = gp % kStages;
              const uint32_t stage = kv_base + s * C::kStage;
              if (kF8) {
                // P as two e4m3 parts (64B-swizzled rows) against V read
                // MN-major from the two 128-dim chunks, K = 32 KV rows a step
                for (int k = 0; k < 2 * (kTile / 32); ++k) {
                  const int part = k >> 1, ks = k & 1;
                  const uint64_t a = smem_desc(p_base + pb * kPBytes + part * kPart8 + ks * 32, 16,
                                               512, kSwizzle64B);
                  const uint64_t b = smem_desc(stage + ks * 32 * 128, kChunk8, 1024, kSwizzle128B);
                  mma_e4m3_ss(tmem + TM_O, a, b, idesc_pv, (pv == 0 && k == 0) ? 0u : 1u);
                }
              } else {
                for (int ks = 0; ks < kTile / 16; ++ks) {
                  const uint64_t a =
                      smem_desc(p_base + pb * kPBytes + ks * 32, 16, 1024, kSwizzle128B);
                  const uint64_t b = smem_desc(stage + ks * 16 * 128, 8192, 1024, kSwizzle128B);
                  mma_bf16_ss(tmem + TM_O, a, b, idesc_pv, (pv == 0 && ks == 0) ? 0u : 1u);
                }
              }
              mma_commit(&c.bars[KV_EMPTY0 + s]);
              // both CTAs' P tiles (of this parity) are free
              mma_commit_multicast(&c.bars[P_FREE0 + pb], 0x3);
              if (pv + 1 == nt) mma_commit(&c.bars[O_FINAL]);
              ++pv;
              pv_state = 0;
              progressed = true;
            }
          }
          if (!progressed && qk < nt && qk <= pv + 2) {
            const uint32_t gq = g0 + qk;
            const int s = gq % kStages, sb = gq & 1;
            if (mbar_test_wait(&c.bars[KV_FULL0 + s], (gq / kStages) & 1) &&
                mbar_test_wait(&c.bars[S_FREE0 + sb], ((gq >> 1) & 1) ^ 1)) {
              tc_fence_after();
              const uint32_t d = tmem + TM_S + 64 * sb;
              const uint32_t stage = kv_base + s * C::kStage;
              if (kF8) {
                for (int part = 0; part < q_parts; ++part) {
                  for (int k = 0; k < 8; ++k) {
                    const int lc = k >> 2, ks = k & 3;
                    const uint64_t b =
                        smem_desc(stage + lc * kChunk8 + ks * 32, 16, 1024, kSwizzle128B);
                    // 32 dims = 8 TMEM columns of four e4m3 codes
                    mma_e4m3_ts(d, tmem + TM_Q + 64 * part + 32 * lc + 8 * ks, b, idesc_qk,
                                (part | k) != 0 ? 1u : 0u);
                  }
                  const uint64_t a = smem_desc(qr_base + part * (kRopeQ / 2), 16, 256, kSwizzle32B);
                  const uint64_t b = smem_desc(stage + 2 * kChunk8, 16, 256, kSwizzle32B);
                  mma_e4m3_ss(d, a, b, idesc_qk, 1u);
                }
              } else {
                for (int k = 0; k < 4 * kLatChunks; ++k) {
                  const int lc = k >> 2, ks = k & 3;
                  const uint64_t b =
                      smem_desc(stage + lc * kChunkKV + ks * 32, 16, 1024, kSwizzle128B);
                  // 16 dims = 8 TMEM columns of bf16 pairs
                  mma_bf16_ts(d, tmem + TM_Q + 32 * lc + 8 * ks, b, idesc_qk, k > 0 ? 1u : 0u);
                }
                for (int ks = 0; ks < 2; ++ks) {
                  const uint64_t a = smem_desc(qr_base + ks * 32, 16, 512, kSwizzle64B);
                  const uint64_t b = smem_desc(stage + kLatChunks * kChunkKV + ks * 32, 16, 512,
                                               kSwizzle64B);
                  mma_bf16_ss(d, a, b, idesc_qk, 1u);
                }
              }
              mma_commit(&c.bars[S_FULL0 + sb]);
              if (++qk == nt) mma_commit(&c.bars[Q_FREE]);
              progressed = true;
            }
          }
          if (progressed) {
            idle = 0;
          } else if (++idle > kWaitLimit || ((idle & 1023) == 0 && *c.abort)) {
            if (idle > kWaitLimit) {
              give_up(c);
            }
            goto done_mma;
          }
        }
        g0 += nt;
      }
    done_mma:
      mma_commit(&c.bars[MMA_DRAIN]);
      drain_wait(&c.bars[MMA_DRAIN], 0);
    }
  } else if (warp >= 2 && warp < 2 + kSoftmaxWarps) {
    // ------------------------------------------------------------ softmax (owned rows)
    // Group grp = (w - 2) / 4 takes the KV tiles of global parity grp.  Its
    // warp w covers the 16 owned lanes of subpartition sp = w mod 4: thread t
    // takes lane 32 sp + 16 r + (t mod 16) and KV columns [32 hh, 32 hh + 32),
    // hh = t / 16, so a row's two threads meet in one shuffle.  Tile g's
    // running-max reference comes from the other group (tile g - 1) through
    // shared memory; each group keeps its own share of the row sum.
    const int sp = warp & 3, grp = (warp - 2) >> 2, hh = lane >> 4;
    const int fw = (warp - 2) & 3;                         // warp within the group
    const int k = 16 * sp + (lane & 15);                   // owned-row index
    const int q = 32 * sp + 16 * (int)rank + (lane & 15);  // query row == TMEM lane
    const uint32_t lane_addr = (uint32_t)(32 * sp + 16 * (int)rank) << 16;
    const bool designated = fw == 0 && lane == 0;
    const int g_tid = fw * 32 + lane;  // thread within the group
    const float bmm1_log2e = run_bmm1(p, c.status) * kLog2e;
    const float* qscale = reinterpret_cast<const float*>(sm + OFF_QSCALE);
    float* mref = reinterpret_cast<float*>(sm + OFF_MREF);  // [tile parity][row]
    float* lx = reinterpret_cast<float*>(sm + OFF_LX);      // [item parity][l, m][row]
    const uint32_t xfree_peer0 = map_to_rank(smem_u32(&c.bars[PEER_X_FREE0]), peer);
    const uint32_t pfull_peer0 = map_to_rank(smem_u32(&c.bars[P_FULL0]), peer);
    const uint32_t p_peer0 = map_to_rank(smem_u32(sm + OFF_P), peer);
    const uint32_t fac_peer0 = map_to_rank(smem_u32(sm + OFF_FAC), peer);
    const uint32_t flag_peer0 = map_to_rank(smem_u32(sm + OFF_FLAG), peer);
    const uint32_t lrow_peer = map_to_rank(smem_u32(sm + OFF_LROW), peer);
    const int W = max(p.cp_world, 1);
    constexpr bool sparse = kSparse;
    const unsigned long long* vmask = reinterpret_cast<const unsigned long long*>(sm + OFF_VMASK);
    uint32_t g = 0;
    int n_item = 0;
    int n_multi = 0;  // items of two or more tiles so far: they alone use the (l, m) hand-off
    for (int idx = item_begin; idx < item_end; ++idx) {
      const WorkItem it = items[idx];
      const int nt = n_tiles_of(it);
      if (nt <= 0) continue;
      const int rows_total = it.q_len * H;
      const int row0 = it.g * R;
      const bool row_ok = q < min(R, rows_total - row0);
      const int qi = (row0 + q) / H;
      // sparse top-k: the producer's usable-row mask of each tile is the mask
      const int last = sparse ? INT_MAX
                              : (p.causal ? causal_last(it.mask_base, qi, W) : it.seq_len - 1);
      // tiles ending at or before `clean_end` need no mask for any valid row
      const int first_qi = row0 / H;
      const int clean_end =
          sparse ? it.kv_begin
                 : min(it.kv_end,
                       p.causal ? causal_last(it.mask_base, first_qi, W) + 1 : it.seq_len);
      const uint32_t g_last = g + (uint32_t)nt - 1;
      // (l, m) hand-off slot of this item and the phase of its barrier: only
      // items of two or more tiles (both groups take part) count
      const int ip = n_multi & 1;
      const uint32_t lx_phase = (uint32_t)(n_multi >> 1) & 1;
      // this group's share of the row sum (this thread's 32 columns), relative
      // to the reference m_grp of the group's latest tile of the item
      float l_part = 0.f, m_grp = -INFINITY;
      // FP8 path: this CTA's partial scores are 2^k times the true ones (the
      // MMAs saw its half of the query times 2^k); the factor 2^-k of the
      // item's row is read at the group's first tile of the item
      const float scale = bmm1_log2e;
      float qs_own = 1.f;
      bool have_scale = !kF8;
      for (int t = 0; t < nt; ++t, ++g) {
        if ((int)(g & 1) != grp) continue;
        const int sb = grp;
        float sv[32];
        if (!have_scale) {
          if (!wait_bar(c, QS_FULL0 + (n_item & 1), (n_item >> 1) & 1)) goto done_softmax;
          qs_own = qscale[(n_item & 1) * kRows + q];
          have_scale = true;
        }
        if (!wait_bar(c, S_FULL0 + sb, (g >> 1) & 1)) goto done_softmax;
        tc_fence_after();
        {
          uint32_t v[32];
          tmem_ld_16x32bx2_x32(tmem + lane_addr + TM_S + 64 * sb, v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) sv[j] = __uint_as_float(v[j]) * qs_own;  // exact: 2^-k
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.bars[S_FREE0 + sb]);
        // add the peer's partial scores of this row (fp32, columns
        // [32 hh, 32 hh + 32) = 16-byte units 8 hh .. 8 hh + 7 of the row)
        if (!wait_bar(c, X_FULL0 + sb, (g >> 1) & 1)) goto done_softmax;
        {
          const unsigned char* xb = sm + OFF_X + sb * kXBytes + k * kXRowBytes;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float4 x = *reinterpret_cast<const float4*>(xb + (((8 * hh + u) ^ (k & 7)) << 4));
            sv[4 * u] += x.x;
            sv[4 * u + 1] += x.y;
            sv[4 * u + 2] += x.z;
            sv[4 * u + 3] += x.w;
          }
        }
        // the buffer's next phase (tile g + 2) completes once the peer's bytes
        // for it land, which the peer sends only after this group released
        // this tile's scores (PEER_X_FREE)
        if (designated) mbar_arrive_expect_tx(&c.bars[X_FULL0 + sb], kXBytes);
        // relaxed: the warp's reads of the buffer have returned their values
        // (release at cluster scope would cost a cluster-wide fence per tile)
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(xfree_peer0 + 8u * sb);
        // mask, then the row maximum of the tile (log2 units)
        const int j0 = it.kv_begin + t * kTile;
        const int c0 = j0 + 32 * hh;  // KV index of sv[0]
        // tiles with masked columns are scaled before the -inf mask goes in,
        // so that bmm1 = 0 never multiplies -inf (the same for the whole tile)
        const bool pre_scaled = j0 + kTile > clean_end;
        const float sc = pre_scaled ? 1.f : scale;  // what the scores still need
        uint32_t usable = 0xffffffffu;              // of this thread's 32 columns
        if (sparse) {
          // the mask was written before the tile's full barrier completed
          if (!wait_bar(c, KV_FULL0 + (int)(g % kStages), (g / kStages) & 1)) goto done_softmax;
          unsigned long long u = 0;
#pragma unroll
          for (int r = 0; r < kGatherWarps; ++r) u |= vmask[kGatherWarps * (g & 7) + r];
          usable = (uint32_t)(u >> (32 * hh));
        }
        float m_tile = -INFINITY;
        if (row_ok) {
          float tm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // 4 chains for ILP
          if (!pre_scaled) {
#pragma unroll
            for (int j = 0; j < 32; ++j) tm[j & 3] = fmaxf(tm[j & 3], sv[j]);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int col = c0 + j;
              sv[j] = (col <= last && col < it.kv_end && ((usable >> j) & 1u)) ? sv[j] * scale
                                                                                : -INFINITY;
              tm[j & 3] = fmaxf(tm[j & 3], sv[j]);
            }
          }
          m_tile = fmaxf(fmaxf(tm[0], tm[1]), fmaxf(tm[2], tm[3]));
        }
        m_tile = fmaxf(m_tile, __shfl_xor_sync(0xffffffffu, m_tile, 16)) * sc;
        // The item's running reference after tile g - 1 (the other group's
        // tile); every tile but the very first waits for it, even where it
        // starts an item and ignores the value, so that the barrier phases of
        // the two groups stay in step.
        float m_prev = -INFINITY;
        if (g > 0) {
          const uint32_t gp = g - 1;
          if (!wait_bar(c, MREF0 + 4 * (gp & 1) + sp, (gp >> 1) & 1)) goto done_softmax;
          if (t > 0) m_prev = mref[(gp & 1) * kRows + q];
        }
        // raised (and O rescaled) only when the tile's maximum passes it by
        // more than the threshold; the first tile of an item sets it
        const float m_new =
            (t == 0 || m_tile > m_prev + kRescaleThreshold) ? (row_ok ? m_tile : m_prev) : m_prev;
        if (hh == 0) mref[sb * kRows + q] = m_new;
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.bars[MREF0 + 4 * sb + sp]);
        const bool need = t > 0 && m_new != m_prev;
        const float f = need ? ex2(m_prev - m_new) : 1.f;  // m_prev = -inf gives 0
        if (m_new > m_grp) {  // rebase this group's share (0 while m_grp = -inf)
          l_part *= ex2(m_grp - m_new);
          m_grp = m_new;
        }
        if (row_ok) {
          const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
          float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            sv[j] = ex2(fmaf(sv[j], sc, -m_use));
            rs[j & 3] += sv[j];
          }
          l_part += (rs[0] + rs[1]) + (rs[2] + rs[3]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) sv[j] = 0.f;
        }
        // zero V rows past the end of the KV range (last tile of the item)
        const int valid = it.kv_end - j0;
        if (valid < kTile) {
          unsigned char* stage = sm + OFF_KV + (g % kStages) * C::kStage;
          constexpr int kChunks = kF8 ? 2 : kLatChunks;  // 128-byte rows per KV row
          constexpr uint32_t kChunkBytes = kF8 ? kChunk8 : kChunkKV;
          const int nz = (kTile - valid) * kChunks * 8;  // 16-byte units
          for (int e = g_tid; e < nz; e += kGroupWarps * 32) {
            const int row = valid + e / (8 * kChunks), ch = (e / 8) % kChunks, u = e % 8;
            *reinterpret_cast<uint4*>(stage + ch * kChunkBytes + row * 128 + u * 16) =
                make_uint4(0, 0, 0, 0);
          }
        }
        // P (bf16) of this row into both CTAs' P tiles of this parity once both
        // CTAs' PV of tile g - 2 read them
        if (!wait_bar(c, P_FREE0 + sb, ((g >> 1) & 1) ^ 1)) goto done_softmax;
        {
          const uint32_t pbar = pfull_peer0 + 8u * sb;
          unsigned char* ptile = sm + OFF_P + sb * kPBytes;
          const uint32_t ppeer = p_peer0 + sb * kPBytes;
          if (kF8) {
            // two e4m3 parts: hi = e4m3(p), lo = e4m3(p - hi); their sum is p to
            // about 2^-8 relative (64B-swizzled rows of 64 codes per part)
            uint32_t hw[8], lw[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const uint32_t h01 = f32x2_to_e4m3x2(sv[4 * e], sv[4 * e + 1]);
              const uint32_t h23 = f32x2_to_e4m3x2(sv[4 * e + 2], sv[4 * e + 3]);
              float f0, f1, f2, f3;
              e4m3x2_to_f32x2(h01, f0, f1);
              e4m3x2_to_f32x2(h23, f2, f3);
              hw[e] = h01 | (h23 << 16);
              lw[e] = f32x2_to_e4m3x2(sv[4 * e] - f0, sv[4 * e + 1] - f1) |
                      (f32x2_to_e4m3x2(sv[4 * e + 2] - f2, sv[4 * e + 3] - f3) << 16);
            }
#pragma unroll
            for (int part = 0; part < 2; ++part) {
              const uint32_t* w = part ? lw : hw;
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const uint32_t off =
                    part * kPart8 + q * 64 + (((2 * hh + u) ^ ((q >> 1) & 3)) << 4);
                const uint4 val = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                *reinterpret_cast<uint4*>(ptile + off) = val;
                st_async_v4_b32(ppeer + off, val, pbar);
              }
            }
          } else {
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) w[e] = pack_bf16(sv[2 * e], sv[2 * e + 1]);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const uint32_t off = q * 128 + (((4 * hh + u) ^ (q & 7)) << 4);
              const uint4 val = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
              *reinterpret_cast<uint4*>(ptile + off) = val;
              st_async_v4_b32(ppeer + off, val, pbar);
            }
          }
          if (hh == 0) {
            fac[sb * kRows + q] = f;
            st_async_b32(fac_peer0 + 4u * (sb * kRows + q), __float_as_uint(f), pbar);
          }
          const bool any = __any_sync(0xffffffffu, need);
          if (lane == 0) {
            const int fv = any ? (int)g : -1;
            flags[16 * sb + fw] = fv;
            st_async_b32(flag_peer0 + 4u * (16 * sb + 8 + fw), (uint32_t)fv, pbar);
          }
        }
        if (g == g_last) {
          // the row sum of the item: this group's share plus the other
          // group's, published when it finished its tiles of the item
          float l_row = l_part + __shfl_xor_sync(0xffffffffu, l_part, 16);
          if (nt > 1) {
            if (!wait_bar(c, LX0 + 4 * ip + sp, lx_phase)) goto done_softmax;
            const float l_o = lx[(2 * ip) * kRows + q];
            const float m_o = lx[(2 * ip + 1) * kRows + q];
            if (l_o > 0.f) l_row += l_o * ex2(m_o - m_new);
          }
          // the previous item's epilogues (both CTAs) have read l
          if (n_item > 0 && !wait_bar_cluster(c, LROW_FREE, (n_item - 1) & 1)) goto done_softmax;
          if (hh == 0) {
            lrow[q] = l_row;
            mrow[q] = m_new;  // a split chunk's LSE is written by the epilogue warps
            st_async_b32(lrow_peer + 4u * q, __float_as_uint(l_row), pfull_peer0 + 8u * sb);
            if (row_ok && it.slot < 0 && p.return_lse) {
              const float lse = l_row > 0.f ? (m_new + log2f(l_row)) * kLn2 : -INFINITY;
              p.lse[(size_t)it.q_start * H + row0 + q] = lse;
            }
          }
        }
        fence_proxy_async_smem();  // P and zeroed V rows are read by the MMA
        __syncwarp();
        if (lane == 0) {
          if (fw == 0)
            mbar_arrive_expect_tx(&c.bars[P_FULL0 + sb],
                                  kPeerPBytes + (g == g_last ? kPeerLBytes : 0u));
          else
            mbar_arrive(&c.bars[P_FULL0 + sb]);
        }
      }
      if (nt > 1 && grp != (int)(g_last & 1)) {
        // hand this group's share of the row sum to the group of the last tile
        const float l_row = l_part + __shfl_xor_sync(0xffffffffu, l_part, 16);
        if (hh == 0) {
          lx[(2 * ip) * kRows + q] = l_row;
          lx[(2 * ip + 1) * kRows + q] = m_grp;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.bars[LX0 + 4 * ip + sp]);
      }
      if (nt > 1) ++n_multi;
      ++n_item;
    }
  done_softmax:;
  } else if (warp >= 2 + kSoftmaxWarps && warp < 2 + kSoftmaxWarps + kCeWarps) {
    // ------------------------------------------------------------ send + correction + epilogue
    // Threads t and t + 16 of warp w push the peer-owned row at lane
    // 32 (w mod 4) + 16 (1 - r) + (t mod 16) of each partial-score tile to the
    // peer as soon as QK lands (columns [32 (t / 16), + 32)).  For correction,
    // the epilogue and the Q load, thread q = 32 (w mod 4) + t covers TMEM lane q.
    const int sp = warp & 3, hh = lane >> 4;
    const int q = 32 * sp + lane;  // query row == TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * sp) << 16;
    const uint32_t peer_lanes = (uint32_t)(32 * sp + 16 * (int)peer) << 16;
    const int kp = 16 * sp + (lane & 15);  // the peer's owned-row index of my send row
    const uint32_t x_peer0 = map_to_rank(smem_u32(sm + OFF_X), peer);
    const uint32_t xfull_peer0 = map_to_rank(smem_u32(&c.bars[X_FULL0]), peer);
    const uint32_t lfree_peer = map_to_rank(smem_u32(&c.bars[LROW_FREE]), peer);
    uint32_t g = 0, n_rescale = 0;
    int n_item = 0;
    // `valid`: KV rows of the tile inside the item's range; the others may hold
    // stale shared memory (an unloaded page) and are masked by the softmax
    // FP8 path: per-row factors 2^-k of the query halves, by item parity
    float* qscale = reinterpret_cast<float*>(sm + OFF_QSCALE);
    auto send = [&](uint32_t gs, int valid) -> bool {
      const int sb = gs & 1;
      if (!wait_bar(c, S_FULL0 + sb, (gs >> 1) & 1)) return false;
      tc_fence_after();
      uint32_t v[32];
      tmem_ld_16x32bx2_x32(tmem + peer_lanes + TM_S + 64 * sb, v);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.bars[S_FREE0 + sb]);
      // the scores go over unrounded (fp32): the logits' error stays that of
      // the MMA's fp32 accumulation whatever the size of bmm1 * |S|.  FP8
      // path: in true units, i.e. times this CTA's factor 2^-k of the row
      // (written by this warp's lane of that row with the item's query)
      if (kF8) {
        const float qs = qscale[(n_item & 1) * kRows + 32 * sp + 16 * (int)peer + (lane & 15)];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * qs);
      }
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (32 * hh + j >= valid) v[j] = 0u;
      // the peer's softmax released the buffer (tile gs - 2's scores)
      if (!wait_bar_cluster(c, PEER_X_FREE0 + sb, ((gs >> 1) & 1) ^ 1)) return false;
      const uint32_t xb = x_peer0 + (uint32_t)(sb * kXBytes + kp * kXRowBytes);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        st_async_v4_b32(xb + (uint32_t)(((8 * hh + u) ^ (kp & 7)) << 4),
                        make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]),
                        xfull_peer0 + 8u * sb);
      return true;
    };
    // Row q of the item's Q latent dims of this CTA ([256 r, 256 r + 256)) into
    // TMEM, where they are the A operand of the ts QK MMAs (and, for an e4m3
    // query, its RoPE dims into smem).  Called only when no QK of an earlier
    // item is pending.
    const long long q_rows = p.total_q * H;
    const float bmm2 = run_bmm2(p);
    // `ordinal`: the item's place among this worker's items (its scale slot)
    auto write_q = [&](const WorkItem& it, int ordinal) {
      const long long qrow = (long long)it.q_start * H + (long long)it.g * R + q;
      const bool in = qrow < q_rows;
      if constexpr (kF8) {
        qscale[(ordinal & 1) * kRows + q] = load_q_row_fp8_mma(
            p, reinterpret_cast<const uint4*>(ws + q_split_offset(lay)), qrow, in, q, rank,
            tmem + lane_base + TM_Q, sm + OFF_QROPE);
      } else if (!p.q_fp8) {
        const uint4* src = reinterpret_cast<const uint4*>(
            reinterpret_cast<const __nv_bfloat16*>(p.query) + (in ? qrow : 0) * kQkDim +
            256 * (int)rank);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t w[64];
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const uint4 x = in ? __ldg(src + 16 * half + u) : make_uint4(0, 0, 0, 0);
            w[4 * u] = x.x;
            w[4 * u + 1] = x.y;
            w[4 * u + 2] = x.z;
            w[4 * u + 3] = x.w;
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tmem_st_32x32b_x16(tmem + lane_base + TM_Q + 64 * half + 16 * j,
                               *reinterpret_cast<const uint32_t(*)[16]>(w + 16 * j));
        }
      } else {
        load_q_row_e4m3(p, qrow, in, q, rank, tmem + lane_base + TM_Q, sm + OFF_QROPE);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&c.bars[QT_FULL]);
        if (kF8) mbar_arrive(&c.bars[QS_FULL0 + (ordinal & 1)]);
      }
    };
    auto correct = [&](uint32_t gc, bool first) -> bool {
      if (!wait_bar(c, P_FULL0 + (gc & 1), (gc >> 1) & 1)) return false;
      if (!first && rescale_requested(sm, gc)) {
        if (!wait_bar(c, O_STABLE, n_rescale & 1)) return false;
        ++n_rescale;
        tc_fence_after();
        const float f = fac[(gc & 1) * kRows + q];
#pragma unroll 1
        for (int c16 = 0; c16 < 16; ++c16) {
          uint32_t x[16];
          const uint32_t addr = tmem + lane_base + TM_O + 16 * c16;
          tmem_ld_32x32b_x16(addr, x);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) x[j] = __float_as_uint(__uint_as_float(x[j]) * f);
          tmem_st_32x32b_x16(addr, x);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.bars[CORR_DONE]);
      }
      return true;
    };
    for (int idx = item_begin; idx < item_end; ++idx) {
      const WorkItem it = items[idx];
      const int nt = n_tiles_of(it);
      if (nt <= 0) continue;
      if (n_item == 0) write_q(it, 0);
      for (int t = 0; t < nt; ++t, ++g) {
        if (!send(g, it.kv_end - (it.kv_begin + t * kTile))) goto done_epi;
        if (t > 0 && !correct(g - 1, t == 1)) goto done_epi;
      }
      // every QK of this item has completed (send saw the last S_FULL): the
      // next item's Q may replace this one in TMEM
      for (int nx = idx + 1; nx < item_end; ++nx) {
        const WorkItem itn = items[nx];
        if (n_tiles_of(itn) > 0) {
          write_q(itn, n_item + 1);
          break;
        }
      }
      if (!correct(g - 1, nt == 1)) goto done_epi;
      // epilogue: O / l for my V dims (l of every row arrived with the last P)
      if (!wait_bar(c, O_FINAL, n_item & 1)) goto done_epi;
      tc_fence_after();
      {
        const int rows_total = it.q_len * H;
        const int row0 = it.g * R;
        const bool row_ok = q < min(R, rows_total - row0);
        const float l = lrow[q];
        const float m = mrow[q];  // meaningful for the rows this CTA owns
        __syncwarp();
        if (lane == 0) {  // both CTAs' softmax may overwrite l (and m) for the next item
          mbar_arrive(&c.bars[LROW_FREE]);
          mbar_arrive_cluster_relaxed(lfree_peer);
        }
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const size_t grow = (size_t)it.q_start * H + row0 + q;
        // a split chunk's natural-log LSE of the rows this CTA owns (lane q is
        // owned by CTA (q / 16) mod 2); made visible with the partial O below
        if (it.slot >= 0 && row_ok && ((q >> 4) & 1) == (int)rank)
          part_lse[(size_t)it.slot * R + q] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
#pragma unroll 1
        for (int c16 = 0; c16 < 16; ++c16) {
          uint32_t x[16];
          tmem_ld_32x32b_x16(tmem + lane_base + TM_O + 16 * c16, x);
          tmem_wait_ld();
          if (!row_ok) continue;
          const int vd = 256 * (int)rank + 16 * c16;  // first output V dim of this chunk
          if (it.slot < 0) {
            const float s2 = inv * bmm2;
            uint32_t o[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              o[k] = pack_bf16(__uint_as_float(x[2 * k]) * s2, __uint_as_float(x[2 * k + 1]) * s2);
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) +
                                                  grow * kVDim + vd);
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
          } else {
            // this row's chunk of the split partial (consecutive rows store
            // consecutive 16-byte units: coalesced)
            const int cidx = 16 * (int)rank + c16;
            if (kPartialBf16) {
              uint32_t o[8];
#pragma unroll
              for (int k = 0; k < 8; ++k)
                o[k] = pack_bf16(__uint_as_float(x[2 * k]) * inv, __uint_as_float(x[2 * k + 1]) * inv);
              part_o[part_unit(it.slot, R, cidx, 0, q)] = make_uint4(o[0], o[1], o[2], o[3]);
              part_o[part_unit(it.slot, R, cidx, 1, q)] = make_uint4(o[4], o[5], o[6], o[7]);
            } else {
#pragma unroll
              for (int k = 0; k < 4; ++k)
                reinterpret_cast<float4*>(part_o)[part_unit(it.slot, R, cidx, k, q)] =
                    make_float4(__uint_as_float(x[4 * k]) * inv, __uint_as_float(x[4 * k + 1]) * inv,
                                __uint_as_float(x[4 * k + 2]) * inv, __uint_as_float(x[4 * k + 3]) * inv);
            }
          }
        }
      }
      tc_fence_before();
      if (it.slot >= 0) __threadfence();  // the partial is visible GPU-wide before it is counted
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.bars[EPI_DONE]);
      if (it.comb >= 0 && warp == 2 + kSoftmaxWarps) {
        // all four warps' partials (and the owners' LSEs) are written: count
        // this CTA's chunk, so the combine can merge the group (it merges
        // once both CTAs of every chunk have counted)
        if (!wait_bar(c, EPI_DONE, n_item & 1)) goto done_epi;
        if (lane == 0) {
          __threadfence();
          atomicAdd(comb_done + it.comb, 1);
        }
      }
      ++n_item;
    }
  done_epi:;
  } else if (kFp8 && warp >= 2 + kSoftmaxWarps + kCeWarps) {
    // ------------------------------------------------------------ e4m3 -> bf16
    // Threads r + 64 p (p = 0..3) convert KV row r of each tile from the
    // staging ring (row-major bytes) into the bf16 ring in the swizzled layouts
    // the MMAs read: latent chunk p, and for p < 2 half p of the RoPE dims.
    const int ct = tid - (2 + kSoftmaxWarps + kCeWarps) * 32;
    const int r = ct & (kTile - 1), part = ct / kTile;
    uint32_t g = 0;
    for (int idx = item_begin; idx < item_end; ++idx) {
      const WorkItem it = items[idx];
      const int nt = n_tiles_of(it);
      if (nt <= 0) continue;
      for (int t = 0; t < nt; ++t, ++g) {
        const int ss = g & 1;        // staging slot (2 deep)
        const int s = g % kStages;   // bf16 slot
        if (!wait_bar(c, STG_FULL0 + ss, (g >> 1) & 1)) goto done_conv;
        if (!wait_bar(c, KV_EMPTY0 + s, ((g / kStages) & 1) ^ 1)) goto done_conv;
        const unsigned char* src = sm + C::OFF_STG + ss * kStgBytes;
        unsigned char* dst = sm + OFF_KV + s * kStageBytes;
        {
          const int lc = part;
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
        if (part < 2) {  // RoPE: 16 of its 32 values -> two 16-byte units (64B swizzle)
          const int k = part;
          const uint4 b =
              *reinterpret_cast<const uint4*>(src + kLatChunks * kTile * 64 + r * 32 + 16 * k);
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
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&c.bars[KV_FULL0 + s]);
          mbar_arrive(&c.bars[STG_EMPTY0 + ss]);
        }
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

template <bool kFp8, bool kSparse, bool kF8 = false>
cudaError_t setup_one(int sm_count, int* n_pairs) {
  using C = Cfg<kFp8, kSparse, kF8>;
  auto kernel = decode_sm103_kernel<kFp8, kSparse, kF8>;
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sm_count / 2), 1, 1);
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
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

// Launch as a programmatic dependent of the previous kernel in the stream.
template <bool kFp8, bool kSparse, bool kF8 = false>
cudaError_t launch_pdl(int grid, cudaStream_t stream, const Problem& p, const Layout& lay, char* ws,
                       const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c) {
  using C = Cfg<kFp8, kSparse, kF8>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_sm103_kernel<kFp8, kSparse, kF8>, p, lay, ws, a, b, c);
}

}  // namespace

cudaError_t decode_sm103_setup(int kv_dtype, int sparse, int f8_mma, int sm_count, int* n_pairs) {
  if (kv_dtype == 1 && f8_mma && !sparse) return setup_one<false, false, true>(sm_count, n_pairs);
  if (kv_dtype == 1)
    return sparse ? setup_one<true, true>(sm_count, n_pairs)
                  : setup_one<true, false>(sm_count, n_pairs);
  return sparse ? setup_one<false, true>(sm_count, n_pairs)
                : setup_one<false, false>(sm_count, n_pairs);
}

cudaError_t launch_decode_sm103(const Problem& p, const Layout& lay, void* ws,
                                cudaStream_t stream) {
  CUtensorMap tm_q_rope, tm_kv, tm_kv_rope;
  const uint64_t q_rows = std::max<uint64_t>(1, (uint64_t)p.total_q * p.num_heads);
  const uint64_t kv_rows = (uint64_t)p.num_pages * p.page_size;
  // sparse top-k gathers single rows (four per copy); otherwise pages are copied
  const uint32_t box_rows = p.sparse_k > 0 ? 1u : (uint32_t)p.page_size;
  // (an e4m3 query, and any query on the FP8 MMA path, is read with plain
  // loads; its map is encoded but unused)
  if (!(p.q_fp8 ? encode_2d(&tm_q_rope, p.query, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, q_rows, 32,
                            kRows, CU_TENSOR_MAP_SWIZZLE_NONE)
                : encode_2d(&tm_q_rope, p.query, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, q_rows, 32,
                            kRows, CU_TENSOR_MAP_SWIZZLE_64B)))
    return cudaErrorInvalidValue;
  if (p.f8_mma) {
    // e4m3 rows straight into the ring for the FP8 MMAs: 128-dim latent chunks
    // (128B swizzle) and the 32 RoPE dims (32B swizzle)
    if (p.kv_dtype != 1 || p.sparse_k > 0 ||
        !encode_2d(&tm_kv, p.kv_cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kv_rows, 128, box_rows,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tm_kv_rope, p.kv_cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kv_rows, 32,
                   box_rows, CU_TENSOR_MAP_SWIZZLE_32B))
      return cudaErrorInvalidValue;
    return launch_pdl<false, false, true>(lay.n_ctas, stream, p, lay, static_cast<char*>(ws),
                                          tm_q_rope, tm_kv, tm_kv_rope);
  }
  if (p.kv_dtype == 1) {
    // e4m3 bytes land row-major in the staging ring; the converter swizzles
    if (!encode_2d(&tm_kv, p.kv_cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kv_rows, 64, box_rows,
                   CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&tm_kv_rope, p.kv_cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kv_rows, 32,
                   box_rows, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
    return p.sparse_k > 0 ? launch_pdl<true, true>(lay.n_ctas, stream, p, lay,
                                                   static_cast<char*>(ws), tm_q_rope, tm_kv,
                                                   tm_kv_rope)
                          : launch_pdl<true, false>(lay.n_ctas, stream, p, lay,
                                                    static_cast<char*>(ws), tm_q_rope, tm_kv,
                                                    tm_kv_rope);
  }
  if (!encode_2d(&tm_kv, p.kv_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kv_rows, 64, box_rows,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tm_kv_rope, p.kv_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kv_rows, 32,
                 box_rows, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  return p.sparse_k > 0 ? launch_pdl<false, true>(lay.n_ctas, stream, p, lay,
                                                  static_cast<char*>(ws), tm_q_rope, tm_kv,
                                                  tm_kv_rope)
                        : launch_pdl<false, false>(lay.n_ctas, stream, p, lay,
                                                   static_cast<char*>(ws), tm_q_rope, tm_kv,
                                                   tm_kv_rope);
}

}  // namespace mla
