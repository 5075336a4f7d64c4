// On-device split-KV work partitioner.
//
// Reads seq_lens / qo_indptr on the device (the problem statement of the
// FlashInfer page "prims_ts_batch_decode_with_kv_cache_mla" forbids
// device-to-host metadata reads on this path) and writes into the workspace
// (a) the list of work items of the decode kernel and, for every persistent
// worker, the contiguous range of items it owns, and (b) the list of split
// (request, row group) pairs the combine kernel merges.
//
// Cost model: a request with q query rows and H heads has G = ceil(q H / R)
// row groups of R rows; each group costs c0 + T units, T = ceil(L / 64) KV
// tiles plus a fixed overhead c0 (query load, epilogue).  Laying all groups
// end to end gives W units; with n' = min(n, W / kMinUnits) workers (a
// worker gets at least about one item's worth; the others stay idle), worker
// p owns units [floor(p W / n'), floor((p+1) W / n')).  A group that
// straddles a range boundary is cut at the corresponding tile and each piece
// becomes a separate item writing a partial; every other group is one item
// writing the output directly.  So workers are balanced to within one tile
// plus one overhead, and there are at most n + #groups items and n - 1 cut
// points.  Under sparse top-k selection a group is one token's H rows and its
// KV range is the token's list of k positions (T = ceil(k / 64)).  One CTA
// of 128-1024 threads; the range boundaries are tabulated in shared memory
// once, so cut points and owners are table lookups.
#include <algorithm>

#include "mla_common.cuh"
#include "sm100_ptx.cuh"

namespace mla {

namespace {

// One CTA of 128..1024 threads, sized by the launch from the plan's bounds
// (fewer warps make the block-wide steps cheaper on small problems).
constexpr int kMaxThreads = 1024;
// the cost model's kOverheadTiles and kMinUnits are in mla_common.cuh (the
// plan bounds its worker count with them)
constexpr int kBoundTable = 512;         // workers whose range boundaries are tabulated

struct Shared {
  long long warp_ll[32];
  int warp_i[32];
  int carry;
  long long carry_ll;
  long long bound[kBoundTable + 1];  // start unit of every worker's range (and W)
};

__device__ int block_or(int v, Shared& sh) {
  for (int o = 16; o > 0; o >>= 1) v |= __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) sh.warp_i[warp] = v;
  __syncthreads();
  int t = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t |= sh.warp_i[w];
  __syncthreads();
  return t;
}

__device__ int block_min(int v, Shared& sh) {
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) sh.warp_i[warp] = v;
  __syncthreads();
  int t = sh.warp_i[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) t = min(t, sh.warp_i[w]);
  __syncthreads();
  return t;
}

__device__ int block_max(int v, Shared& sh) {
  return -block_min(-v, sh);
}

// In-place exclusive prefix sum of data[0, n); returns the total.
template <typename T>
__device__ T block_exclusive_scan(T* data, int n, Shared& sh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  // every thread has read the previous scan's total (returned from carry_ll)
  // before it is reset
  __syncthreads();
  if (threadIdx.x == 0) sh.carry_ll = 0;
  __syncthreads();
  for (int base = 0; base < n; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const T v = i < n ? data[i] : T(0);
    T x = v;
    for (int o = 1; o < 32; o <<= 1) {
      const T y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) sh.warp_ll[warp] = (long long)x;
    __syncthreads();
    if (warp == 0) {
      long long w = lane < nw ? sh.warp_ll[lane] : 0;
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      sh.warp_ll[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const long long warp_excl = warp ? sh.warp_ll[warp - 1] : 0;
    const long long carry = sh.carry_ll;
    if (i < n) data[i] = (T)(carry + warp_excl + (long long)(x - v));
    __syncthreads();
    if (threadIdx.x == 0) sh.carry_ll = carry + sh.warp_ll[nw - 1];
    __syncthreads();
  }
  return (T)sh.carry_ll;
}

// Worker ranges.  The workers form `lanes` lanes of nl workers (leftover
// workers get empty ranges); lane k owns units [k WL, (k + 1) WL) and its
// worker i the units [k WL + floor(i WL / nl), k WL + floor((i + 1) WL / nl)).
// With one lane this is the plain split of [0, W) into n near-equal ranges.
struct Bounds {
  long long W, n, lanes, nl, WL;
  const long long* table;  // boundary(p) for p in [0, n], or nullptr
  // start unit of worker p's range (the arithmetic behind the table)
  __device__ long long boundary_of(long long p) const {
    if (p >= lanes * nl) return W;
    const long long k = p / nl, i = p - k * nl;
    return k * WL + (i * WL) / nl;
  }
  __device__ long long boundary(long long p) const { return table ? table[p] : boundary_of(p); }
  // first worker p whose range starts after unit x (0 <= x < W); boundaries
  // are nondecreasing in p and boundary(n) = W > x
  __device__ long long first_above(long long x) const {
    if (table) {
      long long lo = 0, hi = n;
      while (lo < hi) {
        const long long mid = (lo + hi) >> 1;
        if (table[mid] > x) hi = mid; else lo = mid + 1;
      }
      return lo;
    }
    const long long k = x / WL, r = x - k * WL;
    const long long i = ((r + 1) * nl + WL - 1) / WL;
    return i >= nl ? (k + 1) * nl : k * nl + i;
  }
  // worker that owns unit x (0 <= x < W): the largest p with boundary(p) <= x
  __device__ long long owner_of(long long x) const {
    return min(first_above(x) - 1, n - 1);
  }
};

// Tile cut position of range boundary p inside a group starting at unit S.
__device__ __forceinline__ int cut_tile(const Bounds& bd, long long p, long long S, int T) {
  const long long t = bd.boundary(p) - S - kOverheadTiles;
  return (int)min(max(t, 0LL), (long long)T);
}

}  // namespace

__global__ void __launch_bounds__(kMaxThreads, 1)
partition_kernel(Problem p, Layout lay, char* __restrict__ ws) {
  __shared__ Shared sh;
  // the decode kernel may set up its barriers and TMEM meanwhile; it reads
  // nothing written here before its grid-dependency wait
  ptx::pdl_launch_dependents();
  int* hdr = reinterpret_cast<int*>(ws);
  WorkItem* items = reinterpret_cast<WorkItem*>(ws + lay.items);
  CombineItem* comb = reinterpret_cast<CombineItem*>(ws + lay.combine);
  int* worker_begin = reinterpret_cast<int*>(ws + lay.worker_ranges);
  const int B = p.batch;
  const int R = lay.rows_per_group;
  const int H = p.num_heads;
  const bool sparse = p.sparse_k > 0;
  // KV rows a group of request b walks: its cache rows, or the token's list
  auto kv_rows = [&](int L) { return sparse ? p.sparse_k : L; };
  // per-request and per-group scratch: in shared memory when it fits (no
  // memory round trip between the phases below), else in the workspace
  extern __shared__ __align__(16) unsigned char scratch_smem[];
  char* req_base = lay.scratch_in_smem ? reinterpret_cast<char*>(scratch_smem) : ws + lay.req_scratch;
  char* grp_base = lay.scratch_in_smem
                       ? reinterpret_cast<char*>(scratch_smem) + (lay.group_scratch - lay.req_scratch)
                       : ws + lay.group_scratch;
  int* r_qlen = reinterpret_cast<int*>(req_base);
  int* r_qstart = r_qlen + B;
  int* r_len = r_qstart + B;
  int* r_gbase = r_len + B;  // first group index of the request
  int* r_mbase = r_gbase + B;  // causal mask base of the request (see causal_last)
  int* r_empty = r_mbase + B;  // empty combine entries of the request (DCP, no local rows)
  // per-group scratch
  long long* g_start = reinterpret_cast<long long*>(grp_base);  // unit offset
  int* g_items = reinterpret_cast<int*>(g_start + lay.max_groups);              // -> item base
  int* g_req = g_items + lay.max_groups;
  int* g_nch = g_req + lay.max_groups;
  int* g_slot = g_nch + lay.max_groups;  // partial-slot base
  int* g_comb = g_slot + lay.max_groups;  // combine-entry base
  int* g_k = g_comb + lay.max_groups;     // row group within its request
  int* it_owner = g_k + lay.max_groups;   // per item: owning worker

  // 1. Per-request lengths, clamped so that nothing downstream leaves the
  //    caller's buffers; contract violations are flagged in the status word.
  int status = 0;
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    int q, qs;
    if (p.packed) {
      int lo = p.qo_indptr[b], hi = p.qo_indptr[b + 1];
      const int tq = (int)p.total_q;
      if (lo < 0 || hi > tq || hi - lo < 1 || hi - lo > p.max_q) status |= kStatusQLen;
      lo = min(max(lo, 0), tq);
      hi = min(max(hi, lo), tq);
      q = min(hi - lo, p.max_q);
      qs = lo;
    } else {
      q = p.max_q;
      qs = b * p.max_q;
    }
    int L = p.seq_lens[b];
    int mbase;
    if (p.cp_world > 1) {
      // decode-context parallelism: a rank may hold no row of a request
      if (L < 0 || L > p.max_seq_len) status |= kStatusSeqLen;
      L = min(max(L, 0), p.max_seq_len);
      mbase = 0;
      if (p.causal) {
        const int Lg = p.seq_lens_global[b];
        if (Lg < 1) status |= kStatusSeqLen;
        if (q > Lg) status |= kStatusCausal;
        mbase = Lg - q - p.cp_rank;
      }
    } else {
      if (L < 1 || L > p.max_seq_len) status |= kStatusSeqLen;
      L = min(max(L, 0), p.max_seq_len);
      if (p.causal && !sparse && q > L) status |= kStatusCausal;
      mbase = L - q;
    }
    r_qlen[b] = q;
    r_qstart[b] = qs;
    r_len[b] = L;
    r_mbase[b] = mbase;
    r_gbase[b] = (L > 0) ? (q * H + R - 1) / R : 0;
    // a DCP rank with no row of the request still owes its rows O = 0 and
    // lse = -inf (the empty sum); the combine kernel writes them
    r_empty[b] = (p.cp_world > 1 && L == 0) ? (q * H + R - 1) / R : 0;
  }
  status = __syncthreads_or(status) ? block_or(status, sh) : 0;
  // do all requests that have row groups have the same number of them?
  int g_min = 1 << 30, g_max = 0;
  for (int b = threadIdx.x; b < B; b += blockDim.x)
    if (r_gbase[b] > 0) {
      g_min = min(g_min, r_gbase[b]);
      g_max = max(g_max, r_gbase[b]);
    }
  g_min = block_min(g_min, sh);
  g_max = block_max(g_max, sh);
  __syncthreads();
  int n_groups = block_exclusive_scan(r_gbase, B, sh);
  if (n_groups > lay.max_groups) {  // unreachable within the contract
    status |= kStatusCapacity;
    n_groups = 0;
  }

  // 2. Groups with their unit costs.  When every request that has row
  //    groups has the same number G >= 2 of them (a uniform q_len) and the
  //    workers can be split into G lanes of at least two, group k of every
  //    request goes to lane k (order lane-major), so lane k's worker i walks
  //    the same KV ranges as every other lane's worker i at the same time: a
  //    page comes from DRAM once and from L2 for the other lanes.  Otherwise
  //    groups are laid out in request order on one lane.
  const long long n = lay.n_workers;
  const int G = g_max;
  // groups' total cost first (lane order does not change it), then the
  // number of busy workers and the lanes
  long long W_total = 0;
  for (int b = threadIdx.x; b < B && n_groups > 0; b += blockDim.x) {
    const int gb = r_gbase[b];  // scanned: first group of request b
    const int ge = (b + 1 < B) ? r_gbase[b + 1] : n_groups;
    W_total += (long long)(ge - gb) * (kOverheadTiles + (kv_rows(r_len[b]) + kKvTile - 1) / kKvTile);
  }
  __syncthreads();
  if (threadIdx.x == 0) sh.carry_ll = 0;
  __syncthreads();
  // summed within each warp first, then one add per warp: contended 64-bit
  // shared atomics serialise (one per request cost a few microseconds at B = 64)
  for (int o = 16; o > 0; o >>= 1) W_total += __shfl_xor_sync(0xffffffffu, W_total, o);
  if ((threadIdx.x & 31) == 0 && W_total != 0)
    atomicAdd(reinterpret_cast<unsigned long long*>(&sh.carry_ll), (unsigned long long)W_total);
  __syncthreads();
  W_total = sh.carry_ll;
  const long long n_eff = max(1LL, min(n, W_total / kMinUnits));
  const int lanes = (g_min == g_max && G >= 2 && n_eff / G >= 2) ? G : 1;
  const int n_req_groups = lanes > 1 ? n_groups / G : 0;  // requests that have groups
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int gb = r_gbase[b];
    const int ge = (b + 1 < B) ? r_gbase[b + 1] : n_groups;
    const int T = (kv_rows(r_len[b]) + kKvTile - 1) / kKvTile;
    for (int g = gb; g < ge && g < n_groups; ++g) {
      const int k = g - gb;
      const int slot = lanes > 1 ? k * n_req_groups + gb / G : g;
      g_req[slot] = b;
      g_k[slot] = k;
      g_start[slot] = kOverheadTiles + T;  // cost; scanned into the start unit below
    }
  }
  __syncthreads();
  const long long W = block_exclusive_scan(g_start, n_groups, sh);
  Bounds bd;
  bd.W = W;
  bd.n = n;
  bd.lanes = lanes;
  bd.nl = n_eff / lanes;  // busy workers per lane; the rest get empty ranges
  bd.WL = W / lanes;      // every lane has the same cost
  bd.table = nullptr;
  if (n <= kBoundTable) {
    for (long long q = threadIdx.x; q <= n; q += blockDim.x) sh.bound[q] = bd.boundary_of(q);
    __syncthreads();
    bd.table = sh.bound;
  }

  // 3. Cut points inside each group -> chunk counts.
  for (int g = threadIdx.x; g < n_groups; g += blockDim.x) {
    const int b = g_req[g];
    const int T = (kv_rows(r_len[b]) + kKvTile - 1) / kKvTile;
    const long long S = g_start[g], c = kOverheadTiles + T;
    int nch = 1;
    if (W > 0) {
      const long long p_lo = bd.first_above(S);           // boundaries after the group start
      const long long p_hi = bd.first_above(S + c - 1) - 1;  // ... and before its end
      int prev = 0;
      for (long long q = max(p_lo, 1LL); q <= min(p_hi, n - 1); ++q) {
        const int t = cut_tile(bd, q, S, T);
        if (t > prev && t < T) {
          ++nch;
          prev = t;
        }
      }
    }
    g_nch[g] = nch;
    g_items[g] = nch;
    g_slot[g] = nch > 1 ? nch : 0;
    g_comb[g] = nch > 1 ? 1 : 0;
  }
  __syncthreads();
  int n_items = block_exclusive_scan(g_items, n_groups, sh);
  const int n_partials = block_exclusive_scan(g_slot, n_groups, sh);
  const int n_combine = block_exclusive_scan(g_comb, n_groups, sh);
  if (n_items > lay.max_items || n_partials > lay.max_partials || n_combine > lay.max_combine) {
    status |= kStatusCapacity;  // unreachable within the contract
    n_items = 0;
  }

  // 4. Items (group order, then chunk order) and combine entries.
  if (n_items > 0) {
    for (int g = threadIdx.x; g < n_groups; g += blockDim.x) {
      const int b = g_req[g];
      const int L = r_len[b];
      const int KV = kv_rows(L);
      const int T = (KV + kKvTile - 1) / kKvTile;
      const long long S = g_start[g], c = kOverheadTiles + T;
      const int nch = g_nch[g];
      const int g_local = g_k[g];
      int k = 0, prev = 0;
      // an item belongs to the worker whose range holds its first KV tile
      long long start_unit = S + kOverheadTiles;
      auto emit = [&](int t0, int t1, long long unit) {
        WorkItem it;
        it.b = b;
        it.g = g_local;
        it.kv_begin = t0 * kKvTile;
        it.kv_end = min(KV, t1 * kKvTile);
        it.slot = nch > 1 ? g_slot[g] + k : -1;
        it.comb = nch > 1 ? g_comb[g] : -1;
        it.q_len = r_qlen[b];
        it.seq_len = L;
        it.q_start = r_qstart[b];
        it.mask_base = r_mbase[b];
        items[g_items[g] + k] = it;
        it_owner[g_items[g] + k] = (int)bd.owner_of(unit);
        ++k;
      };
      if (nch > 1 && W > 0) {
        const long long p_lo = bd.first_above(S);
        const long long p_hi = bd.first_above(S + c - 1) - 1;
        for (long long q = max(p_lo, 1LL); q <= min(p_hi, n - 1); ++q) {
          const int t = cut_tile(bd, q, S, T);
          if (t > prev && t < T) {
            emit(prev, t, start_unit);
            start_unit = S + kOverheadTiles + t;
            prev = t;
          }
        }
      }
      emit(prev, T, start_unit);
      if (nch > 1) {
        CombineItem ci;
        ci.b = b;
        ci.g = g_local;
        ci.first_slot = g_slot[g];
        ci.stride = 1;
        ci.n_chunks = nch;
        ci.q_len = r_qlen[b];
        ci.q_start = r_qstart[b];
        ci.pad = 0;
        comb[g_comb[g]] = ci;
      }
    }
  }
  // Empty entries after the split ones: every row group of a request this
  // DCP rank holds no row of (no chunk: the combine writes zeros and -inf).
  const int comb_base = n_items > 0 ? n_combine : 0;
  int n_empty = 0;
  if (p.cp_world > 1) {
    n_empty = block_exclusive_scan(r_empty, B, sh);
    if (comb_base + n_empty > lay.max_combine) {  // unreachable within the contract
      status |= kStatusCapacity;
      n_empty = 0;
    } else {
      for (int b = threadIdx.x; b < B; b += blockDim.x) {
        if (r_len[b] > 0) continue;
        const int cnt = (r_qlen[b] * H + R - 1) / R;
        for (int k = 0; k < cnt; ++k) {
          CombineItem ci;
          ci.b = b;
          ci.g = k;
          ci.first_slot = 0;
          ci.stride = 1;
          ci.n_chunks = 0;
          ci.q_len = r_qlen[b];
          ci.q_start = r_qstart[b];
          ci.pad = 0;
          comb[comb_base + r_empty[b] + k] = ci;
        }
      }
    }
  }
  // completion counters of the combine entries (bumped by the decode kernel)
  int* comb_done = reinterpret_cast<int*>(ws + lay.comb_done);
  for (int e = threadIdx.x; e < lay.max_combine; e += blockDim.x) comb_done[e] = 0;
  __syncthreads();
  // 5. Worker ranges: worker w owns items [begin[w], begin[w + 1]).
  for (int w = threadIdx.x; w <= (int)n; w += blockDim.x) {
    int lo = 0, hi = n_items;  // first item with owner >= w
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (it_owner[mid] < w) lo = mid + 1; else hi = mid;
    }
    worker_begin[w] = (w == (int)n) ? n_items : lo;
  }
  if (threadIdx.x == 0) {
    hdr[kHdrStatus] = status;
    hdr[kHdrNumItems] = n_items;
    hdr[kHdrWorkCounter] = 0;
    hdr[kHdrNumCombine] = comb_base + n_empty;
    hdr[kHdrChunkTiles] = (int)min(W, (long long)1 << 30);
    hdr[kHdrCombineCounter] = 0;
  }
}

// ---------------------------------------------------------------------------
// The same partition computed by one warp.  The block kernel above is a chain
// of block-wide steps, each several barriers deep; here every step is a warp
// scan or reduction over per-lane contiguous runs, ordered by __syncwarp
// alone, and the work list it leaves is the block kernel's, bit for bit (same
// cost model, same Bounds arithmetic, same item order).  Every control path
// that reaches a shuffle is taken by all 32 lanes.
//
// The tables hold up to kWarpMaxReq requests and kWarpMaxGroups row groups,
// but the launch picks this form only while every lane holds at most one
// request and one group (kWarpPickReq, kWarpPickGroups): measured per call on
// GB300, it ends 2 us sooner than the block kernel with one group a lane (B =
// 2) and 2-10 us later with 2-4 groups or requests a lane, whose runs are
// walked serially.
constexpr int kWarpMaxReq = 512;
constexpr int kWarpMaxGroups = 512;
constexpr int kWarpPickReq = 32;
constexpr int kWarpPickGroups = 32;
// items <= groups + cut points, and cut points < workers <= kBoundTable
constexpr int kWarpMaxItems = kWarpMaxGroups + kBoundTable;

struct WarpShared {
  int q[kWarpMaxReq], qs[kWarpMaxReq], len[kWarpMaxReq], mbase[kWarpMaxReq], gbase[kWarpMaxReq];
  long long g_start[kWarpMaxGroups];
  int g_req[kWarpMaxGroups], g_k[kWarpMaxGroups], g_nch[kWarpMaxGroups];
  int g_item[kWarpMaxGroups], g_slot[kWarpMaxGroups], g_comb[kWarpMaxGroups];
  long long bound[kBoundTable + 1];
  int owner[kWarpMaxItems];
};

__host__ __device__ inline bool partition_warp_fits(const Problem& p, const Layout& lay) {
  return p.cp_world <= 1 && p.batch >= 0 && p.batch <= kWarpMaxReq &&
         lay.max_groups <= kWarpMaxGroups && lay.n_workers >= 1 && lay.n_workers <= kBoundTable;
}

// Whether the launch runs the single-warp form (see above).
__host__ __device__ inline bool partition_warp_picked(const Problem& p, const Layout& lay) {
  return partition_warp_fits(p, lay) && p.batch <= kWarpPickReq && lay.max_groups <= kWarpPickGroups;
}

namespace {

constexpr unsigned kFull = 0xffffffffu;

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}
__device__ __forceinline__ int warp_or(int v) {
  for (int o = 16; o > 0; o >>= 1) v |= __shfl_xor_sync(kFull, v, o);
  return v;
}
__device__ __forceinline__ int warp_min(int v) {
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(kFull, v, o));
  return v;
}
__device__ __forceinline__ int warp_max(int v) {
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(kFull, v, o));
  return v;
}
// Exclusive prefix of v over the lanes; *total receives the sum of all lanes.
template <typename T>
__device__ __forceinline__ T warp_excl_scan(T v, T* total) {
  const int lane = threadIdx.x & 31;
  T x = v;
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  *total = __shfl_sync(kFull, x, 31);
  return x - v;
}

// Lane `lane`'s contiguous run [lo, hi) of n elements.
struct Run {
  int lo, hi;
  __device__ Run(int n, int lane) {
    const int per = (n + 31) / 32;
    lo = min(n, lane * per);
    hi = min(n, lo + per);
  }
};

}  // namespace

__global__ void __launch_bounds__(32, 1)
partition_warp_kernel(Problem p, Layout lay, char* __restrict__ ws) {
  __shared__ WarpShared sh;
  ptx::pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  int* hdr = reinterpret_cast<int*>(ws);
  WorkItem* items = reinterpret_cast<WorkItem*>(ws + lay.items);
  CombineItem* comb = reinterpret_cast<CombineItem*>(ws + lay.combine);
  int* worker_begin = reinterpret_cast<int*>(ws + lay.worker_ranges);
  const int B = p.batch;
  const int R = lay.rows_per_group;
  const int H = p.num_heads;
  const bool sparse = p.sparse_k > 0;
  auto tiles_of = [&](int L) { return ((sparse ? p.sparse_k : L) + kKvTile - 1) / kKvTile; };

  // 1. Per-request lengths (clamped and flagged as in the block kernel) and
  //    the request's number of row groups, over the lane's run of requests.
  int status = 0, g_min = 1 << 30, g_max = 0, my_groups = 0;
  long long my_cost = 0;
  const Run rb(B, lane);
  for (int b = rb.lo; b < rb.hi; ++b) {
    int q, qs;
    if (p.packed) {
      int lo = p.qo_indptr[b], hi = p.qo_indptr[b + 1];
      const int tq = (int)p.total_q;
      if (lo < 0 || hi > tq || hi - lo < 1 || hi - lo > p.max_q) status |= kStatusQLen;
      lo = min(max(lo, 0), tq);
      hi = min(max(hi, lo), tq);
      q = min(hi - lo, p.max_q);
      qs = lo;
    } else {
      q = p.max_q;
      qs = b * p.max_q;
    }
    int L = p.seq_lens[b];
    if (L < 1 || L > p.max_seq_len) status |= kStatusSeqLen;
    L = min(max(L, 0), p.max_seq_len);
    if (p.causal && !sparse && q > L) status |= kStatusCausal;
    const int gc = (L > 0) ? (q * H + R - 1) / R : 0;
    sh.q[b] = q;
    sh.qs[b] = qs;
    sh.len[b] = L;
    sh.mbase[b] = L - q;
    sh.gbase[b] = gc;  // count; replaced by the first group index below
    if (gc > 0) {
      g_min = min(g_min, gc);
      g_max = max(g_max, gc);
    }
    my_groups += gc;
    my_cost += (long long)gc * (kOverheadTiles + tiles_of(L));
  }
  status = warp_or(status);
  g_min = warp_min(g_min);
  g_max = warp_max(g_max);
  int n_groups;
  {
    int run = warp_excl_scan(my_groups, &n_groups);
    for (int b = rb.lo; b < rb.hi; ++b) {
      const int c = sh.gbase[b];
      sh.gbase[b] = run;
      run += c;
    }
  }
  if (n_groups > lay.max_groups || n_groups > kWarpMaxGroups) {  // unreachable within the contract
    status |= kStatusCapacity;
    n_groups = 0;
  }
  const long long W_total = warp_sum(my_cost);
  __syncwarp();

  // 2. Groups with their unit costs, lane-major when the lanes of the block
  //    kernel apply (same rule).
  const long long n = lay.n_workers;
  const int G = g_max;
  const long long n_eff = max(1LL, min(n, (n_groups > 0 ? W_total : 0) / kMinUnits));
  const int lanes = (g_min == g_max && G >= 2 && n_eff / G >= 2) ? G : 1;
  const int n_req_groups = lanes > 1 ? n_groups / G : 0;
  for (int b = rb.lo; b < rb.hi; ++b) {
    const int gb = sh.gbase[b];
    const int ge = (b + 1 < B) ? sh.gbase[b + 1] : n_groups;
    const int T = tiles_of(sh.len[b]);
    for (int g = gb; g < ge && g < n_groups; ++g) {
      const int k = g - gb;
      const int slot = lanes > 1 ? k * n_req_groups + gb / G : g;
      if (slot < 0 || slot >= n_groups) continue;  // unreachable: slots are a permutation
      sh.g_req[slot] = b;
      sh.g_k[slot] = k;
      sh.g_start[slot] = kOverheadTiles + T;
    }
  }
  __syncwarp();
  const Run rg(n_groups, lane);
  long long W;
  {
    long long csum = 0;
    for (int g = rg.lo; g < rg.hi; ++g) csum += sh.g_start[g];
    long long run = warp_excl_scan(csum, &W);
    for (int g = rg.lo; g < rg.hi; ++g) {
      const long long c = sh.g_start[g];
      sh.g_start[g] = run;
      run += c;
    }
  }
  Bounds bd;
  bd.W = W;
  bd.n = n;
  bd.lanes = lanes;
  bd.nl = n_eff / lanes;
  bd.WL = W / lanes;
  bd.table = nullptr;
  for (long long q = lane; q <= n; q += 32) sh.bound[q] = bd.boundary_of(q);
  __syncwarp();
  bd.table = sh.bound;

  // 3. Cut points inside each group -> chunk counts, then the item, partial
  //    slot and combine entry bases of every group.
  int s_items = 0, s_slot = 0, s_comb = 0;
  for (int g = rg.lo; g < rg.hi; ++g) {
    const int T = tiles_of(sh.len[sh.g_req[g]]);
    const long long S = sh.g_start[g], c = kOverheadTiles + T;
    int nch = 1;
    if (W > 0) {
      const long long p_lo = bd.first_above(S);
      const long long p_hi = bd.first_above(S + c - 1) - 1;
      int prev = 0;
      for (long long q = max(p_lo, 1LL); q <= min(p_hi, n - 1); ++q) {
        const int t = cut_tile(bd, q, S, T);
        if (t > prev && t < T) {
          ++nch;
          prev = t;
        }
      }
    }
    sh.g_nch[g] = nch;
    s_items += nch;
    s_slot += nch > 1 ? nch : 0;
    s_comb += nch > 1 ? 1 : 0;
  }
  int n_items, n_partials, n_combine;
  {
    int r_items = warp_excl_scan(s_items, &n_items);
    int r_slot = warp_excl_scan(s_slot, &n_partials);
    int r_comb = warp_excl_scan(s_comb, &n_combine);
    for (int g = rg.lo; g < rg.hi; ++g) {
      const int nch = sh.g_nch[g];
      sh.g_item[g] = r_items;
      sh.g_slot[g] = r_slot;
      sh.g_comb[g] = r_comb;
      r_items += nch;
      r_slot += nch > 1 ? nch : 0;
      r_comb += nch > 1 ? 1 : 0;
    }
  }
  if (n_items > lay.max_items || n_partials > lay.max_partials || n_combine > lay.max_combine ||
      n_items > kWarpMaxItems) {
    status |= kStatusCapacity;  // unreachable within the contract
    n_items = 0;
  }

  // 4. Items (group order, then chunk order) and combine entries.
  if (n_items > 0) {
    for (int g = rg.lo; g < rg.hi; ++g) {
      const int b = sh.g_req[g];
      const int L = sh.len[b];
      const int KV = sparse ? p.sparse_k : L;
      const int T = tiles_of(L);
      const long long S = sh.g_start[g], c = kOverheadTiles + T;
      const int nch = sh.g_nch[g];
      int k = 0, prev = 0;
      long long start_unit = S + kOverheadTiles;
      auto emit = [&](int t0, int t1, long long unit) {
        const int idx = sh.g_item[g] + k;
        ++k;
        if (idx < 0 || idx >= n_items) return;  // unreachable: the scan places every item
        WorkItem it;
        it.b = b;
        it.g = sh.g_k[g];
        it.kv_begin = t0 * kKvTile;
        it.kv_end = min(KV, t1 * kKvTile);
        it.slot = nch > 1 ? sh.g_slot[g] + (k - 1) : -1;
        it.comb = nch > 1 ? sh.g_comb[g] : -1;
        it.q_len = sh.q[b];
        it.seq_len = L;
        it.q_start = sh.qs[b];
        it.mask_base = sh.mbase[b];
        items[idx] = it;
        sh.owner[idx] = (int)bd.owner_of(unit);
      };
      if (nch > 1 && W > 0) {
        const long long p_lo = bd.first_above(S);
        const long long p_hi = bd.first_above(S + c - 1) - 1;
        for (long long q = max(p_lo, 1LL); q <= min(p_hi, n - 1); ++q) {
          const int t = cut_tile(bd, q, S, T);
          if (t > prev && t < T) {
            emit(prev, t, start_unit);
            start_unit = S + kOverheadTiles + t;
            prev = t;
          }
        }
      }
      emit(prev, T, start_unit);
      if (nch > 1 && sh.g_comb[g] < n_combine) {
        CombineItem ci;
        ci.b = b;
        ci.g = sh.g_k[g];
        ci.first_slot = sh.g_slot[g];
        ci.stride = 1;
        ci.n_chunks = nch;
        ci.q_len = sh.q[b];
        ci.q_start = sh.qs[b];
        ci.pad = 0;
        comb[sh.g_comb[g]] = ci;
      }
    }
  }
  int* comb_done = reinterpret_cast<int*>(ws + lay.comb_done);
  for (int e = lane; e < lay.max_combine; e += 32) comb_done[e] = 0;
  __syncwarp();
  // 5. Worker ranges: worker w owns items [begin[w], begin[w + 1]).
  for (int w = lane; w <= (int)n; w += 32) {
    int lo = 0, hi = n_items;  // first item with owner >= w
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (sh.owner[mid] < w) lo = mid + 1; else hi = mid;
    }
    worker_begin[w] = (w == (int)n) ? n_items : lo;
  }
  if (lane == 0) {
    hdr[kHdrStatus] = status;
    hdr[kHdrNumItems] = n_items;
    hdr[kHdrWorkCounter] = 0;
    hdr[kHdrNumCombine] = n_items > 0 ? n_combine : 0;
    hdr[kHdrChunkTiles] = (int)min(W, (long long)1 << 30);
    hdr[kHdrCombineCounter] = 0;
  }
}

cudaError_t launch_partition(const Problem& p, const Layout& lay, void* ws, cudaStream_t stream) {
  const size_t smem = lay.scratch_in_smem ? lay.scratch_bytes : 0;
  long long need = std::max<long long>(std::max<long long>(p.batch, lay.max_groups),
                                       (long long)lay.n_workers + 1);
  const int threads = (int)std::min<long long>(kMaxThreads,
                                                std::max<long long>(128, (need + 31) / 32 * 32));
  if (partition_warp_picked(p, lay))
    partition_warp_kernel<<<1, 32, 0, stream>>>(p, lay, static_cast<char*>(ws));
  else
    partition_kernel<<<1, threads, smem, stream>>>(p, lay, static_cast<char*>(ws));
  return cudaGetLastError();
}

cudaError_t partition_setup() {
  return cudaFuncSetAttribute(partition_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kPartitionSmemMax);
}

}  // namespace mla
