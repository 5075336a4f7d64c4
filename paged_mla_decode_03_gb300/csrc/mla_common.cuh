// Shared definitions of the paged MLA decode kernels: the problem record
// passed by value to every kernel, the split-KV work items, and the layout of
// the caller-owned workspace.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mla {

constexpr int kQkDim = 576;       // 512 latent + 64 RoPE
constexpr int kVDim = 512;        // V = the latent part of each cache row
constexpr int kKvTile = 64;       // KV rows per pipeline tile

// Problem record: static plan parameters plus the per-run pointers/scales.
// Largest partitioner scratch kept in shared memory (else in the workspace).
constexpr size_t kPartitionSmemMax = 160 * 1024;

// Status word bits (workspace header word kHdrStatus).
constexpr int kStatusSeqLen = 1, kStatusQLen = 2, kStatusCausal = 4, kStatusCapacity = 8,
              kStatusPage = 16, kStatusTimeout = 32, kStatusScale = 64;

struct Problem {
  int batch, num_heads, max_q, max_seq_len, page_size, max_pages;
  int packed, kv_dtype, causal, return_lse;
  int q_fp8;                     // 1: query is e4m3
  int f8_mma;                    // 1: e4m3 cache on FP8 MMAs (else widened to bf16)
  int cp_world, cp_rank;         // decode-context parallelism (cp_world 1: off)
  int sparse_k;                  // > 0: sparse top-k, k listed KV positions per token
  long long num_pages, total_q;  // total_q: rows of the query tensor (tokens)
  float bmm1_scale, bmm2_scale;
  const float* bmm1_dev;         // non-null: read bmm1 from device memory at run time
  const float* bmm2_dev;         // non-null: read bmm2 from device memory at run time
  const void* query;             // bf16 or e4m3 [tokens, H, 576]
  const void* kv_cache;          // bf16 or e4m3 [num_pages, page_size, 576]
  const int* block_tables;       // [B, max_pages]
  const int* seq_lens;           // [B]
  const int* qo_indptr;          // [B + 1] or nullptr
  const int* seq_lens_global;    // [B] global KV lengths (causal, cp_world > 1) or nullptr
  const int* sparse_idx;         // [tokens, sparse_k] logical KV positions, or nullptr
  void* out;                     // bf16 [tokens, H, 512]
  float* lse;                    // fp32 [tokens, H] or nullptr
};

// bmm1 of this run: the host value, or the device value when one was given.
// A negative or non-finite device value sets kStatusScale and reads as 0.
__device__ __forceinline__ float run_bmm1(const Problem& p, int* status) {
  if (!p.bmm1_dev) return p.bmm1_scale;
  const float v = *p.bmm1_dev;
  if (v >= 0.f && v <= 3.0e38f) return v;
  atomicOr(status, kStatusScale);
  return 0.f;
}
__device__ __forceinline__ float run_bmm2(const Problem& p) {
  return p.bmm2_dev ? *p.bmm2_dev : p.bmm2_scale;
}

// One unit of work of the decode kernel: query rows [R g, R g + R) of request
// b (R = Layout::rows_per_group, clipped to its q_len * H rows) against KV rows
// [kv_begin, kv_end).  Under sparse top-k selection R = H (one token, q_start
// + g) and [kv_begin, kv_end) indexes the token's position list.
// slot < 0: the item covers the whole KV range and writes `out` directly;
// otherwise it writes a normalised partial (bf16 O, fp32 natural-log LSE) into
// partial slot `slot` for the combine kernel.
struct WorkItem {
  int b, g, kv_begin, kv_end;
  int slot, q_len, seq_len, q_start;  // q_start: first token of request b; seq_len: its L
  int comb;                           // combine entry of a split group, else -1
  int mask_base;                      // causal bound of query row i: causal_last(mask_base, i, W)
};

// Last local KV row (inclusive) that query row qi of a request may see under
// causal masking, from the request's mask_base.  On one rank (W = 1)
// mask_base = L - q and the bound is L - q + qi (the bottom-right rule of the
// FlashInfer page "prims_ts_batch_decode_with_kv_cache_mla").  Under
// decode-context parallelism rank r of W holds global row g (g mod W == r)
// as local row g div W, and row qi sees the global rows g <= Lg - q + qi, so
// with mask_base = Lg - q - r the bound is floor((mask_base + qi) / W).
// A negative result means the row sees no local row.
__host__ __device__ inline int causal_last(int mask_base, int qi, int W) {
  const int x = mask_base + qi;
  return x >= 0 ? x / W : -((W - 1 - x) / W);
}

// One split (request, row group): partials live in slots first + k * stride.
struct CombineItem {
  int b, g, first_slot, stride;
  int n_chunks, q_len, q_start, pad;
};

// Header words at the start of the workspace.
enum HeaderWord {
  kHdrStatus = 0,     // contract-violation bits (see mla_decode_status_offset)
  kHdrNumItems = 1,
  kHdrWorkCounter = 2,     // reserved: zeroed by the partitioner, read by no kernel
  kHdrNumCombine = 3,
  kHdrChunkTiles = 4,      // the partition's total cost in units (a diagnostic)
  kHdrCombineCounter = 5,  // reserved: zeroed by the partitioner, read by no kernel
  kHdrWords = 64
};

// Byte layout of the workspace; computed on the host at plan time.
struct Layout {
  size_t items;          // WorkItem[max_items]
  size_t combine;        // CombineItem[max_combine]
  size_t worker_ranges;  // int[n_workers + 1]: worker w owns items [r[w], r[w+1])
  size_t req_scratch;    // int[4 * batch]: partitioner scratch
  size_t group_scratch;  // partitioner scratch per row group / item
  size_t scratch_bytes;  // bytes of the two scratch areas
  int scratch_in_smem;   // 1: the partitioner keeps its scratch in shared memory
  size_t part_o;         // split partials of O, see part_unit
  size_t part_lse;       // float[max_partials][rows_per_group]
  size_t comb_done;      // int[max_combine]: CTAs that finished a chunk of each split group
  size_t total;
  int max_items, max_combine, max_partials, max_groups;
  int n_workers;       // persistent workers (CTAs, or CTA pairs)
  int n_ctas;          // CTAs of the decode grid
  int rows_per_group;  // query rows per work item
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The partitioner's cost model: a row group costs kOverheadTiles + its KV
// tiles (the overhead is the query load and the epilogue, in tile units;
// measured ~3.2), and every busy worker gets at least kMinUnits units.
constexpr long long kOverheadTiles = 3;
constexpr long long kMinUnits = 4;

// The query split of the FP8 MMA path with a bf16 query (mla_qsplit.cu), one
// record of kQSplitUnits 16-byte units per (query row, CTA half): latent hi
// codes (units 0-15), latent lo codes (16-31), RoPE hi (32-33), RoPE lo
// (34-35), each in dim order, then the half's factor 2^-k (the float in the
// first word of unit 36).  The records follow the combine counters; the plans
// that use them size the workspace to hold one per (row, half) of their
// largest query.  (Kept out of Layout: the decode kernel measured 1.5% slower
// on the MTP workload with two more Layout fields, for no reason found.)
constexpr int kQSplitUnits = 37;
__host__ __device__ inline size_t q_split_offset(const Layout& lay) {
  return align_up(lay.comb_done + sizeof(int) * (size_t)(lay.max_combine > 1 ? lay.max_combine : 1),
                  256);
}

// Split partials of O (normalised by their own softmax sum): bf16, or fp32
// when kPartialBf16 is false.  A slot holds R rows x 512 dims as 32 chunks of
// 16 dims; chunk c of row q is kPartUnits 16-byte units, stored unit-major
// over the rows, [slot][c][unit][row], so the epilogue's threads (one row
// each) write consecutive 16-byte units.
constexpr bool kPartialBf16 = true;
constexpr int kPartUnits = kPartialBf16 ? 2 : 4;  // 16-byte units of a 16-dim chunk
constexpr size_t kPartBytesPerRow = 32 * kPartUnits * 16;
__host__ __device__ inline size_t part_unit(size_t slot, int R, int c, int u, int q) {
  return ((slot * 32 + (size_t)c) * kPartUnits + (size_t)u) * (size_t)R + (size_t)q;
}

}  // namespace mla
