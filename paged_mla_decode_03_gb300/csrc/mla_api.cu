// C ABI of the paged MLA decode library (declared in include/mla_decode.h).
//
// mla_decode_plan sizes the workspace from the static parameters (the
// problem statement's "semantic key": head count, page size, the static
// q_len / KV-length / total_q bounds) and the device's SM count.
// mla_decode_run checks what the host can check and enqueues three kernels
// on the caller's stream: the split-KV partitioner, the decode kernel and the
// combine kernel, with the query split between the first two on the FP8 MMA
// path with a bf16 query.  Grid sizes depend only on plan-time values, and nothing
// here allocates, copies or synchronises, so a run can be captured in a CUDA
// graph and replayed with new seq_lens / qo_indptr values.
#include <algorithm>
#include <new>

#include "../../include/mla_decode.h"
#include "mla_common.cuh"

namespace mla {
cudaError_t launch_partition(const Problem& p, const Layout& lay, void* ws, cudaStream_t stream);
cudaError_t partition_setup();
cudaError_t launch_combine(const Problem& p, const Layout& lay, void* ws, int grid,
                           cudaStream_t stream);
cudaError_t decode_sm103_setup(int kv_dtype, int sparse, int f8_mma, int sm_count, int* n_pairs);
cudaError_t launch_merge_states(const void* o_parts, const float* lse_parts, int n, long long rows,
                                float scale, void* out, float* lse_out, cudaStream_t stream);
cudaError_t launch_qsplit(const Problem& p, const Layout& lay, void* ws, int sm_count,
                          cudaStream_t stream);
cudaError_t launch_decode_sm103(const Problem& p, const Layout& lay, void* ws,
                                cudaStream_t stream);
}  // namespace mla

struct mla_plan_s {
  mla_decode_params prm;
  mla::Layout lay;
  int sm_count;
  int combine_grid;
  // mla_decode_run_host copies the query on this stream while the
  // partitioner runs (created with the plan, on its device)
  cudaStream_t side_stream = nullptr;
  ~mla_plan_s() {
    if (side_stream) cudaStreamDestroy(side_stream);
  }
};

namespace {

constexpr size_t kHeaderBytes = sizeof(int) * mla::kHdrWords;

bool supported_heads(int h) { return h == 16 || h == 32 || h == 64 || h == 128; }

// An e4m3 cache runs on the FP8 MMAs unless widening was asked for (sparse
// top-k always widens).
bool uses_f8_mma(const mla_decode_params& p) {
  return p.kv_dtype == MLA_KV_FP8_E4M3 && p.sparse_top_k == 0 && p.e4m3_widen == 0;
}

// the FP8 MMA path with a bf16 query: the query is split before the decode
bool uses_q_split(const mla_decode_params& p) {
  return uses_f8_mma(p) && p.q_dtype == MLA_Q_BF16;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

int make_layout(const mla_decode_params& prm, int n_workers, int n_ctas, int rows_per_group,
                mla::Layout* lay) {
  using namespace mla;
  const long long B = prm.batch;
  const long long R = rows_per_group;
  const long long g_max = ceil_div((long long)prm.max_seq_len_q * prm.num_heads, R);
  long long groups = B * g_max;
  if (prm.packed) groups = std::min(groups, B + ceil_div(prm.max_total_q * prm.num_heads, R));
  groups = std::max(groups, 1LL);
  // each range boundary between two workers cuts at most one group
  const long long max_items = groups + n_workers;
  if (max_items > (1LL << 30)) return MLA_ERR_UNSUPPORTED;
  lay->rows_per_group = rows_per_group;
  lay->n_workers = n_workers;
  lay->n_ctas = n_ctas;
  lay->max_groups = (int)groups;
  lay->max_items = (int)max_items;
  // split groups (at most one per worker boundary), plus, under decode-context
  // parallelism, one empty entry per row group of a request the rank holds no
  // row of: never more than one entry per group
  lay->max_combine =
      (int)(prm.cp_world > 1 ? groups : std::min(groups, (long long)n_workers));
  lay->max_partials = (int)std::min(max_items, 2LL * n_workers);
  size_t off = kHeaderBytes;
  lay->items = off;
  off = align_up(off + sizeof(WorkItem) * lay->max_items, 256);
  lay->combine = off;
  off = align_up(off + sizeof(CombineItem) * lay->max_combine, 256);
  lay->worker_ranges = off;
  off = align_up(off + sizeof(int) * (n_workers + 1), 256);
  lay->req_scratch = off;
  const size_t req_bytes = align_up(sizeof(int) * 6 * std::max(B, 1LL), 256);
  off += req_bytes;
  lay->group_scratch = off;
  const size_t grp_bytes = align_up(sizeof(long long) * lay->max_groups +
                                        sizeof(int) * 6 * lay->max_groups +
                                        sizeof(int) * lay->max_items,
                                    256);
  off += grp_bytes;
  lay->scratch_bytes = req_bytes + grp_bytes;
  lay->scratch_in_smem = lay->scratch_bytes <= kPartitionSmemMax ? 1 : 0;
  lay->part_o = off;
  off = align_up(off + kPartBytesPerRow * R * (size_t)lay->max_partials, 256);
  lay->part_lse = off;
  off = align_up(off + sizeof(float) * R * (size_t)lay->max_partials, 256);
  lay->comb_done = off;
  off = align_up(off + sizeof(int) * (size_t)std::max(lay->max_combine, 1), 256);
  // the FP8 MMA path (e4m3 cache, dense, not widened) with a bf16 query: the
  // query's e4m3 parts, split once per call before the decode (q_split_offset)
  if (prm.kv_dtype == MLA_KV_FP8_E4M3 && prm.sparse_top_k == 0 && prm.e4m3_widen == 0 &&
      prm.q_dtype == MLA_Q_BF16) {
    const long long tokens = prm.packed ? prm.max_total_q : B * prm.max_seq_len_q;
    const size_t halves = 2 * (size_t)std::max(tokens, 1LL) * (size_t)prm.num_heads;
    off = align_up(off + halves * kQSplitUnits * 16, 256);
  }
  lay->total = off;
  return MLA_OK;
}

}  // namespace

extern "C" {

int mla_decode_plan(const mla_decode_params* params, mla_plan_t** plan, size_t* workspace_bytes) {
  if (!params || !plan || !workspace_bytes) return MLA_ERR_INVALID_ARG;
  *plan = nullptr;
  const mla_decode_params& p = *params;
  if (p.batch < 0 || p.max_seq_len_q < 1 || p.max_seq_len < 1 || p.max_pages_per_req < 1 ||
      p.num_pages < 1 || p.device < 0)
    return MLA_ERR_INVALID_ARG;
  if (p.packed != 0 && p.packed != 1) return MLA_ERR_INVALID_ARG;
  if (p.packed && p.max_total_q < 0) return MLA_ERR_INVALID_ARG;
  if (p.kv_dtype != MLA_KV_BF16 && p.kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_INVALID_ARG;
  if (p.q_dtype != MLA_Q_BF16 && p.q_dtype != MLA_Q_FP8_E4M3) return MLA_ERR_INVALID_ARG;
  if (p.mask != MLA_MASK_CAUSAL && p.mask != MLA_MASK_DENSE) return MLA_ERR_INVALID_ARG;
  if (p.cp_world < 0 || (p.cp_world <= 1 && p.cp_rank != 0) ||
      (p.cp_world > 1 && (p.cp_rank < 0 || p.cp_rank >= p.cp_world)))
    return MLA_ERR_INVALID_ARG;
  if (p.sparse_top_k < 0 || p.sparse_top_k > (1 << 24) || (p.sparse_top_k > 0 && p.cp_world > 1))
    return MLA_ERR_INVALID_ARG;
  if (!supported_heads(p.num_heads)) return MLA_ERR_UNSUPPORTED;
  if (p.page_size != 32 && p.page_size != 64) return MLA_ERR_UNSUPPORTED;
  // cache rows are addressed with 32-bit row coordinates
  if (p.num_pages > (1LL << 31) / p.page_size) return MLA_ERR_UNSUPPORTED;
  if ((long long)p.max_pages_per_req * p.page_size < p.max_seq_len) return MLA_ERR_INVALID_ARG;
  if (!p.packed && (long long)p.batch * p.max_seq_len_q > (1LL << 31) / 128)
    return MLA_ERR_UNSUPPORTED;

  int dev_count = 0;
  if (cudaGetDeviceCount(&dev_count) != cudaSuccess || p.device >= dev_count) return MLA_ERR_CUDA;
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaSetDevice(p.device) != cudaSuccess) return MLA_ERR_CUDA;
  int sms = 0, n_pairs = 0;
  cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p.device);
  if (e == cudaSuccess)
    e = mla::decode_sm103_setup(p.kv_dtype, p.sparse_top_k > 0, uses_f8_mma(p), sms, &n_pairs);
  if (e == cudaSuccess) e = mla::partition_setup();
  cudaStream_t side = nullptr;
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&side, cudaStreamNonBlocking);
  cudaSetDevice(prev);
  if (e != cudaSuccess || sms <= 0) {
    if (side) cudaStreamDestroy(side);
    return MLA_ERR_CUDA;
  }

  mla_plan_s* pl = new (std::nothrow) mla_plan_s;
  if (!pl) {
    cudaStreamDestroy(side);
    return MLA_ERR_INVALID_ARG;
  }
  pl->side_stream = side;
  pl->prm = p;
  pl->sm_count = sms;
  // one work item = 128 query rows on one CTA pair; under sparse top-k one
  // token's H rows (its own position list)
  const int rows_per_group = p.sparse_top_k > 0 ? p.num_heads : 128;
  // No run of this plan keeps more workers busy than its largest possible
  // work allows (the partitioner gives a busy worker at least kMinUnits units
  // of kOverheadTiles + tiles per row group), so a small plan launches a
  // smaller grid; the work list is the same as with every pair.
  {
    const long long g_max = ceil_div((long long)p.max_seq_len_q * p.num_heads, rows_per_group);
    long long groups = (long long)p.batch * g_max;
    if (p.packed)
      groups = std::min(groups, (long long)p.batch +
                                    ceil_div(p.max_total_q * p.num_heads, rows_per_group));
    const long long kv_rows = p.sparse_top_k > 0 ? p.sparse_top_k : p.max_seq_len;
    const long long units = std::max(groups, 1LL) * (mla::kOverheadTiles + ceil_div(kv_rows, mla::kKvTile));
    n_pairs = (int)std::max(1LL, std::min<long long>(n_pairs, units / mla::kMinUnits));
  }
  const int rc = make_layout(p, n_pairs, 2 * n_pairs, rows_per_group, &pl->lay);
  if (rc != MLA_OK) {
    delete pl;
    return rc;
  }
  pl->combine_grid = std::min(pl->lay.max_combine, 4 * sms);
  *plan = pl;
  *workspace_bytes = pl->lay.total;
  return MLA_OK;
}

}  // extern "C"

namespace {

// Device staging of mla_decode_run_host: the per-step inputs and results,
// each region 256-byte aligned.
struct HostStaging {
  size_t query, block_tables, seq_lens, qo_indptr, out, lse, total;
  size_t query_bytes, block_tables_bytes, seq_lens_bytes, qo_indptr_bytes, out_bytes, lse_bytes;
};

HostStaging host_staging(const mla_decode_params& prm, int64_t total_q) {
  const size_t B = (size_t)std::max(prm.batch, 0);
  const size_t tokens = prm.packed ? (size_t)std::max<int64_t>(total_q, 0)
                                   : B * (size_t)std::max(prm.max_seq_len_q, 0);
  const size_t H = (size_t)prm.num_heads;
  HostStaging st{};
  st.query_bytes = tokens * H * MLA_HEAD_DIM_QK * (prm.q_dtype == MLA_Q_FP8_E4M3 ? 1 : 2);
  st.block_tables_bytes = B * (size_t)std::max(prm.max_pages_per_req, 0) * sizeof(int32_t);
  st.seq_lens_bytes = B * sizeof(int32_t);
  st.qo_indptr_bytes = prm.packed ? (B + 1) * sizeof(int32_t) : 0;
  st.out_bytes = tokens * H * MLA_HEAD_DIM_V * 2;
  st.lse_bytes = prm.return_lse ? tokens * H * sizeof(float) : 0;
  size_t off = 0;
  auto take = [&](size_t n) {
    const size_t at = off;
    off = mla::align_up(off + n, 256);
    return at;
  };
  st.query = take(st.query_bytes);
  st.block_tables = take(st.block_tables_bytes);
  st.seq_lens = take(st.seq_lens_bytes);
  st.qo_indptr = take(st.qo_indptr_bytes);
  st.out = take(st.out_bytes);
  st.lse = take(st.lse_bytes);
  st.total = std::max<size_t>(off, 256);
  return st;
}

// Shared body of the run entry points.  Device scales (bmm1_dev / bmm2_dev
// non-null) replace the host values and are read by the kernels.
int run_impl(const mla_plan_t* plan, const void* query, const void* kv_cache,
             const int32_t* block_tables, const int32_t* seq_lens, const int32_t* qo_indptr,
             int64_t total_q, float bmm1_scale, float bmm2_scale, const float* bmm1_dev,
             const float* bmm2_dev, void* out, float* lse, void* workspace,
             size_t workspace_bytes, void* stream, void* event_before_decode,
             void* event_after_decode, const int32_t* seq_lens_global = nullptr,
             const int32_t* sparse_idx = nullptr, cudaEvent_t join_before_decode = nullptr) {
  if (!plan) return MLA_ERR_INVALID_ARG;
  const mla_decode_params& prm = plan->prm;
  // a sparse plan needs its position lists; no other plan takes them
  if ((prm.sparse_top_k > 0) != (sparse_idx != nullptr)) return MLA_ERR_INVALID_ARG;
  if (prm.batch == 0) return MLA_OK;
  if (sparse_idx && !aligned(sparse_idx, 4)) return MLA_ERR_ALIGNMENT;
  // a causal decode-context-parallel plan needs the global lengths; no other
  // plan takes them
  const bool dcp = prm.cp_world > 1;
  if (dcp && prm.mask == MLA_MASK_CAUSAL ? !seq_lens_global : seq_lens_global != nullptr)
    return MLA_ERR_INVALID_ARG;
  if (seq_lens_global && !aligned(seq_lens_global, 4)) return MLA_ERR_ALIGNMENT;
  // the plan's SM count, cluster occupancy and kernel attributes belong to
  // params.device, and the kernels launch on the current device
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return MLA_ERR_CUDA;
  if (cur != prm.device) return MLA_ERR_INVALID_ARG;
  if (!query || !kv_cache || !block_tables || !seq_lens || !out || !workspace)
    return MLA_ERR_INVALID_ARG;
  if (prm.return_lse && !lse) return MLA_ERR_INVALID_ARG;
  // the kernel takes the running max of raw scores and scales it afterwards
  if (!bmm1_dev && (!(bmm1_scale >= 0.f) || bmm1_scale > 3.0e38f)) return MLA_ERR_INVALID_ARG;
  if ((bmm1_dev && !aligned(bmm1_dev, 4)) || (bmm2_dev && !aligned(bmm2_dev, 4)))
    return MLA_ERR_ALIGNMENT;
  if (prm.packed) {
    if (!qo_indptr || total_q < 0 || total_q > prm.max_total_q) return MLA_ERR_INVALID_ARG;
  } else if (qo_indptr) {
    return MLA_ERR_INVALID_ARG;
  }
  if (workspace_bytes < plan->lay.total) return MLA_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(query, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) ||
      !aligned(workspace, 256) || !aligned(block_tables, 4) || !aligned(seq_lens, 4) ||
      (lse && !aligned(lse, 4)) || (qo_indptr && !aligned(qo_indptr, 4)))
    return MLA_ERR_ALIGNMENT;

  mla::Problem p;
  p.batch = prm.batch;
  p.num_heads = prm.num_heads;
  p.max_q = prm.max_seq_len_q;
  p.max_seq_len = prm.max_seq_len;
  p.page_size = prm.page_size;
  p.max_pages = prm.max_pages_per_req;
  p.packed = prm.packed;
  p.kv_dtype = prm.kv_dtype;
  p.q_fp8 = prm.q_dtype == MLA_Q_FP8_E4M3;
  p.f8_mma = uses_f8_mma(prm);
  p.cp_world = dcp ? prm.cp_world : 1;
  p.cp_rank = dcp ? prm.cp_rank : 0;
  p.seq_lens_global = seq_lens_global;
  p.sparse_k = prm.sparse_top_k > 0 ? prm.sparse_top_k : 0;
  p.sparse_idx = sparse_idx;
  p.causal = prm.mask == MLA_MASK_CAUSAL;
  p.return_lse = prm.return_lse != 0;
  p.num_pages = prm.num_pages;
  p.total_q = prm.packed ? total_q : (long long)prm.batch * prm.max_seq_len_q;
  p.bmm1_scale = bmm1_scale;
  p.bmm2_scale = bmm2_scale;
  p.bmm1_dev = bmm1_dev;
  p.bmm2_dev = bmm2_dev;
  p.query = query;
  p.kv_cache = kv_cache;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.qo_indptr = prm.packed ? qo_indptr : nullptr;
  p.out = out;
  p.lse = prm.return_lse ? lse : nullptr;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // while the stream is being captured into a graph, the events become
  // event-record nodes of the graph (timed at every replay)
  unsigned int ev_flags = cudaEventRecordDefault;
  if (event_before_decode || event_after_decode) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return MLA_ERR_CUDA;
    if (cs == cudaStreamCaptureStatusActive) ev_flags = cudaEventRecordExternal;
  }
  if (mla::launch_partition(p, plan->lay, workspace, s) != cudaSuccess) return MLA_ERR_CUDA;
  // work enqueued elsewhere that the decode needs (the host entry's query copy)
  if (join_before_decode && cudaStreamWaitEvent(s, join_before_decode, 0) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (uses_q_split(prm) &&
      mla::launch_qsplit(p, plan->lay, workspace, plan->sm_count, s) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (event_before_decode &&
      cudaEventRecordWithFlags(static_cast<cudaEvent_t>(event_before_decode), s, ev_flags) !=
          cudaSuccess)
    return MLA_ERR_CUDA;
  if (mla::launch_decode_sm103(p, plan->lay, workspace, s) != cudaSuccess) return MLA_ERR_CUDA;
  if (event_after_decode &&
      cudaEventRecordWithFlags(static_cast<cudaEvent_t>(event_after_decode), s, ev_flags) !=
          cudaSuccess)
    return MLA_ERR_CUDA;
  if (mla::launch_combine(p, plan->lay, workspace, plan->combine_grid, s) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

}  // namespace

extern "C" {

int mla_decode_run_profiled(const mla_plan_t* plan, const void* query, const void* kv_cache,
                            const int32_t* block_tables, const int32_t* seq_lens,
                            const int32_t* qo_indptr, int64_t total_q,
                            const int32_t* sparse_indices, float bmm1_scale, float bmm2_scale,
                            void* out, float* lse, void* workspace, size_t workspace_bytes,
                            void* stream, void* event_before_decode, void* event_after_decode) {
  return run_impl(plan, query, kv_cache, block_tables, seq_lens, qo_indptr, total_q, bmm1_scale,
                  bmm2_scale, nullptr, nullptr, out, lse, workspace, workspace_bytes, stream,
                  event_before_decode, event_after_decode, nullptr, sparse_indices);
}

int mla_decode_run_device_scales(const mla_plan_t* plan, const void* query, const void* kv_cache,
                                 const int32_t* block_tables, const int32_t* seq_lens,
                                 const int32_t* qo_indptr, int64_t total_q,
                                 const float* bmm1_scale, const float* bmm2_scale, void* out,
                                 float* lse, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  if (!bmm1_scale || !bmm2_scale) return MLA_ERR_INVALID_ARG;
  return run_impl(plan, query, kv_cache, block_tables, seq_lens, qo_indptr, total_q, 0.f, 0.f,
                  bmm1_scale, bmm2_scale, out, lse, workspace, workspace_bytes, stream, nullptr,
                  nullptr);
}

int mla_decode_run(const mla_plan_t* plan, const void* query, const void* kv_cache,
                   const int32_t* block_tables, const int32_t* seq_lens, const int32_t* qo_indptr,
                   int64_t total_q, float bmm1_scale, float bmm2_scale, void* out, float* lse,
                   void* workspace, size_t workspace_bytes, void* stream) {
  return run_impl(plan, query, kv_cache, block_tables, seq_lens, qo_indptr, total_q, bmm1_scale,
                  bmm2_scale, nullptr, nullptr, out, lse, workspace, workspace_bytes, stream,
                  nullptr, nullptr);
}

int mla_decode_run_dcp(const mla_plan_t* plan, const void* query, const void* kv_cache,
                       const int32_t* block_tables, const int32_t* seq_lens,
                       const int32_t* qo_indptr, int64_t total_q,
                       const int32_t* causal_seqlens_kv_global, float bmm1_scale,
                       float bmm2_scale, void* out, float* lse, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (!plan || plan->prm.cp_world <= 1) return MLA_ERR_INVALID_ARG;
  return run_impl(plan, query, kv_cache, block_tables, seq_lens, qo_indptr, total_q, bmm1_scale,
                  bmm2_scale, nullptr, nullptr, out, lse, workspace, workspace_bytes, stream,
                  nullptr, nullptr, causal_seqlens_kv_global);
}

int mla_decode_run_sparse(const mla_plan_t* plan, const void* query, const void* kv_cache,
                          const int32_t* block_tables, const int32_t* seq_lens,
                          const int32_t* qo_indptr, int64_t total_q,
                          const int32_t* sparse_indices, float bmm1_scale, float bmm2_scale,
                          void* out, float* lse, void* workspace, size_t workspace_bytes,
                          void* stream) {
  if (!plan || plan->prm.sparse_top_k <= 0 || !sparse_indices) return MLA_ERR_INVALID_ARG;
  return run_impl(plan, query, kv_cache, block_tables, seq_lens, qo_indptr, total_q, bmm1_scale,
                  bmm2_scale, nullptr, nullptr, out, lse, workspace, workspace_bytes, stream,
                  nullptr, nullptr, nullptr, sparse_indices);
}

int mla_merge_states(const void* o_parts, const float* lse_parts, int32_t n_parts, int64_t rows,
                     float scale, void* out, float* lse_out, void* stream) {
  if (n_parts < 1 || rows < 0 || rows > (1LL << 40) || (double)n_parts * (double)rows > 9.0e15)
    return MLA_ERR_INVALID_ARG;
  if (rows == 0) return MLA_OK;
  if (!o_parts || !lse_parts || !out) return MLA_ERR_INVALID_ARG;
  if (!aligned(o_parts, 16) || !aligned(out, 16) || !aligned(lse_parts, 4) ||
      (lse_out && !aligned(lse_out, 4)))
    return MLA_ERR_ALIGNMENT;
  return mla::launch_merge_states(o_parts, lse_parts, n_parts, rows, scale, out, lse_out,
                                  static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

size_t mla_decode_host_staging_bytes(const mla_plan_t* plan, int64_t total_q) {
  if (!plan) return 0;
  const mla_decode_params& prm = plan->prm;
  if (prm.packed && (total_q < 0 || total_q > prm.max_total_q)) return 0;
  const HostStaging st = host_staging(prm, total_q);
  return st.total;
}

int mla_decode_run_host(const mla_plan_t* plan, const void* h_query, const void* kv_cache,
                        const int32_t* h_block_tables, const int32_t* h_seq_lens,
                        const int32_t* h_qo_indptr, int64_t total_q, float bmm1_scale,
                        float bmm2_scale, void* h_out, float* h_lse, void* staging,
                        size_t staging_bytes, void* workspace, size_t workspace_bytes,
                        void* stream) {
  if (!plan) return MLA_ERR_INVALID_ARG;
  const mla_decode_params& prm = plan->prm;
  if (prm.batch == 0) return MLA_OK;
  if (!h_query || !kv_cache || !h_block_tables || !h_seq_lens || !h_out || !staging ||
      !workspace)
    return MLA_ERR_INVALID_ARG;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return MLA_ERR_CUDA;
  if (cur != prm.device || (prm.cp_world > 1 && prm.mask == MLA_MASK_CAUSAL) ||
      prm.sparse_top_k > 0)
    return MLA_ERR_INVALID_ARG;
  if (prm.return_lse && !h_lse) return MLA_ERR_INVALID_ARG;
  if (prm.packed) {
    if (!h_qo_indptr || total_q < 0 || total_q > prm.max_total_q) return MLA_ERR_INVALID_ARG;
  } else if (h_qo_indptr) {
    return MLA_ERR_INVALID_ARG;
  }
  if (!(bmm1_scale >= 0.f) || bmm1_scale > 3.0e38f) return MLA_ERR_INVALID_ARG;
  const HostStaging st = host_staging(prm, total_q);
  if (staging_bytes < st.total) return MLA_ERR_WORKSPACE_TOO_SMALL;
  if (workspace_bytes < plan->lay.total) return MLA_ERR_WORKSPACE_TOO_SMALL;
  // everything the decode itself would refuse is refused before a copy is enqueued
  if (!aligned(staging, 256) || !aligned(kv_cache, 16) || !aligned(workspace, 256))
    return MLA_ERR_ALIGNMENT;
  char* base = static_cast<char*>(staging);
  void* d_query = base + st.query;
  int32_t* d_bt = reinterpret_cast<int32_t*>(base + st.block_tables);
  int32_t* d_sl = reinterpret_cast<int32_t*>(base + st.seq_lens);
  int32_t* d_qo = prm.packed ? reinterpret_cast<int32_t*>(base + st.qo_indptr) : nullptr;
  void* d_out = base + st.out;
  float* d_lse = prm.return_lse ? reinterpret_cast<float*>(base + st.lse) : nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // One copy per buffer.  The metadata goes first on the caller's stream (the
  // partitioner reads nothing else); the query goes on the plan's side stream,
  // forked after the caller's earlier work (which may still read the staging
  // buffer) and joined before the decode, so it overlaps the partitioner.
  auto h2d = [&](void* dst, const void* src, size_t n, cudaStream_t on) {
    return n == 0 || cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, on) == cudaSuccess;
  };
  if (!h2d(d_bt, h_block_tables, st.block_tables_bytes, s) ||
      !h2d(d_sl, h_seq_lens, st.seq_lens_bytes, s) ||
      (d_qo && !h2d(d_qo, h_qo_indptr, st.qo_indptr_bytes, s)))
    return MLA_ERR_CUDA;
  cudaEvent_t fork = nullptr, join = nullptr;
  auto release = [&]() {  // pending events are released once their work completes
    if (fork) cudaEventDestroy(fork);
    if (join) cudaEventDestroy(join);
  };
  if (cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&join, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventRecord(fork, s) != cudaSuccess ||
      cudaStreamWaitEvent(plan->side_stream, fork, 0) != cudaSuccess ||
      !h2d(d_query, h_query, st.query_bytes, plan->side_stream) ||
      cudaEventRecord(join, plan->side_stream) != cudaSuccess) {
    release();
    return MLA_ERR_CUDA;
  }
  const int rc = run_impl(plan, d_query, kv_cache, d_bt, d_sl, d_qo, total_q, bmm1_scale,
                          bmm2_scale, nullptr, nullptr, d_out, d_lse, workspace, workspace_bytes,
                          stream, nullptr, nullptr, nullptr, nullptr, join);
  release();
  if (rc != MLA_OK) return rc;
  if (st.out_bytes &&
      cudaMemcpyAsync(h_out, d_out, st.out_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (d_lse && st.lse_bytes &&
      cudaMemcpyAsync(h_lse, d_lse, st.lse_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

void mla_decode_destroy(mla_plan_t* plan) {
  if (!plan) return;
  // the plan's side stream belongs to its device
  int prev = -1;
  const bool swap = cudaGetDevice(&prev) == cudaSuccess && prev != plan->prm.device &&
                    cudaSetDevice(plan->prm.device) == cudaSuccess;
  delete plan;
  if (swap) cudaSetDevice(prev);
}

size_t mla_decode_workspace_size(const mla_plan_t* plan) { return plan ? plan->lay.total : 0; }

int mla_decode_work_list_layout(const mla_plan_t* plan, size_t* items_offset,
                                size_t* worker_ranges_offset, int32_t* n_workers) {
  if (!plan || !items_offset || !worker_ranges_offset || !n_workers) return MLA_ERR_INVALID_ARG;
  static_assert(sizeof(mla::WorkItem) == 10 * sizeof(int32_t), "work item record");
  *items_offset = plan->lay.items;
  *worker_ranges_offset = plan->lay.worker_ranges;
  *n_workers = plan->lay.n_workers;
  return MLA_OK;
}

int32_t mla_decode_kernels_per_run(const mla_plan_t* plan) {
  if (!plan) return -1;
  if (plan->prm.batch == 0) return 0;
  return uses_q_split(plan->prm) ? 4 : 3;
}

size_t mla_decode_status_offset(void) { return sizeof(int) * mla::kHdrStatus; }

const char* mla_decode_status_string(int status) {
  switch (status) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "MLA_ERR_WORKSPACE_TOO_SMALL";
    case MLA_ERR_ALIGNMENT: return "MLA_ERR_ALIGNMENT";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    default: return "MLA_ERR_UNKNOWN";
  }
}

}  // extern "C"
