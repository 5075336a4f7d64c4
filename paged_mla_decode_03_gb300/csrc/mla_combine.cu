// Split-KV combine: merges the normalised partials of every split
// (request, row group), stored in bf16 (part_unit in mla_common.cuh), by
// their natural-log LSEs (fp32), accumulating in fp32.
//
// For chunks k with partial output O_k (already divided by its own softmax
// denominator) and lse_k = ln sum_{j in chunk k} exp(s_j):
//   lse = ln sum_k exp(lse_k)          O = bmm2 * sum_k exp(lse_k - lse) * O_k
// which is exactly the single-pass result.  The natural-log LSE is the form
// the vLLM "FlashInferMLAImpl" page uses to merge partial attention across
// decode-context-parallel shards; here the shards are KV chunks of one GPU.
//
// An entry is merged once both CTAs of each of its chunks have counted their
// partial (a bounded acquire spin by one thread of the block), so entries
// whose chunks finished early are merged while the decode kernel still runs.
// An entry with no chunk (a decode-context-parallel rank that holds no row of
// the request) writes the empty sum: O = 0 and lse = -inf.
//
// Grid: (row blocks of 8 rows) x min(entry bound, 4 x SMs), 256 threads; a
// block takes entries blockIdx.y, + gridDim.y, ...; 32 threads per row, 16
// output dims per thread.  Every load of a thread (the LSEs and the 16-dim
// slices of up to kBatch chunks) is issued before any is used, so a row costs
// one memory round trip per kBatch chunks.  Blocks past the live number of
// entries exit at once, so the grid depends only on plan-time bounds.
#include <cuda_bf16.h>

#include <algorithm>

#include "mla_common.cuh"
#include "sm100_ptx.cuh"

namespace mla {

namespace {
constexpr int kThreads = 256;
constexpr int kRowsPerBlock = 8;
// chunks loaded per round trip: 2 keeps the combine at 64 registers, four
// blocks of 256 threads per SM (with 4, 80 registers and three blocks: the
// headline call 0.3 us, MTP 0.8 us and sparse 0.9 us slower, since fewer of the
// blocks waiting on unfinished entries fit beside the decode tail)
constexpr int kBatch = 2;
constexpr int kMergeBatch = 4;  // shards per round trip in merge_states_kernel
}  // namespace

// Waits (bounded) until the counter reaches `target`; acquire ordering makes
// the counted partials visible.  Gives up at once if a wait already timed out.
__device__ bool wait_count(const int* counter, int target, int* status) {
  for (uint32_t i = 0; i < (1u << 22); ++i) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
    if (v >= target) return true;
    if ((i & 255) == 255 && (*reinterpret_cast<volatile int*>(status) & kStatusTimeout)) return false;
    __nanosleep(128);
  }
  atomicOr(status, kStatusTimeout);
  return false;
}

// No grid-dependency wait: launched as a programmatic dependent of the decode
// kernel, whose CTAs release it right after their prologue, the combine's
// CTAs run on SMs the decode kernel has finished with and merge a group as
// soon as both CTAs of every chunk of it have counted their partial.
__global__ void __launch_bounds__(kThreads, 4)
combine_kernel(Problem p, Layout lay, char* __restrict__ ws) {
  int* status = reinterpret_cast<int*>(ws) + kHdrStatus;
  const int* done = reinterpret_cast<const int*>(ws + lay.comb_done);
  const int* hdr = reinterpret_cast<const int*>(ws);
  const CombineItem* comb = reinterpret_cast<const CombineItem*>(ws + lay.combine);
  const uint4* part_o = reinterpret_cast<const uint4*>(ws + lay.part_o);  // see part_unit
  const float* part_lse = reinterpret_cast<const float*>(ws + lay.part_lse);
  const int n_combine = hdr[kHdrNumCombine];
  const int H = p.num_heads;
  const int R = lay.rows_per_group;
  const int row_in_block = threadIdx.x >> 5;  // 0..7
  const int t = threadIdx.x & 31;             // output dims [16 t, 16 t + 16)

  for (int ci = blockIdx.y; ci < n_combine; ci += gridDim.y) {
    const CombineItem c = comb[ci];
    const int rows = min(R, c.q_len * H - c.g * R);
    const int r = blockIdx.x * kRowsPerBlock + row_in_block;
    if (blockIdx.x * kRowsPerBlock >= rows) continue;  // uniform over the block
    // every thread of the block reaches this barrier on every entry it visits
    // (the loop bounds and the test above are uniform); rows past the group's
    // end skip only the merge below
    if (!__syncthreads_and(threadIdx.x != 0 || wait_count(done + ci, 2 * c.n_chunks, status)))
      return;
    if (r < rows) {
      // running merge over batches of chunks: (m, sum, acc) rescaled per batch
      float m = -INFINITY, sum = 0.f;
      float acc[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[e] = 0.f;
      for (int k0 = 0; k0 < c.n_chunks; k0 += kBatch) {
        // this row's 16 dims of each chunk as stored (8 words of bf16 pairs,
        // or 16 fp32 words), widened where they are used: half the registers
        // of widening them here, so more blocks fit on an SM
        uint32_t xw[kBatch][4 * kPartUnits];
        float l[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          l[u] = -INFINITY;
#pragma unroll
          for (int v = 0; v < 4 * kPartUnits; ++v) xw[u][v] = 0u;
          if (k0 + u < c.n_chunks) {
            const size_t slot = (size_t)(c.first_slot + (k0 + u) * c.stride);
#pragma unroll
            for (int v = 0; v < kPartUnits; ++v) {
              const uint4 a = part_o[part_unit(slot, R, t, v, r)];
              xw[u][4 * v] = a.x;
              xw[u][4 * v + 1] = a.y;
              xw[u][4 * v + 2] = a.z;
              xw[u][4 * v + 3] = a.w;
            }
            l[u] = part_lse[slot * R + r];
          }
        }
        float m_new = m;
#pragma unroll
        for (int u = 0; u < kBatch; ++u) m_new = fmaxf(m_new, l[u]);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float f = expf(m - m_use);  // m = -inf: 0
        sum *= f;
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[e] *= f;
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const float w = expf(l[u] - m_use);  // absent chunks: l = -inf, w = 0
          sum += w;
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            // bf16: dim e is the low half of word e / 2 for even e, the high half for odd e
            const float xe = kPartialBf16 ? __uint_as_float((e & 1) ? (xw[u][e >> 1] & 0xFFFF0000u)
                                                                   : (xw[u][e >> 1] << 16))
                                          : __uint_as_float(xw[u][e]);
            acc[e] += w * xe;
          }
        }
        m = m_new;
      }
      const float s2 = sum > 0.f ? run_bmm2(p) / sum : 0.f;
      const size_t grow = (size_t)c.q_start * H + (size_t)c.g * R + r;
      __nv_bfloat162 o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = __floats2bfloat162_rn(acc[2 * e] * s2, acc[2 * e + 1] * s2);
      uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + grow * kVDim +
                                            16 * t);
      dst[0] = *reinterpret_cast<uint4*>(o);
      dst[1] = *reinterpret_cast<uint4*>(o + 4);
      const float m_use = (m == -INFINITY) ? 0.f : m;
      if (p.return_lse && t == 0) p.lse[grow] = (sum > 0.f) ? m_use + logf(sum) : -INFINITY;
    }
  }
}

cudaError_t launch_combine(const Problem& p, const Layout& lay, void* ws, int grid,
                           cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((lay.rows_per_group + kRowsPerBlock - 1) / kRowsPerBlock, grid, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, p, lay, static_cast<char*>(ws));
}

}  // namespace mla

namespace mla {

// Merge of n partial attention states of the same rows (the exchange step of
// decode-context parallelism, where each rank attends over its own KV shard;
// the vLLM "FlashInferMLAImpl" page merges such shards by their natural-log
// LSE).  For row r with shard outputs O_k (already normalised, bf16) and
// lse_k:  lse = ln sum_k exp(lse_k),  out = scale * sum_k exp(lse_k - lse) O_k.
// A shard with no visible key (lse = -inf) contributes nothing.  One warp
// per row, 16 dims per lane, every shard's loads issued before any use
// (batches of kMergeBatch shards).
__global__ void __launch_bounds__(256)
merge_states_kernel(const __nv_bfloat16* __restrict__ o_parts, const float* __restrict__ lse_parts,
                    int n, long long rows, float scale, __nv_bfloat16* __restrict__ out,
                    float* __restrict__ lse_out) {
  const int t = threadIdx.x & 31;  // dims [16 t, 16 t + 16)
  // grid-stride over blocks of 8 rows (rows may exceed what one grid covers)
  for (long long r = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); r < rows;
       r += (long long)gridDim.x * 8) {
    float m = -INFINITY, sum = 0.f;
    float acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = 0.f;
    for (int k0 = 0; k0 < n; k0 += kMergeBatch) {
      uint4 x[kMergeBatch][2];
      float l[kMergeBatch];
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        l[u] = -INFINITY;
        x[u][0] = x[u][1] = make_uint4(0, 0, 0, 0);
        if (k0 + u < n) {
          const size_t base = ((size_t)(k0 + u) * rows + r) * kVDim + 16 * t;
          const uint4* src = reinterpret_cast<const uint4*>(o_parts + base);
          x[u][0] = src[0];
          x[u][1] = src[1];
          l[u] = lse_parts[(size_t)(k0 + u) * rows + r];
        }
      }
      float m_new = m;
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) m_new = fmaxf(m_new, l[u]);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float f = expf(m - m_use);
      sum *= f;
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[e] *= f;
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        const float w = expf(l[u] - m_use);
        sum += w;
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(x[u]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float2 v = __bfloat1622float2(h[e]);
          acc[2 * e] += w * v.x;
          acc[2 * e + 1] += w * v.y;
        }
      }
      m = m_new;
    }
    const float s2 = sum > 0.f ? scale / sum : 0.f;
    __nv_bfloat162 o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = __floats2bfloat162_rn(acc[2 * e] * s2, acc[2 * e + 1] * s2);
    uint4* dst = reinterpret_cast<uint4*>(out + (size_t)r * kVDim + 16 * t);
    dst[0] = *reinterpret_cast<uint4*>(o);
    dst[1] = *reinterpret_cast<uint4*>(o + 4);
    const float m_use = (m == -INFINITY) ? 0.f : m;
    if (lse_out && t == 0) lse_out[r] = (sum > 0.f) ? m_use + logf(sum) : -INFINITY;
  }
}

cudaError_t launch_merge_states(const void* o_parts, const float* lse_parts, int n, long long rows,
                                float scale, void* out, float* lse_out, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const long long blocks = std::min<long long>((rows + 7) / 8, 1LL << 20);
  merge_states_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(o_parts), lse_parts, n, rows, scale,
      static_cast<__nv_bfloat16*>(out), lse_out);
  return cudaGetLastError();
}

}  // namespace mla
