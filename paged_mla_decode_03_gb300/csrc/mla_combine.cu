// Split-KV combine: merges the normalised fp32 partials of every split
// (request, row group) by their natural-log LSEs.
//
// For chunks k with partial output O_k (already divided by its own softmax
// denominator) and lse_k = ln sum_{j in chunk k} exp(s_j):
//   lse = ln sum_k exp(lse_k)          O = bmm2 * sum_k exp(lse_k - lse) * O_k
// which is exactly the single-pass result.  The natural-log LSE is the form
// the vLLM "FlashInferMLAImpl" page uses to merge partial attention across
// decode-context-parallel shards; here the shards are KV chunks of one GPU.
//
// Grid: (row blocks of 4 rows) x (combine entries), 256 threads; 64 threads
// per row, 8 output dims per thread, all chunk loads of a thread issued
// together.  Blocks past the live number of entries exit at once, so the
// grid depends only on plan-time bounds.
#include <cuda_bf16.h>

#include "mla_common.cuh"

namespace mla {

namespace {
constexpr int kThreads = 256;
constexpr int kRowsPerBlock = 4;
constexpr int kUnroll = 8;
}  // namespace

__global__ void __launch_bounds__(kThreads)
combine_kernel(Problem p, Layout lay, char* __restrict__ ws) {
  const int* hdr = reinterpret_cast<const int*>(ws);
  const CombineItem* comb = reinterpret_cast<const CombineItem*>(ws + lay.combine);
  const float* part_o = reinterpret_cast<const float*>(ws + lay.part_o);
  const float* part_lse = reinterpret_cast<const float*>(ws + lay.part_lse);
  const int n_combine = hdr[kHdrNumCombine];
  const int H = p.num_heads;
  const int R = lay.rows_per_group;
  const int row_in_block = threadIdx.x >> 6;  // 0..3
  const int t = threadIdx.x & 63;             // output dims [8 t, 8 t + 8)

  for (int ci = blockIdx.y; ci < n_combine; ci += gridDim.y) {
    const CombineItem c = comb[ci];
    const int rows = min(R, c.q_len * H - c.g * R);
    const int r = blockIdx.x * kRowsPerBlock + row_in_block;
    if (r >= rows) continue;
    float m = -INFINITY;
    for (int k = 0; k < c.n_chunks; ++k)
      m = fmaxf(m, part_lse[(size_t)(c.first_slot + k * c.stride) * R + r]);
    const float m_use = (m == -INFINITY) ? 0.f : m;
    float sum = 0.f;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int k0 = 0; k0 < c.n_chunks; k0 += kUnroll) {
      float4 x[kUnroll][2];
      float w[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        w[u] = 0.f;
        x[u][0] = x[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k0 + u < c.n_chunks) {
          const size_t slot = (size_t)(c.first_slot + (k0 + u) * c.stride);
          const float4* src =
              reinterpret_cast<const float4*>(part_o + (slot * R + r) * kVDim) + 2 * t;
          x[u][0] = src[0];
          x[u][1] = src[1];
          w[u] = expf(part_lse[slot * R + r] - m_use);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        sum += w[u];
        acc[0] += w[u] * x[u][0].x;
        acc[1] += w[u] * x[u][0].y;
        acc[2] += w[u] * x[u][0].z;
        acc[3] += w[u] * x[u][0].w;
        acc[4] += w[u] * x[u][1].x;
        acc[5] += w[u] * x[u][1].y;
        acc[6] += w[u] * x[u][1].z;
        acc[7] += w[u] * x[u][1].w;
      }
    }
    const float s2 = sum > 0.f ? p.bmm2_scale / sum : 0.f;
    const size_t grow = (size_t)c.q_start * H + (size_t)c.g * R + r;
    __nv_bfloat162 o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = __floats2bfloat162_rn(acc[2 * e] * s2, acc[2 * e + 1] * s2);
    *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + grow * kVDim + 8 * t) =
        *reinterpret_cast<uint4*>(o);
    if (p.return_lse && t == 0) p.lse[grow] = (sum > 0.f) ? m_use + logf(sum) : -INFINITY;
  }
}

cudaError_t launch_combine(const Problem& p, const Layout& lay, void* ws, int grid,
                           cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  const dim3 g((lay.rows_per_group + kRowsPerBlock - 1) / kRowsPerBlock, grid, 1);
  combine_kernel<<<g, kThreads, 0, stream>>>(p, lay, static_cast<char*>(ws));
  return cudaGetLastError();
}

}  // namespace mla
