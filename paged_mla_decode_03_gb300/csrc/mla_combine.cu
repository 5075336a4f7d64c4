// Split-KV combine: merges the normalised fp32 partials of every split
// (request, row group) by their natural-log LSEs.
//
// For chunks k with partial output O_k (already divided by its own softmax
// denominator) and lse_k = ln sum_{j in chunk k} exp(s_j):
//   lse = ln sum_k exp(lse_k)          O = bmm2 * sum_k exp(lse_k - lse) * O_k
// which is exactly the single-pass result.  The natural-log LSE is the form
// the vLLM "FlashInferMLAImpl" page uses to merge partial attention across
// decode-context-parallel shards; here the shards are KV chunks of one GPU.
#include <cuda_bf16.h>

#include "mla_common.cuh"

namespace mla {

namespace {
constexpr int kThreads = 256;
}

__global__ void __launch_bounds__(kThreads)
combine_kernel(Problem p, Layout lay, char* __restrict__ ws) {
  const int* hdr = reinterpret_cast<const int*>(ws);
  const CombineItem* comb = reinterpret_cast<const CombineItem*>(ws + lay.combine);
  const float* part_o = reinterpret_cast<const float*>(ws + lay.part_o);
  const float* part_lse = reinterpret_cast<const float*>(ws + lay.part_lse);
  const int n_combine = hdr[kHdrNumCombine];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = p.num_heads;
  const int R = lay.rows_per_group;

  for (int ci = blockIdx.x; ci < n_combine; ci += gridDim.x) {
    const CombineItem c = comb[ci];
    const int rows_total = c.q_len * H;
    const int rows = min(R, rows_total - c.g * R);
    for (int r = warp; r < rows; r += kThreads / 32) {
      // weights: each lane holds up to one chunk's lse per 32-chunk pass
      float m = -INFINITY;
      for (int k = lane; k < c.n_chunks; k += 32) {
        const int slot = c.first_slot + k * c.stride;
        m = fmaxf(m, part_lse[(size_t)slot * R + r]);
      }
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      const float m_use = (m == -INFINITY) ? 0.f : m;
      float sum = 0.f;
      for (int k = lane; k < c.n_chunks; k += 32) {
        const int slot = c.first_slot + k * c.stride;
        sum += expf(part_lse[(size_t)slot * R + r] - m_use);
      }
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      const float inv = sum > 0.f ? 1.f / sum : 0.f;
      // each lane owns 16 output dims: d = lane * 4 + 128 * v, v = 0..3
      float4 acc[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int k = 0; k < c.n_chunks; ++k) {
        const int slot = c.first_slot + k * c.stride;
        const float w = expf(part_lse[(size_t)slot * R + r] - m_use) * inv;
        const float4* src = reinterpret_cast<const float4*>(
            part_o + ((size_t)slot * R + r) * kVDim);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const float4 x = src[lane + 32 * v];
          acc[v].x += w * x.x;
          acc[v].y += w * x.y;
          acc[v].z += w * x.z;
          acc[v].w += w * x.w;
        }
      }
      const size_t grow = (size_t)c.q_start * H + (size_t)c.g * R + r;
      __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.out) + grow * kVDim;
      const float s2 = p.bmm2_scale;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc[v].x * s2, acc[v].y * s2);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc[v].z * s2, acc[v].w * s2);
        uint2 packed;
        packed.x = *reinterpret_cast<uint32_t*>(&lo);
        packed.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(dst + 4 * (lane + 32 * v)) = packed;
      }
      if (p.return_lse && lane == 0)
        p.lse[grow] = (sum > 0.f) ? m_use + logf(sum) : -INFINITY;
    }
  }
}

cudaError_t launch_combine(const Problem& p, const Layout& lay, void* ws, int grid,
                           cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  combine_kernel<<<grid, kThreads, 0, stream>>>(p, lay, static_cast<char*>(ws));
  return cudaGetLastError();
}

}  // namespace mla
