// Paged MLA decode, CUDA-core (SIMT) kernel: fp32 arithmetic on bf16 inputs.
//
// One persistent CTA per SM pulls work items (request, 64-row query group,
// KV chunk) from the partitioner's list and, for each item, streams the KV
// chunk in 64-row tiles gathered through block_tables:
//   S = Q K^T * bmm1 * log2(e)             (576-dim dot products)
//   mask: KV row j visible to query row i iff j <= L - q + i (causal, the
//         bottom-right rule of the FlashInfer page
//         "prims_ts_batch_decode_with_kv_cache_mla") or j < L (dense)
//   online softmax in base 2 (running max m, denominator l)
//   O = O * 2^(m_old - m_new) + P V         (V = first 512 dims of the tile)
// The epilogue writes bf16 O * bmm2 / l and the natural-log LSE
// (m + log2 l) * ln 2, or a normalised fp32 partial for the combine kernel.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "mla_common.cuh"

namespace mla {

namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerGroup = 64;
constexpr int kRowStride = kQkDim + 8;  // bf16 elements per smem row (bank skew)
constexpr int kSStride = kKvTile + 4;   // floats per smem score row (float4 aligned)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct SmemLayout {
  static constexpr size_t q = 0;
  static constexpr size_t kv = q + sizeof(__nv_bfloat16) * kRowsPerGroup * kRowStride;
  static constexpr size_t s = kv + sizeof(__nv_bfloat16) * kKvTile * kRowStride;
  static constexpr size_t stats = s + sizeof(float) * kRowsPerGroup * kSStride;
  static constexpr size_t item = stats + sizeof(float) * 3 * kRowsPerGroup;
  static constexpr size_t total = item + 64;
};

__device__ __forceinline__ float2 bf2_to_f2(uint32_t v) {
  __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&v);
  return __bfloat1622float2(h);
}

// 16 e4m3 bytes -> 16 bf16 values (exact: every e4m3 value is a bf16 value).
__device__ __forceinline__ void e4m3x16_to_bf16(const uint4 src, uint4* dst) {
  const uint32_t w[4] = {src.x, src.y, src.z, src.w};
  uint32_t o[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)((w[k] >> (16 * h)) & 0xFFFF);
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
      __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
      o[2 * k + h] = *reinterpret_cast<uint32_t*>(&b);
    }
  }
  dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
  dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

}  // namespace

template <bool kFp8>
__global__ void __launch_bounds__(kThreads, 1)
decode_simt_kernel(Problem p, Layout lay, char* __restrict__ ws) {
  extern __shared__ __align__(16) unsigned char smem[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem + SmemLayout::q);
  __nv_bfloat16* sK = reinterpret_cast<__nv_bfloat16*>(smem + SmemLayout::kv);
  float* sS = reinterpret_cast<float*>(smem + SmemLayout::s);
  float* sM = reinterpret_cast<float*>(smem + SmemLayout::stats);
  float* sL = sM + kRowsPerGroup;
  float* sA = sL + kRowsPerGroup;

  int* hdr = reinterpret_cast<int*>(ws);
  const WorkItem* items = reinterpret_cast<const WorkItem*>(ws + lay.items);
  float* part_o = reinterpret_cast<float*>(ws + lay.part_o);
  float* part_lse = reinterpret_cast<float*>(ws + lay.part_lse);
  const int* worker_begin = reinterpret_cast<const int*>(ws + lay.worker_ranges);
  const int item_begin = worker_begin[blockIdx.x], item_end = worker_begin[blockIdx.x + 1];
  const int tid = threadIdx.x;
  const int H = p.num_heads;
  const float s_scale = p.bmm1_scale * kLog2e;

  for (int idx = item_begin; idx < item_end; ++idx) {
    __syncthreads();
    const WorkItem it = items[idx];
    const int rows_total = it.q_len * H;
    const int row0 = it.g * kRowsPerGroup;
    const int n_rows = min(kRowsPerGroup, rows_total - row0);
    const size_t grow0 = (size_t)it.q_start * H + row0;

    // Q tile (rows past the group are zero)
    for (int e = tid; e < kRowsPerGroup * (kQkDim / 8); e += kThreads) {
      const int r = e / (kQkDim / 8), c = e % (kQkDim / 8);
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < n_rows)
        v = reinterpret_cast<const uint4*>(p.query)[(grow0 + r) * (kQkDim / 8) + c];
      *reinterpret_cast<uint4*>(sQ + r * kRowStride + c * 8) = v;
    }
    if (tid < kRowsPerGroup) {
      sM[tid] = -INFINITY;
      sL[tid] = 0.f;
    }
    float2 acc[kRowsPerGroup];
#pragma unroll
    for (int r = 0; r < kRowsPerGroup; ++r) acc[r] = make_float2(0.f, 0.f);

    for (int j0 = it.kv_begin; j0 < it.kv_end; j0 += kKvTile) {
      __syncthreads();
      // KV tile gathered through the page table; rows past kv_end are zero
      if (kFp8) {
        for (int e = tid; e < kKvTile * (kQkDim / 16); e += kThreads) {
          const int r = e / (kQkDim / 16), c = e % (kQkDim / 16);
          const int j = j0 + r;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (j < it.kv_end) {
            const int page = p.block_tables[(size_t)it.b * p.max_pages + j / p.page_size];
            if (page >= 0 && page < p.num_pages) {
              const size_t row = (size_t)page * p.page_size + (j % p.page_size);
              v = reinterpret_cast<const uint4*>(p.kv_cache)[row * (kQkDim / 16) + c];
            } else if (c == 0) {
              atomicOr(&hdr[kHdrStatus], 16);
            }
          }
          e4m3x16_to_bf16(v, reinterpret_cast<uint4*>(sK + r * kRowStride + c * 16));
        }
      } else {
        for (int e = tid; e < kKvTile * (kQkDim / 8); e += kThreads) {
          const int r = e / (kQkDim / 8), c = e % (kQkDim / 8);
          const int j = j0 + r;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (j < it.kv_end) {
            const int page = p.block_tables[(size_t)it.b * p.max_pages + j / p.page_size];
            if (page >= 0 && page < p.num_pages) {
              const size_t row = (size_t)page * p.page_size + (j % p.page_size);
              v = reinterpret_cast<const uint4*>(p.kv_cache)[row * (kQkDim / 8) + c];
            } else if (c == 0) {
              atomicOr(&hdr[kHdrStatus], 16);
            }
          }
          *reinterpret_cast<uint4*>(sK + r * kRowStride + c * 8) = v;
        }
      }
      __syncthreads();

      // S: thread owns rows 4*rt .. 4*rt+3 and columns ct + 16*k
      {
        const int rt = tid >> 4, ct = tid & 15;
        float s[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int k = 0; k < 4; ++k) s[a][k] = 0.f;
        const uint32_t* q32 = reinterpret_cast<const uint32_t*>(sQ);
        const uint32_t* k32 = reinterpret_cast<const uint32_t*>(sK);
#pragma unroll 4
        for (int d2 = 0; d2 < kQkDim / 2; ++d2) {
          float2 qv[4], kv[4];
#pragma unroll
          for (int a = 0; a < 4; ++a) qv[a] = bf2_to_f2(q32[(4 * rt + a) * (kRowStride / 2) + d2]);
#pragma unroll
          for (int k = 0; k < 4; ++k) kv[k] = bf2_to_f2(k32[(ct + 16 * k) * (kRowStride / 2) + d2]);
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int k = 0; k < 4; ++k) s[a][k] += qv[a].x * kv[k].x + qv[a].y * kv[k].y;
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const int r = 4 * rt + a;
          const int i = (row0 + r) / H;  // query row within the request
          const int last = p.causal ? it.seq_len - it.q_len + i : it.seq_len - 1;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int c = ct + 16 * k;
            const int j = j0 + c;
            const bool ok = (r < n_rows) && (j < it.kv_end) && (j <= last);
            sS[r * kSStride + c] = ok ? s[a][k] * s_scale : -INFINITY;
          }
        }
      }
      __syncthreads();

      // online softmax: 4 threads per row, 16 columns each
      {
        const int r = tid >> 2, qd = tid & 3;
        float* row = sS + r * kSStride + 16 * qd;
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 16; ++c) mx = fmaxf(mx, row[c]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_old = sM[r];
        const float m_new = fmaxf(m_old, mx);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        float sum = 0.f;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float e = exp2f(row[c] - m_use);
          row[c] = e;
          sum += e;
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        __syncwarp();
        if (qd == 0) {
          const float alpha = exp2f(m_old - m_use);
          sA[r] = alpha;
          sL[r] = sL[r] * alpha + sum;
          sM[r] = m_new;
        }
      }
      __syncthreads();

      // O += P V for this thread's two output dims
      {
        const uint32_t* v32 = reinterpret_cast<const uint32_t*>(sK);
#pragma unroll
        for (int r = 0; r < kRowsPerGroup; ++r) {
          const float a = sA[r];
          acc[r].x *= a;
          acc[r].y *= a;
        }
        for (int jj = 0; jj < kKvTile; jj += 4) {
          float2 v[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) v[u] = bf2_to_f2(v32[(jj + u) * (kRowStride / 2) + tid]);
#pragma unroll
          for (int r = 0; r < kRowsPerGroup; ++r) {
            const float4 pr = *reinterpret_cast<const float4*>(sS + r * kSStride + jj);
            acc[r].x += pr.x * v[0].x + pr.y * v[1].x + pr.z * v[2].x + pr.w * v[3].x;
            acc[r].y += pr.x * v[0].y + pr.y * v[1].y + pr.z * v[2].y + pr.w * v[3].y;
          }
        }
      }
    }
    __syncthreads();

    // epilogue
#pragma unroll
    for (int r = 0; r < kRowsPerGroup; ++r) {
      if (r >= n_rows) break;
      const float l = sL[r];
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if (it.slot < 0) {
        __nv_bfloat162 o = __floats2bfloat162_rn(acc[r].x * inv * p.bmm2_scale,
                                                 acc[r].y * inv * p.bmm2_scale);
        reinterpret_cast<__nv_bfloat162*>(p.out)[(grow0 + r) * (kVDim / 2) + tid] = o;
      } else {
        reinterpret_cast<float2*>(part_o)[((size_t)it.slot * kRowsPerGroup + r) * (kVDim / 2) + tid] =
            make_float2(acc[r].x * inv, acc[r].y * inv);
      }
    }
    if (tid < n_rows) {
      const float l = sL[tid];
      const float lse = l > 0.f ? (sM[tid] + log2f(l)) * kLn2 : -INFINITY;
      if (it.slot < 0) {
        if (p.return_lse) p.lse[grow0 + tid] = lse;
      } else {
        part_lse[(size_t)it.slot * kRowsPerGroup + tid] = lse;
      }
    }
  }
}

size_t decode_simt_smem_bytes() { return SmemLayout::total; }

cudaError_t decode_simt_setup() {
  cudaError_t e = cudaFuncSetAttribute(decode_simt_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SmemLayout::total);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(decode_simt_kernel<true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SmemLayout::total);
}

cudaError_t launch_decode_simt(const Problem& p, const Layout& lay, void* ws,
                               cudaStream_t stream) {
  if (p.kv_dtype == 1)
    decode_simt_kernel<true><<<lay.n_ctas, kThreads, SmemLayout::total, stream>>>(
        p, lay, static_cast<char*>(ws));
  else
    decode_simt_kernel<false><<<lay.n_ctas, kThreads, SmemLayout::total, stream>>>(
        p, lay, static_cast<char*>(ws));
  return cudaGetLastError();
}

}  // namespace mla
