// Query split for the FP8 MMAs (an e4m3 cache read by kind::f8f6f4 MMAs with
// a bf16 query).  The vLLM page "FlashInferMLAImpl" runs the products of a
// quantised cache in FP8 with bmm1 multiplied by the cache's scale; the FP8
// tensor cores take e4m3 for both operands, so a bf16 query row is carried as
// two e4m3 parts whose sum is the row to about bf16's precision.
//
// For every query row and each half of it that one CTA of the decode pair
// reads (rank r: latent dims [256 r, 256 r + 256), RoPE dims [512 + 32 r, +32),
// 288 dims), the row half is scaled by 2^k, the largest power of two with
// max|x| 2^k <= 448 over those 288 dims, and split into hi = e4m3(x) and
// lo = e4m3(x - hi).  hi + lo equals x exactly wherever |x| >= 2^-2 (x is a
// bf16 value times a power of two, and x - hi has at most four significant
// bits at or above 2^-9) and to within 2^-10 below that, i.e. within 2^-17 of
// the half's largest element.  The decode multiplies the half's partial scores
// by 2^-k before the two halves are added.  An all-zero half, or one holding a
// NaN or an infinity, takes k = 0.
//
// Output per (row, half), a record of kQSplitUnits 16-byte units at
// q_split_offset(lay): latent hi (16), latent lo (16), RoPE hi (2), RoPE lo
// (2), codes in dim order, and the factor 2^-k in the first word of the last.
// One warp per row, grid-strided: lane l holds the row's 16-byte units l
// (latent, half 0), 32 + l (latent, half 1) and, for l < 8, 64 + l (RoPE, half
// l / 4), so every load and store of a warp is contiguous; each half's
// largest magnitude is a warp reduction.
//
// Launch: after the partitioner, as its programmatic dependent (it reads only
// the query and writes only its own workspace region, so it may run beside
// the partitioner), and it releases the decode kernel at its start.  The
// decode kernel's grid-dependency wait covers this grid alone, so this grid's
// last step waits for its own primary: when it completes, the partitioner has
// completed too.
#include <cuda_bf16.h>

#include <algorithm>

#include "mla_common.cuh"
#include "sm100_ptx.cuh"

namespace mla {

namespace {

constexpr int kThreads = 256;

// Eight bf16 values (one uint4) times `up` -> two words of hi codes and two of
// lo codes (four codes a word, low byte first).
__device__ __forceinline__ void split8(const uint4 x, float up, uint32_t* hi, uint32_t* lo) {
  const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const float a = __uint_as_float(w4[2 * e] << 16) * up;
    const float b = __uint_as_float(w4[2 * e] & 0xFFFF0000u) * up;
    const float c = __uint_as_float(w4[2 * e + 1] << 16) * up;
    const float d = __uint_as_float(w4[2 * e + 1] & 0xFFFF0000u) * up;
    const uint32_t hab = ptx::f32x2_to_e4m3x2(a, b), hcd = ptx::f32x2_to_e4m3x2(c, d);
    float fa, fb, fc, fd;
    ptx::e4m3x2_to_f32x2(hab, fa, fb);
    ptx::e4m3x2_to_f32x2(hcd, fc, fd);
    hi[e] = hab | (hcd << 16);
    lo[e] = ptx::f32x2_to_e4m3x2(a - fa, b - fb) | (ptx::f32x2_to_e4m3x2(c - fc, d - fd) << 16);
  }
}

// The exponent k of a half whose largest magnitude has the bf16 bit pattern
// `mbits` (sign cleared): the largest k with max|x| 2^k <= 448 = 1.75 * 2^8;
// 0 for an all-zero half or one holding a NaN or an infinity.
__device__ __forceinline__ int split_exponent(uint32_t mbits) {
  const float amax = __uint_as_float(mbits << 16);
  if (!(amax > 0.f && amax <= 3.4028235e38f)) return 0;
  const uint32_t ab = __float_as_uint(amax);
  const int E = (int)(ab >> 23);  // biased exponent, 0 for a subnormal
  const int k = E == 0 ? 126 : ((ab & 0x7FFFFFu) <= 0x600000u ? 135 - E : 134 - E);
  return min(126, max(-126, k));
}

__device__ __forceinline__ uint32_t max_bits(const uint4 x) {  // both halves of each word
  return __vmaxu2(__vmaxu2(x.x & 0x7FFF7FFFu, x.y & 0x7FFF7FFFu),
                  __vmaxu2(x.z & 0x7FFF7FFFu, x.w & 0x7FFF7FFFu));
}

__global__ void __launch_bounds__(kThreads)
qsplit_kernel(Problem p, Layout lay, char* __restrict__ ws) {
  ptx::pdl_launch_dependents();
  const long long rows = p.total_q * p.num_heads;
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (kThreads / 32);
  uint2* out = reinterpret_cast<uint2*>(ws + q_split_offset(lay));  // 2 * kQSplitUnits a record
  // the loop bound is the same for every lane of a warp
  for (long long row = ((long long)blockIdx.x * kThreads + threadIdx.x) >> 5; row < rows;
       row += warps) {
    const uint4* src = reinterpret_cast<const uint4*>(
        reinterpret_cast<const __nv_bfloat16*>(p.query) + row * kQkDim);
    const uint4 a = __ldg(src + lane);
    const uint4 b = __ldg(src + 32 + lane);
    const uint4 c = lane < 8 ? __ldg(src + 64 + lane) : make_uint4(0, 0, 0, 0);
    uint32_t m0 = max_bits(a), m1 = max_bits(b);
    if (lane < 4) m0 = __vmaxu2(m0, max_bits(c));
    else if (lane < 8) m1 = __vmaxu2(m1, max_bits(c));
    for (int o = 16; o > 0; o >>= 1) {
      m0 = __vmaxu2(m0, __shfl_xor_sync(0xffffffffu, m0, o));
      m1 = __vmaxu2(m1, __shfl_xor_sync(0xffffffffu, m1, o));
    }
    const int k0 = split_exponent(max(m0 & 0xFFFFu, m0 >> 16));
    const int k1 = split_exponent(max(m1 & 0xFFFFu, m1 >> 16));
    const float up0 = __uint_as_float((uint32_t)(127 + k0) << 23);
    const float up1 = __uint_as_float((uint32_t)(127 + k1) << 23);
    uint2* d0 = out + (row * 2) * (2 * kQSplitUnits);
    uint2* d1 = d0 + 2 * kQSplitUnits;
    uint32_t hw[2], lw[2];
    split8(a, up0, hw, lw);
    d0[lane] = make_uint2(hw[0], hw[1]);  // latent hi
    d0[32 + lane] = make_uint2(lw[0], lw[1]);  // latent lo
    split8(b, up1, hw, lw);
    d1[lane] = make_uint2(hw[0], hw[1]);
    d1[32 + lane] = make_uint2(lw[0], lw[1]);
    if (lane < 8) {
      uint2* d = lane < 4 ? d0 : d1;
      split8(c, lane < 4 ? up0 : up1, hw, lw);
      d[64 + (lane & 3)] = make_uint2(hw[0], hw[1]);  // RoPE hi
      d[68 + (lane & 3)] = make_uint2(lw[0], lw[1]);  // RoPE lo
    }
    if (lane == 0) {  // the factors 2^-k, in unit 36 of each record
      d0[72] = make_uint2((uint32_t)(127 - k0) << 23, 0u);
      d1[72] = make_uint2((uint32_t)(127 - k1) << 23, 0u);
    }
  }
  // complete only after the partitioner (this grid's primary) has
  ptx::pdl_wait();
}

}  // namespace

cudaError_t launch_qsplit(const Problem& p, const Layout& lay, void* ws, int sm_count,
                          cudaStream_t stream) {
  const long long rows = p.total_q * p.num_heads;
  if (rows <= 0) return cudaSuccess;
  constexpr int kWarps = kThreads / 32;
  const long long blocks =
      std::max<long long>(1, std::min<long long>((rows + kWarps - 1) / kWarps, 4LL * sm_count));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, qsplit_kernel, p, lay, static_cast<char*>(ws));
}

}  // namespace mla
