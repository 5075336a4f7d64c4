// Host stand-ins for the CUDA constructs the partition kernel uses, so that
// its source compiles as C++ and runs with one std::thread per CUDA thread
// (one block): __syncthreads is a std::barrier over the block, __syncwarp one
// over the warp's 32 threads, a warp shuffle is an exchange through a per-warp array between two barriers of
// the warp's 32 threads, and atomics are std::atomic_ref operations.
#pragma once
#include <algorithm>
#include <atomic>
#include <barrier>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

struct HostDim3 {
  unsigned x = 1, y = 1, z = 1;
};
inline thread_local HostDim3 threadIdx;
inline HostDim3 blockDim;

#define __device__
#define __host__
#define __global__
#define __forceinline__ inline
#define __launch_bounds__(...)
#define __shared__ static
#define __align__(n) alignas(n)
#define __restrict__
using std::max;
using std::min;

inline std::barrier<>* g_block_barrier = nullptr;
inline void __syncthreads() { g_block_barrier->arrive_and_wait(); }

struct HostWarp {
  std::barrier<>* bar;
  long long slot[32];
};
inline std::vector<HostWarp*> g_warps;

template <typename T>
T host_exchange(T v, int src_lane) {
  const int lane = threadIdx.x & 31;
  HostWarp* w = g_warps[threadIdx.x >> 5];
  long long bits = 0;
  std::memcpy(&bits, &v, sizeof(T));
  w->slot[lane] = bits;
  w->bar->arrive_and_wait();
  const long long got = w->slot[src_lane];
  w->bar->arrive_and_wait();
  T out;
  std::memcpy(&out, &got, sizeof(T));
  return out;
}
template <typename T>
T __shfl_xor_sync(unsigned, T v, int d) {
  return host_exchange(v, (threadIdx.x & 31) ^ d);
}
template <typename T>
T __shfl_sync(unsigned, T v, int src_lane) {
  return host_exchange(v, src_lane & 31);
}
inline void __syncwarp(unsigned = 0xffffffffu) { g_warps[threadIdx.x >> 5]->bar->arrive_and_wait(); }
template <typename T>
T __shfl_up_sync(unsigned, T v, int d) {
  const int lane = threadIdx.x & 31;
  return host_exchange(v, lane >= d ? lane - d : lane);
}
inline int __syncthreads_or(int v) {
  static std::atomic<int> acc{0};
  static std::atomic<int> round{0};
  (void)round;
  __syncthreads();
  if (threadIdx.x == 0) acc.store(0);
  __syncthreads();
  if (v) acc.fetch_or(1);
  __syncthreads();
  const int r = acc.load();
  __syncthreads();
  return r;
}
inline int atomicOr(int* p, int v) { return std::atomic_ref<int>(*p).fetch_or(v); }
inline unsigned long long atomicAdd(unsigned long long* p, unsigned long long v) {
  return std::atomic_ref<unsigned long long>(*p).fetch_add(v);
}
inline void __threadfence() { std::atomic_thread_fence(std::memory_order_seq_cst); }
typedef int cudaError_t;
typedef void* cudaStream_t;
