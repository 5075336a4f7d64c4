// Runs a partition kernel's source (the block or the single-warp form) on host threads for one problem read
// from a text file and writes the work list it leaves in the workspace.
// Built by tests/test_partition_host.py from generated copies of the kernel
// source (partition_host.inc) and of the plan's layout arithmetic
// (make_layout.inc).
#include <cstdio>
#include <cstdlib>
#include <deque>
#include <string>

#include "partition_host.inc"
#include "mla_decode.h"

namespace {
long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }
constexpr size_t kHeaderBytes = sizeof(int) * mla::kHdrWords;
enum { MLA_OK = 0, MLA_ERR_UNSUPPORTED = -2 };
#include "make_layout.inc"
}  // namespace

int main(int argc, char** argv) {
  // argv[3] = "warp": run the single-warp kernel (exit 4 if the plan does not fit it)
  if (argc != 3 && argc != 4) return 2;
  const bool warp_kernel = argc == 4 && std::string(argv[3]) == "warp";
  FILE* f = std::fopen(argv[1], "r");
  if (!f) return 2;
  int B, H, packed, max_q, max_seq_len, n_workers, sparse_k, causal;
  long long total_q;
  if (std::fscanf(f, "%d %d %d %d %d %d %d %d %lld", &B, &H, &packed, &max_q, &max_seq_len,
                  &n_workers, &sparse_k, &causal, &total_q) != 9)
    return 2;
  std::vector<int> seq_lens(B), qo(B + 1);
  for (auto& x : seq_lens)
    if (std::fscanf(f, "%d", &x) != 1) return 2;
  if (packed)
    for (auto& x : qo)
      if (std::fscanf(f, "%d", &x) != 1) return 2;
  std::fclose(f);
  mla_decode_params prm{};
  prm.batch = B;
  prm.num_heads = H;
  prm.max_seq_len_q = max_q;
  prm.max_seq_len = max_seq_len;
  prm.packed = packed;
  prm.max_total_q = total_q;
  prm.cp_world = 1;
  prm.sparse_top_k = sparse_k;
  mla::Layout lay{};
  if (make_layout(prm, n_workers, 2 * n_workers, sparse_k > 0 ? H : 128, &lay) != 0) return 3;
  std::vector<unsigned char> ws(lay.total, 0xAB);  // dirty, as a reused workspace would be
  std::vector<unsigned char> scratch(lay.scratch_in_smem ? lay.scratch_bytes : 16, 0xCD);
  g_scratch = scratch.data();
  mla::Problem p{};
  p.batch = B;
  p.num_heads = H;
  p.max_q = max_q;
  p.max_seq_len = max_seq_len;
  p.packed = packed;
  p.causal = causal;
  p.cp_world = 1;
  p.sparse_k = sparse_k;
  p.total_q = total_q;
  p.seq_lens = seq_lens.data();
  p.qo_indptr = packed ? qo.data() : nullptr;
  // the launch's block size (launch_partition)
  const long long need = std::max<long long>(std::max<long long>(B, lay.max_groups),
                                             (long long)lay.n_workers + 1);
  if (warp_kernel && !mla::partition_warp_fits(p, lay)) return 4;
  const int threads =
      warp_kernel ? 32
                  : (int)std::min<long long>(1024, std::max<long long>(128, (need + 31) / 32 * 32));
  blockDim.x = threads;
  std::barrier<> block_bar(threads);
  g_block_barrier = &block_bar;
  std::deque<std::barrier<>> warp_bars;  // constructed in place, never moved
  std::vector<HostWarp> warps(threads / 32);
  for (int w = 0; w < threads / 32; ++w) {
    warp_bars.emplace_back(32);
    warps[w].bar = &warp_bars[w];
    g_warps.push_back(&warps[w]);
  }
  std::vector<std::thread> th;
  for (int t = 0; t < threads; ++t)
    th.emplace_back([&, t] {
      threadIdx.x = t;
      if (warp_kernel)
        mla::partition_warp_kernel(p, lay, reinterpret_cast<char*>(ws.data()));
      else
        mla::partition_kernel(p, lay, reinterpret_cast<char*>(ws.data()));
    });
  for (auto& x : th) x.join();
  const int* hdr = reinterpret_cast<const int*>(ws.data());
  FILE* o = std::fopen(argv[2], "w");
  if (!o) return 2;
  std::fprintf(o, "%d %d %d\n", hdr[mla::kHdrStatus], hdr[mla::kHdrNumItems],
               hdr[mla::kHdrNumCombine]);
  const int* items = reinterpret_cast<const int*>(ws.data() + lay.items);
  for (int i = 0; i < hdr[mla::kHdrNumItems] * 10; ++i) std::fprintf(o, "%d ", items[i]);
  std::fprintf(o, "\n");
  const int* wb = reinterpret_cast<const int*>(ws.data() + lay.worker_ranges);
  for (int i = 0; i <= n_workers; ++i) std::fprintf(o, "%d ", wb[i]);
  std::fprintf(o, "\n");
  std::fclose(o);
  return 0;
}
