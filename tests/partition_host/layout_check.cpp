// Checks the workspace layout of the plan's arithmetic (make_layout, from a
// generated copy of mla_api.cu's function) for plans read from a text file,
// one per line:
//   B H packed max_q max_total_q max_seq_len n_workers sparse_k kv_dtype q_dtype widen cp_world
// Every region must start on a 256-byte boundary, in order, and hold what the
// kernels write into it: work items, combine entries, worker ranges, the
// partitioner's scratch, the split partials (part_unit's largest index), their
// LSEs, the combine counters, and, on the FP8 MMA path with a bf16 query, one
// query-split record per (row, CTA half) at q_split_offset.  Prints "ok" or the
// first failed check and the plan's line number.
#include <cstdio>
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
  if (argc != 2) return 2;
  FILE* f = std::fopen(argv[1], "r");
  if (!f) return 2;
  int line = 0;
  long long B, H, packed, max_q, max_total_q, max_seq_len, n_workers, sparse_k, kv, qd, widen, cp;
  while (std::fscanf(f, "%lld %lld %lld %lld %lld %lld %lld %lld %lld %lld %lld %lld", &B, &H,
                     &packed, &max_q, &max_total_q, &max_seq_len, &n_workers, &sparse_k, &kv, &qd,
                     &widen, &cp) == 12) {
    ++line;
    mla_decode_params prm{};
    prm.batch = (int)B;
    prm.num_heads = (int)H;
    prm.packed = (int)packed;
    prm.max_seq_len_q = (int)max_q;
    prm.max_total_q = max_total_q;
    prm.max_seq_len = (int)max_seq_len;
    prm.sparse_top_k = (int)sparse_k;
    prm.kv_dtype = (int)kv;
    prm.q_dtype = (int)qd;
    prm.e4m3_widen = (int)widen;
    prm.cp_world = (int)cp;
    mla::Layout lay{};
    const int R = sparse_k > 0 ? (int)H : 128;
    if (make_layout(prm, (int)n_workers, 2 * (int)n_workers, R, &lay) != 0) {
      std::printf("line %d: make_layout refused the plan\n", line);
      return 1;
    }
    auto fail = [&](const char* what) {
      std::printf("line %d: %s\n", line, what);
      return 1;
    };
    const size_t starts[] = {lay.items,       lay.combine, lay.worker_ranges,
                             lay.req_scratch, lay.part_o,  lay.part_lse,
                             lay.comb_done};
    for (size_t s : starts)
      if (s % 256 != 0) return fail("a region starts off a 256-byte boundary");
    if (lay.items < kHeaderBytes) return fail("work items overlap the header");
    if (lay.combine < lay.items + sizeof(mla::WorkItem) * (size_t)lay.max_items)
      return fail("work items overflow into the combine entries");
    if (lay.worker_ranges < lay.combine + sizeof(mla::CombineItem) * (size_t)lay.max_combine)
      return fail("combine entries overflow into the worker ranges");
    if (lay.req_scratch < lay.worker_ranges + sizeof(int) * (size_t)(lay.n_workers + 1))
      return fail("worker ranges overflow into the partitioner scratch");
    if (lay.part_o < lay.req_scratch + lay.scratch_bytes)
      return fail("partitioner scratch overflows into the partials");
    if (lay.max_partials > 0) {
      const size_t last = mla::part_unit((size_t)lay.max_partials - 1, R, 31, mla::kPartUnits - 1,
                                         R - 1);
      if (lay.part_o + 16 * (last + 1) > lay.part_lse)
        return fail("the last partial unit overflows into the partial LSEs");
    }
    if (lay.comb_done < lay.part_lse + sizeof(float) * (size_t)R * (size_t)lay.max_partials)
      return fail("partial LSEs overflow into the combine counters");
    const size_t counters = sizeof(int) * (size_t)(lay.max_combine > 1 ? lay.max_combine : 1);
    if (lay.total < lay.comb_done + counters) return fail("combine counters overflow the workspace");
    const bool split = kv == MLA_KV_FP8_E4M3 && sparse_k == 0 && widen == 0 && qd == MLA_Q_BF16;
    if (split) {
      const long long tokens = packed ? max_total_q : B * max_q;
      const size_t records = 2 * (size_t)(tokens > 1 ? tokens : 1) * (size_t)H;
      const size_t q0 = mla::q_split_offset(lay);
      if (q0 % 16 != 0) return fail("query-split records are not 16-byte aligned");
      if (q0 < lay.comb_done + counters) return fail("query-split records overlap the counters");
      if (q0 + records * mla::kQSplitUnits * 16 > lay.total)
        return fail("query-split records overflow the workspace");
    }
  }
  std::fclose(f);
  std::printf("ok %d\n", line);
  return line > 0 ? 0 : 3;
}
