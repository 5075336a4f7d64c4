"""The partition kernels' own source, run on CPU threads, against the host model.

The partitioner's arithmetic is pinned twice: by ``tests/partition_model.py``
(a Python restatement, checked for its invariants on CPU and compared with the
kernel's work list on the GPU), and here. The test compiles the CUDA source
of both kernel forms (``partition_kernel``, one block, and
``partition_warp_kernel``, one warp, which the launch picks for small plans) as C++ with host stand-ins for the barriers and warp
shuffles (``tests/partition_host/shim.h``), under AddressSanitizer and
UndefinedBehaviorSanitizer. It runs one std::thread per CUDA thread of the
launch and requires the work list the kernel leaves in a dirty workspace to
equal the host model's, item by item and worker range by worker range. An
out-of-range index or a race on the shared scratch shows up here, on CPU,
before any GPU run.
"""
import os
import re
import shutil
import subprocess

import numpy as np
import pytest

import mla_inputs as mi
from partition_model import partition

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.join(ROOT, "tests", "partition_host")
CSRC = os.path.join(ROOT, "paged_mla_decode_03_gb300", "csrc")


def _function_text(src, head):
    """The text of the function that starts at `head`, through its closing brace."""
    i = src.index(head)
    j = src.index("{", i)
    depth = 0
    for k in range(j, len(src)):
        depth += {"{": 1, "}": -1}.get(src[k], 0)
        if depth == 0:
            return src[i:k + 1]
    raise ValueError(head)


@pytest.fixture(scope="module")
def emulator(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no g++")
    out = tmp_path_factory.mktemp("partition_host")
    common = open(os.path.join(CSRC, "mla_common.cuh")).read()
    common = common.replace("#include <cuda_runtime.h>\n", "")
    common = common.replace("#pragma once", "#pragma once\ninline unsigned char* g_scratch = nullptr;", 1)
    (out / "mla_common_host.h").write_text(common)
    src = open(os.path.join(CSRC, "mla_partition.cu")).read()
    src = src.replace('#include "mla_common.cuh"\n#include "sm100_ptx.cuh"\n',
                      '#include "shim.h"\n#include "mla_common_host.h"\n')
    src = src.replace("ptx::pdl_launch_dependents();", "")
    src = src.replace("extern __shared__ __align__(16) unsigned char scratch_smem[];",
                      "unsigned char* scratch_smem = g_scratch;")
    src = src[:src.index("cudaError_t launch_partition(")] + "}  // namespace mla\n"
    assert "asm" not in src and "__ldg" not in src
    (out / "partition_host.inc").write_text(src)
    api = open(os.path.join(CSRC, "mla_api.cu")).read()
    (out / "make_layout.inc").write_text(_function_text(api, "int make_layout(") + "\n")
    exe = out / "partition_host"
    cmd = [cxx, "-std=c++20", "-O1", "-g", "-fsanitize=address,undefined",
           "-fno-sanitize-recover=undefined", "-pthread", "-I", str(out), "-I", HERE,
           "-I", os.path.join(ROOT, "include"), os.path.join(HERE, "driver.cpp"), "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0 and ("No such file" in r.stderr or "cannot find -l" in r.stderr):
        pytest.skip("host toolchain lacks C++20 <barrier> or the sanitizers: " + r.stderr[-300:])
    assert r.returncode == 0, r.stderr[-3000:]
    return exe, out


def _run(emulator, w, n_workers, kernel="block"):
    """Runs one kernel form on `w`; returns False if the single-warp form was
    asked for and the plan does not fit it."""
    exe, out = emulator
    inp, res = out / "in.txt", out / "out.txt"
    with open(inp, "w") as f:
        f.write(f"{w.batch} {w.num_heads} {int(w.packed)} {w.max_seq_len_q} {w.max_seq_len} "
                f"{n_workers} {w.sparse_k} {int(w.causal)} {w.total_q}\n")
        f.write(" ".join(str(int(x)) for x in w.seq_lens) + "\n")
        if w.packed:
            f.write(" ".join(str(int(x)) for x in w.qo_indptr) + "\n")
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=0:abort_on_error=1")
    args = [str(exe), str(inp), str(res)] + (["warp"] if kernel == "warp" else [])
    r = subprocess.run(args, capture_output=True, text=True, env=env, timeout=300)
    if kernel == "warp" and r.returncode == 4:
        return False
    assert r.returncode == 0, (r.returncode, r.stderr[-3000:])
    lines = open(res).read().split("\n")
    status, n_items, _ = (int(x) for x in lines[0].split())
    vals = [int(x) for x in lines[1].split()]
    got = [vals[10 * i:10 * i + 10] for i in range(n_items)]
    wb = [int(x) for x in lines[2].split()]
    items, ref_wb, _ = partition(w.seq_lens, w.q_lens, w.q_start()[:-1], w.num_heads, n_workers,
                                 w.seq_lens.astype(np.int64) - w.q_lens, sparse_k=w.sparse_k)
    assert status == 0
    assert got == [list(t) for t in items]
    assert wb == ref_wb
    return True


@pytest.mark.parametrize("kernel", ["block", "warp"])
@pytest.mark.parametrize("name", ["tiny", "deepseek_v3", "mtp", "ragged", "fp8_long",
                                  "sparse_topk"])
def test_kernel_source_work_list_equals_host_model_on_bench_workloads(emulator, name, kernel):
    # every one of these plans fits the single-warp form (the launch picks it
    # for tiny and fp8_long)
    assert _run(emulator, mi.WORKLOADS[name](), 76, kernel)


class _Shape:
    """Just the fields the partitioner reads (no KV pool is drawn)."""

    def __init__(self, seq_lens, q_lens, H, packed, sparse_k):
        self.seq_lens = np.asarray(seq_lens, np.int32)
        self.q_lens = np.asarray(q_lens, np.int32)
        self.batch = len(self.seq_lens)
        self.num_heads = H
        self.packed = packed
        self.causal = True
        self.sparse_k = sparse_k
        self.max_seq_len = int(self.seq_lens.max())
        self.max_seq_len_q = int(self.q_lens.max())
        self.total_q = int(self.q_lens.sum())
        self.qo_indptr = np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)

    def q_start(self):
        return self.qo_indptr.astype(np.int64)


@pytest.mark.parametrize("kernel", ["block", "warp"])
@pytest.mark.parametrize("seed", range(10))
def test_kernel_source_work_list_equals_host_model_on_random_shapes(emulator, seed, kernel):
    rng = np.random.default_rng(7000 + seed)
    B = int(rng.integers(1, 200))
    H = int(rng.choice([16, 32, 64, 128]))
    packed = bool(rng.integers(2))
    q = (rng.integers(1, 9, size=B) if packed else np.full(B, int(rng.integers(1, 5))))
    L = rng.integers(q, int(rng.choice([100, 3000, 40000])), endpoint=True)
    sparse_k = int(rng.choice([64, 100, 2048])) if rng.random() < 0.3 else 0
    _run(emulator, _Shape(L, q, H, packed, sparse_k), int(rng.choice([1, 7, 76, 148, 600])),
         kernel)


def _plan_groups(q, H, packed, sparse_k):
    """The plan's bound on row groups (make_layout): R = 128 rows, or H under
    sparse top-k, where a group is one token's heads."""
    R = H if sparse_k else 128
    B, max_q = len(q), int(np.max(q))
    groups = B * -(-max_q * H // R)
    if packed:
        groups = min(groups, B + -(-int(np.sum(q)) * H // R))
    return groups


@pytest.mark.parametrize("seed", range(24))
def test_single_warp_kernel_on_shapes_near_its_bounds(emulator, seed):
    """The single-warp form on shapes up to its table bounds (512 requests,
    512 row groups, 512 workers), with lengths that make many short groups,
    one group longer than all the others, or groups shorter than the overhead;
    every shape must fit it and give the host model's work list."""
    rng = np.random.default_rng(9100 + seed)
    H = int(rng.choice([16, 32, 64, 128]))
    packed = bool(rng.integers(2))
    sparse_k = int(rng.choice([64, 2048])) if rng.random() < 0.25 else 0
    B = int(rng.integers(1, 513))
    q = rng.integers(1, 9, size=B) if packed else np.full(B, int(rng.integers(1, 5)))
    while _plan_groups(q, H, packed, sparse_k) > 512:
        q = q[:max(1, len(q) * 3 // 4)]
    B = len(q)
    kind = seed % 3
    if kind == 0:
        L = rng.integers(q, q + 200, endpoint=True)
    elif kind == 1:
        L = rng.integers(q, 2000, endpoint=True)
        L[int(rng.integers(B))] = 120000
    else:
        L = rng.integers(q, 40000, endpoint=True)
    n_workers = int(rng.choice([1, 2, 76, 148, 511, 512]))
    assert _run(emulator, _Shape(L, q, H, packed, sparse_k), n_workers, "warp")


def test_workspace_layout_regions_hold_what_the_kernels_write(emulator):
    """The plan's layout arithmetic (make_layout) on plans of every kind: bf16
    and e4m3 caches (FP8 MMAs with a bf16 or an e4m3 query, and widened),
    fixed and packed queries from one token to prefill sizes, sparse top-k,
    decode-context parallelism, and worker counts from 1 to 600.  Every region
    must be 256-byte aligned, in order, and large enough for what the kernels
    write (tests/partition_host/layout_check.cpp states the checks)."""
    exe_dir = emulator[1]
    cxx = shutil.which("g++")
    exe = exe_dir / "layout_check"
    r = subprocess.run([cxx, "-std=c++20", "-O1", "-fsanitize=address,undefined",
                        "-fno-sanitize-recover=undefined", "-pthread", "-I", str(exe_dir), "-I",
                        HERE, "-I", os.path.join(ROOT, "include"),
                        os.path.join(HERE, "layout_check.cpp"), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    rows = []
    # B H packed max_q max_total_q max_seq_len n_workers sparse_k kv q widen cp_world
    for kv, q, widen in ((0, 0, 0), (1, 0, 0), (1, 1, 0), (1, 0, 1)):
        rows += [
            (2, 16, 0, 1, 0, 64, 76, 0, kv, q, widen, 1),            # tiny
            (64, 128, 0, 1, 0, 8192, 76, 0, kv, q, widen, 1),        # headline
            (32, 128, 0, 4, 0, 16384, 76, 0, kv, q, widen, 1),       # MTP
            (128, 16, 1, 8, 576, 32768, 76, 0, kv, q, widen, 1),     # ragged
            (8, 128, 0, 2, 0, 131072, 76, 0, kv, q, widen, 1),       # long context
            (512, 128, 1, 48, 18432, 2048, 76, 0, kv, q, widen, 1),  # prefill
            (64, 128, 0, 1, 0, 12288, 76, 2048, kv, q, widen, 1),    # sparse top-k
            (16, 64, 0, 2, 0, 4096, 76, 0, kv, q, widen, 2),         # DCP rank
            (1, 16, 1, 1, 1, 1, 1, 0, kv, q, widen, 1),              # one token, one worker
            (200, 32, 1, 8, 900, 40000, 600, 100, kv, q, widen, 1),  # sparse, many workers
            (300, 128, 1, 8, 2400, 5000, 148, 0, kv, q, widen, 1),
        ]
    inp = exe_dir / "layouts.txt"
    inp.write_text("\n".join(" ".join(str(v) for v in row) for row in rows) + "\n")
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=0:abort_on_error=1")
    r = subprocess.run([str(exe), str(inp)], capture_output=True, text=True, env=env, timeout=60)
    assert r.returncode == 0, (r.stdout, r.stderr[-2000:])
    assert r.stdout.strip() == f"ok {len(rows)}"
