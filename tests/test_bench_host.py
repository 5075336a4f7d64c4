"""CPU tests of bench.py's host logic: the algorithmic work model and the
multi-rank reductions (world_size 2 over gloo on 127.0.0.1)."""
import dataclasses
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import mla_inputs as mi


def test_work_model_counts_visible_pairs_by_enumeration():
    w = mi.build("wm", 3, num_heads=4, page_size=32, seq_lens=[5, 9, 40], q_lens=[2, 3, 1],
                 packed=True, return_lse=True)
    wm = bench.work_model(w)
    n = 0
    for L, q in zip(w.seq_lens, w.q_lens):
        for i in range(q):
            n += sum(1 for j in range(L) if j <= L - q + i)
    assert wm["n_vis"] == n
    assert wm["flops"] == 2 * 4 * (576 + 512) * n
    assert wm["kv_bytes"] == int(w.seq_lens.sum()) * 576 * 2
    wd = mi.build("wm", 3, num_heads=4, page_size=32, seq_lens=[5, 9], q_lens=[2, 2],
                  packed=False, causal=False)
    assert bench.work_model(wd)["n_vis"] == 2 * 5 + 2 * 9


def test_sparse_work_model_counts_usable_entries_and_distinct_rows():
    """Under sparse top-k the FLOPs count every usable listed entry (repeats
    included), the KV bytes only the distinct rows of each request, and a
    list of every position once gives the dense non-causal counts."""
    w = mi.build("wms", 4, num_heads=4, page_size=32, seq_lens=[50, 70], q_lens=[2, 2],
                 packed=False, causal=False)
    dense = bench.work_model(w)
    idx = np.full((4, 70), -1, np.int32)
    for t in range(4):
        L = int(w.seq_lens[t // 2])
        idx[t, :L] = np.random.default_rng(t).permutation(L)
    full = bench.work_model(dataclasses.replace(w, sparse_idx=idx))
    assert full["n_vis"] == dense["n_vis"] and full["flops"] == dense["flops"]
    assert full["kv_bytes"] == dense["kv_bytes"]
    # repeats, -1 and past-the-end entries: 3 + 1 usable for token 0, 2 usable for the rest
    idx2 = np.full((4, 6), -1, np.int32)
    idx2[0] = [3, 3, 7, 50, -1, 9]
    idx2[1] = [0, 1, -1, -1, -1, 70]
    idx2[2] = [5, 6, -1, -1, -1, -1]
    idx2[3] = [5, 6, 70, -1, -1, -1]
    wm = bench.work_model(dataclasses.replace(w, sparse_idx=idx2))
    assert wm["n_vis"] == 4 + 2 + 2 + 2
    # distinct rows: request 0 {0, 1, 3, 7, 9}, request 1 {5, 6}
    assert wm["kv_bytes"] == (5 + 2) * 576 * 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    ws, r = bench.dist_init("gloo")
    assert (ws, r) == (world, rank)
    bench.barrier()
    mx = bench.reduce_max(1.5 + rank)
    sm = bench.reduce_sum(10.0 * (rank + 1))
    out[rank] = (mx, sm)
    dist.destroy_process_group()


def test_two_rank_max_and_sum_over_gloo():
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, join=True,
                       start_method="spawn")
    assert out[0] == (2.5, 30.0) and out[1] == (2.5, 30.0)


def test_roofline_picks_the_binding_resource():
    peaks = {"hbm_gbs": 1000.0, "bf16_tflops": 1000.0}
    w = mi.build("rf", 3, num_heads=128, page_size=64, seq_lens=[64], q_lens=[1], packed=False)
    wm = {"flops": 1e12, "bytes": 1e9}
    r = bench.roofline(w, wm, 2e-3, peaks)          # 1 ms of HBM, 1 ms of tensor: tie -> hbm
    assert r["bound"] == "hbm" and abs(r["frac"] - 0.5) < 1e-12
    wm = {"flops": 4e12, "bytes": 1e9}
    r = bench.roofline(w, wm, 8e-3, peaks)
    assert r["bound"] == "tensor" and abs(r["frac"] - 0.5) < 1e-12


def _dcp_worker(rank, world, port, out, layout):
    """One DCP rank on CPU: its shard's partial state (from the oracle), the
    library's all-gather step over gloo, then the reference LSE merge.
    layout "round_robin": global KV row g on rank g mod world, causal bound on
    global positions (the per-rank decode the vLLM FlashInferMLAImpl page asks
    of the kernel); "prefix_suffix": a dense prefix and a causal suffix."""
    import sys
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    import dcp_shards
    import oracle
    import paged_mla_decode_03_gb300 as mla
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = mi.build("dcp", 77, num_heads=2, page_size=4, seq_lens=[23, 17, 30], q_lens=[3, 3, 3],
                 packed=False, causal=True, return_lse=True, bmm1_scale=0.3, bmm2_scale=1.5)
    if layout == "round_robin":  # shards run with bmm2 = 1; the merge applies w's
        shard = dataclasses.replace(mi.dcp_shard(w, world, rank), bmm2_scale=1.0)
    else:
        shard = dcp_shards.shards(w)[rank]
    o, l = oracle.run(shard)
    outs, lses = mla.dcp_gather(torch.from_numpy(o), torch.from_numpy(l))
    merged, lse = dcp_shards.merge_reference(outs.numpy(), lses.numpy(), w.bmm2_scale)
    ref_o, ref_l = oracle.run(w)
    out[rank] = (float(np.abs(merged - ref_o).max()), float(np.abs(lse - ref_l).max()),
                 tuple(outs.shape))
    dist.destroy_process_group()


@pytest.mark.parametrize("layout", ["round_robin", "prefix_suffix"])
def test_dcp_two_ranks_gather_and_merge_equal_single_pass_over_gloo(layout):
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_dcp_worker, args=(2, _free_port(), out, layout), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        d_o, d_l, shape = out[r]
        assert shape == (2, 9, 2, 512)
        assert d_o < 1e-12 and d_l < 1e-12
