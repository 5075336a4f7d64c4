"""CPU tests of bench.py's host logic: the algorithmic work model and the
multi-rank reductions (world_size 2 over gloo on 127.0.0.1)."""
import os
import socket

import numpy as np
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
