"""GPU test of mla_decode_run_static_workspace, the entry point for callers
that cannot allocate device memory when they enqueue a decode (code running
under CUDA graph capture, plug-ins inside runtimes that own all device
memory).  It must give the same result as mla_decode_run with a
caller-provided workspace, on two calls in a row (the second call reuses the
library's scratch array as the first one left it).

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import mla_inputs as mi
import paged_mla_decode_03_gb300 as mla
from harness import LSE_TOL, TOL, run, to_device

pytestmark = pytest.mark.gpu


def _entry():
    lib = mla.load_library()
    fn = lib.mla_decode_run_static_workspace
    vp = ctypes.c_void_p
    fn.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_int64, ctypes.c_float, ctypes.c_float, vp, vp,
                   vp]
    fn.restype = ctypes.c_int
    return fn


@pytest.mark.parametrize("make", [
    lambda: mi.deepseek_v3(batch=6, lo=100, hi=700, return_lse=True),
    lambda: mi.ragged(batch=12, median=200.0, max_len=1000),
    lambda: mi.fp8_long(batch=2, lo=300, hi=900, return_lse=True),
])
def test_static_workspace_matches_caller_workspace_twice(make):
    w = make()
    d = to_device(w)
    run(w, d)  # reference: caller-provided workspace
    torch.cuda.synchronize()
    ref_o = d.out.float().cpu().numpy()
    ref_l = d.lse.cpu().numpy() if d.lse is not None else None
    fn = _entry()
    stream = torch.cuda.current_stream().cuda_stream
    atol, rtol = TOL[w.kv_dtype]
    for _ in range(2):
        out = torch.full_like(d.out, float("nan"))
        lse = torch.full_like(d.lse, float("nan")) if d.lse is not None else None
        rc = fn(d.plan.handle, d.query.data_ptr(), d.kv_cache.data_ptr(),
                d.block_tables.data_ptr(), d.seq_lens.data_ptr(),
                d.qo_indptr.data_ptr() if d.qo_indptr is not None else None,
                w.total_q if w.packed else 0, w.bmm1_scale, w.bmm2_scale, out.data_ptr(),
                lse.data_ptr() if lse is not None else None, stream)
        assert rc == 0, mla.mla_decode_status_string(rc)
        torch.cuda.synchronize()
        o = out.float().cpu().numpy()
        assert np.isfinite(o).all()
        assert np.all(np.abs(o - ref_o) <= atol + rtol * np.abs(ref_o))
        if lse is not None:
            assert np.abs(lse.cpu().numpy() - ref_l).max() <= LSE_TOL


def test_static_workspace_rejects_plans_that_do_not_fit():
    # A packed plan with a huge total_q bound needs more scratch than the array holds.
    plan = mla.Plan(batch=16384, num_heads=128, max_seq_len_q=64, max_seq_len=4096, page_size=64,
                    max_pages_per_req=64, num_pages=16, packed=True, max_total_q=1 << 21)
    assert plan.workspace_bytes > mla.MLA_STATIC_WORKSPACE_BYTES
    rc = _entry()(plan.handle, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 16, 1.0, 1.0, 1 << 20,
                  None, torch.cuda.current_stream().cuda_stream)
    assert rc == -3  # MLA_ERR_WORKSPACE_TOO_SMALL, nothing enqueued


def test_static_workspace_captured_in_a_graph_follows_new_lengths():
    """The documented sequence for capture: one call outside capture (it
    resolves the array's device address), then a captured call, replayed with
    new seq_lens written in place between replays.  Each replay must equal
    the caller-workspace path on the same lengths."""
    w = mi.build("graph_static", 98, num_heads=16, page_size=32, seq_lens=[300, 120, 77],
                 q_lens=[2, 3, 1], packed=True, return_lse=True, max_seq_len_q=4)
    d = to_device(w)
    fn = _entry()
    s = torch.cuda.Stream()

    def call(out, lse):
        return fn(d.plan.handle, d.query.data_ptr(), d.kv_cache.data_ptr(),
                  d.block_tables.data_ptr(), d.seq_lens.data_ptr(), d.qo_indptr.data_ptr(),
                  w.total_q, w.bmm1_scale, w.bmm2_scale, out.data_ptr(), lse.data_ptr(),
                  s.cuda_stream)

    out_g = torch.full_like(d.out, float("nan"))
    lse_g = torch.full_like(d.lse, float("nan"))
    with torch.cuda.stream(s):
        assert call(out_g, lse_g) == 0  # outside capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        rc = call(out_g, lse_g)
    assert rc == 0
    atol, rtol = TOL["bf16"]
    for lens in ([250, 64, 77], [300, 3, 40]):
        d.seq_lens.copy_(torch.tensor(lens, dtype=torch.int32))
        out_g.fill_(float("nan"))
        lse_g.fill_(float("nan"))
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()
        run(w, d)  # caller workspace, same lengths, into d.out / d.lse
        torch.cuda.synchronize()
        o = out_g.float().cpu().numpy()
        ref_o = d.out.float().cpu().numpy()
        assert np.isfinite(o).all()
        assert np.all(np.abs(o - ref_o) <= atol + rtol * np.abs(ref_o)), lens
        assert np.abs(lse_g.cpu().numpy() - d.lse.cpu().numpy()).max() <= LSE_TOL, lens
