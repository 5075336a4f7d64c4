"""Shared helpers of the GPU tests: move a ``mla_inputs.Workload`` to the
device, run the CUDA library on it through the C ABI binding, and compare
with the fp64 oracle under the tolerances of the problem definition:

* bf16 KV:  |O - ref| <= 1e-2 + 2e-2 |ref|,  |lse - ref| <= 2e-3
* e4m3 KV:  |O - ref| <= 3e-2 + 5e-2 |ref|   (oracle fed the same e4m3 codes)
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import paged_mla_decode_03_gb300 as mla

TOL = {"bf16": (1e-2, 2e-2), "e4m3": (3e-2, 5e-2)}
LSE_TOL = 2e-3


@dataclasses.dataclass
class DeviceCase:
    query: torch.Tensor
    kv_cache: torch.Tensor
    block_tables: torch.Tensor
    seq_lens: torch.Tensor
    qo_indptr: object
    out: torch.Tensor
    lse: object
    workspace: torch.Tensor
    plan: mla.Plan


def to_device(w, *, return_lse=None, causal=None, workspace_fill=None, max_total_q=None,
              plan_batch=None):
    dev = torch.device("cuda", 0)
    if getattr(w, "q_dtype", "bf16") == "e4m3":
        q = torch.from_numpy(w.query).to(dev).view(torch.float8_e4m3fn)
    else:
        q = torch.from_numpy(w.query.view(np.int16)).to(dev).view(torch.bfloat16)
    if w.kv_dtype == "bf16":
        kv = torch.from_numpy(w.kv_cache.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        kv = torch.from_numpy(w.kv_cache).to(dev).view(torch.float8_e4m3fn)
    bt = torch.from_numpy(w.block_tables).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    qo = torch.from_numpy(w.qo_indptr).to(dev) if w.packed else None
    ret = w.return_lse if return_lse is None else return_lse
    cz = w.causal if causal is None else causal
    tokens = w.total_q if w.packed else w.batch * w.sq
    plan = mla.Plan(batch=w.batch, num_heads=w.num_heads, max_seq_len_q=w.max_seq_len_q,
                    max_seq_len=w.max_seq_len, page_size=w.page_size,
                    max_pages_per_req=w.block_tables.shape[1], num_pages=w.num_pages,
                    packed=w.packed, max_total_q=max_total_q if max_total_q else tokens,
                    kv_dtype=w.kv_dtype, causal=cz, return_lse=ret,
                    q_dtype=getattr(w, "q_dtype", "bf16"))
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=dev)
    if workspace_fill is not None:
        ws.fill_(workspace_fill)
    out = torch.full((tokens, w.num_heads, 512), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((tokens, w.num_heads), float("nan"), dtype=torch.float32, device=dev) if ret else None
    return DeviceCase(q, kv, bt, sl, qo, out, lse, ws, plan)


def run(w, d: DeviceCase, stream=None):
    d.plan.run(d.query, d.kv_cache, d.block_tables, d.seq_lens, d.out, qo_indptr=d.qo_indptr,
               total_q=w.total_q if w.packed else 0, lse=d.lse, workspace=d.workspace,
               bmm1_scale=w.bmm1_scale, bmm2_scale=w.bmm2_scale, stream=stream)


def results(d: DeviceCase):
    torch.cuda.synchronize()
    out = d.out.float().cpu().numpy().astype(np.float64)
    lse = d.lse.cpu().numpy().astype(np.float64) if d.lse is not None else None
    return out, lse


def device_status(d: DeviceCase) -> int:
    torch.cuda.synchronize()
    off = mla.mla_decode_status_offset()
    return int(d.workspace[off:off + 4].view(torch.int32).item())


def check(kv_dtype, out, ref_out, lse=None, ref_lse=None, what=""):
    """Element-wise tolerance check; returns the relative-L2 diagnostic."""
    atol, rtol = TOL[kv_dtype]
    assert np.isfinite(out).all(), f"{what}: non-finite output"
    err = np.abs(out - ref_out)
    bound = atol + rtol * np.abs(ref_out)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; "
                           f"max err {err.max():.3g} at {np.unravel_index(err.argmax(), err.shape)}")
    if lse is not None:
        lerr = np.abs(lse - ref_lse)
        assert np.isfinite(lse).all(), f"{what}: non-finite lse"
        assert lerr.max() <= LSE_TOL, f"{what}: lse max err {lerr.max():.3g}"
    denom = np.linalg.norm(ref_out)
    return float(np.linalg.norm(out - ref_out) / denom) if denom > 0 else 0.0


def sample_pairs(w, n, seed=0):
    """(token, head) pairs covering first/last rows of requests plus random ones."""
    rng = np.random.default_rng(seed)
    qs = w.q_start()
    H = w.num_heads
    picks = []
    for b in rng.choice(w.batch, size=min(w.batch, max(1, n // 4)), replace=False):
        t0, t1 = int(qs[b]), int(qs[b + 1])
        picks += [(t0, 0), (t1 - 1, H - 1), (t0 + (t1 - t0) // 2, H // 2)]
    tokens = int(qs[-1])
    while len(picks) < n:
        picks.append((int(rng.integers(tokens)), int(rng.integers(H))))
    return np.array(sorted(set(picks)), dtype=np.int64)
