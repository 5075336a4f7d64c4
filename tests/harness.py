"""Shared helpers of the GPU tests: move a ``mla_inputs.Workload`` to the
device, run the CUDA library on it through the C ABI binding, and compare
with the fp64 oracle under the tolerances of the problem definition:

* bf16 KV:  |O - ref| <= 1e-2 + 2e-2 |ref|,  |lse - ref| <= 2e-3
* e4m3 KV:  |O - ref| <= 3e-2 + 5e-2 |ref|   (oracle fed the same e4m3 codes)

plus a gate on the relative L2 error ||O - ref|| / ||ref|| <= 1e-2.  At long
KV lengths |O| falls below the absolute term of the element-wise bound (an
all-zero output would pass it); the kernel's own rounding (P and the output
rounded to bf16, 2^-9 relative each) puts the relative L2 error near 2e-3, so
1e-2 leaves a 5x margin and still fails any dropped term or zeroed output.
Rows that see no key (a decode-context-parallel rank can hold none) must
come back with lse = -inf exactly where the oracle has it.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import paged_mla_decode_03_gb300 as mla

TOL = {"bf16": (1e-2, 2e-2), "e4m3": (3e-2, 5e-2)}
LSE_TOL = 2e-3
REL_L2_MAX = 1e-2


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
    seq_lens_global: object = None
    sparse_idx: object = None


def to_device(w, *, return_lse=None, causal=None, workspace_fill=None, max_total_q=None,
              plan_batch=None, e4m3_widen=False):
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
                    q_dtype=getattr(w, "q_dtype", "bf16"), cp_world=w.cp_world,
                    cp_rank=w.cp_rank, sparse_top_k=w.sparse_k, e4m3_widen=e4m3_widen)
    sp = torch.from_numpy(w.sparse_idx).to(dev) if w.sparse_idx is not None else None
    slg = None
    if w.cp_world > 1 and cz:
        slg = torch.from_numpy(w.seq_lens_global.astype(np.int32)).to(dev)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=dev)
    if workspace_fill is not None:
        ws.fill_(workspace_fill)
    out = torch.full((tokens, w.num_heads, 512), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((tokens, w.num_heads), float("nan"), dtype=torch.float32, device=dev) if ret else None
    return DeviceCase(q, kv, bt, sl, qo, out, lse, ws, plan, slg, sp)


def run(w, d: DeviceCase, stream=None):
    d.plan.run(d.query, d.kv_cache, d.block_tables, d.seq_lens, d.out, qo_indptr=d.qo_indptr,
               total_q=w.total_q if w.packed else 0, lse=d.lse, workspace=d.workspace,
               bmm1_scale=w.bmm1_scale, bmm2_scale=w.bmm2_scale, stream=stream,
               seq_lens_global=d.seq_lens_global, sparse_indices=d.sparse_idx)


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
    """Element-wise tolerance check plus the relative-L2 gate; returns the
    relative L2 error (printed, and named in every assertion message)."""
    atol, rtol = TOL[kv_dtype]
    out = np.asarray(out, dtype=np.float64)
    ref_out = np.asarray(ref_out, dtype=np.float64).reshape(out.shape)
    assert np.isfinite(out).all(), f"{what}: non-finite output"
    denom = np.linalg.norm(ref_out)
    diff = np.linalg.norm(out - ref_out)
    rel = float(diff / denom) if denom > 0 else float(diff)
    tag = f"{what}: rel-L2 {rel:.3g}"
    print(tag)
    err = np.abs(out - ref_out)
    bound = atol + rtol * np.abs(ref_out)
    bad = err > bound
    assert not bad.any(), (f"{tag}; {bad.sum()} of {bad.size} outside tolerance; "
                           f"max err {err.max():.3g} at {np.unravel_index(err.argmax(), err.shape)}")
    assert rel <= REL_L2_MAX, f"{tag} above {REL_L2_MAX}"
    if lse is not None:
        lse = np.asarray(lse, dtype=np.float64)
        ref_lse = np.asarray(ref_lse, dtype=np.float64).reshape(lse.shape)
        empty = np.isneginf(ref_lse)
        assert np.array_equal(np.isneginf(lse), empty), f"{tag}; lse -inf rows differ"
        assert np.isfinite(lse[~empty]).all(), f"{tag}; non-finite lse"
        if (~empty).any():
            lerr = np.abs(lse[~empty] - ref_lse[~empty]).max()
            assert lerr <= LSE_TOL, f"{tag}; lse max err {lerr:.3g}"
    return rel


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
