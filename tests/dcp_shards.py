"""Decode-context-parallel sharding of a workload, for the DCP tests.

Each request's KV rows are cut at a page boundary into a prefix shard and a
suffix shard that holds at least the request's q_len last rows.  Every query
row sees the whole prefix (dense mask over it) and the suffix under the
bottom-right causal mask, so the two shards' natural-log-LSE merge equals
the single causal pass (the vLLM "FlashInferMLAImpl" page merges DCP shards
by this LSE).
"""
import dataclasses

import numpy as np


def split_points(w):
    """Page-aligned prefix length of each request (>= one page, leaves >= q rows)."""
    ps = w.page_size
    L0 = []
    for L, q in zip(w.seq_lens, w.q_lens):
        cut = ps * ((int(L) - int(q)) // (2 * ps))
        assert cut >= ps, "request too short to shard"
        L0.append(cut)
    return np.array(L0, dtype=np.int32)


def shards(w):
    """(prefix, suffix) workloads sharing w's query and cache; both with LSE
    and bmm2 = 1 (the merge applies w.bmm2_scale)."""
    ps = w.page_size
    L0 = split_points(w)
    bt0 = np.full_like(w.block_tables, -1)
    bt1 = np.full_like(w.block_tables, -1)
    for b in range(w.batch):
        n0 = int(L0[b]) // ps
        n_all = (int(w.seq_lens[b]) + ps - 1) // ps
        bt0[b, :n0] = w.block_tables[b, :n0]
        bt1[b, :n_all - n0] = w.block_tables[b, n0:n_all]
    pre = dataclasses.replace(w, seq_lens=L0, block_tables=bt0, causal=False, return_lse=True,
                              bmm2_scale=1.0, max_seq_len=int(L0.max()))
    suf_lens = (w.seq_lens - L0).astype(np.int32)
    suf = dataclasses.replace(w, seq_lens=suf_lens, block_tables=bt1, causal=True,
                              return_lse=True, bmm2_scale=1.0, max_seq_len=int(suf_lens.max()))
    return pre, suf


def merge_reference(outs, lses, scale):
    """float64 LSE merge of stacked partial states [n, rows..., 512], [n, rows...]."""
    outs = np.asarray(outs, dtype=np.float64)
    lses = np.asarray(lses, dtype=np.float64)
    m = lses.max(axis=0)
    w = np.exp(lses - m)
    z = w.sum(axis=0)
    out = scale * (w[..., None] * outs).sum(axis=0) / z[..., None]
    return out, m + np.log(z)
