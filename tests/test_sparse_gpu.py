"""GPU parity of sparse top-k decode (``mla_decode_run_sparse``) against the
fp64 oracle.

Reading of the pages (the FlashInfer issue's launcher takes a
``sparse_mla_top_k`` argument and says nothing more): query token t attends
exactly the logical KV positions listed in row t of an int32 [tokens, k]
list that fall in [0, seq_len), once per listing; the list replaces the mask.
The kernel gathers the listed rows itself (one token's H query rows per work
item), so these cases cover: lists shorter than the prefix (-1 padding),
ragged last tiles (k not a multiple of 64), repeated and out-of-range
entries, tokens with no usable entry (alone and inside split items), every
head count's row-group size, both cache dtypes and an e4m3 query.
"""
import dataclasses

import numpy as np
import pytest
import torch

import mla_inputs as mi
import oracle
import paged_mla_decode_03_gb300 as mla
from harness import check, device_status, results, run, to_device

pytestmark = pytest.mark.gpu


def parity(w, **kw):
    d = to_device(w, **kw)
    run(w, d)
    out, lse = results(d)
    ref_o, ref_l = oracle.run(w)
    check(w.kv_dtype, out.reshape(-1, w.num_heads, 512), ref_o, lse,
          ref_l if lse is not None else None, what=w.name)
    assert device_status(d) == 0
    return d, out, lse


def topk(seed, k, *, H=128, ps=64, seq_lens, q_lens, packed=False, kv_dtype="bf16",
         q_dtype="bf16", bmm1=None, lse=True):
    kw = {} if bmm1 is None else dict(bmm1_scale=bmm1)
    w = mi.build(f"sparse_h{H}_k{k}", seed, num_heads=H, page_size=ps, seq_lens=seq_lens,
                 q_lens=q_lens, packed=packed, return_lse=lse, kv_dtype=kv_dtype,
                 q_dtype=q_dtype, **kw)
    return mi.with_topk(w, k, seed + 1)


CASES = {
    # lists longer than some prefixes (-1 padded), one 128-row group per token
    "h128_q1_k256": lambda: topk(2001, 256, seq_lens=[100, 3000, 700, 256, 1500, 64],
                                 q_lens=[1] * 6),
    # MTP: four tokens per request, each its own group and its own list
    "h128_q4_k512": lambda: topk(2002, 512, seq_lens=[900, 2500, 520], q_lens=[4] * 3),
    # 16-row groups, packed ragged q, page size 32, k not a multiple of 64
    "h16_packed_k100": lambda: topk(2003, 100, H=16, ps=32, seq_lens=[300, 40, 1000, 99, 5],
                                    q_lens=[3, 1, 4, 2, 1], packed=True),
    "h64_k64": lambda: topk(2004, 64, H=64, seq_lens=[640, 65, 2000], q_lens=[2] * 3),
    "h32_k320": lambda: topk(2005, 320, H=32, seq_lens=[1200, 330, 4000, 321], q_lens=[1] * 4),
    # e4m3 cache (staging ring + converter warps) and a ragged tail tile
    "e4m3_h128_q2_k192": lambda: topk(2006, 192, seq_lens=[1000, 400, 3000], q_lens=[2] * 3,
                                      kv_dtype="e4m3"),
    "e4m3_h16_packed_k77": lambda: topk(2007, 77, H=16, ps=32, seq_lens=[500, 80, 2000],
                                        q_lens=[2, 1, 3], packed=True, kv_dtype="e4m3"),
    # e4m3 query (q_scale folded into bmm1) on a bf16 cache
    "e4m3q_h128_k128": lambda: topk(2008, 128, seq_lens=[700, 129, 2048], q_lens=[1] * 3,
                                    q_dtype="e4m3"),
    # wide logits
    "h128_k256_bmm1_1": lambda: topk(2009, 256, seq_lens=[2000, 600], q_lens=[2] * 2, bmm1=1.0),
}


@pytest.mark.parametrize("name", list(CASES))
def test_sparse_topk_full_parity(name):
    parity(CASES[name]())


def test_sparse_topk_repeated_out_of_range_and_padding_entries():
    """Repeated positions count once per listing; -1, negative and past-the-end
    positions (their pages hold NaN or sit past the table) are never read."""
    w = topk(2010, 128, seq_lens=[600, 1500, 300], q_lens=[2] * 3)
    idx = w.sparse_idx.copy()
    rng = np.random.default_rng(4)
    for t in range(idx.shape[0]):
        b = t // 2
        L = int(w.seq_lens[b])
        used = idx[t][idx[t] >= 0]
        pos = rng.choice(128, size=24, replace=False)
        idx[t, pos[:8]] = used[:8]                     # repeats
        idx[t, pos[8:12]] = -1
        idx[t, pos[12:16]] = -5 - np.arange(4)
        idx[t, pos[16:20]] = L + np.arange(4)          # the poisoned tail of the last page
        idx[t, pos[20:24]] = 10 ** 7
    parity(dataclasses.replace(w, sparse_idx=idx))


def test_sparse_topk_tokens_without_usable_entries_are_empty_sums():
    """Tokens whose lists hold nothing usable get out = 0 and lse = -inf,
    also when the token's list is long enough to be split across workers
    (every chunk then merges an empty state)."""
    w = topk(2011, 4096, seq_lens=[5000, 6000, 300], q_lens=[2] * 3)
    idx = w.sparse_idx.copy()
    idx[1] = -1                       # request 0, token 1: nothing listed
    idx[2, :] = 6000 + np.arange(4096)  # request 1, token 0: all past the end
    idx[5, 1:] = -1                   # request 2, token 1: one entry left
    d, out, lse = parity(dataclasses.replace(w, sparse_idx=idx))
    o = out.reshape(-1, w.num_heads, 512)
    assert np.all(o[[1, 2]] == 0) and np.all(np.isneginf(lse[[1, 2]]))
    assert np.all(np.isfinite(lse[5]))


def test_sparse_list_of_every_position_equals_the_dense_decode():
    """A list of all L positions (shuffled) through the sparse path and the
    plain dense decode agree within the bf16 tolerance, and both match the oracle."""
    w = mi.build("dense_ref", 2012, num_heads=128, page_size=64, seq_lens=[700, 1300, 64],
                 q_lens=[2] * 3, packed=False, causal=False, return_lse=True)
    rng = np.random.default_rng(6)
    k = int(w.seq_lens.max())
    idx = np.full((w.total_q, k), -1, np.int32)
    for t in range(w.total_q):
        L = int(w.seq_lens[t // 2])
        idx[t, :L] = rng.permutation(L)
    ws = dataclasses.replace(w, sparse_idx=idx, name="all_positions")
    _, out_s, lse_s = parity(ws)
    _, out_d, lse_d = parity(w)
    check("bf16", out_s, out_d, lse_s, lse_d, what="sparse vs dense")


def test_sparse_topk_repeats_are_bitwise_equal_with_a_dirty_workspace():
    w = topk(2013, 1024, seq_lens=[3000, 5000, 1100, 2000], q_lens=[1] * 4)
    first = None
    for fill in (0, 255, 77):
        d = to_device(w, workspace_fill=fill)
        run(w, d)
        torch.cuda.synchronize()
        assert device_status(d) == 0
        o, l = d.out.clone(), d.lse.clone()
        if first is None:
            first = (o, l)
        else:
            assert torch.equal(first[0].view(torch.int16), o.view(torch.int16))
            assert torch.equal(first[1], l)


def test_sparse_topk_graph_replay_follows_new_lists_and_lengths():
    """Lists and lengths live on the device: a captured decode replayed after
    both are rewritten in place equals a fresh run on the new values."""
    w = topk(2014, 256, seq_lens=[900, 400, 1600], q_lens=[2] * 3)
    d = to_device(w)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run(w, d, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run(w, d, stream=s)
    w2 = mi.with_topk(dataclasses.replace(w, seq_lens=np.array([800, 399, 1000], np.int32)), 256,
                      seed=99)
    d.seq_lens.copy_(torch.from_numpy(w2.seq_lens))
    d.sparse_idx.copy_(torch.from_numpy(w2.sparse_idx))
    d.out.fill_(float("nan"))
    with torch.cuda.stream(s):
        g.replay()
    s.synchronize()
    out, lse = results(d)
    ref_o, ref_l = oracle.run(w2)
    check("bf16", out.reshape(-1, w.num_heads, 512), ref_o, lse, ref_l, what="graph replay")


def test_sparse_topk_bad_page_id_of_a_listed_row_sets_the_status_bit():
    """A listed position inside [0, L) whose block-table entry is out of range
    (a contract violation) is skipped, flagged in the status word, and
    nothing faults; the other tokens are unaffected."""
    w = topk(2015, 128, seq_lens=[640, 640], q_lens=[1, 1])
    bt = w.block_tables.copy()
    bad_page = 3
    bt[0, bad_page] = w.num_pages + 11
    d = to_device(dataclasses.replace(w, block_tables=bt))
    run(w, d)
    out, lse = results(d)
    assert device_status(d) & 16
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    ref_o, ref_l = oracle.run(dataclasses.replace(w, batch=1, seq_lens=w.seq_lens[1:],
                                                  q_lens=w.q_lens[1:],
                                                  block_tables=w.block_tables[1:],
                                                  query=w.query[1:],
                                                  sparse_idx=w.sparse_idx[1:]))
    check("bf16", out.reshape(-1, w.num_heads, 512)[1:], ref_o, lse[1:], ref_l, what="others")


def test_sparse_and_plain_plans_refuse_each_others_entry_points():
    w = topk(2016, 64, seq_lens=[200], q_lens=[1])
    d = to_device(w)
    with pytest.raises(mla.MlaDecodeError):
        mla.mla_decode_run(d.plan.handle, d.query, d.kv_cache, d.block_tables, d.seq_lens, None,
                           0, w.bmm1_scale, w.bmm2_scale, d.out, d.lse, d.workspace)
    plain = dataclasses.replace(w, sparse_idx=None)
    dp = to_device(plain)
    with pytest.raises(mla.MlaDecodeError):
        mla.mla_decode_run_sparse(dp.plan.handle, dp.query, dp.kv_cache, dp.block_tables,
                                  dp.seq_lens, None, 0, d.sparse_idx, w.bmm1_scale, w.bmm2_scale,
                                  dp.out, dp.lse, dp.workspace)


def test_sparse_topk_through_decode_api():
    w = topk(2017, 192, seq_lens=[500, 1200], q_lens=[3, 3])
    d = to_device(w)
    q = d.query.view(w.batch, 3, w.num_heads, 576)
    out, lse = mla.decode(q, d.kv_cache.unsqueeze(1), d.workspace, d.block_tables, d.seq_lens,
                          w.max_seq_len, bmm1_scale=w.bmm1_scale, bmm2_scale=w.bmm2_scale,
                          return_lse=True, sparse_indices=d.sparse_idx)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.run(w)
    check("bf16", out.float().cpu().numpy().reshape(-1, w.num_heads, 512), ref_o,
          lse.cpu().numpy(), ref_l, what="decode api")


def test_sparse_profiled_entry_times_the_decode_and_equals_the_plain_entry():
    """The bench's entry point (events around the decode kernel) takes the
    lists too and gives the same bits as mla_decode_run_sparse."""
    w = topk(2018, 256, seq_lens=[900, 2000, 400], q_lens=[1] * 3)
    d = to_device(w)
    run(w, d)
    ref = d.out.clone()
    out = torch.full_like(d.out, float("nan"))
    ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    mla.mla_decode_run_profiled(d.plan.handle, d.query, d.kv_cache, d.block_tables, d.seq_lens,
                                None, 0, w.bmm1_scale, w.bmm2_scale, out, d.lse, d.workspace,
                                events=ev, sparse_indices=d.sparse_idx)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert ev[0].elapsed_time(ev[1]) > 0.0
    with pytest.raises(mla.MlaDecodeError):  # a sparse plan needs its lists here too
        mla.mla_decode_run_profiled(d.plan.handle, d.query, d.kv_cache, d.block_tables,
                                    d.seq_lens, None, 0, w.bmm1_scale, w.bmm2_scale, out, d.lse,
                                    d.workspace)


def test_sparse_plan_is_refused_by_the_allocation_free_entry():
    import ctypes
    w = topk(2019, 64, seq_lens=[300], q_lens=[1])
    d = to_device(w)
    lib = mla.load_library()
    fn = lib.mla_decode_run_static_workspace
    vp = ctypes.c_void_p
    fn.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_int64, ctypes.c_float, ctypes.c_float, vp, vp,
                   vp]
    fn.restype = ctypes.c_int
    rc = fn(d.plan.handle, d.query.data_ptr(), d.kv_cache.data_ptr(), d.block_tables.data_ptr(),
            d.seq_lens.data_ptr(), None, 0, w.bmm1_scale, w.bmm2_scale, d.out.data_ptr(),
            d.lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == -1  # MLA_ERR_INVALID_ARG: the static entry has no list argument
