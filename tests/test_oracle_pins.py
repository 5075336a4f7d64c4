"""Pins of the fp64 oracle against facts the problem statement and the
mathematics fix, independently of the oracle's own code.

Each test is chosen so that a plausible slip in the oracle (a dropped RoPE
term, an off-by-one causal bound, a log2 LSE, a transposed page walk, a wrong
scale placement) fails at least one of them.  All run on CPU.
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import mla_inputs as mi
import oracle
from oracle import brute


def small(seed, *, H=2, ps=4, seq_lens=(9, 5), q_lens=(1, 1), packed=False, causal=True,
          kv_dtype="bf16", bmm1=0.125, bmm2=1.0, poison=True, q_dtype="bf16"):
    return mi.build("pin", seed, num_heads=H, page_size=ps, seq_lens=list(seq_lens),
                    q_lens=list(q_lens), packed=packed, causal=causal, kv_dtype=kv_dtype,
                    bmm1_scale=bmm1, bmm2_scale=bmm2, poison=poison, return_lse=True,
                    q_dtype=q_dtype)


def as_f64(bits, kv_dtype="bf16"):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16 if kv_dtype == "bf16" else np.uint8))
    t = t.view(torch.bfloat16) if kv_dtype == "bf16" else t.view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def gather(w, b):
    """Dense [L, 576] float64 rows of request b (numpy fancy indexing)."""
    L = int(w.seq_lens[b])
    j = np.arange(L)
    pages = w.block_tables[b][j // w.page_size]
    return as_f64(w.kv_cache, w.kv_dtype)[pages, j % w.page_size]


# ---------------------------------------------------------------- decoders

def test_bf16_decoder_matches_torch_all_codes():
    codes = np.arange(1 << 16, dtype=np.uint16)
    ref = as_f64(codes)
    got = np.array([oracle.decode_bf16(int(c)) for c in codes])
    got_b = np.array([brute.bf16_value(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and np.array_equal(np.isnan(got_b), nan)
    assert np.array_equal(got[~nan], ref[~nan]) and np.array_equal(got_b[~nan], ref[~nan])


def test_e4m3_decoder_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = as_f64(codes, "e4m3")
    got = np.array([oracle.decode_e4m3(int(c)) for c in codes])
    got_b = np.array([brute.e4m3_value(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert nan.sum() == 2  # S.1111.111 for both signs
    assert np.array_equal(np.isnan(got), nan) and np.array_equal(np.isnan(got_b), nan)
    assert np.array_equal(got[~nan], ref[~nan]) and np.array_equal(got_b[~nan], ref[~nan])
    assert ref[0x7E] == 448.0 and ref[0x01] == 2.0 ** -9


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("case", [
    dict(seq_lens=(9, 5), q_lens=(1, 1)),
    dict(seq_lens=(7, 12), q_lens=(3, 3), causal=True),
    dict(seq_lens=(7, 12), q_lens=(3, 3), causal=False),
    dict(seq_lens=(6, 3, 11), q_lens=(2, 3, 1), packed=True),
    dict(seq_lens=(10, 4), q_lens=(2, 2), kv_dtype="e4m3", bmm1=0.5, bmm2=0.75),
    dict(seq_lens=(13,), q_lens=(4,), ps=8, bmm1=3.0),
    dict(seq_lens=(8, 11), q_lens=(2, 2), q_dtype="e4m3", bmm1=0.5),
    dict(seq_lens=(9, 6), q_lens=(1, 1), q_dtype="e4m3", kv_dtype="e4m3", bmm1=4.0),
])
def test_c_oracle_matches_python_brute_force(case):
    w = small(7, **case)
    out, lse = oracle.run(w)
    bo, bl = brute.mla_decode(w.query_rows(), w.q_start(), w.kv_cache, w.block_tables,
                              w.seq_lens, kv_dtype=w.kv_dtype, causal=w.causal,
                              bmm1_scale=w.bmm1_scale, bmm2_scale=w.bmm2_scale,
                              q_dtype=w.q_dtype)
    np.testing.assert_allclose(out, np.array(bo), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, np.array(bl), rtol=1e-12, atol=1e-12)
    assert np.isfinite(out).all() and np.isfinite(lse).all()


# ---------------------------------------------------------------- closed forms

def test_seq_len_one_returns_scaled_first_row():
    """L = 1: softmax over one row is 1, so O = bmm2 * V_0 and lse = bmm1 * q.k_0."""
    w = small(3, H=3, seq_lens=(1, 1, 1), q_lens=(1, 1, 1), bmm1=0.3, bmm2=1.7)
    out, lse = oracle.run(w)
    Q = as_f64(w.query_rows())
    for b in range(w.batch):
        k0 = gather(w, b)[0]
        for h in range(w.num_heads):
            assert lse[b, h] == pytest.approx(w.bmm1_scale * np.dot(Q[b, h], k0), rel=1e-13, abs=1e-13)
            np.testing.assert_allclose(out[b, h], w.bmm2_scale * k0[:512], rtol=1e-14, atol=0)


def _visible(L, q, i, causal):
    return (L - q + i + 1) if causal else L


@pytest.mark.parametrize("causal", [True, False])
def test_zero_query_gives_uniform_mean_and_log_count(causal):
    """Q = 0 makes every visible score 0: lse = ln(n_visible), O = bmm2 * mean(V)."""
    w = small(11, H=2, seq_lens=(13, 6), q_lens=(4, 4), causal=causal, bmm2=2.0)
    w = dataclasses.replace(w, query=np.zeros_like(w.query))
    out, lse = oracle.run(w)
    for b in range(w.batch):
        rows = gather(w, b)
        L, q = int(w.seq_lens[b]), int(w.q_lens[b])
        for i in range(q):
            n = _visible(L, q, i, causal)
            t = b * q + i
            for h in range(w.num_heads):
                assert lse[t, h] == pytest.approx(math.log(n), abs=1e-14)
                np.testing.assert_allclose(out[t, h], 2.0 * rows[:n, :512].mean(axis=0),
                                           rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("causal", [True, False])
def test_index_encoded_values_expose_each_visible_set(causal):
    """V_j = one-hot(j) and Q = 0: O[d] = 1/n for exactly the visible rows d.

    This reads the mask decision for every (row, KV index) pair exactly,
    including the bottom-right alignment of the causal bound.
    """
    ps, seq_lens, q_lens = 8, [21, 9, 30], [5, 2, 7]
    w = small(13, H=1, ps=ps, seq_lens=seq_lens, q_lens=q_lens, packed=True, causal=causal)
    kv = np.zeros(w.kv_cache.shape, np.float32)
    for b, L in enumerate(seq_lens):
        for j in range(L):
            kv[w.block_tables[b][j // ps], j % ps, j] = 1.0
    w = dataclasses.replace(w, kv_cache=mi.bf16_bits(kv), query=np.zeros_like(w.query))
    out, lse = oracle.run(w)
    qs = w.q_start()
    for b, (L, q) in enumerate(zip(seq_lens, q_lens)):
        for i in range(q):
            t = qs[b] + i
            n = (L - q + i + 1) if causal else L
            expect = np.zeros(512)
            expect[:n] = 1.0 / n
            np.testing.assert_allclose(out[t, 0], expect, rtol=1e-13, atol=1e-16)
            assert (out[t, 0] > 0).sum() == n


def test_constant_scores_give_mean_of_values():
    """Latent query part 0 and one shared RoPE part in every row: all scores
    equal c = bmm1 * q_rope . k_rope, so O = bmm2 * mean(V) and lse = c + ln n."""
    w = small(17, H=2, seq_lens=(11, 7), q_lens=(2, 2), bmm1=0.2, bmm2=0.5)
    rng = np.random.default_rng(5)
    rope = mi.bf16_bits(rng.standard_normal(64).astype(np.float32))
    kv = w.kv_cache.copy()
    kv[..., 512:] = rope
    q = w.query.copy().reshape(-1, w.num_heads, 576)
    q[..., :512] = 0
    w = dataclasses.replace(w, kv_cache=kv, query=q.reshape(w.query.shape))
    out, lse = oracle.run(w)
    Q = as_f64(q)
    rope64 = as_f64(rope)
    for b in range(w.batch):
        rows = gather(w, b)
        L, qn = int(w.seq_lens[b]), int(w.q_lens[b])
        for i in range(qn):
            n = L - qn + i + 1
            t = b * qn + i
            for h in range(w.num_heads):
                c = w.bmm1_scale * np.dot(Q[t, h, 512:], rope64)
                assert lse[t, h] == pytest.approx(c + math.log(n), rel=1e-13, abs=1e-13)
                np.testing.assert_allclose(out[t, h], 0.5 * rows[:n, :512].mean(axis=0),
                                           rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------- invariances

def test_page_permutation_invariance():
    w = small(19, H=3, ps=4, seq_lens=(17, 5, 12), q_lens=(2, 2, 2))
    w2 = mi.permute_pages(w, seed=3)
    assert not np.array_equal(w.block_tables, w2.block_tables)
    o1, l1 = oracle.run(w)
    o2, l2 = oracle.run(w2)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_packed_uniform_equals_fixed():
    w = small(23, H=2, seq_lens=(9, 14, 6), q_lens=(3, 3, 3))
    qo = np.array([0, 3, 6, 9], np.int32)
    wp = dataclasses.replace(w, packed=True, qo_indptr=qo,
                             query=w.query.reshape(9, w.num_heads, 576))
    o1, l1 = oracle.run(w)
    o2, l2 = oracle.run(wp)
    assert np.array_equal(o1.reshape(o2.shape), o2) and np.array_equal(l1.reshape(l2.shape), l2)


def _flatten(w):
    """One request per query row: per-row copies of block_tables/seq_lens
    (the flattening the vLLM FlashInferMLAImpl page applies to dense decode)."""
    qs = w.q_start()
    row_req = np.searchsorted(qs[1:], np.arange(w.total_q), side="right")
    return dataclasses.replace(
        w, batch=w.total_q, packed=True, q_lens=np.ones(w.total_q, np.int32),
        qo_indptr=np.arange(w.total_q + 1, dtype=np.int32),
        query=w.query_rows().copy(), block_tables=w.block_tables[row_req].copy(),
        seq_lens=w.seq_lens[row_req].copy())


def test_dense_multi_token_equals_flattened_single_rows():
    w = small(29, H=2, seq_lens=(10, 4, 13), q_lens=(3, 1, 2), packed=True, causal=False)
    o1, l1 = oracle.run(w)
    o2, l2 = oracle.run(_flatten(w))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_causal_row_equals_truncated_single_row_launch():
    """Row i of a causal request of length L and q rows sees exactly the first
    L - q + i + 1 rows: equal to a q=1 launch over that prefix."""
    w = small(31, H=2, seq_lens=(15, 9), q_lens=(4, 4))
    o1, l1 = oracle.run(w)
    for i in range(4):
        sl = (w.seq_lens - 4 + i + 1).astype(np.int32)
        wi = dataclasses.replace(w, q_lens=np.ones(2, np.int32), seq_lens=sl, max_seq_len_q=1,
                                 query=w.query[:, i:i + 1].copy())
        oi, li = oracle.run(wi)
        assert np.array_equal(o1.reshape(2, 4, 2, 512)[:, i], oi.reshape(2, 2, 512))
        assert np.array_equal(l1.reshape(2, 4, 2)[:, i], li.reshape(2, 2))


def test_split_kv_recombination_equals_single_pass():
    """Attention over [0, a) and [a, L) merged by their natural-log LSEs equals
    one pass over [0, L): lse = ln(e^lse1 + e^lse2), O = sum_k e^(lse_k - lse) O_k."""
    ps = 4
    w = small(37, H=3, ps=ps, seq_lens=(22, 13), q_lens=(1, 1), causal=False, bmm1=0.7)
    full_o, full_l = oracle.run(w)
    for a_pages in (1, 2, 3):
        a = a_pages * ps
        w1 = dataclasses.replace(w, seq_lens=np.full(2, a, np.int32))
        bt2 = np.full_like(w.block_tables, -1)
        bt2[:, :-a_pages] = w.block_tables[:, a_pages:]
        w2 = dataclasses.replace(w, seq_lens=(w.seq_lens - a).astype(np.int32), block_tables=bt2)
        o1, l1 = oracle.run(w1)
        o2, l2 = oracle.run(w2)
        lse = np.logaddexp(l1, l2)
        o = np.exp(l1 - lse)[..., None] * o1 + np.exp(l2 - lse)[..., None] * o2
        np.testing.assert_allclose(lse, full_l, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(o, full_o, rtol=1e-11, atol=1e-14)


def test_bmm2_is_linear_and_leaves_lse_alone():
    w = small(41, H=2, seq_lens=(9, 6), q_lens=(2, 2))
    o1, l1 = oracle.run(w)
    o2, l2 = oracle.run(dataclasses.replace(w, bmm2_scale=4.0))
    assert np.array_equal(o2, 4.0 * o1) and np.array_equal(l1, l2)


def test_large_scores_do_not_overflow():
    """bmm1 = 64 pushes scores to ~1e3: the max-shift keeps exp finite."""
    w = small(43, H=2, seq_lens=(9, 6), q_lens=(1, 1), bmm1=64.0)
    out, lse = oracle.run(w)
    assert np.isfinite(out).all() and np.isfinite(lse).all() and np.abs(lse).max() > 100
    bo, bl = brute.mla_decode(w.query_rows(), w.q_start(), w.kv_cache, w.block_tables,
                              w.seq_lens, kv_dtype="bf16", causal=True,
                              bmm1_scale=w.bmm1_scale, bmm2_scale=w.bmm2_scale)
    np.testing.assert_allclose(out, np.array(bo), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, np.array(bl), rtol=1e-13)


def test_fp8_workload_oracle_equals_dequantised_bf16_free_path():
    """The e4m3 oracle equals the same oracle fed the dequantised values with
    the folded scales: k_scale * e4m3 values re-expressed in fp64 through an
    exact path (float8 -> float64 by torch, then k_scale folded back)."""
    w = mi.build("fp8pin", 5, num_heads=2, page_size=8, seq_lens=[19, 7], q_lens=[2, 2],
                 packed=False, kv_dtype="e4m3", return_lse=True)
    out, lse = oracle.run(w)
    vals = as_f64(w.kv_cache, "e4m3")                      # exact dequantised codes
    Q = as_f64(w.query_rows())
    for b in range(2):
        L = int(w.seq_lens[b])
        j = np.arange(L)
        rows = vals[w.block_tables[b][j // 8], j % 8]
        for i in range(2):
            n = L - 2 + i + 1
            t = 2 * b + i
            for h in range(2):
                s = w.bmm1_scale * (rows[:n] @ Q[t, h])
                ref_l = np.logaddexp.reduce(s)
                p = np.exp(s - ref_l)
                ref_o = w.bmm2_scale * (p @ rows[:n, :512])
                assert lse[t, h] == pytest.approx(ref_l, rel=1e-12, abs=1e-12)
                np.testing.assert_allclose(out[t, h], ref_o, rtol=1e-10, atol=1e-14)


def test_poisoned_memory_is_never_read():
    """Tail rows, unused pages and unused table entries are NaN / invalid in
    every generated workload; a finite result shows none was dereferenced."""
    w = small(47, H=2, ps=8, seq_lens=(13, 3, 17), q_lens=(1, 1, 1))
    assert (w.block_tables < 0).any() or (w.block_tables >= w.num_pages).any()
    assert np.isnan(as_f64(w.kv_cache)).any()
    out, lse = oracle.run(w)
    assert np.isfinite(out).all() and np.isfinite(lse).all()


def test_thread_count_does_not_change_results():
    w = small(53, H=4, seq_lens=(21, 9, 14), q_lens=(2, 2, 2))
    o1, l1 = oracle.run(w, n_threads=1)
    o2, l2 = oracle.run(w, n_threads=5)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_selected_pairs_equal_full_run():
    w = small(59, H=4, seq_lens=(21, 9), q_lens=(3, 3))
    o, l = oracle.run(w)
    sel = np.array([[0, 1], [5, 3], [2, 0], [4, 2]])
    os_, ls = oracle.run(w, sel=sel)
    for k, (t, h) in enumerate(sel):
        assert np.array_equal(os_[k], o[t, h]) and ls[k] == l[t, h]


def test_tiny_workload_matches_recorded_oracle_output():
    """Regression record written by tests/golden/make_golden.py (oracle only)."""
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "tiny_oracle.json")) as f:
        doc = json.load(f)
    w = mi.tiny()
    out, lse = oracle.run(w)
    np.testing.assert_allclose(lse, np.array(doc["lse"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(out[..., doc["out_dims"]], np.array(doc["out"]), rtol=0, atol=1e-12)


def test_e4m3_query_equals_the_same_values_as_bf16():
    """Every e4m3 value is a bf16 value: an e4m3 query and the bf16 query
    holding the decoded values give bitwise-equal oracle outputs, so the query
    decoding is the only thing an e4m3 query changes."""
    w = small(11, H=3, seq_lens=(9, 14), q_lens=(2, 2), q_dtype="e4m3", bmm1=0.7)
    assert w.query.dtype == np.uint8 and w.q_scale is not None
    out8, lse8 = oracle.run(w)
    vals = as_f64(w.query, "e4m3")
    wb = dataclasses.replace(w, query=mi.bf16_bits(vals.astype(np.float32)), q_dtype="bf16")
    assert np.array_equal(as_f64(wb.query), vals)  # exact in bf16
    out16, lse16 = oracle.run(wb)
    assert np.array_equal(out8, out16) and np.array_equal(lse8, lse16)


def test_e4m3_query_quantisation_folds_q_scale_into_bmm1():
    """q_scale = amax / 448 maps the largest |q| to 448 and is folded into
    bmm1, so scores use the dequantised query: q_scale * e4m3(q / q_scale)."""
    wb = small(12, seq_lens=(7,), q_lens=(1,), bmm1=0.25)
    w8 = small(12, seq_lens=(7,), q_lens=(1,), bmm1=0.25, q_dtype="e4m3")
    q = as_f64(wb.query)
    assert np.abs(as_f64(w8.query, "e4m3")).max() == 448.0
    assert w8.bmm1_scale == np.float32(0.25 * w8.q_scale)
    deq = as_f64(w8.query, "e4m3") * w8.q_scale
    assert np.abs(deq - q).max() <= 2.0 ** -4 * np.abs(q).max()  # e4m3 keeps 3 mantissa bits


# ---------------------------------------------------------------- decode-context parallelism

@pytest.mark.parametrize("world,case", [
    (2, dict(seq_lens=(9, 14, 3), q_lens=(3, 3, 3), causal=True)),
    (3, dict(seq_lens=(9, 14, 4), q_lens=(2, 2, 2), causal=True)),
    (4, dict(seq_lens=(2, 11, 7), q_lens=(2, 2, 2), causal=True)),   # ranks with no rows
    (4, dict(seq_lens=(6, 3, 11), q_lens=(2, 3, 1), packed=True)),
    (3, dict(seq_lens=(7, 12), q_lens=(3, 3), causal=False)),
])
def test_dcp_rank_states_merge_to_the_single_pass(world, case):
    """Each rank's oracle state over its round-robin share of the rows, with the
    causal bound taken on global positions, merged across ranks by natural-log
    LSE (the vLLM FlashInferMLAImpl page's DCP merge) equals the one-pass
    oracle on the whole sequence.  A wrong global/local index map or a causal
    bound on local positions double-counts or drops rows and fails this."""
    w = small(61, H=2, **case)
    full_o, full_l = oracle.run(w)
    parts = [oracle.run(mi.dcp_shard(w, world, r)) for r in range(world)]
    lses = np.stack([p[1] for p in parts])
    lse = np.logaddexp.reduce(lses, axis=0)
    o = sum(np.exp(p[1] - lse)[..., None] * p[0] for p in parts)
    np.testing.assert_allclose(lse, full_l, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(o, full_o, rtol=1e-11, atol=1e-14)


def test_dcp_with_one_rank_is_the_plain_oracle():
    w = small(62, H=2, seq_lens=(9, 5), q_lens=(2, 2))
    o1, l1 = oracle.run(w)
    o2, l2 = oracle.run(mi.dcp_shard(w, 1, 0))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_dcp_rows_without_keys_are_empty_sums():
    """Global length 2, q = 2, four ranks: rank 1 sees its one row only from
    query row 1 on, ranks 2 and 3 hold nothing, so those rows are the empty
    sum (O = 0, lse = -inf), which the LSE merge ignores."""
    w = small(63, H=2, seq_lens=(2,), q_lens=(2,))
    o1, l1 = oracle.run(mi.dcp_shard(w, 4, 1))
    assert np.all(np.isneginf(l1[0])) and np.all(o1[0] == 0) and np.all(np.isfinite(l1[1]))
    for r in (2, 3):
        o, l = oracle.run(mi.dcp_shard(w, 4, r))
        assert np.all(np.isneginf(l)) and np.all(o == 0)


@pytest.mark.parametrize("world,rank,causal", [(2, 1, True), (3, 0, True), (3, 2, True),
                                               (4, 3, False)])
def test_dcp_c_oracle_matches_python_brute_force(world, rank, causal):
    w = small(64, H=2, seq_lens=(9, 14, 5), q_lens=(3, 3, 3), causal=causal, bmm1=0.5)
    sh = mi.dcp_shard(w, world, rank)
    out, lse = oracle.run(sh)
    bo, bl = brute.mla_decode(sh.query_rows(), sh.q_start(), sh.kv_cache, sh.block_tables,
                              sh.seq_lens, kv_dtype=sh.kv_dtype, causal=sh.causal,
                              bmm1_scale=sh.bmm1_scale, bmm2_scale=sh.bmm2_scale,
                              cp_world=world, cp_rank=rank, seq_lens_global=sh.seq_lens_global)
    bl = np.array(bl)
    assert np.array_equal(np.isneginf(lse), np.isneginf(bl))
    fin = np.isfinite(bl)
    np.testing.assert_allclose(out, np.array(bo), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse[fin], bl[fin], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- sparse top-k selection

def _with_lists(w, lists):
    """w with the given per-token position lists, -1 padded to a common k."""
    k = max(len(x) for x in lists)
    idx = np.full((len(lists), k), -1, dtype=np.int32)
    for t, x in enumerate(lists):
        idx[t, :len(x)] = x
    return dataclasses.replace(w, sparse_idx=idx)


@pytest.mark.parametrize("causal", [True, False])
def test_sparse_list_of_every_position_is_the_dense_pass(causal):
    """A token whose list holds every row 0 .. L-1 once, in any order, sees
    exactly the dense set; the plan's causal flag is not consulted."""
    w = small(81, H=2, seq_lens=(9, 14, 5), q_lens=(2, 2, 2), causal=causal)
    rng = np.random.default_rng(3)
    qs = w.q_start()
    lists = [list(rng.permutation(int(w.seq_lens[b])))
             for b in range(w.batch) for _ in range(int(qs[b + 1] - qs[b]))]
    o_s, l_s = oracle.run(_with_lists(w, lists))
    o_d, l_d = oracle.run(w, causal=False)
    np.testing.assert_allclose(o_s, o_d, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(l_s, l_d, rtol=1e-13, atol=1e-13)


def test_sparse_list_of_the_causal_prefix_is_the_causal_pass():
    """Token i's list = its causal prefix 0 .. L-q+i (padded with -1 and with
    positions at or past L, which are unused) gives the causal result."""
    w = small(82, H=3, seq_lens=(9, 14, 6), q_lens=(3, 1, 2), packed=True)
    qs = w.q_start()
    lists = []
    for b in range(w.batch):
        L, q = int(w.seq_lens[b]), int(qs[b + 1] - qs[b])
        for i in range(q):
            lists.append(list(range(L - q + i, -1, -1)) + [L, -1, L + 100, -7])
    o_s, l_s = oracle.run(_with_lists(w, lists))
    o_c, l_c = oracle.run(w, causal=True)
    np.testing.assert_allclose(o_s, o_c, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(l_s, l_c, rtol=1e-13, atol=1e-13)


def test_sparse_single_position_returns_that_row():
    """One listed row j: O = bmm2 * V_j and lse = bmm1 * q.k_j (softmax of one)."""
    w = small(83, H=2, seq_lens=(9, 14), q_lens=(1, 1), bmm1=0.3, bmm2=1.5)
    picks = [6, 11]
    out, lse = oracle.run(_with_lists(w, [[-1, picks[0], 9], [picks[1], -1, 14]]))
    Q = as_f64(w.query_rows())
    for b, j in enumerate(picks):
        kj = gather(w, b)[j]
        for h in range(w.num_heads):
            assert lse[b, h] == pytest.approx(w.bmm1_scale * np.dot(Q[b, h], kj), rel=1e-13,
                                              abs=1e-13)
            np.testing.assert_allclose(out[b, h], w.bmm2_scale * kj[:512], rtol=1e-14, atol=0)


def test_sparse_repeated_position_counts_each_listing():
    """[j, j] weighs row j twice: O is unchanged and lse grows by exactly ln 2;
    with Q = 0, [a, a, b] gives O = (2 V_a + V_b) / 3 and lse = ln 3."""
    w = small(84, H=2, seq_lens=(12,), q_lens=(1,), bmm2=1.0)
    o1, l1 = oracle.run(_with_lists(w, [[5]]))
    o2, l2 = oracle.run(_with_lists(w, [[5, 5]]))
    np.testing.assert_allclose(o2, o1, rtol=1e-14, atol=0)
    np.testing.assert_allclose(l2, l1 + math.log(2.0), rtol=0, atol=1e-13)
    wz = dataclasses.replace(w, query=np.zeros_like(w.query))
    o3, l3 = oracle.run(_with_lists(wz, [[3, 3, 8]]))
    rows = gather(w, 0)
    np.testing.assert_allclose(l3, math.log(3.0), atol=1e-14)
    np.testing.assert_allclose(o3[0, 0], (2 * rows[3, :512] + rows[8, :512]) / 3, rtol=1e-13,
                               atol=1e-16)


def test_sparse_list_with_no_usable_entry_is_the_empty_sum():
    w = small(85, H=2, seq_lens=(4, 9), q_lens=(1, 1))
    out, lse = oracle.run(_with_lists(w, [[-1, 4, 100], [3, -1, -1]]))
    assert np.all(np.isneginf(lse[0])) and np.all(out[0] == 0)
    assert np.all(np.isfinite(lse[1]))


def test_sparse_order_of_the_list_does_not_matter():
    w = mi.with_topk(small(86, H=2, seq_lens=(40, 23), q_lens=(2, 2)), 16, seed=5)
    rng = np.random.default_rng(8)
    shuffled = np.stack([rng.permutation(r) for r in w.sparse_idx])
    o1, l1 = oracle.run(w)
    o2, l2 = oracle.run(dataclasses.replace(w, sparse_idx=shuffled))
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(l2, l1, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("case", [
    dict(seq_lens=(40, 23), q_lens=(2, 2), k=16),
    dict(seq_lens=(9, 30, 5), q_lens=(3, 1, 2), packed=True, k=8, kv_dtype="e4m3", bmm1=0.5),
    dict(seq_lens=(70,), q_lens=(1,), k=32, q_dtype="e4m3", bmm1=2.0),
])
def test_sparse_c_oracle_matches_python_brute_force(case):
    k = case.pop("k")
    w = mi.with_topk(small(87, H=2, **case), k, seed=9)
    # add a repeated entry, an out-of-range one and a -1 to every full list
    idx = w.sparse_idx.copy()
    idx[:, -3] = idx[:, 0]
    idx[:, -2] = 10 ** 6
    idx[:, -1] = -1
    w = dataclasses.replace(w, sparse_idx=idx)
    out, lse = oracle.run(w)
    bo, bl = brute.mla_decode(w.query_rows(), w.q_start(), w.kv_cache, w.block_tables,
                              w.seq_lens, kv_dtype=w.kv_dtype, causal=w.causal,
                              bmm1_scale=w.bmm1_scale, bmm2_scale=w.bmm2_scale,
                              q_dtype=w.q_dtype, sparse_idx=w.sparse_idx)
    np.testing.assert_allclose(out, np.array(bo), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, np.array(bl), rtol=1e-12, atol=1e-12)


def test_sparse_lists_stay_inside_each_tokens_causal_prefix():
    """The input generator's lists: distinct, inside [0, L - q + i], -1 padded."""
    w = mi.with_topk(small(88, H=2, seq_lens=(40, 7, 100), q_lens=(3, 3, 3)), 24, seed=2)
    qs = w.q_start()
    for b in range(w.batch):
        L, q = int(w.seq_lens[b]), int(qs[b + 1] - qs[b])
        for i in range(q):
            row = w.sparse_idx[int(qs[b]) + i]
            used = row[row >= 0]
            assert len(used) == min(24, L - q + i + 1) and np.all(row[len(used):] == -1)
            assert len(set(used.tolist())) == len(used) and used.max() <= L - q + i


def test_sparse_selection_is_refused_with_decode_context_parallelism():
    w = mi.with_topk(small(89, H=2, seq_lens=(9, 5), q_lens=(1, 1)), 4)
    with pytest.raises(RuntimeError):
        oracle.run(dataclasses.replace(w, cp_world=2, cp_rank=0,
                                       seq_lens_global=w.seq_lens.copy()))
