"""Seeded random configurations through the C ABI against the fp64 oracle.

Each case draws one launch at random:
- shape: head count, page size, batch, fixed or packed query lengths;
- mask (causal or dense), cache and query dtypes, LSE or none, bmm1;
- for an e4m3 cache, the FP8-MMA path or the exact widening path;
- sparse top-k lists, with random padding, repeated and out-of-range entries;
- a workspace filled with a random byte.

It compares every (token, head) pair when the case is small and a seeded sample otherwise, and
requires a zero status word.  The point is breadth: combinations the hand-written cases do not
reach.
"""
import dataclasses
import math

import numpy as np
import pytest

import mla_inputs as mi
import oracle
from harness import check, device_status, results, run, sample_pairs, to_device

pytestmark = pytest.mark.gpu

N_CASES = 96


def draw(seed):
    rng = np.random.default_rng(50_000 + seed)
    H = int(rng.choice([16, 32, 64, 128]))
    ps = int(rng.choice([32, 64]))
    B = int(rng.integers(1, 24))
    packed = bool(rng.integers(2))
    causal = bool(rng.random() < 0.75)
    if packed:
        q = rng.integers(1, 9, size=B).astype(np.int32)
    else:
        q = np.full(B, int(rng.integers(1, 6)), np.int32)
    L = rng.integers(np.maximum(q, 1), int(rng.choice([80, 600, 2500])), endpoint=True).astype(np.int32)
    kv_dtype = "e4m3" if rng.random() < 0.3 else "bf16"
    q_dtype = "e4m3" if rng.random() < 0.2 else "bf16"
    bmm1 = float(rng.choice([1.0 / math.sqrt(192.0), 0.5, 1.0]))
    w = mi.build(f"fuzz{seed}", 50_000 + seed, num_heads=H, page_size=ps, seq_lens=L, q_lens=q,
                 packed=packed, causal=causal, return_lse=bool(rng.integers(2)), kv_dtype=kv_dtype,
                 q_dtype=q_dtype, bmm1_scale=bmm1, max_seq_len_q=int(q.max()) + int(rng.integers(0, 3)) if packed else None,
                 rng=rng)
    if rng.random() < 0.3:
        k = int(rng.choice([16, 64, 100, 256]))
        w = mi.with_topk(w, k, seed=seed)
        idx = w.sparse_idx.copy()
        qs = w.q_start()
        # sprinkle repeats, -1 and past-the-end entries into some rows
        for t in range(idx.shape[0]):
            if rng.random() < 0.5:
                b = int(np.searchsorted(qs[1:], t, side="right"))
                m = int(rng.integers(1, max(2, k // 4)))
                pos = rng.choice(k, size=min(m, k), replace=False)
                choice = rng.integers(3, size=pos.size)
                used = idx[t][idx[t] >= 0]
                for p_, c in zip(pos, choice):
                    if c == 0 and used.size:
                        idx[t, p_] = int(rng.choice(used))
                    elif c == 1:
                        idx[t, p_] = -1
                    else:
                        idx[t, p_] = int(w.seq_lens[b]) + int(rng.integers(0, 5))
        w = dataclasses.replace(w, sparse_idx=idx)
    fill = int(rng.integers(0, 256))
    widen = w.kv_dtype == "e4m3" and bool(rng.integers(2))
    return w, fill, widen


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_configuration_matches_oracle(seed):
    w, fill, widen = draw(seed)
    d = to_device(w, workspace_fill=fill, e4m3_widen=widen)
    run(w, d)
    out, lse = results(d)
    assert device_status(d) == 0, f"{w.name}: status {device_status(d)}"
    H = w.num_heads
    tokens = w.total_q
    if tokens * H <= 4096:
        ref_o, ref_l = oracle.run(w)
        check(w.kv_dtype, out.reshape(-1, H, 512), ref_o, lse,
              ref_l if lse is not None else None, what=w.name)
    else:
        sel = sample_pairs(w, 96, seed=seed)
        ref_o, ref_l = oracle.run(w, sel=sel)
        got_o = out.reshape(-1, H, 512)[sel[:, 0], sel[:, 1]]
        got_l = lse[sel[:, 0], sel[:, 1]] if lse is not None else None
        check(w.kv_dtype, got_o, ref_o, got_l, ref_l if got_l is not None else None, what=w.name)
        assert np.isfinite(out).all(), f"{w.name}: non-finite output"
