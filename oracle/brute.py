"""Pure-Python brute force of paged MLA decode -- TEST INFRASTRUCTURE ONLY.

Written independently of ``oracle.c`` to cross-check it on tiny inputs: the
bit decoding, the page walk, the mask predicate and the summation order are
all expressed differently here.  Every sum uses ``math.fsum`` (exactly
rounded), so on tiny inputs the two implementations must agree to ~1e-12.

The mask follows the FlashInfer page "prims_ts_batch_decode_with_kv_cache_mla":
query row i of a request with q rows and L cached rows attends through KV row
L - q + i; written here as the predicate ``j - (L - q) <= i`` (causal) or
``j < L`` (dense).  Under decode-context parallelism (the vLLM
``FlashInferMLAImpl`` page passes cp_world, cp_rank and the global KV lengths
to the kernel) local row j of rank r holds global row j * W + r, and the
causal predicate is applied to that global position against the global
length: ``(j * W + r) - (Lg - q) <= i``.  Under sparse top-k selection the
token's list of logical positions is walked as given: an entry e is used iff
``0 <= e < L``, and each use contributes one term (a repeated entry counts
once per listing).
"""
from __future__ import annotations

import math
import struct


def bf16_value(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def e4m3_value(bits: int) -> float:
    bits = int(bits) & 0xFF
    sign = -1.0 if bits & 0x80 else 1.0
    exp_field = (bits & 0x78) >> 3
    frac = (bits & 0x07) / 8.0
    if exp_field == 15 and (bits & 0x07) == 7:
        return float("nan")
    if exp_field == 0:
        return sign * frac * 2.0 ** -6
    return sign * (1.0 + frac) * 2.0 ** (exp_field - 7)


def mla_decode(query, q_start, kv_cache, block_tables, seq_lens, *, kv_dtype, causal,
               bmm1_scale, bmm2_scale, q_dtype="bf16", cp_world=1, cp_rank=0,
               seq_lens_global=None, sparse_idx=None):
    """Return (out[tokens][H][512], lse[tokens][H]) as nested Python lists.
    A row with no visible key gets zeros and -inf."""
    decode = bf16_value if kv_dtype == "bf16" else e4m3_value
    q_decode = bf16_value if q_dtype == "bf16" else e4m3_value
    tokens, H, D = query.shape
    ps = kv_cache.shape[1]
    out = [[None] * H for _ in range(tokens)]
    lse = [[None] * H for _ in range(tokens)]
    for b in range(len(seq_lens)):
        L = int(seq_lens[b])
        t0, t1 = int(q_start[b]), int(q_start[b + 1])
        q = t1 - t0
        rows = []
        for j in range(L):
            page = int(block_tables[b][j // ps])
            rows.append([decode(x) for x in kv_cache[page][j % ps]])
        if cp_world > 1:
            Lg = int(seq_lens_global[b])

            def seen(j, i):
                return (j * cp_world + cp_rank) - (Lg - q) <= i
        else:
            def seen(j, i):
                return j - (L - q) <= i
        for i in range(q):
            if sparse_idx is not None:
                visible = [int(e) for e in sparse_idx[t0 + i] if 0 <= int(e) < L]
            else:
                visible = [j for j in range(L) if (seen(j, i) if causal else True)]
            if not visible:
                for h in range(H):
                    lse[t0 + i][h] = float("-inf")
                    out[t0 + i][h] = [0.0] * 512
                continue
            for h in range(H):
                qv = [q_decode(x) for x in query[t0 + i][h]]
                s = [bmm1_scale * math.fsum(qv[d] * rows[j][d] for d in range(D))
                     for j in visible]
                mx = max(s)
                w = [math.exp(x - mx) for x in s]
                z = math.fsum(w)
                lse[t0 + i][h] = mx + math.log(z)
                out[t0 + i][h] = [bmm2_scale * math.fsum(w[k] * rows[j][d]
                                                          for k, j in enumerate(visible)) / z
                                  for d in range(512)]
    return out, lse
