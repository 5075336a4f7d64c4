"""Seeded synthetic workloads for batched paged MLA decode.

This module draws inputs and nothing else: query rows, a paged latent KV pool,
page tables, KV lengths, packed query offsets and the two scale factors.  It
holds none of the attention arithmetic, so both the fp64 oracle (``oracle/``)
and the CUDA library (``paged_mla_decode_03_gb300``) can be fed from it without
sharing any computation.

Shapes follow the problem statement of the FlashInfer page
"prims_ts_batch_decode_with_kv_cache_mla" (signature and parameter text):

* fixed query   ``[B, SQ, H, 576]``; packed query ``[total_q, H, 576]`` with
  ``qo_indptr`` holding B + 1 cumulative offsets;
* ``kv_cache``  ``[num_pages, page_size, 576]`` (512 latent + 64 RoPE dims, one
  copy: V is the first 512 dims of the same rows);
* ``block_tables`` ``[B, max_pages_per_req]`` int32, ``seq_lens`` ``[B]`` int32.

Values are N(0, 1) rounded to bf16 (round-to-nearest-even).  The fp8 variant
quantises N(0, 1) KV to e4m3 with a per-tensor ``k_scale = amax / 448`` and
folds it into both scales, as the vLLM ``FlashInferMLAImpl.forward_mqa`` page
does for a quantised cache (``bmm1 *= k_scale``, ``bmm2 *= k_scale``).

Memory the computation must never touch is poisoned: rows at or past
``seq_lens[b]`` in a request's last page and every page no request uses hold
NaN, and page-table entries past a request's last page hold -1 or an
out-of-range page id.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

HEAD_DIM_QK = 576      # 512 latent (kv_lora_rank) + 64 RoPE dims
HEAD_DIM_V = 512       # V = first 512 dims of each cache row
BF16_NAN = 0x7FC0
E4M3_NAN = 0x7F
E4M3_MAX = 448.0


@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    batch: int
    num_heads: int
    page_size: int
    packed: bool
    causal: bool
    return_lse: bool
    kv_dtype: str                      # "bf16" or "e4m3"
    q_lens: np.ndarray                 # [B] int32 (uniform when fixed)
    seq_lens: np.ndarray               # [B] int32
    max_seq_len_q: int
    max_seq_len: int
    query: np.ndarray                  # uint16 bf16 bits or uint8 e4m3 codes (q_dtype),
                                       # [B,SQ,H,576] or [total_q,H,576]
    qo_indptr: Optional[np.ndarray]    # [B+1] int32 when packed
    kv_cache: np.ndarray               # uint16 (bf16) or uint8 (e4m3), [pages, ps, 576]
    block_tables: np.ndarray           # [B, max_pages_per_req] int32
    bmm1_scale: float                  # exactly representable in fp32
    bmm2_scale: float
    k_scale: Optional[float] = None
    q_dtype: str = "bf16"              # "bf16" or "e4m3" (query quantised, q_scale in bmm1)
    q_scale: Optional[float] = None
    # decode-context parallelism: this workload is rank cp_rank's share of a
    # sequence sharded over cp_world ranks (seq_lens local, seq_lens_global global)
    cp_world: int = 1
    cp_rank: int = 0
    seq_lens_global: Optional[np.ndarray] = None
    # sparse top-k selection: int32 [tokens, k] logical KV positions per query
    # token (-1: unused entry), or None for the causal / dense mask
    sparse_idx: Optional[np.ndarray] = None

    @property
    def sparse_k(self) -> int:
        return 0 if self.sparse_idx is None else int(self.sparse_idx.shape[1])

    @property
    def total_q(self) -> int:
        return int(self.q_lens.sum())

    @property
    def num_pages(self) -> int:
        return int(self.kv_cache.shape[0])

    @property
    def sq(self) -> int:
        """Per-request query length of a fixed launch (the bound when packed)."""
        return int(self.max_seq_len_q)

    def q_start(self) -> np.ndarray:
        """[B+1] token offsets of each request's first query row."""
        if self.packed:
            return self.qo_indptr.astype(np.int64)
        return np.arange(self.batch + 1, dtype=np.int64) * self.sq

    def query_rows(self) -> np.ndarray:
        """The query viewed as [tokens, H, 576] (fixed shape flattened)."""
        return self.query.reshape(-1, self.num_heads, HEAD_DIM_QK)


def f32(x: float) -> float:
    """Round a Python float to the nearest fp32 value."""
    return float(np.float32(x))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 array -> bf16 bit patterns (round to nearest even) as uint16."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def e4m3_bits(x: np.ndarray) -> np.ndarray:
    """float32 array -> float8_e4m3fn bit patterns (round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _normal(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(size=shape, dtype=np.float32)


def build(name: str, seed: int, *, num_heads: int, page_size: int,
          seq_lens, q_lens, packed: bool, causal: bool = True,
          return_lse: bool = False, kv_dtype: str = "bf16",
          pool_factor: float = 1.25, bmm1_scale: float = 1.0 / math.sqrt(192.0),
          bmm2_scale: float = 1.0, num_pages: Optional[int] = None,
          block_tables: Optional[np.ndarray] = None, poison: bool = True,
          max_seq_len_q: Optional[int] = None, max_seq_len: Optional[int] = None,
          rng: Optional[np.random.Generator] = None, q_dtype: str = "bf16") -> Workload:
    """Draw one workload.  Draw order: pool permutation, query, KV values."""
    rng = rng if rng is not None else np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    q_lens = np.asarray(q_lens, dtype=np.int32)
    B = int(seq_lens.shape[0])
    H = int(num_heads)
    ps = int(page_size)
    if not packed and B > 0:
        assert np.all(q_lens == q_lens[0]), "fixed-shape launches share one q_len"
    n_pages = (seq_lens.astype(np.int64) + ps - 1) // ps
    needed = int(n_pages.sum())
    max_pages = max(1, int(n_pages.max()) if B else 1)

    if block_tables is None:
        pool = num_pages if num_pages is not None else max(1, math.ceil(pool_factor * needed))
        assert pool >= needed
        perm = rng.permutation(pool).astype(np.int32)
        block_tables = np.empty((B, max_pages), dtype=np.int32)
        pos = 0
        for b in range(B):
            k = int(n_pages[b])
            block_tables[b, :k] = perm[pos:pos + k]
            pos += k
            tail = block_tables[b, k:]
            # unused entries: alternate -1 and an out-of-range page id
            tail[0::2] = -1
            tail[1::2] = pool + 7
    else:
        block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
        pool = int(num_pages)

    if packed:
        qo_indptr = np.zeros(B + 1, dtype=np.int32)
        qo_indptr[1:] = np.cumsum(q_lens)
        total_q = int(qo_indptr[-1])
        qshape = (total_q, H, HEAD_DIM_QK)
        sq = int(max_seq_len_q if max_seq_len_q is not None else (q_lens.max() if B else 1))
    else:
        qo_indptr = None
        sq = int(q_lens[0]) if B else int(max_seq_len_q or 1)
        qshape = (B, sq, H, HEAD_DIM_QK)
    q32 = _normal(rng, qshape)
    q_scale = None
    if q_dtype == "bf16":
        query = bf16_bits(q32)
    elif q_dtype == "e4m3":
        # per-tensor q_scale = amax / 448, folded into bmm1 (as for k_scale)
        q_scale = f32(float(np.abs(q32).max()) / E4M3_MAX) if q32.size else 1.0
        query = e4m3_bits(q32 / np.float32(q_scale))
        bmm1_scale = bmm1_scale * q_scale
    else:
        raise ValueError(q_dtype)
    del q32

    kv32 = _normal(rng, (pool, ps, HEAD_DIM_QK))
    used = np.zeros((pool, ps), dtype=bool)
    for b in range(B):
        L = int(seq_lens[b])
        for p in range(int(n_pages[b])):
            rows = min(ps, L - p * ps)
            used[block_tables[b, p], :rows] = True

    k_scale = None
    if kv_dtype == "bf16":
        kv = bf16_bits(kv32)
        if poison:
            kv[~used] = BF16_NAN
    elif kv_dtype == "e4m3":
        amax = float(np.abs(kv32[used]).max()) if used.any() else 1.0
        k_scale = f32(amax / E4M3_MAX)
        kv = e4m3_bits(kv32 / np.float32(k_scale))
        if poison:
            kv[~used] = E4M3_NAN
        bmm1_scale = bmm1_scale * k_scale
        bmm2_scale = bmm2_scale * k_scale
    else:
        raise ValueError(kv_dtype)
    del kv32

    return Workload(
        name=name, seed=seed, batch=B, num_heads=H, page_size=ps, packed=packed,
        causal=causal, return_lse=return_lse, kv_dtype=kv_dtype, q_lens=q_lens,
        seq_lens=seq_lens,
        max_seq_len_q=sq,
        max_seq_len=int(max_seq_len if max_seq_len is not None else (seq_lens.max() if B else 1)),
        query=query, qo_indptr=qo_indptr, kv_cache=kv, block_tables=block_tables,
        bmm1_scale=f32(bmm1_scale), bmm2_scale=f32(bmm2_scale), k_scale=k_scale,
        q_dtype=q_dtype, q_scale=q_scale)


# ---------------------------------------------------------------------------
# The five workloads.  Seeds are 1000 + workload index.  ``scale`` < 1 shrinks
# the batch and the length ranges for parity runs the oracle finishes quickly;
# ``scale`` = 1 is the full-size workload.
# ---------------------------------------------------------------------------

def tiny(seed: int = 1001, poison: bool = True) -> Workload:
    """B=2, H=16, q_len=1, seq_lens {37, 64}, page_size 32, 8 physical pages,
    block_tables = a seeded permutation of the 8 pages viewed as [2, 4]."""
    rng = np.random.default_rng(seed)
    bt = rng.permutation(8).astype(np.int32).reshape(2, 4)
    return build("tiny_b2_h16_q1_ps32", seed, num_heads=16, page_size=32,
                 seq_lens=[37, 64], q_lens=[1, 1], packed=False, return_lse=True,
                 num_pages=8, block_tables=bt, poison=poison, rng=rng)


def _uniform_lens(rng, lo, hi, n):
    return rng.integers(lo, hi, size=n, endpoint=True).astype(np.int32)


def deepseek_v3(seed: int = 1002, batch: int = 64, lo: int = 1024, hi: int = 8192,
                return_lse: bool = False, poison: bool = True, q_dtype: str = "bf16") -> Workload:
    """B=64, H=128, q_len=1, page_size 64, seq_lens ~ U[1024, 8192]."""
    rng = np.random.default_rng(seed)
    L = _uniform_lens(rng, lo, hi, batch)
    return build(f"deepseek_v3_b{batch}_h128_q1_ps64", seed, num_heads=128, page_size=64,
                 seq_lens=L, q_lens=np.ones(batch, np.int32), packed=False,
                 return_lse=return_lse, poison=poison, rng=rng, q_dtype=q_dtype)


def mtp(seed: int = 1003, batch: int = 32, lo: int = 2048, hi: int = 16384,
        q_len: int = 4, return_lse: bool = False, poison: bool = True,
        q_dtype: str = "bf16") -> Workload:
    """B=32, H=128, fixed q_len=4, bottom-right causal, seq_lens ~ U[2048, 16384]."""
    rng = np.random.default_rng(seed)
    L = _uniform_lens(rng, lo, hi, batch)
    return build(f"mtp_b{batch}_h128_q{q_len}_ps64", seed, num_heads=128, page_size=64,
                 seq_lens=L, q_lens=np.full(batch, q_len, np.int32), packed=False,
                 return_lse=return_lse, poison=poison, rng=rng, q_dtype=q_dtype)


def ragged(seed: int = 1004, batch: int = 128, median: float = 4096.0, sigma: float = 1.0,
           max_len: int = 32768, poison: bool = True) -> Workload:
    """B=128, H=16, packed q_len ~ U{1..8} via qo_indptr (max_seq_len_q = 8),
    page_size 32, seq_lens lognormal (median 4096, sigma 1) clipped to
    [q_len, 32768], output plus LSE."""
    rng = np.random.default_rng(seed)
    q = rng.integers(1, 8, size=batch, endpoint=True).astype(np.int32)
    raw = np.rint(np.exp(rng.normal(math.log(median), sigma, size=batch)))
    L = np.clip(raw, q, max_len).astype(np.int32)
    return build(f"ragged_b{batch}_h16_packed_ps32", seed, num_heads=16, page_size=32,
                 seq_lens=L, q_lens=q, packed=True, return_lse=True, max_seq_len_q=8,
                 poison=poison, rng=rng)


def fp8_long(seed: int = 1005, batch: int = 8, lo: int = 65536, hi: int = 131072,
             q_len: int = 2, return_lse: bool = False, poison: bool = True,
             q_dtype: str = "bf16") -> Workload:
    """B=8, H=128, fixed q_len=2, page_size 64, seq_lens ~ U[65536, 131072],
    e4m3 KV with k_scale = amax/448 folded into bmm1 and bmm2."""
    rng = np.random.default_rng(seed)
    L = _uniform_lens(rng, lo, hi, batch)
    return build(f"fp8_long_b{batch}_h128_q{q_len}_ps64", seed, num_heads=128, page_size=64,
                 seq_lens=L, q_lens=np.full(batch, q_len, np.int32), packed=False,
                 kv_dtype="e4m3", return_lse=return_lse, poison=poison, rng=rng,
                 q_dtype=q_dtype)


def prefill(seed: int = 1006, batch: int = 512, q_lo: int = 24, q_hi: int = 48,
            max_len: int = 2048, poison: bool = True) -> Workload:
    """Prefill through the decode path (the FlashInfer issue "Support
    cum_seq_lens_q in trtllm_batch_decode_with_kv_cache_mla", point 1):
    B=512, H=128, packed q_len ~ U{24..48} (about 18k query tokens),
    page_size 64, seq_lens ~ U[q_len + 1, 2048], bottom-right causal, out + LSE.
    Not one of the five decode workloads: a size check of the packed path."""
    rng = np.random.default_rng(seed)
    q = rng.integers(q_lo, q_hi, size=batch, endpoint=True).astype(np.int32)
    L = rng.integers(q + 1, max_len, endpoint=True).astype(np.int32)
    return build(f"prefill_b{batch}_h128_packed_ps64", seed, num_heads=128, page_size=64,
                 seq_lens=L, q_lens=q, packed=True, return_lse=True, max_seq_len_q=q_hi,
                 poison=poison, rng=rng)


def with_topk(w: Workload, k: int, seed: int = 0) -> Workload:
    """``w`` with a sparse top-k list per query token.

    The pages name the launcher argument ``sparse_mla_top_k`` and nothing
    more, so the lists are drawn to look like an indexer's output: token i
    of a request with q tokens and L cached rows picks min(k, L - q + i + 1)
    distinct positions of its causal prefix [0, L - q + i], uniformly at
    random and in random order, and pads the rest of its k entries with -1.
    Sampling only: no attention arithmetic.
    """
    rng = np.random.default_rng(seed)
    qs = w.q_start()
    idx = np.full((int(qs[-1]), int(k)), -1, dtype=np.int32)
    for b in range(w.batch):
        L = int(w.seq_lens[b])
        q = int(qs[b + 1] - qs[b])
        for i in range(q):
            n = max(0, L - q + i + 1)
            m = min(int(k), n)
            if m == 0:
                continue
            if n <= 4 * m:
                pick = rng.permutation(n)[:m]
            else:  # sparse pick from a long prefix without an O(n) permutation
                pick = rng.choice(n, size=m, replace=False)
            idx[int(qs[b]) + i, :m] = pick.astype(np.int32)
    return dataclasses.replace(w, name=f"{w.name}_top{k}", sparse_idx=idx)


def sparse_topk(seed: int = 1007, batch: int = 64, k: int = 2048, lo: int = 3072,
                hi: int = 12288, q_len: int = 1, return_lse: bool = False,
                poison: bool = True, kv_dtype: str = "bf16") -> Workload:
    """Sparse top-k decode: B=64, H=128, q_len=1, page_size 64,
    seq_lens ~ U[3072, 12288], k = 2048 listed positions per token drawn by
    ``with_topk`` (every list full: L > k).  The pages fix no sparse workload;
    the shape is the headline decode shape with the selection on top."""
    rng = np.random.default_rng(seed)
    L = _uniform_lens(rng, lo, hi, batch)
    w = build(f"sparse_b{batch}_h128_q{q_len}_ps64", seed, num_heads=128, page_size=64,
              seq_lens=L, q_lens=[q_len] * batch, packed=False, causal=True,
              return_lse=return_lse, poison=poison, kv_dtype=kv_dtype, rng=rng)
    return with_topk(w, k, seed + 1)


WORKLOADS = {
    "tiny": tiny,
    "deepseek_v3": deepseek_v3,
    "mtp": mtp,
    "ragged": ragged,
    "fp8_long": fp8_long,
    "prefill": prefill,
    "sparse_topk": sparse_topk,
}


def dcp_shard(w: Workload, world: int, rank: int, seed: int = 0) -> Workload:
    """Rank ``rank``'s share of workload ``w`` under decode-context
    parallelism over ``world`` ranks.

    The KV rows of each request are dealt round robin: global row g lives on
    rank g mod world as its local row g div world (the pages do not state the
    layout; this is the plainest reading, with an interleave of one row).  The
    rank's rows are copied, unchanged, into a fresh paged pool of the same
    page size (1.25x the pages needed, shuffled, unused rows NaN-poisoned, as
    ``build`` does); ``seq_lens`` become the local counts, which may be 0, and
    ``seq_lens_global`` keeps the global lengths.  Query, scales and flags are
    w's.  Pure data movement: no attention arithmetic.
    """
    assert w.cp_world == 1 and 0 <= rank < world
    rng = np.random.default_rng(seed + 7919 * rank)
    ps = w.page_size
    B = w.batch
    local = [np.arange(rank, int(L), world, dtype=np.int64) for L in w.seq_lens]
    n_loc = np.array([len(g) for g in local], dtype=np.int32)
    n_pages = (n_loc.astype(np.int64) + ps - 1) // ps
    needed = int(n_pages.sum())
    pool = max(1, math.ceil(1.25 * needed))
    perm = rng.permutation(pool).astype(np.int32)
    max_pages = max(1, int(n_pages.max()) if B else 1)
    bt = np.empty((B, max_pages), dtype=np.int32)
    nan = BF16_NAN if w.kv_dtype == "bf16" else E4M3_NAN
    kv = np.full((pool, ps, HEAD_DIM_QK), nan, dtype=w.kv_cache.dtype)
    pos = 0
    for b in range(B):
        k = int(n_pages[b])
        bt[b, :k] = perm[pos:pos + k]
        pos += k
        tail = bt[b, k:]
        tail[0::2] = -1
        tail[1::2] = pool + 7
        g = local[b]
        src = w.kv_cache[w.block_tables[b, g // ps], g % ps]      # [n_loc, 576]
        j = np.arange(len(g))
        kv[bt[b, j // ps], j % ps] = src
    return dataclasses.replace(
        w, name=f"{w.name}_dcp{rank}of{world}", seq_lens=n_loc, kv_cache=kv, block_tables=bt,
        max_seq_len=max(1, int(n_loc.max()) if B else 1), cp_world=world, cp_rank=rank,
        seq_lens_global=w.seq_lens.copy())


def permute_pages(w: Workload, seed: int) -> Workload:
    """Same logical cache with physical pages shuffled and block_tables rewritten.

    Every valid entry of ``block_tables`` is remapped; poisoned entries are kept.
    """
    rng = np.random.default_rng(seed)
    P = w.num_pages
    perm = rng.permutation(P)               # old page p moves to slot perm[p]
    kv = np.empty_like(w.kv_cache)
    kv[perm] = w.kv_cache
    bt = w.block_tables.copy()
    valid = (bt >= 0) & (bt < P)
    bt[valid] = perm[bt[valid]]
    return dataclasses.replace(w, kv_cache=kv, block_tables=bt.astype(np.int32))
