"""fp64 CPU oracle for batched paged MLA decode -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The CUDA library (``paged_mla_decode_03_gb300``)
never imports it, and this package imports nothing from the library.

Two independent implementations of the same definition live here:

* ``oracle.c`` -- plain C, fp64, threaded over (token, head) pairs; the
  workhorse for parity runs.  Loaded through ctypes.
* ``brute.py`` -- pure Python with ``math.fsum``, for tiny inputs only.

Both compute, for each request b, query row i and head h (problem statement
and causal rule from the FlashInfer page
"prims_ts_batch_decode_with_kv_cache_mla"; natural-log LSE from the vLLM
``FlashInferMLAImpl`` page):

    s_j = bmm1_scale * <Q[b,i,h,:576], K_b[j,:576]>     j visible
    lse = ln sum_j exp(s_j)
    O   = bmm2_scale * sum_j exp(s_j - lse) * K_b[j,:512]

with K_b gathered through ``block_tables`` and row i of a request of q_len q
seeing rows 0 .. seq_len - q + i (causal) or 0 .. seq_len - 1 (dense).  Under
decode-context parallelism (``cp_world`` > 1; the vLLM ``FlashInferMLAImpl``
page passes cp_world, cp_rank and the global KV lengths to the kernel) a
rank's local row j is global row j * cp_world + cp_rank and the causal bound
is taken on that global position against the global length.  Under sparse
top-k selection (``sparse_idx``; the trtllm-gen MLA launcher in the FlashInfer
issue "Support cum_seq_lens_q in trtllm_batch_decode_with_kv_cache_mla" takes a
``sparse_mla_top_k`` argument and the pages say no more) query token t
attends exactly the logical KV positions listed in row t of ``sparse_idx``
that fall in [0, seq_len), once per listing; the list replaces the mask.

Parity status of each function is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

V_DIM = 512
QK_DIM = 576


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, plain C, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC",
                               "-shared", "-o", tmp, _SRC, "-lpthread", "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_mla_decode.restype = ctypes.c_int
        lib.oracle_mla_decode.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_double, ctypes.c_double, ctypes.c_int64, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.oracle_mla_decode_q.restype = ctypes.c_int
        lib.oracle_mla_decode_q.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_double, ctypes.c_double, ctypes.c_int64, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.oracle_mla_decode_dcp.restype = ctypes.c_int
        lib.oracle_mla_decode_dcp.argtypes = lib.oracle_mla_decode_q.argtypes + [
            ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
        lib.oracle_mla_decode_full.restype = ctypes.c_int
        lib.oracle_mla_decode_full.argtypes = lib.oracle_mla_decode_dcp.argtypes + [
            ctypes.c_int, ctypes.c_void_p]
        lib.oracle_decode_bf16.restype = ctypes.c_double
        lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_e4m3.restype = ctypes.c_double
        lib.oracle_decode_e4m3.argtypes = [ctypes.c_uint8]
        _lib = lib
    return _lib


def decode_bf16(bits: int) -> float:
    return _load().oracle_decode_bf16(bits)


def decode_e4m3(bits: int) -> float:
    return _load().oracle_decode_e4m3(bits)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def mla_decode(query: np.ndarray, q_start: np.ndarray, kv_cache: np.ndarray,
               block_tables: np.ndarray, seq_lens: np.ndarray, *, kv_dtype: str,
               causal: bool, bmm1_scale: float, bmm2_scale: float,
               sel: Optional[np.ndarray] = None, n_threads: Optional[int] = None,
               q_dtype: str = "bf16", cp_world: int = 1, cp_rank: int = 0,
               seq_lens_global: Optional[np.ndarray] = None,
               sparse_idx: Optional[np.ndarray] = None):
    """fp64 O and LSE.

    query:   uint16 bf16 bits (q_dtype "bf16") or uint8 e4m3 codes ("e4m3")
             viewed as [tokens, H, 576]
    q_start: [B+1] token offset of each request (fixed launches: b * SQ)
    kv_cache: uint16 (bf16) or uint8 (e4m3) [pages, page_size, 576]
    sel:     optional [n, 2] (token, head) pairs; default every pair.
    cp_world, cp_rank, seq_lens_global: decode-context parallelism -- this
             rank holds the global rows g with g mod cp_world == cp_rank as
             its local rows g div cp_world; the causal bound applies to the
             global positions, with global lengths seq_lens_global [B].
    sparse_idx: optional int32 [tokens, k] logical KV positions per query
             token (sparse top-k): the token attends the listed positions in
             [0, seq_len) (an entry outside, e.g. -1, is unused; a repeated
             one counts each time); ``causal`` is then not consulted.
    Returns (out, lse): [tokens, H, 512] and [tokens, H], or [n, 512] and [n].
    Rows that see no key get O = 0 and lse = -inf (the empty sum).
    """
    lib = _load()
    H = int(query.shape[-2])
    if q_dtype == "bf16":
        assert query.dtype == np.uint16
        qd = 0
    elif q_dtype == "e4m3":
        assert query.dtype == np.uint8
        qd = 1
    else:
        raise ValueError(q_dtype)
    q = np.ascontiguousarray(query.reshape(-1, H, QK_DIM))
    qs = np.ascontiguousarray(q_start, dtype=np.int64)
    kv = np.ascontiguousarray(kv_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B = int(sl.shape[0])
    if kv_dtype == "bf16":
        assert kv.dtype == np.uint16
        kd = 0
    elif kv_dtype == "e4m3":
        assert kv.dtype == np.uint8
        kd = 1
    else:
        raise ValueError(kv_dtype)
    tokens = int(qs[-1]) if B else 0
    if sel is None:
        n = tokens * H
        sel_arr = None
        out_shape, lse_shape = (tokens, H, V_DIM), (tokens, H)
    else:
        sel_arr = np.ascontiguousarray(sel, dtype=np.int64).reshape(-1, 2)
        n = int(sel_arr.shape[0])
        out_shape, lse_shape = (n, V_DIM), (n,)
    out = np.zeros(out_shape, dtype=np.float64)
    lse = np.zeros(lse_shape, dtype=np.float64)
    if n == 0 or B == 0:
        return out, lse
    slg = None
    if cp_world > 1 and seq_lens_global is not None:
        slg = np.ascontiguousarray(seq_lens_global, dtype=np.int32)
        assert slg.shape == sl.shape
    sk, sp = 0, None
    if sparse_idx is not None:
        sp = np.ascontiguousarray(sparse_idx, dtype=np.int32)
        assert sp.ndim == 2 and sp.shape[0] == tokens and sp.shape[1] >= 1
        sk = int(sp.shape[1])
    rc = lib.oracle_mla_decode_full(
        B, H, kd, qd, q.ctypes.data, qs.ctypes.data, kv.ctypes.data, int(kv.shape[0]),
        int(kv.shape[1]), bt.ctypes.data, int(bt.shape[1]), sl.ctypes.data, int(bool(causal)),
        float(bmm1_scale), float(bmm2_scale), n,
        sel_arr.ctypes.data if sel_arr is not None else None,
        out.ctypes.data, lse.ctypes.data, int(n_threads or default_threads()),
        int(cp_world), int(cp_rank), slg.ctypes.data if slg is not None else None,
        sk, sp.ctypes.data if sp is not None else None)
    if rc != 0:
        raise RuntimeError(f"oracle_mla_decode failed with status {rc}")
    return out, lse


def run(w, sel: Optional[np.ndarray] = None, n_threads: Optional[int] = None,
        causal: Optional[bool] = None):
    """Oracle on a ``mla_inputs.Workload`` (see ``mla_decode``)."""
    return mla_decode(w.query_rows(), w.q_start(), w.kv_cache, w.block_tables, w.seq_lens,
                      kv_dtype=w.kv_dtype, causal=w.causal if causal is None else causal,
                      bmm1_scale=w.bmm1_scale, bmm2_scale=w.bmm2_scale, sel=sel,
                      n_threads=n_threads, q_dtype=getattr(w, "q_dtype", "bf16"),
                      cp_world=getattr(w, "cp_world", 1), cp_rank=getattr(w, "cp_rank", 0),
                      seq_lens_global=getattr(w, "seq_lens_global", None),
                      sparse_idx=getattr(w, "sparse_idx", None))
