"""Batched paged MLA decode on GB300 (sm_103a): thin Python binding.

Every step of the computation runs in the CUDA kernels of ``libmla_decode.so``
behind the C ABI in ``include/mla_decode.h``; this module only marshals
arguments (torch tensors for device memory and streams) and caches plans.
There is no CPU fallback: if the library is missing, every call raises.

The high-level entry point mirrors the FlashInfer page
"prims_ts_batch_decode_with_kv_cache_mla" (signature): fixed
``[B, SQ, H, 576]`` or packed ``[total_q, H, 576]`` queries (``qo_indptr``),
a rank-3 or rank-4 paged cache, ``block_tables``/``seq_lens`` on the device,
caller-owned workspace, ``bmm1_scale``/``bmm2_scale``, causal or dense
masking, bf16 output and an optional natural-log LSE.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Tuple

import torch

__all__ = [
    "MLA_OK", "MlaDecodeError", "MlaDecodeParams", "load_library", "library_path",
    "mla_decode_plan", "mla_decode_run", "mla_decode_run_profiled", "mla_decode_run_dcp",
    "mla_decode_run_sparse", "mla_decode_destroy", "mla_decode_workspace_size",
    "mla_decode_status_offset", "mla_decode_status_string", "Plan", "decode",
    "HEAD_DIM_QK", "HEAD_DIM_V",
]

HEAD_DIM_QK = 576
HEAD_DIM_V = 512
MLA_OK = 0
MLA_STATIC_WORKSPACE_BYTES = 48 * 1024 * 1024  # scratch of mla_decode_run_static_workspace
KV_BF16, KV_FP8_E4M3 = 0, 1
Q_BF16, Q_FP8_E4M3 = 0, 1
MASK_CAUSAL, MASK_DENSE = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libmla_decode.so")
_lib = None


class MlaDecodeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {mla_decode_status_string(status)} ({status})")
        self.status = status


class MlaDecodeParams(ctypes.Structure):
    """Mirror of ``mla_decode_params`` (natural C alignment)."""
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("max_seq_len_q", ctypes.c_int32),
        ("max_seq_len", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("max_pages_per_req", ctypes.c_int32),
        ("num_pages", ctypes.c_int64),
        ("packed", ctypes.c_int32),
        ("max_total_q", ctypes.c_int64),
        ("kv_dtype", ctypes.c_int32),
        ("mask", ctypes.c_int32),
        ("return_lse", ctypes.c_int32),
        ("device", ctypes.c_int32),
        ("q_dtype", ctypes.c_int32),
        ("cp_world", ctypes.c_int32),
        ("cp_rank", ctypes.c_int32),
        ("sparse_top_k", ctypes.c_int32),
        ("e4m3_widen", ctypes.c_int32),
    ]


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libmla_decode.so (built by ``paged_mla_decode_03_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                           "`python -m paged_mla_decode_03_gb300.build` (no fallback exists)")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.mla_decode_plan.argtypes = [ctypes.POINTER(MlaDecodeParams), ctypes.POINTER(vp),
                                    ctypes.POINTER(sz)]
    lib.mla_decode_plan.restype = ctypes.c_int
    lib.mla_decode_run.argtypes = [vp, vp, vp, vp, vp, vp, i64, ctypes.c_float, ctypes.c_float,
                                   vp, vp, vp, sz, vp]
    lib.mla_decode_run.restype = ctypes.c_int
    lib.mla_decode_run_profiled.argtypes = [vp, vp, vp, vp, vp, vp, i64, vp, ctypes.c_float,
                                            ctypes.c_float, vp, vp, vp, sz, vp, vp, vp]
    lib.mla_decode_run_profiled.restype = ctypes.c_int
    lib.mla_decode_run_device_scales.argtypes = [vp, vp, vp, vp, vp, vp, i64, vp, vp, vp, vp, vp,
                                                 sz, vp]
    lib.mla_decode_run_device_scales.restype = ctypes.c_int
    lib.mla_decode_host_staging_bytes.argtypes = [vp, i64]
    lib.mla_decode_host_staging_bytes.restype = sz
    lib.mla_decode_run_host.argtypes = [vp, vp, vp, vp, vp, vp, i64, ctypes.c_float,
                                        ctypes.c_float, vp, vp, vp, sz, vp, sz, vp]
    lib.mla_decode_run_host.restype = ctypes.c_int
    lib.mla_decode_run_dcp.argtypes = [vp, vp, vp, vp, vp, vp, i64, vp, ctypes.c_float,
                                       ctypes.c_float, vp, vp, vp, sz, vp]
    lib.mla_decode_run_dcp.restype = ctypes.c_int
    lib.mla_decode_run_sparse.argtypes = [vp, vp, vp, vp, vp, vp, i64, vp, ctypes.c_float,
                                          ctypes.c_float, vp, vp, vp, sz, vp]
    lib.mla_decode_run_sparse.restype = ctypes.c_int
    lib.mla_merge_states.argtypes = [vp, vp, i32, i64, ctypes.c_float, vp, vp, vp]
    lib.mla_merge_states.restype = ctypes.c_int
    lib.mla_decode_destroy.argtypes = [vp]
    lib.mla_decode_destroy.restype = None
    lib.mla_decode_workspace_size.argtypes = [vp]
    lib.mla_decode_workspace_size.restype = sz
    lib.mla_decode_work_list_layout.argtypes = [vp, ctypes.POINTER(sz), ctypes.POINTER(sz),
                                                ctypes.POINTER(i32)]
    lib.mla_decode_work_list_layout.restype = ctypes.c_int
    lib.mla_decode_kernels_per_run.argtypes = [vp]
    lib.mla_decode_kernels_per_run.restype = i32
    lib.mla_decode_status_offset.argtypes = []
    lib.mla_decode_status_offset.restype = sz
    lib.mla_decode_status_string.argtypes = [ctypes.c_int]
    lib.mla_decode_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def mla_decode_status_string(status: int) -> str:
    return load_library().mla_decode_status_string(int(status)).decode()


def mla_decode_status_offset() -> int:
    return int(load_library().mla_decode_status_offset())


def mla_decode_plan(params: MlaDecodeParams) -> Tuple[int, int]:
    """-> (plan handle, workspace bytes).  Raises MlaDecodeError on failure."""
    lib = load_library()
    handle = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    rc = lib.mla_decode_plan(ctypes.byref(params), ctypes.byref(handle), ctypes.byref(ws))
    if rc != MLA_OK:
        raise MlaDecodeError(rc, "mla_decode_plan")
    return handle.value, ws.value


def mla_decode_destroy(plan: Optional[int]) -> None:
    if plan:
        load_library().mla_decode_destroy(ctypes.c_void_p(plan))


def mla_decode_workspace_size(plan: int) -> int:
    return int(load_library().mla_decode_workspace_size(ctypes.c_void_p(plan)))


def mla_decode_work_list_layout(plan: int) -> Tuple[int, int, int]:
    """(items offset, worker-ranges offset, workers) of a plan's work list in
    the workspace (see include/mla_decode.h); for tests and tools."""
    a, b, n = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_int32()
    rc = load_library().mla_decode_work_list_layout(ctypes.c_void_p(plan), ctypes.byref(a),
                                                    ctypes.byref(b), ctypes.byref(n))
    if rc != MLA_OK:
        raise MlaDecodeError(rc, "mla_decode_work_list_layout")
    return a.value, b.value, n.value


def mla_decode_kernels_per_run(plan: int) -> int:
    """Kernels one run of the plan launches (see include/mla_decode.h)."""
    return int(load_library().mla_decode_kernels_per_run(ctypes.c_void_p(plan)))


def _nbytes(x) -> int:
    if x is None or isinstance(x, int):
        return 0
    return x.numel() * x.element_size()


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def mla_decode_run(plan: int, query, kv_cache, block_tables, seq_lens, qo_indptr, total_q: int,
                   bmm1_scale: float, bmm2_scale: float, out, lse, workspace,
                   workspace_bytes: Optional[int] = None, stream=None) -> None:
    """Enqueue one decode (arguments: tensors or raw device pointers)."""
    lib = load_library()
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace)
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    elif isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    rc = lib.mla_decode_run(ctypes.c_void_p(plan), _ptr(query), _ptr(kv_cache), _ptr(block_tables),
                            _ptr(seq_lens), _ptr(qo_indptr), int(total_q), float(bmm1_scale),
                            float(bmm2_scale), _ptr(out), _ptr(lse), _ptr(workspace),
                            int(workspace_bytes), stream)
    if rc != MLA_OK:
        raise MlaDecodeError(rc, "mla_decode_run")


def mla_decode_run_dcp(plan: int, query, kv_cache, block_tables, seq_lens, qo_indptr,
                       total_q: int, seq_lens_global, bmm1_scale: float, bmm2_scale: float,
                       out, lse, workspace, workspace_bytes: Optional[int] = None,
                       stream=None) -> None:
    """One decode-context-parallel rank's decode (``mla_decode_run_dcp``):
    ``seq_lens`` are the rank's local row counts, ``seq_lens_global`` the
    global KV lengths the causal bound is taken against (None for dense)."""
    lib = load_library()
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace)
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    elif isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    rc = lib.mla_decode_run_dcp(ctypes.c_void_p(plan), _ptr(query), _ptr(kv_cache),
                                _ptr(block_tables), _ptr(seq_lens), _ptr(qo_indptr), int(total_q),
                                _ptr(seq_lens_global), float(bmm1_scale), float(bmm2_scale),
                                _ptr(out), _ptr(lse), _ptr(workspace), int(workspace_bytes),
                                stream)
    if rc != MLA_OK:
        raise MlaDecodeError(rc, "mla_decode_run_dcp")


def mla_decode_run_sparse(plan: int, query, kv_cache, block_tables, seq_lens, qo_indptr,
                          total_q: int, sparse_indices, bmm1_scale: float, bmm2_scale: float,
                          out, lse, workspace, workspace_bytes: Optional[int] = None,
                          stream=None) -> None:
    """Sparse top-k decode (``mla_decode_run_sparse``): ``sparse_indices`` is
    an int32 CUDA tensor ``[tokens, k]`` of logical KV positions per query
    token; entries outside ``[0, seq_lens[b])`` are unused."""
    lib = load_library()
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace)
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    elif isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    if isinstance(sparse_indices, torch.Tensor) and (
            sparse_indices.dtype != torch.int32 or not sparse_indices.is_cuda
            or not sparse_indices.is_contiguous()):
        raise TypeError("sparse_indices must be a contiguous int32 CUDA tensor")
    rc = lib.mla_decode_run_sparse(ctypes.c_void_p(plan), _ptr(query), _ptr(kv_cache),
                                   _ptr(block_tables), _ptr(seq_lens), _ptr(qo_indptr),
                                   int(total_q), _ptr(sparse_indices), float(bmm1_scale),
                                   float(bmm2_scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                   int(workspace_bytes), stream)
    if rc != MLA_OK:
        raise MlaDecodeError(rc, "mla_decode_run_sparse")


def mla_decode_host_staging_bytes(plan: int, total_q: int = 0) -> int:
    """Device staging bytes of ``mla_decode_run_host`` for one step."""
    return int(load_library().mla_decode_host_staging_bytes(ctypes.c_void_p(plan), int(total_q)))


def mla_decode_run_host(plan: int, h_query, kv_cache, h_block_tables, h_seq_lens, h_qo_indptr,
                        total_q: int, bmm1_scale: float, bmm2_scale: float, h_out, h_lse,
                        staging, workspace, staging_bytes: Optional[int] = None,
                        workspace_bytes: Optional[int] = None, stream=None) -> None:
    """Enqueue one decode whose query, metadata and results are host buffers
    (CPU tensors, ideally pinned); ``kv_cache``, ``staging`` and ``workspace``
    are device buffers.  The copies are enqueued on ``stream`` with the decode."""
    lib = load_library()
    if staging_bytes is None:
        staging_bytes = _nbytes(staging)
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace)
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    elif isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    rc = lib.mla_decode_run_host(ctypes.c_void_p(plan), _ptr(h_query), _ptr(kv_cache),
                                 _ptr(h_block_tables), _ptr(h_seq_lens), _ptr(h_qo_indptr),
                                 int(total_q), float(bmm1_scale), float(bmm2_scale), _ptr(h_out),
                                 _ptr(h_lse), _ptr(staging), int(staging_bytes), _ptr(workspace),
                                 int(workspace_bytes), stream)
    if rc != MLA_OK:
        raise MlaDecodeError(rc, "mla_decode_run_host")


def mla_decode_run_device_scales(plan: int, query, kv_cache, block_tables, seq_lens, qo_indptr,
                                 total_q: int, bmm1_scale, bmm2_scale, out, lse, workspace,
                                 workspace_bytes: Optional[int] = None, stream=None) -> None:
    """``mla_decode_run`` with the two scales read from device memory at run
    time (``bmm1_scale`` / ``bmm2_scale``: one-element fp32 CUDA tensors or
    raw device pointers), so a captured graph sees new values at every replay."""
    lib = load_library()
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace)
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    elif isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    for t in (bmm1_scale, bmm2_scale):
        if isinstance(t, torch.Tensor) and (t.dtype != torch.float32 or not t.is_cuda
                                            or t.numel() != 1):
            raise TypeError("device scales must be one-element fp32 CUDA tensors")
    rc = lib.mla_decode_run_device_scales(
        ctypes.c_void_p(plan), _ptr(query), _ptr(kv_cache), _ptr(block_tables), _ptr(seq_lens),
        _ptr(qo_indptr), int(total_q), _ptr(bmm1_scale), _ptr(bmm2_scale), _ptr(out), _ptr(lse),
        _ptr(workspace), int(workspace_bytes), stream)
    if rc != 0:
        raise MlaDecodeError(rc, "mla_decode_run_device_scales")


def mla_decode_run_profiled(plan: int, query, kv_cache, block_tables, seq_lens, qo_indptr,
                            total_q: int, bmm1_scale: float, bmm2_scale: float, out, lse,
                            workspace, workspace_bytes: Optional[int] = None, stream=None,
                            events=None, sparse_indices=None) -> None:
    """``mla_decode_run`` (``mla_decode_run_sparse`` with ``sparse_indices``)
    that also records ``events = (before, after)`` (torch.cuda.Event) around
    the decode kernel on the same stream."""
    lib = load_library()
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace)
    if stream is None:
        stream = torch.cuda.current_stream()
    if not isinstance(stream, torch.cuda.Stream):
        raise TypeError("stream must be a torch.cuda.Stream")
    ev0 = ev1 = None
    if events is not None:
        # make sure the events exist (torch creates them lazily on first record)
        events[0].record(stream)
        events[1].record(stream)
        ev0, ev1 = events[0].cuda_event, events[1].cuda_event
    rc = lib.mla_decode_run_profiled(ctypes.c_void_p(plan), _ptr(query), _ptr(kv_cache),
                                     _ptr(block_tables), _ptr(seq_lens), _ptr(qo_indptr),
                                     int(total_q), _ptr(sparse_indices), float(bmm1_scale),
                                     float(bmm2_scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                     int(workspace_bytes), stream.cuda_stream, ev0, ev1)
    if rc != MLA_OK:
        raise MlaDecodeError(rc, "mla_decode_run_profiled")


class Plan:
    """Owns one C plan; ``run`` enqueues a decode with it."""

    def __init__(self, *, batch: int, num_heads: int, max_seq_len_q: int, max_seq_len: int,
                 page_size: int, max_pages_per_req: int, num_pages: int, packed: bool,
                 max_total_q: int = 0, kv_dtype: str = "bf16", causal: bool = True,
                 return_lse: bool = False, device: int = 0, q_dtype: str = "bf16",
                 cp_world: int = 1, cp_rank: int = 0, sparse_top_k: int = 0,
                 e4m3_widen: bool = False):
        self.params = MlaDecodeParams(
            batch=batch, num_heads=num_heads, max_seq_len_q=max_seq_len_q,
            max_seq_len=max_seq_len, page_size=page_size, max_pages_per_req=max_pages_per_req,
            num_pages=num_pages, packed=int(bool(packed)), max_total_q=max_total_q,
            kv_dtype=KV_FP8_E4M3 if kv_dtype in ("e4m3", "fp8", torch.float8_e4m3fn) else KV_BF16,
            mask=MASK_CAUSAL if causal else MASK_DENSE, return_lse=int(bool(return_lse)),
            device=device,
            q_dtype=Q_FP8_E4M3 if q_dtype in ("e4m3", "fp8", torch.float8_e4m3fn) else Q_BF16,
            cp_world=cp_world, cp_rank=cp_rank, sparse_top_k=sparse_top_k,
            e4m3_widen=int(bool(e4m3_widen)))
        self.cp_world = cp_world
        self.sparse_top_k = sparse_top_k
        self.handle, self.workspace_bytes = mla_decode_plan(self.params)

    def run(self, query, kv_cache, block_tables, seq_lens, out, *, qo_indptr=None, total_q=0,
            lse=None, workspace=None, bmm1_scale=1.0, bmm2_scale=1.0, stream=None,
            seq_lens_global=None, sparse_indices=None):
        """Scales are Python floats, or one-element fp32 CUDA tensors (then both
        must be, and the kernels read them when they run).  A plan with
        ``cp_world`` > 1 runs one DCP rank's decode (``seq_lens_global``: the
        global KV lengths, required under causal masking); a plan with
        ``sparse_top_k`` > 0 a sparse top-k decode over ``sparse_indices``."""
        if self.sparse_top_k > 0:
            mla_decode_run_sparse(self.handle, query, kv_cache, block_tables, seq_lens,
                                  qo_indptr, total_q, sparse_indices, bmm1_scale, bmm2_scale,
                                  out, lse, workspace, None, stream)
            return
        if self.cp_world > 1:
            mla_decode_run_dcp(self.handle, query, kv_cache, block_tables, seq_lens, qo_indptr,
                               total_q, seq_lens_global, bmm1_scale, bmm2_scale, out, lse,
                               workspace, None, stream)
            return
        if isinstance(bmm1_scale, torch.Tensor) or isinstance(bmm2_scale, torch.Tensor):
            mla_decode_run_device_scales(self.handle, query, kv_cache, block_tables, seq_lens,
                                         qo_indptr, total_q, bmm1_scale, bmm2_scale, out, lse,
                                         workspace, None, stream)
            return
        mla_decode_run(self.handle, query, kv_cache, block_tables, seq_lens, qo_indptr, total_q,
                       bmm1_scale, bmm2_scale, out, lse, workspace, None, stream)

    def staging_bytes(self, total_q: int = 0) -> int:
        """Device staging bytes ``run_host`` needs for a step of ``total_q`` rows."""
        return mla_decode_host_staging_bytes(self.handle, total_q)

    def run_host(self, h_query, kv_cache, h_block_tables, h_seq_lens, h_out, *, staging,
                 workspace, h_qo_indptr=None, total_q=0, h_lse=None, bmm1_scale=1.0,
                 bmm2_scale=1.0, stream=None):
        """One step with host-side query, metadata and results (see
        ``mla_decode_run_host``); returns once the copies and kernels are enqueued."""
        for name, t in (("h_query", h_query), ("h_block_tables", h_block_tables),
                        ("h_seq_lens", h_seq_lens), ("h_out", h_out), ("h_qo_indptr", h_qo_indptr),
                        ("h_lse", h_lse)):
            if isinstance(t, torch.Tensor) and (t.is_cuda or not t.is_contiguous()):
                raise ValueError(f"{name} must be a contiguous host tensor")
        mla_decode_run_host(self.handle, h_query, kv_cache, h_block_tables, h_seq_lens,
                            h_qo_indptr, total_q, bmm1_scale, bmm2_scale, h_out, h_lse, staging,
                            workspace, None, None, stream)

    def close(self):
        if self.handle:
            mla_decode_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


_plans: Dict[tuple, Plan] = {}


def decode(query: torch.Tensor, kv_cache: torch.Tensor, workspace_buffer: torch.Tensor,
           block_tables: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int, *,
           qo_indptr: Optional[torch.Tensor] = None, max_seq_len_q: Optional[int] = None,
           out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
           bmm1_scale=1.0, bmm2_scale=1.0, mask_type: str = "causal",
           return_lse: bool = False, cp_world: int = 1, cp_rank: int = 0,
           causal_seqlens_kv_global: Optional[torch.Tensor] = None,
           sparse_indices: Optional[torch.Tensor] = None, e4m3_widen: bool = False):
    """Paged MLA decode.  Returns ``out`` (and ``lse`` when ``return_lse``).

    ``query``: bf16 or float8_e4m3fn (quantised with a q_scale the caller folds
    into ``bmm1_scale``), ``[B, SQ, H, 576]`` (qo_indptr None) or ``[total_q, H, 576]``.
    ``kv_cache``: bf16 or float8_e4m3fn, ``[pages, page_size, 576]`` or
    ``[pages, 1, page_size, 576]``.  ``workspace_buffer`` must hold at least
    the plan's workspace bytes (see ``Plan``).  Plans are cached per static key.
    ``bmm1_scale`` / ``bmm2_scale``: floats, or one-element fp32 CUDA tensors the
    kernels read at run time (for scales that change between graph replays).
    ``cp_world`` / ``cp_rank`` / ``causal_seqlens_kv_global``: one rank of a
    decode-context-parallel decode (the vLLM FlashInferMLAImpl page's DCP
    keyword arguments); ``seq_lens`` are then the rank's local row counts.
    ``sparse_indices``: int32 ``[tokens, k]`` logical KV positions per query
    token (sparse top-k, ``sparse_mla_top_k`` = k); the listed positions in
    ``[0, seq_lens[b])`` replace the mask.
    ``e4m3_widen``: with an e4m3 cache, widen every e4m3 value exactly to bf16
    and multiply on bf16 tensor cores instead of the FP8 ones (see
    ``mla_decode_params.e4m3_widen`` in ``include/mla_decode.h``).
    """
    if query.dtype not in (torch.bfloat16, torch.float8_e4m3fn) or not query.is_cuda:
        raise ValueError("query must be a bf16 or float8_e4m3fn CUDA tensor")
    q_dtype = "bf16" if query.dtype == torch.bfloat16 else "e4m3"
    if kv_cache.dim() == 4:
        if kv_cache.shape[1] != 1:
            raise ValueError("rank-4 kv_cache must be [pages, 1, page_size, 576]")
        kv_cache = kv_cache.squeeze(1)
    if kv_cache.dim() != 3 or kv_cache.shape[-1] != HEAD_DIM_QK:
        raise ValueError("kv_cache must be [pages, page_size, 576]")
    if kv_cache.dtype == torch.bfloat16:
        kv_dtype = "bf16"
    elif kv_cache.dtype in (torch.float8_e4m3fn, torch.uint8):
        kv_dtype = "e4m3"
    else:
        raise ValueError(f"unsupported kv_cache dtype {kv_cache.dtype}")
    packed = qo_indptr is not None
    H = int(query.shape[-2])
    B = int(seq_lens.shape[0])
    if packed:
        if max_seq_len_q is None:
            raise ValueError("max_seq_len_q is required for packed launches")
        total_q = int(query.shape[0])
        sq = int(max_seq_len_q)
        out_shape = (total_q, H, HEAD_DIM_V)
        lse_shape = (total_q, H)
    else:
        total_q = 0
        sq = int(query.shape[1])
        out_shape = (B, sq, H, HEAD_DIM_V)
        lse_shape = (B * sq, H)
    causal = mask_type == "causal"
    if mask_type not in ("causal", "dense"):
        raise ValueError(mask_type)
    top_k = int(sparse_indices.shape[-1]) if sparse_indices is not None else 0
    key = (B, H, sq, int(max_seq_len), int(kv_cache.shape[1]), int(block_tables.shape[1]),
           int(kv_cache.shape[0]), packed, total_q if packed else 0, kv_dtype, causal,
           bool(return_lse), query.device.index or 0, q_dtype, int(cp_world), int(cp_rank),
           top_k, bool(e4m3_widen))
    plan = _plans.get(key)
    if plan is None:
        plan = Plan(batch=B, num_heads=H, max_seq_len_q=sq, max_seq_len=int(max_seq_len),
                    page_size=int(kv_cache.shape[1]), max_pages_per_req=int(block_tables.shape[1]),
                    num_pages=int(kv_cache.shape[0]), packed=packed, max_total_q=total_q,
                    kv_dtype=kv_dtype, causal=causal, return_lse=return_lse,
                    device=query.device.index or 0, q_dtype=q_dtype, cp_world=int(cp_world),
                    cp_rank=int(cp_rank), sparse_top_k=top_k, e4m3_widen=e4m3_widen)
        _plans[key] = plan
    if workspace_buffer.numel() * workspace_buffer.element_size() < plan.workspace_bytes:
        raise ValueError(f"workspace_buffer needs {plan.workspace_bytes} bytes")
    if out is None:
        out = torch.empty(out_shape, dtype=torch.bfloat16, device=query.device)
    if return_lse and lse is None:
        lse = torch.empty(lse_shape, dtype=torch.float32, device=query.device)
    plan.run(query, kv_cache, block_tables, seq_lens, out, qo_indptr=qo_indptr, total_q=total_q,
             lse=lse if return_lse else None, workspace=workspace_buffer,
             bmm1_scale=bmm1_scale, bmm2_scale=bmm2_scale,
             seq_lens_global=causal_seqlens_kv_global if causal else None,
             sparse_indices=sparse_indices)
    return (out, lse) if return_lse else out


def merge_states(o_parts: torch.Tensor, lse_parts: torch.Tensor, *, scale: float = 1.0,
                 out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                 stream=None):
    """Merge partial attention states of the same rows by their natural-log
    LSEs (``mla_merge_states``): ``o_parts`` bf16 ``[n, ..., 512]``,
    ``lse_parts`` fp32 ``[n, ...]`` (the leading dims after ``n`` flattened to
    rows).  Returns ``(out, lse)`` with the parts' row shape."""
    if o_parts.dtype != torch.bfloat16 or lse_parts.dtype != torch.float32:
        raise TypeError("o_parts must be bf16 and lse_parts fp32")
    if not (o_parts.is_cuda and lse_parts.is_cuda):
        raise ValueError("merge_states runs on the GPU")
    n = int(o_parts.shape[0])
    row_shape = tuple(o_parts.shape[1:-1])
    if o_parts.shape[-1] != HEAD_DIM_V or tuple(lse_parts.shape) != (n,) + row_shape:
        raise ValueError("o_parts [n, ..., 512] and lse_parts [n, ...] disagree")
    o_parts = o_parts.contiguous()
    lse_parts = lse_parts.contiguous()
    rows = 1
    for d in row_shape:
        rows *= int(d)
    if out is None:
        out = torch.empty(row_shape + (HEAD_DIM_V,), dtype=torch.bfloat16, device=o_parts.device)
    if lse is None:
        lse = torch.empty(row_shape, dtype=torch.float32, device=o_parts.device)
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    elif isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    rc = load_library().mla_merge_states(_ptr(o_parts), _ptr(lse_parts), n, rows, float(scale),
                                         _ptr(out), _ptr(lse), stream)
    if rc != 0:
        raise MlaDecodeError(rc, "mla_merge_states")
    return out, lse


def dcp_gather(out: torch.Tensor, lse: torch.Tensor, group=None):
    """The exchange step of decode-context parallelism: all-gather this rank's
    partial state (``out`` [..., 512], ``lse`` [...]) over ``group`` (a
    torch.distributed process group; default the world) into stacked
    ``[world, ...]`` tensors, to be merged with ``merge_states``."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    outs = [torch.empty_like(out) for _ in range(world)]
    lses = [torch.empty_like(lse) for _ in range(world)]
    dist.all_gather(outs, out.contiguous(), group=group)
    dist.all_gather(lses, lse.contiguous(), group=group)
    return torch.stack(outs), torch.stack(lses)
