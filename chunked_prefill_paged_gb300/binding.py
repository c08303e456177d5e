"""ctypes binding of libcpa (include/cpa.h): argument marshalling only.

Every step of the computation runs in the library's CUDA kernels.  PyTorch
supplies device memory and streams; the binding turns tensors into raw
pointers and fills the C structs.  There is no fallback: if the library is
missing or the device is not supported, calls raise.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional, Sequence

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcpa.so")

SUCCESS = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_CUDA = 3
ERR_DEVICE_TIMEOUT = 4
ERR_BAD_BLOCK_ID = 5
ERR_WORKSPACE = 6

DTYPE_FP32 = 0
DTYPE_BF16 = 1

KV_SAME = 0
KV_FP8_E4M3 = 1

FLAG_FUSE_KV_WRITE = 0x1
FLAG_FORCE_SIMT = 0x2
FLAG_NO_SPLIT = 0x4
FLAG_TAIL_SPLIT = 0x8
FLAG_TEST_STALL = 0x100
# bytes of the static device array behind chunked_prefill_attention_no_alloc
NO_ALLOC_WORKSPACE_BYTES = 32 << 20


class CpaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class _Batch(ctypes.Structure):
    _fields_ = [
        ("num_reqs", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("total_new_tokens", ctypes.c_int32),
        ("cached_seq_len", ctypes.c_void_p),
        ("num_new_tokens", ctypes.c_void_p),
        ("cu_new_tokens", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("h_cached_seq_len", ctypes.c_void_p),
        ("h_num_new_tokens", ctypes.c_void_p),
    ]


class _Params(ctypes.Structure):
    _fields_ = [
        ("num_heads_q", ctypes.c_int32),
        ("num_heads_kv", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("kv_segment_size", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("dtype", ctypes.c_int32),
        ("flags", ctypes.c_uint32),
        ("timeout_cycles", ctypes.c_int64),
        ("rope_theta", ctypes.c_float),
        ("kv_format", ctypes.c_int32),
        ("k_scale", ctypes.c_void_p),
        ("v_scale", ctypes.c_void_p),
    ]


class _EngineConfig(ctypes.Structure):
    _fields_ = [
        ("num_blocks", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("max_batched_tokens", ctypes.c_int32),
        ("chunk_size", ctypes.c_int32),
        ("scope_key", ctypes.c_uint64),
    ]


class _StepPlan(ctypes.Structure):
    _fields_ = [
        ("num_reqs", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("total_new_tokens", ctypes.c_int32),
        ("request_ids", ctypes.POINTER(ctypes.c_int64)),
        ("cached_seq_len", ctypes.POINTER(ctypes.c_int32)),
        ("num_new_tokens", ctypes.POINTER(ctypes.c_int32)),
        ("cu_new_tokens", ctypes.POINTER(ctypes.c_int32)),
        ("block_table", ctypes.POINTER(ctypes.c_int32)),
        ("token_ids", ctypes.POINTER(ctypes.c_int32)),
    ]


EXPORTED = [
    "cpa_engine_create",
    "cpa_engine_destroy",
    "cpa_engine_add_request",
    "cpa_engine_schedule",
    "cpa_engine_commit",
    "cpa_engine_num_free_blocks",
    "cpa_engine_num_unfinished",
    "cpa_engine_prefix_hit_tokens",
    "chunked_prefill_workspace_size",
    "paged_kv_write",
    "chunked_prefill_attention",
    "chunked_prefill_attention_no_alloc",
    "cpa_last_device_error",
    "cpa_status_string",
    "cpa_version",
]

_lib = None


def load(path: str = LIB_PATH):
    """Load libcpa.so (built by chunked_prefill_paged_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: run `python -m chunked_prefill_paged_gb300.build` "
                          "(requires nvcc); there is no fallback path")
    lib = ctypes.CDLL(path)
    P, VP = ctypes.POINTER, ctypes.c_void_p
    lib.chunked_prefill_workspace_size.restype = ctypes.c_size_t
    lib.chunked_prefill_workspace_size.argtypes = [P(_Batch), P(_Params)]
    lib.paged_kv_write.restype = ctypes.c_int
    lib.paged_kv_write.argtypes = [P(_Batch), P(_Params), VP, VP, VP, VP, VP]
    lib.chunked_prefill_attention.restype = ctypes.c_int
    lib.chunked_prefill_attention.argtypes = [P(_Batch), P(_Params), VP, VP, VP, VP, VP, VP, VP, VP,
                                              ctypes.c_size_t, VP]
    lib.chunked_prefill_attention_no_alloc.restype = ctypes.c_int
    lib.chunked_prefill_attention_no_alloc.argtypes = [P(_Batch), P(_Params), VP, VP, VP, VP, VP, VP, VP, VP]
    lib.cpa_last_device_error.restype = ctypes.c_int
    lib.cpa_last_device_error.argtypes = [VP]
    lib.cpa_status_string.restype = ctypes.c_char_p
    lib.cpa_status_string.argtypes = [ctypes.c_int]
    lib.cpa_version.restype = ctypes.c_int32
    lib.cpa_version.argtypes = []
    lib.cpa_engine_create.restype = ctypes.c_int
    lib.cpa_engine_create.argtypes = [P(_EngineConfig), P(VP)]
    lib.cpa_engine_destroy.restype = None
    lib.cpa_engine_destroy.argtypes = [VP]
    lib.cpa_engine_add_request.restype = ctypes.c_int
    lib.cpa_engine_add_request.argtypes = [VP, ctypes.c_int64, VP, ctypes.c_int32, ctypes.c_int32]
    lib.cpa_engine_schedule.restype = ctypes.c_int
    lib.cpa_engine_schedule.argtypes = [VP, P(_StepPlan)]
    lib.cpa_engine_commit.restype = ctypes.c_int
    lib.cpa_engine_commit.argtypes = [VP, VP]
    lib.cpa_engine_num_free_blocks.restype = ctypes.c_int32
    lib.cpa_engine_num_free_blocks.argtypes = [VP]
    lib.cpa_engine_num_unfinished.restype = ctypes.c_int32
    lib.cpa_engine_num_unfinished.argtypes = [VP]
    lib.cpa_engine_prefix_hit_tokens.restype = ctypes.c_int32
    lib.cpa_engine_prefix_hit_tokens.argtypes = [VP, ctypes.c_int64]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().cpa_status_string(int(status)).decode()


@dataclasses.dataclass
class Params:
    """Shape and options of one attention layer (cpa_params)."""
    num_heads_q: int
    num_heads_kv: int
    head_dim: int
    block_size: int
    num_blocks: int
    kv_segment_size: int = 0
    scale: Optional[float] = None
    dtype: int = DTYPE_BF16
    flags: int = FLAG_FUSE_KV_WRITE
    timeout_cycles: int = 0
    rope_theta: float = 0.0
    # FP8 cache: kv_format KV_FP8_E4M3, uint8 pools, and float32 device
    # tensors of H_kv scales for keys and for values
    kv_format: int = KV_SAME
    k_scale: Optional[torch.Tensor] = None
    v_scale: Optional[torch.Tensor] = None

    def c(self) -> _Params:
        scale = self.scale if self.scale is not None else 1.0 / float(np.sqrt(self.head_dim))
        for t in (self.k_scale, self.v_scale):
            if t is not None and t.dtype != torch.float32:
                raise TypeError("k_scale / v_scale must be float32 tensors")
        return _Params(self.num_heads_q, self.num_heads_kv, self.head_dim, self.block_size, self.num_blocks,
                       self.kv_segment_size, scale, self.dtype, self.flags, self.timeout_cycles,
                       self.rope_theta, self.kv_format, _ptr(self.k_scale), _ptr(self.v_scale))


class Batch:
    """Varlen batch descriptor (cpa_batch): device arrays plus host mirrors.

    cached_seq_len / num_new_tokens: per request; block_table: [num_reqs,
    max_blocks_per_seq] int32 (numpy or torch).  The device copies are made
    once here, on `device`."""

    def __init__(self, cached_seq_len: Sequence[int], num_new_tokens: Sequence[int], block_table,
                 device="cuda"):
        self.h_cached = np.ascontiguousarray(np.asarray(cached_seq_len, dtype=np.int32))
        self.h_new = np.ascontiguousarray(np.asarray(num_new_tokens, dtype=np.int32))
        bt = block_table.cpu().numpy() if isinstance(block_table, torch.Tensor) else np.asarray(block_table)
        bt = np.ascontiguousarray(bt, dtype=np.int32)
        if bt.ndim != 2 or bt.shape[0] != self.h_cached.shape[0]:
            raise ValueError("block_table must be [num_reqs, max_blocks_per_seq]")
        cu = np.zeros(len(self.h_new) + 1, dtype=np.int32)
        np.cumsum(self.h_new, out=cu[1:])
        self.h_cu = cu
        self.h_block_table = bt
        dev = torch.device(device)
        self.cached = torch.from_numpy(self.h_cached).to(dev)
        self.new = torch.from_numpy(self.h_new).to(dev)
        self.cu = torch.from_numpy(cu).to(dev)
        self.block_table = torch.from_numpy(bt).to(dev)

    @classmethod
    def from_device(cls, h_cached_seq_len: np.ndarray, h_num_new_tokens: np.ndarray, h_block_table: np.ndarray,
                    cached_seq_len: torch.Tensor, num_new_tokens: torch.Tensor, cu_new_tokens: torch.Tensor,
                    block_table: torch.Tensor) -> "Batch":
        """A batch whose device arrays already exist (int32, contiguous; e.g.
        filled by one host-to-device copy), with host mirrors of the same
        values."""
        b = cls.__new__(cls)
        b.h_cached = np.ascontiguousarray(h_cached_seq_len, dtype=np.int32)
        b.h_new = np.ascontiguousarray(h_num_new_tokens, dtype=np.int32)
        b.h_block_table = np.ascontiguousarray(h_block_table, dtype=np.int32)
        cu = np.zeros(len(b.h_new) + 1, dtype=np.int32)
        np.cumsum(b.h_new, out=cu[1:])
        b.h_cu = cu
        n, cols = b.h_block_table.shape
        for t, size in ((cached_seq_len, n), (num_new_tokens, n), (cu_new_tokens, n + 1), (block_table, n * cols)):
            if t.dtype != torch.int32 or not t.is_contiguous() or t.numel() != size:
                raise ValueError("device arrays must be contiguous int32 of the batch's sizes")
        b.cached, b.new, b.cu, b.block_table = cached_seq_len, num_new_tokens, cu_new_tokens, block_table
        return b

    @property
    def num_reqs(self) -> int:
        return int(self.h_cached.shape[0])

    @property
    def total_new_tokens(self) -> int:
        return int(self.h_cu[-1])

    def c(self) -> _Batch:
        return _Batch(self.num_reqs, int(self.h_block_table.shape[1]), self.total_new_tokens,
                      self.cached.data_ptr(), self.new.data_ptr(), self.cu.data_ptr(),
                      self.block_table.data_ptr(), self.h_cached.ctypes.data, self.h_new.ctypes.data)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libcpa must be contiguous")
    return t.data_ptr()


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def workspace_size(batch: Batch, params: Params) -> int:
    b, p = batch.c(), params.c()
    return int(load().chunked_prefill_workspace_size(ctypes.byref(b), ctypes.byref(p)))


def paged_kv_write(batch: Batch, params: Params, k_new, v_new, k_cache, v_cache, stream=None) -> None:
    b, p = batch.c(), params.c()
    rc = load().paged_kv_write(ctypes.byref(b), ctypes.byref(p), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                               _ptr(v_cache), _stream_ptr(stream))
    if rc != SUCCESS:
        raise CpaError(rc, "paged_kv_write")


def chunked_prefill_attention(batch: Batch, params: Params, q, k_new, v_new, k_cache, v_cache, out,
                              lse=None, workspace=None, stream=None) -> None:
    b, p = batch.c(), params.c()
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = load().chunked_prefill_attention(ctypes.byref(b), ctypes.byref(p), _ptr(q), _ptr(k_new), _ptr(v_new),
                                          _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse), _ptr(workspace),
                                          ws_bytes, _stream_ptr(stream))
    if rc != SUCCESS:
        raise CpaError(rc, "chunked_prefill_attention")


def chunked_prefill_attention_no_alloc(batch: Batch, params: Params, q, k_new, v_new, k_cache, v_cache, out,
                                       lse=None, stream=None) -> None:
    """chunked_prefill_attention without a workspace argument: for callers
    that cannot allocate device memory; the library's static device array
    holds the split-KV partials (see include/cpa.h)."""
    b, p = batch.c(), params.c()
    rc = load().chunked_prefill_attention_no_alloc(ctypes.byref(b), ctypes.byref(p), _ptr(q), _ptr(k_new),
                                                   _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(out),
                                                   _ptr(lse), _stream_ptr(stream))
    if rc != SUCCESS:
        raise CpaError(rc, "chunked_prefill_attention_no_alloc")


def last_device_error(stream=None) -> int:
    return int(load().cpa_last_device_error(_stream_ptr(stream)))


def attention(batch: Batch, params: Params, q, k_new, v_new, k_cache, v_cache, *, with_lse=True, stream=None):
    """Allocate out / lse / workspace with torch and run chunked_prefill_attention."""
    T = batch.total_new_tokens
    out = torch.empty((T, params.num_heads_q, params.head_dim), dtype=q.dtype, device=q.device)
    lse = torch.empty((T, params.num_heads_q), dtype=torch.float32, device=q.device) if with_lse else None
    n = workspace_size(batch, params)
    ws = torch.empty((max(n, 16) + 3) // 4, dtype=torch.float32, device=q.device) if n else None
    chunked_prefill_attention(batch, params, q, k_new, v_new, k_cache, v_cache, out, lse, ws, stream)
    return out, lse


@dataclasses.dataclass
class StepPlan:
    """One step's batch from the engine (host arrays, copied out)."""
    request_ids: np.ndarray      # int64 [num_reqs]
    cached_seq_len: np.ndarray   # int32 [num_reqs]
    num_new_tokens: np.ndarray   # int32 [num_reqs]
    block_table: np.ndarray      # int32 [num_reqs, max_blocks_per_seq]
    token_ids: np.ndarray        # int32 [total_new_tokens]

    @property
    def num_reqs(self) -> int:
        return int(self.request_ids.shape[0])


class Engine:
    """The library's host-side serving harness (include/cpa_engine.h): greedy
    token budget, incremental block allocation, prefix hash chain."""

    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int, max_batched_tokens: int,
                 chunk_size: int, scope_key: int = 0):
        self._lib = load()
        cfg = _EngineConfig(num_blocks, block_size, max_blocks_per_seq, max_batched_tokens, chunk_size,
                            scope_key)
        h = ctypes.c_void_p()
        rc = self._lib.cpa_engine_create(ctypes.byref(cfg), ctypes.byref(h))
        if rc != SUCCESS:
            raise CpaError(rc, "cpa_engine_create")
        self._h = h
        self.max_blocks_per_seq = max_blocks_per_seq
        self._n = 0

    def close(self) -> None:
        if self._h:
            self._lib.cpa_engine_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_request(self, request_id: int, prompt: Sequence[int], max_new_tokens: int) -> None:
        p = np.ascontiguousarray(np.asarray(prompt, dtype=np.int32))
        rc = self._lib.cpa_engine_add_request(self._h, int(request_id), p.ctypes.data, int(p.shape[0]),
                                              int(max_new_tokens))
        if rc != SUCCESS:
            raise CpaError(rc, "cpa_engine_add_request")

    def schedule(self) -> StepPlan:
        pl = _StepPlan()
        rc = self._lib.cpa_engine_schedule(self._h, ctypes.byref(pl))
        if rc != SUCCESS:
            raise CpaError(rc, "cpa_engine_schedule")
        n, cols, t = pl.num_reqs, pl.max_blocks_per_seq, pl.total_new_tokens
        self._n = n

        def arr(ptr, count, dtype):
            if count == 0:
                return np.zeros(0, dtype=dtype)
            return np.ctypeslib.as_array(ptr, shape=(count,)).astype(dtype, copy=True)

        return StepPlan(arr(pl.request_ids, n, np.int64), arr(pl.cached_seq_len, n, np.int32),
                        arr(pl.num_new_tokens, n, np.int32), arr(pl.block_table, n * cols, np.int32).reshape(n, cols),
                        arr(pl.token_ids, t, np.int32))

    def commit(self, sampled_tokens: Sequence[int]) -> None:
        s = np.ascontiguousarray(np.asarray(sampled_tokens, dtype=np.int32))
        if s.shape[0] != self._n:
            raise ValueError("one sampled token per scheduled request")
        rc = self._lib.cpa_engine_commit(self._h, s.ctypes.data if self._n else None)
        if rc != SUCCESS:
            raise CpaError(rc, "cpa_engine_commit")

    def num_free_blocks(self) -> int:
        return int(self._lib.cpa_engine_num_free_blocks(self._h))

    def num_unfinished(self) -> int:
        return int(self._lib.cpa_engine_num_unfinished(self._h))

    def prefix_hit_tokens(self, request_id: int) -> int:
        return int(self._lib.cpa_engine_prefix_hit_tokens(self._h, int(request_id)))
