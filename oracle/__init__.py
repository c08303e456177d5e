"""fp64 CPU oracle for paged chunked-prefill attention -- test infrastructure.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and it shares no code
with that path: the arithmetic lives in ``cpa_oracle.c`` (plain C, fp64),
compiled on first use with the host C compiler.

What the oracle computes is stated, with citations to the pages, at the top
of ``cpa_oracle.c``.  Summary: for active token i of request r (absolute
position p = cached_seq_len[r] + i) and query head h (kv head h // G), the
output is softmax(scale * q . K_j) weighted V over keys j = 0..p, where keys
j < cached_seq_len come from the paged pool through the block table and the
rest from the request's new K/V rows ("Prefill Processing", Key Concepts;
"Prefill Optimisation" section 2, Causal equivalence).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cpa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libcpa_oracle.so")
_lock = threading.Lock()
_lib = None

# Planted mistakes (tests only; see the enum in cpa_oracle.c).
MUT_NONE = 0
MUT_DROP_DIAGONAL = 1
MUT_GQA_MODULO = 2
MUT_NO_POSITION_OFFSET = 3
MUT_DROP_CACHED = 4
MUT_NO_BLOCK_TABLE = 5
MUT_NO_SCALE = 6
MUT_MERGE_NO_RESCALE = 7
MUT_WRITE_OFF_BY_ONE = 8
MUT_ROPE_INTERLEAVED = 9
MUT_ROPE_NO_OFFSET = 10
MUT_FP8_NEW_UNQUANTIZED = 11
MUT_FP8_HEAD0_SCALE = 12
MUT_FP8_TRUNCATE = 13
MUT_SEES_NEXT_KEY = 14


class _Problem(ctypes.Structure):
    _fields_ = [
        ("num_reqs", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("total_new_tokens", ctypes.c_int32),
        ("num_heads_q", ctypes.c_int32),
        ("num_heads_kv", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("mutation", ctypes.c_int32),
        ("scale", ctypes.c_double),
        ("cached_seq_len", ctypes.c_void_p),
        ("num_new_tokens", ctypes.c_void_p),
        ("cu_new_tokens", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("q", ctypes.c_void_p),
        ("k_new", ctypes.c_void_p),
        ("v_new", ctypes.c_void_p),
        ("k_cache", ctypes.c_void_p),
        ("v_cache", ctypes.c_void_p),
        ("kv_fp8", ctypes.c_int32),
        ("k_scale", ctypes.c_void_p),
        ("v_scale", ctypes.c_void_p),
    ]


def build(force: bool = False) -> str:
    """Compile cpa_oracle.c into a shared library next to it (gcc, -O2, no fast-math)."""
    with _lock:
        if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            subprocess.check_call(
                ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
                 _SRC, "-o", tmp, "-lm"])
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.cpa_oracle_attention.restype = ctypes.c_int
        lib.cpa_oracle_attention.argtypes = [
            ctypes.POINTER(_Problem), ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.cpa_oracle_kv_write_fp8.restype = ctypes.c_int
        lib.cpa_oracle_kv_write_fp8.argtypes = [ctypes.POINTER(_Problem), ctypes.c_void_p, ctypes.c_void_p]
        lib.cpa_oracle_e4m3_encode.restype = None
        lib.cpa_oracle_e4m3_encode.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_long, ctypes.c_int]
        lib.cpa_oracle_e4m3_decode.restype = None
        lib.cpa_oracle_e4m3_decode.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_long]
        lib.cpa_oracle_rope.restype = ctypes.c_int
        lib.cpa_oracle_rope.argtypes = [ctypes.POINTER(_Problem), ctypes.c_double, ctypes.c_void_p,
                                        ctypes.c_void_p]
        lib.cpa_oracle_kv_write.restype = ctypes.c_int
        lib.cpa_oracle_kv_write.argtypes = [ctypes.POINTER(_Problem), ctypes.c_int,
                                            ctypes.c_void_p, ctypes.c_void_p]
        _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _as_values(a: np.ndarray):
    """Return (contiguous array, dtype code): float32 values, bfloat16 bits
    (uint16) or float64 values."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, 0
    if a.dtype == np.uint16:
        return a, 1
    if a.dtype == np.float64:
        return a, 2
    raise TypeError(f"oracle inputs must be float32, float64 or bfloat16 bits (uint16), got {a.dtype}")


class Batch:
    """Host description of one step: per-request cached and new token counts
    and block-table rows ("Prefill Processing", Scheduler Output and Block
    Allocation)."""

    def __init__(self, cached_seq_len, num_new_tokens, block_table):
        self.cached_seq_len = np.ascontiguousarray(np.asarray(cached_seq_len, dtype=np.int32))
        self.num_new_tokens = np.ascontiguousarray(np.asarray(num_new_tokens, dtype=np.int32))
        self.block_table = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
        if self.block_table.ndim != 2 or self.block_table.shape[0] != self.cached_seq_len.shape[0]:
            raise ValueError("block_table must be [num_reqs, max_blocks_per_seq]")
        self.cu_new_tokens = np.zeros(self.num_reqs + 1, dtype=np.int32)
        np.cumsum(self.num_new_tokens, out=self.cu_new_tokens[1:])

    @property
    def num_reqs(self) -> int:
        return int(self.cached_seq_len.shape[0])

    @property
    def total_new_tokens(self) -> int:
        return int(self.cu_new_tokens[-1])


def _problem(batch: Batch, q, k_new, v_new, k_cache, v_cache, *, num_heads_q, num_heads_kv,
             head_dim, block_size, scale, mutation, keep, kv_scales=None):
    q, dt = _as_values(q)
    k_new, dt1 = _as_values(k_new)
    v_new, dt2 = _as_values(v_new)
    if kv_scales is None:
        k_cache, dt3 = _as_values(k_cache)
        v_cache, dt4 = _as_values(v_cache)
    else:
        # FP8 pools: E4M3 codes, one byte per element
        k_cache = np.ascontiguousarray(k_cache)
        v_cache = np.ascontiguousarray(v_cache)
        if k_cache.dtype != np.uint8 or v_cache.dtype != np.uint8:
            raise TypeError("FP8 pools must be uint8 arrays of E4M3 codes")
        dt3 = dt4 = dt
        k_scale = np.ascontiguousarray(np.asarray(kv_scales[0], dtype=np.float32))
        v_scale = np.ascontiguousarray(np.asarray(kv_scales[1], dtype=np.float32))
        if k_scale.shape != (num_heads_kv,) or v_scale.shape != (num_heads_kv,):
            raise ValueError("k_scale / v_scale must hold one scale per kv head")
        if not (np.all(np.isfinite(k_scale)) and np.all(k_scale > 0) and np.all(np.isfinite(v_scale))
                and np.all(v_scale > 0)):
            raise ValueError("FP8 scales must be finite and > 0")
        keep.extend([k_scale, v_scale])
    if len({dt, dt1, dt2, dt3, dt4}) != 1:
        raise TypeError("q, k_new, v_new and the pools must share one element type")
    T = batch.total_new_tokens
    if q.size != T * num_heads_q * head_dim or k_new.size != T * num_heads_kv * head_dim:
        raise ValueError("q / k_new sizes do not match the batch")
    num_blocks = k_cache.size // (block_size * num_heads_kv * head_dim)
    keep.extend([q, k_new, v_new, k_cache, v_cache, batch])
    P = _Problem(
        batch.num_reqs, batch.block_table.shape[1], T, num_heads_q, num_heads_kv, head_dim,
        block_size, num_blocks, dt, mutation, float(scale),
        batch.cached_seq_len.ctypes.data, batch.num_new_tokens.ctypes.data,
        batch.cu_new_tokens.ctypes.data, batch.block_table.ctypes.data,
        q.ctypes.data, k_new.ctypes.data, v_new.ctypes.data, k_cache.ctypes.data,
        v_cache.ctypes.data)
    if kv_scales is not None:
        P.kv_fp8 = 1
        P.k_scale = k_scale.ctypes.data
        P.v_scale = v_scale.ctypes.data
    return P


def attention(batch: Batch, q, k_new, v_new, k_cache, v_cache, *, num_heads_q, num_heads_kv,
              head_dim, block_size, scale, rows=None, segmented=False, kv_segment_size=0,
              threads=None, mutation=MUT_NONE, k_scale=None, v_scale=None):
    """fp64 attention output [n_rows, H_q, d] and lse [n_rows, H_q] (natural log).

    rows: token indices into the packed batch (None = all tokens).  With
    segmented=True the cached keys are walked in kv_segment_size pieces and
    combined by the online-softmax merge; otherwise the definition is
    evaluated directly.  Inputs: float32 arrays or bfloat16 bit patterns
    (uint16) of q [T,H_q,d], k_new/v_new [T,H_kv,d], pools
    [num_blocks, block_size, H_kv, d].

    FP8 cache: with k_scale / v_scale ([H_kv] each) the pools are uint8 E4M3
    codes; a code c of kv head g stands for value(c) * scale[g], and the
    active tokens' own K/V rows are taken through the same encoding (as the
    cache holds them).
    """
    lib = _load()
    keep = []
    fp8 = _fp8_scales(k_scale, v_scale)
    P = _problem(batch, q, k_new, v_new, k_cache, v_cache, num_heads_q=num_heads_q,
                 num_heads_kv=num_heads_kv, head_dim=head_dim, block_size=block_size, scale=scale,
                 mutation=mutation, keep=keep, kv_scales=fp8)
    if rows is None:
        n_rows = batch.total_new_tokens
        rows_arr = None
        rows_ptr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
        n_rows = int(rows_arr.shape[0])
        rows_ptr = rows_arr.ctypes.data
    out = np.zeros((n_rows, num_heads_q, head_dim), dtype=np.float64)
    lse = np.zeros((n_rows, num_heads_q), dtype=np.float64)
    if n_rows == 0:
        return out, lse
    rc = lib.cpa_oracle_attention(ctypes.byref(P), rows_ptr, n_rows, 1 if segmented else 0,
                                  int(kv_segment_size), out.ctypes.data, lse.ctypes.data,
                                  int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle attention failed with status {rc}")
    return out, lse


def _fp8_scales(k_scale, v_scale):
    if (k_scale is None) != (v_scale is None):
        raise ValueError("give both k_scale and v_scale, or neither")
    return None if k_scale is None else (k_scale, v_scale)


def kv_write(batch: Batch, k_new, v_new, k_cache, v_cache, *, num_heads_kv, head_dim, block_size,
             mutation=MUT_NONE, k_scale=None, v_scale=None):
    """Return copies of the pools with every active token's K/V row written
    into its slot (block_table[r][(C+i)//bs]*bs + (C+i)%bs).  A byte copy;
    with k_scale / v_scale the pools are uint8 E4M3 codes and each element is
    encoded with its kv head's scale (see e4m3_encode)."""
    lib = _load()
    k_out = np.array(k_cache, copy=True, order="C")
    v_out = np.array(v_cache, copy=True, order="C")
    k_new = np.ascontiguousarray(k_new)
    v_new = np.ascontiguousarray(v_new)
    fp8 = _fp8_scales(k_scale, v_scale)
    if fp8 is not None:
        keep = []
        dummy_q = np.zeros(batch.total_new_tokens * num_heads_kv * head_dim, dtype=k_new.dtype)
        P = _problem(batch, dummy_q, k_new, v_new, k_out, v_out, num_heads_q=num_heads_kv,
                     num_heads_kv=num_heads_kv, head_dim=head_dim, block_size=block_size, scale=1.0,
                     mutation=mutation, keep=keep, kv_scales=fp8)
        rc = lib.cpa_oracle_kv_write_fp8(ctypes.byref(P), k_out.ctypes.data, v_out.ctypes.data)
        if rc != 0:
            raise RuntimeError(f"oracle kv_write (FP8) failed with status {rc}")
        return k_out, v_out
    if k_new.dtype != k_out.dtype or v_new.dtype != v_out.dtype:
        raise TypeError("new rows and pools must share one element type")
    keep = []
    dummy_q = np.zeros(batch.total_new_tokens * num_heads_kv * head_dim, dtype=k_new.dtype)
    P = _problem(batch, dummy_q, k_new, v_new, k_out, v_out, num_heads_q=num_heads_kv,
                 num_heads_kv=num_heads_kv, head_dim=head_dim, block_size=block_size, scale=1.0,
                 mutation=mutation, keep=keep)
    rc = lib.cpa_oracle_kv_write(ctypes.byref(P), k_out.dtype.itemsize, k_out.ctypes.data,
                                 v_out.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"oracle kv_write failed with status {rc}")
    return k_out, v_out


def rope(batch: Batch, q, k_new, *, num_heads_q, num_heads_kv, head_dim, theta, mutation=MUT_NONE):
    """Rotary position embedding (rotate-half form) of the active tokens'
    queries [T, H_q, d] and new keys [T, H_kv, d] at absolute positions
    cached_seq_len[r] + i, in fp64.  Returns (q_rot, k_rot) as float64."""
    lib = _load()
    T = batch.total_new_tokens
    q = np.ascontiguousarray(q)
    k_new = np.ascontiguousarray(k_new)
    keep = []
    v_dummy = np.zeros_like(k_new)
    pool_dummy = np.zeros(num_heads_kv * head_dim, dtype=k_new.dtype)
    P = _problem(batch, q, k_new, v_dummy, pool_dummy, pool_dummy, num_heads_q=num_heads_q,
                 num_heads_kv=num_heads_kv, head_dim=head_dim, block_size=1, scale=1.0,
                 mutation=mutation, keep=keep)
    q_out = np.zeros((T, num_heads_q, head_dim), dtype=np.float64)
    k_out = np.zeros((T, num_heads_kv, head_dim), dtype=np.float64)
    if T == 0:
        return q_out, k_out
    rc = lib.cpa_oracle_rope(ctypes.byref(P), ctypes.c_double(float(theta)), q_out.ctypes.data,
                             k_out.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"oracle rope failed with status {rc}")
    return q_out, k_out


def e4m3_encode(y, mutation=MUT_NONE) -> np.ndarray:
    """FP8 E4M3 codes (uint8) of float32 values: nearest, ties to an even
    mantissa, |y| >= 448 saturated to +-448, NaN to the NaN code 0x7F."""
    lib = _load()
    y = np.ascontiguousarray(np.asarray(y, dtype=np.float32))
    out = np.zeros(y.shape, dtype=np.uint8)
    lib.cpa_oracle_e4m3_encode(y.ctypes.data, out.ctypes.data, ctypes.c_long(y.size), int(mutation))
    return out


def e4m3_decode(codes) -> np.ndarray:
    """Values (float64) of FP8 E4M3 codes."""
    lib = _load()
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.zeros(c.shape, dtype=np.float64)
    lib.cpa_oracle_e4m3_decode(c.ctypes.data, out.ctypes.data, ctypes.c_long(c.size))
    return out
