"""The C ABI library on the CPU: it loads, exports every function declared in
include/*.h, and its host-side checks reject bad arguments before any launch
(no GPU is touched by these calls)."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from chunked_prefill_paged_gb300 import build
    build.build()
    import chunked_prefill_paged_gb300 as cpa
    return cpa


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    names.discard("defined")
    return names


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert {"paged_kv_write", "chunked_prefill_attention", "chunked_prefill_workspace_size"} <= names
    handle = ctypes.CDLL(lib.LIB_PATH)
    for n in names:
        assert hasattr(handle, n), f"{n} declared in include/ but not exported"
    assert set(lib.EXPORTED) <= names


def test_binding_constants_match_the_header(lib):
    text = open(os.path.join(ROOT, "include", "cpa.h")).read()
    m = re.search(r"#define CPA_NO_ALLOC_WORKSPACE_BYTES \((\d+)u << (\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == lib.NO_ALLOC_WORKSPACE_BYTES


def test_version_and_status_strings(lib):
    L = lib.load()
    assert L.cpa_version() >= 100
    for s in range(7):
        assert lib.status_string(s)


def _cbatch(lib, cached, new, max_blocks, dev_ptr=0x1000):
    h_c = np.asarray(cached, dtype=np.int32)
    h_n = np.asarray(new, dtype=np.int32)
    b = lib.binding._Batch(len(h_c), max_blocks, int(h_n.sum()), dev_ptr, dev_ptr, dev_ptr, dev_ptr,
                           h_c.ctypes.data, h_n.ctypes.data)
    return b, (h_c, h_n)


BAD_PARAMS = [
    dict(num_heads_q=30, num_heads_kv=8),    # H_q not a multiple of H_kv
    dict(head_dim=96),
    dict(block_size=8),
    dict(kv_segment_size=768),
    dict(kv_segment_size=512, block_size=128, num_blocks=0),
    dict(dtype=5),
    dict(scale=float("inf")),
    dict(scale=-0.1),
    dict(rope_theta=-1.0),
    dict(rope_theta=float("nan")),
]


@pytest.mark.parametrize("bad", BAD_PARAMS)
def test_bad_params_rejected_before_launch(lib, bad):
    kw = dict(num_heads_q=32, num_heads_kv=8, head_dim=128, block_size=16, num_blocks=100, kv_segment_size=1024)
    kw.update(bad)
    p = lib.Params(**kw).c()
    b, keep = _cbatch(lib, [10], [5], 4)
    L = lib.load()
    rc = L.chunked_prefill_attention(ctypes.byref(b), ctypes.byref(p), 16, 16, 16, 16, 16, 16, None, None, 0, None)
    assert rc == lib.ERR_INVALID_ARG
    rc = L.paged_kv_write(ctypes.byref(b), ctypes.byref(p), 16, 16, 16, 16, None)
    assert rc == lib.ERR_INVALID_ARG


@pytest.mark.parametrize("cached,new,max_blocks", [
    ([10], [-1], 4),          # negative length
    ([-3], [2], 4),
    ([60], [5], 4),           # C + N beyond the block table (4 x 16)
])
def test_bad_batches_rejected(lib, cached, new, max_blocks):
    p = lib.Params(32, 8, 128, 16, 100, 1024).c()
    b, keep = _cbatch(lib, cached, new, max_blocks)
    L = lib.load()
    assert L.chunked_prefill_attention(ctypes.byref(b), ctypes.byref(p), 16, 16, 16, 16, 16, 16, None, None, 0,
                                       None) == lib.ERR_INVALID_ARG


def test_total_tokens_must_match(lib):
    p = lib.Params(32, 8, 128, 16, 100, 1024).c()
    b, keep = _cbatch(lib, [3, 4], [5, 6], 4)
    b.total_new_tokens = 12
    L = lib.load()
    assert L.chunked_prefill_attention(ctypes.byref(b), ctypes.byref(p), 16, 16, 16, 16, 16, 16, None, None, 0,
                                       None) == lib.ERR_INVALID_ARG


def test_misaligned_pointer_rejected(lib):
    p = lib.Params(32, 8, 128, 16, 100, 1024).c()
    b, keep = _cbatch(lib, [3], [5], 4)
    L = lib.load()
    assert L.paged_kv_write(ctypes.byref(b), ctypes.byref(p), 18, 16, 16, 16, None) == lib.ERR_INVALID_ARG


def test_empty_batch_is_a_no_op(lib):
    p = lib.Params(32, 8, 128, 16, 100, 1024).c()
    b = lib.binding._Batch(0, 1, 0, None, None, None, None, None, None)
    L = lib.load()
    assert L.chunked_prefill_attention(ctypes.byref(b), ctypes.byref(p), None, None, None, None, None, None, None,
                                       None, 0, None) == lib.SUCCESS
    assert L.chunked_prefill_workspace_size(ctypes.byref(b), ctypes.byref(p)) == 0


def test_workspace_size_counts_split_partials(lib):
    L = lib.load()
    # 3 decodes (one row group of G = 4 rows each), H_kv 8, d 128, split 1024
    p = lib.Params(32, 8, 128, 16, 10000, 1024).c()
    b, keep = _cbatch(lib, [5000, 100, 2047], [1, 1, 1], 400)
    pieces = [-(-(5000 + 1) // 1024), 1, -(-(2047 + 1) // 1024)]
    partials = sum(8 * n * 4 * (128 + 2) * 4 for n in pieces if n > 1)
    counter = 256  # the tensor-core kernel's work counter, after the partials
    expect = -(-partials // 256) * 256 + counter
    assert L.chunked_prefill_workspace_size(ctypes.byref(b), ctypes.byref(p)) == expect
    # no split requested: only the work counter
    p2 = lib.Params(32, 8, 128, 16, 10000, 1024, flags=lib.FLAG_NO_SPLIT).c()
    assert L.chunked_prefill_workspace_size(ctypes.byref(b), ctypes.byref(p2)) == counter
    # a prefill chunk of 512 tokens spans many query tiles and is never split
    b3, keep3 = _cbatch(lib, [8000], [512], 600)
    assert L.chunked_prefill_workspace_size(ctypes.byref(b3), ctypes.byref(p)) == counter
    # the CUDA-core kernel (forced) keeps no counter
    p4 = lib.Params(32, 8, 128, 16, 10000, 1024, flags=lib.FLAG_NO_SPLIT | lib.FLAG_FORCE_SIMT).c()
    assert L.chunked_prefill_workspace_size(ctypes.byref(b3), ctypes.byref(p4)) == 0


def test_workspace_size_counts_rotated_copies(lib):
    L = lib.load()
    b, keep = _cbatch(lib, [8000], [512], 600)
    rq = 512 * 32 * 128 * 2   # rotated queries, bf16
    rk = 512 * 8 * 128 * 2    # rotated new keys
    # block size 128, the one-pipeline kernel: the queries are rotated in
    # shared memory, so only the keys' copy comes first (256-byte aligned); the
    # counters stay last (the work counter and the rotation's 2 + 4 counts fit
    # the same 256 bytes)
    b128, keep128 = _cbatch(lib, [8064], [512], 80)
    plain = L.chunked_prefill_workspace_size(ctypes.byref(b128),
                                             ctypes.byref(lib.Params(32, 8, 128, 128, 1000, 1024).c()))
    p = lib.Params(32, 8, 128, 128, 1000, 1024, rope_theta=500000.0).c()
    assert L.chunked_prefill_workspace_size(ctypes.byref(b128), ctypes.byref(p)) == rk + plain
    # block size 16 with query tiles to pair, the two-pipeline kernel: the
    # rotation pre-pass writes copies of both
    plain = L.chunked_prefill_workspace_size(ctypes.byref(b), ctypes.byref(lib.Params(32, 8, 128, 16, 10000, 1024).c()))
    p = lib.Params(32, 8, 128, 16, 10000, 1024, rope_theta=500000.0).c()
    assert L.chunked_prefill_workspace_size(ctypes.byref(b), ctypes.byref(p)) == rq + rk + plain
    # the CUDA-core kernel (forced) reads rotated copies of both, and keeps no counter
    ps = lib.Params(32, 8, 128, 16, 10000, 1024, rope_theta=500000.0, flags=lib.FLAG_FORCE_SIMT).c()
    assert L.chunked_prefill_workspace_size(ctypes.byref(b), ctypes.byref(ps)) == rq + rk


def _fp8_params(lib, k_scale=0x1000, v_scale=0x1000, **kw):
    base = dict(num_heads_q=32, num_heads_kv=8, head_dim=128, block_size=16, num_blocks=100, kv_segment_size=1024)
    base.update(kw)
    p = lib.Params(**base).c()
    p.kv_format = lib.KV_FP8_E4M3
    p.k_scale = k_scale
    p.v_scale = v_scale
    return p


@pytest.mark.parametrize("case,expect", [
    (dict(kv_format=2), "invalid"),
    (dict(k_scale=None), "invalid"),
    (dict(v_scale=None), "invalid"),
    (dict(k_scale=0x1002), "invalid"),     # scales must be 4-byte aligned
    (dict(dtype=0), "unsupported"),        # FP8 codes of BF16 rows only
])
def test_fp8_arguments_checked_before_launch(lib, case, expect):
    case = dict(case)
    fmt = case.pop("kv_format", None)
    p = _fp8_params(lib, **case)
    if fmt is not None:
        p.kv_format = fmt
    b, keep = _cbatch(lib, [10], [5], 4)
    L = lib.load()
    want = lib.ERR_INVALID_ARG if expect == "invalid" else lib.ERR_UNSUPPORTED
    assert L.chunked_prefill_attention(ctypes.byref(b), ctypes.byref(p), 16, 16, 16, 16, 16, 16, None, None, 0,
                                       None) == want
    assert L.paged_kv_write(ctypes.byref(b), ctypes.byref(p), 16, 16, 16, 16, None) == want
    assert L.chunked_prefill_workspace_size(ctypes.byref(b), ctypes.byref(p)) == 0


@pytest.mark.parametrize("kw", [dict(head_dim=64), dict(flags=0x2)])
def test_fp8_attention_needs_the_tensor_core_kernel(lib, kw):
    # d = 64 or a forced CUDA-core kernel: the FP8 cache runs on the
    # tensor-core kernel only (a query group that does not divide 128, G = 3,
    # runs there too: 126-row query tiles)
    p = _fp8_params(lib, **kw)
    b, keep = _cbatch(lib, [10], [5], 4)
    L = lib.load()
    assert L.chunked_prefill_attention(ctypes.byref(b), ctypes.byref(p), 16, 16, 16, 16, 16, 16, None, None, 0,
                                       None) == lib.ERR_UNSUPPORTED
    assert L.chunked_prefill_workspace_size(ctypes.byref(b), ctypes.byref(p)) == 0


def test_fp8_attention_takes_query_groups_that_do_not_divide_128(lib):
    p = _fp8_params(lib, num_heads_q=24)  # G = 3
    b, keep = _cbatch(lib, [10], [5], 4)
    assert lib.load().chunked_prefill_workspace_size(ctypes.byref(b), ctypes.byref(p)) > 0


def test_workspace_size_counts_fp8_codes(lib):
    L = lib.load()
    b, keep = _cbatch(lib, [8000], [512], 600)
    plain = L.chunked_prefill_workspace_size(ctypes.byref(b), ctypes.byref(lib.Params(32, 8, 128, 16, 10000, 1024).c()))
    q16 = 512 * 32 * 128 * 2  # fp16 queries
    qs = 512 * 32 * 4         # their row scales
    codes = 512 * 8 * 128     # one byte per element of k_new (and again of v_new)
    p = _fp8_params(lib, num_blocks=10000)
    assert L.chunked_prefill_workspace_size(ctypes.byref(b), ctypes.byref(p)) == q16 + qs + 2 * codes + plain
    # with RoPE the rotation goes straight into those copies
    p.rope_theta = 500000.0
    assert L.chunked_prefill_workspace_size(ctypes.byref(b), ctypes.byref(p)) == q16 + qs + 2 * codes + plain
