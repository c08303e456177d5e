"""Pools larger than 4 GiB per K and per V: the kernels take the pool as a
plain pointer plus num_blocks, and a GB300 holds pools of tens of GB, so
every byte offset into the pool must be computed in 64 bits.

The batch is drawn on a small pool as everywhere else; its blocks are then
moved to the top of a pool of more than 4.5 GiB (every block id shifted by
the same offset, so the request's slots all sit past byte 2^32).  Outputs
and LSE must match the oracle run on the small pool, and the written slots
at the top of the large pool must equal the oracle's write bit for bit.
The rest of the large pool is left uninitialised: nothing outside the block
table may be read.  Covered: the one-pipeline tensor-core kernel (block size
128), the two-pipeline kernel (block size 16, requests of more than 128
rows), the CUDA-core kernel (FP32), split decodes with the merge, the fused
and the standalone write, and the FP8 cache."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import Result, assert_within, bits, params_for, to_oracle

pytestmark = pytest.mark.gpu

LARGE_POOL_BYTES = 9 << 29  # 4.5 GiB per pool: slot offsets past 2^32
REQS = [(0, 300), (700, 130), (3000, 1), (1500, 1), (2048, 256), (33, 1)]


@pytest.fixture(scope="module")
def cpa():
    import chunked_prefill_paged_gb300 as m
    m.load()
    return m


def to_large_pool(w, small: torch.Tensor):
    """The small pool's blocks at the top of a pool of at least
    LARGE_POOL_BYTES; returns (pool, block offset)."""
    block_bytes = small[0].numel() * small.element_size()
    nb = max(-(-LARGE_POOL_BYTES // block_bytes), w.num_blocks) + w.num_blocks
    offset = nb - w.num_blocks
    assert offset * block_bytes >= 1 << 32
    big = torch.empty((nb,) + tuple(small.shape[1:]), dtype=small.dtype, device=small.device)
    big[offset:] = small
    return big, offset


def shifted(block_table: np.ndarray, offset: int) -> np.ndarray:
    bt = block_table.astype(np.int64) + offset
    assert bt.max() < 2 ** 31
    return bt.astype(np.int32)


@pytest.mark.parametrize("dtype,hq,hkv,d,bs,fused", [
    ("bf16", 32, 8, 128, 128, True),   # one-pipeline tensor-core kernel
    ("bf16", 32, 8, 128, 16, True),    # two-pipeline kernel (requests of > 128 rows)
    ("bf16", 32, 8, 128, 16, False),   # standalone write, then attention over the read-only pool
    ("f32", 8, 2, 64, 16, True),       # CUDA-core kernel
])
def test_slots_past_4gib(cpa, dtype, hq, hkv, d, bs, fused):
    sh = W.Shape(hq, hkv, d, bs, 1024, dtype)
    w = W.make_batch_workload(f"large_pool_{dtype}_{bs}", sh, REQS, seed=83)
    t = w.materialize("cuda")
    s = w.steps[0]
    q, kn, vn = t.step_inputs(s)
    ob = oracle.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    qo, kno, vno = to_oracle(q), to_oracle(kn), to_oracle(vn)
    k_small, v_small = to_oracle(t.k_cache), to_oracle(t.v_cache)
    ref_o, ref_l = oracle.attention(ob, qo, kno, vno, k_small, v_small, num_heads_q=hq, num_heads_kv=hkv,
                                    head_dim=d, block_size=bs, scale=sh.scale)
    k_ref, v_ref = oracle.kv_write(ob, kno, vno, k_small, v_small, num_heads_kv=hkv, head_dim=d, block_size=bs)

    k_big, offset = to_large_pool(w, t.k_cache)
    v_big, _ = to_large_pool(w, t.v_cache)
    del t.k_cache, t.v_cache
    p = params_for(w, flags=cpa.FLAG_FUSE_KV_WRITE if fused else 0)
    p.num_blocks = k_big.shape[0]
    b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, shifted(w.block_table, offset), device="cuda")
    if not fused:
        cpa.paged_kv_write(b, p, kn, vn, k_big, v_big)
    out, lse = cpa.attention(b, p, q, kn, vn, k_big, v_big)
    torch.cuda.synchronize()
    assert cpa.last_device_error() == cpa.SUCCESS
    res = Result()
    res.add(out.float().cpu().numpy(), ref_o, lse.cpu().numpy(), ref_l)
    assert_within(res, dtype)
    vt = np.int16 if dtype == "bf16" else np.int32
    assert np.array_equal(bits(k_big[offset:]), k_ref.view(vt)), "K slots differ from the oracle's write"
    assert np.array_equal(bits(v_big[offset:]), v_ref.view(vt)), "V slots differ from the oracle's write"
    del k_big, v_big
    torch.cuda.empty_cache()


def test_fp8_slots_past_4gib(cpa):
    sh = W.Shape(32, 8, 128, 16, 1024, "bf16")
    w = W.make_batch_workload("large_pool_fp8", sh, REQS, seed=84)
    t = w.materialize("cuda")
    s = w.steps[0]
    q, kn, vn = t.step_inputs(s)
    ks, vs = W.fp8_scales(sh.num_heads_kv)
    k8 = W.fp8_pool_codes(t.k_cache, ks)
    v8 = W.fp8_pool_codes(t.v_cache, vs)
    del t.k_cache, t.v_cache
    ob = oracle.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    qo, kno, vno = to_oracle(q), to_oracle(kn), to_oracle(vn)
    k_small, v_small = k8.cpu().numpy(), v8.cpu().numpy()
    ref_o, ref_l = oracle.attention(ob, qo, kno, vno, k_small, v_small, num_heads_q=sh.num_heads_q,
                                    num_heads_kv=sh.num_heads_kv, head_dim=sh.head_dim, block_size=sh.block_size,
                                    scale=sh.scale, k_scale=ks, v_scale=vs)
    k_ref, v_ref = oracle.kv_write(ob, kno, vno, k_small, v_small, num_heads_kv=sh.num_heads_kv,
                                   head_dim=sh.head_dim, block_size=sh.block_size, k_scale=ks, v_scale=vs)

    k_big, offset = to_large_pool(w, k8)
    v_big, _ = to_large_pool(w, v8)
    del k8, v8
    p = params_for(w)
    p.num_blocks = k_big.shape[0]
    p.kv_format = cpa.KV_FP8_E4M3
    p.k_scale = torch.as_tensor(ks, device="cuda")
    p.v_scale = torch.as_tensor(vs, device="cuda")
    b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, shifted(w.block_table, offset), device="cuda")
    out, lse = cpa.attention(b, p, q, kn, vn, k_big, v_big)
    torch.cuda.synchronize()
    assert cpa.last_device_error() == cpa.SUCCESS
    res = Result()
    res.add(out.float().cpu().numpy(), ref_o, lse.cpu().numpy(), ref_l)
    assert_within(res, "bf16")
    assert np.array_equal(k_big[offset:].cpu().numpy(), k_ref), "K codes differ from the oracle's write"
    assert np.array_equal(v_big[offset:].cpu().numpy(), v_ref), "V codes differ from the oracle's write"
    del k_big, v_big
    torch.cuda.empty_cache()
