"""GPU parity for the rotary position embedding (rope_theta > 0) against the
fp64 oracle.  The interface stores rotated queries and keys in the element
type (the cache holds rotated BF16 keys), so the reference is the oracle's
exact fp64 rotation rounded to that type (nearest even), then attention in
fp64.  Outputs within the BF16 / FP32 bounds; pool keys within one rounding
step of the reference (the library rotates in fp32 before rounding); pool
values bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import BF16_ATOL, FP32_ATOL, Result, assert_within, bits, params_for, sample_rows, to_oracle

pytestmark = pytest.mark.gpu

THETA = 500000.0


@pytest.fixture(scope="module")
def cpa():
    import chunked_prefill_paged_gb300 as m
    m.load()
    return m


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rounded(x: np.ndarray, dtype: str) -> np.ndarray:
    """fp64 values rounded to the element type (nearest even) and back."""
    tt = torch.bfloat16 if dtype == "bf16" else torch.float32
    return torch.from_numpy(np.ascontiguousarray(x)).to(tt).to(torch.float64).numpy()


def rope_params(w, flags=None, theta=THETA):
    p = params_for(w, flags)
    p.rope_theta = theta
    return p


def check_pool_keys(t_k, t_v, step, bt, kr, vn, bs, dtype):
    """Rotated keys of the active tokens in their slots (within rounding),
    values bit-exact."""
    k_pool, v_pool = as_f64(t_k), bits(t_v)
    vn_bits = bits(vn)
    cu = step.cu_new_tokens
    # one unit in the last place at the bottom of a binade: the fp32 rotation
    # may land on the other side of a rounding boundary than the fp64 one
    tol_rel = 2.0 ** -7 if dtype == "bf16" else 2.0 ** -22
    for r in range(len(step.num_new_tokens)):
        for i in range(int(step.num_new_tokens[r])):
            pos = int(step.cached_seq_len[r]) + i
            blk, off = int(bt[r, pos // bs]), pos % bs
            tok = int(cu[r]) + i
            ref = kr[tok]
            err = np.abs(k_pool[blk, off] - ref)
            # one rounding step, plus the fp32 rotation's own error near zero crossings
            assert np.all(err <= tol_rel * np.abs(ref) + 1e-6 * np.abs(ref).max()), (r, i, err.max())
            assert np.array_equal(v_pool[blk, off], vn_bits[tok])


@pytest.mark.parametrize("dtype,bs,flags", [("bf16", 16, None), ("bf16", 128, None), ("f32", 16, None),
                                            ("bf16", 16, "force_simt")])
def test_rope_small_batch(cpa, dtype, bs, flags):
    reqs = [(0, 300), (130, 77), (1000, 1), (17, 1), (257, 129), (5, 3), (3000, 1)]
    d = 64 if dtype == "f32" else 128
    w = W.make_batch_workload(f"rope_{dtype}_{bs}", W.Shape(8, 2, d, bs, 512, dtype), reqs, seed=41)
    t = w.materialize("cuda")
    s = w.steps[0]
    sh = w.shape
    fl = cpa.FLAG_FUSE_KV_WRITE | (cpa.FLAG_FORCE_SIMT if flags == "force_simt" else 0)
    p = rope_params(w, fl)
    b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    q, kn, vn = t.step_inputs(s)
    ob = oracle.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    qr, kr = oracle.rope(ob, as_f64(q), as_f64(kn), num_heads_q=sh.num_heads_q, num_heads_kv=sh.num_heads_kv,
                         head_dim=d, theta=THETA)
    qr, kr = rounded(qr, dtype), rounded(kr, dtype)
    k_pool0, v_pool0 = as_f64(t.k_cache), as_f64(t.v_cache)
    ref_o, ref_l = oracle.attention(ob, qr, kr, as_f64(vn), k_pool0, v_pool0, num_heads_q=sh.num_heads_q,
                                    num_heads_kv=sh.num_heads_kv, head_dim=d, block_size=bs, scale=sh.scale)
    out, lse = cpa.attention(b, p, q, kn, vn, t.k_cache, t.v_cache)
    torch.cuda.synchronize()
    assert cpa.last_device_error() == cpa.SUCCESS
    res = Result()
    res.add(out.float().cpu().numpy(), ref_o, lse.cpu().numpy(), ref_l)
    assert_within(res, dtype)
    check_pool_keys(t.k_cache, t.v_cache, s, w.block_table, kr, vn, bs, dtype)
    # the caller's inputs are left as they were
    q2, kn2, _ = t.step_inputs(s)
    assert torch.equal(q, q2) and torch.equal(kn, kn2)


def test_rope_standalone_write_then_read_only_attention(cpa):
    reqs = [(0, 200), (64, 33), (900, 1)]
    w = W.make_batch_workload("rope_write", W.Shape(8, 2, 128, 16, 512, "bf16"), reqs, seed=42)
    t = w.materialize("cuda")
    s = w.steps[0]
    sh = w.shape
    b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    q, kn, vn = t.step_inputs(s)
    ob = oracle.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    qr, kr = oracle.rope(ob, as_f64(q), as_f64(kn), num_heads_q=sh.num_heads_q, num_heads_kv=sh.num_heads_kv,
                         head_dim=128, theta=THETA)
    qr, kr = rounded(qr, "bf16"), rounded(kr, "bf16")
    k_pool0, v_pool0 = as_f64(t.k_cache), as_f64(t.v_cache)
    ref_o, ref_l = oracle.attention(ob, qr, kr, as_f64(vn), k_pool0, v_pool0, num_heads_q=sh.num_heads_q,
                                    num_heads_kv=sh.num_heads_kv, head_dim=128, block_size=16, scale=sh.scale)
    cpa.paged_kv_write(b, rope_params(w), kn, vn, t.k_cache, t.v_cache)
    out, lse = cpa.attention(b, rope_params(w, 0), q, kn, vn, t.k_cache, t.v_cache)
    torch.cuda.synchronize()
    assert cpa.last_device_error() == cpa.SUCCESS
    res = Result()
    res.add(out.float().cpu().numpy(), ref_o, lse.cpu().numpy(), ref_l)
    assert_within(res, "bf16")
    check_pool_keys(t.k_cache, t.v_cache, s, w.block_table, kr, vn, 16, "bf16")


def test_rope_chunked_prompt_matches_oracle(cpa):
    # a 1,000-token prompt in chunks of 384, 384, 232: each chunk's keys are
    # rotated at their absolute positions and kept rotated in the cache
    w = W.make_prompt_workload("rope_prompt", W.Shape(8, 2, 128, 16, 512, "bf16"), 1000, 384, 80, seed=43)
    t = w.materialize("cuda")
    sh = w.shape
    p = rope_params(w)
    k_pool_o = as_f64(t.k_cache)
    v_pool_o = as_f64(t.v_cache)
    res = Result()
    for s in w.steps:
        b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
        q, kn, vn = t.step_inputs(s)
        out, lse = cpa.attention(b, p, q, kn, vn, t.k_cache, t.v_cache)
        torch.cuda.synchronize()
        ob = oracle.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
        qr, kr = oracle.rope(ob, as_f64(q), as_f64(kn), num_heads_q=sh.num_heads_q, num_heads_kv=sh.num_heads_kv,
                             head_dim=128, theta=THETA)
        qr, kr = rounded(qr, "bf16"), rounded(kr, "bf16")
        ref_o, ref_l = oracle.attention(ob, qr, kr, as_f64(vn), k_pool_o, v_pool_o, num_heads_q=sh.num_heads_q,
                                        num_heads_kv=sh.num_heads_kv, head_dim=128, block_size=16, scale=sh.scale)
        res.add(out.float().cpu().numpy(), ref_o, lse.cpu().numpy(), ref_l)
        k_pool_o, v_pool_o = oracle.kv_write(ob, kr, as_f64(vn), k_pool_o, v_pool_o, num_heads_kv=sh.num_heads_kv,
                                             head_dim=128, block_size=16)
    assert cpa.last_device_error() == cpa.SUCCESS
    assert_within(res, "bf16")


def run_rope(cpa, w, *, flags=None, rows_per_req=None, steps_to_check=None, variant="plain", seed=0):
    """Every step of `w` with the rotary embedding applied in the call (fused
    write unless flags say otherwise, then the standalone write): outputs of
    the checked steps (all rows, or a sample) against the oracle's rotation
    rounded to bf16 then attention in fp64; after each step the pool's keys
    within one rounding step of the oracle's rotated keys and its values
    bit-exact."""
    sh = w.shape
    t = w.materialize("cuda")
    W.apply_variant(t, variant, sh.num_heads_q // sh.num_heads_kv)
    fl = cpa.FLAG_FUSE_KV_WRITE if flags is None else flags
    p = rope_params(w, fl)
    k_pool_o, v_pool_o = as_f64(t.k_cache), as_f64(t.v_cache)
    steps_to_check = range(len(w.steps)) if steps_to_check is None else steps_to_check
    res = Result()
    for si, s in enumerate(w.steps):
        b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
        q, kn, vn = t.step_inputs(s)
        out, lse = cpa.attention(b, p, q, kn, vn, t.k_cache, t.v_cache)
        if not fl & cpa.FLAG_FUSE_KV_WRITE:
            cpa.paged_kv_write(b, p, kn, vn, t.k_cache, t.v_cache)
        torch.cuda.synchronize()
        assert cpa.last_device_error() == cpa.SUCCESS
        ob = oracle.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
        qr, kr = oracle.rope(ob, as_f64(q), as_f64(kn), num_heads_q=sh.num_heads_q, num_heads_kv=sh.num_heads_kv,
                             head_dim=sh.head_dim, theta=THETA)
        qr, kr = rounded(qr, "bf16"), rounded(kr, "bf16")
        if si in steps_to_check:
            rows = None if rows_per_req is None else sample_rows(s, rows_per_req, seed + si)
            ref_o, ref_l = oracle.attention(ob, qr, kr, as_f64(vn), k_pool_o, v_pool_o,
                                            num_heads_q=sh.num_heads_q, num_heads_kv=sh.num_heads_kv,
                                            head_dim=sh.head_dim, block_size=sh.block_size, scale=sh.scale,
                                            rows=rows)
            idx = slice(None) if rows is None else torch.as_tensor(rows, device=out.device)
            res.add(out[idx].float().cpu().numpy(), ref_o, lse[idx].cpu().numpy(), ref_l)
        check_pool_keys(t.k_cache, t.v_cache, s, w.block_table, kr, vn, sh.block_size, "bf16")
        k_pool_o, v_pool_o = oracle.kv_write(ob, kr, as_f64(vn), k_pool_o, v_pool_o, num_heads_kv=sh.num_heads_kv,
                                             head_dim=sh.head_dim, block_size=sh.block_size)
    assert_within(res, "bf16")


# Tensor-core shapes with the rotation applied in the attention launch: G = 1
# (every row its own token), G = 16 and 32 (few tokens per query tile), head
# dimension 64 (both halves of a pair in one 128-byte row); prefills with and
# without cached keys, a ragged chunk and decodes (split units) side by side.
@pytest.mark.parametrize("hq,hkv,d,bs", [(8, 8, 128, 16), (16, 1, 128, 128), (8, 2, 64, 16), (64, 2, 128, 32),
                                         (28, 4, 128, 16)])
def test_rope_tensor_core_shapes(cpa, hq, hkv, d, bs):
    reqs = [(0, 300), (130, 77), (1000, 1), (257, 129), (4000, 1)]
    w = W.make_batch_workload(f"rope_tc_{hq}_{hkv}_{d}_{bs}", W.Shape(hq, hkv, d, bs, 512, "bf16"), reqs, seed=44)
    run_rope(cpa, w)


def test_rope_without_fused_write_and_with_tail_pieces(cpa):
    # no fused write: the rotated keys are only read (the standalone write
    # follows); then the opt-in tail cut, whose pieces each rotate their queries
    reqs = [(0, 700), (3000, 900), (50, 1)]
    w = W.make_batch_workload("rope_tail", W.Shape(32, 8, 128, 16, 1024, "bf16"), reqs, seed=45)
    run_rope(cpa, w, flags=0)
    run_rope(cpa, w, flags=cpa.FLAG_FUSE_KV_WRITE | cpa.FLAG_TAIL_SPLIT)


def test_rope_llama3_8b_prompt_sampled(cpa):
    # the 10,000-token prompt in 5 chunks of 2048 with theta 5e5, sharpened
    # queries: the first chunk (every key new: query tiles wait for the
    # rotation of their keys) and the last (8,192 cached keys) on sampled rows
    w = W.llama3_8b_prompt()
    run_rope(cpa, w, rows_per_req=24, steps_to_check=[0, 4], variant="peaky", seed=7)
