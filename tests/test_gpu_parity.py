"""GPU parity: the CUDA library against the fp64 oracle on the same seeded
inputs, through the C ABI.  BF16 outputs within max-abs 2e-2, FP32 within
1e-4, plus a relative gate on every checked (token, head) row and on each
step's relative RMS error; the paged K/V pool bit-exact.

Each measured configuration also runs with peaked queries ("peaky": times
4) and with "needle" queries (each row's own key and the key just past its
causal limit score far above the rest), so that outputs are O(1) and a
mask or position error confined to a few rows fails the gates
(workloads.apply_variant)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import (Result, assert_within, bits, params_for, run_and_compare, to_oracle)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cpa():
    import chunked_prefill_paged_gb300 as m
    m.load()
    return m


def small_batch(hq=8, hkv=2, d=128, bs=16, dtype="bf16", seg=512, reqs=None, seed=7):
    reqs = reqs or [(0, 300), (130, 77), (1000, 1), (17, 1), (257, 129), (0, 0), (64, 0), (5, 3)]
    return W.make_batch_workload(f"small_{hq}_{hkv}_{d}_{bs}_{dtype}", W.Shape(hq, hkv, d, bs, seg, dtype), reqs,
                                 seed=seed)


# ------------------------------------------------------------------ KV write
@pytest.mark.parametrize("dtype,bs,d", [("bf16", 16, 128), ("bf16", 128, 128), ("f32", 16, 64), ("bf16", 32, 64)])
def test_paged_kv_write_bit_exact(cpa, dtype, bs, d):
    w = small_batch(d=d, bs=bs, dtype=dtype)
    t = w.materialize("cuda")
    s = w.steps[0]
    b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    p = params_for(w)
    q, kn, vn = t.step_inputs(s)
    k_ref, v_ref = oracle.kv_write(oracle.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table),
                                   to_oracle(kn), to_oracle(vn), to_oracle(t.k_cache), to_oracle(t.v_cache),
                                   num_heads_kv=w.shape.num_heads_kv, head_dim=d, block_size=bs)
    cpa.paged_kv_write(b, p, kn, vn, t.k_cache, t.v_cache)
    torch.cuda.synchronize()
    vt = np.int16 if dtype == "bf16" else np.int32
    assert np.array_equal(bits(t.k_cache), k_ref.view(vt))
    assert np.array_equal(bits(t.v_cache), v_ref.view(vt))
    assert cpa.last_device_error() == cpa.SUCCESS


# ------------------------------------------------------- small, every row
def test_tiny_fp32_config(cpa):
    w = W.tiny_fp32()
    res = run_and_compare(w)
    assert_within(res, "f32")


@pytest.mark.parametrize("hq,hkv,d,bs", [(8, 2, 128, 16), (8, 2, 128, 128), (8, 1, 128, 32), (16, 2, 64, 64),
                                         (4, 4, 128, 16), (32, 4, 128, 16)])
@pytest.mark.parametrize("variant", W.VARIANTS)
def test_small_batch_tensor_cores(cpa, hq, hkv, d, bs, variant):
    w = small_batch(hq, hkv, d, bs)
    res = run_and_compare(w, variant=variant)
    assert_within(res, "bf16")


# query groups that do not divide 128 run on the tensor cores with query tiles
# of G * floor(128 / G) rows (126, 125, 120): a token's rows never straddle
# two tiles, and the MMA rows past them carry nothing to an output
@pytest.mark.parametrize("hq,hkv,d,bs", [(6, 2, 128, 16), (28, 4, 128, 16), (12, 2, 64, 128), (20, 4, 128, 32),
                                         (24, 2, 128, 16)])
@pytest.mark.parametrize("variant", W.VARIANTS)
def test_small_batch_tensor_cores_uneven_groups(cpa, hq, hkv, d, bs, variant):
    w = small_batch(hq, hkv, d, bs)
    res = run_and_compare(w, variant=variant)
    assert_within(res, "bf16")


def test_uneven_group_with_the_tail_cut_and_no_split(cpa):
    w = small_batch(28, 4, 128, 16, reqs=[(3000, 900), (0, 700), (5000, 1), (70, 3)], seed=9)
    res = run_and_compare(w, flags=cpa.FLAG_FUSE_KV_WRITE | cpa.FLAG_TAIL_SPLIT)
    assert_within(res, "bf16")
    res = run_and_compare(w, flags=cpa.FLAG_FUSE_KV_WRITE | cpa.FLAG_NO_SPLIT, variant="needle")
    assert_within(res, "bf16")


def test_small_batch_cuda_cores_bf16(cpa):
    w = small_batch()
    res = run_and_compare(w, flags=cpa.FLAG_FUSE_KV_WRITE | cpa.FLAG_FORCE_SIMT)
    assert_within(res, "bf16")


def test_small_batch_fp32_cuda_cores(cpa):
    w = small_batch(d=64, dtype="f32")
    res = run_and_compare(w)
    assert_within(res, "f32")


@pytest.mark.parametrize("seg", [512, 1024, 2048, 4096])
def test_split_kv_decodes_every_segment_size(cpa, seg):
    reqs = [(5000, 1), (4095, 1), (4096, 1), (777, 1), (9000, 3), (0, 1), (1, 1), (2300, 16)]
    w = small_batch(reqs=reqs, seg=seg, seed=11)
    res = run_and_compare(w, kv_segment_size=seg)
    assert_within(res, "bf16")


def test_no_split_matches_split(cpa):
    reqs = [(5000, 1), (3000, 2), (123, 1)]
    w = small_batch(reqs=reqs, seed=12)
    res = run_and_compare(w, flags=cpa.FLAG_FUSE_KV_WRITE | cpa.FLAG_NO_SPLIT)
    assert_within(res, "bf16")


def test_standalone_write_then_read_only_attention(cpa):
    w = small_batch(seed=13)
    res = run_and_compare(w, flags=0)
    assert_within(res, "bf16")


@pytest.mark.parametrize("variant", W.VARIANTS)
def test_chunked_prompt_multistep_fused_write(cpa, variant):
    sh = W.Shape(16, 4, 128, 16, 512, "bf16")
    w = W.make_prompt_workload("prompt700", sh, 700, 256, 64, seed=14)
    res = run_and_compare(w, variant=variant)
    assert_within(res, "bf16")


def test_first_token_of_fresh_prompt_returns_its_value_row(cpa):
    # C = 0: token 0 sees only itself, p = 1, l = 1, so out = v_0 exactly
    w = small_batch(reqs=[(0, 40), (0, 1)], seed=15)
    t = w.materialize("cuda")
    s = w.steps[0]
    b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    q, kn, vn = t.step_inputs(s)
    out, _ = cpa.attention(b, params_for(w), q, kn, vn, t.k_cache, t.v_cache)
    G = w.shape.num_heads_q // w.shape.num_heads_kv
    for tok in (0, 40):
        for h in range(w.shape.num_heads_q):
            assert torch.equal(out[tok, h], vn[tok, h // G])


@pytest.mark.parametrize("variant", ["plain", "needle"])
def test_chunking_invariance_against_one_shot_oracle(cpa, variant):
    # the same prompt in one chunk and in uneven chunks: every chunking's
    # outputs match the oracle's one-shot causal attention over the whole
    # prompt ("Prefill Optimisation" section 2, causal equivalence)
    sh = W.Shape(8, 2, 128, 16, 512, "bf16")
    L = 600
    ref = None
    for chunk in (600, 200, 137):
        w = W.make_prompt_workload("inv", sh, L, chunk, 64, seed=16)
        t = w.materialize("cuda")
        W.apply_variant(t, variant, sh.num_heads_q // sh.num_heads_kv)
        p = params_for(w)
        rows, lses = [], []
        for step in w.steps:
            b = cpa.Batch(step.cached_seq_len, step.num_new_tokens, w.block_table)
            q, kn, vn = t.step_inputs(step)
            o, l = cpa.attention(b, p, q, kn, vn, t.k_cache, t.v_cache)
            rows.append(o.float().cpu().numpy())
            lses.append(l.cpu().numpy())
        torch.cuda.synchronize()
        if ref is None:
            # one request, nothing cached, the whole prompt active
            ob = oracle.Batch([0], [L], w.block_table)
            ref = oracle.attention(ob, to_oracle(t.q), to_oracle(t.k), to_oracle(t.v), to_oracle(t.k_cache),
                                   to_oracle(t.v_cache), num_heads_q=sh.num_heads_q,
                                   num_heads_kv=sh.num_heads_kv, head_dim=sh.head_dim,
                                   block_size=sh.block_size, scale=sh.scale)
        res = Result()
        res.add(np.concatenate(rows), ref[0], np.concatenate(lses), ref[1])
        assert_within(res, "bf16")


# ------------------------------------------------------------ edge cases
def test_empty_batch_and_zero_token_requests(cpa):
    w = small_batch(reqs=[(10, 0), (0, 0)], seed=17)
    t = w.materialize("cuda")
    s = w.steps[0]
    b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    q = torch.empty((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    kv = torch.empty((0, 2, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    before = bits(t.k_cache)
    cpa.chunked_prefill_attention(b, params_for(w), q, kv, kv, t.k_cache, t.v_cache, out)
    cpa.paged_kv_write(b, params_for(w), kv, kv, t.k_cache, t.v_cache)
    torch.cuda.synchronize()
    assert np.array_equal(bits(t.k_cache), before)


def test_invalid_arguments_are_rejected(cpa):
    w = small_batch(seed=18)
    t = w.materialize("cuda")
    s = w.steps[0]
    b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    q, kn, vn = t.step_inputs(s)
    out = torch.empty_like(q)
    bad = params_for(w, kv_segment_size=768)
    with pytest.raises(cpa.CpaError) as e:
        cpa.chunked_prefill_attention(b, bad, q, kn, vn, t.k_cache, t.v_cache, out)
    assert e.value.status == cpa.ERR_INVALID_ARG
    decodes = small_batch(reqs=[(5000, 1)], seed=19)
    td = decodes.materialize("cuda")
    sd = decodes.steps[0]
    bd = cpa.Batch(sd.cached_seq_len, sd.num_new_tokens, decodes.block_table)
    qd, knd, vnd = td.step_inputs(sd)
    with pytest.raises(cpa.CpaError) as e:
        cpa.chunked_prefill_attention(bd, params_for(decodes), qd, knd, vnd, td.k_cache, td.v_cache,
                                      torch.empty_like(qd))
    assert e.value.status == cpa.ERR_WORKSPACE


# ------------------------------------------- the measured workloads, sampled
@pytest.mark.parametrize("variant", W.VARIANTS)
def test_config_llama3_8b_prompt(cpa, variant):
    res = run_and_compare(W.llama3_8b_prompt(), rows_per_req=24, variant=variant)
    assert_within(res, "bf16")


@pytest.mark.parametrize("variant", W.VARIANTS)
def test_config_prefix_cache(cpa, variant):
    res = run_and_compare(W.prefix_cache(), rows_per_req=4, variant=variant)
    assert_within(res, "bf16")


@pytest.mark.parametrize("variant", W.VARIANTS)
def test_config_mixed_step(cpa, variant):
    res = run_and_compare(W.mixed_step(), rows_per_req=3, variant=variant)
    assert_within(res, "bf16")


@pytest.mark.parametrize("variant", ["plain", "needle"])
def test_speculative_decode_queries(cpa, variant):
    # short causal chunks (1 + 4 draft tokens) over long contexts, split into
    # kv_segment_size pieces and merged
    res = run_and_compare(W.speculative_decode(num_reqs=16), rows_per_req=2, variant=variant)
    assert_within(res, "bf16")


@pytest.mark.parametrize("variant", W.VARIANTS)
def test_config_long_context(cpa, variant):
    res = run_and_compare(W.long_context(), rows_per_req=6, steps_to_check=[0, 7, 15], variant=variant)
    assert_within(res, "bf16")


# ------------------------------------------------------ two CTA groups (planner)
@pytest.mark.parametrize("C", [2048, 4096, 6144])
def test_two_cta_groups_write_every_row(cpa, C):
    """A chunk of 2048 query tokens over C cached ones (H 32/8, bs 128): 512
    units on 152 SMs, which the planner runs as two CTA groups, each claiming
    from its own counter and then from the other's (the planner tests check
    that choice).  A unit never claimed would leave its rows unwritten: the
    output and LSE start as NaN and every row must be written; sampled rows
    match the oracle and the pool's new rows are the oracle's write."""
    _groups_write_every_row(cpa, small_batch(hq=32, hkv=8, bs=128, seg=1024, reqs=[(C, 2048)], seed=40 + C // 2048),
                            rows_per_req=48, seed=C)


def test_two_cta_groups_head_dim_64(cpa):
    """The same with d 64 and G 1 (H 24/24, bs 128): 384 units, which the
    planner runs as 72 CTAs taking 2 of the heaviest units and 80 taking 3 of
    the lightest; a quarter of the rows against the oracle."""
    _groups_write_every_row(cpa, small_batch(hq=24, hkv=24, d=64, bs=128, seg=1024, reqs=[(2048, 2048)], seed=61),
                            rows_per_req=512, seed=61)


def _groups_write_every_row(cpa, w, rows_per_req, seed):
    hq = w.shape.num_heads_q
    t = w.materialize("cuda")
    s = w.steps[0]
    b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    p = params_for(w)
    q, kn, vn = t.step_inputs(s)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((s.total_new_tokens, hq), float("nan"), dtype=torch.float32, device="cuda")
    n = cpa.workspace_size(b, p)
    ws = torch.empty((max(n, 16) + 3) // 4, dtype=torch.float32, device="cuda")
    cpa.chunked_prefill_attention(b, p, q, kn, vn, t.k_cache, t.v_cache, out, lse, ws)
    torch.cuda.synchronize()
    assert cpa.last_device_error() == cpa.SUCCESS
    assert bool(torch.isfinite(out).all()), "output rows left unwritten"
    assert bool(torch.isfinite(lse).all()), "LSE rows left unwritten"
    res = run_and_compare(w, rows_per_req=rows_per_req, seed=seed)
    assert_within(res, "bf16")
