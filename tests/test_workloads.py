"""The host-side schedules, counters and input recipe against the numbers the
pages print (tests/golden/pages_examples.json, each value cited there)."""
import json
import os

import numpy as np
import pytest

import workloads as W

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_examples.json")))


@pytest.mark.parametrize("case", GOLDEN["pairs"])
def test_pair_counts(case):
    assert W.pairs(case["cached"], case["new"]) == case["pairs"]


@pytest.mark.parametrize("case", GOLDEN["pair_terms"])
def test_pair_terms(case):
    C, N = case["cached"], case["new"]
    assert W.pairs(C, N) - W.pairs(0, N) == case["suffix_prefix"]
    assert W.pairs(0, N) == case["suffix_suffix"]


@pytest.mark.parametrize("case", GOLDEN["prefix_match"])
def test_full_block_prefix_reuse(case):
    bs = case["block_size"]
    cached = (case["matched_prefix"] // bs) * bs
    assert cached == case["cached"]
    assert case["prompt"] - cached == case["fresh"]


@pytest.mark.parametrize("case", GOLDEN["chunk_schedules"])
def test_chunk_schedules(case):
    assert W.chunk_schedule(case["prompt"], case["decodes"], case["budget"]) == case["chunks"]


@pytest.mark.parametrize("case", GOLDEN["budget_exhausted"])
def test_budget_exhaustion_raises(case):
    with pytest.raises(RuntimeError):
        W.chunk_schedule(case["prompt"], case["decodes"], case["budget"])


def test_segmentation_steps_of_the_10k_prompt():
    g = GOLDEN["segmentation_steps"]
    w = W.llama3_8b_prompt()
    assert [int(s.cached_seq_len[0]) for s in w.steps] == g["cached_seq_len"]
    assert [int(s.num_new_tokens[0]) for s in w.steps] == g["active"]
    assert sum(w.pairs_per_step()) == W.pairs(0, g["prompt"])  # chunking keeps the pair count


@pytest.mark.parametrize("case", GOLDEN["segment_counts"])
def test_segment_counts(case):
    assert case["cached_seq_len"] // case["kv_segment_size"] == case["segments"]


def test_partial_segment():
    g = GOLDEN["partial_segment"]
    assert g["cached_seq_len"] // g["kv_segment_size"] == g["full_segments"]
    assert g["cached_seq_len"] % g["kv_segment_size"] == g["partial_valid"]


@pytest.mark.parametrize("case", GOLDEN["blocks_needed"])
def test_blocks_needed(case):
    assert W.cdiv(case["tokens"], case["block_size"]) == case["blocks"]


@pytest.mark.parametrize("case", GOLDEN["kv_bytes"])
def test_kv_bytes_per_token(case):
    # one token, no queries or outputs: only the cache-side K and V rows
    per_layer = W.algorithmic_bytes([1], [0], 0, case["heads_kv"], case["head_dim"], case["elem_bytes"])
    assert per_layer * case["layers"] == case["bytes_per_token"]


def test_mixed_step_schedule_fills_the_budget():
    w = W.mixed_step()
    s = w.steps[0]
    new = s.num_new_tokens
    assert int(new.sum()) == 2048
    assert list(new[:64]) == [1] * 64
    assert list(new[64:]) == [512, 512, 512, 448]
    assert all(1024 <= c <= 32768 for c in s.cached_seq_len[:64])
    assert all(c % 512 == 0 and 0 <= c <= 16384 for c in s.cached_seq_len[64:])


def test_workload_shapes():
    t = W.tiny_fp32()
    assert (t.shape.num_heads_q, t.shape.num_heads_kv, t.shape.head_dim, t.shape.block_size) == (4, 1, 64, 16)
    assert t.num_blocks == 64 and int(t.steps[0].cached_seq_len[0]) == 256
    assert sum(t.pairs_per_step()) == 41024
    p = W.prefix_cache()
    shared = p.block_table[:, :256]
    assert (shared == shared[0]).all()
    own = [set(p.block_table[r, 256:W.cdiv(4096 + int(n), 16)].tolist()) for r, n in
           enumerate(p.steps[0].num_new_tokens)]
    for i in range(16):
        assert not (own[i] & set(shared[0].tolist()))
        for j in range(i):
            assert not (own[i] & own[j])
    lc = W.long_context()
    assert len(lc.steps) == 16 and int(lc.steps[-1].cached_seq_len[0]) == 30720
    assert sum(lc.pairs_per_step()) == 536887296


def test_decode_batch_shape():
    # the small decode-only profiling case: 32 decodes over 8192 cached
    # tokens, 513 blocks of 16 each, pool = needed + 10 %
    w = W.decode_batch()
    s = w.steps[0]
    assert w.num_reqs == 32 and s.cached_seq_len.tolist() == [8192] * 32 and s.num_new_tokens.tolist() == [1] * 32
    need = 32 * W.cdiv(8193, 16)
    assert w.num_blocks == need + -(-need // 10)
    assert (w.shape.num_heads_q, w.shape.num_heads_kv, w.shape.head_dim, w.shape.block_size) == (32, 8, 128, 16)


def test_block_tables_hold_distinct_physical_blocks():
    for w in (W.llama3_8b_prompt(), W.mixed_step(), W.long_context(), W.decode_batch()):
        used = []
        for r in range(w.num_reqs):
            last = w.steps[-1]
            C = int(last.cached_seq_len[r]) if w.num_reqs > 1 else int(last.cached_seq_len[0])
            N = int(last.num_new_tokens[r]) if w.num_reqs > 1 else int(last.num_new_tokens[0])
            used.extend(w.block_table[r, :W.cdiv(C + N, w.shape.block_size)].tolist())
        assert len(used) == len(set(used))
        assert max(used) < w.num_blocks and min(used) >= 0
        assert w.block_table.min() >= 0 and w.block_table.max() < w.num_blocks


def test_materialized_pool_has_sentinels_outside_cached_slots():
    w = W.make_batch_workload("t", W.Shape(4, 2, 8, 16, 512, "bf16"), [(37, 3), (0, 5), (16, 1)], seed=3)
    t = w.materialize("cpu")
    k = t.k_cache.float().numpy()
    # request 0: 37 cached tokens = 2 full blocks + 5 slots of a third
    b = w.block_table[0]
    assert np.isfinite(k[b[0]]).all() and np.isfinite(k[b[1]]).all()
    assert np.isfinite(k[b[2], :5]).all() and np.isnan(k[b[2], 5:]).all()
    n_finite_blocks = int(np.isfinite(k).any(axis=(1, 2, 3)).sum())
    assert n_finite_blocks == 3 + 1  # request 2 holds one full cached block
