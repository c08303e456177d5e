"""The split planner's fine tail on the GPU.  When the planner lengthens the
kv_segment_size pieces of a decode-heavy batch, the last requests in batch
order (enough for three waves of CTAs on the device) cut their keys into
pieces half as long, so the launch's last units are short.  The workspace
size the library asks for pins the plan (partials per piece and kv head);
every row is compared with the fp64 oracle ("Prefill Processing", Partial KV
Segment Handling: the pieces of one query's keys merge to the unsplit
result)."""
import pytest
import torch

import workloads as W
from helpers import assert_within, params_for, run_and_compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cpa():
    import chunked_prefill_paged_gb300 as m
    m.load()
    return m


def partial_floats(rows, d):
    return rows * d + ((2 * rows + 3) & ~3)


def test_fine_tail_plan_and_parity(cpa):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    w = W.decode_batch(num_reqs=32, ctx=8192)
    sh = w.shape
    s = w.steps[0]
    b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    p = params_for(w)
    G, keys = sh.num_heads_q // sh.num_heads_kv, 8192 + 1
    # 32 x 5 pieces of 2048 keys x 8 heads = 1280 units >= 1024, 4096-key
    # pieces would leave 768: the planner takes 2048; the fine pieces are
    # 1024 keys (9 per request, 72 units), for ceil(3 * sms / 72) requests
    fine_reqs = -(-3 * sms // (9 * sh.num_heads_kv))
    pieces = (32 - fine_reqs) * -(-keys // 2048) + fine_reqs * -(-keys // 1024)
    ws_floats = pieces * sh.num_heads_kv * partial_floats(G, sh.head_dim)
    expect = ((ws_floats * 4 + 255) // 256) * 256 + 256  # then the work counter
    assert cpa.workspace_size(b, p) == expect
    res = run_and_compare(w)
    assert_within(res, "bf16")


def test_fine_tail_not_taken_when_pieces_are_not_lengthened(cpa):
    # 8 decodes: the pieces stay at kv_segment_size, so no fine tail
    w = W.decode_batch(num_reqs=8, ctx=8192)
    sh = w.shape
    s = w.steps[0]
    b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    p = params_for(w)
    G = sh.num_heads_q // sh.num_heads_kv
    ws_floats = 8 * -(-8193 // 1024) * sh.num_heads_kv * partial_floats(G, sh.head_dim)
    assert cpa.workspace_size(b, p) == ((ws_floats * 4 + 255) // 256) * 256 + 256
    res = run_and_compare(w)
    assert_within(res, "bf16")
