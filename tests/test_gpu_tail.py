"""Tail pieces on the GPU.  When a prefill batch's query tiles would leave
the last wave of CTAs partly idle, the planner (with CPA_FLAG_TAIL_SPLIT)
cuts the last few tiles (by work index) into pieces by key tiles; each piece
writes a partial (unnormalised output, running maximum, sum) and the CTA
finishing a tile's last piece merges them -- the same online-softmax merge as split decodes ("Prefill
Processing", Partial KV Segment Handling: pieces of one query's keys combine
to the unsplit result).  Each case checks that the cut is active (the
workspace grows by the partials), compares every row of the cut tiles and
a sample of the others with the fp64 oracle, and compares the output with
the same call without CPA_FLAG_TAIL_SPLIT (the cut is opt-in)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import BF16_ATOL, BF16_LSE_ATOL, params_for, to_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cpa():
    import chunked_prefill_paged_gb300 as m
    m.load()
    return m


def run_case(cpa, w, rows):
    sh = w.shape
    t = w.materialize("cuda")
    s = w.steps[0]
    b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    p_tail = params_for(w, flags=cpa.FLAG_TAIL_SPLIT)  # read-only: both calls see the same pool
    p_none = params_for(w, flags=0)
    assert cpa.workspace_size(b, p_tail) > cpa.workspace_size(b, p_none), "no tail cut planned"
    q, kn, vn = t.step_inputs(s)
    out, lse = cpa.attention(b, p_tail, q, kn, vn, t.k_cache, t.v_cache)
    out_n, lse_n = cpa.attention(b, p_none, q, kn, vn, t.k_cache, t.v_cache)
    torch.cuda.synchronize()
    assert cpa.last_device_error() == cpa.SUCCESS
    ob = oracle.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    ref_o, ref_l = oracle.attention(ob, to_oracle(q), to_oracle(kn), to_oracle(vn), to_oracle(t.k_cache),
                                    to_oracle(t.v_cache), num_heads_q=sh.num_heads_q, num_heads_kv=sh.num_heads_kv,
                                    head_dim=sh.head_dim, block_size=sh.block_size, scale=sh.scale, rows=rows)
    idx = torch.as_tensor(rows, device=out.device)
    got = out[idx].float().cpu().numpy()
    assert np.all(np.isfinite(got))
    err = float(np.abs(got - ref_o).max())
    lse_err = float(np.abs(lse[idx].cpu().numpy() - ref_l).max())
    assert err <= BF16_ATOL, err
    assert lse_err <= BF16_LSE_ATOL, lse_err
    # the cut changes only the order of the fp32 sums
    assert float((out.float() - out_n.float()).abs().max()) <= 2e-2
    assert float((lse - lse_n).abs().max()) <= 1e-3


def test_tail_pieces_llama_chunk(cpa):
    # the fourth chunk of the Llama-3-8B-shaped prompt: 512 query tiles of
    # about 56 key tiles on 152 SMs; the last tiles by index are the first
    # query tiles of the chunk (tokens 0 .. 223), kv head innermost
    w = W.make_batch_workload("tail_llama", W.Shape(32, 8, 128, 128, 1024, "bf16"), [(6144, 2048)], seed=91)
    rows = list(range(0, 256)) + [300, 777, 1500, 2047]
    run_case(cpa, w, rows)


def test_tail_pieces_several_requests_block_16(cpa):
    # two prompts continuing from unaligned cached lengths (bs 16), ragged
    # last query tiles; the last units by index are the second request's
    # first query tiles (rows 1003 .. 1258)
    w = W.make_batch_workload("tail_two", W.Shape(32, 8, 128, 16, 1024, "bf16"), [(8100, 1003), (9003, 1040)],
                              seed=92)
    rows = [0, 500, 1002] + list(range(1003, 1300)) + [2042]
    run_case(cpa, w, rows)


def test_tail_pieces_head_major(cpa):
    # K/V larger than half of L2: units walk kv head by kv head, so the cut
    # tiles are the first query tiles of the last kv head (query heads 28-31)
    w = W.make_batch_workload("tail_head_major", W.Shape(32, 8, 128, 16, 1024, "bf16"), [(16384, 2048)], seed=93)
    rows = list(range(0, 1792, 8)) + [2047]
    run_case(cpa, w, rows)
