"""chunked_prefill_attention_no_alloc: the attention call for callers that
cannot allocate device memory (a plugin whose host application owns all
device memory, or a serving loop that must not call cudaMalloc because it can
synchronise the device).  Its workspace lives in the library's static device
array instead of a caller buffer.

Called through the C ABI and compared with chunked_prefill_attention (with a
torch-allocated workspace) on the same inputs: the two run the same plan and
the same kernels, so the outputs must be bit-identical; both are also held
to the fp64 oracle.  Between the two compared calls another no-alloc call on
a different batch (other contexts, tail pieces) leaves unrelated partials
and counters in the static array, so a kernel that read scratch before
writing it would show.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import Result, assert_within, params_for, to_oracle

pytestmark = pytest.mark.gpu


def no_alloc(cpa, lib, b, p, q, kn, vn, kc, vc, out, lse):
    cb, cp = b.c(), p.c()
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.chunked_prefill_attention_no_alloc(ctypes.byref(cb), ctypes.byref(cp), q.data_ptr(), kn.data_ptr(),
                                                vn.data_ptr(), kc.data_ptr(), vc.data_ptr(), out.data_ptr(),
                                                lse.data_ptr(), stream)
    assert rc == cpa.SUCCESS, cpa.status_string(rc)


def test_no_alloc_is_bit_identical_to_the_workspace_entry_point():
    import chunked_prefill_paged_gb300 as cpa
    lib = cpa.load()
    # decodes with long contexts take the split-KV path (the one that needs
    # scratch), the prefill chunks the direct path
    sh = W.Shape(32, 8, 128, 16, 1024, "bf16")
    reqs = [(5000, 1), (3000, 1), (12000, 1), (700, 1), (0, 200), (900, 130)]
    w = W.make_batch_workload("no_alloc", sh, reqs, seed=31)
    t = w.materialize("cuda")
    s = w.steps[0]
    b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    p = params_for(w, flags=0)  # read-only pool: every call sees the same cache
    need = cpa.workspace_size(b, p)
    assert 0 < need <= cpa.NO_ALLOC_WORKSPACE_BYTES
    q, kn, vn = t.step_inputs(s)

    # a different batch that fills the static array with other partials and
    # tail-piece counters: a long chunk cut into tail pieces, and decodes
    w2 = W.make_batch_workload("no_alloc_other", sh, [(6144, 2048), (20000, 1), (9000, 1)], seed=32)
    t2 = w2.materialize("cuda")
    s2 = w2.steps[0]
    b2 = cpa.Batch(s2.cached_seq_len, s2.num_new_tokens, w2.block_table)
    p2 = params_for(w2, flags=cpa.FLAG_TAIL_SPLIT)
    assert cpa.workspace_size(b2, p2) <= cpa.NO_ALLOC_WORKSPACE_BYTES
    q2, kn2, vn2 = t2.step_inputs(s2)

    ref_out, ref_lse = cpa.attention(b, p, q, kn, vn, t.k_cache, t.v_cache)
    torch.cuda.synchronize()
    outs = []
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        no_alloc(cpa, lib, b, p, q, kn, vn, t.k_cache, t.v_cache, out, lse)
        if call == 0:
            o2, l2 = torch.empty_like(q2), torch.empty((q2.shape[0], q2.shape[1]), dtype=torch.float32,
                                                         device="cuda")
            no_alloc(cpa, lib, b2, p2, q2, kn2, vn2, t2.k_cache, t2.v_cache, o2, l2)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out), f"call {call}: output differs from the workspace entry point"
        assert torch.equal(lse, ref_lse), f"call {call}: lse differs from the workspace entry point"
        outs.append(out)
    assert cpa.last_device_error() == cpa.SUCCESS

    ob = oracle.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    ref_o, ref_l = oracle.attention(ob, to_oracle(q), to_oracle(kn), to_oracle(vn), to_oracle(t.k_cache),
                                    to_oracle(t.v_cache), num_heads_q=sh.num_heads_q, num_heads_kv=sh.num_heads_kv,
                                    head_dim=sh.head_dim, block_size=sh.block_size, scale=sh.scale)
    res = Result()
    res.add(outs[1].float().cpu().numpy(), ref_o, ref_lse.cpu().numpy(), ref_l)
    assert_within(res, "bf16")


def test_no_alloc_rejects_batches_beyond_its_array():
    import chunked_prefill_paged_gb300 as cpa
    # 2,000 decodes of 32k context each need far more than 32 MiB of partials
    n = 2000
    b = cpa.Batch([32000] * n, [1] * n, np.zeros((n, 2001), dtype=np.int32))
    p = cpa.Params(32, 8, 128, 16, 100000, 1024)
    assert cpa.workspace_size(b, p) > cpa.NO_ALLOC_WORKSPACE_BYTES
    x = torch.empty((n, 32, 128), dtype=torch.bfloat16, device="cuda")
    kv = torch.empty((n, 8, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cpa.CpaError) as e:
        cpa.chunked_prefill_attention_no_alloc(b, p, x, kv, kv, kv, kv, x)
    assert e.value.status == cpa.ERR_WORKSPACE
