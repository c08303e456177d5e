"""chunked_prefill_attention_no_alloc: the attention call for callers that
cannot allocate device memory (a plugin whose host application owns all
device memory, or a serving loop that must not call cudaMalloc because it can
synchronise the device).  Its split-KV partials live in the library's static
device array instead of a caller workspace.

Called through the C ABI and compared with chunked_prefill_attention (with a
torch-allocated workspace) on the same inputs, twice in a row: the static
array keeps the previous call's contents, and the second call must not
depend on them.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from helpers import BF16_ATOL, BF16_LSE_ATOL, params_for

pytestmark = pytest.mark.gpu


def test_no_alloc_matches_workspace_entry_point_twice():
    import chunked_prefill_paged_gb300 as cpa
    lib = cpa.load()
    # decodes with long contexts take the split-KV path (the one that needs
    # scratch), the prefill chunks the direct path
    reqs = [(5000, 1), (3000, 1), (12000, 1), (700, 1), (0, 200), (900, 130)]
    w = W.make_batch_workload("no_alloc", W.Shape(32, 8, 128, 16, 1024, "bf16"), reqs, seed=31)
    t = w.materialize("cuda")
    s = w.steps[0]
    b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    p = params_for(w)
    need = cpa.workspace_size(b, p)
    assert 0 < need <= (32 << 20)
    q, kn, vn = t.step_inputs(s)

    ref_out, ref_lse = cpa.attention(b, p, q, kn, vn, t.k_cache, t.v_cache)
    torch.cuda.synchronize()

    cb, cp = b.c(), p.c()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        rc = lib.chunked_prefill_attention_no_alloc(ctypes.byref(cb), ctypes.byref(cp), q.data_ptr(), kn.data_ptr(),
                                                    vn.data_ptr(), t.k_cache.data_ptr(), t.v_cache.data_ptr(),
                                                    out.data_ptr(), lse.data_ptr(), stream)
        assert rc == cpa.SUCCESS, cpa.status_string(rc)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        assert (out.float() - ref_out.float()).abs().max().item() <= BF16_ATOL
        assert (lse - ref_lse).abs().max().item() <= BF16_LSE_ATOL
    assert cpa.last_device_error() == cpa.SUCCESS


def test_no_alloc_rejects_batches_beyond_its_array():
    import chunked_prefill_paged_gb300 as cpa
    # 2,000 decodes of 32k context each need far more than 32 MiB of partials
    n = 2000
    b = cpa.Batch([32000] * n, [1] * n, np.zeros((n, 2001), dtype=np.int32))
    p = cpa.Params(32, 8, 128, 16, 100000, 1024)
    assert cpa.workspace_size(b, p) > (32 << 20)
    x = torch.empty((n, 32, 128), dtype=torch.bfloat16, device="cuda")
    kv = torch.empty((n, 8, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cpa.CpaError) as e:
        cpa.chunked_prefill_attention_no_alloc(b, p, x, kv, kv, kv, kv, x)
    assert e.value.status == cpa.ERR_WORKSPACE
