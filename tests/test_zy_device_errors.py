"""Device-side failure reporting without a GPU fault: a block id outside the
pool is skipped and reported; a wait that nothing will satisfy expires after
its bound and the launch reports a timeout; the context stays usable."""
import pytest
import torch

import workloads as W
from helpers import params_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cpa():
    import chunked_prefill_paged_gb300 as m
    m.load()
    assert m.last_device_error() == m.SUCCESS
    return m


def _small(reqs, seed):
    return W.make_batch_workload("err", W.Shape(8, 2, 128, 16, 512, "bf16"), reqs, seed=seed)


@pytest.mark.parametrize("simt", [False, True])
def test_bad_block_id_is_reported(cpa, simt):
    w = _small([(200, 40)], seed=21)
    bt = w.block_table.copy()
    bt[0, 3] = w.num_blocks + 7  # a cached block outside the pool
    t = w.materialize("cuda")
    s = w.steps[0]
    b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, bt)
    flags = cpa.FLAG_FUSE_KV_WRITE | (cpa.FLAG_FORCE_SIMT if simt else 0)
    q, kn, vn = t.step_inputs(s)
    cpa.attention(b, params_for(w, flags=flags), q, kn, vn, t.k_cache, t.v_cache)
    assert cpa.last_device_error() == cpa.ERR_BAD_BLOCK_ID
    assert cpa.last_device_error() == cpa.SUCCESS  # reading clears it


def test_stalled_wait_times_out_and_context_survives(cpa):
    w = _small([(300, 64)], seed=22)
    t = w.materialize("cuda")
    s = w.steps[0]
    b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    q, kn, vn = t.step_inputs(s)
    p = params_for(w, flags=cpa.FLAG_TEST_STALL, timeout_cycles=2_000_000)
    cpa.attention(b, p, q, kn, vn, t.k_cache, t.v_cache)
    assert cpa.last_device_error() == cpa.ERR_DEVICE_TIMEOUT
    # the context is still usable: a normal launch succeeds afterwards
    out, _ = cpa.attention(b, params_for(w), q, kn, vn, t.k_cache, t.v_cache)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    assert cpa.last_device_error() == cpa.SUCCESS
