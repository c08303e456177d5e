"""The GPU parity gates bite at full size: evaluated on the CPU, an oracle
with a planted mask or position mistake fails exactly the gates the GPU
parity tests apply, on the rows those tests sample from the Llama-3-8B
prompt (5 chunks of 2048, bs 128) and from the 32k long-context prompt
(16 chunks of 2048, H_q 64, bs 16), while the unmodified oracle's result
rounded to bf16 passes them.

With N(0, 1) queries over thousands of keys the softmax is nearly flat and
outputs are about 0.01-0.05 in size, so the 2e-2 max-abs bound alone could
not see a one-key mask error on a late chunk.  The "needle" queries
(workloads.apply_variant) put most of each row's weight on its own key and
make the key just past its causal limit just as strong, so a dropped
diagonal or one key too many changes the row by O(1) on every chunk.  No
GPU kernel is involved: the planted mistakes live in the oracle
("Prefill Optimisation" section 2, causal equivalence: token i of a chunk
at cached_seq_len C sees keys 0 .. C + i)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import Result, gate_failures, sample_rows, to_oracle

# (workload, rows sampled per request, checked steps): as in test_gpu_parity.
# Each check here takes about four of the rows those tests sample per step
# (the gates are maxima over rows, so failing on a subset fails on the set).
CASES = {
    "llama3_8b_prompt": (W.llama3_8b_prompt, 24, [0, 1, 2, 3, 4]),
    "long_context": (W.long_context, 6, [15]),
}
MUTATIONS = {
    "drop_diagonal": oracle.MUT_DROP_DIAGONAL,
    "sees_next_key": oracle.MUT_SEES_NEXT_KEY,
    "no_position_offset": oracle.MUT_NO_POSITION_OFFSET,
}


def bf16_values(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x).to(torch.bfloat16).float().numpy()


_views = {}
_refs = {}


def step_views(name, variant):
    """Per checked step: the oracle batch, inputs, pools as the step sees
    them (the oracle's own writes of the earlier chunks) and rows."""
    key = (name, variant)
    if key in _views:
        return _views[key]
    make, per_req, checked = CASES[name]
    w = make()
    sh = w.shape
    t = w.materialize("cpu")
    W.apply_variant(t, variant, sh.num_heads_q // sh.num_heads_kv)
    q, k, v = to_oracle(t.q), to_oracle(t.k), to_oracle(t.v)
    kp, vp = to_oracle(t.k_cache), to_oracle(t.v_cache)
    views = []
    for si, step in enumerate(w.steps):
        ob = oracle.Batch(step.cached_seq_len, step.num_new_tokens, w.block_table)
        rows = step.token_rows
        if si in checked:
            sampled = sample_rows(step, per_req, si)
            views.append((ob, q[rows], k[rows], v[rows], kp, vp, sampled[::max(1, len(sampled) // 4)]))
        if si == max(checked):
            break
        kp, vp = oracle.kv_write(ob, k[rows], v[rows], kp, vp, num_heads_kv=sh.num_heads_kv,
                                 head_dim=sh.head_dim, block_size=sh.block_size)
    _views[key] = (sh, views)
    return _views[key]


def gates_on(name, variant, mutation, steps=None):
    """Gate failures of the (mutated) oracle's bf16-rounded result against
    the unmodified oracle."""
    sh, views = step_views(name, variant)
    kw = dict(num_heads_q=sh.num_heads_q, num_heads_kv=sh.num_heads_kv, head_dim=sh.head_dim,
              block_size=sh.block_size, scale=sh.scale)
    res = Result()
    for i, (ob, q, k, v, kp, vp, rows) in enumerate(views):
        if steps is not None and i not in steps:
            continue
        if (name, variant, i) not in _refs:
            _refs[(name, variant, i)] = oracle.attention(ob, q, k, v, kp, vp, rows=rows, **kw)
        ref_o, ref_l = _refs[(name, variant, i)]
        if mutation == oracle.MUT_NONE:
            got_o, got_l = ref_o, ref_l
        else:
            got_o, got_l = oracle.attention(ob, q, k, v, kp, vp, rows=rows, mutation=mutation, **kw)
        res.add(bf16_values(got_o.astype(np.float32)), ref_o, got_l.astype(np.float32), ref_l)
    return gate_failures(res, "bf16")


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("variant", ["plain", "needle"])
def test_correct_result_rounded_to_bf16_passes(name, variant):
    assert gates_on(name, variant, oracle.MUT_NONE) == []


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_planted_mask_mistake_fails_on_the_last_chunk_alone(name, mutation):
    # the last checked chunk sees about 8k (Llama) or 31k (long context)
    # keys; a one-key error there is caught through the needle queries
    _, views = step_views(name, "needle")
    assert gates_on(name, "needle", MUTATIONS[mutation], steps=[len(views) - 1]) != []
