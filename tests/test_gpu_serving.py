"""Multi-step serving on the GPU: the library's engine plans each step, the
attention call runs it over the paged cache (K/V write fused), and every
output row is compared with dense causal attention over its request's own
token sequence computed by the fp64 oracle ("Prefill Optimisation", section 2:
chunked prefill equals one-shot causal attention; section 3: a reused prefix
block holds exactly the K/V the request would have computed).

The stand-in model gives every (token id, position) fixed q / k / v rows
(a token table plus a position table), so identical prefixes have identical
K/V and a prefix-cache hit is exact.  The engine's plan is checked against the
harness oracle's plan step by step; sampled tokens come from a seeded
generator, independent of the outputs.  Also: one attention call captured in
a CUDA graph and replayed gives the eager call's result."""
import numpy as np
import pytest
import torch

import oracle
from oracle import harness as H

from helpers import BF16_ATOL, BF16_LSE_ATOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cpa():
    import chunked_prefill_paged_gb300 as m
    m.load()
    return m


class Model:
    def __init__(self, vocab, max_pos, hq, hkv, d, seed):
        g = torch.Generator().manual_seed(seed)
        mk = lambda *s: torch.randn(*s, generator=g) * 0.7
        self.tq, self.pq = mk(vocab, hq, d), mk(max_pos, hq, d)
        self.tk, self.pk = mk(vocab, hkv, d), mk(max_pos, hkv, d)
        self.tv, self.pv = mk(vocab, hkv, d), mk(max_pos, hkv, d)

    def rows(self, tokens, positions):
        t = torch.as_tensor(np.asarray(tokens, dtype=np.int64))
        p = torch.as_tensor(np.asarray(positions, dtype=np.int64))
        bf = lambda x: x.to(torch.bfloat16)
        return bf(self.tq[t] + self.pq[p]), bf(self.tk[t] + self.pk[p]), bf(self.tv[t] + self.pv[p])


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def dense_reference(model, seq, rows, hq, hkv, d):
    """fp64 causal attention over the whole sequence; outputs of `rows`."""
    L = len(seq)
    q, k, v = model.rows(seq, range(L))
    ob = oracle.Batch([0], [L], np.zeros((1, 1), np.int32))
    pool = np.zeros((1, 1, hkv, d), np.uint16)
    return oracle.attention(ob, bits(q), bits(k), bits(v), pool, pool, num_heads_q=hq, num_heads_kv=hkv,
                            head_dim=d, block_size=1, scale=1.0 / np.sqrt(d), rows=rows, threads=4)


def test_serving_steps_match_dense_attention(cpa):
    from chunked_prefill_paged_gb300.serving import Server
    hq, hkv, d, bs = 8, 2, 128, 16
    vocab, max_pos = 40, 512
    model = Model(vocab, max_pos, hq, hkv, d, seed=81)
    num_blocks, cols, budget, chunk = 256, 32, 192, 64
    eng = cpa.Engine(num_blocks, bs, cols, budget, chunk, scope_key=5)
    ora = H.Engine(num_blocks, bs, cols, budget, chunk, scope=5)
    params = cpa.Params(hq, hkv, d, bs, num_blocks, 512, 1.0 / np.sqrt(d), cpa.DTYPE_BF16, cpa.FLAG_FUSE_KV_WRITE)
    k_cache = torch.full((num_blocks, bs, hkv, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    v_cache = torch.full_like(k_cache, float("nan"))
    server = Server(eng, params, k_cache, v_cache, max_reqs=64)
    rng = np.random.default_rng(82)
    systems = [list(rng.integers(0, vocab, size=n)) for n in (48, 80)]
    arrivals = []
    for rid in range(14):
        prompt = systems[rid % 2] + list(rng.integers(0, vocab, size=int(rng.integers(5, 120))))
        arrivals.append((int(rng.integers(0, 12)), rid, prompt, int(rng.integers(2, 8))))
    arrivals.sort()
    seqs = {}
    first_cached = {}   # cached tokens of each request's first step (a prefix-cache hit when > 0)
    ai = 0
    worst = worst_lse = 0.0
    for t in range(120):
        while ai < len(arrivals) and arrivals[ai][0] <= t:
            _, rid, prompt, mx = arrivals[ai]
            eng.add_request(rid, prompt, mx)
            ora.add_request(rid, prompt, mx)
            seqs[rid] = list(prompt)
            ai += 1
        so = ora.schedule()
        draws = [int(x) for x in rng.integers(0, vocab, size=len(so.rids))]

        def make_qkv(plan):
            pos = np.concatenate([np.arange(c, c + n) for c, n in zip(plan.cached_seq_len, plan.num_new_tokens)])
            q, k, v = model.rows(plan.token_ids, pos)
            return q.cuda(), k.cuda(), v.cuda()

        plan, out, lse = server.step(make_qkv, lambda plan, out: draws)
        assert plan.request_ids.tolist() == so.rids and plan.cached_seq_len.tolist() == so.cached_seq_len
        assert plan.num_new_tokens.tolist() == so.num_new_tokens
        assert plan.block_table.tolist() == [list(r) for r in so.block_table]
        ora.commit(dict(zip(so.rids, draws)))
        if out is None:
            if ai == len(arrivals) and eng.num_unfinished() == 0:
                break
            continue
        torch.cuda.synchronize()
        out_h, lse_h = out.float().cpu().numpy(), lse.cpu().numpy()
        o = 0
        for rid, c, n in zip(plan.request_ids.tolist(), plan.cached_seq_len.tolist(), plan.num_new_tokens.tolist()):
            seq = seqs[rid][:c + n]
            first_cached.setdefault(rid, c)
            ref_o, ref_l = dense_reference(model, seq, list(range(c, c + n)), hq, hkv, d)
            worst = max(worst, float(np.abs(out_h[o:o + n] - ref_o).max()))
            worst_lse = max(worst_lse, float(np.abs(lse_h[o:o + n] - ref_l).max()))
            o += n
        for rid in plan.request_ids.tolist():   # prompt plus the outputs drawn so far
            seqs[rid] = list(ora._req(rid).tokens)
    assert cpa.last_device_error() == cpa.SUCCESS
    assert ai == len(arrivals) and eng.num_unfinished() == 0
    assert worst <= BF16_ATOL, worst
    assert worst_lse <= BF16_LSE_ATOL, worst_lse
    assert sum(1 for c in first_cached.values() if c > 0) >= 4  # requests that started on cached prefix blocks


def test_attention_call_replays_in_a_cuda_graph(cpa):
    import workloads as W
    w = W.make_batch_workload("graph", W.Shape(16, 4, 128, 16, 512, "bf16"),
                              [(0, 200), (700, 1), (3000, 1), (64, 77)], seed=83)
    t = w.materialize("cuda", sentinel=W.SENTINEL_ZERO)
    s = w.steps[0]
    sh = w.shape
    p = cpa.Params(sh.num_heads_q, sh.num_heads_kv, sh.head_dim, sh.block_size, w.num_blocks, sh.kv_segment_size,
                   sh.scale, cpa.DTYPE_BF16, 0)  # no fused write: replays read the same pool
    b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    q, k, v = t.step_inputs(s)
    eager, eager_lse = cpa.attention(b, p, q, k, v, t.k_cache, t.v_cache)
    out = torch.empty_like(eager)
    lse = torch.empty_like(eager_lse)
    n = cpa.workspace_size(b, p)
    ws = torch.empty(max(n // 4, 4), dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        cpa.chunked_prefill_attention(b, p, q, k, v, t.k_cache, t.v_cache, out, lse, ws)  # warm-up
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cpa.chunked_prefill_attention(b, p, q, k, v, t.k_cache, t.v_cache, out, lse, ws,
                                      torch.cuda.current_stream())
    out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert cpa.last_device_error() == cpa.SUCCESS
    assert torch.allclose(out.float(), eager.float(), atol=1e-2, rtol=0)
    assert torch.allclose(lse, eager_lse, atol=1e-3, rtol=0)
