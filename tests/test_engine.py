"""The library's serving harness (C++, include/cpa_engine.h) against the
harness oracle (oracle/harness.py), on the CPU: every step's plan -- request
order, cached and new token counts, block-table rows and the tokens computed
-- must be identical (integer work: bit-exact), and so must the free-block and
unfinished counts, over seeded scenarios with shared prefixes, staggered
arrivals, pools small enough to refuse allocations and reuse cached free
blocks, and budgets/chunks of every kind."""
import numpy as np
import pytest

from oracle import harness as H


@pytest.fixture(scope="module")
def cpa():
    from chunked_prefill_paged_gb300 import build
    build.build()
    import chunked_prefill_paged_gb300 as m
    return m


def oracle_plan(e: H.Engine, step: H.Step):
    toks = []
    for rid, c, n in zip(step.rids, step.cached_seq_len, step.num_new_tokens):
        toks.extend(e._req(rid).tokens[c:c + n])
    return (list(step.rids), list(step.cached_seq_len), list(step.num_new_tokens),
            [list(r) for r in step.block_table], toks)


def lib_plan(p):
    return (p.request_ids.tolist(), p.cached_seq_len.tolist(), p.num_new_tokens.tolist(), p.block_table.tolist(),
            p.token_ids.tolist())


def scenario(seed):
    rng = np.random.default_rng(seed)
    bs = int(rng.choice([4, 16, 32]))
    num_blocks = int(rng.integers(12, 200))
    max_blocks = int(rng.integers(8, 64))
    budget = int(rng.integers(8, 600))
    chunk = int(rng.integers(1, budget + 1))
    scope = int(rng.integers(0, 2 ** 63))
    systems = [list(rng.integers(0, 50, size=int(rng.integers(1, 6)) * bs)) for _ in range(3)]
    arrivals = []
    for rid in range(int(rng.integers(3, 25))):
        prefix = systems[int(rng.integers(0, 3))] if rng.random() < 0.7 else []
        tail = list(rng.integers(0, 50, size=int(rng.integers(1, 3 * bs + 5))))
        arrivals.append((int(rng.integers(0, 30)), rid, prefix + tail, int(rng.integers(1, 12))))
    return dict(num_blocks=num_blocks, block_size=bs, max_blocks_per_seq=max_blocks, budget=budget, chunk=chunk,
                scope=scope), sorted(arrivals)


@pytest.mark.parametrize("seed", range(40))
def test_engine_matches_oracle_step_by_step(cpa, seed):
    cfg, arrivals = scenario(1100 + seed)
    o = H.Engine(cfg["num_blocks"], cfg["block_size"], cfg["max_blocks_per_seq"], cfg["budget"], cfg["chunk"],
                 cfg["scope"])
    g = cpa.Engine(cfg["num_blocks"], cfg["block_size"], cfg["max_blocks_per_seq"], cfg["budget"], cfg["chunk"],
                   cfg["scope"])
    rng = np.random.default_rng(seed)
    ai = 0
    steps = 0
    for t in range(400):
        while ai < len(arrivals) and arrivals[ai][0] <= t:
            _, rid, prompt, mx = arrivals[ai]
            o.add_request(rid, prompt, mx)
            g.add_request(rid, prompt, mx)
            ai += 1
        so = o.schedule()
        sg = g.schedule()
        assert lib_plan(sg) == oracle_plan(o, so), f"step {t}"
        sampled = [int(x) for x in rng.integers(0, 50, size=len(so.rids))]
        o.commit(dict(zip(so.rids, sampled)))
        g.commit(sampled)
        assert g.num_free_blocks() == o.num_free_blocks()
        assert g.num_unfinished() == sum(1 for r in o.reqs if not r.finished)
        steps += bool(so.rids)
        if ai == len(arrivals) and g.num_unfinished() == 0:
            break
    assert steps > 0


def test_pages_examples_through_the_library(cpa):
    # the 10,240-token request over a cached 4,096-token prefix (block 128):
    # 48 blocks after its first step, 64 after the second, null ids past them
    e = cpa.Engine(200, 128, 80, 2048, 2048)
    prefix = list(range(1000, 1000 + 4096))
    e.add_request(0, prefix + [1], 1)
    while True:
        p = e.schedule()
        e.commit([0] * p.num_reqs)              # every plan is committed, an empty one too
        if p.num_reqs == 0:
            break
    e.add_request(1, prefix + list(range(5000, 5000 + 6144)), 1)
    assert e.prefix_hit_tokens(1) == 4096
    p = e.schedule()
    assert p.cached_seq_len.tolist() == [4096] and p.num_new_tokens.tolist() == [2048]
    assert (p.block_table[0, :48] > 0).all() and (p.block_table[0, 48:] == 0).all()
    e.commit([0])
    p = e.schedule()
    assert int((p.block_table[0] > 0).sum()) == 64


def test_bad_arguments(cpa):
    with pytest.raises(cpa.CpaError):
        cpa.Engine(1, 16, 8, 64, 64)            # no block besides the null block
    e = cpa.Engine(10, 16, 8, 64, 64)
    with pytest.raises(cpa.CpaError):
        e.add_request(0, [], 1)
    with pytest.raises(cpa.CpaError):
        e.add_request(0, [1, 2], 0)
    e.add_request(0, [1, 2], 1)
    with pytest.raises(cpa.CpaError):
        e.add_request(0, [1, 2], 1)             # id already known
    with pytest.raises(cpa.CpaError):
        e.commit([])                            # nothing scheduled yet
    e.schedule()
    with pytest.raises(cpa.CpaError):
        e.schedule()                            # the previous step is not committed
