"""Pins for the harness oracle (block allocation, prefix hash chain, greedy
token budget) against what the pages print and the definitions they give.

* FNV-1a 64: the published test vectors of the FNV hash.
* "Prefill Processing", Block Allocation: a 10,240-token request whose first
  4,096 tokens are cached (block size 128) holds 48 blocks after its first
  2,048-token step (32 claimed from the prefix cache, 16 fresh) and 64 after
  the second; its block-table row has 48 ids, then the null block 0 in every
  other of the cdiv(10240, 128) = 80 columns.
* "Prefill Optimisation", section 2: with a budget of 512 and four running
  decodes a 2,048-token prompt goes in chunks 508, 508, 508, 508, 16 with
  cached positions 508, 1016, 1524, 2032, 2048.
* "Prefill Processing", Key Concepts: the 10,000-token prompt under a 2,048
  budget takes iterations of 2048 x 4 and 1808.
* "Prefill Optimisation", section 3: changing one early token changes every
  later block hash (no reuse); identical prefixes reuse their full blocks
  only.
* "Chunked Prefill": decodes first, then chunks capped at 512.
Each planted mistake in a copy of the engine (decodes after prefills, no
leftover prompt token, a hash without the parent) fails one of these.
"""
import numpy as np
import pytest

from oracle import harness as H


def test_fnv1a64_published_vectors():
    assert H.fnv1a64(b"") == 0xCBF29CE484222325
    assert H.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert H.fnv1a64(b"foobar") == 0x85944171F73967E8


def run_until_done(e, sampled=7, max_steps=1000):
    steps = []
    for _ in range(max_steps):
        s = e.schedule()
        if not s.rids:
            break
        steps.append(s)
        e.commit({rid: sampled for rid in s.rids})
    return steps


def test_block_allocation_example_of_the_pages():
    bs = 128
    e = H.Engine(num_blocks=200, block_size=bs, max_blocks_per_seq=80, budget=2048, chunk=2048)
    prefix = list(range(1000, 1000 + 4096))
    e.add_request(0, prefix + [1], max_new_tokens=1)  # computes and caches the 4096-token prefix
    run_until_done(e)
    e.add_request(1, prefix + list(range(5000, 5000 + 10240 - 4096)), max_new_tokens=1)
    s1 = e.schedule()
    assert s1.rids == [1] and s1.cached_seq_len == [4096] and s1.num_new_tokens == [2048]
    row = s1.block_table[0]
    assert len(row) == 80
    assert all(b > 0 for b in row[:48]) and row[48:] == [0] * 32      # 48 blocks, then null ids
    assert len(set(row[:48])) == 48
    e.commit({1: 0})
    s2 = e.schedule()
    assert s2.cached_seq_len == [6144] and s2.num_new_tokens == [2048]
    assert sum(1 for b in s2.block_table[0] if b) == 64
    assert s2.block_table[0][:48] == row[:48]                          # blocks are kept, only appended


def _budget_trace(engine_cls=H.Engine):
    e = engine_cls(num_blocks=400, block_size=16, max_blocks_per_seq=200, budget=512, chunk=512)
    for rid in range(4):
        e.add_request(rid, [rid] * 4, max_new_tokens=100)
    s = e.schedule()
    e.commit({rid: 1 for rid in s.rids})                               # the four now decode
    e.add_request(9, list(range(2048)), max_new_tokens=1)
    trace = []
    for _ in range(5):
        s = e.schedule()
        dec = sum(1 for n in s.num_new_tokens if n == 1 and s.rids[s.num_new_tokens.index(n)] != 9)
        pf = [n for rid, n in zip(s.rids, s.num_new_tokens) if rid == 9]
        e.commit({rid: 1 for rid in s.rids})
        trace.append((dec, pf[0] if pf else 0, e._req(9).num_computed))
    return trace


def test_budget_trace_of_the_pages():
    assert _budget_trace() == [(4, 508, 508), (4, 508, 1016), (4, 508, 1524), (4, 508, 2032), (4, 16, 2048)]


def test_ten_thousand_token_prompt_iterations():
    e = H.Engine(num_blocks=100, block_size=128, max_blocks_per_seq=80, budget=2048, chunk=2048)
    e.add_request(0, list(range(10000)), max_new_tokens=1)
    steps = run_until_done(e)
    assert [s.num_new_tokens[0] for s in steps] == [2048, 2048, 2048, 2048, 1808]
    assert [s.cached_seq_len[0] for s in steps] == [0, 2048, 4096, 6144, 8192]


def test_decodes_first_then_capped_chunks():
    e = H.Engine(num_blocks=4000, block_size=16, max_blocks_per_seq=400, budget=2048, chunk=512)
    for rid in range(64):
        e.add_request(rid, [rid], max_new_tokens=50)
    s = e.schedule()
    e.commit({r: 1 for r in s.rids})
    for rid in range(100, 104):
        e.add_request(rid, list(range(rid, rid + 3000)), max_new_tokens=1)
    s = e.schedule()
    assert s.num_new_tokens[:64] == [1] * 64 and s.rids[:64] == list(range(64))
    assert s.num_new_tokens[64:] == [512, 512, 512, 448]


def _prefix_case(second, bs=16):
    e = H.Engine(num_blocks=100, block_size=bs, max_blocks_per_seq=20, budget=4096, chunk=4096)
    first = list(range(100, 164))           # 64 tokens = 4 full blocks
    e.add_request(0, first, max_new_tokens=1)
    run_until_done(e)
    e.add_request(1, second, max_new_tokens=1)
    s = e.schedule()
    if not s.rids:
        return None, None           # nothing left to compute: the request never runs
    return s.cached_seq_len[0], s.block_table[0]


def test_prefix_hash_chain_reuse_and_invalidation():
    first = list(range(100, 164))
    c, row = _prefix_case(first[:48] + [7, 8, 9, 10])        # 3 shared full blocks
    assert c == 48
    c, _ = _prefix_case(first[:40] + [7] * 20)               # 2.5 shared blocks: full blocks only
    assert c == 32
    changed = list(first)
    changed[5] = -1                                          # one early token differs
    c, _ = _prefix_case(changed)
    assert c == 0
    c, _ = _prefix_case(list(first))                         # whole prompt cached: leave one token
    assert c == 48


def test_freed_blocks_return_and_cached_ones_survive():
    e = H.Engine(num_blocks=9, block_size=4, max_blocks_per_seq=8, budget=64, chunk=64)
    e.add_request(0, list(range(16)), max_new_tokens=1)      # 4 blocks
    run_until_done(e)
    assert e.num_free_blocks() == 8                          # all returned (block 0 is never handed out)
    e.add_request(1, list(range(16)) + [99], max_new_tokens=1)
    s = e.schedule()
    assert s.cached_seq_len == [16]                          # the cached blocks were still there
    e.add_request(2, [5] * 40, max_new_tokens=1)             # needs 10 blocks: more than the pool
    s2 = e.schedule()
    assert 2 not in s2.rids                                  # skipped, no preemption


# ------------------------------------------------------------ planted mistakes

class DecodesLast(H.Engine):
    def schedule(self):
        # prefills claim the budget before decodes
        active = [r for r in self.reqs if not r.finished]
        self.reqs = [r for r in active if not (r.started and r.num_computed >= r.prompt_len)] + \
                    [r for r in active if r.started and r.num_computed >= r.prompt_len] + \
                    [r for r in self.reqs if r.finished]
        order = {id(r): i for i, r in enumerate(self.reqs)}
        rids, cached, new, used = [], [], [], 0
        for r in sorted((r for r in self.reqs if not r.finished), key=lambda r: order[id(r)]):
            if used >= self.budget:
                break
            if not r.started:
                self._prefix_hit(r)
                r.started = True
            n = 1 if r.num_computed >= r.prompt_len else min(self.chunk, self.budget - used,
                                                             r.prompt_len - r.num_computed)
            if n <= 0 or not self._allocate_slots(r, n):
                continue
            rids.append(r.rid)
            cached.append(r.num_computed)
            new.append(n)
            used += n
        table = [self._req(i).blocks + [0] * (self.max_blocks - len(self._req(i).blocks)) for i in rids]
        self.last = H.Step(rids, cached, new, table)
        return self.last


def test_planted_decodes_last_is_caught():
    assert _budget_trace(DecodesLast) != _budget_trace()


def _same_content_elsewhere():
    # the first request holds blocks [P][P][R][S]; the second starts [P][R]: its
    # second block has the content of the first request's third block at
    # another position (after another prefix), so only its first block may be
    # reused
    P, R, S = [11] * 16, list(range(16)), list(range(50, 66))
    e = H.Engine(num_blocks=100, block_size=16, max_blocks_per_seq=20, budget=4096, chunk=4096)
    e.add_request(0, P + P + R + S, max_new_tokens=1)
    run_until_done(e)
    e.add_request(1, P + R + S, max_new_tokens=1)
    return e.schedule().cached_seq_len[0]


def test_parent_hash_keeps_content_at_other_positions_apart():
    assert _same_content_elsewhere() == 16


def test_planted_hash_without_parent_is_caught(monkeypatch):
    monkeypatch.setattr(H, "block_hash", lambda parent, scope, tokens: H.fnv1a64(
        b"".join(int(t).to_bytes(4, "little", signed=True) for t in tokens)))
    assert _same_content_elsewhere() != 16


def test_planted_full_prompt_reuse_is_caught(monkeypatch):
    def hit_all(self, r):
        parent = 0
        for i in range(r.prompt_len // self.bs):
            h = H.block_hash(parent, self.scope, r.tokens[i * self.bs:(i + 1) * self.bs])
            b = self.cache.get(h)
            if b is None:
                break
            self._claim_cached(b)
            r.blocks.append(b)
            r.hashes.append(h)
            parent = h
        r.num_computed = len(r.blocks) * self.bs
    monkeypatch.setattr(H.Engine, "_prefix_hit", hit_all)
    c, _ = _prefix_case(list(range(100, 164)))
    assert c != 48
