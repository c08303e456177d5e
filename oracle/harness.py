"""Plain-Python oracle of the multi-step host harness -- test infrastructure.

Only the tests (and the bench's CPU leg) may import this module; the library's
own harness (the C++ engine behind include/cpa_engine.h) shares no code with
it.  It restates, step by step and in the pages' terms, what one serving
iteration decides before the attention call:

* Greedy token budget ("Chunked Prefill"; "Prefill Optimisation", section 2,
  Mechanics of chunked scheduling): every running decode claims one token of
  the per-step budget first; the rest goes to prompt chunks in arrival order,
  each at most `chunk` tokens.
* Incremental block allocation ("Prefill Processing", Block Allocation): a
  request holds cdiv(num_computed + num_new, block_size) blocks after
  allocate_slots; cached prefix blocks are claimed first, then fresh ones.
  Block 0 is the null block: unallocated block-table columns hold 0.
* Prefix hash chain ("Prefill Optimisation", section 3, vLLM block hash
  chain): the hash of a full block covers its parent's hash, its ordered token
  ids and the cache scope; a new request reuses its prompt's leading full
  blocks while their hashes are cached (full-block-only policy), leaving at
  least one prompt token to compute (the last token's logits are needed).

Where the pages leave a choice open, the readings taken (the C++ engine
follows the same ones):

* block hash = 64-bit FNV-1a over the little-endian bytes of (parent hash,
  scope key, the block's token ids as int32), parent of the first block 0;
* free blocks form a queue: allocation takes the front; a finished request's
  blocks whose count drops to 0 go to the back, last block first (so the
  most recently used prefix blocks are the last to be reused); a block taken
  from the queue for new data loses its cached hash; a cached free block
  claimed by a prefix hit leaves the queue;
* a request that cannot get its blocks this step is skipped (no preemption);
* after the step a request's completed full blocks are hashed and entered
  into the cache unless the hash is already there; a request whose prompt is
  complete appends one output token per step (the caller's), and finishes
  when it has max_new_tokens outputs, freeing its blocks.
"""
from __future__ import annotations

import collections
import dataclasses
from typing import Dict, List, Optional, Sequence, Tuple

FNV_OFFSET = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3
MASK64 = (1 << 64) - 1


def fnv1a64(data: bytes, h: int = FNV_OFFSET) -> int:
    """FNV-1a, 64 bits: for each byte, xor then multiply by the FNV prime."""
    for b in data:
        h ^= b
        h = (h * FNV_PRIME) & MASK64
    return h


def block_hash(parent: int, scope: int, tokens: Sequence[int]) -> int:
    data = parent.to_bytes(8, "little") + scope.to_bytes(8, "little")
    data += b"".join(int(t).to_bytes(4, "little", signed=True) for t in tokens)
    return fnv1a64(data)


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


@dataclasses.dataclass
class Request:
    rid: int
    tokens: List[int]          # prompt, then outputs
    prompt_len: int
    max_new_tokens: int
    num_computed: int = 0      # tokens whose K/V is in the cache
    blocks: List[int] = dataclasses.field(default_factory=list)
    hashes: List[int] = dataclasses.field(default_factory=list)  # of the full blocks computed so far
    started: bool = False
    finished: bool = False

    @property
    def outputs(self) -> int:
        return len(self.tokens) - self.prompt_len


@dataclasses.dataclass
class Step:
    rids: List[int]
    cached_seq_len: List[int]
    num_new_tokens: List[int]
    block_table: List[List[int]]   # [num_reqs][max_blocks_per_seq], 0 past the allocated blocks


class Engine:
    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int, budget: int, chunk: int,
                 scope: int = 0):
        self.bs = block_size
        self.max_blocks = max_blocks_per_seq
        self.budget = budget
        self.chunk = chunk
        self.scope = scope
        self.free = collections.deque(range(1, num_blocks))   # block 0 is the null block
        self.ref = [0] * num_blocks
        self.block_hash: Dict[int, int] = {}                  # block -> hash of its cached content
        self.cache: Dict[int, int] = {}                       # hash -> block
        self.reqs: List[Request] = []
        self.last: Optional[Step] = None

    # ---------------------------------------------------------------- blocks
    def _take_free(self) -> int:
        b = self.free.popleft()
        h = self.block_hash.pop(b, None)
        if h is not None and self.cache.get(h) == b:
            del self.cache[h]
        self.ref[b] = 1
        return b

    def _claim_cached(self, b: int) -> None:
        if self.ref[b] == 0:
            self.free.remove(b)
        self.ref[b] += 1

    def _allocate_slots(self, r: Request, num_new: int) -> bool:
        need = cdiv(r.num_computed + num_new, self.bs)
        if need > self.max_blocks:
            return False
        extra = need - len(r.blocks)
        if extra > len(self.free):
            return False
        for _ in range(extra):
            r.blocks.append(self._take_free())
        return True

    def _prefix_hit(self, r: Request) -> None:
        """Claim the leading full prompt blocks whose hashes are cached."""
        parent = 0
        limit = (r.prompt_len - 1) // self.bs   # leave at least one prompt token to compute
        for i in range(limit):
            h = block_hash(parent, self.scope, r.tokens[i * self.bs:(i + 1) * self.bs])
            b = self.cache.get(h)
            if b is None:
                break
            self._claim_cached(b)
            r.blocks.append(b)
            r.hashes.append(h)
            parent = h
        r.num_computed = len(r.blocks) * self.bs

    # ------------------------------------------------------------- interface
    def add_request(self, rid: int, prompt: Sequence[int], max_new_tokens: int) -> None:
        self.reqs.append(Request(rid, list(prompt), len(prompt), max_new_tokens))

    def schedule(self) -> Step:
        rids, cached, new = [], [], []
        used = 0
        active = [r for r in self.reqs if not r.finished]
        for r in active:          # decodes first, one token each
            if r.started and r.num_computed >= r.prompt_len:
                if used >= self.budget:
                    break
                if not self._allocate_slots(r, 1):
                    continue
                rids.append(r.rid)
                cached.append(r.num_computed)
                new.append(1)
                used += 1
        for r in active:          # then prompt chunks in arrival order
            if r.started and r.num_computed >= r.prompt_len:
                continue
            if used >= self.budget:
                break
            if not r.started:
                self._prefix_hit(r)
                r.started = True
            take = min(self.chunk, self.budget - used, r.prompt_len - r.num_computed)
            if take <= 0 or not self._allocate_slots(r, take):
                continue
            rids.append(r.rid)
            cached.append(r.num_computed)
            new.append(take)
            used += take
        table = []
        for rid in rids:
            r = self._req(rid)
            table.append(r.blocks + [0] * (self.max_blocks - len(r.blocks)))
        self.last = Step(rids, cached, new, table)
        return self.last

    def commit(self, sampled: Dict[int, int]) -> None:
        """After the step: advance the computed counts, cache completed full
        blocks, append one output token (sampled[rid]) to every request whose
        prompt is complete, retire finished requests."""
        step = self.last
        for rid, n in zip(step.rids, step.num_new_tokens):
            r = self._req(rid)
            r.num_computed += n
            while len(r.hashes) < r.num_computed // self.bs:
                i = len(r.hashes)
                parent = r.hashes[-1] if r.hashes else 0
                h = block_hash(parent, self.scope, r.tokens[i * self.bs:(i + 1) * self.bs])
                r.hashes.append(h)
                b = r.blocks[i]
                if h not in self.cache:
                    self.cache[h] = b
                    self.block_hash[b] = h
            if r.num_computed >= r.prompt_len:
                r.tokens.append(int(sampled[rid]))
                if r.outputs >= r.max_new_tokens:
                    self._finish(r)

    def _finish(self, r: Request) -> None:
        r.finished = True
        for b in reversed(r.blocks):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)
        r.blocks = []

    def _req(self, rid: int) -> Request:
        for r in self.reqs:
            if r.rid == rid:
                return r
        raise KeyError(rid)

    def num_free_blocks(self) -> int:
        return len(self.free)
