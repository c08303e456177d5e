"""Seeded synthetic workloads for paged chunked-prefill attention.

This module is shared by the tests, the bench and the smoke check.  It holds
the input recipe only -- request lengths, block tables, pool contents and
Q/K/V values -- plus the host-side schedules and work counters the pages
print.  It holds none of the attention arithmetic and none of the KV-write
arithmetic: the oracle and the CUDA library each implement those on their
own.

Recipe (every value seeded):
  * Q, K, V: i.i.d. N(0, 1) drawn in float32 and rounded to bfloat16 (RNE)
    when the workload is bfloat16.
  * Physical block ids: a seeded permutation of the pool, so a request's
    blocks are scattered ("vLLM Chunked Prefill ..." section 3.2 on
    fragmentation across chunks).
  * Block-table columns past a request's allocated blocks hold seeded
    random ids ("Prefill Processing", Block Allocation: unallocated columns
    carry no meaning for the kernel).
  * Pool slots that hold no cached token are filled with a sentinel (NaN for
    parity runs, zero for timing runs) so that a stray read shows.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

SENTINEL_NAN = "nan"
SENTINEL_ZERO = "zero"


# ---------------------------------------------------------------------------
# Schedules and counters printed by the pages (host-side policy, no attention
# arithmetic)
# ---------------------------------------------------------------------------

def cdiv(a: int, b: int) -> int:
    return -(-a // b)


def chunk_schedule(total_prompt_tokens: int, active_decodes: int, max_batched_tokens: int) -> List[int]:
    """Prompt chunk sizes when decodes claim the budget first and the rest
    goes to the prompt ("Prefill Optimisation", section 2, Mechanics of
    chunked scheduling; section 7 ChunkedScheduler).  Raises when no prefill
    budget is left."""
    if max_batched_tokens <= 0:
        raise ValueError("max_batched_tokens must be positive")
    if total_prompt_tokens < 0 or active_decodes < 0:
        raise ValueError("token counts must be non-negative")
    avail = max_batched_tokens - active_decodes
    if avail <= 0:
        raise RuntimeError("no prefill progress possible: decodes fill the token budget")
    chunks = []
    left = total_prompt_tokens
    while left > 0:
        c = min(left, avail)
        chunks.append(c)
        left -= c
    return chunks


def greedy_step(decodes: Sequence[int], prefills: Sequence[Tuple[int, int]], budget: int,
                chunk: int) -> List[Tuple[str, int, int]]:
    """One step of the greedy decode-first scheduler with a per-request chunk
    cap ("Chunked Prefill" blog note, From scratch).  decodes: context length
    of each decoding sequence; prefills: (tokens done, prompt length).
    Returns (kind, cached_seq_len, num_new_tokens) per scheduled request."""
    batch = [("decode", int(c), 1) for c in decodes]
    used = len(decodes)
    for done, total in prefills:
        if used >= budget:
            break
        take = min(chunk, budget - used, total - done)
        if take <= 0:
            continue
        batch.append(("prefill", int(done), int(take)))
        used += take
    return batch


def pairs(cached_seq_len: int, num_new_tokens: int) -> int:
    """Visible (query, key) pairs of one request: each new token sees the
    whole cache and, causally, its own chunk ("Prefill Optimisation",
    section 4, Suffix-to-prefix pairs)."""
    C, N = int(cached_seq_len), int(num_new_tokens)
    return N * C + N * (N + 1) // 2


def attention_flops(pairs_total: int, num_heads_q: int, head_dim: int, layers: int = 1) -> int:
    """4 * L * H_Q * pairs * d_head ("Prefill Optimisation", section 4)."""
    return 4 * layers * num_heads_q * int(pairs_total) * head_dim


def algorithmic_bytes(cached: Sequence[int], new: Sequence[int], num_heads_q: int, num_heads_kv: int,
                      head_dim: int, elem_bytes: int, kv_elem_bytes: Optional[int] = None) -> int:
    """Bytes the method must move once: cached K and V read once per kv head,
    Q / K_new / V_new read, new K/V written into the pool, output written
    ("Prefill Optimisation", section 6, per-token KV bytes).  kv_elem_bytes:
    bytes per pool element (1 for the FP8 cache; default elem_bytes)."""
    T = int(sum(int(n) for n in new))
    kv_row = 2 * num_heads_kv * head_dim * (elem_bytes if kv_elem_bytes is None else kv_elem_bytes)
    cached_bytes = sum(int(c) for c in cached) * kv_row
    io = T * (num_heads_q + 2 * num_heads_kv) * head_dim * elem_bytes
    write = T * kv_row
    out = T * num_heads_q * head_dim * elem_bytes
    return cached_bytes + io + write + out


# ---------------------------------------------------------------------------
# Workload description
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class Shape:
    num_heads_q: int
    num_heads_kv: int
    head_dim: int
    block_size: int
    kv_segment_size: int
    dtype: str  # "f32" or "bf16"

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2


@dataclasses.dataclass
class Step:
    cached_seq_len: np.ndarray   # int32 [num_reqs]
    num_new_tokens: np.ndarray   # int32 [num_reqs]
    token_rows: np.ndarray       # int64 [T]: rows of the value tensors this step's tokens use

    @property
    def total_new_tokens(self) -> int:
        return int(self.num_new_tokens.sum())

    @property
    def cu_new_tokens(self) -> np.ndarray:
        cu = np.zeros(len(self.num_new_tokens) + 1, dtype=np.int32)
        np.cumsum(self.num_new_tokens, out=cu[1:])
        return cu


@dataclasses.dataclass
class Workload:
    name: str
    shape: Shape
    num_blocks: int
    block_table: np.ndarray      # int32 [num_reqs, max_blocks_per_seq]
    steps: List[Step]
    num_value_rows: int          # rows of the Q/K/V value tensors
    cached_blocks: List[List[int]]  # per request: physical blocks whose slots hold cached KV
    cached_valid: List[int]      # per request: number of cached tokens present before step 0
    seed: int
    description: str = ""

    @property
    def num_reqs(self) -> int:
        return int(self.block_table.shape[0])

    def pairs_per_step(self) -> List[int]:
        return [sum(pairs(c, n) for c, n in zip(s.cached_seq_len, s.num_new_tokens)) for s in self.steps]

    def flops_per_step(self) -> List[int]:
        sh = self.shape
        return [attention_flops(p, sh.num_heads_q, sh.head_dim) for p in self.pairs_per_step()]

    def bytes_per_step(self, kv_elem_bytes: Optional[int] = None) -> List[int]:
        sh = self.shape
        return [algorithmic_bytes(s.cached_seq_len, s.num_new_tokens, sh.num_heads_q, sh.num_heads_kv,
                                  sh.head_dim, sh.elem_bytes, kv_elem_bytes) for s in self.steps]

    def materialize(self, device="cpu", sentinel: str = SENTINEL_NAN) -> "Tensors":
        return _materialize(self, torch.device(device), sentinel)


@dataclasses.dataclass
class Tensors:
    q: torch.Tensor        # [rows, H_q, d]
    k: torch.Tensor        # [rows, H_kv, d]
    v: torch.Tensor        # [rows, H_kv, d]
    k_cache: torch.Tensor  # [num_blocks, block_size, H_kv, d] before step 0
    v_cache: torch.Tensor

    def step_inputs(self, step: Step):
        idx = torch.as_tensor(step.token_rows, device=self.q.device)
        if len(step.token_rows) and np.all(np.diff(step.token_rows) == 1):
            a = int(step.token_rows[0])
            b = a + len(step.token_rows)
            return self.q[a:b], self.k[a:b], self.v[a:b]
        return self.q[idx].contiguous(), self.k[idx].contiguous(), self.v[idx].contiguous()


VARIANTS = ("plain", "peaky", "needle")


def apply_variant(t: Tensors, variant: str, group: int) -> None:
    """Reshape the query values of materialized inputs, in place, so that a
    parity check cannot pass on a wrong mask.

    plain   N(0, 1) queries as drawn.  Over thousands of keys the softmax is
            nearly flat and outputs are about 0.01-0.05 in size.
    peaky   queries times 4 (a power of two: exact in bf16 and fp32); scores
            then have a standard deviation of about 4, a few keys carry most
            of the weight and outputs are O(1).
    needle  query row t of every query head is the sum of value row t's key
            and value row t + 1's key (of the kv head that serves that query
            head, heads grouped contiguously: kv head h // group), rounded to
            the element type.  In a prompt, value row t + 1 is the next
            position, so a row's own key and the key just past its causal
            limit both score about sqrt(d) above the rest: the output is
            dominated by the row's own value row, and a mask that drops the
            diagonal or lets the next key in changes it by O(1).
    """
    if variant == "plain":
        return
    if variant == "peaky":
        t.q.mul_(4)
        return
    if variant != "needle":
        raise ValueError(f"unknown variant {variant!r}")
    k = t.k.float()
    nxt = torch.zeros_like(k)
    nxt[:-1] = k[1:]
    src = (k + nxt).repeat_interleave(group, dim=1)  # [rows, H_q, d]
    t.q.copy_(src.to(t.q.dtype))


def _gen(device: torch.device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, g, device, dtype) -> torch.Tensor:
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    return x.to(dtype)


def _materialize(w: Workload, device: torch.device, sentinel: str) -> Tensors:
    sh = w.shape
    dt = sh.torch_dtype
    g = _gen(device, w.seed)
    q = _normal((w.num_value_rows, sh.num_heads_q, sh.head_dim), g, device, dt)
    k = _normal((w.num_value_rows, sh.num_heads_kv, sh.head_dim), g, device, dt)
    v = _normal((w.num_value_rows, sh.num_heads_kv, sh.head_dim), g, device, dt)
    pool_shape = (w.num_blocks, sh.block_size, sh.num_heads_kv, sh.head_dim)
    k_cache = torch.empty(pool_shape, dtype=dt, device=device)
    v_cache = torch.empty(pool_shape, dtype=dt, device=device)
    step = 4096
    for b0 in range(0, w.num_blocks, step):
        b1 = min(w.num_blocks, b0 + step)
        k_cache[b0:b1] = _normal((b1 - b0,) + pool_shape[1:], g, device, dt)
        v_cache[b0:b1] = _normal((b1 - b0,) + pool_shape[1:], g, device, dt)
    # Cached KV present before the first step keeps its random values: every
    # slot of a listed block that holds a cached token.  Every other slot
    # (unlisted blocks, the tail of a partly filled block) gets the sentinel.
    fill = float("nan") if sentinel == SENTINEL_NAN else 0.0
    keep = np.zeros(w.num_blocks, dtype=bool)
    tails = []
    for r, blocks in enumerate(w.cached_blocks):
        valid = int(w.cached_valid[r])
        for col, b in enumerate(blocks):
            n_valid = min(sh.block_size, valid - col * sh.block_size)
            if n_valid <= 0:
                continue
            keep[int(b)] = True
            if n_valid < sh.block_size:
                tails.append((int(b), n_valid))
    drop = torch.as_tensor(np.nonzero(~keep)[0], device=device)
    if drop.numel():
        k_cache[drop] = fill
        v_cache[drop] = fill
    for b, n_valid in tails:
        k_cache[b, n_valid:] = fill
        v_cache[b, n_valid:] = fill
    return Tensors(q, k, v, k_cache, v_cache)


# ---------------------------------------------------------------------------
# FP8 cache inputs
# ---------------------------------------------------------------------------

FP8_MAX = 448.0


def fp8_scales(num_heads_kv: int, amax: float = 4.5) -> Tuple[np.ndarray, np.ndarray]:
    """Per-kv-head key and value scales for N(0,1) data: |x| up to about
    `amax` maps onto the E4M3 range, a little differently per head (so that a
    wrong head index shows).  float32 [H_kv] each."""
    g = np.arange(num_heads_kv, dtype=np.float64)
    k = (amax / FP8_MAX) * (1.0 + 0.125 * g)
    v = (amax / FP8_MAX) * (1.0 + 0.0625 * ((g * 5) % num_heads_kv))
    return k.astype(np.float32), v.astype(np.float32)


def fp8_pool_codes(pool: torch.Tensor, scale: np.ndarray, chunk_blocks: int = 2048) -> torch.Tensor:
    """Input generation for FP8 caches: uint8 codes of a pool
    [num_blocks, bs, H_kv, d] (NaN sentinels become NaN codes), from torch's
    own float8_e4m3fn conversion of x / scale clamped to the finite range --
    a library routine, independent of both the library and the oracle; any
    valid code pattern would serve as cached contents."""
    s = torch.as_tensor(np.asarray(scale, dtype=np.float32), device=pool.device)[:, None]
    out = torch.empty(pool.shape, dtype=torch.uint8, device=pool.device)
    for b0 in range(0, pool.shape[0], chunk_blocks):
        b1 = min(pool.shape[0], b0 + chunk_blocks)
        y = (pool[b0:b1].float() / s).clamp(-FP8_MAX, FP8_MAX)
        out[b0:b1] = y.to(torch.float8_e4m3fn).view(torch.uint8)
    return out


def _block_table(rng: np.random.Generator, needs: Sequence[int], num_blocks: int, extra_cols: int,
                 shared: Optional[Sequence[int]] = None, shared_count: int = 0) -> np.ndarray:
    """Rows of physical block ids drawn from a seeded permutation of the pool.
    The first shared_count columns of every row may be one shared list of
    blocks (prefix caching); padding columns get random in-range ids."""
    max_cols = max(needs) + extra_cols if needs else 1
    bt = rng.integers(0, num_blocks, size=(len(needs), max(max_cols, 1)), dtype=np.int64)
    perm = list(rng.permutation(num_blocks))
    if shared is not None:
        shared_set = set(int(b) for b in shared)
        perm = [b for b in perm if int(b) not in shared_set]
    pos = 0
    for r, need in enumerate(needs):
        own = need - (shared_count if shared is not None else 0)
        if shared is not None:
            bt[r, :shared_count] = np.asarray(shared[:shared_count])
            start = shared_count
        else:
            start = 0
        if pos + own > len(perm):
            raise ValueError("pool too small for the requested blocks")
        bt[r, start:start + own] = np.asarray(perm[pos:pos + own], dtype=np.int64)
        pos += own
    return bt.astype(np.int32)


def make_batch_workload(name: str, shape: Shape, reqs: Sequence[Tuple[int, int]], seed: int,
                        num_blocks: Optional[int] = None, spare: float = 0.1, extra_cols: int = 3,
                        description: str = "") -> Workload:
    """One step over independent requests, each (cached_seq_len, num_new_tokens)."""
    rng = np.random.default_rng(seed)
    needs = [cdiv(c + n, shape.block_size) for c, n in reqs]
    total = sum(needs)
    if num_blocks is None:
        num_blocks = max(total + int(math.ceil(total * spare)), 1)
    bt = _block_table(rng, needs, num_blocks, extra_cols)
    cached = np.array([c for c, _ in reqs], dtype=np.int32)
    new = np.array([n for _, n in reqs], dtype=np.int32)
    T = int(new.sum())
    step = Step(cached, new, np.arange(T, dtype=np.int64))
    cached_blocks = [list(bt[r, :cdiv(c, shape.block_size)]) for r, (c, _) in enumerate(reqs)]
    return Workload(name, shape, num_blocks, bt, [step], max(T, 1), cached_blocks,
                    [c for c, _ in reqs], seed, description)


def make_prompt_workload(name: str, shape: Shape, prompt_len: int, chunk: int, num_blocks: int,
                         seed: int, extra_cols: int = 2, description: str = "") -> Workload:
    """One prompt processed in chunks of `chunk` tokens, one request per step;
    the cache starts empty and each step's K/V is written by the step itself
    ("Prefill Processing", Prefill Segmentation)."""
    rng = np.random.default_rng(seed)
    need = cdiv(prompt_len, shape.block_size)
    bt = _block_table(rng, [need], num_blocks, extra_cols)
    steps = []
    done = 0
    while done < prompt_len:
        n = min(chunk, prompt_len - done)
        steps.append(Step(np.array([done], dtype=np.int32), np.array([n], dtype=np.int32),
                          np.arange(done, done + n, dtype=np.int64)))
        done += n
    return Workload(name, shape, num_blocks, bt, steps, prompt_len, [[]], [0], seed, description)


# ---------------------------------------------------------------------------
# The five workloads the measurements are quoted on
# ---------------------------------------------------------------------------

def tiny_fp32(seed: int = 1001) -> Workload:
    """1 request, FP32, H_q 4, H_kv 1, d 64, block 16, 256 cached tokens in 16
    blocks of a 64-block pool, 128 active tokens."""
    sh = Shape(4, 1, 64, 16, 512, "f32")
    return make_batch_workload("tiny_fp32", sh, [(256, 128)], seed, num_blocks=64,
                               description="1 req, C=256, N=128, H 4/1, d 64, bs 16, FP32")


def llama3_8b_prompt(seed: int = 1002) -> Workload:
    """Llama-3-8B-shaped layer: a 10,000-token prompt in 5 chunks of 2048
    (cached 0, 2048, 4096, 6144, 8192), H_q 32, H_kv 8, d 128, block 128,
    kv_segment_size 1024, 128-block pool."""
    sh = Shape(32, 8, 128, 128, 1024, "bf16")
    return make_prompt_workload("llama3_8b_prompt_10k_chunk2048", sh, 10000, 2048, 128, seed,
                                description="10,000-token prompt, 5 chunks of 2048, H 32/8, d 128, bs 128")


def prefix_cache(seed: int = 1003) -> Workload:
    """16 requests sharing one 4096-token cached prefix (the same 256 physical
    blocks), each with a unique suffix of uniform{256..512} active tokens;
    H_q 32, H_kv 8, d 128, block 16, 8192-block pool."""
    sh = Shape(32, 8, 128, 16, 1024, "bf16")
    rng = np.random.default_rng(seed)
    suffix = rng.integers(256, 513, size=16)
    C = 4096
    num_blocks = 8192
    shared = list(rng.permutation(num_blocks)[: C // 16])
    needs = [cdiv(C + int(n), 16) for n in suffix]
    bt = _block_table(rng, needs, num_blocks, 3, shared=shared, shared_count=C // 16)
    cached = np.full(16, C, dtype=np.int32)
    new = suffix.astype(np.int32)
    T = int(new.sum())
    step = Step(cached, new, np.arange(T, dtype=np.int64))
    cached_blocks = [list(bt[r, : C // 16]) for r in range(16)]
    return Workload("prefix_cache_16x4096", sh, num_blocks, bt, [step], T, cached_blocks, [C] * 16,
                    seed, "16 reqs share a 4096-token prefix (256 blocks), suffix U{256..512}, bs 16")


def mixed_step(seed: int = 1004, num_decodes: int = 64, budget: int = 2048, chunk: int = 512) -> Workload:
    """One step under a 2048-token budget: 64 decodes with context
    uniform{1024..32768} claim the budget first, prefill chunks of 512 at
    cached_seq_len uniform over the multiples of 512 in [0, 16384] fill the
    rest (greedy scheduler); H 32/8, d 128, block 16, pool = needed + 10%."""
    sh = Shape(32, 8, 128, 16, 1024, "bf16")
    rng = np.random.default_rng(seed)
    ctx = rng.integers(1024, 32769, size=num_decodes)
    n_prefills = cdiv(budget - num_decodes, chunk)
    starts = rng.integers(0, 16384 // 512 + 1, size=n_prefills) * 512
    prefills = [(int(s), int(s) + 4 * chunk) for s in starts]  # prompts long enough for one chunk
    sched = greedy_step([int(c) for c in ctx], prefills, budget, chunk)
    reqs = [(c, n) for _, c, n in sched]
    w = make_batch_workload("mixed_step_budget2048", sh, reqs, seed, spare=0.1,
                            description="64 decodes C~U{1024..32768} + prefill chunks 512,512,512,448 "
                                        "at C~U{0,512,..,16384}; bs 16")
    return w


def speculative_decode(seed: int = 1006, num_reqs: int = 64, drafts: int = 4) -> Workload:
    """Decodes that verify draft tokens: each request brings 1 + drafts active
    tokens ("Prefill Processing", Attention Metadata: decode_token_threshold =
    1 + max_num_draft_tokens) over a context uniform{1024..32768}; H 32/8,
    d 128, block 16, kv_segment_size 1024, pool = needed + 10%."""
    sh = Shape(32, 8, 128, 16, 1024, "bf16")
    rng = np.random.default_rng(seed)
    ctx = rng.integers(1024, 32769, size=num_reqs)
    reqs = [(int(c), 1 + drafts) for c in ctx]
    return make_batch_workload(f"speculative_decode_{num_reqs}x{1 + drafts}", sh, reqs, seed, spare=0.1,
                               description=f"{num_reqs} requests x {1 + drafts} tokens over C~U{{1024..32768}}; bs 16")


def decode_batch(seed: int = 1007, num_reqs: int = 32, ctx: int = 8192) -> Workload:
    """Plain decodes (one active token each) over equal contexts; H 32/8,
    d 128, block 16, kv_segment_size 1024: a small decode-only case (about
    1 GiB of pool at the defaults) for profiling the split-KV path."""
    sh = Shape(32, 8, 128, 16, 1024, "bf16")
    return make_batch_workload(f"decode_{num_reqs}x{ctx}", sh, [(ctx, 1)] * num_reqs, seed, spare=0.1,
                               description=f"{num_reqs} decodes over {ctx} cached tokens; bs 16")


def long_context(seed: int = 1005) -> Workload:
    """70B-shaped GQA: a 32,768-token prompt in 16 chunks of 2048 (last step
    cached 30,720), H_q 64, H_kv 8, d 128, block 16, kv_segment_size 4096,
    block table over a shuffled 4096-block pool."""
    sh = Shape(64, 8, 128, 16, 4096, "bf16")
    return make_prompt_workload("long_context_32k_chunk2048", sh, 32768, 2048, 4096, seed,
                                description="32,768-token prompt, 16 chunks of 2048, H 64/8, d 128, bs 16")


ALL = {
    "tiny_fp32": tiny_fp32,
    "llama3_8b_prompt": llama3_8b_prompt,
    "prefix_cache": prefix_cache,
    "mixed_step": mixed_step,
    "long_context": long_context,
    "speculative_decode": speculative_decode,
    "decode_batch": decode_batch,
}
