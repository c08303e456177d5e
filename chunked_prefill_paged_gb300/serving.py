"""A serving loop over the library: the engine's plan for a step, its batch
moved to the device in one copy, the attention call, the commit.

The model around attention is the caller's: `make_qkv(plan)` returns the
step's q, k_new, v_new on the device ([T, H, d] packed like the plan's
tokens) and `sample(plan, out)` returns one token per plan row."""
from __future__ import annotations

from typing import Callable, Optional, Tuple

import numpy as np
import torch

from .binding import Batch, Engine, Params, StepPlan, attention


class StepBuffers:
    """Pinned host staging and device arrays for a step's batch descriptor,
    reused across steps (two sets, so that packing step k + 1 never waits
    for the copy of step k).  One host-to-device copy per step carries
    cached_seq_len, num_new_tokens, cu_new_tokens and the block table."""

    def __init__(self, max_reqs: int, max_blocks_per_seq: int, device="cuda"):
        self.max_reqs = max_reqs
        self.cols = max_blocks_per_seq
        n = 3 * max_reqs + 1 + max_reqs * max_blocks_per_seq
        self.host = [torch.empty(n, dtype=torch.int32).pin_memory() for _ in range(2)]
        self.dev = [torch.empty(n, dtype=torch.int32, device=device) for _ in range(2)]
        self.done = [None, None]
        self.k = 0

    def batch(self, plan: StepPlan, stream: Optional[torch.cuda.Stream] = None) -> Batch:
        nr = plan.num_reqs
        if nr > self.max_reqs or plan.block_table.shape[1] != self.cols:
            raise ValueError("plan larger than the step buffers")
        i = self.k
        self.k ^= 1
        if self.done[i] is not None:
            self.done[i].synchronize()      # its previous copy has been read
        h = self.host[i].numpy()
        cu = np.zeros(nr + 1, dtype=np.int32)
        np.cumsum(plan.num_new_tokens, out=cu[1:])
        o = 0
        for part in (plan.cached_seq_len, plan.num_new_tokens, cu, plan.block_table.reshape(-1)):
            h[o:o + part.size] = part
            o += part.size
        stream = stream or torch.cuda.current_stream()
        with torch.cuda.stream(stream):
            self.dev[i][:o].copy_(self.host[i][:o], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(stream)
        self.done[i] = ev
        d = self.dev[i]
        return Batch.from_device(plan.cached_seq_len, plan.num_new_tokens, plan.block_table, d[0:nr], d[nr:2 * nr],
                                 d[2 * nr:3 * nr + 1], d[3 * nr + 1:3 * nr + 1 + nr * self.cols])


class Server:
    """Drives the engine and the attention call step by step."""

    def __init__(self, engine: Engine, params: Params, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 max_reqs: int, device="cuda"):
        self.engine = engine
        self.params = params
        self.k_cache = k_cache
        self.v_cache = v_cache
        self.buffers = StepBuffers(max_reqs, engine.max_blocks_per_seq, device)

    def step(self, make_qkv: Callable[[StepPlan], Tuple[torch.Tensor, torch.Tensor, torch.Tensor]],
             sample: Callable[[StepPlan, torch.Tensor], np.ndarray]):
        """One iteration; returns (plan, out, lse), out / lse None when
        nothing could run."""
        plan = self.engine.schedule()
        if plan.num_reqs == 0:
            self.engine.commit([])
            return plan, None, None
        batch = self.buffers.batch(plan)
        q, k, v = make_qkv(plan)
        out, lse = attention(batch, self.params, q, k, v, self.k_cache, self.v_cache)
        self.engine.commit(sample(plan, out))
        return plan, out, lse
