"""Shared helpers for the GPU parity tests: run a workload through the CUDA
library and through the fp64 oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import math
from typing import List, Optional, Sequence

import numpy as np
import torch

import oracle
import workloads as W

BF16_ATOL = 2e-2   # max-abs error bound for BF16 outputs against the fp64 oracle
FP32_ATOL = 1e-4   # max-abs error bound for FP32 outputs
BF16_LSE_ATOL = 2e-3
FP32_LSE_ATOL = 1e-4
BF16_REL_RMS = 1e-2  # gate on the relative RMS error of each checked step
# Gate on every (token, query head) row: |o_gpu - o_ref|_2 <= ROW_REL * |o_ref|_2.
# BF16 output rounding alone gives about 2^-9 / sqrt(3) relative per row, and
# P rounded to bf16 before the PV product about as much again; a mask or
# offset error confined to one row moves that row by far more once the
# softmax is peaked (the peaky and needle input variants).
BF16_ROW_REL = 2e-2
FP32_ROW_REL = 1e-3
# A BF16 output is stored rounded to bf16: half an ulp, up to 2^-8 |o|.  The
# max-abs bound is applied to the error beyond that rounding, |o - o_ref| <=
# 2e-2 + 2^-8 |o_ref| per element: at |o| >= 4 half an ulp alone is 2^-6, and
# a result whose fp32 value lies near a rounding midpoint (P itself rounded to
# bf16 before the PV product moves it by up to 2^-9 relative) lands one ulp,
# 2^-5, from the exact value.  Below |o| = 0.5 the allowance is under 2e-3.
BF16_ROUNDING_REL = 2.0 ** -8


def to_oracle(t: torch.Tensor) -> np.ndarray:
    """float32 values, or bfloat16 bit patterns as uint16."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(t.dtype)


def bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy()
    return t.view(torch.int32).numpy()


def params_for(w: W.Workload, flags=None, kv_segment_size=None, timeout_cycles=0):
    import chunked_prefill_paged_gb300 as cpa
    sh = w.shape
    return cpa.Params(sh.num_heads_q, sh.num_heads_kv, sh.head_dim, sh.block_size, w.num_blocks,
                      sh.kv_segment_size if kv_segment_size is None else kv_segment_size, sh.scale,
                      cpa.DTYPE_FP32 if sh.dtype == "f32" else cpa.DTYPE_BF16,
                      cpa.FLAG_FUSE_KV_WRITE if flags is None else flags, timeout_cycles)


def sample_rows(step: W.Step, n_per_req: int, seed: int) -> List[int]:
    """First and last token of every request plus random ones (sorted, unique)."""
    rng = np.random.default_rng(seed)
    cu = step.cu_new_tokens
    rows = set()
    for r in range(len(step.num_new_tokens)):
        a, b = int(cu[r]), int(cu[r + 1])
        if b <= a:
            continue
        rows.update([a, b - 1])
        k = min(n_per_req, b - a)
        rows.update(int(x) for x in rng.integers(a, b, size=k))
    return sorted(rows)


class Result:
    def __init__(self):
        self.max_err = 0.0
        self.max_err_beyond_bf16 = 0.0  # max of |o - o_ref| - 2^-8 |o_ref|
        self.max_lse_err = 0.0
        self.rel_rms = []
        self.max_row_rel = 0.0
        self.rows_checked = 0

    def add(self, gpu_out: np.ndarray, ref_out: np.ndarray, gpu_lse: Optional[np.ndarray], ref_lse: np.ndarray):
        assert np.all(np.isfinite(gpu_out)), "non-finite output"
        err = np.abs(gpu_out.astype(np.float64) - ref_out)
        self.max_err = max(self.max_err, float(err.max()) if err.size else 0.0)
        if err.size:
            self.max_err_beyond_bf16 = max(self.max_err_beyond_bf16,
                                           float((err - BF16_ROUNDING_REL * np.abs(ref_out)).max()))
            self.rel_rms.append(float(np.sqrt((err ** 2).mean()) / max(np.sqrt((ref_out ** 2).mean()), 1e-30)))
            e_row = np.sqrt((err ** 2).sum(axis=-1))
            r_row = np.sqrt((ref_out.astype(np.float64) ** 2).sum(axis=-1))
            self.max_row_rel = max(self.max_row_rel, float((e_row / np.maximum(r_row, 1e-30)).max()))
        if gpu_lse is not None and gpu_lse.size:
            self.max_lse_err = max(self.max_lse_err, float(np.abs(gpu_lse.astype(np.float64) - ref_lse).max()))
        self.rows_checked += gpu_out.shape[0]


def run_and_compare(w: W.Workload, *, flags=None, kv_segment_size=None, rows_per_req: Optional[int] = None,
                    steps_to_check: Optional[Sequence[int]] = None, threads=None, check_pool=True,
                    seed: int = 0, device="cuda", variant: str = "plain"):
    """Run every step of `w` on the GPU (fused K/V write unless flags say
    otherwise, then the standalone write) and in the oracle; compare the
    checked steps' outputs (all rows, or a sample) and the final pool.
    variant: the query values (workloads.apply_variant)."""
    import chunked_prefill_paged_gb300 as cpa
    sh = w.shape
    t = w.materialize(device)
    W.apply_variant(t, variant, sh.num_heads_q // sh.num_heads_kv)
    k_pool_o = to_oracle(t.k_cache)
    v_pool_o = to_oracle(t.v_cache)
    params = params_for(w, flags, kv_segment_size)
    fused = bool(params.flags & cpa.FLAG_FUSE_KV_WRITE)
    res = Result()
    steps_to_check = range(len(w.steps)) if steps_to_check is None else steps_to_check
    for si, step in enumerate(w.steps):
        batch = cpa.Batch(step.cached_seq_len, step.num_new_tokens, w.block_table, device=device)
        q, kn, vn = t.step_inputs(step)
        out, lse = cpa.attention(batch, params, q, kn, vn, t.k_cache, t.v_cache)
        if not fused:
            cpa.paged_kv_write(batch, params, kn, vn, t.k_cache, t.v_cache)
        torch.cuda.synchronize()
        ob = oracle.Batch(step.cached_seq_len, step.num_new_tokens, w.block_table)
        qo, kno, vno = to_oracle(q), to_oracle(kn), to_oracle(vn)
        if si in steps_to_check and step.total_new_tokens > 0:
            rows = None if rows_per_req is None else sample_rows(step, rows_per_req, seed + si)
            ref_o, ref_l = oracle.attention(ob, qo, kno, vno, k_pool_o, v_pool_o, num_heads_q=sh.num_heads_q,
                                            num_heads_kv=sh.num_heads_kv, head_dim=sh.head_dim,
                                            block_size=sh.block_size, scale=sh.scale, rows=rows,
                                            threads=threads)
            idx = slice(None) if rows is None else torch.as_tensor(rows, device=out.device)
            res.add(out[idx].float().cpu().numpy(), ref_o, lse[idx].cpu().numpy(), ref_l)
        k_pool_o, v_pool_o = oracle.kv_write(ob, kno, vno, k_pool_o, v_pool_o, num_heads_kv=sh.num_heads_kv,
                                             head_dim=sh.head_dim, block_size=sh.block_size)
    if check_pool:
        assert np.array_equal(bits(t.k_cache), k_pool_o.view(np.int16 if sh.dtype == "bf16" else np.int32)), \
            "K pool differs from the oracle's write"
        assert np.array_equal(bits(t.v_cache), v_pool_o.view(np.int16 if sh.dtype == "bf16" else np.int32)), \
            "V pool differs from the oracle's write"
    assert cpa.last_device_error() == cpa.SUCCESS
    return res


def gate_failures(res: Result, dtype: str) -> List[str]:
    """The gates every parity test applies, as a list of the ones that fail."""
    bad = []
    if dtype == "f32":
        atol, lse_tol, row_tol = FP32_ATOL, FP32_LSE_ATOL, FP32_ROW_REL
        if not res.max_err <= atol:
            bad.append(f"max-abs error {res.max_err:.3e} > {atol}")
    else:
        atol, lse_tol, row_tol = BF16_ATOL, BF16_LSE_ATOL, BF16_ROW_REL
        if not res.max_err_beyond_bf16 <= atol:
            bad.append(f"max-abs error beyond the bf16 rounding {res.max_err_beyond_bf16:.3e} > {atol} "
                       f"(max-abs {res.max_err:.3e})")
    if not res.max_lse_err <= lse_tol:
        bad.append(f"lse error {res.max_lse_err:.3e} > {lse_tol}")
    if not res.max_row_rel <= row_tol:
        bad.append(f"row relative error {res.max_row_rel:.3e} > {row_tol}")
    if dtype != "f32" and res.rel_rms and not max(res.rel_rms) <= BF16_REL_RMS:
        bad.append(f"relative RMS error {max(res.rel_rms):.3e} > {BF16_REL_RMS}")
    return bad


def assert_within(res: Result, dtype: str):
    bad = gate_failures(res, dtype)
    assert not bad, "; ".join(bad)
