#!/usr/bin/env python
"""Throughput of paged chunked-prefill attention on GB300.

One bench step is one pass of the whole hot path over the workload: the
10,000-token Llama-3-8B-shaped prompt (H_q 32, H_kv 8, d 128, block 128,
kv_segment_size 1024) processed as 5 chunks of 2048 tokens, each chunk one
chunked_prefill_attention call (K/V write fused) over the paged cache.

Printed (rank 0, one JSON line): algorithmic attention TFLOP/s =
4 * H_q * d * visible pairs / time, with the roofline of the attention
kernel, the end-to-end number through the Python API with host buffers, the
oracle timed on the host cores, the SM clocks seen during the timed region,
a secondary line for the decode-heavy mixed step (KV-read GB/s), and the
same mixed step over an FP8 (E4M3) cache ("fp8_mixed", pool bytes counted
at one per element).

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]
  python bench.py --case NAME [--steps K --warmup W]

--case times one attention call of a single workload step (for profiling
under ncu and per-configuration timing) and prints {"case": ..., "ms": ...}:
  llama_chunk        last 1808-token chunk of the Llama-3-8B prompt (bs 128)
  llama_chunk_rope   the same with the rotary embedding applied in the call (theta 5e5)
  long_context_last  last 2048-token chunk of the 32,768-token prompt
                     (H_q 64, bs 16, cached 30,720)
  mixed_step         64 decodes + 512-token chunks under a 2048 budget
  prefix_cache       16 requests sharing a 4096-token cached prefix
  speculative_decode 64 requests x 5 tokens (1 + 4 drafts) over contexts U{1024..32768}
  *_fp8              mixed_step, llama_chunk, speculative_decode over FP8 (E4M3) pools
  serving            the library's engine driving many steps: 64 requests on four shared
                     1024-token system prompts (prefix caching), budget 2048, chunk 512
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
import types

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

L2_FLUSH_BYTES = 256 << 20
METRIC = "chunk-attn TFLOP/s (algorithmic, visible pairs only)"
UNIT = "TFLOP/s"


# name -> (workload constructor, step index, rope_theta, FP8 pools)
CASES = {
    "llama_chunk": (W.llama3_8b_prompt, -1, 0.0, False),
    "llama_chunk_rope": (W.llama3_8b_prompt, -1, 500000.0, False),
    "long_context_last": (W.long_context, -1, 0.0, False),
    "mixed_step": (W.mixed_step, 0, 0.0, False),
    "prefix_cache": (W.prefix_cache, 0, 0.0, False),
    "prefix_cache_rope": (W.prefix_cache, 0, 500000.0, False),
    "long_context_last_rope": (W.long_context, -1, 500000.0, False),
    "speculative_decode": (W.speculative_decode, 0, 0.0, False),
    "llama_chunk_fp8": (W.llama3_8b_prompt, -1, 0.0, True),
    "mixed_step_fp8": (W.mixed_step, 0, 0.0, True),
    "speculative_decode_fp8": (W.speculative_decode, 0, 0.0, True),
    "decode_32x8k": (W.decode_batch, 0, 0.0, False),
    "decode_32x8k_fp8": (W.decode_batch, 0, 0.0, True),
}


def fp8_inputs(cpa, w, t, params, dev):
    """Turn a materialized workload's pools into FP8 codes (input
    generation by torch's float8 conversion) and point params at them."""
    ks, vs = W.fp8_scales(w.shape.num_heads_kv)
    k8 = W.fp8_pool_codes(t.k_cache, ks)
    v8 = W.fp8_pool_codes(t.v_cache, vs)
    t.k_cache, t.v_cache = k8, v8
    params.kv_format = cpa.KV_FP8_E4M3
    params.k_scale = torch.as_tensor(ks, device=dev)
    params.v_scale = torch.as_tensor(vs, device=dev)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="--impl reference: seconds of oracle work over the whole run (warm-up included)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    ap.add_argument("--case", choices=sorted(CASES) + ["serving"], default=None,
                    help="time one attention call of this workload step instead of the bench step")
    return ap.parse_args()


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo")
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# nominal dense peaks of one GB300, reported beside the measured fractions
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_HBM_GBS = 8000.0


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [line.split(",") for line in open(self.path).read().strip().splitlines() if line.strip()]
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if len(r) > 5 + i and "Active" == r[5 + i].strip()})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


KERNEL_SOURCES = ("attn_tc2.cu", "attn_tc.cu", "tc_common.cuh", "device_common.cuh", "ptx_sm100.cuh",
                  "cpa_internal.h", "cpa_api.cu")


def kernel_sources_sha256() -> str:
    """One hash over the sources the attention kernel and its launch are built from."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, "chunked_prefill_paged_gb300", "csrc", name), "rb").read())
    return h.hexdigest()


def kernel_traffic_record():
    """dram bytes per launch of the attention kernel from the committed ncu
    summary, only if none of the kernel's sources changed since the capture."""
    p = os.path.join(ROOT, "profiles", "attn_tc_traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p))
    if rec.get("sources_sha256") != kernel_sources_sha256():
        return None
    return rec


# ---------------------------------------------------------------- oracle leg
def oracle_sample(w: W.Workload, t_cpu, seconds: float):
    """Time the fp64 oracle on host cores over a bounded sample of the last
    chunk's rows (the heaviest step).  Returns (TFLOP/s, cores, description)."""
    import oracle
    sh = w.shape
    ob_pool_k = t_cpu["k_cache"]
    ob_pool_v = t_cpu["v_cache"]
    # the cache the last chunk reads: the oracle's own writes of the earlier chunks
    for step in w.steps[:-1]:
        ob = oracle.Batch(step.cached_seq_len, step.num_new_tokens, w.block_table)
        rows = step.token_rows
        ob_pool_k, ob_pool_v = oracle.kv_write(ob, t_cpu["k"][rows], t_cpu["v"][rows], ob_pool_k, ob_pool_v,
                                               num_heads_kv=sh.num_heads_kv, head_dim=sh.head_dim,
                                               block_size=sh.block_size)
    last = w.steps[-1]
    ob = oracle.Batch(last.cached_seq_len, last.num_new_tokens, w.block_table)
    rows = last.token_rows
    q, k, v = t_cpu["q"][rows], t_cpu["k"][rows], t_cpu["v"][rows]
    cores = oracle.default_threads()
    C = int(last.cached_seq_len[0])

    def run(n):
        sel = np.linspace(0, len(rows) - 1, n).astype(np.int64)
        t0 = time.perf_counter()
        oracle.attention(ob, q, k, v, ob_pool_k, ob_pool_v, num_heads_q=sh.num_heads_q,
                         num_heads_kv=sh.num_heads_kv, head_dim=sh.head_dim, block_size=sh.block_size,
                         scale=sh.scale, rows=sel, threads=cores)
        dt = time.perf_counter() - t0
        flops = sum(W.attention_flops(C + int(i) + 1, sh.num_heads_q, sh.head_dim) for i in sel)
        return dt, flops

    dt, _ = run(cores)
    n = int(max(cores, min(len(rows), cores * seconds / max(dt, 1e-3))))
    dt, flops = run(n)
    desc = (f"{n} of {len(rows)} query tokens (all {sh.num_heads_q} heads) of the last 2048-token chunk "
            f"(cached {C}); fp64, {cores} threads, {dt:.1f} s")
    return flops / dt / 1e12, cores, desc


def to_oracle_np(x: torch.Tensor):
    x = x.contiguous().cpu()
    return x.view(torch.int16).numpy().view(np.uint16) if x.dtype == torch.bfloat16 else x.numpy()


# ---------------------------------------------------------------- GPU leg
def run_ours(args, rank, world, local):
    import chunked_prefill_paged_gb300 as cpa
    from chunked_prefill_paged_gb300 import build
    build.build()
    cpa.load()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    hbm_peak, bf16_peak, peak_kind = measured_peaks()

    w = W.llama3_8b_prompt()
    sh = w.shape
    t = w.materialize(dev, sentinel=W.SENTINEL_ZERO)
    params = cpa.Params(sh.num_heads_q, sh.num_heads_kv, sh.head_dim, sh.block_size, w.num_blocks,
                        sh.kv_segment_size, sh.scale, cpa.DTYPE_BF16, cpa.FLAG_FUSE_KV_WRITE)
    batches = [cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table, device=dev) for s in w.steps]
    inputs = [t.step_inputs(s) for s in w.steps]
    outs = [torch.empty((s.total_new_tokens, sh.num_heads_q, sh.head_dim), dtype=torch.bfloat16, device=dev)
            for s in w.steps]
    ws_bytes = max(cpa.workspace_size(b, params) for b in batches)
    ws = torch.empty(max(ws_bytes // 4, 4), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flops_step = sum(w.flops_per_step())
    # attention, plus the merge kernel when some request is split: the workspace
    # then holds partials in front of the 256-byte work counter (the bench's
    # calls use no RoPE, no FP8 and no tail cut, the workspace's other parts)
    launches_per_step = len(w.steps) + sum(1 for b in batches if cpa.workspace_size(b, params) > 256)

    def one_step(evs=None):
        for i, (b, (q, k, v), o) in enumerate(zip(batches, inputs, outs)):
            if evs is not None:
                evs[i][0].record(stream)
            cpa.chunked_prefill_attention(b, params, q, k, v, t.k_cache, t.v_cache, o, None, ws, stream)
            if evs is not None:
                evs[i][1].record(stream)

    for _ in range(max(args.warmup, 3)):
        one_step()
    torch.cuda.synchronize(dev)
    if cpa.last_device_error(stream) != cpa.SUCCESS:
        raise RuntimeError("device error during warm-up")

    barrier(world)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local)
    clocks.start()
    # the timed steps carry no events between their calls; a second pass of
    # the same steps, outside the timed region, times each launch for the
    # roofline's kernel time
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for k in range(args.steps):
        flush.zero_()  # L2 flush, outside the timed region
        step_ev[k][0].record(stream)
        one_step()
        step_ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    barrier(world)
    launch_ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in w.steps] for _ in range(args.steps)]
    for k in range(args.steps):
        flush.zero_()
        one_step(launch_ev[k])
    torch.cuda.synchronize(dev)
    total_ms = sum(a.elapsed_time(b) for a, b in step_ev)
    kernel_ms = sum(a.elapsed_time(b) for row in launch_ev for a, b in row)
    total_ms = reduce_max(total_ms, world)
    ms_per_step = total_ms / args.steps
    value = world * flops_step * args.steps / (total_ms / 1e3) / 1e12
    achieved = flops_step * args.steps / (kernel_ms / 1e3) / 1e12
    status = cpa.last_device_error(stream)
    if status != cpa.SUCCESS:
        raise RuntimeError(f"device error in the timed region: {cpa.status_string(status)}")

    # end to end through the API with host buffers: H2D of each chunk's
    # q / k / v from pinned memory, the call, D2H of the output.  The copies
    # run on their own streams, one per direction, as a serving loop would
    # run them: every chunk's inputs go up at the start of the step, chunk
    # i's call waits for its own inputs, and its output comes back while
    # chunk i + 1 computes and later inputs still go up (the calls stay in
    # order on the compute stream: each chunk reads the K/V the previous one
    # wrote).
    host_in = [tuple(x.cpu().pin_memory() for x in inp) for inp in inputs]
    host_out = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    dev_in = [tuple(torch.empty_like(x) for x in inp) for inp in inputs]
    h2d = sum(x.numel() * x.element_size() for inp in host_in for x in inp)
    d2h = sum(o.numel() * o.element_size() for o in host_out)
    copy_in, copy_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in batches]
    ev_done = [torch.cuda.Event() for _ in batches]

    def e2e_step():
        copy_in.wait_stream(stream)
        copy_out.wait_stream(stream)
        with torch.cuda.stream(copy_in):
            for i, (hin, din) in enumerate(zip(host_in, dev_in)):
                for d_, h_ in zip(din, hin):
                    d_.copy_(h_, non_blocking=True)
                ev_in[i].record(copy_in)
        for i, (b, din, o, ho) in enumerate(zip(batches, dev_in, outs, host_out)):
            stream.wait_event(ev_in[i])
            cpa.chunked_prefill_attention(b, params, din[0], din[1], din[2], t.k_cache, t.v_cache, o, None, ws,
                                          stream)
            ev_done[i].record(stream)
            with torch.cuda.stream(copy_out):
                copy_out.wait_event(ev_done[i])
                ho.copy_(o, non_blocking=True)
        stream.wait_stream(copy_in)
        stream.wait_stream(copy_out)  # the step ends when the last output is on the host

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for k in range(args.steps):
        flush.zero_()
        e_ev[k][0].record(stream)
        e2e_step()
        e_ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(sum(a.elapsed_time(b) for a, b in e_ev), world)
    e2e_value = world * flops_step * args.steps / (e2e_ms / 1e3) / 1e12

    rec = kernel_traffic_record()
    roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": bf16_peak, "unit": "TFLOP/s",
                "frac": round(achieved / bf16_peak, 4), "peak_kind": f"{peak_kind} bf16 burst",
                "frac_of_nominal": round(achieved / NOMINAL_BF16_TFLOPS, 4),
                "traffic": rec["bytes_per_launch"] if rec else None,
                "kernel": "attn_tc_kernel<128, false>",
                "algorithmic_flops_per_launch": flops_step / len(w.steps)}

    host_copies = pinned_copy_rates(dev, h2d, d2h, e2e_ms / args.steps)

    secondary = fp8_mixed = prefix = long_last = rope = None
    if not args.no_secondary:
        secondary = run_mixed(args, dev, stream, hbm_peak, peak_kind, flush)
        fp8_mixed = run_mixed(args, dev, stream, hbm_peak, peak_kind, flush, fp8=True)
        prefix = run_prefill_extra(args, dev, stream, bf16_peak, peak_kind, flush, W.prefix_cache, 0)
        long_last = run_prefill_extra(args, dev, stream, bf16_peak, peak_kind, flush, W.long_context, -1)
        rope = run_rope_overhead(args, dev, stream, flush)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t_cpu = {"q": to_oracle_np(t.q), "k": to_oracle_np(t.k), "v": to_oracle_np(t.v),
                 "k_cache": to_oracle_np(t.k_cache), "v_cache": to_oracle_np(t.v_cache)}
        v_, cores, desc = oracle_sample(w, t_cpu, args.cpu_seconds)
        cpu = {"value": v_, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": bench_config(w, world),
        "roofline": roofline,
        "e2e": {"value": round(e2e_value, 3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "cpu_baseline": cpu,
        "host_copies": host_copies,
        "secondary": secondary,
        "fp8_mixed": fp8_mixed,
        "prefix_cache": prefix,
        "long_context_last": long_last,
        "rope_last_chunk": rope,
    }
    return line


def pinned_copy_rates(dev, h2d_bytes, d2h_bytes, e2e_ms_per_step):
    """Plain pinned-host copy rates on this machine, one cudaMemcpyAsync per
    direction of the e2e leg's byte counts (H2D alone, D2H alone, both at
    once on two streams), beside the rate the e2e leg's copies reach."""
    up_h = torch.empty(h2d_bytes, dtype=torch.uint8).pin_memory()
    up_d = torch.empty(h2d_bytes, dtype=torch.uint8, device=dev)
    dn_d = torch.empty(d2h_bytes, dtype=torch.uint8, device=dev)
    dn_h = torch.empty(d2h_bytes, dtype=torch.uint8).pin_memory()
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn, reps=10):
        for _ in range(2):
            fn()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize(dev)
        return (time.perf_counter() - t0) / reps

    def up():
        with torch.cuda.stream(s1):
            up_d.copy_(up_h, non_blocking=True)

    def down():
        with torch.cuda.stream(s2):
            dn_h.copy_(dn_d, non_blocking=True)

    def both():
        up()
        down()

    t_up, t_dn, t_both = timed(up), timed(down), timed(both)
    gbs = lambda b, t: round(b / t / 1e9, 1)
    return {"h2d_gbs": gbs(h2d_bytes, t_up), "d2h_gbs": gbs(d2h_bytes, t_dn),
            "both_gbs": gbs(h2d_bytes + d2h_bytes, t_both),
            "e2e_leg_gbs": gbs(h2d_bytes + d2h_bytes, e2e_ms_per_step / 1e3),
            "e2e_leg_frac_of_both": round(t_both / (e2e_ms_per_step / 1e3), 3),
            "how": "one pinned cudaMemcpyAsync per direction of the e2e bytes, host wall time over 10 reps"}


def warm_cache(cpa, w, t, params, dev, upto):
    """Write the K/V of steps [0, upto) into the pool (as the earlier chunks'
    calls would have), so a later chunk reads real cached values."""
    for s in w.steps[:upto]:
        b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table, device=dev)
        _, k, v = t.step_inputs(s)
        cpa.paged_kv_write(b, params, k, v, t.k_cache, t.v_cache)


def tc_kernel_name(sh, step, rope=False, fp8=False):
    """The tensor-core kernel the library's planner picks for this batch (its
    rule, restated for labelling): the two-pipeline kernel for BF16 pools at
    block sizes up to 32 with query tiles to pair and a query group dividing
    128 (with the rotary embedding after the rotation pre-pass)."""
    G = sh.num_heads_q // sh.num_heads_kv
    pairs = any(int(n) * G > 128 for n in step.num_new_tokens)
    if not fp8 and 128 % G == 0 and sh.block_size <= 32 and pairs:
        return f"attn_tc2_kernel<{sh.head_dim}>"
    return f"attn_tc_kernel<{sh.head_dim}, {'true' if fp8 else 'false'}>"


def time_prefill_calls(args, dev, stream, flush, w, t, i, thetas):
    """Median CUDA-event time (ms) of one attention call of step i for each
    rope_theta in `thetas`, the calls of the different thetas interleaved
    (each after an L2 flush)."""
    import chunked_prefill_paged_gb300 as cpa
    sh = w.shape
    s = w.steps[i]
    plist = [cpa.Params(sh.num_heads_q, sh.num_heads_kv, sh.head_dim, sh.block_size, w.num_blocks,
                        sh.kv_segment_size, sh.scale, cpa.DTYPE_BF16, cpa.FLAG_FUSE_KV_WRITE, rope_theta=th)
             for th in thetas]
    b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table, device=dev)
    q, k, v = t.step_inputs(s)
    out = torch.empty_like(q)
    n = max(cpa.workspace_size(b, p) for p in plist)
    ws = torch.empty(max(n // 4, 4), dtype=torch.float32, device=dev)
    for _ in range(max(args.warmup, 3)):
        for p in plist:
            cpa.chunked_prefill_attention(b, p, q, k, v, t.k_cache, t.v_cache, out, None, ws, stream)
    torch.cuda.synchronize(dev)
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in plist]
           for _ in range(args.steps)]
    for row in evs:
        for p, (e0, e1) in zip(plist, row):
            flush.zero_()
            e0.record(stream)
            cpa.chunked_prefill_attention(b, p, q, k, v, t.k_cache, t.v_cache, out, None, ws, stream)
            e1.record(stream)
    torch.cuda.synchronize(dev)
    if cpa.last_device_error(stream) != cpa.SUCCESS:
        raise RuntimeError(f"device error in {w.name}")
    return [statistics.median(row[j][0].elapsed_time(row[j][1]) for row in evs) for j in range(len(plist))]


def run_prefill_extra(args, dev, stream, bf16_peak, peak_kind, flush, make, idx):
    """A prefill-heavy configuration's attention call (one workload step,
    its cache holding the earlier chunks' K/V): algorithmic TFLOP/s against
    the measured bf16 peak."""
    import chunked_prefill_paged_gb300 as cpa
    w = make()
    sh = w.shape
    t = w.materialize(dev, sentinel=W.SENTINEL_ZERO)
    i = idx % len(w.steps)
    s = w.steps[i]
    params = cpa.Params(sh.num_heads_q, sh.num_heads_kv, sh.head_dim, sh.block_size, w.num_blocks,
                        sh.kv_segment_size, sh.scale, cpa.DTYPE_BF16, cpa.FLAG_FUSE_KV_WRITE)
    warm_cache(cpa, w, t, params, dev, i)
    (ms,) = time_prefill_calls(args, dev, stream, flush, w, t, i, [0.0])
    flops = w.flops_per_step()[i]
    achieved = flops / (ms / 1e3) / 1e12
    del t
    torch.cuda.empty_cache()
    return {"workload": w.name, "step": i, "cached_seq_len": [int(x) for x in sorted(set(s.cached_seq_len))],
            "tokens": int(s.total_new_tokens), "metric": "chunk-attn TFLOP/s (algorithmic, visible pairs only)",
            "value": round(achieved, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4), "flops_per_step": flops,
            "launches_per_step": 1,
            "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": round(achieved / bf16_peak, 4), "peak_kind": f"{peak_kind} bf16 burst",
                         "frac_of_nominal": round(achieved / NOMINAL_BF16_TFLOPS, 4),
                         "traffic": None, "kernel": tc_kernel_name(sh, s)},
            "l2": "flushed before every timed call (256 MiB write)"}


def run_rope_overhead(args, dev, stream, flush, theta=500000.0):
    """The Llama prompt's last chunk (cached 8192) with the rotary embedding
    applied in the call against the same call without it, interleaved."""
    import chunked_prefill_paged_gb300 as cpa
    w = W.llama3_8b_prompt()
    sh = w.shape
    t = w.materialize(dev, sentinel=W.SENTINEL_ZERO)
    i = len(w.steps) - 1
    params = cpa.Params(sh.num_heads_q, sh.num_heads_kv, sh.head_dim, sh.block_size, w.num_blocks,
                        sh.kv_segment_size, sh.scale, cpa.DTYPE_BF16, cpa.FLAG_FUSE_KV_WRITE)
    warm_cache(cpa, w, t, params, dev, i)
    steps = types.SimpleNamespace(steps=max(args.steps, 20), warmup=args.warmup)
    ms_plain, ms_rope = time_prefill_calls(steps, dev, stream, flush, w, t, i, [0.0, theta])
    del t
    torch.cuda.empty_cache()
    return {"workload": w.name, "step": i, "rope_theta": theta, "ms_no_rope": round(ms_plain, 4),
            "ms_rope": round(ms_rope, 4), "overhead": round(ms_rope / ms_plain - 1.0, 4),
            "kernel": tc_kernel_name(sh, w.steps[i], rope=True), "calls_each": steps.steps,
            "how": "median of interleaved calls, each after a 256 MiB L2 flush"}


def run_mixed(args, dev, stream, hbm_peak, peak_kind, flush, fp8=False):
    """Decode-heavy mixed step (64 decodes + 4 prefill chunks): KV-read GB/s
    (with FP8 pools the pool bytes count one per element)."""
    import chunked_prefill_paged_gb300 as cpa
    w = W.mixed_step()
    sh = w.shape
    t = w.materialize(dev, sentinel=W.SENTINEL_ZERO)
    s = w.steps[0]
    params = cpa.Params(sh.num_heads_q, sh.num_heads_kv, sh.head_dim, sh.block_size, w.num_blocks,
                        sh.kv_segment_size, sh.scale, cpa.DTYPE_BF16, cpa.FLAG_FUSE_KV_WRITE)
    if fp8:
        fp8_inputs(cpa, w, t, params, dev)
    b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table, device=dev)
    q, k, v = t.step_inputs(s)
    out = torch.empty_like(q)
    n = cpa.workspace_size(b, params)
    ws = torch.empty(max(n // 4, 4), dtype=torch.float32, device=dev)
    for _ in range(max(args.warmup, 3)):
        cpa.chunked_prefill_attention(b, params, q, k, v, t.k_cache, t.v_cache, out, None, ws, stream)
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        cpa.chunked_prefill_attention(b, params, q, k, v, t.k_cache, t.v_cache, out, None, ws, stream)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = statistics.median(a.elapsed_time(b_) for a, b_ in evs)
    if cpa.last_device_error(stream) != cpa.SUCCESS:
        raise RuntimeError("device error in the mixed step")
    byts = w.bytes_per_step(1 if fp8 else None)[0]
    gbs = byts / (ms / 1e3) / 1e9
    flops = w.flops_per_step()[0]
    del t
    torch.cuda.empty_cache()
    return {"workload": w.name + ("_fp8" if fp8 else ""), "metric": "mixed-batch algorithmic GB/s",
            "value": round(gbs, 1), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "bytes_per_step": byts, "tflops": round(flops / (ms / 1e3) / 1e12, 2),
            "peak": hbm_peak, "frac": round(gbs / hbm_peak, 4), "peak_kind": f"{peak_kind} HBM copy",
            "frac_of_nominal": round(gbs / NOMINAL_HBM_GBS, 4)}


def run_case(args, local):
    """One attention call of one workload step, timed with CUDA events after
    an L2 flush; for profiling and per-configuration numbers."""
    import chunked_prefill_paged_gb300 as cpa
    from chunked_prefill_paged_gb300 import build
    build.build()
    cpa.load()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    make, idx, rope_theta, fp8 = CASES[args.case]
    w = make()
    sh = w.shape
    t = w.materialize(dev, sentinel=W.SENTINEL_ZERO)
    s = w.steps[idx]
    params = cpa.Params(sh.num_heads_q, sh.num_heads_kv, sh.head_dim, sh.block_size, w.num_blocks,
                        sh.kv_segment_size, sh.scale, cpa.DTYPE_BF16 if sh.dtype == "bf16" else cpa.DTYPE_FP32,
                        cpa.FLAG_FUSE_KV_WRITE, rope_theta=rope_theta)
    if fp8:
        fp8_inputs(cpa, w, t, params, dev)
    warm_cache(cpa, w, t, params, dev, idx % len(w.steps))
    b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table, device=dev)
    q, k, v = t.step_inputs(s)
    out = torch.empty_like(q)
    n = cpa.workspace_size(b, params)
    ws = torch.empty(max(n // 4, 4), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        cpa.chunked_prefill_attention(b, params, q, k, v, t.k_cache, t.v_cache, out, None, ws, stream)
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        cpa.chunked_prefill_attention(b, params, q, k, v, t.k_cache, t.v_cache, out, None, ws, stream)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    if cpa.last_device_error(stream) != cpa.SUCCESS:
        raise RuntimeError("device error")
    ms = statistics.median(a.elapsed_time(b_) for a, b_ in evs)
    i = idx % len(w.steps)
    flops, byts = w.flops_per_step()[i], w.bytes_per_step(1 if fp8 else None)[i]
    return {"case": args.case, "workload": w.name, "steps": args.steps, "warmup": args.warmup, "ms": round(ms, 4),
            "tflops": round(flops / (ms / 1e3) / 1e12, 1), "gbs": round(byts / (ms / 1e3) / 1e9, 1),
            "flops": flops, "bytes": byts, "tokens": int(s.total_new_tokens)}


def run_serving(args, local):
    """Whole serving iterations through the library's engine: its plan, the
    batch's one host-to-device copy, a stand-in model's q / k / v (token and
    position tables on the device), the attention call (K/V write fused) and
    the commit.  Reports tokens per second of the whole loop and the share
    the attention call takes."""
    import chunked_prefill_paged_gb300 as cpa
    from chunked_prefill_paged_gb300 import build
    from chunked_prefill_paged_gb300.serving import Server
    build.build()
    cpa.load()
    dev = torch.device("cuda", local)
    hq, hkv, d, bs = 32, 8, 128, 16
    vocab, max_pos = 1000, 4096
    num_reqs, budget, chunk, max_new = 64, 2048, 512, 64
    g = torch.Generator(device=dev)
    g.manual_seed(1007)
    tab = lambda n, h: (torch.randn(n, h, d, generator=g, device=dev) * 0.5).to(torch.bfloat16)
    tq, pq, tk, pk, tv, pv = tab(vocab, hq), tab(max_pos, hq), tab(vocab, hkv), tab(max_pos, hkv), tab(vocab, hkv), \
        tab(max_pos, hkv)
    rng = np.random.default_rng(1007)
    systems = [rng.integers(0, vocab, size=1024) for _ in range(4)]
    prompts = [np.concatenate([systems[i % 4], rng.integers(0, vocab, size=int(rng.integers(128, 1025)))])
               for i in range(num_reqs)]
    cols = (max(len(p) for p in prompts) + max_new) // bs + 1
    num_blocks = sum(len(p) + max_new for p in prompts) // bs + num_reqs + 1
    eng = cpa.Engine(num_blocks, bs, cols, budget, chunk, scope_key=1007)
    for i, p in enumerate(prompts):
        eng.add_request(i, p, max_new)
    params = cpa.Params(hq, hkv, d, bs, num_blocks, 1024, 1.0 / np.sqrt(d), cpa.DTYPE_BF16, cpa.FLAG_FUSE_KV_WRITE)
    k_cache = torch.zeros((num_blocks, bs, hkv, d), dtype=torch.bfloat16, device=dev)
    v_cache = torch.zeros_like(k_cache)
    server = Server(eng, params, k_cache, v_cache, max_reqs=num_reqs, device=dev)
    stream = torch.cuda.current_stream(dev)
    attn_ev = []

    def make_qkv(plan):
        pos = np.concatenate([np.arange(c, c + n) for c, n in zip(plan.cached_seq_len, plan.num_new_tokens)])
        ti = torch.from_numpy(plan.token_ids.astype(np.int64)).pin_memory().to(dev, non_blocking=True)
        pi = torch.from_numpy(pos.astype(np.int64)).pin_memory().to(dev, non_blocking=True)
        q, k, v = tq[ti] + pq[pi], tk[ti] + pk[pi], tv[ti] + pv[pi]
        e0 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        attn_ev.append(e0)
        return q, k, v

    def sample(plan, out):
        e1 = torch.cuda.Event(enable_timing=True)
        e1.record(stream)
        attn_ev.append(e1)
        return rng.integers(0, vocab, size=plan.num_reqs)

    steps = tokens = 0
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    while eng.num_unfinished() > 0 and steps < 5000:
        plan, out, _ = server.step(make_qkv, sample)
        steps += 1
        tokens += int(plan.num_new_tokens.sum())
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t0
    if cpa.last_device_error(stream) != cpa.SUCCESS:
        raise RuntimeError("device error")
    attn_ms = sum(attn_ev[i].elapsed_time(attn_ev[i + 1]) for i in range(0, len(attn_ev) - 1, 2))
    return {"case": "serving", "requests": num_reqs, "steps": steps, "tokens": tokens,
            "tokens_per_s": round(tokens / wall, 1), "ms_per_step": round(wall * 1e3 / max(steps, 1), 4),
            "attention_ms_per_step": round(attn_ms / max(steps, 1), 4),
            "attention_share": round(attn_ms / (wall * 1e3), 3),
            "config": {"H_q": hq, "H_kv": hkv, "head_dim": d, "block_size": bs, "budget": budget, "chunk": chunk,
                       "system_prompts": "4 x 1024 tokens", "suffix": "U{128..1024}", "max_new_tokens": max_new}}


def bench_config(w: W.Workload, world: int) -> dict:
    """The bench line's config (both arms print the same one)."""
    sh = w.shape
    return {"workload": w.name, "prompt_tokens": 10000, "chunk": 2048, "chunks_per_step": len(w.steps),
            "H_q": sh.num_heads_q, "H_kv": sh.num_heads_kv, "head_dim": sh.head_dim,
            "block_size": sh.block_size, "kv_segment_size": sh.kv_segment_size,
            "flops_per_step": sum(w.flops_per_step()), "l2": "flushed before every timed step (256 MiB write)",
            "parallelism": f"replicas x{world}"}


def run_reference(args, rank, world):
    """The oracle as it stands on the host cores, same metric and workload.
    Each step is a bounded sample of the workload (query rows of the last
    chunk, all heads); value is the algorithmic TFLOP/s of the sampled work,
    ms_per_step the wall time each sampled step took.  The time a whole step
    (all five chunks) would take at that rate is reported separately."""
    if rank != 0:
        return None
    w = W.llama3_8b_prompt()
    t = w.materialize("cpu", sentinel=W.SENTINEL_ZERO)
    t_cpu = {"q": to_oracle_np(t.q), "k": to_oracle_np(t.k), "v": to_oracle_np(t.v),
             "k_cache": to_oracle_np(t.k_cache), "v_cache": to_oracle_np(t.v_cache)}
    per = max(1.0, getattr(args, "ref_seconds", 60.0) / max(args.steps + args.warmup, 1))
    vals, walls = [], []
    desc = ""
    cores = 1
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        v_, cores, desc = oracle_sample(w, t_cpu, per)
        if i >= args.warmup:
            vals.append(v_)
            walls.append(time.perf_counter() - t0)
    value = statistics.mean(vals) if vals else 0.0
    ms_sample = 1e3 * statistics.mean(walls) if walls else None
    full_ms = sum(w.flops_per_step()) / (value * 1e12) * 1e3 if value > 0 else None
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_sample, 1) if ms_sample else None,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(w, world),
        "step_kind": "a bounded sample of the workload per step (see cpu_baseline.sample); "
                     "ms_per_step is the wall time of that sample, including its cache set-up",
        "ms_per_full_step_extrapolated": round(full_ms, 1) if full_ms else None,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    rank, world, local = dist_setup()
    if args.case is not None:
        runner = run_serving if args.case == "serving" else run_case
        line = runner(args, local) if rank == 0 else None
    elif args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
