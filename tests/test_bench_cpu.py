"""bench.py's reference arm on the CPU: the oracle as it stands, timed on a
bounded sample of the same workload, prints the contract's keys with the
same metric and unit as the GPU arm."""
import time
import types


def test_reference_arm_line():
    import bench
    import workloads as W
    args = types.SimpleNamespace(steps=2, warmup=0, ref_seconds=2.0)
    t0 = time.perf_counter()
    line = bench.run_reference(args, 0, 1)
    wall = time.perf_counter() - t0
    # the time it claims for its timed steps is time it actually spent
    assert line["ms_per_step"] * line["steps"] / 1e3 <= wall
    assert line["ms_per_full_step_extrapolated"] > line["ms_per_step"]
    # the same config as the GPU arm prints
    assert line["config"] == bench.bench_config(W.llama3_8b_prompt(), 1)
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    # only rank 0 works; the others return nothing
    assert bench.run_reference(args, 1, 2) is None
