"""The library's host-side work planner (make_plan in csrc/cpa_api.cu) on the
CPU, through tests/plan_harness.cu, which compiles the planner with stub
launchers and runs it for a given SM count.  A GPU is needed for the planner
to see an SM count in the library itself (workspace sizes on a machine with no
device carry no SM-dependent part), so these cases pin the SM-dependent
choices here:

* the split length grows from kv_segment_size while the batch keeps at least
  1024 units, up to 8192 keys;
* the fine tail: the last requests in batch order whose split units, at half
  the piece length, make three waves of CTAs;
* the interleave span: prefill and decode units alternate over the indices
  before the fine tail's units;
* the opt-in tail cut of prefill batches (CPA_FLAG_TAIL_SPLIT);
* the workspace layout (partials, then the counters, 256-byte aligned);
* the kernel and the query tiles per direct unit: the two-pipeline kernel
  for BF16 batches at block sizes 16 and 32 with query tiles to pair, with
  pairs unless single tiles schedule better; else the one-pipeline kernel
  with single tiles.

The expected values restate the rules in plain Python over the same inputs."""
import json
import math
import os
import shutil
import subprocess

import pytest

import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FUSE, NO_SPLIT, TAIL_SPLIT = 0x1, 0x4, 0x8


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc is not available")
    exe = str(tmp_path_factory.mktemp("plan") / "plan_harness")
    subprocess.run([nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a",
                    os.path.join(ROOT, "tests", "plan_harness.cu"), "-o", exe], check=True, capture_output=True)
    return exe


def plan(harness, reqs, sms=152, hq=32, hkv=8, d=128, bs=16, seg=1024, flags=FUSE, kv_format=0, rope=0.0):
    text = f"{sms} {hq} {hkv} {d} {bs} {seg} 1 {flags} {kv_format} {len(reqs)}\n"
    text += "\n".join(f"{c} {n}" for c, n in reqs) + f"\n{rope}\n"
    out = subprocess.run([harness], input=text, capture_output=True, text=True, check=True).stdout
    return json.loads(out)


def split_pieces(C, N, G, length):
    """Pieces of a request whose rows fit one 128-row tile, else 0 (a direct request)."""
    if N <= 0 or math.ceil(N * G / 128) > 1:
        return 0
    k = math.ceil((C + N) / length)
    return k if k > 1 else 0


def direct_units(C, N, G, hkv, length, tiles_per_unit=2):
    if N <= 0 or split_pieces(C, N, G, length):
        return 0
    return hkv * math.ceil(math.ceil(N * G / 128) / tiles_per_unit)


def expected(reqs, sms, G=4, hkv=8, base=1024, tiles_per_unit=2):
    length = base
    while length * 2 <= 8192:
        units = sum(hkv * split_pieces(c, n, G, length * 2) + direct_units(c, n, G, hkv, length * 2, tiles_per_unit)
                    for c, n in reqs)
        if units < 1024:
            break
        length *= 2
    fine_from, fine = -1, 0
    if sms > 0 and length > base:
        fine = max(base, length // 2)
        fu = 0
        r1 = len(reqs)
        for r in range(len(reqs) - 1, -1, -1):
            if fu >= 3 * sms:
                break
            fu += hkv * split_pieces(*reqs[r], G, fine)
            r1 = r
        if fu > 0:
            fine_from = r1
        else:
            fine = 0
    lens = [fine if fine_from >= 0 and r >= fine_from else length for r in range(len(reqs))]
    split = [hkv * split_pieces(c, n, G, l) for (c, n), l in zip(reqs, lens)]
    direct = [direct_units(c, n, G, hkv, l, tiles_per_unit) for (c, n), l in zip(reqs, lens)]
    fine_units = sum(split[r] for r in range(len(reqs)) if fine_from >= 0 and r >= fine_from)
    return dict(split_len=length, split_len_fine=fine if fine_from >= 0 else 0, fine_from=fine_from,
                fine_units=fine_units, split_units=sum(split), direct_units=sum(direct),
                interleave_span=sum(split) + sum(direct) - fine_units)


def check(got, want):
    for k, v in want.items():
        assert got[k] == v, (k, got[k], v)


@pytest.mark.parametrize("sms", [152, 64, 0])
def test_decode_batch_plan(harness, sms):
    reqs = [(8192, 1)] * 32
    got = plan(harness, reqs, sms=sms)
    want = expected(reqs, sms)
    check(got, want)
    if sms == 152:
        # 32 x 5 pieces of 2048 keys; the last 7 requests (9 pieces of 1024
        # each, 72 units apiece, 504 >= 3 x 152) form the fine tail
        assert (got["split_len"], got["split_len_fine"], got["fine_from"], got["fine_units"]) == (2048, 1024, 25, 504)
    if sms == 0:
        assert got["fine_from"] == -1 and got["split_units"] == 32 * 5 * 8
    # partials (4 rows x 128 + 8 floats per piece and head), then one 256-byte counter block
    floats = got["split_units"] * (4 * 128 + 8)
    assert got["sched_off"] == math.ceil(floats * 4 / 256) * 256
    assert got["ws_bytes"] == got["sched_off"] + 256


def test_mixed_step_plan_interleaves_before_the_fine_tail(harness):
    w = W.mixed_step()
    s = w.steps[0]
    reqs = [(int(c), int(n)) for c, n in zip(s.cached_seq_len, s.num_new_tokens)]
    got = plan(harness, reqs)
    check(got, expected(reqs, 152))
    # the fine tail is the last decodes; the prefill chunks (after them in
    # batch order) stay direct, and every direct unit precedes the fine tail
    n_dec = sum(1 for _, n in reqs if n == 1)
    assert 0 <= got["fine_from"] < n_dec
    assert got["fine_units"] >= 3 * 152
    assert got["direct_units"] <= got["interleave_span"] < got["direct_units"] + got["split_units"]


def test_no_split_flag_keeps_every_request_direct(harness):
    reqs = [(8192, 1)] * 32
    got = plan(harness, reqs, flags=FUSE | NO_SPLIT)
    assert got["split_units"] == 0 and got["direct_units"] == 32 * 8 and got["fine_from"] == -1
    assert got["ws_bytes"] == 256  # the work counter only


@pytest.mark.parametrize("flags,sms,cut", [(FUSE | TAIL_SPLIT, 152, (56, 2)), (FUSE, 152, (0, 0)),
                                          (FUSE | TAIL_SPLIT, 0, (0, 0)),
                                          (FUSE | TAIL_SPLIT | NO_SPLIT, 152, (0, 0))])
def test_tail_cut_is_opt_in(harness, flags, sms, cut):
    # a 2048-token chunk over 6144 cached tokens: 512 query tiles of about
    # 56 key tiles, 3.37 waves on 152 SMs; with the flag the planner cuts
    # the last wave's 56 tiles in two
    got = plan(harness, [(6144, 2048)], sms=sms, bs=128, flags=flags)
    # block size 128: the one-pipeline kernel, single query tiles
    assert (got["tc2"], got["tiles_per_unit"]) == (0, 1)
    assert got["direct_units"] == 512 and got["split_units"] == 0
    assert (got["tail_units"], got["tail_pieces"]) == cut
    # partials of the pieces (128 rows x 128 + 256 floats each), then the
    # work counter and eight counters per cut tile
    floats = cut[0] * cut[1] * (128 * 128 + 256)
    counters = math.ceil(4 * (1 + 8 * cut[0]) / 256) * 256
    assert got["ws_bytes"] == math.ceil(floats * 4 / 256) * 256 + counters


def test_fp8_pools_plan_like_bf16(harness):
    reqs = [(8192, 1)] * 32
    bf16 = plan(harness, reqs)
    fp8 = plan(harness, reqs, kv_format=1)
    for k in ("split_len", "split_len_fine", "fine_from", "split_units", "direct_units"):
        assert fp8[k] == bf16[k]


def test_query_tile_pairs_with_bf16_pools_only(harness):
    # a 2048-token chunk: 64 query tiles per kv head, in 32 pairs with BF16
    # pools; FP8 pools keep single tiles (their kernel has one tile per unit)
    bf16 = plan(harness, [(4096, 2048)], bs=16)
    fp8 = plan(harness, [(4096, 2048)], bs=16, kv_format=1)
    assert (bf16["tiles_per_unit"], bf16["direct_units"]) == (2, 8 * 32)
    assert (fp8["tiles_per_unit"], fp8["direct_units"]) == (1, 8 * 64)
    # an odd tile count: the last pair of each head is a single tile
    odd = plan(harness, [(0, 3 * 32)], bs=16)
    assert odd["direct_units"] == 8 * 2


def expected_tiles_per_unit(reqs, sms, G=4, hkv=8, bs=16, d=128):
    """The planner's choice restated: the two-pipeline kernel only at block
    sizes 16 and 32 with some request of more than 128 rows (else single
    tiles on the one-pipeline kernel); there, greedy list schedules of
    pairs and of single query tiles (costs in 1024-cycle periods: a key tile
    max(2, boxes) for a pair, max(1, boxes) for a single tile, boxes = K and
    V TMA boxes x 75 cycles; 4 per unit); singles when they end 3 % sooner."""
    import heapq
    if bs > 32 or not any(n * G > 128 for _, n in reqs):
        return 1
    boxes = 2 * math.ceil(128 / min(bs, 128)) * (d // 64) * 75 / 1024

    def end(tpu):
        h = [0.0] * sms
        for c, n_tok in reqs:
            if n_tok <= 0:
                continue
            rows = n_tok * G
            n_qt = math.ceil(rows / 128)
            for i in range(math.ceil(n_qt / tpu)):
                last = n_qt - 1 - i * tpu
                first = max(0, last - tpu + 1)
                last_tok = (min((last + 1) * 128, rows) - 1) // G
                n = math.ceil(c / 128) + math.ceil((last_tok + 1) / 128)
                cost = n * (max(2, boxes) if last > first else max(1, boxes)) + 4
                for _ in range(hkv):
                    heapq.heappush(h, heapq.heappop(h) + cost)
        return max(h)

    return 1 if end(1) < 0.97 * end(2) else 2


@pytest.mark.parametrize("reqs,bs,hq", [([(8192, 1808)], 128, 32), ([(8192, 1808)], 16, 64),
                                        ([(6144, 2048)], 128, 32), ([(0, 2048)], 128, 32),
                                        ([(4096, 300), (4096, 512), (100, 1000)], 16, 32),
                                        ([(30720, 2048)], 16, 64), ([(2048, 700), (0, 64)], 64, 32)])
def test_tiles_per_unit_choice(harness, reqs, bs, hq):
    got = plan(harness, reqs, bs=bs, hq=hq)
    want = expected_tiles_per_unit(reqs, 152, G=hq // 8, bs=bs)
    assert got["tiles_per_unit"] == want
    assert got["direct_units"] == sum(direct_units(c, n, hq // 8, 8, 1024, want) for c, n in reqs)


def test_kernel_choice(harness):
    # block size 16 with rows to pair: the two-pipeline kernel
    assert plan(harness, [(30720, 2048)], bs=16, hq=64)["tc2"] == 1
    # block size 128, decode-only batches, FP8 pools, the tail cut: one pipeline
    assert plan(harness, [(8192, 1808)], bs=128)["tc2"] == 0
    assert plan(harness, [(8192, 1)] * 8, bs=16)["tc2"] == 0
    assert plan(harness, [(30720, 2048)], bs=16, kv_format=1)["tc2"] == 0
    assert plan(harness, [(30720, 2048)], bs=16, flags=FUSE | TAIL_SPLIT)["tc2"] == 0
    # the rotary embedding: the one-pipeline kernel applies it in the same
    # launch (BF16 pools); the two-pipeline kernel and FP8 pools take the
    # rotation pre-pass
    got = plan(harness, [(30720, 2048)], bs=16, rope=500000.0)
    assert (got["tc2"], got["rope_fused"]) == (1, 0)
    assert plan(harness, [(8192, 1808)], bs=128, rope=500000.0)["rope_fused"] == 1
    assert plan(harness, [(8192, 1808)], bs=128, kv_format=1, rope=500000.0)["rope_fused"] == 0
    assert plan(harness, [(8192, 1808)], bs=128)["rope_fused"] == 0


def test_bench_kernel_labels_follow_the_planner(harness):
    # bench.py names the kernel of each prefill line by restating the
    # planner's choice; the planner itself decides here
    import bench
    import workloads as W
    for make, idx in [(W.prefix_cache, 0), (W.long_context, -1), (W.llama3_8b_prompt, -1), (W.mixed_step, 0)]:
        w = make()
        sh = w.shape
        s = w.steps[idx]
        reqs = list(zip((int(c) for c in s.cached_seq_len), (int(n) for n in s.num_new_tokens)))
        got = plan(harness, reqs, hq=sh.num_heads_q, hkv=sh.num_heads_kv, d=sh.head_dim, bs=sh.block_size,
                   seg=sh.kv_segment_size)
        assert bench.tc_kernel_name(sh, s).startswith("attn_tc2_kernel") == bool(got["tc2"]), w.name
        got_rope = plan(harness, reqs, hq=sh.num_heads_q, hkv=sh.num_heads_kv, d=sh.head_dim, bs=sh.block_size,
                        seg=sh.kv_segment_size, rope=500000.0)
        assert bench.tc_kernel_name(sh, s, rope=True).startswith("attn_tc2_kernel") == bool(got_rope["tc2"])


@pytest.mark.parametrize("hq,hkv,want", [(32, 8, 128), (24, 8, 126), (28, 4, 126), (24, 4, 126), (20, 4, 125),
                                         (96, 8, 120), (128, 1, 128), (100, 1, 100)])
def test_query_tiles_hold_whole_tokens(harness, hq, hkv, want):
    # a tensor-core query tile is G * floor(128 / G) packed rows: whole tokens
    # only, for every query group up to 128; the two-pipeline kernel (which
    # pairs 128-row tiles) takes only groups that divide 128
    G = hq // hkv
    got = plan(harness, [(4096, 700), (100, 1)], hq=hq, hkv=hkv)
    assert got["tile_m"] == want == G * (128 // G)
    if 128 % G:
        assert got["tc2"] == 0


def test_two_cta_groups_for_chunks_over_a_cache(harness):
    """One-pipeline kernel, direct units only: 512 units on 152 CTAs leave a
    last wave of 56.  Chunks of 2048 query tokens over a cache (units of
    17-48 key tiles) pack better as 96 CTAs x 3 of the heaviest units and 56
    CTAs x 4 of the lightest, each group with its own counter."""
    for C in (2048, 4096, 6144):
        p = plan(harness, [(C, 2048)], bs=128)
        assert (p["tc2"], p["direct_units"]) == (0, 512)
        assert (p["group_ctas"], p["group_units"]) == (96, 288)
    # d 64, G 1: 384 units (q 2, R 80): 72 CTAs x 2 heaviest, 80 x 3 lightest
    p = plan(harness, [(2048, 2048)], hq=24, hkv=24, d=64, bs=128)
    assert (p["direct_units"], p["group_ctas"], p["group_units"]) == (384, 72, 144)
    # a prompt's first chunk (units of 1-16 tiles: the single counter already
    # balances them), whole waves, the two-pipeline kernel, split units, the
    # tail cut: one counter
    assert plan(harness, [(0, 2048)], bs=128)["group_ctas"] == 0
    assert plan(harness, [(8192, 1808)], bs=128)["group_ctas"] == 0
    assert plan(harness, [(4096, 2048)], bs=16)["tc2"] == 1
    assert plan(harness, [(4096, 2048)], bs=16)["group_ctas"] == 0
    assert plan(harness, [(4096, 2048), (9000, 1)], bs=128)["group_ctas"] == 0
    assert plan(harness, [(6144, 2048)], bs=128, flags=FUSE | 0x8)["group_ctas"] == 0
    # the second counter follows the others in the zeroed counter block
    one = plan(harness, [(0, 2048)], bs=128)
    two = plan(harness, [(2048, 2048)], bs=128)
    assert two["ws_bytes"] - two["sched_off"] == one["ws_bytes"] - one["sched_off"]
