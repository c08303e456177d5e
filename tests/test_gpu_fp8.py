"""GPU parity for the FP8 (E4M3) key/value cache against the fp64 oracle.

The cache reading ("Prefill Optimisation", section 3, prefix caching: the KV
data type and its quantization scales): a pool element is the E4M3 code of
fl32(x / scale) for its kv head, a code stands for value * scale, and
attention sees every key and value -- the chunk's own rows too -- through
that encoding.  Checked:
  * the K/V write (standalone and fused) against the oracle's codes,
    bit-exact, other slots untouched;
  * attention outputs and LSE within the BF16 bounds over mixed batches,
    chunked prompts, the full mixed step (sampled rows) and with RoPE;
  * the code expansion itself is exact: every finite code read through the
    value path reproduces its value bit-exactly, and through the key path its
    log-sum-exp to fp32 precision, from the pool and from the new rows.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import BF16_ATOL, BF16_LSE_ATOL, Result, assert_within, params_for, sample_rows, to_oracle

pytestmark = pytest.mark.gpu

THETA = 500000.0


@pytest.fixture(scope="module")
def cpa():
    import chunked_prefill_paged_gb300 as m
    m.load()
    return m


def fp8_params(cpa, w, flags=None, rope_theta=0.0, scales=None):
    p = params_for(w, flags)
    ks, vs = scales if scales is not None else W.fp8_scales(w.shape.num_heads_kv)
    p.kv_format = cpa.KV_FP8_E4M3
    p.k_scale = torch.as_tensor(ks, device="cuda")
    p.v_scale = torch.as_tensor(vs, device="cuda")
    p.rope_theta = rope_theta
    return p, ks, vs


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def run_fp8(cpa, w, *, flags=None, rope_theta=0.0, rows_per_req=None, rows=None, check_pool=True, threads=None):
    """Every step of `w` over FP8 pools (fused write unless flags say
    otherwise, then the standalone write), against the oracle."""
    sh = w.shape
    t = w.materialize("cuda")
    p, ks, vs = fp8_params(cpa, w, flags, rope_theta)
    k8 = W.fp8_pool_codes(t.k_cache, ks)
    v8 = W.fp8_pool_codes(t.v_cache, vs)
    del t.k_cache, t.v_cache
    k_pool_o, v_pool_o = k8.cpu().numpy(), v8.cpu().numpy()
    fused = bool(p.flags & cpa.FLAG_FUSE_KV_WRITE)
    res = Result()
    for si, s in enumerate(w.steps):
        b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
        q, kn, vn = t.step_inputs(s)
        out, lse = cpa.attention(b, p, q, kn, vn, k8, v8)
        if not fused:
            cpa.paged_kv_write(b, p, kn, vn, k8, v8)
        torch.cuda.synchronize()
        ob = oracle.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
        if rope_theta > 0:
            qr, kr = oracle.rope(ob, as_f64(q), as_f64(kn), num_heads_q=sh.num_heads_q,
                                 num_heads_kv=sh.num_heads_kv, head_dim=sh.head_dim, theta=rope_theta)
            # the library stores rotated rows in the element type before encoding them
            bf = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).to(torch.float64).numpy()
            qo, kno = bf(qr), bf(kr)
        else:
            qo, kno = to_oracle(q), to_oracle(kn)
        vno = to_oracle(vn) if rope_theta == 0 else as_f64(vn)
        if s.total_new_tokens > 0:
            rs = rows if rows is not None else (None if rows_per_req is None else sample_rows(s, rows_per_req, si))
            ref_o, ref_l = oracle.attention(ob, qo, kno, vno, k_pool_o, v_pool_o, num_heads_q=sh.num_heads_q,
                                            num_heads_kv=sh.num_heads_kv, head_dim=sh.head_dim,
                                            block_size=sh.block_size, scale=sh.scale, rows=rs, threads=threads,
                                            k_scale=ks, v_scale=vs)
            idx = slice(None) if rs is None else torch.as_tensor(rs, device=out.device)
            res.add(out[idx].float().cpu().numpy(), ref_o, lse[idx].cpu().numpy(), ref_l)
        k_pool_o, v_pool_o = oracle.kv_write(ob, kno, vno, k_pool_o, v_pool_o, num_heads_kv=sh.num_heads_kv,
                                             head_dim=sh.head_dim, block_size=sh.block_size, k_scale=ks, v_scale=vs)
    if check_pool:
        k_gpu, v_gpu = k8.cpu().numpy(), v8.cpu().numpy()
        if rope_theta == 0:
            assert np.array_equal(k_gpu, k_pool_o), "K codes differ from the oracle's write"
        else:
            # a rotated bf16 key may sit one rounding step from the fp64 rotation
            # rounded to bf16, so its code may be one step away; elsewhere equal
            dk = np.abs(oracle.e4m3_decode(k_gpu) - oracle.e4m3_decode(k_pool_o))
            step = np.maximum(np.abs(oracle.e4m3_decode(k_pool_o)) * 2.0 ** -3, 2.0 ** -9)
            same = (k_gpu == k_pool_o) | (dk <= step)
            assert np.all(same), "K codes differ from the oracle's write by more than one step"
            assert np.mean(k_gpu == k_pool_o) > 0.999
        assert np.array_equal(v_gpu, v_pool_o), "V codes differ from the oracle's write"
    assert cpa.last_device_error() == cpa.SUCCESS
    return res


REQS = [(0, 300), (130, 77), (1000, 1), (17, 1), (257, 129), (5, 3), (3000, 1), (2048, 256)]


@pytest.mark.parametrize("bs", [16, 128])
def test_fp8_small_batch_fused_write(cpa, bs):
    w = W.make_batch_workload(f"fp8_{bs}", W.Shape(16, 4, 128, bs, 512, "bf16"), REQS, seed=61)
    res = run_fp8(cpa, w)
    assert_within(res, "bf16")


@pytest.mark.parametrize("flags", ["standalone_write", "no_split"])
def test_fp8_small_batch_variants(cpa, flags):
    w = W.make_batch_workload("fp8_var", W.Shape(32, 8, 128, 16, 1024, "bf16"), REQS, seed=62)
    fl = 0 if flags == "standalone_write" else (cpa.FLAG_FUSE_KV_WRITE | cpa.FLAG_NO_SPLIT)
    res = run_fp8(cpa, w, flags=fl)
    assert_within(res, "bf16")


def test_fp8_chunked_prompt_matches_oracle(cpa):
    w = W.make_prompt_workload("fp8_prompt", W.Shape(32, 8, 128, 16, 1024, "bf16"), 1000, 384, 80, seed=63)
    res = run_fp8(cpa, w)
    assert_within(res, "bf16")


def test_fp8_mixed_step_sampled(cpa):
    # the mixed decode/prefill step at full size; sampled rows of every request
    w = W.mixed_step()
    res = run_fp8(cpa, w, rows_per_req=2, check_pool=False)
    assert_within(res, "bf16")


def test_fp8_with_rope(cpa):
    w = W.make_batch_workload("fp8_rope", W.Shape(16, 4, 128, 16, 512, "bf16"), REQS[:6], seed=64)
    res = run_fp8(cpa, w, rope_theta=THETA)
    assert_within(res, "bf16")


def test_fp8_rope_standalone_write(cpa):
    w = W.make_prompt_workload("fp8_rope_prompt", W.Shape(8, 2, 128, 16, 512, "bf16"), 700, 300, 64, seed=65)
    res = run_fp8(cpa, w, flags=0, rope_theta=THETA)
    assert_within(res, "bf16")


def test_fp8_unsupported_shapes_are_refused(cpa):
    w = W.make_batch_workload("fp8_d64", W.Shape(4, 1, 64, 16, 512, "bf16"), [(0, 5)], seed=66)
    t = w.materialize("cuda")
    s = w.steps[0]
    p, ks, vs = fp8_params(cpa, w)
    b = cpa.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    q, kn, vn = t.step_inputs(s)
    k8 = torch.zeros(t.k_cache.shape, dtype=torch.uint8, device="cuda")
    v8 = torch.zeros_like(k8)
    with pytest.raises(cpa.CpaError) as e:
        cpa.attention(b, p, q, kn, vn, k8, v8)
    assert e.value.status == cpa.ERR_UNSUPPORTED
    # the write alone is supported at d = 64
    cpa.paged_kv_write(b, p, kn, vn, k8, v8)
    torch.cuda.synchronize()
    ob = oracle.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    ko, vo = oracle.kv_write(ob, to_oracle(kn), to_oracle(vn), np.zeros(k8.shape, np.uint8),
                             np.zeros(v8.shape, np.uint8), num_heads_kv=1, head_dim=64, block_size=16,
                             k_scale=ks, v_scale=vs)
    assert np.array_equal(k8.cpu().numpy(), ko) and np.array_equal(v8.cpu().numpy(), vo)


# ---------------------------------------------------------------- exactness

FINITE_CODES = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)


class Probe:
    """A hand-built batch with one kv head and scales 1: H_q query heads of
    d = 128, block size 16, request r on blocks 4r .. 4r + 3."""

    def __init__(self, cpa, reqs, hq):
        self.cpa = cpa
        self.hq, self.d, self.bs = hq, 128, 16
        self.cached = np.array([c for c, _ in reqs], np.int32)
        self.new = np.array([n for _, n in reqs], np.int32)
        self.nr = len(reqs)
        self.bt = np.arange(4 * self.nr, dtype=np.int32).reshape(self.nr, 4)
        self.T = int(self.new.sum())
        self.cu = np.concatenate([[0], np.cumsum(self.new)]).astype(np.int64)
        self.q = torch.zeros((self.T, hq, 128), dtype=torch.bfloat16)
        self.k = torch.zeros((self.T, 1, 128), dtype=torch.bfloat16)
        self.v = torch.zeros((self.T, 1, 128), dtype=torch.bfloat16)
        self.k8 = torch.zeros((4 * self.nr, 16, 1, 128), dtype=torch.uint8)
        self.v8 = torch.zeros_like(self.k8)

    def run(self):
        cpa = self.cpa
        p = cpa.Params(self.hq, 1, 128, 16, 4 * self.nr, 512, 1.0, cpa.DTYPE_BF16, cpa.FLAG_FUSE_KV_WRITE)
        p.kv_format = cpa.KV_FP8_E4M3
        p.k_scale = torch.ones(1, dtype=torch.float32, device="cuda")
        p.v_scale = torch.ones(1, dtype=torch.float32, device="cuda")
        b = cpa.Batch(self.cached, self.new, self.bt)
        out, lse = cpa.attention(b, p, self.q.cuda(), self.k.cuda(), self.v.cuda(), self.k8.cuda(), self.v8.cuda())
        torch.cuda.synchronize()
        assert cpa.last_device_error() == cpa.SUCCESS
        return out.cpu(), lse.cpu()


def code_values_bf16(codes: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(oracle.e4m3_decode(codes)).to(torch.bfloat16)  # every E4M3 value is a bf16 value


def test_every_code_reads_back_exactly_through_the_value_path(cpa):
    # requests 0, 1: one new token whose value row holds 128 codes (the output
    # of a lone key is its value); requests 2, 3: the same codes in the pool,
    # the new token's own key scored 448 below the cached one, so its weight
    # underflows to 0 and the output is the cached value row
    chunks = [FINITE_CODES[:128], np.concatenate([FINITE_CODES[128:], np.zeros(2, np.uint8)])]
    pr = Probe(cpa, [(0, 1), (0, 1), (1, 1), (1, 1)], hq=1)
    for r, codes in enumerate(chunks):
        pr.v[r, 0] = code_values_bf16(codes)
        blk = pr.bt[2 + r, 0]
        pr.v8[blk, 0, 0] = torch.from_numpy(codes)
        pr.k8[blk, 0, 0, 0] = 0x7E  # key value 448 at dimension 0
        pr.q[2 + r, 0, 0] = 1.0
    out, _ = pr.run()
    for r, codes in enumerate(chunks):
        # equal as numbers, so every bit of a nonzero value (the padding keys'
        # +0 products turn the code -0 into +0, as IEEE addition does)
        want = code_values_bf16(codes)
        assert torch.equal(out[r, 0], want), f"new-row values, chunk {r}"
        assert torch.equal(out[2 + r, 0], want), f"pooled values, chunk {r}"


def test_every_code_scores_exactly_through_the_key_path(cpa):
    # query head h of the probing token is the unit vector e_h; key 0 carries
    # code c_h at dimension h, the probing token's own key is zero, so
    # lse = log(exp(value(c_h)) + 1).  New-row keys: requests (0, 2), the
    # second token probes.  Pooled keys: requests (1, 1).
    hq = 8
    groups = [FINITE_CODES[i:i + hq] for i in range(0, len(FINITE_CODES), hq)]
    groups[-1] = np.concatenate([groups[-1], np.zeros(hq - len(groups[-1]), np.uint8)])
    n = len(groups)
    pr = Probe(cpa, [(0, 2)] * n + [(1, 1)] * n, hq=hq)
    for g, codes in enumerate(groups):
        t_new = int(pr.cu[g])            # key 0 of request g (new row); token t_new + 1 probes
        pr.k[t_new, 0, :hq] = code_values_bf16(codes)
        blk = pr.bt[n + g, 0]
        pr.k8[blk, 0, 0, :hq] = torch.from_numpy(codes)
        t_pool = int(pr.cu[n + g])        # the probing token of the pooled request
        for h in range(hq):
            pr.q[t_new + 1, h, h] = 1.0
            pr.q[t_pool, h, h] = 1.0
    _, lse = pr.run()
    for g, codes in enumerate(groups):
        vals = oracle.e4m3_decode(codes)
        want = np.logaddexp(vals, 0.0)
        for name, tok in (("new", int(pr.cu[g]) + 1), ("pooled", int(pr.cu[n + g]))):
            got = lse[tok].numpy().astype(np.float64)
            err = np.abs(got - want)
            assert np.all(err <= 2e-6 * np.maximum(1.0, np.abs(want))), (name, codes, got, want)


@pytest.mark.parametrize("bs,hq,hkv", [(32, 16, 4), (64, 64, 8), (16, 28, 4)])
def test_fp8_other_block_sizes_and_groups(cpa, bs, hq, hkv):
    # block sizes 32 / 64 (several code boxes per key tile), G = 8 query heads
    # per kv head (the long-context shape) and G = 7 (126-row query tiles)
    w = W.make_batch_workload(f"fp8_b{bs}_{hq}", W.Shape(hq, hkv, 128, bs, 1024, "bf16"),
                              [(0, 150), (2000, 1), (513, 64), (4096, 1)], seed=67)
    res = run_fp8(cpa, w)
    assert_within(res, "bf16")


def test_fp8_speculative_decode_queries(cpa):
    # multi-token decode queries (1 + draft tokens) over long FP8 contexts:
    # short causal chunks on the split path
    w = W.make_batch_workload("fp8_spec", W.Shape(32, 8, 128, 16, 1024, "bf16"),
                              [(3000, 5), (9000, 5), (17, 5), (12345, 3)], seed=68)
    res = run_fp8(cpa, w)
    assert_within(res, "bf16")


def test_fp8_tail_pieces(cpa):
    # a prefill chunk whose last query tiles are cut into tail pieces (see
    # test_gpu_tail.py): every row of the cut tiles, over FP8 pools
    w = W.make_batch_workload("fp8_tail", W.Shape(32, 8, 128, 128, 1024, "bf16"), [(6144, 2048)], seed=69)
    b = cpa.Batch(w.steps[0].cached_seq_len, w.steps[0].num_new_tokens, w.block_table)
    p, _, _ = fp8_params(cpa, w, flags=cpa.FLAG_FUSE_KV_WRITE | cpa.FLAG_TAIL_SPLIT)
    p_none, _, _ = fp8_params(cpa, w)
    assert cpa.workspace_size(b, p) > cpa.workspace_size(b, p_none), "no tail cut planned"
    res = run_fp8(cpa, w, flags=cpa.FLAG_FUSE_KV_WRITE | cpa.FLAG_TAIL_SPLIT, rows=list(range(0, 256)) + [1000, 2047])
    assert_within(res, "bf16")
