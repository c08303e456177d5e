"""Pins for the oracle's FP8 (E4M3) key/value cache.

The pages name FP8 E4M3 and its quantization scales as one of the things that
fix what cached KV means ("Prefill Optimisation", section 3, prefix caching:
the identity dimensions of reusable KV) and say nothing more, so the format is
the OCP FP8 E4M3 one (bias 7, subnormals m * 2^-9, S.1111.111 NaN, largest
finite 448) and the cache reading is: code = nearest E4M3 value of fl32(x / scale[kv head]), ties to an
even mantissa, saturated to +-448; a code stands for value * scale; attention
sees every key and value (the chunk's own included) through that encoding.
None of these pins compares the oracle with itself:
  * code values fixed by the format definition (closed forms);
  * every finite code decodes and re-encodes to itself;
  * for |y| < 448 the codes equal torch's float8_e4m3fn conversion (an
    independent implementation of the same rounding), ties included;
  * saturation and NaN;
  * the FP8 K/V write equals torch's codes slot by slot, other slots kept;
  * chunked prefill through an FP8 pool equals one-shot attention over the
    prompt quantized by torch (pure-Python fsum brute force), with different
    scales per kv head;
  * each planted mistake (truncating encoder, the chunk's own rows left
    unquantized, one scale for every head, a write one slot off) fails one.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W

from test_oracle import brute_force

MAX_E4M3 = 448.0


def torch_codes(y: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(y, dtype=np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def torch_dequant(x: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """x [..., H, d] through the cache format with per-head scales, by torch:
    fp32 quotient, clamp to the finite range, float8_e4m3fn, times scale."""
    s = np.asarray(scale, dtype=np.float32)[:, None]
    y = (x.astype(np.float32) / s).astype(np.float32)
    y = np.clip(y, -MAX_E4M3, MAX_E4M3)
    v = torch.from_numpy(y).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    return v * s.astype(np.float64)


def test_code_values_fixed_by_the_format():
    table = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x39: 1.125,
             0x3F: 1.875, 0x40: 2.0, 0x77: 240.0, 0x7E: 448.0, 0x80: -0.0, 0xB8: -1.0, 0xFE: -448.0}
    codes = np.array(sorted(table), dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    for c, v in zip(codes, vals):
        assert v == table[int(c)] and math.copysign(1, v) == math.copysign(1, table[int(c)]), hex(c)
    assert np.isnan(oracle.e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    assert np.all(np.diff(vals[(codes < 0x80)]) > 0)  # positive codes are increasing
    assert np.array_equal(oracle.e4m3_encode(vals.astype(np.float32)), codes)


def _in_range_samples():
    rng = np.random.default_rng(51)
    x = 2.0 ** rng.uniform(-14, 8.8, 100000) * rng.choice([-1.0, 1.0], 100000)
    vals = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2  # exact ties, all representable in fp32
    y = np.concatenate([x, mids, -mids]).astype(np.float32)
    return y[np.abs(y) < MAX_E4M3]


def test_encoder_matches_torch_float8_in_range():
    y = _in_range_samples()
    assert np.array_equal(oracle.e4m3_encode(y), torch_codes(y))


def test_ties_go_to_even_mantissa():
    y = np.array([1.0625, 1.1875, 2.0 ** -9 * 1.5, 2.0 ** -9 * 2.5, 0.5 * 2.0 ** -9], dtype=np.float32)
    assert list(oracle.e4m3_encode(y)) == [0x38, 0x3A, 0x02, 0x02, 0x00]


def test_saturation_and_nan():
    y = np.array([448.0, 460.0, 464.0, 480.0, 1e6, np.inf, -1e6, -np.inf, np.nan], dtype=np.float32)
    assert list(oracle.e4m3_encode(y)) == [0x7E] * 6 + [0xFE, 0xFE, 0x7F]


def test_truncating_encoder_is_caught():
    y = _in_range_samples()
    assert not np.array_equal(oracle.e4m3_encode(y, oracle.MUT_FP8_TRUNCATE), torch_codes(y))


def _write_case(seed=52):
    rng = np.random.default_rng(seed)
    hkv, d, bs = 2, 8, 4
    cached, new = [5, 0, 9], [3, 6, 1]
    nb = 16
    bt = rng.permutation(nb)[:12].astype(np.int32).reshape(3, 4)
    b = oracle.Batch(cached, new, bt)
    T = sum(new)
    kn = (rng.standard_normal((T, hkv, d)) * 3).astype(np.float32)
    vn = (rng.standard_normal((T, hkv, d)) * 3).astype(np.float32)
    ks = np.array([0.01, 0.05], dtype=np.float32)
    vs = np.array([0.02, 0.004], dtype=np.float32)
    kc = rng.integers(0, 256, (nb, bs, hkv, d)).astype(np.uint8)
    vc = rng.integers(0, 256, (nb, bs, hkv, d)).astype(np.uint8)
    return b, kn, vn, ks, vs, kc, vc, hkv, d, bs


def _fp8_write_matches(mutation=oracle.MUT_NONE) -> bool:
    b, kn, vn, ks, vs, kc, vc, hkv, d, bs = _write_case()
    ko, vo = oracle.kv_write(b, kn, vn, kc, vc, num_heads_kv=hkv, head_dim=d, block_size=bs, k_scale=ks,
                             v_scale=vs, mutation=mutation)
    ek, ev = kc.copy(), vc.copy()
    for r in range(b.num_reqs):
        for i in range(int(b.num_new_tokens[r])):
            pos = int(b.cached_seq_len[r]) + i
            blk, off = int(b.block_table[r, pos // bs]), pos % bs
            t = int(b.cu_new_tokens[r]) + i
            ek[blk, off] = torch_codes(np.clip(kn[t] / ks[:, None], -MAX_E4M3, MAX_E4M3))
            ev[blk, off] = torch_codes(np.clip(vn[t] / vs[:, None], -MAX_E4M3, MAX_E4M3))
    return bool(np.array_equal(ko, ek) and np.array_equal(vo, ev))


def test_fp8_write_matches_torch_codes_slot_by_slot():
    assert _fp8_write_matches()


@pytest.mark.parametrize("mutation", [oracle.MUT_WRITE_OFF_BY_ONE, oracle.MUT_FP8_HEAD0_SCALE,
                                      oracle.MUT_FP8_TRUNCATE])
def test_planted_write_mistake_is_caught(mutation):
    assert not _fp8_write_matches(mutation)


def _chunked_fp8_pins_pass(mutation=oracle.MUT_NONE) -> bool:
    rng = np.random.default_rng(53)
    hq, hkv, d, bs = 4, 2, 8, 4
    chunks = [6, 5, 8]
    P = sum(chunks)
    q = rng.standard_normal((P, hq, d)).astype(np.float32)
    k = (rng.standard_normal((P, hkv, d)) * 2).astype(np.float32)
    v = rng.standard_normal((P, hkv, d)).astype(np.float32)
    ks = np.array([0.004, 0.03], dtype=np.float32)  # head 0 fine-grained, head 1 coarse
    vs = np.array([0.02, 0.003], dtype=np.float32)
    need = W.cdiv(P, bs)
    nb = need + 3
    bt = np.concatenate([rng.permutation(nb)[:need], [0, 1]]).astype(np.int32)[None, :]
    kc = np.full((nb, bs, hkv, d), 0x7F, dtype=np.uint8)  # NaN codes in every unwritten slot
    vc = np.full((nb, bs, hkv, d), 0x7F, dtype=np.uint8)
    outs = []
    done = 0
    for n in chunks:
        b = oracle.Batch([done], [n], bt)
        sl = slice(done, done + n)
        o, _ = oracle.attention(b, q[sl], k[sl], v[sl], kc, vc, num_heads_q=hq, num_heads_kv=hkv, head_dim=d,
                                block_size=bs, scale=1.0 / math.sqrt(d), threads=2, k_scale=ks, v_scale=vs,
                                mutation=mutation)
        kc, vc = oracle.kv_write(b, k[sl], v[sl], kc, vc, num_heads_kv=hkv, head_dim=d, block_size=bs,
                                 k_scale=ks, v_scale=vs)
        outs.append(o)
        done += n
    out = np.concatenate(outs)
    ref, _ = brute_force(q.astype(np.float64), torch_dequant(k, ks), torch_dequant(v, vs), hq, hkv,
                         1.0 / math.sqrt(d))
    return bool(np.max(np.abs(out - ref)) < 1e-10)


def test_chunked_prefill_over_fp8_cache_equals_one_shot_over_quantized_prompt():
    assert _chunked_fp8_pins_pass()


@pytest.mark.parametrize("mutation", [oracle.MUT_FP8_NEW_UNQUANTIZED, oracle.MUT_FP8_HEAD0_SCALE])
def test_planted_fp8_attention_mistake_is_caught(mutation):
    assert not _chunked_fp8_pins_pass(mutation)
