"""Pins for the fp64 oracle, checked against what the pages and mathematics fix.

None of these compares the oracle with itself.  Each pin is one of:
  * a closed form (first token of a fresh prompt returns its own value row;
    zero queries give the mean of the visible value rows and lse = log of the
    number of visible keys; constant value rows; a one-hot score);
  * a pure-Python math.fsum brute force over the dense, unpaged prompt;
  * chunk invariance: chunked prefill through the paged cache equals one-shot
    causal attention over the full prompt ("Prefill Optimisation", section 2,
    Causal equivalence);
  * segment invariance: walking the cache in kv_segment_size pieces with the
    online merge equals the definition ("Prefill Processing", Kernel
    Interface; Partial KV Segment Handling);
  * prefix-hit equivalence: a request whose prefix sits in shared cached
    blocks gets the same suffix output as recomputing the prefix
    ("Prefill Processing", Prefix Caching);
  * planted mistakes: each known wrong variant of the oracle fails at least
    one of the pins above.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W

TOL = 1e-12


def bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_values(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()


def nan_pool(num_blocks, bs, hkv, d, dtype):
    if dtype == "f32":
        return np.full((num_blocks, bs, hkv, d), np.nan, dtype=np.float32)
    return np.full((num_blocks, bs, hkv, d), 0x7FC1, dtype=np.uint16)


def run_prompt(q, k, v, chunks, *, hq, hkv, d, bs, rng, num_blocks=None, segmented=False, seg=0,
               mutation=0, write_mutation=0, dtype="f32", extra_cols=2):
    """Process one prompt in the given chunks through the paged cache:
    attention of each chunk (cache + chunk), then the chunk's K/V write."""
    P = q.shape[0]
    need = W.cdiv(P, bs)
    num_blocks = num_blocks or need + 5
    bt = np.concatenate([rng.permutation(num_blocks)[:need], rng.integers(0, num_blocks, extra_cols)])
    bt = bt.astype(np.int32)[None, :]
    kc = nan_pool(num_blocks, bs, hkv, d, dtype)
    vc = nan_pool(num_blocks, bs, hkv, d, dtype)
    outs, lses = [], []
    done = 0
    for n in chunks:
        b = oracle.Batch([done], [n], bt)
        sl = slice(done, done + n)
        o, l = oracle.attention(b, q[sl], k[sl], v[sl], kc, vc, num_heads_q=hq, num_heads_kv=hkv,
                                head_dim=d, block_size=bs, scale=1.0 / math.sqrt(d),
                                segmented=segmented, kv_segment_size=seg, threads=4, mutation=mutation)
        kc, vc = oracle.kv_write(b, k[sl], v[sl], kc, vc, num_heads_kv=hkv, head_dim=d, block_size=bs,
                                 mutation=write_mutation)
        outs.append(o)
        lses.append(l)
        done += n
    return np.concatenate(outs), np.concatenate(lses), kc, vc, bt


def brute_force(q, k, v, hq, hkv, scale):
    """Dense causal attention over the whole prompt, pure Python, fsum."""
    P, _, d = q.shape
    G = hq // hkv
    out = np.zeros((P, hq, d))
    lse = np.zeros((P, hq))
    for p in range(P):
        for h in range(hq):
            g = h // G
            s = [scale * math.fsum(float(q[p, h, c]) * float(k[j, g, c]) for c in range(d)) for j in range(p + 1)]
            m = max(s)
            e = [math.exp(x - m) for x in s]
            z = math.fsum(e)
            for c in range(d):
                out[p, h, c] = math.fsum(e[j] * float(v[j, g, c]) for j in range(p + 1)) / z
            lse[p, h] = m + math.log(z)
    return out, lse


def rand_prompt(rng, P, hq, hkv, d):
    q = rng.standard_normal((P, hq, d)).astype(np.float32)
    k = rng.standard_normal((P, hkv, d)).astype(np.float32)
    v = rng.standard_normal((P, hkv, d)).astype(np.float32)
    return q, k, v


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_first_token_returns_its_value_row(dtype):
    rng = np.random.default_rng(1)
    hq, hkv, d, bs = 4, 2, 16, 4
    q, k, v = rand_prompt(rng, 9, hq, hkv, d)
    if dtype == "bf16":
        qb, kb, vb = bf16_bits(q), bf16_bits(k), bf16_bits(v)
        out, _, _, _, _ = run_prompt(qb, kb, vb, [9], hq=hq, hkv=hkv, d=d, bs=bs, rng=rng, dtype="bf16")
        vref = bf16_values(vb)  # decoded by torch, not by the oracle
    else:
        out, _, _, _, _ = run_prompt(q, k, v, [9], hq=hq, hkv=hkv, d=d, bs=bs, rng=rng)
        vref = v
    G = hq // hkv
    for h in range(hq):
        assert np.array_equal(out[0, h], vref[0, h // G].astype(np.float64))


def test_zero_queries_average_visible_values_and_lse_counts_keys():
    rng = np.random.default_rng(2)
    hq, hkv, d, bs = 4, 1, 8, 16
    P = 70
    _, k, v = rand_prompt(rng, P, hq, hkv, d)
    q = np.zeros((P, hq, d), dtype=np.float32)
    out, lse, *_ = run_prompt(q, k, v, [33, 20, 17], hq=hq, hkv=hkv, d=d, bs=bs, rng=rng)
    for p in range(P):
        mean = v[: p + 1, 0].astype(np.float64).mean(axis=0)
        for h in range(hq):
            assert np.allclose(out[p, h], mean, rtol=0, atol=1e-13)
            assert abs(lse[p, h] - math.log(p + 1)) < 1e-13


def test_constant_values_give_the_constant():
    rng = np.random.default_rng(3)
    hq, hkv, d, bs = 2, 2, 8, 8
    P = 40
    q, k, _ = rand_prompt(rng, P, hq, hkv, d)
    c = rng.standard_normal((hkv, d)).astype(np.float32)
    v = np.broadcast_to(c, (P, hkv, d)).copy()
    out, *_ = run_prompt(q, k, v, [16, 8, 16], hq=hq, hkv=hkv, d=d, bs=bs, rng=rng)
    for h in range(hq):
        assert np.allclose(out[:, h], c[h].astype(np.float64), rtol=0, atol=1e-13)


def test_one_hot_score_selects_that_key():
    # keys are basis vectors, the query of token p points at key j*(p) <= p
    rng = np.random.default_rng(4)
    P, d, hq, hkv, bs = 24, 32, 2, 1, 4
    k = np.zeros((P, hkv, d), dtype=np.float32)
    for j in range(P):
        k[j, 0, j] = 1.0
    v = rng.standard_normal((P, hkv, d)).astype(np.float32)
    target = np.array([rng.integers(0, p + 1) for p in range(P)])
    q = np.zeros((P, hq, d), dtype=np.float32)
    A = 60.0
    for p in range(P):
        q[p, :, target[p]] = A * math.sqrt(d)  # scaled score = A for the target key, 0 otherwise
    out, lse, *_ = run_prompt(q, k, v, [10, 7, 7], hq=hq, hkv=hkv, d=d, bs=bs, rng=rng)
    a_eff = float(np.float32(A * math.sqrt(d))) / math.sqrt(d)  # the query is stored in float32
    for p in range(P):
        for h in range(hq):
            assert np.allclose(out[p, h], v[target[p], 0], rtol=1e-20, atol=1e-20 + 1e-24 * p)
            assert abs(lse[p, h] - a_eff) < 1e-12


# ---------------------------------------------------------------------------
# brute force, chunk invariance, segments, prefix hits
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("hq,hkv,chunks", [(4, 2, [7, 5, 9, 1, 1, 3]), (3, 1, [26]), (2, 2, [1] * 6 + [20])])
def test_brute_force_dense_prompt(hq, hkv, chunks):
    rng = np.random.default_rng(5 + hq)
    d, bs = 6, 4
    P = sum(chunks)
    q, k, v = rand_prompt(rng, P, hq, hkv, d)
    out, lse, *_ = run_prompt(q, k, v, chunks, hq=hq, hkv=hkv, d=d, bs=bs, rng=rng)
    ref_o, ref_l = brute_force(q, k, v, hq, hkv, 1.0 / math.sqrt(d))
    assert np.max(np.abs(out - ref_o)) < TOL
    assert np.max(np.abs(lse - ref_l)) < TOL


def test_chunk_invariance_any_chunking():
    rng = np.random.default_rng(6)
    hq, hkv, d, bs = 8, 2, 16, 16
    P = 300
    q, k, v = rand_prompt(rng, P, hq, hkv, d)
    one, one_l, *_ = run_prompt(q, k, v, [P], hq=hq, hkv=hkv, d=d, bs=bs, rng=rng)
    for chunks in ([128, 128, 44], [100] * 3, [1] * 5 + [295], list(np.diff([0, 17, 64, 65, 200, 300]))):
        o, l, *_ = run_prompt(q, k, v, [int(c) for c in chunks], hq=hq, hkv=hkv, d=d, bs=bs, rng=rng)
        assert np.max(np.abs(o - one)) < TOL
        assert np.max(np.abs(l - one_l)) < TOL


def test_kv_write_places_each_token_in_its_slot_and_nothing_else():
    rng = np.random.default_rng(7)
    hq, hkv, d, bs = 2, 2, 4, 8
    P = 45
    q, k, v = rand_prompt(rng, P, hq, hkv, d)
    _, _, kc, vc, bt = run_prompt(q, k, v, [20, 13, 12], hq=hq, hkv=hkv, d=d, bs=bs, rng=rng)
    written = np.zeros(kc.shape[:2], dtype=bool)
    for j in range(P):
        blk, off = bt[0, j // bs], j % bs
        assert np.array_equal(kc[blk, off], k[j]) and np.array_equal(vc[blk, off], v[j])
        written[blk, off] = True
    assert np.all(np.isnan(kc[~written])) and np.all(np.isnan(vc[~written]))


def test_kv_write_is_a_byte_copy_for_bf16():
    rng = np.random.default_rng(8)
    hkv, d, bs = 2, 8, 16
    T = 21
    k = bf16_bits(rng.standard_normal((T, hkv, d)))
    v = bf16_bits(rng.standard_normal((T, hkv, d)))
    bt = np.array([[5, 2, 7, 1]], dtype=np.int32)
    b = oracle.Batch([9], [T], bt)
    kc = nan_pool(8, bs, hkv, d, "bf16")
    vc = nan_pool(8, bs, hkv, d, "bf16")
    kc2, vc2 = oracle.kv_write(b, k, v, kc, vc, num_heads_kv=hkv, head_dim=d, block_size=bs)
    for i in range(T):
        pos = 9 + i
        assert np.array_equal(kc2[bt[0, pos // bs], pos % bs], k[i])
        assert np.array_equal(vc2[bt[0, pos // bs], pos % bs], v[i])
    assert int((kc2 != kc).any(axis=(2, 3)).sum()) == T


@pytest.mark.parametrize("seg", [512, 1024, 2048, 4096, 0])
def test_segment_invariance_with_partial_segment(seg):
    # cached 3584 = 3 full 1024-segments + 512 valid ("Partial KV Segment Handling")
    rng = np.random.default_rng(9)
    hq, hkv, d, bs = 2, 1, 4, 128
    C, N = 3584, 5
    q, k, v = rand_prompt(rng, C + N, hq, hkv, d)
    _, _, kc, vc, bt = run_prompt(q[:C], k[:C], v[:C], [C], hq=hq, hkv=hkv, d=d, bs=bs, rng=rng,
                                  num_blocks=40, extra_cols=W.cdiv(C + N, bs) - W.cdiv(C, bs) + 1)
    b = oracle.Batch([C], [N], bt)
    kw = dict(num_heads_q=hq, num_heads_kv=hkv, head_dim=d, block_size=bs, scale=0.5, threads=4)
    ref_o, ref_l = oracle.attention(b, q[C:], k[C:], v[C:], kc, vc, **kw)
    o, l = oracle.attention(b, q[C:], k[C:], v[C:], kc, vc, segmented=True, kv_segment_size=seg, **kw)
    assert np.max(np.abs(o - ref_o)) < TOL and np.max(np.abs(l - ref_l)) < TOL


def test_prefix_hit_equals_recompute():
    rng = np.random.default_rng(10)
    hq, hkv, d, bs = 4, 2, 8, 16
    prefix, suffixes = 64, [9, 30, 17]
    q, k, v = rand_prompt(rng, prefix + max(suffixes), hq, hkv, d)
    # request A computes the prefix and leaves it in the cache
    _, _, kc, vc, bt = run_prompt(q[:prefix], k[:prefix], v[:prefix], [prefix], hq=hq, hkv=hkv, d=d,
                                  bs=bs, rng=rng, num_blocks=64)
    shared = bt[0, : prefix // bs]
    free = [b for b in range(64) if b not in set(shared.tolist())]
    rows, cached, new = [], [], []
    qs, ks, vs = [], [], []
    for i, n in enumerate(suffixes):
        own = free[i * 4:(i + 1) * 4]
        rows.append(np.concatenate([shared, own]))
        cached.append(prefix)
        new.append(n)
        # every request gets the same prompt, so the suffix tokens are identical
        qs.append(q[prefix:prefix + n])
        ks.append(k[prefix:prefix + n])
        vs.append(v[prefix:prefix + n])
    b = oracle.Batch(cached, new, np.array(rows, dtype=np.int32))
    o, l = oracle.attention(b, np.concatenate(qs), np.concatenate(ks), np.concatenate(vs), kc, vc,
                            num_heads_q=hq, num_heads_kv=hkv, head_dim=d, block_size=bs,
                            scale=1.0 / math.sqrt(d), threads=4)
    full_o, full_l, *_ = run_prompt(q, k, v, [prefix + max(suffixes)], hq=hq, hkv=hkv, d=d, bs=bs, rng=rng)
    off = 0
    for n in suffixes:
        assert np.max(np.abs(o[off:off + n] - full_o[prefix:prefix + n])) < TOL
        assert np.max(np.abs(l[off:off + n] - full_l[prefix:prefix + n])) < TOL
        off += n


def test_sampled_rows_match_full_evaluation():
    rng = np.random.default_rng(11)
    hq, hkv, d, bs = 4, 2, 8, 16
    reqs = [(37, 5), (0, 20), (100, 1), (16, 33)]
    w = W.make_batch_workload("t", W.Shape(hq, hkv, d, bs, 512, "f32"), reqs, seed=11)
    t = w.materialize("cpu")
    s = w.steps[0]
    b = oracle.Batch(s.cached_seq_len, s.num_new_tokens, w.block_table)
    q, kn, vn = t.step_inputs(s)
    kw = dict(num_heads_q=hq, num_heads_kv=hkv, head_dim=d, block_size=bs, scale=0.3, threads=3)
    full_o, full_l = oracle.attention(b, q.numpy(), kn.numpy(), vn.numpy(), t.k_cache.numpy(),
                                      t.v_cache.numpy(), **kw)
    rows = [58, 0, 25, 3, 40]
    o, l = oracle.attention(b, q.numpy(), kn.numpy(), vn.numpy(), t.k_cache.numpy(), t.v_cache.numpy(),
                            rows=rows, **kw)
    assert np.array_equal(o, full_o[rows]) and np.array_equal(l, full_l[rows])
    assert np.all(np.isfinite(full_o))  # NaN sentinels in unused slots never reach the output


# ---------------------------------------------------------------------------
# planted mistakes: every one must be caught by a pin above
# ---------------------------------------------------------------------------

def _pins_pass(mutation=0, write_mutation=0) -> bool:
    rng = np.random.default_rng(12)
    hq, hkv, d, bs = 4, 2, 6, 4
    chunks = [7, 5, 9]
    P = sum(chunks)
    q, k, v = rand_prompt(rng, P, hq, hkv, d)
    try:
        out, lse, kc, vc, bt = run_prompt(q, k, v, chunks, hq=hq, hkv=hkv, d=d, bs=bs, rng=rng,
                                          mutation=mutation, write_mutation=write_mutation)
    except RuntimeError:
        return False
    ref_o, ref_l = brute_force(q, k, v, hq, hkv, 1.0 / math.sqrt(d))
    ok = np.max(np.abs(out - ref_o)) < TOL and np.max(np.abs(lse - ref_l)) < TOL
    # segment invariance on the filled cache
    b = oracle.Batch([P - 2], [2], bt)
    kw = dict(num_heads_q=hq, num_heads_kv=hkv, head_dim=d, block_size=bs, scale=0.4, threads=2,
              mutation=mutation)
    o1, _ = oracle.attention(b, q[P - 2:], k[P - 2:], v[P - 2:], kc, vc, **kw)
    o2, _ = oracle.attention(b, q[P - 2:], k[P - 2:], v[P - 2:], kc, vc, segmented=True,
                             kv_segment_size=8, **kw)
    ok = ok and np.max(np.abs(o1 - o2)) < TOL
    return bool(ok)


def test_pins_pass_on_the_unmodified_oracle():
    assert _pins_pass()


@pytest.mark.parametrize("mutation", [oracle.MUT_DROP_DIAGONAL, oracle.MUT_GQA_MODULO,
                                      oracle.MUT_NO_POSITION_OFFSET, oracle.MUT_DROP_CACHED,
                                      oracle.MUT_NO_BLOCK_TABLE, oracle.MUT_NO_SCALE,
                                      oracle.MUT_MERGE_NO_RESCALE, oracle.MUT_SEES_NEXT_KEY])
def test_planted_attention_mistake_is_caught(mutation):
    assert not _pins_pass(mutation=mutation)


def test_planted_write_mistake_is_caught():
    assert not _pins_pass(write_mutation=oracle.MUT_WRITE_OFF_BY_ONE)
