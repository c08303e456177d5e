"""Pins for the oracle's rotary position embedding.

The pages place the active tokens of a chunk at absolute positions
num_computed_tokens + i ("Prefill Optimisation", section 2; "Chunked
Prefill"), which is where a rotary embedding rotates queries and keys.  The
rotary convention itself is the rotate-half form (pairs (c, c + d/2), angle
p * theta^(-2c/d)).  None of these pins compares the oracle with itself:
  * a rotation keeps every head vector's norm, and position 0 is the identity;
  * scores depend only on the distance between query and key positions;
  * the rotation equals multiplying the complex numbers x_c + i x_{c+d/2} by
    exp(i p theta^(-2c/d)) (numpy complex arithmetic, a separate statement
    of the same map);
  * chunked prefill with the rotation at absolute positions, through the
    paged cache holding rotated keys, equals one-shot causal attention over
    the rotated prompt (pure-Python fsum brute force);
  * each planted mistake (interleaved pairs, no position offset) fails one
    of these.
"""
import math

import numpy as np
import pytest

import oracle
import workloads as W

from test_oracle import brute_force

TOL = 1e-12
THETA = 10000.0


def rot(cached, new, q, k, *, d, theta=THETA, mutation=oracle.MUT_NONE):
    b = oracle.Batch([cached], [new], np.zeros((1, 1), dtype=np.int32))
    return oracle.rope(b, q, k, num_heads_q=q.shape[1], num_heads_kv=k.shape[1], head_dim=d, theta=theta,
                       mutation=mutation)


def test_rotation_keeps_norms_and_position_zero_is_identity():
    rng = np.random.default_rng(31)
    d = 16
    q = rng.standard_normal((9, 4, d))
    k = rng.standard_normal((9, 2, d))
    qr, kr = rot(0, 9, q, k, d=d)
    assert np.max(np.abs(np.linalg.norm(qr, axis=2) - np.linalg.norm(q, axis=2))) < TOL
    assert np.max(np.abs(np.linalg.norm(kr, axis=2) - np.linalg.norm(k, axis=2))) < TOL
    assert np.array_equal(qr[0], q[0]) and np.array_equal(kr[0], k[0])  # token 0 sits at position 0
    assert np.max(np.abs(qr[1:] - q[1:])) > 1e-3  # later positions do rotate


@pytest.mark.parametrize("shift", [1, 37, 4096])
def test_scores_depend_only_on_relative_position(shift):
    rng = np.random.default_rng(32)
    d, n = 8, 12
    q = rng.standard_normal((n, 1, d))
    k = rng.standard_normal((n, 1, d))
    qa, ka = rot(0, n, q, k, d=d)        # positions 0 .. n-1
    qb, kb = rot(shift, n, q, k, d=d)    # the same tokens at positions shift .. shift+n-1
    sa = qa[:, 0] @ ka[:, 0].T
    sb = qb[:, 0] @ kb[:, 0].T
    assert np.max(np.abs(sa - sb)) < 1e-9 * max(1.0, shift / 100)
    assert np.max(np.abs(qa - qb)) > 1e-3  # the vectors themselves did move


def complex_rotation(x, positions, d, theta):
    half = d // 2
    z = x[..., :half] + 1j * x[..., half:]
    freq = theta ** (-2.0 * np.arange(half) / d)
    w = np.exp(1j * positions[:, None, None] * freq[None, None, :])
    y = z * w
    return np.concatenate([y.real, y.imag], axis=-1)


@pytest.mark.parametrize("cached", [0, 5, 3000])
def test_matches_complex_multiplication(cached):
    rng = np.random.default_rng(33)
    d, n = 32, 7
    q = rng.standard_normal((n, 3, d))
    k = rng.standard_normal((n, 1, d))
    qr, kr = rot(cached, n, q, k, d=d, theta=500000.0)
    pos = np.arange(cached, cached + n, dtype=np.float64)
    assert np.max(np.abs(qr - complex_rotation(q, pos, d, 500000.0))) < 1e-9
    assert np.max(np.abs(kr - complex_rotation(k, pos, d, 500000.0))) < 1e-9


def chunked_with_rope(q, k, v, chunks, *, hq, hkv, d, bs, rng, mutation=oracle.MUT_NONE):
    """Chunked prefill through the paged cache, rotating each chunk's queries
    and keys at their absolute positions; the cache keeps rotated keys."""
    P = q.shape[0]
    need = W.cdiv(P, bs)
    num_blocks = need + 3
    bt = np.concatenate([rng.permutation(num_blocks)[:need], [0, 1]]).astype(np.int32)[None, :]
    kc = np.full((num_blocks, bs, hkv, d), np.nan)
    vc = np.full((num_blocks, bs, hkv, d), np.nan)
    outs = []
    done = 0
    for n in chunks:
        b = oracle.Batch([done], [n], bt)
        sl = slice(done, done + n)
        qr, kr = oracle.rope(b, q[sl], k[sl], num_heads_q=hq, num_heads_kv=hkv, head_dim=d, theta=THETA,
                             mutation=mutation)
        o, _ = oracle.attention(b, qr, kr, v[sl], kc, vc, num_heads_q=hq, num_heads_kv=hkv, head_dim=d,
                                block_size=bs, scale=1.0 / math.sqrt(d), threads=2)
        kc, vc = oracle.kv_write(b, kr, v[sl], kc, vc, num_heads_kv=hkv, head_dim=d, block_size=bs)
        outs.append(o)
        done += n
    return np.concatenate(outs)


def _rope_pins_pass(mutation=oracle.MUT_NONE) -> bool:
    rng = np.random.default_rng(34)
    hq, hkv, d, bs = 4, 2, 8, 4
    chunks = [6, 5, 8]
    P = sum(chunks)
    q = rng.standard_normal((P, hq, d))
    k = rng.standard_normal((P, hkv, d))
    v = rng.standard_normal((P, hkv, d))
    out = chunked_with_rope(q, k, v, chunks, hq=hq, hkv=hkv, d=d, bs=bs, rng=rng, mutation=mutation)
    pos = np.arange(P, dtype=np.float64)
    qr, kr = complex_rotation(q, pos, d, THETA), complex_rotation(k, pos, d, THETA)
    ref, _ = brute_force(qr, kr, v, hq, hkv, 1.0 / math.sqrt(d))
    ok = np.max(np.abs(out - ref)) < 1e-10
    # the rotation of a single chunk at an offset
    q2, k2 = rot(9, 4, q[:4], k[:4], d=d, mutation=mutation)
    p2 = np.arange(9, 13, dtype=np.float64)
    ok = ok and np.max(np.abs(q2 - complex_rotation(q[:4], p2, d, THETA))) < 1e-9
    return bool(ok)


def test_chunked_prefill_with_rope_equals_one_shot():
    assert _rope_pins_pass()


@pytest.mark.parametrize("mutation", [oracle.MUT_ROPE_INTERLEAVED, oracle.MUT_ROPE_NO_OFFSET])
def test_planted_rope_mistake_is_caught(mutation):
    assert not _rope_pins_pass(mutation)
