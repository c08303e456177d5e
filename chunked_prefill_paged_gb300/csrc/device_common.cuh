// device_common.cuh -- device helpers shared by the kernels: work-unit
// decoding, the paged-slot lookup of an active token, the fused/standalone
// K/V scatter, and error recording.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "cpa_internal.h"

namespace cpa {

__device__ __forceinline__ void record_error(int *err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// Request owning packed token t: the last r with cu[r] <= t (requests with no
// tokens are skipped because cu[r] == cu[r + 1]).
__device__ __forceinline__ int request_of_token(const int32_t *cu, int num_reqs, int t) {
    int lo = 0, hi = num_reqs;  // answer in [lo, hi)
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (__ldg(cu + mid) <= t)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// A decoded work unit (see cpa_internal.h).
struct Unit {
    int r, g, qt, piece;  // piece < 0: direct unit
    int C, N, cu0;
    int row0, rows;       // packed rows [row0, row0 + rows) of the request (up to
                          // tiles_per_unit * tile_m rows)
    int k_begin, k_end;   // keys [k_begin, k_end) of this unit
    int tail;             // tail piece: index of its direct unit among the tail units, else -1
    long long ws_off;     // float offset of the unit's partial (split units, tail pieces)
};

// Decode unit index `unit`; every lane of the calling warp must take part and
// gets the same result.  Returns false for an index past the last unit.
__device__ __forceinline__ bool decode_unit(const AttnArgs &a, int unit, Unit &u) {
    const int lane = threadIdx.x & 31;
    bool split = unit >= a.num_direct_units;
    int target = split ? unit - a.num_direct_units : unit;
    int tail = -1, tail_piece = 0;
    if (a.tail_units > 0) {
        // the last tail_units direct units as tail_pieces pieces each, in their place
        const int first = a.num_direct_units - a.tail_units;
        const int pieces_end = first + a.tail_units * a.tail_pieces;
        if (unit >= first && unit < pieces_end) {
            tail = (unit - first) / a.tail_pieces;
            tail_piece = (unit - first) - tail * a.tail_pieces;
            split = false;
            target = first + tail;
        } else if (unit >= pieces_end) {
            split = true;
            target = unit - pieces_end;
        }
    }
    if (a.interleave && unit < a.interleave_span) {
        // direct (prefill) and split (decode) units spread evenly over the
        // first T indices, each kind in its own order: index k is direct when
        // floor((k + 1) D / T) > floor(k D / T); the remaining split units follow
        const long long D = a.num_direct_units, T = a.interleave_span;
        const long long before = (long long)unit * D / T, after = ((long long)unit + 1) * D / T;
        split = after == before;
        target = split ? (int)(unit - before) : (int)before;
    }
    int base = 0;
    long long base_ws = 0;
    for (int r0 = 0; r0 < a.num_reqs; r0 += 32) {
        const int r = r0 + lane;
        ReqWork w{0, 0, 0, 0};
        if (r < a.num_reqs) w = request_work(__ldg(a.cached + r), __ldg(a.nnew + r), a.G, a.hkv, a.d, a.tile_m,
                                             split_len_of(a, r), a.tiles_per_unit);
        const int cnt = split ? w.split_units : w.direct_units;
        const long long wsf = split ? w.ws_floats : 0;
        int inc = cnt;
        long long incw = wsf;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int t = __shfl_up_sync(0xffffffffu, inc, o);
            long long tw = __shfl_up_sync(0xffffffffu, incw, o);
            if (lane >= o) {
                inc += t;
                incw += tw;
            }
        }
        const bool hit = cnt > 0 && target >= base + inc - cnt && target < base + inc;
        const unsigned m = __ballot_sync(0xffffffffu, hit);
        if (m) {
            const int src = __ffs(m) - 1;
            const int rr = r0 + src;
            const int first = __shfl_sync(0xffffffffu, base + inc - cnt, src);
            const long long wsb = __shfl_sync(0xffffffffu, base_ws + incw - wsf, src);
            const int local = target - first;
            u.r = rr;
            u.C = __ldg(a.cached + rr);
            u.N = __ldg(a.nnew + rr);
            u.cu0 = __ldg(a.cu + rr);
            u.g = local % a.hkv;
            const int rows_total = u.N * a.G;
            if (!split) {
                // the request's i-th tile group of kv head g covers query tiles
                // [last - tiles_per_unit + 1, last] with last = n_qt - 1 -
                // i * tiles_per_unit: heaviest tiles first.  Kv head innermost
                // (local = i * hkv + g) spreads concurrent CTAs over all heads,
                // which balances causal chunks best; head-major (local = g *
                // groups + i) keeps concurrent CTAs on one or two heads' K/V,
                // which keeps the working set in L2 for long contexts.
                const int n_qt = cdiv(rows_total, a.tile_m);
                const int groups = cdiv(n_qt, a.tiles_per_unit);
                int i = local / a.hkv;
                if (a.head_major) {
                    u.g = local / groups;
                    i = local - u.g * groups;
                }
                const int last = n_qt - 1 - i * a.tiles_per_unit;
                const int first = max(0, last - a.tiles_per_unit + 1);
                u.qt = first;
                u.piece = -1;
                u.row0 = first * a.tile_m;
                u.rows = min((last + 1) * a.tile_m, rows_total) - u.row0;
                const int last_tok = (u.row0 + u.rows - 1) / a.G;
                u.k_begin = 0;
                u.k_end = u.C + last_tok + 1;
                u.tail = tail;
                u.ws_off = 0;
                if (tail >= 0) {
                    // key tiles [j0, j1) of the unit's n (the cached keys in
                    // tiles from key 0, then the new keys in tiles from key C)
                    const int nc = cdiv(u.C, kTcTileN);
                    const int n = nc + cdiv(u.k_end - u.C, kTcTileN);
                    const int j0 = tail_piece * n / a.tail_pieces, j1 = (tail_piece + 1) * n / a.tail_pieces;
                    u.piece = tail_piece;
                    u.k_begin = j0 < nc ? j0 * kTcTileN : u.C + (j0 - nc) * kTcTileN;
                    if (j1 < n) u.k_end = j1 < nc ? j1 * kTcTileN : u.C + (j1 - nc) * kTcTileN;
                    u.ws_off = a.tail_ws + ((long long)tail * a.tail_pieces + tail_piece) *
                                               partial_floats(a.tile_m, a.d);
                }
            } else {
                u.qt = 0;
                u.piece = local / a.hkv;
                u.row0 = 0;
                u.rows = rows_total;
                const int len = split_len_of(a, rr);
                u.k_begin = u.piece * len;
                u.k_end = min(u.k_begin + len, u.C + u.N);
                u.tail = -1;
                u.ws_off = wsb + (long long)local * partial_floats(rows_total, a.d);
            }
            return true;
        }
        base += __shfl_sync(0xffffffffu, inc, 31);
        base_ws += __shfl_sync(0xffffffffu, incw, 31);
    }
    return false;
}

// Physical pool row (slot) of absolute position `pos` of request r, or -1
// when the block id is outside [0, num_blocks) (recorded in *err).
__device__ __forceinline__ long long slot_of(const int32_t *bt, int max_blocks, int bs, int num_blocks, int r,
                                             int pos, int *err) {
    const int blk = __ldg(bt + (long long)r * max_blocks + pos / bs);
    if (blk < 0 || blk >= num_blocks) {
        record_error(err, kErrBadBlock);
        return -1;
    }
    return (long long)blk * bs + pos % bs;
}

// Scatter 16-byte pieces [begin, end) of the new K/V rows into the pool.
// Piece index = ((t * hkv + g) * pieces_per_head + p): consecutive threads
// copy consecutive 16 bytes of one token's row, so loads and stores are
// coalesced.  Active token t of request r lands on the slot of position
// cached[r] + (t - cu[r]).
__device__ __forceinline__ void scatter_new_kv(const int32_t *cached, const int32_t *cu, const int32_t *bt,
                                               int num_reqs, int max_blocks, int hkv, int bs, int num_blocks,
                                               int head_bytes, const void *k_new, const void *v_new,
                                               void *k_cache, void *v_cache, long long begin, long long end,
                                               int stride_start, int stride, int *err) {
    const int pieces_per_head = head_bytes >> 4;
    const long long per_token = (long long)hkv * pieces_per_head;
    for (long long i = begin + stride_start; i < end; i += stride) {
        const int t = (int)(i / per_token);
        const int rem = (int)(i - (long long)t * per_token);
        const int g = rem / pieces_per_head;
        const int p = rem - g * pieces_per_head;
        const int r = request_of_token(cu, num_reqs, t);
        const int pos = __ldg(cached + r) + (t - __ldg(cu + r));
        const long long slot = slot_of(bt, max_blocks, bs, num_blocks, r, pos, err);
        if (slot < 0) continue;
        const long long src = ((long long)t * hkv + g) * head_bytes + p * 16;
        const long long dst = (slot * hkv + g) * head_bytes + p * 16;
        const uint4 kv = __ldg(reinterpret_cast<const uint4 *>(static_cast<const char *>(k_new) + src));
        const uint4 vv = __ldg(reinterpret_cast<const uint4 *>(static_cast<const char *>(v_new) + src));
        *reinterpret_cast<uint4 *>(static_cast<char *>(k_cache) + dst) = kv;
        *reinterpret_cast<uint4 *>(static_cast<char *>(v_cache) + dst) = vv;
    }
}

// The K and V rows of new tokens [t0, t1) into their pool slots, by
// nthreads threads (index tid).  A token's row (all kv heads, row_bytes) is
// contiguous both in k_new / v_new and in its slot, so a thread copies fixed
// 16-byte columns of kBatch tokens at a time: the tokens' slots first (one
// block-table read per token, no per-piece index arithmetic), then all loads,
// then all stores.  kKWritten: k_new was written earlier in this launch (the
// rotated keys) and is read through the coherent path.
template <int kBatch, bool kKWritten>
__device__ __forceinline__ void write_token_rows(const int32_t *cached, const int32_t *cu, const int32_t *bt,
                                                 int num_reqs, int max_blocks, int bs, int num_blocks, int row_bytes,
                                                 const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                                                 int t0, int t1, int tid, int nthreads, int *err) {
    if (t0 >= t1) return;
    const int cols = row_bytes >> 4;
    const char *kn = static_cast<const char *>(k_new);
    const char *vn = static_cast<const char *>(v_new);
    char *kc = static_cast<char *>(k_cache);
    char *vc = static_cast<char *>(v_cache);
    int r = request_of_token(cu, num_reqs, t0);
    for (int t = t0; t < t1; t += kBatch) {
        long long src[kBatch], dst[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int tt = t + k;
            src[k] = 0;
            dst[k] = -1;
            if (tt < t1) {
                while (r + 1 < num_reqs && __ldg(cu + r + 1) <= tt) ++r;
                const int pos = __ldg(cached + r) + (tt - __ldg(cu + r));
                const long long slot = slot_of(bt, max_blocks, bs, num_blocks, r, pos, err);
                src[k] = (long long)tt * row_bytes;
                if (slot >= 0) dst[k] = slot * row_bytes;
            }
        }
        for (int c = tid; c < cols; c += nthreads) {
            uint4 kv[kBatch], vv[kBatch];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                if (dst[k] >= 0) {
                    const uint4 *ks = reinterpret_cast<const uint4 *>(kn + src[k]) + c;
                    kv[k] = kKWritten ? *ks : __ldg(ks);
                    vv[k] = __ldg(reinterpret_cast<const uint4 *>(vn + src[k]) + c);
                }
            }
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                if (dst[k] >= 0) {
                    reinterpret_cast<uint4 *>(kc + dst[k])[c] = kv[k];
                    reinterpret_cast<uint4 *>(vc + dst[k])[c] = vv[k];
                }
            }
        }
    }
}

// Share of the fused K/V write done by CTA `cta` of `ctas` (called by
// `nthreads` threads of the CTA, thread index `tid`).
__device__ __forceinline__ void fused_write_share(const AttnArgs &a, int cta, int ctas, int tid, int nthreads,
                                                  int elem_bytes) {
    const int head_bytes = a.d * elem_bytes;
    const long long total = (long long)a.total_tokens * a.hkv * (head_bytes >> 4);
    const long long per = (total + ctas - 1) / ctas;
    const long long b = (long long)cta * per;
    const long long e = b + per < total ? b + per : total;
    if (b >= e) return;
    scatter_new_kv(a.cached, a.cu, a.bt, a.num_reqs, a.max_blocks, a.hkv, a.bs, a.num_blocks, head_bytes,
                   a.k_new, a.v_new, a.k_cache, a.v_cache, b, e, tid, nthreads, a.err);
}

// Rotary embedding ("Prefill Optimisation", section 2; the chunk's tokens
// at their absolute positions, "Chunked Prefill"): pair (c, c + d/2) of a row
// at position pos turns by the angle pos * theta^(-2c/d).  frac is that rate
// in turns, theta^(-2c/d) / (2 pi), as a 64-bit binary fraction, so pos *
// frac modulo 2^64 is the angle reduced to one turn; its top 24 bits, as the
// exact float x in [0, 2) with angle = pi x, go to sincospif (whose own
// reduction is exact, so no large-argument path).
__device__ __forceinline__ void rope_cos_sin(int pos, unsigned long long frac, float &c, float &s) {
    const unsigned long long turn = (unsigned long long)pos * frac;  // wraps: modulo one turn
    const float x = (float)(unsigned)(turn >> 40) * (1.0f / 8388608.0f);  // 2 * turns, exact
    sincospif(x, &s, &c);
}

// (x0, x1) turned by the angle whose cosine and sine are (c, s), in fp32 with
// a fixed rounding order, so every kernel that rotates a row gets the same bits
__device__ __forceinline__ void rope_turn(float x0, float x1, float c, float s, float &y0, float &y1) {
    y0 = __fmaf_rn(x0, c, -__fmul_rn(x1, s));
    y1 = __fmaf_rn(x1, c, __fmul_rn(x0, s));
}

__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ float from_float<float>(float x) {
    return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

}  // namespace cpa
