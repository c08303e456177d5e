// kernels_basic.cu -- the standalone paged K/V write, the CUDA-core
// attention kernel (FP32 path, and a BF16 cross-check), and the merge of
// split-KV partials.
//
// Attention semantics ("Prefill Processing", Key Concepts and Kernel
// Interface; "Prefill Optimisation", section 2): packed row (token t, query
// head h) of request r sees keys j <= cached_seq_len[r] + (t - cu[r]); keys
// below cached_seq_len come from the pool through the block table, the rest
// from the request's new K/V rows.  The running maximum / sum / output are
// carried across key tiles (online softmax), in the log2 domain: scores are
// multiplied by scale * log2(e) and exponentiated with exp2.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_common.cuh"
#include "launch.h"

namespace cpa {

// ------------------------------------------------------------------ KV write
__global__ void __launch_bounds__(256) kv_write_kernel(KvWriteArgs a) {
    const long long total = (long long)a.total_tokens * a.hkv * (a.head_bytes >> 4);
    const int stride = gridDim.x * blockDim.x;
    scatter_new_kv(a.cached, a.cu, a.bt, a.num_reqs, a.max_blocks, a.hkv, a.bs, a.num_blocks, a.head_bytes,
                   a.k_new, a.v_new, a.k_cache, a.v_cache, 0, total, blockIdx.x * blockDim.x + threadIdx.x,
                   stride, a.err);
}

cudaError_t launch_kv_write(const KvWriteArgs &a, int num_sms, cudaStream_t stream) {
    const long long total = (long long)a.total_tokens * a.hkv * (a.head_bytes >> 4);
    if (total == 0) return cudaSuccess;
    long long blocks = (total + 255) / 256;
    const long long cap = (long long)num_sms * 8;
    if (blocks > cap) blocks = cap;
    kv_write_kernel<<<(int)blocks, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

// ------------------------------------------------ rotary / FP8 pre-pass
// rope_kernel (FP8 pools, fp32 elements): one warp per (active token, group
// of kHeadsPerWarp heads; query heads first, then key heads; query heads only
// when rotated queries are wanted).  16-bit rotation alone: rope_rows_kernel
// below.
//
// Rotation: the angle of pair c is reduced to one turn exactly in integer
// arithmetic: turn_frac[c] holds theta^(-2c/d) / (2 pi) as a 64-bit binary
// fraction, so pos * turn_frac[c] modulo 2^64 (a wrapping 64-bit product) is
// the fraction of a turn; its top 24 bits give the angle in [0, 2 pi), whose
// cosine and sine are taken in fp32.  The rotation runs in fp32 and is
// rounded to the element type.
//
// FP8 cache: each key (after rotation, as the element type) and value
// element x of kv head g becomes the E4M3 code of fl32(x / scale[g]) --
// correctly rounded division, then the hardware conversion, round to
// nearest even with saturation to +-448.  The attention over FP8 pools runs
// its score MMAs on E4M3 operands, so each query row (after rotation, as the
// element type) is scaled by 2^e, e chosen so that the row's largest
// magnitude lands in [2^7, 2^8) (below the E4M3 maximum 448), and written as
// two E4M3 planes: a = E4M3(y) and b = E4M3(y - a), y the scaled element
// (y - a is exact in fp32).  a + b is within 2^-8 |y| of y (plus 2^-10 near
// the bottom of the range, 2^-18 of the row's maximum), about the precision
// of bf16; 2^-e goes to q_rscale for the softmax to undo.
//
// Lane l owns pairs c = 2l, 2l + 1 (d = 128) or c = l (d = 64), so the warp's
// accesses to each half row are contiguous.
constexpr int kHeadsPerWarp = 8;

// PPL consecutive elements of a lane moved as one access
template <int BYTES> struct LaneVec;
template <> struct LaneVec<1> { using type = unsigned char; };
template <> struct LaneVec<2> { using type = unsigned short; };
template <> struct LaneVec<4> { using type = unsigned int; };
template <> struct LaneVec<8> { using type = uint2; };

__device__ __forceinline__ uint8_t e4m3_code(float x, float scale) {
    return (uint8_t)__nv_cvt_float_to_fp8(__fdiv_rn(x, scale), __NV_SATFINITE, __NV_E4M3);
}

// y as two E4M3 codes: a = E4M3(y), b = E4M3(y - value(a)) (nearest even,
// saturating; y - value(a) is exact in fp32)
__device__ __forceinline__ void e4m3_split(float y, uint8_t &a, uint8_t &b) {
    a = (uint8_t)__nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3);
    const float va = __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)a, __NV_E4M3)));
    b = (uint8_t)__nv_cvt_float_to_fp8(y - va, __NV_SATFINITE, __NV_E4M3);
}

// the PPL codes of a lane's elements, packed as they lie in memory
template <int PPL, typename T>
__device__ __forceinline__ typename LaneVec<PPL>::type e4m3_lane(const T (&e)[PPL], float scale) {
    union {
        typename LaneVec<PPL>::type v;
        uint8_t b[PPL];
    } c;
#pragma unroll
    for (int i = 0; i < PPL; ++i) c.b[i] = e4m3_code(to_float(e[i]), scale);
    return c.v;
}

template <int D, typename T>
__global__ void __launch_bounds__(256) rope_kernel(RopeArgs a) {
    constexpr int PPL = D / 64;   // pairs per lane
    constexpr int HALF = D / 2;
    __shared__ unsigned long long frac_s[HALF];
    for (int c = threadIdx.x; c < HALF; c += blockDim.x) frac_s[c] = a.turn_frac[c];
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int head_lo = (a.q_rot || a.q8) ? 0 : a.hq;  // key heads only unless queries are written
    const int heads = a.hq + a.hkv;
    const int groups = (heads - head_lo + kHeadsPerWarp - 1) / kHeadsPerWarp;
    const long long wid = blockIdx.x * (long long)(blockDim.x >> 5) + (threadIdx.x >> 5);
    if (wid >= (long long)a.total_tokens * groups) return;
    const int t = (int)(wid / groups), grp = (int)(wid % groups);
    const int r = request_of_token(a.cu, a.num_reqs, t);
    const int pos = __ldg(a.cached + r) + (t - __ldg(a.cu + r));
    float cs[PPL], sn[PPL];
#pragma unroll
    for (int e = 0; e < PPL; ++e) {
        cs[e] = 1.f;
        sn[e] = 0.f;
        if (a.rotate) rope_cos_sin(pos, frac_s[lane * PPL + e], cs[e], sn[e]);
    }
    long long slot = -1;
    if (a.write_pool) slot = slot_of(a.bt, a.max_blocks, a.bs, a.num_blocks, r, pos, a.err);
    using V = typename LaneVec<PPL * (int)sizeof(T)>::type;
    using C8 = typename LaneVec<PPL>::type;
    union Lane {
        V v;
        T e[PPL];
    };
    const int h_begin = head_lo + grp * kHeadsPerWarp;
    const int h_end = min(heads, h_begin + kHeadsPerWarp);
    // every head's elements (and value chunk) are loaded before any is
    // written: one round of memory latency per warp instead of one per head
    Lane xls[kHeadsPerWarp], xhs[kHeadsPerWarp];
    uint4 vvs[kHeadsPerWarp];
    const bool copy_v = a.write_pool && !a.kv_fp8 && lane < D * (int)sizeof(T) / 16;
#pragma unroll
    for (int i = 0; i < kHeadsPerWarp; ++i) {
        const int head = h_begin + i;
        if (head < h_end) {
            const bool is_q = head < a.hq;
            const int hh = is_q ? head : head - a.hq;
            const long long row = ((long long)t * (is_q ? a.hq : a.hkv) + hh) * D;
            const T *src = static_cast<const T *>(is_q ? a.q : a.k_new) + row + lane * PPL;
            xls[i].v = __ldg(reinterpret_cast<const V *>(src));
            xhs[i].v = __ldg(reinterpret_cast<const V *>(src + HALF));
            if (!is_q && copy_v) vvs[i] = __ldg(reinterpret_cast<const uint4 *>(static_cast<const T *>(a.v_new) + row) + lane);
        }
    }
#pragma unroll
    for (int i = 0; i < kHeadsPerWarp; ++i) {
        const int head = h_begin + i;
        if (head >= h_end) break;
        const bool is_q = head < a.hq;
        const int hh = is_q ? head : head - a.hq;
        const long long row = ((long long)t * (is_q ? a.hq : a.hkv) + hh) * D;
        Lane xl = xls[i], xh = xhs[i];
        if (a.rotate) {
#pragma unroll
            for (int e = 0; e < PPL; ++e) {
                float y0, y1;
                rope_turn(to_float(xl.e[e]), to_float(xh.e[e]), cs[e], sn[e], y0, y1);
                xl.e[e] = from_float<T>(y0);
                xh.e[e] = from_float<T>(y1);
            }
        }
        if (is_q && a.q8) {
            // two E4M3 planes of the row scaled by 2^e (see above)
            float amax = 0.f;
#pragma unroll
            for (int e = 0; e < PPL; ++e) amax = fmaxf(amax, fmaxf(fabsf(to_float(xl.e[e])), fabsf(to_float(xh.e[e]))));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            int ex = 0;
            if (amax > 0.f) frexpf(amax, &ex);  // amax in [2^(ex-1), 2^ex)
            const int e = max(-100, min(100, amax > 0.f ? 8 - ex : 0));
            const float up = __int_as_float((127 + e) << 23), down = __int_as_float((127 - e) << 23);
            union Codes {
                C8 v;
                uint8_t b[PPL];
            } pa_lo, pa_hi, pb_lo, pb_hi;
#pragma unroll
            for (int e2 = 0; e2 < PPL; ++e2) {
                e4m3_split(to_float(xl.e[e2]) * up, pa_lo.b[e2], pb_lo.b[e2]);
                e4m3_split(to_float(xh.e[e2]) * up, pa_hi.b[e2], pb_hi.b[e2]);
            }
            uint8_t *dst = static_cast<uint8_t *>(a.q8) + row;
            const long long plane = (long long)a.total_tokens * a.hq * D;
            *reinterpret_cast<C8 *>(dst + lane * PPL) = pa_lo.v;
            *reinterpret_cast<C8 *>(dst + HALF + lane * PPL) = pa_hi.v;
            *reinterpret_cast<C8 *>(dst + plane + lane * PPL) = pb_lo.v;
            *reinterpret_cast<C8 *>(dst + plane + HALF + lane * PPL) = pb_hi.v;
            if (lane == 0) a.q_rscale[(long long)t * a.hq + hh] = down;
            continue;
        }
        if (is_q) {
            T *dst = static_cast<T *>(a.q_rot) + row;
            *reinterpret_cast<V *>(dst + lane * PPL) = xl.v;
            *reinterpret_cast<V *>(dst + HALF + lane * PPL) = xh.v;
            continue;
        }
        const long long prow = slot >= 0 ? (slot * a.hkv + hh) * D : -1;  // pool row of this head
        if (!a.kv_fp8) {
            if (a.k_rot) {
                T *dst = static_cast<T *>(a.k_rot) + row;
                *reinterpret_cast<V *>(dst + lane * PPL) = xl.v;
                *reinterpret_cast<V *>(dst + HALF + lane * PPL) = xh.v;
            }
            if (prow >= 0) {
                T *kp = static_cast<T *>(a.k_cache) + prow;
                *reinterpret_cast<V *>(kp + lane * PPL) = xl.v;
                *reinterpret_cast<V *>(kp + HALF + lane * PPL) = xh.v;
                // the value row goes to the same slot unchanged, 16 bytes per lane
                if (copy_v) reinterpret_cast<uint4 *>(static_cast<T *>(a.v_cache) + prow)[lane] = vvs[i];
            }
            continue;
        }
        // FP8 cache: codes of the key and of the value elements this lane owns
        const float ks = __ldg(a.k_scale + hh), vsc = __ldg(a.v_scale + hh);
        const C8 kl = e4m3_lane<PPL>(xl.e, ks), kh = e4m3_lane<PPL>(xh.e, ks);
        Lane yl, yh;
        const T *vsrc = static_cast<const T *>(a.v_new) + row + lane * PPL;
        yl.v = *reinterpret_cast<const V *>(vsrc);
        yh.v = *reinterpret_cast<const V *>(vsrc + HALF);
        const C8 vl = e4m3_lane<PPL>(yl.e, vsc), vh = e4m3_lane<PPL>(yh.e, vsc);
        uint8_t *dsts[4] = {a.k_q8 ? static_cast<uint8_t *>(a.k_q8) + row : nullptr,
                            a.v_q8 ? static_cast<uint8_t *>(a.v_q8) + row : nullptr,
                            prow >= 0 ? static_cast<uint8_t *>(a.k_cache) + prow : nullptr,
                            prow >= 0 ? static_cast<uint8_t *>(a.v_cache) + prow : nullptr};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (!dsts[i]) continue;
            *reinterpret_cast<C8 *>(dsts[i] + lane * PPL) = (i & 1) ? vl : kl;
            *reinterpret_cast<C8 *>(dsts[i] + HALF + lane * PPL) = (i & 1) ? vh : kh;
        }
    }
}

// Rotation only (16-bit elements, no FP8 cache): one warp per active token.
// Lane l owns the 8-pair chunk c = l mod (d / 16) of a head's half rows --
// 16 bytes of the first half and the matching 16 bytes of the second -- so it
// forms its 8 angles once for the token and rotates that chunk of every
// head, 32 / (d / 16) heads per warp step (query heads first when rotated
// queries are wanted, then key heads).  kSteps steps have their loads in
// flight before any of them stores; then the token's value rows go to its
// pool slot for a fused write.  Same angles and rounding as rope_kernel.
template <int D, typename T>
__global__ void __launch_bounds__(256) rope_rows_kernel(RopeArgs a) {
    static_assert(sizeof(T) == 2, "16-bit elements");
    constexpr int HALF = D / 2;
    constexpr int CPH = HALF / 8;        // 8-pair chunks per half row
    constexpr int HPS = 32 / CPH;        // heads per warp step
    constexpr int kSteps = 4;            // warp steps with loads in flight at once
    __shared__ unsigned long long frac_s[HALF];
    for (int c = threadIdx.x; c < HALF; c += blockDim.x) frac_s[c] = a.turn_frac[c];
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const long long t64 = blockIdx.x * (long long)(blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t64 >= a.total_tokens) return;
    const int t = (int)t64;
    const int r = request_of_token(a.cu, a.num_reqs, t);
    const int pos = __ldg(a.cached + r) + (t - __ldg(a.cu + r));
    const int c = lane % CPH, hs = lane / CPH;
    float cs[8], sn[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) rope_cos_sin(pos, frac_s[8 * c + e], cs[e], sn[e]);
    long long slot = -1;
    if (a.write_pool) slot = slot_of(a.bt, a.max_blocks, a.bs, a.num_blocks, r, pos, a.err);
    union Chunk {
        uint4 v;
        T e[8];
    };
    const int head_lo = a.q_rot ? 0 : a.hq;
    const int heads = a.hq + a.hkv;
    for (int h0 = head_lo; h0 < heads; h0 += HPS * kSteps) {
        Chunk lo[kSteps], hi[kSteps];
#pragma unroll
        for (int k = 0; k < kSteps; ++k) {
            const int head = h0 + k * HPS + hs;
            if (head < heads) {
                const bool is_q = head < a.hq;
                const long long row = is_q ? ((long long)t * a.hq + head) * D : ((long long)t * a.hkv + head - a.hq) * D;
                const T *src = static_cast<const T *>(is_q ? a.q : a.k_new) + row + 8 * c;
                lo[k].v = __ldg(reinterpret_cast<const uint4 *>(src));
                hi[k].v = __ldg(reinterpret_cast<const uint4 *>(src + HALF));
            }
        }
#pragma unroll
        for (int k = 0; k < kSteps; ++k) {
            const int head = h0 + k * HPS + hs;
            if (head >= heads) continue;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float y0, y1;
                rope_turn(to_float(lo[k].e[e]), to_float(hi[k].e[e]), cs[e], sn[e], y0, y1);
                lo[k].e[e] = from_float<T>(y0);
                hi[k].e[e] = from_float<T>(y1);
            }
            const bool is_q = head < a.hq;
            const int hh = is_q ? head : head - a.hq;
            const long long off = ((long long)t * (is_q ? a.hq : a.hkv) + hh) * D + 8 * c;
            T *dst = static_cast<T *>(is_q ? a.q_rot : a.k_rot);
            if (dst) {
                *reinterpret_cast<uint4 *>(dst + off) = lo[k].v;
                *reinterpret_cast<uint4 *>(dst + off + HALF) = hi[k].v;
            }
            if (!is_q && slot >= 0) {
                T *kp = static_cast<T *>(a.k_cache) + (slot * a.hkv + hh) * D + 8 * c;
                *reinterpret_cast<uint4 *>(kp) = lo[k].v;
                *reinterpret_cast<uint4 *>(kp + HALF) = hi[k].v;
            }
        }
    }
    if (slot >= 0) {
        // the token's value rows (all kv heads, contiguous in v_new and in
        // the slot), unchanged, 16 bytes per lane per step
        const int chunks = a.hkv * D * 2 / 16;
        const uint4 *vs = reinterpret_cast<const uint4 *>(static_cast<const T *>(a.v_new) + (long long)t * a.hkv * D);
        uint4 *vd = reinterpret_cast<uint4 *>(static_cast<T *>(a.v_cache) + slot * a.hkv * D);
        for (int i0 = lane; i0 < chunks; i0 += 32 * kSteps) {
            uint4 v[kSteps];
#pragma unroll
            for (int k = 0; k < kSteps; ++k)
                if (i0 + 32 * k < chunks) v[k] = __ldg(vs + i0 + 32 * k);
#pragma unroll
            for (int k = 0; k < kSteps; ++k)
                if (i0 + 32 * k < chunks) vd[i0 + 32 * k] = v[k];
        }
    }
}

cudaError_t launch_rope(const RopeArgs &a, int num_sms, cudaStream_t stream) {
    (void)num_sms;
    if (a.total_tokens == 0) return cudaSuccess;
    const int warps = 8;
    if (a.elem_bytes == 2 && a.rotate && !a.kv_fp8 && !a.q8) {
        const int blocks = (a.total_tokens + warps - 1) / warps;
        if (a.d == 128)
            rope_rows_kernel<128, __nv_bfloat16><<<blocks, warps * 32, 0, stream>>>(a);
        else
            rope_rows_kernel<64, __nv_bfloat16><<<blocks, warps * 32, 0, stream>>>(a);
        return cudaGetLastError();
    }
    const int heads = (a.q_rot || a.q8) ? a.hq + a.hkv : a.hkv;
    const long long work = (long long)a.total_tokens * ((heads + kHeadsPerWarp - 1) / kHeadsPerWarp);
    const int blocks = (int)((work + warps - 1) / warps);
    if (a.elem_bytes == 2) {
        if (a.d == 128)
            rope_kernel<128, __nv_bfloat16><<<blocks, warps * 32, 0, stream>>>(a);
        else
            rope_kernel<64, __nv_bfloat16><<<blocks, warps * 32, 0, stream>>>(a);
    } else {
        if (a.d == 128)
            rope_kernel<128, float><<<blocks, warps * 32, 0, stream>>>(a);
        else
            rope_kernel<64, float><<<blocks, warps * 32, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

// ------------------------------------------------------- CUDA-core attention
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <typename T, int D>
__global__ void __launch_bounds__(128) attn_simt_kernel(AttnArgs a) {
    constexpr int KT = 32;        // keys per shared-memory tile
    constexpr int RPW = 4;        // rows per warp (4 warps x 4 = kSimtTileM)
    constexpr int DPL = D / 32;   // output elements per lane
    static_assert(RPW * 4 == kSimtTileM, "tile rows");
    __shared__ float q_s[kSimtTileM][D];
    __shared__ float k_s[KT][D + 1];
    __shared__ float v_s[KT][D];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (a.fuse_write) fused_write_share(a, blockIdx.x, gridDim.x, tid, 128, (int)sizeof(T));

    Unit u;
    if (!decode_unit(a, blockIdx.x, u)) return;
    const T *q = static_cast<const T *>(a.q);
    const T *k_new = static_cast<const T *>(a.k_new);
    const T *v_new = static_cast<const T *>(a.v_new);
    const T *k_pool = static_cast<const T *>(a.k_cache);
    const T *v_pool = static_cast<const T *>(a.v_cache);
    const int G = a.G;

    for (int idx = tid; idx < kSimtTileM * D; idx += 128) {
        const int lr = idx / D, c = idx % D;
        float x = 0.f;
        if (lr < u.rows) {
            const int pr = u.row0 + lr;
            const int t = u.cu0 + pr / G, h = u.g * G + pr % G;
            x = to_float(q[((long long)t * a.hq + h) * D + c]) * a.scale_log2;
        }
        q_s[lr][c] = x;
    }

    float m[RPW], l[RPW], o[RPW][DPL];
    int pos[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int c = 0; c < DPL; ++c) o[i][c] = 0.f;
        const int lr = warp * RPW + i;
        pos[i] = (lr < u.rows) ? u.C + (u.row0 + lr) / G : -1;
    }

    for (int kb = u.k_begin; kb < u.k_end; kb += KT) {
        __syncthreads();
        for (int idx = tid; idx < KT * D; idx += 128) {
            const int kk = idx / D, c = idx % D;
            const int j = kb + kk;
            float kx = 0.f, vx = 0.f;
            if (j < u.k_end) {
                if (j < u.C) {
                    const long long slot = slot_of(a.bt, a.max_blocks, a.bs, a.num_blocks, u.r, j, a.err);
                    if (slot >= 0) {
                        const long long e = (slot * a.hkv + u.g) * D + c;
                        kx = to_float(k_pool[e]);
                        vx = to_float(v_pool[e]);
                    }
                } else {
                    const long long e = ((long long)(u.cu0 + j - u.C) * a.hkv + u.g) * D + c;
                    kx = to_float(k_new[e]);
                    vx = to_float(v_new[e]);
                }
            }
            k_s[kk][c] = kx;
            v_s[kk][c] = vx;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
            const int lr = warp * RPW + i;
            if (lr >= u.rows) continue;  // uniform across the warp
            const int j = kb + lane;
            float s = -INFINITY;
            if (j < u.k_end && j <= pos[i]) {
                float acc = 0.f;
#pragma unroll 16
                for (int c = 0; c < D; ++c) acc = fmaf(q_s[lr][c], k_s[lane][c], acc);
                s = acc;
            }
            const float mn = fmaxf(m[i], warp_max(s));
            const float mu = (mn == -INFINITY) ? 0.f : mn;
            const float p = exp2f(s - mu);
            const float alpha = exp2f(m[i] - mu);
            l[i] = l[i] * alpha + warp_sum(p);
#pragma unroll
            for (int c = 0; c < DPL; ++c) o[i][c] *= alpha;
#pragma unroll 8
            for (int jj = 0; jj < KT; ++jj) {
                const float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
                for (int c = 0; c < DPL; ++c) o[i][c] = fmaf(pj, v_s[jj][lane + 32 * c], o[i][c]);
            }
            m[i] = mn;
        }
    }

    T *out = static_cast<T *>(a.out);
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const int lr = warp * RPW + i;
        if (lr >= u.rows) continue;
        if (u.piece >= 0) {
            float *ws = a.ws + u.ws_off;
#pragma unroll
            for (int c = 0; c < DPL; ++c) ws[(long long)lr * D + lane + 32 * c] = o[i][c];
            if (lane == 0) {
                ws[(long long)u.rows * D + lr] = m[i];
                ws[(long long)u.rows * D + u.rows + lr] = l[i];
            }
        } else {
            const int pr = u.row0 + lr;
            const int t = u.cu0 + pr / G, h = u.g * G + pr % G;
            const float inv = 1.f / l[i];
#pragma unroll
            for (int c = 0; c < DPL; ++c) out[((long long)t * a.hq + h) * D + lane + 32 * c] = from_float<T>(o[i][c] * inv);
            if (a.lse && lane == 0) a.lse[(long long)t * a.hq + h] = (m[i] + log2f(l[i])) * 0.69314718055994531f;
        }
    }
}

cudaError_t launch_attn_simt(const AttnArgs &a, int dtype, cudaStream_t stream) {
    const int grid = a.num_direct_units + a.num_split_units;
    if (grid == 0) return cudaSuccess;
    if (dtype == CPA_DTYPE_FP32) {
        if (a.d == 64)
            attn_simt_kernel<float, 64><<<grid, 128, 0, stream>>>(a);
        else
            attn_simt_kernel<float, 128><<<grid, 128, 0, stream>>>(a);
    } else {
        if (a.d == 64)
            attn_simt_kernel<__nv_bfloat16, 64><<<grid, 128, 0, stream>>>(a);
        else
            attn_simt_kernel<__nv_bfloat16, 128><<<grid, 128, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

// ------------------------------------------------------------ split merge
// Combine the partials of the pieces of one split request for one kv head:
// M = max_s m_s, L = sum_s l_s 2^(m_s - M), O = sum_s O_s 2^(m_s - M) / L,
// lse = (M + log2 L) ln 2.  Pieces that saw no key (l_s = 0) are skipped.
template <typename T, int D>
__global__ void __launch_bounds__(128) attn_merge_kernel(AttnArgs a) {
    constexpr int DPL = D / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sr = blockIdx.x / a.hkv;  // index among split requests
    const int g = blockIdx.x % a.hkv;
    // find the sr-th split request and its workspace base
    int r = -1, pieces = 0;
    long long wsb = 0;
    {
        int base = 0;
        long long base_ws = 0;
        for (int r0 = 0; r0 < a.num_reqs && r < 0; r0 += 32) {
            const int rr = r0 + lane;
            ReqWork w{0, 0, 0, 0};
            if (rr < a.num_reqs) w = request_work(__ldg(a.cached + rr), __ldg(a.nnew + rr), a.G, a.hkv, a.d,
                                                  a.tile_m, split_len_of(a, rr), a.tiles_per_unit);
            const int cnt = w.split_units > 0 ? 1 : 0;
            int inc = cnt;
            long long incw = w.ws_floats;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int t = __shfl_up_sync(0xffffffffu, inc, o);
                long long tw = __shfl_up_sync(0xffffffffu, incw, o);
                if (lane >= o) {
                    inc += t;
                    incw += tw;
                }
            }
            const bool hit = cnt > 0 && sr == base + inc - 1;
            const unsigned m = __ballot_sync(0xffffffffu, hit);
            if (m) {
                const int src = __ffs(m) - 1;
                r = r0 + src;
                wsb = __shfl_sync(0xffffffffu, base_ws + incw - w.ws_floats, src);
                pieces = __shfl_sync(0xffffffffu, w.pieces, src);
            }
            base += __shfl_sync(0xffffffffu, inc, 31);
            base_ws += __shfl_sync(0xffffffffu, incw, 31);
        }
    }
    if (r < 0) return;
    const int N = __ldg(a.nnew + r), cu0 = __ldg(a.cu + r);
    const int rows = N * a.G;
    const long long unit_floats = partial_floats(rows, D);
    T *out = static_cast<T *>(a.out);
    for (int lr = warp; lr < rows; lr += 4) {
        float M = -INFINITY;
        for (int s = 0; s < pieces; ++s) {
            const float *p = a.ws + wsb + (long long)(s * a.hkv + g) * unit_floats;
            const float ls = p[(long long)rows * D + rows + lr];
            if (ls > 0.f) M = fmaxf(M, p[(long long)rows * D + lr]);
        }
        float L = 0.f, o[DPL];
#pragma unroll
        for (int c = 0; c < DPL; ++c) o[c] = 0.f;
        for (int s = 0; s < pieces; ++s) {
            const float *p = a.ws + wsb + (long long)(s * a.hkv + g) * unit_floats;
            const float ls = p[(long long)rows * D + rows + lr];
            if (!(ls > 0.f)) continue;
            const float w = exp2f(p[(long long)rows * D + lr] - M);
            L += ls * w;
#pragma unroll
            for (int c = 0; c < DPL; ++c) o[c] = fmaf(w, p[(long long)lr * D + lane + 32 * c], o[c]);
        }
        const int t = cu0 + lr / a.G, h = g * a.G + lr % a.G;
        const float inv = 1.f / L;
#pragma unroll
        for (int c = 0; c < DPL; ++c) out[((long long)t * a.hq + h) * D + lane + 32 * c] = from_float<T>(o[c] * inv);
        if (a.lse && lane == 0) a.lse[(long long)t * a.hq + h] = (M + log2f(L)) * 0.69314718055994531f;
    }
}

cudaError_t launch_attn_merge(const AttnArgs &a, int dtype, int num_split_reqs, cudaStream_t stream) {
    const int grid = num_split_reqs * a.hkv;
    if (grid == 0) return cudaSuccess;
    if (dtype == CPA_DTYPE_FP32) {
        if (a.d == 64)
            attn_merge_kernel<float, 64><<<grid, 128, 0, stream>>>(a);
        else
            attn_merge_kernel<float, 128><<<grid, 128, 0, stream>>>(a);
    } else {
        if (a.d == 64)
            attn_merge_kernel<__nv_bfloat16, 64><<<grid, 128, 0, stream>>>(a);
        else
            attn_merge_kernel<__nv_bfloat16, 128><<<grid, 128, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace cpa
