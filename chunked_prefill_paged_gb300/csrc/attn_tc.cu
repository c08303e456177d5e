// attn_tc.cu -- tensor-core (tcgen05 + TMEM + TMA) attention over the
// paged K/V cache for BF16, one work unit (see cpa_internal.h) per CTA.
//
// What one unit computes ("Prefill Processing", How Segmentation Works with
// KV Segments, Kernel Interface, Partial KV Segment Handling; "Prefill
// Optimisation", section 2, Causal equivalence): 128 packed query rows
// (tokens x the G query heads of one kv head) against the keys
// [k_begin, k_end) of their request -- cached keys from the pool through the
// block table, new keys from k_new/v_new -- causally masked at absolute
// position cached_seq_len + i, with the online softmax carried across
// 128-key tiles.
//
// Warp roles (192 threads):
//   warps 0-3  softmax / correction / epilogue; thread i owns query row i,
//              which is TMEM lane i.  They also do this CTA's share of the
//              fused K/V write before the first tile.
//   warp 4     TMA producer: Q once, then K and V tiles into an NS-stage ring.
//              A pool tile is block_size-row boxes, one per block of the
//              block table; a new-token tile is one 128-row box of k_new.
//   warp 5     MMA issuer (one lane): S_j = Q K_j^T into TMEM buffer j % 2,
//              then O += P_{j-1} V_{j-1} with P read from TMEM, so the tensor
//              core computes the next scores while softmax runs.
//
// TMEM (512 columns): S0 [0,128), S1 [128,256), O [256, 256 + D).  P_j, as
// bf16 pairs, overwrites the first 64 columns of its S buffer.
// Rescaling is lazy: the reference maximum of a row only moves (and O is
// rescaled) when a tile's maximum exceeds it by more than 2^8 in the exp2
// domain; the final O / l is exact whichever reference was used.
// Every mbarrier wait is bounded; on expiry the CTA records
// CPA_ERR_DEVICE_TIMEOUT, drains its in-flight copies and MMAs (bounded),
// frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_common.cuh"
#include "launch.h"
#include "ptx_sm100.cuh"

namespace cpa {
namespace {

using namespace ptx;

constexpr int kThreads = 192;
constexpr int kSoftmaxThreads = 128;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct TcCfg {
    static constexpr int kHalves = D / 64;                 // 64-element (128 B) column chunks
    static constexpr int kTileBytes = 128 * D * 2;         // 128 rows of D bf16
    static constexpr int kStages = (D == 128) ? 3 : 4;
    static constexpr int kSmemBytes = 1024 /*align*/ + kTileBytes * (1 + 2 * kStages);
};

struct __align__(8) TcShared {
    uint64_t q_full;
    uint64_t k_full[4], v_full[4];
    uint64_t k_empty[4], v_empty[4];
    uint64_t s_full[2], p_full[2], o_done[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Key tiles of a unit: the cached part [k_begin, min(k_end, C)) then the new
// part [max(k_begin, C), k_end), each cut into 128-key tiles.
struct TileList {
    int n_cached, n_total;
    int cached_end, new_begin;
    int k_begin, k_end;
    __device__ __forceinline__ void init(const Unit &u) {
        k_begin = u.k_begin;
        k_end = u.k_end;
        cached_end = min(u.k_end, u.C);
        new_begin = max(u.k_begin, u.C);
        const int nc = cached_end > k_begin ? cdiv(cached_end - k_begin, kTcTileN) : 0;
        const int nn = k_end > new_begin ? cdiv(k_end - new_begin, kTcTileN) : 0;
        n_cached = nc;
        n_total = nc + nn;
    }
    // first key of tile j, keys valid in it, and whether it comes from the pool
    __device__ __forceinline__ void tile(int j, int &key0, int &valid, bool &pooled) const {
        if (j < n_cached) {
            key0 = k_begin + j * kTcTileN;
            valid = min(kTcTileN, cached_end - key0);
            pooled = true;
        } else {
            key0 = new_begin + (j - n_cached) * kTcTileN;
            valid = min(kTcTileN, k_end - key0);
            pooled = false;
        }
    }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k_new, const __grid_constant__ CUtensorMap tm_v_new,
                   const __grid_constant__ CUtensorMap tm_k_pool, const __grid_constant__ CUtensorMap tm_v_pool) {
    using Cfg = TcCfg<D>;
    constexpr int NS = Cfg::kStages;
    constexpr int TB = Cfg::kTileBytes;
    extern __shared__ uint8_t smem_raw[];
    __shared__ TcShared sh;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = smem;
    uint8_t *sK = smem + TB;              // NS stages
    uint8_t *sV = smem + TB * (1 + NS);   // NS stages

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const long long LIM = a.timeout_cycles;

    if (tid == 0) {
        mbar_init(&sh.q_full, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(&sh.k_full[s], 1);
            mbar_init(&sh.v_full[s], 1);
            mbar_init(&sh.k_empty[s], 1);
            mbar_init(&sh.v_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sh.s_full[b], 1);
            mbar_init(&sh.p_full[b], kSoftmaxThreads);
            mbar_init(&sh.o_done[b], 1);
        }
        mbar_init(&sh.mma_done, 1);
        sh.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&sh.tmem_base, 512);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k_new);
        prefetch_tmap(&tm_v_new);
        prefetch_tmap(&tm_k_pool);
        prefetch_tmap(&tm_v_pool);
    }
    Unit u;
    const bool have_unit = decode_unit(a, blockIdx.x, u);  // every warp decodes the same unit
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    TileList tl;
    if (have_unit) tl.init(u);
    const int n_tiles = have_unit ? tl.n_total : 0;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ TMA
        if (lane == 0 && n_tiles > 0) {
            bool ok = true;
            mbar_arrive_expect_tx(&sh.q_full, TB);
            const int tok0 = u.cu0 + u.row0 / a.G;
            for (int h = 0; h < Cfg::kHalves; ++h)
                tma_load_3d(sQ + h * (TB / Cfg::kHalves), &tm_q, &sh.q_full, h * 64, u.g * a.G, tok0);
            const int32_t *bt_row = a.bt + (long long)u.r * a.max_blocks;
            int issued[2] = {0, 0};  // tiles whose K (0) / V (1) copies were issued
            for (int j = 0; j < n_tiles && ok; ++j) {
                const int st = j % NS;
                const uint32_t ph = (uint32_t)((j / NS) & 1);
                int key0, valid;
                bool pooled;
                tl.tile(j, key0, valid, pooled);
                for (int kv = 0; kv < 2 && ok; ++kv) {
                    uint64_t *empty = kv ? &sh.v_empty[st] : &sh.k_empty[st];
                    uint64_t *full = kv ? &sh.v_full[st] : &sh.k_full[st];
                    uint8_t *dst = (kv ? sV : sK) + st * TB;
                    if (!mbar_wait(empty, ph ^ 1u, LIM) || *(volatile int *)&sh.abort_flag) {
                        ok = false;
                        break;
                    }
                    if (a.test_stall && j == 0 && kv == 0) {
                        // testing only: arm the barrier but never copy, so the MMA
                        // warp's bounded wait on this tile expires
                        mbar_arrive_expect_tx(full, (uint32_t)TB);
                    } else if (pooled) {
                        const int nblk = cdiv(valid, a.bs);
                        mbar_arrive_expect_tx(full, (uint32_t)(nblk * a.bs * D * 2));
                        const int col0 = key0 / a.bs;
                        for (int b = 0; b < nblk; ++b) {
                            int blk = __ldg(bt_row + col0 + b);
                            if (blk < 0 || blk >= a.num_blocks) {
                                record_error(a.err, kErrBadBlock);
                                blk = 0;  // keep the byte count; the output of this unit is void
                            }
                            for (int h = 0; h < Cfg::kHalves; ++h)
                                tma_load_4d(dst + h * (TB / Cfg::kHalves) + b * a.bs * 128, kv ? &tm_v_pool : &tm_k_pool,
                                            full, h * 64, u.g, 0, blk);
                        }
                    } else {
                        mbar_arrive_expect_tx(full, (uint32_t)TB);
                        const int row = u.cu0 + (key0 - u.C);
                        for (int h = 0; h < Cfg::kHalves; ++h)
                            tma_load_3d(dst + h * (TB / Cfg::kHalves), kv ? &tm_v_new : &tm_k_new, full, h * 64, u.g,
                                        row);
                    }
                    issued[kv] = j + 1;
                }
            }
            if (!ok) {
                record_error(a.err, kErrTimeout);
                sh.abort_flag = 1;
            }
            // drain: every issued copy must land before the CTA may exit
            mbar_wait(&sh.q_full, 0, LIM);
            for (int kv = 0; kv < 2; ++kv)
                for (int j = (issued[kv] > NS ? issued[kv] - NS : 0); j < issued[kv]; ++j)
                    mbar_wait(kv ? &sh.v_full[j % NS] : &sh.k_full[j % NS], (uint32_t)((j / NS) & 1), LIM);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA
        if (lane == 0 && n_tiles > 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, 0, 1);
            const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK), sVa = smem_u32(sV);
            const uint32_t tO = tmem + 256;
            bool ok = mbar_wait(&sh.q_full, 0, LIM);
            auto issue_pv = [&](int i) -> bool {
                const int b = i & 1, st = i % NS;
                if (!mbar_wait(&sh.p_full[b], (uint32_t)((i >> 1) & 1), LIM)) return false;
                if (!mbar_wait(&sh.v_full[st], (uint32_t)((i / NS) & 1), LIM)) return false;
                tc_fence_after();
                const uint32_t vbase = sVa + st * TB;
#pragma unroll
                for (int kk = 0; kk < kTcTileN / 16; ++kk) {
                    const uint64_t bd = smem_desc(vbase + kk * 2048, 16384, 1024, kSwizzle128B);
                    umma_ts(tO, tmem + b * 128 + kk * 8, bd, idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(&sh.v_empty[st]);
                umma_commit(&sh.o_done[b]);
                return true;
            };
            for (int j = 0; j < n_tiles && ok; ++j) {
                const int b = j & 1, st = j % NS;
                if (!mbar_wait(&sh.k_full[st], (uint32_t)((j / NS) & 1), LIM) || *(volatile int *)&sh.abort_flag) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t kbase = sKa + st * TB;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (TB / Cfg::kHalves) + (kk & 3) * 32;
                    const uint64_t ad = smem_desc(sQa + off, 16, 1024, kSwizzle128B);
                    const uint64_t bd = smem_desc(kbase + off, 16, 1024, kSwizzle128B);
                    umma_ss(tmem + b * 128, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
                }
                umma_commit(&sh.k_empty[st]);
                umma_commit(&sh.s_full[b]);
                if (j >= 1 && !issue_pv(j - 1)) ok = false;
            }
            if (ok && !issue_pv(n_tiles - 1)) ok = false;
            if (!ok) {
                record_error(a.err, kErrTimeout);
                sh.abort_flag = 1;
            }
            // every MMA issued so far must finish before TMEM is freed
            umma_commit(&sh.mma_done);
            mbar_wait(&sh.mma_done, 0, LIM);
        }
    } else {
        // ------------------------------------------------- softmax (warps 0-3)
        if (a.fuse_write) fused_write_share(a, blockIdx.x, a.write_ctas, tid, kSoftmaxThreads, 2);
        if (n_tiles > 0) {
            const int lr = tid;  // query row == TMEM lane
            const bool row_valid = lr < u.rows;
            const int pos = row_valid ? u.C + (u.row0 + lr) / a.G : -1;
            const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
            float m_ref = -INFINITY, l = 0.f;
            bool ok = true;
            for (int j = 0; j < n_tiles; ++j) {
                const int b = j & 1, st = j % NS;
                if (!__all_sync(0xffffffffu, mbar_wait(&sh.s_full[b], (uint32_t)((j >> 1) & 1), LIM) &&
                                                 !*(volatile int *)&sh.abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                int key0, valid;
                bool pooled;
                tl.tile(j, key0, valid, pooled);
                // scores of this row
                float s[kTcTileN];
#pragma unroll
                for (int c = 0; c < kTcTileN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(lane_base + b * 128 + c * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(r[i]);
                }
                const int lim = min(valid, pos - key0 + 1);  // keys [0, lim) of the tile are visible
                float tmax = -INFINITY;
#pragma unroll
                for (int k = 0; k < kTcTileN; ++k) {
                    s[k] = (k < lim) ? s[k] * a.scale_log2 : -INFINITY;
                    tmax = fmaxf(tmax, s[k]);
                }
                // O may only be touched once the PV that last wrote it is done
                if (j >= 2 &&
                    !__all_sync(0xffffffffu, mbar_wait(&sh.o_done[(j - 2) & 1], (uint32_t)(((j - 2) >> 1) & 1), LIM))) {
                    ok = false;
                    break;
                }
                const bool move = (tmax > m_ref + kRescaleThreshold) || (m_ref == -INFINITY && tmax > -INFINITY);
                float alpha = 1.f;
                if (move) {
                    alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - tmax);
                    m_ref = tmax;
                    l *= alpha;
                }
                if (j >= 1 && __any_sync(0xffffffffu, move)) {
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait(&sh.o_done[(j - 1) & 1], (uint32_t)(((j - 1) >> 1) & 1), LIM))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld32(lane_base + 256 + c * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                        tmem_st32(lane_base + 256 + c * 32, r);
                    }
                }
                const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;
                float rsum = 0.f;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t r[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float p0 = ex2(s[c * 64 + 2 * i] - mu);
                        const float p1 = ex2(s[c * 64 + 2 * i + 1] - mu);
                        rsum += p0 + p1;
                        r[i] = pack_bf16(p0, p1);
                    }
                    tmem_st32(lane_base + b * 128 + c * 32, r);
                }
                l += rsum;
                if (valid < kTcTileN) {
                    // keys past the valid range of this tile: zero their V rows so that
                    // P = 0 never meets a NaN or Inf left in the pool or in shared memory
                    if (!__all_sync(0xffffffffu, mbar_wait(&sh.v_full[st], (uint32_t)((j / NS) & 1), LIM))) {
                        ok = false;
                        break;
                    }
                    if (tid >= valid) {
                        uint8_t *vrow = sV + st * TB + tid * 128;
#pragma unroll
                        for (int h = 0; h < Cfg::kHalves; ++h) {
                            uint4 *p = reinterpret_cast<uint4 *>(vrow + h * (TB / Cfg::kHalves));
#pragma unroll
                            for (int i = 0; i < 8; ++i) p[i] = make_uint4(0, 0, 0, 0);
                        }
                    }
                    fence_proxy_async_smem();
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&sh.p_full[b]);
            }
            if (ok) {
                const int n = n_tiles;
                if (n >= 2) ok = __all_sync(0xffffffffu, mbar_wait(&sh.o_done[(n - 2) & 1], (uint32_t)(((n - 2) >> 1) & 1), LIM));
                if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&sh.o_done[(n - 1) & 1], (uint32_t)(((n - 1) >> 1) & 1), LIM));
            }
            if (!ok) {
                record_error(a.err, kErrTimeout);
                sh.abort_flag = 1;
            }
            tc_fence_after();
            if (ok) {
                // epilogue: O row from TMEM
                float o[D];
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(lane_base + 256 + c * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[c * 32 + i] = __uint_as_float(r[i]);
                }
                if (row_valid) {
                    if (u.piece >= 0) {
                        float *ws = a.ws + u.ws_off;
                        float4 *dst = reinterpret_cast<float4 *>(ws + (long long)lr * D);
#pragma unroll
                        for (int i = 0; i < D / 4; ++i) dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                        ws[(long long)u.rows * D + lr] = m_ref;
                        ws[(long long)u.rows * D + u.rows + lr] = l;
                    } else {
                        const int pr = u.row0 + lr;
                        const int t = u.cu0 + pr / a.G, h = u.g * a.G + pr % a.G;
                        const float inv = 1.f / l;
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) +
                                                               ((long long)t * a.hq + h) * D);
#pragma unroll
                        for (int i = 0; i < D / 8; ++i) {
                            uint4 w;
                            w.x = pack_bf16(o[8 * i + 0] * inv, o[8 * i + 1] * inv);
                            w.y = pack_bf16(o[8 * i + 2] * inv, o[8 * i + 3] * inv);
                            w.z = pack_bf16(o[8 * i + 4] * inv, o[8 * i + 5] * inv);
                            w.w = pack_bf16(o[8 * i + 6] * inv, o[8 * i + 7] * inv);
                            dst[i] = w;
                        }
                        if (a.lse) a.lse[(long long)t * a.hq + h] = (m_ref + __log2f(l)) * 0.69314718055994531f;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) {
        __syncwarp();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_attn_tc(const AttnArgs &a, const TcMaps &m, cudaStream_t stream) {
    const int grid = a.num_direct_units + a.num_split_units;
    if (grid == 0) return cudaSuccess;
    cudaError_t e;
    if (a.d == 128) {
        constexpr int smem = TcCfg<128>::kSmemBytes;
        e = cudaFuncSetAttribute(attn_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attn_tc_kernel<128><<<grid, kThreads, smem, stream>>>(a, m.q, m.k_new, m.v_new, m.k_pool, m.v_pool);
    } else {
        constexpr int smem = TcCfg<64>::kSmemBytes;
        e = cudaFuncSetAttribute(attn_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attn_tc_kernel<64><<<grid, kThreads, smem, stream>>>(a, m.q, m.k_new, m.v_new, m.k_pool, m.v_pool);
    }
    return cudaGetLastError();
}

}  // namespace cpa
