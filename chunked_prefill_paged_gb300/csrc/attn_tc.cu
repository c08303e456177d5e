// attn_tc.cu -- tensor-core (tcgen05 + TMEM + TMA) attention over the paged
// K/V cache for BF16.  Persistent: one CTA per SM walks the work units (see
// cpa_internal.h) in order blockIdx.x, blockIdx.x + gridDim.x, ...
//
// What a unit computes ("Prefill Processing", How Segmentation Works with KV
// Segments, Kernel Interface, Partial KV Segment Handling; "Prefill
// Optimisation", section 2, Causal equivalence): one 128-row query tile --
// packed (token, query head) rows of one request and one kv head -- against
// the keys [k_begin, k_end) of the request, cached keys read from the pool
// through the block table and new keys from k_new/v_new, masked causally at
// absolute position cached_seq_len + i.  The online softmax is carried
// across 128-key tiles; a split unit (one piece of a decode's keys) writes
// its unnormalised partial for attn_merge instead.
//
// Warp roles (384 threads):
//   warps 0-7  softmax / correction / epilogue.  Two threads own one query
//              row: warp w covers TMEM lanes 32 (w % 4) + 16 (w / 4) .. +15,
//              its threads 0-15 the row's keys 0-63 (output columns 0 .. D/2-1)
//              and threads 16-31 keys 64-127 (columns D/2 .. D-1); the row
//              maximum and sum are combined with one shuffle.  They also do
//              this CTA's share of the fused K/V write first.
//   warp 8     TMA producer of Q per unit and of the K tiles; warp 10 of the V
//              tiles, each into its own ring, so a V slot still in use never
//              holds up the next K copy.  A pool tile is one box per cache
//              block (found through the block table), a new-token tile one
//              128-row box of k_new / v_new.  Warp 11 idles.
//   warp 9     MMA issuer (converged; one elected lane issues).  Scores run one tile ahead: for key tile
//              j it issues S(j+1) = Q K(j+1)^T into the other score buffer,
//              then O += P(j) V(j) once the softmax has written P(j), so the
//              tensor core computes the next scores while softmax runs.
//
// TMEM (512 columns): two score buffers S0 [0,128) and S1 [128,256), O
// [256, 256 + D).  P(j), as bf16 pairs, overwrites the first 64 columns of
// the buffer that held S(j); S(j+2) reuses that buffer only after PV(j) was
// issued (tensor-core ops from one thread run in order).  Rescaling is lazy:
// a row's reference maximum moves (and O is rescaled, after waiting for the
// previous PV) only when a tile's maximum exceeds it by more than 2^8 in the
// exp2 domain; the final O / l is exact whichever reference was used.
// Every mbarrier wait is bounded; on expiry the CTA records
// CPA_ERR_DEVICE_TIMEOUT, drains its copies and MMAs, frees TMEM and returns.
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

constexpr int kThreads = 384;
constexpr int kSoftmaxThreads = 256;  // warps 0-7
constexpr int kProducerWarp = 8;      // Q and K copies
constexpr int kMmaWarp = 9;
constexpr int kVProducerWarp = 10;    // V copies (warp 11 idles)
constexpr int kKT = kTcTileN;         // keys per K/V tile (128)
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct TcCfg {
    static constexpr int kHalves = D / 64;           // 64-element (128 B) column chunks
    static constexpr int kTileBytes = 128 * D * 2;   // 128 rows of D bf16 (Q, K or V tile)
    static constexpr int kHalfBytes = kTileBytes / kHalves;
    static constexpr int kKStages = (D == 128) ? 3 : 6;
    static constexpr int kVStages = (D == 128) ? 3 : 6;
    static constexpr int kSmemBytes = 1024 /*align*/ + kTileBytes * (1 + kKStages + kVStages);
};

struct __align__(8) TcShared {
    uint64_t q_full, q_empty;
    uint64_t k_full[6], k_empty[6];
    uint64_t v_full[6], v_empty[6];
    uint64_t s_full[2];  // per score buffer
    uint64_t p_full[2];  // per score buffer: P(j) written over S(j)
    uint64_t pv_done;
    uint64_t o_full, o_empty;
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
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
        n_cached = cached_end > k_begin ? cdiv(cached_end - k_begin, kKT) : 0;
        const int nn = k_end > new_begin ? cdiv(k_end - new_begin, kKT) : 0;
        n_total = n_cached + nn;
    }
    // first key of tile j, keys valid in it, and whether it comes from the pool
    __device__ __forceinline__ void tile(int j, int &key0, int &valid, bool &pooled) const {
        if (j < n_cached) {
            key0 = k_begin + j * kKT;
            valid = min(kKT, cached_end - key0);
            pooled = true;
        } else {
            key0 = new_begin + (j - n_cached) * kKT;
            valid = min(kKT, k_end - key0);
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
    constexpr int NSK = Cfg::kKStages;
    constexpr int NSV = Cfg::kVStages;
    constexpr int TB = Cfg::kTileBytes;
    constexpr int HB = Cfg::kHalfBytes;
    extern __shared__ uint8_t smem_raw[];
    __shared__ TcShared sh;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = smem;
    uint8_t *sK = smem + TB;           // NSK stages
    uint8_t *sV = sK + NSK * TB;       // NSV stages

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const long long LIM = a.timeout_cycles;
    const int total_units = a.num_direct_units + a.num_split_units;

    if (tid == 0) {
        mbar_init(&sh.q_full, 1);
        mbar_init(&sh.q_empty, 1);
        for (int s = 0; s < NSK; ++s) {
            mbar_init(&sh.k_full[s], 1);
            mbar_init(&sh.k_empty[s], 1);
        }
        for (int s = 0; s < NSV; ++s) {
            mbar_init(&sh.v_full[s], 1);
            mbar_init(&sh.v_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sh.s_full[b], 1);
            mbar_init(&sh.p_full[b], kSoftmaxThreads);
        }
        mbar_init(&sh.pv_done, 1);
        mbar_init(&sh.o_full, 1);
        mbar_init(&sh.o_empty, kSoftmaxThreads);
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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    volatile int *abort_flag = &sh.abort_flag;

    if (warp == kProducerWarp || warp == kVProducerWarp) {
        // ================================================================ TMA
        const int kv_role = (warp == kVProducerWarp) ? 1 : 0;  // copies K (0) or V (1)
        long long gt = 0;  // key tiles of the units before this one
        int it = 0;        // units started by this CTA
        bool ok = true;
        long long issued = 0;  // tiles (counted in gt) whose copies this warp issued
        for (int unit = blockIdx.x; unit < total_units; unit += gridDim.x, ++it) {
            if (__any_sync(0xffffffffu, !ok || *abort_flag)) break;
            Unit u;
            decode_unit(a, unit, u);
            TileList tl;
            tl.init(u);
            const int n = tl.n_total;
            // The warp runs converged: every lane takes the waits, lane 0 arms
            // the barriers, and the copies of one tile are spread over the lanes
            // (one cache block and 64-column half per lane).
            const int32_t *bt_row = a.bt + (long long)u.r * a.max_blocks;
            // copies of key tile j (K when kv = 0, V when kv = 1) into their ring slot
            auto load_kv = [&](int j, int kv) -> bool {
                const long long g = gt + j;
                const int ns = kv ? NSV : NSK;
                const int st = (int)(g % ns);
                const uint32_t ph = (uint32_t)((g / ns) & 1);
                uint64_t *empty = kv ? &sh.v_empty[st] : &sh.k_empty[st];
                uint64_t *full = kv ? &sh.v_full[st] : &sh.k_full[st];
                uint8_t *dst = (kv ? sV : sK) + st * TB;
                if (!__all_sync(0xffffffffu, mbar_wait(empty, ph ^ 1u, LIM)) || __any_sync(0xffffffffu, *abort_flag))
                    return false;
                int key0, valid;
                bool pooled;
                tl.tile(j, key0, valid, pooled);
                if (a.test_stall && it == 0 && j == 0 && kv == 0) {
                    // testing only: arm the barrier but never copy, so the
                    // MMA warp's bounded wait on this tile expires
                    if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)TB);
                } else if (pooled) {
                    const int nblk = cdiv(valid, a.bs);
                    if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)(nblk * a.bs * D * 2));
                    __syncwarp();
                    const int col0 = key0 / a.bs;
                    for (int i = lane; i < nblk * Cfg::kHalves; i += 32) {
                        const int b = i / Cfg::kHalves, h = i % Cfg::kHalves;
                        int blk = __ldg(bt_row + col0 + b);
                        if (blk < 0 || blk >= a.num_blocks) {
                            record_error(a.err, kErrBadBlock);
                            blk = 0;  // keep the byte count; this unit's output is void
                        }
                        tma_load_4d(dst + h * HB + b * a.bs * 128, kv ? &tm_v_pool : &tm_k_pool, full, h * 64, u.g,
                                    0, blk);
                    }
                } else {
                    if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)TB);
                    __syncwarp();
                    const int row = u.cu0 + (key0 - u.C);
                    if (lane < Cfg::kHalves)
                        tma_load_3d(dst + lane * HB, kv ? &tm_v_new : &tm_k_new, full, lane * 64, u.g, row);
                }
                issued = g + 1;
                return true;
            };
            if (kv_role == 0) {
                // the first K tile does not depend on the Q buffer: issue it
                // before waiting for the previous unit's last score MMA
                ok = load_kv(0, 0);
                if (ok && it > 0 && !__all_sync(0xffffffffu, mbar_wait(&sh.q_empty, (uint32_t)((it - 1) & 1), LIM)))
                    ok = false;
                if (ok) {
                    if (lane == 0) mbar_arrive_expect_tx(&sh.q_full, TB);
                    __syncwarp();
                    const int tok0 = u.cu0 + u.row0 / a.G;
                    if (lane < Cfg::kHalves) tma_load_3d(sQ + lane * HB, &tm_q, &sh.q_full, lane * 64, u.g * a.G, tok0);
                }
                for (int j = 1; j < n && ok; ++j) ok = load_kv(j, 0);
            } else {
                for (int j = 0; j < n && ok; ++j) ok = load_kv(j, 1);
            }
            gt += n;
        }
        if (!ok) {
            if (lane == 0) record_error(a.err, kErrTimeout);
            *abort_flag = 1;
        }
        // drain: every issued copy must land before the CTA may exit
        {
            const int ns = kv_role ? NSV : NSK;
            for (long long g = (issued > ns ? issued - ns : 0); g < issued; ++g)
                mbar_wait(kv_role ? &sh.v_full[(int)(g % ns)] : &sh.k_full[(int)(g % ns)], (uint32_t)((g / ns) & 1),
                          LIM);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ================================================================ MMA
        long long gt = 0;
        int qcnt = 0;  // units started
        int gs = 0;    // score tiles issued (buffer gs & 1)
        int pc = 0;    // P tiles consumed
        int oc = 0;    // units finished
        bool ok = true;
        constexpr uint32_t idesc_s = idesc_bf16_f32(128, kKT, 0, 0);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, 0, 1);
        // Shared-memory descriptors are built once; a k-step or ring slot only
        // advances the start-address field (bytes >> 4), which stays below 2^14
        // for any shared-memory address.
        const uint64_t q_desc = smem_desc(smem_u32(sQ), 16, 1024, kSwizzle128B);
        const uint64_t k_desc0 = smem_desc(smem_u32(sK), 16, 1024, kSwizzle128B);
        const uint64_t v_desc0 = smem_desc(smem_u32(sV), HB, 1024, kSwizzle128B);
        const uint32_t tO = tmem + 256;
        for (int unit = blockIdx.x; unit < total_units; unit += gridDim.x) {
            if (__any_sync(0xffffffffu, !ok || *abort_flag)) break;
            Unit u;
            decode_unit(a, unit, u);
            TileList tl;
            tl.init(u);
            const int n = tl.n_total;
            // The whole warp runs this converged; one elected lane issues each
            // MMA and commit, and every wait is taken by all lanes.
            // S(jj) = Q K(jj)^T into the next score buffer
            auto issue_s = [&](int jj) -> bool {
                const long long g = gt + jj;
                const int st = (int)(g % NSK);
                if (!__all_sync(0xffffffffu, mbar_wait(&sh.k_full[st], (uint32_t)((g / NSK) & 1), LIM)) ||
                    __any_sync(0xffffffffu, *abort_flag))
                    return false;
                tc_fence_after();
                const uint64_t kd = k_desc0 + (uint64_t)((st * TB) >> 4);
                const uint32_t d_tmem = tmem + (gs & 1) * kKT;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (uint64_t)(((kk >> 2) * HB + (kk & 3) * 32) >> 4);
                    umma_ss_warp(d_tmem, q_desc + off, kd + off, idesc_s, kk > 0 ? 1u : 0u);
                }
                umma_commit_warp(&sh.s_full[gs & 1]);
                umma_commit_warp(&sh.k_empty[st]);
                ++gs;
                if (jj == n - 1) umma_commit_warp(&sh.q_empty);  // Q is free once the last S is done
                return true;
            };
            if (!__all_sync(0xffffffffu, mbar_wait(&sh.q_full, (uint32_t)(qcnt++ & 1), LIM))) ok = false;
            tc_fence_after();
            if (ok) ok = issue_s(0);
            for (int j = 0; j < n && ok; ++j) {
                // the next scores go first, into the buffer PV(j-1) has finished reading
                if (j + 1 < n && !issue_s(j + 1)) {
                    ok = false;
                    break;
                }
                const int b = pc & 1;  // P(j) sits in the buffer S(j) used
                if (!__all_sync(0xffffffffu, mbar_wait(&sh.p_full[b], (uint32_t)((pc >> 1) & 1), LIM))) {
                    ok = false;
                    break;
                }
                ++pc;
                if (j == 0 && !__all_sync(0xffffffffu, mbar_wait(&sh.o_empty, (uint32_t)((oc & 1) ^ 1), LIM))) {
                    ok = false;
                    break;
                }
                const long long g = gt + j;
                const int st = (int)(g % NSV);
                if (!__all_sync(0xffffffffu, mbar_wait(&sh.v_full[st], (uint32_t)((g / NSV) & 1), LIM))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t vd = v_desc0 + (uint64_t)((st * TB) >> 4);
                const uint32_t tP = tmem + b * kKT;
#pragma unroll
                for (int kk = 0; kk < kKT / 16; ++kk)
                    umma_ts_warp(tO, tP + kk * 8, vd + (uint64_t)((kk * 2048) >> 4), idesc_pv,
                                 (j > 0 || kk > 0) ? 1u : 0u);
                umma_commit_warp(&sh.v_empty[st]);
                umma_commit_warp(&sh.pv_done);
                if (j == n - 1) {
                    umma_commit_warp(&sh.o_full);
                    ++oc;
                }
            }
            gt += n;
        }
        if (!ok) {
            if (lane == 0) record_error(a.err, kErrTimeout);
            *abort_flag = 1;
        }
        // every MMA issued so far must finish before TMEM is freed
        umma_commit_warp(&sh.mma_done);
        mbar_wait(&sh.mma_done, 0, LIM);
        __syncwarp();
    } else if (warp < 8) {
        // ============================================== softmax (warps 0-7)
        const int half = lane >> 4;                                // 0: keys 0-63, 1: keys 64-127
        const int lr = 32 * (warp & 3) + 16 * (warp >> 2) + (lane & 15);  // row of the tile == TMEM lane
        if (a.fuse_write) fused_write_share(a, blockIdx.x, gridDim.x, tid, kSoftmaxThreads, 2);
        const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3) + 16 * (warp >> 2)) << 16);
        const uint32_t tO = lane_base + 256;
        const float sl = a.scale_log2;
        long long gt = 0;
        int gs = 0;  // score tiles consumed (== P tiles produced)
        int oc = 0;
        bool ok = true;
        for (int unit = blockIdx.x; unit < total_units; unit += gridDim.x) {
            if (__any_sync(0xffffffffu, !ok || *abort_flag)) break;
            Unit u;
            decode_unit(a, unit, u);
            TileList tl;
            tl.init(u);
            const int n = tl.n_total;
            const bool row_valid = lr < u.rows;
            const int pos = row_valid ? u.C + (u.row0 + lr) / a.G : -1;
            float m_ref = -INFINITY, l = 0.f;
            for (int j = 0; j < n; ++j) {
                const int b = gs & 1;
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&sh.s_full[b], (uint32_t)((gs >> 1) & 1), LIM) && !*abort_flag)) {
                    ok = false;
                    break;
                }
                ++gs;
                tc_fence_after();
                const uint32_t tS = lane_base + b * kKT;
                int key0, valid;
                bool pooled;
                tl.tile(j, key0, valid, pooled);
                float s[64];  // keys half*64 .. half*64 + 63 of the tile
                {
                    uint32_t r0[32], r1[32];
                    tmem_ld16x2_32<64>(tS, r0);  // threads 0-15: keys 0-31, 16-31: keys 64-95
                    tmem_ld16x2_32<64>(tS + 32, r1);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        s[i] = __uint_as_float(r0[i]);
                        s[32 + i] = __uint_as_float(r1[i]);
                    }
                }
                // keys [0, lim) of the tile are visible to this row
                const int lim = min(valid, pos - key0 + 1) - half * 64;
                if (!__all_sync(0xffffffffu, lim >= 64)) {
#pragma unroll
                    for (int k = 0; k < 64; ++k) s[k] = (k < lim) ? s[k] : -INFINITY;
                }
                float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
                for (int k = 4; k < 60; k += 8) {
                    mx0 = max3(mx0, s[k], s[k + 1]);
                    mx1 = max3(mx1, s[k + 2], s[k + 3]);
                    mx2 = max3(mx2, s[k + 4], s[k + 5]);
                    mx3 = max3(mx3, s[k + 6], s[k + 7]);
                }
                mx0 = max3(mx0, s[60], s[61]);
                mx1 = max3(mx1, s[62], s[63]);
                float tmax = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
                tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16)) * sl;  // whole row
                const bool move = (tmax > m_ref + kRescaleThreshold) || (m_ref == -INFINITY && tmax > -INFINITY);
                float alpha = 1.f;
                if (move) {
                    alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - tmax);
                    m_ref = tmax;
                    l *= alpha;
                }
                const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref;
                float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
                {
                    uint32_t r[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float e0 = ex2(fmaf(s[2 * i], sl, neg));
                        const float e1 = ex2(fmaf(s[2 * i + 1], sl, neg));
                        if (i & 1) {
                            a2 += e0;
                            a3 += e1;
                        } else {
                            a0 += e0;
                            a1 += e1;
                        }
                        r[i] = pack_bf16(e0, e1);
                    }
                    tmem_st16x2_32<32>(tS, r);  // threads 0-15: P columns 0-31, 16-31: 32-63
                }
                l += (a0 + a1) + (a2 + a3);
                if (j >= 1 && __any_sync(0xffffffffu, move)) {
                    // rescale O once PV(j-1) (global P tile gs - 2) has completed;
                    // PV(j) cannot start before this group's arrival below
                    if (!__all_sync(0xffffffffu, mbar_wait(&sh.pv_done, (uint32_t)((gs - 2) & 1), LIM))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) {
                        uint32_t r[32];
                        tmem_ld16x2_32<D / 2>(tO + c * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                        tmem_st16x2_32<D / 2>(tO + c * 32, r);
                    }
                }
                if (valid < kKT) {
                    // keys past the tile's valid range: zero their V rows so that
                    // P = 0 never meets a NaN or Inf left in the pool or in smem
                    const long long g = gt + j;
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait(&sh.v_full[(int)(g % NSV)], (uint32_t)((g / NSV) & 1), LIM))) {
                        ok = false;
                        break;
                    }
                    const int vr = tid >> 1, vh = tid & 1;  // V row, 64-column chunk
                    if (vr >= valid && vh < Cfg::kHalves) {
                        uint4 *q4 = reinterpret_cast<uint4 *>(sV + (int)(g % NSV) * TB + vh * HB + vr * 128);
#pragma unroll
                        for (int i = 0; i < 8; ++i) q4[i] = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&sh.p_full[b]);
            }
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&sh.o_full, (uint32_t)(oc & 1), LIM));
            if (!ok) break;
            tc_fence_after();
            l += __shfl_xor_sync(0xffffffffu, l, 16);  // whole row
            // epilogue: this thread's half of the O row, then release O
            const int pr = u.row0 + lr;  // packed row of the request
            const float inv = 1.f / l;
            const int t = u.cu0 + pr / a.G, h = u.g * a.G + pr % a.G;
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t r[32];
                tmem_ld16x2_32<D / 2>(tO + c * 32, r);  // output columns half * D/2 + c * 32 + i
                tmem_wait_ld();
                const int col0 = half * (D / 2) + c * 32;
                if (row_valid) {
                    if (u.piece >= 0) {
                        float4 *dst = reinterpret_cast<float4 *>(a.ws + u.ws_off + (long long)pr * D + col0);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                                 __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
                    } else {
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) +
                                                               ((long long)t * a.hq + h) * D + col0);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            uint4 w;
                            w.x = pack_bf16(__uint_as_float(r[8 * i + 0]) * inv, __uint_as_float(r[8 * i + 1]) * inv);
                            w.y = pack_bf16(__uint_as_float(r[8 * i + 2]) * inv, __uint_as_float(r[8 * i + 3]) * inv);
                            w.z = pack_bf16(__uint_as_float(r[8 * i + 4]) * inv, __uint_as_float(r[8 * i + 5]) * inv);
                            w.w = pack_bf16(__uint_as_float(r[8 * i + 6]) * inv, __uint_as_float(r[8 * i + 7]) * inv);
                            dst[i] = w;
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&sh.o_empty);
            ++oc;
            if (row_valid && half == 0) {
                if (u.piece >= 0) {
                    float *ws = a.ws + u.ws_off;
                    ws[(long long)u.rows * D + pr] = m_ref;
                    ws[(long long)u.rows * D + u.rows + pr] = l;
                } else if (a.lse) {
                    a.lse[(long long)t * a.hq + h] = (m_ref + __log2f(l)) * 0.69314718055994531f;
                }
            }
            gt += n;
        }
        if (!ok) {
            record_error(a.err, kErrTimeout);
            *abort_flag = 1;
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
    const int grid = a.write_ctas;  // persistent: min(units, SMs)
    if (grid <= 0 || a.num_direct_units + a.num_split_units == 0) return cudaSuccess;
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
