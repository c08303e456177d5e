// attn_tc2.cu -- tensor-core attention over BF16 pools with two query tiles
// per unit (attn_tc2_kernel<D>).  Same computation and unit decomposition as
// attn_tc.cu ("Prefill Processing", How Segmentation Works with KV Segments,
// Kernel Interface; "Prefill Optimisation", section 2, Causal equivalence):
// a unit is one request and one kv head, here two consecutive 128-row query
// tiles A and B (packed (token, query head) rows) that share every K and V
// tile the unit walks.  A split unit (one piece of a decode's keys) has tile
// A only and writes its unnormalised partial for attn_merge.
//
// Why two tiles.  One 128 x 128 key tile costs 1024 tensor cycles (S = Q K^T
// and O += P V, 512 each); the softmax of one tile (128 rows x 128 keys)
// takes longer than that on a single tile's pipeline.  With two tiles the
// MMA warp issues, per key tile j,
//     S_A(j), PV_B(j-1), S_B(j), PV_A(j)
// so the softmax of tile A has the time of PV_B(j-1) and S_B(j) (1024
// tensor cycles) to turn S_A(j) into P_A(j), and likewise for B, while the
// tensor pipe stays busy.  Every K / V tile then serves 256 query rows, which
// halves the copies (and the TMA boxes: 16 per operand tile at block size
// 16) per FLOP.
//
// TMEM (512 columns): S_A [0, 128), S_B [128, 256), O_A [256, 256 + D),
// O_B [256 + D, 256 + 2D).  P_X(j), as bf16 pairs, overwrites the first 64
// columns of S_X; S_X(j + 1) is issued after PV_X(j) by the same thread, and
// tcgen05 MMAs of one CTA execute in issue order, so S_X(j + 1) cannot
// overwrite P_X(j) before PV_X(j) has read it.
//
// Warp roles (512 threads):
//   warps 0-3   softmax of tile A, warps 4-7 of tile B: one thread per row
//               (TMEM lane 32 (w % 4) + lane), all 128 keys of a tile; lazy
//               rescale of the row's O (only when its maximum grows by more
//               than 2^8 in the exp2 domain).  They also take the pieces of
//               the fused K/V write.  These two warpgroups run with more
//               registers (setmaxnreg) than the others.
//   warp 8      unit scheduler (claims units from the launch's work counter,
//               decodes each once and publishes it) and TMA producer of K.
//   warp 9      MMA issuer (all four MMA kinds, one elected lane).
//   warp 10     TMA producer of V; zeroes the rows of a partial V tile past
//               its valid keys once it has landed (P = 0 must not meet a NaN
//               left in the pool or a stale value in the slot).
//   warp 11     TMA producer of Q: tile A's stage is reloaded as soon as the
//               unit's last S_A MMA has completed, tile B's after the last
//               S_B; each unit's Q is prefetched into L2 when the unit is
//               published, ahead of that.
//   warps 12-15 epilogue: warp 12 + e reads TMEM lanes 32e .. 32e + 31 of O_A
//               and then O_B, one thread per output row, and writes the rows
//               (or a split unit's fp32 partial) and the LSE.
// Every mbarrier wait is bounded; on expiry the CTA records
// CPA_ERR_DEVICE_TIMEOUT, drains its copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "device_common.cuh"
#include "launch.h"
#include "ptx_sm100.cuh"
#include "tc_common.cuh"

namespace cpa {
namespace {

using namespace ptx;
using namespace tc;

constexpr int kThreads2 = 512;
constexpr int kSoftmaxThreads2 = 256;  // warps 0-7
constexpr int kKWarp = 8;              // scheduler and K copies
constexpr int kMmaWarp2 = 9;
constexpr int kVWarp = 10;             // V copies and partial-tile zeroing
constexpr int kQWarp = 11;             // Q copies
constexpr int kEpiWarp2 = 12;          // warps 12-15
constexpr int kReaders2 = 15;          // every warp but 8 reads every unit
constexpr float kRescaleThreshold2 = 8.0f;  // log2 units
// Registers per thread: the launch gives 128 to each of the 512 threads; the
// two softmax warpgroups take 184 (a row's 128 scores stay in registers),
// warps 8-11 keep 80 and the epilogue warpgroup 64 (2 x 184 + 80 + 64 =
// 4 x 128; a split that compiles without spills).
constexpr uint32_t kRegsSoftmax = 184;
constexpr uint32_t kRegsOther = 80;
constexpr uint32_t kRegsEpilogue = 64;
constexpr int kLaunchRegs = 128;

template <int D>
struct Tc2Cfg {
    static constexpr int kHalves = D / 64;          // 64-element (128 B) column chunks
    static constexpr int kTileBytes = 128 * D * 2;  // 128 rows of D bf16 (a Q, K or V tile)
    static constexpr int kHalfBytes = kTileBytes / kHalves;
    static constexpr int kQSlots = 3;  // a unit's Q tiles take the next one or two
    static constexpr int kKStages = (D == 128) ? 2 : 6;
    static constexpr int kVStages = (D == 128) ? 2 : 4;
    // Q_A, Q_B, the K ring, the V ring; the barriers and small arrays follow
    static constexpr int kTileArea = kTileBytes * (kQSlots + kKStages + kVStages);
    static constexpr uint32_t kTmemO = 256;         // O_A; O_B at kTmemO + D
};

struct __align__(8) Tc2Shared {
    uint64_t q_full[3], q_empty[3];  // per Q slot
    uint64_t k_full[6], k_empty[6];
    uint64_t v_full[4], v_empty[4];
    uint64_t v_ready[4];             // a V tile may be read: landed, partial rows zeroed
    uint64_t s_full[2];              // per query tile: S_X(j) is in TMEM
    uint64_t p_full[2];              // P_X(j) written (one arrival per softmax warp of X)
    uint64_t o_full[2], o_empty[2];  // a unit's O_X complete / read by the epilogue
    uint64_t epi_full, epi_empty;    // row maxima and sums handed to the epilogue
    uint64_t mma_done;
    UnitRing ring;
    uint32_t tmem_base;
    int abort_flag;
    float epi_m[256], epi_l[256];
};

// How a unit's work splits over the two pipelines (X = A, B: score buffer
// S_X, output O_X, softmax warps 4X .. 4X + 3).
//   Row pair (more than 128 rows): pipeline A takes query tile A (rows
//   0-127), B takes tile B (rows 128 .. rows - 1); both walk the unit's key
//   tiles in order and share every K / V tile.  Tile A's rows are earlier
//   tokens: its key tiles are a prefix of the unit's.
//   Key split (at most 128 rows: decodes, small chunks, a request's odd last
//   query tile): both pipelines take the one query tile, A the even key
//   tiles and B the odd ones, each with its own running maximum and sum;
//   the epilogue merges the two.
struct UnitShape {
    bool key_split;
    int nt0, nt1;  // key tiles pipelines A and B process
};
__device__ __forceinline__ UnitShape unit_shape(const AttnArgs &a, const Unit &u, const TileList &tl) {
    UnitShape s;
    const int n = tl.n_total;
    s.key_split = u.rows <= kTcTileM;
    if (s.key_split) {
        s.nt0 = (n + 1) / 2;
        s.nt1 = n / 2;
    } else {
        const int last_tok_a = (u.row0 + kTcTileM - 1) / a.G;
        s.nt0 = tl.tiles_until(u.C + last_tok_a + 1);
        s.nt1 = n;
    }
    return s;
}

template <int D>
__global__ void __launch_bounds__(kThreads2, 1)
    attn_tc2_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k_new, const __grid_constant__ CUtensorMap tm_v_new,
                    const __grid_constant__ CUtensorMap tm_k_pool, const __grid_constant__ CUtensorMap tm_v_pool) {
    using Cfg = Tc2Cfg<D>;
    constexpr int NSK = Cfg::kKStages;
    constexpr int NSV = Cfg::kVStages;
    constexpr int TB = Cfg::kTileBytes;
    constexpr int HB = Cfg::kHalfBytes;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // The 128-byte swizzled tiles need a 1024-byte aligned base; the kernel
    // declares no static shared memory, so the dynamic area starts aligned.
    // Checked (uniformly, before any barrier) rather than padded: the tiles
    // leave no room for a pad.
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) record_error(a.err, kErrTimeout);
        return;
    }
    uint8_t *sQ = smem_raw;  // Cfg::kQSlots Q slots
    uint8_t *sK = smem_raw + Cfg::kQSlots * TB;
    uint8_t *sV = sK + NSK * TB;
    Tc2Shared &sh = *reinterpret_cast<Tc2Shared *>(smem_raw + Cfg::kTileArea);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const long long LIM = a.timeout_cycles;
    const int total_units = attention_units(a);
    const int end_index = total_units + a.write_chunks;  // then the fused K/V write

    if (tid == 0) {
        for (int q = 0; q < Cfg::kQSlots; ++q) {
            mbar_init(&sh.q_full[q], 1);
            mbar_init(&sh.q_empty[q], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&sh.s_full[x], 1);
            mbar_init(&sh.p_full[x], 4);  // the four softmax warps of the tile
            mbar_init(&sh.o_full[x], 1);
            mbar_init(&sh.o_empty[x], 4);  // the four epilogue warps
        }
        for (int s = 0; s < NSK; ++s) {
            mbar_init(&sh.k_full[s], 1);
            mbar_init(&sh.k_empty[s], 1);
        }
        for (int s = 0; s < NSV; ++s) {
            mbar_init(&sh.v_full[s], 1);
            mbar_init(&sh.v_empty[s], 1);
            mbar_init(&sh.v_ready[s], 1);
        }
        mbar_init(&sh.epi_full, 8);   // one arrival per softmax warp
        mbar_init(&sh.epi_empty, 4);  // one per epilogue warp
        mbar_init(&sh.mma_done, 1);
        for (int i = 0; i < kUnitRing; ++i) {
            mbar_init(&sh.ring.full[i], 1);
            mbar_init(&sh.ring.empty[i], kReaders2);
        }
        sh.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp2) {
        tmem_alloc(&sh.tmem_base, 512);
        tmem_relinquish();
    }
    if (warp == kKWarp && lane == 0) {
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
    // The register split is set per warpgroup, one setmaxnreg each, at the
    // top of that warpgroup's branch: warps 8-15 give registers back before
    // warps 0-7 can take them.
    if (warp >= 8 && warp < kEpiWarp2) {
        regs_dec<kRegsOther>();
        if (warp == kKWarp || warp == kVWarp) {
            // ============================================================ K, V
            const int kv = (warp == kVWarp) ? 1 : 0;
            bool ok = true;
            const int ns = kv ? NSV : NSK;
            uint64_t *const ring_full = kv ? sh.v_full : sh.k_full;
            uint64_t *const ring_empty = kv ? sh.v_empty : sh.k_empty;
            uint8_t *const ring = kv ? sV : sK;
            int slot = 0;     // ring slot of the next copy
            uint32_t ph = 0;  // parity of that slot's current fill
            int pending = 0;  // fills issued and not yet drained (<= ns)
            // V: the rows of a partial tile past its valid keys are zeroed once
            // the copy has landed (eight lanes per 128-byte row, four rows at
            // a time, then a proxy fence: the MMA reads through the async
            // proxy), and only then is the tile ready.  The zeroing waits for
            // the copy, so it is put off until the next copy has been issued
            // (or the unit ring shows no attention work) and the V stream keeps
            // a copy in flight meanwhile.
            int zero_slot = -1, zero_valid = 0;
            uint32_t zero_ph = 0;
            auto zero_deferred = [&]() -> bool {
                if (zero_slot < 0) return true;
                if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&ring_full[zero_slot], zero_ph, LIM, abort_flag)))
                    return false;
                uint8_t *vs = ring + zero_slot * TB + (lane & 7) * 16;
                for (int r = zero_valid + (lane >> 3); r < kKT; r += 4) {
#pragma unroll
                    for (int h = 0; h < Cfg::kHalves; ++h)
                        *reinterpret_cast<uint4 *>(vs + h * HB + r * 128) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.v_ready[zero_slot]);
                zero_slot = -1;
                return true;
            };
            // warp 8 also schedules: lane 0 claims the next unit once the
            // current unit's K copies are all issued, and publishes it
            int taken = (kv == 0 && lane == 0) ? atomicAdd(a.sched, 1) : 0;
            for (int it = 0;; ++it) {
                int unit;
                Unit u;
                if (kv == 0) {
                    unit = __shfl_sync(0xffffffffu, taken, 0);
                    const int s = it % kUnitRing;
                    if (it >= kUnitRing &&
                        !__all_sync(0xffffffffu, mbar_wait_or_abort(&sh.ring.empty[s],
                                                                    (uint32_t)((it / kUnitRing - 1) & 1), LIM, abort_flag))) {
                        ok = false;
                        break;
                    }
                    if (unit < total_units) decode_unit(a, unit, u);
                    if (lane == 0) {
                        publish_unit(sh.ring, it, unit, u);
                        if (unit >= total_units && unit < end_index) taken = atomicAdd(a.sched, 1);
                    }
                } else {
                    unit = read_unit(sh.ring, it, LIM, abort_flag, u);
                    if (unit < 0) {
                        ok = false;
                        break;
                    }
                }
                if (unit >= total_units && kv == 1 && !zero_deferred()) {
                    // no attention work follows in this CTA: the last partial
                    // tile is zeroed now (the unit ring may not advance until
                    // the softmax warps finish with it)
                    ok = false;
                    break;
                }
                if (unit >= end_index) break;
                if (unit >= total_units) continue;  // a piece of the K/V write: the softmax warps' job
                if (__any_sync(0xffffffffu, !ok || *abort_flag)) break;
                TileList tl;
                tl.init(u);
                const int n = tl.n_total;
                const bool hinted = a.interleave && u.piece >= 0;
                const uint64_t pol = hinted ? policy_evict_first() : 0;
                const int32_t *bt_row = a.bt + (long long)u.r * a.max_blocks;
                for (int j = 0; j < n && ok; ++j) {
                    uint64_t *empty = &ring_empty[slot];
                    uint64_t *full = &ring_full[slot];
                    uint8_t *dst = ring + slot * TB;
                    if (!__all_sync(0xffffffffu, mbar_wait_or_abort(empty, ph ^ 1u, LIM, abort_flag))) {
                        ok = false;
                        break;
                    }
                    int key0, valid;
                    bool pooled;
                    tl.tile(j, key0, valid, pooled);
                    if (a.test_stall && it == 0 && j == 0 && kv == 0) {
                        // testing only: arm the barrier but never copy, so the
                        // MMA warp's bounded wait on this tile expires
                        if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)TB);
                    } else if (pooled) {
                        // one box per cache block and 64-column half
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
                            if (hinted)
                                tma_load_4d_hint(dst + h * HB + b * a.bs * 128, kv ? &tm_v_pool : &tm_k_pool, full,
                                                 h * 64, u.g, 0, blk, pol);
                            else
                                tma_load_4d(dst + h * HB + b * a.bs * 128, kv ? &tm_v_pool : &tm_k_pool, full, h * 64,
                                            u.g, 0, blk);
                        }
                    } else {
                        if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)TB);
                        __syncwarp();
                        const int row = u.cu0 + (key0 - u.C);
                        if (lane < Cfg::kHalves)
                            tma_load_3d(dst + lane * HB, kv ? &tm_v_new : &tm_k_new, full, lane * 64, u.g, row);
                    }
                    const int filled = slot;
                    const uint32_t filled_ph = ph;
                    if (++slot == ns) {
                        slot = 0;
                        ph ^= 1u;
                    }
                    if (pending < ns) ++pending;
                    if (kv == 1) {
                        // the previous partial tile, now that this copy is in flight
                        if (!zero_deferred()) {
                            ok = false;
                            break;
                        }
                        if (valid < kKT) {
                            zero_slot = filled;
                            zero_ph = filled_ph;
                            zero_valid = valid;
                        } else {
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&sh.v_ready[filled]);  // full: ready when it lands
                        }
                    }
                }
                if (kv == 0 && lane == 0) taken = atomicAdd(a.sched, 1);  // this unit's K copies are all issued
            }
            if (!ok) {
                if (lane == 0) record_error(a.err, kErrTimeout);
                *abort_flag = 1;
            }
            // drain: every issued copy must land before the CTA may exit
            for (int i = pending; i >= 1; --i) {
                int st = slot - i;
                uint32_t p = ph;
                if (st < 0) {
                    st += ns;
                    p ^= 1u;
                }
                mbar_wait(&ring_full[st], p, LIM);
            }
            __syncwarp();
        } else if (warp == kQWarp) {
            // ============================================================== Q
            // A unit's query tiles go to the next one or two of three Q slots
            // (tile A, then tile B of a row pair), so the next unit's tile A
            // lands in the slot no running unit holds while this one runs.
            bool ok = true;
            uint32_t qpos = 0;      // Q slots handed out
            uint32_t filled = 0;    // bit q: slot q has been filled
            uint32_t fill_par = 0;  // bit q: parity of slot q's fills
            auto load_q = [&](int tok, int g) -> bool {
                const int q = (int)(qpos % Cfg::kQSlots);
                // the slot's previous tile must be done with: the commit after
                // the last S MMA that read it
                if (((filled >> q) & 1u) &&
                    !__all_sync(0xffffffffu, mbar_wait_or_abort(&sh.q_empty[q], ((fill_par >> q) & 1u) ^ 1u, LIM,
                                                                abort_flag)))
                    return false;
                if (lane == 0) mbar_arrive_expect_tx(&sh.q_full[q], (uint32_t)TB);
                __syncwarp();
                if (lane < Cfg::kHalves)
                    tma_load_3d(sQ + q * TB + lane * HB, &tm_q, &sh.q_full[q], lane * 64, g * a.G, tok);
                filled |= 1u << q;
                fill_par ^= 1u << q;
                ++qpos;
                return true;
            };
            for (int it = 0;; ++it) {
                Unit u;
                const int unit = read_unit(sh.ring, it, LIM, abort_flag, u);
                if (unit < 0) {
                    ok = false;
                    break;
                }
                if (unit >= end_index) break;
                if (unit >= total_units) continue;
                if (__any_sync(0xffffffffu, !ok || *abort_flag)) break;
                const int ntiles = u.rows > kTcTileM ? 2 : 1;
                const int tok0 = u.cu0 + u.row0 / a.G;
                const int tok_per_tile = kTcTileM / a.G;
                // into L2 now; the copies below wait for their slots
                if (lane < ntiles * Cfg::kHalves)
                    tma_prefetch_l2_3d(&tm_q, (lane % Cfg::kHalves) * 64, u.g * a.G,
                                       tok0 + (lane / Cfg::kHalves) * tok_per_tile);
                if (!load_q(tok0, u.g) || (ntiles == 2 && !load_q(tok0 + tok_per_tile, u.g))) {
                    ok = false;
                    break;
                }
            }
            if (!ok) {
                if (lane == 0) record_error(a.err, kErrTimeout);
                *abort_flag = 1;
            }
            // drain: every slot's last copy must land before the CTA may exit
            for (int q = 0; q < Cfg::kQSlots; ++q)
                if ((filled >> q) & 1u) mbar_wait(&sh.q_full[q], ((fill_par >> q) & 1u) ^ 1u, LIM);
            __syncwarp();
        } else if (warp == kMmaWarp2) {
            // ============================================================ MMA
            bool ok = true;
            constexpr uint32_t idesc_s = idesc_bf16_f32(128, kKT, 0, 0);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, 0, 1);
            const uint64_t q_desc = smem_desc(smem_u32(sQ), 16, 1024, kSwizzle128B);
            const uint32_t desc_hi = (uint32_t)(q_desc >> 32);
            const uint32_t q_lo0 = (uint32_t)q_desc;
            const uint32_t k_lo0 = (uint32_t)smem_desc(smem_u32(sK), 16, 1024, kSwizzle128B);
            const uint32_t v_lo0 = (uint32_t)smem_desc(smem_u32(sV), HB, 1024, kSwizzle128B);
            uint32_t k_it = 0, v_it = 0;     // K / V tiles consumed (ring position)
            uint32_t qpos = 0;     // Q slots taken (as the Q warp hands them out)
            uint32_t q_par = 0;    // bit q: parity of the uses of Q slot q
            uint32_t pv_cnt_a = 0, pv_cnt_b = 0;  // PV_X issued (p_full parity)
            uint32_t o_use_a = 0, o_use_b = 0;    // units that accumulated into O_X
            auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
                if (__all_sync(0xffffffffu, mbar_wait_or_abort(bar, parity, LIM, abort_flag))) return true;
                ok = false;
                return false;
            };
            // S_X(j) = Q K(kt)^T into S_X (Q: the unit's tile X, or tile A for
            // both pipelines of a key-split unit), then its commit
            auto issue_s = [&](int x, uint32_t qd, uint32_t k_lo) {
                if constexpr (D == 128) {
                    umma_s_tile128(tmem + x * kKT, qd, k_lo, desc_hi, idesc_s, (uint32_t)(HB >> 4));
                } else {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (uint32_t)(((kk >> 2) * HB + (kk & 3) * 32) >> 4);
                        umma_ss_warp2(tmem + x * kKT, qd + off, k_lo + off, desc_hi, idesc_s, kk > 0 ? 1u : 0u);
                    }
                }
                umma_commit_warp(&sh.s_full[x]);
            };
            const TileList *tl_cur = nullptr;  // the unit being issued (for the V tiles' valid keys)
            // O_X += P_X(j) V(vt) once the softmax has written P_X(j).  The
            // first PV to read a V tile waits for it: for a full tile until it
            // has landed, for a partial one until its rows past the valid keys
            // are zeroed too (which the V producer does after it has landed).
            auto issue_pv = [&](int x, int j, uint32_t vt, int vtile, bool first, uint32_t &pv_cnt,
                                uint32_t o_use) -> bool {
                const int vs = (int)(vt % NSV);
                if (first) {
                    int key0, valid;
                    bool pooled;
                    tl_cur->tile(vtile, key0, valid, pooled);
                    if (!wait(valid < kKT ? &sh.v_ready[vs] : &sh.v_full[vs], (vt / NSV) & 1u)) return false;
                }
                if (j == 0 && o_use >= 1 && !wait(&sh.o_empty[x], (o_use - 1) & 1u)) return false;
                if (!wait(&sh.p_full[x], pv_cnt & 1u)) return false;
                tc_fence_after();
                const uint32_t v_lo = v_lo0 + (uint32_t)vs * (uint32_t)(TB >> 4);
                const uint32_t tP = tmem + x * kKT;
                const uint32_t tO = tmem + Cfg::kTmemO + x * D;
                umma_pv_tile128(tO, tP, v_lo, desc_hi, idesc_pv, j > 0 ? 1u : 0u);
                ++pv_cnt;
                return true;
            };
            for (int ucnt = 0;; ++ucnt) {
                Unit u;
                const int unit = read_unit(sh.ring, ucnt, LIM, abort_flag, u);
                if (unit < 0) {
                    ok = false;
                    break;
                }
                if (unit >= end_index) break;
                if (unit >= total_units) continue;
                if (__any_sync(0xffffffffu, !ok || *abort_flag)) break;
                TileList tl;
                tl.init(u);
                tl_cur = &tl;
                const int n = tl.n_total;
                const UnitShape us = unit_shape(a, u, tl);
                const bool ks = us.key_split;
                // S_X(j) and PV_X(j) read key tile key_tile(x, j) of the unit
                auto key_tile = [&](int x, int j) -> uint32_t { return (uint32_t)(ks ? 2 * j + x : j); };
                const int steps = ks ? us.nt0 : n;
                // Q slots of tile A and (row pair) tile B, as the Q warp filled them
                const int qa = (int)(qpos % Cfg::kQSlots), qb = (int)((qpos + 1) % Cfg::kQSlots);
                const uint32_t qa_lo = q_lo0 + (uint32_t)qa * (uint32_t)(TB >> 4);
                const uint32_t qb_lo = q_lo0 + (uint32_t)qb * (uint32_t)(TB >> 4);
                // K(kt) is freed after its last S: S_B in row pairs, the one S otherwise
                const bool k_after_a = ks || us.nt1 == 0;
                for (int j = 0; j < steps && ok; ++j) {
                    if (j < us.nt0) {
                        const uint32_t kt = k_it + key_tile(0, j);
                        const int ks_ = (int)(kt % NSK);
                        if (!wait(&sh.k_full[ks_], (kt / NSK) & 1u)) break;
                        if (j == 0 && !wait(&sh.q_full[qa], (q_par >> qa) & 1u)) break;
                        tc_fence_after();
                        issue_s(0, qa_lo, k_lo0 + (uint32_t)ks_ * (uint32_t)(TB >> 4));
                        if (k_after_a) umma_commit_warp(&sh.k_empty[ks_]);
                        // Q_A is free after the last S that reads it
                        if ((int)key_tile(0, j) == (ks ? n - 1 : us.nt0 - 1)) umma_commit_warp(&sh.q_empty[qa]);
                    }
                    // PV_B(j - 1): tile B is the last reader of its V tile
                    if (j >= 1 && j - 1 < us.nt1) {
                        const uint32_t vt = v_it + key_tile(1, j - 1);
                        if (!issue_pv(1, j - 1, vt, (int)key_tile(1, j - 1), ks || j - 1 >= us.nt0, pv_cnt_b, o_use_b))
                            break;
                        umma_commit_warp(&sh.v_empty[vt % NSV]);
                        if (j - 1 == us.nt1 - 1) umma_commit_warp(&sh.o_full[1]);  // O_B complete
                    }
                    if (j < us.nt1) {
                        const uint32_t kt = k_it + key_tile(1, j);
                        const int ks_ = (int)(kt % NSK);
                        // a key-split unit's own K tile; in a row pair, K(j) when
                        // tile A's keys ended before it
                        if ((ks || j >= us.nt0) && !wait(&sh.k_full[ks_], (kt / NSK) & 1u)) break;
                        if (!ks && j == 0 && !wait(&sh.q_full[qb], (q_par >> qb) & 1u)) break;
                        tc_fence_after();
                        issue_s(1, ks ? qa_lo : qb_lo, k_lo0 + (uint32_t)ks_ * (uint32_t)(TB >> 4));
                        umma_commit_warp(&sh.k_empty[ks_]);
                        if (ks ? (int)key_tile(1, j) == n - 1 : j == us.nt1 - 1)
                            umma_commit_warp(&sh.q_empty[ks ? qa : qb]);
                    }
                    if (j < us.nt0) {
                        const uint32_t vt = v_it + key_tile(0, j);
                        if (!issue_pv(0, j, vt, (int)key_tile(0, j), true, pv_cnt_a, o_use_a)) break;
                        if (k_after_a) umma_commit_warp(&sh.v_empty[vt % NSV]);
                        if (j == us.nt0 - 1) umma_commit_warp(&sh.o_full[0]);  // O_A complete
                    }
                }
                if (ok && us.nt1 > 0 && steps - 1 < us.nt1) {
                    // the last PV_B, after the loop
                    const uint32_t vt = v_it + key_tile(1, steps - 1);
                    if (issue_pv(1, steps - 1, vt, (int)key_tile(1, steps - 1), ks || steps - 1 >= us.nt0, pv_cnt_b,
                                 o_use_b)) {
                        umma_commit_warp(&sh.v_empty[vt % NSV]);
                        umma_commit_warp(&sh.o_full[1]);
                    }
                }
                if (!ok) break;
                q_par ^= 1u << qa;
                if (!ks) q_par ^= 1u << qb;
                qpos += ks ? 1 : 2;
                ++o_use_a;
                if (us.nt1 > 0) ++o_use_b;
                k_it += (uint32_t)n;
                v_it += (uint32_t)n;
            }
            if (!ok) {
                if (lane == 0) record_error(a.err, kErrTimeout);
                *abort_flag = 1;
            }
            // every MMA issued so far must finish before TMEM is freed
            umma_commit_warp(&sh.mma_done);
            mbar_wait(&sh.mma_done, 0, LIM);
            __syncwarp();
        }
    } else if (warp >= kEpiWarp2) {
        regs_dec<kRegsEpilogue>();
        // ======================================================= epilogue
        const int e = warp - kEpiWarp2;
        bool ok = true;
        uint32_t o_use_a = 0, o_use_b = 0;  // units whose O_A / O_B this warp has read
        uint32_t ecnt = 0;
        auto wait_o = [&](int x, uint32_t &o_use) -> bool {
            if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&sh.o_full[x], o_use & 1u, LIM, abort_flag))) return false;
            ++o_use;
            return true;
        };
        // One output row (or a split unit's fp32 partial) from O_X, or, with
        // wb != 0, from wa O_A + wb O_B; then O_X (and O_B) are released.
        auto emit = [&](const Unit &u, int x, int lr, bool merge, float M, float L, float wa, float wb) {
            const bool row_valid = lr < u.rows;
            const bool warp_rows = __any_sync(0xffffffffu, row_valid);
            const uint32_t tO = tmem + ((uint32_t)(32 * e) << 16) + Cfg::kTmemO + x * D;
            const int pr = u.row0 + lr;  // packed row of the request
            const long long t = u.cu0 + pr / a.G;
            const int h = u.g * a.G + pr % a.G;
            const bool partial = u.piece >= 0;  // a split unit's unnormalised fp32 row
            const float inv = partial ? 1.f : 1.f / L;
#pragma unroll 1
            for (int c = 0; c < D / 16 && warp_rows; ++c) {
                uint32_t r[16];
                tmem_ld16(tO + c * 16, r);
                if (merge) {
                    uint32_t rb[16];
                    tmem_ld16(tO + D + c * 16, rb);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        r[i] = __float_as_uint(fmaf(wb, __uint_as_float(rb[i]), wa * __uint_as_float(r[i])));
                } else {
                    tmem_wait_ld();
                }
                if (!row_valid) continue;
                if (partial) {
                    float4 *d4 = reinterpret_cast<float4 *>(a.ws + u.ws_off + (long long)lr * D + c * 16);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        d4[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                            __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
                } else {
                    uint4 *d = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) + (t * a.hq + h) * D);
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        uint4 w;
                        w.x = pack_bf16(__uint_as_float(r[8 * i + 0]) * inv, __uint_as_float(r[8 * i + 1]) * inv);
                        w.y = pack_bf16(__uint_as_float(r[8 * i + 2]) * inv, __uint_as_float(r[8 * i + 3]) * inv);
                        w.z = pack_bf16(__uint_as_float(r[8 * i + 4]) * inv, __uint_as_float(r[8 * i + 5]) * inv);
                        w.w = pack_bf16(__uint_as_float(r[8 * i + 6]) * inv, __uint_as_float(r[8 * i + 7]) * inv);
                        d[2 * c + i] = w;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sh.o_empty[x]);
                if (merge) mbar_arrive(&sh.o_empty[1]);
            }
            if (row_valid) {
                if (partial) {
                    float *ws = a.ws + u.ws_off;
                    ws[(long long)u.rows * D + lr] = L > 0.f ? M : -INFINITY;
                    ws[(long long)u.rows * D + u.rows + lr] = L;
                } else if (a.lse) {
                    a.lse[t * a.hq + h] = (M + __log2f(L)) * 0.69314718055994531f;
                }
            }
        };
        for (int it = 0;; ++it) {
            Unit u;
            const int unit = read_unit(sh.ring, it, LIM, abort_flag, u);
            if (unit < 0) {
                ok = false;
                break;
            }
            if (unit >= end_index) break;
            if (unit >= total_units) continue;
            if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&sh.epi_full, ecnt & 1u, LIM, abort_flag))) {
                ok = false;
                break;
            }
            const float m0 = sh.epi_m[32 * e + lane], l0 = sh.epi_l[32 * e + lane];
            const float m1 = sh.epi_m[128 + 32 * e + lane], l1 = sh.epi_l[128 + 32 * e + lane];
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.epi_empty);
            ++ecnt;
            TileList tl;
            tl.init(u);
            const UnitShape us = unit_shape(a, u, tl);
            if (!us.key_split) {
                // a row pair: one output row from each pipeline
                if (!wait_o(0, o_use_a)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                emit(u, 0, 32 * e + lane, false, m0, l0, 1.f, 0.f);
                if (!wait_o(1, o_use_b)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                emit(u, 1, 128 + 32 * e + lane, false, m1, l1, 1.f, 0.f);
            } else if (us.nt1 == 0) {
                // a key split with one key tile: pipeline A alone
                if (!wait_o(0, o_use_a)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                emit(u, 0, 32 * e + lane, false, m0, l0, 1.f, 0.f);
            } else {
                // a key split: the row from both pipelines, merged with the
                // online-softmax rescale -- M = max(m_A, m_B), w_X = 2^(m_X - M)
                // (0 for a pipeline that saw no key of the row), O = w_A O_A +
                // w_B O_B, l = w_A l_A + w_B l_B
                if (!wait_o(0, o_use_a) || !wait_o(1, o_use_b)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float M = fmaxf(m0, m1);
                const float wa = l0 > 0.f ? ex2(m0 - M) : 0.f;
                const float wb = l1 > 0.f ? ex2(m1 - M) : 0.f;
                emit(u, 0, 32 * e + lane, true, M, wa * l0 + wb * l1, wa, wb);
            }
        }
        if (!ok) {
            if (lane == 0) record_error(a.err, kErrTimeout);
            *abort_flag = 1;
        }
    } else {
        regs_inc<kRegsSoftmax>();
        // ======================================================== softmax
        const int x = warp >> 2;  // query tile
        const int lr = 32 * (warp & 3) + lane;  // row of the tile == TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        const uint32_t tS = lane_base + x * kKT;
        const uint32_t tO = lane_base + Cfg::kTmemO + x * D;
        const float sl = a.scale_log2;
        uint32_t tcnt = 0;  // tiles of this pipeline processed (s_full phases)
        uint32_t ecnt = 0;  // units handed to the epilogue
        bool ok = true;
        for (int it = 0;; ++it) {
            Unit u;
            const int unit = read_unit(sh.ring, it, LIM, abort_flag, u);
            if (unit < 0) {
                ok = false;
                break;
            }
            if (unit >= end_index) break;
            if (unit >= total_units) {
                // a piece of the fused K/V write (this kernel reads new keys
                // from k_new / v_new, so the pool rows are only for the next
                // call); CTAs take these once attention work runs out
                const long long total = (long long)a.total_tokens * a.hkv * (D * 2 / 16);
                const long long b = (long long)(unit - total_units) * kWriteChunkPieces;
                const long long e = b + kWriteChunkPieces < total ? b + kWriteChunkPieces : total;
                scatter_new_kv(a.cached, a.cu, a.bt, a.num_reqs, a.max_blocks, a.hkv, a.bs, a.num_blocks, D * 2,
                               a.k_new, a.v_new, a.k_cache, a.v_cache, b, e, tid, kSoftmaxThreads2, a.err);
                continue;
            }
            if (__any_sync(0xffffffffu, !ok || *abort_flag)) break;
            TileList tl;
            tl.init(u);
            const UnitShape us = unit_shape(a, u, tl);
            const int nx = x ? us.nt1 : us.nt0;
            const int prow = us.key_split ? lr : x * 128 + lr;  // row of the unit
            const bool row_valid = prow < u.rows;
            const int pos = row_valid ? u.C + (u.row0 + prow) / a.G : -1;
            // a warp whose 32 rows are all padding skips the math; each O row
            // depends on its own P row only
            const bool warp_rows = __any_sync(0xffffffffu, row_valid);
            float m_ref = -INFINITY, l = 0.f;
            for (int j = 0; j < nx; ++j, ++tcnt) {
                if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&sh.s_full[x], tcnt & 1u, LIM, abort_flag))) {
                    ok = false;
                    break;
                }
                if (warp_rows) {
                    tc_fence_after();
                    int key0, valid;
                    bool pooled;
                    tl.tile(us.key_split ? 2 * j + x : j, key0, valid, pooled);
                    float s[128];
                    {
                        // all four loads in flight before the one wait
                        uint32_t r0[32], r1[32], r2[32], r3[32];
                        tmem_ld32(tS, r0);
                        tmem_ld32(tS + 32, r1);
                        tmem_ld32(tS + 64, r2);
                        tmem_ld32(tS + 96, r3);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            s[i] = __uint_as_float(r0[i]);
                            s[32 + i] = __uint_as_float(r1[i]);
                            s[64 + i] = __uint_as_float(r2[i]);
                            s[96 + i] = __uint_as_float(r3[i]);
                        }
                    }
                    // keys [0, lim) of the tile are visible to this row
                    const int lim = min(valid, pos - key0 + 1);
                    if (!__all_sync(0xffffffffu, lim >= kKT)) {
#pragma unroll
                        for (int k = 0; k < 128; ++k) s[k] = (k < lim) ? s[k] : -INFINITY;
                    }
                    // row maximum: eight independent max3 chains, then a tree
                    float mx[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c) mx[c] = s[c];
#pragma unroll
                    for (int k = 8; k < 120; k += 16) {
#pragma unroll
                        for (int c = 0; c < 8; ++c) mx[c] = max3(mx[c], s[k + 2 * c], s[k + 2 * c + 1]);
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c) mx[c] = max3(mx[c], s[120 + 2 * c], s[121 + 2 * c]);
                    const float tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) *
                                       sl;
                    const bool move =
                        (tmax > m_ref + kRescaleThreshold2) || (m_ref == -INFINITY && tmax > -INFINITY);
                    float alpha = 1.f;
                    if (move) {
                        alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - tmax);
                        m_ref = tmax;
                        l *= alpha;
                    }
                    const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref;
                    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
                    const float2 sl2 = make_float2(sl, sl), neg2 = make_float2(neg, neg);
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        // keys 64c .. 64c + 63 -> P columns 32c .. 32c + 31
                        uint32_t r[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const float2 xx =
                                __ffma2_rn(make_float2(s[64 * c + 2 * i], s[64 * c + 2 * i + 1]), sl2, neg2);
                            float2 ee;
                            ee.x = ex2(xx.x);
                            ee.y = ex2(xx.y);
                            if (i & 1)
                                acc1 = __fadd2_rn(acc1, ee);
                            else
                                acc0 = __fadd2_rn(acc0, ee);
                            r[i] = pack_bf16(ee.x, ee.y);
                        }
                        tmem_st32(tS + c * 32, r);
                    }
                    l += (acc0.x + acc0.y) + (acc1.x + acc1.y);
                    if (j >= 1 && __any_sync(0xffffffffu, move)) {
                        // rescale O: PV_X(j - 1) has completed, as the commit
                        // behind s_full (after S_X(j)) tracks every MMA the MMA
                        // warp issued before it; PV_X(j) cannot start before
                        // this warp's arrival below
#pragma unroll 1
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t r[32];
                            tmem_ld32(tO + c * 32, r);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                            tmem_st32(tO + c * 32, r);
                        }
                    }
                    tmem_wait_st();
                    tc_fence_before();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.p_full[x]);
            }
            if (!ok) break;
            // hand the rows' maxima and sums to the epilogue warps once they
            // have read the previous unit's
            if (ecnt >= 1 &&
                !__all_sync(0xffffffffu, mbar_wait_or_abort(&sh.epi_empty, (ecnt - 1) & 1u, LIM, abort_flag))) {
                ok = false;
                break;
            }
            sh.epi_m[x * 128 + lr] = m_ref;
            sh.epi_l[x * 128 + lr] = l;
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.epi_full);
            ++ecnt;
        }
        if (!ok) {
            record_error(a.err, kErrTimeout);
            *abort_flag = 1;
        }
    }
    // warp 11 done, every role drained: free TMEM
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp2) {
        __syncwarp();
        tmem_dealloc(tmem, 512);
    }
}

template <int D>
cudaError_t launch_tc2(const AttnArgs &a, const TcMaps &m, int grid, cudaStream_t stream) {
    constexpr int smem = Tc2Cfg<D>::kTileArea + (int)sizeof(Tc2Shared);
    // Set once per device: the shared-memory size, and a check that the
    // kernel was built for the 128 registers per thread the register split
    // draws on (a mismatch would leave setmaxnreg.inc waiting forever, so the
    // kernel is not launched then).
    static std::mutex attr_mutex;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lock(attr_mutex);
        if (dev < 0 || dev >= 64 || !attr_set[dev]) {
            cudaFuncAttributes fa{};
            e = cudaFuncGetAttributes(&fa, attn_tc2_kernel<D>);
            if (e != cudaSuccess) return e;
            if (fa.numRegs != kLaunchRegs || fa.sharedSizeBytes != 0) return cudaErrorInvalidConfiguration;
            e = cudaFuncSetAttribute(attn_tc2_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) attr_set[dev] = true;
        }
    }
    attn_tc2_kernel<D><<<grid, kThreads2, smem, stream>>>(a, m.q, m.k_new, m.v_new, m.k_pool, m.v_pool);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_tc2(const AttnArgs &a, const TcMaps &m, cudaStream_t stream) {
    const int grid = a.write_ctas;  // persistent: min(units + write pieces, SMs)
    if (grid <= 0 || attention_units(a) == 0) return cudaSuccess;
    // the one-pipeline kernel's cases (a.rope: fused RoPE; two CTA groups)
    if (a.rope || a.kv_fp8 || a.group_ctas) return cudaErrorNotSupported;
    return a.d == 128 ? launch_tc2<128>(a, m, grid, stream) : launch_tc2<64>(a, m, grid, stream);
}

}  // namespace cpa
