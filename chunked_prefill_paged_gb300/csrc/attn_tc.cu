// attn_tc.cu -- tensor-core (tcgen05 + TMEM + TMA) attention over the paged
// K/V cache: BF16 pools (attn_tc_kernel<D, false>) and FP8 E4M3 pools
// (attn_tc_kernel<128, true>).  Persistent: one CTA per SM takes work units
// (see cpa_internal.h) from a per-launch counter in the workspace, in index
// order (a request's heaviest units first), so that CTAs that finish early
// take more units.  For some prefill batches the planner splits the CTAs into
// two groups with a counter each (the heaviest units for one, the lightest
// for the other, claim_unit below), which packs the last wave better.
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
// Warp roles (384 threads; 512 with FP8 pools):
//   warps 0-7  softmax / correction / epilogue.  Two threads own one query
//              row: warp w covers TMEM lanes 32 (w % 4) + 16 (w / 4) .. +15,
//              its threads 0-15 the row's keys 0-63 (output columns 0 .. D/2-1)
//              and threads 16-31 keys 64-127 (columns D/2 .. D-1); the row
//              maximum and sum are combined with one shuffle.
//              With the rotary embedding they first rotate the launch's new
//              keys, once, from k_src into the workspace copy k_new that the
//              new-key tiles and the fused write read: pieces of 16 tokens
//              taken from their own counter, each counted done per 128-row
//              tile of the new rows, which the K copies of a new-key tile
//              wait for.
//   warp 8     unit scheduler (it claims each unit, decodes it once and passes
//              the decoded unit to the other roles through a ring) and TMA
//              producer of Q per unit and of the K tiles; warp 10 of the V
//              tiles, each into its own ring, so a V slot still in use never
//              holds up the next K copy.  A pool tile is one box per cache
//              block (found through the block table), a new-token tile one
//              128-row box of k_new / v_new.
//   warp 9     score MMA issuer: S(j) = Q K(j)^T into score buffer j % 3 as
//              soon as K(j) is in and the PV that last read that buffer has
//              completed, so scores run up to three tiles ahead of the PVs.
//   warp 11    PV MMA issuer: O += P(j) V(j) once the softmax has written P(j).
//              Issuing from two warps on different SM sub-partitions halves
//              the instruction stream each shares with the softmax warps.
//   warps 12-15 (BF16 pools) output epilogue; with the rotary embedding they
//              also rotate each unit's query tile in its Q stage once it has
//              landed, one unit ahead of the outputs, and the score MMAs wait
//              for that (q_rot) instead of the copy.  They also do the fused
//              K/V write, an even share per CTA while its first unit runs
//              (this kernel reads new keys from k_new / v_new, so the pool
//              rows are only needed by the next call).
//   warps 12-15 (FP8 pools) expand E4M3 value code tiles in place into the
//              fp16 tiles the PV MMAs read (32 rows each).  The score MMAs read
//              the key codes as they landed (E4M3 operands, .kind::f8f6f4), with
//              the queries as two E4M3 planes (a row and its rounding residual).
//
// TMEM (512 columns): three score buffers S0 [0,128), S1 [128,256) and
// S2 [256,384), O [384, 384 + D).  P(j), as bf16 (fp16) pairs, overwrites the first
// 64 columns of the buffer that held S(j); S(j+3) reuses that buffer only
// after PV(j) has completed.  With three buffers the chain softmax(j) ->
// PV(j) -> S(j+3) -> softmax(j+3) spans two other softmax tiles.  Rescaling is lazy:
// a row's reference maximum moves (and O is rescaled, after waiting for the
// previous PV) only when a tile's maximum exceeds it by more than 2^8 in the
// exp2 domain; the final O / l is exact whichever reference was used.
// Every mbarrier wait is bounded; on expiry the CTA records
// CPA_ERR_DEVICE_TIMEOUT, drains its copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <type_traits>

#include "device_common.cuh"
#include "launch.h"
#include "ptx_sm100.cuh"
#include "tc_common.cuh"

namespace cpa {
namespace {

using namespace ptx;
using namespace tc;

constexpr int kSoftmaxThreads = 256;  // warps 0-7
constexpr int kProducerWarp = 8;      // Q and K copies
constexpr int kMmaWarp = 9;
constexpr int kVProducerWarp = 10;    // V copies
constexpr int kPvWarp = 11;           // PV MMA issuer
constexpr int kSBuf = 3;              // score buffers in TMEM
constexpr uint32_t kTmemO = kSBuf * kKT;  // first TMEM column of O
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// BF16 pools: during a direct unit of at least kEarlyClaimMinTiles key tiles,
// and during every unit with the rotary embedding, the next unit is claimed
// after issuing the K copies of all but the last kClaimAhead + 1 tiles
// (measured on the 10k-token Llama prompt: the last chunk 0.194 -> 0.189 ms,
// with RoPE 0.200 -> 0.194 ms; shorter units, decode pieces among them, keep
// the late claim, which balances the launch's last wave better)
constexpr int kClaimAhead = 6;
constexpr int kEarlyClaimMinTiles = 24;
constexpr int kKConvWarp = 12;              // FP8 cache: warps 12-13 expand K tiles, 14-15 V tiles
constexpr int kEpiWarp = 12;                // BF16 cache: warps 12-15 write the outputs

// Roles of the two kernel flavours (16 warps each): with BF16 pools warps
// 12-15 take the output epilogue off the softmax warps; with FP8 pools they
// expand the codes and the softmax warps write the outputs themselves.
template <bool F8>
struct TcRoles {
    static constexpr int kThreads = 512;
    static constexpr int kUnitReaders = 15;  // every warp but 8 reads every index
    static constexpr bool kEpiWarps = !F8;
};

template <int D, bool F8>
struct TcCfg {
    static constexpr int kHalves = D / 64;           // 64-element (128 B) column chunks
    static constexpr int kTileBytes = 128 * D * 2;   // 128 rows of D 16-bit values (Q, K or V tile)
    static constexpr int kHalfBytes = kTileBytes / kHalves;
    // BF16 pools: two Q stages, so the next unit's Q loads while this one
    // runs.  FP8 pools: one, and a third V stage instead: there a V tile's
    // slot turns over through its code copy, the expansion and the PV, and
    // two stages left the PVs waiting (measured: mixed step 1.06 -> 0.99 ms,
    // 32 decodes 0.226 -> 0.215 ms; a K stage given up instead was slower)
    static constexpr int kQStages = F8 ? 1 : 2;
    static constexpr int kKStages = (D == 128) ? 3 : 6;
    static constexpr int kVStages = (D == 128) ? (F8 ? 3 : 2) : 5;
    // FP8 pools: a K copy brings a code tile (128 rows x D bytes, 128-byte
    // swizzled) to the start of its ring slot, where the score MMA reads it;
    // a V copy brings one (plain rows) into the upper half of its slot, and
    // the expansion warps turn it in place into the fp16 tile the PV MMA reads
    static constexpr int kCodeTileBytes = 128 * D;
    static constexpr int kSmemBytes = 1024 /*align*/ + kTileBytes * (kQStages + kKStages + kVStages);
};

struct __align__(8) TcShared {
    uint64_t q_full[2], q_empty[2];
    uint64_t q_rot[2];  // rotary embedding: the stage's queries are rotated (four epilogue warps)
    uint64_t k_full[6], k_empty[6];
    uint64_t v_full[6], v_empty[6];
    uint64_t s_full[kSBuf];  // per score buffer
    uint64_t p_full[kSBuf];  // per score buffer: P(j) written over S(j)
    uint64_t pv_done[kSBuf];  // per score buffer: the PV that read its P has completed
    uint64_t o_full, o_empty;
    uint64_t mma_done;
    // BF16 pools: the softmax warps hand each finished unit's row maxima and
    // sums to the epilogue warps (epi_full), which free the arrays once read
    uint64_t epi_full, epi_empty;
    float epi_m[128], epi_l[128];
    uint64_t v8_full[6];  // FP8 pools: a V slot's code tile has landed
    // unit scheduler: warp 8 takes unit indices from the launch's work
    // counter and passes them to the other roles through this ring
    UnitRing ring;
    uint32_t tmem_base;
    int abort_flag;
    int rope_claim;  // the softmax warps' current piece of the key rotation
};

// Four E4M3 codes (bytes of w, lowest address first) as fp16 pairs: codes
// 0, 1 in the first word, 2, 3 in the second, lower column in the low half.
// Every E4M3 value is an fp16 value (3 mantissa bits; exponents 2^-9 .. 2^8),
// so the conversion is exact.
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const unsigned short a = (unsigned short)(w & 0xffffu), b = (unsigned short)(w >> 16);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"(a));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"(b));
}

// Rows [r0, r0 + 32) of a 128 x 128 code tile, held in the upper half of its
// ring slot (rows of 128 bytes at slot + 16 KB), expanded in place into the
// 16-bit tile the MMAs read: two 64-column halves of 128 rows x 128 B at
// slot and slot + 16 KB, 16-byte chunk c of row r at chunk position
// c ^ (r % 8) (the 128-byte swizzle).  Half 1 of row r overwrites code row r
// only, so reading each row before writing it keeps the expansion in place;
// the eight rows of each lane are read before any of them is written (the
// loads then overlap), and the four warps of a tile own disjoint rows.
// Rows at or past `valid` become zeros (code 0).  Eight lanes share a row: lane piece p (16
// codes, columns 16p .. 16p + 15) fills chunks 2(p % 4) and 2(p % 4) + 1 of
// half p / 4.  Which of its two chunks a lane handles first alternates with
// the half and with the row's parity: then every store instruction covers all
// eight chunk positions of each row, and every 8-byte load instruction reads
// row pairs whose byte ranges fall on complementary banks -- neither
// conflicts.
__device__ __forceinline__ void expand_code_rows(uint8_t *slot, int r0, int valid, int lane, int half_bytes) {
    const uint8_t *codes = slot + half_bytes;
    const int p = lane & 7;
    const int h = p >> 2;
    const int f = h ^ ((lane >> 3) & 1);  // r0 is even, so (lane >> 3) & 1 is the row's parity
    const int c_first = 2 * (p & 3) + f, c_second = 2 * (p & 3) + 1 - f;
    constexpr int kBatch = 8;  // 8 x 4 = 32 rows, every load before any store
    {
        const int it0 = 0;
        uint2 w0[kBatch], w1[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int r = r0 + (it0 + i) * 4 + (lane >> 3);
            w0[i] = make_uint2(0, 0);
            w1[i] = make_uint2(0, 0);
            if (r < valid) {
                const uint8_t *in = codes + r * 128 + p * 16;
                w0[i] = *reinterpret_cast<const uint2 *>(in + 8 * f);        // codes of chunk c_first
                w1[i] = *reinterpret_cast<const uint2 *>(in + 8 * (1 - f));  // codes of chunk c_second
            }
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int r = r0 + (it0 + i) * 4 + (lane >> 3);
            uint4 o0, o1;
            e4m3x4_to_f16(w0[i].x, o0.x, o0.y);
            e4m3x4_to_f16(w0[i].y, o0.z, o0.w);
            e4m3x4_to_f16(w1[i].x, o1.x, o1.y);
            e4m3x4_to_f16(w1[i].y, o1.z, o1.w);
            uint8_t *row = slot + h * half_bytes + r * 128;
            const int sw = r & 7;
            *reinterpret_cast<uint4 *>(row + ((c_first ^ sw) << 4)) = o0;
            *reinterpret_cast<uint4 *>(row + ((c_second ^ sw) << 4)) = o1;
        }
    }
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// The 16 output rows [lr0, lr0 + 16) of a unit run as tail pieces, merged by
// one warp from the pieces' partials: each holds O_q = sum over its keys of
// 2^(s - m_q) v (times the value scale), m_q and l_q; a row is
// sum_q 2^(m_q - M) O_q / sum_q 2^(m_q - M) l_q with M the largest m_q of the
// pieces that saw a key.  Lane j < 16 forms row lr0 + j's weights; the rows
// are then read whole (D floats over the warp's lanes, from L2, where the
// other CTAs' partials are) and written as bf16.
template <int D>
__device__ __forceinline__ void merge_tail_rows(const AttnArgs &a, const Unit &u, int lr0, int lane) {
    constexpr int F = D / 4;     // float4 per row
    constexpr int RPP = 32 / F;  // rows per pass
    const int P = a.tail_pieces;
    const long long pf = partial_floats(a.tile_m, D);
    const float *base = a.ws + a.tail_ws + (long long)u.tail * P * pf;
    const long long ml = (long long)u.rows * D;  // row maxima, then sums
    float w[kMaxTailPieces];
    float inv;
    {
        const int r = lr0 + (lane & 15);
        const bool valid = r < u.rows;
        float mq[kMaxTailPieces], lq[kMaxTailPieces], M = -INFINITY;
#pragma unroll
        for (int q = 0; q < kMaxTailPieces; ++q) {
            lq[q] = (q < P && valid) ? __ldcg(base + q * pf + ml + u.rows + r) : 0.f;
            mq[q] = lq[q] > 0.f ? __ldcg(base + q * pf + ml + r) : -INFINITY;
            M = fmaxf(M, mq[q]);
        }
        float L = 0.f;
#pragma unroll
        for (int q = 0; q < kMaxTailPieces; ++q) {
            w[q] = lq[q] > 0.f ? ex2(mq[q] - M) : 0.f;
            L = fmaf(lq[q], w[q], L);
        }
        inv = L > 0.f ? 1.f / L : 0.f;
        if (lane < 16 && valid && a.lse) {
            const int pr = u.row0 + r;
            a.lse[(long long)(u.cu0 + pr / a.G) * a.hq + u.g * a.G + pr % a.G] =
                (M + __log2f(L)) * 0.69314718055994531f;
        }
    }
    const int sub = lane / F, f = lane % F;
#pragma unroll 4
    for (int i = 0; i < 16; i += RPP) {
        const int j = i + sub;
        float wj[kMaxTailPieces];
#pragma unroll
        for (int q = 0; q < kMaxTailPieces; ++q) wj[q] = __shfl_sync(0xffffffffu, w[q], j);
        const float invj = __shfl_sync(0xffffffffu, inv, j);
        const int r = lr0 + j;
        if (r < u.rows) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int q = 0; q < kMaxTailPieces; ++q) {
                if (q < P) {
                    const float4 v = __ldcg(reinterpret_cast<const float4 *>(base + q * pf + (long long)r * D) + f);
                    acc.x = fmaf(wj[q], v.x, acc.x);
                    acc.y = fmaf(wj[q], v.y, acc.y);
                    acc.z = fmaf(wj[q], v.z, acc.z);
                    acc.w = fmaf(wj[q], v.w, acc.w);
                }
            }
            const int pr = u.row0 + r;
            const long long t = u.cu0 + pr / a.G, h = u.g * a.G + pr % a.G;
            uint2 o;
            o.x = pack_bf16(acc.x * invj, acc.y * invj);
            o.y = pack_bf16(acc.z * invj, acc.w * invj);
            reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(a.out) + (t * a.hq + h) * D)[f] = o;
        }
    }
}

// Piece `piece` of the key rotation: new tokens [16 piece, 16 piece + 16) of
// every kv head, from k_src into k_new, by the 256 softmax threads.  Thread
// (tl, j, s) takes the pairs (c, c + D/2), c = 8 j .. 8 j + 7, of token tl's
// rows for kv heads s, s + S, ... (S threads per (token, j)): two 16-byte
// loads per row, every load of the piece in flight before the first store.
template <int D>
__device__ __forceinline__ void rope_keys_piece(const AttnArgs &a, int piece, int tid) {
    constexpr int J = D / 16;                            // 8-pair chunks of a row
    constexpr int S = kSoftmaxThreads / (kRopePieceTokens * J);  // threads per (token, chunk)
    constexpr int HB = 4;                                // heads per batch of loads
    static_assert(S >= 1 && S * kRopePieceTokens * J == kSoftmaxThreads, "one (token, chunk, s) per thread");
    const int s = tid % S, combo = tid / S;
    const int tl = combo / J, j = combo - tl * J;
    const int t = piece * kRopePieceTokens + tl;
    if (t >= a.total_tokens) return;
    const long long row0 = (long long)t * a.hkv * D + 8 * j;
    const __nv_bfloat16 *src = static_cast<const __nv_bfloat16 *>(a.k_src) + row0;
    __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(const_cast<void *>(a.k_new)) + row0;
    float cs[8], sn[8];
    for (int h0 = s; h0 < a.hkv; h0 += HB * S) {
        uint4 x[HB], y[HB];
#pragma unroll
        for (int i = 0; i < HB; ++i) {
            const int h = h0 + i * S;
            if (h < a.hkv) {
                x[i] = __ldg(reinterpret_cast<const uint4 *>(src + h * D));
                y[i] = __ldg(reinterpret_cast<const uint4 *>(src + h * D + D / 2));
            }
        }
        if (h0 == s) {
            // the position and the angles while the first rows load
            const int r = request_of_token(a.cu, a.num_reqs, t);
            const int pos = __ldg(a.cached + r) + (t - __ldg(a.cu + r));
#pragma unroll
            for (int k = 0; k < 8; ++k) rope_cos_sin(pos, a.turn_frac[8 * j + k], cs[k], sn[k]);
        }
#pragma unroll
        for (int i = 0; i < HB; ++i) {
            const int h = h0 + i * S;
            if (h >= a.hkv) break;
            const uint32_t xw[4] = {x[i].x, x[i].y, x[i].z, x[i].w}, yw[4] = {y[i].x, y[i].y, y[i].z, y[i].w};
            uint32_t ow[4], pw[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                // element 2k in the low half of word k
                float a0, b0, a1, b1;
                rope_turn(__uint_as_float(xw[k] << 16), __uint_as_float(yw[k] << 16), cs[2 * k], sn[2 * k], a0, b0);
                rope_turn(__uint_as_float(xw[k] & 0xffff0000u), __uint_as_float(yw[k] & 0xffff0000u), cs[2 * k + 1],
                          sn[2 * k + 1], a1, b1);
                ow[k] = pack_bf16(a0, a1);
                pw[k] = pack_bf16(b0, b1);
            }
            *reinterpret_cast<uint4 *>(dst + h * D) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
            *reinterpret_cast<uint4 *>(dst + h * D + D / 2) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
        }
    }
}

// Whether the key rotation's pieces of the new rows [row_begin, row_end) are
// done: waits (bounded)
// for the pieces of their 128-row tiles, or of the whole launch once `all`
// is known.  The calling thread's acquire orders its later reads after them.
__device__ __forceinline__ bool rope_rows_done(const AttnArgs &a, int row_begin, int row_end, bool &all,
                                               long long limit, const volatile int *abort_flag) {
    if (!all) {
        const long long t0 = clock64();
        for (;;) {
            if (ld_acquire_gpu(a.rope_count + 1) >= a.rope_pieces) {
                all = true;
                break;
            }
            bool have = true;
            for (int i = row_begin / kTcTileN; i <= (row_end - 1) / kTcTileN && have; ++i)
                have = ld_acquire_gpu(a.rope_count + 2 + i) >= rope_pieces_of_tile(a.total_tokens, i);
            if (have) break;
            if (*abort_flag || clock64() - t0 > limit) return false;
            __nanosleep(128);
        }
    }
    return true;
}

// As rope_rows_done, for the lane that then issues copies of the rotated
// rows: its proxy fence orders them before its TMA reads too.
__device__ __forceinline__ bool rope_rows_ready(const AttnArgs &a, int row_begin, int row_end, bool &all,
                                                long long limit, const volatile int *abort_flag) {
    if (!rope_rows_done(a, row_begin, row_end, all, limit, abort_flag)) return false;
    fence_proxy_async_global();
    return true;
}

// Rotate the queries of unit u in place in its Q stage (128 rows of D bf16
// values, in 64-column halves of 128-byte swizzled rows), by the 128
// epilogue threads (thread lr).  Item (tl, fc): the pairs (c, c + D/2), c =
// 8 fc .. 8 fc + 7, of the G rows of the tile's local token tl, all at
// position C + row0 / G + tl; thread lr takes items lr, lr + 128, ..., so
// its fc = lr mod D/16 is fixed, and it reads those pairs' turn rates once
// per tile.  The top 32 bits of pos * rate modulo 2^64 (the high word's
// product plus the carry-in from the low word's: exact to 2^-32 turn) give
// the angle, whose top 24 bits go to sincospif as for the keys, so the
// rotated queries round as an exact rotation's do but for rare ties.
// Elements c and c + D/2 sit in 16-byte chunks at the same place of their
// halves (D = 128) or four chunks apart in one half (D = 64).
template <int D>
__device__ __forceinline__ void rope_q_tile(const AttnArgs &a, const Unit &u, uint8_t *tile, int lr) {
    constexpr int FC = D / 16;
    constexpr int HB = 128 * 128;  // bytes of a 64-column half
    const int G = a.G;
    const int items = cdiv(u.rows, G) * FC;
    const int fc = lr % FC;
    uint32_t fh[8], fl[8];  // the pairs' turn rates, high and low words
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const unsigned long long f = a.turn_frac[fc * 8 + k];
        fh[k] = (uint32_t)(f >> 32);
        fl[k] = (uint32_t)f;
    }
    const int e0 = fc * 8, e1 = e0 + D / 2;
    const int off0 = (e0 >> 6) * HB, c0 = (e0 & 63) >> 3;
    const int off1 = (e1 >> 6) * HB, c1 = (e1 & 63) >> 3;
    for (int it = lr; it < items; it += 128) {
        const int tl = it / FC;
        const uint32_t pos = (uint32_t)(u.C + u.row0 / G + tl);
        float2 c2[4], s2[4];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            // the angle's top 24 bits (units of 2^-24 turn) as an exact float
            // x in [0, 2) half turns
            const uint32_t v = (pos * fh[k] + __umulhi(pos, fl[k])) >> 8;
            const float x = __uint2float_rn(v) * (1.0f / 8388608.0f);
            float sv, cv;
            sincospif(x, &sv, &cv);
            (k & 1 ? c2[k >> 1].y : c2[k >> 1].x) = cv;
            (k & 1 ? s2[k >> 1].y : s2[k >> 1].x) = sv;
        }
#pragma unroll 2
        for (int g = 0; g < G; ++g) {
            const int m = tl * G + g;
            uint4 *p0 = reinterpret_cast<uint4 *>(tile + off0 + m * 128 + ((c0 ^ (m & 7)) << 4));
            uint4 *p1 = reinterpret_cast<uint4 *>(tile + off1 + m * 128 + ((c1 ^ (m & 7)) << 4));
            const uint4 x = *p0, y = *p1;
            const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
            uint32_t ow[4], pw[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                // elements 2k (low half of word k) and 2k + 1: (x c - y s, y c + x s)
                const float2 xf = make_float2(__uint_as_float(xw[k] << 16), __uint_as_float(xw[k] & 0xffff0000u));
                const float2 yf = make_float2(__uint_as_float(yw[k] << 16), __uint_as_float(yw[k] & 0xffff0000u));
                const float2 o = __ffma2_rn(xf, c2[k], __fmul2_rn(yf, make_float2(-s2[k].x, -s2[k].y)));
                const float2 q = __ffma2_rn(yf, c2[k], __fmul2_rn(xf, s2[k]));
                ow[k] = pack_bf16(o.x, o.y);
                pw[k] = pack_bf16(q.x, q.y);
            }
            *p0 = make_uint4(ow[0], ow[1], ow[2], ow[3]);
            *p1 = make_uint4(pw[0], pw[1], pw[2], pw[3]);
        }
    }
}

// Work indices.  A CTA's first unit needs no atomic: CTA b starts with
// index b of its group (the grid is min(units, SMs), and a group of c CTAs
// holds at least c units).  Later claims take the group's next index past
// those, from its counter (zeroed before the launch), then, once the group
// has run out, the other group's; total_units when both have.
__device__ __forceinline__ int first_unit(const AttnArgs &a) {
    if (!a.group_ctas) return (int)blockIdx.x;
    return (int)blockIdx.x < a.group_ctas ? (int)blockIdx.x : a.group_units + ((int)blockIdx.x - a.group_ctas);
}
__device__ __forceinline__ int claim_unit(const AttnArgs &a, int total_units) {
    if (!a.group_ctas) return (int)gridDim.x + atomicAdd(a.sched, 1);
    const bool first = (int)blockIdx.x < a.group_ctas;
    const int b_ctas = (int)gridDim.x - a.group_ctas;
    for (int k = 0; k < 2; ++k) {
        if (first == (k == 0)) {
            const int i = a.group_ctas + atomicAdd(a.sched, 1);
            if (i < a.group_units) return i;
        } else {
            const int i = a.group_units + b_ctas + atomicAdd(a.sched_b, 1);
            if (i < total_units) return i;
        }
    }
    return total_units;
}

template <int D, bool F8>
__global__ void __launch_bounds__(TcRoles<F8>::kThreads, 1)
    attn_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k_new, const __grid_constant__ CUtensorMap tm_v_new,
                   const __grid_constant__ CUtensorMap tm_k_pool, const __grid_constant__ CUtensorMap tm_v_pool) {
    using Cfg = TcCfg<D, F8>;
    constexpr int NSK = Cfg::kKStages;
    constexpr int NSV = Cfg::kVStages;
    constexpr int TB = Cfg::kTileBytes;
    constexpr int HB = Cfg::kHalfBytes;
    constexpr int CB = Cfg::kCodeTileBytes;
    static_assert(!F8 || D == 128, "FP8 pools: head_dim 128");
    extern __shared__ uint8_t smem_raw[];
    __shared__ TcShared sh;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = smem;                // 2 stages
    uint8_t *sK = smem + Cfg::kQStages * TB;  // NSK stages
    uint8_t *sV = sK + NSK * TB;       // NSV stages

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const long long LIM = a.timeout_cycles;
    const int total_units = attention_units(a);
    const int end_index = total_units;  // the counter's indices past the work

    if (tid == 0) {
        for (int b = 0; b < Cfg::kQStages; ++b) {
            mbar_init(&sh.q_full[b], 1);
            mbar_init(&sh.q_rot[b], 4);
            // the last score MMA's commit, and with BF16 pools the four
            // epilogue warps, which stage the unit's output rows there
            mbar_init(&sh.q_empty[b], TcRoles<F8>::kEpiWarps ? 1 + 4 : 1);
        }
        // 16-bit tiles: filled by one TMA arrival, or (FP8 pools) by the two
        // expansion warps once the code tile's copies (k8 / v8_full) landed
        for (int s = 0; s < NSK; ++s) {
            mbar_init(&sh.k_full[s], 1);
            mbar_init(&sh.k_empty[s], 1);
        }
        for (int s = 0; s < NSV; ++s) {
            mbar_init(&sh.v_full[s], F8 ? 4 : 1);
            mbar_init(&sh.v_empty[s], 1);
            mbar_init(&sh.v8_full[s], 1);
        }
        for (int b = 0; b < kSBuf; ++b) {
            mbar_init(&sh.s_full[b], 1);
            mbar_init(&sh.p_full[b], kSoftmaxThreads);
        }
        for (int b = 0; b < kSBuf; ++b) mbar_init(&sh.pv_done[b], 1);
        mbar_init(&sh.o_full, 1);
        mbar_init(&sh.o_empty, TcRoles<F8>::kEpiWarps ? 128 : kSoftmaxThreads);
        mbar_init(&sh.epi_full, 8);   // one arrival per softmax warp
        mbar_init(&sh.epi_empty, 4);  // one per epilogue warp
        mbar_init(&sh.mma_done, 2);  // one commit from each MMA warp
        for (int i = 0; i < kUnitRing; ++i) {
            mbar_init(&sh.ring.full[i], 1);
            mbar_init(&sh.ring.empty[i], TcRoles<F8>::kUnitReaders);
        }
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
        bool ok = true;
        // the copies' ring; with FP8 pools a value code tile goes to the upper
        // half of its slot and its own barrier (the expansion then fills the
        // slot), a key code tile to the start of its slot
        const int ns = kv_role ? NSV : NSK;
        uint64_t *const ring_full = kv_role ? (F8 ? sh.v8_full : sh.v_full) : sh.k_full;
        uint64_t *const ring_empty = kv_role ? sh.v_empty : sh.k_empty;
        uint8_t *const ring = kv_role ? sV + (F8 ? HB : 0) : sK;
        constexpr int slot_bytes = F8 ? CB : TB;
        int slot = 0;         // ring slot of the next copy
        uint32_t ph = 0;      // parity of that slot's current fill
        int pending = 0;      // fills of the ring issued and not yet drained (<= ns)
        bool rope_all = false;  // rotary embedding: every rotated key row is known written (lane 0)
        // Warp 8 is also the scheduler: lane 0 takes the next unit from the
        // work counter once it has issued the current unit's last K copies,
        // a few tiles before the CTA runs out of work (claimed much earlier,
        // the last units would wait behind busy CTAs while others idle), and
        // publishes it to the other roles through the unit ring.
        //
        // Long direct units (BF16 pools), and with the rotary embedding every
        // unit, claim the next unit kClaimAhead tiles earlier and publish it a
        // tile after that, with its Q copy issued then if its stage is free:
        // the next unit's first score MMA need not wait for its queries (nor,
        // with the rotary embedding, for their rotation by the epilogue warps).
        int taken = (kv_role == 0 && lane == 0) ? first_unit(a) : 0;
        int early = -1;        // ring entry published during the previous unit (rotary embedding)
        bool early_q = false;  // and its Q copy issued
        for (int it = 0;; ++it) {  // it: units started by this CTA
            int unit;
            Unit u;
            if (kv_role == 0) {
                if (early == it) {
                    unit = *reinterpret_cast<volatile int *>(&sh.ring.index[it % kUnitRing]);
                    if (unit < total_units) get_unit(u, sh.ring.desc[it % kUnitRing]);
                } else {
                    unit = __shfl_sync(0xffffffffu, taken, 0);
                    const int s = it % kUnitRing;
                    if (it >= kUnitRing &&
                        !__all_sync(0xffffffffu, mbar_wait_or_abort(&sh.ring.empty[s], (uint32_t)((it / kUnitRing - 1) & 1),
                                                                    LIM, abort_flag))) {
                        ok = false;
                        break;
                    }
                    if (unit < total_units) decode_unit(a, unit, u);  // once, for every role
                    if (lane == 0) publish_unit(sh.ring, it, unit, u);
                    __syncwarp();
                }
            } else {
                unit = read_unit(sh.ring, it, LIM, abort_flag, u);
                if (unit < 0) {
                    ok = false;
                    break;
                }
            }
            if (unit >= end_index) break;
            if (__any_sync(0xffffffffu, !ok || *abort_flag)) break;
            TileList tl;
            tl.init(u);
            const int n = tl.n_total;
            // in a batch that mixes prefill and decode units, a decode piece's
            // cached K/V (read once) may leave L2 first, ahead of the prefill
            // units' K/V that other query tiles read again; elsewhere the
            // copies take no policy
            const bool hinted = a.interleave && u.piece >= 0;
            const uint64_t pol = hinted ? policy_evict_first() : 0;
            // The warp runs converged: every lane takes the waits, lane 0 arms
            // the barriers, and the copies of one tile are spread over the lanes
            // (one cache block and 64-column half per lane).
            const int32_t *bt_row = a.bt + (long long)u.r * a.max_blocks;
            // copies of key tile j (K when kv = 0, V when kv = 1) into their ring slot
            auto load_kv = [&](int j, int kv) -> bool {
                uint64_t *empty = &ring_empty[slot];
                uint64_t *full = &ring_full[slot];
                uint8_t *dst = ring + slot * TB;
                if (!__all_sync(0xffffffffu, mbar_wait_or_abort(empty, ph ^ 1u, LIM, abort_flag))) return false;
                int key0, valid;
                bool pooled;
                tl.tile(j, key0, valid, pooled);
                if (a.test_stall && it == 0 && j == 0 && kv == 0) {
                    // testing only: arm the barrier but never copy, so the
                    // MMA warp's bounded wait on this tile expires
                    if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)slot_bytes);
                } else if (F8 && pooled) {
                    // code tile: one box of bs rows x D bytes per cache block
                    const int nblk = cdiv(valid, a.bs);
                    if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)(nblk * a.bs * D));
                    __syncwarp();
                    const int col0 = key0 / a.bs;
                    for (int b = lane; b < nblk; b += 32) {
                        int blk = __ldg(bt_row + col0 + b);
                        if (blk < 0 || blk >= a.num_blocks) {
                            record_error(a.err, kErrBadBlock);
                            blk = 0;  // keep the byte count; this unit's output is void
                        }
                        if (hinted)
                            tma_load_4d_hint(dst + b * a.bs * D, kv ? &tm_v_pool : &tm_k_pool, full, 0, u.g, 0, blk,
                                             pol);
                        else
                            tma_load_4d(dst + b * a.bs * D, kv ? &tm_v_pool : &tm_k_pool, full, 0, u.g, 0, blk);
                    }
                } else if (F8) {
                    // the new rows' codes: one 128-row box of the workspace copy
                    if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)CB);
                    __syncwarp();
                    if (lane == 0)
                        tma_load_3d(dst, kv ? &tm_v_new : &tm_k_new, full, 0, u.g, u.cu0 + (key0 - u.C));
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
                        if (hinted)
                            tma_load_4d_hint(dst + h * HB + b * a.bs * 128, kv ? &tm_v_pool : &tm_k_pool, full,
                                             h * 64, u.g, 0, blk, pol);
                        else
                            tma_load_4d(dst + h * HB + b * a.bs * 128, kv ? &tm_v_pool : &tm_k_pool, full, h * 64,
                                        u.g, 0, blk);
                    }
                } else if (!F8 && a.rope && kv == 0) {
                    // rotated keys: lane 0 waits until the rows are written,
                    // then issues the copies itself
                    const int row = u.cu0 + (key0 - u.C);
                    int ready = 1;
                    if (lane == 0) ready = rope_rows_ready(a, row, row + valid, rope_all, LIM, abort_flag) ? 1 : 0;
                    if (!__shfl_sync(0xffffffffu, ready, 0)) return false;
                    if (lane == 0) {
                        mbar_arrive_expect_tx(full, (uint32_t)TB);
#pragma unroll
                        for (int h = 0; h < Cfg::kHalves; ++h)
                            tma_load_3d(dst + h * HB, &tm_k_new, full, h * 64, u.g, row);
                    }
                } else {
                    if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)TB);
                    __syncwarp();
                    const int row = u.cu0 + (key0 - u.C);
                    if (lane < Cfg::kHalves)
                        tma_load_3d(dst + lane * HB, kv ? &tm_v_new : &tm_k_new, full, lane * 64, u.g, row);
                }
                if (++slot == ns) {
                    slot = 0;
                    ph ^= 1u;
                }
                if (pending < ns) ++pending;
                return true;
            };
            if (kv_role == 0) {
                // Q first: its stage (it % kQStages) was last used two units
                // ago and is free by now, while the first K tile waits for a
                // ring slot that the current unit's last score MMAs release
                constexpr int QS = Cfg::kQStages;
                // the Q copy of ring entry i (unit fields uq) into stage i % QS
                // once its previous user released it (wait), or only if it
                // already has (!wait)
                auto copy_q = [&](int i, const Unit &uq, bool wait) -> bool {
                    const int qb = i % QS;
                    if (i >= QS) {
                        const uint32_t par = (uint32_t)(((i - QS) / QS) & 1);
                        if (!__all_sync(0xffffffffu, wait ? mbar_wait_or_abort(&sh.q_empty[qb], par, LIM, abort_flag)
                                                          : mbar_try_wait(&sh.q_empty[qb], par)))
                            return false;
                    }
                    if (lane == 0) mbar_arrive_expect_tx(&sh.q_full[qb], (uint32_t)(a.tile_m * D * 2));  // tile_m rows
                    __syncwarp();
                    const int tok0 = uq.cu0 + uq.row0 / a.G;
                    if (F8) {
                        // the two E4M3 planes of the queries
                        if (lane < 2)
                            tma_load_4d(sQ + qb * TB + lane * HB, &tm_q, &sh.q_full[qb], 0, uq.g * a.G, tok0, lane);
                    } else if (lane < Cfg::kHalves) {
                        tma_load_3d(sQ + qb * TB + lane * HB, &tm_q, &sh.q_full[qb], lane * 64, uq.g * a.G, tok0);
                    }
                    return true;
                };
                if (ok && !(early == it && early_q) && !copy_q(it, u, true)) ok = false;
                const int jc = (!F8 && (a.rope || (u.piece < 0 && n >= kEarlyClaimMinTiles))) ? max(0, n - 1 - kClaimAhead) : n;
                early_q = false;
                for (int j = 0; j < n && ok; ++j) {
                    ok = load_kv(j, 0);
                    if (!ok || j < jc) continue;
                    if (j == jc) {
                        if (lane == 0) taken = claim_unit(a, total_units);
                        continue;
                    }
                    if (early != it + 1) {
                        // publish the next unit (its claim has had a tile to return)
                        const int un = __shfl_sync(0xffffffffu, taken, 0);
                        const int s = (it + 1) % kUnitRing;
                        if (it + 1 >= kUnitRing &&
                            !__all_sync(0xffffffffu, mbar_wait_or_abort(&sh.ring.empty[s],
                                                                        (uint32_t)(((it + 1) / kUnitRing - 1) & 1), LIM,
                                                                        abort_flag))) {
                            ok = false;
                            break;
                        }
                        Unit uu;
                        if (un < total_units) decode_unit(a, un, uu);
                        if (lane == 0) publish_unit(sh.ring, it + 1, un, uu);
                        __syncwarp();
                        early = it + 1;
                    }
                    if (!early_q) {
                        const int un = *reinterpret_cast<volatile int *>(&sh.ring.index[(it + 1) % kUnitRing]);
                        if (un < total_units) {
                            Unit uu;
                            get_unit(uu, sh.ring.desc[(it + 1) % kUnitRing]);
                            early_q = copy_q(it + 1, uu, false);
                        }
                    }
                }
                // this unit's copies are all issued: claim the next unit now
                // unless that was done above
                if (ok && jc >= n && lane == 0) taken = claim_unit(a, total_units);
            } else {
                for (int j = 0; j < n && ok; ++j) ok = load_kv(j, 1);
            }
        }
        if (!ok) {
            if (lane == 0) record_error(a.err, kErrTimeout);
            *abort_flag = 1;
        }
        // drain: every issued copy must land before the CTA may exit.  The
        // last `pending` fills occupy the slots just before `slot`.
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
    } else if (warp == kMmaWarp || warp == kPvWarp) {
        // ================================================================ MMA
        // Two issuing warps on different SM sub-partitions: warp 9 issues the
        // score MMAs, warp 11 the PV MMAs.  Each runs converged; one elected
        // lane issues each MMA and commit, and every wait is taken by all
        // lanes.  A score buffer is reused only once the PV that read its P
        // has completed (pv_done of that buffer).
        int ub = 0;                  // score buffer of this warp's next tile
        uint32_t uph = 0;            // use parity of that buffer
        int rs = 0;                  // ring slot (K for warp 9, V for warp 11)
        uint32_t rph = 0;            // and the parity of its fill
        long long issued = 0;        // tiles issued by this warp
        bool ok = true;
        // bf16 operands; fp16 with FP8 pools (queries scaled per row, codes
        // expanded exactly, probabilities rounded to fp16)
        constexpr uint32_t idesc_s = F8 ? idesc_e4m3_f32(128, kKT) : idesc_16bit_f32(128, kKT, 0, 0, true);
        constexpr uint32_t idesc_pv = idesc_16bit_f32(128, D, 0, 1, !F8);
        // Shared-memory descriptors: the high halves (stride, version,
        // swizzle) are common to Q, K and V; only the low halves (start
        // address >> 4 and leading byte offset) differ.  Addresses stay below
        // 2^18 bytes, so adding (bytes >> 4) never carries out of the field.
        const uint64_t q_desc = smem_desc(smem_u32(sQ), 16, 1024, kSwizzle128B);
        const uint32_t desc_hi = (uint32_t)(q_desc >> 32);
        const uint32_t q_lo = (uint32_t)q_desc;
        const uint32_t k_lo0 = (uint32_t)smem_desc(smem_u32(sK), 16, 1024, kSwizzle128B);
        const uint32_t v_lo0 = (uint32_t)smem_desc(smem_u32(sV), HB, 1024, kSwizzle128B);
        const uint32_t tO = tmem + kTmemO;
        const bool s_role = (warp == kMmaWarp);
        for (int ucnt = 0;; ++ucnt) {  // ucnt: units started
            Unit u;
            const int unit = read_unit(sh.ring, ucnt, LIM, abort_flag, u);
            if (unit < 0) {
                ok = false;
                break;
            }
            if (unit >= end_index) break;
            if (__any_sync(0xffffffffu, !ok || *abort_flag)) break;
            TileList tl;
            tl.init(u);
            const int n = tl.n_total;
            if (s_role) {
                // S(j) = Q K(j)^T, as far ahead as the score buffers allow
                // (with the rotary embedding, once the epilogue warps rotated Q)
                const int qb = ucnt % Cfg::kQStages;
                uint64_t *q_ready = (!F8 && a.rope) ? &sh.q_rot[qb] : &sh.q_full[qb];
                if (!__all_sync(0xffffffffu,
                                mbar_wait_or_abort(q_ready, (uint32_t)((ucnt / Cfg::kQStages) & 1), LIM, abort_flag))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t q_lo_u = q_lo + (uint32_t)qb * (uint32_t)(TB >> 4);
                for (int j = 0; j < n; ++j) {
                    if (issued >= kSBuf &&
                        !__all_sync(0xffffffffu, mbar_wait_or_abort(&sh.pv_done[ub], uph ^ 1u, LIM, abort_flag))) {
                        ok = false;
                        break;
                    }
                    if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&sh.k_full[rs], rph, LIM, abort_flag))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t k_lo = k_lo0 + (uint32_t)rs * (uint32_t)(TB >> 4);
                    const uint32_t d_tmem = tmem + ub * kKT;
                    if constexpr (F8) {
                        umma_s_tile_e4m3(d_tmem, q_lo_u, k_lo, desc_hi, idesc_s, (uint32_t)(HB >> 4));
                    } else if constexpr (D == 128) {
                        umma_s_tile128(d_tmem, q_lo_u, k_lo, desc_hi, idesc_s, (uint32_t)(HB >> 4));
                    } else {
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = (uint32_t)(((kk >> 2) * HB + (kk & 3) * 32) >> 4);
                            umma_ss_warp2(d_tmem, q_lo_u + off, k_lo + off, desc_hi, idesc_s, kk > 0 ? 1u : 0u);
                        }
                    }
                    umma_commit_warp(&sh.s_full[ub]);
                    umma_commit_warp(&sh.k_empty[rs]);
                    if (j == n - 1) umma_commit_warp(&sh.q_empty[qb]);  // Q is free once the last S is done
                    ++issued;
                    if (++ub == kSBuf) {
                        ub = 0;
                        uph ^= 1u;
                    }
                    if (++rs == NSK) {
                        rs = 0;
                        rph ^= 1u;
                    }
                }
            } else {
                // O += P(j) V(j) once the softmax has written P(j)
                for (int j = 0; j < n; ++j) {
                    // V(j) first: a partial tile's zeroing then overlaps the
                    // softmax of tile j
                    if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&sh.v_full[rs], rph, LIM, abort_flag))) {
                        ok = false;
                        break;
                    }
                    int key0, valid;
                    bool pooled;
                    tl.tile(j, key0, valid, pooled);
                    if (!F8 && valid < kKT) {
                        // keys past the tile's valid range: zero their V rows so
                        // that P = 0 never meets a NaN or Inf left in the pool or
                        // in this ring slot (eight lanes per 128-byte row, four
                        // rows at a time; then a proxy fence, as the MMA reads
                        // through the async proxy)
                        uint8_t *vs_ = sV + rs * TB + (lane & 7) * 16;
                        for (int r = valid + (lane >> 3); r < kKT; r += 4) {
#pragma unroll
                            for (int h = 0; h < Cfg::kHalves; ++h)
                                *reinterpret_cast<uint4 *>(vs_ + h * HB + r * 128) = make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                    if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&sh.p_full[ub], uph, LIM, abort_flag))) {
                        ok = false;
                        break;
                    }
                    if (j == 0 && !__all_sync(0xffffffffu, mbar_wait_or_abort(&sh.o_empty, (uint32_t)((ucnt & 1) ^ 1),
                                                                               LIM, abort_flag))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t v_lo = v_lo0 + (uint32_t)rs * (uint32_t)(TB >> 4);
                    const uint32_t tP = tmem + ub * kKT;
                    umma_pv_tile128(tO, tP, v_lo, desc_hi, idesc_pv, j > 0 ? 1u : 0u);
                    umma_commit_warp(&sh.v_empty[rs]);
                    umma_commit_warp(&sh.pv_done[ub]);
                    if (j == n - 1) umma_commit_warp(&sh.o_full);
                    if (++ub == kSBuf) {
                        ub = 0;
                        uph ^= 1u;
                    }
                    if (++rs == NSV) {
                        rs = 0;
                        rph ^= 1u;
                    }
                }
                if (!ok) break;
            }
        }
        if (!ok) {
            if (lane == 0) record_error(a.err, kErrTimeout);
            *abort_flag = 1;
        }
        // every MMA issued so far (by both warps) must finish before TMEM is freed
        umma_commit_warp(&sh.mma_done);
        mbar_wait(&sh.mma_done, 0, LIM);
        __syncwarp();
    } else if (TcRoles<F8>::kEpiWarps && warp >= kEpiWarp) {
        // =============================================== epilogue (warps 12-15)
        // Warp 12 + e reads TMEM lanes 32e .. 32e + 31: one thread per output
        // row with all its D columns.  Per unit: take the rows' maxima and
        // sums from the softmax warps, wait for the last PV, read O, free it
        // for the next unit's PVs, and write the rows (a split unit's or tail
        // piece's partial: unnormalised, with its maxima and sums).
        //
        // With the rotary embedding these warps rotate each unit's queries in
        // its Q stage, one unit ahead: the next unit's as soon as its copy
        // has landed, before this unit's outputs (which wait for its last PV).
        //
        // They also copy this CTA's share of the fused K/V write while the
        // first unit runs (attention reads the new rows from k_new / v_new,
        // never from these pool rows): at once, or with the rotary embedding
        // after the first unit's queries and once the share's keys are rotated.
        const int e = warp - kEpiWarp;
        const int lr = 32 * e + lane;
        const bool rope = !F8 && a.rope;
        auto write_share = [&]() -> bool {
            const int per = cdiv(a.total_tokens, (int)gridDim.x);
            const int t0 = (int)blockIdx.x * per;
            const int t1 = t0 + per < a.total_tokens ? t0 + per : a.total_tokens;
            if (t0 >= t1) return true;
            const int row_bytes = a.hkv * D * 2;
            if (rope) {
                bool all = false;
                if (!__all_sync(0xffffffffu, rope_rows_done(a, t0, t1, all, LIM, abort_flag))) return false;
                write_token_rows<4, true>(a.cached, a.cu, a.bt, a.num_reqs, a.max_blocks, a.bs, a.num_blocks,
                                          row_bytes, a.k_new, a.v_new, a.k_cache, a.v_cache, t0, t1, lr, 128, a.err);
            } else {
                write_token_rows<4, false>(a.cached, a.cu, a.bt, a.num_reqs, a.max_blocks, a.bs, a.num_blocks,
                                           row_bytes, a.k_new, a.v_new, a.k_cache, a.v_cache, t0, t1, lr, 128, a.err);
            }
            return true;
        };
        if (a.write_share && !rope) write_share();
        const uint32_t tO = tmem + ((uint32_t)(32 * e) << 16) + kTmemO;
        bool ok = true;
        // the queries of ring entry i (an attention unit uq), rotated in place
        auto rotate_q = [&](int i, const Unit &uq) -> bool {
            const int qb = i % Cfg::kQStages;
            if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&sh.q_full[qb], (uint32_t)((i / Cfg::kQStages) & 1), LIM,
                                                            abort_flag)))
                return false;
            rope_q_tile<D>(a, uq, sQ + qb * TB, lr);
            fence_proxy_async_smem();  // the score MMAs read Q through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.q_rot[qb]);
            return true;
        };
        // (each entry's ring slot is held from its first read until its
        // fields are read again, after the next unit's rotation: so the
        // fields are not kept in registers meanwhile)
        Unit u;
        int unit = read_unit(sh.ring, 0, LIM, abort_flag, u, false);
        if (rope && unit >= 0 && unit < total_units && !rotate_q(0, u)) unit = -1;
        if (a.write_share && rope && unit >= 0 && !write_share()) unit = -1;
        for (int ec = 0;; ++ec) {
            if (unit < 0) {
                ok = false;
                break;
            }
            if (unit >= end_index) break;
            int unit_n = 0;
            if (rope) {
                Unit un;
                unit_n = read_unit(sh.ring, ec + 1, LIM, abort_flag, un, false);
                if (unit_n >= 0 && unit_n < total_units && !rotate_q(ec + 1, un)) unit_n = -1;
            }
            reread_unit(sh.ring, ec, u);
            const uint32_t ph = (uint32_t)(ec & 1);
            if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&sh.epi_full, ph, LIM, abort_flag))) {
                ok = false;
                break;
            }
            const float m = sh.epi_m[lr], l = sh.epi_l[lr];
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.epi_empty);
            if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&sh.o_full, ph, LIM, abort_flag))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const bool row_valid = lr < u.rows;
            const bool warp_rows = __any_sync(0xffffffffu, row_valid);
            const int pr = u.row0 + lr;  // packed row of the request
            const int t = u.cu0 + pr / a.G, h = u.g * a.G + pr % a.G;
            const float inv = 1.f / l;
            if (u.piece >= 0) {
                // a partial: the fp32 row goes out before O is freed
#pragma unroll
                for (int c = 0; c < D / 64 && warp_rows; ++c) {
                    uint32_t r0[32], r1[32];  // columns 64c .. 64c + 63
                    tmem_ld32(tO + c * 64, r0);
                    tmem_ld32(tO + c * 64 + 32, r1);
                    tmem_wait_ld();
                    if (row_valid) {
                        float4 *dst = reinterpret_cast<float4 *>(a.ws + u.ws_off + (long long)lr * D + c * 64);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            dst[i] = make_float4(__uint_as_float(r0[4 * i]), __uint_as_float(r0[4 * i + 1]),
                                                 __uint_as_float(r0[4 * i + 2]), __uint_as_float(r0[4 * i + 3]));
                            dst[8 + i] = make_float4(__uint_as_float(r1[4 * i]), __uint_as_float(r1[4 * i + 1]),
                                                     __uint_as_float(r1[4 * i + 2]), __uint_as_float(r1[4 * i + 3]));
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&sh.o_empty);
            } else {
                // the row as bf16 in registers (D / 2 words), O freed for the
                // next unit's PVs, then the stores
                uint32_t o[D / 2];
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];  // columns 32c .. 32c + 31
                    if (warp_rows) {
                        tmem_ld32(tO + c * 32, r);
                        tmem_wait_ld();
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        o[16 * c + i] = pack_bf16(__uint_as_float(r[2 * i]) * inv, __uint_as_float(r[2 * i + 1]) * inv);
                }
                tc_fence_before();
                mbar_arrive(&sh.o_empty);
                // The stores go through this unit's Q stage, free since its
                // last score MMA completed (before the softmax could finish
                // the last tile) and until the warps below release it: each
                // lane puts its row there (16-byte chunk c of row r at
                // position (c + r) mod CPR, which spreads a store instruction
                // over all banks), then every store instruction writes whole
                // rows (RPI rows of CPR chunks) instead of one chunk of each
                // of 32 rows.
                if (warp_rows) {
                    constexpr int CPR = D / 8;     // 16-byte chunks per row
                    constexpr int RPI = 32 / CPR;  // rows per store instruction
                    uint8_t *stage = sQ + (ec % Cfg::kQStages) * TB + e * 32 * (D * 2);
#pragma unroll
                    for (int c = 0; c < CPR; ++c)
                        *reinterpret_cast<uint4 *>(stage + lane * (D * 2) + (((c + lane) % CPR) << 4)) =
                            make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
                    __syncwarp();
                    const long long row_off = row_valid ? ((long long)t * a.hq + h) * D : -1;
                    const int c = lane % CPR;
#pragma unroll 4
                    for (int i = 0; i < 32 / RPI; ++i) {
                        const int r = RPI * i + lane / CPR;
                        const long long off = __shfl_sync(0xffffffffu, row_off, r);
                        const uint4 v = *reinterpret_cast<const uint4 *>(stage + r * (D * 2) + (((c + r) % CPR) << 4));
                        if (off >= 0) reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) + off)[c] = v;
                    }
                }
            }
            // the stage's next user is a TMA copy (async proxy)
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.q_empty[ec % Cfg::kQStages]);
            if (row_valid) {
                if (u.piece >= 0) {
                    float *ws = a.ws + u.ws_off;
                    ws[(long long)u.rows * D + lr] = m;
                    ws[(long long)u.rows * D + u.rows + lr] = l;
                } else if (a.lse) {
                    a.lse[(long long)t * a.hq + h] = (m + __log2f(l)) * 0.69314718055994531f;
                }
            }
            if (u.tail >= 0 && warp_rows) {
                // a tail piece: the warp that completes the unit's last piece
                // for its 32 rows (warp 12 + e of every piece's CTA writes
                // them) merges the pieces' partials of those rows.  The warp
                // barrier orders the lanes' partial writes before lane 0's
                // release, and lane 0's acquire before the lanes' reads.
                __syncwarp();
                int last = 0;
                if (lane == 0)
                    last = atom_add_acq_rel_gpu(a.tail_count + u.tail * kSoftmaxWarpsMax + e, 1) ==
                           a.tail_pieces - 1;
                if (__shfl_sync(0xffffffffu, last, 0)) {
                    __syncwarp();
                    merge_tail_rows<D>(a, u, 32 * e, lane);
                    merge_tail_rows<D>(a, u, 32 * e + 16, lane);
                }
            }
            unit = rope ? unit_n : read_unit(sh.ring, ec + 1, LIM, abort_flag, u, false);
        }
        if (!ok) {
            if (lane == 0) record_error(a.err, kErrTimeout);
            *abort_flag = 1;
        }
    } else if (F8 && warp >= kKConvWarp) {
        // ==================================== FP8 expansion (warps 12-15)
        // Warp 12 + w expands rows 32w .. 32w + 31 of every V code tile in its
        // ring slot.  V rows past a tile's valid keys become zeros (P = 0 must
        // not meet a NaN code left in the pool or a stale value).  Key code
        // rows there are left as they are: the softmax masks their scores.
        const int r0 = (warp - kKConvWarp) * 32;
        const int nsb = NSV;
        int sb = 0;
        uint32_t phb = 0;
        bool ok = true;
        for (int cc = 0;; ++cc) {
            Unit u;
            const int unit = read_unit(sh.ring, cc, LIM, abort_flag, u);
            if (unit < 0) {
                ok = false;
                break;
            }
            if (unit >= end_index) break;
            if (__any_sync(0xffffffffu, !ok || *abort_flag)) break;
            TileList tl;
            tl.init(u);
            for (int j = 0; j < tl.n_total; ++j) {
                uint64_t *code_full = &sh.v8_full[sb];
                uint64_t *tile_full = &sh.v_full[sb];
                if (!__all_sync(0xffffffffu, mbar_wait_or_abort(code_full, phb, LIM, abort_flag))) {
                    ok = false;
                    break;
                }
                int key0, valid;
                bool pooled;
                tl.tile(j, key0, valid, pooled);
                expand_code_rows(sV + sb * TB, r0, valid, lane, HB);
                fence_proxy_async_smem();  // the MMA reads the tile through the async proxy
                __syncwarp();
                if (lane == 0) mbar_arrive(tile_full);
                if (++sb == nsb) {
                    sb = 0;
                    phb ^= 1u;
                }
            }
            if (!ok) break;
        }
        if (!ok) {
            if (lane == 0) record_error(a.err, kErrTimeout);
            *abort_flag = 1;
        }
        __syncwarp();
    } else if (warp < 8) {
        // ============================================== softmax (warps 0-7)
        const int half = lane >> 4;                                // 0: keys 0-63, 1: keys 64-127
        const int lr = 32 * (warp & 3) + 16 * (warp >> 2) + (lane & 15);  // row of the tile == TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3) + 16 * (warp >> 2)) << 16);
        const uint32_t tO = lane_base + kTmemO;
        float sl = a.scale_log2;  // with FP8 pools times the unit's key scale
        int cb = 0;          // score buffer of the next tile
        uint32_t cph = 0;    // and its use parity
        int prev_b = 0;      // buffer and use parity of the previous tile (for the PV(j-1) wait)
        uint32_t prev_ph = 0;
        bool ok = true;
        if (!F8 && a.rope) {
            // the rotary embedding: rotate the new keys once, before any unit.
            // Thread 0 claims the pieces for the eight warps, each one piece
            // ahead; once every thread's rows are out (the barrier), it counts
            // the piece done (release) for its 128-row tile and the launch.
            int next = 0;
            if (tid == 0) next = atomicAdd(a.rope_count, 1);
            for (;;) {
                if (tid == 0) sh.rope_claim = next;
                named_bar_sync(1, kSoftmaxThreads);
                const int piece = sh.rope_claim;
                if (piece >= a.rope_pieces) break;
                if (tid == 0) next = atomicAdd(a.rope_count, 1);
                rope_keys_piece<D>(a, piece, tid);
                fence_proxy_async_global();
                named_bar_sync(1, kSoftmaxThreads);  // also: every thread has read rope_claim
                if (tid == 0) {
                    red_release_gpu_add(a.rope_count + 2 + piece / (kTcTileN / kRopePieceTokens), 1);
                    red_release_gpu_add(a.rope_count + 1, 1);
                }
            }
        }
        for (int oc = 0;; ++oc) {  // oc: units started
            Unit u;
            const int unit = read_unit(sh.ring, oc, LIM, abort_flag, u);
            if (unit < 0) {
                ok = false;
                break;
            }
            if (unit >= end_index) break;
            if (__any_sync(0xffffffffu, !ok || *abort_flag)) break;
            TileList tl;
            tl.init(u);
            const int n = tl.n_total;
            const bool row_valid = lr < u.rows;
            const int pos = row_valid ? u.C + (u.row0 + lr) / a.G : -1;
            // FP8 pools: the tiles hold code values and the queries were
            // scaled by a power of two per row; the key scale and the row's
            // inverse query scale multiply its scores, the value scale the output
            float v_mul = 1.f;
            if (F8) {
                const int pr = u.row0 + lr;
                const float q_mul =
                    row_valid ? __ldg(a.q_rscale + (long long)(u.cu0 + pr / a.G) * a.hq + u.g * a.G + pr % a.G) : 1.f;
                sl = a.scale_log2 * __ldg(a.k_scale + u.g) * q_mul;
                v_mul = __ldg(a.v_scale + u.g);
            }
            float m_ref = -INFINITY, l = 0.f;
            // a warp whose 16 rows are all padding (a decode has G rows of
            // 128) skips the math; each O row depends on its own P row only,
            // so whatever its P rows hold never reaches a written output
            const bool warp_rows = __any_sync(0xffffffffu, row_valid);
            for (int j = 0; j < n; ++j) {
                const int b = cb;
                const uint32_t bph = cph;
                if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&sh.s_full[b], cph, LIM, abort_flag))) {
                    ok = false;
                    break;
                }
                if (++cb == kSBuf) {
                    cb = 0;
                    cph ^= 1u;
                }
                if (!warp_rows) {
                    mbar_arrive(&sh.p_full[b]);
                    prev_b = b;
                    prev_ph = bph;
                    continue;
                }
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
                float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
                {
                    // exponentials in pairs: paired FMAs and adds, ex2 on the MUFU
                    uint32_t r[32];
                    const float2 sl2 = make_float2(sl, sl), neg2 = make_float2(neg, neg);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float2 x = __ffma2_rn(make_float2(s[2 * i], s[2 * i + 1]), sl2, neg2);
                        float2 e;
                        e.x = ex2(x.x);
                        e.y = ex2(x.y);
                        if (i & 1)
                            acc1 = __fadd2_rn(acc1, e);
                        else
                            acc0 = __fadd2_rn(acc0, e);
                        r[i] = F8 ? pack_f16(e.x, e.y) : pack_bf16(e.x, e.y);
                    }
                    tmem_st16x2_32<32>(tS, r);  // threads 0-15: P columns 0-31, 16-31: 32-63
                }
                l += (acc0.x + acc0.y) + (acc1.x + acc1.y);
                if (j >= 1 && __any_sync(0xffffffffu, move)) {
                    // rescale O once PV(j-1) has completed; PV(j) cannot start
                    // before this group's arrival below
                    if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&sh.pv_done[prev_b], prev_ph, LIM, abort_flag))) {
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
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&sh.p_full[b]);
                prev_b = b;
                prev_ph = bph;
            }
            if (!ok) break;
            if constexpr (TcRoles<F8>::kEpiWarps) {
                // the epilogue warps write this unit's rows: hand them each
                // row's maximum and sum once they have read the previous unit's
                l += __shfl_xor_sync(0xffffffffu, l, 16);  // whole row
                if (oc >= 1 && !__all_sync(0xffffffffu, mbar_wait_or_abort(&sh.epi_empty, (uint32_t)((oc - 1) & 1),
                                                                            LIM, abort_flag))) {
                    ok = false;
                    break;
                }
                if (half == 0) {
                    sh.epi_m[lr] = m_ref;
                    sh.epi_l[lr] = l;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.epi_full);
                continue;
            }
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait_or_abort(&sh.o_full, (uint32_t)(oc & 1), LIM, abort_flag));
            if (!ok) break;
            tc_fence_after();
            l += __shfl_xor_sync(0xffffffffu, l, 16);  // whole row
            // epilogue: this thread's half of the O row, then release O
            const int pr = u.row0 + lr;  // packed row of the request
            const float inv = v_mul / l;
            const int t = u.cu0 + pr / a.G, h = u.g * a.G + pr % a.G;
#pragma unroll
            for (int c = 0; c < D / 64 && warp_rows; ++c) {
                uint32_t r[32];
                tmem_ld16x2_32<D / 2>(tO + c * 32, r);  // output columns half * D/2 + c * 32 + i
                tmem_wait_ld();
                const int col0 = half * (D / 2) + c * 32;
                if (row_valid) {
                    if (u.piece >= 0) {
                        float4 *dst = reinterpret_cast<float4 *>(a.ws + u.ws_off + (long long)lr * D + col0);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[i] = make_float4(__uint_as_float(r[4 * i]) * v_mul, __uint_as_float(r[4 * i + 1]) * v_mul,
                                                 __uint_as_float(r[4 * i + 2]) * v_mul,
                                                 __uint_as_float(r[4 * i + 3]) * v_mul);
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
            if (row_valid && half == 0) {
                if (u.piece >= 0) {
                    float *ws = a.ws + u.ws_off;
                    ws[(long long)u.rows * D + lr] = m_ref;
                    ws[(long long)u.rows * D + u.rows + lr] = l;
                } else if (a.lse) {
                    a.lse[(long long)t * a.hq + h] = (m_ref + __log2f(l)) * 0.69314718055994531f;
                }
            }
            if (u.tail >= 0 && warp_rows) {
                // a tail piece: the warp that completes the unit's last piece
                // for its 16 rows (the same warp of every piece's CTA writes
                // them) merges the pieces' partials of those rows.  The warp
                // barrier orders the lanes' partial writes before lane 0's
                // release, and lane 0's acquire before the lanes' reads.
                __syncwarp();
                int last = 0;
                if (lane == 0)
                    last = atom_add_acq_rel_gpu(a.tail_count + u.tail * kSoftmaxWarpsMax + warp, 1) ==
                           a.tail_pieces - 1;
                if (__shfl_sync(0xffffffffu, last, 0)) {
                    __syncwarp();
                    merge_tail_rows<D>(a, u, 32 * (warp & 3) + 16 * (warp >> 2), lane);
                }
            }
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

template <int D, bool F8>
cudaError_t launch_tc(const AttnArgs &a, const TcMaps &m, int grid, cudaStream_t stream) {
    constexpr int smem = TcCfg<D, F8>::kSmemBytes;
    // set once per device (a repeated set is harmless), so that later calls
    // make no attribute call and can be captured into a CUDA graph; host
    // threads launching at once take the lock
    static std::mutex attr_mutex;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lock(attr_mutex);
        if (dev < 0 || dev >= 64 || !attr_set[dev]) {
            e = cudaFuncSetAttribute(attn_tc_kernel<D, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) attr_set[dev] = true;
        }
    }
    attn_tc_kernel<D, F8><<<grid, TcRoles<F8>::kThreads, smem, stream>>>(a, m.q, m.k_new, m.v_new, m.k_pool,
                                                                          m.v_pool);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_tc(const AttnArgs &a, const TcMaps &m, cudaStream_t stream) {
    const int grid = a.write_ctas;  // persistent: min(units, SMs)
    if (grid <= 0 || attention_units(a) == 0) return cudaSuccess;
    // the fused write is the epilogue warps' share (BF16 pools), never
    // pieces of the work counter
    if (a.write_chunks != 0 || (a.write_share && a.kv_fp8)) return cudaErrorInvalidValue;
    if (a.kv_fp8) return a.d == 128 ? launch_tc<128, true>(a, m, grid, stream) : cudaErrorInvalidValue;
    return a.d == 128 ? launch_tc<128, false>(a, m, grid, stream) : launch_tc<64, false>(a, m, grid, stream);
}

}  // namespace cpa
