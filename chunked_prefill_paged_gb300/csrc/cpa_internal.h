// cpa_internal.h -- definitions shared by the host planner and the kernels
// of libcpa (not part of the public ABI).
//
// Work decomposition.  The active rows of a request are its N_r tokens times
// the G = H_q / H_kv query heads that share one key/value head ("Prefill
// Optimisation", section 6, grouped-query attention); they are packed
// token-major, head-minor, so one tile of rows reads one stream of K/V.  A
// work unit is (request, kv head, query tile, key range):
//   * direct units: a query tile with all keys it can see, walked in order
//     with the running (max, sum, output) carried along;
//   * split units: requests whose rows fit one tile (decodes, tiny chunks)
//     are cut into pieces of split_len keys -- the kv_segment_size segments
//     of "Prefill Processing" (Kernel Interface, Partial KV Segment
//     Handling) -- each written as a partial (unnormalised output, max,
//     sum) and merged by attn_merge.
//   * tail pieces: on the tensor-core kernel, when the direct units would
//     leave the last wave of CTAs partly idle, the planner may cut each of
//     the last few direct units (by index) into a few pieces by key tiles.
//     Each piece writes a partial like a split unit; the CTA that finishes a
//     unit's last piece merges them into the output, in the same launch.
// Direct units are numbered first (the heaviest query tiles of each request
// first), the tail pieces in place of the last direct units, then split
// units.  Host and device both use request_work() so the launch size and the
// device-side decode agree.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define CPA_HD __host__ __device__ __forceinline__
#else
#define CPA_HD inline
#endif

namespace cpa {

constexpr int kTcTileM = 128;    // packed query rows per tensor-core tile
constexpr int kTcTileN = 128;    // keys per K/V tile of the tensor-core kernel
constexpr int kSimtTileM = 16;   // packed query rows per CUDA-core tile
constexpr int kDefaultSplit = 1024;
// A CTA takes several consecutive kv_segment_size pieces of a decode's keys
// (carried by its online softmax) while the batch still has at least this
// many units -- about seven per SM on a 152-SM GB300, enough for the dynamic
// scheduler to balance -- up to kMaxSplitLen keys per unit.
constexpr int kSplitTargetUnits = 1024;
constexpr int kMaxSplitLen = 8192;
// When the planner lengthened the pieces, the last decode requests (in batch
// order) take pieces half as long (at least the base length), enough for
// this many waves of CTAs: their units are the last of the launch, so the
// last wave ends evenly instead of with some CTAs deep in a long piece
// (measured on a 64-decode mixed step: half-length pieces for three waves
// beat quarter-length ones and four or six waves).
constexpr int kFineTailWaves = 3;
// 16-byte pieces of the new K/V rows per fused-write chunk of the tensor-core
// kernel (each piece index copies 16 bytes of K and 16 bytes of V)
constexpr int kWriteChunkPieces = 1024;
// Tensor-core kernel with the rotary embedding: new tokens per piece of the
// key rotation at the start of the launch (a 128-row tile of the new rows is
// complete once its 128 / kRopePieceTokens pieces are).
constexpr int kRopePieceTokens = 16;
// Batches whose K/V (all requests, cached + new) exceed this many bytes walk
// their direct units kv head by kv head (about half of GB300's L2).
constexpr double kHeadMajorKvBytes = 64.0 * 1024 * 1024;

// device error codes (match cpa_status)
constexpr int kErrTimeout = 4;
constexpr int kErrBadBlock = 5;

CPA_HD int cdiv(int a, int b) { return (a + b - 1) / b; }

// Floats of one split unit's partial: output [rows][d], then the row maxima
// [rows] and sums [rows], padded to a multiple of 4 floats so that every
// unit's output block starts 16-byte aligned.
CPA_HD long long partial_floats(int rows, int d) { return (long long)rows * d + ((2 * rows + 3) & ~3); }

// Softmax warps of the tensor-core kernel (counters per tail unit), and the
// most pieces a tail unit is cut into.
constexpr int kSoftmaxWarpsMax = 8;
constexpr int kMaxTailPieces = 4;

struct ReqWork {
    int direct_units;    // H_kv * query tiles, or 0
    int split_units;     // H_kv * pieces, or 0
    int pieces;          // key pieces of a split request (0 when direct)
    long long ws_floats; // floats of partials for a split request
};

// tiles_per_unit: query tiles one direct unit covers (the tensor-core kernel
// pairs two consecutive tiles of a request so they share every K/V tile).
CPA_HD ReqWork request_work(int C, int N, int G, int hkv, int d, int tile_m, int split_len, int tiles_per_unit) {
    ReqWork w{0, 0, 0, 0};
    if (N <= 0) return w;
    const int rows = N * G;
    const int n_qt = cdiv(rows, tile_m);
    if (split_len > 0 && n_qt == 1) {
        const int pieces = cdiv(C + N, split_len);
        if (pieces > 1) {
            w.split_units = hkv * pieces;
            w.pieces = pieces;
            w.ws_floats = (long long)w.split_units * partial_floats(rows, d);
            return w;
        }
    }
    w.direct_units = hkv * cdiv(n_qt, tiles_per_unit);
    return w;
}

// Arguments of every attention kernel (passed by value).
struct AttnArgs {
    // batch
    int num_reqs;
    int max_blocks;
    int total_tokens;
    const int32_t *cached;
    const int32_t *nnew;
    const int32_t *cu;
    const int32_t *bt;
    // shape
    int hq, hkv, G, d, bs, num_blocks;
    float scale_log2;  // softmax scale * log2(e)
    int split_len;     // 0: no split units
    int split_len_fine; // requests fine_from .. num_reqs - 1 cut their keys in pieces of this
    int fine_from;      // length (the launch's last split units); see split_len_of
    int tile_m;
    int tiles_per_unit; // query tiles per direct unit
    int head_major;     // direct units of a request ordered kv head by kv head
                        // (else kv head innermost); see decode_unit
    int num_direct_units;
    int num_split_units;
    int tail_units;     // tensor-core kernel, no split units: the last tail_units direct units
                        // run as tail_pieces pieces each, numbered unit-major in their place
    int tail_pieces;
    long long tail_ws;  // float offset in ws of the tail pieces' partials (one per piece)
    int *tail_count;    // [tail_units * kSoftmaxWarpsMax]: pieces of a unit whose rows of one
                        // softmax warp are written (zeroed before the launch)
    int interleave;     // tensor-core kernel, batches with both kinds: direct and split units
                        // alternate over indices [0, interleave_span) (see decode_unit), so
                        // that prefill (tensor-bound) and decode (HBM-bound) units run side
                        // by side; the split units past the span (the fine ones) come last
    int interleave_span;
    // data
    const void *q;
    const void *k_new;
    const void *v_new;
    void *k_cache;
    void *v_cache;
    void *out;
    float *lse;
    float *ws;          // partials of split units
    int *sched;         // tensor-core kernel: work counter (zeroed before the launch)
    int group_ctas;     // one-pipeline kernel, two CTA groups (0: one): CTAs [0, group_ctas)
    int group_units;    // claim indices [0, group_units) from sched, the others the rest
    int *sched_b;       // from this second counter; each then takes the other group's
    int write_chunks;   // two-pipeline kernel with the fused write: indices [units, units +
                        // write_chunks) of the counter are pieces of the K/V write, taken
                        // by CTAs whose attention work has run out
    int fuse_write;     // write new K/V into the pool in the same launch
    int write_share;    // one-pipeline kernel: each CTA's epilogue warps copy an even share
                        // of the K/V write near the start (they are idle until the first
                        // unit ends), instead of counter pieces
    int write_ctas;     // grid size: the tensor-core kernel's persistent CTAs (units and
                        // write pieces, at most one per SM); the CUDA-core kernel's units
    int *err;           // device error word (first error wins)
    long long timeout_cycles;
    int test_stall;     // testing only: withhold the first K tile's copies
    // FP8 cache: pools and k_new / v_new (the workspace copies of the new rows'
    // codes) hold E4M3 codes; a code of kv head g stands for value * scale[g].
    // q is then two E4M3 planes [2][T, hq, d] (a row scaled by 2^e, and its
    // rounding residual); q_rscale[t * hq + h] = 2^-e.
    int kv_fp8;
    const float *k_scale;  // [hkv]
    const float *v_scale;  // [hkv]
    const float *q_rscale; // [T, hq]
    // Rotary embedding in the tensor-core kernel (BF16 pools): the queries are
    // rotated in shared memory once their tile has landed; the new keys are
    // rotated once, at the start of the launch, from k_src into k_new (a
    // workspace copy that the new-key tiles and the fused write read).
    // rope_count: [0] pieces claimed, [1] pieces done, [2 + i] pieces done of
    // 128-row tile i of the new rows (zeroed before the launch).
    int rope;
    int rope_pieces;       // cdiv(total_tokens, kRopePieceTokens)
    const void *k_src;     // [T, hkv, d] the caller's (unrotated) new keys
    int *rope_count;
    // turns per position of pair c, theta^(-2c/d) / (2 pi), as a 64-bit binary
    // fraction (see RopeArgs)
    unsigned long long turn_frac[64];
};

// Pieces of the key rotation that cover 128-row tile i of the new rows.
CPA_HD int rope_pieces_of_tile(int total_tokens, int i) {
    const int rows = total_tokens - i * kTcTileN;
    return cdiv(rows < kTcTileN ? rows : kTcTileN, kRopePieceTokens);
}

// Piece length of request r's keys when its rows fit one tile.
CPA_HD int split_len_of(const AttnArgs &a, int r) { return r >= a.fine_from ? a.split_len_fine : a.split_len; }

// Work indices of attention (direct units, tail pieces, split units).
CPA_HD int attention_units(const AttnArgs &a) {
    return a.num_direct_units + a.num_split_units + a.tail_units * (a.tail_pieces - 1);
}

// Arguments of the pre-pass over the active tokens' rows: with rotate, turns
// queries and new keys at absolute position cached[r] + i (pairs (c, c + d/2)
// by p * theta^(-2c/d)) into q_rot / k_rot; with kv_fp8, encodes the (rotated)
// keys and the values as E4M3 codes into k_q8 / v_q8; with write_pool, stores
// the keys and values (rotated, encoded as the pool holds them) into their
// pool slots.
struct RopeArgs {
    int num_reqs, max_blocks, total_tokens;
    const int32_t *cached;
    const int32_t *cu;
    const int32_t *bt;
    int hq, hkv, d, bs, num_blocks;
    int elem_bytes;       // 2 (bf16) or 4 (fp32)
    // turns per position of pair c, theta^(-2c/d) / (2 pi), as a 64-bit binary
    // fraction: pos * turn_frac[c] modulo 2^64 is the angle reduced to one turn
    unsigned long long turn_frac[64];
    const void *q;        // [T, hq, d] (may be null when q_rot is null)
    const void *k_new;    // [T, hkv, d]
    const void *v_new;    // [T, hkv, d]
    void *q_rot;          // [T, hq, d] or null
    void *k_rot;          // [T, hkv, d] or null
    int write_pool;
    void *k_cache;
    void *v_cache;
    int *err;
    int rotate;           // 0: keys pass unrotated (turn_frac unused)
    int kv_fp8;           // pools hold E4M3 codes (element type bf16)
    const float *k_scale; // [hkv]
    const float *v_scale; // [hkv]
    void *k_q8;           // [T, hkv, d] codes of the keys, or null
    void *v_q8;           // [T, hkv, d] codes of the values, or null
    void *q8;             // [2][T, hq, d] E4M3 planes of the scaled queries (FP8-cache attention), or null
    float *q_rscale;      // [T, hq] inverse power-of-two scale of each q8 row
};

// Arguments of the standalone KV write.
struct KvWriteArgs {
    int num_reqs, max_blocks, total_tokens;
    const int32_t *cached;
    const int32_t *cu;
    const int32_t *bt;
    int hkv, bs, num_blocks;
    int head_bytes;  // d * element bytes: one head's row
    const void *k_new;
    const void *v_new;
    void *k_cache;
    void *v_cache;
    int *err;
};

}  // namespace cpa
