// cpa_api.cu -- the C ABI of libcpa: host-side checks, work planning, tensor
// maps, and the launches.  Every entry point is declared in include/cpa.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <functional>
#include <mutex>
#include <queue>
#include <utility>
#include <vector>

#include "../../include/cpa.h"
#include "cpa_internal.h"
#include "launch.h"

namespace cpa {

__device__ int g_device_error;  // first error a kernel recorded (0: none)

namespace {

constexpr int kMaxDevices = 64;
constexpr long long kDefaultTimeoutCycles = 2000000000LL;

struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    int cc_major = 0, cc_minor = 0;
    int *err = nullptr;  // device address of g_device_error
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];

cpa_status device_info(DeviceInfo &out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CPA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo &d = g_devices[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return CPA_ERR_CUDA;
        if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return CPA_ERR_CUDA;
        if (cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return CPA_ERR_CUDA;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return CPA_ERR_CUDA;
        d.err = static_cast<int *>(p);
        d.ready = true;
    }
    out = d;
    // the library is built for sm_103a only
    if (out.cc_major != 10 || out.cc_minor != 3) return CPA_ERR_UNSUPPORTED;
    return CPA_SUCCESS;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks every argument that the host can see.  Nothing is launched when
// this fails.
cpa_status validate(const cpa_batch *b, const cpa_params *p) {
    if (!b || !p) return CPA_ERR_INVALID_ARG;
    if (p->dtype != CPA_DTYPE_FP32 && p->dtype != CPA_DTYPE_BF16) return CPA_ERR_INVALID_ARG;
    if (p->num_heads_q <= 0 || p->num_heads_kv <= 0 || p->num_heads_q % p->num_heads_kv != 0)
        return CPA_ERR_INVALID_ARG;
    if (p->head_dim != 64 && p->head_dim != 128) return CPA_ERR_INVALID_ARG;
    if (p->block_size != 16 && p->block_size != 32 && p->block_size != 64 && p->block_size != 128)
        return CPA_ERR_INVALID_ARG;
    if (p->num_blocks <= 0) return CPA_ERR_INVALID_ARG;
    const int ks = p->kv_segment_size;
    if (ks != 0 && ks != 512 && ks != 1024 && ks != 2048 && ks != 4096) return CPA_ERR_INVALID_ARG;
    if (ks != 0 && ks % p->block_size != 0) return CPA_ERR_INVALID_ARG;
    if (!isfinite(p->scale) || !(p->scale > 0.f)) return CPA_ERR_INVALID_ARG;
    if (!isfinite(p->rope_theta) || p->rope_theta < 0.f) return CPA_ERR_INVALID_ARG;
    if (p->timeout_cycles < 0) return CPA_ERR_INVALID_ARG;
    if (p->kv_format != CPA_KV_SAME && p->kv_format != CPA_KV_FP8_E4M3) return CPA_ERR_INVALID_ARG;
    if (p->kv_format == CPA_KV_FP8_E4M3) {
        if (!p->k_scale || !p->v_scale || (reinterpret_cast<uintptr_t>(p->k_scale) & 3u) ||
            (reinterpret_cast<uintptr_t>(p->v_scale) & 3u))
            return CPA_ERR_INVALID_ARG;
        if (p->dtype != CPA_DTYPE_BF16) return CPA_ERR_UNSUPPORTED;  // FP8 codes of BF16 rows only
    }
    if (b->num_reqs < 0 || b->total_new_tokens < 0) return CPA_ERR_INVALID_ARG;
    if (b->num_reqs == 0) return b->total_new_tokens == 0 ? CPA_SUCCESS : CPA_ERR_INVALID_ARG;
    if (b->max_blocks_per_seq <= 0) return CPA_ERR_INVALID_ARG;
    if (!b->h_cached_seq_len || !b->h_num_new_tokens) return CPA_ERR_INVALID_ARG;
    if (!b->cached_seq_len || !b->num_new_tokens || !b->cu_new_tokens || !b->block_table)
        return CPA_ERR_INVALID_ARG;
    long long total = 0;
    const long long cap = (long long)b->max_blocks_per_seq * p->block_size;
    for (int r = 0; r < b->num_reqs; ++r) {
        const long long C = b->h_cached_seq_len[r], N = b->h_num_new_tokens[r];
        if (C < 0 || N < 0 || C + N > cap || C + N > INT32_MAX / 2) return CPA_ERR_INVALID_ARG;
        total += N;
    }
    if (total != b->total_new_tokens) return CPA_ERR_INVALID_ARG;
    return CPA_SUCCESS;
}

bool kv_fp8(const cpa_params *p) { return p->kv_format == CPA_KV_FP8_E4M3; }

bool use_tensor_cores(const cpa_params *p) {
    if (p->dtype != CPA_DTYPE_BF16) return false;
    if (p->flags & CPA_FLAG_FORCE_SIMT) return false;
    const int G = p->num_heads_q / p->num_heads_kv;
    return G <= kTcTileM;
}

// Packed query rows of a tensor-core tile: the whole tokens that fit 128 MMA
// rows (a query tile is one TMA box of (d, G, 128 / G) -- G query heads of
// floor(128 / G) tokens), so that no token's rows straddle two tiles; the
// MMA rows past it (128 mod G of them) carry nothing that reaches an output.
int tc_tile_m(int G) { return G * (kTcTileM / G); }

struct Plan {
    int tile_m = 0;
    bool tc = false;         // the tensor-core kernels (else the CUDA-core one)
    bool tc2 = false;        // the two-pipeline tensor-core kernel (attn_tc2.cu)
    bool rope_fused = false; // the one-pipeline kernel rotates queries and keys itself
    int tiles_per_unit = 1;
    int head_major = 0;
    size_t sched_off = 0;   // byte offset of the work counter in the workspace
    size_t rq_off = 0, rk_off = 0;  // rotated q / k_new copies (rope_theta > 0)
    size_t kq_off = 0, vq_off = 0;  // FP8 cache: codes of k_new / v_new
    size_t q8_off = 0, qs_off = 0;  // FP8 cache: two E4M3 planes of the queries, their row scales
    size_t ws_bytes = 0;    // workspace bytes: partials, then (tensor-core path) the counter
    int split_len = 0;
    int split_len_fine = 0;
    int fine_from = INT32_MAX;  // first request whose pieces are split_len_fine long
    int fine_units = 0;         // their split units (the launch's last)
    int tail_units = 0;     // the last direct units run as tail_pieces pieces each
    int tail_pieces = 0;
    int group_ctas = 0;     // one-pipeline kernel: CTAs [0, group_ctas) take indices [0,
    int group_units = 0;    // group_units) first, the others the rest (0: one group)
    long long tail_ws_floats = 0;  // float offset of their partials
    int direct_units = 0;
    int split_units = 0;
    int split_reqs = 0;
    long long ws_floats = 0;
};

int elem_bytes(const cpa_params *p) { return p->dtype == CPA_DTYPE_FP32 ? 4 : 2; }
int pool_elem_bytes(const cpa_params *p) { return kv_fp8(p) ? 1 : elem_bytes(p); }

// Attention over FP8 pools runs on the tensor-core kernel only (d = 128).
cpa_status check_attention_support(const cpa_params *p) {
    if (kv_fp8(p) && (p->head_dim != 128 || !use_tensor_cores(p))) return CPA_ERR_UNSUPPORTED;
    return CPA_SUCCESS;
}

// Cost of a unit in periods of one key tile: its tiles plus the switch to it
// (the previous unit's last PV and epilogue, refilling the copy pipeline),
// about six tile periods by clock64 traces of the kernel.  A tail piece costs
// about twelve periods more (measured: chunks of 2048 query tokens cut this
// way ran 5 % slower over 2048 cached tokens, as fast over 4096, 3.5 %
// faster over 6144): its partial's write, the count, and the merge.
constexpr double kUnitSwitchTiles = 6.0;
constexpr double kTailPieceTiles = 12.0;

// Greedy list schedule, as the kernel's work counter hands out indices: each
// of the CTAs (a min-heap of their finish times) takes the next unit when it
// is free.
using FinishHeap = std::priority_queue<double, std::vector<double>, std::greater<double>>;

double schedule_end(FinishHeap h) {
    double end = 0;
    while (!h.empty()) {
        end = h.top();
        h.pop();
    }
    return end;
}

// Tail pieces for a batch of direct units only.  With U units of similar size
// on S SMs the last wave holds U mod S units and leaves the other SMs idle;
// cutting those units into p pieces by key tiles (each piece writes a partial,
// merged by the CTA that finishes the unit's last piece) spreads that work
// over more SMs.  Simulates the schedule without pieces and with the last k
// units in p pieces (k the last wave's units, and that plus half the SMs;
// p = 2, 3, 4) and keeps the best cut if it ends at least 2% sooner.
// Key tiles of every direct unit of a one-tile-per-unit plan, in work-counter
// order (the order decode_unit uses).
std::vector<int> direct_unit_tiles(const cpa_batch *b, const cpa_params *p, const Plan &pl) {
    const int G = p->num_heads_q / p->num_heads_kv, hkv = p->num_heads_kv;
    std::vector<int> tiles;
    tiles.reserve(pl.direct_units);
    for (int r = 0; r < b->num_reqs; ++r) {
        const int C = b->h_cached_seq_len[r], N = b->h_num_new_tokens[r];
        const ReqWork w = request_work(C, N, G, hkv, p->head_dim, pl.tile_m, pl.split_len, pl.tiles_per_unit);
        const int rows = N * G, n_qt = cdiv(rows, pl.tile_m);
        for (int local = 0; local < w.direct_units; ++local) {
            const int i = pl.head_major ? local % n_qt : local / hkv;
            const int last = n_qt - 1 - i;
            const int last_tok = (std::min((last + 1) * pl.tile_m, rows) - 1) / G;
            tiles.push_back(cdiv(C, kTcTileN) + cdiv(last_tok + 1, kTcTileN));
        }
    }
    return tiles;
}

void plan_tail(const cpa_batch *b, const cpa_params *p, int sms, Plan &pl) {
    const int D = pl.direct_units;
    if (sms <= 0 || D < sms || D > 8 * sms || pl.split_units > 0 || !(p->flags & CPA_FLAG_TAIL_SPLIT) ||
        (p->flags & CPA_FLAG_NO_SPLIT))
        return;
    // key tiles of every direct unit in index order
    const std::vector<int> tiles = direct_unit_tiles(b, p, pl);
    if ((int)tiles.size() != D) return;
    const int R = D % sms;
    std::vector<int> cuts;
    if (R > 0) cuts.push_back(R);
    if (R + sms / 2 <= D) cuts.push_back(R + sms / 2);
    if (cuts.empty()) return;
    std::sort(cuts.begin(), cuts.end(), std::greater<int>());  // head lengths D - k ascending
    FinishHeap h;
    for (int c = 0; c < sms; ++c) h.push(0.0);
    double best = -1;
    size_t next_cut = 0;
    for (int u = 0; u <= D; ++u) {
        while (next_cut < cuts.size() && D - cuts[next_cut] == u) {
            const int k = cuts[next_cut++];
            for (int pieces = 2; pieces <= kMaxTailPieces; ++pieces) {
                bool fits = true;
                for (int v = D - k; v < D && fits; ++v) fits = tiles[v] >= 2 * pieces;
                if (!fits) break;
                FinishHeap t = h;
                for (int v = D - k; v < D; ++v) {
                    for (int q = 0; q < pieces; ++q) {
                        const int n = (q + 1) * tiles[v] / pieces - q * tiles[v] / pieces;
                        const double f = t.top() + n + kUnitSwitchTiles + kTailPieceTiles;
                        t.pop();
                        t.push(f);
                    }
                }
                const double end = schedule_end(t);
                if (best < 0 || end < best) {
                    best = end;
                    pl.tail_units = k;
                    pl.tail_pieces = pieces;
                }
            }
        }
        if (u == D) break;
        const double f = h.top() + tiles[u] + kUnitSwitchTiles;
        h.pop();
        h.push(f);
    }
    if (best < 0 || best > 0.98 * schedule_end(h)) {
        pl.tail_units = 0;
        pl.tail_pieces = 0;
    }
}

// Two groups of CTAs for a batch of direct units only (one-pipeline kernel).
// With U units, heaviest first, on S CTAs (U = q S + R, 0 < R), a single
// work counter ends in a last wave of R units that the other CTAs wait for.
// The better packing gives S - R CTAs q of the heaviest units each and R CTAs
// q + 1 of the lightest: so CTAs [0, S - R) take indices [0, (S - R) q) from
// the work counter and the others the rest from a second counter, each group
// in its own greedy order, and a CTA whose group has run out takes the other
// group's next index.  Simulates both schedules (a unit costs its key tiles
// plus kGroupSwitchTiles) and keeps the groups if they end at least 2 %
// sooner: chunks of causal prompts over a cache gain (their units differ by
// at most 16 tiles of 17-48), a prompt's first chunk (units of 1-16 tiles,
// already balanced by the single counter) does not, and is not simulated.
constexpr int kGroupSwitchTiles = 3;
constexpr int kGroupMaxWaves = 8;

// End of the greedy schedule of units with integer costs (key tiles + the
// switch) on `sms` CTAs, the first group_ctas of them taking indices
// [0, group_units) first and the rest the others (group_ctas = 0: one
// counter).  CTAs of a group are alike, so the simulation keeps, per time
// step, how many CTAs of each group become free then: no heap.
int grouped_end(const std::vector<int> &tiles, int sms, int group_ctas, int group_units) {
    const int U = (int)tiles.size();
    long long total = 0;
    int longest = 0;
    for (int t : tiles) {
        total += t + kGroupSwitchTiles;
        longest = std::max(longest, t + kGroupSwitchTiles);
    }
    // every CTA is free again by total / sms + longest (a greedy list
    // schedule ends within one unit of the mean load)
    const int horizon = (int)(total / sms) + 2 * longest + 2;
    std::vector<int> free_at[2] = {std::vector<int>(horizon, 0), std::vector<int>(horizon, 0)};
    free_at[0][0] = group_ctas ? group_ctas : sms;
    free_at[1][0] = group_ctas ? sms - group_ctas : 0;
    int next[2] = {0, group_ctas ? group_units : U};
    const int end[2] = {group_ctas ? group_units : U, U};
    int last = 0;
    for (int t = 0; t < horizon; ++t) {
        for (int g = 0; g < 2; ++g) {
            for (int c = free_at[g][t]; c > 0; --c) {
                int u = -1;
                if (next[g] < end[g])
                    u = next[g]++;
                else if (next[1 - g] < end[1 - g])
                    u = next[1 - g]++;
                if (u < 0) {
                    last = t;
                    continue;
                }
                const int f = t + tiles[u] + kGroupSwitchTiles;
                if (f >= horizon) return INT32_MAX;  // not expected: treated as no gain
                ++free_at[g][f];
            }
        }
    }
    return last;
}

void plan_groups(const cpa_batch *b, const cpa_params *p, int sms, Plan &pl) {
    const int U = pl.direct_units;
    if (!pl.tc || pl.tc2 || sms <= 0 || pl.split_units > 0 || pl.tail_units > 0 || pl.head_major || U <= sms ||
        U > kGroupMaxWaves * sms || U % sms == 0)
        return;
    // units more than twice as long as others (a prompt's first chunk) are
    // balanced by the single counter already: no simulation (host time).  A
    // request's heaviest unit has all its keys, its lightest those of its
    // first query tile.
    const int G = p->num_heads_q / p->num_heads_kv;
    int lightest = INT32_MAX, heaviest = 0;
    for (int r = 0; r < b->num_reqs; ++r) {
        const int C = b->h_cached_seq_len[r], N = b->h_num_new_tokens[r];
        if (N <= 0) continue;
        const int first_tok = (std::min(pl.tile_m, N * G) - 1) / G;
        lightest = std::min(lightest, cdiv(C, kTcTileN) + cdiv(first_tok + 1, kTcTileN));
        heaviest = std::max(heaviest, cdiv(C, kTcTileN) + cdiv(N, kTcTileN));
    }
    if (2 * lightest < heaviest) return;
    const std::vector<int> tiles = direct_unit_tiles(b, p, pl);
    if ((int)tiles.size() != U) return;
    const int q = U / sms, R = U % sms;
    const int one = grouped_end(tiles, sms, 0, 0);
    const int two = grouped_end(tiles, sms, sms - R, (sms - R) * q);
    if (two < INT32_MAX && (double)two < 0.98 * one) {
        pl.group_ctas = sms - R;
        pl.group_units = (sms - R) * q;
    }
}

// Query tiles per direct unit for the two-pipeline kernel on a batch of
// direct units only: pairs, whose K/V tiles serve 256 rows, or single tiles
// split by keys over the two pipelines.  Both do the same tensor work; pairs
// halve the K/V copies (and TMA boxes) per FLOP, single tiles make twice as
// many units, which can fill the launch's last wave of CTAs better.  A greedy
// list schedule of the units (the work counter's order: requests in turn,
// each request's heaviest query tiles first, kv heads innermost) on `sms`
// CTAs, with costs in periods of 1024 cycles -- a key tile costs a pair 2
// periods and a single tile 1, or the TMA issue time of its K and V boxes
// (about 75 cycles a box) when that is longer, plus a switch of 4 periods per
// unit -- picks the one that ends sooner (pairs unless singles end 3 %
// sooner).  Batches with split units keep pairs.
constexpr double kBoxCycles = 75.0;
constexpr double kUnitSwitchPeriods = 4.0;

int choose_tiles_per_unit(const cpa_batch *b, const cpa_params *p, int sms, const Plan &pl) {
    if (sms <= 0 || pl.split_units > 0 || pl.direct_units == 0) return 2;
    const int G = p->num_heads_q / p->num_heads_kv, hkv = p->num_heads_kv;
    const int bs = std::min(p->block_size, kTcTileN);
    const double boxes = 2.0 * cdiv(kTcTileN, bs) * (p->head_dim / 64) * kBoxCycles / 1024.0;
    auto end_time = [&](int tpu) {
        FinishHeap h;
        for (int c = 0; c < sms; ++c) h.push(0.0);
        for (int r = 0; r < b->num_reqs; ++r) {
            const int C = b->h_cached_seq_len[r], N = b->h_num_new_tokens[r];
            if (N <= 0) continue;
            const int rows = N * G, n_qt = cdiv(rows, kTcTileM), groups = cdiv(n_qt, tpu);
            for (int i = 0; i < groups; ++i) {
                const int last = n_qt - 1 - i * tpu, first = std::max(0, last - tpu + 1);
                const int last_tok = (std::min((last + 1) * kTcTileM, rows) - 1) / G;
                const int n = cdiv(C, kTcTileN) + cdiv(last_tok + 1, kTcTileN);
                const double per_tile = last > first ? std::max(2.0, boxes) : std::max(1.0, boxes);
                const double cost = n * per_tile + kUnitSwitchPeriods;
                for (int g = 0; g < hkv; ++g) {
                    const double f = h.top() + cost;
                    h.pop();
                    h.push(f);
                }
            }
        }
        return schedule_end(h);
    };
    return end_time(1) < 0.97 * end_time(2) ? 1 : 2;
}

// Ints at the workspace's counter offset, zeroed before each tensor-core
// launch: the work counter, kSoftmaxWarpsMax per tail unit, with the rotary
// embedding the rotation's claim and done counts and one done count per
// 128-row tile of the new rows, and with two CTA groups the second group's
// work counter.
size_t counter_ints(const cpa_batch *b, const Plan &pl) {
    size_t n = 1 + (size_t)pl.tail_units * kSoftmaxWarpsMax;
    if (pl.rope_fused) n += 2 + (size_t)cdiv(b->total_new_tokens, kTcTileN);
    if (pl.group_ctas) n += 1;  // the second group's work counter, last
    return n;
}

Plan make_plan(const cpa_batch *b, const cpa_params *p, int sms) {
    Plan pl;
    const bool tc = use_tensor_cores(p);
    const int G = p->num_heads_q / p->num_heads_kv;
    pl.tc = tc;
    pl.tile_m = tc ? tc_tile_m(G) : kSimtTileM;
    // The two-pipeline kernel (attn_tc2.cu) runs BF16 batches at block sizes
    // 16 and 32 that have query tiles to pair: a 128-key tile there takes 16
    // or 8 TMA boxes per operand, and pairs halve the boxes per FLOP.  The
    // one-pipeline kernel (attn_tc.cu) runs the rest -- block sizes 64 and
    // 128, decode-only batches (both measured faster on it), FP8 pools and
    // the opt-in tail cut, and query groups that do not divide 128.  Pairs
    // unless a batch of direct units only schedules better with single tiles
    // (choose_tiles_per_unit, below).
    bool pairs = false;
    for (int r = 0; r < b->num_reqs && !pairs; ++r)
        pairs = (long long)b->h_num_new_tokens[r] * G > kTcTileM;
    const bool rope = p->rope_theta > 0.f;
    pl.tc2 = tc && (kTcTileM % G) == 0 && !kv_fp8(p) && !(p->flags & CPA_FLAG_TAIL_SPLIT) && p->block_size <= 32 &&
             pairs;
    // the one-pipeline kernel applies the rotary embedding in the same launch;
    // the two-pipeline kernel reads rotated copies from the pre-pass
    pl.rope_fused = tc && !kv_fp8(p) && rope && !pl.tc2;
    pl.tiles_per_unit = pl.tc2 ? 2 : 1;
    pl.split_len = (p->flags & CPA_FLAG_NO_SPLIT) ? 0 : (p->kv_segment_size > 0 ? p->kv_segment_size : kDefaultSplit);
    // fewer, longer split units while the batch keeps enough of them: every
    // unit costs a switch (its lookups, the epilogue, the pipeline's refill)
    for (int len = pl.split_len * 2; pl.split_len > 0 && len <= kMaxSplitLen; len *= 2) {
        long long units = 0;
        for (int r = 0; r < b->num_reqs; ++r) {
            const ReqWork w = request_work(b->h_cached_seq_len[r], b->h_num_new_tokens[r], G, p->num_heads_kv,
                                           p->head_dim, pl.tile_m, len, pl.tiles_per_unit);
            units += w.direct_units + w.split_units;
        }
        if (units < kSplitTargetUnits) break;
        pl.split_len = len;
    }
    // the persistent kernel's last wave: the last decode requests' keys in
    // shorter pieces, enough for kFineTailWaves waves of CTAs
    const int base = (p->flags & CPA_FLAG_NO_SPLIT) ? 0 : (p->kv_segment_size > 0 ? p->kv_segment_size : kDefaultSplit);
    if (tc && sms > 0 && base > 0 && pl.split_len > base) {
        const int fine = std::max(base, pl.split_len / 2);
        long long fu = 0;
        int r1 = b->num_reqs;
        for (int r = b->num_reqs - 1; r >= 0 && fu < (long long)kFineTailWaves * sms; --r) {
            fu += request_work(b->h_cached_seq_len[r], b->h_num_new_tokens[r], G, p->num_heads_kv, p->head_dim,
                               pl.tile_m, fine, pl.tiles_per_unit)
                      .split_units;
            r1 = r;
        }
        if (fu > 0) {
            pl.fine_from = r1;
            pl.split_len_fine = fine;
        }
    }
    double kv_bytes = 0;
    for (int r = 0; r < b->num_reqs; ++r) {
        const int len = r >= pl.fine_from ? pl.split_len_fine : pl.split_len;
        const ReqWork w = request_work(b->h_cached_seq_len[r], b->h_num_new_tokens[r], G, p->num_heads_kv,
                                       p->head_dim, pl.tile_m, len, pl.tiles_per_unit);
        pl.direct_units += w.direct_units;
        pl.split_units += w.split_units;
        if (r >= pl.fine_from) pl.fine_units += w.split_units;
        pl.split_reqs += w.split_units > 0 ? 1 : 0;
        pl.ws_floats += w.ws_floats;
        kv_bytes += (double)(b->h_cached_seq_len[r] + b->h_num_new_tokens[r]) * p->num_heads_kv * p->head_dim * 2.0 *
                    pool_elem_bytes(p);
    }
    // K/V of the batch larger than about half of L2: walk the direct units
    // head by head so that concurrent CTAs share K/V tiles in L2
    pl.head_major = kv_bytes > kHeadMajorKvBytes ? 1 : 0;
    if (pl.tc2 && choose_tiles_per_unit(b, p, sms, pl) == 1) {
        pl.tiles_per_unit = 1;
        pl.direct_units = 0;
        for (int r = 0; r < b->num_reqs; ++r)
            pl.direct_units += request_work(b->h_cached_seq_len[r], b->h_num_new_tokens[r], G, p->num_heads_kv,
                                            p->head_dim, pl.tile_m, pl.split_len, 1)
                                   .direct_units;
    }
    if (tc) plan_tail(b, p, sms, pl);
    if (tc) plan_groups(b, p, sms, pl);
    if (pl.tail_units > 0) {
        pl.tail_ws_floats = pl.ws_floats;
        pl.ws_floats += (long long)pl.tail_units * pl.tail_pieces * partial_floats(pl.tile_m, p->head_dim);
    }
    pl.ws_bytes = (size_t)pl.ws_floats * sizeof(float);
    const size_t T = (size_t)b->total_new_tokens, es = (size_t)elem_bytes(p), d = (size_t)p->head_dim;
    auto take = [&](size_t bytes) {  // next 256-byte aligned part of the workspace
        const size_t off = (pl.ws_bytes + 255) & ~(size_t)255;
        pl.ws_bytes = off + bytes;
        return off;
    };
    if (kv_fp8(p)) {
        // the (rotated) queries as two E4M3 planes with their row scales, and
        // the new rows as the FP8 cache holds them, which the attention reads
        pl.q8_off = take(2 * T * p->num_heads_q * d);
        pl.qs_off = take(T * p->num_heads_q * sizeof(float));
        pl.kq_off = take(T * p->num_heads_kv * d);
        pl.vq_off = take(T * p->num_heads_kv * d);
    } else if (pl.rope_fused) {
        // the rotated copy of k_new, which the tensor-core kernel writes and
        // reads (its queries are rotated in shared memory)
        pl.rk_off = take(T * p->num_heads_kv * d * es);
    } else if (p->rope_theta > 0.f) {
        // rotated copies of q and k_new, which the attention then reads
        pl.rq_off = take(T * p->num_heads_q * d * es);
        pl.rk_off = take(T * p->num_heads_kv * d * es);
    }
    if (tc) {
        // the persistent kernel's work counter, the tail units' counters and
        // the key rotation's counters, after the partials
        pl.sched_off = (pl.ws_bytes + 255) & ~(size_t)255;
        const size_t counters = sizeof(int) * counter_ints(b, pl);
        pl.ws_bytes = pl.sched_off + ((counters + 255) & ~(size_t)255);
    }
    return pl;
}


// 16-bit tiles land 128-byte swizzled (the MMA operand layout), as do the
// E4M3 tiles the score MMA reads (kCodesMma: query planes, key codes); value
// code tiles land as plain rows for the expansion warps (kCodes)
enum class MapType { kBf16, kF16, kCodes, kCodesMma };

cpa_status encode(CUtensorMap *map, const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                  const cuuint32_t *box, MapType type = MapType::kBf16) {
    auto enc = tensor_map_encoder();
    if (!enc) return CPA_ERR_CUDA;
    const cuuint32_t es[4] = {1, 1, 1, 1};
    const bool codes = type == MapType::kCodes || type == MapType::kCodesMma;
    const CUtensorMapDataType dt = codes ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : type == MapType::kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                           : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUresult r = enc(map, dt, (cuuint32_t)rank,
                     const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     type == MapType::kCodes ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? CPA_SUCCESS : CPA_ERR_CUDA;
}

cpa_status make_tc_maps(const cpa_batch *b, const cpa_params *p, const void *q, const void *k_new, const void *v_new,
                        const void *k_cache, const void *v_cache, TcMaps &m) {
    const cuuint64_t D = (cuuint64_t)p->head_dim, Hq = (cuuint64_t)p->num_heads_q, Hkv = (cuuint64_t)p->num_heads_kv;
    const cuuint64_t T = (cuuint64_t)b->total_new_tokens, bs = (cuuint64_t)p->block_size;
    const cuuint32_t G = (cuuint32_t)(p->num_heads_q / p->num_heads_kv);
    if (kv_fp8(p)) {
        // with the FP8 cache q is the pre-pass's two E4M3 planes [2][T, H_q, d]:
        // a box is one plane's (d bytes, G heads, 128 / G tokens)
        const cuuint64_t dims[4] = {D, Hq, T, 2};
        const cuuint64_t strides[3] = {D, Hq * D, T * Hq * D};
        const cuuint32_t box[4] = {(cuuint32_t)D, G, (cuuint32_t)kTcTileM / G, 1};
        if (cpa_status s = encode(&m.q, q, 4, dims, strides, box, MapType::kCodesMma)) return s;
    } else {
        const cuuint64_t dims[3] = {D, Hq, T};
        const cuuint64_t strides[2] = {D * 2, Hq * D * 2};
        const cuuint32_t box[3] = {64, G, (cuuint32_t)kTcTileM / G};
        if (cpa_status s = encode(&m.q, q, 3, dims, strides, box)) return s;
    }
    const cuuint32_t box_rows = (cuuint32_t)(bs < (cuuint64_t)kTcTileN ? bs : (cuuint64_t)kTcTileN);
    if (kv_fp8(p)) {
        // codes: one byte per element, a box spans the whole d-byte head row
        const cuuint64_t dims3[3] = {D, Hkv, T};
        const cuuint64_t strides3[2] = {D, Hkv * D};
        const cuuint32_t box3[3] = {(cuuint32_t)D, 1, (cuuint32_t)kTcTileN};
        if (cpa_status s = encode(&m.k_new, k_new, 3, dims3, strides3, box3, MapType::kCodesMma)) return s;
        if (cpa_status s = encode(&m.v_new, v_new, 3, dims3, strides3, box3, MapType::kCodes)) return s;
        const cuuint64_t dims4[4] = {D, Hkv, bs, (cuuint64_t)p->num_blocks};
        const cuuint64_t strides4[3] = {D, Hkv * D, bs * Hkv * D};
        const cuuint32_t box4[4] = {(cuuint32_t)D, 1, box_rows, 1};
        if (cpa_status s = encode(&m.k_pool, k_cache, 4, dims4, strides4, box4, MapType::kCodesMma)) return s;
        return encode(&m.v_pool, v_cache, 4, dims4, strides4, box4, MapType::kCodes);
    }
    {
        const cuuint64_t dims[3] = {D, Hkv, T};
        const cuuint64_t strides[2] = {D * 2, Hkv * D * 2};
        const cuuint32_t box[3] = {64, 1, (cuuint32_t)kTcTileN};
        if (cpa_status s = encode(&m.k_new, k_new, 3, dims, strides, box)) return s;
        if (cpa_status s = encode(&m.v_new, v_new, 3, dims, strides, box)) return s;
    }
    {
        const cuuint64_t dims[4] = {D, Hkv, bs, (cuuint64_t)p->num_blocks};
        const cuuint64_t strides[3] = {D * 2, Hkv * D * 2, bs * Hkv * D * 2};
        // one box is one block (or the 128 rows of a block one key tile covers)
        const cuuint32_t box[4] = {64, 1, box_rows, 1};
        if (cpa_status s = encode(&m.k_pool, k_cache, 4, dims, strides, box)) return s;
        if (cpa_status s = encode(&m.v_pool, v_cache, 4, dims, strides, box)) return s;
    }
    return CPA_SUCCESS;
}

RopeArgs rope_args(const cpa_batch *batch, const cpa_params *params, int *err) {
    RopeArgs r{};
    r.num_reqs = batch->num_reqs;
    r.max_blocks = batch->max_blocks_per_seq;
    r.total_tokens = batch->total_new_tokens;
    r.cached = batch->cached_seq_len;
    r.cu = batch->cu_new_tokens;
    r.bt = batch->block_table;
    r.hq = params->num_heads_q;
    r.hkv = params->num_heads_kv;
    r.d = params->head_dim;
    r.bs = params->block_size;
    r.num_blocks = params->num_blocks;
    r.elem_bytes = elem_bytes(params);
    r.rotate = params->rope_theta > 0.f ? 1 : 0;
    r.kv_fp8 = kv_fp8(params) ? 1 : 0;
    r.k_scale = params->k_scale;
    r.v_scale = params->v_scale;
    for (int c = 0; c < params->head_dim / 2 && r.rotate; ++c) {
        const double turns = pow((double)params->rope_theta, -2.0 * c / params->head_dim) / 6.283185307179586477;
        r.turn_frac[c] = (unsigned long long)ldexp(turns, 64);  // turns < 1 / (2 pi): fits
    }
    r.err = err;
    return r;
}

}  // namespace
}  // namespace cpa

using namespace cpa;

extern "C" {

int32_t cpa_version(void) { return 100; }

const char *cpa_status_string(cpa_status s) {
    switch (s) {
        case CPA_SUCCESS: return "success";
        case CPA_ERR_INVALID_ARG: return "invalid argument";
        case CPA_ERR_UNSUPPORTED: return "unsupported configuration or device";
        case CPA_ERR_CUDA: return "CUDA error";
        case CPA_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        case CPA_ERR_BAD_BLOCK_ID: return "block id outside the pool";
        case CPA_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

size_t chunked_prefill_workspace_size(const cpa_batch *batch, const cpa_params *params) {
    if (validate(batch, params) != CPA_SUCCESS || batch->num_reqs == 0) return 0;
    if (check_attention_support(params) != CPA_SUCCESS) return 0;
    DeviceInfo dev;  // the SM count shapes the plan (tail pieces); none without a device
    const int sms = device_info(dev) == CPA_SUCCESS ? dev.sms : 0;
    const Plan pl = make_plan(batch, params, sms);
    return pl.ws_bytes;
}

cpa_status paged_kv_write(const cpa_batch *batch, const cpa_params *params, const void *k_new, const void *v_new,
                          void *k_cache, void *v_cache, void *stream) {
    if (cpa_status s = validate(batch, params)) return s;
    if (batch->total_new_tokens == 0) return CPA_SUCCESS;
    if (!k_new || !v_new || !k_cache || !v_cache) return CPA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return CPA_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (cpa_status s = device_info(dev)) return s;
    if (params->rope_theta > 0.f || kv_fp8(params)) {
        // rotated keys (and the values) go to the pool, as E4M3 codes with the
        // FP8 cache; no copies are kept
        RopeArgs r = rope_args(batch, params, dev.err);
        r.k_new = k_new;
        r.v_new = v_new;
        r.write_pool = 1;
        r.k_cache = k_cache;
        r.v_cache = v_cache;
        return launch_rope(r, dev.sms, static_cast<cudaStream_t>(stream)) == cudaSuccess ? CPA_SUCCESS : CPA_ERR_CUDA;
    }
    KvWriteArgs a{};
    a.num_reqs = batch->num_reqs;
    a.max_blocks = batch->max_blocks_per_seq;
    a.total_tokens = batch->total_new_tokens;
    a.cached = batch->cached_seq_len;
    a.cu = batch->cu_new_tokens;
    a.bt = batch->block_table;
    a.hkv = params->num_heads_kv;
    a.bs = params->block_size;
    a.num_blocks = params->num_blocks;
    a.head_bytes = params->head_dim * elem_bytes(params);
    a.k_new = k_new;
    a.v_new = v_new;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.err = dev.err;
    return launch_kv_write(a, dev.sms, static_cast<cudaStream_t>(stream)) == cudaSuccess ? CPA_SUCCESS : CPA_ERR_CUDA;
}

cpa_status chunked_prefill_attention(const cpa_batch *batch, const cpa_params *params, const void *q,
                                     const void *k_new, const void *v_new, void *k_cache, void *v_cache, void *out,
                                     float *lse, void *workspace, size_t workspace_bytes, void *stream) {
    if (cpa_status s = validate(batch, params)) return s;
    if (batch->total_new_tokens == 0) return CPA_SUCCESS;
    if (!q || !k_new || !v_new || !k_cache || !v_cache || !out) return CPA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned16(out) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
        return CPA_ERR_INVALID_ARG;
    if (cpa_status s = check_attention_support(params)) return s;
    DeviceInfo dev;
    if (cpa_status s = device_info(dev)) return s;
    const Plan pl = make_plan(batch, params, dev.sms);
    const size_t need = pl.ws_bytes;
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace))) return CPA_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    bool fuse_write = (params->flags & CPA_FLAG_FUSE_KV_WRITE) != 0;
    const float *q_rscale = nullptr;
    const bool prepass = (params->rope_theta > 0.f && !pl.rope_fused) || kv_fp8(params);
    RopeArgs r{};
    if (prepass) {
        // pre-pass over the new rows: rotate q and k_new, encode the keys and
        // values for the FP8 cache, into workspace copies that the attention
        // then reads (and, for a fused write, put the rows as the pool holds
        // them into their slots).  Launched below, once every host-side step
        // that can fail is done.
        char *ws = static_cast<char *>(workspace);
        r = rope_args(batch, params, dev.err);
        r.q = q;
        r.k_new = k_new;
        r.v_new = v_new;
        r.q_rot = (r.rotate && !r.kv_fp8) ? ws + pl.rq_off : nullptr;
        r.k_rot = (r.rotate && !r.kv_fp8) ? ws + pl.rk_off : nullptr;
        r.k_q8 = r.kv_fp8 ? ws + pl.kq_off : nullptr;
        r.v_q8 = r.kv_fp8 ? ws + pl.vq_off : nullptr;
        r.q8 = r.kv_fp8 ? ws + pl.q8_off : nullptr;
        r.q_rscale = r.kv_fp8 ? reinterpret_cast<float *>(ws + pl.qs_off) : nullptr;
        r.write_pool = fuse_write ? 1 : 0;
        r.k_cache = k_cache;
        r.v_cache = v_cache;
        if (r.q_rot) q = r.q_rot;
        if (r.k_rot) k_new = r.k_rot;
        if (r.kv_fp8) {
            q = r.q8;
            k_new = r.k_q8;
            v_new = r.v_q8;
            q_rscale = r.q_rscale;
        }
        fuse_write = false;
    }

    AttnArgs a{};
    a.num_reqs = batch->num_reqs;
    a.max_blocks = batch->max_blocks_per_seq;
    a.total_tokens = batch->total_new_tokens;
    a.cached = batch->cached_seq_len;
    a.nnew = batch->num_new_tokens;
    a.cu = batch->cu_new_tokens;
    a.bt = batch->block_table;
    a.hq = params->num_heads_q;
    a.hkv = params->num_heads_kv;
    a.G = params->num_heads_q / params->num_heads_kv;
    a.d = params->head_dim;
    a.bs = params->block_size;
    a.num_blocks = params->num_blocks;
    a.scale_log2 = params->scale * 1.4426950408889634f;
    a.split_len = pl.split_len;
    a.split_len_fine = pl.split_len_fine;
    a.fine_from = pl.fine_from;
    a.tile_m = pl.tile_m;
    a.tiles_per_unit = pl.tiles_per_unit;
    a.head_major = pl.head_major;
    a.interleave = (pl.tc && pl.direct_units > 0 && pl.split_units > 0) ? 1 : 0;
    a.interleave_span = pl.direct_units + pl.split_units - pl.fine_units;
    a.num_direct_units = pl.direct_units;
    a.num_split_units = pl.split_units;
    a.tail_units = pl.tail_units;
    a.group_ctas = pl.group_ctas;
    a.group_units = pl.group_units;
    a.tail_pieces = pl.tail_pieces;
    a.tail_ws = pl.tail_ws_floats;
    a.q = q;
    a.k_new = k_new;
    a.v_new = v_new;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.out = out;
    a.lse = lse;
    a.ws = static_cast<float *>(workspace);
    a.fuse_write = fuse_write ? 1 : 0;
    if (pl.tc && fuse_write) {
        if (!pl.tc2) {
            // the one-pipeline kernel's epilogue warps copy it while the
            // first units run
            a.write_share = 1;
        } else {
            const long long pieces = (long long)batch->total_new_tokens * params->num_heads_kv *
                                     (params->head_dim * elem_bytes(params) / 16);
            a.write_chunks = (int)((pieces + kWriteChunkPieces - 1) / kWriteChunkPieces);
        }
    }
    const int units = attention_units(a);
    // the tensor-core kernel is persistent: at most one CTA per SM, and no
    // more than it has attention units and write pieces
    const int work = units + a.write_chunks;
    a.write_ctas = pl.tc ? (work < dev.sms ? work : dev.sms) : units;
    a.err = dev.err;
    a.timeout_cycles = params->timeout_cycles > 0 ? params->timeout_cycles : kDefaultTimeoutCycles;
    a.test_stall = (params->flags & CPA_FLAG_TEST_STALL) ? 1 : 0;
    a.kv_fp8 = kv_fp8(params) ? 1 : 0;
    a.k_scale = params->k_scale;
    a.v_scale = params->v_scale;
    a.q_rscale = q_rscale;
    if (pl.rope_fused) {
        // the kernel rotates the keys from the caller's k_new into the
        // workspace copy, which then stands for k_new (its tiles, the write)
        const RopeArgs ra = rope_args(batch, params, dev.err);
        a.rope = 1;
        a.rope_pieces = cdiv(batch->total_new_tokens, kRopePieceTokens);
        a.k_src = k_new;
        k_new = static_cast<char *>(workspace) + pl.rk_off;
        a.k_new = k_new;
        for (int c = 0; c < 64; ++c) a.turn_frac[c] = ra.turn_frac[c];
    }

    cudaError_t e;
    if (pl.tc) {
        TcMaps maps;
        if (cpa_status s = make_tc_maps(batch, params, q, k_new, v_new, k_cache, v_cache, maps)) return s;
        if (prepass && launch_rope(r, dev.sms, st) != cudaSuccess) return CPA_ERR_CUDA;
        a.sched = reinterpret_cast<int *>(static_cast<char *>(workspace) + pl.sched_off);
        a.tail_count = pl.tail_units > 0 ? a.sched + 1 : nullptr;
        a.rope_count = pl.rope_fused ? a.sched + 1 + (size_t)pl.tail_units * kSoftmaxWarpsMax : nullptr;
        a.sched_b = pl.group_ctas ? a.sched + counter_ints(batch, pl) - 1 : nullptr;
        e = cudaMemsetAsync(a.sched, 0, sizeof(int) * counter_ints(batch, pl), st);
        if (e == cudaSuccess) e = pl.tc2 ? launch_attn_tc2(a, maps, st) : launch_attn_tc(a, maps, st);
    } else {
        // the CUDA-core kernel (its pre-pass is RoPE only: FP8 pools need the
        // tensor-core kernel)
        e = prepass ? launch_rope(r, dev.sms, st) : cudaSuccess;
        if (e == cudaSuccess) e = launch_attn_simt(a, params->dtype, st);
    }
    if (e != cudaSuccess) return CPA_ERR_CUDA;
    if (pl.split_reqs > 0) {
        e = launch_attn_merge(a, params->dtype, pl.split_reqs, st);
        if (e != cudaSuccess) return CPA_ERR_CUDA;
    }
    return CPA_SUCCESS;
}

cpa_status cpa_last_device_error(void *stream) {
    DeviceInfo dev;
    if (cpa_status s = device_info(dev)) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaMemcpyAsync(&v, dev.err, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return CPA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return CPA_ERR_CUDA;
    if (v != 0) {
        if (cudaMemsetAsync(dev.err, 0, sizeof(int), st) != cudaSuccess) return CPA_ERR_CUDA;
        if (cudaStreamSynchronize(st) != cudaSuccess) return CPA_ERR_CUDA;
    }
    return static_cast<cpa_status>(v);
}

}  // extern "C"
