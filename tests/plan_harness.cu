// plan_harness.cu -- test infrastructure: runs the library's host-side work
// planner (make_plan) for a batch read from stdin, with a given SM count, and
// prints the plan.  The planner's source is included in this translation unit;
// the kernel launchers it refers to are stubs (nothing here touches a GPU).
//
// stdin: sms hq hkv d bs kv_segment_size dtype flags kv_format num_reqs, then
// num_reqs pairs (cached_seq_len num_new_tokens), then optionally rope_theta.
#include "../chunked_prefill_paged_gb300/csrc/cpa_api.cu"

#include <stdio.h>
#include <vector>

namespace cpa {
cudaError_t launch_kv_write(const KvWriteArgs &, int, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_rope(const RopeArgs &, int, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_attn_simt(const AttnArgs &, int, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_attn_merge(const AttnArgs &, int, int, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_attn_tc(const AttnArgs &, const TcMaps &, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_attn_tc2(const AttnArgs &, const TcMaps &, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace cpa

int main() {
    int sms, hq, hkv, d, bs, seg, dtype, kv_format, n;
    unsigned flags;
    if (scanf("%d %d %d %d %d %d %d %u %d %d", &sms, &hq, &hkv, &d, &bs, &seg, &dtype, &flags, &kv_format, &n) != 10)
        return 2;
    std::vector<int32_t> C(n), N(n);
    int total = 0, longest = 0;
    for (int r = 0; r < n; ++r) {
        if (scanf("%d %d", &C[r], &N[r]) != 2) return 2;
        total += N[r];
        longest = C[r] + N[r] > longest ? C[r] + N[r] : longest;
    }
    float rope_theta = 0.f;
    if (scanf("%f", &rope_theta) != 1) rope_theta = 0.f;
    cpa_batch b{};
    b.num_reqs = n;
    b.max_blocks_per_seq = (longest + bs - 1) / bs;
    b.total_new_tokens = total;
    b.h_cached_seq_len = C.data();
    b.h_num_new_tokens = N.data();
    cpa_params p{};
    p.num_heads_q = hq;
    p.num_heads_kv = hkv;
    p.head_dim = d;
    p.block_size = bs;
    p.num_blocks = 1 << 30;
    p.kv_segment_size = seg;
    p.scale = 1.f;
    p.dtype = dtype;
    p.flags = flags;
    p.kv_format = kv_format;
    p.rope_theta = rope_theta;
    const cpa::Plan pl = cpa::make_plan(&b, &p, sms);
    printf("{\"split_len\": %d, \"split_len_fine\": %d, \"fine_from\": %d, \"fine_units\": %d, "
           "\"direct_units\": %d, \"split_units\": %d, \"split_reqs\": %d, \"tail_units\": %d, \"tail_pieces\": %d, "
           "\"head_major\": %d, \"interleave_span\": %d, \"ws_bytes\": %zu, \"sched_off\": %zu, "
           "\"tiles_per_unit\": %d, \"tc2\": %d, \"rope_fused\": %d, \"tile_m\": %d, \"group_ctas\": %d, "
           "\"group_units\": %d}\n",
           pl.split_len, pl.split_len_fine, pl.fine_from == INT32_MAX ? -1 : pl.fine_from, pl.fine_units,
           pl.direct_units, pl.split_units, pl.split_reqs, pl.tail_units, pl.tail_pieces, pl.head_major,
           pl.direct_units + pl.split_units - pl.fine_units, pl.ws_bytes, pl.sched_off, pl.tiles_per_unit, pl.tc2 ? 1 : 0,
           pl.rope_fused ? 1 : 0, pl.tile_m, pl.group_ctas, pl.group_units);
    return 0;
}
