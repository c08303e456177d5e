// tc_common.cuh -- pieces shared by the tensor-core attention kernels
// (attn_tc.cu: one query tile per unit, BF16 and FP8 pools; attn_tc2.cu: two
// query tiles per unit, BF16 pools): the key-tile walk of a unit, the ring
// through which the scheduling warp hands decoded units to the other roles,
// and small math helpers.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "device_common.cuh"
#include "ptx_sm100.cuh"

namespace cpa {
namespace tc {

constexpr int kKT = kTcTileN;  // keys per K/V tile (128)
constexpr int kUnitRing = 4;   // unit indices passed ahead to the other roles

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
    // tiles of the keys [k_begin, kend) for kend <= k_end: a prefix of the list
    __device__ __forceinline__ int tiles_until(int kend) const {
        const int ce = min(kend, cached_end);
        const int nc = ce > k_begin ? cdiv(ce - k_begin, kKT) : 0;
        return nc + (kend > new_begin ? cdiv(kend - new_begin, kKT) : 0);
    }
};

// The ring through which the scheduling warp publishes each claimed unit:
// its index and its decoded fields, one mbarrier pair per slot.
struct UnitRing {
    uint64_t full[kUnitRing], empty[kUnitRing];
    int index[kUnitRing];
    Unit desc[kUnitRing];
};

// A decoded unit through a ring slot: the scheduling warp decodes each unit
// once, as soon as it has claimed it, and every other role copies the fields
// (the slot's mbarrier orders the stores before the loads).
__device__ __forceinline__ void put_unit(Unit &dst, const Unit &u) {
    volatile int *d = reinterpret_cast<volatile int *>(&dst);
    const int *v = reinterpret_cast<const int *>(&u);
#pragma unroll
    for (int k = 0; k < (int)(sizeof(Unit) / 4); ++k) d[k] = v[k];
}
__device__ __forceinline__ void get_unit(Unit &u, const Unit &src) {
    const volatile int *d = reinterpret_cast<const volatile int *>(&src);
    int *v = reinterpret_cast<int *>(&u);
#pragma unroll
    for (int k = 0; k < (int)(sizeof(Unit) / 4); ++k) v[k] = d[k];
}

// The i-th unit of this CTA, as published by the scheduling warp (every lane
// of the calling warp takes part): its index, and for an attention unit its
// decoded fields in u.  The index is >= the unit count for a piece of the K/V
// write or when the CTA is done; -1 when the wait gave up (timeout or abort).
// With release = false the slot stays held (its fields valid) until
// reread_unit(ring, i, u) copies them again and releases it.
__device__ __forceinline__ int read_unit(UnitRing &ring, int i, long long limit, const volatile int *abort_flag,
                                         Unit &u, bool release = true) {
    const int s = i % kUnitRing;
    if (!__all_sync(0xffffffffu, ptx::mbar_wait_or_abort(&ring.full[s], (uint32_t)((i / kUnitRing) & 1), limit,
                                                         abort_flag)))
        return -1;
    const int unit = *reinterpret_cast<volatile int *>(&ring.index[s]);
    get_unit(u, ring.desc[s]);
    __syncwarp();
    if (release && (threadIdx.x & 31) == 0) ptx::mbar_arrive(&ring.empty[s]);
    return unit;
}

// The unit of held slot i (read before with release = false), released now.
__device__ __forceinline__ int reread_unit(UnitRing &ring, int i, Unit &u) {
    const int s = i % kUnitRing;
    const int unit = *reinterpret_cast<volatile int *>(&ring.index[s]);
    get_unit(u, ring.desc[s]);
    __syncwarp();
    if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(&ring.empty[s]);
    return unit;
}

// Publish unit index `unit` (decoded into u when it is an attention unit) in
// ring slot i % kUnitRing; called by lane 0 of the scheduling warp once every
// reader has released the slot's previous use.
__device__ __forceinline__ void publish_unit(UnitRing &ring, int i, int unit, const Unit &u) {
    const int s = i % kUnitRing;
    put_unit(ring.desc[s], u);
    ring.index[s] = unit;
    ptx::mbar_arrive(&ring.full[s]);  // release: index and fields are visible to every waiter
}

}  // namespace tc
}  // namespace cpa
