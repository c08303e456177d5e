// ptx_sm100.cuh -- thin inline-PTX wrappers for the Blackwell (sm_100 family,
// built here for sm_103a) features the kernels use: mbarriers, TMA tensor
// loads, and the 5th-generation tensor cores (tcgen05) with their tensor
// memory (TMEM).  Each wrapper is one PTX instruction; the encodings of the
// shared-memory matrix descriptor and of the instruction descriptor follow
// the PTX ISA's tcgen05 chapter (Matrix Descriptors; Instruction
// descriptor for .kind::f16).
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace cpa {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the phase with the given parity has completed, for at most
// `limit` SM clock cycles.  Returns false when the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, long long limit) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) return false;
    }
    return true;
}

// As mbar_wait, and also gives up (returns false) once *abort is set.  The
// flag is read only while the phase is still open, so a wait on a phase
// that has already completed costs one try_wait.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t *bar, uint32_t parity, long long limit,
                                                   const volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort || clock64() - t0 > limit) return false;
    }
    return true;
}

// ------------------------------------------------------- register budget
// Move registers between warpgroups of a running CTA (every warp of the
// warpgroup executes it).  `dec` returns registers to the CTA's pool, `inc`
// waits until the pool can give them.
template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar, int c0, int c1,
                                            int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, uint64_t *bar, int c0, int c1,
                                            int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// as tma_load_4d, with an L2 eviction-priority policy made by createpolicy
__device__ __forceinline__ void tma_load_4d_hint(void *dst, const CUtensorMap *map, uint64_t *bar, int c0, int c1,
                                                 int c2, int c3, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(policy)
        : "memory");
}

// bring a tile of a 3-D tensor map into L2 (no shared-memory destination,
// no completion to wait for)
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap *map, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

// L2 policy: lines a copy brings in are the first to go (data read once)
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// make generic-proxy writes to shared memory visible to the async proxy
// (TMA, tensor cores)
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// order this thread's view of global memory (its own writes, and those of
// other threads that an acquire or a barrier ordered before this point)
// before its later async-proxy (TMA) accesses
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Add v to a global counter with release semantics at GPU scope: the
// caller's earlier writes (and those that a barrier ordered before it) are
// visible to whoever acquires the counter and reads the sum.
__device__ __forceinline__ void red_release_gpu_add(int *p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// barrier `id` (1..15) for `count` threads (a multiple of 32) of the CTA
__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------------------- tcgen05
// Allocation is warp-wide; the allocated column base is written to smem.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Add v to a global counter with acquire-release semantics at GPU scope and
// return the previous value: the caller's earlier writes (and those that a
// warp or CTA barrier ordered before it) are visible to whoever later
// acquires the counter, and the caller's later reads see the writes released
// by earlier adders.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int *p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Warp-wide forms of the two MMA shapes and of the commit: the whole warp
// executes them converged and one elected lane issues the instruction.
// Issuing from a converged warp keeps the descriptors in uniform registers;
// a lone lane in a divergent branch pays a much longer issue latency per MMA.
__device__ __forceinline__ void umma_ss_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// As umma_ss_warp / umma_ts_warp with each shared-memory descriptor passed as
// its two 32-bit halves.  The start address (bits 0-13) and the leading
// byte offset (bits 16-29) sit in the low half, so a k-step or a ring slot
// changes only that half: one 32-bit add per operand instead of 64-bit math.
__device__ __forceinline__ void umma_ss_warp2(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t desc_hi,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t.reg .b64 ad, bd;\n\t"
        "mov.b64 ad, {%1, %3};\n\t"
        "mov.b64 bd, {%2, %3};\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %4, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_lo), "r"(b_lo), "r"(desc_hi), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_ts_warp2(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t desc_hi,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t.reg .b64 bd;\n\t"
        "mov.b64 bd, {%2, %3};\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"(desc_hi), "r"(idesc), "r"(accumulate)
        : "memory");
}

// One score tile S = Q K^T at head_dim 128: eight MMAs (K steps of 16
// elements) issued by one elected lane under a single elect.sync.  Q and K
// are K-major 128-byte-swizzled tiles of two 64-column halves; a K step
// advances both descriptors' start address by 32 bytes (2 in 16-byte units)
// and the second half starts half_units later.  The first MMA overwrites D.
__device__ __forceinline__ void umma_s_tile128(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t desc_hi,
                                               uint32_t idesc, uint32_t half_units) {
    asm volatile(
        "{\n\t.reg .pred e, pf, pt;\n\t.reg .b32 a, b;\n\t.reg .b64 ad, bd;\n\t"
        "setp.ne.b32 pf, 0, 0;\n\t"
        "setp.eq.b32 pt, 0, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "mov.b64 ad, {%1, %3};\n\tmov.b64 bd, {%2, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %4, pf;\n\t"
        "add.u32 a, %1, 2;\n\tadd.u32 b, %2, 2;\n\tmov.b64 ad, {a, %3};\n\tmov.b64 bd, {b, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %4, pt;\n\t"
        "add.u32 a, %1, 4;\n\tadd.u32 b, %2, 4;\n\tmov.b64 ad, {a, %3};\n\tmov.b64 bd, {b, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %4, pt;\n\t"
        "add.u32 a, %1, 6;\n\tadd.u32 b, %2, 6;\n\tmov.b64 ad, {a, %3};\n\tmov.b64 bd, {b, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %4, pt;\n\t"
        "add.u32 a, %1, %5;\n\tadd.u32 b, %2, %5;\n\tmov.b64 ad, {a, %3};\n\tmov.b64 bd, {b, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %4, pt;\n\t"
        "add.u32 a, a, 2;\n\tadd.u32 b, b, 2;\n\tmov.b64 ad, {a, %3};\n\tmov.b64 bd, {b, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %4, pt;\n\t"
        "add.u32 a, a, 2;\n\tadd.u32 b, b, 2;\n\tmov.b64 ad, {a, %3};\n\tmov.b64 bd, {b, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %4, pt;\n\t"
        "add.u32 a, a, 2;\n\tadd.u32 b, b, 2;\n\tmov.b64 ad, {a, %3};\n\tmov.b64 bd, {b, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %4, pt;\n\t}\n" ::"r"(d_tmem),
        "r"(a_lo), "r"(b_lo), "r"(desc_hi), "r"(idesc), "r"(half_units)
        : "memory");
}

// One score tile S = (Qa + Qb) K^T at head_dim 128 with E4M3 operands: the
// queries as two E4M3 planes (a row and its rounding residual), each a
// K-major 128-byte-swizzled tile of 128 one-byte columns, and K one such
// tile of codes.  Four .kind::f8f6f4 MMAs per plane (K steps of 32 elements
// = 32 bytes = 2 units), the eight under one elect.sync; plane b starts
// plane_units after plane a.  The first MMA overwrites D.
__device__ __forceinline__ void umma_s_tile_e4m3(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t desc_hi,
                                                 uint32_t idesc, uint32_t plane_units) {
    asm volatile(
        "{\n\t.reg .pred e, pf, pt;\n\t.reg .b32 a, b;\n\t.reg .b64 ad, bd;\n\t"
        "setp.ne.b32 pf, 0, 0;\n\t"
        "setp.eq.b32 pt, 0, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "mov.b64 ad, {%1, %3};\n\tmov.b64 bd, {%2, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], ad, bd, %4, pf;\n\t"
        "add.u32 a, %1, 2;\n\tadd.u32 b, %2, 2;\n\tmov.b64 ad, {a, %3};\n\tmov.b64 bd, {b, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], ad, bd, %4, pt;\n\t"
        "add.u32 a, %1, 4;\n\tadd.u32 b, %2, 4;\n\tmov.b64 ad, {a, %3};\n\tmov.b64 bd, {b, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], ad, bd, %4, pt;\n\t"
        "add.u32 a, %1, 6;\n\tadd.u32 b, %2, 6;\n\tmov.b64 ad, {a, %3};\n\tmov.b64 bd, {b, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], ad, bd, %4, pt;\n\t"
        "add.u32 a, %1, %5;\n\tmov.b64 ad, {a, %3};\n\tmov.b64 bd, {%2, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], ad, bd, %4, pt;\n\t"
        "add.u32 a, a, 2;\n\tadd.u32 b, %2, 2;\n\tmov.b64 ad, {a, %3};\n\tmov.b64 bd, {b, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], ad, bd, %4, pt;\n\t"
        "add.u32 a, a, 2;\n\tadd.u32 b, b, 2;\n\tmov.b64 ad, {a, %3};\n\tmov.b64 bd, {b, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], ad, bd, %4, pt;\n\t"
        "add.u32 a, a, 2;\n\tadd.u32 b, b, 2;\n\tmov.b64 ad, {a, %3};\n\tmov.b64 bd, {b, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], ad, bd, %4, pt;\n\t}\n" ::"r"(d_tmem),
        "r"(a_lo), "r"(b_lo), "r"(desc_hi), "r"(idesc), "r"(plane_units)
        : "memory");
}

// One PV product over a 128-key tile: O (+)= P V with P read from TMEM
// (16 keys = 8 columns of bf16 pairs per MMA) and V an MN-major tile (16 key
// rows = 2048 bytes = 128 units per MMA); eight MMAs under one elect.sync.
// The first MMA accumulates only when accumulate is non-zero.
__device__ __forceinline__ void umma_pv_tile128(uint32_t d_tmem, uint32_t p_tmem, uint32_t b_lo, uint32_t desc_hi,
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p0, pt;\n\t.reg .b32 t, b;\n\t.reg .b64 bd;\n\t"
        "setp.ne.b32 p0, %5, 0;\n\t"
        "setp.eq.b32 pt, 0, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "mov.b64 bd, {%2, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, p0;\n\t"
        "add.u32 t, %1, 8;\n\tadd.u32 b, %2, 128;\n\tmov.b64 bd, {b, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t], bd, %4, pt;\n\t"
        "add.u32 t, t, 8;\n\tadd.u32 b, b, 128;\n\tmov.b64 bd, {b, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t], bd, %4, pt;\n\t"
        "add.u32 t, t, 8;\n\tadd.u32 b, b, 128;\n\tmov.b64 bd, {b, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t], bd, %4, pt;\n\t"
        "add.u32 t, t, 8;\n\tadd.u32 b, b, 128;\n\tmov.b64 bd, {b, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t], bd, %4, pt;\n\t"
        "add.u32 t, t, 8;\n\tadd.u32 b, b, 128;\n\tmov.b64 bd, {b, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t], bd, %4, pt;\n\t"
        "add.u32 t, t, 8;\n\tadd.u32 b, b, 128;\n\tmov.b64 bd, {b, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t], bd, %4, pt;\n\t"
        "add.u32 t, t, 8;\n\tadd.u32 b, b, 128;\n\tmov.b64 bd, {b, %3};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [t], bd, %4, pt;\n\t}\n" ::"r"(d_tmem),
        "r"(p_tmem), "r"(b_lo), "r"(desc_hi), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit_warp(uint64_t *bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}\n" ::"r"(smem_u32(bar))
        : "memory");
}

// Arrive once on `bar` when every tcgen05 MMA issued so far by this thread
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp gets lane
// (taddr.lane + t), columns taddr.col .. +31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns (thread t: lane taddr.lane + t).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// 16 lanes x 32-bit columns, two halves: threads 0-15 access lanes
// taddr.lane + t, columns taddr.col .. +31; threads 16-31 the same lanes at
// columns taddr.col + SPLIT .. +31.  Two threads thus share one TMEM lane
// (matrix row), each holding part of its columns.
template <int SPLIT>
__device__ __forceinline__ void tmem_ld16x2_32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32], %33;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr), "n"(SPLIT)
        : "memory");
}

template <int SPLIT>
__device__ __forceinline__ void tmem_st16x2_32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x32bx2.x32.b32 [%0], %33, "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "n"(SPLIT)
        : "memory");
}

// Shared-memory matrix descriptor (tcgen05): start address, leading and
// stride byte offsets (all >> 4), version 1, base offset 0, swizzle mode.
constexpr uint64_t kSwizzle128B = 2;

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint64_t swizzle) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
    d |= swizzle << 61;
    return d;
}

// Instruction descriptor, .kind::f16 with bf16 inputs and f32 accumulate.
// a_mn / b_mn: operand stored MN-major (1) instead of K-major (0).
// kind::f16 with fp32 accumulation; A and B both bf16 (bf16 = true) or both
// fp16 (bf16 = false)
__host__ __device__ constexpr uint32_t idesc_16bit_f32(int M, int N, int a_mn, int b_mn, bool bf16) {
    return (1u << 4)                      // D format: f32
           | ((bf16 ? 1u : 0u) << 7)      // A format: bf16 (1) or f16 (0)
           | ((bf16 ? 1u : 0u) << 10)     // B format: likewise
           | ((uint32_t)a_mn << 15)       // A major
           | ((uint32_t)b_mn << 16)       // B major
           | ((uint32_t)(N >> 3) << 17)   // N / 8
           | ((uint32_t)(M >> 4) << 24);  // M / 16
}

__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn, int b_mn) {
    return idesc_16bit_f32(M, N, a_mn, b_mn, true);
}

// Instruction descriptor, .kind::f8f6f4 with E4M3 A and B (format code 0 in
// bits 7-9 and 10-12), both K-major, fp32 accumulate.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
    return (1u << 4)                      // D format: f32
           | ((uint32_t)(N >> 3) << 17)   // N / 8
           | ((uint32_t)(M >> 4) << 24);  // M / 16
}

}  // namespace ptx
}  // namespace cpa
