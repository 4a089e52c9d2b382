// device_common.cuh -- inline-PTX helpers for sm_103a kernels of this library:
// shared-memory mbarriers, bulk / tensor TMA copies, bounded waits and the
// device status word.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/pagedkv.h"

namespace pkv {

// A wait on an on-chip barrier that has not completed after this long is a
// bug (every wait here is for a copy already issued); the waiting thread
// records PF_DEV_WAIT_TIMEOUT and gives up instead of hanging the GPU.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy and to the
// other threads; follow with __syncthreads().
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

// Suspend hint for try_wait: the hardware parks a waiting thread until the
// phase completes or this many nanoseconds pass, so waits cost no issue slots.
constexpr uint32_t kSuspendHintNs = 200000;

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}

// Wait until the phase with the given parity has completed.  Bounded: after
// kWaitLimitNs it ORs PF_DEV_WAIT_TIMEOUT into *status and returns false.
// sleep_ns > 0 backs off between polls (for waits off the critical path).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int *status, uint32_t sleep_ns = 0) {
    if (mbar_try_wait(bar, parity)) return true;
    unsigned long long t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (sleep_ns) __nanosleep(sleep_ns);
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            atomicOr(status, PF_DEV_WAIT_TIMEOUT);
            return false;
        }
    }
}

// Warp-uniform bounded wait: lane 0 polls, the result is broadcast, and the
// __shfl_sync orders the other lanes' later shared-memory reads after it.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int *status, int lane,
                                          uint32_t sleep_ns = 0) {
    int ok = 1;
    if (lane == 0) ok = mbar_wait(bar, parity, status, sleep_ns) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Barrier among `count` warps built on an mbarrier initialised with that
// count: each warp's lane 0 arrives after the warp's writes, then waits
// (bounded) for the phase.  `phase` counts this barrier's uses.
__device__ __forceinline__ bool warps_sync(uint32_t bar, uint32_t &phase, int *status, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
    const bool ok = warp_wait(bar, phase & 1u, status, lane);
    ++phase;
    return ok;
}

// Atomic add with acquire-release semantics at GPU scope: publishes this
// thread's (and, by cumulativity, its CTA's synchronised) earlier writes and
// observes those published by earlier adders.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int *p, int v) {
    int old;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Wrapping increment at GPU scope, relaxed: returns the old value and stores
// (old >= limit) ? 0 : old + 1.  With fence_acq_rel_gpu before it, it
// releases the thread's earlier writes; with the fence after it, it acquires.
__device__ __forceinline__ unsigned atomic_inc_relaxed_gpu(unsigned *p, unsigned limit) {
    unsigned old;
    asm volatile("atom.relaxed.gpu.global.inc.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(limit) : "memory");
    return old;
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// One 64-bit word of a record shared between CTAs: the value's bits in the
// low half and the writing launch's epoch in the high half, stored and loaded
// as single 64-bit relaxed GPU-scope accesses (each indivisible), so a reader
// that finds the current epoch in a word holds that launch's value, with no
// fence on either side.
__device__ __forceinline__ void st_tagged(unsigned long long *p, float v, unsigned epoch) {
    const unsigned long long w = (unsigned long long)__float_as_uint(v) | ((unsigned long long)epoch << 32);
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}

__device__ __forceinline__ unsigned long long ld_tagged(const unsigned long long *p) {
    unsigned long long w;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}

__device__ __forceinline__ float tagged_value(unsigned long long w) { return __uint_as_float((unsigned)w); }
__device__ __forceinline__ unsigned tagged_epoch(unsigned long long w) { return (unsigned)(w >> 32); }

// 1-D bulk copy global -> shared, completing `bytes` on the mbarrier.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// 1-D bulk copy shared -> global (the async proxy reads shared memory),
// tracked by the issuing thread's bulk groups: commit with bulk_commit(),
// then bulk_wait_read<N>() before the shared bytes are written again and
// bulk_wait<N>() for the global writes to complete.  Both addresses 16-byte
// aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_store(void *dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// 3-D tiled TMA load of one box at coordinates (c0, c1, c2); c0 is the
// innermost (contiguous) coordinate and must be 16-byte aligned in bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
        : "memory");
}

// L2 prefetch of one tile through a tensor map: nothing is copied into the
// CTA and no barrier is involved.
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

// 4-D tiled TMA load into shared memory (same completion as tma_load_3d).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2, int c3,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap *map, int c0, int c1, int c2, int c3) {
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}

// Order this thread's earlier generic-proxy shared-memory writes before later
// async-proxy (TMA) writes to the same bytes.
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16-byte cp.async (L2 only) from global to shared memory.
__device__ __forceinline__ void cp_async16_cg(uint32_t smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem), "l"(gmem) : "memory");
}

// The mbarrier counts one arrival when every cp.async this thread issued so
// far has completed (.noinc: the arrival counts toward the barrier's expected
// count, which must include it).
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Four 8x8 b16 matrices from shared memory: lanes 8i .. 8i + 7 give the row
// addresses (16 bytes each) of matrix i; register i receives matrix i, lane l
// holding row l / 4, columns 2 (l % 4) and 2 (l % 4) + 1.  With .trans, lane l
// holds column l / 4, rows 2 (l % 4) and 2 (l % 4) + 1.
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

// Warp-wide D = A * B + D with A 16x16 (row), B 16x8 (column) fp16 and D
// 16x8 fp32.  Fragments (g = lane / 4, t = lane % 4): a0 (row g, k 2t..2t+1),
// a1 (row g + 8), a2 (row g, k + 8), a3 (row g + 8, k + 8); b0 (k 2t..2t+1,
// column g), b1 (k + 8); d0, d1 (row g, columns 2t, 2t + 1), d2, d3 (row g + 8).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Order this thread's earlier generic-proxy global writes before its later
// async-proxy (TMA) accesses of global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Hint: bring the 128-byte line holding p into L2.
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// L2 policy for data read exactly once per call: evict first.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 16-byte streaming global loads/stores (read once / written once).
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_stream(uint4 *p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// Eight fp16 values packed in a uint4 -> eight floats (exact).
__device__ __forceinline__ void half8_to_float(const uint4 &v, float (&f)[8]) {
    const __half2 *h = reinterpret_cast<const __half2 *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 x = __half22float2(h[i]);
        f[2 * i] = x.x;
        f[2 * i + 1] = x.y;
    }
}

}  // namespace pkv
