// moe_device.cuh -- device helpers shared by the libmoe kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// ----------------------------------------------------------------- lanes

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// ------------------------------------------------- programmatic launches

// Every kernel of the layer starts with pdl_begin: it waits until the previous
// kernel in the stream has completed and its writes are visible, and all of
// the kernel's global loads and stores come after it, so stream order is
// kept.  Each kernel ends with pdl_end, after its last load, which lets the
// next kernel be scheduled while this one's last blocks finish: what overlaps
// is launch latency.  The trigger is not given earlier on purpose: a kernel
// two launches ahead could then become resident while this one still loads,
// and lines that this kernel leaves in a shared L1 could be stale by the time
// that kernel reads the addresses (rewritten in between by the kernel in the
// middle).  Both instructions are no-ops for a kernel launched without the
// programmatic-serialization attribute.
__device__ __forceinline__ void pdl_begin() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_end() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------- numerics

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// silu with the fast exponential and division: a few fp32 ulp from silu(),
// so a product rounded to bf16 afterwards differs from the correctly rounded
// one only where it lies within those ulps of a bf16 rounding boundary (one
// bf16 ulp then).  For g below about -88 the exponential overflows and the
// quotient is 0, as silu's limit is.
__device__ __forceinline__ float silu_fast(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
    __nv_bfloat16 b = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t*>(&b);
}

// ------------------------------------------- bf16 rows as scaled f16 rows

// The power-of-two shift sigma that moves a bf16 row's largest magnitude into
// [2^14, 2^15), from the largest |bf16| bit pattern mx of the row (0 for an
// all-zero row), clamped to [-113, 112].  bf16 has fewer significant bits
// than f16, so every element that stays in the f16 normal range converts
// exactly.
__device__ __forceinline__ int row_f16_shift(uint32_t mx) {
    if (mx == 0) return 0;
    // floor(log2) of a bf16 magnitude: its exponent field, or for a subnormal
    // the position of its top mantissa bit
    const int ef = (int)(mx >> 7);
    const int e = ef > 0 ? ef - 127 : (31 - __clz((int)mx)) - 133;
    return min(max(14 - e, -113), 112);
}

// The power-of-two shift that moves an fp32 magnitude with bit pattern mx
// (the largest |value| of a group) into [2^14, 2^15), clamped to [-120, 120]
// so that 2^shift and 2^-shift are normal fp32 values; 0 for mx == 0.
__device__ __forceinline__ int f32_f16_shift(uint32_t mx) {
    if (mx == 0) return 0;
    const int e = (mx >> 23) ? (int)(mx >> 23) - 127 : (31 - __clz((int)mx)) - 149;
    return min(max(14 - e, -120), 120);
}

// Two bf16 (low half first) times `up` (= 2^sigma) as an f16x2.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t w, float up) {
    const float lo = __uint_as_float(w << 16) * up;
    const float hi = __uint_as_float(w & 0xFFFF0000u) * up;
    const __half2 hv = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&hv);
}

// ------------------------------------------------ async copies, mbarriers

// Device error flag of this translation unit: set by a kernel whose bounded
// wait gave up (each kernel file has its own; moe_device_error() reads all).
static __device__ int g_device_error = 0;
// Set when a kernel meets an index outside its inputs' range (a tile's expert,
// a pair index, the tile count) and skips that work instead of reading or
// writing out of bounds.  Not read by the waits: every role skips the same
// work, so the pipelines stay in step.
static __device__ int g_index_error = 0;
__device__ __forceinline__ void flag_index_error() { atomicOr(&g_index_error, 1); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// One bounded try: the thread may sleep up to ~0.5 ms inside the instruction
// until the phase completes, instead of spinning on the issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(500000u)
        : "memory");
    return ok != 0;
}

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Bounded wait for the phase with the given parity.  Gives up (returns
// false) after kWaitLimitNs, or as soon as another CTA of the same kernel
// file has raised the device error flag, so one failure cannot stall a grid.
// The flag and the clock are checked only every 64 polls, keeping the poll
// itself a single shared-memory barrier test.
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 63) == 0) {
            if (*(volatile int*)&g_device_error) return false;
            if (global_ns() - t0 > limit_ns) {
                atomicExch(&g_device_error, 1);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    return mbar_wait_for(bar, parity, kWaitLimitNs);
}

// A bounded wait whose outcome is the same on every lane of the warp: if one
// lane gave up, all of them do.  A wait's result is otherwise taken per
// thread, and a lane that stopped while the others went on would leave them
// in a warp-collective instruction (a shuffle, tcgen05.ld / st, ldmatrix,
// mma.sync) that it never reaches.  All 32 lanes must call it.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity) {
    const bool ok = mbar_wait(bar, parity);
    return __all_sync(0xFFFFFFFFu, ok) != 0;
}

// `ok` reduced with AND over the `nthreads` threads (whole warps) that meet
// at named barrier `id`; every one of them must call it.  Threads that then
// synchronise at that barrier again act on the same outcome, so none is left
// waiting there for threads that stopped.
__device__ __forceinline__ bool all_at_barrier(bool ok, int id, int nthreads) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// ------------------------------------------------- CTA pairs (clusters of 2)

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster; orders the threads' earlier
// shared-memory writes (barrier inits among them) before the other CTAs'
// later accesses.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// Arrive on the mbarrier at the same shared-memory offset in CTA `rank` of
// the cluster, with the arrive's default semantics (release at CTA scope): no
// cluster-scope fence, which stalled every arriving warp for microseconds.
// The data the arrival announces is either ordered by the tensor-core fences
// around it (tensor-memory stores) or was itself announced to this thread by
// an mbarrier phase (TMA writes).
__device__ __forceinline__ void mbar_arrive_remote(uint64_t* bar, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(bar)), "r"(rank));
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}

// Prefetch one 2D box of a tensor map into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_2d(const void* tmap, int c0, int c1) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(tmap),
                 "r"(c0), "r"(c1)
                 : "memory");
}

// 2D tiled TMA load of one box into shared memory, completing on the mbarrier.
// c0 is the inner coordinate (bytes for a uint8 map; a multiple of 16).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int c0, int c1,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(tmap), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
            smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

// Bulk (TMA engine) copy global -> shared, completing `bytes` on the mbarrier.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t r[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// D = A * B with a zero accumulator (m16n8k16, f16 in, fp32 out).
__device__ __forceinline__ void mma_f16_16816_z(float d[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// D += A * B (m16n8k16, f16 in, fp32 accumulate).
__device__ __forceinline__ void mma_f16_16816_acc(float d[4], uint32_t a0, uint32_t a1,
                                                  uint32_t a2, uint32_t a3, uint32_t b0,
                                                  uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace moe
