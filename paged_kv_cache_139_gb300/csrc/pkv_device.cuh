// Device-side helpers for the sm_103a kernels: the latched status word,
// programmatic dependent launch, mbarriers with bounded waits, 1-D bulk
// (TMA) copies into shared memory, and 16-bit <-> fp32 conversion.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace pkv {

// ---- per-device status word ---------------------------------------------

struct DeviceStatus {
    unsigned int flags;        // kFlag* bits; sticky until pkv_check clears them
    unsigned int have_first;   // 1 once first_bad/first_flag hold a value
    long long first_bad;       // the first offending value (slot, block id, ...)
    unsigned int first_flag;
    unsigned int pad;
};

enum : unsigned int {
    kFlagBadSlot = 1u,         // slot outside the pool
    kFlagBadBlock = 2u,        // block-table entry outside the pool
    kFlagBadPair = 4u,         // copy pair with a block id outside the pool
    kFlagTimeout = 8u,         // a bounded wait gave up
    kFlagBadContext = 16u,     // context length negative or beyond the table
    kFlagBadWorkspace = 32u,   // attention workspace not initialised
    kFlagSlotNotLast = 64u,    // fused decode write: slot is not position context_len - 1 of its table
};

__device__ __forceinline__ void latch(DeviceStatus *st, unsigned int flag, long long value) {
    atomicOr(&st->flags, flag);
    if (atomicCAS(&st->have_first, 0u, 1u) == 0u) {
        st->first_bad = value;
        st->first_flag = flag;
    }
}

// Head of an attention workspace (paged_attention_workspace_init zeroes the
// buffer and sets the magic): work-ticket counters of the persistent kernels.
// A kernel's last CTA leaves the counters at zero for the next call.
struct WsHeader {
    unsigned int next;        // next ticket
    unsigned int done;        // CTAs that have taken their last ticket
    unsigned int magic;       // kWsMagic once paged_attention_workspace_init has run
    unsigned int pad;
};
constexpr unsigned int kWsMagic = 0x31766b70u;
constexpr size_t kWsHeaderBytes = 256;

// Cycles a wait on an mbarrier may take before the kernel gives up (about
// 0.14 s at 1.9 GHz; a stage normally lands within microseconds).
constexpr long long kWaitLimitCycles = 1ll << 28;
// After one wait has given up: how long to wait for copies still in flight.
constexpr long long kDrainLimitCycles = 1ll << 25;

// True once any kernel has latched a timeout that pkv_check has not yet
// cleared; kernels then return at once instead of waiting again.
__device__ __forceinline__ bool timed_out(const DeviceStatus *st) {
    return (*reinterpret_cast<const volatile unsigned int *>(&st->flags) & kFlagTimeout) != 0;
}

// ---- programmatic dependent launch ---------------------------------------

// Blocks until the grids this one depends on have completed and their
// memory is visible; a no-op for a launch without the PDL attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next grid in the stream start launching.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- mbarrier --------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the phase with the given parity to complete; false if it has not
// within `limit` cycles.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, long long limit) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t it = 0; it < (1u << 28); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > limit) return false;
    }
    return false;
}

// ---- 1-D bulk copy (TMA, no tensor map) -----------------------------------

// bytes from global to this CTA's shared memory; completion is counted on
// `bar` as transaction bytes.  Both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void *smem_dst, const void *gmem_src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Same, with an L2 cache-policy hint (a createpolicy result).
__device__ __forceinline__ void bulk_g2s_hint(void *smem_dst, const void *gmem_src, uint32_t bytes,
                                              uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---- tiled (tensor-map) TMA copy ------------------------------------------

// A 3-D box at coordinates (x, y, z) (innermost first); x * element size a
// multiple of 16 bytes.
__device__ __forceinline__ void tma_load_3d(void *smem_dst, const void *tmap, int x, int y, int z, uint64_t *bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// A 4-D box of the tensor map at coordinates (x, y, z, w) (innermost first)
// into shared memory, completing on `bar`.  x * element size must be a
// multiple of 16 bytes.
__device__ __forceinline__ void tma_load_4d(void *smem_dst, const void *tmap, int x, int y, int z, int w,
                                            uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// ---- fp32 arithmetic on 16-bit inputs and on pairs ---------------------------

// a * b + c with 16-bit a, b (bit patterns) and fp32 c, d: the inputs widen
// exactly, so the result equals fmaf((float)a, (float)b, c).
template <typename T> __device__ __forceinline__ float fma_mixed(unsigned short a, unsigned short b, float c);
template <> __device__ __forceinline__ float fma_mixed<__half>(unsigned short a, unsigned short b, float c) {
    float d;
    asm("fma.rn.f32.f16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(c));
    return d;
}
template <> __device__ __forceinline__ float fma_mixed<__nv_bfloat16>(unsigned short a, unsigned short b, float c) {
    float d;
    asm("fma.rn.f32.bf16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(c));
    return d;
}

// Two fp32 lanes at once.
__device__ __forceinline__ unsigned long long pack2(float x, float y) {
    return (unsigned long long)__float_as_uint(x) | ((unsigned long long)__float_as_uint(y) << 32);
}
__device__ __forceinline__ float lo2(unsigned long long v) { return __uint_as_float((unsigned)v); }
__device__ __forceinline__ float hi2(unsigned long long v) { return __uint_as_float((unsigned)(v >> 32)); }
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// ---- warp-level tensor-core fragments ---------------------------------------

// Four 8x8 16-bit matrices; lane L gives the row address of matrix L / 8.
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void *row_addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(row_addr)));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], const void *row_addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(row_addr)));
}

template <typename T> struct Mma;

// D(16x8, f32) += A(16x16, row) * B(16x8, col), 16-bit inputs.
template <> struct Mma<__nv_bfloat16> {
    static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                     "{%8, %9}, {%0, %1, %2, %3};"
                     : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    // two fp32 -> one register of two bf16 (lo = x in the low half), round to nearest even
    static __device__ __forceinline__ uint32_t pack(float x, float y) {
        __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
        return *reinterpret_cast<uint32_t *>(&h);
    }
};

template <> struct Mma<__half> {
    static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                     "{%8, %9}, {%0, %1, %2, %3};"
                     : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    static __device__ __forceinline__ uint32_t pack(float x, float y) {
        __half2 h = __floats2half2_rn(x, y);
        return *reinterpret_cast<uint32_t *>(&h);
    }
};

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---- 16-bit element types --------------------------------------------------

template <typename T> struct F16Traits;

template <> struct F16Traits<__half> {
    // Eight halves (one 16-byte vector) to fp32.
    static __device__ __forceinline__ void to_f32(const uint4 &raw, float f[8]) {
        const __half2 *h = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            float2 v = __half22float2(h[i]);
            f[2 * i] = v.x;
            f[2 * i + 1] = v.y;
        }
    }
    static __device__ __forceinline__ __half from_f32(float x) { return __float2half_rn(x); }
};

template <> struct F16Traits<__nv_bfloat16> {
    static __device__ __forceinline__ void to_f32(const uint4 &raw, float f[8]) {
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            float2 v = __bfloat1622float2(h[i]);
            f[2 * i] = v.x;
            f[2 * i + 1] = v.y;
        }
    }
    static __device__ __forceinline__ __nv_bfloat16 from_f32(float x) { return __float2bfloat16_rn(x); }
};

}  // namespace pkv
