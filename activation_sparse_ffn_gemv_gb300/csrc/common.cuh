// common.cuh -- device helpers shared by the sffn kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sffn.h"

#define SFFN_DEV __device__ __forceinline__
#define SFFN_HOST_DEV __host__ __device__ __forceinline__

namespace sffn {

// ---------------------------------------------------------------------------
// Memory access
// ---------------------------------------------------------------------------

// 128-bit streaming load through the non-coherent path, not kept in L1:
// weights are read once per call and must not evict the staged activations.
SFFN_DEV uint4 ldg_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 32-bit streaming load (read once; no L1 allocation).
SFFN_DEV uint32_t ldg_stream_u32(const void *p) {
    uint32_t r;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

SFFN_DEV uint4 ldg_v4(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// ---------------------------------------------------------------------------
// Shared-memory barriers and bulk (1-D TMA) copies
// ---------------------------------------------------------------------------

SFFN_DEV uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

SFFN_DEV uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

SFFN_DEV void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// Make barrier initialisation visible to the async (TMA) proxy.
SFFN_DEV void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

SFFN_DEV void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
SFFN_DEV void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
SFFN_DEV bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for the barrier phase with the given parity to complete; gives up after
// limit_ns of wall time and returns false (the caller records a timeout).
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s
SFFN_DEV bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > limit_ns) return false;
    return true;
}

// L2 policy for data read exactly once (weights): evict first.
SFFN_DEV uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Order this thread's earlier generic-proxy shared-memory accesses (made
// visible to it, e.g. by a barrier) before its subsequent async-proxy (TMA)
// accesses to shared memory.
SFFN_DEV void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Per-thread asynchronous global -> shared copies (completion by
// cp_async_wait_all); addresses aligned to the copy size.
SFFN_DEV void cp_async_16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
SFFN_DEV void cp_async_4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
SFFN_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Bulk prefetch of [src, src + bytes) into L2 (16-byte aligned, multiple of 16).
SFFN_DEV void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Global -> shared bulk copy (16-byte aligned addresses, size a multiple of 16)
// completing `bytes` of transaction count on `bar`.
SFFN_DEV void bulk_load(void *dst_smem, const void *src, uint32_t bytes, uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch
// ---------------------------------------------------------------------------

// Block until the preceding kernel in the stream has completed and its memory
// is visible.  Every kernel calls this (in every CTA) before it touches
// workspace or outputs, so completion of any kernel implies completion of all
// earlier ones.
SFFN_DEV void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Barrier over `count` threads (whole warps) of the CTA on hardware barrier id
// (1..15; id 0 is __syncthreads).
SFFN_DEV void named_barrier_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Allow the next kernel in the stream to begin launching its CTAs.
SFFN_DEV void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Number formats
// ---------------------------------------------------------------------------

// bf16 pair packed in a 32-bit word -> two fp32 (exact widening).
SFFN_DEV float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
SFFN_DEV float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

SFFN_DEV float bf16_to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

// Round fp32 -> bf16, nearest-even.
SFFN_DEV uint16_t f32_to_bf16_bits(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&h);
}

// Correctly rounded bf16 sum of two bf16 pairs (one rounding of the exact sum):
// fma.rn.bf16x2 computes a * 1 + b exactly before its single rounding.
SFFN_DEV uint32_t bf16x2_add_rn(uint32_t a, uint32_t b) {
    uint32_t d;
    const uint32_t one = 0x3f803f80u;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(one), "r"(b));
    return d;
}

// ---------------------------------------------------------------------------
// Reductions
// ---------------------------------------------------------------------------

SFFN_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

SFFN_DEV float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

SFFN_DEV int warp_incl_scan(int v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// Block-wide exclusive scan of one int per thread (blockDim.x <= 1024, a
// multiple of 32).  `scratch` holds >= 33 ints.  Returns the exclusive prefix;
// *total receives the block total.  Contains __syncthreads().
SFFN_DEV int block_excl_scan(int v, int *scratch, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int incl = warp_incl_scan(v, lane);
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nw ? scratch[lane] : 0;
        int wi = warp_incl_scan(w, lane);
        if (lane < nw) scratch[lane] = wi - w;
        if (lane == 31) scratch[32] = wi;
    }
    __syncthreads();
    int r = scratch[warp] + incl - v;
    *total = scratch[32];
    __syncthreads();
    return r;
}

// Record a device-side contract violation (first error wins).
SFFN_DEV void record_error(int32_t *err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// ReLU, or SiLU(g) = g * sigmoid(g) with the accurate expf (the selection
// decisions are compared against an fp64 reference at 1e-6 relative).
SFFN_DEV float act_fn(int act, float g) {
    if (act == SFFN_ACT_RELU) return g > 0.f ? g : 0.f;
    return g / (1.f + expf(-g));
}

}  // namespace sffn
