// Device-side helpers of the gx_gemm kernels: inline PTX for mbarriers, TMA (cp.async.bulk.tensor), L2 prefetch,
// programmatic dependent launch and the global timer. sm_103a only.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace sdmgx {
namespace dev {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- programmatic dependent launch ----------------------------------------------------------------------------------
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- mbarrier -------------------------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// true once the phase with the given parity has completed. A thread whose phase is not complete yet may be suspended
// (it issues nothing) until the phase completes or a time limit of the hardware's own passes. No suspend-time hint is
// given: on the large step a hint of 1 ms (or 32 us, or 1 us) woke the waiting warps later, 0.05-0.1 us a step.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: false if the phase did not complete within timeout_ns (the caller then reports and unwinds). Waiting
// threads sleep inside try_wait instead of spinning, so a waiting warp leaves its issue slots to the warps that
// compute (a test_wait spin in every wait made the large step 3% slower).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (static_cast<int64_t>(global_timer_ns() - t0) > timeout_ns) return false;
    }
}

// ---- TMA ------------------------------------------------------------------------------------------------------------
// 3-D tiled load of one box into this CTA's shared memory; completion is counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int32_t c0, int32_t c1, int32_t c2,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}
// 4-D tiled load of one box (used for a tensor viewed with a split row dimension)
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int32_t c0, int32_t c1, int32_t c2,
                                            int32_t c3, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
        "%5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}
// L2 prefetch of one box (no shared-memory destination, no completion)
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int32_t c0, int32_t c1, int32_t c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 1-D bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from global memory into this CTA's
// shared memory; completion is counted in bytes on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

// 1-D bulk copy of `bytes` from this CTA's shared memory to global memory, committed as its own bulk group; the caller
// waits for it with bulk_wait_all.
__device__ __forceinline__ void bulk_store(void *dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n\t"
                 "cp.async.bulk.commit_group;" ::"l"(reinterpret_cast<uint64_t>(dst)),
                 "r"(src), "r"(bytes)
                 : "memory");
}
// 3-D tiled store of one box from this CTA's shared memory to global memory, committed as its own bulk group.
// Elements of the box outside the tensor's extents are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, int32_t c0, int32_t c1, int32_t c2, uint32_t src) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];\n\t"
        "cp.async.bulk.commit_group;" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(c0), "r"(c1), "r"(c2), "r"(src)
        : "memory");
}
// waits until every bulk group this thread committed has completed (its writes performed)
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// waits until every bulk group this thread committed has read its shared-memory source (which may then be reused)
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// ---- flags between CTAs (global memory, GPU scope) ---------------------------------------------------------------------
__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(v) : "memory");
}
// orders this thread's view of global memory between the generic proxy (ordinary loads / stores) and the async proxy
// (bulk copies)
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Bounded wait until the flag holds `want`; false if that took longer than timeout_ns. Polls with relaxed loads;
// once it matches, an acquire fence orders the caller's later reads after the flag writer's release.
__device__ __forceinline__ bool wait_flag(const uint32_t *f, uint32_t want, int64_t timeout_ns) {
    uint64_t t0 = 0;
    bool timed = false;
    while (true) {
        uint32_t v;
        asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(reinterpret_cast<uint64_t>(f)) : "memory");
        if (v == want) {
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
            return true;
        }
        if (!timed) {
            t0 = global_timer_ns();
            timed = true;
        }
        __nanosleep(100);
        if (static_cast<int64_t>(global_timer_ns() - t0) > timeout_ns) return false;
    }
}

// ---- packed FP32 FMA ------------------------------------------------------------------------------------------------
// (c0, c1) = (fma(a0, b0, c0), fma(a1, b1, c1)): one fma.rn.f32x2 instruction, each lane an IEEE fused multiply-add
// rounded to nearest even with subnormals kept, i.e. bit for bit the same as two fmaf calls; half the issue slots.
__device__ __forceinline__ void fma2(float &c0, float &c1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%0, %1};\n\t"
        "fma.rn.f32x2 rc, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rc;\n\t}"
        : "+f"(c0), "+f"(c1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// ---- vector shared-memory loads and global stores --------------------------------------------------------------------
template <int V>
struct Vec;
template <>
struct Vec<1> {
    __device__ __forceinline__ static void load(const float *p, float *o) { o[0] = *p; }
    __device__ __forceinline__ static void store(float *p, const float *v) { *p = v[0]; }
};
template <>
struct Vec<2> {
    __device__ __forceinline__ static void load(const float *p, float *o) {
        const float2 t = *reinterpret_cast<const float2 *>(p);
        o[0] = t.x;
        o[1] = t.y;
    }
    __device__ __forceinline__ static void store(float *p, const float *v) {
        *reinterpret_cast<float2 *>(p) = make_float2(v[0], v[1]);
    }
};
template <>
struct Vec<4> {
    __device__ __forceinline__ static void load(const float *p, float *o) {
        const float4 t = *reinterpret_cast<const float4 *>(p);
        o[0] = t.x;
        o[1] = t.y;
        o[2] = t.z;
        o[3] = t.w;
    }
    __device__ __forceinline__ static void store(float *p, const float *v) {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};

}  // namespace dev
}  // namespace sdmgx
