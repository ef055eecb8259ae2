// Device helpers shared by the scan and state-update kernels (sm_103a).
//
// Inline PTX for mbarrier / TMA (cp.async.bulk.tensor), bounded waits that
// report a timeout through a device error word instead of hanging, and the
// fp32 math used on the hot path.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mscan {


constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- math ----

// 2^x on the MUFU (relative error a few ulp; flushes denormal results to 0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// log1p(v) for v in [0, 1] as v * q(v); q is the degree-7 fit of log1p(v)/v on
// [0, 1] that fit_log1p.py derives (relative error of the fit <= 2.2e-7).
__device__ __forceinline__ float log1p_unit(float v) {
    float q = -0.008574675768613815f;
    q = fmaf(q, v, 0.044214192777872086f);
    q = fmaf(q, v, -0.10785368084907532f);
    q = fmaf(q, v, 0.17757023870944977f);
    q = fmaf(q, v, -0.2449961155653f);
    q = fmaf(q, v, 0.3327617645263672f);
    q = fmaf(q, v, -0.49997448921203613f);
    q = fmaf(q, v, 0.9999998211860657f);
    return v * q;
}

// q(v) of log1p_unit for two values at once, on the packed FP32 pipe.
__device__ __forceinline__ float2 log1p_unit_q2(float2 v) {
    float2 q = make_float2(-0.008574675768613815f, -0.008574675768613815f);
    q = __ffma2_rn(q, v, make_float2(0.044214192777872086f, 0.044214192777872086f));
    q = __ffma2_rn(q, v, make_float2(-0.10785368084907532f, -0.10785368084907532f));
    q = __ffma2_rn(q, v, make_float2(0.17757023870944977f, 0.17757023870944977f));
    q = __ffma2_rn(q, v, make_float2(-0.2449961155653f, -0.2449961155653f));
    q = __ffma2_rn(q, v, make_float2(0.3327617645263672f, 0.3327617645263672f));
    q = __ffma2_rn(q, v, make_float2(-0.49997448921203613f, -0.49997448921203613f));
    q = __ffma2_rn(q, v, make_float2(0.9999998211860657f, 0.9999998211860657f));
    return q;
}

// softplus(x) = log(1 + e^x) = max(x, 0) + log1p(e^{-|x|}); accurate in relative
// terms for small results (x << 0), where log2-based forms are not.
__device__ __forceinline__ float softplus_f(float x) {
    const float v = ex2_approx(-fabsf(x) * kLog2e);
    return fmaxf(x, 0.f) + log1p_unit(v);
}

// silu(z) = z * sigmoid(z) = z / (1 + e^{-z}); -> -0 for z << 0, z for z >> 0.
__device__ __forceinline__ float silu_f(float z) {
    return z * rcp_approx(1.f + ex2_approx(-z * kLog2e));
}

// --------------------------------------------------------- io types -------

template <typename T> struct Io;

template <> struct Io<float> {
    static constexpr int kBytes = 4;
    static constexpr CUtensorMapDataType kTmaType = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    __device__ __forceinline__ static float to_f(float x) { return x; }
    __device__ __forceinline__ static float from_f(float x) { return x; }
};

template <> struct Io<__nv_bfloat16> {
    static constexpr int kBytes = 2;
    static constexpr CUtensorMapDataType kTmaType = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    __device__ __forceinline__ static float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    __device__ __forceinline__ static __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

// --------------------------------------------------- mbarrier / TMA -------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before later
// async-proxy (TMA) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// Plain arrival (count 1) on `bar`, release semantics at CTA scope.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
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

// try_wait with a suspend-time hint: a thread whose phase has not completed may
// sleep (up to `ns` nanoseconds) until it does, instead of spinning on issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// 16-byte asynchronous copy global -> shared (both 16-byte aligned) that holds
// no register while in flight; cp_async_wait_all waits for this thread's.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for phase `parity` of `bar` to complete. Gives up after about one second
// of wall time (a TMA load normally lands in microseconds) and returns false.
// The common case, a phase that has already completed, costs one try_wait
// without a suspend hint (measured on B300: about 30 cycles, against about 75
// with the hint) and no timer read.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t start = global_timer_ns();
    for (uint32_t i = 1; i < (1u << 30); ++i) {
        if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
        if (global_timer_ns() - start > 1000000000ull) return false;
    }
    return false;
}

// Records `code` in the device error word (0 = fine, otherwise the mamba_status
// a kernel reported) unless an earlier error is already there. The word lives
// in the library's host file, which passes its address to the kernels and
// reads (and clears) it in mamba_check_device_error.
__device__ __forceinline__ void report_device_error(int* err, int code) { atomicCAS(err, 0, code); }

// ------------------------------------------------- checked-bounds build ----
// Built with -DMAMBA_DEBUG_BOUNDS, every global load and store that a kernel
// makes with ordinary instructions is first checked to lie inside the tensor
// it belongs to (its base pointer and its extent, from the call's sizes). An
// access outside is skipped (a load yields zero) and the kernel records
// MAMBA_ERR_DEVICE_BOUNDS in the device error word: nothing traps. TMA copies
// need no check, the tensor map encoded from the same sizes bounds them (and
// fills zeros outside). In the normal build the checks compile to nothing.
#ifdef MAMBA_DEBUG_BOUNDS
constexpr bool kCheckBounds = true;
#else
constexpr bool kCheckBounds = false;
#endif
constexpr int kErrDeviceBounds = -9;  // MAMBA_ERR_DEVICE_BOUNDS

// Whether the `count` values of type U at p lie inside the tensor that starts
// at `base` and holds `extent` values of type T (a null tensor holds none).
template <typename T, typename U>
__host__ __device__ __forceinline__ bool span_inside(const T* base, size_t extent, const U* p, long long count) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(base), q = reinterpret_cast<uintptr_t>(p);
    return base != nullptr && count >= 0 && q >= lo &&
           q + sizeof(U) * static_cast<size_t>(count) <= lo + sizeof(T) * extent;
}

// True when the access lies inside its tensor (span_inside); in the checked
// build an access outside it is recorded in *err and the caller skips it. In
// the normal build: true, and nothing is computed.
template <typename T, typename U>
__device__ __forceinline__ bool in_bounds(int* err, const T* base, size_t extent, const U* p, long long count = 1) {
    if constexpr (kCheckBounds) {
        if (!span_inside(base, extent, p, count)) {
            report_device_error(err, kErrDeviceBounds);
            return false;
        }
    }
    return true;
}

// 3-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

}  // namespace mscan
