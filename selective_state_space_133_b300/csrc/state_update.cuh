// Single-token recurrent state update (decode), sm_103a.
//
// One step of the selective SSM recurrence applied in place to a resident fp32
// state ("mamba->jamba", blog.csdn.net, §2.2: constant-time recurrent inference;
// "Mamba 论文精读", youngju.dev, §6: fixed-size state, O(1) per token):
//     dt = softplus(delta + bias)  (or delta + bias)
//     h  = exp(dt*A[d,:]) * h + dt*B[b,:]*u
//     y  = (C[b,:] . h + D[d]*u) * silu(z)
//
// The step is bound by HBM: the state (64 bytes per row) is read and written
// once, everything else is a few bytes per row or shared by a whole batch row
// (B, C) or channel (A). Four lanes share a row, each owning 4 consecutive
// states, so a warp moves 512 contiguous bytes of state per load and store;
// the partial C.h sums are added with two xor-shuffles inside the 4-lane group.
// All of a row's loads are issued before any arithmetic. The grid is
// (channels / 64, batch), so no thread divides to find its row.
#pragma once

#include "common.cuh"

namespace mscan {

struct UpdateArgs {
    float* state;
    const void* u;
    const void* delta;
    const void* z;      // may be null
    const void* B;
    const void* C;
    const float* A;
    const float* D;     // may be null
    const float* bias;  // may be null
    void* y;
    int batch, dim;
    int softplus;
};

constexpr int kUpdateThreads = 256;   // 64 channels per pass, 4 lanes each
constexpr int kUpdateRows = 1;         // rows per lane (2 doubles the registers and halves the warps: slower)
constexpr int kUpdateCh = kUpdateThreads / 4 * kUpdateRows;  // channels per block

// Four consecutive values (16-byte aligned for fp32, 8-byte for bf16) as fp32 pairs.
__device__ __forceinline__ void ldg4(const float* p, float2& lo, float2& hi) {
    const float4 q = *reinterpret_cast<const float4*>(p);
    lo = make_float2(q.x, q.y);
    hi = make_float2(q.z, q.w);
}
__device__ __forceinline__ void ldg4(const __nv_bfloat16* p, float2& lo, float2& hi) {
    const uint2 q = *reinterpret_cast<const uint2*>(p);
    lo = make_float2(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xffff0000u));
    hi = make_float2(__uint_as_float(q.y << 16), __uint_as_float(q.y & 0xffff0000u));
}

template <typename T>
__global__ void __launch_bounds__(kUpdateThreads) state_update_kernel(const UpdateArgs a) {
    const int b = blockIdx.y;
    const int q = threadIdx.x & 3;
    const T* u = static_cast<const T*>(a.u);
    const T* dl = static_cast<const T*>(a.delta);

    // B, C of this batch row: the same for every lane of the block
    float2 B01, B23, C01, C23;
    ldg4(static_cast<const T*>(a.B) + static_cast<size_t>(b) * kDState + 4 * q, B01, B23);
    ldg4(static_cast<const T*>(a.C) + static_cast<size_t>(b) * kDState + 4 * q, C01, C23);

    int d[kUpdateRows], dc[kUpdateRows];
    size_t row[kUpdateRows];
    float4 s4[kUpdateRows];
    float2 A01[kUpdateRows], A23[kUpdateRows];
    float uu[kUpdateRows], dv[kUpdateRows];
    // all loads first
#pragma unroll
    for (int r = 0; r < kUpdateRows; ++r) {
        d[r] = blockIdx.x * kUpdateCh + r * (kUpdateThreads / 4) + (threadIdx.x >> 2);
        dc[r] = d[r] < a.dim ? d[r] : a.dim - 1;  // padding lanes recompute the last channel, store nothing
        row[r] = static_cast<size_t>(b) * a.dim + dc[r];
        s4[r] = *reinterpret_cast<const float4*>(a.state + row[r] * kDState + 4 * q);
        ldg4(a.A + static_cast<size_t>(dc[r]) * kDState + 4 * q, A01[r], A23[r]);
        uu[r] = Io<T>::to_f(u[row[r]]);
        dv[r] = Io<T>::to_f(dl[row[r]]);
    }
#pragma unroll
    for (int r = 0; r < kUpdateRows; ++r) {
        float dt = dv[r] + (a.bias ? a.bias[dc[r]] : 0.f);
        if (a.softplus) dt = softplus_f(dt);
        const float2 dlt = make_float2(dt * kLog2e, dt * kLog2e);
        const float2 w = make_float2(dt * uu[r], dt * uu[r]);
        float2 h01 = make_float2(s4[r].x, s4[r].y), h23 = make_float2(s4[r].z, s4[r].w);
        const float2 x01 = __fmul2_rn(dlt, A01[r]), x23 = __fmul2_rn(dlt, A23[r]);
        h01 = __ffma2_rn(make_float2(ex2_approx(x01.x), ex2_approx(x01.y)), h01, __fmul2_rn(w, B01));
        h23 = __ffma2_rn(make_float2(ex2_approx(x23.x), ex2_approx(x23.y)), h23, __fmul2_rn(w, B23));
        const float2 acc = __ffma2_rn(C23, h23, __fmul2_rn(C01, h01));
        float yp = acc.x + acc.y;
        yp += __shfl_xor_sync(0xffffffffu, yp, 1);
        yp += __shfl_xor_sync(0xffffffffu, yp, 2);
        if (d[r] < a.dim) {
            *reinterpret_cast<float4*>(a.state + row[r] * kDState + 4 * q) = make_float4(h01.x, h01.y, h23.x, h23.y);
            if (q == 0) {
                float yy = a.D ? fmaf(a.D[d[r]], uu[r], yp) : yp;
                if (a.z) yy *= silu_f(Io<T>::to_f(static_cast<const T*>(a.z)[row[r]]));
                static_cast<T*>(a.y)[row[r]] = Io<T>::from_f(yy);
            }
        }
    }
}

}  // namespace mscan
