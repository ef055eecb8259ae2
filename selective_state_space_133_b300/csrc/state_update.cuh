// Single-token recurrent state update (decode), sm_103a.
//
// One step of the selective SSM recurrence applied in place to a resident fp32
// state ("mamba->jamba", blog.csdn.net, §2.2: constant-time recurrent inference;
// "Mamba 论文精读", youngju.dev, §6: fixed-size state, O(1) per token):
//     dt = softplus(delta + bias)  (or delta + bias)
//     h  = exp(dt*A[d,:]) * h + dt*B[b,:]*u
//     y  = (C[b,:] . h + D[d]*u) * silu(z)
//
// The step is bound by HBM: the state (64 bytes per channel) is read and written
// once, everything else is a few bytes per channel. Four lanes share a channel,
// each owning 4 consecutive states (one 16-byte load and store), so a warp moves
// 512 contiguous bytes of state per instruction; the partial C.h sums are added
// with two xor-shuffles inside the 4-lane group.
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

template <typename T>
__device__ __forceinline__ void load4(const T* p, float (&v)[4]);

template <>
__device__ __forceinline__ void load4<float>(const float* p, float (&v)[4]) {
    const float4 q = *reinterpret_cast<const float4*>(p);
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
}

template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[4]) {
    const uint2 q = *reinterpret_cast<const uint2*>(p);
    v[0] = __uint_as_float(q.x << 16); v[1] = __uint_as_float(q.x & 0xffff0000u);
    v[2] = __uint_as_float(q.y << 16); v[3] = __uint_as_float(q.y & 0xffff0000u);
}

constexpr int kUpdateThreads = 256;  // 64 channels per block

template <typename T>
__global__ void __launch_bounds__(kUpdateThreads) state_update_kernel(const UpdateArgs a) {
    const long long rows = static_cast<long long>(a.batch) * a.dim;
    const long long row = static_cast<long long>(blockIdx.x) * (kUpdateThreads / 4) + (threadIdx.x >> 2);
    const int q = threadIdx.x & 3;
    const bool valid = row < rows;
    const long long rr = valid ? row : rows - 1;  // padding lanes recompute the last row, store nothing
    const int b = static_cast<int>(rr / a.dim);
    const int d = static_cast<int>(rr % a.dim);

    const T* u = static_cast<const T*>(a.u);
    const T* dl = static_cast<const T*>(a.delta);
    float dt = Io<T>::to_f(dl[rr]) + (a.bias ? a.bias[d] : 0.f);
    if (a.softplus) dt = softplus_f(dt);
    const float uu = Io<T>::to_f(u[rr]);

    float hs[4], av[4], bv[4], cv[4];
    float4* sp = reinterpret_cast<float4*>(a.state + rr * kDState + 4 * q);
    {
        const float4 s4 = *sp;
        hs[0] = s4.x; hs[1] = s4.y; hs[2] = s4.z; hs[3] = s4.w;
    }
    load4<float>(a.A + static_cast<size_t>(d) * kDState + 4 * q, av);
    load4<T>(static_cast<const T*>(a.B) + static_cast<size_t>(b) * kDState + 4 * q, bv);
    load4<T>(static_cast<const T*>(a.C) + static_cast<size_t>(b) * kDState + 4 * q, cv);

    const float w = dt * uu;
    float yp = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float e = ex2_approx(dt * (av[j] * kLog2e));
        hs[j] = fmaf(e, hs[j], w * bv[j]);
        yp = fmaf(cv[j], hs[j], yp);
    }
    yp += __shfl_xor_sync(0xffffffffu, yp, 1);
    yp += __shfl_xor_sync(0xffffffffu, yp, 2);

    if (valid) {
        *sp = make_float4(hs[0], hs[1], hs[2], hs[3]);
        if (q == 0) {
            float yy = a.D ? fmaf(a.D[d], uu, yp) : yp;
            if (a.z) yy *= silu_f(Io<T>::to_f(static_cast<const T*>(a.z)[rr]));
            static_cast<T*>(a.y)[rr] = Io<T>::from_f(yy);
        }
    }
}

}  // namespace mscan
