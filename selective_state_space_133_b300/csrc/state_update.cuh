// Single-token recurrent state update (decode), sm_103a.
//
// One step of the selective SSM recurrence applied in place to a resident fp32
// state ("mamba->jamba", blog.csdn.net, §2.2: constant-time recurrent inference;
// "Mamba 论文精读", youngju.dev, §6: fixed-size state, O(1) per token):
//     dt = softplus(delta + bias)  (or delta + bias)
//     h  = exp(dt*A[d,:]) * h + dt*B[b,:]*u
//     y  = (C[b,:] . h + D[d]*u) * silu(z)
//
// With the ZOH instantiation the input gain dt*B is the exact zero-order-hold
// B_bar = (exp(dt*A) - 1) / A * B ("Mamba 论文精读" §2.2), taken with expm1.
//
// The step is bound by HBM: the state (4N bytes per row) is read and written
// once, everything else is a few bytes per row or shared by a whole batch row
// (B, C) or channel (A). N/4 lanes share a row, each owning 4 consecutive
// states, so a warp moves 512 contiguous bytes of state per load and store;
// the partial C.h sums are added with xor-shuffles inside the lane group.
// A thread takes the same channel in kR consecutive batch rows: A, D and the
// bias of the channel are loaded once for all of them, and their states
// (16 bytes each) are copied into shared memory with asynchronous copies
// before any arithmetic, so that the copies in flight hold no registers and a
// full SM of threads keeps enough bytes in flight to cover the memory latency
// at full bandwidth. The block's B and C rows are staged in shared memory as
// fp32. The grid is (channels / channels per block, batch rows / kR).
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
    int* err;           // device error word
    int batch, dim;
    int softplus;
};

constexpr int kUpdateThreads = 128;

// Lanes per row and rows per block of the state update for state size NS.
template <int NS>
struct UpdateGeo {
    static_assert(NS == 8 || NS == 16 || NS == 32 || NS == 64, "state sizes 8, 16, 32 and 64 are compiled");
    // states per lane: 4 (measured on B300 at 256 x 5120, N = 16: 30.7 us,
    // against 42.9 us with 8 and 47.1 us with 16, which take fewer lanes a row)
    static constexpr int kV = 4;
    static constexpr int kQ = NS / kV;                      // lanes per row
    static constexpr int kCh = kUpdateThreads / kQ;         // channels per block
    static constexpr int kR = 4;                            // batch rows per thread (and per block)
};

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

template <typename T, int NS, bool ZOH>
__global__ void __launch_bounds__(kUpdateThreads) state_update_kernel(const UpdateArgs a) {
    using G = UpdateGeo<NS>;
    constexpr int kQ = G::kQ, kR = G::kR, kV = G::kV, kV4 = kV / 4;
    __shared__ float4 stage[kR][kV4][kUpdateThreads];  // the state of each of this thread's rows
    __shared__ alignas(16) float bc[kR][2][NS];         // B and C of the block's batch rows
    const int tid = threadIdx.x;
    const int q = tid % kQ;
    const int b0 = blockIdx.y * kR;
    const int d = blockIdx.x * G::kCh + tid / kQ;
    const int dc = d < a.dim ? d : a.dim - 1;  // padding lanes recompute the last channel, store nothing
    const T* u = static_cast<const T*>(a.u);
    const T* dl = static_cast<const T*>(a.delta);
    const T* zg = static_cast<const T*>(a.z);
    const size_t nrows = static_cast<size_t>(a.batch) * a.dim;  // extents, for the checked-bounds build

    // every load first: the states (asynchronous), then the rest
#pragma unroll
    for (int r = 0; r < kR; ++r) {
        const float* sp = a.state + (static_cast<size_t>(b0 + r) * a.dim + dc) * NS + kV * q;
#pragma unroll
        for (int v = 0; v < kV4; ++v)
            if (b0 + r < a.batch && in_bounds(a.err, a.state, nrows * NS, sp + 4 * v, 4))
                cp_async16(&stage[r][v][tid], sp + 4 * v);
    }
    for (int i = tid; i < kR * 2 * NS; i += kUpdateThreads) {
        const int r = i / (2 * NS), which = (i / NS) % 2, n = i % NS;
        const T* src = static_cast<const T*>(which ? a.C : a.B) + static_cast<size_t>(b0 + r) * NS + n;
        bc[r][which][n] = b0 + r < a.batch && in_bounds(a.err, static_cast<const T*>(which ? a.C : a.B),
                                                        static_cast<size_t>(a.batch) * NS, src)
            ? Io<T>::to_f(*src) : 0.f;
    }
    float2 Av[2 * kV4];  // this lane's kV values of A as pairs
#pragma unroll
    for (int v = 0; v < kV4; ++v) {
        Av[2 * v] = Av[2 * v + 1] = make_float2(-1.f, -1.f);
        const float* Ap = a.A + static_cast<size_t>(dc) * NS + kV * q + 4 * v;
        if (in_bounds(a.err, a.A, static_cast<size_t>(a.dim) * NS, Ap, 4)) ldg4(Ap, Av[2 * v], Av[2 * v + 1]);
    }
    const float bias = a.bias && in_bounds(a.err, a.bias, a.dim, a.bias + dc) ? a.bias[dc] : 0.f;
    const float Dd = a.D && q == 0 && in_bounds(a.err, a.D, a.dim, a.D + dc) ? a.D[dc] : 0.f;
    float uu[kR], dv[kR], zz[kR];
#pragma unroll
    for (int r = 0; r < kR; ++r) {
        const size_t row = static_cast<size_t>(b0 + r < a.batch ? b0 + r : a.batch - 1) * a.dim + dc;
        uu[r] = in_bounds(a.err, u, nrows, u + row) ? Io<T>::to_f(u[row]) : 0.f;
        dv[r] = in_bounds(a.err, dl, nrows, dl + row) ? Io<T>::to_f(dl[row]) : 0.f;
        zz[r] = zg && q == 0 && in_bounds(a.err, zg, nrows, zg + row) ? Io<T>::to_f(zg[row]) : 0.f;
    }
    cp_async_wait_all();
    __syncthreads();  // bc, written by other threads

#pragma unroll
    for (int r = 0; r < kR; ++r) {
        if (b0 + r >= a.batch) break;
        float dt = dv[r] + bias;
        if (a.softplus) dt = softplus_f(dt);
        const float2 dlt = make_float2(dt * kLog2e, dt * kLog2e);
        const float2 w = make_float2(dt * uu[r], dt * uu[r]);
        float4 hn[kV4];
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int v = 0; v < kV4; ++v) {
            const float4 s4 = stage[r][v][tid];
            const float4 b4 = *reinterpret_cast<const float4*>(&bc[r][0][kV * q + 4 * v]);
            const float4 c4 = *reinterpret_cast<const float4*>(&bc[r][1][kV * q + 4 * v]);
            const float2 A01 = Av[2 * v], A23 = Av[2 * v + 1];
            const float2 B01 = make_float2(b4.x, b4.y), B23 = make_float2(b4.z, b4.w);
            float2 h01 = make_float2(s4.x, s4.y), h23 = make_float2(s4.z, s4.w);
            const float2 x01 = __fmul2_rn(dlt, A01), x23 = __fmul2_rn(dlt, A23);
            float2 g01, g23;  // input terms
            if (ZOH) {
                // (exp(dt a) - 1) / a per state, dt where dt*a = 0 (its limit)
                const float av[4] = {A01.x, A01.y, A23.x, A23.y};
                float gv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float x = dt * av[i];
                    gv[i] = (x == 0.f ? dt : expm1f(x) / av[i]) * uu[r];
                }
                g01 = __fmul2_rn(make_float2(gv[0], gv[1]), B01);
                g23 = __fmul2_rn(make_float2(gv[2], gv[3]), B23);
            } else {
                g01 = __fmul2_rn(w, B01);
                g23 = __fmul2_rn(w, B23);
            }
            h01 = __ffma2_rn(make_float2(ex2_approx(x01.x), ex2_approx(x01.y)), h01, g01);
            h23 = __ffma2_rn(make_float2(ex2_approx(x23.x), ex2_approx(x23.y)), h23, g23);
            acc = __ffma2_rn(make_float2(c4.z, c4.w), h23, __ffma2_rn(make_float2(c4.x, c4.y), h01, acc));
            hn[v] = make_float4(h01.x, h01.y, h23.x, h23.y);
        }
        float yp = acc.x + acc.y;
#pragma unroll
        for (int o = 1; o < kQ; o <<= 1) yp += __shfl_xor_sync(0xffffffffu, yp, o);
        if (d < a.dim) {
            const size_t row = static_cast<size_t>(b0 + r) * a.dim + d;
            float* sp = a.state + row * NS + kV * q;
#pragma unroll
            for (int v = 0; v < kV4; ++v)
                if (in_bounds(a.err, a.state, nrows * NS, sp + 4 * v, 4))
                    *reinterpret_cast<float4*>(sp + 4 * v) = hn[v];
            if (q == 0) {
                float yy = a.D ? fmaf(Dd, uu[r], yp) : yp;
                if (zg) yy *= silu_f(zz[r]);
                T* yg = static_cast<T*>(a.y);
                if (in_bounds(a.err, yg, nrows, yg + row)) yg[row] = Io<T>::from_f(yy);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Single-token step of the SSD (Mamba-2) form: per batch row b and head h the
// state is a (headdim x N) matrix with one decay per step ("Mamba 论文精读"
// §4.1: h_t = A_t h_{t-1} + B_t x_t, y_t = C_t h_t; §5.2 the multi-head layer):
//     dt = softplus(delta[b,h] + bias[h])   (or delta + bias)
//     S[p,:] = exp(dt A[h]) S[p,:] + dt x[b,h*P+p] B[b,:]
//     y[b,h*P+p] = S[p,:] . C[b,:] + D[h] x[b,h*P+p]
// Bound by HBM like the scan's state update: each state row (4N bytes) is
// read and written once. N/4 lanes share a row, 4 states each, and add their
// partial C.S with xor-shuffles (8 states a lane at N = 256, so that a row
// fits one warp). A thread takes kR rows of the same batch row,
// which share B and C (loaded once), and copies their states into shared
// memory with asynchronous copies before any arithmetic.

struct SsdUpdateArgs {
    float* state;        // (batch, nheads, headdim, N) fp32, in place
    const void* x;       // (batch, nheads * headdim)
    const void* delta;   // (batch, nheads)
    const void* B;       // (batch, N)
    const void* C;       // (batch, N)
    const float* A;      // (nheads)
    const float* D;      // (nheads) or null
    const float* bias;   // (nheads) or null
    void* y;             // (batch, nheads * headdim)
    int* err;            // device error word
    int batch, nheads, headdim;
    int softplus;
};

template <int NS>
struct SsdUpdateGeo {
    static_assert(NS == 64 || NS == 128 || NS == 256, "state sizes 64, 128 and 256 are compiled");
    static constexpr int kV = NS == 256 ? 8 : 4;         // states per lane (a row fits one warp)
    static constexpr int kQ = NS / kV;                   // lanes per row (a power of two up to 32)
    static constexpr int kPass = kUpdateThreads / kQ;    // rows the block's threads cover at once
    static constexpr int kR = 4;                         // rows per thread
    static constexpr int kRows = kPass * kR;             // rows per block
};

template <typename T, int NS>
__global__ void __launch_bounds__(kUpdateThreads) ssd_update_kernel(const SsdUpdateArgs a) {
    using G = SsdUpdateGeo<NS>;
    constexpr int kQ = G::kQ, kR = G::kR, kV4 = G::kV / 4;
    __shared__ float4 stage[kR][kV4][kUpdateThreads];  // the state of each of this thread's rows
    const int tid = threadIdx.x;
    const int b = blockIdx.y;
    const int q = tid % kQ;
    const int dim = a.nheads * a.headdim;
    const size_t nrows = static_cast<size_t>(a.batch) * dim;  // extents, for the checked-bounds build
    const T* xg = static_cast<const T*>(a.x);
    const T* dg = static_cast<const T*>(a.delta);
    // every load first: the states (asynchronous), then the rest
    int dcs[kR];
#pragma unroll
    for (int r = 0; r < kR; ++r) {
        const int d = blockIdx.x * G::kRows + r * G::kPass + tid / kQ;
        dcs[r] = d < dim ? d : dim - 1;  // padding lanes recompute the last row, store nothing
        const float* sp = a.state + (static_cast<size_t>(b) * dim + dcs[r]) * NS + G::kV * q;
#pragma unroll
        for (int v = 0; v < kV4; ++v) {
            if (in_bounds(a.err, a.state, nrows * NS, sp + 4 * v, 4)) cp_async16(&stage[r][v][tid], sp + 4 * v);
            else stage[r][v][tid] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    float2 Bv[2 * kV4], Cv[2 * kV4];  // this lane's kV values of B and C as pairs
#pragma unroll
    for (int v = 0; v < kV4; ++v) {
        Bv[2 * v] = Bv[2 * v + 1] = Cv[2 * v] = Cv[2 * v + 1] = make_float2(0.f, 0.f);
        const T* Bp = static_cast<const T*>(a.B) + static_cast<size_t>(b) * NS + G::kV * q + 4 * v;
        const T* Cp = static_cast<const T*>(a.C) + static_cast<size_t>(b) * NS + G::kV * q + 4 * v;
        if (in_bounds(a.err, static_cast<const T*>(a.B), static_cast<size_t>(a.batch) * NS, Bp, 4))
            ldg4(Bp, Bv[2 * v], Bv[2 * v + 1]);
        if (in_bounds(a.err, static_cast<const T*>(a.C), static_cast<size_t>(a.batch) * NS, Cp, 4))
            ldg4(Cp, Cv[2 * v], Cv[2 * v + 1]);
    }
    float xv[kR], dt[kR], Ah[kR], Dh[kR];
#pragma unroll
    for (int r = 0; r < kR; ++r) {
        const int h = dcs[r] / a.headdim;
        const size_t row = static_cast<size_t>(b) * dim + dcs[r];
        const size_t hrow = static_cast<size_t>(b) * a.nheads + h;
        xv[r] = in_bounds(a.err, xg, nrows, xg + row) ? Io<T>::to_f(xg[row]) : 0.f;
        dt[r] = (in_bounds(a.err, dg, static_cast<size_t>(a.batch) * a.nheads, dg + hrow) ? Io<T>::to_f(dg[hrow])
                                                                                           : 0.f) +
                (a.bias && in_bounds(a.err, a.bias, a.nheads, a.bias + h) ? a.bias[h] : 0.f);
        Ah[r] = in_bounds(a.err, a.A, a.nheads, a.A + h) ? a.A[h] : -1.f;
        Dh[r] = a.D && q == 0 && in_bounds(a.err, a.D, a.nheads, a.D + h) ? a.D[h] : 0.f;
    }
    cp_async_wait_all();  // this thread's own copies: no other thread reads them

#pragma unroll
    for (int r = 0; r < kR; ++r) {
        float dtr = dt[r];
        if (a.softplus) dtr = softplus_f(dtr);
        const float decay = ex2_approx(dtr * Ah[r] * kLog2e);
        const float2 ea = make_float2(decay, decay);
        const float2 w = make_float2(dtr * xv[r], dtr * xv[r]);
        float4 hn[kV4];
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int v = 0; v < kV4; ++v) {
            const float4 s4 = stage[r][v][tid];
            const float2 h01 = __ffma2_rn(ea, make_float2(s4.x, s4.y), __fmul2_rn(w, Bv[2 * v]));
            const float2 h23 = __ffma2_rn(ea, make_float2(s4.z, s4.w), __fmul2_rn(w, Bv[2 * v + 1]));
            acc = __ffma2_rn(Cv[2 * v + 1], h23, __ffma2_rn(Cv[2 * v], h01, acc));
            hn[v] = make_float4(h01.x, h01.y, h23.x, h23.y);
        }
        float yp = acc.x + acc.y;
#pragma unroll
        for (int o = 1; o < kQ; o <<= 1) yp += __shfl_xor_sync(0xffffffffu, yp, o);
        const int d = blockIdx.x * G::kRows + r * G::kPass + tid / kQ;
        if (d < dim) {
            const size_t row = static_cast<size_t>(b) * dim + d;
            float* sp = a.state + row * NS + G::kV * q;
#pragma unroll
            for (int v = 0; v < kV4; ++v)
                if (in_bounds(a.err, a.state, nrows * NS, sp + 4 * v, 4))
                    *reinterpret_cast<float4*>(sp + 4 * v) = hn[v];
            if (q == 0) {
                const float yy = a.D ? fmaf(Dh[r], xv[r], yp) : yp;
                T* yg = static_cast<T*>(a.y);
                if (in_bounds(a.err, yg, nrows, yg + row)) yg[row] = Io<T>::from_f(yy);
            }
        }
    }
}

}  // namespace mscan
