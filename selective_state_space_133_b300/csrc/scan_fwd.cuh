// Selective-scan forward kernel (prefill), sm_103a.
//
// Computes, for every (batch b, channel d), the recurrence of the selective SSM
// ("Mamba 论文精读", youngju.dev, §2.2 and §3.3; gate from §3.4; D skip term from
// "Mamba的基础知识", weblog-19d, 状态空间模型 section):
//     dt = softplus(delta + bias)            (or delta + bias)
//     h  = exp(dt*A[d,:]) * h + dt*B[b,:,l]*u   (h = 0 before l = 0)
//     y  = (C[b,:,l] . h + D[d]*u) * silu(z)
// with the state kept in registers for the whole sequence and nothing but y
// (and the optional final state) written back ("mamba->jamba", blog.csdn.net,
// §2.3: discretise, scan and contract on chip; HBM traffic O(BLD + BLN)).
//
// Design (B300-first, not the pages' kernel):
//  * The path is bound by the SM's issue slots, the FP32 pipe and the MUFU exp
//    (one exp per (b,l,d,n) element), not by HBM. Each thread therefore walks
//    the WHOLE sequence for its rows sequentially: no warp-level scan, no carry
//    fix-ups; the recurrence costs 4 FP32 lane-ops + 1 exp per element, issued
//    as packed FFMA2/FMUL2 on pairs of states.
//  * CTA = one warp = ROWS channels of one batch, two lanes per channel, each
//    lane holding 8 of the 16 states. One-warp CTAs keep the grid balanced over
//    148 SMs (7 resident per SM).
//  * The sequence is cut into TL-step chunks. Lane 0 issues 3-D TMA loads of a
//    chunk's u/delta/z (ROWS x TL) and B/C (16 x TL) tiles into a STAGES-deep
//    ring (one mbarrier per slot, bounded waits).
//  * Per chunk there are three phases: the pre-pass (dt and dt*u once per
//    (row, step); B/C transposed into per-step fp32 pairs), the recurrence, and
//    the epilogue (two half-state partial sums + D*u, times silu(z), stored as
//    16-byte vectors). They are software-pipelined: iteration c runs the
//    recurrence of chunk c, the pre-pass of chunk c+1 and the epilogue of chunk
//    c-1 as one straight-line block, so the three independent instruction
//    streams hide each other's latencies inside a single warp.
//  * The last chunk's recurrence runs only its valid steps; padding steps are
//    never applied, so the final state needs no masking.
#pragma once

#include <type_traits>

#include "common.cuh"

namespace mscan {

struct ScanArgs {
    const void* u;
    const void* delta;
    const void* z;       // may be null
    const void* B;
    const void* C;
    const float* A;
    const float* D;      // may be null
    const float* bias;   // may be null
    void* y;
    float* final_state;  // may be null
    int batch, dim, seqlen;
    int softplus;
    int use_tma;         // 1: TMA tiles; 0: plain loads (row pitch not 16-byte aligned)
};

template <typename T, int ROWS, int TL>
struct RawTiles {
    alignas(128) T u[ROWS][TL];
    alignas(128) T dl[ROWS][TL];
    alignas(128) T z[ROWS][TL];
    alignas(128) T B[kDState][TL];
    alignas(128) T C[kDState][TL];
};

template <typename T, int ROWS, int TL, int STAGES>
struct ScanSmem {
    RawTiles<T, ROWS, TL> raw[STAGES];
    alignas(16) float2 W[2][ROWS][TL + 1];            // {dt, dt*u}; odd pitch: conflict-free scan reads
    alignas(16) float4 BC[2][TL][kDState / 2 + 1];    // per step {B_2k, B_2k+1, C_2k, C_2k+1}; +1 pad
    alignas(16) float Y[2][2][ROWS][TL + 4];          // partial C.h per half of the states
    alignas(8) uint64_t full[STAGES];
};

// Plain (non-TMA) fill of one raw slot, zero outside the tensor. Used when the
// row pitch seqlen*sizeof(T) is not a multiple of 16 bytes, which TMA cannot map.
template <typename T, int ROWS, int TL>
__device__ __forceinline__ void fill_raw_plain(RawTiles<T, ROWS, TL>& R, const ScanArgs& a, int b, int d0, int l0,
                                               int lane) {
    const T* u = static_cast<const T*>(a.u);
    const T* dl = static_cast<const T*>(a.delta);
    const T* z = static_cast<const T*>(a.z);
    const T* Bm = static_cast<const T*>(a.B);
    const T* Cm = static_cast<const T*>(a.C);
    const T zero = Io<T>::from_f(0.f);
    for (int i = lane; i < ROWS * TL; i += 32) {
        const int r = i / TL, t = i % TL;
        const int d = d0 + r, l = l0 + t;
        const bool ok = d < a.dim && l < a.seqlen;
        const size_t off = (static_cast<size_t>(b) * a.dim + d) * a.seqlen + l;
        R.u[r][t] = ok ? u[off] : zero;
        R.dl[r][t] = ok ? dl[off] : zero;
        if (z) R.z[r][t] = ok ? z[off] : zero;
    }
    for (int i = lane; i < kDState * TL; i += 32) {
        const int n = i / TL, t = i % TL;
        const int l = l0 + t;
        const bool ok = l < a.seqlen;
        const size_t off = (static_cast<size_t>(b) * kDState + n) * a.seqlen + l;
        R.B[n][t] = ok ? Bm[off] : zero;
        R.C[n][t] = ok ? Cm[off] : zero;
    }
}

// Load 8 consecutive values (16-byte aligned in shared memory) as fp32.
__device__ __forceinline__ void lds8_f32(const float* p, float (&v)[8]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0];
    const float4 b = reinterpret_cast<const float4*>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void lds8_f32(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 q = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        v[2 * j + 0] = __uint_as_float(w[j] << 16);
        v[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
}

// Store 8 consecutive outputs (16-byte aligned in global memory).
__device__ __forceinline__ void stg8(float* p, const float (&v)[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void stg8(__nv_bfloat16* p, const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __nv_bfloat162 q = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
        w[j] = *reinterpret_cast<const uint32_t*>(&q);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Per-lane state and the three phases of one CTA.
template <typename T, int ROWS, int TL, int STAGES, bool SOFTPLUS, bool HAS_Z>
struct ScanCta {
    using Smem = ScanSmem<T, ROWS, TL, STAGES>;
    using Raw = RawTiles<T, ROWS, TL>;
    static_assert(ROWS * 2 == 32, "one warp: two lanes per row");
    static_assert(TL == 16, "pre-pass/epilogue: 8 steps per lane; transpose: one step per lane pair");

    Smem& S;
    const ScanArgs& a;
    int lane, r, g, b, d0, d;
    float bias, Dd;
    float2 a2[4];  // A[d, 8g .. 8g+7] * log2(e), as pairs
    float2 h[4];   // this lane's 8 states

    __device__ __forceinline__ ScanCta(Smem& S_, const ScanArgs& a_) : S(S_), a(a_) {}

    // dt and dt*u for steps 8g..8g+7 of row r; B/C of step lane/2 transposed.
    __device__ __forceinline__ void prepass(const Raw& R, int buf) {
        const int t0 = 8 * g;
        float dv[8], uv[8];
        lds8_f32(&R.dl[r][t0], dv);
        lds8_f32(&R.u[r][t0], uv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float dt = dv[i] + bias;
            if (SOFTPLUS) dt = softplus_f(dt);
            S.W[buf][r][t0 + i] = make_float2(dt, dt * uv[i]);
        }
        const int t = lane >> 1;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int q = 2 * j + (lane & 1);
            S.BC[buf][t][q] = make_float4(Io<T>::to_f(R.B[2 * q][t]), Io<T>::to_f(R.B[2 * q + 1][t]),
                                          Io<T>::to_f(R.C[2 * q][t]), Io<T>::to_f(R.C[2 * q + 1][t]));
        }
    }

    // One step of the recurrence for this lane's 8 states; returns its part of C.h.
    // The C.h sum runs as two independent FFMA2 chains (states 0-3, 4-7).
    __device__ __forceinline__ float step(int buf, int t) {
        const float2 dw = S.W[buf][r][t];
        const float2 dd = make_float2(dw.x, dw.x);
        const float2 ww = make_float2(dw.y, dw.y);
        float2 yp[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 bc = S.BC[buf][t][4 * g + q];
            const float2 x = __fmul2_rn(dd, a2[q]);
            float2 e;
            e.x = ex2_approx(x.x);
            e.y = ex2_approx(x.y);
            const float2 pb = __fmul2_rn(ww, make_float2(bc.x, bc.y));
            h[q] = __ffma2_rn(e, h[q], pb);
            yp[q >> 1] = __ffma2_rn(make_float2(bc.z, bc.w), h[q], yp[q >> 1]);
        }
        const float2 ys = __fadd2_rn(yp[0], yp[1]);
        return ys.x + ys.y;
    }

    // All TL steps of a chunk (fully unrolled), partial sums to Y[buf][g][r][:].
    __device__ __forceinline__ void scan_full(int buf) {
#pragma unroll
        for (int t = 0; t < TL; t += 4) {
            float yv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) yv[j] = step(buf, t + j);
            *reinterpret_cast<float4*>(&S.Y[buf][g][r][t]) = make_float4(yv[0], yv[1], yv[2], yv[3]);
        }
    }

    // The first `steps` steps of a chunk (the sequence's last, partial chunk).
    __device__ __forceinline__ void scan_partial(int buf, int steps) {
#pragma unroll 1
        for (int t = 0; t < steps; ++t) S.Y[buf][g][r][t] = step(buf, t);
    }

    // y = (Y0 + Y1 + D*u) * silu(z) for steps 8g..8g+7 of row r, stored to global.
    // FULL: the chunk lies entirely inside the sequence.
    template <bool FULL>
    __device__ __forceinline__ void epilogue(const Raw& R, int buf, int l0) {
        const int t0 = 8 * g;
        float uv[8], zv[8], y0[8], y1[8], out[8];
        lds8_f32(&R.u[r][t0], uv);
        if (HAS_Z) lds8_f32(&R.z[r][t0], zv);
        lds8_f32(&S.Y[buf][0][r][t0], y0);
        lds8_f32(&S.Y[buf][1][r][t0], y1);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float yy = fmaf(Dd, uv[i], y0[i] + y1[i]);
            if (HAS_Z) yy *= silu_f(zv[i]);
            out[i] = yy;
        }
        if (d < a.dim) {
            T* yrow = static_cast<T*>(a.y) + (static_cast<size_t>(b) * a.dim + d) * a.seqlen;
            const int lb = l0 + t0;
            if (a.use_tma && (FULL || lb + 8 <= a.seqlen)) {
                stg8(yrow + lb, out);  // row pitch is a multiple of 16 bytes on this path
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (FULL || lb + i < a.seqlen) yrow[lb + i] = Io<T>::from_f(out[i]);
            }
        }
    }
};

template <typename T, int ROWS, int TL, int STAGES, bool SOFTPLUS, bool HAS_Z>
__global__ void __launch_bounds__(32)
scan_fwd_kernel(const ScanArgs a, const __grid_constant__ CUtensorMap tm_u,
                const __grid_constant__ CUtensorMap tm_dl, const __grid_constant__ CUtensorMap tm_z,
                const __grid_constant__ CUtensorMap tm_B, const __grid_constant__ CUtensorMap tm_C) {
    using Cta = ScanCta<T, ROWS, TL, STAGES, SOFTPLUS, HAS_Z>;
    __shared__ typename Cta::Smem S;
    Cta k(S, a);
    k.lane = threadIdx.x;
    k.b = blockIdx.y;
    k.d0 = blockIdx.x * ROWS;
    k.r = k.lane >> 1;
    k.g = k.lane & 1;
    k.d = k.d0 + k.r;
    const int dc = k.d < a.dim ? k.d : a.dim - 1;  // clamped for parameter loads of padding rows
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 av =
            *reinterpret_cast<const float2*>(a.A + static_cast<size_t>(dc) * kDState + 8 * k.g + 2 * q);
        k.a2[q] = make_float2(av.x * kLog2e, av.y * kLog2e);
        k.h[q] = make_float2(0.f, 0.f);
    }
    k.bias = a.bias ? a.bias[dc] : 0.f;
    k.Dd = a.D ? a.D[dc] : 0.f;

    const int n = (a.seqlen + TL - 1) / TL;
    const int lane = k.lane;
    constexpr uint32_t kTile = ROWS * TL * sizeof(T);
    constexpr uint32_t kBC = kDState * TL * sizeof(T);
    constexpr uint32_t kSlotBytes = (HAS_Z ? 3u : 2u) * kTile + 2u * kBC;
    int issued = 0;

    auto issue = [&](int c) {  // lane 0 only
        RawTiles<T, ROWS, TL>& R = S.raw[c % STAGES];
        uint64_t* bar = &S.full[c % STAGES];
        mbar_arrive_expect_tx(bar, kSlotBytes);
        const int l0 = c * TL;
        tma_load_3d(&R.u[0][0], &tm_u, bar, l0, k.d0, k.b);
        tma_load_3d(&R.dl[0][0], &tm_dl, bar, l0, k.d0, k.b);
        if (HAS_Z) tma_load_3d(&R.z[0][0], &tm_z, bar, l0, k.d0, k.b);
        tma_load_3d(&R.B[0][0], &tm_B, bar, l0, 0, k.b);
        tma_load_3d(&R.C[0][0], &tm_C, bar, l0, 0, k.b);
    };
    // Makes chunk c's raw tiles available in slot c % STAGES, first refilling the
    // ring up to chunk c + STAGES - 3: when chunk c is acquired, the epilogue of
    // chunk c-2 is done, so only chunks c-1 .. c+STAGES-3 hold slots. Returns
    // false if a TMA wait timed out (after draining what is still in flight).
    auto acquire = [&](int c) -> bool {
        if (!a.use_tma) {
            fill_raw_plain<T, ROWS, TL>(S.raw[c % STAGES], a, k.b, k.d0, c * TL, lane);
            __syncwarp();
            return true;
        }
        const int want = min(n, c + STAGES - 2);
        if (issued < want) {
            if (lane == 0) {
                fence_proxy_async_smem();
                for (int q = issued; q < want; ++q) issue(q);
            }
            issued = want;
        }
        if (mbar_wait_bounded(&S.full[c % STAGES], (c / STAGES) & 1)) return true;
        report_device_error(-6);
        for (int q = c + 1; q < issued; ++q) mbar_wait_bounded(&S.full[q % STAGES], (q / STAGES) & 1);
        return false;
    };

    if (a.use_tma) {
        if (lane == 0) {
#pragma unroll
            for (int s = 0; s < STAGES; ++s) mbar_init(&S.full[s], 1);
            fence_barrier_init();
        }
        __syncwarp();
    }

    // One steady-state iteration: recurrence of chunk c, pre-pass of c+1, epilogue
    // of c-1. P = c & 1 is a compile-time constant so that every shared-memory
    // buffer index is static and the three phases can be interleaved freely.
    auto steady = [&](auto parity, int c) -> bool {
        constexpr int P = decltype(parity)::value;
        if (!acquire(c + 1)) return false;
        k.scan_full(P);
        k.prepass(S.raw[(c + 1) % STAGES], P ^ 1);
        k.template epilogue<true>(S.raw[(c - 1) % STAGES], P ^ 1, (c - 1) * TL);
        __syncwarp();
        return true;
    };

    if (n > 0) {
        if (!acquire(0)) return;
        k.prepass(S.raw[0], 0);
        __syncwarp();
        const int last_steps = a.seqlen - (n - 1) * TL;
        if (n == 1) {
            if (last_steps == TL) k.scan_full(0); else k.scan_partial(0, last_steps);
            __syncwarp();
            k.template epilogue<false>(S.raw[0], 0, 0);
        } else {
            // c = 0: recurrence of chunk 0 and pre-pass of chunk 1
            if (!acquire(1)) return;
            k.scan_full(0);
            k.prepass(S.raw[1 % STAGES], 1);
            __syncwarp();
            // steady state, two iterations per trip (odd c, then even c)
            int c = 1;
#pragma unroll 1
            for (; c + 1 < n - 1; c += 2) {
                if (!steady(std::integral_constant<int, 1>{}, c)) return;
                if (!steady(std::integral_constant<int, 0>{}, c + 1)) return;
            }
            if (c < n - 1) {
                if (!steady(std::integral_constant<int, 1>{}, c)) return;
                ++c;
            }
            // c = n-1: recurrence of the last chunk, epilogue of chunk n-2
            if (last_steps == TL) k.scan_full(c & 1); else k.scan_partial(c & 1, last_steps);
            k.template epilogue<true>(S.raw[(c - 1) % STAGES], (c - 1) & 1, (c - 1) * TL);
            __syncwarp();
            k.template epilogue<false>(S.raw[c % STAGES], c & 1, c * TL);
        }
    }

    if (a.final_state && k.d < a.dim) {
        float4* fs = reinterpret_cast<float4*>(a.final_state + (static_cast<size_t>(k.b) * a.dim + k.d) * kDState +
                                               8 * k.g);
        fs[0] = make_float4(k.h[0].x, k.h[0].y, k.h[1].x, k.h[1].y);
        fs[1] = make_float4(k.h[2].x, k.h[2].y, k.h[3].x, k.h[3].y);
    }
}

}  // namespace mscan
