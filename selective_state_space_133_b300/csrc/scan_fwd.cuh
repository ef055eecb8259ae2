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
//  * At N = 16 the path is bound by the SM, not by HBM: every (b,l,d,n)
//    element costs one MUFU ex2 and four FP32 operations (dt*A, dt*u*B, the
//    recurrence FMA, the C.h FMA), B300 retires about 32 ex2 and 128 FP32
//    lane-operations per clock per SM, and every element also needs its B and
//    C values delivered from shared memory (256 bytes per wavefront at best,
//    one wavefront per clock per SM). Each thread therefore walks the whole
//    sequence for its states sequentially: no cross-thread scan and no carry
//    fix-up pass, which would add work per element.
//  * A CTA is one warp = 16 channels of one batch row with its own copy ring,
//    so no warp ever waits for another. In the recurrence, lane (h, c) =
//    (lane >> 4, lane & 15) owns states 8h..8h+7 of channel c: each half-warp
//    reads one B/C address per step (a 16-byte broadcast load, 2 wavefronts),
//    and the per-(channel, step) values dt and dt*u are shared by two lanes.
//  * The sequence is cut into 16-step chunks. Lane 0 issues 3-D TMA loads of
//    a chunk's u/delta/z tiles (16 channels x 16 steps) and of the chunk's
//    packed B/C rows (fp32, [step][B0..15 C0..15], written once per call by
//    bc_pack_kernel) into a 4-deep ring with one "full" mbarrier per slot (TMA
//    transaction count); a slot is refilled as soon as the warp is done with
//    it, and the waits for data are bounded and report a timeout instead of
//    hanging.
//  * Per chunk there are three phases, run in order:
//      pre-pass   once per (channel, step), lane (c, j) = (lane >> 1, lane & 1)
//                 taking steps 8j..8j+7 of channel c: dt and dt*u, stored as
//                 float2 pairs that the recurrence uses, each value broadcast
//                 to both halves, as packed f32x2 operands;
//      recurrence per lane, 16 steps x 8 states with packed FMUL2/FFMA2 and
//                 software-pipelined by one step; the step's partial C.h of
//                 the lane's 8 states goes to shared memory (one 16-byte store
//                 per 4 steps);
//      epilogue   once per (channel, step), same lanes as the pre-pass: the two
//                 partials + D*u, times silu(z), rounded, one 16-byte store.
//    All shared-memory strides are chosen so that these accesses are free of
//    bank conflicts.
//  * Steps past the end of the sequence get dt = 0 (exp(0) = 1, zero input),
//    so the padded tail leaves the state unchanged and the final state needs
//    no masking.
#pragma once

#include "common.cuh"

namespace mscan {

constexpr int kTL = 16;                  // steps per chunk
constexpr int kCtaCh = 16;               // channels per CTA (one warp)
constexpr int kBCW = 2 * kDState;        // floats per step in the packed B/C buffer
constexpr int kWP = kTL + 2;             // W row stride (float2): 16-byte rows, distinct banks
constexpr int kPJ = kCtaCh * 4 + 8;      // partial sums: stride between 4-step groups (floats)
constexpr int kPH = (kTL / 4) * kPJ;     // partial sums: stride between state halves (floats)
constexpr int kStages = 4;               // TMA ring depth
constexpr int kScanThreads = 32;

constexpr int kConvW = 4;  // width of the causal convolution fused in front of the scan

struct ScanArgs {
    const float* A;
    const float* D;      // may be null
    const float* bias;   // may be null
    const float* h0;     // state before the first step, may be null (zero)
    void* y;
    float* final_state;  // may be null
    float* chunk_states; // (batch, dim, ceil(seqlen / 16), 16): the state before every chunk; may be null
    int batch, dim, seqlen;
    // With the fused convolution (the kernel's CONV instantiation) the u tiles
    // hold the convolution's input x, and u = silu(sum_k w[k] x[l-3+k] + b):
    const float* conv_w;     // (dim, kConvW) fp32
    const float* conv_b;     // (dim) fp32, may be null
    const void* conv_state;  // (batch, dim, kConvW - 1) io dtype: x before step 0, oldest first; may be null
};

template <typename T>
struct ScanStage {
    alignas(128) T u[kCtaCh][kTL];
    alignas(128) T dl[kCtaCh][kTL];
    alignas(128) T z[kCtaCh][kTL];
    alignas(128) float bc[kTL][kBCW];
};

template <typename T>
struct ScanSmem {
    ScanStage<T> st[kStages];
    alignas(16) float2 W[kCtaCh][kWP];   // {dt, dt*u} per (channel, step)
    alignas(16) float P[2 * kPH];        // [state half][4-step group][channel][4 steps]
    alignas(8) uint64_t full[kStages];   // TMA transaction barrier per slot
    alignas(16) float U[kCtaCh][kTL + 1];  // u after the convolution (CONV only)
    float XH[2][kCtaCh][kConvW - 1];     // the last inputs x of the previous chunk (CONV only)
};

// ------------------------------------------------------------ helpers ------

// Eight consecutive values (16-byte aligned for bf16, 32-byte for fp32) as fp32.
__device__ __forceinline__ void lds8(const float* p, float (&v)[8]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0];
    const float4 b = reinterpret_cast<const float4*>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void lds8(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 q = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        v[2 * j + 0] = __uint_as_float(w[j] << 16);
        v[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
}

// Eight consecutive outputs to global memory; `vec` = all 8 are in range and
// the address is aligned for vector stores; otherwise the first `valid` go out
// one by one.
__device__ __forceinline__ void stg8(float* p, const float (&v)[8], bool vec, int valid) {
    if (vec) {
        reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < valid) p[i] = v[i];
    }
}
__device__ __forceinline__ void stg8(__nv_bfloat16* p, const float (&v)[8], bool vec, int valid) {
    __nv_bfloat162 o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
    if (vec) {
        *reinterpret_cast<uint4*>(p) = make_uint4(*reinterpret_cast<const uint32_t*>(&o[0]),
                                                  *reinterpret_cast<const uint32_t*>(&o[1]),
                                                  *reinterpret_cast<const uint32_t*>(&o[2]),
                                                  *reinterpret_cast<const uint32_t*>(&o[3]));
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < valid) p[i] = (i & 1) ? o[i >> 1].y : o[i >> 1].x;
    }
}

// softplus on a pair: max(x,0) + log1p(e^{-|x|}), log1p on the FP32 pipe.
__device__ __forceinline__ float2 softplus2(float2 x) {
    const float2 v = make_float2(ex2_approx(-fabsf(x.x) * kLog2e), ex2_approx(-fabsf(x.y) * kLog2e));
    return __fadd2_rn(make_float2(fmaxf(x.x, 0.f), fmaxf(x.y, 0.f)), __fmul2_rn(v, log1p_unit_q2(v)));
}

// y * silu(z) on a pair: y * z / (1 + e^{-z}).
__device__ __forceinline__ float2 gate2(float2 y, float2 z) {
    const float2 e = make_float2(ex2_approx(-z.x * kLog2e), ex2_approx(-z.y * kLog2e));
    const float2 den = __fadd2_rn(e, make_float2(1.f, 1.f));
    const float2 r = make_float2(rcp_approx(den.x), rcp_approx(den.y));
    return __fmul2_rn(__fmul2_rn(y, z), r);
}

// ------------------------------------------------------------- kernel ------

template <typename T, bool SOFTPLUS, bool HAS_Z, bool CONV>
__global__ void __launch_bounds__(kScanThreads)
scan_fwd_kernel(const ScanArgs a, const __grid_constant__ CUtensorMap tm_u,
                const __grid_constant__ CUtensorMap tm_dl, const __grid_constant__ CUtensorMap tm_z,
                const __grid_constant__ CUtensorMap tm_bc) {
    __shared__ ScanSmem<T> sm;
    const int lane = threadIdx.x;
    const int b = blockIdx.y;
    const int d0 = blockIdx.x * kCtaCh;
    const int L = a.seqlen;
    const int n = (L + kTL - 1) / kTL;

    // Chunk k's tiles into slot k % kStages (lane 0 only).
    auto issue = [&](int k) {
        constexpr uint32_t kTile = kCtaCh * kTL * sizeof(T);
        constexpr uint32_t kStageBytes = (HAS_Z ? 3u : 2u) * kTile + kTL * kBCW * 4u;
        ScanStage<T>& S = sm.st[k % kStages];
        uint64_t* bar = &sm.full[k % kStages];
        mbar_arrive_expect_tx(bar, kStageBytes);
        const int l0 = k * kTL;
        tma_load_3d(&S.u[0][0], &tm_u, bar, l0, d0, b);
        tma_load_3d(&S.dl[0][0], &tm_dl, bar, l0, d0, b);
        if (HAS_Z) tma_load_3d(&S.z[0][0], &tm_z, bar, l0, d0, b);
        tma_load_3d(&S.bc[0][0], &tm_bc, bar, 0, l0, b);
    };

    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kStages; ++s) mbar_init(&sm.full[s], 1);
        fence_barrier_init();
        for (int k = 0; k < n && k < kStages; ++k) issue(k);
    }
    __syncwarp();

    // Recurrence lanes: channel rc, states 8*rh .. 8*rh+7.
    const int rc = lane & 15, rh = lane >> 4;
    // Pre-pass / epilogue lanes: channel ec, steps 8*ej .. 8*ej+7 of each chunk.
    const int ec = lane >> 1, ej = lane & 1;

    const int rd = d0 + rc < a.dim ? d0 + rc : a.dim - 1;  // clamped for parameter loads
    float2 A2[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 av = *reinterpret_cast<const float2*>(a.A + static_cast<size_t>(rd) * kDState + 8 * rh + 2 * i);
        A2[i] = make_float2(av.x * kLog2e, av.y * kLog2e);
    }
    float2 h[4];
    if (a.h0) {
        const float4* hp = reinterpret_cast<const float4*>(a.h0 + (static_cast<size_t>(b) * a.dim + rd) * kDState +
                                                           8 * rh);
        const float4 p0 = hp[0], p1 = hp[1];
        h[0] = make_float2(p0.x, p0.y); h[1] = make_float2(p0.z, p0.w);
        h[2] = make_float2(p1.x, p1.y); h[3] = make_float2(p1.z, p1.w);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = make_float2(0.f, 0.f);
    }

    const int ed = d0 + ec;
    const bool eactive = ed < a.dim;
    const int edc = eactive ? ed : a.dim - 1;
    const float bias = a.bias ? a.bias[edc] : 0.f;
    const float Dd = a.D ? a.D[edc] : 0.f;
    float cw[kConvW] = {0.f, 0.f, 0.f, 0.f}, cb = 0.f;
    if (CONV) {
        const float4 w4 = *reinterpret_cast<const float4*>(a.conv_w + static_cast<size_t>(edc) * kConvW);
        cw[0] = w4.x; cw[1] = w4.y; cw[2] = w4.z; cw[3] = w4.w;
        cb = a.conv_b ? a.conv_b[edc] : 0.f;
        // the inputs before step 0 (read by the same lane in the first pre-pass)
        if (ej == 0) {
#pragma unroll
            for (int m = 0; m < kConvW - 1; ++m)
                sm.XH[1][ec][m] = (a.conv_state && eactive)
                    ? Io<T>::to_f(static_cast<const T*>(a.conv_state)[(static_cast<size_t>(b) * a.dim + ed) *
                                                                          (kConvW - 1) + m])
                    : 0.f;
        }
    }
    // this lane's output: steps 8*ej .. 8*ej+7 of every chunk of channel ed
    T* const yrow = static_cast<T*>(a.y) + (static_cast<size_t>(b) * a.dim + edc) * L + 8 * ej;
    const bool vec_ok = eactive && (L & 7) == 0;

    // Bounded wait for the tiles of chunk k in slot s; warp-uniform verdict. On
    // a timeout the warp records the error and waits (bounded again) for the
    // copies that may still be in flight, so that none lands after it exits.
    auto wait_full = [&](int s, int k) -> bool {
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&sm.full[s], (k / kStages) & 1));
        if (!ok) {
            report_device_error(-6);
            for (int j = k + 1; j < n && j < k + kStages; ++j)
                mbar_wait_bounded(&sm.full[j % kStages], (j / kStages) & 1);
        }
        return ok;
    };

    // Slot s is free once every lane is done with chunk k: lane 0 refills it
    // with chunk k + kStages (the proxy fence orders the lanes' generic reads
    // of the slot before the TMA's writes).
    auto release = [&](int k) {
        if (lane == 0 && k + kStages < n) {
            fence_proxy_async_smem();
            issue(k + kStages);
        }
    };

    // --- the three phases --------------------------------------------------
    auto prepass = [&](const ScanStage<T>& S, int k) {
        float uv[8], dv[8];
        lds8(&S.u[ec][8 * ej], uv);
        lds8(&S.dl[ec][8 * ej], dv);
        if (CONV) {
            // the 3 inputs before this lane's first step: from this chunk (second
            // half) or from the previous chunk's last inputs (first half)
            float xm[kConvW - 1];
#pragma unroll
            for (int m = 0; m < kConvW - 1; ++m)
                xm[m] = ej ? Io<T>::to_f(S.u[ec][8 - (kConvW - 1) + m]) : sm.XH[(k + 1) & 1][ec][m];
            if (ej) {
#pragma unroll
                for (int m = 0; m < kConvW - 1; ++m) sm.XH[k & 1][ec][m] = uv[8 - (kConvW - 1) + m];
            }
            float xs[8 + kConvW - 1];
#pragma unroll
            for (int m = 0; m < kConvW - 1; ++m) xs[m] = xm[m];
#pragma unroll
            for (int i = 0; i < 8; ++i) xs[kConvW - 1 + i] = uv[i];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float acc = cb;
#pragma unroll
                for (int m = 0; m < kConvW; ++m) acc = fmaf(cw[m], xs[i + m], acc);
                uv[i] = silu_f(acc);
                sm.U[ec][8 * ej + i] = uv[i];
            }
        }
        const float2 bb = make_float2(bias, bias);
        float4* W = reinterpret_cast<float4*>(&sm.W[ec][8 * ej]);
        const int lr = k * kTL + 8 * ej;  // first step of this lane's eight
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 x = __fadd2_rn(make_float2(dv[2 * i], dv[2 * i + 1]), bb);
            if (SOFTPLUS) x = softplus2(x);
            float2 w = __fmul2_rn(x, make_float2(uv[2 * i], uv[2 * i + 1]));
            if (lr + 8 > L) {  // sequence tail: padding steps leave the state unchanged
                if (lr + 2 * i >= L) { x.x = 0.f; w.x = 0.f; }
                if (lr + 2 * i + 1 >= L) { x.y = 0.f; w.y = 0.f; }
            }
            W[i] = make_float4(x.x, w.x, x.y, w.y);
        }
    };

    // The recurrence is software-pipelined by one step: the loads, the ex2 of
    // dt*A and dt*u*B of step t+1 are issued before the state update of step t
    // uses them. The next step's ex2 sit between the current step's C.h FMAs,
    // so the MUFU and FMA pipes are fed alternately.
    auto recurrence = [&](const ScanStage<T>& S) {
        const float2* W = &sm.W[rc][0];
        const float* bc = &S.bc[0][0];
        float* P = &sm.P[rh * kPH + 4 * rc];
        float2 e[4], pb[4], cv[4];
        // step 0's operands
        {
            const float2 w = W[0];
            const float4 b0 = *reinterpret_cast<const float4*>(bc + 8 * rh);
            const float4 b1 = *reinterpret_cast<const float4*>(bc + 8 * rh + 4);
            const float4 c0 = *reinterpret_cast<const float4*>(bc + kDState + 8 * rh);
            const float4 c1 = *reinterpret_cast<const float4*>(bc + kDState + 8 * rh + 4);
            const float2 dd = make_float2(w.x, w.x), du = make_float2(w.y, w.y);
            const float2 bv[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w), make_float2(b1.x, b1.y),
                                  make_float2(b1.z, b1.w)};
            cv[0] = make_float2(c0.x, c0.y); cv[1] = make_float2(c0.z, c0.w);
            cv[2] = make_float2(c1.x, c1.y); cv[3] = make_float2(c1.z, c1.w);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 x = __fmul2_rn(dd, A2[i]);
                e[i] = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                pb[i] = __fmul2_rn(du, bv[i]);
            }
        }
#pragma unroll
        for (int t0 = 0; t0 < kTL; t0 += 4) {
            float p[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = t0 + i;
                const int tn = t + 1 < kTL ? t + 1 : t;  // the last step loads nothing new (values unused)
                const float2 w = W[tn];
                const float4 b0 = *reinterpret_cast<const float4*>(bc + tn * kBCW + 8 * rh);
                const float4 b1 = *reinterpret_cast<const float4*>(bc + tn * kBCW + 8 * rh + 4);
                const float4 c0 = *reinterpret_cast<const float4*>(bc + tn * kBCW + kDState + 8 * rh);
                const float4 c1 = *reinterpret_cast<const float4*>(bc + tn * kBCW + kDState + 8 * rh + 4);
                const float2 dd = make_float2(w.x, w.x), du = make_float2(w.y, w.y);
                const float2 bn[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w), make_float2(b1.x, b1.y),
                                      make_float2(b1.z, b1.w)};
                const float2 cn[4] = {make_float2(c0.x, c0.y), make_float2(c0.z, c0.w), make_float2(c1.x, c1.y),
                                      make_float2(c1.z, c1.w)};
                // Written in an issue-friendly order (a warp issues in order):
                // every result is consumed a few independent instructions later.
#pragma unroll
                for (int j = 0; j < 4; ++j) h[j] = __ffma2_rn(e[j], h[j], pb[j]);   // step t
                float2 x[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) x[j] = __fmul2_rn(dd, A2[j]);             // step t+1
                float2 acc = __fmul2_rn(cv[0], h[0]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (t + 1 < kTL) e[j] = make_float2(ex2_approx(x[j].x), ex2_approx(x[j].y));
                    if (j < 3) acc = __ffma2_rn(cv[j + 1], h[j + 1], acc);
                }
                if (t + 1 < kTL) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        pb[j] = __fmul2_rn(du, bn[j]);
                        cv[j] = cn[j];
                    }
                }
                p[i] = acc.x + acc.y;
            }
            *reinterpret_cast<float4*>(P + (t0 / 4) * kPJ) = make_float4(p[0], p[1], p[2], p[3]);
        }
    };

    auto epilogue = [&](const ScanStage<T>& S, int k) {
        // steps 8*ej .. 8*ej+7 are the 4-step groups 2*ej and 2*ej+1
        const float* P0 = &sm.P[(2 * ej) * kPJ + 4 * ec];
        const float4 a0 = *reinterpret_cast<const float4*>(P0);
        const float4 a1 = *reinterpret_cast<const float4*>(P0 + kPJ);
        const float4 b0 = *reinterpret_cast<const float4*>(P0 + kPH);
        const float4 b1 = *reinterpret_cast<const float4*>(P0 + kPH + kPJ);
        float2 y[4] = {__fadd2_rn(make_float2(a0.x, a0.y), make_float2(b0.x, b0.y)),
                       __fadd2_rn(make_float2(a0.z, a0.w), make_float2(b0.z, b0.w)),
                       __fadd2_rn(make_float2(a1.x, a1.y), make_float2(b1.x, b1.y)),
                       __fadd2_rn(make_float2(a1.z, a1.w), make_float2(b1.z, b1.w))};
        float uv[8];
        if (CONV) {
#pragma unroll
            for (int i = 0; i < 8; ++i) uv[i] = sm.U[ec][8 * ej + i];
        } else {
            lds8(&S.u[ec][8 * ej], uv);
        }
        const float2 DD = make_float2(Dd, Dd);
#pragma unroll
        for (int i = 0; i < 4; ++i) y[i] = __ffma2_rn(DD, make_float2(uv[2 * i], uv[2 * i + 1]), y[i]);
        if (HAS_Z) {
            float zv[8];
            lds8(&S.z[ec][8 * ej], zv);
#pragma unroll
            for (int i = 0; i < 4; ++i) y[i] = gate2(y[i], make_float2(zv[2 * i], zv[2 * i + 1]));
        }
        const float out[8] = {y[0].x, y[0].y, y[1].x, y[1].y, y[2].x, y[2].y, y[3].x, y[3].y};
        const int l = k * kTL + 8 * ej;
        if (vec_ok && l + 8 <= L) {
            stg8(yrow + k * kTL, out, true, 8);
        } else if (eactive && l < L) {
            stg8(yrow + k * kTL, out, false, L - l);
        }
    };

    // --- main loop ----------------------------------------------------------
    // The phases run in order (recurrence k, epilogue k, pre-pass k+1), so W
    // and P are single-buffered; the other warps on the SM fill the issue
    // slots each phase leaves idle. The loop body is not unrolled over the
    // ring: one copy of the (fully unrolled) chunk code stays in the
    // instruction cache.
    if (n > 0) {
        if (!wait_full(0, 0)) return;
        prepass(sm.st[0], 0);
        __syncwarp();
        float* const ck = a.chunk_states ? a.chunk_states + (static_cast<size_t>(b) * a.dim + rd) * n * kDState + 8 * rh
                                         : nullptr;
        const bool ck_store = ck && d0 + rc < a.dim;
#pragma unroll 1
        for (int k = 0; k < n; ++k) {
            const ScanStage<T>& S = sm.st[k % kStages];
            if (ck_store) {  // the state before chunk k, for the backward
                float4* p = reinterpret_cast<float4*>(ck + static_cast<size_t>(k) * kDState);
                p[0] = make_float4(h[0].x, h[0].y, h[1].x, h[1].y);
                p[1] = make_float4(h[2].x, h[2].y, h[3].x, h[3].y);
            }
            recurrence(S);
            __syncwarp();
            epilogue(S, k);
            __syncwarp();
            release(k);
            if (k + 1 < n) {
                const int s1 = (k + 1) % kStages;
                if (!wait_full(s1, k + 1)) return;
                prepass(sm.st[s1], k + 1);
            }
            __syncwarp();
        }
    }

    if (a.final_state && d0 + rc < a.dim) {
        float4* fs = reinterpret_cast<float4*>(a.final_state +
                                               (static_cast<size_t>(b) * a.dim + d0 + rc) * kDState + 8 * rh);
        fs[0] = make_float4(h[0].x, h[0].y, h[1].x, h[1].y);
        fs[1] = make_float4(h[2].x, h[2].y, h[3].x, h[3].y);
    }
}

// Packs B and C ((batch, 16, L) each, io dtype) into one fp32 buffer
// (batch, Lp, 32): row l holds B[:, l] then C[:, l]; rows l >= L are zero.
// One thread per (batch, row): strided reads coalesce across threads, and each
// thread writes its 128-byte row with eight 16-byte stores.
template <typename T>
__global__ void __launch_bounds__(256)
bc_pack_kernel(const T* __restrict__ B, const T* __restrict__ C, float* __restrict__ out, int batch, int L,
               int Lp) {
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= static_cast<long long>(batch) * Lp) return;
    const int b = static_cast<int>(i / Lp);
    const int l = static_cast<int>(i % Lp);
    float v[kBCW];
    const bool ok = l < L;
    const size_t base = static_cast<size_t>(b) * kDState * L + l;
#pragma unroll
    for (int s = 0; s < kDState; ++s) {
        v[s] = ok ? Io<T>::to_f(B[base + static_cast<size_t>(s) * L]) : 0.f;
        v[kDState + s] = ok ? Io<T>::to_f(C[base + static_cast<size_t>(s) * L]) : 0.f;
    }
    float4* o = reinterpret_cast<float4*>(out + i * kBCW);
#pragma unroll
    for (int j = 0; j < kBCW / 4; ++j) o[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
}

// Copies rows of length L into rows of pitch Lpitch >= L (the tail is left as
// is: TMA boxes read it, but padding steps are masked in the pre-pass). Used
// only when L * sizeof(T) is not a multiple of 16 bytes, which a TMA tensor
// map cannot stride over.
template <typename T>
__global__ void __launch_bounds__(256)
row_pitch_kernel(const T* __restrict__ src, T* __restrict__ dst, long long rows, int L, int Lpitch) {
    const long long total = rows * L;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long r = i / L;
        const int l = static_cast<int>(i - r * L);
        dst[r * Lpitch + l] = src[i];
    }
}

}  // namespace mscan
