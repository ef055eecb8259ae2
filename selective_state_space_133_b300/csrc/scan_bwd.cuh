// Backward of the selective scan (training), sm_103a.
//
// Gradients of L = sum(dy * y) with respect to u, delta, z, A, B, C, D,
// delta_bias and the initial state, for the scan of scan_fwd.cuh. The pages
// describe the backward as recomputing A_bar and B_bar from the inputs instead
// of storing them ("mamba->jamba", blog.csdn.net, §2.3); this kernel does the
// same, and keeps only one fp32 state per row every 16 steps between its two
// sweeps. Per step, with dp = dy * silu(z) (or dy) and gh the gradient
// reaching h_l (reverse-mode differentiation of h_l = e h_{l-1} + dt u B,
// e = exp(dt A), y = (C.h + D u) silu(z)):
//     gh     = g + dp C                dC += dp h_l        dB += gh dt u
//     d(dtu) = sum_n gh B              de = gh h_{l-1}     d(dt) += sum_n de e A
//     dA    += de e dt                 g  = gh e           (to h_{l-1})
//     du     = dp D + d(dtu) dt        d(dt) += d(dtu) u   ddelta = d(dt) sigmoid(x)
//
// Layout: one warp per CTA = 16 channels of one batch row, as in the forward.
// Recurrence lanes (rh, rc) = (lane >> 4, lane & 15) own states 8rh..8rh+7 of
// channel rc; pre-pass/epilogue lanes (ec, ej) = (lane >> 1, lane & 1) own
// steps 8ej..8ej+7 of channel ec.
//   Sweep 1 (forward, chunk by chunk): dt and dt*u, the recurrence, and the
//            state before each chunk stored to the workspace; skipped when the
//            forward already stored them (its chunk_states output).
//   Sweep 2 (reverse, chunk by chunk): reload the chunk's starting state,
//            recompute its 16 states into shared memory with C.h; form dp and
//            dz; run the reverse recurrence over the 16 steps; per step, the
//            channel sums of dB and dC are formed in shared memory and added
//            into an fp32 buffer (vector atomics, one per 4 steps); finally
//            du and ddelta per (channel, step).
// dA, dD and delta_bias's gradient are summed over the sequence in registers
// and added atomically into the caller's (zeroed) fp32 outputs.
#pragma once

#include "common.cuh"

namespace mscan {

constexpr int kBwdTL = 16;   // steps per chunk (the checkpoint interval)
constexpr int kBwdCh = 16;   // channels per CTA (one warp)

struct ScanBwdArgs {
    const void* u;
    const void* delta;
    const void* z;          // may be null
    const void* dy;
    const float* bc;        // packed B/C rows, (batch, Lp, 32) fp32
    const float* A;
    const float* D;         // may be null
    const float* bias;      // may be null
    const float* h0;        // may be null
    float* hck;             // (batch, dim, n_chunks, 16) fp32: the workspace, or the forward's chunk states
    int have_hck;           // 1: hck already holds the states (from the forward): skip sweep 1
    float* dbc;             // workspace: (batch, 2, 16, Lp) fp32 sums of dB, dC (zeroed by the host)
    void* du;
    void* ddelta;
    void* dz;               // null iff z is null
    float* dA;              // (dim, 16), zeroed by the host
    float* dD;              // (dim) or null, zeroed by the host
    float* dbias;           // (dim) or null, zeroed by the host
    float* dh0;             // (batch, dim, 16) or null
    int batch, dim, seqlen, Lp;
    int softplus;
};

struct ScanBwdSmem {
    alignas(16) float2 W[kBwdCh][kBwdTL + 1];        // {dt, dt*u}; odd row pitch: distinct banks per channel
    alignas(16) float SG[kBwdCh][kBwdTL + 1];        // d(dt)/d(delta + bias)
    alignas(16) float DP[kBwdCh][kBwdTL + 1];        // dp = dy * silu(z)
    alignas(16) float U[kBwdCh][kBwdTL + 1];         // u
    alignas(16) float4 traj[kBwdTL][2][32];          // recomputed states: [step][half of the 8][lane]
    alignas(16) float P[2][kBwdTL / 4][kBwdCh * 4 + 8];  // partial C.h: [state half][4-step group][channel][4]
    alignas(16) float2 Q[kBwdCh][kBwdTL + 1];        // {d(dtu), d(dt)} per (channel, step), both halves summed
    alignas(16) float RB[kBwdCh][36];                // one step's dB (cols 0..15) and dC (16..31) per channel
    alignas(16) float BC[kBwdTL][32];                // the chunk's packed B/C rows
};

// Eight consecutive values of a row as fp32, zero where l >= L. `vec`: the 8
// are in range and 16-byte (bf16) / 32-byte (fp32) aligned.
__device__ __forceinline__ void ldg8(const float* p, float (&v)[8], bool vec, int valid) {
    if (vec) {
        const float4 a = reinterpret_cast<const float4*>(p)[0];
        const float4 b = reinterpret_cast<const float4*>(p)[1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = i < valid ? p[i] : 0.f;
    }
}
__device__ __forceinline__ void ldg8(const __nv_bfloat16* p, float (&v)[8], bool vec, int valid) {
    if (vec) {
        const uint4 q = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[2 * j + 0] = __uint_as_float(w[j] << 16);
            v[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = i < valid ? __bfloat162float(p[i]) : 0.f;
    }
}

// Eight outputs (same rules as ldg8); reuses the forward's stores.
__device__ __forceinline__ void stg8b(float* p, const float (&v)[8], bool vec, int valid) {
    if (vec) {
        reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < valid) p[i] = v[i];
    }
}
__device__ __forceinline__ void stg8b(__nv_bfloat16* p, const float (&v)[8], bool vec, int valid) {
    if (vec) {
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __nv_bfloat162 q = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
            w[j] = *reinterpret_cast<const uint32_t*>(&q);
        }
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < valid) p[i] = __float2bfloat16_rn(v[i]);
    }
}

// Adds four consecutive floats (16-byte aligned) to global memory atomically.
__device__ __forceinline__ void red_add4(float* p, float4 v) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}

template <typename T, bool SOFTPLUS, bool HAS_Z>
__global__ void __launch_bounds__(32) scan_bwd_kernel(const ScanBwdArgs a) {
    __shared__ ScanBwdSmem sm;
    constexpr float kLn2 = 0.6931471805599453f;
    const int lane = threadIdx.x;
    const int b = blockIdx.y, d0 = blockIdx.x * kBwdCh;
    const int L = a.seqlen, n = (L + kBwdTL - 1) / kBwdTL;
    const int rc = lane & 15, rh = lane >> 4;   // recurrence lanes
    const int ec = lane >> 1, ej = lane & 1;    // pre-pass / epilogue lanes
    const bool ractive = d0 + rc < a.dim;
    const int rd = ractive ? d0 + rc : a.dim - 1;  // clamped for loads of padding channels
    const bool eactive = d0 + ec < a.dim;
    const int ed = eactive ? d0 + ec : a.dim - 1;
    const size_t rrow = static_cast<size_t>(b) * a.dim + rd;
    const size_t erow = static_cast<size_t>(b) * a.dim + ed;
    const bool vec_ok = eactive && (L & 7) == 0;

    float2 A2[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 av = *reinterpret_cast<const float2*>(a.A + static_cast<size_t>(rd) * kDState + 8 * rh + 2 * i);
        A2[i] = make_float2(av.x * kLog2e, av.y * kLog2e);
    }
    const float bias = a.bias ? a.bias[ed] : 0.f;
    const float Dd = a.D ? a.D[ed] : 0.f;
    float* const hck = a.hck + rrow * n * kDState + 8 * rh;
    const float* const bcb = a.bc + static_cast<size_t>(b) * a.Lp * 32;

    // the 8 values of the pre-pass lane's row at steps k*16 + 8ej .. +7 (zero past L)
    auto load8 = [&](const void* base, int k, float (&v)[8]) {
        const int l = k * kBwdTL + 8 * ej;
        ldg8(static_cast<const T*>(base) + erow * L + l, v, vec_ok && l + 8 <= L, eactive ? L - l : 0);
    };
    // the chunk's packed B/C rows (2 KB, contiguous) into shared memory: each
    // 16-byte load and store of the warp covers 512 contiguous bytes
    auto stage_bc = [&](int k) {
        const float4* src = reinterpret_cast<const float4*>(bcb + static_cast<size_t>(k) * kBwdTL * 32);
        float4* dst = reinterpret_cast<float4*>(&sm.BC[0][0]);
#pragma unroll
        for (int j = 0; j < 4; ++j) dst[32 * j + lane] = src[32 * j + lane];
    };
    auto loadB = [&](int t, float2 (&v)[4]) {
        const float4 p0 = *reinterpret_cast<const float4*>(&sm.BC[t][8 * rh]);
        const float4 p1 = *reinterpret_cast<const float4*>(&sm.BC[t][8 * rh + 4]);
        v[0] = make_float2(p0.x, p0.y); v[1] = make_float2(p0.z, p0.w);
        v[2] = make_float2(p1.x, p1.y); v[3] = make_float2(p1.z, p1.w);
    };
    auto loadC = [&](int t, float2 (&v)[4]) {
        const float4 p0 = *reinterpret_cast<const float4*>(&sm.BC[t][kDState + 8 * rh]);
        const float4 p1 = *reinterpret_cast<const float4*>(&sm.BC[t][kDState + 8 * rh + 4]);
        v[0] = make_float2(p0.x, p0.y); v[1] = make_float2(p0.z, p0.w);
        v[2] = make_float2(p1.x, p1.y); v[3] = make_float2(p1.z, p1.w);
    };
    auto ex2_pair = [](float2 x) { return make_float2(ex2_approx(x.x), ex2_approx(x.y)); };

    // ---------------------------------------------------- sweep 1: forward ----
    float2 h[4];
    if (a.h0) {
        const float4* hp = reinterpret_cast<const float4*>(a.h0 + rrow * kDState + 8 * rh);
        const float4 p0 = hp[0], p1 = hp[1];
        h[0] = make_float2(p0.x, p0.y); h[1] = make_float2(p0.z, p0.w);
        h[2] = make_float2(p1.x, p1.y); h[3] = make_float2(p1.z, p1.w);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = make_float2(0.f, 0.f);
    }
#pragma unroll 1
    for (int k = 0; k < (a.have_hck ? 0 : n); ++k) {
        {
            float uv[8], dv[8];
            load8(a.u, k, uv);
            load8(a.delta, k, dv);
            const int l = k * kBwdTL + 8 * ej;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float dt = dv[i] + bias;
                if (SOFTPLUS) dt = softplus_f(dt);
                if (l + i >= L) dt = 0.f;   // padding steps leave the state unchanged
                sm.W[ec][8 * ej + i] = make_float2(dt, dt * uv[i]);
            }
        }
        stage_bc(k);
        __syncwarp();
        if (ractive) {
            float4* hp = reinterpret_cast<float4*>(hck + k * kDState);
            hp[0] = make_float4(h[0].x, h[0].y, h[1].x, h[1].y);
            hp[1] = make_float4(h[2].x, h[2].y, h[3].x, h[3].y);
        }
#pragma unroll
        for (int t = 0; t < kBwdTL; ++t) {
            const float2 w = sm.W[rc][t];
            float2 Bv[4];
            loadB(t, Bv);
            const float2 dd = make_float2(w.x, w.x), du = make_float2(w.y, w.y);
#pragma unroll
            for (int j = 0; j < 4; ++j) h[j] = __ffma2_rn(ex2_pair(__fmul2_rn(dd, A2[j])), h[j], __fmul2_rn(du, Bv[j]));
        }
        __syncwarp();
    }

    // ---------------------------------------------------- sweep 2: reverse ----
    float2 g[4], dAacc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) { g[i] = make_float2(0.f, 0.f); dAacc[i] = make_float2(0.f, 0.f); }
    float dDacc = 0.f, dbacc = 0.f;
    const int col_which = lane >> 4, col_n = lane & 15;  // the dB/dC column this lane sums
#pragma unroll 1
    for (int k = n - 1; k >= 0; --k) {
        const int l0 = k * kBwdTL;
        const int le = l0 + 8 * ej;  // first step of the pre-pass lane's eight
        // the chunk's checkpoint (issued first: its latency overlaps the pre-pass)
        float2 hs[4];
        {
            const float4* hp = reinterpret_cast<const float4*>(hck + k * kDState);
            const float4 p0 = hp[0], p1 = hp[1];
            hs[0] = make_float2(p0.x, p0.y); hs[1] = make_float2(p0.z, p0.w);
            hs[2] = make_float2(p1.x, p1.y); hs[3] = make_float2(p1.z, p1.w);
        }
        // (i) dt, dt*u, d(dt)/dx and u per (channel, step), into shared memory
        {
            float uv[8], dv[8];
            load8(a.u, k, uv);
            load8(a.delta, k, dv);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float x = dv[i] + bias;
                float dt = x, sg = 1.f;
                if (SOFTPLUS) {
                    dt = softplus_f(x);
                    sg = rcp_approx(1.f + ex2_approx(-x * kLog2e));  // softplus'(x) = sigmoid(x)
                }
                if (le + i >= L) dt = 0.f;
                sm.W[ec][8 * ej + i] = make_float2(dt, dt * uv[i]);
                sm.SG[ec][8 * ej + i] = sg;
                sm.U[ec][8 * ej + i] = uv[i];
            }
        }
        stage_bc(k);
        __syncwarp();

        // (ii) the chunk's states, recomputed from its checkpoint, and C.h
        {
            float2 hc[4] = {hs[0], hs[1], hs[2], hs[3]};
            float* Pw = &sm.P[rh][0][4 * rc];
#pragma unroll 1
            for (int t0 = 0; t0 < kBwdTL; t0 += 4) {
                float p[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int t = t0 + i;
                    const float2 w = sm.W[rc][t];
                    float2 Bv[4], Cv[4];
                    loadB(t, Bv);
                    loadC(t, Cv);
                    const float2 dd = make_float2(w.x, w.x), du = make_float2(w.y, w.y);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        hc[j] = __ffma2_rn(ex2_pair(__fmul2_rn(dd, A2[j])), hc[j], __fmul2_rn(du, Bv[j]));
                    sm.traj[t][0][lane] = make_float4(hc[0].x, hc[0].y, hc[1].x, hc[1].y);
                    sm.traj[t][1][lane] = make_float4(hc[2].x, hc[2].y, hc[3].x, hc[3].y);
                    float2 acc = __fmul2_rn(Cv[0], hc[0]);
                    acc = __ffma2_rn(Cv[1], hc[1], acc);
                    acc = __ffma2_rn(Cv[2], hc[2], acc);
                    acc = __ffma2_rn(Cv[3], hc[3], acc);
                    p[i] = acc.x + acc.y;
                }
                *reinterpret_cast<float4*>(Pw + (t0 / 4) * (kBwdCh * 4 + 8)) = make_float4(p[0], p[1], p[2], p[3]);
            }
        }
        __syncwarp();

        // (iii) dp = dy * silu(z) and dz = dy * (C.h + D u) * silu'(z)
        {
            float gy[8], zv[8], pre[8];
            load8(a.dy, k, gy);
            if (HAS_Z) load8(a.z, k, zv);
#pragma unroll
            for (int gq = 0; gq < 2; ++gq) {
                const float4 x0 = *reinterpret_cast<const float4*>(&sm.P[0][2 * ej + gq][4 * ec]);
                const float4 x1 = *reinterpret_cast<const float4*>(&sm.P[1][2 * ej + gq][4 * ec]);
                pre[4 * gq + 0] = x0.x + x1.x; pre[4 * gq + 1] = x0.y + x1.y;
                pre[4 * gq + 2] = x0.z + x1.z; pre[4 * gq + 3] = x0.w + x1.w;
            }
            float dzv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float uu = sm.U[ec][8 * ej + i];
                const float p = fmaf(Dd, uu, pre[i]);
                float dp = gy[i];
                if (HAS_Z) {
                    const float s = rcp_approx(1.f + ex2_approx(-zv[i] * kLog2e));
                    dzv[i] = gy[i] * p * s * fmaf(zv[i], 1.f - s, 1.f);
                    dp = gy[i] * zv[i] * s;
                }
                dDacc = fmaf(dp, uu, dDacc);
                sm.DP[ec][8 * ej + i] = dp;
            }
            if (HAS_Z) {
                T* dzp = static_cast<T*>(a.dz) + erow * L + le;
                if (eactive && le < L) stg8b(dzp, dzv, vec_ok && le + 8 <= L, L - le);
            }
        }
        __syncwarp();

        // (iv) the reverse recurrence over the chunk's 16 steps; this lane's
        // dB/dC column (the channel sum) goes to the fp32 sums 4 steps at a time
        float* const dcol = a.dbc + ((static_cast<size_t>(b) * 2 + col_which) * kDState + col_n) * a.Lp + l0;
#pragma unroll 1
        for (int t0 = kBwdTL - 4; t0 >= 0; t0 -= 4) {
          float accBC[4];
#pragma unroll
          for (int ti = 3; ti >= 0; --ti) {
            const int t = t0 + ti;
            const float2 w = sm.W[rc][t];
            const float dp = sm.DP[rc][t];
            float2 Bv[4], Cv[4], hT[4], hP[4];
            loadB(t, Bv);
            loadC(t, Cv);
            {
                const float4 q0 = sm.traj[t][0][lane], q1 = sm.traj[t][1][lane];
                hT[0] = make_float2(q0.x, q0.y); hT[1] = make_float2(q0.z, q0.w);
                hT[2] = make_float2(q1.x, q1.y); hT[3] = make_float2(q1.z, q1.w);
            }
            if (t > 0) {
                const float4 q0 = sm.traj[t - 1][0][lane], q1 = sm.traj[t - 1][1][lane];
                hP[0] = make_float2(q0.x, q0.y); hP[1] = make_float2(q0.z, q0.w);
                hP[2] = make_float2(q1.x, q1.y); hP[3] = make_float2(q1.z, q1.w);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) hP[j] = hs[j];
            }
            const float2 dd = make_float2(w.x, w.x), du = make_float2(w.y, w.y), dpp = make_float2(dp, dp);
            float2 sdtu = make_float2(0.f, 0.f), sdt = make_float2(0.f, 0.f);
            float2 dBv[4], dCv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 e = ex2_pair(__fmul2_rn(dd, A2[j]));
                const float2 gh = __ffma2_rn(dpp, Cv[j], g[j]);
                dCv[j] = __fmul2_rn(dpp, hT[j]);
                dBv[j] = __fmul2_rn(gh, du);
                sdtu = __ffma2_rn(gh, Bv[j], sdtu);
                const float2 dee = __fmul2_rn(__fmul2_rn(gh, hP[j]), e);
                sdt = __ffma2_rn(dee, A2[j], sdt);
                dAacc[j] = __ffma2_rn(dee, dd, dAacc[j]);
                g[j] = __fmul2_rn(gh, e);
            }
            {   // both state halves of the channel: lanes rc and rc + 16
                float qa = sdtu.x + sdtu.y, qb = sdt.x + sdt.y;
                qa += __shfl_xor_sync(0xffffffffu, qa, 16);
                qb += __shfl_xor_sync(0xffffffffu, qb, 16);
                if (rh == 0) sm.Q[rc][t] = make_float2(qa, qb * kLn2);
            }
            // channel sums of this step's dB and dC
            float4* rb = reinterpret_cast<float4*>(&sm.RB[rc][0]);
            rb[2 * rh] = make_float4(dBv[0].x, dBv[0].y, dBv[1].x, dBv[1].y);
            rb[2 * rh + 1] = make_float4(dBv[2].x, dBv[2].y, dBv[3].x, dBv[3].y);
            rb[4 + 2 * rh] = make_float4(dCv[0].x, dCv[0].y, dCv[1].x, dCv[1].y);
            rb[4 + 2 * rh + 1] = make_float4(dCv[2].x, dCv[2].y, dCv[3].x, dCv[3].y);
            __syncwarp();
            float2 sacc = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < kBwdCh; c += 2) sacc = __fadd2_rn(sacc, make_float2(sm.RB[c][lane], sm.RB[c + 1][lane]));
            accBC[ti] = sacc.x + sacc.y;
            __syncwarp();
          }
          red_add4(dcol + t0, make_float4(accBC[0], accBC[1], accBC[2], accBC[3]));
        }

        // (v) du and ddelta per (channel, step)
        {
            float duv[8], dxv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int t = 8 * ej + i;
                const float2 q = sm.Q[ec][t];
                const float sdtu = q.x;
                const float sdt = fmaf(sdtu, sm.U[ec][t], q.y);
                duv[i] = fmaf(sm.DP[ec][t], Dd, sdtu * sm.W[ec][t].x);
                dxv[i] = le + i < L ? sdt * sm.SG[ec][t] : 0.f;
                dbacc += dxv[i];
            }
            if (eactive && le < L) {
                stg8b(static_cast<T*>(a.du) + erow * L + le, duv, vec_ok && le + 8 <= L, L - le);
                stg8b(static_cast<T*>(a.ddelta) + erow * L + le, dxv, vec_ok && le + 8 <= L, L - le);
            }
        }
        __syncwarp();
    }

    // the gradient of the initial state, dA, dD and the bias's gradient
    if (a.dh0 && ractive) {
        float4* p = reinterpret_cast<float4*>(a.dh0 + rrow * kDState + 8 * rh);
        p[0] = make_float4(g[0].x, g[0].y, g[1].x, g[1].y);
        p[1] = make_float4(g[2].x, g[2].y, g[3].x, g[3].y);
    }
    if (ractive) {
        float* p = a.dA + static_cast<size_t>(rd) * kDState + 8 * rh;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            atomicAdd(p + 2 * j, dAacc[j].x);
            atomicAdd(p + 2 * j + 1, dAacc[j].y);
        }
    }
    dDacc += __shfl_xor_sync(0xffffffffu, dDacc, 1);
    dbacc += __shfl_xor_sync(0xffffffffu, dbacc, 1);
    if (eactive && ej == 0) {
        if (a.dD) atomicAdd(a.dD + ed, dDacc);
        if (a.dbias) atomicAdd(a.dbias + ed, dbacc);
    }
}

// dB and dC in the I/O dtype from the fp32 sums: out[b][n][l] = dbc[b][which][n][l].
template <typename T>
__global__ void __launch_bounds__(256)
dbc_unpack_kernel(const float* __restrict__ dbc, T* __restrict__ dB, T* __restrict__ dC, int batch, int L, int Lp) {
    const long long total = static_cast<long long>(batch) * 2 * kDState * L;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int l = static_cast<int>(i % L);
        const long long r = i / L;  // (b, which, n)
        const int nn = static_cast<int>(r % kDState);
        const int which = static_cast<int>((r / kDState) % 2);
        const int bb = static_cast<int>(r / (2 * kDState));
        const float v = dbc[r * Lp + l];
        T* out = which ? dC : dB;
        out[(static_cast<size_t>(bb) * kDState + nn) * L + l] = Io<T>::from_f(v);
    }
}

}  // namespace mscan
