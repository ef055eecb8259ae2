// Backward of the selective scan (training), sm_103a.
//
// Gradients of L = sum(dy * y) with respect to u, delta, z, A, B, C, D,
// delta_bias and the initial state, for the scan of scan_fwd.cuh. The pages
// describe the backward as recomputing A_bar and B_bar from the inputs instead
// of storing them ("mamba->jamba", blog.csdn.net, §2.3); this kernel does the
// same, and keeps only one fp32 state per row every 16 steps between its two
// sweeps. Per step, with dp = dy * silu(z) (or dy) and gh the gradient
// reaching h_l (reverse-mode differentiation of h_l = e h_{l-1} + gain u B,
// e = exp(dt A), gain = dt, y = (C.h + D u) silu(z)):
//     gh     = g + dp C                dC += dp h_l        dB += gh gain u
//     de     = gh h_{l-1}              d(dt) += sum_n de e A
//     dA    += de e dt                 g  = gh e           (to h_{l-1})
//     du     = dp D + sum_n gh B gain  d(dt) += sum_n gh B u (d gain / d dt)
//     ddelta = d(dt) sigmoid(x)
// With the exact zero-order-hold gain (ZOH; "Mamba 论文精读" §2.2) gain =
// (e - 1) / A, d gain / d dt = e, and dA also gains gh B u (d gain / dA),
// d gain / dA = (dt e - gain) / A, taken from its series
// dt^2 (1/2 + x/3 + x^2/8), x = dt A, where |x| < 1/64 (next term <= 1e-7
// relative).
//
// Layout as in the forward with 8 states a lane (4 at N = 8; ScanBwdGeo):
// one warp per CTA; recurrence lane
// (rh, rc) = (lane / kCh, lane % kCh) owns states kS*rh .. kS*rh + kS - 1 of
// channel rc; pre-pass/epilogue lanes (ec, ej) = (lane / kG, lane % kG) own
// steps kSP*ej .. kSP*ej + kSP - 1 of channel ec.
//   Sweep 1 (forward, chunk by chunk): dt and dt*u, the recurrence, and the
//            state before each chunk stored to the workspace; skipped when the
//            forward already stored them (its chunk_states output).
//   Sweep 2 (reverse, chunk by chunk): reload the chunk's starting state,
//            recompute the states of its 16 steps into shared memory with C.h; form dp and
//            dz; run the reverse recurrence over the 16 steps; per step, the
//            channel sums of dB and dC are formed in shared memory and added
//            into an fp32 buffer (vector atomics, one per 4 steps); finally
//            du and ddelta per (channel, step).
// dA, dD and delta_bias's gradient are summed over the sequence in registers
// and added atomically into the caller's (zeroed) fp32 outputs.
#pragma once

#include "scan_fwd.cuh"

namespace mscan {

constexpr int kBwdTL = 16;   // steps per chunk (the checkpoint interval)

// The backward's lane geometry: the forward's with 8 states per lane (4 at
// N = 8); wider lanes would take it past the register file.
template <int NS>
using ScanBwdGeo = FwdGeo<NS, NS == 8 ? 4 : 8>;

struct ScanBwdArgs {
    const void* u;
    const void* delta;
    const void* z;          // may be null
    const void* dy;
    const float* bc;        // packed B/C rows, (batch, Lp, 2N) fp32
    const float* A;
    const float* D;         // may be null
    const float* bias;      // may be null
    const float* h0;        // may be null
    float* hck;             // (batch, dim, n_chunks, N) fp32: the workspace, or the forward's chunk states
    int have_hck;           // 1: hck already holds the states (from the forward): skip sweep 1
    float* dbc;             // workspace: (batch, 2, N, Lp) fp32 sums of dB, dC (zeroed by the host)
    void* du;
    void* ddelta;
    void* dz;               // null iff z is null
    float* dA;              // (dim, N), zeroed by the host
    float* dD;              // (dim) or null, zeroed by the host
    float* dbias;           // (dim) or null, zeroed by the host
    float* dh0;             // (batch, dim, N) or null
    int* err;               // device error word
    int batch, dim, seqlen, Lp;
};

template <int NS, bool ZOH>
struct ScanBwdSmem {
    using G = ScanBwdGeo<NS>;
    alignas(16) float2 W[G::kCh][kBwdTL + 1];        // {dt, dt*u} ({dt, u} with ZOH); odd row pitch
    alignas(16) float SG[G::kCh][kBwdTL + 1];        // d(dt)/d(delta + bias)
    alignas(16) float DP[G::kCh][kBwdTL + 1];        // dp = dy * silu(z)
    alignas(16) float U[ZOH ? 1 : G::kCh][kBwdTL + 1];  // u (with ZOH, W's second value holds it)
    alignas(16) float4 traj[kBwdTL][G::kS / 4][32];  // recomputed states: [step][4-state group][lane]
    alignas(16) float P[G::kG][kBwdTL / 4][G::kCh * 4 + 8];  // partial C.h: [state group][4-step group][channel][4]
    alignas(16) float2 Q[G::kCh][kBwdTL + 1];        // per (channel, step), all state groups summed:
                                                     // {sum gh B gain', d(dt) so far}: gain' = 1 for dt*B
                                                     // (du and d(dt) take their dt / u factors later);
                                                     // with ZOH gain' = gain and d(dt) is complete
    alignas(16) float RB[G::kCh][2 * NS + 4];        // one step's dB (cols 0..N-1) and dC (N..2N-1) per channel
    alignas(16) float BC[kBwdTL][2 * NS];            // the chunk's packed B/C rows
};

// n consecutive values of a row in global memory as fp32, zero where past the
// end: `vec` = all n are in range and aligned for vector loads of at most 16
// bytes (as stg_n's stores); otherwise the first `valid` one by one.
template <int n>
__device__ __forceinline__ void ldg_n(const float* p, float (&v)[n], bool vec, int valid) {
    if (vec) {
        lds_n<n>(p, v);  // same vector shapes in global memory
    } else {
#pragma unroll
        for (int i = 0; i < n; ++i) v[i] = i < valid ? p[i] : 0.f;
    }
}
template <int n>
__device__ __forceinline__ void ldg_n(const __nv_bfloat16* p, float (&v)[n], bool vec, int valid) {
    if (vec) {
        lds_n<n>(p, v);
    } else {
#pragma unroll
        for (int i = 0; i < n; ++i) v[i] = i < valid ? __bfloat162float(p[i]) : 0.f;
    }
}

// A float2 in shared memory read and written with volatile instructions,
// which the compiler may not hoist out of a loop (so that it does not keep
// the value in registers across the loop instead) and keeps in order among
// themselves.
__device__ __forceinline__ float2 lds2_pinned(const float2* p) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(smem_u32(p)));
    return v;
}
__device__ __forceinline__ void sts2_pinned(float2* p, float2 v) {
    asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(smem_u32(p)), "f"(v.x), "f"(v.y));
}

// Adds four consecutive floats (16-byte aligned) to global memory atomically.
__device__ __forceinline__ void red_add4(float* p, float4 v) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}

// d gain / dA of the ZOH gain on a pair of states, with x2 = dt*a*log2(e),
// e = exp(dt a), gain = (e - 1)/a (zoh_gain2), dt and 1/a.
__device__ __forceinline__ float2 zoh_dgain_da2(float2 x2, float2 e, float2 gain, float2 dt, float2 inv_a) {
    constexpr float kLn2 = 0.6931471805599453f;
    constexpr float kSmall = 0.022542110013890053f;  // |dt a| < 1/64, as in zoh_gain2
    const float2 x = __fmul2_rn(x2, make_float2(kLn2, kLn2));
    float2 t = __ffma2_rn(x, make_float2(0.125f, 0.125f), make_float2(1.f / 3.f, 1.f / 3.f));
    t = __ffma2_rn(t, x, make_float2(0.5f, 0.5f));
    const float2 ss = __fmul2_rn(__fmul2_rn(dt, dt), t);
    const float2 sl = __fmul2_rn(__ffma2_rn(dt, e, make_float2(-gain.x, -gain.y)), inv_a);
    return make_float2(fabsf(x2.x) < kSmall ? ss.x : sl.x, fabsf(x2.y) < kSmall ? ss.y : sl.y);
}

template <typename T, int NS, bool SOFTPLUS, bool HAS_Z, bool ZOH>
__global__ void __launch_bounds__(32) scan_bwd_kernel(const ScanBwdArgs a) {
    using G = ScanBwdGeo<NS>;
    constexpr int kS = G::kS, kG = G::kG, kCh = G::kCh, kSP = G::kSP;
    constexpr int H = kS / 2;                              // state pairs per recurrence lane
    constexpr int kPJ = kCh * 4 + 8;
    constexpr int kCols = 2 * NS;                          // dB and dC columns of a step
    constexpr int kCPL = kCols >= 32 ? kCols / 32 : 1;     // columns summed per lane
    constexpr float kLn2 = 0.6931471805599453f;
    __shared__ ScanBwdSmem<NS, ZOH> sm;
    const int lane = threadIdx.x;
    const int b = blockIdx.y, d0 = blockIdx.x * kCh;
    const int L = a.seqlen, n = (L + kBwdTL - 1) / kBwdTL;
    const int rc = lane % kCh, rh = lane / kCh;   // recurrence lanes
    const int ec = lane / kG, ej = lane % kG;     // pre-pass / epilogue lanes
    const bool ractive = d0 + rc < a.dim;
    const int rd = ractive ? d0 + rc : a.dim - 1;  // clamped for loads of padding channels
    const bool eactive = d0 + ec < a.dim;
    const int ed = eactive ? d0 + ec : a.dim - 1;
    const size_t rrow = static_cast<size_t>(b) * a.dim + rd;
    const size_t erow = static_cast<size_t>(b) * a.dim + ed;
    const bool vec_ok = eactive && (L % G::template vec_steps<T>()) == 0;
    // extents (elements) of the tensors, for the checked-bounds build
    const size_t nrows = static_cast<size_t>(a.batch) * a.dim;   // (batch, channel) rows
    const size_t nx = nrows * L;                                  // u, delta, z, dy, du, ddelta, dz
    const size_t npk = static_cast<size_t>(a.batch) * a.Lp;       // packed B/C rows, dB/dC sum columns

    // With ZOH, 1/a of this lane's states and their dA sums live in shared
    // memory (each lane reads back only what it wrote): in registers they
    // would take the kernel past the register file.
    __shared__ float2 inv_a[ZOH ? H : 1][32];
    __shared__ float2 dA_zoh[ZOH ? H : 1][32];
    float2 A2[H];
#pragma unroll
    for (int i = 0; i < H; ++i) {
        const float* ap = a.A + static_cast<size_t>(rd) * NS + kS * rh + 2 * i;
        const float2 av = in_bounds(a.err, a.A, static_cast<size_t>(a.dim) * NS, ap, 2)
            ? *reinterpret_cast<const float2*>(ap) : make_float2(-1.f, -1.f);
        A2[i] = make_float2(av.x * kLog2e, av.y * kLog2e);
        if (ZOH) {
            sts2_pinned(&inv_a[i][lane], make_float2(1.f / av.x, 1.f / av.y));
            sts2_pinned(&dA_zoh[i][lane], make_float2(0.f, 0.f));
        }
    }
    auto IA = [&](int j) -> float2 { return lds2_pinned(&inv_a[ZOH ? j : 0][lane]); };
    // u of (channel c, step t) of the chunk in shared memory
    auto u_at = [&](int c, int t) -> float { return ZOH ? sm.W[c][t].y : sm.U[ZOH ? 0 : c][t]; };
    const float bias = a.bias && in_bounds(a.err, a.bias, a.dim, a.bias + ed) ? a.bias[ed] : 0.f;
    const float Dd = a.D && in_bounds(a.err, a.D, a.dim, a.D + ed) ? a.D[ed] : 0.f;
    float* const hck = a.hck + rrow * n * NS + kS * rh;
    const float* const bcb = a.bc + static_cast<size_t>(b) * a.Lp * kCols;

    // the kSP values of the pre-pass lane's row at steps k*16 + kSP*ej .. (zero past L)
    auto loadN = [&](const void* base, int k, float (&v)[kSP]) {
        const int l = k * kBwdTL + kSP * ej;
        const T* tb = static_cast<const T*>(base);
        const bool vec = vec_ok && l + kSP <= L;
        const int valid = eactive ? L - l : 0;
        if constexpr (kCheckBounds) {
            if ((vec || valid > 0) && !in_bounds(a.err, tb, nx, tb + erow * L + l, vec ? kSP : min(valid, kSP))) {
#pragma unroll
                for (int i = 0; i < kSP; ++i) v[i] = 0.f;
                return;
            }
        }
        ldg_n<kSP>(tb + erow * L + l, v, vec, valid);
    };
    // the chunk's packed B/C rows (16 x 2N floats, contiguous) into shared memory
    auto stage_bc = [&](int k) {
        const float* srcf = bcb + static_cast<size_t>(k) * kBwdTL * kCols;
        if (!in_bounds(a.err, a.bc, npk * kCols, srcf, kBwdTL * kCols)) return;
        const float4* src = reinterpret_cast<const float4*>(srcf);
        float4* dst = reinterpret_cast<float4*>(&sm.BC[0][0]);
#pragma unroll
        for (int j = 0; j < kBwdTL * kCols / 128; ++j) dst[32 * j + lane] = src[32 * j + lane];
    };
    auto loadBC = [&](int t, int off, float2 (&v)[H]) {  // off = 0: B, NS: C
#pragma unroll
        for (int q = 0; q < kS / 4; ++q) {
            const float4 p = *reinterpret_cast<const float4*>(&sm.BC[t][off + kS * rh + 4 * q]);
            v[2 * q] = make_float2(p.x, p.y);
            v[2 * q + 1] = make_float2(p.z, p.w);
        }
    };
    auto ex2_pair = [](float2 x) { return make_float2(ex2_approx(x.x), ex2_approx(x.y)); };
    // the input term of one step on pair j: dt*u*B, or the ZOH gain times u*B (du holds u then)
    auto input_term = [&](float2 x2, float2 e, float2 dd, float2 du, float2 Bj, int j) {
        const float2 t = __fmul2_rn(du, Bj);
        return ZOH ? __fmul2_rn(zoh_gain2(x2, e, dd, IA(j)), t) : t;
    };
    // pre-pass of chunk k: dt and its second operand (dt*u, or u with ZOH) per (channel, step)
    auto prepass = [&](int k, bool full) {
        float uv[kSP], dv[kSP];
        loadN(a.u, k, uv);
        loadN(a.delta, k, dv);
        const int le = k * kBwdTL + kSP * ej;
#pragma unroll
        for (int i = 0; i < kSP; ++i) {
            const float x = dv[i] + bias;
            float dt = x, sg = 1.f;
            if (SOFTPLUS) {
                dt = softplus_f(x);
                if (full) sg = rcp_approx(1.f + ex2_approx(-x * kLog2e));  // softplus'(x) = sigmoid(x)
            }
            if (le + i >= L) dt = 0.f;   // padding steps leave the state unchanged
            sm.W[ec][kSP * ej + i] = make_float2(dt, ZOH ? uv[i] : dt * uv[i]);
            if (full) {
                sm.SG[ec][kSP * ej + i] = sg;
                if (!ZOH) sm.U[ec][kSP * ej + i] = uv[i];
            }
        }
    };
    auto store_h = [&](float* base, size_t extent, float* p, const float2 (&v)[H]) {
        if (!in_bounds(a.err, base, extent, p, kS)) return;
#pragma unroll
        for (int q = 0; q < kS / 4; ++q)
            reinterpret_cast<float4*>(p)[q] = make_float4(v[2 * q].x, v[2 * q].y, v[2 * q + 1].x, v[2 * q + 1].y);
    };
    auto load_h = [&](const float* base, size_t extent, const float* p, float2 (&v)[H]) {
        const bool ok = in_bounds(a.err, base, extent, p, kS);
#pragma unroll
        for (int q = 0; q < kS / 4; ++q) {
            const float4 t = ok ? reinterpret_cast<const float4*>(p)[q] : make_float4(0.f, 0.f, 0.f, 0.f);
            v[2 * q] = make_float2(t.x, t.y);
            v[2 * q + 1] = make_float2(t.z, t.w);
        }
    };

    // ---------------------------------------------------- sweep 1: forward ----
    float2 h[H];
    if (a.h0) {
        load_h(a.h0, nrows * NS, a.h0 + rrow * NS + kS * rh, h);
    } else {
#pragma unroll
        for (int i = 0; i < H; ++i) h[i] = make_float2(0.f, 0.f);
    }
#pragma unroll 1
    for (int k = 0; k < (a.have_hck ? 0 : n); ++k) {
        prepass(k, false);
        stage_bc(k);
        __syncwarp();
        if (ractive) store_h(a.hck, nrows * n * NS, hck + static_cast<size_t>(k) * NS, h);
#pragma unroll
        for (int t = 0; t < kBwdTL; ++t) {
            const float2 w = sm.W[rc][t];
            float2 Bv[H];
            loadBC(t, 0, Bv);
            const float2 dd = make_float2(w.x, w.x), du = make_float2(w.y, w.y);
#pragma unroll
            for (int j = 0; j < H; ++j) {
                const float2 x2 = __fmul2_rn(dd, A2[j]);
                const float2 e = ex2_pair(x2);
                h[j] = __ffma2_rn(e, h[j], input_term(x2, e, dd, du, Bv[j], j));
            }
        }
        __syncwarp();
    }

    // ---------------------------------------------------- sweep 2: reverse ----
    float2 g[H], dAacc[H];
#pragma unroll
    for (int i = 0; i < H; ++i) { g[i] = make_float2(0.f, 0.f); dAacc[i] = make_float2(0.f, 0.f); }
    float dDacc = 0.f, dbacc = 0.f;
#pragma unroll 1
    for (int k = n - 1; k >= 0; --k) {
        const int l0 = k * kBwdTL;
        const int le = l0 + kSP * ej;  // first step of the pre-pass lane's kSP
        // the chunk's checkpoint (issued first: its latency overlaps the pre-pass)
        float2 hs[H];
        load_h(a.hck, nrows * n * NS, hck + static_cast<size_t>(k) * NS, hs);
        // (i) dt, its second operand, d(dt)/dx and u per (channel, step), into shared memory
        prepass(k, true);
        stage_bc(k);
        __syncwarp();

        // (ii) the chunk's states, recomputed from its checkpoint, and C.h
        {
            float2 hc[H];
#pragma unroll
            for (int j = 0; j < H; ++j) hc[j] = hs[j];
            float* Pw = &sm.P[rh][0][4 * rc];
#pragma unroll 1
            for (int t0 = 0; t0 < kBwdTL; t0 += 4) {
                float p[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int t = t0 + i;
                    const float2 w = sm.W[rc][t];
                    float2 Bv[H], Cv[H];
                    loadBC(t, 0, Bv);
                    loadBC(t, NS, Cv);
                    const float2 dd = make_float2(w.x, w.x), du = make_float2(w.y, w.y);
#pragma unroll
                    for (int j = 0; j < H; ++j) {
                        const float2 x2 = __fmul2_rn(dd, A2[j]);
                        const float2 e = ex2_pair(x2);
                        hc[j] = __ffma2_rn(e, hc[j], input_term(x2, e, dd, du, Bv[j], j));
                    }
#pragma unroll
                    for (int q = 0; q < kS / 4; ++q)
                        sm.traj[t][q][lane] = make_float4(hc[2 * q].x, hc[2 * q].y, hc[2 * q + 1].x, hc[2 * q + 1].y);
                    float2 acc = __fmul2_rn(Cv[0], hc[0]);
#pragma unroll
                    for (int j = 1; j < H; ++j) acc = __ffma2_rn(Cv[j], hc[j], acc);
                    p[i] = acc.x + acc.y;
                }
                *reinterpret_cast<float4*>(Pw + (t0 / 4) * kPJ) = make_float4(p[0], p[1], p[2], p[3]);
            }
        }
        __syncwarp();

        // (iii) dp = dy * silu(z) and dz = dy * (C.h + D u) * silu'(z)
        {
            float gy[kSP], zv[kSP], pre[kSP];
            loadN(a.dy, k, gy);
            if (HAS_Z) loadN(a.z, k, zv);
            if constexpr (kSP >= 4) {
#pragma unroll
                for (int gq = 0; gq < kSP / 4; ++gq) {
                    const int grp = (kSP / 4) * ej + gq;
                    float4 s = *reinterpret_cast<const float4*>(&sm.P[0][grp][4 * ec]);
#pragma unroll
                    for (int r = 1; r < kG; ++r) {
                        const float4 x = *reinterpret_cast<const float4*>(&sm.P[r][grp][4 * ec]);
                        s.x += x.x; s.y += x.y; s.z += x.z; s.w += x.w;
                    }
                    pre[4 * gq] = s.x; pre[4 * gq + 1] = s.y; pre[4 * gq + 2] = s.z; pre[4 * gq + 3] = s.w;
                }
            } else {  // two steps: half of a 4-step group
                const int grp = ej / 2, off = 2 * (ej % 2);
                float2 s = *reinterpret_cast<const float2*>(&sm.P[0][grp][4 * ec + off]);
#pragma unroll
                for (int r = 1; r < kG; ++r) {
                    const float2 x = *reinterpret_cast<const float2*>(&sm.P[r][grp][4 * ec + off]);
                    s.x += x.x; s.y += x.y;
                }
                pre[0] = s.x; pre[1] = s.y;
            }
            float dzv[kSP];
#pragma unroll
            for (int i = 0; i < kSP; ++i) {
                const float uu = u_at(ec, kSP * ej + i);
                const float p = fmaf(Dd, uu, pre[i]);
                float dp = gy[i];
                if (HAS_Z) {
                    const float s = rcp_approx(1.f + ex2_approx(-zv[i] * kLog2e));
                    dzv[i] = gy[i] * p * s * fmaf(zv[i], 1.f - s, 1.f);
                    dp = gy[i] * zv[i] * s;
                }
                dDacc = fmaf(dp, uu, dDacc);
                sm.DP[ec][kSP * ej + i] = dp;
            }
            if (HAS_Z) {
                T* dzp = static_cast<T*>(a.dz) + erow * L + le;
                const bool vec = vec_ok && le + kSP <= L;
                if (eactive && le < L && in_bounds(a.err, static_cast<T*>(a.dz), nx, dzp, vec ? kSP : min(L - le, kSP)))
                    stg_n<kSP>(dzp, dzv, vec, L - le);
            }
        }
        __syncwarp();

        // (iv) the reverse recurrence over the chunk's 16 steps; this lane's
        // dB/dC columns (channel sums) go to the fp32 sums 4 steps at a time
#pragma unroll 1
        for (int t0 = kBwdTL - 4; t0 >= 0; t0 -= 4) {
          float accBC[kCPL][4];
#pragma unroll
          for (int ti = 3; ti >= 0; --ti) {
            const int t = t0 + ti;
            const float2 w = sm.W[rc][t];
            const float dp = sm.DP[rc][t];
            float2 Bv[H], Cv[H], hT[H], hP[H];
            loadBC(t, 0, Bv);
            loadBC(t, NS, Cv);
#pragma unroll
            for (int q = 0; q < kS / 4; ++q) {
                const float4 v = sm.traj[t][q][lane];
                hT[2 * q] = make_float2(v.x, v.y);
                hT[2 * q + 1] = make_float2(v.z, v.w);
            }
            if (t > 0) {
#pragma unroll
                for (int q = 0; q < kS / 4; ++q) {
                    const float4 v = sm.traj[t - 1][q][lane];
                    hP[2 * q] = make_float2(v.x, v.y);
                    hP[2 * q + 1] = make_float2(v.z, v.w);
                }
            } else {
#pragma unroll
                for (int j = 0; j < H; ++j) hP[j] = hs[j];
            }
            const float2 dd = make_float2(w.x, w.x), du = make_float2(w.y, w.y), dpp = make_float2(dp, dp);
            float2 sa = make_float2(0.f, 0.f), sb = make_float2(0.f, 0.f), sc = make_float2(0.f, 0.f);
            float2 dBv[H], dCv[H];
#pragma unroll
            for (int j = 0; j < H; ++j) {
                const float2 x2 = __fmul2_rn(dd, A2[j]);
                const float2 e = ex2_pair(x2);
                const float2 gh = __ffma2_rn(dpp, Cv[j], g[j]);
                dCv[j] = __fmul2_rn(dpp, hT[j]);
                if (ZOH) {  // du holds u
                    const float2 gain = zoh_gain2(x2, e, dd, IA(j));
                    const float2 ghB = __fmul2_rn(gh, Bv[j]);
                    dBv[j] = __fmul2_rn(__fmul2_rn(gh, gain), du);
                    sa = __ffma2_rn(ghB, gain, sa);
                    sc = __ffma2_rn(ghB, e, sc);
                    const float2 dee = __fmul2_rn(__fmul2_rn(gh, hP[j]), e);
                    sb = __ffma2_rn(dee, A2[j], sb);
                    float2* da = &dA_zoh[ZOH ? j : 0][lane];
                    sts2_pinned(da, __ffma2_rn(__fmul2_rn(ghB, du), zoh_dgain_da2(x2, e, gain, dd, IA(j)),
                                               __ffma2_rn(dee, dd, lds2_pinned(da))));
                } else {    // du holds dt*u
                    dBv[j] = __fmul2_rn(gh, du);
                    sa = __ffma2_rn(gh, Bv[j], sa);
                    const float2 dee = __fmul2_rn(__fmul2_rn(gh, hP[j]), e);
                    sb = __ffma2_rn(dee, A2[j], sb);
                    dAacc[j] = __ffma2_rn(dee, dd, dAacc[j]);
                }
                g[j] = __fmul2_rn(gh, e);
            }
            {   // all state groups of the channel: lanes rc + kCh * m
                float qa = sa.x + sa.y, qb = sb.x + sb.y, qc = sc.x + sc.y;
#pragma unroll
                for (int o = kCh; o < 32; o <<= 1) {
                    qa += __shfl_xor_sync(0xffffffffu, qa, o);
                    qb += __shfl_xor_sync(0xffffffffu, qb, o);
                    if (ZOH) qc += __shfl_xor_sync(0xffffffffu, qc, o);
                }
                // with ZOH the term sum_n gh B u e (d gain / d dt = e) completes d(dt) here
                if (rh == 0) sm.Q[rc][t] = make_float2(qa, ZOH ? fmaf(qc, u_at(rc, t), qb * kLn2) : qb * kLn2);
            }
            // channel sums of this step's dB and dC
#pragma unroll
            for (int q = 0; q < kS / 4; ++q) {
                reinterpret_cast<float4*>(&sm.RB[rc][kS * rh])[q] =
                    make_float4(dBv[2 * q].x, dBv[2 * q].y, dBv[2 * q + 1].x, dBv[2 * q + 1].y);
                reinterpret_cast<float4*>(&sm.RB[rc][NS + kS * rh])[q] =
                    make_float4(dCv[2 * q].x, dCv[2 * q].y, dCv[2 * q + 1].x, dCv[2 * q + 1].y);
            }
            __syncwarp();
#pragma unroll
            for (int c = 0; c < kCPL; ++c) {
                const int col = lane + 32 * c;
                float2 sacc = make_float2(0.f, 0.f);
                if (col < kCols) {
#pragma unroll
                    for (int ch = 0; ch < kCh; ch += 2)
                        sacc = __fadd2_rn(sacc, make_float2(sm.RB[ch][col], sm.RB[ch + 1][col]));
                }
                accBC[c][ti] = sacc.x + sacc.y;
            }
            __syncwarp();
          }
#pragma unroll
          for (int c = 0; c < kCPL; ++c) {
              const int col = lane + 32 * c;
              if (col < kCols) {
                  float* dcol = a.dbc + ((static_cast<size_t>(b) * 2 + col / NS) * NS + col % NS) * a.Lp + l0;
                  if (in_bounds(a.err, a.dbc, npk * kCols, dcol + t0, 4))
                      red_add4(dcol + t0, make_float4(accBC[c][0], accBC[c][1], accBC[c][2], accBC[c][3]));
              }
          }
        }

        // (v) du and ddelta per (channel, step)
        {
            float duv[kSP], dxv[kSP];
#pragma unroll
            for (int i = 0; i < kSP; ++i) {
                const int t = kSP * ej + i;
                const float2 q = sm.Q[ec][t];
                const float dsum = ZOH ? q.x : q.x * sm.W[ec][t].x;      // sum_n gh B gain
                const float sdt = ZOH ? q.y : fmaf(q.x, u_at(ec, t), q.y);  // d(dt)
                duv[i] = fmaf(sm.DP[ec][t], Dd, dsum);
                dxv[i] = le + i < L ? sdt * sm.SG[ec][t] : 0.f;
                dbacc += dxv[i];
            }
            if (eactive && le < L) {
                const bool vec = vec_ok && le + kSP <= L;
                T* dup = static_cast<T*>(a.du) + erow * L + le;
                T* ddp = static_cast<T*>(a.ddelta) + erow * L + le;
                if (in_bounds(a.err, static_cast<T*>(a.du), nx, dup, vec ? kSP : min(L - le, kSP)))
                    stg_n<kSP>(dup, duv, vec, L - le);
                if (in_bounds(a.err, static_cast<T*>(a.ddelta), nx, ddp, vec ? kSP : min(L - le, kSP)))
                    stg_n<kSP>(ddp, dxv, vec, L - le);
            }
        }
        __syncwarp();
    }

    // the gradient of the initial state, dA, dD and the bias's gradient
    if (a.dh0 && ractive) store_h(a.dh0, nrows * NS, a.dh0 + rrow * NS + kS * rh, g);
    if (ractive && in_bounds(a.err, a.dA, static_cast<size_t>(a.dim) * NS, a.dA + static_cast<size_t>(rd) * NS + kS * rh,
                             kS)) {
        float* p = a.dA + static_cast<size_t>(rd) * NS + kS * rh;
#pragma unroll
        for (int j = 0; j < H; ++j) {
            const float2 v = ZOH ? lds2_pinned(&dA_zoh[ZOH ? j : 0][lane]) : dAacc[j];
            atomicAdd(p + 2 * j, v.x);
            atomicAdd(p + 2 * j + 1, v.y);
        }
    }
#pragma unroll
    for (int o = 1; o < kG; o <<= 1) {   // the kG pre-pass lanes of a channel
        dDacc += __shfl_xor_sync(0xffffffffu, dDacc, o);
        dbacc += __shfl_xor_sync(0xffffffffu, dbacc, o);
    }
    if (eactive && ej == 0) {
        if (a.dD && in_bounds(a.err, a.dD, a.dim, a.dD + ed)) atomicAdd(a.dD + ed, dDacc);
        if (a.dbias && in_bounds(a.err, a.dbias, a.dim, a.dbias + ed)) atomicAdd(a.dbias + ed, dbacc);
    }
}

// dB and dC in the I/O dtype from the fp32 sums: out[b][n][l] = dbc[b][which][n][l].
template <typename T>
__global__ void __launch_bounds__(256)
dbc_unpack_kernel(const float* __restrict__ dbc, T* __restrict__ dB, T* __restrict__ dC, int batch, int ns, int L,
                  int Lp, int* err) {
    const long long total = static_cast<long long>(batch) * 2 * ns * L;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int l = static_cast<int>(i % L);
        const long long r = i / L;  // (b, which, n)
        const int nn = static_cast<int>(r % ns);
        const int which = static_cast<int>((r / ns) % 2);
        const int bb = static_cast<int>(r / (2 * ns));
        const size_t nout = static_cast<size_t>(batch) * ns * L;
        if (!in_bounds(err, dbc, static_cast<size_t>(batch) * 2 * ns * Lp, dbc + r * Lp + l)) continue;
        const float v = dbc[r * Lp + l];
        T* out = which ? dC : dB;
        T* o = out + (static_cast<size_t>(bb) * ns + nn) * L + l;
        if (in_bounds(err, out, nout, o)) *o = Io<T>::from_f(v);
    }
}

}  // namespace mscan
