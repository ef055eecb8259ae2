// State-space dual (SSD) layer, chunked form on the tensor cores, sm_103a.
//
// The Mamba-2 form of the selective SSM ("Mamba 论文精读", youngju.dev, §4.1:
// the recurrence h_t = A_t h_{t-1} + B_t x_t, y_t = C_t h_t is dual to the
// masked product Y = (T o M) X with M semiseparable; §5.2: multi-head,
// headdim 64, larger states). Per batch row b and head h the state S is a
// (64 x N) matrix, the decay a_t = exp(dt_t A_h) one scalar per step:
//     S_t = a_t S_{t-1} + dt_t x_t B_t^T,   y_t = S_t C_t + D_h x_t.
// Over a chunk of Q = 64 steps with c_l = sum_{r<=l} dt_r A_h (inclusive):
//     y_l = sum_{s<=l} (C_l . B_s) e^{c_l - c_s} dt_s x_s        (intra-chunk)
//         + e^{c_l} S_prev C_l                                    (carried state)
//         + D_h x_l
//     S_new = e^{c_Q} S_prev + sum_s x_s (e^{c_Q - c_s} dt_s) B_s^T.
// The four contractions (C B^T, its masked product with X, the state update
// and C S^T) run on the tensor cores: bf16 operands, fp32 accumulation.
// Three operands are not bf16 inputs but values computed in fp32 (the masked
// C B^T, the decay-weighted x and the carried state); each is split into a
// bf16 high part and a bf16 remainder and multiplied twice, which keeps them
// to ~2^-17 relative (one bf16 rounding of those operands alone costs up to
// 1e-2 relative error in y at N = 128, over the bf16 I/O tolerance).
//
// One CTA (8 warps) per (head, batch row) walks the chunks in order; the fp32
// state never leaves the registers (it is the state-update product's
// accumulator). Warp w owns row block w & 3 (16 rows: steps l of the outputs
// and of C B^T, channels p of the state) and column half w >> 2 of every
// per-chunk product, so that two CTAs (16 warps) fit on an SM and hide each
// other's latencies. The x, B and C tiles arrive by 3-D TMA (128-byte swizzled
// rows), each on its own barrier and refilled for the next chunk as soon as
// its last reader is done (C after C S^T and C B^T, x after the outputs, B
// after the state update); the operands the CTA writes itself use padded
// rows. Within each product the high-part MMAs of all column tiles are issued
// before the low-part ones, so no two consecutive MMAs share an accumulator.
// Steps past the end of the sequence get dt = 0, so they leave the state
// unchanged.
#pragma once

#include "common.cuh"

namespace mscan {

constexpr int kSsdQ = 64;         // chunk length
constexpr int kSsdP = 64;         // head dimension
constexpr int kSsdThreads = 256;  // 8 warps
constexpr int kSsdPad = 8;        // row padding (bf16) of the operands written in shared memory

struct SsdArgs {
    const void* delta;   // (batch, nheads, L) bf16
    const float* A;      // (nheads)
    const float* D;      // (nheads) or null
    const float* bias;   // (nheads) or null
    const float* h0;     // (batch, nheads, 64, N) or null
    void* y;             // (batch, nheads * 64, L) bf16
    float* final_state;  // (batch, nheads, 64, N) or null
    int* err;            // device error word
    int batch, nheads, seqlen;
    int softplus;
};

template <int NS>
struct SsdSmem {
    // TMA tiles: rows of 64 bf16 (128 bytes), 128-byte swizzle
    alignas(1024) __nv_bfloat16 X[kSsdP][kSsdQ];   // x   [p][s]
    alignas(1024) __nv_bfloat16 Bt[NS][kSsdQ];     // B   [n][s]
    alignas(1024) __nv_bfloat16 Ct[NS][kSsdQ];     // C   [n][l]
    // operands computed here, high and low bf16 parts: the masked C B^T [l][s]
    // until its product with x is done, then the decay-weighted x [p][s]
    alignas(16) __nv_bfloat16 Oh[kSsdQ][kSsdQ + kSsdPad], Ol[kSsdQ][kSsdQ + kSsdPad];
    alignas(16) __nv_bfloat16 Sh[kSsdP][NS + kSsdPad], Sl[kSsdP][NS + kSsdPad];  // state [p][n]
    alignas(16) float Yt[kSsdP][kSsdQ + 4];  // the chunk's outputs [p][l], for row-contiguous stores
    float c2[2][kSsdQ];                      // c_l * log2(e), chunk k in [k & 1]
    float dt[2][kSsdQ];
    alignas(8) uint64_t full[3];             // x, B, C tiles
};
static_assert(kSsdQ == kSsdP, "the O buffers hold both Q x Q and P x Q operands");

// ------------------------------------------------------------ helpers ------

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t (&r)[2]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}
// D += A B, A 16x16 (row), B 16x8 (col), bf16 operands, fp32 accumulators
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Element (row, col) of a tile of 128-byte rows written by TMA with the
// 128-byte swizzle (16-byte unit u of row r stored at unit u ^ (r & 7); tile
// base 1024-aligned).
__device__ __forceinline__ float swz_ld(const __nv_bfloat16* tile, int row, int col) {
    const unsigned char* p = reinterpret_cast<const unsigned char*>(tile) + row * 128 +
                             ((((col >> 3) ^ (row & 7)) << 4) | ((col & 7) << 1));
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
}
// v as a bf16 pair hi + lo: hi = bf16(v), lo = bf16(v - hi).
__device__ __forceinline__ void split2(float v0, float v1, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(v0 - hf.x, v1 - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}


// ------------------------------------------------------------- kernel ------

template <int NS>
__global__ void __launch_bounds__(kSsdThreads, 2)
ssd_fwd_kernel(const SsdArgs a, const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
               const __grid_constant__ CUtensorMap tm_c) {
    extern __shared__ unsigned char ssd_smem_raw[];
    // 1024-byte aligned view of the dynamic shared memory, derived from the
    // shared array itself so that every access stays a shared-memory access
    SsdSmem<NS>& sm = *reinterpret_cast<SsdSmem<NS>*>(ssd_smem_raw + ((1024u - (smem_u32(ssd_smem_raw) & 1023u)) & 1023u));
    constexpr int kNH = NS / 16;  // 8-column state tiles of a warp (half of the state)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, tq = lane & 3;      // accumulator row group / column pair
    const int mi = lane >> 3, rr = lane & 7;     // ldmatrix: which 8x8 matrix, which row of it
    const int rb = warp & 3, chalf = warp >> 2;
    const int m0 = 16 * rb;                      // this warp's rows
    const int c0 = 32 * chalf;                   // its half of the 64 columns (channels p, or steps s of C B^T)
    const int n0 = chalf * (NS / 2);             // its half of the state columns
    const int h = blockIdx.x, b = blockIdx.y;
    const int L = a.seqlen;
    const int n = (L + kSsdQ - 1) / kSsdQ;
    const int dim = a.nheads * kSsdP;
    const int ch0 = h * kSsdP;                   // first channel of the head
    const float Ah2 = a.A[h] * kLog2e;
    const float bias = a.bias ? a.bias[h] : 0.f;
    const float Dh = a.D ? a.D[h] : 0.f;
    const size_t head_row = static_cast<size_t>(b) * a.nheads + h;

    // tile loads of chunk k (thread 0): barrier 0 = x, 1 = B, 2 = C; parity k & 1
    int last[3] = {-1, -1, -1};
    auto issue = [&](int which, int k) {
        uint64_t* bar = &sm.full[which];
        const int l0 = k * kSsdQ;
        if (which == 0) {
            mbar_arrive_expect_tx(bar, kSsdP * kSsdQ * 2);
            tma_load_3d(&sm.X[0][0], &tm_x, bar, l0, ch0, b);
        } else {
            mbar_arrive_expect_tx(bar, NS * kSsdQ * 2);
            tma_load_3d(which == 1 ? &sm.Bt[0][0] : &sm.Ct[0][0], which == 1 ? &tm_b : &tm_c, bar, l0, 0, b);
        }
        last[which] = k;
    };
    // after a timeout: wait (bounded) for this thread's copies still in flight
    auto drain = [&]() {
        for (int i = 0; i < 3; ++i)
            if (last[i] >= 0) mbar_wait_bounded(&sm.full[i], static_cast<uint32_t>(last[i] & 1));
    };
    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&sm.full[i], 1);
        fence_barrier_init();
        if (n > 0) { issue(2, 0); issue(1, 0); issue(0, 0); }
    }

    // The state: rows m0 + g (+8), columns n0 + 8j + 2tq (+1).
    float S[kNH][4];
    const bool have_state = a.h0 != nullptr;
#pragma unroll
    for (int j = 0; j < kNH; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int p = m0 + g + 8 * (e >> 1), c = n0 + 8 * j + 2 * tq + (e & 1);
            S[j][e] = have_state ? a.h0[(head_row * kSsdP + p) * NS + c] : 0.f;
        }
    }
    auto store_state_parts = [&]() {
#pragma unroll
        for (int j = 0; j < kNH; ++j) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t hi, lo;
                split2(S[j][2 * hf], S[j][2 * hf + 1], hi, lo);
                const int p = m0 + g + 8 * hf, c = n0 + 8 * j + 2 * tq;
                *reinterpret_cast<uint32_t*>(&sm.Sh[p][c]) = hi;
                *reinterpret_cast<uint32_t*>(&sm.Sl[p][c]) = lo;
            }
        }
    };
    if (have_state) store_state_parts();
    __syncthreads();

    const __nv_bfloat16* dl = static_cast<const __nv_bfloat16*>(a.delta) + head_row * L;
    __nv_bfloat16* yb = static_cast<__nv_bfloat16*>(a.y) + (static_cast<size_t>(b) * dim + ch0) * L;
    const bool vec_ok = (L & 7) == 0;
    const uint32_t xt = smem_u32(&sm.X[0][0]);
    const uint32_t bt = smem_u32(&sm.Bt[0][0]);
    const uint32_t ct = smem_u32(&sm.Ct[0][0]);
    // Loop-invariant parts of the ldmatrix addresses. Rows of the swizzled
    // tiles advance in steps of 8, so their swizzle term (row & 7) is fixed.
    const int ra = rr + ((mi >> 1) << 3);        // row of this lane in matrices ordered (row, row, row+8, row+8)
    const int rc = rr + ((mi & 1) << 3);         // ... ordered (row, row+8, row, row+8)
    // Outputs (C S^T, the masked product, y): two row blocks of equal causal
    // work, {0, 3} or {1, 2}, and one quarter (16) of the head's channels.
    const int yrb[2] = {(warp & 1) ? 1 : 0, (warp & 1) ? 2 : 3};
    const int pq = warp >> 1;
    uint32_t a_y[2];                             // C^T rows of the two output row blocks, at k0 = 0
#pragma unroll
    for (int r = 0; r < 2; ++r) a_y[r] = ct + ra * 128 + (((2 * yrb[r] + (mi & 1)) ^ (ra & 7)) << 4);
    const uint32_t x_q = xt + (16 * pq + ra) * 128;  // X rows of the channel quarter
    const int sw = ra & 7;
    // C B^T: the 20 (row block, column block, 8-column half) units of the causal
    // triangle, dealt round-robin: units warp, warp + 8, warp + 16
    const int krow = (lane & 7) + 8 * ((lane >> 3) & 1);  // ldmatrix.x2 row of this lane
    const uint32_t b_row = bt + (n0 + ra) * 128;  // Bt rows n0 + ra (+16 jp)

    // dt and the cumulative decay of chunk k into buffer k & 1 (warp 0);
    // padding steps get dt = 0
    auto decay_prefix = [&](int k) {
        float v[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int l = 2 * lane + i, gl = k * kSsdQ + l;
            float d = 0.f;
            if (gl < L) {
                d = __bfloat162float(dl[gl]) + bias;
                if (a.softplus) d = softplus_f(d);
            }
            sm.dt[k & 1][l] = d;
            v[i] = d * Ah2;
        }
        const float pair = v[0] + v[1];
        float incl = pair;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        const float excl = incl - pair;
        sm.c2[k & 1][2 * lane] = excl + v[0];
        sm.c2[k & 1][2 * lane + 1] = excl + pair;
    };
    if (warp == 0 && n > 0) decay_prefix(0);
    __syncthreads();

    // A wait that runs out sets `timed_out`; the chunk is finished with
    // whatever the tiles hold and the kernel leaves at the chunk's last
    // barrier, so that no thread is ever left waiting at a barrier.
    bool timed_out = false;
#pragma unroll 1
    for (int k = 0; k < n; ++k) {
        const uint32_t par = static_cast<uint32_t>(k & 1);
        const float* c2 = sm.c2[k & 1];
        const float* dtv = sm.dt[k & 1];
        if (!mbar_wait_bounded(&sm.full[2], par)) timed_out = true;  // C

        // --- C S^T (carried state) for this warp's two row blocks and channel quarter ---
        float Y[2][2][4];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) Y[r][j][e] = 0.f;
        const bool carry = have_state || k > 0;
        if (carry) {
#pragma unroll
            for (int k0 = 0; k0 < NS; k0 += 16) {
                uint32_t af[2][4], bh[4], bl[4];  // A = C^T rows from Ct[n][l]; B = S^T from Sh/Sl[p][n]
                ldsm_x4_t(a_y[0] + k0 * 128, af[0]);
                ldsm_x4_t(a_y[1] + k0 * 128, af[1]);
                ldsm_x4(smem_u32(&sm.Sh[16 * pq + ra][k0 + 8 * (mi & 1)]), bh);
                ldsm_x4(smem_u32(&sm.Sl[16 * pq + ra][k0 + 8 * (mi & 1)]), bl);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    mma_bf16(Y[r][0], af[r], bh[0], bh[1]);
                    mma_bf16(Y[r][1], af[r], bh[2], bh[3]);
                }
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    mma_bf16(Y[r][0], af[r], bl[0], bl[1]);
                    mma_bf16(Y[r][1], af[r], bl[2], bl[3]);
                }
            }
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const float e0 = ex2_approx(c2[16 * yrb[r] + g]), e1 = ex2_approx(c2[16 * yrb[r] + g + 8]);
#pragma unroll
                for (int j = 0; j < 2; ++j) { Y[r][j][0] *= e0; Y[r][j][1] *= e0; Y[r][j][2] *= e1; Y[r][j][3] *= e1; }
            }
        }
        if (!mbar_wait_bounded(&sm.full[1], par)) timed_out = true;  // B
        // --- C B^T over this warp's units of the causal triangle, masked and weighted ---
        {
            float G[3][4];
            int urb[3], ucol[3];  // row block and first column of each unit
#pragma unroll
            for (int i = 0; i < 3; ++i) {
                // unit u -> (row block, column block, half): u = rb (rb + 1) + 2 sb + nt
                const int u = warp + 8 * i;
                const int rbu = u < 2 ? 0 : (u < 6 ? 1 : (u < 12 ? 2 : 3));
                const int rem = u - rbu * (rbu + 1);
                urb[i] = rbu;
                ucol[i] = 8 * rem;            // 16 sb + 8 nt
#pragma unroll
                for (int e = 0; e < 4; ++e) G[i][e] = 0.f;
            }
#pragma unroll
            for (int k0 = 0; k0 < NS; k0 += 16) {
#pragma unroll
                for (int i = 0; i < 3; ++i) {
                    if (warp + 8 * i < 20) {
                        uint32_t af[4], bf[2];
                        ldsm_x4_t(ct + (k0 + ra) * 128 + (((2 * urb[i] + (mi & 1)) ^ (ra & 7)) << 4), af);
                        ldsm_x2_t(bt + (k0 + krow) * 128 + (((ucol[i] >> 3) ^ (krow & 7)) << 4), bf);
                        mma_bf16(G[i], af, bf[0], bf[1]);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 3; ++i) {
                if (warp + 8 * i < 20) {
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int l = 16 * urb[i] + g + 8 * hf;
                        const float cl = c2[l];
                        float v[2];
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            const int sc = ucol[i] + 2 * tq + c;
                            v[c] = sc <= l ? G[i][2 * hf + c] * ex2_approx(cl - c2[sc]) * dtv[sc] : 0.f;
                        }
                        uint32_t hi, lo;
                        split2(v[0], v[1], hi, lo);
                        *reinterpret_cast<uint32_t*>(&sm.Oh[l][ucol[i] + 2 * tq]) = hi;
                        *reinterpret_cast<uint32_t*>(&sm.Ol[l][ucol[i] + 2 * tq]) = lo;
                    }
                }
            }
        }
        __syncthreads();  // every unit of the triangle is in; C is consumed
        if (tid == 0 && k + 1 < n && !timed_out) {  // (never refill a tile whose load may be in flight)
            fence_proxy_async_smem();
            issue(2, k + 1);
        }
        if (!mbar_wait_bounded(&sm.full[0], par)) timed_out = true;  // x
        // --- Y += (masked C B^T) X^T over s < 16 (row block + 1) ---
#pragma unroll
        for (int r = 0; r < 2; ++r) {
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
                if (kb <= yrb[r]) {
                    uint32_t ah[4], al[4], bx[4];
                    const int arow = 16 * yrb[r] + rc, acol = 16 * kb + 8 * (mi >> 1);
                    ldsm_x4(smem_u32(&sm.Oh[arow][acol]), ah);
                    ldsm_x4(smem_u32(&sm.Ol[arow][acol]), al);
                    ldsm_x4(x_q + (((2 * kb + (mi & 1)) ^ sw) << 4), bx);  // B = X^T from X[p][s]
                    mma_bf16(Y[r][0], ah, bx[0], bx[1]);
                    mma_bf16(Y[r][1], ah, bx[2], bx[3]);
                    mma_bf16(Y[r][0], al, bx[0], bx[1]);
                    mma_bf16(Y[r][1], al, bx[2], bx[3]);
                }
            }
        }
        __syncthreads();  // every warp is done with the masked rows: the O buffers take the weighted x
        // --- outputs (+ D x) into Yt; decay-weighted x into the O buffers ---
#pragma unroll
        for (int r = 0; r < 2; ++r) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int l = 16 * yrb[r] + g + 8 * (e >> 1), p = 16 * pq + 8 * j + 2 * tq + (e & 1);
                    sm.Yt[p][l] = Y[r][j][e] + Dh * swz_ld(&sm.X[0][0], p, l);
                }
            }
        }
        const float clast = c2[kSsdQ - 1];
        {
            const int p = m0 + (lane >> 1);
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                const int sc = c0 + 16 * (lane & 1) + i;
                const float w0 = ex2_approx(clast - c2[sc]) * dtv[sc];
                const float w1 = ex2_approx(clast - c2[sc + 1]) * dtv[sc + 1];
                uint32_t hi, lo;
                split2(swz_ld(&sm.X[0][0], p, sc) * w0, swz_ld(&sm.X[0][0], p, sc + 1) * w1, hi, lo);
                *reinterpret_cast<uint32_t*>(&sm.Oh[p][sc]) = hi;
                *reinterpret_cast<uint32_t*>(&sm.Ol[p][sc]) = lo;
            }
        }
        __syncthreads();  // Yt and the weighted x complete; x is consumed
        if (tid == 0 && k + 1 < n && !timed_out) {  // (never refill a tile whose load may be in flight)
            fence_proxy_async_smem();
            issue(0, k + 1);
        }
        if (warp == 0 && k + 1 < n) decay_prefix(k + 1);  // the next chunk's dt and decay, other buffer
        // y rows of the head's 64 channels, 8 steps per store
#pragma unroll
        for (int v = tid; v < kSsdP * (kSsdQ / 8); v += kSsdThreads) {
            const int p = v >> 3, lc = (v & 7) * 8, gl = k * kSsdQ + lc;
            if (gl >= L) continue;
            __nv_bfloat16* dst = yb + static_cast<size_t>(p) * L + gl;
            const float* src = &sm.Yt[p][lc];
            if (vec_ok && gl + 8 <= L) {
                uint32_t w[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const __nv_bfloat162 o = __floats2bfloat162_rn(src[2 * q], src[2 * q + 1]);
                    w[q] = *reinterpret_cast<const uint32_t*>(&o);
                }
                *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
            } else {
                for (int q = 0; q < 8 && gl + q < L; ++q) dst[q] = __float2bfloat16_rn(src[q]);
            }
        }
        // --- state: S = e^{c_Q} S + (weighted x) B^T: rows m0.., this warp's state half ---
        const float ed = ex2_approx(clast);
#pragma unroll
        for (int j = 0; j < kNH; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) S[j][e] *= ed;
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
            uint32_t ah[4], al[4], bb[kNH / 2][4];
            const int arow = m0 + rr + ((mi & 1) << 3), acol = 16 * kb + 8 * (mi >> 1);
            ldsm_x4(smem_u32(&sm.Oh[arow][acol]), ah);
            ldsm_x4(smem_u32(&sm.Ol[arow][acol]), al);
#pragma unroll
            for (int jp = 0; jp < kNH / 2; ++jp)  // B = Bt^T from Bt[n][s]
                ldsm_x4(b_row + jp * 16 * 128 + (((2 * kb + (mi & 1)) ^ sw) << 4), bb[jp]);
#pragma unroll
            for (int jp = 0; jp < kNH / 2; ++jp) {
                mma_bf16(S[2 * jp], ah, bb[jp][0], bb[jp][1]);
                mma_bf16(S[2 * jp + 1], ah, bb[jp][2], bb[jp][3]);
            }
#pragma unroll
            for (int jp = 0; jp < kNH / 2; ++jp) {
                mma_bf16(S[2 * jp], al, bb[jp][0], bb[jp][1]);
                mma_bf16(S[2 * jp + 1], al, bb[jp][2], bb[jp][3]);
            }
        }
        store_state_parts();
        // state parts and the next chunk's decay complete; B is consumed
        if (__syncthreads_or(timed_out)) {
            if (tid == 0) { report_device_error(a.err, -6); drain(); }
            return;
        }
        if (tid == 0 && k + 1 < n && !timed_out) {  // (never refill a tile whose load may be in flight)
            fence_proxy_async_smem();
            issue(1, k + 1);
        }
    }

    if (a.final_state) {
#pragma unroll
        for (int j = 0; j < kNH; ++j) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int p = m0 + g + 8 * hf, c = n0 + 8 * j + 2 * tq;
                *reinterpret_cast<float2*>(a.final_state + (head_row * kSsdP + p) * NS + c) =
                    make_float2(S[j][2 * hf], S[j][2 * hf + 1]);
            }
        }
    }
}

}  // namespace mscan
