// State-space dual (SSD) layer, chunked form on the 5th-generation tensor cores, sm_103a.
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
// Four contractions per chunk, all `tcgen05.mma` (bf16 operands from shared
// memory, fp32 accumulators in tensor memory), issued by one thread:
//     G  = C^T B            M = 64 (l), N = 64 (s), K = N      -> TMEM cols   0..63
//     Y1 = C^T S_prev^T     M = 64 (l), N = 64 (p), K = N      -> TMEM cols  64..127
//     Y2 = Gm X^T           M = 64 (l), N = 64 (p), K = 64 (s) -> TMEM cols 128..191
//     U  = B W^T            M = N (n),  N = 64 (p), K = 64 (s) -> TMEM cols 192..255
// with Gm the causally masked, decay-weighted G and W the decay-weighted x
// (W[p][s] = x[p][s] e^{c_Q - c_s} dt_s). C and B are used straight from their
// TMA tiles ([n][l] rows): as MN-major operands where the contraction runs over
// n, as a K-major one (B in U) where it runs over s; the carried state is
// written in the same [n][p] form (16-byte row pieces). Three operands are not bf16
// inputs but values computed in fp32 (Gm, W and the carried state); each is
// split into a bf16 high part and a bf16 remainder and multiplied twice, which
// keeps them to ~2^-17 relative (one bf16 rounding of those operands alone
// costs up to 1e-2 relative error in y at N = 128, over the bf16 tolerance).
//
// One CTA (8 warps) per (head, batch row) walks the chunks in order; the fp32
// state stays in registers (a thread holds one state column n for 32 of the
// channels), updated from U as S = e^{c_Q} S + U and written back, split, as
// the next chunk's operand. Two CTAs share an SM (104 KB of shared memory and
// 256 TMEM columns each), so one's elementwise work overlaps the other's
// contractions and loads. At N = 256 (the Mamba-2 section's largest state) U
// is two M = 128 products and a CTA takes the SM (177 KB, 512 TMEM columns),
// each thread holding one state column for all 64 channels. Per chunk: one thread issues G and Y1 as soon as C and
// B are in; every thread forms W; barrier; it issues U while every
// thread forms Gm from G (tcgen05.ld, mask, decay weights, split), with D_h
// added on its diagonal so that Y2 = Gm X^T carries the skip term D x;
// barrier; it issues Y2 and reloads the B, C and x tiles for the next
// chunk as soon as the products reading them are done; every thread forms the
// outputs y = e^{c_l} Y1 + Y2 (staged in shared memory and stored, 16 bytes a
// row piece, at the start of the next chunk) and the new state; barrier. The
// tiles arrive by 3-D TMA (128-byte swizzle) on their own barriers, so their
// loads overlap the second half of the previous chunk. Steps past the end of the
// sequence get dt = 0, so they leave the state unchanged. Every wait is
// bounded: a wait that runs out is reported through the device error word,
// the chunk finishes and the kernel leaves with its tensor memory freed.
#pragma once

#include "common.cuh"

namespace mscan {

constexpr int kSsdQ = 64;          // chunk length
constexpr int kSsdP = 64;          // head dimension
constexpr int kSsdThreads = 256;   // 8 warps
constexpr int kSsdTmemCols = 256;  // G, Y1, Y2, U: 64 fp32 columns each
constexpr int kSsdYPitch = 72;     // row pitch (bf16) of the output staging tile

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

// All tiles are rows of 64 bf16 (128 bytes) in the 128-byte swizzle (16-byte
// unit u of row r stored at unit u ^ (r & 7), tiles 1024-aligned): the layout
// TMA writes and the tensor cores read.
template <int NS>
struct SsdSmem {
    alignas(1024) __nv_bfloat16 X[kSsdP][kSsdQ];   // x [p][s]            (TMA)
    alignas(1024) __nv_bfloat16 Bt[NS][kSsdQ];     // B [n][s]            (TMA)
    alignas(1024) __nv_bfloat16 Ct[NS][kSsdQ];     // C [n][l]            (TMA)
    // Gm [l][s] high and low parts; once the Y2 product is done, the staging
    // tile of the chunk's outputs y [p][l] (bf16, pitch kSsdYPitch)
    alignas(1024) __nv_bfloat16 Gh[kSsdQ][kSsdQ];
    alignas(1024) __nv_bfloat16 Gl[kSsdQ][kSsdQ];
    alignas(1024) __nv_bfloat16 Wh[kSsdP][kSsdQ];  // W [p][s], high part
    alignas(1024) __nv_bfloat16 Wl[kSsdP][kSsdQ];  //           low part
    alignas(1024) __nv_bfloat16 Sh[NS][kSsdP];     // carried state [n][p], high part
    alignas(1024) __nv_bfloat16 Sl[NS][kSsdP];     //                       low part
    alignas(16) float c2[2][kSsdQ];  // c_l * log2(e), chunk k in [k & 1]
    alignas(16) float dt[2][kSsdQ];
    alignas(16) float wq[2][kSsdQ + 8];  // e^{c_Q - c_s} dt_s at wq_at(s): 4 floats of padding after
                                         // each 32 steps keep the W phase's 16-byte reads of steps
                                         // 8u.. (u = 0, 2, 4, 6 in one quarter-warp) in distinct banks
    alignas(8) uint64_t full[3];     // TMA: x, B, C
    alignas(8) uint64_t done[4];     // MMA completion: G, Y1, U, Y2 (each also covers the earlier ones)
    uint32_t tmem;                   // base address of this CTA's tensor memory
};
static_assert(kSsdP * kSsdYPitch * 2 <= 2 * kSsdQ * kSsdQ * 2, "the y staging tile fits in the Gm buffers");

// ------------------------------------------------------------ helpers ------

// Index of step s in the padded decay-weight row (SsdSmem::wq).
__device__ __forceinline__ int wq_at(int s) { return s + ((s >> 5) << 2); }

// Byte offset of element (row, col) in a swizzled tile of 128-byte rows.
__device__ __forceinline__ int swz(int row, int col) {
    return row * 128 + ((((col >> 3) ^ (row & 7))) << 4) + ((col & 7) << 1);
}
__device__ __forceinline__ float swz_ld(const __nv_bfloat16* tile, int row, int col) {
    return __bfloat162float(
        *reinterpret_cast<const __nv_bfloat16*>(reinterpret_cast<const unsigned char*>(tile) + swz(row, col)));
}
// v as a bf16 pair hi + lo: hi = bf16(v), lo = bf16(v - hi).
__device__ __forceinline__ void split2(float v0, float v1, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(v0 - hf.x, v1 - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}
__device__ __forceinline__ float2 bf2_to_f2(uint32_t v) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
}

// Shared-memory matrix descriptor (tcgen05): start address, leading and stride
// byte offsets, descriptor version 1 (bit 46), 128-byte swizzle (2 << 61).
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}
// K-major operand: rows (M or N) of 128 bytes along K, groups of 8 rows 1024
// bytes apart; one K16 step is a 32-byte offset inside the swizzled rows.
__device__ __forceinline__ uint64_t desc_k(uint32_t saddr) { return umma_desc(saddr, 16, 1024); }
// MN-major operand of one 64-wide block along M (or N): rows along K, 128
// bytes each, groups of 8 rows 1024 bytes apart; one K16 step is 2048 bytes.
__device__ __forceinline__ uint64_t desc_mn(uint32_t saddr) { return umma_desc(saddr, 1024, 1024); }
// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A/B
// MN-major (transposed) flags, N / 8 and M / 16.
__host__ __device__ constexpr uint32_t umma_idesc(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
// D (tensor memory) = A B (+ D if acc); issued by one thread.
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc ? 1u : 0u)
        : "memory");
}
// `bar` receives one arrival once every MMA this thread has issued is done.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 16 lanes x 256 bits: thread t gets rows t/4 and t/4 + 8 (from the lane base),
// columns 2(t%4) and 2(t%4) + 1 of the 8 at `taddr`: r = {(r0,c0), (r0,c1), (r8,c0), (r8,c1)}.
__device__ __forceinline__ void tmem_ld_16x256b(uint32_t taddr, uint32_t (&r)[4]) {
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
}
// 32 lanes x 32 bits, 16 columns: thread t gets lane (base + t), columns c..c+15.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------- kernel ------

template <int NS>
__global__ void __launch_bounds__(kSsdThreads, NS == 256 ? 1 : 2)
ssd_fwd_kernel(const SsdArgs a, const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
               const __grid_constant__ CUtensorMap tm_c) {
    static_assert(NS == 64 || NS == 128 || NS == 256, "state sizes 64, 128 and 256 are compiled");
    // At N = 256 U is two M = 128 products (rows n < 128 and n >= 128) into
    // 64 more TMEM columns, so a CTA takes all 512 (and, at 177 KB of shared
    // memory, the SM); a thread then holds one state column for all 64
    // channels.
    constexpr int kTmemCols = NS == 256 ? 512 : kSsdTmemCols;
    constexpr int kSC = NS == 256 ? 64 : 32;      // state channels a thread holds
    constexpr int kUM = NS == 256 ? 128 : NS;     // M of each U product
    extern __shared__ unsigned char ssd_smem_raw[];
    // 1024-byte aligned view of the dynamic shared memory, derived from the
    // shared array itself so that every access stays a shared-memory access
    SsdSmem<NS>& sm = *reinterpret_cast<SsdSmem<NS>*>(ssd_smem_raw + ((1024u - (smem_u32(ssd_smem_raw) & 1023u)) & 1023u));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q = warp & 3;      // the TMEM lane quarter this warp may access
    const int half = warp >> 2;  // its half (32 columns) of every per-chunk product
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    // Warps 4 and 5 own blocks of Gm that lie above the diagonal (no TMEM
    // read, no mask arithmetic), so they take the serial work: thread 0 of
    // warp 4 issues the loads and the MMAs, warp 5 forms each chunk's decay.
    constexpr int kIssuer = 128, kDecayWarp = 5;
    const int h = blockIdx.x, b = blockIdx.y;
    const int L = a.seqlen;
    const int n = (L + kSsdQ - 1) / kSsdQ;
    const int dim = a.nheads * kSsdP;
    const int ch0 = h * kSsdP;  // first channel of the head
    const float Ah2 = (in_bounds(a.err, a.A, a.nheads, a.A + h) ? a.A[h] : -1.f) * kLog2e;
    const float bias = a.bias && in_bounds(a.err, a.bias, a.nheads, a.bias + h) ? a.bias[h] : 0.f;
    const float Dh = a.D && in_bounds(a.err, a.D, a.nheads, a.D + h) ? a.D[h] : 0.f;
    const size_t head_row = static_cast<size_t>(b) * a.nheads + h;
    // extents (elements) of the tensors, for the checked-bounds build
    const size_t nheads_all = static_cast<size_t>(a.batch) * a.nheads;   // (batch, head) rows
    const size_t nstate = nheads_all * kSsdP * NS;                         // h0, final state
    const size_t ny = nheads_all * kSsdP * L;                              // y

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sm.tmem)),
                     "n"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // tile loads of chunk k (the issuing thread): barrier 0 = x, 1 = B, 2 = C; parity k & 1
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
    if (tid == kIssuer) {
        for (int i = 0; i < 3; ++i) mbar_init(&sm.full[i], 1);
        for (int i = 0; i < 4; ++i) mbar_init(&sm.done[i], 1);
        fence_barrier_init();
        if (n > 0) { issue(2, 0); issue(1, 0); issue(0, 0); }
    }
    __syncwarp();

    // The state: this thread holds column sn of it for channels p = pc0 + j,
    // j < kSC. U's row n lies in TMEM lane n at N = 128 (M = 128), in lane
    // 32 (n / 16) + n % 16 at N = 64 (M = 64), where lanes 16..31 of a warp
    // hold none, and at N = 256 in lane n % 128 of the product of its half.
    const bool sact = NS != 64 || lane < 16;
    const int sn = NS == 256 ? 32 * q + lane + 128 * half : NS == 128 ? 32 * q + lane : 16 * q + (lane & 15);
    const int pc0 = NS == 256 ? 0 : 32 * half;
    const bool have_state = a.h0 != nullptr;
    float S[kSC];
#pragma unroll
    for (int j = 0; j < kSC; ++j) {
        const float* hp = a.h0 + (head_row * kSsdP + pc0 + j) * NS + sn;
        S[j] = (have_state && sact && in_bounds(a.err, a.h0, nstate, hp)) ? *hp : 0.f;
    }
    // the state's high and low parts as the Y1 product's operand: row n, this
    // thread's kSC channels as 16-byte units of each part
    auto store_state_parts = [&]() {
        if (!sact) return;
        unsigned char* hb = reinterpret_cast<unsigned char*>(&sm.Sh[sn][0]);
        unsigned char* lb = reinterpret_cast<unsigned char*>(&sm.Sl[sn][0]);
#pragma unroll
        for (int c = 0; c < kSC / 8; ++c) {
            uint4 hi, lo;
            split2(S[8 * c], S[8 * c + 1], hi.x, lo.x);
            split2(S[8 * c + 2], S[8 * c + 3], hi.y, lo.y);
            split2(S[8 * c + 4], S[8 * c + 5], hi.z, lo.z);
            split2(S[8 * c + 6], S[8 * c + 7], hi.w, lo.w);
            const int off = ((pc0 / 8 + c) ^ (sn & 7)) << 4;
            *reinterpret_cast<uint4*>(hb + off) = hi;
            *reinterpret_cast<uint4*>(lb + off) = lo;
        }
    };
    if (have_state) store_state_parts();
    // dt, the cumulative decay and the state-update weights of chunk k into
    // buffer k & 1 (one warp); padding steps get dt = 0
    const __nv_bfloat16* dl = static_cast<const __nv_bfloat16*>(a.delta) + head_row * L;
    // Δ of chunk k (steps 2 lane, 2 lane + 1), loaded a chunk ahead of its use
    auto load_delta = [&](int k, float (&r)[2]) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int gl = k * kSsdQ + 2 * lane + i;
            r[i] = gl < L && in_bounds(a.err, static_cast<const __nv_bfloat16*>(a.delta), nheads_all * L, dl + gl)
                ? __bfloat162float(dl[gl]) : 0.f;
        }
    };
    auto decay_prefix = [&](int k, const float (&r)[2]) {
        float v[2], d[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int l = 2 * lane + i, gl = k * kSsdQ + l;
            d[i] = 0.f;
            if (gl < L) {
                d[i] = r[i] + bias;
                if (a.softplus) d[i] = softplus_f(d[i]);
            }
            v[i] = d[i] * Ah2;
        }
        *reinterpret_cast<float2*>(&sm.dt[k & 1][2 * lane]) = make_float2(d[0], d[1]);
        const float pair = v[0] + v[1];
        float incl = pair;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        const float excl = incl - pair;
        const float cq = __shfl_sync(0xffffffffu, incl, 31);
        const float c0 = excl + v[0], c1 = excl + pair;
        *reinterpret_cast<float2*>(&sm.c2[k & 1][2 * lane]) = make_float2(c0, c1);
        *reinterpret_cast<float2*>(&sm.wq[k & 1][wq_at(2 * lane)]) =
            make_float2(ex2_approx(cq - c0) * d[0], ex2_approx(cq - c1) * d[1]);
    };
    if (warp == kDecayWarp && n > 0) {
        float r[2];
        load_delta(0, r);
        decay_prefix(0, r);
    }
    fence_proxy_async_smem();  // the state parts, for the tensor cores
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem = sm.tmem;
    const uint32_t tG = tmem, tY1 = tmem + 64, tY2 = tmem + 128, tU = tmem + 192, tU2 = tmem + 256;
    const uint32_t xs = smem_u32(&sm.X[0][0]), bs = smem_u32(&sm.Bt[0][0]), cs = smem_u32(&sm.Ct[0][0]);
    const uint32_t ghs = smem_u32(&sm.Gh[0][0]), gls = smem_u32(&sm.Gl[0][0]);
    const uint32_t whs = smem_u32(&sm.Wh[0][0]), wls = smem_u32(&sm.Wl[0][0]);
    const uint32_t shs = smem_u32(&sm.Sh[0][0]), sls = smem_u32(&sm.Sl[0][0]);
    constexpr uint32_t kIdG = umma_idesc(64, 64, true, true);     // C^T (MN-major) x B (MN-major)
    constexpr uint32_t kIdY1 = umma_idesc(64, 64, true, true);    // C^T (MN-major) x S^T (MN-major)
    constexpr uint32_t kIdY2 = umma_idesc(64, 64, false, false);  // Gm x X^T
    constexpr uint32_t kIdU = umma_idesc(kUM, 64, false, false);  // B x W^T (each half of B at N = 256)

    __nv_bfloat16* yb = static_cast<__nv_bfloat16*>(a.y) + (static_cast<size_t>(b) * dim + ch0) * L;
    // Output staging [p][kSsdYPitch] over the Gm buffers: written once the
    // masked product is done, stored to HBM at the start of the next chunk.
    __nv_bfloat16* yt = &sm.Gh[0][0];
    const bool vec_ok = (L & 7) == 0;
    const int l0 = 16 * q + (lane >> 2), l1 = l0 + 8;  // this thread's rows in the M = 64 products
    const int cp = 2 * (lane & 3);                     // and its column pair in each group of 8
    // y rows of the head's 64 channels for chunk k, 8 steps per store
    auto store_y = [&](int k) {
#pragma unroll
        for (int v = tid; v < kSsdP * (kSsdQ / 8); v += kSsdThreads) {
            const int p = v >> 3, lc = (v & 7) * 8, gl = k * kSsdQ + lc;
            if (gl >= L) continue;
            __nv_bfloat16* dst = yb + static_cast<size_t>(p) * L + gl;
            const __nv_bfloat16* src = yt + p * kSsdYPitch + lc;
            if (!in_bounds(a.err, static_cast<__nv_bfloat16*>(a.y), ny, dst, min(8, L - gl))) continue;
            if (vec_ok && gl + 8 <= L) {
                *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
            } else {
                for (int i = 0; i < 8 && gl + i < L; ++i) dst[i] = src[i];
            }
        }
    };

    // A wait that runs out sets `timed_out`; the chunk is finished with
    // whatever the tiles hold and the kernel leaves at the chunk's last
    // barrier, so that no thread is ever left waiting at a barrier.
    bool timed_out = false;
#pragma unroll 1
    for (int k = 0; k < n; ++k) {
        const uint32_t par = static_cast<uint32_t>(k & 1);
        const float* c2 = sm.c2[k & 1];
        const float* dtv = sm.dt[k & 1];
        const float* wq = sm.wq[k & 1];
        const bool carry = have_state || k > 0;
        float dnext[2] = {0.f, 0.f};
        if (warp == kDecayWarp && k + 1 < n) load_delta(k + 1, dnext);

        // --- G = C^T B and Y1 = C^T S^T as soon as C and B are in ---
        if (tid == kIssuer) {
            if (!mbar_wait_bounded(&sm.full[2], par)) timed_out = true;
            if (!mbar_wait_bounded(&sm.full[1], par)) timed_out = true;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < NS / 16; ++kk) umma(tG, desc_mn(cs + kk * 2048), desc_mn(bs + kk * 2048), kIdG, kk > 0);
            umma_commit(&sm.done[0]);
            if (carry) {
#pragma unroll
                for (int kk = 0; kk < NS / 16; ++kk) {
                    umma(tY1, desc_mn(cs + kk * 2048), desc_mn(shs + kk * 2048), kIdY1, kk > 0);
                    umma(tY1, desc_mn(cs + kk * 2048), desc_mn(sls + kk * 2048), kIdY1, true);
                }
            }
            umma_commit(&sm.done[1]);
        }
        __syncwarp();
        if (k > 0) store_y(k - 1);

        // --- W = x e^{c_Q - c_s} dt_s, split: thread = channel p, 16 steps ---
        if (!mbar_wait_bounded(&sm.full[0], par)) timed_out = true;
        {
            const int p = tid >> 2;
            const unsigned char* xb = reinterpret_cast<const unsigned char*>(&sm.X[0][0]);
            unsigned char* whb = reinterpret_cast<unsigned char*>(&sm.Wh[0][0]);
            unsigned char* wlb = reinterpret_cast<unsigned char*>(&sm.Wl[0][0]);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int u = 2 * (tid & 3) + i;  // 16-byte unit: steps 8u .. 8u + 7
                const int off = p * 128 + ((u ^ (p & 7)) << 4);
                const uint4 xv = *reinterpret_cast<const uint4*>(xb + off);
                const float4 w0 = *reinterpret_cast<const float4*>(&wq[wq_at(8 * u)]);
                const float4 w1 = *reinterpret_cast<const float4*>(&wq[wq_at(8 * u) + 4]);
                const float2 x0 = bf2_to_f2(xv.x), x1 = bf2_to_f2(xv.y), x2 = bf2_to_f2(xv.z), x3 = bf2_to_f2(xv.w);
                uint4 hi, lo;
                split2(x0.x * w0.x, x0.y * w0.y, hi.x, lo.x);
                split2(x1.x * w0.z, x1.y * w0.w, hi.y, lo.y);
                split2(x2.x * w1.x, x2.y * w1.y, hi.z, lo.z);
                split2(x3.x * w1.z, x3.y * w1.w, hi.w, lo.w);
                *reinterpret_cast<uint4*>(whb + off) = hi;
                *reinterpret_cast<uint4*>(wlb + off) = lo;
            }
        }
        fence_proxy_async_smem();  // W, for the tensor cores
        tc_fence_before();
        __syncthreads();  // W is complete; the staging tile is read out

        // --- U = B W^T, while the masked operand is formed ---
        if (tid == kIssuer) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kSsdQ / 16; ++kk) {
                umma(tU, desc_k(bs + kk * 32), desc_k(whs + kk * 32), kIdU, kk > 0);
                umma(tU, desc_k(bs + kk * 32), desc_k(wls + kk * 32), kIdU, true);
                if (NS == 256) {  // rows n = 128..255 of B: 128 rows of 128 bytes further
                    umma(tU2, desc_k(bs + 16384 + kk * 32), desc_k(whs + kk * 32), kIdU, kk > 0);
                    umma(tU2, desc_k(bs + 16384 + kk * 32), desc_k(wls + kk * 32), kIdU, true);
                }
            }
            umma_commit(&sm.done[2]);
            if (k + 1 < n && !timed_out && mbar_try_wait(&sm.done[1], par)) issue(2, k + 1);  // C is free already
        }
        __syncwarp();

        // --- Gm = G e^{c_l - c_s} dt_s for s <= l, plus D on the diagonal
        //     (so that Y2 carries the skip term D x), split ---
        if (!mbar_wait_bounded(&sm.done[0], par)) timed_out = true;
        tc_fence_after();
        {
            unsigned char* ghb = reinterpret_cast<unsigned char*>(&sm.Gh[0][0]);
            unsigned char* glb = reinterpret_cast<unsigned char*>(&sm.Gl[0][0]);
            if (32 * half <= 16 * q + 15) {  // (the warp's block has steps s <= l)
                uint32_t g[4][4];
#pragma unroll
                for (int j = 0; j < 4; ++j) tmem_ld_16x256b(tG + lane_base + 32 * half + 8 * j, g[j]);
                tmem_wait_ld();
                const float cl0 = c2[l0], cl1 = c2[l1];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int s = 32 * half + 8 * j + cp;
                    const float2 cs2 = *reinterpret_cast<const float2*>(&c2[s]);
                    const float2 ds = *reinterpret_cast<const float2*>(&dtv[s]);
                    float v00 = s <= l0 ? __uint_as_float(g[j][0]) * ex2_approx(cl0 - cs2.x) * ds.x : 0.f;
                    float v01 = s + 1 <= l0 ? __uint_as_float(g[j][1]) * ex2_approx(cl0 - cs2.y) * ds.y : 0.f;
                    float v10 = s <= l1 ? __uint_as_float(g[j][2]) * ex2_approx(cl1 - cs2.x) * ds.x : 0.f;
                    float v11 = s + 1 <= l1 ? __uint_as_float(g[j][3]) * ex2_approx(cl1 - cs2.y) * ds.y : 0.f;
                    if (s == l0) v00 += Dh;
                    if (s + 1 == l0) v01 += Dh;
                    if (s == l1) v10 += Dh;
                    if (s + 1 == l1) v11 += Dh;
                    uint32_t hi, lo;
                    split2(v00, v01, hi, lo);
                    *reinterpret_cast<uint32_t*>(ghb + swz(l0, s)) = hi;
                    *reinterpret_cast<uint32_t*>(glb + swz(l0, s)) = lo;
                    split2(v10, v11, hi, lo);
                    *reinterpret_cast<uint32_t*>(ghb + swz(l1, s)) = hi;
                    *reinterpret_cast<uint32_t*>(glb + swz(l1, s)) = lo;
                }
            } else {  // above the diagonal (the staging tile overwrote it)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int s = 32 * half + 8 * j + cp;
                    *reinterpret_cast<uint32_t*>(ghb + swz(l0, s)) = 0u;
                    *reinterpret_cast<uint32_t*>(glb + swz(l0, s)) = 0u;
                    *reinterpret_cast<uint32_t*>(ghb + swz(l1, s)) = 0u;
                    *reinterpret_cast<uint32_t*>(glb + swz(l1, s)) = 0u;
                }
            }
        }
        fence_proxy_async_smem();  // Gm, for the tensor cores
        tc_fence_before();
        __syncthreads();

        // --- Y2 = Gm X^T; B and C are reloaded for the next chunk once free ---
        if (tid == kIssuer) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kSsdQ / 16; ++kk) {
                umma(tY2, desc_k(ghs + kk * 32), desc_k(xs + kk * 32), kIdY2, kk > 0);
                umma(tY2, desc_k(gls + kk * 32), desc_k(xs + kk * 32), kIdY2, true);
            }
            umma_commit(&sm.done[3]);
            if (k + 1 < n) {
                if (!mbar_wait_bounded(&sm.done[2], par)) timed_out = true;  // G and U: B is free
                if (!timed_out) issue(1, k + 1);
                if (last[2] != k + 1) {  // C not reloaded yet
                    if (!mbar_wait_bounded(&sm.done[1], par)) timed_out = true;  // G and Y1: C is free
                    if (!timed_out) issue(2, k + 1);
                }
            }
        }
        __syncwarp();

        // --- state: S = e^{c_Q} S + U, split into the next chunk's operand ---
        if (!mbar_wait_bounded(&sm.done[2], par)) timed_out = true;  // U
        tc_fence_after();
        {
            const float ed = ex2_approx(c2[kSsdQ - 1]);
            // this thread's row of U (its TMEM lane), kSC columns, 32 at a time
            const uint32_t urow = (NS == 256 ? (half ? tU2 : tU) : tU + 32 * half) + lane_base;
#pragma unroll
            for (int j0 = 0; j0 < kSC; j0 += 32) {
                uint32_t u[2][16];
                tmem_ld_32x32b_x16(urow + j0, u[0]);
                tmem_ld_32x32b_x16(urow + j0 + 16, u[1]);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) S[j0 + j] = fmaf(ed, S[j0 + j], __uint_as_float(u[j >> 4][j & 15]));
            }
        }
        if (!mbar_wait_bounded(&sm.done[1], par)) timed_out = true;  // Y1, the parts' last reader, is done
        store_state_parts();

        // --- outputs y = e^{c_l} Y1 + Y2, staged as bf16 [p][l] over Gm ---
        if (!mbar_wait_bounded(&sm.done[3], par)) timed_out = true;  // every product of the chunk
        tc_fence_after();
        if (tid == kIssuer && k + 1 < n && !timed_out) {  // x is free
            fence_proxy_async_smem();
            issue(0, k + 1);
        }
        __syncwarp();
        {
            uint32_t y1[4][4], y2[4][4];
#pragma unroll
            for (int j = 0; j < 4; ++j) tmem_ld_16x256b(tY2 + lane_base + 32 * half + 8 * j, y2[j]);
            if (carry) {
#pragma unroll
                for (int j = 0; j < 4; ++j) tmem_ld_16x256b(tY1 + lane_base + 32 * half + 8 * j, y1[j]);
            }
            tmem_wait_ld();
            const float e0 = carry ? ex2_approx(c2[l0]) : 0.f, e1 = carry ? ex2_approx(c2[l1]) : 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int p = 32 * half + 8 * j + cp;
                float v00 = __uint_as_float(y2[j][0]), v01 = __uint_as_float(y2[j][1]);
                float v10 = __uint_as_float(y2[j][2]), v11 = __uint_as_float(y2[j][3]);
                if (carry) {
                    v00 = fmaf(e0, __uint_as_float(y1[j][0]), v00);
                    v01 = fmaf(e0, __uint_as_float(y1[j][1]), v01);
                    v10 = fmaf(e1, __uint_as_float(y1[j][2]), v10);
                    v11 = fmaf(e1, __uint_as_float(y1[j][3]), v11);
                }
                yt[p * kSsdYPitch + l0] = __float2bfloat16_rn(v00);
                yt[(p + 1) * kSsdYPitch + l0] = __float2bfloat16_rn(v01);
                yt[p * kSsdYPitch + l1] = __float2bfloat16_rn(v10);
                yt[(p + 1) * kSsdYPitch + l1] = __float2bfloat16_rn(v11);
            }
        }

        if (warp == kDecayWarp && k + 1 < n) decay_prefix(k + 1, dnext);  // the next chunk's dt and decay, other buffer
        fence_proxy_async_smem();  // the state parts, for the next chunk's Y1 product
        tc_fence_before();
        // the staging tile, the state parts and the next chunk's decay are complete
        if (__syncthreads_or(timed_out)) {
            if (tid == kIssuer) {
                report_device_error(a.err, -6);
                drain();
                for (int i = 0; i < 4; ++i) mbar_wait_bounded(&sm.done[i], par);  // this chunk's products
            }
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            if (warp == 0)
                asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols)
                             : "memory");
            return;
        }
        tc_fence_after();
    }
    if (n > 0) store_y(n - 1);

    if (a.final_state && sact) {
#pragma unroll
        for (int j = 0; j < kSC; ++j) {
            float* fp = a.final_state + (head_row * kSsdP + pc0 + j) * NS + sn;
            if (in_bounds(a.err, a.final_state, nstate, fp)) *fp = S[j];
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
}

}  // namespace mscan
