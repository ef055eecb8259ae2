// C ABI of libmambascan.so: argument validation, workspaces, dispatch.
//
// Declared in include/mamba_scan.h. Every check runs on the host before any
// launch; a rejected call launches nothing and writes nothing. The library
// keeps no state besides the device error word; mamba_scan_fwd allocates its
// workspace stream-ordered, mamba_scan_fwd_ws takes it from the caller. The
// forward-scan kernels themselves are launched from scan_fwd_n*.cu (one file
// per state size, see host.h).
#include <algorithm>
#include <cstring>
#include <mutex>

#include "../../include/mamba_scan.h"
#include "host.h"
#include "scan_bwd.cuh"
#include "state_update.cuh"

// Device error word: 0 = fine, otherwise the mamba_status a kernel reported
// (kernels get its address in their arguments). Read and cleared by
// mamba_check_device_error.
static __device__ int g_device_error = 0;

namespace {

using mhost::aligned;
using mhost::round_up;

constexpr int kKnownFlags = MAMBA_FLAG_SOFTPLUS | MAMBA_FLAG_ZOH;
static_assert(mscan::kErrDeviceBounds == MAMBA_ERR_DEVICE_BOUNDS, "the kernels' bounds status is the ABI's");

bool forward_dstate(int dstate) { return dstate == 8 || dstate == 16 || dstate == 32 || dstate == 64; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Device address of a file-scope __device__ object on the current device. In
// host code such an object's name is only a host-side stand-in, so the address
// comes from cudaGetSymbolAddress, looked up once per device (with that device
// current) and cached in `cache`. Returns nullptr if the lookup fails.
constexpr int kMaxDevices = 64;
std::mutex g_symbol_mutex;

template <typename Sym>
void* symbol_address(const Sym& sym, void* (&cache)[kMaxDevices]) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_symbol_mutex);
    if (!cache[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, sym) != cudaSuccess) return nullptr;
        cache[dev] = p;
    }
    return cache[dev];
}

void* g_error_addr[kMaxDevices] = {};

int* device_error_word() { return static_cast<int*>(symbol_address(g_device_error, g_error_addr)); }

}  // namespace

bool mhost::make_map_3d(CUtensorMap* m, CUtensorMapDataType t, size_t es, const void* base, uint64_t e0,
                        uint64_t e1, uint64_t e2, uint64_t pitch0, uint32_t b0, uint32_t b1,
                        CUtensorMapSwizzle swizzle) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {e0, e1, e2};
    const cuuint64_t strides[2] = {pitch0 * es, pitch0 * e1 * es};
    const cuuint32_t box[3] = {b0, b1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, t, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

template <typename T, int NS>
void launch_pack(const void* B, const void* C, float* bc, int batch, int L, int Lp, int* err, cudaStream_t stream) {
    const long long threads = static_cast<long long>(batch) * Lp;
    mscan::bc_pack_kernel<T, NS><<<static_cast<unsigned>((threads + 255) / 256), 256, 0, stream>>>(
        static_cast<const T*>(B), static_cast<const T*>(C), bc, batch, L, Lp, err);
}

// Streaming multiprocessors of the current device (looked up once per device).
int device_sms() {
    static int cache[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    if (!cache[dev]) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = sms;
    }
    return cache[dev];
}

// Sequence split of the forward scan. A CTA is one warp that walks its
// channels' whole sequence; when there are too few of them to keep the
// schedulers busy (a long sequence over few channels), the chunks are cut
// into segments: a state-only pass finds each segment's end state (from
// zero), and the full pass starts every segment from the combination of the
// ones before it. The state-only pass costs about 60% of a full pass per
// element, but a lone warp per scheduler runs at a fraction of the rate of
// several: measured on B300 over 131072 steps, 5120 channels ran 1.5x and
// 2048 channels 3.6x faster split into segments for about 12 warps a
// scheduler (at most 32 segments) than in one pass, and no target beat it.
// The split is taken only where the grid is under one warp per scheduler,
// into segments of at least 64 chunks.
constexpr int kSplitWarpsPerScheduler = 12;
constexpr int kMaxSegments = 32;
constexpr int kMinSegmentChunks = 64;

struct SplitPlan {
    int nseg = 1;        // segments (1: no split)
    int seg_chunks = 0;  // chunks per segment (0: no split)
    size_t carry = 0, carry_dt = 0, bytes = 0;  // workspace layout: end states, sums of dt, total
};

// The split of a (batch, dim, L) scan; with `max_bytes`, the largest segment
// count (if any) whose carries fit in that many bytes.
SplitPlan plan_split(long long batch, long long dim, long long L, int dstate, size_t max_bytes = ~size_t(0)) {
    SplitPlan p;
    const int sms = device_sms();
    if (batch <= 0 || dim <= 0 || L <= 0 || sms <= 0) return p;
    const long long kch = dstate == 8    ? mscan::FwdGeo<8>::kCh    // channels per warp
                          : dstate == 16 ? mscan::FwdGeo<16>::kCh
                          : dstate == 32 ? mscan::FwdGeo<32>::kCh
                                         : mscan::FwdGeo<64>::kCh;
    const long long warps = batch * ((dim + kch - 1) / kch);
    const long long schedulers = 4ll * sms;
    if (warps >= schedulers) return p;
    const long long chunks = (L + mscan::kTL - 1) / mscan::kTL;
    long long k = (kSplitWarpsPerScheduler * schedulers + warps / 2) / warps;
    k = std::min<long long>(std::min<long long>(k, kMaxSegments), chunks / kMinSegmentChunks);
    for (; k >= 2; --k) {
        p.seg_chunks = static_cast<int>((chunks + k - 1) / k);
        p.nseg = static_cast<int>((chunks + p.seg_chunks - 1) / p.seg_chunks);
        const size_t rows = static_cast<size_t>(p.nseg - 1) * batch * dim;
        p.carry = 0;
        p.carry_dt = round_up(rows * dstate * sizeof(float), 256);
        p.bytes = p.carry_dt + round_up(rows * sizeof(float), 256);
        if (p.nseg >= 2 && p.bytes <= max_bytes) return p;
    }
    return SplitPlan();
}

// The forward scan, split as `plan` says when `ws` (at least plan.bytes) is
// given, else in one pass.
template <typename T>
int launch_scan(mscan::ScanArgs a, int flags, int dstate, const SplitPlan& plan, char* ws, cudaStream_t stream) {
    if (!(a.err = device_error_word())) return MAMBA_ERR_CUDA;
    auto launch = [&](int nseg, bool state_pass) {
        switch (dstate) {
            case 8: return mhost::launch_scan_n<T, 8>(a, flags, nseg, state_pass, stream);
            case 16: return mhost::launch_scan_n<T, 16>(a, flags, nseg, state_pass, stream);
            case 32: return mhost::launch_scan_n<T, 32>(a, flags, nseg, state_pass, stream);
            default: return mhost::launch_scan_n<T, 64>(a, flags, nseg, state_pass, stream);
        }
    };
    if (plan.nseg < 2 || !ws) {
        a.seg_chunks = 0;
        return launch(1, false);
    }
    a.seg_chunks = plan.seg_chunks;
    a.carry = reinterpret_cast<float*>(ws + plan.carry);
    a.carry_dt = reinterpret_cast<float*>(ws + plan.carry_dt);
    const int st = launch(plan.nseg, true);
    return st != MAMBA_OK ? st : launch(plan.nseg, false);
}

template <typename T, int NS>
void launch_update_n(const mscan::UpdateArgs& a, bool zoh, cudaStream_t stream) {
    using G = mscan::UpdateGeo<NS>;
    const dim3 grid((a.dim + G::kCh - 1) / G::kCh, (a.batch + G::kR - 1) / G::kR);
    if (zoh) mscan::state_update_kernel<T, NS, true><<<grid, mscan::kUpdateThreads, 0, stream>>>(a);
    else mscan::state_update_kernel<T, NS, false><<<grid, mscan::kUpdateThreads, 0, stream>>>(a);
}

template <typename T, int NS>
void launch_ssd_update_n(const mscan::SsdUpdateArgs& a, cudaStream_t s) {
    constexpr int rows = mscan::SsdUpdateGeo<NS>::kRows;
    const dim3 grid((a.nheads * a.headdim + rows - 1) / rows, a.batch);
    mscan::ssd_update_kernel<T, NS><<<grid, mscan::kUpdateThreads, 0, s>>>(a);
}

template <typename T>
int launch_update(const mscan::UpdateArgs& a, int dstate, bool zoh, cudaStream_t stream) {
    switch (dstate) {
        case 8: launch_update_n<T, 8>(a, zoh, stream); break;
        case 16: launch_update_n<T, 16>(a, zoh, stream); break;
        case 32: launch_update_n<T, 32>(a, zoh, stream); break;
        default: launch_update_n<T, 64>(a, zoh, stream); break;
    }
    return cudaGetLastError() == cudaSuccess ? MAMBA_OK : MAMBA_ERR_CUDA;
}

// Workspace of one backward call: packed B/C rows, one fp32 state per row per
// 16-step chunk, and the fp32 sums of dB and dC.
struct BwdWorkspace {
    int Lp, n;
    size_t bc, hck, dbc, total;
};

BwdWorkspace bwd_workspace(long long batch, long long dim, long long L, int dstate) {
    BwdWorkspace w;
    w.Lp = static_cast<int>(round_up(static_cast<size_t>(L), mscan::kBwdTL));
    w.n = w.Lp / mscan::kBwdTL;
    w.bc = 0;
    size_t off = round_up(static_cast<size_t>(batch) * w.Lp * 2 * dstate * sizeof(float), 256);
    w.hck = off;
    off += round_up(static_cast<size_t>(batch) * dim * w.n * dstate * sizeof(float), 256);
    w.dbc = off;
    off += round_up(static_cast<size_t>(batch) * 2 * dstate * w.Lp * sizeof(float), 256);
    w.total = L > 0 ? off : 0;
    return w;
}

template <typename T>
int launch_bwd(mscan::ScanBwdArgs a, int flags, int dstate, const void* B, const void* C, void* dB, void* dC,
               char* ws, cudaStream_t stream) {
    const BwdWorkspace w = bwd_workspace(a.batch, a.dim, a.seqlen, dstate);
    a.Lp = w.Lp;
    if (!(a.err = device_error_word())) return MAMBA_ERR_CUDA;
    if (cudaMemsetAsync(a.dA, 0, static_cast<size_t>(a.dim) * dstate * sizeof(float), stream) != cudaSuccess)
        return MAMBA_ERR_CUDA;
    if (a.dD && cudaMemsetAsync(a.dD, 0, a.dim * sizeof(float), stream) != cudaSuccess) return MAMBA_ERR_CUDA;
    if (a.dbias && cudaMemsetAsync(a.dbias, 0, a.dim * sizeof(float), stream) != cudaSuccess) return MAMBA_ERR_CUDA;
    if (a.seqlen > 0) {
        a.bc = reinterpret_cast<const float*>(ws + w.bc);
        if (!a.have_hck) a.hck = reinterpret_cast<float*>(ws + w.hck);
        a.dbc = reinterpret_cast<float*>(ws + w.dbc);
        if (cudaMemsetAsync(a.dbc, 0, static_cast<size_t>(a.batch) * 2 * dstate * w.Lp * sizeof(float), stream) !=
            cudaSuccess)
            return MAMBA_ERR_CUDA;
        float* bc = const_cast<float*>(a.bc);
        switch (dstate) {
            case 8: launch_pack<T, 8>(B, C, bc, a.batch, a.seqlen, w.Lp, a.err, stream); break;
            case 16: launch_pack<T, 16>(B, C, bc, a.batch, a.seqlen, w.Lp, a.err, stream); break;
            case 32: launch_pack<T, 32>(B, C, bc, a.batch, a.seqlen, w.Lp, a.err, stream); break;
            default: launch_pack<T, 64>(B, C, bc, a.batch, a.seqlen, w.Lp, a.err, stream); break;
        }
    }
    int st;
    switch (dstate) {
        case 8: st = mhost::launch_bwd_n<T, 8>(a, flags, stream); break;
        case 16: st = mhost::launch_bwd_n<T, 16>(a, flags, stream); break;
        case 32: st = mhost::launch_bwd_n<T, 32>(a, flags, stream); break;
        default: st = mhost::launch_bwd_n<T, 64>(a, flags, stream); break;
    }
    if (st != MAMBA_OK) return st;
    if (a.seqlen > 0) {
        const long long total = static_cast<long long>(a.batch) * 2 * dstate * a.seqlen;
        const unsigned blocks = static_cast<unsigned>(std::min<long long>((total + 255) / 256, 148ll * 32));
        mscan::dbc_unpack_kernel<T><<<blocks, 256, 0, stream>>>(a.dbc, static_cast<T*>(dB), static_cast<T*>(dC),
                                                               a.batch, dstate, a.seqlen, w.Lp, a.err);
    }
    return cudaGetLastError() == cudaSuccess ? MAMBA_OK : MAMBA_ERR_CUDA;
}

size_t dtype_size(int io_dtype) { return io_dtype == MAMBA_BF16 ? 2 : 4; }

}  // namespace

extern "C" {

// Argument checks shared by the scan entry points (MAMBA_OK or the error code).
static int check_scan_args(const void* u, const void* delta, const float* A, const void* B, const void* C,
                           const float* D, const void* z, const float* delta_bias, int flags, const void* y,
                           const float* final_state, int batch, int dim, int seqlen, int dstate, int io_dtype,
                           const float* initial_state = nullptr) {
    if (io_dtype != MAMBA_F32 && io_dtype != MAMBA_BF16) return MAMBA_ERR_DTYPE;
    if (flags & ~kKnownFlags) return MAMBA_ERR_FLAGS;
    if (batch < 0 || dim < 0 || seqlen < 0 || !forward_dstate(dstate)) return MAMBA_ERR_SHAPE;
    if (batch > 65535) return MAMBA_ERR_SHAPE;  // grid.y
    const size_t es = dtype_size(io_dtype);
    // every flat index must fit in 63 bits of bytes, and TMA strides in 40 bits
    const unsigned long long elems = static_cast<unsigned long long>(batch) * dim * seqlen;
    if (dim > 0 && seqlen > 0 && elems / dim / seqlen != static_cast<unsigned long long>(batch)) return MAMBA_ERR_SHAPE;
    if ((static_cast<unsigned long long>(seqlen) + 16) * dim * es >= (1ull << 40)) return MAMBA_ERR_SHAPE;
    if ((static_cast<unsigned long long>(seqlen) + 16) * 2 * dstate * sizeof(float) >= (1ull << 40))
        return MAMBA_ERR_SHAPE;
    if (batch == 0 || dim == 0) return MAMBA_OK;
    if (!A) return MAMBA_ERR_NULL;
    if (seqlen > 0 && (!u || !delta || !B || !C || !y)) return MAMBA_ERR_NULL;
    const void* p16[] = {u, delta, z, B, C, y, A, final_state, initial_state};
    for (const void* p : p16)
        if (p && !aligned(p, 16)) return MAMBA_ERR_ALIGN;
    if ((D && !aligned(D, 4)) || (delta_bias && !aligned(delta_bias, 4))) return MAMBA_ERR_ALIGN;
    return MAMBA_OK;
}

struct ConvArgs {
    const float* w = nullptr;     // (dim, 4) or null: no convolution
    const float* b = nullptr;
    const void* state = nullptr;
};

static int run_scan(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
                    const void* z, const float* delta_bias, int flags, void* y, float* final_state, int batch,
                    int dim, int seqlen, int dstate, int io_dtype, cudaStream_t s,
                    const float* initial_state = nullptr, ConvArgs conv = ConvArgs(),
                    float* chunk_states = nullptr, void* workspace = nullptr,
                    const SplitPlan* plan_in = nullptr) {
    mscan::ScanArgs a;
    memset(&a, 0, sizeof(a));
    a.u = u; a.delta = delta; a.z = z; a.B = B; a.C = C;
    a.A = A; a.D = D; a.bias = delta_bias; a.h0 = initial_state; a.y = y; a.final_state = final_state;
    a.conv_w = conv.w; a.conv_b = conv.b; a.conv_state = conv.state;
    a.chunk_states = chunk_states;
    a.batch = batch; a.dim = dim; a.seqlen = seqlen;
    const SplitPlan plan = plan_in ? *plan_in : plan_split(batch, dim, seqlen, dstate);
    char* ws = static_cast<char*>(workspace);
    return io_dtype == MAMBA_BF16 ? launch_scan<__nv_bfloat16>(a, flags, dstate, plan, ws, s)
                                  : launch_scan<float>(a, flags, dstate, plan, ws, s);
}

// Checks a caller's workspace against the split plan's need: NULL runs the
// scan in one pass; otherwise it must hold `need` bytes, 256-byte aligned.
static int check_workspace(void* workspace, size_t workspace_bytes, size_t need) {
    if (!workspace || need == 0) return MAMBA_OK;
    if (workspace_bytes < need) return MAMBA_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return MAMBA_ERR_ALIGN;
    return MAMBA_OK;
}

size_t mamba_scan_workspace_size(int batch, int dim, int seqlen, int dstate, int io_dtype) {
    if (batch <= 0 || dim <= 0 || seqlen <= 0 || !forward_dstate(dstate)) return 0;
    if (io_dtype != MAMBA_F32 && io_dtype != MAMBA_BF16) return 0;
    return plan_split(batch, dim, seqlen, dstate).bytes;
}

int mamba_scan_fwd_ws(const void* u, const void* delta, const float* A, const void* B, const void* C,
                      const float* D, const void* z, const float* delta_bias, int flags,
                      const float* initial_state, void* y, float* final_state, float* chunk_states, int batch,
                      int dim, int seqlen, int dstate, int io_dtype, void* workspace, size_t workspace_bytes,
                      void* stream) {
    int st = check_scan_args(u, delta, A, B, C, D, z, delta_bias, flags, y, final_state, batch, dim, seqlen, dstate,
                             io_dtype, initial_state);
    if (st != MAMBA_OK || batch == 0 || dim == 0) return st;
    if (chunk_states && !aligned(chunk_states, 16)) return MAMBA_ERR_ALIGN;
    st = check_workspace(workspace, workspace_bytes, plan_split(batch, dim, seqlen, dstate).bytes);
    if (st != MAMBA_OK) return st;
    return run_scan(u, delta, A, B, C, D, z, delta_bias, flags, y, final_state, batch, dim, seqlen, dstate,
                    io_dtype, static_cast<cudaStream_t>(stream), initial_state, ConvArgs(), chunk_states, workspace);
}

int mamba_conv_scan_fwd_ws(const void* x, const float* conv_weight, const float* conv_bias,
                           const void* conv_state, int conv_width, const void* delta, const float* A, const void* B,
                           const void* C, const float* D, const void* z, const float* delta_bias, int flags,
                           const float* initial_state, void* y, float* final_state, int batch, int dim,
                           int seqlen, int dstate, int io_dtype, void* workspace, size_t workspace_bytes,
                           void* stream) {
    int st = check_scan_args(x, delta, A, B, C, D, z, delta_bias, flags, y, final_state, batch, dim, seqlen, dstate,
                             io_dtype, initial_state);
    if (st != MAMBA_OK) return st;
    if (conv_width != mscan::kConvW) return MAMBA_ERR_SHAPE;
    if (batch == 0 || dim == 0) return MAMBA_OK;
    if (!conv_weight) return MAMBA_ERR_NULL;
    if (!aligned(conv_weight, 16) || (conv_bias && !aligned(conv_bias, 4)) ||
        (conv_state && !aligned(conv_state, dtype_size(io_dtype))))
        return MAMBA_ERR_ALIGN;
    st = check_workspace(workspace, workspace_bytes, plan_split(batch, dim, seqlen, dstate).bytes);
    if (st != MAMBA_OK) return st;
    ConvArgs conv;
    conv.w = conv_weight; conv.b = conv_bias; conv.state = conv_state;
    return run_scan(x, delta, A, B, C, D, z, delta_bias, flags, y, final_state, batch, dim, seqlen, dstate,
                    io_dtype, static_cast<cudaStream_t>(stream), initial_state, conv, nullptr, workspace);
}

int mamba_scan_fwd(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
                   const void* z, const float* delta_bias, int flags, void* y, float* final_state,
                   int batch, int dim, int seqlen, int dstate, int io_dtype, void* stream) {
    int st = check_scan_args(u, delta, A, B, C, D, z, delta_bias, flags, y, final_state, batch, dim, seqlen, dstate,
                             io_dtype);
    if (st != MAMBA_OK || batch == 0 || dim == 0) return st;
    return run_scan(u, delta, A, B, C, D, z, delta_bias, flags, y, final_state, batch, dim, seqlen, dstate,
                    io_dtype, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free scan: a fixed scratch array instead of a workspace.
//
// Some callers cannot allocate device memory at call time: serving loops that
// reserve all their memory at start-up and must not allocate afterwards,
// plugins running inside a host framework that owns every device allocation,
// and programs that have no allocator of their own to hand us a workspace.
// The only scratch the forward scan uses is the carries of a split sequence
// (long sequences over few channels, see plan_split). mamba_scan_fwd_noalloc
// keeps them in this file-scope device array, which every GPU that loads the
// library holds until the process exits, so it splits exactly where
// mamba_scan_fwd_ws given a workspace does, into as many segments as it
// would take whose carries fit: (segments - 1) * batch * dim * (N + 1) fp32
// values within 1 MiB (on a 148-SM B300, 4 segments of 1 x 5120 channels at
// N = 16, where the workspace entry point takes 22; the split still runs,
// with fewer segments, never in more memory).
constexpr size_t kStaticScratchBytes = 1u << 20;  // 1 MiB
static __device__ __align__(256) unsigned char g_scan_scratch[kStaticScratchBytes];

namespace {

void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_scan_scratch on the current device (looked up once per
// device with that device current, then cached); nullptr if the lookup fails.
void* scratch_address() { return symbol_address(g_scan_scratch, g_scratch_addr); }

}  // namespace

extern "C" int mamba_scan_fwd_noalloc(const void* u, const void* delta, const float* A, const void* B,
                                      const void* C, const float* D, const void* z, const float* delta_bias,
                                      int flags, void* y, float* final_state, int batch, int dim,
                                      int seqlen, int dstate, int io_dtype, void* stream) {
    int st = check_scan_args(u, delta, A, B, C, D, z, delta_bias, flags, y, final_state, batch, dim, seqlen, dstate,
                             io_dtype);
    if (st != MAMBA_OK || batch == 0 || dim == 0) return st;
    // The array's address is the current device's: a stream of another
    // device would make the kernels touch that device's memory.
    int dev = 0, sdev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MAMBA_ERR_CUDA;
    if (stream && (cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev) != cudaSuccess || sdev != dev))
        return MAMBA_ERR_CUDA;
    const SplitPlan plan = plan_split(batch, dim, seqlen, dstate, kStaticScratchBytes);
    void* scratch = nullptr;
    if (plan.bytes > 0 && !(scratch = scratch_address())) return MAMBA_ERR_CUDA;
    // The state-only pass writes every carry the full pass reads, so the
    // array needs no clearing between calls.
    return run_scan(u, delta, A, B, C, D, z, delta_bias, flags, y, final_state, batch, dim, seqlen, dstate,
                    io_dtype, static_cast<cudaStream_t>(stream), nullptr, ConvArgs(), nullptr, scratch, &plan);
}

extern "C" {

size_t mamba_scan_bwd_workspace_size(int batch, int dim, int seqlen, int dstate, int io_dtype) {
    if (batch <= 0 || dim <= 0 || seqlen <= 0 || !forward_dstate(dstate)) return 0;
    if (io_dtype != MAMBA_F32 && io_dtype != MAMBA_BF16) return 0;
    return bwd_workspace(batch, dim, seqlen, dstate).total;
}

int mamba_scan_bwd(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
                   const void* z, const float* delta_bias, int flags, const float* initial_state,
                   const float* chunk_states, const void* dy, void* du, void* ddelta, float* dA, void* dB, void* dC, float* dD, void* dz,
                   float* ddelta_bias, float* dinitial_state, int batch, int dim, int seqlen, int dstate,
                   int io_dtype, void* workspace, size_t workspace_bytes, void* stream) {
    int st = check_scan_args(u, delta, A, B, C, D, z, delta_bias, flags, dy, nullptr, batch, dim, seqlen, dstate, io_dtype,
                             initial_state);
    if (st != MAMBA_OK) return st;
    if (batch == 0 || dim == 0) return MAMBA_OK;
    if (!dA) return MAMBA_ERR_NULL;
    if (seqlen > 0 && (!du || !ddelta || !dB || !dC)) return MAMBA_ERR_NULL;
    if (z && seqlen > 0 && !dz) return MAMBA_ERR_NULL;
    if ((dD && !D) || (ddelta_bias && !delta_bias)) return MAMBA_ERR_NULL;  // a gradient of an absent input
    const void* p16[] = {du, ddelta, dA, dB, dC, dz, dinitial_state, chunk_states};
    for (const void* p : p16)
        if (p && !aligned(p, 16)) return MAMBA_ERR_ALIGN;
    if ((dD && !aligned(dD, 4)) || (ddelta_bias && !aligned(ddelta_bias, 4))) return MAMBA_ERR_ALIGN;
    const size_t need = bwd_workspace(batch, dim, seqlen, dstate).total;
    if (need > 0) {
        if (!workspace) return MAMBA_ERR_NULL;
        if (workspace_bytes < need) return MAMBA_ERR_WORKSPACE;
        if (!aligned(workspace, 256)) return MAMBA_ERR_ALIGN;
    }
    mscan::ScanBwdArgs a;
    memset(&a, 0, sizeof(a));
    a.u = u; a.delta = delta; a.z = z; a.dy = dy; a.A = A; a.D = D; a.bias = delta_bias; a.h0 = initial_state;
    a.du = du; a.ddelta = ddelta; a.dz = z ? dz : nullptr; a.dA = dA; a.dD = dD; a.dbias = ddelta_bias;
    a.dh0 = dinitial_state;
    a.hck = const_cast<float*>(chunk_states);  // read only when given
    a.have_hck = chunk_states != nullptr;
    a.batch = batch; a.dim = dim; a.seqlen = seqlen;
    char* ws = static_cast<char*>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return io_dtype == MAMBA_BF16 ? launch_bwd<__nv_bfloat16>(a, flags, dstate, B, C, dB, dC, ws, s)
                                  : launch_bwd<float>(a, flags, dstate, B, C, dB, dC, ws, s);
}

int mamba_state_update(float* state, const void* u, const void* delta, const float* A, const void* B, const void* C,
                       const float* D, const void* z, const float* delta_bias, int flags, void* y, int batch,
                       int dim, int dstate, int io_dtype, void* stream) {
    if (io_dtype != MAMBA_F32 && io_dtype != MAMBA_BF16) return MAMBA_ERR_DTYPE;
    if (flags & ~kKnownFlags) return MAMBA_ERR_FLAGS;
    if (batch < 0 || dim < 0 || !forward_dstate(dstate)) return MAMBA_ERR_SHAPE;
    if (batch > 65535) return MAMBA_ERR_SHAPE;  // grid.y
    if (batch == 0 || dim == 0) return MAMBA_OK;
    if (!state || !u || !delta || !A || !B || !C || !y) return MAMBA_ERR_NULL;
    const void* p16[] = {state, A};
    for (const void* p : p16)
        if (!aligned(p, 16)) return MAMBA_ERR_ALIGN;
    const size_t es = dtype_size(io_dtype);
    // B/C rows are read 4 values at a time (16-byte base alignment as for every entry point)
    if (!aligned(B, 16) || !aligned(C, 16)) return MAMBA_ERR_ALIGN;
    const void* pe[] = {u, delta, z, y};
    for (const void* p : pe)
        if (p && !aligned(p, es)) return MAMBA_ERR_ALIGN;
    if ((D && !aligned(D, 4)) || (delta_bias && !aligned(delta_bias, 4))) return MAMBA_ERR_ALIGN;

    mscan::UpdateArgs a;
    a.state = state; a.u = u; a.delta = delta; a.z = z; a.B = B; a.C = C; a.A = A; a.D = D; a.bias = delta_bias;
    a.y = y; a.batch = batch; a.dim = dim; a.softplus = (flags & MAMBA_FLAG_SOFTPLUS) != 0;
    if (!(a.err = device_error_word())) return MAMBA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool zoh = (flags & MAMBA_FLAG_ZOH) != 0;
    return io_dtype == MAMBA_BF16 ? launch_update<__nv_bfloat16>(a, dstate, zoh, s)
                                  : launch_update<float>(a, dstate, zoh, s);
}

// --- SSD (Mamba-2 chunked form) ---------------------------------------------

static bool ssd_dstate(int dstate) { return dstate == 64 || dstate == 128 || dstate == 256; }

// Workspace of one SSD call: row-pitched copies of x, B and C when a row of
// seqlen bf16 values is not a whole number of 16-byte units (a TMA stride rule).
struct SsdWorkspace {
    int pitch;
    bool copy_rows;
    size_t x, b, c, total;
};

static SsdWorkspace ssd_workspace(long long batch, long long nheads, long long L, int dstate) {
    SsdWorkspace w;
    w.copy_rows = (L * 2) % 16 != 0;
    w.pitch = w.copy_rows ? static_cast<int>(round_up(static_cast<size_t>(L), 8)) : static_cast<int>(L);
    const size_t xr = static_cast<size_t>(batch) * nheads * mscan::kSsdP * w.pitch * 2;
    const size_t br = static_cast<size_t>(batch) * dstate * w.pitch * 2;
    w.x = 0;
    w.b = round_up(xr, 256);
    w.c = w.b + round_up(br, 256);
    w.total = (w.copy_rows && L > 0) ? w.c + round_up(br, 256) : 0;
    return w;
}

size_t mamba_ssd_workspace_size(int batch, int nheads, int headdim, int seqlen, int dstate, int io_dtype) {
    if (batch <= 0 || nheads <= 0 || seqlen <= 0 || headdim != mscan::kSsdP || !ssd_dstate(dstate)) return 0;
    if (io_dtype != MAMBA_BF16) return 0;
    return ssd_workspace(batch, nheads, seqlen, dstate).total;
}

int mamba_ssd_fwd(const void* x, const void* delta, const float* A, const void* B, const void* C, const float* D,
                  const float* delta_bias, int flags, const float* initial_state, void* y, float* final_state,
                  int batch, int nheads, int headdim, int seqlen, int dstate, int io_dtype, void* workspace,
                  size_t workspace_bytes, void* stream) {
    if (io_dtype != MAMBA_BF16) return MAMBA_ERR_DTYPE;
    if (flags & ~MAMBA_FLAG_SOFTPLUS) return MAMBA_ERR_FLAGS;
    if (batch < 0 || nheads < 0 || seqlen < 0 || headdim != mscan::kSsdP || !ssd_dstate(dstate))
        return MAMBA_ERR_SHAPE;
    if (batch > 65535) return MAMBA_ERR_SHAPE;  // grid.y
    const unsigned long long dim = static_cast<unsigned long long>(nheads) * headdim;
    if ((static_cast<unsigned long long>(seqlen) + 16) * dim * 2 >= (1ull << 40)) return MAMBA_ERR_SHAPE;
    if (dim > 0 && seqlen > 0 &&
        static_cast<unsigned long long>(batch) * dim * static_cast<unsigned long long>(seqlen) >= (1ull << 62))
        return MAMBA_ERR_SHAPE;
    if (batch == 0 || nheads == 0) return MAMBA_OK;
    if (!A) return MAMBA_ERR_NULL;
    if (seqlen > 0 && (!x || !delta || !B || !C || !y)) return MAMBA_ERR_NULL;
    const void* p16[] = {x, B, C, y, initial_state, final_state};
    for (const void* p : p16)
        if (p && !aligned(p, 16)) return MAMBA_ERR_ALIGN;
    if ((delta && !aligned(delta, 2)) || !aligned(A, 4) || (D && !aligned(D, 4)) ||
        (delta_bias && !aligned(delta_bias, 4)))
        return MAMBA_ERR_ALIGN;
    const SsdWorkspace w = ssd_workspace(batch, nheads, seqlen, dstate);
    if (w.total > 0) {
        if (!workspace) return MAMBA_ERR_NULL;
        if (workspace_bytes < w.total) return MAMBA_ERR_WORKSPACE;
        if (!aligned(workspace, 256)) return MAMBA_ERR_ALIGN;
    }
    mscan::SsdArgs a;
    memset(&a, 0, sizeof(a));
    a.delta = delta; a.A = A; a.D = D; a.bias = delta_bias; a.h0 = initial_state; a.y = y;
    a.final_state = final_state; a.batch = batch; a.nheads = nheads; a.seqlen = seqlen;
    a.softplus = (flags & MAMBA_FLAG_SOFTPLUS) != 0;
    if (!(a.err = device_error_word())) return MAMBA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (w.total > 0) {  // rows of x, B and C at a 16-byte pitch
        char* ws = static_cast<char*>(workspace);
        const long long rows[3] = {static_cast<long long>(batch) * nheads * headdim,
                                   static_cast<long long>(batch) * dstate, static_cast<long long>(batch) * dstate};
        const void* src[3] = {x, B, C};
        const size_t dst[3] = {w.x, w.b, w.c};
        for (int i = 0; i < 3; ++i) {
            const unsigned blocks = static_cast<unsigned>(std::min<long long>((rows[i] * seqlen + 255) / 256, 148ll * 16));
            mscan::row_pitch_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
                static_cast<const __nv_bfloat16*>(src[i]), reinterpret_cast<__nv_bfloat16*>(ws + dst[i]), rows[i],
                seqlen, w.pitch, a.err);
        }
        if (cudaGetLastError() != cudaSuccess) return MAMBA_ERR_CUDA;
        x = ws + w.x; B = ws + w.b; C = ws + w.c;
    }
    return dstate == 64    ? mhost::launch_ssd_n<64>(a, x, B, C, w.pitch, s)
           : dstate == 128 ? mhost::launch_ssd_n<128>(a, x, B, C, w.pitch, s)
                           : mhost::launch_ssd_n<256>(a, x, B, C, w.pitch, s);
}

int mamba_ssd_update(float* state, const void* x, const void* delta, const float* A, const void* B, const void* C,
                     const float* D, const float* delta_bias, int flags, void* y, int batch, int nheads, int headdim,
                     int dstate, int io_dtype, void* stream) {
    if (io_dtype != MAMBA_F32 && io_dtype != MAMBA_BF16) return MAMBA_ERR_DTYPE;
    if (flags & ~MAMBA_FLAG_SOFTPLUS) return MAMBA_ERR_FLAGS;
    if (batch < 0 || nheads < 0 || headdim != mscan::kSsdP || !ssd_dstate(dstate)) return MAMBA_ERR_SHAPE;
    if (batch > 65535) return MAMBA_ERR_SHAPE;  // grid.y
    if (static_cast<long long>(nheads) * headdim > (1ll << 30)) return MAMBA_ERR_SHAPE;
    if (batch == 0 || nheads == 0) return MAMBA_OK;
    if (!state || !x || !delta || !A || !B || !C || !y) return MAMBA_ERR_NULL;
    const size_t es = dtype_size(io_dtype);
    const void* p16[] = {state, B, C};
    for (const void* p : p16)
        if (!aligned(p, 16)) return MAMBA_ERR_ALIGN;
    const void* pe[] = {x, delta, y};
    for (const void* p : pe)
        if (!aligned(p, es)) return MAMBA_ERR_ALIGN;
    if (!aligned(A, 4) || (D && !aligned(D, 4)) || (delta_bias && !aligned(delta_bias, 4))) return MAMBA_ERR_ALIGN;
    mscan::SsdUpdateArgs a;
    a.state = state; a.x = x; a.delta = delta; a.B = B; a.C = C; a.A = A; a.D = D; a.bias = delta_bias; a.y = y;
    a.batch = batch; a.nheads = nheads; a.headdim = headdim; a.softplus = (flags & MAMBA_FLAG_SOFTPLUS) != 0;
    if (!(a.err = device_error_word())) return MAMBA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (io_dtype == MAMBA_BF16) {
        if (dstate == 64) launch_ssd_update_n<__nv_bfloat16, 64>(a, s);
        else if (dstate == 128) launch_ssd_update_n<__nv_bfloat16, 128>(a, s);
        else launch_ssd_update_n<__nv_bfloat16, 256>(a, s);
    } else {
        if (dstate == 64) launch_ssd_update_n<float, 64>(a, s);
        else if (dstate == 128) launch_ssd_update_n<float, 128>(a, s);
        else launch_ssd_update_n<float, 256>(a, s);
    }
    return cudaGetLastError() == cudaSuccess ? MAMBA_OK : MAMBA_ERR_CUDA;
}

int mamba_check_device_error(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MAMBA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return MAMBA_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return MAMBA_ERR_CUDA;
        return v;
    }
    return MAMBA_OK;
}

const char* mamba_status_string(int status) {
    switch (status) {
        case MAMBA_OK: return "MAMBA_OK";
        case MAMBA_ERR_NULL: return "MAMBA_ERR_NULL: a required pointer is NULL";
        case MAMBA_ERR_SHAPE: return "MAMBA_ERR_SHAPE: unsupported or out-of-range size";
        case MAMBA_ERR_DTYPE: return "MAMBA_ERR_DTYPE: io_dtype is not MAMBA_F32 or MAMBA_BF16";
        case MAMBA_ERR_ALIGN: return "MAMBA_ERR_ALIGN: a base pointer is not aligned as required";
        case MAMBA_ERR_CUDA: return "MAMBA_ERR_CUDA: a CUDA call failed";
        case MAMBA_ERR_DEVICE_TIMEOUT: return "MAMBA_ERR_DEVICE_TIMEOUT: a kernel gave up waiting on its copies";
        case MAMBA_ERR_WORKSPACE: return "MAMBA_ERR_WORKSPACE: the workspace is smaller than mamba_scan_workspace_size";
        case MAMBA_ERR_FLAGS: return "MAMBA_ERR_FLAGS: an unknown flag bit, or one this entry point does not support";
        case MAMBA_ERR_DEVICE_BOUNDS: return "MAMBA_ERR_DEVICE_BOUNDS: a kernel computed an index outside a tensor";
        default: return "unknown mamba_status";
    }
}

int mamba_version(void) { return 300; }

int mamba_checked_bounds(void) { return mscan::kCheckBounds ? 1 : 0; }

}  // extern "C"
