// C ABI of libmambascan.so: argument validation, TMA tensor maps, dispatch.
//
// Declared in include/mamba_scan.h. Every check runs on the host before any
// launch; a rejected call launches nothing and writes nothing. The library
// allocates no device memory and keeps no state besides the device error word.
#include <cstring>
#include <mutex>

#include "../../include/mamba_scan.h"
#include "scan_fwd.cuh"
#include "state_update.cuh"

namespace {

using mscan::kDState;

constexpr int kRows = 16;    // channels per CTA (one warp, two lanes per channel)
constexpr int kTL = 16;      // steps per chunk

// TMA ring depth: two chunks of look-ahead on top of the three chunks a CTA
// works on (bf16: 27 KB of shared memory per CTA, 7 CTAs per SM).
template <typename T> constexpr int kStages = 5;
template <> constexpr int kStages<float> = 4;

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

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// 3-D map over a (d2, d1, d0) row-major tensor (d0 innermost) with box (b0, b1, 1).
bool make_map_3d(CUtensorMap* m, CUtensorMapDataType t, size_t es, const void* base, uint64_t d0, uint64_t d1,
                 uint64_t d2, uint32_t b0, uint32_t b1) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {d0 * es, d0 * d1 * es};
    const cuuint32_t box[3] = {b0, b1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, t, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T>
int launch_scan(const mscan::ScanArgs& a, cudaStream_t stream) {
    constexpr size_t es = sizeof(T);
    CUtensorMap tm_u, tm_dl, tm_z, tm_B, tm_C;
    memset(&tm_u, 0, sizeof(tm_u)); memset(&tm_dl, 0, sizeof(tm_dl)); memset(&tm_z, 0, sizeof(tm_z));
    memset(&tm_B, 0, sizeof(tm_B)); memset(&tm_C, 0, sizeof(tm_C));
    mscan::ScanArgs args = a;
    args.use_tma = (static_cast<uint64_t>(a.seqlen) * es) % 16 == 0 && a.seqlen > 0;
    if (args.use_tma) {
        const auto ty = mscan::Io<T>::kTmaType;
        bool ok = make_map_3d(&tm_u, ty, es, a.u, a.seqlen, a.dim, a.batch, kTL, kRows) &&
                  make_map_3d(&tm_dl, ty, es, a.delta, a.seqlen, a.dim, a.batch, kTL, kRows) &&
                  make_map_3d(&tm_B, ty, es, a.B, a.seqlen, kDState, a.batch, kTL, kDState) &&
                  make_map_3d(&tm_C, ty, es, a.C, a.seqlen, kDState, a.batch, kTL, kDState);
        if (ok && a.z) ok = make_map_3d(&tm_z, ty, es, a.z, a.seqlen, a.dim, a.batch, kTL, kRows);
        if (!ok) return MAMBA_ERR_CUDA;
    }
    const dim3 grid((a.dim + kRows - 1) / kRows, a.batch);
    constexpr int S = kStages<T>;
    if (a.softplus) {
        if (a.z) mscan::scan_fwd_kernel<T, kRows, kTL, S, true, true><<<grid, 32, 0, stream>>>(args, tm_u, tm_dl, tm_z, tm_B, tm_C);
        else     mscan::scan_fwd_kernel<T, kRows, kTL, S, true, false><<<grid, 32, 0, stream>>>(args, tm_u, tm_dl, tm_z, tm_B, tm_C);
    } else {
        if (a.z) mscan::scan_fwd_kernel<T, kRows, kTL, S, false, true><<<grid, 32, 0, stream>>>(args, tm_u, tm_dl, tm_z, tm_B, tm_C);
        else     mscan::scan_fwd_kernel<T, kRows, kTL, S, false, false><<<grid, 32, 0, stream>>>(args, tm_u, tm_dl, tm_z, tm_B, tm_C);
    }
    return cudaGetLastError() == cudaSuccess ? MAMBA_OK : MAMBA_ERR_CUDA;
}

template <typename T>
int launch_update(const mscan::UpdateArgs& a, cudaStream_t stream) {
    const long long rows = static_cast<long long>(a.batch) * a.dim;
    constexpr int kRowsPerBlock = mscan::kUpdateThreads / 4;
    const long long blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
    mscan::state_update_kernel<T><<<static_cast<unsigned>(blocks), mscan::kUpdateThreads, 0, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? MAMBA_OK : MAMBA_ERR_CUDA;
}

size_t dtype_size(int io_dtype) { return io_dtype == MAMBA_BF16 ? 2 : 4; }

}  // namespace

extern "C" {

int mamba_scan_fwd(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
                   const void* z, const float* delta_bias, int softplus_flag, void* y, float* final_state,
                   int batch, int dim, int seqlen, int dstate, int io_dtype, void* stream) {
    if (io_dtype != MAMBA_F32 && io_dtype != MAMBA_BF16) return MAMBA_ERR_DTYPE;
    if (batch < 0 || dim < 0 || seqlen < 0 || dstate != kDState) return MAMBA_ERR_SHAPE;
    if (batch > 65535) return MAMBA_ERR_SHAPE;  // grid.y
    const size_t es = dtype_size(io_dtype);
    // every flat index must fit in 63 bits of bytes, and TMA strides in 40 bits
    const unsigned long long elems = static_cast<unsigned long long>(batch) * dim * seqlen;
    if (dim > 0 && seqlen > 0 && elems / dim / seqlen != static_cast<unsigned long long>(batch)) return MAMBA_ERR_SHAPE;
    if (static_cast<unsigned long long>(seqlen) * dim * es >= (1ull << 40)) return MAMBA_ERR_SHAPE;
    if (batch == 0 || dim == 0) return MAMBA_OK;
    if (!A) return MAMBA_ERR_NULL;
    if (seqlen > 0 && (!u || !delta || !B || !C || !y)) return MAMBA_ERR_NULL;
    const void* p16[] = {u, delta, z, B, C, y, A, final_state};
    for (const void* p : p16)
        if (p && !aligned(p, 16)) return MAMBA_ERR_ALIGN;
    if ((D && !aligned(D, 4)) || (delta_bias && !aligned(delta_bias, 4))) return MAMBA_ERR_ALIGN;

    mscan::ScanArgs a;
    a.u = u; a.delta = delta; a.z = z; a.B = B; a.C = C; a.A = A; a.D = D; a.bias = delta_bias;
    a.y = y; a.final_state = final_state;
    a.batch = batch; a.dim = dim; a.seqlen = seqlen; a.softplus = softplus_flag != 0; a.use_tma = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return io_dtype == MAMBA_BF16 ? launch_scan<__nv_bfloat16>(a, s) : launch_scan<float>(a, s);
}

int mamba_state_update(float* state, const void* u, const void* delta, const float* A, const void* B, const void* C,
                       const float* D, const void* z, const float* delta_bias, int softplus_flag, void* y, int batch,
                       int dim, int dstate, int io_dtype, void* stream) {
    if (io_dtype != MAMBA_F32 && io_dtype != MAMBA_BF16) return MAMBA_ERR_DTYPE;
    if (batch < 0 || dim < 0 || dstate != kDState) return MAMBA_ERR_SHAPE;
    const unsigned long long rows = static_cast<unsigned long long>(batch) * dim;
    if (rows / 64 >= (1ull << 31)) return MAMBA_ERR_SHAPE;  // grid.x
    if (rows == 0) return MAMBA_OK;
    if (!state || !u || !delta || !A || !B || !C || !y) return MAMBA_ERR_NULL;
    const void* p16[] = {state, A};
    for (const void* p : p16)
        if (!aligned(p, 16)) return MAMBA_ERR_ALIGN;
    const size_t es = dtype_size(io_dtype);
    // B/C rows are read 4 elements at a time
    if (!aligned(B, 4 * es) || !aligned(C, 4 * es)) return MAMBA_ERR_ALIGN;
    const void* pe[] = {u, delta, z, y};
    for (const void* p : pe)
        if (p && !aligned(p, es)) return MAMBA_ERR_ALIGN;
    if ((D && !aligned(D, 4)) || (delta_bias && !aligned(delta_bias, 4))) return MAMBA_ERR_ALIGN;

    mscan::UpdateArgs a;
    a.state = state; a.u = u; a.delta = delta; a.z = z; a.B = B; a.C = C; a.A = A; a.D = D; a.bias = delta_bias;
    a.y = y; a.batch = batch; a.dim = dim; a.softplus = softplus_flag != 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return io_dtype == MAMBA_BF16 ? launch_update<__nv_bfloat16>(a, s) : launch_update<float>(a, s);
}

int mamba_check_device_error(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MAMBA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, mscan::g_device_error, sizeof(int)) != cudaSuccess) return MAMBA_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(mscan::g_device_error, &zero, sizeof(int)) != cudaSuccess) return MAMBA_ERR_CUDA;
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
        default: return "unknown mamba_status";
    }
}

int mamba_version(void) { return 100; }

}  // extern "C"
