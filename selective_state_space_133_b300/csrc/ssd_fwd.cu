// SSD (Mamba-2 chunked form) kernels, state sizes 64, 128 and 256: tensor maps and launch.
#include <string.h>

#include "../../include/mamba_scan.h"
#include "host.h"

namespace mhost {

template <int NS>
int launch_ssd_n(const mscan::SsdArgs& a, const void* x, const void* B, const void* C, int pitch,
                 cudaStream_t stream) {
    CUtensorMap tm_x, tm_b, tm_c;
    memset(&tm_x, 0, sizeof(tm_x)); memset(&tm_b, 0, sizeof(tm_b)); memset(&tm_c, 0, sizeof(tm_c));
    if (a.seqlen > 0) {
        const auto ty = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;  // rows of 64 bf16 = 128 bytes
        const uint64_t dim = static_cast<uint64_t>(a.nheads) * mscan::kSsdP;
        const bool ok = make_map_3d(&tm_x, ty, 2, x, a.seqlen, dim, a.batch, pitch, mscan::kSsdQ, mscan::kSsdP, sw) &&
                        make_map_3d(&tm_b, ty, 2, B, a.seqlen, NS, a.batch, pitch, mscan::kSsdQ, NS, sw) &&
                        make_map_3d(&tm_c, ty, 2, C, a.seqlen, NS, a.batch, pitch, mscan::kSsdQ, NS, sw);
        if (!ok) return MAMBA_ERR_CUDA;
    }
    // the tiles need 1024-byte alignment inside the dynamic shared memory
    const size_t smem = sizeof(mscan::SsdSmem<NS>) + 1024;
    // two CTAs (110 KB each at N = 128) share an SM, one (177 KB) at N = 256:
    // ask for the whole carveout
    if (cudaFuncSetAttribute(mscan::ssd_fwd_kernel<NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess ||
        cudaFuncSetAttribute(mscan::ssd_fwd_kernel<NS>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return MAMBA_ERR_CUDA;
    const dim3 grid(a.nheads, a.batch);
    mscan::ssd_fwd_kernel<NS><<<grid, mscan::kSsdThreads, smem, stream>>>(a, tm_x, tm_b, tm_c);
    return cudaGetLastError() == cudaSuccess ? MAMBA_OK : MAMBA_ERR_CUDA;
}

template int launch_ssd_n<64>(const mscan::SsdArgs&, const void*, const void*, const void*, int, cudaStream_t);
template int launch_ssd_n<128>(const mscan::SsdArgs&, const void*, const void*, const void*, int, cudaStream_t);
template int launch_ssd_n<256>(const mscan::SsdArgs&, const void*, const void*, const void*, int, cudaStream_t);

}  // namespace mhost
