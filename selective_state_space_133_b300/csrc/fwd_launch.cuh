// Definition of mhost::launch_scan_n, included by the per-state-size files
// scan_fwd_n*.cu, each of which instantiates it for its own state size.
#pragma once

#include <string.h>

#include <type_traits>

#include "../../include/mamba_scan.h"
#include "host.h"

namespace mhost {

template <typename T, int NS>
int launch_scan_n(const mscan::ScanArgs& a, const FwdInputs& in, int flags, cudaStream_t stream) {
    using G = mscan::FwdGeo<NS>;
    constexpr size_t es = sizeof(T);
    CUtensorMap tm_u, tm_dl, tm_z, tm_bc;
    memset(&tm_u, 0, sizeof(tm_u)); memset(&tm_dl, 0, sizeof(tm_dl));
    memset(&tm_z, 0, sizeof(tm_z)); memset(&tm_bc, 0, sizeof(tm_bc));
    if (a.seqlen > 0) {
        const auto ty = mscan::Io<T>::kTmaType;
        const uint32_t bl = mscan::kTL, bd = G::kCh;
        bool ok = make_map_3d(&tm_u, ty, es, in.u, a.seqlen, a.dim, a.batch, in.pitch, bl, bd) &&
                  make_map_3d(&tm_dl, ty, es, in.delta, a.seqlen, a.dim, a.batch, in.pitch, bl, bd) &&
                  make_map_3d(&tm_bc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, sizeof(float), in.bc, G::kBCW, in.Lp,
                              a.batch, G::kBCW, G::kBCW, bl);
        if (ok && in.z) ok = make_map_3d(&tm_z, ty, es, in.z, a.seqlen, a.dim, a.batch, in.pitch, bl, bd);
        if (!ok) return MAMBA_ERR_CUDA;
    }
    const dim3 grid((a.dim + G::kCh - 1) / G::kCh, a.batch);
    auto go = [&](auto sp, auto hz, auto cv, auto zo) {
        mscan::scan_fwd_kernel<T, NS, decltype(sp)::value, decltype(hz)::value, decltype(cv)::value,
                               decltype(zo)::value>
            <<<grid, mscan::kScanThreads, 0, stream>>>(a, tm_u, tm_dl, tm_z, tm_bc);
    };
    using Y = std::true_type;
    using N = std::false_type;
    const bool conv = a.conv_w != nullptr;
    const bool hz = in.z != nullptr;
    // 16 instantiations: softplus x gate x convolution x ZOH gain
    auto pick_zoh = [&](auto sp, auto z, auto cv) {
        if (flags & MAMBA_FLAG_ZOH) go(sp, z, cv, Y{});
        else go(sp, z, cv, N{});
    };
    auto pick_conv = [&](auto sp, auto z) {
        if (conv) pick_zoh(sp, z, Y{});
        else pick_zoh(sp, z, N{});
    };
    auto pick_z = [&](auto sp) {
        if (hz) pick_conv(sp, Y{});
        else pick_conv(sp, N{});
    };
    if (flags & MAMBA_FLAG_SOFTPLUS) pick_z(Y{});
    else pick_z(N{});
    return cudaGetLastError() == cudaSuccess ? MAMBA_OK : MAMBA_ERR_CUDA;
}

}  // namespace mhost
