// Definition of mhost::launch_bwd_n, included by the per-state-size files
// scan_bwd_n*.cu, each of which instantiates it for its own state size.
#pragma once

#include <type_traits>

#include "../../include/mamba_scan.h"
#include "host.h"

namespace mhost {

template <typename T, int NS>
int launch_bwd_n(const mscan::ScanBwdArgs& a, int flags, cudaStream_t stream) {
    const dim3 grid((a.dim + mscan::ScanBwdGeo<NS>::kCh - 1) / mscan::ScanBwdGeo<NS>::kCh, a.batch);
    auto go = [&](auto sp, auto hz, auto zo) {
        mscan::scan_bwd_kernel<T, NS, decltype(sp)::value, decltype(hz)::value, decltype(zo)::value>
            <<<grid, 32, 0, stream>>>(a);
    };
    using Y = std::true_type;
    using N = std::false_type;
    const bool hz = a.z != nullptr;
    auto pick_zoh = [&](auto sp, auto z) {
        if (flags & MAMBA_FLAG_ZOH) go(sp, z, Y{});
        else go(sp, z, N{});
    };
    auto pick_z = [&](auto sp) {
        if (hz) pick_zoh(sp, Y{});
        else pick_zoh(sp, N{});
    };
    if (flags & MAMBA_FLAG_SOFTPLUS) pick_z(Y{});
    else pick_z(N{});
    return cudaGetLastError() == cudaSuccess ? MAMBA_OK : MAMBA_ERR_CUDA;
}

}  // namespace mhost
