// Definition of mhost::launch_scan_n, included by the per-state-size files
// scan_fwd_n*.cu, each of which instantiates it for its own state size.
#pragma once

#include <string.h>

#include <type_traits>

#include "../../include/mamba_scan.h"
#include "host.h"

namespace mhost {

template <typename T, int NS>
int launch_scan_n(const mscan::ScanArgs& args, int flags, int nseg, bool state_pass, cudaStream_t stream) {
    using G = mscan::FwdGeo<NS>;
    constexpr size_t es = sizeof(T);
    mscan::ScanArgs a = args;
    CUtensorMap tm_u, tm_dl, tm_z, tm_b, tm_c;
    memset(&tm_u, 0, sizeof(tm_u)); memset(&tm_dl, 0, sizeof(tm_dl)); memset(&tm_z, 0, sizeof(tm_z));
    memset(&tm_b, 0, sizeof(tm_b)); memset(&tm_c, 0, sizeof(tm_c));
    // TMA needs every row stride to be a whole number of 16-byte units; other
    // lengths take the kernel's plain-load path (no tensor maps).
    a.plain = (static_cast<size_t>(a.seqlen) * es) % 16 != 0;
    if (a.seqlen > 0 && !a.plain) {
        const auto ty = mscan::Io<T>::kTmaType;
        const uint32_t bl = mscan::kTL, bd = G::kCh;
        bool ok = make_map_3d(&tm_u, ty, es, a.u, a.seqlen, a.dim, a.batch, a.seqlen, bl, bd) &&
                  make_map_3d(&tm_dl, ty, es, a.delta, a.seqlen, a.dim, a.batch, a.seqlen, bl, bd) &&
                  make_map_3d(&tm_b, ty, es, a.B, a.seqlen, NS, a.batch, a.seqlen, bl, NS) &&
                  make_map_3d(&tm_c, ty, es, a.C, a.seqlen, NS, a.batch, a.seqlen, bl, NS);
        if (ok && a.z && !state_pass) ok = make_map_3d(&tm_z, ty, es, a.z, a.seqlen, a.dim, a.batch, a.seqlen, bl, bd);
        if (!ok) return MAMBA_ERR_CUDA;
    }
    // the state-only pass runs every segment but the last
    const dim3 grid((a.dim + G::kCh - 1) / G::kCh, a.batch, state_pass ? nseg - 1 : nseg);
    auto go = [&](auto sp, auto hz, auto cv, auto zo, auto st) {
        mscan::scan_fwd_kernel<T, NS, decltype(sp)::value, decltype(hz)::value, decltype(cv)::value,
                               decltype(zo)::value, decltype(st)::value>
            <<<grid, mscan::kScanThreads, 0, stream>>>(a, tm_u, tm_dl, tm_z, tm_b, tm_c);
    };
    using Y = std::true_type;
    using N = std::false_type;
    const bool conv = a.conv_w != nullptr;
    const bool hz = a.z != nullptr;
    // 16 + 8 instantiations: softplus x gate x convolution x ZOH gain, and the
    // state-only pass (no gate) of each
    auto pick_pass = [&](auto sp, auto z, auto cv, auto zo) {
        if (state_pass) go(sp, N{}, cv, zo, Y{});
        else go(sp, z, cv, zo, N{});
    };
    auto pick_zoh = [&](auto sp, auto z, auto cv) {
        if (flags & MAMBA_FLAG_ZOH) pick_pass(sp, z, cv, Y{});
        else pick_pass(sp, z, cv, N{});
    };
    auto pick_conv = [&](auto sp, auto z) {
        if (conv) pick_zoh(sp, z, Y{});
        else pick_zoh(sp, z, N{});
    };
    auto pick_z = [&](auto sp) {
        if (hz && !state_pass) pick_conv(sp, Y{});
        else pick_conv(sp, N{});
    };
    if (flags & MAMBA_FLAG_SOFTPLUS) pick_z(Y{});
    else pick_z(N{});
    return cudaGetLastError() == cudaSuccess ? MAMBA_OK : MAMBA_ERR_CUDA;
}

}  // namespace mhost
