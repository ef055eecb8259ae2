// Host-side pieces shared by the library's translation units.
//
// The forward-scan kernels are instantiated per state size in their own files
// (scan_fwd_n8.cu ... scan_fwd_n64.cu, compiled in parallel); each of those
// files defines launch_scan_n for its state size and instantiates no other
// kernel; scan_bwd_n*.cu do the same for the backward (launch_bwd_n) and
// ssd_fwd.cu for the SSD kernels (launch_ssd_n).
// Everything else (argument checks, workspace layouts, the backward's B/C
// pack, the row copies of the SSD and the state update) lives in mamba_scan.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "scan_bwd.cuh"
#include "scan_fwd.cuh"
#include "ssd_fwd.cuh"

namespace mhost {

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// 3-D TMA tensor map over a tensor with extents (e0, e1, e2), e0 innermost, row
// pitch `pitch0` elements (>= e0) and plane pitch pitch0 * e1; box (b0, b1, 1).
// Defined in mamba_scan.cu. Returns false if the map cannot be encoded.
bool make_map_3d(CUtensorMap* m, CUtensorMapDataType t, size_t es, const void* base, uint64_t e0, uint64_t e1,
                 uint64_t e2, uint64_t pitch0, uint32_t b0, uint32_t b1,
                 CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE);

// Encodes the tensor maps and launches the forward kernel of state size NS
// (the instantiation picked by `flags`, bits MAMBA_FLAG_*, and by whether the
// convolution and z are given) on the inputs named in `a`, over `nseg`
// segments of a.seg_chunks chunks (nseg = 1, a.seg_chunks = 0: no split);
// `state_pass` launches the state-only pass of a split sequence instead.
// Returns a mamba_status.
template <typename T, int NS>
int launch_scan_n(const mscan::ScanArgs& a, int flags, int nseg, bool state_pass, cudaStream_t stream);

// Launches the backward kernel of state size NS picked by `flags` and by
// whether z is given (defined in bwd_launch.cuh). Returns a mamba_status.
template <typename T, int NS>
int launch_bwd_n(const mscan::ScanBwdArgs& a, int flags, cudaStream_t stream);

// Launches the SSD kernel of state size NS (64 or 128) on x, B and C at row
// pitch `pitch` elements (defined in ssd_fwd.cu). Returns a mamba_status.
template <int NS>
int launch_ssd_n(const mscan::SsdArgs& a, const void* x, const void* B, const void* C, int pitch,
                 cudaStream_t stream);

}  // namespace mhost
