// Forward-scan kernels for state size N = 64 (all 16 flag combinations and their state-only passes, fp32 and bf16 I/O).
#include "fwd_launch.cuh"

namespace mhost {
template int launch_scan_n<float, 64>(const mscan::ScanArgs&, int, int, bool, cudaStream_t);
template int launch_scan_n<__nv_bfloat16, 64>(const mscan::ScanArgs&, int, int, bool, cudaStream_t);
}  // namespace mhost
