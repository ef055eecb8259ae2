// Forward-scan kernels for state size N = 16 (all 16 flag combinations, fp32 and bf16 I/O).
#include "fwd_launch.cuh"

namespace mhost {
template int launch_scan_n<float, 16>(const mscan::ScanArgs&, const FwdInputs&, int, cudaStream_t);
template int launch_scan_n<__nv_bfloat16, 16>(const mscan::ScanArgs&, const FwdInputs&, int, cudaStream_t);
}  // namespace mhost
