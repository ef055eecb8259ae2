// Backward-scan kernels for state size N = 32 (softplus x gate x ZOH gain, fp32 and bf16 I/O).
#include "bwd_launch.cuh"

namespace mhost {
template int launch_bwd_n<float, 32>(const mscan::ScanBwdArgs&, int, cudaStream_t);
template int launch_bwd_n<__nv_bfloat16, 32>(const mscan::ScanBwdArgs&, int, cudaStream_t);
}  // namespace mhost
