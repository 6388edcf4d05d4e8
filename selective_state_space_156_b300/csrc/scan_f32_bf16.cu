// Scan kernels for f32 inputs and bf16 output (one translation unit per dtype pair keeps builds parallel).
#include "scan_kernels.cuh"

namespace ssm {
cudaError_t launch_scan_f32_bf16(const ScanKernelArgs& a, int zoh, cudaStream_t s) {
    return launch_scan_typed<F32, BF16>(a, zoh, s);
}
}  // namespace ssm
