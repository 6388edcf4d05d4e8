// Scan kernels for f32 inputs and f32 output (one translation unit per dtype pair keeps builds parallel).
#include "scan_kernels.cuh"

namespace ssm {
cudaError_t launch_scan_f32_f32(const ScanKernelArgs& a, int zoh, cudaStream_t s) {
    return launch_scan_typed<F32, F32>(a, zoh, s);
}
}  // namespace ssm
