// Scan kernels for bf16 inputs and bf16 output.  Aligned problems run the packed-pairs kernel with 1, 2
// or 4 lanes per channel (N <= 16) or the four-lanes-per-channel tensor-core kernel (16 < N <= 64); the
// rest run the element-wise one-row-per-thread kernel.
#include "scan_g4.cuh"
#include "scan_kernels.cuh"
#include "scan_p16.cuh"

namespace ssm {
cudaError_t launch_scan_bf16_bf16(const ScanKernelArgs& a, int zoh, cudaStream_t s) {
    if (a.kind == kScanP16) {
        if (a.N <= 4) return launch_p16<4, 1>(a, zoh, s);
        if (a.N <= 8) return a.lpc >= 2 ? launch_p16<8, 2>(a, zoh, s) : launch_p16<8, 1>(a, zoh, s);
        if (a.lpc >= 4) return launch_p16<16, 4>(a, zoh, s);
        if (a.lpc == 2) return launch_p16<16, 2>(a, zoh, s);
        return launch_p16<16, 1>(a, zoh, s);
    }
    if (a.kind == kScanG4) {
        if (a.N <= 32) return launch_g4_nsl<8>(a, zoh, s);
        return launch_g4_nsl<16>(a, zoh, s);
    }
    return launch_scan_typed<BF16, BF16>(a, zoh, s);
}

cudaError_t take_scan_wait_error(unsigned* flags) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_scan_wait_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_scan_wait_error, &zero, sizeof(unsigned));
}
}  // namespace ssm
