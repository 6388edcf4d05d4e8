// Host-side declarations shared by the translation units of libssm_b300.so.
#pragma once

#include <cstddef>
#include <string>
#include <utility>

#include <cuda_runtime.h>

#include "../../include/ssm_scan.h"

namespace ssm {

// Everything a scan launch needs, after host-side validation.
struct ScanKernelArgs {
    int Bsz, D, N, L;
    const void* u;
    const void* delta;
    const float* A;
    const void* Bm;
    const void* Cm;
    const float* Dskip;
    const float* delta_bias;
    const void* z;
    const float* conv_w;
    const float* conv_b;
    int conv_width;
    const void* conv_init;  // (rows, conv_width - 1) x before t = 0 (in dtype), or NULL for zeros
    const int* state_indices;  // (B) slot of each batch row in h0 / h_out / conv_init, or NULL (slot = b)
    float* h_all;              // (B, ceil(L / hall_every), D, N): the state after every hall_every-th step
                               // (entry c after step min(c hall_every + hall_every - 1, L - 1)), or NULL
    int hall_every;            // 1 (h_all) or SSM_CKPT_STEPS (h_ckpt)
    const float* h0;
    float* h_out;
    void* y;
    int softplus;
    int vec;       // 1: every (b, d) row of u/delta/z/y starts 16-byte aligned and L % 8 == 0
    int nseg;      // number of L segments (1 = one pass, no workspace)
    int seg_len;   // timesteps per segment (a multiple of 8); the last one may be shorter
    int seg0_len;  // kScanP16: > 0 when segment 0 has its own length (then [0, seg0_len), and seg_len steps
                   // per later segment) and runs its final pass in the split's first launch; 0 otherwise
    float* ws_h;     // (nseg - 1, B*D, N) end state of each segment but the last, from a zero start (with
                     // seg0_len > 0, entry 0 is segment 0's end state from h0)
    float* ws_dsum;  // (nseg - 1, B*D) sum of dt over each segment but the last
    float* ws_h0;    // (B*D, N) copy of h0 taken before any block may write h_out (h0 may alias h_out)
    int kind;        // kScanSeq, kScanP16 or kScanG4
    int lpc;         // kScanP16: lanes per channel (1, 2 or 4)
    int withhold;    // test only: block (0, 0) of the packed kernel's final pass never copies its first chunk
};

constexpr int kScanSeq = 0;  // one (b, d) row per thread, all states in registers (any dtype, any alignment)
constexpr int kScanP16 = 2;  // one row per thread, cp.async staging, packed fp32 pairs (bf16, aligned, N <= 16)
constexpr int kScanG4 = 1;   // four lanes per channel, tensor-core readout (bf16, aligned, 16 < N <= 64)

constexpr int kScanThreads = 128;  // channels per block in the scan kernels
constexpr int kScanChunk = 64;     // timesteps of B/C staged in shared memory at a time

// Launches the summary (when nseg > 1) and final scan kernels.  in/out: 0 = f32, 1 = bf16.
cudaError_t launch_scan(const ScanKernelArgs& a, int in_dtype, int out_dtype, int zoh, cudaStream_t stream);

// conv_final[s, i] = x_{L - W1 + i} of the batch row whose slot is s (from conv_init where that time is
// negative, zero without it), W1 = conv_width - 1; conv_final may be conv_init itself.
cudaError_t launch_conv_history(const void* x, const void* conv_init, void* conv_final, const int* state_indices,
                                int Bsz, int D, int L, int W1, int dtype, cudaStream_t stream);

cudaError_t launch_causal_conv1d(const void* x, const float* w, const float* b, void* y, int Bsz, int D, int L,
                                 int width, int silu, int dtype, cudaStream_t stream);

// One decode step after host-side validation.  x is u, or the conv input when conv_w != NULL.
struct DecodeStep {
    float* state;
    const void* x;
    const void* delta;
    const float* A;
    const void* Bm;
    const void* Cm;
    const float* Dskip;
    const float* delta_bias;
    const void* z;
    void* y;
    const float* conv_w;  // (D, conv_width) or NULL
    const float* conv_b;  // (D) or NULL
    void* conv_state;     // (B, D, conv_width - 1) or NULL (conv_width == 1)
    int conv_width;
    const int* state_indices;  // (B) slot of each batch row in state / conv_state, or NULL (slot = b)
    int Bsz, D, N, softplus, zoh, dtype;  // dtype: 0 = f32, 1 = bf16
};

cudaError_t launch_state_update(const DecodeStep& s, cudaStream_t stream);

// The streamed decode kernel (state_update_bulk.cu): eligibility, launch, and the flag its bounded
// waits set on a timeout (read and cleared by take_bulk_wait_error, which synchronises).
bool state_update_bulk_eligible(const DecodeStep& s);
cudaError_t launch_state_update_bulk(const DecodeStep& s, cudaStream_t stream);
cudaError_t take_bulk_wait_error(unsigned* flags);
// The packed scan kernel's flag for a chunk whose bulk tensor copies it stopped waiting for.
cudaError_t take_scan_wait_error(unsigned* flags);

// The backward pass (scan_bwd.cu), after host-side validation and zeroing of the accumulated outputs.
struct ScanBwdArgs {
    int Bsz, D, N, L;
    const void* u;
    const void* delta;
    const float* A;
    const void* Bm;
    const void* Cm;
    const float* Dskip;
    const float* delta_bias;
    const void* z;
    const float* conv_w;
    const float* conv_b;
    int conv_width;
    const void* conv_init;
    const float* h0;
    const float* h_ckpt;  // (B, ceil(L / 8), D, N) the forward's state after steps 7, 15, ... (and L - 1)
    const void* dy;
    const float* dh_out;  // (B, D, N) or NULL
    void* du;
    void* ddelta;
    void* dz;
    float* dA;
    float* dB;
    float* dC;
    float* dDskip;
    float* ddelta_bias;
    float* dconv_w;
    float* dconv_b;
    void* dconv_init;
    float* dh0;
    int softplus;
    int vec;  // every (b, d) row of u / delta / z / dy / du / ddelta / dz is 16-byte aligned and L % 8 == 0
    int nseg, seg_len;  // L split: segments of seg_len steps (a multiple of 64); 1 = none
    float* ws_g;        // (nseg - 1, B*D, N) adjoint each segment >= 1 hands back from a zero start
    float* ws_dsum;     // (nseg - 1, B*D) sum of dt over each segment >= 1
    float* ws_pend;     // (nseg - 1, B*D, 3) input gradients each segment >= 1 owes to the 3 steps before it
};

cudaError_t launch_scan_bwd(const ScanBwdArgs& a, int dtype, int zoh, cudaStream_t stream);
// Blocks of the backward kernel a problem of this kind would run that the device keeps resident at once.
cudaError_t scan_bwd_resident_blocks(int dtype, int N, int zoh, bool conv, int* slots);

// The Mamba-2 (SSD) chunked scan on the tensor cores (ssd_tc.cu), after host-side validation.
struct SsdArgs {
    int Bsz, H, G, L, N;       // batch, heads, groups, steps, state (64 or 128); head dim 64 (ssd_tc_supported)
    const void* x;             // (B, H*64, L) bf16
    const void* dt;            // (B, H, L) bf16
    const float* A;            // (H)
    const void* Bm;            // (B, G, L, N) bf16
    const void* Cm;            // (B, G, L, N) bf16
    const float* Dskip;        // (H) or NULL
    const float* dt_bias;      // (H) or NULL
    const void* z;             // (B, H*64, L) bf16 or NULL
    const float* h0;           // (B, H, 64, N) or NULL
    float* h_out;              // (B, H, 64, N) or NULL
    void* y;                   // (B, H*64, L) bf16
    int softplus, zoh;
    int withhold;              // test only: chunk 0's C is never copied (every wait for it runs out)
};

bool ssd_tc_supported(int N, int P);

// Test hook for the bounded waits (ssm_test_withhold_first_copy, a process-wide flag read at each launch):
// while set, the streamed decode kernel (block 0), the packed scan's TMA-staged final pass without an L
// split (block (0, 0)) and the SSD kernel (every block) leave out their first copy, so that waits for it
// run out after about a second and the kernel reports it through ssm_device_error.  Nothing faults or
// hangs; the outputs of the affected tiles are left unwritten.
bool withhold_first_copy();
cudaError_t launch_ssd_chunked(const SsdArgs& a, cudaStream_t stream);
// The SSD kernel's flag for a copy or MMA it stopped waiting for.
cudaError_t take_ssd_wait_error(unsigned* flags);

// cudaFuncSetAttribute(kernel, MaxDynamicSharedMemorySize, bytes) once per kernel, size and device, not
// on every launch (the call costs microseconds of host time; a prefill in chunks launches many times).
cudaError_t set_dynamic_smem(const void* kernel, int bytes);

// Launch with programmatic stream serialization (the kernel must call pdl_wait before its first global
// access), unless SSM_PDL=0; then a plain launch.
bool pdl_enabled();

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Blocks of `kernel` that the current device keeps resident at once (SMs x occupancy), cached per
// kernel, launch shape and device.
cudaError_t resident_blocks(const void* kernel, int threads, int smem_bytes, int* slots);

template <typename K>
inline cudaError_t set_dynamic_smem_once(K* kernel, int bytes) {
    return set_dynamic_smem(reinterpret_cast<const void*>(kernel), bytes);
}

// Launch geometry of each kernel kind, used by the host to plan the L split.
constexpr int kSeqChanPerBlock = 128, kSeqBlocksPerSM = 3, kSeqChunk = 64;
constexpr int kG4ChanPerBlock = 32, kG4BlocksPerSM = 7, kG4ChunkSteps = 32;
constexpr int kP16Threads_ = 128, kP16ChunkSteps = 48;  // kScanP16: channels per block = 128 / lpc

// Per-dtype-combination entry points defined in scan_<in>_<out>.cu.
cudaError_t launch_scan_f32_f32(const ScanKernelArgs& a, int zoh, cudaStream_t s);
cudaError_t launch_scan_bf16_bf16(const ScanKernelArgs& a, int zoh, cudaStream_t s);
cudaError_t launch_scan_bf16_f32(const ScanKernelArgs& a, int zoh, cudaStream_t s);
cudaError_t launch_scan_f32_bf16(const ScanKernelArgs& a, int zoh, cudaStream_t s);

}  // namespace ssm
