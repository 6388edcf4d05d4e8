// extern "C" entry points of libssm_b300.so: argument validation, launch-shape choice and dispatch.
// Declarations, argument meaning, layouts, ownership and error behaviour: include/ssm_scan.h.
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <string>

#include "ssm_internal.h"

namespace {

thread_local std::string g_last_error;

ssm_status fail(ssm_status code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

ssm_status cuda_status(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return SSM_OK;
    return fail(SSM_ERR_CUDA, "%s: CUDA error %d (%s)", what, (int)e, cudaGetErrorString(e));
}

size_t esize(int dtype) { return dtype == SSM_BF16 ? 2 : 4; }

bool overlaps(const void* a, size_t abytes, const void* b, size_t bbytes) {
    if (a == nullptr || b == nullptr) return false;
    uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    return n;
}

// Which kernel runs a problem: the four-lanes-per-channel kernel for aligned bf16-in/bf16-out
// problems (its tensor-core readout rounds h to tf32, fine for a bf16 result), the one-row-per-thread
// kernel otherwise.
bool aligned_rows(const ssm_scan_params* p) {
    const size_t ib = esize(p->in_dtype), ob = esize(p->out_dtype);
    return ((size_t)p->seqlen % 8 == 0) && aligned16(p->u) && aligned16(p->delta) && aligned16(p->y) &&
           (p->z == nullptr || aligned16(p->z)) && aligned16(p->Bm) && aligned16(p->Cm) && ib * 8 % 16 == 0 &&
           ob * 8 % 16 == 0;
}

int scan_kind(const ssm_scan_params* p) {
    // state slots are implemented by the element-wise kernel; the per-step state output by it and by the
    // packed kernel (16-byte-aligned h_all)
    if (p->state_indices != nullptr) return ssm::kScanSeq;
    const float* hs = p->h_all != nullptr ? p->h_all : p->h_ckpt;  // the state output (every step or every 8th)
    if (p->in_dtype == SSM_BF16 && p->out_dtype == SSM_BF16 && aligned_rows(p)) {
        if (p->dstate <= 16 && (hs == nullptr || aligned16(hs))) return ssm::kScanP16;
        if (p->dstate <= 64 && hs == nullptr) return ssm::kScanG4;
    }
    return ssm::kScanSeq;
}

struct KindGeom {
    int chan_per_block, blocks_per_sm, chunk;
};

// Resident blocks per SM of the packed kernel by lanes per channel (its launch bounds).
int p16_blocks_per_sm(int lpc) { return lpc == 1 ? 2 : (lpc == 2 ? 4 : 6); }  // registers, or shared memory (lpc 4)

KindGeom kind_geom(int kind, int lpc) {
    if (kind == ssm::kScanG4) return {ssm::kG4ChanPerBlock, ssm::kG4BlocksPerSM, ssm::kG4ChunkSteps};
    if (kind == ssm::kScanP16) return {ssm::kP16Threads_ / lpc, p16_blocks_per_sm(lpc), ssm::kP16ChunkSteps};
    return {ssm::kSeqChanPerBlock, ssm::kSeqBlocksPerSM, ssm::kSeqChunk};
}

// Lanes per channel of the packed kernel.  More lanes per channel give more warps (better latency
// hiding) at a higher per-step cost.  SSM_SCAN_LANES_PER_CHANNEL (1, 2 or 4), read once per process,
// overrides the choice (for comparisons).
int lpc_override() {
    static const int v = [] {
        const char* env = getenv("SSM_SCAN_LANES_PER_CHANNEL");
        const int x = env != nullptr ? atoi(env) : 0;
        return (x == 1 || x == 2 || x == 4) ? x : 0;
    }();
    return v;
}

int choose_lpc(const ssm_scan_params* p) {
    if (const int v = lpc_override()) return p->dstate <= 4 ? 1 : (p->dstate <= 8 && v > 2 ? 2 : v);
    return 1;  // measured fastest on the 8 x 4096 x 16 x 2048 and 1 x 5120 x 16 x 65536 workloads
}

// Segmenting of L.  One segment while the (b, channel-block) grid fills at least half of the GPU's
// resident block slots; otherwise L is cut into as many segments (each >= 256 steps) as still fit in
// one round of resident blocks, so the final pass never needs a second wave.
struct SegPlan {
    int nseg;
    int seg_len;
    int seg0_len;  // > 0: segment 0 has this length and runs its final pass beside the summaries
};

// A summary launch costs about this much of a final launch per step (percent; ncu on 2048-step calls on
// 5120 channels: 48.2 us for 272-step summaries against 60.4 us for 272-step final passes): segment 0,
// whose final pass runs beside the summaries, is this much shorter than the others so that both end
// together.
constexpr int kSummaryCostPct = 80;

SegPlan plan_segments(int kind, int lpc, int Bsz, int D, int L) {
    const KindGeom kg = kind_geom(kind, lpc);
    const int cpb = kg.chan_per_block, bps = kg.blocks_per_sm, chunk = kg.chunk;
    const long long blocks = (long long)((D + cpb - 1) / cpb) * Bsz;
    const long long slots = (long long)sm_count() * bps;
    SegPlan p{1, ((L + chunk - 1) / chunk) * chunk};
    if (blocks * 2 >= slots) return p;
    long long want = slots / blocks;
    const long long maxseg = L / 256;  // 256: 32 chained 2048-step calls on 5120 channels 4.55 -> 3.78 ms (512)
    if (want > maxseg) want = maxseg;
    if (want > 64) want = 64;
    if (want <= 1) return p;
    if (kind == ssm::kScanP16) {
        // Segment 0 needs no carry, so its final pass runs in the first launch beside the summaries of
        // segments 1 .. want - 1, and its end state is the first carry; the second launch runs the final
        // passes of segments 1 .. want.  That is want + 1 segments at want blocks per channel block in each
        // launch.  Segment starts need 8-step boundaries only (16-byte staged rows, 8-step groups and
        // checkpoints); segment 0 is shorter by the summary's cost.
        long long ls = ((100LL * L + 100LL * want + kSummaryCostPct - 1) / (100LL * want + kSummaryCostPct) + 7) / 8 * 8;
        long long l0 = L - want * ls;
        while (l0 < 8 && ls > 8) {
            ls -= 8;
            l0 = L - want * ls;
        }
        if (l0 >= 8) {
            p.nseg = (int)want + 1;
            p.seg_len = (int)ls;
            p.seg0_len = (int)l0;
            return p;
        }
    }
    const int seg = (int)(((L + want - 1) / want + chunk - 1) / chunk) * chunk;
    p.seg_len = seg;
    p.nseg = (L + seg - 1) / seg;
    return p;
}

// The plan of one call: state slots are never split (the split's h0 copy is indexed by batch row).
SegPlan scan_plan(const ssm_scan_params* p, int kind, int lpc) {
    if (p->state_indices != nullptr) {
        const int chunk = kind_geom(kind, lpc).chunk;
        return SegPlan{1, ((p->seqlen + chunk - 1) / chunk) * chunk};
    }
    return plan_segments(kind, lpc, p->batch, p->dim, p->seqlen);
}

size_t workspace_bytes_for(const ssm_scan_params* p, const SegPlan& sp) {
    if (sp.nseg <= 1) return 0;
    const size_t rows = (size_t)p->batch * p->dim;
    size_t bytes = (size_t)(sp.nseg - 1) * rows * ((size_t)p->dstate + 1) * sizeof(float);
    if (p->h0 != nullptr) bytes += rows * (size_t)p->dstate * sizeof(float);
    return bytes + 256;
}

bool dstate_supported(const ssm_scan_params* p) {
    if (p->dstate >= 1 && p->dstate <= 16) return true;
    return (p->dstate == 32 || p->dstate == 64) && scan_kind(p) == ssm::kScanG4;
}

ssm_status validate_scan(const ssm_scan_params* p) {
    if (p == nullptr) return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd: params is NULL");
    if (p->batch <= 0 || p->dim <= 0 || p->dstate <= 0 || p->seqlen <= 0)
        return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd: sizes must be positive (batch=%d dim=%d dstate=%d seqlen=%d)",
                    p->batch, p->dim, p->dstate, p->seqlen);
    if (p->batch > 65535) return fail(SSM_ERR_UNSUPPORTED, "ssm_scan_fwd: batch %d exceeds 65535", p->batch);
    if ((p->in_dtype != SSM_F32 && p->in_dtype != SSM_BF16) || (p->out_dtype != SSM_F32 && p->out_dtype != SSM_BF16))
        return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd: bad dtype (in=%d out=%d)", (int)p->in_dtype, (int)p->out_dtype);
    if (!p->u || !p->delta || !p->A || !p->Bm || !p->Cm || !p->y)
        return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd: u, delta, A, Bm, Cm and y are required");
    if ((p->delta_softplus != 0 && p->delta_softplus != 1) || (p->zoh != 0 && p->zoh != 1))
        return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd: delta_softplus and zoh must be 0 or 1");
    if (p->conv_w != nullptr && (p->conv_width < 1 || p->conv_width > 4))
        return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd: conv_width %d outside 1..4", p->conv_width);
    if (p->h_all != nullptr && p->h_ckpt != nullptr)
        return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd: h_all and h_ckpt are alternatives (give one)");
    if (p->h_ckpt != nullptr && p->state_indices != nullptr)
        return fail(SSM_ERR_UNSUPPORTED, "ssm_scan_fwd: h_ckpt is not offered with state_indices");
    if (!dstate_supported(p))
        return fail(SSM_ERR_UNSUPPORTED,
                    "ssm_scan_fwd: dstate %d not supported (1..16; 32 and 64 need bf16 in/out, 16-byte-aligned "
                    "rows, seqlen %% 8 == 0 and none of state_indices, h_all, h_ckpt)", p->dstate);
    const size_t rows = (size_t)p->batch * p->dim;
    if (rows * (size_t)p->seqlen >= ((size_t)1 << 40))
        return fail(SSM_ERR_UNSUPPORTED, "ssm_scan_fwd: batch*dim*seqlen too large");
    const size_t ib = esize(p->in_dtype), ob = esize(p->out_dtype);
    const size_t nbdl = rows * (size_t)p->seqlen;
    const size_t nbnl = (size_t)p->batch * p->dstate * p->seqlen;
    const size_t ybytes = nbdl * ob;
    if (overlaps(p->y, ybytes, p->u, nbdl * ib) || overlaps(p->y, ybytes, p->delta, nbdl * ib) ||
        overlaps(p->y, ybytes, p->z, nbdl * ib) || overlaps(p->y, ybytes, p->Bm, nbnl * ib) ||
        overlaps(p->y, ybytes, p->Cm, nbnl * ib))
        return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd: y overlaps an input");
    if (p->h_out != nullptr && overlaps(p->h_out, rows * p->dstate * 4, p->y, ybytes))
        return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd: h_out overlaps y");
    if (p->h_all != nullptr) {
        const size_t hb = nbdl * (size_t)p->dstate * 4;
        if (overlaps(p->h_all, hb, p->u, nbdl * ib) || overlaps(p->h_all, hb, p->delta, nbdl * ib) ||
            overlaps(p->h_all, hb, p->z, nbdl * ib) || overlaps(p->h_all, hb, p->Bm, nbnl * ib) ||
            overlaps(p->h_all, hb, p->Cm, nbnl * ib) || overlaps(p->h_all, hb, p->y, ybytes) ||
            (p->h_out && !p->state_indices && overlaps(p->h_all, hb, p->h_out, rows * p->dstate * 4)) ||
            (p->h0 && !p->state_indices && overlaps(p->h_all, hb, p->h0, rows * p->dstate * 4)))
            return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd: h_all overlaps another tensor");
    }
    if (p->h_ckpt != nullptr) {
        const size_t ck = (size_t)(p->seqlen + SSM_CKPT_STEPS - 1) / SSM_CKPT_STEPS;
        const size_t hb = rows * ck * (size_t)p->dstate * 4;
        if (overlaps(p->h_ckpt, hb, p->u, nbdl * ib) || overlaps(p->h_ckpt, hb, p->delta, nbdl * ib) ||
            overlaps(p->h_ckpt, hb, p->z, nbdl * ib) || overlaps(p->h_ckpt, hb, p->Bm, nbnl * ib) ||
            overlaps(p->h_ckpt, hb, p->Cm, nbnl * ib) || overlaps(p->h_ckpt, hb, p->y, ybytes) ||
            (p->h_out && overlaps(p->h_ckpt, hb, p->h_out, rows * p->dstate * 4)) ||
            (p->h0 && overlaps(p->h_ckpt, hb, p->h0, rows * p->dstate * 4)))
            return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd: h_ckpt overlaps another tensor");
    }
    if (p->conv_w != nullptr && p->conv_width > 1 && p->state_indices == nullptr) {
        const size_t cbytes = rows * (size_t)(p->conv_width - 1) * ib;
        if (p->conv_init != nullptr && (overlaps(p->conv_init, cbytes, p->y, ybytes) ||
                                        (p->h_out && overlaps(p->conv_init, cbytes, p->h_out, rows * p->dstate * 4))))
            return fail(SSM_ERR_INVALID_ARG, "ssm_scan_fwd: conv_init overlaps an output");
        if (p->conv_final != nullptr) {
            const void* f = p->conv_final;
            if (overlaps(f, cbytes, p->u, nbdl * ib) || overlaps(f, cbytes, p->delta, nbdl * ib) ||
                overlaps(f, cbytes, p->z, nbdl * ib) || overlaps(f, cbytes, p->Bm, nbnl * ib) ||
                overlaps(f, cbytes, p->Cm, nbnl * ib) || overlaps(f, cbytes, p->y, ybytes) ||
                (p->h_out && overlaps(f, cbytes, p->h_out, rows * p->dstate * 4)) ||
                (p->h0 && overlaps(f, cbytes, p->h0, rows * p->dstate * 4)) ||
                (p->conv_init && p->conv_init != f && overlaps(f, cbytes, p->conv_init, cbytes)))
                return fail(SSM_ERR_INVALID_ARG,
                            "ssm_scan_fwd: conv_final overlaps another tensor (it may only be conv_init itself)");
        }
    }
    return SSM_OK;
}

// The kernel arguments every scan entry point derives from the parameters the same way.
ssm::ScanKernelArgs scan_args(const ssm_scan_params* p) {
    ssm::ScanKernelArgs a{};
    a.Bsz = p->batch; a.D = p->dim; a.N = p->dstate; a.L = p->seqlen;
    a.u = p->u; a.delta = p->delta; a.A = p->A; a.Bm = p->Bm; a.Cm = p->Cm;
    a.Dskip = p->Dskip; a.delta_bias = p->delta_bias; a.z = p->z;
    a.conv_w = p->conv_w; a.conv_b = p->conv_w ? p->conv_b : nullptr; a.conv_width = p->conv_w ? p->conv_width : 0;
    a.conv_init = (p->conv_w && p->conv_width > 1) ? p->conv_init : nullptr;
    a.state_indices = p->state_indices;
    a.h_all = p->h_all != nullptr ? p->h_all : p->h_ckpt;
    a.hall_every = p->h_ckpt != nullptr ? SSM_CKPT_STEPS : 1;
    a.h0 = p->h0; a.h_out = p->h_out; a.y = p->y;
    a.softplus = p->delta_softplus;
    a.vec = aligned_rows(p);
    a.kind = scan_kind(p);
    a.lpc = choose_lpc(p);
    return a;
}

// The scan launches, then (when asked) the conv-history copy, which runs after the scan so that a
// conv_final aliasing conv_init is only written once every block has read its history.
ssm_status launch_scan_and_history(const ssm::ScanKernelArgs& a, const ssm_scan_params* p, ssm_stream_t stream,
                                   const char* who) {
    cudaError_t e = ssm::launch_scan(a, (int)p->in_dtype, (int)p->out_dtype, p->zoh, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_status(e, who);
    if (p->conv_w != nullptr && p->conv_width > 1 && p->conv_final != nullptr) {
        e = ssm::launch_conv_history(p->u, a.conv_init, p->conv_final, p->state_indices, p->batch, p->dim,
                                     p->seqlen, p->conv_width - 1, (int)p->in_dtype, (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_status(e, who);
    }
    return SSM_OK;
}

// ---------------------------------------------------------------------------------------------
// Scratch for ssm_scan_fwd_static: a fixed buffer in the library's own device memory, for callers
// that cannot allocate.  Every GPU that loads the library holds these bytes until the process exits.
// ---------------------------------------------------------------------------------------------
constexpr size_t kStaticScratchBytes = (size_t)4 << 20;  // 4 MiB
constexpr int kStaticScratchMaxDevices = 64;

std::mutex g_static_scratch_mu;
void* g_static_scratch_addr[kStaticScratchMaxDevices] = {};
void* g_static_scratch_ctx[kStaticScratchMaxDevices] = {};  // the context the address was taken in

// The calling thread's current driver context (cuCtxGetCurrent, looked up through the runtime so that
// the library does not link against libcuda), or nullptr when it cannot be had.
void* current_context() {
    using Fn = int (*)(void**);
    static Fn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<Fn>(p);
        return static_cast<Fn>(nullptr);
    }();
    void* ctx = nullptr;
    if (fn == nullptr || fn(&ctx) != 0) return nullptr;
    return ctx;
}

}  // namespace

static __device__ __align__(256) unsigned char ssm_static_scratch[kStaticScratchBytes];

namespace {

// Device address of ssm_static_scratch on the current device.  The host-side name of the array is
// only a stand-in, so the address is asked of the runtime once per device, with that device current,
// and cached.
ssm_status static_scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e, "ssm_scan_fwd_static: cudaGetDevice");
    if (dev < 0 || dev >= kStaticScratchMaxDevices)
        return fail(SSM_ERR_UNSUPPORTED, "ssm_scan_fwd_static: device %d is beyond the %d devices it tracks", dev,
                    kStaticScratchMaxDevices);
    std::lock_guard<std::mutex> lock(g_static_scratch_mu);
    // asked again when the device's context is not the one the address was taken in (after a
    // cudaDeviceReset the module is loaded anew and the old address is stale)
    void* ctx = current_context();
    if (g_static_scratch_addr[dev] == nullptr || ctx == nullptr || ctx != g_static_scratch_ctx[dev]) {
        void* addr = nullptr;
        e = cudaGetSymbolAddress(&addr, ssm_static_scratch);
        if (e != cudaSuccess) return cuda_status(e, "ssm_scan_fwd_static: cudaGetSymbolAddress");
        if (addr == nullptr) return fail(SSM_ERR_CUDA, "ssm_scan_fwd_static: no device address for the scratch buffer");
        g_static_scratch_addr[dev] = addr;
        g_static_scratch_ctx[dev] = current_context();
    }
    *out = g_static_scratch_addr[dev];
    return SSM_OK;
}

}  // namespace

extern "C" {

const char* ssm_last_error(void) { return g_last_error.c_str(); }

const char* ssm_version(void) { return "ssm_b300 0.1 (sm_103a)"; }

}  // extern "C"

namespace {

// The backward's L split: as for the forward (a split only when the (b, channel-block) grid fills less
// than half the resident block slots, so that the split grid still runs in one wave), with the backward
// kernel's 128 channels per block and the resident blocks the device reports for the instantiation
// that will run; segments of a multiple of 64 steps.
SegPlan bwd_plan(const ssm_scan_bwd_params* p) {
    const int cpb = 128, chunk = 64;
    const long long blocks = (long long)((p->dim + cpb - 1) / cpb) * p->batch;
    int rs = 0;
    if (ssm::scan_bwd_resident_blocks((int)p->in_dtype, p->dstate, p->zoh, p->conv_w != nullptr, &rs) !=
            cudaSuccess ||
        rs <= 0)
        rs = sm_count() * 2;
    const long long slots = rs;
    SegPlan sp{1, ((p->seqlen + chunk - 1) / chunk) * chunk};
    if (blocks * 2 >= slots) return sp;
    long long want = slots / blocks;
    if (want > p->seqlen / 512) want = p->seqlen / 512;
    if (want > 64) want = 64;
    if (want <= 1) return sp;
    const int seg = (int)(((p->seqlen + want - 1) / want + chunk - 1) / chunk) * chunk;
    sp.seg_len = seg;
    sp.nseg = (p->seqlen + seg - 1) / seg;
    return sp;
}

size_t bwd_workspace_bytes(const ssm_scan_bwd_params* p, const SegPlan& sp) {
    if (sp.nseg <= 1) return 0;
    const size_t rows = (size_t)p->batch * p->dim;
    return (size_t)(sp.nseg - 1) * rows * ((size_t)p->dstate + 1 + 3) * sizeof(float) + 3 * 256;
}

ssm_status validate_bwd(const ssm_scan_bwd_params* p) {
    const char* who = "ssm_scan_bwd";
    if (p == nullptr) return fail(SSM_ERR_INVALID_ARG, "%s: params is NULL", who);
    if (p->batch <= 0 || p->dim <= 0 || p->dstate <= 0 || p->seqlen <= 0)
        return fail(SSM_ERR_INVALID_ARG, "%s: sizes must be positive", who);
    if (p->batch > 65535) return fail(SSM_ERR_UNSUPPORTED, "%s: batch %d exceeds 65535", who, p->batch);
    if (p->dstate > 16) return fail(SSM_ERR_UNSUPPORTED, "%s: dstate %d not supported (1..16)", who, p->dstate);
    if (p->in_dtype != SSM_F32 && p->in_dtype != SSM_BF16) return fail(SSM_ERR_INVALID_ARG, "%s: bad dtype", who);
    if ((p->delta_softplus != 0 && p->delta_softplus != 1) || (p->zoh != 0 && p->zoh != 1))
        return fail(SSM_ERR_INVALID_ARG, "%s: delta_softplus and zoh must be 0 or 1", who);
    if (!p->u || !p->delta || !p->A || !p->Bm || !p->Cm || !p->h_ckpt || !p->dy || !p->du || !p->ddelta || !p->dA ||
        !p->dB || !p->dC)
        return fail(SSM_ERR_INVALID_ARG, "%s: u, delta, A, Bm, Cm, h_ckpt, dy, du, ddelta, dA, dB and dC are required",
                    who);
    if (p->z && !p->dz) return fail(SSM_ERR_INVALID_ARG, "%s: dz is required with z", who);
    if (p->conv_w && (p->conv_width < 1 || p->conv_width > 4))
        return fail(SSM_ERR_INVALID_ARG, "%s: conv_width %d outside 1..4", who, p->conv_width);
    const size_t rows = (size_t)p->batch * p->dim, nbdl = rows * p->seqlen;
    const size_t eb = esize(p->in_dtype);
    const size_t nbnl = (size_t)p->batch * p->dstate * p->seqlen;
    const size_t W = p->conv_w ? (size_t)p->conv_width : 0, W1 = W > 0 ? W - 1 : 0;  // conv taps, history
    struct Range { const void* p; size_t n; };
    const Range ins[] = {{p->u, nbdl * eb}, {p->delta, nbdl * eb}, {p->z, nbdl * eb}, {p->Bm, nbnl * eb},
                         {p->Cm, nbnl * eb}, {p->dy, nbdl * eb},
                         {p->h_ckpt, rows * (size_t)((p->seqlen + SSM_CKPT_STEPS - 1) / SSM_CKPT_STEPS) * p->dstate * 4},
                         {p->A, (size_t)p->dim * p->dstate * 4}, {p->h0, rows * p->dstate * 4},
                         {p->Dskip, (size_t)p->dim * 4}, {p->delta_bias, (size_t)p->dim * 4},
                         {p->conv_w, (size_t)p->dim * W * 4}, {p->conv_b, W ? (size_t)p->dim * 4 : 0},
                         {p->conv_init, rows * W1 * eb}, {p->dh_out, rows * p->dstate * 4}};
    const Range outs[] = {{p->du, nbdl * eb}, {p->ddelta, nbdl * eb}, {p->dz, nbdl * eb},
                          {p->dA, (size_t)p->dim * p->dstate * 4}, {p->dB, nbnl * 4}, {p->dC, nbnl * 4},
                          {p->dDskip, (size_t)p->dim * 4}, {p->ddelta_bias, (size_t)p->dim * 4},
                          {p->dconv_w, (size_t)p->dim * W * 4}, {p->dconv_b, W ? (size_t)p->dim * 4 : 0},
                          {p->dconv_init, rows * W1 * eb}, {p->dh0, rows * p->dstate * 4}};
    for (const Range& o : outs) {
        if (!o.p) continue;
        for (const Range& i : ins)
            if (overlaps(o.p, o.n, i.p, i.n)) return fail(SSM_ERR_INVALID_ARG, "%s: an output overlaps an input", who);
        for (const Range& q : outs)
            if (&q != &o && overlaps(o.p, o.n, q.p, q.n))
                return fail(SSM_ERR_INVALID_ARG, "%s: two outputs overlap", who);
    }
    return SSM_OK;
}

}  // namespace

extern "C" {

size_t ssm_scan_bwd_workspace_size(const ssm_scan_bwd_params* p) {
    if (validate_bwd(p) != SSM_OK) return 0;
    return bwd_workspace_bytes(p, bwd_plan(p));
}

ssm_status ssm_scan_bwd(const ssm_scan_bwd_params* p, ssm_stream_t stream) {
    const char* who = "ssm_scan_bwd";
    ssm_status vs = validate_bwd(p);
    if (vs != SSM_OK) return vs;
    const size_t rows = (size_t)p->batch * p->dim;
    const size_t eb = esize(p->in_dtype);
    const size_t nbnl = (size_t)p->batch * p->dstate * p->seqlen;
    struct Range { const void* p; size_t n; };
    ssm::ScanBwdArgs a{};
    a.Bsz = p->batch; a.D = p->dim; a.N = p->dstate; a.L = p->seqlen;
    a.u = p->u; a.delta = p->delta; a.A = p->A; a.Bm = p->Bm; a.Cm = p->Cm; a.Dskip = p->Dskip;
    a.delta_bias = p->delta_bias; a.z = p->z; a.conv_w = p->conv_w; a.conv_b = p->conv_w ? p->conv_b : nullptr;
    a.conv_width = p->conv_w ? p->conv_width : 0;
    a.conv_init = (p->conv_w && p->conv_width > 1) ? p->conv_init : nullptr;
    a.h0 = p->h0; a.h_ckpt = p->h_ckpt; a.dy = p->dy; a.dh_out = p->dh_out;
    a.du = p->du; a.ddelta = p->ddelta; a.dz = p->z ? p->dz : nullptr; a.dA = p->dA; a.dB = p->dB; a.dC = p->dC;
    a.dDskip = p->Dskip ? p->dDskip : nullptr; a.ddelta_bias = p->delta_bias ? p->ddelta_bias : nullptr;
    a.dconv_w = p->conv_w ? p->dconv_w : nullptr; a.dconv_b = (p->conv_w && p->conv_b) ? p->dconv_b : nullptr;
    a.dconv_init = (p->conv_w && p->conv_width > 1) ? p->dconv_init : nullptr;
    a.dh0 = p->dh0;
    a.softplus = p->delta_softplus;
    const bool a16 = ((size_t)p->seqlen * eb) % 16 == 0 && aligned16(p->u) && aligned16(p->delta) &&
                     aligned16(p->dy) && aligned16(p->du) && aligned16(p->ddelta) && (!p->z || aligned16(p->z)) &&
                     (!p->z || aligned16(p->dz)) && p->seqlen % 8 == 0;
    a.vec = a16 ? 1 : 0;
    SegPlan sp = bwd_plan(p);
    if (sp.nseg > 1 && (p->workspace == nullptr || p->workspace_bytes < bwd_workspace_bytes(p, sp)))
        sp = SegPlan{1, ((p->seqlen + 63) / 64) * 64};
    a.nseg = sp.nseg;
    a.seg_len = sp.seg_len;
    if (sp.nseg > 1) {
        uintptr_t base = (reinterpret_cast<uintptr_t>(p->workspace) + 255) & ~(uintptr_t)255;
        float* w = reinterpret_cast<float*>(base);
        a.ws_g = w;
        w += (size_t)(sp.nseg - 1) * rows * p->dstate;
        w = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(w) + 255) & ~(uintptr_t)255);
        a.ws_dsum = w;
        w += (size_t)(sp.nseg - 1) * rows;
        w = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(w) + 255) & ~(uintptr_t)255);
        a.ws_pend = w;
    }
    cudaStream_t st = (cudaStream_t)stream;
    // the accumulated outputs start from zero
    const Range acc[] = {{a.dA, (size_t)p->dim * p->dstate * 4}, {a.dB, nbnl * 4}, {a.dC, nbnl * 4},
                         {a.dDskip, (size_t)p->dim * 4}, {a.ddelta_bias, (size_t)p->dim * 4},
                         {a.dconv_w, (size_t)p->dim * (p->conv_w ? p->conv_width : 0) * 4},
                         {a.dconv_b, (size_t)p->dim * 4}};
    for (const Range& r : acc) {
        if (!r.p || r.n == 0) continue;
        cudaError_t e = cudaMemsetAsync(const_cast<void*>(r.p), 0, r.n, st);
        if (e != cudaSuccess) return cuda_status(e, who);
    }
    return cuda_status(ssm::launch_scan_bwd(a, (int)p->in_dtype, p->zoh, st), who);
}

ssm_status ssm_device_error(unsigned* flags) {
    if (flags == nullptr) return fail(SSM_ERR_INVALID_ARG, "ssm_device_error: flags is NULL");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_status(e, "ssm_device_error: cudaDeviceSynchronize");
    unsigned dec = 0, scan = 0, ssd = 0;
    e = ssm::take_bulk_wait_error(&dec);
    if (e != cudaSuccess) return cuda_status(e, "ssm_device_error: reading the decode flag");
    e = ssm::take_scan_wait_error(&scan);
    if (e != cudaSuccess) return cuda_status(e, "ssm_device_error: reading the scan flag");
    e = ssm::take_ssd_wait_error(&ssd);
    if (e != cudaSuccess) return cuda_status(e, "ssm_device_error: reading the SSD flag");
    *flags = (dec ? 1u : 0u) | (scan ? 2u : 0u) | (ssd ? 4u : 0u);
    return SSM_OK;
}

size_t ssm_scan_workspace_size(const ssm_scan_params* p) {
    if (validate_scan(p) != SSM_OK) return 0;
    return workspace_bytes_for(p, scan_plan(p, scan_kind(p), choose_lpc(p)));
}

ssm_status ssm_scan_fwd(const ssm_scan_params* p, ssm_stream_t stream) {
    ssm_status st = validate_scan(p);
    if (st != SSM_OK) return st;

    ssm::ScanKernelArgs a = scan_args(p);

    SegPlan sp = scan_plan(p, a.kind, a.lpc);
    const size_t need = workspace_bytes_for(p, sp);
    if (sp.nseg > 1 && (p->workspace == nullptr || p->workspace_bytes < need)) {
        const int chunk = kind_geom(a.kind, a.lpc).chunk;
        sp = SegPlan{1, ((p->seqlen + chunk - 1) / chunk) * chunk};
    }
    a.nseg = sp.nseg;
    a.seg_len = sp.seg_len;
    a.seg0_len = sp.seg0_len;
    if (sp.nseg > 1) {
        uintptr_t base = (reinterpret_cast<uintptr_t>(p->workspace) + 255) & ~(uintptr_t)255;
        const size_t rows = (size_t)p->batch * p->dim;
        float* w = reinterpret_cast<float*>(base);
        a.ws_dsum = w;
        a.ws_h = w + (size_t)(sp.nseg - 1) * rows;
        a.ws_h0 = p->h0 != nullptr ? a.ws_h + (size_t)(sp.nseg - 1) * rows * p->dstate : nullptr;
    }
    return launch_scan_and_history(a, p, stream, "ssm_scan_fwd launch");
}

ssm_status causal_conv1d_fwd(const void* x, const float* w, const float* b, void* y, int batch, int dim, int seqlen,
                             int width, int silu, ssm_dtype dtype, ssm_stream_t stream) {
    if (!x || !w || !y) return fail(SSM_ERR_INVALID_ARG, "causal_conv1d_fwd: x, w and y are required");
    if (batch <= 0 || dim <= 0 || seqlen <= 0)
        return fail(SSM_ERR_INVALID_ARG, "causal_conv1d_fwd: sizes must be positive");
    if (batch > 65535) return fail(SSM_ERR_UNSUPPORTED, "causal_conv1d_fwd: batch %d exceeds 65535", batch);
    if (width < 1 || width > 4) return fail(SSM_ERR_INVALID_ARG, "causal_conv1d_fwd: width %d outside 1..4", width);
    if (silu != 0 && silu != 1) return fail(SSM_ERR_INVALID_ARG, "causal_conv1d_fwd: silu must be 0 or 1");
    if (dtype != SSM_F32 && dtype != SSM_BF16) return fail(SSM_ERR_INVALID_ARG, "causal_conv1d_fwd: bad dtype");
    const size_t bytes = (size_t)batch * dim * seqlen * esize(dtype);
    if (overlaps(x, bytes, y, bytes)) return fail(SSM_ERR_INVALID_ARG, "causal_conv1d_fwd: y overlaps x");
    return cuda_status(ssm::launch_causal_conv1d(x, w, b, y, batch, dim, seqlen, width, silu, (int)dtype,
                                                 (cudaStream_t)stream),
                       "causal_conv1d_fwd launch");
}

}  // extern "C"

namespace {

// Host-side checks and launch of one decode step (ssm_state_update and ssm_state_update_conv).
ssm_status run_decode_step(const ssm::DecodeStep& st, ssm_dtype dtype, const char* who, cudaStream_t stream) {
    if (!st.state || !st.x || !st.delta || !st.A || !st.Bm || !st.Cm || !st.y)
        return fail(SSM_ERR_INVALID_ARG, "%s: state, x (u), delta, A, Bm, Cm and y are required", who);
    if (st.Bsz <= 0 || st.D <= 0 || st.N <= 0) return fail(SSM_ERR_INVALID_ARG, "%s: sizes must be positive", who);
    if (st.Bsz > 65535) return fail(SSM_ERR_UNSUPPORTED, "%s: batch %d exceeds 65535", who, st.Bsz);
    if (!(st.N <= 16 || st.N == 32 || st.N == 64))
        return fail(SSM_ERR_UNSUPPORTED, "%s: dstate %d not supported (1..16, 32, 64)", who, st.N);
    if ((st.softplus != 0 && st.softplus != 1) || (st.zoh != 0 && st.zoh != 1))
        return fail(SSM_ERR_INVALID_ARG, "%s: delta_softplus and zoh must be 0 or 1", who);
    if (dtype != SSM_F32 && dtype != SSM_BF16) return fail(SSM_ERR_INVALID_ARG, "%s: bad dtype", who);
    if (st.conv_w != nullptr) {
        if (st.conv_width < 1 || st.conv_width > 4)
            return fail(SSM_ERR_INVALID_ARG, "%s: conv_width %d outside 1..4", who, st.conv_width);
        if (st.conv_width > 1 && st.conv_state == nullptr)
            return fail(SSM_ERR_INVALID_ARG, "%s: conv_state is required when conv_width > 1", who);
    }
    const size_t bd = (size_t)st.Bsz * st.D * esize(dtype);
    const size_t bn = (size_t)st.Bsz * st.N * esize(dtype);
    // with state slots the cache holds an unknown number of slots: its checks below cover one slot per row
    const size_t sb = (size_t)st.Bsz * st.D * st.N * 4;
    const void* y = st.y;
    if (overlaps(y, bd, st.x, bd) || overlaps(y, bd, st.delta, bd) || overlaps(y, bd, st.z, bd) ||
        overlaps(y, bd, st.Bm, bn) || overlaps(y, bd, st.Cm, bn) || overlaps(y, bd, st.state, sb))
        return fail(SSM_ERR_INVALID_ARG, "%s: y overlaps an input or the state", who);
    if (st.conv_w != nullptr && st.conv_width > 1) {
        const size_t cb = (size_t)st.Bsz * st.D * (st.conv_width - 1) * esize(dtype);
        const void* c = st.conv_state;
        if (overlaps(c, cb, st.x, bd) || overlaps(c, cb, st.delta, bd) || overlaps(c, cb, st.z, bd) ||
            overlaps(c, cb, st.Bm, bn) || overlaps(c, cb, st.Cm, bn) || overlaps(c, cb, st.state, sb) ||
            overlaps(c, cb, y, bd))
            return fail(SSM_ERR_INVALID_ARG, "%s: conv_state overlaps another tensor", who);
    }
    return cuda_status(ssm::launch_state_update(st, stream), who);
}

ssm::DecodeStep decode_step(float* state, const void* x, const void* delta, const float* A, const void* Bm,
                            const void* Cm, const float* Dskip, const float* delta_bias, const void* z, void* y,
                            int batch, int dim, int dstate, int delta_softplus, int zoh, ssm_dtype dtype) {
    ssm::DecodeStep st{};
    st.state = state; st.x = x; st.delta = delta; st.A = A; st.Bm = Bm; st.Cm = Cm;
    st.Dskip = Dskip; st.delta_bias = delta_bias; st.z = z; st.y = y;
    st.Bsz = batch; st.D = dim; st.N = dstate; st.softplus = delta_softplus; st.zoh = zoh; st.dtype = (int)dtype;
    st.conv_width = 1;
    return st;
}

}  // namespace

extern "C" {

ssm_status ssm_state_update(float* state, const void* u, const void* delta, const float* A, const void* Bm,
                            const void* Cm, const float* Dskip, const float* delta_bias, const void* z, void* y,
                            int batch, int dim, int dstate, int delta_softplus, int zoh, ssm_dtype dtype,
                            ssm_stream_t stream) {
    const ssm::DecodeStep st = decode_step(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y, batch, dim, dstate,
                                           delta_softplus, zoh, dtype);
    return run_decode_step(st, dtype, "ssm_state_update", (cudaStream_t)stream);
}

ssm_status ssm_state_update_conv(const ssm_step_params* p, ssm_stream_t stream) {
    if (p == nullptr) return fail(SSM_ERR_INVALID_ARG, "ssm_state_update_conv: params is NULL");
    ssm::DecodeStep st = decode_step(p->state, p->x, p->delta, p->A, p->Bm, p->Cm, p->Dskip, p->delta_bias, p->z,
                                     p->y, p->batch, p->dim, p->dstate, p->delta_softplus, p->zoh, p->dtype);
    if (p->conv_w != nullptr) {
        st.conv_w = p->conv_w;
        st.conv_b = p->conv_b;
        st.conv_width = p->conv_width;
        st.conv_state = p->conv_width > 1 ? p->conv_state : nullptr;
    }
    st.state_indices = p->state_indices;
    return run_decode_step(st, p->dtype, "ssm_state_update_conv", (cudaStream_t)stream);
}

ssm_status ssm_scan_fwd_static(const ssm_scan_params* p, ssm_stream_t stream) {
    ssm_status st = validate_scan(p);
    if (st != SSM_OK) return st;

    ssm::ScanKernelArgs a = scan_args(p);

    // the same launch plan as ssm_scan_fwd with a large enough workspace; p->workspace is ignored
    const SegPlan sp = scan_plan(p, a.kind, a.lpc);
    const size_t need = workspace_bytes_for(p, sp);
    if (need > kStaticScratchBytes)
        return fail(SSM_ERR_UNSUPPORTED,
                    "ssm_scan_fwd_static: this problem needs %zu bytes of scratch, more than the %zu-byte static "
                    "buffer; call ssm_scan_fwd with a caller workspace instead",
                    need, kStaticScratchBytes);
    a.nseg = sp.nseg;
    a.seg_len = sp.seg_len;
    a.seg0_len = sp.seg0_len;
    if (sp.nseg > 1) {
        // Nothing here has to start at zero: the first launch of this call writes every word of the
        // scratch that its final pass reads (segment sums, segment end states, the copy of h0 where it is
        // used).
        void* base = nullptr;
        st = static_scratch_address(&base);
        if (st != SSM_OK) return st;
        const size_t rows = (size_t)p->batch * p->dim;
        float* w = reinterpret_cast<float*>(base);
        a.ws_dsum = w;
        a.ws_h = w + (size_t)(sp.nseg - 1) * rows;
        a.ws_h0 = p->h0 != nullptr ? a.ws_h + (size_t)(sp.nseg - 1) * rows * p->dstate : nullptr;
    }
    return launch_scan_and_history(a, p, stream, "ssm_scan_fwd_static launch");
}

ssm_status ssd_scan_fwd(const ssd_scan_params* p, ssm_stream_t stream) {
    const char* who = "ssd_scan_fwd";
    if (p == nullptr) return fail(SSM_ERR_INVALID_ARG, "%s: params is NULL", who);
    if (p->batch <= 0 || p->nheads <= 0 || p->headdim <= 0 || p->ngroups <= 0 || p->dstate <= 0 || p->seqlen <= 0)
        return fail(SSM_ERR_INVALID_ARG, "%s: sizes must be positive (batch=%d nheads=%d headdim=%d ngroups=%d "
                    "dstate=%d seqlen=%d)", who, p->batch, p->nheads, p->headdim, p->ngroups, p->dstate, p->seqlen);
    if (!p->x || !p->dt || !p->A || !p->Bm || !p->Cm || !p->y)
        return fail(SSM_ERR_INVALID_ARG, "%s: x, dt, A, Bm, Cm and y are required", who);
    if ((p->delta_softplus != 0 && p->delta_softplus != 1) || (p->zoh != 0 && p->zoh != 1))
        return fail(SSM_ERR_INVALID_ARG, "%s: delta_softplus and zoh must be 0 or 1", who);
    if (p->nheads % p->ngroups != 0)
        return fail(SSM_ERR_INVALID_ARG, "%s: ngroups %d does not divide nheads %d", who, p->ngroups, p->nheads);
    if (!ssm::ssd_tc_supported(p->dstate, p->headdim))
        return fail(SSM_ERR_UNSUPPORTED, "%s: headdim %d / dstate %d not supported (64 / 64 or 128)", who, p->headdim,
                    p->dstate);
    if (p->seqlen % 8 != 0)
        return fail(SSM_ERR_UNSUPPORTED, "%s: seqlen %d is not a multiple of 8", who, p->seqlen);
    if (!aligned16(p->x) || !aligned16(p->dt) || !aligned16(p->Bm) || !aligned16(p->Cm) || !aligned16(p->y))
        return fail(SSM_ERR_UNSUPPORTED, "%s: x, dt, Bm, Cm and y must be 16-byte aligned", who);
    const size_t B = (size_t)p->batch, H = (size_t)p->nheads, L = (size_t)p->seqlen;
    const size_t D = H * (size_t)p->headdim, N = (size_t)p->dstate, G = (size_t)p->ngroups;
    if (B * H > 0x7fffffffu || B * D > 0x7fffffffu || B * G * L * N > ((size_t)1 << 40))
        return fail(SSM_ERR_UNSUPPORTED, "%s: problem too large", who);
    const size_t xb = B * D * L * 2, db = B * H * L * 2, bcb = B * G * L * N * 2, hb = B * D * N * 4;
    struct Span {
        const void* p;
        size_t n;
    };
    const Span in[] = {{p->x, xb}, {p->dt, db}, {p->A, H * 4}, {p->Bm, bcb}, {p->Cm, bcb}, {p->Dskip, H * 4},
                       {p->dt_bias, H * 4}, {p->z, xb}, {p->h0, hb}};
    for (const Span& i : in)
        if (overlaps(p->y, xb, i.p, i.n)) return fail(SSM_ERR_INVALID_ARG, "%s: y overlaps an input", who);
    if (p->h_out) {
        if (overlaps(p->h_out, hb, p->y, xb)) return fail(SSM_ERR_INVALID_ARG, "%s: h_out overlaps y", who);
        for (const Span& i : in)
            if (i.p != p->h0 && overlaps(p->h_out, hb, i.p, i.n))
                return fail(SSM_ERR_INVALID_ARG, "%s: h_out overlaps an input", who);
        if (p->h0 && p->h0 != p->h_out && overlaps(p->h_out, hb, p->h0, hb))
            return fail(SSM_ERR_INVALID_ARG, "%s: h_out partly overlaps h0", who);
    }
    ssm::SsdArgs a{p->batch, p->nheads, p->ngroups, p->seqlen, p->dstate, p->x, p->dt, p->A, p->Bm, p->Cm, p->Dskip,
                   p->dt_bias, p->z, p->h0, p->h_out, p->y, p->delta_softplus, p->zoh};
    cudaError_t e = ssm::launch_ssd_chunked(a, (cudaStream_t)stream);
    if (e == cudaErrorInvalidValue) return fail(SSM_ERR_UNSUPPORTED, "%s: tensor map encoding refused the layout", who);
    return cuda_status(e, "ssd_scan_fwd launch");
}

}  // extern "C"

namespace ssm {
cudaError_t launch_scan(const ScanKernelArgs& a, int in_dtype, int out_dtype, int zoh, cudaStream_t stream) {
    if (in_dtype == 0 && out_dtype == 0) return launch_scan_f32_f32(a, zoh, stream);
    if (in_dtype == 1 && out_dtype == 1) return launch_scan_bf16_bf16(a, zoh, stream);
    if (in_dtype == 1 && out_dtype == 0) return launch_scan_bf16_f32(a, zoh, stream);
    return launch_scan_f32_bf16(a, zoh, stream);
}
}  // namespace ssm
