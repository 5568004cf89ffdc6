// spec_verify_noalloc: the streaming path with its scratch memory in a
// static device array of this library instead of a caller-owned workspace.
//
// For callers that cannot allocate device memory themselves: a plugin that
// another runtime hands only its input and output tensors, or a serving loop
// whose device memory is fixed at start-up and that must not call cudaMalloc
// on its hot path (cudaMalloc can synchronize the device and grows the
// process's footprint). The entry point allocates nothing: the scratch is the
// file-scope array below, which every GPU that loads this library holds, at
// its full size, until the process exits.
#include <cuda.h>

#include <mutex>

#include "sv_internal.h"

namespace sv {
namespace {

// The scratch (the header and completion counters, partial row
// statistics, draw jobs, draw sums). Its size is SV_NOALLOC_SCRATCH_BYTES; shapes that need more are
// rejected with SV_ERR_SCRATCH_LIMIT.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct ScratchAddr {
    unsigned long long ctx_id = 0;  // the driver's id of the context the address belongs to (0: none)
    void* ptr = nullptr;
};
ScratchAddr g_scratch[kMaxDevices];

// The driver's current-context calls, reached through the runtime (the
// library links no driver library of its own). Null where the driver lacks
// them; every call then asks the runtime for the address afresh.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;
std::once_flag g_entry_once;

void load_entry_points() {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_ctx_id = reinterpret_cast<CtxGetIdFn>(f);
    cudaGetLastError();
}

// The id of the calling thread's current context, 0 when it cannot be told.
unsigned long long current_context_id() {
    if (!g_ctx_current || !g_ctx_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (g_ctx_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of g_noalloc_scratch in the current context. In host code
// the array's name is only a host-side handle; the address comes from
// cudaGetSymbolAddress with the device current, once per context: it is
// kept with the driver's id of that context, so that after a device reset
// (a new context, where the module may load at another address) it is asked
// for again instead of reused.
cudaError_t scratch_address(int device, void** ptr) {
    std::call_once(g_entry_once, load_entry_points);
    std::lock_guard<std::mutex> lock(g_mu);
    ScratchAddr& c = g_scratch[device];
    const unsigned long long id = current_context_id();
    if (id == 0 || c.ctx_id != id || !c.ptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        c.ptr = p;
        c.ctx_id = current_context_id();  // the call above made the device's context current if it was not
    }
    *ptr = c.ptr;
    return cudaSuccess;
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" sv_status spec_verify_noalloc(const void* target_logits, const void* draft_logits,
                                         sv_dtype dtype, int B, int gamma, int V,
                                         const int32_t* draft_tokens, const float* u_accept,
                                         const float* u_sample, const float* temperature,
                                         int32_t* out_tokens, int32_t* out_num_accepted,
                                         sv_stream_t stream) {
    set_last_launch_count(0);
    if (B < 0 || gamma < 1 || gamma > SV_MAX_GAMMA || V < 1 || V > SV_MAX_V ||
        (dtype != SV_F32 && dtype != SV_BF16))
        return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!target_logits || !draft_logits || !draft_tokens || !u_accept || !u_sample || !temperature ||
        !out_tokens || !out_num_accepted)
        return SV_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (!current_device(&dev)) return SV_ERR_UNSUPPORTED;
    if (dev.cc_major != 10 || dev.cc_minor != 3 || dev.device >= kMaxDevices) return SV_ERR_UNSUPPORTED;

    Args a = {};
    a.target = target_logits;
    a.draft = draft_logits;
    a.dtype = dtype;
    a.B = B;
    a.gamma = gamma;
    a.V = V;
    a.tokens = draft_tokens;
    a.u_accept = u_accept;
    a.u_sample = u_sample;
    a.temperature = temperature;
    a.out_tokens = out_tokens;
    a.out_num_accepted = out_num_accepted;
    a.peer_wait_ns = 2000000000ull;

    const int grid = streaming_default_grid(dev);
    if (!streaming_applicable(a) || !streaming_grid_ok(B, grid)) return SV_ERR_INVALID_ARG;
    if (streaming_workspace_bytes(B, gamma, V, dtype, grid) > SV_NOALLOC_SCRATCH_BYTES)
        return SV_ERR_SCRATCH_LIMIT;
    void* scratch = nullptr;
    if (scratch_address(dev.device, &scratch) != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    // launch_streaming clears the header and the completion counters at the
    // start of the scratch (the only parts that must start at zero) before it
    // launches.
    const cudaError_t e = launch_streaming(a, dev, grid, scratch, SV_NOALLOC_SCRATCH_BYTES,
                                           reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SV_ERR_CUDA;
    }
    set_last_launch_count(1);
    return SV_OK;
}
