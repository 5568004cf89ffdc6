// extern "C" entry points of libspecverify (declared in include/specverify.h):
// argument validation, device query, choice of execution path, and the
// host-buffer variant that stages inputs and outputs through device memory.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "sv_internal.h"

namespace sv {
namespace {

thread_local int g_last_launches = 0;

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices];

size_t elem_bytes(int dtype) { return dtype == SV_F32 ? 4 : 2; }

bool shape_ok(int B, int gamma, int V, sv_dtype dtype) {
    return B >= 0 && gamma >= 1 && gamma <= SV_MAX_GAMMA && V >= 1 && V <= SV_MAX_V &&
           (dtype == SV_F32 || dtype == SV_BF16);
}

size_t align16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }

// Bytes the call needs in its workspace for this shape and device.
size_t workspace_need(int B, int gamma, int V, sv_dtype dtype, const DeviceInfo& dev) {
    return streaming_workspace_bytes(B, gamma, V, dtype, streaming_default_grid(dev));
}

}  // namespace

void set_last_launch_count(int n) { g_last_launches = n; }

bool current_device(DeviceInfo* info) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return false;
    }
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (d.device != dev) {
        DeviceInfo n;
        n.device = dev;
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        n.num_sms = v;
        cudaDeviceGetAttribute(&n.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&n.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        n.smem_optin = static_cast<size_t>(v);
        d = n;
    }
    *info = d;
    return true;
}

}  // namespace sv

using namespace sv;

extern "C" {

int spec_verify_version(void) { return 10000; }

int spec_verify_last_launch_count(void) { return g_last_launches; }

const char* spec_verify_status_string(sv_status s) {
    switch (s) {
        case SV_OK: return "ok";
        case SV_ERR_INVALID_ARG: return "invalid argument (null pointer, size out of range or unknown dtype)";
        case SV_ERR_UNSUPPORTED: return "unsupported device (needs a CUDA device of compute capability 10.3)";
        case SV_ERR_CUDA: return "a CUDA call failed while enqueueing";
        case SV_ERR_WORKSPACE: return "workspace missing or smaller than spec_verify_workspace_size()";
        case SV_ERR_TIMEOUT: return "a bounded wait ran out";
        case SV_ERR_SCRATCH_LIMIT: return "shape needs more scratch than spec_verify_noalloc holds (SV_NOALLOC_SCRATCH_BYTES)";
        default: return "unknown status";
    }
}

sv_status spec_verify_workspace_size(int B, int gamma, int V, sv_dtype dtype, size_t* bytes) {
    if (!bytes || !shape_ok(B, gamma, V, dtype)) return SV_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (!current_device(&dev)) return SV_ERR_UNSUPPORTED;
    *bytes = workspace_need(B, gamma, V, dtype, dev);
    return SV_OK;
}

// Picks the kernel and launches it. On SV_PATH_AUTO: one cluster per request
// for small batches (at most kClusterMaxB requests) of rows of at least
// kClusterMinRow bytes where it applies, the streaming kernel where it
// applies and the target logits reach 64 KB, else one block per request.
constexpr int kClusterMaxB = 16;
constexpr size_t kClusterMinRow = 16u << 10;
static sv_status dispatch(const Args& a, const DeviceInfo& dev, int path, int grid_ctas, void* workspace,
                   size_t workspace_bytes, sv_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int grid = streaming_default_grid(dev);
    if (grid_ctas > 0) grid = std::min(grid, grid_ctas);
    const bool stream_ok = streaming_applicable(a) && streaming_grid_ok(a.B, grid);
    bool use_stream = false, use_cluster = false;
    if (path == SV_PATH_STREAMING) {
        if (!stream_ok) return SV_ERR_INVALID_ARG;
        use_stream = true;
    } else if (path == SV_PATH_CLUSTER) {
        if (!cluster_applicable(a)) return SV_ERR_INVALID_ARG;
        use_cluster = true;
    } else if (path == SV_PATH_AUTO) {
        const size_t target_bytes = static_cast<size_t>(a.B) * (a.gamma + 1) * a.V * elem_bytes(a.dtype);
        use_cluster = a.B <= kClusterMaxB && static_cast<size_t>(a.V) * elem_bytes(a.dtype) >= kClusterMinRow &&
                      cluster_applicable(a);
        use_stream = !use_cluster && stream_ok && target_bytes >= (64u << 10);
    }
    cudaError_t err;
    if (use_cluster) {
        err = launch_cluster(a, dev, s);
    } else if (use_stream) {
        const size_t need = streaming_workspace_bytes(a.B, a.gamma, a.V, a.dtype, grid);
        if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 15))
            return SV_ERR_WORKSPACE;
        err = launch_streaming(a, dev, grid, workspace, workspace_bytes, s);
    } else {
        err = launch_rowwise(a, dev, s);
    }
    if (err != cudaSuccess) return SV_ERR_CUDA;
    g_last_launches = 1;
    return SV_OK;
}

sv_status spec_verify_ex(const void* target_logits, const void* draft_logits, sv_dtype dtype, int B,
                         int gamma, int V, const int32_t* draft_tokens, const float* u_accept,
                         const float* u_sample, const float* temperature, int32_t* out_tokens,
                         int32_t* out_num_accepted, void* workspace, size_t workspace_bytes,
                         sv_stream_t stream, const sv_debug_out* dbg, int32_t* d_status,
                         const sv_options* opts) {
    g_last_launches = 0;
    if (!shape_ok(B, gamma, V, dtype)) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    // draft_logits == NULL: deterministic (one-hot) proposals, see spec_verify_onehot
    if (!target_logits || !draft_tokens || !u_accept || !u_sample || !temperature || !out_tokens ||
        !out_num_accepted)
        return SV_ERR_INVALID_ARG;
    const int path = opts ? opts->path : SV_PATH_AUTO;
    if (path != SV_PATH_AUTO && path != SV_PATH_ROWWISE && path != SV_PATH_STREAMING && path != SV_PATH_CLUSTER)
        return SV_ERR_INVALID_ARG;
    if (opts && (opts->grid_ctas < 0 || opts->peer_wait_us < 0)) return SV_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (!current_device(&dev)) return SV_ERR_UNSUPPORTED;
    if (dev.cc_major != 10 || dev.cc_minor != 3) return SV_ERR_UNSUPPORTED;

    Args a = {};  // every field not set below is zero (no tree, no parents)
    a.target = target_logits;
    a.draft = draft_logits;
    a.onehot = draft_logits == nullptr;
    a.early = opts && opts->early_exit != 0;
    a.num_draft = (a.onehot && opts) ? opts->num_draft : nullptr;
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
    std::memset(&a.dbg, 0, sizeof a.dbg);
    if (dbg) a.dbg = *dbg;
    a.d_status = d_status;
    a.peer_wait_ns = (opts && opts->peer_wait_us > 0) ? 1000ull * static_cast<unsigned>(opts->peer_wait_us)
                                                     : 2000000000ull;
    a.hold_flag = opts ? opts->hold_flag : nullptr;

    return dispatch(a, dev, path, opts ? opts->grid_ctas : 0, workspace, workspace_bytes, stream);
}

sv_status spec_verify_tree(const void* target_logits, sv_dtype dtype, int B, int gamma, int V,
                           const int32_t* node_tokens, const int32_t* parents, const int32_t* num_nodes,
                           const float* u_accept, const float* u_sample, const float* temperature,
                           int32_t* out_tokens, int32_t* out_num_accepted, int32_t* out_nodes, void* workspace,
                           size_t workspace_bytes, sv_stream_t stream, const sv_debug_out* dbg, int32_t* d_status,
                           const sv_options* opts) {
    g_last_launches = 0;
    if (!shape_ok(B, gamma, V, dtype)) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!target_logits || !node_tokens || !parents || !num_nodes || !u_accept || !u_sample || !temperature ||
        !out_tokens || !out_num_accepted)
        return SV_ERR_INVALID_ARG;
    const int path = opts ? opts->path : SV_PATH_AUTO;
    if (path != SV_PATH_AUTO && path != SV_PATH_ROWWISE && path != SV_PATH_STREAMING) return SV_ERR_INVALID_ARG;
    if (opts && (opts->grid_ctas < 0 || opts->peer_wait_us < 0 || opts->early_exit)) return SV_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (!current_device(&dev)) return SV_ERR_UNSUPPORTED;
    if (dev.cc_major != 10 || dev.cc_minor != 3) return SV_ERR_UNSUPPORTED;
    Args a = {};
    a.target = target_logits;
    a.dtype = dtype;
    a.B = B;
    a.gamma = gamma;
    a.V = V;
    a.tokens = node_tokens;
    a.u_accept = u_accept;
    a.u_sample = u_sample;
    a.temperature = temperature;
    a.out_tokens = out_tokens;
    a.out_num_accepted = out_num_accepted;
    if (dbg) a.dbg = *dbg;
    a.d_status = d_status;
    a.peer_wait_ns = (opts && opts->peer_wait_us > 0) ? 1000ull * static_cast<unsigned>(opts->peer_wait_us)
                                                     : 2000000000ull;
    a.hold_flag = opts ? opts->hold_flag : nullptr;
    a.onehot = true;  // candidates are tokens, not draws from a draft distribution
    a.num_draft = num_nodes;
    a.tree = true;
    a.parents = parents;
    a.out_nodes = out_nodes;
    return dispatch(a, dev, path, opts ? opts->grid_ctas : 0, workspace, workspace_bytes, stream);
}

sv_status spec_verify_onehot(const void* target_logits, sv_dtype dtype, int B, int gamma, int V,
                             const int32_t* draft_tokens, const int32_t* num_draft, const float* u_accept,
                             const float* u_sample, const float* temperature, int32_t* out_tokens,
                             int32_t* out_num_accepted, void* workspace, size_t workspace_bytes,
                             sv_stream_t stream) {
    sv_options o;
    std::memset(&o, 0, sizeof o);
    o.num_draft = num_draft;
    return spec_verify_ex(target_logits, nullptr, dtype, B, gamma, V, draft_tokens, u_accept, u_sample,
                          temperature, out_tokens, out_num_accepted, workspace, workspace_bytes, stream,
                          nullptr, nullptr, &o);
}

sv_status spec_verify(const void* target_logits, const void* draft_logits, sv_dtype dtype, int B,
                      int gamma, int V, const int32_t* draft_tokens, const float* u_accept,
                      const float* u_sample, const float* temperature, int32_t* out_tokens,
                      int32_t* out_num_accepted, void* workspace, size_t workspace_bytes,
                      sv_stream_t stream) {
    g_last_launches = 0;
    if (!draft_logits && B > 0) return SV_ERR_INVALID_ARG;  // one-hot proposals: spec_verify_onehot
    return spec_verify_ex(target_logits, draft_logits, dtype, B, gamma, V, draft_tokens, u_accept,
                          u_sample, temperature, out_tokens, out_num_accepted, workspace,
                          workspace_bytes, stream, nullptr, nullptr, nullptr);
}

// ---------------------------------------------------------------- host path

namespace {

struct Staging {
    size_t target, draft, tokens, u_accept, u_sample, temperature, out_tokens, out_num, workspace,
        end;
};

// Request slices of one spec_verify_host call: at most kHostSlices, each of
// at least kHostSliceMinBytes of input (fewer for small batches).
constexpr int kHostSlices = 8;
constexpr size_t kHostSliceMinBytes = size_t(32) << 20;

// Per device: the stream the host entry copies on, and its events. Made by the
// first call on the device and kept until the process exits; calls hold
// g_copy_mu while they enqueue, so they never share an event in flight.
struct CopyLane {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr;
    cudaEvent_t ready[kHostSlices] = {};
};
std::mutex g_copy_mu;
CopyLane g_lane[kMaxDevices];

CopyLane* copy_lane(int device) {
    if (device < 0 || device >= kMaxDevices) return nullptr;
    CopyLane& c = g_lane[device];
    if (c.stream) return &c;
    CopyLane n;
    bool ok = cudaStreamCreateWithFlags(&n.stream, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&n.fork, cudaEventDisableTiming) == cudaSuccess;
    for (int k = 0; ok && k < kHostSlices; ++k)
        ok = cudaEventCreateWithFlags(&n.ready[k], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        if (n.fork) cudaEventDestroy(n.fork);
        for (cudaEvent_t e : n.ready)
            if (e) cudaEventDestroy(e);
        if (n.stream) cudaStreamDestroy(n.stream);
        return nullptr;
    }
    c = n;
    return &c;
}

Staging staging_layout(int B, int gamma, int V, sv_dtype dtype, size_t ws) {
    const size_t es = elem_bytes(dtype);
    Staging l;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = align16(off + bytes);
        return at;
    };
    l.target = take(static_cast<size_t>(B) * (gamma + 1) * V * es);
    l.draft = take(static_cast<size_t>(B) * gamma * V * es);
    l.tokens = take(static_cast<size_t>(B) * gamma * 4);
    l.u_accept = take(static_cast<size_t>(B) * gamma * 4);
    l.u_sample = take(static_cast<size_t>(B) * 4);
    l.temperature = take(static_cast<size_t>(B) * 4);
    l.out_tokens = take(static_cast<size_t>(B) * (gamma + 1) * 4);
    l.out_num = take(static_cast<size_t>(B) * 4);
    l.workspace = take(ws);
    l.end = off;
    return l;
}

}  // namespace

sv_status spec_verify_host_staging_size(int B, int gamma, int V, sv_dtype dtype, size_t* bytes) {
    if (!bytes || !shape_ok(B, gamma, V, dtype)) return SV_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (!current_device(&dev)) return SV_ERR_UNSUPPORTED;
    *bytes = staging_layout(B, gamma, V, dtype, workspace_need(B, gamma, V, dtype, dev)).end;
    return SV_OK;
}

sv_status spec_verify_host(const void* target_logits, const void* draft_logits, sv_dtype dtype, int B,
                           int gamma, int V, const int32_t* draft_tokens, const float* u_accept,
                           const float* u_sample, const float* temperature, int32_t* out_tokens,
                           int32_t* out_num_accepted, void* staging, size_t staging_bytes,
                           sv_stream_t stream) {
    g_last_launches = 0;
    if (!shape_ok(B, gamma, V, dtype)) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!target_logits || !draft_logits || !draft_tokens || !u_accept || !u_sample || !temperature ||
        !out_tokens || !out_num_accepted)
        return SV_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (!current_device(&dev)) return SV_ERR_UNSUPPORTED;
    const size_t ws = workspace_need(B, gamma, V, dtype, dev);
    const Staging l = staging_layout(B, gamma, V, dtype, ws);
    if (!staging || staging_bytes < l.end || (reinterpret_cast<uintptr_t>(staging) & 15))
        return SV_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(staging);
    const size_t es = elem_bytes(dtype);
    const size_t trow_bytes = static_cast<size_t>(gamma + 1) * V * es;  // one request's target rows
    const size_t drow_bytes = static_cast<size_t>(gamma) * V * es;      // one request's draft rows

    // The inputs cross the host link far slower than the kernel reads them
    // from HBM, so the batch is cut into request slices: the copy stream moves
    // slice k while the caller's stream verifies slice k - 1 (requests are
    // independent, so the outputs are those of one call over the batch).
    size_t in_bytes = static_cast<size_t>(B) * trow_bytes;
    for (int b = 0; b < B; ++b)
        if (temperature[b] > 0.0f) in_bytes += drow_bytes;
    const int slices = static_cast<int>(std::max<size_t>(
        1, std::min<size_t>({static_cast<size_t>(kHostSlices), static_cast<size_t>(B),
                             in_bytes / kHostSliceMinBytes})));

    std::lock_guard<std::mutex> lock(g_copy_mu);
    CopyLane* lane = copy_lane(dev.device);
    if (!lane) return SV_ERR_CUDA;
    cudaStream_t cs = lane->stream;
    auto fail = [&]() {
        cudaGetLastError();
        g_last_launches = 0;
        return SV_ERR_CUDA;
    };
    auto h2d = [&](size_t off, const void* src, size_t bytes) {
        return cudaMemcpyAsync(base + off, src, bytes, cudaMemcpyHostToDevice, cs);
    };
    // The copies overwrite staging: they wait for the caller's earlier work.
    if (cudaEventRecord(lane->fork, s) != cudaSuccess || cudaStreamWaitEvent(cs, lane->fork, 0) != cudaSuccess)
        return fail();
    cudaError_t err = h2d(l.tokens, draft_tokens, static_cast<size_t>(B) * gamma * 4);
    if (err == cudaSuccess) err = h2d(l.u_accept, u_accept, static_cast<size_t>(B) * gamma * 4);
    if (err == cudaSuccess) err = h2d(l.u_sample, u_sample, static_cast<size_t>(B) * 4);
    if (err == cudaSuccess) err = h2d(l.temperature, temperature, static_cast<size_t>(B) * 4);
    if (err != cudaSuccess) return fail();

    int launches = 0;
    for (int k = 0; k < slices; ++k) {
        const int b0 = static_cast<int>(static_cast<int64_t>(B) * k / slices);
        const int b1 = static_cast<int>(static_cast<int64_t>(B) * (k + 1) / slices);
        const int nb = b1 - b0;
        err = h2d(l.target + b0 * trow_bytes, static_cast<const char*>(target_logits) + b0 * trow_bytes,
                  static_cast<size_t>(nb) * trow_bytes);
        // Draft rows: only requests with T > 0 are read, copied in runs of
        // consecutive such requests.
        for (int b = b0; b < b1 && err == cudaSuccess;) {
            if (!(temperature[b] > 0.0f)) {
                ++b;
                continue;
            }
            int e = b + 1;
            while (e < b1 && temperature[e] > 0.0f) ++e;
            err = h2d(l.draft + b * drow_bytes, static_cast<const char*>(draft_logits) + b * drow_bytes,
                      static_cast<size_t>(e - b) * drow_bytes);
            b = e;
        }
        if (err != cudaSuccess || cudaEventRecord(lane->ready[k], cs) != cudaSuccess ||
            cudaStreamWaitEvent(s, lane->ready[k], 0) != cudaSuccess)
            return fail();
        sv_status st = spec_verify(
            base + l.target + b0 * trow_bytes, base + l.draft + b0 * drow_bytes, dtype, nb, gamma, V,
            reinterpret_cast<const int32_t*>(base + l.tokens) + static_cast<size_t>(b0) * gamma,
            reinterpret_cast<const float*>(base + l.u_accept) + static_cast<size_t>(b0) * gamma,
            reinterpret_cast<const float*>(base + l.u_sample) + b0,
            reinterpret_cast<const float*>(base + l.temperature) + b0,
            reinterpret_cast<int32_t*>(base + l.out_tokens) + static_cast<size_t>(b0) * (gamma + 1),
            reinterpret_cast<int32_t*>(base + l.out_num) + b0, base + l.workspace, ws, stream);
        if (st != SV_OK) {
            g_last_launches = 0;
            return st;
        }
        launches += g_last_launches;
    }
    err = cudaMemcpyAsync(out_tokens, base + l.out_tokens, static_cast<size_t>(B) * (gamma + 1) * 4,
                          cudaMemcpyDeviceToHost, s);
    if (err == cudaSuccess)
        err = cudaMemcpyAsync(out_num_accepted, base + l.out_num, static_cast<size_t>(B) * 4,
                              cudaMemcpyDeviceToHost, s);
    if (err != cudaSuccess) return fail();
    g_last_launches = launches;
    return SV_OK;
}

}  // extern "C"
