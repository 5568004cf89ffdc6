// Internal declarations shared by the translation units of libspecverify.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "specverify.h"

namespace sv {

// All arguments of one verification call, after host-side validation.
struct Args {
    const void* target;  // [B, gamma+1, V]
    const void* draft;   // [B, gamma, V]; null in one-hot mode
    bool onehot;               // deterministic proposals: q_i one-hot at x_i, no draft logits
    bool early;                // early exit: nothing after a request's first rejection is read
    bool tree;                 // tree verification (one-hot candidates; num_draft = nodes in use)
    const int32_t* parents;    // tree: [B, gamma] parent of node j at j - 1
    int32_t* out_nodes;        // tree: [B, gamma] accepted node indices, may be null
    const int32_t* num_draft;  // one-hot mode: proposals per request [B] (null: gamma each)
    int dtype;           // SV_F32 / SV_BF16
    int B, gamma, V;
    const int32_t* tokens;      // [B, gamma]
    const float* u_accept;      // [B, gamma]
    const float* u_sample;      // [B]
    const float* temperature;   // [B]
    int32_t* out_tokens;        // [B, gamma+1]
    int32_t* out_num_accepted;  // [B]
    sv_debug_out dbg;           // device pointers, each may be null
    int32_t* d_status;          // may be null
    unsigned long long peer_wait_ns;  // streaming path: limit of each wait on other blocks' work
    const int32_t* hold_flag;         // streaming path, checking only (sv_options.hold_flag)
};

struct DeviceInfo {
    int device = -1;
    int num_sms = 0;
    int cc_major = 0, cc_minor = 0;
    size_t smem_optin = 0;
};

// Sets what spec_verify_last_launch_count() reports on this host thread.
void set_last_launch_count(int n);

// Cached properties of the current device; false when there is none.
bool current_device(DeviceInfo* info);

// Rowwise path: one thread block per request. Enqueues one kernel.
cudaError_t launch_rowwise(const Args& a, const DeviceInfo& dev, cudaStream_t stream);

// Streaming path: persistent grid. Workspace layout and launch.
bool streaming_applicable(const Args& a);
bool streaming_grid_ok(int B, int grid);
size_t streaming_workspace_bytes(int B, int gamma, int V, int dtype, int grid);
int streaming_default_grid(const DeviceInfo& dev);
cudaError_t launch_streaming(const Args& a, const DeviceInfo& dev, int grid, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream);

// Cluster path: one thread-block cluster per request (small batches).
bool cluster_applicable(const Args& a);
int cluster_size(int V, int dtype);
cudaError_t launch_cluster(const Args& a, const DeviceInfo& dev, cudaStream_t stream);

}  // namespace sv
