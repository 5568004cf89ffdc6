// spec_commit: post-verify bookkeeping on the GPU.
//
// "Accélérer Sonar grâce à la spéculation", §Planification MTP pour un jeton
// unique: once the draft tokens are verified, a kernel inserts the next
// target tokens into their slots, so the host never waits for the accepted
// length. Here each request's emitted tokens (the n accepted draft tokens,
// then the target's token: "Speculative Decoding : accélérer l'inférence des
// LLM", §Principe et garanties mathématiques) are appended to its token
// buffer and its length is advanced.
//
// One warp per request: the lanes check the emitted tokens and copy them;
// lane 0 updates the length and the next input token. The request's
// validity is decided warp-uniformly before anything is written.
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kCommitThreads = 256;

__global__ void __launch_bounds__(kCommitThreads) commit_kernel(const int32_t* __restrict__ out_tokens,
                                                                const int32_t* __restrict__ out_num_accepted,
                                                                int B, int gamma, int32_t* __restrict__ token_buf,
                                                                int max_len, int32_t* __restrict__ seq_lens,
                                                                int32_t* __restrict__ next_input,
                                                                int32_t* __restrict__ d_status) {
    const int b = static_cast<int>((static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (b >= B) return;  // whole warps only: blockDim is a multiple of 32
    const int n = out_num_accepted[b];
    const int L = seq_lens[b];
    const int32_t* emitted = out_tokens + static_cast<size_t>(b) * (gamma + 1);
    bool bad = n < 0 || n > gamma || L < 0 || L > max_len;
    if (!bad) {
        int neg = 0;
        for (int j = lane; j <= n; j += 32) neg |= emitted[j] < 0;
        bad = __any_sync(0xffffffffu, neg) != 0;
    }
    if (bad) {
        if (lane == 0) {
            if (next_input) next_input[b] = -1;
            if (d_status) atomicOr(d_status, SV_STATUS_BAD_REQUEST);
        }
        return;
    }
    const int count = min(n + 1, max_len - L);  // tokens that fit
    int32_t* row = token_buf + static_cast<size_t>(b) * max_len;
    for (int j = lane; j < count; j += 32) row[L + j] = emitted[j];
    if (lane == 0) {
        seq_lens[b] = L + count;
        if (next_input) next_input[b] = count > 0 ? emitted[count - 1] : (L > 0 ? row[L - 1] : -1);
        if (count < n + 1 && d_status) atomicOr(d_status, SV_STATUS_TRUNCATED);
    }
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" sv_status spec_commit(const int32_t* out_tokens, const int32_t* out_num_accepted, int B, int gamma,
                                 int32_t* token_buf, int max_len, int32_t* seq_lens, int32_t* next_input,
                                 int32_t* d_status, sv_stream_t stream) {
    set_last_launch_count(0);
    if (B < 0 || gamma < 1 || gamma > SV_MAX_GAMMA || max_len < 1) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!out_tokens || !out_num_accepted || !token_buf || !seq_lens) return SV_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (!current_device(&dev)) return SV_ERR_UNSUPPORTED;
    const long long threads = static_cast<long long>(B) * 32;
    const unsigned blocks = static_cast<unsigned>((threads + kCommitThreads - 1) / kCommitThreads);
    commit_kernel<<<blocks, kCommitThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        out_tokens, out_num_accepted, B, gamma, token_buf, max_len, seq_lens, next_input, d_status);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return SV_ERR_CUDA;
    set_last_launch_count(1);
    return SV_OK;
}
