// spec_ngram_propose: model-free draft tokens by n-gram (prompt) lookup.
//
// "Speculative Decoding : accélérer l'inférence des LLM", §N-gram lookup et
// variantes sans modèle: find the last n tokens of the context earlier in the
// context and propose the tokens that followed them; §Mise en œuvre dans
// vLLM: n from prompt_lookup_min = 2 to prompt_lookup_max = 5.
//
// One block per request. For every candidate end position e <= L - 1 a
// thread counts how many tokens before e match the history's last tokens,
// backwards, up to n_max: m(e). The proposal uses the longest match (the
// largest m, at least n_min) and, among those, the latest occurrence (the
// largest e): both at once as the maximum of the 64-bit key (m << 32) | e over
// the block. Tokens h[e .. e + k - 1] follow, k = min(gamma, L - e).
//
// The history is read once: the block copies up to 8192 tokens into shared
// memory with eight independent loads per thread (one memory latency instead
// of a chain of dependent loads per candidate), then compares there. Longer
// histories take several passes of 8176 candidates, each tile starting
// SV_NGRAM_MAX_N tokens before its first candidate so a match can reach back.
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kNgramThreads = 1024;
constexpr int kNgramLoads = 8;                                  // tokens each thread copies per pass
constexpr int kNgramTile = kNgramThreads * kNgramLoads;         // tokens staged per pass
constexpr int kNgramChunk = kNgramTile - SV_NGRAM_MAX_N;        // candidates per pass

__global__ void __launch_bounds__(kNgramThreads) ngram_kernel(const int32_t* __restrict__ token_buf, int max_len,
                                                              const int32_t* __restrict__ seq_lens, int gamma,
                                                              int n_min, int n_max, int32_t* __restrict__ draft_tokens,
                                                              int32_t* __restrict__ num_draft,
                                                              int32_t* __restrict__ d_status) {
    __shared__ int32_t query[SV_NGRAM_MAX_N];  // query[t] = h[L - 1 - t]
    __shared__ int32_t tile[kNgramTile];        // tile[i - lo] = h[i]
    __shared__ unsigned long long warp_best[kNgramThreads / 32];
    const int b = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int L = seq_lens[b];
    int32_t* out = draft_tokens + static_cast<size_t>(b) * gamma;
    if (L < 0 || L > max_len) {
        for (int i = t; i < gamma; i += kNgramThreads) out[i] = -1;
        if (t == 0) {
            num_draft[b] = 0;
            if (d_status) atomicOr(d_status, SV_STATUS_BAD_REQUEST);
        }
        return;
    }
    const int32_t* h = token_buf + static_cast<size_t>(b) * max_len;
    if (t < n_max && t < L) query[t] = h[L - 1 - t];
    unsigned long long best = 0ull;  // (m << 32) | e; 0 = no match of at least n_min
    // Candidates e in [e0, e1) read h[e - 1 - m] for m < min(n_max, e): tokens
    // [lo, hi) with lo >= e0 - SV_NGRAM_MAX_N and hi = e1 - 1, at most
    // kNgramTile of them. The loop bounds are the same for every thread.
    for (int e0 = n_min; e0 <= L - 1; e0 += kNgramChunk) {
        const int e1 = min(e0 + kNgramChunk, L);
        const int lo = max(0, e0 - SV_NGRAM_MAX_N), hi = e1 - 1;
        __syncthreads();  // the previous pass is done with the tile; query is written
        int32_t v[kNgramLoads];
#pragma unroll
        for (int r = 0; r < kNgramLoads; ++r) {
            const int i = lo + r * kNgramThreads + t;
            v[r] = i < hi ? h[i] : 0;
        }
#pragma unroll
        for (int r = 0; r < kNgramLoads; ++r) {
            const int i = lo + r * kNgramThreads + t;
            if (i < hi) tile[i - lo] = v[r];
        }
        __syncthreads();
        for (int e = e0 + t; e < e1; e += kNgramThreads) {
            int m = 0;
            const int lim = min(n_max, e);
            while (m < lim && tile[e - 1 - m - lo] == query[m]) ++m;
            if (m >= n_min) {
                const unsigned long long key = (static_cast<unsigned long long>(m) << 32) | static_cast<unsigned>(e);
                best = key > best ? key : best;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
        best = other > best ? other : best;
    }
    if (lane == 0) warp_best[warp] = best;
    __syncthreads();
    if (warp == 0) {
        best = lane < kNgramThreads / 32 ? warp_best[lane] : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
            best = other > best ? other : best;
        }
        const int e = static_cast<int>(best & 0xffffffffull);
        const int k = best ? min(gamma, L - e) : 0;
        for (int i = lane; i < gamma; i += 32) out[i] = i < k ? h[e + i] : -1;
        if (lane == 0) num_draft[b] = k;
    }
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" sv_status spec_ngram_propose(const int32_t* token_buf, int B, int max_len, const int32_t* seq_lens,
                                        int gamma, int n_min, int n_max, int32_t* draft_tokens,
                                        int32_t* num_draft, int32_t* d_status, sv_stream_t stream) {
    set_last_launch_count(0);
    if (B < 0 || max_len < 1 || gamma < 1 || gamma > SV_MAX_GAMMA || n_min < 1 || n_max < n_min ||
        n_max > SV_NGRAM_MAX_N)
        return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!token_buf || !seq_lens || !draft_tokens || !num_draft) return SV_ERR_INVALID_ARG;
    DeviceInfo dev;
    if (!current_device(&dev)) return SV_ERR_UNSUPPORTED;
    ngram_kernel<<<B, kNgramThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        token_buf, max_len, seq_lens, gamma, n_min, n_max, draft_tokens, num_draft, d_status);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
    set_last_launch_count(1);
    return SV_OK;
}
