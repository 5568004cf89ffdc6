// Rowwise path of libspecverify: one thread block verifies one request.
//
// The block reduces each of the request's rows in turn (target rows 0..gamma,
// then the draft rows 0..gamma-1 of a T > 0 request) to a (max, sum) or an
// argmax, runs the left-to-right acceptance scan on one thread, and draws the
// replacement or extra token with a block-wide inverse CDF. It handles any V
// and any alignment, with scalar loads; the streaming path is the fast one.
//
// Method: "Speculative Decoding : accélérer l'inférence des LLM",
// §Principe et garanties mathématiques and §Pourquoi la qualité est
// préservée; wiki "Speculative Decoding", eq. alpha(x) and eq. p_corr;
// "Accélérer Sonar grâce à la spéculation", §Décodage spéculatif.
#include <cmath>

#include "sv_common.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;

struct RowStat {
    float m;      // max (T > 0) or max value (T == 0)
    float s;      // sum 2^(l c - fl(m c)) (T > 0)
    int32_t idx;  // lowest-index argmax (T == 0)
    int32_t bad;  // NaN, +inf, or only -inf
};

struct Shared {
    RowStat st[2 * SV_MAX_GAMMA + 1];
    MaxSum ms[kWarps];
    ArgMax am[kWarps];
    int bad[kWarps];
    unsigned long long scan[kWarps + 1];
    DrawParams draw;
    int n;
    int request_bad;
    int last_row;  // early exit: the last position whose rows were read
    int stop;
};

template <int DT>
__device__ RowStat row_maxsum(const void* base, size_t row, int V, float c, Shared& sh) {
    MaxSum st = maxsum_empty();
    int bad = 0;
    const size_t off = row * static_cast<size_t>(V);
    for (int x = threadIdx.x; x < V; x += kThreads) {
        float l = load_logit<DT>(base, off + x);
        if (bad_logit(l)) {
            bad = 1;
        } else {
            maxsum_add(st, l, c);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        MaxSum other{__shfl_xor_sync(0xffffffffu, st.m, o), __shfl_xor_sync(0xffffffffu, st.s, o)};
        st = maxsum_merge(st, other, c);
    }
    bad = __any_sync(0xffffffffu, bad);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        sh.ms[warp] = st;
        sh.bad[warp] = bad;
    }
    __syncthreads();
    RowStat r;
    if (threadIdx.x == 0) {
        MaxSum acc = sh.ms[0];
        int b = sh.bad[0];
        for (int w = 1; w < kWarps; ++w) {
            acc = maxsum_merge(acc, sh.ms[w], c);
            b |= sh.bad[w];
        }
        r = {acc.m, acc.s, -1, (b || acc.m == neg_inf()) ? 1 : 0};
    }
    __syncthreads();
    return r;  // meaningful on thread 0 only
}

template <int DT>
__device__ RowStat row_argmax(const void* base, size_t row, int V, Shared& sh) {
    ArgMax st = argmax_empty();
    int bad = 0;
    const size_t off = row * static_cast<size_t>(V);
    for (int x = threadIdx.x; x < V; x += kThreads) {
        float l = load_logit<DT>(base, off + x);
        if (bad_logit(l)) bad = 1;
        if (l > st.v) st = {l, x};  // increasing x: the first maximum stays
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ArgMax other{__shfl_xor_sync(0xffffffffu, st.v, o), __shfl_xor_sync(0xffffffffu, st.i, o)};
        st = argmax_merge(st, other);
    }
    bad = __any_sync(0xffffffffu, bad);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        sh.am[warp] = st;
        sh.bad[warp] = bad;
    }
    __syncthreads();
    RowStat r;
    if (threadIdx.x == 0) {
        ArgMax acc = sh.am[0];
        int b = sh.bad[0];
        for (int w = 1; w < kWarps; ++w) {
            acc = argmax_merge(acc, sh.am[w]);
            b |= sh.bad[w];
        }
        if (acc.i == 0x7fffffff) acc.i = 0;
        r = {acc.v, 0.0f, acc.i, (b || acc.v == neg_inf()) ? 1 : 0};
    }
    __syncthreads();
    return r;
}

// Sum of the draw weights over [lo, hi) in index order (binary32).
template <int DT>
__device__ __forceinline__ float run_weights(const void* tgt, const void* dft, size_t trow,
                                             size_t drow, int lo, int hi, const DrawParams& d,
                                             int kind) {
    float run = 0.0f;
    for (int e = lo; e < hi; ++e) {
        float lt = load_logit<DT>(tgt, trow + e);
        float w = kind == kKindResidual ? weight_residual(lt, load_logit<DT>(dft, drow + e), d)
                                        : weight_target_excl(lt, e, d, kind);
        run = __fadd_rn(run, w);
    }
    return run;
}

template <int DT>
__global__ void __launch_bounds__(kThreads) rowwise_kernel(Args a) {
    __shared__ Shared sh;
    const int G = a.gamma, V = a.V;
    for (int b = blockIdx.x; b < a.B; b += gridDim.x) {
        const float T = a.temperature[b];
        const bool t_ok = (T >= 0.0f) && (T < pos_inf());
        const bool greedy = t_ok && T == 0.0f;
        const float c = (t_ok && !greedy) ? temp_scale(T) : 0.0f;
        // proposals: gamma, or num_draft[b] for one-hot proposals (no draft
        // rows; target rows past num_draft[b] take no part)
        const int kb = a.onehot && a.num_draft ? a.num_draft[b] : G;
        const bool range_ok = t_ok && kb >= 0 && kb <= G;
        const int np = range_ok ? kb : 0;
        int bad = range_ok ? 0 : 1;
        for (int i = threadIdx.x; i < np; i += kThreads) {
            int x = a.tokens[static_cast<size_t>(b) * G + i];
            if (x < 0 || x >= V) bad = 1;
        }
        bad = __syncthreads_or(bad);
        if (!bad && a.early) {
            // Early exit: position i's rows, then its decision on thread 0; nothing
            // after the first rejection (or mismatch at T = 0) is read. The scan
            // below then meets the same decisions from these rows.
            const int32_t* tok = a.tokens + static_cast<size_t>(b) * G;
            for (int i = 0; i <= np; ++i) {
                const size_t trow = static_cast<size_t>(b) * (G + 1) + i;
                const RowStat st = greedy ? row_argmax<DT>(a.target, trow, V, sh)
                                          : row_maxsum<DT>(a.target, trow, V, c, sh);
                const bool has_draft = !greedy && !a.onehot && i < np;
                RowStat sd;
                if (has_draft) sd = row_maxsum<DT>(a.draft, static_cast<size_t>(b) * G + i, V, c, sh);
                if (threadIdx.x == 0) {
                    sh.st[i] = st;
                    if (has_draft) sh.st[G + 1 + i] = sd;
                    int stop = (st.bad || (has_draft && sd.bad)) ? 2 : 0;
                    if (!stop) {
                        if (i == np) {
                            stop = 1;
                        } else if (greedy) {
                            stop = tok[i] != st.idx ? 1 : 0;
                        } else {
                            const int x = tok[i];
                            const double p = prob_from_stats(
                                load_logit<DT>(a.target, trow * V + x), st.m, st.s, c);
                            const double q = a.onehot ? 1.0
                                                      : prob_from_stats(load_logit<DT>(
                                                                            a.draft, (static_cast<size_t>(b) * G + i) * V + x),
                                                                        sd.m, sd.s, c);
                            stop = accept_draft(p, q, a.u_accept[static_cast<size_t>(b) * G + i]) ? 0 : 1;
                        }
                    }
                    sh.stop = stop;
                    sh.last_row = i;
                }
                __syncthreads();
                if (sh.stop) break;
            }
            bad = sh.stop == 2;
        } else if (!bad) {
            const int nrows = (greedy || a.onehot) ? np + 1 : 2 * G + 1;
            for (int r = 0; r < nrows; ++r) {
                RowStat st;
                if (r <= G) {
                    size_t row = static_cast<size_t>(b) * (G + 1) + r;
                    st = greedy ? row_argmax<DT>(a.target, row, V, sh)
                                : row_maxsum<DT>(a.target, row, V, c, sh);
                } else {
                    size_t row = static_cast<size_t>(b) * G + (r - G - 1);
                    st = row_maxsum<DT>(a.draft, row, V, c, sh);
                }
                if (threadIdx.x == 0) sh.st[r] = st;
            }
            if (threadIdx.x == 0) {
                int any = 0;
                for (int r = 0; r < nrows; ++r) any |= sh.st[r].bad;
                sh.request_bad = any;
            }
            __syncthreads();
            bad = sh.request_bad;
        }

        int32_t* out = a.out_tokens + static_cast<size_t>(b) * (G + 1);
        if (bad) {
            for (int j = threadIdx.x; j <= G; j += kThreads) out[j] = -1;
            if (threadIdx.x == 0) {
                a.out_num_accepted[b] = -1;
                if (a.d_status) atomicOr(a.d_status, SV_STATUS_BAD_REQUEST);
                if (a.dbg.kind) a.dbg.kind[b] = kKindInvalid;
                if (a.dbg.w_total) a.dbg.w_total[b] = nan("");
            }
            for (int j = threadIdx.x; j <= G; j += kThreads) {
                size_t r = static_cast<size_t>(b) * (G + 1) + j;
                if (a.dbg.max_target) a.dbg.max_target[r] = nanf("");
                if (a.dbg.lse_target) a.dbg.lse_target[r] = nan("");
                if (a.dbg.argmax_target) a.dbg.argmax_target[r] = -1;
            }
            for (int j = threadIdx.x; j < G; j += kThreads) {
                size_t r = static_cast<size_t>(b) * G + j;
                if (a.dbg.max_draft) a.dbg.max_draft[r] = nanf("");
                if (a.dbg.lse_draft) a.dbg.lse_draft[r] = nan("");
                if (a.dbg.p_x) a.dbg.p_x[r] = nan("");
                if (a.dbg.q_x) a.dbg.q_x[r] = nan("");
            }
            __syncthreads();
            continue;
        }

        // Per-row checking outputs.
        const int last = a.early ? sh.last_row : (a.onehot ? np : G);  // last target row read
        for (int j = threadIdx.x; j <= G; j += kThreads) {
            size_t r = static_cast<size_t>(b) * (G + 1) + j;
            const bool read = j <= last;
            const RowStat& st = sh.st[j];
            if (a.dbg.max_target) a.dbg.max_target[r] = read ? st.m : nanf("");
            if (a.dbg.lse_target)
                a.dbg.lse_target[r] = (greedy || !read) ? nan("") : lse_from_stats(st.m, st.s, c, T);
            if (a.dbg.argmax_target) a.dbg.argmax_target[r] = (greedy && read) ? st.idx : -1;
        }
        for (int j = threadIdx.x; j < G; j += kThreads) {
            size_t r = static_cast<size_t>(b) * G + j;
            const bool draft = !greedy && !a.onehot && (!a.early || (j <= last && j < np));
            const RowStat& st = sh.st[G + 1 + j];
            if (a.dbg.max_draft) a.dbg.max_draft[r] = draft ? st.m : nanf("");
            if (a.dbg.lse_draft) a.dbg.lse_draft[r] = draft ? lse_from_stats(st.m, st.s, c, T) : nan("");
            if (a.dbg.p_x) a.dbg.p_x[r] = nan("");
            if (a.dbg.q_x) a.dbg.q_x[r] = nan("");
        }
        __syncthreads();

        // Left-to-right acceptance scan on one thread.
        if (threadIdx.x == 0) {
            const int32_t* tok = a.tokens + static_cast<size_t>(b) * G;
            int n = np;
            if (greedy) {
                for (int i = 0; i < np; ++i) {
                    if (tok[i] != sh.st[i].idx) {
                        n = i;
                        break;
                    }
                    out[i] = tok[i];
                }
                out[n] = sh.st[n].idx;
                if (a.dbg.kind) a.dbg.kind[b] = kKindGreedy;
                if (a.dbg.w_total) a.dbg.w_total[b] = nan("");
            } else {
                const float* ua = a.u_accept + static_cast<size_t>(b) * G;
                for (int i = 0; i < np; ++i) {
                    const int x = tok[i];
                    const size_t tr = static_cast<size_t>(b) * (G + 1) + i;
                    const size_t dr = static_cast<size_t>(b) * G + i;
                    const RowStat& sp = sh.st[i];
                    const RowStat& sq = sh.st[G + 1 + i];
                    double p = prob_from_stats(load_logit<DT>(a.target, tr * V + x), sp.m, sp.s, c);
                    // a one-hot proposal has q(x) = 1
                    double q = a.onehot ? 1.0 : prob_from_stats(load_logit<DT>(a.draft, dr * V + x), sq.m, sq.s, c);
                    if (a.dbg.p_x) a.dbg.p_x[dr] = p;
                    if (a.dbg.q_x) a.dbg.q_x[dr] = q;
                    if (!accept_draft(p, q, ua[i])) {
                        n = i;
                        break;
                    }
                    out[i] = x;
                }
                DrawParams d;
                d.c = c;
                d.mcp = scaled_max(sh.st[n].m, c);
                d.isp = __frcp_rn(sh.st[n].s);
                d.excl = -1;
                if (n < np && !a.onehot) {
                    d.kind = kKindResidual;
                    d.mcq = scaled_max(sh.st[G + 1 + n].m, c);
                    d.isq = __frcp_rn(sh.st[G + 1 + n].s);
                    d.fix = kFixResidual;
                } else {
                    // the extra token, or the residual of a one-hot proposal
                    // (p_n without x_n, unnormalised weights)
                    d.kind = n < np ? kKindResidualOnehot : kKindBonus;
                    d.excl = n < np ? tok[n] : -1;
                    d.mcq = 0.0f;
                    d.isq = 0.0f;
                    d.fix = kFixTarget;
                }
                sh.draw = d;
                if (a.dbg.kind) a.dbg.kind[b] = d.kind == kKindResidualOnehot ? kKindResidual : d.kind;
            }
            for (int j = n + 1; j <= G; ++j) out[j] = -1;
            a.out_num_accepted[b] = n;
            sh.n = n;
        }
        __syncthreads();

        if (!greedy) {
            // Inverse-CDF draw over row n: thread t owns tokens [t*E, t*E + E).
            const int n = sh.n;
            DrawParams d = sh.draw;
            const size_t trow = (static_cast<size_t>(b) * (G + 1) + n) * V;
            const size_t drow = (static_cast<size_t>(b) * G + (n < G ? n : 0)) * V;
            const int E = (V + kThreads - 1) / kThreads;
            const int lo = min(V, static_cast<int>(threadIdx.x) * E), hi = min(V, lo + E);
            int kind = d.kind;
            float run = run_weights<DT>(a.target, a.draft, trow, drow, lo, hi, d, kind);
            unsigned long long qv = to_fixed(run, d.fix), total;
            unsigned long long excl = block_excl_scan_u64<kThreads>(qv, sh.scan, &total);
            if (total == 0ull) {
                // Residual weights that round to zero everywhere: draw from p_n.
                kind = kKindBonus;
                d.fix = kFixTarget;
                run = run_weights<DT>(a.target, a.draft, trow, drow, lo, hi, d, kind);
                qv = to_fixed(run, d.fix);
                excl = block_excl_scan_u64<kThreads>(qv, sh.scan, &total);
            }
            const unsigned long long t = scale_uniform(a.u_sample[b], total);
            if (excl <= t && t < excl + qv) {
                float run2 = 0.0f;
                int token = hi - 1;
                for (int e = lo; e < hi; ++e) {
                    float lt = load_logit<DT>(a.target, trow + e);
                    float w = kind == kKindResidual
                                  ? weight_residual(lt, load_logit<DT>(a.draft, drow + e), d)
                                  : weight_target_excl(lt, e, d, kind);
                    run2 = __fadd_rn(run2, w);
                    if (excl + to_fixed(run2, d.fix) > t) {
                        token = e;
                        break;
                    }
                }
                out[n] = token;
            }
            if (threadIdx.x == 0 && a.dbg.w_total)  // target weights reported normalised by s
                a.dbg.w_total[b] = kind == kKindResidual
                                       ? static_cast<double>(total) * kFixResidualInv
                                       : static_cast<double>(total) * kFixTargetInv /
                                             static_cast<double>(sh.st[n].s);
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_rowwise(const Args& a, const DeviceInfo& dev, cudaStream_t stream) {
    const int grid = static_cast<int>(std::min<long long>(a.B, static_cast<long long>(dev.num_sms) * 16));
    if (a.dtype == SV_F32)
        rowwise_kernel<SV_F32><<<grid, kThreads, 0, stream>>>(a);
    else
        rowwise_kernel<SV_BF16><<<grid, kThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace sv
