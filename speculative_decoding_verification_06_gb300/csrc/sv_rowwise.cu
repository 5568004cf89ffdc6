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
#include <type_traits>

#include "sv_common.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;

struct RowStat {
    float m;      // max (T > 0) or max value (T == 0)
    float s;      // sum of the terms of the row (T > 0), anchored or plain
    int32_t idx;  // lowest-index argmax (T == 0)
    int32_t bad;  // NaN, +inf, or only -inf
    int32_t plain;  // s is in the plain form (T > 0)
};

__device__ __forceinline__ MaxSum ms_of(const RowStat& r) { return MaxSum{r.m, r.s, r.plain}; }

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
    int excl[SV_MAX_GAMMA];  // tree: tokens of the rejected children at the last node
    int nexcl;
    int draw_row;            // the row of the draw (tree: the last node)
    int row_flag;            // the last row pass found the anchored form out of range
    // the scan's inputs, read by one thread a position before the scan
    int px[SV_MAX_GAMMA];    // proposed token
    float pu[SV_MAX_GAMMA];  // its uniform
    float plt[SV_MAX_GAMMA]; // target logit at the token
    float pld[SV_MAX_GAMMA]; // draft logit at the token
};

// Logits a thread folds into one partial before the partial joins its running
// state: the binary32 sums then stay short at any V (a thread sees V / 128 of a
// row, 131072 logits at V = 2^24).
constexpr int kInner = 64;

// One pass over a row: the anchored form (PLAIN false; a thread whose
// anchor leaves its range sets the row's plain flag) or the plain form.
template <int DT, bool PLAIN>
__device__ RowStat row_pass(const void* base, size_t row, int V, const Scale& c, Shared& sh) {
    using State = typename std::conditional<PLAIN, MaxSum, MaxSumA>::type;
    auto empty = []() -> State {
        if constexpr (PLAIN) return MaxSum{neg_inf(), 0.0f, 1};
        else return MaxSumA{neg_inf(), 0.0f};
    };
    auto merge = [&](State a, State b) -> State {
        if constexpr (PLAIN) return maxsum_merge(a, b, c);
        else return maxsum_merge_a(a, b, c.c);
    };
    State st = empty();
    int bad = 0, flag = 0;
    const size_t off = row * static_cast<size_t>(V);
    for (int x0 = threadIdx.x; x0 < V; x0 += kThreads * kInner) {
        State part = empty();
        const int x1 = static_cast<int>(min(static_cast<long long>(V), static_cast<long long>(x0) + kThreads * kInner));
        for (int x = x0; x < x1; x += kThreads) {
            const float l = load_logit<DT>(base, off + x);
            if (bad_logit(l)) {
                bad = 1;
            } else {
                if constexpr (PLAIN) maxsum_add(part, l, c);
                else maxsum_add_a(part, l, c.c, flag);
            }
        }
        st = merge(st, part);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        State other = st;
        other.m = __shfl_xor_sync(0xffffffffu, st.m, o);
        other.s = __shfl_xor_sync(0xffffffffu, st.s, o);
        st = merge(st, other);
    }
    bad = __any_sync(0xffffffffu, bad);
    flag = __any_sync(0xffffffffu, flag);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        sh.ms[warp] = MaxSum{st.m, st.s, PLAIN ? 1 : 0};
        sh.bad[warp] = bad | (flag << 1);
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
        r = {acc.m, acc.s, -1, ((b & 1) || acc.m == neg_inf()) ? 1 : 0, acc.plain};
        sh.row_flag = (b & 2) && !(r.bad);
    }
    __syncthreads();
    return r;  // meaningful on thread 0 only
}

// A row's statistics in the anchored form, or (when its anchor left the
// range, or c overflowed) recomputed in the plain form by a second pass.
template <int DT>
__device__ RowStat row_maxsum(const void* base, size_t row, int V, const Scale& c, Shared& sh) {
    const RowStat r = row_pass<DT, false>(base, row, V, c, sh);
    if (!sh.row_flag) return r;
    __syncthreads();  // every thread has read the flag before the next pass clears it
    return row_pass<DT, true>(base, row, V, c, sh);
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
        r = {acc.v, 0.0f, acc.i, (b || acc.v == neg_inf()) ? 1 : 0, 0};
    }
    __syncthreads();
    return r;
}

// Rows of at most kWarpRow logits are reduced by one warp each (at most 64
// logits a lane, so one partial, as in the block pass), with no block
// barrier: the block's warps take the request's rows kWarps at a time and
// their loads overlap. Same forms and flags as row_pass / row_argmax; the
// result is on every lane.
constexpr int kWarpRow = 32 * kInner;

template <int DT, bool PLAIN>
__device__ RowStat warp_row_pass(const void* base, size_t row, int V, const Scale& c, int& flag_out) {
    using State = typename std::conditional<PLAIN, MaxSum, MaxSumA>::type;
    State st;
    if constexpr (PLAIN) st = MaxSum{neg_inf(), 0.0f, 1};
    else st = MaxSumA{neg_inf(), 0.0f};
    int bad = 0, flag = 0;
    const size_t off = row * static_cast<size_t>(V);
    for (int x = threadIdx.x & 31; x < V; x += 32) {
        const float l = load_logit<DT>(base, off + x);
        if (bad_logit(l)) {
            bad = 1;
        } else {
            if constexpr (PLAIN) maxsum_add(st, l, c);
            else maxsum_add_a(st, l, c.c, flag);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        State other = st;
        other.m = __shfl_xor_sync(0xffffffffu, st.m, o);
        other.s = __shfl_xor_sync(0xffffffffu, st.s, o);
        if constexpr (PLAIN) st = maxsum_merge(st, other, c);
        else st = maxsum_merge_a(st, other, c.c);
    }
    bad = __any_sync(0xffffffffu, bad);
    flag = __any_sync(0xffffffffu, flag);
    const RowStat r{st.m, st.s, -1, (bad || st.m == neg_inf()) ? 1 : 0, PLAIN ? 1 : 0};
    flag_out = flag && !r.bad;
    return r;
}

template <int DT>
__device__ RowStat warp_row_maxsum(const void* base, size_t row, int V, const Scale& c) {
    int flag = 0;
    const RowStat r = warp_row_pass<DT, false>(base, row, V, c, flag);
    if (!flag) return r;
    return warp_row_pass<DT, true>(base, row, V, c, flag);
}

template <int DT>
__device__ RowStat warp_row_argmax(const void* base, size_t row, int V) {
    ArgMax st = argmax_empty();
    int bad = 0;
    const size_t off = row * static_cast<size_t>(V);
    for (int x = threadIdx.x & 31; x < V; x += 32) {
        const float l = load_logit<DT>(base, off + x);
        if (bad_logit(l)) bad = 1;
        if (l > st.v) st = {l, x};  // increasing x: the first maximum stays
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ArgMax other{__shfl_xor_sync(0xffffffffu, st.v, o), __shfl_xor_sync(0xffffffffu, st.i, o)};
        st = argmax_merge(st, other);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (st.i == 0x7fffffff) st.i = 0;
    return RowStat{st.v, 0.0f, st.i, (bad || st.v == neg_inf()) ? 1 : 0, 0};
}

// Sum of the draw weights over [lo, hi) in index order (binary32).
// Weight of token e of a draw (residual, extra token, one-hot or tree residual).
template <int DT>
__device__ __forceinline__ float draw_weight(const void* tgt, const void* dft, size_t trow, size_t drow, int e,
                                             const DrawParams& d, int kind, const int* excl, int nexcl) {
    const float lt = load_logit<DT>(tgt, trow + e);
    if (kind == kKindResidual) return weight_residual(lt, load_logit<DT>(dft, drow + e), d);
    if (kind == kKindResidualTree) return in_set(e, excl, nexcl) ? 0.0f : weight_target(lt, d);
    return weight_target_excl(lt, e, d, kind);
}

// A thread's tokens are summed in runs of kRun: each run in binary32 in index
// order, converted to fixed point, and the runs added exactly, so that no
// binary32 sum is longer than kRun at any V.
constexpr int kRun = 32;

template <int DT>
__device__ __forceinline__ float run_weights(const void* tgt, const void* dft, size_t trow,
                                             size_t drow, int lo, int hi, const DrawParams& d,
                                             int kind, const int* excl, int nexcl) {
    float run = 0.0f;
    for (int e = lo; e < hi; ++e) run = __fadd_rn(run, draw_weight<DT>(tgt, dft, trow, drow, e, d, kind, excl, nexcl));
    return run;
}

// The fixed-point sum of tokens [lo, hi), run by run.
template <int DT>
__device__ unsigned long long range_weights(const void* tgt, const void* dft, size_t trow, size_t drow, int lo,
                                            int hi, const DrawParams& d, int kind, const int* excl, int nexcl) {
    unsigned long long q = 0ull;
    for (int r = lo; r < hi; r += kRun)
        q += to_fixed(run_weights<DT>(tgt, dft, trow, drow, r, min(hi, r + kRun), d, kind, excl, nexcl), d.fix);
    return q;
}

template <int DT>
__global__ void __launch_bounds__(kThreads) rowwise_kernel(Args a) {
    __shared__ Shared sh;
    const int G = a.gamma, V = a.V;
    for (int b = blockIdx.x; b < a.B; b += gridDim.x) {
        const float T = a.temperature[b];
        const bool t_ok = (T >= 0.0f) && (T < pos_inf());
        const bool greedy = t_ok && T == 0.0f;
        const Scale c = (t_ok && !greedy) ? temp_scale(T) : Scale{0.0f, 0.0f};
        // proposals: gamma, or num_draft[b] for one-hot proposals (no draft
        // rows; target rows past num_draft[b] take no part)
        const int kb = a.onehot && a.num_draft ? a.num_draft[b] : G;
        const bool range_ok = t_ok && kb >= 0 && kb <= G;
        const int np = range_ok ? kb : 0;
        int bad = range_ok ? 0 : 1;
        for (int i = threadIdx.x; i < np; i += kThreads) {
            int x = a.tokens[static_cast<size_t>(b) * G + i];
            if (x < 0 || x >= V) bad = 1;
            // tree: node i + 1's parent is an earlier node
            if (a.tree) {
                const int par = a.parents[static_cast<size_t>(b) * G + i];
                if (par < 0 || par > i) bad = 1;
            }
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
                            const float lt = load_logit<DT>(a.target, trow * V + x);
                            const float u = a.u_accept[static_cast<size_t>(b) * G + i];
                            // alpha from the logits: p(x) and q(x) may both lie below
                            // the floating-point range while their ratio does not
                            const bool acc =
                                a.onehot ? accept_from_logits(lt, 0.0f, ms_of(st), MaxSum{0.0f, 1.0f, 0}, c, u)
                                         : accept_from_logits(
                                               lt, load_logit<DT>(a.draft, (static_cast<size_t>(b) * G + i) * V + x),
                                               ms_of(st), ms_of(sd), c, u);
                            stop = acc ? 0 : 1;
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
            if (V <= kWarpRow) {
                // a warp a row (the warp's loop is uniform: r depends on the warp only)
                for (int r = threadIdx.x >> 5; r < nrows; r += kWarps) {
                    RowStat st;
                    if (r <= G) {
                        size_t row = static_cast<size_t>(b) * (G + 1) + r;
                        st = greedy ? warp_row_argmax<DT>(a.target, row, V) : warp_row_maxsum<DT>(a.target, row, V, c);
                    } else {
                        st = warp_row_maxsum<DT>(a.draft, static_cast<size_t>(b) * G + (r - G - 1), V, c);
                    }
                    if ((threadIdx.x & 31) == 0) sh.st[r] = st;
                }
                __syncthreads();
            } else {
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
                a.dbg.lse_target[r] = (greedy || !read) ? nan("") : lse_from_stats(ms_of(st), c, T);
            if (a.dbg.argmax_target) a.dbg.argmax_target[r] = (greedy && read) ? st.idx : -1;
        }
        for (int j = threadIdx.x; j < G; j += kThreads) {
            size_t r = static_cast<size_t>(b) * G + j;
            const bool draft = !greedy && !a.onehot && (!a.early || (j <= last && j < np));
            const RowStat& st = sh.st[G + 1 + j];
            if (a.dbg.max_draft) a.dbg.max_draft[r] = draft ? st.m : nanf("");
            if (a.dbg.lse_draft) a.dbg.lse_draft[r] = draft ? lse_from_stats(ms_of(st), c, T) : nan("");
            if (a.dbg.p_x) a.dbg.p_x[r] = nan("");
            if (a.dbg.q_x) a.dbg.q_x[r] = nan("");
        }
        // The linear scan's inputs, a thread a position, so that the scan on
        // one thread does not wait on a read per position (positions up to
        // the last row read: early exit reads nothing past it).
        if (!a.tree) {
            const int npre = min(np, last + 1);
            for (int i = threadIdx.x; i < npre; i += kThreads) {
                const int x = a.tokens[static_cast<size_t>(b) * G + i];
                sh.px[i] = x;
                if (!greedy) {
                    sh.pu[i] = a.u_accept[static_cast<size_t>(b) * G + i];
                    sh.plt[i] = load_logit<DT>(a.target, (static_cast<size_t>(b) * (G + 1) + i) * V + x);
                    sh.pld[i] = a.onehot ? 0.0f : load_logit<DT>(a.draft, (static_cast<size_t>(b) * G + i) * V + x);
                }
            }
        }
        __syncthreads();

        // Left-to-right acceptance scan on one thread.
        if (threadIdx.x == 0 && a.tree) {
            // Tree walk: at node u the children (nodes whose parent is u) are tried
            // in index order; child c is accepted with min(1, p'(x_c)), p' being
            // p without the tokens of the children rejected so far, renormalised;
            // an accepted child becomes u. With every child rejected (or a leaf)
            // the last token is drawn from p'; at T = 0 the first child whose
            // token is the argmax is taken.
            const int32_t* tok = a.tokens + static_cast<size_t>(b) * G;
            const int32_t* par = a.parents + static_cast<size_t>(b) * G;
            const float* ua = a.u_accept + static_cast<size_t>(b) * G;
            int u = 0, n = 0, ne = 0;
            for (;;) {
                if (greedy) {
                    const int am = sh.st[u].idx;
                    int next = -1;
                    for (int cn = 1; cn <= np && next < 0; ++cn)
                        if (par[cn - 1] == u && tok[cn - 1] == am) next = cn;
                    out[n] = am;
                    if (next < 0) break;
                    if (a.out_nodes) a.out_nodes[static_cast<size_t>(b) * G + n] = next;
                    ++n;
                    u = next;
                    continue;
                }
                const size_t tr = static_cast<size_t>(b) * (G + 1) + u;
                double R = 0.0;  // probability of the rejected children
                int next = -1;
                ne = 0;
                for (int cn = 1; cn <= np && next < 0; ++cn) {
                    if (par[cn - 1] != u) continue;
                    const int x = tok[cn - 1];
                    const bool seen = in_set(x, sh.excl, ne);
                    const double px =
                        seen ? 0.0 : prob_from_stats(load_logit<DT>(a.target, tr * V + x), ms_of(sh.st[u]), c);
                    const double rest = 1.0 - R;
                    const double alpha = rest > 0.0 ? fmin(1.0, px / rest) : 0.0;
                    const size_t dr = static_cast<size_t>(b) * G + (cn - 1);
                    if (a.dbg.p_x) a.dbg.p_x[dr] = px;
                    if (a.dbg.q_x) a.dbg.q_x[dr] = 1.0;
                    // u = 0 accepts whenever p'(x) > 0, also where it underflows
                    if (ua[cn - 1] < alpha || (ua[cn - 1] == 0.0f && !seen && rest > 0.0 &&
                                               load_logit<DT>(a.target, tr * V + x) > neg_inf())) {
                        next = cn;
                    } else if (!seen) {
                        sh.excl[ne++] = x;
                        R += px;
                    }
                }
                if (next < 0) break;
                out[n] = tok[next - 1];
                if (a.out_nodes) a.out_nodes[static_cast<size_t>(b) * G + n] = next;
                ++n;
                u = next;
            }
            if (a.out_nodes)
                for (int j = n; j < G; ++j) a.out_nodes[static_cast<size_t>(b) * G + j] = -1;
            if (greedy) {
                if (a.dbg.kind) a.dbg.kind[b] = kKindGreedy;
                if (a.dbg.w_total) a.dbg.w_total[b] = nan("");
            } else {
                DrawParams d;
                draw_rows(d, ne > 0 ? kKindResidualTree : kKindBonus, ms_of(sh.st[u]), nullptr, c);
                d.excl = -1;
                d.fix = kFixTarget;
                sh.draw = d;
                if (a.dbg.kind) a.dbg.kind[b] = ne > 0 ? kKindResidual : kKindBonus;
            }
            sh.nexcl = ne;
            sh.draw_row = u;
            for (int j = n + 1; j <= G; ++j) out[j] = -1;
            a.out_num_accepted[b] = n;
            sh.n = n;
        } else if (threadIdx.x == 0) {
            const int32_t* tok = a.tokens + static_cast<size_t>(b) * G;
            int n = np;
            if (greedy) {
                for (int i = 0; i < np; ++i) {
                    if (sh.px[i] != sh.st[i].idx) {
                        n = i;
                        break;
                    }
                    out[i] = sh.px[i];
                }
                out[n] = sh.st[n].idx;
                if (a.dbg.kind) a.dbg.kind[b] = kKindGreedy;
                if (a.dbg.w_total) a.dbg.w_total[b] = nan("");
            } else {
                for (int i = 0; i < np; ++i) {
                    const int x = sh.px[i];
                    const size_t dr = static_cast<size_t>(b) * G + i;
                    const RowStat& sp = sh.st[i];
                    const RowStat& sq = sh.st[G + 1 + i];
                    const float lt = sh.plt[i], ld = sh.pld[i];
                    if (a.dbg.p_x) a.dbg.p_x[dr] = prob_from_stats(lt, ms_of(sp), c);
                    // a one-hot proposal has q(x) = 1
                    if (a.dbg.q_x) a.dbg.q_x[dr] = a.onehot ? 1.0 : prob_from_stats(ld, ms_of(sq), c);
                    // alpha from the logits: p(x) and q(x) may both lie below the
                    // floating-point range while their ratio does not
                    const bool acc = a.onehot ? accept_from_logits(lt, 0.0f, ms_of(sp), MaxSum{0.0f, 1.0f, 0}, c, sh.pu[i])
                                              : accept_from_logits(lt, ld, ms_of(sp), ms_of(sq), c, sh.pu[i]);
                    if (!acc) {
                        n = i;
                        break;
                    }
                    out[i] = x;
                }
                DrawParams d;
                d.excl = -1;
                if (n < np && !a.onehot) {
                    const MaxSum sq = ms_of(sh.st[G + 1 + n]);
                    draw_rows(d, kKindResidual, ms_of(sh.st[n]), &sq, c);
                    d.fix = kFixResidual;
                } else {
                    // the extra token, or the residual of a one-hot proposal
                    // (p_n without x_n, unnormalised weights)
                    draw_rows(d, n < np ? kKindResidualOnehot : kKindBonus, ms_of(sh.st[n]), nullptr, c);
                    d.excl = n < np ? tok[n] : -1;
                    d.fix = kFixTarget;
                }
                sh.draw = d;
                if (a.dbg.kind) a.dbg.kind[b] = d.base_kind() == kKindResidualOnehot ? kKindResidual : d.base_kind();
            }
            for (int j = n + 1; j <= G; ++j) out[j] = -1;
            a.out_num_accepted[b] = n;
            sh.n = n;
            sh.nexcl = 0;
            sh.draw_row = n;
        }
        __syncthreads();

        if (!greedy) {
            // Inverse-CDF draw over row n: thread t owns tokens [t*E, t*E + E).
            const int n = sh.n, row = sh.draw_row, nexcl = sh.nexcl;
            DrawParams d = sh.draw;
            const size_t trow = (static_cast<size_t>(b) * (G + 1) + row) * V;
            const size_t drow = (static_cast<size_t>(b) * G + (row < G ? row : 0)) * V;
            const int E = (V + kThreads - 1) / kThreads;
            const int lo = min(V, static_cast<int>(threadIdx.x) * E), hi = min(V, lo + E);
            int kind = d.base_kind();
            unsigned long long qv = range_weights<DT>(a.target, a.draft, trow, drow, lo, hi, d, kind, sh.excl, nexcl);
            unsigned long long total;
            unsigned long long excl = block_excl_scan_u64<kThreads>(qv, sh.scan, &total);
            if (total == 0ull) {
                // Residual weights that round to zero everywhere: draw from p_n.
                kind = kKindBonus;
                d.fix = kFixTarget;
                qv = range_weights<DT>(a.target, a.draft, trow, drow, lo, hi, d, kind, sh.excl, nexcl);
                excl = block_excl_scan_u64<kThreads>(qv, sh.scan, &total);
            }
            const unsigned long long t = scale_uniform(a.u_sample[b], total);
            if (excl <= t && t < excl + qv) {
                // the run holding t, then the token, with the same run sums
                int token = hi - 1;
                unsigned long long before = excl;
                for (int r = lo; r < hi; r += kRun) {
                    const int r1 = min(hi, r + kRun);
                    const unsigned long long qr = to_fixed(
                        run_weights<DT>(a.target, a.draft, trow, drow, r, r1, d, kind, sh.excl, nexcl), d.fix);
                    if (before + qr > t) {
                        float run2 = 0.0f;
                        token = r1 - 1;
                        for (int e = r; e < r1; ++e) {
                            run2 = __fadd_rn(run2,
                                             draw_weight<DT>(a.target, a.draft, trow, drow, e, d, kind, sh.excl, nexcl));
                            if (before + to_fixed(run2, d.fix) > t) {
                                token = e;
                                break;
                            }
                        }
                        break;
                    }
                    before += qr;
                }
                out[n] = token;
            }
            if (threadIdx.x == 0 && a.dbg.w_total)  // target weights reported normalised by s
                a.dbg.w_total[b] = kind == kKindResidual
                                       ? static_cast<double>(total) * kFixResidualInv
                                       : static_cast<double>(total) * kFixTargetInv * static_cast<double>(d.isp);
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
