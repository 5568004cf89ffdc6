// Cluster path of libspecverify: one thread-block cluster verifies one request.
//
// For batches too small to keep 152 SMs streaming through the persistent
// kernel (a few requests, or short rows), every row of a request is cut into
// C equal 16-byte-aligned slices, one per CTA of the request's cluster
// (C <= 16). Each CTA folds its slice of every row the request needs into a
// (max, sum) or argmax record and pushes it into the leader's (rank 0's)
// shared memory over distributed shared memory (mapa + st.shared::cluster);
// after a cluster barrier the leader merges the C records of each row in rank
// order and runs the acceptance scan on one warp. A draw is made by the whole cluster: each CTA sums the weights of
// its slice of the draw row in runs of 32 tokens (fixed point, exact), the
// leader finds the CTA whose share holds u * W, and that CTA finds the run,
// then the token. Four cluster barriers separate the phases; nothing goes
// through global memory but the inputs and the outputs, so there is no
// workspace, no memset and no cross-block polling.
//
// Method: "Speculative Decoding : accélérer l'inférence des LLM", §Pourquoi la
// qualité est préservée (accept with min(1, p(x)/q(x)); residual max(p - q, 0)
// renormalised; greedy rule); wiki "Speculative Decoding", eq. alpha(x) and
// eq. p_corr; "Accélérer Sonar grâce à la spéculation", §Décodage spéculatif
// (the extra token after the last accepted draft token).
#include <algorithm>
#include <cmath>

#include "sv_common.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 16;
constexpr int kMaxPieces = 8;  // pieces a CTA's slice of one row is cut into (handed to warps round-robin)
constexpr int kMaxRows = 2 * SV_MAX_GAMMA + 1;
constexpr int kRun = 32;        // draw: tokens summed in binary32 before conversion to fixed point
constexpr int kMaxSlice = 65536;  // elements of one row in one CTA (V <= 16 * 65536)

// A row record: (max, sum; idx = 1 for a plain sum, else -1) or (max value,
// lowest-index argmax), and the data-error flag.
struct CRec {
    float m;
    float s;
    int32_t idx;
    int32_t bad;
};

__device__ __forceinline__ MaxSum ms_of(const CRec& r) { return MaxSum{r.m, r.s, r.idx == 1 ? 1 : 0}; }

// The draw as the leader hands it to every CTA.
struct CJob {
    DrawParams d;
    int draw;  // 1 when a draw runs (a valid sampled request)
    int kind;  // its kind
    int row;   // target (and draft) row of the draw
    int slot;  // output position of the drawn token
};

// Shared memory of each CTA. Nothing is read from another CTA's shared
// memory: each CTA pushes what the leader needs into the leader's (its row
// records, its draw total) and the leader pushes the draw and the choice of
// the CTA that searches into every CTA's, each before a cluster barrier.
struct CShared {
    CJob job;                              // pushed by the leader
    int redo;                              // pushed by the leader: every residual weight was zero, draw from p
    int sel;                               // pushed by the leader: the rank whose share holds t
    unsigned long long sel_t;              // pushed by the leader: t less the shares of the ranks before sel
    unsigned long long totals[kMaxCluster];  // leader: pushed by each rank, its draw total
    CRec st[kMaxRows];                     // leader: the merged record of each row
    unsigned long long wsum[kWarps];
    int x[64];                             // leader: proposed tokens 0..63
    float u[64], lt[64], ld[64];           // leader: their uniforms, target and draft logits
    float us;                              // leader: the draw's uniform
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ int cluster_rank() {
    int r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The address of `p` (this CTA's shared memory) in the shared memory of CTA
// `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(const void* p, int rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, const uint4& v) {
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void st_cluster_u64(uint32_t addr, unsigned long long v) {
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

// Every thread of every CTA of the cluster: the writes to shared memory
// before it are visible to the reads after it, in any CTA of the cluster.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ CRec crec_merge(CRec x, const CRec& y, bool argmax, const Scale& sc) {
    const int bad = x.bad | y.bad;
    if (argmax) {
        const ArgMax m = argmax_merge(ArgMax{x.m, x.idx}, ArgMax{y.m, y.idx});
        return CRec{m.v, 0.0f, m.i, bad};
    }
    const MaxSum m = maxsum_merge(ms_of(x), ms_of(y), sc);
    return CRec{m.m, m.s, m.plain ? 1 : -1, bad};
}

__device__ __forceinline__ CRec crec_empty(bool argmax) {
    return argmax ? CRec{neg_inf(), 0.0f, 0x7fffffff, 0} : CRec{neg_inf(), 0.0f, -1, 0};
}

// Maxima that propagate NaN (a NaN logit makes its row invalid).
__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t x, uint32_t y) {
    uint32_t r;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(y));
    return r;
}
__device__ __forceinline__ float f32_max_nan(float x, float y) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(x), "f"(y));
    return r;
}

// [lo, hi) of part g of n equal parts of [0, len), cut on multiples of vec.
__device__ __forceinline__ int part_at(int len, int n, int g, int vec) {
    if (g <= 0) return 0;
    if (g >= n) return len;
    const long long x = static_cast<long long>(len) * g / n;
    return static_cast<int>(x - x % vec);
}

template <int DT>
struct Cluster {
    static constexpr int ES = DT == SV_F32 ? 4 : 2;
    static constexpr int kVec = 16 / ES;  // elements per 16-byte vector

    const Args& a;
    CShared& sh;
    CRec* pieces;               // [rows][P] records of this CTA's pieces
    unsigned long long* runs;   // draw: fixed-point sum of each run of this CTA's slice
    int C, c, b, lo, len;

    // Row r of the request: target rows 0..gamma, then draft rows.
    __device__ const void* row_base(int r) const {
        const int GM = a.gamma;
        return r <= GM ? static_cast<const void*>(static_cast<const char*>(a.target) +
                                                  (static_cast<size_t>(b) * (GM + 1) + r) * a.V * ES)
                       : static_cast<const void*>(static_cast<const char*>(a.draft) +
                                                  (static_cast<size_t>(b) * GM + (r - GM - 1)) * a.V * ES);
    }

    // The logits of a 16-byte vector.
    __device__ static void unpack(const uint4& v, float (&l)[kVec]) {
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < kVec; ++k)
            l[k] = DT == SV_BF16 ? ((k & 1) ? bf16x2_hi(w4[k >> 1]) : bf16x2_lo(w4[k >> 1])) : __uint_as_float(w4[k]);
    }

    // v[q] for a q known only at run time, by selects (the array stays in
    // registers; no local memory).
    template <int N>
    __device__ static uint4 pick(const uint4 (&v)[N], int q) {
        uint4 r = v[0];
#pragma unroll
        for (int k = 1; k < N; ++k)
            if (q == k) r = v[k];
        return r;
    }

    // One warp folds elements [e0, e1) of a row (row-relative, multiples of
    // kVec) into a record: lanes take 16-byte vectors lane, lane + 32, ... in
    // order (eight loads in flight per lane), each lane folds its elements in
    // index order, then the lanes merge in a fixed order. The loops are kept
    // rolled: these kernels are short, and their time goes to fetching code
    // as much as to fetching data.
    __device__ CRec fold_piece(const void* row, int e0, int e1, bool argmax, const Scale& sc) const {
        const int lane = threadIdx.x & 31;
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const char*>(row) + static_cast<size_t>(e0) * ES);
        const int nvec = (e1 - e0) / kVec;
        ArgMax am = argmax_empty();
        MaxSum ms = maxsum_empty();
        int bad = 0;
        for (int v0 = 0; v0 < nvec; v0 += 32 * 8) {
            uint4 v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int vi = v0 + q * 32 + lane;
                v[q] = vi < nvec ? __ldg(src + vi) : make_uint4(0u, 0u, 0u, 0u);
            }
            if (argmax) {
                // the lane's max over the eight vectors (packed, NaN-propagating;
                // vectors past the piece hold -inf), then, only when it beats
                // the running max, the first position holding it
                float tmax;
                if (DT == SV_BF16) {
                    uint32_t m2 = 0xff80ff80u;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const uint4 w = v0 + q * 32 + lane < nvec ? v[q] : make_uint4(0xff80ff80u, 0xff80ff80u,
                                                                                          0xff80ff80u, 0xff80ff80u);
                        m2 = bf16x2_max_nan(m2, bf16x2_max_nan(bf16x2_max_nan(w.x, w.y), bf16x2_max_nan(w.z, w.w)));
                    }
                    tmax = f32_max_nan(bf16x2_lo(m2), bf16x2_hi(m2));
                } else {
                    tmax = neg_inf();
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        if (v0 + q * 32 + lane >= nvec) continue;
                        tmax = f32_max_nan(tmax, f32_max_nan(f32_max_nan(__uint_as_float(v[q].x), __uint_as_float(v[q].y)),
                                                             f32_max_nan(__uint_as_float(v[q].z), __uint_as_float(v[q].w))));
                    }
                }
                if (bad_logit(tmax)) {
                    bad = 1;
                } else if (tmax > am.v) {
                    int found = -1;
#pragma unroll 1
                    for (int q = 0; q < 8 && found < 0; ++q) {
                        const int vi = v0 + q * 32 + lane;
                        if (vi >= nvec) break;
                        float l[kVec];
                        unpack(pick(v, q), l);
#pragma unroll
                        for (int k = kVec - 1; k >= 0; --k)
                            if (l[k] == tmax) found = e0 + vi * kVec + k;
                    }
                    am = ArgMax{tmax, found};
                }
                continue;
            }
#pragma unroll 1
            for (int q = 0; q < 8; ++q) {
                const int vi = v0 + q * 32 + lane;
                if (vi >= nvec) break;
                float l[kVec];
                unpack(pick(v, q), l);
#pragma unroll
                for (int k = 0; k < kVec; ++k) {
                    if (bad_logit(l[k]))
                        bad = 1;
                    else
                        maxsum_add(ms, l[k], sc);
                }
            }
        }
        bad = __any_sync(0xffffffffu, bad);
        CRec r;
        if (argmax) {
#pragma unroll 1
            for (int o = 16; o > 0; o >>= 1) {
                ArgMax ot{__shfl_xor_sync(0xffffffffu, am.v, o), __shfl_xor_sync(0xffffffffu, am.i, o)};
                am = argmax_merge(am, ot);
            }
            r = CRec{am.v, 0.0f, am.i, bad};
        } else {
#pragma unroll 1
            for (int o = 16; o > 0; o >>= 1) {
                MaxSum ot{__shfl_xor_sync(0xffffffffu, ms.m, o), __shfl_xor_sync(0xffffffffu, ms.s, o),
                          __shfl_xor_sync(0xffffffffu, ms.plain, o)};
                ms = maxsum_merge(ms, ot, sc);
            }
            r = CRec{ms.m, ms.s, ms.plain ? 1 : -1, bad};
        }
        return r;
    }

    // Weight of token e of the draw (kind, d) from its target logit lt (and
    // draft logit ld for a residual).
    __device__ static float weight(float lt, float ld, int e, int kind, const DrawParams& d) {
        if (kind == kKindResidual) return weight_residual(lt, ld, d);
        if (kind == kKindResidualOnehot && e == d.excl) return 0.0f;
        return weight_target(lt, d);
    }

    // The 16-byte vectors of run i of this CTA's slice, tokens [lo + 32 i,
    // lo + 32 i + 32) cut at the slice's end (on a 16-byte boundary), loaded
    // all at once; returns the run's length and its first token in e0.
    static constexpr int kRunVec = kRun / kVec;
    __device__ int load_run(const void* row, int i, uint4 (&v)[kRunVec], int& e0) const {
        e0 = lo + i * kRun;
        const int n = min(kRun, lo + len - e0);
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const char*>(row) + static_cast<size_t>(e0) * ES);
#pragma unroll
        for (int q = 0; q < kRunVec; ++q) v[q] = q * kVec < n ? __ldg(src + q) : make_uint4(0u, 0u, 0u, 0u);
        return n;
    }

    // Fixed-point weight sum of run i: its tokens in index order, in binary32.
    __device__ unsigned long long run_sum(int i, int kind, const DrawParams& d, const void* trow,
                                          const void* drow) const {
        uint4 vt[kRunVec], vd[kRunVec];
        int e0;
        const int n = load_run(trow, i, vt, e0);
        if (kind == kKindResidual) load_run(drow, i, vd, e0);
        float s = 0.0f;
#pragma unroll 1
        for (int q = 0; q * kVec < n; ++q) {
            float lt[kVec], ld[kVec];
            unpack(pick(vt, q), lt);
            unpack(kind == kKindResidual ? pick(vd, q) : make_uint4(0u, 0u, 0u, 0u), ld);
#pragma unroll
            for (int k = 0; k < kVec; ++k) s = __fadd_rn(s, weight(lt[k], ld[k], e0 + q * kVec + k, kind, d));
        }
        return to_fixed(s, d.fix);
    }

    // The token of run i whose prefix (run start `start` plus the run's
    // partial sums, in the order run_sum adds them) first passes tt.
    __device__ int run_token(int i, int kind, const DrawParams& d, const void* trow, const void* drow,
                             unsigned long long start, unsigned long long tt) const {
        uint4 vt[kRunVec], vd[kRunVec];
        int e0;
        const int n = load_run(trow, i, vt, e0);
        if (kind == kKindResidual) load_run(drow, i, vd, e0);
        float part = 0.0f;
        int last_pos = -1;
#pragma unroll 1
        for (int q = 0; q * kVec < n; ++q) {
            float lt[kVec], ld[kVec];
            unpack(pick(vt, q), lt);
            unpack(kind == kKindResidual ? pick(vd, q) : make_uint4(0u, 0u, 0u, 0u), ld);
#pragma unroll
            for (int k = 0; k < kVec; ++k) {
                const float w = weight(lt[k], ld[k], e0 + q * kVec + k, kind, d);
                part = __fadd_rn(part, w);
                if (w > 0.0f) last_pos = e0 + q * kVec + k;
                if (start + to_fixed(part, d.fix) > tt) return e0 + q * kVec + k;
            }
        }
        return last_pos;  // cannot happen: the run's total passes tt
    }
};

// CS: the cluster size, fixed at compile time (1, 2, 4, 8 or 16), so that the
// launch is a plain one.
template <int DT, int CS>
__global__ void __cluster_dims__(CS, 1, 1) __launch_bounds__(kThreads)
    cluster_kernel(Args a, int rows_off, int pieces_off, int runs_off) {
    constexpr int C = CS;
    extern __shared__ __align__(16) char csmem[];
    CShared& sh = *reinterpret_cast<CShared*>(csmem);
    CRec* rows_all = reinterpret_cast<CRec*>(csmem + rows_off);  // leader: [rank][row] records pushed by each rank
    CRec* pieces = reinterpret_cast<CRec*>(csmem + pieces_off);
    unsigned long long* runs = reinterpret_cast<unsigned long long*>(csmem + runs_off);
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int c = cluster_rank();
    const int b = blockIdx.x / C;
    const int GM = a.gamma, V = a.V;
    const int nmax = 2 * GM + 1;  // rows_all's row stride
    using CL = Cluster<DT>;
    const int lo = part_at(V, C, c, CL::kVec);
    const int len = part_at(V, C, c + 1, CL::kVec) - lo;
    const int nruns = (len + kRun - 1) / kRun;
    CL K{a, sh, pieces, runs, C, c, b, lo, len};

    // This CTA's slices of the target rows (read by every request but an
    // invalid one) are asked into L2 before anything else, so that the loads
    // below, which wait for the request's temperature, find them there.
    if (t <= GM && len > 0)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                         static_cast<const char*>(a.target) + ((static_cast<size_t>(b) * (GM + 1) + t) * V + lo) * CL::ES),
                     "r"(static_cast<unsigned>(len * CL::ES))
                     : "memory");

    // the request's parameters (every CTA reads them)
    const float T = a.temperature[b];
    const bool t_ok = (T >= 0.0f) && (T < pos_inf());
    const bool greedy = t_ok && T == 0.0f;
    const bool samp = T > 0.0f && T < pos_inf();
    const Scale sc = samp ? temp_scale(T) : Scale{0.0f, 0.0f};
    const bool onehot = a.onehot;
    const int kb = onehot && a.num_draft ? a.num_draft[b] : GM;
    const bool range_ok = t_ok && kb >= 0 && kb <= GM;
    const int np = range_ok ? kb : 0;
    const int nrows = !range_ok ? 0 : (samp && !onehot ? 2 * GM + 1 : np + 1);
    // pieces per row slice: about one piece per warp, none shorter than 256 elements
    const int P = max(1, min(min(kMaxPieces, kWarps / max(1, nrows)), len / 256));

    // what the scan reads besides the rows' records: the proposed tokens, their
    // uniforms and their two logits, fetched by the leader's last warp while the
    // rows stream (proposals beyond 64 are read by the scan itself)
    if (c == 0 && warp == kWarps - 1 && range_ok) {
        if (lane == 0 && samp) sh.us = a.u_sample[b];
        for (int i = lane; i < np && i < 64; i += 32) {
            const int x = a.tokens[static_cast<size_t>(b) * GM + i];
            sh.x[i] = x;
            if (samp) {
                sh.u[i] = a.u_accept[static_cast<size_t>(b) * GM + i];
                const bool in = x >= 0 && x < V;
                sh.lt[i] = in ? load_logit<DT>(a.target, (static_cast<size_t>(b) * (GM + 1) + i) * V + x) : 0.0f;
                sh.ld[i] = (in && !onehot) ? load_logit<DT>(a.draft, (static_cast<size_t>(b) * GM + i) * V + x) : 0.0f;
            }
        }
    }

    // ---- phase 1: this CTA's slice of every row, cut into P pieces per row;
    // each row's record is pushed into the leader's shared memory
    for (int q = warp; q < nrows * P; q += kWarps) {
        const int r = q / P, j = q - r * P;
        const int e0 = lo + part_at(len, P, j, CL::kVec), e1 = lo + part_at(len, P, j + 1, CL::kVec);
        const bool am = r <= GM && !samp;
        const CRec x = K.fold_piece(K.row_base(r), e0, e1, am, sc);
        if (lane == 0) pieces[q] = x;
    }
    __syncthreads();
    for (int r = t; r < nrows; r += kThreads) {
        const bool am = r <= GM && !samp;
        CRec acc = crec_empty(am);
        for (int j = 0; j < P; ++j) acc = crec_merge(acc, pieces[r * P + j], am, sc);
        const uint4 v{__float_as_uint(acc.m), __float_as_uint(acc.s), static_cast<uint32_t>(acc.idx),
                      static_cast<uint32_t>(acc.bad)};
        st_cluster_v4(cluster_map(&rows_all[c * nmax + r], 0), v);
    }
    cluster_sync();
    // a request that is not sampled has no draw: only the leader has work left
    if (c != 0 && !samp) return;

    // ---- the leader merges each row's records (in rank order) and scans
    if (c == 0 && warp == 0) {
        const int32_t* tok = a.tokens + static_cast<size_t>(b) * GM;
        const sv_debug_out& dbg = a.dbg;
        int32_t* out = a.out_tokens + static_cast<size_t>(b) * (GM + 1);
        int bad = range_ok ? 0 : 1;
        for (int i = lane; i < np; i += 32) {
            const int x = i < 64 ? sh.x[i] : tok[i];
            if (x < 0 || x >= V) bad = 1;
        }
        for (int r = lane; r < nrows; r += 32) {
            const bool am = r <= GM && !samp;
            CRec acc = crec_empty(am);
#pragma unroll 4
            for (int k = 0; k < C; ++k) acc = crec_merge(acc, rows_all[k * nmax + r], am, sc);
            if (am) {
                if (acc.idx == 0x7fffffff) acc.idx = 0;
                if (acc.m == neg_inf()) acc.bad = 1;
            } else if (acc.m == neg_inf()) {
                acc.bad = 1;
            }
            sh.st[r] = acc;
            if (acc.bad) bad = 1;
        }
        bad = __any_sync(0xffffffffu, bad);
        __syncwarp();
        const CRec* st = sh.st;
        CJob job;
        job.draw = 0;
        if (bad) {
            for (int j = lane; j <= GM; j += 32) {
                out[j] = -1;
                const size_t r = static_cast<size_t>(b) * (GM + 1) + j;
                if (dbg.max_target) dbg.max_target[r] = nanf("");
                if (dbg.lse_target) dbg.lse_target[r] = nan("");
                if (dbg.argmax_target) dbg.argmax_target[r] = -1;
            }
            for (int j = lane; j < GM; j += 32) {
                const size_t r = static_cast<size_t>(b) * GM + j;
                if (dbg.max_draft) dbg.max_draft[r] = nanf("");
                if (dbg.lse_draft) dbg.lse_draft[r] = nan("");
                if (dbg.p_x) dbg.p_x[r] = nan("");
                if (dbg.q_x) dbg.q_x[r] = nan("");
            }
            if (lane == 0) {
                a.out_num_accepted[b] = -1;
                if (a.d_status) atomicOr(a.d_status, SV_STATUS_BAD_REQUEST);
                if (dbg.kind) dbg.kind[b] = kKindInvalid;
                if (dbg.w_total) dbg.w_total[b] = nan("");
            }
        } else {
            for (int j = lane; j <= GM; j += 32) {
                const size_t r = static_cast<size_t>(b) * (GM + 1) + j;
                const bool read = j <= np;  // one-hot: rows past the proposals are not part of the request
                if (dbg.max_target) dbg.max_target[r] = read ? st[j].m : nanf("");
                if (dbg.lse_target) dbg.lse_target[r] = (greedy || !read) ? nan("") : lse_from_stats(ms_of(st[j]), sc, T);
                if (dbg.argmax_target) dbg.argmax_target[r] = (greedy && read) ? st[j].idx : -1;
            }
            for (int j = lane; j < GM; j += 32) {
                const size_t r = static_cast<size_t>(b) * GM + j;
                const bool draft = !greedy && !onehot;
                if (dbg.max_draft) dbg.max_draft[r] = draft ? st[GM + 1 + j].m : nanf("");
                if (dbg.lse_draft) dbg.lse_draft[r] = draft ? lse_from_stats(ms_of(st[GM + 1 + j]), sc, T) : nan("");
            }
            // first failing position over all lanes (gamma may exceed 32)
            int n = np;
            for (int base = 0; base < np; base += 32) {
                const int i = base + lane;
                bool fail = false;
                if (i < np) {
                    const int x = i < 64 ? sh.x[i] : tok[i];
                    if (greedy) {
                        fail = x != st[i].idx;
                    } else {
                        const size_t tr = static_cast<size_t>(b) * (GM + 1) + i;
                        const size_t dr = static_cast<size_t>(b) * GM + i;
                        const float lt = i < 64 ? sh.lt[i] : load_logit<DT>(a.target, tr * V + x);
                        const float u = i < 64 ? sh.u[i] : a.u_accept[dr];
                        if (dbg.p_x) dbg.p_x[dr] = prob_from_stats(lt, ms_of(st[i]), sc);
                        if (onehot) {
                            if (dbg.q_x) dbg.q_x[dr] = 1.0;
                            fail = !accept_from_logits(lt, 0.0f, ms_of(st[i]), MaxSum{0.0f, 1.0f, 0}, sc, u);
                        } else {
                            const float ld = i < 64 ? sh.ld[i] : load_logit<DT>(a.draft, dr * V + x);
                            if (dbg.q_x) dbg.q_x[dr] = prob_from_stats(ld, ms_of(st[GM + 1 + i]), sc);
                            fail = !accept_from_logits(lt, ld, ms_of(st[i]), ms_of(st[GM + 1 + i]), sc, u);
                        }
                    }
                }
                const unsigned ball = __ballot_sync(0xffffffffu, fail);
                if (n == np && ball) n = base + __ffs(ball) - 1;
            }
            for (int i = lane; i < GM; i += 32)
                if (greedy || i > n || i >= np) {
                    const size_t dr = static_cast<size_t>(b) * GM + i;
                    if (dbg.p_x) dbg.p_x[dr] = nan("");
                    if (dbg.q_x) dbg.q_x[dr] = nan("");
                }
            for (int j = lane; j <= GM; j += 32) {
                if (j < n)
                    out[j] = j < 64 ? sh.x[j] : tok[j];
                else if (j == n)
                    out[j] = greedy ? st[n].idx : -1;  // the draw fills it in
                else
                    out[j] = -1;
            }
            if (greedy) {
                if (lane == 0) {
                    a.out_num_accepted[b] = n;
                    if (dbg.kind) dbg.kind[b] = kKindGreedy;
                    if (dbg.w_total) dbg.w_total[b] = nan("");
                }
            } else {
                DrawParams& d = job.d;
                d.excl = -1;
                if (n < np && !onehot) {
                    const MaxSum sq = ms_of(st[GM + 1 + n]);
                    draw_rows(d, kKindResidual, ms_of(st[n]), &sq, sc);
                    d.fix = kFixResidual;
                } else {
                    draw_rows(d, n < np ? kKindResidualOnehot : kKindBonus, ms_of(st[n]), nullptr, sc);
                    d.excl = n < np ? sh.x[n] : -1;  // n < np <= 64 when n < np reads the prefetch
                    d.fix = kFixTarget;
                }
                job.draw = 1;
                job.kind = d.base_kind();
                job.row = n;
                job.slot = n;
                if (lane == 0 && dbg.kind)
                    dbg.kind[b] = job.kind == kKindResidualOnehot ? kKindResidual : job.kind;
            }
        }
        // the draw goes to every rank (lane k writes rank k's copy)
        if (samp && lane < C) {
            const uint32_t dst = cluster_map(&sh.job, lane);
            const uint32_t* w = reinterpret_cast<const uint32_t*>(&job);
#pragma unroll 1
            for (int q = 0; q < static_cast<int>(sizeof(CJob) / 4); ++q) st_cluster_u32(dst + 4 * q, w[q]);
        }
    }
    if (!samp) return;
    cluster_sync();

    // ---- the draw, by the whole cluster (at most twice: the second from p
    // when every residual weight rounded to zero)
    if (!sh.job.draw) return;  // nothing reads another CTA's shared memory any more
    DrawParams d = sh.job.d;
    int kind = sh.job.kind;
    const void* trow = K.row_base(sh.job.row);
    const void* drow = kind == kKindResidual ? K.row_base(GM + 1 + sh.job.row) : nullptr;
    for (int pass = 0; pass < 2; ++pass) {
        if (pass == 1) {
            kind = kKindBonus;  // p at the same row, unnormalised weights
            d.fix = kFixTarget;
        }
        // each thread sums runs t, t + 256, ...; the CTA's total is exact
        unsigned long long mine = 0;
        for (int i = t; i < nruns; i += kThreads) {
            const unsigned long long q = K.run_sum(i, kind, d, trow, drow);
            runs[i] = q;
            mine += q;
        }
        mine = warp_sum_u64(mine);
        if (lane == 0) sh.wsum[warp] = mine;
        __syncthreads();
        if (t == 0) {
            unsigned long long tot = 0;
            for (int w = 0; w < kWarps; ++w) tot += sh.wsum[w];
            st_cluster_u64(cluster_map(&sh.totals[c], 0), tot);
        }
        cluster_sync();
        if (c == 0 && warp == 0) {
            // the leader picks the rank whose share holds t = floor(u W) and
            // tells every rank (lane k writes rank k's copy)
            int redo = 0, sel = 0;
            unsigned long long sel_t = 0;
            if (lane == 0) {
                unsigned long long total = 0;
                for (int k = 0; k < C; ++k) total += sh.totals[k];
                if (total == 0ull && pass == 0) {
                    redo = 1;
                } else {
                    const unsigned long long tt = scale_uniform(sh.us, total);
                    unsigned long long before = 0;
                    sel = -1;
                    for (int k = 0; k < C && sel < 0; ++k) {
                        if (sh.totals[k] > 0 && tt < before + sh.totals[k])
                            sel = k;
                        else
                            before += sh.totals[k];
                    }
                    if (sel < 0) {  // cannot happen: tt < total; the last rank with weight
                        for (int k = C - 1; k >= 0 && sel < 0; --k)
                            if (sh.totals[k] > 0) sel = k;
                        if (sel < 0) sel = 0;
                        before = 0;
                        for (int k = 0; k < sel; ++k) before += sh.totals[k];
                    }
                    sel_t = tt - before;
                    if (a.dbg.w_total)
                        a.dbg.w_total[b] = kind == kKindResidual ? static_cast<double>(total) * kFixResidualInv
                                                                 : static_cast<double>(total) * kFixTargetInv *
                                                                       static_cast<double>(d.isp);
                }
            }
            redo = __shfl_sync(0xffffffffu, redo, 0);
            sel = __shfl_sync(0xffffffffu, sel, 0);
            sel_t = __shfl_sync(0xffffffffu, sel_t, 0);
            if (lane < C) {
                st_cluster_u32(cluster_map(&sh.redo, lane), static_cast<uint32_t>(redo));
                st_cluster_u32(cluster_map(&sh.sel, lane), static_cast<uint32_t>(sel));
                st_cluster_u64(cluster_map(&sh.sel_t, lane), sel_t);
            }
        }
        cluster_sync();
        if (sh.redo) continue;
        // the rank whose share holds t finds the run, then the token
        if (sh.sel == c && warp == 0) {
            const unsigned long long tt = sh.sel_t;
            unsigned long long before = 0;
            int token = -1;
            for (int i0 = 0; i0 < nruns && token < 0; i0 += 32) {
                const int i = i0 + lane;
                const unsigned long long q = i < nruns ? runs[i] : 0ull;
                unsigned long long incl = q;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                const unsigned long long start = before + incl - q;
                const unsigned hit = __ballot_sync(0xffffffffu, q > 0 && start <= tt && tt < start + q);
                if (hit) {
                    const int src = __ffs(hit) - 1;
                    int found = -1;
                    if (lane == src) found = K.run_token(i, kind, d, trow, drow, start, tt);
                    token = __shfl_sync(0xffffffffu, found, src);
                }
                before += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (lane == 0) {
                a.out_tokens[static_cast<size_t>(b) * (GM + 1) + sh.job.slot] = token >= 0 ? token : lo + len - 1;
                a.out_num_accepted[b] = sh.job.slot;  // the request is final
            }
        }
        break;
    }
}

// Dynamic shared memory of a CTA for this shape: CShared, the records each
// rank pushes to the leader (C ranks x (2 gamma + 1) rows), the piece records
// ((2 gamma + 1) rows x the most pieces a slice is cut into), then the run sums
// of the longest slice. Returns the offsets of the last three.
struct CLayout {
    int rows_off, pieces_off, runs_off;
    size_t total;
};

CLayout cluster_layout(int V, int gamma, int es, int C) {
    const int vec = 16 / es;
    const int slice = (V + C - 1) / C + vec;
    const int P = std::max(1, std::min(kMaxPieces, slice / 256));  // the kernel's P never exceeds it
    auto up16 = [](size_t x) { return (x + 15) & ~static_cast<size_t>(15); };
    CLayout L;
    size_t off = up16(sizeof(CShared));
    L.rows_off = static_cast<int>(off);
    off = up16(off + sizeof(CRec) * static_cast<size_t>(C) * (2 * gamma + 1));
    L.pieces_off = static_cast<int>(off);
    off = up16(off + sizeof(CRec) * static_cast<size_t>(2 * gamma + 1) * P);
    L.runs_off = static_cast<int>(off);
    L.total = off + sizeof(unsigned long long) * ((slice + kRun - 1) / kRun);
    return L;
}

}  // namespace

// Cluster size for a row of V elements: about 4 KB of each row per CTA,
// rounded up to a power of two, at most 16 CTAs.
int cluster_size(int V, int dtype) {
    const long long row_bytes = static_cast<long long>(V) * (dtype == SV_F32 ? 4 : 2);
    const long long want = std::max<long long>(1, std::min<long long>(kMaxCluster, (row_bytes + 4095) / 4096));
    int C = 1;
    while (C < want) C *= 2;
    return C;
}

bool cluster_applicable(const Args& a) {
    const size_t es = a.dtype == SV_F32 ? 4 : 2;
    if (a.tree || a.early) return false;
    if ((static_cast<size_t>(a.V) * es) % 16 != 0) return false;
    if ((reinterpret_cast<uintptr_t>(a.target) & 15) || (reinterpret_cast<uintptr_t>(a.draft) & 15)) return false;
    const int C = cluster_size(a.V, a.dtype);
    if ((a.V + C - 1) / C > kMaxSlice) return false;
    return static_cast<long long>(a.B) * C <= 0x7fffffffLL;
}

namespace {

template <int DT, int CS>
cudaError_t launch_one(const Args& a, const CLayout& L, cudaStream_t stream) {
    cluster_kernel<DT, CS><<<static_cast<unsigned>(a.B) * CS, kThreads, L.total, stream>>>(a, L.rows_off, L.pieces_off,
                                                                                             L.runs_off);
    return cudaGetLastError();
}

template <int DT>
cudaError_t launch_dt(const Args& a, int C, const CLayout& L, cudaStream_t stream) {
    switch (C) {
        case 1: return launch_one<DT, 1>(a, L, stream);
        case 2: return launch_one<DT, 2>(a, L, stream);
        case 4: return launch_one<DT, 4>(a, L, stream);
        case 8: return launch_one<DT, 8>(a, L, stream);
        default: return launch_one<DT, 16>(a, L, stream);
    }
}

template <int DT>
cudaError_t set_attributes(int smem_max) {
    const void* fns[] = {reinterpret_cast<const void*>(&cluster_kernel<DT, 1>),
                         reinterpret_cast<const void*>(&cluster_kernel<DT, 2>),
                         reinterpret_cast<const void*>(&cluster_kernel<DT, 4>),
                         reinterpret_cast<const void*>(&cluster_kernel<DT, 8>),
                         reinterpret_cast<const void*>(&cluster_kernel<DT, 16>)};
    for (const void* f : fns) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_cluster(const Args& a, const DeviceInfo& dev, cudaStream_t stream) {
    const int C = cluster_size(a.V, a.dtype);
    const CLayout L = cluster_layout(a.V, a.gamma, a.dtype == SV_F32 ? 4 : 2, C);
    static thread_local int attr_device = -1;
    if (attr_device != dev.device) {
        // the attribute is set once, for the largest shape the path takes
        const int smem_max = static_cast<int>(cluster_layout(kMaxSlice * kMaxCluster, SV_MAX_GAMMA, 2, kMaxCluster).total);
        cudaError_t e = set_attributes<SV_F32>(smem_max);
        if (e == cudaSuccess) e = set_attributes<SV_BF16>(smem_max);
        if (e != cudaSuccess) return e;
        attr_device = dev.device;
    }
    return a.dtype == SV_F32 ? launch_dt<SV_F32>(a, C, L, stream) : launch_dt<SV_BF16>(a, C, L, stream);
}

}  // namespace sv
