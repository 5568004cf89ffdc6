// Streaming path of libspecverify: one persistent, co-resident grid per call.
//
// The method ("Speculative Decoding : accélérer l'inférence des LLM",
// §Pourquoi la qualité est préservée; wiki "Speculative Decoding", eq. alpha(x)
// and eq. p_corr; "Accélérer Sonar grâce à la spéculation", §Décodage
// spéculatif) needs, per request, the normaliser (or argmax) of gamma+1
// target rows and gamma draft rows, a left-to-right scan, and one draw over a
// row that is known only after the scan. The kernel runs that as three phases
// separated by grid barriers:
//
//  1. Row statistics. The target rows of all requests, then the draft rows of
//     the T > 0 requests (compacted), form one virtual stream of logits that
//     is cut into G equal 16-byte-aligned slices, one per thread block. A
//     producer warp copies its slice through a ring of kStages shared-memory
//     stages with cp.async.bulk (completion on mbarriers); eight consumer warps
//     fold each stage into per-thread (max, sum of 2^((l-m)c)) or argmax
//     states. When the stream moves to a new row each warp writes its partial
//     result for the row piece; there is no block-wide barrier in the stream.
//  2. Acceptance scan. One warp per request merges the pieces of its rows in
//     a fixed order, evaluates p(x_i) and q(x_i) in double, finds the first
//     rejection, writes the accepted tokens and a draw job.
//  3. Draw. The rows the draws need (target row n and draft row n for a
//     residual, target row gamma for the extra token) are streamed again in
//     chunks of one stage; each thread sums the weights of a run of
//     consecutive tokens, and the runs are added into per-chunk totals as
//     64-bit fixed-point integers (exact and order-independent). After a grid
//     barrier one warp per job picks the chunk holding u * W, re-reads that one
//     chunk and finds the token.
//
// Every wait is bounded (about two seconds, by the global timer): a barrier or
// a stage that never completes sets SV_STATUS_TIMEOUT and the kernel returns.
#include <algorithm>
#include <cmath>

#include "sv_common.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kStages = 8;
constexpr int kStageBytes = 16384;
constexpr int kVecPerThread = kStageBytes / 16 / kConsumers;  // 4
constexpr int kMapMax = 256;
constexpr int kMaxB = 4096;
constexpr int kMaxRowsPerReq = 2 * SV_MAX_GAMMA + 1;
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;

// Named barriers (0 is __syncthreads).
constexpr int kBarConsumers = 1;  // the 256 consumer threads
constexpr int kBarHandoff = 2;    // consumers arrive, producer waits (288)

struct Rec {
    float m;      // max value (both modes)
    float s;      // sum 2^((l - m) c) (max/sum mode)
    int32_t idx;  // argmax (argmax mode)
    int32_t bad;  // NaN or +inf seen
};

struct Job {
    int32_t b, n, kind, pad;
    DrawParams d;
};

// Byte offsets into the caller's workspace and the partition constants.
struct Layout {
    long long Et;  // target elements B*(gamma+1)*V
    int G, MT, MD, NCH, vec, chunk_elems;
    size_t hdr, prefix, req, rec_t, rec_d, jobs, chunks, total;
};

__host__ __device__ inline long long part_begin(long long E, int G, int g, int vec) {
    if (g <= 0) return 0;
    if (g >= G) return E;
    long long x = (E * g) / G;
    return x - x % vec;
}

__device__ inline int part_owner(long long E, int G, int vec, long long e) {
    int g = static_cast<int>(min(static_cast<long long>(G - 1), (e * G) / E));
    while (g + 1 < G && part_begin(E, G, g + 1, vec) <= e) ++g;
    while (g > 0 && part_begin(E, G, g, vec) > e) --g;
    return g;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

Layout make_layout(int B, int gamma, int V, int es, int G) {
    Layout L;
    L.G = G;
    L.vec = 16 / es;
    L.Et = static_cast<long long>(B) * (gamma + 1) * V;
    const long long Ed_max = static_cast<long long>(B) * gamma * V;
    L.MT = static_cast<int>(((L.Et + G - 1) / G + L.vec - 1) / V + 2);
    L.MD = static_cast<int>(((Ed_max + G - 1) / G + L.vec - 1) / V + 2);
    L.chunk_elems = kStageBytes / es;
    L.NCH = (V + L.chunk_elems - 1) / L.chunk_elems;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = align256(off + bytes);
        return at;
    };
    L.hdr = take(256);
    L.prefix = take(static_cast<size_t>(B) * 4);
    L.req = take(static_cast<size_t>(B) * 4);
    L.rec_t = take(static_cast<size_t>(G) * L.MT * kConsumerWarps * sizeof(Rec));
    L.rec_d = take(static_cast<size_t>(G) * L.MD * kConsumerWarps * sizeof(Rec));
    L.jobs = take(static_cast<size_t>(B) * sizeof(Job));
    L.chunks = take(static_cast<size_t>(B) * L.NCH * 8);
    L.total = off;
    return L;
}

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase of `bar` with the given parity to complete; false after
// the time limit.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (unsigned it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 0 && global_ns() - t0 > kWaitTimeoutNs) return false;
    }
}

__device__ __forceinline__ void bulk_copy(void* dst_smem, const void* src, unsigned bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive(int id, int count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ float f32_max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// Packed pairs of binary32 (sm_100 family f32x2 arithmetic).
__device__ __forceinline__ unsigned long long f2(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2_sub(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// ---------------------------------------------------------------- barriers

struct Hdr {
    unsigned count;
    unsigned gen;
    int status;
};

// Grid-wide barrier of the co-resident grid; false (and SV_STATUS_TIMEOUT)
// when the other blocks do not arrive within the time limit.
__device__ bool grid_sync(Hdr* h, int32_t* d_status, int* s_flag) {
    __syncthreads();
    if (threadIdx.x == 0) {
        volatile unsigned* vgen = &h->gen;
        const unsigned my_gen = *vgen;
        __threadfence();
        const unsigned prev = atomicAdd(&h->count, 1u);
        int ok = 1;
        if (prev == gridDim.x - 1) {
            atomicExch(&h->count, 0u);
            __threadfence();
            atomicAdd(&h->gen, 1u);
        } else {
            const unsigned long long t0 = global_ns();
            while (*vgen == my_gen) {
                if (global_ns() - t0 > kWaitTimeoutNs) {
                    ok = 0;
                    atomicOr(&h->status, SV_STATUS_TIMEOUT);
                    if (d_status) atomicOr(d_status, SV_STATUS_TIMEOUT);
                    break;
                }
                __nanosleep(100);
            }
        }
        __threadfence();
        *s_flag = ok;
    }
    __syncthreads();
    return *s_flag != 0;
}

// ------------------------------------------------------------ kernel context

struct Ctl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    int n_samp;
    int k_lo;   // first compacted request of this block's draft slice
    int abort;
    int flag;
    int map[kMapMax];
    int wtmp[kConsumerWarps + 1];
};

struct RowLoc {
    int kind;        // 0 target row, 1 draft row
    long long row;   // target row index, or compacted draft row index
    int req;         // request b
    int slot;        // row slot of this block
};

// One stage of the phase-1 stream.
struct Stage1 {
    const char* src;
    unsigned bytes;
    int elems;
    long long e0;  // first element, offset within the row
    RowLoc loc;
};

template <int DT>
struct Kern {
    static constexpr int ES = DT == SV_F32 ? 4 : 2;
    static constexpr int kChunkElems = kStageBytes / ES;
    static constexpr int kTPT = kChunkElems / kConsumers;  // tokens per thread run

    const Args& a;
    const Layout& L;
    char* ws;
    Ctl& ctl;
    char* stages;
    int G, g;

    __device__ Hdr* hdr() const { return reinterpret_cast<Hdr*>(ws + L.hdr); }
    __device__ int* prefix() const { return reinterpret_cast<int*>(ws + L.prefix); }
    __device__ int* req() const { return reinterpret_cast<int*>(ws + L.req); }
    __device__ Rec* rec_t() const { return reinterpret_cast<Rec*>(ws + L.rec_t); }
    __device__ Rec* rec_d() const { return reinterpret_cast<Rec*>(ws + L.rec_d); }
    __device__ Job* jobs() const { return reinterpret_cast<Job*>(ws + L.jobs); }
    __device__ unsigned long long* chunks() const {
        return reinterpret_cast<unsigned long long*>(ws + L.chunks);
    }

    __device__ static bool sampled(float T) { return T > 0.0f && T < pos_inf(); }

    __device__ long long Ed() const {
        return static_cast<long long>(ctl.n_samp) * a.gamma * a.V;
    }

    // ---- phase-1 stage schedule, shared by the producer and the consumers:
    // this block's slice of the target rows, then of the compacted draft rows
    // (the latter needs the prologue's n_samp and map).
    template <typename F>
    __device__ void for_each_target_stage(F&& f) const {
        const int V = a.V, GM = a.gamma;
        const long long ts = part_begin(L.Et, G, g, L.vec), te = part_begin(L.Et, G, g + 1, L.vec);
        const long long first_t = ts / V;
        for (long long e = ts; e < te;) {
            const long long r = e / V;
            const long long seg_end = min(te, (r + 1) * V);
            while (e < seg_end) {
                const int n = static_cast<int>(min(seg_end - e, static_cast<long long>(kChunkElems)));
                Stage1 st;
                st.src = static_cast<const char*>(a.target) + e * ES;
                st.bytes = static_cast<unsigned>(n * ES);
                st.elems = n;
                st.e0 = e - r * V;
                st.loc = {0, r, static_cast<int>(r / (GM + 1)), static_cast<int>(r - first_t)};
                f(st);
                e += n;
            }
        }
    }

    template <typename F>
    __device__ void for_each_draft_stage(F&& f) const {
        const int V = a.V, GM = a.gamma;
        const long long E2 = Ed();
        if (E2 == 0) return;
        const long long ds = part_begin(E2, G, g, L.vec), de = part_begin(E2, G, g + 1, L.vec);
        const long long first_d = ds / V;
        for (long long e = ds; e < de;) {
            const long long kr = e / V;
            const long long seg_end = min(de, (kr + 1) * V);
            const int k = static_cast<int>(kr / GM), i = static_cast<int>(kr % GM);
            const int rel = k - ctl.k_lo;
            const int b = (rel >= 0 && rel < kMapMax) ? ctl.map[rel] : -1;
            if (b < 0 || b >= a.B) {  // cannot happen when the host checks hold
                ctl.abort = 1;
                return;
            }
            const long long base = (static_cast<long long>(b) * GM + i) * V;
            while (e < seg_end) {
                const int n = static_cast<int>(min(seg_end - e, static_cast<long long>(kChunkElems)));
                Stage1 st;
                st.src = static_cast<const char*>(a.draft) + (base + (e - kr * V)) * ES;
                st.bytes = static_cast<unsigned>(n * ES);
                st.elems = n;
                st.e0 = e - kr * V;
                st.loc = {1, kr, b, static_cast<int>(kr - first_d)};
                f(st);
                e += n;
            }
        }
    }

    // ---- producer: lane 0 issues the copies of a schedule into the ring
    struct Producer {
        unsigned it = 0;
    };

    __device__ bool produce(Producer& p, const char* src, unsigned bytes) const {
        const int slot = p.it % kStages;
        const unsigned round = p.it / kStages;
        if (round > 0 && !mbar_wait(&ctl.empty[slot], (round - 1) & 1)) return false;
        if ((threadIdx.x & 31) == 0) {
            mbar_expect_tx(&ctl.full[slot], bytes);
            bulk_copy(stages + static_cast<size_t>(slot) * kStageBytes, src, bytes, &ctl.full[slot]);
        }
        __syncwarp();
        ++p.it;
        return true;
    }

    // Waits (bounded) until every copy the producer issued has landed.
    __device__ void drain(const Producer& p) const {
        const unsigned n = p.it;
        for (unsigned j = (n > kStages ? n - kStages : 0); j < n; ++j)
            mbar_wait(&ctl.full[j % kStages], (j / kStages) & 1);
    }

    struct Consumer {
        unsigned it = 0;
    };

    __device__ const char* consume_begin(Consumer& c) const {
        const int slot = c.it % kStages;
        if (!mbar_wait(&ctl.full[slot], (c.it / kStages) & 1)) return nullptr;
        return stages + static_cast<size_t>(slot) * kStageBytes;
    }
    __device__ void consume_end(Consumer& c) const {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(&ctl.empty[c.it % kStages]);
        ++c.it;
    }

    __device__ void set_abort(int32_t* d_status) const {
        ctl.abort = 1;
        atomicOr(&hdr()->status, SV_STATUS_TIMEOUT);
        if (d_status) atomicOr(d_status, SV_STATUS_TIMEOUT);
    }

    // ---- phase-1 prologue (consumers): count the T > 0 requests, map this
    // block's draft slice to requests; block 0 publishes the compaction.
    __device__ void prologue() const {
        const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
        int cnt = 0;
        for (int b = t; b < a.B; b += kConsumers) cnt += sampled(a.temperature[b]) ? 1 : 0;
        cnt = __reduce_add_sync(0xffffffffu, cnt);
        if (lane == 0) ctl.wtmp[warp] = cnt;
        bar_sync(kBarConsumers, kConsumers);
        if (t == 0) {
            int n = 0;
            for (int w = 0; w < kConsumerWarps; ++w) n += ctl.wtmp[w];
            ctl.n_samp = n;
            const long long E2 = static_cast<long long>(n) * a.gamma * a.V;
            const long long ds = part_begin(E2, G, g, L.vec);
            ctl.k_lo = n > 0 ? static_cast<int>(ds / (static_cast<long long>(a.gamma) * a.V)) : 0;
        }
        bar_sync(kBarConsumers, kConsumers);
        const int k_lo = ctl.k_lo;
        int carry = 0;
        for (int base = 0; base < a.B; base += kConsumers) {
            const int b = base + t;
            const int f = (b < a.B && sampled(a.temperature[b])) ? 1 : 0;
            const unsigned ball = __ballot_sync(0xffffffffu, f);
            const int in_warp = __popc(ball & ((1u << lane) - 1u));
            if (lane == 0) ctl.wtmp[warp] = __popc(ball);
            bar_sync(kBarConsumers, kConsumers);
            int before = carry;
            for (int w = 0; w < warp; ++w) before += ctl.wtmp[w];
            int total = 0;
            for (int w = 0; w < kConsumerWarps; ++w) total += ctl.wtmp[w];
            const int k = before + in_warp;
            if (b < a.B) {
                if (f) {
                    const int rel = k - k_lo;
                    if (rel >= 0 && rel < kMapMax) ctl.map[rel] = b;
                    if (g == 0) req()[k] = b;
                }
                if (g == 0) prefix()[b] = f ? k : -1;
            }
            carry += total;
            bar_sync(kBarConsumers, kConsumers);
        }
    }

    // ---- phase-1 consumer: fold stages into per-thread row states
    struct RowState {
        float m, s;    // max/sum mode
        int idx;       // argmax mode
        int bad;
        bool argmax;   // mode of the current row
        float c;
        long long key; // kind * 2^62 + row, -1 = none
        RowLoc loc;
    };

    __device__ void flush_row(RowState& rs) const {
        if (rs.key < 0) return;
        int bad = __any_sync(0xffffffffu, rs.bad);
        Rec rec;
        if (rs.argmax) {
            ArgMax st{rs.m, rs.idx};
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                ArgMax ot{__shfl_xor_sync(0xffffffffu, st.v, o), __shfl_xor_sync(0xffffffffu, st.i, o)};
                st = argmax_merge(st, ot);
            }
            rec = {st.v, 0.0f, st.i, bad};
        } else {
            MaxSum st{rs.m, rs.s};
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                MaxSum ot{__shfl_xor_sync(0xffffffffu, st.m, o), __shfl_xor_sync(0xffffffffu, st.s, o)};
                st = maxsum_merge(st, ot, rs.c);
            }
            rec = {st.m, st.s, -1, bad};
        }
        if ((threadIdx.x & 31) == 0) {
            const int warp = threadIdx.x >> 5;
            Rec* dst = rs.loc.kind == 0 ? rec_t() + ((static_cast<size_t>(g) * L.MT + rs.loc.slot) * kConsumerWarps + warp)
                                        : rec_d() + ((static_cast<size_t>(g) * L.MD + rs.loc.slot) * kConsumerWarps + warp);
            *dst = rec;
        }
    }

    __device__ void start_row(RowState& rs, const RowLoc& loc) const {
        rs.loc = loc;
        rs.key = (static_cast<long long>(loc.kind) << 62) + loc.row;
        const float T = a.temperature[loc.req];
        rs.argmax = loc.kind == 0 && !sampled(T);
        rs.c = rs.argmax ? 0.0f : temp_scale(T);
        rs.m = neg_inf();
        rs.s = 0.0f;
        rs.idx = 0x7fffffff;
        rs.bad = 0;
    }

    __device__ void fold_stage(RowState& rs, const char* sm, const Stage1& st) const {
        const int t = threadIdx.x;
        const int nvec = static_cast<int>(st.bytes / 16);
        uint4 v[kVecPerThread];
#pragma unroll
        for (int k = 0; k < kVecPerThread; ++k) {
            const int vi = t + k * kConsumers;
            if (vi < nvec) {
                v[k] = *reinterpret_cast<const uint4*>(sm + static_cast<size_t>(vi) * 16);
            } else if (DT == SV_BF16) {
                v[k] = make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
            } else {
                v[k] = make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
            }
        }
        // tile max, NaN-propagating
        float tmax;
        if (DT == SV_BF16) {
            uint32_t m2 = bf16x2_max_nan(bf16x2_max_nan(v[0].x, v[0].y), bf16x2_max_nan(v[0].z, v[0].w));
#pragma unroll
            for (int k = 1; k < kVecPerThread; ++k)
                m2 = bf16x2_max_nan(m2, bf16x2_max_nan(bf16x2_max_nan(v[k].x, v[k].y),
                                                       bf16x2_max_nan(v[k].z, v[k].w)));
            tmax = f32_max_nan(bf16x2_lo(m2), bf16x2_hi(m2));
        } else {
            tmax = neg_inf();
#pragma unroll
            for (int k = 0; k < kVecPerThread; ++k)
                tmax = f32_max_nan(tmax, f32_max_nan(f32_max_nan(__uint_as_float(v[k].x), __uint_as_float(v[k].y)),
                                                     f32_max_nan(__uint_as_float(v[k].z), __uint_as_float(v[k].w))));
        }
        if (bad_logit(tmax)) {
            rs.bad = 1;
            return;
        }
        if (tmax == neg_inf()) return;
        if (rs.argmax) {
            if (tmax > rs.m) {
                // first position of tmax among this thread's elements (increasing index)
                int found = -1;
#pragma unroll
                for (int k = 0; k < kVecPerThread; ++k) {
                    const uint32_t w4[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (DT == SV_BF16) {
                            if (found < 0 && bf16x2_lo(w4[q]) == tmax) found = (t + k * kConsumers) * 8 + 2 * q;
                            if (found < 0 && bf16x2_hi(w4[q]) == tmax) found = (t + k * kConsumers) * 8 + 2 * q + 1;
                        } else {
                            if (found < 0 && __uint_as_float(w4[q]) == tmax) found = (t + k * kConsumers) * 4 + q;
                        }
                    }
                }
                rs.m = tmax;
                rs.idx = static_cast<int>(st.e0) + found;
            }
            return;
        }
        const float c = rs.c;
        if (tmax > rs.m) {
            rs.s = (rs.m == neg_inf()) ? 0.0f : __fmul_rn(rs.s, ex2(__fmul_rn(__fsub_rn(rs.m, tmax), c)));
            rs.m = tmax;
        }
        const unsigned long long mm = f2(rs.m, rs.m), cc = f2(c, c);
        unsigned long long acc = f2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < kVecPerThread; ++k) {
            const uint32_t w4[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
            if (DT == SV_BF16) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const unsigned long long d = f2_mul(f2_sub(f2(bf16x2_lo(w4[q]), bf16x2_hi(w4[q])), mm), cc);
                    float d0, d1;
                    f2_unpack(d, d0, d1);
                    acc = f2_add(acc, f2(ex2(d0), ex2(d1)));
                }
            } else {
#pragma unroll
                for (int q = 0; q < 4; q += 2) {
                    const unsigned long long d =
                        f2_mul(f2_sub(f2(__uint_as_float(w4[q]), __uint_as_float(w4[q + 1])), mm), cc);
                    float d0, d1;
                    f2_unpack(d, d0, d1);
                    acc = f2_add(acc, f2(ex2(d0), ex2(d1)));
                }
            }
        }
        float a0, a1;
        f2_unpack(acc, a0, a1);
        rs.s = __fadd_rn(rs.s, __fadd_rn(a0, a1));
    }

    // ---- phase 2: merge of a row's pieces
    __device__ Rec merge_row(int kind, long long row, bool argmax, float c) const {
        const long long E = kind == 0 ? L.Et : Ed();
        const int MM = kind == 0 ? L.MT : L.MD;
        const Rec* base = kind == 0 ? rec_t() : rec_d();
        const long long e0 = row * a.V, e1 = e0 + a.V - 1;
        const int g0 = part_owner(E, G, L.vec, e0), g1 = part_owner(E, G, L.vec, e1);
        MaxSum ms = maxsum_empty();
        ArgMax am = argmax_empty();
        int bad = 0;
        for (int gg = g0; gg <= g1; ++gg) {
            const long long b0 = part_begin(E, G, gg, L.vec), b1 = part_begin(E, G, gg + 1, L.vec);
            if (b1 <= b0) continue;
            const int slot = static_cast<int>(row - b0 / a.V);
            const Rec* r = base + (static_cast<size_t>(gg) * MM + slot) * kConsumerWarps;
            for (int w = 0; w < kConsumerWarps; ++w) {
                const Rec x = r[w];
                bad |= x.bad;
                if (argmax)
                    am = argmax_merge(am, ArgMax{x.m, x.idx});
                else
                    ms = maxsum_merge(ms, MaxSum{x.m, x.s}, c);
            }
        }
        Rec out;
        if (argmax)
            out = {am.v, 0.0f, am.i == 0x7fffffff ? 0 : am.i, (bad || am.v == neg_inf()) ? 1 : 0};
        else
            out = {ms.m, ms.s, -1, (bad || ms.m == neg_inf()) ? 1 : 0};
        return out;
    }

    // Phase 2 for request b on one warp; `st` is this warp's shared scratch.
    __device__ void verify_request(int b, Rec* st) const {
        const int lane = threadIdx.x & 31, GM = a.gamma, V = a.V;
        const float T = a.temperature[b];
        const bool t_ok = (T >= 0.0f) && (T < pos_inf());
        const bool greedy = t_ok && T == 0.0f;
        const bool samp = sampled(T);
        const float c = samp ? temp_scale(T) : 0.0f;
        const int k = prefix()[b];
        const int32_t* tok = a.tokens + static_cast<size_t>(b) * GM;
        int bad = t_ok ? 0 : 1;
        for (int i = lane; i < GM; i += 32) {
            const int x = tok[i];
            if (x < 0 || x >= V) bad = 1;
        }
        const int nrows = samp ? 2 * GM + 1 : GM + 1;
        for (int r = lane; r < nrows; r += 32) {
            Rec x;
            if (r <= GM)
                x = merge_row(0, static_cast<long long>(b) * (GM + 1) + r, !samp, c);
            else
                x = merge_row(1, static_cast<long long>(k) * GM + (r - GM - 1), false, c);
            st[r] = x;
            bad |= x.bad;
        }
        bad = __any_sync(0xffffffffu, bad);
        __syncwarp();
        int32_t* out = a.out_tokens + static_cast<size_t>(b) * (GM + 1);
        const sv_debug_out& dbg = a.dbg;
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
                if (k >= 0) jobs()[k].kind = kKindInvalid;
            }
            return;
        }
        for (int j = lane; j <= GM; j += 32) {
            const size_t r = static_cast<size_t>(b) * (GM + 1) + j;
            if (dbg.max_target) dbg.max_target[r] = st[j].m;
            if (dbg.lse_target) dbg.lse_target[r] = greedy ? nan("") : lse_from_stats(st[j].m, st[j].s, T);
            if (dbg.argmax_target) dbg.argmax_target[r] = greedy ? st[j].idx : -1;
        }
        for (int j = lane; j < GM; j += 32) {
            const size_t r = static_cast<size_t>(b) * GM + j;
            if (dbg.max_draft) dbg.max_draft[r] = greedy ? nanf("") : st[GM + 1 + j].m;
            if (dbg.lse_draft) dbg.lse_draft[r] = greedy ? nan("") : lse_from_stats(st[GM + 1 + j].m, st[GM + 1 + j].s, T);
        }
        // first failing position over all lanes (gamma may exceed 32)
        int n = GM;
        for (int base = 0; base < GM; base += 32) {
            const int i = base + lane;
            bool fail = false;
            if (i < GM) {
                const int x = tok[i];
                if (greedy) {
                    fail = x != st[i].idx;
                } else {
                    const size_t tr = static_cast<size_t>(b) * (GM + 1) + i;
                    const size_t dr = static_cast<size_t>(b) * GM + i;
                    const double p = prob_from_stats(load_logit<DT>(a.target, tr * V + x), st[i].m, st[i].s, c);
                    const double q = prob_from_stats(load_logit<DT>(a.draft, dr * V + x), st[GM + 1 + i].m,
                                                     st[GM + 1 + i].s, c);
                    if (dbg.p_x) dbg.p_x[dr] = p;
                    if (dbg.q_x) dbg.q_x[dr] = q;
                    fail = !accept_draft(p, q, a.u_accept[dr]);
                }
            }
            const unsigned ball = __ballot_sync(0xffffffffu, fail);
            if (n == GM && ball) n = base + __ffs(ball) - 1;
        }
        // positions after the first rejection (all of them at T = 0) are not evaluated
        for (int i = lane; i < GM; i += 32)
            if (greedy || i > n) {
                const size_t dr = static_cast<size_t>(b) * GM + i;
                if (dbg.p_x) dbg.p_x[dr] = nan("");
                if (dbg.q_x) dbg.q_x[dr] = nan("");
            }
        for (int j = lane; j <= GM; j += 32) {
            if (j < n)
                out[j] = tok[j];
            else if (j == n)
                out[j] = greedy ? st[n].idx : -1;  // the draw fills it in phase 3
            else
                out[j] = -1;
        }
        if (lane == 0) {
            a.out_num_accepted[b] = n;
            if (greedy) {
                if (dbg.kind) dbg.kind[b] = kKindGreedy;
                if (dbg.w_total) dbg.w_total[b] = nan("");
            } else {
                Job j;
                j.b = b;
                j.n = n;
                j.pad = 0;
                DrawParams& d = j.d;
                d.c = c;
                d.mp = st[n].m;
                d.isp = __double2float_rn(1.0 / static_cast<double>(st[n].s));
                if (n < GM) {
                    d.kind = kKindResidual;
                    d.mq = st[GM + 1 + n].m;
                    d.isq = __double2float_rn(1.0 / static_cast<double>(st[GM + 1 + n].s));
                    d.fix = kFixResidual;
                } else {
                    d.kind = kKindBonus;
                    d.mq = 0.0f;
                    d.isq = 0.0f;
                    d.fix = kFixTarget;
                }
                j.kind = d.kind;
                jobs()[k] = j;
                if (dbg.kind) dbg.kind[b] = d.kind;
            }
        }
        if (!greedy)
            for (int j = lane; j < L.NCH; j += 32) chunks()[static_cast<size_t>(k) * L.NCH + j] = 0ull;
    }

    // ---- phase 3 schedule: draw items (job k, chunk j) of this block
    __device__ static int job_cost(int kind) { return kind == kKindResidual ? 2 : (kind == kKindBonus ? 1 : 0); }

    // Calls f(k, j) for every item whose first cost unit falls in this
    // block's share. `pre` holds the cost prefix over jobs (n_samp + 1).
    template <typename F>
    __device__ void for_each_item(const int* pre, F&& f) const {
        const int ns = ctl.n_samp;
        const long long U = static_cast<long long>(pre[ns]) * L.NCH;
        if (U == 0) return;
        const long long u_lo = part_begin(U, G, g, 1), u_hi = part_begin(U, G, g + 1, 1);
        if (u_hi <= u_lo) return;
        // first job whose units end after u_lo
        int lo = 0, hi = ns - 1;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (static_cast<long long>(pre[mid + 1]) * L.NCH > u_lo)
                hi = mid;
            else
                lo = mid + 1;
        }
        for (int k = lo; k < ns; ++k) {
            const int cost = pre[k + 1] - pre[k];
            if (cost == 0) continue;
            const long long base = static_cast<long long>(pre[k]) * L.NCH;
            if (base >= u_hi) break;
            int j0 = 0;
            if (base < u_lo) j0 = static_cast<int>((u_lo - base + cost - 1) / cost);
            for (int j = j0; j < L.NCH; ++j) {
                const long long u0 = base + static_cast<long long>(j) * cost;
                if (u0 >= u_hi) return;
                f(k, j);
            }
        }
    }

    // Weight sum of one thread run: tokens [j*CH + t*TPT, ... + TPT) of the
    // chunk, in index order. `tv`/`dv` hold the run's logits.
    __device__ static float run_sum(const float* lt, const float* ld, int valid, const DrawParams& d,
                                    int kind) {
        float run = 0.0f;
#pragma unroll
        for (int e = 0; e < kTPT; ++e) {
            if (e < valid) {
                const float w = kind == kKindResidual ? weight_residual(lt[e], ld[e], d) : weight_target(lt[e], d);
                run = __fadd_rn(run, w);
            }
        }
        return run;
    }

    // Loads a thread run from shared memory (64 bytes, swizzled order to
    // avoid bank conflicts) into binary32 values.
    __device__ static void load_run_smem(const char* sm, int t, float* out) {
        uint4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int q = (k + (t >> 1)) & 3;
            v[q] = *reinterpret_cast<const uint4*>(sm + static_cast<size_t>(t) * 64 + q * 16);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t w4[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (DT == SV_BF16) {
                    out[q * 8 + 2 * i] = bf16x2_lo(w4[i]);
                    out[q * 8 + 2 * i + 1] = bf16x2_hi(w4[i]);
                } else {
                    out[q * 4 + i] = __uint_as_float(w4[i]);
                }
            }
        }
    }

    __device__ static void load_run_global(const void* base, long long row_elem0, int count, float* out) {
#pragma unroll
        for (int e = 0; e < kTPT; ++e) out[e] = e < count ? load_logit<DT>(base, row_elem0 + e) : 0.0f;
    }
};

template <int DT>
__global__ void __launch_bounds__(kThreads, 1) stream_kernel(Args a, Layout L, char* ws) {
    extern __shared__ __align__(128) char smem[];
    char* stages = smem;
    Ctl& ctl = *reinterpret_cast<Ctl*>(smem + static_cast<size_t>(kStages) * kStageBytes);
    Rec* warp_rows = reinterpret_cast<Rec*>(smem + static_cast<size_t>(kStages) * kStageBytes + sizeof(Ctl));
    int* pre = reinterpret_cast<int*>(warp_rows + kConsumerWarps * kMaxRowsPerReq);

    Kern<DT> K{a, L, ws, ctl, stages, static_cast<int>(gridDim.x), static_cast<int>(blockIdx.x)};
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const bool producer = warp == kConsumerWarps;

    if (t == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl.full[s], 1);
            mbar_init(&ctl.empty[s], kConsumerWarps);
        }
        ctl.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int i = t; i < kMapMax; i += kThreads) ctl.map[i] = -1;
    __syncthreads();

    // -------------------------------------------------------------- phase 1
    typename Kern<DT>::Producer prod;
    typename Kern<DT>::Consumer cons;
    if (producer) {
        bool ok = true;
        auto issue = [&](const Stage1& st) {
            if (!ok || ctl.abort) return;
            ok = K.produce(prod, st.src, st.bytes);
        };
        K.for_each_target_stage(issue);
        bar_sync(kBarHandoff, kThreads);  // the consumers' prologue is done
        K.for_each_draft_stage(issue);
        if (!ok) K.set_abort(a.d_status);
        if (ctl.abort) K.drain(prod);
    } else {
        // target stages do not depend on the prologue, but the consumers
        // compute it first: the ring holds kStages stages meanwhile.
        K.prologue();
        bar_arrive(kBarHandoff, kThreads);
        typename Kern<DT>::RowState rs;
        rs.key = -1;
        bool ok = true;
        auto fold = [&](const Stage1& st) {
            if (!ok) return;
            const long long key = (static_cast<long long>(st.loc.kind) << 62) + st.loc.row;
            if (key != rs.key) {
                K.flush_row(rs);
                K.start_row(rs, st.loc);
            }
            const char* sm = K.consume_begin(cons);
            if (!sm) {
                ok = false;
                K.set_abort(a.d_status);
                return;
            }
            K.fold_stage(rs, sm, st);
            K.consume_end(cons);
        };
        K.for_each_target_stage(fold);
        K.for_each_draft_stage(fold);
        if (ok) K.flush_row(rs);
    }
    Hdr* hdr = K.hdr();
    if (!grid_sync(hdr, a.d_status, &ctl.flag)) return;
    if (ctl.abort) return;

    // -------------------------------------------------------------- phase 2
    if (!producer) {
        Rec* st = warp_rows + warp * kMaxRowsPerReq;
        for (int b = blockIdx.x * kConsumerWarps + warp; b < a.B; b += gridDim.x * kConsumerWarps) {
            K.verify_request(b, st);
            __syncwarp();
        }
    }
    if (ctl.n_samp == 0) return;
    if (!grid_sync(hdr, a.d_status, &ctl.flag)) return;

    // -------------------------------------------------------------- phase 3a
    const int ns = ctl.n_samp;
    if (!producer) {
        // cost prefix over jobs, on the consumers
        Job* jobs = K.jobs();
        int carry = 0;
        for (int base = 0; base < ns; base += kConsumers) {
            const int k = base + t;
            const int cost = k < ns ? Kern<DT>::job_cost(jobs[k].kind) : 0;
            int x = cost;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (lane == 31) ctl.wtmp[warp] = x;
            bar_sync(kBarConsumers, kConsumers);
            int before = carry;
            for (int w = 0; w < warp; ++w) before += ctl.wtmp[w];
            int total = 0;
            for (int w = 0; w < kConsumerWarps; ++w) total += ctl.wtmp[w];
            if (k < ns) pre[k] = before + x - cost;
            carry += total;
            bar_sync(kBarConsumers, kConsumers);
        }
        if (t == 0) pre[ns] = carry;
        bar_sync(kBarConsumers, kConsumers);
        bar_arrive(kBarHandoff, kThreads);
    }
    if (producer) {
        bar_sync(kBarHandoff, kThreads);
        bool ok = true;
        Job* jobs = K.jobs();
        K.for_each_item(pre, [&](int k, int j) {
            if (!ok || ctl.abort) return;
            const Job& jb = jobs[k];
            const long long e0 = static_cast<long long>(j) * Kern<DT>::kChunkElems;
            const int cnt = static_cast<int>(min(static_cast<long long>(Kern<DT>::kChunkElems), a.V - e0));
            const unsigned bytes = static_cast<unsigned>(cnt * Kern<DT>::ES);
            const long long trow = static_cast<long long>(jb.b) * (a.gamma + 1) + jb.n;
            ok = K.produce(prod, static_cast<const char*>(a.target) + (trow * a.V + e0) * Kern<DT>::ES, bytes);
            if (ok && jb.kind == kKindResidual) {
                const long long drow = static_cast<long long>(jb.b) * a.gamma + jb.n;
                ok = K.produce(prod, static_cast<const char*>(a.draft) + (drow * a.V + e0) * Kern<DT>::ES, bytes);
            }
        });
        if (!ok) K.set_abort(a.d_status);
        if (ctl.abort) K.drain(prod);
    } else {
        bool ok = true;
        Job* jobs = K.jobs();
        unsigned long long* csum = K.chunks();
        K.for_each_item(pre, [&](int k, int j) {
            if (!ok) return;
            const Job jb = jobs[k];
            const long long e0 = static_cast<long long>(j) * Kern<DT>::kChunkElems;
            const int cnt = static_cast<int>(min(static_cast<long long>(Kern<DT>::kChunkElems), a.V - e0));
            const int valid = max(0, min(Kern<DT>::kTPT, cnt - t * Kern<DT>::kTPT));
            float lt[Kern<DT>::kTPT], ld[Kern<DT>::kTPT];
            const char* smt = K.consume_begin(cons);
            if (!smt) {
                ok = false;
                K.set_abort(a.d_status);
                return;
            }
            if (valid > 0) Kern<DT>::load_run_smem(smt, t, lt);
            const bool resid = jb.kind == kKindResidual;
            if (resid) {
                K.consume_end(cons);  // release the target stage after loading
                const char* smd = K.consume_begin(cons);
                if (!smd) {
                    ok = false;
                    K.set_abort(a.d_status);
                    return;
                }
                if (valid > 0) Kern<DT>::load_run_smem(smd, t, ld);
            }
            K.consume_end(cons);
            const float run = valid > 0 ? Kern<DT>::run_sum(lt, ld, valid, jb.d, jb.kind) : 0.0f;
            const unsigned long long wsum = warp_sum_u64(to_fixed(run, jb.d.fix));
            if (lane == 0 && wsum) atomicAdd(csum + static_cast<size_t>(k) * L.NCH + j, wsum);
        });
    }
    if (!grid_sync(hdr, a.d_status, &ctl.flag)) return;
    if (ctl.abort || producer) return;

    // -------------------------------------------------------------- phase 3b
    Job* jobs = K.jobs();
    const unsigned long long* csum = K.chunks();
    constexpr int TPT = Kern<DT>::kTPT;
    constexpr int CH = Kern<DT>::kChunkElems;
    for (int k = blockIdx.x * kConsumerWarps + warp; k < ns; k += gridDim.x * kConsumerWarps) {
        const Job jb = jobs[k];
        if (jb.kind != kKindResidual && jb.kind != kKindBonus) continue;
        DrawParams d = jb.d;
        int kind = jb.kind;
        const long long trow = (static_cast<long long>(jb.b) * (a.gamma + 1) + jb.n) * a.V;
        const long long drow = (static_cast<long long>(jb.b) * a.gamma + jb.n) * a.V;
        // chunk totals of this job (recomputed on the warp for the fallback)
        unsigned long long total = 0;
        for (int j = lane; j < L.NCH; j += 32) total += csum[static_cast<size_t>(k) * L.NCH + j];
        total = warp_sum_u64(total);
        bool fallback = false;
        if (total == 0ull) {
            // residual weights rounded to zero everywhere: draw from p_n
            fallback = true;
            kind = kKindBonus;
            d.fix = kFixTarget;
        }
        auto chunk_total = [&](int j) -> unsigned long long {
            // sum over the chunk's 256 runs, on this warp
            unsigned long long acc = 0;
            const long long e0 = static_cast<long long>(j) * CH;
            const int cnt = static_cast<int>(min(static_cast<long long>(CH), a.V - e0));
            for (int vt = lane; vt < kConsumers; vt += 32) {
                const int valid = max(0, min(TPT, cnt - vt * TPT));
                if (valid <= 0) continue;
                float lt[TPT], ld[TPT];
                Kern<DT>::load_run_global(a.target, trow + e0 + vt * TPT, valid, lt);
                if (kind == kKindResidual) Kern<DT>::load_run_global(a.draft, drow + e0 + vt * TPT, valid, ld);
                acc += to_fixed(Kern<DT>::run_sum(lt, ld, valid, d, kind), d.fix);
            }
            return warp_sum_u64(acc);
        };
        if (fallback) {
            total = 0;
            for (int j = 0; j < L.NCH; ++j) total += chunk_total(j);
        }
        const unsigned long long tt =
            __double2ull_rz(static_cast<double>(a.u_sample[jb.b]) * static_cast<double>(total));
        // the chunk holding tt (prefix over chunks, exact integers)
        unsigned long long before = 0;
        int jsel = L.NCH - 1;
        for (int j = 0; j < L.NCH; ++j) {
            const unsigned long long cs = fallback ? chunk_total(j) : csum[static_cast<size_t>(k) * L.NCH + j];
            if (tt < before + cs) {
                jsel = j;
                break;
            }
            before += cs;
        }
        // runs of chunk jsel: values, exclusive prefix in run order
        const long long e0 = static_cast<long long>(jsel) * CH;
        const int cnt = static_cast<int>(min(static_cast<long long>(CH), a.V - e0));
        const unsigned long long tin = tt - before;
        unsigned long long carry = 0;
        int found_vt = -1;
        unsigned long long found_start = 0;
        for (int r0 = 0; r0 < kConsumers && found_vt < 0; r0 += 32) {
            const int vt = r0 + lane;
            const int valid = max(0, min(TPT, cnt - vt * TPT));
            unsigned long long q = 0;
            if (valid > 0) {
                float lt[TPT], ld[TPT];
                Kern<DT>::load_run_global(a.target, trow + e0 + vt * TPT, valid, lt);
                if (kind == kKindResidual) Kern<DT>::load_run_global(a.draft, drow + e0 + vt * TPT, valid, ld);
                q = to_fixed(Kern<DT>::run_sum(lt, ld, valid, d, kind), d.fix);
            }
            unsigned long long x = q;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            const unsigned long long start = carry + x - q;
            const bool mine = q > 0 && start <= tin && tin < start + q;
            const unsigned ball = __ballot_sync(0xffffffffu, mine);
            if (ball) {
                const int src = __ffs(ball) - 1;
                found_vt = r0 + src;
                found_start = __shfl_sync(0xffffffffu, start, src);
            }
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) {
            int token = a.V - 1;
            if (found_vt >= 0) {
                const int valid = max(0, min(TPT, cnt - found_vt * TPT));
                float lt[TPT], ld[TPT];
                Kern<DT>::load_run_global(a.target, trow + e0 + found_vt * TPT, valid, lt);
                if (kind == kKindResidual) Kern<DT>::load_run_global(a.draft, drow + e0 + found_vt * TPT, valid, ld);
                float run = 0.0f;
                int last_pos = -1;
                token = -1;
                for (int e = 0; e < valid; ++e) {
                    const float w = kind == kKindResidual ? weight_residual(lt[e], ld[e], d) : weight_target(lt[e], d);
                    run = __fadd_rn(run, w);
                    if (w > 0.0f) last_pos = e;
                    if (found_start + to_fixed(run, d.fix) > tin) {
                        token = e;
                        break;
                    }
                }
                if (token < 0) token = last_pos;
                token += static_cast<int>(e0) + found_vt * TPT;
            }
            a.out_tokens[static_cast<size_t>(jb.b) * (a.gamma + 1) + jb.n] = token;
            if (a.dbg.w_total) {
                const double W = static_cast<double>(total);
                a.dbg.w_total[jb.b] = kind == kKindResidual ? W * kFixResidualInv
                                                            : W * kFixTargetInv * static_cast<double>(d.isp);
            }
        }
        __syncwarp();
    }
}

size_t smem_bytes() {
    return static_cast<size_t>(kStages) * kStageBytes + sizeof(Ctl) +
           sizeof(Rec) * kConsumerWarps * kMaxRowsPerReq + sizeof(int) * (kMaxB + 1);
}

}  // namespace

bool streaming_applicable(const Args& a) {
    const size_t es = a.dtype == SV_F32 ? 4 : 2;
    if ((static_cast<size_t>(a.V) * es) % 16 != 0) return false;
    if ((reinterpret_cast<uintptr_t>(a.target) & 15) || (reinterpret_cast<uintptr_t>(a.draft) & 15)) return false;
    if (a.B > kMaxB) return false;
    return true;
}

int streaming_default_grid(const DeviceInfo& dev) { return dev.num_sms; }

bool streaming_grid_ok(int B, int grid) { return (B + grid - 1) / grid + 3 <= kMapMax; }

size_t streaming_workspace_bytes(int B, int gamma, int V, int dtype, int grid) {
    return make_layout(B, gamma, V, dtype == SV_F32 ? 4 : 2, grid).total;
}

cudaError_t launch_streaming(const Args& a, const DeviceInfo& dev, int grid, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
    const int es = a.dtype == SV_F32 ? 4 : 2;
    if (!streaming_grid_ok(a.B, grid)) return cudaErrorInvalidValue;
    const Layout L = make_layout(a.B, a.gamma, a.V, es, grid);
    if (workspace_bytes < L.total) return cudaErrorInvalidValue;
    const size_t smem = smem_bytes();
    const void* fn = a.dtype == SV_F32 ? reinterpret_cast<const void*>(&stream_kernel<SV_F32>)
                                       : reinterpret_cast<const void*>(&stream_kernel<SV_BF16>);
    static thread_local int attr_device = -1;
    if (attr_device != dev.device) {
        cudaError_t e = cudaFuncSetAttribute(&stream_kernel<SV_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(&stream_kernel<SV_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, &stream_kernel<SV_BF16>, kThreads, smem);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        attr_device = dev.device;
    }
    if (grid > dev.num_sms) return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(workspace, 0, 256, stream);
    if (e != cudaSuccess) return e;
    Args args = a;
    Layout lay = L;
    char* ws = static_cast<char*>(workspace);
    void* params[] = {&args, &lay, &ws};
    return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kThreads), params, smem, stream);
}

}  // namespace sv
