// Streaming path of libspecverify: one persistent, co-resident grid per call.
//
// The method ("Speculative Decoding : accélérer l'inférence des LLM",
// §Pourquoi la qualité est préservée; wiki "Speculative Decoding", eq. alpha(x)
// and eq. p_corr; "Accélérer Sonar grâce à la spéculation", §Décodage
// spéculatif) needs, per request, the normaliser (or argmax) of gamma+1
// target rows and gamma draft rows, a left-to-right scan, and one draw over a
// row that is known only after the scan. Each block has twelve consumer
// warps, one producer warp, one finisher warp and one search warp; there is
// no grid barrier.
//
//  1. Row statistics. Three streams of logits are cut into equal
//     16-byte-aligned slices: the target rows of the T > 0 requests, their
//     draft rows, and the target rows of the others (greedy, or invalid).
//     The first two are cut into W waves of G slices each (slice w G + g
//     goes to block g), the third into G slices. A block streams, wave by
//     wave, its target slice and its draft slice, then its slice of the
//     third stream. The requests of wave w are complete once wave w has
//     streamed, so their scans and draw jobs are done while later waves
//     still stream, and only the last wave's draws wait at the end; the
//     requests that need no draw come last. The
//     producer copies its slices through a ring of kStages shared-memory
//     stages with cp.async.bulk (completion on mbarriers; an evict-first L2
//     policy, so the streamed lines leave L2 before the small data the scans
//     and searches read); the consumers fold
//     each stage into per-thread (max, sum of 2^(l c - fl(m c))) or argmax
//     states, and the last warp to finish a row piece writes the block's
//     record for it. When a block's share of a request's rows is written, a
//     consumer posts it to the finisher; the finisher adds it to the
//     request's global count of folded logits, and the block that completes
//     the count runs the request's acceptance scan at once, while the other
//     blocks are still streaming: it merges the pieces of each row in a fixed
//     order, finds the first rejection, writes the accepted tokens and
//     publishes a draw job.
//  2. Draw. After its slice, a block's producer takes draw items (a job in
//     publication order, a chunk of kChunkBytes of the row it needs: target
//     row n and draft row n for a residual, target row n otherwise) from a
//     global counter; each thread sums the weights of a run of consecutive
//     tokens and each warp stores the sum of its 32 runs as a 64-bit
//     fixed-point integer (exact, so any order of addition gives the same
//     prefix sums). A job's chunks are counted in global memory, and the
//     search warp of the block that owns the job finds the chunk, then the
//     warp, then the run holding u * W, re-reads those 32 runs and finds the
//     token.
//
// Every wait is bounded (about two seconds, by the global timer): a stage or
// a message that never comes sets SV_STATUS_TIMEOUT and the kernel returns.
#include <algorithm>
#include <cmath>

#include "sv_common.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kConsumerWarps = 12;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kProducerWarp = kConsumerWarps;      // issues the bulk copies
constexpr int kFinisherWarp = kConsumerWarps + 1;  // counts, acceptance scans
constexpr int kSearchWarp = kConsumerWarps + 2;    // token searches of the jobs this block owns
constexpr int kThreads = kConsumers + 96;
constexpr int kHandoffThreads = kConsumers + 32;   // consumers + producer
constexpr int kQueue = 256;                        // finisher message ring (slots)
constexpr int kStages = 4;
constexpr int kStageBytes = 49152;
constexpr int kVecPerThread = kStageBytes / 16 / kConsumers;  // 8
constexpr int kChunkBytes = 24576;  // draw-phase chunk of one row (a residual item fills a stage)
constexpr int kMapMax = 256;   // requests in one block's slices of one stream (all waves)
// Waves of the T > 0 requests' streams. More waves let the early requests'
// scans and draws run while later waves stream, but every wave adds row pieces
// to each block (each ends in a reduction across the block's warps and a
// partial stage), and a wave's scans fall on the blocks whose pieces finish
// last; on GB300 4 and 16 waves were slower than one on the sampling, mixed
// and large batches. One wave (the general slicing passed the GPU tests at 16).
constexpr int kMaxWaves = 1;
constexpr long long kWaveSliceBytes = 256 << 10;  // a block's target slice of one wave, at least
constexpr int kPrePieces = 3;  // row pieces the acceptance scan reads in its first round
constexpr int kMaxGrid = 256;  // blocks (partition tables live in shared memory)
constexpr int kGrab = 4;       // draw items a producer takes per atomic
constexpr int kEeItemsPerProducer2 = 11;  // early exit: position-0 items a producer takes, about, times 2
constexpr int kEeGroupMax = 8;            // early exit: chunks of one task in one item, at most
constexpr int kJobMsg = 0x40000000;  // finisher message flag: a draw item of job (item & ~flag)
constexpr int kEndKind = -2;   // stage descriptor kind: no more draw items
constexpr int kMaxB = 4096;
constexpr int kMaxRowsPerReq = 2 * SV_MAX_GAMMA + 1;
constexpr int kFlushSlots = 16;  // row pieces in flight between the fastest and slowest warp
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;

// Named barriers (0 is __syncthreads).
constexpr int kBarConsumers = 1;  // the 256 consumer threads
constexpr int kBarHandoff = 2;    // consumers arrive, producer waits (kHandoffThreads)

struct Rec {
    float m;      // max value (both modes)
    float s;      // sum 2^(l c - fl(m c)) (max/sum mode; plain where idx says so)
    int32_t idx;  // argmax (argmax mode); max/sum mode: kRecPlain for a plain sum, else -1
    int32_t bad;  // kBadData: NaN or +inf seen; kBadPlain: the anchor left its range
};
constexpr uint32_t kNoPiece = 0xffffffffu;  // Rec.bad of a piece that does not exist
constexpr int32_t kRecPlain = 1;
constexpr int kBadData = 1;   // a NaN or +inf logit, or a row of only -inf: the request is invalid
constexpr int kBadPlain = 2;  // |fl(m c)| >= 2^23 or c overflowed: the row is recomputed plain

__device__ __forceinline__ MaxSum ms_of(const Rec& r) { return MaxSum{r.m, r.s, r.idx == kRecPlain ? 1 : 0}; }

struct Job {
    int32_t b, n, kind, pad;  // request, the draw's row, kind, u_sample bits
    int32_t slot;             // output position of the drawn token (the row n, except in trees)
    DrawParams d;
};

// What a draw-phase stage holds: chunk j of job k (kind kEndKind: none). In
// the early-exit kernel: chunk j of task k, a row-statistics task (type
// kTaskStats: request job.b, position job.n, scale job.d.c, flags) or a draw
// task (type kTaskDraw, the job itself).
struct StageDesc {
    Job job;
    int32_t k, j;
    int32_t type, flags;
    int32_t item, nch;  // early exit: the chunk's item within its task, chunks of the item up to it
};

// Early-exit tasks: the row statistics of one position of one request (the
// target row, and the draft row for model proposals at T > 0), or one draw.
constexpr int kTaskStats = 0;
constexpr int kTaskDraw = 1;
constexpr int kStatsArgmax = 1;  // StageDesc.flags: argmax (T == 0) instead of (max, sum)
constexpr int kStatsDraft = 2;   // StageDesc.flags: the stage also holds the draft row's chunk
constexpr int kItemFirst = 4;    // StageDesc.flags: the first stage of an early-exit item
constexpr int kItemLast = 8;     // StageDesc.flags: the last stage of an early-exit item

// Byte offsets into the caller's workspace and the partition constants.
struct Layout {
    long long Et;  // target elements B*(gamma+1)*V
    int G, NRT, NRD, NCH, vec;  // NRT, NRD: row-piece records of the target and draft streams
    int NI;   // early exit: items per task, groups of GRP chunks
    int GRP;  // early exit: chunks of one task taken as one item
    size_t hdr, req_done, job_done, ready, ee_tasks, ee_done, clear_bytes, rec_t, rec_d, ee_rec, jobs, jobset,
        wsums, total;
    int ee_cap;  // early exit: task slots, B (gamma + 2)
};

// A stream of E elements cut into NS slices of S elements (S a multiple of
// the 16-byte vector; the last slices may be short or empty): slice i is
// [min(E, i S), min(E, (i + 1) S)).
struct Slicing {
    long long E, S;
    int NS;
};
__host__ __device__ inline Slicing make_slicing(long long E, int NS, int vec) {
    long long S = (E + NS - 1) / NS;
    S = (S + vec - 1) / vec * vec;
    return Slicing{E, S > vec ? S : vec, NS};
}
__device__ __forceinline__ long long slice_begin(const Slicing& s, long long i) { return min(s.E, i * s.S); }
// The slice holding element e (0 <= e < E).
__device__ __forceinline__ int slice_of(const Slicing& s, long long e) {
    return static_cast<int>(min(static_cast<long long>(s.NS - 1), e / s.S));
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

Layout make_layout(int B, int gamma, int V, int es, int G) {
    Layout L;
    L.G = G;
    L.vec = 16 / es;
    L.Et = static_cast<long long>(B) * (gamma + 1) * V;
    const long long Ed_max = static_cast<long long>(B) * gamma * V;
    // the piece of row r in slice i has record r + i (see piece_rec): at most
    // the rows plus the slices of each stream (W G of the T > 0 requests'
    // target rows, then 2G of the others')
    L.NRT = static_cast<int>(L.Et / V) + (kMaxWaves + 2) * G;
    L.NRD = static_cast<int>(Ed_max / V) + kMaxWaves * G;
    const int chunk_elems = kChunkBytes / es;
    L.NCH = (V + chunk_elems - 1) / chunk_elems;
    // Early exit: items of GRP chunks. Large items amortise the per-item costs
    // (the grab, the task lookup, the flush) when the batch keeps every
    // producer busy; small ones spread a task over more blocks, which
    // shortens the chain of a request that keeps accepting. GRP is chosen so
    // that the position-0 tasks (B of them) make about 5.5 items a producer
    // (same-box sweeps: 2 chunks best for B = 64 fp32 rows of 128256, 3 for
    // 256 bf16 rows of 128256, 6 to 8 for 512 bf16 rows of 152064).
    {
        const long long x = 2LL * B * L.NCH, d = static_cast<long long>(kEeItemsPerProducer2) * G;
        L.GRP = static_cast<int>(std::min<long long>(kEeGroupMax, std::max<long long>(1, (x + d / 2) / d)));
    }
    L.NI = (L.NCH + L.GRP - 1) / L.GRP;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = align256(off + bytes);
        return at;
    };
    L.hdr = take(256);
    L.req_done = take(static_cast<size_t>(B) * 4);  // logits folded, per request
    L.job_done = take(static_cast<size_t>(B) * 4);  // chunks summed, per draw job
    L.ready = take(static_cast<size_t>(B) * 4);     // published draw jobs (k + 1), in order
    // early exit: B position-0 tasks, then at most gamma more positions and one
    // draw per request
    L.ee_cap = B * (gamma + 2);
    L.ee_tasks = take(static_cast<size_t>(L.ee_cap) * 8);  // published tasks: code (low word), scale c
    L.ee_done = take(static_cast<size_t>(L.ee_cap) * 4);   // chunks done, per task
    L.clear_bytes = off;  // cleared before every launch (up to ee_tasks without early exit)
    L.rec_t = take(static_cast<size_t>(L.NRT) * sizeof(Rec));
    L.rec_d = take(static_cast<size_t>(L.NRD) * sizeof(Rec));
    L.ee_rec = take(static_cast<size_t>(L.ee_cap) * L.NI * 2 * sizeof(Rec));  // per (task, item): target, draft
    L.jobs = take(static_cast<size_t>(B) * sizeof(Job));
    L.jobset = take(static_cast<size_t>(B) * gamma * 4);  // tree jobs: tokens excluded from the last draw
    L.wsums = take(static_cast<size_t>(B) * L.NCH * kConsumerWarps * 8);
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

// The same copy with an L2 eviction policy (a createpolicy value).
__device__ __forceinline__ void bulk_copy_hint(void* dst_smem, const void* src, unsigned bytes, uint64_t* bar,
                                               uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_u32(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// An L2 policy whose lines are evicted before the others'.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Adds v to a global counter with release semantics at GPU scope, without
// waiting for the result.
__device__ __forceinline__ void red_release_add(unsigned* addr, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}

// Polled words in global memory are read and written with device-scope
// relaxed accesses (a volatile access has system scope, more than these
// words need); the orderings they need come from explicit fences or from
// release and acquire-release operations (st_release, atom_add_acq_rel).
__device__ __forceinline__ int ld_relaxed(const int* p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned ld_relaxed(const unsigned* p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Publishes a word after the writer's earlier stores (release at GPU scope).
__device__ __forceinline__ void st_release(int* p, int v) {
    asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Adds v to a global counter and returns the old value; release orders the
// caller's earlier writes before the add, acquire its later reads after it.
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ unsigned long long ld_relaxed(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
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

// Byte permute: the bytes of x selected by `sel` (zero bytes come from the
// second operand, 0).
__device__ __forceinline__ uint32_t prmt(uint32_t x, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(x), "r"(sel));
    return r;
}

// Packed pairs of binary32 (the sm_100-family f32x2 arithmetic).
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ unsigned long long f2_pack_bits(uint32_t lo, uint32_t hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// ---------------------------------------------------------------- barriers

struct Hdr {
    int status;          // SV_STATUS_* bits of this call
    unsigned n_pub;      // draw jobs (early exit: tasks past the first B) published so far
    unsigned next_item;  // draw items handed out so far
    unsigned n_fin;      // early exit: requests finished
};

// Checking output: global-timer stamps (see sv_debug_out.phase_ns).
__device__ __forceinline__ void stamp(unsigned long long* slots, int i, bool who) {
    if (slots && who) {
        const unsigned long long now = global_ns();
        if (i == 0) {
            atomicMin(slots, now);
            atomicMax(slots + 1, now);
        } else {
            atomicMax(slots + i, now);
        }
    }
}

// ------------------------------------------------------------ kernel context

struct Ctl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    // the three streams (after the prologue): the sampled requests' target
    // rows (virtual elements 0..E1), their draft rows, the others' target rows
    // (virtual elements E1..Et, sliced from 0)
    Slicing sl[3];
    int nwave;                     // W: waves of the first two streams (slices W G each)
    StageDesc desc[kStages];       // draw phase: the item in each stage
    int n_samp;
    int j3_lo;  // first other request (by its index among them) of this block's other-target slice
    int abort;
    // this block's slices of the first two streams, wave by wave: the first
    // compacted request (lo) and the place of its entry in the map (off)
    int wlo[2][kMaxWaves];
    int woff[2][kMaxWaves + 1];
    short wmap[2][kMapMax];  // request b of each compacted index those slices hold
    int wtmp[kConsumerWarps + 1];
    Rec wrec[kFlushSlots][kConsumerWarps];  // per-warp partials of a row piece
    Rec wrec2[kFlushSlots][kConsumerWarps]; // early exit: per-warp partials of the draft row
    int wcnt[kFlushSlots];                  // warps that have flushed the piece
    int fq_item[kQueue];                    // finisher ring: request (phase 1) or job (phase 2)
    unsigned fq_val[kQueue];                // logits (phase 1) or chunks (phase 2) it covers
    unsigned fq_seq[kQueue];                // reservation number + 1 of the entry in the slot
    unsigned fq_tail;                       // reservations so far
    unsigned fq_head;                       // entries the finisher has taken
    int cons_done;                          // consumer warps done with both phases
    short kmap[kMaxB];                      // compacted index k of each T > 0 request, else -(j + 1),
                                            // j its index among the others
    short map3[kMapMax];                    // other-target slice: request of other index j3_lo + i
    int dset[kStages][SV_MAX_GAMMA];        // tree draws: the excluded tokens of the item in each stage
    int fset[SV_MAX_GAMMA];                 // tree draws: the excluded tokens of the job being searched
    int wset[kConsumerWarps][SV_MAX_GAMMA]; // tree draws: each consumer warp's copy of its item's set
};

struct RowLoc {
    int kind;       // 0 target row, 1 draft row
    long long row;  // target row index, or compacted draft row index
    int req;        // request b
    int slot;       // row slot of this block
};

// A piece of one row inside this block's slice.
struct Segment {
    const char* src;
    long long elems;
    long long e0;  // first element, offset within the row
    RowLoc loc;
    bool last;     // the last piece of this request's rows in the slice
};


template <int DT>
struct Kern {
    static constexpr int ES = DT == SV_F32 ? 4 : 2;
    static constexpr int kStageElems = kStageBytes / ES;  // phase-1 stage
    static constexpr int kChunkElems = kChunkBytes / ES;  // draw-phase chunk
    static constexpr int kTPT = kChunkElems / kConsumers;  // tokens per thread run (64 bytes)

    const Args& a;
    const Layout& L;
    char* ws;
    Ctl& ctl;
    char* stages;
    int G, g;

    __device__ Hdr* hdr() const { return reinterpret_cast<Hdr*>(ws + L.hdr); }
    __device__ Rec* rec_t() const { return reinterpret_cast<Rec*>(ws + L.rec_t); }
    __device__ Rec* rec_d() const { return reinterpret_cast<Rec*>(ws + L.rec_d); }
    __device__ Job* jobs() const { return reinterpret_cast<Job*>(ws + L.jobs); }
    __device__ int* jobset() const { return reinterpret_cast<int*>(ws + L.jobset); }
    __device__ unsigned* req_done() const { return reinterpret_cast<unsigned*>(ws + L.req_done); }
    __device__ unsigned* job_done() const { return reinterpret_cast<unsigned*>(ws + L.job_done); }
    __device__ int* ready() const { return reinterpret_cast<int*>(ws + L.ready); }
    // Task slot p: the task's code in the low word (0 until published), and for
    // a statistics task the bits of its scale c in the high word.
    __device__ unsigned long long* ee_slot(int p) const {
        return reinterpret_cast<unsigned long long*>(ws + L.ee_tasks) + p;
    }
    __device__ unsigned* ee_done() const { return reinterpret_cast<unsigned*>(ws + L.ee_done); }
    __device__ Rec* ee_rec() const { return reinterpret_cast<Rec*>(ws + L.ee_rec); }
    __device__ unsigned long long* wsums() const {
        return reinterpret_cast<unsigned long long*>(ws + L.wsums);
    }

    __device__ static bool sampled(float T) { return T > 0.0f && T < pos_inf(); }

    // ---- phase-1 schedule: row pieces of this block's slices, in order.
    // Target rows are streamed in a virtual order: the T > 0 requests' rows
    // (request of compacted index k at virtual rows k (gamma+1) ...), then the
    // other requests' (index j among them, after all n_samp of the former).
    // Wave by wave, a block streams its slice of the first and its slice of
    // the T > 0 requests' draft rows; then its slice of the others' rows, so
    // that the requests that need a draw are complete (scanned, their jobs
    // published) while the rows of those that need none still stream. The
    // piece of row r in slice i of a stream has record r + i (slices of the
    // others' rows count after the first stream's W G).

    // Request b of compacted index k in this block's slices of stream st
    // (0 target, 1 draft) of wave w; -1 if it is not there.
    __device__ int wave_req(int st, int w, long long k) const {
        const long long rel = k - ctl.wlo[st][w];
        return (rel >= 0 && rel < ctl.woff[st][w + 1] - ctl.woff[st][w]) ? ctl.wmap[st][ctl.woff[st][w] + rel] : -1;
    }

    // Virtual target elements [vs, ve) of slice `is` (wave w of the first
    // stream; w < 0: the others' rows).
    // The row, request and position advance by increments from the slice's
    // first element (one division per slice, none per piece).
    template <typename F>
    __device__ void for_each_target_segment(long long vs, long long ve, int is, int w, F& f) const {
        const int V = a.V, GM = a.gamma, ns = ctl.n_samp;
        if (vs >= ve) return;
        long long vr = vs / V;
        long long pos = vr / (GM + 1);
        int i = static_cast<int>(vr - pos * (GM + 1));
        for (long long e = vs; e < ve; ++vr) {
            const long long end = min(ve, (vr + 1) * V);
            int b = -1;
            if (pos < ns) {
                if (w >= 0) b = wave_req(0, w, pos);
            } else {
                const long long rel = pos - ns - ctl.j3_lo;
                if (rel >= 0 && rel < kMapMax) b = ctl.map3[rel];
            }
            const long long slot = vr + is;
            if (b < 0 || b >= a.B || slot >= L.NRT) {  // cannot happen when the host checks hold
                ctl.abort = 1;
                return;
            }
            const long long row = static_cast<long long>(b) * (GM + 1) + i;  // its place in memory
            Segment sg;
            sg.src = static_cast<const char*>(a.target) + (row * V + (e - vr * V)) * ES;
            sg.elems = end - e;
            sg.e0 = e - vr * V;
            sg.loc = {0, vr, b, static_cast<int>(slot)};
            sg.last = end == ve || i == GM;
            f(sg);
            e = end;
            if (++i > GM) {
                i = 0;
                ++pos;
            }
        }
    }

    // Compacted draft elements [ds, de) of slice `is` (wave w).
    template <typename F>
    __device__ void for_each_draft_segment(long long ds, long long de, int is, int w, F& f) const {
        const int V = a.V, GM = a.gamma;
        if (ds >= de) return;
        long long kr = ds / V;
        int k = static_cast<int>(kr / GM), i = static_cast<int>(kr - static_cast<long long>(k) * GM);
        for (long long e = ds; e < de; ++kr) {
            const long long end = min(de, (kr + 1) * V);
            const int b = wave_req(1, w, k);
            const long long slot = kr + is;
            if (b < 0 || b >= a.B || slot >= L.NRD) {  // cannot happen when the host checks hold
                ctl.abort = 1;
                return;
            }
            const long long base = (static_cast<long long>(b) * GM + i) * V;
            Segment sg;
            sg.src = static_cast<const char*>(a.draft) + (base + (e - kr * V)) * ES;
            sg.elems = end - e;
            sg.e0 = e - kr * V;
            sg.loc = {1, kr, b, static_cast<int>(slot)};
            sg.last = end == de || i == GM - 1;
            f(sg);
            e = end;
            if (++i == GM) {
                i = 0;
                ++k;
            }
        }
    }

    // Every row piece of this block, in streaming order: its slices of the
    // T > 0 requests' rows, wave by wave, then its two slices of the others'
    // rows (cut into 2G slices, block g taking 2g and 2g + 1: measured a
    // little faster than one slice a block, its fp32 build spilling 24 bytes a
    // thread instead of 48).
    template <typename F>
    __device__ void for_each_segment(F&& f) const {
        const int W = ctl.nwave;
        for (int w = 0; w < W; ++w) {
            const int is = w * G + g;
            for_each_target_segment(slice_begin(ctl.sl[0], is), slice_begin(ctl.sl[0], is + 1), is, w, f);
            for_each_draft_segment(slice_begin(ctl.sl[1], is), slice_begin(ctl.sl[1], is + 1), is, w, f);
        }
        const long long E1 = ctl.sl[0].E;
        for (int i3 = 2 * g; i3 < 2 * g + 2; ++i3)
            for_each_target_segment(E1 + slice_begin(ctl.sl[2], i3), E1 + slice_begin(ctl.sl[2], i3 + 1), W * G + i3,
                                    -1, f);
    }

    // ---- the ring: producer and consumer cursors
    struct Cursor {
        unsigned it = 0;
    };

    // Producer warp: fill the next stage with one copy, or two (the second at
    // byte offset kChunkBytes); lane 0 issues. In the draw phase lane 0 first
    // writes the stage's descriptor; `src` null with `desc` sends the end
    // marker (the stage completes with no bytes).
    // `set0`, `set1`: a tree draw's excluded tokens lane and lane + 32 (nset
    // of them), copied into the stage's descriptor area.
    __device__ bool produce(Cursor& p, const char* src, unsigned bytes, const char* src2 = nullptr,
                            unsigned bytes2 = 0, const StageDesc* desc = nullptr, int set0 = 0, int set1 = 0,
                            int nset = 0) const {
        const int slot = p.it % kStages;
        const unsigned round = p.it / kStages;
        // the verdict is made warp-uniform so that a timeout cannot split the warp
        if (round > 0 && !__all_sync(0xffffffffu, mbar_wait(&ctl.empty[slot], (round - 1) & 1))) return false;
        // a tree draw's excluded tokens travel with the stage
        if (nset > 0) {
            const int lane = threadIdx.x & 31;
            if (lane < nset) ctl.dset[slot][lane] = set0;
            if (lane + 32 < nset) ctl.dset[slot][lane + 32] = set1;
            __syncwarp();
        }
        if ((threadIdx.x & 31) == 0) {
            if (desc) ctl.desc[slot] = *desc;
            if (src) {
                char* dst = stages + static_cast<size_t>(slot) * kStageBytes;
                mbar_expect_tx(&ctl.full[slot], bytes + bytes2);
                bulk_copy(dst, src, bytes, &ctl.full[slot]);
                if (src2) bulk_copy(dst + kChunkBytes, src2, bytes2, &ctl.full[slot]);
            } else {
                mbar_arrive(&ctl.full[slot]);  // release: the descriptor is visible to the waiters
            }
        }
        __syncwarp();
        ++p.it;
        return true;
    }

    // A row-stream stage: one copy with an L2 eviction policy (lane 0 issues).
    __device__ bool produce_stream(Cursor& p, const char* src, unsigned bytes, uint64_t policy) const {
        const int slot = p.it % kStages;
        const unsigned round = p.it / kStages;
        if (round > 0 && !__all_sync(0xffffffffu, mbar_wait(&ctl.empty[slot], (round - 1) & 1))) return false;
        if ((threadIdx.x & 31) == 0) {
            char* dst = stages + static_cast<size_t>(slot) * kStageBytes;
            mbar_expect_tx(&ctl.full[slot], bytes);
            bulk_copy_hint(dst, src, bytes, &ctl.full[slot], policy);
        }
        __syncwarp();
        ++p.it;
        return true;
    }

    // Waits (bounded) until every copy the producer issued has landed.
    __device__ void drain(const Cursor& p) const {
        const unsigned n = p.it;
        for (unsigned j = (n > kStages ? n - kStages : 0); j < n; ++j)
            mbar_wait(&ctl.full[j % kStages], (j / kStages) & 1);
    }

    __device__ const char* consume_begin(Cursor& c) const {
        const int slot = c.it % kStages;
        if (!__all_sync(0xffffffffu, mbar_wait(&ctl.full[slot], (c.it / kStages) & 1))) return nullptr;
        return stages + static_cast<size_t>(slot) * kStageBytes;
    }
    __device__ void consume_end(Cursor& c) const {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(&ctl.empty[c.it % kStages]);
        ++c.it;
    }

    // A bounded wait ran out: the block stops and the status bit is set.
    __device__ void set_abort(int32_t* d_status) const {
        ctl.abort = 1;
        atomicOr(&hdr()->status, SV_STATUS_TIMEOUT);
        if (d_status) atomicOr(d_status, SV_STATUS_TIMEOUT);
    }

    // Publishes draw job k (its record written by this thread): the producers
    // of every block take draw items from the jobs in publication order.
    __device__ void publish(int k) const {
        const unsigned p = atomicAdd(&hdr()->n_pub, 1u);
        st_release(ready() + p, k + 1);  // the job's record lands before its entry
    }

    // Search warp: the token searches of the jobs published at positions
    // g, g + G, g + 2G, ... belong to block g, so that consecutive jobs, which
    // complete at about the same time, are searched by different blocks. Lane
    // 0 keeps the next owned position (own_p) and its job once published
    // (own_k); a poll reads one global word and runs the search when the job's
    // last chunk is counted. Returns whether it made progress.
    __device__ bool poll_owned(int& own_p, int& own_k) const {
        int k = -1, moved = 0;
        if ((threadIdx.x & 31) == 0) {
            const int ns = *reinterpret_cast<const volatile int*>(&ctl.n_samp);
            if (own_p < ns) {
                if (own_k < 0) {
                    const int v = ld_relaxed(ready() + own_p);
                    if (v) {
                        __threadfence();
                        own_k = v - 1;
                        const int kind = __ldcg(&jobs()[own_k].kind);
                        if (kind != kKindResidual && kind != kKindBonus && kind != kKindResidualOnehot &&
                            kind != kKindResidualTree) {  // no items, no search
                            own_p += G;
                            own_k = -1;
                            moved = 1;
                        }
                    }
                }
                if (own_k >= 0 &&
                    ld_relaxed(job_done() + own_k) == static_cast<unsigned>(L.NCH)) {
                    __threadfence();  // the other blocks' chunk sums before they are read
                    k = own_k;
                    own_p += G;
                    own_k = -1;
                }
            }
        }
        k = __shfl_sync(0xffffffffu, k, 0);
        moved = __shfl_sync(0xffffffffu, moved, 0);
        if (k < 0) return moved != 0;
        search_job(k);
        __syncwarp();
        stamp(reinterpret_cast<unsigned long long*>(a.dbg.phase_ns), 7, (threadIdx.x & 31) == 0);
        return true;
    }

    // ---- the finisher's message ring. One consumer lane posts a message once
    // this block's share of a request (phase 1) or of a draw job (phase 2) is
    // in global memory; the finisher warp adds the share to the item's global
    // counter, and the block whose share completes the item finishes it. The
    // consumers never wait on a global atomic or fence.
    //
    // Posts (one lane): false if the ring stayed full for the time limit.
    __device__ bool post(int item, unsigned val) const {
        const unsigned s = atomicAdd(&ctl.fq_tail, 1u);
        volatile unsigned* vhead = &ctl.fq_head;
        volatile int* vabort = &ctl.abort;
        if (s - *vhead >= static_cast<unsigned>(kQueue)) {
            const unsigned long long t0 = global_ns();
            while (s - *vhead >= static_cast<unsigned>(kQueue)) {
                if (*vabort || global_ns() - t0 > kWaitTimeoutNs) return false;
                __nanosleep(128);
            }
        }
        const int i = static_cast<int>(s % kQueue);
        ctl.fq_item[i] = item;
        ctl.fq_val[i] = val;
        __threadfence_block();  // the entry, then its sequence number
        reinterpret_cast<volatile unsigned*>(ctl.fq_seq)[i] = s + 1;
        return true;
    }

    // A consumer warp is done with both phases (after its last post).
    __device__ void consumer_done() const {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) {
            __threadfence_block();
            atomicAdd(&ctl.cons_done, 1);
        }
    }

    // Finisher warp: takes the ring's messages in batches of up to 32; with
    // the ring empty it polls its owned token searches (at most every half
    // microsecond). It returns once every consumer warp is done, the ring is
    // empty and every owned search has run.
    // count(item, val), one lane per message, adds the share to the item's
    // global counter (with the ordering its reader needs) and returns whether
    // that completed the item; work(item), on the whole warp, then finishes
    // each completed item.
    // poll(), on the whole warp, runs owned work that became ready and says
    // whether it did; owned_done(), on lane 0, says that no owned work remains.
    template <typename C, typename W, typename P, typename D>
    __device__ void finish(C&& count, W&& work, P&& poll, D&& owned_done) const {
        const int lane = threadIdx.x & 31;
        volatile unsigned* vseq = ctl.fq_seq;
        volatile int* vdone = &ctl.cons_done;
        unsigned head = 0;
        volatile int* vabort = &ctl.abort;
        unsigned long long t0 = global_ns(), last_poll = 0;
        for (;;) {
            const unsigned s = head + lane;
            const unsigned ready = __ballot_sync(0xffffffffu, vseq[s % kQueue] == s + 1);
            const int n = ready == 0xffffffffu ? 32 : __ffs(~ready) - 1;  // ready entries from head on
            if (n > 0) {
                __threadfence_block();
                int item = -1;
                unsigned val = 0;
                if (lane < n) {
                    item = ctl.fq_item[s % kQueue];
                    val = ctl.fq_val[s % kQueue];
                }
                __syncwarp();
                head += n;
                if (lane == 0) *reinterpret_cast<volatile unsigned*>(&ctl.fq_head) = head;
                bool completed = false;
                if (lane < n) completed = count(item, val);
                unsigned done = __ballot_sync(0xffffffffu, completed);
                while (done) {
                    const int src = __ffs(done) - 1;
                    done &= done - 1;
                    work(__shfl_sync(0xffffffffu, item, src));
                    __syncwarp();
                }
                t0 = global_ns();
                continue;
            }
            if (global_ns() - last_poll > 500ull) {
                if (poll()) {
                    t0 = global_ns();
                    continue;
                }
                last_poll = global_ns();
            }
            int stop = 0;
            if (lane == 0) {
                if (*vabort) {
                    stop = 1;
                } else if (*vdone == kConsumerWarps) {
                    __threadfence_block();
                    if (*reinterpret_cast<volatile unsigned*>(&ctl.fq_tail) == head && owned_done()) stop = 1;
                }
                if (!stop && global_ns() - t0 > kWaitTimeoutNs) {
                    set_abort(a.d_status);
                    stop = 1;
                }
            }
            if (__shfl_sync(0xffffffffu, stop, 0)) return;
            __nanosleep(200);
        }
    }

    // ---- phase-1 prologue (consumers): the count of T > 0 requests, the
    // partition tables of the three streams (the T > 0 requests' target rows,
    // their draft rows, the other requests' target rows), and the maps of this
    // block's slices to requests.
    __device__ void prologue() const {
        const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
        int cnt = 0;
        for (int b = t; b < a.B; b += kConsumers) cnt += sampled(a.temperature[b]) ? 1 : 0;
        cnt = __reduce_add_sync(0xffffffffu, cnt);
        if (lane == 0) ctl.wtmp[warp] = cnt;
        bar_sync(kBarConsumers, kConsumers);
        int n = 0;
        for (int w = 0; w < kConsumerWarps; ++w) n += ctl.wtmp[w];
        // the streams: the T > 0 requests' target rows (E1) and draft rows (E2,
        // none for one-hot proposals) in W waves, the others' target rows (E3)
        const long long R = static_cast<long long>(a.gamma + 1) * a.V;
        const long long D = static_cast<long long>(a.gamma) * a.V;
        const long long E1 = static_cast<long long>(n) * R, E3 = static_cast<long long>(a.B - n) * R;
        const long long E2 = a.onehot ? 0ll : static_cast<long long>(n) * D;
        // waves: a block's target slice of one wave holds kWaveSliceBytes or
        // more, and its slices of all waves fit the maps (each slice holds at
        // most (S - 1) / R + 2 requests, so W waves at most n / G + 3 W)
        int W = static_cast<int>(min(static_cast<long long>(kMaxWaves),
                                     max(1ll, E1 * ES / (static_cast<long long>(G) * kWaveSliceBytes))));
        while (W > 1 && (n + G - 1) / G + 3 * W + 1 > kMapMax) --W;
        const Slicing s1 = make_slicing(E1, W * G, L.vec), s2 = make_slicing(E2, W * G, L.vec);
        const Slicing s3 = make_slicing(E3, 2 * G, L.vec);
        const int j3_lo = static_cast<int>(slice_begin(s3, 2 * g) / R);
        if (t == 0) {
            ctl.n_samp = n;
            ctl.nwave = W;
            ctl.sl[0] = s1;
            ctl.sl[1] = s2;
            ctl.sl[2] = s3;
            ctl.j3_lo = j3_lo;
            // the compacted requests of this block's slices, wave by wave
            for (int st = 0; st < 2; ++st) {
                const Slicing& sl = st == 0 ? s1 : s2;
                const long long per = st == 0 ? R : D;
                int off = 0;
                for (int w = 0; w < W; ++w) {
                    const long long b0 = slice_begin(sl, static_cast<long long>(w) * G + g);
                    const long long b1 = slice_begin(sl, static_cast<long long>(w) * G + g + 1);
                    const int lo = b1 > b0 ? static_cast<int>(b0 / per) : 0;
                    const int cnt = b1 > b0 ? static_cast<int>((b1 - 1) / per) - lo + 1 : 0;
                    ctl.wlo[st][w] = lo;
                    ctl.woff[st][w] = off;
                    off = min(off + cnt, kMapMax);
                }
                ctl.woff[st][W] = off;
            }
        }
        bar_sync(kBarConsumers, kConsumers);
        int carry = 0;
        for (int base = 0; base < a.B; base += kConsumers) {
            const int b = base + t;
            const int f = (b < a.B && sampled(a.temperature[b])) ? 1 : 0;
            const unsigned ball = __ballot_sync(0xffffffffu, f);
            const int in_warp = __popc(ball & ((1u << lane) - 1u));
            if (lane == 0) ctl.wtmp[warp] = __popc(ball);
            bar_sync(kBarConsumers, kConsumers);
            int before = carry, total = 0;
            for (int w = 0; w < kConsumerWarps; ++w) {
                if (w < warp) before += ctl.wtmp[w];
                total += ctl.wtmp[w];
            }
            const int k = before + in_warp;  // T > 0 requests before b
            if (b < a.B) {
                if (f) {
                    for (int st = 0; st < 2; ++st)
                        for (int w = 0; w < W; ++w) {
                            const int rel = k - ctl.wlo[st][w];
                            if (rel >= 0 && rel < ctl.woff[st][w + 1] - ctl.woff[st][w])
                                ctl.wmap[st][ctl.woff[st][w] + rel] = static_cast<short>(b);
                        }
                    ctl.kmap[b] = static_cast<short>(k);
                } else {
                    const int j = b - k;  // the others before b
                    const int rel3 = j - j3_lo;
                    if (rel3 >= 0 && rel3 < kMapMax) ctl.map3[rel3] = static_cast<short>(b);
                    ctl.kmap[b] = static_cast<short>(-(j + 1));
                }
                // A request's count stays -1 until the request is final (then its
                // scan, or its draw, writes it), so that a call that gives up on a
                // wait shows -1 for every request not yet final. The block whose
                // slice holds the first element of the request's target rows
                // clears it here, before it posts any share (the scan comes after
                // every share).
                const int first_block = f ? slice_of(s1, static_cast<long long>(k) * R) % G
                                          : slice_of(s3, static_cast<long long>(b - k) * R) / 2;
                if (first_block == g) a.out_num_accepted[b] = -1;
            }
            carry += total;
            bar_sync(kBarConsumers, kConsumers);
        }
        __threadfence();  // the cleared counts, before this block's first post
    }

    // ---- phase-1 consumer: per-thread state of the current row piece
    struct RowState {
        float m, mc, s;  // max/sum mode (mc = fl(m c))
        int idx;         // argmax mode
        int bad;
        bool argmax;
        float c;
    };

    // The request's temperature turned into (sampled, c), kept for the pieces
    // of the same request that follow (a request's rows are consecutive).
    struct ReqScale {
        int req = -1;
        bool samp = false;
        float c = 0.0f;
    };
    __device__ void start_row(RowState& rs, const RowLoc& loc, ReqScale& rq) const {
        if (loc.req != rq.req) {
            const float T = a.temperature[loc.req];
            rq.req = loc.req;
            rq.samp = sampled(T);
            rq.c = rq.samp ? temp_scale(T).c : 0.0f;
        }
        rs.argmax = loc.kind == 0 && !rq.samp;
        rs.c = rs.argmax ? 0.0f : rq.c;
        rs.m = neg_inf();
        rs.mc = neg_inf();
        rs.s = 0.0f;
        rs.idx = 0x7fffffff;
        rs.bad = 0;
    }

    // The records of a warp's lanes merged (every lane gets the result): the
    // lowest-index argmax, or for (max, sum) the max first and then each
    // lane's sum rescaled to it and added up in a butterfly, so that the
    // dependent chain holds one 2^x rather than one a level. Lanes with
    // nothing to add hold (-inf, 0).
    __device__ static Rec rec_reduce(Rec x, bool argmax, float c) {
        const int bad = static_cast<int>(__reduce_or_sync(0xffffffffu, static_cast<unsigned>(x.bad)));
        if (argmax) {
            ArgMax st{x.m, x.idx};
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                ArgMax ot{__shfl_xor_sync(0xffffffffu, st.v, o), __shfl_xor_sync(0xffffffffu, st.i, o)};
                st = argmax_merge(st, ot);
            }
            return Rec{st.v, 0.0f, st.i, bad};
        }
        float m = x.m;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float t = x.m == neg_inf() ? 0.0f : __fmul_rn(x.s, ex2(__fsub_rn(scaled_max(x.m, c), scaled_max(m, c))));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, o));
        return Rec{m, t, -1, bad};
    }
    __device__ static Rec lane_rec(const RowState& rs) { return Rec{rs.m, rs.s, rs.idx, rs.bad}; }
    __device__ static Rec no_rec() { return Rec{neg_inf(), 0.0f, 0x7fffffff, 0}; }

    // The warps of a block fold disjoint parts of each row piece. Each warp
    // reduces its lanes, parks the result in shared slot `seq % kFlushSlots`,
    // and the last warp to arrive merges the 12 partials (lane w holding warp
    // w's) and writes the block's record for the piece (no block-wide
    // barrier). When `share` is non-zero this piece ends the request's rows in
    // the slice: the merging warp then posts the request with the share's
    // element count.
    __device__ void flush_row(const RowState& rs, const RowLoc& loc, unsigned seq, unsigned share) const {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        const Rec rec = rec_reduce(lane_rec(rs), rs.argmax, rs.c);
        const int fs = static_cast<int>(seq % kFlushSlots);
        int last = 0;
        if (lane == 0) {
            ctl.wrec[fs][warp] = rec;
            __threadfence_block();
            last = atomicAdd(&ctl.wcnt[fs], 1) == kConsumerWarps - 1;
        }
        if (!__shfl_sync(0xffffffffu, last, 0)) return;
        __threadfence_block();
        const Rec out = rec_reduce(lane < kConsumerWarps ? ctl.wrec[fs][lane] : no_rec(), rs.argmax, rs.c);
        if (lane == 0) {
            ctl.wcnt[fs] = 0;
            Rec* dst = (loc.kind == 0 ? rec_t() : rec_d()) + loc.slot;
            *dst = out;
            if (share && !post(loc.req, share)) set_abort(a.d_status);
        }
    }

    // This thread's NV vectors of a stage (nvec 16-byte vectors; -inf past
    // them): a phase-1 stage (kVecPerThread) or one draw-sized chunk of a row
    // (kVecPerThread / 2, early exit). Full stages take a path without
    // per-vector bounds. Callers release the stage as soon as these are in
    // registers and fold them afterwards (fold_vectors), so that a ring slot
    // is held only for the copy, not for the arithmetic.
    template <int NV = kVecPerThread>
    __device__ __forceinline__ static void load_stage(const char* sm, int nvec, uint4 (&v)[NV]) {
        const int t = threadIdx.x;
        if (nvec == NV * kConsumers) {
#pragma unroll
            for (int k = 0; k < NV; ++k)
                v[k] = *reinterpret_cast<const uint4*>(sm + static_cast<size_t>(t + k * kConsumers) * 16);
        } else {
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int vi = t + k * kConsumers;
                if (vi < nvec)
                    v[k] = *reinterpret_cast<const uint4*>(sm + static_cast<size_t>(vi) * 16);
                else if (DT == SV_BF16)
                    v[k] = make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
                else
                    v[k] = make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
            }
        }
    }

    template <int NV>
    __device__ __forceinline__ void fold_vectors(RowState& rs, const uint4 (&v)[NV], long long e0) const {
        const int t = threadIdx.x;
        float tmax;
        if (DT == SV_BF16) {
            uint32_t m2 = bf16x2_max_nan(bf16x2_max_nan(v[0].x, v[0].y), bf16x2_max_nan(v[0].z, v[0].w));
#pragma unroll
            for (int k = 1; k < NV; ++k)
                m2 = bf16x2_max_nan(m2, bf16x2_max_nan(bf16x2_max_nan(v[k].x, v[k].y),
                                                       bf16x2_max_nan(v[k].z, v[k].w)));
            tmax = f32_max_nan(bf16x2_lo(m2), bf16x2_hi(m2));
        } else {
            tmax = neg_inf();
#pragma unroll
            for (int k = 0; k < NV; ++k)
                tmax = f32_max_nan(tmax, f32_max_nan(f32_max_nan(__uint_as_float(v[k].x), __uint_as_float(v[k].y)),
                                                     f32_max_nan(__uint_as_float(v[k].z), __uint_as_float(v[k].w))));
        }
        if (bad_logit(tmax)) {
            rs.bad |= kBadData;
            return;
        }
        if (tmax == neg_inf()) return;
        if (rs.argmax) {
            if (tmax > rs.m) {
                // first position of tmax among this thread's elements (increasing index)
                int found = -1;
#pragma unroll
                for (int k = NV - 1; k >= 0; --k) {
                    const uint32_t w4[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
                    for (int q = 3; q >= 0; --q) {
                        if (DT == SV_BF16) {
                            if (bf16x2_hi(w4[q]) == tmax) found = (t + k * kConsumers) * 8 + 2 * q + 1;
                            if (bf16x2_lo(w4[q]) == tmax) found = (t + k * kConsumers) * 8 + 2 * q;
                        } else {
                            if (__uint_as_float(w4[q]) == tmax) found = (t + k * kConsumers) * 4 + q;
                        }
                    }
                }
                rs.m = tmax;
                rs.idx = static_cast<int>(e0) + found;
            }
            return;
        }
        const float c = rs.c;
        if (tmax > rs.m) {
            const float mc = scaled_max(tmax, c);
            // beyond the anchored form's range (or c overflowed): flagged, and
            // recomputed in the plain form by the warp that decides the request
            if (!(fabsf(mc) < 8388608.0f)) rs.bad |= kBadPlain;
            rs.s = (rs.m == neg_inf()) ? 0.0f : __fmul_rn(rs.s, ex2(__fsub_rn(rs.mc, mc)));
            rs.m = tmax;
            rs.mc = mc;
        }
        // Pairs of logits in packed binary32 arithmetic: fma.rn.f32x2 and
        // add.rn.f32x2 round each lane exactly as two scalar instructions would.
        const unsigned long long cc = f2_pack(c, c), nmc = f2_pack(-rs.mc, -rs.mc);
        unsigned long long acc = f2_pack(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const uint32_t w4[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
            for (int q = 0; q < 4; q += (DT == SV_BF16 ? 1 : 2)) {
                unsigned long long x2;
                if (DT == SV_BF16)
                    x2 = f2_pack_bits(prmt(w4[q], 0x1044u), prmt(w4[q], 0x3244u));
                else
                    x2 = f2_pack_bits(w4[q], w4[q + 1]);
                float d0, d1;
                f2_unpack(f2_fma(x2, cc, nmc), d0, d1);
                acc = f2_add(acc, f2_pack(ex2(d0), ex2(d1)));
            }
        }
        float a0, a1;
        f2_unpack(acc, a0, a1);
        rs.s = __fadd_rn(rs.s, __fadd_rn(a0, a1));
    }

    // ---- acceptance scan: merge of a row's pieces, in slice and warp order.
    // The records of a row's first kPrePieces pieces are read first
    // (row_load) and merged once the request's temperature is known
    // (row_combine); a row over more slices reads the rest then.
    // Row kinds: 0 a target row of a T > 0 request, 2 a target row of another
    // request (`row` virtual in both), 1 a draft row (compacted).
    struct RowRaw {
        uint4 x[kPrePieces];
        int i0, i1;  // the row's first and last slice
    };
    __device__ const Slicing& row_slicing(int kind) const { return ctl.sl[kind == 1 ? 1 : kind == 2 ? 2 : 0]; }
    // The record of `row`'s piece in slice i.
    __device__ const uint4* piece_rec(int kind, int i, long long row) const {
        const Rec* base = kind == 1 ? rec_d() : rec_t() + (kind == 2 ? ctl.nwave * G : 0);
        return reinterpret_cast<const uint4*>(base + row + i);
    }
    __device__ void row_load(int kind, long long row, RowRaw& rr) const {
        const Slicing& sl = row_slicing(kind);
        const long long e0 = row * a.V - (kind == 2 ? ctl.sl[0].E : 0ll);
        rr.i0 = slice_of(sl, e0);
        rr.i1 = slice_of(sl, e0 + a.V - 1);
#pragma unroll
        for (int q = 0; q < kPrePieces; ++q)
            rr.x[q] = rr.i0 + q <= rr.i1 ? __ldcg(piece_rec(kind, rr.i0 + q, row)) : make_uint4(0u, 0u, 0u, kNoPiece);
    }
    __device__ Rec row_combine(int kind, long long row, const RowRaw& rr, bool argmax, float c) const {
        MaxSumA ms{neg_inf(), 0.0f};
        ArgMax am = argmax_empty();
        int bad = 0;
        auto take = [&](const uint4& x) {
            if (x.w == kNoPiece) return;
            const float m = __uint_as_float(x.x), s = __uint_as_float(x.y);
            bad |= static_cast<int>(x.w);
            if (argmax)
                am = argmax_merge(am, ArgMax{m, static_cast<int32_t>(x.z)});
            else
                ms = maxsum_merge_a(ms, MaxSumA{m, s}, c);
        };
#pragma unroll
        for (int q = 0; q < kPrePieces; ++q) take(rr.x[q]);
        for (int i = rr.i0 + kPrePieces; i <= rr.i1; ++i) take(__ldcg(piece_rec(kind, i, row)));
        Rec out;
        if (argmax)
            out = {am.v, 0.0f, am.i == 0x7fffffff ? 0 : am.i, (bad || am.v == neg_inf()) ? kBadData : 0};
        else
            out = {ms.m, ms.s, -1, (bad & kBadPlain) | (((bad & kBadData) || ms.m == neg_inf()) ? kBadData : 0)};
        return out;
    }
    __device__ Rec merge_row(int kind, long long row, bool argmax, float c) const {
        RowRaw rr;
        row_load(kind, row, rr);
        return row_combine(kind, row, rr, argmax, c);
    }

    // Acceptance scan of request b on one warp (the finisher); `st` is its
    // shared scratch of 2 gamma + 1 row records.
    __device__ void verify_request(int b, Rec* st) const {
        const int lane = threadIdx.x & 31, GM = a.gamma, V = a.V;
        const int k = ctl.kmap[b];  // compacted index of a T > 0 request, else negative
        // the request's place in the virtual order of target rows, and their kind
        const int vpos = k >= 0 ? k : ctl.n_samp - k - 1;
        const int tkind = k >= 0 ? 0 : 2;
        const int32_t* tok = a.tokens + static_cast<size_t>(b) * GM;
        const bool onehot = a.onehot;
        // The reads come in two rounds. First everything that depends on no
        // other read: the temperature, the draw's uniform, the proposal
        // count, this lane's token and uniform, and the first piece records
        // of row `lane` (rows numbered target 0..gamma, then draft
        // gamma+1..2 gamma; rows from 32 on are read in the second round).
        // Then the logits at this lane's token, which need only the token
        // (read even when the request turns out greedy).
        const float T = a.temperature[b];
        const int us_bits = __float_as_int(a.u_sample[b]);  // the draw's uniform
        // proposals of this request: gamma, or num_draft[b] for one-hot proposals
        // (whose rows past it take no part)
        const int kb = onehot && a.num_draft ? a.num_draft[b] : GM;
        const int x_l = lane < GM ? tok[lane] : -1;
        const float u_l = lane < GM ? a.u_accept[static_cast<size_t>(b) * GM + lane] : 0.0f;
        const int nrows_max = (k >= 0 && !onehot) ? 2 * GM + 1 : GM + 1;
        auto row_of = [&](int r) -> long long {
            return r <= GM ? static_cast<long long>(vpos) * (GM + 1) + r : static_cast<long long>(k) * GM + (r - GM - 1);
        };
        auto kind_of = [&](int r) { return r <= GM ? tkind : 1; };
        RowRaw raw0;
        if (lane < nrows_max) row_load(kind_of(lane), row_of(lane), raw0);
        float lt_l = 0.0f, ld_l = 0.0f;
        if (!a.tree && x_l >= 0 && x_l < V) {
            lt_l = load_logit<DT>(a.target, (static_cast<size_t>(b) * (GM + 1) + lane) * V + x_l);
            if (k >= 0 && !onehot) ld_l = load_logit<DT>(a.draft, (static_cast<size_t>(b) * GM + lane) * V + x_l);
        }
        const bool t_ok = (T >= 0.0f) && (T < pos_inf());
        const bool greedy = t_ok && T == 0.0f;
        const bool samp = sampled(T);
        const Scale sc = samp ? temp_scale(T) : Scale{0.0f, 0.0f};
        const float c = sc.c;
        const bool range_ok = t_ok && kb >= 0 && kb <= GM;
        int bad = range_ok ? 0 : 1;
        const int np = range_ok ? kb : 0;
        for (int i = lane; i < np; i += 32) {
            const int x = i < 32 ? x_l : tok[i];
            if (x < 0 || x >= V) bad = 1;
            if (a.tree) {  // node i + 1's parent is an earlier node
                const int par = a.parents[static_cast<size_t>(b) * GM + i];
                if (par < 0 || par > i) bad = 1;
            }
        }
        const int nrows = !range_ok ? 0 : (samp && !onehot ? 2 * GM + 1 : np + 1);
        int plain = 0;  // a row flagged kBadPlain
        for (int r = lane; r < nrows; r += 32) {
            const int kind = kind_of(r);
            const bool am = r <= GM && !samp;
            Rec x;
            if (r == lane)
                x = row_combine(kind, row_of(r), raw0, am, c);
            else
                x = merge_row(kind, row_of(r), am, c);
            st[r] = x;
            if (x.bad & kBadData) bad = 1;
            if (x.bad & kBadPlain) plain = 1;
        }
        bad = __any_sync(0xffffffffu, bad);
        __syncwarp();
        if (!bad && __any_sync(0xffffffffu, plain)) recompute_plain(b, st, nrows, sc);
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
            __syncwarp();
            if (lane == 0) {
                a.out_num_accepted[b] = -1;
                if (a.d_status) atomicOr(a.d_status, SV_STATUS_BAD_REQUEST);
                if (dbg.kind) dbg.kind[b] = kKindInvalid;
                if (dbg.w_total) dbg.w_total[b] = nan("");
                if (k >= 0) {  // its draw job is published as invalid (no items, no search)
                    jobs()[k].kind = kKindInvalid;
                    publish(k);
                }
            }
            return;
        }
        for (int j = lane; j <= GM; j += 32) {
            const size_t r = static_cast<size_t>(b) * (GM + 1) + j;
            const bool read = j <= np;  // one-hot: rows past the proposals are not part of the request
            if (dbg.max_target) dbg.max_target[r] = read ? st[j].m : nanf("");
            if (dbg.lse_target)
                dbg.lse_target[r] = (greedy || !read) ? nan("") : lse_from_stats(ms_of(st[j]), sc, T);
            if (dbg.argmax_target) dbg.argmax_target[r] = (greedy && read) ? st[j].idx : -1;
        }
        for (int j = lane; j < GM; j += 32) {
            const size_t r = static_cast<size_t>(b) * GM + j;
            const bool draft = !greedy && !onehot;
            if (dbg.max_draft) dbg.max_draft[r] = draft ? st[GM + 1 + j].m : nanf("");
            if (dbg.lse_draft)
                dbg.lse_draft[r] = draft ? lse_from_stats(ms_of(st[GM + 1 + j]), sc, T) : nan("");
        }
        const ScanPre pre{x_l, u_l, lt_l, ld_l, us_bits};
        Job j;
        const int* set = nullptr;  // a tree draw's excluded tokens
        if (a.tree ? tree_walk(b, k, st, greedy, sc, np, j, set) : linear_scan(b, st, greedy, sc, np, pre, j))
            finish_job(k, j, set);
    }

    // What the acceptance scan reads before it knows the temperature: lane's
    // token, uniform and the logits at the token (rows lane < 32), and the
    // request's draw uniform.
    struct ScanPre {
        int x_l;
        float u_l, lt_l, ld_l;
        int us_bits;  // u_sample[b]
    };

    // The left-to-right scan of request b (not a tree): writes the accepted
    // tokens and count; for a draw fills job j and returns true.
    __device__ bool linear_scan(int b, const Rec* st, bool greedy, const Scale& sc, int np, const ScanPre& pre,
                                Job& j) const {
        const int lane = threadIdx.x & 31, GM = a.gamma, V = a.V;
        const bool onehot = a.onehot;
        const int32_t* tok = a.tokens + static_cast<size_t>(b) * GM;
        const sv_debug_out& dbg = a.dbg;
        int32_t* out = a.out_tokens + static_cast<size_t>(b) * (GM + 1);
        const int x_l = pre.x_l;
        const float u_l = pre.u_l, lt_l = pre.lt_l, ld_l = pre.ld_l;
        // first failing position over all lanes (gamma may exceed 32)
        int n = np;
        for (int base = 0; base < np; base += 32) {
            const int i = base + lane;
            bool fail = false;
            if (i < np) {
                const int x = base == 0 ? x_l : tok[i];
                if (greedy) {
                    fail = x != st[i].idx;
                } else {
                    const size_t tr = static_cast<size_t>(b) * (GM + 1) + i;
                    const size_t dr = static_cast<size_t>(b) * GM + i;
                    const bool pre_loaded = base == 0;
                    const float lt = pre_loaded ? lt_l : load_logit<DT>(a.target, tr * V + x);
                    const float u = pre_loaded ? u_l : a.u_accept[dr];
                    if (dbg.p_x) dbg.p_x[dr] = prob_from_stats(lt, ms_of(st[i]), sc);
                    if (onehot) {
                        // q(x) = 1: the draft side of the test is a row whose only
                        // logit is 0 (max 0, sum 1)
                        if (dbg.q_x) dbg.q_x[dr] = 1.0;
                        fail = !accept_from_logits(lt, 0.0f, ms_of(st[i]), MaxSum{0.0f, 1.0f, 0}, sc, u);
                    } else {
                        const float ld = pre_loaded ? ld_l : load_logit<DT>(a.draft, dr * V + x);
                        if (dbg.q_x) dbg.q_x[dr] = prob_from_stats(ld, ms_of(st[GM + 1 + i]), sc);
                        fail = !accept_from_logits(lt, ld, ms_of(st[i]), ms_of(st[GM + 1 + i]), sc, u);
                    }
                }
            }
            const unsigned ball = __ballot_sync(0xffffffffu, fail);
            if (n == np && ball) n = base + __ffs(ball) - 1;
        }
        // positions after the first rejection, or not proposed (all of them at
        // T = 0), are not evaluated
        for (int i = lane; i < GM; i += 32)
            if (greedy || i > n || i >= np) {
                const size_t dr = static_cast<size_t>(b) * GM + i;
                if (dbg.p_x) dbg.p_x[dr] = nan("");
                if (dbg.q_x) dbg.q_x[dr] = nan("");
            }
        for (int j = lane; j <= GM; j += 32) {
            if (j < n)
                out[j] = j < 32 ? x_l : tok[j];  // lane j read token j in the first round
            else if (j == n)
                out[j] = greedy ? st[n].idx : -1;  // the draw fills it in phase 2
            else
                out[j] = -1;
        }
        // the count is written once the request is final: here at T = 0, else
        // with the drawn token (until then it stays -1, see prologue)
        if (lane == 0 && greedy) {
            a.out_num_accepted[b] = n;
            if (dbg.kind) dbg.kind[b] = kKindGreedy;
            if (dbg.w_total) dbg.w_total[b] = nan("");
        }
        if (greedy) return false;
        j.b = b;
        j.n = n;
        j.slot = n;
        j.pad = pre.us_bits;  // the draw's uniform
        DrawParams& d = j.d;
        d.excl = -1;
        if (n < np && !onehot) {
            const MaxSum sq = ms_of(st[GM + 1 + n]);
            draw_rows(d, kKindResidual, ms_of(st[n]), &sq, sc);
            d.fix = kFixResidual;
        } else {
            // the extra token (n = np), or the residual of a one-hot
            // proposal: p_n without x_n, unnormalised weights
            draw_rows(d, n < np ? kKindResidualOnehot : kKindBonus, ms_of(st[n]), nullptr, sc);
            d.excl = n < np ? tok[n] : -1;
            d.fix = kFixTarget;
        }
        j.kind = d.base_kind();
        if (lane == 0 && dbg.kind) dbg.kind[b] = j.kind == kKindResidualOnehot ? kKindResidual : j.kind;
        return true;
    }

    // Lane 0 publishes draw job k of request j.b. An anchored draw goes to the
    // draw stream (items, then the owner's search); a plain draw (large logits
    // or a tiny T) is drawn here by the whole warp and published as done, so
    // that the producers and the owner pass over it. `set`: a tree draw's
    // excluded tokens.
    __device__ void finish_job(int k, Job j, const int* set) const {
        const int lane = threadIdx.x & 31;
        if (j.d.plain()) {
            plain_draw_warp(j, set);
            j.kind = kKindDrawn;
        }
        if (lane == 0) {
            jobs()[k] = j;
            publish(k);
        }
    }

    // ---- the plain form on one warp. The consumers fold every row in the
    // anchored form and flag (kBadPlain) a row whose anchor leaves its range
    // (logits beyond about 5.8e6 T, or c = log2(e)/T overflowed); the warp
    // that decides the request recomputes such rows here, off the streams,
    // and draws over them itself (sv_common.cuh states both forms).

    // Plain statistics of row `row` of `base`: max m and s = sum 2^((l - m) c),
    // each lane over the logits lane, lane + 32, ... in order, then the lanes
    // merged in a fixed order.
    __device__ MaxSum plain_row_warp(const void* base, long long row, const Scale& sc) const {
        const int lane = threadIdx.x & 31, V = a.V;
        const long long e0 = row * V;
        MaxSum st{neg_inf(), 0.0f, 1};
        for (int x = lane; x < V; x += 128) {
            float l[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) l[q] = x + 32 * q < V ? load_logit<DT>(base, e0 + x + 32 * q) : neg_inf();
#pragma unroll
            for (int q = 0; q < 4; ++q) maxsum_add(st, l[q], sc);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            MaxSum ot{__shfl_xor_sync(0xffffffffu, st.m, o), __shfl_xor_sync(0xffffffffu, st.s, o), 1};
            st = maxsum_merge(st, ot, sc);
        }
        return st;
    }

    // Rows 0..nrows-1 of request b (target rows 0..gamma, then draft rows) whose
    // records are flagged kBadPlain get plain statistics (whole warp).
    __device__ void recompute_plain(int b, Rec* st, int nrows, const Scale& sc) const {
        const int lane = threadIdx.x & 31, GM = a.gamma;
        for (int base = 0; base < nrows; base += 32) {
            unsigned flagged = __ballot_sync(0xffffffffu, base + lane < nrows && (st[base + lane].bad & kBadPlain));
            while (flagged) {
                const int r = base + __ffs(flagged) - 1;
                flagged &= flagged - 1;
                const MaxSum ms = r <= GM ? plain_row_warp(a.target, static_cast<long long>(b) * (GM + 1) + r, sc)
                                          : plain_row_warp(a.draft, static_cast<long long>(b) * GM + (r - GM - 1), sc);
                __syncwarp();
                if (lane == 0) st[r] = Rec{ms.m, ms.s, kRecPlain, 0};
                __syncwarp();
            }
        }
    }

    // The draw of a plain job on one warp: weights from sv_common.cuh in their
    // plain form, summed in runs of 32 tokens (lane l of each step of 1024
    // tokens takes run l), each run in binary32 in index order and converted
    // to fixed point, so prefix sums are exact; the token is the smallest k
    // with C_k > u W. Residual weights that are all zero fall back to p.
    __device__ void plain_draw_warp(const Job& jb, const int* set) const {
        const int lane = threadIdx.x & 31, V = a.V, GM = a.gamma;
        constexpr int RUN = 32;
        DrawParams d = jb.d;
        int kind = jb.kind;
        const long long trow = (static_cast<long long>(jb.b) * (GM + 1) + jb.n) * V;
        const long long drow = (static_cast<long long>(jb.b) * GM + (jb.n < GM ? jb.n : 0)) * V;
        auto weight = [&](int e) -> float {
            const float lt = load_logit<DT>(a.target, trow + e);
            if (kind == kKindResidual) return weight_residual(lt, load_logit<DT>(a.draft, drow + e), d);
            if (kind == kKindResidualOnehot && e == d.excl) return 0.0f;
            if (kind == kKindResidualTree && in_set(e, set, d.excl)) return 0.0f;
            return weight_target(lt, d);
        };
        auto run_fixed = [&](int r0) -> unsigned long long {
            float sum = 0.0f;
            for (int e = r0; e < min(V, r0 + RUN); ++e) sum = __fadd_rn(sum, weight(e));
            return r0 < V ? to_fixed(sum, d.fix) : 0ull;
        };
        auto total_of = [&]() {
            unsigned long long tot = 0;
            for (int s0 = 0; s0 < V; s0 += 32 * RUN) tot += warp_sum_u64(run_fixed(s0 + lane * RUN));
            return tot;
        };
        unsigned long long total = total_of();
        if (total == 0ull) {  // residual weights rounded to zero everywhere: draw from p_n
            kind = kKindBonus;
            d.fix = kFixTarget;
            total = total_of();
        }
        const unsigned long long t = scale_uniform(__int_as_float(jb.pad), total);
        unsigned long long before = 0;
        int token = -1;
        for (int s0 = 0; s0 < V && token < 0; s0 += 32 * RUN) {
            const int r0 = s0 + lane * RUN;
            const unsigned long long q = run_fixed(r0);
            unsigned long long incl = q;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const unsigned long long start = before + incl - q;
            const unsigned hit = __ballot_sync(0xffffffffu, q > 0 && start <= t && t < start + q);
            if (hit) {
                int mine = -1;
                if (lane == __ffs(hit) - 1) {
                    float part = 0.0f;
                    int last_pos = -1;
                    for (int e = r0; e < min(V, r0 + RUN) && mine < 0; ++e) {
                        const float w = weight(e);
                        part = __fadd_rn(part, w);
                        if (w > 0.0f) last_pos = e;
                        if (start + to_fixed(part, d.fix) > t) mine = e;
                    }
                    if (mine < 0) mine = last_pos;  // cannot happen: the run's total passes t
                }
                token = __shfl_sync(0xffffffffu, mine, __ffs(hit) - 1);
            }
            before += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            a.out_tokens[static_cast<size_t>(jb.b) * (GM + 1) + jb.slot] = token >= 0 ? token : V - 1;
            a.out_num_accepted[jb.b] = jb.slot;  // the request is final
            if (a.dbg.w_total)
                a.dbg.w_total[jb.b] = kind == kKindResidual ? static_cast<double>(total) * kFixResidualInv
                                                            : static_cast<double>(total) * kFixTargetInv *
                                                                  static_cast<double>(d.isp);
        }
    }

    // Tree walk of request b (rows' statistics in st; np proposal nodes).
    // At node u the children (the nodes whose parent is u) are tried in index
    // order; child c is accepted with min(1, p'(x_c)), p' being p_u without
    // the tokens of the children rejected so far, renormalised, and an
    // accepted child becomes u. When every child is rejected (or u is a
    // leaf) the last token is drawn from p' of u: its excluded tokens go to
    // the job's set. At T = 0 the first child whose token is the argmax of
    // p_u is followed. The test is made in binary64 on lane 0, as the
    // one-block-per-request kernel makes it.
    __device__ bool tree_walk(int b, int k, const Rec* st, bool greedy, const Scale& c, int np, Job& j,
                              const int*& set_out) const {
        const int lane = threadIdx.x & 31, GM = a.gamma, V = a.V;
        const sv_debug_out& dbg = a.dbg;
        int32_t* out = a.out_tokens + static_cast<size_t>(b) * (GM + 1);
        for (int i = lane; i < GM; i += 32) {
            const size_t dr = static_cast<size_t>(b) * GM + i;
            if (dbg.p_x) dbg.p_x[dr] = nan("");  // children never tried
            if (dbg.q_x) dbg.q_x[dr] = nan("");
            if (a.out_nodes) a.out_nodes[dr] = -1;
        }
        for (int j = lane; j <= GM; j += 32) out[j] = -1;
        __syncwarp();
        const int32_t* tok = a.tokens + static_cast<size_t>(b) * GM;
        const int32_t* par = a.parents + static_cast<size_t>(b) * GM;
        const float* ua = a.u_accept + static_cast<size_t>(b) * GM;
        int* set = greedy ? nullptr : jobset() + static_cast<size_t>(k) * GM;
        int u = 0, n = 0, ne = 0;
        while (lane == 0) {  // the walk, on lane 0
            int next = -1;
            if (greedy) {
                const int am = st[u].idx;
                for (int cn = 1; cn <= np && next < 0; ++cn)
                    if (par[cn - 1] == u && tok[cn - 1] == am) next = cn;
                if (next < 0) {
                    out[n] = am;
                    break;
                }
            } else {
                const size_t tr = static_cast<size_t>(b) * (GM + 1) + u;
                double R = 0.0;  // p_u of the rejected children
                ne = 0;
                for (int cn = 1; cn <= np && next < 0; ++cn) {
                    if (par[cn - 1] != u) continue;
                    const int x = tok[cn - 1];
                    const bool seen = in_set(x, set, ne);
                    const float lx = load_logit<DT>(a.target, tr * V + x);
                    const double px = seen ? 0.0 : prob_from_stats(lx, ms_of(st[u]), c);
                    const double rest = 1.0 - R;
                    const double alpha = rest > 0.0 ? fmin(1.0, px / rest) : 0.0;
                    const size_t dr = static_cast<size_t>(b) * GM + (cn - 1);
                    if (dbg.p_x) dbg.p_x[dr] = px;
                    if (dbg.q_x) dbg.q_x[dr] = 1.0;
                    // u = 0 accepts whenever p'(x) > 0, also where it underflows
                    if (ua[cn - 1] < alpha || (ua[cn - 1] == 0.0f && !seen && rest > 0.0 && lx > neg_inf())) {
                        next = cn;
                    } else if (!seen) {
                        set[ne++] = x;
                        R += px;
                    }
                }
                if (next < 0) break;
            }
            out[n] = tok[next - 1];
            if (a.out_nodes) a.out_nodes[static_cast<size_t>(b) * GM + n] = next;
            ++n;
            u = next;
        }
        if (lane == 0) {
            if (greedy) {
                a.out_num_accepted[b] = n;
                if (dbg.kind) dbg.kind[b] = kKindGreedy;
                if (dbg.w_total) dbg.w_total[b] = nan("");
            } else if (dbg.kind) {
                dbg.kind[b] = ne > 0 ? kKindResidual : kKindBonus;
            }
        }
        if (greedy) return false;
        u = __shfl_sync(0xffffffffu, u, 0);
        n = __shfl_sync(0xffffffffu, n, 0);
        ne = __shfl_sync(0xffffffffu, ne, 0);
        j.b = b;
        j.n = u;  // the draw's row: the last node
        j.slot = n;
        j.pad = __float_as_int(a.u_sample[b]);
        DrawParams& d = j.d;
        draw_rows(d, ne > 0 ? kKindResidualTree : kKindBonus, ms_of(st[u]), nullptr, c);
        d.excl = ne > 0 ? ne : -1;
        d.fix = kFixTarget;
        j.kind = d.base_kind();
        __syncwarp();  // lane 0's set, before the other lanes read it
        set_out = set;  // publish's release store also orders the set before the job
        return true;
    }

    // A run is kTPT consecutive tokens, 64 bytes, held packed as 4 vectors of
    // kTPV tokens. Its weight sum is defined vector by vector: S_q adds the
    // weights of vector q in index order, and the run total is
    // ((S_0 + S_1) + S_2) + S_3. The token search walks the same order, so
    // the prefix at a run's last token is the total the stream pass stored.
    using Run = uint4[4];
    static constexpr int kTPV = 16 / ES;  // tokens per 16-byte vector

    // The weights of one vector's tokens (target vt, draft vd). The exponent
    // arguments l c - mc are formed pair by pair with fma.rn.f32x2 (each lane
    // rounded as a scalar fma), so every weight equals weight_residual or
    // weight_target of that token.
    // `set` (shared memory): the tokens a tree residual excludes, d.excl of
    // them; unused by the other kinds.
    __device__ static __forceinline__ void vec_weights(const uint4& vt, const uint4& vd, const DrawParams& d,
                                                       int kind, int first, float (&w)[kTPV],
                                                       const int* set = nullptr) {
        const uint32_t t4[4] = {vt.x, vt.y, vt.z, vt.w};
        const uint32_t d4[4] = {vd.x, vd.y, vd.z, vd.w};
        const unsigned long long cc = f2_pack(d.c, d.c), nmp = f2_pack(-d.mcp, -d.mcp);
#pragma unroll
        for (int i = 0; i < kTPV / 2; ++i) {
            const unsigned long long xt = DT == SV_BF16 ? f2_pack_bits(prmt(t4[i], 0x1044u), prmt(t4[i], 0x3244u))
                                                        : f2_pack_bits(t4[2 * i], t4[2 * i + 1]);
            float e0, e1;
            f2_unpack(f2_fma(xt, cc, nmp), e0, e1);
            if (kind == kKindResidual) {
                const unsigned long long xd = DT == SV_BF16
                                                  ? f2_pack_bits(prmt(d4[i], 0x1044u), prmt(d4[i], 0x3244u))
                                                  : f2_pack_bits(d4[2 * i], d4[2 * i + 1]);
                float g0, g1;
                f2_unpack(f2_fma(xd, cc, f2_pack(-d.mcq, -d.mcq)), g0, g1);
                // p and q are each rounded to binary32 before the difference:
                // scalar __fmul_rn/__fsub_rn are never merged into a fused
                // multiply-add, so weights that cancel in binary32 are exactly 0
                w[2 * i] = fmaxf(__fsub_rn(__fmul_rn(ex2(e0), d.isp), __fmul_rn(ex2(g0), d.isq)), 0.0f);
                w[2 * i + 1] = fmaxf(__fsub_rn(__fmul_rn(ex2(e1), d.isp), __fmul_rn(ex2(g1), d.isq)), 0.0f);
            } else {
                w[2 * i] = ex2(e0);
                w[2 * i + 1] = ex2(e1);
            }
        }
        if (kind == kKindResidualOnehot) {  // p without the proposed token (first = this vector's first token)
            const int rel = d.excl - first;
#pragma unroll
            for (int e = 0; e < kTPV; ++e) w[e] = e == rel ? 0.0f : w[e];
        } else if (kind == kKindResidualTree) {  // p without the rejected children's tokens
            for (int i = 0; i < d.excl; ++i) {
                const int rel = set[i] - first;
                if (static_cast<unsigned>(rel) < static_cast<unsigned>(kTPV)) {
#pragma unroll
                    for (int e = 0; e < kTPV; ++e) w[e] = e == rel ? 0.0f : w[e];
                }
            }
        }
    }

    // S_q of one vector: its weights added in index order.
    __device__ static __forceinline__ float vec_sum(const uint4& vt, const uint4& vd, const DrawParams& d, int kind,
                                                    int first, const int* set = nullptr) {
        float w[kTPV];
        vec_weights(vt, vd, d, kind, first, w, set);
        float s = w[0];
#pragma unroll
        for (int e = 1; e < kTPV; ++e) s = __fadd_rn(s, w[e]);
        return s;
    }

    __device__ static __forceinline__ float run_total(const float (&S)[4]) {
        return __fadd_rn(__fadd_rn(__fadd_rn(S[0], S[1]), S[2]), S[3]);
    }

    // S_0..S_3 of a run held in index order; vectors at or past `valid`
    // tokens weigh 0 (rows end on 16-byte boundaries, so a vector is either
    // wholly in the row or wholly past it).
    __device__ static __forceinline__ void run_vec_sums(const Run& vt, const Run& vd, int valid, const DrawParams& d,
                                                        int kind, int first, float (&S)[4], const int* set = nullptr) {
        // all four are computed (straight-line code), then the ones past the
        // row are dropped; `first` is the run's first token
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float x = vec_sum(vt[q], vd[q], d, kind, first + q * kTPV, set);
            S[q] = q * kTPV < valid ? x : 0.0f;
        }
    }

    // Run t of a stage in shared memory, read in rotated order so that the 8
    // lanes of each shared-memory wavefront hit distinct banks: raw[k] is
    // vector (k + r) & 3 with r = (t >> 1) & 3.
    __device__ static __forceinline__ void load_run_smem(const char* sm, int t, Run& raw) {
        const int r = (t >> 1) & 3;
        const uint4* base = reinterpret_cast<const uint4*>(sm + static_cast<size_t>(t) * 64);
#pragma unroll
        for (int k = 0; k < 4; ++k) raw[k] = base[(k + r) & 3];
    }

    // Run total of a run read by load_run_smem: the vector sums are computed
    // in the rotated order and put back in index order (rotate by 2 if r & 2,
    // then by 1 if r & 1; selects on constant indices) before they are added.
    __device__ static __forceinline__ float run_total_rotated(const Run& rt, const Run& rd, int t, int valid,
                                                              const DrawParams& d, int kind, int first,
                                                              const int* set = nullptr) {
        const int r = (t >> 1) & 3;
        float Sr[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            // stale shared memory past the row is dropped
            const float x = vec_sum(rt[k], rd[k], d, kind, first + ((k + r) & 3) * kTPV, set);
            Sr[k] = ((k + r) & 3) * kTPV < valid ? x : 0.0f;
        }
        const bool r2 = (r & 2) != 0, r1 = (r & 1) != 0;
        float m[4], S[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) m[q] = r2 ? Sr[(q + 2) & 3] : Sr[q];
#pragma unroll
        for (int q = 0; q < 4; ++q) S[q] = r1 ? m[(q + 3) & 3] : m[q];
        return run_total(S);
    }

    // run_total_rotated with the draw kind a compile-time constant: one
    // straight-line body per kind, chosen once per stage.
    __device__ static __forceinline__ float run_total_by_kind(const Run& rt, const Run& rd, int t, int valid,
                                                              const DrawParams& d, int kind, int first,
                                                              const int* set) {
        switch (kind) {
            case kKindResidual: return run_total_rotated(rt, rd, t, valid, d, kKindResidual, first, set);
            case kKindResidualOnehot: return run_total_rotated(rt, rd, t, valid, d, kKindResidualOnehot, first, set);
            case kKindResidualTree: return run_total_rotated(rt, rd, t, valid, d, kKindResidualTree, first, set);
            default: return run_total_rotated(rt, rd, t, valid, d, kKindBonus, first, set);
        }
    }

    // A run from global memory starting at element `e` (64-byte aligned in the
    // row); its first `valid` tokens are whole 16-byte vectors because rows
    // end on 16-byte boundaries. The rest is zero.
    __device__ static __forceinline__ void load_run_global(const void* base, long long e, int valid, Run& v) {
        const uint4* p = reinterpret_cast<const uint4*>(static_cast<const char*>(base) + e * ES);
        const int nv = valid * ES / 16;
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] = q < nv ? __ldg(p + q) : make_uint4(0u, 0u, 0u, 0u);
    }

    // Fixed-point weight sum of run r of chunk j of a job, from global memory.
    __device__ __forceinline__ unsigned long long run_fixed_global(long long trow, long long drow, int j, int r,
                                                   const DrawParams& d, int kind, const int* set = nullptr) const {
        const long long e0 = static_cast<long long>(j) * kChunkElems;
        const int cnt = static_cast<int>(min(static_cast<long long>(kChunkElems), a.V - e0));
        const int valid = max(0, min(kTPT, cnt - r * kTPT));
        if (valid <= 0) return 0ull;
        Run vt, vd;
        load_run_global(a.target, trow + e0 + r * kTPT, valid, vt);
        if (kind == kKindResidual) load_run_global(a.draft, drow + e0 + r * kTPT, valid, vd);
        float S[4];
        run_vec_sums(vt, vd, valid, d, kind, static_cast<int>(e0) + r * kTPT, S, set);
        return to_fixed(run_total(S), d.fix);
    }

    // ---- phase 2, search warp of the job's owner: the token of draw job k. The chunk holding
    // floor(u W), then the warp within it, from the stored fixed-point sums;
    // then that warp's 32 runs are re-read and summed exactly as in the
    // streaming pass, and one lane walks its run token by token.
    __device__ void search_job(int k) const {
        constexpr int TPT = kTPT;
        constexpr int CH = kChunkElems;
        const int lane = threadIdx.x & 31;
        const Job* gjobs = jobs();
        const unsigned long long* js = wsums() + static_cast<size_t>(k) * L.NCH * kConsumerWarps;
        // this lane's chunk totals (lane j holds chunks j, j+32, ...; NCH <= 128),
        // loaded together with the job: they depend on k only
        const int nch_lane = (L.NCH + 31) / 32;
        unsigned long long ctot[4];
        unsigned long long wp0[kConsumerWarps];  // per-warp sums of chunk `lane` (kept: the search's next step)
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const int j = h * 32 + lane;
            unsigned long long sum = 0;
            if (h < nch_lane && j < L.NCH) {
                const ulonglong2* p = reinterpret_cast<const ulonglong2*>(js + static_cast<size_t>(j) * kConsumerWarps);
#pragma unroll
                for (int hh = 0; hh < kConsumerWarps / 2; ++hh) {
                    const ulonglong2 x = __ldcg(p + hh);
                    sum += x.x + x.y;
                    if (h == 0) {
                        wp0[2 * hh] = x.x;
                        wp0[2 * hh + 1] = x.y;
                    }
                }
            } else if (h == 0) {
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) wp0[w] = 0ull;
            }
            ctot[h] = sum;
        }
        // a tree draw's excluded tokens, read in the same round (gamma <= 64)
        const int* gset = jobset() + static_cast<size_t>(k) * a.gamma;
        const int set0 = lane < a.gamma ? __ldcg(gset + lane) : 0;
        const int set1 = lane + 32 < a.gamma ? __ldcg(gset + lane + 32) : 0;
        // the job comes from L2: it was written by another block, and a job
        // sharing its cache line may have been read here earlier
        Job jb;
        {
            const int* src = reinterpret_cast<const int*>(gjobs + k);
            int* dst = reinterpret_cast<int*>(&jb);
#pragma unroll
            for (int q = 0; q < static_cast<int>(sizeof(Job) / 4); ++q) dst[q] = __ldcg(src + q);
        }
        if (jb.kind != kKindResidual && jb.kind != kKindBonus && jb.kind != kKindResidualOnehot &&
            jb.kind != kKindResidualTree)
            return;
        if (jb.kind == kKindResidualTree) {
            if (lane < jb.d.excl) ctl.fset[lane] = set0;
            if (lane + 32 < jb.d.excl) ctl.fset[lane + 32] = set1;
            __syncwarp();
        }
        const int* set = ctl.fset;
        DrawParams d = jb.d;
        int kind = jb.kind;
        const long long trow = (static_cast<long long>(jb.b) * (a.gamma + 1) + jb.n) * a.V;
        const long long drow = (static_cast<long long>(jb.b) * a.gamma + jb.n) * a.V;
        // per-warp sums of chunk j (from the draw stream, or recomputed on the fallback)
        bool fallback = false;
        auto warp_part = [&](int j, int w) -> unsigned long long {
            if (!fallback) return __ldcg(js + static_cast<size_t>(j) * kConsumerWarps + w);
            return warp_sum_u64(run_fixed_global(trow, drow, j, w * 32 + lane, d, kind, set));
        };
        // total of chunk j on the fallback, computed by the whole warp
        auto chunk_total_warp = [&](int j) -> unsigned long long {
            unsigned long long s = 0;
            for (int w = 0; w < kConsumerWarps; ++w) s += warp_part(j, w);
            return s;
        };
        unsigned long long total = 0;
#pragma unroll
        for (int h = 0; h < 4; ++h) total += ctot[h];
        total = warp_sum_u64(total);
        if (total == 0ull) {
            // residual weights rounded to zero everywhere: draw from p_n
            fallback = true;
            kind = kKindBonus;
            d.fix = kFixTarget;
            total = 0;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                unsigned long long mine = 0;
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = h * 32 + jj;
                    if (h < nch_lane && j < L.NCH) {
                        const unsigned long long c = chunk_total_warp(j);
                        if (jj == lane) mine = c;
                    }
                }
                ctot[h] = mine;
                total += warp_sum_u64(mine);
            }
        }
        const unsigned long long tt =
            scale_uniform(__int_as_float(jb.pad), total);
        unsigned long long before = 0;
        int jsel = -1;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            if (jsel >= 0 || h >= nch_lane) break;
            const int j0 = h * 32;
            const unsigned long long cs = ctot[h];
            unsigned long long incl = cs;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const unsigned long long st0 = before + incl - cs;
            const unsigned hit = __ballot_sync(0xffffffffu, cs > 0 && st0 <= tt && tt < st0 + cs);
            if (hit) {
                const int src = __ffs(hit) - 1;
                jsel = j0 + src;
                before = __shfl_sync(0xffffffffu, st0, src);
            } else {
                before += __shfl_sync(0xffffffffu, incl, 31);
            }
        }
        if (jsel < 0) jsel = L.NCH - 1;  // cannot happen: tt < total
        // the warp of that chunk: lanes 0..7 hold its per-warp sums (on the
        // fallback warp_part is warp-collective, so every lane calls it)
        unsigned long long part = 0ull;
        if (!fallback && jsel < 32) {
            // held by lane jsel since the first round
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const unsigned long long v = __shfl_sync(0xffffffffu, wp0[w], jsel);
                if (lane == w) part = v;
            }
        } else if (!fallback) {
            if (lane < kConsumerWarps) part = __ldcg(js + static_cast<size_t>(jsel) * kConsumerWarps + lane);
        } else {
            for (int w = 0; w < kConsumerWarps; ++w) {
                const unsigned long long v = warp_part(jsel, w);
                if (lane == w) part = v;
            }
        }
        unsigned long long pincl = part;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, pincl, o);
            if (lane >= o) pincl += y;
        }
        const unsigned long long pst = before + pincl - part;
        const unsigned whit = __ballot_sync(0xffffffffu, part > 0 && pst <= tt && tt < pst + part);
        const int wsel = whit ? __ffs(whit) - 1 : kConsumerWarps - 1;
        before = __shfl_sync(0xffffffffu, pst, wsel);
        // its 32 runs, one per lane, re-read with the weights of the draw stream
        const long long e0 = static_cast<long long>(jsel) * CH;
        const int cnt = static_cast<int>(min(static_cast<long long>(CH), a.V - e0));
        const int vt = wsel * 32 + lane;
        const int valid = max(0, min(TPT, cnt - vt * TPT));
        Run lt, ld;
        if (valid > 0) {
            load_run_global(a.target, trow + e0 + vt * TPT, valid, lt);
            if (kind == kKindResidual) load_run_global(a.draft, drow + e0 + vt * TPT, valid, ld);
        }
        float S[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (valid > 0) run_vec_sums(lt, ld, valid, d, kind, static_cast<int>(e0) + vt * TPT, S, set);
        const unsigned long long q = to_fixed(run_total(S), d.fix);
        unsigned long long x = q;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        const unsigned long long start = before + x - q;
        const bool mine = q > 0 && start <= tt && tt < start + q;
        const unsigned ball = __ballot_sync(0xffffffffu, mine);
        if (mine && lane == __ffs(ball) - 1) {
            // the vector, then the token, whose prefix passes tt: the prefix
            // after vector v is P_{v+1} = P_v + S_v (P_0 = 0), and within vector
            // v it is P_v plus the vector's partial sum
            float P = 0.0f, Pv = 0.0f;
            int vsel = -1;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const float next = __fadd_rn(P, S[v]);
                if (vsel < 0 && S[v] > 0.0f && start + to_fixed(next, d.fix) > tt) {
                    vsel = v;
                    Pv = P;
                }
                P = next;
            }
            int token = -1;
            if (vsel >= 0) {
                const uint4 wt = vsel == 0 ? lt[0] : vsel == 1 ? lt[1] : vsel == 2 ? lt[2] : lt[3];
                const uint4 wd = vsel == 0 ? ld[0] : vsel == 1 ? ld[1] : vsel == 2 ? ld[2] : ld[3];
                float w[kTPV];
                vec_weights(wt, wd, d, kind, static_cast<int>(e0) + vt * TPT + vsel * kTPV, w, set);
                float part = w[0];
                int last_pos = w[0] > 0.0f ? 0 : -1;
                if (start + to_fixed(__fadd_rn(Pv, part), d.fix) > tt) token = 0;
#pragma unroll
                for (int e = 1; e < kTPV; ++e) {
                    part = __fadd_rn(part, w[e]);
                    if (w[e] > 0.0f) last_pos = e;
                    if (token < 0 && start + to_fixed(__fadd_rn(Pv, part), d.fix) > tt) token = e;
                }
                if (token < 0) token = last_pos;  // cannot happen: the vector's last prefix passes tt
                token += vsel * kTPV;
            } else {
                token = valid - 1;  // cannot happen: the run's total passes tt
            }
            a.out_tokens[static_cast<size_t>(jb.b) * (a.gamma + 1) + jb.slot] = static_cast<int>(e0) + vt * TPT + token;
        }
        if (!ball && lane == 0) {
            // cannot happen: the runs partition [0, total) exactly
            a.out_tokens[static_cast<size_t>(jb.b) * (a.gamma + 1) + jb.slot] = a.V - 1;
        }
        __syncwarp();
        if (lane == 0) a.out_num_accepted[jb.b] = jb.slot;  // the request is final
        if (lane == 0 && a.dbg.w_total) {
            const double W = static_cast<double>(total);
            a.dbg.w_total[jb.b] =
                kind == kKindResidual ? W * kFixResidualInv : W * kFixTargetInv * static_cast<double>(d.isp);
        }
    }

    // ================================================================ early exit
    // "Speculative Decoding — Come Accelerare l'Inferenza LLM di 2-3x Senza
    // Perdere Qualità", §Il meccanismo: after the first rejection the later draft
    // tokens are discarded, so their rows need not be read. The work is a list of
    // tasks, each cut into L.NCH chunks of kChunkBytes of a row: the row
    // statistics of one position of one request (its target row, and its draft
    // row for model proposals at T > 0), or one draw. Tasks 0..B-1 are position 0
    // of every request; the owner of a statistics task (block p mod G) decides
    // that position and publishes the request's next task: its next position,
    // or its draw. Producers take items, fixed groups of GRP consecutive
    // chunks of one task (L.NI per task), in publication order; an item's
    // statistics are folded into one record, so that the per-chunk costs (the
    // grab, the task lookup, the cross-warp flush) are paid once per group,
    // while a task's chunks still spread over several blocks.

    // A task's code: type, the statistics flags (kStatsArgmax, kStatsDraft) of
    // a published statistics task, request b < 4096, position; plus one.
    __device__ static int ee_encode(int type, int b, int pos, int sflags = 0) {
        return ((type << 28) | (sflags << 20) | (b << 8) | pos) + 1;
    }

    // Proposals of request b (range-checked by the owner of its position 0).
    __device__ int ee_kb(int b) const { return a.onehot && a.num_draft ? a.num_draft[b] : a.gamma; }

    // One lane: appends a task. A draw task's job is written before it is
    // published (the fence); a statistics task carries nothing its readers need
    // from the publisher (they read the inputs, and the records of its own
    // chunks), so it goes out without waiting for the publisher's earlier
    // stores. The slot is stored after the count's increment has returned.
    // A statistics task travels with its flags and scale, so that the producers
    // that take it need no read of their own before issuing its copies.
    __device__ void ee_publish(int type, int b, int pos, float c = 0.0f, int sflags = 0) const {
        if (type != kTaskStats) __threadfence();
        const unsigned q = atomicAdd(&hdr()->n_pub, 1u);
        if (static_cast<long long>(a.B) + q < static_cast<long long>(L.ee_cap))  // always: at most gamma + 1 per request
            st_relaxed(ee_slot(a.B + static_cast<int>(q)),
                       (static_cast<unsigned long long>(__float_as_uint(c)) << 32) |
                           static_cast<unsigned>(ee_encode(type, b, pos, sflags)));
    }

    // One lane: request b is done (its outputs are written).
    __device__ void ee_finish_request(int b) const {
        (void)b;
        __threadfence();
        atomicAdd(&hdr()->n_fin, 1u);
    }

    // One lane: task slot p will stay empty (every request is finished and the
    // published tasks end before p).
    __device__ bool ee_no_task(int p) const {
        if (p >= L.ee_cap) return true;
        if (ld_relaxed(&hdr()->n_fin) < static_cast<unsigned>(a.B)) return false;
        __threadfence();
        return static_cast<long long>(p) >=
               static_cast<long long>(a.B) + ld_relaxed(&hdr()->n_pub);
    }

    __device__ void start_row_mode(RowState& rs, bool argmax, float c) const {
        rs.argmax = argmax;
        rs.c = c;
        rs.m = neg_inf();
        rs.mc = neg_inf();
        rs.s = 0.0f;
        rs.idx = 0x7fffffff;
        rs.bad = 0;
    }

    // The lanes of a warp reduced to one record (every lane holds it).
    __device__ static Rec warp_rec(const RowState& rs) { return rec_reduce(lane_rec(rs), rs.argmax, rs.c); }

    __device__ static Rec rec_merge(Rec x, const Rec& y, bool argmax, float c) {
        x.bad |= y.bad;
        if (argmax) {
            const ArgMax m = argmax_merge(ArgMax{x.m, x.idx}, ArgMax{y.m, y.idx});
            x.m = m.v;
            x.idx = m.i;
        } else {
            const MaxSumA m = maxsum_merge_a(MaxSumA{x.m, x.s}, MaxSumA{y.m, y.s}, c);
            x.m = m.m;
            x.s = m.s;
        }
        return x;
    }

    // End of a statistics item (group grp of task p, nch chunks): each warp
    // parks its records; the last warp merges the twelve (lane w holding warp
    // w's), writes the item's records and posts its chunks to the finisher.
    __device__ void ee_flush_item(const RowState& rt, const RowState& rd, bool has_draft, unsigned seq, int p,
                                  int grp, unsigned nch) const {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        const Rec t = warp_rec(rt);
        Rec d = t;
        if (has_draft) d = warp_rec(rd);
        const int fs = static_cast<int>(seq % kFlushSlots);
        int last = 0;
        if (lane == 0) {
            ctl.wrec[fs][warp] = t;
            ctl.wrec2[fs][warp] = d;
            __threadfence_block();
            last = atomicAdd(&ctl.wcnt[fs], 1) == kConsumerWarps - 1;
        }
        if (!__shfl_sync(0xffffffffu, last, 0)) return;
        __threadfence_block();
        const Rec ot = rec_reduce(lane < kConsumerWarps ? ctl.wrec[fs][lane] : no_rec(), rt.argmax, rt.c);
        Rec od = ot;
        if (has_draft) od = rec_reduce(lane < kConsumerWarps ? ctl.wrec2[fs][lane] : no_rec(), false, rd.c);
        if (lane == 0) {
            ctl.wcnt[fs] = 0;
            Rec* dst = ee_rec() + (static_cast<size_t>(p) * L.NI + grp) * 2;
            dst[0] = ot;
            dst[1] = od;
            if (!post(p | kJobMsg, nch)) set_abort(a.d_status);
        }
    }

    // Producer warp: items of tasks in publication order, one at a time from the
    // global counter (a task's items then run on as many blocks), each as one
    // stage per chunk, until every request is finished; then the end marker.
    __device__ void ee_produce(Cursor& prod) const {
        const int lane = threadIdx.x & 31;
        volatile int* vabort = &ctl.abort;
        Hdr* h = hdr();
        const int NCH = L.NCH, NI = L.NI, GM = a.gamma;
        constexpr int CH = kChunkElems;
        unsigned next = 0;
        if (lane == 0) next = atomicAdd(&h->next_item, 1u);
        int cur_p = -1;
        int task_flags = 0;  // lane 0: the statistics flags of the current task
        StageDesc desc;  // lane 0's copy of the current task
        desc.k = -1;
        desc.type = -1;
        desc.flags = 0;
        desc.job.b = 0;
        desc.job.n = 0;
        desc.job.kind = 0;
        bool ok = true;
        while (ok && !*vabort) {
            const long long i = __shfl_sync(0xffffffffu, next, 0);
            if (lane == 0) next = atomicAdd(&h->next_item, 1u);  // the next item, in flight meanwhile
            const int p = static_cast<int>(static_cast<unsigned>(i) / static_cast<unsigned>(NI));
            const int grp = static_cast<int>(i) - p * NI;
            if (p != cur_p) {
                int state = 1;  // 1 task known, 0 no more tasks, -1 the wait ran out
                if (lane == 0) {
                    int v = 0;
                    float cs = 0.0f;  // a published statistics task's scale
                    if (p < a.B) {
                        v = ee_encode(kTaskStats, p, 0);
                    } else if (p >= L.ee_cap) {
                        state = 0;
                    } else {
                        const unsigned long long* tp = ee_slot(p);
                        const unsigned long long t0 = global_ns();
                        unsigned long long e;
                        while ((e = ld_relaxed(tp)) == 0ull) {
                            if (ee_no_task(p)) {
                                state = 0;
                                break;
                            }
                            if (*vabort || global_ns() - t0 > a.peer_wait_ns) {
                                state = -1;
                                break;
                            }
                            __nanosleep(64);
                        }
                        v = static_cast<int>(static_cast<unsigned>(e));
                        cs = __uint_as_float(static_cast<unsigned>(e >> 32));
                    }
                    if (state == 1) {
                        v -= 1;
                        const int type = v >> 28, b = (v >> 8) & 0xfff, pos = v & 0xff;
                        desc.k = p;
                        desc.type = type;
                        if (type == kTaskStats) {
                            desc.job.b = b;
                            desc.job.n = pos;
                            desc.job.kind = 0;
                            if (p < a.B) {  // position 0: from the request's inputs
                                const float T = a.temperature[b];
                                const bool samp = sampled(T);
                                const int kb = ee_kb(b);
                                desc.job.d.c = samp ? temp_scale(T).c : 0.0f;
                                task_flags = (samp ? 0 : kStatsArgmax) |
                                             ((samp && !a.onehot && pos < kb && pos < GM) ? kStatsDraft : 0);
                            } else {  // published with its scale and flags
                                desc.job.d.c = cs;
                                task_flags = (v >> 20) & (kStatsArgmax | kStatsDraft);
                            }
                        } else {
                            __threadfence();  // the job, written before its task was published
                            const int* src = reinterpret_cast<const int*>(jobs() + b);
                            int* dst = reinterpret_cast<int*>(&desc.job);
#pragma unroll
                            for (int q = 0; q < static_cast<int>(sizeof(Job) / 4); ++q) dst[q] = __ldcg(src + q);
                            task_flags = 0;
                        }
                    }
                }
                state = __shfl_sync(0xffffffffu, state, 0);
                if (state <= 0) {
                    if (state < 0 && lane == 0) set_abort(a.d_status);
                    break;
                }
                cur_p = p;
            }
            const int type = __shfl_sync(0xffffffffu, desc.type, 0);
            const int flags = __shfl_sync(0xffffffffu, task_flags, 0);
            const int b = __shfl_sync(0xffffffffu, desc.job.b, 0);
            const int pos = __shfl_sync(0xffffffffu, desc.job.n, 0);
            const int kind = __shfl_sync(0xffffffffu, desc.job.kind, 0);
            const long long trow = static_cast<long long>(b) * (GM + 1) + pos;  // pos: the draw's row n for draws
            const long long drow = static_cast<long long>(b) * GM + pos;
            const bool two = type == kTaskStats ? (flags & kStatsDraft) != 0 : kind == kKindResidual;
            const int j0 = grp * L.GRP, j1 = min(NCH, j0 + L.GRP);
            desc.item = grp;
            for (int j = j0; ok && j < j1; ++j) {
                desc.j = j;
                desc.nch = j - j0 + 1;
                desc.flags = flags | (j == j0 ? kItemFirst : 0) | (j == j1 - 1 ? kItemLast : 0);
                const long long e0 = static_cast<long long>(j) * CH;
                const int cnt = static_cast<int>(min(static_cast<long long>(CH), a.V - e0));
                const unsigned bytes = static_cast<unsigned>(cnt * ES);
                const char* src_t = static_cast<const char*>(a.target) + (trow * a.V + e0) * ES;
                if (two)
                    ok = produce(prod, src_t, bytes, static_cast<const char*>(a.draft) + (drow * a.V + e0) * ES,
                                 bytes, &desc);
                else
                    ok = produce(prod, src_t, bytes, nullptr, 0u, &desc);
            }
        }
        if (!ok && lane == 0) set_abort(a.d_status);
        __syncwarp();
        StageDesc end;
        end.job.kind = kEndKind;
        end.k = -1;
        end.j = -1;
        end.type = -1;
        end.flags = 0;
        produce(prod, nullptr, 0u, nullptr, 0u, &end);  // bounded; the consumers' own waits are too
    }

    // Consumer warps: the stages of statistics items and draw items until the
    // end marker. A statistics item's chunks fold into one state; a draw item's
    // chunks each get their per-warp sums. Either posts once, at its last stage.
    __device__ void ee_consume(Cursor& cons) const {
        const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
        constexpr int CH = kChunkElems, TPT = kTPT, NVC = kChunkBytes / 16 / kConsumers;
        unsigned long long* ws_sum = wsums();
        RowState rt, rd;  // the statistics item in progress
        start_row_mode(rt, false, 0.0f);
        start_row_mode(rd, false, 0.0f);
        for (unsigned nitem = 0;;) {
            const int slot = static_cast<int>(cons.it % kStages);
            const char* smt = consume_begin(cons);
            if (!smt) {
                set_abort(a.d_status);
                break;
            }
            const StageDesc ds = ctl.desc[slot];
            if (ds.job.kind == kEndKind) {
                consume_end(cons);
                break;
            }
            const long long e0 = static_cast<long long>(ds.j) * CH;
            const int n = static_cast<int>(min(static_cast<long long>(CH), a.V - e0));
            const unsigned nch = static_cast<unsigned>(ds.nch);  // chunks of the item so far
            if (ds.type == kTaskStats) {
                const bool argmax = (ds.flags & kStatsArgmax) != 0, has_draft = (ds.flags & kStatsDraft) != 0;
                if (ds.flags & kItemFirst) {
                    start_row_mode(rt, argmax, ds.job.d.c);
                    start_row_mode(rd, false, ds.job.d.c);
                }
                uint4 vt[NVC], vd[NVC];
                load_stage<NVC>(smt, n * ES / 16, vt);
                if (has_draft) load_stage<NVC>(smt + kChunkBytes, n * ES / 16, vd);
                consume_end(cons);
                fold_vectors<NVC>(rt, vt, e0);
                if (has_draft) fold_vectors<NVC>(rd, vd, e0);
                if (ds.flags & kItemLast) ee_flush_item(rt, rd, has_draft, nitem++, ds.k, ds.item, nch);
            } else {
                const int valid = max(0, min(TPT, n - t * TPT));
                Run lt, ld;
                if (valid > 0) {
                    load_run_smem(smt, t, lt);
                    if (ds.job.kind == kKindResidual) load_run_smem(smt + kChunkBytes, t, ld);
                }
                consume_end(cons);
                const float run = valid > 0 ? run_total_by_kind(lt, ld, t, valid, ds.job.d, ds.job.kind,
                                                                static_cast<int>(e0) + t * TPT, nullptr)
                                            : 0.0f;
                const unsigned long long wsum = warp_sum_u64(to_fixed(run, ds.job.d.fix));
                if (lane == 0) {
                    ws_sum[(static_cast<size_t>(ds.job.b) * L.NCH + ds.j) * kConsumerWarps + warp] = wsum;
                    if (ds.flags & kItemLast) {
                        const int fs = static_cast<int>(nitem % kFlushSlots);
                        __threadfence_block();
                        if (atomicAdd(&ctl.wcnt[fs], 1) == kConsumerWarps - 1) {
                            __threadfence_block();
                            ctl.wcnt[fs] = 0;
                            if (!post(ds.k | kJobMsg, nch)) set_abort(a.d_status);
                        }
                    }
                }
                if (ds.flags & kItemLast) ++nitem;
            }
        }
    }

    // One lane: the request ends at n (-1: invalid); positions after n are -1,
    // and the checking outputs of the rows not read are NaN / -1. The count
    // is written when the request is final (`final`); a pending draw writes it
    // with its token.
    __device__ void ee_close(int b, int n, int from_row, bool final = true) const {
        const int GM = a.gamma;
        int32_t* out = a.out_tokens + static_cast<size_t>(b) * (GM + 1);
        const sv_debug_out& dbg = a.dbg;
        for (int j = n < 0 ? 0 : n + 1; j <= GM; ++j) out[j] = -1;
        if (final) a.out_num_accepted[b] = n;
        for (int j = from_row; j <= GM; ++j) {
            const size_t r = static_cast<size_t>(b) * (GM + 1) + j;
            if (dbg.max_target) dbg.max_target[r] = nanf("");
            if (dbg.lse_target) dbg.lse_target[r] = nan("");
            if (dbg.argmax_target) dbg.argmax_target[r] = -1;
        }
        for (int j = from_row; j < GM; ++j) {
            const size_t r = static_cast<size_t>(b) * GM + j;
            if (dbg.max_draft) dbg.max_draft[r] = nanf("");
            if (dbg.lse_draft) dbg.lse_draft[r] = nan("");
            if (dbg.p_x) dbg.p_x[r] = nan("");
            if (dbg.q_x) dbg.q_x[r] = nan("");
        }
    }

    // What a position's decision reads besides its rows' records: the request's
    // temperature and proposal count, the proposed token, its two logits and
    // its uniform (lane 0), and the request-wide token checks at position 0
    // (each lane its share). The owner reads them as soon as it knows the task,
    // while the task's chunks are still being read.
    struct EePre {
        float T, lt, ld, u;
        int kb, x, bad;
    };

    __device__ EePre ee_prefetch(int b, int pos) const {
        const int lane = threadIdx.x & 31, GM = a.gamma, V = a.V;
        EePre e;
        e.T = a.temperature[b];
        e.kb = ee_kb(b);
        const bool t_ok = (e.T >= 0.0f) && (e.T < pos_inf());
        const bool samp = sampled(e.T);
        const bool range_ok = t_ok && e.kb >= 0 && e.kb <= GM;
        const int32_t* tok = a.tokens + static_cast<size_t>(b) * GM;
        e.x = -1;
        e.lt = 0.0f;
        e.ld = 0.0f;
        e.u = 0.0f;
        if (lane == 0 && range_ok && pos < e.kb) {
            e.x = tok[pos];
            if (samp && e.x >= 0 && e.x < V) {
                const size_t tr = static_cast<size_t>(b) * (GM + 1) + pos, dr = static_cast<size_t>(b) * GM + pos;
                e.lt = load_logit<DT>(a.target, tr * V + e.x);
                if (!a.onehot) e.ld = load_logit<DT>(a.draft, dr * V + e.x);
                e.u = a.u_accept[dr];
            }
        }
        // request-wide checks at position 0: T, the proposal count, every proposed token
        e.bad = range_ok ? 0 : 1;
        if (pos == 0 && range_ok)
            for (int q = lane; q < e.kb; q += 32) {
                const int y = tok[q];
                if (y < 0 || y >= V) e.bad = 1;
            }
        return e;
    }

    // Search warp: the decision at position pos of request b, from the item
    // records of statistics task p and its prefetched inputs.
    __device__ void ee_decide(int p, int b, int pos, const EePre& e) const {
        const int lane = threadIdx.x & 31, GM = a.gamma, NI = L.NI;
        const float T = e.T;
        const bool t_ok = (T >= 0.0f) && (T < pos_inf());
        const bool samp = sampled(T);
        const Scale sc = samp ? temp_scale(T) : Scale{0.0f, 0.0f};
        const float c = sc.c;
        const int kb = e.kb;
        const bool range_ok = t_ok && kb >= 0 && kb <= GM;
        const bool proposal = range_ok && pos < kb;
        const bool has_draft = samp && !a.onehot && proposal;
        int bad = e.bad;
        // the item records of the position's rows, merged in item order per lane
        // and then across lanes; lane 0's result is used
        const bool argmax = !samp;
        Rec rt{neg_inf(), 0.0f, 0x7fffffff, 0}, rd{neg_inf(), 0.0f, -1, 0};
        bool first = true;
        for (int jj = lane; jj < NI; jj += 32) {
            const uint4* src = reinterpret_cast<const uint4*>(ee_rec() + (static_cast<size_t>(p) * NI + jj) * 2);
            const uint4 vt = __ldcg(src), vd = __ldcg(src + 1);
            const Rec xt{__uint_as_float(vt.x), __uint_as_float(vt.y), static_cast<int32_t>(vt.z), static_cast<int32_t>(vt.w)};
            const Rec xd{__uint_as_float(vd.x), __uint_as_float(vd.y), static_cast<int32_t>(vd.z), static_cast<int32_t>(vd.w)};
            if (first) {
                rt = xt;
                rd = xd;
                first = false;
            } else {
                rt = rec_merge(rt, xt, argmax, c);
                if (has_draft) rd = rec_merge(rd, xd, false, c);
            }
        }
        const bool have = !first;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            Rec ot{__shfl_down_sync(0xffffffffu, rt.m, o), __shfl_down_sync(0xffffffffu, rt.s, o),
                   __shfl_down_sync(0xffffffffu, rt.idx, o), __shfl_down_sync(0xffffffffu, rt.bad, o)};
            Rec od{__shfl_down_sync(0xffffffffu, rd.m, o), __shfl_down_sync(0xffffffffu, rd.s, o),
                   __shfl_down_sync(0xffffffffu, rd.idx, o), __shfl_down_sync(0xffffffffu, rd.bad, o)};
            const bool oh = __shfl_down_sync(0xffffffffu, have ? 1 : 0, o) != 0;
            if ((lane & (2 * o - 1)) == 0 && lane + o < 32 && oh) {
                rt = rec_merge(rt, ot, argmax, c);
                if (has_draft) rd = rec_merge(rd, od, false, c);
            }
        }
        bad = __any_sync(0xffffffffu, bad);
        // rows flagged kBadPlain get plain statistics (whole warp; lane 0's
        // merged records decide)
        {
            const int tb = __shfl_sync(0xffffffffu, rt.bad, 0), db = __shfl_sync(0xffffffffu, rd.bad, 0);
            const bool ok = !bad && !(tb & kBadData) && !(has_draft && (db & kBadData));
            for (int w = 0; w < 2; ++w) {  // the target row, then the draft row
                if (!(ok && (w == 0 ? samp && (tb & kBadPlain) : has_draft && (db & kBadPlain)))) continue;
                const MaxSum ms = plain_row_warp(w == 0 ? a.target : a.draft,
                                                 w == 0 ? static_cast<long long>(b) * (GM + 1) + pos
                                                        : static_cast<long long>(b) * GM + pos,
                                                 sc);
                const Rec r{ms.m, ms.s, kRecPlain, 0};
                if (w == 0)
                    rt = r;
                else
                    rd = r;
            }
        }
        int plain_draw = 0;
        if (lane == 0) plain_draw = ee_decide_lane0(p, b, pos, e, rt, rd, sc, bad);
        if (__shfl_sync(0xffffffffu, plain_draw, 0)) ee_plain_draw(b);
    }

    // A plain draw of request b (its job written by lane 0), made by the whole
    // warp; the request is then finished.
    __device__ void ee_plain_draw(int b) const {
        __syncwarp();
        Job j;
        const int* src = reinterpret_cast<const int*>(jobs() + b);
        int* dst = reinterpret_cast<int*>(&j);
        for (int q = 0; q < static_cast<int>(sizeof(Job) / 4); ++q) dst[q] = src[q];
        plain_draw_warp(j, nullptr);
        __syncwarp();
        if ((threadIdx.x & 31) == 0) ee_finish_request(b);
    }

    // The decision at position pos of request b on lane 0, from the merged
    // records rt (target row) and rd (draft row). Returns 1 when the decision
    // is a plain draw, which the caller's warp then makes (job j); the
    // request's other outputs are written here.
    __device__ int ee_decide_lane0(int p, int b, int pos, const EePre& e, Rec rt, Rec rd, const Scale& sc,
                                   int bad) const {
        const int GM = a.gamma;
        const float T = e.T;
        const bool t_ok = (T >= 0.0f) && (T < pos_inf());
        const bool greedy = t_ok && T == 0.0f;
        const bool samp = sampled(T);
        const float c = sc.c;
        const int kb = e.kb;
        const bool range_ok = t_ok && kb >= 0 && kb <= GM;
        const bool proposal = range_ok && pos < kb;
        const bool has_draft = samp && !a.onehot && proposal;
        const int x = e.x;
        const float lt = e.lt, ld = e.ld, u = e.u;
        (void)p;
        const bool row_bad = (rt.bad & kBadData) || rt.m == neg_inf() ||
                             (has_draft && ((rd.bad & kBadData) || rd.m == neg_inf()));
        int32_t* out = a.out_tokens + static_cast<size_t>(b) * (GM + 1);
        const sv_debug_out& dbg = a.dbg;
        if (bad || row_bad) {
            ee_close(b, -1, 0);
            for (int q = 0; q <= GM; ++q) out[q] = -1;
            if (a.d_status) atomicOr(a.d_status, SV_STATUS_BAD_REQUEST);
            if (dbg.kind) dbg.kind[b] = kKindInvalid;
            if (dbg.w_total) dbg.w_total[b] = nan("");
            ee_finish_request(b);
            return 0;
        }
        {  // this position's checking outputs
            const size_t r = static_cast<size_t>(b) * (GM + 1) + pos;
            if (dbg.max_target) dbg.max_target[r] = rt.m;
            if (dbg.lse_target) dbg.lse_target[r] = greedy ? nan("") : lse_from_stats(ms_of(rt), sc, T);
            if (dbg.argmax_target) dbg.argmax_target[r] = greedy ? (rt.idx == 0x7fffffff ? 0 : rt.idx) : -1;
            if (pos < GM) {
                const size_t q = static_cast<size_t>(b) * GM + pos;
                if (dbg.max_draft) dbg.max_draft[q] = has_draft ? rd.m : nanf("");
                if (dbg.lse_draft) dbg.lse_draft[q] = has_draft ? lse_from_stats(ms_of(rd), sc, T) : nan("");
                if (dbg.p_x) dbg.p_x[q] = (samp && proposal) ? prob_from_stats(lt, ms_of(rt), sc) : nan("");
                if (dbg.q_x)
                    dbg.q_x[q] = (samp && proposal) ? (a.onehot ? 1.0 : prob_from_stats(ld, ms_of(rd), sc)) : nan("");
            }
        }
        if (greedy) {
            const int am = rt.idx == 0x7fffffff ? 0 : rt.idx;
            if (proposal && x == am) {
                out[pos] = am;
                ee_publish(kTaskStats, b, pos + 1, 0.0f, kStatsArgmax);
                return 0;
            }
            out[pos] = am;
            ee_close(b, pos, pos + 1);
            if (dbg.kind) dbg.kind[b] = kKindGreedy;
            if (dbg.w_total) dbg.w_total[b] = nan("");
            ee_finish_request(b);
            return 0;
        }
        if (proposal) {
            const bool acc = a.onehot ? accept_from_logits(lt, 0.0f, ms_of(rt), MaxSum{0.0f, 1.0f, 0}, sc, u)
                                      : accept_from_logits(lt, ld, ms_of(rt), ms_of(rd), sc, u);
            if (acc) {
                out[pos] = x;
                ee_publish(kTaskStats, b, pos + 1, c,
                           (!a.onehot && pos + 1 < kb && pos + 1 < GM) ? kStatsDraft : 0);
                return 0;
            }
        }
        // the draw: the residual at a rejection, or the extra token from row kb
        Job j;
        j.b = b;
        j.n = pos;
        j.slot = pos;
        j.pad = __float_as_int(a.u_sample[b]);
        DrawParams& d = j.d;
        d.excl = -1;
        if (proposal && !a.onehot) {
            const MaxSum sq = ms_of(rd);
            draw_rows(d, kKindResidual, ms_of(rt), &sq, sc);
            d.fix = kFixResidual;
        } else {
            draw_rows(d, proposal ? kKindResidualOnehot : kKindBonus, ms_of(rt), nullptr, sc);
            d.excl = proposal ? x : -1;
            d.fix = kFixTarget;
        }
        j.kind = d.base_kind();
        out[pos] = -1;  // the search (or the plain draw) fills it in
        ee_close(b, pos, pos + 1, false);
        if (dbg.kind) dbg.kind[b] = j.kind == kKindResidualOnehot ? kKindResidual : j.kind;
        jobs()[b] = j;
        if (d.plain()) return 1;  // drawn by the caller's warp
        ee_publish(kTaskDraw, b, pos);
        return 0;
    }

    // Search warp: the next owned task (g, g + G, g + 2G, ...), decided or
    // searched once all its chunks are counted. Lane 0 keeps own_p and the
    // task's code (own_v, 0 until it is published); a statistics task's inputs
    // are prefetched into `pre` (for task pre_p) as soon as its code is known.
    __device__ bool ee_poll_owned(int& own_p, int& own_v, EePre& pre, int& pre_p) const {
        int act_p = -1, act_v = 0, known_p = -1, known_v = 0;
        if ((threadIdx.x & 31) == 0 && own_p < L.ee_cap) {
            if (own_v == 0) {
                if (own_p < a.B) {
                    own_v = ee_encode(kTaskStats, own_p, 0);
                } else {
                    const int v = ld_relaxed(reinterpret_cast<const int*>(ee_slot(own_p)));  // the code
                    if (v) {
                        __threadfence();
                        own_v = v;
                    }
                }
            }
            known_p = own_p;
            known_v = own_v;
            if (own_v != 0 &&
                ld_relaxed(ee_done() + own_p) >= static_cast<unsigned>(L.NCH)) {
                __threadfence();  // the other blocks' item records and chunk sums
                act_p = own_p;
                act_v = own_v;
                own_v = 0;
                own_p += G;
            }
        }
        known_p = __shfl_sync(0xffffffffu, known_p, 0);
        known_v = __shfl_sync(0xffffffffu, known_v, 0);
        act_p = __shfl_sync(0xffffffffu, act_p, 0);
        act_v = __shfl_sync(0xffffffffu, act_v, 0);
        if (known_v != 0 && known_p != pre_p && ((known_v - 1) >> 28) == kTaskStats) {
            const int v = known_v - 1;
            pre = ee_prefetch((v >> 8) & 0xfff, v & 0xff);
            pre_p = known_p;
        }
        if (act_p < 0) return false;
        const int v = act_v - 1, type = v >> 28, b = (v >> 8) & 0xfff, pos = v & 0xff;
        if (type == kTaskStats) {
            ee_decide(act_p, b, pos, pre);  // act_p == pre_p: its code was known above at the latest
            pre_p = -1;
        } else {
            search_job(b);
            __syncwarp();
            if ((threadIdx.x & 31) == 0) ee_finish_request(b);
        }
        __syncwarp();
        return true;
    }
};

template <int DT>
__global__ void __launch_bounds__(kThreads, 1) stream_kernel(Args a, Layout L, char* ws) {
    extern __shared__ __align__(128) char smem[];
    char* stages = smem;
    Ctl& ctl = *reinterpret_cast<Ctl*>(smem + static_cast<size_t>(kStages) * kStageBytes);
    Rec* fin_rows = reinterpret_cast<Rec*>(smem + static_cast<size_t>(kStages) * kStageBytes + sizeof(Ctl));

    using KT = Kern<DT>;
    KT K{a, L, ws, ctl, stages, static_cast<int>(gridDim.x), static_cast<int>(blockIdx.x)};
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const bool producer = warp == kProducerWarp, finisher = warp == kFinisherWarp, searcher = warp == kSearchWarp;
    unsigned long long* ph = reinterpret_cast<unsigned long long*>(a.dbg.phase_ns);
    stamp(ph, 0, t == 0);

    if (t == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl.full[s], 1);
            mbar_init(&ctl.empty[s], kConsumerWarps);
        }
        ctl.abort = 0;
        ctl.n_samp = -1;  // set by the consumers' prologue
        ctl.fq_tail = 0;
        ctl.fq_head = 0;
        ctl.cons_done = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int i = t; i < kMapMax; i += kThreads) {
        ctl.wmap[0][i] = -1;
        ctl.wmap[1][i] = -1;
        ctl.map3[i] = -1;
    }
    for (int i = t; i < kFlushSlots; i += kThreads) ctl.wcnt[i] = 0;
    for (int i = t; i < kQueue; i += kThreads) ctl.fq_seq[i] = 0;
    __syncthreads();

    // ------------------------------------------------------------ finisher
    if (finisher) {
        // a request is scanned by the block whose share completes its 2 gamma + 1
        // rows (gamma + 1 at T = 0); a draw job's chunks are counted here and
        // the job is searched by its owner's search warp
        const unsigned V = static_cast<unsigned>(a.V), GM = static_cast<unsigned>(a.gamma);
        unsigned* req_done = K.req_done();
        unsigned* job_done = K.job_done();
        K.finish(
            [&](int item, unsigned share) {
                if (item & kJobMsg) {
                    // fire and forget: the job's owner polls the count; the
                    // release orders this block's chunk sums before it
                    red_release_add(job_done + (item & ~kJobMsg), share);
                    return false;
                }
                // the rows the request streams (kmap: T > 0 or not, from the
                // prologue, so no global read per message)
                const unsigned need = (!a.onehot && ctl.kmap[item] >= 0 ? 2 * GM + 1 : GM + 1) * V;
                // release: this block's row records are visible before they are
                // counted; acquire: the other blocks' records before they are read
                return atom_add_acq_rel(req_done + item, share) + share == need;
            },
            [&](int item) {
                if (!(item & kJobMsg)) {
                    K.verify_request(item, fin_rows);
                    stamp(ph, 3, lane == 0);
                }
            },
            [&]() { return false; }, [&]() { return true; });
        stamp(ph, 9, lane == 0);
        return;
    }

    // ------------------------------------------------------------ searcher
    if (searcher) {
        // the jobs published at positions g, g + G, ...: searched as soon as
        // their last chunk is counted, beside the finisher's scans
        int own_p = blockIdx.x, own_k = -1;  // lane 0: next owned job position, its job
        volatile int* vab = &ctl.abort;
        unsigned long long t0 = global_ns();
        for (;;) {
            if (K.poll_owned(own_p, own_k)) {
                t0 = global_ns();
                continue;
            }
            int stop = 0;
            if (lane == 0) {
                const int ns = *reinterpret_cast<volatile int*>(&ctl.n_samp);  // -1 until the consumers' prologue
                if (*vab) {
                    stop = 1;
                } else if (ns >= 0 && own_p >= ns) {
                    stop = 1;
                } else if (global_ns() - t0 > kWaitTimeoutNs) {
                    K.set_abort(a.d_status);
                    stop = 1;
                }
            }
            if (__shfl_sync(0xffffffffu, stop, 0)) break;
            __nanosleep(100);
        }
        stamp(ph, 9, lane == 0);
        return;
    }

    typename KT::Cursor prod, cons;
    constexpr int TPT = KT::kTPT;
    constexpr int CH = KT::kChunkElems;
    volatile int* vabort = &ctl.abort;

    // ------------------------------------------------------------ producer
    if (producer) {
        bool ok = true;
        // The row streams' lines go first from L2: each logit is read once
        // there (a draw re-reads its rows with copies of its own, at the normal
        // policy), and the small records, jobs and counters the scans and
        // searches read stay. Same box, µs per call, sampling / mixed / large:
        // 77.1 / 174.9 / 382.8 at the normal policy, 68.8 / 167.5 / 375.8
        // with it; the draws' copies at evict-first as well: 73.0 / 170.6 / 380.8.
        const uint64_t pol = l2_evict_first_policy();
        auto issue = [&](const Segment& sg) {
            for (long long off = 0; off < sg.elems && ok && !*vabort; off += KT::kStageElems) {
                const long long n = min(static_cast<long long>(KT::kStageElems), sg.elems - off);
                ok = K.produce_stream(prod, sg.src + off * KT::ES, static_cast<unsigned>(n * KT::ES), pol);
            }
        };
        bar_sync(kBarHandoff, kHandoffThreads);  // the consumers' prologue (partitions, maps) is done
        K.for_each_segment(issue);
        const int ns = ctl.n_samp;
        if (ns > 0) {
            // draw items i = 0 .. ns * NCH - 1: chunk i % NCH of the job published
            // i / NCH-th, taken kGrab at a time from the global counter (the next
            // batch is requested while the current one is issued)
            if (a.hold_flag && ok && lane == 0) {  // checking only: a flag that holds the draw phase
                const unsigned long long t0 = global_ns();
                while (ld_relaxed(a.hold_flag) == 0) {
                    if (global_ns() - t0 > a.peer_wait_ns) {
                        K.set_abort(a.d_status);
                        break;
                    }
                    __nanosleep(256);
                }
            }
            __syncwarp();
            Hdr* h = K.hdr();
            const long long n_items = static_cast<long long>(ns) * L.NCH;
            unsigned next = 0;
            if (lane == 0) next = atomicAdd(&h->next_item, static_cast<unsigned>(kGrab));
            long long i = 0, i_end = 0;
            int ip = 0, ij = 0;  // item i's job position and chunk (advanced by increments within a grab)
            int cur_p = -1;
            StageDesc desc;  // lane 0's copy of the current job
            desc.k = -1;
            int set0 = 0, set1 = 0;  // a tree job's excluded tokens (lane, lane + 32), read once per job
            while (ok && !*vabort) {
                if (i == i_end) {
                    i = __shfl_sync(0xffffffffu, next, 0);
                    i_end = i + kGrab;
                    if (i >= n_items) break;
                    if (lane == 0) next = atomicAdd(&h->next_item, static_cast<unsigned>(kGrab));
                    ip = static_cast<int>(static_cast<unsigned>(i) / static_cast<unsigned>(L.NCH));
                    ij = static_cast<int>(i) - ip * L.NCH;
                }
                if (i >= n_items) break;
                const int p = ip, j = ij;
                if (++ij == L.NCH) {
                    ij = 0;
                    ++ip;
                }
                if (p != cur_p) {
                    // the p-th published job (bounded wait: it is published by the
                    // finisher of the block that completes its request)
                    int got = 1;
                    if (lane == 0) {
                        int v = ld_relaxed(K.ready() + p);
                        if (v == 0) {
                            const unsigned long long t0 = global_ns();
                            while ((v = ld_relaxed(K.ready() + p)) == 0) {
                                if (*vabort || global_ns() - t0 > a.peer_wait_ns) {
                                    got = 0;
                                    break;
                                }
                                __nanosleep(64);
                            }
                        }
                        if (got) {
                            __threadfence();
                            desc.k = v - 1;
                            const int* src = reinterpret_cast<const int*>(K.jobs() + desc.k);
                            int* dst = reinterpret_cast<int*>(&desc.job);
#pragma unroll
                            for (int q = 0; q < static_cast<int>(sizeof(Job) / 4); ++q) dst[q] = __ldcg(src + q);
                        }
                    }
                    if (!__shfl_sync(0xffffffffu, got, 0)) {
                        if (lane == 0) K.set_abort(a.d_status);
                        ok = false;
                        break;
                    }
                    if (__shfl_sync(0xffffffffu, desc.job.kind, 0) == kKindResidualTree) {
                        // written by the finisher that published the job: read from L2
                        const int* gs = K.jobset() + static_cast<size_t>(__shfl_sync(0xffffffffu, desc.k, 0)) * a.gamma;
                        set0 = lane < a.gamma ? __ldcg(gs + lane) : 0;
                        set1 = lane + 32 < a.gamma ? __ldcg(gs + lane + 32) : 0;
                    }
                    if (cur_p < 0) stamp(ph, 4, lane == 0);
                    cur_p = p;
                }
                const int kind = __shfl_sync(0xffffffffu, desc.job.kind, 0);
                if (kind == kKindResidual || kind == kKindBonus || kind == kKindResidualOnehot ||
                    kind == kKindResidualTree) {
                    const int b = __shfl_sync(0xffffffffu, desc.job.b, 0), n = __shfl_sync(0xffffffffu, desc.job.n, 0);
                    desc.j = j;
                    const long long e0 = static_cast<long long>(j) * CH;
                    const int cnt = static_cast<int>(min(static_cast<long long>(CH), a.V - e0));
                    const unsigned bytes = static_cast<unsigned>(cnt * KT::ES);
                    const long long trow = static_cast<long long>(b) * (a.gamma + 1) + n;
                    const char* src_t = static_cast<const char*>(a.target) + (trow * a.V + e0) * KT::ES;
                    if (kind == kKindResidual) {
                        const long long drow = static_cast<long long>(b) * a.gamma + n;
                        ok = K.produce(prod, src_t, bytes,
                                       static_cast<const char*>(a.draft) + (drow * a.V + e0) * KT::ES, bytes, &desc);
                    } else if (kind == kKindResidualTree) {
                        const int ne = __shfl_sync(0xffffffffu, desc.job.d.excl, 0);
                        ok = K.produce(prod, src_t, bytes, nullptr, 0u, &desc, set0, set1, ne);
                    } else {
                        ok = K.produce(prod, src_t, bytes, nullptr, 0u, &desc);
                    }
                }
                ++i;
            }
            if (!ok && lane == 0) K.set_abort(a.d_status);
            __syncwarp();
            // the end marker, also after a failure (bounded: the consumers'
            // own waits are bounded too)
            StageDesc end;
            end.job.kind = kEndKind;
            end.k = -1;
            end.j = -1;
            K.produce(prod, nullptr, 0u, nullptr, 0u, &end);
        }
        if (!ok && lane == 0) K.set_abort(a.d_status);
        if (*vabort) K.drain(prod);
        return;
    }

    // ------------------------------------------------------------ consumers
    // the producer starts once the prologue has laid out the three streams
    K.prologue();
    bar_arrive(kBarHandoff, kHandoffThreads);
    bool ok = true;
    unsigned seq = 0;    // row pieces folded so far (the same on every consumer warp)
    unsigned share = 0;  // elements of the current request folded in this slice
    typename KT::ReqScale rq;
    auto fold = [&](const Segment& sg) {
        if (!ok) return;
        typename KT::RowState rs;
        K.start_row(rs, sg.loc, rq);
        for (long long off = 0; off < sg.elems; off += KT::kStageElems) {
            const long long n = min(static_cast<long long>(KT::kStageElems), sg.elems - off);
            const char* sm = K.consume_begin(cons);
            if (!sm) {
                ok = false;
                K.set_abort(a.d_status);
                return;
            }
            uint4 v[kVecPerThread];
            KT::load_stage(sm, static_cast<int>(n * KT::ES / 16), v);
            K.consume_end(cons);
            K.fold_vectors(rs, v, sg.e0 + off);
        }
        share += static_cast<unsigned>(sg.elems);
        K.flush_row(rs, sg.loc, seq++, sg.last ? share : 0u);
        if (sg.last) share = 0;
    };
    K.for_each_segment(fold);
    stamp(ph, 2, lane == 0);

    if (ctl.n_samp > 0 && ok) {
        // draw items until the producer's end marker; each warp stores the
        // fixed-point sum of its 32 runs, and the last warp done with an item
        // posts it to the finisher
        unsigned long long* wsums = K.wsums();
        for (unsigned iseq = 0;; ++iseq) {
            const int slot = static_cast<int>(cons.it % kStages);
            const char* smt = K.consume_begin(cons);
            if (!smt) {
                K.set_abort(a.d_status);
                break;
            }
            const StageDesc ds = ctl.desc[slot];
            if (ds.job.kind == kEndKind) {
                K.consume_end(cons);
                break;
            }
            const long long e0 = static_cast<long long>(ds.j) * CH;
            const int n = static_cast<int>(min(static_cast<long long>(CH), a.V - e0));
            const int valid = max(0, min(TPT, n - t * TPT));
            typename KT::Run lt, ld;
            if (valid > 0) {
                KT::load_run_smem(smt, t, lt);
                if (ds.job.kind == kKindResidual) KT::load_run_smem(smt + kChunkBytes, t, ld);
            }
            // a tree draw's excluded tokens: this warp's own copy, so that the
            // stage is released before the weights like the other kinds
            int* wset = ctl.wset[warp];
            if (ds.job.kind == kKindResidualTree) {
                if (lane < ds.job.d.excl) wset[lane] = ctl.dset[slot][lane];
                if (lane + 32 < ds.job.d.excl) wset[lane + 32] = ctl.dset[slot][lane + 32];
                __syncwarp();
            }
            K.consume_end(cons);
            const float run = valid > 0 ? KT::run_total_by_kind(lt, ld, t, valid, ds.job.d, ds.job.kind,
                                                                static_cast<int>(e0) + t * TPT, wset)
                                        : 0.0f;
            const unsigned long long wsum = warp_sum_u64(to_fixed(run, ds.job.d.fix));
            if (lane == 0) {
                wsums[(static_cast<size_t>(ds.k) * L.NCH + ds.j) * kConsumerWarps + warp] = wsum;
                // items continue the row pieces' numbering: a warp that starts
                // the draw phase early never shares a slot with a piece that
                // slower warps are still flushing
                const int fs = static_cast<int>((seq + iseq) % kFlushSlots);
                __threadfence_block();
                if (atomicAdd(&ctl.wcnt[fs], 1) == kConsumerWarps - 1) {
                    __threadfence_block();
                    ctl.wcnt[fs] = 0;
                    if (!K.post(ds.k | kJobMsg, 1u)) K.set_abort(a.d_status);
                }
            }
        }
    }
    K.consumer_done();
    stamp(ph, 6, lane == 0);
}

// Early-exit verification: the same producer and consumer warps, with tasks
// (one position's row statistics, or one draw) taken in publication order
// instead of a static row schedule and a draw phase; the finisher only counts
// the chunks done, and the search warp owns tasks g, g + G, ...: it decides
// them (or searches their draws) and publishes what follows.
template <int DT>
__global__ void __launch_bounds__(kThreads, 1) early_kernel(Args a, Layout L, char* ws) {
    extern __shared__ __align__(128) char smem[];
    char* stages = smem;
    Ctl& ctl = *reinterpret_cast<Ctl*>(smem + static_cast<size_t>(kStages) * kStageBytes);
    using KT = Kern<DT>;
    KT K{a, L, ws, ctl, stages, static_cast<int>(gridDim.x), static_cast<int>(blockIdx.x)};
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    unsigned long long* ph = reinterpret_cast<unsigned long long*>(a.dbg.phase_ns);
    stamp(ph, 0, t == 0);
    if (t == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl.full[s], 1);
            mbar_init(&ctl.empty[s], kConsumerWarps);
        }
        ctl.abort = 0;
        ctl.n_samp = 0;
        ctl.fq_tail = 0;
        ctl.fq_head = 0;
        ctl.cons_done = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int i = t; i < kFlushSlots; i += kThreads) ctl.wcnt[i] = 0;
    for (int i = t; i < kQueue; i += kThreads) ctl.fq_seq[i] = 0;
    __syncthreads();

    typename KT::Cursor prod, cons;
    if (warp == kSearchWarp) {
        // the owned tasks g, g + G, ...: decided or searched as soon as their
        // last chunk is counted
        // a request's count stays -1 until it is final (the owner of its
        // position 0 clears it before deciding anything)
        for (int b = blockIdx.x + lane * K.G; b < a.B; b += 32 * K.G) a.out_num_accepted[b] = -1;
        __threadfence();
        int own_p = blockIdx.x, own_v = 0, pre_p = -1;  // lane 0: next owned task, its code once published
        typename KT::EePre pre{};
        volatile int* vab = &ctl.abort;
        unsigned long long t0 = global_ns();
        for (;;) {
            if (K.ee_poll_owned(own_p, own_v, pre, pre_p)) {
                t0 = global_ns();
                continue;
            }
            int stop = 0;
            if (lane == 0) {
                if (*vab) {
                    stop = 1;
                } else if (own_p >= L.ee_cap || (own_v == 0 && K.ee_no_task(own_p))) {
                    stop = 1;
                } else if (global_ns() - t0 > kWaitTimeoutNs) {
                    K.set_abort(a.d_status);
                    stop = 1;
                }
            }
            if (__shfl_sync(0xffffffffu, stop, 0)) break;
            __nanosleep(64);
        }
        stamp(ph, 9, lane == 0);
        return;
    }
    if (warp == kFinisherWarp) {
        unsigned* done = K.ee_done();
        K.finish([&](int item, unsigned v) {
                     red_release_add(done + (item & ~kJobMsg), v);  // the task's owner polls the count
                     return false;
                 },
                 [&](int) {}, [&]() { return false; }, [&]() { return true; });
        stamp(ph, 9, lane == 0);
        return;
    }
    if (warp == kProducerWarp) {
        K.ee_produce(prod);
        if (ctl.abort) K.drain(prod);
        return;
    }
    K.ee_consume(cons);
    K.consumer_done();
    stamp(ph, 6, lane == 0);
}

constexpr size_t kSmemBytes = static_cast<size_t>(kStages) * kStageBytes + sizeof(Ctl) + sizeof(Rec) * kMaxRowsPerReq;
static_assert(kSmemBytes <= 232448, "dynamic shared memory above the 227 KB a block may opt in to");

size_t smem_bytes() { return kSmemBytes; }

}  // namespace

bool streaming_applicable(const Args& a) {
    const size_t es = a.dtype == SV_F32 ? 4 : 2;
    if ((static_cast<size_t>(a.V) * es) % 16 != 0) return false;
    if ((reinterpret_cast<uintptr_t>(a.target) & 15) || (reinterpret_cast<uintptr_t>(a.draft) & 15)) return false;
    if (a.B > kMaxB) return false;
    if (static_cast<size_t>(a.V) * es > static_cast<size_t>(128) * kChunkBytes) return false;  // <= 128 chunks per row
    return true;
}

int streaming_default_grid(const DeviceInfo& dev) { return std::min(dev.num_sms, kMaxGrid); }

bool streaming_grid_ok(int B, int grid) { return grid <= kMaxGrid && (B + grid - 1) / grid + 4 <= kMapMax; }

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
    const void* fn = a.early ? (a.dtype == SV_F32 ? reinterpret_cast<const void*>(&early_kernel<SV_F32>)
                                                   : reinterpret_cast<const void*>(&early_kernel<SV_BF16>))
                             : (a.dtype == SV_F32 ? reinterpret_cast<const void*>(&stream_kernel<SV_F32>)
                                                  : reinterpret_cast<const void*>(&stream_kernel<SV_BF16>));
    static thread_local int attr_device = -1;
    if (attr_device != dev.device) {
        cudaError_t e = cudaFuncSetAttribute(&stream_kernel<SV_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(&stream_kernel<SV_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(&early_kernel<SV_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(&early_kernel<SV_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, &stream_kernel<SV_BF16>, kThreads, smem);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        attr_device = dev.device;
    }
    if (grid > dev.num_sms) return cudaErrorInvalidValue;
    // the header and the completion counters start at zero
    cudaError_t e = cudaMemsetAsync(workspace, 0, a.early ? L.clear_bytes : L.ee_tasks, stream);
    if (e != cudaSuccess) return e;
    Args args = a;
    Layout lay = L;
    char* ws = static_cast<char*>(workspace);
    void* params[] = {&args, &lay, &ws};
    return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kThreads), params, smem, stream);
}

}  // namespace sv
