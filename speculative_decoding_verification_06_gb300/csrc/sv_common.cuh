// Device-side building blocks shared by the two execution paths of
// libspecverify: logit loads, the per-row online (max, sum) state, the
// argmax state, the acceptance test and the inverse-CDF weights.
//
// Arithmetic conventions (both paths):
//  * c = log2(e) / T, rounded once to binary32 (taken as +inf below T = 2^-64;
//    ck = log2(e) / (T 2^64) then stands in for it, applied to differences
//    scaled by 2^64, exactly). A row's
//    normaliser is kept as (m, s) in one of two forms:
//     - anchored: s = sum_x 2^(l(x) * c - mc), mc = fl(m * c) the binary32
//       product. Each term is one fused multiply-add and one 2^x; the
//       rounding r = m c - mc of the anchor is a common factor 2^r of every
//       term of the row, and every consumer of (m, s) recomputes mc the same
//       way, so it cancels exactly in p(x) = 2^(l(x) c - mc) / s. Used while
//       c is finite and |mc| < 2^23, so that |r| <= 1/2 and no term exceeds
//       2^(1/2);
//     - plain: s = sum_x 2^(fl(l(x) - m) c), each exponent formed from the
//       difference to the row max (fl(l - m) is exact for every logit close
//       enough to the max to matter), whatever the magnitude of the logits
//       and for any T > 0. Used for rows with |fl(m c)| >= 2^23 (logits
//       beyond about 5.8e6 T) and for T small enough that c overflows.
//    The two forms differ by the factor 2^r; states are merged in the
//    anchored form when both are anchored, else both are turned plain
//    (s * 2^-r) first.
//  * 2^x uses the special-function unit (PTX ex2.approx.ftz.f32).
//  * The acceptance test of "Speculative Decoding : accélérer l'inférence des
//    LLM", §Pourquoi la qualité est préservée, u < min(1, p(x)/q(x)), is
//    evaluated from the gathered logits and the rows' statistics.
//  * Inverse-CDF draws: each thread sums the binary32 weights of a run of
//    consecutive tokens; the run sums are converted to unsigned 64-bit fixed
//    point (2^-60 units for residual weights, which sum to at most 1; 2^-39
//    for unnormalised target weights, each at most 2^(1/2) and at most 2^24
//    of them) so that every prefix sum is exact and independent of the order
//    in which a reduction or scan adds them.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "specverify.h"

namespace sv {

constexpr double kLog2e = 1.4426950408889634073599246810019;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000u); }
__device__ __forceinline__ float pos_inf() { return __int_as_float(0x7f800000u); }

// 2^x on the special-function unit; results below 2^-126 flush to zero.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The scale of a sampled row: c = log2(e) / T, one correctly rounded binary32
// division of the binary32 log2(e) (no FP64 on the hot path: FP64 is a small
// fraction of FP32 here). Below T = 2^-64 (where c overflows for T under about
// 4.2e-39, and no row of ordinary logits could be anchored anyway) c is +inf,
// so every such row takes the plain form, and ck = log2(e) / (T 2^64) scales
// it instead (T 2^64 is exact and at least 2^-85, so ck is finite); else ck = 0.
constexpr float kLog2eF = 1.44269504088896340736f;
constexpr float kTwo64 = 18446744073709551616.0f;  // 2^64
struct Scale {
    float c;
    float ck;
};
__device__ __forceinline__ Scale temp_scale(float T) {
    const bool tiny = T < 5.42101086242752217004e-20f;  // 2^-64
    const float q = __fdiv_rn(kLog2eF, tiny ? __fmul_rn(T, kTwo64) : T);
    return Scale{tiny ? __int_as_float(0x7f800000u) : q, tiny ? q : 0.0f};
}

// The exponent d log2(e) / T of a difference d = l - m <= 0 to the row max,
// for the plain form: d * c, or (d 2^64) * ck where c overflowed (d 2^64 is
// exact, or -inf where the true exponent is below -2^64 anyway).
__device__ __forceinline__ float plain_arg(float d, const Scale& sc) {
    if (sc.c < __int_as_float(0x7f800000u)) return __fmul_rn(d, sc.c);
    return __fmul_rn(__fmul_rn(d, kTwo64), sc.ck);
}

__device__ __forceinline__ float bf16_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }
__device__ __forceinline__ float bf16x2_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16x2_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// A logit that must not be read: NaN or +inf.
__device__ __forceinline__ bool bad_logit(float x) { return !(x < pos_inf()); }

template <int DT>
__device__ __forceinline__ float load_logit(const void* base, size_t idx);

template <>
__device__ __forceinline__ float load_logit<SV_F32>(const void* base, size_t idx) {
    return __ldg(static_cast<const float*>(base) + idx);
}

template <>
__device__ __forceinline__ float load_logit<SV_BF16>(const void* base, size_t idx) {
    return bf16_to_float(__ldg(static_cast<const unsigned short*>(base) + idx));
}

// ---------------------------------------------------------------- row state

// Online normaliser state: s = sum 2^(l c - fl(m c)) over the logits seen
// (anchored form, plain = 0) or s = sum 2^((l - m) c) (plain form, plain = 1).
struct MaxSum {
    float m;
    float s;
    int plain;
};

__device__ __forceinline__ MaxSum maxsum_empty() { return {neg_inf(), 0.0f, 0}; }

__device__ __forceinline__ float scaled_max(float m, float c) { return __fmul_rn(m, c); }

// Whether a row whose max is m may be kept in the anchored form: c finite
// and |fl(m c)| < 2^23 (NaN, from 0 * inf, fails too).
__device__ __forceinline__ bool anchor_ok(float m, float c) { return fabsf(scaled_max(m, c)) < 8388608.0f; }

// r = m c - fl(m c), exact (the error of a product is a binary32 number and a
// fused multiply-add forms it without rounding).
__device__ __forceinline__ float anchor_err(float m, float c) { return __fmaf_rn(m, c, -scaled_max(m, c)); }

// 2^(l c - mc), the term of logit l in an anchored row whose scaled max is mc.
__device__ __forceinline__ float row_term(float l, float c, float mc) { return ex2(__fmaf_rn(l, c, -mc)); }

// 2^((l - m) c), the term of logit l in a plain row whose max is m.
__device__ __forceinline__ float plain_term(float l, float m, const Scale& sc) {
    return ex2(plain_arg(__fsub_rn(l, m), sc));
}

// The sum of an anchored state in the plain form: s 2^-r.
__device__ __forceinline__ float plain_sum(float m, float s, float c) {
    return m == neg_inf() ? s : __fmul_rn(s, ex2(-anchor_err(m, c)));
}

__device__ __forceinline__ void maxsum_to_plain(MaxSum& st, const Scale& sc) {
    if (!st.plain) {
        st.s = plain_sum(st.m, st.s, sc.c);
        st.plain = 1;
    }
}

// Adds one logit (the caller screens NaN and +inf).
__device__ __forceinline__ void maxsum_add(MaxSum& st, float x, const Scale& sc) {
    const float c = sc.c;
    if (x > st.m) {
        if (!st.plain && anchor_ok(x, c)) {
            const float mc = scaled_max(x, c);
            st.s = (st.m == neg_inf()) ? 0.0f : __fmul_rn(st.s, ex2(__fsub_rn(scaled_max(st.m, c), mc)));
            st.m = x;
            st.s = __fadd_rn(st.s, row_term(x, c, mc));
        } else {
            maxsum_to_plain(st, sc);
            st.s = (st.m == neg_inf()) ? 0.0f : __fmul_rn(st.s, plain_term(st.m, x, sc));
            st.m = x;
            st.s = __fadd_rn(st.s, 1.0f);
        }
    } else if (x != neg_inf()) {
        st.s = __fadd_rn(st.s, st.plain ? plain_term(x, st.m, sc) : row_term(x, c, scaled_max(st.m, c)));
    }
}

// Merges b into a.
__device__ __forceinline__ MaxSum maxsum_merge(MaxSum a, MaxSum b, const Scale& sc) {
    if (b.m > a.m) {
        MaxSum t = a;
        a = b;
        b = t;
    }
    if (b.m == neg_inf()) return a;
    if (!a.plain && !b.plain) {
        a.s = __fadd_rn(a.s, __fmul_rn(b.s, ex2(__fsub_rn(scaled_max(b.m, sc.c), scaled_max(a.m, sc.c)))));
        return a;
    }
    maxsum_to_plain(a, sc);
    maxsum_to_plain(b, sc);
    a.s = __fadd_rn(a.s, __fmul_rn(b.s, plain_term(b.m, a.m, sc)));
    return a;
}

// The anchored state alone, as the streaming kernels' consumers keep it: they
// flag a row whose anchor leaves the range (kBadPlain) instead of switching
// forms, and the warp that decides the request recomputes that row plain.
struct MaxSumA {
    float m;
    float s;
};

// Adds one logit to an anchored state (the caller screens NaN and +inf);
// sets `flag` when the anchor leaves its range (the row is then recomputed
// plain).
__device__ __forceinline__ void maxsum_add_a(MaxSumA& st, float x, float c, int& flag) {
    if (x > st.m) {
        const float mc = scaled_max(x, c);
        if (!(fabsf(mc) < 8388608.0f)) flag = 1;
        st.s = (st.m == neg_inf()) ? 0.0f : __fmul_rn(st.s, ex2(__fsub_rn(scaled_max(st.m, c), mc)));
        st.m = x;
        st.s = __fadd_rn(st.s, row_term(x, c, mc));
    } else if (x != neg_inf()) {
        st.s = __fadd_rn(st.s, row_term(x, c, scaled_max(st.m, c)));
    }
}

__device__ __forceinline__ MaxSumA maxsum_merge_a(MaxSumA a, MaxSumA b, float c) {
    if (b.m > a.m) {
        MaxSumA t = a;
        a = b;
        b = t;
    }
    if (b.m == neg_inf()) return a;
    a.s = __fadd_rn(a.s, __fmul_rn(b.s, ex2(__fsub_rn(scaled_max(b.m, c), scaled_max(a.m, c)))));
    return a;
}

// Argmax state with the lowest index winning ties.
struct ArgMax {
    float v;
    int32_t i;
};

__device__ __forceinline__ ArgMax argmax_empty() { return {neg_inf(), 0x7fffffff}; }

__device__ __forceinline__ ArgMax argmax_merge(ArgMax a, ArgMax b) {
    return (b.v > a.v || (b.v == a.v && b.i < a.i)) ? b : a;
}

// ------------------------------------------------------------ decisions

// p(x) from the row's statistics, in double: 2^(l c - fl(m c)) / s
// (anchored) or 2^((l - m) c) / s (plain).
__device__ __forceinline__ double prob_from_stats(float l, const MaxSum& st, const Scale& sc) {
    if (!st.plain) {
        const double mc = static_cast<double>(scaled_max(st.m, sc.c));
        return exp2(static_cast<double>(l) * static_cast<double>(sc.c) - mc) / static_cast<double>(st.s);
    }
    const double d = static_cast<double>(l) - static_cast<double>(st.m);
    const double e = sc.c < pos_inf() ? d * static_cast<double>(sc.c)
                                      : d * static_cast<double>(kTwo64) * static_cast<double>(sc.ck);
    return exp2(e) / static_cast<double>(st.s);
}

// The accept test u < min(1, p(x)/q(x)) from the gathered logits and the two
// rows' statistics. q(x) = 0 (ld = -inf) gives alpha = 1 if p(x) > 0, else 0;
// u = 0 accepts whenever p(x) > 0, even where p/q underflows.
// Two anchored rows: p/q = 2^e * s_q / s_p with e = (lt - ld) c - (fl(mp c) -
// fl(mq c)) formed with error-free transformations in binary32, rounded once
// and raised on the SFU (relative error about 3e-7; no FP64 on the common
// path). Otherwise (a plain row: large logits or tiny T) in double:
// e = ((lt - mp) - (ld - mq)) c + r_p - r_q, r the anchor rounding of an
// anchored row (0 for a plain one); the differences to the maxima keep e
// accurate whatever the magnitude of the logits.
__device__ __forceinline__ bool accept_from_logits(float lt, float ld, const MaxSum& P, const MaxSum& Q,
                                                   const Scale& sc, float u) {
    if (lt == neg_inf()) return false;  // p(x) = 0 < alpha requires p(x) > 0
    if (ld == neg_inf() || u == 0.0f) return true;
    const float c = sc.c;
    if (!P.plain && !Q.plain) {
        const float d = __fsub_rn(lt, ld);
        const float dz = __fsub_rn(d, lt), d_lo = __fadd_rn(__fsub_rn(lt, __fsub_rn(d, dz)), __fsub_rn(-ld, dz));
        const float mcp = scaled_max(P.m, c), mcq = scaled_max(Q.m, c);
        const float m = __fsub_rn(mcp, mcq);
        const float mz = __fsub_rn(m, mcp), m_lo = __fadd_rn(__fsub_rn(mcp, __fsub_rn(m, mz)), __fsub_rn(-mcq, mz));
        const float p_hi = __fmul_rn(d, c), p_lo = __fmaf_rn(d, c, -p_hi);
        const float e = __fadd_rn(__fsub_rn(p_hi, m), __fsub_rn(__fmaf_rn(d_lo, c, p_lo), m_lo));
        const float alpha = __fmul_rn(ex2(e), __fdiv_rn(Q.s, P.s));
        return u < alpha;
    }
    const double D = (static_cast<double>(lt) - static_cast<double>(P.m)) -
                     (static_cast<double>(ld) - static_cast<double>(Q.m));
    double e;
    if (c < pos_inf()) {
        const double rp = P.plain ? 0.0 : static_cast<double>(anchor_err(P.m, c));
        const double rq = Q.plain ? 0.0 : static_cast<double>(anchor_err(Q.m, c));
        e = D * static_cast<double>(c) + (rp - rq);
    } else {
        e = D * static_cast<double>(kTwo64) * static_cast<double>(sc.ck);  // no anchored row without a finite c
    }
    const double alpha = exp2(e) * (static_cast<double>(Q.s) / static_cast<double>(P.s));
    return static_cast<double>(u) < alpha;
}

// log sum_x exp(l(x)/T) from the statistics: m/T + ln s, less r ln 2 for an
// anchored row (its s carries the factor 2^r, r = m c - fl(m c)), with m/T and
// m c in double.
__device__ __forceinline__ double lse_from_stats(const MaxSum& st, const Scale& sc, float T) {
    const double base = static_cast<double>(st.m) / static_cast<double>(T) + log(static_cast<double>(st.s));
    if (st.plain) return base;
    const double mc_exact = static_cast<double>(st.m) * static_cast<double>(sc.c);
    const double mc = static_cast<double>(scaled_max(st.m, sc.c));
    return base - (mc_exact - mc) * 0.69314718055994530942;
}

// ------------------------------------------------------- inverse-CDF weights

// Draw kinds, also reported in sv_debug_out.kind.
constexpr int kDrawPlain = 0x100;  // DrawParams.kind flag: the draw's exponents are plain
constexpr int kKindInvalid = -1;
constexpr int kKindGreedy = 0;
constexpr int kKindResidual = 1;
constexpr int kKindBonus = 2;
// Internal draw kind, reported as kKindResidual: the residual of a one-hot
// (deterministic) proposal, p_n without the proposed token x_n.
constexpr int kKindResidualOnehot = 3;
// Internal job kind of the streaming kernels: a draw already made by the
// warp that published the job (a plain draw); no items, no search.
constexpr int kKindDrawn = 5;

constexpr float kFixResidual = 1152921504606846976.0f;  // 2^60
constexpr float kFixTarget = 549755813888.0f;           // 2^39
constexpr double kFixResidualInv = 1.0 / 1152921504606846976.0;
constexpr double kFixTargetInv = 1.0 / 549755813888.0;

// Weights of one draw. Residual: max(p - q, 0) from target row n and draft
// row n ("Speculative Decoding" wiki, eq. p_corr). Target: 2^((l - m) c),
// proportional to p at the target row (the extra token, or the fallback when
// residual weights sum to zero). Anchored draws (every row anchored) form the
// exponents with one fused multiply-add against fl(m c); plain draws from the
// difference to the row max (the maxima in mcp, mcq and the plain sums'
// reciprocals in isp, isq).
struct DrawParams {
    int kind;       // kKindResidual, kKindBonus, ... (| kDrawPlain for a plain draw)
    float c;        // c; a plain draw whose c overflowed holds -ck (see draw_scale)
    float mcp, isp; // target row: fl(max * c) (plain: the max) and 1/s
    float mcq, isq; // draft row (residual only)
    float fix;      // fixed-point scale
    int excl;       // kKindResidualOnehot: the token whose weight is zero
    __device__ bool plain() const { return (kind & kDrawPlain) != 0; }
    __device__ int base_kind() const { return kind & ~kDrawPlain; }
};

// The scale of a draw: c, or (+inf, ck) where c overflowed (stored as -ck).
__device__ __forceinline__ Scale draw_scale(const DrawParams& d) {
    return d.c > 0.0f ? Scale{d.c, 0.0f} : Scale{pos_inf(), -d.c};
}

// Fills the row part of a draw's parameters from the statistics of its target
// row P and, for a residual, its draft row Q, and sets the draw's kind.
__device__ __forceinline__ void draw_rows(DrawParams& d, int kind, const MaxSum& P, const MaxSum* Q,
                                          const Scale& sc) {
    const bool plain = P.plain || (Q && Q->plain);
    d.kind = kind | (plain ? kDrawPlain : 0);
    d.c = sc.c < pos_inf() ? sc.c : -sc.ck;
    if (!plain) {
        d.mcp = scaled_max(P.m, sc.c);
        d.isp = __frcp_rn(P.s);
        d.mcq = Q ? scaled_max(Q->m, sc.c) : 0.0f;
        d.isq = Q ? __frcp_rn(Q->s) : 0.0f;
    } else {
        d.mcp = P.m;
        d.isp = __frcp_rn(P.plain ? P.s : plain_sum(P.m, P.s, sc.c));
        d.mcq = Q ? Q->m : 0.0f;
        d.isq = Q ? __frcp_rn(Q->plain ? Q->s : plain_sum(Q->m, Q->s, sc.c)) : 0.0f;
    }
}

__device__ __forceinline__ float weight_target(float lt, const DrawParams& d) {
    return d.plain() ? plain_term(lt, d.mcp, draw_scale(d)) : row_term(lt, d.c, d.mcp);
}

__device__ __forceinline__ float weight_residual(float lt, float ld, const DrawParams& d) {
    const float p = __fmul_rn(weight_target(lt, d), d.isp);
    const float q = __fmul_rn(d.plain() ? plain_term(ld, d.mcq, draw_scale(d)) : row_term(ld, d.c, d.mcq), d.isq);
    return fmaxf(__fsub_rn(p, q), 0.0f);
}

// Weight of token `e` of the target row for a draw of kind kBonus or
// kResidualOnehot: 2^((l - m) c), zero for the excluded token of a one-hot
// residual (max(p - q, 0) with q one-hot at x_n is p without x_n).
__device__ __forceinline__ float weight_target_excl(float lt, int e, const DrawParams& d, int kind) {
    return (kind == kKindResidualOnehot && e == d.excl) ? 0.0f : weight_target(lt, d);
}

// Tree verification: the last token is drawn from p without the tokens of the
// rejected children (at most SV_MAX_GAMMA of them).
constexpr int kKindResidualTree = 4;  // internal, reported as kKindResidual

__device__ __forceinline__ bool in_set(int e, const int* set, int n) {
    for (int i = 0; i < n; ++i)
        if (set[i] == e) return true;
    return false;
}

// floor(u * total) exactly, for u in [0, 1): u = M 2^e with an integer M < 2^24,
// so the product is a 128-bit integer shifted right by -e.
__device__ __forceinline__ unsigned long long scale_uniform(float u, unsigned long long total) {
    const uint32_t bits = __float_as_uint(u);
    const uint32_t ex = (bits >> 23) & 0xffu;
    if (u <= 0.0f || total == 0ull) return 0ull;
    const unsigned long long M = ex ? ((bits & 0x7fffffu) | 0x800000u) : (bits & 0x7fffffu);
    const int shift = 150 - static_cast<int>(ex ? ex : 1);  // u = M 2^-shift
    const unsigned long long lo = total * M, hi = __umul64hi(total, M);
    if (shift >= 128) return 0ull;
    if (shift >= 64) return hi >> (shift - 64);
    return (hi << (64 - shift)) | (lo >> shift);
}

__device__ __forceinline__ unsigned long long to_fixed(float run_sum, float fix) {
    return __float2ull_rz(__fmul_rn(run_sum, fix));
}

// ------------------------------------------------------------ reductions

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Exclusive prefix sum of v over the threads of a block of NT threads (exact:
// integers). `scratch` holds NT/32 + 1 values. Also returns the block total.
template <int NT>
__device__ __forceinline__ unsigned long long block_excl_scan_u64(unsigned long long v,
                                                                  unsigned long long* scratch,
                                                                  unsigned long long* total) {
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long run = 0;
        for (int w = 0; w < NW; ++w) {
            unsigned long long t = scratch[w];
            scratch[w] = run;
            run += t;
        }
        scratch[NW] = run;
    }
    __syncthreads();
    unsigned long long excl = scratch[warp] + (x - v);
    *total = scratch[NW];
    __syncthreads();
    return excl;
}

}  // namespace sv
