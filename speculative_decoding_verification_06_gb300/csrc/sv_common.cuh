// Device-side building blocks shared by the two execution paths of
// libspecverify: logit loads, the per-row online (max, sum) state, the
// argmax state, the acceptance test and the inverse-CDF weights.
//
// Arithmetic conventions (both paths):
//  * c = log2(e) / T, rounded once to binary32. A row's normaliser is kept as
//    (m, s): m the row max and s = sum_x 2^(l(x) * c - mc), mc = fl(m * c)
//    (the binary32 product). Each term is one fused multiply-add and one
//    2^x; the rounding of mc is a common factor 2^(m*c - mc) of every term of
//    the row, and every consumer of (m, s) recomputes mc the same way, so it
//    cancels exactly in p(x) = 2^(l(x) c - mc) / s.
//  * 2^x uses the special-function unit (PTX ex2.approx.ftz.f32).
//  * The acceptance test of "Speculative Decoding : accélérer l'inférence des
//    LLM", §Pourquoi la qualité est préservée, u < min(1, p(x)/q(x)), is
//    evaluated in double from the row statistics.
//  * Inverse-CDF draws: each thread sums the binary32 weights of a run of
//    consecutive tokens; the run sums are converted to unsigned 64-bit fixed
//    point (2^-60 units for residual weights, which sum to at most 1; 2^-39
//    for unnormalised target weights, each at most 1 and at most 2^24 of
//    them) so that every prefix sum is exact and independent of the order in
//    which a reduction or scan adds them.
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

// c = log2(e) / T, one correctly rounded binary32 division of the binary32
// log2(e) (no FP64 on the hot path: FP64 is a small fraction of FP32 here).
// Temperatures in (0, 2^-16) are read as 2^-16. The row statistics sum
// 2^(l c - fl(m c)) with c = log2(e) / T; the largest term is 2^r, r the
// rounding error of fl(m c), which stays far from overflow while |m c| < 2^31
// (logits up to ~2.2e4 at T = 2^-16). At T = 2^-16, p is one-hot (uniform over
// exact ties) to within e^-128 for logits more than 2^-9 apart.
constexpr float kTempMin = 1.52587890625e-05f;  // 2^-16
__device__ __forceinline__ float temp_floor(float T) { return (T > 0.0f && T < kTempMin) ? kTempMin : T; }
__device__ __forceinline__ float temp_scale(float T) { return __fdiv_rn(1.44269504088896340736f, temp_floor(T)); }

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

// Online normaliser state: s = sum 2^(l c - fl(m c)) over the logits seen.
struct MaxSum {
    float m;
    float s;
};

__device__ __forceinline__ MaxSum maxsum_empty() { return {neg_inf(), 0.0f}; }

__device__ __forceinline__ float scaled_max(float m, float c) { return __fmul_rn(m, c); }

// A sampled row is in range while its scaled max fl(m c) stays below 2^31 in
// magnitude: the largest term of its statistics is 2^r with r the rounding
// error of fl(m c), at most half an ulp of it. A row out of range makes its
// request invalid (the same test, in binary32, as the reading on both sides).
__device__ __forceinline__ bool scaled_in_range(float m, float c) {
    return fabsf(scaled_max(m, c)) < 2147483648.0f;
}

// 2^(l c - mc), the term of logit l in a row whose scaled max is mc.
__device__ __forceinline__ float row_term(float l, float c, float mc) { return ex2(__fmaf_rn(l, c, -mc)); }

// Adds one logit (the caller screens NaN and +inf).
__device__ __forceinline__ void maxsum_add(MaxSum& st, float x, float c) {
    if (x > st.m) {
        const float mc = scaled_max(x, c);
        st.s = (st.m == neg_inf()) ? 0.0f : __fmul_rn(st.s, ex2(__fsub_rn(scaled_max(st.m, c), mc)));
        st.m = x;
        st.s = __fadd_rn(st.s, row_term(x, c, mc));
    } else if (x != neg_inf()) {
        st.s = __fadd_rn(st.s, row_term(x, c, scaled_max(st.m, c)));
    }
}

// Merges b into a.
__device__ __forceinline__ MaxSum maxsum_merge(MaxSum a, MaxSum b, float c) {
    if (b.m > a.m) {
        MaxSum t = a;
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

// p(x) = 2^(l c - fl(m c)) / s, in double.
__device__ __forceinline__ double prob_from_stats(float l, float m, float s, float c) {
    const double mc = static_cast<double>(scaled_max(m, c));
    return exp2(static_cast<double>(l) * static_cast<double>(c) - mc) / static_cast<double>(s);
}

// The accept test u < min(1, p(x)/q(x)) from the gathered logits and the two
// rows' (m, s): p/q = 2^e * s_q / s_p with e = (lt - ld) c - (fl(mp c) - fl(mq c)),
// e formed exactly in double, then rounded once and raised on the SFU (relative
// error about 3e-7). q(x) = 0 (ld = -inf) gives alpha = 1 if p(x) > 0, else 0;
// u = 0 accepts whenever p(x) > 0, even where 2^e underflows.
__device__ __forceinline__ bool accept_from_logits(float lt, float ld, float mp, float sp, float mq, float sq,
                                                   float c, float u) {
    if (lt == neg_inf()) return false;  // p(x) = 0 < alpha requires p(x) > 0
    if (ld == neg_inf() || u == 0.0f) return true;
    // e with error-free transformations in binary32: d = lt - ld and
    // m = fl(mp c) - fl(mq c) as two-sums, d * c as a two-product
    const float d = __fsub_rn(lt, ld);
    const float dz = __fsub_rn(d, lt), d_lo = __fadd_rn(__fsub_rn(lt, __fsub_rn(d, dz)), __fsub_rn(-ld, dz));
    const float mcp = scaled_max(mp, c), mcq = scaled_max(mq, c);
    const float m = __fsub_rn(mcp, mcq);
    const float mz = __fsub_rn(m, mcp), m_lo = __fadd_rn(__fsub_rn(mcp, __fsub_rn(m, mz)), __fsub_rn(-mcq, mz));
    const float p_hi = __fmul_rn(d, c), p_lo = __fmaf_rn(d, c, -p_hi);
    const float e = __fadd_rn(__fsub_rn(p_hi, m), __fsub_rn(__fmaf_rn(d_lo, c, p_lo), m_lo));
    const float alpha = __fmul_rn(ex2(e), __fdiv_rn(sq, sp));
    return u < alpha;
}

// log sum_x exp(l(x)/T) from (m, s, c): s = 2^(m c - fl(m c)) sum 2^((l - m) c),
// so the log is m/T + ln s - (m c - fl(m c)) ln 2, with m/T and m c in double.
__device__ __forceinline__ double lse_from_stats(float m, float s, float c, float T) {
    const double mc_exact = static_cast<double>(m) * static_cast<double>(c);
    const double mc = static_cast<double>(scaled_max(m, c));
    return static_cast<double>(m) / static_cast<double>(temp_floor(T)) + log(static_cast<double>(s)) -
           (mc_exact - mc) * 0.69314718055994530942;
}

// ------------------------------------------------------- inverse-CDF weights

// Draw kinds, also reported in sv_debug_out.kind.
constexpr int kKindInvalid = -1;
constexpr int kKindGreedy = 0;
constexpr int kKindResidual = 1;
constexpr int kKindBonus = 2;
// Internal draw kind, reported as kKindResidual: the residual of a one-hot
// (deterministic) proposal, p_n without the proposed token x_n.
constexpr int kKindResidualOnehot = 3;

constexpr float kFixResidual = 1152921504606846976.0f;  // 2^60
constexpr float kFixTarget = 549755813888.0f;           // 2^39
constexpr double kFixResidualInv = 1.0 / 1152921504606846976.0;
constexpr double kFixTargetInv = 1.0 / 549755813888.0;

// Weights of one draw. Residual: max(p - q, 0) from target row n and draft
// row n ("Speculative Decoding" wiki, eq. p_corr). Target: 2^((l - m) c),
// proportional to p at the target row (the extra token, or the fallback when
// residual weights sum to zero).
struct DrawParams {
    int kind;       // kKindResidual, kKindBonus or kKindResidualOnehot
    float c;
    float mcp, isp; // target row: fl(max * c) and 1/s
    float mcq, isq; // draft row (residual only)
    float fix;      // fixed-point scale
    int excl;       // kKindResidualOnehot: the token whose weight is zero
};

__device__ __forceinline__ float weight_target(float lt, const DrawParams& d) {
    return row_term(lt, d.c, d.mcp);
}

__device__ __forceinline__ float weight_residual(float lt, float ld, const DrawParams& d) {
    const float p = __fmul_rn(row_term(lt, d.c, d.mcp), d.isp);
    const float q = __fmul_rn(row_term(ld, d.c, d.mcq), d.isq);
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
