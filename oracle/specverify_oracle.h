/*
 * specverify_oracle.h -- the CPU oracle of the speculative-decoding
 * verification step.
 *
 * TEST INFRASTRUCTURE ONLY. This header and specverify_oracle.c are the
 * plain, slow, fp64 restatement of the method that the CUDA library is
 * checked against. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load it. It shares no code, header, table or helper
 * with the CUDA library (speculative_decoding_verification_06_gb300/csrc),
 * and the CUDA library never calls it.
 *
 * Sources (page title, section):
 *  - "Speculative Decoding : accélérer l'inférence des LLM",
 *    §Principe et garanties mathématiques (propose gamma tokens, verify in one
 *    target pass, accept while compatible, correct the first rejection, at
 *    least one and at most gamma+1 tokens per cycle) and
 *    §Pourquoi la qualité est préservée (accept with probability
 *    min(1, p(x)/q(x)); on rejection draw from p - q clipped at zero and
 *    renormalised; at temperature zero accept iff the token is the target
 *    argmax, else replace it by that argmax).
 *  - "Speculative Decoding — Come Accelerare l'Inferenza LLM di 2-3x Senza
 *    Perdere Qualità", §Il meccanismo: draft model, target model, rejection
 *    sampling (the later draft tokens are discarded after a rejection).
 *  - "Speculative Decoding" (wiki), §数式で見る speculative decoding の正しさ,
 *    eq. alpha(x) and eq. p_corr.
 *  - "Accélérer Sonar grâce à la spéculation", §Décodage spéculatif (up to
 *    n + 1 tokens per step; the target logits at the mismatch position or at
 *    the end of the sequence give the extra token).
 *
 * Readings where the pages are silent:
 *  - temperature: p = softmax(l_target / T), q = softmax(l_draft / T), the
 *    same T for both rows, for every finite T > 0 and every finite logit;
 *    T == 0 is the greedy rule;
 *  - accept iff u_accept < alpha, u in [0, 1); alpha = min(1, p/q); q == 0
 *    gives alpha = 1 when p > 0 and alpha = 0 when p == 0;
 *  - one uniform u_sample per request draws the replacement or the bonus
 *    token by inverse CDF in index order: the token is the smallest k with
 *    C_k > u * W, C_k the inclusive prefix sum of the weights, W their total;
 *    if rounding leaves no such k, the last k with a positive weight;
 *  - if the residual weights sum to zero (impossible in exact arithmetic),
 *    the replacement is drawn from p at that position instead;
 *  - argmax ties go to the lowest index;
 *  - a request is invalid (num_accepted = -1, every output token -1) when T
 *    is NaN, negative or infinite, a draft token is outside [0, V), or a row
 *    the request reads holds a NaN or +inf or only -inf values (the draft
 *    rows of a T == 0 request are never read).
 */
#ifndef SPECVERIFY_ORACLE_H
#define SPECVERIFY_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORACLE_F32 0  /* logits stored as IEEE binary32 */
#define ORACLE_BF16 1 /* logits stored as bfloat16 bit patterns (uint16) */

#define ORACLE_KIND_ERROR (-1)
#define ORACLE_KIND_GREEDY 0
#define ORACLE_KIND_RESIDUAL 1
#define ORACLE_KIND_BONUS 2

/* Optional per-row and per-request facts the checker compares. Every pointer
 * may be NULL. Entries the algorithm does not reach hold NaN (doubles) or -1
 * (integers). Row arrays are indexed like the logits: target [B, gamma+1],
 * draft [B, gamma]. */
typedef struct {
    double* max_target;    /* [B*(gamma+1)] max_x l(x) of every target row */
    double* lse_target;    /* [B*(gamma+1)] log sum_x exp(l(x)/T), T > 0 rows */
    int32_t* argmax_target;/* [B*(gamma+1)] lowest-index argmax of every row */
    double* max_draft;     /* [B*gamma] rows of T > 0 requests */
    double* lse_draft;     /* [B*gamma] rows of T > 0 requests */
    double* p_x;           /* [B*gamma] p_i(x_i) at the evaluated positions */
    double* q_x;           /* [B*gamma] q_i(x_i) at the evaluated positions */
    double* alpha;         /* [B*gamma] min(1, p/q) at the evaluated positions */
    double* accept_margin; /* [B*gamma] |u - alpha| / alpha (inf if alpha == 0) */
    double* w_total;       /* [B] W of the residual or bonus draw */
    double* sample_margin; /* [B] min(t - C_{k-1}, C_k - t) / W of that draw */
    int32_t* kind;         /* [B] ORACLE_KIND_* */
    double* tie_measure;   /* [B] for the checker: the probability, over u_sample
                              uniform on [0, 1), that t = u W lies within
                              ORACLE_TIE_MARGIN * W of an edge of that draw's CDF
                              (0, C_0, ..., C_{V-1} = W), in fp64 */
} oracle_detail;

/* The checker's margin for near-tie draws, relative to W. */
#define ORACLE_TIE_MARGIN 1e-5

/* The verification step for B independent requests, all on host memory.
 *   target      [B, gamma+1, V] logits (dtype), row i scores draft token i,
 *               row gamma is the bonus row
 *   draft       [B, gamma, V] logits (dtype)
 *   tokens      [B, gamma] draft tokens
 *   u_accept    [B, gamma] uniforms in [0, 1)
 *   u_sample    [B] uniforms in [0, 1)
 *   temperature [B]
 *   out_tokens  [B, gamma+1]: accepted tokens, then the replacement or bonus
 *               token, then -1
 *   out_num_accepted [B]: n in [0, gamma], or -1 for an invalid request
 * Returns 0, or -1 for a bad argument (nothing written). */
int oracle_spec_verify(const void* target, const void* draft, int dtype,
                       int B, int gamma, int V,
                       const int32_t* tokens, const float* u_accept,
                       const float* u_sample, const float* temperature,
                       int32_t* out_tokens, int32_t* out_num_accepted,
                       const oracle_detail* detail);

int oracle_version(void);

/* The same step for deterministic proposals (n-gram lookup): q_i is one-hot
 * at x_i, so alpha_i = min(1, p_i(x_i)) and the residual is p_n without x_n.
 * Request b proposes num_draft[b] in [0, gamma] tokens (outside: invalid);
 * target rows past num_draft[b] are never read; tokens past it are ignored.
 * No draft logits. Detail: q_x = 1 at the evaluated positions, draft rows NaN. */
int oracle_spec_verify_onehot(const void* target, int dtype, int B, int gamma, int V,
                              const int32_t* tokens, const int32_t* num_draft,
                              const float* u_accept, const float* u_sample,
                              const float* temperature, int32_t* out_tokens,
                              int32_t* out_num_accepted, const oracle_detail* detail);

/* Early exit: the same decisions as oracle_spec_verify (draft != NULL) or
 * oracle_spec_verify_onehot (draft == NULL, num_draft given), taking positions
 * in order and reading nothing after the first rejection. A request is
 * invalid only when a row it reads is bad, or T, the proposal count or a
 * proposed token is. Detail holds NaN / -1 for the rows not read. */
int oracle_spec_verify_early(const void* target, const void* draft, int dtype, int B, int gamma, int V,
                             const int32_t* tokens, const int32_t* num_draft, const float* u_accept,
                             const float* u_sample, const float* temperature, int32_t* out_tokens,
                             int32_t* out_num_accepted, const oracle_detail* detail);

/* Tree verification with deterministic candidates (see the comment above
 * oracle_spec_verify_tree in the .c file for the rule). gamma = the most
 * non-root nodes (at most 64); tokens, parents, u_accept [B, gamma] are
 * indexed by node - 1; num_nodes [B] non-root nodes in use; target
 * [B, gamma+1, V], row j for node j. Outputs: out_tokens [B, gamma+1] (the
 * accepted path's tokens, then the last token, then -1), out_num_accepted [B]
 * (path length, -1 invalid), out_nodes [B, gamma] (the accepted node indices,
 * then -1). Detail p_x / alpha / accept_margin are indexed by node - 1. */
int oracle_spec_verify_tree(const void* target, int dtype, int B, int gamma, int V, const int32_t* tokens,
                            const int32_t* parents, const int32_t* num_nodes, const float* u_accept,
                            const float* u_sample, const float* temperature, int32_t* out_tokens,
                            int32_t* out_num_accepted, int32_t* out_nodes, const oracle_detail* detail);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_ORACLE_H */
