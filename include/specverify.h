/*
 * specverify.h -- C ABI of libspecverify, the GB300 (sm_103a) speculative-
 * decoding verification step.
 *
 * The operation (page title, section):
 *  - "Speculative Decoding : accélérer l'inférence des LLM",
 *    §Principe et garanties mathématiques: a draft proposes gamma tokens, the
 *    target scores all of them in one pass, candidates are accepted while they
 *    are compatible and the first rejection is corrected by a token drawn from
 *    the target, so one cycle emits between 1 and gamma + 1 tokens;
 *    §Pourquoi la qualité est préservée: x is accepted with probability
 *    min(1, p(x)/q(x)); on rejection the replacement is drawn from p - q
 *    clipped at zero and renormalised; at temperature zero a token is
 *    accepted iff it equals the target argmax, else replaced by that argmax.
 *  - "Speculative Decoding — Come Accelerare l'Inferenza LLM di 2-3x Senza
 *    Perdere Qualità", §Il meccanismo: the later draft tokens are discarded
 *    after a rejection.
 *  - wiki "Speculative Decoding", §数式で見る speculative decoding の正しさ:
 *    eq. alpha(x) = min(1, p(x)/q(x)) and eq. p_corr(x) = max(p-q,0)/sum.
 *  - "Accélérer Sonar grâce à la spéculation", §Décodage spéculatif: with n
 *    draft tokens up to n + 1 tokens are emitted; the target logits at the
 *    mismatch position, or after the last draft token, give the extra token.
 *
 * Readings where the pages are silent: p = softmax(target_logits / T) and
 * q = softmax(draft_logits / T) with the request's temperature T; accept iff
 * u_accept < alpha; alpha = 1 when q(x) == 0 < p(x) and 0 when both are 0;
 * the replacement (or the extra token after gamma acceptances) is the
 * smallest k with C_k > u_sample * W, C_k the inclusive prefix sum of the
 * weights in index order and W their total (if rounding leaves none, the last
 * k with a positive weight); residual weights that sum to zero fall back to
 * p at that position; argmax ties go to the lowest index. Every finite T > 0
 * and every finite logit is verified: alpha is evaluated from the logits, so
 * it stays exact when p(x) and q(x) both lie below the floating-point range,
 * and rows whose logits are large against T (beyond about 5.8e6 T) or whose T
 * is so small that log2(e)/T overflows binary32 are summed from the
 * differences to the row max (2^((l - max) log2(e) / T)) instead of the
 * faster fused form, on both execution paths.
 *
 * Conventions for every entry point:
 *  - Memory: the caller owns every buffer. Array arguments of spec_verify and
 *    spec_verify_ex are DEVICE pointers on the current CUDA device. Nothing is
 *    allocated by the library.
 *  - Stream: work is enqueued on `stream` (NULL = the legacy default stream)
 *    and the call returns without waiting for it.
 *  - Layout: row-major and contiguous. Logit rows are V values; target row i
 *    of request b is at element (b*(gamma+1) + i)*V, draft row i at
 *    (b*gamma + i)*V. Row i scores draft token i; target row gamma is the
 *    bonus row.
 *  - Argument errors (NULL pointers, B < 0, gamma < 1, V < 1, an unknown
 *    dtype, a workspace too small, sizes above the limits below) are
 *    returned before anything is enqueued. B == 0 is a no-op.
 *  - Data errors never trap: a request whose temperature is NaN, negative or
 *    infinite, whose draft token lies outside [0, V), or whose rows hold a
 *    NaN, a +inf or only -inf values gets out_num_accepted = -1 and all its
 *    out_tokens -1; the draft rows of a T == 0 request are never read.
 *  - Determinism: the same inputs on the same device give bit-identical
 *    outputs.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The same type as the CUDA runtime's cudaStream_t. */
typedef struct CUstream_st* sv_stream_t;

typedef int32_t sv_dtype;
#define SV_F32 0  /* IEEE binary32 logits */
#define SV_BF16 1 /* bfloat16 logits (16-bit patterns) */

typedef int32_t sv_status;
#define SV_OK 0
#define SV_ERR_INVALID_ARG 1 /* a NULL pointer, a size out of range, an unknown dtype */
#define SV_ERR_UNSUPPORTED 2 /* no CUDA device, or not compute capability 10.3 */
#define SV_ERR_CUDA 3        /* a CUDA call failed while enqueueing */
#define SV_ERR_WORKSPACE 4   /* workspace NULL or smaller than the size query says */
#define SV_ERR_TIMEOUT 5     /* reserved for host-side waits; kernels report timeouts
                                through the device status word */
#define SV_ERR_SCRATCH_LIMIT 6 /* spec_verify_noalloc: the shape needs more scratch than
                                  SV_NOALLOC_SCRATCH_BYTES */

/* Bits of the optional device status word (int32), OR-ed in by the kernels. */
#define SV_STATUS_BAD_REQUEST 0x1 /* at least one request was invalid (-1) */
#define SV_STATUS_TIMEOUT 0x2     /* a bounded wait inside a streaming kernel ran
                                     out. Whether or not a status word was given, every
                                     request that was not final by then keeps
                                     out_num_accepted = -1 (the kernels write a count
                                     only once its request is final); its out_tokens
                                     may hold a partial result */
#define SV_STATUS_TRUNCATED 0x4   /* spec_commit: not every emitted token of a request
                                     fitted in its token buffer */

/* Size limits checked before launch. */
#define SV_MAX_GAMMA 64
#define SV_MAX_V (1 << 24)

/* Execution paths of spec_verify_ex (sv_options.path). */
#define SV_PATH_AUTO 0      /* the library chooses (the streaming path where it applies) */
#define SV_PATH_ROWWISE 1   /* one thread block per request; any V and alignment */
#define SV_PATH_STREAMING 2 /* persistent grid streaming all rows with bulk copies into
                               shared memory; needs V * element size to be a multiple of
                               16 bytes and 16-byte aligned logit pointers */
#define SV_PATH_CLUSTER 3   /* one thread-block cluster per request: each row cut into up to
                               16 slices, one per CTA, merged over distributed shared memory;
                               no workspace. Needs V * element size a multiple of 16 bytes,
                               16-byte aligned logits, V <= 2^20, no tree, no early exit */

/* Bytes of device workspace spec_verify needs for this shape on the current
 * device (the streaming path's per-row partial results, draw jobs, sampling
 * partial sums, and the header and completion counters it clears itself). Writes the size to *bytes. Needs the current CUDA
 * device to read its SM count; returns SV_ERR_UNSUPPORTED without one. */
sv_status spec_verify_workspace_size(int B, int gamma, int V, sv_dtype dtype, size_t* bytes);

/* The verification step.
 *  target_logits    [B, gamma+1, V] dtype, device.
 *  draft_logits     [B, gamma, V] dtype, device; rows of T == 0 requests are never read.
 *  draft_tokens     [B, gamma] int32, device.
 *  u_accept         [B, gamma] float, device, uniforms in [0, 1).
 *  u_sample         [B] float, device, uniforms in [0, 1).
 *  temperature      [B] float, device; 0 selects the greedy rule.
 *  out_tokens       [B, gamma+1] int32, device: the n accepted draft tokens,
 *                   then the replacement (n < gamma) or extra (n == gamma)
 *                   token, then -1.
 *  out_num_accepted [B] int32, device: n in [0, gamma], or -1 (invalid request).
 *  workspace        device, at least spec_verify_workspace_size() bytes,
 *                   16-byte aligned; its contents need no initialisation and
 *                   are overwritten. Two calls in flight at once must not share
 *                   a workspace.
 * Enqueues work on `stream` and returns SV_OK, or an error before enqueueing. */
sv_status spec_verify(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                      int B, int gamma, int V, const int32_t* draft_tokens,
                      const float* u_accept, const float* u_sample, const float* temperature,
                      int32_t* out_tokens, int32_t* out_num_accepted, void* workspace,
                      size_t workspace_bytes, sv_stream_t stream);

/* Optional per-row and per-request facts for checking, all DEVICE pointers,
 * each may be NULL. Entries the kernels do not compute are written as NaN
 * (floating point) or -1 (integers). lse is log sum_x exp(l(x)/T), the log
 * of the softmax normaliser. */
typedef struct {
    float* max_target;      /* [B*(gamma+1)] row max */
    double* lse_target;     /* [B*(gamma+1)] rows of T > 0 requests */
    int32_t* argmax_target; /* [B*(gamma+1)] rows of T == 0 requests */
    float* max_draft;       /* [B*gamma] rows of T > 0 requests */
    double* lse_draft;      /* [B*gamma] rows of T > 0 requests */
    double* p_x;            /* [B*gamma] p_i(x_i) at the positions evaluated (T > 0) */
    double* q_x;            /* [B*gamma] q_i(x_i) at the positions evaluated (T > 0) */
    double* w_total;        /* [B] total weight W of the replacement or extra draw (T > 0) */
    int32_t* kind;          /* [B] -1 invalid, 0 greedy, 1 residual draw, 2 extra-token draw */
    uint64_t* phase_ns;     /* [SV_PHASE_SLOTS] streaming path only: global-timer stamps
                               (ns). Slot 0 is the earliest block start and slot 1 the
                               latest; slots 2, 3, 4, 6, 7 and 9 are the latest time over
                               all blocks at which: 2 a block's row-statistics stream
                               ended, 3 an acceptance scan ended, 4 a block's producer
                               took its first draw job, 6 a block's draw stream ended,
                               7 a token search ended, 9 a block ended. Slots 5 and 8
                               are not written; 4, 6 and 7 stay untouched when no request
                               has T > 0. The caller fills slot 0 with UINT64_MAX and the
                               others with 0 before the call. */
} sv_debug_out;

#define SV_PHASE_SLOTS 10

typedef struct {
    int32_t path;      /* SV_PATH_* */
    int32_t grid_ctas; /* streaming path: thread blocks in the persistent grid; 0 = the
                          device's full co-resident grid. Smaller grids split rows over
                          fewer blocks (used by tests to exercise every split). */
    int32_t peer_wait_us; /* streaming path: limit of each wait on work of other thread
                             blocks (a draw job to be published, the hold flag), in
                             microseconds; 0 = the default (about 2 s). A block whose wait
                             runs out sets SV_STATUS_TIMEOUT, ends its draw phase and
                             returns; the call's outputs are then not valid. */
    int32_t early_exit; /* non-zero: early-exit verification. Positions are taken in
                           order and nothing after a request's first rejection (first
                           mismatch at T = 0) is read: same outputs, fewer bytes; a
                           request is then invalid only when a row it reads is bad.
                           Checking outputs hold NaN / -1 for the rows not read. */
    const int32_t* hold_flag; /* streaming path, checking only; NULL normally. A device
                                 int32: every block waits, for at most peer_wait_us, until
                                 it is non-zero before its draw phase. A flag nothing sets
                                 makes every such wait run out, which exercises the
                                 SV_STATUS_TIMEOUT report deterministically. */
    const int32_t* num_draft; /* one-hot proposals only (draft_logits NULL): device [B]
                                 int32 proposals per request, see spec_verify_onehot;
                                 NULL = gamma each */
} sv_options;

/* spec_verify with checking outputs and options. `dbg`, `d_status` and
 * `opts` may be NULL. `d_status` is a device int32 into which the kernels OR
 * SV_STATUS_* bits; the caller clears it. `draft_logits` NULL selects
 * deterministic (one-hot) proposals with opts->num_draft, as
 * spec_verify_onehot. */
sv_status spec_verify_ex(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                         int B, int gamma, int V, const int32_t* draft_tokens,
                         const float* u_accept, const float* u_sample, const float* temperature,
                         int32_t* out_tokens, int32_t* out_num_accepted, void* workspace,
                         size_t workspace_bytes, sv_stream_t stream, const sv_debug_out* dbg,
                         int32_t* d_status, const sv_options* opts);

/* Bytes of device staging memory spec_verify_host needs (inputs, outputs and
 * workspace) on the current device. */
sv_status spec_verify_host_staging_size(int B, int gamma, int V, sv_dtype dtype, size_t* bytes);

/* The verification step on HOST buffers: the same arguments as spec_verify
 * with every array in host memory (page-locked memory keeps the copies
 * asynchronous), plus one caller-owned DEVICE staging buffer of
 * spec_verify_host_staging_size() bytes. Enqueues on `stream`: the host to
 * device copies of the inputs (draft rows only for T > 0 requests, whose
 * temperatures the host reads here), the verification, and the device to
 * host copies of out_tokens and out_num_accepted. The outputs are valid once
 * the stream has reached that point (e.g. after cudaStreamSynchronize).
 * The host link is ~30x slower than HBM, so a batch of more than 64 MB of
 * inputs is cut into up to 8 request slices (each >= 32 MB): the copies run on
 * a library-owned copy stream of the current device, and `stream` verifies
 * slice k (one spec_verify launch) as soon as it has landed, while slice k + 1
 * is still being copied. The copies first wait for the work already on
 * `stream`; `stream` waits for every copy, so the call stays ordered on it
 * like one operation. Requests are independent: the outputs are those of one
 * spec_verify over the whole batch (within the parity bar: row sums split at
 * other places). The first call on a device creates that copy stream and its
 * events, kept until the process exits (make it outside stream capture);
 * calls take a lock while they enqueue. Calls that overlap on one staging
 * buffer from different streams race on it. */
sv_status spec_verify_host(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                           int B, int gamma, int V, const int32_t* draft_tokens,
                           const float* u_accept, const float* u_sample,
                           const float* temperature, int32_t* out_tokens,
                           int32_t* out_num_accepted, void* staging, size_t staging_bytes,
                           sv_stream_t stream);

/* Size of the static scratch of spec_verify_noalloc: 8 MiB of device memory,
 * held on every GPU that loads this library until the process exits. */
#define SV_NOALLOC_SCRATCH_BYTES (8u << 20)

/* spec_verify without a workspace argument, for callers that cannot allocate
 * device memory: a plugin that a host runtime gives only its input and output
 * tensors, or a serving loop whose device memory is fixed at start-up and that
 * must not call cudaMalloc on its hot path (cudaMalloc may synchronize the
 * device). The pages describe no such entry point; it has no counterpart
 * there. Arguments and results are those of spec_verify; it always runs the
 * streaming path, so V * element size must be a multiple of 16 bytes, the
 * logit pointers 16-byte aligned and B at most 4096 (else SV_ERR_INVALID_ARG).
 * Its scratch is a static device array of SV_NOALLOC_SCRATCH_BYTES inside the
 * library; a shape that needs more returns SV_ERR_SCRATCH_LIMIT before
 * anything is enqueued. Nothing is allocated: no cudaMalloc, no cudaFree.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current, and keeps it with the
 * driver's id of the current context; a call in another context (after a
 * device reset, say) looks it up again. Make the first call on a device, and
 * the first after a reset, before any stream capture. All calls in the
 * process share the one array, which keeps the previous call's contents (the
 * call clears the part that must start at zero itself): two calls that
 * overlap on the GPU, on any streams, race on it and give undefined results.
 * There is no status word: if a bounded wait inside the kernel runs out (see
 * SV_STATUS_TIMEOUT), every request that was not final keeps
 * out_num_accepted = -1. */
sv_status spec_verify_noalloc(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                              int B, int gamma, int V, const int32_t* draft_tokens,
                              const float* u_accept, const float* u_sample, const float* temperature,
                              int32_t* out_tokens, int32_t* out_num_accepted, sv_stream_t stream);

/* Number of kernel launches the last successful spec_verify* call on this
 * host thread enqueued (memsets and copies not counted). */
int spec_verify_last_launch_count(void);

/* A static English description of a status code. */
const char* spec_verify_status_string(sv_status status);

/* Library version: major * 10000 + minor * 100 + patch. */
int spec_verify_version(void);

/* ---------------------------------------------------------------------------
 * Verification of deterministic proposals ("Speculative Decoding : accélérer
 * l'inférence des LLM", §N-gram lookup et variantes sans modèle: the draft
 * tokens come from a lookup, not from a model). Such a proposer puts all its
 * probability on the token it proposes, so q_i is one-hot at x_i and the rule
 * of §Pourquoi la qualité est préservée becomes: accept x_i iff
 * u_accept < min(1, p_i(x_i)); at the first rejection n, draw from p_n
 * without x_n (max(p_n - q_n, 0) renormalised); after k acceptances draw the
 * extra token from target row k. T == 0 is the greedy rule. No draft logits
 * are read (half the bytes of spec_verify at equal gamma).
 *   num_draft  [B] int32, device: request b proposes num_draft[b] in
 *              [0, gamma] tokens, draft_tokens[b, :num_draft[b]]; the rest of
 *              its row is ignored, and so are its target rows past
 *              num_draft[b] (a NaN there is not an error). A count outside
 *              [0, gamma] makes the request invalid (-1, SV_STATUS_BAD_REQUEST).
 * Every other argument, the outputs, the workspace (spec_verify_workspace_size)
 * and the error behaviour are those of spec_verify. */
sv_status spec_verify_onehot(const void* target_logits, sv_dtype dtype, int B, int gamma, int V,
                             const int32_t* draft_tokens, const int32_t* num_draft, const float* u_accept,
                             const float* u_sample, const float* temperature, int32_t* out_tokens,
                             int32_t* out_num_accepted, void* workspace, size_t workspace_bytes,
                             sv_stream_t stream);

/* ---------------------------------------------------------------------------
 * Tree verification ("Speculative Decoding : accélérer l'inférence des LLM",
 * §Medusa : plusieurs têtes de prédiction and §EAGLE: candidate continuations
 * arranged in a tree, verified in one target pass). The pages do not state the
 * rule for several candidates; this library applies the acceptance rule of
 * §Pourquoi la qualité est préservée candidate after candidate, with
 * deterministic candidates (q one-hot), which keeps the target distribution:
 *  - node 0 is the root; node j in 1..num_nodes[b] has token
 *    node_tokens[b, j-1] and parent parents[b, j-1] in [0, j-1]; target row j
 *    ([B, gamma+1, V], row-major) holds the logits for the token after node j
 *    (row 0: after the context);
 *  - at node u the children are tried in index order; child c is accepted iff
 *    u_accept[b, c-1] < min(1, p'(x_c)), p' = softmax(row u / T) without the
 *    tokens of the children rejected so far, renormalised; it becomes u;
 *  - when every child is rejected, or u is a leaf, the last token is drawn from
 *    p' with u_sample[b] by inverse CDF;
 *  - T == 0: the first child whose token is the argmax of row u is taken;
 *    with none, the argmax ends the walk.
 * A chain (parents[b, j-1] = j-1) gives spec_verify_onehot.
 *   out_tokens [B, gamma+1]: the accepted path's tokens, the last token, -1
 *   out_num_accepted [B]: path length (-1: invalid request)
 *   out_nodes [B, gamma] or NULL: the accepted node indices, then -1
 *   dbg, d_status: as spec_verify_ex (p_x, q_x indexed by node - 1), may be NULL
 * Invalid requests (-1, SV_STATUS_BAD_REQUEST): T NaN, negative or infinite;
 * num_nodes[b] outside [0, gamma]; a parent not an earlier node; a token
 * outside [0, V); a bad row among 0..num_nodes[b]. Rows past num_nodes[b] are
 * not read.
 *   workspace, workspace_bytes: as spec_verify (spec_verify_workspace_size of
 *              the same B, gamma, V, dtype); NULL keeps the call on one thread
 *              block per request, which needs none (SV_PATH_STREAMING with a
 *              NULL or short workspace returns SV_ERR_WORKSPACE)
 *   opts       NULL, or path, grid_ctas, peer_wait_us and hold_flag as in
 *              spec_verify_ex; early_exit must be 0 and num_draft is not read
 *              (SV_ERR_INVALID_ARG otherwise). */
sv_status spec_verify_tree(const void* target_logits, sv_dtype dtype, int B, int gamma, int V,
                           const int32_t* node_tokens, const int32_t* parents, const int32_t* num_nodes,
                           const float* u_accept, const float* u_sample, const float* temperature,
                           int32_t* out_tokens, int32_t* out_num_accepted, int32_t* out_nodes, void* workspace,
                           size_t workspace_bytes, sv_stream_t stream, const sv_debug_out* dbg, int32_t* d_status,
                           const sv_options* opts);

/* ---------------------------------------------------------------------------
 * Post-verify bookkeeping ("Accélérer Sonar grâce à la spéculation",
 * §Planification MTP pour un jeton unique: a kernel inserts the next target
 * tokens into their slots, so the accepted length needs no CPU
 * synchronisation before the next step; "Speculative Decoding : accélérer
 * l'inférence des LLM", §Principe et garanties mathématiques: a pass emits
 * the n accepted draft tokens and one token of the target).
 *
 * Appends the tokens request b emitted, out_tokens[b, 0..n] with
 * n = out_num_accepted[b], to token_buf[b] at seq_lens[b] and advances
 * seq_lens[b]. All pointers are DEVICE pointers owned by the caller; the call
 * enqueues one kernel on `stream` and returns without synchronising.
 *   out_tokens        [B, gamma+1] int32 (spec_verify's output)
 *   out_num_accepted  [B] int32
 *   token_buf         [B, max_len] int32, row-major; updated in place
 *   seq_lens          [B] int32; updated in place
 *   next_input        [B] int32 or NULL: the last token of each history after
 *                     the commit (the next draft step's input), -1 if empty
 *   d_status          int32 or NULL; the kernel ORs in
 *                     SV_STATUS_BAD_REQUEST: n outside [0, gamma], a negative
 *                       emitted token, or seq_lens[b] outside [0, max_len];
 *                       that request is left unchanged, next_input[b] = -1;
 *                     SV_STATUS_TRUNCATED: not every emitted token fitted in
 *                       max_len; the ones that fit are appended.
 * Returns SV_ERR_INVALID_ARG for B < 0, gamma outside [1, SV_MAX_GAMMA],
 * max_len < 1 or a NULL required pointer (nothing enqueued); B == 0 enqueues
 * nothing. */
sv_status spec_commit(const int32_t* out_tokens, const int32_t* out_num_accepted, int B, int gamma,
                      int32_t* token_buf, int max_len, int32_t* seq_lens, int32_t* next_input,
                      int32_t* d_status, sv_stream_t stream);

/* ---------------------------------------------------------------------------
 * Model-free draft tokens by n-gram (prompt) lookup ("Speculative Decoding :
 * accélérer l'inférence des LLM", §N-gram lookup et variantes sans modèle:
 * find the context's last n tokens earlier in the context and propose the
 * tokens that followed them; §Mise en œuvre dans vLLM: prompt_lookup_min = 2,
 * prompt_lookup_max = 5). The page leaves open which occurrence and what to
 * do at the end of the history; this library takes: n from n_max down to
 * n_min, the first (longest) n with an earlier occurrence wins; of its
 * occurrences ending at or before L - 1 the latest is used; the proposal is
 * the up to gamma tokens that follow it, cut at the end of the history.
 *
 * All pointers are DEVICE pointers owned by the caller; one kernel on
 * `stream`, no synchronisation.
 *   token_buf     [B, max_len] int32: request b's history is
 *                 token_buf[b, :seq_lens[b]] (prompt and generated tokens)
 *   seq_lens      [B] int32
 *   draft_tokens  [B, gamma] int32 out: the proposal, then -1
 *   num_draft     [B] int32 out: proposal length k in [0, gamma] (0: none)
 *   d_status      int32 or NULL: ORs SV_STATUS_BAD_REQUEST for a length
 *                 outside [0, max_len] (that request proposes nothing)
 * Returns SV_ERR_INVALID_ARG for B < 0, max_len < 1, gamma outside
 * [1, SV_MAX_GAMMA], n_min < 1, n_max < n_min, n_max > SV_NGRAM_MAX_N or a
 * NULL required pointer; B == 0 enqueues nothing. */
#define SV_NGRAM_MAX_N 16
sv_status spec_ngram_propose(const int32_t* token_buf, int B, int max_len, const int32_t* seq_lens,
                             int gamma, int n_min, int n_max, int32_t* draft_tokens, int32_t* num_draft,
                             int32_t* d_status, sv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
