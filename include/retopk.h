/*
 * retopk.h -- C ABI of the GB300 (sm_103a) decode-time Top-K sparse attention
 * library: ReTopK similarity-guided support reuse and the Exact Top-K path it
 * falls back to.
 *
 * Method: "Recall Before You Rank: Similarity-Guided Top-K Reuse for Efficient
 * Long-Context Attention" (ReTopK), §Methodology.  Each entry point names the
 * equations it executes.
 *
 * Conventions shared by every entry point
 *   - Tensors are raw device pointers owned by the caller.  bf16 tensors are
 *     passed as retopk_bf16 (the IEEE bfloat16 bit pattern).  Every tensor must
 *     be 16-byte aligned and contiguous in the layout stated for it.
 *   - head_dim d must be 128.  Query head h reads KV head h / (Hq / Hkv)
 *     (consecutive GQA groups).
 *   - K cache / V cache layout: [B, Hkv, max_len, d] bf16, row-major.  Row i of
 *     (b, h_kv) is the key (value) of token i, 0-based.
 *   - seqlens: device int32 [B].  seqlens[b] = L_b, the number of valid rows of
 *     sequence b, INCLUDING the token being decoded (its key and value are in
 *     the cache before the step runs).
 *   - `stream` is a cudaStream_t.  Every call is asynchronous on it, never
 *     synchronises the device (except where stated: create, init, export,
 *     import, status and counter reads) and never allocates device memory:
 *     the caller provides the workspace.
 *   - The library's kernels use programmatic dependent launch among
 *     themselves, and the last kernel of a call may let the next grid on the
 *     stream launch before it completes.  A plain launch after a
 *     call is ordered as usual; a kernel the caller launches with
 *     programmatic stream serialisation behind a call must wait for its grid
 *     dependency (griddepcontrol.wait / cudaGridDependencySynchronize) before
 *     it reads the call's outputs.
 *   - Return value: RETOPK_OK (0) or a negative RETOPK_ERR_* code.  Argument
 *     errors are detected on the host before anything is launched.  Faults the
 *     device detects (an out-of-range support index in the cache, a full KV
 *     cache on append) set bits in a sticky status word (retopk_get_status);
 *     no kernel traps or asserts.
 *   - Top-K ties are broken towards the lower key index; when fewer than K
 *     keys (or candidates) exist, the support is all of them.
 */
#ifndef RETOPK_H
#define RETOPK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t retopk_bf16;           /* raw bfloat16 bits */
typedef struct retopk_ctx retopk_ctx;   /* opaque, host-side */

enum {
    RETOPK_OK = 0,
    RETOPK_ERR_INVALID = -1,      /* bad pointer, size or hyper-parameter           */
    RETOPK_ERR_UNSUPPORTED = -2,  /* head_dim != 128, group too large, length too big */
    RETOPK_ERR_WORKSPACE = -3,    /* workspace too small or misaligned              */
    RETOPK_ERR_CUDA = -4,         /* a CUDA runtime call or launch failed           */
    RETOPK_ERR_ALIGN = -5,        /* a tensor pointer is not 16-byte aligned        */
    RETOPK_ERR_STATE = -6,        /* state buffer of the wrong size or version      */
    RETOPK_ERR_SCRATCH = -7       /* exceeds the static scratch of the _noalloc call */
};

/* Status bits (sticky, set by device code). */
#define RETOPK_STATUS_BAD_INDEX   0x1u  /* cached support index outside [0, L)      */
#define RETOPK_STATUS_KV_FULL     0x2u  /* append with seqlens[b] == max_len        */
#define RETOPK_STATUS_NONFINITE   0x4u  /* a non-finite score was produced          */
#define RETOPK_STATUS_TIMEOUT     0x8u  /* a bounded pipeline wait expired (the step's
                                           results are not valid)                  */
#define RETOPK_STATUS_GATHER      0x10u /* a gathered K/V row index outside [0, L) was
                                          skipped: checked by builds with
                                          RETOPK_CHECKED defined, and always by
                                          retopk_fidelity (against max_len)      */

/* Path codes reported per (sequence, query head), Eq. (13). */
#define RETOPK_PATH_REUSE    0
#define RETOPK_PATH_FALLBACK 1          /* rho_max < tau                            */
#define RETOPK_PATH_REFRESH  2          /* T_r > 0 and t_dec a multiple of T_r       */

/* ReTopK hyper-parameters (§Reliable Reuse, §Implementation settings):
 * K support size, C cache capacity, W recent window, R retrieved entries,
 * T_r refresh period (0 disables refresh), tau similarity threshold.
 * Limits: d = 128; 1 <= Hq/Hkv <= 16; B * Hkv <= 512; 1 <= K <= 4096;
 * 1 <= R <= C <= 256; 0 <= W; R*K + W <= 18432; max_len <= 2^23 and
 * B * Hkv * max_len <= 2^29; B * Hq * C * K < 2^31.  The reuse path keeps, per
 * CTA of a head's cluster of CL (`cluster`; 8 when chosen automatically and
 * the smaller sizes do not fit), a bitmap over max_len/CL key positions and
 * three lists of R*K + W words in shared memory, which must fit 227 KB:
 * 5376 + 4 * (max(ceil(max_len/CL)/32, R*K + W) + max(R*K + W, 3096) + R*K + W)
 * bytes, each count of words rounded up to 32 positions or 4 words (e.g., at
 * CL = 8, max_len = 2^23 with R*K + W = 2080, or R*K + W = 18432 with
 * max_len <= 5095424).  Larger combinations return RETOPK_ERR_UNSUPPORTED. */
typedef struct retopk_config {
    int32_t batch;        /* B                                                  */
    int32_t n_q_heads;    /* Hq                                                 */
    int32_t n_kv_heads;   /* Hkv, divides Hq                                    */
    int32_t head_dim;     /* d, must be 128                                     */
    int32_t max_len;      /* rows per (b, h_kv) in the caller's KV cache        */
    int32_t K, C, W, R, T_r;
    float tau;
    int32_t retrieval;    /* RETOPK_RETRIEVE_SIMILAR (0): the R most similar
                             cached queries, Eq. (7) -- the method; or
                             RETOPK_RETRIEVE_RECENT (1): the R most recent
                             entries, rho_max over them (the paper's Table 3
                             "recent-R retrieval" ablation)                  */
    int32_t cluster;      /* CTAs per head in the step's back end (reuse body
                             and exact select): 0 chooses -- the largest of
                             8, 4, 2, 1 for which one wave of B*Hq clusters
                             fits the GPU at two CTAs per SM, raised while
                             the reuse path's candidate bitmap (L / cluster
                             positions per CTA) would not fit its shared
                             memory; or 1, 2, 4, 8 to fix it.  Results do not
                             depend on it.  The stateless exact step chooses
                             the same way for its B*Hq heads.            */
} retopk_config;
#define RETOPK_RETRIEVE_SIMILAR 0
#define RETOPK_RETRIEVE_RECENT  1

/* ---- context ------------------------------------------------------------ */

/* Bytes of device workspace a context with this configuration needs.
 * Returns 0 if the configuration is invalid. */
size_t retopk_workspace_bytes(const retopk_config *cfg);

/* Creates a context that keeps all its state (the per-head query-support
 * cache of Eq. (5), decode counters, scratch) in the caller's device
 * workspace `d_workspace` (>= retopk_workspace_bytes, 256-byte aligned).
 * The context object itself is host memory owned by the library; free it
 * with retopk_destroy.  Synchronises the current device once (clears the
 * workspace).  The workspace must outlive the context. */
int retopk_create(const retopk_config *cfg, void *d_workspace, size_t bytes, retopk_ctx **out);
int retopk_destroy(retopk_ctx *ctx);

/* The same context with its device memory in two parts, so that several
 * contexts -- the layers of a model, each with its own configuration of the
 * same sizes and its own caches -- can share the larger one.
 *   state   (>= retopk_state_workspace_bytes, 256-byte aligned): the context's
 *           own query-support cache (Eq. (5)), ring words, counters and status
 *           word; cleared here.
 *   scratch (>= retopk_scratch_bytes, 256-byte aligned): what a decode step
 *           writes and reads within the step (path decisions, candidate lists,
 *           scores, histograms) and the last step's diagnostics.  Contexts may
 *           share one scratch when their calls never overlap on the GPU: calls
 *           on one stream one after another (captured into one graph or not) are
 *           fine, calls on concurrent streams are not.  retopk_get_diagnostics
 *           and retopk_fidelity report the last step run with the scratch, by
 *           whichever context.
 * (The ReTopK paper's fused implementation likewise reuses per-layer
 * workspaces, §Experiments Table 4.)  Synchronises the current device once.
 * Both buffers must outlive the context. */
size_t retopk_state_workspace_bytes(const retopk_config *cfg);
size_t retopk_scratch_bytes(const retopk_config *cfg);
int retopk_create_shared(const retopk_config *cfg, void *d_state, size_t state_bytes, void *d_scratch,
                         size_t scratch_bytes, retopk_ctx **out);

/* ---- ReTopK decode ------------------------------------------------------ */

/* Cache initialisation from the final C prompt tokens (§Recall-Before-Rerank,
 * "query-support cache"): for prompt position p = L0_b - C + c, c = 0..C-1,
 * stores the query and its Exact Top-K support over the causal prefix
 * 0..p (Eq. (1)).  q_last: [B, Hq, C, d] bf16, the queries of positions
 * L0-C .. L0-1.  d_prompt_len: device int32 [B] = L0_b (each >= C).
 * Resets the decode counter t_dec to 0.  Synchronises `stream` once to read
 * the prompt lengths (set-up, not part of the decode step). */
int retopk_init_cache(retopk_ctx *ctx, const retopk_bf16 *q_last, const retopk_bf16 *k_cache,
                      const int32_t *d_prompt_len, void *stream);

/* Appends one token per sequence: writes k_new / v_new ([B, Hkv, d]) into
 * row seqlens[b] of the caches and increments seqlens[b] on the device.
 * A full cache (seqlens[b] == max_len) sets RETOPK_STATUS_KV_FULL and leaves
 * that sequence unchanged.  Graph-capturable. */
int retopk_append_kv(retopk_ctx *ctx, const retopk_bf16 *k_new, const retopk_bf16 *v_new,
                     retopk_bf16 *k_cache, retopk_bf16 *v_cache, int32_t *d_seqlens,
                     void *stream);

/* One ReTopK decode step for every (sequence, query head):
 *   Eq. (6)-(7)  cosine recall of q against the head's cached queries, Top-R
 *   Eq. (13)     path: refresh / similarity fallback / reuse (decided on device)
 *   reuse:       Eq. (8)-(9) candidates = retrieved supports U recent window,
 *                Eq. (10) exact rerank scores of the candidates only,
 *                Eq. (11) Top-K of the candidates
 *   exact:       Eq. (4) full-history scores, Eq. (1) global Top-K
 *   both:        Eq. (12) softmax-value aggregation over the support, then the
 *                cache insertion of (q, support) and t_dec += 1.
 * q: [B, Hq, d] bf16; out: [B, Hq, d] bf16.  No host round trip: the path
 * switch lives on the device, so the call can be captured in a CUDA graph.
 * Three kernels on `stream`: the path decision, the scan of the KV groups
 * with an exact-path head, and one back-end launch serving every head on its
 * path. */
int retopk_decode_step(retopk_ctx *ctx, const retopk_bf16 *q, const retopk_bf16 *k_cache,
                       const retopk_bf16 *v_cache, const int32_t *d_seqlens,
                       retopk_bf16 *out, void *stream);

/* retopk_append_kv followed by retopk_decode_step, in one fewer launch: the
 * path-decision kernel also writes the new K/V rows and advances the length
 * (same results, same KV_FULL behaviour; the ReTopK paper has no separate
 * notion of this fusion -- it is the decode step with the token's K/V append
 * of Eq. (4)'s L_t folded in).  k_new / v_new: [B, Hkv, d] bf16.
 * Graph-capturable. */
int retopk_decode_step_kv(retopk_ctx *ctx, const retopk_bf16 *k_new, const retopk_bf16 *v_new,
                          const retopk_bf16 *q, retopk_bf16 *k_cache, retopk_bf16 *v_cache,
                          int32_t *d_seqlens, retopk_bf16 *out, void *stream);

/* retopk_decode_step_kv with the token's inputs and the output in HOST memory
 * (pageable or pinned): k_new / v_new [B, Hkv, d], q [B, Hq, d], out
 * [B, Hq, d], all bf16 on the host; k_cache, v_cache, d_seqlens stay on the
 * device.  Synchronous: returns once `out` holds the step's output.  The
 * inputs are copied into library-owned pinned, device-mapped memory; the
 * kernels of retopk_decode_step_kv are replayed as a CUDA graph on
 * `stream` (captured on the first call and again whenever k_cache, v_cache or
 * d_seqlens change), the path-decision kernel reading the token's q, k_new,
 * v_new across the host link (and copying q to device memory for the later
 * kernels) and the back end writing the output rows into the mapped buffer,
 * which is then copied to `out`.  The first call allocates the pinned host
 * staging (2 B Hq d * 2 + 2 B Hkv d * 2 bytes), freed by retopk_destroy; the
 * device copy of q is part of the workspace (no device allocation).  Not to be called from several threads on one
 * context; on a capturing stream it returns RETOPK_ERR_INVALID.  Same
 * results as retopk_decode_step_kv on the same inputs. */
int retopk_decode_step_host(retopk_ctx *ctx, const retopk_bf16 *k_new, const retopk_bf16 *v_new,
                            const retopk_bf16 *q, retopk_bf16 *k_cache, retopk_bf16 *v_cache,
                            int32_t *d_seqlens, retopk_bf16 *out, void *stream);

/* Per-step diagnostics of the last decode step, copied to HOST buffers
 * (synchronises `stream`).  Any pointer may be NULL.
 *   path     [B*Hq] int32   RETOPK_PATH_*
 *   rho_max  [B*Hq] float   max cosine (-inf for an empty cache)
 *   topR     [B*Hq*R] int32 retrieved entries as logical positions
 *                           (0 = oldest live entry), -1 padded
 *   M        [B*Hq] int32   |A_t| on reuse heads, L on exact heads
 *   cand     [B*Hq*(R*K+W)] int32  A_t ascending on reuse heads, -1 padded
 *   support  [B*Hq*K] int32 the selected support ascending, -1 padded
 *   sup_len  [B*Hq] int32
 *   out_f32  [B*Hq*d] float the step output before bf16 rounding */
int retopk_get_diagnostics(retopk_ctx *ctx, int32_t *path, float *rho_max, int32_t *topR,
                           int32_t *M, int32_t *cand, int32_t *support, int32_t *sup_len,
                           float *out_f32, void *stream);

/* Path counters since create/init (host buffers, synchronises):
 * counts[0..2] = steps x heads on reuse / fallback / refresh,
 * counts[3] = sum of M_t over reuse head-steps, counts[4] = max M_t. */
int retopk_get_counters(retopk_ctx *ctx, int64_t counts[5], void *stream);

/* Cache state export / import (checkpoint, and state-forced testing).
 * Host buffer layout, little-endian, contiguous:
 *   fifo_q   [B, Hq, C, d]  uint16 (raw bf16 query bits)
 *   fifo_sup [B, Hq, C, K]  int32  (ascending support, -1 padded)
 *   fifo_len [B, Hq, C]     int32
 *   seq      [B, 3]         int32  (next slot, live count, t_dec)
 * Live entry c (0 = oldest) of sequence b sits in slot
 * (seq[b][0] - seq[b][1] + c) mod C.  Both calls synchronise `stream`.
 * Import refuses (RETOPK_ERR_STATE, device untouched) a slot or count out of
 * range, a length outside [0, K], and a support whose first `len` entries are
 * not strictly ascending and nonnegative; a support index at or beyond the
 * sequence's current length is reported when a step reads it
 * (RETOPK_STATUS_BAD_INDEX) and left out of the candidates. */
size_t retopk_state_bytes(const retopk_ctx *ctx);
int retopk_export_state(retopk_ctx *ctx, void *host_buf, size_t bytes, void *stream);
int retopk_import_state(retopk_ctx *ctx, const void *host_buf, size_t bytes, void *stream);

/* Sticky device status word (RETOPK_STATUS_* bits); `clear` resets it.
 * Synchronises `stream`. */
int retopk_get_status(retopk_ctx *ctx, uint32_t *bits, int clear, void *stream);

/* Failure-path self-test: launches one thread that waits on a barrier nothing
 * arrives on, gives up after `wait_cycles` SM clock cycles (0..8e9), sets
 * RETOPK_STATUS_TIMEOUT in the context's status word and returns -- the same
 * bounded-wait path every pipeline wait of the scan kernel takes.  The
 * context stays usable.  Asynchronous on `stream`. */
int retopk_selftest_wait(retopk_ctx *ctx, int64_t wait_cycles, void *stream);

const char *retopk_strerror(int code);

/* The CUDA runtime's message for the last CUDA error that made a call of this
 * thread return RETOPK_ERR_CUDA (a static string; never NULL). */
const char *retopk_cuda_error_string(void);

/* ---- Exact Top-K (stateless) -------------------------------------------- */

/* Device workspace for exact_topk_attention_step with these sizes
 * (0 if invalid). */
size_t exact_topk_workspace_bytes(int B, int Hq, int Hkv, int d, int max_len, int K);

/* Exact Top-K attention (§Motivation Eq. (1), §Problem Setup Eq. (4),
 * §Recall-Before-Rerank Eq. (12)): for every (b, h) scores all L_b keys,
 * selects the K best (ties to the lower index) and aggregates their values
 * with softmax weights.  q: [B, Hq, d]; out: [B, Hq, d] bf16.
 * idx_out: optional device int32 [B, Hq, K], the support ascending, -1
 * padded when L_b < K.  d_workspace: >= exact_topk_workspace_bytes,
 * 256-byte aligned.  Graph-capturable. */
int exact_topk_attention_step(const retopk_bf16 *q, const retopk_bf16 *k_cache,
                              const retopk_bf16 *v_cache, const int32_t *d_seqlens,
                              int B, int Hq, int Hkv, int d, int max_len, int K,
                              retopk_bf16 *out, int32_t *idx_out,
                              void *d_workspace, size_t bytes, void *stream);

/* The two halves of exact_topk_attention_step, for callers that place other
 * work between them or time them apart; run back to back on one stream with
 * the same workspace (and the same q, seqlens and sizes) they give the same
 * results as exact_topk_attention_step.
 *   exact_topk_scan:   §Problem Setup Eq. (4), e_i = q.k_i / sqrt(d) for every
 *                      key of every (b, h), left in the workspace together with
 *                      the histogram of their first radix digit (the
 *                      workspace's histograms are cleared first).
 *   exact_topk_select: §Motivation Eq. (1), the K best of those scores (ties
 *                      to the lower index), then §Recall-Before-Rerank
 *                      Eq. (12) over them; out / idx_out as for
 *                      exact_topk_attention_step.
 * The select half must follow a scan half with the same workspace; anything
 * else that writes the workspace in between invalidates it.  Both are
 * asynchronous on `stream` and graph-capturable. */
int exact_topk_scan(const retopk_bf16 *q, const retopk_bf16 *k_cache, const int32_t *d_seqlens, int B, int Hq,
                    int Hkv, int d, int max_len, int K, void *d_workspace, size_t bytes, void *stream);
int exact_topk_select(const retopk_bf16 *q, const retopk_bf16 *v_cache, const int32_t *d_seqlens, int B, int Hq,
                      int Hkv, int d, int max_len, int K, retopk_bf16 *out, int32_t *idx_out, void *d_workspace,
                      size_t bytes, void *stream);

/* Allocation-free variant of exact_topk_attention_step (the paper has no
 * counterpart; it exists for callers that cannot allocate device memory at
 * all -- code where allocation is forbidden or unavailable, e.g. an external
 * memory manager owning the whole device, or a plain C host with no allocator
 * to provide a workspace).  Same inputs, outputs and results as
 * exact_topk_attention_step, but the scratch comes from one 16 MiB file-scope
 * device array in the library instead of a caller workspace, so the call
 * allocates nothing (no cudaMalloc / cudaFree, no allocating library call).
 *   - Sizes whose workspace (exact_topk_workspace_bytes) exceeds 16 MiB are
 *     rejected with RETOPK_ERR_SCRATCH before anything is launched (at
 *     Hq = 28, Hkv = 4, K = 512 and B = 1 that allows max_len <= 49024).
 *   - The array is shared by every call in the process and keeps the last
 *     call's contents; each call clears what must start at zero.  Calls that
 *     overlap on the GPU (other streams, other threads) race on it.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - The 16 MiB are reserved on a device when the library's module is loaded
 *     there.  Under CUDA's default lazy module loading that is this first
 *     call, which can therefore return RETOPK_ERR_CUDA if the device has no
 *     16 MiB left: make it at start-up.  From then on the device holds the
 *     array until the process exits, and no later call takes device memory. */
int exact_topk_attention_step_noalloc(const retopk_bf16 *q, const retopk_bf16 *k_cache,
                                      const retopk_bf16 *v_cache, const int32_t *d_seqlens,
                                      int B, int Hq, int Hkv, int d, int max_len, int K,
                                      retopk_bf16 *out, int32_t *idx_out, void *stream);

/* ---- fidelity diagnostics ------------------------------------------------ */

/* Attention-support fidelity of the last decode step (ReTopK paper,
 * §Experiments "Attention-support fidelity", Figs. 5-6; §Motivation
 * Eq. (2)): for every (sequence, query head), the support that step used
 * (its reranked support on the reuse path) against `exact_idx`, the Exact
 * Top-K support of the same query (e.g. idx_out of exact_topk_attention_step
 * run on the same q and caches), and the step's output `out` against the
 * exact output `out_exact`.  Scores are recomputed from q and k_cache (call it
 * before the caches change).  metrics: device float [B, Hq, 4] =
 *   [0] support recall |S^ n S| / |S|,
 *   [1] retained mass: the Exact Top-K softmax mass that falls on S^,
 *   [2] cosine of the two head outputs,
 *   [3] cosine of the two attention distributions.
 * exact_idx: [B, Hq, K] int32 ascending, -1 padded; out / out_exact / q:
 * [B, Hq, d] bf16.  An exact_idx entry outside [0, max_len) is not read (it
 * scores 0) and sets RETOPK_STATUS_GATHER in the context's status word.
 * A diagnostic beside the decode loop, not part of it. */
int retopk_fidelity(retopk_ctx *ctx, const retopk_bf16 *q, const retopk_bf16 *k_cache, const int32_t *exact_idx,
                    const retopk_bf16 *out_exact, const retopk_bf16 *out, float *metrics, void *stream);

/* Support overlap and coverage (ReTopK paper, §Motivation Eqs. (2)-(3)): for
 * each of `rows` rows, S [rows, K] is a support (e.g. the Exact Top-K support
 * S_t) and others [rows, R, K] the R supports it is compared with (e.g. the
 * Exact Top-K supports of the R most similar preceding queries, most similar
 * first); all ascending, -1 padded, device int32.  out: device float
 * [rows, 2] = (|S n others[0]| / K  -- Eq. (2)'s Overlap with the most
 * similar one --, |S n U| / K with U the union of the R supports -- Eq. (3)'s
 * Coverage(R)).  1 <= R <= 256, 1 <= K <= 4096.  Asynchronous on `stream`;
 * a diagnostic, not part of the decode step. */
int retopk_support_overlap(const int32_t *S, const int32_t *others, int rows, int R, int K, float *out,
                           void *stream);

/* ---- profiling ----------------------------------------------------------- */

/* Kernel classes reported by retopk_profile_read. */
#define RETOPK_PROF_APPEND   0   /* K/V row append                                 */
#define RETOPK_PROF_FINISH   1   /* decode back end: reuse path or exact select    */
#define RETOPK_PROF_SCAN     2   /* full-history QK scan + first radix digit       */
#define RETOPK_PROF_SELECT   3   /* exact path: candidate filter, Top-K,
                                    softmax-value, cache insert                    */
#define RETOPK_PROF_CLEAR    4   /* histogram clear of the stateless exact step    */
#define RETOPK_PROF_DECIDE   5   /* recall, Top-R and path switch of a decode step */
#define RETOPK_PROF_KERNELS  6

/* Optional per-kernel timing (off by default).  While enabled, every launch of
 * retopk_append_kv, retopk_decode_step and exact_topk_attention_step is
 * bracketed by two CUDA events on its stream.  Launches made while the stream
 * is being captured get event-record nodes inside the graph; those events are
 * kept, so each replay re-times them.  retopk_profile_read (synchronises on the
 * events) returns, per kernel class, the number of timed launches and their
 * summed duration in milliseconds: eager launches since the previous read, plus
 * the latest replay of every captured launch.  retopk_profile_reset drops all
 * events (call it before destroying graphs that hold them). */
int retopk_profile_enable(int on);
int retopk_profile_read(int64_t launches[RETOPK_PROF_KERNELS], double ms[RETOPK_PROF_KERNELS]);
int retopk_profile_reset(void);

#ifdef __cplusplus
}
#endif
#endif /* RETOPK_H */
