/*
 * sffn.h -- C ABI of libsffn.so: the activation-sparse gated FFN on one GB300
 * (sm_103a).
 *
 * The layer computed is the gated FFN
 *
 *     out = W_down . ( act(W_gate . x + b) (.) (W_up . x) )
 *
 * where intermediate neuron j owns row j of W_gate, row j of W_up and column j
 * of W_down (denseflux, "skipping most of a dense FFN", sec. 1 Motivation).
 * Two ways of skipping work are provided:
 *
 *   decode  -- per token, only the W_up rows and W_down columns of the *active*
 *              neurons are read.  Active means act(g_j) != 0 (exact ReLU/ReGLU
 *              gating, denseflux sec. 5.1-5.2), or a weight-aware score
 *              score_j = |a_j| * ||W_down[:, j]||_2 at or above a threshold, or
 *              among the top floor(F * keep_ratio) scores (WiSparse write-up,
 *              kwkr.cn/news/623085, sec. 1.2, 2.3 and 3.2).
 *   prefill -- token-selective FFN: tokens are chosen by the L2 norm of their
 *              attention-output row up to a cumulative mass threshold, the last
 *              recent_n tokens and at least min_keep tokens are always kept, and
 *              only the chosen tokens run the FFN; the rest pass through the
 *              residual with Z = 0 (RedKnot token-selective sparse FFN,
 *              bhfrc.com/news/43276, Algorithm 1 and its selection rules).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument except `w` (a host struct) and `code` in
 *    sffn_read_device_error is a DEVICE pointer on the current CUDA device.
 *    The caller owns all memory and the stream; the library never allocates
 *    or frees on these calls: scratch memory comes from the caller's
 *    `workspace` (size from sffn_workspace_size, 256-byte aligned).
 *  - The first 16 bytes of every workspace are a control block: the device
 *    error word (below) and two counters with which sffn_decode's CTAs meet at
 *    a grid barrier.  Zero-fill a workspace once before its first use (one
 *    cudaMemset at allocation); every call leaves the control block valid for
 *    the next one, whichever entry point it is, and sffn_read_device_error
 *    clears it.  A workspace serves one call at a time (calls on one stream,
 *    or ordered between streams).
 *  - Calls are asynchronous and stream-ordered on `stream` (NULL = the legacy
 *    default stream); nothing is read back to the host, so a sequence of calls
 *    can be captured in a CUDA graph.  Counts (n_active, n_sel) stay on the
 *    device.  Consecutive kernels use programmatic dependent launch; a decode
 *    call's kernel starts reading its weight matrices, scales and gate bias
 *    before it waits for the preceding kernel of this library on the stream
 *    (no call of this library writes them).
 *  - Argument errors are detected on the host before anything is launched and
 *    returned as a status; a failed launch returns SFFN_ERR_CUDA.  Contract
 *    violations that only the device can see (an out-of-range selected-token
 *    index, n_sel > L) are recorded in an error word at the start of the
 *    workspace (read it with sffn_read_device_error); the offending element is
 *    skipped, nothing traps.
 *  - All device pointers must be 16-byte aligned (128-bit loads) unless stated.
 *  - Matrices are row-major.  The three weight matrices are stored neuron-major,
 *    each [d_ff, d_model]: w_gate[j,:], w_up[j,:] and w_downT[j,:] = W_down[:,j].
 *  - Shape limits: d_model % 8 == 0 (fp32/bf16), d_model % 64 == 0 (int4-g64),
 *    8 <= d_model <= 8192, 1 <= d_ff <= 65536, 1 <= B <= 8.  Decode also needs
 *    d_model <= 4096, and for int4-g64 d_model % 512 == 0 (one row's scales are a
 *    multiple of 16 bytes); int4-g64 decode supports every rule.
 */
#ifndef SFFN_H
#define SFFN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st *sffn_stream_t;

typedef enum {
    SFFN_OK = 0,
    SFFN_ERR_INVALID_ARG = 1, /* null pointer, unknown enum value, parameter out of range */
    SFFN_ERR_SHAPE = 2,       /* dimension out of the supported range                    */
    SFFN_ERR_ALIGNMENT = 3,   /* a pointer is not 16-byte aligned                         */
    SFFN_ERR_UNSUPPORTED = 4, /* valid but not implemented combination / device           */
    SFFN_ERR_WORKSPACE = 5,   /* workspace missing, misaligned or smaller than required   */
    SFFN_ERR_CUDA = 6,        /* a CUDA runtime call or launch failed                     */
    SFFN_ERR_TIMEOUT = 7,     /* a bounded device-side wait gave up (device error word)   */
    SFFN_ERR_DEVICE = 8       /* a device-side contract violation was recorded            */
} sffn_status;

typedef enum { SFFN_MODE_EXACT = 0, SFFN_MODE_THRESHOLD = 1, SFFN_MODE_KEEP_RATIO = 2 } sffn_mode;
typedef enum { SFFN_ACT_RELU = 0, SFFN_ACT_SILU = 1 } sffn_act;
/* Weight storage.  INT4_G64: symmetric int4, two's-complement codes packed two
 * per byte (low nibble = even column), one fp16 scale per 64 consecutive
 * elements of a stored row; value = code * scale. */
typedef enum { SFFN_F32 = 0, SFFN_BF16 = 1, SFFN_INT4_G64 = 2 } sffn_wdtype;
/* Score used by the threshold and keep-ratio modes:
 *   GATE     score_j = |act(g_j)| * ||W_down[:, j]||_2          (W_up stays sparse)
 *   GATE_UP  score_j = |act(g_j) * u_j| * ||W_down[:, j]||_2    (needs every u_j,
 *            so W_up is read in full and only W_down stays sparse). */
typedef enum { SFFN_SCORE_GATE = 0, SFFN_SCORE_GATE_UP = 1 } sffn_score;

/* One FFN layer.  Host struct holding device pointers. */
typedef struct {
    int32_t wdtype;          /* sffn_wdtype                                           */
    int32_t act;             /* sffn_act                                              */
    int32_t d_model, d_ff;
    const void *w_gate;      /* [d_ff, d_model] (int4: uint8 [d_ff, d_model/2])       */
    const void *w_up;        /* [d_ff, d_model]                                       */
    const void *w_downT;     /* [d_ff, d_model], row j = column j of W_down           */
    const void *s_gate;      /* int4 only: fp16 [d_ff, d_model/64]; else NULL         */
    const void *s_up;        /* int4 only                                             */
    const void *s_downT;     /* int4 only                                             */
    const float *b_gate;     /* [d_ff] fp32 gate bias, or NULL                         */
    const float *down_norms; /* [d_ff] fp32 ||W_down[:, j]||_2 (see sffn_down_norms);
                                needed by the threshold / keep-ratio modes, else may be NULL */
} sffn_ffn_weights;

/* Bytes of workspace needed by a call.  which: 0 = sffn_decode (n = B),
 * 1 = sffn_token_select (n = L), 2 = sffn_prefill (n = L).  Returns 0 for an
 * invalid request.  The size depends on the device's SM count (current device). */
size_t sffn_workspace_size(int which, int n, const sffn_ffn_weights *w);

/* norms[j] = ||W_down[:, j]||_2 = sqrt(sum_i w_downT[j, i]^2) of the
 * (dequantised) weights, fp32 [d_ff].  The weight-aware prior of the WiSparse
 * write-up, sec. 2.3, with p = 2 on the down projection's column. */
sffn_status sffn_down_norms(const sffn_ffn_weights *w, float *norms, sffn_stream_t stream);

/* Decode B tokens (1 <= B <= 8) through one layer, skipping inactive neurons.
 *   x          [B, d_model]: fp32 when wdtype == F32, else bf16.
 *   mode       sffn_mode; param = tau for THRESHOLD (keep iff score >= tau,
 *              tau >= 0), keep_ratio in (0, 1] for KEEP_RATIO (keep the
 *              k = max(1, floor(d_ff * keep_ratio)) largest scores, ties to the
 *              lower index), ignored for EXACT (keep iff act(g_j) != 0).
 *   score      sffn_score (threshold / keep-ratio only).
 *   out        [B, d_model], same dtype as x: sum over the token's active j of
 *              act(g_j) * u_j * W_down[:, j], fp32 accumulation, rounded once.
 *   active_idx [B, d_ff] int32: row b holds the token's active neurons in
 *              ascending order in its first n_active[b] entries (the rest is
 *              unspecified).  n_active [B] int32.
 * For B > 1 the W_up / W_down rows of the union of the tokens' active sets are
 * read once and each token is masked to its own set. */
sffn_status sffn_decode(const void *x, int B, const sffn_ffn_weights *w, int mode, int score,
                        float param, void *out, int32_t *active_idx, int32_t *n_active,
                        void *workspace, size_t ws_bytes, sffn_stream_t stream);

/* The dense layer, nothing skipped: out = W_down (act(W_gate x + b) (.) (W_up x))
 * over every neuron, the baseline that denseflux sec. 5.3 measures the sparse
 * layer against (breakeven active fraction, speedup at 10% active).  Reads all
 * three matrices once; no index lists.  x, out: bf16 [B, d_model]; weights bf16
 * or int4-g64; workspace as sffn_decode's (sffn_workspace_size(0, B, w)).
 * Needs d_model in {1024, 2048, 4096} and d_ff <= 128 * (#SMs); a single
 * token with int4-g64 weights also takes d_model 512 and d_ff up to
 * 256 * (#SMs).  Other shapes and fp32 weights return SFFN_ERR_UNSUPPORTED. */
sffn_status sffn_decode_dense(const void *x, int B, const sffn_ffn_weights *w, void *out, void *workspace,
                              size_t ws_bytes, sffn_stream_t stream);

/* Decode one token through one layer with the low-rank gate predictor of the
 * denseflux write-up ("skipping most of a dense FFN", sec. 4.3, cheap
 * predictors: the best untrained predictor is low-rank).  The factors
 * W_gate ~= A B are made offline (e.g. a rank-r truncated SVD of the dequantised
 * gate); per token
 *   y = B x,  p_j = A[j, :] . y + b_gate[j],  candidates P = { j : p_j >= -alpha },
 * the exact gate g_j = W_gate[j, :] . x + b_gate[j] only for j in P, and
 * j active iff j in P and act(g_j) != 0 (the exact rule).  A neuron outside P
 * is skipped even when it would have been active.
 *   x          [d_model], bf16 (fp32 with fp32 weights); 16-byte aligned.
 *   w          bf16 or fp32 weights (int4-g64: SFFN_ERR_UNSUPPORTED).
 *   factor_a   A [d_ff, rank] fp32 row-major, device memory.
 *   factor_b   B [rank, d_model] fp32 row-major, device memory, 16-byte aligned.
 *   rank       1 <= rank <= min(d_ff, 4096).
 *   alpha      >= 0; +INFINITY makes every neuron a candidate (the factors are
 *              then not read and may be NULL): the exact decode.
 *   out, active_idx [d_ff], n_active [1]: as sffn_decode with B = 1 (active
 *              neurons ascending).
 *   workspace  sffn_workspace_size(0, 1, w) bytes, 16-byte aligned.
 * The caller owns every buffer; nothing is allocated.  Argument errors are
 * returned before anything is enqueued. */
sffn_status sffn_decode_predicted(const void *x, const sffn_ffn_weights *w, const float *factor_a,
                                  const float *factor_b, int rank, float alpha, void *out, int32_t *active_idx,
                                  int32_t *n_active, void *workspace, size_t ws_bytes, sffn_stream_t stream);

/* Keep-ratio decode with a per-layer core set (WiSparse write-up, sec. 2.2,
 * the paragraph after the score definition: the columns kept most often at a
 * tier form a guaranteed base set, and each token completes its selection
 * dynamically; sec. 5 FAQ: batch > 1 shares one tier).  Per token:
 *   keep = core  U  the (k - |core|) largest scores among the columns outside
 *          the core (ties to the lower index), k = max(1, floor(d_ff * keep_ratio));
 * with |core| >= k the token keeps the core alone.  Arguments and results as
 * sffn_decode in SFFN_MODE_KEEP_RATIO (B tokens: the union of their sets is
 * read once, each token masked to its own set), plus
 *   core_idx   [n_core] int32 device array: the core's columns (ascending,
 *              distinct, as sffn_tier_core_set writes them); an index outside
 *              [0, d_ff) is skipped and recorded as SFFN_ERR_DEVICE in the
 *              workspace's error word (sffn_read_device_error).
 *   n_core     0 <= n_core <= d_ff (0: the plain keep-ratio selection).
 * Every weight format (fp32, bf16, int4-g64). */
sffn_status sffn_decode_tiered(const void *x, int B, const sffn_ffn_weights *w, int score, float keep_ratio,
                               const int32_t *core_idx, int n_core, void *out, int32_t *active_idx, int32_t *n_active,
                               void *workspace, size_t ws_bytes, sffn_stream_t stream);

/* Bytes of workspace for sffn_tier_core_set (0 for an invalid request). */
size_t sffn_tier_core_workspace_size(int n_calib, int d_ff);

/* The core set of a keep-ratio tier from calibration scores (WiSparse
 * write-up, sec. 2.2): for each calibration token its top-k columns (the k
 * largest scores, ties to the lower index); per column the number of tokens
 * that kept it; the core is the n_core columns with the largest counts (count
 * ties to the lower index), written ascending to core_idx [n_core].
 *   calib_scores [n_calib, d_ff] fp32 device array of non-negative scores (as
 *                sffn_gate_scores writes them); 1 <= n_calib <= 65536.
 *   k            the tier's k, 1 <= k <= d_ff; 0 <= n_core <= d_ff (core_idx may be
 *                NULL when n_core is 0).
 *   workspace    sffn_tier_core_workspace_size(n_calib, d_ff) bytes. */
sffn_status sffn_tier_core_set(const float *calib_scores, int n_calib, int d_ff, int k, int n_core, int32_t *core_idx,
                               void *workspace, size_t ws_bytes, sffn_stream_t stream);

/* ---- MoE layers (RedKnot write-up, bhfrc.com/news/43276, section "adaptive
 * expert Top-K") ---- */

/* The progressive top-K by depth: 6 experts for layers 0-15, 5 for 16-39, 4 for
 * 40-60 (and past 60); -1 for a negative layer. */
int sffn_moe_progressive_k(int layer);

/* Adaptive expert top-K for T tokens.  Per token (logits [T, E] fp32, device):
 * probabilities p = softmax(logits) (fp32); experts ranked by probability
 * descending, ties to the lower expert index; K = the smallest bucket b (from
 * buckets[0..n_buckets), ascending, host memory) with b <= cap whose top-b mass
 * reaches `mass` (the page's default 0.50), else cap (the layer's progressive
 * K).  Writes k_out [T], experts [T, kmax] (the K experts ascending, then -1)
 * and weights [T, kmax] (their probabilities renormalised to sum 1, then 0).
 * 1 <= E <= 512, 1 <= cap <= min(E, 8), cap <= kmax <= 8, bucket values in
 * [1, 8].  Nothing is allocated; T = 0 is a no-op. */
sffn_status sffn_moe_route(const float *logits, int T, int E, int cap, float mass, const int32_t *buckets,
                           int n_buckets, int kmax, int32_t *k_out, int32_t *experts, float *weights,
                           sffn_stream_t stream);

/* Bytes of workspace for sffn_moe_block_budget (0 for an invalid request). */
size_t sffn_moe_budget_workspace_size(int L, int d_model);

/* The block token budget of an MoE layer over one sequence, on the GPU with no
 * host synchronisation.  A token's importance is the L2 norm of its attention
 * output row (y_attn [L, d_model] bf16, as sffn_token_select); f = the share of
 * tokens the mass rule keeps (sffn_token_select with this mass, no recent tail,
 * no minimum) clamped to [min_ratio, max_ratio] (the page's 0.10 / 0.50);
 * nsel = max(1, ceil(f * nblocks)) of the nblocks = ceil(L / block) blocks of
 * `block` consecutive tokens (the page's 128), those with the largest summed
 * importance (ties to the lower block index), run the MoE.  Writes
 * token_idx [L] (the chosen blocks' tokens ascending, first *n_tokens entries)
 * and ranges [2 * nblocks] (the *n_ranges maximal contiguous [start, end) token
 * ranges, ascending).  The list feeds sffn_prefill's sel_idx / n_sel as it is.
 * nblocks <= 8192; workspace sffn_moe_budget_workspace_size(L, d_model) bytes. */
sffn_status sffn_moe_block_budget(const void *y_attn, int L, int d_model, float mass, float min_ratio,
                                  float max_ratio, int block, int32_t *token_idx, int32_t *n_tokens, int32_t *ranges,
                                  int32_t *n_ranges, void *workspace, size_t ws_bytes, sffn_stream_t stream);

/* Size of the scratch array built into the library for sffn_decode_noalloc. */
#define SFFN_NOALLOC_SCRATCH_BYTES (4u << 20)

/* sffn_decode without a workspace argument.  No page describes this call: it
 * exists for callers that cannot allocate device memory themselves -- code that
 * is handed its input and output buffers by a host framework or plugin
 * interface and has no device allocator of its own, or that must not allocate
 * once it is running (a latency-critical serving loop with a fixed memory
 * budget).  Such callers cannot provide the `workspace` that sffn_decode takes.
 *
 * Instead the scratch memory comes from one fixed array of
 * SFFN_NOALLOC_SCRATCH_BYTES (4 MiB) compiled into the library; every GPU that
 * loads the library holds that array until the process exits.  Arguments and
 * results are exactly those of sffn_decode.  The call allocates nothing: no
 * cudaMalloc, no cudaFree, no allocating library routine.
 *  - A request whose workspace (sffn_workspace_size(0, B, w)) would exceed the
 *    array is rejected with SFFN_ERR_WORKSPACE before anything is launched.
 *    On a 152-SM GB300 that admits B = 1 at d_model 4096 / d_ff 11008 and
 *    B <= 2 at d_model 2048 / d_ff 11008.
 *  - The first call on each device looks up the array's device address (with
 *    that device current); make that first call before any stream capture.
 *  - Argument errors are reported exactly as sffn_decode reports them, before
 *    anything is enqueued.
 *  - All calls share the one array, which keeps the previous call's contents
 *    (every word is written before it is read; the grid-barrier counters are
 *    reset at the start of each call).  The device error word is not reset by
 *    a call: it keeps the first error recorded since it was last read with
 *    sffn_decode_noalloc_read_error.  Calls that can overlap on the GPU
 *    (different streams, different host threads) race on the array: issue them
 *    in one stream order. */
sffn_status sffn_decode_noalloc(const void *x, int B, const sffn_ffn_weights *w, int mode, int score,
                                float param, void *out, int32_t *active_idx, int32_t *n_active,
                                sffn_stream_t stream);

/* sffn_read_device_error for the built-in array of sffn_decode_noalloc on the
 * current device: copies its device error word to *code (host) and clears it,
 * waiting for `stream`.  0 = no error; SFFN_ERR_TIMEOUT = a bounded wait of an
 * earlier sffn_decode_noalloc call gave up (its outputs are incomplete). */
sffn_status sffn_decode_noalloc_read_error(int32_t *code, sffn_stream_t stream);

/* Scores of every neuron for B tokens, fp32 [B, d_ff] (score kind as in
 * sffn_decode; down_norms required).  Reads the gate (and for GATE_UP the up
 * projection) in full; used to calibrate thresholds offline. */
sffn_status sffn_gate_scores(const void *x, int B, const sffn_ffn_weights *w, int score,
                             float *scores, void *workspace, size_t ws_bytes, sffn_stream_t stream);

/* Token selection for a prefill of L tokens (RedKnot selection rules):
 *   importance s_t = ||y_attn[t, :]||_2 (y_attn bf16 [L, d_model]);
 *   if mass_thresh >= 1 or sum_t s_t == 0: every token;
 *   else the shortest prefix of the tokens ordered by (s desc, t asc) whose
 *   importance sum reaches mass_thresh * sum_t s_t (the crossing token is
 *   included; none if mass_thresh <= 0), united with the last recent_n tokens,
 *   then extended in the same order up to min(min_keep, L) tokens.
 * Writes sel_idx[0 .. n_sel) ascending (int32 [L]) and n_sel (int32 [1]).
 * recent_n >= 0, min_keep >= 1, 1 <= L <= 1048576, d_model % 8 == 0. */
sffn_status sffn_token_select(const void *y_attn, int L, int d_model, float mass_thresh,
                              int recent_n, int min_keep, int32_t *sel_idx, int32_t *n_sel,
                              void *workspace, size_t ws_bytes, sffn_stream_t stream);

/* Token-selective prefill (RedKnot Algorithm 1): Y = bf16(x + y_attn) for every
 * row; for the selected rows out[t] = bf16(Y[t] + FFN(Y[t])) with
 * FFN(y) = W_down . (SiLU(W_gate . y) (.) (W_up . y)); for the others
 * out[t] = Y[t] (Z = 0).  x, y_attn, out: bf16 [L, d_model].  sel_idx / n_sel as
 * written by sffn_token_select (ascending, device).  Weights: bf16 or int4-g64
 * (the INT4 setting the RedKnot write-up measures: each weight becomes
 * code * scale rounded once to bf16 for the tensor cores), act SILU, no gate
 * bias, d_model % 64 == 0, d_ff % 128 == 0. */
sffn_status sffn_prefill(const void *x, const void *y_attn, int L, const sffn_ffn_weights *w,
                         const int32_t *sel_idx, const int32_t *n_sel, void *out, void *workspace,
                         size_t ws_bytes, sffn_stream_t stream);

/* Per-layer sparsity schedule of a multi-layer token-selective prefill (RedKnot
 * write-up, the three-tier SparseFFNSchedule):
 *   layer <  dense_until                       dense FFN (a selection with mass 1:
 *                                              every token)
 *   dense_until <= layer < deep_layer_start    select with mass_thresh
 *   layer >= deep_layer_start                  select with mass_thresh_deep
 * recent_n and min_keep apply to every layer.  Valid when dense_until >= 0,
 * deep_layer_start >= 0, both masses >= 0, recent_n >= 0 and min_keep >= 1.
 * Host struct. */
typedef struct {
    int32_t dense_until;
    int32_t deep_layer_start;
    float mass_thresh;
    float mass_thresh_deep;
    int32_t recent_n;
    int32_t min_keep;
} sffn_ffn_schedule;

typedef enum {
    SFFN_PRESET_SPEED = 0,     /* dense_until 3,  mass 0.3, recent_n 64  */
    SFFN_PRESET_BALANCED = 1,  /* dense_until 20, mass 0.5, recent_n 128 */
    SFFN_PRESET_QUALITY = 2,   /* dense_until 32, mass 0.7, recent_n 128 */
    SFFN_PRESET_DENSE = 3      /* dense_until 80, mass 1.0, recent_n 128 (the dense baseline) */
} sffn_preset;

/* The write-up's FFN presets table.  The table names no deep tier, so
 * deep_layer_start = INT32_MAX and mass_thresh_deep = mass_thresh; min_keep = 1.
 * Returns SFFN_ERR_INVALID_ARG for an unknown preset or out == NULL. */
sffn_status sffn_schedule_preset(int preset, sffn_ffn_schedule *out);

/* Mass threshold the schedule gives layer `layer` (1 for a dense layer), or a
 * negative value for an invalid schedule or layer < 0.  Host only. */
float sffn_schedule_mass(const sffn_ffn_schedule *s, int layer);

/* Workspace bytes for sffn_prefill_layers with L tokens and layers shaped like w
 * (one selection/prefill region plus one bf16 [L, d_model] buffer); 0 if invalid. */
size_t sffn_prefill_layers_workspace_size(int L, const sffn_ffn_weights *w);

/* A stack of n_layers token-selective prefill layers, enqueued on `stream`
 * without a host synchronisation.  Layer i (schedule index first_layer + i)
 * selects tokens of y_attn[i] with sffn_schedule_mass(s, first_layer + i),
 * s->recent_n and s->min_keep, then runs sffn_prefill with weights w[i] on the
 * previous layer's output (x for i = 0).  The last layer's output goes to out.
 *   x, out      bf16 [L, d_model], distinct buffers.
 *   y_attn      HOST array of n_layers device pointers, bf16 [L, d_model] each.
 *   w           HOST array of n_layers weight structs (same d_model; each as
 *               sffn_prefill requires).
 *   sel_idx     int32 [n_layers, L]: row i holds layer i's selection; n_sel
 *               int32 [n_layers].
 *   workspace   the largest sffn_prefill_layers_workspace_size over the layers
 *               (zero-filled before first use, like every workspace).
 * Errors as sffn_token_select / sffn_prefill; SFFN_ERR_SHAPE if the layers'
 * d_model differ. */
sffn_status sffn_prefill_layers(const void *x, const void *const *y_attn, int L, int n_layers,
                                const sffn_ffn_weights *w, const sffn_ffn_schedule *s, int first_layer,
                                void *out, int32_t *sel_idx, int32_t *n_sel, void *workspace,
                                size_t ws_bytes, sffn_stream_t stream);

/* Copy the workspace's device error word to *code (host) and clear it; waits
 * for `stream`.  0 = no error; otherwise an sffn_status value. */
sffn_status sffn_read_device_error(void *workspace, int32_t *code, sffn_stream_t stream);

/* Static description of a status code. */
const char *sffn_status_string(sffn_status s);

#ifdef __cplusplus
}
#endif
#endif /* SFFN_H */
