/*
 * sel.h -- C ABI of the GB300 (sm_103a) decode-step token-selection library.
 *
 * Four operations over batched fp32 logits rows of a vocabulary of V entries:
 * argmax, exact top-k, filtered sampling and speculative acceptance. Every
 * entry point takes device pointers, sizes, the policy parameters, a
 * caller-owned workspace and a cudaStream_t, validates its arguments on the
 * host, enqueues its kernels on that stream and returns. It never allocates,
 * never synchronises and never touches another stream.
 *
 * Conventions shared by every entry point
 *  - Memory. All pointers except the parameter structs are device pointers
 *    owned by the caller. Logits are row-major: row r starts at
 *    logits + r * V (a row stride of exactly V floats). The vector path needs
 *    logits 16-byte aligned and V % 4 == 0; any other 4-byte-aligned layout
 *    takes the scalar path, with identical results.
 *  - Workspace. d_ws holds per-row partial results, and the slots that the
 *    finishing launches combine and clear again. Size it with
 *    sel_workspace_bytes() for the largest call it will serve, zero it once
 *    with sel_workspace_init() after allocating it, then reuse it: every call
 *    leaves its counters at zero again. Calls that may run concurrently (on
 *    different streams) need separate workspaces. d_ws must be 256-byte
 *    aligned.
 *  - Errors. The return value reports what the host can see: bad arguments
 *    (SEL_EINVAL), a workspace too small (SEL_EWORKSPACE), an unsupported
 *    size (SEL_EUNSUPPORTED) or a launch failure (SEL_ECUDA). rows == 0 (or
 *    S == 0) is a no-op returning SEL_OK. Data errors found on the device do
 *    not fail the call: they make that row's (sequence's) ids
 *    SEL_INVALID_ID, with NaN values and probabilities. A row is invalid when
 *    it holds a NaN or +-Inf logit, or when its uniform lies outside [0, 1)
 *    (fail closed: the greedy serving variant of the Muser book's argmax
 *    latches nonfinite logits and returns 0xffffffff, "Ch 21 -- Sampling,
 *    argmax, and grammar", 21.4 and 21.6).
 *  - Ids are 31-bit: V must be below 2^31 (bit 31 of an id is the
 *    nonfinite flag of that design).
 *  - Determinism. Results do not depend on block scheduling: every combine
 *    runs in a fixed order, and ties between equal logits always go to the
 *    lower token id.
 */
#ifndef SEL_H
#define SEL_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sel_status {
    SEL_OK = 0,
    SEL_EINVAL = 1,       /* null/misaligned pointer, bad size or parameter */
    SEL_EWORKSPACE = 2,   /* ws_bytes below sel_workspace_bytes() */
    SEL_ECUDA = 3,        /* a CUDA call or kernel launch failed */
    SEL_EUNSUPPORTED = 4  /* valid request outside what the kernels cover */
} sel_status;

#define SEL_INVALID_ID 0xFFFFFFFFu  /* per-row (per-sequence) error sentinel */
#define SEL_MAX_K 1024u             /* largest k of sel_topk / top_k of sel_sample */
#define SEL_MAX_V 0x7FFFFFFFu       /* V must be <= SEL_MAX_V (31-bit ids) */
#define SEL_WS_ALIGN 256u

/* Operation codes for sel_workspace_bytes. */
enum { SEL_OP_ARGMAX = 0, SEL_OP_TOPK = 1, SEL_OP_SAMPLE = 2, SEL_OP_SPEC = 3,
       SEL_OP_SPEC_SAMPLER = 4, SEL_OP_SPEC_DIAG = 5, SEL_OP_SHARD_DRAW = 6,
       SEL_OP_SPEC_SHARD_DRAW = 7 };

/* Order of temperature and filters in sel_sample. */
enum {
    SEL_ORDER_TEMP_FIRST = 0, /* scale by 1/T, then top-k, top-p, min-p */
    SEL_ORDER_TEMP_LAST = 1   /* top-k, top-p, min-p on the untempered
                                 distribution; temperature only in the draw
                                 ("Speculative-decoding acceptance rules",
                                 The rules: filtering on the untempered
                                 distribution, temperature scaling last) */
};

/* Acceptance rule of spec_accept. */
enum {
    SPEC_MODE_REJECTION = 0, /* modified rejection sampling (lossless) */
    SPEC_MODE_ARGMAX = 1     /* argmax-against-argmax (greedy stream) */
};

/*
 * Bytes of workspace an operation needs.
 *   op SEL_OP_ARGMAX: rows, V (k ignored)
 *   op SEL_OP_TOPK:   rows, V, k
 *   op SEL_OP_SAMPLE: rows, V, k = the policy's top_k
 *   op SEL_OP_SPEC:   rows = S (sequences), V, k = K (draft positions)
 *   op SEL_OP_SPEC_SAMPLER: rows = S * (K + 1) (target rows), V,
 *                     k = the policy's top_k
 *   op SEL_OP_SPEC_DIAG: rows = S, V, k = K
 *   op SEL_OP_SHARD_DRAW: rows, V = the shard's slice width (k ignored)
 *   op SEL_OP_SPEC_SHARD_DRAW: rows = S, V = the shard's slice width
 * The size depends only on these arguments, not on the device. Returns 0
 * when the arguments are invalid (the entry point would refuse them anyway).
 */
size_t sel_workspace_bytes(int op, uint32_t rows, uint32_t V, uint32_t k);

/*
 * Zero a freshly allocated workspace: one cudaMemsetAsync on `stream`.
 * Needed once per allocation; the entry points keep it zeroed afterwards.
 */
sel_status sel_workspace_init(void *d_ws, size_t ws_bytes, cudaStream_t stream);

/*
 * sel_argmax -- per row, the lowest index attaining the maximum logit.
 *
 * Defined by the Muser book chapter "Ch 21 -- Sampling, argmax, and
 * grammar": 21.3 (a reduction of each row to one (value, index) pair; the
 * comparison is strictly greater, so a tie keeps the lower index), 21.4 (the
 * greedy serving variant: any NaN/Inf latches a flag and the result is
 * 0xffffffff), 21.5 ("encode_argmax_f32_rows": one winner per row of a
 * logits matrix).
 *
 *   d_logits   [rows][V] f32, device
 *   d_out_ids  [rows] u32, device: the winning id, or SEL_INVALID_ID when the
 *              row holds a nonfinite logit
 *   d_ws       workspace of sel_workspace_bytes(SEL_OP_ARGMAX, rows, V, 0)
 */
sel_status sel_argmax(const float *d_logits, uint32_t rows, uint32_t V,
                      uint32_t *d_out_ids, void *d_ws, size_t ws_bytes,
                      cudaStream_t stream);

/*
 * sel_topk -- per row, the k largest logits with their token ids, sorted by
 * value descending, equal values by lower id; only these k entries per row
 * leave the kernel.
 *
 * Defined by the llama.cpp pull request 49 ("Change": llama_set_logits_topk
 * runs top_k on the logits so only the k candidates per row are copied, and
 * the candidates hold the k largest logits of each row with their tokens and
 * values), with the lower-id tie rule of the Muser book, 21.3.
 *
 *   d_logits    [rows][V] f32, device
 *   k           1 <= k <= min(V, SEL_MAX_K)
 *   d_out_vals  [rows][k] f32, device: the values (copies of the logits);
 *               NaN for an invalid row
 *   d_out_ids   [rows][k] u32, device: their ids; SEL_INVALID_ID for an
 *               invalid row
 *   d_ws        workspace of sel_workspace_bytes(SEL_OP_TOPK, rows, V, k)
 */
sel_status sel_topk(const float *d_logits, uint32_t rows, uint32_t V,
                    uint32_t k, float *d_out_vals, uint32_t *d_out_ids,
                    void *d_ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Sampling policy.
 *   temperature  >= 0; 0 means greedy (the argmax, probability 1)
 *   top_k        1 <= top_k <= SEL_MAX_K (top_k > V means V); 0 means no
 *                truncation: full-row sampling, the chain over all V ids
 *                (see sel_sample)
 *   top_p        (0, 1]; 1 disables it
 *   min_p        [0, 1); 0 disables it
 *   order        SEL_ORDER_TEMP_FIRST or SEL_ORDER_TEMP_LAST
 *   top_n_sigma  >= 0, finite; 0 disables it. Keeps only ids whose logit is
 *                at least max - top_n_sigma * sigma, sigma the population
 *                standard deviation of the row's V logits (a mask against the
 *                maximum, independent of T), before top-k (Muser book 21.7,
 *                the sampler chain: top-n-sigma, then top-k)
 *   typical_p    [0, 1]; 0 and 1 disable it. Locally typical sampling on the
 *                candidates (after top-k, before top-p; Muser book 21.7):
 *                with H the entropy of P over the candidates, keep the ids
 *                of smallest |-ln P - H| (ties: the more probable one) until
 *                their P reaches typical_p; they keep their order and P is
 *                renormalised over them
 * The last two fields were appended; a zero-initialised struct leaves both
 * filters off.
 */
typedef struct sel_sample_params {
    float temperature;
    uint32_t top_k;
    float top_p;
    float min_p;
    int32_t order;
    float top_n_sigma;
    float typical_p;
} sel_sample_params;

/*
 * sel_sample -- per row, one token drawn by inverse CDF from the filtered,
 * temperature-scaled softmax, with a caller-supplied uniform.
 *
 * Steps (TEMP_FIRST): z = x / T; the top-n-sigma mask (if on); the top_k
 * candidates of z (the sel_topk definition); P = softmax over the
 * candidates; the locally typical window (if on); top-p keeps the shortest
 * prefix, in (P desc, id asc) order, whose cumulative P reaches top_p (the
 * crossing token included); min-p keeps candidates with P >= min_p * P_max;
 * Q = P renormalised over the survivors; the draw is the first survivor, in
 * the same order, whose cumulative Q exceeds u (the last survivor if
 * rounding leaves none). TEMP_LAST computes the filters with T = 1 and Q with
 * the tempered weights.
 * Full-row sampling (top_k == 0, temperature > 0): the same chain with every
 * id of the row as a candidate; the draw walks the survivors in ascending
 * token id instead (the same distribution, without sorting the row). The
 * row is read twice. The filters are decided from the row's 64 most probable
 * ids against sums over the whole row; a top-p cut or a locally typical
 * window that needs ids beyond those 64 is found by a search over the row (a
 * radix select weighted by probability mass, on the value for top-p and on
 * the distance to the typical logit M + Tf * mean(g) for the typical window,
 * then top-p inside that window; passes that L2 mostly serves), so every
 * such row is decided. (Under top-n-sigma the search first sums the
 * candidate set's mass and mean log-weight over the row.)
 * Sources: Muser book 21.1 (temperature-scaled softmax, then a draw
 * restricted to top-k / top-p candidates) and 21.7 (top-k truncation before
 * the top-p cutoff); llama.cpp pull 49, "Change" (a chain with top-k first
 * needs only the k candidates; top-p and min-p then act on them);
 * "Speculative-decoding acceptance rules", The rules (the temperature-last
 * order).
 *
 *   d_uniforms  [rows] f32, device: u in [0, 1); anything else (NaN
 *               included) makes the row invalid
 *   d_out_ids   [rows] u32, device: the drawn id or SEL_INVALID_ID
 *   d_out_probs [rows] f32, device: Q of the drawn id (1 for greedy), NaN
 *               for an invalid row
 *   d_ws        workspace of sel_workspace_bytes(SEL_OP_SAMPLE, rows, V, top_k)
 */
sel_status sel_sample(const float *d_logits, uint32_t rows, uint32_t V,
                      const sel_sample_params *params,
                      const float *d_uniforms, uint32_t *d_out_ids,
                      float *d_out_probs, void *d_ws, size_t ws_bytes,
                      cudaStream_t stream);

/*
 * Speculative-acceptance policy.
 *   temperature  >= 0; p and q are softmax(logits / T); 0 selects the argmax
 *                rule whatever the mode (greedy draws nothing)
 *   mode         SPEC_MODE_REJECTION or SPEC_MODE_ARGMAX
 */
typedef struct spec_params {
    float temperature;
    int32_t mode;
} spec_params;

/*
 * spec_accept -- verify K draft tokens per sequence against the target.
 *
 * SPEC_MODE_REJECTION ("Speculative-decoding acceptance rules", Modified
 * rejection sampling, steps 1-3; Muser book 21.9): for j = 0..K-1, accept
 * draft token t_j iff u_acc[j] * q_j(t_j) <= p_j(t_j); at the first
 * rejection j* draw one token with u_fin from normalize(max(p_j* - q_j*, 0))
 * (from p_j* if that residual sums to <= 0) and stop; if all K are accepted
 * draw a bonus token with u_fin from p_K. Draws walk the vocabulary in
 * ascending token id.
 * SPEC_MODE_ARGMAX (same page, Argmax-against-argmax): accept t_j iff it
 * equals argmax(target_j); emit that argmax at the first mismatch, or the
 * bonus argmax(target_K) when all match. d_draft and the uniforms may be
 * NULL.
 *
 *   d_target        [S][K+1][V] f32, device
 *   d_draft         [S][K][V] f32, device (rejection mode)
 *   d_draft_tokens  [S][K] u32, device
 *   d_u_acc         [S][K] f32, device: one uniform per draft position
 *   d_u_fin         [S] f32, device: one uniform for the final draw
 *   d_accepted      [S] u32, device: accepted count n, or SEL_INVALID_ID
 *   d_emitted       [S][K+1] u32, device: t_0..t_{n-1}, the drawn token,
 *                   then SEL_INVALID_ID
 *   d_ws            workspace of sel_workspace_bytes(SEL_OP_SPEC, S, V, K)
 * A sequence is invalid (accepted and emitted all SEL_INVALID_ID) when any
 * of its rows holds a nonfinite logit, a draft token is >= V, or (rejection
 * mode) a uniform lies outside [0, 1).
 */
sel_status spec_accept(const float *d_target, const float *d_draft,
                       const uint32_t *d_draft_tokens, uint32_t S,
                       uint32_t K, uint32_t V, const spec_params *params,
                       const float *d_u_acc, const float *d_u_fin,
                       uint32_t *d_accepted, uint32_t *d_emitted, void *d_ws,
                       size_t ws_bytes, cudaStream_t stream);

/*
 * spec_accept_sampler -- the sampler-match rule of "Speculative-decoding
 * acceptance rules" (mlxcel), "Sampler-match": each verified position j
 * draws a fresh token from the target's sampler -- the sel_sample chain with
 * policy `p` over target row j and the uniform u[s][j] -- and the drafted
 * token t_j is accepted iff it equals that draw. The first mismatch emits
 * the draw and ends the chain; if all K drafts match, the draw at position K
 * is the bonus token. Lossless: every emitted token is a draw from the target
 * sampler; the acceptance probability is sum_x p(x) q(x).
 *
 *   d_target        [S][K+1][V] f32 target logits
 *   d_draft_tokens  [S][K] u32
 *   p               the target sampler, as for sel_sample (temperature == 0
 *                   is greedy; top_k == 0 samples the whole row, and a draw
 *                   that fails closed there fails its sequence closed)
 *   d_u             [S][K+1] f32, one uniform per verified position
 *   d_accepted, d_emitted  as for spec_accept
 *   d_ws            workspace of sel_workspace_bytes(SEL_OP_SPEC_SAMPLER,
 *                   S * (K + 1), V, p->top_k)
 * A sequence with a nonfinite target row, a draft token >= V or any of its
 * K + 1 uniforms outside [0, 1) gets 0xFFFFFFFF everywhere. Two launches.
 */
sel_status spec_accept_sampler(const float *d_target,
                               const uint32_t *d_draft_tokens, uint32_t S,
                               uint32_t K, uint32_t V,
                               const sel_sample_params *p, const float *d_u,
                               uint32_t *d_accepted, uint32_t *d_emitted,
                               void *d_ws, size_t ws_bytes,
                               cudaStream_t stream);

/*
 * spec_diagnostics -- the closed-form acceptance diagnostics of
 * "Speculative-decoding acceptance rules" (mlxcel), "Verifying the gain
 * before trusting a throughput number": per verified position j < K,
 * sum_x min(p_j(x), q_j(x)) (the acceptance probability of modified rejection
 * sampling) and sum_x p_j(x) q_j(x) (that of sampler-match), with
 * p_j = softmax(target_j / T) and q_j = softmax(draft_j / T), T > 0.
 *
 *   d_target [S][K+1][V], d_draft [S][K][V] f32 (target row K is read but
 *            not used)
 *   d_sum_min, d_sum_prod  [S][K] f32 outputs; NaN for a position whose
 *            target or draft row holds a NaN or Inf
 *   d_ws     workspace of sel_workspace_bytes(SEL_OP_SPEC_DIAG, S, V, K)
 * Reads every row once for its statistics and each position's pair of rows
 * once more. Two launches.
 */
sel_status spec_diagnostics(const float *d_target, const float *d_draft,
                            uint32_t S, uint32_t K, uint32_t V,
                            float temperature, float *d_sum_min,
                            float *d_sum_prod, void *d_ws, size_t ws_bytes,
                            cudaStream_t stream);

/*
 * sel_argmax_noalloc -- sel_argmax for callers that cannot allocate device
 * memory (a runtime that plans all device memory up front, or a plugin
 * interface that passes a stream but no workspace). The pages have no
 * counterpart: it is the same per-row argmax as sel_argmax, computed by the
 * same kernel, with its scratch taken from an array of
 * SEL_NOALLOC_SCRATCH_BYTES that the library reserves on every GPU it is
 * loaded on and keeps until the process exits.
 *
 *   d_logits, rows, V, d_out_ids  as for sel_argmax
 * Requests whose workspace would not fit (sel_workspace_bytes(SEL_OP_ARGMAX,
 * rows, V, 0) > SEL_NOALLOC_SCRATCH_BYTES: more than 131,040 rows, at any
 * V) return SEL_EWORKSPACE. The call allocates and frees nothing;
 * it zeroes the part of the array it uses with cudaMemsetAsync on `stream` and
 * launches on `stream`. The first call on a device looks the array's device
 * address up (cudaGetSymbolAddress), so make that first call before any
 * stream capture. Later calls look it up again unless their stream is being
 * captured, so a cudaDeviceReset or another context made current between
 * calls is followed. Every call on a device shares the one array: calls that
 * may overlap on the GPU (different streams without ordering) race; order
 * them (one stream, or an event between streams).
 */
#define SEL_NOALLOC_SCRATCH_BYTES (1u << 20)
sel_status sel_argmax_noalloc(const float *d_logits, uint32_t rows, uint32_t V,
                              uint32_t *d_out_ids, cudaStream_t stream);

/*
 * sel_argmax_excluding -- Muser ch. 21, 21.4, the greedy serving variant: the
 * request's end-of-generation ids are masked out inside the reduction only
 * (the logits are left untouched, for log-probabilities and sessions), while
 * the NaN/Inf latch still covers every logit. Per row: the lowest id of the
 * maximum over the ids not in the set.
 *
 *   d_excluded  device array of n_excluded ids, one set for every row; ids
 *               >= V are ignored, duplicates do not matter, any order
 *   n_excluded  0 <= n_excluded <= SEL_MAX_EXCLUDED (0: plain sel_argmax)
 *   the rest    as for sel_argmax (same workspace: SEL_OP_ARGMAX)
 * A row with a nonfinite logit (excluded or not), or whose ids are all
 * excluded, gets 0xFFFFFFFF.
 */
#define SEL_MAX_EXCLUDED 256u
sel_status sel_argmax_excluding(const float *d_logits, uint32_t rows, uint32_t V,
                                const uint32_t *d_excluded, uint32_t n_excluded,
                                uint32_t *d_out_ids, void *d_ws, size_t ws_bytes,
                                cudaStream_t stream);

/*
 * Vocabulary shards -- llama.cpp PR 49, "Problem": under a tensor split each
 * GPU holds a share of the output head (about 155k and 93k of the 248k
 * columns there), so each computes the logits of one contiguous id range.
 * A shard runs sel_topk on its own slice (shard-local ids); the lists of all
 * shards of a row, gathered into one buffer, merge into the top k of the
 * whole row, with the same values, ids and order as sel_topk on the
 * unsharded row (ties: lower global id). Argmax is the case k = 1.
 *
 *   d_vals     [rows][G][k] f32: shard g's sel_topk values for each row
 *   d_ids      [rows][G][k] u32: shard g's sel_topk ids (local to the shard)
 *   G          number of shards, 1 <= G <= SEL_MAX_SHARDS
 *   k          entries per shard list, 1 <= k <= SEL_MAX_K
 *   h_offsets  HOST array of G + 1 increasing ids: shard g covers global
 *              ids [h_offsets[g], h_offsets[g+1]), at least k of them;
 *              h_offsets[G] <= SEL_MAX_V. Read during the call only.
 *   d_out_vals, d_out_ids  [rows][k]: the merged top k, global ids
 * A row in which any shard reported 0xFFFFFFFF (nonfinite logits), or whose
 * lists are malformed (an id outside its shard, a nonfinite value, a list
 * out of order), gets NaN values and 0xFFFFFFFF ids. No workspace: one block
 * per row, launched on `stream`. The gather itself (all-gather of the lists
 * between GPUs) is the caller's.
 */
#define SEL_MAX_SHARDS 64u
sel_status sel_merge_shards(const float *d_vals, const uint32_t *d_ids,
                            uint32_t rows, uint32_t G, uint32_t k,
                            const uint32_t *h_offsets, float *d_out_vals,
                            uint32_t *d_out_ids, cudaStream_t stream);

/*
 * Per-shard row statistics: what a shard's slice adds to the whole row's
 * softmax normaliser, mean log-weight and standard deviation, so that the
 * filters that look at the whole row (top-n-sigma, and sampling with
 * top_k == 0) can run on vocabulary shards. Written by sel_topk_stats, one
 * record per row of the slice; the caller all-gathers them with the lists.
 * With Tf the filter temperature (the policy's temperature, or 1 in the
 * temperature-last order, or 1 for a greedy policy) and m the slice's
 * largest logit:
 */
typedef struct sel_row_stats {
    float max;      /* m: the slice's largest logit */
    uint32_t flags; /* bit 0: the slice holds a NaN or +-Inf logit (the
                       other fields are then meaningless) */
    float x0;       /* shift of s1 and s2: the slice's first logit */
    uint32_t n;     /* logits in the slice */
    double s1;      /* sum over the slice of (x - x0) */
    double s2;      /* sum over the slice of (x - x0)^2 */
    double z;       /* sum of exp((x - m) / Tf) */
    double h;       /* sum of exp((x - m) / Tf) * (x - m) / Tf; 0 unless the
                       policy's typical_p filter is on */
} sel_row_stats;    /* 48 bytes */

/*
 * sel_topk_stats -- sel_topk on a shard's slice plus that slice's
 * sel_row_stats, from one read of the slice.
 *
 *   d_logits, rows, V, k, d_out_vals, d_out_ids  as for sel_topk (V is the
 *              slice's width; ids local to the slice)
 *   p          the sampling policy (host pointer, read during the call):
 *              fixes Tf and whether h is summed
 *   d_stats    [rows] sel_row_stats, device
 *   d_ws       workspace of sel_workspace_bytes(SEL_OP_TOPK, rows, V, k)
 * A row with a nonfinite logit gets SEL_INVALID_ID ids (as sel_topk) and
 * flags bit 0.
 */
sel_status sel_topk_stats(const float *d_logits, uint32_t rows, uint32_t V,
                          uint32_t k, const sel_sample_params *p,
                          float *d_out_vals, uint32_t *d_out_ids,
                          sel_row_stats *d_stats, void *d_ws, size_t ws_bytes,
                          cudaStream_t stream);

/*
 * The survivor set and draw of one row of full-row sampling on shards:
 * written by sel_sample_shards, read by sel_shard_draw_mass and
 * sel_shard_draw. Opaque; every rank holds the same copy when it ran
 * sel_sample_shards on the same gathered inputs.
 */
typedef struct sel_shard_plan {
    uint32_t opaque[12];
} sel_shard_plan;   /* 48 bytes */

/*
 * sel_sample_shards -- the sampling chain of sel_sample over a row split
 * into vocabulary shards, from the shards' gathered lists and statistics.
 *
 * With top_k > 0 the top-k filter comes first in the chain (Muser ch. 21,
 * 21.7), so the rest of the chain needs only the top_k candidates (llama.cpp
 * PR 49, "Change"): the merged lists give exactly the candidates sel_sample
 * finds in the whole row, and the call writes (id, probability) directly.
 * Top-n-sigma needs the whole row's standard deviation as well, merged here
 * from the shards' (n, x0, s1, s2): pass d_stats.
 *
 * With top_k == 0 (full-row sampling) the call decides each row's survivor
 * set from the merged 64 most probable candidates and the merged
 * normaliser (sum of z rescaled to the row's maximum), as sel_sample does,
 * and writes it to d_plan; the draw over the survivors, in ascending global
 * id, then runs on the shards: sel_shard_draw_mass on every shard,
 * an all-gather of the masses, sel_shard_draw on every shard, and an
 * all-reduce of the shards' outputs (minimum of the ids, sum of the
 * probabilities). A row whose top-p cut lies past the 64 candidates (the
 * unsharded call finds it by a search over the row) and a row whose
 * typical window runs past them fail closed in this form, with error bit 8
 * raised by sel_shard_draw.
 *
 *   d_vals, d_ids  [rows][G][k], as for sel_merge_shards; each shard list is
 *              sel_topk (or sel_topk_stats) of the slice with k = p->top_k,
 *              or with k = min(64, smallest slice) when p->top_k == 0 (any
 *              k when p->temperature == 0: greedy takes the top candidate)
 *   d_stats    [rows][G] sel_row_stats from sel_topk_stats on each slice with
 *              the same policy, or NULL when top_k > 0 and top-n-sigma is off
 *   rows, G, k, h_offsets  as for sel_merge_shards
 *   p, d_uniforms  as for sel_sample
 *   d_out_ids, d_out_probs  [rows], as for sel_sample (top_k > 0 or greedy);
 *              unused (may be NULL) when top_k == 0
 *   d_plan     [rows] sel_shard_plan (top_k == 0; may be NULL otherwise)
 * Per-row errors as for sel_sample (0xFFFFFFFF, probability NaN): a shard
 * whose list or statistics report a nonfinite logit, a malformed list, or
 * statistics whose n differs from the shard's width fail the row closed.
 * Returns SEL_EINVAL when d_stats is NULL but top-n-sigma is on or
 * top_k == 0, or d_plan is NULL with top_k == 0.
 */
sel_status sel_sample_shards(const float *d_vals, const uint32_t *d_ids,
                             const sel_row_stats *d_stats, uint32_t rows,
                             uint32_t G, uint32_t k, const uint32_t *h_offsets,
                             const sel_sample_params *p,
                             const float *d_uniforms, uint32_t *d_out_ids,
                             float *d_out_probs, sel_shard_plan *d_plan,
                             cudaStream_t stream);

/*
 * sel_shard_draw_mass -- step 1 of the full-row draw on shards: each
 * shard's mass of the row's survivors, sum of exp((x - max) / T) over the
 * survivors in its slice (the row's maximum and T from the plan). Also
 * leaves per-chunk sums in d_ws for sel_shard_draw.
 *
 *   d_logits   [rows][V] f32: this shard's slice (V its width)
 *   offset     the slice's first global id (h_offsets[g])
 *   d_plan     [rows] from sel_sample_shards
 *   d_mass     [rows] f64, device: this shard's survivor mass (0 for a row
 *              that fails closed)
 *   d_ws       workspace of sel_workspace_bytes(SEL_OP_SHARD_DRAW, rows, V,
 *              0), kept untouched until the matching sel_shard_draw
 */
sel_status sel_shard_draw_mass(const float *d_logits, uint32_t rows, uint32_t V,
                               uint32_t offset, const sel_shard_plan *d_plan,
                               double *d_mass, void *d_ws, size_t ws_bytes,
                               cudaStream_t stream);

/*
 * sel_shard_draw -- step 2: with every shard's mass gathered, the draw
 * u * total falls in one shard (shards in id order, a fixed-order scan);
 * that shard walks its survivors in ascending id and writes the global id
 * and its probability (weight / total). Every other shard writes
 * SEL_OTHER_SHARD and probability 0, so an all-reduce (minimum of the ids,
 * sum of the probabilities) over the shards gives the row's result on
 * every rank. A row that fails closed gets SEL_INVALID_ID and NaN on every
 * shard.
 *
 *   d_logits, rows, V, offset, d_plan  as for sel_shard_draw_mass
 *   g, G       this shard's index and the number of shards
 *   d_masses   [rows][G] f64: every shard's d_mass, gathered in shard order
 *   d_out_ids, d_out_probs  [rows]
 *   d_ws       the workspace of this shard's sel_shard_draw_mass call; its
 *              first word collects error bit 8 (a cut past the candidates)
 */
#define SEL_OTHER_SHARD 0xFFFFFFFEu
sel_status sel_shard_draw(const float *d_logits, uint32_t rows, uint32_t V,
                          uint32_t offset, uint32_t g, uint32_t G,
                          const sel_shard_plan *d_plan, const double *d_masses,
                          uint32_t *d_out_ids, float *d_out_probs, void *d_ws,
                          size_t ws_bytes, cudaStream_t stream);

/*
 * Speculative acceptance on vocabulary shards. Under a tensor split each
 * rank holds one id range of every target and draft row (llama.cpp PR 49,
 * "Problem"). The acceptance rules ("Speculative-decoding acceptance rules",
 * Modified rejection sampling and Argmax-against-argmax) need, per row, the
 * softmax normaliser (or the argmax) of the whole row and the logits at the
 * draft tokens; the final draw needs the residual's mass on every shard
 * (one exchange of per-shard totals). The steps, on every rank:
 *   1. spec_shard_stats on the rank's slices: one spec_shard_part per row;
 *   2. all-gather the parts into [S][G][2K+1];
 *   3. spec_accept_shards: the merged statistics, the acceptance chain (the
 *      same on every rank), accepted counts and emitted tokens, and, in the
 *      rejection rule, a draw plan per sequence;
 *   4. (rejection rule) spec_shard_draw_mass on the slices, all-gather the
 *      [S][2] masses into [S][G][2], spec_shard_draw on the slices, and an
 *      all-reduce (minimum) of the emitted arrays over the ranks: the shard
 *      the draw falls in writes the token's global id, the others
 *      SEL_OTHER_SHARD.
 */
typedef struct spec_shard_part {
    float max;        /* the slice's largest logit */
    uint32_t idx;     /* argmax rule: global id of the slice's first maximum;
                         bit 31: the slice holds a NaN or +-Inf logit */
    float x_tok;      /* rejection rule: the row's logit at its draft token,
                         when has_tok */
    uint32_t has_tok; /* 1: the row's draft token lies in this slice */
    double z;         /* rejection rule: sum of exp((x - max) / T) */
    uint32_t pad[2];
} spec_shard_part;    /* 32 bytes */

typedef struct spec_shard_plan {
    uint32_t opaque[8];
} spec_shard_plan;    /* 32 bytes */

#define SPEC_SHARD_MAX_K 64u

/*
 * spec_shard_stats -- step 1 on one shard.
 *
 *   d_target   [S][K+1][V] f32: this shard's slice of every target row
 *   d_draft    [S][K][V] f32: the slices of the draft rows (rejection rule)
 *   d_draft_tokens [S][K] u32: the draft tokens, GLOBAL ids
 *   V, offset  the slice's width and first global id
 *   params     as for spec_accept
 *   d_parts    [S][2K+1] spec_shard_part: per sequence, target rows 0..K,
 *              then draft rows 0..K-1 (unused in the argmax rule)
 *   d_ws       workspace of sel_workspace_bytes(SEL_OP_SPEC, S, V, K)
 * K <= SPEC_SHARD_MAX_K (else SEL_EUNSUPPORTED).
 */
sel_status spec_shard_stats(const float *d_target, const float *d_draft,
                            const uint32_t *d_draft_tokens, uint32_t S,
                            uint32_t K, uint32_t V, uint32_t offset,
                            const spec_params *params, spec_shard_part *d_parts,
                            void *d_ws, size_t ws_bytes, cudaStream_t stream);

/*
 * spec_accept_shards -- step 3: the acceptance chain of spec_accept from the
 * gathered parts.
 *
 *   d_parts    [S][G][2K+1]: every shard's spec_shard_stats output, shard
 *              order = id order
 *   G, h_offsets  as for sel_merge_shards (h_offsets[G] = V)
 *   d_draft_tokens, params, d_u_acc, d_u_fin, d_accepted, d_emitted  as for
 *              spec_accept; in the rejection rule the emitted entry at the
 *              accepted count is left SEL_INVALID_ID for the draw
 *   d_plan     [S] spec_shard_plan (rejection rule; may be NULL in the
 *              argmax rule, which emits its final token here)
 * Per-sequence errors as for spec_accept; parts that do not fit their shard
 * (a draft token's logit on no shard or on two) also invalidate the sequence.
 */
sel_status spec_accept_shards(const spec_shard_part *d_parts,
                              const uint32_t *d_draft_tokens, uint32_t S,
                              uint32_t K, uint32_t G,
                              const uint32_t *h_offsets,
                              const spec_params *params, const float *d_u_acc,
                              const float *d_u_fin, uint32_t *d_accepted,
                              uint32_t *d_emitted, spec_shard_plan *d_plan,
                              cudaStream_t stream);

/*
 * spec_shard_draw_mass -- step 4a on one shard: the residual mass
 * sum max(p - q, 0) and the target mass sum p over this slice of the rows
 * each sequence's plan names (the rejecting position's target and draft
 * rows, or target row K for a bonus draw).
 *
 *   d_target, d_draft, S, K, V  as for spec_shard_stats
 *   d_plan     [S] from spec_accept_shards
 *   d_mass     [S][2] f64: (residual, target) masses of this slice
 *   d_ws       workspace of sel_workspace_bytes(SEL_OP_SPEC_SHARD_DRAW, S,
 *              V, 0), kept untouched until the matching spec_shard_draw
 */
sel_status spec_shard_draw_mass(const float *d_target, const float *d_draft,
                                uint32_t S, uint32_t K, uint32_t V,
                                const spec_shard_plan *d_plan, double *d_mass,
                                void *d_ws, size_t ws_bytes,
                                cudaStream_t stream);

/*
 * spec_shard_draw -- step 4b on shard g: the draw with u_fin over the
 * residual (over p when the residual's total is <= 0), in ascending global
 * id across the shards; writes d_emitted[s][accepted] (the token's global
 * id on the shard it falls in, SEL_OTHER_SHARD on the others).
 *
 *   d_target, d_draft, S, K, V, offset  as for spec_shard_stats
 *   g, G       this shard and the number of shards
 *   d_plan     [S] from spec_accept_shards
 *   d_masses   [S][G][2] f64: every shard's d_mass, gathered in shard order
 *   d_emitted  [S][K+1] u32: this rank's spec_accept_shards output
 *   d_ws       this shard's spec_shard_draw_mass workspace
 */
sel_status spec_shard_draw(const float *d_target, const float *d_draft,
                           uint32_t S, uint32_t K, uint32_t V, uint32_t offset,
                           uint32_t g, uint32_t G,
                           const spec_shard_plan *d_plan,
                           const double *d_masses, uint32_t *d_emitted,
                           void *d_ws, size_t ws_bytes, cudaStream_t stream);

/* Static description of a status code. */
const char *sel_status_string(sel_status status);

#ifdef __cplusplus
}
#endif

#endif /* SEL_H */
