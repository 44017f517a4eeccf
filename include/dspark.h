/*
 * dspark.h - C ABI of the GB300 DSpark/DFlash block drafter.
 *
 * The drafter reads the target model's hidden states at m tapped layers for
 * every context token, keeps a per-layer context K/V cache, and drafts a block
 * of gamma tokens in one parallel pass followed by a short sequential Markov
 * chain.  Sources (by page and section):
 *   "module-dflash.ts" (mlx-bun 0.0.7 -> 0.0.9): the header comment (Eq 2,
 *       Eq 3), #buildContext, #buildBlock, #maskBias, #layer, #backbone,
 *       #baseLogits, #markov, #confidence, forwardInfer, initFromDims;
 *   "src/dspark-runtime.js" (minicpm5-2b-webgpu): updateContext (context
 *       K/V computed once per token and stored per layer), propose (draft
 *       step with the Markov chain and argmax kept on the device).
 *
 * Conventions for every call:
 *   - Pointers named *_dev are CUDA device pointers on the handle's device;
 *     pointers named *_host are host pointers (pageable or pinned).
 *   - Matrices are row-major [out, in] (the input dimension is contiguous).
 *   - "dtype" tensors are bf16 (raw 16-bit patterns) when cfg.dtype is
 *     DSPARK_BF16 and IEEE float32 when it is DSPARK_FP32.  Norm vectors are
 *     always float32.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Device-pointer
 *     calls are asynchronous on it and never synchronise the host; *_host calls
 *     synchronise `stream` before they return.
 *   - Errors the host can see (bad configuration, NULL pointer, token outside
 *     [0, vocab), context over capacity) are returned at once and nothing is
 *     launched.  Violations only the device can see (a batched token or
 *     sequence id out of range, a batched context over capacity) set a device
 *     error word; dspark_check() and dspark_context_length() report it as
 *     DSPARK_ERR_DEVICE.  dspark_last_error() describes the last failure.
 *   - A handle is not thread-safe; calls on one handle are ordered by the
 *     caller.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DSPARK_OK = 0,
    DSPARK_ERR_INVALID_ARG = 1,  /* bad config, NULL pointer, token out of range          */
    DSPARK_ERR_CAPACITY = 2,     /* context longer than max_ctx, too many sequences        */
    DSPARK_ERR_CUDA = 3,         /* a CUDA runtime call failed (message in last_error)     */
    DSPARK_ERR_UNSUPPORTED = 4,  /* shape outside what the kernels implement                */
    DSPARK_ERR_TIMEOUT = 5,      /* a bounded device wait gave up                           */
    DSPARK_ERR_OOM = 6,          /* device allocation failed                                */
    DSPARK_ERR_DEVICE = 7        /* the device error word was set (see dspark_check)        */
} dspark_status;

typedef enum { DSPARK_BF16 = 0, DSPARK_FP32 = 1 } dspark_dtype;

/* FFN activation of the gated FFN in #layer: SiLU(gate)*up (the "silu" kernel of
 * "src/dspark-runtime.js", propose) or tanh-GELU(gate)*up (MLX geluApprox). */
typedef enum { DSPARK_ACT_SILU = 0, DSPARK_ACT_GELU_TANH = 1 } dspark_act;

/* Drafter dimensions: DflashConfig and TargetDims of "module-dflash.ts". */
typedef struct dspark_config {
    int32_t hidden;       /* H: target hidden size                                     */
    int32_t n_taps;       /* m: tapped target layers; features are [T, m*H]             */
    int32_t d_draft;      /* d: drafter width; multiple of 64                           */
    int32_t n_heads;      /* d % n_heads == 0; head_dim = d / n_heads, <= 256, even     */
    int32_t n_layers;     /* draft layers                                               */
    int32_t ff_mult;      /* F = ff_mult * d                                            */
    int32_t gamma;        /* block size, 1 <= gamma <= 16                               */
    int32_t vocab;        /* V                                                          */
    int32_t markov_rank;  /* r, multiple of 8, <= 1024                                  */
    float eps;            /* RMSNorm epsilon                                            */
    int32_t dtype;        /* dspark_dtype                                               */
    int32_t act;          /* dspark_act                                                 */
    int32_t max_ctx;      /* context capacity per sequence (tokens)                     */
    int32_t max_seqs;     /* number of sequences with their own caches (>= 1)           */
    /* The variant of "src/dspark-runtime.js" (noiseNormRope / contextNormRope, K/V
     * width below H).  All zero: multi-head attention without either transform.   */
    int32_t n_kv_heads;   /* K/V heads (0: n_heads); n_heads % n_kv_heads == 0; query   */
                          /* head h reads K/V head h / (n_heads / n_kv_heads)           */
    int32_t qk_norm;      /* 1: RMSNorm of every head of Q and K (weights q_norm,       */
                          /* k_norm [head_dim] per layer, the same eps)                 */
    float rope_theta;     /* > 0: rotary embedding of Q and K after the norm, rotate-   */
                          /* half layout: entries e, e + hd/2 turned by                 */
                          /* pos * theta^(-2e/hd); context row t at pos t, block row j  */
                          /* at pos L + j (L = context length)                          */
} dspark_config;

/* Weights, as device pointers in cfg.dtype unless noted (norm vectors float32).
 * Names follow buildNames of "module-dflash.ts"; shapes are [out, in]. */
typedef struct dspark_weights {
    const void* W_c;          /* [d, m*H]      Eq 2 projection                           */
    const float* ctx_norm;    /* [d]                                                     */
    const void* embed;        /* [V, H]        the target's token embedding (BORROWED:   */
                              /*               must stay valid while the handle lives)   */
    const void* tok_proj;     /* [d, H]                                                  */
    const void* mask_emb;     /* [gamma-1, d]  (may be NULL when gamma == 1)             */
    const void* block_pos;    /* [gamma, d]                                              */
    const float* const* attn_norm;  /* host array of n_layers device pointers, each [d]  */
    const void* const* wq;          /* ... each [d, d]                                   */
    const void* const* wk;          /* ... each [d_kv, d], d_kv = n_kv_heads * head_dim   */
    const void* const* wv;          /* ... each [d_kv, d]                                */
    const void* const* wo;          /* ... each [d, d]                                   */
    const float* const* ff_norm;    /* ... each [d]                                      */
    const void* const* w_gate;      /* ... each [F, d]                                   */
    const void* const* w_up;        /* ... each [F, d]                                   */
    const void* const* w_down;      /* ... each [d, F]                                   */
    const float* out_norm;    /* [d]                                                     */
    const void* out_proj;     /* [V, d]        d -> vocab head                           */
    const void* markov_w1;    /* [V, r]        previous-token factor (row gather)        */
    const void* markov_w2;    /* [V, r]        vocab factor (bias = w2 . w1[prev])       */
    const void* conf_w;       /* [d + r]       confidence head weight                    */
    const void* conf_b;       /* [1]           confidence head bias                      */
    const float* const* q_norm;     /* host array of n_layers device pointers, each       */
    const float* const* k_norm;     /* [head_dim] (read only when cfg.qk_norm)            */
} dspark_weights;

typedef struct dspark_handle dspark_handle;

/* Create a drafter on the current CUDA device.  Copies and repacks every weight
 * except `embed` into library-owned device memory (the caller may free them
 * once this returns, after synchronising `stream`), and allocates the context
 * caches: n_layers x max_seqs x 2 x (max_ctx + gamma) x d_kv elements of dtype.
 * Source: initFromDims / DflashDrafter constructor ("module-dflash.ts"), which
 * also rejects d % n_heads != 0.  Returns DSPARK_ERR_INVALID_ARG for a bad
 * config or NULL weight, DSPARK_ERR_UNSUPPORTED for shapes outside the limits
 * above, DSPARK_ERR_OOM if the device is full.  *out is NULL on failure. */
dspark_status dspark_create(const dspark_config* cfg, const dspark_weights* w, void* stream,
                            dspark_handle** out);

/* Free every library-owned buffer.  Synchronises the device first.  NULL is a no-op. */
void dspark_destroy(dspark_handle* h);

/* Context ingest for sequence 0 (Eq 2 + Eq 3; "src/dspark-runtime.js"
 * updateContext): for T new context rows feats_dev [T, m*H] (dtype, taps
 * concatenated on the feature axis), compute H_ctx = RMSNorm(W_c x) * ctx_norm
 * and, for every layer i, append W_k,i n and W_v,i n with
 * n = RMSNorm(H_ctx) * attn_norm_i to the layer's cache (with the variant fields of the
 * config, the K heads normalised and turned at their positions first).  T = 0 is a no-op.
 * DSPARK_ERR_CAPACITY if the context would exceed max_ctx (nothing launched). */
dspark_status dspark_ingest_context(dspark_handle* h, const void* feats_dev, int32_t T, void* stream);

/* Draft one block for sequence 0 ("module-dflash.ts" forwardInfer, greedy):
 * block rows (#buildBlock: tok_proj E[last_token] + block_pos[0], then
 * mask_emb[j-1] + block_pos[j]), n_layers of #layer attending over
 * [context ++ block] with no mask, out_norm, base logits U = out_proj y, then
 * for k = 0..gamma-1: logits_k = U_k + w2 w1[prev_k] (prev_0 = last_token,
 * prev_k = token_{k-1}), token_k = argmax (lowest index on ties; a draw instead
 * when dspark_set_sampling set a temperature), conf_k = sigmoid(conf_w . [y_k ; w1[prev_k]] + conf_b).
 * With the variant fields of the config, the heads of Q and of the block's K rows are
 * normalised and turned at positions L + j before the attention.
 * Outputs: tokens_dev [gamma] int32, conf_dev [gamma] float, and, if not NULL,
 * logits_dev [gamma, V] float.  The context is not modified. */
dspark_status dspark_draft(dspark_handle* h, int32_t last_token, int32_t* tokens_dev, float* conf_dev,
                           float* logits_dev, void* stream);

/* dspark_ingest_context(h, feats_dev, T) followed by dspark_draft(h, last_token, ...), with the same
 * arguments, errors and results (page 1's updateContext then propose, "src/dspark-runtime.js"), as one
 * call: the block rows, which read no context, are built on the handle's side stream while the T
 * rows are ingested on `stream`, and so is layer 0's QKV projection where its norm comes through the
 * block build (it writes the block's K/V rows at the length after the ingest); the draft continues
 * on `stream` once both are done.  The side stream's launches use scratch of their own.  The draft
 * runs without the handle's captured graph.  The call returns once everything is enqueued on
 * `stream`; feats_dev must stay valid until the work completes.  T = 0 drafts only. */
dspark_status dspark_ingest_and_draft(dspark_handle* h, const void* feats_dev, int32_t T, int32_t last_token,
                                      int32_t* tokens_dev, float* conf_dev, float* logits_dev, void* stream);

/* Batched ingest: sequences seq_ids_dev[i] (i < n_seqs) receive the feature rows
 * cu_tokens_dev[i] .. cu_tokens_dev[i+1]-1 of feats_dev [total_tokens, m*H]
 * (cu_tokens_dev: n_seqs+1 prefix sums, cu[0] = 0, cu[n] = total_tokens).  Each
 * sequence is ingested exactly as dspark_ingest_context would.  Sequence ids
 * must be distinct.  A sequence whose context would exceed max_ctx is left
 * unchanged and sets the device error word. */
dspark_status dspark_ingest_context_batched(dspark_handle* h, int32_t n_seqs, const int32_t* seq_ids_dev,
                                            const int32_t* cu_tokens_dev, const void* feats_dev,
                                            int32_t total_tokens, void* stream);

/* Batched draft: one block per sequence seq_ids_dev[i] with anchor
 * last_tokens_dev[i]; outputs tokens_dev [n_seqs, gamma], conf_dev [n_seqs, gamma],
 * logits_dev [n_seqs, gamma, V] or NULL.  Results equal n_seqs calls of
 * dspark_draft on the sequences' own caches.  n_seqs <= max_seqs. */
dspark_status dspark_draft_batched(dspark_handle* h, int32_t n_seqs, const int32_t* seq_ids_dev,
                                   const int32_t* last_tokens_dev, int32_t* tokens_dev, float* conf_dev,
                                   float* logits_dev, void* stream);

/* Host-buffer forms of ingest and draft for sequence 0, same arithmetic as the
 * device-pointer calls.  dspark_ingest_context_host copies feats_host [T, m*H] in
 * (through a library staging buffer, on `stream`), enqueues the ingest and returns
 * once feats_host has been read; the ingest completes in stream order.
 * dspark_draft_host runs the draft, copies tokens/conf (and logits, if logits_host
 * is not NULL) out and synchronises `stream`.  Consecutive host-buffer calls of one
 * handle go on one stream (the staging buffers are reused). */
dspark_status dspark_ingest_context_host(dspark_handle* h, const void* feats_host, int32_t T, void* stream);
dspark_status dspark_draft_host(dspark_handle* h, int32_t last_token, int32_t* tokens_host, float* conf_host,
                                float* logits_host, void* stream);

/* Token choice of the Markov chain ("module-dflash.ts", forwardInfer: processLogits +
 * sampleToken with a seeded KeyStream; "src/dspark-runtime.js", propose: the
 * temperature > 0 branch).  temperature = 0 (the default): argmax, lowest index on ties.
 * temperature > 0: the token of block position k is drawn from softmax(l / temperature)
 * over the top_k largest logits (ties to the lower index; top_k = 0: the whole
 * vocabulary), as argmax of l_v / temperature - ln(-ln u_v), where u_v is built from the
 * SplitMix64 output number c + 1 of the stream seeded with `seed`,
 * c = slot * 2^48 + (draw mod 2^24) * 2^24 + v, u = (top 24 bits + 0.5) / 2^24, and draw =
 * the slot's draw counter + k; every draft call advances the counters of its sequences by
 * gamma.  This call resets every counter to 0 (stream-ordered on `stream`) and applies to
 * the following draft calls.  Errors: INVALID_ARG (temperature negative or not finite,
 * top_k outside [0, 64]), UNSUPPORTED (vocabulary above 256 x 2048 entries or rank above
 * 1024 with sampling on). */
dspark_status dspark_set_sampling(dspark_handle* h, float temperature, int32_t top_k, uint64_t seed, void* stream);

/* Set the context length of seq_id to 0 (stream-ordered on `stream`). */
dspark_status dspark_reset(dspark_handle* h, int32_t seq_id, void* stream);

/* Context length of seq_id, read from the device (synchronises the device);
 * returns DSPARK_ERR_DEVICE if the device error word is set. */
dspark_status dspark_context_length(dspark_handle* h, int32_t seq_id, int32_t* out_host);

/* Self-test of the bounded device waits (failure detection without a fault): runs
 * one of the library's waits on device words that nothing completes, in a small
 * kernel of its own on a private stream: which = 0 the single-sequence Markov
 * chain's arrival count, 1 the resident chain's barrier, 2 the cooperative
 * chain's barrier, 3 the one-launch layers' grid barrier, 4 the tensor-core
 * kernels' mbarrier wait, 5 the one-launch step's grid barrier (whose outcome
 * every thread of the CTA takes alike).  The wait gives up after its limit (about one second)
 * and the kernel returns normally; *word_host (may be NULL) receives the error
 * word it recorded, DSPARK_DEVERR_TIMEOUT when the wait gave up.  The device
 * stays usable.  Synchronises that stream; INVALID_ARG for another `which`. */
dspark_status dspark_selftest_wait(int32_t which, int32_t* word_host);

/* Read and clear the device error word (synchronises the device).  *word_host
 * (may be NULL) receives it: 0 = none, otherwise a DSPARK_DEVERR_* bit set. */
#define DSPARK_DEVERR_TOKEN_RANGE 1   /* a batched anchor token outside [0, V)        */
#define DSPARK_DEVERR_SEQ_RANGE 2     /* a batched sequence id outside [0, max_seqs)  */
#define DSPARK_DEVERR_CAPACITY 4      /* a batched ingest would exceed max_ctx        */
#define DSPARK_DEVERR_NONFINITE 8     /* a logit row had no finite maximum            */
#define DSPARK_DEVERR_TIMEOUT 16      /* a bounded wait inside a kernel gave up       */
dspark_status dspark_check(dspark_handle* h, int32_t* word_host);

/* Device pointers to the library-owned cache of (seq_id, layer): K and V rows
 * [max_ctx + gamma, d] of dtype, row stride d elements; rows [0, length) hold
 * the context.  For inspection only: the pointers stay valid until destroy. */
dspark_status dspark_get_cache(dspark_handle* h, int32_t seq_id, int32_t layer, const void** k_dev,
                               const void** v_dev);

/* Description of the last error on this handle (or of the last failed create
 * when h is NULL).  Never NULL. */
const char* dspark_last_error(const dspark_handle* h);

/* Timing of the step's kernel classes with CUDA events recorded on the calls'
 * own stream around each class of launches (no extra synchronisation).
 * dspark_profile(h, mask) with mask != 0 clears the counters and starts
 * recording the classes whose bit is set (bit i = the i-th class name that
 * dspark_profile_read reports; -1 = all); mask 0 stops.
 * dspark_profile_read fills up to `max` entries (class name, summed device
 * milliseconds, number of timed ranges, kernel launches in those ranges),
 * synchronising the recorded events first, and returns the number of classes
 * (negative on error). */
dspark_status dspark_profile(dspark_handle* h, int32_t class_mask);
int32_t dspark_profile_read(dspark_handle* h, int32_t max, const char** names_host, double* ms_host,
                            int64_t* ranges_host, int64_t* launches_host);

/* The contraction inside every projection of the step ("module-dflash.ts":
 * the ops.matmul calls of #buildContext, #buildBlock, #layer, #baseLogits),
 * as a standalone call: out[m, n] = sum_k A[m, k] W[n, k], fp32 result.
 * A_dev [M, K] (row stride lda elements) and W_dev [N, K] are both bf16
 * (dtype DSPARK_BF16) or both float32 (DSPARK_FP32); out_dev [M, N] float32
 * with row stride ldo.  `kernel` selects the implementation: 0 the one the step
 * would use for this shape, 1 SIMT tiles, 2 weight streaming (M <= 16, K % 8 == 0),
 * 3 tcgen05 tensor cores in 128 x 256 tiles (bf16, K >= 64, K % 8 == 0, 16-byte
 * aligned rows), 4 tcgen05 weight streaming (as 3, and M <= 16), 5 the wide tcgen05
 * form (as 3, and M <= 320): W's rows on the MMA's 128-row side and A's rows on its
 * N side in one or two groups, so no A tile is padded to 128 rows; kernel 0 takes it
 * where M <= 160 or 257 <= M <= 320, and N is at least 128 x the SM count.
 * DSPARK_ERR_UNSUPPORTED if the chosen kernel cannot take the shape. */
dspark_status dspark_linear(int32_t dtype, const void* A_dev, int64_t lda, const void* W_dev, int32_t M, int32_t N,
                            int32_t K, float* out_dev, int64_t ldo, int32_t kernel, void* stream);

/* out = A W^T with the weight-streaming tensor-core kernel (dspark_linear's
 * kernel 4), for callers that cannot allocate device memory: code living in
 * another runtime's memory pool, allocator-free serving loops, contexts whose
 * allocations are frozen after start-up.  The pages have no counterpart of
 * this call; it is an interface of this library.  It allocates nothing: the
 * kernel's split-K scratch is a static device array of
 * DSPARK_NOALLOC_SCRATCH_FLOATS floats plus DSPARK_NOALLOC_MAX_TILES tickets,
 * held by every GPU that loads the library until the process exits.  The first
 * call on a device looks up the array's device address (cudaGetSymbolAddress)
 * with that device current, so make that first call before any stream
 * capture.  Every call shares the array: the tickets are cleared on each call,
 * and calls whose work overlaps on the GPU race.
 * Shapes: bf16 A_dev [M, K] (row stride lda), bf16 W_dev [N, K], float out_dev
 * [M, N] (row stride ldo); 1 <= M <= 16, K >= 64, K % 8 == 0, lda % 8 == 0,
 * 16-byte aligned A and W, N <= 128 * DSPARK_NOALLOC_MAX_TILES
 * (DSPARK_ERR_CAPACITY beyond).  dspark_noalloc_last_error() describes a failure. */
#define DSPARK_NOALLOC_SCRATCH_FLOATS 4194304
#define DSPARK_NOALLOC_MAX_TILES 4096
dspark_status dspark_linear_stream_noalloc(const void* A_dev, int64_t lda, const void* W_dev, int32_t M, int32_t N,
                                           int32_t K, float* out_dev, int64_t ldo, void* stream);
/* Read and clear the error word that dspark_linear_stream_noalloc's kernels
 * share on the current device (a static device int, like their scratch).  The
 * kernel records DSPARK_DEVERR_TIMEOUT there when one of its bounded waits gives
 * up; the call that launched it has already returned DSPARK_OK, and its output
 * is incomplete.  Synchronous: waits for the device's earlier work, copies the
 * word into *word_host and, if it was set, clears it and returns
 * DSPARK_ERR_DEVICE (DSPARK_OK when it was 0).  Allocates nothing. */
dspark_status dspark_noalloc_check(int32_t* word_host);
const char* dspark_noalloc_last_error(void);

/* Choose between forms of the same computation, per handle (the library picks
 * by shape when a choice is 0, its default).  The forms compute the same
 * function up to floating-point rounding order; the choice exists so that each
 * form can be exercised and measured.  Captured draft graphs are dropped.
 *   DSPARK_PATH_LAYERS      batch-1 draft layers: 0 auto (the same as 1), 1 one
 *                           kernel per projection, 2 every layer in one launch on warp
 *                           MMAs, 3 the whole step up to the logits in one
 *                           launch on tcgen05 (block build, layers, out_proj)
 *   DSPARK_PATH_MARKOV      Markov chain of 1-2 sequences: 0 FMA-pipe chain,
 *                           1 the warp-MMA chain
 *   DSPARK_PATH_NORM_CHAIN  batch-1 per-kernel layers: 0 RMSNorm through the
 *                           residual epilogues, 1 separate normalisation launches
 *   DSPARK_PATH_GRAPHS      draft steps: 0 captured and replayed as CUDA graphs,
 *                           1 launched directly
 * DSPARK_ERR_INVALID_ARG for an unknown choice or value.  A forced form that
 * does not apply to the drafter or batch falls back to the default. */
#define DSPARK_PATH_LAYERS 0
#define DSPARK_PATH_MARKOV 1
#define DSPARK_PATH_NORM_CHAIN 2
#define DSPARK_PATH_GRAPHS 3
dspark_status dspark_set_path(dspark_handle* h, int32_t what, int32_t value);

/* Number of kernel launches issued by this handle since creation (all calls). */
int64_t dspark_launch_count(const dspark_handle* h);

/* Library version string. */
const char* dspark_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
