// Internal launchers of the drafter kernels (host side).  Every launcher
// enqueues on `st` and returns cudaGetLastError() of its launch.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dspark {

enum DType { DT_BF16 = 0, DT_F32 = 1 };

// ------------------------------------------------------------------ GEMM epilogues
// Every GEMM here computes acc[m, n] = sum_k A[m, k] * W[n, k] (W is [N, K],
// K contiguous) and hands acc to one of these epilogues.
enum EpiKind {
    EPI_STORE_F32 = 0,  // out_f32[m * ldo + n] = acc
    EPI_ADD_F32 = 1,    // out_f32[m * ldo + n] += acc            (residual add)
    EPI_SWIGLU = 2,     // columns come in (gate, up) pairs: out_act[m * ld_act + n/2] = act(gate) * up
    EPI_KV_CACHE = 3,   // columns [0, d) -> K cache, [d, 2d) -> V cache, row -> (seq, position)
    EPI_QKV = 4,        // columns [0, d) -> out_f32 (Q), [d, 2d) -> K cache, [2d, 3d) -> V cache
    EPI_MARKOV_T = 5,   // row m = vocabulary entry, column n = sequence: l = acc + U[n*gamma + k][m];
                        // logits (optional); argmax partial per sequence and 32 rows (tensor-core GEMM only)
};

struct EpiParams {
    int kind = EPI_STORE_F32;
    float* out_f32 = nullptr;
    int64_t ldo = 0;
    int split_rows = 0;          // EPI_STORE_F32 of a K-split tensor-core GEMM: rows between the ranges' outputs
    int64_t group_stride = 0;    // EPI_KV_CACHE of a grouped tensor-core GEMM: cache elements between groups
    int group_cols = 0;          // EPI_KV_CACHE of one product over several groups side by side: columns per
                                 // group (group = n / group_cols); 0: one group
    void* out_act = nullptr;     // EPI_SWIGLU output, element type act_dtype
    int act_dtype = DT_F32;
    int64_t ld_act = 0;
    int act = 0;                 // 0 SiLU, 1 tanh-GELU
    // cache epilogues
    void* cache = nullptr;       // layer base: K of seq s at cache + s*seq_stride, V at + kv_off
    int cache_dtype = DT_BF16;
    int64_t seq_stride = 0;      // elements between sequences
    int64_t kv_off = 0;          // elements from K to V of one sequence
    int d = 0;
    int d_kv = 0;                // cache row width (0: d); EPI_QKV: Q is columns [0, d), K and V d_kv each
    int max_rows = 0;            // rows per sequence cache (positions must be < max_rows)
    const int* row_seq = nullptr;  // EPI_KV_CACHE: sequence slot per GEMM row (nullptr: slot 0)
    const int* row_pos = nullptr;  // EPI_KV_CACHE: position per GEMM row, -1 = drop (nullptr: len[slot] + m)
    const int* seq_len = nullptr;  // device context lengths per slot
    int gamma = 1;                 // EPI_QKV: GEMM row m is block row m % gamma of sequence m / gamma
    const int* seq_ids = nullptr;  // EPI_QKV: slot of sequence b (nullptr: slot b)
    // EPI_MARKOV_T (row m = vocabulary entry, column n = sequence, block position mk_k)
    const float* mk_U = nullptr;   // [B*gamma, ldo] base logits
    float* mk_logits = nullptr;    // [B*gamma, ldo] or nullptr
    float* mk_part_v = nullptr;    // [B, mk_nch] best value of each 32-entry vocabulary chunk
    int* mk_part_i = nullptr;      // [B, mk_nch] its index
    int mk_nch = 0;                // ceil(V / 32)
    int mk_k = 0;
    // EPI_ADD_F32 of the weight-streaming GEMM, when ssp is set: besides x += acc, the next
    // projection's operand xb[m * ld_xb + n] = bf16(x * xb_g[n]) and the row sums of x^2 over each
    // 8 columns, ssp[(n / 8) * 16 + m] (what that projection's row-sum form reads)
    void* xb = nullptr;
    int64_t ld_xb = 0;
    const float* xb_g = nullptr;
    float* ssp = nullptr;
};

// Generic tiled SIMT GEMM (fp32 FMA), any M, N, K.  A rows may be gathered:
// A row m is at A + (a_rows ? a_rows[m] : m) * lda.
cudaError_t gemm_simt(int a_dtype, const void* A, int64_t lda, const int* a_rows, int w_dtype, const void* W,
                      int M, int N, int K, const EpiParams& ep, cudaStream_t st);

// Weight-streaming GEMM for M <= 16 activation rows: W is read once from HBM
// with 16-byte non-allocating loads, fp32 FMA.  A (fp32, or w_dtype when
// a_dtype says so) row m is at A + (a_rows ? a_rows[m] : a_row0 + m) * lda.
// K must be a multiple of 8.  When the rows of W alone cannot fill the GPU, K
// is split over CTAs; the partial sums go to `ws` (ws_floats capacity) and are
// added in a fixed order, so results do not depend on scheduling.
bool skinny_ok(int M, int K);
cudaError_t gemm_skinny(int a_dtype, const void* A, int64_t lda, const int* a_rows, int a_row0, int w_dtype,
                        const void* W, int M, int N, int K, const EpiParams& ep, float* ws, size_t ws_floats,
                        int num_sms, cudaStream_t st);

// ------------------------------------------------------------------ norms and block set-up
// out[r] = x[r] / sqrt(mean(x[r]^2) + eps) * w   (rows of length n, x fp32)
// With parts (nparts > 0): x += the partial products parts[s * part_stride + row * ldx + col], s in
// order, written back to x, before the norm (the residual of a K-split projection).
cudaError_t rmsnorm_rows(const float* x, int64_t ldx, const float* w, int rows, int n, float eps, int out_dtype,
                         void* out, int64_t ldo, cudaStream_t st, const float* parts = nullptr, int nparts = 0,
                         int64_t part_stride = 0);

// Ingest normalisation: H = RMSNorm(P) * ctx_norm, then for each layer i
// N_i = RMSNorm(H) * attn_norm_i, written to out + i * layer_stride (out_dtype).
// P holds nsplit partial products (K ranges) at P + s * split_stride; they are summed first.
cudaError_t ingest_norm(const float* P, int nsplit, int64_t split_stride, int rows, int d, float eps,
                        const float* ctx_norm, const float* const* attn_norm_dev, int n_layers, int out_dtype,
                        void* out, int64_t layer_stride, cudaStream_t st);

// x[b * gamma + j] = block_const[j] for b < B, j < gamma (fp32).
// x = the block rows of every sequence; with xb (one sequence only) also the first projection's
// chained operand: xb = bf16(x * g) and the 8-column sums of x^2 (the layout of EpiParams::ssp).
// Wd = bf16(W * g) column-wise: W, Wd bf16 [rows, K], g fp32 [K] (the attn_norm folded into weights).
cudaError_t scale_cols(const void* W, const float* g, int rows, int K, void* Wd, cudaStream_t st);
cudaError_t block_init(float* x, const float* block_const, int B, int gamma, int d, cudaStream_t st,
                       void* xb = nullptr, const float* g = nullptr, float* ssp = nullptr);
// block_const[0] = block_pos[0]; block_const[j] = mask_emb[j-1] + block_pos[j] (fp32 out).
cudaError_t block_const_init(int dtype, const void* mask_emb, const void* block_pos, int gamma, int d, float* out,
                             cudaStream_t st);
// out[i] = float(in[i]) for n elements of dtype.
cudaError_t to_float(int dtype, const void* in, int64_t n, float* out, cudaStream_t st);

// Kernel launches issued by this library so far (all handles); for accounting.
long long launch_count();
void note_launch(int n = 1);

// ------------------------------------------------------------------ attention
struct AttnParams {
    const float* q;          // [B*gamma, d], row b*gamma + j
    const void* cache;       // layer base (see EpiParams)
    int cache_dtype;
    int64_t seq_stride, kv_off;
    const int* seq_len;      // context length per slot (block rows sit at len .. len+gamma-1)
    const int* seq_ids;      // slot of sequence b (nullptr: b)
    int B, gamma, d, n_heads;
    int d_kv = 0, n_kv_heads = 0;  // cache row width and K/V heads (0: d, n_heads); head h reads K/V head
                                   // h / (n_heads / n_kv_heads)
    int n_chunks;            // split of the (len + gamma) keys of one sequence, 1 .. attn_max_chunks()
    int max_keys = 0;        // bound on any sequence's len + gamma (0: none known); picks the ring depth
    float* part;             // scratch: B * n_heads * n_chunks * gamma * (head_dim + 2) floats
    unsigned int* tickets;   // scratch: B * n_heads counters, zero before and after every launch
    void* out;               // [B*gamma, d] attention output, out_dtype
    int out_dtype;
};
size_t attn_scratch_floats(int B, int n_heads, int n_chunks, int gamma, int head_dim);
int attn_max_chunks(int cache_dtype, int head_dim, int gamma);
cudaError_t attention_init();  // once per process/device, before any launch or capture
// bf16 caches with head_dim 64 or 128 run on the tensor cores (mma.sync, key
// ranges of whole 64-key tiles, empty ranges exit); the rest on the SIMT kernel.
cudaError_t attention(const AttnParams& p, cudaStream_t st);
bool attention_tc_ok(int cache_dtype, int head_dim, int gamma);
int attention_tc_max_chunks();
// The key-range count at which the tensor-core attention merges the ranges of a (sequence, head) as
// one thread-block cluster, for sequences of up to max_keys keys; 0 when that form does not apply.
int attention_tc_cluster_chunks(int max_keys);
cudaError_t attention_tc_init();
cudaError_t attention_tc(const AttnParams& p, cudaStream_t st);

// ------------------------------------------------------------------ per-head Q/K norm and rotation
// The variant of "src/dspark-runtime.js" (noiseNormRope, contextNormRope): every head of a Q
// or K row is RMS-normalised with a [head_dim] weight (when given) and then turned by the
// rotary embedding (when theta > 0), rotate-half layout: entries e and e + hd/2 by the angle
// pos * theta^(-2e/hd).  In place: Q rows in fp32, K rows in the cache (dtype).
struct QkRope {
    float* q = nullptr;                  // block form: Q rows [B*gamma, ldq] (row b*gamma + j)
    int64_t ldq = 0;
    const float* q_norm = nullptr;       // [head_dim] or nullptr (no norm)
    const float* k_norm = nullptr;       // block form: this layer's [head_dim] or nullptr
    const float* const* k_norm_layers = nullptr;  // ingest form: device array of n_layers pointers, or nullptr
    void* cache = nullptr;               // layer base (block form) / layer 0 base (ingest form)
    int cache_dtype = DT_BF16;
    int64_t layer_stride = 0, seq_stride = 0;
    int d_kv = 0, max_rows = 0;
    const int* seq_len = nullptr;        // device context length per slot
    int n_heads = 0, n_kv_heads = 0, head_dim = 0, n_layers = 1;
    float eps = 0.f, theta = 0.f;
    const double* freq = nullptr;        // [head_dim / 2] theta^(-2e/hd), e < hd/2 (required when theta > 0)
    int B = 0, gamma = 0;                // block form: rows b*gamma + j at position len[slot] + j
    const int* seq_ids = nullptr;        // block form: slot of sequence b (nullptr: b)
    int rows = 0;                        // ingest form: context rows just written
    const int* row_seq = nullptr;        // ingest form: slot per row (nullptr: slot 0)
    const int* row_pos = nullptr;        // ingest form: position per row, -1 = dropped (nullptr: len[slot] + m)
};
// Fill dev[0, head_dim / 2) with theta^(-2e/hd), computed on the host in double (theta > 0).
cudaError_t qk_rope_freq_fill(float theta, int head_dim, double* dev, cudaStream_t st);
cudaError_t qk_rope_block(const QkRope& a, cudaStream_t st);   // the block's Q rows and K rows of one layer
cudaError_t qk_rope_ingest(const QkRope& a, cudaStream_t st);  // K rows of new context rows, every layer

// ------------------------------------------------------------------ persistent draft layers
// Every draft layer of sequence slot 0 (batch 1, bf16) in one cooperative launch,
// one CTA per SM: x (the block rows after the block build) -> x after the last
// layer; Q, the block's K/V cache rows, the attention output and the SwiGLU
// output pass through q, the cache, act and hact.  Host arrays of layer pointers.
struct DraftPersistArgs {
    float* x;
    float* q;
    void* act;                  // [gamma, d] bf16
    void* hact;                 // [gamma, F] bf16
    float* part;                // n_heads * nchunks * gamma * (head_dim + 4) floats
    void* cache;                // layer 0 base (bf16), slot 0
    int64_t layer_stride, kv_off;
    int max_rows;
    const int* seq_len;         // device; entry 0
    const void* const* wqkv;    // [n_layers] of [3d, d]
    const void* const* wo;      // [n_layers] of [d, d]
    const void* const* wgu;     // [n_layers] of [2F, d], rows (gate f, up f) interleaved
    const void* const* wd;      // [n_layers] of [d, F]
    const float* const* attn_norm;
    const float* const* ff_norm;
    int d, F, nh, nL, gamma, act_kind, nchunks;
    float eps;
    const void* maps;           // device [n_layers][4] slot tensor maps (tc_encode_slot_map) of wqkv, wo, wgu, wd
    int map3d;                  // the maps are 3-D
    unsigned long long* bar;    // 2 zero-initialised words
    unsigned int* epoch;        // zero-initialised
    int* err;
};
cudaError_t draft_persistent_init();  // once per process/device
bool draft_persistent_ok(const DraftPersistArgs& a);
cudaError_t draft_persistent(const DraftPersistArgs& a, int num_sms, cudaStream_t st);

// Batch-1 draft step up to the logits in one cooperative launch with tcgen05 projections
// (draft_step_tc.cu): block build, every layer, out_norm and out_proj.
struct DraftStepArgs {
    float* x;                   // [gamma, d]
    float* qkv;                 // [gamma, 3d] (the kernel zeroes it before use)
    float* gu;                  // [gamma, 2F] (idem)
    float* y;                   // [gamma, d]
    float* U;                   // [gamma, V]
    void* act;                  // [gamma, d] bf16 attention output
    float* apart;               // n_heads * nchunks * gamma * (head_dim + 4) floats
    unsigned int* hcnt;         // [2, n_heads] zero-initialised
    void* cache;                // layer 0 base (bf16), slot 0
    int64_t layer_stride, kv_off;
    int max_rows;
    const int* seq_len;         // device; entry 0
    const void* embed;          // [V, H] bf16
    const int* anchor_dev;      // device [1] or nullptr
    int anchor;
    const float* block_const;   // [gamma, d]
    const float* const* attn_norm;
    const float* const* ff_norm;
    const float* out_norm;
    const void* maps;           // device [2 + 4 n_layers] weight tensor maps (box 64 x 128, 128-byte swizzle)
    int d, F, H, V, nh, nL, gamma, act_kind, nchunks;
    float eps;
    unsigned long long* bar;    // 2 zero-initialised words
    unsigned int* epoch;        // zero-initialised
    int* err;
    // the Markov chain, argmax and confidences in the same launch (chain != 0; bf16 w1/w2, r % 64 == 0)
    int chain = 0, r = 0;
    const void* w1 = nullptr;
    const void* w2 = nullptr;
    const float* conf_w = nullptr;      // [d + r + 1]
    int* tokens = nullptr;              // [gamma]
    float* conf = nullptr;              // [gamma]
    float* logits = nullptr;            // [gamma, V] or nullptr
    unsigned long long* mk = nullptr;   // [2][17][num_sms] zero-initialised exchange words and counters
};
cudaError_t draft_step_tc_init();  // per device
bool draft_step_tc_ok(const DraftStepArgs& a, int num_sms);
cudaError_t draft_step_tc(const DraftStepArgs& a, int num_sms, cudaStream_t st);

// ------------------------------------------------------------------ Markov chain, argmax, confidence
struct MarkovParams {
    const float* U;          // [B*gamma, V] base logits
    const void* w1;          // [V, r], w_dtype
    const void* w2;          // [V, r], w_dtype
    int w_dtype;
    const float* y;          // [B*gamma, d] out-normed block rows
    const float* conf_w;     // [d + r + 1] fp32: weight, then the bias
    int B, gamma, V, r, d;
    int k;                   // block position
    const int* anchors;      // [B] device, or nullptr: use `anchor`
    int anchor;
    int* tokens;             // [B, gamma]
    float* conf;             // [B, gamma]
    float* logits;           // [B, gamma, V] or nullptr
    float* part_v;           // scratch: B * ctas floats
    int* part_i;             // scratch: B * ctas ints
    unsigned int* counters;  // scratch: B counters, zero between launches
    int* err;                // device error word
    int ctas;                // CTAs per sequence over V
    unsigned long long* keys = nullptr;  // markov_chain: 2 sets of keys_stride argmax words (sequence b, position k
                                         // at b * 16 + k), zero before the first launch
    int keys_stride = 0;                 // >= 16 * B
    unsigned int* epoch = nullptr;       // markov_chain: launch counter (selects the word set), zero-initialised
    unsigned long long* bar = nullptr;   // markov_chain_resident: 2 arrival counters, zero-initialised
};
int markov_ctas(int V);
cudaError_t markov_step(const MarkovParams& p, cudaStream_t st);
// All gamma positions in one cooperative launch (p.ctas CTAs per sequence, one
// bounded grid barrier per position, the argmax through 64-bit atomic max words
// p.keys; bar_count/bar_gen: zeroed words, left reusable).  markov_chain_max_ctas is the
// largest co-resident grid.
int markov_chain_max_ctas(int w_dtype);
// Many-sequence form: per position k, gather E[b] = w1[prev_b] (bf16, [B, r]),
// a tensor-core GEMM w2 . E^T ([V, B]) with the EPI_MARKOV_T epilogue, then
// markov_finish reduces the chunk partials of every sequence to its token and
// confidence.
cudaError_t markov_gather(const void* w1, int r, int V, const int* anchors, const int* tokens, int gamma, int k, int B,
                          void* E, cudaStream_t st);
cudaError_t markov_finish(const float* part_v, const int* part_i, int nchunks, const void* w1, int w_dtype,
                          const float* y, const float* conf_w, const int* anchors, int* tokens, float* conf, int B,
                          int gamma, int k, int d, int r, int V, int* err, cudaStream_t st);
cudaError_t markov_chain(const MarkovParams& p, unsigned int* bar_count, unsigned int* bar_gen, cudaStream_t st);
// Up to 8 sequences with bf16 weights and r in {64, 128, 256}: one cooperative CTA
// per SM keeps its slice of w2 in shared memory for the whole chain and runs the
// dot products on the warp MMA (the sequences are its N columns).  The draft step
// takes it for 3 to 8 sequences; one or two take the FMA form below.
cudaError_t markov_chain_resident_init();  // once per process/device
bool markov_chain_resident_ok(const MarkovParams& p);
cudaError_t markov_chain_resident(const MarkovParams& p, int num_sms, cudaStream_t st);
// One or two sequences (bf16, r = 64, 128 or 256): the resident slice with FMA dot
// products; p.keys holds 2 sets of p.keys_stride >= 16 * B * (num_sms + 1) exchange
// words and arrival counters (zero before the first launch), selected by the parity
// of p.epoch, which the launch advances.  They must not be shared with the other chains.
// Sampling form of the chain (temperature > 0): per block position k, CTAs over the
// vocabulary compute the logits and publish candidate words, then one CTA per sequence
// draws the token (Gumbel-max over the top_k candidates, SplitMix64 uniforms keyed by
// slot, draw counter + k and vocabulary entry) and its confidence; the last position
// advances draws[slot] by gamma.
struct SampleParams {
    const float* U = nullptr;          // [B*gamma, V] base logits
    const void* w1 = nullptr;          // [V, r], w_dtype
    const void* w2 = nullptr;
    int w_dtype = DT_BF16;
    const float* y = nullptr;          // [B*gamma, d] out-normed block rows
    const float* conf_w = nullptr;     // [d + r + 1]
    int B = 0, gamma = 0, V = 0, r = 0, d = 0, k = 0;
    const int* anchors = nullptr;      // [B] device, or nullptr: `anchor`
    int anchor = 0;
    const int* seq_ids = nullptr;      // [B] slots, or nullptr: slot b
    int n_slots = 0;                   // slots with a draw counter
    int* tokens = nullptr;             // [B, gamma]
    float* conf = nullptr;
    float* logits = nullptr;           // [B, gamma, V] or nullptr
    float temperature = 0.f;
    int top_k = 0;                     // 0: the whole vocabulary; else 1..64
    unsigned long long seed = 0;
    unsigned int* draws = nullptr;     // [n_slots] draw counters
    unsigned long long* cand = nullptr;  // [B, ctas, cand_stride] candidate words
    int cand_stride = 0;
    int* err = nullptr;
};
int sample_ctas(int V, int num_sms);
bool sample_ok(int V, int r, int top_k, int num_sms);
cudaError_t sample_init();
cudaError_t markov_sample_step(const SampleParams& p, int num_sms, cudaStream_t st);

// Self-tests of the bounded device waits (each on words that nothing completes; every one gives
// up after about a second and ORs DEVERR_TIMEOUT into *err): which = 0 the FMA chain's arrival
// count, 1 the resident chain's barrier, 2 the cooperative chain's barrier (scratch: 64 zeroed
// bytes); the persistent layers' grid barrier; the tensor-core kernels' mbarrier wait.
cudaError_t markov_wait_selftest(int which, void* scratch, int* err, cudaStream_t st);
cudaError_t persistent_wait_selftest(void* scratch, int* err, cudaStream_t st);
cudaError_t mbar_wait_selftest(int* err, cudaStream_t st);
cudaError_t step_wait_selftest(void* scratch, int* err, cudaStream_t st);

bool markov_chain_fma_ok(const MarkovParams& p, int num_sms);
cudaError_t markov_chain_fma(const MarkovParams& p, int num_sms, cudaStream_t st);

// ------------------------------------------------------------------ bookkeeping kernels
// For a batched ingest: per feature row t, its slot and cache position
// (len[slot] + t - cu[i]); -1 and an error bit if over capacity or bad id.
cudaError_t ingest_rowmap(const int* seq_ids, const int* cu, int n_seqs, int total, const int* seq_len,
                          int max_seqs, int max_ctx, int* row_seq, int* row_pos, int* err, cudaStream_t st);
// len[slot] += cu[i+1] - cu[i] for sequences whose rows were all accepted.
cudaError_t ingest_commit(const int* seq_ids, const int* cu, int n_seqs, int* seq_len, int max_seqs, int max_ctx,
                          cudaStream_t st);
cudaError_t add_len(int* seq_len, int slot, int delta, cudaStream_t st);
cudaError_t set_len(int* seq_len, int slot, int value, cudaStream_t st);
// Validate batched draft inputs: ids in [0, max_seqs), anchors in [0, V).
// Bad entries set err bits; safe_ids gets -1 for a bad id (the sequence is then
// skipped by every kernel) and safe_anchors the anchor clamped into [0, V).
cudaError_t check_draft_inputs(const int* seq_ids, const int* anchors, int n, int max_seqs, int V, int* err,
                               int* safe_ids, int* safe_anchors, cudaStream_t st);

}  // namespace dspark
