// C ABI of the drafter library: handle, weight packing, caches, workspaces
// and the ingest / draft step orchestration (see include/dspark.h).
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <string>
#include <vector>

#include "../../include/dspark.h"
#include "kernels.cuh"
#include "tc_gemm.cuh"

using namespace dspark;

namespace {

thread_local std::string g_create_error = "no error";

// Forms of the batch-1 draft layers (dspark_set_path, DSPARK_PATH_LAYERS).
enum { LAYERS_AUTO = 0, LAYERS_PER_KERNEL = 1, LAYERS_PERSISTENT_MMA = 2, LAYERS_STEP_TC = 3 };

struct DevBuf {
    void* p = nullptr;
    size_t bytes = 0;
};

// Kernel classes of the step, timed by dspark_profile.
enum Cat {
    CAT_INGEST_PROJ, CAT_INGEST_NORM, CAT_INGEST_KV, CAT_BLOCK, CAT_NORM, CAT_QKV, CAT_ATTN, CAT_O, CAT_GATE_UP,
    CAT_DOWN, CAT_OUT_PROJ, CAT_MARKOV, CAT_LAYERS, CAT_STEP,
    CAT_QKV_SIDE,  // layer 0's QKV beside an ingest (its range spans the ingest it overlaps)
    CAT_COUNT
};
const char* const kCatNames[CAT_COUNT] = {"ingest_proj", "ingest_norm", "ingest_kv", "block_build", "rmsnorm",
                                          "qkv_proj", "attention", "o_proj", "gate_up_proj", "down_proj",
                                          "out_proj", "markov_argmax", "draft_layers", "draft_step",
                                          "qkv_proj_beside_ingest"};

struct ProfRange {
    int cat;
    cudaEvent_t a, b;
    long long launches;
    cudaGraphNode_t na = nullptr, nb = nullptr;  // event-record nodes when captured in a graph
};

// A captured draft step, replayed while its inputs and outputs stay the same.
struct DraftGraph {
    int B = 0;
    const int* seq_ids = nullptr;
    const int* anchors = nullptr;
    int* tokens = nullptr;
    float* conf = nullptr;
    float* logits = nullptr;
    uint32_t mask = 0;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    std::vector<ProfRange> ranges;
    long long kernels = 0;
    uint64_t last_use = 0;
};

}  // namespace

struct dspark_handle {
    dspark_config cfg{};
    int device = 0;
    int num_sms = 148;
    int dt = DT_BF16;
    size_t esz = 2;
    int d = 0, F = 0, hd = 0, mH = 0, R = 0;  // R: rows of the largest draft batch (max_seqs * gamma)

    std::vector<void*> allocs;
    // packed weights (library-owned)
    void* W_c = nullptr;
    float* ctx_norm = nullptr;
    const void* embed = nullptr;
    void* tok_proj = nullptr;
    float* block_const = nullptr;            // [gamma, d]
    std::vector<void*> wqkv, wo, wgu, wd;    // wqkv [3d, d]; wgu [2F, d] rows (gate f, up f) interleaved
    std::vector<float*> attn_norm, ff_norm;
    std::vector<float*> q_norm, k_norm;      // [head_dim] per layer (qk_norm)
    float** k_norm_dev = nullptr;            // device array of the k_norm pointers
    int nkv = 0, dkv = 0;                    // K/V heads and K/V width
    bool qk_rope = false;                    // per-head norm and/or rotation of Q and K
    double* rope_freq = nullptr;             // [head_dim / 2] rotation frequencies (rope_theta > 0)
    float** attn_norm_dev = nullptr;         // device array of the attn_norm pointers
    float* out_norm = nullptr;
    void* out_proj = nullptr;
    void* w1 = nullptr;
    void* w2 = nullptr;
    float* conf_wb = nullptr;                // [d + r + 1]
    TcWeight tc_wc, tc_out_proj;             // tensor-core views (bf16 only), rows >= 17
    std::vector<TcWeight> tc_kv, tc_qkv, tc_wo, tc_wgu, tc_wd;
    TcWeight tc_kv_a, tc_kv_w;               // every layer's ingest K/V product as one grouped GEMM (A: Nbuf)
    // the same product with each layer's attn_norm folded into its K/V weights: A is one copy of
    // RMSNorm(H_ctx) shared by every layer (tc_kv_a2, 2-D) and the weights are bf16([W_k; W_v] * g)
    void* wkv_s = nullptr;                   // [n_layers][2 d_kv][d] bf16
    TcWeight tc_kv_a2, tc_kv_ws;
    TcWeightStream ts_wc, ts_out_proj;       // weight-streaming tensor-core views, rows <= 16
    TcWeightStream ts_kv_all;                // wkv_s as one [n_layers * 2 d_kv, d] weight (short ingests)
    std::vector<TcWeightStream> ts_kv, ts_qkv, ts_wo, ts_wgu, ts_wd;
    // batched residual projections split over K: their partials wait here for the next row norm,
    // which adds kp_pending of them into x in order
    float* kp_part = nullptr;
    size_t kp_floats = 0;
    int kp_pending = 0;
    float* ts_part = nullptr;                // split-K partials of the streaming GEMM
    size_t ts_part_floats = 0;
    unsigned int* ts_tickets = nullptr;
    size_t ts_n_tickets = 0;
    // caches: [layer][seq][K|V][rows][d]
    void* cache = nullptr;
    int64_t rows = 0, seq_stride = 0, kv_off = 0, layer_stride = 0;
    int* d_len = nullptr;
    int* d_len_next = nullptr;  // sequence 0's length after an ingest in flight (the early layer-0 QKV)
    int* d_err = nullptr;
    std::vector<int> len_host;
    std::vector<char> len_known;
    // draft workspaces
    float *x = nullptr, *act = nullptr, *hbuf = nullptr, *q = nullptr, *y = nullptr, *U = nullptr;
    void* act_lp = nullptr;                  // bf16 copies of A operands for the tensor-core path
    void* h_lp = nullptr;
    void* xb = nullptr;                      // [16, d] bf16 operand x * g written by the residual epilogues
    float* ssp = nullptr;                    // [d / 8, 16] their 8-column sums of x^2
    bool chain_norm = true;                  // batch-1 layers: norms through the residual epilogues
    // sampling instead of argmax (temperature > 0)
    float samp_t = 0.f;
    int samp_k = 0;
    unsigned long long samp_seed = 0;
    unsigned int* samp_draws = nullptr;      // [max_seqs] draw counters
    unsigned long long* samp_cand = nullptr; // [max_seqs, sample_ctas, 64] candidate words
    float* attn_part = nullptr;
    size_t attn_part_floats = 0;
    unsigned int* attn_tickets = nullptr;    // [max_seqs * n_heads]
    float* mk_v = nullptr;
    int* mk_i = nullptr;
    unsigned int* mk_cnt = nullptr;
    int mk_ctas = 1;
    int mk_chain_max = 0;                    // largest co-resident grid of the one-launch Markov chain
    TcWeight tc_mk_E;                        // mk_E as the N operand of the many-sequence Markov GEMM
    TcWeight tc_tok_proj;                    // tok_proj [d, H] for the many-sequence block build
    void* emb_rows = nullptr;                // [max_seqs, H] gathered anchor embeddings (bf16)
    void* mk_E = nullptr;                    // [max_seqs, r] gathered w1 rows (bf16)
    float* mk_pv = nullptr;                  // [max_seqs, ceil(V/32)] chunk partials
    int* mk_pi = nullptr;
    unsigned int* mk_bar = nullptr;          // [2] grid-barrier words, the chain's launch epoch, the FMA chain's
    unsigned long long* mk_slots = nullptr;  // [2, 16 * 2 * (num_sms + 1)] exchange words and counters, FMA chain
    bool mk_fma = true;                      // one or two sequences: the FMA chain
    unsigned long long* mk_keys = nullptr;   // [2, max_seqs, 16] argmax words of the Markov chain, then 2 counters
    unsigned long long* pk_bar = nullptr;    // persistent draft layers: 2 barrier counters, then the launch epoch
    TcWeightStream ts_tok_proj;              // tok_proj [d, H] as a 128-row weight stream
    void* ds_maps = nullptr;                 // one-launch tcgen05 step: [2 + 4 n_layers] weight tensor maps
    float* ds_qkv = nullptr;                 // [gamma, 3d] QKV products
    float* ds_gu = nullptr;                  // [gamma, 2F] gate/up products
    unsigned int* ds_hcnt = nullptr;         // [2, n_heads] arrivals of a head's key ranges
    float* ds_apart = nullptr;               // attention partials
    size_t ds_apart_floats = 0;
    unsigned long long* ds_bar = nullptr;    // 2 barrier counters, then the launch epoch
    unsigned long long* ds_mk = nullptr;     // [2][17][num_sms] Markov exchange words and counters
    void* pk_maps = nullptr;                 // [n_layers][4] weight-slice tensor maps of the persistent layers
    int pk_map3d = 0;
    int layers_path = 0;                     // DSPARK_PATH_LAYERS: 0 auto, else the forced form
    float* ws = nullptr;
    size_t ws_floats = 0;
    // a second set of split-K scratch (SIMT and weight-streaming) for launches on the side stream
    // beside an ingest (SideScratch)
    float* ws_side = nullptr;
    size_t ws_side_floats = 0;
    float* ts_part_side = nullptr;
    size_t ts_part_side_floats = 0;
    unsigned int* ts_tickets_side = nullptr;
    size_t ts_n_tickets_side = 0;
    int* safe_ids = nullptr;                 // [max_seqs] validated batched sequence slots (-1: rejected)
    int* safe_anchors = nullptr;             // [max_seqs] batched anchors clamped into [0, V)
    // ingest workspaces
    int ingest_rows = 0;
    int P_rows = 0;                          // rows of P: room for the K ranges of a split projection
    float* P = nullptr;
    void* Nbuf = nullptr;
    DevBuf rowmap;                           // row_seq, row_pos (grow-only)
    DevBuf stage_in, stage_out;              // host-call staging (grow-only)
    cudaEvent_t in_copied = nullptr;         // the host features are in stage_in

    std::string err = "no error";
    long long launches_at_create = 0;
    // CUDA graphs of the draft step
    bool use_graphs = true;
    cudaStream_t cap_stream = nullptr;
    // side branch of the step: work that no launch on the main stream waits for right away
    // (forked from and joined back into the main stream with the two events)
    cudaStream_t side_stream = nullptr;
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
    cudaEvent_t ev_block = nullptr;          // the block build of dspark_ingest_and_draft, on the side stream
    std::vector<DraftGraph> graphs;
    uint64_t graph_clock = 0;
    std::vector<ProfRange>* cap_ranges = nullptr;  // set while capturing
    int* anchor_dev = nullptr;                     // [1] anchor of the non-batched draft
    // profiling
    bool prof_on = false;
    uint32_t prof_mask = 0;
    std::vector<ProfRange> prof_ranges;
    std::vector<cudaEvent_t> prof_pool;
    size_t prof_next = 0;
};

namespace {

dspark_status fail(dspark_handle* h, dspark_status st, const std::string& msg) {
    if (h) h->err = msg;
    else g_create_error = msg;
    return st;
}

#define CUDA_TRY(h, expr)                                                                     \
    do {                                                                                      \
        cudaError_t _e = (expr);                                                              \
        if (_e != cudaSuccess)                                                                \
            return fail((h), _e == cudaErrorMemoryAllocation ? DSPARK_ERR_OOM : DSPARK_ERR_CUDA, \
                        std::string(#expr) + ": " + cudaGetErrorString(_e));                  \
    } while (0)

cudaError_t dalloc(dspark_handle* h, void** p, size_t bytes) {
    if (bytes == 0) bytes = 16;
    cudaError_t e = cudaMalloc(p, bytes);
    if (e == cudaSuccess) h->allocs.push_back(*p);
    return e;
}

cudaError_t grow(DevBuf& b, size_t bytes) {
    if (b.bytes >= bytes) return cudaSuccess;
    if (b.p) cudaFree(b.p);
    b.p = nullptr;
    b.bytes = 0;
    size_t want = std::max<size_t>(bytes, 1 << 20);
    cudaError_t e = cudaMalloc(&b.p, want);
    if (e == cudaSuccess) b.bytes = want;
    return e;
}

int attn_chunks(const dspark_handle* h, int B, int max_keys) {
    // Few (sequence, head) pairs: at most one CTA per SM (the tensor-core kernel
    // then runs a deeper cp.async ring), so that each range is long and the last
    // CTA merges few partials.  Many pairs: about a dozen CTAs per SM over the
    // launch, so that sequences of unequal length balance.  At least 64 keys
    // (one tile) per range either way.
    const int nh = h->cfg.n_heads;
    const int pairs = nh * B;
    int want = pairs <= h->num_sms ? h->num_sms / pairs : (12 * h->num_sms + pairs - 1) / pairs;
    int by_keys = (max_keys + 63) / 64;
    int n = std::max(1, std::min(std::min(want, by_keys), attn_max_chunks(h->dt, h->hd, h->cfg.gamma)));
    // short enough ranges merge inside a thread-block cluster, which holds at most so many of them
    if (h->dt == DT_BF16 && attention_tc_ok(h->dt, h->hd, h->cfg.gamma)) {
        const int cl = attention_tc_cluster_chunks(max_keys);
        if (cl >= 2 && n > cl) n = cl;
    }
    return n;
}

// A weight and its tensor-core views.
struct WView {
    const void* W;
    const TcWeight* tc;
    const TcWeightStream* ts;
};
template <typename V>
const V* at_or_null(const std::vector<V>& v, int i) {
    return v.empty() ? nullptr : &v[i];
}

// acc = A . W^T with the best kernel for the shape:
//   rows <= 16, bf16: weight-streaming tcgen05 (swap-AB) kernel;
//   rows <= 16 otherwise (fp32 drafter, gathered rows): SIMT weight streaming;
//   rows >= 17, bf16: persistent tcgen05 GEMM;  anything else: SIMT tiles.
cudaError_t gemm(dspark_handle* h, int a_dtype, const void* A, int64_t lda, const int* a_rows, int a_row0,
                 const WView& wv, int M, int N, int K, const EpiParams& ep, cudaStream_t st) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    const void* W = wv.W;
    const TcWeight* tcw = wv.tc;
    if (M <= 16 && wv.ts && wv.ts->ready && a_dtype == DT_BF16 && a_rows == nullptr && tc_stream_ok(M, N, K))
        return tc_stream((const char*)A + (size_t)a_row0 * lda * 2, lda, *wv.ts, M, N, K, ep, h->ts_part,
                         h->ts_part_floats, h->ts_tickets, h->ts_n_tickets, h->num_sms, h->d_err, st);
    // only the weight-streaming epilogues (tensor-core, and the SIMT one of a single row) hand over the
    // next operand
    if (ep.ssp && !(M <= 16 && skinny_ok(M, K))) return cudaErrorInvalidValue;
    if (M <= 16 && skinny_ok(M, K))
        return gemm_skinny(a_dtype, A, lda, a_rows, a_row0, h->dt, W, M, N, K, ep, h->ws, h->ws_floats, h->num_sms, st);
    if (tcw && tcw->ready && a_dtype == DT_BF16 && a_rows == nullptr && tc_wide_preferred(M, N, h->num_sms) &&
        tc_wide_ok(*tcw, M, N, K, ep))
        return tc_gemm_wide((const char*)A + (size_t)a_row0 * lda * 2, lda, *tcw, M, N, K, ep, h->num_sms, h->d_err,
                            st);
    if (tcw && tcw->ready && a_dtype == DT_BF16 && a_rows == nullptr && tc_gemm_ok(M, N, K))
        return tc_gemm((const char*)A + (size_t)a_row0 * lda * 2, lda, *tcw, M, N, K, ep, h->num_sms, h->d_err, st);
    const char* a = (const char*)A;
    if (!a_rows) a += (size_t)a_row0 * lda * (a_dtype == DT_BF16 ? 2 : 4);
    return gemm_simt(a_dtype, a, lda, a_rows, h->dt, W, M, N, K, ep, st);
}

// RMSNorm(x) * w for the R block rows, then (that) . W^T.  Where the weight-streaming
// tensor-core kernel runs the product, the normalisation is folded into it (the
// operand is x * w, the row scale multiplies the accumulator); otherwise a
// normalisation kernel writes the operand to actA first.
cudaError_t norm_gemm(dspark_handle* h, const float* w, int R, const WView& wv, int N, int K, const EpiParams& ep,
                      void* actA, int adt, cudaStream_t st, int norm_cat);


// Next event of the handle's reusable timing-event pool (nullptr if none can be made).
cudaEvent_t pool_event(dspark_handle* h) {
    if (h->prof_next >= h->prof_pool.size()) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        h->prof_pool.push_back(e);
    }
    return h->prof_pool[h->prof_next++];
}

// Records an event pair around one class of launches when profiling is on.
struct Prof {
    dspark_handle* h;
    cudaStream_t st;
    int idx = -1;
    long long l0 = 0;
    cudaEvent_t ev() { return pool_event(h); }
    std::vector<ProfRange>& list() { return h->cap_ranges ? *h->cap_ranges : h->prof_ranges; }
    void record(cudaEvent_t e) {
        if (h->cap_ranges) cudaEventRecordWithFlags(e, st, cudaEventRecordExternal);
        else cudaEventRecord(e, st);
    }
    Prof(dspark_handle* h_, int cat, cudaStream_t st_) : h(h_), st(st_) {
        if (!h->prof_on || !(h->prof_mask & (1u << cat))) return;
        cudaEvent_t a, b;
        if (h->cap_ranges) {  // placeholders: every replay gets fresh events
            if (cudaEventCreate(&a) != cudaSuccess) return;
            if (cudaEventCreate(&b) != cudaSuccess) return;
        } else {
            a = ev();
            b = ev();
            if (!a || !b) return;
        }
        record(a);
        list().push_back({cat, a, b, 0});
        idx = (int)list().size() - 1;
        l0 = launch_count();
    }
    void end() {
        if (idx < 0) return;
        record(list()[idx].b);
        list()[idx].launches = launch_count() - l0;
        idx = -1;
    }
    ~Prof() { end(); }
};

cudaError_t norm_gemm(dspark_handle* h, const float* w, int R, const WView& wv, int N, int K, const EpiParams& ep,
                      void* actA, int adt, cudaStream_t st, int norm_cat) {
    const int d = h->d;
    {
        Prof pr(h, CAT_NORM, st);
        cudaError_t e = rmsnorm_rows(h->x, d, w, R, d, h->cfg.eps, adt, actA, d, st,
                                     h->kp_pending ? h->kp_part : nullptr, h->kp_pending, (int64_t)R * d);
        h->kp_pending = 0;
        if (e != cudaSuccess) return e;
    }
    Prof pr(h, norm_cat, st);
    return gemm(h, adt, actA, d, nullptr, 0, wv, R, N, K, ep, st);
}

// A projection whose RMSNorm comes through the previous residual epilogue: X = h->xb holds
// bf16(x * g) and h->ssp the 8-column sums of x^2, from which the kernel forms the row scales.
cudaError_t chained_gemm(dspark_handle* h, int R, const WView& wv, int N, int K, const EpiParams& ep, cudaStream_t st,
                         int cat) {
    Prof pr(h, cat, st);
    StreamNorm sn;
    sn.ssp = h->ssp;
    sn.eps = h->cfg.eps;
    return tc_stream(h->xb, K, *wv.ts, R, N, K, ep, h->ts_part, h->ts_part_floats, h->ts_tickets, h->ts_n_tickets,
                     h->num_sms, h->d_err, st, &sn);
}

// x += A . W^T for many block rows.  When the output tiles would leave most SMs idle, K is cut into
// ranges whose partial products wait in kp_part; the next row norm adds them into x in order.
cudaError_t residual_gemm(dspark_handle* h, int a_dtype, const void* A, int64_t lda, const WView& wv, int R, int N, int K,
                          const EpiParams& res, cudaStream_t st) {
    if (R >= 17 && a_dtype == DT_BF16 && wv.tc && wv.tc->ready && tc_gemm_ok(R, N, K) && !res.ssp && h->kp_part &&
        h->kp_pending == 0 && res.kind == EPI_ADD_F32 && res.out_f32 == h->x && res.ldo == N && N == h->d) {
        const int tiles = ((R + 127) / 128) * ((N + 255) / 256);
        const int nkb = (K + 63) / 64;
        int ks = std::min({h->num_sms / tiles, nkb, 12});
        while (ks > 1 && (size_t)ks * R * N > h->kp_floats) --ks;
        if (ks >= 2) {
            EpiParams ep;
            ep.kind = EPI_STORE_F32;
            ep.out_f32 = h->kp_part;
            ep.ldo = N;
            ep.split_rows = R;
            cudaError_t e = tc_gemm(A, lda, *wv.tc, R, N, K, ep, h->num_sms, h->d_err, st, ks);
            if (e == cudaSuccess) h->kp_pending = ks;
            return e;
        }
    }
    return gemm(h, a_dtype, A, lda, nullptr, 0, wv, R, N, K, res, st);
}

// Every batch-1 projection streams (so the residual epilogues can hand over the next norm's operand).
bool norm_chain_ok(const dspark_handle* h, int R, bool lowp) {
    if (!h->chain_norm || !lowp || R > 16 || !h->ts_out_proj.ready || !tc_stream_ok(R, h->cfg.vocab, h->d) ||
        h->d % 64 != 0)
        return false;
    const int d = h->d, F = h->F;
    for (int i = 0; i < h->cfg.n_layers; ++i) {
        const TcWeightStream* v[4] = {at_or_null(h->ts_qkv, i), at_or_null(h->ts_wo, i), at_or_null(h->ts_wgu, i),
                                      at_or_null(h->ts_wd, i)};
        for (const TcWeightStream* w : v)
            if (!w || !w->ready) return false;
    }
    return tc_stream_ok(R, d + 2 * h->dkv, d) && tc_stream_ok(R, d, d) && tc_stream_ok(R, 2 * F, d) &&
           tc_stream_ok(R, d, F);
}

// Per-head norm / rotation arguments shared by the block and ingest forms (layer `layer`).
QkRope qk_rope_args(const dspark_handle* h, int layer) {
    QkRope a;
    a.cache = (char*)h->cache + (size_t)layer * h->layer_stride * h->esz;
    a.cache_dtype = h->dt;
    a.layer_stride = h->layer_stride;
    a.seq_stride = h->seq_stride;
    a.d_kv = h->dkv;
    a.max_rows = (int)h->rows;
    a.seq_len = h->d_len;
    a.k_norm = h->cfg.qk_norm ? h->k_norm[layer] : nullptr;
    a.n_heads = h->cfg.n_heads;
    a.n_kv_heads = h->nkv;
    a.head_dim = h->hd;
    a.eps = h->cfg.eps;
    a.theta = h->cfg.rope_theta;
    a.freq = h->rope_freq;
    return a;
}

// The context rows just projected: per-head K norm / rotation in every layer's cache, at the
// rows' positions (slot 0 at len + m, or the batched row_seq / row_pos), before the length moves.
cudaError_t ingest_qk(dspark_handle* h, int n, const int* row_seq, const int* row_pos, cudaStream_t st) {
    if (!h->qk_rope || n <= 0) return cudaSuccess;
    QkRope a = qk_rope_args(h, 0);
    a.k_norm_layers = h->cfg.qk_norm ? h->k_norm_dev : nullptr;
    a.n_layers = h->cfg.n_layers;
    a.rows = n;
    a.row_seq = row_seq;
    a.row_pos = row_pos;
    return qk_rope_ingest(a, st);
}

EpiParams cache_epi(const dspark_handle* h, int layer) {
    EpiParams ep;
    ep.cache = (char*)h->cache + (size_t)layer * h->layer_stride * h->esz;
    ep.cache_dtype = h->dt;
    ep.seq_stride = h->seq_stride;
    ep.kv_off = h->kv_off;
    ep.d = h->d;
    ep.d_kv = h->dkv;
    ep.max_rows = (int)h->rows;
    ep.seq_len = h->d_len;
    return ep;
}

dspark_status check_cfg(const dspark_config* c, std::string& why) {
    if (!c) { why = "config is NULL"; return DSPARK_ERR_INVALID_ARG; }
    if (c->hidden <= 0 || c->n_taps <= 0 || c->d_draft <= 0 || c->n_heads <= 0 || c->n_layers <= 0 ||
        c->ff_mult <= 0 || c->gamma <= 0 || c->vocab <= 0 || c->markov_rank <= 0 || c->max_ctx < 0 ||
        c->max_seqs <= 0 || !(c->eps >= 0.f)) {
        why = "config has a non-positive dimension";
        return DSPARK_ERR_INVALID_ARG;
    }
    if (c->d_draft % c->n_heads != 0) {
        why = "d_draft " + std::to_string(c->d_draft) + " not divisible by n_heads " + std::to_string(c->n_heads);
        return DSPARK_ERR_INVALID_ARG;
    }
    if (c->dtype != DSPARK_BF16 && c->dtype != DSPARK_FP32) { why = "unknown dtype"; return DSPARK_ERR_INVALID_ARG; }
    if (c->act != DSPARK_ACT_SILU && c->act != DSPARK_ACT_GELU_TANH) { why = "unknown act"; return DSPARK_ERR_INVALID_ARG; }
    const int hd = c->d_draft / c->n_heads;
    if (c->gamma > 16) { why = "gamma > 16"; return DSPARK_ERR_UNSUPPORTED; }
    if (hd > 256 || hd % 8 != 0) { why = "head_dim must be a multiple of 8 and <= 256"; return DSPARK_ERR_UNSUPPORTED; }
    if (256 % (hd / 8) != 0 || c->gamma > 256 / (hd / 8)) { why = "gamma * head_dim must be <= 2048 with head_dim / 8 dividing 256"; return DSPARK_ERR_UNSUPPORTED; }
    if (c->dtype == DSPARK_FP32 && hd > 128) { why = "fp32 drafters take head_dim <= 128"; return DSPARK_ERR_UNSUPPORTED; }
    if (c->d_draft % 64 != 0 || c->d_draft > 4096) { why = "d_draft must be a multiple of 64, <= 4096"; return DSPARK_ERR_UNSUPPORTED; }
    if (c->markov_rank % 8 != 0 || c->markov_rank > 1024) { why = "markov_rank must be a multiple of 8, <= 1024"; return DSPARK_ERR_UNSUPPORTED; }
    if (c->hidden % 8 != 0) { why = "hidden must be a multiple of 8"; return DSPARK_ERR_UNSUPPORTED; }
    if ((int64_t)c->max_ctx + c->gamma > (1 << 30)) { why = "max_ctx too large"; return DSPARK_ERR_UNSUPPORTED; }
    if (c->n_kv_heads < 0 || c->n_heads % (c->n_kv_heads ? c->n_kv_heads : c->n_heads) != 0) {
        why = "n_heads must be a multiple of n_kv_heads";
        return DSPARK_ERR_INVALID_ARG;
    }
    if (c->qk_norm != 0 && c->qk_norm != 1) { why = "qk_norm must be 0 or 1"; return DSPARK_ERR_INVALID_ARG; }
    if (!(c->rope_theta >= 0.f) || !std::isfinite(c->rope_theta)) { why = "rope_theta must be finite and >= 0"; return DSPARK_ERR_INVALID_ARG; }
    return DSPARK_OK;
}

dspark_status sync_len(dspark_handle* h, int slot) {
    if (h->len_known[slot]) return DSPARK_OK;
    int v = 0;
    CUDA_TRY(h, cudaDeviceSynchronize());
    CUDA_TRY(h, cudaMemcpy(&v, h->d_len + slot, sizeof(int), cudaMemcpyDeviceToHost));
    h->len_host[slot] = v;
    h->len_known[slot] = 1;
    return DSPARK_OK;
}

// Eq 2 + Eq 3 for `T` feature rows; rows map to (slot, position) through
// row_seq/row_pos (batched) or slot 0 at len[0] + t (row_seq == nullptr).
dspark_status ingest_rows(dspark_handle* h, const void* feats, int T, const int* row_seq, const int* row_pos,
                          cudaStream_t st) {
    const int d = h->d, nL = h->cfg.n_layers;
    for (int t0 = 0; t0 < T; t0 += h->ingest_rows) {
        const int n = std::min(h->ingest_rows, T - t0);
        const void* X = (const char*)feats + (size_t)t0 * h->mH * h->esz;
        EpiParams ep;
        ep.kind = EPI_STORE_F32;
        ep.out_f32 = h->P;
        ep.ldo = d;
        // Too few output tiles for the SMs: cut K into ranges (separate work units
        // whose partial products the normalisation sums).
        int ks = 1;
        if (n > 16 && h->tc_wc.ready && tc_gemm_ok(n, d, h->mH)) {
            const int tiles = ((n + 127) / 128) * ((d + 255) / 256);
            ks = std::max(1, std::min({h->num_sms / tiles, 4, h->P_rows / n, h->mH / (64 * 8)}));
        }
        {
            Prof pr(h, CAT_INGEST_PROJ, st);
            if (ks > 1) {
                ep.split_rows = n;
                CUDA_TRY(h, tc_gemm(X, h->mH, h->tc_wc, n, d, h->mH, ep, h->num_sms, h->d_err, st, ks));
            } else {
                CUDA_TRY(h, gemm(h, h->dt, X, h->mH, nullptr, 0, WView{h->W_c, &h->tc_wc, &h->ts_wc}, n, d, h->mH, ep,
                                 st));
            }
        }
        const int lp = h->dt;  // normalised rows in the storage type (bf16 feeds the tensor cores)
        const bool grouped = n > 16 && h->tc_kv_a.ready && h->tc_kv_w.ready && tc_gemm_ok(n, 2 * h->dkv, d);
        // a short ingest streams every layer's scaled K/V weights in one launch
        const bool stream_all = !grouped && n <= 16 && lp == DT_BF16 && h->ts_kv_all.ready &&
                                tc_stream_ok(n, nL * 2 * h->dkv, d);
        // the attn_norm rides on the scaled K/V weights: one normalised copy serves every layer
        const bool shared = (grouped && h->tc_kv_ws.ready && h->tc_kv_a2.ready128) || stream_all;
        {
            Prof pr(h, CAT_INGEST_NORM, st);
            CUDA_TRY(h, ingest_norm(h->P, ks, (int64_t)n * d, n, d, h->cfg.eps, h->ctx_norm,
                                    shared ? nullptr : h->attn_norm_dev, shared ? 1 : nL, lp, h->Nbuf,
                                    (int64_t)h->ingest_rows * d, st));
        }
        Prof pr_kv(h, CAT_INGEST_KV, st);
        if (grouped) {
            // all layers in one launch: [nL x row tiles x column tiles] work units
            EpiParams kv = cache_epi(h, 0);
            kv.kind = EPI_KV_CACHE;
            kv.group_stride = h->layer_stride;
            if (row_seq) {
                kv.row_seq = row_seq + t0;
                kv.row_pos = row_pos + t0;
            }
            if (shared)
                CUDA_TRY(h, tc_gemm_grouped(h->tc_kv_a2, h->tc_kv_ws, nL, n, 2 * h->dkv, d, kv, h->num_sms, h->d_err, st,
                                            true));
            else
                CUDA_TRY(h, tc_gemm_grouped(h->tc_kv_a, h->tc_kv_w, nL, n, 2 * h->dkv, d, kv, h->num_sms, h->d_err, st));
            CUDA_TRY(h, ingest_qk(h, n, row_seq ? row_seq + t0 : nullptr, row_seq ? row_pos + t0 : nullptr, st));
            if (!row_seq) CUDA_TRY(h, add_len(h->d_len, 0, n, st));
            continue;
        }
        if (stream_all) {
            // one product [n, nL * 2 d_kv]: column block l is layer l's K/V rows
            EpiParams kv = cache_epi(h, 0);
            kv.kind = EPI_KV_CACHE;
            kv.group_stride = h->layer_stride;
            kv.group_cols = 2 * h->dkv;
            if (row_seq) {
                kv.row_seq = row_seq + t0;
                kv.row_pos = row_pos + t0;
            }
            CUDA_TRY(h, tc_stream(h->Nbuf, d, h->ts_kv_all, n, nL * 2 * h->dkv, d, kv, h->ts_part, h->ts_part_floats,
                                  h->ts_tickets, h->ts_n_tickets, h->num_sms, h->d_err, st));
            CUDA_TRY(h, ingest_qk(h, n, row_seq ? row_seq + t0 : nullptr, row_seq ? row_pos + t0 : nullptr, st));
            if (!row_seq) CUDA_TRY(h, add_len(h->d_len, 0, n, st));
            continue;
        }
        for (int i = 0; i < nL; ++i) {
            EpiParams kv = cache_epi(h, i);
            kv.kind = EPI_KV_CACHE;
            if (row_seq) {
                kv.row_seq = row_seq + t0;
                kv.row_pos = row_pos + t0;
            }
            // otherwise slot 0 at len[0] + m: the device length advances after every chunk
            const void* Ni = (const char*)h->Nbuf + (size_t)i * h->ingest_rows * d * h->esz;
            const void* Wkv = (const char*)h->wqkv[i] + (size_t)d * d * h->esz;  // rows [d, d + 2 d_kv) = [W_k; W_v]
            CUDA_TRY(h, gemm(h, lp, Ni, d, nullptr, 0, WView{Wkv, at_or_null(h->tc_kv, i), at_or_null(h->ts_kv, i)}, n,
                             2 * h->dkv, d, kv, st));
        }
        CUDA_TRY(h, ingest_qk(h, n, row_seq ? row_seq + t0 : nullptr, row_seq ? row_pos + t0 : nullptr, st));
        if (!row_seq) CUDA_TRY(h, add_len(h->d_len, 0, n, st));
    }
    return DSPARK_OK;
}

// The draft step for B sequences (slots seq_ids[b], or slot b when NULL).
// The one-launch tcgen05 step (block build, every layer, out_norm, out_proj) for a batch-1 draft
// of a bf16 multi-head drafter without the per-head Q/K transforms; false if it does not apply.
bool draft_step_args(dspark_handle* h, int B, const int* seq_ids, const int* anchors_dev, int anchor, int max_keys,
                     int* tokens, float* conf, float* logits, DraftStepArgs& a) {
    const dspark_config& c = h->cfg;
    if (B != 1 || seq_ids || h->dt != DT_BF16 || !h->ds_maps || h->qk_rope || h->nkv != c.n_heads) return false;
    a = DraftStepArgs{};
    a.x = h->x;
    a.qkv = h->ds_qkv;
    a.gu = h->ds_gu;
    a.y = h->y;
    a.U = h->U;
    a.act = h->act_lp;
    a.apart = h->ds_apart;
    a.hcnt = h->ds_hcnt;
    a.cache = h->cache;
    a.layer_stride = h->layer_stride;
    a.kv_off = h->kv_off;
    a.max_rows = (int)h->rows;
    a.seq_len = h->d_len;
    a.embed = h->embed;
    a.anchor_dev = anchors_dev;
    a.anchor = anchor;
    a.block_const = h->block_const;
    a.attn_norm = h->attn_norm.data();
    a.ff_norm = h->ff_norm.data();
    a.out_norm = h->out_norm;
    a.maps = h->ds_maps;
    a.d = h->d;
    a.F = h->F;
    a.H = c.hidden;
    a.V = c.vocab;
    a.nh = c.n_heads;
    a.nL = c.n_layers;
    a.gamma = c.gamma;
    a.act_kind = c.act;
    // one attention item (head, key range) per CTA, at least one 64-key tile per range
    a.nchunks = std::max(1, std::min(h->num_sms / c.n_heads, (max_keys + 63) / 64));
    a.eps = c.eps;
    a.bar = h->ds_bar;
    a.epoch = reinterpret_cast<unsigned int*>(h->ds_bar + 2);
    a.err = h->d_err;
    // the Markov chain in the same launch, unless the tokens are sampled
    const int r = c.markov_rank;
    if (h->samp_t <= 0.f && h->ds_mk && (r == 64 || r == 128 || r == 256 || r == 512)) {
        a.chain = 1;
        a.r = c.markov_rank;
        a.w1 = h->w1;
        a.w2 = h->w2;
        a.conf_w = h->conf_wb;
        a.tokens = tokens;
        a.conf = conf;
        a.logits = logits;
        a.mk = h->ds_mk;
    }
    return draft_step_tc_ok(a, h->num_sms) && (size_t)c.n_heads * a.nchunks * c.gamma * (h->hd + 4) <= h->ds_apart_floats;
}

// The block rows ("module-dflash.ts" #buildBlock: x_0 = E[anchor] tok_proj^T + block_pos[0], x_j =
// mask_emb[j-1] + block_pos[j]) and, for one sequence, layer 0's chained operand; *chain0 says whether
// that operand was written.  Reads no context: it may run beside an ingest.
dspark_status block_build(dspark_handle* h, int B, const int* seq_ids, const int* anchors_dev, int anchor,
                          cudaStream_t st, bool* chain0_out) {
    const dspark_config& c = h->cfg;
    const int d = h->d, R = B * c.gamma;
    const bool lowp0 = h->dt == DT_BF16;
    // one sequence: the block build also writes layer 0's chained operand (bf16(x * attn_norm) and
    // the 8-column sums of x^2), so the first QKV projection needs no normalisation launch
    const bool chain0 = B == 1 && !seq_ids && norm_chain_ok(h, R, lowp0) && d % 8 == 0 && h->ws &&
                        h->ws_floats >= 2 * (size_t)d && !(h->tc_tok_proj.ready && B >= 8);
    CUDA_TRY(h, block_init(h->x, h->block_const, B, c.gamma, d, st, chain0 ? h->xb : nullptr,
                           chain0 ? h->attn_norm[0] : nullptr, chain0 ? h->ssp : nullptr));
    {
        EpiParams ep;
        ep.kind = EPI_ADD_F32;
        ep.out_f32 = h->x;
        ep.ldo = (int64_t)c.gamma * d;  // row b of the product lands on block row 0 of sequence b
        if (chain0) {
            ep.xb = h->xb;
            ep.ld_xb = d;
            ep.ssp = h->ssp;
            ep.xb_g = h->attn_norm[0];
        }
        if (B >= 8 && h->tc_tok_proj.ready && h->emb_rows && anchors_dev && tc_gemm_ok(B, d, c.hidden)) {
            // many sequences: gather the anchor embeddings, then one tensor-core GEMM
            CUDA_TRY(h, markov_gather(h->embed, c.hidden, c.vocab, anchors_dev, nullptr, c.gamma, 0, B, h->emb_rows, st));
            CUDA_TRY(h, tc_gemm(h->emb_rows, c.hidden, h->tc_tok_proj, B, d, c.hidden, ep, h->num_sms, h->d_err, st));
        } else {
            CUDA_TRY(h, gemm(h, h->dt, h->embed, c.hidden, anchors_dev, anchors_dev ? 0 : anchor,
                             WView{h->tok_proj, nullptr, nullptr}, B, d, c.hidden, ep, st));
        }
    }
    *chain0_out = chain0;
    return DSPARK_OK;
}

// The QKV epilogue of layer `layer`: Q rows to h->q, the block's K/V rows into the cache after the
// context (whose lengths are read from seq_len).
EpiParams qkv_epi(const dspark_handle* h, int layer, const int* seq_ids, const int* seq_len) {
    EpiParams qkv = cache_epi(h, layer);
    qkv.kind = EPI_QKV;
    qkv.out_f32 = h->q;
    qkv.ldo = h->d;
    qkv.gamma = h->cfg.gamma;
    qkv.seq_ids = seq_ids;
    qkv.seq_len = seq_len;
    return qkv;
}

// While alive, the handle's split-K scratch is the side stream's set: launches on the side stream
// beside an ingest never share scratch with the ingest's own GEMMs.
struct SideScratch {
    dspark_handle* h;
    explicit SideScratch(dspark_handle* hh) : h(hh) { swap(); }
    ~SideScratch() { swap(); }
    void swap() {
        std::swap(h->ws, h->ws_side);
        std::swap(h->ws_floats, h->ws_side_floats);
        std::swap(h->ts_part, h->ts_part_side);
        std::swap(h->ts_part_floats, h->ts_part_side_floats);
        std::swap(h->ts_tickets, h->ts_tickets_side);
        std::swap(h->ts_n_tickets, h->ts_n_tickets_side);
    }
};

// prebuilt: -1 build the block rows here, 0 / 1 already built (1: with the chained operand);
// qkv0_done: layer 0's QKV projection has been issued already (dspark_ingest_and_draft)
dspark_status draft_rows(dspark_handle* h, int B, const int* seq_ids, const int* anchors_dev, int anchor, int max_keys,
                         int* tokens, float* conf, float* logits, cudaStream_t st, int prebuilt = -1,
                         bool qkv0_done = false) {
    const dspark_config& c = h->cfg;
    const int d = h->d, F = h->F, R = B * c.gamma, V = c.vocab;
    h->kp_pending = 0;  // partials of an earlier, interrupted draft are never applied
    DraftStepArgs dsa;
    const bool one_launch = h->layers_path == LAYERS_STEP_TC &&
                            draft_step_args(h, B, seq_ids, anchors_dev, anchor, max_keys, tokens, conf, logits, dsa);
    if (one_launch) {
        Prof pr(h, CAT_STEP, st);
        CUDA_TRY(h, draft_step_tc(dsa, h->num_sms, st));
        if (dsa.chain) return DSPARK_OK;  // the chain, argmax and confidences ran in the same launch
    }
    if (!one_launch) {
        Prof pr_block(h, CAT_BLOCK, st);
        bool chain0 = prebuilt > 0;
        if (prebuilt < 0) {
            const dspark_status bs = block_build(h, B, seq_ids, anchors_dev, anchor, st, &chain0);
            if (bs != DSPARK_OK) return bs;
        }
        const bool lowp = (h->dt == DT_BF16);  // the tensor-core kernels take bf16 activations
        void* actA = lowp ? h->act_lp : (void*)h->act;
        const int adt = lowp ? DT_BF16 : DT_F32;
        bool layers_done = false;
        // Every layer in one persistent launch on the warp MMA, only when asked for: the per-kernel
        // tcgen05 path is faster on both drafter shapes (for the small Gemma-shaped layers too).
        // (the one-launch layers keep one K/V head per query head and no per-head transform)
        if (B == 1 && !seq_ids && lowp && h->layers_path == LAYERS_PERSISTENT_MMA && !h->qk_rope &&
            h->nkv == c.n_heads) {
            // every layer in one persistent launch
            DraftPersistArgs a{};
            a.x = h->x;
            a.q = h->q;
            a.act = h->act_lp;
            a.hact = h->h_lp;
            a.part = h->attn_part;
            a.cache = h->cache;
            a.layer_stride = h->layer_stride;
            a.kv_off = h->kv_off;
            a.max_rows = (int)h->rows;
            a.seq_len = h->d_len;
            a.wqkv = h->wqkv.data();
            a.wo = h->wo.data();
            a.wgu = h->wgu.data();
            a.wd = h->wd.data();
            a.attn_norm = h->attn_norm.data();
            a.ff_norm = h->ff_norm.data();
            a.d = d;
            a.F = F;
            a.nh = c.n_heads;
            a.nL = c.n_layers;
            a.gamma = c.gamma;
            a.act_kind = c.act;
            a.nchunks = std::max(1, std::min(h->num_sms / c.n_heads, (max_keys + 63) / 64));
            a.eps = c.eps;
            a.maps = h->pk_maps;
            a.map3d = h->pk_map3d;
            a.bar = h->pk_bar;
            a.epoch = reinterpret_cast<unsigned int*>(h->pk_bar + 2);
            a.err = h->d_err;
            if (draft_persistent_ok(a) &&
                attn_scratch_floats(1, c.n_heads, a.nchunks, c.gamma, h->hd) <= h->attn_part_floats) {
                pr_block.end();
                Prof pr(h, CAT_LAYERS, st);
                CUDA_TRY(h, draft_persistent(a, h->num_sms, st));
                layers_done = true;
            }
        }
        // Batch 1: the residual epilogues of W_o and W_down also write the next projection's operand
        // bf16(x * g) and the row sums of x^2, so no normalisation launch sits between the layers.
        const bool chain = !layers_done && norm_chain_ok(h, R, lowp);
        for (int i = 0; i < c.n_layers && !layers_done; ++i) {
            if (i == 0) pr_block.end();
            const EpiParams qkv = qkv_epi(h, i, seq_ids, h->d_len);
            const WView wqkv{h->wqkv[i], at_or_null(h->tc_qkv, i), at_or_null(h->ts_qkv, i)};
            if (i == 0 && qkv0_done && chain && chain0) {
                // issued beside the ingest
            } else if (chain && (i > 0 || chain0))
                CUDA_TRY(h, chained_gemm(h, R, wqkv, d + 2 * h->dkv, d, qkv, st, CAT_QKV));
            else
                CUDA_TRY(h, norm_gemm(h, h->attn_norm[i], R, wqkv, d + 2 * h->dkv, d, qkv, actA, adt, st, CAT_QKV));
            if (h->qk_rope) {
                Prof pq(h, CAT_QKV, st);
                QkRope qr = qk_rope_args(h, i);
                qr.q = h->q;
                qr.ldq = d;
                qr.q_norm = h->cfg.qk_norm ? h->q_norm[i] : nullptr;
                qr.B = B;
                qr.gamma = c.gamma;
                qr.seq_ids = seq_ids;
                CUDA_TRY(h, qk_rope_block(qr, st));
            }
            AttnParams ap;
            ap.q = h->q;
            ap.cache = (char*)h->cache + (size_t)i * h->layer_stride * h->esz;
            ap.cache_dtype = h->dt;
            ap.seq_stride = h->seq_stride;
            ap.kv_off = h->kv_off;
            ap.seq_len = h->d_len;
            ap.seq_ids = seq_ids;
            ap.B = B;
            ap.gamma = c.gamma;
            ap.d = d;
            ap.n_heads = c.n_heads;
            ap.d_kv = h->dkv;
            ap.n_kv_heads = h->nkv;
            ap.n_chunks = attn_chunks(h, B, max_keys);
            ap.max_keys = max_keys;
            ap.part = h->attn_part;
            ap.tickets = h->attn_tickets;
            ap.out = actA;
            ap.out_dtype = adt;
            if (attn_scratch_floats(B, c.n_heads, ap.n_chunks, c.gamma, h->hd) > h->attn_part_floats)
                return fail(h, DSPARK_ERR_CAPACITY, "attention scratch too small");
            {
                Prof pr(h, CAT_ATTN, st);
                CUDA_TRY(h, attention(ap, st));
            }
            EpiParams res;
            res.kind = EPI_ADD_F32;
            res.out_f32 = h->x;
            res.ldo = d;
            if (chain) {
                res.xb = h->xb;
                res.ld_xb = d;
                res.ssp = h->ssp;
                res.xb_g = h->ff_norm[i];
            }
            {
                Prof pr(h, CAT_O, st);
                CUDA_TRY(h, residual_gemm(h, adt, actA, d,
                                          WView{h->wo[i], at_or_null(h->tc_wo, i), at_or_null(h->ts_wo, i)}, R, d, d,
                                          res, st));
            }
            EpiParams sw;
            sw.kind = EPI_SWIGLU;
            sw.out_act = lowp ? h->h_lp : (void*)h->hbuf;
            sw.act_dtype = adt;
            sw.ld_act = F;
            sw.act = c.act;
            const WView wgu{h->wgu[i], at_or_null(h->tc_wgu, i), at_or_null(h->ts_wgu, i)};
            if (chain)
                CUDA_TRY(h, chained_gemm(h, R, wgu, 2 * F, d, sw, st, CAT_GATE_UP));
            else
                CUDA_TRY(h, norm_gemm(h, h->ff_norm[i], R, wgu, 2 * F, d, sw, actA, adt, st, CAT_GATE_UP));
            if (chain) res.xb_g = i + 1 < c.n_layers ? h->attn_norm[i + 1] : h->out_norm;
            {
                Prof pr(h, CAT_DOWN, st);
                CUDA_TRY(h, residual_gemm(h, adt, sw.out_act, F,
                                          WView{h->wd[i], at_or_null(h->tc_wd, i), at_or_null(h->ts_wd, i)}, R, d, F,
                                          res, st));
            }
        }
        if (chain) {
            // out_proj takes its norm through the chain; y (the confidence head's input) is needed
            // only by the Markov launch, so it is computed on a side branch beside out_proj
            CUDA_TRY(h, cudaEventRecord(h->ev_fork, st));
            CUDA_TRY(h, cudaStreamWaitEvent(h->side_stream, h->ev_fork, 0));
            {
                Prof pr(h, CAT_NORM, h->side_stream);
                CUDA_TRY(h, rmsnorm_rows(h->x, d, h->out_norm, R, d, c.eps, DT_F32, h->y, d, h->side_stream));
            }
            CUDA_TRY(h, cudaEventRecord(h->ev_join, h->side_stream));
        } else {
            Prof pr(h, CAT_NORM, st);
            CUDA_TRY(h, rmsnorm_rows(h->x, d, h->out_norm, R, d, c.eps, DT_F32, h->y, d, st,
                                     h->kp_pending ? h->kp_part : nullptr, h->kp_pending, (int64_t)R * d));
            h->kp_pending = 0;
        }
        {
            EpiParams ep;
            ep.kind = EPI_STORE_F32;
            ep.out_f32 = h->U;
            ep.ldo = V;
            if (chain) {
                CUDA_TRY(h, chained_gemm(h, R, WView{h->out_proj, &h->tc_out_proj, &h->ts_out_proj}, V, d, ep, st,
                                         CAT_OUT_PROJ));
                CUDA_TRY(h, cudaStreamWaitEvent(st, h->ev_join, 0));
            } else if (lowp) {
                // norm_gemm opens its own normalisation and projection ranges
                CUDA_TRY(h, norm_gemm(h, h->out_norm, R, WView{h->out_proj, &h->tc_out_proj, &h->ts_out_proj}, V, d, ep,
                                      h->act_lp, DT_BF16, st, CAT_OUT_PROJ));
            } else {
                Prof pr(h, CAT_OUT_PROJ, st);
                CUDA_TRY(h, gemm(h, DT_F32, h->y, d, nullptr, 0, WView{h->out_proj, &h->tc_out_proj, &h->ts_out_proj}, R, V,
                                 d, ep, st));
            }
        }
    }
    MarkovParams mp;
    mp.U = h->U;
    mp.w1 = h->w1;
    mp.w2 = h->w2;
    mp.w_dtype = h->dt;
    mp.y = h->y;
    mp.conf_w = h->conf_wb;
    mp.B = B;
    mp.gamma = c.gamma;
    mp.V = V;
    mp.r = c.markov_rank;
    mp.d = d;
    mp.anchors = anchors_dev;
    mp.anchor = anchor;
    mp.tokens = tokens;
    mp.conf = conf;
    mp.logits = logits;
    mp.part_v = h->mk_v;
    mp.part_i = h->mk_i;
    mp.counters = h->mk_cnt;
    mp.err = h->d_err;
    mp.ctas = h->mk_ctas;
    mp.keys = h->mk_keys;
    mp.keys_stride = 16 * h->cfg.max_seqs;
    mp.epoch = h->mk_bar + 2;
    mp.bar = h->mk_keys + 2 * (size_t)h->cfg.max_seqs * 16;
    Prof pr(h, CAT_MARKOV, st);
    if (h->samp_t > 0.f) {
        SampleParams sp;
        sp.U = h->U;
        sp.w1 = h->w1;
        sp.w2 = h->w2;
        sp.w_dtype = h->dt;
        sp.y = h->y;
        sp.conf_w = h->conf_wb;
        sp.B = B;
        sp.gamma = c.gamma;
        sp.V = V;
        sp.r = c.markov_rank;
        sp.d = d;
        sp.anchors = anchors_dev;
        sp.anchor = anchor;
        sp.seq_ids = seq_ids;
        sp.n_slots = c.max_seqs;
        sp.tokens = tokens;
        sp.conf = conf;
        sp.logits = logits;
        sp.temperature = h->samp_t;
        sp.top_k = h->samp_k;
        sp.seed = h->samp_seed;
        sp.draws = h->samp_draws;
        sp.cand = h->samp_cand;
        sp.cand_stride = 64;
        sp.err = h->d_err;
        for (int k = 0; k < c.gamma; ++k) {
            sp.k = k;
            CUDA_TRY(h, markov_sample_step(sp, h->num_sms, st));
        }
        return DSPARK_OK;
    }
    if (B >= 8 && h->tc_mk_E.ready && tc_gemm_ok(V, B, c.markov_rank) && anchors_dev) {
        // many sequences: per position a [V, r] x [B, r]^T tensor-core GEMM reads w2 once for all of
        // them; vocabulary entries are the rows, so the base logits are read along their rows
        const int nch = (V + 31) / 32;
        for (int k = 0; k < c.gamma; ++k) {
            CUDA_TRY(h, markov_gather(h->w1, c.markov_rank, V, anchors_dev, tokens, c.gamma, k, B, h->mk_E, st));
            EpiParams ep;
            ep.kind = EPI_MARKOV_T;
            ep.ldo = V;
            ep.mk_nch = nch;
            ep.gamma = c.gamma;
            ep.mk_U = h->U;
            ep.mk_logits = logits;
            ep.mk_part_v = h->mk_pv;
            ep.mk_part_i = h->mk_pi;
            ep.mk_k = k;
            CUDA_TRY(h, tc_gemm(h->w2, c.markov_rank, h->tc_mk_E, V, B, c.markov_rank, ep, h->num_sms, h->d_err, st));
            CUDA_TRY(h, markov_finish(h->mk_pv, h->mk_pi, nch, h->w1, h->dt, h->y, h->conf_wb, anchors_dev, tokens, conf,
                                      B, c.gamma, k, d, c.markov_rank, V, h->d_err, st));
        }
        return DSPARK_OK;
    }
    if (h->mk_fma && h->mk_slots) {
        MarkovParams fp = mp;
        fp.keys = h->mk_slots;
        fp.keys_stride = 16 * 2 * (h->num_sms + 1);
        fp.epoch = h->mk_bar + 3;
        fp.bar = nullptr;
        if (markov_chain_fma_ok(fp, h->num_sms)) {
            CUDA_TRY(h, markov_chain_fma(fp, h->num_sms, st));
            return DSPARK_OK;
        }
    }
    if (markov_chain_resident_ok(mp)) {
        CUDA_TRY(h, markov_chain_resident(mp, h->num_sms, st));
        return DSPARK_OK;
    }
    // one cooperative launch when B sequences x ctas fit co-resident, else one launch per position
    const int chain_ctas = std::min(h->mk_ctas, h->mk_chain_max / std::max(B, 1));
    if (chain_ctas >= 8 || chain_ctas >= h->mk_ctas) {
        mp.ctas = chain_ctas;
        CUDA_TRY(h, markov_chain(mp, h->mk_bar, h->mk_bar + 1, st));
        return DSPARK_OK;
    }
    for (int k = 0; k < c.gamma; ++k) {
        mp.k = k;
        CUDA_TRY(h, markov_step(mp, st));
    }
    return DSPARK_OK;
}

void destroy_graph(DraftGraph& g) {
    if (g.exec) cudaGraphExecDestroy(g.exec);
    if (g.graph) cudaGraphDestroy(g.graph);
    for (auto& r : g.ranges) {
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    g = DraftGraph();
}

// The draft step through a cached CUDA graph: captured on the handle's own
// stream the first time (inputs, outputs, B and the profiling mask form the
// key), then replayed on `st`.  Kernels read every per-call value (context
// lengths, anchors, previous tokens) from device memory, so a replay needs no
// parameter updates.
dspark_status draft_graphed(dspark_handle* h, int B, const int* seq_ids, const int* anchors, int max_keys,
                            int* tokens, float* conf, float* logits, cudaStream_t st) {
    const uint32_t mask = h->prof_on ? h->prof_mask : 0u;
    DraftGraph* g = nullptr;
    for (auto& c : h->graphs)
        if (c.exec && c.B == B && c.seq_ids == seq_ids && c.anchors == anchors && c.tokens == tokens &&
            c.conf == conf && c.logits == logits && c.mask == mask)
            g = &c;
    if (!g) {
        if (h->graphs.size() >= 8) {
            auto old = std::min_element(h->graphs.begin(), h->graphs.end(),
                                        [](const DraftGraph& a, const DraftGraph& b) { return a.last_use < b.last_use; });
            destroy_graph(*old);
            h->graphs.erase(old);
        }
        DraftGraph ng;
        ng.B = B;
        ng.seq_ids = seq_ids;
        ng.anchors = anchors;
        ng.tokens = tokens;
        ng.conf = conf;
        ng.logits = logits;
        ng.mask = mask;
        const long long l0 = launch_count();
        CUDA_TRY(h, cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeRelaxed));
        h->cap_ranges = &ng.ranges;
        dspark_status s = draft_rows(h, B, seq_ids, anchors, 0, max_keys, tokens, conf, logits, h->cap_stream);
        h->cap_ranges = nullptr;
        cudaError_t ce = cudaStreamEndCapture(h->cap_stream, &ng.graph);
        ng.kernels = launch_count() - l0;
        note_launch(-(int)ng.kernels);  // capturing is not launching
        if (s != DSPARK_OK || ce != cudaSuccess) {
            destroy_graph(ng);
            if (s != DSPARK_OK) return s;
            return fail(h, DSPARK_ERR_CUDA, std::string("graph capture: ") + cudaGetErrorString(ce));
        }
        cudaError_t ie = cudaGraphInstantiate(&ng.exec, ng.graph, 0);
        if (ie != cudaSuccess) {
            destroy_graph(ng);
            return fail(h, DSPARK_ERR_CUDA, std::string("graph instantiate: ") + cudaGetErrorString(ie));
        }
        if (!ng.ranges.empty()) {
            size_t n = 0;
            cudaGraphGetNodes(ng.graph, nullptr, &n);
            std::vector<cudaGraphNode_t> nodes(n);
            cudaGraphGetNodes(ng.graph, nodes.data(), &n);
            for (auto node : nodes) {
                cudaGraphNodeType t;
                if (cudaGraphNodeGetType(node, &t) != cudaSuccess || t != cudaGraphNodeTypeEventRecord) continue;
                cudaEvent_t e;
                if (cudaGraphEventRecordNodeGetEvent(node, &e) != cudaSuccess) continue;
                for (auto& r : ng.ranges) {
                    if (r.a == e) r.na = node;
                    if (r.b == e) r.nb = node;
                }
            }
        }
        h->graphs.push_back(std::move(ng));
        g = &h->graphs.back();
    }
    g->last_use = ++h->graph_clock;
    if (mask) {
        for (auto& r : g->ranges) {
            if (!r.na || !r.nb) continue;
            cudaEvent_t a = pool_event(h), b = pool_event(h);
            if (!a || !b) break;
            CUDA_TRY(h, cudaGraphExecEventRecordNodeSetEvent(g->exec, r.na, a));
            CUDA_TRY(h, cudaGraphExecEventRecordNodeSetEvent(g->exec, r.nb, b));
            h->prof_ranges.push_back({r.cat, a, b, r.launches});
        }
    }
    CUDA_TRY(h, cudaGraphLaunch(g->exec, st));
    note_launch((int)g->kernels);
    return DSPARK_OK;
}

}  // namespace

extern "C" {

dspark_status dspark_profile(dspark_handle* h, int32_t class_mask) {
    if (!h) return fail(nullptr, DSPARK_ERR_INVALID_ARG, "handle is NULL");
    if (class_mask) {
        CUDA_TRY(h, cudaDeviceSynchronize());
        h->prof_ranges.clear();
        h->prof_next = 0;
    }
    h->prof_on = class_mask != 0;
    h->prof_mask = (uint32_t)class_mask;
    return DSPARK_OK;
}

int32_t dspark_profile_read(dspark_handle* h, int32_t max, const char** names_host, double* ms_host,
                            int64_t* ranges_host, int64_t* launches_host) {
    if (!h) return -1;
    double ms[CAT_COUNT] = {0};
    int64_t nr[CAT_COUNT] = {0}, nl[CAT_COUNT] = {0};
    for (auto& r : h->prof_ranges) {
        if (cudaEventSynchronize(r.b) != cudaSuccess) return -1;
        float t = 0.f;
        if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return -1;
        ms[r.cat] += t;
        nr[r.cat] += 1;
        nl[r.cat] += r.launches;
    }
    for (int c = 0; c < CAT_COUNT && c < max; ++c) {
        if (names_host) names_host[c] = kCatNames[c];
        if (ms_host) ms_host[c] = ms[c];
        if (ranges_host) ranges_host[c] = nr[c];
        if (launches_host) launches_host[c] = nl[c];
    }
    return CAT_COUNT;
}

dspark_status dspark_linear(int32_t dtype, const void* A_dev, int64_t lda, const void* W_dev, int32_t M, int32_t N,
                            int32_t K, float* out_dev, int64_t ldo, int32_t kernel, void* stream) {
    if (!A_dev || !W_dev || !out_dev) return fail(nullptr, DSPARK_ERR_INVALID_ARG, "a pointer is NULL");
    if (M < 0 || N < 0 || K <= 0 || lda < K || ldo < N) return fail(nullptr, DSPARK_ERR_INVALID_ARG, "bad shape");
    if (dtype != DSPARK_BF16 && dtype != DSPARK_FP32) return fail(nullptr, DSPARK_ERR_INVALID_ARG, "unknown dtype");
    if (M == 0 || N == 0) return DSPARK_OK;
    cudaStream_t st = (cudaStream_t)stream;
    const int dt = dtype == DSPARK_BF16 ? DT_BF16 : DT_F32;
    EpiParams ep;
    ep.kind = EPI_STORE_F32;
    ep.out_f32 = out_dev;
    ep.ldo = ldo;
    static int* err_word = nullptr;
    int num_sms = 148, dev = 0;
    CUDA_TRY(nullptr, cudaGetDevice(&dev));
    CUDA_TRY(nullptr, cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev));
    if (kernel == 0) {
        if (M <= 16 && dt == DT_BF16 && tc_stream_ok(M, N, K)) kernel = 4;
        else if (M <= 16 && skinny_ok(M, K)) kernel = 2;
        else if (dt == DT_BF16 && tc_available() && tc_gemm_ok(M, N, K)) kernel = tc_wide_preferred(M, N, num_sms) ? 5 : 3;
        else kernel = 1;
    }
    if (kernel == 1) {
        CUDA_TRY(nullptr, gemm_simt(dt, A_dev, lda, nullptr, dt, W_dev, M, N, K, ep, st));
    } else if (kernel == 2) {
        if (!skinny_ok(M, K) || lda % 8 != 0) return fail(nullptr, DSPARK_ERR_UNSUPPORTED, "shape not for weight streaming");
        CUDA_TRY(nullptr, gemm_skinny(dt, A_dev, lda, nullptr, 0, dt, W_dev, M, N, K, ep, nullptr, 0, num_sms, st));
    } else if (kernel == 3) {
        if (dt != DT_BF16 || !tc_available() || !tc_gemm_ok(M, N, K) || lda % 8 != 0 || ((uintptr_t)A_dev & 15) ||
            ((uintptr_t)W_dev & 15))
            return fail(nullptr, DSPARK_ERR_UNSUPPORTED, "shape not for the tensor-core GEMM");
        if (!err_word) CUDA_TRY(nullptr, cudaMalloc((void**)&err_word, sizeof(int)));
        TcWeight w;
        CUDA_TRY(nullptr, tc_prepare(w, W_dev, N, K));
        if (!w.ready) return fail(nullptr, DSPARK_ERR_UNSUPPORTED, "tensor map rejected");
        CUDA_TRY(nullptr, tc_gemm(A_dev, lda, w, M, N, K, ep, num_sms, err_word, st));
    } else if (kernel == 5) {
        if (dt != DT_BF16 || !tc_available() || lda % 8 != 0 || ((uintptr_t)A_dev & 15) || ((uintptr_t)W_dev & 15))
            return fail(nullptr, DSPARK_ERR_UNSUPPORTED, "shape not for the wide tensor-core GEMM");
        if (!err_word) CUDA_TRY(nullptr, cudaMalloc((void**)&err_word, sizeof(int)));
        TcWeight w;
        CUDA_TRY(nullptr, tc_prepare(w, W_dev, N, K));
        if (!tc_wide_ok(w, M, N, K, ep)) return fail(nullptr, DSPARK_ERR_UNSUPPORTED, "shape not for the wide tensor-core GEMM");
        CUDA_TRY(nullptr, tc_gemm_wide(A_dev, lda, w, M, N, K, ep, num_sms, err_word, st));
    } else if (kernel == 4) {
        if (dt != DT_BF16 || !tc_stream_ok(M, N, K) || lda % 8 != 0 || ((uintptr_t)A_dev & 15) ||
            ((uintptr_t)W_dev & 15))
            return fail(nullptr, DSPARK_ERR_UNSUPPORTED, "shape not for the streaming tensor-core GEMM");
        // process-wide scratch for this standalone call (grow-only; counters stay zeroed between launches)
        static float* part = nullptr;
        static size_t part_floats = 0;
        static unsigned int* tickets = nullptr;
        static size_t n_tickets = 0;
        if (!err_word) CUDA_TRY(nullptr, cudaMalloc((void**)&err_word, sizeof(int)));
        const size_t need = tc_stream_scratch_floats(N, K, num_sms), tiles = (size_t)(N + 127) / 128;
        if (need > part_floats) {
            CUDA_TRY(nullptr, cudaDeviceSynchronize());
            if (part) cudaFree(part);
            part = nullptr;
            part_floats = 0;
            CUDA_TRY(nullptr, cudaMalloc((void**)&part, need * 4));
            part_floats = need;
        }
        if (tiles > n_tickets) {
            CUDA_TRY(nullptr, cudaDeviceSynchronize());
            if (tickets) cudaFree(tickets);
            tickets = nullptr;
            n_tickets = 0;
            CUDA_TRY(nullptr, cudaMalloc((void**)&tickets, tiles * sizeof(unsigned int)));
            CUDA_TRY(nullptr, cudaMemset(tickets, 0, tiles * sizeof(unsigned int)));
            n_tickets = tiles;
        }
        TcWeightStream w;
        CUDA_TRY(nullptr, tc_stream_prepare(w, W_dev, N, K));
        if (!w.ready) return fail(nullptr, DSPARK_ERR_UNSUPPORTED, "tensor map rejected");
        CUDA_TRY(nullptr, tc_stream(A_dev, lda, w, M, N, K, ep, part, part_floats, tickets, n_tickets, num_sms, err_word, st));
    } else {
        return fail(nullptr, DSPARK_ERR_INVALID_ARG, "unknown kernel");
    }
    return DSPARK_OK;
}

const char* dspark_version(void) { return "dspark-gb300 0.1"; }

const char* dspark_last_error(const dspark_handle* h) { return h ? h->err.c_str() : g_create_error.c_str(); }

int64_t dspark_launch_count(const dspark_handle* h) {
    return h ? (int64_t)(launch_count() - h->launches_at_create) : (int64_t)launch_count();
}

void dspark_destroy(dspark_handle* h) {
    if (!h) return;
    cudaDeviceSynchronize();
    for (void* p : h->allocs) cudaFree(p);
    if (h->rowmap.p) cudaFree(h->rowmap.p);
    if (h->stage_in.p) cudaFree(h->stage_in.p);
    if (h->in_copied) cudaEventDestroy(h->in_copied);
    if (h->stage_out.p) cudaFree(h->stage_out.p);
    for (auto& g : h->graphs) destroy_graph(g);
    if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
    if (h->side_stream) cudaStreamDestroy(h->side_stream);
    if (h->ev_fork) cudaEventDestroy(h->ev_fork);
    if (h->ev_join) cudaEventDestroy(h->ev_join);
    if (h->ev_block) cudaEventDestroy(h->ev_block);
    for (cudaEvent_t e : h->prof_pool) cudaEventDestroy(e);
    tc_release(h->tc_wc);
    tc_release(h->tc_out_proj);
    tc_release(h->tc_mk_E);
    tc_release(h->tc_tok_proj);
    for (auto* v : {&h->tc_kv, &h->tc_qkv, &h->tc_wo, &h->tc_wgu, &h->tc_wd})
        for (auto& w : *v) tc_release(w);
    delete h;
}

dspark_status dspark_create(const dspark_config* cfg, const dspark_weights* w, void* stream, dspark_handle** out) {
    if (!out) return fail(nullptr, DSPARK_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    std::string why;
    dspark_status s = check_cfg(cfg, why);
    if (s != DSPARK_OK) return fail(nullptr, s, why);
    if (!w) return fail(nullptr, DSPARK_ERR_INVALID_ARG, "weights are NULL");
    const int nL = cfg->n_layers;
    if (!w->W_c || !w->ctx_norm || !w->embed || !w->tok_proj || !w->block_pos || (cfg->gamma > 1 && !w->mask_emb) ||
        !w->attn_norm || !w->wq || !w->wk || !w->wv || !w->wo || !w->ff_norm || !w->w_gate || !w->w_up ||
        !w->w_down || !w->out_norm || !w->out_proj || !w->markov_w1 || !w->markov_w2 || !w->conf_w || !w->conf_b)
        return fail(nullptr, DSPARK_ERR_INVALID_ARG, "a weight pointer is NULL");
    for (int i = 0; i < nL; ++i)
        if (!w->attn_norm[i] || !w->wq[i] || !w->wk[i] || !w->wv[i] || !w->wo[i] || !w->ff_norm[i] ||
            !w->w_gate[i] || !w->w_up[i] || !w->w_down[i])
            return fail(nullptr, DSPARK_ERR_INVALID_ARG, "layer " + std::to_string(i) + " has a NULL weight");
    if (cfg->qk_norm) {
        if (!w->q_norm || !w->k_norm) return fail(nullptr, DSPARK_ERR_INVALID_ARG, "q_norm / k_norm are NULL");
        for (int i = 0; i < nL; ++i)
            if (!w->q_norm[i] || !w->k_norm[i])
                return fail(nullptr, DSPARK_ERR_INVALID_ARG, "layer " + std::to_string(i) + " has a NULL q/k norm");
    }

    dspark_handle* h = new dspark_handle();
    h->cfg = *cfg;
    h->launches_at_create = launch_count();
    cudaStream_t st = (cudaStream_t)stream;
    auto bail = [&](dspark_status code) {
        g_create_error = h->err;
        dspark_destroy(h);
        return code;
    };
#define CTRY(expr)                                                                                   \
    do {                                                                                             \
        cudaError_t _e = (expr);                                                                     \
        if (_e != cudaSuccess) {                                                                     \
            h->err = std::string(#expr) + ": " + cudaGetErrorString(_e);                             \
            return bail(_e == cudaErrorMemoryAllocation ? DSPARK_ERR_OOM : DSPARK_ERR_CUDA);         \
        }                                                                                            \
    } while (0)
    CTRY(cudaGetDevice(&h->device));
    CTRY(cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device));
    h->dt = cfg->dtype == DSPARK_BF16 ? DT_BF16 : DT_F32;
    h->esz = h->dt == DT_BF16 ? 2 : 4;
    const int d = cfg->d_draft, F = cfg->ff_mult * d, H = cfg->hidden, V = cfg->vocab, r = cfg->markov_rank;
    const size_t es = h->esz;
    h->d = d;
    h->F = F;
    h->hd = d / cfg->n_heads;
    h->nkv = cfg->n_kv_heads ? cfg->n_kv_heads : cfg->n_heads;
    h->dkv = h->nkv * h->hd;
    h->qk_rope = cfg->qk_norm != 0 || cfg->rope_theta > 0.f;
    h->mH = cfg->n_taps * H;
    h->R = cfg->max_seqs * cfg->gamma;
    const int R = h->R;

    auto copy_mat = [&](void** dst, const void* src, size_t elems) -> cudaError_t {
        cudaError_t e = dalloc(h, dst, elems * es);
        if (e != cudaSuccess) return e;
        return cudaMemcpyAsync(*dst, src, elems * es, cudaMemcpyDeviceToDevice, st);
    };
    auto copy_f32 = [&](float** dst, const float* src, size_t n) -> cudaError_t {
        cudaError_t e = dalloc(h, (void**)dst, n * 4);
        if (e != cudaSuccess) return e;
        return cudaMemcpyAsync(*dst, src, n * 4, cudaMemcpyDeviceToDevice, st);
    };
    CTRY(copy_mat(&h->W_c, w->W_c, (size_t)d * h->mH));
    CTRY(copy_f32(&h->ctx_norm, w->ctx_norm, d));
    h->embed = w->embed;
    CTRY(copy_mat(&h->tok_proj, w->tok_proj, (size_t)d * H));
    CTRY(dalloc(h, (void**)&h->block_const, (size_t)cfg->gamma * d * 4));
    CTRY(block_const_init(h->dt, cfg->gamma > 1 ? w->mask_emb : w->block_pos, w->block_pos, cfg->gamma, d,
                          h->block_const, st));
    h->wqkv.resize(nL);
    h->wo.resize(nL);
    h->wgu.resize(nL);
    h->wd.resize(nL);
    h->attn_norm.resize(nL);
    h->ff_norm.resize(nL);
    const int dkv = h->dkv;
    if (cfg->qk_norm) {
        h->q_norm.resize(nL);
        h->k_norm.resize(nL);
    }
    for (int i = 0; i < nL; ++i) {
        const size_t dd = (size_t)d * d, kd = (size_t)dkv * d, qkv = dd + 2 * kd;
        if (i == 0) CTRY(dalloc(h, &h->wqkv[0], (size_t)nL * qkv * es));  // layers back to back
        else h->wqkv[i] = (char*)h->wqkv[0] + (size_t)i * qkv * es;
        CTRY(cudaMemcpyAsync(h->wqkv[i], w->wq[i], dd * es, cudaMemcpyDeviceToDevice, st));
        CTRY(cudaMemcpyAsync((char*)h->wqkv[i] + dd * es, w->wk[i], kd * es, cudaMemcpyDeviceToDevice, st));
        CTRY(cudaMemcpyAsync((char*)h->wqkv[i] + (dd + kd) * es, w->wv[i], kd * es, cudaMemcpyDeviceToDevice, st));
        if (cfg->qk_norm) {
            CTRY(copy_f32(&h->q_norm[i], w->q_norm[i], h->hd));
            CTRY(copy_f32(&h->k_norm[i], w->k_norm[i], h->hd));
        }
        CTRY(copy_mat(&h->wo[i], w->wo[i], dd));
        CTRY(dalloc(h, &h->wgu[i], 2 * (size_t)F * d * es));
        CTRY(cudaMemcpy2DAsync(h->wgu[i], 2 * d * es, w->w_gate[i], d * es, d * es, F, cudaMemcpyDeviceToDevice, st));
        CTRY(cudaMemcpy2DAsync((char*)h->wgu[i] + d * es, 2 * d * es, w->w_up[i], d * es, d * es, F,
                               cudaMemcpyDeviceToDevice, st));
        CTRY(copy_mat(&h->wd[i], w->w_down[i], (size_t)d * F));
        CTRY(copy_f32(&h->attn_norm[i], w->attn_norm[i], d));
        CTRY(copy_f32(&h->ff_norm[i], w->ff_norm[i], d));
    }
    if (cfg->rope_theta > 0.f) {
        CTRY(dalloc(h, (void**)&h->rope_freq, (size_t)(h->hd / 2) * sizeof(double)));
        CTRY(qk_rope_freq_fill(cfg->rope_theta, h->hd, h->rope_freq, st));
    }
    if (cfg->qk_norm) {
        CTRY(dalloc(h, (void**)&h->k_norm_dev, sizeof(float*) * nL));
        CTRY(cudaMemcpyAsync(h->k_norm_dev, h->k_norm.data(), sizeof(float*) * nL, cudaMemcpyHostToDevice, st));
    }
    CTRY(dalloc(h, (void**)&h->attn_norm_dev, sizeof(float*) * nL));
    CTRY(cudaMemcpyAsync(h->attn_norm_dev, h->attn_norm.data(), sizeof(float*) * nL, cudaMemcpyHostToDevice, st));
    CTRY(copy_f32(&h->out_norm, w->out_norm, d));
    CTRY(copy_mat(&h->out_proj, w->out_proj, (size_t)V * d));
    CTRY(copy_mat(&h->w1, w->markov_w1, (size_t)V * r));
    CTRY(copy_mat(&h->w2, w->markov_w2, (size_t)V * r));
    CTRY(dalloc(h, (void**)&h->conf_wb, (size_t)(d + r + 1) * 4));
    CTRY(to_float(h->dt, w->conf_w, d + r, h->conf_wb, st));
    CTRY(to_float(h->dt, w->conf_b, 1, h->conf_wb + d + r, st));

    // caches
    h->rows = (int64_t)cfg->max_ctx + cfg->gamma;
    h->kv_off = h->rows * dkv;
    h->seq_stride = 2 * h->kv_off;
    h->layer_stride = h->seq_stride * cfg->max_seqs;
    CTRY(dalloc(h, &h->cache, (size_t)h->layer_stride * nL * es));
    CTRY(dalloc(h, (void**)&h->d_len, sizeof(int) * cfg->max_seqs));
    CTRY(dalloc(h, (void**)&h->d_len_next, sizeof(int)));
    CTRY(cudaMemsetAsync(h->d_len, 0, sizeof(int) * cfg->max_seqs, st));
    CTRY(dalloc(h, (void**)&h->d_err, sizeof(int)));
    CTRY(cudaMemsetAsync(h->d_err, 0, sizeof(int), st));
    h->len_host.assign(cfg->max_seqs, 0);
    h->len_known.assign(cfg->max_seqs, 1);

    // draft workspaces
    const int wide = std::max(d, F);
    CTRY(dalloc(h, (void**)&h->x, (size_t)R * d * 4));
    CTRY(dalloc(h, (void**)&h->act, (size_t)R * wide * 4));
    CTRY(dalloc(h, (void**)&h->hbuf, (size_t)R * F * 4));
    CTRY(dalloc(h, (void**)&h->q, (size_t)R * d * 4));
    CTRY(dalloc(h, (void**)&h->y, (size_t)R * d * 4));
    CTRY(dalloc(h, (void**)&h->U, (size_t)R * V * 4));
    CTRY(dalloc(h, &h->act_lp, (size_t)R * wide * 2));
    CTRY(dalloc(h, &h->h_lp, (size_t)R * F * 2));
    CTRY(dalloc(h, &h->xb, (size_t)16 * d * 2));
    CTRY(dalloc(h, (void**)&h->ssp, (size_t)(d / 8 + 1) * 16 * sizeof(float)));
    CTRY(cudaMemsetAsync(h->ssp, 0, (size_t)(d / 8 + 1) * 16 * sizeof(float), st));
    {
        size_t worst = 0;
        for (int B = 1; B <= cfg->max_seqs; ++B) {
            int ch = attn_chunks(h, B, cfg->max_ctx + cfg->gamma);
            worst = std::max(worst, attn_scratch_floats(B, cfg->n_heads, ch, cfg->gamma, h->hd));
        }
        h->attn_part_floats = worst;
        CTRY(dalloc(h, (void**)&h->attn_part, worst * 4));
        const size_t nt = (size_t)cfg->max_seqs * cfg->n_heads;
        CTRY(dalloc(h, (void**)&h->attn_tickets, nt * sizeof(unsigned int)));
        CTRY(cudaMemsetAsync(h->attn_tickets, 0, nt * sizeof(unsigned int), st));
    }
    h->mk_ctas = markov_ctas(V);
    h->mk_chain_max = markov_chain_max_ctas(h->dt);
    CTRY(dalloc(h, (void**)&h->mk_v, 2 * (size_t)cfg->max_seqs * h->mk_ctas * 4));
    CTRY(dalloc(h, (void**)&h->mk_i, 2 * (size_t)cfg->max_seqs * h->mk_ctas * 4));
    CTRY(dalloc(h, (void**)&h->mk_bar, 4 * sizeof(unsigned int)));
    CTRY(cudaMemsetAsync(h->mk_bar, 0, 4 * sizeof(unsigned int), st));
    {
        const size_t n_slots = 2 * (size_t)16 * 2 * (h->num_sms + 1);
        CTRY(dalloc(h, (void**)&h->mk_slots, n_slots * sizeof(unsigned long long)));
        CTRY(cudaMemsetAsync(h->mk_slots, 0, n_slots * sizeof(unsigned long long), st));
    }
    CTRY(dalloc(h, (void**)&h->mk_keys, (2 * (size_t)cfg->max_seqs * 16 + 2) * sizeof(unsigned long long)));
    CTRY(cudaMemsetAsync(h->mk_keys, 0, (2 * (size_t)cfg->max_seqs * 16 + 2) * sizeof(unsigned long long), st));
    CTRY(dalloc(h, (void**)&h->mk_cnt, (size_t)cfg->max_seqs * 4));
    CTRY(dalloc(h, (void**)&h->safe_ids, (size_t)cfg->max_seqs * 4));
    CTRY(dalloc(h, (void**)&h->anchor_dev, sizeof(int)));
    CTRY(attention_init());
    CTRY(markov_chain_resident_init());
    CTRY(sample_init());
    CTRY(dalloc(h, (void**)&h->samp_draws, (size_t)cfg->max_seqs * sizeof(unsigned int)));
    CTRY(cudaMemsetAsync(h->samp_draws, 0, (size_t)cfg->max_seqs * sizeof(unsigned int), st));
    CTRY(dalloc(h, (void**)&h->samp_cand,
                (size_t)cfg->max_seqs * sample_ctas(cfg->vocab, h->num_sms) * 64 * sizeof(unsigned long long)));
    CTRY(draft_persistent_init());
    CTRY(dalloc(h, (void**)&h->pk_bar, 3 * sizeof(unsigned long long)));
    CTRY(cudaMemsetAsync(h->pk_bar, 0, 3 * sizeof(unsigned long long), st));
    if (h->dt == DT_BF16 && d % 512 == 0 && F % 512 == 0 && tc_available()) {
        // weight-slice tensor maps of the persistent draft layers (3-D if the driver takes it)
        struct alignas(64) Map128 {
            unsigned char b[128];
        };
        std::vector<Map128> maps((size_t)4 * nL);
        for (int three = 1; three >= 0 && !h->pk_maps; --three) {
            bool ok = true;
            for (int i = 0; i < nL && ok; ++i) {
                ok = tc_encode_slot_map(&maps[4 * i + 0], h->wqkv[i], 3 * (int64_t)d, d, three) &&
                     tc_encode_slot_map(&maps[4 * i + 1], h->wo[i], d, d, three) &&
                     tc_encode_slot_map(&maps[4 * i + 2], h->wgu[i], 2 * (int64_t)F, d, three) &&
                     tc_encode_slot_map(&maps[4 * i + 3], h->wd[i], d, F, three);
            }
            if (!ok) continue;
            CTRY(dalloc(h, &h->pk_maps, maps.size() * sizeof(Map128)));
            CTRY(cudaMemcpyAsync(h->pk_maps, maps.data(), maps.size() * sizeof(Map128), cudaMemcpyHostToDevice, st));
            CTRY(cudaStreamSynchronize(st));  // the host array goes out of scope
            h->pk_map3d = three;
        }
    }
    CTRY(cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking));
    CTRY(cudaStreamCreateWithFlags(&h->side_stream, cudaStreamNonBlocking));
    CTRY(cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming));
    CTRY(cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming));
    CTRY(cudaEventCreateWithFlags(&h->ev_block, cudaEventDisableTiming));
    CTRY(dalloc(h, (void**)&h->safe_anchors, (size_t)cfg->max_seqs * 4));
    CTRY(cudaMemsetAsync(h->mk_cnt, 0, (size_t)cfg->max_seqs * 4, st));
    h->ws_floats = (size_t)4 << 20;
    CTRY(dalloc(h, (void**)&h->ws, h->ws_floats * 4));
    h->ws_side_floats = (size_t)1 << 20;
    CTRY(dalloc(h, (void**)&h->ws_side, h->ws_side_floats * 4));
    // ingest workspaces
    h->ingest_rows = std::max(1, std::min(std::max(cfg->max_ctx, 16), 16384));
    h->P_rows = h->ingest_rows * (h->ingest_rows <= 4096 ? 4 : 1);
    CTRY(dalloc(h, (void**)&h->P, (size_t)h->P_rows * d * 4));
    CTRY(dalloc(h, &h->Nbuf, (size_t)nL * h->ingest_rows * d * es));

    // tensor-core views of the big weights (bf16 only)
    if (h->dt == DT_BF16 && tc_available()) {
        CTRY(tc_prepare(h->tc_wc, h->W_c, d, h->mH));
        CTRY(tc_prepare(h->tc_out_proj, h->out_proj, V, d));
        h->tc_kv.resize(nL);
        h->tc_qkv.resize(nL);
        h->tc_wo.resize(nL);
        h->tc_wgu.resize(nL);
        h->tc_wd.resize(nL);
        for (int i = 0; i < nL; ++i) {
            CTRY(tc_prepare(h->tc_kv[i], (char*)h->wqkv[i] + (size_t)d * d * es, 2 * dkv, d));
            if (i == 0) {
                tc_prepare_grouped(h->tc_kv_a, h->Nbuf, nL, (int64_t)h->ingest_rows * d, h->ingest_rows, d, true);
                tc_prepare_grouped(h->tc_kv_w, (char*)h->wqkv[0] + (size_t)d * d * es, nL,
                                   (int64_t)(d + 2 * dkv) * d, 2 * dkv, d, false);
                // attn_norm folded into the ingest K/V weights (the grouped product's shared-operand form)
                CTRY(dalloc(h, &h->wkv_s, (size_t)nL * 2 * dkv * d * es));
                for (int l = 0; l < nL; ++l)
                    CTRY(scale_cols((char*)h->wqkv[l] + (size_t)d * d * es, h->attn_norm[l], 2 * dkv, d,
                                    (char*)h->wkv_s + (size_t)l * 2 * dkv * d * es, st));
                tc_prepare_grouped(h->tc_kv_ws, h->wkv_s, nL, (int64_t)2 * dkv * d, 2 * dkv, d, false);
                CTRY(tc_prepare(h->tc_kv_a2, h->Nbuf, h->ingest_rows, d));
            }
            CTRY(tc_prepare(h->tc_qkv[i], h->wqkv[i], d + 2 * dkv, d));
            CTRY(tc_prepare(h->tc_wo[i], h->wo[i], d, d));
            CTRY(tc_prepare(h->tc_wgu[i], h->wgu[i], 2 * F, d));
            CTRY(tc_prepare(h->tc_wd[i], h->wd[i], d, F));
        }
        // K-range partials of the batched residual projections: up to 12 ranges of every block row
        const size_t rmax = (size_t)cfg->max_seqs * cfg->gamma;
        if (rmax >= 17) {
            h->kp_floats = std::min<size_t>(12 * rmax * d, (size_t)64 << 20);
            CTRY(dalloc(h, (void**)&h->kp_part, h->kp_floats * 4));
        }
    }
    if (h->dt == DT_BF16 && tc_available() && cfg->max_seqs >= 8) {
        CTRY(tc_prepare(h->tc_tok_proj, h->tok_proj, d, H));
        CTRY(dalloc(h, &h->emb_rows, (size_t)cfg->max_seqs * H * 2));
        CTRY(dalloc(h, &h->mk_E, (size_t)cfg->max_seqs * r * 2));
        CTRY(tc_prepare(h->tc_mk_E, h->mk_E, cfg->max_seqs, r));
        const size_t nch = (size_t)(V + 31) / 32;
        CTRY(dalloc(h, (void**)&h->mk_pv, (size_t)cfg->max_seqs * nch * 4));
        CTRY(dalloc(h, (void**)&h->mk_pi, (size_t)cfg->max_seqs * nch * 4));
    }
    if (h->dt == DT_BF16 && tc_stream_ok(1, 1, 64)) {
        size_t part = 0, tiles = 0;
        auto prep = [&](TcWeightStream& v, const void* p, int N, int K) -> cudaError_t {
            part = std::max(part, tc_stream_scratch_floats(N, K, h->num_sms));
            tiles = std::max(tiles, (size_t)(N + 127) / 128);
            return tc_stream_prepare(v, p, N, K);
        };
        CTRY(prep(h->ts_wc, h->W_c, d, h->mH));
        CTRY(prep(h->ts_out_proj, h->out_proj, V, d));
        if (h->wkv_s) CTRY(prep(h->ts_kv_all, h->wkv_s, nL * 2 * dkv, d));
        h->ts_kv.resize(nL);
        h->ts_qkv.resize(nL);
        h->ts_wo.resize(nL);
        h->ts_wgu.resize(nL);
        h->ts_wd.resize(nL);
        for (int i = 0; i < nL; ++i) {
            CTRY(prep(h->ts_kv[i], (char*)h->wqkv[i] + (size_t)d * d * es, 2 * dkv, d));
            CTRY(prep(h->ts_qkv[i], h->wqkv[i], d + 2 * dkv, d));
            CTRY(prep(h->ts_wo[i], h->wo[i], d, d));
            CTRY(prep(h->ts_wgu[i], h->wgu[i], 2 * F, d));
            CTRY(prep(h->ts_wd[i], h->wd[i], d, F));
        }
        h->ts_part_floats = part;
        h->ts_n_tickets = tiles;
        CTRY(dalloc(h, (void**)&h->ts_part, std::max<size_t>(part, 4) * 4));
        CTRY(dalloc(h, (void**)&h->ts_tickets, tiles * sizeof(unsigned int)));
        CTRY(cudaMemsetAsync(h->ts_tickets, 0, tiles * sizeof(unsigned int), st));
        // the side stream's set, for layer 0's QKV projection beside an ingest
        h->ts_part_side_floats = tc_stream_scratch_floats(d + 2 * dkv, d, h->num_sms);
        h->ts_n_tickets_side = (size_t)(d + 2 * dkv + 127) / 128;
        CTRY(dalloc(h, (void**)&h->ts_part_side, std::max<size_t>(h->ts_part_side_floats, 4) * 4));
        CTRY(dalloc(h, (void**)&h->ts_tickets_side, h->ts_n_tickets_side * sizeof(unsigned int)));
        CTRY(cudaMemsetAsync(h->ts_tickets_side, 0, h->ts_n_tickets_side * sizeof(unsigned int), st));
        // the one-launch tcgen05 draft step: its weight maps in launch order, and its scratch
        CTRY(tc_stream_prepare(h->ts_tok_proj, h->tok_proj, d, H));
        CTRY(draft_step_tc_init());
        bool maps_ok = h->ts_tok_proj.ready && h->ts_out_proj.ready;
        for (int i = 0; i < nL; ++i)
            maps_ok = maps_ok && h->ts_qkv[i].ready && h->ts_wo[i].ready && h->ts_wgu[i].ready && h->ts_wd[i].ready;
        if (maps_ok && dkv == d && d % 128 == 0) {
            struct alignas(64) Map128 {
                unsigned char b[128];
            };
            std::vector<Map128> maps((size_t)2 + 4 * nL);
            auto put = [&](size_t k, const TcWeightStream& w) { memcpy(maps[k].b, w.tmap, 128); };
            put(0, h->ts_tok_proj);
            for (int i = 0; i < nL; ++i) {
                put(1 + 4 * i, h->ts_qkv[i]);
                put(2 + 4 * i, h->ts_wo[i]);
                put(3 + 4 * i, h->ts_wgu[i]);
                put(4 + 4 * i, h->ts_wd[i]);
            }
            put(1 + 4 * (size_t)nL, h->ts_out_proj);
            CTRY(dalloc(h, &h->ds_maps, maps.size() * sizeof(Map128)));
            CTRY(cudaMemcpyAsync(h->ds_maps, maps.data(), maps.size() * sizeof(Map128), cudaMemcpyHostToDevice, st));
            CTRY(cudaStreamSynchronize(st));  // the host array goes out of scope
            const int G = h->num_sms;
            CTRY(dalloc(h, (void**)&h->ds_hcnt, 2 * (size_t)cfg->n_heads * sizeof(unsigned int)));
            CTRY(cudaMemsetAsync(h->ds_hcnt, 0, 2 * (size_t)cfg->n_heads * sizeof(unsigned int), st));
            CTRY(dalloc(h, (void**)&h->ds_qkv, (size_t)cfg->gamma * 3 * d * sizeof(float)));
            CTRY(dalloc(h, (void**)&h->ds_gu, (size_t)cfg->gamma * 2 * F * sizeof(float)));
            h->ds_apart_floats = (size_t)G * cfg->gamma * (h->hd + 4);
            CTRY(dalloc(h, (void**)&h->ds_apart, h->ds_apart_floats * 4));
            CTRY(dalloc(h, (void**)&h->ds_bar, 3 * sizeof(unsigned long long)));
            CTRY(cudaMemsetAsync(h->ds_bar, 0, 3 * sizeof(unsigned long long), st));
            const size_t nmk = 2 * (size_t)17 * G;
            CTRY(dalloc(h, (void**)&h->ds_mk, nmk * sizeof(unsigned long long)));
            CTRY(cudaMemsetAsync(h->ds_mk, 0, nmk * sizeof(unsigned long long), st));
        }
    }
    CTRY(cudaStreamSynchronize(st));
#undef CTRY
    *out = h;
    return DSPARK_OK;
}

dspark_status dspark_ingest_context(dspark_handle* h, const void* feats_dev, int32_t T, void* stream) {
    if (!h) return fail(nullptr, DSPARK_ERR_INVALID_ARG, "handle is NULL");
    if (T < 0) return fail(h, DSPARK_ERR_INVALID_ARG, "T < 0");
    if (T == 0) return DSPARK_OK;
    if (!feats_dev) return fail(h, DSPARK_ERR_INVALID_ARG, "feats is NULL");
    dspark_status s = sync_len(h, 0);
    if (s != DSPARK_OK) return s;
    if ((int64_t)h->len_host[0] + T > h->cfg.max_ctx)
        return fail(h, DSPARK_ERR_CAPACITY, "context would exceed max_ctx (" + std::to_string(h->len_host[0]) + " + " +
                                                std::to_string(T) + " > " + std::to_string(h->cfg.max_ctx) + ")");
    s = ingest_rows(h, feats_dev, T, nullptr, nullptr, (cudaStream_t)stream);
    if (s != DSPARK_OK) return s;
    h->len_host[0] += T;
    return DSPARK_OK;
}

dspark_status dspark_draft(dspark_handle* h, int32_t last_token, int32_t* tokens_dev, float* conf_dev,
                           float* logits_dev, void* stream) {
    if (!h) return fail(nullptr, DSPARK_ERR_INVALID_ARG, "handle is NULL");
    if (!tokens_dev || !conf_dev) return fail(h, DSPARK_ERR_INVALID_ARG, "tokens or conf is NULL");
    if (last_token < 0 || last_token >= h->cfg.vocab)
        return fail(h, DSPARK_ERR_INVALID_ARG, "last_token " + std::to_string(last_token) + " outside [0, vocab)");
    cudaStream_t st = (cudaStream_t)stream;
    if (h->use_graphs) {
        CUDA_TRY(h, set_len(h->anchor_dev, 0, last_token, st));
        return draft_graphed(h, 1, nullptr, h->anchor_dev, h->cfg.max_ctx + h->cfg.gamma, tokens_dev, conf_dev,
                             logits_dev, st);
    }
    dspark_status s = sync_len(h, 0);
    if (s != DSPARK_OK) return s;
    return draft_rows(h, 1, nullptr, nullptr, last_token, h->len_host[0] + h->cfg.gamma, tokens_dev, conf_dev,
                      logits_dev, st);
}

dspark_status dspark_ingest_and_draft(dspark_handle* h, const void* feats_dev, int32_t T, int32_t last_token,
                                      int32_t* tokens_dev, float* conf_dev, float* logits_dev, void* stream) {
    if (!h) return fail(nullptr, DSPARK_ERR_INVALID_ARG, "handle is NULL");
    if (T < 0) return fail(h, DSPARK_ERR_INVALID_ARG, "T < 0");
    if (T > 0 && !feats_dev) return fail(h, DSPARK_ERR_INVALID_ARG, "feats is NULL");
    if (!tokens_dev || !conf_dev) return fail(h, DSPARK_ERR_INVALID_ARG, "tokens or conf is NULL");
    if (last_token < 0 || last_token >= h->cfg.vocab)
        return fail(h, DSPARK_ERR_INVALID_ARG, "last_token " + std::to_string(last_token) + " outside [0, vocab)");
    dspark_status s = sync_len(h, 0);
    if (s != DSPARK_OK) return s;
    if ((int64_t)h->len_host[0] + T > h->cfg.max_ctx)
        return fail(h, DSPARK_ERR_CAPACITY, "context would exceed max_ctx (" + std::to_string(h->len_host[0]) + " + " +
                                                std::to_string(T) + " > " + std::to_string(h->cfg.max_ctx) + ")");
    cudaStream_t st = (cudaStream_t)stream;
    if (h->layers_path == LAYERS_STEP_TC) {  // the one-launch step builds its block itself
        if (T > 0) {
            s = ingest_rows(h, feats_dev, T, nullptr, nullptr, st);
            if (s != DSPARK_OK) return s;
            h->len_host[0] += T;
        }
        return draft_rows(h, 1, nullptr, nullptr, last_token, h->len_host[0] + h->cfg.gamma, tokens_dev, conf_dev,
                          logits_dev, st);
    }
    // The block rows read no context: they are built on the side stream while the context is
    // ingested.  So is layer 0's QKV projection when its norm comes through the block build: it
    // reads only the block rows, and it writes the block's K/V rows after the new context, at the
    // length the host already knows (a word of its own, as the ingest updates the device length).
    CUDA_TRY(h, cudaEventRecord(h->ev_fork, st));
    CUDA_TRY(h, cudaStreamWaitEvent(h->side_stream, h->ev_fork, 0));
    bool chain0 = false, qkv0_early = false;
    {
        SideScratch side(h);
        s = block_build(h, 1, nullptr, nullptr, last_token, h->side_stream, &chain0);
        if (s != DSPARK_OK) return s;
        qkv0_early = T > 0 && chain0 && !h->qk_rope && h->ts_part &&
                     (h->layers_path == LAYERS_AUTO || h->layers_path == LAYERS_PER_KERNEL) &&
                     norm_chain_ok(h, h->cfg.gamma, h->dt == DT_BF16);
        if (qkv0_early) {
            CUDA_TRY(h, set_len(h->d_len_next, 0, h->len_host[0] + T, h->side_stream));
            const WView wqkv{h->wqkv[0], at_or_null(h->tc_qkv, 0), at_or_null(h->ts_qkv, 0)};
            CUDA_TRY(h, chained_gemm(h, h->cfg.gamma, wqkv, h->d + 2 * h->dkv, h->d,
                                     qkv_epi(h, 0, nullptr, h->d_len_next), h->side_stream, CAT_QKV_SIDE));
        }
    }
    CUDA_TRY(h, cudaEventRecord(h->ev_block, h->side_stream));
    if (T > 0) {
        s = ingest_rows(h, feats_dev, T, nullptr, nullptr, st);
        if (s != DSPARK_OK) return s;
        h->len_host[0] += T;
    }
    CUDA_TRY(h, cudaStreamWaitEvent(st, h->ev_block, 0));
    return draft_rows(h, 1, nullptr, nullptr, last_token, h->len_host[0] + h->cfg.gamma, tokens_dev, conf_dev,
                      logits_dev, st, chain0 ? 1 : 0, qkv0_early);
}

dspark_status dspark_ingest_context_batched(dspark_handle* h, int32_t n_seqs, const int32_t* seq_ids_dev,
                                            const int32_t* cu_tokens_dev, const void* feats_dev, int32_t total_tokens,
                                            void* stream) {
    if (!h) return fail(nullptr, DSPARK_ERR_INVALID_ARG, "handle is NULL");
    if (n_seqs < 0 || total_tokens < 0) return fail(h, DSPARK_ERR_INVALID_ARG, "negative count");
    if (n_seqs == 0 || total_tokens == 0) return DSPARK_OK;
    if (n_seqs > h->cfg.max_seqs) return fail(h, DSPARK_ERR_CAPACITY, "n_seqs > max_seqs");
    if (!seq_ids_dev || !cu_tokens_dev || !feats_dev) return fail(h, DSPARK_ERR_INVALID_ARG, "a pointer is NULL");
    cudaStream_t st = (cudaStream_t)stream;
    CUDA_TRY(h, grow(h->rowmap, (size_t)total_tokens * 2 * sizeof(int)));
    int* row_seq = (int*)h->rowmap.p;
    int* row_pos = row_seq + total_tokens;
    CUDA_TRY(h, ingest_rowmap(seq_ids_dev, cu_tokens_dev, n_seqs, total_tokens, h->d_len, h->cfg.max_seqs,
                              h->cfg.max_ctx, row_seq, row_pos, h->d_err, st));
    dspark_status s = ingest_rows(h, feats_dev, total_tokens, row_seq, row_pos, st);
    if (s != DSPARK_OK) return s;
    CUDA_TRY(h, ingest_commit(seq_ids_dev, cu_tokens_dev, n_seqs, h->d_len, h->cfg.max_seqs, h->cfg.max_ctx, st));
    std::fill(h->len_known.begin(), h->len_known.end(), 0);
    return DSPARK_OK;
}

dspark_status dspark_draft_batched(dspark_handle* h, int32_t n_seqs, const int32_t* seq_ids_dev,
                                   const int32_t* last_tokens_dev, int32_t* tokens_dev, float* conf_dev,
                                   float* logits_dev, void* stream) {
    if (!h) return fail(nullptr, DSPARK_ERR_INVALID_ARG, "handle is NULL");
    if (n_seqs < 0) return fail(h, DSPARK_ERR_INVALID_ARG, "n_seqs < 0");
    if (n_seqs == 0) return DSPARK_OK;
    if (n_seqs > h->cfg.max_seqs) return fail(h, DSPARK_ERR_CAPACITY, "n_seqs > max_seqs");
    if (!seq_ids_dev || !last_tokens_dev || !tokens_dev || !conf_dev)
        return fail(h, DSPARK_ERR_INVALID_ARG, "a pointer is NULL");
    cudaStream_t st = (cudaStream_t)stream;
    CUDA_TRY(h, check_draft_inputs(seq_ids_dev, last_tokens_dev, n_seqs, h->cfg.max_seqs, h->cfg.vocab, h->d_err,
                                   h->safe_ids, h->safe_anchors, st));
    if (h->use_graphs)
        return draft_graphed(h, n_seqs, h->safe_ids, h->safe_anchors, h->cfg.max_ctx + h->cfg.gamma, tokens_dev,
                             conf_dev, logits_dev, st);
    return draft_rows(h, n_seqs, h->safe_ids, h->safe_anchors, 0, h->cfg.max_ctx + h->cfg.gamma, tokens_dev, conf_dev,
                      logits_dev, st);
}

dspark_status dspark_ingest_context_host(dspark_handle* h, const void* feats_host, int32_t T, void* stream) {
    if (!h) return fail(nullptr, DSPARK_ERR_INVALID_ARG, "handle is NULL");
    if (T < 0) return fail(h, DSPARK_ERR_INVALID_ARG, "T < 0");
    if (T == 0) return DSPARK_OK;
    if (!feats_host) return fail(h, DSPARK_ERR_INVALID_ARG, "feats is NULL");
    cudaStream_t st = (cudaStream_t)stream;
    const size_t bytes = (size_t)T * h->mH * h->esz;
    CUDA_TRY(h, grow(h->stage_in, bytes));
    if (!h->in_copied) CUDA_TRY(h, cudaEventCreateWithFlags(&h->in_copied, cudaEventDisableTiming));
    CUDA_TRY(h, cudaMemcpyAsync(h->stage_in.p, feats_host, bytes, cudaMemcpyHostToDevice, st));
    CUDA_TRY(h, cudaEventRecord(h->in_copied, st));
    dspark_status s = dspark_ingest_context(h, h->stage_in.p, T, stream);
    if (s != DSPARK_OK) return s;
    // the caller may reuse feats_host once it has been read; the ingest itself finishes in stream
    // order, so a draft submitted next queues behind it without an idle gap on the device
    CUDA_TRY(h, cudaEventSynchronize(h->in_copied));
    return DSPARK_OK;
}

dspark_status dspark_draft_host(dspark_handle* h, int32_t last_token, int32_t* tokens_host, float* conf_host,
                                float* logits_host, void* stream) {
    if (!h) return fail(nullptr, DSPARK_ERR_INVALID_ARG, "handle is NULL");
    if (!tokens_host || !conf_host) return fail(h, DSPARK_ERR_INVALID_ARG, "tokens or conf is NULL");
    cudaStream_t st = (cudaStream_t)stream;
    const int g = h->cfg.gamma;
    const size_t lbytes = logits_host ? (size_t)g * h->cfg.vocab * 4 : 0;
    CUDA_TRY(h, grow(h->stage_out, (size_t)g * 8 + 256 + lbytes));
    int* tok = (int*)h->stage_out.p;
    float* cf = (float*)((char*)h->stage_out.p + 128);
    float* lg = logits_host ? (float*)((char*)h->stage_out.p + 256) : nullptr;
    dspark_status s = dspark_draft(h, last_token, tok, cf, lg, stream);
    if (s != DSPARK_OK) return s;
    CUDA_TRY(h, cudaMemcpyAsync(tokens_host, tok, (size_t)g * 4, cudaMemcpyDeviceToHost, st));
    CUDA_TRY(h, cudaMemcpyAsync(conf_host, cf, (size_t)g * 4, cudaMemcpyDeviceToHost, st));
    if (logits_host) CUDA_TRY(h, cudaMemcpyAsync(logits_host, lg, lbytes, cudaMemcpyDeviceToHost, st));
    CUDA_TRY(h, cudaStreamSynchronize(st));
    return DSPARK_OK;
}

dspark_status dspark_reset(dspark_handle* h, int32_t seq_id, void* stream) {
    if (!h) return fail(nullptr, DSPARK_ERR_INVALID_ARG, "handle is NULL");
    if (seq_id < 0 || seq_id >= h->cfg.max_seqs) return fail(h, DSPARK_ERR_INVALID_ARG, "seq_id out of range");
    CUDA_TRY(h, set_len(h->d_len, seq_id, 0, (cudaStream_t)stream));
    h->len_host[seq_id] = 0;
    h->len_known[seq_id] = 1;
    return DSPARK_OK;
}

dspark_status dspark_set_sampling(dspark_handle* h, float temperature, int32_t top_k, uint64_t seed, void* stream) {
    if (!h) return fail(nullptr, DSPARK_ERR_INVALID_ARG, "handle is NULL");
    if (!(temperature >= 0.f) || !std::isfinite(temperature))
        return fail(h, DSPARK_ERR_INVALID_ARG, "temperature must be finite and >= 0");
    if (top_k < 0 || top_k > 64) return fail(h, DSPARK_ERR_INVALID_ARG, "top_k must be in [0, 64]");
    if (temperature > 0.f && !sample_ok(h->cfg.vocab, h->cfg.markov_rank, top_k, h->num_sms))
        return fail(h, DSPARK_ERR_UNSUPPORTED, "sampling is not available for this vocabulary and rank");
    CUDA_TRY(h, cudaMemsetAsync(h->samp_draws, 0, (size_t)h->cfg.max_seqs * sizeof(unsigned int),
                                (cudaStream_t)stream));
    h->samp_t = temperature;
    h->samp_k = top_k;
    h->samp_seed = seed;
    for (auto& g : h->graphs) destroy_graph(g);  // the captured steps carry the old settings
    h->graphs.clear();
    return DSPARK_OK;
}

dspark_status dspark_set_path(dspark_handle* h, int32_t what, int32_t value) {
    if (!h) return fail(nullptr, DSPARK_ERR_INVALID_ARG, "handle is NULL");
    switch (what) {
        case DSPARK_PATH_LAYERS:
            if (value < 0 || value > 3) return fail(h, DSPARK_ERR_INVALID_ARG, "layers path must be in [0, 3]");
            h->layers_path = value;
            break;
        case DSPARK_PATH_MARKOV:
            if (value < 0 || value > 1) return fail(h, DSPARK_ERR_INVALID_ARG, "Markov path must be 0 or 1");
            h->mk_fma = value == 0;
            break;
        case DSPARK_PATH_NORM_CHAIN:
            if (value < 0 || value > 1) return fail(h, DSPARK_ERR_INVALID_ARG, "norm-chain path must be 0 or 1");
            h->chain_norm = value == 0;
            break;
        case DSPARK_PATH_GRAPHS:
            if (value < 0 || value > 1) return fail(h, DSPARK_ERR_INVALID_ARG, "graphs path must be 0 or 1");
            h->use_graphs = value == 0;
            break;
        default:
            return fail(h, DSPARK_ERR_INVALID_ARG, "unknown path");
    }
    // captured draft steps were recorded with the old choice
    for (auto& g : h->graphs) destroy_graph(g);
    h->graphs.clear();
    return DSPARK_OK;
}

dspark_status dspark_selftest_wait(int32_t which, int32_t* word_host) {
    if (which < 0 || which > 5) return fail(nullptr, DSPARK_ERR_INVALID_ARG, "which must be in [0, 5]");
    void* scratch = nullptr;
    int* err = nullptr;
    cudaStream_t st = nullptr;
    auto done = [&](dspark_status s, const std::string& why) {
        if (st) cudaStreamDestroy(st);
        if (scratch) cudaFree(scratch);
        if (err) cudaFree(err);
        return s == DSPARK_OK ? s : fail(nullptr, s, why);
    };
    cudaError_t e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaMalloc(&scratch, 64);
    if (e == cudaSuccess) e = cudaMalloc((void**)&err, sizeof(int));
    if (e == cudaSuccess) e = cudaMemsetAsync(scratch, 0, 64, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(err, 0, sizeof(int), st);
    if (e == cudaSuccess) {
        if (which <= 2) e = markov_wait_selftest(which, scratch, err, st);
        else if (which == 3) e = persistent_wait_selftest(scratch, err, st);
        else if (which == 4) e = mbar_wait_selftest(err, st);
        else e = step_wait_selftest(scratch, err, st);
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    int v = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&v, err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return done(DSPARK_ERR_CUDA, std::string("self-test: ") + cudaGetErrorString(e));
    if (word_host) *word_host = v;
    return done(DSPARK_OK, "");
}

dspark_status dspark_check(dspark_handle* h, int32_t* word_host) {
    if (!h) return fail(nullptr, DSPARK_ERR_INVALID_ARG, "handle is NULL");
    int v = 0;
    CUDA_TRY(h, cudaDeviceSynchronize());
    CUDA_TRY(h, cudaMemcpy(&v, h->d_err, sizeof(int), cudaMemcpyDeviceToHost));
    CUDA_TRY(h, cudaMemset(h->d_err, 0, sizeof(int)));
    if (word_host) *word_host = v;
    if (v) return fail(h, DSPARK_ERR_DEVICE, "device error word " + std::to_string(v));
    return DSPARK_OK;
}

dspark_status dspark_context_length(dspark_handle* h, int32_t seq_id, int32_t* out_host) {
    if (!h) return fail(nullptr, DSPARK_ERR_INVALID_ARG, "handle is NULL");
    if (!out_host) return fail(h, DSPARK_ERR_INVALID_ARG, "out is NULL");
    if (seq_id < 0 || seq_id >= h->cfg.max_seqs) return fail(h, DSPARK_ERR_INVALID_ARG, "seq_id out of range");
    int v = 0, e = 0;
    CUDA_TRY(h, cudaDeviceSynchronize());
    CUDA_TRY(h, cudaMemcpy(&v, h->d_len + seq_id, sizeof(int), cudaMemcpyDeviceToHost));
    CUDA_TRY(h, cudaMemcpy(&e, h->d_err, sizeof(int), cudaMemcpyDeviceToHost));
    *out_host = v;
    h->len_host[seq_id] = v;
    h->len_known[seq_id] = 1;
    if (e) return fail(h, DSPARK_ERR_DEVICE, "device error word " + std::to_string(e));
    return DSPARK_OK;
}

dspark_status dspark_get_cache(dspark_handle* h, int32_t seq_id, int32_t layer, const void** k_dev,
                               const void** v_dev) {
    if (!h) return fail(nullptr, DSPARK_ERR_INVALID_ARG, "handle is NULL");
    if (seq_id < 0 || seq_id >= h->cfg.max_seqs || layer < 0 || layer >= h->cfg.n_layers)
        return fail(h, DSPARK_ERR_INVALID_ARG, "seq_id or layer out of range");
    const char* base = (const char*)h->cache + ((size_t)layer * h->layer_stride + (size_t)seq_id * h->seq_stride) * h->esz;
    if (k_dev) *k_dev = base;
    if (v_dev) *v_dev = base + (size_t)h->kv_off * h->esz;
    return DSPARK_OK;
}

}  // extern "C"
