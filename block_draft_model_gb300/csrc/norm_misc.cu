// Row normalisations, block set-up and per-sequence bookkeeping kernels.
#include <stdlib.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"

namespace dspark {

namespace {

constexpr int NT = 256;

constexpr int KP_MAX = 12;  // most K-range partials a row norm adds

// ACC: first x += the nparts partial products at parts + s * part_stride (same row layout as x), added
// in order and written back (each element by the thread that later reads it), then the norm.
template <typename TO, bool ACC>
__global__ void __launch_bounds__(NT) k_rmsnorm_rows(float* __restrict__ x, int64_t ldx,
                                                     const float* __restrict__ w, int n, float eps, TO* out,
                                                     int64_t ldo, const float* __restrict__ parts, int nparts,
                                                     int64_t part_stride) {
    pdl_wait();
    pdl_trigger();
    __shared__ float red[32];
    float* xr = x + (int64_t)blockIdx.x * ldx;
    float ss = 0.f;
    for (int c = threadIdx.x; c < n; c += NT) {
        float v = xr[c];
        if constexpr (ACC) {
            // every partial requested at once (at most KP_MAX of them), then added in order
            const float* pr = parts + (int64_t)blockIdx.x * ldx + c;
            float pv[KP_MAX];
#pragma unroll
            for (int sp = 0; sp < KP_MAX; ++sp) pv[sp] = sp < nparts ? pr[sp * part_stride] : 0.f;
#pragma unroll
            for (int sp = 0; sp < KP_MAX; ++sp) v += pv[sp];
            xr[c] = v;
        }
        ss = fmaf(v, v, ss);
    }
    ss = block_sum(ss, red);
    const float s = rsqrtf(ss / (float)n + eps);
    TO* o = out + (int64_t)blockIdx.x * ldo;
    for (int c = threadIdx.x; c < n; c += NT) o[c] = from_f32<TO>(xr[c] * s * w[c]);
}

// Four consecutive outputs with one 8-byte (bf16) or 16-byte (fp32) store.
__device__ __forceinline__ void store4(bf16* o, float a, float b, float c, float d) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(o) = u;
}
__device__ __forceinline__ void store4(float* o, float a, float b, float c, float d) {
    *reinterpret_cast<float4*>(o) = make_float4(a, b, c, d);
}

// Ingest normalisation, one warp per context row (rows_per_warp rows in turn):
// H = RMSNorm(P) * ctx_norm in registers, then every layer's normalised copy
// RMSNorm(H) * attn_norm_i with 8/16-byte stores.  The norm vectors are read
// where they are used (they stay in L1/L2), so the CTAs carry no shared memory
// and many of them are resident at once.
constexpr int INW = 4;  // warps per CTA

// ONE: the instance for one unweighted copy (attn_norm == nullptr), without the per-layer loop.
template <typename TO, int MAXV, bool ONE>
__global__ void __launch_bounds__(INW * 32) k_ingest_norm(const float* __restrict__ P, int nsplit, int64_t split_stride,
                                                         int rows, int d, float eps,
                                                         const float* __restrict__ ctx_norm,
                                                         const float* const* __restrict__ attn_norm, int n_layers,
                                                         TO* out, int64_t layer_stride, int rows_per_warp) {
    pdl_wait();
    pdl_trigger();
    const int nv = d / 4;
    const int lane = threadIdx.x & 31;
    const int row0 = (blockIdx.x * INW + (threadIdx.x >> 5)) * rows_per_warp;
    for (int rr = 0; rr < rows_per_warp; ++rr) {
        const int row = row0 + rr;
        if (row >= rows) break;
        const float4* pr = reinterpret_cast<const float4*>(P + (int64_t)row * d);
        float4 h[MAXV];
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < MAXV; ++i) {
            const int v = lane + 32 * i;
            h[i] = v < nv ? pr[v] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int sp = 1; sp < nsplit; ++sp) {  // partial products of the other K ranges
            const float4* ps = reinterpret_cast<const float4*>(P + sp * split_stride + (int64_t)row * d);
#pragma unroll
            for (int i = 0; i < MAXV; ++i) {
                const int v = lane + 32 * i;
                if (v < nv) {
                    const float4 a = ps[v];
                    h[i] = make_float4(h[i].x + a.x, h[i].y + a.y, h[i].z + a.z, h[i].w + a.w);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < MAXV; ++i) ss += h[i].x * h[i].x + h[i].y * h[i].y + h[i].z * h[i].z + h[i].w * h[i].w;
        ss = warp_sum(ss);
        const float s1 = rsqrtf(ss / (float)d + eps);
        const float4* cn = reinterpret_cast<const float4*>(ctx_norm);
        float ss2 = 0.f;
#pragma unroll
        for (int i = 0; i < MAXV; ++i) {
            const int v = lane + 32 * i;
            if (v < nv) {
                const float4 w = __ldg(cn + v);
                h[i] = make_float4(h[i].x * s1 * w.x, h[i].y * s1 * w.y, h[i].z * s1 * w.z, h[i].w * s1 * w.w);
                ss2 += h[i].x * h[i].x + h[i].y * h[i].y + h[i].z * h[i].z + h[i].w * h[i].w;
            }
        }
        ss2 = warp_sum(ss2);
        const float s2 = rsqrtf(ss2 / (float)d + eps);
        if (ONE) {  // one copy without a norm weight (the weights carry each layer's attn_norm)
            TO* o = out + (int64_t)row * d;
#pragma unroll
            for (int i = 0; i < MAXV; ++i) {
                const int v = lane + 32 * i;
                if (v < nv) store4(o + 4 * v, h[i].x * s2, h[i].y * s2, h[i].z * s2, h[i].w * s2);
            }
            continue;
        }
        if constexpr (!ONE)
        for (int l = 0; l < n_layers; ++l) {
            const float4* an = reinterpret_cast<const float4*>(attn_norm[l]);
            TO* o = out + l * layer_stride + (int64_t)row * d;
#pragma unroll
            for (int i = 0; i < MAXV; ++i) {
                const int v = lane + 32 * i;
                if (v < nv) {
                    const float4 w = __ldg(an + v);
                    store4(o + 4 * v, h[i].x * s2 * w.x, h[i].y * s2 * w.y, h[i].z * s2 * w.z, h[i].w * s2 * w.w);
                }
            }
        }
    }
}

// x = the block rows; with xb set (one sequence, d a multiple of 8) also the first projection's
// operand xb = bf16(x * g) and the 8-column sums of x^2, ssp[(n / 8) * 16 + row].
__global__ void k_block_init(float* __restrict__ x, const float* __restrict__ bc, int B, int gamma, int d,
                             bf16* __restrict__ xb, const float* __restrict__ g, float* __restrict__ ssp) {
    pdl_wait();
    pdl_trigger();
    const int64_t total = (int64_t)B * gamma * d, per = (int64_t)gamma * d;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const float v = bc[i % per];
        x[i] = v;
        if (xb) {  // whole 8-lane groups are active together: total and the strides are multiples of 8
            const int row = (int)(i / d), n = (int)(i - (int64_t)row * d);
            xb[i] = __float2bfloat16(v * g[n]);
            float s2 = v * v;
            const unsigned mask = __activemask();
            s2 += __shfl_xor_sync(mask, s2, 1, 8);
            s2 += __shfl_xor_sync(mask, s2, 2, 8);
            s2 += __shfl_xor_sync(mask, s2, 4, 8);
            if ((n & 7) == 0) ssp[(n >> 3) * 16 + row] = s2;
        }
    }
}

// Wd[r][k] = bf16(W[r][k] * g[k]) for r < rows, k < K (both bf16, K contiguous).
__global__ void k_scale_cols(const bf16* __restrict__ W, const float* __restrict__ g, int rows, int K, bf16* __restrict__ Wd) {
    pdl_wait();
    pdl_trigger();
    const int64_t total = (int64_t)rows * K;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x)
        Wd[i] = __float2bfloat16(__bfloat162float(W[i]) * g[i % K]);
}

__global__ void k_ingest_rowmap(const int* __restrict__ seq_ids, const int* __restrict__ cu, int n_seqs, int total,
                                const int* __restrict__ seq_len, int max_seqs, int max_ctx, int* row_seq, int* row_pos,
                                int* err) {
    pdl_wait();
    pdl_trigger();
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < total; t += gridDim.x * blockDim.x) {
        // sequence i with cu[i] <= t < cu[i+1] (binary search over the prefix sums)
        int lo = 0, hi = n_seqs - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (cu[mid] <= t) lo = mid;
            else hi = mid - 1;
        }
        const int sid = seq_ids[lo];
        if (sid < 0 || sid >= max_seqs) {
            row_seq[t] = 0;
            row_pos[t] = -1;
            atomicOr(err, 2);
            continue;
        }
        const int cnt = cu[lo + 1] - cu[lo];
        const int len = seq_len[sid];
        row_seq[t] = sid;
        if (len + cnt > max_ctx) {
            row_pos[t] = -1;
            if (t == cu[lo]) atomicOr(err, 4);
        } else {
            row_pos[t] = len + (t - cu[lo]);
        }
    }
}

__global__ void k_ingest_commit(const int* __restrict__ seq_ids, const int* __restrict__ cu, int n_seqs, int* seq_len,
                                int max_seqs, int max_ctx) {
    pdl_wait();
    pdl_trigger();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_seqs; i += gridDim.x * blockDim.x) {
        const int sid = seq_ids[i];
        if (sid < 0 || sid >= max_seqs) continue;
        const int cnt = cu[i + 1] - cu[i];
        if (seq_len[sid] + cnt <= max_ctx) seq_len[sid] += cnt;
    }
}

__global__ void k_add_len(int* seq_len, int slot, int delta) {
    pdl_wait();
    pdl_trigger(); seq_len[slot] += delta; }
__global__ void k_set_len(int* seq_len, int slot, int value) {
    pdl_wait();
    pdl_trigger(); seq_len[slot] = value; }

__global__ void k_check_draft(const int* __restrict__ seq_ids, const int* __restrict__ anchors, int n, int max_seqs,
                              int V, int* err, int* safe_ids, int* safe_anchors) {
    pdl_wait();
    pdl_trigger();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const int sid = seq_ids[i];
        const bool bad_id = sid < 0 || sid >= max_seqs;
        if (bad_id) atomicOr(err, 2);
        safe_ids[i] = bad_id ? -1 : sid;
        const int a = anchors[i];
        if (a < 0 || a >= V) atomicOr(err, 1);
        safe_anchors[i] = min(max(a, 0), V - 1);
    }
}

template <typename T>
__global__ void k_block_const(const T* __restrict__ mask_emb, const T* __restrict__ block_pos, int gamma, int d,
                              float* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < gamma * d; i += gridDim.x * blockDim.x) {
        const int j = i / d;
        float v = to_f32(block_pos[i]);
        if (j > 0) v += to_f32(mask_emb[i - d]);
        out[i] = v;
    }
}

template <typename T>
__global__ void k_to_float(const T* __restrict__ in, int64_t n, float* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = to_f32(in[i]);
}

}  // namespace

// Every launch of the step uses programmatic dependent launch.
bool pdl_enabled() { return true; }

static long long g_launches = 0;
long long launch_count() { return __atomic_load_n(&g_launches, __ATOMIC_RELAXED); }
void note_launch(int n) { __atomic_fetch_add(&g_launches, (long long)n, __ATOMIC_RELAXED); }

cudaError_t block_const_init(int dtype, const void* mask_emb, const void* block_pos, int gamma, int d, float* out,
                             cudaStream_t st) {
    const int blocks = std::max(1, std::min((gamma * d + 255) / 256, 1024));
    if (dtype == DT_BF16)
        launch(k_block_const<bf16>, blocks, 256, 0, st, (const bf16*)mask_emb, (const bf16*)block_pos, gamma, d, out);
    else
        launch(k_block_const<float>, blocks, 256, 0, st, (const float*)mask_emb, (const float*)block_pos, gamma, d, out);
    note_launch();
    return cudaGetLastError();
}

cudaError_t to_float(int dtype, const void* in, int64_t n, float* out, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, 1024));
    if (dtype == DT_BF16)
        launch(k_to_float<bf16>, blocks, 256, 0, st, (const bf16*)in, n, out);
    else
        launch(k_to_float<float>, blocks, 256, 0, st, (const float*)in, n, out);
    note_launch();
    return cudaGetLastError();
}

cudaError_t rmsnorm_rows(const float* x, int64_t ldx, const float* w, int rows, int n, float eps, int out_dtype,
                         void* out, int64_t ldo, cudaStream_t st, const float* parts, int nparts, int64_t part_stride) {
    if (rows <= 0) return cudaSuccess;
    float* xm = const_cast<float*>(x);  // written only when partials are added
    const bool acc = parts && nparts > 0;
    if (nparts > KP_MAX) return cudaErrorInvalidValue;
    if (out_dtype == DT_BF16) {
        if (acc) launch(k_rmsnorm_rows<bf16, true>, rows, NT, 0, st, xm, ldx, w, n, eps, (bf16*)out, ldo, parts, nparts, part_stride);
        else launch(k_rmsnorm_rows<bf16, false>, rows, NT, 0, st, xm, ldx, w, n, eps, (bf16*)out, ldo, parts, 0, part_stride);
    } else {
        if (acc) launch(k_rmsnorm_rows<float, true>, rows, NT, 0, st, xm, ldx, w, n, eps, (float*)out, ldo, parts, nparts, part_stride);
        else launch(k_rmsnorm_rows<float, false>, rows, NT, 0, st, xm, ldx, w, n, eps, (float*)out, ldo, parts, 0, part_stride);
    }
    note_launch();
    return cudaGetLastError();
}

template <typename TO, int MAXV>
cudaError_t launch_ingest_norm(const float* P, int nsplit, int64_t split_stride, int rows, int d, float eps,
                               const float* ctx_norm,
                               const float* const* attn_norm_dev, int n_layers, void* out, int64_t layer_stride,
                               cudaStream_t st) {
    // up to four CTAs per SM before a warp takes more than one row
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int rpw = std::max(1, (rows + INW * 4 * sms - 1) / (INW * 4 * sms));
    const int blocks = (rows + INW * rpw - 1) / (INW * rpw);
    if (attn_norm_dev)
        launch(k_ingest_norm<TO, MAXV, false>, blocks, INW * 32, 0, st, P, nsplit, split_stride, rows, d, eps, ctx_norm,
               attn_norm_dev, n_layers, (TO*)out, layer_stride, rpw);
    else
        launch(k_ingest_norm<TO, MAXV, true>, blocks, INW * 32, 0, st, P, nsplit, split_stride, rows, d, eps, ctx_norm,
               attn_norm_dev, n_layers, (TO*)out, layer_stride, rpw);
    note_launch();
    return cudaGetLastError();
}

template <typename TO>
cudaError_t ingest_norm_t(const float* P, int nsplit, int64_t split_stride, int rows, int d, float eps,
                          const float* ctx_norm,
                          const float* const* attn_norm_dev, int n_layers, void* out, int64_t layer_stride,
                          cudaStream_t st) {
    const int per_lane = (d / 4 + 31) / 32;
    if (per_lane <= 2) return launch_ingest_norm<TO, 2>(P, nsplit, split_stride, rows, d, eps, ctx_norm, attn_norm_dev, n_layers, out, layer_stride, st);
    if (per_lane <= 4) return launch_ingest_norm<TO, 4>(P, nsplit, split_stride, rows, d, eps, ctx_norm, attn_norm_dev, n_layers, out, layer_stride, st);
    if (per_lane <= 8) return launch_ingest_norm<TO, 8>(P, nsplit, split_stride, rows, d, eps, ctx_norm, attn_norm_dev, n_layers, out, layer_stride, st);
    if (per_lane <= 16) return launch_ingest_norm<TO, 16>(P, nsplit, split_stride, rows, d, eps, ctx_norm, attn_norm_dev, n_layers, out, layer_stride, st);
    return launch_ingest_norm<TO, 32>(P, nsplit, split_stride, rows, d, eps, ctx_norm, attn_norm_dev, n_layers, out, layer_stride, st);
}

cudaError_t ingest_norm(const float* P, int nsplit, int64_t split_stride, int rows, int d, float eps,
                        const float* ctx_norm, const float* const* attn_norm_dev, int n_layers, int out_dtype,
                        void* out, int64_t layer_stride, cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    if (nsplit < 1 || (nsplit > 1 && split_stride < (int64_t)rows * d)) return cudaErrorInvalidValue;
    if (d % 4 != 0 || d > 4096) return cudaErrorInvalidValue;
    if (out_dtype == DT_BF16)
        return ingest_norm_t<bf16>(P, nsplit, split_stride, rows, d, eps, ctx_norm, attn_norm_dev, n_layers, out,
                                   layer_stride, st);
    return ingest_norm_t<float>(P, nsplit, split_stride, rows, d, eps, ctx_norm, attn_norm_dev, n_layers, out,
                                layer_stride, st);
}

cudaError_t block_init(float* x, const float* block_const, int B, int gamma, int d, cudaStream_t st, void* xb_,
                       const float* g, float* ssp) {
    bf16* xb = static_cast<bf16*>(xb_);
    if (xb && (B != 1 || gamma > 16 || d % 8 != 0 || !g || !ssp)) return cudaErrorInvalidValue;
    int64_t total = (int64_t)B * gamma * d;
    int blocks = (int)std::min<int64_t>((total + 255) / 256, 1024);
    launch(k_block_init, blocks, 256, 0, st, x, block_const, B, gamma, d, xb, g, ssp);
    note_launch();
    return cudaGetLastError();
}

cudaError_t scale_cols(const void* W, const float* g, int rows, int K, void* Wd, cudaStream_t st) {
    if (rows <= 0 || K <= 0) return cudaSuccess;
    const int blocks = (int)std::min<int64_t>(((int64_t)rows * K + 255) / 256, 4096);
    launch(k_scale_cols, blocks, 256, 0, st, (const bf16*)W, g, rows, K, (bf16*)Wd);
    note_launch();
    return cudaGetLastError();
}

cudaError_t ingest_rowmap(const int* seq_ids, const int* cu, int n_seqs, int total, const int* seq_len, int max_seqs,
                          int max_ctx, int* row_seq, int* row_pos, int* err, cudaStream_t st) {
    if (total <= 0) return cudaSuccess;
    int blocks = std::min((total + 255) / 256, 1024);
    launch(k_ingest_rowmap, blocks, 256, 0, st, seq_ids, cu, n_seqs, total, seq_len, max_seqs, max_ctx, row_seq, row_pos, err);
    note_launch();
    return cudaGetLastError();
}

cudaError_t ingest_commit(const int* seq_ids, const int* cu, int n_seqs, int* seq_len, int max_seqs, int max_ctx,
                          cudaStream_t st) {
    if (n_seqs <= 0) return cudaSuccess;
    launch(k_ingest_commit, (n_seqs + 255) / 256, 256, 0, st, seq_ids, cu, n_seqs, seq_len, max_seqs, max_ctx);
    note_launch();
    return cudaGetLastError();
}

cudaError_t add_len(int* seq_len, int slot, int delta, cudaStream_t st) {
    launch(k_add_len, 1, 1, 0, st, seq_len, slot, delta);
    note_launch();
    return cudaGetLastError();
}

cudaError_t set_len(int* seq_len, int slot, int value, cudaStream_t st) {
    launch(k_set_len, 1, 1, 0, st, seq_len, slot, value);
    note_launch();
    return cudaGetLastError();
}

cudaError_t check_draft_inputs(const int* seq_ids, const int* anchors, int n, int max_seqs, int V, int* err,
                               int* safe_ids, int* safe_anchors, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    launch(k_check_draft, (n + 255) / 256, 256, 0, st, seq_ids, anchors, n, max_seqs, V, err, safe_ids, safe_anchors);
    note_launch();
    return cudaGetLastError();
}

}  // namespace dspark
