// Per-head RMSNorm and rotary embedding of Q and K rows: the variant of
// "src/dspark-runtime.js" (kernels noiseNormRope for the block rows and
// contextNormRope for the context rows, with the qNorm / kNorm weights).  One
// warp per (row, head): lane l holds the rotation pairs (e, e + hd/2) for
// e = l, l + 32, ... (hd <= 256), the RMS over the head comes from a warp sum,
// and the angle pos * theta^(-2e/hd) is formed and reduced modulo 2 pi in
// double precision before the single-precision sine and cosine (a float angle
// would be off by about 2e-3 rad at position 32768); the frequencies come from a
// table built once on the host, so each pair costs a few double operations.
#include <math.h>
#include <stdint.h>

#include <vector>

#include "common.cuh"
#include "kernels.cuh"

namespace dspark {

namespace {

constexpr int MAXP = 4;  // rotation pairs per lane: head_dim <= 256

__device__ __forceinline__ float ld_elem(const float* p) { return *p; }
__device__ __forceinline__ float ld_elem(const bf16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_elem(float* p, float v) { *p = v; }
__device__ __forceinline__ void st_elem(bf16* p, float v) { *p = __float2bfloat16_rn(v); }

// One head vector v[0, hd) in place: optional RMSNorm with weight w, then optional rotation at pos.
template <typename T>
__device__ __forceinline__ void head_norm_rope(T* v, int hd, const float* w, float eps, const double* freq, int pos) {
    const int lane = threadIdx.x & 31, half = hd >> 1;
    float a[MAXP], b[MAXP];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < MAXP; ++i) {
        const int e = lane + 32 * i;
        a[i] = e < half ? ld_elem(v + e) : 0.f;
        b[i] = e < half ? ld_elem(v + e + half) : 0.f;
        ss += a[i] * a[i] + b[i] * b[i];
    }
    if (w) {
        ss = warp_sum(ss);
        const float r = rsqrtf(ss / (float)hd + eps);
#pragma unroll
        for (int i = 0; i < MAXP; ++i) {
            const int e = lane + 32 * i;
            if (e < half) {
                a[i] *= r * w[e];
                b[i] *= r * w[e + half];
            }
        }
    }
    if (freq) {
        const double two_pi = 6.283185307179586476925286766559;
#pragma unroll
        for (int i = 0; i < MAXP; ++i) {
            const int e = lane + 32 * i;
            if (e < half) {
                double ang = (double)pos * freq[e];
                ang -= two_pi * rint(ang * (1.0 / two_pi));
                float sn, cs;
                sincosf((float)ang, &sn, &cs);
                const float na = a[i] * cs - b[i] * sn, nb = b[i] * cs + a[i] * sn;
                a[i] = na;
                b[i] = nb;
            }
        }
    }
#pragma unroll
    for (int i = 0; i < MAXP; ++i) {
        const int e = lane + 32 * i;
        if (e < half) {
            st_elem(v + e, a[i]);
            st_elem(v + e + half, b[i]);
        }
    }
}

// Block rows: grid (B*gamma, n_heads + n_kv_heads); heads below n_heads are Q heads (fp32
// rows), the rest K heads of the block row in this layer's cache at position len + j.
template <typename TC>
__global__ void __launch_bounds__(32) k_qk_block(QkRope a) {
    pdl_wait();
    pdl_trigger();
    const int m = blockIdx.x, head = blockIdx.y;
    const int b = m / a.gamma, j = m - b * a.gamma;
    const int slot = a.seq_ids ? a.seq_ids[b] : b;
    if (slot < 0) return;
    const int pos = a.seq_len[slot] + j;
    if (head < a.n_heads) {
        head_norm_rope(a.q + (int64_t)m * a.ldq + (int64_t)head * a.head_dim, a.head_dim, a.q_norm, a.eps, a.freq, pos);
    } else {
        if (pos < 0 || pos >= a.max_rows) return;
        TC* k = reinterpret_cast<TC*>(a.cache) + (int64_t)slot * a.seq_stride + (int64_t)pos * a.d_kv +
                (int64_t)(head - a.n_heads) * a.head_dim;
        head_norm_rope(k, a.head_dim, a.k_norm, a.eps, a.freq, pos);
    }
}

// Context rows: grid (rows, n_kv_heads, n_layers); row m of slot row_seq[m] (or 0) at
// row_pos[m] (or len[slot] + m, the length before it moves).
template <typename TC>
__global__ void __launch_bounds__(32) k_qk_ingest(QkRope a) {
    pdl_wait();
    pdl_trigger();
    const int m = blockIdx.x, kvh = blockIdx.y, layer = blockIdx.z;
    const int slot = a.row_seq ? a.row_seq[m] : 0;
    if (slot < 0) return;
    const int pos = a.row_pos ? a.row_pos[m] : a.seq_len[slot] + m;
    if (pos < 0 || pos >= a.max_rows) return;
    TC* k = reinterpret_cast<TC*>(a.cache) + (int64_t)layer * a.layer_stride + (int64_t)slot * a.seq_stride +
            (int64_t)pos * a.d_kv + (int64_t)kvh * a.head_dim;
    head_norm_rope(k, a.head_dim, a.k_norm_layers ? a.k_norm_layers[layer] : nullptr, a.eps, a.freq, pos);
}

bool args_ok(const QkRope& a) {
    return a.cache && a.seq_len && a.head_dim >= 2 && a.head_dim <= 2 * 32 * MAXP && a.head_dim % 2 == 0 &&
           a.n_kv_heads >= 1 && a.d_kv == a.n_kv_heads * a.head_dim && (a.theta <= 0.f || a.freq);
}

}  // namespace

cudaError_t qk_rope_freq_fill(float theta, int head_dim, double* dev, cudaStream_t st) {
    if (!(theta > 0.f) || head_dim < 2 || !dev) return cudaErrorInvalidValue;
    std::vector<double> f(head_dim / 2);
    for (int e = 0; e < head_dim / 2; ++e) f[e] = pow((double)theta, -2.0 * (double)e / (double)head_dim);
    cudaError_t err = cudaMemcpyAsync(dev, f.data(), f.size() * sizeof(double), cudaMemcpyHostToDevice, st);
    if (err == cudaSuccess) err = cudaStreamSynchronize(st);  // the host table goes out of scope
    return err;
}

cudaError_t qk_rope_block(const QkRope& a, cudaStream_t st) {
    if (!args_ok(a) || !a.q || a.n_heads < 1 || a.B < 1 || a.gamma < 1) return cudaErrorInvalidValue;
    const dim3 grid(a.B * a.gamma, a.n_heads + a.n_kv_heads);
    if (a.cache_dtype == DT_BF16) launch(k_qk_block<bf16>, grid, 32, 0, st, a);
    else launch(k_qk_block<float>, grid, 32, 0, st, a);
    note_launch();
    return cudaGetLastError();
}

cudaError_t qk_rope_ingest(const QkRope& a, cudaStream_t st) {
    if (!args_ok(a) || a.rows < 1 || a.n_layers < 1) return cudaErrorInvalidValue;
    const dim3 grid(a.rows, a.n_kv_heads, a.n_layers);
    if (a.cache_dtype == DT_BF16) launch(k_qk_ingest<bf16>, grid, 32, 0, st, a);
    else launch(k_qk_ingest<float>, grid, 32, 0, st, a);
    note_launch();
    return cudaGetLastError();
}

}  // namespace dspark
