// Block attention of a draft layer ("module-dflash.ts", #layer: the gamma
// block queries attend bidirectionally over [context ++ block], scale
// head_dim^-1/2, no mask).  The block's own K/V rows have already been written
// to the cache right after the context (rows len .. len+gamma-1), so every key
// is a cache row.
//
// Split-K flash decoding: the keys of one (sequence, head) are cut into
// n_chunks ranges; each CTA keeps a running (max, sum, unnormalised output)
// per query over its range (the "attention" pass of "src/dspark-runtime.js",
// propose, with its partial/md buffers), and a second kernel merges the
// ranges (the "combine" pass).  fp32 throughout; keys and values are read
// from the bf16 (or fp32) cache once.
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"

namespace dspark {

namespace {

constexpr int TK = 32;    // keys per tile
constexpr int NT = 128;   // threads per CTA
constexpr int GMAX = 16;  // largest block size
constexpr int HMAX = 256; // largest head dim

struct Smem {
    static size_t bytes(int gamma, int hd) {
        return sizeof(float) * ((size_t)gamma * hd + (size_t)TK * (hd + 1) + (size_t)TK * hd + (size_t)gamma * TK +
                                3 * (size_t)gamma);
    }
};

template <typename TC>
__device__ __forceinline__ void load_tile(float* dst, int dst_ld, const TC* src_base, int64_t row_stride, int nk,
                                          int hd) {
    constexpr int VE = Vec16<TC>::N;
    const int vecs_per_row = hd / VE;
    for (int idx = threadIdx.x; idx < nk * vecs_per_row; idx += NT) {
        const int row = idx / vecs_per_row, v = idx - row * vecs_per_row;
        uint4 u = *reinterpret_cast<const uint4*>(src_base + row * row_stride + v * VE);
        float f[VE];
        Vec16<TC>::unpack(u, f);
#pragma unroll
        for (int e = 0; e < VE; ++e) dst[row * dst_ld + v * VE + e] = f[e];
    }
}

template <typename TC>
__global__ void __launch_bounds__(NT) k_attn_partial(AttnParams p) {
    extern __shared__ float sm[];
    const int gamma = p.gamma, d = p.d, hd = d / p.n_heads;
    float* q = sm;                          // [gamma][hd]
    float* Ks = q + gamma * hd;             // [TK][hd+1]
    float* Vs = Ks + TK * (hd + 1);         // [TK][hd]
    float* S = Vs + TK * hd;                // [gamma][TK]
    float* m_run = S + gamma * TK;          // [gamma]
    float* l_run = m_run + gamma;           // [gamma]
    float* alpha = l_run + gamma;           // [gamma]

    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int slot = p.seq_ids ? p.seq_ids[b] : b;
    const int n_keys = slot < 0 ? 0 : p.seq_len[slot] + gamma;  // a rejected sequence has no keys
    const int chunk = (n_keys + p.n_chunks - 1) / p.n_chunks;
    const int start = c * chunk, end = min(n_keys, start + chunk);
    const float scale = rsqrtf((float)hd);

    const TC* Kb = reinterpret_cast<const TC*>(p.cache) + (int64_t)max(slot, 0) * p.seq_stride + h * hd;
    const TC* Vb = Kb + p.kv_off;

    for (int idx = threadIdx.x; idx < gamma * hd; idx += NT) {
        const int j = idx / hd, e = idx - j * hd;
        q[idx] = p.q[(int64_t)(b * gamma + j) * d + h * hd + e] * scale;
    }
    for (int j = threadIdx.x; j < gamma; j += NT) {
        m_run[j] = -INFINITY;
        l_run[j] = 0.f;
    }
    float o[GMAX][HMAX / NT];
#pragma unroll
    for (int j = 0; j < GMAX; ++j)
#pragma unroll
        for (int x = 0; x < HMAX / NT; ++x) o[j][x] = 0.f;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int t0 = start; t0 < end; t0 += TK) {
        const int nk = min(TK, end - t0);
        __syncthreads();
        load_tile<TC>(Ks, hd + 1, Kb + (int64_t)t0 * d, d, nk, hd);
        load_tile<TC>(Vs, hd, Vb + (int64_t)t0 * d, d, nk, hd);
        __syncthreads();
        for (int pi = threadIdx.x; pi < gamma * TK; pi += NT) {
            const int j = pi / TK, key = pi - j * TK;
            float s = -INFINITY;
            if (key < nk) {
                const float* qr = q + j * hd;
                const float* kr = Ks + key * (hd + 1);
                float acc = 0.f;
                for (int e = 0; e < hd; ++e) acc = fmaf(qr[e], kr[e], acc);
                s = acc;
            }
            S[pi] = s;
        }
        __syncthreads();
        for (int j = warp; j < gamma; j += NT / 32) {
            const float s = S[j * TK + lane];
            const float mt = warp_max(s);
            const float m_old = m_run[j];
            const float m_new = fmaxf(m_old, mt);
            const float pr = (lane < nk) ? __expf(s - m_new) : 0.f;
            const float sum = warp_sum(pr);
            S[j * TK + lane] = pr;
            __syncwarp();
            if (lane == 0) {
                const float a = (m_old == -INFINITY) ? 0.f : __expf(m_old - m_new);
                alpha[j] = a;
                l_run[j] = l_run[j] * a + sum;
                m_run[j] = m_new;
            }
        }
        __syncthreads();
#pragma unroll
        for (int x = 0; x < HMAX / NT; ++x) {
            const int e = threadIdx.x + x * NT;
            if (e >= hd) break;
#pragma unroll
            for (int j = 0; j < GMAX; ++j)
                if (j < gamma) o[j][x] *= alpha[j];
            for (int key = 0; key < nk; ++key) {
                const float v = Vs[key * hd + e];
#pragma unroll
                for (int j = 0; j < GMAX; ++j)
                    if (j < gamma) o[j][x] = fmaf(S[j * TK + key], v, o[j][x]);
            }
        }
    }
    __syncthreads();
    const int w = hd + 2;
    float* base = p.part + ((((int64_t)b * p.n_heads + h) * p.n_chunks + c) * gamma) * w;
#pragma unroll
    for (int x = 0; x < HMAX / NT; ++x) {
        const int e = threadIdx.x + x * NT;
        if (e >= hd) break;
#pragma unroll
        for (int j = 0; j < GMAX; ++j)
            if (j < gamma) base[j * w + 2 + e] = o[j][x];
    }
    for (int j = threadIdx.x; j < gamma; j += NT) {
        base[j * w] = m_run[j];
        base[j * w + 1] = l_run[j];
    }
}

template <typename TO>
__global__ void __launch_bounds__(NT) k_attn_combine(AttnParams p) {
    const int h = blockIdx.x, b = blockIdx.y;
    const int gamma = p.gamma, d = p.d, hd = d / p.n_heads, w = hd + 2;
    const float* base = p.part + (((int64_t)b * p.n_heads + h) * p.n_chunks) * gamma * w;
    TO* out = reinterpret_cast<TO*>(p.out);
    for (int j = 0; j < gamma; ++j) {
        float M = -INFINITY;
        for (int c = 0; c < p.n_chunks; ++c) M = fmaxf(M, base[((int64_t)c * gamma + j) * w]);
        float L = 0.f;
        for (int c = 0; c < p.n_chunks; ++c) {
            const float mc = base[((int64_t)c * gamma + j) * w];
            if (mc != -INFINITY) L += __expf(mc - M) * base[((int64_t)c * gamma + j) * w + 1];
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        for (int e = threadIdx.x; e < hd; e += NT) {
            float acc = 0.f;
            for (int c = 0; c < p.n_chunks; ++c) {
                const float mc = base[((int64_t)c * gamma + j) * w];
                if (mc != -INFINITY) acc += __expf(mc - M) * base[((int64_t)c * gamma + j) * w + 2 + e];
            }
            out[(int64_t)(b * gamma + j) * d + h * hd + e] = from_f32<TO>(acc * inv);
        }
    }
}

}  // namespace

size_t attn_scratch_floats(int B, int n_heads, int n_chunks, int gamma, int head_dim) {
    return (size_t)B * n_heads * n_chunks * gamma * (head_dim + 2);
}

cudaError_t attention_init() {
    const int sm = (int)Smem::bytes(GMAX, HMAX);
    cudaError_t e = cudaFuncSetAttribute(k_attn_partial<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k_attn_partial<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm);
}

cudaError_t attention(const AttnParams& p, cudaStream_t st) {
    const int hd = p.d / p.n_heads;
    if (p.gamma > GMAX || hd > HMAX || hd % 8 != 0) return cudaErrorInvalidValue;
    const size_t sm = Smem::bytes(p.gamma, hd);
    dim3 g1(p.n_chunks, p.n_heads, p.B);
    if (p.cache_dtype == DT_BF16)
        k_attn_partial<bf16><<<g1, NT, sm, st>>>(p);
    else
        k_attn_partial<float><<<g1, NT, sm, st>>>(p);
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dim3 g2(p.n_heads, p.B);
    if (p.out_dtype == DT_BF16)
        k_attn_combine<bf16><<<g2, NT, 0, st>>>(p);
    else
        k_attn_combine<float><<<g2, NT, 0, st>>>(p);
    note_launch();
    return cudaGetLastError();
}

}  // namespace dspark
