// GEMM epilogues shared by the SIMT, weight-streaming and tensor-core GEMMs.
#pragma once

#include "common.cuh"
#include "kernels.cuh"

#include <climits>

namespace dspark {

__device__ __forceinline__ float act_fn(int act, float g) {
    if (act == 0) return g / (1.f + expf(-g));  // SiLU
    const float c = 0.7978845608028654f;        // sqrt(2/pi)
    return 0.5f * g * (1.f + tanhf(c * (g + 0.044715f * g * g * g)));
}

// Column c of a K/V product ([0, w): K, [w, 2w): V, w = the cache row width) of (slot, pos).
__device__ __forceinline__ void cache_store(const EpiParams& ep, int slot, int pos, int c, float v, int grp = 0) {
    if (pos < 0 || pos >= ep.max_rows) return;
    const int w = ep.d_kv ? ep.d_kv : ep.d;
    int64_t off = grp * ep.group_stride + (int64_t)slot * ep.seq_stride + (c >= w ? ep.kv_off : 0) +
                  (int64_t)pos * w + (c >= w ? c - w : c);
    if (ep.cache_dtype == DT_BF16)
        reinterpret_cast<bf16*>(ep.cache)[off] = __float2bfloat16_rn(v);
    else
        reinterpret_cast<float*>(ep.cache)[off] = v;
}

// EPI_QKV for one element: Q columns to out_f32, K/V columns into the cache after the context.
__device__ __forceinline__ void epi_qkv(const EpiParams& ep, int m, int n, float v) {
    if (n < ep.d) {
        ep.out_f32[(int64_t)m * ep.ldo + n] = v;
    } else {
        int b = m / ep.gamma, j = m - b * ep.gamma;
        int slot = ep.seq_ids ? ep.seq_ids[b] : b;
        if (slot >= 0) cache_store(ep, slot, ep.seq_len[slot] + j, n - ep.d, v);
    }
}

// One output element (every kind except EPI_SWIGLU).
__device__ __forceinline__ void epi_one(const EpiParams& ep, int m, int n, float v, int grp = 0) {
    switch (ep.kind) {
        case EPI_STORE_F32:
            ep.out_f32[(int64_t)m * ep.ldo + n] = v;
            break;
        case EPI_ADD_F32:
            ep.out_f32[(int64_t)m * ep.ldo + n] += v;
            break;
        case EPI_KV_CACHE: {
            int slot = ep.row_seq ? ep.row_seq[m] : 0;
            int pos = ep.row_pos ? ep.row_pos[m] : ep.seq_len[slot] + m;
            if (ep.group_cols > 0) {  // the groups side by side in one product
                grp = n / ep.group_cols;
                n -= grp * ep.group_cols;
            }
            cache_store(ep, slot, pos, n, v, grp);
            break;
        }
        case EPI_QKV:
            epi_qkv(ep, m, n, v);
            break;
        default:
            break;
    }
}

// epi_one for a kernel instance compiled for one epilogue kind (EK >= 0; EK < 0: the kind of ep),
// so that the instance carries only that kind's code.
template <int EK>
__device__ __forceinline__ void epi_one_k(const EpiParams& ep, int m, int n, float v) {
    if constexpr (EK == EPI_STORE_F32) ep.out_f32[(int64_t)m * ep.ldo + n] = v;
    else if constexpr (EK == EPI_ADD_F32) ep.out_f32[(int64_t)m * ep.ldo + n] += v;
    else if constexpr (EK == EPI_QKV) epi_qkv(ep, m, n, v);
    else if constexpr (EK < 0) epi_one(ep, m, n, v);
}

// epi_one_k with the group of a grouped launch (EPI_KV_CACHE).
template <int EK>
__device__ __forceinline__ void epi_one_kg(const EpiParams& ep, int m, int n, float v, int grp) {
    if constexpr (EK == EPI_STORE_F32 || EK == EPI_ADD_F32 || EK == EPI_QKV) epi_one_k<EK>(ep, m, n, v);
    else epi_one(ep, m, n, v, grp);
}

// A (gate, up) column pair of EPI_SWIGLU: columns 2f and 2f+1 give output f.
__device__ __forceinline__ void epi_pair(const EpiParams& ep, int m, int n_even, float g, float u) {
    float h = act_fn(ep.act, g) * u;
    int64_t off = (int64_t)m * ep.ld_act + (n_even >> 1);
    if (ep.act_dtype == DT_BF16)
        reinterpret_cast<bf16*>(ep.out_act)[off] = __float2bfloat16_rn(h);
    else
        reinterpret_cast<float*>(ep.out_act)[off] = h;
}

// 32 consecutive columns [n, n + 32) of row m (n a multiple of 32), with
// 16-byte vector stores where the layout allows; falls back to one element at
// a time at the right edge or for unaligned leading dimensions.
__device__ __forceinline__ void store_bf16x32(bf16* dst, const float* v) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 p = __floats2bfloat162_rn(v[8 * q + 2 * i], v[8 * q + 2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t*>(&p);
        }
        d4[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}
__device__ __forceinline__ void store_f32x32(float* dst, const float* v) {
    float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int q = 0; q < 8; ++q) d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

__device__ __forceinline__ void cache_store32(const EpiParams& ep, int slot, int pos, int c, const float* v,
                                              int grp = 0) {
    if (pos < 0 || pos >= ep.max_rows) return;
    const int w = ep.d_kv ? ep.d_kv : ep.d;
    const int64_t off = grp * ep.group_stride + (int64_t)slot * ep.seq_stride + (c >= w ? ep.kv_off : 0) +
                        (int64_t)pos * w + (c >= w ? c - w : c);
    if (ep.cache_dtype == DT_BF16) store_bf16x32(reinterpret_cast<bf16*>(ep.cache) + off, v);
    else store_f32x32(reinterpret_cast<float*>(ep.cache) + off, v);
}

// EPI_MARKOV_T for one warp: lane l holds the accumulators of vocabulary row
// `vrow` (valid: vrow < V) for sequences nb .. nb+31 (those >= N are absent).
// Adds the base logits (consecutive lanes read consecutive entries of a U row),
// stores the logits if asked, then a reduce-scatter over the lanes (5 exchange
// steps, halving the columns each time) leaves in lane l the best of the
// warp's 32 rows for sequence nb + l: larger value, then lower index.  Called
// by all 32 lanes; vrow - lane is the warp's first row, a multiple of 32.
// Reduce-scatter over the warp's lanes (5 exchange steps, halving the columns each time): lane l
// holds the best of the 32 lanes' column-l entries in val[0] / idx[0] (larger value, then lower
// index).  Called by all 32 lanes.
__device__ __forceinline__ void markov_reduce_scatter(float* val, int* idx) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
        const bool upper = (lane & w) != 0;  // keep columns [w, 2w), else [0, w)
#pragma unroll
        for (int i = 0; i < w; ++i) {
            const float sv = upper ? val[i] : val[i + w];
            const int si = upper ? idx[i] : idx[i + w];
            float kv = upper ? val[i + w] : val[i];
            int ki = upper ? idx[i + w] : idx[i];
            const float ov = __shfl_xor_sync(0xffffffffu, sv, w);
            const int oi = __shfl_xor_sync(0xffffffffu, si, w);
            if (better(ov, oi, kv, ki)) {
                kv = ov;
                ki = oi;
            }
            val[i] = kv;
            idx[i] = ki;
        }
    }
}

// The base logits of markov_t32: u[j] = U[(nb + j) * gamma + k][vrow] (0 where absent).  They do not
// depend on the accumulators, so a caller may issue them before the accumulators are ready.
__device__ __forceinline__ void markov_u32_load(const EpiParams& ep, int vrow, bool valid, int nb, int N, float* u) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const bool ok = valid && nb + j < N;
        const int64_t row = (int64_t)(nb + j) * ep.gamma + ep.mk_k;
        u[j] = ok ? __ldcs(ep.mk_U + row * ep.ldo + vrow) : 0.f;
    }
}

// markov_t32 with the base logits already loaded (u from markov_u32_load).
__device__ __forceinline__ void markov_t32_u(const EpiParams& ep, int vrow, bool valid, int nb, int N, const float* acc,
                                             const float* u);

__device__ __forceinline__ void markov_t32(const EpiParams& ep, int vrow, bool valid, int nb, int N, const float* acc) {
    // all 32 loads first: a logits store between them would have to wait for
    // the load before it (the compiler cannot rule out that the buffers overlap)
    float u[32];
    markov_u32_load(ep, vrow, valid, nb, N, u);
    markov_t32_u(ep, vrow, valid, nb, N, acc, u);
}

__device__ __forceinline__ void markov_t32_u(const EpiParams& ep, int vrow, bool valid, int nb, int N, const float* acc,
                                             const float* u) {
    const int lane = threadIdx.x & 31;
    float val[32];
    int idx[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const bool ok = valid && nb + j < N;
        val[j] = ok ? acc[j] + u[j] : -INFINITY;
        idx[j] = ok ? vrow : INT_MAX;
    }
    if (ep.mk_logits) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (valid && nb + j < N) ep.mk_logits[((int64_t)(nb + j) * ep.gamma + ep.mk_k) * ep.ldo + vrow] = val[j];
    }
    markov_reduce_scatter(val, idx);
    if (nb + lane < N) {
        const int64_t o = (int64_t)(nb + lane) * ep.mk_nch + ((vrow - lane) >> 5);
        ep.mk_part_v[o] = val[0];
        ep.mk_part_i[o] = idx[0];
    }
}

// epi_row32 for a kernel instance compiled for one epilogue kind (EK >= 0; EK < 0: the kind of ep).
template <int EK>
__device__ __forceinline__ void epi_row32_k(const EpiParams& ep, int m, int n, int N, const float* v, int grp) {
    const int kind = EK >= 0 ? EK : ep.kind;
    const bool full = n + 32 <= N;
    switch (kind) {
        case EPI_STORE_F32:
        case EPI_ADD_F32:
            if (full && (ep.ldo & 3) == 0 && ((uintptr_t)ep.out_f32 & 15) == 0) {
                float* dst = ep.out_f32 + (int64_t)m * ep.ldo + n;
                if (kind == EPI_ADD_F32) {
                    float t[32];
                    const float4* s4 = reinterpret_cast<const float4*>(dst);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 a = s4[q];
                        t[4 * q] = a.x + v[4 * q];
                        t[4 * q + 1] = a.y + v[4 * q + 1];
                        t[4 * q + 2] = a.z + v[4 * q + 2];
                        t[4 * q + 3] = a.w + v[4 * q + 3];
                    }
                    store_f32x32(dst, t);
                } else {
                    store_f32x32(dst, v);
                }
                return;
            }
            break;
        case EPI_KV_CACHE:
            // 32 columns never straddle K and V when the cache row width is a multiple of 32
            if (full && ep.group_cols == 0 && (ep.d & 31) == 0 && ((ep.d_kv ? ep.d_kv : ep.d) & 31) == 0 &&
                ((uintptr_t)ep.cache & 15) == 0) {
                const int slot = ep.row_seq ? ep.row_seq[m] : 0;
                const int pos = ep.row_pos ? ep.row_pos[m] : ep.seq_len[slot] + m;
                cache_store32(ep, slot, pos, n, v, grp);
                return;
            }
            break;
        case EPI_QKV:
            if (full && (ep.d & 31) == 0 && ((ep.d_kv ? ep.d_kv : ep.d) & 31) == 0 && ((uintptr_t)ep.cache & 15) == 0) {
                if (n < ep.d) {
                    if ((ep.ldo & 3) == 0 && ((uintptr_t)ep.out_f32 & 15) == 0) {
                        store_f32x32(ep.out_f32 + (int64_t)m * ep.ldo + n, v);
                        return;
                    }
                    break;
                }
                const int b = m / ep.gamma, j = m - b * ep.gamma;
                const int slot = ep.seq_ids ? ep.seq_ids[b] : b;
                if (slot >= 0) cache_store32(ep, slot, ep.seq_len[slot] + j, n - ep.d, v);
                return;
            }
            break;
        case EPI_SWIGLU:
            if (full && (ep.ld_act & 15) == 0 && ((uintptr_t)ep.out_act & 15) == 0) {
                float h[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) h[i] = act_fn(ep.act, v[2 * i]) * v[2 * i + 1];
                const int64_t off = (int64_t)m * ep.ld_act + (n >> 1);
                if (ep.act_dtype == DT_BF16) {
                    uint4* d4 = reinterpret_cast<uint4*>(reinterpret_cast<bf16*>(ep.out_act) + off);
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        uint32_t w[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            __nv_bfloat162 p = __floats2bfloat162_rn(h[8 * q + 2 * i], h[8 * q + 2 * i + 1]);
                            w[i] = *reinterpret_cast<uint32_t*>(&p);
                        }
                        d4[q] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                } else {
                    float4* d4 = reinterpret_cast<float4*>(reinterpret_cast<float*>(ep.out_act) + off);
#pragma unroll
                    for (int q = 0; q < 4; ++q) d4[q] = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
                }
                return;
            }
            break;
        default:
            return;
    }
    // unrolled so that v stays in registers
    if (kind == EPI_SWIGLU) {
#pragma unroll
        for (int j = 0; j < 32; j += 2)
            if (n + j + 1 < N) epi_pair(ep, m, n + j, v[j], v[j + 1]);
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (n + j < N) epi_one_kg<EK>(ep, m, n + j, v[j], grp);
    }
}

__device__ __forceinline__ void epi_row32(const EpiParams& ep, int m, int n, int N, const float* v, int grp = 0) {
    epi_row32_k<-1>(ep, m, n, N, v, grp);
}

}  // namespace dspark
