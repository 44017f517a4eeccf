// GEMM epilogues shared by the SIMT, weight-streaming and tensor-core GEMMs.
#pragma once

#include "common.cuh"
#include "kernels.cuh"

namespace dspark {

__device__ __forceinline__ float act_fn(int act, float g) {
    if (act == 0) return g / (1.f + expf(-g));  // SiLU
    const float c = 0.7978845608028654f;        // sqrt(2/pi)
    return 0.5f * g * (1.f + tanhf(c * (g + 0.044715f * g * g * g)));
}

__device__ __forceinline__ void cache_store(const EpiParams& ep, int slot, int pos, int c, float v) {
    if (pos < 0 || pos >= ep.max_rows) return;
    int64_t off = (int64_t)slot * ep.seq_stride + (c >= ep.d ? ep.kv_off : 0) + (int64_t)pos * ep.d + (c % ep.d);
    if (ep.cache_dtype == DT_BF16)
        reinterpret_cast<bf16*>(ep.cache)[off] = __float2bfloat16_rn(v);
    else
        reinterpret_cast<float*>(ep.cache)[off] = v;
}

// One output element (every kind except EPI_SWIGLU).
__device__ __forceinline__ void epi_one(const EpiParams& ep, int m, int n, float v) {
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
            cache_store(ep, slot, pos, n, v);
            break;
        }
        case EPI_QKV: {
            if (n < ep.d) {
                ep.out_f32[(int64_t)m * ep.ldo + n] = v;
            } else {
                int b = m / ep.gamma, j = m - b * ep.gamma;
                int slot = ep.seq_ids ? ep.seq_ids[b] : b;
                if (slot >= 0) cache_store(ep, slot, ep.seq_len[slot] + j, n - ep.d, v);
            }
            break;
        }
        default:
            break;
    }
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

}  // namespace dspark
