// Block attention of a draft layer ("module-dflash.ts", #layer: the gamma
// block queries attend bidirectionally over [context ++ block], scale
// head_dim^-1/2, no mask).  The block's own K/V rows have already been written
// to the cache right after the context (rows len .. len+gamma-1), so every key
// is a cache row.
//
// Split-K flash decoding in one launch: the keys of one (sequence, head) are
// cut into n_chunks ranges, one CTA each ("attention" pass of
// "src/dspark-runtime.js", propose, with its partial/md buffers).  A CTA
// streams its range in 64-key tiles through a cp.async double buffer (bf16 or
// fp32 rows, 16-byte padded so the shared-memory reads are conflict-free), and
// keeps a running (max, sum, unnormalised output) per query in fp32.  The last
// CTA of a (sequence, head) - found with a ticket counter, no spinning - merges
// the ranges ("combine" pass) in a fixed order and writes the output.
//
// Work split per 64-key tile (256 threads):
//   scores   thread = (key pair, 8-element interleaved slice of head_dim): 2 keys
//            x gamma queries in registers, 3-step shuffle reduction over slices;
//   softmax  warp = query: running max/sum over the tile with warp shuffles;
//   P.V      thread = (query, 8 consecutive head_dim elements): 16-byte V reads.
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"

namespace dspark {

namespace {

constexpr int TK = 64;     // keys per tile
constexpr int NT = 256;    // threads per CTA
constexpr int GMAX = 16;   // largest block size
constexpr int HMAX = 256;  // largest head dim
constexpr int CMAX = 64;   // largest number of key ranges per (sequence, head)

template <typename TC>
struct Layout {
    int hd, gamma;
    int row_bytes;  // padded shared-memory row of a K or V tile
    __host__ __device__ Layout(int hd_, int g_) : hd(hd_), gamma(g_), row_bytes(hd_ * (int)sizeof(TC) + 16) {}
    __host__ __device__ int tile_bytes() const { return TK * row_bytes; }
    // [K0 V0 K1 V1] tiles, then Q [gamma][hd] fp32, S [gamma][TK] fp32, then per-query state and merge weights
    __host__ __device__ int q_off() const { return 4 * tile_bytes(); }
    __host__ __device__ int s_off() const { return q_off() + gamma * hd * 4; }
    __host__ __device__ int st_off() const { return s_off() + gamma * TK * 4; }
    __host__ __device__ int w_off() const { return st_off() + 3 * GMAX * 4; }
    __host__ __device__ int bytes() const { return w_off() + GMAX * CMAX * 4 + 16; }
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Issue the copies of keys [t0, t0 + TK) (rows at or beyond `end` are zero-filled) into tile buffers.
template <typename TC>
__device__ __forceinline__ void load_tile(uint8_t* ksm, uint8_t* vsm, const TC* Kb, const TC* Vb, int64_t row_stride,
                                          int t0, int end, const Layout<TC>& L) {
    const int vec_per_row = L.hd * (int)sizeof(TC) / 16;
    const uint32_t kbase = (uint32_t)__cvta_generic_to_shared(ksm), vbase = (uint32_t)__cvta_generic_to_shared(vsm);
    for (int i = threadIdx.x; i < TK * vec_per_row; i += NT) {
        const int r = i / vec_per_row, v = i - r * vec_per_row;
        const int key = t0 + r;
        const bool ok = key < end;
        const int64_t off = (int64_t)(ok ? key : t0) * row_stride + v * (16 / (int)sizeof(TC));
        const uint32_t so = r * L.row_bytes + v * 16;
        cp_async16(kbase + so, Kb + off, ok ? 16 : 0);
        cp_async16(vbase + so, Vb + off, ok ? 16 : 0);
    }
}

template <typename TC>
__device__ __forceinline__ void unpack8(const uint8_t* p, float* f) {
    if (sizeof(TC) == 2) {
        Vec16<bf16>::unpack(*reinterpret_cast<const uint4*>(p), f);
    } else {
        Vec16<float>::unpack(*reinterpret_cast<const uint4*>(p), f);
        Vec16<float>::unpack(*reinterpret_cast<const uint4*>(p + 16), f + 4);
    }
}

template <typename TC, typename TO>
__global__ void __launch_bounds__(NT) k_attention(AttnParams p) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) uint8_t sm[];
    const int gamma = p.gamma, d = p.d, hd = d / p.n_heads;
    const Layout<TC> L(hd, gamma);
    float* Q = reinterpret_cast<float*>(sm + L.q_off());
    float* S = reinterpret_cast<float*>(sm + L.s_off());
    float* m_run = reinterpret_cast<float*>(sm + L.st_off());
    float* l_run = m_run + GMAX;
    float* alpha = l_run + GMAX;
    float* Wm = reinterpret_cast<float*>(sm + L.w_off());
    __shared__ int is_last;

    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int slot = p.seq_ids ? p.seq_ids[b] : b;
    const int n_keys = slot < 0 ? 0 : p.seq_len[slot] + gamma;  // a rejected sequence has no keys
    const int chunk = (n_keys + p.n_chunks - 1) / p.n_chunks;
    const int start = min(n_keys, c * chunk), end = min(n_keys, start + chunk);

    // K/V head of query head h and the cache row width (grouped-query attention)
    const int dkv = p.d_kv ? p.d_kv : d;
    const int kvh = p.n_kv_heads ? h / (p.n_heads / p.n_kv_heads) : h;
    const TC* Kb = reinterpret_cast<const TC*>(p.cache) + (int64_t)max(slot, 0) * p.seq_stride + kvh * hd;
    const TC* Vb = Kb + p.kv_off;
    if (start < end) load_tile<TC>(sm, sm + L.tile_bytes(), Kb, Vb, dkv, start, end, L);
    cp_async_commit();

    const float scale = rsqrtf((float)hd);
    for (int i = tid; i < gamma * hd; i += NT) {
        const int j = i / hd, e = i - j * hd;
        Q[i] = p.q[(int64_t)(b * gamma + j) * d + h * hd + e] * scale;
    }
    if (tid < GMAX) {
        m_run[tid] = -INFINITY;
        l_run[tid] = 0.f;
    }
    // P.V ownership: 8 consecutive head_dim elements of one query
    const int ng = hd / 8;
    const int pv_eg = tid % ng, pv_j = tid / ng;
    float o[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) o[u] = 0.f;
    // score ownership: key pair kp, interleaved slice sl (groups of 8 head_dim elements g = sl, sl+8, ...)
    const int kp = tid >> 3, sl = tid & 7;

    int buf = 0;
    for (int t0 = start; t0 < end; t0 += TK) {
        const int nk = min(TK, end - t0);
        if (t0 + TK < end) {
            uint8_t* nxt = sm + (buf ^ 1) * 2 * L.tile_bytes();
            load_tile<TC>(nxt, nxt + L.tile_bytes(), Kb, Vb, dkv, t0 + TK, end, L);
        }
        cp_async_commit();
        cp_async_wait_1();
        __syncthreads();
        const uint8_t* Ks = sm + buf * 2 * L.tile_bytes();
        const uint8_t* Vs = Ks + L.tile_bytes();
        // ---- scores S[j][key] for keys 2kp, 2kp+1
        {
            float acc[GMAX][2];
#pragma unroll
            for (int j = 0; j < GMAX; ++j) acc[j][0] = acc[j][1] = 0.f;
            for (int g = sl; g < ng; g += 8) {
                float k0[8], k1[8];
                unpack8<TC>(Ks + (2 * kp) * L.row_bytes + g * 8 * sizeof(TC), k0);
                unpack8<TC>(Ks + (2 * kp + 1) * L.row_bytes + g * 8 * sizeof(TC), k1);
#pragma unroll
                for (int j = 0; j < GMAX; ++j) {
                    if (j >= gamma) break;
                    const float4 qa = *reinterpret_cast<const float4*>(Q + j * hd + g * 8);
                    const float4 qb = *reinterpret_cast<const float4*>(Q + j * hd + g * 8 + 4);
                    const float q[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        acc[j][0] = fmaf(q[u], k0[u], acc[j][0]);
                        acc[j][1] = fmaf(q[u], k1[u], acc[j][1]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < GMAX; ++j) {
                if (j >= gamma) break;
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    float v = acc[j][x];
                    v += __shfl_xor_sync(0xffffffffu, v, 1);
                    v += __shfl_xor_sync(0xffffffffu, v, 2);
                    v += __shfl_xor_sync(0xffffffffu, v, 4);
                    acc[j][x] = v;
                }
                if (sl == (j & 7)) {
                    S[j * TK + 2 * kp] = (2 * kp < nk) ? acc[j][0] : -INFINITY;
                    S[j * TK + 2 * kp + 1] = (2 * kp + 1 < nk) ? acc[j][1] : -INFINITY;
                }
            }
        }
        __syncthreads();
        // ---- online softmax, one warp per query
        for (int j = warp; j < gamma; j += NT / 32) {
            const float s0 = S[j * TK + 2 * lane], s1 = S[j * TK + 2 * lane + 1];
            const float mt = warp_max(fmaxf(s0, s1));
            const float m_old = m_run[j];
            const float m_new = fmaxf(m_old, mt);
            const float p0 = __expf(s0 - m_new), p1 = __expf(s1 - m_new);  // exp(-inf) = 0 for padded keys
            const float sum = warp_sum(p0 + p1);
            S[j * TK + 2 * lane] = p0;
            S[j * TK + 2 * lane + 1] = p1;
            if (lane == 0) {
                const float a = (m_old == -INFINITY) ? 0.f : __expf(m_old - m_new);
                alpha[j] = a;
                l_run[j] = l_run[j] * a + sum;
                m_run[j] = m_new;
            }
        }
        __syncthreads();
        // ---- O[j][eg*8 .. +8] = alpha O + sum_key P[j][key] V[key]
        if (pv_j < gamma) {
            const float a = alpha[pv_j];
#pragma unroll
            for (int u = 0; u < 8; ++u) o[u] *= a;
            const float* pr = S + pv_j * TK;
            for (int key = 0; key < nk; ++key) {
                float v[8];
                unpack8<TC>(Vs + key * L.row_bytes + pv_eg * 8 * sizeof(TC), v);
                const float pk = pr[key];
#pragma unroll
                for (int u = 0; u < 8; ++u) o[u] = fmaf(pk, v[u], o[u]);
            }
        }
        buf ^= 1;
        __syncthreads();  // every thread is done with this buffer before it is refilled
    }
    cp_async_wait_0();
    __syncthreads();

    // ---- this range's partial: (m, l, o[hd]) per query; rows are hd + 2 floats (8-byte aligned)
    const int w = hd + 2;
    const int64_t bh = (int64_t)b * p.n_heads + h;
    float* base = p.part + (bh * p.n_chunks + c) * gamma * w;
    if (pv_j < gamma) {
        float2* d2 = reinterpret_cast<float2*>(base + pv_j * w + 2 + pv_eg * 8);
        d2[0] = make_float2(o[0], o[1]);
        d2[1] = make_float2(o[2], o[3]);
        d2[2] = make_float2(o[4], o[5]);
        d2[3] = make_float2(o[6], o[7]);
    }
    if (tid < gamma) {
        base[tid * w] = m_run[tid];
        base[tid * w + 1] = l_run[tid];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) is_last = (atomicAdd(&p.tickets[bh], 1u) == (unsigned int)p.n_chunks - 1);
    __syncthreads();
    if (!is_last) return;
    __threadfence();

    // ---- last CTA of (b, h): merge the n_chunks ranges in order
    const float* all = p.part + bh * p.n_chunks * gamma * w;
    for (int j = warp; j < gamma; j += NT / 32) {
        float M = -INFINITY;
        for (int cc = lane; cc < p.n_chunks; cc += 32) M = fmaxf(M, __ldcg(all + ((int64_t)cc * gamma + j) * w));
        M = warp_max(M);
        float Lsum = 0.f;
        for (int cc = lane; cc < p.n_chunks; cc += 32) {
            const float mc = __ldcg(all + ((int64_t)cc * gamma + j) * w);
            const float lc = __ldcg(all + ((int64_t)cc * gamma + j) * w + 1);
            Lsum += (mc == -INFINITY) ? 0.f : __expf(mc - M) * lc;
        }
        Lsum = warp_sum(Lsum);
        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
        for (int cc = lane; cc < p.n_chunks; cc += 32) {
            const float mc = __ldcg(all + ((int64_t)cc * gamma + j) * w);
            Wm[j * CMAX + cc] = (mc == -INFINITY) ? 0.f : __expf(mc - M) * inv;
        }
    }
    __syncthreads();
    if (pv_j < gamma) {
        float acc[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u] = 0.f;
        const float* wj = Wm + pv_j * CMAX;
        int cc = 0;
        for (; cc + 2 <= p.n_chunks; cc += 2) {
            const float2* s0 = reinterpret_cast<const float2*>(all + ((int64_t)cc * gamma + pv_j) * w + 2 + pv_eg * 8);
            const float2* s1 =
                reinterpret_cast<const float2*>(all + ((int64_t)(cc + 1) * gamma + pv_j) * w + 2 + pv_eg * 8);
            float2 a[4], bb[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                a[q] = __ldcg(s0 + q);
                bb[q] = __ldcg(s1 + q);
            }
            const float w0 = wj[cc], w1 = wj[cc + 1];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc[2 * q] = fmaf(w1, bb[q].x, fmaf(w0, a[q].x, acc[2 * q]));
                acc[2 * q + 1] = fmaf(w1, bb[q].y, fmaf(w0, a[q].y, acc[2 * q + 1]));
            }
        }
        for (; cc < p.n_chunks; ++cc) {
            const float2* s0 = reinterpret_cast<const float2*>(all + ((int64_t)cc * gamma + pv_j) * w + 2 + pv_eg * 8);
            const float w0 = wj[cc];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 a = __ldcg(s0 + q);
                acc[2 * q] = fmaf(w0, a.x, acc[2 * q]);
                acc[2 * q + 1] = fmaf(w0, a.y, acc[2 * q + 1]);
            }
        }
        TO* out = reinterpret_cast<TO*>(p.out) + (int64_t)(b * gamma + pv_j) * d + h * hd + pv_eg * 8;
#pragma unroll
        for (int u = 0; u < 8; ++u) out[u] = from_f32<TO>(acc[u]);
    }
    if (tid == 0) p.tickets[bh] = 0u;
}

int g_smem_limit = 0;  // largest dynamic shared memory the kernels may request on this device

template <typename TC, typename TO>
cudaError_t set_attr() {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, k_attention<TC, TO>);
    if (e != cudaSuccess) return e;
    int dev = 0, optin = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
    const int limit = optin - (int)fa.sharedSizeBytes;
    g_smem_limit = limit;
    const int sm = Layout<TC>(HMAX, GMAX).bytes();
    return cudaFuncSetAttribute(k_attention<TC, TO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                sm < limit ? sm : limit);
}

}  // namespace

size_t attn_scratch_floats(int B, int n_heads, int n_chunks, int gamma, int head_dim) {
    // partial rows of head_dim + 2 floats (SIMT kernel) or head_dim + 4 (tensor-core kernel)
    return (size_t)B * n_heads * n_chunks * gamma * (head_dim + 4);
}

int attn_max_chunks(int cache_dtype, int head_dim, int gamma) {
    return attention_tc_ok(cache_dtype, head_dim, gamma) ? attention_tc_max_chunks() : CMAX;
}

cudaError_t attention_init() {
    cudaError_t e;
    if ((e = attention_tc_init()) != cudaSuccess) return e;
    if ((e = set_attr<bf16, bf16>()) != cudaSuccess) return e;
    if ((e = set_attr<bf16, float>()) != cudaSuccess) return e;
    if ((e = set_attr<float, bf16>()) != cudaSuccess) return e;
    return set_attr<float, float>();
}

cudaError_t attention(const AttnParams& p, cudaStream_t st) {
    const int hd = p.d / p.n_heads;
    if (attention_tc_ok(p.cache_dtype, hd, p.gamma)) return attention_tc(p, st);
    if (p.gamma > GMAX || hd > HMAX || hd % 8 != 0 || p.n_chunks < 1 || p.n_chunks > CMAX || NT % (hd / 8) != 0 ||
        p.gamma > NT / (hd / 8))
        return cudaErrorInvalidValue;
    const int need = p.cache_dtype == DT_BF16 ? Layout<bf16>(hd, p.gamma).bytes() : Layout<float>(hd, p.gamma).bytes();
    if (need > g_smem_limit) return cudaErrorInvalidValue;
    dim3 grid(p.n_chunks, p.n_heads, p.B);
    if (p.cache_dtype == DT_BF16) {
        const size_t sm = Layout<bf16>(hd, p.gamma).bytes();
        if (p.out_dtype == DT_BF16) launch(k_attention<bf16, bf16>, grid, NT, sm, st, p);
        else launch(k_attention<bf16, float>, grid, NT, sm, st, p);
    } else {
        const size_t sm = Layout<float>(hd, p.gamma).bytes();
        if (p.out_dtype == DT_BF16) launch(k_attention<float, bf16>, grid, NT, sm, st, p);
        else launch(k_attention<float, float>, grid, NT, sm, st, p);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace dspark
