// Sampling form of the Markov chain's token choice ("module-dflash.ts", forwardInfer:
// processLogits + sampleToken with a KeyStream; "src/dspark-runtime.js", propose: the
// temperature > 0 branch that keeps 64 or 256 candidates).  The pages name a temperature,
// a top-k and a seeded key stream but define none of them; the reading implemented here:
//   candidates = the top_k largest logits of the position (ties to the lower index), or
//                the whole vocabulary when top_k = 0;
//   token      = argmax over the candidates of l_v / t + g_v, g_v = -ln(-ln u_v)
//                (the Gumbel-max rule: an exact draw from softmax(l / t) over them);
//   u_v        = (floor(z / 2^40) + 0.5) / 2^24, z the (c + 1)-th SplitMix64 output
//                (Steele, Lea and Flood, 2014) of the stream seeded with `seed`,
//                c = slot * 2^48 + (draw mod 2^24) * 2^24 + v, draw = the slot's draw
//                counter + k (the counter advances by gamma per draft call).
// Two launches per block position:
//   k_sample_logits: CTAs over the vocabulary compute l = U_k + w2 . w1[prev], write the
//     logits, and publish either their best Gumbel key (top_k = 0) or their own top_k
//     logits as 64-bit words (order-preserving float bits << 32 | ~index), found by the
//     same radix select;
//   k_sample_pick: one CTA per sequence gathers the words, finds the top_k-th largest by
//     an 8-pass radix select (the union of the CTAs' lists holds the global top_k), draws
//     among the words at or above it, and writes the token and the confidence.
#include <climits>
#include <stdint.h>
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"

namespace dspark {

namespace {

constexpr int NT_L = 512;        // k_sample_logits threads
constexpr int NT_P = 1024;       // k_sample_pick threads
constexpr int LPR_S = 4;         // lanes per vocabulary row
constexpr int RPW_S = 32 / LPR_S;
constexpr int RMAX_S = 1024;     // largest Markov rank
constexpr int ROWS_MAX = 2048;   // vocabulary rows per CTA (the local selection's size)
constexpr int TOPK_MAX = 64;
constexpr int MAX_CTAS = 256;

__device__ __forceinline__ uint32_t order_bits(float v) {
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float order_value(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}
__device__ __forceinline__ unsigned long long word_of(float v, int i) {
    return ((unsigned long long)order_bits(v) << 32) | (unsigned long long)(~(uint32_t)i);
}

// The Gumbel noise of vocabulary entry v for draw `draw` of sequence slot `slot`.
__device__ __forceinline__ float gumbel_noise(unsigned long long seed, uint32_t slot, uint32_t draw, uint32_t v) {
    const unsigned long long c = ((unsigned long long)(slot & 0xffffu) << 48) |
                                 ((unsigned long long)(draw & 0xffffffu) << 24) | (unsigned long long)(v & 0xffffffu);
    unsigned long long z = seed + (c + 1ull) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    const float u = ((float)(uint32_t)(z >> 40) + 0.5f) * (1.0f / 16777216.0f);
    return -logf(-logf(u));
}

__device__ __forceinline__ unsigned long long warp_max64(unsigned long long w) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long x = __shfl_xor_sync(0xffffffffu, w, o);
        w = x > w ? x : w;
    }
    return w;
}

// Largest word over the block; every thread gets it.  `red` holds >= 32 words.
__device__ __forceinline__ unsigned long long block_max64(unsigned long long w, unsigned long long* red) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    w = warp_max64(w);
    __syncthreads();
    if (lane == 0) red[wid] = w;
    __syncthreads();
    unsigned long long t = lane < nw ? red[lane] : 0ull;
    return warp_max64(t);
}

struct KthShared {
    unsigned int hist[256];
    unsigned long long prefix;
    unsigned int rem;
    int count;
    int done;
};

// The K-th largest of the nonzero words w[0, n) (they are distinct), for the whole block;
// 1 when there are no more than K of them.  MSB-first radix select on 8-bit digits; it
// stops once every word under the chosen prefix is wanted.
__device__ unsigned long long block_kth_word(const unsigned long long* w, int n, int K, KthShared& ks) {
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        ks.prefix = 0ull;
        ks.rem = (unsigned int)K;
        ks.count = 0;
        ks.done = 0;
    }
    __syncthreads();
    int nz = 0;
    for (int i = tid; i < n; i += nt) nz += w[i] != 0ull;
    nz = __reduce_add_sync(0xffffffffu, nz);
    if (lane == 0 && nz) atomicAdd(&ks.count, nz);
    __syncthreads();
    if (ks.count <= K) return 1ull;
    unsigned long long mask = 0ull;
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += nt) ks.hist[i] = 0u;
        __syncthreads();
        const unsigned long long prefix = ks.prefix;
        // block-uniform trip count, so that every lane takes part in the match; the lanes of a
        // warp that fall in the same bin add once (the high digits crowd into few bins)
        for (int i0 = 0; i0 < n; i0 += nt) {
            const int i = i0 + tid;
            const unsigned long long x = i < n ? w[i] : 0ull;
            const bool in = x != 0ull && (x & mask) == prefix;
            const uint32_t bin = in ? ((uint32_t)(x >> shift) & 255u) : 256u;
            const uint32_t peers = __match_any_sync(0xffffffffu, bin);
            if (in && lane == __ffs(peers) - 1) atomicAdd(&ks.hist[bin], (unsigned int)__popc(peers));
        }
        __syncthreads();
        if (warp == 0) {
            // lane l holds digits 255 - 8l down to 248 - 8l; find where the count from the top
            // reaches the rank still wanted
            unsigned int h8[8], loc = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                h8[q] = ks.hist[255 - 8 * lane - q];
                loc += h8[q];
            }
            unsigned int incl = loc;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned int t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            const unsigned int rem = ks.rem, excl = incl - loc;
            const unsigned int hit = __ballot_sync(0xffffffffu, excl < rem && rem <= incl);
            if (hit != 0u && lane == __ffs(hit) - 1) {
                unsigned int cum = excl, hq = 0;
                int qs = 7;
                bool found = false;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (!found && cum + h8[q] >= rem) {
                        qs = q;
                        hq = h8[q];
                        found = true;
                    } else if (!found) {
                        cum += h8[q];
                    }
                }
                ks.prefix = prefix | ((unsigned long long)(255 - 8 * lane - qs) << shift);
                ks.rem = rem - cum;
                ks.done = (hq == rem - cum);  // every word under the new prefix is wanted
            }
        }
        mask |= 0xffull << shift;
        __syncthreads();
        if (ks.done) break;
    }
    return ks.prefix;
}

__device__ __forceinline__ int sample_prev(const SampleParams& p, int b) {
    const int prev = p.k == 0 ? (p.anchors ? p.anchors[b] : p.anchor) : p.tokens[b * p.gamma + p.k - 1];
    return min(max(prev, 0), p.V - 1);
}

// The sequence's slot (its draw counter); an out-of-range id is reported and mapped to slot 0.
__device__ __forceinline__ uint32_t sample_slot(const SampleParams& p, int b) {
    const int s = p.seq_ids ? p.seq_ids[b] : b;
    if (s < 0 || s >= p.n_slots) {
        if (threadIdx.x == 0) atomicOr(p.err, 2);  // a sequence id outside [0, max_seqs)
        return 0u;
    }
    return (uint32_t)s;
}

template <typename TW>
__global__ void __launch_bounds__(NT_L) k_sample_logits(SampleParams p) {
    pdl_wait();
    pdl_trigger();
    constexpr int VE = Vec16<TW>::N;
    __shared__ __align__(16) float e[RMAX_S];
    __shared__ unsigned long long keys[ROWS_MAX];
    __shared__ unsigned long long red[32];
    __shared__ KthShared ks;
    __shared__ int n_out;

    const int b = blockIdx.y, k = p.k, r = p.r, V = p.V, K = p.top_k;
    const int prev = sample_prev(p, b);
    const uint32_t slot = sample_slot(p, b);
    const uint32_t draw = p.draws[slot] + (uint32_t)k;
    const TW* w1 = reinterpret_cast<const TW*>(p.w1);
    const TW* w2 = reinterpret_cast<const TW*>(p.w2);
    for (int c = threadIdx.x; c < r; c += NT_L) e[c] = to_f32(w1[(int64_t)prev * r + c]);

    const int rows = (V + gridDim.x - 1) / gridDim.x;
    const int v_begin = blockIdx.x * rows, v_end = min(V, v_begin + rows);
    const int nrows = max(0, v_end - v_begin);
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane & (LPR_S - 1), rw = lane / LPR_S;
    const int64_t urow = (int64_t)(b * p.gamma + k) * V;
    const int nvec = r / VE;
    unsigned long long zbest = 0ull;
    // two rows per lane group per pass, eight 16-byte chunks of each requested before any is used
    constexpr int QL = 8;
    for (int v0 = v_begin + warp * (2 * RPW_S); v0 < v_end; v0 += (NT_L / 32) * (2 * RPW_S)) {
        int vr[2] = {v0 + rw, v0 + RPW_S + rw};
        float acc[2] = {0.f, 0.f};
        for (int x0 = sub; x0 < nvec; x0 += QL * LPR_S) {
            uint4 u[2][QL];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const TW* row = w2 + (int64_t)min(vr[h], v_end - 1) * r;
#pragma unroll
                for (int q = 0; q < QL; ++q) {
                    const int x = x0 + q * LPR_S;
                    u[h][q] = x < nvec ? __ldg(reinterpret_cast<const uint4*>(row + x * VE)) : make_uint4(0, 0, 0, 0);
                }
            }
#pragma unroll
            for (int q = 0; q < QL; ++q) {
                const int x = x0 + q * LPR_S;
                if (x < nvec) {
                    const float* ep = e + x * VE;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        float f[VE];
                        Vec16<TW>::unpack(u[h][q], f);
#pragma unroll
                        for (int t = 0; t < VE; ++t) acc[h] = fmaf(f[t], ep[t], acc[h]);
                    }
                }
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int o = 1; o < LPR_S; o <<= 1) acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], o);
            const int v = vr[h];
            if (sub == 0 && v < v_end) {
                const float l = p.U[urow + v] + acc[h];
                if (p.logits) p.logits[urow + v] = l;
                if (K > 0) {
                    keys[v - v_begin] = word_of(l, v);
                } else {
                    const unsigned long long zw = word_of(l / p.temperature + gumbel_noise(p.seed, slot, draw, v), v);
                    zbest = zw > zbest ? zw : zbest;
                }
            }
        }
    }
    unsigned long long* out = p.cand + ((size_t)b * gridDim.x + blockIdx.x) * p.cand_stride;
    if (K == 0) {
        const unsigned long long m = block_max64(zbest, red);
        if (threadIdx.x == 0) out[0] = m;
        return;
    }
    __syncthreads();
    // this CTA's top_k words (unordered): the ones at or above its top_k-th largest
    const unsigned long long thr = block_kth_word(keys, nrows, K, ks);
    if (threadIdx.x == 0) n_out = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < nrows; i += NT_L) {
        const unsigned long long w = keys[i];
        if (w != 0ull && w >= thr) out[atomicAdd(&n_out, 1)] = w;
    }
    __syncthreads();
    for (int j = n_out + threadIdx.x; j < K; j += NT_L) out[j] = 0ull;
}

template <typename TW>
__global__ void __launch_bounds__(NT_P) k_sample_pick(SampleParams p, int ctas) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ unsigned long long words[];  // [ctas * cand_stride]
    __shared__ KthShared ks;
    __shared__ unsigned long long red[32];
    __shared__ float redf[32];

    const int b = blockIdx.x, k = p.k, r = p.r, V = p.V;
    const int K = p.top_k;
    const int per = K > 0 ? K : 1;
    const int n = ctas * per;
    const uint32_t slot = sample_slot(p, b);
    const uint32_t draw = p.draws[slot] + (uint32_t)k;
    const unsigned long long* src = p.cand + (size_t)b * ctas * p.cand_stride;
    for (int i = threadIdx.x; i < n; i += NT_P) {
        const int c = i / per, j = i - c * per;
        words[i] = __ldcg(src + (size_t)c * p.cand_stride + j);
    }
    __syncthreads();
    unsigned long long pick = 0ull;
    if (K == 0) {
        unsigned long long m = 0ull;
        for (int i = threadIdx.x; i < n; i += NT_P) m = words[i] > m ? words[i] : m;
        pick = block_max64(m, red);
    } else {
        const unsigned long long thr = block_kth_word(words, n, K, ks);
        unsigned long long m = 0ull;
        for (int i = threadIdx.x; i < n; i += NT_P) {
            const unsigned long long w = words[i];
            if (w != 0ull && w >= thr) {
                const int v = (int)(~(uint32_t)w);
                const float l = order_value((uint32_t)(w >> 32));
                const unsigned long long zw = word_of(l / p.temperature + gumbel_noise(p.seed, slot, draw, v), v);
                m = zw > m ? zw : m;
            }
        }
        pick = block_max64(m, red);
    }
    // confidence: sigmoid(conf_w . [y_k ; w1[prev]] + conf_b)
    const int prev = sample_prev(p, b);
    const TW* w1 = reinterpret_cast<const TW*>(p.w1);
    const float* yr = p.y + (int64_t)(b * p.gamma + k) * p.d;
    float z = 0.f;
    for (int c = threadIdx.x; c < p.d; c += NT_P) z = fmaf(yr[c], p.conf_w[c], z);
    for (int c = threadIdx.x; c < r; c += NT_P) z = fmaf(to_f32(w1[(int64_t)prev * r + c]), p.conf_w[p.d + c], z);
    z = block_sum(z, redf);
    if (threadIdx.x == 0) {
        int tok = (int)(~(uint32_t)pick);
        if (pick == 0ull || !(order_value((uint32_t)(pick >> 32)) > -INFINITY) || tok < 0 || tok >= V) {
            atomicOr(p.err, 8);
            tok = 0;
        }
        p.tokens[b * p.gamma + k] = tok;
        p.conf[b * p.gamma + k] = 1.f / (1.f + expf(-(z + p.conf_w[p.d + r])));
        if (k == p.gamma - 1) p.draws[slot] += (uint32_t)p.gamma;  // every launch of this call has read it
    }
}

bool g_sample_ready = false;

}  // namespace

int sample_ctas(int V, int num_sms) {
    int c = num_sms;
    if ((V + c - 1) / c > ROWS_MAX) c = (V + ROWS_MAX - 1) / ROWS_MAX;
    return c;
}

bool sample_ok(int V, int r, int top_k, int num_sms) {
    return g_sample_ready && V >= 1 && r >= 8 && r <= RMAX_S && r % 8 == 0 && top_k >= 0 && top_k <= TOPK_MAX &&
           sample_ctas(V, num_sms) <= MAX_CTAS;
}

cudaError_t sample_init() {
    const int bytes = MAX_CTAS * TOPK_MAX * 8;
    cudaError_t e = cudaFuncSetAttribute(k_sample_pick<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_sample_pick<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    g_sample_ready = e == cudaSuccess;
    (void)cudaGetLastError();
    return cudaSuccess;
}

cudaError_t markov_sample_step(const SampleParams& p, int num_sms, cudaStream_t st) {
    if (!(p.temperature > 0.f) || !sample_ok(p.V, p.r, p.top_k, num_sms) || p.B < 1 || !p.draws || !p.cand)
        return cudaErrorInvalidValue;
    const int ctas = sample_ctas(p.V, num_sms);
    if (p.cand_stride < (p.top_k > 0 ? p.top_k : 1)) return cudaErrorInvalidValue;
    const size_t smem = (size_t)ctas * (p.top_k > 0 ? p.top_k : 1) * 8;
    if (p.w_dtype == DT_BF16) {
        launch(k_sample_logits<bf16>, dim3(ctas, p.B), NT_L, 0, st, p);
        note_launch();
        launch(k_sample_pick<bf16>, p.B, NT_P, smem, st, p, ctas);
    } else {
        launch(k_sample_logits<float>, dim3(ctas, p.B), NT_L, 0, st, p);
        note_launch();
        launch(k_sample_pick<float>, p.B, NT_P, smem, st, p, ctas);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace dspark
