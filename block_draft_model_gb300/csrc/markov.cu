// One position k of the sequential Markov chain ("module-dflash.ts",
// forwardInfer / #markov / #confidence; "src/dspark-runtime.js", propose:
// markovEmbed, markov, addBias, argmax, argmaxFinal):
//   e       = w1[prev]            prev = anchor (k = 0) or the token drafted at k-1
//   logits  = U_k + w2 e          (w2 stored [V, r], one row per vocabulary entry)
//   token_k = argmax logits       (lowest index on ties)
//   conf_k  = sigmoid(conf_w . [y_k ; e] + conf_b)
// One fused launch per position: every CTA streams a slice of w2, adds the
// base logits, keeps its best (value, index); the last CTA to finish (ticket
// counter, no spinning) reduces the CTA results, writes the token and the
// confidence, and re-arms the counter.  Four lanes share a vocabulary row (128
// bytes each for r = 256), so every load is a full 32-byte sector and a row
// needs a two-step shuffle; two rows per lane group are in flight at once.  The token stays on the
// device, where the next position's launch reads it.
#include <climits>
#include <stdint.h>
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"

namespace dspark {

namespace {

constexpr int NT = 256;
constexpr int LPR = 4;         // lanes per vocabulary row
constexpr int RPW = 32 / LPR;  // rows per warp pass
constexpr int RMAX = 1024;     // largest Markov rank

template <typename TW>
__global__ void __launch_bounds__(NT) k_markov(MarkovParams p) {
    pdl_trigger();
    pdl_wait();
    constexpr int VE = Vec16<TW>::N;
    __shared__ __align__(16) float e[RMAX];
    __shared__ float red_v[NT / 32];
    __shared__ int red_i[NT / 32];
    __shared__ int is_last;
    __shared__ float redf[32];

    const int b = blockIdx.y, k = p.k, r = p.r, V = p.V;
    int prev = (k == 0) ? (p.anchors ? p.anchors[b] : p.anchor) : p.tokens[b * p.gamma + k - 1];
    prev = min(max(prev, 0), V - 1);
    const TW* w1 = reinterpret_cast<const TW*>(p.w1);
    const TW* w2 = reinterpret_cast<const TW*>(p.w2);
    for (int c = threadIdx.x; c < r; c += NT) e[c] = to_f32(w1[(int64_t)prev * r + c]);
    __syncthreads();

    const int rows = (V + gridDim.x - 1) / gridDim.x;
    const int v_begin = blockIdx.x * rows, v_end = min(V, v_begin + rows);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane & (LPR - 1), rw = lane / LPR;
    const int64_t urow = (int64_t)(b * p.gamma + k) * V;
    const int nvec = r / VE;

    ArgBest best{-INFINITY, INT_MAX};
    // each pass: 8 rows per warp, 4 lanes per row, two passes in flight
    for (int v0 = v_begin + warp * (2 * RPW); v0 < v_end; v0 += (NT / 32) * (2 * RPW)) {
        const int va = v0 + rw, vb = v0 + RPW + rw;
        const TW* ra = w2 + (int64_t)min(va, v_end - 1) * r;
        const TW* rb = w2 + (int64_t)min(vb, v_end - 1) * r;
        float aa = 0.f, ab = 0.f;
        for (int vi = sub; vi < nvec; vi += 4 * LPR) {
            uint4 ua[4], ub[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int x = vi + q * LPR;
                ua[q] = x < nvec ? __ldg(reinterpret_cast<const uint4*>(ra + x * VE)) : make_uint4(0, 0, 0, 0);
                ub[q] = x < nvec ? __ldg(reinterpret_cast<const uint4*>(rb + x * VE)) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int x = vi + q * LPR;
                if (x >= nvec) break;
                float fa[VE], fb[VE];
                Vec16<TW>::unpack(ua[q], fa);
                Vec16<TW>::unpack(ub[q], fb);
                const float* ep = e + x * VE;
#pragma unroll
                for (int t = 0; t < VE; ++t) {
                    aa = fmaf(fa[t], ep[t], aa);
                    ab = fmaf(fb[t], ep[t], ab);
                }
            }
        }
#pragma unroll
        for (int o = 1; o < LPR; o <<= 1) {
            aa += __shfl_xor_sync(0xffffffffu, aa, o);
            ab += __shfl_xor_sync(0xffffffffu, ab, o);
        }
        if (sub == 0) {
            if (va < v_end) {
                const float l = p.U[urow + va] + aa;
                if (p.logits) p.logits[urow + va] = l;
                if (better(l, va, best.v, best.i)) {
                    best.v = l;
                    best.i = va;
                }
            }
            if (vb < v_end) {
                const float l = p.U[urow + vb] + ab;
                if (p.logits) p.logits[urow + vb] = l;
                if (better(l, vb, best.v, best.i)) {
                    best.v = l;
                    best.i = vb;
                }
            }
        }
    }
    best = warp_argbest(best);
    if (lane == 0) {
        red_v[warp] = best.v;
        red_i[warp] = best.i;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        ArgBest cb{-INFINITY, INT_MAX};
        for (int w = 0; w < NT / 32; ++w)
            if (better(red_v[w], red_i[w], cb.v, cb.i)) {
                cb.v = red_v[w];
                cb.i = red_i[w];
            }
        p.part_v[b * gridDim.x + blockIdx.x] = cb.v;
        p.part_i[b * gridDim.x + blockIdx.x] = cb.i;
        __threadfence();
        const unsigned int ticket = atomicAdd(&p.counters[b], 1u);
        is_last = (ticket == gridDim.x - 1);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // last CTA of this sequence: reduction of the CTA results (the key is a total order, so the
    // result does not depend on the order of arrival)
    ArgBest fb{-INFINITY, INT_MAX};
    for (int c = threadIdx.x; c < (int)gridDim.x; c += NT) {
        const float v = __ldcg(p.part_v + b * gridDim.x + c);
        const int i = __ldcg(p.part_i + b * gridDim.x + c);
        if (better(v, i, fb.v, fb.i)) {
            fb.v = v;
            fb.i = i;
        }
    }
    fb = warp_argbest(fb);
    if (lane == 0) {
        red_v[warp] = fb.v;
        red_i[warp] = fb.i;
    }
    // confidence: sigmoid(conf_w . [y_k ; e] + conf_b)
    const float* yr = p.y + (int64_t)(b * p.gamma + k) * p.d;
    float z = 0.f;
    for (int c = threadIdx.x; c < p.d; c += NT) z = fmaf(yr[c], p.conf_w[c], z);
    for (int c = threadIdx.x; c < r; c += NT) z = fmaf(e[c], p.conf_w[p.d + c], z);
    z = block_sum(z, redf);  // contains __syncthreads, so red_v/red_i are complete
    if (threadIdx.x == 0) {
        ArgBest tb{-INFINITY, INT_MAX};
        for (int w = 0; w < NT / 32; ++w)
            if (better(red_v[w], red_i[w], tb.v, tb.i)) {
                tb.v = red_v[w];
                tb.i = red_i[w];
            }
        int tok = tb.i;
        if (tok == INT_MAX || !(tb.v > -INFINITY)) {
            atomicOr(p.err, 8);
            tok = 0;
        }
        p.tokens[b * p.gamma + k] = tok;
        p.conf[b * p.gamma + k] = 1.f / (1.f + expf(-(z + p.conf_w[p.d + r])));
        p.counters[b] = 0u;
    }
}

// Bounded grid-wide barrier for a cooperative launch: `count` and `gen` are
// zero-initialised device words shared by all CTAs.  Gives up after about a
// second (sets DSPARK_DEVERR_TIMEOUT in *err and returns false).
__device__ __forceinline__ bool grid_sync(unsigned int* count, unsigned int* gen, unsigned int n_ctas, int* err) {
    __shared__ int ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        ok = 1;
        const unsigned int g = *(volatile unsigned int*)gen;
        __threadfence();
        if (atomicAdd(count, 1u) == n_ctas - 1) {
            *(volatile unsigned int*)count = 0u;
            __threadfence();
            atomicAdd(gen, 1u);
        } else {
            uint64_t t0, t;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
            while (*(volatile unsigned int*)gen == g) {
                asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
                if (t - t0 > 1000000000ull) {
                    atomicOr(err, 16);
                    ok = 0;
                    break;
                }
            }
        }
        __threadfence();
    }
    __syncthreads();
    return ok != 0;
}

// The whole chain in one cooperative launch: grid = ctas * B CTAs, CTA c of
// sequence b = blockIdx.x / ctas streams its slice of w2 at every position;
// after one grid barrier per position every CTA of the sequence reduces the
// CTA winners itself (the key is a total order, so all agree), and CTA 0 of the
// sequence writes the token and the confidence.  Partials are double-buffered
// by position parity: a buffer is rewritten two positions later, after a
// barrier every CTA passed only once done reading it.
template <typename TW>
__global__ void __launch_bounds__(NT) k_markov_chain(MarkovParams p, unsigned int* bar_count, unsigned int* bar_gen) {
    constexpr int VE = Vec16<TW>::N;
    __shared__ __align__(16) float e[RMAX];
    __shared__ float red_v[NT / 32];
    __shared__ int red_i[NT / 32];
    __shared__ float redf[32];
    __shared__ int prev_s;

    const int ctas = p.ctas;
    const int b = blockIdx.x / ctas, cta = blockIdx.x - b * ctas;
    const int r = p.r, V = p.V;
    const TW* w1 = reinterpret_cast<const TW*>(p.w1);
    const TW* w2 = reinterpret_cast<const TW*>(p.w2);
    const int rows = (V + ctas - 1) / ctas;
    const int v_begin = cta * rows, v_end = min(V, v_begin + rows);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane & (LPR - 1), rw = lane / LPR;
    const int nvec = r / VE;
    if (threadIdx.x == 0) prev_s = min(max(p.anchors ? p.anchors[b] : p.anchor, 0), V - 1);
    __syncthreads();

    for (int k = 0; k < p.gamma; ++k) {
        const int prev = prev_s;
        for (int c = threadIdx.x; c < r; c += NT) e[c] = to_f32(w1[(int64_t)prev * r + c]);
        __syncthreads();
        const int64_t urow = (int64_t)(b * p.gamma + k) * V;
        ArgBest best{-INFINITY, INT_MAX};
        for (int v0 = v_begin + warp * (2 * RPW); v0 < v_end; v0 += (NT / 32) * (2 * RPW)) {
            const int va = v0 + rw, vb = v0 + RPW + rw;
            const TW* ra = w2 + (int64_t)min(va, v_end - 1) * r;
            const TW* rb = w2 + (int64_t)min(vb, v_end - 1) * r;
            float aa = 0.f, ab = 0.f;
            for (int vi = sub; vi < nvec; vi += 4 * LPR) {
                uint4 ua[4], ub[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int x = vi + q * LPR;
                    ua[q] = x < nvec ? __ldg(reinterpret_cast<const uint4*>(ra + x * VE)) : make_uint4(0, 0, 0, 0);
                    ub[q] = x < nvec ? __ldg(reinterpret_cast<const uint4*>(rb + x * VE)) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int x = vi + q * LPR;
                    if (x >= nvec) break;
                    float fa[VE], fb[VE];
                    Vec16<TW>::unpack(ua[q], fa);
                    Vec16<TW>::unpack(ub[q], fb);
                    const float* ep = e + x * VE;
#pragma unroll
                    for (int t = 0; t < VE; ++t) {
                        aa = fmaf(fa[t], ep[t], aa);
                        ab = fmaf(fb[t], ep[t], ab);
                    }
                }
            }
#pragma unroll
            for (int o = 1; o < LPR; o <<= 1) {
                aa += __shfl_xor_sync(0xffffffffu, aa, o);
                ab += __shfl_xor_sync(0xffffffffu, ab, o);
            }
            if (sub == 0) {
                if (va < v_end) {
                    const float l = p.U[urow + va] + aa;
                    if (p.logits) p.logits[urow + va] = l;
                    if (better(l, va, best.v, best.i)) {
                        best.v = l;
                        best.i = va;
                    }
                }
                if (vb < v_end) {
                    const float l = p.U[urow + vb] + ab;
                    if (p.logits) p.logits[urow + vb] = l;
                    if (better(l, vb, best.v, best.i)) {
                        best.v = l;
                        best.i = vb;
                    }
                }
            }
        }
        best = warp_argbest(best);
        if (lane == 0) {
            red_v[warp] = best.v;
            red_i[warp] = best.i;
        }
        __syncthreads();
        const int64_t pb = (int64_t)(k & 1) * p.B * ctas + (int64_t)b * ctas;
        if (threadIdx.x == 0) {
            ArgBest cb{-INFINITY, INT_MAX};
            for (int w = 0; w < NT / 32; ++w)
                if (better(red_v[w], red_i[w], cb.v, cb.i)) {
                    cb.v = red_v[w];
                    cb.i = red_i[w];
                }
            p.part_v[pb + cta] = cb.v;
            p.part_i[pb + cta] = cb.i;
        }
        grid_sync(bar_count, bar_gen, gridDim.x, p.err);
        // every CTA of the sequence: the winner over the CTA results
        ArgBest fb{-INFINITY, INT_MAX};
        for (int c = threadIdx.x; c < ctas; c += NT) {
            const float v = __ldcg(p.part_v + pb + c);
            const int i = __ldcg(p.part_i + pb + c);
            if (better(v, i, fb.v, fb.i)) {
                fb.v = v;
                fb.i = i;
            }
        }
        fb = warp_argbest(fb);
        __syncthreads();  // red_v/red_i reuse
        if (lane == 0) {
            red_v[warp] = fb.v;
            red_i[warp] = fb.i;
        }
        float z = 0.f;
        if (cta == 0) {
            const float* yr = p.y + (int64_t)(b * p.gamma + k) * p.d;
            for (int c = threadIdx.x; c < p.d; c += NT) z = fmaf(yr[c], p.conf_w[c], z);
            for (int c = threadIdx.x; c < r; c += NT) z = fmaf(e[c], p.conf_w[p.d + c], z);
        }
        z = block_sum(z, redf);  // contains __syncthreads: red_v/red_i are complete
        if (threadIdx.x == 0) {
            ArgBest tb{-INFINITY, INT_MAX};
            for (int w = 0; w < NT / 32; ++w)
                if (better(red_v[w], red_i[w], tb.v, tb.i)) {
                    tb.v = red_v[w];
                    tb.i = red_i[w];
                }
            int tok = tb.i;
            if (tok == INT_MAX || !(tb.v > -INFINITY)) {
                if (cta == 0) atomicOr(p.err, 8);
                tok = 0;
            }
            prev_s = tok;
            if (cta == 0) {
                p.tokens[b * p.gamma + k] = tok;
                p.conf[b * p.gamma + k] = 1.f / (1.f + expf(-(z + p.conf_w[p.d + r])));
            }
        }
        __syncthreads();
    }
}

// E[b][:] = w1[prev_b] for the many-sequence form (prev_b = anchor at k = 0, else token k-1).
template <typename TW>
__global__ void k_markov_gather(const TW* __restrict__ w1, int r, int V, const int* __restrict__ anchors,
                                const int* __restrict__ tokens, int gamma, int k, TW* __restrict__ E) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x;
    int prev = k == 0 ? anchors[b] : tokens[b * gamma + k - 1];
    prev = min(max(prev, 0), V - 1);
    for (int c = threadIdx.x; c < r; c += blockDim.x) E[(int64_t)b * r + c] = w1[(int64_t)prev * r + c];
}

// Per sequence: the best of the 32-column chunk partials, then token and confidence.
template <typename TW>
__global__ void __launch_bounds__(NT) k_markov_finish(const float* __restrict__ part_v, const int* __restrict__ part_i,
                                                      int nchunks, const TW* __restrict__ w1,
                                                      const float* __restrict__ y, const float* __restrict__ conf_w,
                                                      const int* __restrict__ anchors, int* tokens, float* conf,
                                                      int gamma, int k, int d, int r, int V, int* err) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red_v[NT / 32];
    __shared__ int red_i[NT / 32];
    __shared__ float redf[32];
    const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    ArgBest best{-INFINITY, INT_MAX};
    for (int c = threadIdx.x; c < nchunks; c += NT) {
        const float v = part_v[(int64_t)b * nchunks + c];
        const int i = part_i[(int64_t)b * nchunks + c];
        if (better(v, i, best.v, best.i)) {
            best.v = v;
            best.i = i;
        }
    }
    best = warp_argbest(best);
    if (lane == 0) {
        red_v[warp] = best.v;
        red_i[warp] = best.i;
    }
    int prev = k == 0 ? anchors[b] : tokens[b * gamma + k - 1];
    prev = min(max(prev, 0), V - 1);
    const float* yr = y + (int64_t)(b * gamma + k) * d;
    float z = 0.f;
    for (int c = threadIdx.x; c < d; c += NT) z = fmaf(yr[c], conf_w[c], z);
    for (int c = threadIdx.x; c < r; c += NT) z = fmaf(to_f32(w1[(int64_t)prev * r + c]), conf_w[d + c], z);
    z = block_sum(z, redf);
    if (threadIdx.x == 0) {
        ArgBest tb{-INFINITY, INT_MAX};
        for (int w = 0; w < NT / 32; ++w)
            if (better(red_v[w], red_i[w], tb.v, tb.i)) {
                tb.v = red_v[w];
                tb.i = red_i[w];
            }
        int tok = tb.i;
        if (tok == INT_MAX || !(tb.v > -INFINITY)) {
            atomicOr(err, 8);
            tok = 0;
        }
        tokens[b * gamma + k] = tok;
        conf[b * gamma + k] = 1.f / (1.f + expf(-(z + conf_w[d + r])));
    }
}

}  // namespace

cudaError_t markov_gather(const void* w1, int r, int V, const int* anchors, const int* tokens, int gamma, int k, int B,
                          void* E, cudaStream_t st) {
    launch(k_markov_gather<bf16>, B, 128, 0, st, (const bf16*)w1, r, V, anchors, tokens, gamma, k, (bf16*)E);
    note_launch();
    return cudaGetLastError();
}

cudaError_t markov_finish(const float* part_v, const int* part_i, int nchunks, const void* w1, int w_dtype,
                          const float* y, const float* conf_w, const int* anchors, int* tokens, float* conf, int B,
                          int gamma, int k, int d, int r, int V, int* err, cudaStream_t st) {
    if (w_dtype == DT_BF16)
        launch(k_markov_finish<bf16>, B, NT, 0, st, part_v, part_i, nchunks, (const bf16*)w1, y, conf_w, anchors,
               tokens, conf, gamma, k, d, r, V, err);
    else
        launch(k_markov_finish<float>, B, NT, 0, st, part_v, part_i, nchunks, (const float*)w1, y, conf_w, anchors,
               tokens, conf, gamma, k, d, r, V, err);
    note_launch();
    return cudaGetLastError();
}

int markov_ctas(int V) {
    int c = (V + 127) / 128;  // 128 vocabulary rows per CTA
    return c < 1 ? 1 : (c > 4096 ? 4096 : c);
}

int markov_chain_max_ctas(int w_dtype) {
    int per_sm = 0, dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cudaError_t e = w_dtype == DT_BF16
                        ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_markov_chain<bf16>, NT, 0)
                        : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_markov_chain<float>, NT, 0);
    if (e != cudaSuccess) return 0;
    return per_sm * sms;
}

cudaError_t markov_chain(const MarkovParams& p, unsigned int* bar_count, unsigned int* bar_gen, cudaStream_t st) {
    if (p.r > RMAX || p.r % 8 != 0) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.ctas * p.B);
    cfg.blockDim = dim3(NT);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = p.w_dtype == DT_BF16 ? cudaLaunchKernelEx(&cfg, k_markov_chain<bf16>, p, bar_count, bar_gen)
                                         : cudaLaunchKernelEx(&cfg, k_markov_chain<float>, p, bar_count, bar_gen);
    note_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t markov_step(const MarkovParams& p, cudaStream_t st) {
    if (p.r > RMAX || p.r % 8 != 0) return cudaErrorInvalidValue;
    dim3 grid(p.ctas, p.B);
    if (p.w_dtype == DT_BF16)
        launch(k_markov<bf16>, grid, NT, 0, st, p);
    else
        launch(k_markov<float>, grid, NT, 0, st, p);
    note_launch();
    return cudaGetLastError();
}

}  // namespace dspark
