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
#include <algorithm>
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
constexpr int GMAX_CHAIN = 16; // largest block size (key words per sequence)

template <typename TW>
__global__ void __launch_bounds__(NT) k_markov(MarkovParams p) {
    pdl_wait();
    pdl_trigger();
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

// (value, index) -> one 64-bit key whose unsigned order is the argmax order:
// larger value first, then lower index.  Key 0 is below every candidate.
__device__ __forceinline__ unsigned long long arg_key(float v, int i) {
    unsigned int u = __float_as_uint(v);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)u << 32) | (unsigned long long)(~(unsigned int)i);
}
__device__ __forceinline__ float key_value(unsigned long long key) {
    unsigned int u = (unsigned int)(key >> 32);
    u = (u & 0x80000000u) ? (u & 0x7fffffffu) : ~u;
    return __uint_as_float(u);
}

// The whole chain in one cooperative launch: grid = ctas * B CTAs, CTA c of
// sequence b = blockIdx.x / ctas streams its slice of w2 at every position and
// folds its best (value, index) into one 64-bit word per (sequence, position)
// with an atomic max; after one grid barrier per position every CTA reads the
// token from that word.  The confidences need only the tokens, so CTA 0 of
// each sequence computes them after the last position.  The words alternate
// between two sets by launch parity (a device epoch counter): a launch clears
// the other set, which the next launch uses.
template <typename TW>
__global__ void __launch_bounds__(NT) k_markov_chain(MarkovParams p, unsigned int* bar_count, unsigned int* bar_gen) {
    constexpr int VE = Vec16<TW>::N;
    __shared__ __align__(16) float e[RMAX];
    __shared__ float red_v[NT / 32];
    __shared__ int red_i[NT / 32];
    __shared__ float redf[32];
    __shared__ int toks[GMAX_CHAIN + 1];

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
    const unsigned int par = *(volatile unsigned int*)p.epoch & 1u;
    unsigned long long* keys = p.keys + (size_t)par * p.keys_stride + (size_t)b * GMAX_CHAIN;
    if (blockIdx.x == 0) {
        unsigned long long* other = p.keys + (size_t)(par ^ 1u) * p.keys_stride;
        for (int i = threadIdx.x; i < p.keys_stride; i += NT) other[i] = 0ull;
        if (p.bar && threadIdx.x == 0) p.bar[par ^ 1u] = 0ull;  // shared with the resident form
    }
    if (threadIdx.x == 0) toks[0] = min(max(p.anchors ? p.anchors[b] : p.anchor, 0), V - 1);
    __syncthreads();

    for (int k = 0; k < p.gamma; ++k) {
        const int prev = toks[k];
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
        if (threadIdx.x == 0) {
            ArgBest cb{-INFINITY, INT_MAX};
            for (int w = 0; w < NT / 32; ++w)
                if (better(red_v[w], red_i[w], cb.v, cb.i)) {
                    cb.v = red_v[w];
                    cb.i = red_i[w];
                }
            if (cb.i != INT_MAX) atomicMax(keys + k, arg_key(cb.v, cb.i));
        }
        grid_sync(bar_count, bar_gen, gridDim.x, p.err);  // orders the atomic before the arrival
        if (threadIdx.x == 0) {
            const unsigned long long key = __ldcg(keys + k);
            int tok = (int)(~(unsigned int)key);
            if (key == 0ull || !(key_value(key) > -INFINITY) || tok < 0 || tok >= V) {
                if (cta == 0) atomicOr(p.err, 8);
                tok = 0;
            }
            toks[k + 1] = tok;
            if (cta == 0) p.tokens[b * p.gamma + k] = tok;
        }
        __syncthreads();
    }
    // confidences of every position: sigmoid(conf_w . [y_k ; w1[prev_k]] + conf_b)
    if (cta == 0) {
        for (int k = 0; k < p.gamma; ++k) {
            const float* yr = p.y + (int64_t)(b * p.gamma + k) * p.d;
            const TW* er = w1 + (int64_t)toks[k] * r;
            float z = 0.f;
            for (int c = threadIdx.x; c < p.d; c += NT) z = fmaf(yr[c], p.conf_w[c], z);
            for (int c = threadIdx.x; c < r; c += NT) z = fmaf(to_f32(er[c]), p.conf_w[p.d + c], z);
            z = block_sum(z, redf);
            if (threadIdx.x == 0) p.conf[b * p.gamma + k] = 1.f / (1.f + expf(-(z + p.conf_w[p.d + r])));
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicAdd(p.epoch, 1u);  // every CTA read it before the first barrier
}

// ---- resident form: up to 8 sequences, bf16 weights, r = 64, 128 or 256 ------------
// (the draft step uses it for 3 to 8 sequences; one or two take the FMA form further down)
// One CTA per SM for the whole chain.  CTA c owns vocabulary rows
// [c * rows, (c + 1) * rows) for every sequence and keeps as many of its w2
// rows as fit in shared memory for all gamma positions (the rest are read
// from global memory each position), so w2 crosses the memory system once
// per chain instead of once per position.  The dot products w2 . e_b run on
// the tensor cores: mma.m16n8k16 with 16 vocabulary rows as M, the (up to 8)
// sequences' e = w1[prev] as the N columns, r as K.  Inside each 32-wide slice
// of r the K order is permuted so that a lane's A fragments for two k-steps
// are one 16-byte chunk of a row and its B fragments one 16-byte chunk of its
// sequence's e (the same permutation on both sides leaves every dot product
// unchanged).  Resident rows are stored with their 16-byte chunks XOR-swizzled
// by row, so the fragment loads are free of bank conflicts.  Per position:
// base logits (prefetched into shared memory during the previous barrier), a
// (value, index) atomic max per sequence, then one grid barrier on a 64-bit
// arrival counter (release add, acquire poll; it counts up through the launch,
// barrier k opens at (k + 1) * gridDim.x).  Counters and argmax words
// alternate between two sets by launch parity.
constexpr int NT_RES = 512;
constexpr int NB_RES = 8;  // sequences: the N of the MMA

__device__ __forceinline__ void cp_async16_res(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// c[16x8] += a[16x16] . b[16x8], bf16 inputs, fp32 accumulators
__device__ __forceinline__ void mma_bf16_16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// the two k-steps held by one 16-byte chunk of rows g, g+8 (lo, hi) and of e
__device__ __forceinline__ void mma_chunk(float* c, const uint4& lo, const uint4& hi, const uint4& ev) {
    mma_bf16_16816(c, lo.x, hi.x, lo.y, hi.y, ev.x, ev.y);
    mma_bf16_16816(c, lo.z, hi.z, lo.w, hi.w, ev.z, ev.w);
}

// Bounded barrier of the resident chain: true when every CTA has arrived.
__device__ __forceinline__ bool res_barrier(unsigned long long* bar, unsigned long long target, int* err) {
    __shared__ int ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        ok = 1;
        asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(bar) : "memory");
        uint64_t t0, t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
        while (true) {
            unsigned long long cur;
            asm volatile("ld.acquire.gpu.u64 %0, [%1];" : "=l"(cur) : "l"(bar) : "memory");
            if (cur >= target) break;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
            if (t - t0 > 1000000000ull) {
                atomicOr(err, 16);
                ok = 0;
                break;
            }
        }
    }
    __syncthreads();
    return ok != 0;
}

template <int KD>  // r = 32 * KD
__global__ void __launch_bounds__(NT_RES, 1) k_markov_chain_res(MarkovParams p, int n_cache) {
    constexpr int R = KD * 32;
    constexpr int ROWB = R * 2;   // bytes of one w2 row
    constexpr int CPR = ROWB / 16;  // 16-byte chunks per row (a multiple of 8)
    // dynamic shared memory: [n_cache][ROWB] resident w2 rows (swizzled chunks),
    // then the base logits of the next position, [2 buffers][B][rows] fp32
    extern __shared__ __align__(128) uint8_t w2s[];
    __shared__ float red_v[NB_RES][NT_RES / 32];
    __shared__ int red_i[NB_RES][NT_RES / 32];
    __shared__ float redf[32];
    __shared__ int toks[NB_RES][GMAX_CHAIN + 1];

    const int V = p.V, gamma = p.gamma, NB = p.B;
    const bf16* __restrict__ w1 = reinterpret_cast<const bf16*>(p.w1);
    const bf16* __restrict__ w2 = reinterpret_cast<const bf16*>(p.w2);
    float* __restrict__ lg = p.logits;
    const int rows = (V + gridDim.x - 1) / gridDim.x;
    const int v_begin = blockIdx.x * rows;
    const int nrows = max(0, min(V, v_begin + rows) - v_begin);
    const int nc = min(n_cache, nrows);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    float* ubuf = reinterpret_cast<float*>(w2s + (size_t)n_cache * ROWB);  // [2][NB][rows]
    const uint32_t ubuf_s = (uint32_t)__cvta_generic_to_shared(ubuf);
    const uint32_t w2s_s = (uint32_t)__cvta_generic_to_shared(w2s);

    {  // the resident rows: chunk c of row li at chunk c ^ (li & 7)
        const uint8_t* src = reinterpret_cast<const uint8_t*>(w2 + (int64_t)v_begin * R);
        for (int i = tid; i < nc * CPR; i += NT_RES) {
            const int li = i / CPR, c = i - li * CPR;
            cp_async16_res(w2s_s + li * ROWB + ((c ^ (li & 7)) * 16), src + (size_t)i * 16);
        }
    }
    auto load_u = [&](int k) {  // base logits of position k for this CTA's rows, into buffer k & 1
        for (int i = tid; i < NB * nrows; i += NT_RES) {
            const int b = i / nrows, li = i - b * nrows;
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                             ubuf_s + (uint32_t)((((k & 1) * NB + b) * rows + li) * 4)),
                         "l"(p.U + (int64_t)(b * gamma + k) * V + v_begin + li)
                         : "memory");
        }
    };
    load_u(0);
    asm volatile("cp.async.commit_group;" ::: "memory");
    const unsigned int par = *(volatile unsigned int*)p.epoch & 1u;
    unsigned long long* keys = p.keys + (size_t)par * p.keys_stride;
    unsigned long long* bar = p.bar + par;
    if (blockIdx.x == 0) {
        unsigned long long* other = p.keys + (size_t)(par ^ 1u) * p.keys_stride;
        for (int i = tid; i < p.keys_stride; i += NT_RES) other[i] = 0ull;
        if (tid == 0) p.bar[par ^ 1u] = 0ull;
    }
    if (tid < NB) toks[tid][0] = min(max(p.anchors ? p.anchors[tid] : p.anchor, 0), V - 1);

    const int tiles = (nrows + 15) / 16;
    for (int k = 0; k < gamma; ++k) {
        asm volatile("cp.async.wait_group 0;" ::: "memory");  // resident rows (k = 0) and this position's U
        __syncthreads();
        const float* uk = ubuf + (k & 1) * NB * rows;
        // B fragments: lane (g, t) supplies sequence g's e = w1[prev_g], chunk 4j + t of every slice j
        uint4 ev[KD];
#pragma unroll
        for (int j = 0; j < KD; ++j)
            ev[j] = g < NB ? __ldg(reinterpret_cast<const uint4*>(w1 + (int64_t)toks[g][k] * R + (4 * j + t) * 8))
                           : make_uint4(0, 0, 0, 0);
        ArgBest best[2] = {{-INFINITY, INT_MAX}, {-INFINITY, INT_MAX}};  // sequences 2t, 2t+1
        // the highest tiles (rows read from global memory) first: their loads overlap the load of e
        for (int tile = warp + (tiles - 1 - warp) / 16 * 16; tile >= 0 && warp < tiles; tile -= 16) {
            const int la = tile * 16 + g, lb = la + 8;
            float c[4] = {0.f, 0.f, 0.f, 0.f};
            if (tile * 16 + 16 <= nc) {
#pragma unroll
                for (int j = 0; j < KD; ++j) {
                    const int ch = 4 * j + t;
                    const uint4 lo = *reinterpret_cast<const uint4*>(w2s + la * ROWB + ((ch ^ (la & 7)) * 16));
                    const uint4 hi = *reinterpret_cast<const uint4*>(w2s + lb * ROWB + ((ch ^ (lb & 7)) * 16));
                    mma_chunk(c, lo, hi, ev[j]);
                }
            } else {
                uint4 lo[KD], hi[KD];
#pragma unroll
                for (int j = 0; j < KD; ++j) {
                    const int ch = 4 * j + t;
                    lo[j] = la < nc ? *reinterpret_cast<const uint4*>(w2s + la * ROWB + ((ch ^ (la & 7)) * 16))
                            : la < nrows ? __ldg(reinterpret_cast<const uint4*>(w2 + (int64_t)(v_begin + la) * R + ch * 8))
                                         : make_uint4(0, 0, 0, 0);
                    hi[j] = lb < nc ? *reinterpret_cast<const uint4*>(w2s + lb * ROWB + ((ch ^ (lb & 7)) * 16))
                            : lb < nrows ? __ldg(reinterpret_cast<const uint4*>(w2 + (int64_t)(v_begin + lb) * R + ch * 8))
                                         : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int j = 0; j < KD; ++j) mma_chunk(c, lo[j], hi[j], ev[j]);
            }
            // c[0], c[1]: row la, sequences 2t, 2t+1; c[2], c[3]: row lb
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int li = q < 2 ? la : lb, n = 2 * t + (q & 1);
                if (li < nrows && n < NB) {
                    const int v = v_begin + li;
                    const float l = c[q] + uk[n * rows + li];
                    if (lg) lg[(int64_t)(n * gamma + k) * V + v] = l;
                    if (better(l, v, best[q & 1].v, best[q & 1].i)) {
                        best[q & 1].v = l;
                        best[q & 1].i = v;
                    }
                }
            }
        }
        // over the 8 row groups of the warp (lanes with equal t hold the same sequences)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, best[h].v, o);
                const int oi = __shfl_xor_sync(0xffffffffu, best[h].i, o);
                if (better(ov, oi, best[h].v, best[h].i)) {
                    best[h].v = ov;
                    best[h].i = oi;
                }
            }
            if (g == 0 && 2 * t + h < NB) {
                red_v[2 * t + h][warp] = best[h].v;
                red_i[2 * t + h][warp] = best[h].i;
            }
        }
        __syncthreads();
        if (warp < NB) {  // warp b reduces sequence b's 16 warp results
            ArgBest cb{lane < NT_RES / 32 ? red_v[warp][lane] : -INFINITY,
                       lane < NT_RES / 32 ? red_i[warp][lane] : INT_MAX};
            cb = warp_argbest(cb);
            if (lane == 0 && cb.i != INT_MAX) atomicMax(keys + warp * GMAX_CHAIN + k, arg_key(cb.v, cb.i));
        }
        if (k + 1 < gamma) load_u(k + 1);  // its buffer was last read two positions ago
        asm volatile("cp.async.commit_group;" ::: "memory");
        res_barrier(bar, (unsigned long long)(k + 1) * gridDim.x, p.err);
        if (tid < NB) {
            const unsigned long long key = __ldcg(keys + tid * GMAX_CHAIN + k);
            int tok = (int)(~(unsigned int)key);
            if (key == 0ull || !(key_value(key) > -INFINITY) || tok < 0 || tok >= V) {
                if (blockIdx.x == 0) atomicOr(p.err, 8);
                tok = 0;
            }
            toks[tid][k + 1] = tok;
            if (blockIdx.x == 0) p.tokens[tid * gamma + k] = tok;
        }
    }
    __syncthreads();
    // confidences: sigmoid(conf_w . [y_k ; w1[prev_k]] + conf_b), by CTA 0
    if (blockIdx.x == 0) {
        for (int b = 0; b < NB; ++b)
            for (int k = 0; k < gamma; ++k) {
                const float* yr = p.y + (int64_t)(b * gamma + k) * p.d;
                const bf16* er = w1 + (int64_t)toks[b][k] * R;
                float z = 0.f;
                for (int c = tid; c < p.d; c += NT_RES) z = fmaf(yr[c], p.conf_w[c], z);
                for (int c = tid; c < R; c += NT_RES) z = fmaf(to_f32(er[c]), p.conf_w[p.d + c], z);
                z = block_sum(z, redf);
                if (tid == 0) p.conf[b * gamma + k] = 1.f / (1.f + expf(-(z + p.conf_w[p.d + R])));
            }
        if (tid == 0) atomicAdd(p.epoch, 1u);  // every CTA read it before the first barrier
    }
}

// One or two sequences: the same resident w2 slice, but the dot products run on
// the FMA pipes (bf16 x bf16 + fp32, one rounding each), since a warp MMA would
// spend 7 of its 8 columns on nothing.  An 8-lane group takes 8 rows of a
// 512-row pass, strided by 64 so that the rows read from global memory (past
// the resident ones) spread over every group; lane s holds the 16-byte chunks
// s, s + 8, ... of each row and of e = w1[prev], and a butterfly over the group
// leaves lane s with the whole dot product of the group's row s.  The
// position's argmax goes through one 64-bit word per CTA and an arrival
// counter (word stored, then a release add); one lane per CTA polls the
// counter with a bound and its warp then reads every word once, which keeps
// the polling off the words' cache lines.  Before publishing, each CTA pulls
// the w1 row of its own best into L2, which holds the next position's e
// wherever the winner came from.
constexpr int NT_FMA = 512;
constexpr int NB_FMA = 2;  // sequences the FMA chain serves

__device__ __forceinline__ uint64_t chain_clock() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// One thread waits (bounded, about a second) until *counter >= target; true when it gave up.
__device__ __forceinline__ bool wait_arrivals(const unsigned long long* counter, unsigned long long target) {
    const uint64_t t0 = chain_clock();
    while (true) {
        unsigned long long cur;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(cur) : "l"(counter) : "memory");
        if (cur >= target) return false;
        if (chain_clock() - t0 > 1000000000ull) return true;
    }
}

// 16-byte read-only load with an L2 eviction policy (from createpolicy)
__device__ __forceinline__ uint4 ld_nc_policy(const uint4* a, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(a), "l"(pol));
    return v;
}

// acc += sum over the 8 bf16 pairs of w and e, in order
__device__ __forceinline__ float fma_chunk(const uint4& w, const uint4& e, float acc) {
    asm("{\n\t.reg .b16 a0, a1, a2, a3, a4, a5, a6, a7, b0, b1, b2, b3, b4, b5, b6, b7;\n\t"
        "mov.b32 {a0, a1}, %1;\n\tmov.b32 {a2, a3}, %2;\n\tmov.b32 {a4, a5}, %3;\n\tmov.b32 {a6, a7}, %4;\n\t"
        "mov.b32 {b0, b1}, %5;\n\tmov.b32 {b2, b3}, %6;\n\tmov.b32 {b4, b5}, %7;\n\tmov.b32 {b6, b7}, %8;\n\t"
        "fma.rn.f32.bf16 %0, a0, b0, %0;\n\tfma.rn.f32.bf16 %0, a1, b1, %0;\n\t"
        "fma.rn.f32.bf16 %0, a2, b2, %0;\n\tfma.rn.f32.bf16 %0, a3, b3, %0;\n\t"
        "fma.rn.f32.bf16 %0, a4, b4, %0;\n\tfma.rn.f32.bf16 %0, a5, b5, %0;\n\t"
        "fma.rn.f32.bf16 %0, a6, b6, %0;\n\tfma.rn.f32.bf16 %0, a7, b7, %0;\n\t}"
        : "+f"(acc)
        : "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w), "r"(e.x), "r"(e.y), "r"(e.z), "r"(e.w));
    return acc;
}

// 8 row partials per lane of an 8-lane group -> lane s holds the group sum of row s
__device__ __forceinline__ float reduce_scatter8(const float (&a)[8], int s) {
    float h[4], q[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float give = (s & 4) ? a[i] : a[i + 4];
        h[i] = ((s & 4) ? a[i + 4] : a[i]) + __shfl_xor_sync(0xffffffffu, give, 4);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float give = (s & 2) ? h[i] : h[i + 2];
        q[i] = ((s & 2) ? h[i + 2] : h[i]) + __shfl_xor_sync(0xffffffffu, give, 2);
    }
    const float give = (s & 1) ? q[0] : q[1];
    return ((s & 1) ? q[1] : q[0]) + __shfl_xor_sync(0xffffffffu, give, 1);
}

// NSTG > 0: the rows past the resident ones stream through a per-thread cp.async ring of NSTG
// 64-row blocks (n_cache a multiple of 64), so that their loads run ahead across passes and across
// the argmax exchange; each thread copies exactly the 16-byte chunks it reads, and its own copy
// groups are its only synchronisation.  The arithmetic is the same as without the ring.
constexpr int MAX_SBLK = 64;  // streamed 64-row blocks per CTA in the ring form
constexpr int RING_STAGES = 3;

template <int KD, int NF, int NSTG = 0>  // r = 32 * KD, NF sequences
__global__ void __launch_bounds__(NT_FMA, 1) k_markov_chain_fma(MarkovParams p, int n_cache, int n_keep) {
    constexpr int R = KD * 32;
    constexpr int ROWB = R * 2;
    constexpr int CPR = ROWB / 16;  // 16-byte chunks per row
    constexpr int CPL = CPR / 8;    // chunks per lane
    constexpr int GROUPS = NT_FMA / 8;
    constexpr int PASS = GROUPS * 8;  // rows per pass
    extern __shared__ __align__(128) uint8_t w2s[];
    __shared__ float red_v[NF][NT_FMA / 32];
    __shared__ int red_i[NF][NT_FMA / 32];
    __shared__ float redf[32];
    __shared__ int toks[NF][GMAX_CHAIN + 1];

    const int V = p.V, gamma = p.gamma, G = gridDim.x;
    const bf16* __restrict__ w1 = reinterpret_cast<const bf16*>(p.w1);
    const bf16* __restrict__ w2 = reinterpret_cast<const bf16*>(p.w2);
    float* __restrict__ lg = p.logits;
    const int rows = (V + G - 1) / G;
    const int v_begin = blockIdx.x * rows;
    const int nrows = max(0, min(V, v_begin + rows) - v_begin);
    const int nc = min(n_cache, nrows);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, s = lane & 7, grp = tid >> 3;
    constexpr int RING_BYTES = NSTG * 64 * ROWB;
    float* ubuf = reinterpret_cast<float*>(w2s + (size_t)n_cache * ROWB + RING_BYTES);  // [2][NF][rows]
    const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(w2s + (size_t)n_cache * ROWB);
    __shared__ short sblk[NSTG > 0 ? MAX_SBLK : 1];  // first rows of the streamed blocks, in consumption order
    __shared__ int n_sblk;
    const uint32_t ubuf_s = (uint32_t)__cvta_generic_to_shared(ubuf);
    const uint32_t w2s_s = (uint32_t)__cvta_generic_to_shared(w2s);
    const uint4* __restrict__ w2g = reinterpret_cast<const uint4*>(w2 + (int64_t)v_begin * R);

    {  // the resident rows: chunk c of row li at chunk c ^ (li & 7)
        const uint8_t* src = reinterpret_cast<const uint8_t*>(w2 + (int64_t)v_begin * R);
        for (int i = tid; i < nc * CPR; i += NT_FMA) {
            const int li = i / CPR, c = i - li * CPR;
            cp_async16_res(w2s_s + li * ROWB + ((c ^ (li & 7)) * 16), src + (size_t)i * 16);
        }
    }
    auto load_u = [&](int k) {
        for (int i = tid; i < NF * nrows; i += NT_FMA) {
            const int b = i / nrows, li = i - b * nrows;
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                             ubuf_s + (uint32_t)((((k & 1) * NF + b) * rows + li) * 4)),
                         "l"(p.U + (int64_t)(b * gamma + k) * V + v_begin + li)
                         : "memory");
        }
    };
    load_u(0);
    asm volatile("cp.async.commit_group;" ::: "memory");
    const unsigned int par = *(volatile unsigned int*)p.epoch & 1u;
    unsigned long long* slots = p.keys + (size_t)par * p.keys_stride;  // [16][NF][G] words
    unsigned long long* arrived = slots + (size_t)GMAX_CHAIN * NF * G;   // [16][NF] arrival counters
    if (blockIdx.x == 0) {
        unsigned long long* other = p.keys + (size_t)(par ^ 1u) * p.keys_stride;
        for (int i = tid; i < p.keys_stride; i += NT_FMA) other[i] = 0ull;
    }
    if (tid < NF) toks[tid][0] = min(max(p.anchors ? p.anchors[tid] : p.anchor, 0), V - 1);

    // The rows past the resident ones are read again at every position, and together they can
    // exceed what L2 keeps: least-recently-used replacement then drops each line before its
    // next use. The first n_keep of them (a share of L2 chosen by the host) are loaded with
    // evict-last and the rest with evict-first, so the kept share hits in L2 at every position
    // after the first; the last position loads everything evict-first to release the lines.
    uint64_t pol_keep, pol_pass;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_keep));
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_pass));
    // ring form: the streamed blocks in the order the passes take them (rows ascending by pass,
    // blocks descending inside a pass), then the first NSTG - 1 of them requested
    int nsb = 0, qc = 0;
    auto issue = [&](int q) {  // this thread's chunks of the q-th streamed block, over all positions
        if (q < gamma * nsb) {
            const int kq = q / nsb, li = sblk[q - kq * nsb] + grp;
            const bool in = li < nrows;
            const uint64_t pol = (kq + 1 < gamma && li < nc + n_keep) ? pol_keep : pol_pass;
            const uint4* src = w2g + (int64_t)(in ? li : 0) * CPR;
            const uint32_t dst = ring_s + (uint32_t)((q % (NSTG > 0 ? NSTG : 1)) * 64 + grp) * ROWB;
#pragma unroll
            for (int j = 0; j < CPL; ++j)
                asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(
                                 dst + (uint32_t)((s + 8 * j) * 16)),
                             "l"(src + s + 8 * j), "r"(in ? 16 : 0), "l"(pol)
                             : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    if constexpr (NSTG > 0) {
        if (tid == 0) {
            int n = 0;
            for (int base = 0; base < nrows; base += PASS)
                for (int i = 7; i >= 0; --i) {
                    const int row0 = base + 64 * i;
                    if (row0 >= nc && row0 < nrows && n < MAX_SBLK) sblk[n++] = (short)row0;
                }
            n_sblk = n;
        }
        __syncthreads();
        nsb = n_sblk;
        for (int q = 0; q < NSTG - 1; ++q) issue(q);
    }
    for (int k = 0; k < gamma; ++k) {
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();
        const float* uk = ubuf + (k & 1) * NF * rows;
        const int keep_end = k + 1 < gamma ? nc + n_keep : nc;
        uint4 ev[NF][CPL];
#pragma unroll
        for (int n = 0; n < NF; ++n)
#pragma unroll
            for (int j = 0; j < CPL; ++j)
                ev[n][j] = __ldg(reinterpret_cast<const uint4*>(w1 + (int64_t)toks[n][k] * R) + s + 8 * j);
        ArgBest best[NF];
#pragma unroll
        for (int n = 0; n < NF; ++n) best[n] = {-INFINITY, INT_MAX};
        for (int base = 0; base < nrows; base += PASS) {
            float acc[NF][8];
            // the highest rows (read from global memory) first: their loads overlap the load of e
#pragma unroll
            for (int i = 7; i >= 0; --i) {
                const int li = base + grp + GROUPS * i;
                uint4 w[CPL];
                const int row0 = base + GROUPS * i;  // the first row of this 64-row block (warp-uniform)
                if (li < nc) {
#pragma unroll
                    for (int j = 0; j < CPL; ++j)
                        w[j] = *reinterpret_cast<const uint4*>(w2s + li * ROWB + (((s + 8 * j) ^ (li & 7)) * 16));
                } else if (NSTG > 0 && row0 >= nc && row0 < nrows) {
                    // (every thread of the CTA takes this branch for the block, so the group counts agree)
                    issue(qc + NSTG - 1);
                    asm volatile("cp.async.wait_group %0;" ::"n"(NSTG > 0 ? NSTG - 1 : 0) : "memory");
                    const uint8_t* rr = w2s + (size_t)n_cache * ROWB + (size_t)((qc % (NSTG > 0 ? NSTG : 1)) * 64 + grp) * ROWB;
#pragma unroll
                    for (int j = 0; j < CPL; ++j) w[j] = *reinterpret_cast<const uint4*>(rr + (s + 8 * j) * 16);
                    ++qc;
                } else if (li < nrows) {
                    const uint64_t pol = li < keep_end ? pol_keep : pol_pass;
#pragma unroll
                    for (int j = 0; j < CPL; ++j) w[j] = ld_nc_policy(w2g + (int64_t)li * CPR + s + 8 * j, pol);
                } else {
#pragma unroll
                    for (int j = 0; j < CPL; ++j) w[j] = make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int n = 0; n < NF; ++n) {
                    float a = 0.f;
#pragma unroll
                    for (int j = 0; j < CPL; ++j) a = fma_chunk(w[j], ev[n][j], a);
                    acc[n][i] = a;
                }
            }
            const int li = base + grp + GROUPS * s;
#pragma unroll
            for (int n = 0; n < NF; ++n) {
                const float dot = reduce_scatter8(acc[n], s);
                if (li < nrows) {
                    const int v = v_begin + li;
                    const float l = dot + uk[n * rows + li];
                    if (lg) lg[(int64_t)(n * gamma + k) * V + v] = l;
                    if (better(l, v, best[n].v, best[n].i)) {
                        best[n].v = l;
                        best[n].i = v;
                    }
                }
            }
        }
#pragma unroll
        for (int n = 0; n < NF; ++n) {
            const ArgBest wb = warp_argbest(best[n]);
            if (lane == 0) {
                red_v[n][warp] = wb.v;
                red_i[n][warp] = wb.i;
            }
        }
        __syncthreads();
        if (k + 1 < gamma) load_u(k + 1);  // its buffer was last read two positions ago
        asm volatile("cp.async.commit_group;" ::: "memory");
        if (warp < NF) {
            const int n = warp;
            unsigned long long* sl = slots + (size_t)(k * NF + n) * G;
            ArgBest cb{lane < NT_FMA / 32 ? red_v[n][lane] : -INFINITY, lane < NT_FMA / 32 ? red_i[n][lane] : INT_MAX};
            cb = warp_argbest(cb);
            if (lane == 0) {
                // a CTA without rows still arrives, with a word below every real one
                const unsigned long long key = cb.i != INT_MAX ? arg_key(cb.v, cb.i) : 1ull;
                if (cb.i != INT_MAX) {
                    const char* row = reinterpret_cast<const char*>(w1 + (int64_t)cb.i * R);
#pragma unroll
                    for (int o = 0; o < ROWB; o += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(row + o));
                }
                asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(sl + blockIdx.x), "l"(key) : "memory");
                asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(arrived + k * NF + n) : "memory");
            }
            // lane 0 waits (bounded) for every CTA's arrival, then the warp reads the words once
            bool timed_out = false;
            if (lane == 0) timed_out = wait_arrivals(arrived + k * NF + n, (unsigned long long)G);
            __syncwarp();
            unsigned long long m = 0ull;
            for (int c = lane; c < G; c += 32) {
                unsigned long long w;
                asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(sl + c) : "memory");
                m = w > m ? w : m;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long om = __shfl_xor_sync(0xffffffffu, m, o);
                m = om > m ? om : m;
            }
            if (lane == 0) {
                int tok = (int)(~(unsigned int)m);
                if (timed_out) atomicOr(p.err, 16);
                if (m <= 1ull || !(key_value(m) > -INFINITY) || tok < 0 || tok >= V) {
                    if (blockIdx.x == 0) atomicOr(p.err, 8);
                    tok = 0;
                }
                toks[n][k + 1] = tok;
                if (blockIdx.x == 0) p.tokens[n * gamma + k] = tok;
            }
        }
    }
    __syncthreads();
    // confidences: sigmoid(conf_w . [y_k ; w1[prev_k]] + conf_b), by CTA 0
    if (blockIdx.x == 0) {
        for (int b = 0; b < NF; ++b)
            for (int k = 0; k < gamma; ++k) {
                const float* yr = p.y + (int64_t)(b * gamma + k) * p.d;
                const bf16* er = w1 + (int64_t)toks[b][k] * R;
                float z = 0.f;
                for (int c = tid; c < p.d; c += NT_FMA) z = fmaf(yr[c], p.conf_w[c], z);
                for (int c = tid; c < R; c += NT_FMA) z = fmaf(to_f32(er[c]), p.conf_w[p.d + c], z);
                z = block_sum(z, redf);
                if (tid == 0) p.conf[b * gamma + k] = 1.f / (1.f + expf(-(z + p.conf_w[p.d + R])));
            }
        // every CTA read the parity before its first release add; CTA 0's last acquire follows them all
        if (tid == 0) atomicAdd(p.epoch, 1u);
    }
}

int g_res_ok[3] = {0, 0, 0};  // the resident chain's kernels for r = 64, 128, 256
int g_res_budget = 0;         // its dynamic shared memory
int g_l2_bytes = 0;           // the device's L2 size

bool g_fma_ok = false;         // the FMA chain's kernels

// Each bounded wait of the chains on words that nothing completes: one CTA, so the FMA chain's
// arrival count (target 1, nobody arrives), the resident chain's barrier and the cooperative
// chain's barrier (two CTAs expected) all give up after their limit and record the timeout.
__global__ void k_wait_selftest(int which, unsigned long long* w64, unsigned int* w32, int* err) {
    if (which == 0) {
        if (threadIdx.x == 0 && wait_arrivals(w64, 1ull)) atomicOr(err, 16);
    } else if (which == 1) {
        res_barrier(w64, 2ull, err);
    } else {
        grid_sync(w32, w32 + 1, 2u, err);
    }
}

template <int KD, int NF, int NSTG = 0>
cudaError_t fma_attr(int bytes) {
    return cudaFuncSetAttribute(k_markov_chain_fma<KD, NF, NSTG>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int KD>
cudaError_t res_attr(int bytes) {
    return cudaFuncSetAttribute(k_markov_chain_res<KD>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// E[b][:] = w1[prev_b] for the many-sequence form (prev_b = anchor at k = 0, else token k-1).
template <typename TW>
__global__ void k_markov_gather(const TW* __restrict__ w1, int r, int V, const int* __restrict__ anchors,
                                const int* __restrict__ tokens, int gamma, int k, TW* __restrict__ E) {
    pdl_wait();
    pdl_trigger();
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
    pdl_wait();
    pdl_trigger();
    __shared__ float red_v[NT / 32];
    __shared__ int red_i[NT / 32];
    __shared__ float redf[32];
    const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // every thread's first 32 partials are requested at once (one L2 round trip), the rest in turn
    const float* pv = part_v + (int64_t)b * nchunks;
    const int* pi = part_i + (int64_t)b * nchunks;
    float v[32];
    int iv[32];
#pragma unroll
    for (int q = 0; q < 32; ++q) {
        const int c = threadIdx.x + q * NT;
        v[q] = c < nchunks ? pv[c] : -INFINITY;
        iv[q] = c < nchunks ? pi[c] : INT_MAX;
    }
    ArgBest best{-INFINITY, INT_MAX};
#pragma unroll
    for (int q = 0; q < 32; ++q)
        if (better(v[q], iv[q], best.v, best.i)) best = ArgBest{v[q], iv[q]};
    for (int c = threadIdx.x + 32 * NT; c < nchunks; c += NT)
        if (better(pv[c], pi[c], best.v, best.i)) best = ArgBest{pv[c], pi[c]};
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
    if (p.r > RMAX || p.r % 8 != 0 || p.gamma > GMAX_CHAIN || !p.keys || !p.epoch || p.keys_stride < 16 * p.B)
        return cudaErrorInvalidValue;
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

bool markov_chain_resident_ok(const MarkovParams& p) {
    const int kd = p.r / 32;
    return p.w_dtype == DT_BF16 && p.B >= 1 && p.B <= NB_RES && p.r % 32 == 0 && (kd == 2 || kd == 4 || kd == 8) &&
           p.gamma >= 1 && p.gamma <= GMAX_CHAIN && p.keys && p.epoch && p.bar && p.keys_stride >= 16 * p.B &&
           g_res_ok[kd == 8 ? 2 : kd / 2 - 1];
}

cudaError_t markov_chain_resident_init() {
    int dev = 0, optin = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
    g_res_budget = (optin - 4096) / 16 * 16;  // static shared memory and headroom
    if ((e = cudaDeviceGetAttribute(&g_l2_bytes, cudaDevAttrL2CacheSize, dev)) != cudaSuccess) return e;
    g_res_ok[0] = res_attr<2>(g_res_budget) == cudaSuccess;
    g_res_ok[1] = res_attr<4>(g_res_budget) == cudaSuccess;
    g_res_ok[2] = res_attr<8>(g_res_budget) == cudaSuccess;
    g_fma_ok = fma_attr<2, 1>(g_res_budget) == cudaSuccess && fma_attr<2, 2>(g_res_budget) == cudaSuccess &&
               fma_attr<4, 1>(g_res_budget) == cudaSuccess && fma_attr<4, 2>(g_res_budget) == cudaSuccess &&
               fma_attr<8, 1>(g_res_budget) == cudaSuccess && fma_attr<8, 2>(g_res_budget) == cudaSuccess &&
               fma_attr<8, 1, RING_STAGES>(g_res_budget) == cudaSuccess;
    (void)cudaGetLastError();
    return cudaSuccess;
}

cudaError_t markov_chain_resident(const MarkovParams& p, int num_sms, cudaStream_t st) {
    if (!markov_chain_resident_ok(p)) return cudaErrorInvalidValue;
    const int kd = p.r / 32;
    // what the base-logit buffers leave of the budget holds resident rows
    const int rows = (p.V + num_sms - 1) / num_sms;
    const int ubytes = (2 * p.B * rows * 4 + 15) / 16 * 16;
    const int n_cache = std::max(0, std::min(rows, (g_res_budget - ubytes) / (p.r * 2)));
    const size_t smem = (size_t)n_cache * p.r * 2 + ubytes;
    if ((int)smem > g_res_budget) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(NT_RES);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (kd == 2) e = cudaLaunchKernelEx(&cfg, k_markov_chain_res<2>, p, n_cache);
    else if (kd == 4) e = cudaLaunchKernelEx(&cfg, k_markov_chain_res<4>, p, n_cache);
    else e = cudaLaunchKernelEx(&cfg, k_markov_chain_res<8>, p, n_cache);
    note_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t markov_wait_selftest(int which, void* scratch, int* err, cudaStream_t st) {
    if (which < 0 || which > 2 || !scratch || !err) return cudaErrorInvalidValue;
    k_wait_selftest<<<1, 64, 0, st>>>(which, reinterpret_cast<unsigned long long*>(scratch),
                                       reinterpret_cast<unsigned int*>(scratch) + 4, err);
    note_launch();
    return cudaGetLastError();
}

bool markov_chain_fma_ok(const MarkovParams& p, int num_sms) {
    const int kd = p.r / 32;
    return g_fma_ok && p.w_dtype == DT_BF16 && p.B >= 1 && p.B <= NB_FMA && p.r % 32 == 0 &&
           (kd == 2 || kd == 4 || kd == 8) && p.gamma >= 1 && p.gamma <= GMAX_CHAIN && p.keys && p.epoch &&
           (int64_t)p.keys_stride >= (int64_t)GMAX_CHAIN * p.B * (num_sms + 1);
}

cudaError_t markov_chain_fma(const MarkovParams& p, int num_sms, cudaStream_t st) {
    if (!markov_chain_fma_ok(p, num_sms)) return cudaErrorInvalidValue;
    const int kd = p.r / 32;
    const int rows = (p.V + num_sms - 1) / num_sms;
    const int ubytes = (2 * p.B * rows * 4 + 15) / 16 * 16;
    int n_cache = std::max(0, std::min(rows, (g_res_budget - ubytes) / (p.r * 2)));
    // Where most of a CTA's rows do not fit in shared memory, the rest stream through the ring form:
    // fewer resident rows (a multiple of 64) make room for the ring's blocks.
    const int ring_bytes = RING_STAGES * 64 * p.r * 2;
    const int n_cache_ring = std::max(0, (g_res_budget - ubytes - ring_bytes) / (p.r * 2)) & ~63;
    const bool ring = kd == 8 && p.B == 1 && rows - n_cache >= 6 * 64 && n_cache_ring > 0 &&
                      (rows - n_cache_ring + 63) / 64 <= MAX_SBLK;
    if (ring) n_cache = n_cache_ring;
    const size_t smem = (size_t)n_cache * p.r * 2 + (ring ? ring_bytes : 0) + ubytes;
    if ((int)smem > g_res_budget) return cudaErrorInvalidValue;
    // streamed rows kept in L2 across positions: 60% of L2 over the grid (the best of 25, 40, 60, 80%)
    const int n_keep = (int)std::min<int64_t>(rows, (int64_t)g_l2_bytes * 3 / 5 / ((int64_t)num_sms * p.r * 2));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // every CTA polls the others' words
    attr[0].val.cooperative = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(NT_FMA);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    const bool one = p.B == 1;
    if (kd == 2) e = one ? cudaLaunchKernelEx(&cfg, k_markov_chain_fma<2, 1>, p, n_cache, n_keep)
                         : cudaLaunchKernelEx(&cfg, k_markov_chain_fma<2, 2>, p, n_cache, n_keep);
    else if (kd == 4) e = one ? cudaLaunchKernelEx(&cfg, k_markov_chain_fma<4, 1>, p, n_cache, n_keep)
                              : cudaLaunchKernelEx(&cfg, k_markov_chain_fma<4, 2>, p, n_cache, n_keep);
    else if (ring) e = cudaLaunchKernelEx(&cfg, k_markov_chain_fma<8, 1, RING_STAGES>, p, n_cache, n_keep);
    else e = one ? cudaLaunchKernelEx(&cfg, k_markov_chain_fma<8, 1>, p, n_cache, n_keep)
                 : cudaLaunchKernelEx(&cfg, k_markov_chain_fma<8, 2>, p, n_cache, n_keep);
    note_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace dspark
