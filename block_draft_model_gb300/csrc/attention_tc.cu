// Block attention of a draft layer on the tensor cores, for a bf16 K/V cache
// ("module-dflash.ts", #layer: the gamma block queries attend bidirectionally
// over [context ++ block], scale head_dim^-1/2, no mask; the block's own K/V
// rows sit in the cache right after the context, so every key is a cache row).
//
// Same split-K flash-decoding structure as the SIMT kernel ("attention" and
// "combine" passes of "src/dspark-runtime.js", propose): the keys of one
// (sequence, head) are cut into ranges, one CTA each, and the last CTA of the
// (sequence, head), found with a ticket counter, merges the ranges in a fixed
// order.  Ranges are whole 64-key tiles, sized on the device from the actual
// length; CTAs past the last range exit at once.
//
// Inside a CTA (4 warps) the keys stream through a 3-stage cp.async ring of
// 64-key K and V tiles (rows padded by 16 bytes, so ldmatrix is conflict-free).
// Each warp owns 16 keys of every tile and keeps its own running softmax state,
// with the keys on the 16-row M side of mma.m16n8k16 and the block queries on
// its 8-wide N side (one or two tiles of 8):
//   S^T  = K Q^T  K fragments from ldmatrix, Q (pre-scaled by head_dim^-1/2
//                 log2 e, rounded to bf16) held in registers as B fragments;
//   P^T  = 2^(S^T - m)  in registers, rounded to bf16; movmatrix transposes
//                 each 8 x 8 block into the B fragment of the next product;
//   O^T += V^T P^T  V^T fragments from ldmatrix.trans of the V tile.
// The row sums add the bf16-rounded P, so every range's output is a convex
// combination of V rows.  At the end the four warps merge through shared
// memory into the range's (m, l, o) partial (log2 domain, rows of head_dim + 4
// floats so that the last CTA can stage them with 16-byte cp.async copies).
#include <limits.h>
#include <math.h>
#include <stdlib.h>

#include "common.cuh"
#include "kernels.cuh"

namespace dspark {

namespace {

constexpr int TK = 64;      // keys per tile
constexpr int NW = 4;       // warps per CTA, 16 keys of each tile per warp
constexpr int NT = NW * 32;
constexpr int GMAX = 16;    // queries per block (the M of the MMA)
constexpr int CMAX = 128;   // largest number of key ranges per (sequence, head)
constexpr int CL_MAX_TILES = 6;  // longest ranges (in 64-key tiles) merged as a cluster; longer ones keep the
                                 // deep ring and the ticketed merge, which their length amortises
constexpr int RFAST = 12;   // up to this many ranges the last CTA merges in one pass per thread
static_assert(NT == GMAX * 8, "the merge gives each query eight threads");

// NS: cp.async ring depth; 3 when two CTAs share an SM, 6 when one CTA has it alone
template <int HD, int NS>
struct TLayout {
    static constexpr int RB = HD * 2 + 16;  // padded bytes of one K or V row
    static constexpr int TILE = TK * RB;
    static constexpr int STAGE = 2 * TILE;  // K tile, then V tile
    static constexpr int BYTES = NS * STAGE;
    // after the key loop the ring is reused:
    //   this CTA's four warps: their outputs and (m, l)
    static constexpr int OWS = HD + 8;                      // padded row of a warp's output, floats
    static constexpr int OW = 0;                            // [NW][GMAX][OWS] fp32
    static constexpr int ML = OW + NW * GMAX * OWS * 4;     // [NW][GMAX] m, then [NW][GMAX] l
    static_assert(ML + 2 * NW * GMAX * 4 <= BYTES, "warp merge buffers must fit in the tile ring");
    //   the cluster form: this range's partial [GMAX][PW] (m, l, 2 unused, o[HD]), read by the cluster
    static constexpr int CP = ML + 2 * NW * GMAX * 4;
    //   the last CTA's merge of the ranges, staged piece by piece: per query the
    //   piece's range weights, the running (max, sum, rescale), then the partials
    static constexpr int PW = HD + 4;                       // partial row: m, l, 2 unused, o[HD] (16-byte rows)
    static constexpr int WM = 0;                            // [GMAX][CMAX] range weights of the piece
    static constexpr int MJ = WM + GMAX * CMAX * 4;         // [GMAX] running max, [GMAX] sum, [GMAX] rescale
    static constexpr int STG = MJ + 4 * GMAX * 4;           // staged partials (16-byte aligned)
    static_assert(STG + GMAX * PW * 4 <= BYTES, "one range of partials must fit beside the merge state");
    static_assert(CP + GMAX * PW * 4 <= BYTES, "the cluster partial must fit in the tile ring");
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}
// c[16x8] += a[16x16] . b[16x8], bf16 inputs, fp32 accumulators
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// 2^x (hardware approximation; 2^-inf = 0)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// (lo, hi) -> bf16x2 with lo in the low half; the rounded values are returned through lo/hi
__device__ __forceinline__ uint32_t pack_round(float& lo, float& hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    lo = __low2float(v);
    hi = __high2float(v);
    return *reinterpret_cast<uint32_t*>(&v);
}

template <typename TO>
__device__ __forceinline__ void store4(TO* dst, float a, float b, float c, float d);
template <>
__device__ __forceinline__ void store4<float>(float* dst, float a, float b, float c, float d) {
    *reinterpret_cast<float4*>(dst) = make_float4(a, b, c, d);
}
template <>
__device__ __forceinline__ void store4<bf16>(bf16* dst, float a, float b, float c, float d) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dst) = u;
}

// Copies of keys [t0, t0 + TK) into one ring stage; keys at or past `end` are zero-filled.  Only
// the rows whose key lies in [klo, khi) are touched (the default: every row).
template <int HD>
__device__ __forceinline__ void load_kv(uint32_t dst, const bf16* Kb, const bf16* Vb, int64_t stride, int t0,
                                        int end, int klo = INT_MIN, int khi = INT_MAX) {
    constexpr int RB = HD * 2 + 16, TILE = TK * RB;  // as in TLayout
    constexpr int VPR = HD * 2 / 16;
#pragma unroll 4
    for (int i = threadIdx.x; i < TK * VPR; i += NT) {
        const int r = i / VPR, v = i - r * VPR;
        const int key = t0 + r;
        if (key < klo || key >= khi) continue;
        const bool ok = key < end;
        const int64_t off = (int64_t)(ok ? key : t0) * stride + v * 8;
        const uint32_t so = r * RB + v * 16;
        cp_async16(dst + so, Kb + off, ok ? 16 : 0);
        cp_async16(dst + TILE + so, Vb + off, ok ? 16 : 0);
    }
}

// CL: the key ranges of one (sequence, head) are the CTAs of one thread-block cluster (grid.x =
// cluster size = n_chunks <= 16) and merge through distributed shared memory: no partials in global
// memory, no ticket, no restaging by a last CTA.
__device__ __forceinline__ void cluster_sync_release_acquire() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t laddr, int rank) {
    uint32_t ra;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(laddr), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
    return v;
}
__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t laddr, int rank) {
    uint32_t ra;
    float4 v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(laddr), "r"(rank));
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(ra)
                 : "memory");
    return v;
}

// NQ: tiles of 8 block queries (1 up to 8 queries, 2 up to 16)
template <int HD, typename TO, int NS, bool CL, int NQ>
__global__ void __launch_bounds__(NT, 2) k_attention_tc(AttnParams p) {
    using L = TLayout<HD, NS>;
    constexpr int KS = HD / 16;  // 16-wide head_dim steps of K Q^T; 16-row head_dim tiles of V^T P^T
    extern __shared__ __align__(128) uint8_t sm[];
    __shared__ int is_last;

    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gamma = p.gamma, d = p.d;
    // Up to pdl_wait() this kernel reads only what kernels at least two launches back wrote (the slot
    // map, the context lengths and the context rows of the cache): its predecessor, the projection
    // that wrote Q and the block's K/V rows, has passed its own wait before this kernel starts.
    const int slot = p.seq_ids ? p.seq_ids[b] : b;
    const int n_keys = slot < 0 ? 0 : p.seq_len[slot] + gamma;  // a rejected sequence has no keys
    TO* out = reinterpret_cast<TO*>(p.out) + (int64_t)b * gamma * d + h * HD;
    if (n_keys == 0) {
        pdl_wait();
        pdl_trigger();
        if (c == 0)
            for (int i = tid; i < gamma * (HD / 4); i += NT)
                store4<TO>(out + (int64_t)(i / (HD / 4)) * d + (i % (HD / 4)) * 4, 0.f, 0.f, 0.f, 0.f);
        return;
    }
    const int per = (n_keys + p.n_chunks - 1) / p.n_chunks;
    const int chunk = (per + TK - 1) / TK * TK;
    const int n_real = (n_keys + chunk - 1) / chunk;
    if (!CL && c >= n_real) {
        pdl_wait();
        pdl_trigger();
        return;
    }
    // (in the cluster form a CTA past the last range stays for the cluster barriers, with no keys)
    const int start = c * chunk, end = min(n_keys, start + chunk);
    const int n_tiles = c < n_real ? (end - start + TK - 1) / TK : 0;

    // K/V head of query head h, and the cache row width (grouped-query attention shares one K/V head
    // between n_heads / n_kv_heads query heads)
    const int dkv = p.d_kv ? p.d_kv : d;
    const int kvh = p.n_kv_heads ? h / (p.n_heads / p.n_kv_heads) : h;
    const bf16* Kb = reinterpret_cast<const bf16*>(p.cache) + (int64_t)slot * p.seq_stride + kvh * HD;
    const bf16* Vb = Kb + p.kv_off;
    const uint32_t ring = (uint32_t)__cvta_generic_to_shared(sm);
    const int n_ctx = n_keys - gamma;  // keys below this are context rows, written before the step
#pragma unroll
    for (int s = 0; s < NS - 1; ++s) {
        if (s < n_tiles) load_kv<HD>(ring + s * L::STAGE, Kb, Vb, dkv, start + s * TK, end, INT_MIN, n_ctx);
        cp_async_commit();
    }
    pdl_wait();
    pdl_trigger();
    // the block's own K/V rows of the tiles above (and the zero rows past the range end)
#pragma unroll
    for (int s = 0; s < NS - 1; ++s)
        if (s < n_tiles && start + (s + 1) * TK > n_ctx)
            load_kv<HD>(ring + s * L::STAGE, Kb, Vb, dkv, start + s * TK, end, n_ctx, INT_MAX);
    cp_async_commit();

    // Keys are the MMA's 16-row M side and the block queries its 8-wide N side (NQ tiles of 8), so
    // at most 8 queries no MMA column is spent on rows that do not exist:
    //   S^T = K Q^T  (A: 16 keys x 16 of head_dim from ldmatrix, B: Q^T from registers),
    //   O^T += V^T P^T  (A: 16 of head_dim x 16 keys, ldmatrix.trans of the V tile; B: P^T).
    // The S^T accumulator of each 8 x 8 (keys x queries) block is, once rounded to bf16 pairs, the
    // register layout of an 8 x 8 matrix; movmatrix transposes it into the B fragment of P^T.
    // Thread (g = lane / 4, cq = 2 * (lane % 4)) holds keys g, g + 8 and queries cq, cq + 1 of every
    // query tile; the per-query max is reduced over the 8 threads that share cq.
    const int g = lane >> 2, cq = (lane & 3) * 2;
    uint32_t qb[KS][NQ][2];  // B fragments of Q^T: query nq * 8 + g, head_dim ks * 16 + cq (+1) and + 8 (+9)
    {
        const float qs = rsqrtf((float)HD) * 1.4426950408889634f;
#pragma unroll
        for (int nq = 0; nq < NQ; ++nq) {
            const int qi = nq * 8 + g;
            const bool v = qi < gamma;
            const float* q0 = p.q + (int64_t)(b * gamma + (v ? qi : 0)) * d + h * HD;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int col = ks * 16 + cq;
                float2 x = v ? *reinterpret_cast<const float2*>(q0 + col) : make_float2(0.f, 0.f);
                float2 y = v ? *reinterpret_cast<const float2*>(q0 + col + 8) : make_float2(0.f, 0.f);
                float x0 = x.x * qs, x1 = x.y * qs, y0 = y.x * qs, y1 = y.y * qs;
                qb[ks][nq][0] = pack_round(x0, x1);
                qb[ks][nq][1] = pack_round(y0, y1);
            }
        }
    }

    float o[KS][NQ][4];  // O^T: head_dim ks * 16 + g (+8) x queries nq * 8 + cq (+1)
#pragma unroll
    for (int n = 0; n < KS; ++n)
#pragma unroll
        for (int nq = 0; nq < NQ; ++nq) o[n][nq][0] = o[n][nq][1] = o[n][nq][2] = o[n][nq][3] = 0.f;
    float mq[NQ][2], lq[NQ][2];  // queries nq * 8 + cq (+1): running max; this thread's keys' sum
#pragma unroll
    for (int nq = 0; nq < NQ; ++nq) mq[nq][0] = mq[nq][1] = -INFINITY, lq[nq][0] = lq[nq][1] = 0.f;

    // ldmatrix row addresses: lane -> matrix lane/8, row lane%8.  K as A (non-transposed): matrices
    // (keys 0-7 | 8-15) x (head_dim 0-7 | 8-15) in fragment order; V^T as A (transposed): the V rows
    // of keys 0-7 | 8-15, columns head_dim 0-7 | 8-15, in the order that transposes into fragments.
    const int lr = lane & 7, lm = lane >> 3, kw = warp * 16;
    const uint32_t k_lane = (uint32_t)((kw + (lm & 1) * 8 + lr) * L::RB + (lm >> 1) * 16);
    const uint32_t v_lane = (uint32_t)((kw + (lm >> 1) * 8 + lr) * L::RB + (lm & 1) * 16);

    for (int t = 0; t < n_tiles; ++t) {
        if (t == 0) cp_async_wait<0>();  // the first tiles' context and block rows came in two groups
        else cp_async_wait<NS - 2>();
        __syncthreads();  // tile t is visible; every warp is done with tile t-1, whose stage is refilled next
        {
            const int tn = t + NS - 1;
            if (tn < n_tiles) load_kv<HD>(ring + (tn % NS) * L::STAGE, Kb, Vb, dkv, start + tn * TK, end);
            cp_async_commit();
        }
        const int nk = min(TK, end - (start + t * TK));
        if (kw >= nk) continue;
        const uint32_t kbase = ring + (t % NS) * L::STAGE;
        const uint32_t vbase = kbase + L::TILE;

        float s[NQ][4];
#pragma unroll
        for (int nq = 0; nq < NQ; ++nq) s[nq][0] = s[nq][1] = s[nq][2] = s[nq][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint32_t ka[4];
            ldsm_x4(kbase + k_lane + ks * 32, ka[0], ka[1], ka[2], ka[3]);
#pragma unroll
            for (int nq = 0; nq < NQ; ++nq) mma16816(s[nq], ka, qb[ks][nq][0], qb[ks][nq][1]);
        }
        if (kw + 16 > nk) {  // keys past the range end (zero rows) take no weight
#pragma unroll
            for (int nq = 0; nq < NQ; ++nq) {
                if (kw + g >= nk) s[nq][0] = s[nq][1] = -INFINITY;
                if (kw + g + 8 >= nk) s[nq][2] = s[nq][3] = -INFINITY;
            }
        }
        uint32_t pb[NQ][2];
        float al[NQ][2];
#pragma unroll
        for (int nq = 0; nq < NQ; ++nq) {
            float mx0 = fmaxf(s[nq][0], s[nq][2]), mx1 = fmaxf(s[nq][1], s[nq][3]);
#pragma unroll
            for (int o2 = 4; o2 < 32; o2 <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o2));
            }
            const float mn0 = fmaxf(mq[nq][0], mx0), mn1 = fmaxf(mq[nq][1], mx1);
            const float ms0 = mn0 == -INFINITY ? 0.f : mn0, ms1 = mn1 == -INFINITY ? 0.f : mn1;
            al[nq][0] = ex2(mq[nq][0] - ms0);
            al[nq][1] = ex2(mq[nq][1] - ms1);
            mq[nq][0] = mn0;
            mq[nq][1] = mn1;
            float p0 = ex2(s[nq][0] - ms0), p1 = ex2(s[nq][1] - ms1);  // key g:     queries cq, cq+1
            float p2 = ex2(s[nq][2] - ms0), p3 = ex2(s[nq][3] - ms1);  // key g + 8: queries cq, cq+1
            const uint32_t x0 = pack_round(p0, p1), x1 = pack_round(p2, p3);
            lq[nq][0] = lq[nq][0] * al[nq][0] + (p0 + p2);
            lq[nq][1] = lq[nq][1] * al[nq][1] + (p1 + p3);
            asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(pb[nq][0]) : "r"(x0));
            asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(pb[nq][1]) : "r"(x1));
        }
#pragma unroll
        for (int n = 0; n < KS; ++n)
#pragma unroll
            for (int nq = 0; nq < NQ; ++nq) {
                o[n][nq][0] *= al[nq][0];
                o[n][nq][1] *= al[nq][1];
                o[n][nq][2] *= al[nq][0];
                o[n][nq][3] *= al[nq][1];
            }
#pragma unroll
        for (int n = 0; n < KS; ++n) {
            uint32_t va[4];
            ldsm_x4_t(vbase + v_lane + n * 32, va[0], va[1], va[2], va[3]);
#pragma unroll
            for (int nq = 0; nq < NQ; ++nq) mma16816(o[n][nq], va, pb[nq][0], pb[nq][1]);
        }
    }
    cp_async_wait<0>();
    __syncthreads();  // the ring is free for the merge buffers

    // ---- merge the four warps into this range's partial
    float* Ow = reinterpret_cast<float*>(sm + L::OW);
    float* Mw = reinterpret_cast<float*>(sm + L::ML);
    float* Lw = Mw + NW * GMAX;
#pragma unroll
    for (int nq = 0; nq < NQ; ++nq) {
        float l0 = lq[nq][0], l1 = lq[nq][1];
#pragma unroll
        for (int o2 = 4; o2 < 32; o2 <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, o2);
            l1 += __shfl_xor_sync(0xffffffffu, l1, o2);
        }
        const int q0 = warp * GMAX + nq * 8 + cq;
#pragma unroll
        for (int n = 0; n < KS; ++n) {
            Ow[q0 * L::OWS + n * 16 + g] = o[n][nq][0];
            Ow[(q0 + 1) * L::OWS + n * 16 + g] = o[n][nq][1];
            Ow[q0 * L::OWS + n * 16 + g + 8] = o[n][nq][2];
            Ow[(q0 + 1) * L::OWS + n * 16 + g + 8] = o[n][nq][3];
        }
        if (g == 0) {
            Mw[q0] = mq[nq][0];
            Mw[q0 + 1] = mq[nq][1];
            Lw[q0] = l0;
            Lw[q0 + 1] = l1;
        }
    }
    __syncthreads();

    constexpr int w = L::PW;
    const int64_t bh = (int64_t)b * p.n_heads + h;
    if (CL && n_real > 1) {
        // this range's partial into shared memory, then the cluster merges every range's partial
        float* cp = reinterpret_cast<float*>(sm + L::CP);
        for (int i = tid; i < gamma * (HD / 4); i += NT) {
            const int j = i / (HD / 4), e = (i % (HD / 4)) * 4;
            float M = -INFINITY;
#pragma unroll
            for (int v = 0; v < NW; ++v) M = fmaxf(M, Mw[v * GMAX + j]);
            float l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int v = 0; v < NW; ++v) {
                const float mv = Mw[v * GMAX + j];
                const float wt = mv == -INFINITY ? 0.f : ex2(mv - M);
                l += wt * Lw[v * GMAX + j];
                const float4 ov = *reinterpret_cast<const float4*>(Ow + (v * GMAX + j) * L::OWS + e);
                acc[0] += wt * ov.x;
                acc[1] += wt * ov.y;
                acc[2] += wt * ov.z;
                acc[3] += wt * ov.w;
            }
            *reinterpret_cast<float4*>(cp + j * w + 4 + e) = make_float4(acc[0], acc[1], acc[2], acc[3]);
            if (e == 0) *reinterpret_cast<float2*>(cp + j * w) = make_float2(M, l);
        }
        cluster_sync_release_acquire();  // every range's partial is written and visible to the cluster
        const uint32_t cpa = (uint32_t)__cvta_generic_to_shared(cp);
        for (int i = c * NT + tid; i < gamma * (HD / 4); i += (int)gridDim.x * NT) {
            const int j = i / (HD / 4), e = (i % (HD / 4)) * 4;
            float M = -INFINITY;
            for (int q = 0; q < n_real; ++q) M = fmaxf(M, ld_cluster_f32(cpa + j * w * 4, q));
            const float Ms = M == -INFINITY ? 0.f : M;
            float l = 0.f, a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
            for (int q = 0; q < n_real; ++q) {
                const float mq = ld_cluster_f32(cpa + j * w * 4, q);
                const float lq = ld_cluster_f32(cpa + (j * w + 1) * 4, q);
                const float4 x = ld_cluster_f32x4(cpa + (j * w + 4 + e) * 4, q);
                const float wt = mq == -INFINITY ? 0.f : ex2(mq - Ms);
                l = fmaf(wt, lq, l);
                a0 = fmaf(wt, x.x, a0);
                a1 = fmaf(wt, x.y, a1);
                a2 = fmaf(wt, x.z, a2);
                a3 = fmaf(wt, x.w, a3);
            }
            const float inv = 1.f / l;  // every range holds at least one key, so the sum is >= 1
            store4<TO>(out + (int64_t)j * d + e, a0 * inv, a1 * inv, a2 * inv, a3 * inv);
        }
        // no CTA leaves while another may still read its partial
        asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
        return;
    }
    if (CL && c >= n_real) return;  // one range: the first CTA writes the output on its own
    float* part = p.part + (bh * p.n_chunks + c) * gamma * w;
    for (int i = tid; i < gamma * (HD / 4); i += NT) {
        const int j = i / (HD / 4), e = (i % (HD / 4)) * 4;
        float M = -INFINITY;
#pragma unroll
        for (int v = 0; v < NW; ++v) M = fmaxf(M, Mw[v * GMAX + j]);
        float l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int v = 0; v < NW; ++v) {
            const float mv = Mw[v * GMAX + j];
            const float wt = mv == -INFINITY ? 0.f : ex2(mv - M);
            l += wt * Lw[v * GMAX + j];
            const float4 ov = *reinterpret_cast<const float4*>(Ow + (v * GMAX + j) * L::OWS + e);
            acc[0] += wt * ov.x;
            acc[1] += wt * ov.y;
            acc[2] += wt * ov.z;
            acc[3] += wt * ov.w;
        }
        if (n_real == 1) {
            const float inv = 1.f / l;  // the range holds at least one key, so l >= 1
            store4<TO>(out + (int64_t)j * d + e, acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
        } else {
            *reinterpret_cast<float4*>(part + j * w + 4 + e) = make_float4(acc[0], acc[1], acc[2], acc[3]);
            if (e == 0) *reinterpret_cast<float2*>(part + j * w) = make_float2(M, l);
        }
    }
    if (n_real == 1) return;
    if constexpr (CL) return;  // (the cluster form has merged above; no ticketed merge in its code)
    // Ticket: after the barrier, one acquire-release atomic publishes this CTA's
    // partial (release, cumulative over the barrier) and, in the last CTA, makes
    // every other CTA's partial visible (acquire, passed on by the next barrier).
    __syncthreads();
    if (tid == 0) {
        unsigned int prev;
        asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;" : "=r"(prev) : "l"(p.tickets + bh) : "memory");
        is_last = prev == (unsigned int)n_real - 1;
    }
    __syncthreads();
    if (!is_last) return;

    // ---- last CTA of (b, h): merge the n_real ranges in order.  The partials
    // (m, l and o of every query) are staged into shared memory with cp.async,
    // as many ranges as fit per piece (usually all: one round trip), and merged
    // piece by piece with a running max, sum and rescale per query.
    const float* all = p.part + bh * p.n_chunks * gamma * w;  // range cc, query j at (cc * gamma + j) * w
    constexpr int ITEMS = (GMAX * (HD / 4) + NT - 1) / NT;  // (query, 4 columns) items per thread
    const int rbytes = gamma * w * 4;
    const uint32_t stg = ring + L::STG;
    const float* S = reinterpret_cast<const float*>(sm + L::STG);
    if (n_real <= RFAST && n_real <= (L::BYTES - L::STG) / rbytes) {
        // Few ranges: one staging round trip, then each thread merges its own items over the
        // ranges (two passes over the (m, l) pairs, no shared weight tables, no further block
        // barriers).  The loops stay rolled: this code runs once per launch, cold in the
        // instruction cache, and unrolled it is slower to fetch than to execute.  With more
        // ranges the per-thread chain grows long and the piecewise merge below, which spreads
        // the ranges of a query over eight threads, is faster.
        const char* src = reinterpret_cast<const char*>(all);
        for (int i = tid; i < n_real * rbytes / 16; i += NT) cp_async16(stg + i * 16, src + i * 16, 16);
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
#pragma unroll 1
        for (int k = 0; k < ITEMS; ++k) {
            const int i = tid + k * NT;
            if (i < gamma * (HD / 4)) {
                const int j = i / (HD / 4), e = (i % (HD / 4)) * 4;
                const float* sj = S + j * w;  // range cc at sj + cc * gamma * w
                const int cs = gamma * w;
                float M = -INFINITY;
#pragma unroll 1
                for (int cc = 0; cc < n_real; ++cc) M = fmaxf(M, sj[cc * cs]);
                const float Ms = M == -INFINITY ? 0.f : M;
                float l = 0.f, a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 1
                for (int cc = 0; cc < n_real; ++cc) {
                    const float2 ml = *reinterpret_cast<const float2*>(sj + cc * cs);
                    const float4 x = *reinterpret_cast<const float4*>(sj + cc * cs + 4 + e);
                    const float wt = ml.x == -INFINITY ? 0.f : ex2(ml.x - Ms);
                    l = fmaf(wt, ml.y, l);
                    a0 = fmaf(wt, x.x, a0);
                    a1 = fmaf(wt, x.y, a1);
                    a2 = fmaf(wt, x.z, a2);
                    a3 = fmaf(wt, x.w, a3);
                }
                const float inv = 1.f / l;  // every range holds at least one key, so the sum is >= 1
                store4<TO>(out + (int64_t)j * d + e, a0 * inv, a1 * inv, a2 * inv, a3 * inv);
            }
        }
        if (tid == 0) p.tickets[bh] = 0u;
        return;
    }
    float* Wm = reinterpret_cast<float*>(sm + L::WM);
    float* Mj = reinterpret_cast<float*>(sm + L::MJ);
    float* Lj = Mj + GMAX;
    float* Sc = Lj + GMAX;
    if (tid < GMAX) {
        Mj[tid] = -INFINITY;
        Lj[tid] = 0.f;
    }
    float acc[ITEMS][4];
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) acc[k][0] = acc[k][1] = acc[k][2] = acc[k][3] = 0.f;
    const int fit = min((L::BYTES - L::STG) / rbytes, CMAX);
    for (int c0 = 0; c0 < n_real; c0 += fit) {
        const int nr = min(fit, n_real - c0);
        __syncthreads();  // the previous piece has been consumed
        const char* src = reinterpret_cast<const char*>(all + (int64_t)c0 * gamma * w);
        for (int i = tid; i < nr * rbytes / 16; i += NT) cp_async16(stg + i * 16, src + i * 16, 16);
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
        {
            // per query j: eight threads (one per range residue mod 8) find the piece's max and sum
            const int j = tid >> 3, sub = tid & 7;
            const bool qv = j < gamma;
            float pm = -INFINITY;
            if (qv)
                for (int cc = sub; cc < nr; cc += 8) pm = fmaxf(pm, S[(cc * gamma + j) * w]);
            pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 1));
            pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 2));
            pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 4));
            const float m_old = qv ? Mj[j] : -INFINITY, m_new = fmaxf(m_old, pm);
            const float ms = m_new == -INFINITY ? 0.f : m_new;
            float lsum = 0.f;
            if (qv)
                for (int cc = sub; cc < nr; cc += 8) {
                    const float2 ml = *reinterpret_cast<const float2*>(S + (cc * gamma + j) * w);
                    const float wt = ml.x == -INFINITY ? 0.f : ex2(ml.x - ms);
                    Wm[j * CMAX + cc] = wt;
                    lsum += wt * ml.y;
                }
            lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
            lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
            lsum += __shfl_xor_sync(0xffffffffu, lsum, 4);
            if (qv && sub == 0) {
                const float sc = m_old == -INFINITY ? 0.f : ex2(m_old - ms);
                Sc[j] = sc;
                Lj[j] = Lj[j] * sc + lsum;
                Mj[j] = m_new;
            }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < ITEMS; ++k) {
            const int i = tid + k * NT;
            if (i < gamma * (HD / 4)) {
                const int j = i / (HD / 4), e = (i % (HD / 4)) * 4;
                const float sc = Sc[j];
                float a0 = acc[k][0] * sc, a1 = acc[k][1] * sc, a2 = acc[k][2] * sc, a3 = acc[k][3] * sc;
                const float* wj = Wm + j * CMAX;
                const float* sj = S + j * w + 4 + e;  // range cc at sj + cc * gamma * w
                const int cs = gamma * w;
                float b0 = 0.f, b1 = 0.f, b2 = 0.f, b3 = 0.f;  // second accumulator set: two chains
                int cc = 0;
                for (; cc + 2 <= nr; cc += 2) {
                    const float w0 = wj[cc], w1 = wj[cc + 1];
                    const float4 x = *reinterpret_cast<const float4*>(sj + cc * cs);
                    const float4 y = *reinterpret_cast<const float4*>(sj + (cc + 1) * cs);
                    a0 = fmaf(w0, x.x, a0);
                    a1 = fmaf(w0, x.y, a1);
                    a2 = fmaf(w0, x.z, a2);
                    a3 = fmaf(w0, x.w, a3);
                    b0 = fmaf(w1, y.x, b0);
                    b1 = fmaf(w1, y.y, b1);
                    b2 = fmaf(w1, y.z, b2);
                    b3 = fmaf(w1, y.w, b3);
                }
                if (cc < nr) {
                    const float w0 = wj[cc];
                    const float4 x = *reinterpret_cast<const float4*>(sj + cc * cs);
                    a0 = fmaf(w0, x.x, a0);
                    a1 = fmaf(w0, x.y, a1);
                    a2 = fmaf(w0, x.z, a2);
                    a3 = fmaf(w0, x.w, a3);
                }
                acc[k][0] = a0 + b0;
                acc[k][1] = a1 + b1;
                acc[k][2] = a2 + b2;
                acc[k][3] = a3 + b3;
            }
        }
    }
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
        const int i = tid + k * NT;
        if (i < gamma * (HD / 4)) {
            const int j = i / (HD / 4), e = (i % (HD / 4)) * 4;
            const float inv = 1.f / Lj[j];  // every range holds at least one key, so the sum is >= 1
            store4<TO>(out + (int64_t)j * d + e, acc[k][0] * inv, acc[k][1] * inv, acc[k][2] * inv, acc[k][3] * inv);
        }
    }
    if (tid == 0) p.tickets[bh] = 0u;
}

template <int HD, typename TO, int NS, int NQ>
cudaError_t set_attr_tc_q() {
    cudaError_t e = cudaFuncSetAttribute(k_attention_tc<HD, TO, NS, false, NQ>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, TLayout<HD, NS>::BYTES);
    if (e != cudaSuccess || NS != 3) return e;
    e = cudaFuncSetAttribute(k_attention_tc<HD, TO, 3, true, NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             TLayout<HD, 3>::BYTES);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k_attention_tc<HD, TO, 3, true, NQ>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}
template <int HD, typename TO, int NS>
cudaError_t set_attr_tc() {
    cudaError_t e = set_attr_tc_q<HD, TO, NS, 1>();
    return e != cudaSuccess ? e : set_attr_tc_q<HD, TO, NS, 2>();
}

int g_num_sms = 0;
// largest key-range count launched as one cluster (0: the cluster form is off); set at init from
// how many clusters of that size the device can hold at once
int g_cluster_max = 0;

template <int HD, typename TO, int NQ>
void launch_tc(const AttnParams& p, dim3 grid, cudaStream_t st) {
    // A grid that fits one CTA per SM gives each CTA the SM's whole shared memory: a deeper ring,
    // where the ranges are long enough to use it.  Ranges of a few tiles keep the 3-stage ring, so
    // that the next kernel's CTAs (launched early, programmatic dependent launch) fit beside them.
    const int per_range = p.max_keys > 0 ? (p.max_keys + (int)grid.x * TK - 1) / ((int)grid.x * TK) : 1 << 30;
    if (grid.x >= 2 && (int)grid.x <= g_cluster_max && per_range <= CL_MAX_TILES) {
        // the ranges of one (sequence, head) as one cluster, merged through distributed shared memory
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = grid.x;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(NT);
        cfg.dynamicSmemBytes = TLayout<HD, 3>::BYTES;
        cfg.stream = st;
        cfg.attrs = attr;
        cfg.numAttrs = pdl_enabled() ? 2 : 1;
        cudaLaunchKernelEx(&cfg, k_attention_tc<HD, TO, 3, true, NQ>, p);
    } else if ((int)(grid.x * grid.y * grid.z) <= g_num_sms && per_range > 2) {
        launch(k_attention_tc<HD, TO, 6, false, NQ>, grid, NT, (size_t)TLayout<HD, 6>::BYTES, st, p);
    } else {
        launch(k_attention_tc<HD, TO, 3, false, NQ>, grid, NT, (size_t)TLayout<HD, 3>::BYTES, st, p);
    }
}

}  // namespace

bool attention_tc_ok(int cache_dtype, int head_dim, int gamma) {
    return cache_dtype == DT_BF16 && (head_dim == 64 || head_dim == 128) && gamma >= 1 && gamma <= GMAX;
}

int attention_tc_max_chunks() { return CMAX; }

int attention_tc_cluster_chunks(int max_keys) {
    if (g_cluster_max < 2) return 0;
    const int per_range = (max_keys + g_cluster_max * TK - 1) / (g_cluster_max * TK);
    return per_range <= CL_MAX_TILES ? g_cluster_max : 0;
}

cudaError_t attention_tc_init() {
    cudaError_t e;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = set_attr_tc<64, bf16, 3>()) != cudaSuccess) return e;
    if ((e = set_attr_tc<64, float, 3>()) != cudaSuccess) return e;
    if ((e = set_attr_tc<128, bf16, 3>()) != cudaSuccess) return e;
    if ((e = set_attr_tc<128, float, 3>()) != cudaSuccess) return e;
    if ((e = set_attr_tc<64, bf16, 6>()) != cudaSuccess) return e;
    if ((e = set_attr_tc<64, float, 6>()) != cudaSuccess) return e;
    if ((e = set_attr_tc<128, bf16, 6>()) != cudaSuccess) return e;
    if ((e = set_attr_tc<128, float, 6>()) != cudaSuccess) return e;
    // the largest cluster of the short-range form that the device can hold (16, else the portable 8)
    g_cluster_max = 0;
    for (int n : {16, 8}) {
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = n;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(n, 1, 1);
        cfg.blockDim = dim3(NT);
        cfg.dynamicSmemBytes = TLayout<128, 3>::BYTES;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, k_attention_tc<128, float, 3, true, 2>, &cfg) == cudaSuccess &&
            clusters >= 1) {
            g_cluster_max = n;
            break;
        }
    }
    (void)cudaGetLastError();  // a refused probe leaves nothing behind
    return cudaSuccess;
}

cudaError_t attention_tc(const AttnParams& p, cudaStream_t st) {
    const int hd = p.d / p.n_heads;
    if (!attention_tc_ok(p.cache_dtype, hd, p.gamma) || p.n_chunks < 1 || p.n_chunks > CMAX ||
        (p.out_dtype != DT_BF16 && p.out_dtype != DT_F32))
        return cudaErrorInvalidValue;
    dim3 grid(p.n_chunks, p.n_heads, p.B);
    const bool o16 = p.out_dtype == DT_BF16;
    const bool q8 = p.gamma <= 8;
    if (hd == 64) {
        if (o16) q8 ? launch_tc<64, bf16, 1>(p, grid, st) : launch_tc<64, bf16, 2>(p, grid, st);
        else q8 ? launch_tc<64, float, 1>(p, grid, st) : launch_tc<64, float, 2>(p, grid, st);
    } else {
        if (o16) q8 ? launch_tc<128, bf16, 1>(p, grid, st) : launch_tc<128, bf16, 2>(p, grid, st);
        else q8 ? launch_tc<128, float, 1>(p, grid, st) : launch_tc<128, float, 2>(p, grid, st);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace dspark
