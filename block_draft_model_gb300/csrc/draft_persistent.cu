// All draft layers of one sequence in one persistent launch ("module-dflash.ts",
// #layer: pre-norm bidirectional block attention over [context ++ block] and a
// SwiGLU FFN, each with a residual add; "src/dspark-runtime.js", propose).
//
// One cooperative CTA per SM.  Each layer runs as phases separated by bounded
// grid barriers:
//   A  x -> RMSNorm * attn_norm (every CTA, into shared memory); the CTA's
//      16-row tiles of [Wq; Wk; Wv]: Q rows to q, K/V rows into the cache
//   B  attention: work item (head, key range) per CTA, flash-decoding partials
//   C  merge of the key ranges (skipped when one range covers the keys)
//   D  O projection, residual add into x
//   E  x -> RMSNorm * ff_norm; [gate; up] tiles, SwiGLU into hact
//   F  down projection, residual add into x
// The projections are weight streams with at most 16 activation rows, so the
// weight rows are the M side of mma.m16n8k16 and the block rows the N side
// ("swap AB").  A producer warp streams every weight tile of every layer, in
// the order the CTA consumes them, into a ring of shared-memory slots with
// bulk copies (one per 16-row tile row and 512-element K slice, rows padded by
// 16 bytes); it never waits for a grid barrier, so the weights of the next
// phases arrive while the CTA waits for the other CTAs.  Eight consumer warps
// take the CTA's tiles of a phase in turn.  Inside each 32-wide slice of K
// the K order is permuted so that a lane's A fragments for two k-steps are one
// 16-byte chunk of a weight row and its B fragments one chunk of an
// activation row (the same permutation on both sides leaves the products
// unchanged); activation rows in shared memory have their chunks
// XOR-swizzled by row.  Every wait is bounded (about a second); a timeout
// sets DSPARK_DEVERR_TIMEOUT and every role drains and returns.
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.cuh"
#include "tc_common.cuh"

namespace dspark {

namespace {

using namespace tc;

constexpr int NCW = 8;                  // consumer warps
constexpr int NTP = (NCW + 1) * 32;     // plus the producer warp
constexpr int KSLOT = 512;              // K elements of one ring slot
constexpr int SLOT_BYTES = 16 * KSLOT * 2;  // a 16-row tile slice: 8 blocks of [16 rows][64], 128-byte swizzle
constexpr int MAXL = 16;
constexpr int TKA = 64;                 // attention keys per tile
constexpr int GMAXP = 16;               // block rows
constexpr int MAXCH = 32;               // key ranges per head

struct PersistParams {
    float* x;        // [gamma, d] residual
    float* q;        // [gamma, d]
    bf16* act;       // [gamma, d] attention output
    bf16* hact;      // [gamma, F] SwiGLU output
    float* part;     // [nh][nchunks][gamma][hd + 4] attention partials
    bf16* cache;     // layer 0, slot 0: K rows at + pos * d, V rows at + kv_off
    int64_t layer_stride, kv_off;
    int max_rows;    // cache rows per sequence
    const int* seq_len;
    const bf16* wqkv[MAXL];
    const bf16* wo[MAXL];
    const bf16* wgu[MAXL];
    const bf16* wd[MAXL];
    const float* attn_norm[MAXL];
    const float* ff_norm[MAXL];
    int d, F, nh, nL, gamma, act_kind, nchunks, nslot, xs_bytes;
    float eps;
    const CUtensorMap* maps;  // [n_layers][4] slot maps of wqkv, wo, wgu, wd (global memory)
    int map3d;                // one 3-D copy per slot, else eight 2-D copies
    unsigned long long* bar;  // 2 arrival counters (launch parity)
    unsigned int* epoch;
    int* err;
};

__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ void cons_sync() { named_sync(1, NCW * 32); }
__device__ __forceinline__ void attn_sync() { named_sync(2, 128); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16z(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void tma3d(uint32_t dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
            dst),
        "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
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
__device__ __forceinline__ void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// the two k-steps held by one 16-byte chunk of weight rows g, g+8 (lo, hi) and of activation row g
__device__ __forceinline__ void mma_chunk(float* c, const uint4& lo, const uint4& hi, const uint4& xv) {
    mma16816(c, lo.x, hi.x, lo.y, hi.y, xv.x, xv.y);
    mma16816(c, lo.z, hi.z, lo.w, hi.w, xv.z, xv.w);
}
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t pack_round(float& lo, float& hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    lo = __low2float(v);
    hi = __high2float(v);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Grid barrier among the consumer warps of every CTA: a 64-bit arrival counter
// that counts up through the launch (barrier number `n` opens at n * gridDim.x).
__device__ __forceinline__ void grid_barrier(unsigned long long* bar, unsigned long long target, int* err,
                                             volatile int* abort_flag) {
    cons_sync();
    if (threadIdx.x == 0) {
        asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(bar) : "memory");
        const uint64_t t0 = globaltimer();
        while (true) {
            unsigned long long cur;
            asm volatile("ld.acquire.gpu.u64 %0, [%1];" : "=l"(cur) : "l"(bar) : "memory");
            if (cur >= target || *abort_flag) break;
            if (globaltimer() - t0 > TIMEOUT_NS) {
                atomicOr(err, DEVERR_TIMEOUT);
                *abort_flag = 1;
                break;
            }
        }
    }
    cons_sync();
}

// Tiles of a projection phase that CTA c owns: c, c + G, c + 2G, ... below n_tiles.
__device__ __forceinline__ int my_tiles(int n_tiles, int c, int G) { return n_tiles > c ? (n_tiles - 1 - c) / G + 1 : 0; }

enum Phase { PH_QKV = 0, PH_O = 1, PH_GU = 2, PH_D = 3 };

__device__ __forceinline__ void phase_shape(const PersistParams& p, int layer, int ph, const bf16*& W, int& N,
                                            int& K) {
    if (ph == PH_QKV) {
        W = p.wqkv[layer];
        N = 3 * p.d;
        K = p.d;
    } else if (ph == PH_O) {
        W = p.wo[layer];
        N = p.d;
        K = p.d;
    } else if (ph == PH_GU) {
        W = p.wgu[layer];
        N = 2 * p.F;
        K = p.d;
    } else {
        W = p.wd[layer];
        N = p.d;
        K = p.F;
    }
}

// Activation rows [gamma, K] bf16 from global into the swizzled staging area
// (rows gamma .. 8*NT-1 zeroed); chunk c of row n at n * K * 2 + ((c ^ (n & 7)) * 16).
template <int NT>
__device__ __forceinline__ void stage_rows(uint8_t* xs, const bf16* src, int K, int gamma) {
    const int cpr = K / 8;
    const uint32_t xs_s = smem_u32(xs);
    for (int i = threadIdx.x; i < NT * 8 * cpr; i += NCW * 32) {
        const int n = i / cpr, c = i - n * cpr;
        const uint32_t dst = xs_s + n * K * 2 + ((c ^ (n & 7)) * 16);
        if (n < gamma) cp_async16(dst, src + (int64_t)n * K + c * 8);
        else *reinterpret_cast<uint4*>(xs + n * K * 2 + ((c ^ (n & 7)) * 16)) = make_uint4(0, 0, 0, 0);
    }
    cp_commit();
    cp_wait<0>();
    cons_sync();
}

// RMSNorm(x) * w of the gamma block rows into the swizzled staging area (bf16);
// a warp per row, the row held in registers (d <= 32 * 4 * DMAXV).
constexpr int DMAXV = 16;
template <int NT>
__device__ __forceinline__ void stage_norm(uint8_t* xs, const float* x, const float* w, int d, int gamma, float eps) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nv = d / 4;
    for (int n = warp; n < NT * 8; n += NCW) {
        uint8_t* row = xs + n * d * 2;
        if (n >= gamma) {
            for (int e4 = lane; e4 < nv; e4 += 32)
                *reinterpret_cast<uint2*>(row + (((e4 >> 1) ^ (n & 7)) * 16) + (e4 & 1) * 8) = make_uint2(0, 0);
            continue;
        }
        const float4* xr = reinterpret_cast<const float4*>(x + (int64_t)n * d);
        float4 v[DMAXV];
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < DMAXV; ++i) {
            const int e4 = lane + 32 * i;
            v[i] = e4 < nv ? __ldcg(xr + e4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < DMAXV; ++i) ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
        ss = warp_sum(ss);
        const float rs = rsqrtf(ss / (float)d + eps);
        const float4* w4 = reinterpret_cast<const float4*>(w);
#pragma unroll
        for (int i = 0; i < DMAXV; ++i) {
            const int e4 = lane + 32 * i;
            if (e4 < nv) {
                const float4 g = w4[e4];
                *reinterpret_cast<uint2*>(row + (((e4 >> 1) ^ (n & 7)) * 16) + (e4 & 1) * 8) =
                    make_uint2(pack2(v[i].x * rs * g.x, v[i].y * rs * g.y), pack2(v[i].z * rs * g.z, v[i].w * rs * g.w));
            }
        }
    }
    cons_sync();
}

// One ring slot (16 weight rows x KSLOT) against the staged activations,
// accumulated into c; two accumulator chains (even and odd k slices).
template <int NT>
__device__ __forceinline__ void slot_mma(float (&c)[NT][4], const uint8_t* sb, int ks, int K, const uint8_t* xs) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    float c2[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) c2[n][0] = c2[n][1] = c2[n][2] = c2[n][3] = 0.f;
#pragma unroll 4
    for (int j = 0; j < KSLOT / 32; j += 2) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int ch = 4 * (j + u) + t;  // 16-byte chunk of the slice: block ch / 8, chunk ch % 8
            const uint8_t* blk = sb + (ch >> 3) * 2048 + (((ch & 7) ^ g) * 16);  // rows g and g + 8 share g & 7
            const uint4 lo = *reinterpret_cast<const uint4*>(blk + g * 128);
            const uint4 hi = *reinterpret_cast<const uint4*>(blk + (g + 8) * 128);
            const int xc = ks * (KSLOT / 8) + ch;  // chunk of the activation row
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const int xr = n * 8 + g;
                const uint4 xv = *reinterpret_cast<const uint4*>(xs + xr * K * 2 + ((xc ^ (xr & 7)) * 16));
                mma_chunk(u ? c2[n] : c[n], lo, hi, xv);
            }
        }
    }
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) c[n][e] += c2[n][e];
}

// Warps per weight tile of a phase: a power of two that divides the eight
// consumer warps among the CTA's tiles and does not exceed the slots per tile.
__device__ __forceinline__ int warps_per_tile(int mine, int spt) {
    int w = 1;
    while (w * 2 <= NCW && w * 2 <= spt && mine * w * 2 <= NCW) w *= 2;
    return w;
}

// Attention of one (head, key range) by warps 0-3: the flash-decoding loop of
// the tensor-core attention kernel over a two-stage cp.async ring in `ab`.
template <int HD>
__device__ void attn_item(const PersistParams& p, int layer, int h, int start, int end, int n_real, int rg,
                          uint8_t* ab) {
    constexpr int RB = HD * 2 + 16, TILE = TKA * RB, STAGE = 2 * TILE, KS = HD / 16;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gamma = p.gamma, d = p.d;
    const bf16* Kb = p.cache + (int64_t)layer * p.layer_stride + h * HD;
    const bf16* Vb = Kb + p.kv_off;
    const uint32_t ring = smem_u32(ab);
    const int n_tiles = (end - start + TKA - 1) / TKA;
    auto load = [&](int st, int t0) {
        constexpr int VPR = HD * 2 / 16;
        for (int i = tid; i < TKA * VPR; i += 128) {
            const int r = i / VPR, v = i - r * VPR;
            const int key = t0 + r;
            const bool ok = key < end;
            const int64_t off = (int64_t)(ok ? key : t0) * d + v * 8;
            const uint32_t so = ring + st * STAGE + r * RB + v * 16;
            cp_async16z(so, Kb + off, ok ? 16 : 0);
            cp_async16z(so + TILE, Vb + off, ok ? 16 : 0);
        }
        cp_commit();
    };
    load(0, start);
    const int g = lane >> 2, cq = (lane & 3) * 2;
    uint32_t qf[KS][4];
    {
        const float qs = rsqrtf((float)HD) * 1.4426950408889634f;
        const float* q0 = p.q + (int64_t)g * d + h * HD;
        const float* q1 = q0 + (int64_t)8 * d;
        const bool v0 = g < gamma, v1 = g + 8 < gamma;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int col = ks * 16 + cq;
            const float2 a = v0 ? __ldcg(reinterpret_cast<const float2*>(q0 + col)) : make_float2(0.f, 0.f);
            const float2 b = v1 ? __ldcg(reinterpret_cast<const float2*>(q1 + col)) : make_float2(0.f, 0.f);
            const float2 c = v0 ? __ldcg(reinterpret_cast<const float2*>(q0 + col + 8)) : make_float2(0.f, 0.f);
            const float2 e = v1 ? __ldcg(reinterpret_cast<const float2*>(q1 + col + 8)) : make_float2(0.f, 0.f);
            float x0 = a.x * qs, x1 = a.y * qs, y0 = b.x * qs, y1 = b.y * qs;
            float z0 = c.x * qs, z1 = c.y * qs, w0 = e.x * qs, w1 = e.y * qs;
            qf[ks][0] = pack_round(x0, x1);
            qf[ks][1] = pack_round(y0, y1);
            qf[ks][2] = pack_round(z0, z1);
            qf[ks][3] = pack_round(w0, w1);
        }
    }
    float o[2 * KS][4];
#pragma unroll
    for (int n = 0; n < 2 * KS; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const int lr = lane & 7, lm = lane >> 3, kw = warp * 16;
    const uint32_t k_lane = (uint32_t)((kw + (lm >> 1) * 8 + lr) * RB + (lm & 1) * 16);
    const uint32_t v_lane = (uint32_t)((kw + (lm & 1) * 8 + lr) * RB + (lm >> 1) * 16);
    for (int t = 0; t < n_tiles; ++t) {
        if (t + 1 < n_tiles) load((t + 1) & 1, start + (t + 1) * TKA);
        else cp_commit();
        cp_wait<1>();
        attn_sync();
        const int nk = min(TKA, end - (start + t * TKA));
        if (kw < nk) {
            const uint32_t kbase = ring + (t & 1) * STAGE, vbase = kbase + TILE;
            float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kbase + k_lane + ks * 32, b0, b1, b2, b3);
                mma16816(s[0], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b0, b1);
                mma16816(s[1], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b2, b3);
            }
            if (kw + 16 > nk) {
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        if (kw + n * 8 + cq + e >= nk) s[n][e] = s[n][2 + e] = -INFINITY;
            }
            float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
            float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float ms0 = mn0 == -INFINITY ? 0.f : mn0, ms1 = mn1 == -INFINITY ? 0.f : mn1;
            const float a0 = ex2(m0 - ms0), a1 = ex2(m1 - ms1);
            m0 = mn0;
            m1 = mn1;
            float p00 = ex2(s[0][0] - ms0), p01 = ex2(s[0][1] - ms0), p02 = ex2(s[0][2] - ms1), p03 = ex2(s[0][3] - ms1);
            float p10 = ex2(s[1][0] - ms0), p11 = ex2(s[1][1] - ms0), p12 = ex2(s[1][2] - ms1), p13 = ex2(s[1][3] - ms1);
            const uint32_t pf0 = pack_round(p00, p01), pf1 = pack_round(p02, p03);
            const uint32_t pf2 = pack_round(p10, p11), pf3 = pack_round(p12, p13);
            l0 = l0 * a0 + ((p00 + p01) + (p10 + p11));
            l1 = l1 * a1 + ((p02 + p03) + (p12 + p13));
#pragma unroll
            for (int n = 0; n < 2 * KS; ++n) {
                o[n][0] *= a0;
                o[n][1] *= a0;
                o[n][2] *= a1;
                o[n][3] *= a1;
            }
#pragma unroll
            for (int n2 = 0; n2 < KS; ++n2) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vbase + v_lane + n2 * 32, b0, b1, b2, b3);
                mma16816(o[2 * n2], pf0, pf1, pf2, pf3, b0, b1);
                mma16816(o[2 * n2 + 1], pf0, pf1, pf2, pf3, b2, b3);
            }
        }
        attn_sync();  // every warp is done with this stage before it is refilled
    }
    cp_wait<0>();
    attn_sync();
    // merge the four warps through shared memory, then this range's partial (or the output)
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    constexpr int OWS = HD + 8;
    float* Ow = reinterpret_cast<float*>(ab);
    float* Mw = Ow + 4 * GMAXP * OWS;
    float* Lw = Mw + 4 * GMAXP;
#pragma unroll
    for (int n = 0; n < 2 * KS; ++n) {
        *reinterpret_cast<float2*>(Ow + (warp * GMAXP + g) * OWS + n * 8 + cq) = make_float2(o[n][0], o[n][1]);
        *reinterpret_cast<float2*>(Ow + (warp * GMAXP + g + 8) * OWS + n * 8 + cq) = make_float2(o[n][2], o[n][3]);
    }
    if ((lane & 3) == 0) {
        Mw[warp * GMAXP + g] = m0;
        Mw[warp * GMAXP + g + 8] = m1;
        Lw[warp * GMAXP + g] = l0;
        Lw[warp * GMAXP + g + 8] = l1;
    }
    attn_sync();
    constexpr int PW = HD + 4;
    for (int i = tid; i < gamma * (HD / 4); i += 128) {
        const int j = i / (HD / 4), e = (i % (HD / 4)) * 4;
        float M = -INFINITY;
#pragma unroll
        for (int v = 0; v < 4; ++v) M = fmaxf(M, Mw[v * GMAXP + j]);
        float l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const float mv = Mw[v * GMAXP + j];
            const float wt = mv == -INFINITY ? 0.f : ex2(mv - M);
            l += wt * Lw[v * GMAXP + j];
            const float4 ov = *reinterpret_cast<const float4*>(Ow + (v * GMAXP + j) * OWS + e);
            acc[0] += wt * ov.x;
            acc[1] += wt * ov.y;
            acc[2] += wt * ov.z;
            acc[3] += wt * ov.w;
        }
        if (n_real == 1) {
            const float inv = 1.f / l;
            *reinterpret_cast<uint2*>(p.act + (int64_t)j * d + h * HD + e) =
                make_uint2(pack2(acc[0] * inv, acc[1] * inv), pack2(acc[2] * inv, acc[3] * inv));
        } else {
            float* pr = p.part + ((int64_t)(h * p.nchunks + rg) * gamma + j) * PW;
            *reinterpret_cast<float4*>(pr + 4 + e) = make_float4(acc[0], acc[1], acc[2], acc[3]);
            if (e == 0) *reinterpret_cast<float2*>(pr) = make_float2(M, l);
        }
    }
}

template <int NT, int HD>
__global__ void __launch_bounds__(NTP, 1) k_draft_persistent(const __grid_constant__ PersistParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    // the 128-byte swizzle of the weight slices follows address bits 7-9: 1024-byte aligned ring
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t* ring = smem;
    uint8_t* xs = smem + (size_t)p.nslot * SLOT_BYTES;
    float* red = reinterpret_cast<float*>(xs + p.xs_bytes);  // [NCW][NT][32 lanes][4] tile partials
    uint64_t* full = reinterpret_cast<uint64_t*>(red + NCW * NT * 32 * 4);
    uint64_t* empty = full + p.nslot;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + p.nslot);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x, G = gridDim.x;
    const int d = p.d, gamma = p.gamma;
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.nslot; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    const unsigned int par = *(volatile unsigned int*)p.epoch & 1u;
    unsigned long long* bar = p.bar + par;
    if (c == 0 && threadIdx.x == 0) p.bar[par ^ 1u] = 0ull;  // the next launch's counter
    __syncthreads();

    if (warp == NCW) {
        // ---- producer: every weight tile of every layer, in consumption order.  Before
        // a phase's slices, the CTA's tiles of the phase after next are prefetched into L2
        // (two phases of weights fit there), so the slice copies hit L2.
        uint32_t idx = 0;
        bool ok = true;
        auto prefetch_l2 = [&](int q) {  // q: phase number layer * 4 + ph
            if (q >= p.nL * 4) return;
            const bf16* W2;
            int N2, K2;
            phase_shape(p, q / 4, q % 4, W2, N2, K2);
            const int tiles2 = (N2 + 15) / 16;
            for (int tt = c; tt < tiles2; tt += G) {  // a tile's rows are one contiguous block
                const char* base = reinterpret_cast<const char*>(W2 + (int64_t)tt * 16 * K2);
                const int bytes = min(16, N2 - tt * 16) * K2 * 2;
                for (int off = lane * 128; off < bytes; off += 32 * 128)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(base + off));
            }
        };
        prefetch_l2(0);
        prefetch_l2(1);
        for (int layer = 0; layer < p.nL && ok; ++layer)
            for (int ph = 0; ph < 4 && ok; ++ph) {
                const bf16* W;
                int N, K;
                phase_shape(p, layer, ph, W, N, K);
                prefetch_l2(layer * 4 + ph + 2);
                const int tiles = (N + 15) / 16, spt = K / KSLOT;
                for (int tt = c; tt < tiles && ok; tt += G)
                    for (int ks = 0; ks < spt; ++ks, ++idx) {
                        const int slot = (int)(idx % (uint32_t)p.nslot);
                        if (!mbar_wait(&empty[slot], ((idx / (uint32_t)p.nslot) & 1u) ^ 1u, abort_flag)) {
                            ok = false;
                            break;
                        }
                        if (lane == 0) {
                            const CUtensorMap* map = p.maps + layer * 4 + ph;
                            const uint32_t dst = smem_u32(ring + (size_t)slot * SLOT_BYTES);
                            mbar_arrive_expect_tx(&full[slot], SLOT_BYTES);  // rows past N arrive as zeros
                            if (p.map3d) {
                                tma3d(dst, map, &full[slot], 0, tt * 16, ks * 8);
                            } else {
                                for (int b = 0; b < 8; ++b)
                                    tma_load_2d(dst + b * 2048, map, &full[slot], (ks * 8 + b) * 64, tt * 16);
                            }
                        }
                    }
            }
        // no copy may still be in flight when the CTA exits (only possible after an abort)
        if (lane == 0) {
            volatile int never = 0;
            for (uint32_t i = idx > (uint32_t)p.nslot ? idx - (uint32_t)p.nslot : 0u; i < idx; ++i)
                mbar_wait(&full[i % (uint32_t)p.nslot], (i / (uint32_t)p.nslot) & 1u, &never);
        }
        __syncwarp();
    } else {
        // ---- consumers
        const int g = lane >> 2, t = lane & 3;
        const int L = p.seq_len[0];
        const int n_keys = L + gamma;
        const int per = (n_keys + p.nchunks - 1) / p.nchunks;
        const int chunk = (per + TKA - 1) / TKA * TKA;
        const int n_real = (n_keys + chunk - 1) / chunk;
        unsigned long long nbar = 0;
        uint32_t idx = 0;  // ring slots consumed by this CTA before the current phase
        for (int layer = 0; layer < p.nL; ++layer) {
            bf16* cache = p.cache + (int64_t)layer * p.layer_stride;
            for (int ph = 0; ph < 4; ++ph) {
                const bf16* W;
                int N, K;
                phase_shape(p, layer, ph, W, N, K);
                // activations of this phase
                if (ph == PH_QKV) stage_norm<NT>(xs, p.x, p.attn_norm[layer], d, gamma, p.eps);
                else if (ph == PH_O) stage_rows<NT>(xs, p.act, d, gamma);
                else if (ph == PH_GU) stage_norm<NT>(xs, p.x, p.ff_norm[layer], d, gamma, p.eps);
                else stage_rows<NT>(xs, p.hact, p.F, gamma);
                const int tiles = (N + 15) / 16, spt = K / KSLOT, mine = my_tiles(tiles, c, G);
                // groups of wpt warps share a tile, each taking every wpt-th slot of it; the
                // group's first warp sums the partials in warp order and applies the epilogue
                const int wpt = warps_per_tile(mine, spt), ngrp = NCW / wpt, grp = warp / wpt, gi = warp % wpt;
                for (int r0 = 0; r0 < mine; r0 += ngrp) {
                    const int k = r0 + grp;
                    float acc[NT][4];
#pragma unroll
                    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
                    if (k < mine) {
                        for (int ks = gi; ks < spt; ks += wpt) {
                            const uint32_t si = idx + (uint32_t)(k * spt + ks);
                            const int slot = (int)(si % (uint32_t)p.nslot);
                            if (!mbar_wait(&full[slot], (si / (uint32_t)p.nslot) & 1u, abort_flag)) break;
                            slot_mma<NT>(acc, ring + (size_t)slot * SLOT_BYTES, ks, K, xs);
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&empty[slot]);
                        }
                        if (wpt > 1) {
#pragma unroll
                            for (int n = 0; n < NT; ++n)
                                *reinterpret_cast<float4*>(red + ((warp * NT + n) * 32 + lane) * 4) =
                                    make_float4(acc[n][0], acc[n][1], acc[n][2], acc[n][3]);
                        }
                    }
                    if (wpt > 1) cons_sync();
                    if (k < mine && gi == 0) {
                        for (int o = 1; o < wpt; ++o)
#pragma unroll
                            for (int n = 0; n < NT; ++n) {
                                const float4 r = *reinterpret_cast<const float4*>(red + (((warp + o) * NT + n) * 32 + lane) * 4);
                                acc[n][0] += r.x;
                                acc[n][1] += r.y;
                                acc[n][2] += r.z;
                                acc[n][3] += r.w;
                            }
                        const int tt = c + k * G;
                        // acc[n][0..1]: weight row tt*16+g, block rows n*8+2t, +1; acc[n][2..3]: row +8
                        if (ph == PH_GU) {
                            // rows 2f (gate) and 2f+1 (up) are lanes g and g+1 (lane + 4)
    #pragma unroll
                            for (int n = 0; n < NT; ++n) {
                                float up[4];
    #pragma unroll
                                for (int e = 0; e < 4; ++e) up[e] = __shfl_down_sync(0xffffffffu, acc[n][e], 4);
                                if ((g & 1) == 0) {
    #pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const int row = tt * 16 + g + (e >> 1) * 8, j = n * 8 + 2 * t + (e & 1);
                                        if (row < N && j < gamma)
                                            p.hact[(int64_t)j * p.F + (row >> 1)] =
                                                __float2bfloat16_rn(act_fn(p.act_kind, acc[n][e]) * up[e]);
                                    }
                                }
                            }
                        } else {
    #pragma unroll
                            for (int n = 0; n < NT; ++n)
    #pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const int row = tt * 16 + g + (e >> 1) * 8, j = n * 8 + 2 * t + (e & 1);
                                    if (row >= N || j >= gamma) continue;
                                    const float v = acc[n][e];
                                    if (ph == PH_QKV) {
                                        if (row < d) {
                                            p.q[(int64_t)j * d + row] = v;
                                        } else if (L + j < p.max_rows) {
                                            const int64_t off = (int64_t)(L + j) * d + (row < 2 * d ? row - d : row - 2 * d);
                                            cache[(row < 2 * d ? 0 : p.kv_off) + off] = __float2bfloat16_rn(v);
                                        }
                                    } else {
                                        float* xp = p.x + (int64_t)j * d + row;
                                        *xp = __ldcg(xp) + v;
                                    }
                                }
                        }

                    }
                    if (wpt > 1) cons_sync();  // partials are rewritten next round
                }
                idx += (uint32_t)(mine * spt);
                if (layer == p.nL - 1 && ph == PH_D) break;  // the launch's end orders the last phase
                grid_barrier(bar, (++nbar) * G, p.err, abort_flag);
                if (ph == PH_QKV) {
                    // ---- attention: item c = (head, key range) by warps 0-3
                    const int items = p.nh * p.nchunks;
                    if (c < items && warp < 4) {
                        const int h = c / p.nchunks, rg = c - h * p.nchunks;
                        const int start = rg * chunk, end = min(n_keys, start + chunk);
                        if (rg < n_real) attn_item<HD>(p, layer, h, start, end, n_real, rg, xs);
                    }
                    grid_barrier(bar, (++nbar) * G, p.err, abort_flag);
                    if (n_real > 1) {
                        // ---- merge of the key ranges: warp per (head, block row)
                        constexpr int PW = HD + 4;
                        for (int it = c + G * warp; it < p.nh * gamma; it += G * NCW) {
                            const int h = it / gamma, j = it - h * gamma;
                            const float* base = p.part + ((int64_t)h * p.nchunks * gamma + j) * PW;
                            const int64_t cs = (int64_t)gamma * PW;
                            float mv = -INFINITY, lv = 0.f;
                            if (lane < n_real) {
                                const float2 ml = __ldcg(reinterpret_cast<const float2*>(base + lane * cs));
                                mv = ml.x;
                                lv = ml.y;
                            }
                            const float M = warp_max(mv);
                            const float wt = (lane < n_real && mv != -INFINITY) ? ex2(mv - M) : 0.f;
                            const float inv = 1.f / warp_sum(wt * lv);
                            // every lane runs the same iterations (the shuffle needs the whole warp)
                            for (int e0 = 0; e0 < HD; e0 += 128) {
                                const int e = e0 + lane * 4;
                                const bool mine_e = e < HD;
                                float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 8
                                for (int cc = 0; cc < n_real; ++cc) {
                                    const float wc = __shfl_sync(0xffffffffu, wt, cc);
                                    if (mine_e) {
                                        const float4 ov = __ldcg(reinterpret_cast<const float4*>(base + cc * cs + 4 + e));
                                        a0 = fmaf(wc, ov.x, a0);
                                        a1 = fmaf(wc, ov.y, a1);
                                        a2 = fmaf(wc, ov.z, a2);
                                        a3 = fmaf(wc, ov.w, a3);
                                    }
                                }
                                if (mine_e)
                                    *reinterpret_cast<uint2*>(p.act + (int64_t)j * d + h * HD + e) =
                                        make_uint2(pack2(a0 * inv, a1 * inv), pack2(a2 * inv, a3 * inv));
                            }
                        }
                        grid_barrier(bar, (++nbar) * G, p.err, abort_flag);
                    }
                }
            }
        }
    }
    __syncthreads();
    if (c == 0 && threadIdx.x == 0) atomicAdd(p.epoch, 1u);  // every CTA read it before the first barrier
}

template <int NT, int HD>
cudaError_t set_attr(int bytes) {
    return cudaFuncSetAttribute(k_draft_persistent<NT, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

int g_budget = 0;  // dynamic shared memory of the persistent kernel (0: unavailable)

}  // namespace

cudaError_t draft_persistent_init() {
    int dev = 0, optin = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
    const int budget = (optin - 2048) / 128 * 128;
    bool ok = set_attr<1, 64>(budget) == cudaSuccess && set_attr<1, 128>(budget) == cudaSuccess &&
              set_attr<2, 64>(budget) == cudaSuccess && set_attr<2, 128>(budget) == cudaSuccess;
    (void)cudaGetLastError();
    g_budget = ok ? budget : 0;
    return cudaSuccess;
}

// Shared memory: the ring, then max(activation staging, attention ring), then the slot barriers.
static int xs_bytes_for(int d, int F, int gamma, int hd) {
    const int nt = (gamma + 7) / 8;
    const int stage = nt * 8 * (d > F ? d : F) * 2;
    const int attn = 2 * 2 * TKA * (hd * 2 + 16);
    return ((stage > attn ? stage : attn) + 127) / 128 * 128;
}

static int red_bytes(int gamma) { return NCW * ((gamma + 7) / 8) * 32 * 4 * 4; }

bool draft_persistent_ok(const DraftPersistArgs& a) {
    const int hd = a.d / a.nh;
    if (g_budget == 0 || a.gamma < 1 || a.gamma > GMAXP || a.nL < 1 || a.nL > MAXL) return false;
    if ((hd != 64 && hd != 128) || a.d % KSLOT != 0 || a.F % KSLOT != 0 || a.nchunks < 1 || a.nchunks > MAXCH)
        return false;
    if (a.d > 32 * 4 * DMAXV) return false;
    const int xs = xs_bytes_for(a.d, a.F, a.gamma, hd);
    const int nslot = (g_budget - xs - red_bytes(a.gamma) - 2048) / SLOT_BYTES;
    return nslot >= 4 && a.maps;
}

namespace {
// The layers' grid barrier with one CTA where two are expected: it gives up after its limit.
__global__ void __launch_bounds__(NCW * 32) k_barrier_selftest(unsigned long long* bar, int* err) {
    __shared__ int abort_flag;
    if (threadIdx.x == 0) abort_flag = 0;
    __syncthreads();
    grid_barrier(bar, 2ull, err, &abort_flag);
}
}  // namespace

cudaError_t persistent_wait_selftest(void* scratch, int* err, cudaStream_t st) {
    if (!scratch || !err) return cudaErrorInvalidValue;
    k_barrier_selftest<<<1, NCW * 32, 0, st>>>(reinterpret_cast<unsigned long long*>(scratch), err);
    note_launch();
    return cudaGetLastError();
}

cudaError_t draft_persistent(const DraftPersistArgs& a, int num_sms, cudaStream_t st) {
    if (!draft_persistent_ok(a)) return cudaErrorInvalidValue;
    PersistParams p{};
    p.x = a.x;
    p.q = a.q;
    p.act = reinterpret_cast<bf16*>(a.act);
    p.hact = reinterpret_cast<bf16*>(a.hact);
    p.part = a.part;
    p.cache = reinterpret_cast<bf16*>(a.cache);
    p.layer_stride = a.layer_stride;
    p.kv_off = a.kv_off;
    p.max_rows = a.max_rows;
    p.seq_len = a.seq_len;
    for (int i = 0; i < a.nL; ++i) {
        p.wqkv[i] = reinterpret_cast<const bf16*>(a.wqkv[i]);
        p.wo[i] = reinterpret_cast<const bf16*>(a.wo[i]);
        p.wgu[i] = reinterpret_cast<const bf16*>(a.wgu[i]);
        p.wd[i] = reinterpret_cast<const bf16*>(a.wd[i]);
        p.attn_norm[i] = a.attn_norm[i];
        p.ff_norm[i] = a.ff_norm[i];
    }
    p.d = a.d;
    p.F = a.F;
    p.nh = a.nh;
    p.nL = a.nL;
    p.gamma = a.gamma;
    p.act_kind = a.act_kind;
    p.nchunks = a.nchunks;
    p.eps = a.eps;
    p.bar = a.bar;
    p.epoch = a.epoch;
    p.err = a.err;
    const int hd = a.d / a.nh;
    p.xs_bytes = xs_bytes_for(a.d, a.F, a.gamma, hd);
    p.nslot = (g_budget - p.xs_bytes - red_bytes(a.gamma) - 2048) / SLOT_BYTES;
    p.maps = reinterpret_cast<const CUtensorMap*>(a.maps);
    p.map3d = a.map3d;
    const size_t smem = 1024 + (size_t)p.nslot * SLOT_BYTES + p.xs_bytes + red_bytes(a.gamma) + 2 * p.nslot * 8 + 16;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(NTP);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int nt = (a.gamma + 7) / 8;
    cudaError_t e;
    if (nt == 1)
        e = hd == 64 ? cudaLaunchKernelEx(&cfg, k_draft_persistent<1, 64>, p)
                     : cudaLaunchKernelEx(&cfg, k_draft_persistent<1, 128>, p);
    else
        e = hd == 64 ? cudaLaunchKernelEx(&cfg, k_draft_persistent<2, 64>, p)
                     : cudaLaunchKernelEx(&cfg, k_draft_persistent<2, 128>, p);
    note_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace dspark
