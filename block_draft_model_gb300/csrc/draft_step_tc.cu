// One persistent launch for a batch-1 draft step up to the base logits, with
// every projection on the tcgen05 tensor cores:
//   "module-dflash.ts" #buildBlock   x_0 = E[a] tok_proj^T + block_pos[0], x_j = mask_emb[j-1] + block_pos[j]
//   "module-dflash.ts" #layer        pre-norm bidirectional attention over [context ++ block] and a
//                                    SwiGLU FFN, each with a residual add (every draft layer)
//   "module-dflash.ts" #baseLogits   y = RMSNorm(x) * out_norm, U = y out_proj^T
// ("src/dspark-runtime.js", propose: the same chain, kept on the device).
//
// Phases, separated by bounded grid barriers (one cooperative CTA per SM):
//   TOK   x = E[a] tok_proj^T (row 0 only) + block rows
//   per layer:  QKV  [q | k | v] = RMSNorm(x) * attn_norm . W_qkv^T
//               ATT  attention items (head, key range): partial (max, sum, output) per range,
//                    then the head's ranges merge them into O
//               WO   x += O W_o^T
//               GU   [gate | up] = RMSNorm(x) * ff_norm . W_gu^T
//               DOWN x += (act(gate) * up) W_down^T
//   OUT   U = RMSNorm(x) * out_norm . out_proj^T (and y)
//   MKV   optionally the Markov chain ("module-dflash.ts" #markov, #confidence, forwardInfer):
//         for k < gamma, l_k = U_k + w2 . w1[prev_k], tok_k = argmax l_k (lowest index on ties),
//         prev_0 = anchor, prev_{k+1} = tok_k; conf_k = sigmoid(conf_w . [y_k ; w1[prev_k]] + conf_b)
//
// Every projection phase is a weight stream with at most 16 activation rows:
// the weights are the MMA's M side (128-row tiles, 64-wide K blocks of 16 KB
// moved by TMA with the 128-byte swizzle) and the block rows its N = 16 side.
// A phase's K blocks, taken tile by tile, are cut into one contiguous range
// per CTA, so every CTA streams the same number of bytes.  The four 16-wide
// K slices of a K block go to four accumulators (16 TMEM columns each), so
// consecutive MMAs do not wait for one another; the epilogue adds them.
// RMSNorm is split: the operand is bf16(x * g) and each accumulator row is
// scaled by 1 / sqrt(mean(x^2) + eps) of its block row, computed while the
// MMAs run.  Every phase adds its partial products into fp32 buffers with
// fire-and-forget atomic adds (x itself for the block build, W_o and W_down;
// U for out_proj), so a tile shared by several CTAs needs no second pass;
// the buffers are zeroed (x set to the block rows) in earlier phases.  The
// key ranges of one attention head merge their partials cooperatively once
// all of them have arrived (a per-head count), so the W_o operand is a copy.
//
// Roles: warp 0 (one lane) streams every weight K block of every phase into a
// ring of shared-memory stages in the order the CTA consumes them and never
// waits for a grid barrier, so the next phases' weights arrive while the CTA
// waits for the others.  Warp 1 owns TMEM and one lane issues the MMAs.
// Warps 2-9 build the operands, read the accumulators back, run the epilogues
// and the attention, and take part in the grid barriers.
//
// Every wait is bounded (about one second); a timeout sets DSPARK_DEVERR_TIMEOUT
// in the error word, every role stops, in-flight copies and MMAs are waited
// for, TMEM is freed and the kernel returns.
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.cuh"
#include "tc_common.cuh"

namespace dspark {

namespace {

using namespace tc;

constexpr int NCW = 8;                    // consumer warps (warps 2..9)
constexpr int NCT = NCW * 32;             // consumer threads
constexpr int NTHR = (NCW + 2) * 32;      // plus the producer and MMA warps
constexpr int TM = 128;                   // weight rows per tile (MMA M)
constexpr int KB = 64;                    // K elements per ring stage
constexpr int STAGE_BYTES = TM * KB * 2;  // 16 KB
constexpr int BSLOT_BYTES = 16 * KB * 2;  // one K block of the 16-row operand: 2 KB
constexpr int CH = 4;                     // independent accumulator chains per tile (the K slices of a K block)
constexpr int UCOLS = CH * 16;            // TMEM columns of one tile's accumulators
constexpr int NACC = 8;                   // tiles whose accumulators are in TMEM at once
constexpr int TMEM_COLS = NACC * UCOLS;   // 512: the whole TMEM of the SM
constexpr int TKA = 64;                   // attention keys per tile
constexpr int MAXL = 16;                  // layers
constexpr int GMAX = 16;                  // block rows

enum Kind { K_TOK = 0, K_QKV = 1, K_WO = 2, K_GU = 3, K_DOWN = 4, K_OUT = 5 };

struct StepParams {
    float* x;          // [gamma, d] residual stream
    float* qkv;        // [gamma, 3d] QKV products (added into; zero before the phase)
    float* gu;         // [gamma, 2F] gate/up products, rows (gate f, up f) interleaved (idem)
    float* y;          // [gamma, d] out-normed rows
    float* U;          // [gamma, V] logits before the Markov bias
    bf16* act;         // [gamma, d] attention output O
    float* apart;      // attention partials [nh][nchunks][gamma][hd + 4]: max, sum, -, -, output
    unsigned int* hcnt;      // [2][nh] arrivals of a head's key ranges, counting up through the launch
    bf16* cache;       // layer 0, slot 0: K rows at + pos * d, V rows at + kv_off + pos * d
    int64_t layer_stride, kv_off;
    int max_rows;
    const int* seq_len;       // [0]: context length
    const bf16* embed;        // [V, H]
    const int* anchor_dev;    // [0]: anchor token, or nullptr (then `anchor`)
    int anchor;
    const float* block_const; // [gamma, d]: mask_emb + block_pos (row 0: block_pos[0])
    const float* attn_norm[MAXL];
    const float* ff_norm[MAXL];
    const float* out_norm;
    const CUtensorMap* maps;  // [2 + 4 * nL]: tok_proj, per layer (qkv, wo, gate/up, down), out_proj
    int d, F, H, V, nh, nL, gamma, act_kind, nchunks;
    float eps;
    int nstage;               // ring stages
    int ubytes;               // operand / attention staging area
    unsigned long long* bar;  // 2 arrival counters (launch parity)
    unsigned int* epoch;
    int* err;
    // the Markov chain (chain != 0)
    int chain, r;
    const bf16* w1;           // [V, r]
    const bf16* w2;           // [V, r]
    const float* conf_w;      // [d + r + 1]: the weight, then the bias
    int* tokens;              // [gamma]
    float* conf;              // [gamma]
    float* logits;            // [gamma, V] or nullptr
    unsigned long long* mk;   // [2][GMAX + 1][G] per position: one word per CTA, then the arrival counters
};

__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void cons_sync() { named_sync(1, NCT); }
// Consumer barrier that also returns the OR of `v` over the consumer threads: a decision every
// consumer takes alike (the abort flag can be raised by the other roles at any time).
__device__ __forceinline__ bool cons_sync_or(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(NCT)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void attn_sync() { named_sync(2, 128); }

__device__ __forceinline__ void cp_async16z(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
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
__device__ __forceinline__ void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
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

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- the schedule
// Phase s: 0 TOK; 1 + 4 i + k: layer i, k = 0 QKV, 1 WO, 2 GU, 3 DOWN; 1 + 4 nL: OUT.
struct Shape {
    int kind, layer, N, K, nT, nkb;
};
__device__ __forceinline__ Shape phase_shape(const StepParams& p, int s) {
    Shape sh;
    if (s == 0) {
        sh.kind = K_TOK;
        sh.layer = 0;
        sh.N = p.d;
        sh.K = p.H;
    } else if (s == 1 + 4 * p.nL) {
        sh.kind = K_OUT;
        sh.layer = 0;
        sh.N = p.V;
        sh.K = p.d;
    } else {
        const int k = (s - 1) & 3;
        sh.layer = (s - 1) >> 2;
        sh.kind = K_QKV + k;
        sh.N = k == 0 ? 3 * p.d : (k == 1 ? p.d : (k == 2 ? 2 * p.F : p.d));
        sh.K = k == 3 ? p.F : p.d;
    }
    sh.nT = (sh.N + TM - 1) / TM;
    sh.nkb = (sh.K + KB - 1) / KB;
    return sh;
}

// The phase's K blocks (tile-major) cut into contiguous ranges over the first
// min(G, T) CTAs: CTA c owns [c T / g, (c + 1) T / g).
__device__ __forceinline__ void my_range(const Shape& sh, int c, int G, int& lo, int& hi) {
    const int T = sh.nT * sh.nkb;
    const int g = min(G, T);
    if (c >= g) {
        lo = hi = 0;
        return;
    }
    lo = (int)((int64_t)c * T / g);
    hi = (int)((int64_t)(c + 1) * T / g);
}
// The CTA that owns K block j of the phase.
__device__ __forceinline__ int owner(const Shape& sh, int G, int j) {
    const int64_t T = (int64_t)sh.nT * sh.nkb;
    const int64_t g = min((int64_t)G, T);
    return (int)(((int64_t)(j + 1) * g + T - 1) / T - 1);
}

// Bounded mbarrier wait for a thread that may wait long (the epilogue warps): backs off with
// short sleeps so that it does not compete with the MMA thread for the barrier unit.
__device__ __forceinline__ bool mbar_wait_sleepy(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (globaltimer() - t0 > TIMEOUT_NS) {
            *abort_flag = 1;
            return false;
        }
        __nanosleep(64);
    }
    return true;
}

// ---------------------------------------------------------------- grid barrier
// Arrival counter counting up through the launch: barrier n opens at n * G.  Returns true
// (on every consumer thread alike) when the CTA has to stop.
__device__ __forceinline__ bool grid_barrier(unsigned long long* bar, unsigned long long target, int* err,
                                             volatile int* abort_flag) {
    cons_sync();
    if (threadIdx.x == 64) {
        __threadfence();
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
    return cons_sync_or(*abort_flag != 0);
}

// ---------------------------------------------------------------- operand staging
// The phase's operand for the CTA's K blocks: slot i holds K block (kb_first + i) mod nkb
// as [16 rows][64] bf16, row n at n * 128 bytes, 16-byte chunk c at (c ^ (n & 7)) * 16 (the
// layout a 128-byte-swizzled TMA copy gives).  Only the block rows are written: a row n past
// them feeds accumulator column n alone, which no epilogue reads (the block build uses row 0).
//   TOK: the anchor's embedding row;  QKV / GU / OUT: x * g (the row scale comes later);
//   WO: the attention output O;  DOWN: act(gate) * up.
// Every thread takes an equal share of the (slot, row, chunk) items and issues all of its
// loads before any of the arithmetic, so the staging costs one round trip to L2.
__device__ __forceinline__ void st_chunk(uint8_t* ub, int slot, int n, int ch, const float* f) {
    *reinterpret_cast<uint4*>(ub + slot * BSLOT_BYTES + n * 128 + ((ch ^ (n & 7)) * 16)) =
        make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
}

__device__ __forceinline__ void stage_operand(const StepParams& p, const Shape& sh, int kb_first, int nslots,
                                              uint8_t* ub, int anchor) {
    const int t = threadIdx.x - 64;
    const int K = sh.K, gamma = p.gamma;
    const int rows = sh.kind == K_TOK ? 1 : gamma;
    const int total = nslots * rows * 8;
    // item i: slot i / (rows * 8), row (i / 8) % rows, chunk i % 8
    auto decode = [&](int i, int& slot, int& n, int& ch, int& k0) {
        slot = i / (rows * 8);
        const int rem = i - slot * rows * 8;
        n = rem >> 3;
        ch = rem & 7;
        k0 = ((kb_first + slot) % sh.nkb) * KB + ch * 8;
    };
    {
        constexpr int BATCH = 4;  // items per thread whose loads are in flight together
        const float* g =
            sh.kind == K_QKV ? p.attn_norm[sh.layer] : (sh.kind == K_GU ? p.ff_norm[sh.layer] : p.out_norm);
        for (int i0 = t; i0 < total; i0 += BATCH * NCT) {
            float4 a[BATCH][4];
            // loads
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                const int i = i0 + b * NCT;
                int slot, n, ch, k0;
                decode(i, slot, n, ch, k0);
                const bool ok = i < total && k0 < K;
#pragma unroll
                for (int q = 0; q < 4; ++q) a[b][q] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (!ok) continue;
                if (sh.kind == K_TOK) {
                    a[b][0] = __ldg(reinterpret_cast<const float4*>(p.embed + (int64_t)anchor * p.H + k0));
                } else if (sh.kind == K_WO) {
                    a[b][0] = __ldcg(reinterpret_cast<const float4*>(p.act + (int64_t)n * p.d + k0));
                } else if (sh.kind == K_DOWN) {
                    // columns k0 .. k0 + 7 of act(gate) * up are the (gate, up) pairs 2 k0 .. 2 k0 + 15 of gu
                    const float4* gr = reinterpret_cast<const float4*>(p.gu + (int64_t)n * 2 * p.F + 2 * k0);
#pragma unroll
                    for (int q = 0; q < 4; ++q) a[b][q] = __ldcg(gr + q);
                } else {
                    const float4* xr = reinterpret_cast<const float4*>(p.x + (int64_t)n * p.d + k0);
                    const float4* gr = reinterpret_cast<const float4*>(g + k0);
                    a[b][0] = __ldcg(xr);
                    a[b][1] = __ldcg(xr + 1);
                    a[b][2] = __ldg(gr);
                    a[b][3] = __ldg(gr + 1);
                }
            }
            // arithmetic and stores
#pragma unroll
            for (int b = 0; b < BATCH; ++b) {
                const int i = i0 + b * NCT;
                if (i >= total) continue;
                int slot, n, ch, k0;
                decode(i, slot, n, ch, k0);
                if (sh.kind == K_TOK || sh.kind == K_WO) {
                    // bf16 already (the embedding row; the attention output): the chunk as is
                    *reinterpret_cast<float4*>(ub + slot * BSLOT_BYTES + n * 128 + ((ch ^ (n & 7)) * 16)) = a[b][0];
                    continue;
                }
                float f[8];
                if (sh.kind == K_DOWN) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        f[2 * q] = act_fn(p.act_kind, a[b][q].x) * a[b][q].y;
                        f[2 * q + 1] = act_fn(p.act_kind, a[b][q].z) * a[b][q].w;
                    }
                } else {
                    f[0] = a[b][0].x * a[b][2].x;
                    f[1] = a[b][0].y * a[b][2].y;
                    f[2] = a[b][0].z * a[b][2].z;
                    f[3] = a[b][0].w * a[b][2].w;
                    f[4] = a[b][1].x * a[b][3].x;
                    f[5] = a[b][1].y * a[b][3].y;
                    f[6] = a[b][1].z * a[b][3].z;
                    f[7] = a[b][1].w * a[b][3].w;
                }
                st_chunk(ub, slot, n, ch, f);
            }
        }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor cores
}

// rs[j] = 1 / sqrt(mean(x[j]^2) + eps) over the whole row, a warp per block row.
__device__ __forceinline__ void row_scales(const StepParams& p, float* rs) {
    const int w = (threadIdx.x >> 5) - 2, lane = threadIdx.x & 31;
    for (int j = w; j < p.gamma; j += NCW) {
        const float4* xr = reinterpret_cast<const float4*>(p.x + (int64_t)j * p.d);
        float a = 0.f;
        for (int k4 = lane; k4 < p.d / 4; k4 += 32) {
            const float4 v = __ldcg(xr + k4);
            a += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
        a = warp_sum(a);
        if (lane == 0) rs[j] = rsqrtf(a / (float)p.d + p.eps);
    }
}

// Zero a CTA's share of a buffer of n floats (16-byte aligned): float4 shares, and the last
// CTA also takes the n % 4 trailing floats.
__device__ __forceinline__ void zero_share(float* buf, int64_t n, int c, int G) {
    const int64_t n4 = n / 4;
    const int64_t a = n4 * c / G, b = n4 * (c + 1) / G;
    float4* b4 = reinterpret_cast<float4*>(buf);
    for (int64_t i = a + (threadIdx.x - 64); i < b; i += NCT) b4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c == G - 1 && threadIdx.x - 64 < (int)(n - 4 * n4)) buf[4 * n4 + (threadIdx.x - 64)] = 0.f;
}

// ---------------------------------------------------------------- epilogues
// Thread (row r of the tile, column group cg) holds v[i] = acc[r][cg * 8 + i], scaled.  Every
// phase adds into its output; nothing else touches those entries during the phase.
__device__ __forceinline__ void epi_add(const StepParams& p, const Shape& sh, int t, int r, int cg, const float* v) {
    const int n = t * TM + r;
    if (n >= sh.N) return;
    float* dst;
    int64_t ld;
    int rows = p.gamma;
    if (sh.kind == K_QKV) {
        dst = p.qkv;
        ld = 3 * (int64_t)p.d;
    } else if (sh.kind == K_GU) {
        dst = p.gu;
        ld = 2 * (int64_t)p.F;
    } else if (sh.kind == K_OUT) {
        dst = p.U;
        ld = p.V;
    } else {
        dst = p.x;
        ld = p.d;
        if (sh.kind == K_TOK) rows = 1;  // only operand row 0 (the anchor) is staged
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int j = cg * 8 + i;
        if (j < rows) atomicAdd(dst + j * ld + n, v[i]);  // result unused: a fire-and-forget reduction
    }
}

// ---------------------------------------------------------------- attention
// One (head, key range) item on warps 2-5: flash decoding over 64-key tiles of a two-stage
// cp.async ring in `ab`; scores in the log2 domain; the range's partial (max, sum, output)
// goes to apart.  The range that holds the block's own keys (rows L .. L + gamma - 1) first
// writes the head's block K/V rows into the cache, in the cache's bf16 format.
template <int HD>
__device__ void attn_item(const StepParams& p, int layer, int h, int start, int end, int L, int rg, uint8_t* ab) {
    constexpr int RB = HD * 2 + 16, TILE = TKA * RB, STAGE = 2 * TILE, KS = HD / 16;
    const int tid = threadIdx.x - 64, warp = tid >> 5, lane = tid & 31;
    const int gamma = p.gamma, d = p.d;
    bf16* Kw = p.cache + (int64_t)layer * p.layer_stride + h * HD;
    const bf16* Kb = Kw;
    const bf16* Vb = Kb + p.kv_off;
    const uint32_t ring = smem_u32(ab);
    if (end > L) {
        for (int i = tid; i < gamma * HD / 4; i += 128) {
            const int j = i / (HD / 4), e = (i - j * (HD / 4)) * 4;
            if (L + j >= p.max_rows) continue;
            const float* src = p.qkv + (int64_t)j * 3 * d + h * HD + e;
            const float4 kv = __ldcg(reinterpret_cast<const float4*>(src + d));
            const float4 vv = __ldcg(reinterpret_cast<const float4*>(src + 2 * d));
            bf16* kd = Kw + (int64_t)(L + j) * d + e;
            *reinterpret_cast<uint2*>(kd) = make_uint2(pack2(kv.x, kv.y), pack2(kv.z, kv.w));
            *reinterpret_cast<uint2*>(kd + p.kv_off) = make_uint2(pack2(vv.x, vv.y), pack2(vv.z, vv.w));
        }
        __threadfence();
        attn_sync();  // the rows are in global memory before any copy of this CTA reads them
    }
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
        const float* q0 = p.qkv + (int64_t)g * 3 * d + h * HD;
        const float* q1 = q0 + (int64_t)8 * 3 * d;
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
    // the four warps' key slices merged through shared memory, then this range's partial (or the output)
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    constexpr int OWS = HD + 8;
    float* Ow = reinterpret_cast<float*>(ab);
    float* Mw = Ow + 4 * GMAX * OWS;
    float* Lw = Mw + 4 * GMAX;
#pragma unroll
    for (int n = 0; n < 2 * KS; ++n) {
        *reinterpret_cast<float2*>(Ow + (warp * GMAX + g) * OWS + n * 8 + cq) = make_float2(o[n][0], o[n][1]);
        *reinterpret_cast<float2*>(Ow + (warp * GMAX + g + 8) * OWS + n * 8 + cq) = make_float2(o[n][2], o[n][3]);
    }
    if ((lane & 3) == 0) {
        Mw[warp * GMAX + g] = m0;
        Mw[warp * GMAX + g + 8] = m1;
        Lw[warp * GMAX + g] = l0;
        Lw[warp * GMAX + g + 8] = l1;
    }
    attn_sync();
    constexpr int PW = HD + 4;
    for (int i = tid; i < gamma * (HD / 4); i += 128) {
        const int j = i / (HD / 4), e = (i % (HD / 4)) * 4;
        float M = -INFINITY;
#pragma unroll
        for (int v = 0; v < 4; ++v) M = fmaxf(M, Mw[v * GMAX + j]);
        float l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const float mv = Mw[v * GMAX + j];
            const float wt = mv == -INFINITY ? 0.f : ex2(mv - M);
            l += wt * Lw[v * GMAX + j];
            const float4 ov = *reinterpret_cast<const float4*>(Ow + (v * GMAX + j) * OWS + e);
            acc[0] += wt * ov.x;
            acc[1] += wt * ov.y;
            acc[2] += wt * ov.z;
            acc[3] += wt * ov.w;
        }
        float* pr = p.apart + ((int64_t)(h * p.nchunks + rg) * gamma + j) * PW;
        *reinterpret_cast<float4*>(pr + 4 + e) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        if (e == 0) *reinterpret_cast<float2*>(pr) = make_float2(M, l);
    }
}

// After every key range of head h has written its partial (the head's arrival count reached
// `target`), range rg merges its share of the head's gamma x HD outputs:
// O = sum_r exp2(m_r - M) o_r / sum_r exp2(m_r - M) l_r, M = max_r m_r, ranges in order.
template <int HD>
__device__ void attn_merge(const StepParams& p, unsigned int* cnt, unsigned int target, int h, int rg, int n_real,
                           volatile int* abort_flag) {
    constexpr int PW = HD + 4;
    const int tid = threadIdx.x - 64;
    __threadfence();
    attn_sync();
    if (tid == 0) {
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(cnt) : "memory");
        const uint64_t t0 = globaltimer();
        while (true) {
            unsigned int cur;
            asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(cur) : "l"(cnt) : "memory");
            if (cur >= target || *abort_flag) break;
            if (globaltimer() - t0 > TIMEOUT_NS) {
                atomicOr(p.err, DEVERR_TIMEOUT);
                *abort_flag = 1;
                break;
            }
            __nanosleep(32);
        }
    }
    attn_sync();
    const int gamma = p.gamma, groups = gamma * (HD / 4);
    const int g0 = (int)((int64_t)rg * groups / n_real), g1 = (int)((int64_t)(rg + 1) * groups / n_real);
    for (int gi = g0 + tid; gi < g1; gi += 128) {
        const int j = gi / (HD / 4), e = (gi - j * (HD / 4)) * 4;
        const float* base = p.apart + ((int64_t)h * p.nchunks * gamma + j) * PW;
        const int64_t cs = (int64_t)gamma * PW;
        constexpr int RB = 16;  // ranges whose loads are in flight together
        float M = -INFINITY, l = 0.f, a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        for (int r0 = 0; r0 < n_real; r0 += RB) {
            float2 ml[RB];
            float4 ov[RB];
#pragma unroll
            for (int u = 0; u < RB; ++u) {
                const int r = min(r0 + u, n_real - 1);
                ml[u] = __ldcg(reinterpret_cast<const float2*>(base + r * cs));
                ov[u] = __ldcg(reinterpret_cast<const float4*>(base + r * cs + 4 + e));
            }
            float Mn = M;
#pragma unroll
            for (int u = 0; u < RB; ++u)
                if (r0 + u < n_real) Mn = fmaxf(Mn, ml[u].x);
            const float sc = M == -INFINITY ? 0.f : ex2(M - Mn);
            l *= sc;
            a0 *= sc;
            a1 *= sc;
            a2 *= sc;
            a3 *= sc;
#pragma unroll
            for (int u = 0; u < RB; ++u) {
                const float wt = (r0 + u < n_real && ml[u].x != -INFINITY) ? ex2(ml[u].x - Mn) : 0.f;
                l = fmaf(wt, ml[u].y, l);
                a0 = fmaf(wt, ov[u].x, a0);
                a1 = fmaf(wt, ov[u].y, a1);
                a2 = fmaf(wt, ov[u].z, a2);
                a3 = fmaf(wt, ov[u].w, a3);
            }
            M = Mn;
        }
        const float inv = 1.f / l;
        *reinterpret_cast<uint2*>(p.act + (int64_t)j * p.d + h * HD + e) =
            make_uint2(pack2(a0 * inv, a1 * inv), pack2(a2 * inv, a3 * inv));
    }
}

// ---------------------------------------------------------------- the Markov chain
// acc += the 8 bf16 products of w and e, each as one bf16 x bf16 + fp32 fused multiply-add
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

// (value, index) as one word whose unsigned order is: larger value first, then lower index
__device__ __forceinline__ unsigned long long best_key(float v, int i) {
    uint32_t u = __float_as_uint(v);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)u << 32) | (unsigned long long)(~(uint32_t)i);
}

// The chain over the CTA's vocabulary rows [v0, v1) (consumer warps).  An 8-lane group takes a
// row at a time (lane s holds the 16-byte chunks s, s + 8, ... of the w2 row and of e, so the
// group reads whole 128-byte segments); w2 (read once per position) stays in L2 after the first.
// Each position's argmax: the CTA's best word, then one word per CTA and an arrival counter; one
// lane waits (bounded) for every CTA and its warp reads the words.
template <int CPL>
__device__ void markov_chain(const StepParams& p, int anchor, unsigned long long* words, int* toks, float* redv,
                             int* redi, const uint8_t* w2s, int n_res, uint64_t* w2_full, float* us,
                             volatile int* abort_flag) {
    const int c = blockIdx.x, G = gridDim.x, V = p.V, r = p.r, gamma = p.gamma;
    const int tt = threadIdx.x - 64, warp = tt >> 5, lane = threadIdx.x & 31, grp = tt >> 3, s = tt & 7;
    constexpr int GROUPS = NCT / 8, UR = 4;  // row groups; rows of a group in flight together
    constexpr int ROWB = CPL * 128;          // bytes of a w2 row
    const int v0 = (int)((int64_t)c * V / G), v1 = (int)((int64_t)(c + 1) * V / G);
    if (tt == 0) toks[0] = anchor;
    // the slice's base logits of every position into shared memory at once: us[k * nrows + li]
    const int nrows = v1 - v0;
    for (int i = tt; i < gamma * nrows; i += NCT) {
        const int k = i / nrows, li = i - k * nrows;
        us[i] = __ldcg(p.U + (int64_t)k * V + v0 + li);
    }
    // the first n_res rows of the slice arrive in shared memory (row li at li * ROWB); an 8-lane group
    // reads one whole 128-byte segment of a row at a time, so the rows need no swizzle
    if (n_res > 0 && lane == 0 && !mbar_wait_sleepy(w2_full, 0, abort_flag)) atomicOr(p.err, DEVERR_TIMEOUT);
    cons_sync();
    for (int k = 0; k < gamma; ++k) {
        const int prev = toks[k];
        uint4 ev[CPL];
#pragma unroll
        for (int j = 0; j < CPL; ++j) ev[j] = __ldg(reinterpret_cast<const uint4*>(p.w1 + (int64_t)prev * r) + s + 8 * j);
        float bv = -INFINITY;
        int bi = INT_MAX;
        // the loop bound is the same for every lane: the shuffles below take the whole warp.  The
        // highest rows (past the resident ones, read from global memory) come first, so that their
        // loads overlap the load of e.
        for (int base = v0 + (nrows > 0 ? (nrows - 1) / (GROUPS * UR) : -1) * (GROUPS * UR); base >= v0;
             base -= GROUPS * UR) {
            uint4 w[UR][CPL];
            float u[UR];
#pragma unroll
            for (int q = 0; q < UR; ++q) {
                const int row = base + grp + GROUPS * q;
                const bool ok = row < v1;
                const bool res = row - v0 < n_res;
#pragma unroll
                for (int j = 0; j < CPL; ++j)
                    w[q][j] = !ok ? make_uint4(0, 0, 0, 0)
                                  : res ? *reinterpret_cast<const uint4*>(w2s + (size_t)(row - v0) * ROWB + (s + 8 * j) * 16)
                                        : __ldg(reinterpret_cast<const uint4*>(p.w2 + (int64_t)row * r) + s + 8 * j);
                u[q] = (ok && s == 0) ? us[k * nrows + (row - v0)] : 0.f;
            }
#pragma unroll
            for (int q = 0; q < UR; ++q) {
                float dot = 0.f;
#pragma unroll
                for (int j = 0; j < CPL; ++j) dot = fma_chunk(w[q][j], ev[j], dot);
                dot += __shfl_xor_sync(0xffffffffu, dot, 4);
                dot += __shfl_xor_sync(0xffffffffu, dot, 2);
                dot += __shfl_xor_sync(0xffffffffu, dot, 1);
                const int row = base + grp + GROUPS * q;
                if (s == 0 && row < v1) {
                    const float l = u[q] + dot;
                    if (p.logits) p.logits[(int64_t)k * V + row] = l;
                    if (better(l, row, bv, bi)) {
                        bv = l;
                        bi = row;
                    }
                }
            }
        }
        ArgBest b = warp_argbest({bv, bi});
        if (lane == 0) {
            redv[warp] = b.v;
            redi[warp] = b.i;
        }
        cons_sync();
        if (warp == 0) {
            ArgBest cb{lane < NCW ? redv[lane] : -INFINITY, lane < NCW ? redi[lane] : INT_MAX};
            cb = warp_argbest(cb);
            unsigned long long* wk = words + (size_t)k * G;
            unsigned long long* cnt = words + (size_t)GMAX * G + k;
            if (lane == 0) {
                // a CTA without rows still arrives, with a word below every real one
                const unsigned long long key = cb.i != INT_MAX ? best_key(cb.v, cb.i) : 1ull;
                if (cb.i != INT_MAX) {  // the next position's e wherever it comes from: this CTA's best row
                    const char* row = reinterpret_cast<const char*>(p.w1 + (int64_t)cb.i * r);
                    for (int o = 0; o < r * 2; o += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(row + o));
                }
                asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(wk + c), "l"(key) : "memory");
                asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(cnt) : "memory");
                const uint64_t t0 = globaltimer();
                while (true) {
                    unsigned long long cur;
                    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(cur) : "l"(cnt) : "memory");
                    if (cur >= (unsigned long long)G || *abort_flag) break;
                    if (globaltimer() - t0 > TIMEOUT_NS) {
                        atomicOr(p.err, DEVERR_TIMEOUT);
                        *abort_flag = 1;
                        break;
                    }
                }
            }
            __syncwarp();
            unsigned long long m = 0ull;
            for (int i = lane; i < G; i += 32) {
                unsigned long long w;
                asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(wk + i) : "memory");
                m = w > m ? w : m;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long om = __shfl_xor_sync(0xffffffffu, m, o);
                m = om > m ? om : m;
            }
            if (lane == 0) {
                int tok = (int)(~(uint32_t)m);
                if (m <= 1ull || tok < 0 || tok >= V) {  // no valid word (an aborted or broken exchange)
                    if (c == 0) atomicOr(p.err, 8);
                    tok = 0;
                }
                toks[k + 1] = tok;
                if (c == 0) p.tokens[k] = tok;
            }
        }
        cons_sync();
    }
    // confidences, by CTA 0: sigmoid(conf_w . [y_k ; w1[prev_k]] + conf_b)
    if (c == 0) {
        for (int k = 0; k < gamma; ++k) {
            const float* yr = p.y + (int64_t)k * p.d;
            const bf16* er = p.w1 + (int64_t)toks[k] * r;
            float z = 0.f;
            for (int i = tt; i < p.d; i += NCT) z = fmaf(__ldcg(yr + i), __ldg(p.conf_w + i), z);
            for (int i = tt; i < r; i += NCT) z = fmaf(__bfloat162float(er[i]), __ldg(p.conf_w + p.d + i), z);
            z = warp_sum(z);
            if (lane == 0) redv[warp] = z;
            cons_sync();
            if (tt == 0) {
                float a = 0.f;
                for (int w2i = 0; w2i < NCW; ++w2i) a += redv[w2i];
                p.conf[k] = 1.f / (1.f + expf(-(a + __ldg(p.conf_w + p.d + r))));
            }
            cons_sync();
        }
    }
}

// ---------------------------------------------------------------- the kernel
template <int HD>
__global__ void __launch_bounds__(NTHR, 1) k_draft_step_tc(const __grid_constant__ StepParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // 128-byte swizzle: 1024-byte aligned
    uint8_t* ring = smem;
    uint8_t* ub = ring + (size_t)p.nstage * STAGE_BYTES;           // operand slots / attention staging
    uint64_t* full = reinterpret_cast<uint64_t*>(ub + p.ubytes);
    uint64_t* empty = full + p.nstage;
    uint64_t* acc_full = empty + p.nstage;
    uint64_t* acc_empty = acc_full + NACC;
    uint64_t* b_full = acc_empty + NACC;
    uint64_t* b_taken = b_full + 1;  // the MMA warp has seen the phase's b_full
    uint64_t* drain = b_taken + 1;
    uint64_t* w2_full = drain + 1;   // the Markov chain's resident w2 rows have arrived
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(w2_full + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* rs = reinterpret_cast<float*>(tmem_slot + 4);   // [16] row scales
    int* toks = reinterpret_cast<int*>(rs + GMAX);          // [GMAX + 1] the chain's tokens
    float* redv = reinterpret_cast<float*>(toks + GMAX + 4);  // [NCW] the chain's per-warp bests
    int* redi = reinterpret_cast<int*>(redv + NCW);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x, G = gridDim.x;
    const int nph = 2 + 4 * p.nL;
    const int S = p.nstage;
    // rows of this CTA's w2 slice kept in shared memory for the chain (the ring and staging area)
    const int v0c = (int)((int64_t)c * p.V / G), v1c = (int)((int64_t)(c + 1) * p.V / G);
    // (the slice's base logits of every position take the end of that area)
    const size_t ures = ((size_t)p.gamma * (v1c - v0c) * 4 + 127) / 128 * 128;
    const size_t area = (size_t)S * STAGE_BYTES + p.ubytes;
    const int n_res = p.chain && area > ures ? min(v1c - v0c, (int)((area - ures) / ((size_t)p.r * 2))) : 0;
    float* us = reinterpret_cast<float*>(ring + (area - ures));

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < NACC; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], NCW);  // every consumer warp has read the accumulators
        }
        mbar_init(b_full, 1);
        mbar_init(b_taken, 1);
        mbar_init(drain, 1);
        mbar_init(w2_full, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    const unsigned int par = *(volatile unsigned int*)p.epoch & 1u;
    unsigned long long* bar = p.bar + par;
    if (c == 0 && threadIdx.x == 0) p.bar[par ^ 1u] = 0ull;  // the next launch's counters
    if (c == 0 && threadIdx.x < p.nh) p.hcnt[(par ^ 1u) * p.nh + threadIdx.x] = 0u;
    if (c == 0 && p.chain) {
        unsigned long long* other = p.mk + (size_t)(par ^ 1u) * (GMAX + 1) * G;
        for (int i = threadIdx.x; i < (GMAX + 1) * G; i += NTHR) other[i] = 0ull;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---- producer: every K block of every phase, in consumption order (ring position
        // st / phase bit ph and the K block coordinates advance incrementally)
        if (lane == 0) {
            uint32_t st = 0, ph = 0, issued = 0;
            bool ok = true;
            for (int s = 0; s < nph && ok; ++s) {
                const Shape sh = phase_shape(p, s);
                const CUtensorMap* map = p.maps + s;
                asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
                int lo, hi;
                my_range(sh, c, G, lo, hi);
                int t = lo / sh.nkb, kb = lo - t * sh.nkb;
                for (int j = lo; j < hi; ++j) {
                    if (!mbar_wait(&empty[st], ph ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[st], STAGE_BYTES);  // rows / columns past the matrix arrive as zeros
                    tma_load_2d(smem_u32(ring + (size_t)st * STAGE_BYTES), map, &full[st], kb * KB, t * TM);
                    ++issued;
                    if (++kb == sh.nkb) {
                        kb = 0;
                        ++t;
                    }
                    if (++st == (uint32_t)S) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
            }
            // the Markov chain's resident w2 rows, once every MMA (and so every read of the ring and of
            // the operand slots) has retired: contiguous rows, in bulk copies of at most 32 KB
            if (ok && n_res > 0) {
                if (mbar_wait(drain, 0, abort_flag)) {
                    const size_t bytes = (size_t)n_res * p.r * 2;
                    const char* src = reinterpret_cast<const char*>(p.w2 + (int64_t)v0c * p.r);
                    mbar_arrive_expect_tx(w2_full, (uint32_t)bytes);
                    for (size_t o = 0; o < bytes; o += 32768) {
                        const uint32_t n = (uint32_t)min((size_t)32768, bytes - o);
                        asm volatile(
                            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                                smem_u32(ring) + (uint32_t)o),
                            "l"(src + o), "r"(n), "r"(smem_u32(w2_full))
                            : "memory");
                    }
                    // wait for them here too: no copy may be in flight when the CTA exits
                    volatile int never = 0;
                    mbar_wait(w2_full, 0, &never);
                }
            }
            // no copy may still be in flight when the CTA exits (only possible after an abort):
            // the last min(S, issued) copies, newest first
            volatile int never = 0;
            for (uint32_t i = 0; i < (uint32_t)S && i < issued; ++i) {
                if (st == 0) {
                    st = (uint32_t)S;
                    ph ^= 1u;
                }
                --st;
                mbar_wait(&full[st], ph, &never);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA issuer: K slice k of every K block into accumulator chain k of the tile
        if (lane == 0) {
            const uint32_t id = idesc(TM, 16);
            const uint32_t ub_s = smem_u32(ub), ring_s = smem_u32(ring);
            uint32_t st = 0, ph = 0, acc = 0, aph = 0, bph = 0;
            bool ok = true;
            for (int s = 0; s < nph && ok; ++s) {
                const Shape sh = phase_shape(p, s);
                int lo, hi;
                my_range(sh, c, G, lo, hi);
                if (!mbar_wait(b_full, bph, abort_flag)) break;  // the phase's operand is staged
                bph ^= 1u;
                mbar_arrive(b_taken);
                tc_fence_after();
                int slot = 0;  // the i-th K block of the CTA's range is operand slot i mod nkb
                for (int j = lo; j < hi && ok;) {
                    const int t = j / sh.nkb, kb0 = j - t * sh.nkb, kb1 = min(sh.nkb, kb0 + (hi - j));
                    if (!mbar_wait(&acc_empty[acc], aph ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem + acc * (uint32_t)UCOLS;
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait(&full[st], ph, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t dw = sdesc(ring_s + st * (uint32_t)STAGE_BYTES);
                        const uint64_t dx = sdesc(ub_s + (uint32_t)slot * (uint32_t)BSLOT_BYTES);
#pragma unroll
                        for (int k = 0; k < CH; ++k)
                            umma(d_tmem + (uint32_t)(k * 16), dw + (uint64_t)(2 * k), dx + (uint64_t)(2 * k), id,
                                 kb > kb0 ? 1u : 0u);
                        umma_commit(&empty[st]);
                        if (++st == (uint32_t)S) {
                            st = 0;
                            ph ^= 1u;
                        }
                        if (++slot == sh.nkb) slot = 0;
                    }
                    if (!ok) break;
                    umma_commit(&acc_full[acc]);
                    if (++acc == (uint32_t)NACC) {
                        acc = 0;
                        aph ^= 1u;
                    }
                    j += kb1 - kb0;
                }
            }
            // every MMA issued above has retired before TMEM is freed
            umma_commit(drain);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(drain, 0) && globaltimer() - t0 < TIMEOUT_NS) {
            }
        }
        __syncwarp();
    } else {
        // ---- consumers: operands, epilogues, attention, grid barriers
        const int tt = threadIdx.x - 64;
        const int q4 = warp & 3, cg = (warp - 2) >> 2;  // TMEM lane quarter, column group
        const int r = q4 * 32 + lane;                    // row of the tile
        const int L = __ldcg(p.seq_len);
        const int anchor = p.anchor_dev ? __ldcg(p.anchor_dev) : p.anchor;
        const int n_keys = L + p.gamma;
        const int per = (n_keys + p.nchunks - 1) / p.nchunks;
        const int chunk = (per + TKA - 1) / TKA * TKA;
        const int n_real = (n_keys + chunk - 1) / chunk;
        // buffers that phases add into: x starts as the block rows (the block build adds the anchor's
        // projection to row 0), qkv and U at zero (later layers' qkv: zeroed after their attention);
        // a grid barrier after the block build's operand orders these before any addition
        {
            const int64_t n4 = (int64_t)p.gamma * p.d / 4;
            const int64_t a4 = n4 * c / G, b4 = n4 * (c + 1) / G;
            for (int64_t i = a4 + tt; i < b4; i += NCT)
                reinterpret_cast<float4*>(p.x)[i] = __ldg(reinterpret_cast<const float4*>(p.block_const) + i);
        }
        zero_share(p.qkv, (int64_t)p.gamma * 3 * p.d, c, G);
        zero_share(p.U, (int64_t)p.gamma * p.V, c, G);
        unsigned long long nbar = 0;
        uint32_t acc = 0, aph = 0;
        for (int s = 0; s < nph; ++s) {
            const Shape sh = phase_shape(p, s);
            int lo, hi;
            my_range(sh, c, G, lo, hi);
            const int kb_first = hi > lo ? lo % sh.nkb : 0;
            const int nslots = min(sh.nkb, hi - lo);
            const bool scaled = sh.kind == K_QKV || sh.kind == K_GU || sh.kind == K_OUT;
            stage_operand(p, sh, kb_first, nslots, ub, anchor);
            cons_sync();
            if (tt == 0) {
                // b_full completes once per phase: the MMA warp must have seen the previous one
                if (s == 0 || mbar_wait(b_taken, (uint32_t)(s - 1) & 1u, abort_flag)) mbar_arrive(b_full);
                else *abort_flag = 1;
            }
            // while the MMAs run: buffers for later phases, and the row scales of this one
            if (s == 0 && grid_barrier(bar, (++nbar) * G, p.err, abort_flag)) break;  // x, qkv, U set everywhere
            if (sh.kind == K_QKV) zero_share(p.gu, (int64_t)p.gamma * 2 * p.F, c, G);
            if (sh.kind == K_WO) zero_share(p.qkv, (int64_t)p.gamma * 3 * p.d, c, G);
            if (scaled) {
                row_scales(p, rs);
                cons_sync();
            }
            if (sh.kind == K_OUT) {
                // y = RMSNorm(x) * out_norm in fp32 (the confidence head's input): a column range per CTA
                const int c0 = (int)((int64_t)c * p.d / G), c1 = (int)((int64_t)(c + 1) * p.d / G);
                for (int i = tt; i < p.gamma * (c1 - c0); i += NCT) {
                    const int j = i / (c1 - c0), k = c0 + i % (c1 - c0);
                    p.y[(int64_t)j * p.d + k] = __ldcg(p.x + (int64_t)j * p.d + k) * rs[j] * __ldg(p.out_norm + k);
                }
            }
            // epilogues of the CTA's tiles, in MMA order
            for (int j = lo; j < hi;) {
                const int t = j / sh.nkb, kb0 = j - t * sh.nkb, kb1 = min(sh.nkb, kb0 + (hi - j));
                j += kb1 - kb0;
                const int a = (int)acc;
                // one lane of the warp polls (the MMA thread shares the barrier unit), then the warp goes on
                bool got = true;
                if (lane == 0) got = mbar_wait_sleepy(&acc_full[a], aph, abort_flag);
                got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
                if (++acc == (uint32_t)NACC) {
                    acc = 0;
                    aph ^= 1u;
                }
                tc_fence_after();
                float v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = 0.f;
                // tcgen05.ld is warp-wide: the whole warp takes the same branch
                const bool ld_ok = got && __shfl_sync(0xffffffffu, *abort_flag, 0) == 0;
                if (ld_ok && cg * 8 < p.gamma) {
#pragma unroll
                    for (int k = 0; k < CH; ++k) {
                        uint32_t rr[8];
                        tmem_ld8(tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(a * UCOLS + k * 16 + cg * 8), rr);
#pragma unroll
                        for (int i = 0; i < 8; ++i) v[i] += __uint_as_float(rr[i]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[a]);  // this warp is done with the accumulators
                if (!ld_ok) continue;
                if (scaled)
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[i] *= rs[min(cg * 8 + i, GMAX - 1)];
                epi_add(p, sh, t, r, cg, v);
            }
            if (cons_sync_or(*abort_flag != 0)) break;
            if (s == nph - 1) {
                if (p.chain && !grid_barrier(bar, (++nbar) * G, p.err, abort_flag)) {
                    // U, y and the logits' base are complete everywhere: the chain, in the staging area
                    unsigned long long* words = p.mk + (size_t)par * (GMAX + 1) * G;
                    const int cpl = p.r / 64;
                    if (cpl == 4) markov_chain<4>(p, anchor, words, toks, redv, redi, ring, n_res, w2_full, us, abort_flag);
                    else if (cpl == 2) markov_chain<2>(p, anchor, words, toks, redv, redi, ring, n_res, w2_full, us, abort_flag);
                    else if (cpl == 1) markov_chain<1>(p, anchor, words, toks, redv, redi, ring, n_res, w2_full, us, abort_flag);
                    else if (cpl == 8) markov_chain<8>(p, anchor, words, toks, redv, redi, ring, n_res, w2_full, us, abort_flag);
                }
                break;
            }
            if (grid_barrier(bar, (++nbar) * G, p.err, abort_flag)) break;
            if (sh.kind == K_QKV) {
                // ---- attention of layer sh.layer: item c = (head, key range) on warps 2-5
                const int h = c / p.nchunks, rg = c - h * p.nchunks;
                if (c < p.nh * p.nchunks && rg < n_real && warp < 6) {
                    const int start = rg * chunk, end = min(n_keys, start + chunk);
                    attn_item<HD>(p, sh.layer, h, start, end, L, rg, ub);
                    attn_merge<HD>(p, p.hcnt + par * p.nh + h, (unsigned int)((sh.layer + 1) * n_real), h, rg, n_real,
                                   abort_flag);
                }
                if (grid_barrier(bar, (++nbar) * G, p.err, abort_flag)) break;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) atomicOr(p.err, DEVERR_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
    if (c == 0 && threadIdx.x == 0) atomicAdd(p.epoch, 1u);  // every CTA read it before the first barrier
}

// The step's grid barrier with one CTA where two are expected: it gives up after its limit and
// every consumer thread sees the same outcome.
__global__ void __launch_bounds__(NTHR, 1) k_step_barrier_selftest(unsigned long long* bar, int* err) {
    __shared__ int abort_flag;
    if (threadIdx.x == 0) abort_flag = 0;
    __syncthreads();
    if (threadIdx.x >= 64) {
        const bool stop = grid_barrier(bar, 2ull, err, &abort_flag);
        if (threadIdx.x == 64 && !stop) atomicOr(err, 1);  // not expected: the barrier cannot open
    }
}

int g_budget = 0;  // dynamic shared memory the kernel may take (0: unavailable)

// Staging area: the operand slots of the widest phase, or the attention's two-stage ring and its
// merge scratch, whichever is larger.
int ubytes_for(const DraftStepArgs& a, int G) {
    // (the operand slots of every phase, or the attention's ring and merge scratch)
    const int hd = a.d / a.nh;
    auto slots = [&](int N, int K) {
        const int nT = (N + TM - 1) / TM, nkb = (K + KB - 1) / KB;
        const int64_t T = (int64_t)nT * nkb;
        const int g = (int)std::min<int64_t>(G, T);
        const int mx = (int)((T + g - 1) / g) + 1;  // a range can straddle one more K block than the mean
        return std::min(nkb, mx);
    };
    int ns = std::max({slots(a.d, a.H), slots(3 * a.d, a.d), slots(a.d, a.d), slots(2 * a.F, a.d), slots(a.d, a.F),
                       slots(a.V, a.d)});
    const int attn = 2 * 2 * TKA * (hd * 2 + 16);
    const int merge = (4 * GMAX * (hd + 8) + 8 * GMAX) * 4;
    return std::max({ns * BSLOT_BYTES, attn, merge});
}

}  // namespace

cudaError_t step_wait_selftest(void* scratch, int* err, cudaStream_t st) {
    if (!scratch || !err) return cudaErrorInvalidValue;
    k_step_barrier_selftest<<<1, NTHR, 0, st>>>(reinterpret_cast<unsigned long long*>(scratch), err);
    note_launch();
    return cudaGetLastError();
}

cudaError_t draft_step_tc_init() {
    int dev = 0, optin = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
    const int budget = (optin - 1024) / 1024 * 1024;
    const bool ok =
        cudaFuncSetAttribute(k_draft_step_tc<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, budget) == cudaSuccess &&
        cudaFuncSetAttribute(k_draft_step_tc<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, budget) == cudaSuccess;
    (void)cudaGetLastError();
    g_budget = ok ? budget : 0;
    return cudaSuccess;
}

// Bytes after the ring and staging area: barriers, TMEM slot, flags and row scales.
static constexpr int kTail = 1024;

static int stages_for(const DraftStepArgs& a, int G) {
    const int s = (g_budget - 1024 - ubytes_for(a, G) - kTail) / STAGE_BYTES;
    // the tail holds 2 s + 2 NACC + 4 mbarriers, the TMEM slot and flags (16 B), rs[16], the chain's
    // tokens [20] and per-warp bests [2][8]
    return (2 * s + 2 * NACC + 4) * 8 + 16 + (16 + 20 + 16) * 4 <= kTail ? s : 0;
}

bool draft_step_tc_ok(const DraftStepArgs& a, int G) {
    if (g_budget == 0 || !a.maps) return false;
    const int hd = a.nh > 0 ? a.d / a.nh : 0;
    if (a.gamma < 1 || a.gamma > GMAX || a.nL < 1 || a.nL > MAXL || (hd != 64 && hd != 128) || a.d % TM != 0 ||
        a.F % KB != 0 || a.H % 8 != 0 || a.d % a.nh != 0 || a.V < 1 || a.nchunks < 1)
        return false;
    if (a.nh * a.nchunks > G || a.nh > NTHR) return false;  // one attention item per CTA
    // the chain's lanes hold r / 64 16-byte chunks of a row: r in {64, 128, 256, 512}
    if (a.chain && ((a.r != 64 && a.r != 128 && a.r != 256 && a.r != 512) || !a.mk || !a.w1 || !a.w2 || !a.conf_w ||
                    !a.tokens || !a.conf))
        return false;
    const int S = stages_for(a, G);
    if (S < 4) return false;
    // the chain keeps its slice's base logits (every position) in the ring and staging area
    if (a.chain && (size_t)a.gamma * ((a.V + G - 1) / G) * 4 + 128 > (size_t)S * STAGE_BYTES + ubytes_for(a, G))
        return false;
    return true;
}

cudaError_t draft_step_tc(const DraftStepArgs& a, int G, cudaStream_t st) {
    if (!draft_step_tc_ok(a, G)) return cudaErrorInvalidValue;
    StepParams p{};
    p.x = a.x;
    p.qkv = a.qkv;
    p.gu = a.gu;
    p.y = a.y;
    p.U = a.U;
    p.act = reinterpret_cast<bf16*>(a.act);
    p.apart = a.apart;
    p.hcnt = a.hcnt;
    p.cache = reinterpret_cast<bf16*>(a.cache);
    p.layer_stride = a.layer_stride;
    p.kv_off = a.kv_off;
    p.max_rows = a.max_rows;
    p.seq_len = a.seq_len;
    p.embed = reinterpret_cast<const bf16*>(a.embed);
    p.anchor_dev = a.anchor_dev;
    p.anchor = a.anchor;
    p.block_const = a.block_const;
    for (int i = 0; i < a.nL; ++i) {
        p.attn_norm[i] = a.attn_norm[i];
        p.ff_norm[i] = a.ff_norm[i];
    }
    p.out_norm = a.out_norm;
    p.maps = reinterpret_cast<const CUtensorMap*>(a.maps);
    p.d = a.d;
    p.F = a.F;
    p.H = a.H;
    p.V = a.V;
    p.nh = a.nh;
    p.nL = a.nL;
    p.gamma = a.gamma;
    p.act_kind = a.act_kind;
    p.nchunks = a.nchunks;
    p.eps = a.eps;
    p.ubytes = ubytes_for(a, G);
    p.nstage = stages_for(a, G);
    p.bar = a.bar;
    p.epoch = a.epoch;
    p.err = a.err;
    p.chain = a.chain;
    p.r = a.r;
    p.w1 = reinterpret_cast<const bf16*>(a.w1);
    p.w2 = reinterpret_cast<const bf16*>(a.w2);
    p.conf_w = a.conf_w;
    p.tokens = a.tokens;
    p.conf = a.conf;
    p.logits = a.logits;
    p.mk = a.mk;
    const size_t smem = 1024 + (size_t)p.nstage * STAGE_BYTES + p.ubytes + kTail;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(NTHR);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int hd = a.d / a.nh;
    cudaError_t e = hd == 64 ? cudaLaunchKernelEx(&cfg, k_draft_step_tc<64>, p)
                             : cudaLaunchKernelEx(&cfg, k_draft_step_tc<128>, p);
    note_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace dspark
