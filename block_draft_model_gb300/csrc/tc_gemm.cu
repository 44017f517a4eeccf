// Tensor-core GEMM for sm_100-family GPUs (tcgen05 + TMA + TMEM), bf16 in, fp32 accumulate:
//   acc[m, n] = sum_k A[m, k] W[n, k]     A: [M, K] bf16, W: [N, K] bf16 (K contiguous)
// and the GEMM epilogues of epilogue.cuh.
//
// Persistent, warp-specialised CTA (one per SM, 192 threads):
//   warp 0     TMA producer: 128x64 A and 256x64 W tiles (128-byte swizzle) into a
//              STAGES-deep shared-memory ring, one mbarrier (with transaction
//              bytes) per stage;
//   warp 1     allocates 512 TMEM columns (two 128x256 fp32 accumulators) and one
//              elected lane issues tcgen05.mma (M 128, N 256, K 16) per 16-wide
//              K slice; tcgen05.commit frees a stage when its MMAs retire and
//              signals the epilogue when a tile's accumulator is complete;
//   warps 2-5  epilogue: tcgen05.ld of their 32 TMEM lanes (= tile rows), then
//              the epilogue functor, while the MMA warp fills the other
//              accumulator.
// Every mbarrier wait is bounded (about one second of %globaltimer); on a
// timeout the kernel records DSPARK_DEVERR_TIMEOUT, stops every role, drains
// its own MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdio.h>

#include "epilogue.cuh"
#include "tc_common.cuh"
#include "tc_gemm.cuh"

namespace dspark {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int TMEM_COLS = 2 * BN;     // two accumulators
constexpr int NTHREADS = 192;
using namespace tc;

// Per epilogue warp, a 32 x 32 fp32 block (rows padded to 36 floats) through which the
// plain fp32 store is transposed: each warp store then writes four whole 128-byte lines
// instead of touching 32 lines with 16 bytes each.
constexpr int STG_LD = 36;
constexpr int STG_BYTES = 4 * 32 * STG_LD * 4;
constexpr size_t smem_bytes() { return 1024 + (size_t)STAGES * (A_BYTES + B_BYTES) + 256 + STG_BYTES; }
// The EPI_MARKOV_T instance: B (the <= 128 sequences) in 128-row stages, and per epilogue warp two 32 x 32
// fp32 buffers of base logits, filled by cp.async a tile ahead of their use.
constexpr int BN_MK = 128;
constexpr int B_BYTES_MK = BN_MK * BK * 2;      // 16 KB
constexpr int UBUF_BYTES = 32 * 32 * 4;         // one warp's 32 sequences x 32 vocabulary rows
constexpr int STAGES_MK = 4;
constexpr size_t smem_bytes_mk() { return 1024 + (size_t)STAGES_MK * (A_BYTES + B_BYTES_MK) + 256 + 8 * 2 * UBUF_BYTES; }

struct TileMap {
    int nM, nN;
    bool n_fast;
    int ks;      // K ranges per output tile (consecutive work units)
    int groups;  // independent problems of the same shape (third map coordinate = group)
    int map3d;   // the tensor maps are 3-D (grouped launches, also with one group)
    int a2d;     // grouped launch whose A is one 2-D matrix shared by every group
    int bn;      // columns per tile
    __device__ __forceinline__ void at(int t, int& m0, int& n0, int& s, int& g) const {
        const int per = nM * nN * ks;
        g = t / per;
        t -= g * per;
        s = t % ks;
        t /= ks;
        int mi, ni;
        if (n_fast) {
            mi = t / nN;
            ni = t - mi * nN;
        } else {
            ni = t / nM;
            mi = t - ni * nM;
        }
        m0 = mi * BM;
        n0 = ni * bn;
    }
};

// MK: the instance for EPI_MARKOV_T, with eight epilogue warps (two per TMEM lane quarter, taking
// alternate 32-column chunks) that issue their chunk's base-logit loads before the accumulator is ready.
constexpr int NTHREADS_MK = 320;
// EK: the epilogue kind the instance is compiled for (EK < 0: any, read from ep at run time);
// EPI_MARKOV_T is the instance MK described above.
template <int EK>
__global__ void __launch_bounds__(EK == EPI_MARKOV_T ? NTHREADS_MK : NTHREADS, 1)
    k_tc_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int M, int N, int K,
              TileMap tm, EpiParams ep, int* err) {
    constexpr bool MK = EK == EPI_MARKOV_T;
    const int kind = EK >= 0 ? EK : ep.kind;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sA = smem_u32(smem);
    constexpr int BNk = MK ? BN_MK : BN;
    constexpr int STAGESk = MK ? STAGES_MK : STAGES;
    constexpr int B_BYTESk = BNk * BK * 2;
    const uint32_t sB = sA + STAGESk * A_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGESk * (A_BYTES + B_BYTESk));
    uint64_t* full = bars;                      // [STAGESk]
    uint64_t* empty = bars + STAGESk;            // [STAGESk]
    uint64_t* acc_full = bars + 2 * STAGESk;     // [2]
    uint64_t* acc_empty = bars + 2 * STAGESk + 2;  // [2]
    uint64_t* drain = bars + 2 * STAGESk + 4;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGESk + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* stage_f32 = reinterpret_cast<float*>(smem + STAGESk * (A_BYTES + B_BYTESk) + 256);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles = tm.nM * tm.nN * tm.ks * tm.groups;
    const int nkb = (K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGESk; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], MK ? 8 : 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();  // operands and outputs are shared with earlier kernels of the stream
    pdl_trigger();

    if (warp == 0) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(&tmB) : "memory");
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                int m0, n0, s, g;
                tm.at(t, m0, n0, s, g);
                if constexpr (MK) {
                    // the tile's base-logit rows into L2, a tile ahead of the epilogue that reads them
                    const int span = (min(M, m0 + BM) - m0) * 4 & ~15;
                    if (span > 0 && (ep.ldo & 3) == 0 && ((uintptr_t)ep.mk_U & 15) == 0)
                        for (int j = n0; j < min(N, n0 + BNk); ++j)
                            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                                             ep.mk_U + ((int64_t)j * ep.gamma + ep.mk_k) * ep.ldo + m0),
                                         "r"(span)
                                         : "memory");
                }
                const int kb1 = (s + 1) * nkb / tm.ks;
                for (int kb = s * nkb / tm.ks; kb < kb1; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], A_BYTES + B_BYTESk);
                    if (tm.map3d) {
                        if (tm.a2d) tma_load_2d(sA + stage * A_BYTES, &tmA, &full[stage], kb * BK, m0);
                        else tma_load_3d(sA + stage * A_BYTES, &tmA, &full[stage], kb * BK, m0, g);
                        tma_load_3d(sB + stage * B_BYTESk, &tmB, &full[stage], kb * BK, n0, g);
                    } else {
                        tma_load_2d(sA + stage * A_BYTES, &tmA, &full[stage], kb * BK, m0);
                        tma_load_2d(sB + stage * B_BYTESk, &tmB, &full[stage], kb * BK, n0);
                    }
                    if (++stage == STAGESk) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        __syncwarp();  // lane 0 rejoins its warp before the CTA-wide barrier
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, buf = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                if (!mbar_wait(&acc_empty[buf], acc_phase ^ 1u, abort_flag)) break;
                tc_fence_after();
                int m0, n0, s, g;
                tm.at(t, m0, n0, s, g);
                const int kb0 = s * nkb / tm.ks, kb1 = (s + 1) * nkb / tm.ks;
                // a narrow last (or only) column tile multiplies only its 16-aligned width
                const int n_rem = N - n0;
                const uint32_t id = idesc(BM, n_rem >= BNk ? BNk : (n_rem + 15) & ~15);
                const uint32_t d_tmem = tmem + buf * BNk;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t da = sdesc(sA + stage * A_BYTES);
                    const uint64_t db = sdesc(sB + stage * B_BYTESk);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)  // +32 bytes per 16-wide K slice inside the swizzled row
                        umma(d_tmem, da + (uint64_t)(2 * k), db + (uint64_t)(2 * k), id, (kb > kb0 || k) ? 1u : 0u);
                    umma_commit(&empty[stage]);
                    if (++stage == STAGESk) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(&acc_full[buf]);
                if (++buf == 2) {
                    buf = 0;
                    acc_phase ^= 1u;
                }
            }
            // drain: every MMA issued by this thread has retired once `drain` completes
            umma_commit(drain);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(drain, 0) && globaltimer() - t0 < TIMEOUT_NS) {
            }
        }
        __syncwarp();
    } else if constexpr (MK) {
        // epilogue warps 2..9: TMEM lanes 32*(warp % 4) .. +31 (vocabulary rows), chunks half, half + 2, ...
        // The base logits of the warp's first chunk come through its two shared-memory buffers, copied a
        // tile ahead (cp.async, 16-byte pieces): tile t's block is [32 sequences][32 vocabulary rows].
        const int q = warp & 3, half = (warp - 2) >> 2;
        float* ub = reinterpret_cast<float*>(smem + STAGESk * (A_BYTES + B_BYTESk) + 256) + (warp - 2) * 2 * 1024;
        const bool cp_ok = (ep.ldo & 3) == 0 && ((uintptr_t)ep.mk_U & 15) == 0;
        auto fill = [&](int t, float* dst) {
            int m0, n0, s, g;
            tm.at(t, m0, n0, s, g);
            const int nb0 = n0 + half * 32, c0 = m0 + q * 32;
#pragma unroll
            for (int i = 0; i < 8; ++i) {  // 256 pieces: sequence j = piece / 8, columns 4 * (piece % 8) ..
                const int pc = lane + 32 * i, j = pc >> 3, col = c0 + (pc & 7) * 4;
                const int bytes = nb0 + j < N && col < M ? min(4, M - col) * 4 : 0;
                const float* src = bytes ? ep.mk_U + ((int64_t)(nb0 + j) * ep.gamma + ep.mk_k) * ep.ldo + col : ep.mk_U;
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst + j * 32 + (pc & 7) * 4)),
                             "l"(src), "r"(bytes)
                             : "memory");
            }
        };
        int buf = 0, it = 0;
        uint32_t acc_phase = 0;
        if (cp_ok && (int)blockIdx.x < tiles) fill(blockIdx.x, ub);
        asm volatile("cp.async.commit_group;" ::: "memory");
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
            __syncwarp();  // every lane is done with the buffer the next copy overwrites
            if (cp_ok && t + (int)gridDim.x < tiles) fill(t + gridDim.x, ub + ((it + 1) & 1) * 1024);
            asm volatile("cp.async.commit_group;" ::: "memory");
            int m0, n0, s, g;
            tm.at(t, m0, n0, s, g);
            const int row = m0 + q * 32 + lane;
            const bool rows_in = m0 + q * 32 < M;  // warp-uniform
            const float* us = ub + (it & 1) * 1024;
            if (!mbar_wait(&acc_full[buf], acc_phase, abort_flag)) break;
            tc_fence_after();
            asm volatile("cp.async.wait_group 1;" ::: "memory");  // this tile's block (the next may be in flight)
            __syncwarp();
            const uint32_t base = tmem + buf * BNk + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
            for (int c = half; c < BNk / 32; c += 2) {
                const int nb = n0 + c * 32;
                if (nb >= N) break;  // columns past N were not multiplied
                uint32_t r[32];
                tmem_ld32(base + c * 32, r);
                if (rows_in) {
                    float v[32], u[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                    if (c == half && cp_ok) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) u[j] = us[j * 32 + lane];
                    } else {
                        markov_u32_load(ep, row, row < M, nb, N, u);
                    }
                    markov_t32_u(ep, row, row < M, nb, N, v, u);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
            if (++buf == 2) {
                buf = 0;
                acc_phase ^= 1u;
            }
        }
        asm volatile("cp.async.wait_group 0;" ::: "memory");  // no copy outlives the kernel
    } else {
        // epilogue warps 2..5: TMEM lanes 32*(warp % 4) .. +31
        const int q = warp & 3;
        int buf = 0;
        uint32_t acc_phase = 0;
        float* stg = stage_f32 + q * 32 * STG_LD;
        const bool coalesce = kind == EPI_STORE_F32 && (ep.ldo & 3) == 0 && ((uintptr_t)ep.out_f32 & 15) == 0;
        // bf16 K/V cache rows, 64 columns at a time (whole 128-byte lines); a 64-column pair never
        // straddles K and V when the cache row width is a multiple of 64
        const int kvw = ep.d_kv ? ep.d_kv : ep.d;
        const bool kv16 = kind == EPI_KV_CACHE && ep.cache_dtype == DT_BF16 && (kvw & 63) == 0 &&
                          ((uintptr_t)ep.cache & 15) == 0 && ((ep.seq_stride | ep.kv_off | ep.group_stride) & 7) == 0;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
            int m0, n0, s, g;
            tm.at(t, m0, n0, s, g);
            if (!mbar_wait(&acc_full[buf], acc_phase, abort_flag)) break;
            tc_fence_after();
            const int row = m0 + q * 32 + lane;
            const int orow = row + s * ep.split_rows;  // output row (K range s of a split product)
            const uint32_t base = tmem + buf * BN + ((uint32_t)(q * 32) << 16);
            // K/V cache element offset of this lane's row (without the column), and whether it is stored
            int64_t kv_row = 0;
            int kv_ok = 0;
            if (kv16 && row < M) {
                const int slot = ep.row_seq ? ep.row_seq[row] : 0;
                const int pos = ep.row_pos ? ep.row_pos[row] : (slot >= 0 ? ep.seq_len[slot] + row : -1);
                kv_ok = slot >= 0 && pos >= 0 && pos < ep.max_rows;
                kv_row = g * ep.group_stride + (int64_t)slot * ep.seq_stride + (int64_t)pos * kvw;
            }
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                const int nb = n0 + c * 32;
                if (nb >= N) break;  // columns past N were not multiplied
                if (kv16 && (c & 1) == 0 && nb + 64 <= N) {  // warp-wide: every lane takes part
                    uint32_t r0[32], r1[32];
                    tmem_ld32(base + c * 32, r0);
                    tmem_ld32(base + c * 32 + 32, r1);
                    // lane l's 64 bf16 into row l of the block (144-byte rows), then 8 lanes per row
                    // store its 128 bytes: 4 rows per warp store
                    uint4* srow = reinterpret_cast<uint4*>(stg + lane * STG_LD);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t* rr = j < 4 ? r0 + 8 * j : r1 + 8 * (j - 4);
                        uint32_t w4[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            __nv_bfloat162 pr = __floats2bfloat162_rn(__uint_as_float(rr[2 * i]), __uint_as_float(rr[2 * i + 1]));
                            w4[i] = *reinterpret_cast<uint32_t*>(&pr);
                        }
                        srow[j] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                    __syncwarp();
                    const int64_t col = nb < kvw ? nb : ep.kv_off + (nb - kvw);
                    bf16* cache = reinterpret_cast<bf16*>(ep.cache);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int rr = (lane >> 3) + 4 * i;
                        const uint4 val = *reinterpret_cast<const uint4*>(stg + rr * STG_LD + (lane & 7) * 4);
                        const int64_t rb = __shfl_sync(0xffffffffu, kv_row, rr);
                        if (__shfl_sync(0xffffffffu, kv_ok, rr))
                            *reinterpret_cast<uint4*>(cache + rb + col + (lane & 7) * 8) = val;
                    }
                    __syncwarp();
                    ++c;
                    continue;
                }
                uint32_t r[32];
                tmem_ld32(base + c * 32, r);
                if (coalesce && nb + 32 <= N) {  // warp-wide: every lane takes part
                    // lane l's row (32 columns) into row l of the block, then each lane
                    // takes 4 columns of rows l/8, l/8 + 4, ...: 8 lanes cover one row's 128 bytes
                    float4* srow = reinterpret_cast<float4*>(stg + lane * STG_LD);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        srow[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                              __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                    __syncwarp();
                    const int c4 = (lane & 7) * 4;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int rr = (lane >> 3) + 4 * i;
                        const int mrow = m0 + q * 32 + rr;
                        const float4 val = *reinterpret_cast<const float4*>(stg + rr * STG_LD + c4);
                        if (mrow < M)
                            *reinterpret_cast<float4*>(ep.out_f32 + (int64_t)(mrow + s * ep.split_rows) * ep.ldo + nb +
                                                       c4) = val;
                    }
                    __syncwarp();
                } else if (EK < 0 && kind == EPI_MARKOV_T) {  // warp-wide: every lane takes part
                    if (m0 + q * 32 < M) {
                        float v[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                        markov_t32(ep, row, row < M, nb, N, v);
                    }
                } else if (row < M) {
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                    epi_row32_k<EK>(ep, orow, nb, N, v, g);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
            if (++buf == 2) {
                buf = 0;
                acc_phase ^= 1u;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) atomicOr(err, DEVERR_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

// ---------------------------------------------------------------------------------------------
// Wide form for few activation rows against many weight rows (the vocabulary projection of a
// batched draft): the weights are the MMA's 128-row side and the activation rows its N side,
// so the fp32 result rows are written along the vocabulary (a warp store covers 32 consecutive
// entries of one output row) and no activation tile is padded to 128 rows.
//   acc[n, m] = sum_k W[n, k] A[m, k]  for a 128-row weight tile and a group of <= 160 rows m.
// The M rows are cut into ng groups of at most 160 (ng <= 2); tile t is weight tile t / ng and
// group t % ng, so the groups of one weight tile run on neighbouring CTAs at the same time and
// the weight tile comes from DRAM once.  Each tile's accumulator takes one of three 160-column
// TMEM slots in turn (the CTA's u-th tile, slot u % 3): the MMAs of a tile overlap the epilogues
// of the two before it.  Warps 2-5 drain the even tiles and warps 6-9 the odd ones; each set
// waits on barriers of its own (u % 6), so it always observes its tiles' completions in order.
namespace wide {
constexpr int UW = 160;          // most columns per tile
constexpr int SLOTS = 3;
constexpr int NTHREADS = 320;    // producer, MMA, 2 x 4 epilogue warps
constexpr int W_BYTES = 128 * BK * 2;  // 16 KB weight tile per stage
constexpr int MAX_M = 2 * UW;
constexpr int SMEM_MAX = 232448;  // 227 KB, the opt-in maximum per CTA
constexpr int BAR_BYTES = 256;
inline int groups(int M) { return M > UW ? 2 : 1; }
// rows per group, a multiple of 16 (the last group may be narrower)
inline int group_w(int M) {
    const int na = (M + 15) & ~15, g = groups(M);
    return (((na + g - 1) / g) + 15) & ~15;
}
inline int stage_bytes(int M) { return W_BYTES + group_w(M) * BK * 2; }
inline int stages(int M) {
    const int s = (SMEM_MAX - 1024 - BAR_BYTES) / stage_bytes(M);
    return s > 8 ? 8 : s;
}
inline size_t smem(int M) { return 1024 + (size_t)stages(M) * stage_bytes(M) + BAR_BYTES; }
}  // namespace wide

__global__ void __launch_bounds__(wide::NTHREADS, 1)
    k_tc_wide(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW, int M, int N, int K,
              int S, int gw, EpiParams ep, int* err) {
    using namespace wide;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int na = (M + 15) & ~15;
    const int ng = (na + gw - 1) / gw;
    const uint32_t sbytes = W_BYTES + gw * BK * 2;
    const uint32_t s0 = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)S * sbytes);
    uint64_t* full = bars;                 // [S]
    uint64_t* empty = bars + 8;            // [S]
    uint64_t* acc_full = bars + 16;        // [6]
    uint64_t* acc_empty = bars + 22;       // [SLOTS]
    uint64_t* drain = bars + 25;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 26);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles = ((N + 127) / 128) * ng;
    const int nkb = (K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 6; ++b) mbar_init(&acc_full[b], 1);
        for (int b = 0; b < SLOTS; ++b) mbar_init(&acc_empty[b], 4);
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(&tmW) : "memory");
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                const int wt = t / ng, g = t - wt * ng;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sb = s0 + stage * sbytes;
                    mbar_arrive_expect_tx(&full[stage], sbytes);
                    tma_load_2d(sb, &tmW, &full[stage], kb * BK, wt * 128);
                    tma_load_2d(sb + W_BYTES, &tmA, &full[stage], kb * BK, g * gw);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, u = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++u) {
                const int g = t % ng;
                const int width = na - g * gw < gw ? na - g * gw : gw;
                const uint32_t id = idesc(128, width);
                const uint32_t d_tmem = tmem + (u % SLOTS) * UW;
                if (!mbar_wait(&acc_empty[u % SLOTS], ((u / SLOTS) & 1u) ^ 1u, abort_flag)) break;
                tc_fence_after();
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sb = s0 + stage * sbytes;
                    const uint64_t dw = sdesc(sb), da = sdesc(sb + W_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        umma(d_tmem, dw + (uint64_t)(2 * k), da + (uint64_t)(2 * k), id, (kb || k) ? 1u : 0u);
                    umma_commit(&empty[stage]);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(&acc_full[u % 6]);
            }
            umma_commit(drain);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(drain, 0) && globaltimer() - t0 < TIMEOUT_NS) {
            }
        }
        __syncwarp();
    } else {
        // epilogue: set h drains the CTA's tiles u with u % 2 == h; TMEM lanes 32*(warp % 4) .. +31
        // are weight rows
        const int h = (warp - 2) >> 2, q = warp & 3;
        int u = h;
        for (int t = blockIdx.x + h * gridDim.x; t < tiles; t += 2 * gridDim.x, u += 2) {
            if (!mbar_wait(&acc_full[u % 6], (uint32_t)(u / 6) & 1u, abort_flag)) break;
            tc_fence_after();
            const int wt = t / ng, g = t - wt * ng;
            const int width = na - g * gw < gw ? na - g * gw : gw;
            const int n = wt * 128 + q * 32 + lane;
            const int mend = g * gw + width < M ? g * gw + width : M;  // the group's rows end here
            const uint32_t base = tmem + (u % SLOTS) * UW + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < width; c += 32) {
                uint32_t r[32];
                tmem_ld32(base + c, r);
                const int m0 = g * gw + c;
                if (n < N) {
                    float* o = ep.out_f32 + (int64_t)m0 * ep.ldo + n;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (m0 + i < mend) o[(int64_t)i * ep.ldo] = __uint_as_float(r[i]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[u % SLOTS]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) atomicOr(err, DEVERR_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
    }
}

// The instance for an epilogue kind (the Markov one is launched on its own): one per kind the path
// uses, so that each carries only its own epilogue code; other kinds take the generic one.
decltype(&k_tc_gemm<-1>) gemm_kernel(int kind) {
    switch (kind) {
        case EPI_STORE_F32: return k_tc_gemm<EPI_STORE_F32>;
        case EPI_ADD_F32: return k_tc_gemm<EPI_ADD_F32>;
        case EPI_QKV: return k_tc_gemm<EPI_QKV>;
        case EPI_SWIGLU: return k_tc_gemm<EPI_SWIGLU>;
        case EPI_KV_CACHE: return k_tc_gemm<EPI_KV_CACHE>;
        default: return k_tc_gemm<-1>;
    }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
// Per device (the shared-memory attribute belongs to the device's context):
// -1 unknown, 0 unavailable, 1 available.
constexpr int kMaxDev = 64;
int g_state[kMaxDev] = {-1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1,
                        -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1,
                        -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1};

bool init_encode() {
    int dev = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return false;
    if (g_state[dev] >= 0) return g_state[dev] == 1;
    g_state[dev] = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
    if (major != 10) return false;
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return false;
        g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    }
    for (auto fn : {k_tc_gemm<-1>, k_tc_gemm<EPI_STORE_F32>, k_tc_gemm<EPI_ADD_F32>, k_tc_gemm<EPI_QKV>,
                    k_tc_gemm<EPI_SWIGLU>, k_tc_gemm<EPI_KV_CACHE>})
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes()) != cudaSuccess)
            return false;
    if (cudaFuncSetAttribute(k_tc_gemm<EPI_MARKOV_T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_bytes_mk()) != cudaSuccess)
        return false;
    if (cudaFuncSetAttribute(k_tc_wide, cudaFuncAttributeMaxDynamicSharedMemorySize, wide::SMEM_MAX) != cudaSuccess)
        return false;
    g_state[dev] = 1;
    return true;
}

// 2-D bf16 tensor map: rows x cols (cols contiguous, row stride ld elements), box box_rows x 64.
bool encode(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

bool tc_available() { return init_encode(); }

bool tc_prepare_grouped(TcWeight& w, const void* ptr, int groups, int64_t group_stride, int rows, int K, bool a_side) {
    w.ready = false;
    w.ready128 = false;
    w.ptr = ptr;
    w.N = rows;
    w.K = K;
    if (!init_encode() || groups < 1 || K % 8 != 0 || ((uintptr_t)ptr & 15) != 0 || group_stride % 8 != 0) return false;
    cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)rows, (cuuint64_t)groups};
    cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)group_stride * 2};
    cuuint32_t box[3] = {(cuuint32_t)BK, (cuuint32_t)(a_side ? BM : BN), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(reinterpret_cast<CUtensorMap*>(w.tmap), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                          const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    w.ready = r == CUDA_SUCCESS;
    return w.ready;
}

cudaError_t tc_gemm_grouped(const TcWeight& a, const TcWeight& w, int groups, int M, int N, int K, const EpiParams& ep,
                            int num_sms, int* err, cudaStream_t st, bool a_shared) {
    if (!a.ready || !w.ready || groups < 1 || !tc_gemm_ok(M, N, K) || M > a.N || N > w.N || K != w.K || K != a.K)
        return cudaErrorInvalidValue;
    if (a_shared && !a.ready128) return cudaErrorInvalidValue;
    TileMap tm;
    tm.nM = (M + BM - 1) / BM;
    tm.nN = (N + BN - 1) / BN;
    tm.bn = BN;
    tm.n_fast = tm.nN <= tm.nM;
    tm.ks = 1;
    tm.groups = groups;
    tm.map3d = 1;
    tm.a2d = a_shared ? 1 : 0;
    const int tiles = tm.nM * tm.nN * groups;
    const int grid = tiles < num_sms ? tiles : num_sms;
    launch(gemm_kernel(ep.kind), grid, NTHREADS, smem_bytes(), st,
           *reinterpret_cast<const CUtensorMap*>(a_shared ? a.tmap128 : a.tmap),
           *reinterpret_cast<const CUtensorMap*>(w.tmap), M, N, K, tm, ep, err);
    note_launch();
    return cudaGetLastError();
}

bool tc_encode_slot_map(void* map, const void* W, int64_t rows, int64_t K, bool three_d) {
    if (!init_encode() || K % 512 != 0 || ((uintptr_t)W & 15) != 0) return false;
    CUresult r;
    if (three_d) {
        // (64 elements of a 128-byte column block, row, column block): one box = 16 rows x 512
        cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(K / 64)};
        cuuint64_t strides[2] = {(cuuint64_t)(K * 2), 128};
        cuuint32_t box[3] = {64, 16, 8};
        cuuint32_t estr[3] = {1, 1, 1};
        r = g_encode(reinterpret_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(W), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
        cuuint64_t strides[1] = {(cuuint64_t)(K * 2)};
        cuuint32_t box[2] = {64, 16};
        cuuint32_t estr[2] = {1, 1};
        r = g_encode(reinterpret_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS;
}

cudaError_t tc_prepare(TcWeight& w, const void* ptr, int N, int K) {
    w.ready = false;
    w.ready128 = false;
    w.ptr = ptr;
    w.N = N;
    w.K = K;
    if (!init_encode()) return cudaSuccess;
    if (K % 8 != 0 || ((uintptr_t)ptr & 15) != 0) return cudaSuccess;
    if (!encode(reinterpret_cast<CUtensorMap*>(w.tmap), ptr, N, K, K, BN)) return cudaSuccess;
    w.ready = true;
    w.ready128 = encode(reinterpret_cast<CUtensorMap*>(w.tmap128), ptr, N, K, K, 128);
    return cudaSuccess;
}

void tc_release(TcWeight& w) { w.ready = w.ready128 = false; }

bool tc_gemm_ok(int M, int N, int K) { return init_encode() && M >= 1 && N >= 1 && K >= BK && K % 8 == 0; }

// Measured on the 262144-row vocabulary projection (K 1024): the wide form wins at M <= 160 (one
// group; the tiles pad M to 128 or 256) and at 257..320 (the tiles pad to 384); in between the
// tiles' 256 rows carry little padding and they are the faster form.
bool tc_wide_preferred(int M, int N, int num_sms) {
    return (M <= wide::UW || (M > 2 * BM && M <= wide::MAX_M)) && (N + 127) / 128 >= num_sms;
}

bool tc_wide_ok(const TcWeight& w, int M, int N, int K, const EpiParams& ep) {
    return w.ready128 && tc_gemm_ok(M, N, K) && M <= wide::MAX_M && N <= w.N && K == w.K &&
           ep.kind == EPI_STORE_F32 && ep.out_f32 != nullptr;
}

cudaError_t tc_gemm_wide(const void* A, int64_t lda, const TcWeight& w, int M, int N, int K, const EpiParams& ep,
                         int num_sms, int* err, cudaStream_t st) {
    if (!tc_wide_ok(w, M, N, K, ep)) return cudaErrorInvalidValue;
    if (lda % 8 != 0 || ((uintptr_t)A & 15) != 0) return cudaErrorInvalidValue;
    CUtensorMap tmA;
    const int gw = wide::group_w(M);
    if (!encode(&tmA, A, M, K, lda, gw)) return cudaErrorInvalidValue;
    const int S = wide::stages(M);
    if (S < 2) return cudaErrorInvalidValue;
    const int tiles = (N + 127) / 128 * wide::groups(M);
    const int grid = tiles < num_sms ? tiles : num_sms;
    launch(k_tc_wide, grid, wide::NTHREADS, wide::smem(M), st, tmA, *reinterpret_cast<const CUtensorMap*>(w.tmap128),
           M, N, K, S, gw, ep, err);
    note_launch();
    return cudaGetLastError();
}

cudaError_t tc_gemm(const void* A, int64_t lda, const TcWeight& w, int M, int N, int K, const EpiParams& ep,
                    int num_sms, int* err, cudaStream_t st, int ksplit) {
    if (!w.ready || !tc_gemm_ok(M, N, K) || N > w.N || K != w.K) return cudaErrorInvalidValue;
    if (ksplit < 1 || (ksplit > 1 && (ep.kind != EPI_STORE_F32 || ep.split_rows < M || ksplit > (K + BK - 1) / BK)))
        return cudaErrorInvalidValue;
    if (lda % 8 != 0 || ((uintptr_t)A & 15) != 0) return cudaErrorInvalidValue;
    CUtensorMap tmA;
    if (!encode(&tmA, A, M, K, lda, BM)) return cudaErrorInvalidValue;
    // the Markov instance takes B (the sequences) in 128-row tiles through the 128-row-box map
    const bool mk = ep.kind == EPI_MARKOV_T;
    if (mk && !w.ready128) return cudaErrorInvalidValue;
    TileMap tm;
    tm.bn = mk ? BN_MK : BN;
    tm.nM = (M + BM - 1) / BM;
    tm.nN = (N + tm.bn - 1) / tm.bn;
    tm.n_fast = tm.nN <= tm.nM;
    tm.ks = ksplit;
    tm.groups = 1;
    tm.map3d = 0;
    tm.a2d = 0;
    const int tiles = tm.nM * tm.nN * ksplit;
    const int grid = tiles < num_sms ? tiles : num_sms;
    if (mk)
        launch(k_tc_gemm<EPI_MARKOV_T>, grid, NTHREADS_MK, smem_bytes_mk(), st, tmA,
               *reinterpret_cast<const CUtensorMap*>(w.tmap128), M, N, K, tm, ep, err);
    else
        launch(gemm_kernel(ep.kind), grid, NTHREADS, smem_bytes(), st, tmA, *reinterpret_cast<const CUtensorMap*>(w.tmap), M,
               N, K, tm, ep, err);
    note_launch();
    return cudaGetLastError();
}

}  // namespace dspark
