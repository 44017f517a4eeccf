// Weight-streaming tensor-core GEMM for a handful of activation rows (the
// batch-1 draft step: M = gamma <= 16), "swap-AB" on tcgen05:
//   acc[m, n] = sum_k X[m, k] W[n, k]       W: [N, K] bf16, X: [M <= 16, K] bf16
// W supplies the MMA's M side (128 weight rows per tile, streamed once from
// HBM by TMA with the 128-byte swizzle) and X the N side (16 columns; TMA fills
// the rows beyond M with zeros).  Each tcgen05.mma is 128x16x16; the fp32
// accumulator is 16 TMEM columns.
//
// The work is HBM-bound, so the layout serves bytes in flight: a CTA owns one
// (128-row tile, K slice) unit, keeps STAGES 18 KB stages in flight, and two
// CTAs fit on an SM.  When the weight rows alone cannot fill the GPU, K is split
// over CTAs; each CTA writes its 128x16 partial to scratch and the last CTA of
// the tile (ticket counter, no spinning) adds the partials in split order and
// applies the epilogue, so results do not depend on scheduling.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdlib.h>

#include "epilogue.cuh"
#include "tc_common.cuh"
#include "tc_gemm.cuh"

namespace dspark {

namespace {

using namespace tc;

constexpr int BM = 128, BN = 16, BK = 64, STAGES = 6;
constexpr int W_BYTES = BM * BK * 2;  // 16 KB
constexpr int X_BYTES = BN * BK * 2;  // 2 KB
constexpr int TMEM_COLS = 32;
constexpr int NTHREADS = 192;

// tail after the ring: barriers and flags (256 B), then the row-scale partials [8][16] (512 B)
constexpr size_t smem_bytes() { return 1024 + (size_t)STAGES * (W_BYTES + X_BYTES) + 768; }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Row-sum form: rsc[m] = 1 / sqrt(mean(x[m]^2) + eps) from the producer's 8-column sums
// (K / 8 of them per row), added by the four epilogue warps in a fixed order.
__device__ __forceinline__ void build_rowscale(const StreamNorm& sn, int K, float* red, float* rsc) {
    const int t = threadIdx.x - 64;  // 0..127
    const int m = t & 15, part = t >> 4;
    const int nP = K >> 3;
    float s = 0.f;
#pragma unroll 8
    for (int j = part; j < nP; j += 8) s += __ldcg(sn.ssp + j * 16 + m);
    red[part * 16 + m] = s;
    epi_bar();
    if (t < 16) {
        float a = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) a += red[q * 16 + t];
        rsc[t] = rsqrtf(a / (float)K + sn.eps);
    }
    epi_bar();
}

// EPI_ADD_F32 with the next projection's operand: x += v, xb = bf16(x * g[n]); returns x^2.
__device__ __forceinline__ float epi_add_xb(const EpiParams& ep, int m, int n, float v) {
    float* p = ep.out_f32 + (int64_t)m * ep.ldo + n;
    const float x = *p + v;
    *p = x;
    reinterpret_cast<bf16*>(ep.xb)[(int64_t)m * ep.ld_xb + n] = __float2bfloat16(x * ep.xb_g[n]);
    return x * x;
}

// grid: n_tiles * splits CTAs; CTA b handles tile b / splits, K blocks
// [s * kb_per, min(nkb, (s + 1) * kb_per)) with s = b % splits.
// EK: the epilogue kind the instance is compiled for (EK < 0: any, read from ep at run time);
// CLU: split-K partials reduced inside the cluster (else through scratch and tile tickets).
template <int EK, bool CLU>
__global__ void __launch_bounds__(NTHREADS, 2)
    k_tc_stream(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, int M, int N, int K,
                int splits, int kb_per, int cluster_reduce_arg, EpiParams ep, float* __restrict__ part,
                unsigned int* __restrict__ tickets, int* err, StreamNorm sn) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sW = smem_u32(smem);
    const uint32_t sX = sW + STAGES * W_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * (W_BYTES + X_BYTES));
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* acc_full = bars + 2 * STAGES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* is_last = reinterpret_cast<volatile int*>(tmem_slot + 2);
    float* rsc = reinterpret_cast<float*>(bars + 16);    // row scales [BN]
    float* rs_red = reinterpret_cast<float*>(bars + 32);  // row-sum partials [8][16]
    const bool rowscale = sn.ssp != nullptr;
    const int kind = EK >= 0 ? EK : ep.kind;
    constexpr bool cluster_reduce = CLU;
    (void)cluster_reduce_arg;
    // EPI_ADD_F32 that also writes the next operand and row sums
    const bool xbm = (EK < 0 || EK == EPI_ADD_F32) && ep.ssp != nullptr;
    // EPI_ADD_F32 reduced in the cluster: the residual entries this thread will own in the final
    // epilogue (at most two items of four activation rows), loaded while the weights stream; no other
    // thread of the kernel touches them
    const bool xpre_on = splits > 1 && cluster_reduce && kind == EPI_ADD_F32;
    float xpre[2][4];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x / splits, split = blockIdx.x - tile * splits;
    const int nkb = (K + BK - 1) / BK;
    const int kb0 = split * kb_per, kb1 = min(nkb, kb0 + kb_per);
    const int n0 = tile * BM;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
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

    if (warp == 0) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(&tmW) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(&tmX) : "memory");
            const uint32_t stage_tx = W_BYTES + X_BYTES;
            // The weights are never written by the step: the first ring of weight tiles
            // is requested before waiting for the kernels that produce X.
            const int pre = min(STAGES, kb1 - kb0);
            for (int i = 0; i < pre; ++i) {
                mbar_arrive_expect_tx(&full[i], stage_tx);
                tma_load_2d(sW + i * W_BYTES, &tmW, &full[i], (kb0 + i) * BK, n0);
            }
            pdl_wait();
            pdl_trigger();
            for (int i = 0; i < pre; ++i) tma_load_2d(sX + i * X_BYTES, &tmX, &full[i], (kb0 + i) * BK, 0);
            int stage = pre % STAGES;
            uint32_t phase = pre == STAGES ? 1u : 0u;
            for (int kb = kb0 + pre; kb < kb1; ++kb) {
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) break;
                mbar_arrive_expect_tx(&full[stage], stage_tx);
                tma_load_2d(sW + stage * W_BYTES, &tmW, &full[stage], kb * BK, n0);
                tma_load_2d(sX + stage * X_BYTES, &tmX, &full[stage], kb * BK, 0);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        } else {
            pdl_wait();
            pdl_trigger();
        }
        __syncwarp();  // lane 0 rejoins its warp before the CTA-wide barrier
    } else if (warp == 1) {
        pdl_wait();
        pdl_trigger();
        if (lane == 0) {
            const uint32_t id = idesc(BM, BN);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait(&full[stage], phase, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t dw = sdesc(sW + stage * W_BYTES);
                const uint64_t dx = sdesc(sX + stage * X_BYTES);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    umma(tmem, dw + (uint64_t)(2 * k), dx + (uint64_t)(2 * k), id, (kb > kb0 || k > 0) ? 1u : 0u);
                umma_commit(&empty[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            umma_commit(acc_full);  // also drains: completes once every MMA above has retired
            if (ok) {
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(acc_full, 0) && globaltimer() - t0 < TIMEOUT_NS) {
                }
            }
        }
        __syncwarp();
    } else {
        pdl_wait();  // the epilogue reads and writes buffers shared with earlier kernels
        pdl_trigger();
        if (xpre_on) {
            const int t = threadIdx.x - 64, rps = BM / splits;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int it = h * 128 + t;
                const int nn = n0 + split * rps + (it >> 2), cg = it & 3;
#pragma unroll
                for (int qq = 0; qq < 4; ++qq)
                    xpre[h][qq] = (it < rps * 4 && nn < N && 4 * cg + qq < M)
                                      ? __ldcg(ep.out_f32 + (int64_t)(4 * cg + qq) * ep.ldo + nn)
                                      : 0.f;
            }
        }
        if (rowscale) build_rowscale(sn, K, rs_red, rsc);
        const int q = warp & 3;
        const int row = q * 32 + lane;  // weight row within the tile
        const int n = n0 + row;
        float v[BN];
        bool have = mbar_wait(acc_full, 0, abort_flag) && !*abort_flag;
        if (have) {
            tc_fence_after();
            uint32_t r[BN];
            tmem_ld16(tmem + ((uint32_t)(q * 32) << 16), r);
#pragma unroll
            for (int m = 0; m < BN; ++m) v[m] = __uint_as_float(r[m]) * (rowscale ? rsc[m] : 1.f);
        } else {
#pragma unroll
            for (int m = 0; m < BN; ++m) v[m] = 0.f;
        }
        bool final_ = (splits == 1);
        if (splits > 1 && cluster_reduce) {
            // partial tile [128 rows][16] into this CTA's (now idle) first weight stage; the cluster
            // reduction below reads it through distributed shared memory
            float4* red = reinterpret_cast<float4*>(smem) + row * (BN / 4);
#pragma unroll
            for (int c = 0; c < BN / 4; ++c) red[c] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
        } else if (splits > 1) {
            float4* dst = reinterpret_cast<float4*>(part + (((int64_t)tile * splits + split) * BM + row) * BN);
#pragma unroll
            for (int c = 0; c < BN / 4; ++c) dst[c] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
            __threadfence();
            epi_bar();
            if (threadIdx.x == 64) {
                const unsigned int t = atomicAdd(&tickets[tile], 1u);
                *is_last = (t == (unsigned int)splits - 1);
            }
            epi_bar();
            if (*is_last) {
                __threadfence();
#pragma unroll
                for (int m = 0; m < BN; ++m) v[m] = 0.f;
                // splits added in order; four splits' loads in flight at a time
                int s = 0;
                for (; s + 4 <= splits; s += 4) {
                    float4 t[4][BN / 4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float4* src =
                            reinterpret_cast<const float4*>(part + (((int64_t)tile * splits + s + u) * BM + row) * BN);
#pragma unroll
                        for (int c = 0; c < BN / 4; ++c) t[u][c] = __ldcg(src + c);
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int c = 0; c < BN / 4; ++c) {
                            v[4 * c] += t[u][c].x;
                            v[4 * c + 1] += t[u][c].y;
                            v[4 * c + 2] += t[u][c].z;
                            v[4 * c + 3] += t[u][c].w;
                        }
                }
                for (; s < splits; ++s) {
                    const float4* src = reinterpret_cast<const float4*>(part + (((int64_t)tile * splits + s) * BM + row) * BN);
#pragma unroll
                    for (int c = 0; c < BN / 4; ++c) {
                        const float4 t = __ldcg(src + c);
                        v[4 * c] += t.x;
                        v[4 * c + 1] += t.y;
                        v[4 * c + 2] += t.z;
                        v[4 * c + 3] += t.w;
                    }
                }
                if (threadIdx.x == 64) tickets[tile] = 0u;
                final_ = true;
            }
        }
        if (final_ && have) {
            if (kind == EPI_SWIGLU) {
                // (gate, up) rows are adjacent lanes: even lanes take their odd neighbour's value
#pragma unroll
                for (int m = 0; m < BN; ++m) {
                    const float up = __shfl_down_sync(0xffffffffu, v[m], 1);
                    if (m < M && !(lane & 1) && n + 1 < N) epi_pair(ep, m, n, v[m], up);
                }
            } else if (n < N) {
#pragma unroll
                for (int m = 0; m < BN; ++m)
                    if (m < M) {
                        if (xbm) v[m] = epi_add_xb(ep, m, n, v[m]);
                        else epi_one_k<EK>(ep, m, n, v[m]);
                    }
            }
        }
        if (xbm && final_) {
            // 8-column sums of x^2: lanes are consecutive columns
#pragma unroll
            for (int m = 0; m < BN; ++m) {
                float a = (have && n < N && m < M) ? v[m] : 0.f;
                a += __shfl_xor_sync(0xffffffffu, a, 1);
                a += __shfl_xor_sync(0xffffffffu, a, 2);
                a += __shfl_xor_sync(0xffffffffu, a, 4);
                if ((lane & 7) == 0 && n < N && m < M) ep.ssp[(n >> 3) * 16 + m] = a;
            }
        }
    }
    if (splits > 1 && cluster_reduce) {
        // Split-K reduction inside the cluster (the tile's `splits` CTAs): after the first cluster
        // barrier every partial is in its CTA's shared memory; CTA s reduces rows
        // [s * 128 / splits, (s + 1) * 128 / splits) over all CTAs in split order and applies the
        // epilogue; the second barrier keeps every CTA's shared memory alive until all reads are done.
        asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
        if (warp >= 2) {
            // item = (row of my share, group of 4 activation columns); all splits' float4s of an
            // item are requested together, then added in split order
            const int t = threadIdx.x - 64;  // 0..127
            const int rps = BM / splits;
            const bool swiglu = kind == EPI_SWIGLU;
            for (int it0 = 0; it0 < rps * 4; it0 += 128) {
                const int it = it0 + t;
                const bool mine = it < rps * 4;
                const int r = mine ? it >> 2 : 0, cg = it & 3;
                const int row = split * rps + r;
                const uint32_t laddr = smem_u32(smem) + (uint32_t)(row * BN * 4 + cg * 16);
                float4 part4[8];
#pragma unroll
                for (int s2 = 0; s2 < 8; ++s2) {
                    part4[s2] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (s2 < splits) {
                        uint32_t raddr;
                        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(laddr), "r"(s2));
                        asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                                     : "=f"(part4[s2].x), "=f"(part4[s2].y), "=f"(part4[s2].z), "=f"(part4[s2].w)
                                     : "r"(raddr)
                                     : "memory");
                    }
                }
                float v4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int s2 = 0; s2 < 8; ++s2) {
                    v4[0] += part4[s2].x;
                    v4[1] += part4[s2].y;
                    v4[2] += part4[s2].z;
                    v4[3] += part4[s2].w;
                }
                const int n = n0 + row;
                const bool ok = mine && !*abort_flag;
                if (swiglu) {
                    // (gate, up) rows 2j, 2j+1 are items four apart in the same warp
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float up = __shfl_down_sync(0xffffffffu, v4[q], 4);
                        const int m = 4 * cg + q;
                        if (ok && m < M && !(row & 1) && n + 1 < N) epi_pair(ep, m, n, v4[q], up);
                    }
                } else {
                    float x2[4] = {0.f, 0.f, 0.f, 0.f};
                    if (ok && n < N) {
                        const int h = it0 >> 7;  // 0 or 1: the prefetched residual of this item
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (4 * cg + q < M) {
                                if (xpre_on) {
                                    const float xn = (h ? xpre[1][q] : xpre[0][q]) + v4[q];
                                    ep.out_f32[(int64_t)(4 * cg + q) * ep.ldo + n] = xn;
                                    if (xbm) {
                                        reinterpret_cast<bf16*>(ep.xb)[(int64_t)(4 * cg + q) * ep.ld_xb + n] =
                                            __float2bfloat16(xn * ep.xb_g[n]);
                                        x2[q] = xn * xn;
                                    }
                                } else if (xbm) {
                                    x2[q] = epi_add_xb(ep, 4 * cg + q, n, v4[q]);
                                } else {
                                    epi_one_k<EK>(ep, 4 * cg + q, n, v4[q]);
                                }
                            }
                    }
                    if (xbm) {
                        // 8-column sums of x^2: the 8 lanes of an activation-row group hold 8 consecutive
                        // columns (lane bits 2..4); their first lane writes the group's four rows
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            x2[q] += __shfl_xor_sync(0xffffffffu, x2[q], 4);
                            x2[q] += __shfl_xor_sync(0xffffffffu, x2[q], 8);
                            x2[q] += __shfl_xor_sync(0xffffffffu, x2[q], 16);
                        }
                        if ((lane >> 2) == 0 && mine && n < N)
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                if (4 * cg + q < M) ep.ssp[(n >> 3) * 16 + 4 * cg + q] = x2[q];
                    }
                }
            }
        }
        // only the shared-memory reads above must be done before any CTA of the cluster exits
        asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) atomicOr(err, DEVERR_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

// Per device: the raised shared-memory limit is an attribute of the device's context.
constexpr int kMaxDev = 64;
bool g_ready[kMaxDev] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_enc = nullptr;

bool ready() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return false;
    if (g_ready[dev]) return true;
    if (!tc_available()) return false;
    if (!g_enc) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return false;
        g_enc = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    }
    for (auto fn : {k_tc_stream<-1, false>, k_tc_stream<EPI_STORE_F32, false>, k_tc_stream<EPI_ADD_F32, false>,
                    k_tc_stream<EPI_QKV, false>, k_tc_stream<EPI_SWIGLU, false>, k_tc_stream<-1, true>,
                    k_tc_stream<EPI_STORE_F32, true>, k_tc_stream<EPI_ADD_F32, true>, k_tc_stream<EPI_QKV, true>,
                    k_tc_stream<EPI_SWIGLU, true>})
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes()) != cudaSuccess)
            return false;
    g_ready[dev] = true;
    return true;
}

bool encode(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return g_enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tensor-core kernels' mbarrier wait on a barrier that nothing arrives at: it gives up after
// its limit, as a stalled copy or MMA would make it.
__global__ void k_mbar_selftest(int* err) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0, &abort_flag)) atomicOr(err, DEVERR_TIMEOUT);
}

}  // namespace

cudaError_t mbar_wait_selftest(int* err, cudaStream_t st) {
    if (!err) return cudaErrorInvalidValue;
    k_mbar_selftest<<<1, 32, 0, st>>>(err);
    note_launch();
    return cudaGetLastError();
}

// The instance for an epilogue kind: one per kind the step uses, so that each carries only its own
// epilogue code (it runs once per launch, from a cold instruction cache); others take the generic one.
template <bool CLU>
decltype(&k_tc_stream<-1, CLU>) stream_kernel(int kind) {
    switch (kind) {
        case EPI_STORE_F32: return k_tc_stream<EPI_STORE_F32, CLU>;
        case EPI_ADD_F32: return k_tc_stream<EPI_ADD_F32, CLU>;
        case EPI_QKV: return k_tc_stream<EPI_QKV, CLU>;
        case EPI_SWIGLU: return k_tc_stream<EPI_SWIGLU, CLU>;
        default: return k_tc_stream<-1, CLU>;
    }
}

bool tc_stream_ok(int M, int N, int K) { return ready() && M >= 1 && M <= BN && N >= 1 && K >= BK && K % 8 == 0; }

// Largest split of K; split-K partial sums are reduced inside a thread-block cluster through
// distributed shared memory where the split allows, else through scratch and tile tickets.
constexpr int kMaxSplits = 8;

int choose_splits(int nT, int nkb, int num_sms) {
    int splits = (2 * num_sms + nT - 1) / nT;
    return splits < 1 ? 1 : (splits > nkb ? nkb : (splits > kMaxSplits ? kMaxSplits : splits));
}

size_t tc_stream_scratch_floats(int N, int K, int num_sms) {
    const int nT = (N + BM - 1) / BM, nkb = (K + BK - 1) / BK;
    const int splits = choose_splits(nT, nkb, num_sms);
    return splits > 1 ? (size_t)nT * splits * BM * BN : 0;
}

cudaError_t tc_stream(const void* X, int64_t ldx, const TcWeightStream& w, int M, int N, int K, const EpiParams& ep,
                      float* part, size_t part_floats, unsigned int* tickets, size_t n_tickets, int num_sms, int* err,
                      cudaStream_t st, const StreamNorm* norm) {
    if (!w.ready || !tc_stream_ok(M, N, K) || N != w.N || K != w.K) return cudaErrorInvalidValue;
    StreamNorm sn{};
    CUtensorMap tmX;
    if (ep.ssp && (ep.kind != EPI_ADD_F32 || !ep.xb || !ep.xb_g || N % 8 != 0)) return cudaErrorInvalidValue;
    if (norm) {
        if (!norm->ssp || K % 8 != 0) return cudaErrorInvalidValue;
        sn.ssp = norm->ssp;
        sn.eps = norm->eps;
    }
    if (ldx % 8 != 0 || ((uintptr_t)X & 15) != 0) return cudaErrorInvalidValue;
    if (!encode(&tmX, X, M, K, ldx, BN)) return cudaErrorInvalidValue;
    const int nT = (N + BM - 1) / BM, nkb = (K + BK - 1) / BK;
    int splits = choose_splits(nT, nkb, num_sms);
    while (splits > 1 && ((size_t)nT * splits * BM * BN > part_floats || (size_t)nT > n_tickets)) --splits;
    const CUtensorMap& tmW = *reinterpret_cast<const CUtensorMap*>(w.tmap);
    if (part_floats != 0) {
        // cluster reduction: splits is a power of two (cluster size <= 8) and every split non-empty
        int cs = 1;
        while (cs * 2 <= choose_splits(nT, nkb, num_sms) && cs * 2 <= 8 && cs * 2 <= nkb) cs *= 2;
        if (cs > 1) {
            const int kbp = (nkb + cs - 1) / cs;
            if ((cs - 1) * kbp < nkb) {
                cudaLaunchAttribute attr[2];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = cs;
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = 1;
                attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
                attr[1].val.programmaticStreamSerializationAllowed = 1;
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3(nT * cs);
                cfg.blockDim = dim3(NTHREADS);
                cfg.dynamicSmemBytes = smem_bytes();
                cfg.stream = st;
                cfg.attrs = attr;
                cfg.numAttrs = pdl_enabled() ? 2 : 1;
                cudaError_t e = cudaLaunchKernelEx(&cfg, stream_kernel<true>(ep.kind), tmW, tmX, M, N, K, cs, kbp, 1, ep,
                                                   part, tickets, err, sn);
                note_launch();
                if (e != cudaSuccess) return e;
                return cudaGetLastError();
            }
        }
    }
    int kb_per = (nkb + splits - 1) / splits;
    splits = (nkb + kb_per - 1) / kb_per;  // no empty splits
    launch(stream_kernel<false>(ep.kind), nT * splits, NTHREADS, smem_bytes(), st, tmW, tmX, M, N, K, splits, kb_per, 0,
           ep, part, tickets, err, sn);
    note_launch();
    return cudaGetLastError();
}

cudaError_t tc_stream_prepare(TcWeightStream& w, const void* ptr, int N, int K) {
    w.ready = false;
    w.ptr = ptr;
    w.N = N;
    w.K = K;
    if (!ready()) return cudaSuccess;
    if (K % 8 != 0 || ((uintptr_t)ptr & 15) != 0) return cudaSuccess;
    if (!encode(reinterpret_cast<CUtensorMap*>(w.tmap), ptr, N, K, K, BM)) return cudaSuccess;
    w.ready = true;
    return cudaSuccess;
}

}  // namespace dspark
