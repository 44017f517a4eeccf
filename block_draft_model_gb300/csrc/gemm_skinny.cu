// Weight-streaming GEMM for a handful of activation rows (the batch-1 draft
// step, where M = gamma <= 16): every weight row is read from HBM exactly once
// with 16-byte non-allocating loads and used for all M rows at once.  The work
// is bound by HBM bandwidth, so the kernel is built for bytes in flight, not
// for tensor-core rate: each warp owns two weight rows, each lane streams
// four 16-byte vectors of each row before consuming them, and the activations
// sit in shared memory as fp32.
#include <algorithm>

#include "epilogue.cuh"

namespace dspark {

namespace {

constexpr int NT = 256;            // 8 warps
constexpr int WARPS = NT / 32;
constexpr int RPW = 2;             // weight rows per warp
constexpr int ROWS_PER_CTA = WARPS * RPW;
constexpr int SMEM_FLOATS = 8192;  // 32 KB of activations per chunk
constexpr int UNROLL = 4;

template <typename TW, typename TA, int MR>
__global__ void __launch_bounds__(NT) k_skinny(const TA* __restrict__ A, int64_t lda, const int* __restrict__ a_rows,
                                               int a_row0, const TW* __restrict__ W, int M, int N, int K,
                                               int k_per_split, EpiParams ep, float* __restrict__ ws) {
    pdl_wait();
    pdl_trigger();
    constexpr int VE = Vec16<TW>::N;         // weight elements per 16-byte vector
    constexpr int KC = SMEM_FLOATS / MR;     // activation chunk (columns)
    __shared__ __align__(16) float As[MR * KC];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * ROWS_PER_CTA + warp * RPW;
    const int ks = blockIdx.y * k_per_split;
    const int ke = min(K, ks + k_per_split);

    float acc[RPW][MR];
#pragma unroll
    for (int r = 0; r < RPW; ++r)
#pragma unroll
        for (int m = 0; m < MR; ++m) acc[r][m] = 0.f;

    const TW* wrow[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) wrow[r] = W + (int64_t)min(n0 + r, N - 1) * K;

    for (int kc0 = ks; kc0 < ke; kc0 += KC) {
        const int kcn = min(KC, ke - kc0);
        __syncthreads();
        for (int idx = threadIdx.x; idx < MR * KC; idx += NT) {
            const int m = idx / KC, kk = idx - m * KC;
            float v = 0.f;
            if (m < M && kk < kcn) {
                const int64_t row = a_rows ? a_rows[m] : (int64_t)a_row0 + m;
                v = to_f32(A[row * lda + kc0 + kk]);
            }
            As[idx] = v;
        }
        __syncthreads();
        // lane covers elements [kk, kk + VE) for kk = lane*VE + i*32*VE
        for (int kb = 0; kb < kcn; kb += 32 * VE * UNROLL) {
            uint4 wv[UNROLL][RPW];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int kk = kb + (u * 32 + lane) * VE;
#pragma unroll
                for (int r = 0; r < RPW; ++r)
                    wv[u][r] = (kk < kcn) ? ld_stream16(wrow[r] + kc0 + kk) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int kk = kb + (u * 32 + lane) * VE;
                if (kk >= kcn) break;
                float wf[RPW][VE];
#pragma unroll
                for (int r = 0; r < RPW; ++r) Vec16<TW>::unpack(wv[u][r], wf[r]);
#pragma unroll
                for (int m = 0; m < MR; ++m) {
                    const float4* ap = reinterpret_cast<const float4*>(As + m * KC + kk);
                    float a[VE];
#pragma unroll
                    for (int q = 0; q < VE / 4; ++q) {
                        float4 t = ap[q];
                        a[4 * q] = t.x;
                        a[4 * q + 1] = t.y;
                        a[4 * q + 2] = t.z;
                        a[4 * q + 3] = t.w;
                    }
#pragma unroll
                    for (int r = 0; r < RPW; ++r)
#pragma unroll
                        for (int e = 0; e < VE; ++e) acc[r][m] = fmaf(a[e], wf[r][e], acc[r][m]);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < RPW; ++r)
#pragma unroll
        for (int m = 0; m < MR; ++m) acc[r][m] = warp_sum(acc[r][m]);

    if (lane != 0) return;
    if (gridDim.y > 1) {
        // partial sums: ws[split][m][n]
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const int n = n0 + r;
            if (n >= N) continue;
#pragma unroll
            for (int m = 0; m < MR; ++m)
                if (m < M) ws[((int64_t)blockIdx.y * M + m) * N + n] = acc[r][m];
        }
        return;
    }
#pragma unroll
    for (int m = 0; m < MR; ++m) {
        if (m >= M) break;
        if (ep.kind == EPI_SWIGLU) {
            if (n0 + 1 < N) epi_pair(ep, m, n0, acc[0][m], acc[1][m]);
        } else {
#pragma unroll
            for (int r = 0; r < RPW; ++r)
                if (n0 + r < N) epi_one(ep, m, n0 + r, acc[r][m]);
        }
    }
}

// Fixed-order sum of the split-K partials, then the epilogue.  ADD_XB: the instance for the one
// row of a residual add that also hands over the next operand (only that code, which runs once
// per launch from a cold instruction cache).
template <bool ADD_XB>
__global__ void k_splitk_reduce(const float* __restrict__ ws, int splits, int M, int N, EpiParams ep) {
    pdl_wait();
    pdl_trigger();
    const int64_t total = (int64_t)M * N;
    const bool pairs = !ADD_XB && ep.kind == EPI_SWIGLU;
    const int64_t items = pairs ? total / 2 : total;
    for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < items; it += (int64_t)gridDim.x * blockDim.x) {
        if (pairs) {
            const int64_t idx = it * 2;
            const int m = (int)(idx / N), n = (int)(idx - (int64_t)m * N);
            float g = 0.f, u = 0.f;
            for (int s = 0; s < splits; ++s) {
                g += ws[(int64_t)s * total + idx];
                u += ws[(int64_t)s * total + idx + 1];
            }
            epi_pair(ep, m, n, g, u);
        } else {
            const int m = (int)(it / N), n = (int)(it - (int64_t)m * N);
            float v = 0.f;
            for (int s = 0; s < splits; ++s) v += ws[(int64_t)s * total + it];
            if (ADD_XB) {
                // EPI_ADD_F32 of one row (M = 1, N a multiple of 8) that also writes the next projection's
                // operand bf16(x * g) and the row's 8-column sums of x^2; whole 8-lane groups are active
                float* px = ep.out_f32 + n;
                const float x = *px + v;
                *px = x;
                reinterpret_cast<bf16*>(ep.xb)[n] = __float2bfloat16(x * ep.xb_g[n]);
                float s2 = x * x;
                const unsigned mask = __activemask();
                s2 += __shfl_xor_sync(mask, s2, 1, 8);
                s2 += __shfl_xor_sync(mask, s2, 2, 8);
                s2 += __shfl_xor_sync(mask, s2, 4, 8);
                if ((n & 7) == 0) ep.ssp[(n >> 3) * 16] = s2;
            } else if constexpr (!ADD_XB) {
                epi_one(ep, m, n, v);
            }
        }
    }
}

template <typename TW, typename TA, int MR>
cudaError_t launch(const void* A, int64_t lda, const int* a_rows, int a_row0, const void* W, int M, int N, int K,
                   const EpiParams& ep, float* ws, size_t ws_floats, int num_sms, cudaStream_t st) {
    const int row_ctas = (N + ROWS_PER_CTA - 1) / ROWS_PER_CTA;
    // split K until there are about four CTAs per SM, keeping >= 512 columns per split
    int splits = 1;
    const int want = 4 * num_sms;
    while (row_ctas * splits < want && K / (splits * 2) >= 512 && splits < 32) splits *= 2;
    while (splits > 1 && (size_t)splits * M * N > ws_floats) splits /= 2;
    if (ep.ssp && splits == 1) splits = 2;  // the chained operand is written by the reduce
    int kps = (K + splits - 1) / splits;
    kps = (kps + 7) / 8 * 8;
    splits = (K + kps - 1) / kps;
    dim3 grid(row_ctas, splits);
    launch(k_skinny<TW, TA, MR>, grid, NT, 0, st, (const TA*)A, lda, a_rows, a_row0, (const TW*)W, M, N, K, kps, ep, ws);
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || splits == 1) return e;
    int64_t items = (int64_t)M * N;
    int blocks = (int)std::min<int64_t>((items + 255) / 256, 8 * num_sms);
    if (ep.ssp) launch(k_splitk_reduce<true>, blocks, 256, 0, st, ws, splits, M, N, ep);
    else launch(k_splitk_reduce<false>, blocks, 256, 0, st, ws, splits, M, N, ep);
    note_launch();
    return cudaGetLastError();
}

template <typename TW, typename TA>
cudaError_t dispatch_m(const void* A, int64_t lda, const int* a_rows, int a_row0, const void* W, int M, int N, int K,
                       const EpiParams& ep, float* ws, size_t ws_floats, int num_sms, cudaStream_t st) {
    if (M <= 1) return launch<TW, TA, 1>(A, lda, a_rows, a_row0, W, M, N, K, ep, ws, ws_floats, num_sms, st);
    if (M <= 2) return launch<TW, TA, 2>(A, lda, a_rows, a_row0, W, M, N, K, ep, ws, ws_floats, num_sms, st);
    if (M <= 4) return launch<TW, TA, 4>(A, lda, a_rows, a_row0, W, M, N, K, ep, ws, ws_floats, num_sms, st);
    if (M <= 8) return launch<TW, TA, 8>(A, lda, a_rows, a_row0, W, M, N, K, ep, ws, ws_floats, num_sms, st);
    return launch<TW, TA, 16>(A, lda, a_rows, a_row0, W, M, N, K, ep, ws, ws_floats, num_sms, st);
}

}  // namespace

bool skinny_ok(int M, int K) { return M >= 1 && M <= 16 && K % 8 == 0 && K > 0; }

cudaError_t gemm_skinny(int a_dtype, const void* A, int64_t lda, const int* a_rows, int a_row0, int w_dtype,
                        const void* W, int M, int N, int K, const EpiParams& ep, float* ws, size_t ws_floats,
                        int num_sms, cudaStream_t st) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    if (!skinny_ok(M, K)) return cudaErrorInvalidValue;
    // the chained operand: one row, an added residual, whole 8-column groups, and a reduce to write it
    if (ep.ssp && (M != 1 || ep.kind != EPI_ADD_F32 || N % 8 != 0 || K < 16 || !ws || ws_floats < 2 * (size_t)N))
        return cudaErrorInvalidValue;
    if (w_dtype == DT_BF16) {
        if (a_dtype == DT_BF16)
            return dispatch_m<bf16, bf16>(A, lda, a_rows, a_row0, W, M, N, K, ep, ws, ws_floats, num_sms, st);
        return dispatch_m<bf16, float>(A, lda, a_rows, a_row0, W, M, N, K, ep, ws, ws_floats, num_sms, st);
    }
    return dispatch_m<float, float>(A, lda, a_rows, a_row0, W, M, N, K, ep, ws, ws_floats, num_sms, st);
}

}  // namespace dspark
