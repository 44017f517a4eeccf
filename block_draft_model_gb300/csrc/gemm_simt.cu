// Generic tiled SIMT GEMM: acc[m, n] = sum_k A[m, k] W[n, k] in fp32 FMA.
// Used for the fp32 drafter (which must hold 1e-4 relative accuracy, beyond
// bf16 tensor cores) and for any shape the specialised kernels do not take.
#include "epilogue.cuh"

namespace dspark {

namespace {

constexpr int BM = 64, BN = 64, BK = 32, NT = 256;

template <typename T>
__device__ __forceinline__ void load8(const T* row, int64_t k, int K, float* f) {
    // eight consecutive elements starting at k, zero beyond K
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = (k + i < K) ? to_f32(row[k + i]) : 0.f;
}

template <typename TA, typename TW>
__global__ void __launch_bounds__(NT) k_gemm_simt(const TA* __restrict__ A, int64_t lda, const int* __restrict__ a_rows,
                                                  const TW* __restrict__ W, int M, int N, int K, EpiParams ep) {
    pdl_wait();
    pdl_trigger();
    __shared__ float As[BK][BM + 4];
    __shared__ float Ws[BK][BN + 4];
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    // loader mapping: 256 threads x 8 elements = 64 rows x 32 k
    const int lr = tid >> 2, lk = (tid & 3) * 8;
    const int am = m0 + lr, wn = n0 + lr;
    const TA* arow = nullptr;
    if (am < M) arow = A + (int64_t)(a_rows ? a_rows[am] : am) * lda;
    const TW* wrow = (wn < N) ? W + (int64_t)wn * K : nullptr;

    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    for (int k0 = 0; k0 < K; k0 += BK) {
        float fa[8], fw[8];
        if (arow) load8(arow, k0 + lk, K, fa);
        else
#pragma unroll
            for (int i = 0; i < 8; ++i) fa[i] = 0.f;
        if (wrow) load8(wrow, k0 + lk, K, fw);
        else
#pragma unroll
            for (int i = 0; i < 8; ++i) fw[i] = 0.f;
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            As[lk + i][lr] = fa[i];
            Ws[lk + i][lr] = fw[i];
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < BK; ++kk) {
            float a[4], w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) w[j] = Ws[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], w[j], acc[i][j]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= M) continue;
        const int nb = n0 + tx * 4;
        if (ep.kind == EPI_SWIGLU) {
#pragma unroll
            for (int j = 0; j < 4; j += 2)
                if (nb + j + 1 < N) epi_pair(ep, m, nb + j, acc[i][j], acc[i][j + 1]);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (nb + j < N) epi_one(ep, m, nb + j, acc[i][j]);
        }
    }
}

}  // namespace

cudaError_t gemm_simt(int a_dtype, const void* A, int64_t lda, const int* a_rows, int w_dtype, const void* W, int M,
                      int N, int K, const EpiParams& ep, cudaStream_t st) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM);
    if (a_dtype == DT_F32 && w_dtype == DT_F32)
        launch(k_gemm_simt<float, float>, grid, NT, 0, st, (const float*)A, lda, a_rows, (const float*)W, M, N, K, ep);
    else if (a_dtype == DT_BF16 && w_dtype == DT_BF16)
        launch(k_gemm_simt<bf16, bf16>, grid, NT, 0, st, (const bf16*)A, lda, a_rows, (const bf16*)W, M, N, K, ep);
    else if (a_dtype == DT_F32 && w_dtype == DT_BF16)
        launch(k_gemm_simt<float, bf16>, grid, NT, 0, st, (const float*)A, lda, a_rows, (const bf16*)W, M, N, K, ep);
    else
        launch(k_gemm_simt<bf16, float>, grid, NT, 0, st, (const bf16*)A, lda, a_rows, (const float*)W, M, N, K, ep);
    note_launch();
    return cudaGetLastError();
}

}  // namespace dspark
