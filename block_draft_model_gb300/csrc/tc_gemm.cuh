// Tensor-core GEMM (tcgen05 + TMA + TMEM) for bf16 operands:
// acc[m, n] = sum_k A[m, k] W[n, k], fp32 accumulation, GEMM epilogues of epilogue.cuh.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.cuh"

namespace dspark {

// A weight matrix W [N, K] (bf16, K contiguous) with its TMA descriptor.
struct TcWeight {
    bool ready = false;
    bool ready128 = false;  // tmap128 (128-row boxes, the wide form's weight side) is valid
    const void* ptr = nullptr;
    int N = 0, K = 0;
    alignas(64) unsigned char tmap[128];
    alignas(64) unsigned char tmap128[128];
};

bool tc_available();
// Tensor map (128 bytes at `map`, host memory) over a bf16 weight [rows, K] whose
// one box is a 16-row x 512-column slice laid out as 8 column blocks of
// [16 rows][64] with the 128-byte swizzle: a 3-D map (one copy per slice) or,
// with three_d false, a 2-D map with [16][64] boxes (eight copies per slice).
bool tc_encode_slot_map(void* map, const void* W, int64_t rows, int64_t K, bool three_d);
cudaError_t tc_prepare(TcWeight& w, const void* ptr, int N, int K);
void tc_release(TcWeight& w);
bool tc_gemm_ok(int M, int N, int K);
// `groups` problems of one shape in one launch: acc_g = A_g . W_g^T.  Both sides are
// 3-D views (bf16 rows of K, group g at ptr + g * group_stride elements) made by
// tc_prepare_grouped (a_side: 128-row boxes of A, else 256-row boxes of W); the
// EPI_KV_CACHE epilogue of group g writes at ep.cache + g * ep.group_stride.
bool tc_prepare_grouped(TcWeight& w, const void* ptr, int groups, int64_t group_stride, int rows, int K, bool a_side);
// a_shared: A is one 2-D matrix (a made by tc_prepare, its 128-row boxes) read by every group.
cudaError_t tc_gemm_grouped(const TcWeight& a, const TcWeight& w, int groups, int M, int N, int K, const EpiParams& ep,
                            int num_sms, int* err, cudaStream_t st, bool a_shared = false);
// A: [M, K] bf16 with row stride lda (16-byte aligned).  A bounded device wait
// that gives up sets bit 16 of *err (the handle's device error word).
// ksplit > 1 (EPI_STORE_F32 only) cuts K into ksplit ranges, each a separate
// work unit: range s stores its partial product at rows s * ep.split_rows + m
// of ep.out_f32, and the consumer sums the ranges.
cudaError_t tc_gemm(const void* A, int64_t lda, const TcWeight& w, int M, int N, int K, const EpiParams& ep,
                    int num_sms, int* err, cudaStream_t st, int ksplit = 1);
// The wide form on its own: the weights are the MMA's 128-row side and all M <= 320 rows of A
// its N side (EPI_STORE_F32; every weight tile read once).
bool tc_wide_ok(const TcWeight& w, int M, int N, int K, const EpiParams& ep);
// The shapes where the wide form beats the 128 x 256 tiles: M <= 160 or 257..320, and at
// least one 128-row weight tile per SM.
bool tc_wide_preferred(int M, int N, int num_sms);
cudaError_t tc_gemm_wide(const void* A, int64_t lda, const TcWeight& w, int M, int N, int K, const EpiParams& ep,
                         int num_sms, int* err, cudaStream_t st);

// Weight-streaming variant for M <= 16 activation rows (tc_stream.cu): the
// weights are the MMA's 128-row side.  `part`/`tickets` are scratch for the
// split-K partials (tc_stream_scratch_floats floats; one zeroed counter per
// 128-row tile, left zeroed after every launch).
struct TcWeightStream {
    bool ready = false;
    const void* ptr = nullptr;
    int N = 0, K = 0;
    alignas(64) unsigned char tmap[128];
};
bool tc_stream_ok(int M, int N, int K);
size_t tc_stream_scratch_floats(int N, int K, int num_sms);
cudaError_t tc_stream_prepare(TcWeightStream& w, const void* ptr, int N, int K);
// Row scales of tc_stream: X is bf16(x * g) already, and the accumulator row m is scaled by
// 1 / sqrt(mean_k(x[m][k]^2) + eps) from the 8-column sums of x^2 written by the epilogue that
// produced x: the product with RMSNorm(x) * g without a separate normalisation kernel.
struct StreamNorm {
    const float* ssp = nullptr;  // ssp[(k / 8) * 16 + m] = sum of x[m]^2 over columns [k, k + 8)
    float eps = 0.f;
};
cudaError_t tc_stream(const void* X, int64_t ldx, const TcWeightStream& w, int M, int N, int K, const EpiParams& ep,
                      float* part, size_t part_floats, unsigned int* tickets, size_t n_tickets, int num_sms, int* err,
                      cudaStream_t st, const StreamNorm* norm = nullptr);

}  // namespace dspark
