// A weight-streaming linear call that allocates no device memory.
//
// Some callers cannot call cudaMalloc: code running inside another runtime's
// memory pool, allocator-free serving loops, or a context whose allocations
// are frozen after start-up.  dspark_linear_stream_noalloc serves them: it
// runs the same weight-streaming tensor-core kernel as dspark_linear
// (kernel 4), but the kernel's split-K scratch (partial sums, per-tile
// tickets and the error word) lives in file-scope __device__ arrays of this
// library, which every GPU that loads the library holds until the process
// exits.
//
// In host code the arrays' names are host-side stand-ins, not device
// addresses; the device addresses come from cudaGetSymbolAddress, once per
// device, with that device current, on the first call made on it.  That
// first call should therefore come before any stream capture.  All calls share
// the arrays: the tickets are cleared on every call, and two calls whose work
// overlaps on the GPU race on the scratch.  A kernel that gives up on a bounded
// wait records DSPARK_DEVERR_TIMEOUT in the shared error word, which
// dspark_noalloc_check reads and clears.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/dspark.h"
#include "kernels.cuh"
#include "tc_gemm.cuh"

namespace {

constexpr size_t kPartFloats = DSPARK_NOALLOC_SCRATCH_FLOATS;  // split-K partial sums (16 MB)
constexpr size_t kTickets = DSPARK_NOALLOC_MAX_TILES;          // one counter per 128-row weight tile

static __device__ __align__(256) float g_part[kPartFloats];
static __device__ __align__(256) unsigned int g_tickets[kTickets];
static __device__ __align__(256) int g_err;

struct DevicePtrs {
    float* part = nullptr;
    unsigned int* tickets = nullptr;
    int* err = nullptr;
    int num_sms = 0;
    bool ready = false;
};

constexpr int kMaxDevices = 64;
DevicePtrs g_dev[kMaxDevices];
std::mutex g_mu;

thread_local const char* g_msg = "no error";

dspark_status setup(int dev, DevicePtrs** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    DevicePtrs& p = g_dev[dev];
    if (!p.ready) {
        if (cudaGetSymbolAddress((void**)&p.part, g_part) != cudaSuccess ||
            cudaGetSymbolAddress((void**)&p.tickets, g_tickets) != cudaSuccess ||
            cudaGetSymbolAddress((void**)&p.err, g_err) != cudaSuccess ||
            cudaDeviceGetAttribute(&p.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            g_msg = "cudaGetSymbolAddress failed for the scratch arrays";
            return DSPARK_ERR_CUDA;
        }
        p.ready = true;
    }
    *out = &p;
    return DSPARK_OK;
}

}  // namespace

extern "C" {

dspark_status dspark_linear_stream_noalloc(const void* A_dev, int64_t lda, const void* W_dev, int32_t M, int32_t N,
                                           int32_t K, float* out_dev, int64_t ldo, void* stream) {
    using namespace dspark;
    if (!A_dev || !W_dev || !out_dev) {
        g_msg = "a pointer is NULL";
        return DSPARK_ERR_INVALID_ARG;
    }
    if (M < 1 || M > 16 || N < 1 || K < 64 || K % 8 != 0 || lda < K || lda % 8 != 0 || ldo < N) {
        g_msg = "shape outside 1 <= M <= 16, K >= 64, K % 8 == 0, lda % 8 == 0, ldo >= N";
        return DSPARK_ERR_INVALID_ARG;
    }
    if (((uintptr_t)A_dev & 15) || ((uintptr_t)W_dev & 15)) {
        g_msg = "A and W must be 16-byte aligned";
        return DSPARK_ERR_INVALID_ARG;
    }
    const size_t tiles = (size_t)(N + 127) / 128;
    if (tiles > kTickets) {
        g_msg = "N exceeds the static scratch (DSPARK_NOALLOC_MAX_TILES * 128 rows)";
        return DSPARK_ERR_CAPACITY;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        g_msg = "no current CUDA device";
        return DSPARK_ERR_CUDA;
    }
    DevicePtrs* p = nullptr;
    dspark_status s = setup(dev, &p);
    if (s != DSPARK_OK) return s;
    if (!tc_stream_ok(M, N, K)) {
        g_msg = "the weight-streaming tensor-core kernel is not available on this device";
        return DSPARK_ERR_UNSUPPORTED;
    }
    TcWeightStream w;
    if (tc_stream_prepare(w, W_dev, N, K) != cudaSuccess || !w.ready) {
        g_msg = "tensor map for W rejected";
        return DSPARK_ERR_UNSUPPORTED;
    }
    cudaStream_t st = (cudaStream_t)stream;
    // tickets must start at zero; a call that gave up on a bounded wait could have left them armed
    if (cudaMemsetAsync(p->tickets, 0, tiles * sizeof(unsigned int), st) != cudaSuccess) {
        g_msg = "clearing the tickets failed";
        return DSPARK_ERR_CUDA;
    }
    EpiParams ep;
    ep.kind = EPI_STORE_F32;
    ep.out_f32 = out_dev;
    ep.ldo = ldo;
    // tc_stream reduces its split of K until the partial sums fit kPartFloats
    if (tc_stream(A_dev, lda, w, M, N, K, ep, p->part, kPartFloats, p->tickets, kTickets, p->num_sms, p->err, st) !=
        cudaSuccess) {
        g_msg = "kernel launch failed";
        return DSPARK_ERR_CUDA;
    }
    return DSPARK_OK;
}

dspark_status dspark_noalloc_check(int32_t* word_host) {
    if (!word_host) {
        g_msg = "word_host is NULL";
        return DSPARK_ERR_INVALID_ARG;
    }
    *word_host = 0;
    // the symbol copies go through the current device's copy of g_err and allocate nothing;
    // they wait for the device's earlier work, so every call before this one is covered
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_err, sizeof(int)) != cudaSuccess) {
        g_msg = "reading the error word failed";
        return DSPARK_ERR_CUDA;
    }
    *word_host = v;
    if (v == 0) return DSPARK_OK;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_err, &zero, sizeof(int)) != cudaSuccess) {
        g_msg = "clearing the error word failed";
        return DSPARK_ERR_CUDA;
    }
    g_msg = "a bounded device wait gave up (DSPARK_DEVERR_TIMEOUT); the output of that call is incomplete";
    return DSPARK_ERR_DEVICE;
}

const char* dspark_noalloc_last_error(void) { return g_msg; }

}  // extern "C"
