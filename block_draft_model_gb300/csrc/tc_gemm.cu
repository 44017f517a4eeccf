// Tensor-core GEMM: not enabled yet (the SIMT kernels serve every shape).
#include "tc_gemm.cuh"

namespace dspark {

bool tc_available() { return false; }
cudaError_t tc_prepare(TcWeight& w, const void* ptr, int N, int K) {
    w.ready = false;
    w.ptr = ptr;
    w.N = N;
    w.K = K;
    return cudaSuccess;
}
void tc_release(TcWeight& w) { w.ready = false; }
bool tc_gemm_ok(int, int, int) { return false; }
cudaError_t tc_gemm(const void*, int64_t, const TcWeight&, int, int, int, const EpiParams&, int, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace dspark
