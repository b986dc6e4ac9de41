// selftest.cu -- exercises the failure path the GEMMs rely on, without a
// fault: one CTA waits, with the same bounded mbarrier wait the GEMM roles
// use, on a barrier that nothing ever arrives on.  After the limit the wait
// gives up, raises the CTA's abort flag and sets the timeout bit of the
// handle's device status word; the kernel then returns normally.  A second
// self-test fails one index check, which a debug build (-DLMOE_DEBUG) reports.
#include "kernels.h"
#include "ptx.cuh"

namespace lmoe {

namespace {

__global__ void bounded_wait_kernel(unsigned *err, uint64_t limit_ns, int *gave_up) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);   // expects one arrival; none will come
        abort_flag = 0u;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const bool ok = mbar_wait(smem_u32(&bar), 0u, &abort_flag, err, limit_ns);
        if (gave_up) *gave_up = ok ? 0 : 1;
    }
}

// One index check that fails (1 is not below 1); no memory is accessed.
__global__ void index_check_kernel() { idx_ok(1, 1); }

}  // namespace

cudaError_t launch_index_check_selftest(cudaStream_t st) {
    index_check_kernel<<<1, 1, 0, st>>>();
    return cudaGetLastError();
}

cudaError_t launch_bounded_wait_selftest(unsigned *err, uint64_t limit_ns, int *gave_up, cudaStream_t st) {
    bounded_wait_kernel<<<1, 32, 0, st>>>(err, limit_ns, gave_up);
    return cudaGetLastError();
}

LMOE_DEBUG_WORD_READER(debug_word_selftest)

}  // namespace lmoe
