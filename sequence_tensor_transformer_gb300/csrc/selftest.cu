// Failure-detection self-test: runs the library's bounded waits against a
// flag that nothing sets and an mbarrier that never completes, so that the
// timeout path (status word, early exit) is exercised without hanging the GPU.
#include "sptp_ptx.cuh"

namespace sptp {

namespace {

__global__ void wait_selftest_kernel(DeviceStatus* st, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // one arrival expected; none is ever made
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        WaitCtx w{st, &abort_flag, limit_ns};
        const bool flag_ok = flag_wait_geq(&st->flag, 1, w, kWhereSelftestFlag, 0);
        // a fresh context so the second wait runs its own limit
        int local_abort = 0;
        WaitCtx w2{st, &local_abort, limit_ns};
        const bool bar_ok = mbar_wait(&bar, 0, w2, kWhereSelftestBarrier, flag_ok ? 1 : 0);
        (void)bar_ok;
    }
    __syncthreads();
}

}  // namespace

cudaError_t launch_wait_selftest(DeviceStatus* st, unsigned long long limit_ns, cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(st, limit_ns);
    return cudaGetLastError();
}

}  // namespace sptp
