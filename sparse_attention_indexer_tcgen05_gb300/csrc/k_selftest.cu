// k_selftest.cu -- a bounded wait that runs out, so that the device-side timeout reporting of the tensor-core
// kernels can be exercised without making any GPU fault or hang.
//
// One warp initialises an mbarrier that nothing ever arrives on and waits on it with wait_bar_for, the bounded
// wait every tensor-core kernel uses, with a limit of about 1 ms instead of about 2 s.  The wait runs out, records
// its site code in this file's device error word and returns; the kernel then ends with no copy or MMA in flight.
// csa_check_device_status reads the word (CSA_ERR_TIMEOUT) and clears it.
#include "csa_tc.cuh"
#include "tc_ptx.cuh"

namespace csa {

static __device__ int g_selftest_error = 0;

cudaError_t selftest_read_clear_error(int *flag)
{
    cudaError_t e = cudaMemcpyFromSymbol(flag, g_selftest_error, sizeof(int));
    if (e != cudaSuccess || *flag == 0) return e;
    int zero = 0;
    return cudaMemcpyToSymbol(g_selftest_error, &zero, sizeof(int));
}

__global__ void bounded_wait_selftest_kernel(long long limit_cycles)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) ptx::wait_bar_for(&bar, 0, &abort_flag, &g_selftest_error, 90, limit_cycles);
    __syncthreads();
}

cudaError_t launch_bounded_wait_selftest(cudaStream_t st)
{
    bounded_wait_selftest_kernel<<<1, 32, 0, st>>>(2000000LL);  // about 1 ms at 2 GHz
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace csa
