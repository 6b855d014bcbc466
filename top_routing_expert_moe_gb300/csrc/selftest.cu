// selftest.cu -- exercises the bounded-wait failure path on the device.
//
// Every mbarrier wait in the TMA-fed kernels gives up after a time limit,
// records MOE_ERR_TIMEOUT in the device status word and lets the kernel
// return, so a lost arrival cannot hang the GPU.  This kernel waits, with the
// same wait routine and a caller-chosen limit, on a barrier that nothing ever
// arrives on: the wait must run out, record the status and return.
#include "common.cuh"
#include "kernels.h"
#include "tma.cuh"

namespace moe {
namespace {

__global__ void selftest_wait_kernel(int* status, unsigned long long limit_ns) {
    pdl_wait();
    pdl_trigger();
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);   // expects one arrival, which never comes
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0)
        (void)mbar_wait(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
}

}  // namespace
}  // namespace moe

extern "C" int moe_selftest_bounded_wait(unsigned long long limit_ns, moe_stream_t stream) {
    using namespace moe;
    if (limit_ns == 0 || limit_ns > 1000000000ull) return MOE_ERR_INVALID_ARG;
    MOE_LAUNCH(selftest_wait_kernel, 1, 32, 0, (cudaStream_t)stream, device_status_ptr(), limit_ns);
    return MOE_OK;
}
