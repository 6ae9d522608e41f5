// ct_selftest.cu -- a kernel whose bounded wait is made to run out, so that
// the timeout path every pipelined kernel shares (bounded mbarrier wait ->
// device status word -> ct_last_device_error) can be exercised without a
// fault or a hang.  Not part of any forward computation.
#include "ct_internal.h"
#include "ct_tma.h"

namespace ct {
namespace {

// One thread initialises an mbarrier that expects one arrival, never arrives,
// and waits for it with the given limit; the wait gives up, the status word
// records the timeout, and the kernel returns normally.
__global__ void wait_timeout_kernel(uint64_t limit_ns, unsigned int *status)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    dev::mbar_init(&bar, 1);
    dev::fence_mbar_init();
    if (!dev::mbar_wait_bounded(&bar, 0, limit_ns)) atomicExch(status, (unsigned)CT_ERR_DEVICE_TIMEOUT);
}

}  // namespace
}  // namespace ct

extern "C" ct_status ct_selftest_wait_timeout(uint64_t limit_ns, void *stream)
{
    if (limit_ns == 0 || limit_ns > 1000000000ull) return CT_ERR_ARG;
    unsigned int *status = ct::device_status_ptr();
    if (!status) return CT_ERR_CUDA;
    ct::wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(limit_ns, status);
    return cudaGetLastError() == cudaSuccess ? CT_OK : CT_ERR_CUDA;
}
