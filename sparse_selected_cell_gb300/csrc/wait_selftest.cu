// wait_selftest.cu -- a check of the bounded-wait machinery every pipelined
// kernel of this library relies on (tc::mbar_wait): one warp waits on an
// mbarrier that nothing arrives on, gives up after `limit_ns`, and records
// QSA_DEV_WAIT_TIMEOUT in *dev_status the way the attention kernels do.  It
// faults nothing and cannot hang: the wait ends by wall time.
#include "qsa_common.cuh"
#include "tc_ptx.cuh"

namespace qsa {
namespace {

__global__ void __launch_bounds__(32) wait_selftest_kernel(uint64_t limit_ns, int32_t* dev_status) {
    __shared__ __align__(8) uint64_t bar_mem;
    __shared__ int abort_flag;
    const uint32_t bar = smem_u32(&bar_mem);
    if (threadIdx.x == 0) {
        tc::mbar_init(bar, 1);   // one arrival expected; none ever comes
        abort_flag = 0;
        tc::fence_mbar_init();
    }
    __syncwarp();
    if (!tc::mbar_wait(bar, 0, reinterpret_cast<volatile int*>(&abort_flag), limit_ns) && threadIdx.x == 0)
        report(dev_status, QSA_DEV_WAIT_TIMEOUT);
}

}  // namespace
}  // namespace qsa

extern "C" int qsa_wait_selftest(int32_t limit_us, int32_t* dev_status, void* stream) {
    if (limit_us <= 0 || limit_us > 10000000 || !dev_status) return QSA_ERR_ARG;
    qsa::wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((uint64_t)limit_us * 1000u,
                                                                               dev_status);
    return cudaGetLastError() == cudaSuccess ? QSA_OK : QSA_ERR_CUDA;
}
