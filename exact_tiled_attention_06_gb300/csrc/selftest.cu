// selftest.cu -- failure detection without a fault: one block whose barrier wait is
// never satisfied. Every pipeline wait in the library is bounded (mbar_wait gives up after
// kWaitLimitCycles, about 2 s at 2 GHz, and records a timeout in the device error word);
// this entry point lets a test make such a wait run out and check that the host reads the
// status and that the context stays usable afterwards.
#include "internal.h"
#include "ptx.cuh"

#define ATTN_API extern "C" __attribute__((visibility("default")))

namespace attn {
namespace {

__global__ void __launch_bounds__(64) attn_selftest_wait(unsigned* err)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ volatile int abort_flag;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);  // one arrival would complete phase 0; none ever comes
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // Warp 0 waits on the barrier until its time limit; warp 1 waits too and leaves when
    // warp 0's timeout raises the block's abort flag.
    mbar_wait(b, 0, &abort_flag, err);
}

}  // namespace
}  // namespace attn

using namespace attn;

ATTN_API int attn_selftest_wait_timeout(void* stream)
{
    int dev = 0;
    int rc = check_device(&dev);
    if (rc != kOk) return rc;
    unsigned* err = device_error_word();
    if (!err) return kErrCuda;
    attn_selftest_wait<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(err);
    return cudaGetLastError() == cudaSuccess ? kOk : kErrLaunch;
}
