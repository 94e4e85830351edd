// tree_attn_selftest_timeout: exercise the bounded-wait error path on the GPU.
//
// Every pipelined kernel of this library waits on shared-memory mbarriers with a time limit;
// when a wait expires the kernel sets a bit in the plan's status words, leaves its pipeline
// and returns, and tree_attn_check reports TA_ERR_DEVICE_TIMEOUT.  That path only runs when
// something has gone wrong, so this entry point makes it run on purpose in the one safe way:
// a single thread waits, with a short limit, on an mbarrier that nothing ever arrives on.
// No trap, no assert, no bad address; the kernel returns normally and the context stays
// usable, which the caller can confirm by running an ordinary call afterwards.
#include <cuda_runtime.h>

#include <string>

#include "../../include/treeattn.h"
#include "plan.h"
#include "ptx.cuh"

namespace treeattn {
namespace {

__global__ void __launch_bounds__(32) timeout_selftest_kernel(int *status, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_barrier_init();
    // The barrier's phase 0 needs one arrival and gets none: the wait below always runs out.
    mbar_wait_for(b, 0, nullptr, status, limit_ns);
}

}  // namespace
}  // namespace treeattn

using namespace treeattn;

int tree_attn_selftest_timeout(const ta_plan *plan, int64_t limit_us, void *stream) {
    if (!plan) {
        set_error("plan is NULL");
        return TA_ERR_INVALID;
    }
    if (limit_us < 100 || limit_us > 1000000) {
        set_error("limit_us must lie in [100, 1000000]");
        return TA_ERR_INVALID;
    }
    if (plan->d_status == nullptr) {
        set_error("the plan was built with TA_PLAN_HOST_ONLY");
        return TA_ERR_INVALID;
    }
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != plan->device) {
        set_error("tree_attn_selftest_timeout: the plan's device is not the current device");
        return TA_ERR_INVALID;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    timeout_selftest_kernel<<<1, 32, 0, s>>>(plan->d_status + 3,
                                             static_cast<unsigned long long>(limit_us) * 1000ull);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error(std::string("selftest launch: ") + cudaGetErrorString(e));
        return TA_ERR_CUDA;
    }
    return TA_OK;
}
