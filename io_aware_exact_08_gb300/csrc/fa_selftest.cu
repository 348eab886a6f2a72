// Self-test of the device failure path: a kernel waits, with the same
// bounded mbarrier wait the tensor-core kernels use, on a barrier that
// nothing arrives at. The wait gives up after `limit_ns`, records
// FA_ERR_DEVICE_TIMEOUT and a site id in the device status word and the
// kernel returns normally, so the context stays usable. Nothing faults,
// traps or hangs.
#include <cstdint>

#include "fa_internal.h"
#include "fa_sm103.cuh"

namespace fa {
namespace {

constexpr int kSelfTestSite = 900;

__global__ void wait_timeout_kernel(int* status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        sm103::mbar_init(&bar, 1);
        abort_flag = 0;
        sm103::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        sm103::WaitCtx w{&abort_flag, status, limit_ns};
        sm103::mbar_wait(&bar, 0, w, kSelfTestSite);  // no arrival ever comes
    }
}

}  // namespace
}  // namespace fa

extern "C" int fa_test_wait_timeout(uint64_t limit_ns, void* stream) {
    int* status = nullptr;
    if (fa::status_address(&status) != FA_OK) return FA_ERR_CUDA;
    fa::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, limit_ns);
    fa::note_launches(1);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
