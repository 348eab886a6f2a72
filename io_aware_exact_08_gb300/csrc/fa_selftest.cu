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

// Throughput of ex2.approx.f32, the instruction the softmax spends most of
// its exponentials on: every thread runs `iters` rounds of eight independent
// ex2 (the chains keep the multifunction unit's pipeline full) and writes one
// value so the work is not discarded.
__global__ void __launch_bounds__(512) ex2_probe_kernel(float* out, int iters) {
    float a[8];
#pragma unroll
    for (int x = 0; x < 8; ++x) a[x] = -1e-3f * (float)(threadIdx.x + x);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            a[x] = sm103::ex2_approx(a[x]);
            a[x] -= 1.f;  // keeps the argument in (-1, 0]
        }
    }
    out[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = a[0] + a[1] + a[2] + a[3] + a[4] + a[5] + a[6] + a[7];
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

extern "C" int fa_ex2_probe(float* out, int n_blocks, int iters, void* stream) {
    if (!out || n_blocks < 1 || iters < 1) return FA_ERR_INVALID_ARG;
    fa::ex2_probe_kernel<<<n_blocks, 512, 0, static_cast<cudaStream_t>(stream)>>>(out, iters);
    fa::note_launches(1);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
