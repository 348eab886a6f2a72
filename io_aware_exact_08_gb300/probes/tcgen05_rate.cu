// Throughput probe for tcgen05.mma kind::f16 (bf16 in, fp32 accumulate) on
// one GPU: one CTA per SM, one thread issuing M = 128 MMAs back to back over
// zero-filled shared-memory operands (K = 128 per group of 8 instructions),
// with a commit and a bounded wait every 16 groups. It measures the rates the
// attention kernels are designed around:
//   - N = 64 / 128 / 256, A from shared memory or from TMEM;
//   - B operand K-major or MN-major;
//   - two accumulators alternated per group, issued as straight-line code
//     and through a branch on the group index.
// Build and run (any CUDA 13 toolkit, on a GB300):
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 \
//        io_aware_exact_08_gb300/probes/tcgen05_rate.cu -o /tmp/tcgen05_rate && /tmp/tcgen05_rate
#include <cstdint>
#include <cstdio>

#include <cuda_runtime.h>

#include "../csrc/fa_sm103.cuh"

using namespace fa::sm103;

enum Pattern { kUniformSS = 0, kUniformTS = 1, kAltStraight = 2, kAltBranch = 3 };

template <int N, int BMN, int PATTERN>
__global__ void __launch_bounds__(128, 1) probe(int iters, int* status) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar;
    __shared__ uint32_t taddr;
    __shared__ int abort_flag;
    // A: 128 x 128 bf16 (32 KB); B: up to 256 x 128 bf16 (64 KB)
    for (int i = threadIdx.x; i < (32768 + 65536) / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (threadIdx.x < 32) {
        tmem_alloc(&taddr, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t t = taddr;
    WaitCtx w{&abort_flag, status};
    if (threadIdx.x == 0) {
        const uint32_t a = smem_u32(smem), b = a + 32768;
        constexpr uint32_t id = idesc_bf16_f32(128, N, 0, BMN);
        const uint64_t ad = smem_desc_sw128(a, 16, 1024);
        const uint64_t bd = BMN ? smem_desc_sw128(b, N * 128, 1024) : smem_desc_sw128(b, 16, 1024);
        for (int it = 0; it < iters; ++it) {
            const bool odd = PATTERN == kAltBranch ? (it & 1) : false;
#pragma unroll
            for (int g = 0; g < (PATTERN == kAltStraight ? 2 : 1); ++g) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t ao = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;
                    const uint32_t bo = BMN ? (kk * 2048) >> 4 : ((kk / 4) * (N * 128) + (kk % 4) * 32) >> 4;
                    if (PATTERN == kUniformTS)
                        mma_ts(t, t + 256 + kk * 8, bd + bo, id, kk > 0);
                    else if (PATTERN == kAltStraight)
                        mma_ss(t + 128 * g, ad + ao, bd + bo, id, kk > 0);
                    else if (PATTERN == kAltBranch && odd)
                        mma_ss(t + 128, ad + ao, bd + bo, id, kk > 0);
                    else
                        mma_ss(t, ad + ao, bd + bo, id, kk > 0);
                }
            }
            if ((it & 15) == 15) {
                mma_commit(&bar);
                mbar_wait(&bar, (it >> 4) & 1, w, 1);
            }
        }
        mma_commit(&bar);
        mbar_wait(&bar, (iters >> 4) & 1, w, 2);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x < 32) tmem_dealloc(t, 512);
}

template <int N, int BMN, int PATTERN>
void run(const char* name, int sms, int* status) {
    const int smem = 1024 + 32768 + 65536;
    cudaFuncSetAttribute(probe<N, BMN, PATTERN>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    probe<N, BMN, PATTERN><<<sms, 128, smem>>>(16, status);
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    const int iters = 4096;
    cudaEventRecord(e0);
    probe<N, BMN, PATTERN><<<sms, 128, smem>>>(iters, status);
    cudaEventRecord(e1);
    cudaEventSynchronize(e1);
    float ms = 0.f;
    cudaEventElapsedTime(&ms, e0, e1);
    const double groups = (double)iters * (PATTERN == kAltStraight ? 2 : 1);
    const double flop = 2.0 * 128 * N * 128 * groups * sms;
    int st = 0;
    cudaMemcpy(&st, status, sizeof(int), cudaMemcpyDeviceToHost);
    std::printf("%-44s %8.1f TFLOP/s  (status %d, %s)\n", name, flop / ms / 1e9, st,
                cudaGetErrorString(cudaGetLastError()));
}

int main() {
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    int* status = nullptr;
    cudaMalloc(&status, 2 * sizeof(int));
    cudaMemset(status, 0, 2 * sizeof(int));
    std::printf("SMs: %d\n", sms);
    run<128, 0, kUniformSS>("SS N=128, B K-major", sms, status);
    run<256, 0, kUniformSS>("SS N=256, B K-major", sms, status);
    run<64, 0, kUniformSS>("SS N=64, B K-major", sms, status);
    run<128, 1, kUniformSS>("SS N=128, B MN-major", sms, status);
    run<128, 1, kUniformTS>("TS N=128 (A from TMEM), B MN-major", sms, status);
    run<64, 1, kUniformTS>("TS N=64 (A from TMEM), B MN-major", sms, status);
    run<128, 0, kAltStraight>("SS N=128, 2 accumulators, straight-line", sms, status);
    run<128, 0, kAltBranch>("SS N=128, 2 accumulators, branch per group", sms, status);
    cudaFree(status);
    return 0;
}
