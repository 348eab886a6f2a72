// fa_bwd_noalloc: the backward pass for callers that cannot allocate device
// memory themselves.
//
// fa_bwd needs a workspace (the per-row statistics -LSE and rowsum(dO o O)
// and the fp32 dQ accumulator). Some callers have no way to provide one: a host framework
// whose caching allocator has already reserved the device's memory, a
// latency-bound serving path where cudaMalloc (which can synchronise the
// device and take unbounded time) is not allowed, or a plugin that is handed
// only its inputs and outputs. For them, this entry point takes its
// workspace from a fixed array in device memory that is part of the loaded
// library, so nothing is allocated per call.
//
// Costs and rules of that array:
//  - Its size is FA_BWD_NOALLOC_SCRATCH_BYTES. Every GPU on which the library
//    is loaded keeps that much memory reserved until the process exits.
//  - Problems whose workspace (fa_bwd_workspace_size) exceeds it are refused
//    with FA_ERR_WORKSPACE before anything is launched.
//  - All calls share the one array. The backward kernels zero the dQ
//    accumulator and overwrite the row sums at the start of every call, so
//    leftovers from an earlier call do not matter; but two calls whose
//    kernels can run at the same time on the GPU (different streams without
//    ordering between them) race on the array and give wrong results.
//  - The array's address on a device is looked up once, on that device's
//    first call, with that device current. That first call should happen
//    before any stream capture begins.
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/fa.h"

namespace {

constexpr int kMaxDevices = 64;

// The workspace shared by every fa_bwd_noalloc call on a device. In host
// code this name is only a handle: its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_BWD_NOALLOC_SCRATCH_BYTES];

std::mutex g_lock;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up once
// per device), or nullptr on failure.
void* scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> guard(g_lock);
    if (!g_scratch_addr[dev]) {
        void* ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) {
            if (std::getenv("FA_DEBUG"))
                std::fprintf(stderr, "fa_bwd_noalloc: cudaGetSymbolAddress failed: %s\n", cudaGetErrorString(e));
            return nullptr;
        }
        g_scratch_addr[dev] = ptr;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                              const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                              int causal, const uint8_t* block_mask, float dropout_p, uint64_t seed, fa_dtype dtype,
                              const int32_t* kv_len, void* stream) {
    const size_t need = fa_bwd_workspace_size(B, H, N, d);
    if (need > (size_t)FA_BWD_NOALLOC_SCRATCH_BYTES) {
        if (std::getenv("FA_DEBUG"))
            std::fprintf(stderr, "fa_bwd_noalloc: needs %zu bytes of workspace, the fixed array holds %zu\n", need,
                         (size_t)FA_BWD_NOALLOC_SCRATCH_BYTES);
        return FA_ERR_WORKSPACE;
    }
    void* scratch = nullptr;
    if (need > 0 && N > 0) {
        scratch = scratch_address();
        if (!scratch) return FA_ERR_CUDA;
    }
    return fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, block_mask, dropout_p, seed, dtype,
                  kv_len, scratch, (size_t)FA_BWD_NOALLOC_SCRATCH_BYTES, stream);
}
