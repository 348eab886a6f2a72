// C entry points of the attention library: argument validation, workspace
// layout, kernel selection and the device status word. See include/fa.h for
// the contract of each call.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>

#include "fa_internal.h"

namespace fa {
namespace {

// Device status word: kernels whose bounded waits run out write
// FA_ERR_DEVICE_TIMEOUT (and the id of the wait) here instead of trapping.
__device__ int g_status[2];

int g_kernel_path = 0;  // 0 = default, 1 = CUDA-core kernels only
std::atomic<uint64_t> g_launches{0};
// fa_set_main_kernel_events: events recorded around the next calls' main
// kernels (null = off)
cudaEvent_t g_main_start = nullptr, g_main_stop = nullptr;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Backward workspace for the per-row statistics: kColTableFloats floats per
// (b*h, 128-row query tile), which also holds the plain [B,H,N] row sums.
size_t stats_bytes(int B, int H, int N) {
    return (size_t)B * H * ((N + kMaskBlock - 1) / kMaskBlock) * kColTableFloats * sizeof(float);
}

uint32_t keep_threshold(float p) {
    const double t = std::floor((double)p * 4294967296.0);
    if (t <= 0.0) return 0u;
    if (t >= 4294967295.0) return 0xffffffffu;
    return (uint32_t)t;
}

int check_common(int B, int H, int N, int d, float scale, float dropout_p, fa_dtype dtype) {
    if (B < 1 || H < 1 || N < 0) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (!(dropout_p >= 0.f && dropout_p < 1.f)) return FA_ERR_INVALID_ARG;
    if (dtype != FA_BF16 && dtype != FA_FP32 && dtype != FA_FP16) return FA_ERR_UNSUPPORTED;
    if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
    if ((long long)B * H > 65535) return FA_ERR_UNSUPPORTED;
    if (N > (1 << 24)) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

void fill_common(Problem& p, int B, int H, int N, int d, float scale, int causal, const uint8_t* block_mask,
                 float dropout_p, uint64_t seed, fa_dtype dtype, const int32_t* kv_len, void* stream) {
    p.B = B;
    p.H = H;
    p.N = N;
    p.d = d;
    p.scale = scale;
    p.causal = causal ? 1 : 0;
    p.block_mask = block_mask;
    p.nb = (N + kMaskBlock - 1) / kMaskBlock;
    p.dropout_p = dropout_p;
    p.drop_threshold = keep_threshold(dropout_p);
    p.seed = seed;
    p.dtype = dtype;
    p.kv_len = kv_len;
    p.stream = static_cast<cudaStream_t>(stream);
}

int from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return FA_OK;
    if (std::getenv("FA_DEBUG")) std::fprintf(stderr, "fa: CUDA error %s\n", cudaGetErrorString(e));
    return FA_ERR_CUDA;
}

// Which kernels serve a problem. 16-bit inputs run on the tensor-core
// kernels and fp32 on the CUDA-core kernels (or every dtype, when the caller
// forced them with fa_set_kernel_path(1)). A 16-bit problem the tensor-core
// kernels do not take is refused with FA_ERR_UNSUPPORTED rather than sent to
// the far slower CUDA-core kernels behind the caller's back: scale <= 0
// (their online softmax takes the running maximum of the unscaled scores), or
// a block mask with more key tiles per row (query tiles per column in the
// backward) than their shared-memory tile lists hold.
int pick_path(const Problem& p, bool backward, bool* tensor_cores) {
    *tensor_cores = false;
    if (g_kernel_path != 0 || (p.dtype != FA_BF16 && p.dtype != FA_FP16)) return FA_OK;
    if (!(p.scale > 0.f)) return FA_ERR_UNSUPPORTED;
    if (p.block_mask) {
        const int tiles = (p.N + kMaskBlock - 1) / kMaskBlock;
        const int cap = !backward ? kMaskListCap
                        : p.d == 64 ? kMaskListCap
                        : p.d == 128 ? kMaskListCapBwd128 : kMaskListCapBwd256;
        if (tiles > cap) return FA_ERR_UNSUPPORTED;
    }
    *tensor_cores = true;
    return FA_OK;
}

}  // namespace

void note_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

void record_main_start(cudaStream_t s) {
    if (g_main_start) cudaEventRecord(g_main_start, s);
}

void record_main_stop(cudaStream_t s) {
    if (g_main_stop) cudaEventRecord(g_main_stop, s);
}

int status_address(int** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    static int* cached[64] = {nullptr};
    if (dev < 0 || dev >= 64) return FA_ERR_CUDA;
    if (!cached[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_status) != cudaSuccess) return FA_ERR_CUDA;
        cached[dev] = static_cast<int*>(ptr);
    }
    *out = cached[dev];
    return FA_OK;
}



}  // namespace fa

using namespace fa;

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
           float scale, int causal, const uint8_t* block_mask, float dropout_p, uint64_t seed, fa_dtype dtype,
           const int32_t* kv_len, void* stream) {
    int rc = check_common(B, H, N, d, scale, dropout_p, dtype);
    if (rc != FA_OK) return rc;
    if (N == 0) return FA_OK;
    if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
        return FA_ERR_INVALID_ARG;
    Problem p{};
    fill_common(p, B, H, N, d, scale, causal, block_mask, dropout_p, seed, dtype, kv_len, stream);
    p.q = q;
    p.k = k;
    p.v = v;
    p.o = o;
    p.lse = lse;
    bool tc = false;
    rc = pick_path(p, false, &tc);
    if (rc != FA_OK) return rc;
    rc = status_address(&p.status);
    if (rc != FA_OK) return rc;
    if (tc) return launch_fwd_tc(p);
    record_main_start(p.stream);
    rc = from_cuda(launch_fwd_simt(p));
    record_main_stop(p.stream);
    return rc;
}

int fa_fwd_fp8(const void* q, const void* k, const void* vt, const float* descale_q, const float* descale_k,
               const float* descale_v, void* o, float* lse, int B, int H, int N, int d, float scale, int causal,
               const uint8_t* block_mask, const int32_t* kv_len, void* stream) {
    int rc = check_common(B, H, N, d, scale, 0.f, FA_BF16);
    if (rc != FA_OK) return rc;
    if (d != 128) return FA_ERR_UNSUPPORTED;
    if (!(scale > 0.f)) return FA_ERR_UNSUPPORTED;
    if (N == 0) return FA_OK;
    if (N % 16 != 0) return FA_ERR_UNSUPPORTED;  // rows of vt must start 16-byte aligned
    if (!q || !k || !vt || !o || !lse || !descale_q || !descale_k || !descale_v) return FA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(vt, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
        !aligned(descale_q, 4) || !aligned(descale_k, 4) || !aligned(descale_v, 4))
        return FA_ERR_INVALID_ARG;
    if (block_mask && (N + kMaskBlock - 1) / kMaskBlock > kMaskListCap) return FA_ERR_UNSUPPORTED;
    Problem p{};
    fill_common(p, B, H, N, d, scale, causal, block_mask, 0.f, 0, FA_BF16, kv_len, stream);
    p.q = q;
    p.k = k;
    p.v = vt;
    p.o = o;
    p.lse = lse;
    rc = status_address(&p.status);
    if (rc != FA_OK) return rc;
    return launch_fwd_fp8(p, Fp8Inputs{descale_q, descale_k, descale_v});
}

size_t fa_fwd_splitkv_workspace_size(int B, int H, int N, int d, int n_splits) {
    if (B < 1 || H < 1 || N < 0 || (d != 64 && d != 128 && d != 256) || n_splits < 1 || n_splits > kMaxSplits)
        return 0;
    const size_t rows = (size_t)B * H * N;
    return round256((size_t)n_splits * rows * d * sizeof(float)) + round256((size_t)n_splits * rows * sizeof(float));
}

int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                   float scale, int causal, const uint8_t* block_mask, float dropout_p, uint64_t seed, fa_dtype dtype,
                   const int32_t* kv_len, int n_splits, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_common(B, H, N, d, scale, dropout_p, dtype);
    if (rc != FA_OK) return rc;
    if (n_splits < 1 || n_splits > kMaxSplits) return FA_ERR_INVALID_ARG;
    if (N == 0) return FA_OK;
    if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
        return FA_ERR_INVALID_ARG;
    const size_t need = fa_fwd_splitkv_workspace_size(B, H, N, d, n_splits);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return FA_ERR_WORKSPACE;
    Problem p{};
    fill_common(p, B, H, N, d, scale, causal, block_mask, dropout_p, seed, dtype, kv_len, stream);
    p.q = q;
    p.k = k;
    p.v = v;
    p.o = o;
    p.lse = lse;
    bool tc = false;
    rc = pick_path(p, false, &tc);
    if (rc != FA_OK) return rc;
    rc = status_address(&p.status);
    if (rc != FA_OK) return rc;
    // one split, or the CUDA-core kernels: the plain forward computes the
    // same result
    if (n_splits == 1 || !tc) {
        if (tc) return launch_fwd_tc(p);
        record_main_start(p.stream);
        rc = from_cuda(launch_fwd_simt(p));
        record_main_stop(p.stream);
        return rc;
    }
    const size_t rows = (size_t)B * H * N;
    p.n_splits = n_splits;
    p.o_part = static_cast<float*>(workspace);
    p.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + round256((size_t)n_splits * rows * d * sizeof(float)));
    return launch_fwd_tc(p);
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
    if (B < 1 || H < 1 || N < 0 || (d != 64 && d != 128 && d != 256)) return 0;
    const size_t rows = (size_t)B * H * N;
    // the per-row statistics (1 KB per 128-row tile: -LSE and -rowsum(dO o O)
    // of the tile's rows, or the plain row sums), the fp32 dQ accumulator,
    // the backward's work counter
    return round256(stats_bytes(B, H, N)) + round256(rows * (size_t)d * sizeof(float)) + 256;
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO, void* dq,
           void* dk, void* dv, int B, int H, int N, int d, float scale, int causal, const uint8_t* block_mask,
           float dropout_p, uint64_t seed, fa_dtype dtype, const int32_t* kv_len, void* workspace,
           size_t workspace_bytes, void* stream) {
    int rc = check_common(B, H, N, d, scale, dropout_p, dtype);
    if (rc != FA_OK) return rc;
    if (N == 0) return FA_OK;
    if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dO, 16) ||
        !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4))
        return FA_ERR_INVALID_ARG;
    const size_t need = fa_bwd_workspace_size(B, H, N, d);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return FA_ERR_WORKSPACE;
    Problem p{};
    fill_common(p, B, H, N, d, scale, causal, block_mask, dropout_p, seed, dtype, kv_len, stream);
    p.q = q;
    p.k = k;
    p.v = v;
    p.o = const_cast<void*>(o);
    p.lse = const_cast<float*>(lse);
    p.dO = dO;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    const size_t rows = (size_t)B * H * N;
    const size_t stats = round256(stats_bytes(B, H, N));
    p.delta = static_cast<float*>(workspace);
    p.col_table = static_cast<float*>(workspace);
    p.dq_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + stats);
    p.item_ctr = reinterpret_cast<int*>(static_cast<char*>(workspace) + stats + round256(rows * (size_t)d * sizeof(float)));
    bool tc = false;
    rc = pick_path(p, true, &tc);
    if (rc != FA_OK) return rc;
    rc = status_address(&p.status);
    if (rc != FA_OK) return rc;
    if (tc) return launch_bwd_tc(p);
    record_main_start(p.stream);
    rc = from_cuda(launch_bwd_simt(p));
    record_main_stop(p.stream);
    return rc;
}

int fa_dropout_mask(uint8_t* keep, int B, int H, int N, float p, uint64_t seed, void* stream) {
    if (B < 1 || H < 1 || N < 0 || !(p >= 0.f && p < 1.f)) return FA_ERR_INVALID_ARG;
    if (N == 0) return FA_OK;
    if (!keep) return FA_ERR_INVALID_ARG;
    return from_cuda(launch_dropout_mask(keep, B, H, N, keep_threshold(p), seed, static_cast<cudaStream_t>(stream)));
}

int fa_check_device_status(void* stream, int* site) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
    int host[2] = {0, 0};
    if (cudaMemcpyFromSymbol(host, g_status, sizeof(host)) != cudaSuccess) return FA_ERR_CUDA;
    if (host[0] != 0) {
        const int zero[2] = {0, 0};
        if (cudaMemcpyToSymbol(g_status, zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
    }
    if (site) *site = host[1];
    return host[0];
}

const char* fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid argument";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: unsupported head dim, dtype or size";
        case FA_ERR_CUDA: return "FA_ERR_CUDA: CUDA runtime error";
        case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: workspace missing, too small or misaligned";
        case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT: a device-side bounded wait ran out";
        default: return "unknown fa status";
    }
}

uint64_t fa_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int fa_set_main_kernel_events(void* ev_start, void* ev_stop) {
    if ((ev_start == nullptr) != (ev_stop == nullptr)) return FA_ERR_INVALID_ARG;
    g_main_start = static_cast<cudaEvent_t>(ev_start);
    g_main_stop = static_cast<cudaEvent_t>(ev_stop);
    return FA_OK;
}

int fa_set_kernel_path(int path) {
    const int old = g_kernel_path;
    g_kernel_path = (path == 1) ? 1 : 0;
    return old;
}

}  // extern "C"
