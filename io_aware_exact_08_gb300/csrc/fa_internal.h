// Internal declarations shared by the library's translation units.
// Not part of the public ABI (that is include/fa.h).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/fa.h"

namespace fa {

// Everything a launch needs; filled and validated by the C entry points.
struct Problem {
    const void* q;
    const void* k;
    const void* v;
    void* o;
    float* lse;
    const void* dO;
    void* dq;
    void* dk;
    void* dv;
    int B, H, N, d;
    float scale;
    int causal;
    const uint8_t* block_mask;  // nb x nb or nullptr
    int nb;                     // ceil(N / 128)
    float dropout_p;
    uint32_t drop_threshold;    // keep iff philox word >= drop_threshold
    uint64_t seed;
    fa_dtype dtype;
    const int32_t* kv_len;      // [B] or nullptr
    float* delta;               // workspace: rowsum(dO o O), fp32 [B,H,N] (d = 256 and CUDA-core backward)
    // workspace, the same bytes as delta (tensor-core backward at d = 64, 128):
    // per (b*h, 128-row query tile) 128 floats -LSE*log2(e) then 128 floats
    // -rowsum(dO o O), rows past N padded with -inf and 0 (kColTableFloats
    // floats a tile)
    float* col_table;
    float* dq_acc;              // workspace: fp32 [B,H,N,d]
    int* item_ctr = nullptr;    // workspace: the backward's work counter (zeroed by its first kernel)
    int* status;                // device status word (timeouts)
    cudaStream_t stream;
    // split-KV forward: n_splits key-tile ranges per pair of query tiles,
    // partial O / LSE in the caller's workspace, merged after (1 = off)
    int n_splits = 1;
    float* o_part = nullptr;    // [n_splits][B*H][N][d] fp32
    float* lse_part = nullptr;  // [n_splits][B*H][N] fp32
};

constexpr int kMaxSplits = 64;

constexpr int kColTableFloats = 256;

constexpr int kMaskBlock = 128;
// With a block mask the tensor-core kernels keep each CTA's list of visible
// tiles in shared memory: at most kMaskListCap entries (kMaskListCapBwd128
// in the d = 128 backward and kMaskListCapBwd256 in the d = 256 backward,
// whose shared memory is otherwise full). Larger masks run on the CUDA-core
// kernels.
constexpr int kMaskListCap = 1024;
constexpr int kMaskListCapBwd128 = 256;
constexpr int kMaskListCapBwd256 = 256;

// Counts kernel launches for fa_launch_count (thread-safe).
void note_launches(int n);

// Diagnostic timing (fa_set_main_kernel_events): record the caller's events
// on `s` right before and right after the launch(es) of a call's main
// kernel; no-ops while no events are set.
void record_main_start(cudaStream_t s);
void record_main_stop(cudaStream_t s);

// Device address of the status word on the current device (looked up once
// per device).
int status_address(int** out);

// CUDA-core kernels (any dtype, d in {64,128,256}); implemented in fa_simt.cu.
cudaError_t launch_fwd_simt(const Problem& p);
cudaError_t launch_bwd_simt(const Problem& p);
cudaError_t launch_bwd_preprocess(const Problem& p);
cudaError_t launch_dropout_mask(uint8_t* keep, int B, int H, int N, uint32_t thr, uint64_t seed,
                                cudaStream_t s);

// tcgen05 kernels (bf16, fp16): forward d in {64,128,256} (fa_fwd_sm103.cu),
// backward d in {64,128} (fa_bwd_sm103.cu) and d = 256 (fa_bwd256_sm103.cu).
int launch_fwd_tc(const Problem& p);
// head dim 64, one query tile per CTA, two CTAs per SM (fa_fwd1t_sm103.cu)
int launch_fwd_1t(const Problem& p);

// FP8 forward (fa_fwd_fp8.cu): E4M3 q, k (Problem::q, k) and the transposed
// vt (Problem::v), with per-head dequantisation factors; head dim 128.
struct Fp8Inputs {
    const float* descale_q;
    const float* descale_k;
    const float* descale_v;
};
int launch_fwd_fp8(const Problem& p, const Fp8Inputs& in);
int launch_bwd_tc(const Problem& p);
int launch_bwd256_tc(const Problem& p);

}  // namespace fa
