// Device helpers shared by the CUDA-core and tensor-core kernels:
// element conversion, the dropout keep bit (Philox4x32-10), warp reductions.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace fa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw: "Parallel Random Numbers: As
// Easy as 1, 2, 3", SC'11). Counter (c0..c3), key (k0, k1); ten rounds, each
// two 32x32->64 products; the key advances by the Weyl increments between
// rounds.
struct Philox4 {
    uint32_t x, y, z, w;
};

// The full 64-bit product of two 32-bit words in one instruction
// (mul.wide.u32): both halves of each round's two products come from it.
__device__ __forceinline__ void mul_wide(uint32_t a, uint32_t b, uint32_t& hi, uint32_t& lo) {
    uint64_t prod;
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(prod) : "r"(a), "r"(b));
    lo = (uint32_t)prod;
    hi = (uint32_t)(prod >> 32);
}

__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                uint32_t k0, uint32_t k1) {
    constexpr uint32_t kMul0 = 0xD2511F53u, kMul1 = 0xCD9E8D57u;
    constexpr uint32_t kInc0 = 0x9E3779B9u, kInc1 = 0xBB67AE85u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        uint32_t hi0, lo0, hi1, lo1;
        mul_wide(kMul0, c0, hi0, lo0);
        mul_wide(kMul1, c2, hi1, lo1);
        const uint32_t n0 = hi1 ^ c1 ^ k0;
        const uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
        k0 += kInc0;
        k1 += kInc1;
    }
    return {c0, c1, c2, c3};
}

// The 4 keep bits of keys j4*4 .. j4*4+3 for query row i of head (b, h):
// bit w set iff word w of Philox((j4, i, h, b), (lo32(seed), hi32(seed))) >= thr.
__device__ __forceinline__ uint32_t keep_bits4(uint64_t seed, uint32_t thr, int b, int h, int i, int j4) {
    const Philox4 r = philox4x32_10((uint32_t)j4, (uint32_t)i, (uint32_t)h, (uint32_t)b,
                                    (uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32));
    return (uint32_t)(r.x >= thr) | ((uint32_t)(r.y >= thr) << 1) | ((uint32_t)(r.z >= thr) << 2) |
           ((uint32_t)(r.w >= thr) << 3);
}

__device__ __forceinline__ bool keep_bit(uint64_t seed, uint32_t thr, int b, int h, int i, int j) {
    return (keep_bits4(seed, thr, b, h, i, j >> 2) >> (j & 3)) & 1u;
}

// Warp-cooperative list of the block-mask entries that are set: the indices
// t in [lo, hi) with mask[t * stride] != 0, in increasing order, written to
// `list` (shared memory). Returns the count on every lane. The loads of four
// 32-entry chunks are issued before any of them is used, so a scan of up to
// 128 entries waits for one memory latency rather than four.
__device__ __forceinline__ int warp_list_visible(const uint8_t* mask, size_t stride, int lo, int hi, uint16_t* list,
                                                 int lane) {
    int cnt = 0;
    for (int c = lo & ~31; c < hi; c += 128) {
        bool act[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int t = c + 32 * k + lane;
            act[k] = t >= lo && t < hi && mask[(size_t)t * stride] != 0;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t bal = __ballot_sync(0xffffffffu, act[k]);
            if (act[k]) list[cnt + __popc(bal & ((1u << lane) - 1u))] = (uint16_t)(c + 32 * k + lane);
            cnt += __popc(bal);
        }
    }
    return cnt;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace fa
