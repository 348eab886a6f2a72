// CUDA-core (fp32 FMA) kernels for exact tiled attention, any element type
// (fp32, bf16, fp16).
//
// These serve the fp32 inputs (where a single tf32 tensor-core pass cannot
// meet 1e-4 on O) and act as a second, independent GPU path for the bf16
// tensor-core kernels. They follow the same tiled algorithm: K/V tiles of
// 32 keys are staged in shared memory, each warp keeps the running row max
// m and row sum l of its query rows, and the output is rescaled by
// exp(m_old - m_new) whenever the max grows ("FlashAttention: Fast and
// Memory-Efficient Exact Attention with IO-Awareness", section "Metode",
// steps 1-4, with the normalisation deferred to the end as in the
// FlashAttention-2 section of the "Flash Attention" guide). The backward
// recomputes P from the stored log-sum-exp and splits into a dK/dV pass
// (one warp per key row, looping over query tiles) and a dQ pass (one warp
// per query row, looping over key tiles), so no atomics are needed.
#include <cmath>
#include <cstdint>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kRowsPerWarp = 4;
constexpr int kWarps = 4;
constexpr int kRowsPerCta = kRowsPerWarp * kWarps;  // 16
constexpr int kTile = 32;                           // keys (or queries) per staged tile

struct SimtArgs {
    const void* q;
    const void* k;
    const void* v;
    void* o;
    float* lse;
    const void* dO;
    void* dq;
    void* dk;
    void* dv;
    const float* delta_in;
    float* delta_out;
    int H, N;
    float scale;
    int causal;
    const uint8_t* block_mask;
    int nb;
    uint32_t thr;
    float inv_keep;
    int dropout;
    uint64_t seed;
    const int32_t* kv_len;
};

__device__ __forceinline__ bool visible(const SimtArgs& a, int L, int i, int j) {
    if (j >= L) return false;
    if (a.causal && j > i) return false;
    if (a.block_mask && !a.block_mask[(size_t)(i / kMaskBlock) * a.nb + (j / kMaskBlock)]) return false;
    return true;
}

// ---------------------------------------------------------------------------
// Forward: grid (ceil(N/16), B*H), 128 threads; warp w owns rows
// row0 + 4w .. row0 + 4w + 3; lane l scores key j0 + l of each staged tile.
// ---------------------------------------------------------------------------
template <int D>
constexpr size_t fwd_simt_smem() {
    return sizeof(float) * ((size_t)kRowsPerCta * D + (size_t)kTile * (D + 1) + (size_t)kTile * D);
}

template <typename T, int D>
__global__ void __launch_bounds__(128) fwd_simt_kernel(SimtArgs a) {
    constexpr int DPL = D / 32;  // output columns per lane
    // dynamic shared memory (at d = 256 the tiles pass the 48 KB static limit)
    extern __shared__ float simt_smem[];
    float(*sQ)[D] = reinterpret_cast<float(*)[D]>(simt_smem);                        // [kRowsPerCta][D]
    float(*sK)[D + 1] = reinterpret_cast<float(*)[D + 1]>(simt_smem + kRowsPerCta * D);  // [kTile][D + 1]
    float(*sV)[D] = reinterpret_cast<float(*)[D]>(simt_smem + kRowsPerCta * D + kTile * (D + 1));  // [kTile][D]

    const int bh = blockIdx.y, b = bh / a.H, h = bh % a.H;
    const int row0 = blockIdx.x * kRowsPerCta;
    const int N = a.N;
    const size_t base = (size_t)bh * N * D;
    const T* Q = static_cast<const T*>(a.q) + base;
    const T* K = static_cast<const T*>(a.k) + base;
    const T* V = static_cast<const T*>(a.v) + base;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (int e = tid; e < kRowsPerCta * D; e += blockDim.x) {
        const int r = e / D, c = e % D;
        sQ[r][c] = (row0 + r < N) ? to_f32(Q[(size_t)(row0 + r) * D + c]) : 0.f;
    }

    const int L = a.kv_len ? min(a.kv_len[b], N) : N;
    int kend = L;
    if (a.causal) kend = min(kend, min(N, row0 + kRowsPerCta));
    const float sl2 = a.scale * kLog2e;

    float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][DPL];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int t = 0; t < DPL; ++t) acc[r][t] = 0.f;
    }

    for (int j0 = 0; j0 < kend; j0 += kTile) {
        // 16 query rows and 32 keys each sit inside one 128 x 128 mask block.
        if (a.block_mask && !a.block_mask[(size_t)(row0 / kMaskBlock) * a.nb + j0 / kMaskBlock]) continue;
        __syncthreads();
        for (int e = tid; e < kTile * D; e += blockDim.x) {
            const int r = e / D, c = e % D;
            const int j = j0 + r;
            sK[r][c] = (j < N) ? to_f32(K[(size_t)j * D + c]) : 0.f;
            sV[r][c] = (j < N) ? to_f32(V[(size_t)j * D + c]) : 0.f;
        }
        __syncthreads();
        const int j = j0 + lane;
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const int lr = warp * kRowsPerWarp + r;
            const int i = row0 + lr;
            float s = 0.f;
#pragma unroll 8
            for (int c = 0; c < D; ++c) s = fmaf(sQ[lr][c], sK[lane][c], s);
            s = (i < N && visible(a, L, i, j)) ? s * sl2 : -INFINITY;
            const float mnew = fmaxf(m[r], warp_max(s));
            const float mref = (mnew == -INFINITY) ? 0.f : mnew;
            const float alpha = exp2f(m[r] - mref);
            const float pe = exp2f(s - mref);
            l[r] = l[r] * alpha + warp_sum(pe);
            float pd = pe;
            if (a.dropout && pe != 0.f && !keep_bit(a.seed, a.thr, b, bh % a.H, i, j)) pd = 0.f;
#pragma unroll
            for (int t = 0; t < DPL; ++t) acc[r][t] *= alpha;
#pragma unroll 4
            for (int jj = 0; jj < kTile; ++jj) {
                const float pj = __shfl_sync(0xffffffffu, pd, jj);
#pragma unroll
                for (int t = 0; t < DPL; ++t) acc[r][t] = fmaf(pj, sV[jj][lane + 32 * t], acc[r][t]);
            }
            m[r] = mnew;
        }
    }
    (void)h;

    T* O = static_cast<T*>(a.o) + base;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int i = row0 + warp * kRowsPerWarp + r;
        if (i >= N) continue;
        const float inv = (l[r] > 0.f) ? a.inv_keep / l[r] : 0.f;
#pragma unroll
        for (int t = 0; t < DPL; ++t) O[(size_t)i * D + lane + 32 * t] = from_f32<T>(acc[r][t] * inv);
        if (lane == 0) a.lse[(size_t)bh * N + i] = (l[r] > 0.f) ? (m[r] + log2f(l[r])) * kLn2 : -INFINITY;
    }
}

// ---------------------------------------------------------------------------
// Backward preprocess: delta[i] = sum_c dO[i][c] * O[i][c]; one warp per row.
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const T* __restrict__ O, const T* __restrict__ dO,
                                                             float* __restrict__ delta, size_t rows) {
    const size_t row = (size_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    float s = 0.f;
#pragma unroll
    for (int t = 0; t < D / 32; ++t) {
        const size_t e = row * D + lane + 32 * t;
        s = fmaf(to_f32(O[e]), to_f32(dO[e]), s);
    }
    s = warp_sum(s);
    if (lane == 0) delta[row] = s;
}

// ---------------------------------------------------------------------------
// Backward dK/dV: grid (ceil(N/16), B*H); warp w owns key rows
// key0 + 4w .. +3; lane l handles query i0 + l of each staged query tile.
// ---------------------------------------------------------------------------
template <int D>
constexpr size_t bwd_simt_smem() {  // either backward kernel
    return sizeof(float) * (2 * (size_t)kRowsPerCta * D + 2 * (size_t)kTile * (D + 1) + 2 * (size_t)kTile);
}

template <typename T, int D>
__global__ void __launch_bounds__(128) bwd_dkdv_simt_kernel(SimtArgs a) {
    constexpr int DPL = D / 32;
    extern __shared__ float simt_smem[];
    float(*sKr)[D] = reinterpret_cast<float(*)[D]>(simt_smem);                     // [kRowsPerCta][D]
    float(*sVr)[D] = reinterpret_cast<float(*)[D]>(simt_smem + kRowsPerCta * D);   // [kRowsPerCta][D]
    float(*sQ)[D + 1] = reinterpret_cast<float(*)[D + 1]>(simt_smem + 2 * kRowsPerCta * D);  // [kTile][D + 1]
    float(*sdO)[D + 1] =
        reinterpret_cast<float(*)[D + 1]>(simt_smem + 2 * kRowsPerCta * D + kTile * (D + 1));  // [kTile][D + 1]
    float* sLse = simt_smem + 2 * kRowsPerCta * D + 2 * kTile * (D + 1);  // [kTile]
    float* sDelta = sLse + kTile;                                          // [kTile]

    const int bh = blockIdx.y, b = bh / a.H, h = bh % a.H;
    const int key0 = blockIdx.x * kRowsPerCta;
    const int N = a.N;
    const size_t base = (size_t)bh * N * D;
    const T* Q = static_cast<const T*>(a.q) + base;
    const T* K = static_cast<const T*>(a.k) + base;
    const T* V = static_cast<const T*>(a.v) + base;
    const T* dO = static_cast<const T*>(a.dO) + base;
    const float* lse = a.lse + (size_t)bh * N;
    const float* delta = a.delta_in + (size_t)bh * N;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = a.kv_len ? min(a.kv_len[b], N) : N;

    for (int e = tid; e < kRowsPerCta * D; e += blockDim.x) {
        const int r = e / D, c = e % D;
        const bool in = key0 + r < N;
        sKr[r][c] = in ? to_f32(K[(size_t)(key0 + r) * D + c]) : 0.f;
        sVr[r][c] = in ? to_f32(V[(size_t)(key0 + r) * D + c]) : 0.f;
    }

    float dk[kRowsPerWarp][DPL], dv[kRowsPerWarp][DPL];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int t = 0; t < DPL; ++t) dk[r][t] = dv[r][t] = 0.f;

    const float sl2 = a.scale * kLog2e;
    const int istart = a.causal ? (key0 / kTile) * kTile : 0;
    if (key0 < L) {
        for (int i0 = istart; i0 < N; i0 += kTile) {
            if (a.block_mask && !a.block_mask[(size_t)(i0 / kMaskBlock) * a.nb + key0 / kMaskBlock]) continue;
            __syncthreads();
            for (int e = tid; e < kTile * D; e += blockDim.x) {
                const int r = e / D, c = e % D;
                const int i = i0 + r;
                sQ[r][c] = (i < N) ? to_f32(Q[(size_t)i * D + c]) : 0.f;
                sdO[r][c] = (i < N) ? to_f32(dO[(size_t)i * D + c]) : 0.f;
            }
            if (tid < kTile) {
                const int i = i0 + tid;
                sLse[tid] = (i < N) ? lse[i] : -INFINITY;
                sDelta[tid] = (i < N) ? delta[i] : 0.f;
            }
            __syncthreads();
            const int i = i0 + lane;
            const float lse2 = sLse[lane] * kLog2e;
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                const int lr = warp * kRowsPerWarp + r;
                const int j = key0 + lr;
                float s = 0.f, dph = 0.f;
#pragma unroll 8
                for (int c = 0; c < D; ++c) {
                    s = fmaf(sQ[lane][c], sKr[lr][c], s);
                    dph = fmaf(sdO[lane][c], sVr[lr][c], dph);
                }
                const bool vis = i < N && j < N && sLse[lane] != -INFINITY && visible(a, L, i, j);
                const float p = vis ? exp2f(s * sl2 - lse2) : 0.f;
                float zk = a.inv_keep;
                if (a.dropout && vis && !keep_bit(a.seed, a.thr, b, h, i, j)) zk = 0.f;
                const float pd = p * zk;
                const float ds = p * (dph * zk - sDelta[lane]);
#pragma unroll 4
                for (int ii = 0; ii < kTile; ++ii) {
                    const float pdi = __shfl_sync(0xffffffffu, pd, ii);
                    const float dsi = __shfl_sync(0xffffffffu, ds, ii);
#pragma unroll
                    for (int t = 0; t < DPL; ++t) {
                        dv[r][t] = fmaf(pdi, sdO[ii][lane + 32 * t], dv[r][t]);
                        dk[r][t] = fmaf(dsi, sQ[ii][lane + 32 * t], dk[r][t]);
                    }
                }
            }
        }
    }

    T* dK = static_cast<T*>(a.dk) + base;
    T* dV = static_cast<T*>(a.dv) + base;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int j = key0 + warp * kRowsPerWarp + r;
        if (j >= N) continue;
#pragma unroll
        for (int t = 0; t < DPL; ++t) {
            dK[(size_t)j * D + lane + 32 * t] = from_f32<T>(dk[r][t] * a.scale);
            dV[(size_t)j * D + lane + 32 * t] = from_f32<T>(dv[r][t]);
        }
    }
}

// ---------------------------------------------------------------------------
// Backward dQ: grid (ceil(N/16), B*H); warp w owns query rows; lane l
// handles key j0 + l of each staged key tile.
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(128) bwd_dq_simt_kernel(SimtArgs a) {
    constexpr int DPL = D / 32;
    extern __shared__ float simt_smem[];
    float(*sQ)[D] = reinterpret_cast<float(*)[D]>(simt_smem);                    // [kRowsPerCta][D]
    float(*sdO)[D] = reinterpret_cast<float(*)[D]>(simt_smem + kRowsPerCta * D);  // [kRowsPerCta][D]
    float(*sK)[D + 1] = reinterpret_cast<float(*)[D + 1]>(simt_smem + 2 * kRowsPerCta * D);  // [kTile][D + 1]
    float(*sV)[D + 1] =
        reinterpret_cast<float(*)[D + 1]>(simt_smem + 2 * kRowsPerCta * D + kTile * (D + 1));  // [kTile][D + 1]

    const int bh = blockIdx.y, b = bh / a.H, h = bh % a.H;
    const int row0 = blockIdx.x * kRowsPerCta;
    const int N = a.N;
    const size_t base = (size_t)bh * N * D;
    const T* Q = static_cast<const T*>(a.q) + base;
    const T* K = static_cast<const T*>(a.k) + base;
    const T* V = static_cast<const T*>(a.v) + base;
    const T* dO = static_cast<const T*>(a.dO) + base;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = a.kv_len ? min(a.kv_len[b], N) : N;

    for (int e = tid; e < kRowsPerCta * D; e += blockDim.x) {
        const int r = e / D, c = e % D;
        const bool in = row0 + r < N;
        sQ[r][c] = in ? to_f32(Q[(size_t)(row0 + r) * D + c]) : 0.f;
        sdO[r][c] = in ? to_f32(dO[(size_t)(row0 + r) * D + c]) : 0.f;
    }
    float lse2[kRowsPerWarp], dlt[kRowsPerWarp], dq[kRowsPerWarp][DPL];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int i = row0 + warp * kRowsPerWarp + r;
        lse2[r] = (i < N) ? a.lse[(size_t)bh * N + i] * kLog2e : -INFINITY;
        dlt[r] = (i < N) ? a.delta_in[(size_t)bh * N + i] : 0.f;
#pragma unroll
        for (int t = 0; t < DPL; ++t) dq[r][t] = 0.f;
    }

    int kend = L;
    if (a.causal) kend = min(kend, min(N, row0 + kRowsPerCta));
    const float sl2 = a.scale * kLog2e;
    for (int j0 = 0; j0 < kend; j0 += kTile) {
        if (a.block_mask && !a.block_mask[(size_t)(row0 / kMaskBlock) * a.nb + j0 / kMaskBlock]) continue;
        __syncthreads();
        for (int e = tid; e < kTile * D; e += blockDim.x) {
            const int r = e / D, c = e % D;
            const int j = j0 + r;
            sK[r][c] = (j < N) ? to_f32(K[(size_t)j * D + c]) : 0.f;
            sV[r][c] = (j < N) ? to_f32(V[(size_t)j * D + c]) : 0.f;
        }
        __syncthreads();
        const int j = j0 + lane;
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const int lr = warp * kRowsPerWarp + r;
            const int i = row0 + lr;
            float s = 0.f, dph = 0.f;
#pragma unroll 8
            for (int c = 0; c < D; ++c) {
                s = fmaf(sQ[lr][c], sK[lane][c], s);
                dph = fmaf(sdO[lr][c], sV[lane][c], dph);
            }
            const bool vis = i < N && lse2[r] != -INFINITY && visible(a, L, i, j);
            const float p = vis ? exp2f(s * sl2 - lse2[r]) : 0.f;
            float zk = a.inv_keep;
            if (a.dropout && vis && !keep_bit(a.seed, a.thr, b, h, i, j)) zk = 0.f;
            const float ds = p * (dph * zk - dlt[r]);
#pragma unroll 4
            for (int jj = 0; jj < kTile; ++jj) {
                const float dsj = __shfl_sync(0xffffffffu, ds, jj);
#pragma unroll
                for (int t = 0; t < DPL; ++t) dq[r][t] = fmaf(dsj, sK[jj][lane + 32 * t], dq[r][t]);
            }
        }
    }

    T* dQ = static_cast<T*>(a.dq) + base;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int i = row0 + warp * kRowsPerWarp + r;
        if (i >= N) continue;
#pragma unroll
        for (int t = 0; t < DPL; ++t) dQ[(size_t)i * D + lane + 32 * t] = from_f32<T>(dq[r][t] * a.scale);
    }
}

// One thread per (row, group of 4 keys): one Philox call gives 4 keep bits.
__global__ void dropout_mask_kernel(uint8_t* keep, int H, int N, uint32_t thr, uint64_t seed, size_t rows) {
    const int groups = (N + 3) / 4;
    const size_t gid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= rows * groups) return;
    const size_t row = gid / groups;
    const int j4 = (int)(gid % groups);
    const int i = (int)(row % N);
    const int h = (int)((row / N) % H);
    const int b = (int)(row / ((size_t)N * H));
    const uint32_t bits = keep_bits4(seed, thr, b, h, i, j4);
    uint8_t* out = keep + row * N + 4 * j4;
    for (int w = 0; w < 4 && 4 * j4 + w < N; ++w) out[w] = (bits >> w) & 1u;
}

SimtArgs make_args(const Problem& p) {
    SimtArgs a{};
    a.q = p.q;
    a.k = p.k;
    a.v = p.v;
    a.o = p.o;
    a.lse = p.lse;
    a.dO = p.dO;
    a.dq = p.dq;
    a.dk = p.dk;
    a.dv = p.dv;
    a.delta_in = p.delta;
    a.delta_out = p.delta;
    a.H = p.H;
    a.N = p.N;
    a.scale = p.scale;
    a.causal = p.causal;
    a.block_mask = p.block_mask;
    a.nb = p.nb;
    a.thr = p.drop_threshold;
    a.inv_keep = 1.0f / (1.0f - p.dropout_p);
    a.dropout = p.dropout_p > 0.f;
    a.seed = p.seed;
    a.kv_len = p.kv_len;
    return a;
}

// Opts a kernel into more than 48 KB of dynamic shared memory (once).
template <typename K>
cudaError_t allow_smem(K kernel, size_t bytes, bool& done) {
    if (done || bytes <= 48 * 1024) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) done = true;
    return e;
}

template <typename T, int D>
cudaError_t fwd_simt(const Problem& p) {
    constexpr size_t smem = fwd_simt_smem<D>();
    static bool attr = false;
    cudaError_t e = allow_smem(fwd_simt_kernel<T, D>, smem, attr);
    if (e != cudaSuccess) return e;
    dim3 grid((p.N + kRowsPerCta - 1) / kRowsPerCta, p.B * p.H);
    fwd_simt_kernel<T, D><<<grid, 128, smem, p.stream>>>(make_args(p));
    note_launches(1);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t bwd_pre(const Problem& p) {
    const size_t rows = (size_t)p.B * p.H * p.N;
    const unsigned blocks = (unsigned)((rows + 7) / 8);
    bwd_preprocess_kernel<T, D><<<blocks, 256, 0, p.stream>>>(static_cast<const T*>(p.o),
                                                              static_cast<const T*>(p.dO), p.delta, rows);
    note_launches(1);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t bwd_simt(const Problem& p) {
    cudaError_t e = bwd_pre<T, D>(p);
    if (e != cudaSuccess) return e;
    constexpr size_t smem = bwd_simt_smem<D>();
    static bool attr_kv = false, attr_q = false;
    if ((e = allow_smem(bwd_dkdv_simt_kernel<T, D>, smem, attr_kv)) != cudaSuccess) return e;
    if ((e = allow_smem(bwd_dq_simt_kernel<T, D>, smem, attr_q)) != cudaSuccess) return e;
    dim3 grid((p.N + kRowsPerCta - 1) / kRowsPerCta, p.B * p.H);
    const SimtArgs a = make_args(p);
    bwd_dkdv_simt_kernel<T, D><<<grid, 128, smem, p.stream>>>(a);
    note_launches(1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_dq_simt_kernel<T, D><<<grid, 128, smem, p.stream>>>(a);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace

// head dims 64, 128 and 256 (the caller has checked d)
#define FA_SIMT_BY_D(fn, T) (p.d == 64 ? fn<T, 64>(p) : p.d == 128 ? fn<T, 128>(p) : fn<T, 256>(p))

cudaError_t launch_fwd_simt(const Problem& p) {
    if (p.dtype == FA_BF16) return FA_SIMT_BY_D(fwd_simt, __nv_bfloat16);
    if (p.dtype == FA_FP16) return FA_SIMT_BY_D(fwd_simt, __half);
    return FA_SIMT_BY_D(fwd_simt, float);
}

cudaError_t launch_bwd_preprocess(const Problem& p) {
    if (p.dtype == FA_BF16) return FA_SIMT_BY_D(bwd_pre, __nv_bfloat16);
    if (p.dtype == FA_FP16) return FA_SIMT_BY_D(bwd_pre, __half);
    return FA_SIMT_BY_D(bwd_pre, float);
}

cudaError_t launch_bwd_simt(const Problem& p) {
    if (p.dtype == FA_BF16) return FA_SIMT_BY_D(bwd_simt, __nv_bfloat16);
    if (p.dtype == FA_FP16) return FA_SIMT_BY_D(bwd_simt, __half);
    return FA_SIMT_BY_D(bwd_simt, float);
}

cudaError_t launch_dropout_mask(uint8_t* keep, int B, int H, int N, uint32_t thr, uint64_t seed, cudaStream_t s) {
    const size_t rows = (size_t)B * H * N;
    const size_t work = rows * (size_t)((N + 3) / 4);
    if (work == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((work + 255) / 256);
    dropout_mask_kernel<<<blocks, 256, 0, s>>>(keep, H, N, thr, seed, rows);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace fa
