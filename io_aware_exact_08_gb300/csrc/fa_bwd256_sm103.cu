// Backward attention at head dim 256 on the tensor cores, in three passes.
//
// The gradients are those of the d <= 128 kernel (recomputation of S and P
// from the stored log-sum-exp, "FlashAttention: Fast and Memory-Efficient
// Exact Attention with IO-Awareness", section "Ide Utama", third point):
//   dV = P^T dO,  dP = (dO V^T) o Z/(1-p),  dS = P o (dP - delta),
//   dK = scale dS^T Q,  dQ = scale dS K,  delta_i = sum_c dO_ic O_ic.
// At d = 256 one 128 x 256 fp32 accumulator takes 256 of the 512 TMEM
// columns, so dK and dV cannot both stay in TMEM next to S^T and dP^T. Each
// pass therefore keeps one accumulator and recomputes what it needs:
//   pass dV (CTA = key tile j):   S^T = K_j Q_i^T,  dV_j += P^T dO_i
//   pass dK (CTA = key tile j):   S^T, dP^T = V_j dO_i^T,  dK_j += dS^T Q_i
//   pass dQ (CTA = query tile i): S = Q_i K_j^T, dP = dO_i V_j^T,  dQ_i += dS K_j
// (8 products of 128 x 128 x 256 per tile pair instead of 5), and writes its
// gradient directly: no fp32 accumulator in global memory, no atomics.
//
// TMEM: X (S or S^T) in columns 0-127, Y (dP or dP^T) in 128-255, the
// accumulator in 256-511. The 16-bit operand of the accumulating product (P
// or dS) is written back over X: the 64 values of a warp's column half go to
// the first 32 of that half's 64 columns, which the warp has read.
// Shared memory: the CTA's own tiles (1 or 2 of 64 KB) stay resident; the
// streamed tiles pass through a ring of six 16 KB slots, one 64-column box
// each, in the order the MMAs use them. The accumulating product reads its
// B operand two boxes (128 columns) at a time from adjacent slots; the
// loads come in groups of 4, so a pair never wraps around the ring.
// Roles (320 threads): warps 0-7 compute (thread = TMEM lane = row, warp
// half w / 4 takes 64 of the 128 columns), warp 8 TMA producer, warp 9 MMA
// issuer (all lanes run its loop, one elected lane issues).
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>

#include <cuda.h>

#include "fa_device.cuh"
#include "fa_internal.h"
#include "fa_sm103.cuh"

namespace fa {

bool make_tmap16(CUtensorMap* map, const void* base, int BH, int N, int d, int box_rows, CUtensorMapDataType type);

namespace {

using namespace sm103;

constexpr int D = 256;
constexpr int kTile = 128;
constexpr int kThreads = 320;
constexpr int kComputeWarps = 8;
constexpr int kBoxBytes = kTile * 128;      // 128 rows x 64 columns, 16-bit
constexpr int kTileBytes = 4 * kBoxBytes;   // 128 x 256
constexpr int kSlots = 6;
constexpr uint32_t kColX = 0, kColY = 128, kColAcc = 256;

enum Mode { kDV = 0, kDK = 1, kDQ = 2 };

template <int kMode>
struct Bwd256Cfg {
    static constexpr int kResident = (kMode == kDV) ? 1 : 2;    // resident 128 x 256 tiles
    static constexpr int kListBytes = kMaskListCapBwd256 * 2;
    // resident tiles, ring, -LSE / -delta of the step's columns (two
    // buffers each, dV/dK passes), barriers, block-mask list
    static constexpr int kSmem = kResident * kTileBytes + kSlots * kBoxBytes + 4 * kTile * 4 + 256 + kListBytes;
};

struct Bwd256Params {
    const float* lse;
    const float* delta;
    void* out;  // dV, dK or dQ
    const uint8_t* block_mask;
    const int32_t* kv_len;
    int* status;
    int H, N, nb;
    float scale;
    float scale_log2;
    float keep_scale;  // 1/(1-p)
    uint32_t drop_thr;
    int dropout;
    int causal;
    uint64_t seed;
};

struct Bwd256Shared {
    uint64_t res_full;
    uint64_t slot_full[kSlots];
    uint64_t slot_empty[kSlots];
    uint64_t x_full;    // X (and Y) of the step in TMEM
    uint64_t op_ready;  // the 16-bit operand written over X, X and Y read
    uint64_t col_ready[2];  // per column half: the step's -LSE / -delta staged
    uint64_t acc_done;
    uint64_t teardown;
    uint32_t tmem_base;
    int abort_flag;
    int n_list;
};
static_assert(sizeof(Bwd256Shared) <= 256, "barrier block");

// The tiles a CTA visits, in increasing order. dV/dK passes (key tile jt):
// query tiles [causal ? jt : 0, nqt) whose rows see a key of the tile;
// dQ pass (query tile qt): key tiles [0, causal ? qt + 1 : nkt). With a block
// mask, the list built in shared memory.
struct Sched256 {
    int first, end;  // range without a mask
    const uint16_t* list;
    int n_list;
    bool mask;
    __device__ int count() const { return mask ? n_list : max(0, end - first); }
    __device__ int tile(int u) const { return mask ? (int)list[u] : first + u; }
};

template <typename T, int kMode, bool kMask>
__global__ void __launch_bounds__(kThreads, 1)
    bwd256_kernel(const __grid_constant__ CUtensorMap tm_r0, const __grid_constant__ CUtensorMap tm_r1,
                  const __grid_constant__ CUtensorMap tm_s0, const __grid_constant__ CUtensorMap tm_s1,
                  const Bwd256Params p) {
    using Cfg = Bwd256Cfg<kMode>;
    constexpr bool kKeyRows = (kMode != kDQ);  // TMEM lanes are key rows (dV, dK) or query rows (dQ)
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {  // swizzled tiles need 1024-byte alignment
        if (threadIdx.x == 0 && atomicCAS(p.status, 0, (int)FA_ERR_CUDA) == 0) atomicExch(p.status + 1, 230);
        return;
    }
    uint8_t* sRes = smem_raw;                                   // resident tiles
    uint8_t* sRing = sRes + Cfg::kResident * kTileBytes;        // kSlots boxes
    float* sNegLse = reinterpret_cast<float*>(sRing + kSlots * kBoxBytes);  // [2][128]
    float* sNegDelta = sNegLse + 2 * kTile;                     // [2][128]
    Bwd256Shared* st = reinterpret_cast<Bwd256Shared*>(sNegDelta + 2 * kTile);
    uint16_t* sList = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(st) + 256);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x;
    const int b = bh / p.H, h = bh % p.H;
    const int ntiles = (p.N + kTile - 1) / kTile;
    const int L = p.kv_len ? min(max(p.kv_len[b], 0), p.N) : p.N;
    const int nkt = (L + kTile - 1) / kTile;  // key tiles with a visible key
    // own tile: key tile (dV, dK; lowest first, the heaviest under a causal
    // mask) or query tile (dQ; highest first)
    const int own = kKeyRows ? (int)blockIdx.y : (p.causal ? ntiles - 1 - (int)blockIdx.y : (int)blockIdx.y);
    const int own0 = own * kTile;

    Sched256 sched;
    sched.list = sList;
    sched.n_list = 0;
    sched.mask = kMask;
    if (kKeyRows) {
        sched.first = p.causal ? own : 0;
        sched.end = (own < nkt) ? ntiles : 0;  // a key tile past kv_len contributes nothing
    } else {
        sched.first = 0;
        sched.end = p.causal ? min(nkt, own + 1) : nkt;
    }
    WaitCtx wctx{&st->abort_flag, p.status};
    if (kMask && warp == 0) {
        // dV, dK: query tiles i with block (i, own) set; dQ: key tiles j with
        // block (own, j) set; within the unmasked range, 32 at a time
        const int cnt = kKeyRows ? warp_list_visible(p.block_mask + own, (size_t)p.nb, sched.first, sched.end, sList, lane)
                                 : warp_list_visible(p.block_mask + (size_t)own * p.nb, 1, sched.first, sched.end,
                                                     sList, lane);
        if (lane == 0) st->n_list = cnt;
    }
    if (tid == 0) {
        mbar_init(&st->res_full, 1);
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&st->slot_full[s], 1);
            mbar_init(&st->slot_empty[s], 1);
        }
        mbar_init(&st->x_full, 1);
        mbar_init(&st->op_ready, kComputeWarps);
        mbar_init(&st->col_ready[0], kComputeWarps / 2);
        mbar_init(&st->col_ready[1], kComputeWarps / 2);
        mbar_init(&st->acc_done, 1);
        mbar_init(&st->teardown, 1);
        st->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(&st->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = st->tmem_base;
    if constexpr (kMask) sched.n_list = st->n_list;
    const int n = sched.count();

    if (warp == 8) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && n > 0) {
            prefetch_tmap(&tm_r0);
            if (Cfg::kResident > 1) prefetch_tmap(&tm_r1);
            prefetch_tmap(&tm_s0);
            prefetch_tmap(&tm_s1);
            mbar_arrive_expect_tx(&st->res_full, Cfg::kResident * kTileBytes);
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                tma_load_3d(sRes + x * kBoxBytes, &tm_r0, &st->res_full, x * 64, own0, bh);
                if (Cfg::kResident > 1)
                    tma_load_3d(sRes + kTileBytes + x * kBoxBytes, &tm_r1, &st->res_full, x * 64, own0, bh);
            }
            int t = 0;  // load counter
            bool okp = true;
            auto load = [&](const CUtensorMap* map, int x, int row) {
                const int s = t % kSlots;
                const uint32_t ph = (t / kSlots) & 1;
                if (!mbar_wait(&st->slot_empty[s], ph ^ 1, wctx, 201)) {
                    okp = false;
                    return;
                }
                mbar_arrive_expect_tx(&st->slot_full[s], kBoxBytes);
                tma_load_3d(sRing + s * kBoxBytes, map, &st->slot_full[s], x * 64, row, bh);
                ++t;
            };
            // per step: the 4 boxes of s0 (X), of s1 (Y; dO for the dV pass's
            // accumulation), and of s0 again (the dK and dQ accumulation)
            for (int u = 0; okp && u < n; ++u) {
                const int row = sched.tile(u) * kTile;
                for (int x = 0; okp && x < 4; ++x) load(&tm_s0, x, row);
                for (int x = 0; okp && x < 4; ++x) load(&tm_s1, x, row);
                if (kMode != kDV)
                    for (int x = 0; okp && x < 4; ++x) load(&tm_s0, x, row);
            }
            for (int l = max(0, t - kSlots); l < t; ++l)
                mbar_wait(&st->slot_full[l % kSlots], (l / kSlots) & 1, wctx, 202);
            mbar_wait(&st->res_full, 0, wctx, 203);
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        if (n > 0) {
            constexpr uint32_t idesc_x = idesc_f32acc(Elem16<T>::kFmt, kTile, kTile, 0, 0);
            constexpr uint32_t idesc_acc = idesc_f32acc(Elem16<T>::kFmt, kTile, 128, 0, 1);
            const uint32_t ring = smem_u32(sRing);
            const uint64_t r0d = smem_desc_sw128(smem_u32(sRes), 16, 1024);
            const uint64_t r1d = smem_desc_sw128(smem_u32(sRes + kTileBytes), 16, 1024);
            const uint64_t ring_k = smem_desc_sw128(ring, 16, 1024);         // K-major box
            const uint64_t ring_mn = smem_desc_sw128(ring, kBoxBytes, 1024);  // MN-major, 2 boxes
            constexpr uint32_t kSlotUnits = kBoxBytes >> 4;
            bool ok = mbar_wait_warp(&st->res_full, 0, wctx, 210);
            tc_fence_after();
            int ld = 0;  // next load to use
            // D[col] = R . box^T over the 4 boxes of one streamed tile
            auto product = [&](uint32_t col, uint64_t rd) -> bool {
#pragma unroll 1
                for (int x = 0; x < 4; ++x) {
                    const int s = ld % kSlots;
                    if (!mbar_wait_warp(&st->slot_full[s], (ld / kSlots) & 1, wctx, 211)) return false;
                    tc_fence_after();
                    const uint64_t bd = ring_k + (uint64_t)(s * kSlotUnits);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_ss_warp(tmem + col, desc_add(rd, x * kBoxBytes + kk * 32), desc_add(bd, kk * 32), idesc_x,
                                    (x > 0 || kk > 0) ? 1u : 0u);
                    mma_commit_warp(&st->slot_empty[s]);
                    ++ld;
                }
                return true;
            };
            for (int u = 0; ok && u < n; ++u) {
                // X = R0 . s0^T (and Y = R1 . s1^T)
                ok = product(kColX, r0d);
                if (ok && kMode != kDV) ok = product(kColY, r1d);
                if (!ok) break;
                mma_commit_warp(&st->x_full);
                if (!mbar_wait_warp(&st->op_ready, u & 1, wctx, 212)) break;
                tc_fence_after();
                // acc[:, 128 g .. 128 g + 127] += op . (boxes 2g, 2g+1 of the
                // streamed tile), A = op from TMEM (16-bit, 128 columns of
                // K packed into TMEM columns 0-31 and 64-95)
#pragma unroll 1
                for (int g = 0; g < 2 && ok; ++g) {
                    const int s0 = ld % kSlots, s1 = (ld + 1) % kSlots;
                    if (!mbar_wait_warp(&st->slot_full[s0], (ld / kSlots) & 1, wctx, 213) ||
                        !mbar_wait_warp(&st->slot_full[s1], ((ld + 1) / kSlots) & 1, wctx, 214)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bd = ring_mn + (uint64_t)(s0 * kSlotUnits);
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk)
                        mma_ts_warp(tmem + kColAcc + g * 128, tmem + kColX + (kk / 4) * 64 + (kk % 4) * 8,
                                    desc_add(bd, kk * 16 * 128), idesc_acc, (u > 0 || kk > 0) ? 1u : 0u);
                    mma_commit_warp(&st->slot_empty[s0]);
                    mma_commit_warp(&st->slot_empty[s1]);
                    ld += 2;
                }
            }
            mma_commit_warp(&st->acc_done);
            mma_commit_warp(&st->teardown);
            mbar_wait_warp(&st->teardown, 0, wctx, 215);
        }
    } else {
        // ------------------------------------------------------------ compute
        const int quarter = warp & 3;
        const int half = warp >> 2;  // columns [64 half, 64 half + 64)
        const int r = quarter * 32 + lane;
        const int rabs = own0 + r;  // key row (dV, dK) or query row (dQ)
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const float sl2 = p.scale_log2;
        bool ok = true;
        // dQ pass: this row's -LSE (log2 units; -inf for a row that sees no
        // key, so P = 0) and -delta
        float row_nlse = -INFINITY, row_ndelta = 0.f;
        if (!kKeyRows && rabs < p.N) {
            const float lv = p.lse[(size_t)bh * p.N + rabs];
            row_nlse = (lv == -INFINITY) ? -INFINITY : -(lv * kLog2e);
            row_ndelta = -p.delta[(size_t)bh * p.N + rabs];
        }
        const bool key_ok = rabs < L;  // dV, dK: the key row is not padding
        // dV, dK: each column half stages its 64 columns' -LSE (rows r < 64)
        // and -delta (rows r >= 64), two buffers by step parity
        const int col = 64 * half + (r & 63);
        const bool stage_lse = r < 64;
        for (int u = 0; u < n; ++u) {
            const int other0 = sched.tile(u) * kTile;  // first column's query (dV, dK) or key (dQ)
            const int lbuf = (u & 1) * kTile;
            if (kKeyRows) {
                const int qi = other0 + col;
                if (stage_lse) {
                    const float lv = (qi < p.N) ? p.lse[(size_t)bh * p.N + qi] : -INFINITY;
                    sNegLse[lbuf + col] = (lv == -INFINITY) ? -INFINITY : -(lv * kLog2e);
                } else {
                    sNegDelta[lbuf + col] = (qi < p.N) ? -p.delta[(size_t)bh * p.N + qi] : 0.f;
                }
                mbar_arrive_warp(&st->col_ready[half]);
                if (!mbar_wait_warp(&st->col_ready[half], u & 1, wctx, 220)) {
                    ok = false;
                    break;
                }
            }
            if (!mbar_wait_warp(&st->x_full, u & 1, wctx, 221)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // visible columns of this row form [cmin, cmax)
            int cmin = 0, cmax;
            if (kKeyRows) {
                if (p.causal) cmin = max(0, rabs - other0);
                cmax = key_ok ? min(kTile, p.N - other0) : 0;
            } else {
                cmax = min(kTile, L - other0);
                if (p.causal) cmax = min(cmax, rabs - other0 + 1);
                if (rabs >= p.N) cmax = 0;
            }
#pragma unroll 1
            for (int ch = 0; ch < 2; ++ch) {
                const int cb = half * 64 + ch * 32;
                uint32_t xr[32], yr[32];
                tmem_ld32(tmem + lane_base + kColX + cb, xr);
                if (kMode != kDV) tmem_ld32(tmem + lane_base + kColY + cb, yr);
                tmem_ld_wait();
                reg_fence(xr);
                if (kMode != kDV) reg_fence(yr);
                // keep bits of the 32 columns (bit x = column cb + x)
                uint32_t keep = 0xffffffffu;
                if (p.dropout) {
                    keep = 0;
                    if (kKeyRows) {
                        // lane (4a + w) draws the bits of keys 4a..4a+3 for
                        // query cb + 4g + w; the group of 4 lanes exchanges them
#pragma unroll
                        for (int g = 0; g < 8; ++g) {
                            const int qi = other0 + cb + 4 * g + (lane & 3);
                            const uint32_t bits = keep_bits4(p.seed, p.drop_thr, b, h, qi, rabs >> 2);
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const uint32_t v = __shfl_sync(0xffffffffu, bits, (lane & ~3) | q);
                                keep |= ((v >> (lane & 3)) & 1u) << (4 * g + q);
                            }
                        }
                    } else {
#pragma unroll
                        for (int g = 0; g < 8; ++g)
                            keep |= keep_bits4(p.seed, p.drop_thr, b, h, rabs, (other0 + cb) / 4 + g) << (4 * g);
                    }
                }
                uint32_t pk[16];
#pragma unroll
                for (int x = 0; x < 32; x += 2) {
                    float e[2], outv[2];
#pragma unroll
                    for (int y = 0; y < 2; ++y) {
                        const int c = cb + x + y;
                        const bool vis = c >= cmin && c < cmax;
                        const float nl = kKeyRows ? sNegLse[lbuf + c] : row_nlse;
                        e[y] = vis ? ex2_approx(fmaf(__uint_as_float(xr[x + y]), sl2, nl)) : 0.f;
                        const float z = ((keep >> (x + y)) & 1u) ? p.keep_scale : 0.f;
                        if (kMode == kDV) {
                            outv[y] = p.dropout ? e[y] * z : e[y];  // P^ = P Z/(1-p)
                        } else {
                            // dS = P (dP Z/(1-p) - delta)
                            const float nd = kKeyRows ? sNegDelta[lbuf + c] : row_ndelta;
                            const float dpv = p.dropout ? __uint_as_float(yr[x + y]) * z : __uint_as_float(yr[x + y]);
                            outv[y] = e[y] * (dpv + nd);
                        }
                    }
                    pk[x / 2] = Elem16<T>::pack2(outv[0], outv[1]);
                }
                // 32 values -> 16 columns inside the 64 this warp half has read
                tmem_st16(tmem + lane_base + kColX + half * 64 + ch * 16, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive_warp(&st->op_ready);
        }
        // epilogue: out = mul * acc; each warp half writes 128 of the 256 columns
        T* out = static_cast<T*>(p.out) + ((size_t)bh * p.N) * D;
        const float mul = (kMode == kDV) ? 1.f : p.scale;
        const bool have = ok && n > 0 && mbar_wait_warp(&st->acc_done, 0, wctx, 222);
        if (have) tc_fence_after();
        // ok and have are warp-uniform: tcgen05.ld is a warp-collective
        // instruction, so every lane loads and only the stores test the row
        if (ok) {
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                const int c0 = half * 128 + c * 32;
                uint32_t ar[32];
                if (have) {
                    tmem_ld32(tmem + lane_base + kColAcc + c0, ar);
                    tmem_ld_wait();
                    reg_fence(ar);
                } else {
#pragma unroll
                    for (int x = 0; x < 32; ++x) ar[x] = 0u;
                }
                if (rabs >= p.N) continue;
                uint4* dst = reinterpret_cast<uint4*>(out + (size_t)rabs * D + c0);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    uint4 w4;
                    w4.x = Elem16<T>::pack2(__uint_as_float(ar[8 * v + 0]) * mul, __uint_as_float(ar[8 * v + 1]) * mul);
                    w4.y = Elem16<T>::pack2(__uint_as_float(ar[8 * v + 2]) * mul, __uint_as_float(ar[8 * v + 3]) * mul);
                    w4.z = Elem16<T>::pack2(__uint_as_float(ar[8 * v + 4]) * mul, __uint_as_float(ar[8 * v + 5]) * mul);
                    w4.w = Elem16<T>::pack2(__uint_as_float(ar[8 * v + 6]) * mul, __uint_as_float(ar[8 * v + 7]) * mul);
                    dst[v] = w4;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem, 512);
}

template <typename T, int kMode, bool kMask>
int launch_pass(const Problem& pr, const CUtensorMap& r0, const CUtensorMap& r1, const CUtensorMap& s0,
                const CUtensorMap& s1, void* out) {
    using Cfg = Bwd256Cfg<kMode>;
    auto kernel = bwd256_kernel<T, kMode, kMask>;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem) != cudaSuccess)
            return FA_ERR_CUDA;
        attr_set = true;
    }
    Bwd256Params p{};
    p.lse = pr.lse;
    p.delta = pr.delta;
    p.out = out;
    p.block_mask = pr.block_mask;
    p.kv_len = pr.kv_len;
    p.status = pr.status;
    p.H = pr.H;
    p.N = pr.N;
    p.nb = pr.nb;
    p.scale = pr.scale;
    p.scale_log2 = pr.scale * kLog2e;
    p.keep_scale = 1.0f / (1.0f - pr.dropout_p);
    p.drop_thr = pr.drop_threshold;
    p.dropout = pr.dropout_p > 0.f;
    p.causal = pr.causal;
    p.seed = pr.seed;
    dim3 grid(pr.B * pr.H, (pr.N + kTile - 1) / kTile);
    kernel<<<grid, kThreads, Cfg::kSmem, pr.stream>>>(r0, r1, s0, s1, p);
    note_launches(1);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        if (std::getenv("FA_DEBUG")) std::fprintf(stderr, "fa: bwd256 launch: %s\n", cudaGetErrorString(e));
        return FA_ERR_CUDA;
    }
    return FA_OK;
}

template <typename T, bool kMask>
int launch_bwd256_t(const Problem& pr) {
    constexpr CUtensorMapDataType tt = Elem16<T>::kTmaType;
    const int BH = pr.B * pr.H;
    CUtensorMap tq, tk, tv, tdo;
    if (!make_tmap16(&tq, pr.q, BH, pr.N, D, kTile, tt) || !make_tmap16(&tk, pr.k, BH, pr.N, D, kTile, tt) ||
        !make_tmap16(&tv, pr.v, BH, pr.N, D, kTile, tt) || !make_tmap16(&tdo, pr.dO, BH, pr.N, D, kTile, tt))
        return FA_ERR_CUDA;
    // delta_i = sum_c dO_ic O_ic, then the three passes
    if (launch_bwd_preprocess(pr) != cudaSuccess) return FA_ERR_CUDA;
    record_main_start(pr.stream);
    int rc = launch_pass<T, kDV, kMask>(pr, tk, tk, tq, tdo, pr.dv);
    if (rc == FA_OK) rc = launch_pass<T, kDK, kMask>(pr, tk, tv, tq, tdo, pr.dk);
    if (rc == FA_OK) rc = launch_pass<T, kDQ, kMask>(pr, tq, tdo, tk, tv, pr.dq);
    record_main_stop(pr.stream);
    return rc;
}

}  // namespace

int launch_bwd256_tc(const Problem& p) {
    if (p.dtype == FA_FP16) return p.block_mask ? launch_bwd256_t<__half, true>(p) : launch_bwd256_t<__half, false>(p);
    if (p.dtype == FA_BF16)
        return p.block_mask ? launch_bwd256_t<__nv_bfloat16, true>(p) : launch_bwd256_t<__nv_bfloat16, false>(p);
    return FA_ERR_UNSUPPORTED;
}

}  // namespace fa
