// Forward attention on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// One CTA computes two 128-row query tiles of one (batch, head) and walks the
// key/value tiles K_j, V_j (128 keys each) that are not masked out, following
// the per-block update of "FlashAttention: Fast and Memory-Efficient Exact
// Attention with IO-Awareness" (section "Metode", steps 1-4): S_ij = Q_i K_j^T,
// running row max m and row sum l, and O_i <- e^{m_old - m_new} O_i +
// P~_ij V_j, with the division by l deferred to the end (FlashAttention-2
// section of the "Flash Attention" guide). Fully masked tiles are skipped
// (causal future, key padding, zero blocks of the block-sparse mask,
// "Ekstensi: Block-Sparse FlashAttention"). Warp specialisation follows the
// FlashAttention-3 section of the guide and the two-tile ping-pong its
// FlashAttention-4 section.
//
// The running max is only raised when a row's new maximum exceeds the one
// in use by more than 2^8 (log2 units); between raises P <= 2^8, which fp32
// accumulation holds exactly enough, and the final O/l and LSE use the same
// m, so the result is unchanged while most O rescales are skipped.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>

#include <cuda.h>
#include <cuda_bf16.h>

#include "fa_device.cuh"
#include "fa_internal.h"
#include "fa_sm103.cuh"

namespace fa {
namespace {

using namespace sm103;

constexpr int kBlockM = 128;  // query rows per CTA
constexpr int kBlockN = 128;  // keys per tile
constexpr int kSoftmaxThreads = 128;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct FwdParams {
    float* lse;
    void* o;
    const uint8_t* block_mask;
    const int32_t* kv_len;
    int* status;
    int H, N, nb, n_qtiles;
    // split-KV: the key tiles of each pair of query tiles are cut into
    // n_splits ranges, one CTA each, which write the partial O (fp32,
    // normalised over their range) and LSE to o_part / lse_part
    // ([n_splits][B*H][N][D] and [n_splits][B*H][N]); 1 and null otherwise
    int n_splits;
    float* o_part;
    float* lse_part;
    int BH;
    float scale_log2;
    float out_scale;  // 1/(1-p)
    uint32_t drop_thr;
    int dropout;
    int causal;
    uint64_t seed;
};

// ---------------------------------------------------------------------------
// Two query tiles per CTA (256 rows), one softmax warpgroup per tile. The MMA
// warp issues, per step u,
//     P_0(u) V, S_0(u+1), P_1(u) V, S_1(u+1)
// so the softmax of one tile runs while the tensor core works on the other
// (the ping-pong of the FlashAttention-4 design). Without a block mask tile t
// visits key tiles 0 .. n_t - 1 and both tiles share one K/V stream (K_u,
// V_u); with one (kSplit) each tile visits the tiles of its own list and the
// producer loads them in the order of use.
// Roles (384 threads, three warpgroups): warps 0-3 softmax of tile 0, warps
// 4-7 softmax of tile 1, warp 8 TMA producer, warp 9 MMA issuer (all 32 lanes
// run its loop, one elected lane issues), warps 10-11 idle. setmaxnreg moves
// registers from the third warpgroup to the softmax warpgroups (208 each
// thread against 80; launched at 168), which removes the softmax spills.
// ---------------------------------------------------------------------------
constexpr int kThreadsPP = 384;
constexpr int kSoftmaxRegs = 208, kIssueRegs = 80;
// setmaxnreg.inc takes registers from the CTA's launch allocation (384
// threads at 168, the most a 384-thread launch gets) and waits until they
// are free, so the budgets must fit in it
static_assert(256 * kSoftmaxRegs + 128 * kIssueRegs <= kThreadsPP * 168, "register budgets above the launch");

template <int D>
struct FwdPPCfg {
    static constexpr int kStages = (D == 128) ? 4 : 8;
    static constexpr int kTileBytes = kBlockN * D * 2;
    static constexpr int kQBytes = kBlockM * D * 2;  // per query tile
    static constexpr int kBoxes = D / 64;
    static constexpr int kBoxBytes = kBlockN * 128;
    // + the two query tiles' lists of visible key tiles (block masks)
    static constexpr int kSmem = 1024 + 2 * kQBytes + kStages * kTileBytes + 256 + 2 * kMaskListCap * 2;
    static constexpr uint32_t kTmemCols = 512;
    // S_t at columns 128 t, O_t at 256 + D t
};

struct SharedPP {
    uint64_t kv_full[8];
    uint64_t kv_empty[8];
    uint64_t q_full;
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t o_final[2];
    uint64_t o_staged[2];  // every softmax warp of tile t has written its rows of O over Q_t
    uint64_t teardown;
    uint32_t tmem_base;
    int abort_flag;
    int n_list[2];  // kSplit: visible key tiles of each query tile
};
static_assert(sizeof(SharedPP) <= 256, "barrier block");

template <typename T, int D, bool kSplit, bool kPartial>
__global__ void __launch_bounds__(kThreadsPP, 1)
    fwd_pp_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const FwdParams p) {
    using Cfg = FwdPPCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;  // tile t at t * kQBytes
    uint8_t* sKV = smem + 2 * Cfg::kQBytes;
    SharedPP* st = reinterpret_cast<SharedPP*>(sKV + Cfg::kStages * Cfg::kTileBytes);
    uint16_t* sList = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(st) + 256);  // [2][kMaskListCap]

    // launched with programmatic stream serialization: wait for the kernel
    // ahead (it may have written Q, K, V, kv_len or the mask), then let the
    // next one (the backward's preprocess) start launching behind this grid
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // grid (B*H, pairs x splits): the hardware dispatches x fastest, so every
    // head's heaviest pair (causal) goes out before any lighter one
    const int bh = blockIdx.x;
    const int b = bh / p.H, h = bh % p.H;
    const int n_pairs = (p.n_qtiles + 1) / 2;
    // kPartial (split-KV): blockIdx.y = rank * n_splits + split
    const int rank = kPartial ? (int)blockIdx.y / p.n_splits : (int)blockIdx.y;
    const int split = kPartial ? (int)blockIdx.y % p.n_splits : 0;
    const int pair = p.causal ? (n_pairs - 1 - rank) : rank;
    const int L = p.kv_len ? min(max(p.kv_len[b], 0), p.N) : p.N;
    const int nkt = (L + kBlockN - 1) / kBlockN;  // key tiles with a visible key
    // key tiles visited by query tile t of this CTA (0 if the tile is past N)
    int n_t[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int qt = 2 * pair + t;
        n_t[t] = (qt < p.n_qtiles) ? (p.causal ? min(nkt, qt + 1) : nkt) : 0;
    }
    // this CTA's range [kb, ke) of the pair's key tiles (all of them unless
    // split-KV); tile t visits key tiles kb .. kb + n_t - 1
    int kb = 0, ke = 1 << 30;
    if constexpr (kPartial) {
        const int chunk = (max(n_t[0], n_t[1]) + p.n_splits - 1) / p.n_splits;
        kb = split * chunk;
        ke = kb + chunk;
#pragma unroll
        for (int t = 0; t < 2; ++t) n_t[t] = max(0, min(n_t[t], ke) - kb);
    }
    WaitCtx wctx{&st->abort_flag, p.status};
    // kSplit (block mask): each query tile walks its own list of visible key
    // tiles, built here by warp 0 from its mask row (coalesced loads and a
    // ballot), and the K/V tiles of the two lists are loaded one after the
    // other in the order the MMA warp uses them
    if (kSplit && warp == 0) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int qt = 2 * pair + t;
            int e = (qt < p.n_qtiles) ? nkt : 0;
            if (p.causal) e = min(e, qt + 1);
            e = min(e, ke);
            const int cnt =
                warp_list_visible(p.block_mask + (size_t)qt * p.nb, 1, kb, e, sList + t * kMaskListCap, lane);
            if (lane == 0) st->n_list[t] = cnt;
        }
    }

    if (tid == 0) {
        for (int s = 0; s < Cfg::kStages; ++s) {
            mbar_init(&st->kv_full[s], 1);
            mbar_init(&st->kv_empty[s], 1);
        }
        mbar_init(&st->q_full, 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(&st->s_full[t], 1);
            mbar_init(&st->p_full[t], kSoftmaxThreads / 32);
            mbar_init(&st->o_final[t], 1);
            mbar_init(&st->o_staged[t], kSoftmaxThreads / 32);  // the 4 softmax warps of tile t
        }
        mbar_init(&st->teardown, 1);
        st->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(&st->tmem_base, Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = st->tmem_base;
    if constexpr (kSplit) {
        n_t[0] = st->n_list[0];
        n_t[1] = st->n_list[1];
    }
    const int n_max = max(n_t[0], n_t[1]);
    const uint16_t* list0 = sList;
    const uint16_t* list1 = sList + kMaskListCap;

    if (warp == 8) {
        // ------------------------------------------------------------ producer
        regs_dec<kIssueRegs>();
        if (lane == 0 && n_max > 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            const int nq = (n_t[1] > 0) ? 2 : 1;
            mbar_arrive_expect_tx(&st->q_full, nq * Cfg::kQBytes);
            for (int t = 0; t < nq; ++t)
#pragma unroll
                for (int x = 0; x < Cfg::kBoxes; ++x)
                    tma_load_3d(sQ + t * Cfg::kQBytes + x * Cfg::kBoxBytes, &tm_q, &st->q_full, x * 64,
                                (2 * pair + t) * kBlockM, bh);
            int t = 0;  // load counter
            if constexpr (!kSplit) {
                // load index 2u = K_u, 2u + 1 = V_u
                for (; t < 2 * n_max; ++t) {
                    const int s = t % Cfg::kStages;
                    const uint32_t ph = (t / Cfg::kStages) & 1;
                    if (!mbar_wait(&st->kv_empty[s], ph ^ 1, wctx, 61)) break;
                    mbar_arrive_expect_tx(&st->kv_full[s], Cfg::kTileBytes);
                    uint8_t* dst = sKV + s * Cfg::kTileBytes;
                    const CUtensorMap* map = (t & 1) ? &tm_v : &tm_k;
#pragma unroll
                    for (int x = 0; x < Cfg::kBoxes; ++x)
                        tma_load_3d(dst + x * Cfg::kBoxBytes, map, &st->kv_full[s], x * 64, (kb + (t >> 1)) * kBlockN,
                                    bh);
                }
            } else {
                // K of S_0(0), K of S_1(0), then per step u and tile t: V of
                // P_t V, K of the tile's next S
                auto load = [&](const CUtensorMap* map, int j) -> bool {
                    const int s = t % Cfg::kStages;
                    const uint32_t ph = (t / Cfg::kStages) & 1;
                    if (!mbar_wait(&st->kv_empty[s], ph ^ 1, wctx, 61)) return false;
                    mbar_arrive_expect_tx(&st->kv_full[s], Cfg::kTileBytes);
                    uint8_t* dst = sKV + s * Cfg::kTileBytes;
#pragma unroll
                    for (int x = 0; x < Cfg::kBoxes; ++x)
                        tma_load_3d(dst + x * Cfg::kBoxBytes, map, &st->kv_full[s], x * 64, j * kBlockN, bh);
                    ++t;
                    return true;
                };
                bool okp = true;
                if (n_t[0] > 0) okp = load(&tm_k, list0[0]);
                if (okp && n_t[1] > 0) okp = load(&tm_k, list1[0]);
                for (int u = 0; okp && u < n_max; ++u) {
                    if (u < n_t[0]) {
                        okp = load(&tm_v, list0[u]);
                        if (okp && u + 1 < n_t[0]) okp = load(&tm_k, list0[u + 1]);
                    }
                    if (okp && u < n_t[1]) {
                        okp = load(&tm_v, list1[u]);
                        if (okp && u + 1 < n_t[1]) okp = load(&tm_k, list1[u + 1]);
                    }
                }
            }
            // drain: the last load issued into each stage has landed
            for (int l = max(0, t - Cfg::kStages); l < t; ++l)
                mbar_wait(&st->kv_full[l % Cfg::kStages], (l / Cfg::kStages) & 1, wctx, 62);
            mbar_wait(&st->q_full, 0, wctx, 63);
        }
    } else if (warp == 10 || warp == 11) {
        regs_dec<kIssueRegs>();  // idle: the rest of the producer / MMA warpgroup
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        regs_dec<kIssueRegs>();
        if (n_max > 0) {
            constexpr uint32_t idesc_s = idesc_f32acc(Elem16<T>::kFmt, kBlockM, kBlockN, 0, 0);
            constexpr uint32_t idesc_o = idesc_f32acc(Elem16<T>::kFmt, kBlockM, D, 0, 1);
            const uint32_t kv_base = smem_u32(sKV);
            const uint64_t qd0 = smem_desc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t qd1 = smem_desc_sw128(smem_u32(sQ + Cfg::kQBytes), 16, 1024);
            bool ok = mbar_wait_warp(&st->q_full, 0, wctx, 70);
            tc_fence_after();
            // Straight-line issue code with every counter in registers, run
            // by the whole warp (one elected lane issues): the issuing path
            // has about 64 cycles per MMA to spare.
            // Each load index is waited on once, before its first use.
            const int c0 = n_t[0], c1 = n_t[1];
            const uint64_t kvd_k = smem_desc_sw128(kv_base, 16, 1024);              // K tiles, K-major
            const uint64_t kvd_v = smem_desc_sw128(kv_base, Cfg::kBoxBytes, 1024);  // V tiles, MN-major
            constexpr uint32_t kStageUnits = Cfg::kTileBytes >> 4;
            if constexpr (!kSplit) {
            // S_t(0) = Q_t K_0^T
            if (ok) {
                ok = mbar_wait_warp(&st->kv_full[0], 0, wctx, 71);
                tc_fence_after();
            }
            if (ok) {
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if ((t ? c1 : c0) == 0) continue;
                    const uint64_t qd = t ? qd1 : qd0;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk / 4) * Cfg::kBoxBytes + (kk % 4) * 32;
                        mma_ss_warp(tmem + t * 128, desc_add(qd, off), desc_add(kvd_k, off), idesc_s, kk > 0);
                    }
                    mma_commit_warp(&st->s_full[t]);
                }
                mma_commit_warp(&st->kv_empty[0]);
            }
            for (int u = 0; ok && u < n_max; ++u) {
                const int lv = 2 * u + 1, lk = 2 * u + 2;  // load indices of V_u and K_{u+1}
                const int sv = lv % Cfg::kStages, sk = lk % Cfg::kStages;
                const uint64_t vd = kvd_v + (uint64_t)(sv * kStageUnits);
                const uint64_t kd = kvd_k + (uint64_t)(sk * kStageUnits);
                const bool need_k = (u + 1 < c0) || (u + 1 < c1);
                bool v_ready = false, k_ready = false;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const int ct = t ? c1 : c0;
                    if (u >= ct) continue;
                    // P_t(u) V_u
                    if (!mbar_wait_warp(&st->p_full[t], u & 1, wctx, 72)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (!v_ready) {
                        if (!mbar_wait_warp(&st->kv_full[sv], (lv / Cfg::kStages) & 1, wctx, 74)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        v_ready = true;
                    }
#pragma unroll
                    for (int kk = 0; kk < kBlockN / 16; ++kk)
                        mma_ts_warp(tmem + 256 + t * D, tmem + t * 128 + kk * 8, desc_add(vd, kk * 16 * 128), idesc_o,
                               (u > 0 || kk > 0) ? 1u : 0u);
                    if (u + 1 == ct) mma_commit_warp(&st->o_final[t]);
                    // S_t(u+1) = Q_t K_{u+1}^T over the S/P columns just read
                    if (u + 1 < ct) {
                        if (!k_ready) {
                            if (!mbar_wait_warp(&st->kv_full[sk], (lk / Cfg::kStages) & 1, wctx, 75)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            k_ready = true;
                        }
                        const uint64_t qd = t ? qd1 : qd0;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = (kk / 4) * Cfg::kBoxBytes + (kk % 4) * 32;
                            mma_ss_warp(tmem + t * 128, desc_add(qd, off), desc_add(kd, off), idesc_s, kk > 0);
                        }
                        mma_commit_warp(&st->s_full[t]);
                    }
                }
                if (!ok) break;
                // V_u and K_{u+1} are released after their last MMA
                mma_commit_warp(&st->kv_empty[sv]);
                if (need_k) mma_commit_warp(&st->kv_empty[sk]);
            }
            } else {
            int ld = 0;  // next load to use, in the producer's order
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (!ok || (t ? c1 : c0) == 0) continue;
                const int s = ld % Cfg::kStages;
                ok = mbar_wait_warp(&st->kv_full[s], (ld / Cfg::kStages) & 1, wctx, 71);
                if (!ok) break;
                tc_fence_after();
                const uint64_t qd = t ? qd1 : qd0;
                const uint64_t kd = kvd_k + (uint64_t)(s * kStageUnits);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk / 4) * Cfg::kBoxBytes + (kk % 4) * 32;
                    mma_ss_warp(tmem + t * 128, desc_add(qd, off), desc_add(kd, off), idesc_s, kk > 0);
                }
                mma_commit_warp(&st->s_full[t]);
                mma_commit_warp(&st->kv_empty[s]);
                ++ld;
            }
            for (int u = 0; ok && u < n_max; ++u) {
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const int ct = t ? c1 : c0;
                    if (u >= ct) continue;
                    // P_t(u) V
                    if (!mbar_wait_warp(&st->p_full[t], u & 1, wctx, 72)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    int s = ld % Cfg::kStages;
                    if (!mbar_wait_warp(&st->kv_full[s], (ld / Cfg::kStages) & 1, wctx, 74)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t vd = kvd_v + (uint64_t)(s * kStageUnits);
#pragma unroll
                    for (int kk = 0; kk < kBlockN / 16; ++kk)
                        mma_ts_warp(tmem + 256 + t * D, tmem + t * 128 + kk * 8, desc_add(vd, kk * 16 * 128), idesc_o,
                                    (u > 0 || kk > 0) ? 1u : 0u);
                    mma_commit_warp(&st->kv_empty[s]);
                    ++ld;
                    if (u + 1 == ct) mma_commit_warp(&st->o_final[t]);
                    if (u + 1 < ct) {
                        // S_t of the tile's next key tile over the S/P columns just read
                        s = ld % Cfg::kStages;
                        if (!mbar_wait_warp(&st->kv_full[s], (ld / Cfg::kStages) & 1, wctx, 75)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t qd = t ? qd1 : qd0;
                        const uint64_t kd = kvd_k + (uint64_t)(s * kStageUnits);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = (kk / 4) * Cfg::kBoxBytes + (kk % 4) * 32;
                            mma_ss_warp(tmem + t * 128, desc_add(qd, off), desc_add(kd, off), idesc_s, kk > 0);
                        }
                        mma_commit_warp(&st->s_full[t]);
                        mma_commit_warp(&st->kv_empty[s]);
                        ++ld;
                    }
                }
            }
            }
            mma_commit_warp(&st->teardown);
            mbar_wait_warp(&st->teardown, 0, wctx, 73);
        }
    } else {
        // ------------------------------------------------------------ softmax
        regs_inc<kSoftmaxRegs>();
        const int t = warp >> 2;  // query tile of this warpgroup
        const int r = tid & 127;
        const int i = (2 * pair + t) * kBlockM + r;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t sbase = tmem + lane_base + t * 128;
        const uint32_t obase = tmem + lane_base + 256 + t * D;
        const int n = n_t[t];
        float m = -INFINITY;
        float l = 0.f;
        bool ok = true;
        // key tile of step u: u itself, or the u-th entry of this tile's list
        const uint16_t* my_list = t ? list1 : list0;
        for (int u = 0; u < n; ++u) {
            const int ktile = kSplit ? (int)my_list[u] : kb + u;
            // dropout keep bits of this row's 128 keys (bit x of keep[c] is
            // key 32c + x), drawn before S arrives
            uint32_t keep[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
            if (p.dropout) {
#pragma unroll 8
                for (int g = 0; g < 32; ++g) {
                    const uint32_t bits = keep_bits4(p.seed, p.drop_thr, b, h, i, ktile * (kBlockN / 4) + g);
                    if (g == 0) keep[0] = keep[1] = keep[2] = keep[3] = 0;
                    const uint32_t sh = bits << (4 * (g & 7));
                    if ((g >> 3) == 0) keep[0] |= sh;
                    else if ((g >> 3) == 1) keep[1] |= sh;
                    else if ((g >> 3) == 2) keep[2] |= sh;
                    else keep[3] |= sh;
                }
            }
            if (!mbar_wait_warp(&st->s_full[t], u & 1, wctx, 80)) {
                ok = false;
                break;
            }
            // S_t(u) was issued after P_t(u-1) V: O_t is complete here
            tc_fence_after();
            const int k0 = ktile * kBlockN;
            int lim = min(kBlockN, L - k0);
            if (p.causal) lim = min(lim, i - k0 + 1);
            const bool full = lim >= kBlockN;
            // the whole row of S in registers, one TMEM wait
            uint32_t sr[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(sbase + c * 32, sr[c]);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 4; ++c) reg_fence(sr[c]);
            if (!full) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int x = 0; x < 32; ++x)
                        if (c * 32 + x >= lim) sr[c][x] = __float_as_uint(-INFINITY);
            }
            float pm[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) pm[x] = -INFINITY;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int x = 0; x < 32; x += 2)
                    pm[(x >> 1) & 7] =
                        fmax3(pm[(x >> 1) & 7], __uint_as_float(sr[c][x]), __uint_as_float(sr[c][x + 1]));
            pm[0] = fmax3(pm[0], pm[1], pm[2]);
            pm[3] = fmax3(pm[3], pm[4], pm[5]);
            pm[6] = fmaxf(pm[6], pm[7]);
            pm[0] = fmax3(pm[0], pm[3], pm[6]);
            const float mt = pm[0] * p.scale_log2;
            const bool raise = mt > m + kRescaleThreshold;
            if (__any_sync(0xffffffffu, raise) && u > 0) {
                const float alpha = raise ? ex2_approx(m - mt) : 1.f;
#pragma unroll 1
                for (int c = 0; c < D / 8; ++c) {
                    uint32_t orr[8];
                    tmem_ld8(obase + c * 8, orr);
                    tmem_ld_wait();
                    reg_fence8(orr);
#pragma unroll
                    for (int x = 0; x < 8; ++x) orr[x] = __float_as_uint(__uint_as_float(orr[x]) * alpha);
                    tmem_st8(obase + c * 8, orr);
                }
                if (raise) l *= alpha;
            }
            if (raise) m = mt;
            const float nmref = (m == -INFINITY) ? 0.f : -m;
            const float sl2 = p.scale_log2;
            // row-sum partials, four pairs
            float ps[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) ps[x] = 0.f;
            // exponentials packed in place: pair x/2 overwrites word x/2,
            // which has already been consumed; P chunk c lands in columns
            // 16c..16c+15, already read. The sum takes every exponential,
            // the dropout mask only what goes to P.
            if (!p.dropout) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
#pragma unroll
                    for (int x = 0; x < 32; x += 2) {
                        float a0, a1;
                        ffma2(a0, a1, __uint_as_float(sr[c][x]), __uint_as_float(sr[c][x + 1]), sl2, sl2, nmref, nmref);
                        const float e0 = ex2_approx(a0), e1 = ex2_approx(a1);
                        const int k = (x >> 1) & 3;
                        fadd2(ps[2 * k], ps[2 * k + 1], ps[2 * k], ps[2 * k + 1], e0, e1);
                        sr[c][x >> 1] = Elem16<T>::pack2(e0, e1);
                    }
                    tmem_st16(sbase + c * 16, *reinterpret_cast<const uint32_t(*)[16]>(&sr[c][0]));
                }
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
#pragma unroll
                    for (int x = 0; x < 32; x += 2) {
                        float a0, a1;
                        ffma2(a0, a1, __uint_as_float(sr[c][x]), __uint_as_float(sr[c][x + 1]), sl2, sl2, nmref, nmref);
                        const float e0 = ex2_approx(a0), e1 = ex2_approx(a1);
                        const int k = (x >> 1) & 3;
                        fadd2(ps[2 * k], ps[2 * k + 1], ps[2 * k], ps[2 * k + 1], e0, e1);
                        sr[c][x >> 1] =
                            Elem16<T>::pack2(((keep[c] >> x) & 1u) ? e0 : 0.f, ((keep[c] >> (x + 1)) & 1u) ? e1 : 0.f);
                    }
                    tmem_st16(sbase + c * 16, *reinterpret_cast<const uint32_t(*)[16]>(&sr[c][0]));
                }
            }
            fadd2(ps[0], ps[1], ps[0], ps[1], ps[4], ps[5]);
            fadd2(ps[2], ps[3], ps[2], ps[3], ps[6], ps[7]);
            fadd2(ps[0], ps[1], ps[0], ps[1], ps[2], ps[3]);
            l += ps[0] + ps[1];
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive_warp(&st->p_full[t]);
        }
        T* O = static_cast<T*>(p.o) + ((size_t)bh * p.N) * D;
        // split-KV partials of this split and head
        const size_t prow = ((size_t)split * p.BH + bh) * p.N;
        if (ok && n > 0) {
            if (mbar_wait_warp(&st->o_final[t], 0, wctx, 81)) {
                tc_fence_after();
                const float inv = (l > 0.f) ? p.out_scale / l : 0.f;
                // 16-bit O: written over Q_t (every product of tile t has
                // completed, its last S before its last P V) as D / 64 boxes of
                // 128 rows x 64 columns, 128-byte swizzled (16-byte chunk c of
                // row r at chunk position c ^ (r & 7)), then stored by the TMA
                // engine: rows past N are outside the tensor and not written.
                // Split-KV partials (fp32) are stored row by row.
                uint8_t* qt_tile = sQ + t * Cfg::kQBytes;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t orr[32];
                    tmem_ld32(obase + c * 32, orr);
                    tmem_ld_wait();
                    reg_fence(orr);
                    if constexpr (kPartial) {
                        if (i < p.N) {
                            float4* dst = reinterpret_cast<float4*>(p.o_part + (prow + i) * D + c * 32);
#pragma unroll
                            for (int v = 0; v < 8; ++v)
                                dst[v] = make_float4(__uint_as_float(orr[4 * v]) * inv, __uint_as_float(orr[4 * v + 1]) * inv,
                                                     __uint_as_float(orr[4 * v + 2]) * inv,
                                                     __uint_as_float(orr[4 * v + 3]) * inv);
                        }
                    } else {
                        uint8_t* row = qt_tile + (c >> 1) * Cfg::kBoxBytes + r * 128;
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint4 w4;
                            w4.x = Elem16<T>::pack2(__uint_as_float(orr[8 * v + 0]) * inv, __uint_as_float(orr[8 * v + 1]) * inv);
                            w4.y = Elem16<T>::pack2(__uint_as_float(orr[8 * v + 2]) * inv, __uint_as_float(orr[8 * v + 3]) * inv);
                            w4.z = Elem16<T>::pack2(__uint_as_float(orr[8 * v + 4]) * inv, __uint_as_float(orr[8 * v + 5]) * inv);
                            w4.w = Elem16<T>::pack2(__uint_as_float(orr[8 * v + 6]) * inv, __uint_as_float(orr[8 * v + 7]) * inv);
                            const int chunk = (c & 1) * 4 + v;
                            *reinterpret_cast<uint4*>(row + ((chunk ^ (r & 7)) << 4)) = w4;
                        }
                    }
                }
                if (i < p.N) {
                    const float lse_i = (l > 0.f) ? (m + __log2f(l)) * kLn2 : -INFINITY;
                    if (kPartial) p.lse_part[prow + i] = lse_i;
                    else p.lse[(size_t)bh * p.N + i] = lse_i;
                }
                if constexpr (!kPartial) {
                    fence_proxy_async_smem();
                    mbar_arrive_warp(&st->o_staged[t]);
                    if ((warp & 3) == 0 && mbar_wait_warp(&st->o_staged[t], 0, wctx, 86) && lane == 0) {
#pragma unroll
                        for (int x = 0; x < Cfg::kBoxes; ++x)
                            tma_store_3d(&tm_o, qt_tile + x * Cfg::kBoxBytes, x * 64, (2 * pair + t) * kBlockM, bh);
                        bulk_commit_group();
                        bulk_wait_all();  // complete before the CTA ends
                    }
                }
            }
        } else if (n == 0 && i < p.N) {
            if (kPartial) {
                float4* dst = reinterpret_cast<float4*>(p.o_part + (prow + i) * D);
#pragma unroll
                for (int v = 0; v < D / 4; ++v) dst[v] = make_float4(0.f, 0.f, 0.f, 0.f);
                p.lse_part[prow + i] = -INFINITY;
            } else {
                uint4 z = make_uint4(0, 0, 0, 0);
                uint4* dst = reinterpret_cast<uint4*>(O + (size_t)i * D);
#pragma unroll
                for (int v = 0; v < D / 8; ++v) dst[v] = z;
                p.lse[(size_t)bh * p.N + i] = -INFINITY;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem, Cfg::kTmemCols);
}

// ---------------------------------------------------------------------------
// Head dim 256: one 128-row query tile per CTA. Two query tiles would need
// 2 x (128 + 256) = 768 TMEM columns; one tile with a double-buffered S needs
// 2 x 128 + 256 = 512, the whole TMEM. S(u) lives in buffer u % 2 (columns
// 128 (u % 2)), O in columns 256-511. The MMA warp issues S(u+1) before
// P(u) V, so the softmax of key tile u+1 runs while the tensor core computes
// P(u) V_u and S(u+2):
//     S(0), S(1), [P(0)] P(0) V_0, S(2), [P(1)] P(1) V_1, S(3), ...
// Because P(u) V may still be running when the softmax of tile u+1 wants to
// rescale O, that rescale (rare: only when the row max rises by more than
// 2^8) first waits for the P(u) V commit.
// Roles (192 threads): warps 0-3 softmax (one thread per query row), warp 4
// TMA producer, warp 5 MMA issuer (all lanes run its loop, one elected lane
// issues). K/V tiles are 64 KB, so the ring has two stages; each load has
// the softmax of one key tile to land in.
// ---------------------------------------------------------------------------
constexpr int kThreads256 = 192;

struct Fwd256Cfg {
    static constexpr int D = 256;
    static constexpr int kStages = 2;
    static constexpr int kTileBytes = kBlockN * D * 2;  // one K or V tile, 64 KB
    static constexpr int kQBytes = kBlockM * D * 2;     // 64 KB
    static constexpr int kBoxes = D / 64;
    static constexpr int kBoxBytes = kBlockN * 128;
    // + the query tile's list of visible key tiles (block masks)
    static constexpr int kSmem = 1024 + kQBytes + kStages * kTileBytes + 256 + kMaskListCap * 2;
};

struct Shared256 {
    uint64_t kv_full[2];
    uint64_t kv_empty[2];
    uint64_t q_full;
    uint64_t s_full[2];  // buffer b: S(u) for u % 2 == b
    uint64_t p_full[2];  // buffer b: P(u) written over S(u)
    uint64_t o_done;     // one commit after every P(u) V
    uint64_t o_final;
    uint64_t teardown;
    uint32_t tmem_base;
    int abort_flag;
    int n_list;
};
static_assert(sizeof(Shared256) <= 256, "barrier block");

template <typename T, bool kSplit, bool kPartial>
__global__ void __launch_bounds__(kThreads256, 1)
    fwd_d256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
    using Cfg = Fwd256Cfg;
    constexpr int D = Cfg::D;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sKV = smem + Cfg::kQBytes;
    Shared256* st = reinterpret_cast<Shared256*>(sKV + Cfg::kStages * Cfg::kTileBytes);
    uint16_t* sList = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(st) + 256);  // [kMaskListCap]

    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // grid (B*H, query tiles x splits), x fastest: every head's heaviest
    // causal tile goes out first
    const int bh = blockIdx.x;
    const int b = bh / p.H, h = bh % p.H;
    const int rank = kPartial ? (int)blockIdx.y / p.n_splits : (int)blockIdx.y;
    const int split = kPartial ? (int)blockIdx.y % p.n_splits : 0;
    const int qt = p.causal ? (p.n_qtiles - 1 - rank) : rank;
    const int L = p.kv_len ? min(max(p.kv_len[b], 0), p.N) : p.N;
    const int nkt = (L + kBlockN - 1) / kBlockN;
    int n = p.causal ? min(nkt, qt + 1) : nkt;
    // this CTA's range [kb, ke) of key tiles (all of them unless split-KV)
    int kb = 0, ke = 1 << 30;
    if constexpr (kPartial) {
        const int chunk = (n + p.n_splits - 1) / p.n_splits;
        kb = split * chunk;
        ke = kb + chunk;
        n = max(0, min(n, ke) - kb);
    }
    WaitCtx wctx{&st->abort_flag, p.status};
    if (kSplit && warp == 0) {
        int e = p.causal ? min(nkt, qt + 1) : nkt;
        e = min(e, ke);
        const int cnt = warp_list_visible(p.block_mask + (size_t)qt * p.nb, 1, kb, e, sList, lane);
        if (lane == 0) st->n_list = cnt;
    }
    if (tid == 0) {
        for (int s = 0; s < Cfg::kStages; ++s) {
            mbar_init(&st->kv_full[s], 1);
            mbar_init(&st->kv_empty[s], 1);
        }
        mbar_init(&st->q_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&st->s_full[s], 1);
            mbar_init(&st->p_full[s], kSoftmaxThreads / 32);
        }
        mbar_init(&st->o_done, 1);
        mbar_init(&st->o_final, 1);
        mbar_init(&st->teardown, 1);
        st->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(&st->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = st->tmem_base;
    if constexpr (kSplit) n = st->n_list;

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        // load order: K(0), K(1), then per step u: V(u), K(u+2)
        if (lane == 0 && n > 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            mbar_arrive_expect_tx(&st->q_full, Cfg::kQBytes);
#pragma unroll
            for (int x = 0; x < Cfg::kBoxes; ++x)
                tma_load_3d(sQ + x * Cfg::kBoxBytes, &tm_q, &st->q_full, x * 64, qt * kBlockM, bh);
            int t = 0;  // load counter
            auto load = [&](const CUtensorMap* map, int u) -> bool {
                const int j = kSplit ? (int)sList[u] : kb + u;
                const int s = t % Cfg::kStages;
                const uint32_t ph = (t / Cfg::kStages) & 1;
                if (!mbar_wait(&st->kv_empty[s], ph ^ 1, wctx, 161)) return false;
                mbar_arrive_expect_tx(&st->kv_full[s], Cfg::kTileBytes);
                uint8_t* dst = sKV + s * Cfg::kTileBytes;
#pragma unroll
                for (int x = 0; x < Cfg::kBoxes; ++x)
                    tma_load_3d(dst + x * Cfg::kBoxBytes, map, &st->kv_full[s], x * 64, j * kBlockN, bh);
                ++t;
                return true;
            };
            bool okp = load(&tm_k, 0);
            if (okp && n > 1) okp = load(&tm_k, 1);
            for (int u = 0; okp && u < n; ++u) {
                okp = load(&tm_v, u);
                if (okp && u + 2 < n) okp = load(&tm_k, u + 2);
            }
            // drain: the last load issued into each stage has landed
            for (int l = max(0, t - Cfg::kStages); l < t; ++l)
                mbar_wait(&st->kv_full[l % Cfg::kStages], (l / Cfg::kStages) & 1, wctx, 162);
            mbar_wait(&st->q_full, 0, wctx, 163);
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (n > 0) {
            constexpr uint32_t idesc_s = idesc_f32acc(Elem16<T>::kFmt, kBlockM, kBlockN, 0, 0);
            constexpr uint32_t idesc_o = idesc_f32acc(Elem16<T>::kFmt, kBlockM, D, 0, 1);
            constexpr uint32_t kStageUnits = Cfg::kTileBytes >> 4;
            const uint32_t kv_base = smem_u32(sKV);
            const uint64_t qd = smem_desc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t kvd_k = smem_desc_sw128(kv_base, 16, 1024);              // K tiles, K-major
            const uint64_t kvd_v = smem_desc_sw128(kv_base, Cfg::kBoxBytes, 1024);  // V tiles, MN-major
            bool ok = mbar_wait_warp(&st->q_full, 0, wctx, 170);
            tc_fence_after();
            int ld = 0;  // next load to use, in the producer's order
            // S(u) = Q K_u^T into buffer u % 2
            auto issue_s = [&](int u) -> bool {
                const int s = ld % Cfg::kStages;
                if (!mbar_wait_warp(&st->kv_full[s], (ld / Cfg::kStages) & 1, wctx, 171)) return false;
                tc_fence_after();
                const uint64_t kd = kvd_k + (uint64_t)(s * kStageUnits);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk / 4) * Cfg::kBoxBytes + (kk % 4) * 32;
                    mma_ss_warp(tmem + (u & 1) * 128, desc_add(qd, off), desc_add(kd, off), idesc_s, kk > 0);
                }
                mma_commit_warp(&st->s_full[u & 1]);
                mma_commit_warp(&st->kv_empty[s]);
                ++ld;
                return true;
            };
            if (ok) ok = issue_s(0);
            if (ok && n > 1) ok = issue_s(1);
            for (int u = 0; ok && u < n; ++u) {
                // O += P(u) V_u, A = P(u) from TMEM
                if (!mbar_wait_warp(&st->p_full[u & 1], (u >> 1) & 1, wctx, 172)) break;
                tc_fence_after();
                const int s = ld % Cfg::kStages;
                if (!mbar_wait_warp(&st->kv_full[s], (ld / Cfg::kStages) & 1, wctx, 174)) break;
                tc_fence_after();
                const uint64_t vd = kvd_v + (uint64_t)(s * kStageUnits);
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk)
                    mma_ts_warp(tmem + 256, tmem + (u & 1) * 128 + kk * 8, desc_add(vd, kk * 16 * 128), idesc_o,
                                (u > 0 || kk > 0) ? 1u : 0u);
                mma_commit_warp(&st->kv_empty[s]);
                ++ld;
                mma_commit_warp(&st->o_done);
                if (u + 1 == n) mma_commit_warp(&st->o_final);
                // S(u+2) over the P(u) columns just read (MMAs run in order)
                if (u + 2 < n) ok = issue_s(u + 2);
            }
            mma_commit_warp(&st->teardown);
            mbar_wait_warp(&st->teardown, 0, wctx, 173);
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int r = tid;  // 0..127
        const int i = qt * kBlockM + r;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const uint32_t obase = tmem + lane_base + 256;
        float m = -INFINITY;
        float l = 0.f;
        bool ok = true;
        for (int u = 0; u < n; ++u) {
            const int ktile = kSplit ? (int)sList[u] : kb + u;
            const uint32_t sbase = tmem + lane_base + (u & 1) * 128;
            uint32_t keep[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
            if (p.dropout) {
#pragma unroll 8
                for (int g = 0; g < 32; ++g) {
                    const uint32_t bits = keep_bits4(p.seed, p.drop_thr, b, h, i, ktile * (kBlockN / 4) + g);
                    if (g == 0) keep[0] = keep[1] = keep[2] = keep[3] = 0;
                    const uint32_t sh = bits << (4 * (g & 7));
                    if ((g >> 3) == 0) keep[0] |= sh;
                    else if ((g >> 3) == 1) keep[1] |= sh;
                    else if ((g >> 3) == 2) keep[2] |= sh;
                    else keep[3] |= sh;
                }
            }
            if (!mbar_wait_warp(&st->s_full[u & 1], (u >> 1) & 1, wctx, 180)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int k0 = ktile * kBlockN;
            int lim = min(kBlockN, L - k0);
            if (p.causal) lim = min(lim, i - k0 + 1);
            const bool full = lim >= kBlockN;
            uint32_t sr[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(sbase + c * 32, sr[c]);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 4; ++c) reg_fence(sr[c]);
            if (!full) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int x = 0; x < 32; ++x)
                        if (c * 32 + x >= lim) sr[c][x] = __float_as_uint(-INFINITY);
            }
            float pm[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) pm[x] = -INFINITY;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int x = 0; x < 32; x += 2)
                    pm[(x >> 1) & 7] =
                        fmax3(pm[(x >> 1) & 7], __uint_as_float(sr[c][x]), __uint_as_float(sr[c][x + 1]));
            pm[0] = fmax3(pm[0], pm[1], pm[2]);
            pm[3] = fmax3(pm[3], pm[4], pm[5]);
            pm[6] = fmaxf(pm[6], pm[7]);
            pm[0] = fmax3(pm[0], pm[3], pm[6]);
            const float mt = pm[0] * p.scale_log2;
            const bool raise = mt > m + kRescaleThreshold;
            if (__any_sync(0xffffffffu, raise) && u > 0) {
                // O must hold P(u-1) V before it is rescaled
                if (!mbar_wait_warp(&st->o_done, (u - 1) & 1, wctx, 181)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float alpha = raise ? ex2_approx(m - mt) : 1.f;
#pragma unroll 1
                for (int c = 0; c < D / 8; ++c) {
                    uint32_t orr[8];
                    tmem_ld8(obase + c * 8, orr);
                    tmem_ld_wait();
                    reg_fence8(orr);
#pragma unroll
                    for (int x = 0; x < 8; ++x) orr[x] = __float_as_uint(__uint_as_float(orr[x]) * alpha);
                    tmem_st8(obase + c * 8, orr);
                }
                if (raise) l *= alpha;
            }
            if (raise) m = mt;
            const float nmref = (m == -INFINITY) ? 0.f : -m;
            const float sl2 = p.scale_log2;
            float ps[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) ps[x] = 0.f;
            // exponentials packed in place (P chunk c in columns 16c..16c+15,
            // already read); the sum takes every exponential, the dropout
            // mask only what goes to P
            if (!p.dropout) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
#pragma unroll
                    for (int x = 0; x < 32; x += 2) {
                        float a0, a1;
                        ffma2(a0, a1, __uint_as_float(sr[c][x]), __uint_as_float(sr[c][x + 1]), sl2, sl2, nmref, nmref);
                        const float e0 = ex2_approx(a0), e1 = ex2_approx(a1);
                        const int k = (x >> 1) & 3;
                        fadd2(ps[2 * k], ps[2 * k + 1], ps[2 * k], ps[2 * k + 1], e0, e1);
                        sr[c][x >> 1] = Elem16<T>::pack2(e0, e1);
                    }
                    tmem_st16(sbase + c * 16, *reinterpret_cast<const uint32_t(*)[16]>(&sr[c][0]));
                }
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
#pragma unroll
                    for (int x = 0; x < 32; x += 2) {
                        float a0, a1;
                        ffma2(a0, a1, __uint_as_float(sr[c][x]), __uint_as_float(sr[c][x + 1]), sl2, sl2, nmref, nmref);
                        const float e0 = ex2_approx(a0), e1 = ex2_approx(a1);
                        const int k = (x >> 1) & 3;
                        fadd2(ps[2 * k], ps[2 * k + 1], ps[2 * k], ps[2 * k + 1], e0, e1);
                        sr[c][x >> 1] =
                            Elem16<T>::pack2(((keep[c] >> x) & 1u) ? e0 : 0.f, ((keep[c] >> (x + 1)) & 1u) ? e1 : 0.f);
                    }
                    tmem_st16(sbase + c * 16, *reinterpret_cast<const uint32_t(*)[16]>(&sr[c][0]));
                }
            }
            fadd2(ps[0], ps[1], ps[0], ps[1], ps[4], ps[5]);
            fadd2(ps[2], ps[3], ps[2], ps[3], ps[6], ps[7]);
            fadd2(ps[0], ps[1], ps[0], ps[1], ps[2], ps[3]);
            l += ps[0] + ps[1];
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive_warp(&st->p_full[u & 1]);
        }
        T* O = static_cast<T*>(p.o) + ((size_t)bh * p.N) * D;
        const size_t prow = ((size_t)split * p.BH + bh) * p.N;  // split-KV partials
        if (ok && n > 0) {
            if (mbar_wait_warp(&st->o_final, 0, wctx, 182)) {
                tc_fence_after();
                const float inv = (l > 0.f) ? p.out_scale / l : 0.f;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t orr[32];
                    tmem_ld32(obase + c * 32, orr);
                    tmem_ld_wait();
                    reg_fence(orr);
                    if (kPartial && i < p.N) {
                        float4* dst = reinterpret_cast<float4*>(p.o_part + (prow + i) * D + c * 32);
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            dst[v] = make_float4(__uint_as_float(orr[4 * v]) * inv, __uint_as_float(orr[4 * v + 1]) * inv,
                                                 __uint_as_float(orr[4 * v + 2]) * inv,
                                                 __uint_as_float(orr[4 * v + 3]) * inv);
                    } else if (i < p.N) {
                        uint4* dst = reinterpret_cast<uint4*>(O + (size_t)i * D + c * 32);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint4 w4;
                            w4.x = Elem16<T>::pack2(__uint_as_float(orr[8 * v + 0]) * inv, __uint_as_float(orr[8 * v + 1]) * inv);
                            w4.y = Elem16<T>::pack2(__uint_as_float(orr[8 * v + 2]) * inv, __uint_as_float(orr[8 * v + 3]) * inv);
                            w4.z = Elem16<T>::pack2(__uint_as_float(orr[8 * v + 4]) * inv, __uint_as_float(orr[8 * v + 5]) * inv);
                            w4.w = Elem16<T>::pack2(__uint_as_float(orr[8 * v + 6]) * inv, __uint_as_float(orr[8 * v + 7]) * inv);
                            dst[v] = w4;
                        }
                    }
                }
                if (i < p.N) {
                    const float lse_i = (l > 0.f) ? (m + __log2f(l)) * kLn2 : -INFINITY;
                    if (kPartial) p.lse_part[prow + i] = lse_i;
                    else p.lse[(size_t)bh * p.N + i] = lse_i;
                }
            }
        } else if (n == 0 && i < p.N) {
            if (kPartial) {
                float4* dst = reinterpret_cast<float4*>(p.o_part + (prow + i) * D);
#pragma unroll 4
                for (int v = 0; v < D / 4; ++v) dst[v] = make_float4(0.f, 0.f, 0.f, 0.f);
                p.lse_part[prow + i] = -INFINITY;
            } else {
                uint4 z = make_uint4(0, 0, 0, 0);
                uint4* dst = reinterpret_cast<uint4*>(O + (size_t)i * D);
#pragma unroll 4
                for (int v = 0; v < D / 8; ++v) dst[v] = z;
                p.lse[(size_t)bh * p.N + i] = -INFINITY;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

}  // namespace

// [B*H, N, d] of a 16-bit type viewed as a 3-D tensor (d fastest); boxes of
// 64 x rows.
bool make_tmap16(CUtensorMap* map, const void* base, int BH, int N, int d, int box_rows, CUtensorMapDataType type) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, type, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// [B*H, N, d] fp32 (the backward's dQ accumulator) viewed as a 3-D tensor (d
// fastest); boxes of 32 columns (128 bytes, 128-byte swizzle) x 32 rows.
bool make_tmap_f32_acc(CUtensorMap* map, float* base, int BH, int N, int d) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)N * d * 4};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Merges the n_splits partial results of split-KV: with w_s = e^{LSE_s - M},
// O = sum_s w_s O_s / sum_s w_s and LSE = M + log sum_s w_s (M = max_s LSE_s),
// the combination of softmax partials over disjoint key blocks of the
// "FlashAttention" blog post (section "Tiling") and of the paper summary's
// incremental softmax (section "Pelacakan Softmax Inkremental"). One warp per
// row; rows without a visible key (every LSE_s = -inf) get O = 0, LSE = -inf.
template <typename T, int D>
__global__ void __launch_bounds__(256) splitkv_merge_kernel(const float* __restrict__ o_part,
                                                            const float* __restrict__ lse_part,
                                                            T* __restrict__ o, float* __restrict__ lse,
                                                            int n_splits, size_t rows) {
    pdl_wait();  // the partials come from the forward kernel
    const size_t row = (size_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    constexpr int PER = D / 32;  // 2 or 4 floats per lane
    float mx = -INFINITY;
    for (int s = 0; s < n_splits; ++s) mx = fmaxf(mx, lse_part[(size_t)s * rows + row]);
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    float wsum = 0.f;
    if (mx != -INFINITY) {
        for (int s = 0; s < n_splits; ++s) {
            const float ls = lse_part[(size_t)s * rows + row];
            const float w = (ls == -INFINITY) ? 0.f : expf(ls - mx);
            wsum += w;
            const float* src = o_part + ((size_t)s * rows + row) * D + lane * PER;
#pragma unroll
            for (int e = 0; e < PER; ++e) acc[e] = fmaf(w, src[e], acc[e]);
        }
    }
    const float inv = (wsum > 0.f) ? 1.f / wsum : 0.f;
    T* dst = o + row * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; e += 2)
        *reinterpret_cast<uint32_t*>(dst + e) = Elem16<T>::pack2(acc[e] * inv, acc[e + 1] * inv);
    if (lane == 0) lse[row] = (wsum > 0.f) ? mx + logf(wsum) : -INFINITY;
}

FwdParams fwd_params(const Problem& pr) {
    const int BH = pr.B * pr.H;
    FwdParams p{};
    p.lse = pr.lse;
    p.o = pr.o;
    p.block_mask = pr.block_mask;
    p.kv_len = pr.kv_len;
    p.status = pr.status;
    p.H = pr.H;
    p.N = pr.N;
    p.nb = pr.nb;
    p.n_qtiles = (pr.N + kBlockM - 1) / kBlockM;
    p.BH = BH;
    p.n_splits = pr.o_part ? pr.n_splits : 1;
    p.o_part = pr.o_part;
    p.lse_part = pr.lse_part;
    p.scale_log2 = pr.scale * kLog2e;
    p.out_scale = 1.0f / (1.0f - pr.dropout_p);
    p.drop_thr = pr.drop_threshold;
    p.dropout = pr.dropout_p > 0.f;
    p.causal = pr.causal;
    p.seed = pr.seed;
    return p;
}

// split-KV: merges the partial results into O and LSE (launched behind the
// forward kernel with programmatic stream serialization)
template <typename T, int D>
int launch_merge(const Problem& pr, const FwdParams& p, cudaLaunchConfig_t cfg) {
    const size_t rows = (size_t)p.BH * pr.N;
    cfg.gridDim = dim3((unsigned)((rows + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, splitkv_merge_kernel<T, D>, (const float*)p.o_part,
                                             (const float*)p.lse_part, static_cast<T*>(pr.o), pr.lse, p.n_splits, rows);
    note_launches(1);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <typename T, int D, bool kSplit, bool kPartial>
int launch_fwd_tc_d(const Problem& pr) {
    constexpr int kSmem = FwdPPCfg<D>::kSmem;
    constexpr CUtensorMapDataType tt = Elem16<T>::kTmaType;
    CUtensorMap tq, tk, tv, to;
    const int BH = pr.B * pr.H;
    if (!make_tmap16(&tq, pr.q, BH, pr.N, D, kBlockM, tt) || !make_tmap16(&tk, pr.k, BH, pr.N, D, kBlockN, tt) ||
        !make_tmap16(&tv, pr.v, BH, pr.N, D, kBlockN, tt))
        return FA_ERR_CUDA;
    // O's tensor map (split-KV partials are fp32 and stored row by row)
    if (kPartial) to = tq;
    else if (!make_tmap16(&to, pr.o, BH, pr.N, D, kBlockM, tt)) return FA_ERR_CUDA;
    const FwdParams p = fwd_params(pr);
    auto kernel = fwd_pp_kernel<T, D, kSplit, kPartial>;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
            return FA_ERR_CUDA;
        // the setmaxnreg budgets must fit in the registers the kernel is
        // actually launched with, or the softmax warps would wait forever
        cudaFuncAttributes a{};
        if (cudaFuncGetAttributes(&a, kernel) != cudaSuccess ||
            a.numRegs * kThreadsPP < 256 * kSoftmaxRegs + 128 * kIssueRegs) {
            if (std::getenv("FA_DEBUG"))
                std::fprintf(stderr, "fa: fwd register budget exceeds the launch allocation (%d regs)\n", a.numRegs);
            return FA_ERR_CUDA;
        }
        attr_set = true;
    }
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    const long long grid_y = (long long)((p.n_qtiles + 1) / 2) * p.n_splits;
    if (grid_y > 65535) return FA_ERR_UNSUPPORTED;
    cfg.gridDim = dim3(BH, (unsigned)grid_y);
    cfg.blockDim = dim3(kThreadsPP);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = pr.stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    record_main_start(pr.stream);
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, to, p);
    record_main_stop(pr.stream);
    note_launches(1);
    if (e != cudaSuccess) {
        if (std::getenv("FA_DEBUG")) std::fprintf(stderr, "fa: fwd_tc launch: %s\n", cudaGetErrorString(e));
        return FA_ERR_CUDA;
    }
    if (p.o_part) return launch_merge<T, D>(pr, p, cfg);
    return FA_OK;
}

template <typename T, bool kSplit, bool kPartial>
int launch_fwd256(const Problem& pr) {
    constexpr int kSmem = Fwd256Cfg::kSmem;
    constexpr CUtensorMapDataType tt = Elem16<T>::kTmaType;
    CUtensorMap tq, tk, tv;
    const int BH = pr.B * pr.H;
    if (!make_tmap16(&tq, pr.q, BH, pr.N, 256, kBlockM, tt) || !make_tmap16(&tk, pr.k, BH, pr.N, 256, kBlockN, tt) ||
        !make_tmap16(&tv, pr.v, BH, pr.N, 256, kBlockN, tt))
        return FA_ERR_CUDA;
    const FwdParams p = fwd_params(pr);
    auto kernel = fwd_d256_kernel<T, kSplit, kPartial>;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
            return FA_ERR_CUDA;
        attr_set = true;
    }
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    const long long grid_y = (long long)p.n_qtiles * p.n_splits;
    if (grid_y > 65535) return FA_ERR_UNSUPPORTED;
    cfg.gridDim = dim3(BH, (unsigned)grid_y);
    cfg.blockDim = dim3(kThreads256);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = pr.stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    record_main_start(pr.stream);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, p);
    record_main_stop(pr.stream);
    note_launches(1);
    if (e != cudaSuccess) {
        if (std::getenv("FA_DEBUG")) std::fprintf(stderr, "fa: fwd_d256 launch: %s\n", cudaGetErrorString(e));
        return FA_ERR_CUDA;
    }
    if (p.o_part) return launch_merge<T, 256>(pr, p, cfg);
    return FA_OK;
}

template <typename T>
int launch_fwd_tc_t(const Problem& p) {
    if (p.d == 256) {  // one query tile per CTA
        if (p.o_part) return p.block_mask ? launch_fwd256<T, true, true>(p) : launch_fwd256<T, false, true>(p);
        return p.block_mask ? launch_fwd256<T, true, false>(p) : launch_fwd256<T, false, false>(p);
    }
    // head dim 64 (not split-KV): one query tile per CTA, two CTAs per SM
    if (p.d == 64 && !p.o_part) return launch_fwd_1t(p);
    // without a block mask both tiles' key lists are prefixes of one list and
    // share its K/V loads; with one, each tile has its own list (kSplit)
    if (p.o_part) {  // split-KV
        if (p.block_mask)
            return p.d == 64 ? launch_fwd_tc_d<T, 64, true, true>(p) : launch_fwd_tc_d<T, 128, true, true>(p);
        return p.d == 64 ? launch_fwd_tc_d<T, 64, false, true>(p) : launch_fwd_tc_d<T, 128, false, true>(p);
    }
    if (p.block_mask)
        return p.d == 64 ? launch_fwd_tc_d<T, 64, true, false>(p) : launch_fwd_tc_d<T, 128, true, false>(p);
    return p.d == 64 ? launch_fwd_tc_d<T, 64, false, false>(p) : launch_fwd_tc_d<T, 128, false, false>(p);
}

int launch_fwd_tc(const Problem& p) {
    if (!(p.scale > 0.f)) {
        record_main_start(p.stream);
        const cudaError_t e = launch_fwd_simt(p);
        record_main_stop(p.stream);
        return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
    }
    if (p.dtype == FA_FP16) return launch_fwd_tc_t<__half>(p);
    if (p.dtype == FA_BF16) return launch_fwd_tc_t<__nv_bfloat16>(p);
    return FA_ERR_UNSUPPORTED;
}

}  // namespace fa
