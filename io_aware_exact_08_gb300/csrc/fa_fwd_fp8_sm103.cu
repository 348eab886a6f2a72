// Forward attention with 8-bit (E4M3) inputs on the tcgen05 tensor cores.
//
// The FP8 path of the FlashAttention-3 section of "Penjelasan Flash
// Attention: Panduan Komprehensif" ("Presisi FP8 native"): both products of
// the forward run on 8-bit operands (tcgen05.mma kind::f8f6f4, twice the
// 16-bit rate), with fp32 accumulation in TMEM. The algorithm is the same
// block-by-block update as the 16-bit forward ("FlashAttention: Fast and
// Memory-Efficient Exact Attention with IO-Awareness", section "Metode",
// steps 1-4): S_ij = Q_i K_j^T, running row max m and row sum l,
// O_i <- e^{m_old - m_new} O_i + P~_ij V_j, O = O / l at the end.
//
// Inputs and scaling (the pages fix none of this; the reading is this
// library's):
//  - q, k are E4M3 codes [B*H, N, 128]; v is passed transposed, vt =
//    [B*H, 128, N] (keys contiguous), so that both operands of P V are
//    K-major like those of Q K^T;
//  - each head has one dequantisation factor per tensor (descale_q, _k, _v,
//    fp32 [B*H]): the real input is code * factor. The factors of Q and K
//    fold into the softmax scale, V's into the final division by l;
//  - P~ is quantised to E4M3 for the P V product. It is computed as
//    2^(s - m + 5) in log2 units, i.e. shifted up by 2^5 so that the
//    probabilities that matter sit in E4M3's normal range (the smallest
//    normal, 2^-6, stands for 2^-11 of the running maximum; smaller ones
//    round as subnormals, to within 2^-15 of it), and the running max is
//    raised when the row max exceeds it by more than 3.5, so
//    P~ <= 2^8.5 < 448, the largest finite E4M3 value. l sums the fp32
//    values before quantisation; the shift cancels in O = sum P V / l and is
//    taken off LSE. A raise rescales O in TMEM for the whole warp, so the
//    threshold is as large as the E4M3 range allows (a threshold of 1/2
//    with a 2^8 shift measured 1305 against 1698 TFLOP/s on a causal
//    N = 8K, d = 128 problem).
// One CTA computes two 128-row query tiles (ping-pong between two softmax
// warpgroups, as in the 16-bit kernel); head dimension 128 only.
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

constexpr int kD = 128;
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
constexpr int kSoftmaxThreads = 128;
constexpr int kThreads = 384;
constexpr int kSoftmaxRegs = 208, kIssueRegs = 80;
static_assert(256 * kSoftmaxRegs + 128 * kIssueRegs <= kThreads * 168, "register budgets above the launch");
constexpr float kRaise = 3.5f;   // raise the running max when the row max exceeds it by this (log2 units)
constexpr float kPShift = 5.0f;  // P~ = 2^(s - m + 5)
constexpr int kStages = 8;
constexpr int kTileBytes = kBlockN * kD;  // one 128 x 128 E4M3 tile: Q_t, K_j or Vt_j
constexpr int kSmem = 1024 + 2 * kTileBytes + kStages * kTileBytes + 256 + 2 * kMaskListCap * 2;

struct Fp8Params {
    float* lse;
    __nv_bfloat16* o;
    const uint8_t* block_mask;
    const int32_t* kv_len;
    const float* descale_q;
    const float* descale_k;
    const float* descale_v;
    int* status;
    int H, N, nb, n_qtiles;
    float scale_log2;  // scale * log2(e), before the per-head factors
    int causal;
};

struct SharedF8 {
    uint64_t kv_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t q_full;
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t o_final[2];
    uint64_t teardown;
    uint32_t tmem_base;
    int abort_flag;
    int n_list[2];
};
static_assert(sizeof(SharedF8) <= 256, "barrier block");

// TMEM: S_t at columns 128 t (P~ of tile t, E4M3, four to a column, over the
// first 32 of them), O_t at 256 + 128 t.
template <bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_vt, const Fp8Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;  // tile t at t * kTileBytes
    uint8_t* sKV = smem + 2 * kTileBytes;
    SharedF8* st = reinterpret_cast<SharedF8*>(sKV + kStages * kTileBytes);
    uint16_t* sList = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(st) + 256);  // [2][kMaskListCap]

    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // grid (B*H, pairs), x fastest: every head's heaviest causal pair first
    const int bh = blockIdx.x;
    const int b = bh / p.H;
    const int n_pairs = (p.n_qtiles + 1) / 2;
    const int pair = p.causal ? (n_pairs - 1 - (int)blockIdx.y) : (int)blockIdx.y;
    const int L = p.kv_len ? min(max(p.kv_len[b], 0), p.N) : p.N;
    const int nkt = (L + kBlockN - 1) / kBlockN;
    int n_t[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int qt = 2 * pair + t;
        n_t[t] = (qt < p.n_qtiles) ? (p.causal ? min(nkt, qt + 1) : nkt) : 0;
    }
    WaitCtx wctx{&st->abort_flag, p.status};
    if (kSplit && warp == 0) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int qt = 2 * pair + t;
            const int e = n_t[t];
            const int cnt =
                warp_list_visible(p.block_mask + (size_t)qt * p.nb, 1, 0, e, sList + t * kMaskListCap, lane);
            if (lane == 0) st->n_list[t] = cnt;
        }
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&st->kv_full[s], 1);
            mbar_init(&st->kv_empty[s], 1);
        }
        mbar_init(&st->q_full, 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(&st->s_full[t], 1);
            mbar_init(&st->p_full[t], kSoftmaxThreads / 32);
            mbar_init(&st->o_final[t], 1);
        }
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
            prefetch_tmap(&tm_vt);
            const int nq = (n_t[1] > 0) ? 2 : 1;
            mbar_arrive_expect_tx(&st->q_full, nq * kTileBytes);
            for (int t = 0; t < nq; ++t)
                tma_load_3d(sQ + t * kTileBytes, &tm_q, &st->q_full, 0, (2 * pair + t) * kBlockM, bh);
            int t = 0;  // load counter
            // K_j: (d, key row) box at (0, 128 j); Vt_j: (key, d row) box at (128 j, 0)
            auto load = [&](bool is_v, int j) -> bool {
                const int s = t % kStages;
                const uint32_t ph = (t / kStages) & 1;
                if (!mbar_wait(&st->kv_empty[s], ph ^ 1, wctx, 261)) return false;
                mbar_arrive_expect_tx(&st->kv_full[s], kTileBytes);
                uint8_t* dst = sKV + s * kTileBytes;
                if (is_v)
                    tma_load_3d(dst, &tm_vt, &st->kv_full[s], j * kBlockN, 0, bh);
                else
                    tma_load_3d(dst, &tm_k, &st->kv_full[s], 0, j * kBlockN, bh);
                ++t;
                return true;
            };
            bool okp = true;
            if constexpr (!kSplit) {
                // load 2u = K_u, 2u + 1 = Vt_u, shared by both tiles
                for (int u = 0; okp && u < n_max; ++u) {
                    okp = load(false, u);
                    if (okp) okp = load(true, u);
                }
            } else {
                // K of S_0(0), K of S_1(0), then per step u and tile t: Vt of
                // P_t V, K of the tile's next S
                if (n_t[0] > 0) okp = load(false, list0[0]);
                if (okp && n_t[1] > 0) okp = load(false, list1[0]);
                for (int u = 0; okp && u < n_max; ++u) {
                    if (u < n_t[0]) {
                        okp = load(true, list0[u]);
                        if (okp && u + 1 < n_t[0]) okp = load(false, list0[u + 1]);
                    }
                    if (okp && u < n_t[1]) {
                        okp = load(true, list1[u]);
                        if (okp && u + 1 < n_t[1]) okp = load(false, list1[u + 1]);
                    }
                }
            }
            for (int l = max(0, t - kStages); l < t; ++l)
                mbar_wait(&st->kv_full[l % kStages], (l / kStages) & 1, wctx, 262);
            mbar_wait(&st->q_full, 0, wctx, 263);
        }
    } else if (warp == 10 || warp == 11) {
        regs_dec<kIssueRegs>();
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        regs_dec<kIssueRegs>();
        if (n_max > 0) {
            // E4M3 is format code 0 of kind::f8f6f4; every operand K-major
            constexpr uint32_t idesc = idesc_f32acc(0u, kBlockM, 128, 0, 0);
            constexpr uint32_t kStageUnits = kTileBytes >> 4;
            const uint32_t kv_base = smem_u32(sKV);
            const uint64_t qd0 = smem_desc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t qd1 = smem_desc_sw128(smem_u32(sQ + kTileBytes), 16, 1024);
            const uint64_t kvd = smem_desc_sw128(kv_base, 16, 1024);
            bool ok = mbar_wait_warp(&st->q_full, 0, wctx, 270);
            tc_fence_after();
            const int c0 = n_t[0], c1 = n_t[1];
            auto issue_s = [&](int t, int s) {
                const uint64_t qd = t ? qd1 : qd0;
                const uint64_t kd = kvd + (uint64_t)(s * kStageUnits);
#pragma unroll
                for (int kk = 0; kk < kD / 32; ++kk)
                    mma_f8_ss_warp(tmem + t * 128, desc_add(qd, kk * 32), desc_add(kd, kk * 32), idesc, kk > 0);
                mma_commit_warp(&st->s_full[t]);
            };
            auto issue_pv = [&](int t, int s, int u) {
                const uint64_t vd = kvd + (uint64_t)(s * kStageUnits);
#pragma unroll
                for (int kk = 0; kk < kBlockN / 32; ++kk)
                    mma_f8_ts_warp(tmem + 256 + t * 128, tmem + t * 128 + kk * 8, desc_add(vd, kk * 32), idesc,
                                   (u > 0 || kk > 0) ? 1u : 0u);
            };
            if constexpr (!kSplit) {
                if (ok) {
                    ok = mbar_wait_warp(&st->kv_full[0], 0, wctx, 271);
                    tc_fence_after();
                }
                if (ok) {
                    if (c0 > 0) issue_s(0, 0);
                    if (c1 > 0) issue_s(1, 0);
                    mma_commit_warp(&st->kv_empty[0]);
                }
                for (int u = 0; ok && u < n_max; ++u) {
                    const int lv = 2 * u + 1, lk = 2 * u + 2;  // loads of Vt_u and K_{u+1}
                    const int sv = lv % kStages, sk = lk % kStages;
                    const bool need_k = (u + 1 < c0) || (u + 1 < c1);
                    bool v_ready = false, k_ready = false;
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const int ct = t ? c1 : c0;
                        if (u >= ct) continue;
                        if (!mbar_wait_warp(&st->p_full[t], u & 1, wctx, 272)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        if (!v_ready) {
                            if (!mbar_wait_warp(&st->kv_full[sv], (lv / kStages) & 1, wctx, 274)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            v_ready = true;
                        }
                        issue_pv(t, sv, u);
                        if (u + 1 == ct) mma_commit_warp(&st->o_final[t]);
                        if (u + 1 < ct) {
                            if (!k_ready) {
                                if (!mbar_wait_warp(&st->kv_full[sk], (lk / kStages) & 1, wctx, 275)) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after();
                                k_ready = true;
                            }
                            issue_s(t, sk);
                        }
                    }
                    if (!ok) break;
                    mma_commit_warp(&st->kv_empty[sv]);
                    if (need_k) mma_commit_warp(&st->kv_empty[sk]);
                }
            } else {
                int ld = 0;  // next load to use, in the producer's order
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (!ok || (t ? c1 : c0) == 0) continue;
                    const int s = ld % kStages;
                    ok = mbar_wait_warp(&st->kv_full[s], (ld / kStages) & 1, wctx, 271);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(t, s);
                    mma_commit_warp(&st->kv_empty[s]);
                    ++ld;
                }
                for (int u = 0; ok && u < n_max; ++u) {
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const int ct = t ? c1 : c0;
                        if (u >= ct) continue;
                        if (!mbar_wait_warp(&st->p_full[t], u & 1, wctx, 272)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        int s = ld % kStages;
                        if (!mbar_wait_warp(&st->kv_full[s], (ld / kStages) & 1, wctx, 274)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_pv(t, s, u);
                        mma_commit_warp(&st->kv_empty[s]);
                        ++ld;
                        if (u + 1 == ct) mma_commit_warp(&st->o_final[t]);
                        if (u + 1 < ct) {
                            s = ld % kStages;
                            if (!mbar_wait_warp(&st->kv_full[s], (ld / kStages) & 1, wctx, 275)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            issue_s(t, s);
                            mma_commit_warp(&st->kv_empty[s]);
                            ++ld;
                        }
                    }
                }
            }
            mma_commit_warp(&st->teardown);
            mbar_wait_warp(&st->teardown, 0, wctx, 273);
        }
    } else {
        // ------------------------------------------------------------ softmax
        regs_inc<kSoftmaxRegs>();
        const int t = warp >> 2;
        const int r = tid & 127;
        const int i = (2 * pair + t) * kBlockM + r;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t sbase = tmem + lane_base + t * 128;
        const uint32_t obase = tmem + lane_base + 256 + t * 128;
        const int n = n_t[t];
        // scores in log2 units: raw Q8.K8 times scale * log2(e) * the two factors
        const float sl2 = p.scale_log2 * p.descale_q[bh] * p.descale_k[bh];
        float m = -INFINITY;
        float l = 0.f;
        bool ok = true;
        const uint16_t* my_list = t ? list1 : list0;
        for (int u = 0; u < n; ++u) {
            const int ktile = kSplit ? (int)my_list[u] : u;
            if (!mbar_wait_warp(&st->s_full[t], u & 1, wctx, 280)) {
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
            const float mt = pm[0] * sl2;
            const bool raise = mt > m + kRaise;
            if (__any_sync(0xffffffffu, raise) && u > 0) {
                // S_t(u) was issued after P_t(u-1) V: O_t is complete here
                const float alpha = raise ? ex2_approx(m - mt) : 1.f;
#pragma unroll 1
                for (int c = 0; c < kD / 8; ++c) {
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
            // P~ = 2^(s - m + 5): at most 2^8.5 < 448
            const float nmref = (m == -INFINITY) ? 0.f : kPShift - m;
            float ps[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) ps[x] = 0.f;
            // four E4M3 values per word; word x/4 of chunk c overwrites a
            // register already consumed
#pragma unroll
            for (int c = 0; c < 4; ++c) {
#pragma unroll
                for (int x = 0; x < 32; x += 4) {
                    float a0, a1, a2, a3;
                    ffma2(a0, a1, __uint_as_float(sr[c][x]), __uint_as_float(sr[c][x + 1]), sl2, sl2, nmref, nmref);
                    ffma2(a2, a3, __uint_as_float(sr[c][x + 2]), __uint_as_float(sr[c][x + 3]), sl2, sl2, nmref, nmref);
                    const float e0 = ex2_approx(a0), e1 = ex2_approx(a1), e2 = ex2_approx(a2), e3 = ex2_approx(a3);
                    const int k = (x >> 2) & 3;
                    fadd2(ps[2 * k], ps[2 * k + 1], ps[2 * k], ps[2 * k + 1], e0, e1);
                    fadd2(ps[2 * k], ps[2 * k + 1], ps[2 * k], ps[2 * k + 1], e2, e3);
                    sr[c][x >> 2] = pack_e4m3x4(e0, e1, e2, e3);
                }
                tmem_st8(sbase + c * 8, *reinterpret_cast<uint32_t(*)[8]>(&sr[c][0]));
            }
            fadd2(ps[0], ps[1], ps[0], ps[1], ps[4], ps[5]);
            fadd2(ps[2], ps[3], ps[2], ps[3], ps[6], ps[7]);
            fadd2(ps[0], ps[1], ps[0], ps[1], ps[2], ps[3]);
            l += ps[0] + ps[1];
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive_warp(&st->p_full[t]);
        }
        __nv_bfloat16* O = p.o + ((size_t)bh * p.N) * kD;
        if (ok && n > 0) {
            if (mbar_wait_warp(&st->o_final[t], 0, wctx, 281)) {
                tc_fence_after();
                const float inv = (l > 0.f) ? p.descale_v[bh] / l : 0.f;
#pragma unroll
                for (int c = 0; c < kD / 32; ++c) {
                    uint32_t orr[32];
                    tmem_ld32(obase + c * 32, orr);
                    tmem_ld_wait();
                    reg_fence(orr);
                    if (i < p.N) {
                        uint4* dst = reinterpret_cast<uint4*>(O + (size_t)i * kD + c * 32);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint4 w4;
                            w4.x = pack_bf16x2(__uint_as_float(orr[8 * v + 0]) * inv, __uint_as_float(orr[8 * v + 1]) * inv);
                            w4.y = pack_bf16x2(__uint_as_float(orr[8 * v + 2]) * inv, __uint_as_float(orr[8 * v + 3]) * inv);
                            w4.z = pack_bf16x2(__uint_as_float(orr[8 * v + 4]) * inv, __uint_as_float(orr[8 * v + 5]) * inv);
                            w4.w = pack_bf16x2(__uint_as_float(orr[8 * v + 6]) * inv, __uint_as_float(orr[8 * v + 7]) * inv);
                            dst[v] = w4;
                        }
                    }
                }
                if (i < p.N) p.lse[(size_t)bh * p.N + i] = (l > 0.f) ? (m - kPShift + __log2f(l)) * kLn2 : -INFINITY;
            }
        } else if (n == 0 && i < p.N) {
            const uint4 z = make_uint4(0, 0, 0, 0);
            uint4* dst = reinterpret_cast<uint4*>(O + (size_t)i * kD);
#pragma unroll
            for (int v = 0; v < kD / 8; ++v) dst[v] = z;
            p.lse[(size_t)bh * p.N + i] = -INFINITY;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem, 512);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn8() {
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

// A [BH, rows, cols] byte tensor (cols fastest) as a 3-D tensor map with
// 128 x 128 boxes and the 128-byte swizzle; cols must be a multiple of 16.
bool make_tmap8(CUtensorMap* map, const void* base, int BH, int rows, int cols) {
    EncodeTiledFn fn = encode_fn8();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)cols, (cuuint64_t)rows * cols};
    cuuint32_t box[3] = {128, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kSplit>
int launch_fp8_t(const Problem& pr, const Fp8Inputs& in) {
    const int BH = pr.B * pr.H;
    CUtensorMap tq, tk, tvt;
    if (!make_tmap8(&tq, pr.q, BH, pr.N, kD) || !make_tmap8(&tk, pr.k, BH, pr.N, kD) ||
        !make_tmap8(&tvt, pr.v, BH, kD, pr.N))
        return FA_ERR_CUDA;
    Fp8Params p{};
    p.lse = pr.lse;
    p.o = static_cast<__nv_bfloat16*>(pr.o);
    p.block_mask = pr.block_mask;
    p.kv_len = pr.kv_len;
    p.descale_q = in.descale_q;
    p.descale_k = in.descale_k;
    p.descale_v = in.descale_v;
    p.status = pr.status;
    p.H = pr.H;
    p.N = pr.N;
    p.nb = pr.nb;
    p.n_qtiles = (pr.N + kBlockM - 1) / kBlockM;
    p.scale_log2 = pr.scale * kLog2e;
    p.causal = pr.causal;
    auto kernel = fwd_fp8_kernel<kSplit>;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
            return FA_ERR_CUDA;
        cudaFuncAttributes a{};
        if (cudaFuncGetAttributes(&a, kernel) != cudaSuccess ||
            a.numRegs * kThreads < 256 * kSoftmaxRegs + 128 * kIssueRegs) {
            if (std::getenv("FA_DEBUG"))
                std::fprintf(stderr, "fa: fp8 register budget exceeds the launch allocation (%d regs)\n", a.numRegs);
            return FA_ERR_CUDA;
        }
        attr_set = true;
    }
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    const int grid_y = (p.n_qtiles + 1) / 2;
    if (grid_y > 65535) return FA_ERR_UNSUPPORTED;
    cfg.gridDim = dim3(BH, grid_y);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = pr.stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    record_main_start(pr.stream);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tq, tk, tvt, p);
    record_main_stop(pr.stream);
    note_launches(1);
    if (e != cudaSuccess) {
        if (std::getenv("FA_DEBUG")) std::fprintf(stderr, "fa: fwd_fp8 launch: %s\n", cudaGetErrorString(e));
        return FA_ERR_CUDA;
    }
    return FA_OK;
}

}  // namespace

int launch_fwd_fp8(const Problem& p, const Fp8Inputs& in) {
    return p.block_mask ? launch_fp8_t<true>(p, in) : launch_fp8_t<false>(p, in);
}

}  // namespace fa
