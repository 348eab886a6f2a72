// Forward attention at head dimension 64, one 128-row query tile per CTA,
// two CTAs per SM.
//
// The same per-block update as the two-tile kernel ("FlashAttention: Fast and
// Memory-Efficient Exact Attention with IO-Awareness", section "Metode",
// steps 1-4; the division by l deferred to the end as in the FlashAttention-2
// section of the "Flash Attention" guide), laid out so that two CTAs fit on
// one SM: TMEM holds S (128 columns), O (64) and P (64 columns of packed
// 16-bit pairs) in a 256-column allocation, and shared memory holds Q and a
// five-stage K/V ring (about 100 KB). P has columns of its own so that
// S(u+1) = Q K_{u+1}^T is issued as soon as the softmax has read S(u) into
// registers: the tensor core computes the next scores and P(u-1) V while the
// softmax of tile u runs. The MMA order is S(0), S(1), P(0)V, S(2), P(1)V, ...
// and the loads follow it (K0, K1, V0, K2, V1, ...). Each query row is shared
// by two softmax threads, one per 64-key half of the tile, which halves the
// per-thread chain (TMEM load, exponentials, P store) that bounds a CTA's
// pace; the halves exchange their maxima once per tile. The tensor core
// alternates between the two CTAs of the SM, and one CTA's start (barriers,
// TMEM, the Q and first K/V loads) and end (the O and LSE stores) overlap the
// other's main loop.
// Roles (384 threads): warps 0-7 softmax (thread = query row, column half),
// warp 8 TMA producer, warp 9 MMA issuer (all 32 lanes run its loop, one
// elected lane issues), warps 10-11 idle. setmaxnreg gives the softmax
// warpgroups 96 registers a thread and the other 48 (launched at 80).
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

bool make_tmap16(CUtensorMap* map, const void* base, int BH, int N, int d, int box_rows, CUtensorMapDataType type);

namespace {

using namespace sm103;

constexpr int kD = 64;
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
// Thread layout, chosen by whether dropout applies. With dropout the keep
// bits (one Philox4x32-10 call per four keys) dominate a tile, and two
// threads per query row (one per 64-key half) halve them per thread
// (bert_pad_dropout forward 192 -> 239 TFLOP/s). Without dropout the
// exchange of the halves' maxima costs more than the shorter chain saves
// (block_sparse forward 650 against 563 TFLOP/s), so one thread takes a row.
template <bool kDrop>
struct Layout1t {
    static constexpr int kHalves = kDrop ? 2 : 1;           // softmax threads per query row
    static constexpr int kSoftWarps = 4 * kHalves;
    static constexpr int kThreads = 32 * kSoftWarps + 128;  // + producer, MMA issuer, two idle warps
    // two CTAs per SM; setmaxnreg moves registers to the softmax warps
    static constexpr int kLaunchRegs = 65536 / (2 * kThreads) / 8 * 8;
    static constexpr int kSoftRegs = kDrop ? 96 : 208, kIssueRegs = 48;
    static constexpr int kBudget = 32 * kSoftWarps * kSoftRegs + 128 * kIssueRegs;
    static_assert(kBudget <= kThreads * kLaunchRegs, "register budgets above the launch");
    static constexpr int kCols = kBlockN / kHalves;  // keys of a tile per thread
    static constexpr int kChunks = kCols / 32;
    static constexpr int kOCols = kD / kHalves;      // columns of O per thread
};
constexpr float kRescaleThreshold = 8.0f;  // log2 units, as in the two-tile kernel
constexpr int kStages = 5;
constexpr int kTileBytes = kBlockN * kD * 2;  // one 128 x 64 16-bit tile (one 128-byte-wide box)
// barrier block, the two column halves' row maxima (double-buffered by tile
// parity) and row-sum shares, the block-mask tile list
constexpr int kSmem = 1024 + kTileBytes + kStages * kTileBytes + 256 + (2 * 2 * 128 + 2 * 128) * 4 + kMaskListCap * 2;
static_assert(2 * (kSmem + 1024) <= 228 * 1024, "two CTAs per SM");
constexpr uint32_t kColS = 0, kColO = 128, kColP = 192, kTmemCols = 256;

struct Fwd1tParams {
    float* lse;
    void* o;
    const uint8_t* block_mask;
    const int32_t* kv_len;
    int* status;
    int H, N, nb, n_qtiles;
    float scale_log2;
    float out_scale;  // 1/(1-p)
    uint32_t drop_thr;
    int causal;
    uint64_t seed;
};

struct Shared1t {
    uint64_t kv_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t q_full;
    uint64_t s_full;   // S(u) in TMEM
    uint64_t s_free;   // the softmax has read S(u): S(u+1) may be written
    uint64_t p_full;   // P(u) in TMEM
    uint64_t pv_done;  // P(u) V has completed: O may be rescaled, P overwritten
    uint64_t mx_ready[2][4];  // both column halves' maxima of tile u (buffer u & 1), rows of quarter q, written
    uint64_t l_ready;      // both halves' row-sum shares written
    uint64_t o_final;
    uint64_t o_staged;  // every softmax warp has written its rows of O over Q
    uint64_t teardown;
    uint32_t tmem_base;
    int abort_flag;
    int n_list;
};
static_assert(sizeof(Shared1t) <= 256, "barrier block");

template <typename T, bool kSplit, bool kDrop>
__global__ void __launch_bounds__(Layout1t<kDrop>::kThreads, 2)
    fwd_1t_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const Fwd1tParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sKV = smem + kTileBytes;
    Shared1t* st = reinterpret_cast<Shared1t*>(sKV + kStages * kTileBytes);
    float* sMax = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(st) + 256);  // [2 parities][2 halves][128 rows]
    float* sL = sMax + 2 * 2 * 128;                                                // [2 halves][128 rows]
    uint16_t* sList = reinterpret_cast<uint16_t*>(sL + 2 * 128);                   // [kMaskListCap]

    using Lay = Layout1t<kDrop>;
    constexpr int kProdWarp = Lay::kSoftWarps, kMmaWarp = Lay::kSoftWarps + 1;
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // grid (B*H, query tiles), x fastest: every head's heaviest causal tile first
    const int bh = blockIdx.x;
    const int b = bh / p.H, h = bh % p.H;
    const int qt = p.causal ? (p.n_qtiles - 1 - (int)blockIdx.y) : (int)blockIdx.y;
    const int L = p.kv_len ? min(max(p.kv_len[b], 0), p.N) : p.N;
    const int nkt = (L + kBlockN - 1) / kBlockN;
    int n = p.causal ? min(nkt, qt + 1) : nkt;
    WaitCtx wctx{&st->abort_flag, p.status};
    if (kSplit && warp == 0) {
        const int cnt = warp_list_visible(p.block_mask + (size_t)qt * p.nb, 1, 0, n, sList, lane);
        if (lane == 0) st->n_list = cnt;
    }
    if (warp == kProdWarp && lane == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&st->kv_full[s], 1);
            mbar_init(&st->kv_empty[s], 1);
        }
        mbar_init(&st->q_full, 1);
        mbar_init(&st->s_full, 1);
        mbar_init(&st->s_free, Lay::kSoftWarps);
        mbar_init(&st->p_full, Lay::kSoftWarps);
        mbar_init(&st->pv_done, 1);
        for (int q = 0; q < 4; ++q) {  // the two warps (one per column half) of lane quarter q
            mbar_init(&st->mx_ready[0][q], Lay::kHalves);
            mbar_init(&st->mx_ready[1][q], Lay::kHalves);
        }
        mbar_init(&st->l_ready, Lay::kSoftWarps);
        mbar_init(&st->o_final, 1);
        mbar_init(&st->o_staged, Lay::kSoftWarps);
        mbar_init(&st->teardown, 1);
        st->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&st->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = st->tmem_base;
    if constexpr (kSplit) n = st->n_list;

    if (warp == kProdWarp) {
        // ------------------------------------------------------------ producer
        regs_dec<Lay::kIssueRegs>();
        if (lane == 0 && n > 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            mbar_arrive_expect_tx(&st->q_full, kTileBytes);
            tma_load_3d(sQ, &tm_q, &st->q_full, 0, qt * kBlockM, bh);
            // loads in the order the MMA warp uses them: K(0), then for each
            // u, K(u+1) (if any) and V(u)
            int t = 0;
            bool okp = true;
            for (int x = 0; okp && x < 2 * n; ++x) {
                const bool is_v = x > 0 && ((x & 1) == 0 || x == 2 * n - 1);
                const int u = is_v ? (x == 2 * n - 1 ? n - 1 : x / 2 - 1) : (x + 1) / 2;
                const int j = kSplit ? (int)sList[u] : u;
                const int s = t % kStages;
                const uint32_t ph = (t / kStages) & 1;
                if (!mbar_wait(&st->kv_empty[s], ph ^ 1, wctx, 361)) {
                    okp = false;
                    break;
                }
                mbar_arrive_expect_tx(&st->kv_full[s], kTileBytes);
                tma_load_3d(sKV + s * kTileBytes, is_v ? &tm_v : &tm_k, &st->kv_full[s], 0, j * kBlockN, bh);
                ++t;
            }
            // drain: the last load issued into each stage has landed
            for (int l = max(0, t - kStages); l < t; ++l)
                mbar_wait(&st->kv_full[l % kStages], (l / kStages) & 1, wctx, 362);
            mbar_wait(&st->q_full, 0, wctx, 363);
        }
    } else if (warp > kMmaWarp) {
        regs_dec<Lay::kIssueRegs>();  // idle: the rest of the producer / MMA warpgroup
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        regs_dec<Lay::kIssueRegs>();
        if (n > 0) {
            constexpr uint32_t idesc_s = idesc_f32acc(Elem16<T>::kFmt, kBlockM, kBlockN, 0, 0);
            constexpr uint32_t idesc_o = idesc_f32acc(Elem16<T>::kFmt, kBlockM, kD, 0, 1);
            constexpr uint32_t kStageUnits = kTileBytes >> 4;
            const uint32_t kv_base = smem_u32(sKV);
            const uint64_t qd = smem_desc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t kvd_k = smem_desc_sw128(kv_base, 16, 1024);               // K tiles, K-major
            const uint64_t kvd_v = smem_desc_sw128(kv_base, kBlockN * 128, 1024);    // V tiles, MN-major
            bool ok = mbar_wait_warp(&st->q_full, 0, wctx, 370);
            tc_fence_after();
            int ld = 0;  // next load to use
            // S(u) = Q K_u^T over the S columns (S(u-1) has been read)
            auto issue_s = [&]() -> bool {
                const int s = ld % kStages;
                if (!mbar_wait_warp(&st->kv_full[s], (ld / kStages) & 1, wctx, 371)) return false;
                tc_fence_after();
                const uint64_t kd = kvd_k + (uint64_t)(s * kStageUnits);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk)
                    mma_ss_warp(tmem + kColS, desc_add(qd, kk * 32), desc_add(kd, kk * 32), idesc_s, kk > 0);
                mma_commit_warp(&st->s_full);
                mma_commit_warp(&st->kv_empty[s]);
                ++ld;
                return true;
            };
            if (ok) ok = issue_s();
            for (int u = 0; ok && u < n; ++u) {
                if (u + 1 < n) {
                    if (!mbar_wait_warp(&st->s_free, u & 1, wctx, 375)) break;
                    tc_fence_after();
                    if (!issue_s()) break;
                }
                // O += P(u) V_u, A = P(u) from TMEM
                if (!mbar_wait_warp(&st->p_full, u & 1, wctx, 372)) break;
                tc_fence_after();
                const int s = ld % kStages;
                if (!mbar_wait_warp(&st->kv_full[s], (ld / kStages) & 1, wctx, 374)) break;
                tc_fence_after();
                const uint64_t vd = kvd_v + (uint64_t)(s * kStageUnits);
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk)
                    mma_ts_warp(tmem + kColO, tmem + kColP + kk * 8, desc_add(vd, kk * 16 * 128), idesc_o,
                                (u > 0 || kk > 0) ? 1u : 0u);
                mma_commit_warp(&st->kv_empty[s]);
                mma_commit_warp(&st->pv_done);
                ++ld;
                if (u + 1 == n) mma_commit_warp(&st->o_final);
            }
            mma_commit_warp(&st->teardown);
            mbar_wait_warp(&st->teardown, 0, wctx, 373);
        }
    } else {
        // ------------------------------------------------------------ softmax
        // warp w reads TMEM lane quarter w & 3 (query rows 32 (w & 3) .. + 31)
        // and column part w >> 2 of every score tile. With two parts (the
        // dropout layout) a row is shared by two threads, one per 64-key half:
        // both take the tile's row maximum from the two halves' maxima
        // (exchanged through shared memory), so they keep the same running
        // maximum m and make the same rescaling decisions; each rescales and
        // stores its columns of O and keeps its share of the row sum l, and
        // the shares are added at the end.
        regs_inc<Lay::kSoftRegs>();
        constexpr int kCols = Lay::kCols, kChunks = Lay::kChunks, kOCols = Lay::kOCols;
        const int quarter = warp & 3;
        const int half = warp >> 2;  // column part (0 in the one-part layout)
        const int r = quarter * 32 + lane;  // query row within the tile
        const int i = qt * kBlockM + r;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const uint32_t sbase = tmem + lane_base + kColS + kCols * half;
        const uint32_t obase = tmem + lane_base + kColO + kOCols * half;
        const uint32_t pbase = tmem + lane_base + kColP + (kCols / 2) * half;
        float m = -INFINITY;
        float l = 0.f;
        bool ok = true;
        for (int u = 0; u < n; ++u) {
            const int ktile = kSplit ? (int)sList[u] : u;
            // dropout keep bits of this thread's keys (bit x of keep[c] is
            // key kCols half + 32 c + x of the tile), drawn before S arrives
            uint32_t keep[kChunks];
#pragma unroll
            for (int c = 0; c < kChunks; ++c) keep[c] = 0xffffffffu;
            if constexpr (kDrop) {
#pragma unroll
                for (int c = 0; c < kChunks; ++c) keep[c] = 0;
#pragma unroll 8
                for (int g = 0; g < kCols / 4; ++g) {
                    const uint32_t bits =
                        keep_bits4(p.seed, p.drop_thr, b, h, i, ktile * (kBlockN / 4) + (kCols / 4) * half + g);
                    keep[g >> 3] |= bits << (4 * (g & 7));
                }
            }
            if (!mbar_wait_warp(&st->s_full, u & 1, wctx, 380)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int k0 = ktile * kBlockN + kCols * half;  // first key of this thread's part
            int lim = min(kCols, L - k0);
            if (p.causal) lim = min(lim, i - k0 + 1);
            uint32_t sr[kChunks][32];
#pragma unroll
            for (int c = 0; c < kChunks; ++c) tmem_ld32(sbase + c * 32, sr[c]);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < kChunks; ++c) reg_fence(sr[c]);
            // S(u) is in registers: the S columns may take S(u+1)
            tc_fence_before();
            mbar_arrive_warp(&st->s_free);
            if (lim < kCols) {
#pragma unroll
                for (int c = 0; c < kChunks; ++c)
#pragma unroll
                    for (int x = 0; x < 32; ++x)
                        if (c * 32 + x >= lim) sr[c][x] = __float_as_uint(-INFINITY);
            }
            float pm[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) pm[x] = -INFINITY;
#pragma unroll
            for (int c = 0; c < kChunks; ++c)
#pragma unroll
                for (int x = 0; x < 32; x += 2)
                    pm[(x >> 1) & 7] =
                        fmax3(pm[(x >> 1) & 7], __uint_as_float(sr[c][x]), __uint_as_float(sr[c][x + 1]));
            pm[0] = fmax3(pm[0], pm[1], pm[2]);
            pm[3] = fmax3(pm[3], pm[4], pm[5]);
            pm[6] = fmaxf(pm[6], pm[7]);
            pm[0] = fmax3(pm[0], pm[3], pm[6]);
            if constexpr (Lay::kHalves == 2) {
                // the row maximum of the tile from both halves, exchanged
                // between the two warps that share these 32 rows (a barrier
                // per lane quarter; buffer u & 1: a warp writes it again at
                // u + 2 only after both have passed the exchange of u + 1, so
                // after this one's reads)
                float* mx = sMax + (u & 1) * 256;
                mx[half * 128 + r] = pm[0];
                mbar_arrive_warp(&st->mx_ready[u & 1][quarter]);
                if (!mbar_wait_warp(&st->mx_ready[u & 1][quarter], (u >> 1) & 1, wctx, 384)) {
                    ok = false;
                    break;
                }
                pm[0] = fmaxf(pm[0], mx[(half ^ 1) * 128 + r]);
            }
            const float mt = pm[0] * p.scale_log2;
            const bool raise = mt > m + kRescaleThreshold;
            // P(u-1) V must have completed before O is rescaled or P(u)
            // written over P(u-1)
            bool pv_waited = (u == 0);
            if (__any_sync(0xffffffffu, raise) && u > 0) {
                if (!mbar_wait_warp(&st->pv_done, (u - 1) & 1, wctx, 382)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                pv_waited = true;
                const float alpha = raise ? ex2_approx(m - mt) : 1.f;
#pragma unroll 1
                for (int c = 0; c < kOCols / 8; ++c) {
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
            // exponentials packed in place (P chunk c in sr[c][0..15], this
            // thread's P columns 16c..16c+15); the sum takes every
            // exponential, the dropout mask only what goes to P. Without
            // dropout all chunks are stored after the last exponential, so the
            // wait for P(u-1) V comes as late as possible; with dropout the
            // wait comes first and each chunk is stored as soon as it is
            // packed, which keeps fewer registers live.
            if constexpr (!kDrop) {
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
#pragma unroll
                    for (int x = 0; x < 32; x += 2) {
                        float a0, a1;
                        ffma2(a0, a1, __uint_as_float(sr[c][x]), __uint_as_float(sr[c][x + 1]), sl2, sl2, nmref, nmref);
                        const float e0 = ex2_approx(a0), e1 = ex2_approx(a1);
                        const int k = (x >> 1) & 3;
                        fadd2(ps[2 * k], ps[2 * k + 1], ps[2 * k], ps[2 * k + 1], e0, e1);
                        sr[c][x >> 1] = Elem16<T>::pack2(e0, e1);
                    }
                }
            } else {
                if (!pv_waited) {
                    if (!mbar_wait_warp(&st->pv_done, (u - 1) & 1, wctx, 383)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    pv_waited = true;
                }
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
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
                    tmem_st16(pbase + c * 16, *reinterpret_cast<const uint32_t(*)[16]>(&sr[c][0]));
                }
            }
            fadd2(ps[0], ps[1], ps[0], ps[1], ps[4], ps[5]);
            fadd2(ps[2], ps[3], ps[2], ps[3], ps[6], ps[7]);
            fadd2(ps[0], ps[1], ps[0], ps[1], ps[2], ps[3]);
            l += ps[0] + ps[1];
            if constexpr (!kDrop) {
                if (!pv_waited) {
                    if (!mbar_wait_warp(&st->pv_done, (u - 1) & 1, wctx, 383)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
#pragma unroll
                for (int c = 0; c < kChunks; ++c)
                    tmem_st16(pbase + c * 16, *reinterpret_cast<const uint32_t(*)[16]>(&sr[c][0]));
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive_warp(&st->p_full);
        }
        T* O = static_cast<T*>(p.o) + ((size_t)bh * p.N) * kD;
        if (ok && n > 0) {
            bool ready = true;
            float lt = l;
            if constexpr (Lay::kHalves == 2) {
                // the row sum is the two halves' shares
                sL[half * 128 + r] = l;
                mbar_arrive_warp(&st->l_ready);
                ready = mbar_wait_warp(&st->l_ready, 0, wctx, 385);
                if (ready) lt += sL[(half ^ 1) * 128 + r];
            }
            if (ready && mbar_wait_warp(&st->o_final, 0, wctx, 381)) {
                tc_fence_after();
                // O = acc / l in 16 bits, written over Q (every product has
                // completed, the last S before the last P V) as one 128 x 64
                // tile, 128-byte swizzled (16-byte chunk c of row r at chunk
                // position c ^ (r & 7)), then stored by the TMA engine: rows
                // past N are outside the tensor and not written
                const float inv = (lt > 0.f) ? p.out_scale / lt : 0.f;
#pragma unroll
                for (int c = 0; c < kOCols / 32; ++c) {
                    uint32_t orr[32];
                    tmem_ld32(obase + c * 32, orr);
                    tmem_ld_wait();
                    reg_fence(orr);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 w4;
                        w4.x = Elem16<T>::pack2(__uint_as_float(orr[8 * v + 0]) * inv, __uint_as_float(orr[8 * v + 1]) * inv);
                        w4.y = Elem16<T>::pack2(__uint_as_float(orr[8 * v + 2]) * inv, __uint_as_float(orr[8 * v + 3]) * inv);
                        w4.z = Elem16<T>::pack2(__uint_as_float(orr[8 * v + 4]) * inv, __uint_as_float(orr[8 * v + 5]) * inv);
                        w4.w = Elem16<T>::pack2(__uint_as_float(orr[8 * v + 6]) * inv, __uint_as_float(orr[8 * v + 7]) * inv);
                        const int chunk = (kOCols * half + c * 32) / 8 + v;
                        *reinterpret_cast<uint4*>(sQ + r * 128 + ((chunk ^ (r & 7)) << 4)) = w4;
                    }
                }
                if (half == 0 && i < p.N) p.lse[(size_t)bh * p.N + i] = (lt > 0.f) ? (m + __log2f(lt)) * kLn2 : -INFINITY;
                fence_proxy_async_smem();
                mbar_arrive_warp(&st->o_staged);
                if (warp == 0 && mbar_wait_warp(&st->o_staged, 0, wctx, 386) && lane == 0) {
                    tma_store_3d(&tm_o, sQ, 0, qt * kBlockM, bh);
                    bulk_commit_group();
                    bulk_wait_all();  // complete before the CTA ends
                }
            }
        } else if (n == 0 && i < p.N) {
            const uint4 z = make_uint4(0, 0, 0, 0);
            uint4* dst = reinterpret_cast<uint4*>(O + (size_t)i * kD + kOCols * half);
#pragma unroll
            for (int v = 0; v < kOCols / 8; ++v) dst[v] = z;
            if (half == 0) p.lse[(size_t)bh * p.N + i] = -INFINITY;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

template <typename T, bool kSplit, bool kDrop>
int launch_1t(const Problem& pr) {
    constexpr CUtensorMapDataType tt = Elem16<T>::kTmaType;
    CUtensorMap tq, tk, tv, to;
    const int BH = pr.B * pr.H;
    if (!make_tmap16(&tq, pr.q, BH, pr.N, kD, kBlockM, tt) || !make_tmap16(&tk, pr.k, BH, pr.N, kD, kBlockN, tt) ||
        !make_tmap16(&tv, pr.v, BH, pr.N, kD, kBlockN, tt) || !make_tmap16(&to, pr.o, BH, pr.N, kD, kBlockM, tt))
        return FA_ERR_CUDA;
    Fwd1tParams p{};
    p.lse = pr.lse;
    p.o = pr.o;
    p.block_mask = pr.block_mask;
    p.kv_len = pr.kv_len;
    p.status = pr.status;
    p.H = pr.H;
    p.N = pr.N;
    p.nb = pr.nb;
    p.n_qtiles = (pr.N + kBlockM - 1) / kBlockM;
    p.scale_log2 = pr.scale * kLog2e;
    p.out_scale = 1.0f / (1.0f - pr.dropout_p);
    p.drop_thr = pr.drop_threshold;
    p.causal = pr.causal;
    p.seed = pr.seed;
    auto kernel = fwd_1t_kernel<T, kSplit, kDrop>;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
            return FA_ERR_CUDA;
        // the setmaxnreg budgets must fit in the registers the kernel is
        // launched with, or the softmax warps would wait forever
        cudaFuncAttributes a{};
        if (cudaFuncGetAttributes(&a, kernel) != cudaSuccess ||
            a.numRegs * Layout1t<kDrop>::kThreads < Layout1t<kDrop>::kBudget) {
            if (std::getenv("FA_DEBUG"))
                std::fprintf(stderr, "fa: fwd_1t register budget exceeds the launch allocation (%d regs)\n", a.numRegs);
            return FA_ERR_CUDA;
        }
        attr_set = true;
    }
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    if (p.n_qtiles > 65535) return FA_ERR_UNSUPPORTED;
    cfg.gridDim = dim3(BH, p.n_qtiles);
    cfg.blockDim = dim3(Layout1t<kDrop>::kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = pr.stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    record_main_start(pr.stream);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, to, p);
    record_main_stop(pr.stream);
    note_launches(1);
    if (e != cudaSuccess) {
        if (std::getenv("FA_DEBUG")) std::fprintf(stderr, "fa: fwd_1t launch: %s\n", cudaGetErrorString(e));
        return FA_ERR_CUDA;
    }
    return FA_OK;
}

template <typename T>
int launch_1t_for(const Problem& p) {
    const bool drop = p.dropout_p > 0.f;
    if (p.block_mask) return drop ? launch_1t<T, true, true>(p) : launch_1t<T, true, false>(p);
    return drop ? launch_1t<T, false, true>(p) : launch_1t<T, false, false>(p);
}

}  // namespace

int launch_fwd_1t(const Problem& p) {
    if (p.dtype == FA_FP16) return launch_1t_for<__half>(p);
    if (p.dtype == FA_BF16) return launch_1t_for<__nv_bfloat16>(p);
    return FA_ERR_UNSUPPORTED;
}

}  // namespace fa
