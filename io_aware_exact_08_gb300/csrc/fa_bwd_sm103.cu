// Backward attention on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// The backward keeps only O and the per-row log-sum-exp from the forward and
// recomputes S and P tile by tile on chip ("FlashAttention: Fast and
// Memory-Efficient Exact Attention with IO-Awareness", section "Ide Utama",
// third point; "FlashAttention" blog post, section "Recomputation"). With
// P^ = P o Z/(1-p) the dropped-out probabilities, the gradients are
//   dV = P^T dO,  dP = (dO V^T) o Z/(1-p),  dS = P o (dP - rowsum(dO o O)),
//   dK = scale dS^T Q,  dQ = scale dS K.
//
// Three launches:
//   1. preprocess: per 128-row query tile a column table of -LSE_i log2(e)
//      and -delta_i, delta_i = sum_c dO_ic O_ic (fp32, rows past N padded),
//      dQacc = 0 and the work counter = 0;
//   2. main: work items are (128-key tile K_j/V_j, batch*head) pairs, each
//      looping over the query tiles i that see it; one CTA per item, or (the
//      persistent grid) one CTA per SM claiming items in order. The TMA
//      engine loads each step's Q_i, dO_i and column table into one stage.
//      Per tile, on tensor cores:
//        S^T = K_j Q_i^T,  dP^T = V_j dO_i^T          (TMEM, fp32)
//      (D = 64: over all 128 queries; D = 128: per 64-query half), eight
//      compute warps (thread = key row, half of the 128 query columns each)
//      rebuild P^T = exp(S^T - LSE), apply masks and dropout, and form
//      dS^T = P^T o (dP^T - delta); P^T (16-bit) goes back into TMEM and dS^T
//      (16-bit) into a swizzled shared-memory tile, then
//        dV_j += P^T dO_i  (A from TMEM),  dK_j += dS^T Q_i,
//        dQ_i = dS K_j (both operands read MN-major)
//      (at D = 128 computed transposed, dQ_i^T = K_j^T dS^T, so that a
//      warp's reduction covers 32 consecutive floats of one row), and the
//      reduction warps add it into the fp32 accumulator in global memory
//      (D = 128: red.global.add; D = 64: TMA bulk tensor reduce-adds of
//      32 x 32 boxes staged in shared memory). dK_j, dV_j stay in TMEM until
//      the item's end.
//   3. convert: dq = dtype(scale * dQacc).
// Roles: warps 0-7 compute, warp 8 TMA producer, warp 9 MMA issuer (all 32
// lanes run its loop, one elected lane issues), warp 10 claims the persistent
// grid's items and builds their block-mask tile lists, warp 11 stores dK and
// dV at D = 64 (TMA stores of tiles the compute warps stage in the item's K/V
// buffer; idle at D = 128), warps 12-15 dQ reduction (one per TMEM lane
// quarter), so that the compute warps never wait for the dQ product or for
// the reductions to drain into L2. At D = 64 K_j, V_j alternate between two
// buffers by item, so the next item's tiles load during this one.
#include <algorithm>
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
bool make_tmap_f32_acc(CUtensorMap* map, float* base, int BH, int N, int d);

namespace {

using namespace sm103;

constexpr int kTile = 128;          // keys per CTA, queries per step
constexpr int kComputeThreads = 256;

template <int D>
struct BwdCfg {
    // 512 threads in four warpgroups (compute, compute, producer + MMA + two
    // idle warps, dQ reduction), launched at 128 registers a thread; the
    // setmaxnreg budgets below move registers to the compute warps. They must
    // fit in the launch allocation (512 * 128), or .inc would wait forever.
    static constexpr int kThreads = 512;
    static constexpr int kReduceWarp0 = 12;
    static constexpr int kComputeRegs = (D == 64) ? 184 : 168;
    static constexpr int kIssueRegs = (D == 64) ? 40 : 72;
    static constexpr int kReduceRegs = 96;
    static constexpr int kRegBudget = 256 * kComputeRegs + 128 * kIssueRegs + 128 * kReduceRegs;
    static_assert(kRegBudget <= kThreads * 128, "register budgets above the launch allocation");
    static constexpr int kStages = 2;
    static constexpr int kTileBytes = kTile * D * 2;  // one 128 x D 16-bit tile
    // D = 64: K_j, V_j in two buffers alternating by item, so the next
    // item's tiles load while this one runs (D = 128: one, shared memory is
    // full)
    static constexpr int kKvBuffers = (D == 64) ? 2 : 1;
    static constexpr int kKvBytes = 2 * kTileBytes;  // K_j then V_j
    static constexpr int kBoxBytes = kTile * 128;     // 128 rows x 64 columns
    static constexpr int kBoxes = D / 64;
    // a step's stage: Q_i, dO_i and the column table of its 128 queries
    // (-LSE in log2 units, then -delta), loaded together by the TMA engine
    static constexpr int kColBytes = kColTableFloats * 4;
    static constexpr int kStageBytes = 2 * kTileBytes + kColBytes;
    static_assert(kStageBytes % 1024 == 0, "stages keep the swizzled tiles 1024-byte aligned");
    static constexpr int kDsBytes = kTile * kTile * 2;  // dS^T, 128 x 128, 16-bit
    // D = 64 runs the next step's S^T/dP^T products while the current step's
    // dQ product still reads dS^T, so the tile is double-buffered by step
    // parity there
    static constexpr int kDsBuffers = (D == 64) ? 2 : 1;
    // D = 64: dQ leaves through the TMA engine (bulk reduce-add of 32 x 32
    // fp32 boxes staged in shared memory, 4 KB per reduction warp). Row-
    // per-thread reductions there sent 32 scattered L2 requests per
    // instruction through the load/store path, and the compute warps' shared
    // memory accesses queued behind them.
    static constexpr bool kDqBulk = (D == 64);
    static constexpr int kDqStageBytes = kDqBulk ? 4 * 32 * 128 : 0;
    // D = 64: dK, dV leave through TMA stores (issued by warp 11) of two
    // 128 x 64 tiles staged in the item's own K/V buffer, whose products have
    // completed when the accumulators are read; the buffer takes the next
    // K/V tiles once the stores have read it. D = 128 stores rows from the
    // compute warps.
    static constexpr bool kTmaOut = (D == 64);
    // (no alignment slack: the dynamic shared memory window starts 1024-byte
    // aligned, which the kernel checks)
    // block masks: this key tile's list of visible query tiles
    static constexpr int kListCap = (D == 128) ? kMaskListCapBwd128 : kMaskListCap;
    static constexpr int kBarBytes = 512;
    static constexpr int kSmemBase =
        kKvBuffers * kKvBytes + kStages * kStageBytes + kDsBuffers * kDsBytes + kDqStageBytes + kBarBytes;
    static_assert(kSmemBase + kListCap * 2 <= 232448, "shared memory");
    // a persistent CTA with a block mask keeps two item lists (D = 64 only)
    static_assert(D != 64 || kSmemBase + kListCap * 4 <= 232448, "shared memory");
    static constexpr int smem(bool mask, bool ring) { return kSmemBase + (mask ? kListCap * 2 * (ring ? 2 : 1) : 0); }
    static constexpr uint32_t kColS = 0, kColDP = 128;
    // dQ accumulator. D = 128: dQ^T (lanes = head-dim rows, 128 query
    // columns), aliasing dP^T. D = 64: dQ (lanes = query rows, 64 columns).
    static constexpr bool kDqTransposed = (D == 128);
    static constexpr uint32_t kColDQ = (D == 128) ? 128 : 256;
    static constexpr uint32_t kColDV = (D == 128) ? 256 : 320;
    static constexpr uint32_t kColDK = 384;
    // D = 64: P^T (16-bit pairs, 128 keys x 128 queries) in columns of its
    // own, so the next step's S^T may be written while dV still reads P^T
    static constexpr uint32_t kColP = 448;
};


struct BwdParams {
    const float* col_table;  // per (bh, query tile): -LSE log2(e), -delta of its 128 rows
    float* dq_acc;
    void* dk;
    void* dv;
    const uint8_t* block_mask;
    const int32_t* kv_len;
    int* status;
    int H, N, nb;
    int BH, nkt;  // heads x batch, key tiles: the work items are (bh, key tile)
    int* item_ctr;  // persistent grid: items claimed past each CTA's first (zeroed by the preprocess kernel)
    float scale;
    float scale_log2;
    float keep_scale;  // 1/(1-p)
    uint32_t drop_thr;
    int dropout;
    int causal;
    uint64_t seed;
};

struct BwdShared {
    uint64_t kv_full[2];   // K_j, V_j of the item in buffer b loaded
    uint64_t st_full[2];
    uint64_t st_empty[2];
    uint64_t s_full[2];    // D = 128: per 64-query half h, S^T_h and dP^T_h in TMEM; D = 64: [0], the whole tile
    uint64_t p_ready[2];   // P^T_h in TMEM and dS^T_h in shared memory (D = 64: [0], both halves)
    uint64_t s_free;       // D = 64: S^T, dP^T read into the compute warps' registers
    uint64_t p_free;       // D = 64: P^T read by the dV product
    uint64_t dq_full[2];   // dQ of half h (D = 128) / of the tile (D = 64, [0])
    uint64_t dq_free[2];   // that dQ read out of TMEM by the reduction warps
    uint64_t acc_done;
    uint64_t acc_free;     // dK, dV of the item read out of TMEM by the compute warps
    uint64_t kv_empty[2];  // buffer b free: its K_j, V_j read by the item's MMAs (D = 64: and its dK, dV stored)
    uint64_t out_staged[2];  // D = 64: the item's dK, dV tiles staged in K/V buffer b (8 compute warps)
    uint64_t teardown;
    uint64_t list_full[2];  // block mask, persistent: item list of buffer b built
    uint64_t list_free[2];  // ... and released by every warp that reads it
    uint32_t tmem_base;
    int abort_flag;
    int n_list[2];  // block mask: visible query tiles of the item's key tile (per list buffer)
    int ring_item[2];  // persistent grid: the item of ring buffer b (n_items: no more work)
};
static_assert(sizeof(BwdShared) <= 512, "barrier block");

// Query tiles that see key tile j, in increasing order: without a block
// mask (kMask false) the suffix [first, nqt) (first = j when causal), with
// one the list built in shared memory at the start.
template <bool kMask>
struct QSched {
    int jt, nqt, L, causal;
    const uint16_t* list;
    int n_list;
    __device__ bool key_tile_live() const { return jt * kTile < L; }
    // without a block mask the query tiles that see key tile j are the range
    // [j, nqt) under a causal mask (tile i holds a query at or after key
    // 128 j exactly when i >= j) and [0, nqt) otherwise
    __device__ int lo() const { return causal ? jt : 0; }
    __device__ int next(int i) const { return min(max(i, lo()), nqt); }
    __device__ int count() const {
        if (!key_tile_live()) return 0;
        if constexpr (kMask) return n_list;
        return max(nqt - lo(), 0);
    }
    // the first query tile, and the one after i, the k-th (k from 0); nqt
    // past the last
    __device__ int first() const {
        if constexpr (kMask) return n_list > 0 ? (int)list[0] : nqt;
        else return next(0);
    }
    __device__ int after(int i, int k) const {
        if constexpr (kMask) return k + 1 < n_list ? (int)list[k + 1] : nqt;
        else return next(i + 1);
    }
};

// *dst += a (fp32, no return value, relaxed, L2).
__device__ __forceinline__ void red_add_f32(float* dst, float a) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(dst), "f"(a) : "memory");
}


template <typename T, int D, bool kMask, bool kPersist>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
                  const __grid_constant__ CUtensorMap tm_dv, const BwdParams p) {
    using Cfg = BwdCfg<D>;
    // kPersist: a CTA walks several items (persistent grid); otherwise every
    // CTA runs exactly one item. With a block mask and a persistent grid
    // (kRing) each item's list of query tiles goes into one of two buffers
    constexpr bool kRing = kMask && kPersist;
    static_assert(!kRing || D == 64, "two item lists fit in shared memory at D = 64 only");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {  // swizzled tiles need 1024-byte alignment
        if (threadIdx.x == 0 && atomicCAS(p.status, 0, (int)FA_ERR_CUDA) == 0) atomicExch(p.status + 1, 130);
        return;
    }
    uint8_t* sK = smem_raw;  // K/V buffer b: K at sK + b kKvBytes, V kTileBytes after it
    uint8_t* sStages = sK + Cfg::kKvBuffers * Cfg::kKvBytes;
    uint8_t* sDS = sStages + Cfg::kStages * Cfg::kStageBytes;
    uint8_t* sDQ = sDS + Cfg::kDsBuffers * Cfg::kDsBytes;  // D = 64: dQ staging, 4 KB per reduction warp
    BwdShared* st = reinterpret_cast<BwdShared*>(sDQ + Cfg::kDqStageBytes);
    uint16_t* sList = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(st) + Cfg::kBarBytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Work items are (bh, key tile) pairs, item = bh + BH * key tile, so
    // under a causal mask the heaviest key tiles (lowest j) of every head come
    // first. A CTA of the one-item grid takes item = its index. In the
    // persistent grid (one CTA per SM) a CTA's first item is its index too
    // and warp 10 claims each further one from a counter in the workspace, so
    // items go out in order to whichever CTA is free (the balance of the
    // hardware's dispatch, without the CTA set-up between items), and
    // publishes it, with its list of query tiles under a block mask, in one of
    // two alternating buffers that every other role reads before the item;
    // the barriers run on across items, counted by the global step gs + it
    // and the item count gi, so the next item's loads and first products
    // overlap the previous item's last products and its dK/dV stores.
    const int n_items = p.BH * p.nkt;
    const int n_ctas = gridDim.x * gridDim.y;
    const int cta = blockIdx.x + blockIdx.y * gridDim.x;
    const int item0 = cta;
    const int nqt = (p.N + kTile - 1) / kTile;
    auto make_sched = [&](int item, int rr) {
        QSched<kMask> q;
        const int bh_ = item % p.BH;
        q.jt = item / p.BH;
        q.nqt = nqt;
        q.L = p.kv_len ? min(max(p.kv_len[bh_ / p.H], 0), p.N) : p.N;
        q.causal = p.causal;
        q.list = sList + (kRing ? (rr & 1) * Cfg::kListCap : 0);
        q.n_list = 0;
        return q;
    };
    WaitCtx wctx{&st->abort_flag, p.status};
    // block mask (one item per CTA): warp 0 lists the query tiles whose mask
    // block (i, j) is set (strided loads of one mask column and a ballot)
    if (kMask && !kRing && warp == 0 && item0 < n_items) {
        const int jt0 = item0 / p.BH;
        const int first = p.causal ? jt0 : 0;
        const int cnt = warp_list_visible(p.block_mask + jt0, (size_t)p.nb, first, nqt, sList, lane);
        if (lane == 0) st->n_list[0] = cnt;
    }

    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&st->kv_full[b], 1);
            mbar_init(&st->kv_empty[b], Cfg::kTmaOut ? 2 : 1);  // the MMA commit (+ warp 11 after the stores)
            mbar_init(&st->out_staged[b], kComputeThreads / 32);
        }
        for (int s = 0; s < Cfg::kStages; ++s) {
            mbar_init(&st->st_full[s], 1);
            mbar_init(&st->st_empty[s], 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(&st->s_full[h], 1);
            mbar_init(&st->p_ready[h], kComputeThreads / (D == 64 ? 32 : 64));
            mbar_init(&st->dq_full[h], 1);
            mbar_init(&st->dq_free[h], kComputeThreads / 64);
        }
        mbar_init(&st->s_free, kComputeThreads / 32);
        mbar_init(&st->p_free, 1);
        mbar_init(&st->acc_done, 1);
        mbar_init(&st->acc_free, kComputeThreads / 32);
        mbar_init(&st->teardown, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&st->list_full[b], 1);
            // producer, MMA, 8 compute and 4 reduction warps (+ warp 11, the
            // dK/dV store warp at D = 64)
            mbar_init(&st->list_free[b], Cfg::kTmaOut ? 15 : 14);
        }
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
    // the item's query-step schedule and number of steps
    auto item_sched = [&](int item, int rr, int& n_active) {
        QSched<kMask> q = make_sched(item, rr);
        if constexpr (kMask) q.n_list = st->n_list[kRing ? (rr & 1) : 0];
        n_active = q.count();
        return q;
    };
    // persistent grid: before its rr-th item a reading warp releases ring
    // buffer (rr - 1) & 1 and waits until buffer rr & 1 holds the next item
    // (one thread per warp arrives; the producer's loop runs on one lane)
    auto list_acquire = [&](int rr, bool warp_wide) -> bool {
        if constexpr (!kPersist) return true;
        if (rr > 0) {
            if (warp_wide) mbar_arrive_warp(&st->list_free[(rr - 1) & 1]);
            else mbar_arrive(&st->list_free[(rr - 1) & 1]);
        }
        return warp_wide ? mbar_wait_warp(&st->list_full[rr & 1], (rr >> 1) & 1, wctx, 140)
                         : mbar_wait(&st->list_full[rr & 1], (rr >> 1) & 1, wctx, 140);
    };
    // The next kernel (dq conversion) may start launching once every CTA is
    // here. Q, K, V, dO and LSE were complete before the preprocess kernel
    // ran, so the producer and MMA warps start at once; the compute and
    // reduction warps wait for the preprocess kernel (delta, dQacc = 0).
    pdl_trigger();

    if (warp == 8) {
        // ------------------------------------------------------------ producer
        regs_dec<Cfg::kIssueRegs>();
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_do);
            // bit s: a load was issued into stage s / the phase of its last one
            uint32_t issued_any = 0, issued_phase = 0;
            bool okp = true;
            bool pre_done = false;  // the preprocess kernel's column table is visible
            int gs = 0, gi = 0;  // steps and items with work, so far
            for (int rr = 0; okp && (kPersist || rr == 0); ++rr) {
                if (!list_acquire(rr, false)) break;
                const int item = kPersist ? st->ring_item[rr & 1] : item0;
                if (item >= n_items) break;
                int n_active;
                const QSched<kMask> sched = item_sched(item, rr, n_active);
                if (n_active == 0) continue;
                const int bh = item % p.BH;
                const int j0 = sched.jt * kTile;
                // Q_i, dO_i and the column table of query tile i, step t
                // (global step gs + t), into its stage
                auto load_step = [&](int i, int t) -> bool {
                    const int g = gs + t;
                    const int s = g % Cfg::kStages;
                    const uint32_t ph = (g / Cfg::kStages) & 1;
                    if (!mbar_wait(&st->st_empty[s], ph ^ 1, wctx, 101)) return false;
                    mbar_arrive_expect_tx(&st->st_full[s], Cfg::kStageBytes);
                    uint8_t* dq = sStages + s * Cfg::kStageBytes;
                    uint8_t* ddo = dq + Cfg::kTileBytes;
#pragma unroll
                    for (int x = 0; x < Cfg::kBoxes; ++x) {
                        tma_load_3d(dq + x * Cfg::kBoxBytes, &tm_q, &st->st_full[s], x * 64, i * kTile, bh);
                        tma_load_3d(ddo + x * Cfg::kBoxBytes, &tm_do, &st->st_full[s], x * 64, i * kTile, bh);
                    }
                    // the table is written by the preprocess kernel: the first
                    // copy waits for it (Q_i, dO_i are already on their way)
                    if (!pre_done) {
                        pdl_wait();
                        pre_done = true;
                    }
                    bulk_load_1d(dq + 2 * Cfg::kTileBytes, p.col_table + ((size_t)bh * nqt + i) * kColTableFloats,
                                 Cfg::kColBytes, &st->st_full[s]);
                    issued_phase = (issued_phase & ~(1u << s)) | (ph << s);
                    issued_any |= 1u << s;
                    return true;
                };
                // With one K/V buffer the item's first Q_i, dO_i go ahead of
                // K_j, V_j (their stage frees before the previous item's last
                // MMA has run); with two, K_j and V_j go first, into buffer
                // gi % 2, which the item before the previous one has released
                // long before.
                int i = sched.first();
                int t0 = 0;
                if constexpr (Cfg::kKvBuffers == 1) {
                    if (!load_step(i, 0)) break;
                    i = sched.after(i, 0);
                    t0 = 1;
                }
                const int kb = gi % Cfg::kKvBuffers;
                const int g_prev = gi - Cfg::kKvBuffers;  // the item that last used buffer kb
                if (g_prev >= 0 && !mbar_wait(&st->kv_empty[kb], (g_prev / Cfg::kKvBuffers) & 1, wctx, 104)) break;
                mbar_arrive_expect_tx(&st->kv_full[kb], Cfg::kKvBytes);
                uint8_t* kv = sK + kb * Cfg::kKvBytes;
#pragma unroll
                for (int x = 0; x < Cfg::kBoxes; ++x) {
                    tma_load_3d(kv + x * Cfg::kBoxBytes, &tm_k, &st->kv_full[kb], x * 64, j0, bh);
                    tma_load_3d(kv + Cfg::kTileBytes + x * Cfg::kBoxBytes, &tm_v, &st->kv_full[kb], x * 64, j0, bh);
                }
                for (int t = t0; i < sched.nqt; i = sched.after(i, t), ++t) {
                    if (!load_step(i, t)) {
                        okp = false;
                        break;
                    }
                }
                gs += n_active;
                ++gi;
            }
            // drain: the last load issued into each stage, and the last K/V
            for (int s = 0; s < Cfg::kStages; ++s)
                if ((issued_any >> s) & 1u) mbar_wait(&st->st_full[s], (issued_phase >> s) & 1u, wctx, 102);
            if (gi > 0) mbar_wait(&st->kv_full[(gi - 1) % Cfg::kKvBuffers], ((gi - 1) / Cfg::kKvBuffers) & 1, wctx, 103);
        }
    } else if (warp == 10 || warp == 11) {
        // the rest of the producer / MMA warpgroup. In the persistent grid
        // warp 10 fills the item ring: buffer rr & 1, once every reader has
        // released the item before it there (rr - 2), gets the CTA's rr-th
        // item (its index for rr = 0, then claimed from the counter, n_items
        // once none is left) and, with a block mask, the item's query tiles.
        // Warp 11 is idle.
        regs_dec<Cfg::kIssueRegs>();
        if constexpr (kPersist) {
            if (warp == 10) {
                for (int rr = 0;; ++rr) {
                    if (rr >= 2 && !mbar_wait_warp(&st->list_free[rr & 1], ((rr - 2) >> 1) & 1, wctx, 141)) break;
                    int item = item0;
                    if (rr > 0) {
                        if (rr == 1) pdl_wait();  // the counter is zeroed by the preprocess kernel
                        int claimed = 0;
                        if (lane == 0) claimed = atomicAdd(p.item_ctr, 1);
                        item = n_ctas + __shfl_sync(0xffffffffu, claimed, 0);
                    }
                    item = min(item, n_items);
                    if (kMask && item < n_items) {
                        const int jt = item / p.BH;
                        const int cnt = warp_list_visible(p.block_mask + jt, (size_t)p.nb, p.causal ? jt : 0, nqt,
                                                          sList + (rr & 1) * Cfg::kListCap, lane);
                        if (lane == 0) st->n_list[rr & 1] = cnt;
                    }
                    if (lane == 0) st->ring_item[rr & 1] = item;
                    mbar_arrive_warp(&st->list_full[rr & 1]);
                    if (item >= n_items) break;
                }
            }
        }
        if constexpr (Cfg::kTmaOut) {
            if (warp == 11) {
                // dK/dV stores: per item with work, once the compute warps have
                // staged the tiles in the item's K/V buffer, two TMA stores
                // (rows past N are outside the tensor and not written); the
                // buffer is released to the producer when they have read it
                if (lane == 0) {
                    prefetch_tmap(&tm_dk);
                    prefetch_tmap(&tm_dv);
                }
                int gi = 0;  // items with work, so far
                for (int rr = 0; kPersist || rr == 0; ++rr) {
                    if (!list_acquire(rr, true)) break;
                    const int item = kPersist ? st->ring_item[rr & 1] : item0;
                    if (item >= n_items) break;
                    int n_active;
                    const QSched<kMask> sched = item_sched(item, rr, n_active);
                    if (n_active == 0) continue;
                    const int kb = gi % Cfg::kKvBuffers;
                    if (!mbar_wait_warp(&st->out_staged[kb], (gi / Cfg::kKvBuffers) & 1, wctx, 127)) break;
                    if (lane == 0) {
                        uint8_t* kv = sK + kb * Cfg::kKvBytes;
                        tma_store_3d(&tm_dk, kv, 0, sched.jt * kTile, item % p.BH);
                        tma_store_3d(&tm_dv, kv + Cfg::kTileBytes, 0, sched.jt * kTile, item % p.BH);
                        bulk_commit_group();
                        bulk_wait_read();
                    }
                    __syncwarp();
                    mbar_arrive_warp(&st->kv_empty[kb]);
                    ++gi;
                }
                // the stores have completed before the CTA ends
                if (lane == 0) bulk_wait_all();
            }
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        regs_dec<Cfg::kIssueRegs>();
        // the whole warp runs the issue loop; one elected lane issues
        {
            constexpr uint32_t id_sh = idesc_f32acc(Elem16<T>::kFmt, kTile, 64, 0, 0);      // S^T_h, dP^T_h (N = 64)
            constexpr uint32_t id_dv = idesc_f32acc(Elem16<T>::kFmt, kTile, D, 0, 1);      // dV (A tmem), dK (A K-major)
            constexpr uint32_t id_dqt_h = idesc_f32acc(Elem16<T>::kFmt, kTile, 64, 1, 1);   // dQ^T_h (A, B MN-major, N = 64)
            constexpr uint32_t id_dq = idesc_f32acc(Elem16<T>::kFmt, kTile, D, 1, 1);       // dQ (A, B MN-major)
            const uint32_t ds_base = smem_u32(sDS);
            // descriptors built once (K and V per item, from the item's
            // buffer), advanced by constants per MMA
            const uint64_t dsd_k = smem_desc_sw128(ds_base, 16, 1024);       // dS^T, K-major
            const uint64_t dsd_mn = smem_desc_sw128(ds_base, kTile * 128, 1024);  // dS^T, MN-major
            bool ok = true;
            int gs = 0, gi = 0;  // steps and items with work, so far
            for (int rr = 0; ok && (kPersist || rr == 0); ++rr) {
            if (!list_acquire(rr, true)) break;
            const int item = kPersist ? st->ring_item[rr & 1] : item0;
            if (item >= n_items) break;
            int n_active;
            (void)item_sched(item, rr, n_active);
            if (n_active == 0) continue;
            const int kb = gi % Cfg::kKvBuffers;
            if (!mbar_wait_warp(&st->kv_full[kb], (gi / Cfg::kKvBuffers) & 1, wctx, 110)) break;
            tc_fence_after();
            const uint32_t k_base = smem_u32(sK + kb * Cfg::kKvBytes), v_base = k_base + Cfg::kTileBytes;
            const uint64_t kd_k = smem_desc_sw128(k_base, 16, 1024);               // K, K-major
            const uint64_t vd_k = smem_desc_sw128(v_base, 16, 1024);               // V, K-major
            const uint64_t kd_mn = smem_desc_sw128(k_base, Cfg::kBoxBytes, 1024);  // K, MN-major (N = d)
            const uint64_t kd_mn2 = smem_desc_sw128(k_base, kTile * 128, 1024);    // K, MN-major (M = d)
            if constexpr (D == 64) {
            // Software-pipelined order: the next step's S^T, dP^T (over all
            // 128 queries, N = 128) are issued as soon as the compute warps
            // have read this step's into registers (s_free), ahead of this
            // step's gradient products, so the compute warps work on step
            // t + 1 while the tensor core runs dV, dK, dQ of step t:
            //   [S dP](t+1) [dV dK dQ](t) [S dP](t+2) [dV dK dQ](t+1) ...
            // P^T has TMEM columns of its own; the compute warps write P^T of
            // step t + 1 once dV(t) has read P^T(t) (p_free). dS^T alternates
            // between two shared-memory tiles by step parity: dK, dQ of step t
            // read their tile while step t + 1 writes the other, and step
            // t + 2 writes it again only after S^T(t + 2), issued after dQ(t),
            // is complete.
            constexpr uint32_t id_s = idesc_f32acc(Elem16<T>::kFmt, kTile, kTile, 0, 0);  // S^T, dP^T (N = 128)
            auto issue_sdp = [&](int g2) {  // g2: global step
                const uint32_t qb = smem_u32(sStages + (g2 % Cfg::kStages) * Cfg::kStageBytes);
                const uint64_t qk = smem_desc_sw128(qb, 16, 1024);
                const uint64_t dk = smem_desc_sw128(qb + Cfg::kTileBytes, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss_warp(tmem + Cfg::kColS, desc_add(kd_k, kk * 32), desc_add(qk, kk * 32), id_s, kk > 0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_ss_warp(tmem + Cfg::kColDP, desc_add(vd_k, kk * 32), desc_add(dk, kk * 32), id_s, kk > 0);
                mma_commit_warp(&st->s_full[0]);
            };
            if (ok) ok = mbar_wait_warp(&st->st_full[gs % Cfg::kStages], (gs / Cfg::kStages) & 1, wctx, 111);
            if (ok) {
                tc_fence_after();
                issue_sdp(gs);
            }
            for (int it = 0; ok && it < n_active; ++it) {
                const int g = gs + it;
                const int s = g % Cfg::kStages;
                const uint32_t q_base = smem_u32(sStages + s * Cfg::kStageBytes);
                const uint32_t do_base = q_base + Cfg::kTileBytes;
                const uint64_t qd_mn = smem_desc_sw128(q_base, Cfg::kBoxBytes, 1024);
                const uint64_t dod_mn = smem_desc_sw128(do_base, Cfg::kBoxBytes, 1024);
                const uint32_t dsb = (uint32_t)((g & 1) * Cfg::kDsBytes);
                if (it + 1 < n_active) {
                    const int s1 = (g + 1) % Cfg::kStages;
                    if (!mbar_wait_warp(&st->s_free, g & 1, wctx, 117) ||
                        !mbar_wait_warp(&st->st_full[s1], ((g + 1) / Cfg::kStages) & 1, wctx, 111)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_sdp(g + 1);
                }
                if (!mbar_wait_warp(&st->p_ready[0], g & 1, wctx, 113)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // the item's first products overwrite dV, dK: the compute
                // warps must have read out the previous item's
                if (it == 0 && gi > 0) {
                    if (!mbar_wait_warp(&st->acc_free, (gi - 1) & 1, wctx, 116)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                const uint32_t acc = (it > 0) ? 1u : 0u;
                // dV += P^T dO (A from TMEM: query columns 16 kk.. of P^T in
                // packed columns 8 kk..), then dK += dS^T Q (dS^T query half
                // kk / 4 is shared-memory box kk / 4)
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk)
                    mma_ts_warp(tmem + Cfg::kColDV, tmem + Cfg::kColP + kk * 8, desc_add(dod_mn, kk * 2048), id_dv,
                                (acc || kk > 0) ? 1u : 0u);
                mma_commit_warp(&st->p_free);
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk)
                    mma_ss_warp(tmem + Cfg::kColDK, desc_add(dsd_k, dsb + (kk >> 2) * (kTile * 128) + (kk & 3) * 32),
                                desc_add(qd_mn, kk * 2048), id_dv, (acc || kk > 0) ? 1u : 0u);
                mma_commit_warp(&st->st_empty[s]);  // Q_i, dO_i read
                // dQ = dS K_j over the whole tile, over the previous step's dQ
                // once it has been read out
                if (g > 0) {
                    if (!mbar_wait_warp(&st->dq_free[0], (g - 1) & 1, wctx, 115)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk)
                    mma_ss_warp(tmem + Cfg::kColDQ, desc_add(dsd_mn, dsb + kk * 2048), desc_add(kd_mn, kk * 2048), id_dq,
                                kk > 0);
                mma_commit_warp(&st->dq_full[0]);
            }
            } else {
            // D = 128: per 64-query half h, S^T_h = K_j Q_{i,h}^T and
            // dP^T_h = V_j dO_{i,h}^T (N = 64); half 1's products run while
            // the compute warps of half 0 work, and half 0's gradient MMAs
            // while half 1's do. dP^T_h overwrites the previous step's dQ^T_h
            // once the reduction warps have read it out.
            for (int it = 0; ok && it < n_active; ++it) {
                const int g = gs + it;
                const int s = g % Cfg::kStages;
                if (!mbar_wait_warp(&st->st_full[s], (g / Cfg::kStages) & 1, wctx, 111)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t q_base = smem_u32(sStages + s * Cfg::kStageBytes);
                const uint32_t do_base = q_base + Cfg::kTileBytes;
                const uint64_t qd_k = smem_desc_sw128(q_base, 16, 1024);
                const uint64_t dod_k = smem_desc_sw128(do_base, 16, 1024);
                const uint64_t qd_mn = smem_desc_sw128(q_base, Cfg::kBoxBytes, 1024);
                const uint64_t dod_mn = smem_desc_sw128(do_base, Cfg::kBoxBytes, 1024);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk / 4) * Cfg::kBoxBytes + (kk % 4) * 32;
                        mma_ss_warp(tmem + Cfg::kColS + 64 * h, desc_add(kd_k, off), desc_add(qd_k, off + 8192 * h), id_sh,
                               kk > 0);
                    }
                    if (g > 0) {
                        if (!mbar_wait_warp(&st->dq_free[h], (g - 1) & 1, wctx, 112)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk / 4) * Cfg::kBoxBytes + (kk % 4) * 32;
                        mma_ss_warp(tmem + Cfg::kColDP + 64 * h, desc_add(vd_k, off), desc_add(dod_k, off + 8192 * h), id_sh,
                               kk > 0);
                    }
                    mma_commit_warp(&st->s_full[h]);
                }
                if (!ok) break;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (!mbar_wait_warp(&st->p_ready[h], g & 1, wctx, 113)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // the item's first products overwrite dV, dK: the compute
                    // warps must have read out the previous item's
                    if (it == 0 && h == 0 && gi > 0) {
                        if (!mbar_wait_warp(&st->acc_free, (gi - 1) & 1, wctx, 116)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    // dV += P^T_h dO_h (P^T_h, 16-bit, in TMEM columns
                    // 64h..64h+31) and dK += dS^T_h Q_h (dS^T half h is
                    // shared-memory box h), interleaved with
                    // dQ^T_h = K_j^T dS^T_h (M = head dim, N = 64 queries:
                    // lane = head-dim index, so one reduction instruction
                    // covers 32 consecutive floats of a row) so that
                    // consecutive MMAs go to different accumulators
                    const uint32_t acc = (it > 0 || h > 0) ? 1u : 0u;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        mma_ts_warp(tmem + Cfg::kColDV, tmem + Cfg::kColS + 64 * h + kk * 8,
                                    desc_add(dod_mn, 8192 * h + kk * 2048), id_dv, (acc || kk > 0) ? 1u : 0u);
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int k2 = 2 * kk + e;
                            mma_ss_warp(tmem + Cfg::kColDQ + 64 * h, desc_add(kd_mn2, k2 * 2048),
                                        desc_add(dsd_mn, h * (kTile * 128) + k2 * 2048), id_dqt_h, k2 > 0);
                            if (e == 0)
                                mma_ss_warp(tmem + Cfg::kColDK, desc_add(dsd_k, h * (kTile * 128) + kk * 32),
                                            desc_add(qd_mn, 8192 * h + kk * 2048), id_dv, (acc || kk > 0) ? 1u : 0u);
                        }
                    }
                    if (h == 1) mma_commit_warp(&st->st_empty[s]);  // Q_i, dO_i read
                    mma_commit_warp(&st->dq_full[h]);
                }
            }
            }
            // the item's K_j, V_j are read by every MMA issued so far; dK, dV
            // are complete when these arrive
            mma_commit_warp(&st->kv_empty[kb]);
            mma_commit_warp(&st->acc_done);
            gs += n_active;
            ++gi;
            }
            if (gi > 0) {
                mma_commit_warp(&st->teardown);
                mbar_wait_warp(&st->teardown, 0, wctx, 114);
            }
        }
    } else if (warp >= Cfg::kReduceWarp0) {
        // ------------------------------------------------------------ dQ reduction
        regs_dec<Cfg::kReduceRegs>();
        // D = 128: dQ^T, lane = head-dim index, so one reduction instruction
        // covers 32 consecutive floats of one query row. D = 64: dQ, lane =
        // query row, added by bulk tensor reductions (below).
        const int quarter = warp & 3;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const int r = quarter * 32 + lane;
        bool ok = true;
        int gs = 0;  // steps with work, so far
        uint8_t* dq_buf = sDQ + quarter * 4096;  // D = 64: this warp's 32 x 32 fp32 box
        if (Cfg::kDqBulk && lane == 0) prefetch_tmap(&tm_dq);
        pdl_wait();
        for (int rr = 0; ok && (kPersist || rr == 0); ++rr) {
        if (!list_acquire(rr, true)) break;
        const int item = kPersist ? st->ring_item[rr & 1] : item0;
        if (item >= n_items) break;
        int n_active;
        const QSched<kMask> sched = item_sched(item, rr, n_active);
        if (n_active == 0) continue;
        const int bh = item % p.BH;
        int it = 0;
        for (int i = sched.first(); ok && i < sched.nqt; i = sched.after(i, it), ++it) {
            const int g = gs + it;
            const int i0 = i * kTile;
            const int nvalid = min(kTile, p.N - i0);
#pragma unroll
            for (int h = 0; h < (Cfg::kDqTransposed ? 2 : 1); ++h) {
                if (!mbar_wait_warp(&st->dq_full[h], g & 1, wctx, 121)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // read out, release the TMEM (the next dP^T / dQ may
                // overwrite it), then reduce
                uint32_t qa[32], qb[32];
                tmem_ld32(tmem + lane_base + Cfg::kColDQ + h * 64, qa);
                tmem_ld32(tmem + lane_base + Cfg::kColDQ + h * 64 + 32, qb);
                tmem_ld_wait();
                reg_fence(qa);
                reg_fence(qb);
                tc_fence_before();
                mbar_arrive_warp(&st->dq_free[h]);
                if (Cfg::kDqTransposed) {
                    float* dst = p.dq_acc + ((size_t)bh * p.N + i0 + h * 64) * D + r;
#pragma unroll
                    for (int x = 0; x < 32; ++x)
                        if (h * 64 + x < nvalid) red_add_f32(dst + (size_t)x * D, __uint_as_float(qa[x]));
#pragma unroll
                    for (int x = 0; x < 32; ++x)
                        if (h * 64 + 32 + x < nvalid) red_add_f32(dst + (size_t)(32 + x) * D, __uint_as_float(qb[x]));
                } else if (Cfg::kDqBulk) {
                    // this warp's 32 query rows in two boxes of 32 columns,
                    // each staged with the 128-byte swizzle (16-byte chunk c
                    // of row x at chunk position c ^ (x & 7)) and added into
                    // the accumulator by the TMA engine; rows past N are
                    // outside the tensor map and skipped
                    if (quarter * 32 < nvalid) {
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            const uint32_t* q = c ? qb : qa;
                            if (lane == 0) bulk_wait_read();  // the previous box has been read
                            __syncwarp();
#pragma unroll
                            for (int v = 0; v < 8; ++v)
                                *reinterpret_cast<uint4*>(dq_buf + lane * 128 + ((v ^ (lane & 7)) << 4)) =
                                    make_uint4(q[4 * v], q[4 * v + 1], q[4 * v + 2], q[4 * v + 3]);
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tma_reduce_add_3d(&tm_dq, dq_buf, 32 * c, i0 + quarter * 32, bh);
                                bulk_commit_group();
                            }
                        }
                    }
                }
            }
        }
        gs += n_active;
        }
        // the accumulator writes are complete before the CTA ends
        if (Cfg::kDqBulk && lane == 0) bulk_wait_all();
    } else {
        // ------------------------------------------------------------ compute
        regs_inc<Cfg::kComputeRegs>();
        const int quarter = warp & 3;      // TMEM lane quarter
        const int half = warp >> 2;        // query columns [64*half, 64*half + 64)
        const int r = quarter * 32 + lane;  // key row within the tile
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        bool ok = true;
        int gs = 0, gi = 0;  // steps and items with work, so far
        for (int rr = 0; ok && (kPersist || rr == 0); ++rr) {
        if (!list_acquire(rr, true)) {
            ok = false;
            break;
        }
        const int item = kPersist ? st->ring_item[rr & 1] : item0;
        if (item >= n_items) break;
        int n_active;
        const QSched<kMask> sched = item_sched(item, rr, n_active);
        const int bh = item % p.BH;
        const int b = bh / p.H, h = bh % p.H;
        const int j0 = sched.jt * kTile;
        const int jrow = j0 + r;
        const bool key_ok = jrow < sched.L;
        if (n_active == 0) {
            // no query sees this key tile: dK = dV = 0 on its rows
            if (jrow < p.N) {
#pragma unroll
                for (int which = 0; which < 2; ++which) {
                    T* out = static_cast<T*>(which ? p.dv : p.dk) + ((size_t)bh * p.N + jrow) * D;
                    uint4* dst = reinterpret_cast<uint4*>(out + half * (D / 2));
#pragma unroll
                    for (int v = 0; v < D / 16; ++v) dst[v] = make_uint4(0, 0, 0, 0);
                }
            }
            continue;
        }
        int it = 0;
        for (int i = sched.first(); i < sched.nqt; ++it) {
            const int g = gs + it;
            const int i0 = i * kTile;
            const int i_next = sched.after(i, it);
            // per-query -LSE (log2 units; -inf for masked rows and rows past
            // N, so P = 0) and -delta, negated so that each pair of columns
            // takes one paired fma / add: the column table in the step's
            // stage, loaded with Q_i and dO_i
            const int sidx = g % Cfg::kStages;
            const float* colt = reinterpret_cast<const float*>(sStages + sidx * Cfg::kStageBytes + 2 * Cfg::kTileBytes);
            // dropout keep bits of this row's 64 query columns, drawn before
            // S^T arrives (bit x of keep_w[ch] is query column
            // 64 half + 32 ch + x). Lane (4a + w) draws, for the 8 queries
            // 4g + w of each 32-column chunk, the 4 keep bits of keys
            // 4a..4a+3 and packs them into one word (bits 4g..4g+3); the key
            // of lane 4a + w for query 4g + q is then bit 4g + w of lane
            // 4a + q's word, so one shuffle per group mate moves all of them
            uint32_t keep_w[2] = {0xffffffffu, 0xffffffffu};
            if (p.dropout) {
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    const int cb = half * 64 + ch * 32;
                    uint32_t word = 0;
#pragma unroll
                    for (int g = 0; g < 8; ++g) {
                        const int qi = i0 + cb + 4 * g + (lane & 3);
                        word |= keep_bits4(p.seed, p.drop_thr, b, h, qi, jrow >> 2) << (4 * g);
                    }
                    uint32_t keep = 0;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t v = __shfl_sync(0xffffffffu, word, (lane & ~3) | q);
                        keep |= ((v >> (lane & 3)) & 0x11111111u) << q;
                    }
                    keep_w[ch] = keep;
                }
            }
            if (!mbar_wait_warp(&st->s_full[D == 64 ? 0 : half], g & 1, wctx, 120) ||
                !mbar_wait_warp(&st->st_full[sidx], (g / Cfg::kStages) & 1, wctx, 123)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // visible queries of this key row form a suffix [cmin, 128) of the tile
            int cmin = 0;
            if (p.causal) cmin = max(0, jrow - i0);
            const int cmax = key_ok ? min(kTile, p.N - i0) : 0;
            // at D = 64 both chunks of S^T and dP^T are loaded with one TMEM
            // wait (the registers allow it there); at D = 128 one chunk at a
            // time
            constexpr bool kLoadBoth = (D == 64);
            uint32_t sr2[2][32], dr2[2][32];
            // D = 64: both chunks' P^T (TMEM) and dS^T (shared memory) are
            // stored after the second chunk is computed, so that the second
            // chunk's shared-memory reads of LSE and delta do not queue
            // behind the first chunk's stores; the 16-bit results are packed
            // in place over the scores they came from (P^T pairs into S^T's
            // registers, dS^T pairs into dP^T's: pair x/2 is written once
            // elements x..x+3 are read), which leaves the compiler the
            // registers to load LSE and delta ahead of their use. D = 128
            // packs one chunk at a time into separate arrays.
            uint32_t pk2[1][16];
            uint32_t dsk2[1][16];
            if constexpr (kLoadBoth) {
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    tmem_ld32(tmem + lane_base + Cfg::kColS + half * 64 + ch * 32, sr2[ch]);
                    tmem_ld32(tmem + lane_base + Cfg::kColDP + half * 64 + ch * 32, dr2[ch]);
                }
                tmem_ld_wait();
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    reg_fence(sr2[ch]);
                    reg_fence(dr2[ch]);
                }
                // S^T, dP^T are in registers: the next step's may be written
                tc_fence_before();
                mbar_arrive_warp(&st->s_free);
            }
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
                const int cb = half * 64 + ch * 32;  // first query column of this chunk
                uint32_t(&sr)[32] = sr2[ch];
                uint32_t(&dr)[32] = dr2[ch];
                if constexpr (!kLoadBoth) {
                    tmem_ld32(tmem + lane_base + Cfg::kColS + cb, sr);
                    tmem_ld32(tmem + lane_base + Cfg::kColDP + cb, dr);
                    tmem_ld_wait();
                    reg_fence(sr);
                    reg_fence(dr);
                }
                const uint32_t keep = keep_w[ch];
                const bool edge = (cmin > cb) || (cmax < cb + 32);
                uint32_t(&pk)[16] = pk2[0];
                uint32_t(&dsk)[16] = dsk2[0];
                auto put = [&](int idx, uint32_t pv, uint32_t dv) {
                    if constexpr (kLoadBoth) {
                        sr[idx] = pv;
                        dr[idx] = dv;
                    } else {
                        pk[idx] = pv;
                        dsk[idx] = dv;
                    }
                };
                // columns outside [cmin, cmax) (causal diagonal, key padding,
                // sequence end) are zeroed in S first, so the element loop
                // below carries no per-element mask test
                if (edge) {
#pragma unroll
                    for (int x = 0; x < 32; ++x)
                        if (cb + x < cmin || cb + x >= cmax) sr[x] = __float_as_uint(-INFINITY);
                }
                const float sl2 = p.scale_log2;
                if (!p.dropout) {
#pragma unroll
                    for (int x = 0; x < 32; x += 4) {
                        const float4 l4 = *reinterpret_cast<const float4*>(colt + cb + x);
                        const float4 d4 = *reinterpret_cast<const float4*>(colt + kTile + cb + x);
                        float a[4], e[4], t[4], g[4];
                        ffma2(a[0], a[1], __uint_as_float(sr[x]), __uint_as_float(sr[x + 1]), sl2, sl2, l4.x, l4.y);
                        ffma2(a[2], a[3], __uint_as_float(sr[x + 2]), __uint_as_float(sr[x + 3]), sl2, sl2, l4.z, l4.w);
#pragma unroll
                        for (int y = 0; y < 4; ++y) e[y] = ex2_approx(a[y]);
                        // dS = P (dP - delta)
                        fadd2(t[0], t[1], __uint_as_float(dr[x]), __uint_as_float(dr[x + 1]), d4.x, d4.y);
                        fadd2(t[2], t[3], __uint_as_float(dr[x + 2]), __uint_as_float(dr[x + 3]), d4.z, d4.w);
                        fmul2(g[0], g[1], e[0], e[1], t[0], t[1]);
                        fmul2(g[2], g[3], e[2], e[3], t[2], t[3]);
                        put(x / 2, Elem16<T>::pack2(e[0], e[1]), Elem16<T>::pack2(g[0], g[1]));
                        put(x / 2 + 1, Elem16<T>::pack2(e[2], e[3]), Elem16<T>::pack2(g[2], g[3]));
                    }
                } else {
#pragma unroll
                    for (int x = 0; x < 32; x += 4) {
                        const float4 l4 = *reinterpret_cast<const float4*>(colt + cb + x);
                        const float4 d4 = *reinterpret_cast<const float4*>(colt + kTile + cb + x);
                        float a[4], e[4], z[4], t[4], g[4], pv[4];
                        ffma2(a[0], a[1], __uint_as_float(sr[x]), __uint_as_float(sr[x + 1]), sl2, sl2, l4.x, l4.y);
                        ffma2(a[2], a[3], __uint_as_float(sr[x + 2]), __uint_as_float(sr[x + 3]), sl2, sl2, l4.z, l4.w);
#pragma unroll
                        for (int y = 0; y < 4; ++y) {
                            e[y] = ex2_approx(a[y]);
                            z[y] = ((keep >> (x + y)) & 1u) ? p.keep_scale : 0.f;
                        }
                        // P^ = P Z/(1-p);  dS = P (dP Z/(1-p) - delta)
                        fmul2(pv[0], pv[1], e[0], e[1], z[0], z[1]);
                        fmul2(pv[2], pv[3], e[2], e[3], z[2], z[3]);
                        ffma2(t[0], t[1], __uint_as_float(dr[x]), __uint_as_float(dr[x + 1]), z[0], z[1], d4.x, d4.y);
                        ffma2(t[2], t[3], __uint_as_float(dr[x + 2]), __uint_as_float(dr[x + 3]), z[2], z[3], d4.z, d4.w);
                        fmul2(g[0], g[1], e[0], e[1], t[0], t[1]);
                        fmul2(g[2], g[3], e[2], e[3], t[2], t[3]);
                        put(x / 2, Elem16<T>::pack2(pv[0], pv[1]), Elem16<T>::pack2(g[0], g[1]));
                        put(x / 2 + 1, Elem16<T>::pack2(pv[2], pv[3]), Elem16<T>::pack2(g[2], g[3]));
                    }
                }
                // P^T into TMEM columns this warp has already read
                if constexpr (!kLoadBoth) tmem_st16(tmem + lane_base + Cfg::kColS + half * 64 + ch * 16, pk);
                // dS^T row r, queries cb..cb+31: 4 swizzled 16-byte chunks
                uint8_t* row = sDS + (g & (Cfg::kDsBuffers - 1)) * Cfg::kDsBytes + half * (kTile * 128) + r * 128;
                if constexpr (!kLoadBoth) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const int chunk = ch * 4 + v;
                        uint4 w4 = make_uint4(dsk[4 * v], dsk[4 * v + 1], dsk[4 * v + 2], dsk[4 * v + 3]);
                        *reinterpret_cast<uint4*>(row + ((chunk ^ (r & 7)) << 4)) = w4;
                    }
                }
            }
            if constexpr (kLoadBoth) {
                // dS^T first (its buffer is free since S^T of this step
                // completed), then P^T (own columns: query column c in packed
                // column c / 2) once the previous step's dV product has read it
                uint8_t* row = sDS + (g & (Cfg::kDsBuffers - 1)) * Cfg::kDsBytes + half * (kTile * 128) + r * 128;
#pragma unroll
                for (int chunk = 0; chunk < 8; ++chunk) {
                    const uint32_t* d4 = &dr2[chunk >> 2][4 * (chunk & 3)];
                    *reinterpret_cast<uint4*>(row + ((chunk ^ (r & 7)) << 4)) = make_uint4(d4[0], d4[1], d4[2], d4[3]);
                }
                if (g > 0) {
                    if (!mbar_wait_warp(&st->p_free, (g - 1) & 1, wctx, 124)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
#pragma unroll
                for (int ch = 0; ch < 2; ++ch)
                    tmem_st16(tmem + lane_base + Cfg::kColP + half * 32 + ch * 16,
                              *reinterpret_cast<const uint32_t(*)[16]>(&sr2[ch][0]));
            }
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive_warp(&st->p_ready[D == 64 ? 0 : half]);
            i = i_next;
        }
        if (!ok) break;
        // epilogue: dK = scale * acc, dV = acc, rows of this key tile. The
        // accumulators are read out of TMEM and released (acc_free) before
        // the stores, so the next item's products can start meanwhile.
        if (!mbar_wait_warp(&st->acc_done, gi & 1, wctx, 122)) {
            ok = false;
            break;
        }
        tc_fence_after();
        uint32_t ar[2][D / 64][32];
#pragma unroll
        for (int which = 0; which < 2; ++which)
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
                tmem_ld32(tmem + lane_base + (which ? Cfg::kColDV : Cfg::kColDK) + half * (D / 2) + c * 32, ar[which][c]);
        tmem_ld_wait();
#pragma unroll
        for (int which = 0; which < 2; ++which)
#pragma unroll
            for (int c = 0; c < D / 64; ++c) reg_fence(ar[which][c]);
        tc_fence_before();
        mbar_arrive_warp(&st->acc_free);
        if constexpr (Cfg::kTmaOut) {
            // dK (scaled) and dV as two 128 x 64 tiles, 128-byte swizzled, over
            // the item's K_j and V_j (every product of the item has completed:
            // acc_done); warp 11 stores them
            uint8_t* tile = sK + (gi % Cfg::kKvBuffers) * Cfg::kKvBytes;
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const float mul = which ? 1.f : p.scale;
                uint8_t* row = tile + which * Cfg::kTileBytes + r * 128;
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const uint32_t* a = &ar[which][0][8 * v];
                    uint4 w4;
                    w4.x = Elem16<T>::pack2(__uint_as_float(a[0]) * mul, __uint_as_float(a[1]) * mul);
                    w4.y = Elem16<T>::pack2(__uint_as_float(a[2]) * mul, __uint_as_float(a[3]) * mul);
                    w4.z = Elem16<T>::pack2(__uint_as_float(a[4]) * mul, __uint_as_float(a[5]) * mul);
                    w4.w = Elem16<T>::pack2(__uint_as_float(a[6]) * mul, __uint_as_float(a[7]) * mul);
                    const int chunk = half * 4 + v;  // 16-byte chunk of the 128-byte row
                    *reinterpret_cast<uint4*>(row + ((chunk ^ (r & 7)) << 4)) = w4;
                }
            }
            fence_proxy_async_smem();
            mbar_arrive_warp(&st->out_staged[gi % Cfg::kKvBuffers]);
        } else if (jrow < p.N) {
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                T* out = static_cast<T*>(which ? p.dv : p.dk) + ((size_t)bh * p.N) * D;
                const float mul = which ? 1.f : p.scale;
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    uint4* dst = reinterpret_cast<uint4*>(out + (size_t)jrow * D + half * (D / 2) + c * 32);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 w4;
                        w4.x = Elem16<T>::pack2(__uint_as_float(ar[which][c][8 * v + 0]) * mul,
                                                __uint_as_float(ar[which][c][8 * v + 1]) * mul);
                        w4.y = Elem16<T>::pack2(__uint_as_float(ar[which][c][8 * v + 2]) * mul,
                                                __uint_as_float(ar[which][c][8 * v + 3]) * mul);
                        w4.z = Elem16<T>::pack2(__uint_as_float(ar[which][c][8 * v + 4]) * mul,
                                                __uint_as_float(ar[which][c][8 * v + 5]) * mul);
                        w4.w = Elem16<T>::pack2(__uint_as_float(ar[which][c][8 * v + 6]) * mul,
                                                __uint_as_float(ar[which][c][8 * v + 7]) * mul);
                        dst[v] = w4;
                    }
                }
            }
        }
        gs += n_active;
        ++gi;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem, 512);
}

// The column table and dQacc = 0 (16-bit inputs). Rows are padded to whole
// 128-row tiles per head (Np = 128 nqt); for row i of head bh the table entry
// of query tile i / 128 gets -LSE_i log2(e) (-inf where LSE_i = -inf, so
// P = 0) and -delta_i, delta_i = sum_c dO_ic O_ic, and rows past N get -inf
// and 0. D/8 threads per row, 16-byte loads and stores, the row sum reduced
// across those threads.
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_pre_tc_kernel(const T* __restrict__ O, const T* __restrict__ dO,
                                                         const float* __restrict__ lse, float* __restrict__ col_table,
                                                         float* __restrict__ dq_acc, int* __restrict__ item_ctr, int N,
                                                         int nqt, size_t padded_rows) {
    constexpr int TPR = D / 8;  // threads per row (8 or 16)
    pdl_wait();               // O and LSE come from the forward kernel
    pdl_trigger();
    if (blockIdx.x == 0 && threadIdx.x == 0) *item_ctr = 0;  // the main kernel's work counter
    const size_t prow = ((size_t)blockIdx.x * 256 + threadIdx.x) / TPR;
    const int t = threadIdx.x % TPR;
    const size_t np = (size_t)nqt * kTile;
    const size_t bh = prow / np;
    const int i = (int)(prow - bh * np);
    // every lane takes part in the shuffles below; rows past N or past the
    // last head contribute zeros and load nothing
    const bool in_range = prow < padded_rows;
    const bool valid = in_range && i < N;
    const size_t row = bh * (size_t)N + (size_t)i;
    const uint4 zero4 = make_uint4(0, 0, 0, 0);
    const uint4 o4 = valid ? reinterpret_cast<const uint4*>(O + row * D)[t] : zero4;
    const uint4 g4 = valid ? reinterpret_cast<const uint4*>(dO + row * D)[t] : zero4;
    const uint32_t ow[4] = {o4.x, o4.y, o4.z, o4.w}, gw[4] = {g4.x, g4.y, g4.z, g4.w};
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 of = Elem16<T>::unpack2(ow[e]);
        const float2 gf = Elem16<T>::unpack2(gw[e]);
        s = fmaf(of.x, gf.x, s);
        s = fmaf(of.y, gf.y, s);
    }
#pragma unroll
    for (int w = TPR / 2; w > 0; w >>= 1) s += __shfl_xor_sync(0xffffffffu, s, w);
    if (!in_range) return;
    if (t == 0) {
        float* ent = col_table + (bh * nqt + (size_t)(i / kTile)) * kColTableFloats + (i % kTile);
        float nl = -INFINITY, nd = 0.f;
        if (valid) {
            const float l = lse[row];
            nl = (l == -INFINITY) ? -INFINITY : -(l * kLog2e);
            nd = -s;
        }
        ent[0] = nl;
        ent[kTile] = nd;
    }
    if (!valid) return;
    float4* acc = reinterpret_cast<float4*>(dq_acc + row * D) + 2 * t;
    acc[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    acc[1] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// dq = T(scale * dQacc), 4 elements per thread.
template <typename T>
__global__ void __launch_bounds__(256) dq_convert_kernel(const float4* __restrict__ acc, uint2* __restrict__ dq,
                                                         float scale, size_t n4) {
    pdl_wait();  // the accumulator is complete only when the main kernel is
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n4) return;
    const float4 a = acc[idx];
    uint2 w;
    w.x = Elem16<T>::pack2(a.x * scale, a.y * scale);
    w.y = Elem16<T>::pack2(a.z * scale, a.w * scale);
    dq[idx] = w;
}

template <typename T, int D>
int launch_bwd_tc_d(const Problem& pr) {
    using Cfg = BwdCfg<D>;
    constexpr CUtensorMapDataType tt = Elem16<T>::kTmaType;
    const int BH = pr.B * pr.H;
    CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;
    if (!make_tmap16(&tq, pr.q, BH, pr.N, D, kTile, tt) || !make_tmap16(&tk, pr.k, BH, pr.N, D, kTile, tt) ||
        !make_tmap16(&tv, pr.v, BH, pr.N, D, kTile, tt) || !make_tmap16(&tdo, pr.dO, BH, pr.N, D, kTile, tt) ||
        !make_tmap_f32_acc(&tdq, pr.dq_acc, BH, pr.N, D) || !make_tmap16(&tdk, pr.dk, BH, pr.N, D, kTile, tt) ||
        !make_tmap16(&tdv, pr.dv, BH, pr.N, D, kTile, tt))
        return FA_ERR_CUDA;
    const size_t rows = (size_t)BH * pr.N;
    const int nqt = (pr.N + kTile - 1) / kTile;
    const size_t padded_rows = (size_t)BH * nqt * kTile;
    // The three kernels are launched with programmatic stream serialization:
    // each may start while the previous one drains and waits (pdl_wait) only
    // where it reads what that one wrote.
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = pr.stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(256);
    cfg.gridDim = dim3((unsigned)((padded_rows * (D / 8) + 255) / 256));
    if (cudaLaunchKernelEx(&cfg, bwd_pre_tc_kernel<T, D>, static_cast<const T*>(pr.o), static_cast<const T*>(pr.dO),
                           static_cast<const float*>(pr.lse), pr.col_table, pr.dq_acc, pr.item_ctr, pr.N, nqt,
                           padded_rows) != cudaSuccess)
        return FA_ERR_CUDA;
    note_launches(1);

    BwdParams p{};
    p.col_table = pr.col_table;
    p.dq_acc = pr.dq_acc;
    p.dk = pr.dk;
    p.dv = pr.dv;
    p.block_mask = pr.block_mask;
    p.kv_len = pr.kv_len;
    p.status = pr.status;
    p.H = pr.H;
    p.N = pr.N;
    p.nb = pr.nb;
    p.BH = BH;
    p.nkt = (pr.N + kTile - 1) / kTile;
    p.item_ctr = pr.item_ctr;
    p.scale = pr.scale;
    p.scale_log2 = pr.scale * kLog2e;
    p.keep_scale = 1.0f / (1.0f - pr.dropout_p);
    p.drop_thr = pr.drop_threshold;
    p.dropout = pr.dropout_p > 0.f;
    p.causal = pr.causal;
    p.seed = pr.seed;
    // The grid is persistent (one CTA per SM claiming items in order from the
    // workspace counter), so that one item's last products and dK/dV stores
    // overlap the next one's loads and first products; with a block mask the
    // persistent CTA needs two item lists in shared memory, which fit at
    // D = 64 only, and D = 128 keeps one CTA per item.
    const bool persist = !pr.block_mask || D == 64;
    using KernelFn = decltype(&bwd_tc_kernel<T, D, false, false>);
    KernelFn kernel = nullptr;
    KernelFn all[4] = {bwd_tc_kernel<T, D, false, false>, bwd_tc_kernel<T, D, false, true>,
                       bwd_tc_kernel<T, D, true, false>, nullptr};
    if constexpr (D == 64) all[3] = bwd_tc_kernel<T, D, true, true>;
    kernel = all[(pr.block_mask ? 2 : 0) + (persist ? 1 : 0)];
    if (!kernel) return FA_ERR_UNSUPPORTED;
    static bool attr_set = false;
    if (!attr_set) {
        // setmaxnreg.inc takes registers from what the CTA was launched with
        // and waits (without bound) until they are free: refuse to launch
        // unless the budgets fit in that allocation
        for (int x = 0; x < 4; ++x) {
            if (!all[x]) continue;
            cudaFuncAttributes a{};
            if (cudaFuncSetAttribute(all[x], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     Cfg::smem(x >= 2, x == 3)) != cudaSuccess ||
                cudaFuncGetAttributes(&a, all[x]) != cudaSuccess || a.numRegs * Cfg::kThreads < Cfg::kRegBudget) {
                if (std::getenv("FA_DEBUG"))
                    std::fprintf(stderr, "fa: bwd register budget %d exceeds the launch allocation (%d regs)\n",
                                 Cfg::kRegBudget, a.numRegs);
                return FA_ERR_CUDA;
            }
        }
        attr_set = true;
    }
    if (!persist) {
        cfg.gridDim = dim3(BH, p.nkt);
    } else {
        int dev = 0, nsm = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nsm < 1)
            return FA_ERR_CUDA;
        const long long n_items = (long long)BH * p.nkt;
        cfg.gridDim = dim3((unsigned)std::min<long long>(n_items, nsm), 1);
    }
    cfg.blockDim = dim3(Cfg::kThreads);
    cfg.dynamicSmemBytes = Cfg::smem(pr.block_mask != nullptr, pr.block_mask != nullptr && persist);
    record_main_start(pr.stream);
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, tdo, tdq, tdk, tdv, p);
    record_main_stop(pr.stream);
    note_launches(1);
    if (e != cudaSuccess) {
        if (std::getenv("FA_DEBUG")) std::fprintf(stderr, "fa: bwd_tc launch: %s\n", cudaGetErrorString(e));
        return FA_ERR_CUDA;
    }
    const size_t n4 = rows * D / 4;
    cfg.gridDim = dim3((unsigned)((n4 + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    e = cudaLaunchKernelEx(&cfg, dq_convert_kernel<T>, reinterpret_cast<const float4*>(pr.dq_acc),
                           static_cast<uint2*>(pr.dq), pr.scale, n4);
    note_launches(1);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

int launch_bwd_tc(const Problem& p) {
    if (!(p.scale > 0.f)) {
        record_main_start(p.stream);
        const cudaError_t e = launch_bwd_simt(p);
        record_main_stop(p.stream);
        return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
    }
    if (p.d == 256) return launch_bwd256_tc(p);
    if (p.dtype == FA_FP16) return p.d == 64 ? launch_bwd_tc_d<__half, 64>(p) : launch_bwd_tc_d<__half, 128>(p);
    if (p.dtype == FA_BF16)
        return p.d == 64 ? launch_bwd_tc_d<__nv_bfloat16, 64>(p) : launch_bwd_tc_d<__nv_bfloat16, 128>(p);
    return FA_ERR_UNSUPPORTED;
}

}  // namespace fa
