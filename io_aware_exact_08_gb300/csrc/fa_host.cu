// fa_fwd_bwd_host: one attention training step (forward and backward) on
// tensors that live in host memory.
//
// The method starts from Q, K, V already in HBM and ends with O written to
// HBM (blog post "Flash Attention", section "Flash Attention"). A caller
// whose tensors start in host memory pays two more transfers per step: q, k,
// v, dO over the host link into HBM, and o, lse, dq, dk, dv back. Run one
// after another, those copies take longer than the kernels on GB300 (a
// quarter of a gigabyte each way for a B=2 H=16 N=8K d=128 step). This entry
// point overlaps them with the kernels:
//  - Heads are independent in both passes, so the step is cut into chunks of
//    whole heads, each a smaller fa_fwd + fa_bwd problem.
//  - The chunks move through a ring of three device slots in the caller's
//    workspace. Host-to-device copies run on one internal stream,
//    device-to-host copies on another, and the kernels alternately on the
//    caller's stream and a second internal one: chunk c+1 is copied in and
//    chunk c-1 copied out while chunk c computes, and a chunk's forward
//    takes the SMs the previous chunk's backward frees as it ends.
//  - Events order each slot's reuse: a chunk's inputs are overwritten only
//    after the backward that read them has finished, and its outputs only
//    after they have been copied out.
//  - The call ends by making the caller's stream wait for the internal
//    streams, so work queued on it afterwards sees every result in host
//    memory.
//
// What constrains the chunks:
//  - The dropout keep bit of (b, h, i, j) is drawn from a counter that holds
//    the absolute batch and head. A chunk is launched as its own problem and
//    would number its heads from zero, so with dropout the step runs as one
//    chunk (the copies then do not overlap the kernels).
//  - Key padding (kv_len) is per batch. Chunks then either hold whole
//    batches, or lie inside one batch, and are given kv_len from their first
//    batch on.
//  - Without those, any run of consecutive heads is a valid chunk.
//
// The three internal streams and their events are created on a device's first
// call and kept until the process exits. Calls on one device are serialised
// on the host while they enqueue work.
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <initializer_list>
#include <mutex>
#include <utility>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/fa.h"

namespace {

constexpr int kSlots = 3;          // device slots in the ring
// Chunks per step when the caller leaves the size open: at most four, each
// of at least 8 heads' worth of 128-row query tiles, and no fewer than 256
// or more than 512 tiles, where the step has that many.
//  - The host link of a GB300 moves ~200 GB/s each way (~340 GB/s both ways
//    at once), so at N = 8K the copies of a step take about as long as its
//    kernels. Four chunks keep the first chunk's copy-in and the last
//    chunk's copy-out short while each chunk still fills the GPU.
//  - Long sequences need more tiles per chunk: a key tile of the causal
//    backward meets every query tile of its head, so a chunk of few long
//    heads lasts as long as that one item.
// Measured (one step on host buffers, with the kernels on one stream; the
// second compute stream moves these choices by under 1 %):
//  - B=2 H=16 N=8K d=128 causal: 3 chunks 2.46 ms, 4 chunks 2.34, 6 chunks
//    2.72, 8 chunks 3.15;
//  - B=8 H=12 N=1K d=64 causal: 3 chunks 0.459 ms, 6 chunks 0.482,
//    12 chunks 0.574, one chunk 0.538;
//  - B=1 H=4 N=16K d=128 causal: one chunk 1.375 ms, 2 chunks 1.633;
//  - B=1 H=16 N=16K d=128 causal: 4 chunks 3.905 ms, 2 chunks 4.236;
//  - B=2 H=8 N=4K d=256 causal: 2 chunks 1.396 ms, one chunk 1.869.
constexpr int kMaxChunks = 4;
constexpr long long kMinChunkTiles = 256, kMaxChunkTiles = 512, kMinChunkHeads = 8;
constexpr int kMaxDevices = 64;

struct Chunk {
    long long head0;  // first head, numbered b * H + h
    int B, H;         // shape of the chunk's fa_fwd / fa_bwd problem
    int b0;           // first batch of the chunk (its kv_len offset)
};

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

size_t elem_bytes(fa_dtype t) { return t == FA_FP32 ? 4 : 2; }

bool valid_shape(int B, int H, int N, int d, fa_dtype dtype) {
    if (B < 1 || H < 1 || N < 0) return false;
    if ((long long)B * H > 65535) return false;
    if (d != 64 && d != 128 && d != 256) return false;
    return dtype == FA_BF16 || dtype == FA_FP16 || dtype == FA_FP32;
}

// The chunks of a step, in head order. Every head appears in exactly one
// chunk; the chunks' problems are independent.
std::vector<Chunk> plan_chunks(int B, int H, int N, bool has_kv_len, bool dropout, int chunk_heads) {
    std::vector<Chunk> out;
    const long long F = (long long)B * H;
    if (dropout) {
        out.push_back({0, B, H, 0});
        return out;
    }
    long long G;
    if (chunk_heads > 0) {
        G = std::min<long long>(chunk_heads, F);
    } else {
        const long long nt = std::max(1, (N + 127) / 128);
        const long long tiles = std::min(kMaxChunkTiles, std::max(kMinChunkTiles, kMinChunkHeads * nt));
        const long long gmin = (tiles + nt - 1) / nt;
        const long long n = std::max(1LL, std::min<long long>(kMaxChunks, F / gmin));
        G = (F + n - 1) / n;
    }
    // n pieces of `total` units, as even as possible: piece i has
    // total / n units, plus one for the first total % n pieces
    auto piece = [](long long total, long long n, long long i) { return total / n + (i < total % n ? 1 : 0); };
    if (has_kv_len) {
        if (G >= H) {  // whole batches, at most G / H of them per chunk
            const long long n = (B + G / H - 1) / (G / H);
            for (long long i = 0, b = 0; i < n; b += piece(B, n, i), ++i)
                out.push_back({b * H, (int)piece(B, n, i), H, (int)b});
        } else {  // runs of heads inside each batch
            const long long n = (H + G - 1) / G;
            for (int b = 0; b < B; ++b)
                for (long long i = 0, h = 0; i < n; h += piece(H, n, i), ++i)
                    out.push_back({(long long)b * H + h, 1, (int)piece(H, n, i), b});
        }
    } else {
        const long long n = (F + G - 1) / G;
        for (long long i = 0, f = 0; i < n; f += piece(F, n, i), ++i) out.push_back({f, 1, (int)piece(F, n, i), 0});
    }
    return out;
}

int slot_heads(const std::vector<Chunk>& chunks) {
    int s = 0;
    for (const Chunk& c : chunks) s = std::max(s, c.B * c.H);
    return s;
}

// Workspace layout: kv_len (if given), the block mask (if given), then the
// slots. A slot holds q, k, v, dO, o, dq, dk, dv of `heads` heads, their lse
// and the backward workspace of that many heads, each part 256-byte aligned.
struct Layout {
    size_t kv_len_off, mask_off, slots_off;
    size_t tensor_bytes, lse_bytes, bwd_ws_bytes, slot_bytes;
    int n_slots;
    size_t total;
};

Layout make_layout(int B, int N, int d, fa_dtype dtype, bool has_mask, bool has_kv_len, int heads, int n_chunks) {
    Layout L{};
    const size_t nb = (size_t)(N + 127) / 128;
    L.kv_len_off = 0;
    L.mask_off = has_kv_len ? round256((size_t)B * sizeof(int32_t)) : 0;
    L.slots_off = L.mask_off + (has_mask ? round256(nb * nb) : 0);
    L.tensor_bytes = round256((size_t)heads * N * d * elem_bytes(dtype));
    L.lse_bytes = round256((size_t)heads * N * sizeof(float));
    L.bwd_ws_bytes = round256(fa_bwd_workspace_size(1, heads, N, d));
    L.slot_bytes = 8 * L.tensor_bytes + L.lse_bytes + L.bwd_ws_bytes;
    L.n_slots = std::min(kSlots, n_chunks);
    L.total = L.slots_off + (size_t)L.n_slots * L.slot_bytes;
    return L;
}

// Per-device copy streams and the events that order the ring.
struct DeviceCtx {
    bool ready = false;
    cudaStream_t s_in = nullptr, s_out = nullptr, s_comp = nullptr;
    cudaEvent_t ev_start = nullptr, ev_in_done = nullptr, ev_out_done = nullptr, ev_comp_done = nullptr;
    cudaEvent_t ev_qkv[kSlots] = {}, ev_do[kSlots] = {}, ev_fwd[kSlots] = {}, ev_bwd[kSlots] = {},
                ev_out[kSlots] = {};
};

std::mutex g_lock[kMaxDevices];
DeviceCtx g_ctx[kMaxDevices];

bool make_event(cudaEvent_t* e) { return cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess; }

void destroy_ctx(DeviceCtx& c) {
    for (cudaStream_t* st : {&c.s_in, &c.s_out, &c.s_comp})
        if (*st) cudaStreamDestroy(*st);
    for (cudaEvent_t* e : {&c.ev_start, &c.ev_in_done, &c.ev_out_done, &c.ev_comp_done})
        if (*e) cudaEventDestroy(*e);
    for (int s = 0; s < kSlots; ++s)
        for (cudaEvent_t* e : {&c.ev_qkv[s], &c.ev_do[s], &c.ev_fwd[s], &c.ev_bwd[s], &c.ev_out[s]})
            if (*e) cudaEventDestroy(*e);
    c = DeviceCtx{};
}

// The context of the current device, created on first use (under its lock);
// a failed creation releases what it made, so a later call starts afresh.
DeviceCtx* device_ctx(int dev) {
    DeviceCtx& c = g_ctx[dev];
    if (c.ready) return &c;
    bool ok = cudaStreamCreateWithFlags(&c.s_in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&c.s_out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&c.s_comp, cudaStreamNonBlocking) == cudaSuccess &&
              make_event(&c.ev_start) && make_event(&c.ev_in_done) && make_event(&c.ev_out_done) &&
              make_event(&c.ev_comp_done);
    for (int s = 0; ok && s < kSlots; ++s)
        ok = make_event(&c.ev_qkv[s]) && make_event(&c.ev_do[s]) && make_event(&c.ev_fwd[s]) &&
             make_event(&c.ev_bwd[s]) && make_event(&c.ev_out[s]);
    if (!ok) {
        destroy_ctx(c);
        return nullptr;
    }
    c.ready = true;
    return &c;
}

int from_cuda(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return FA_OK;
    if (std::getenv("FA_DEBUG")) std::fprintf(stderr, "fa_fwd_bwd_host: %s: %s\n", what, cudaGetErrorString(e));
    return FA_ERR_CUDA;
}

char* at(void* base, size_t off) { return static_cast<char*>(base) + off; }
const char* at(const void* base, size_t off) { return static_cast<const char*>(base) + off; }

}  // namespace

extern "C" size_t fa_fwd_bwd_host_workspace_size(int B, int H, int N, int d, fa_dtype dtype,
                                                 const uint8_t* block_mask, float dropout_p, const int32_t* kv_len,
                                                 int chunk_heads) {
    if (!valid_shape(B, H, N, d, dtype) || chunk_heads < 0) return 0;
    if (N == 0) return 0;
    const std::vector<Chunk> chunks = plan_chunks(B, H, N, kv_len != nullptr, dropout_p > 0.f, chunk_heads);
    return make_layout(B, N, d, dtype, block_mask != nullptr, kv_len != nullptr, slot_heads(chunks),
                       (int)chunks.size())
        .total;
}

extern "C" int fa_fwd_bwd_host_chunks(int B, int H, int N, const int32_t* kv_len, float dropout_p,
                                      int chunk_heads, int* desc, int max_chunks) {
    if (B < 1 || H < 1 || N < 0 || (long long)B * H > 65535 || chunk_heads < 0 || max_chunks < 0)
        return FA_ERR_INVALID_ARG;
    const std::vector<Chunk> chunks = plan_chunks(B, H, N, kv_len != nullptr, dropout_p > 0.f, chunk_heads);
    if (desc) {
        for (int i = 0; i < (int)chunks.size() && i < max_chunks; ++i) {
            desc[4 * i + 0] = (int)chunks[i].head0;
            desc[4 * i + 1] = chunks[i].B;
            desc[4 * i + 2] = chunks[i].H;
            desc[4 * i + 3] = chunks[i].b0;
        }
    }
    return (int)chunks.size();
}

extern "C" int fa_fwd_bwd_host(const void* q, const void* k, const void* v, const void* dO, void* o, float* lse,
                               void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                               const uint8_t* block_mask, float dropout_p, uint64_t seed, fa_dtype dtype,
                               const int32_t* kv_len, int chunk_heads, void* workspace, size_t workspace_bytes,
                               void* stream) {
    if (B < 1 || H < 1 || N < 0 || chunk_heads < 0) return FA_ERR_INVALID_ARG;
    if (!(dropout_p >= 0.f && dropout_p < 1.f)) return FA_ERR_INVALID_ARG;
    if (!valid_shape(B, H, N, d, dtype)) return FA_ERR_UNSUPPORTED;
    if (N == 0) return FA_OK;
    if (!q || !k || !v || !dO || !o || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
    const std::vector<Chunk> chunks = plan_chunks(B, H, N, kv_len != nullptr, dropout_p > 0.f, chunk_heads);
    const Layout L = make_layout(B, N, d, dtype, block_mask != nullptr, kv_len != nullptr, slot_heads(chunks),
                                 (int)chunks.size());
    if (!workspace || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
        return FA_ERR_WORKSPACE;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> guard(g_lock[dev]);
    DeviceCtx* c = device_ctx(dev);
    if (!c) return FA_ERR_CUDA;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);

    const size_t head_elems = (size_t)N * d;
    const size_t eb = elem_bytes(dtype);
    const size_t nb = (size_t)(N + 127) / 128;
    int32_t* kv_dev = kv_len ? reinterpret_cast<int32_t*>(at(workspace, L.kv_len_off)) : nullptr;
    uint8_t* mask_dev = block_mask ? reinterpret_cast<uint8_t*>(at(workspace, L.mask_off)) : nullptr;

    int rc = FA_OK;
    // the copies start after the work already queued on the caller's stream
    // (an earlier step may still be using the workspace)
    rc = from_cuda(cudaEventRecord(c->ev_start, cs), "record start");
    if (rc == FA_OK) rc = from_cuda(cudaStreamWaitEvent(c->s_in, c->ev_start, 0), "wait start");
    if (rc == FA_OK) rc = from_cuda(cudaStreamWaitEvent(c->s_comp, c->ev_start, 0), "wait start");
    if (rc == FA_OK && kv_dev)
        rc = from_cuda(cudaMemcpyAsync(kv_dev, kv_len, (size_t)B * sizeof(int32_t), cudaMemcpyHostToDevice, c->s_in),
                       "copy kv_len");
    if (rc == FA_OK && mask_dev)
        rc = from_cuda(cudaMemcpyAsync(mask_dev, block_mask, nb * nb, cudaMemcpyHostToDevice, c->s_in),
                       "copy block mask");

    for (size_t i = 0; rc == FA_OK && i < chunks.size(); ++i) {
        const Chunk& ch = chunks[i];
        const int s = (int)(i % L.n_slots);
        const bool reuse = i >= (size_t)L.n_slots;
        char* slot = at(workspace, L.slots_off + (size_t)s * L.slot_bytes);
        char* t[8];
        for (int j = 0; j < 8; ++j) t[j] = slot + (size_t)j * L.tensor_bytes;  // q k v dO o dq dk dv
        float* lse_d = reinterpret_cast<float*>(slot + 8 * L.tensor_bytes);
        void* bwd_ws = slot + 8 * L.tensor_bytes + L.lse_bytes;
        const size_t heads = (size_t)ch.B * ch.H;
        const size_t off = (size_t)ch.head0 * head_elems * eb;
        const size_t bytes = heads * head_elems * eb;
        const size_t lse_off = (size_t)ch.head0 * N * sizeof(float);
        const size_t lse_bytes = heads * N * sizeof(float);
        const void* src_in[4] = {q, k, v, dO};
        void* dst_out[4] = {o, dq, dk, dv};

        // in: the slot's inputs are free once the backward of the chunk that
        // used the slot before has finished
        if (reuse) rc = from_cuda(cudaStreamWaitEvent(c->s_in, c->ev_bwd[s], 0), "wait slot inputs");
        for (int j = 0; rc == FA_OK && j < 3; ++j)
            rc = from_cuda(cudaMemcpyAsync(t[j], at(src_in[j], off), bytes, cudaMemcpyHostToDevice, c->s_in),
                           "copy in");
        if (rc == FA_OK) rc = from_cuda(cudaEventRecord(c->ev_qkv[s], c->s_in), "record qkv");
        if (rc == FA_OK)
            rc = from_cuda(cudaMemcpyAsync(t[3], at(dO, off), bytes, cudaMemcpyHostToDevice, c->s_in), "copy dO");
        if (rc == FA_OK) rc = from_cuda(cudaEventRecord(c->ev_do[s], c->s_in), "record dO");

        // compute, alternately on the caller's stream and the second compute
        // stream, so that a chunk's forward can start on the SMs the
        // previous chunk's backward leaves idle as it finishes. The slot's
        // outputs are free once the chunk that used the slot before has been
        // copied out.
        cudaStream_t ks = (i % 2 == 0) ? cs : c->s_comp;
        if (rc == FA_OK) rc = from_cuda(cudaStreamWaitEvent(ks, c->ev_qkv[s], 0), "wait qkv");
        if (rc == FA_OK && reuse) rc = from_cuda(cudaStreamWaitEvent(ks, c->ev_out[s], 0), "wait slot outputs");
        const int32_t* kv_chunk = kv_dev ? kv_dev + ch.b0 : nullptr;
        if (rc == FA_OK)
            rc = fa_fwd(t[0], t[1], t[2], t[4], lse_d, ch.B, ch.H, N, d, scale, causal, mask_dev, dropout_p, seed,
                        dtype, kv_chunk, ks);
        if (rc == FA_OK) rc = from_cuda(cudaEventRecord(c->ev_fwd[s], ks), "record fwd");
        if (rc == FA_OK) rc = from_cuda(cudaStreamWaitEvent(ks, c->ev_do[s], 0), "wait dO");
        if (rc == FA_OK)
            rc = fa_bwd(t[0], t[1], t[2], t[4], lse_d, t[3], t[5], t[6], t[7], ch.B, ch.H, N, d, scale, causal,
                        mask_dev, dropout_p, seed, dtype, kv_chunk, bwd_ws, L.bwd_ws_bytes, ks);
        if (rc == FA_OK) rc = from_cuda(cudaEventRecord(c->ev_bwd[s], ks), "record bwd");

        // out: o and lse as soon as the forward is done, the gradients after
        // the backward
        if (rc == FA_OK) rc = from_cuda(cudaStreamWaitEvent(c->s_out, c->ev_fwd[s], 0), "wait fwd");
        if (rc == FA_OK)
            rc = from_cuda(cudaMemcpyAsync(at(o, off), t[4], bytes, cudaMemcpyDeviceToHost, c->s_out), "copy o");
        if (rc == FA_OK)
            rc = from_cuda(cudaMemcpyAsync(reinterpret_cast<char*>(lse) + lse_off, lse_d, lse_bytes,
                                           cudaMemcpyDeviceToHost, c->s_out),
                           "copy lse");
        if (rc == FA_OK) rc = from_cuda(cudaStreamWaitEvent(c->s_out, c->ev_bwd[s], 0), "wait bwd");
        for (int j = 1; rc == FA_OK && j < 4; ++j)
            rc = from_cuda(cudaMemcpyAsync(at(dst_out[j], off), t[4 + j], bytes, cudaMemcpyDeviceToHost, c->s_out),
                           "copy out");
        if (rc == FA_OK) rc = from_cuda(cudaEventRecord(c->ev_out[s], c->s_out), "record out");
    }

    // join: the caller's stream waits for the other three streams, also
    // after an error, so that nothing of this call is left unordered behind
    // it
    int rc_join = FA_OK;
    const std::pair<cudaStream_t, cudaEvent_t> joins[3] = {
        {c->s_in, c->ev_in_done}, {c->s_comp, c->ev_comp_done}, {c->s_out, c->ev_out_done}};
    for (const auto& j : joins) {
        int r = from_cuda(cudaEventRecord(j.second, j.first), "record done");
        if (r == FA_OK) r = from_cuda(cudaStreamWaitEvent(cs, j.second, 0), "join");
        if (rc_join == FA_OK) rc_join = r;
    }
    return rc != FA_OK ? rc : rc_join;
}
