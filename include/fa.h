/*
 * fa.h - C ABI of the exact IO-aware attention library (GB300, sm_103a).
 *
 * The library computes exact attention O = softmax(scale * Q K^T + mask) V
 * block by block with the running row-max / row-sum rescaling, so the N x N
 * score matrix never reaches HBM ("FlashAttention: Fast and Memory-Efficient
 * Exact Attention with IO-Awareness", sections "Ide Utama" and "Metode",
 * steps 1-4), and the backward pass that keeps only O and the per-row
 * log-sum-exp and recomputes S and P tile by tile (same page, "Ide Utama",
 * third point; "FlashAttention" blog post, section "Recomputation").
 *
 * Conventions shared by every entry point:
 *  - Tensors are contiguous [B, H, N, d] row-major (d fastest), in device
 *    memory (host memory for fa_fwd_bwd_host), 16-byte aligned. q, k, v, o,
 *    dO, dq, dk, dv all have that shape and the element type `dtype`. lse is fp32 [B, H, N] in natural log:
 *    lse = m + ln(l), which carries the same information as the pair (l, m)
 *    the pages keep for the backward pass.
 *  - d must be 64, 128 or 256. B, H >= 1, N >= 0 (N == 0 is a no-op).
 *    d = 256 is the largest head dimension of the FlashAttention-2 section
 *    of "Penjelasan Flash Attention: Panduan Komprehensif" ("Dukungan untuk
 *    dimensi head yang lebih besar"); its backward runs in three passes
 *    (dV, dK, dQ) on the tensor cores for 16-bit inputs.
 *  - Masks combine by AND: causal (key j > query i is masked, top-left
 *    aligned), key padding (j >= kv_len[b] masked; kv_len is int32[B] in
 *    device memory, or NULL), block mask (block_mask[(i/128)*nb + j/128] == 0
 *    masks the block; nb = ceil(N/128); uint8 in device memory, or NULL).
 *    The block-sparse form follows "FlashAttention: Fast and Memory-Efficient
 *    Exact Attention with IO-Awareness", section "Ekstensi: Block-Sparse
 *    FlashAttention"; the block edge is fixed at 128 for queries and keys.
 *  - A query row with every key masked gives O = 0, lse = -inf and no
 *    gradient.
 *  - Dropout (0 <= dropout_p < 1) is applied to the normalised P for the
 *    P V product only (inverted: kept entries scaled by 1/(1-p)); lse does
 *    not include it. The keep bit of (b, h, i, j) is word (j mod 4) of
 *    Philox4x32-10 (Salmon et al., SC'11) with key (lo32(seed), hi32(seed))
 *    and counter (j/4, i, h, b), kept iff that word >= floor(p * 2^32)
 *    (clamped to 2^32 - 1). It is independent of tiling, so the forward,
 *    the backward and fa_dropout_mask agree bit for bit.
 *  - stream is a cudaStream_t (NULL = the legacy default stream). Calls are
 *    asynchronous on it and synchronise nothing except
 *    fa_check_device_status. The library allocates no device memory per
 *    call; the only device memory it holds is static: a status word of two
 *    ints and the fixed FA_BWD_NOALLOC_SCRATCH_BYTES (32 MiB) array of
 *    fa_bwd_noalloc, present on every GPU that loads the library
 *    (fa_fwd_bwd_host also keeps two streams and a few events per device).
 *  - The device addresses of those two static objects are looked up once
 *    per device and cached for the life of the process, so resetting a
 *    device (cudaDeviceReset, or a reset of its primary context) while the
 *    library is in use is not supported.
 *  - Every call returns FA_OK (0) or a negative fa_status. Argument errors
 *    are detected on the host before any launch; nothing is thrown across
 *    the ABI. Device-side bounded waits that run out set a status word that
 *    fa_check_device_status reports.
 */
#ifndef FA_GB300_FA_H
#define FA_GB300_FA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of q, k, v, o, dO, dq, dk, dv. The 16-bit types run on the
 * tcgen05 tensor-core kernels (fp32 accumulation); fp32 runs on fp32
 * CUDA-core kernels. */
typedef enum { FA_BF16 = 0, FA_FP32 = 1, FA_FP16 = 2 } fa_dtype;

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = -1,   /* null pointer, negative size, p outside [0,1), misalignment */
    FA_ERR_UNSUPPORTED = -2,   /* d not in {64,128,256}, unknown dtype, or a 16-bit problem the
                                  tensor-core kernels do not take (see fa_fwd) */
    FA_ERR_CUDA = -3,          /* a CUDA runtime call failed (launch, attribute, symbol) */
    FA_ERR_WORKSPACE = -4,     /* workspace missing or smaller than fa_bwd_workspace_size */
    FA_ERR_DEVICE_TIMEOUT = -5 /* a device-side bounded wait ran out (see fa_check_device_status) */
} fa_status;

/*
 * Forward: o = softmax(scale * q k^T + mask) v with optional dropout, and
 * lse[b,h,i] = log-sum-exp of row i's (masked, scaled) scores.
 * Inputs q, k, v; outputs o (dtype) and lse (fp32). All device pointers,
 * owned by the caller. bf16 and fp16 run on the tcgen05 tensor-core kernel;
 * fp32 on an fp32 CUDA-core kernel.
 * 16-bit problems the tensor-core kernels do not take are refused with
 * FA_ERR_UNSUPPORTED before any launch, not run on the (far slower)
 * CUDA-core kernels: scale <= 0, or a block mask with more than 1024 key
 * tiles per row (N > 131072). The backward's limit on block masks is 1024
 * tiles at d = 64 and 256 tiles (N <= 32768) at d = 128 and 256. Callers who
 * want the CUDA-core kernels for such a problem select them explicitly with
 * fa_set_kernel_path(1).
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int N, int d, float scale, int causal,
           const uint8_t* block_mask, float dropout_p, uint64_t seed,
           fa_dtype dtype, const int32_t* kv_len, void* stream);

/*
 * Backward: given the forward's inputs, its outputs o and lse, and the
 * output gradient dO, writes dq, dk, dv (dtype, [B,H,N,d]). S and P are
 * recomputed tile by tile from lse; the same masks, scale and dropout
 * (seed, p) as the forward must be passed. workspace is caller-owned device
 * memory of at least fa_bwd_workspace_size(B,H,N,d) bytes, 256-byte aligned
 * (rowsum(dO o O), the fp32 dQ accumulator and a work counter: about
 * B*H*N*(d+1)*4 + 256 bytes); its contents on entry do not matter and on
 * exit are unspecified.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dO, void* dq, void* dk, void* dv,
           int B, int H, int N, int d, float scale, int causal,
           const uint8_t* block_mask, float dropout_p, uint64_t seed,
           fa_dtype dtype, const int32_t* kv_len,
           void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward for callers that cannot allocate device memory (a framework whose
 * allocator already owns the device, a latency-bound path where cudaMalloc
 * is not allowed, a plugin given only its tensors). The paper has no
 * counterpart: this is a packaging of fa_bwd, with the same arguments and
 * results minus the workspace. The workspace comes from a fixed array of
 * FA_BWD_NOALLOC_SCRATCH_BYTES in device memory that the library holds on
 * every GPU it is loaded on until exit; nothing is allocated per call.
 *  - Returns FA_ERR_WORKSPACE, without launching, when
 *    fa_bwd_workspace_size(B,H,N,d) exceeds that size (about
 *    B*H*N*(d+2)*4 bytes).
 *  - Calls share the array: calls whose kernels may overlap on the GPU
 *    (unordered streams) race and give wrong results. Each call clears the
 *    parts that must start at zero.
 *  - The first call on a device looks up the array's device address with
 *    that device current; make that first call before any stream capture.
 */
#define FA_BWD_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dO, void* dq, void* dk, void* dv,
                   int B, int H, int N, int d, float scale, int causal,
                   const uint8_t* block_mask, float dropout_p, uint64_t seed,
                   fa_dtype dtype, const int32_t* kv_len, void* stream);

/*
 * One training step on HOST tensors: o, lse = forward(q, k, v) and
 * dq, dk, dv = backward(q, k, v, o, lse, dO), the same computation as fa_fwd
 * followed by fa_bwd, for callers whose tensors are in host memory. The
 * method itself starts from Q, K, V in HBM and ends with O in HBM (blog post
 * "Flash Attention", section "Flash Attention"); this call adds the
 * transfers and hides them behind the kernels. The heads are cut into
 * chunks that pass through a ring of three device slots in the workspace:
 * the copies of chunk c+1 in and chunk c-1 out run on two internal streams
 * while chunk c computes on `stream`.
 *   q, k, v, dO    inputs, host memory, [B, H, N, d] of `dtype`.
 *   o, dq, dk, dv  outputs, host memory, [B, H, N, d] of `dtype`.
 *   lse            output, host memory, fp32 [B, H, N].
 *   block_mask, kv_len
 *                  as in fa_fwd but in HOST memory (copied into the
 *                  workspace), or NULL.
 *   chunk_heads    heads per chunk; 0 picks it (at most 4 chunks, each of
 *                  at least 8 heads' worth of 128-row query tiles, clamped
 *                  to 256..512 tiles, where the problem has that many). With key padding a chunk holds whole batches
 *                  or lies within one. With dropout the step is one chunk:
 *                  the keep bits are drawn from the absolute (b, h).
 *   workspace      caller-owned device memory, 256-byte aligned, of at least
 *                  fa_fwd_bwd_host_workspace_size bytes (about three chunks'
 *                  tensors plus their backward workspace).
 *   other arguments as in fa_fwd / fa_bwd.
 * Runs on the current device; `stream` must belong to it.
 * Asynchronous like a cudaMemcpyAsync: on return the work is queued and
 * `stream` waits for all of it; the host buffers must stay valid and
 * unchanged until the stream reaches that point. The copies overlap the
 * kernels only for page-locked host memory (cudaHostAlloc,
 * cudaHostRegister); with pageable memory the results are the same but
 * the call returns only after its copies are done. The library creates two
 * streams and a few events per device on the first call and keeps them
 * until exit; calls on one device are serialised on the host while they
 * queue their work.
 * Returns the errors of fa_fwd and fa_bwd (FA_ERR_INVALID_ARG for a null
 * host pointer or chunk_heads < 0; FA_ERR_WORKSPACE for a missing, small or
 * misaligned workspace). An error from the kernels' entry points stops the
 * call after the chunks already queued; `stream` still waits for them.
 */
int fa_fwd_bwd_host(const void* q, const void* k, const void* v, const void* dO,
                    void* o, float* lse, void* dq, void* dk, void* dv,
                    int B, int H, int N, int d, float scale, int causal,
                    const uint8_t* block_mask, float dropout_p, uint64_t seed,
                    fa_dtype dtype, const int32_t* kv_len, int chunk_heads,
                    void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace fa_fwd_bwd_host needs for these arguments (only
 * whether block_mask and kv_len are NULL, and whether dropout_p > 0,
 * matter); 0 for invalid sizes or N == 0. */
size_t fa_fwd_bwd_host_workspace_size(int B, int H, int N, int d, fa_dtype dtype,
                                      const uint8_t* block_mask, float dropout_p,
                                      const int32_t* kv_len, int chunk_heads);

/* Diagnostic: the chunks fa_fwd_bwd_host would use, in order. Writes up to
 * max_chunks records of four ints (first head numbered b*H + h, the chunk's
 * B, its H, its first batch) to desc (may be NULL) and returns the number
 * of chunks, or FA_ERR_INVALID_ARG. */
int fa_fwd_bwd_host_chunks(int B, int H, int N, const int32_t* kv_len, float dropout_p,
                           int chunk_heads, int* desc, int max_chunks);

/*
 * Split-KV forward: the same result as fa_fwd (O and LSE up to rounding),
 * computed with the key tiles of every pair of 128-row query tiles cut into
 * n_splits ranges, one CTA each, for problems whose B*H*ceil(N/256) work items
 * would not fill the GPU (sequence parallelism across the key dimension,
 * "Flash Attention" guide, section "Flash Attention 2 / Paralelisme sepanjang
 * panjang sekuens"). Each CTA writes its range's O (normalised over the range)
 * and LSE to the workspace; a second kernel merges them with the
 * incremental-softmax combination of the paper summary (section "Pelacakan
 * Softmax Inkremental"): M = max_s LSE_s, w_s = e^{LSE_s - M},
 * O = sum_s w_s O_s / sum_s w_s, LSE = M + log sum_s w_s.
 *   n_splits   1 .. 64 (1 runs fa_fwd); arguments otherwise as fa_fwd.
 *   workspace  caller-owned device memory, >= fa_fwd_splitkv_workspace_size
 *              bytes, 256-byte aligned; contents undefined on return.
 * Returns as fa_fwd, plus FA_ERR_INVALID_ARG for n_splits outside 1..64 and
 * FA_ERR_WORKSPACE for a missing, small or misaligned workspace. With the
 * CUDA-core kernels (fp32, or fa_set_kernel_path(1)) it runs fa_fwd.
 */
int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int H, int N, int d, float scale, int causal,
                   const uint8_t* block_mask, float dropout_p, uint64_t seed,
                   fa_dtype dtype, const int32_t* kv_len, int n_splits,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * FP8 forward ("Flash Attention" guide, section "Flash Attention 3 / Presisi
 * FP8 native"): o = softmax(scale * Q K^T + mask) V on 8-bit inputs, both
 * products on the tensor cores in E4M3 with fp32 accumulation.
 *   q, k       E4M3 codes (OCP 8-bit floating point, 1-4-3, bias 7), uint8
 *              [B, H, N, 128], device memory, 16-byte aligned.
 *   vt         V transposed: E4M3 codes [B, H, 128, N] (keys contiguous), so
 *              that every operand of both products is K-major.
 *   descale_q, descale_k, descale_v
 *              per-head dequantisation factors, fp32 [B*H] in device memory:
 *              the real input is code * factor (per-tensor, per-head
 *              scaling; the caller chooses them, e.g. max|x| / 448).
 *   o          bf16 [B, H, N, 128]; lse fp32 [B, H, N] (natural log).
 *   causal, block_mask, kv_len as in fa_fwd; no dropout.
 * P is quantised to E4M3 for the P V product, scaled by 2^5 before
 * rounding (the running maximum is raised when a row's maximum exceeds it
 * by 3.5 in log2 units, so the scaled values stay below 2^8.5 < 448;
 * probabilities below 2^-11 of the running maximum round as E4M3
 * subnormals); the row sum uses the unquantised values. The error this adds to O is that
 * of rounding each P_ij to E4M3 (relative 2^-4): |dO_ic| is within a few
 * (2^-4/sqrt 3) sqrt(sum_j P_ij^2 V_jc^2) for independent roundings.
 * Returns FA_ERR_UNSUPPORTED for d != 128, N not a multiple of 16 (the rows
 * of vt must be 16-byte aligned), scale <= 0 or a block mask with more than
 * 1024 key tiles per row; otherwise as fa_fwd.
 */
int fa_fwd_fp8(const void* q, const void* k, const void* vt,
               const float* descale_q, const float* descale_k, const float* descale_v,
               void* o, float* lse, int B, int H, int N, int d, float scale, int causal,
               const uint8_t* block_mask, const int32_t* kv_len, void* stream);

/* Bytes of split-KV workspace: n_splits * B*H*N*(d + 1) floats (partial O,
 * then partial LSE), each part rounded up to 256 bytes; 0 for invalid sizes. */
size_t fa_fwd_splitkv_workspace_size(int B, int H, int N, int d, int n_splits);

/*
 * Bytes of backward workspace: the per-row statistics (1 KB per 128-row tile
 * of each head: -LSE and -rowsum(dO o O) of the tile's rows, padded past N)
 * plus the fp32 dQ accumulator ([B,H,N,d]), each rounded up to 256 bytes,
 * plus 256 bytes for the counter through which the backward's CTAs claim
 * work. O(B*H*N*d): the backward keeps no N x N state. Returns 0 for invalid
 * sizes.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Test hook: writes the dropout keep mask Z (uint8 0/1, [B,H,N,N], device
 * memory owned by the caller) that fa_fwd/fa_bwd apply for (p, seed).
 */
int fa_dropout_mask(uint8_t* keep, int B, int H, int N, float p, uint64_t seed, void* stream);

/*
 * Synchronises `stream`, returns the device status word (FA_OK, or
 * FA_ERR_DEVICE_TIMEOUT when a kernel's bounded wait ran out), then clears
 * it. *site (optional) receives the id of the wait that gave up.
 */
int fa_check_device_status(void* stream, int* site);

/* Human-readable name of a status code (static string). */
const char* fa_status_string(int status);

/*
 * Diagnostic: 0 = default kernels (tcgen05 for bf16 and fp16), 1 = force the
 * CUDA-core kernels for every dtype. Process-wide; returns the old value.
 */
int fa_set_kernel_path(int path);

/*
 * Test hook for the device failure path: launches one small kernel whose
 * bounded mbarrier wait (the same routine the tensor-core kernels use) waits
 * on a barrier nothing arrives at, gives up after limit_ns nanoseconds,
 * records FA_ERR_DEVICE_TIMEOUT with site 900 in the status word and returns.
 * Nothing faults or hangs; read the result with fa_check_device_status.
 */
int fa_test_wait_timeout(uint64_t limit_ns, void* stream);

/*
 * Diagnostic for the exponential roofline: launches n_blocks blocks of 512
 * threads, each thread running iters rounds of 8 independent ex2.approx.f32
 * (the softmax's exponential), so that timing the call gives the GPU's
 * exponential throughput: n_blocks * 512 * iters * 8 / time. out is
 * caller-owned device memory of n_blocks * 512 floats (a result that keeps
 * the work live). Returns FA_ERR_INVALID_ARG for a null out or counts < 1.
 */
int fa_ex2_probe(float* out, int n_blocks, int iters, void* stream);

/*
 * Diagnostic: number of CUDA kernels this library has launched in the
 * calling process (all devices, all entry points).
 */
uint64_t fa_launch_count(void);

/*
 * Diagnostic timing of a call's main kernel. While set, every fa_fwd,
 * fa_fwd_splitkv, fa_fwd_fp8 and fa_bwd call records ev_start (a cudaEvent_t) on its
 * stream immediately before launching its main kernel (the forward kernel;
 * the backward's tile kernel, or its three d = 256 passes; the CUDA-core
 * kernels) and ev_stop immediately after, so that cudaEventElapsedTime gives
 * that kernel's duration without the backward's preprocess and dQ
 * conversion. An event between two launches ends their programmatic
 * overlap, so set the events only for timing runs. Both NULL turns it off;
 * exactly one NULL returns FA_ERR_INVALID_ARG. Process-wide, not
 * thread-safe; the events stay owned by the caller.
 */
int fa_set_main_kernel_events(void* ev_start, void* ev_stop);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_H */
