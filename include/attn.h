/*
 * attn.h -- C ABI of the GB300 (sm_103a) exact tiled attention library (libattn.so).
 *
 * Exact scaled-dot-product attention computed tile by tile with the online-softmax
 * update; the N x N score matrix never reaches device memory.
 *
 * Pages cited (by title and section):
 *   "Modern attention kernels" (blog.ecitis.org)                -- MAK
 *   "Flash attention and IO-aware attention" (aigrafen.se)      -- IOA
 *   "Attention kernels" (inference.tusharamrit.in)              -- AK
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers on the current CUDA device, row-major
 *    and contiguous. bf16 tensors and workspaces must be 16-byte aligned; fp32 and
 *    int32 arrays 4-byte aligned. bf16 tensors are passed as void*.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *    Every launch is asynchronous on that stream; the library never synchronises it.
 *  - The caller owns every buffer (inputs, outputs, workspace). The library never
 *    allocates or frees device memory. The one fixed device allocation it carries is
 *    attn_decode_noalloc's static 64 MiB scratch array, which sits in a module of its own:
 *    a GPU holds it only after attn_decode_noalloc has been called on it.
 *  - Host-detectable problems return a negative attn_status before anything is
 *    launched. Problems the kernels detect (a block-table entry out of range, a
 *    pipeline wait that ran out of time) set a device error word that
 *    attn_get_device_error() reads and clears. Kernels never trap.
 *  - Supported head dimensions: d in {64, 128}. Device: compute capability 10.3.
 */
#ifndef ATTN_H
#define ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum attn_status {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = -1,     /* null pointer, bad size, Hq % Hkv != 0, scale <= 0 ... */
    ATTN_ERR_UNSUPPORTED = -2,     /* d not in {64,128}, block_size not a multiple of 16, non-sm_103 device */
    ATTN_ERR_MISALIGNED = -3,      /* a pointer is not 16-byte aligned */
    ATTN_ERR_WORKSPACE = -4,       /* workspace missing or smaller than the *_workspace_size() figure */
    ATTN_ERR_LAUNCH = -5,          /* a kernel launch failed */
    ATTN_ERR_DEVICE_TIMEOUT = -6,  /* a bounded pipeline wait inside a kernel ran out of time */
    ATTN_ERR_DEVICE_BOUNDS = -7,   /* a kernel met a block-table entry outside [0, num_blocks) */
    ATTN_ERR_CUDA = -8             /* a CUDA runtime call made by the host side failed */
} attn_status;

/*
 * attn_fwd -- prefill attention: O = softmax(scale * Q K^T + mask) V, plus per-row lse.
 *
 *   MAK "Standard attention materializes quadratic state" (S = Q K^T / sqrt(d),
 *   P = softmax(S), O = P V); MAK "Online softmax makes tiling exact" (running max m,
 *   running sum l, unnormalised accumulator o, rescaled by exp(m - m') and divided by
 *   l once at the end); MAK "Kernel structure" (causal tiles above the diagonal are
 *   skipped, the boundary tile is masked; local attention narrows the visited range);
 *   MAK "Backward pass recomputes scores" (the per-row statistic that is saved).
 *
 *   q   : bf16 [B][Hq][Nq][d]          (input)
 *   k, v: bf16 [B][Hkv][Nk][d]         (input)  query head h reads kv head h / (Hq/Hkv)
 *   o   : bf16 [B][Hq][Nq][d]          (output) rounded to nearest even from fp32
 *   lse : fp32 [B][Hq][Nq]             (output) natural-log sum of exp of the scaled
 *                                       scores of the row; -inf for a row with no key
 *   scale  : > 0, multiplies q.k (1/sqrt(d) for standard attention)
 *   causal : nonzero -> row i sees keys j <= i + (Nk - Nq) (bottom-right alignment)
 *   window : >= 0 -> row i also needs j >= i + (Nk - Nq) - window; < 0 -> no left limit
 *   A row with no allowed key gets O = 0 and lse = -inf.
 *   Sizes: B, Hq, Hkv >= 1; Nq, Nk >= 0 (0 is a no-op); every product fits in int32 rows.
 *   Returns ATTN_OK or a negative attn_status.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale,
             int causal, int window, void* stream);

/*
 * attn_fwd_fp8 -- prefill attention over 8-bit E4M3 Q, K and V with per-tensor scales.
 *
 *   AK, the FlashAttention-3 paragraph (FP8 operands), with the tiled online-softmax
 *   computation of attn_fwd. The real inputs are Q = q_descale * q, K = k_descale * k and
 *   V = v_descale * v, where q, k, v hold E4M3 codes (OCP 8-bit floating point: sign,
 *   4-bit exponent with bias 7, 3-bit mantissa, subnormals, one NaN code per sign, no
 *   infinity). O and lse are those of attn_fwd on these real inputs with one extra
 *   rounding: each unnormalised probability, held as p = 2^6 * 2^(s - m) with m a
 *   running maximum that lags the true one by less than a factor 4 (so p <= 2^8), is
 *   rounded to E4M3 for the P V product (nearest even: relative error at most 2^-4 for
 *   p >= 2^-6, i.e. probabilities down to 2^-12 of the row maximum's weight; absolute
 *   error at most 2^-10 in p below), while the row sum uses the unrounded values.
 *
 *   q  : E4M3 bytes [B][Hq][Nq][128]      (input)
 *   k  : E4M3 bytes [B][Hkv][Nk][128]     (input)
 *   vt : E4M3 bytes [B][Hkv][128][Nk]     (input) V transposed: element (key j, column t)
 *                                          of kv head h is vt[h][t][j]
 *   o  : bf16 [B][Hq][Nq][128]            (output)
 *   lse: fp32 [B][Hq][Nq]                 (output) as attn_fwd
 *   scale, causal, window, B, Hq, Hkv, Nq, Nk: as attn_fwd. q_descale, k_descale,
 *   v_descale: > 0 and finite (else ATTN_ERR_INVALID_ARG). d must be 128 and Nk a
 *   multiple of 16 (the V^T rows must stay 16-byte aligned); otherwise
 *   ATTN_ERR_UNSUPPORTED. NaN codes in the inputs propagate as in any IEEE arithmetic.
 *   Enqueues one kernel on `stream`. Returns ATTN_OK or a negative attn_status.
 */
int attn_fwd_fp8(const void* q, const void* k, const void* vt, void* o, float* lse,
                 int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale,
                 float q_descale, float k_descale, float v_descale,
                 int causal, int window, void* stream);

/*
 * attn_fwd_blocksparse -- prefill restricted to the 128 x 128 score blocks a block index
 * lists.
 *
 *   MAK "Kernel structure" (an arbitrary sparse mask needs an index structure telling the
 *   kernel which blocks exist; tiles that do not exist are never visited); MAK, the table
 *   of attention variants (sparse attention visits selected score blocks); AK, sparse
 *   attention (global plus local patterns keep softmax attention and restrict positions).
 *
 *   q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale: as attn_fwd.
 *   row_ptr : int32 [ceil(Nq / 128) + 1] (device) CSR offsets into col_idx, row_ptr[0] = 0
 *   col_idx : int32 [row_ptr[last]] (device) key blocks (keys [128 c, 128 c + 128)) listed
 *             for each query block (rows [128 r, 128 r + 128)), strictly ascending, each
 *             below ceil(Nk / 128); one index serves every batch entry and head.
 *   causal, window: as attn_fwd, applied element by element inside the listed blocks.
 *   Row i attends key j when block (i / 128, j / 128) is listed and the causal / window
 *   mask allows (i, j); a row with no such key gets O = 0 and lse = -inf.
 *   Nk <= 262144 and at most 2048 blocks per query block. An entry out of range or out of
 *   order sets ATTN_ERR_DEVICE_BOUNDS in the device error word and is skipped.
 *   Enqueues one kernel on `stream`. Returns ATTN_OK or a negative attn_status.
 */
int attn_fwd_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale,
                         int causal, int window, const int32_t* row_ptr, const int32_t* col_idx,
                         void* stream);

/*
 * attn_prefill_paged -- prefill of several sequences against a paged KV cache (chunked
 * prefill): each sequence's new queries attend to its cached tokens, the new ones included.
 *
 *   MAK "Paged attention changes addressing" (logical block = pos / block_size, offset =
 *   pos % block_size, physical = block_table[seq, block], address = base + physical *
 *   block_stride + offset * token_stride); MAK "Prefill and decode need different
 *   kernels" and AK (tiled prefill, paged cache: one engine uses both), with the tiled
 *   online-softmax computation of attn_fwd.
 *
 *   q          : bf16 [num_seqs][Hq][max_q][d]      (input) rows i >= q_lens[s] are not read
 *   k_cache,
 *   v_cache    : bf16 [num_blocks][Hkv][block_size][d] (input, layout version 1)
 *   block_table: int32 [num_seqs][max_blocks_per_seq] (input, device)
 *   q_lens     : int32 [num_seqs] (device) new queries of each sequence, 0 <= q_len <= max_q
 *   kv_lens    : int32 [num_seqs] (device) tokens of each sequence in the cache, new ones
 *                included: q_len <= kv_len <= max_blocks_per_seq * block_size. Query row i
 *                of sequence s is position kv_len - q_len + i (bottom-right alignment).
 *   o          : bf16 [num_seqs][Hq][max_q][d]      (output) rows i >= q_lens[s] untouched
 *   lse        : fp32 [num_seqs][Hq][max_q]         (output) as attn_fwd; rows past q_len untouched
 *   block_size : a power of two in [16, 256]. causal, window, scale: as attn_fwd, with
 *                Nq = q_len and Nk = kv_len per sequence.
 *   Cache slots past a sequence's end (the tail of its last block) are never used, whatever
 *   they hold. A block-table entry outside [0, num_blocks), or lengths breaking the bounds
 *   above, set ATTN_ERR_DEVICE_BOUNDS in the device error word (that sequence's output is
 *   then undefined). num_blocks * Hkv * block_size must stay below 2^31.
 *   Enqueues one kernel on `stream`. Returns ATTN_OK or a negative attn_status.
 */
int attn_prefill_paged(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_table, const int32_t* q_lens, const int32_t* kv_lens,
                       void* o, float* lse, int num_seqs, int Hq, int Hkv, int d, int block_size,
                       int max_blocks_per_seq, int num_blocks, int max_q, float scale,
                       int causal, int window, void* stream);

/*
 * attn_bwd_workspace_size -- bytes of scratch attn_bwd needs: D_i = rowsum(dO o O) in
 * fp32 [B][Hq][Nq] (256-byte aligned), then an fp32 dQ accumulator [B][Hq][Nq][d].
 * Returns 0 for invalid sizes.
 */
size_t attn_bwd_workspace_size(int B, int Hq, int Nq, int d);

/*
 * attn_bwd -- gradients of attention: dQ, dK, dV of L = sum(dO o O) for the O that
 *   attn_fwd computes from the same q, k, v, scale, causal and window.
 *
 *   MAK "Backward pass recomputes scores" (keeping P for the backward would cost
 *   quadratic memory, so only a per-row statistic is kept and the score tiles are
 *   formed again); IOA, the backward-pass paragraph (two numbers per row kept, the
 *   probabilities rebuilt tile by tile); AK, the rematerialisation passage (more FLOPs,
 *   less memory traffic).
 *   With P_ij = exp(scale q_i.k_j - lse_i) (0 where masked):
 *     dV_j = sum_i P_ij dO_i,   dP_ij = dO_i . v_j,   D_i = dO_i . O_i,
 *     dS_ij = P_ij (dP_ij - D_i),   dQ_i = scale sum_j dS_ij k_j,   dK_j = scale sum_i dS_ij q_i.
 *
 *   q, o, dout : bf16 [B][Hq][Nq][d]     (input) o and lse as written by attn_fwd
 *   k, v       : bf16 [B][Hkv][Nk][d]    (input)
 *   lse        : fp32 [B][Hq][Nq]        (input) from attn_fwd
 *   dq         : bf16 [B][Hq][Nq][d]     (output)
 *   dk, dv     : bf16 [B][Hkv][Nk][d]    (output) summed over the Hq/Hkv query heads
 *                                         that share each kv head
 *   scale, causal, window: as for attn_fwd.  A row with no allowed key (lse = -inf)
 *   contributes nothing and gets dQ = 0.
 *   P and dS are rounded to bf16 before they enter the tensor-core products, with fp32
 *   accumulation (the same precision as the forward's P V product).
 *   workspace : device scratch of at least attn_bwd_workspace_size(B, Hq, Nq, d) bytes,
 *               16-byte aligned; no initialisation needed; clobbered. Two calls that
 *               share a workspace must not overlap on the device. No output may alias
 *               an input or the workspace.
 *   Sizes: as for attn_fwd; Nq = 0 gives dK = dV = 0, Nk = 0 gives dQ = 0.
 *   Enqueues three kernels on `stream` (statistics, main, dQ conversion).
 *   Returns ATTN_OK or a negative attn_status.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
             const float* lse, void* dq, void* dk, void* dv,
             int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale,
             int causal, int window, void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_decode_workspace_size -- bytes of scratch attn_decode needs for these sizes.
 *
 *   AK FlashDecoding: each chunk of a sequence's keys produces a partial output with
 *   its own max and sum; the partials are merged afterwards. The workspace holds
 *   the work counters (four completion counters per sequence and kv head group, one
 *   per column slice a team of warps merges) and those partials (fp32) for the largest
 *   possible split count of the batch.
 *   Returns 0 for invalid sizes.
 */
size_t attn_decode_workspace_size(int num_seqs, int Hq, int Hkv, int d, int block_size,
                                  int max_blocks_per_seq);

/*
 * attn_decode -- one query token per sequence against a paged KV cache.
 *
 *   MAK "Prefill and decode need different kernels" (decode is memory-bound: read the
 *   cache in wide contiguous pieces, spread one query's context over many blocks and
 *   combine their results, let a kv head serve all of its query heads, follow the
 *   block table); MAK "Paged attention changes addressing" (logical block =
 *   pos / block_size, offset = pos % block_size, physical = block_table[seq, block],
 *   address = base + physical * block_stride + offset * token_stride);
 *   AK FlashDecoding (split-KV partials merged with the online-softmax rescaling);
 *   AK GQA (the query heads of one kv head read it once).
 *
 *   q          : bf16 [num_seqs][Hq][d]                         (input)
 *   k_cache,
 *   v_cache    : bf16 [num_blocks][Hkv][block_size][d]          (input, layout version 1)
 *   block_table: int32 [num_seqs][max_blocks_per_seq]          (input) physical block of
 *                each logical block; entries past a sequence's length are never read
 *   seq_lens   : int32 [num_seqs]                               (input, device) keys per
 *                sequence, 0 <= L <= max_blocks_per_seq * block_size (not read by the host)
 *   o          : bf16 [num_seqs][Hq][d]                         (output)
 *   lse        : fp32 [num_seqs][Hq]                            (output) -inf when L = 0
 *   block_size : multiple of 16, at most 256.  num_seqs <= 65535 (0 is a no-op).
 *   num_blocks * Hkv * block_size must stay below 2^31 (cache rows are addressed
 *   with 32-bit TMA coordinates).
 *   workspace  : device scratch of at least attn_decode_workspace_size(...) bytes,
 *                16-byte aligned; contents need no initialisation and are clobbered.
 *   Two calls that share a workspace must not overlap on the device.
 *   Cache slots past a sequence's length (the tail of its last block) are never used,
 *   whatever they hold. A block-table entry outside [0, num_blocks) sets
 *   ATTN_ERR_DEVICE_BOUNDS in the device error word (the output is then undefined).
 *   Enqueues a 4-byte-granular memset of the workspace's counters and one kernel per
 *   2048 sequences on `stream`. Returns ATTN_OK or a negative attn_status.
 */
int attn_decode(const void* q, const void* k_cache, const void* v_cache,
                const int32_t* block_table, const int32_t* seq_lens, void* o, float* lse,
                int num_seqs, int Hq, int Hkv, int d, int block_size, int max_blocks_per_seq,
                int num_blocks, float scale, void* workspace, size_t workspace_bytes,
                void* stream);

/*
 * attn_decode_noalloc -- attn_decode without a caller-supplied workspace.
 *
 *   No counterpart in the pages: this is a deployment convenience. Some callers cannot
 *   allocate device memory where they run decode (a serving runtime that reserved
 *   nearly all of HBM for its KV-cache pool and forbids further cudaMalloc, or a
 *   plugin running inside another framework's execution plan, where allocation calls
 *   are not allowed). This variant keeps the split-KV partials in a static device
 *   array inside libattn.so instead: 64 MiB, in a module that holds nothing else, so a
 *   GPU holds it from the first attn_decode_noalloc call on that device (the runtime
 *   loads the module then) until the process exits; processes that never call it never
 *   hold it. It allocates nothing (no cudaMalloc, cudaFree or allocating library call);
 *   the caller still passes every input and output, with the same meaning, layout and
 *   alignment as attn_decode, and gets the same argument checks and statuses.
 *
 *   Returns ATTN_ERR_WORKSPACE when attn_decode_workspace_size(...) for these sizes
 *   exceeds 64 MiB, before anything is launched. The first call on a device, with that
 *   device current, looks up the array's device address (cudaGetSymbolAddress) and
 *   caches it; make that first call before any stream capture. Every call shares the
 *   one array, so calls that overlap on the GPU (on different streams, or from different
 *   threads) race and corrupt each other's results; serialise them. The array keeps the
 *   last call's contents: each call first zeroes the counters it needs on the stream
 *   (one small cudaMemsetAsync), and reads only partials it has written itself.
 */
int attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_table, const int32_t* seq_lens, void* o, float* lse,
                        int num_seqs, int Hq, int Hkv, int d, int block_size, int max_blocks_per_seq,
                        int num_blocks, float scale, void* stream);

/*
 * attn_decode_graph_create / _launch / _layers / _destroy -- one decode step over many
 * layers, captured once as a CUDA graph and replayed with a single launch per step.
 *
 *   AK, the passage on launch overhead at decode and its remedies (a decode step repeats
 *   identical launches, so they are recorded a single time and re-issued together: the
 *   host pays per step instead of per launch, while the bytes moved do not change),
 *   applied to the decode of attn_decode.
 *
 *   create: n_layers in [1, 4096]. q, k_cache, v_cache, o, lse are HOST arrays of
 *     n_layers DEVICE pointers, layer l's tensors with the layouts of attn_decode; the
 *     arrays are read during the call only. block_table, seq_lens, the sizes, scale and
 *     workspace are those of attn_decode and are shared by every layer (one block table
 *     per sequence; each layer has its own cache). The layers run in order, one after
 *     another, so one workspace of attn_decode_workspace_size(...) bytes serves them all.
 *     Captures, on a private stream, one counter memset and then each layer's decode
 *     kernel(s); a decode launch leaves its completion counters at zero and zeroes the
 *     claim counter of the next launch (two alternate), so layers after the first need
 *     no memset and are launched as programmatic dependents of the layer
 *     before (their set-up and first cache reads overlap its tail; everything they write
 *     waits for it to complete). Then instantiates the graph; nothing runs. On success
 *     *graph_out holds an opaque handle (host memory and CUDA graph objects owned by the
 *     library until attn_decode_graph_destroy); on failure it is NULL. Errors: the
 *     attn_decode statuses, checked for every layer before any CUDA call; ATTN_ERR_CUDA if
 *     the capture or the instantiation fails. Call it outside any stream capture of the
 *     calling thread.
 *   launch: enqueues the captured step on `stream` (a stream of the device that was
 *     current at create; another device gives ATTN_ERR_INVALID_ARG). The graph holds
 *     every pointer and size given at create: keep those buffers alive and in place. It
 *     reads the CONTENTS at launch time, so between launches the caller may rewrite the
 *     queries, the cache rows, the block table and seq_lens (the lengths may grow up to
 *     max_blocks_per_seq * block_size: the split plan depends on sizes only). A layer's
 *     caches must not overlap an earlier layer's o or lse (a dependent layer starts
 *     reading its caches before its predecessor ends; it reads q only after). Two launches
 *     of one graph, or a launch and another call that share its workspace, must not
 *     overlap on the device. The device error word works as for attn_decode.
 *   layers: the layer count of a handle (0 for NULL).
 *   destroy: releases the handle (NULL is a no-op). Do not destroy a graph whose launch
 *     may still be running on the device; synchronise the stream first.
 */
int attn_decode_graph_create(int n_layers, const void* const* q, const void* const* k_cache,
                             const void* const* v_cache, void* const* o, float* const* lse,
                             const int32_t* block_table, const int32_t* seq_lens, int num_seqs, int Hq,
                             int Hkv, int d, int block_size, int max_blocks_per_seq, int num_blocks,
                             float scale, void* workspace, size_t workspace_bytes, void** graph_out);
int attn_decode_graph_launch(void* graph, void* stream);
int attn_decode_graph_layers(const void* graph);
int attn_decode_graph_destroy(void* graph);

/*
 * attn_fwd_host / attn_decode_host -- attn_fwd and attn_decode from HOST buffers: the
 * copies to the device and back are part of the call.
 *
 *   No counterpart in the pages: the end-to-end entry points of the library.
 *   The *_h arguments are host pointers, the *_d arguments device buffers of the same
 *   shapes and layouts (the caller owns both; inputs are copied into the *_d buffers, the
 *   outputs computed there and copied back to the *_h buffers). Page-locked host memory
 *   (cudaHostAlloc / cudaHostRegister) is needed for the copies to overlap anything; with
 *   pageable memory the result is the same and the copies are synchronous. Sizes, scale,
 *   masks, workspace and errors are those of attn_fwd / attn_decode; d_* pointers must meet
 *   their alignment rules. Everything is ordered after the work already queued on `stream`
 *   and complete on `stream` when the last copy back is; the host buffers must stay valid
 *   and unchanged until then. The results are bitwise those of attn_fwd / attn_decode.
 *
 *   attn_fwd_host pipelines chunks of chunk_kv_heads kv heads (with their query heads) of
 *   one batch entry over the library's two copy streams (created on first use, per device,
 *   kept until exit) and `stream`: chunk c+1 is copied in while chunk c is computed and
 *   chunk c-1 is copied out. chunk_kv_heads <= 0 picks max(1, Hkv / 4).
 *   attn_decode_host copies q, the block table, the lengths and both caches in, runs the
 *   decode, and copies O and lse out, all in order on `stream` (the decode reads the whole
 *   cache, so there is nothing to overlap within one call).
 */
int attn_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* o_h, float* lse_h,
                  void* q_d, void* k_d, void* v_d, void* o_d, float* lse_d,
                  int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale, int causal, int window,
                  int chunk_kv_heads, void* stream);
int attn_decode_host(const void* q_h, const void* k_cache_h, const void* v_cache_h,
                     const int32_t* block_table_h, const int32_t* seq_lens_h, void* o_h, float* lse_h,
                     void* q_d, void* k_cache_d, void* v_cache_d, int32_t* block_table_d,
                     int32_t* seq_lens_d, void* o_d, float* lse_d, int num_seqs, int Hq, int Hkv, int d,
                     int block_size, int max_blocks_per_seq, int num_blocks, float scale,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_selftest_wait_timeout -- failure detection without a fault: launches one block
 * whose pipeline-barrier wait is never satisfied. The wait gives up after its time limit
 * (about 2 s, as every wait in the library) and records ATTN_ERR_DEVICE_TIMEOUT in the
 * device error word; attn_get_device_error() then returns it, and the context stays
 * usable. For tests of the error path; nothing else calls it. Enqueues one kernel on
 * `stream`; returns ATTN_OK or a negative attn_status.
 */
int attn_selftest_wait_timeout(void* stream);

/*
 * attn_decode_chunk_tokens -- keys per split-KV chunk attn_decode uses for these sizes
 * (AK FlashDecoding: the chunk length of the split). 512 keys, halved (down to 128, and
 * staying a multiple of block_size) while the work items -- chunks of the longest
 * possible sequence x num_seqs x kv heads x groups of 16 query heads -- number fewer
 * than the 1216 worker warps of a full GB300. Depends on sizes only, never on the
 * lengths. Informational; 0 if invalid.
 */
int attn_decode_chunk_tokens(int num_seqs, int Hq, int Hkv, int block_size, int max_blocks_per_seq);

/*
 * attn_get_device_error -- wait for `stream`, then read and clear the device error
 * word of the current device. Returns ATTN_OK, ATTN_ERR_DEVICE_TIMEOUT,
 * ATTN_ERR_DEVICE_BOUNDS, or ATTN_ERR_CUDA if the synchronisation itself failed.
 */
int attn_get_device_error(void* stream);

/*
 * attn_kv_layout_version -- identity of the paged-cache layout the library reads
 * (MAK "Failure modes", page-table mismatch: encode layout identity).
 * Version 1 = [num_blocks][Hkv][block_size][d], bf16, block_table int32 row-major.
 */
int attn_kv_layout_version(void);

/* attn_status_string -- static, human-readable name of a status code. */
const char* attn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H */
