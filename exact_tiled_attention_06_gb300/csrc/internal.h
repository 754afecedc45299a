// internal.h -- host-side declarations shared by the translation units of libattn.so.
// Nothing here is exported; the public interface is include/attn.h.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

// Status values (same numbers as attn_status in include/attn.h).
enum : int {
    kOk = 0,
    kErrInvalidArg = -1,
    kErrUnsupported = -2,
    kErrMisaligned = -3,
    kErrWorkspace = -4,
    kErrLaunch = -5,
    kErrDeviceTimeout = -6,
    kErrDeviceBounds = -7,
    kErrCuda = -8,
};

// Encode a tiled TMA descriptor over a bf16 tensor with the 128-byte swizzle.
// dims[0] is the innermost (contiguous) extent; strides_bytes[i] is the byte stride
// of dimension i+1. Out-of-range box elements read as zero.
int encode_bf16_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box);

// Encode a tiled TMA descriptor over an fp32 tensor without swizzle (a box is stored
// densely, row after row); used as the target of TMA reductions.
int encode_f32_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                   const uint32_t* box);

// The current device in *dev_out; ATTN_ERR_UNSUPPORTED unless it is compute capability 10.3.
int check_device(int* dev_out);
// Number of SMs of the current device (0 on failure), looked up once per device.
int sm_count();
// Encode a tiled TMA descriptor over an 8-bit tensor (E4M3 bytes) with the 128-byte swizzle.
int encode_u8_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                  const uint32_t* box);
// Device address of the library's error word on the current device (nullptr on failure).
unsigned* device_error_word();

// Prefill (implemented in fwd_kernel.cu). Arguments are already validated.
int launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
               int Nq, int Nk, int d, float scale, int causal, int window, cudaStream_t stream,
               unsigned* err);

// FP8 prefill (implemented in fwd_kernel.cu): E4M3 q, k and transposed v, per-tensor
// scales; d = 128. Arguments are already validated.
int launch_fwd_fp8(const void* q, const void* k, const void* vt, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                   int Nk, int d, float scale, float q_descale, float k_descale, float v_descale, int causal,
                   int window, cudaStream_t stream, unsigned* err);
// Block-sparse prefill (implemented in fwd_kernel.cu): 128 x 128 blocks listed in CSR form
// (row_ptr [ceil(Nq / 128) + 1], col_idx), device pointers. Arguments are already validated.
constexpr int kSparseMaxKeys = 2048 * 128;  // the merged walk holds 4096 entries
int launch_fwd_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                           int Nq, int Nk, int d, float scale, int causal, int window, const int32_t* row_ptr,
                           const int32_t* col_idx, cudaStream_t stream, unsigned* err);

// Paged prefill (implemented in fwd_kernel.cu). Arguments are already validated.
int launch_fwd_paged(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                     const int32_t* q_lens, const int32_t* kv_lens, void* o, float* lse, int S, int Hq, int Hkv, int d,
                     int block_size, int max_blocks, int num_blocks, int max_q, float scale, int causal, int window,
                     cudaStream_t stream, unsigned* err);

// Split-KV decode plan: the chunk length and the workspace carve-up.
struct DecodePlan {
    int chunk;              // keys per split (multiple of 16 and of block_size)
    int n_split_max;        // splits of the longest possible sequence
    int n_hgroups;          // groups of at most 16 query heads per kv head
    size_t counters_bytes;  // claim counter (8 bytes), exit counter (4 + 4 pad), one completion counter
                            // per (sequence, head group)
    size_t lse_offset;      // byte offset of the partial log-sums  [n_split_max][num_seqs][Hq] fp32
    size_t o_offset;        // byte offset of the partial outputs   [n_split_max][num_seqs][Hq][d] fp32
    size_t bytes;           // total workspace bytes
};
bool decode_plan(int num_seqs, int Hq, int Hkv, int d, int block_size, int max_blocks_per_seq,
                 DecodePlan* plan);

// Decode (implemented in decode_kernel.cu). Arguments are already validated. A launch
// claims work from one of the workspace's two claim counters, and zeroes the other for
// the next launch of a chain once its own predecessor has completed. chain_slot (may be
// null: slot 0) holds the first launch's counter and receives the next launch's. flags:
//   kDecodeCountersZeroed -- the workspace's counters are known to be zero (the previous
//                            launch of the chain completed normally): no memset is enqueued;
//   kDecodeChained        -- launch as a programmatic dependent of the previous launch on
//                            the stream (its set-up and cache reads overlap that launch's
//                            tail; everything else waits for it to complete).
constexpr int kDecodeCountersZeroed = 1;
constexpr int kDecodeChained = 2;
// Host-side checks of attn_decode's arguments, shared by every decode entry point (no CUDA
// call). On kOk, *plan holds the split plan and *empty is true when there is nothing to
// compute (num_seqs == 0). The workspace is the caller's to check against plan->bytes.
int validate_decode_args(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                         const int32_t* seq_lens, const void* o, const float* lse, int num_seqs, int Hq, int Hkv,
                         int d, int block_size, int max_blocks_per_seq, int num_blocks, float scale,
                         DecodePlan* plan, bool* empty);

int launch_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                  const int32_t* seq_lens, void* o, float* lse, int num_seqs, int Hq, int Hkv, int d,
                  int block_size, int max_blocks_per_seq, int num_blocks, float scale, void* workspace,
                  const DecodePlan& plan, cudaStream_t stream, unsigned* err, int flags,
                  int* chain_slot = nullptr);

// Backward workspace: D_i [B][Hq][Nq] fp32 at dvec_offset, then the fp32 dQ accumulator
// [B][Hq][Nq][d] at dq_offset (256-byte aligned).
struct BwdLayout {
    size_t dvec_offset;
    size_t dq_offset;
    size_t bytes;
};
BwdLayout bwd_layout(int B, int Hq, int Nq, int d);

// Backward (implemented in bwd_kernel.cu). Arguments are already validated.
int launch_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
               void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale, int causal,
               int window, void* workspace, cudaStream_t stream, unsigned* err);

}  // namespace attn
