// attn_api.cu -- the exported C ABI of libattn.so (declared in include/attn.h):
// argument validation, TMA descriptor encoding, the device error word, and the
// dispatch to the prefill and decode launchers.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "attn.h"
#include "internal.h"
#include "ptx.cuh"

#define ATTN_API __attribute__((visibility("default")))

// Device-detected problems land here (0 = none); read and cleared by attn_get_device_error.
__device__ unsigned g_attn_device_error;

namespace attn {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned* g_err_ptr[kMaxDevices] = {};
int g_arch_ok[kMaxDevices] = {};  // 0 unknown, 1 sm_103, -1 other
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_encode_tried = false;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

// Compute capability 10.3 (GB300) is the only target this library is built for.
int check_device(int* dev_out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return kErrCuda;
    if (dev < 0 || dev >= kMaxDevices) return kErrUnsupported;
    *dev_out = dev;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_arch_ok[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return kErrCuda;
        g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    return g_arch_ok[dev] == 1 ? kOk : kErrUnsupported;
}

namespace {
int g_num_sms[kMaxDevices] = {};
std::mutex g_sm_mu;
}  // namespace

int sm_count()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lk(g_sm_mu);
    if (g_num_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_num_sms[dev] = n;
    }
    return g_num_sms[dev];
}

unsigned* device_error_word()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attn_device_error) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<unsigned*>(p);
    }
    return g_err_ptr[dev];
}

namespace {

int encode_map(CUtensorMap* map, CUtensorMapDataType dtype, CUtensorMapSwizzle swizzle, const void* base, int rank,
               const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box)
{
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_encode_tried) {
            g_encode_tried = true;
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                    cudaSuccess &&
                q == cudaDriverEntryPointSuccess)
                g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
    }
    if (!g_encode) return kErrCuda;
    cuuint64_t gdim[5];
    cuuint64_t gstride[4];
    cuuint32_t bdim[5];
    cuuint32_t estride[5];
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i];
        bdim[i] = box[i];
        estride[i] = 1;
        if (i + 1 < rank) gstride[i] = strides_bytes[i];
    }
    const CUresult r = g_encode(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(base), gdim, gstride, bdim,
                                estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? kOk : kErrCuda;
}

}  // namespace

int encode_bf16_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box)
{
    return encode_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_SWIZZLE_128B, base, rank, dims,
                      strides_bytes, box);
}

int encode_u8_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                  const uint32_t* box)
{
    return encode_map(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_128B, base, rank, dims, strides_bytes,
                      box);
}

int encode_f32_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                   const uint32_t* box)
{
    return encode_map(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, CU_TENSOR_MAP_SWIZZLE_NONE, base, rank, dims,
                      strides_bytes, box);
}

int validate_decode_args(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                         const int32_t* seq_lens, const void* o, const float* lse, int num_seqs, int Hq, int Hkv,
                         int d, int block_size, int max_blocks_per_seq, int num_blocks, float scale,
                         DecodePlan* plan, bool* empty)
{
    *empty = false;
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !o || !lse) return kErrInvalidArg;
    if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || max_blocks_per_seq < 0 || num_blocks <= 0) return kErrInvalidArg;
    if (Hq % Hkv != 0) return kErrInvalidArg;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return kErrInvalidArg;
    if (num_seqs > 65535) return kErrInvalidArg;
    if (d != 64 && d != 128) return kErrUnsupported;
    if (block_size < 16 || block_size > 256 || block_size % 16 != 0) return kErrUnsupported;
    if (static_cast<long long>(num_blocks) * Hkv * block_size > INT32_MAX) return kErrUnsupported;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) || !aligned4(lse) ||
        !aligned4(block_table) || !aligned4(seq_lens))
        return kErrMisaligned;
    if (num_seqs == 0) {
        *empty = true;
        return kOk;
    }
    if (!decode_plan(num_seqs, Hq, Hkv, d, block_size, max_blocks_per_seq, plan)) return kErrInvalidArg;
    return kOk;
}

}  // namespace attn

using namespace attn;

extern "C" {

ATTN_API int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                      int Nq, int Nk, int d, float scale, int causal, int window, void* stream)
{
    // ---- arguments (no CUDA call before these checks)
    if ((!q || !o || !lse) && Nq != 0) return kErrInvalidArg;  // no queries: nothing is read or written
    if ((!k || !v) && Nk != 0) return kErrInvalidArg;  // no keys: k and v are never read
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq < 0 || Nk < 0) return kErrInvalidArg;
    if (Hq % Hkv != 0) return kErrInvalidArg;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return kErrInvalidArg;
    if (static_cast<long long>(B) * Hq > INT32_MAX / 2 || static_cast<long long>(B) * Hkv > INT32_MAX / 2)
        return kErrInvalidArg;
    if (d != 64 && d != 128) return kErrUnsupported;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse)) return kErrMisaligned;  // null is aligned
    if (Nq == 0) return kOk;
    // ---- device
    int dev = 0;
    int rc = check_device(&dev);
    if (rc != kOk) return rc;
    unsigned* err = device_error_word();
    if (!err) return kErrCuda;
    return launch_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, window,
                      static_cast<cudaStream_t>(stream), err);
}

ATTN_API int attn_fwd_fp8(const void* q, const void* k, const void* vt, void* o, float* lse, int B, int Hq, int Hkv,
                          int Nq, int Nk, int d, float scale, float q_descale, float k_descale, float v_descale,
                          int causal, int window, void* stream)
{
    // ---- arguments (no CUDA call before these checks)
    if ((!q || !o || !lse) && Nq != 0) return kErrInvalidArg;  // no queries: nothing is read or written
    if ((!k || !vt) && Nk != 0) return kErrInvalidArg;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq < 0 || Nk < 0) return kErrInvalidArg;
    if (Hq % Hkv != 0) return kErrInvalidArg;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return kErrInvalidArg;
    if (!(q_descale > 0.0f) || !std::isfinite(q_descale) || !(k_descale > 0.0f) || !std::isfinite(k_descale) ||
        !(v_descale > 0.0f) || !std::isfinite(v_descale))
        return kErrInvalidArg;
    if (static_cast<long long>(B) * Hq > INT32_MAX / 2 || static_cast<long long>(B) * Hkv > INT32_MAX / 2)
        return kErrInvalidArg;
    if (d != 128) return kErrUnsupported;
    if (Nk % 16 != 0) return kErrUnsupported;  // the V^T rows (Nk bytes) must stay 16-byte aligned
    if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(o) || !aligned4(lse)) return kErrMisaligned;
    if (Nq == 0) return kOk;
    // ---- device
    int dev = 0;
    int rc = check_device(&dev);
    if (rc != kOk) return rc;
    unsigned* err = device_error_word();
    if (!err) return kErrCuda;
    return launch_fwd_fp8(q, k, vt, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, q_descale, k_descale, v_descale, causal,
                          window, static_cast<cudaStream_t>(stream), err);
}

ATTN_API int attn_fwd_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                                  int Hkv, int Nq, int Nk, int d, float scale, int causal, int window,
                                  const int32_t* row_ptr, const int32_t* col_idx, void* stream)
{
    // ---- arguments (no CUDA call before these checks)
    if (!q || !o || !lse || !row_ptr || !col_idx) return kErrInvalidArg;
    if ((!k || !v) && Nk != 0) return kErrInvalidArg;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq < 0 || Nk < 0) return kErrInvalidArg;
    if (Hq % Hkv != 0) return kErrInvalidArg;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return kErrInvalidArg;
    if (static_cast<long long>(B) * Hq > INT32_MAX / 2 || static_cast<long long>(B) * Hkv > INT32_MAX / 2)
        return kErrInvalidArg;
    if (d != 64 && d != 128) return kErrUnsupported;
    if (Nk > kSparseMaxKeys) return kErrUnsupported;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse) || !aligned4(row_ptr) ||
        !aligned4(col_idx))
        return kErrMisaligned;
    if (Nq == 0) return kOk;
    // ---- device
    int dev = 0;
    int rc = check_device(&dev);
    if (rc != kOk) return rc;
    unsigned* err = device_error_word();
    if (!err) return kErrCuda;
    return launch_fwd_blocksparse(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, window, row_ptr, col_idx,
                                  static_cast<cudaStream_t>(stream), err);
}

ATTN_API int attn_prefill_paged(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                                const int32_t* q_lens, const int32_t* kv_lens, void* o, float* lse, int num_seqs,
                                int Hq, int Hkv, int d, int block_size, int max_blocks_per_seq, int num_blocks,
                                int max_q, float scale, int causal, int window, void* stream)
{
    // ---- arguments (no CUDA call before these checks)
    if (!q || !k_cache || !v_cache || !block_table || !q_lens || !kv_lens || !o || !lse) return kErrInvalidArg;
    if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || max_blocks_per_seq < 0 || num_blocks <= 0 || max_q < 0)
        return kErrInvalidArg;
    if (Hq % Hkv != 0) return kErrInvalidArg;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return kErrInvalidArg;
    if (static_cast<long long>(num_seqs) * Hq > INT32_MAX / 2) return kErrInvalidArg;
    if (d != 64 && d != 128) return kErrUnsupported;
    if (block_size < 16 || block_size > 256 || (block_size & (block_size - 1)) != 0) return kErrUnsupported;
    if (static_cast<long long>(num_blocks) * Hkv * block_size > INT32_MAX) return kErrUnsupported;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) || !aligned4(lse) ||
        !aligned4(block_table) || !aligned4(q_lens) || !aligned4(kv_lens))
        return kErrMisaligned;
    if (num_seqs == 0 || max_q == 0) return kOk;
    // ---- device
    int dev = 0;
    int rc = check_device(&dev);
    if (rc != kOk) return rc;
    unsigned* err = device_error_word();
    if (!err) return kErrCuda;
    return launch_fwd_paged(q, k_cache, v_cache, block_table, q_lens, kv_lens, o, lse, num_seqs, Hq, Hkv, d,
                            block_size, max_blocks_per_seq, num_blocks, max_q, scale, causal, window,
                            static_cast<cudaStream_t>(stream), err);
}

ATTN_API size_t attn_bwd_workspace_size(int B, int Hq, int Nq, int d)
{
    if (B <= 0 || Hq <= 0 || Nq < 0 || (d != 64 && d != 128)) return 0;
    if (static_cast<long long>(B) * Hq > INT32_MAX / 2) return 0;
    return bwd_layout(B, Hq, Nq, d).bytes;
}

ATTN_API int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                      const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk,
                      int d, float scale, int causal, int window, void* workspace, size_t workspace_bytes,
                      void* stream)
{
    // ---- arguments (no CUDA call before these checks)
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq < 0 || Nk < 0) return kErrInvalidArg;
    if (Nq > 0 && (!q || !o || !dout || !lse || !dq)) return kErrInvalidArg;
    if (Nk > 0 && (!k || !v || !dk || !dv)) return kErrInvalidArg;
    if (Hq % Hkv != 0) return kErrInvalidArg;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return kErrInvalidArg;
    if (static_cast<long long>(B) * Hq > INT32_MAX / 2 || static_cast<long long>(B) * Hkv > INT32_MAX / 2)
        return kErrInvalidArg;
    if (d != 64 && d != 128) return kErrUnsupported;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned4(lse) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return kErrMisaligned;  // null is aligned
    if (Nq == 0 && Nk == 0) return kOk;
    const BwdLayout lay = bwd_layout(B, Hq, Nq, d);
    if (!workspace || workspace_bytes < lay.bytes) return kErrWorkspace;
    if (!aligned16(workspace)) return kErrMisaligned;
    // ---- device
    int dev = 0;
    int rc = check_device(&dev);
    if (rc != kOk) return rc;
    unsigned* err = device_error_word();
    if (!err) return kErrCuda;
    return launch_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, Nq, Nk, d, scale, causal, window, workspace,
                      static_cast<cudaStream_t>(stream), err);
}

ATTN_API size_t attn_decode_workspace_size(int num_seqs, int Hq, int Hkv, int d, int block_size,
                                           int max_blocks_per_seq)
{
    if (d != 64 && d != 128) return 0;
    DecodePlan plan;
    if (!decode_plan(num_seqs, Hq, Hkv, d, block_size, max_blocks_per_seq, &plan)) return 0;
    return plan.bytes;
}

ATTN_API int attn_decode_chunk_tokens(int num_seqs, int Hq, int Hkv, int block_size, int max_blocks_per_seq)
{
    DecodePlan plan;
    if (!decode_plan(num_seqs, Hq, Hkv, 128, block_size, max_blocks_per_seq, &plan)) return 0;
    return plan.chunk;
}

ATTN_API int attn_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                         const int32_t* seq_lens, void* o, float* lse, int num_seqs, int Hq, int Hkv, int d,
                         int block_size, int max_blocks_per_seq, int num_blocks, float scale, void* workspace,
                         size_t workspace_bytes, void* stream)
{
    // ---- arguments (no CUDA call before these checks)
    DecodePlan plan;
    bool empty = false;
    int rc = validate_decode_args(q, k_cache, v_cache, block_table, seq_lens, o, lse, num_seqs, Hq, Hkv, d,
                                  block_size, max_blocks_per_seq, num_blocks, scale, &plan, &empty);
    if (rc != kOk || empty) return rc;
    if (!workspace || workspace_bytes < plan.bytes) return kErrWorkspace;
    if (!aligned16(workspace)) return kErrMisaligned;
    // ---- device
    int dev = 0;
    rc = check_device(&dev);
    if (rc != kOk) return rc;
    unsigned* err = device_error_word();
    if (!err) return kErrCuda;
    return launch_decode(q, k_cache, v_cache, block_table, seq_lens, o, lse, num_seqs, Hq, Hkv, d, block_size,
                         max_blocks_per_seq, num_blocks, scale, workspace, plan, static_cast<cudaStream_t>(stream),
                         err, 0);
}

ATTN_API int attn_get_device_error(void* stream)
{
    unsigned* err = device_error_word();
    if (!err) return kErrCuda;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned host = 0;
    if (cudaMemcpyAsync(&host, err, sizeof(unsigned), cudaMemcpyDeviceToHost, s) != cudaSuccess) return kErrCuda;
    if (cudaMemsetAsync(err, 0, sizeof(unsigned), s) != cudaSuccess) return kErrCuda;
    if (cudaStreamSynchronize(s) != cudaSuccess) return kErrCuda;
    if (host == 0) return kOk;
    if (host == kDevErrTimeout) return kErrDeviceTimeout;
    return kErrDeviceBounds;
}

ATTN_API int attn_kv_layout_version(void) { return 1; }

ATTN_API const char* attn_status_string(int status)
{
    switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_MISALIGNED: return "ATTN_ERR_MISALIGNED";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
    case ATTN_ERR_LAUNCH: return "ATTN_ERR_LAUNCH";
    case ATTN_ERR_DEVICE_TIMEOUT: return "ATTN_ERR_DEVICE_TIMEOUT";
    case ATTN_ERR_DEVICE_BOUNDS: return "ATTN_ERR_DEVICE_BOUNDS";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    default: return "ATTN_ERR_UNKNOWN";
    }
}

}  // extern "C"
