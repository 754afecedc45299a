// host_api.cu -- prefill and decode from HOST buffers: the copies to and from the device
// are part of the call.
//
// attn_fwd_host cuts the work into chunks of kv heads (with their query heads) of one
// batch entry, whose Q, K, V, O and lse rows are contiguous, and pipelines them over three
// streams: chunk c+1 is copied in while chunk c is computed and chunk c-1 is copied out,
// so the host link, the tensor cores and the return link work at the same time. The
// computation of each chunk is attn_fwd's kernel on that chunk.
#include <climits>
#include <cmath>
#include <mutex>

#include "internal.h"

#define ATTN_API extern "C" __attribute__((visibility("default")))

namespace attn {
namespace {

constexpr int kMaxHostDevices = 64;
std::mutex g_host_mu;
cudaStream_t g_copy_in[kMaxHostDevices] = {};
cudaStream_t g_copy_out[kMaxHostDevices] = {};

// The library's two copy streams of the current device, created on first use and kept
// until the process exits.
int copy_streams(int dev, cudaStream_t* in, cudaStream_t* out)
{
    std::lock_guard<std::mutex> lk(g_host_mu);
    if (!g_copy_in[dev]) {
        cudaStream_t a = nullptr, b = nullptr;
        if (cudaStreamCreateWithFlags(&a, cudaStreamNonBlocking) != cudaSuccess) return kErrCuda;
        if (cudaStreamCreateWithFlags(&b, cudaStreamNonBlocking) != cudaSuccess) {
            cudaStreamDestroy(a);
            return kErrCuda;
        }
        g_copy_in[dev] = a;
        g_copy_out[dev] = b;
    }
    *in = g_copy_in[dev];
    *out = g_copy_out[dev];
    return kOk;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Record an event on `from` and make `to` wait for it (the event is released at once; the
// dependency stays).
int link(cudaStream_t from, cudaStream_t to)
{
    cudaEvent_t e = nullptr;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return kErrCuda;
    const bool ok = cudaEventRecord(e, from) == cudaSuccess && cudaStreamWaitEvent(to, e, 0) == cudaSuccess;
    cudaEventDestroy(e);
    return ok ? kOk : kErrCuda;
}

}  // namespace
}  // namespace attn

using namespace attn;

ATTN_API int attn_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* o_h, float* lse_h, void* q_d,
                           void* k_d, void* v_d, void* o_d, float* lse_d, int B, int Hq, int Hkv, int Nq, int Nk,
                           int d, float scale, int causal, int window, int chunk_kv_heads, void* stream)
{
    // ---- arguments (no CUDA call before these checks)
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq < 0 || Nk < 0) return kErrInvalidArg;
    if (Hq % Hkv != 0) return kErrInvalidArg;
    if (Nq > 0 && (!q_h || !o_h || !lse_h || !q_d || !o_d || !lse_d)) return kErrInvalidArg;
    if (Nk > 0 && (!k_h || !v_h || !k_d || !v_d)) return kErrInvalidArg;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return kErrInvalidArg;
    if (static_cast<long long>(B) * Hq > INT32_MAX / 2 || static_cast<long long>(B) * Hkv > INT32_MAX / 2)
        return kErrInvalidArg;
    if (d != 64 && d != 128) return kErrUnsupported;
    if (!aligned16(q_d) || !aligned16(k_d) || !aligned16(v_d) || !aligned16(o_d) || !aligned4(lse_d))
        return kErrMisaligned;
    if (Nq == 0) return kOk;
    // ---- device
    int dev = 0;
    int rc = check_device(&dev);
    if (rc != kOk) return rc;
    unsigned* err = device_error_word();
    if (!err) return kErrCuda;
    cudaStream_t s_in = nullptr, s_out = nullptr;
    rc = copy_streams(dev, &s_in, &s_out);
    if (rc != kOk) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int G = Hq / Hkv;
    int c = chunk_kv_heads;
    if (c <= 0) c = Hkv >= 4 ? Hkv / 4 : 1;  // about four chunks per batch entry
    if (c > Hkv) c = Hkv;
    const size_t eq = static_cast<size_t>(Nq) * d * 2;  // bytes of one query head's Q (and O)
    const size_t ek = static_cast<size_t>(Nk) * d * 2;  // bytes of one kv head's K (and V)
    const size_t el = static_cast<size_t>(Nq) * 4;      // bytes of one query head's lse
    auto byte = [](const void* p, size_t off) { return static_cast<const char*>(p) + off; };
    auto wbyte = [](void* p, size_t off) { return static_cast<char*>(p) + off; };
    // everything queued before this call on `stream` comes first
    if ((rc = link(s, s_in)) != kOk) return rc;
    if ((rc = link(s, s_out)) != kOk) return rc;
    for (int b = 0; b < B && rc == kOk; ++b) {
        for (int h0 = 0; h0 < Hkv && rc == kOk; h0 += c) {
            const int nh = h0 + c <= Hkv ? c : Hkv - h0;
            const size_t kq = (static_cast<size_t>(b) * Hq + static_cast<size_t>(h0) * G);  // first query head
            const size_t kk = static_cast<size_t>(b) * Hkv + h0;                            // first kv head
            const size_t nq_heads = static_cast<size_t>(nh) * G;
            // in: Q, K, V of the chunk
            if (cudaMemcpyAsync(wbyte(q_d, kq * eq), byte(q_h, kq * eq), nq_heads * eq, cudaMemcpyHostToDevice,
                                s_in) != cudaSuccess)
                return kErrCuda;
            if (Nk > 0) {
                if (cudaMemcpyAsync(wbyte(k_d, kk * ek), byte(k_h, kk * ek), nh * ek, cudaMemcpyHostToDevice, s_in) !=
                        cudaSuccess ||
                    cudaMemcpyAsync(wbyte(v_d, kk * ek), byte(v_h, kk * ek), nh * ek, cudaMemcpyHostToDevice, s_in) !=
                        cudaSuccess)
                    return kErrCuda;
            }
            if ((rc = link(s_in, s)) != kOk) return rc;
            // compute the chunk on the caller's stream
            rc = launch_fwd(wbyte(q_d, kq * eq), Nk > 0 ? byte(k_d, kk * ek) : nullptr,
                            Nk > 0 ? byte(v_d, kk * ek) : nullptr, wbyte(o_d, kq * eq),
                            reinterpret_cast<float*>(wbyte(lse_d, kq * el)), 1, static_cast<int>(nq_heads), nh, Nq,
                            Nk, d, scale, causal, window, s, err);
            if (rc != kOk) return rc;
            // out: O and lse of the chunk once it is computed
            if ((rc = link(s, s_out)) != kOk) return rc;
            if (cudaMemcpyAsync(wbyte(o_h, kq * eq), byte(o_d, kq * eq), nq_heads * eq, cudaMemcpyDeviceToHost,
                                s_out) != cudaSuccess ||
                cudaMemcpyAsync(wbyte(lse_h, kq * el), byte(lse_d, kq * el), nq_heads * el, cudaMemcpyDeviceToHost,
                                s_out) != cudaSuccess)
                return kErrCuda;
        }
    }
    // the call is complete on `stream` once the last copy out is
    return link(s_out, s);
}

ATTN_API int attn_decode_host(const void* q_h, const void* k_cache_h, const void* v_cache_h,
                              const int32_t* block_table_h, const int32_t* seq_lens_h, void* o_h, float* lse_h,
                              void* q_d, void* k_cache_d, void* v_cache_d, int32_t* block_table_d,
                              int32_t* seq_lens_d, void* o_d, float* lse_d, int num_seqs, int Hq, int Hkv, int d,
                              int block_size, int max_blocks_per_seq, int num_blocks, float scale, void* workspace,
                              size_t workspace_bytes, void* stream)
{
    // ---- arguments (no CUDA call before these checks)
    if (!q_h || !k_cache_h || !v_cache_h || !block_table_h || !seq_lens_h || !o_h || !lse_h) return kErrInvalidArg;
    if (!q_d || !k_cache_d || !v_cache_d || !block_table_d || !seq_lens_d || !o_d || !lse_d) return kErrInvalidArg;
    if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || max_blocks_per_seq < 0 || num_blocks <= 0) return kErrInvalidArg;
    if (Hq % Hkv != 0) return kErrInvalidArg;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return kErrInvalidArg;
    if (num_seqs > 65535) return kErrInvalidArg;
    if (d != 64 && d != 128) return kErrUnsupported;
    if (block_size < 16 || block_size > 256 || block_size % 16 != 0) return kErrUnsupported;
    if (static_cast<long long>(num_blocks) * Hkv * block_size > INT32_MAX) return kErrUnsupported;
    if (!aligned16(q_d) || !aligned16(k_cache_d) || !aligned16(v_cache_d) || !aligned16(o_d) || !aligned4(lse_d) ||
        !aligned4(block_table_d) || !aligned4(seq_lens_d))
        return kErrMisaligned;
    if (num_seqs == 0) return kOk;
    DecodePlan plan;
    if (!decode_plan(num_seqs, Hq, Hkv, d, block_size, max_blocks_per_seq, &plan)) return kErrInvalidArg;
    if (!workspace || workspace_bytes < plan.bytes) return kErrWorkspace;
    if (!aligned16(workspace)) return kErrMisaligned;
    // ---- device
    int dev = 0;
    int rc = check_device(&dev);
    if (rc != kOk) return rc;
    unsigned* err = device_error_word();
    if (!err) return kErrCuda;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t cache = static_cast<size_t>(num_blocks) * Hkv * block_size * d * 2;
    const size_t qb = static_cast<size_t>(num_seqs) * Hq * d * 2;
    // decode needs the whole cache before it starts: the copies go in order on `stream`
    if (cudaMemcpyAsync(q_d, q_h, qb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(block_table_d, block_table_h, static_cast<size_t>(num_seqs) * max_blocks_per_seq * 4,
                        cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(seq_lens_d, seq_lens_h, static_cast<size_t>(num_seqs) * 4, cudaMemcpyHostToDevice, s) !=
            cudaSuccess ||
        cudaMemcpyAsync(k_cache_d, k_cache_h, cache, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(v_cache_d, v_cache_h, cache, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return kErrCuda;
    rc = launch_decode(q_d, k_cache_d, v_cache_d, block_table_d, seq_lens_d, o_d, lse_d, num_seqs, Hq, Hkv, d,
                       block_size, max_blocks_per_seq, num_blocks, scale, workspace, plan, s, err, 0);
    if (rc != kOk) return rc;
    if (cudaMemcpyAsync(o_h, o_d, qb, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(lse_h, lse_d, static_cast<size_t>(num_seqs) * Hq * 4, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess)
        return kErrCuda;
    return kOk;
}
