// noalloc.cu -- attn_decode_noalloc: paged decode with its scratch in a static device array.
//
// Some callers cannot allocate device memory where they run decode: a serving runtime
// that has reserved nearly all of HBM for its KV-cache pool and forbids any further
// cudaMalloc, or a plugin that runs inside another framework's execution plan, where
// allocation calls are not allowed. They cannot supply the workspace attn_decode needs,
// so this entry point keeps the split-KV partials in a fixed array of this library
// instead. It allocates nothing (no cudaMalloc, cudaFree or allocating library call);
// the caller still passes every input and output.
//
// This file holds no kernel, so the array sits in a module of its own: with the CUDA
// runtime's lazy module loading (the default), a GPU holds the array's bytes only once a
// process calls attn_decode_noalloc on it, and then until the process exits. Processes
// that use only the other entry points never load it.
#include <climits>
#include <mutex>

#include "internal.h"

namespace attn {
namespace {

// Upper bound of the split-KV partials (and counters) this entry point can hold: 64 MiB.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;

// The scratch itself. On the host this name is only a stand-in for the symbol, not a
// device address: host code must never hand it to a kernel. Its address on a device
// comes from cudaGetSymbolAddress, below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device (with
// that device current) and cached.
int noalloc_scratch(int dev, void** out)
{
    if (dev < 0 || dev >= kNoAllocMaxDevices) return kErrUnsupported;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return kErrCuda;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return kOk;
}

}  // namespace
}  // namespace attn

extern "C" __attribute__((visibility("default"))) int attn_decode_noalloc(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table, const int32_t* seq_lens,
    void* o, float* lse, int num_seqs, int Hq, int Hkv, int d, int block_size, int max_blocks_per_seq,
    int num_blocks, float scale, void* stream)
{
    using namespace attn;
    // ---- arguments: the same checks as attn_decode (no CUDA call before them)
    DecodePlan plan;
    bool empty = false;
    int rc = validate_decode_args(q, k_cache, v_cache, block_table, seq_lens, o, lse, num_seqs, Hq, Hkv, d,
                                  block_size, max_blocks_per_seq, num_blocks, scale, &plan, &empty);
    if (rc != kOk || empty) return rc;
    if (plan.bytes > kNoAllocScratchBytes) return kErrWorkspace;  // sizes beyond the static scratch
    // ---- device
    int dev = 0;
    rc = check_device(&dev);
    if (rc != kOk) return rc;
    void* scratch = nullptr;
    rc = noalloc_scratch(dev, &scratch);
    if (rc != kOk) return rc;
    unsigned* err = device_error_word();
    if (!err) return kErrCuda;
    // flags = 0: the launch first zeroes the scratch's counters on the stream, so whatever
    // an earlier call left in the array does not matter
    return launch_decode(q, k_cache, v_cache, block_table, seq_lens, o, lse, num_seqs, Hq, Hkv, d, block_size,
                         max_blocks_per_seq, num_blocks, scale, scratch, plan, static_cast<cudaStream_t>(stream),
                         err, 0);
}
