// decode_graph.cu -- a decode step over many layers captured once as a CUDA graph.
//
// "Attention kernels" (inference.tusharamrit.in), the passage on launch overhead at
// decode and its remedies: a decode step repeats the same launches with the same shapes
// every token, so the whole sequence of launches can be captured once and replayed as a
// single unit, which removes nearly all of the per-launch CPU cost without changing the
// memory traffic.
//
// The decode kernel reads the sequence lengths on the device and its split plan depends
// only on host-side sizes (num_seqs, heads, block size, max_blocks_per_seq), so one
// captured step stays valid while the sequences grow, as long as every buffer keeps its
// address: the caller writes the next token's queries, cache rows, block-table entries
// and lengths in place and replays the graph.
#include <climits>
#include <cmath>
#include <new>

#include "internal.h"

#define ATTN_API extern "C" __attribute__((visibility("default")))

namespace attn {
namespace {

constexpr int kMaxGraphLayers = 4096;

struct DecodeGraph {
    cudaGraphExec_t exec;
    int dev;
    int n_layers;
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace
}  // namespace attn

using namespace attn;

ATTN_API int attn_decode_graph_create(int n_layers, const void* const* q, const void* const* k_cache,
                                      const void* const* v_cache, void* const* o, float* const* lse,
                                      const int32_t* block_table, const int32_t* seq_lens, int num_seqs, int Hq,
                                      int Hkv, int d, int block_size, int max_blocks_per_seq, int num_blocks,
                                      float scale, void* workspace, size_t workspace_bytes, void** graph_out)
{
    // ---- arguments (no CUDA call before these checks)
    if (!graph_out) return kErrInvalidArg;
    *graph_out = nullptr;
    if (n_layers <= 0 || n_layers > kMaxGraphLayers) return kErrInvalidArg;
    if (!q || !k_cache || !v_cache || !o || !lse || !block_table || !seq_lens) return kErrInvalidArg;
    if (num_seqs <= 0 || Hq <= 0 || Hkv <= 0 || max_blocks_per_seq < 0 || num_blocks <= 0) return kErrInvalidArg;
    if (Hq % Hkv != 0) return kErrInvalidArg;
    if (!(scale > 0.0f) || !(scale < INFINITY)) return kErrInvalidArg;
    if (num_seqs > 65535) return kErrInvalidArg;
    if (d != 64 && d != 128) return kErrUnsupported;
    if (block_size < 16 || block_size > 256 || block_size % 16 != 0) return kErrUnsupported;
    if (static_cast<long long>(num_blocks) * Hkv * block_size > INT32_MAX) return kErrUnsupported;
    if (!aligned4(block_table) || !aligned4(seq_lens)) return kErrMisaligned;
    for (int l = 0; l < n_layers; ++l) {
        if (!q[l] || !k_cache[l] || !v_cache[l] || !o[l] || !lse[l]) return kErrInvalidArg;
        if (!aligned16(q[l]) || !aligned16(k_cache[l]) || !aligned16(v_cache[l]) || !aligned16(o[l]) ||
            !aligned4(lse[l]))
            return kErrMisaligned;
    }
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
    // ---- capture: the layers' decode launches in order on a private stream (one chain)
    cudaStream_t s = nullptr;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return kErrCuda;
    if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        cudaStreamDestroy(s);
        return kErrCuda;
    }
    // Layer 0 zeroes the counters; each launch zeroes the claim counter the next one uses
    // (the two alternate), so the later layers skip the memset and launch as programmatic
    // dependents of the layer before: their set-up and first cache reads overlap its tail.
    int slot = 0;
    for (int l = 0; l < n_layers && rc == kOk; ++l)
        rc = launch_decode(q[l], k_cache[l], v_cache[l], block_table, seq_lens, o[l], lse[l], num_seqs, Hq, Hkv, d,
                           block_size, max_blocks_per_seq, num_blocks, scale, workspace, plan, s, err,
                           l == 0 ? 0 : (kDecodeCountersZeroed | kDecodeChained), &slot);
    cudaGraph_t graph = nullptr;
    const cudaError_t end = cudaStreamEndCapture(s, &graph);
    cudaStreamDestroy(s);
    if (rc != kOk || end != cudaSuccess || !graph) {
        if (graph) cudaGraphDestroy(graph);
        cudaGetLastError();  // clear a capture error so later calls start clean
        return rc != kOk ? rc : kErrCuda;
    }
    cudaGraphExec_t exec = nullptr;
    const cudaError_t inst = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (inst != cudaSuccess || !exec) {
        cudaGetLastError();
        return kErrCuda;
    }
    DecodeGraph* h = new (std::nothrow) DecodeGraph{exec, dev, n_layers};
    if (!h) {
        cudaGraphExecDestroy(exec);
        return kErrCuda;
    }
    *graph_out = h;
    return kOk;
}

ATTN_API int attn_decode_graph_launch(void* graph, void* stream)
{
    if (!graph) return kErrInvalidArg;
    const DecodeGraph* h = static_cast<const DecodeGraph*>(graph);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return kErrCuda;
    if (dev != h->dev) return kErrInvalidArg;
    return cudaGraphLaunch(h->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess ? kOk : kErrLaunch;
}

ATTN_API int attn_decode_graph_layers(const void* graph)
{
    return graph ? static_cast<const DecodeGraph*>(graph)->n_layers : 0;
}

ATTN_API int attn_decode_graph_destroy(void* graph)
{
    if (!graph) return kOk;
    DecodeGraph* h = static_cast<DecodeGraph*>(graph);
    const cudaError_t e = cudaGraphExecDestroy(h->exec);
    delete h;
    return e == cudaSuccess ? kOk : kErrCuda;
}
