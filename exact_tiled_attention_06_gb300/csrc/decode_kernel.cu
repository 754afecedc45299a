// decode_kernel.cu -- one-query-per-sequence attention over a paged KV cache, sm_103a.
//
// Split kernel: one CTA per (key chunk, kv head [, group of 16 query heads], sequence).
//   warp 4     producer: prefetches the chunk's block-table entries, then one thread
//              streams 16-token K and V sub-pages into an 8-stage shared-memory ring
//              with TMA (128-byte swizzle), one mbarrier pair per stage
//   warps 0-3  consumers: sub-pages round-robin; S = q K^T and O += P V with
//              mma.sync m16n8k16 (the up-to-16 query heads of the kv head are the M
//              rows, so every K/V byte is read once for all of them); per-row online
//              softmax in registers; a final merge of the four warps' (m, l, o)
//              writes the chunk's normalised partial output and log-sum (log2 units).
// Combine kernel: one warp per (sequence, query head) merges the chunk partials with
//   the log-sum weights and writes bf16 O and the natural-log lse.
//
// Pages: "Modern attention kernels", "Prefill and decode need different kernels"
// (coalesced cache reads, parallel reduction across the context, grouped-query
// sharing, block indirection) and "Paged attention changes addressing" (logical
// block = pos / block_size, offset = pos % block_size, physical = table[seq, block]);
// "Attention kernels", FlashDecoding (chunk partials O_c, m_c, l_c merged with the
// online-softmax rescaling) and the GQA paragraph (read a kv head once for its
// query heads). Decode is memory-bound, so the design goal is bytes in flight, not
// tensor-core rate: mma.sync is only a compact dot-product engine here.
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kDecWarps = 4;                       // consumer warps
constexpr int kDecThreads = (kDecWarps + 1) * 32;  // + producer warp
constexpr int kDecStages = 8;
constexpr int kSub = 16;            // tokens per sub-page (one TMA box height)
constexpr int kMaxChunkBlocks = 64; // block-table entries prefetched per split
constexpr int kChunkTokens = 512;   // keys per split
constexpr int kRowsPerCta = 16;     // query heads per CTA (mma M)
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct DecCfg {
    static constexpr int kBoxes = D / 64;
    static constexpr int kBoxBytes = kSub * 128;              // 16 rows x 128 bytes
    static constexpr int kSubBytes = kBoxes * kBoxBytes;      // one K (or V) sub-page
    static constexpr int kStageBytes = 2 * kSubBytes;         // K + V
    static constexpr int kRingBytes = kDecStages * kStageBytes;
    static constexpr int kMergeStride = D + 2;                // o[D], m, l
    static constexpr int kMergeBytes = kDecWarps * kRowsPerCta * kMergeStride * 4;
    static constexpr int kDataBytes = kRingBytes > kMergeBytes ? kRingBytes : kMergeBytes;
    static constexpr int kTableOff = kDataBytes;
    static constexpr int kBarOff = kTableOff + kMaxChunkBlocks * 4;
    static constexpr int kAbortOff = kBarOff + 2 * kDecStages * 8;
    static constexpr int kUsedBytes = kAbortOff + 16;
    static constexpr int kSmemBytes = kUsedBytes + 1024;
};

struct DecParams {
    const __nv_bfloat16* q;
    const int32_t* block_table;
    const int32_t* seq_lens;
    float* part_o;    // [n_split_max][num_seqs][Hq][D]
    float* part_lse;  // [n_split_max][num_seqs][Hq], log2 units
    int num_seqs, Hq, Hkv, G, block_size, max_blocks, num_blocks;
    int chunk;
    int n_hgroups;
    float scale_log2;
    unsigned* err;
};

__device__ __forceinline__ int clamp_len(const DecParams& p, int L)
{
    const long long cap = static_cast<long long>(p.max_blocks) * p.block_size;
    if (L < 0 || L > cap) {
        report_error(p.err, kDevErrBounds);
        return L < 0 ? 0 : static_cast<int>(cap);
    }
    return L;
}

__device__ __forceinline__ uint32_t ld_u32(const __nv_bfloat16* p)
{
    return *reinterpret_cast<const uint32_t*>(p);
}

template <int D>
__global__ void __launch_bounds__(kDecThreads)
    attn_decode_split_sm103(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                            const DecParams p)
{
    using C = DecCfg<D>;
    const int split = blockIdx.x;
    const int hkv = blockIdx.y / p.n_hgroups;
    const int hg = blockIdx.y % p.n_hgroups;
    const int seq = blockIdx.z;
    const int L = clamp_len(p, p.seq_lens[seq]);
    const int tok0 = split * p.chunk;
    if (tok0 >= L) return;  // whole block: this split lies past the sequence
    const int tok1 = min(L, tok0 + p.chunk);
    const int n_sub = (tok1 - tok0 + kSub - 1) / kSub;
    const int hq0 = hkv * p.G + hg * kRowsPerCta;
    const int nvalid = min(kRowsPerCta, p.G - hg * kRowsPerCta);

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(smem);
    int* table_s = reinterpret_cast<int*>(smem + C::kTableOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbortOff);
    const uint32_t bar0 = sb + C::kBarOff;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (kDecStages + s); };
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kDecStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kDecWarps) {
        // ============================================================ producer
        const int lb0 = tok0 / p.block_size;
        const int n_lb = (tok1 - 1) / p.block_size - lb0 + 1;
        for (int i = lane; i < n_lb; i += 32) {
            int phys = p.block_table[static_cast<size_t>(seq) * p.max_blocks + lb0 + i];
            if (phys < 0 || phys >= p.num_blocks) {
                report_error(p.err, kDevErrBounds);
                phys = 0;
            }
            table_s[i] = phys;
        }
        __syncwarp();
        if (lane == 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            int issued = 0;
            for (int i = 0; i < n_sub; ++i) {
                const int s = i % kDecStages;
                if (i >= kDecStages && !mbar_wait(empty(s), ((i / kDecStages) - 1) & 1, abort_flag, p.err)) break;
                const int tok = tok0 + i * kSub;
                const int lb = tok / p.block_size;
                const int off = tok - lb * p.block_size;
                const int row = (table_s[lb - lb0] * p.Hkv + hkv) * p.block_size + off;
                const uint32_t dst = sb + s * C::kStageBytes;
                mbar_arrive_expect_tx(full(s), C::kStageBytes);
#pragma unroll
                for (int x = 0; x < C::kBoxes; ++x) tma_load_2d(dst + x * C::kBoxBytes, &tm_k, full(s), 64 * x, row);
#pragma unroll
                for (int x = 0; x < C::kBoxes; ++x)
                    tma_load_2d(dst + C::kSubBytes + x * C::kBoxBytes, &tm_v, full(s), 64 * x, row);
                ++issued;
            }
            // never leave while a copy into this block's shared memory is in flight
            for (int s = 0; s < kDecStages; ++s) {
                const int fills = issued / kDecStages + (s < issued % kDecStages ? 1 : 0);
                if (fills > 0) mbar_wait(full(s), (fills - 1) & 1, nullptr, p.err);
            }
        }
        return;
    }

    // ================================================================ consumers
    const int g = lane >> 2;   // fragment row group
    const int tig = lane & 3;  // thread in group
    const float sl2 = p.scale_log2;

    // q as A fragments (rows = query heads of this kv head, zero past nvalid)
    uint32_t qa[D / 16][4];
    {
        const __nv_bfloat16* qb = p.q + (static_cast<size_t>(seq) * p.Hq + hq0) * D;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const int col = 16 * kk + 2 * tig;
            qa[kk][0] = g < nvalid ? ld_u32(qb + g * D + col) : 0u;
            qa[kk][1] = g + 8 < nvalid ? ld_u32(qb + (g + 8) * D + col) : 0u;
            qa[kk][2] = g < nvalid ? ld_u32(qb + g * D + col + 8) : 0u;
            qa[kk][3] = g + 8 < nvalid ? ld_u32(qb + (g + 8) * D + col + 8) : 0u;
        }
    }
    float m[2] = {-INFINITY, -INFINITY};  // rows g and g + 8, scaled log2 units
    float l[2] = {0.0f, 0.0f};            // per-lane partial sums
    float o[D / 8][4];
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.0f;

    // ldmatrix lane addressing inside a 128-byte-swizzled 16-row box
    const int mat = lane >> 3, rr = lane & 7;
    const int k_token = 8 * (mat >> 1) + rr, k_unit = mat & 1;
    const int v_token = 8 * (mat & 1) + rr, v_unit = mat >> 1;

    bool ok = true;
    for (int i = warp; i < n_sub; i += kDecWarps) {
        const int s = i % kDecStages;
        if (!mbar_wait(full(s), (i / kDecStages) & 1, abort_flag, p.err)) {
            ok = false;
            break;
        }
        const uint32_t sK = sb + s * C::kStageBytes;
        const uint32_t sV = sK + C::kSubBytes;
        const int ntok = min(kSub, tok1 - (tok0 + i * kSub));
        if (ntok < kSub) {
            // Slots past the sequence end are never used: zero those V rows (they may
            // hold anything, NaN included) so that 0 * V stays 0 in the P V product.
            uint8_t* vrow = smem + s * C::kStageBytes + C::kSubBytes;
            const int units = (kSub - ntok) * 8;  // 16-byte units per box
            for (int x = 0; x < C::kBoxes; ++x)
                for (int u = lane; u < units; u += 32)
                    reinterpret_cast<uint4*>(vrow + x * C::kBoxBytes + ntok * 128)[u] = make_uint4(0u, 0u, 0u, 0u);
            __syncwarp();
        }
        // ---- S = q K^T (16 heads x 16 tokens)
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const int U = 2 * kk + k_unit;
            const uint32_t addr = sK + (U >> 3) * C::kBoxBytes + k_token * 128 + (((U & 7) ^ rr) << 4);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(addr, b0, b1, b2, b3);
            mma_16816(sc[0], qa[kk], b0, b1);
            mma_16816(sc[1], qa[kk], b2, b3);
        }
        if (ntok < kSub) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (8 * nt + 2 * tig + (e & 1) >= ntok) sc[nt][e] = -INFINITY;
        }
        // ---- online softmax per row (rows g: e = 0,1; rows g+8: e = 2,3)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float mx = fmaxf(fmaxf(sc[0][2 * h], sc[0][2 * h + 1]), fmaxf(sc[1][2 * h], sc[1][2 * h + 1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float m_cand = mx * sl2;
            if (m_cand > m[h] + kRescaleThreshold || (m[h] == -INFINITY && m_cand > -INFINITY)) {
                const float m_new = fmaxf(m[h], m_cand);
                const float alpha = (m[h] == -INFINITY) ? 0.0f : ex2_approx(m[h] - m_new);
                m[h] = m_new;
                l[h] *= alpha;
#pragma unroll
                for (int nt = 0; nt < D / 8; ++nt) {
                    o[nt][2 * h] *= alpha;
                    o[nt][2 * h + 1] *= alpha;
                }
            }
            const float base = (m[h] == -INFINITY) ? 0.0f : m[h];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 2 * h; e < 2 * h + 2; ++e) {
                    sc[nt][e] = ex2_approx(fmaf(sc[nt][e], sl2, -base));
                    l[h] += sc[nt][e];
                }
        }
        if (g >= nvalid) sc[0][0] = sc[0][1] = sc[1][0] = sc[1][1] = 0.0f;
        if (g + 8 >= nvalid) sc[0][2] = sc[0][3] = sc[1][2] = sc[1][3] = 0.0f;
        uint32_t pa[4];
        pa[0] = pack_bf16x2(sc[0][0], sc[0][1]);
        pa[1] = pack_bf16x2(sc[0][2], sc[0][3]);
        pa[2] = pack_bf16x2(sc[1][0], sc[1][1]);
        pa[3] = pack_bf16x2(sc[1][2], sc[1][3]);
        // ---- O += P V
#pragma unroll
        for (int np = 0; np < D / 16; ++np) {
            const int U = 2 * np + v_unit;
            const uint32_t addr = sV + (U >> 3) * C::kBoxBytes + v_token * 128 + (((U & 7) ^ rr) << 4);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_trans(addr, b0, b1, b2, b3);
            mma_16816(o[2 * np], pa, b0, b1);
            mma_16816(o[2 * np + 1], pa, b2, b3);
        }
        if (ntok < kSub) fence_proxy_async_smem();  // generic writes before the next TMA fill
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(s));
    }

    // ---- merge the four warps' states and write this split's partial
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
    }
    named_bar_sync(1, kDecWarps * 32);  // every consumer is done with the ring
    const bool aborted = !ok || *abort_flag;
    float* mg = reinterpret_cast<float*>(smem);
    if (!aborted) {
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int row = g + 8 * (e >> 1);
                const int col = 8 * nt + 2 * tig + (e & 1);
                mg[(warp * kRowsPerCta + row) * C::kMergeStride + col] = o[nt][e];
            }
        if (tig == 0) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = g + 8 * h;
                mg[(warp * kRowsPerCta + row) * C::kMergeStride + D] = m[h];
                mg[(warp * kRowsPerCta + row) * C::kMergeStride + D + 1] = l[h];
            }
        }
    }
    named_bar_sync(1, kDecWarps * 32);
    if (aborted || *abort_flag) return;
    const size_t part_row0 = (static_cast<size_t>(split) * p.num_seqs + seq) * p.Hq + hq0;
    for (int idx = threadIdx.x; idx < nvalid * D; idx += kDecWarps * 32) {
        const int row = idx / D, col = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, mg[(w * kRowsPerCta + row) * C::kMergeStride + D]);
        float Ls = 0.0f, Os = 0.0f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) {
            const float* st = mg + (w * kRowsPerCta + row) * C::kMergeStride;
            if (st[D] == -INFINITY) continue;
            const float wgt = ex2_approx(st[D] - M);
            Ls += st[D + 1] * wgt;
            Os += st[col] * wgt;
        }
        p.part_o[(part_row0 + row) * D + col] = Os / Ls;
        if (col == 0) p.part_lse[part_row0 + row] = M + log2f(Ls);
    }
}

template <int D>
__global__ void __launch_bounds__(128)
    attn_decode_combine_sm103(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                              const int32_t* __restrict__ seq_lens, __nv_bfloat16* __restrict__ o,
                              float* __restrict__ lse, int num_seqs, int Hq, int chunk, int max_blocks,
                              int block_size, unsigned* err)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hq = blockIdx.x * 4 + warp;
    const int seq = blockIdx.y;
    if (hq >= Hq) return;
    int L = seq_lens[seq];
    const long long cap = static_cast<long long>(max_blocks) * block_size;
    if (L < 0 || L > cap) {
        report_error(err, kDevErrBounds);
        L = L < 0 ? 0 : static_cast<int>(cap);
    }
    const int n = (L + chunk - 1) / chunk;
    const size_t out = static_cast<size_t>(seq) * Hq + hq;
    __nv_bfloat16* orow = o + out * D;
    if (n == 0) {
#pragma unroll
        for (int i = 0; i < D / 32; ++i) orow[lane + 32 * i] = __float2bfloat16_rn(0.0f);
        if (lane == 0) lse[out] = -INFINITY;
        return;
    }
    float M = -INFINITY;
    for (int c = lane; c < n; c += 32) M = fmaxf(M, part_lse[(static_cast<size_t>(c) * num_seqs + seq) * Hq + hq]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float acc[D / 32];
#pragma unroll
    for (int i = 0; i < D / 32; ++i) acc[i] = 0.0f;
    float S = 0.0f;
    for (int c = 0; c < n; ++c) {
        const size_t r = (static_cast<size_t>(c) * num_seqs + seq) * Hq + hq;
        const float w = ex2_approx(part_lse[r] - M);
        S += w;
        const float* po = part_o + r * D;
#pragma unroll
        for (int i = 0; i < D / 32; ++i) acc[i] = fmaf(w, po[lane + 32 * i], acc[i]);
    }
    const float inv = 1.0f / S;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) orow[lane + 32 * i] = __float2bfloat16_rn(acc[i] * inv);
    if (lane == 0) lse[out] = (M + log2f(S)) * kLn2;
}

template <int D>
int launch_decode_d(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                    const int32_t* seq_lens, void* o, float* lse, int num_seqs, int Hq, int Hkv, int block_size,
                    int max_blocks, int num_blocks, float scale, void* workspace, const DecodePlan& plan,
                    cudaStream_t stream, unsigned* err)
{
    using C = DecCfg<D>;
    float* part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + plan.lse_offset);
    float* part_o = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + plan.o_offset);
    if (plan.n_split_max > 0) {
        CUtensorMap tk, tv;
        const uint64_t dims[2] = {static_cast<uint64_t>(D),
                                  static_cast<uint64_t>(num_blocks) * Hkv * static_cast<uint64_t>(block_size)};
        const uint64_t strides[1] = {static_cast<uint64_t>(D) * 2};
        const uint32_t box[2] = {64u, static_cast<uint32_t>(kSub)};
        int rc = encode_bf16_map(&tk, k_cache, 2, dims, strides, box);
        if (rc != kOk) return rc;
        rc = encode_bf16_map(&tv, v_cache, 2, dims, strides, box);
        if (rc != kOk) return rc;
        DecParams prm;
        prm.q = static_cast<const __nv_bfloat16*>(q);
        prm.block_table = block_table;
        prm.seq_lens = seq_lens;
        prm.part_o = part_o;
        prm.part_lse = part_lse;
        prm.num_seqs = num_seqs;
        prm.Hq = Hq;
        prm.Hkv = Hkv;
        prm.G = Hq / Hkv;
        prm.block_size = block_size;
        prm.max_blocks = max_blocks;
        prm.num_blocks = num_blocks;
        prm.chunk = plan.chunk;
        prm.n_hgroups = plan.n_hgroups;
        prm.scale_log2 = scale * kLog2e;
        prm.err = err;
        if (cudaFuncSetAttribute(attn_decode_split_sm103<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmemBytes) != cudaSuccess)
            return kErrCuda;
        const dim3 grid(static_cast<unsigned>(plan.n_split_max), static_cast<unsigned>(Hkv * plan.n_hgroups),
                        static_cast<unsigned>(num_seqs));
        attn_decode_split_sm103<D><<<grid, kDecThreads, C::kSmemBytes, stream>>>(tk, tv, prm);
        if (cudaGetLastError() != cudaSuccess) return kErrLaunch;
    }
    const dim3 cgrid(static_cast<unsigned>((Hq + 3) / 4), static_cast<unsigned>(num_seqs));
    attn_decode_combine_sm103<D><<<cgrid, 128, 0, stream>>>(part_o, part_lse, seq_lens,
                                                           static_cast<__nv_bfloat16*>(o), lse, num_seqs, Hq,
                                                           plan.chunk, max_blocks, block_size, err);
    return cudaGetLastError() == cudaSuccess ? kOk : kErrLaunch;
}

}  // namespace

bool decode_plan(int num_seqs, int Hq, int Hkv, int d, int block_size, int max_blocks_per_seq, DecodePlan* plan)
{
    if (num_seqs <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || block_size <= 0 || max_blocks_per_seq < 0) return false;
    if (Hq % Hkv != 0 || block_size % kSub != 0 || block_size > 256) return false;
    // Split length: a whole number of blocks, at most kMaxChunkBlocks table entries.
    int chunk = kChunkTokens;
    if (chunk < block_size) chunk = block_size;
    chunk = (chunk / block_size) * block_size;
    if (chunk / block_size > kMaxChunkBlocks) chunk = kMaxChunkBlocks * block_size;
    const long long max_ctx = static_cast<long long>(max_blocks_per_seq) * block_size;
    const long long n_split = (max_ctx + chunk - 1) / chunk;
    if (n_split > 65535) return false;
    const int G = Hq / Hkv;
    plan->chunk = chunk;
    plan->n_split_max = static_cast<int>(n_split);
    plan->n_hgroups = (G + kRowsPerCta - 1) / kRowsPerCta;
    const size_t rows = static_cast<size_t>(n_split) * num_seqs * Hq;
    plan->lse_offset = 0;
    plan->o_offset = ((rows * 4 + 255) / 256) * 256;
    plan->bytes = plan->o_offset + rows * static_cast<size_t>(d) * 4;
    if (plan->bytes == 0) plan->bytes = 256;
    return true;
}

int launch_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                  const int32_t* seq_lens, void* o, float* lse, int num_seqs, int Hq, int Hkv, int d, int block_size,
                  int max_blocks_per_seq, int num_blocks, float scale, void* workspace, const DecodePlan& plan,
                  cudaStream_t stream, unsigned* err)
{
    if (d == 128)
        return launch_decode_d<128>(q, k_cache, v_cache, block_table, seq_lens, o, lse, num_seqs, Hq, Hkv, block_size,
                                    max_blocks_per_seq, num_blocks, scale, workspace, plan, stream, err);
    if (d == 64)
        return launch_decode_d<64>(q, k_cache, v_cache, block_table, seq_lens, o, lse, num_seqs, Hq, Hkv, block_size,
                                   max_blocks_per_seq, num_blocks, scale, workspace, plan, stream, err);
    return kErrUnsupported;
}

}  // namespace attn

// ============================================================================
// attn_decode_noalloc: the decode above with its scratch in a static device array.
//
// Some callers cannot allocate device memory where they run decode: a serving
// runtime that has reserved nearly all of HBM for its KV-cache pool and forbids any
// further cudaMalloc, or a plugin that runs inside another framework's execution
// plan, where allocation calls are not allowed. They cannot supply the workspace
// attn_decode needs, so this entry point uses a fixed array that lives in the
// library's module instead: every GPU that loads libattn.so holds these bytes until
// the process exits. It allocates nothing (no cudaMalloc, cudaFree or allocating
// library call); the caller still passes every input and output.
// ============================================================================
namespace attn {
namespace {

// Upper bound of the split-KV partials this entry point can hold (64 MiB).
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;

// The scratch itself. Host code must not pass this name to a kernel: on the host it
// is only a stand-in for the symbol, not a device address.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device.
int noalloc_scratch(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return kErrCuda;
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
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    auto a4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !o || !lse) return kErrInvalidArg;
    if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || max_blocks_per_seq < 0 || num_blocks <= 0) return kErrInvalidArg;
    if (Hq % Hkv != 0) return kErrInvalidArg;
    if (!(scale > 0.0f) || !isfinite(scale)) return kErrInvalidArg;
    if (num_seqs > 65535) return kErrInvalidArg;
    if (d != 64 && d != 128) return kErrUnsupported;
    if (block_size < 16 || block_size > 256 || block_size % 16 != 0) return kErrUnsupported;
    if (static_cast<long long>(num_blocks) * Hkv * block_size > INT32_MAX) return kErrUnsupported;
    if (!a16(q) || !a16(k_cache) || !a16(v_cache) || !a16(o) || !a4(lse) || !a4(block_table) || !a4(seq_lens))
        return kErrMisaligned;
    if (num_seqs == 0) return kOk;
    DecodePlan plan;
    if (!decode_plan(num_seqs, Hq, Hkv, d, block_size, max_blocks_per_seq, &plan)) return kErrInvalidArg;
    if (plan.bytes > kNoAllocScratchBytes) return kErrWorkspace;  // sizes beyond the static scratch
    int major = 0, minor = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return kErrCuda;
    if (major != 10 || minor != 3) return kErrUnsupported;
    void* scratch = nullptr;
    int rc = noalloc_scratch(&scratch);
    if (rc != kOk) return rc;
    unsigned* err = device_error_word();
    if (!err) return kErrCuda;
    return launch_decode(q, k_cache, v_cache, block_table, seq_lens, o, lse, num_seqs, Hq, Hkv, d, block_size,
                         max_blocks_per_seq, num_blocks, scale, scratch, plan, static_cast<cudaStream_t>(stream),
                         err);
}
