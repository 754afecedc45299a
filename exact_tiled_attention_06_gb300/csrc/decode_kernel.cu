// decode_kernel.cu -- one-query-per-sequence attention over a paged KV cache, sm_103a.
//
// One persistent kernel, one block per SM, eight independent worker warps per block.
// A work item is (key chunk of 512 tokens -- fewer for a small batch, down to 128 -- kv
// head [, group of 16 query heads], sequence). Each block first reads the sequence
// lengths (on the device: the host never reads them), orders the sequences by chunk
// count and prefix-sums the counts in shared memory, so items exist only inside
// sequences. When the launch has at most half as many items as warps, a team of T = 2
// or 4 warps of a block shares each item (its sub-pages dealt round-robin); otherwise
// T = 1. Each team then repeatedly:
//   * takes an item: its own index first, then the next one from a device-wide counter
//     (items in sequence order -- most chunks first -- then head group, then chunk),
//   * loads the item's block-table entries (one per lane) and the query heads of its
//     kv head as mma.sync A fragments,
//   * streams the chunk's 16-token K and V sub-pages with TMA (128-byte swizzle) into
//     its own 3-stage shared-memory ring, re-filling a stage as soon as it is used,
//   * computes S = q K^T and O += P V with mma.sync m16n8k16 (the query heads of the kv
//     head are the M rows: every K/V byte is read once for the whole group) with a
//     per-row online softmax in registers,
//   * (a team) combines its members' partials in shared memory, member w taking the
//     columns [w D/T, (w + 1) D/T),
//   * writes the chunk's normalised partial and log-sum; the warp that completes the
//     last chunk of a (sequence, head group) -- per column slice for a team -- merges
//     all its partials and writes O and lse. A sequence that fits in one chunk is
//     written directly.
// A launch leaves its completion counters at zero (each is reset by the warp that merges)
// and claims from one of two counters, zeroing the other for the next launch of a chain;
// every block signals programmatic dependents at its start and waits for its own
// predecessor before touching outputs or workspace, so a chain of decode launches (the
// layers of a captured step) needs one memset, no block waits at its exit, and each
// launch's set-up overlaps the previous one's tail.
//
// Pages: "Modern attention kernels", "Prefill and decode need different kernels"
// (decode is memory-bound: wide contiguous cache reads, one query's context spread over
// many blocks and combined, a kv head read once for its query heads, the block table
// followed, many sequences in one launch) and "Paged attention changes
// addressing" (logical block = pos / block_size, offset = pos % block_size, physical =
// table[seq, block]); "Attention kernels", FlashDecoding (chunk partials O_c, m_c, l_c
// merged with the online-softmax rescaling) and the GQA paragraph. Decode is
// memory-bound, so the design goal is bytes in flight (8 warps x 3 stages x 8 KB per
// SM), not tensor-core rate: mma.sync is only a compact dot-product engine here.
#include <climits>
#include <cmath>
#include <cstdint>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kDecWarps = 8;          // independent worker warps per block
constexpr int kSub = 16;              // tokens per sub-page (one TMA box height)
constexpr int kChunkTokens = 512;     // keys per work item (the most)
constexpr int kMinChunkTokens = 128;  // keys per work item (the fewest the planner goes down to)
constexpr long long kTargetItems = 152 * 8;  // worker warps of a full GB300 (152 SMs x 8)
constexpr int kMaxChunkBlocks = 32;   // block-table entries per item (one per lane)
constexpr int kRowsPerItem = 16;      // query heads per item (mma M)
constexpr int kPlanMaxSeqs = 2048;    // sequences per launch (the block's length table)
constexpr int kMaxTeamAll = 4;        // warps sharing an item at most, any head size
static_assert(kPlanMaxSeqs <= 2048, "the sort key holds the sequence in 11 bits");
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct DecCfg {
    static constexpr int kBoxes = D / 64;
    static constexpr int kBoxBytes = kSub * 128;              // 16 rows x 128 bytes
    static constexpr int kSubBytes = kBoxes * kBoxBytes;      // one K (or V) sub-page
    static constexpr int kStageBytes = 2 * kSubBytes;         // K + V
    static constexpr int kStages = (D == 128) ? 3 : 6;        // per warp
    static constexpr int kWarpRingBytes = kStages * kStageBytes;
    static constexpr int kBarOff = kDecWarps * kWarpRingBytes;
    static constexpr int kUsedBytes = kBarOff + kDecWarps * kStages * 8;
    // lengths, chunk prefix, per-warp scan totals, sequences in heaviest-first order
    static constexpr int kPlanOff = kUsedBytes;
    static constexpr int kPlanBytes = (3 * kPlanMaxSeqs + 2 + kDecWarps) * 4;
    // teams: claimed item per team (two slots, by iteration parity), abort flags, and
    // each warp's (m, l) per row for the team's combine
    static constexpr int kMaxTeam = D / 32;  // warps per item at most (a lane owns >= 4 columns)
    static_assert(kMaxTeam <= kMaxTeamAll, "completion counters per (sequence, head group)");
    static constexpr int kTeamOff = kPlanOff + kPlanBytes;
    static constexpr int kTeamBytes = kDecWarps * 2 * 8 + kDecWarps * 4 + kDecWarps * kRowsPerItem * 8;
    static constexpr int kRowF = D + 8;      // floats per row of a warp's partial O in its ring
    static_assert(kRowsPerItem * kRowF * 4 <= kStages * 2 * kBoxes * kBoxBytes, "partial O fits the ring");
    static constexpr int kSmemBytes = kTeamOff + kTeamBytes + 1024;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static_assert(kTeamOff % 8 == 0, "team area alignment");
};

struct DecParams {
    const __nv_bfloat16* q;
    const int32_t* block_table;
    const int32_t* seq_lens;
    __nv_bfloat16* o;
    float* lse;
    unsigned long long* work;       // dynamic items claimed after each team's first
    unsigned long long* work_next;  // the claim counter of the next launch of a chain
    int* done;                 // [num_seqs][HG] chunks finished
    float* part_o;             // [n_split_max][num_seqs][Hq][D]
    float* part_lse;           // [n_split_max][num_seqs][Hq], log2 units
    int num_seqs, Hq, Hkv, G, block_size, max_blocks, num_blocks;
    int chunk;
    int n_hgroups;
    int HG;                    // Hkv * n_hgroups
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

// A completion count with acquire-release semantics at GPU scope. Called by one lane after
// a warp barrier: the release covers the partial the whole warp stored before the barrier,
// and for the last arriver the acquire makes every other chunk's partial visible to the
// loads its warp makes after the next warp barrier. (A fence before a relaxed count and
// another after it cost the small-batch step 0.4 us per layer.)
__device__ __forceinline__ int atom_add_acq_rel(int* addr, int v)
{
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ uint32_t ld_u32(const __nv_bfloat16* p)
{
    return *reinterpret_cast<const uint32_t*>(p);
}

// Merge of one (sequence, head group)'s chunk partials for the column slice
// [tw S, (tw + 1) S), S = 32 VEC: eight lanes per query head (four heads at a time), each
// lane owning VEC float4 (4 VEC consecutive columns) of the slice. The chunks' log-sums
// are spread over a head's eight lanes (chunk c on lane c % 8, up to 64 chunks held in
// registers) and reduced there; their weights reach the other lanes by shuffle. A lane
// holds kLoads float4 of partial rows at once, kLoads / VEC chunks, so the rows of up to
// 4 (VEC 4), 16 (VEC 2) or 32 (VEC 1) chunks arrive in one round trip; the first group is
// requested before the log-sums.
template <int D, int VEC>
__device__ __forceinline__ void merge_slice(const DecParams& p, int seq, int hq0, int nvalid, int n_splits, int tw,
                                            int lane)
{
    constexpr int kCols = 4 * VEC;     // this lane's columns
    constexpr int kSlice = 8 * kCols;  // the slice's columns
    // float4 of partial rows a lane holds at once: 32 for a team's narrow slice (a small
    // batch: its merges end the launch, one round trip matters), 16 for a whole row (a large
    // batch: merges overlap other warps' streaming, fewer registers in flight measured better)
    constexpr int kLoads = VEC == 4 ? 16 : 32;
    constexpr int kGroup = kLoads / VEC;  // chunks per group of loads
    constexpr int kRun = kGroup < 8 ? kGroup : 8;  // chunks whose weights one register holds
    static_assert(kGroup % kRun == 0 && 8 % kRun == 0, "weight runs tile the group");
    constexpr int kHeld = 8;           // log-sums per lane in registers
    static_assert(kSlice <= D, "slice within the head");
    const int slot_row = lane >> 3;    // head within the group of four
    const int cg = lane & 7;           // column group (and chunk c = cg mod 8)
    const int src0 = slot_row * 8;
    const size_t split_stride = static_cast<size_t>(p.num_seqs) * p.Hq;  // rows per chunk
    const size_t cstride = split_stride * (D / 4);                       // float4 per chunk
    for (int rb = 0; rb < nvalid; rb += 4) {
        const int row = rb + slot_row;
        const bool live = row < nvalid;
        const size_t r0 = static_cast<size_t>(seq) * p.Hq + hq0 + (live ? row : nvalid - 1);
        const float* lse_r = p.part_lse + r0;
        const int col0 = tw * kSlice + cg * kCols;
        const float4* po = reinterpret_cast<const float4*>(p.part_o + r0 * D + col0);
        float acc[kCols];
#pragma unroll
        for (int t = 0; t < kCols; ++t) acc[t] = 0.0f;
        float4 v[kGroup][VEC];
        auto load_group = [&](int c) {
#pragma unroll
            for (int k = 0; k < kGroup; ++k)
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    v[k][j] = c + k < n_splits ? __ldcg(po + (c + k) * cstride + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        };
        // chunks r kRun .. r kRun + kRun - 1 of the loaded group, weights from register hreg
        // of lanes src0 + off .. src0 + off + kRun - 1
        auto add_run = [&](int r, float hreg, int off) {
#pragma unroll
            for (int k = 0; k < kRun; ++k) {
                const float w = __shfl_sync(0xffffffffu, hreg, src0 + off + k);
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    const float4 x = v[kRun * r + k][j];
                    acc[4 * j + 0] = fmaf(w, x.x, acc[4 * j + 0]);
                    acc[4 * j + 1] = fmaf(w, x.y, acc[4 * j + 1]);
                    acc[4 * j + 2] = fmaf(w, x.z, acc[4 * j + 2]);
                    acc[4 * j + 3] = fmaf(w, x.w, acc[4 * j + 3]);
                }
            }
        };
        float M = -INFINITY, S = 0.0f;
        if (n_splits <= 8 * kHeld) {
            load_group(0);
            float hl[kHeld];
#pragma unroll
            for (int k = 0; k < kHeld; ++k) {
                const int c = cg + 8 * k;
                hl[k] = c < n_splits ? __ldcg(lse_r + c * split_stride) : -INFINITY;
            }
#pragma unroll
            for (int k = 0; k < kHeld; ++k) M = fmaxf(M, hl[k]);
            M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 1));
            M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 2));
            M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 4));
#pragma unroll
            for (int k = 0; k < kHeld; ++k) {
                hl[k] = ex2_approx(hl[k] - M);  // the chunk's weight (0 past n_splits)
                S += hl[k];
            }
            S += __shfl_xor_sync(0xffffffffu, S, 1);
            S += __shfl_xor_sync(0xffffffffu, S, 2);
            S += __shfl_xor_sync(0xffffffffu, S, 4);
            for (int c = 0; c < n_splits; c += kGroup) {
                if (c > 0) load_group(c);
#pragma unroll
                for (int r = 0; r < kGroup / kRun; ++r) {
                    const int c0 = c + kRun * r;
                    if (c0 >= n_splits) break;
                    const int hb = c0 >> 3;  // register holding these weights
                    float hreg = hl[0];
#pragma unroll
                    for (int j = 1; j < kHeld; ++j)
                        if (j == hb) hreg = hl[j];
                    add_run(r, hreg, c0 & 7);
                }
            }
        } else {
            // more chunks than registers hold: log-sums read twice
            for (int c = cg; c < n_splits; c += 8) M = fmaxf(M, __ldcg(lse_r + c * split_stride));
            M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 1));
            M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 2));
            M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 4));
            for (int c = cg; c < n_splits; c += 8) S += ex2_approx(__ldcg(lse_r + c * split_stride) - M);
            S += __shfl_xor_sync(0xffffffffu, S, 1);
            S += __shfl_xor_sync(0xffffffffu, S, 2);
            S += __shfl_xor_sync(0xffffffffu, S, 4);
            for (int c = 0; c < n_splits; c += kGroup) {
                load_group(c);
                float hw[kGroup / kRun];  // lane cg < kRun: weight of chunk c + kRun r + cg
#pragma unroll
                for (int r = 0; r < kGroup / kRun; ++r) {
                    const int ch = c + kRun * r + cg;
                    hw[r] = cg < kRun && ch < n_splits ? ex2_approx(__ldcg(lse_r + ch * split_stride) - M) : 0.0f;
                }
#pragma unroll
                for (int r = 0; r < kGroup / kRun; ++r) add_run(r, hw[r], 0);
            }
        }
        if (live) {
            const float inv = 1.0f / S;
            __nv_bfloat16* ob = p.o + r0 * D + col0;
            if constexpr (kCols >= 8) {
                uint4* orow = reinterpret_cast<uint4*>(ob);
#pragma unroll
                for (int x = 0; x < kCols / 8; ++x)
                    orow[x] = make_uint4(pack_bf16x2(acc[8 * x + 0] * inv, acc[8 * x + 1] * inv),
                                         pack_bf16x2(acc[8 * x + 2] * inv, acc[8 * x + 3] * inv),
                                         pack_bf16x2(acc[8 * x + 4] * inv, acc[8 * x + 5] * inv),
                                         pack_bf16x2(acc[8 * x + 6] * inv, acc[8 * x + 7] * inv));
            } else {
                *reinterpret_cast<uint2*>(ob) = make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv),
                                                           pack_bf16x2(acc[2] * inv, acc[3] * inv));
            }
            if (tw == 0 && cg == 0) p.lse[r0] = (M + log2f(S)) * kLn2;
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kDecWarps * 32, 1)
    attn_decode_sm103(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const DecParams p)
{
    using C = DecCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t ring = smem_u32(smem) + warp * C::kWarpRingBytes;
    uint8_t* ring_ptr = smem + warp * C::kWarpRingBytes;
    const uint32_t bar0 = smem_u32(smem) + C::kBarOff + warp * C::kStages * 8;
    auto full = [&](int s) { return bar0 + 8u * s; };

    if (threadIdx.x == 0) griddep_launch_dependents();  // the next launch may start its set-up
    if (lane == 0) {
        for (int s = 0; s < C::kStages; ++s) mbar_init(full(s), 1);
        fence_mbar_init();
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    // ---- the block's plan: every sequence's length and its number of chunks (an empty
    // sequence has one item, which writes O = 0 and lse = -inf); the sequences sorted by
    // chunk count, most first (the longest work is taken first, so the last items of the
    // launch are short ones); the chunk counts prefix-summed in that order, so that item t
    // maps to (sequence, chunk, head group) with no item past a sequence's end.
    int* sL = reinterpret_cast<int*>(smem + C::kPlanOff);  // [num_seqs] lengths
    int* sP = sL + kPlanMaxSeqs;                            // [num_seqs + 1] prefix, sorted order
    int* warp_tot = sP + kPlanMaxSeqs + 1;                  // [kDecWarps]
    volatile int* sDry = warp_tot + kDecWarps;              // a warp of this block found no item left
    int* sKey = warp_tot + kDecWarps + 1;                   // [pow2 >= num_seqs] sort keys
    {
        constexpr int kThreads = kDecWarps * 32;
        const int S = p.num_seqs;
        // key = (65535 - chunks) << 11 | sequence: ascending keys = most chunks first, ties
        // in sequence order (chunks <= 65535 and sequence < 2048 per launch)
        if (S <= kThreads) {
            // One sequence per thread: its place in the order and its prefix by counting the
            // smaller keys (the unsorted keys wait in the upper half of the key array).
            constexpr int kTmp = kPlanMaxSeqs - kThreads;
            const int i = threadIdx.x;
            int key = 0, n = 0;
            if (i < S) {
                const int L = clamp_len(p, p.seq_lens[i]);
                sL[i] = L;
                n = L > 0 ? (L + p.chunk - 1) / p.chunk : 1;
                key = ((65535 - n) << 11) | i;
                sKey[kTmp + i] = key;
            }
            __syncthreads();
            if (i < S) {
                int rank = 0, pre = 0;
                for (int j = 0; j < S; ++j) {
                    const int kj = sKey[kTmp + j];
                    if (kj < key) {
                        ++rank;
                        pre += 65535 - (kj >> 11);
                    }
                }
                sKey[rank] = key;
                sP[rank] = pre;
                if (rank == S - 1) sP[S] = pre + n;
            }
        } else {
            int N = 1;
            while (N < S) N <<= 1;
            for (int i = threadIdx.x; i < N; i += kThreads) {
                int key = INT_MAX;
                if (i < S) {
                    const int L = clamp_len(p, p.seq_lens[i]);
                    sL[i] = L;
                    const int n = L > 0 ? (L + p.chunk - 1) / p.chunk : 1;
                    key = ((65535 - n) << 11) | i;
                }
                sKey[i] = key;
            }
            __syncthreads();
            for (int k = 2; k <= N; k <<= 1) {  // bitonic sort in shared memory
                for (int jj = k >> 1; jj > 0; jj >>= 1) {
                    for (int i = threadIdx.x; i < N; i += kThreads) {
                        const int ixj = i ^ jj;
                        if (ixj > i) {
                            const int a = sKey[i], b = sKey[ixj];
                            if ((a > b) == ((i & k) == 0)) {
                                sKey[i] = b;
                                sKey[ixj] = a;
                            }
                        }
                    }
                    __syncthreads();
                }
            }
            // exclusive prefix of the chunk counts in sorted order (contiguous runs per thread)
            const int per = (S + kThreads - 1) / kThreads;
            const int b0 = threadIdx.x * per;
            const int b1 = min(S, b0 + per);
            int mine = 0;
            for (int i = b0; i < b1; ++i) mine += 65535 - (sKey[i] >> 11);
            int incl = mine;  // inclusive scan over the warp, then over the warps
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            if (lane == 31) warp_tot[warp] = incl;
            __syncthreads();
            int base = 0;
            for (int w = 0; w < warp; ++w) base += warp_tot[w];
            int run = base + incl - mine;
            for (int i = b0; i < b1; ++i) {
                sP[i] = run;
                run += 65535 - (sKey[i] >> 11);
            }
            if (threadIdx.x == kThreads - 1) sP[S] = base + incl;
        }
        if (threadIdx.x == 0) *sDry = 0;
        if (threadIdx.x < kDecWarps) reinterpret_cast<int*>(smem + C::kTeamOff + kDecWarps * 16)[threadIdx.x] = 0;
        __syncthreads();
    }

    const int g = lane >> 2;   // fragment row group
    const int tig = lane & 3;  // thread in group
    const float sl2 = p.scale_log2;
    // ldmatrix lane addressing inside a 128-byte-swizzled 16-row box
    const int mat = lane >> 3, rr = lane & 7;
    const int k_token = 8 * (mat >> 1) + rr, k_unit = mat & 1;
    const int v_token = 8 * (mat & 1) + rr, v_unit = mat >> 1;
    uint32_t uses = 0;  // sub-pages this warp has streamed (ring position)

    // Items in heaviest-first sequence order, then head group, then chunk: a sequence's
    // chunks are taken together, so its merge can start early. Each team's first item is its
    // own index (nothing to claim); later ones come from a device-wide counter.
    const int n_warps = static_cast<int>(gridDim.x) * kDecWarps;
    const long long n_items = static_cast<long long>(sP[p.num_seqs]) * p.HG;
    // Team size T: with at most half as many items as warps, T warps of a block share an
    // item (sub-pages dealt round-robin, partials combined in shared memory), so that a
    // small batch's cache reads spread over more warps. Every block derives the same T.
    int T = 1;
    while (T * 2 <= C::kMaxTeam && n_items * (T * 2) <= n_warps) T *= 2;
    const int team = warp / T;  // team within the block
    const int tw = warp % T;    // rank in the team = column slice of the merge
    const long long n_teams = static_cast<long long>(gridDim.x) * (kDecWarps / T);
    long long* sTeamT = reinterpret_cast<long long*>(smem + C::kTeamOff);           // [team][2]
    volatile int* sTeamAbort = reinterpret_cast<int*>(smem + C::kTeamOff + kDecWarps * 16);  // [team]
    float2* sML = reinterpret_cast<float2*>(smem + C::kTeamOff + kDecWarps * 20);   // [warp][row]
    auto team_sync = [&]() {
        asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(T * 32) : "memory");
    };
    bool first = true;
    bool waited = false;
    uint32_t iter = 0;  // items this team has taken (its claim slot parity)
    // Work written by the previous launch (outputs, this launch's workspace) is touched
    // only after it has completed; set-up and cache reads may overlap its tail.
    auto wait_prior = [&]() {
        if (!waited) {
            griddep_wait();
            waited = true;
        }
    };
    while (true) {
        // ---------------------------------------------------------------- next item
        long long t = 0;
        if (first) {
            t = static_cast<long long>(blockIdx.x) * (kDecWarps / T) + team;
            first = false;
        } else if (T == 1) {
            // nothing to claim when the first items covered everything, or once another
            // warp of this block has found the counter exhausted
            int dry = 0;
            if (lane == 0) dry = *sDry;
            dry = __shfl_sync(0xffffffffu, dry, 0);  // one decision for the whole warp
            if (n_items <= n_warps || dry) break;
            wait_prior();
            if (lane == 0) t = n_warps + static_cast<long long>(atomicAdd(p.work, 1ull));
            t = __shfl_sync(0xffffffffu, t, 0);
            if (t >= n_items && lane == 0) *sDry = 1;
        } else {
            if (n_items <= n_teams) break;  // the first items covered everything
            wait_prior();
            // the leader claims; the team reads the claim after the barrier (two slots by
            // parity, so a slot is rewritten only after every member has read it)
            if (tw == 0 && lane == 0) {
                long long c = n_items;
                if (!*sDry) {
                    c = n_teams + static_cast<long long>(atomicAdd(p.work, 1ull));
                    if (c >= n_items) *sDry = 1;
                }
                sTeamT[team * 2 + (iter & 1)] = c;
            }
            team_sync();
            t = sTeamT[team * 2 + (iter & 1)];
        }
        ++iter;
        if (t >= n_items) break;
        // in chunk units: sP[pos] <= qi < sP[pos + 1] (32-bit division when the items allow)
        const int qi = n_items <= INT_MAX ? static_cast<int>(t) / p.HG : static_cast<int>(t / p.HG);
        int pos = 0;                                 // place in the heaviest-first order
        {
            int lo = 0, hi = p.num_seqs - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (sP[mid] <= qi) lo = mid;
                else hi = mid - 1;
            }
            pos = lo;
        }
        const int seq = sKey[pos] & 2047;
        const int n_chunks = sP[pos + 1] - sP[pos];
        const int rem = static_cast<int>(t - static_cast<long long>(sP[pos]) * p.HG);
        const int hg = rem / n_chunks;
        const int split = rem - hg * n_chunks;
        const int L = sL[seq];
        const int hkv = p.n_hgroups == 1 ? hg : hg / p.n_hgroups;
        const int grp = hg - hkv * p.n_hgroups;
        const int hq0 = hkv * p.G + grp * kRowsPerItem;
        const int nvalid = min(kRowsPerItem, p.G - grp * kRowsPerItem);
        const size_t out_row0 = static_cast<size_t>(seq) * p.Hq + hq0;

        if (L == 0) {
            // an empty sequence: O = 0, lse = -inf (written by the team's first warp)
            wait_prior();
            if (tw == 0) {
                for (int idx = lane; idx < nvalid * D; idx += 32)
                    p.o[out_row0 * D + idx] = __float2bfloat16_rn(0.0f);
                if (lane < nvalid) p.lse[out_row0 + lane] = -INFINITY;
            }
            continue;
        }
        const int tok0 = split * p.chunk;
        const int tok1 = min(L, tok0 + p.chunk);
        const int n_sub = (tok1 - tok0 + kSub - 1) / kSub;
        const int lb0 = tok0 / p.block_size;
        const int n_lb = (tok1 - 1) / p.block_size - lb0 + 1;
        // this warp's sub-pages: tw, tw + T, tw + 2T, ... (none when n_sub <= tw)
        const int n_mine = tw < n_sub ? (n_sub - tw + T - 1) / T : 0;
        int phys = 0;
        if (lane < n_lb) {
            phys = p.block_table[static_cast<size_t>(seq) * p.max_blocks + lb0 + lane];
            if (phys < 0 || phys >= p.num_blocks) {
                report_error(p.err, kDevErrBounds);
                phys = 0;
            }
        }
        // Cache row of every sub-page of the item, one per lane (n_sub <= 32): the first
        // row of its 16 tokens in the [block][kv head][token] row space.
        int sub_row = 0;
        {
            const int tok = tok0 + min(lane, n_sub - 1) * kSub;
            const int lb = tok / p.block_size;
            const int ph = __shfl_sync(0xffffffffu, phys, lb - lb0);
            sub_row = (ph * p.Hkv + hkv) * p.block_size + (tok - lb * p.block_size);
        }
        // Issue the TMA copies of this warp's k-th sub-page (item sub-page tw + k T) into
        // its ring stage: one copy for K and one for V, each landing as kBoxes 16-row
        // boxes of 128 bytes.
        auto issue = [&](int k) {
            const int row = __shfl_sync(0xffffffffu, sub_row, tw + k * T);
            if (lane == 0) {
                const int s = static_cast<int>((uses + k) % C::kStages);
                const uint32_t dst = ring + s * C::kStageBytes;
                mbar_arrive_expect_tx(full(s), C::kStageBytes);
                tma_load_3d(dst, &tm_k, full(s), 0, row, 0);
                tma_load_3d(dst + C::kSubBytes, &tm_v, full(s), 0, row, 0);
            }
        };
        const int primed = min(C::kStages, n_mine);
        for (int k = 0; k < primed; ++k) issue(k);
        int issued = primed;
        wait_prior();
        // q as A fragments (rows = query heads of this kv head, zero past nvalid)
        uint32_t qa[D / 16][4];
        {
            const __nv_bfloat16* qb = p.q + out_row0 * D;
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

        bool ok = true;
        for (int k = 0; k < n_mine; ++k) {
            const int i = tw + k * T;  // sub-page of the item
            const int s = static_cast<int>((uses + k) % C::kStages);
            if (!mbar_wait(full(s), ((uses + k) / C::kStages) & 1, nullptr, p.err)) {
                ok = false;
                // never leave while a copy into this warp's ring is in flight
                for (int j = k + 1; j < issued; ++j)
                    mbar_wait(full(static_cast<int>((uses + j) % C::kStages)), ((uses + j) / C::kStages) & 1,
                              nullptr, p.err);
                break;
            }
            const uint32_t sK = ring + s * C::kStageBytes;
            const uint32_t sV = sK + C::kSubBytes;
            const int ntok = min(kSub, tok1 - (tok0 + i * kSub));
            if (ntok < kSub) {
                // Slots past the sequence end are never used: zero those V rows (they may
                // hold anything, NaN included) so that 0 * V stays 0 in the P V product.
                uint8_t* vrow = ring_ptr + s * C::kStageBytes + C::kSubBytes;
                const int units = (kSub - ntok) * 8;  // 16-byte units per box
                for (int x = 0; x < C::kBoxes; ++x)
                    for (int u = lane; u < units; u += 32)
                        reinterpret_cast<uint4*>(vrow + x * C::kBoxBytes + ntok * 128)[u] = make_uint4(0u, 0u, 0u, 0u);
                // these generic-proxy writes precede the stage's next TMA fill
                fence_proxy_async_smem();
                __syncwarp();
            }
            // ---- S = q K^T (16 heads x 16 tokens)
            // (even and odd k steps accumulate separately: four short chains, not two long)
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            float sd[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int U = 2 * kk + k_unit;
                const uint32_t addr = sK + (U >> 3) * C::kBoxBytes + k_token * 128 + (((U & 7) ^ rr) << 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(addr, b0, b1, b2, b3);
                mma_16816((kk & 1) ? sd[0] : sc[0], qa[kk], b0, b1);
                mma_16816((kk & 1) ? sd[1] : sc[1], qa[kk], b2, b3);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[nt][e] += sd[nt][e];
            if (ntok < kSub) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (8 * nt + 2 * tig + (e & 1) >= ntok) sc[nt][e] = -INFINITY;
            }
            // ---- online softmax per row (rows g: e = 0,1; rows g+8: e = 2,3)
            float mx[2];
#pragma unroll
            for (int h = 0; h < 2; ++h)
                mx[h] = fmaxf(fmaxf(sc[0][2 * h], sc[0][2 * h + 1]), fmaxf(sc[1][2 * h], sc[1][2 * h + 1]));
#pragma unroll
            for (int h = 0; h < 2; ++h) mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
#pragma unroll
            for (int h = 0; h < 2; ++h) mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
            bool grow[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float m_cand = mx[h] * sl2;
                grow[h] = m_cand > m[h] + kRescaleThreshold || (m[h] == -INFINITY && m_cand > -INFINITY);
                mx[h] = m_cand;
            }
            if (grow[0] || grow[1]) {
                // the running maximum moved by more than the threshold: rescale O and l
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float m_new = grow[h] ? fmaxf(m[h], mx[h]) : m[h];
                    const float alpha = !grow[h] ? 1.0f : (m[h] == -INFINITY) ? 0.0f : ex2_approx(m[h] - m_new);
                    m[h] = m_new;
                    l[h] *= alpha;
#pragma unroll
                    for (int nt = 0; nt < D / 8; ++nt) {
                        o[nt][2 * h] *= alpha;
                        o[nt][2 * h + 1] *= alpha;
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
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
            __syncwarp();
            if (k + C::kStages < n_mine) {
                // every read of the stage has returned (the P V products consumed them)
                issue(k + C::kStages);
                ++issued;
            }
        }
        uses += static_cast<uint32_t>(issued);
        if (T == 1 && !ok) break;  // a copy timed out (reported): leave through the exit count

        // ---------------------------------------------------------------- item result
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
            l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
        }
        const int n_splits = (L + p.chunk - 1) / p.chunk;
        // completion counter of this (sequence, head group) and column slice
        const size_t done_idx = (static_cast<size_t>(seq) * p.HG + hg) * C::kMaxTeam + tw;
        if (T > 1) {
            // ---- team combine: each warp leaves its unnormalised O (rows x D, padded rows)
            // in its own ring, idle now, and (m, l) per row; then warp tw combines columns
            // [tw D/T, (tw + 1) D/T) of the team's T partials.
            float* mine = reinterpret_cast<float*>(ring_ptr);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = g + 8 * h;
                if (row >= nvalid) continue;
#pragma unroll
                for (int nt = 0; nt < D / 8; ++nt)
                    *reinterpret_cast<float2*>(mine + row * C::kRowF + 8 * nt + 2 * tig) =
                        make_float2(o[nt][2 * h], o[nt][2 * h + 1]);
                if (tig == 0) sML[warp * kRowsPerItem + row] = make_float2(m[h], l[h]);
            }
            if (!ok && lane == 0) sTeamAbort[team] = 1;
            fence_proxy_async_smem();  // these writes precede the ring's next TMA fills
            team_sync();
            if (sTeamAbort[team]) break;  // a member's copy timed out (reported): leave together
            // lane r < nvalid: the weights 2^(m_w - M) of row r's members and 1 / L
            float wt[C::kMaxTeam];
            float inv_r = 0.0f;
            {
                const int r = lane < nvalid ? lane : 0;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < C::kMaxTeam; ++w)
                    if (w < T) M = fmaxf(M, sML[(team * T + w) * kRowsPerItem + r].x);
                float Ls = 0.0f;
#pragma unroll
                for (int w = 0; w < C::kMaxTeam; ++w) {
                    wt[w] = 0.0f;
                    if (w < T) {
                        const float2 ml = sML[(team * T + w) * kRowsPerItem + r];
                        wt[w] = ex2_approx(ml.x - M);  // 0 for a member with no sub-page
                        Ls += wt[w] * ml.y;
                    }
                }
                inv_r = 1.0f / Ls;
                if (lane < nvalid) {
                    if (n_splits == 1) {
                        if (tw == 0) p.lse[out_row0 + r] = (M + log2f(Ls)) * kLn2;
                    } else {
                        // every member writes the row's log-sum (the same value): each column
                        // slice's merge then reads one its own counter orders
                        p.part_lse[(static_cast<size_t>(split) * p.num_seqs + seq) * p.Hq + hq0 + r] = M + log2f(Ls);
                    }
                }
            }
            const int cpl = D / 32 / T;   // columns per lane: 1, 2 or 4
            const int c0 = tw * (D / T) + lane * cpl;
            for (int r = 0; r < nvalid; ++r) {
                float a[C::kMaxTeam];
#pragma unroll
                for (int w = 0; w < C::kMaxTeam; ++w) a[w] = __shfl_sync(0xffffffffu, wt[w], r);
                const float inv = __shfl_sync(0xffffffffu, inv_r, r);
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int w = 0; w < C::kMaxTeam; ++w) {
                    if (w >= T) break;
                    const float* src = reinterpret_cast<const float*>(smem + (team * T + w) * C::kWarpRingBytes) +
                                       r * C::kRowF + c0;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (j < cpl) acc[j] = fmaf(a[w], src[j], acc[j]);
                }
                if (n_splits == 1) {
                    __nv_bfloat16* orow = p.o + (out_row0 + r) * D + c0;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (j < cpl) orow[j] = __float2bfloat16_rn(acc[j] * inv);
                } else {
                    float* dst = p.part_o + ((static_cast<size_t>(split) * p.num_seqs + seq) * p.Hq + hq0 + r) * D + c0;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (j < cpl) dst[j] = acc[j] * inv;
                }
            }
            if (n_splits == 1) continue;
            __syncwarp();
            int last_t = 0;
            if (lane == 0) last_t = atom_add_acq_rel(p.done + done_idx, 1) == n_splits - 1;
            last_t = __shfl_sync(0xffffffffu, last_t, 0);
            if (!last_t) continue;
        }
        if (T == 1 && n_splits == 1) {
            // the whole sequence was this chunk: write O and lse directly
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = g + 8 * h;
                if (row >= nvalid) continue;
                const float inv = 1.0f / l[h];
                __nv_bfloat16* orow = p.o + (out_row0 + row) * D;
#pragma unroll
                for (int nt = 0; nt < D / 8; ++nt)
                    *reinterpret_cast<uint32_t*>(orow + 8 * nt + 2 * tig) =
                        pack_bf16x2(o[nt][2 * h] * inv, o[nt][2 * h + 1] * inv);
                if (tig == 0) p.lse[out_row0 + row] = (m[h] + log2f(l[h])) * kLn2;
            }
            continue;
        }
        if (T == 1) {
        // several chunks: write this one's normalised partial and log-sum
        const size_t part_row0 = (static_cast<size_t>(split) * p.num_seqs + seq) * p.Hq + hq0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = g + 8 * h;
            if (row >= nvalid) continue;
            const float inv = 1.0f / l[h];
            float* prow = p.part_o + (part_row0 + row) * D;
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt)
                *reinterpret_cast<float2*>(prow + 8 * nt + 2 * tig) = make_float2(o[nt][2 * h] * inv,
                                                                                 o[nt][2 * h + 1] * inv);
            if (tig == 0) p.part_lse[part_row0 + row] = m[h] + log2f(l[h]);
        }
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atom_add_acq_rel(p.done + done_idx, 1) == n_splits - 1;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (!last) continue;
        }
        // ---- this warp finished the last chunk of (seq, head group) for its column slice
        // (all D columns when T = 1): merge that slice of every partial (the warp barrier
        // orders every lane's loads after lane 0's acquiring count)
        __syncwarp();
        {
            const int vec = D / 32 / T;  // float4 per lane of the slice
            if constexpr (D >= 128) {
                if (vec == 4) merge_slice<D, 4>(p, seq, hq0, nvalid, n_splits, tw, lane);
            }
            if (vec == 2) merge_slice<D, 2>(p, seq, hq0, nvalid, n_splits, tw, lane);
            else if (vec == 1) merge_slice<D, 1>(p, seq, hq0, nvalid, n_splits, tw, lane);
        }
        if (lane == 0) p.done[done_idx] = 0;  // the last to touch it
    }
    // ---- leave. The next launch of a chain claims from the other counter, last used by
    // this launch's predecessor, which has completed once wait_prior returns: block 0
    // zeroes it, so the chain needs one memset and no block waits at its exit (the
    // completion counters were reset by the warps that merged). The wait also keeps this
    // launch from completing before its predecessor.
    wait_prior();
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.work_next = 0ull;
}


template <int D>
int launch_decode_d(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                    const int32_t* seq_lens, void* o, float* lse, int num_seqs, int Hq, int Hkv, int block_size,
                    int max_blocks, int num_blocks, float scale, void* workspace, const DecodePlan& plan,
                    cudaStream_t stream, unsigned* err, int flags, int* chain_slot)
{
    using C = DecCfg<D>;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    // the claim counters and the completion counters must start at zero; a launch leaves
    // its completion counters at zero and zeroes the next launch's claim counter, so a
    // chain of launches needs this only once
    if (!(flags & kDecodeCountersZeroed) && cudaMemsetAsync(ws, 0, plan.counters_bytes, stream) != cudaSuccess)
        return kErrCuda;
    // The cache as rows of D elements, each row seen as kBoxes 64-column pieces: dims
    // {column in piece, row, piece}, so that one copy brings a sub-page's 16 rows as kBoxes
    // boxes of 16 x 128 bytes (piece-major, each box swizzled on its own).
    CUtensorMap tk, tv;
    const uint64_t dims[3] = {64u, static_cast<uint64_t>(num_blocks) * Hkv * static_cast<uint64_t>(block_size),
                              static_cast<uint64_t>(C::kBoxes)};
    const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, 128u};
    const uint32_t box[3] = {64u, static_cast<uint32_t>(kSub), static_cast<uint32_t>(C::kBoxes)};
    int rc = encode_bf16_map(&tk, k_cache, 3, dims, strides, box);
    if (rc != kOk) return rc;
    rc = encode_bf16_map(&tv, v_cache, 3, dims, strides, box);
    if (rc != kOk) return rc;
    const int sms = sm_count();
    if (sms <= 0) return kErrCuda;
    if (cudaFuncSetAttribute(attn_decode_sm103<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
        cudaSuccess)
        return kErrCuda;
    DecParams prm;
    int slot = chain_slot ? (*chain_slot & 1) : 0;  // claim counters at ws and ws + 8
    prm.done = reinterpret_cast<int*>(ws + 16);
    prm.part_lse = reinterpret_cast<float*>(ws + plan.lse_offset);
    prm.part_o = reinterpret_cast<float*>(ws + plan.o_offset);
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.G = Hq / Hkv;
    prm.block_size = block_size;
    prm.max_blocks = max_blocks;
    prm.num_blocks = num_blocks;
    prm.chunk = plan.chunk;
    prm.n_hgroups = plan.n_hgroups;
    prm.HG = Hkv * plan.n_hgroups;
    prm.scale_log2 = scale * kLog2e;
    prm.err = err;
    // A block holds the lengths of at most kPlanMaxSeqs sequences: larger batches run as
    // consecutive launches over ranges of sequences (the later ones chained to the earlier).
    for (int s0 = 0; s0 < num_seqs; s0 += kPlanMaxSeqs) {
        const int S = num_seqs - s0 < kPlanMaxSeqs ? num_seqs - s0 : kPlanMaxSeqs;
        prm.q = static_cast<const __nv_bfloat16*>(q) + static_cast<size_t>(s0) * Hq * D;
        prm.block_table = block_table + static_cast<size_t>(s0) * max_blocks;
        prm.seq_lens = seq_lens + s0;
        prm.o = static_cast<__nv_bfloat16*>(o) + static_cast<size_t>(s0) * Hq * D;
        prm.lse = lse + static_cast<size_t>(s0) * Hq;
        prm.num_seqs = S;
        // at most one warp per item and team member beyond what the batch can hold
        const long long max_items =
            static_cast<long long>(plan.n_split_max > 0 ? plan.n_split_max : 1) * S * prm.HG * C::kMaxTeam;
        long long grid = sms;
        if (grid * kDecWarps > max_items) grid = (max_items + kDecWarps - 1) / kDecWarps;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(kDecWarps * 32);
        cfg.dynamicSmemBytes = C::kSmemBytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        const bool chained = (flags & kDecodeChained) || s0 > 0;
        cfg.attrs = chained ? attr : nullptr;
        cfg.numAttrs = chained ? 1 : 0;
        prm.work = reinterpret_cast<unsigned long long*>(ws + 8 * slot);
        prm.work_next = reinterpret_cast<unsigned long long*>(ws + 8 * (slot ^ 1));
        if (cudaLaunchKernelEx(&cfg, attn_decode_sm103<D>, tk, tv, prm) != cudaSuccess) return kErrLaunch;
        slot ^= 1;
    }
    if (chain_slot) *chain_slot = slot;
    return cudaGetLastError() == cudaSuccess ? kOk : kErrLaunch;
}

}  // namespace

bool decode_plan(int num_seqs, int Hq, int Hkv, int d, int block_size, int max_blocks_per_seq, DecodePlan* plan)
{
    if (num_seqs <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || block_size <= 0 || max_blocks_per_seq < 0) return false;
    if (Hq % Hkv != 0 || block_size % kSub != 0 || block_size > 256) return false;
    // Split length: a whole number of blocks, at most one block-table entry per lane.
    int chunk = kChunkTokens;
    if (chunk < block_size) chunk = block_size;
    chunk = (chunk / block_size) * block_size;
    if (chunk / block_size > kMaxChunkBlocks) chunk = kMaxChunkBlocks * block_size;
    const long long max_ctx = static_cast<long long>(max_blocks_per_seq) * block_size;
    const int G = Hq / Hkv;
    plan->n_hgroups = (G + kRowsPerItem - 1) / kRowsPerItem;
    const size_t hg = static_cast<size_t>(Hkv) * plan->n_hgroups;
    // A small batch (few, short sequences) gives fewer items than there are worker warps,
    // and a warp streams one item at a time: halve the chunk until the items cover the
    // warps, so that the cache reads spread over the whole GPU (more, smaller partials).
    long long n_split = (max_ctx + chunk - 1) / chunk;
    while (n_split * num_seqs * static_cast<long long>(hg) < kTargetItems && chunk / 2 >= kMinChunkTokens &&
           (chunk / 2) % block_size == 0) {
        chunk /= 2;
        n_split = (max_ctx + chunk - 1) / chunk;
    }
    if (n_split > 65535) return false;
    plan->chunk = chunk;
    plan->n_split_max = static_cast<int>(n_split);
    // one completion counter per (sequence, head group, merge column slice of a team)
    plan->counters_bytes = ((16 + 4 * static_cast<size_t>(num_seqs) * hg * kMaxTeamAll + 255) / 256) * 256;
    const size_t rows = static_cast<size_t>(n_split) * num_seqs * Hq;
    plan->lse_offset = plan->counters_bytes;
    plan->o_offset = plan->lse_offset + ((rows * 4 + 255) / 256) * 256;
    plan->bytes = plan->o_offset + rows * static_cast<size_t>(d) * 4;
    return true;
}

int launch_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                  const int32_t* seq_lens, void* o, float* lse, int num_seqs, int Hq, int Hkv, int d, int block_size,
                  int max_blocks_per_seq, int num_blocks, float scale, void* workspace, const DecodePlan& plan,
                  cudaStream_t stream, unsigned* err, int flags, int* chain_slot)
{
    if (d == 128)
        return launch_decode_d<128>(q, k_cache, v_cache, block_table, seq_lens, o, lse, num_seqs, Hq, Hkv, block_size,
                                    max_blocks_per_seq, num_blocks, scale, workspace, plan, stream, err, flags,
                                   chain_slot);
    if (d == 64)
        return launch_decode_d<64>(q, k_cache, v_cache, block_table, seq_lens, o, lse, num_seqs, Hq, Hkv, block_size,
                                   max_blocks_per_seq, num_blocks, scale, workspace, plan, stream, err, flags,
                                   chain_slot);
    return kErrUnsupported;
}

}  // namespace attn
