// fwd_kernel.cu -- prefill attention for sm_103a.
//
// One CTA owns two 128-row query tiles that read the same K/V stream (two query
// heads of one kv head when the GQA group is even, else two consecutive row tiles
// of one head). Roles, by warp:
//   warps 0-3  softmax for query tile 0 (thread = row = TMEM lane)
//   warps 4-7  softmax for query tile 1
//   warp  8    tcgen05 MMA issue (one thread) and TMEM allocation
//   warp  9    TMA producer (one thread): Q tiles, then the K/V ring
//
// Per key tile j and query tile t (pages: "Modern attention kernels", sections
// "Online softmax makes tiling exact" and "Kernel structure"; "Attention kernels",
// the FlashAttention-2/3 paragraphs on query-outer order, warp specialisation and
// asynchronous copies):
//   S_t = Q_t K_j^T           tcgen05.mma, bf16 x bf16 -> fp32 in TMEM (128 x 128)
//   softmax warps             m' = max(m, rowmax), p = 2^(s*scale*log2e - m'),
//                             l = alpha*l + sum p, P (bf16) written back over S_t
//   O_t = alpha*O_t + P_t V_j tcgen05.mma with P from TMEM, V from shared memory
// and after the last tile O/l (bf16) and lse = ln2 * (m + log2 l) are written.
// The running max is only moved when a row's max rises by more than 2^8 (lazy
// rescale); the result is unchanged because l and O always share the same max.
//
// Key tiles wholly outside the causal/window band are never visited; the tiles that
// cross the band edge or the end of the keys are masked per element.
//
// PAGED = true is prefill of several sequences against a paged KV cache (chunked
// prefill): sequence b has q_lens[b] new queries, the last of its kv_lens[b] cached
// tokens (bottom-right causal alignment), and its keys are read through the block table
// ("Modern attention kernels", "Paged attention changes addressing"). The producer
// copies each 128-key tile as min(block_size, 128)-row boxes from the cache's physical
// blocks and skips blocks past the sequence; in the last, partial tile it zeroes the V
// rows past the sequence (whatever the cache holds there) before P V may read them.
//
// MODE = sparse visits only the 128 x 128 score blocks a CSR block index lists
// ("Modern attention kernels", "Kernel structure": an arbitrary sparse mask needs an
// index of the blocks that exist; sparse attention visits the selected score blocks),
// intersected element by element with the causal / window masks. The block's two query
// tiles' lists are merged once into a shared-memory walk (key tile, tiles it is active
// for); the producer, the MMA thread and the softmax warps all step through that walk.
#include <climits>
#include <cmath>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int BM = 128;  // query rows per tile (= TMEM lanes)
constexpr int BN = 128;  // keys per tile
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr int kFwdThreads = 320;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: move the max only if it rises by > 256x
// FP8: the max moves once it rises by > 4x, and p is computed as 2^6 * 2^(s - m), so
// p <= 2^8 stays inside E4M3's range (448) while probabilities down to 2^-12 of the row's
// weight keep E4M3's normal (relative) precision. l carries the same 2^6.
constexpr float kFp8RescaleThreshold = 2.0f;
constexpr float kFp8PShift = 6.0f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kModeDense = 0, kModePaged = 1, kModeSparse = 2;
constexpr int kModeFp8 = 3;  // dense over E4M3 Q, K and transposed V (d = 128)
constexpr int kMaxWalk = 4096;                        // sparse: entries of the merged walk
constexpr int kWalkBytes = kMaxWalk * 4 + 16;         // entries + {count, last entry of tile 0 / 1}

template <int D, int EB = 2>  // EB: bytes per Q/K/V element (2: bf16, 1: E4M3)
struct FwdCfg {
    static constexpr int kBoxCols = 128 / EB;        // elements per 128-byte box row
    static constexpr int kBoxes = D * EB / 128;      // 128-byte-wide TMA boxes per row
    static constexpr int kBoxBytes = 128 * 128;      // 128 rows x 128 bytes
    static constexpr int kTileBytes = kBoxes * kBoxBytes;
    static constexpr int kStages = (kTileBytes == 2 * kBoxBytes) ? 4 : 8;  // K/V ring slots (K and V alternate)
    static constexpr int kQOff = 0;
    static constexpr int kRingOff = 2 * kTileBytes;
    static constexpr int kBarOff = kRingOff + kStages * kTileBytes;
    static constexpr int kNumBars = 1 + 2 * kStages + 8;
    static constexpr int kHolderOff = kBarOff + 8 * kNumBars;
    static constexpr int kAbortOff = kHolderOff + 4;
    static constexpr int kUsedBytes = kAbortOff + 4;
    static constexpr int kSmemBytes = kUsedBytes + 1024;  // slack for the 1024-byte alignment
    static constexpr uint32_t kTmemCols = 512;            // S0 | S1 | O0 | O1
    static constexpr uint32_t kOCol = 2 * BN;
    static_assert(kUsedBytes + 1024 + kWalkBytes <= 227 * 1024, "shared memory budget (with the sparse walk)");
    static_assert(kOCol + 2 * D <= kTmemCols, "TMEM budget");
};

struct FwdParams {
    __nv_bfloat16* o;
    float* lse;
    int B, Hq, Hkv, Nq, Nk, G;  // paged: B = sequences, Nq = max_q (row stride), Nk unused
    const int32_t* block_table;  // paged: [B][max_blocks] physical block of each logical block
    const int32_t* q_lens;       // paged: [B] new queries per sequence (device)
    const int32_t* kv_lens;      // paged: [B] cached tokens per sequence, new ones included (device)
    int max_blocks, block_size, bs_log2, num_blocks;
    const int32_t* row_ptr;      // sparse: [ceil(Nq / 128) + 1] CSR row offsets (device)
    const int32_t* col_idx;      // sparse: listed key blocks, ascending per query block (device)
    float scale_log2;  // scale * log2(e)
    int causal, window;
    int pair_heads;    // 1: tiles are query heads (2u, 2u+1) at one row tile; 0: row tiles (2r, 2r+1);
                       // 2: one tile per block (row tile r of head u), for grids smaller than the GPU
    int n_row_units;   // row units per (batch, head unit)
    int n_hunits;      // head units per batch entry
    int next_stride;   // dense / sparse: units between a block and the one that will take its SM
    float out_scale;   // multiplies O (FP8: V's scale; else 1)
    unsigned* err;
};

struct TileWork {
    int head;   // query head
    int row0;   // first query row
    int rows;   // valid rows in the tile (0: no tile)
    int kv_lo;  // first key tile visited
    int kv_hi;  // one past the last key tile visited
};

// Key tiles a query tile must visit: causal keeps keys j <= i + (Nk - Nq); a window
// w >= 0 also needs j >= i + (Nk - Nq) - w.
__device__ __forceinline__ TileWork make_tile(const FwdParams& p, int head, int row0, int nq, int nk)
{
    TileWork t{head, row0, 0, 0, 0};
    int rows = nq - row0;
    if (rows > BM) rows = BM;
    if (rows <= 0) return t;
    t.rows = rows;
    const long long delta = static_cast<long long>(nk) - nq;
    long long key_hi = nk;
    if (p.causal) {
        const long long h = static_cast<long long>(row0) + rows + delta;
        if (h < key_hi) key_hi = h;
    }
    long long key_lo = 0;
    if (p.window >= 0) {
        const long long l = static_cast<long long>(row0) + delta - p.window;
        if (l > key_lo) key_lo = l;
    }
    if (key_hi > key_lo) {
        t.kv_lo = static_cast<int>(key_lo / BN);
        t.kv_hi = static_cast<int>((key_hi + BN - 1) / BN);
    }
    return t;
}

// True when every key of tile j is allowed for every valid row of the query tile.
__device__ __forceinline__ bool tile_unmasked(const FwdParams& p, const TileWork& t, int j, int nq, int nk)
{
    const long long k0 = static_cast<long long>(j) * BN, k1 = k0 + BN;
    const long long delta = static_cast<long long>(nk) - nq;
    if (k1 > nk) return false;
    if (p.causal && k1 - 1 > t.row0 + delta) return false;
    if (p.window >= 0 && k0 < static_cast<long long>(t.row0) + t.rows - 1 + delta - p.window) return false;
    return true;
}

__device__ __forceinline__ bool tile_active(const TileWork& t, int j)
{
    return t.rows > 0 && t.kv_lo <= j && j < t.kv_hi;
}

template <int D, int MODE>
__global__ void __launch_bounds__(kFwdThreads, 1)
    attn_fwd_sm103(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const FwdParams p)
{
    constexpr bool FP8 = MODE == kModeFp8;
    using C = FwdCfg<D, FP8 ? 1 : 2>;
    constexpr bool PAGED = MODE == kModePaged;
    constexpr bool SPARSE = MODE == kModeSparse;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work unit. Dense: heaviest row units first, which balances the causal triangle.
    // Paged: sequence outer, then kv head, then row units (heaviest first) and the head
    // units of that kv head, so that the blocks running together read the same K/V pages
    // and the cache stays in L2 (sequences have different lengths; their order is kept).
    const int unit = blockIdx.x;
    int ru, b, hu;
    if constexpr (PAGED) {
        const int per_seq = p.n_hunits * p.n_row_units;
        const int hpg = p.n_hunits / p.Hkv;  // head units per kv head
        b = unit / per_seq;
        const int r = unit % per_seq;
        const int grp = r / (hpg * p.n_row_units);
        const int r2 = r % (hpg * p.n_row_units);
        ru = p.n_row_units - 1 - r2 / hpg;
        hu = grp * hpg + r2 % hpg;
    } else {
        const int n_bh = p.B * p.n_hunits;
        ru = p.n_row_units - 1 - unit / n_bh;
        const int bh = unit % n_bh;
        b = bh / p.n_hunits;
        hu = bh % p.n_hunits;
    }
    // rows and keys of this (batch entry | sequence)
    int nq = p.Nq, nk = p.Nk;
    if constexpr (PAGED) {
        nq = p.q_lens[b];
        nk = p.kv_lens[b];
        if (nq < 0 || nq > p.Nq || nk < nq || static_cast<long long>(nk) > static_cast<long long>(p.max_blocks) * p.block_size) {
            if (threadIdx.x == 0) report_error(p.err, kDevErrBounds);
            nq = 0;
            nk = 0;
        }
    }
    TileWork tw[2];
    if (p.pair_heads == 2) {
        tw[0] = make_tile(p, hu, ru * BM, nq, nk);
        tw[1] = TileWork{hu, 0, 0, 0, 0};
    } else if (p.pair_heads) {
        tw[0] = make_tile(p, 2 * hu, ru * BM, nq, nk);
        tw[1] = make_tile(p, 2 * hu + 1, ru * BM, nq, nk);
    } else {
        tw[0] = make_tile(p, hu, 2 * ru * BM, nq, nk);
        tw[1] = make_tile(p, hu, (2 * ru + 1) * BM, nq, nk);
    }
    const int hkv = tw[0].head / p.G;
    bool act[2] = {tw[0].rows > 0 && tw[0].kv_lo < tw[0].kv_hi, tw[1].rows > 0 && tw[1].kv_lo < tw[1].kv_hi};
    int lo = INT_MAX, hi = 0;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        if (act[t]) {
            lo = min(lo, tw[t].kv_lo);
            hi = max(hi, tw[t].kv_hi);
        }
    }
    bool has_work = lo < hi;

    // ---- barriers
    const uint32_t bar0 = sb + C::kBarOff;
    const uint32_t bar_q = bar0;
    auto kv_full = [&](int s) { return bar0 + 8u * (1 + s); };
    auto kv_empty = [&](int s) { return bar0 + 8u * (1 + C::kStages + s); };
    // Copy n of the ring (K and V alternate: n even K_j, odd V_j) may start once copy
    // n - kStages has been released. bf16: a V tile is released by the commit that releases
    // the K tile after it, issued once every product of that key step was issued (so after
    // the V tile's P V products): one commit fewer per key step. FP8, whose steps are
    // shorter, releases every tile on its own (the later V releases measured slower there).
    constexpr bool kVByK = !FP8;
    auto slot_free = [&](int n, int kind) { return kVByK && kind ? kv_empty((n + 1) % C::kStages) : kv_empty(n % C::kStages); };
    auto slot_free_parity = [&](int n, int kind) {
        return static_cast<uint32_t>((kVByK && kind ? (n + 1 - C::kStages) / C::kStages : n / C::kStages - 1) & 1);
    };
    auto s_full = [&](int t) { return bar0 + 8u * (1 + 2 * C::kStages + t); };
    auto p_full = [&](int t) { return bar0 + 8u * (3 + 2 * C::kStages + t); };
    auto o_done = [&](int t) { return bar0 + 8u * (5 + 2 * C::kStages + t); };
    const uint32_t bar_drain = bar0 + 8u * (7 + 2 * C::kStages);
    const uint32_t bar_vtail = bar0 + 8u * (8 + 2 * C::kStages);  // paged: the partial tile's V rows zeroed
    // paged: the key tile that holds the sequence's last key when it is partial, else -1
    const int tail_j = (PAGED && nk % BN != 0) ? nk / BN : -1;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kHolderOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbortOff);

    if (threadIdx.x == 0) {
        mbar_init(bar_q, 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(kv_full(s), 1);
            mbar_init(kv_empty(s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(s_full(t), 1);
            mbar_init(p_full(t), 128);
            mbar_init(o_done(t), 1);
        }
        mbar_init(bar_drain, 1);
        mbar_init(bar_vtail, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    // ---- dense and sparse: the Q tiles (and, dense, the first K/V tiles) are requested as
    // soon as the barriers exist, ahead of the TMEM allocation and (sparse) the walk: their
    // latency is the longest part of a short block's start. Sparse: both tiles' Q is loaded
    // even if the walk later finds a tile with no listed block. Paged: the producer loads Q
    // (measured: issuing it here does not help there).
    auto issue_q = [&]() {
        uint32_t qbytes = 0;
#pragma unroll
        for (int t = 0; t < 2; ++t)
            if (act[t]) qbytes += C::kTileBytes;
        mbar_arrive_expect_tx(bar_q, qbytes);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            if (!act[t]) continue;
#pragma unroll
            for (int x = 0; x < C::kBoxes; ++x)
                tma_load_3d(sb + C::kQOff + t * C::kTileBytes + x * C::kBoxBytes, &tm_q, bar_q, C::kBoxCols * x,
                            tw[t].row0, b * p.Hq + tw[t].head);
        }
    };
    // One K (kind 0) or V (kind 1) tile of key tile j into ring slot s. FP8 V is stored
    // transposed ([d][Nk] per head): its tile is the 128 keys of every d row, one box.
    auto load_kv = [&](int kind, int s, int j) {
        const uint32_t dst = sb + C::kRingOff + s * C::kTileBytes;
        if (FP8 && kind == 1) {
            tma_load_3d(dst, &tm_v, kv_full(s), j * BN, 0, b * p.Hkv + hkv);
        } else {
            const CUtensorMap* map = kind == 0 ? &tm_k : &tm_v;
#pragma unroll
            for (int x = 0; x < C::kBoxes; ++x)
                tma_load_3d(dst + x * C::kBoxBytes, map, kv_full(s), C::kBoxCols * x, j * BN, b * p.Hkv + hkv);
        }
    };
    const bool q_early = has_work && !PAGED;
    const int n_pre = ((MODE == kModeDense || FP8) && has_work) ? min(C::kStages, 2 * (hi - lo)) : 0;  // even
    if (threadIdx.x == 0 && q_early) {
        fence_proxy_async_smem();
        issue_q();
        for (int i = 0; i < n_pre; ++i) {  // first fill of each ring slot: K_lo, V_lo, K_lo+1, ...
            mbar_arrive_expect_tx(kv_full(i), C::kTileBytes);
            load_kv(i & 1, i, lo + i / 2);
        }
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == kLoadWarp && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    // ---- sparse: merge the two query tiles' listed key blocks into the walk
    uint32_t* walk = reinterpret_cast<uint32_t*>(smem + C::kUsedBytes);  // sparse only (kWalkBytes)
    if constexpr (SPARSE) {
        // the lists, copied by every thread into the (still unused) K/V ring
        int32_t* raw = reinterpret_cast<int32_t*>(smem + C::kRingOff);
        int beg[2] = {0, 0}, len[2] = {0, 0};
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            if (!act[t]) continue;
            const int qb = tw[t].row0 / BM;
            beg[t] = p.row_ptr[qb];
            len[t] = p.row_ptr[qb + 1] - beg[t];
            if (len[t] < 0 || len[t] > kMaxWalk / 2) {
                if (threadIdx.x == 0) report_error(p.err, kDevErrBounds);
                len[t] = 0;
            }
        }
        for (int e = threadIdx.x; e < len[0] + len[1]; e += kFwdThreads)
            raw[e] = e < len[0] ? p.col_idx[beg[0] + e] : p.col_idx[beg[1] + e - len[0]];
        __syncthreads();
        if (threadIdx.x == 0) {
            // entry = key tile | bit 30 + t when tile t lists it inside its causal / window
            // range; listed tiles must ascend strictly and lie below ceil(Nk / 128)
            const int n_kblk = (nk + BN - 1) / BN;
            int i0 = 0, i1 = 0, n = 0, prev = -1, last0 = -1, last1 = -1;
            while (i0 < len[0] || i1 < len[1]) {
                const int c0 = i0 < len[0] ? raw[i0] : INT_MAX;
                const int c1 = i1 < len[1] ? raw[len[0] + i1] : INT_MAX;
                const int j = c0 < c1 ? c0 : c1;
                uint32_t m = 0;
                if (c0 == j) {
                    ++i0;
                    if (tw[0].kv_lo <= j && j < tw[0].kv_hi) m |= 1u;
                }
                if (c1 == j) {
                    ++i1;
                    if (tw[1].kv_lo <= j && j < tw[1].kv_hi) m |= 2u;
                }
                if (j < 0 || j >= n_kblk || j <= prev) {
                    report_error(p.err, kDevErrBounds);
                    continue;
                }
                prev = j;
                if (m == 0) continue;
                walk[4 + n] = static_cast<uint32_t>(j) | (m << 30);
                if (m & 1u) last0 = n;
                if (m & 2u) last1 = n;
                ++n;
            }
            walk[0] = static_cast<uint32_t>(n);
            walk[1] = static_cast<uint32_t>(last0);
            walk[2] = static_cast<uint32_t>(last1);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    // ---- key-tile walk: entry e -> key tile walk_j(e), active for query tile t when
    // walk_act(t, e); the last entry of tile t is last_e[t]. Dense and paged: the range
    // [lo, hi) with each tile's own band.
    int n_walk = has_work ? hi - lo : 0;
    int last_e[2] = {tw[0].kv_hi - 1 - lo, tw[1].kv_hi - 1 - lo};
    if constexpr (SPARSE) {
        n_walk = static_cast<int>(walk[0]);
        last_e[0] = static_cast<int>(walk[1]);
        last_e[1] = static_cast<int>(walk[2]);
        act[0] = last_e[0] >= 0;
        act[1] = last_e[1] >= 0;
        has_work = n_walk > 0;
    }
    auto walk_j = [&](int e) -> int {
        if constexpr (SPARSE) return static_cast<int>(walk[4 + e] & 0x3FFFFFFFu);
        else return lo + e;
    };
    auto walk_act = [&](int t, int e) -> bool {
        if constexpr (SPARSE) return ((walk[4 + e] >> (30 + t)) & 1u) != 0u;
        else return tile_active(t ? tw[1] : tw[0], lo + e);
    };

    const uint32_t sQ = sb + C::kQOff;
    const uint32_t sRing = sb + C::kRingOff;

    if (warp == kLoadWarp) {
        // ================================================================ producer
        if (PAGED && has_work && lane == 0) issue_q();
        int n = n_pre;  // K/V copies issued (K and V alternate in the ring)
        if constexpr (!PAGED) {
            if (has_work && lane == 0) {
                bool ok = true;
                for (int e = n_pre / 2; e < n_walk && ok; ++e) {
                    const int j = walk_j(e);
#pragma unroll
                    for (int kind = 0; kind < 2; ++kind) {
                        const int s = n % C::kStages;
                        if (n >= C::kStages &&
                            !mbar_wait(slot_free(n, kind), slot_free_parity(n, kind), abort_flag, p.err)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(kv_full(s), C::kTileBytes);
                        load_kv(kind, s, j);
                        ++n;
                    }
                }
                // The block that will run on this SM after this one is about next_stride
                // units further on: bring its Q tiles and first K/V tile into L2 now, so that
                // its start does not wait on DRAM.
                const long long un = static_cast<long long>(blockIdx.x) + p.next_stride;
                if (p.next_stride > 0 && un < gridDim.x) {
                    const int u2 = static_cast<int>(un);
                    const int n_bh = p.B * p.n_hunits;
                    const int ru2 = p.n_row_units - 1 - u2 / n_bh;
                    const int bh2 = u2 % n_bh;
                    const int b2 = bh2 / p.n_hunits, hu2 = bh2 % p.n_hunits;
                    TileWork t2[2];
                    if (p.pair_heads == 2) {
                        t2[0] = make_tile(p, hu2, ru2 * BM, p.Nq, p.Nk);
                        t2[1] = TileWork{hu2, 0, 0, 0, 0};
                    } else if (p.pair_heads) {
                        t2[0] = make_tile(p, 2 * hu2, ru2 * BM, p.Nq, p.Nk);
                        t2[1] = make_tile(p, 2 * hu2 + 1, ru2 * BM, p.Nq, p.Nk);
                    } else {
                        t2[0] = make_tile(p, hu2, 2 * ru2 * BM, p.Nq, p.Nk);
                        t2[1] = make_tile(p, hu2, (2 * ru2 + 1) * BM, p.Nq, p.Nk);
                    }
                    int lo2 = INT_MAX;
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        if (t2[t].rows <= 0) continue;
#pragma unroll
                        for (int x = 0; x < C::kBoxes; ++x)
                            tma_prefetch_l2_3d(&tm_q, C::kBoxCols * x, t2[t].row0, b2 * p.Hq + t2[t].head);
                        if (t2[t].kv_lo < t2[t].kv_hi) lo2 = min(lo2, t2[t].kv_lo);
                    }
                    if (!SPARSE && lo2 != INT_MAX && p.Nk > 0) {
                        const int hkv2 = t2[0].head / p.G;
#pragma unroll
                        for (int x = 0; x < C::kBoxes; ++x) {
                            tma_prefetch_l2_3d(&tm_k, C::kBoxCols * x, lo2 * BN, b2 * p.Hkv + hkv2);
                            if (FP8) tma_prefetch_l2_3d(&tm_v, lo2 * BN, 0, b2 * p.Hkv + hkv2);
                            else tma_prefetch_l2_3d(&tm_v, C::kBoxCols * x, lo2 * BN, b2 * p.Hkv + hkv2);
                        }
                    }
                }
            }
        } else if (has_work) {
            // Paged: the whole warp. A 128-key tile is `subs` sub-blocks of min(block_size,
            // 128) rows; lane (u, x) = (lane / kBoxes, lane % kBoxes) copies sub-block u's
            // column box x, reading its block-table entry one tile ahead. Sub-blocks past the
            // sequence are not copied.
            const int sub_rows = p.block_size < BN ? p.block_size : BN;
            const int subs = BN / sub_rows;
            const int my_u = lane / C::kBoxes, my_x = lane % C::kBoxes;
            const bool mine = my_u < subs;
            auto entry = [&](int jt) -> int {
                const int key = jt * BN + my_u * sub_rows;
                return (mine && key < nk) ? __ldg(p.block_table + static_cast<long long>(b) * p.max_blocks +
                                                  (key >> p.bs_log2))
                                          : 0;
            };
            int ent_next = entry(walk_j(0));
            bool ok = true;
            for (int e = 0; e < n_walk && ok; ++e) {
                const int j = walk_j(e);
                const int ent = ent_next;
                if (e + 1 < n_walk) ent_next = entry(walk_j(e + 1));
                const int key = j * BN + my_u * sub_rows;
                const bool copy = mine && key < nk;
                int row = 0;
                if (copy) {
                    int phys = ent;
                    if (phys < 0 || phys >= p.num_blocks) {
                        report_error(p.err, kDevErrBounds);
                        phys = 0;
                    }
                    row = (phys * p.Hkv + hkv) * p.block_size + (key & (p.block_size - 1));
                }
                const int valid = min(BN, nk - j * BN);  // keys of this tile inside the sequence
                const int n_sub = (valid + sub_rows - 1) / sub_rows;
#pragma unroll
                for (int kind = 0; kind < 2; ++kind) {
                    const int s = n % C::kStages;
                    bool w = true;
                    if (lane == 0) {
                        if (n >= C::kStages) w = mbar_wait(slot_free(n, kind), slot_free_parity(n, kind), abort_flag, p.err);
                        if (w)
                            mbar_arrive_expect_tx(kv_full(s), static_cast<uint32_t>(n_sub * sub_rows * 128 * C::kBoxes));
                    }
                    if (!__shfl_sync(0xffffffffu, w, 0)) {  // (also orders the copies after expect_tx)
                        ok = false;
                        break;
                    }
                    const uint32_t dst = sRing + s * C::kTileBytes;
                    if (copy)
                        tma_load_2d(dst + my_x * C::kBoxBytes + my_u * sub_rows * 128, kind == 0 ? &tm_k : &tm_v,
                                    kv_full(s), 64 * my_x, row);
                    ++n;
                    if (kind == 1 && j == tail_j) {
                        // V of the partial tile: once it has landed, zero the rows past the
                        // sequence (stale or unwritten cache slots) so that P V never meets a
                        // NaN under a zero weight; then hand the tile to the MMA thread
                        bool f = true;
                        if (lane == 0) f = mbar_wait(kv_full(s), ((n - 1) / C::kStages) & 1, abort_flag, p.err);
                        if (!__shfl_sync(0xffffffffu, f, 0)) {
                            ok = false;
                            break;
                        }
                        for (int r = valid + lane; r < BN; r += 32)
#pragma unroll
                            for (int x = 0; x < C::kBoxes; ++x)
#pragma unroll
                                for (int c = 0; c < 8; ++c)
                                    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};"
                                                 ::"r"(dst + x * C::kBoxBytes + r * 128 + 16 * c), "r"(0u)
                                                 : "memory");
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar_vtail);
                    }
                }
            }
        }
        if ((has_work || q_early) && lane == 0) {
            // Never leave while a copy into this block's shared memory is in flight.
            mbar_wait(bar_q, 0, nullptr, p.err);
            for (int s = 0; s < C::kStages; ++s) {
                const int fills = n / C::kStages + (s < n % C::kStages ? 1 : 0);
                if (fills > 0) mbar_wait(kv_full(s), (fills - 1) & 1, nullptr, p.err);
            }
        }
    } else if (warp == kMmaWarp) {
        // ================================================================ MMA issue
        if (lane == 0 && has_work) {
            constexpr uint32_t idesc_qk = FP8 ? idesc_e4m3_f32(BM, BN) : idesc_bf16_f32(BM, BN, false, false);
            constexpr uint32_t idesc_pv = FP8 ? idesc_e4m3_f32(BM, D) : idesc_bf16_f32(BM, D, false, true);
            // S_t = Q_t K^T: both operands K-major; a 16-wide k step is 32 bytes inside a
            // 128-byte swizzle row, and every 64 columns start a new box.
            // Descriptors are built once; another k step, slot or tile only adds its byte
            // offset / 16 to the start-address field (every address stays below 256 KB).
            const uint64_t qdesc0 = smem_desc_sw128(sQ, 16, 1024);
            const uint64_t kdesc0 = smem_desc_sw128(sRing, 16, 1024);
            // bf16 V is MN-major (d contiguous); FP8 V arrives transposed, K-major like K.
            const uint64_t vdesc0 = FP8 ? smem_desc_sw128(sRing, 16, 1024) : smem_desc_sw128(sRing, C::kBoxBytes, 1024);
            auto issue_qk = [&](int t, int slot) {
                const uint32_t d_tmem = tmem + static_cast<uint32_t>(t * BN);
                const uint64_t qd = qdesc0 + static_cast<uint64_t>((t * C::kTileBytes) >> 4);
                const uint64_t kd = kdesc0 + static_cast<uint64_t>((slot * C::kTileBytes) >> 4);
                if constexpr (FP8) {
                    // 32 E4M3 elements (32 bytes) per step, all inside the one 128-byte row
#pragma unroll
                    for (int kk = 0; kk < D / 32; ++kk)
                        mma_ss_f8(d_tmem, qd + 2 * kk, kd + 2 * kk, idesc_qk, kk > 0 ? 1u : 0u);
                } else {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t off = static_cast<uint64_t>(((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4);
                        mma_ss(d_tmem, qd + off, kd + off, idesc_qk, kk > 0 ? 1u : 0u);
                    }
                }
            };
            // O_t (+)= P_t V: P from TMEM (8 columns = 16 bf16 keys per step); V is
            // MN-major in shared memory: 16 keys = 2048 bytes per step, the two
            // 64-column halves of d are one box (kBoxBytes) apart.
            auto issue_pv = [&](int t, int slot, bool accumulate) {
                const uint32_t d_tmem = tmem + C::kOCol + static_cast<uint32_t>(t * D);
                const uint32_t a_tmem = tmem + static_cast<uint32_t>(t * BN);
                const uint64_t vd = vdesc0 + static_cast<uint64_t>((slot * C::kTileBytes) >> 4);
                if constexpr (FP8) {
                    // P as E4M3 in TMEM: 32 keys = 8 columns per step; V^T K-major: +32 bytes
#pragma unroll
                    for (int kk = 0; kk < BN / 32; ++kk)
                        mma_ts_f8(d_tmem, a_tmem + kk * 8, vd + static_cast<uint64_t>(2 * kk), idesc_pv,
                                  (accumulate || kk > 0) ? 1u : 0u);
                } else {
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        mma_ts(d_tmem, a_tmem + kk * 8, vd + static_cast<uint64_t>(kk * 128), idesc_pv,
                               (accumulate || kk > 0) ? 1u : 0u);
                }
            };

            bool ok = mbar_wait(bar_q, 0, abort_flag, p.err);
            tc_fence_after();
            int n = 0;
            uint32_t pphase[2] = {0u, 0u};
            bool first_pv[2] = {true, true};
            if (ok) {
                const int ks = n % C::kStages;
                ok = mbar_wait(kv_full(ks), (n / C::kStages) & 1, abort_flag, p.err);
                tc_fence_after();
                ++n;
                if (ok) {
#pragma unroll
                    for (int t = 0; t < 2; ++t)
                        if (walk_act(t, 0)) {
                            issue_qk(t, ks);
                            tc_commit(s_full(t));
                        }
                    tc_commit(kv_empty(ks));
                }
            }
            for (int e = 0; e < n_walk && ok; ++e) {
                const int j = walk_j(e);
                const int vs = n % C::kStages;
                if (!mbar_wait(kv_full(vs), (n / C::kStages) & 1, abort_flag, p.err)) break;
                // paged: the partial tile's V is usable once its tail rows are zeroed
                if (PAGED && j == tail_j && !mbar_wait(bar_vtail, 0, abort_flag, p.err)) break;
                tc_fence_after();
                ++n;
                const bool has_next = e + 1 < n_walk;
                const int ks = n % C::kStages;
                // tile 0: O0 += P0 V_j, then S0 for the next key tile
                if (walk_act(0, e)) {
                    if (!mbar_wait(p_full(0), pphase[0], abort_flag, p.err)) break;
                    pphase[0] ^= 1u;
                    tc_fence_after();
                    issue_pv(0, vs, !first_pv[0]);
                    first_pv[0] = false;
                    if (e == last_e[0]) tc_commit(o_done(0));
                }
                if (has_next) {
                    if (!mbar_wait(kv_full(ks), (n / C::kStages) & 1, abort_flag, p.err)) break;
                    tc_fence_after();
                    ++n;
                    if (walk_act(0, e + 1)) {
                        issue_qk(0, ks);
                        tc_commit(s_full(0));
                    }
                }
                // tile 1: O1 += P1 V_j, then S1 for the next key tile
                if (walk_act(1, e)) {
                    if (!mbar_wait(p_full(1), pphase[1], abort_flag, p.err)) break;
                    pphase[1] ^= 1u;
                    tc_fence_after();
                    issue_pv(1, vs, !first_pv[1]);
                    first_pv[1] = false;
                    if (e == last_e[1]) tc_commit(o_done(1));
                }
                if constexpr (!kVByK) tc_commit(kv_empty(vs));
                if (has_next) {
                    if (walk_act(1, e + 1)) {
                        issue_qk(1, ks);
                        tc_commit(s_full(1));
                    }
                    tc_commit(kv_empty(ks));
                }
            }
            // Never release TMEM while an MMA may still be running.
            tc_commit(bar_drain);
            mbar_wait(bar_drain, 0, nullptr, p.err);
        }
    } else {
        // ================================================================ softmax (warps 0-7)
        const int t = warp >> 2;
        const int quarter = warp & 3;
        const TileWork T = t ? tw[1] : tw[0];
        const int r = quarter * 32 + lane;  // row in the tile = TMEM lane
        const int row = T.row0 + r;
        const uint32_t lane_sel = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t s_tmem = tmem + lane_sel + static_cast<uint32_t>(t * BN);
        const uint32_t o_tmem = tmem + lane_sel + C::kOCol + static_cast<uint32_t>(t * D);
        const float sl2 = p.scale_log2;
        float m = -INFINITY;  // running max, scaled log2 units
        float l = 0.0f;       // running sum
        int n_act = 0;
        bool ok = true;
        const bool tile_has = t ? act[1] : act[0];
        if (tile_has) {
            const long long diag = static_cast<long long>(row) + (static_cast<long long>(nk) - nq);
            long long key_max = static_cast<long long>(nk) - 1;
            if (p.causal && diag < key_max) key_max = diag;
            const long long key_min = p.window >= 0 ? diag - p.window : LLONG_MIN / 4;
            for (int e = 0; e < n_walk; ++e) {
                bool mine;  // (warp-uniform)
                if constexpr (SPARSE) mine = ((walk[4 + e] >> (30 + t)) & 1u) != 0u;
                else mine = tile_active(T, lo + e);
                if (!mine) continue;
                const int j = walk_j(e);
                if (!mbar_wait(s_full(t), n_act & 1, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t sr[BN];
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) tmem_ld32(s_tmem + 32 * c, sr + 32 * c);
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) tmem_ld_wait_dep32(sr + 32 * c);
                float s[BN];
#pragma unroll
                for (int c = 0; c < BN; ++c) s[c] = __uint_as_float(sr[c]);
                if (!tile_unmasked(p, T, j, nq, nk)) {
                    const long long kbase = static_cast<long long>(j) * BN;
                    long long hi_rel = key_max - kbase;
                    long long lo_rel = key_min - kbase;
                    const int hi_c = hi_rel < -1 ? -1 : (hi_rel > BN ? BN : static_cast<int>(hi_rel));
                    const int lo_c = lo_rel < 0 ? 0 : (lo_rel > BN + 1 ? BN + 1 : static_cast<int>(lo_rel));
#pragma unroll
                    for (int c = 0; c < BN; ++c)
                        if (c > hi_c || c < lo_c) s[c] = -INFINITY;
                }
                float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
                for (int c = 0; c < BN; c += 8) {
                    mx0 = fmax3(mx0, s[c], s[c + 1]);
                    mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
                    mx2 = fmax3(mx2, s[c + 4], s[c + 5]);
                    mx3 = fmax3(mx3, s[c + 6], s[c + 7]);
                }
                const float m_cand = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
                const bool need = m_cand > m + (FP8 ? kFp8RescaleThreshold : kRescaleThreshold) ||
                                   (m == -INFINITY && m_cand > -INFINITY);
                float alpha = 1.0f;
                const bool rescale = __any_sync(0xffffffffu, need);
                if (rescale) {
                    const float m_new = fmaxf(m, m_cand);
                    alpha = (m == -INFINITY) ? 0.0f : ex2_approx(m - m_new);
                    m = m_new;
                }
                const float base = (m == -INFINITY) ? 0.0f : (FP8 ? m - kFp8PShift : m);
                float sum0 = 0.0f, sum1 = 0.0f;
                // p = 2^(s * scale * log2e - m) with paired fp32 FMAs; P as bf16 pairs over
                // the first 64 columns of S_t
                const uint64_t scale2 = f2pack(sl2, sl2);
                const uint64_t nbase2 = f2pack(-base, -base);
                uint64_t sum2 = f2pack(0.0f, 0.0f);
                if constexpr (FP8) {
                    // P as E4M3, four keys per 32-bit TMEM column (the first 32 columns of S_t);
                    // p = 2^6 * 2^(s - m) <= 2^8 (max moved at a 4x rise), inside E4M3's range (448)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t pk[16];
#pragma unroll
                        for (int c = h * BN / 2; c < (h + 1) * BN / 2; c += 4) {
                            float t0, t1, t2, t3;
                            f2unpack(f2fma(f2pack(s[c], s[c + 1]), scale2, nbase2), t0, t1);
                            f2unpack(f2fma(f2pack(s[c + 2], s[c + 3]), scale2, nbase2), t2, t3);
                            const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
                            const float p2 = ex2_approx(t2), p3 = ex2_approx(t3);
                            sum2 = f2add(sum2, f2add(f2pack(p0, p1), f2pack(p2, p3)));
                            pk[(c - h * BN / 2) / 4] = pack_e4m3x4(p0, p1, p2, p3);
                        }
                        tmem_st16(s_tmem + 16 * h, pk);
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t pk[BN / 4];
#pragma unroll
                        for (int c = h * BN / 2; c < (h + 1) * BN / 2; c += 2) {
                            float t0, t1;
                            f2unpack(f2fma(f2pack(s[c], s[c + 1]), scale2, nbase2), t0, t1);
                            const float p0 = ex2_approx(t0);
                            const float p1 = ex2_approx(t1);
                            sum2 = f2add(sum2, f2pack(p0, p1));
                            pk[(c - h * BN / 2) / 2] = pack_bf16x2(p0, p1);
                        }
                        tmem_st32(s_tmem + 32 * h, pk);
                    }
                }
                f2unpack(sum2, sum0, sum1);
                l = l * alpha + (sum0 + sum1);
                if (rescale && n_act > 0) {
                    // O <- alpha * O. The previous P V has finished: it was issued before
                    // the S MMA whose completion was just observed.
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t ov[32];
                        tmem_ld32(o_tmem + 32 * c, ov);
                        tmem_ld_wait_dep32(ov);
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                        tmem_st32(o_tmem + 32 * c, ov);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(p_full(t));
                ++n_act;
            }
        }
        // ---- epilogue: O / l -> bf16, lse = ln2 * (m + log2 l)
        if (T.rows > 0 && ok) {
            const bool valid_row = row < nq;
            const size_t row_idx = (static_cast<size_t>(b) * p.Hq + T.head) * p.Nq + row;
            const float inv_l = l > 0.0f ? p.out_scale / l : 0.0f;
            if (tile_has) {
                if (mbar_wait(o_done(t), 0, abort_flag, p.err)) {
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t ov[32];
                        tmem_ld32(o_tmem + 32 * c, ov);
                        tmem_ld_wait_dep32(ov);
                        if (valid_row) {
                            uint4* dst = reinterpret_cast<uint4*>(p.o + row_idx * D + 32 * c);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                uint4 w;
                                w.x = pack_bf16x2(__uint_as_float(ov[8 * i + 0]) * inv_l,
                                                  __uint_as_float(ov[8 * i + 1]) * inv_l);
                                w.y = pack_bf16x2(__uint_as_float(ov[8 * i + 2]) * inv_l,
                                                  __uint_as_float(ov[8 * i + 3]) * inv_l);
                                w.z = pack_bf16x2(__uint_as_float(ov[8 * i + 4]) * inv_l,
                                                  __uint_as_float(ov[8 * i + 5]) * inv_l);
                                w.w = pack_bf16x2(__uint_as_float(ov[8 * i + 6]) * inv_l,
                                                  __uint_as_float(ov[8 * i + 7]) * inv_l);
                                dst[i] = w;
                            }
                        }
                    }
                    if (valid_row)
                        p.lse[row_idx] = l > 0.0f ? (m + log2f(l) - (FP8 ? kFp8PShift : 0.0f)) * kLn2 : -INFINITY;
                }
            } else if (valid_row) {
                // no key is allowed for any row of this tile
                uint4* dst = reinterpret_cast<uint4*>(p.o + row_idx * D);
#pragma unroll
                for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
                p.lse[row_idx] = -INFINITY;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D>
int launch_fwd_d(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                 int Nk, float scale, int causal, int window, const int32_t* row_ptr, const int32_t* col_idx,
                 cudaStream_t stream, unsigned* err)
{
    using C = FwdCfg<D>;
    CUtensorMap tq, tk, tv;
    const uint32_t box[3] = {64u, 128u, 1u};
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Nq),
                                  static_cast<uint64_t>(B) * Hq};
        const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(Nq) * D * 2};
        int rc = encode_bf16_map(&tq, q, 3, dims, strides, box);
        if (rc != kOk) return rc;
    }
    if (Nk > 0) {
        const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Nk), static_cast<uint64_t>(B) * Hkv};
        const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(Nk) * D * 2};
        int rc = encode_bf16_map(&tk, k, 3, dims, strides, box);
        if (rc != kOk) return rc;
        rc = encode_bf16_map(&tv, v, 3, dims, strides, box);
        if (rc != kOk) return rc;
    } else {
        // No keys: no K/V tile is ever loaded, the descriptors are placeholders.
        tk = tq;
        tv = tq;
    }
    FwdParams prm;
    prm.o = static_cast<__nv_bfloat16*>(o);
    prm.lse = lse;
    prm.B = B;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.Nq = Nq;
    prm.Nk = Nk;
    prm.G = Hq / Hkv;
    prm.scale_log2 = scale * kLog2e;
    prm.causal = causal ? 1 : 0;
    prm.window = window < 0 ? -1 : window;
    prm.pair_heads = (prm.G % 2 == 0) ? 1 : 0;
    const int n_row_tiles = (Nq + BM - 1) / BM;
    prm.n_row_units = prm.pair_heads ? n_row_tiles : (n_row_tiles + 1) / 2;
    prm.n_hunits = prm.pair_heads ? Hq / 2 : Hq;
    prm.block_table = nullptr;
    prm.q_lens = nullptr;
    prm.kv_lens = nullptr;
    prm.max_blocks = prm.block_size = prm.bs_log2 = prm.num_blocks = 0;
    prm.row_ptr = row_ptr;
    prm.col_idx = col_idx;
    prm.next_stride = sm_count();  // one block per SM: the block launched next is about this far on
    prm.out_scale = 1.0f;
    prm.err = err;
    if (2 * static_cast<long long>(B) * prm.n_hunits * prm.n_row_units <= prm.next_stride) {
        // a grid of at most half the SMs: one query tile per block instead (still one wave),
        // so the tiles run side by side
        prm.pair_heads = 2;
        prm.n_row_units = n_row_tiles;
        prm.n_hunits = Hq;
    }
    const long long grid = static_cast<long long>(B) * prm.n_hunits * prm.n_row_units;
    if (grid <= 0) return kOk;
    if (grid > INT_MAX) return kErrInvalidArg;

    if (row_ptr) {  // block-sparse: the walk follows the used bytes
        if (cudaFuncSetAttribute(attn_fwd_sm103<D, kModeSparse>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmemBytes + kWalkBytes) != cudaSuccess)
            return kErrCuda;
        attn_fwd_sm103<D, kModeSparse><<<static_cast<unsigned>(grid), kFwdThreads, C::kSmemBytes + kWalkBytes, stream>>>(
            tq, tk, tv, prm);
        return cudaGetLastError() == cudaSuccess ? kOk : kErrLaunch;
    }
    if (cudaFuncSetAttribute(attn_fwd_sm103<D, kModeDense>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes) != cudaSuccess)
        return kErrCuda;
    attn_fwd_sm103<D, kModeDense><<<static_cast<unsigned>(grid), kFwdThreads, C::kSmemBytes, stream>>>(tq, tk, tv, prm);
    return cudaGetLastError() == cudaSuccess ? kOk : kErrLaunch;
}

// FP8 prefill (d = 128): q [B][Hq][Nq][128], k [B][Hkv][Nk][128] and vt [B][Hkv][128][Nk]
// as E4M3 bytes, read through 8-bit TMA views with 128 x 128-byte boxes (a Q/K tile is
// 128 rows of 128 bytes; a V^T tile is the 128 d rows of 128 keys). Arguments are already
// validated (Nk a multiple of 16: the V^T row stride must be 16-byte aligned).
int launch_fwd_fp8_128(const void* q, const void* k, const void* vt, void* o, float* lse, int B, int Hq, int Hkv,
                       int Nq, int Nk, float scale, float q_descale, float k_descale, float v_descale, int causal,
                       int window, cudaStream_t stream, unsigned* err)
{
    constexpr int D = 128;
    using C = FwdCfg<D, 1>;
    CUtensorMap tq, tk, tv;
    const uint32_t box[3] = {128u, 128u, 1u};
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Nq), static_cast<uint64_t>(B) * Hq};
        const uint64_t strides[2] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Nq) * D};
        int rc = encode_u8_map(&tq, q, 3, dims, strides, box);
        if (rc != kOk) return rc;
    }
    if (Nk > 0) {
        const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Nk), static_cast<uint64_t>(B) * Hkv};
        const uint64_t strides[2] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Nk) * D};
        int rc = encode_u8_map(&tk, k, 3, dims, strides, box);
        if (rc != kOk) return rc;
        const uint64_t vdims[3] = {static_cast<uint64_t>(Nk), static_cast<uint64_t>(D), static_cast<uint64_t>(B) * Hkv};
        const uint64_t vstrides[2] = {static_cast<uint64_t>(Nk), static_cast<uint64_t>(D) * Nk};
        rc = encode_u8_map(&tv, vt, 3, vdims, vstrides, box);
        if (rc != kOk) return rc;
    } else {
        tk = tq;  // no keys: never loaded
        tv = tq;
    }
    FwdParams prm;
    prm.o = static_cast<__nv_bfloat16*>(o);
    prm.lse = lse;
    prm.B = B;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.Nq = Nq;
    prm.Nk = Nk;
    prm.G = Hq / Hkv;
    // S comes out of the MMA in code units: the scales of Q and K join the softmax scale
    prm.scale_log2 = scale * q_descale * k_descale * kLog2e;
    prm.causal = causal ? 1 : 0;
    prm.window = window < 0 ? -1 : window;
    prm.pair_heads = (prm.G % 2 == 0) ? 1 : 0;
    const int n_row_tiles = (Nq + BM - 1) / BM;
    prm.n_row_units = prm.pair_heads ? n_row_tiles : (n_row_tiles + 1) / 2;
    prm.n_hunits = prm.pair_heads ? Hq / 2 : Hq;
    prm.block_table = nullptr;
    prm.q_lens = nullptr;
    prm.kv_lens = nullptr;
    prm.max_blocks = prm.block_size = prm.bs_log2 = prm.num_blocks = 0;
    prm.row_ptr = nullptr;
    prm.col_idx = nullptr;
    prm.next_stride = sm_count();
    prm.out_scale = v_descale;
    prm.err = err;
    if (2 * static_cast<long long>(B) * prm.n_hunits * prm.n_row_units <= prm.next_stride) {
        prm.pair_heads = 2;  // a grid of at most half the SMs: one query tile per block (one wave)
        prm.n_row_units = n_row_tiles;
        prm.n_hunits = Hq;
    }
    const long long grid = static_cast<long long>(B) * prm.n_hunits * prm.n_row_units;
    if (grid <= 0) return kOk;
    if (grid > INT_MAX) return kErrInvalidArg;
    if (cudaFuncSetAttribute(attn_fwd_sm103<D, kModeFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes) != cudaSuccess)
        return kErrCuda;
    attn_fwd_sm103<D, kModeFp8><<<static_cast<unsigned>(grid), kFwdThreads, C::kSmemBytes, stream>>>(tq, tk, tv, prm);
    return cudaGetLastError() == cudaSuccess ? kOk : kErrLaunch;
}

// Paged prefill: q, o [S][Hq][max_q][d]; caches [num_blocks][Hkv][block_size][d] read
// through 2-D TMA views {d, num_blocks * Hkv * block_size} with min(block_size, 128)-row
// boxes. Arguments are already validated (block_size a power of two in [16, 256]).
template <int D>
int launch_fwd_paged_d(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                       const int32_t* q_lens, const int32_t* kv_lens, void* o, float* lse, int S, int Hq, int Hkv,
                       int block_size, int max_blocks, int num_blocks, int max_q, float scale, int causal, int window,
                       cudaStream_t stream, unsigned* err)
{
    using C = FwdCfg<D>;
    CUtensorMap tq, tk, tv;
    {
        const uint32_t box[3] = {64u, 128u, 1u};
        const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(max_q), static_cast<uint64_t>(S) * Hq};
        const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(max_q) * D * 2};
        int rc = encode_bf16_map(&tq, q, 3, dims, strides, box);
        if (rc != kOk) return rc;
    }
    {
        const uint32_t box[2] = {64u, static_cast<uint32_t>(block_size < BN ? block_size : BN)};
        const uint64_t dims[2] = {static_cast<uint64_t>(D), static_cast<uint64_t>(num_blocks) * Hkv * block_size};
        const uint64_t strides[1] = {static_cast<uint64_t>(D) * 2};
        int rc = encode_bf16_map(&tk, k_cache, 2, dims, strides, box);
        if (rc != kOk) return rc;
        rc = encode_bf16_map(&tv, v_cache, 2, dims, strides, box);
        if (rc != kOk) return rc;
    }
    FwdParams prm;
    prm.o = static_cast<__nv_bfloat16*>(o);
    prm.lse = lse;
    prm.B = S;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.Nq = max_q;
    prm.Nk = 0;
    prm.G = Hq / Hkv;
    prm.block_table = block_table;
    prm.q_lens = q_lens;
    prm.kv_lens = kv_lens;
    prm.max_blocks = max_blocks;
    prm.block_size = block_size;
    prm.bs_log2 = 31 - __builtin_clz(static_cast<unsigned>(block_size));
    prm.num_blocks = num_blocks;
    prm.row_ptr = nullptr;
    prm.col_idx = nullptr;
    prm.scale_log2 = scale * kLog2e;
    prm.causal = causal ? 1 : 0;
    prm.window = window < 0 ? -1 : window;
    prm.pair_heads = (prm.G % 2 == 0) ? 1 : 0;
    const int n_row_tiles = (max_q + BM - 1) / BM;
    prm.n_row_units = prm.pair_heads ? n_row_tiles : (n_row_tiles + 1) / 2;
    prm.n_hunits = prm.pair_heads ? Hq / 2 : Hq;
    prm.next_stride = 0;
    prm.out_scale = 1.0f;
    prm.err = err;
    const long long grid = static_cast<long long>(S) * prm.n_hunits * prm.n_row_units;
    if (grid <= 0) return kOk;
    if (grid > INT_MAX) return kErrInvalidArg;
    if (cudaFuncSetAttribute(attn_fwd_sm103<D, kModePaged>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes) != cudaSuccess)
        return kErrCuda;
    attn_fwd_sm103<D, kModePaged><<<static_cast<unsigned>(grid), kFwdThreads, C::kSmemBytes, stream>>>(tq, tk, tv, prm);
    return cudaGetLastError() == cudaSuccess ? kOk : kErrLaunch;
}

}  // namespace

int launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
               int Nk, int d, float scale, int causal, int window, cudaStream_t stream, unsigned* err)
{
    if (Nq == 0) return kOk;
    if (d == 128)
        return launch_fwd_d<128>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, window, nullptr, nullptr, stream,
                                 err);
    if (d == 64)
        return launch_fwd_d<64>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, window, nullptr, nullptr, stream,
                                err);
    return kErrUnsupported;
}

int launch_fwd_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                           int Nq, int Nk, int d, float scale, int causal, int window, const int32_t* row_ptr,
                           const int32_t* col_idx, cudaStream_t stream, unsigned* err)
{
    if (Nq == 0) return kOk;
    if (d == 128)
        return launch_fwd_d<128>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, window, row_ptr, col_idx, stream,
                                 err);
    if (d == 64)
        return launch_fwd_d<64>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, window, row_ptr, col_idx, stream,
                                err);
    return kErrUnsupported;
}

int launch_fwd_fp8(const void* q, const void* k, const void* vt, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                   int Nk, int d, float scale, float q_descale, float k_descale, float v_descale, int causal,
                   int window, cudaStream_t stream, unsigned* err)
{
    if (d != 128) return kErrUnsupported;
    return launch_fwd_fp8_128(q, k, vt, o, lse, B, Hq, Hkv, Nq, Nk, scale, q_descale, k_descale, v_descale, causal,
                              window, stream, err);
}

int launch_fwd_paged(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                     const int32_t* q_lens, const int32_t* kv_lens, void* o, float* lse, int S, int Hq, int Hkv, int d,
                     int block_size, int max_blocks, int num_blocks, int max_q, float scale, int causal, int window,
                     cudaStream_t stream, unsigned* err)
{
    if (S == 0 || max_q == 0) return kOk;
    if (d == 128)
        return launch_fwd_paged_d<128>(q, k_cache, v_cache, block_table, q_lens, kv_lens, o, lse, S, Hq, Hkv,
                                       block_size, max_blocks, num_blocks, max_q, scale, causal, window, stream, err);
    if (d == 64)
        return launch_fwd_paged_d<64>(q, k_cache, v_cache, block_table, q_lens, kv_lens, o, lse, S, Hq, Hkv,
                                      block_size, max_blocks, num_blocks, max_q, scale, causal, window, stream, err);
    return kErrUnsupported;
}

}  // namespace attn
