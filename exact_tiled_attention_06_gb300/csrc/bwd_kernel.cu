// bwd_kernel.cu -- attention backward for sm_103a: dQ, dK, dV from Q, K, V, O, dO and
// the forward's per-row lse, with the score tiles recomputed.
//
// Pages: "Modern attention kernels", "Backward pass recomputes scores" (the forward
// saves compact per-row statistics; the backward recomputes score tiles instead of
// storing P); "Flash attention and IO-aware attention" (save only the row statistics,
// recompute P block by block); "Attention kernels" (recompute from Q, K, V on the fly).
//
// For a row i and key j (P_ij = 2^(s_ij * scale * log2e - lse_i * log2e), 0 if masked):
//   dV_j = sum_i P_ij dO_i          dP_ij = dO_i . v_j          D_i = dO_i . O_i
//   dS_ij = P_ij (dP_ij - D_i)      dQ_i = scale sum_j dS_ij k_j      dK_j = scale sum_i dS_ij q_i
// (D_i equals sum_j P_ij dP_ij because O_i = sum_j P_ij v_j.)
//
// Three launches:
//   attn_bwd_prep      D_i = rowsum(dO o O) in fp32, and a zeroed fp32 dQ accumulator
//   attn_bwd_sm103     one CTA per (128-key tile, kv head): dK, dV accumulate in TMEM
//                      over every query head of the group and every query tile that sees
//                      the keys; each tile's dQ partial is added to the fp32 accumulator
//   attn_bwd_dq_out    dQ = scale * accumulator, rounded to bf16
//
// Main kernel roles (192 threads):
//   warps 0-3  element-wise work, thread = TMEM lane: P^T and dS^T rows (lane = key),
//              then the dQ partial (lane = d for d = 128, lane = query for d = 64) and
//              the final dK, dV (lane = key)
//   warp  4    TMEM allocation and tcgen05 MMA issue (one thread)
//   warp  5    TMA producer (one thread): K and V once, then Q and dO per query tile
//              into two stages, so that the next tile loads while the current one is used
// TMEM columns: [0,128) S^T, then P^T packed bf16 in [64,128); [128,256) dP^T, then dS^T
// packed in [192,256); the dQ partial goes to the columns freed by the softmax ([0,64) and
// [128,192): dQ^T's query halves for d = 128, dQ's 64 columns for d = 64), so that no MMA
// writes a column another MMA of the same tile still reads; dV and dK accumulate in
// [256,256+d) and [256+d,256+2d).
#include <climits>
#include <cmath>
#include <cstdint>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int BQ = 128;  // query rows per tile
constexpr int BK = 128;  // keys per tile (TMEM lanes in the key-major products)
constexpr int kBwdThreads = 192;
constexpr int kMmaWarpB = 4;
constexpr int kLoadWarpB = 5;
constexpr float kLog2eB = 1.4426950408889634f;

template <int D>
struct BwdCfg {
    static constexpr int kBoxes = D / 64;
    static constexpr int kBoxBytes = 128 * 128;         // 128 rows x 128 bytes
    static constexpr int kTileBytes = kBoxes * kBoxBytes;
    static constexpr int kKOff = 0;                     // K tile (resident)
    static constexpr int kVOff = kTileBytes;            // V tile (resident)
    static constexpr int kQOff = 2 * kTileBytes;        // Q tile, stage s at + s * kStageStride
    static constexpr int kDOOff = 3 * kTileBytes;       // dO tile, stage s at + s * kStageStride
    static constexpr int kStageStride = 2 * kTileBytes; // two stages: the next query tile loads
                                                        // while the current one is in use
    static constexpr int kDSOff = 6 * kTileBytes;       // dS^T, bf16, MN-major operand (32 KB)
    // lse (log2 units) and D of the tile's queries, 128 + 128 fp32, two buffers
    static constexpr int kVecOff = kDSOff + 2 * kBoxBytes;
    static constexpr int kBarOff = kVecOff + 2 * 2 * BQ * 4;
    static constexpr int kNumBars = 12;
    static constexpr int kHolderOff = kBarOff + 8 * kNumBars;
    static constexpr int kAbortOff = kHolderOff + 4;
    static constexpr int kUsedBytes = kAbortOff + 4;
    // Dynamic shared memory: the used bytes plus what is left for aligning the base to
    // 1024 bytes, within the 227 KB a block may have; at least ~120 KB so that two
    // blocks never share an SM (each takes all of TMEM). The kernel checks that the
    // aligned layout fits before it touches anything.
    static constexpr int kMaxDynSmem = 227 * 1024;
    static constexpr int kPadded = (kUsedBytes + 1024) < kMaxDynSmem ? (kUsedBytes + 1024) : kMaxDynSmem;
    static constexpr int kSmemBytes = kPadded > 122880 ? kPadded : 122880;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kSCol = 0, kPCol = 64, kDPCol = 128, kDSCol = 192;
    static constexpr uint32_t kDQCol0 = 0, kDQCol1 = 128;  // dQ partial, d in [0,64) and [64,128)
    static constexpr uint32_t kDVCol = 256, kDKCol = 256 + D;
    static_assert(kUsedBytes <= kMaxDynSmem, "shared memory budget");
    static_assert(kDKCol + D <= kTmemCols, "TMEM budget");
    static_assert(kDQCol1 + 64 <= kDSCol && kDQCol0 + 64 <= kPCol, "dQ columns overlap P^T or dS^T");
};

struct BwdParams {
    const __nv_bfloat16* o;
    const __nv_bfloat16* dout;
    const float* lse;
    const float* dvec;   // D_i, fp32 [B][Hq][Nq]
    float* dq_acc;       // fp32 [B][Hq][Nq][d]
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    int B, Hq, Hkv, Nq, Nk, G;
    float scale, scale_log2;
    int causal, window;
    int n_ktiles;
    unsigned* err;
};

// ---------------------------------------------------------------------------- prep
// One warp per row: D_i = sum_c dO_ic O_ic (fp32), and the row of the dQ accumulator
// set to zero.
template <int D>
__global__ void __launch_bounds__(256)
    attn_bwd_prep(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                  float* __restrict__ dvec, float* __restrict__ dq_acc, long long rows)
{
    const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const __nv_bfloat16* orow = o + row * D;
    const __nv_bfloat16* drow = dout + row * D;
    float acc = 0.0f;
#pragma unroll
    for (int c = lane * 2; c < D; c += 64) {
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(orow + c));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(drow + c));
        acc = fmaf(a.x, b.x, fmaf(a.y, b.y, acc));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) dvec[row] = acc;
    float4* z = reinterpret_cast<float4*>(dq_acc + row * D);
    for (int c = lane; c < D / 4; c += 32) z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ---------------------------------------------------------------------------- dQ out
template <int D>
__global__ void __launch_bounds__(256)
    attn_bwd_dq_out(const float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dq, float scale, long long n4)
{
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n4) return;
    const float4 a = reinterpret_cast<const float4*>(dq_acc)[i];
    uint2 w;
    w.x = pack_bf16x2(a.x * scale, a.y * scale);
    w.y = pack_bf16x2(a.z * scale, a.w * scale);
    reinterpret_cast<uint2*>(dq)[i] = w;
}

// Query tiles that see some key of tile kt: causal keeps queries with i + delta >= k0;
// a window w keeps queries with i + delta - w <= k1 - 1.
__device__ __forceinline__ void query_tile_range(const BwdParams& p, int kt, int& qlo, int& qhi)
{
    const long long delta = static_cast<long long>(p.Nk) - p.Nq;
    const long long k0 = static_cast<long long>(kt) * BK;
    long long k1 = k0 + BK;
    if (k1 > p.Nk) k1 = p.Nk;
    long long i_lo = 0, i_hi = p.Nq;  // queries [i_lo, i_hi)
    if (p.causal && k0 - delta > i_lo) i_lo = k0 - delta;
    if (p.window >= 0) {
        const long long h = k1 - 1 + p.window - delta + 1;
        if (h < i_hi) i_hi = h;
    }
    if (i_hi <= i_lo) {
        qlo = qhi = 0;
        return;
    }
    qlo = static_cast<int>(i_lo / BQ);
    qhi = static_cast<int>((i_hi + BQ - 1) / BQ);
}

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_sm103(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const BwdParams p)
{
    using C = BwdCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Block order: key tile outer, (batch, kv head) inner, so that under a causal mask the
    // tiles that see the most query tiles (the first key tiles) are scheduled first.
    const int n_bk = p.B * p.Hkv;
    const int kt = static_cast<int>(blockIdx.x) / n_bk;
    const int bk = static_cast<int>(blockIdx.x) % n_bk;  // batch * Hkv + kv head
    const int b = bk / p.Hkv;
    const int hkv = bk % p.Hkv;
    int qlo, qhi;
    query_tile_range(p, kt, qlo, qhi);
    const int n_it = p.G * (qhi - qlo);  // (query head of the group, query tile) pairs

    const uint32_t bar0 = sb + C::kBarOff;
    const uint32_t kv_full = bar0;             // K and V tiles landed
    const uint32_t st_full = bar0 + 8u;        // two barriers: Q and dO of stage 0 / 1 landed
    const uint32_t st_empty = bar0 + 24u;      // two barriers: every MMA reading stage 0 / 1 done
    const uint32_t sdp_full = bar0 + 40u;      // S^T and dP^T are in TMEM
    const uint32_t p_ready = bar0 + 48u;       // P^T, dS^T written (TMEM and shared memory)
    const uint32_t dq_full = bar0 + 56u;       // the dQ partial is in TMEM
    const uint32_t dq_read = bar0 + 64u;       // the dQ partial has been read out
    const uint32_t fin = bar0 + 72u;           // every MMA is done
    const uint32_t vec_full = bar0 + 80u;      // two barriers: statistics buffer 0 / 1 written
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kHolderOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbortOff);

    // The 1024-byte aligned layout must fit in what was requested (uniform for the block).
    if (static_cast<int>(smem - smem_raw) + C::kUsedBytes > C::kSmemBytes) {
        if (threadIdx.x == 0) report_error(p.err, kDevErrBounds);
        return;
    }
    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        mbar_init(st_full, 1);
        mbar_init(st_full + 8u, 1);
        mbar_init(st_empty, 1);
        mbar_init(st_empty + 8u, 1);
        mbar_init(sdp_full, 1);
        mbar_init(p_ready, 128);
        mbar_init(dq_full, 1);
        mbar_init(dq_read, 128);
        mbar_init(fin, 1);
        mbar_init(vec_full, 128);
        mbar_init(vec_full + 8u, 128);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarpB) {
        tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t sK = sb + C::kKOff, sV = sb + C::kVOff, sQ = sb + C::kQOff, sDO = sb + C::kDOOff;
    const uint32_t sDS = sb + C::kDSOff;

    if (warp == kLoadWarpB) {
        // ================================================================ producer
        if (lane == 0 && n_it > 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_do);
            mbar_arrive_expect_tx(kv_full, 2 * C::kTileBytes);
#pragma unroll
            for (int x = 0; x < C::kBoxes; ++x) {
                tma_load_3d(sK + x * C::kBoxBytes, &tm_k, kv_full, 64 * x, kt * BK, bk);
                tma_load_3d(sV + x * C::kBoxBytes, &tm_v, kv_full, 64 * x, kt * BK, bk);
            }
            int it = 0;  // query tiles issued; tile t uses stage t % 2, its (t / 2)-th use
            for (int g = 0; g < p.G; ++g) {
                const int hq = hkv * p.G + g;
                for (int qt = qlo; qt < qhi; ++qt, ++it) {
                    const int st = it & 1;
                    const uint32_t full = st_full + 8u * st;
                    if (it >= 2 && !mbar_wait(st_empty + 8u * st, ((it >> 1) - 1) & 1, abort_flag, p.err))
                        goto producer_done;
                    mbar_arrive_expect_tx(full, 2 * C::kTileBytes);
                    const uint32_t so = st * C::kStageStride;
#pragma unroll
                    for (int x = 0; x < C::kBoxes; ++x) {
                        tma_load_3d(sQ + so + x * C::kBoxBytes, &tm_q, full, 64 * x, qt * BQ, b * p.Hq + hq);
                        tma_load_3d(sDO + so + x * C::kBoxBytes, &tm_do, full, 64 * x, qt * BQ, b * p.Hq + hq);
                    }
                }
            }
        producer_done:
            // never leave while a copy into this block's shared memory is in flight: wait
            // for the last tile issued on each stage
            mbar_wait(kv_full, 0, nullptr, p.err);
            for (int t = it >= 2 ? it - 2 : 0; t < it; ++t) mbar_wait(st_full + 8u * (t & 1), (t >> 1) & 1, nullptr, p.err);
        }
    } else if (warp == kMmaWarpB) {
        // ================================================================ MMA issue
        if (lane == 0 && n_it > 0) {
            constexpr uint32_t idesc_kq = idesc_bf16_f32(BK, BQ, false, false);  // S^T, dP^T
            constexpr uint32_t idesc_pd = idesc_bf16_f32(BK, D, false, true);    // dV, dK (A in TMEM)
            // dQ: d = 128 computes dQ^T = K^T dS^T (lane = d, so that the accumulator adds are
            // coalesced along d), one 64-query half at a time; d = 64 computes dQ = dS K
            // (lane = query, N = 64).
            constexpr uint32_t idesc_dq = D == 128 ? idesc_bf16_f32(D, 64, true, true) : idesc_bf16_f32(BQ, 64, true, true);
            // K-major descriptors (16-wide k steps inside 128-byte rows, a new box every 64)
            const uint64_t kd = smem_desc_sw128(sK, 16, 1024), vd = smem_desc_sw128(sV, 16, 1024);
            const uint64_t qd = smem_desc_sw128(sQ, 16, 1024), dod = smem_desc_sw128(sDO, 16, 1024);
            // MN-major descriptors (16 rows of the reduction dimension = 2048 bytes per step,
            // the two 64-wide halves of the other dimension one box apart)
            const uint64_t q_mn = smem_desc_sw128(sQ, C::kBoxBytes, 1024);
            const uint64_t do_mn = smem_desc_sw128(sDO, C::kBoxBytes, 1024);
            const uint64_t k_mn = smem_desc_sw128(sK, C::kBoxBytes, 1024);
            const uint64_t ds_mn = smem_desc_sw128(sDS, C::kBoxBytes, 1024);
            bool ok = mbar_wait(kv_full, 0, abort_flag, p.err);
            for (int it = 0; it < n_it && ok; ++it) {
                const int st = it & 1;
                if (!mbar_wait(st_full + 8u * st, (it >> 1) & 1, abort_flag, p.err)) break;
                if (it > 0 && !mbar_wait(dq_read, (it - 1) & 1, abort_flag, p.err)) break;
                tc_fence_after();
                const uint64_t so = static_cast<uint64_t>((st * C::kStageStride) >> 4);  // stage offset
                // S^T = K Q^T and dP^T = V dO^T (keys x queries)
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = static_cast<uint64_t>(((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4);
                    mma_ss(tmem + C::kSCol, kd + off, qd + so + off, idesc_kq, kk > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = static_cast<uint64_t>(((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4);
                    mma_ss(tmem + C::kDPCol, vd + off, dod + so + off, idesc_kq, kk > 0 ? 1u : 0u);
                }
                tc_commit(sdp_full);
                if (!mbar_wait(p_ready, it & 1, abort_flag, p.err)) break;
                tc_fence_after();
                // dV += P^T dO and dK += dS^T Q (A from TMEM, 16 queries = 8 columns per step)
#pragma unroll
                for (int kk = 0; kk < BQ / 16; ++kk)
                    mma_ts(tmem + C::kDVCol, tmem + C::kPCol + kk * 8, do_mn + so + static_cast<uint64_t>(kk * 128),
                           idesc_pd, (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < BQ / 16; ++kk)
                    mma_ts(tmem + C::kDKCol, tmem + C::kDSCol + kk * 8, q_mn + so + static_cast<uint64_t>(kk * 128),
                           idesc_pd, (it > 0 || kk > 0) ? 1u : 0u);
                tc_commit(st_empty + 8u * st);  // Q and dO of this stage are no longer read
                // dQ partial, into columns that neither dV nor dK reads
                if constexpr (D == 128) {
                    // dQ^T (d x queries) = K^T dS^T: A = K MN-major, B = dS^T MN-major, one
                    // 64-query half (one 16 KB block of the dS^T buffer) at a time
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            mma_ss(tmem + (h == 0 ? C::kDQCol0 : C::kDQCol1), k_mn + static_cast<uint64_t>(kk * 128),
                                   ds_mn + static_cast<uint64_t>((h * C::kBoxBytes) >> 4) +
                                       static_cast<uint64_t>(kk * 128),
                                   idesc_dq, kk > 0 ? 1u : 0u);
                } else {
                    // dQ (queries x d) = dS K: A = dS MN-major, B = K MN-major
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_ss(tmem + C::kDQCol0, ds_mn + static_cast<uint64_t>(kk * 128),
                               k_mn + static_cast<uint64_t>(kk * 128), idesc_dq, kk > 0 ? 1u : 0u);
                }
                tc_commit(dq_full);
            }
            tc_commit(fin);
            mbar_wait(fin, 0, nullptr, p.err);
        }
    } else {
        // ================================================================ warps 0-3
        const int row = threadIdx.x;                       // TMEM lane owned by this thread
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const long long delta = static_cast<long long>(p.Nk) - p.Nq;
        // Queries allowed to see key j (the key of this thread in the S^T, dP^T products):
        // i in [i_min, i_max]; causal j <= i + delta, window j >= i + delta - w.
        const long long j = static_cast<long long>(kt) * BK + row;
        long long i_min = 0, i_max = static_cast<long long>(p.Nq) - 1;
        if (p.causal && j - delta > i_min) i_min = j - delta;
        if (p.window >= 0 && j - delta + p.window < i_max) i_max = j - delta + p.window;
        if (j >= p.Nk) i_max = -1;
        bool ok = true;
        int it = 0;
        for (int g = 0; g < p.G && ok; ++g) {
            const int hq = hkv * p.G + g;
            const long long rowbase = (static_cast<long long>(b) * p.Hq + hq) * p.Nq;
            for (int qt = qlo; qt < qhi; ++qt, ++it) {
                // ---- per-query statistics of this tile, in buffer it % 2. Every thread
                // finished reading that buffer (two tiles ago) before it arrived on p_ready
                // of the previous tile, which this thread's dq_full wait has seen complete.
                const int u = it & 1;
                float* s_lse2 = reinterpret_cast<float*>(smem + C::kVecOff) + u * 2 * BQ;  // lse * log2(e)
                float* s_dvec = s_lse2 + BQ;                                                // D
                {
                    const int q = qt * BQ + row;
                    float l2 = INFINITY, dd = 0.0f;
                    if (q < p.Nq) {
                        l2 = p.lse[rowbase + q] * kLog2eB;
                        dd = p.dvec[rowbase + q];
                    }
                    s_lse2[row] = l2;
                    s_dvec[row] = dd;
                }
                mbar_arrive(vec_full + 8u * u);
                // (wait results are made warp-uniform: the tcgen05 loads and stores below are
                // warp-collective and must be reached by all 32 lanes or by none)
                if (!__all_sync(0xffffffffu, mbar_wait(vec_full + 8u * u, (it >> 1) & 1, abort_flag, p.err))) {
                    ok = false;
                    break;
                }
                const long long q0 = static_cast<long long>(qt) * BQ;
                const int c_lo = static_cast<int>(max(-1ll, min(static_cast<long long>(BQ), i_min - q0)));
                const int c_hi = static_cast<int>(max(-1ll, min(static_cast<long long>(BQ), i_max - q0)));
                const bool full = c_lo <= 0 && c_hi >= BQ - 1;
                if (!__all_sync(0xffffffffu, mbar_wait(sdp_full, it & 1, abort_flag, p.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // ---- P^T and dS^T, 64 queries at a time (32 packed bf16 pairs per half).
                // The upper half goes first: its packed rows land in columns whose fp32
                // scores it has just read, and the lower half's packed rows land in
                // columns the upper half has already consumed.
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    const int half = 1 - hh;
                    uint32_t pp[32], pd[32];
#pragma unroll
                    for (int sub = 0; sub < 2; ++sub) {
                        const int c0 = half * 64 + sub * 32;
                        uint32_t sr[32], dr[32];
                        tmem_ld32(tmem + lane_base + C::kSCol + c0, sr);
                        tmem_ld32(tmem + lane_base + C::kDPCol + c0, dr);
                        tmem_ld_wait_dep32(sr);
                        tmem_ld_wait_dep32(dr);
#pragma unroll
                        for (int k = 0; k < 32; k += 2) {
                            float pv[2], dv[2];
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int c = c0 + k + e;
                                const float pe =
                                    ex2_approx(fmaf(__uint_as_float(sr[k + e]), p.scale_log2, -s_lse2[c]));
                                const float de = pe * (__uint_as_float(dr[k + e]) - s_dvec[c]);
                                const bool allowed = full || (c >= c_lo && c <= c_hi);
                                pv[e] = allowed ? pe : 0.0f;
                                dv[e] = allowed ? de : 0.0f;
                            }
                            pp[sub * 16 + k / 2] = pack_bf16x2(pv[0], pv[1]);
                            pd[sub * 16 + k / 2] = pack_bf16x2(dv[0], dv[1]);
                        }
                    }
                    // P^T and dS^T rows into TMEM (A operands of dV and dK) ...
                    tmem_st32(tmem + lane_base + C::kPCol + half * 32, pp);
                    tmem_st32(tmem + lane_base + C::kDSCol + half * 32, pd);
                    // ... and dS^T into shared memory as the MN-major A operand of dQ:
                    // queries [64 half, 64 half + 64) form one 16 KB block, key `row` is a
                    // 128-byte row, its 16-byte chunks XOR-swizzled with (row mod 8).
                    const uint32_t rbase = sDS + half * C::kBoxBytes + row * 128;
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        const uint32_t addr = rbase + ((cc ^ (row & 7)) << 4);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pd[4 * cc]),
                                     "r"(pd[4 * cc + 1]), "r"(pd[4 * cc + 2]), "r"(pd[4 * cc + 3])
                                     : "memory");
                    }
                }
                tmem_st_wait();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(p_ready);
                // ---- the dQ partial: add it to the fp32 accumulator
                if (!__all_sync(0xffffffffu, mbar_wait(dq_full, it & 1, abort_flag, p.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if constexpr (D == 128) {
                    // dQ^T: lane = d (this thread's row), column = query. For each query the
                    // 32 lanes of a warp add 32 consecutive floats: one 128-byte line.
                    float* dst = p.dq_acc + (rowbase + q0) * D + row;
#pragma unroll 1
                    for (int c0 = 0; c0 < BQ; c0 += 32) {
                        uint32_t r[32];
                        __syncwarp();
                        tmem_ld32(tmem + lane_base + (c0 < 64 ? C::kDQCol0 + c0 : C::kDQCol1 + (c0 - 64)), r);
                        tmem_ld_wait_dep32(r);
                        const int n_valid = static_cast<int>(min(32ll, static_cast<long long>(p.Nq) - (q0 + c0)));
#pragma unroll
                        for (int m = 0; m < 32; ++m)
                            if (m < n_valid)
                                asm volatile("red.global.add.f32 [%0], %1;" ::"l"(dst + static_cast<long long>(c0 + m) * D),
                                             "f"(__uint_as_float(r[m]))
                                             : "memory");
                    }
                } else {
                    // dQ: lane = query (this thread's row), column = d
                    const long long q = q0 + row;
                    float* dst = p.dq_acc + (rowbase + q) * D;
                    uint32_t r[32];
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        __syncwarp();
                        tmem_ld32(tmem + lane_base + C::kDQCol0 + c0, r);
                        tmem_ld_wait_dep32(r);
                        if (q < p.Nq) {
#pragma unroll
                            for (int m = 0; m < 8; ++m)
                                asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + c0 + 4 * m),
                                             "f"(__uint_as_float(r[4 * m])), "f"(__uint_as_float(r[4 * m + 1])),
                                             "f"(__uint_as_float(r[4 * m + 2])), "f"(__uint_as_float(r[4 * m + 3]))
                                             : "memory");
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(dq_read);
            }
        }
        // ---- dK, dV (lane = key) once every MMA is done. Every lane loads (the TMEM
        // loads are warp-collective); only lanes with a key inside the sequence store.
        const bool have = n_it > 0 ? mbar_wait(fin, 0, nullptr, p.err) : true;
        tc_fence_after();
        if (__all_sync(0xffffffffu, have && ok && *abort_flag == 0)) {
            const long long obase = ((static_cast<long long>(b) * p.Hkv + hkv) * p.Nk + j) * D;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t rv[32], rk[32];
                __syncwarp();
                if (n_it > 0) {
                    tmem_ld32(tmem + lane_base + C::kDVCol + c0, rv);
                    tmem_ld32(tmem + lane_base + C::kDKCol + c0, rk);
                    tmem_ld_wait_dep32(rv);
                    tmem_ld_wait_dep32(rk);
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k) rv[k] = rk[k] = 0u;
                }
                if (j < p.Nk) {
                    uint4* pv = reinterpret_cast<uint4*>(p.dv + obase + c0);
                    uint4* pk = reinterpret_cast<uint4*>(p.dk + obase + c0);
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        uint4 wv, wk;
                        wv.x = pack_bf16x2(__uint_as_float(rv[8 * m + 0]), __uint_as_float(rv[8 * m + 1]));
                        wv.y = pack_bf16x2(__uint_as_float(rv[8 * m + 2]), __uint_as_float(rv[8 * m + 3]));
                        wv.z = pack_bf16x2(__uint_as_float(rv[8 * m + 4]), __uint_as_float(rv[8 * m + 5]));
                        wv.w = pack_bf16x2(__uint_as_float(rv[8 * m + 6]), __uint_as_float(rv[8 * m + 7]));
                        wk.x = pack_bf16x2(__uint_as_float(rk[8 * m + 0]) * p.scale, __uint_as_float(rk[8 * m + 1]) * p.scale);
                        wk.y = pack_bf16x2(__uint_as_float(rk[8 * m + 2]) * p.scale, __uint_as_float(rk[8 * m + 3]) * p.scale);
                        wk.z = pack_bf16x2(__uint_as_float(rk[8 * m + 4]) * p.scale, __uint_as_float(rk[8 * m + 5]) * p.scale);
                        wk.w = pack_bf16x2(__uint_as_float(rk[8 * m + 6]) * p.scale, __uint_as_float(rk[8 * m + 7]) * p.scale);
                        pv[m] = wv;
                        pk[m] = wk;
                    }
                }
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarpB) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D>
int launch_bwd_d(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                 void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk, float scale, int causal,
                 int window, void* workspace, cudaStream_t stream, unsigned* err)
{
    using C = BwdCfg<D>;
    const long long rows = static_cast<long long>(B) * Hq * Nq;
    const BwdLayout lay = bwd_layout(B, Hq, Nq, D);
    float* dvec = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + lay.dvec_offset);
    float* dq_acc = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + lay.dq_offset);
    if ((rows + 7) / 8 > INT_MAX || (rows * D / 4 + 255) / 256 > INT_MAX) return kErrInvalidArg;

    // ---- D_i and the zeroed dQ accumulator
    if (rows > 0) {
        attn_bwd_prep<D><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), dvec, dq_acc, rows);
        if (cudaGetLastError() != cudaSuccess) return kErrLaunch;
    }

    // ---- dK, dV and the dQ partials
    const int n_ktiles = (Nk + BK - 1) / BK;
    const long long grid = static_cast<long long>(n_ktiles) * B * Hkv;
    if (grid > INT_MAX) return kErrInvalidArg;
    if (grid > 0) {
        CUtensorMap tq, tk, tv, tdo;
        const uint32_t box[3] = {64u, 128u, 1u};
        {
            const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Nk),
                                      static_cast<uint64_t>(B) * Hkv};
            const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(Nk) * D * 2};
            int rc = encode_bf16_map(&tk, k, 3, dims, strides, box);
            if (rc != kOk) return rc;
            rc = encode_bf16_map(&tv, v, 3, dims, strides, box);
            if (rc != kOk) return rc;
        }
        if (Nq > 0) {
            const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Nq),
                                      static_cast<uint64_t>(B) * Hq};
            const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(Nq) * D * 2};
            int rc = encode_bf16_map(&tq, q, 3, dims, strides, box);
            if (rc != kOk) return rc;
            rc = encode_bf16_map(&tdo, dout, 3, dims, strides, box);
            if (rc != kOk) return rc;
        } else {
            // No queries: no query tile is ever loaded and every block writes zero dK, dV.
            tq = tk;
            tdo = tk;
        }
        BwdParams prm;
        prm.o = static_cast<const __nv_bfloat16*>(o);
        prm.dout = static_cast<const __nv_bfloat16*>(dout);
        prm.lse = lse;
        prm.dvec = dvec;
        prm.dq_acc = dq_acc;
        prm.dk = static_cast<__nv_bfloat16*>(dk);
        prm.dv = static_cast<__nv_bfloat16*>(dv);
        prm.B = B;
        prm.Hq = Hq;
        prm.Hkv = Hkv;
        prm.Nq = Nq;
        prm.Nk = Nk;
        prm.G = Hq / Hkv;
        prm.scale = scale;
        prm.scale_log2 = scale * kLog2eB;
        prm.causal = causal ? 1 : 0;
        prm.window = window < 0 ? -1 : window;
        prm.n_ktiles = n_ktiles;
        prm.err = err;
        if (cudaFuncSetAttribute(attn_bwd_sm103<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
            cudaSuccess)
            return kErrCuda;
        attn_bwd_sm103<D><<<static_cast<unsigned>(grid), kBwdThreads, C::kSmemBytes, stream>>>(tq, tk, tv, tdo, prm);
        if (cudaGetLastError() != cudaSuccess) return kErrLaunch;
    }

    // ---- dQ = scale * accumulator in bf16
    if (rows > 0) {
        const long long n4 = rows * D / 4;
        attn_bwd_dq_out<D><<<static_cast<unsigned>((n4 + 255) / 256), 256, 0, stream>>>(
            dq_acc, static_cast<__nv_bfloat16*>(dq), scale, n4);
        if (cudaGetLastError() != cudaSuccess) return kErrLaunch;
    }
    return kOk;
}

}  // namespace

BwdLayout bwd_layout(int B, int Hq, int Nq, int d)
{
    const size_t rows = static_cast<size_t>(B) * Hq * Nq;
    BwdLayout lay;
    lay.dvec_offset = 0;
    lay.dq_offset = (rows * sizeof(float) + 255) / 256 * 256;
    lay.bytes = lay.dq_offset + rows * static_cast<size_t>(d) * sizeof(float);
    if (lay.bytes == 0) lay.bytes = 256;
    return lay;
}

int launch_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
               void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale, int causal,
               int window, void* workspace, cudaStream_t stream, unsigned* err)
{
    if (d == 128)
        return launch_bwd_d<128>(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, Nq, Nk, scale, causal, window,
                                 workspace, stream, err);
    if (d == 64)
        return launch_bwd_d<64>(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, Nq, Nk, scale, causal, window,
                                workspace, stream, err);
    return kErrUnsupported;
}

}  // namespace attn
