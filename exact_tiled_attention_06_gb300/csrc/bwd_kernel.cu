// bwd_kernel.cu -- attention backward for sm_103a: dQ, dK, dV from Q, K, V, O, dO and
// the forward's per-row lse, with the score tiles recomputed.
//
// Pages: "Modern attention kernels", "Backward pass recomputes scores" (storing P would
// cost quadratic memory: a per-row statistic is kept and the score tiles are formed
// again); "Flash attention and IO-aware attention", the backward-pass paragraph (two
// numbers per row kept, probabilities rebuilt tile by tile); "Attention kernels", the
// rematerialisation passage (extra FLOPs traded for memory traffic).
//
// For a row i and key j (P_ij = 2^(s_ij * scale * log2e - lse_i * log2e), 0 if masked):
//   dV_j = sum_i P_ij dO_i          dP_ij = dO_i . v_j          D_i = dO_i . O_i
//   dS_ij = P_ij (dP_ij - D_i)      dQ_i = scale sum_j dS_ij k_j      dK_j = scale sum_i dS_ij q_i
// (D_i equals sum_j P_ij dP_ij because O_i = sum_j P_ij v_j.)
//
// Three launches:
//   attn_bwd_prep      D_i = rowsum(dO o O) in fp32, and a zeroed fp32 dQ accumulator
//   attn_bwd_sm103     one CTA per (128-key tile, kv head): dK, dV accumulate in TMEM
//                      over every query head of the group and every 128-query tile that
//                      sees the keys; each tile's dQ partial is added to the accumulator
//   attn_bwd_dq_out    dQ = scale * accumulator, rounded to bf16
//
// Main kernel, per 128-query tile t (keys are the TMEM lanes of every product but dQ^T):
//   S^T  = K Q^T        (128 x 128)       dP^T = V dO^T       (128 x 128)
//   P^T, dS^T           element-wise, written back to TMEM as bf16 (A operands), dS^T
//                       also to shared memory (B operand of dQ^T)
//   dV  += P^T dO       dK += dS^T Q      dQ^T = K^T dS^T     (d x 128, lane = d)
// Every product has N = 128: a tcgen05.mma instruction costs nearly the same for N = 64,
// so narrower tiles would halve the tensor throughput.
// Roles (448 threads):
//   warps 0-7   softmax: warp w owns TMEM lane quadrant w % 4 (32 keys) and the query
//               half w / 4 (queries [64 h, 64 h + 64) of the tile)
//   warps 8-11  dQ readout: copy the tile's dQ^T (lane = d) from TMEM into the tile's Q/dO
//               stage (free once every MMA of the tile is done), release the TMEM, and
//               have one thread add the staged tile to the fp32 accumulator with TMA
//               tensor reductions; the stage returns to the producer when the TMA unit has
//               read it. (Per-thread atomic adds would occupy the SM's memory-instruction
//               queue while L2 drains them and stall the softmax's exp and shared loads.)
//   warp  12    TMEM allocation and tcgen05 MMA issue (one thread)
//   warp  13    TMA producer (one thread): K and V once, Q and dO per tile (2 stages)
// TMEM columns: S^T in [0,128) and dP^T in [128,256); the softmax packs P^T (bf16) into
// [64 h, 64 h + 32) and dS^T into [64 h + 32, 64 h + 64) (query half h), and dQ^T then
// lands in [128,256). dV and dK accumulate in [256, 256 + d) and [256 + d, 256 + 2 d).
// MMA issue order: dV(t) as soon as P^T(t) is written (while dS^T(t) is computed),
// dK(t), dQ^T(t), S^T(t + 1) (once dV(t), dK(t) are done), dP^T(t + 1) (once dQ^T(t)
// has been copied out): the tensor pipe stays busy while the softmax of tile t + 1
// computes P^T from S^T(t + 1) during dP^T(t + 1).
// For d = 64 the dQ^T product still has M = 128: rows 64..127 of its A operand point at
// a zero-filled block of shared memory, and the readout skips those lanes.
#include <climits>
#include <cmath>
#include <cstdint>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int BQ = 128;  // queries per tile
constexpr int BK = 128;  // keys per CTA (TMEM lanes of S^T, dP^T, dV, dK)
constexpr int kSoftmaxThreads = 256;  // warps 0-7
constexpr int kReadoutWarp0 = 8;      // warps 8-11
constexpr int kMmaWarpB = 12;
constexpr int kLoadWarpB = 13;
constexpr int kBwdThreads = 14 * 32;
constexpr int kStagesB = 2;           // Q / dO stages
constexpr float kLog2eB = 1.4426950408889634f;

template <int D>
struct BwdCfg {
    static constexpr int kBoxes = D / 64;               // 64-column (128-byte) boxes
    static constexpr int kBox = 128 * 128;              // one box of a 128-row tile: 16 KB
    static constexpr int kTile = kBoxes * kBox;         // K, V, Q or dO tile
    static constexpr int kKOff = 0;                     // K tile (resident)
    static constexpr int kVOff = kTile;                 // V tile (resident)
    static constexpr int kZOff = 2 * kTile;             // d = 64: zeros standing in for d 64..127
    static constexpr int kZBytes = D == 64 ? kBox : 0;
    static constexpr int kStageOff = kZOff + kZBytes;   // stage s: Q at + s * kStageBytes, dO after Q
    static constexpr int kStageBytes = 2 * kTile;
    static constexpr int kDSOff = kStageOff + kStagesB * kStageBytes;  // dS^T: 128 keys x 128 queries
    static constexpr int kDSBytes = 2 * kBox;           // two 64-query blocks of 16 KB
    static constexpr int kVecOff = kDSOff + kDSBytes;   // two buffers: lse * log2(e) [128], D [128]
    static constexpr int kBarOff = kVecOff + 2 * 2 * BQ * 4;
    static constexpr int kNumBars = 16;
    // dQ^T staging inside a consumed Q/dO stage: box b (d in [32 b, 32 b + 32)) is 128
    // query rows of 32 fp32 (128 bytes), 16 KB per box
    static constexpr int kStgBox = 128 * 32 * 4;
    static_assert((D / 32) * kStgBox <= kStageBytes, "dQ^T staging must fit in one stage");
    static constexpr int kHolderOff = kBarOff + 8 * kNumBars;
    static constexpr int kAbortOff = kHolderOff + 4;
    static constexpr int kUsedBytes = kAbortOff + 4;
    // Dynamic shared memory: what is used plus room to align the base to 1024 bytes
    // (capped at the 227 KB a block may have; the kernel checks that the aligned layout
    // fits), at least ~120 KB so that two blocks never share an SM (each takes all of TMEM).
    static constexpr int kMaxDynSmem = 227 * 1024;
    static constexpr int kPadded = (kUsedBytes + 1024) < kMaxDynSmem ? (kUsedBytes + 1024) : kMaxDynSmem;
    static constexpr int kSmemBytes = kPadded > 122880 ? kPadded : 122880;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kSCol = 0, kDPCol = 128;  // S^T, dP^T (then dQ^T)
    static constexpr uint32_t kDVCol = 256, kDKCol = 256 + D;
    static_assert(kUsedBytes <= kMaxDynSmem, "shared memory budget");
    static_assert(kDKCol + D <= kTmemCols, "TMEM budget");
    static_assert(kStageOff % 1024 == 0 && kDSOff % 1024 == 0 && kZOff % 1024 == 0,
                  "swizzled tiles need 1024-byte alignment");
};

// Barrier slots (8 bytes each) from kBarOff. Per-tile barriers complete once per tile.
enum BwdBar : uint32_t {
    kBarKV = 0,          // K and V landed
    kBarStFull = 1,      // + s: stage s of Q and dO landed (2)
    kBarStFree = 3,      // + s: stage s may be reloaded: its tile's MMAs are done and the
                         //      staged dQ^T it then held has been read by the TMA unit (2)
    kBarSFull = 5,       // S^T in TMEM
    kBarDPFull = 6,      // dP^T in TMEM (and every earlier MMA done)
    kBarPReady = 7,      // P^T written to TMEM (256 arrivals)
    kBarDSReady = 8,     // dS^T written to TMEM and shared memory (256 arrivals)
    kBarPDSDone = 9,     // dV and dK of the tile done: the S^T columns may be rewritten
    kBarDQFull = 10,     // dQ^T in TMEM
    kBarDQRead = 11,     // dQ^T copied to registers (128 arrivals)
    kBarVec = 12,        // + u: statistics buffer u written (2; 256 arrivals)
    kBarFin = 14,        // every MMA done
    kBarRoSync = 15,     // dQ^T staged in shared memory (128 arrivals)
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
__global__ void __launch_bounds__(kBwdThreads, 1)  // 14 warps: at most 128 registers a thread
    attn_bwd_sm103(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_dq, const BwdParams p)
{
    using C = BwdCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    // The 1024-byte aligned layout must fit in what was requested (uniform for the block).
    if (static_cast<int>(smem - smem_raw) + C::kUsedBytes > C::kSmemBytes) {
        if (threadIdx.x == 0) report_error(p.err, kDevErrBounds);
        return;
    }
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
    const int n_it = p.G * (qhi - qlo);  // tiles: (query head of the group, 128-query tile)

    const uint32_t bar0 = sb + C::kBarOff;
#define BWD_BAR(i) (bar0 + 8u * static_cast<uint32_t>(i))
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kHolderOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbortOff);

    if (threadIdx.x == 0) {
        mbar_init(BWD_BAR(kBarKV), 1);
        for (int s = 0; s < kStagesB; ++s) {
            mbar_init(BWD_BAR(kBarStFull + s), 1);
            mbar_init(BWD_BAR(kBarStFree + s), 1);
        }
        mbar_init(BWD_BAR(kBarVec), kSoftmaxThreads);
        mbar_init(BWD_BAR(kBarVec + 1), kSoftmaxThreads);
        mbar_init(BWD_BAR(kBarSFull), 1);
        mbar_init(BWD_BAR(kBarDPFull), 1);
        mbar_init(BWD_BAR(kBarPReady), kSoftmaxThreads);
        mbar_init(BWD_BAR(kBarDSReady), kSoftmaxThreads);
        mbar_init(BWD_BAR(kBarPDSDone), 1);
        mbar_init(BWD_BAR(kBarDQFull), 1);
        mbar_init(BWD_BAR(kBarDQRead), 128);
        mbar_init(BWD_BAR(kBarFin), 1);
        mbar_init(BWD_BAR(kBarRoSync), 128);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if constexpr (C::kZBytes > 0) {
        // zeros read by the tensor cores as rows 64..127 of the dQ^T product's A operand
        for (int i = threadIdx.x; i < C::kZBytes / 16; i += kBwdThreads)
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(sb + C::kZOff + 16 * i), "r"(0u)
                         : "memory");
        fence_proxy_async_smem();
    }
    if (warp == kMmaWarpB) {
        tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t sK = sb + C::kKOff, sV = sb + C::kVOff;
    const uint32_t sStage = sb + C::kStageOff, sDS = sb + C::kDSOff;

    if (warp == kLoadWarpB) {
        // ================================================================ producer
        if (lane == 0 && n_it > 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_do);
            mbar_arrive_expect_tx(BWD_BAR(kBarKV), 2 * C::kTile);
#pragma unroll
            for (int x = 0; x < C::kBoxes; ++x) {
                tma_load_3d(sK + x * C::kBox, &tm_k, BWD_BAR(kBarKV), 64 * x, kt * BK, bk);
                tma_load_3d(sV + x * C::kBox, &tm_v, BWD_BAR(kBarKV), 64 * x, kt * BK, bk);
            }
            int it = 0;  // tile it uses stage it % 2 for the (it / 2)-th time
            for (int gq = 0; gq < p.G; ++gq) {
                const int zq = b * p.Hq + hkv * p.G + gq;
                for (int qt = qlo; qt < qhi; ++qt, ++it) {
                    const int s = it & 1;
                    if (it >= kStagesB &&
                        !mbar_wait(BWD_BAR(kBarStFree + s), ((it >> 1) - 1) & 1, abort_flag, p.err))
                        goto producer_done;
                    const uint32_t full = BWD_BAR(kBarStFull + s);
                    mbar_arrive_expect_tx(full, 2 * C::kTile);
                    const uint32_t so = sStage + s * C::kStageBytes;
#pragma unroll
                    for (int x = 0; x < C::kBoxes; ++x) {
                        tma_load_3d(so + x * C::kBox, &tm_q, full, 64 * x, qt * BQ, zq);
                        tma_load_3d(so + C::kTile + x * C::kBox, &tm_do, full, 64 * x, qt * BQ, zq);
                    }
                }
            }
        producer_done:
            // never leave while a copy into this block's shared memory is in flight: wait
            // for K, V and for the last tile issued on each stage
            mbar_wait(BWD_BAR(kBarKV), 0, nullptr, p.err);
            for (int t = it > kStagesB ? it - kStagesB : 0; t < it; ++t)
                mbar_wait(BWD_BAR(kBarStFull + (t & 1)), (t >> 1) & 1, nullptr, p.err);
        }
    } else if (warp == kMmaWarpB) {
        // ================================================================ MMA issue
        if (lane == 0 && n_it > 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(BK, BQ, false, false);   // S^T, dP^T
            constexpr uint32_t idesc_g = idesc_bf16_f32(BK, D, false, true);     // dV, dK (A in TMEM)
            constexpr uint32_t idesc_q = idesc_bf16_f32(128, BQ, true, true);    // dQ^T (M = 128 d rows)
            // K-major operands of S^T and dP^T: 16-column k steps inside 128-byte rows, a
            // new 16 KB box every 64 columns
            const uint64_t kd = smem_desc_sw128(sK, 16, 1024), vd = smem_desc_sw128(sV, 16, 1024);
            const uint64_t st_k = smem_desc_sw128(sStage, 16, 1024);           // stage 0, K-major
            // MN-major operands: 16 rows of the reduction dimension (2048 bytes) per k step,
            // the two 64-wide halves of the other dimension one box apart
            const uint64_t st_mn = smem_desc_sw128(sStage, C::kBox, 1024);     // stage 0, MN-major
            const uint64_t k_mn = smem_desc_sw128(sK, D == 128 ? C::kBox : C::kZOff - C::kKOff, 1024);
            const uint64_t ds_mn = smem_desc_sw128(sDS, C::kBox, 1024);
            const uint32_t tS = tmem + C::kSCol, tDP = tmem + C::kDPCol;

            auto issue_s = [&](int t) {  // S^T(t) = K Q(t)^T
                const uint64_t qd = st_k + static_cast<uint64_t>(((t & 1) * C::kStageBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = static_cast<uint64_t>(((kk >> 2) * C::kBox + (kk & 3) * 32) >> 4);
                    mma_ss(tS, kd + off, qd + off, idesc_s, kk > 0 ? 1u : 0u);
                }
                tc_commit(BWD_BAR(kBarSFull));
            };
            auto issue_dp = [&](int t) {  // dP^T(t) = V dO(t)^T
                const uint64_t dod = st_k + static_cast<uint64_t>(((t & 1) * C::kStageBytes + C::kTile) >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = static_cast<uint64_t>(((kk >> 2) * C::kBox + (kk & 3) * 32) >> 4);
                    mma_ss(tDP, vd + off, dod + off, idesc_s, kk > 0 ? 1u : 0u);
                }
                tc_commit(BWD_BAR(kBarDPFull));
            };

            bool ok = mbar_wait(BWD_BAR(kBarKV), 0, abort_flag, p.err) &&
                      mbar_wait(BWD_BAR(kBarStFull), 0, abort_flag, p.err);
            if (ok) {
                tc_fence_after();
                issue_s(0);
                issue_dp(0);
            }
            for (int t = 0; t < n_it && ok; ++t) {
                const uint32_t tp = t & 1;
                const int s = t & 1;
                const uint64_t qm = st_mn + static_cast<uint64_t>((s * C::kStageBytes) >> 4);
                const uint64_t dom = qm + static_cast<uint64_t>(C::kTile >> 4);
                // dV += P^T dO as soon as P^T is written (16 queries per k step: query half
                // kk / 4, its P^T at 64 h, dS^T at 64 h + 32)
                if (!mbar_wait(BWD_BAR(kBarPReady), tp, abort_flag, p.err)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < BQ / 16; ++kk)
                    mma_ts(tmem + C::kDVCol, tS + 64 * (kk >> 2) + 8 * (kk & 3),
                           dom + static_cast<uint64_t>(kk * 128), idesc_g, (t > 0 || kk > 0) ? 1u : 0u);
                // dK += dS^T Q
                if (!mbar_wait(BWD_BAR(kBarDSReady), tp, abort_flag, p.err)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < BQ / 16; ++kk)
                    mma_ts(tmem + C::kDKCol, tS + 64 * (kk >> 2) + 32 + 8 * (kk & 3),
                           qm + static_cast<uint64_t>(kk * 128), idesc_g, (t > 0 || kk > 0) ? 1u : 0u);
                tc_commit(BWD_BAR(kBarPDSDone));      // P^T, dS^T (the S^T columns) are no longer read
                // dQ^T = K^T dS^T into the dP^T columns (the softmax has read dP^T)
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    mma_ss(tDP, k_mn + static_cast<uint64_t>(kk * 128), ds_mn + static_cast<uint64_t>(kk * 128),
                           idesc_q, kk > 0 ? 1u : 0u);
                tc_commit(BWD_BAR(kBarDQFull));
                if (t + 1 < n_it) {
                    // S^T(t+1) once dV(t), dK(t) are done; dP^T(t+1) once dQ^T(t) is copied out
                    if (!mbar_wait(BWD_BAR(kBarStFull + ((t + 1) & 1)), ((t + 1) >> 1) & 1, abort_flag, p.err)) break;
                    if (!mbar_wait(BWD_BAR(kBarPDSDone), tp, abort_flag, p.err)) break;
                    tc_fence_after();
                    issue_s(t + 1);
                    if (!mbar_wait(BWD_BAR(kBarDQRead), tp, abort_flag, p.err)) break;
                    tc_fence_after();
                    issue_dp(t + 1);
                }
            }
            tc_commit(BWD_BAR(kBarFin));
            mbar_wait(BWD_BAR(kBarFin), 0, nullptr, p.err);
        }
    } else if (warp < kReadoutWarp0) {
        // ================================================================ softmax warps 0-7
        const int tid = threadIdx.x;
        const int qd = warp & 3;                  // TMEM lane quadrant
        const int hh = warp >> 2;                 // query half: queries [64 hh, 64 hh + 64)
        const int krow = 32 * qd + lane;          // key row in the tile = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
        const long long delta = static_cast<long long>(p.Nk) - p.Nq;
        // Queries allowed to see this thread's key j: i in [i_min, i_max] (causal:
        // j <= i + delta; window w: j >= i + delta - w; inside the sequence).
        const long long j = static_cast<long long>(kt) * BK + krow;
        long long i_min = 0, i_max = static_cast<long long>(p.Nq) - 1;
        if (p.causal && j - delta > i_min) i_min = j - delta;
        if (p.window >= 0 && j - delta + p.window < i_max) i_max = j - delta + p.window;
        if (j >= p.Nk) i_max = -1;
        const uint32_t tS = tmem + lane_base + C::kSCol + 64 * hh;    // this half's S^T, then P^T | dS^T
        const uint32_t tDP = tmem + lane_base + C::kDPCol + 64 * hh;  // this half's dP^T
        const uint32_t ds_row = sDS + hh * C::kBox + krow * 128;      // this key's row of this half's dS^T
        bool ok = true;
        int it = 0;
        for (int gq = 0; gq < p.G && ok; ++gq) {
            const long long rowbase = (static_cast<long long>(b) * p.Hq + hkv * p.G + gq) * p.Nq;
            for (int qt = qlo; qt < qhi; ++qt, ++it) {
                const uint32_t tp = it & 1;               // per-tile barrier parity
                const int u = it & 1;                     // statistics buffer
                const long long q0 = static_cast<long long>(qt) * BQ;
                // ---- -lse * log2(e) and -D of the tile's 128 queries. The buffer was last read
                // two tiles ago; every thread arrived on the previous tile's barrier after
                // that read, and this thread has passed that barrier.
                float* vec = reinterpret_cast<float*>(smem + C::kVecOff) + u * 2 * BQ;
                if (tid < BQ) {
                    const long long q = q0 + tid;
                    float l2 = INFINITY, dd = 0.0f;
                    if (q < p.Nq) {
                        l2 = p.lse[rowbase + q] * kLog2eB;
                        dd = p.dvec[rowbase + q];
                    }
                    vec[tid] = -l2;
                    vec[BQ + tid] = -dd;
                }
                mbar_arrive(BWD_BAR(kBarVec + u));
                // (wait results are made warp-uniform: the tcgen05 loads and stores below are
                // warp-collective and must be reached by all 32 lanes or by none)
                if (!__all_sync(0xffffffffu, mbar_wait(BWD_BAR(kBarVec + u), (it >> 1) & 1, abort_flag, p.err))) {
                    ok = false;
                    break;
                }
                const long long c0q = q0 + 64 * hh;  // first query of this half
                const int c_lo = static_cast<int>(max(-1ll, min(64ll, i_min - c0q)));
                const int c_hi = static_cast<int>(max(-1ll, min(64ll, i_max - c0q)));
                const bool full = c_lo <= 0 && c_hi >= 63;
                const float* nl2v = vec + 64 * hh;      // -lse * log2(e) of this half's queries
                const float* nddv = vec + BQ + 64 * hh;  // -D of this half's queries
                // off the diagonal (and inside a window) every key of the warp sees every query
                // of the half: no per-element mask
                const bool all_full = __all_sync(0xffffffffu, full);
                // ---- P^T = exp2(S^T * scale * log2e - lse * log2e), masked, into TMEM as bf16
                if (!__all_sync(0xffffffffu, mbar_wait(BWD_BAR(kBarSFull), tp, abort_flag, p.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // (exponent and product in paired fp32: one instruction per two elements)
                const uint64_t c2 = f2pack(p.scale_log2, p.scale_log2);
                float pv[64];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t sr[32];
                    tmem_ld32(tS + 32 * c, sr);
                    tmem_ld_wait_dep32(sr);
                    float nl2[32];  // read here, not hoisted (keeps registers for the products)
#pragma unroll
                    for (int k = 0; k < 32; k += 4)
                        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                     : "=f"(nl2[k]), "=f"(nl2[k + 1]), "=f"(nl2[k + 2]), "=f"(nl2[k + 3])
                                     : "r"(smem_u32(nl2v + 32 * c + k)));
#pragma unroll
                    for (int k = 0; k < 32; k += 2) {
                        float x0, x1;
                        f2unpack(f2fma(f2pack(__uint_as_float(sr[k]), __uint_as_float(sr[k + 1])), c2,
                                       f2pack(nl2[k], nl2[k + 1])),
                                 x0, x1);
                        pv[32 * c + k] = ex2_approx(x0);
                        pv[32 * c + k + 1] = ex2_approx(x1);
                    }
                    if (!all_full) {
#pragma unroll
                        for (int k = 0; k < 32; ++k) {
                            const int q = 32 * c + k;
                            pv[q] = (q >= c_lo && q <= c_hi) ? pv[q] : 0.0f;
                        }
                    }
                }
                {
                    uint32_t pp[32];
#pragma unroll
                    for (int k = 0; k < 32; ++k) pp[k] = pack_bf16x2(pv[2 * k], pv[2 * k + 1]);
                    tmem_st32(tS, pp);  // over S^T columns this half has read
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(BWD_BAR(kBarPReady));
                // ---- dS^T = P^T (dP^T - D), 32 queries at a time, into TMEM (bf16) and into
                // shared memory as the MN-major B operand of dQ^T: key krow is a 128-byte row
                // of this half's 64 queries, its 16-byte chunks XOR-swizzled with (krow mod 8)
                if (!__all_sync(0xffffffffu, mbar_wait(BWD_BAR(kBarDPFull), tp, abort_flag, p.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t pd[16];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {  // 16 columns of dP^T at a time keep registers low
                        uint32_t dr[16];
                        tmem_ld16(tDP + 32 * c + 16 * e, dr);
                        tmem_ld_wait_dep16(dr);
                        float ndd[16];  // -D of these 16 queries, read here (not hoisted)
#pragma unroll
                        for (int k = 0; k < 16; k += 4)
                            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                         : "=f"(ndd[k]), "=f"(ndd[k + 1]), "=f"(ndd[k + 2]), "=f"(ndd[k + 3])
                                         : "r"(smem_u32(nddv + 32 * c + 16 * e + k)));
#pragma unroll
                        for (int k = 0; k < 16; k += 2) {
                            const int q = 32 * c + 16 * e + k;
                            float d0, d1;
                            f2unpack(f2mul(f2pack(pv[q], pv[q + 1]),
                                           f2add(f2pack(__uint_as_float(dr[k]), __uint_as_float(dr[k + 1])),
                                                 f2pack(ndd[k], ndd[k + 1]))),
                                     d0, d1);
                            pd[8 * e + k / 2] = pack_bf16x2(d0, d1);
                        }
                    }
                    tmem_st16(tS + 32 + 16 * c, pd);  // over S^T columns this half has read
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const uint32_t addr = ds_row + (((4 * c + cc) ^ (krow & 7)) << 4);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pd[4 * cc]),
                                     "r"(pd[4 * cc + 1]), "r"(pd[4 * cc + 2]), "r"(pd[4 * cc + 3])
                                     : "memory");
                    }
                }
                tmem_st_wait();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(BWD_BAR(kBarDSReady));
            }
        }
        // ---- epilogue once every MMA is done: warps 0-3 write dV, warps 4-7 write dK
        // (lane = key). Every lane loads (the TMEM loads are warp-collective); only lanes
        // with a key inside the sequence store.
        const bool have = n_it > 0 ? mbar_wait(BWD_BAR(kBarFin), 0, nullptr, p.err) : true;
        tc_fence_after();
        if (__all_sync(0xffffffffu, have && ok && *abort_flag == 0)) {
            const long long obase = ((static_cast<long long>(b) * p.Hkv + hkv) * p.Nk + j) * D;
            __nv_bfloat16* out = hh == 0 ? p.dv : p.dk;
            const float mul = hh == 0 ? 1.0f : p.scale;
            const uint32_t col = hh == 0 ? C::kDVCol : C::kDKCol;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t r[32];
                __syncwarp();
                if (n_it > 0) {
                    tmem_ld32(tmem + lane_base + col + c0, r);
                    tmem_ld_wait_dep32(r);
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k) r[k] = 0u;
                }
                if (j < p.Nk) {
                    uint4* dst = reinterpret_cast<uint4*>(out + obase + c0);
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(r[8 * m + 0]) * mul, __uint_as_float(r[8 * m + 1]) * mul);
                        w.y = pack_bf16x2(__uint_as_float(r[8 * m + 2]) * mul, __uint_as_float(r[8 * m + 3]) * mul);
                        w.z = pack_bf16x2(__uint_as_float(r[8 * m + 4]) * mul, __uint_as_float(r[8 * m + 5]) * mul);
                        w.w = pack_bf16x2(__uint_as_float(r[8 * m + 6]) * mul, __uint_as_float(r[8 * m + 7]) * mul);
                        dst[m] = w;
                    }
                }
            }
        }
    } else {
        // ================================================================ dQ readout warps 8-11
        const int qd = warp & 3;                  // TMEM lane quadrant = d rows [32 qd, 32 qd + 32)
        const uint32_t src = tmem + (static_cast<uint32_t>(32 * qd) << 16) + C::kDPCol;
        const bool active = 32 * qd < D;          // d = 64: lanes 64..127 hold the zero padding
        const bool leader = threadIdx.x == 32 * kReadoutWarp0;
        int it = 0;
        bool ok = true;
        for (int gq = 0; gq < p.G && ok; ++gq) {
            const int zq = b * p.Hq + hkv * p.G + gq;
            for (int qt = qlo; qt < qhi; ++qt, ++it) {
                const int s = it & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(BWD_BAR(kBarDQFull), it & 1, abort_flag, p.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // Every MMA of this tile is done (the commit behind dq_full covers them), so
                // its Q/dO stage is free: stage dQ^T there, box qd, row = query, column = lane.
                const uint32_t stg = sStage + s * C::kStageBytes;
                const uint32_t stg_lane = stg + qd * C::kStgBox + 4 * lane;
#pragma unroll 1
                for (int c = 0; c < BQ; c += 32) {
                    uint32_t r[32];
                    __syncwarp();
                    tmem_ld32(src + c, r);
                    tmem_ld_wait_dep32(r);
                    if (c + 32 == BQ) {
                        tc_fence_before();
                        mbar_arrive(BWD_BAR(kBarDQRead));  // the dP^T / dQ^T columns may be rewritten
                    }
                    if (active) {
#pragma unroll
                        for (int m = 0; m < 32; ++m)
                            asm volatile("st.shared.b32 [%0], %1;" ::"r"(stg_lane + (c + m) * 128), "r"(r[m])
                                         : "memory");
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(BWD_BAR(kBarRoSync));
                if (leader) {
                    // one thread: add the staged boxes to the accumulator (rows past Nq are
                    // clipped by the tensor map), then hand the stage back to the producer
                    // once the TMA unit has read it
                    if (!mbar_wait(BWD_BAR(kBarRoSync), it & 1, abort_flag, p.err)) {
                        ok = false;
                    } else {
#pragma unroll
                        for (int x = 0; x < D / 32; ++x)
                            tma_reduce_add_3d(&tm_dq, stg + x * C::kStgBox, 32 * x, qt * BQ, zq);
                        bulk_commit_group();
                        bulk_wait_group_read0();
                        mbar_arrive(BWD_BAR(kBarStFree + s));
                    }
                }
                if (!__all_sync(0xffffffffu, ok)) break;
            }
        }
        if (leader) bulk_wait_group0();  // every reduction performed before the block exits
    }
#undef BWD_BAR

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
        {
            const uint32_t box[3] = {64u, static_cast<uint32_t>(BK), 1u};
            const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Nk),
                                      static_cast<uint64_t>(B) * Hkv};
            const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(Nk) * D * 2};
            int rc = encode_bf16_map(&tk, k, 3, dims, strides, box);
            if (rc != kOk) return rc;
            rc = encode_bf16_map(&tv, v, 3, dims, strides, box);
            if (rc != kOk) return rc;
        }
        CUtensorMap tdq;
        if (Nq > 0) {
            const uint32_t box[3] = {64u, static_cast<uint32_t>(BQ), 1u};
            const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Nq),
                                      static_cast<uint64_t>(B) * Hq};
            const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(Nq) * D * 2};
            int rc = encode_bf16_map(&tq, q, 3, dims, strides, box);
            if (rc != kOk) return rc;
            rc = encode_bf16_map(&tdo, dout, 3, dims, strides, box);
            if (rc != kOk) return rc;
            // fp32 dQ accumulator [B][Hq][Nq][d], reduced into box by box (32 d x 128 queries)
            const uint32_t box_dq[3] = {32u, static_cast<uint32_t>(BQ), 1u};
            const uint64_t strides_dq[2] = {static_cast<uint64_t>(D) * 4, static_cast<uint64_t>(Nq) * D * 4};
            rc = encode_f32_map(&tdq, dq_acc, 3, dims, strides_dq, box_dq);
            if (rc != kOk) return rc;
        } else {
            // No queries: no query tile is ever loaded and every block writes zero dK, dV.
            tq = tk;
            tdo = tk;
            tdq = tk;
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
        attn_bwd_sm103<D><<<static_cast<unsigned>(grid), kBwdThreads, C::kSmemBytes, stream>>>(tq, tk, tv, tdo, tdq, prm);
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
