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
//                      over every query head of the group and every 64-query step that
//                      sees the keys; each step's dQ partial is added to the accumulator
//   attn_bwd_dq_out    dQ = scale * accumulator, rounded to bf16
//
// Main kernel, per 64-query step j (keys are the TMEM lanes of every product but dQ^T):
//   S^T  = K Q^T        (128 x 64)        dP^T = V dO^T       (128 x 64)
//   P^T, dS^T           element-wise, written back to TMEM as bf16 (A operands), dS^T
//                       also to shared memory (B operand of dQ^T)
//   dV  += P^T dO       dK += dS^T Q      dQ^T = K^T dS^T     (d x 64, lane = d)
// Roles (448 threads):
//   warps 0-7   softmax: warp w owns TMEM lane quadrant w % 4 (32 keys) and the query
//               group w / 4 (queries [32 g, 32 g + 32) of the step)
//   warps 8-11  dQ readout: copy the step's dQ^T tile (lane = d) from TMEM to registers,
//               release it, then add it to the fp32 accumulator; each warp instruction
//               covers 32 consecutive d of one query (one 128-byte line)
//   warp  12    TMEM allocation and tcgen05 MMA issue (one thread)
//   warp  13    TMA producer (one thread): K and V once, Q and dO per step (3 stages)
// TMEM columns: two step buffers (step j uses buffer j % 2, 128 columns at 128 (j % 2)):
// S^T in its first 64 columns, dP^T in the last 64. The softmax packs P^T and dS^T (bf16)
// into the S^T half (query group g: P^T at 32 g, dS^T at 32 g + 16), and dQ^T then lands
// in the dP^T half. dV and dK accumulate in [256, 256 + d) and [256 + d, 256 + 2 d).
// The MMA thread issues S^T and dP^T of step j + 1 before the gradient products of step
// j, so that each step's softmax overlaps the tensor work of its neighbours.
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

constexpr int BQ = 64;   // queries per step
constexpr int BK = 128;  // keys per CTA (TMEM lanes of S^T, dP^T, dV, dK)
constexpr int kSoftmaxThreads = 256;  // warps 0-7
constexpr int kReadoutWarp0 = 8;      // warps 8-11
constexpr int kMmaWarpB = 12;
constexpr int kLoadWarpB = 13;
constexpr int kBwdThreads = 14 * 32;
constexpr int kStagesB = 3;           // Q / dO stages
constexpr float kLog2eB = 1.4426950408889634f;

template <int D>
struct BwdCfg {
    static constexpr int kBoxes = D / 64;               // 64-column (128-byte) boxes
    static constexpr int kKBox = BK * 128;              // one box of the K or V tile: 16 KB
    static constexpr int kKVTile = kBoxes * kKBox;
    static constexpr int kQBox = BQ * 128;              // one box of a Q or dO step tile: 8 KB
    static constexpr int kQTile = kBoxes * kQBox;
    static constexpr int kKOff = 0;                     // K tile (resident)
    static constexpr int kVOff = kKVTile;               // V tile (resident)
    static constexpr int kZOff = 2 * kKVTile;           // d = 64: zeros standing in for d 64..127
    static constexpr int kZBytes = D == 64 ? kKBox : 0;
    static constexpr int kStageOff = kZOff + kZBytes;   // stage s: Q at + s * kStageBytes, dO after Q
    static constexpr int kStageBytes = 2 * kQTile;
    static constexpr int kDSOff = kStageOff + kStagesB * kStageBytes;  // dS^T, two buffers
    static constexpr int kDSBytes = BK * 128;           // 128 keys x 64 queries x bf16
    static constexpr int kVecOff = kDSOff + 2 * kDSBytes;  // two buffers: lse * log2(e) [64], D [64]
    static constexpr int kBarOff = kVecOff + 2 * 2 * BQ * 4;
    static constexpr int kNumBars = 20;
    static constexpr int kHolderOff = kBarOff + 8 * kNumBars;
    static constexpr int kAbortOff = kHolderOff + 4;
    static constexpr int kUsedBytes = kAbortOff + 4;
    // Dynamic shared memory: what is used plus room to align the base to 1024 bytes;
    // at least ~120 KB so that two blocks never share an SM (each takes all of TMEM).
    static constexpr int kSmemBytes = (kUsedBytes + 1024) > 122880 ? (kUsedBytes + 1024) : 122880;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kBufCols = 128;           // one step buffer
    static constexpr uint32_t kDPHalf = 64;             // dP^T, then dQ^T, within a buffer
    static constexpr uint32_t kDVCol = 256, kDKCol = 256 + D;
    static_assert(kUsedBytes + 1024 <= 227 * 1024, "shared memory budget");
    static_assert(kDKCol + D <= kTmemCols, "TMEM budget");
    static_assert(kStageOff % 1024 == 0 && kDSOff % 1024 == 0 && kZOff % 1024 == 0,
                  "swizzled tiles need 1024-byte alignment");
};

// Barrier slots (8 bytes each) from kBarOff.
enum BwdBar : uint32_t {
    kBarKV = 0,          // K and V landed
    kBarStFull = 1,      // + s: stage s of Q and dO landed (3)
    kBarStEmpty = 4,     // + s: every MMA reading stage s is done (3)
    kBarSFull = 7,       // + b: S^T of buffer b in TMEM (2)
    kBarDPFull = 9,      // + b: dP^T of buffer b in TMEM (2)
    kBarPReady = 11,     // + b: P^T, dS^T of buffer b written, TMEM and shared (2; 256 arrivals)
    kBarDQFull = 13,     // + b: dQ^T of buffer b in TMEM (2)
    kBarDQRead = 15,     // + b: dQ^T of buffer b copied to registers (2; 128 arrivals)
    kBarVec = 17,        // + u: statistics buffer u written (2; 256 arrivals)
    kBarFin = 19,        // every MMA done
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
    // tiles that see the most query steps (the first key tiles) are scheduled first.
    const int n_bk = p.B * p.Hkv;
    const int kt = static_cast<int>(blockIdx.x) / n_bk;
    const int bk = static_cast<int>(blockIdx.x) % n_bk;  // batch * Hkv + kv head
    const int b = bk / p.Hkv;
    const int hkv = bk % p.Hkv;
    int qlo, qhi;
    query_tile_range(p, kt, qlo, qhi);
    const int n_it = p.G * (qhi - qlo);  // steps: (query head of the group, 64-query tile)

    const uint32_t bar0 = sb + C::kBarOff;
#define BWD_BAR(i) (bar0 + 8u * static_cast<uint32_t>(i))
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kHolderOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbortOff);

    if (threadIdx.x == 0) {
        mbar_init(BWD_BAR(kBarKV), 1);
        for (int s = 0; s < kStagesB; ++s) {
            mbar_init(BWD_BAR(kBarStFull + s), 1);
            mbar_init(BWD_BAR(kBarStEmpty + s), 1);
        }
        for (int u = 0; u < 2; ++u) {
            mbar_init(BWD_BAR(kBarSFull + u), 1);
            mbar_init(BWD_BAR(kBarDPFull + u), 1);
            mbar_init(BWD_BAR(kBarPReady + u), kSoftmaxThreads);
            mbar_init(BWD_BAR(kBarDQFull + u), 1);
            mbar_init(BWD_BAR(kBarDQRead + u), 128);
            mbar_init(BWD_BAR(kBarVec + u), kSoftmaxThreads);
        }
        mbar_init(BWD_BAR(kBarFin), 1);
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
            mbar_arrive_expect_tx(BWD_BAR(kBarKV), 2 * C::kKVTile);
#pragma unroll
            for (int x = 0; x < C::kBoxes; ++x) {
                tma_load_3d(sK + x * C::kKBox, &tm_k, BWD_BAR(kBarKV), 64 * x, kt * BK, bk);
                tma_load_3d(sV + x * C::kKBox, &tm_v, BWD_BAR(kBarKV), 64 * x, kt * BK, bk);
            }
            int it = 0, s = 0, ph = 0;  // step it uses stage s = it % 3 for the (it / 3)-th time, ph = that & 1
            for (int gq = 0; gq < p.G; ++gq) {
                const int zq = b * p.Hq + hkv * p.G + gq;
                for (int qt = qlo; qt < qhi; ++qt, ++it) {
                    // the previous use of this stage must be released (its ((it / 3) - 1)-th release)
                    if (it >= kStagesB && !mbar_wait(BWD_BAR(kBarStEmpty + s), ph ^ 1, abort_flag, p.err))
                        goto producer_done;
                    const uint32_t full = BWD_BAR(kBarStFull + s);
                    mbar_arrive_expect_tx(full, 2 * C::kQTile);
                    const uint32_t so = sStage + s * C::kStageBytes;
#pragma unroll
                    for (int x = 0; x < C::kBoxes; ++x) {
                        tma_load_3d(so + x * C::kQBox, &tm_q, full, 64 * x, qt * BQ, zq);
                        tma_load_3d(so + C::kQTile + x * C::kQBox, &tm_do, full, 64 * x, qt * BQ, zq);
                    }
                    if (++s == kStagesB) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
        producer_done:
            // never leave while a copy into this block's shared memory is in flight: wait
            // for K, V and for the last step issued on each stage
            mbar_wait(BWD_BAR(kBarKV), 0, nullptr, p.err);
            for (int t = it > kStagesB ? it - kStagesB : 0; t < it; ++t)
                mbar_wait(BWD_BAR(kBarStFull + t % kStagesB), (t / kStagesB) & 1, nullptr, p.err);
        }
    } else if (warp == kMmaWarpB) {
        // ================================================================ MMA issue
        if (lane == 0 && n_it > 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(BK, BQ, false, false);   // S^T, dP^T
            constexpr uint32_t idesc_g = idesc_bf16_f32(BK, D, false, true);     // dV, dK (A in TMEM)
            constexpr uint32_t idesc_q = idesc_bf16_f32(128, BQ, true, true);    // dQ^T (M = 128 d rows)
            // K-major operands of S^T and dP^T: 16-column k steps inside 128-byte rows, a
            // new box every 64 columns (16 KB apart in K / V, 8 KB apart in Q / dO)
            const uint64_t kd = smem_desc_sw128(sK, 16, 1024), vd = smem_desc_sw128(sV, 16, 1024);
            // MN-major operands: 16 rows of the reduction dimension (2048 bytes) per k step
            const uint64_t k_mn = smem_desc_sw128(sK, D == 128 ? C::kKBox : C::kZOff - C::kKOff, 1024);
            const uint64_t st_k = smem_desc_sw128(sStage, 16, 1024);         // stage 0, K-major
            const uint64_t st_mn = smem_desc_sw128(sStage, C::kQBox, 1024);  // stage 0, MN-major
            const uint64_t ds_mn = smem_desc_sw128(sDS, C::kDSBytes, 1024);  // dS^T buffer 0
            bool ok = mbar_wait(BWD_BAR(kBarKV), 0, abort_flag, p.err);

            // S^T and dP^T of step j into buffer j % 2
            auto issue_sdp = [&](int j) -> bool {
                const int s = j % kStagesB, bf = j & 1;
                if (!mbar_wait(BWD_BAR(kBarStFull + s), (j / kStagesB) & 1, abort_flag, p.err)) return false;
                // buffer bf last held step j - 2: its dQ^T was copied out (and, by the commit
                // that preceded, every MMA of step j - 2 is complete)
                if (j >= 2 && !mbar_wait(BWD_BAR(kBarDQRead + bf), ((j >> 1) - 1) & 1, abort_flag, p.err))
                    return false;
                tc_fence_after();
                const uint32_t dbuf = tmem + bf * C::kBufCols;
                const uint64_t qd = st_k + static_cast<uint64_t>((s * C::kStageBytes) >> 4);
                const uint64_t dod = qd + static_cast<uint64_t>(C::kQTile >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t oa = static_cast<uint64_t>(((kk >> 2) * C::kKBox + (kk & 3) * 32) >> 4);
                    const uint64_t ob = static_cast<uint64_t>(((kk >> 2) * C::kQBox + (kk & 3) * 32) >> 4);
                    mma_ss(dbuf, kd + oa, qd + ob, idesc_s, kk > 0 ? 1u : 0u);
                }
                tc_commit(BWD_BAR(kBarSFull + bf));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t oa = static_cast<uint64_t>(((kk >> 2) * C::kKBox + (kk & 3) * 32) >> 4);
                    const uint64_t ob = static_cast<uint64_t>(((kk >> 2) * C::kQBox + (kk & 3) * 32) >> 4);
                    mma_ss(dbuf + C::kDPHalf, vd + oa, dod + ob, idesc_s, kk > 0 ? 1u : 0u);
                }
                tc_commit(BWD_BAR(kBarDPFull + bf));
                return true;
            };
            // dV, dK and dQ^T of step j
            auto issue_grad = [&](int j) -> bool {
                const int s = j % kStagesB, bf = j & 1;
                if (!mbar_wait(BWD_BAR(kBarPReady + bf), (j >> 1) & 1, abort_flag, p.err)) return false;
                tc_fence_after();
                const uint32_t dbuf = tmem + bf * C::kBufCols;
                const uint64_t qm = st_mn + static_cast<uint64_t>((s * C::kStageBytes) >> 4);
                const uint64_t dom = qm + static_cast<uint64_t>(C::kQTile >> 4);
                // 16 queries per k step: query group kk / 2, its P^T at 32 g, dS^T at 32 g + 16
#pragma unroll
                for (int kk = 0; kk < BQ / 16; ++kk)
                    mma_ts(tmem + C::kDVCol, dbuf + 32 * (kk >> 1) + 8 * (kk & 1),
                           dom + static_cast<uint64_t>(kk * 128), idesc_g, (j > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < BQ / 16; ++kk)
                    mma_ts(tmem + C::kDKCol, dbuf + 32 * (kk >> 1) + 16 + 8 * (kk & 1),
                           qm + static_cast<uint64_t>(kk * 128), idesc_g, (j > 0 || kk > 0) ? 1u : 0u);
                tc_commit(BWD_BAR(kBarStEmpty + s));  // Q and dO of this stage are no longer read
                const uint64_t dsd = ds_mn + static_cast<uint64_t>((bf * C::kDSBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    mma_ss(dbuf + C::kDPHalf, k_mn + static_cast<uint64_t>(kk * 128),
                           dsd + static_cast<uint64_t>(kk * 128), idesc_q, kk > 0 ? 1u : 0u);
                tc_commit(BWD_BAR(kBarDQFull + bf));
                return true;
            };

            ok = ok && issue_sdp(0);
            for (int j = 0; j < n_it && ok; ++j) {
                if (j + 1 < n_it && !issue_sdp(j + 1)) break;
                if (!issue_grad(j)) break;
            }
            tc_commit(BWD_BAR(kBarFin));
            mbar_wait(BWD_BAR(kBarFin), 0, nullptr, p.err);
        }
    } else if (warp < kReadoutWarp0) {
        // ================================================================ softmax warps 0-7
        const int tid = threadIdx.x;
        const int qd = warp & 3;                  // TMEM lane quadrant
        const int grp = warp >> 2;                // query group: queries [32 grp, 32 grp + 32)
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
        bool ok = true;
        int it = 0;
        for (int gq = 0; gq < p.G && ok; ++gq) {
            const long long rowbase = (static_cast<long long>(b) * p.Hq + hkv * p.G + gq) * p.Nq;
            for (int qt = qlo; qt < qhi; ++qt, ++it) {
                const int bf = it & 1;                 // TMEM step buffer, statistics buffer
                const uint32_t par = (it >> 1) & 1;    // phase parity of this buffer's barriers
                const long long q0 = static_cast<long long>(qt) * BQ;
                // ---- lse * log2(e) and D of the step's 64 queries. The buffer was last read
                // two steps ago; every thread arrived on the previous step's barrier after
                // that read, and this thread has passed that barrier.
                float* vec = reinterpret_cast<float*>(smem + C::kVecOff) + bf * 2 * BQ;
                if (tid < BQ) {
                    const long long q = q0 + tid;
                    float l2 = INFINITY, dd = 0.0f;
                    if (q < p.Nq) {
                        l2 = p.lse[rowbase + q] * kLog2eB;
                        dd = p.dvec[rowbase + q];
                    }
                    vec[tid] = l2;
                    vec[BQ + tid] = dd;
                }
                mbar_arrive(BWD_BAR(kBarVec + bf));
                // (wait results are made warp-uniform: the tcgen05 loads and stores below are
                // warp-collective and must be reached by all 32 lanes or by none)
                if (!__all_sync(0xffffffffu, mbar_wait(BWD_BAR(kBarVec + bf), par, abort_flag, p.err))) {
                    ok = false;
                    break;
                }
                const long long c0q = q0 + 32 * grp;  // first query of this group
                const int c_lo = static_cast<int>(max(-1ll, min(32ll, i_min - c0q)));
                const int c_hi = static_cast<int>(max(-1ll, min(32ll, i_max - c0q)));
                const bool full = c_lo <= 0 && c_hi >= 31;
                const float* l2v = vec + 32 * grp;
                const float* ddv = vec + BQ + 32 * grp;
                const uint32_t dbuf = tmem + lane_base + bf * C::kBufCols;
                // ---- P^T = exp2(S^T * scale * log2e - lse * log2e), masked
                if (!__all_sync(0xffffffffu, mbar_wait(BWD_BAR(kBarSFull + bf), par, abort_flag, p.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t sr[32];
                tmem_ld32(dbuf + 32 * grp, sr);
                tmem_ld_wait_dep32(sr);
                float pv[32];
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const float pe = ex2_approx(fmaf(__uint_as_float(sr[k]), p.scale_log2, -l2v[k]));
                    pv[k] = (full || (k >= c_lo && k <= c_hi)) ? pe : 0.0f;
                }
                // ---- dS^T = P^T (dP^T - D)
                if (!__all_sync(0xffffffffu, mbar_wait(BWD_BAR(kBarDPFull + bf), par, abort_flag, p.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t dr[32];
                tmem_ld32(dbuf + C::kDPHalf + 32 * grp, dr);
                tmem_ld_wait_dep32(dr);
                uint32_t pp[16], pd[16];
#pragma unroll
                for (int k = 0; k < 32; k += 2) {
                    const float d0 = pv[k] * (__uint_as_float(dr[k]) - ddv[k]);
                    const float d1 = pv[k + 1] * (__uint_as_float(dr[k + 1]) - ddv[k + 1]);
                    pp[k / 2] = pack_bf16x2(pv[k], pv[k + 1]);
                    pd[k / 2] = pack_bf16x2(d0, d1);
                }
                // P^T and dS^T into the columns this group has just read (A operands of dV, dK)
                tmem_st16(dbuf + 32 * grp, pp);
                tmem_st16(dbuf + 32 * grp + 16, pd);
                // dS^T into shared memory, the MN-major B operand of dQ^T: key krow is a
                // 128-byte row of 64 queries, this group's 32 queries are its 16-byte chunks
                // 4 grp .. 4 grp + 3, XOR-swizzled with (krow mod 8)
                const uint32_t rbase = sDS + bf * C::kDSBytes + krow * 128;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const uint32_t addr = rbase + (((4 * grp + cc) ^ (krow & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pd[4 * cc]),
                                 "r"(pd[4 * cc + 1]), "r"(pd[4 * cc + 2]), "r"(pd[4 * cc + 3])
                                 : "memory");
                }
                tmem_st_wait();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(BWD_BAR(kBarPReady + bf));
            }
        }
        // ---- epilogue once every MMA is done: warps 0-3 write dV, warps 4-7 write dK
        // (lane = key). Every lane loads (the TMEM loads are warp-collective); only lanes
        // with a key inside the sequence store.
        const bool have = n_it > 0 ? mbar_wait(BWD_BAR(kBarFin), 0, nullptr, p.err) : true;
        tc_fence_after();
        if (__all_sync(0xffffffffu, have && ok && *abort_flag == 0)) {
            const long long obase = ((static_cast<long long>(b) * p.Hkv + hkv) * p.Nk + j) * D;
            __nv_bfloat16* out = grp == 0 ? p.dv : p.dk;
            const float mul = grp == 0 ? 1.0f : p.scale;
            const uint32_t col = grp == 0 ? C::kDVCol : C::kDKCol;
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
        const int drow = 32 * qd + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
        const bool active = 32 * qd < D;          // d = 64: lanes 64..127 hold the zero padding
        int it = 0;
        bool ok = true;
        for (int gq = 0; gq < p.G && ok; ++gq) {
            const long long rowbase = (static_cast<long long>(b) * p.Hq + hkv * p.G + gq) * p.Nq;
            for (int qt = qlo; qt < qhi; ++qt, ++it) {
                const int bf = it & 1;
                const uint32_t par = (it >> 1) & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(BWD_BAR(kBarDQFull + bf), par, abort_flag, p.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t src = tmem + lane_base + bf * C::kBufCols + C::kDPHalf;
                uint32_t r[64];
                tmem_ld32(src, r);
                tmem_ld32(src + 32, r + 32);
                tmem_ld_wait_dep32(r);
                tmem_ld_wait_dep32(r + 32);
                tc_fence_before();
                mbar_arrive(BWD_BAR(kBarDQRead + bf));  // the TMEM buffer may be reused
                if (active) {
                    const long long q0 = static_cast<long long>(qt) * BQ;
                    const int n_valid = static_cast<int>(min(static_cast<long long>(BQ), p.Nq - q0));
                    float* dst = p.dq_acc + (rowbase + q0) * D + drow;
                    if (n_valid == BQ) {
#pragma unroll
                        for (int m = 0; m < BQ; ++m) {
                            asm volatile("red.global.add.f32 [%0], %1;" ::"l"(dst), "f"(__uint_as_float(r[m])) : "memory");
                            dst += D;
                        }
                    } else {
#pragma unroll
                        for (int m = 0; m < BQ; ++m) {
                            if (m < n_valid)
                                asm volatile("red.global.add.f32 [%0], %1;" ::"l"(dst), "f"(__uint_as_float(r[m])) : "memory");
                            dst += D;
                        }
                    }
                }
            }
        }
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
        if (Nq > 0) {
            const uint32_t box[3] = {64u, static_cast<uint32_t>(BQ), 1u};
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
