// Exact attention backward, bf16 in / f32 accumulate, for sm_103a.
//
// What it computes: for O = softmax(Q K^T * scale + mask) V ("Is Flash
// Attention Stable?" §II-A) and an upstream gradient dO, the gradients
//     dV = P^T dO,   dS = P o (dO V^T - D),   dQ = scale dS K,   dK = scale dS^T Q
// with P the attention weights and D_i = sum_c dO_ic O_ic (which equals
// sum_j P_ij (dO V^T)_ij, the softmax Jacobian's rank-one term).  As the
// yadro-code.ru FlashAttention tutorial notes for the method's backward pass,
// nothing of size N x N is stored by the forward: P is recomputed tile by tile
// from Q, K and the per-row LSE the forward wrote, P = exp(s - LSE).
//
// Three launches:
//   prep   one warp per query row: D_i, LSE in log2 units (+inf for a row
//          without any allowed key, so its P is 0), and the row of the f32
//          dQ accumulator set to zero.
//   main   one CTA per (batch*head, key tile of BC = 128 keys), K_j and V_j
//          resident in shared memory, query tiles of BR = 64 rows streamed:
//            warps 0..7  two warpgroups, each thread one key row (tensor
//                        memory lane = key); warpgroup h owns query columns
//                        32h .. 32h+31 of S^T and dP^T.  They load S^T and
//                        dP^T and release them at once, form P and dS in
//                        registers, and write P^T and dS^T (bf16) into their
//                        own tensor-memory columns and dS^T into shared memory
//                        (an operand of the dQ product).  Then the previous
//                        step's dQ^T partial goes to shared memory as dQ rows
//                        and one bulk tensor reduction per warpgroup adds them
//                        into the f32 accumulator in global memory.
//            warp 8      TMA producer: K_j, V_j once; Q_i, dO_i tiles and the
//                        step's LSE / D slices into a ring of NS stages.
//            warp 9      MMA issuer: S^T = K Q_i^T and dP^T = V dO_i^T (both
//                        operands in shared memory), issued for step i+1 as
//                        soon as the warps hold step i's; then dV += P^T dO_i
//                        and dK += dS^T Q_i (A from tensor memory, B MN-major
//                        in shared memory) and dQ_i^T = K_j^T dS_i^T (both
//                        MN-major in shared memory, M = d).
//          Epilogue: dV and scale * dK to bf16, staged over the K / V tiles,
//          TMA-stored.
//   finish dQ = bf16(scale * accumulator).
// Tensor memory (512 columns for d = 128):
//   S^T | dP^T (64 each) | P^T | dS^T (bf16, 32 each) | dV | dK (d each) | dQ^T (64).
#include <cuda_bf16.h>

#include <atomic>
#include <cstdio>
#include <mutex>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace eta {
namespace {

constexpr float kLog2eBw = 1.4426950408889634f;
constexpr float kNegInfBw = -__builtin_huge_valf();
constexpr float kPosInfBw = __builtin_huge_valf();

// Element-wise add of a shared-memory tile into global memory through a tensor
// map (float32 here), as one bulk-group operation; rows outside the tensor are
// dropped.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap *m, uint32_t src, int x, int y, int z) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(m)),
        "r"(src), "r"(x), "r"(y), "r"(z)
        : "memory");
}

template <int D>
struct BwdShape {
    static constexpr int BR = 64;    // query rows per step (streamed)
    static constexpr int BC = 128;   // key rows per CTA (resident)
    static constexpr int CB = D / 64;                // 128-byte column blocks per row
    static constexpr int KV_BYTES = BC * D * 2;      // one K or V tile
    static constexpr int QT_BYTES = BR * D * 2;      // one Q or dO tile
    static constexpr int STAGE_BYTES = 2 * QT_BYTES; // Q_i | dO_i
    static constexpr int STAT_BYTES = 2 * BR * 4;    // LSE (log2) | D of the step's rows
    static constexpr int DS_BYTES = BR * BC * 2;     // dS^T, MN-major B operand of K^T dS^T
    static constexpr int DQ_BYTES = BR * D * 4;      // dQ partial rows (f32), staged for the bulk reduction
    static constexpr int NS = 3;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = KV_BYTES;
    static constexpr int OFF_RING = 2 * KV_BYTES;
    static constexpr int OFF_DS = OFF_RING + NS * STAGE_BYTES;
    static constexpr int OFF_DQ = OFF_DS + DS_BYTES;
    static constexpr int OFF_STAT = OFF_DQ + DQ_BYTES;
    static constexpr int OFF_BAR = OFF_STAT + NS * STAT_BYTES;
    // barriers: kv_full, full[NS], empty[NS], s_full, s_free, ds_ready, b_done, done
    static constexpr int BAR_KV = 0;
    static constexpr int BAR_FULL = 1;
    static constexpr int BAR_EMPTY = BAR_FULL + NS;
    static constexpr int BAR_SFULL = BAR_EMPTY + NS;    // S^T, dP^T of a step are in tensor memory
    static constexpr int BAR_SFREE = BAR_SFULL + 1;     // ... and the warps hold them in registers
    static constexpr int BAR_DSREADY = BAR_SFREE + 1;   // P^T, dS^T, dS^T (shared) of a step written
    static constexpr int BAR_BDONE = BAR_DSREADY + 1;   // the step's dV, dK, dQ^T products are done
    static constexpr int BAR_DONE = BAR_BDONE + 1;
    static constexpr int NBARS = BAR_DONE + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
    // + alignment slack; at least 117 KB so that no second CTA is resident
    // (its 512-column tensor-memory allocation would wait for this one)
    static constexpr int SMEM_MIN = OFF_MISC + 16 + 1024;
    static constexpr int SMEM_BYTES = SMEM_MIN < 117 * 1024 ? 117 * 1024 : SMEM_MIN;
    // tensor memory columns
    static constexpr int C_S = 0;              // S^T (f32)
    static constexpr int C_DP = BR;            // dP^T (f32)
    static constexpr int C_P = 2 * BR;         // P^T (bf16 pairs)
    static constexpr int C_DS = 2 * BR + BR / 2;   // dS^T (bf16 pairs)
    static constexpr int C_DV = 3 * BR;
    static constexpr int C_DK = 3 * BR + D;
    static constexpr int C_DQ = 3 * BR + 2 * D;    // dQ^T: M = d rows (lanes), BR columns
    static constexpr int TMEM_COLS = 512;
    static constexpr int COMPUTE_WARPS = 8;
    static constexpr int WARP_TMA = COMPUTE_WARPS;
    static constexpr int WARP_MMA = COMPUTE_WARPS + 1;
    static constexpr int THREADS = 32 * (COMPUTE_WARPS + 2);

    static_assert(D == 64 || D == 128, "head dim");
    static_assert(C_DQ + BR <= TMEM_COLS, "tensor memory budget");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static_assert(BR == 64 && COMPUTE_WARPS == 8, "two warpgroups of 32 query columns each");
};

struct BwdParams {
    int N;
    int BH;
    int nkt;            // key tiles per head
    int nqt;            // query tiles per head
    int npad;           // padded row count of the LSE / D vectors
    int causal;
    float scale_log2;   // scale * log2(e)
    float scale;
    const float *key_mask;   // [BH][N] additive, or null
    const float *lse2;       // [BH][npad] LSE * log2(e); +inf for padding and empty rows
    const float *dvec;       // [BH][npad] D; 0 for padding
    float *dq_acc;           // [BH][N][D]
    int *err;
};

template <int D>
__global__ void __launch_bounds__(BwdShape<D>::THREADS, 1)
    attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                       const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
    using S = BwdShape<D>;
    constexpr int BR = S::BR, BC = S::BC;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work item: key tile j of head bh ----
    // Causal: key tiles near the start see the most query tiles; they go first.
    int j, bh;
    if (p.causal) {
        j = blockIdx.x / p.BH;
        bh = blockIdx.x % p.BH;
    } else {
        bh = blockIdx.x / p.nkt;
        j = blockIdx.x % p.nkt;
    }
    const int N = p.N;
    const int key0 = j * BC;
    // first query tile with a row that may see a key of this tile
    const int it0 = p.causal ? key0 / BR : 0;
    const int nit = p.nqt - it0;

    auto bar = [&](int i) -> uint32_t { return sbase + S::OFF_BAR + 8 * i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + S::OFF_MISC);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + S::OFF_MISC + 4);
    const uint32_t sK = sbase + S::OFF_K;
    const uint32_t sV = sbase + S::OFF_V;
    const uint32_t sRing = sbase + S::OFF_RING;
    const uint32_t sDS = sbase + S::OFF_DS;
    const uint32_t sDQ = sbase + S::OFF_DQ;
    const uint32_t sStat = sbase + S::OFF_STAT;

    if (threadIdx.x == 0) {
        mbar_init(bar(S::BAR_KV), 1);
        for (int s = 0; s < S::NS; ++s) {
            mbar_init(bar(S::BAR_FULL + s), 1);
            mbar_init(bar(S::BAR_EMPTY + s), 1);
        }
        mbar_init(bar(S::BAR_SFULL), 1);
        mbar_init(bar(S::BAR_SFREE), 32 * S::COMPUTE_WARPS);
        mbar_init(bar(S::BAR_DSREADY), 32 * S::COMPUTE_WARPS);
        mbar_init(bar(S::BAR_BDONE), 1);
        mbar_init(bar(S::BAR_DONE), 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == S::WARP_MMA) {
        tmem_alloc(smem_u32(tmem_slot), S::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Launched as a programmatic dependent of the prep kernel: no global
    // memory is read or written before that grid has completed.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp >= S::COMPUTE_WARPS) {
        // All 32 lanes run the loop with warp-uniform values; one elected lane
        // issues each copy, MMA and commit.  A wait fails for the whole warp
        // if any lane's bounded wait gave up.
        auto wwait = [&](uint32_t b, uint32_t parity, int site) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(b, parity, abort_flag, p.err, site));
        };
        const bool leader = elect_one();
        if (warp == S::WARP_TMA) {
            // --------------------------------------------------------------
            // TMA producer
            // --------------------------------------------------------------
            if (leader) {
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_k);
                tma_prefetch_desc(&tm_v);
                tma_prefetch_desc(&tm_do);
            }
            const uint64_t pol_once = l2_policy_evict_first();   // K_j, V_j: read by this CTA only
            const uint64_t pol_rows = l2_policy_evict_last();    // Q, dO, LSE, D: read by every key tile
            if (leader) {
                mbar_arrive_expect_tx(bar(S::BAR_KV), 2 * S::KV_BYTES);
#pragma unroll
                for (int cb = 0; cb < S::CB; ++cb) {
                    tma_load_3d_hint(sK + cb * (BC * 128), &tm_k, bar(S::BAR_KV), cb * 64, key0, bh, pol_once);
                    tma_load_3d_hint(sV + cb * (BC * 128), &tm_v, bar(S::BAR_KV), cb * 64, key0, bh, pol_once);
                }
            }
            int issued = 0;
            for (int t = 0; t < nit; ++t) {
                const int slot = t % S::NS, round = t / S::NS;
                if (round > 0 && !wwait(bar(S::BAR_EMPTY + slot), (round - 1) & 1, 1)) break;
                const int q0 = (it0 + t) * BR;
                if (leader) {
                    const uint32_t fb = bar(S::BAR_FULL + slot);
                    const uint32_t st = sRing + slot * S::STAGE_BYTES;
                    mbar_arrive_expect_tx(fb, S::STAGE_BYTES + S::STAT_BYTES);
#pragma unroll
                    for (int cb = 0; cb < S::CB; ++cb) {
                        tma_load_3d_hint(st + cb * (BR * 128), &tm_q, fb, cb * 64, q0, bh, pol_rows);
                        tma_load_3d_hint(st + S::QT_BYTES + cb * (BR * 128), &tm_do, fb, cb * 64, q0, bh, pol_rows);
                    }
                    const size_t srow = static_cast<size_t>(bh) * p.npad + q0;
                    bulk_load(sStat + slot * S::STAT_BYTES, p.lse2 + srow, BR * 4, fb, pol_rows);
                    bulk_load(sStat + slot * S::STAT_BYTES + BR * 4, p.dvec + srow, BR * 4, fb, pol_rows);
                }
                issued = t + 1;
            }
            // Drain: every copy this warp started has landed before the CTA may exit.
            for (int t = max(0, issued - S::NS); t < issued; ++t)
                wwait(bar(S::BAR_FULL + t % S::NS), (t / S::NS) & 1, 2);
            wwait(bar(S::BAR_KV), 0, 3);
            __syncwarp();
        } else {
            // --------------------------------------------------------------
            // MMA issuer
            // --------------------------------------------------------------
            constexpr uint32_t idesc_s = idesc_bf16_f32(128, BR, false, false);  // S^T, dP^T: K-major A and B
            constexpr uint32_t idesc_g = idesc_bf16_f32(128, D, false, true);    // dV, dK: A in TMEM, B MN-major
            constexpr uint32_t idesc_q = idesc_bf16_f32(D, BR, true, true);      // dQ^T: A, B MN-major
            bool ok = wwait(bar(S::BAR_KV), 0, 10);
            const uint64_t kdesc = sdesc_sw128(sK, 16, 1024);              // K as K-major A
            const uint64_t vdesc = sdesc_sw128(sV, 16, 1024);              // V as K-major A
            const uint64_t ktdesc = sdesc_sw128(sK, BC * 128, 1024);       // K^T as MN-major A (keys = K dim)
            const uint64_t dsdesc = sdesc_sw128(sDS, 16, 1024);            // dS^T as MN-major B (one 64-wide atom)
            // S^T = K Q_t^T and dP^T = V dO_t^T of step t (stage t % NS)
            auto issue_a = [&](int t) -> bool {
                const int slot = t % S::NS;
                if (!wwait(bar(S::BAR_FULL + slot), (t / S::NS) & 1, 11)) return false;
                tc_fence_after();
                const uint32_t st = sRing + slot * S::STAGE_BYTES;
                const uint64_t qdesc = sdesc_sw128(st, 16, 1024);                  // Q_t as K-major B
                const uint64_t dodesc = sdesc_sw128(st + S::QT_BYTES, 16, 1024);   // dO_t as K-major B
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const int cb = kk >> 2, off = (kk & 3) * 32;
                        mma_bf16_ss(tmem + S::C_S, kdesc + static_cast<uint64_t>((cb * (BC * 128) + off) >> 4),
                                    qdesc + static_cast<uint64_t>((cb * (BR * 128) + off) >> 4), idesc_s,
                                    kk > 0 ? 1u : 0u);
                    }
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const int cb = kk >> 2, off = (kk & 3) * 32;
                        mma_bf16_ss(tmem + S::C_DP, vdesc + static_cast<uint64_t>((cb * (BC * 128) + off) >> 4),
                                    dodesc + static_cast<uint64_t>((cb * (BR * 128) + off) >> 4), idesc_s,
                                    kk > 0 ? 1u : 0u);
                    }
                    tc_commit(bar(S::BAR_SFULL));
                }
                __syncwarp();
                return true;
            };
            if (ok) ok = issue_a(0);
            for (int t = 0; ok && t < nit; ++t) {
                // step t+1's S^T, dP^T overwrite step t's once the warps hold them
                if (t + 1 < nit) {
                    if (!wwait(bar(S::BAR_SFREE), t & 1, 12) || !issue_a(t + 1)) break;
                }
                if (!wwait(bar(S::BAR_DSREADY), t & 1, 13)) break;
                tc_fence_after();
                const int slot = t % S::NS;
                const uint32_t st = sRing + slot * S::STAGE_BYTES;
                const uint64_t qdesc_mn = sdesc_sw128(st, BR * 128, 1024);              // Q_t as MN-major B
                const uint64_t dodesc_mn = sdesc_sw128(st + S::QT_BYTES, BR * 128, 1024);
                if (leader) {
                    // K = BR query columns: 16 queries = 8 columns of bf16 pairs
#pragma unroll
                    for (int kk = 0; kk < BR / 16; ++kk)
                        mma_bf16_ts(tmem + S::C_DV, tmem + S::C_P + 8 * kk,
                                    dodesc_mn + static_cast<uint64_t>((kk * 2048) >> 4), idesc_g,
                                    (t > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                    for (int kk = 0; kk < BR / 16; ++kk)
                        mma_bf16_ts(tmem + S::C_DK, tmem + S::C_DS + 8 * kk,
                                    qdesc_mn + static_cast<uint64_t>((kk * 2048) >> 4), idesc_g,
                                    (t > 0 || kk > 0) ? 1u : 0u);
                    // dQ_t^T = K^T dS^T over K = BC keys (16 keys = 2048 bytes of both operands)
#pragma unroll
                    for (int kk = 0; kk < BC / 16; ++kk)
                        mma_bf16_ss(tmem + S::C_DQ, ktdesc + static_cast<uint64_t>((kk * 2048) >> 4),
                                    dsdesc + static_cast<uint64_t>((kk * 2048) >> 4), idesc_q, kk > 0 ? 1u : 0u);
                    tc_commit(bar(S::BAR_BDONE));
                    tc_commit(bar(S::BAR_EMPTY + slot));
                }
                __syncwarp();
            }
            if (leader) tc_commit(bar(S::BAR_DONE));
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------------
        // Compute warpgroups: thread = key row of the tile
        // ------------------------------------------------------------------
        const int wq = warp & 3, h = warp >> 2;
        const int key_in = wq * 32 + lane;
        const int key = key0 + key_in;
        const uint32_t t_lane = static_cast<uint32_t>(wq * 32) << 16;
        const float sl2 = p.scale_log2;
        // This key's additive term in log2 units; keys past N take no part.
        float mask2 = 0.f;
        if (key >= N) mask2 = kNegInfBw;
        else if (p.key_mask) mask2 = __ldg(p.key_mask + static_cast<size_t>(bh) * N + key) * kLog2eBw;
        const float *stat = reinterpret_cast<const float *>(smem + S::OFF_STAT);
        // dQ^T rows: lane = head-dim index c (M = 128), or lanes 0..15 of each
        // warp (M = 64, rows 16 wq .. 16 wq + 15)
        const bool dq_lane = (D == 128) || (lane < 16);
        const int dq_c = (D == 128) ? wq * 32 + lane : wq * 16 + (lane & 15);
        // One thread per warpgroup issues that warpgroup's bulk reductions.
        const bool issuer = (wq == 0) && (lane == 0);
        const uint32_t stage_dq = sDQ + h * (32 * D * 4);   // 32 query rows x D floats
        // Adds the dQ^T partial of step tq (queries (it0+tq)*BR + 32h + e, e < 32)
        // into the accumulator: the rows go to shared memory, then one bulk
        // tensor reduction adds them (rows past N are dropped by the copy).
        auto drain_dq = [&](int tq, bool live) {
            uint32_t r[32];
            tmem_ld32(tmem + t_lane + S::C_DQ + 32 * h, r);
            tmem_ld_wait();
            reg_fence32(r);
            if (issuer) tma_store_wait_read0();   // the previous reduction has read the staging rows
            named_bar_sync(2 + h, 128);
            if (dq_lane) {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(stage_dq + (e * D + dq_c) * 4), "r"(r[e]) : "memory");
            }
            fence_proxy_async_smem();
            named_bar_sync(2 + h, 128);
            const int y = (it0 + tq) * BR + 32 * h;
            if (issuer && live && y < N) {
                tma_reduce_add_3d(&tm_dq, stage_dq, 0, y, bh);
                tma_store_commit();
            }
        };
        // A wait that gives up (the error word records it; every later wait then
        // gives up at once) does not end the loop: every warp still takes part
        // in every named barrier, on whatever the buffers hold, and nothing is
        // reduced into global memory.
        bool ok = true;
        for (int t = 0; t < nit; ++t) {
            const int slot = t % S::NS;
            const int q0 = (it0 + t) * BR;
            ok = __all_sync(0xffffffffu, mbar_wait(bar(S::BAR_SFULL), t & 1, abort_flag, p.err, 20)) && ok;
            tc_fence_after();
            uint32_t s[32], dp[32];
            tmem_ld32(tmem + t_lane + S::C_S + 32 * h, s);
            tmem_ld32(tmem + t_lane + S::C_DP + 32 * h, dp);
            tmem_ld_wait();
            reg_fence32(s);
            reg_fence32(dp);
            tc_fence_before();
            mbar_arrive(bar(S::BAR_SFREE));
            // this warpgroup's queries q0 + 32h + c; lane c holds query c's LSE (log2) and D
            const float *st_h = stat + slot * (S::STAT_BYTES / 4) + 32 * h;
            const float my_l2 = st_h[lane], my_dv = st_h[BR + lane];
            const int qb = q0 + 32 * h;
            const bool diag = p.causal && (qb <= key0 + BC - 1);   // some query here precedes some key of the tile
            uint32_t pk[16], dk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                float pr[2], ds[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int c = 2 * e + u;
                    float x = fmaf(__uint_as_float(s[c]), sl2, mask2) - __shfl_sync(0xffffffffu, my_l2, c);
                    if (diag && qb + c < key) x = kNegInfBw;
                    pr[u] = ex2(x);
                    ds[u] = pr[u] * (__uint_as_float(dp[c]) - __shfl_sync(0xffffffffu, my_dv, c));
                }
                pk[e] = pack_bf16x2(pr[0], pr[1]);
                dk[e] = pack_bf16x2(ds[0], ds[1]);
            }
            // The previous step's products have read P^T, dS^T and the shared dS^T:
            // reduce its dQ^T, then overwrite them.
            if (t > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar(S::BAR_BDONE), (t - 1) & 1, abort_flag, p.err, 21)) && ok;
                tc_fence_after();
                drain_dq(t - 1, ok);
            }
            tmem_st16(tmem + t_lane + S::C_P + 16 * h, pk);
            tmem_st16(tmem + t_lane + S::C_DS + 16 * h, dk);
            // dS^T into shared memory: row key_in of the MN-major tile (64 queries
            // = one 128-byte row, 16-byte chunks XOR-swizzled by key_in % 8);
            // this warpgroup's 32 queries are chunks 4h .. 4h+3.
            {
                const uint32_t rowaddr = sDS + (key_in >> 3) * 1024 + (key_in & 7) * 128;
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    const int ch = 4 * h + k4;
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(rowaddr + ((ch ^ (key_in & 7)) << 4)),
                                 "r"(dk[4 * k4]), "r"(dk[4 * k4 + 1]), "r"(dk[4 * k4 + 2]), "r"(dk[4 * k4 + 3])
                                 : "memory");
                }
            }
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(S::BAR_DSREADY));
        }
        ok = __all_sync(0xffffffffu, mbar_wait(bar(S::BAR_BDONE), (nit - 1) & 1, abort_flag, p.err, 23)) && ok;
        tc_fence_after();
        drain_dq(nit - 1, ok);
        if (issuer) tma_store_wait0();   // every reduction of this warpgroup has completed
        // ---------------- epilogue: dV, scale * dK ----------------
        mbar_wait(bar(S::BAR_DONE), 0, abort_flag, p.err, 22);
        tc_fence_after();
        const float sc = p.scale;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const uint32_t tcol = which == 0 ? S::C_DV : S::C_DK;
            const uint32_t stage = which == 0 ? sV : sK;   // K_j, V_j are no longer read
            const float mul = which == 0 ? 1.f : sc;
#pragma unroll
            for (int c = h * (D / 64); c < (h + 1) * (D / 64); ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + t_lane + tcol + 32 * c, r);
                tmem_ld_wait();
                reg_fence32(r);
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    w[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * mul, __uint_as_float(r[2 * e + 1]) * mul);
                const int cb = c >> 1;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int ch = (c & 1) * 4 + k;
                    const uint32_t addr = stage + cb * (BC * 128) + key_in * 128 + ((ch ^ (key_in & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[4 * k]),
                                 "r"(w[4 * k + 1]), "r"(w[4 * k + 2]), "r"(w[4 * k + 3])
                                 : "memory");
                }
            }
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 32 * S::COMPUTE_WARPS);
        if (warp == 0 && lane == 0 && !*abort_flag) {
#pragma unroll
            for (int cb = 0; cb < S::CB; ++cb) {
                tma_store_3d(&tm_dv, sV + cb * (BC * 128), cb * 64, key0, bh);
                tma_store_3d(&tm_dk, sK + cb * (BC * 128), cb * 64, key0, bh);
            }
            tma_store_commit();
            tma_store_wait0();
        }
    }

    // The finish kernel may be scheduled now (it waits for this grid's
    // completion before it reads the accumulator).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    if (warp == S::WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, S::TMEM_COLS);
    }
}

// Per (padded) query row: D_i = <dO_i, O_i>, LSE in log2 units, and the row
// of the dQ accumulator cleared.  A warp takes RPW consecutive rows of one
// head and issues all their loads before it uses one.
constexpr int kPrepRowsPerWarp = 4;   // divides npad (a multiple of 64)

template <int D>
__global__ void attn_bwd_prep_kernel(const __nv_bfloat16 *__restrict__ O, const __nv_bfloat16 *__restrict__ dO,
                                     const float *__restrict__ LSE, float *__restrict__ lse2,
                                     float *__restrict__ dvec, float *__restrict__ dq_acc, int BH, int N, int npad) {
    constexpr int RPW = kPrepRowsPerWarp;
    // a programmatic dependent of the kernel before it in the stream: no
    // global memory is touched before that grid has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw * RPW < static_cast<long long>(BH) * npad) {
        const int bh = static_cast<int>(gw * RPW / npad);
        const int i0 = static_cast<int>(gw * RPW % npad);   // the RPW rows are i0 .. i0 + RPW - 1 of head bh
        constexpr int PER = D / 32;   // elements per lane (2 or 4), one vector load each
        using V = typename std::conditional<PER == 4, uint2, uint32_t>::type;
        V ov[RPW], gv[RPW];
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            if (i0 + r < N) {
                const size_t row = static_cast<size_t>(bh) * N + i0 + r;
                ov[r] = *reinterpret_cast<const V *>(O + row * D + lane * PER);
                gv[r] = *reinterpret_cast<const V *>(dO + row * D + lane * PER);
            }
        }
        float acc[RPW];
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            acc[r] = 0.f;
            if (i0 + r < N) {
                if constexpr (PER == 4) {
                    acc[r] = fmaf(bf16lo_to_f32(ov[r].x), bf16lo_to_f32(gv[r].x), acc[r]);
                    acc[r] = fmaf(bf16hi_to_f32(ov[r].x), bf16hi_to_f32(gv[r].x), acc[r]);
                    acc[r] = fmaf(bf16lo_to_f32(ov[r].y), bf16lo_to_f32(gv[r].y), acc[r]);
                    acc[r] = fmaf(bf16hi_to_f32(ov[r].y), bf16hi_to_f32(gv[r].y), acc[r]);
                } else {
                    acc[r] = fmaf(bf16lo_to_f32(ov[r]), bf16lo_to_f32(gv[r]), acc[r]);
                    acc[r] = fmaf(bf16hi_to_f32(ov[r]), bf16hi_to_f32(gv[r]), acc[r]);
                }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int r = 0; r < RPW; ++r) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const size_t srow = static_cast<size_t>(bh) * npad + i0 + r;
            if (i0 + r >= N) {
                if (lane == 0) {
                    lse2[srow] = kPosInfBw;
                    dvec[srow] = 0.f;
                }
                continue;
            }
            const size_t row = static_cast<size_t>(bh) * N + i0 + r;
            float *z = dq_acc + row * D + lane * PER;
            if constexpr (PER == 4) *reinterpret_cast<float4 *>(z) = make_float4(0.f, 0.f, 0.f, 0.f);
            else *reinterpret_cast<float2 *>(z) = make_float2(0.f, 0.f);
            if (lane == 0) {
                const float l = LSE[row];
                lse2[srow] = (l == kNegInfBw) ? kPosInfBw : l * kLog2eBw;
                dvec[srow] = acc[r];
            }
        }
    }
    // The main kernel (a programmatic dependent launch) may be scheduled now.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// dQ = bf16(scale * accumulator), four elements per thread.
__global__ void attn_bwd_finish_kernel(const float4 *__restrict__ acc, uint2 *__restrict__ dq, long long n4,
                                       float scale) {
    // a programmatic dependent of the main kernel: its reductions are complete first
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (long long k = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; k < n4;
         k += static_cast<long long>(gridDim.x) * blockDim.x) {
        const float4 a = acc[k];
        uint2 w;
        w.x = pack_bf16x2(a.x * scale, a.y * scale);
        w.y = pack_bf16x2(a.z * scale, a.w * scale);
        dq[k] = w;
    }
    // the next kernel in the stream may be scheduled now (it waits for this grid)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// The float32 dQ accumulator [BH][N][D] as a tensor of 32-row boxes (no swizzle).
bool make_acc_map(CUtensorMap *m, const float *base, int D, int N, int BH) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 4, static_cast<cuuint64_t>(N) * D * 4};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(D), 32u, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int npad_of(int N) { return (N + 63) / 64 * 64; }

template <int D>
int launch_bwd_d(const void *Q, const void *K, const void *V, const void *O, const void *dO, const float *LSE,
                 void *dQ, void *dK, void *dV, int BH, int N, int causal, float scale, const float *key_mask,
                 void *workspace, cudaStream_t stream) {
    using S = BwdShape<D>;
    auto kern = attn_bwd_tc_kernel<D>;
    // The shared-memory opt-in, once per device (calls may come from several
    // host threads).
    constexpr int kMaxDevBw = 64;
    static std::atomic<int> ready[kMaxDevBw];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevBw) return kErrCuda;
    if (ready[dev].load(std::memory_order_acquire) == 0) {
        std::lock_guard<std::mutex> lk(mu);
        if (ready[dev].load(std::memory_order_relaxed) == 0) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM_BYTES) != cudaSuccess)
                return kErrCuda;
            ready[dev].store(1, std::memory_order_release);
        }
    }
    const int npad = npad_of(N);
    char *ws = static_cast<char *>(workspace);
    float *lse2 = reinterpret_cast<float *>(ws);
    float *dvec = reinterpret_cast<float *>(ws + round256(static_cast<size_t>(BH) * npad * 4));
    float *acc = reinterpret_cast<float *>(ws + 2 * round256(static_cast<size_t>(BH) * npad * 4));

    CUtensorMap tq, tk, tv, tdo, tdk, tdv, tdq;
    if (!make_bf16_rows_map(&tq, Q, D, N, BH, S::BR) || !make_bf16_rows_map(&tk, K, D, N, BH, S::BC) ||
        !make_bf16_rows_map(&tv, V, D, N, BH, S::BC) || !make_bf16_rows_map(&tdo, dO, D, N, BH, S::BR) ||
        !make_bf16_rows_map(&tdk, dK, D, N, BH, S::BC) || !make_bf16_rows_map(&tdv, dV, D, N, BH, S::BC) ||
        !make_acc_map(&tdq, acc, D, N, BH))
        return kErrCuda;
    int *err = device_error_word();
    if (!err) return kErrCuda;

    {
        const long long warps = static_cast<long long>(BH) * npad / kPrepRowsPerWarp;
        const long long blocks = (warps * 32 + 255) / 256;
        if (blocks > 0x7fffffffLL) return kErrUnsupported;
        // a programmatic dependent launch, like the two kernels after it
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(blocks));
        cfg.blockDim = dim3(256);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const __nv_bfloat16 *o16 = static_cast<const __nv_bfloat16 *>(O);
        const __nv_bfloat16 *do16 = static_cast<const __nv_bfloat16 *>(dO);
        if (cudaLaunchKernelEx(&cfg, attn_bwd_prep_kernel<D>, o16, do16, LSE, lse2, dvec, acc, BH, N, npad) !=
            cudaSuccess) {
            (void)cudaGetLastError();
            attn_bwd_prep_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(o16, do16, LSE, lse2, dvec,
                                                                                     acc, BH, N, npad);
            if (cudaGetLastError() != cudaSuccess) return kErrCuda;
        }
    }
    BwdParams p;
    p.N = N;
    p.BH = BH;
    p.nkt = (N + S::BC - 1) / S::BC;
    p.nqt = (N + S::BR - 1) / S::BR;
    p.npad = npad;
    p.causal = causal;
    p.scale_log2 = scale * kLog2eBw;
    p.scale = scale;
    p.key_mask = key_mask;
    p.lse2 = lse2;
    p.dvec = dvec;
    p.dq_acc = acc;
    p.err = err;
    const long long grid = static_cast<long long>(BH) * p.nkt;
    if (grid > 0x7fffffffLL) return kErrUnsupported;
    // The main and finish kernels are programmatic dependent launches: each
    // grid's launch overlaps the end of the one before, and each waits for it
    // (griddepcontrol.wait) before touching global memory.  An ordinary launch
    // is the fallback.
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(S::THREADS);
        cfg.dynamicSmemBytes = S::SMEM_BYTES;
        cfg.stream = stream;
        cfg.attrs = pdl;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, tdo, tdk, tdv, tdq, p) != cudaSuccess) {
            (void)cudaGetLastError();
            kern<<<static_cast<unsigned>(grid), S::THREADS, S::SMEM_BYTES, stream>>>(tq, tk, tv, tdo, tdk, tdv, tdq,
                                                                                   p);
            if (cudaGetLastError() != cudaSuccess) return kErrCuda;
        }
    }
    {
        const long long n4 = static_cast<long long>(BH) * N * D / 4;
        long long blocks = (n4 + 255) / 256;
        if (blocks > 4 * 152 * 8) blocks = 4 * 152 * 8;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(blocks));
        cfg.blockDim = dim3(256);
        cfg.stream = stream;
        cfg.attrs = pdl;
        cfg.numAttrs = 1;
        const float4 *a4 = reinterpret_cast<const float4 *>(acc);
        uint2 *q2 = static_cast<uint2 *>(dQ);
        if (cudaLaunchKernelEx(&cfg, attn_bwd_finish_kernel, a4, q2, n4, scale) != cudaSuccess) {
            (void)cudaGetLastError();
            attn_bwd_finish_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a4, q2, n4, scale);
            if (cudaGetLastError() != cudaSuccess) return kErrCuda;
        }
    }
    return kOk;
}

}  // namespace

size_t bwd_workspace_bytes(int BH, int N, int d) {
    const size_t stats = round256(static_cast<size_t>(BH) * npad_of(N) * 4);
    return 2 * stats + round256(static_cast<size_t>(BH) * N * d * 4);
}

int launch_bwd_tc_bf16(const void *Q, const void *K, const void *V, const void *O, const void *dO, const float *LSE,
                       void *dQ, void *dK, void *dV, int B, int H, int N, int d, int causal, float scale,
                       const float *key_mask, void *workspace, cudaStream_t stream) {
    const int BH = B * H;
    if (d == 64)
        return launch_bwd_d<64>(Q, K, V, O, dO, LSE, dQ, dK, dV, BH, N, causal, scale, key_mask, workspace, stream);
    if (d == 128)
        return launch_bwd_d<128>(Q, K, V, O, dO, LSE, dQ, dK, dV, BH, N, causal, scale, key_mask, workspace, stream);
    return kErrUnsupported;
}

}  // namespace eta
