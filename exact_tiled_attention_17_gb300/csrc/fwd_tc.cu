// Exact tiled attention forward, bf16 in / f32 accumulate, for sm_103a.
//
// What it computes: O = softmax(Q K^T * scale + mask) V and the per-row
// natural-log LSE ("Is Flash Attention Stable?" §II-A), tile by tile as in
// its §II-B / Fig. 1, never forming the N x N score matrix.  Each query row
// carries the online-softmax state of the yadro-code.ru FlashAttention
// tutorial: a running maximum m, a running denominator l and an
// unnormalised accumulator that is multiplied by exp(m_old - m_new) when the
// maximum grows, with one division at the end.
//
// GB300 mapping: at most one CTA per SM, each running a list of work units:
// a group of NQ consecutive BR-row query tiles of one (batch, head), or one
// part of such a group split along K/V (the last round; merged in a cluster).
// Causal: heaviest groups (largest row index) first.
//   warps 0 .. 4*NQ*NH-1  softmax warpgroups: NH per query tile (NH = 2 for
//                  BC = 128: each owns half of the tile's key columns and half
//                  of O's columns).  One thread per row (tensor-memory lane =
//                  row).  Reads its S columns, applies the scale (and the
//                  causal and length masks on edge tiles), keeps the row
//                  state (m, l), rescales its O columns in tensor memory when
//                  needed, writes its part of P as bf16 back over its S
//                  columns, then the epilogue (normalise, bf16 stores; LSE).
//   next warp      TMA producer: each unit's Q tiles, then K_j / V_j tiles
//                  into a ring of NS shared-memory slots (128-byte swizzle).
//   next warp      MMA issuer (one elected lane): S_q = Q_q K_j^T (both
//                  operands in shared memory; with a key mask one more K step,
//                  ones x mask operand, adds mask / scale to every row) and
//                  O_q += P_q V_j (P from tensor memory, V MN-major in shared
//                  memory) on tcgen05, f32 accumulators in tensor memory.
//   next warp      (with a key mask) writes each K tile's mask / scale into
//                  the ring slot as a 16-wide bf16 operand, three exact parts
//                  per key, and arrives on the slot's full barrier too.  A
//                  masked tile thus reaches the softmax like any other.
// The MMA issue order S_0(j+1) after P_0 V_j, S_1(j+1) after P_1 V_j lets the
// tensor pipe work on one tile while the other tile's softmax runs.  P_q is
// handed over on one barrier that both warpgroups of the tile arrive on, so
// the MMA warp wakes once per tile (waking once per warpgroup cost ~3%), and
// P_q V starts only after both warpgroups have rescaled their O columns.
// Where tensor memory has room (BC = 64) each query tile has two S buffers
// and S_q(j+2) is issued right after P_q V_j, so the softmax never waits for
// its own P V.
//
// BR = 64 uses M = 64 MMAs, whose accumulator rows r sit in tensor-memory lane
// 32*(r/16) + r%16: lanes 0..15 of each warp carry rows, lanes 16..31 idle.
//
// Each tile's row maximum is taken first (with the tensor-memory loads of S,
// which return it on sm_103a; the two warpgroups of a tile exchange theirs),
// then the exponentials.  The reference maximum m moves only to a tile
// maximum more than kRescaleThresh above it, so O is rescaled rarely and
// every p stays below 2^kRescaleThresh.
// Exact up to rounding: O / l does not depend on the reference point.
// One denominator per row, the float32 sum of the bf16-rounded p that P V
// applies, so the weights that reach O sum to one (a row whose weight sits
// on one key gets that key's V exactly, wherever the reference maximum is);
// it also gives the LSE.
//
// Block-sparse variant (BSPARSE): a byte mask over 128 x 128 (query block, key
// block) pairs says which blocks take part; every other score is -inf.  The
// unit runs only the key tiles marked for at least one of its query tiles (a
// list that one warp builds while the previous unit runs, in one of three
// rotating buffers); a listed tile that is not marked for a query tile is
// masked whole for it.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <mutex>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace eta {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThresh = 8.0f;
constexpr float kNegInf = -__builtin_huge_valf();

constexpr int kBsListCap = 1024;   // key tiles a block-sparse CTA can list (N <= 131072)

template <int D, int BR, int BC, int NQ, bool MASKED, bool BSPARSE = false>
struct TcShape {
    static constexpr int CB = D / 64;               // 128-byte column blocks per row
    static constexpr int Q_BYTES = BR * D * 2;      // one Q (or O staging) tile
    static constexpr int SLOT_BYTES = BC * D * 2;   // one K or V tile
    static constexpr int SMEM_BUDGET = 225 * 1024;  // leaves room for barriers and alignment
    // Key mask as one more K = 16 step of S = Q K^T: a constant A operand of
    // ones (128 rows, k = 0..2 one, the rest zero) times a B operand holding
    // each key's mask / scale as three bf16 parts (hi + mid + lo, k = 0..2).
    // Both are K-major without swizzle: 32 bytes per row, 8-row groups of
    // 256 bytes.  One B operand per ring slot (written with the K tile).
    static constexpr int MOP_ROW = 32;
    static constexpr int MOP_ONES = MASKED ? 128 * MOP_ROW : 0;
    static constexpr int MOP_SLOT = MASKED ? BC * MOP_ROW : 0;
    // Two S buffers per query tile when tensor memory has room: S_q(j+2) is
    // computed while the softmax works on S_q(j+1) and P_q(j) waits for its
    // P V, instead of after P V.
    static constexpr bool DBS = 2 * NQ * BC + NQ * D <= 512;
    static constexpr int NSB = DBS ? 2 : 1;
    // BC = 128: two softmax warpgroups share each query tile, one per half of
    // its columns (and of O's columns).
    static constexpr int NH = BC == 128 ? 2 : 1;
    // two warpgroups per tile exchange per-row values (half maxima, partial sums)
    static constexpr int XCH_BYTES = NH == 2 ? NQ * 2 * 128 * 8 : 0;
    // block-sparse: the listed key tiles (index | per-query-tile marks << 14) and per-tile counts
    // block-sparse: three unit lists in rotation (a unit's list is built while
    // the previous unit runs; no warp is ever two units behind another)
    static constexpr int LIST_ONE = kBsListCap * 2 + 16;
    static constexpr int LIST_BYTES = BSPARSE ? 3 * LIST_ONE : 0;
    static constexpr int NS_RAW = (SMEM_BUDGET - NQ * Q_BYTES - MOP_ONES - XCH_BYTES - LIST_BYTES) / (SLOT_BYTES + MOP_SLOT);
    static constexpr int NS = NS_RAW > 8 ? 8 : (NS_RAW < 2 ? 2 : NS_RAW);
    static constexpr int MASK_BYTES = MOP_ONES + NS * MOP_SLOT;
    static constexpr int TMEM_USED = NQ * (NSB * BC + D);
    static constexpr int TMEM_COLS = TMEM_USED <= 32 ? 32
                                     : TMEM_USED <= 64 ? 64
                                     : TMEM_USED <= 128 ? 128
                                     : TMEM_USED <= 256 ? 256 : 512;
    static constexpr int SOFTMAX_WARPS = 4 * NQ * NH;
    static constexpr int WARP_TMA = SOFTMAX_WARPS;
    static constexpr int WARP_MMA = SOFTMAX_WARPS + 1;
    // key mask: one more warp writes each K tile's mask operand (off the
    // TMA producer's path; with 18 or 10 other warps it costs no registers)
    static constexpr int WARP_MASK = SOFTMAX_WARPS + 2;
    static constexpr int EXTRA_WARPS = MASKED ? 3 : 2;

    // setmaxnreg could move registers from the producer/MMA warpgroup to the
    // softmax warpgroups; every shape here fits the launch share, and the
    // move only makes ptxas spill around it.
    static constexpr bool MOVE_REGS = false;
    // softmax warps + TMA + MMA (a whole warpgroup for those two when
    // registers are moved, since setmaxnreg acts per warpgroup)
    static constexpr int THREADS = MOVE_REGS ? 32 * SOFTMAX_WARPS + 128 : 32 * (SOFTMAX_WARPS + EXTRA_WARPS);
    static constexpr int LAUNCH_REGS = NH == 2 ? 96 : 168;   // 65536 / THREADS, rounded down to 8
    static constexpr int REGS_SOFTMAX = NH == 2 ? 112 : 208;
    static constexpr int REGS_OTHER = NH == 2 ? 32 : 88;     // softmax + other shares == THREADS * LAUNCH_REGS
    // shared memory layout (offsets from a 1024-byte aligned base)
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_RING = NQ * Q_BYTES;
    static constexpr int OFF_MASK = OFF_RING + NS * SLOT_BYTES;
    static constexpr int OFF_XCH = OFF_MASK + MASK_BYTES;
    static constexpr int OFF_LIST = OFF_XCH + XCH_BYTES;
    static constexpr int OFF_BAR = OFF_LIST + LIST_BYTES;
    // barriers: q_full[NQ] full[NS] empty[NS] s_full[NQ][NSB] p_full[NQ][NSB][NH] o_full[NQ]
    // pv_done[NQ] q_free[NQ] o_free[NQ] done part
    static constexpr int BAR_QFULL = 0;
    static constexpr int BAR_FULL = BAR_QFULL + NQ;
    static constexpr int BAR_EMPTY = BAR_FULL + NS;
    static constexpr int BAR_SFULL = BAR_EMPTY + NS;
    static constexpr int BAR_PFULL = BAR_SFULL + NQ * NSB;
    static constexpr int BAR_OFULL = BAR_PFULL + NQ * NSB;
    static constexpr int BAR_PVDONE = BAR_OFULL + NQ;   // two S buffers: each P_q V has completed
    // A CTA runs several work units: Q_q may be reloaded once the unit's last
    // S_q product has completed, and O_q rewritten once the epilogue has read it.
    static constexpr int BAR_QFREE = BAR_PVDONE + NQ;
    static constexpr int BAR_OFREE = BAR_QFREE + NQ;
    static constexpr int BAR_DONE = BAR_OFREE + NQ;
    static constexpr int BAR_PART = BAR_DONE + 1;       // split K/V: partials of the other parts are ready
    static constexpr int BAR_LIST = BAR_PART + 1;       // block-sparse: unit list b is built (3)
    static constexpr int NBARS = BAR_LIST + 3;
    // split K/V: a part's partial results, staged in the (then idle) Q tiles and K/V ring:
    // unnormalised O (float32) and the per-row m, l.  O is stored as 16-byte
    // pieces [query tile][32-column chunk][piece k of 8][row], so the 32 lanes
    // of a warp (32 consecutive rows) read 512 contiguous bytes per load.
    static constexpr int PART_BYTES = (NQ * 128 * D + 2 * NQ * 128) * 4;
    static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
    // + alignment slack; a 512-column tensor-memory user also claims enough
    // shared memory that no second CTA can be resident (its allocation would wait)
    static constexpr int SMEM_MIN = OFF_MISC + 16 + 1024;
    static constexpr int SMEM_BYTES = (TMEM_COLS == 512 && SMEM_MIN <= 116 * 1024) ? 117 * 1024 : SMEM_MIN;

    __host__ __device__ static constexpr int s_col(int q, int b) { return (q * NSB + b) * BC; }
    __host__ __device__ static constexpr int o_col(int q) { return NQ * NSB * BC + q * D; }

    static_assert(D == 64 || D == 128, "head dim");
    static_assert(BR == 64 || BR == 128, "query tile");
    static_assert(BC == 64 || BC == 128 || BC == 256, "key tile");
    static_assert(TMEM_USED <= 512, "tensor memory budget");
    // A 512-column allocation must never wait for another resident CTA.
    static_assert(TMEM_COLS < 512 || SMEM_BYTES > 116 * 1024, "one CTA per SM for full TMEM");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static_assert(!MOVE_REGS || 32 * SOFTMAX_WARPS * REGS_SOFTMAX + 128 * REGS_OTHER == THREADS * LAUNCH_REGS,
                  "register split must equal the launch allocation");
    // two S buffers: K_{j+2} is waited for while V_j still holds its slot
    static_assert(!DBS || NS >= 4, "ring depth for two S buffers");
    static constexpr bool CAN_SPLIT = (PART_BYTES <= NQ * Q_BYTES + NS * SLOT_BYTES) && (BR == 128) && !BSPARSE;
    static_assert(!BSPARSE || (BR == 128 && BC == 128 && NQ <= 2), "block-sparse tiles are the 128 x 128 blocks");
};

struct TcParams {
    int N;              // sequence length
    int BH;             // B * H
    int num_qg;         // query groups (NQ * BR rows) per head
    int causal;
    float scale;        // multiplies Q K^T
    float inv_scale;    // 1 / scale (rounded once from double)
    float scale_log2;   // scale * log2(e)
    const float *key_mask;  // [BH][N] additive, or null
    const uint8_t *block_mask;  // block-sparse: [BH][nkb][nkb] bytes, non-zero = take part
    int nkb;                    // 128-row blocks per head
    __nv_bfloat16 *o;       // [BH][N][D]
    float *lse;             // [BH][N], or null
    int *err;               // device error word
    // Work items (groups of NQ query tiles of one head) are numbered heaviest
    // first for causal (largest rows first) and head-major otherwise.  Every
    // CTA of the grid (G CTAs, at most one per SM) runs a list of work units:
    // items [0, n_full) whole, CTA c taking items c, c + G, c + 2G, ...
    // (causal: every other round in reverse, so long and short items mix);
    // then each item in [n_full, items) split along K/V into `split` parts,
    // run as the last unit of the `split` CTAs of one cluster; the parts swap
    // partials and each merges and stores a share of O's columns.
    int items;
    int n_full;
    int split;
    int split_shift;   // log2(split)
};

// The u-th work unit of CTA c in a grid of G CTAs (see TcParams); false when
// the CTA has no u-th unit.
__device__ __forceinline__ bool work_unit(const TcParams &p, int c, int G, int u, int &item, int &part,
                                          int &nparts) {
    auto full = [&](int r) { return r * G + ((p.causal && (r & 1)) ? G - 1 - c : c); };
    const int f = full(u);
    if (f < p.n_full) {
        item = f;
        part = 0;
        nparts = 1;
        return true;
    }
    if (u > 0 && full(u - 1) >= p.n_full) return false;   // the tail unit comes right after the full ones
    if (c >= (p.items - p.n_full) << p.split_shift) return false;
    item = p.n_full + (c >> p.split_shift);
    part = c & (p.split - 1);   // equals the rank in the cluster
    nparts = p.split;
    return true;
}

template <int D, int BR, int BC, int NQ, bool MASKED, bool BSPARSE>
__global__ void __launch_bounds__(TcShape<D, BR, BC, NQ, MASKED, BSPARSE>::THREADS, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
    using S = TcShape<D, BR, BC, NQ, MASKED, BSPARSE>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int N = p.N;
    const int nkv_all = (N + BC - 1) / BC;
    const int cta = blockIdx.x;
    const int G = gridDim.x;
    // block-sparse: the listed key tiles of unit u (index | per-query-tile marks
    // << 14) and, after them, the per-query-tile list lengths
    auto list_of = [&](int u) { return reinterpret_cast<uint16_t *>(smem + S::OFF_LIST + (u % 3) * S::LIST_ONE); };
    uint16_t *kv_list = list_of(0);   // the current unit's list

    // ---- geometry of one work unit ----
    // Causal: heaviest query groups (largest rows) first.  Non-causal: all
    // query groups of one head together, so a head's K/V stay hot in L2.
    // Query tile q starts at row r0[q] and runs the K/V tiles
    // [kv_lo, kv_lo + nkv[q]) (a part's share of a split item; block-sparse:
    // the first nkv[q] entries of the CTA's list).
    int bh = 0, kv_lo = 0, nkv_max = 0;
    int r0[NQ], nkv[NQ];
    // (32-bit arithmetic only: nkv_all * 8 < 2^31, and nparts = 2^split_shift)
    auto geometry = [&](int u, int item, int part, int nparts) {
        if constexpr (BSPARSE) kv_list = list_of(u);
        const int dq = p.causal ? p.BH : p.num_qg;
        const int quo = item / dq, rem = item - quo * dq;
        const int qg = p.causal ? p.num_qg - 1 - quo : rem;
        bh = p.causal ? rem : quo;
        const int sh = nparts > 1 ? p.split_shift : 0;
        kv_lo = (nkv_all * part) >> sh;
        const int kv_hi = (nkv_all * (part + 1)) >> sh;
        nkv_max = 0;
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            r0[q] = (qg * NQ + q) * BR;
            if (r0[q] >= N) {
                nkv[q] = 0;
            } else if constexpr (BSPARSE) {
                // (clamped: after a failed wait the list may not have been built)
                nkv[q] = min(max(reinterpret_cast<const int *>(kv_list + kBsListCap)[q], 0), kBsListCap);
            } else if (p.causal) {
                const int last_row = min(r0[q] + BR - 1, N - 1);
                nkv[q] = min(nkv_all, last_row / BC + 1);
            } else {
                nkv[q] = kv_hi - kv_lo;
            }
            nkv_max = max(nkv_max, nkv[q]);
        }
    };

    auto bar = [&](int i) -> uint32_t { return sbase + S::OFF_BAR + 8 * i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + S::OFF_MISC);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + S::OFF_MISC + 4);
    const uint32_t sQ = sbase + S::OFF_Q;
    const uint32_t sRing = sbase + S::OFF_RING;

    if (threadIdx.x == 0) {
        for (int q = 0; q < NQ; ++q) {
            mbar_init(bar(S::BAR_QFULL + q), 1);
            for (int b = 0; b < S::NSB; ++b) {
                mbar_init(bar(S::BAR_SFULL + q * S::NSB + b), 1);
                // every softmax thread of the tile (both warpgroups): the MMA
                // warp wakes once per tile, not once per warpgroup
                mbar_init(bar(S::BAR_PFULL + q * S::NSB + b), 128 * S::NH);
            }
            mbar_init(bar(S::BAR_OFULL + q), 1);
            mbar_init(bar(S::BAR_PVDONE + q), 1);
            mbar_init(bar(S::BAR_QFREE + q), 1);
            mbar_init(bar(S::BAR_OFREE + q), 128 * S::NH);
        }
        for (int s = 0; s < S::NS; ++s) {
            mbar_init(bar(S::BAR_FULL + s), MASKED ? 2 : 1);   // (+ the mask warp)
            mbar_init(bar(S::BAR_EMPTY + s), 1);
        }
        mbar_init(bar(S::BAR_DONE), 1);
        mbar_init(bar(S::BAR_PART), static_cast<uint32_t>((p.split > 1 ? p.split - 1 : 1) * S::SOFTMAX_WARPS * 32));
        for (int b = 0; b < 3; ++b) mbar_init(bar(S::BAR_LIST + b), 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == S::WARP_MMA) {
        tmem_alloc(smem_u32(tmem_slot), S::TMEM_COLS);
        tmem_relinquish();
    }
    // Block-sparse: warp 1 builds unit u's list into buffer u % 3 (key tiles
    // marked for at least one of the unit's query tiles, in order, with the
    // per-tile marks in bits 14..15, and per query tile how many entries reach
    // its last marked tile) and arrives on that buffer's barrier.  A query
    // tile inside N with no marked tile still runs one fully masked tile,
    // which writes O = 0 and LSE = -inf.
    auto build_list = [&](int u) {
        int item, part, nparts;
        if (!work_unit(p, cta, G, u, item, part, nparts)) return;
        const int dq = p.causal ? p.BH : p.num_qg;
        const int quo = item / dq, rem = item - quo * dq;
        const int qg = p.causal ? p.num_qg - 1 - quo : rem;
        const int bhu = p.causal ? rem : quo;
        int r0u[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) r0u[q] = (qg * NQ + q) * BR;
        uint16_t *lst = list_of(u);
        int *counts = reinterpret_cast<int *>(lst + kBsListCap);
        const int nkb = p.nkb;
        const uint8_t *bm = p.block_mask + static_cast<size_t>(bhu) * nkb * nkb;
        int cnt = 0, last[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) last[q] = 0;
        for (int j0 = 0; j0 < nkb; j0 += 32) {
            const int jt = j0 + lane;
            uint32_t marks = 0;
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                if (r0u[q] < N && jt < nkb) {
                    bool a = bm[static_cast<size_t>(r0u[q] / 128) * nkb + jt] != 0;
                    if (p.causal) a = a && (jt * BC <= min(r0u[q] + BR - 1, N - 1));
                    if (a) marks |= 1u << q;
                }
            }
            const uint32_t ball = __ballot_sync(0xffffffffu, marks != 0);
            if (marks) lst[cnt + __popc(ball & ((1u << lane) - 1u))] = static_cast<uint16_t>(jt | (marks << 14));
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const uint32_t bq = __ballot_sync(0xffffffffu, (marks >> q) & 1u);
                if (bq) {
                    const int L = 31 - __clz(bq);
                    last[q] = cnt + __popc(ball & ((1u << L) - 1u)) + 1;
                }
            }
            cnt += __popc(ball);
        }
        bool empty_tile = false;
#pragma unroll
        for (int q = 0; q < NQ; ++q) empty_tile = empty_tile || (r0u[q] < N && last[q] == 0);
        if (empty_tile && cnt == 0 && lane == 0) lst[0] = 0;
        if (lane == 0) {
#pragma unroll
            for (int q = 0; q < NQ; ++q) counts[q] = (r0u[q] < N && last[q] == 0) ? 1 : last[q];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(S::BAR_LIST + u % 3));
    };
    // Every role waits for unit u's list before reading it.
    auto wait_list = [&](int u) -> bool {
        if constexpr (BSPARSE) return mbar_wait(bar(S::BAR_LIST + u % 3), (u / 3) & 1, abort_flag, p.err, 26);
        return true;
    };
    if constexpr (MASKED) {
        // The ones operand (16-byte unit i: k-chunk (i >> 3) & 1, whose chunk 0
        // holds 1, 1, 1, 0 ... in bf16) and every slot's B operand zeroed (its
        // k = 8..15 chunk stays zero; k = 0..7 is rewritten per K tile).
        for (int i = threadIdx.x; i < S::MASK_BYTES / 16; i += S::THREADS) {
            const bool one = i < S::MOP_ONES / 16 && ((i >> 3) & 1) == 0;
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sbase + S::OFF_MASK + 16 * i),
                         "r"(one ? 0x3F803F80u : 0u), "r"(one ? 0x00003F80u : 0u), "r"(0u), "r"(0u)
                         : "memory");
        }
        fence_proxy_async_smem();   // read by the tensor core
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // first key tile of the unit's j-th K/V tile
    auto kv_tile = [&](int jj) -> int {
        if constexpr (BSPARSE) return kv_list[jj] & 0x3FFF;
        else return kv_lo + jj;
    };
    // Launched as a programmatic dependent of the kernel before it in the
    // stream: no global memory is read or written before that grid has
    // completed (the set-up above touches only this CTA's memories).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if constexpr (S::CAN_SPLIT) {
        // Parts of a split item arrive on each other's barriers: all of the
        // cluster's barriers must be initialised first.
        if (p.split > 1) cluster_sync();
    }

    if (warp >= S::SOFTMAX_WARPS) {
        if constexpr (S::MOVE_REGS) regs_dec<S::REGS_OTHER>();
        // The producer and MMA warps run their loops on all 32 lanes with
        // warp-uniform values (so address and descriptor arithmetic stays on
        // the uniform datapath) and one elected lane issues each copy, MMA
        // and commit.  A wait counts as failed for the warp if any lane's
        // bounded wait gave up, so every lane leaves a loop together.
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
            }
            const uint64_t pol_kv = l2_policy_evict_last();   // K/V are re-read by every query group
            const uint64_t pol_q = l2_policy_evict_first();   // Q is read once
            int t = 0;                 // K/V tiles issued so far, all units: K_0 V_0 K_1 V_1 ...
            int uo[NQ];                // units so far in which query tile q ran
#pragma unroll
            for (int q = 0; q < NQ; ++q) uo[q] = 0;
            bool ok = true;
            for (int u = 0; ok; ++u) {
                int item, part, nparts;
                if (!work_unit(p, cta, G, u, item, part, nparts)) break;
                if constexpr (BSPARSE) {
                    if (!wwait(bar(S::BAR_LIST + u % 3), (u / 3) & 1, 26)) {
                        ok = false;
                        break;
                    }
                }
                geometry(u, item, part, nparts);
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    if (nkv[q] == 0) continue;
                    // Q_q of the previous unit is still read by its last S products.
                    if (uo[q] > 0 && !wwait(bar(S::BAR_QFREE + q), (uo[q] - 1) & 1, 4)) ok = false;
                    if (ok && leader) {
                        mbar_arrive_expect_tx(bar(S::BAR_QFULL + q), S::Q_BYTES);
#pragma unroll
                        for (int cb = 0; cb < S::CB; ++cb)
                            tma_load_3d_hint(sQ + q * S::Q_BYTES + cb * (BR * 128), &tm_q, bar(S::BAR_QFULL + q),
                                             cb * 64, r0[q], bh, pol_q);
                    }
                    ++uo[q];
                }
                for (int tt = 0; ok && tt < 2 * nkv_max; ++tt, ++t) {
                    const int slot = t % S::NS, round = t / S::NS;
                    if (round > 0 && !wwait(bar(S::BAR_EMPTY + slot), (round - 1) & 1, 1)) {
                        ok = false;
                        break;
                    }
                    if (leader) {
                        mbar_arrive_expect_tx(bar(S::BAR_FULL + slot), S::SLOT_BYTES);
                        const CUtensorMap *m = (tt & 1) ? &tm_v : &tm_k;
#pragma unroll
                        for (int cb = 0; cb < S::CB; ++cb)
                            tma_load_3d_hint(sRing + slot * S::SLOT_BYTES + cb * (BC * 128), m,
                                             bar(S::BAR_FULL + slot), cb * 64, kv_tile(tt >> 1) * BC, bh, pol_kv);
                    }
                }
            }
            // Drain: every copy this warp started has landed before the CTA
            // may exit (normally already true).
            for (int tt = max(0, t - S::NS); tt < t; ++tt)
                wwait(bar(S::BAR_FULL + tt % S::NS), (tt / S::NS) & 1, 2);
#pragma unroll
            for (int q = 0; q < NQ; ++q)
                if (uo[q] > 0) wwait(bar(S::BAR_QFULL + q), (uo[q] - 1) & 1, 3);
            __syncwarp();
        } else if (MASKED && warp == S::WARP_MASK) {
            // --------------------------------------------------------------
            // Key-mask operand: for each K tile, mask / scale of its keys as
            // hi + mid + lo (bf16 each, round to nearest: 24 bits in all, so
            // the float is exact), k = 0..2 of the slot's B operand.  A finite
            // value past the bf16 range is clamped to it; -inf stays -inf with
            // zero mid and lo.  Arrives on every slot's full barrier (V tiles
            // too: the ring depth may be odd), the next K tile's values
            // already fetched while the warp waits.
            // --------------------------------------------------------------
            constexpr int MPL = BC / 32;   // keys per lane
            int t = 0;                     // K/V tiles so far, all units (as the producer counts)
            bool ok = true;
            for (int u = 0; ok; ++u) {
                int item, part, nparts;
                if (!work_unit(p, cta, G, u, item, part, nparts)) break;
                if constexpr (BSPARSE) {
                    if (!wwait(bar(S::BAR_LIST + u % 3), (u / 3) & 1, 26)) {
                        ok = false;
                        break;
                    }
                }
                geometry(u, item, part, nparts);
                const float *mrow = p.key_mask + static_cast<size_t>(bh) * N;
                float mv[MPL];
                auto fetch = [&](int jj) {
                    const int key0 = kv_tile(jj) * BC;
#pragma unroll
                    for (int i = 0; i < MPL; ++i) {
                        const int key = key0 + 32 * i + lane;
                        mv[i] = 0.f;
                        if (key < N) asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(mv[i]) : "l"(mrow + key));
                    }
                };
                if (nkv_max > 0) fetch(0);
                for (int tt = 0; ok && tt < 2 * nkv_max; ++tt, ++t) {
                    const int slot = t % S::NS, round = t / S::NS;
                    if (round > 0 && !wwait(bar(S::BAR_EMPTY + slot), (round - 1) & 1, 5)) {
                        ok = false;
                        break;
                    }
                    if ((tt & 1) == 0) {
                        const uint32_t mop = sbase + S::OFF_MASK + S::MOP_ONES + slot * S::MOP_SLOT;
#pragma unroll
                        for (int i = 0; i < MPL; ++i) {
                            const int r = 32 * i + lane;
                            // (a product, not a quotient: a division by
                            // the IEEE routine takes its slow path for an
                            // infinite mask value, and one such key per warp
                            // made this warp gate the ring, ~7 %)
                            float w = mv[i] * p.inv_scale;
                            constexpr float kBf16Max = 3.3895313892515355e38f;
                            if (isinf(w) && !isinf(mv[i])) w = copysignf(kBf16Max, w);
                            uint32_t w0, w1;
                            if (isfinite(w)) {
                                const __nv_bfloat16 hi = __float2bfloat16_rn(w);
                                const float r1 = w - __bfloat162float(hi);
                                const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
                                const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
                                w0 = static_cast<uint32_t>(__bfloat16_as_ushort(hi)) |
                                     (static_cast<uint32_t>(__bfloat16_as_ushort(mid)) << 16);
                                w1 = static_cast<uint32_t>(__bfloat16_as_ushort(lo));
                            } else {
                                w0 = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(w)));
                                w1 = 0u;
                            }
                            asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(mop + (r >> 3) * 256 + (r & 7) * 16),
                                         "r"(w0), "r"(w1)
                                         : "memory");
                        }
                        fence_proxy_async_smem();   // read by the tensor core
                        __syncwarp();
                        if ((tt >> 1) + 1 < nkv_max) fetch((tt >> 1) + 1);
                    }
                    if (leader) mbar_arrive(bar(S::BAR_FULL + slot));
                }
            }
            __syncwarp();
        } else if (warp == S::WARP_MMA) {
            // --------------------------------------------------------------
            // MMA issuer (one elected lane)
            // --------------------------------------------------------------
            constexpr uint32_t idesc_s = idesc_bf16_f32(BR, BC, false, false);  // Q, K both K-major
            constexpr uint32_t idesc_o = idesc_bf16_f32(BR, D, false, true);    // P (TMEM), V MN-major
            // Descriptors differ only in their start-address field (bits
            // 0..13, address >> 4): build one base per operand and add.
            const uint64_t qdesc0 = sdesc_sw128(sQ, 16, 1024);
            const uint64_t kdesc0 = sdesc_sw128(sRing, 16, 1024);
            const uint64_t vdesc0 = sdesc_sw128(sRing, BC * 128, 1024);
            // key mask: the ones operand and slot 0's mask operand
            const uint64_t onesdesc = sdesc_kmajor_plain(sbase + S::OFF_MASK, 128, 256);
            const uint64_t mopdesc0 = sdesc_kmajor_plain(sbase + S::OFF_MASK + S::MOP_ONES, 128, 256);
            // Running counts over all units: K/V tiles (t_base: the unit's K_0),
            // S tiles of each query tile, and units in which each query tile ran.
            int t_base = 0;
            int sq[NQ], uo[NQ];
#pragma unroll
            for (int q = 0; q < NQ; ++q) sq[q] = uo[q] = 0;
            auto commit = [&](int b) {
                if (leader) tc_commit(bar(b));
            };
            // S_q(j) of the unit goes to S buffer (sq[q] + j) % NSB and is
            // signalled on that buffer's barrier; after the unit's last S_q,
            // Q_q may be reloaded.
            auto issue_s = [&](int q, int j, int nkvq) {
                const int b = (sq[q] + j) & (S::NSB - 1);
                const uint64_t a0 = qdesc0 + static_cast<uint64_t>((q * S::Q_BYTES) >> 4);
                const uint64_t b0 =
                    kdesc0 + static_cast<uint64_t>((((t_base + 2 * j) % S::NS) * S::SLOT_BYTES) >> 4);
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const int cb = kk >> 2, off = (kk & 3) * 32;
                        mma_bf16_ss(tmem + S::s_col(q, b), a0 + static_cast<uint64_t>((cb * (BR * 128) + off) >> 4),
                                    b0 + static_cast<uint64_t>((cb * (BC * 128) + off) >> 4), idesc_s,
                                    kk > 0 ? 1u : 0u);
                    }
                    if constexpr (MASKED)   // S += mask / scale
                        mma_bf16_ss(tmem + S::s_col(q, b), onesdesc,
                                    mopdesc0 + static_cast<uint64_t>((((t_base + 2 * j) % S::NS) * S::MOP_SLOT) >> 4),
                                    idesc_s, 1u);
                    tc_commit(bar(S::BAR_SFULL + q * S::NSB + b));
                }
                if (j == nkvq - 1) commit(S::BAR_QFREE + q);
            };
            // P_q V_j over K steps [BC/16 * h / NH, BC/16 * (h+1) / NH): half h of P,
            // which its warpgroup wrote over the first columns of its half of S
            constexpr int KPH = (BC / 16) / S::NH;   // K steps per half
            auto issue_pv = [&](int q, int j, int h) {
                const int b = (sq[q] + j) & (S::NSB - 1);
                const uint64_t b0 =
                    vdesc0 + static_cast<uint64_t>((((t_base + 2 * j + 1) % S::NS) * S::SLOT_BYTES) >> 4);
                if (leader) {
#pragma unroll
                    for (int kk = (BC / 16) * h / S::NH; kk < (BC / 16) * (h + 1) / S::NH; ++kk) {
                        mma_bf16_ts(tmem + S::o_col(q), tmem + S::s_col(q, b) + (kk / KPH) * (BC / S::NH) + (kk % KPH) * 8,
                                    b0 + static_cast<uint64_t>((kk * 2048) >> 4), idesc_o,
                                    (j > 0 || kk > 0) ? 1u : 0u);
                    }
                }
            };
            // Before the unit's first P_q V (which overwrites O_q): the previous
            // unit's epilogue has read O_q.  Then all of P_q(j).
            auto wait_p = [&](int q, int j) -> bool {
                if (j == 0 && uo[q] > 0 && !wwait(bar(S::BAR_OFREE + q), (uo[q] - 1) & 1, 16))
                    return false;
                const int g = sq[q] + j;
                if (!wwait(bar(S::BAR_PFULL + q * S::NSB + (g & (S::NSB - 1))), (g / S::NSB) & 1, 13))
                    return false;
                tc_fence_after();
                return true;
            };

            bool ok = true;
            for (int u = 0; ok; ++u) {
                int item, part, nparts;
                if (!work_unit(p, cta, G, u, item, part, nparts)) break;
                if constexpr (BSPARSE) {
                    if (!wwait(bar(S::BAR_LIST + u % 3), (u / 3) & 1, 26)) {
                        ok = false;
                        break;
                    }
                }
                geometry(u, item, part, nparts);
#pragma unroll
                for (int q = 0; q < NQ; ++q)
                    if (ok && nkv[q] > 0) ok = wwait(bar(S::BAR_QFULL + q), uo[q] & 1, 10);
                if (!ok) break;
                auto full_wait = [&](int tt, int site) -> bool {   // tile tt of the unit has landed
                    const int tg = t_base + tt;
                    if (!wwait(bar(S::BAR_FULL + tg % S::NS), (tg / S::NS) & 1, site)) return false;
                    tc_fence_after();
                    return true;
                };
                auto slot_of = [&](int tt) { return S::BAR_EMPTY + (t_base + tt) % S::NS; };

                // The loops over q and h have compile-time bounds and no early
                // exit, so q and h are constants after unrolling and the
                // per-tile counts stay in registers.
                if constexpr (S::DBS) {
                    // Two S buffers per query tile.  Order: S(0), S(1) for both
                    // tiles; then per step j: P_0 V_j, S_0(j+2), P_1 V_j, S_1(j+2).
                    // S_q(j+2) overwrites the buffer P_q(j) was read from, after it
                    // in the tensor pipe; it is ready long before the softmax wants
                    // it, so the softmax never waits for P V.
                    for (int jj = 0; ok && jj < 2 && jj < nkv_max; ++jj) {
                        if (!full_wait(2 * jj, 11)) {
                            ok = false;
                            break;
                        }
#pragma unroll
                        for (int q = 0; q < NQ; ++q)
                            if (jj < nkv[q]) issue_s(q, jj, nkv[q]);
                        commit(slot_of(2 * jj));
                    }
                    for (int j = 0; ok && j < nkv_max; ++j) {
                        if (!full_wait(2 * j + 1, 12)) {
                            ok = false;
                            break;
                        }
                        bool k_ready = false;
#pragma unroll
                        for (int q = 0; q < NQ; ++q) {
                            if (!ok || j >= nkv[q]) continue;
                            if (wait_p(q, j)) {
#pragma unroll
                                for (int h = 0; h < S::NH; ++h) issue_pv(q, j, h);
                            } else {
                                ok = false;
                            }
                            if (!ok) continue;
                            commit(S::BAR_PVDONE + q);
                            if (j == nkv[q] - 1) commit(S::BAR_OFULL + q);
                            if (j + 2 < nkv[q]) {
                                if (!k_ready) {
                                    if (!full_wait(2 * j + 4, 14)) {
                                        ok = false;
                                        continue;
                                    }
                                    k_ready = true;
                                }
                                issue_s(q, j + 2, nkv[q]);
                            }
                        }
                        commit(slot_of(2 * j + 1));               // V_j slot
                        if (k_ready) commit(slot_of(2 * j + 4));  // K_{j+2} slot
                    }
                } else {
                    if (ok && nkv_max > 0) {
                        ok = full_wait(0, 11);  // K_0
                        if (ok) {
#pragma unroll
                            for (int q = 0; q < NQ; ++q)
                                if (nkv[q] > 0) issue_s(q, 0, nkv[q]);
                            commit(slot_of(0));
                        }
                    }
                    for (int j = 0; ok && j < nkv_max; ++j) {
                        if (!full_wait(2 * j + 1, 12)) {
                            ok = false;
                            break;
                        }
                        bool k_ready = false;
#pragma unroll
                        for (int q = 0; q < NQ; ++q) {
                            if (!ok || j >= nkv[q]) continue;
                            if (wait_p(q, j)) {
#pragma unroll
                                for (int h = 0; h < S::NH; ++h) issue_pv(q, j, h);
                            } else {
                                ok = false;
                            }
                            if (!ok) continue;
                            if (j == nkv[q] - 1) commit(S::BAR_OFULL + q);
                            if (j + 1 < nkv[q]) {
                                if (!k_ready) {
                                    if (!full_wait(2 * j + 2, 14)) {
                                        ok = false;
                                        continue;
                                    }
                                    k_ready = true;
                                }
                                issue_s(q, j + 1, nkv[q]);
                            }
                        }
                        commit(slot_of(2 * j + 1));               // V_j slot
                        if (k_ready) commit(slot_of(2 * j + 2));  // K_{j+1} slot
                    }
                }
                t_base += 2 * nkv_max;
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    sq[q] += nkv[q];
                    uo[q] += nkv[q] > 0 ? 1 : 0;
                }
            }
            // Every MMA issued has completed before tensor memory is released.
            commit(S::BAR_DONE);
            wwait(bar(S::BAR_DONE), 0, 15);
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------------
        // Softmax warpgroup h of query tile q.  NH = 2: warpgroup h owns S
        // columns [BC/2*h, BC/2*(h+1)), the matching half of P (written over
        // the first BC/4 of those columns) and half of O's columns; the two
        // warpgroups of a tile agree on every row's reference maximum.
        // ------------------------------------------------------------------
        if constexpr (S::MOVE_REGS) regs_inc<S::REGS_SOFTMAX>();
        const int q = warp / (4 * S::NH);
        const int h = (warp >> 2) & (S::NH - 1);
        const int wq = warp & 3;
        // Row of this thread.  M = 128: lane l of warp w holds row 32w + l.
        // M = 64: lanes 0..15 of warp w hold rows 16w .. 16w+15.
        const bool active = (BR == 128) || (lane < 16);
        const int row_in = (BR == 128) ? wq * 32 + lane : wq * 16 + (lane & 15);
        const uint32_t t_lane = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tO = tmem + t_lane + S::o_col(q);
        const float sl2 = p.scale_log2;
        constexpr int CW = BC / S::NH;       // S columns of this warpgroup
        constexpr int OC = D / 32 / S::NH;   // 32-column chunks of O of this warpgroup
        bool ok = true;
        // per-row exchange slot of warpgroup hh of this tile; barrier of the pair
        auto xch = [&](int hh) -> uint32_t { return sbase + S::OFF_XCH + ((q * 2 + hh) * 128 + row_in) * 8; };
        auto pair_sync = [&]() { named_bar_sync(7 + q, 256); };
        // (a, b) of this row from the other warpgroup, after publishing our own
        // (M = 64: only the lane that carries the row writes its slot)
        auto exchange = [&](float a, float b, float &ao, float &bo) {
            if (active) asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(xch(h)), "f"(a), "f"(b) : "memory");
            pair_sync();
            asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(ao), "=f"(bo) : "r"(xch(1 - h)) : "memory");
        };
        int sq = 0;   // S tiles of this query tile so far, all units
        int uo = 0;   // units so far in which this query tile ran

        for (int u = 0;; ++u) {
            int item, part, nparts;
            if (!work_unit(p, cta, G, u, item, part, nparts)) break;
            if constexpr (BSPARSE) {
                // warp 1 lists this unit's key tiles (the first unit) and the
                // next unit's, while this one runs
                if (warp == 1) {
                    if (u == 0) build_list(0);
                    build_list(u + 1);
                }
                if (!wait_list(u)) ok = false;
            }
            geometry(u, item, part, nparts);
            // This tile's row offset and K/V tile count as plain registers (a
            // run-time index into r0[] / nkv[] would place them in local memory).
            int r0q = r0[0], nkvq = nkv[0];
#pragma unroll
            for (int i = 1; i < NQ; ++i)
                if (q == i) {
                    r0q = r0[i];
                    nkvq = nkv[i];
                }
            const int row = r0q + row_in;
            float m = kNegInf;    // reference maximum, log2 units (the same in both warpgroups)
            float l = 0.f;        // sum of the bf16-rounded p over this warpgroup's columns

            // A wait that gives up (the error word records it; every later wait
            // then gives up at once) does not end the loop: the tile is computed
            // from whatever tensor memory holds, so every warp still takes part in
            // every named barrier of the loop and no partner is left waiting.
            for (int j = 0; j < nkvq; ++j) {
                const int g = sq + j;              // this S tile's index over all units
                const int sb = g & (S::NSB - 1);   // S buffer of this tile
                if (!mbar_wait(bar(S::BAR_SFULL + q * S::NSB + sb), (g / S::NSB) & 1, abort_flag, p.err, 20)) ok = false;
                tc_fence_after();
                const uint32_t tS = tmem + t_lane + S::s_col(q, sb);
                const int key0 = kv_tile(j) * BC;
                // block-sparse: a listed tile not marked for this query tile is masked whole
                bool dead = false;
                if constexpr (BSPARSE) dead = !((kv_list[j] >> (14 + q)) & 1);
                // Tiles that need per-element masking: the N tail and the causal
                // diagonal.  (A key mask is already part of S.)
                const bool edge = dead || (key0 + BC > N) || (p.causal && key0 + BC - 1 > r0q);

                const bool diag = p.causal && key0 + BC - 1 > r0q;   // tile crosses the causal diagonal
                // One loaded 32-column chunk -> log2-domain scores
                // x = s*scale*log2(e), -inf where not allowed (past N, above
                // the causal diagonal, a dead block-sparse tile).
                auto mask_chunk = [&](int c, uint32_t *r) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int key = key0 + 32 * c + e;
                        float x = __uint_as_float(r[e]);
                        x = (key < N) ? x * sl2 : kNegInf;
                        if (diag) x = (key <= row) ? x : kNegInf;
                        if constexpr (BSPARSE) x = dead ? kNegInf : x;
                        r[e] = __float_as_uint(x);
                    }
                };
                auto chunk_max = [&](const uint32_t *r, float mx) {
#pragma unroll
                    for (int e = 0; e < 32; e += 2) mx = fmax3(mx, __uint_as_float(r[e]), __uint_as_float(r[e + 1]));
                    return mx;
                };
                // p = 2^(x - m_use) for one 32-column chunk, packed to bf16 pairs
                // and written to the 16 columns from pcol.  EDGE: the chunk is
                // already scaled and masked (a compile-time branch, so the
                // inner loop carries no select).
                // Partial sums per chunk keep the add chains short: sa / sb sum the
                // bf16-rounded p of the even / odd columns.
                auto exp_chunk = [&](auto edge_c, int pcol, const uint32_t *r, uint64_t negm2, float &sa, float &sb) {
                    constexpr bool EDGE = decltype(edge_c)::value;
                    const uint64_t sl2x2 = f2_pack(sl2, sl2);
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const uint64_t xx = f2_pack(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
                        uint64_t y;
                        if constexpr (EDGE) y = f2_add(xx, negm2);
                        else y = f2_fma(xx, sl2x2, negm2);
                        float y0, y1;
                        f2_unpack(y, y0, y1);
                        const float p0 = ex2(y0), p1 = ex2(y1);
                        uint32_t w = pack_bf16x2(p0, p1);
                        if (!active) w = 0u;
                        pk[e] = w;
                        add_bf16x2_f32(sa, sb, w);
                    }
                    tmem_st16(tS + pcol, pk);
                };

                // O_q *= alpha for this warp's rows and this warpgroup's columns
                // (warp-collective; alpha = 1 for rows whose reference did not move).
                auto rescale_o = [&](float alpha) {
                    const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
                    for (int c = h * OC; c < (h + 1) * OC; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tO + 32 * c, o);
                        tmem_ld_wait();
                        reg_fence32(o);
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const uint64_t v = f2_mul(f2_pack(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), a2);
                            float v0, v1;
                            f2_unpack(v, v0, v1);
                            o[e] = __float_as_uint(v0);
                            o[e + 1] = __float_as_uint(v1);
                        }
                        tmem_st32(tO + 32 * c, o);
                    }
                };

                // With two S buffers the P V of tile j-1 may still run: O_q holds
                // it only after that P V has completed.
                auto o_settled = [&]() {
                    if constexpr (S::DBS) {
                        mbar_wait(bar(S::BAR_PVDONE + q), (g - 1) & 1, abort_flag, p.err, 25);
                        tc_fence_after();
                    }
                };
                // This warpgroup's part of P_q is in tensor memory (and its part
                // of O rescaled): once both warpgroups have arrived, P_q V may
                // be issued.  (Each half of P V accumulates into all of O's
                // columns, so it must not start before both rescales.)
                auto release_p = [&]() {
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(bar(S::BAR_PFULL + q * S::NSB + sb));
                };
                constexpr int NC = CW / 32;   // 32-column chunks of this warpgroup
                if constexpr (NC <= 2) {
                    // One pass: this warpgroup's S columns stay in registers.
                    // The tile's row maximum comes with the loads (interior
                    // tiles) or after masking (edge tiles); two warpgroups
                    // exchange theirs.
                    uint32_t sr[NC][32];
                    float mxc[NC];
                    float mx = kNegInf;
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        if (edge) tmem_ld32(tS + h * CW + 32 * c, sr[c]);
                        else tmem_ld32_max(tS + h * CW + 32 * c, sr[c], mxc[c]);
                    }
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        reg_fence32(sr[c]);
                        if (!edge) reg_fence_f32(mxc[c]);
                        if (edge) {
                            mask_chunk(h * NC + c, sr[c]);
                            mx = chunk_max(sr[c], mx);
                        } else {
                            mx = fmaxf(mx, mxc[c]);
                        }
                    }
                    if (!edge) mx *= sl2;
                    if constexpr (S::NH == 2) {
                        // The row maximum over both halves is needed only if some
                        // row's half maximum would move the reference: one vote,
                        // and the exchange only then.
                        if (named_bar_red_or(7 + q, 256, active && mx > m + kRescaleThresh)) {
                            float mo, unused;
                            exchange(mx, 0.f, mo, unused);
                            mx = fmaxf(mx, mo);
                        } else {
                            mx = m;
                        }
                    }
                    // The reference moves only to a maximum more than
                    // kRescaleThresh above it (from -inf: to any finite
                    // maximum), so every p stays below 2^kRescaleThresh and O
                    // is rescaled only then.
                    const float m_new = (active && mx > m + kRescaleThresh) ? mx : m;
                    const bool moved = m_new != m;
                    const float a = moved ? ex2(m - m_new) : 1.f;
                    m = m_new;
                    const float m_use = (m == kNegInf) ? 0.f : m;
                    const uint64_t negm2 = f2_pack(-m_use, -m_use);
                    // P chunk c goes over this half's columns 16c .. 16c+15,
                    // already read into registers.
                    float ls = 0.f;
                    auto exps = [&](auto edge_c) {
#pragma unroll
                        for (int c = 0; c < NC; ++c) {
                            float sa = 0.f, sb = 0.f;
                            exp_chunk(edge_c, h * CW + 16 * c, sr[c], negm2, sa, sb);
                            ls += sa + sb;
                        }
                    };
                    if (edge) exps(std::true_type{});
                    else exps(std::false_type{});
                    // O_q takes the new reference before this tile's P V
                    // accumulates into it (S is no longer held).
                    if (j > 0 && __any_sync(0xffffffffu, moved)) {
                        o_settled();
                        rescale_o(a);
                    }
                    l = l * a + ls;
                    release_p();
                } else {
                    // Two passes (the columns do not fit in registers): the
                    // row maximum first, then the exponentials.
                    float mx = kNegInf;
#pragma unroll 1
                    for (int c = 0; c < NC; ++c) {
                        uint32_t sr[32];
                        float mc;
                        if (edge) {
                            tmem_ld32(tS + h * CW + 32 * c, sr);
                            tmem_ld_wait();
                            reg_fence32(sr);
                            mask_chunk(h * NC + c, sr);
                            mx = chunk_max(sr, mx);
                        } else {
                            tmem_ld32_max(tS + h * CW + 32 * c, sr, mc);
                            tmem_ld_wait();
                            reg_fence32(sr);
                            reg_fence_f32(mc);
                            mx = fmaxf(mx, mc);
                        }
                    }
                    if (!edge) mx *= sl2;
                    if constexpr (S::NH == 2) {
                        float mo, unused;
                        exchange(mx, 0.f, mo, unused);
                        mx = fmaxf(mx, mo);
                    }
                    const float m_new = (active && mx > m + kRescaleThresh) ? mx : m;
                    const bool moved = m_new != m;
                    const float a = moved ? ex2(m - m_new) : 1.f;
                    if (j > 0 && __any_sync(0xffffffffu, moved)) {
                        o_settled();
                        rescale_o(a);
                    }
                    m = m_new;
                    l *= a;
                    const float m_use = (m == kNegInf) ? 0.f : m;
                    const uint64_t negm2 = f2_pack(-m_use, -m_use);
                    // P chunk c goes over this half's columns 16c .. 16c+15,
                    // never ahead of the columns still to be read.
                    float ls = 0.f;
                    uint32_t sr[2][32];
                    tmem_ld32(tS + h * CW, sr[0]);
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        tmem_ld_wait();
                        reg_fence32(sr[c & 1]);
                        if (c + 1 < NC) tmem_ld32(tS + h * CW + 32 * (c + 1), sr[(c + 1) & 1]);
                        if (edge) mask_chunk(h * NC + c, sr[c & 1]);
                        float sa = 0.f, sb = 0.f;
                        if (edge) exp_chunk(std::true_type{}, h * CW + 16 * c, sr[c & 1], negm2, sa, sb);
                        else exp_chunk(std::false_type{}, h * CW + 16 * c, sr[c & 1], negm2, sa, sb);
                        ls += sa + sb;
                    }
                    l += ls;
                    release_p();
                }
            }

            // ---------------- epilogue ----------------
            // Two warpgroups per tile: each row's sum over all columns.
            if constexpr (S::NH == 2) {
                float lo, unused;
                pair_sync();   // the other warpgroup has read the last tile's exchange
                exchange(l, 0.f, lo, unused);
                l += lo;
                pair_sync();   // both have read it: the next unit may exchange again
            }
            if (nkvq > 0 && ok) ok = mbar_wait(bar(S::BAR_OFULL + q), uo & 1, abort_flag, p.err, 21);
            tc_fence_after();
            // Chunk c (32 columns) of this thread's row of O, times 1 / l, as
            // bf16: two 32-byte stores (whole sectors) when O is 32-byte aligned.
            const bool wide = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
            auto store_chunk = [&](int c, const uint32_t (&o)[32], uint64_t inv2, bool store) {
                __nv_bfloat16 *orow = p.o + (static_cast<size_t>(bh) * N + (store ? row : 0)) * D;
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const uint64_t v = f2_mul(f2_pack(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), inv2);
                    float v0, v1;
                    f2_unpack(v, v0, v1);
                    w[e] = pack_bf16x2(v0, v1);
                }
                if (store && wide) {
#pragma unroll
                    for (int k = 0; k < 2; ++k)
                        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(orow + 32 * c + 16 * k),
                                     "r"(w[8 * k]), "r"(w[8 * k + 1]), "r"(w[8 * k + 2]), "r"(w[8 * k + 3]),
                                     "r"(w[8 * k + 4]), "r"(w[8 * k + 5]), "r"(w[8 * k + 6]), "r"(w[8 * k + 7])
                                     : "memory");
                } else if (store) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(orow + 32 * c + 8 * k),
                                     "r"(w[4 * k]), "r"(w[4 * k + 1]), "r"(w[4 * k + 2]), "r"(w[4 * k + 3])
                                     : "memory");
                }
            };
            bool split_unit = false;
            if constexpr (S::CAN_SPLIT) {
                if (nparts > 1) {
                    // A split item: the parts swap their partial results
                    // (unnormalised O, m, l per row) through shared memory across
                    // the cluster.  Part r merges and stores the 32-column chunks c
                    // of O with c mod nparts = r (part 0 also the LSE), with the
                    // same rescale as between tiles: M = max_r m_r, weights
                    // 2^(m_r - M).  Every part forms l the same way (ranks in
                    // order), so a row's chunks share one normaliser.
                    split_unit = true;
                    const uint32_t sPart = sQ;   // partials live in the (now idle) Q tiles and K/V ring
                    // piece k of chunk c of this thread's row; the row's m (k = 0) and l (k = 1)
                    auto part_at = [&](int c, int k) { return sPart + (((q * (D / 32) + c) * 8 + k) * 128 + row_in) * 16; };
                    auto stat_addr = [&](int k) { return sPart + (NQ * 128 * D + k * NQ * 128 + q * 128 + row_in) * 4; };
                    // The ring is reused only after every MMA of the CTA (both query
                    // tiles) has completed: the other tile's last PV may still read V.
                    mbar_wait(bar(S::BAR_DONE), 0, abort_flag, p.err, 24);
                    tc_fence_after();
                    if (nkvq > 0) {
#pragma unroll
                        for (int c = h * OC; c < (h + 1) * OC; ++c) {
                            if ((c & (nparts - 1)) == part) continue;   // merged here
                            uint32_t o[32];
                            tmem_ld32(tO + 32 * c, o);
                            tmem_ld_wait();
                            reg_fence32(o);
#pragma unroll
                            for (int k = 0; k < 8; ++k)
                                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(part_at(c, k)),
                                             "r"(o[4 * k]), "r"(o[4 * k + 1]), "r"(o[4 * k + 2]), "r"(o[4 * k + 3])
                                             : "memory");
                        }
                    }
                    if (h == 0) {
                        asm volatile("st.shared.f32 [%0], %1;" ::"r"(stat_addr(0)), "f"(m) : "memory");
                        asm volatile("st.shared.f32 [%0], %1;" ::"r"(stat_addr(1)), "f"(l) : "memory");
                    }
#pragma unroll
                    for (int r = 0; r < 8; ++r)
                        if (r < nparts && r != part) mbar_arrive_remote(mapa_shared(bar(S::BAR_PART), r));
                    // This CTA's shared memory outlives the other parts' reads: every
                    // thread of every part meets at the cluster barrier at the end.
                    // A failed wait (the error word has it) reads no partial: the
                    // merge then has only this part's keys, and the O / LSE stores
                    // below are skipped because the abort flag is set.
                    // Every part's (m, l) is read in one round trip over the
                    // cluster (all loads issued before any is used).
                    const bool parts_ok = mbar_wait_cluster(bar(S::BAR_PART), 0, abort_flag, p.err, 23);
                    float mr[8], lr[8];
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        mr[r] = kNegInf;
                        lr[r] = 0.f;
                        if (r == part) {
                            mr[r] = m;
                            lr[r] = l;
                        } else if (parts_ok && r < nparts) {
                            mr[r] = ld_cluster_f32(mapa_shared(stat_addr(0), r));
                            lr[r] = ld_cluster_f32(mapa_shared(stat_addr(1), r));
                        }
                    }
                    float m_fin = mr[0];
#pragma unroll
                    for (int r = 1; r < 8; ++r) m_fin = fmaxf(m_fin, mr[r]);
                    float a_r[8];   // weight of part r's O (0: nothing to add)
                    float l_fin = 0.f, a_own = 0.f;
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        a_r[r] = (mr[r] == kNegInf || m_fin == kNegInf) ? 0.f : ex2(mr[r] - m_fin);
                        l_fin = r == 0 ? a_r[0] * lr[0] : l_fin + a_r[r] * lr[r];
                        if (r == part) a_own = a_r[r];
                    }
                    if (nkvq > 0) {
                        const bool any = l_fin > 0.f;
                        const float inv = any ? 1.f / l_fin : 0.f;
                        const bool store = active && row < N && !*abort_flag;
#pragma unroll
                        for (int c = h * OC; c < (h + 1) * OC; ++c) {
                            if ((c & (nparts - 1)) != part) continue;   // another part's chunk
                            uint32_t o[32];
                            tmem_ld32(tO + 32 * c, o);
                            tmem_ld_wait();
                            reg_fence32(o);
                            // O = a_part O_part + sum_r a_r O_r (the other parts' O read
                            // from their shared memory through the cluster)
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * a_own);
#pragma unroll
                            for (int r = 0; r < 8; ++r) {
                                const float ar = a_r[r];
                                if (r >= nparts || r == part || ar == 0.f) continue;
                                const uint32_t src = mapa_shared(part_at(c, 0), r);
                                // the chunk's 8 loads are issued before the first is used
                                float v[32];
#pragma unroll
                                for (int k = 0; k < 8; ++k)
                                    ld_cluster_v4(src + 128 * 16 * k, v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
#pragma unroll
                                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(fmaf(ar, v[e], __uint_as_float(o[e])));
                            }
                            store_chunk(c, o, f2_pack(inv, inv), store);
                        }
                        if (h == 0 && part == 0 && active && p.lse != nullptr && row < N && !*abort_flag)
                            p.lse[static_cast<size_t>(bh) * N + row] = any ? (m_fin + log2f(l_fin)) * kLn2 : kNegInf;
                    }
                }
            }
            if (!split_unit && nkvq > 0) {
                const bool any = l > 0.f;
                const float inv = any ? 1.f / l : 0.f;
                const uint64_t inv2 = f2_pack(inv, inv);
                const bool store = active && row < N && !*abort_flag;
#pragma unroll
                for (int c = h * OC; c < (h + 1) * OC; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tO + 32 * c, o);
                    tmem_ld_wait();
                    reg_fence32(o);
                    store_chunk(c, o, inv2, store);
                }
                if (h == 0 && active && p.lse != nullptr && row < N && !*abort_flag)
                    p.lse[static_cast<size_t>(bh) * N + row] = any ? (m + log2f(l)) * kLn2 : kNegInf;
            }
            if (nkvq > 0) {
                // The epilogue has read O_q: the next unit's first P V may overwrite it.
                tc_fence_before();
                mbar_arrive(bar(S::BAR_OFREE + q));
            }
            sq += nkvq;
            uo += nkvq > 0 ? 1 : 0;
        }   // work units
    }

    // The next kernel in the stream may be scheduled now (it waits for this
    // grid's completion before it touches global memory).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    if (warp == S::WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, S::TMEM_COLS);
    }
    if constexpr (S::CAN_SPLIT) {
        // Split item: no part exits while another part may still read its
        // shared memory.  Every thread reaches this point on every path (all
        // waits above are bounded), so the barrier always completes.
        if (p.split > 1) cluster_sync();
    }
}

constexpr int kMaxDev = 64;
std::mutex g_launch_mu;   // serialises the once-per-device set-up below

int sm_count(int dev) {
    static std::atomic<int> counts[kMaxDev];
    if (dev < 0 || dev >= kMaxDev) return 0;
    int n = counts[dev].load(std::memory_order_acquire);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        counts[dev].store(n, std::memory_order_release);
    }
    return n;
}

template <int D, int BR, int BC, int NQ, bool MASKED, bool BSPARSE = false>
int launch_variant(const void *Q, const void *K, const void *V, void *O, float *LSE, int BH, int N,
                   int causal, float scale, const float *key_mask, cudaStream_t stream, int *split_out,
                   const uint8_t *block_mask = nullptr) {
    using S = TcShape<D, BR, BC, NQ, MASKED, BSPARSE>;
    auto kern = attn_fwd_tc_kernel<D, BR, BC, NQ, MASKED, BSPARSE>;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return kErrCuda;
    // Once per device: the shared-memory opt-in, and how many clusters of 2,
    // 4 and 8 CTAs can be resident at once (a split tail is used only if
    // every cluster of it fits in one wave).
    static std::atomic<int> ready[kMaxDev];
    static int max_clusters[kMaxDev][4];
    if (ready[dev].load(std::memory_order_acquire) == 0) {
        std::lock_guard<std::mutex> lk(g_launch_mu);
        if (ready[dev].load(std::memory_order_relaxed) == 0) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM_BYTES) != cudaSuccess)
                return kErrCuda;
            if (S::MOVE_REGS) {
                // setmaxnreg moves registers within the launch allocation; the split
                // above is exact only for this per-thread count.
                cudaFuncAttributes fa;
                if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return kErrCuda;
                if (fa.numRegs != S::LAUNCH_REGS) return kErrUnsupported;
            }
            for (int i = 1; i < 4; ++i) {
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3(8u);
                cfg.blockDim = dim3(S::THREADS);
                cfg.dynamicSmemBytes = S::SMEM_BYTES;
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = 1u << i;
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = 1;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                int n = 0;
                if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
                    (void)cudaGetLastError();
                    n = 0;
                }
                max_clusters[dev][i] = n;
            }
            ready[dev].store(1, std::memory_order_release);
        }
    }
    CUtensorMap tq, tk, tv;
    if (!make_bf16_rows_map(&tq, Q, D, N, BH, BR) || !make_bf16_rows_map(&tk, K, D, N, BH, BC) ||
        !make_bf16_rows_map(&tv, V, D, N, BH, BC))
        return kErrCuda;
    TcParams p;
    p.N = N;
    p.BH = BH;
    p.num_qg = (N + NQ * BR - 1) / (NQ * BR);
    p.causal = causal;
    p.scale = scale;
    p.inv_scale = static_cast<float>(1.0 / static_cast<double>(scale));
    p.scale_log2 = scale * kLog2e;
    p.key_mask = key_mask;
    p.block_mask = block_mask;
    p.nkb = (N + 127) / 128;
    p.o = static_cast<__nv_bfloat16 *>(O);
    p.lse = LSE;
    p.err = device_error_word();
    if (!p.err) return kErrCuda;
    const long long items = static_cast<long long>(p.num_qg) * BH;
    if (items > 0x7fffffffLL) return kErrUnsupported;
    const int nsm = sm_count(dev);
    if (nsm <= 0) return kErrCuda;
    // Work: one CTA per SM, each running a list of work units (TcParams).
    // Non-causal items past the last full round are split along K/V into s
    // parts, s the largest power of two with s * (items mod SMs) <= SMs, run
    // by clusters of s CTAs; causal and block-sparse work stays unsplit.
    long long grid = std::min<long long>(items, nsm);
    long long n_full = items;
    int split = 1;
    if (S::CAN_SPLIT && !causal) {
        const long long R = items % nsm;
        const int nkv_all = (N + BC - 1) / BC;
        int sp = 1;
        while (R > 0 && sp * 2 <= 8 && sp * 2 * R <= nsm && sp * 2 <= nkv_all && nsm % (sp * 2) == 0) sp *= 2;
        const int si = sp == 8 ? 3 : sp == 4 ? 2 : sp == 2 ? 1 : 0;
        const long long g = (items - R > 0) ? nsm : R * sp;
        if (sp > 1 && static_cast<long long>(max_clusters[dev][si]) * sp >= g) {
            split = sp;
            n_full = items - R;
            grid = g;
        }
    }
    p.items = static_cast<int>(items);
    p.n_full = static_cast<int>(n_full);
    p.split = split;
    p.split_shift = split == 8 ? 3 : split == 4 ? 2 : split == 2 ? 1 : 0;
    if (split > 1) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(S::THREADS);
        cfg.dynamicSmemBytes = S::SMEM_BYTES;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(split);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        if (cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, p) == cudaSuccess) {
            if (split_out) *split_out = split;
            return kOk;
        }
        (void)cudaGetLastError();   // cluster not schedulable: run unsplit
        p.n_full = p.items;
        p.split = 1;
        p.split_shift = 0;
        grid = std::min<long long>(items, nsm);
    }
    if (split_out) *split_out = 1;
    // a programmatic dependent launch: its launch overlaps the end of the
    // kernel before it in the stream (an ordinary launch is the fallback)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(S::THREADS);
    cfg.dynamicSmemBytes = S::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, p) == cudaSuccess) return kOk;
    (void)cudaGetLastError();
    kern<<<static_cast<unsigned>(grid), S::THREADS, S::SMEM_BYTES, stream>>>(tq, tk, tv, p);
    return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

template <int D, int BR, int BC>
int launch_shape(const void *Q, const void *K, const void *V, void *O, float *LSE, int BH, int N, int causal,
                 float scale, const float *key_mask, cudaStream_t stream, const char **variant) {
    constexpr int NQ = (2 * (BC + D) <= 512) ? 2 : 1;
    static char names[2][4][64];
    int split = 1;
    const int rc = key_mask
        ? launch_variant<D, BR, BC, NQ, true>(Q, K, V, O, LSE, BH, N, causal, scale, key_mask, stream, &split)
        : launch_variant<D, BR, BC, NQ, false>(Q, K, V, O, LSE, BH, N, causal, scale, key_mask, stream, &split);
    const int si = split >= 8 ? 3 : split >= 4 ? 2 : split >= 2 ? 1 : 0;
    char *name = names[key_mask ? 1 : 0][si];
    snprintf(name, 64, "tc_bf16_d%d_br%d_bc%d_nq%d%s%s", D, BR, BC, NQ, key_mask ? "_mask" : "",
             si == 0 ? "" : si == 1 ? "_kvsplit2" : si == 2 ? "_kvsplit4" : "_kvsplit8");
    if (variant) *variant = name;
    return rc;
}

template <int D, int BR>
int launch_br(int Bc, const void *Q, const void *K, const void *V, void *O, float *LSE, int BH, int N, int causal,
              float scale, const float *key_mask, cudaStream_t stream, const char **variant) {
    switch (Bc) {
        case 64: return launch_shape<D, BR, 64>(Q, K, V, O, LSE, BH, N, causal, scale, key_mask, stream, variant);
        case 128: return launch_shape<D, BR, 128>(Q, K, V, O, LSE, BH, N, causal, scale, key_mask, stream, variant);
        case 256: return launch_shape<D, BR, 256>(Q, K, V, O, LSE, BH, N, causal, scale, key_mask, stream, variant);
        default: return kErrUnsupported;
    }
}

}  // namespace

int launch_fwd_tc_bf16_bsparse(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                               int N, int d, int causal, float scale, const uint8_t *block_mask,
                               const float *key_mask, cudaStream_t stream, const char **variant) {
    const int BH = B * H;
    int split = 1;
    int rc;
    if (d == 128) {
        rc = key_mask ? launch_variant<128, 128, 128, 2, true, true>(Q, K, V, O, LSE, BH, N, causal, scale, key_mask,
                                                                     stream, &split, block_mask)
                      : launch_variant<128, 128, 128, 2, false, true>(Q, K, V, O, LSE, BH, N, causal, scale, key_mask,
                                                                      stream, &split, block_mask);
        if (variant) *variant = key_mask ? "tc_bf16_d128_br128_bc128_nq2_mask_bsparse" : "tc_bf16_d128_br128_bc128_nq2_bsparse";
    } else if (d == 64) {
        rc = key_mask ? launch_variant<64, 128, 128, 2, true, true>(Q, K, V, O, LSE, BH, N, causal, scale, key_mask,
                                                                    stream, &split, block_mask)
                      : launch_variant<64, 128, 128, 2, false, true>(Q, K, V, O, LSE, BH, N, causal, scale, key_mask,
                                                                     stream, &split, block_mask);
        if (variant) *variant = key_mask ? "tc_bf16_d64_br128_bc128_nq2_mask_bsparse" : "tc_bf16_d64_br128_bc128_nq2_bsparse";
    } else {
        return kErrUnsupported;
    }
    return rc;
}

int launch_fwd_tc_bf16(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H, int N,
                       int d, int causal, float scale, int Br, int Bc, const float *key_mask,
                       cudaStream_t stream, const char **variant) {
    if (Br == 0) Br = 128;
    if (Bc == 0) Bc = 128;
    const int BH = B * H;
    if (d == 64 && Br == 128) return launch_br<64, 128>(Bc, Q, K, V, O, LSE, BH, N, causal, scale, key_mask, stream, variant);
    if (d == 64 && Br == 64) return launch_br<64, 64>(Bc, Q, K, V, O, LSE, BH, N, causal, scale, key_mask, stream, variant);
    if (d == 128 && Br == 128) return launch_br<128, 128>(Bc, Q, K, V, O, LSE, BH, N, causal, scale, key_mask, stream, variant);
    if (d == 128 && Br == 64) return launch_br<128, 64>(Bc, Q, K, V, O, LSE, BH, N, causal, scale, key_mask, stream, variant);
    return kErrUnsupported;
}

}  // namespace eta
