// Decode with a key/value cache: attention of a few new query rows against a
// long cache of keys and values.  The same exact attention as the tiled
// forward ("Is Flash Attention Stable?" §II-A), split over the keys: every
// CTA reduces one chunk of the cache to a partial result (running maximum m,
// denominator l, unnormalised output o, as in the yadro-code.ru tutorial's
// online merge), and the partials are merged with the tutorial's rule for
// joining two blocks: common maximum M, weights 2^(m - M).
//
// With a handful of query rows the work is a stream over K and V (a few
// FLOPs per byte), so this path is HBM-bound and runs on the CUDA cores:
//   partial kernel, grid (splits, B*H); per CTA one producer warp and four
//     consumer warps.  The producer streams the chunk's keys, 32 at a time,
//     into a ring of shared-memory stages with bulk copies (the K rows and
//     the V rows of 32 keys are two contiguous runs).  A consumer warp takes
//     one stage: the lanes split d; each lane's partial dot products for the
//     32 keys are summed across lanes by a butterfly that leaves key `lane`'s
//     score in lane `lane`; a warp-wide maximum and sum per query row; then
//     O += P V with each key's probability broadcast by shuffle.  The
//     consumers' states are merged in shared memory; one partial per (split,
//     b, h, row) goes to the workspace (or straight to O and LSE when there is
//     one split).
//   merge kernel, one CTA per (b, h, row), 128 threads.
// Causal decoding: query row i is the token at position Nk - Nq + i and sees
// keys j <= Nk - Nq + i.
#include <cuda_bf16.h>
#include <cmath>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace eta {
namespace {

constexpr int kDecWarps = 4;     // consumer warps per CTA (plus one producer warp)
constexpr int kDecMaxStages = 8; // ring stages of 32 keys (K rows and V rows): 8, or 4 if 8 do not fit
// Group t goes to stage t % stages and to consumer warp t % kDecWarps: with the
// stage count a multiple of the warp count every stage has one consumer, which
// takes its groups in order, so a phase-parity wait on a stage can never see
// an older phase of another warp's group as complete.
static_assert(kDecMaxStages % kDecWarps == 0 && (kDecMaxStages / 2) % kDecWarps == 0, "one consumer warp per stage");
constexpr float kLog2eD = 1.4426950408889634f;
constexpr float kLn2D = 0.6931471805599453f;

struct DecParams {
    const void *Q, *K, *V;
    void *O;
    float *LSE;
    const float *key_mask;
    int BH, Nq, Nk, d, causal, bf16;
    float scale_log2;
    int splits, chunk, stages;
    float *pm, *pl, *po;   // partials [splits][BH][Nq] and [splits][BH][Nq][d]
    int *err;              // device error word (bounded waits)
};

// 8 consecutive elements of a row, as float
__device__ __forceinline__ void load8(const void *base, int bf16, long long idx, float *f) {
    if (bf16) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(base) + idx));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            f[2 * e] = __uint_as_float(w[e] << 16);
            f[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
        }
    } else {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(base) + idx));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(base) + idx + 4));
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
}

// E consecutive elements (E = d / 32: 1, 2, 3 or 4), as float
template <int E>
__device__ __forceinline__ void loadE(const void *base, int bf16, long long idx, float *f) {
    if (bf16) {
        const __nv_bfloat16 *p = static_cast<const __nv_bfloat16 *>(base) + idx;
        if constexpr (E == 4) {   // 8 bytes, aligned: idx is a multiple of 4
            const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
            f[0] = __uint_as_float(u.x << 16);
            f[1] = __uint_as_float(u.x & 0xFFFF0000u);
            f[2] = __uint_as_float(u.y << 16);
            f[3] = __uint_as_float(u.y & 0xFFFF0000u);
        } else if constexpr (E == 2) {   // 4 bytes, aligned
            const uint32_t u = __ldg(reinterpret_cast<const unsigned int *>(p));
            f[0] = __uint_as_float(u << 16);
            f[1] = __uint_as_float(u & 0xFFFF0000u);
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) f[e] = __bfloat162float(p[e]);
        }
    } else {
        const float *p = static_cast<const float *>(base) + idx;
#pragma unroll
        for (int e = 0; e < E; ++e) f[e] = __ldg(p + e);
    }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ void store_out(void *O, int bf16, long long idx, float v) {
    if (bf16) static_cast<__nv_bfloat16 *>(O)[idx] = __float2bfloat16_rn(v);
    else static_cast<float *>(O)[idx] = v;
}

// NQ: the number of query rows (compile time), E = d / 32.
// Warp kDecWarps is the producer: one lane streams the chunk's keys in groups
// of 32 (the K rows and the V rows of a group are two contiguous runs of
// memory) into a ring of shared-memory stages with bulk copies.
// Consumer warp w takes groups w, w + kDecWarps, ...
template <int NQ, int E>
__global__ void __launch_bounds__(32 * (kDecWarps + 1)) decode_partial_kernel(const DecParams p) {
    constexpr int D = 32 * E;
    extern __shared__ __align__(128) unsigned char dsm[];
    const int elt = p.bf16 ? 2 : 4;
    const int group_bytes = 32 * D * elt;                    // one group of K (or V) rows
    const int NS = p.stages;
    unsigned char *stage0 = dsm;                             // [NS][K group | V group]
    float *qs = reinterpret_cast<float *>(dsm + NS * 2 * group_bytes);   // [NQ][D]
    float *wm = qs + NQ * D;                                  // [kDecWarps][NQ]
    float *wl = wm + kDecWarps * NQ;                          // [kDecWarps][NQ]
    float *wo = wl + kDecWarps * NQ;                          // [kDecWarps][NQ][D]
    uint64_t *bars = reinterpret_cast<uint64_t *>(wo + kDecWarps * NQ * D);   // full[S], empty[S]
    __shared__ uint32_t abort_flag;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + NS);
    const int split = blockIdx.x, bh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k0 = split * p.chunk;
    const int k1 = min(k0 + p.chunk, p.Nk);
    const int ngroups = (k1 - k0 + 31) / 32;
    const long long qbase = static_cast<long long>(bh) * NQ * D;
    const long long kvrow0 = static_cast<long long>(bh) * p.Nk + k0;   // first key row of the chunk
    if (threadIdx.x == 0) {
        for (int st = 0; st < NS; ++st) {
            mbar_init(full0 + 8 * st, 1);
            mbar_init(empty0 + 8 * st, 1);
        }
        abort_flag = 0u;
        fence_mbar_init();
    }
    // Launched as a programmatic dependent of the kernel before it in the
    // stream: no global memory is touched before that grid has completed.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int t = threadIdx.x; t < NQ * D; t += blockDim.x) {
        float f[1];
        loadE<1>(p.Q, p.bf16, qbase + t, f);
        qs[t] = f[0];
    }
    __syncthreads();
    volatile uint32_t *abortp = &abort_flag;

    if (warp == kDecWarps) {
        // producer: one lane issues every copy
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();   // the cache is read once
            int issued = 0;
            for (int t = 0; t < ngroups; ++t) {
                const int st = t % NS;
                if (t >= NS && !mbar_wait(empty0 + 8 * st, ((t / NS) - 1) & 1, abortp, p.err, 40))
                    break;
                const int nk = min(32, k1 - k0 - 32 * t);
                const uint32_t bytes = static_cast<uint32_t>(nk * D * elt);
                const long long row = kvrow0 + 32LL * t;
                const uint32_t dst = smem_u32(stage0 + st * 2 * group_bytes);
                mbar_arrive_expect_tx(full0 + 8 * st, 2 * bytes);
                bulk_load(dst, static_cast<const unsigned char *>(p.K) + row * D * elt, bytes, full0 + 8 * st, pol);
                bulk_load(dst + group_bytes, static_cast<const unsigned char *>(p.V) + row * D * elt, bytes,
                          full0 + 8 * st, pol);
                issued = t + 1;
            }
            // every copy has landed before this thread leaves (normally the
            // consumers have seen them all already)
            for (int t = max(0, issued - NS); t < issued; ++t)
                mbar_wait(full0 + 8 * (t % NS), (t / NS) & 1, abortp, p.err, 42);
        }
        __syncwarp();
        return;
    }

    // consumer warp: lane owns columns [E*lane, E*lane + E) of q, o and the rows
    float qr[NQ][E];
#pragma unroll
    for (int i = 0; i < NQ; ++i)
#pragma unroll
        for (int e = 0; e < E; ++e) qr[i][e] = qs[i * D + E * lane + e];
    float m[NQ], l[NQ], o[NQ][E];
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) o[i][e] = 0.f;
    }
    auto row_vals = [&](const unsigned char *base, int jj, float *f) {   // E values of row jj from shared memory
        if (p.bf16) {
            const __nv_bfloat16 *r = reinterpret_cast<const __nv_bfloat16 *>(base) + jj * D + E * lane;
#pragma unroll
            for (int e = 0; e < E; ++e) f[e] = __bfloat162float(r[e]);
        } else {
            const float *r = reinterpret_cast<const float *>(base) + jj * D + E * lane;
#pragma unroll
            for (int e = 0; e < E; ++e) f[e] = r[e];
        }
    };
    for (int t = warp; t < ngroups; t += kDecWarps) {
        const int st = t % NS;
        if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * st, (t / NS) & 1, abortp, p.err, 41))) break;
        const unsigned char *kb = stage0 + st * 2 * group_bytes;
        const unsigned char *vb = kb + group_bytes;
        const int g = k0 + 32 * t;
        const int nk = min(32, k1 - g);
        const int j = g + lane;   // the key whose score this lane ends up holding
        float pr[NQ];
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            // partial dot products of every key of the group over this lane's
            // columns, then a butterfly that leaves key `lane`'s full sum in
            // lane `lane` (each step keeps the half of the keys whose index bit
            // matches the lane's and adds the partner's other half)
            float part[32];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                float kf[E];
                if (jj < nk) {
                    row_vals(kb, jj, kf);
                } else {
#pragma unroll
                    for (int e = 0; e < E; ++e) kf[e] = 0.f;
                }
                float acc = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) acc = fmaf(qr[i][e], kf[e], acc);
                part[jj] = acc;
            }
#pragma unroll
            for (int w = 16; w >= 1; w >>= 1) {
                const bool upper = (lane & w) != 0;
#pragma unroll
                for (int a = 0; a < w; ++a) {
                    // keep index a + (upper ? w : 0), send the other one
                    const float keep = upper ? part[a + w] : part[a];
                    const float send = upper ? part[a] : part[a + w];
                    part[a] = keep + __shfl_xor_sync(0xffffffffu, send, w);
                }
            }
            const bool valid = lane < nk;
            const float mk = (valid && p.key_mask) ? p.key_mask[static_cast<long long>(bh) * p.Nk + j] * kLog2eD : 0.f;
            float x = valid ? fmaf(part[0], p.scale_log2, mk) : -INFINITY;
            if (p.causal && j > p.Nk - p.Nq + i) x = -INFINITY;
            const float mnew = fmaxf(m[i], warp_max(x));
            const float mu = (mnew == -INFINITY) ? 0.f : mnew;
            const float alpha = (m[i] == -INFINITY) ? 0.f : ex2(m[i] - mu);
            pr[i] = ex2(x - mu);   // 0 for -inf
            l[i] = l[i] * alpha + warp_sum(pr[i]);
#pragma unroll
            for (int e = 0; e < E; ++e) o[i][e] *= alpha;
            m[i] = mnew;
        }
        // O += P V with each key's probability broadcast from its lane
        for (int jj = 0; jj < nk; ++jj) {
            float vf[E];
            row_vals(vb, jj, vf);
#pragma unroll
            for (int i = 0; i < NQ; ++i) {
                const float pj = __shfl_sync(0xffffffffu, pr[i], jj);
#pragma unroll
                for (int e = 0; e < E; ++e) o[i][e] = fmaf(pj, vf[e], o[i][e]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * st);   // this stage may be refilled
    }
    // merge the consumer warps: common maximum, weights 2^(m_w - M)
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        if (lane == 0) {
            wm[warp * NQ + i] = m[i];
            wl[warp * NQ + i] = l[i];
        }
#pragma unroll
        for (int e = 0; e < E; ++e) wo[(warp * NQ + i) * D + E * lane + e] = o[i][e];
    }
    named_bar_sync(1, 32 * kDecWarps);
    for (int t = threadIdx.x; t < NQ * D; t += 32 * kDecWarps) {
        const int i = t / D, c = t % D;
        float M = -INFINITY;
        for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, wm[w * NQ + i]);
        const float mu = (M == -INFINITY) ? 0.f : M;
        float L = 0.f, acc = 0.f;
        for (int w = 0; w < kDecWarps; ++w) {
            const float a = (wm[w * NQ + i] == -INFINITY) ? 0.f : ex2(wm[w * NQ + i] - mu);
            L += a * wl[w * NQ + i];
            acc += a * wo[(w * NQ + i) * D + c];
        }
        const long long row = static_cast<long long>(bh) * NQ + i;
        if (p.splits == 1) {
            store_out(p.O, p.bf16, row * D + c, L > 0.f ? acc / L : 0.f);
            if (c == 0 && p.LSE) p.LSE[row] = L > 0.f ? (M + log2f(L)) * kLn2D : -INFINITY;
        } else {
            const long long prow = static_cast<long long>(split) * p.BH * NQ + row;
            p.po[prow * D + c] = acc;
            if (c == 0) {
                p.pm[prow] = M;
                p.pl[prow] = L;
            }
        }
    }
    // The merge kernel (a programmatic dependent launch) may be scheduled now;
    // it waits for this grid's completion before it reads a partial.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// one CTA per (b, h, row): merge the splits' partials.  Every split's (m, l)
// is read in one round trip and the weights 2^(m_s - M) kept in shared
// memory; the per-column sums over the splits load eight splits' values
// before using the first (a dependent load per split made the merge a chain
// of round trips), and add them in split order.
__global__ void __launch_bounds__(128) decode_merge_kernel(const DecParams p) {
    __shared__ float wsh[kDecodeMaxSplits];
    __shared__ float red[4];
    // Launched as a programmatic dependent of the partial kernel: wait until
    // that grid has completed and its writes are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const long long row = blockIdx.x;   // bh * Nq + i
    const long long nrow = static_cast<long long>(p.BH) * p.Nq;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const float ms = t < p.splits ? p.pm[t * nrow + row] : -INFINITY;
    const float ls = t < p.splits ? p.pl[t * nrow + row] : 0.f;
    float M = warp_max(ms);
    if (lane == 0) red[warp] = M;
    __syncthreads();
    M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    __syncthreads();
    const float mu = (M == -INFINITY) ? 0.f : M;
    const float w = (ms == -INFINITY) ? 0.f : ex2(ms - mu);
    if (t < p.splits) wsh[t] = w;
    float L = warp_sum(t < p.splits ? w * ls : 0.f);
    if (lane == 0) red[warp] = L;
    __syncthreads();
    L = red[0] + red[1] + red[2] + red[3];
    for (int c = t; c < p.d; c += blockDim.x) {
        float acc = 0.f;
        for (int s0 = 0; s0 < p.splits; s0 += 8) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = s0 + u < p.splits ? p.po[((s0 + u) * nrow + row) * p.d + c] : 0.f;
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (s0 + u < p.splits) acc += wsh[s0 + u] * v[u];
        }
        store_out(p.O, p.bf16, row * p.d + c, L > 0.f ? acc / L : 0.f);
    }
    if (t == 0 && p.LSE) p.LSE[row] = L > 0.f ? (M + log2f(L)) * kLn2D : -INFINITY;
    // the next call's partial kernel may be scheduled now (it waits for this grid)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <int NQ, int E>
size_t partial_smem(int bf16, int stages) {
    const size_t group = 32 * 32 * E * (bf16 ? 2 : 4);
    return stages * 2 * group + (NQ * 32 * E + 2 * kDecWarps * NQ + kDecWarps * NQ * 32 * E) * sizeof(float) +
           2 * stages * sizeof(uint64_t);
}

// Splits of the cache (and the keys per split) for a grid of BH x splits
// CTAs, `slots` of which are resident at once.  Every CTA streams the same
// number of keys, so CTAs run in waves, and a part-filled last wave leaves
// SMs idle while the rest of the grid waits for it.  Take the fewest splits
// that fill whole waves to at least 95% (fewer, longer CTAs pay the start-up
// and the merge less often); else the best filling.  At least 256 keys per
// split, at most kDecodeMaxSplits.  Measured on 1x32 heads x 32768 keys: 14
// splits (one wave of 448 CTAs) 84.9 us, 28 (1.96 waves) 87.4, 38 (2.67
// waves) 91.3, 19 (1.33 waves) 105.1.
void choose_splits(DecParams &p, int slots) {
    const int cap = std::max(1, std::min((p.Nk + 255) / 256, kDecodeMaxSplits));
    int best = 1, best_chunk = p.Nk;
    double best_fill = -1.0;
    for (int s = 1; s <= cap; ++s) {
        const int chunk = ((p.Nk + s - 1) / s + 31) / 32 * 32;
        const int splits = (p.Nk + chunk - 1) / chunk;   // no empty split after rounding the chunk up
        const long long ctas = static_cast<long long>(p.BH) * splits;
        const long long waves = (ctas + slots - 1) / slots;
        const double fill = static_cast<double>(ctas) / static_cast<double>(waves * slots);
        if (fill > best_fill + 1e-9) {
            best_fill = fill;
            best = splits;
            best_chunk = chunk;
        }
        if (fill >= 0.95) break;
    }
    p.splits = best;
    p.chunk = best_chunk;
}

template <int NQ, int E>
int launch_partial(DecParams &p, cudaStream_t stream) {
    // deep ring only while two CTAs still fit on an SM (one CTA's start-up
    // then overlaps another's stream)
    p.stages = kDecMaxStages;
    if (partial_smem<NQ, E>(p.bf16, p.stages) > 100 * 1024) p.stages = kDecMaxStages / 2;
    const size_t smem = partial_smem<NQ, E>(p.bf16, p.stages);
    const int threads = 32 * (kDecWarps + 1);
    if (cudaFuncSetAttribute(decode_partial_kernel<NQ, E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return kErrCuda;
    int dev = 0, nsm = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_partial_kernel<NQ, E>, threads, smem) !=
            cudaSuccess)
        return kErrCuda;
    choose_splits(p, std::max(1, per_sm) * std::max(1, nsm));
    // a programmatic dependent launch (an ordinary launch is the fallback)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.splits), static_cast<unsigned>(p.BH));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, decode_partial_kernel<NQ, E>, p) != cudaSuccess) {
        (void)cudaGetLastError();
        decode_partial_kernel<NQ, E><<<dim3(p.splits, p.BH), threads, smem, stream>>>(p);
    }
    return kOk;
}

template <int NQ>
int launch_nq(DecParams &p, cudaStream_t stream) {
    switch (p.d) {
        case 32: return launch_partial<NQ, 1>(p, stream);
        case 64: return launch_partial<NQ, 2>(p, stream);
        case 96: return launch_partial<NQ, 3>(p, stream);
        case 128: return launch_partial<NQ, 4>(p, stream);
        default: return kErrUnsupported;
    }
}

}  // namespace

size_t decode_workspace_bytes(int BH, int Nq, int d) {
    const size_t rows = static_cast<size_t>(kDecodeMaxSplits) * BH * Nq;
    return rows * (2 + static_cast<size_t>(d)) * sizeof(float);
}

int launch_decode(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H, int Nq, int Nk,
                  int d, int causal, float scale, int bf16, const float *key_mask, void *workspace,
                  cudaStream_t stream) {
    DecParams p;
    p.Q = Q;
    p.K = K;
    p.V = V;
    p.O = O;
    p.LSE = LSE;
    p.key_mask = key_mask;
    p.BH = B * H;
    p.Nq = Nq;
    p.Nk = Nk;
    p.d = d;
    p.causal = causal;
    p.bf16 = bf16;
    p.scale_log2 = scale * kLog2eD;
    p.err = device_error_word();
    if (!p.err) return kErrCuda;
    p.splits = 1;   // set with the chunk by the launch (choose_splits)
    p.chunk = Nk;
    const size_t rows = static_cast<size_t>(kDecodeMaxSplits) * p.BH * Nq;
    float *ws = static_cast<float *>(workspace);
    p.pm = ws;
    p.pl = ws + rows;
    p.po = ws + 2 * rows;
    int rc;
    switch (Nq) {
        case 1: rc = launch_nq<1>(p, stream); break;
        case 2: rc = launch_nq<2>(p, stream); break;
        case 3: rc = launch_nq<3>(p, stream); break;
        case 4: rc = launch_nq<4>(p, stream); break;
        case 5: rc = launch_nq<5>(p, stream); break;
        case 6: rc = launch_nq<6>(p, stream); break;
        case 7: rc = launch_nq<7>(p, stream); break;
        case 8: rc = launch_nq<8>(p, stream); break;
        default: return kErrUnsupported;
    }
    if (rc != kOk) return rc;
    if (cudaGetLastError() != cudaSuccess) return kErrCuda;
    if (p.splits > 1) {
        // programmatic dependent launch: the merge grid's launch overlaps the
        // end of the partial grid (the kernel waits for it, griddepcontrol)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(p.BH * Nq));
        cfg.blockDim = dim3(128);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, decode_merge_kernel, p) != cudaSuccess) {
            (void)cudaGetLastError();   // not available: an ordinary launch (the wait is then a no-op)
            decode_merge_kernel<<<static_cast<unsigned>(p.BH * Nq), 128, 0, stream>>>(p);
            if (cudaGetLastError() != cudaSuccess) return kErrCuda;
        }
    }
    return kOk;
}

}  // namespace eta
