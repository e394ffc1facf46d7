// Gradients of exact attention in true float32 on the CUDA cores.
//
// The same gradients as the tensor-core backward (the chain rule through the
// softmax of "Is Flash Attention Stable?" §II-A's attention; the weights
// recomputed from the forward's LSE, as the yadro-code.ru FlashAttention
// tutorial describes for the method's backward pass), with every operation
// in IEEE float32, no TF32 and no atomics:
//   prep     D_i = sum_c dO_ic O_ic per query row (into the workspace)
//   dkdv     one CTA of 8 warps per 64-key tile of one (batch, head); query
//            tiles of 64 rows staged in shared memory; each warp owns 8 keys:
//            lane t forms P and dS for queries t and t+32 of the tile, and
//            lane t accumulates dims t, t+32, t+64, t+96 of dV and dK
//   dq       one CTA of 8 warps per 64-query tile; K/V tiles staged; each
//            warp owns 8 query rows: lane t forms dS for keys t and t+32 and
//            accumulates dims t, t+32, ... of dQ
// P = exp(s - LSE) with s in natural-log units (expf); a row whose LSE is
// -inf (no allowed key) has P = 0.
#include <cmath>

#include "internal.h"

namespace eta {
namespace {

constexpr int kTile = 64;   // query rows or keys per tile
constexpr int kWarpsB = 8;
constexpr int kPerWarp = kTile / kWarpsB;

__global__ void bwd_f32_prep_kernel(const float *__restrict__ O, const float *__restrict__ dO, float *__restrict__ Dv,
                                    long long rows, int d) {
    const long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    float acc = 0.f;
    for (int c = lane; c < d; c += 32) acc = fmaf(O[r * d + c], dO[r * d + c], acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) Dv[r] = acc;
}

// P and dS of (query q, key k) from the score's pieces; 0 where not allowed.
__device__ __forceinline__ void p_ds(float dot, float dpv, float mask_k, float lse_q, float d_q, float scale,
                                     bool allowed, float &p, float &ds) {
    const float s = fmaf(dot, scale, mask_k);
    p = (allowed && lse_q != -INFINITY) ? expf(s - lse_q) : 0.f;
    ds = p * (dpv - d_q);
}

template <int DPL>
__global__ void __launch_bounds__(kWarpsB * 32)
    bwd_f32_dkdv_kernel(const float *__restrict__ Q, const float *__restrict__ K, const float *__restrict__ V,
                        const float *__restrict__ dO, const float *__restrict__ LSE, const float *__restrict__ Dv,
                        float *__restrict__ dK, float *__restrict__ dV, int N, int d, int causal, float scale,
                        const float *__restrict__ key_mask) {
    extern __shared__ float sm[];
    const int ld = d + 1;               // padded row stride: lane t reads row t, column c without conflicts
    float *Qs = sm;                      // [kTile][d+1]
    float *dOs = Qs + kTile * ld;        // [kTile][d+1]
    float *Ls = dOs + kTile * ld;        // [kTile] LSE of the tile's rows (-inf past N)
    float *Ds = Ls + kTile;              // [kTile] D of the tile's rows
    const int ntk = (N + kTile - 1) / kTile;
    const int bh = blockIdx.x / ntk;
    const int key0 = (blockIdx.x % ntk) * kTile;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t head = static_cast<size_t>(bh) * N * d;

    float kreg[kPerWarp][DPL], vreg[kPerWarp][DPL], mk[kPerWarp];
    float adk[kPerWarp][DPL], adv[kPerWarp][DPL];
#pragma unroll
    for (int r = 0; r < kPerWarp; ++r) {
        const int key = key0 + warp * kPerWarp + r;
        mk[r] = (key < N) ? (key_mask ? key_mask[static_cast<size_t>(bh) * N + key] : 0.f) : -INFINITY;
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
            const int c = lane + 32 * e;
            const bool in = key < N && c < d;
            kreg[r][e] = in ? K[head + static_cast<size_t>(key) * d + c] : 0.f;
            vreg[r][e] = in ? V[head + static_cast<size_t>(key) * d + c] : 0.f;
            adk[r][e] = 0.f;
            adv[r][e] = 0.f;
        }
    }
    const int qt0 = causal ? key0 / kTile : 0;
    const int nqt = (N + kTile - 1) / kTile;
    for (int qt = qt0; qt < nqt; ++qt) {
        const int q0 = qt * kTile;
        __syncthreads();
        for (int i = threadIdx.x; i < kTile * d; i += blockDim.x) {
            const int r = i / d, c = i % d;
            const bool in = q0 + r < N;
            const size_t g = head + static_cast<size_t>(q0 + r) * d + c;
            Qs[r * ld + c] = in ? Q[g] : 0.f;
            dOs[r * ld + c] = in ? dO[g] : 0.f;
        }
        for (int i = threadIdx.x; i < kTile; i += blockDim.x) {
            const bool in = q0 + i < N;
            Ls[i] = in ? LSE[static_cast<size_t>(bh) * N + q0 + i] : -INFINITY;
            Ds[i] = in ? Dv[static_cast<size_t>(bh) * N + q0 + i] : 0.f;
        }
        __syncthreads();
#pragma unroll 1
        for (int r = 0; r < kPerWarp; ++r) {
            const int key = key0 + warp * kPerWarp + r;
            if (key >= N) continue;   // warp-uniform
            float p[2], ds[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int ql = lane + 32 * hh;
                // q . k and dO . v over the head dim: k and v are spread over the
                // lanes, so each partial product is summed across the warp
                float dot = 0.f, dpv = 0.f;
#pragma unroll
                for (int e = 0; e < DPL; ++e) {
                    const int cn = min(32, d - 32 * e);
                    for (int cc = 0; cc < cn; ++cc) {
                        const int c = 32 * e + cc;
                        const float kc = __shfl_sync(0xffffffffu, kreg[r][e], cc);
                        const float vc = __shfl_sync(0xffffffffu, vreg[r][e], cc);
                        dot = fmaf(Qs[ql * ld + c], kc, dot);
                        dpv = fmaf(dOs[ql * ld + c], vc, dpv);
                    }
                }
                const bool allowed = (q0 + ql < N) && !(causal && key > q0 + ql);
                p_ds(dot, dpv, mk[r], Ls[ql], Ds[ql], scale, allowed, p[hh], ds[hh]);
            }
#pragma unroll 4
            for (int t = 0; t < kTile; ++t) {
                const float pt = __shfl_sync(0xffffffffu, t < 32 ? p[0] : p[1], t & 31);
                const float st = __shfl_sync(0xffffffffu, t < 32 ? ds[0] : ds[1], t & 31);
#pragma unroll
                for (int e = 0; e < DPL; ++e) {
                    const int c = lane + 32 * e;
                    if (c < d) {
                        adv[r][e] = fmaf(pt, dOs[t * ld + c], adv[r][e]);
                        adk[r][e] = fmaf(st, Qs[t * ld + c], adk[r][e]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kPerWarp; ++r) {
        const int key = key0 + warp * kPerWarp + r;
        if (key >= N) continue;
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
            const int c = lane + 32 * e;
            if (c < d) {
                dV[head + static_cast<size_t>(key) * d + c] = adv[r][e];
                dK[head + static_cast<size_t>(key) * d + c] = adk[r][e] * scale;
            }
        }
    }
}

template <int DPL>
__global__ void __launch_bounds__(kWarpsB * 32)
    bwd_f32_dq_kernel(const float *__restrict__ Q, const float *__restrict__ K, const float *__restrict__ V,
                      const float *__restrict__ dO, const float *__restrict__ LSE, const float *__restrict__ Dv,
                      float *__restrict__ dQ, int N, int d, int causal, float scale,
                      const float *__restrict__ key_mask) {
    extern __shared__ float sm[];
    const int ld = d + 1;
    float *Ks = sm;                      // [kTile][d+1]
    float *Vs = Ks + kTile * ld;         // [kTile][d+1]
    float *Ms = Vs + kTile * ld;         // [kTile] additive mask (-inf past N)
    const int ntq = (N + kTile - 1) / kTile;
    const int bh = blockIdx.x / ntq;
    const int q0 = (blockIdx.x % ntq) * kTile;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t head = static_cast<size_t>(bh) * N * d;

    float qreg[kPerWarp][DPL], oreg[kPerWarp][DPL], acc[kPerWarp][DPL], lse[kPerWarp], dq_d[kPerWarp];
#pragma unroll
    for (int r = 0; r < kPerWarp; ++r) {
        const int row = q0 + warp * kPerWarp + r;
        lse[r] = (row < N) ? LSE[static_cast<size_t>(bh) * N + row] : -INFINITY;
        dq_d[r] = (row < N) ? Dv[static_cast<size_t>(bh) * N + row] : 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
            const int c = lane + 32 * e;
            const bool in = row < N && c < d;
            qreg[r][e] = in ? Q[head + static_cast<size_t>(row) * d + c] : 0.f;
            oreg[r][e] = in ? dO[head + static_cast<size_t>(row) * d + c] : 0.f;
            acc[r][e] = 0.f;
        }
    }
    const int last_row = min(q0 + kTile - 1, N - 1);
    const int nkt = causal ? (last_row / kTile + 1) : (N + kTile - 1) / kTile;
    for (int kt = 0; kt < nkt; ++kt) {
        const int key0 = kt * kTile;
        __syncthreads();
        for (int i = threadIdx.x; i < kTile * d; i += blockDim.x) {
            const int r = i / d, c = i % d;
            const bool in = key0 + r < N;
            const size_t g = head + static_cast<size_t>(key0 + r) * d + c;
            Ks[r * ld + c] = in ? K[g] : 0.f;
            Vs[r * ld + c] = in ? V[g] : 0.f;
        }
        for (int i = threadIdx.x; i < kTile; i += blockDim.x) {
            const int key = key0 + i;
            Ms[i] = (key < N) ? (key_mask ? key_mask[static_cast<size_t>(bh) * N + key] : 0.f) : -INFINITY;
        }
        __syncthreads();
#pragma unroll 1
        for (int r = 0; r < kPerWarp; ++r) {
            const int row = q0 + warp * kPerWarp + r;
            if (row >= N) continue;   // warp-uniform
            float ds[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int kl = lane + 32 * hh;
                float dot = 0.f, dpv = 0.f;
#pragma unroll
                for (int e = 0; e < DPL; ++e) {
                    const int cn = min(32, d - 32 * e);
                    for (int cc = 0; cc < cn; ++cc) {
                        const int c = 32 * e + cc;
                        const float qc = __shfl_sync(0xffffffffu, qreg[r][e], cc);
                        const float oc = __shfl_sync(0xffffffffu, oreg[r][e], cc);
                        dot = fmaf(qc, Ks[kl * ld + c], dot);
                        dpv = fmaf(oc, Vs[kl * ld + c], dpv);
                    }
                }
                const bool allowed = (key0 + kl < N) && !(causal && key0 + kl > row);
                float p;
                p_ds(dot, dpv, Ms[kl], lse[r], dq_d[r], scale, allowed, p, ds[hh]);
            }
#pragma unroll 4
            for (int t = 0; t < kTile; ++t) {
                const float st = __shfl_sync(0xffffffffu, t < 32 ? ds[0] : ds[1], t & 31);
#pragma unroll
                for (int e = 0; e < DPL; ++e) {
                    const int c = lane + 32 * e;
                    if (c < d) acc[r][e] = fmaf(st, Ks[t * ld + c], acc[r][e]);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kPerWarp; ++r) {
        const int row = q0 + warp * kPerWarp + r;
        if (row >= N) continue;
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
            const int c = lane + 32 * e;
            if (c < d) dQ[head + static_cast<size_t>(row) * d + c] = acc[r][e] * scale;
        }
    }
}

template <int DPL>
int launch_bwd_f32_dpl(const float *Q, const float *K, const float *V, const float *O, const float *dO,
                       const float *LSE, float *dQ, float *dK, float *dV, int BH, int N, int d, int causal,
                       float scale, const float *key_mask, float *Dv, cudaStream_t stream) {
    const long long rows = static_cast<long long>(BH) * N;
    const long long pblocks = (rows * 32 + 255) / 256;
    if (pblocks > 0x7fffffffLL) return kErrUnsupported;
    bwd_f32_prep_kernel<<<static_cast<unsigned>(pblocks), 256, 0, stream>>>(O, dO, Dv, rows, d);
    if (cudaGetLastError() != cudaSuccess) return kErrCuda;
    const size_t smem_kv = sizeof(float) * (2 * static_cast<size_t>(kTile) * (d + 1) + 2 * kTile);
    const size_t smem_q = sizeof(float) * (2 * static_cast<size_t>(kTile) * (d + 1) + kTile);
    auto k1 = bwd_f32_dkdv_kernel<DPL>;
    auto k2 = bwd_f32_dq_kernel<DPL>;
    if (cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_kv)) !=
            cudaSuccess ||
        cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_q)) != cudaSuccess)
        return kErrCuda;
    const long long grid = static_cast<long long>((N + kTile - 1) / kTile) * BH;
    if (grid > 0x7fffffffLL) return kErrUnsupported;
    k1<<<static_cast<unsigned>(grid), kWarpsB * 32, smem_kv, stream>>>(Q, K, V, dO, LSE, Dv, dK, dV, N, d, causal,
                                                                       scale, key_mask);
    if (cudaGetLastError() != cudaSuccess) return kErrCuda;
    k2<<<static_cast<unsigned>(grid), kWarpsB * 32, smem_q, stream>>>(Q, K, V, dO, LSE, Dv, dQ, N, d, causal, scale,
                                                                      key_mask);
    return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

}  // namespace

int launch_bwd_f32(const float *Q, const float *K, const float *V, const float *O, const float *dO, const float *LSE,
                   float *dQ, float *dK, float *dV, int B, int H, int N, int d, int causal, float scale,
                   const float *key_mask, void *workspace, cudaStream_t stream) {
    const int BH = B * H;
    float *Dv = static_cast<float *>(workspace);
    switch ((d + 31) / 32) {
        case 1: return launch_bwd_f32_dpl<1>(Q, K, V, O, dO, LSE, dQ, dK, dV, BH, N, d, causal, scale, key_mask, Dv, stream);
        case 2: return launch_bwd_f32_dpl<2>(Q, K, V, O, dO, LSE, dQ, dK, dV, BH, N, d, causal, scale, key_mask, Dv, stream);
        case 3: return launch_bwd_f32_dpl<3>(Q, K, V, O, dO, LSE, dQ, dK, dV, BH, N, d, causal, scale, key_mask, Dv, stream);
        case 4: return launch_bwd_f32_dpl<4>(Q, K, V, O, dO, LSE, dQ, dK, dV, BH, N, d, causal, scale, key_mask, Dv, stream);
        default: return kErrUnsupported;
    }
}

}  // namespace eta
