// Exact tiled attention forward in true float32 on the CUDA cores.
//
// Same computation as the tensor-core path ("Is Flash Attention Stable?"
// §II-A/§II-B; the yadro-code.ru tutorial's online merge), with every
// operation in IEEE float32 and no TF32: the rescale exp(m_old - m_new) is
// applied whenever a tile raises a row's maximum, exactly as the tutorial
// describes, and scores are differenced in natural-log units before the
// exponential (expf) so that large scores such as 1000..1004 keep their
// exact differences.
//
// Layout: one CTA of 8 warps per 64-row query tile of one (batch, head); K/V
// tiles of 64 keys staged in shared memory; each warp owns 8 query rows and
// one row at a time: lane t computes the scores of keys t and t+32, the row
// max and sum are warp reductions, and lane t accumulates output dims
// t, t+32, t+64, t+96.
#include <cmath>

#include "internal.h"

namespace eta {
namespace {

constexpr int kRows = 64;      // query rows per CTA
constexpr int kKeys = 64;      // keys per tile
constexpr int kWarps = 8;
constexpr int kRowsPerWarp = kRows / kWarps;

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

template <int DPL>  // output dims per lane: ceil(d / 32)
__global__ void __launch_bounds__(kWarps * 32)
    attn_fwd_f32_kernel(const float *__restrict__ Q, const float *__restrict__ K, const float *__restrict__ V,
                        float *__restrict__ O, float *__restrict__ LSE, int N, int d, int causal, float scale,
                        const float *__restrict__ key_mask) {
    extern __shared__ float sm[];
    const int ldk = d + 1;  // padded row stride of the K tile (bank-conflict-free column reads)
    float *Qs = sm;                      // [kRows][d]
    float *Ks = Qs + kRows * d;          // [kKeys][d+1]
    float *Vs = Ks + kKeys * ldk;        // [kKeys][d]
    float *Ms = Vs + kKeys * d;          // [kKeys] additive mask of the tile

    const int ntiles = (N + kRows - 1) / kRows;
    const int bh = blockIdx.x / ntiles;
    const int row0 = (blockIdx.x % ntiles) * kRows;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t head = static_cast<size_t>(bh) * N * d;
    const float ninf = -INFINITY;

    for (int i = threadIdx.x; i < kRows * d; i += blockDim.x) {
        const int r = i / d, c = i % d;
        Qs[i] = (row0 + r < N) ? Q[head + static_cast<size_t>(row0 + r) * d + c] : 0.f;
    }

    float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][DPL];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        m[r] = ninf;
        l[r] = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[r][e] = 0.f;
    }

    const int last_row = min(row0 + kRows - 1, N - 1);
    const int nkt = causal ? (last_row / kKeys + 1) : (N + kKeys - 1) / kKeys;
    for (int kt = 0; kt < nkt; ++kt) {
        const int key0 = kt * kKeys;
        __syncthreads();
        for (int i = threadIdx.x; i < kKeys * d; i += blockDim.x) {
            const int r = i / d, c = i % d;
            const bool in = key0 + r < N;
            const size_t g = head + static_cast<size_t>(key0 + r) * d + c;
            Ks[r * ldk + c] = in ? K[g] : 0.f;
            Vs[i] = in ? V[g] : 0.f;
        }
        for (int i = threadIdx.x; i < kKeys; i += blockDim.x) {
            const int key = key0 + i;
            Ms[i] = (key < N) ? (key_mask ? key_mask[static_cast<size_t>(bh) * N + key] : 0.f) : ninf;
        }
        __syncthreads();

#pragma unroll 1
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const int rl = warp * kRowsPerWarp + r;
            const int row = row0 + rl;
            if (row >= N) continue;  // warp-uniform
            const float *qr = Qs + rl * d;
            float s[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int kl = lane + 32 * h;
                const float *kr = Ks + kl * ldk;
                float dot = 0.f;
                for (int c = 0; c < d; ++c) dot = fmaf(qr[c], kr[c], dot);
                float x = fmaf(dot, scale, Ms[kl]);
                if (causal && key0 + kl > row) x = ninf;
                s[h] = x;
            }
            const float mx = warp_max(fmaxf(s[0], s[1]));
            const float m_new = fmaxf(m[r], mx);
            // the tutorial's rescale of the old sums; -inf max means nothing seen yet
            const float alpha = (m_new == ninf) ? 1.f : expf(m[r] - m_new);
            const float mu = (m_new == ninf) ? 0.f : m_new;
            const float p0 = expf(s[0] - mu), p1 = expf(s[1] - mu);
            l[r] = l[r] * alpha + warp_sum(p0 + p1);
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc[r][e] *= alpha;
#pragma unroll 4
            for (int t = 0; t < kKeys; ++t) {
                const float pt = __shfl_sync(0xffffffffu, t < 32 ? p0 : p1, t & 31);
                const float *vr = Vs + t * d;
#pragma unroll
                for (int e = 0; e < DPL; ++e) {
                    const int c = lane + 32 * e;
                    if (c < d) acc[r][e] = fmaf(pt, vr[c], acc[r][e]);
                }
            }
            m[r] = m_new;
        }
    }

#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int row = row0 + warp * kRowsPerWarp + r;
        if (row >= N) continue;
        const bool any = l[r] > 0.f;
        float *orow = O + head + static_cast<size_t>(row) * d;
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
            const int c = lane + 32 * e;
            if (c < d) orow[c] = any ? acc[r][e] / l[r] : 0.f;
        }
        if (LSE && lane == 0) LSE[static_cast<size_t>(bh) * N + row] = any ? m[r] + logf(l[r]) : ninf;
    }
}

template <int DPL>
int launch_dpl(const float *Q, const float *K, const float *V, float *O, float *LSE, int BH, int N, int d,
               int causal, float scale, const float *key_mask, cudaStream_t stream) {
    const size_t smem = sizeof(float) * (static_cast<size_t>(kRows) * d + kKeys * (d + 1) + kKeys * d + kKeys);
    auto kern = attn_fwd_f32_kernel<DPL>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
        return kErrCuda;
    const long long grid = static_cast<long long>((N + kRows - 1) / kRows) * BH;
    if (grid > 0x7fffffffLL) return kErrUnsupported;
    kern<<<static_cast<unsigned>(grid), kWarps * 32, smem, stream>>>(Q, K, V, O, LSE, N, d, causal, scale, key_mask);
    return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

}  // namespace

int launch_fwd_f32(const float *Q, const float *K, const float *V, float *O, float *LSE, int B, int H, int N,
                   int d, int causal, float scale, const float *key_mask, cudaStream_t stream,
                   const char **variant) {
    const int BH = B * H;
    const int dpl = (d + 31) / 32;
    static const char *names[4] = {"simt_f32_br64_bc64_dpl1", "simt_f32_br64_bc64_dpl2", "simt_f32_br64_bc64_dpl3",
                                   "simt_f32_br64_bc64_dpl4"};
    if (dpl < 1 || dpl > 4) return kErrUnsupported;
    if (variant) *variant = names[dpl - 1];
    switch (dpl) {
        case 1: return launch_dpl<1>(Q, K, V, O, LSE, BH, N, d, causal, scale, key_mask, stream);
        case 2: return launch_dpl<2>(Q, K, V, O, LSE, BH, N, d, causal, scale, key_mask, stream);
        case 3: return launch_dpl<3>(Q, K, V, O, LSE, BH, N, d, causal, scale, key_mask, stream);
        default: return launch_dpl<4>(Q, K, V, O, LSE, BH, N, d, causal, scale, key_mask, stream);
    }
}

}  // namespace eta
