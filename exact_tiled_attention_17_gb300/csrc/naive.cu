// Materialising baseline attention ("baseline attention" of "Is Flash
// Attention Stable?" §IV): the full score matrix S = Q K^T * scale + mask is
// written to the caller's workspace in the input dtype, a row softmax with
// float32 arithmetic overwrites it with P (input dtype), and O = P V is
// accumulated in float32 and stored in the input dtype.  Three launches on
// the caller's stream.  The workspace holds B*H*N*N elements, the quadratic
// intermediate the tiled kernel avoids (the yadro-code.ru tutorial's
// 128 MiB per head at 8192 tokens in 2-byte elements).
#include <cuda_bf16.h>

#include <cmath>

#include "internal.h"

namespace eta {
namespace {

constexpr int kTM = 64, kTN = 64, kTK = 16;  // output tile and k step
constexpr int kGemmThreads = 256;            // 16 x 16 threads, 4 x 4 outputs each

template <typename T>
__device__ __forceinline__ float ld_f(const T *p, size_t i);
template <>
__device__ __forceinline__ float ld_f<float>(const float *p, size_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}
template <typename T>
__device__ __forceinline__ void st_f(T *p, size_t i, float v);
template <>
__device__ __forceinline__ void st_f<float>(float *p, size_t i, float v) { p[i] = v; }
template <>
__device__ __forceinline__ void st_f<__nv_bfloat16>(__nv_bfloat16 *p, size_t i, float v) {
    p[i] = __float2bfloat16_rn(v);
}

// C[M][Ncols] = A[M][Kd] * op(B) for one head; op(B)[k][c] = B[c][k] when
// B_ROWS_ARE_COLS (B is [Ncols][Kd], as K is for S = Q K^T), else B[k][c].
// EPI_SCORES applies scale, key mask, causal and tail masking (-inf) for S.
template <typename T, bool B_ROWS_ARE_COLS, bool EPI_SCORES>
__global__ void __launch_bounds__(kGemmThreads)
    naive_gemm_kernel(const T *__restrict__ A, const T *__restrict__ Bm, T *__restrict__ C, int M, int Ncols,
                      int Kd, size_t strideA, size_t strideB, size_t strideC, float scale,
                      const float *__restrict__ key_mask, int causal) {
    __shared__ float As[kTK][kTM + 4];
    __shared__ float Bs[kTK][kTN + 4];
    const int bh = blockIdx.z;
    const int m0 = blockIdx.y * kTM, n0 = blockIdx.x * kTN;
    const T *Ah = A + bh * strideA;
    const T *Bh = Bm + bh * strideB;
    T *Ch = C + bh * strideC;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < Kd; k0 += kTK) {
        for (int i = threadIdx.x; i < kTM * kTK; i += kGemmThreads) {
            const int r = i / kTK, k = i % kTK;
            const int gm = m0 + r, gk = k0 + k;
            As[k][r] = (gm < M && gk < Kd) ? ld_f(Ah, static_cast<size_t>(gm) * Kd + gk) : 0.f;
        }
        for (int i = threadIdx.x; i < kTN * kTK; i += kGemmThreads) {
            if (B_ROWS_ARE_COLS) {
                const int c = i / kTK, k = i % kTK;
                const int gc = n0 + c, gk = k0 + k;
                Bs[k][c] = (gc < Ncols && gk < Kd) ? ld_f(Bh, static_cast<size_t>(gc) * Kd + gk) : 0.f;
            } else {
                const int k = i / kTN, c = i % kTN;
                const int gc = n0 + c, gk = k0 + k;
                Bs[k][c] = (gc < Ncols && gk < Kd) ? ld_f(Bh, static_cast<size_t>(gk) * Ncols + gc) : 0.f;
            }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kTK; ++k) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[k][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[k][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int gm = m0 + ty * 4 + i;
        if (gm >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int gc = n0 + tx * 4 + j;
            if (gc >= Ncols) continue;
            float v = acc[i][j];
            if (EPI_SCORES) {
                v *= scale;
                if (key_mask) v += key_mask[static_cast<size_t>(bh) * Ncols + gc];
                if (causal && gc > gm) v = -INFINITY;
            }
            st_f(Ch, static_cast<size_t>(gm) * Ncols + gc, v);
        }
    }
}

__device__ __forceinline__ float block_reduce_max(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    v = (threadIdx.x < (blockDim.x >> 5)) ? red[threadIdx.x] : -INFINITY;
    if (w == 0) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (l == 0) red[0] = v;
    }
    __syncthreads();
    return red[0];
}
__device__ __forceinline__ float block_reduce_sum(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    v = (threadIdx.x < (blockDim.x >> 5)) ? red[threadIdx.x] : 0.f;
    if (w == 0) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (l == 0) red[0] = v;
    }
    __syncthreads();
    return red[0];
}

// One block per row: P = exp(s - max) / sum (float32 math), stored over S.
template <typename T>
__global__ void __launch_bounds__(256) naive_softmax_kernel(T *__restrict__ S, float *__restrict__ LSE, int N) {
    __shared__ float red[32];
    const size_t row = blockIdx.x;
    T *s = S + row * N;
    float mx = -INFINITY;
    for (int j = threadIdx.x; j < N; j += blockDim.x) mx = fmaxf(mx, ld_f(s, j));
    mx = block_reduce_max(mx, red);
    if (mx == -INFINITY) {  // fully masked row
        for (int j = threadIdx.x; j < N; j += blockDim.x) st_f(s, j, 0.f);
        if (LSE && threadIdx.x == 0) LSE[row] = -INFINITY;
        return;
    }
    float sum = 0.f;
    for (int j = threadIdx.x; j < N; j += blockDim.x) sum += expf(ld_f(s, j) - mx);
    sum = block_reduce_sum(sum, red);
    const float inv = 1.f / sum;
    for (int j = threadIdx.x; j < N; j += blockDim.x) st_f(s, j, expf(ld_f(s, j) - mx) * inv);
    if (LSE && threadIdx.x == 0) LSE[row] = mx + logf(sum);
}

template <typename T>
int run(const T *Q, const T *K, const T *V, T *O, float *LSE, int BH, int N, int d, int causal, float scale,
        const float *key_mask, T *S, cudaStream_t stream) {
    if (BH > 65535) return kErrUnsupported;
    const size_t hqk = static_cast<size_t>(N) * d, hs = static_cast<size_t>(N) * N;
    dim3 g1((N + kTN - 1) / kTN, (N + kTM - 1) / kTM, BH);
    naive_gemm_kernel<T, true, true><<<g1, kGemmThreads, 0, stream>>>(Q, K, S, N, N, d, hqk, hqk, hs, scale,
                                                                       key_mask, causal);
    naive_softmax_kernel<T><<<static_cast<unsigned>(static_cast<size_t>(BH) * N), 256, 0, stream>>>(S, LSE, N);
    dim3 g3((d + kTN - 1) / kTN, (N + kTM - 1) / kTM, BH);
    naive_gemm_kernel<T, false, false><<<g3, kGemmThreads, 0, stream>>>(S, V, O, N, d, N, hs, hqk, hqk, 1.f,
                                                                         nullptr, 0);
    return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

}  // namespace

int launch_naive(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H, int N, int d,
                 int causal, float scale, int dtype, const float *key_mask, void *workspace, cudaStream_t stream) {
    const int BH = B * H;
    if (dtype == 1)
        return run(static_cast<const __nv_bfloat16 *>(Q), static_cast<const __nv_bfloat16 *>(K),
                   static_cast<const __nv_bfloat16 *>(V), static_cast<__nv_bfloat16 *>(O), LSE, BH, N, d, causal,
                   scale, key_mask, static_cast<__nv_bfloat16 *>(workspace), stream);
    return run(static_cast<const float *>(Q), static_cast<const float *>(K), static_cast<const float *>(V),
               static_cast<float *>(O), LSE, BH, N, d, causal, scale, key_mask, static_cast<float *>(workspace),
               stream);
}

}  // namespace eta
