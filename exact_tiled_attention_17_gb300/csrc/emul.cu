// Number-format emulation of attention: the precision and perturbation
// instrument of "Is Flash Attention Stable?" §III (Fig. 2: a numerical
// re-implementation of FlashAttention and of the baseline, run in any number
// format and with the algorithm's internals open to change), used for its
// format sweep (§IV-A, Fig. 3) and its block-size perturbations (§IV-B,
// Fig. 6).  The pages give no code; the reading implemented here:
//
//   A format F has `mbits` fraction bits and `ebits` exponent bits (IEEE
//   style: subnormals, round to nearest with ties to even, overflow to
//   infinity); fl(x) rounds an exact value to F.  Every tensor operation
//   produces its result in F: an elementwise operation is evaluated in
//   binary64 and rounded once; a reduction (row sum, row maximum) or a matrix
//   product accumulates in binary64 and rounds its result once.  Q, K and V
//   are rounded to F first.
//
//   scores   s_j = fl(scale * (q . k_j)); fl(s_j + mask_j) with a key mask;
//            -inf for a masked or (causal) future key.
//   baseline P = fl(softmax(s)) as one operation, then O = fl(P V).
//   tiled    the online merge over key blocks of width Bc, in order
//            (§II-B, Fig. 1; running maximum m, denominator l, unnormalised
//            output o):  M = max(m, max_j s_j), M' = (M == -inf ? 0 : M),
//            a = fl(exp(fl(m - M'))) (0 while m == -inf),
//            p_j = fl(exp(fl(s_j - M'))), l = fl(fl(a l) + fl(sum_j p_j)),
//            o = fl(fl(a o) + fl(sum_j p_j v_j)); finally o = fl(o / l), or 0
//            for a row with no allowed key.
//
// Only the tiled algorithm's per-row arithmetic depends on the tile shape,
// through the key-block width Bc; the query-block height only groups rows.
//
// GPU mapping: one CTA of 128 threads per output row.  Threads split the
// keys of a block for the scores and the exponentials, and the d output
// columns for the products with V.  This is a measurement tool, not a fast
// path: binary64 arithmetic throughout.
#include <cuda_bf16.h>
#include <cmath>

#include "internal.h"

namespace eta {
namespace {

constexpr int kEmulThreads = 128;

// fl(x): x rounded to the format with `mbits` fraction and `ebits` exponent
// bits.  Near x the format's values are spaced 2^(e - mbits), e being x's
// binary exponent, clamped below at the smallest normal exponent (so the
// subnormals share one spacing); x is rounded to the nearest multiple of
// that spacing (ties to even) and a result beyond the largest finite value
// becomes infinite.
__device__ double fmt_round(double x, int mbits, int ebits) {
    if (x != x || isinf(x) || x == 0.0) return x;
    if (mbits >= 52 && ebits >= 11) return x;
    const int emax = (1 << (ebits - 1)) - 1;
    const int emin = 1 - emax;
    int e2;
    (void)frexp(fabs(x), &e2);
    int e = e2 - 1;
    if (e < emin) e = emin;
    const double spacing = ldexp(1.0, e - mbits);
    double y = rint(x / spacing) * spacing;
    const double maxfinite = ldexp(2.0 - ldexp(1.0, -mbits), emax);
    if (fabs(y) > maxfinite) y = copysign(__longlong_as_double(0x7ff0000000000000LL), x);
    return y;
}

__device__ double load_in(const void *base, int dtype, long long i) {
    if (dtype == 1) return static_cast<double>(__bfloat162float(static_cast<const __nv_bfloat16 *>(base)[i]));
    if (dtype == 2) return static_cast<const double *>(base)[i];
    return static_cast<double>(static_cast<const float *>(base)[i]);
}

struct EmulParams {
    const void *Q, *K, *V;
    int dtype;   // 0 float32, 1 bfloat16, 2 float64
    double *O;   // [nrows][d]
    int N, d, causal;
    double scale;
    const float *key_mask;   // [BH][N] or null
    int algo, Bc, mbits, ebits;
    const long long *rows;   // flat row ids or null (rows 0 .. nrows-1)
    long long nrows, nflat;
    int *err;
};

// block-wide maximum or sum of one value per thread (binary64); red has
// kEmulThreads/32 slots
__device__ double block_max(double v, double *red) {
    for (int o = 16; o > 0; o >>= 1) v = fmax(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    double r = red[0];
    for (int w = 1; w < kEmulThreads / 32; ++w) r = fmax(r, red[w]);
    __syncthreads();
    return r;
}
__device__ double block_sum(double v, double *red) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    double r = red[0];
    for (int w = 1; w < kEmulThreads / 32; ++w) r += red[w];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kEmulThreads) attn_emul_kernel(const EmulParams p) {
    extern __shared__ double sm[];
    double *qrow = sm;                 // d values of the query row, in F
    double *red = qrow + 128;          // reduction slots
    double *s = red + kEmulThreads / 32;   // scores / probabilities of the current block
    const long long r = blockIdx.x;
    const long long flat = p.rows ? p.rows[r] : r;
    if (flat < 0 || flat >= p.nflat) {
        if (threadIdx.x == 0) atomicOr(p.err, kErrWordBadRow);
        return;
    }
    const int N = p.N, d = p.d, mb = p.mbits, eb = p.ebits;
    const long long bh = flat / N;
    const int i = static_cast<int>(flat % N);
    const long long base = bh * N * static_cast<long long>(d);
    for (int c = threadIdx.x; c < d; c += kEmulThreads) qrow[c] = fmt_round(load_in(p.Q, p.dtype, base + static_cast<long long>(i) * d + c), mb, eb);
    __syncthreads();

    auto score = [&](int j) -> double {
        if (p.causal && j > i) return -INFINITY;
        const long long kb = base + static_cast<long long>(j) * d;
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += qrow[c] * fmt_round(load_in(p.K, p.dtype, kb + c), mb, eb);
        double x = fmt_round(p.scale * dot, mb, eb);
        if (p.key_mask) {
            const float mk = p.key_mask[bh * N + j];
            x = (isinf(mk) && mk < 0.f) ? -INFINITY : fmt_round(x + static_cast<double>(mk), mb, eb);
        }
        return x;
    };
    // sum_j w[j] * fl(v_j[c]) for j in [j0, j1), w indexed from 0, binary64
    auto pv = [&](int c, int j0, int j1, const double *w) -> double {
        double acc = 0.0;
        for (int j = j0; j < j1; ++j)
            acc += w[j - j0] * fmt_round(load_in(p.V, p.dtype, base + static_cast<long long>(j) * d + c), mb, eb);
        return acc;
    };
    double *orow = p.O + r * static_cast<long long>(d);

    if (p.algo == 0) {
        // baseline: one softmax op over all N scores, then one matrix product
        double mx = -INFINITY;
        for (int j = threadIdx.x; j < N; j += kEmulThreads) {
            s[j] = score(j);
            mx = fmax(mx, s[j]);
        }
        mx = block_max(mx, red);
        if (mx == -INFINITY) {
            for (int c = threadIdx.x; c < d; c += kEmulThreads) orow[c] = 0.0;
            return;
        }
        double part = 0.0;
        for (int j = threadIdx.x; j < N; j += kEmulThreads) {
            s[j] = exp(s[j] - mx);
            part += s[j];
        }
        const double sum = block_sum(part, red);
        for (int j = threadIdx.x; j < N; j += kEmulThreads) s[j] = fmt_round(s[j] / sum, mb, eb);
        __syncthreads();
        for (int c = threadIdx.x; c < d; c += kEmulThreads) orow[c] = fmt_round(pv(c, 0, N, s), mb, eb);
        return;
    }

    // tiled: online merge over key blocks of width Bc
    double m = -INFINITY, l = 0.0;
    double o = 0.0;   // column threadIdx.x of o (threads >= d carry nothing)
    for (int j0 = 0; j0 < N; j0 += p.Bc) {
        const int j1 = min(j0 + p.Bc, N);
        double mx = -INFINITY;
        for (int j = j0 + threadIdx.x; j < j1; j += kEmulThreads) {
            s[j - j0] = score(j);
            mx = fmax(mx, s[j - j0]);
        }
        const double M = fmax(m, block_max(mx, red));
        const double Mu = (M == -INFINITY) ? 0.0 : M;
        const double a = (m == -INFINITY) ? 0.0 : fmt_round(exp(fmt_round(m - Mu, mb, eb)), mb, eb);
        double part = 0.0;
        for (int j = j0 + threadIdx.x; j < j1; j += kEmulThreads) {
            const double x = s[j - j0];
            s[j - j0] = (x == -INFINITY) ? 0.0 : fmt_round(exp(fmt_round(x - Mu, mb, eb)), mb, eb);
            part += s[j - j0];
        }
        const double rs = block_sum(part, red);   // also orders the writes of s before the reads below
        l = fmt_round(fmt_round(a * l, mb, eb) + fmt_round(rs, mb, eb), mb, eb);
        if (threadIdx.x < d)
            o = fmt_round(fmt_round(a * o, mb, eb) + fmt_round(pv(threadIdx.x, j0, j1, s), mb, eb), mb, eb);
        m = M;
        __syncthreads();   // s is overwritten by the next block
    }
    if (threadIdx.x < d) orow[threadIdx.x] = (l == 0.0) ? 0.0 : fmt_round(o / l, mb, eb);
}

__global__ void fmt_round_kernel(const double *x, double *y, long long n, int mbits, int ebits) {
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < n; t += stride)
        y[t] = fmt_round(x[t], mbits, ebits);
}

}  // namespace

size_t emul_smem_bytes(int algo, int N, int Bc) {
    const long long nbuf = algo == 0 ? N : Bc;
    return static_cast<size_t>(128 + kEmulThreads / 32 + nbuf) * sizeof(double);
}

int launch_emul(const void *Q, const void *K, const void *V, int dtype, double *O, int B, int H, int N, int d,
                int causal, float scale, const float *key_mask, int algo, int Bc, int mbits, int ebits,
                const long long *rows, long long nrows, cudaStream_t stream) {
    int *err = device_error_word();
    if (!err) return kErrCuda;
    EmulParams p;
    p.Q = Q;
    p.K = K;
    p.V = V;
    p.dtype = dtype;
    p.O = O;
    p.N = N;
    p.d = d;
    p.causal = causal;
    p.scale = static_cast<double>(scale);
    p.key_mask = key_mask;
    p.algo = algo;
    p.Bc = Bc;
    p.mbits = mbits;
    p.ebits = ebits;
    p.rows = rows;
    p.nflat = static_cast<long long>(B) * H * N;
    p.nrows = rows ? nrows : p.nflat;
    p.err = err;
    if (p.nrows == 0) return kOk;
    if (p.nrows > 0x7fffffffLL) return kErrUnsupported;
    const size_t smem = emul_smem_bytes(algo, N, Bc);
    if (cudaFuncSetAttribute(attn_emul_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return kErrCuda;
    attn_emul_kernel<<<static_cast<unsigned>(p.nrows), kEmulThreads, smem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

int launch_fmt_round(const double *x, double *y, long long n, int mbits, int ebits, cudaStream_t stream) {
    const long long blocks = (n + 255) / 256;
    fmt_round_kernel<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(x, y, n, mbits,
                                                                                                ebits);
    return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

}  // namespace eta
