// Deviation measures between two tensors, on the GPU, in float64:
// max |a-b| (the paper's §IV-A element-wise maximum difference), the 1-D
// Wasserstein-1 distance of the two value distributions (its §V measure),
// computed by sorting both tensors, and mean / std of |a-b| and the signed
// mean.  The sort is a stable least-significant-digit radix sort (8 passes of
// 8 bits) on order-preserving 64-bit keys of the float64 values.  All
// reductions use a fixed grid and a fixed combination order, so results are
// reproducible run to run.
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "internal.h"

namespace eta {
namespace {

constexpr int kSortThreads = 256;
constexpr int kSortItems = 16;
constexpr int kTile = kSortThreads * kSortItems;  // keys per radix block
constexpr int kRedBlocks = 1024;
constexpr int kRedThreads = 256;
constexpr int kScanChunk = 1024;

constexpr size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct Layout {
    size_t keys_a, keys_b, tmp, hist, chunk_sums, part, result, total;
    long long nb, hist_len, nchunks;
};

constexpr Layout layout(long long n) {
    Layout L{};
    L.nb = (n + kTile - 1) / kTile;
    L.hist_len = 256 * L.nb;
    L.nchunks = (L.hist_len + kScanChunk - 1) / kScanChunk;
    size_t off = 0;
    L.keys_a = off; off = align256(off + sizeof(uint64_t) * n);
    L.keys_b = off; off = align256(off + sizeof(uint64_t) * n);
    L.tmp = off; off = align256(off + sizeof(uint64_t) * n);
    L.hist = off; off = align256(off + sizeof(uint32_t) * L.hist_len);
    L.chunk_sums = off; off = align256(off + sizeof(uint32_t) * L.nchunks);
    L.part = off; off = align256(off + sizeof(double) * 3 * kRedBlocks);
    L.result = off; off = align256(off + sizeof(double) * 8);
    L.total = off;
    return L;
}

__device__ __forceinline__ double load_as_f64(const void *p, int t, long long i) {
    if (t == 0) return static_cast<double>(static_cast<const float *>(p)[i]);
    if (t == 1) return static_cast<double>(__bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]));
    return static_cast<const double *>(p)[i];
}
// Order-preserving map of float64 bits to unsigned 64-bit keys.
__device__ __forceinline__ uint64_t f64_to_key(double v) {
    const uint64_t u = static_cast<uint64_t>(__double_as_longlong(v));
    return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}
__device__ __forceinline__ double key_to_f64(uint64_t k) {
    const uint64_t u = (k >> 63) ? (k & 0x7FFFFFFFFFFFFFFFull) : ~k;
    return __longlong_as_double(static_cast<long long>(u));
}
// |a - b| with equal values (including equal infinities) giving 0.
__device__ __forceinline__ double absdiff(double a, double b) { return (a == b) ? 0.0 : fabs(a - b); }
__device__ __forceinline__ double nanmax(double x, double y) {
    return isnan(x) ? x : (isnan(y) ? y : fmax(x, y));
}

// Deterministic block reduction of up to 3 doubles (sum or NaN-propagating max).
template <int K>
__device__ void block_reduce(double (&v)[K], const bool (&is_max)[K], double *red /* [K][32] */) {
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
#pragma unroll
    for (int k = 0; k < K; ++k) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const double u = __shfl_xor_sync(0xffffffffu, v[k], o);
            v[k] = is_max[k] ? nanmax(v[k], u) : v[k] + u;
        }
    }
    __syncthreads();
    if (l == 0)
#pragma unroll
        for (int k = 0; k < K; ++k) red[k * 32 + w] = v[k];
    __syncthreads();
    if (w == 0) {
        const int nw = blockDim.x >> 5;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            double x = (l < nw) ? red[k * 32 + l] : (is_max[k] ? 0.0 : 0.0);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const double u = __shfl_xor_sync(0xffffffffu, x, o);
                x = is_max[k] ? nanmax(x, u) : x + u;
            }
            v[k] = x;
        }
    }
}

// Pass 1: keys of a and b; per-block max |a-b|, sum |a-b|, sum (a-b).
__global__ void __launch_bounds__(kRedThreads)
    dev_convert_kernel(const void *a, int ta, const void *b, int tb, long long n, uint64_t *ka, uint64_t *kb,
                       double *part) {
    __shared__ double red[3 * 32];
    double v[3] = {0.0, 0.0, 0.0};
    const bool is_max[3] = {true, false, false};
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const double x = load_as_f64(a, ta, i), y = load_as_f64(b, tb, i);
        ka[i] = f64_to_key(x);
        kb[i] = f64_to_key(y);
        const double ad = absdiff(x, y);
        v[0] = nanmax(v[0], ad);
        v[1] += ad;
        v[2] += (x == y) ? 0.0 : x - y;
    }
    block_reduce<3>(v, is_max, red);
    if (threadIdx.x == 0)
        for (int k = 0; k < 3; ++k) part[blockIdx.x * 3 + k] = v[k];
}

// Pass 2: per-block sum of (|a-b| - mean)^2; mean read from result[2].
__global__ void __launch_bounds__(kRedThreads)
    dev_var_kernel(const void *a, int ta, const void *b, int tb, long long n, const double *result, double *part) {
    __shared__ double red[32];
    const double mean = result[2];
    double v[1] = {0.0};
    const bool is_max[1] = {false};
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const double ad = absdiff(load_as_f64(a, ta, i), load_as_f64(b, tb, i));
        v[0] += (ad - mean) * (ad - mean);
    }
    block_reduce<1>(v, is_max, red);
    if (threadIdx.x == 0) part[blockIdx.x * 3] = v[0];
}

// Pass 3 (after sorting): per-block sum |sort(a)_i - sort(b)_i|.
__global__ void __launch_bounds__(kRedThreads)
    dev_w1_kernel(const uint64_t *ka, const uint64_t *kb, long long n, double *part) {
    __shared__ double red[32];
    double v[1] = {0.0};
    const bool is_max[1] = {false};
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        v[0] += absdiff(key_to_f64(ka[i]), key_to_f64(kb[i]));
    block_reduce<1>(v, is_max, red);
    if (threadIdx.x == 0) part[blockIdx.x * 3] = v[0];
}

// Combine the per-block partials in a fixed order.  stage 0: max/mean/signed
// mean; stage 1: std; stage 2: w1.
__global__ void __launch_bounds__(kRedThreads) dev_finalize_kernel(const double *part, int nparts, long long n,
                                                                   int stage, double *result) {
    __shared__ double red[3 * 32];
    double v[3] = {0.0, 0.0, 0.0};
    const bool is_max[3] = {stage == 0, false, false};
    for (int i = threadIdx.x; i < nparts; i += blockDim.x) {
        if (stage == 0) {
            v[0] = nanmax(v[0], part[i * 3]);
            v[1] += part[i * 3 + 1];
            v[2] += part[i * 3 + 2];
        } else {
            v[0] += part[i * 3];
        }
    }
    block_reduce<3>(v, is_max, red);
    if (threadIdx.x == 0) {
        const double dn = static_cast<double>(n);
        if (stage == 0) {
            result[0] = v[0];
            result[2] = v[1] / dn;
            result[4] = v[2] / dn;
        } else if (stage == 1) {
            result[3] = sqrt(v[0] / dn);
        } else {
            result[1] = v[0] / dn;
        }
    }
}

// ---------------- radix sort ----------------

__global__ void __launch_bounds__(kSortThreads)
    radix_hist_kernel(const uint64_t *keys, long long n, int shift, uint32_t *hist, long long nb) {
    __shared__ uint32_t cnt[256];
    cnt[threadIdx.x] = 0;
    __syncthreads();
    const long long base = blockIdx.x * static_cast<long long>(kTile);
    for (int i = threadIdx.x; i < kTile; i += kSortThreads) {
        const long long idx = base + i;
        if (idx < n) atomicAdd(&cnt[(keys[idx] >> shift) & 255u], 1u);
    }
    __syncthreads();
    hist[static_cast<long long>(threadIdx.x) * nb + blockIdx.x] = cnt[threadIdx.x];
}

// Exclusive scan, three phases: chunk sums, scan of chunk sums (one block,
// sequential over tiles with a carry), per-chunk scan with the chunk offset.
__global__ void __launch_bounds__(kScanChunk) scan_chunk_sums_kernel(const uint32_t *x, long long len, uint32_t *sums) {
    __shared__ uint32_t red[32];
    const long long i = blockIdx.x * static_cast<long long>(kScanChunk) + threadIdx.x;
    uint32_t v = (i < len) ? x[i] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        uint32_t w = red[threadIdx.x];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
        if (threadIdx.x == 0) sums[blockIdx.x] = w;
    }
}

__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t *warp_tot, uint32_t &total) {
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    uint32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(0xffffffffu, inc, o);
        if (l >= o) inc += u;
    }
    if (l == 31) warp_tot[w] = inc;
    __syncthreads();
    if (w == 0) {
        const int nw = blockDim.x >> 5;
        uint32_t t = (l < nw) ? warp_tot[l] : 0u;
        uint32_t ti = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_up_sync(0xffffffffu, ti, o);
            if (l >= o) ti += u;
        }
        if (l < nw) warp_tot[l] = ti - t;  // exclusive warp offsets
        if (l == 31) warp_tot[32] = ti;
    }
    __syncthreads();
    total = warp_tot[32];
    const uint32_t r = warp_tot[w] + inc - v;
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kScanChunk) scan_sums_kernel(uint32_t *sums, long long nchunks) {
    __shared__ uint32_t warp_tot[33];
    uint32_t carry = 0;
    for (long long t0 = 0; t0 < nchunks; t0 += kScanChunk) {
        const long long i = t0 + threadIdx.x;
        const uint32_t v = (i < nchunks) ? sums[i] : 0u;
        uint32_t total;
        const uint32_t ex = block_exclusive_scan(v, warp_tot, total);
        if (i < nchunks) sums[i] = carry + ex;
        carry += total;
    }
}

__global__ void __launch_bounds__(kScanChunk) scan_apply_kernel(uint32_t *x, long long len, const uint32_t *sums) {
    __shared__ uint32_t warp_tot[33];
    const long long i = blockIdx.x * static_cast<long long>(kScanChunk) + threadIdx.x;
    const uint32_t v = (i < len) ? x[i] : 0u;
    uint32_t total;
    const uint32_t ex = block_exclusive_scan(v, warp_tot, total);
    if (i < len) x[i] = sums[blockIdx.x] + ex;
}

// Stable scatter.  Warp w of block b ranks keys [b*kTile + w*512, +512) in 16
// rounds of 32 consecutive keys: peers with the same digit are found with
// match.any, ranked by lane order, and counted into the warp's private digit
// histogram; a per-digit exclusive scan over warps then gives each warp's
// offset inside the block, and the scanned global histogram the block's.
__global__ void __launch_bounds__(kSortThreads)
    radix_scatter_kernel(const uint64_t *__restrict__ in, uint64_t *__restrict__ out, long long n, int shift,
                         const uint32_t *__restrict__ offs, long long nb) {
    constexpr int kWarps = kSortThreads / 32;
    constexpr int kPerWarp = kTile / kWarps;  // 512
    __shared__ uint32_t wh[kWarps][256];
    for (int i = threadIdx.x; i < kWarps * 256; i += kSortThreads) (&wh[0][0])[i] = 0u;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long base = blockIdx.x * static_cast<long long>(kTile) + warp * kPerWarp;
    uint64_t key[kSortItems];
    uint32_t dig[kSortItems], rank[kSortItems];
#pragma unroll
    for (int r = 0; r < kSortItems; ++r) {
        const long long idx = base + r * 32 + lane;
        const bool valid = idx < n;
        key[r] = valid ? in[idx] : 0ull;
        dig[r] = valid ? static_cast<uint32_t>((key[r] >> shift) & 255u) : 256u;
        const unsigned active = __ballot_sync(0xffffffffu, valid);
        unsigned peers = 0;
        rank[r] = 0;
        if (valid) {
            peers = __match_any_sync(active, dig[r]);
            rank[r] = wh[warp][dig[r]] + __popc(peers & ((1u << lane) - 1u));
        }
        __syncwarp();
        if (valid && lane == __ffs(peers) - 1) wh[warp][dig[r]] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    {
        uint32_t run = 0;
        for (int w = 0; w < kWarps; ++w) {
            const uint32_t c = wh[w][threadIdx.x];
            wh[w][threadIdx.x] = run;
            run += c;
        }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kSortItems; ++r) {
        if (dig[r] == 256u) continue;
        const uint32_t pos = offs[static_cast<long long>(dig[r]) * nb + blockIdx.x] + wh[warp][dig[r]] + rank[r];
        out[pos] = key[r];
    }
}

int radix_sort(uint64_t *keys, uint64_t *tmp, long long n, const Layout &L, char *ws, cudaStream_t st) {
    uint32_t *hist = reinterpret_cast<uint32_t *>(ws + L.hist);
    uint32_t *sums = reinterpret_cast<uint32_t *>(ws + L.chunk_sums);
    uint64_t *src = keys, *dst = tmp;
    for (int shift = 0; shift < 64; shift += 8) {
        radix_hist_kernel<<<static_cast<unsigned>(L.nb), kSortThreads, 0, st>>>(src, n, shift, hist, L.nb);
        scan_chunk_sums_kernel<<<static_cast<unsigned>(L.nchunks), kScanChunk, 0, st>>>(hist, L.hist_len, sums);
        scan_sums_kernel<<<1, kScanChunk, 0, st>>>(sums, L.nchunks);
        scan_apply_kernel<<<static_cast<unsigned>(L.nchunks), kScanChunk, 0, st>>>(hist, L.hist_len, sums);
        radix_scatter_kernel<<<static_cast<unsigned>(L.nb), kSortThreads, 0, st>>>(src, dst, n, shift, hist, L.nb);
        uint64_t *t = src;
        src = dst;
        dst = t;
    }
    // 8 passes: the sorted keys are back in `keys`.
    return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

}  // namespace

// ---------------------------------------------------------------------------
// Allocation-free entry: the same kernels with their scratch in a file-scope
// device array instead of a caller workspace.
// ---------------------------------------------------------------------------
constexpr size_t kNoAllocBytes = layout(kDeviationNoAllocMaxN).total;
static __device__ __align__(256) unsigned char g_deviation_scratch[kNoAllocBytes];

namespace {
std::mutex g_scratch_mu;
void *g_scratch_ptr[64];   // device address of g_deviation_scratch, per device (stale after a
                           // cudaDeviceReset of that device: the header says not to call then)
}  // namespace

int launch_deviation_noalloc(const void *a, int ta, const void *b, int tb, long long n, cudaStream_t stream,
                             double *host_result) {
    if (n > kDeviationNoAllocMaxN) return kErrUnsupported;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return kErrCuda;
    void *ws = nullptr;
    {
        // Set-up, once per device, with that device current: the host-side
        // name of the array is only a stand-in, so ask the runtime for its
        // device address.
        std::lock_guard<std::mutex> lk(g_scratch_mu);
        if (!g_scratch_ptr[dev]) {
            void *ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_deviation_scratch) != cudaSuccess || ptr == nullptr) return kErrCuda;
            g_scratch_ptr[dev] = ptr;
        }
        ws = g_scratch_ptr[dev];
    }
    // Every scratch word the kernels read is written earlier in the same call
    // (keys, histograms, scans, partial sums, result), so nothing needs clearing.
    double *dev_result = reinterpret_cast<double *>(static_cast<char *>(ws) + layout(n).result);
    const int rc = launch_deviation(a, ta, b, tb, n, ws, stream, dev_result);
    if (rc != kOk) return rc;
    if (cudaMemcpyAsync(host_result, dev_result, 5 * sizeof(double), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return kErrCuda;
    return cudaStreamSynchronize(stream) == cudaSuccess ? kOk : kErrCuda;
}

size_t deviation_workspace_bytes(long long n) { return layout(n).total; }
size_t deviation_result_offset(long long n) { return layout(n).result; }

int launch_deviation(const void *a, int ta, const void *b, int tb, long long n, void *workspace,
                     cudaStream_t stream, double *dev_result) {
    if (n >= (1LL << 32) - 1) return kErrUnsupported;
    const Layout L = layout(n);
    char *ws = static_cast<char *>(workspace);
    uint64_t *ka = reinterpret_cast<uint64_t *>(ws + L.keys_a);
    uint64_t *kb = reinterpret_cast<uint64_t *>(ws + L.keys_b);
    uint64_t *tmp = reinterpret_cast<uint64_t *>(ws + L.tmp);
    double *part = reinterpret_cast<double *>(ws + L.part);
    dev_convert_kernel<<<kRedBlocks, kRedThreads, 0, stream>>>(a, ta, b, tb, n, ka, kb, part);
    dev_finalize_kernel<<<1, kRedThreads, 0, stream>>>(part, kRedBlocks, n, 0, dev_result);
    dev_var_kernel<<<kRedBlocks, kRedThreads, 0, stream>>>(a, ta, b, tb, n, dev_result, part);
    dev_finalize_kernel<<<1, kRedThreads, 0, stream>>>(part, kRedBlocks, n, 1, dev_result);
    int rc = radix_sort(ka, tmp, n, L, ws, stream);
    if (rc != kOk) return rc;
    rc = radix_sort(kb, tmp, n, L, ws, stream);
    if (rc != kOk) return rc;
    dev_w1_kernel<<<kRedBlocks, kRedThreads, 0, stream>>>(ka, kb, n, part);
    dev_finalize_kernel<<<1, kRedThreads, 0, stream>>>(part, kRedBlocks, n, 2, dev_result);
    return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

}  // namespace eta
