// Internal interfaces between the C-ABI layer (attn_api.cu) and the kernel
// translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cstddef>
#include <cuda.h>
#include <cuda_runtime.h>

namespace eta {

// Status codes (mirror attn_status_t in include/attn.h).
constexpr int kOk = 0;
constexpr int kErrArg = -1;
constexpr int kErrUnsupported = -2;
constexpr int kErrWorkspace = -3;
constexpr int kErrCuda = -4;
constexpr int kErrDeviceTimeout = -5;

// cuTensorMapEncodeTiled, fetched from the driver at run time.
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

// Tensor map of a bf16 [BH][N][D] tensor for 128-byte-swizzled boxes of
// 64 columns x box_rows rows (the tile layout of the tcgen05 kernels); rows
// past N read as zero and are dropped on store.
bool make_bf16_rows_map(CUtensorMap *m, const void *base, int D, int N, int BH, int box_rows);

// Error-word bit set by the emulation kernel for an out-of-range row id
// (timed-out waits use the low bits).
constexpr int kErrWordBadRow = 1 << 24;

// Device address of the library's error word on the current device (or null).
int *device_error_word();

// BF16 tiled forward on tcgen05 (fwd_tc.cu).  variant receives a static name.
int launch_fwd_tc_bf16(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                       int N, int d, int causal, float scale, int Br, int Bc, const float *key_mask,
                       cudaStream_t stream, const char **variant);

// Block-sparse BF16 forward (fwd_tc.cu): 128 x 128 blocks, block_mask [B*H][nb][nb] bytes.
constexpr int kBlockSparseBlock = 128;
constexpr int kBlockSparseMaxN = 131072;
int launch_fwd_tc_bf16_bsparse(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                               int N, int d, int causal, float scale, const unsigned char *block_mask,
                               const float *key_mask, cudaStream_t stream, const char **variant);

// FP32 tiled forward on the CUDA cores (fwd_f32.cu).
int launch_fwd_f32(const float *Q, const float *K, const float *V, float *O, float *LSE, int B, int H,
                   int N, int d, int causal, float scale, const float *key_mask, cudaStream_t stream,
                   const char **variant);

// Materialising baseline (naive.cu).  dtype: 0 f32, 1 bf16.
int launch_naive(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H, int N,
                 int d, int causal, float scale, int dtype, const float *key_mask, void *workspace,
                 cudaStream_t stream);

// Deviation measures (deviation.cu).
size_t deviation_workspace_bytes(long long n);
int launch_deviation(const void *a, int ta, const void *b, int tb, long long n, void *workspace,
                     cudaStream_t stream, double *dev_result /* 5 doubles inside workspace */);
size_t deviation_result_offset(long long n);

// Allocation-free deviation (scratch in a static device array of deviation.cu).
constexpr long long kDeviationNoAllocMaxN = 1LL << 20;
int launch_deviation_noalloc(const void *a, int ta, const void *b, int tb, long long n, cudaStream_t stream,
                             double *host_result /* 5 doubles */);

// Number-format emulation (emul.cu).  dtype: 0 f32, 1 bf16, 2 f64.
size_t emul_smem_bytes(int algo, int N, int Bc);
int launch_emul(const void *Q, const void *K, const void *V, int dtype, double *O, int B, int H, int N, int d,
                int causal, float scale, const float *key_mask, int algo, int Bc, int mbits, int ebits,
                const long long *rows, long long nrows, cudaStream_t stream);
int launch_fmt_round(const double *x, double *y, long long n, int mbits, int ebits, cudaStream_t stream);

// Decode with a key/value cache (decode.cu).
constexpr int kDecodeMaxSplits = 128;
size_t decode_workspace_bytes(int BH, int Nq, int d);
int launch_decode(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H, int Nq, int Nk,
                  int d, int causal, float scale, int bf16, const float *key_mask, void *workspace,
                  cudaStream_t stream);

// FP32 backward on the CUDA cores (bwd_f32.cu); workspace: B*H*N floats.
int launch_bwd_f32(const float *Q, const float *K, const float *V, const float *O, const float *dO, const float *LSE,
                   float *dQ, float *dK, float *dV, int B, int H, int N, int d, int causal, float scale,
                   const float *key_mask, void *workspace, cudaStream_t stream);

// Backward on tcgen05 (bwd_tc.cu).
size_t bwd_workspace_bytes(int BH, int N, int d);
int launch_bwd_tc_bf16(const void *Q, const void *K, const void *V, const void *O, const void *dO, const float *LSE,
                       void *dQ, void *dK, void *dV, int B, int H, int N, int d, int causal, float scale,
                       const float *key_mask, void *workspace, cudaStream_t stream);

// Bounded-wait self-test kernel (attn_api.cu).
int launch_wait_timeout_probe(unsigned timeout_us, cudaStream_t stream);

}  // namespace eta
