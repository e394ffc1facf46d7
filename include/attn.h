/*
 * Exact tiled attention forward on one NVIDIA GB300 (sm_103a): C ABI.
 *
 * Library: exact_tiled_attention_17_gb300/libattn.so.  Every entry point has
 * C linkage and takes plain pointers and sizes.  No entry point allocates
 * device memory: tensors and workspaces are owned by the caller.  Work is
 * enqueued on the caller's stream (a cudaStream_t passed as void*; NULL means
 * the legacy default stream) on the current device.  The tensor-core forward,
 * the backward and the decode kernels are programmatic dependent launches:
 * each may be scheduled while the kernel before it in the stream finishes,
 * but reads or writes no global memory until that grid has completed, so
 * stream order holds as for an ordinary launch.
 *
 * Errors are reported synchronously through the return value and nothing is
 * launched when an argument is rejected.  There is no CPU fallback and no
 * other backend: a missing GPU or an unsupported device returns
 * ATTN_ERR_CUDA / ATTN_ERR_UNSUPPORTED.  Errors found while a kernel runs
 * (a bounded wait that ran out) are recorded in a device-side error word that
 * attn_status() reads.
 *
 * The computation is the attention of "Is Flash Attention Stable?" §II-A,
 *     O = softmax(Q K^T * scale + mask) V,
 * evaluated as in its §II-B (Fig. 1): tile by tile, without materialising the
 * N x N score matrix, with the online-softmax rescale of the yadro-code.ru
 * FlashAttention tutorial (running row maximum m, running denominator l,
 * unnormalised accumulator multiplied by exp(m_old - m_new) when the maximum
 * grows, one division at the end).
 *
 * Common conventions
 *   Q, K, V, O   [B][H][N][d] row-major, contiguous, device memory, base
 *                pointers 16-byte aligned.  O has the dtype of Q/K/V.
 *   LSE          [B][H][N] float32, device memory, natural-log log-sum-exp of
 *                each row's scaled and masked scores; may be NULL (not written).
 *   causal       0 or 1.  Top-left aligned: query i sees keys j <= i (the
 *                tutorial's causal prefixes).
 *   scale        multiplies Q K^T; callers normally pass 1/sqrt(d).  Must be
 *                finite and > 0.
 *   key_mask     NULL, or [B][H][N] float32 device memory added to every row's
 *                score of key j (a key-padding mask).  Entries must be finite
 *                or -inf; -inf removes the key.  There is no finite "masked"
 *                sentinel anywhere in the library: the aicompass.dev note on
 *                FlashInfer kernels shows why a hard-coded -50,000 is wrong.
 *                On the bf16 tensor-core path the mask enters the score
 *                product: mask / scale (formed as mask times the float32
 *                reciprocal of scale), split into three bf16 parts that carry
 *                that float32 value exactly, is added to q.k before the scale
 *                is applied (equal to scale * q.k + mask up to float32
 *                rounding); a finite mask / scale beyond the bf16 range
 *                (about 3.39e38) is clamped to it.
 *   A row whose every score is -inf (fully masked) outputs O = 0 and
 *   LSE = -inf, with no NaN.  (The tutorial assumes each row has an allowed
 *   key and leaves this case to be defined; this is the definition.)
 */
#ifndef EXACT_TILED_ATTENTION_ATTN_H
#define EXACT_TILED_ATTENTION_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { ATTN_F32 = 0, ATTN_BF16 = 1, ATTN_F64 = 2 } attn_dtype_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_ARG = -1,            /* null pointer, bad size, bad alignment, bad scale      */
    ATTN_ERR_UNSUPPORTED = -2,    /* valid but not implemented: d, Br/Bc, dtype, device    */
    ATTN_ERR_WORKSPACE = -3,      /* workspace NULL or smaller than the size query returns */
    ATTN_ERR_CUDA = -4,           /* a CUDA runtime/driver call failed                     */
    ATTN_ERR_DEVICE_TIMEOUT = -5  /* a kernel's bounded wait ran out (see attn_status)     */
} attn_status_t;

/*
 * attn_fwd — the tiled exact forward pass ("Is Flash Attention Stable?"
 * §II-B and Fig. 1; the tutorial's online merge).
 *
 * dtype ATTN_BF16: Q/K/V/O bfloat16.  Both contractions run on the tcgen05
 *   tensor cores with bf16 operands and float32 accumulation in tensor
 *   memory; softmax state (m, l) and the accumulator stay float32; the
 *   probabilities P are rounded to bf16 (round-to-nearest-even) as the
 *   operand of the second contraction and O is rounded to bf16 at the end.
 *   d must be 64 or 128.  Br in {64, 128}, Bc in {64, 128, 256}; 0 selects
 *   128 for either, except Bc = 0 with causal, d = 64 and N <= 1024, which
 *   selects 64.
 * dtype ATTN_F32: Q/K/V/O float32, every operation in float32 on the CUDA
 *   cores (no TF32).  1 <= d <= 128.  Br and Bc must be 0 or 64.
 * N >= 1 with any tail; B, H >= 1; B*H*N < 2^31 rows.
 * Asynchronous: returns after enqueueing on `stream`.
 */
int attn_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE,
             int B, int H, int N, int d, int causal, float scale, int Br, int Bc,
             int dtype, const float *key_mask, void *stream);

/*
 * attn_fwd_host — attn_fwd on host memory: the same computation ("Is Flash
 * Attention Stable?" §II-A), for a caller whose Q, K, V live in host memory
 * (the end-to-end path: inputs in, results out).  On `stream` it copies Q, K,
 * V (and the key mask) into `workspace`, runs attn_fwd there, and copies O
 * (and LSE) back.
 *
 * Qh, Kh, Vh: host [B][H][N][d] of `dtype`; Oh: host [B][H][N][d] of `dtype`
 * (written); LSEh: host [B][H][N] float32 (written) or NULL; key_mask_h: host
 * [B][H][N] float32 additive mask or NULL.  All host buffers are the
 * caller's; page-locked (pinned) memory lets the copies overlap other work,
 * pageable memory also works but the copies then wait for the host.
 * workspace: device memory of at least attn_fwd_host_workspace_size(B, H, N,
 * d, dtype, key_mask_h != NULL) bytes, 256-byte aligned, owned by the caller
 * and holding the device copies while the call runs.  Other arguments and
 * errors as for attn_fwd; argument errors are returned before anything is
 * enqueued.  Asynchronous: Oh / LSEh hold the result once `stream` has been
 * synchronised, and the host buffers must stay valid until then.
 */
size_t attn_fwd_host_workspace_size(int B, int H, int N, int d, int dtype, int with_mask);
int attn_fwd_host(const void *Qh, const void *Kh, const void *Vh, void *Oh, float *LSEh, int B, int H, int N, int d,
                  int causal, float scale, int Br, int Bc, int dtype, const float *key_mask_h, void *workspace,
                  size_t ws_bytes, void *stream);

/*
 * attn_fwd_block_sparse — the forward of attn_fwd restricted to marked blocks
 * of the score matrix.  The yadro-code.ru FlashAttention tutorial notes that
 * the method's paper also treats a block-sparse extension; read plainly, a
 * block mask says which (query block, key block) pairs take part, every other
 * score is -inf before the softmax, and the kernel skips the key tiles no
 * query tile of a CTA needs.  A query row whose blocks are all unmarked (or
 * that sees no allowed key inside them) gets O = 0, LSE = -inf.
 *
 * block_mask: [B][H][nb][nb] bytes, nb = ceil(N / ATTN_BLOCK_SPARSE_BLOCK),
 * device memory, non-zero = the block takes part; block (i, j) covers query
 * rows 128i .. 128i+127 and keys 128j .. 128j+127.  Other arguments as
 * attn_fwd (key_mask and causal apply on top of the block mask).  dtype must
 * be ATTN_BF16, d 64 or 128 and N <= ATTN_BLOCK_SPARSE_MAX_N, else
 * ATTN_ERR_UNSUPPORTED; block_mask NULL is ATTN_ERR_ARG.  Asynchronous.
 */
#define ATTN_BLOCK_SPARSE_BLOCK 128
#define ATTN_BLOCK_SPARSE_MAX_N 131072
int attn_fwd_block_sparse(const void *Q, const void *K, const void *V, void *O, float *LSE,
                          int B, int H, int N, int d, int causal, float scale, int dtype,
                          const unsigned char *block_mask, const float *key_mask, void *stream);

/*
 * attn_naive_workspace_size — bytes of workspace attn_naive_fwd needs:
 * B*H*N*N elements of the input dtype (the materialised score matrix; the
 * tutorial's arithmetic: 8192 tokens x 2 bytes = 128 MiB per head, 4 GiB for
 * 32 heads).  Returns 0 for invalid arguments or on overflow.
 */
size_t attn_naive_workspace_size(int B, int H, int N, int dtype);

/*
 * attn_naive_fwd — "baseline attention" (the paper's §IV comparison point):
 * materialises S = Q K^T * scale + mask in the caller's workspace, stored in
 * the input dtype; a row softmax with float32 arithmetic overwrites S with
 * P, stored in the input dtype; then O = P V with float32 accumulation,
 * stored in the input dtype.  Same masking, causal and fully-masked-row
 * conventions as attn_fwd.  dtype ATTN_F32 or ATTN_BF16, 1 <= d <= 128.
 * workspace: device memory of at least attn_naive_workspace_size() bytes.
 * Asynchronous.
 */
int attn_naive_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE,
                   int B, int H, int N, int d, int causal, float scale, int dtype,
                   const float *key_mask, void *workspace, size_t ws_bytes, void *stream);

/*
 * Deviation between two tensors (the paper's §IV-A maximum element-wise
 * difference and §V Wasserstein distance; the pages' own formulas were lost
 * in extraction, these are the standard definitions):
 *   max_abs     = max_i |a_i - b_i|
 *   w1          = 1-D Wasserstein-1 between the empirical value distributions
 *                 of a and b, (1/n) * sum_i |sort(a)_i - sort(b)_i|
 *   mean_abs    = mean of |a_i - b_i|;   std_abs = its population std
 *   mean_signed = mean of (a_i - b_i)
 * Elements where a_i == b_i (including equal infinities) contribute 0.
 * All arithmetic is float64; inputs are converted exactly.
 */
typedef struct {
    double max_abs, w1, mean_abs, std_abs, mean_signed;
    long long n;
} attn_dev_t;

/* Bytes of device workspace attn_deviation needs for n elements (0 if n <= 0). */
size_t attn_deviation_workspace_size(long long n);

/*
 * attn_deviation — a (dtype ta) and b (dtype tb): n elements each, device
 * memory, any of ATTN_F32 / ATTN_BF16 / ATTN_F64, naturally aligned.
 * workspace: device memory of at least attn_deviation_workspace_size(n)
 * bytes, 256-byte aligned.  Synchronous: waits for `stream` and writes the
 * result to the host struct *out.
 */
int attn_deviation(const void *a, int ta, const void *b, int tb, long long n,
                   void *workspace, size_t ws_bytes, void *stream, attn_dev_t *out);

/*
 * attn_deviation_noalloc — the same measures as attn_deviation for callers
 * that cannot allocate device memory: for example a plain C host program
 * with no device allocator of its own, or a process whose device memory is
 * already reserved up front by another framework's caching pool, where a
 * cudaMalloc for a workspace would fail or break that pool's accounting.
 * (The paper has no counterpart: this is a convenience of the library.)
 *
 * Instead of a caller workspace it uses one scratch array that the library
 * keeps in device memory for the life of the process on every GPU that loads
 * it: about 24 MiB, enough for n <= ATTN_DEVIATION_NOALLOC_MAX_N elements.
 * Larger n returns ATTN_ERR_UNSUPPORTED (use attn_deviation with a workspace).
 * It calls no cudaMalloc or cudaFree.  The first call on a device looks up
 * the array's device address on that device; make that first call before
 * any stream capture begins.  That address is kept for the life of the
 * process: after a cudaDeviceReset of a device it is stale (the runtime loads
 * the array again elsewhere), so do not call this entry point on a device
 * that has been reset.  All calls share the one array, so calls that
 * can overlap on the GPU (different streams or threads at the same time)
 * race with each other and must be serialised by the caller.  Arguments and
 * result as for attn_deviation; synchronous.
 */
#define ATTN_DEVIATION_NOALLOC_MAX_N 1048576LL
int attn_deviation_noalloc(const void *a, int ta, const void *b, int tb, long long n, void *stream,
                           attn_dev_t *out);

/*
 * attn_decode_fwd — decode with a key/value cache: attention of Nq new query
 * rows against Nk cached keys and values, the same exact attention as
 * attn_fwd ("Is Flash Attention Stable?" §II-A), evaluated by splitting the
 * keys into chunks and merging the chunks' partial results with the
 * yadro-code.ru tutorial's rule for joining two blocks (common maximum,
 * weights exp(m - M)).
 *
 * Q: [B][H][Nq][d]; K, V: [B][H][Nk][d] (the cache); O: [B][H][Nq][d], all of
 * `dtype` (ATTN_BF16 or ATTN_F32), 16-byte aligned.  LSE: [B][H][Nq] float32
 * natural log, or NULL.  key_mask: NULL or [B][H][Nk] additive (finite or
 * -inf).  causal: query row i is the token at position Nk - Nq + i and sees
 * keys j <= Nk - Nq + i (needs Nq <= Nk); otherwise every row sees every
 * key.  A row with no allowed key gives O = 0, LSE = -inf.
 * 1 <= Nq <= ATTN_DECODE_MAX_NQ and d in {32, 64, 96, 128}, else
 * ATTN_ERR_UNSUPPORTED.  workspace: device memory of at least
 * attn_decode_workspace_size(B, H, Nq, d) bytes, 16-byte aligned, for the
 * chunks' partial results.  HBM-bound: runs on the CUDA cores.  Asynchronous.
 */
#define ATTN_DECODE_MAX_NQ 8
size_t attn_decode_workspace_size(int B, int H, int Nq, int d);
int attn_decode_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE,
                    int B, int H, int Nq, int Nk, int d, int causal, float scale, int dtype,
                    const float *key_mask, void *workspace, size_t ws_bytes, void *stream);

/*
 * attn_bwd — gradients of exact attention: for O = softmax(Q K^T * scale +
 * mask) V ("Is Flash Attention Stable?" §II-A) and an upstream gradient dO,
 * dQ, dK and dV.  As the yadro-code.ru FlashAttention tutorial describes for
 * the method's backward pass, intermediate values are recomputed rather than
 * stored: the attention weights are formed again, tile by tile, from Q, K and
 * the forward's per-row LSE, P = exp(s - LSE); nothing of size N x N is kept.
 *
 * Q, K, V, O, dO: [B][H][N][d] bfloat16 (O and LSE as attn_fwd wrote them for
 * these Q, K, V, causal, scale and mask); LSE: [B][H][N] float32 natural log
 * (-inf for a row with no allowed key: its gradients are 0).  dQ, dK, dV:
 * [B][H][N][d] bfloat16, written.  All tensor pointers 16-byte aligned,
 * caller-owned device memory.  key_mask: NULL or [B][H][N] additive (finite
 * or -inf), a constant (no gradient is formed for it).  causal as attn_fwd.
 * dtype ATTN_BF16 (tensor cores; d 64 or 128) or ATTN_F32 (all tensors
 * float32, including dQ, dK, dV; CUDA cores, IEEE float32 throughout, no
 * atomics; d <= 128), else ATTN_ERR_UNSUPPORTED.
 * workspace: at least attn_bwd_workspace_size(B, H, N, d) bytes of device
 * memory, 256-byte aligned (the rows' LSE and D = rowsum(dO * O) vectors and
 * a float32 dQ accumulator), else ATTN_ERR_WORKSPACE.  Asynchronous: three
 * launches on `stream`; errors in the arguments are returned before any
 * launch.  bf16: dQ is accumulated with floating-point reductions from many
 * CTAs, so its last bits can differ from run to run; dK and dV are
 * deterministic.  float32: all three are deterministic.
 */
size_t attn_bwd_workspace_size(int B, int H, int N, int d);
int attn_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO, const float *LSE,
             void *dQ, void *dK, void *dV, int B, int H, int N, int d, int causal, float scale, int dtype,
             const float *key_mask, void *workspace, size_t ws_bytes, void *stream);

/*
 * Number-format emulation — the instrument of "Is Flash Attention Stable?"
 * §III (Fig. 2): a numerical re-implementation of FlashAttention and of the
 * baseline that can run in any number format and whose internals can be
 * changed, used for the format sweep of §IV-A (Fig. 3) and the block-size
 * perturbations of §IV-B (Fig. 6).  The pages give no code for it; the
 * reading implemented here:
 *
 *  - A format has `mbits` fraction bits (1..52) and `ebits` exponent bits
 *    (2..11), IEEE style: subnormals, round to nearest with ties to even,
 *    overflow to infinity.  bf16 = (7, 8), fp16 = (10, 5), tf32 = (10, 8),
 *    fp32 = (23, 8), fp64 = (52, 11).  fl(x) is x rounded to the format.
 *  - Every tensor operation produces its result in the format: elementwise
 *    operations are evaluated in binary64 and rounded once; reductions (row
 *    sum, row maximum) and matrix products accumulate in binary64 and round
 *    their result once.  Q, K and V are rounded to the format first.
 *  - scores s_j = fl(scale * (q . k_j)), then fl(s_j + mask_j) with a key
 *    mask (a -inf mask entry, or a causal future key, gives -inf).
 *  - ATTN_EMUL_BASELINE: P = fl(softmax(s)) as one operation, O = fl(P V).
 *  - ATTN_EMUL_TILED: the online merge over key blocks of width Bc, in
 *    order: M = max(m, max_j s_j), M' = (M == -inf ? 0 : M),
 *    a = fl(exp(fl(m - M'))) (0 while m is -inf), p_j = fl(exp(fl(s_j - M'))),
 *    l = fl(fl(a*l) + fl(sum_j p_j)), o = fl(fl(a*o) + fl(sum_j p_j v_j));
 *    finally O = fl(o / l), or 0 for a row with no allowed key.  Only the key
 *    block width Bc changes a row's arithmetic; the query block height only
 *    groups rows.
 *
 * attn_emul_fwd — Q, K, V: device, [B][H][N][d] of `dtype` (ATTN_F32,
 * ATTN_BF16 or ATTN_F64), naturally aligned; key_mask as for attn_fwd.
 * rows: device array of `nrows` flat row ids (bh * N + i), 8-byte aligned,
 * or NULL for every row (nrows ignored).  O: device float64 [nrows][d]
 * (or [B*H*N][d]), 8-byte aligned, row r for rows[r].  1 <= d <= 128;
 * ATTN_EMUL_BASELINE needs N <= ATTN_EMUL_MAX_N_BASELINE (else
 * ATTN_ERR_UNSUPPORTED); ATTN_EMUL_TILED needs 1 <= Bc <= ATTN_EMUL_MAX_BC.
 * A row id out of range is skipped (its output row is left as it was) and
 * the next attn_status() returns ATTN_ERR_ARG.  Binary64 arithmetic on the
 * CUDA cores: a measurement tool, not a fast path.  Asynchronous.
 */
#define ATTN_EMUL_BASELINE 0
#define ATTN_EMUL_TILED 1
#define ATTN_EMUL_MAX_N_BASELINE 16384
#define ATTN_EMUL_MAX_BC 4096
int attn_emul_fwd(const void *Q, const void *K, const void *V, int dtype, double *O,
                  int B, int H, int N, int d, int causal, float scale, const float *key_mask,
                  int algo, int Bc, int mbits, int ebits, const long long *rows, long long nrows,
                  void *stream);

/*
 * attn_emul_round — y[i] = fl(x[i]) for n float64 values in device memory
 * (8-byte aligned; y may equal x), in the format (mbits, ebits) described
 * above.  Asynchronous.
 */
int attn_emul_round(const double *x, double *y, long long n, int mbits, int ebits, void *stream);

/*
 * attn_status — waits for `stream`, then returns ATTN_ERR_DEVICE_TIMEOUT if a
 * kernel of this library recorded a timed-out wait since the last call,
 * ATTN_ERR_ARG if attn_emul_fwd met an out-of-range row id, and clears the
 * record; ATTN_ERR_CUDA if the stream reports a CUDA error, else ATTN_OK.
 */
int attn_status(void *stream);

/* attn_strerror — static text for a status code. */
const char *attn_strerror(int status);

/*
 * attn_last_variant — writes the name of the kernel variant the last
 * successful attn_fwd call on this thread launched (e.g.
 * "tc_bf16_d128_br128_bc128_nq2") into buf (NUL-terminated, truncated to
 * len).  Returns the full length, or ATTN_ERR_ARG.
 */
int attn_last_variant(char *buf, int len);

/*
 * attn_debug_wait_timeout — self-test of the device-side failure path: one
 * small kernel waits on a shared-memory barrier that nothing will ever
 * complete, gives up after `timeout_us` microseconds (1 .. 10^6), records
 * ATTN_ERR_DEVICE_TIMEOUT in the error word and returns.  The context stays
 * usable; the next attn_status() reports the timeout and clears it.
 */
int attn_debug_wait_timeout(unsigned timeout_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_TILED_ATTENTION_ATTN_H */
