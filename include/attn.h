/*
 * attn.h -- C ABI of libattn, exact softmax attention (forward and backward)
 * for NVIDIA GB300 (sm_103a).
 *
 * What is computed.  For every (b, h) head independently, with Q, K, V of
 * shape (n, d) and s_ij = scale * q_i . k_j:
 *
 *   forward   O = softmax(S) V,  LSE_i = ln sum_j exp(s_ij)
 *             ("Chapter 3.1 -- The cost of attention", section 2, the scaled
 *             dot-product formula; "Flash Attention: Revolutionizing
 *             Transformer Efficiency", "Standard attention: a quick summary")
 *   backward  for a scalar loss with gradient dO = dL/dO:
 *             P = exp(S - LSE), dV = P^T dO, dP = dO V^T, D_i = dO_i . O_i,
 *             dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q
 *             (the pages name the backward pass and its recomputation of P --
 *             "Chapter 3.1", section 5; "On the fine-grained I/O complexity
 *             of attention backward passes", Methodology -- but print no
 *             formulas; these are the exact chain-rule derivatives).
 *   causal    optional mask: s_ij = -inf for j > i (applied before the row
 *             maximum, so P_ij = 0 there).
 *
 * Conventions shared by every entry point:
 *   - Tensors are DEVICE pointers to contiguous row-major [B][H][n][d]
 *     arrays (d innermost).  LSE and D are fp32 [B][H][n], natural log.
 *     Q, K, V, O, dO, dQ, dK, dV share one element type (attn_dtype).
 *   - Every pointer must be 16-byte aligned.  Outputs are fully
 *     overwritten and must not alias any input.
 *   - The caller owns every buffer.  The library never allocates device
 *     memory, never frees, and never synchronises, except attn_status().
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and runs asynchronously.  The return value reports argument
 *     and launch errors only (attn_status_t, 0 = success).  Errors detected
 *     on the device (a bounded wait that ran out) are recorded in a device
 *     status word read by attn_status().
 *   - bf16 path: d in {64, 128, 256}; fp32 path: 1 <= d <= 256.  Any n with
 *     1 <= n <= 8388480 (65535 tiles of 128 rows; ATTN_ERR_UNSUPPORTED above),
 *     B * H <= 65535.
 *   - Thread-safe: the only global state is the device status word, the
 *     fixed scratch of attn_bwd_noalloc and an atomic launch counter.
 */
#ifndef ATTN_H
#define ATTN_H

#include <stddef.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { ATTN_BF16 = 0, ATTN_F32 = 1 } attn_dtype;

/* How attn_bwd combines dQ = scale * sum_j dS_ij k_j across key tiles. */
typedef enum {
  ATTN_DQ_AUTO = 0,   /* the measured default for the shape: ATTN_DQ_ATOMIC
                         for d <= 128; for d = 256 ATTN_DQ_SPILL when that
                         mode applies and its dS^T buffer is at most 4 GiB,
                         else ATTN_DQ_PASS (the workspace-size functions
                         make the same choice) */
  ATTN_DQ_ATOMIC = 1, /* key-tile kernel adds its dQ share into an fp32
                         workspace accumulator with atomics, then converts */
  ATTN_DQ_PASS = 2,   /* separate query-tile kernel recomputes S, dP, dS and
                         sums dQ with no atomics */
  ATTN_DQ_SPILL = 3   /* d = 256, non-causal, dense, one key/value head per
                         query head: the key-tile kernel also writes dS^T
                         (bf16, n x n per head) to the workspace and dQ =
                         scale dS K is one tensor-core GEMM; the workspace
                         grows by B*H*n*round_up(n, 8)*2 bytes.  Trades the
                         pass's second recomputation of S and dP for one
                         n x n write and read through HBM.
                         ATTN_ERR_UNSUPPORTED for other shapes. */
} attn_dq_mode;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, size < 1, bad scale */
  ATTN_ERR_UNSUPPORTED = 2,   /* head dim not supported for this dtype/path */
  ATTN_ERR_WORKSPACE = 3,     /* workspace null, not 256-byte aligned or too small */
  ATTN_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
  ATTN_ERR_DEVICE_TIMEOUT = 5 /* a bounded device-side wait ran out */
} attn_status_t;

/*
 * attn_fwd -- forward pass.
 *   Q, K, V : inputs  [B][H][n][d]
 *   O       : output  [B][H][n][d]
 *   LSE     : output  fp32 [B][H][n], LSE_i = ln sum_j exp(s_ij)
 *   scale   : finite score multiplier (usually 1/sqrt(d))
 *   causal  : 0 or 1
 * bf16: one fused tensor-core kernel (TMA tiles, tcgen05 MMAs with TMEM
 * accumulators, online softmax: "Flash Attention: Revolutionizing
 * Transformer Efficiency", "The mathematics behind Flash Attention",
 * formulas 1-2, with the running-sum factor restored).  fp32: exact fp32
 * SIMT kernel.
 */
ATTN_API int attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
             int B, int H, int n, int d, attn_dtype dtype, float scale,
             int causal, void* stream);

/*
 * attn_bwd_workspace_size -- bytes of device workspace attn_bwd needs for
 * this shape and dQ mode (row statistics, plus the fp32 dQ accumulator in
 * ATTN_DQ_ATOMIC mode).  Returns 0 for invalid arguments.
 */
ATTN_API size_t attn_bwd_workspace_size(int B, int H, int n, int d, attn_dtype dtype,
                               int causal, attn_dq_mode mode);

/*
 * attn_bwd -- backward pass.
 *   Q, K, V, O, dO : inputs [B][H][n][d]; O is the forward output.
 *   LSE            : input fp32 [B][H][n] from attn_fwd.
 *   dQ, dK, dV     : outputs [B][H][n][d].
 *   workspace      : device buffer of at least attn_bwd_workspace_size(...)
 *                    bytes, 256-byte aligned, owned by the caller; contents
 *                    on entry are ignored.
 * Computes D = rowsum(dO o O) in a preprocessing kernel, then recomputes P
 * from LSE tile by tile (P is never stored), accumulating dK and dV per key
 * tile in tensor memory.
 */
ATTN_API int attn_bwd(const void* Q, const void* K, const void* V, const void* O,
             const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
             int B, int H, int n, int d, attn_dtype dtype, float scale,
             int causal, attn_dq_mode mode, void* workspace,
             size_t workspace_bytes, void* stream);

/*
 * Grouped-query and multi-query attention ("Flash Attention: Revolutionizing
 * Transformer Efficiency", section FlashAttention-2, item 3, names both as
 * variants the method supports).  H query heads share H_kv key/value heads:
 * query head h of batch b reads key/value head h / (H / H_kv) of batch b.
 * H_kv must divide H; H_kv = H is attn_fwd / attn_bwd, H_kv = 1 is
 * multi-query attention.
 *   Q, O, dO, dQ : [B][H][n][d];  LSE : fp32 [B][H][n]
 *   K, V, dK, dV : [B][H_kv][n][d]
 * dK and dV of a key/value head are the sums over the query heads that read
 * it: the key-tile kernel walks the query tiles of every head of the group,
 * so the sums accumulate in tensor memory.  When B * H_kv * ceil(n / 128)
 * key-tile CTAs would leave the GPU short of work, the group is split over
 * several CTAs per key/value head that add their partial sums into fp32
 * accumulators in the workspace (then converted); the workspace is
 * attn_bwd_gqa_workspace_size(...) bytes (0 for invalid arguments).  Other
 * arguments, layouts and errors as attn_fwd / attn_bwd, plus
 * ATTN_ERR_INVALID_ARG when H_kv < 1 or H_kv does not divide H.  The
 * materialise-P comparison path (attn_mat_*) has no grouped form.
 */
ATTN_API int attn_fwd_gqa(const void* Q, const void* K, const void* V, void* O, float* LSE,
                          int B, int H, int H_kv, int n, int d, attn_dtype dtype, float scale,
                          int causal, void* stream);
/*
 * attn_fwd_fp8 -- forward pass with FP8 (e4m3) operands on the FP8 tensor
 * cores ("Flash Attention: Revolutionizing Transformer Efficiency", section
 * FlashAttention-3, item 2: FP8 computation).  Head dim 128 only; n a
 * multiple of 16 (ATTN_ERR_UNSUPPORTED otherwise).
 *   Q8, K8 : DEVICE e4m3 bytes [B][H][n][128]
 *   Vt8    : DEVICE e4m3 bytes [B][H][128][n]  (V transposed: every FP8
 *            operand of the tensor cores is then K-major)
 *   O      : output bf16 [B][H][n][128];  LSE : output fp32 [B][H][n]
 *   descale_q, descale_k, descale_v : DEVICE fp32 [B*H] per-head scales
 *            (real value = descale x e4m3 value), or NULL for 1; as written
 *            by attn_quantize_fp8.  4-byte aligned.
 * Computes softmax(scale * dq[h] * dk[h] * Q8 K8^T) (dv[h] V8) with fp32
 * accumulation; the probabilities P are rounded to e4m3 before the P V
 * product, while the row sums use the unrounded fp32 values, so
 * O - O_ref = sum_j (e4m3(p_j) - p_j) v_j / l.  Each rounding is at most
 * 2^-4 of p_j (P <= 2^8 by the running-maximum rule, inside e4m3's range)
 * and, for random inputs, unbiased, which puts the RMS of O - O_ref near
 * 0.027 of the RMS of O_ref (the RMS relative rounding error of e4m3).
 * Tested against the exact result on the same e4m3 inputs: RMS ratio
 * <= 0.035, max|O - O_ref| <= 0.08 max|O_ref|, LSE to 1e-5 relative.
 */
ATTN_API int attn_fwd_fp8(const void* Q8, const void* K8, const void* Vt8, void* O, float* LSE,
                          int B, int H, int n, int d, float scale, const float* descale_q,
                          const float* descale_k, const float* descale_v, int causal,
                          void* stream);

/*
 * attn_quantize_fp8 -- per-head e4m3 encoding of a bf16 attention operand
 * for attn_fwd_fp8, with the optional rotation of incoherent processing
 * ("Flash Attention: Revolutionizing Transformer Efficiency", section
 * FlashAttention-3, items 2 and 3).
 *   X        : DEVICE bf16 [BH][n][d], d = 128 (ATTN_ERR_UNSUPPORTED else)
 *   X8       : DEVICE output e4m3 bytes, [BH][n][128], or [BH][128][n] when
 *              transpose = 1 (for V; n must then be a multiple of 16)
 *   descale  : DEVICE output fp32 [BH]: amax_h / 448 (1 for a zero head)
 *   signs    : DEVICE fp32 [128] of +1 / -1, or NULL.  When given, each row
 *              x is replaced by x diag(signs) H_128 / sqrt(128) (H the
 *              Sylvester Hadamard matrix) before encoding; use the same
 *              signs for Q and K (their scores are unchanged) and none for V
 *              (transpose with signs is ATTN_ERR_INVALID_ARG).
 *   workspace: DEVICE scratch of attn_quantize_fp8_workspace_size bytes.
 * codes = round-to-nearest-even e4m3 of y * (448 / amax_h), saturating at
 * 448.  X, X8 16-byte aligned; descale, signs, workspace 4-byte aligned.
 * Two kernels (head maximum, then codes); no synchronisation.
 */
ATTN_API size_t attn_quantize_fp8_workspace_size(int BH, int n, int d);
ATTN_API int attn_quantize_fp8(const void* X, void* X8, float* descale, int BH, int n, int d,
                               int transpose, const float* signs, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * Block-sparse exact attention.  A block pattern keeps or drops 128 x 128
 * blocks of the score matrix: block_mask is a DEVICE uint8 array
 * [ceil(n/128)][ceil(n/128)] (row = block of 128 queries, column = block of
 * 128 keys; nonzero = kept), shared by every batch and head.  Scores in
 * dropped blocks are -inf (and, when causal, j > i as usual); the kept
 * scores go through the exact softmax, so the result is sparse attention
 * over the pattern ("Chapter 3.1 -- The cost of attention", section 3:
 * Longformer's local windows and global tokens, BigBird's random links;
 * "On the fine-grained I/O complexity of attention backward passes", item
 * 2: sparse attention with Z_QK kept entries).  A query row whose blocks
 * keep no score attends to nothing: O = 0, LSE = -inf, zero gradients (the
 * pages are silent; this is the plain reading).  The kernels visit only the
 * tiles of kept blocks, from per-tile lists they build in the workspace on
 * each call (a few microseconds).  One key/value head per query head only
 * (ATTN_ERR_UNSUPPORTED otherwise); no materialise-P form.
 *   attn_fwd_sparse : workspace of attn_fwd_sparse_workspace_size(n, d)
 *                     bytes (256-byte aligned).
 *   attn_bwd_sparse : workspace of attn_bwd_sparse_workspace_size(...)
 *                     bytes (the attn_bwd workspace plus the lists).
 * Other arguments, layouts and errors as attn_fwd / attn_bwd; a null
 * block_mask is ATTN_ERR_INVALID_ARG.
 */
ATTN_API size_t attn_fwd_sparse_workspace_size(int n, int d);
ATTN_API int attn_fwd_sparse(const void* Q, const void* K, const void* V, void* O, float* LSE,
                             int B, int H, int n, int d, attn_dtype dtype, float scale,
                             int causal, const unsigned char* block_mask, void* workspace,
                             size_t workspace_bytes, void* stream);
ATTN_API size_t attn_bwd_sparse_workspace_size(int B, int H, int n, int d, attn_dtype dtype,
                                               int causal, attn_dq_mode mode);
ATTN_API int attn_bwd_sparse(const void* Q, const void* K, const void* V, const void* O,
                             const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                             int B, int H, int n, int d, attn_dtype dtype, float scale,
                             int causal, attn_dq_mode mode, const unsigned char* block_mask,
                             void* workspace, size_t workspace_bytes, void* stream);

ATTN_API size_t attn_bwd_gqa_workspace_size(int B, int H, int H_kv, int n, int d,
                                            attn_dtype dtype, int causal, attn_dq_mode mode);
ATTN_API int attn_bwd_gqa(const void* Q, const void* K, const void* V, const void* O,
                          const void* dO, const float* LSE, void* dQ, void* dK, void* dV, int B,
                          int H, int H_kv, int n, int d, attn_dtype dtype, float scale,
                          int causal, attn_dq_mode mode, void* workspace,
                          size_t workspace_bytes, void* stream);

/*
 * The three stages attn_bwd runs, exported so a caller can schedule or time
 * them separately (same arguments and workspace as attn_bwd; call them in
 * this order on one stream, with the same dQ mode):
 *   attn_bwd_preprocess  D_i = dO_i . O_i and the log2-scaled LSE into the
 *                        workspace; zeroes the fp32 dQ accumulator
 *                        (ATTN_DQ_ATOMIC).  Bandwidth-bound.
 *   attn_bwd_dkdv        the fused key-tile kernel: recomputes P from LSE and
 *                        writes dK and dV; in ATTN_DQ_ATOMIC mode it also adds
 *                        every dQ share into the workspace accumulator.
 *   attn_bwd_dq          ATTN_DQ_ATOMIC: converts the accumulator to dQ;
 *                        ATTN_DQ_PASS: the query-tile kernel computes dQ.
 * Pointers not used by a stage may be NULL.  attn_bwd_dkdv and attn_bwd_dq
 * are bf16 only: the fp32 kernels read LSE, which these stages do not take,
 * so ATTN_F32 returns ATTN_ERR_INVALID_ARG there (attn_bwd runs fp32).
 */
ATTN_API int attn_bwd_preprocess(const void* O, const void* dO, const float* LSE,
             int B, int H, int n, int d, attn_dtype dtype, int causal,
             attn_dq_mode mode, void* workspace, size_t workspace_bytes,
             void* stream);
ATTN_API int attn_bwd_dkdv(const void* Q, const void* K, const void* V,
             const void* dO, void* dK, void* dV, int B, int H, int n, int d,
             attn_dtype dtype, float scale, int causal, attn_dq_mode mode,
             void* workspace, size_t workspace_bytes, void* stream);
ATTN_API int attn_bwd_dq(const void* Q, const void* K, const void* V,
             const void* dO, void* dQ, int B, int H, int n, int d,
             attn_dtype dtype, float scale, int causal, attn_dq_mode mode,
             void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_bwd_dkdv_keys -- attn_bwd_dkdv with key tiles of key_rows keys (128,
 * 64 or 32; ATTN_ERR_INVALID_ARG otherwise), for measuring how the
 * backward's memory traffic depends on the on-chip memory it works with
 * ("On the fine-grained I/O complexity of attention backward passes",
 * Theorem 1.1: with a cache of M words the tiled backward moves
 * Theta((n^2 d^2 + n d^3) / M) words).  A CTA keeps the K and V rows of its
 * key tile on chip and streams every Q and dO tile past them, so halving
 * key_rows doubles that stream (and the dQ shares added per key tile).  Each
 * CTA still runs the 128-key tile computation but owns only its first
 * key_rows keys (the other keys' probabilities are set to 0), so smaller
 * tiles are also slower; key_rows = 128 is attn_bwd_dkdv.  Results equal
 * attn_bwd_dkdv's up to the order of the dQ additions.  Same arguments and
 * workspace as attn_bwd_dkdv; bf16, one key/value head per query head; d = 64
 * and 128 in ATTN_DQ_ATOMIC (or AUTO) mode only (ATTN_ERR_UNSUPPORTED for
 * ATTN_DQ_PASS), d = 256 in pass mode.
 */
ATTN_API int attn_bwd_dkdv_keys(const void* Q, const void* K, const void* V,
             const void* dO, void* dK, void* dV, int B, int H, int n, int d,
             attn_dtype dtype, float scale, int causal, attn_dq_mode mode,
             int key_rows, void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_bwd_noalloc -- the backward pass for callers that cannot allocate.
 * The pages have no counterpart to this entry point; it is a deployment aid.
 * Some callers cannot pass a workspace: they hold no device allocator of
 * their own, or their device-memory budget is fixed at start-up, or they must
 * not call cudaMalloc where they run the backward because it can block the
 * host or synchronise the device.  This variant takes the same tensors as
 * attn_bwd but keeps its scratch (the LSE and D row statistics) in a fixed
 * 16 MiB device array inside the library, present on every GPU that loads
 * the library until the process exits.  It allocates nothing.
 *   - Computes dQ with the query-tile pass (bf16 results equal attn_bwd with
 *     ATTN_DQ_PASS); fp32 uses the SIMT kernels.
 *   - Size limit: bf16 B*H*n_pad <= 2,097,152 (n_pad = n rounded up to 128),
 *     fp32 B*H*n <= 4,194,304; larger problems return ATTN_ERR_WORKSPACE
 *     before any launch.
 *   - All calls share the array.  Calls whose work overlaps on the GPU (two
 *     streams, or two threads without ordering) race: keep them on one stream
 *     or synchronise in between.  Nothing in the array needs to start at zero.
 *   - The first call on each device looks up the array's address on that
 *     device; make that first call before capturing any stream.  The address
 *     is kept per CUDA context: after cudaDeviceReset, or under another
 *     context made current on the device, the next call looks it up again.
 */
ATTN_API int attn_bwd_noalloc(const void* Q, const void* K, const void* V,
             const void* O, const void* dO, const float* LSE, void* dQ,
             void* dK, void* dV, int B, int H, int n, int d, attn_dtype dtype,
             float scale, int causal, void* stream);

/*
 * Materialise-P comparison path (bf16 only, d in {64,128,256}).  The plainest
 * reading of the small-cache algorithm of "On the fine-grained I/O
 * complexity of attention backward passes" (Methodology step 3: it reads
 * and writes the n x n attention matrices and n x d intermediates
 * explicitly), which is also the standard attention of "Flash Attention:
 * Revolutionizing Transformer Efficiency" ("Standard attention", the score
 * matrix written to and read back from HBM).  Every n x n matrix goes
 * through HBM: forward S (fp32) -> P (bf16) -> O = PV; backward
 * dV = P^T dO, dP = dO V^T (fp32), dS (bf16), dQ = scale dS K,
 * dK = scale dS^T Q.  Results equal attn_fwd/attn_bwd up to rounding.
 * Workspace: attn_mat_workspace_size bytes, 256-byte aligned; the forward
 * leaves P in the workspace and attn_mat_bwd reads it, so pass the same
 * workspace to both without touching it in between.
 */
ATTN_API size_t attn_mat_workspace_size(int B, int H, int n, int d);
ATTN_API int attn_mat_fwd(const void* Q, const void* K, const void* V, void* O,
                 float* LSE, int B, int H, int n, int d, float scale,
                 int causal, void* workspace, size_t workspace_bytes,
                 void* stream);
ATTN_API int attn_mat_bwd(const void* Q, const void* K, const void* V, const void* O,
                 const void* dO, const float* LSE, void* dQ, void* dK,
                 void* dV, int B, int H, int n, int d, float scale,
                 int causal, void* workspace, size_t workspace_bytes,
                 void* stream);

/*
 * attn_gemm_bf16 -- batched tensor-core GEMM used by the materialise-P path,
 * exported for testing the tcgen05/TMA building blocks in isolation:
 *   C[b] = alpha * op(A[b]) * op(B[b]),  b in [0, batch)
 * A[b] is M x K: row-major [M][K] if a_kmajor, else stored as [K][M].
 * B[b] is K x N: stored [N][K] if b_kmajor, else row-major [K][N].
 * C[b] is row-major [M][N], fp32 if c_f32 else bf16.  Batches are packed
 * with strides M*K, K*N, M*N elements.  K must be a multiple of 8 and the
 * contiguous dimension of every operand a multiple of 8 elements.
 */
ATTN_API int attn_gemm_bf16(const void* A, const void* Bm, void* C, int batch, int M,
                   int N, int K, int a_kmajor, int b_kmajor, int c_f32,
                   float alpha, void* stream);

/* Synchronises `stream`, then returns and clears the first device-side
 * error recorded since the last call (ATTN_OK if none). */
ATTN_API int attn_status(void* stream);

/*
 * attn_selftest_wait_timeout -- checks that device-side failure detection
 * reaches the host.  Every barrier wait inside the library's kernels is
 * bounded: when it runs out it records ATTN_ERR_DEVICE_TIMEOUT (and the wait
 * site) in the device status word and the kernel returns instead of hanging.
 * This launches one block whose single wait has no arrival, with the limit
 * timeout_ns (1 us .. 10 s; ATTN_ERR_INVALID_ARG otherwise): after it, the
 * next attn_status(stream) returns ATTN_ERR_DEVICE_TIMEOUT and the context
 * stays usable.  No fault is involved.
 */
ATTN_API int attn_selftest_wait_timeout(unsigned long long timeout_ns, void* stream);

/* Number of kernels the library has enqueued in this process so far
 * (every launch by every entry point, counted on the host when it is
 * issued).  The difference across a region is how many of the library's
 * kernels that region launched. */
ATTN_API unsigned long long attn_launch_count(void);

/* Static description of a status code. */
ATTN_API const char* attn_strerror(int code);

/* Library version string. */
ATTN_API const char* attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H */
