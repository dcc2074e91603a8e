/*
 * w4a16.h -- C ABI of the W4A16 group-128 linear layer for GB300 (sm_103a).
 *
 *     y[B][N] = x[B][K] . dequant(Wq[K][N], S[K/128][N], Z?)
 *
 * with bf16 activations x, 4-bit weight codes q, one bf16 scale s per 128
 * consecutive weights along K, and w = (q - z) * s rounded once to bf16,
 * where z = 8 for the symmetric (GPTQ, "uint4 bias 8") format or a stored
 * 4-bit zero-point per (group, column) for the asymmetric format.
 *
 * Sources, by page title and section:
 *  - "Give Me BF16 or Give Me Death" (summary), section "W4A16-INT
 *    Quantization", paragraphs "Group-wise quantization granularity" (one
 *    16-bit scale per 128 consecutive weights along the input dimension) and
 *    "Inference with W4A16" (weights rebuilt on the fly inside the matrix
 *    multiplication, 16-bit tensor-core products, higher-precision
 *    accumulation).
 *  - "When quantization pays -- and when it does not", section "Counting c
 *    from the kernel, not from intuition" (bias-8 unsigned codes decoded by
 *    the bf16 magic number 128, exact subtraction of 136, then the group
 *    scale), and the opening model of a decode step (memory pipe vs. math pipe).
 *
 * Conventions shared by every call:
 *  - All buffer pointers are DEVICE pointers on the current CUDA device and
 *    must be 16-byte aligned.  The caller owns every buffer; the library never
 *    allocates device memory.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call only enqueues work and returns; it never
 *    synchronises.
 *  - Shapes are validated on the host before anything is enqueued: on any
 *    error nothing is launched and a status is returned.  No C++ exception
 *    crosses this boundary.  Inputs are never padded: K must be a multiple of
 *    128 and N a multiple of 8.
 *  - group_size must be 128 (the only group the format defines here).
 *  - bf16 buffers are passed as void* and hold IEEE bfloat16 bit patterns.
 *
 * Data layouts:
 *  - canonical codes   qweight uint32 [K/8][N]: nibble j (bits 4j..4j+3) of
 *                      word [kk][n] is the code of row k = 8*kk + j, column n.
 *  - canonical zeros   qzeros  uint32 [K/128][N/8]: nibble j of word [g][nn]
 *                      is the zero-point of group g, column 8*nn + j.
 *  - scales            bf16 [K/128][N], row-major.
 *  - x                 bf16 [B][K], row-major (row stride K).
 *  - y                 bf16 [B][N], row-major (row stride N).
 *  - packed blob       opaque, w4a16_packed_bytes() bytes, written by
 *                      w4a16_pack(); its last 16 bytes are a tag (a magic
 *                      word, the layout version W4A16_PACKED_LAYOUT, K, and
 *                      N with the zero-point flag in bit 31) that
 *                      w4a16_packed_check and every GEMM check.
 */
#ifndef W4A16_H_
#define W4A16_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define W4A16_GROUP 128
#define W4A16_PACKED_LAYOUT 4 /* version tag of the packed blob's layout */

typedef enum {
    W4A16_OK = 0,
    W4A16_ERR_NULL = 1,        /* a required pointer is NULL */
    W4A16_ERR_SHAPE = 2,       /* B < 1, K % 128 != 0, N % 8 != 0, or sizes too large */
    W4A16_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned */
    W4A16_ERR_UNSUPPORTED = 4, /* group_size != 128, or an unknown path id */
    W4A16_ERR_WORKSPACE = 5,   /* workspace smaller than w4a16_workspace_bytes() */
    W4A16_ERR_CUDA = 6,        /* a CUDA runtime call or launch failed */
    W4A16_ERR_TIMEOUT = 7,     /* a device-side bounded wait ran out (see
                                  w4a16_device_status) */
    W4A16_ERR_BOUNDS = 8       /* a device-side bounds check failed; only the
                                  debug build (W4A16_DEBUG) checks, reported by
                                  w4a16_device_status */
} w4a16_status;

/* Kernel paths the dispatcher chooses from (w4a16_select_path, forcing). */
typedef enum {
    W4A16_PATH_AUTO = -1,
    W4A16_PATH_SKINNY = 0,  /* small-batch split-K kernel (mma.sync), B <= 16 */
    W4A16_PATH_TCGEN05 = 1  /* tcgen05 tensor-core kernels: the wide-batch kernel
                               above 16 batch rows, the multi-issuer kernel when
                               forced at 16 or fewer (both keep the dequantised
                               weight tile in TMEM) */
} w4a16_path;

/* Bytes of the packed blob for a K x N layer (codes, plus zero-points when
 * has_zeros != 0, plus the 16-byte layout tag): K*N/2 [+ (K/128)*R*4] + 16,
 * where R = N/8 rounded up to a multiple of 4 (each group's row of zero-point
 * words is padded to 16 bytes).  Storage per weight at group 128: 4 bits of
 * code + 16/128 bits of scale = 4.125 bits ("When quantization pays -- and
 * when it does not", section "The three regimes": 0.5156 bytes per weight;
 * "Give Me BF16 or Give Me Death", "W4A16-INT Quantization", paragraph
 * "Group-wise quantization granularity": 0.125 bit of scale overhead), plus
 * 0.03125 bit with zero-points; the tag is a fixed 16 bytes.
 * Returns 0 for invalid shapes. */
size_t w4a16_packed_bytes(int K, int N, int group_size, int has_zeros);

/* Bytes of device workspace w4a16_gemm needs for this shape (0 if none).
 * The workspace holds arrival counters, the small-batch kernel's work
 * scheduler and an fp32 accumulator for split-K sums.  It must be
 * zero-filled once before its first use; every call that completes (device
 * status OK) leaves it all-zero again, so later calls of any shape on the
 * same stream can reuse it.  A call whose bounded wait expired
 * (w4a16_device_status reports W4A16_ERR_TIMEOUT) stops part-way and may
 * leave partial sums and counts in it: the caller must zero-fill the
 * workspace again before reusing it.  Calls that run concurrently must use
 * different workspaces.  (Split-K sums are accumulated in arrival order, so
 * outputs may differ in the last bit between calls; every one is within the
 * error bound.)
 * Returns (size_t)-1 for invalid shapes. */
size_t w4a16_workspace_bytes(int B, int K, int N, int group_size);

/* Offline repack ("Counting c from the kernel": the lop3 magic-number decode
 * takes one nibble from each 16-bit half of a 32-bit word, so the codes of
 * each pair of consecutive k are moved into the two halves of one word).
 *   qweight  device, canonical codes uint32 [K/8][N]            (read)
 *   qzeros   device, canonical zeros uint32 [K/128][N/8], or NULL for the
 *            symmetric format                                   (read)
 *   packed   device, w4a16_packed_bytes(K, N, 128, qzeros != NULL) bytes
 *                                                               (written)
 * Integer-only; the result is a pure permutation of the input nibbles. */
w4a16_status w4a16_pack(const uint32_t *qweight, const uint32_t *qzeros, int K, int N,
                        int group_size, void *packed, void *stream);

/* y = x . dequant(packed, scales) with fp32 accumulation and one final
 * round-to-nearest-even to bf16 ("Inference with W4A16").
 *   x          device bf16 [B][K]                              (read)
 *   packed     device blob from w4a16_pack                     (read)
 *   scales     device bf16 [K/128][N]                          (read)
 *   has_zeros  1 if the blob was packed with zero-points, else 0
 *   y          device bf16 [B][N]                              (written)
 *   workspace  device, >= w4a16_workspace_bytes(B, K, N, 128) bytes,
 *              zero-filled before first use (may be NULL when that size is 0)
 * The kernel path is chosen from (B, K, N) by w4a16_select_path. */
w4a16_status w4a16_gemm(const void *x, const void *packed, const void *scales, int has_zeros,
                        void *y, int B, int K, int N, int group_size,
                        void *workspace, size_t ws_bytes, void *stream);

/* Fused output epilogues (flags, may be combined): the sums are converted
 * once, after the K reduction, so nothing extra goes through HBM.
 *   W4A16_EPI_BIAS      y[b][n] = bf16(acc[b][n] + bias[n])
 *   W4A16_EPI_SILU_MUL  gated MLP: the N columns are interleaved gate / up
 *                       (column 2j = gate j, column 2j + 1 = up j) and
 *                       y[b][j] = bf16(silu(g) * u), silu(g) = g / (1 + e^-g),
 *                       with g and u the (biased) fp32 sums; y is [B][N/2]. */
enum {
    W4A16_EPI_NONE = 0,
    W4A16_EPI_BIAS = 1,
    W4A16_EPI_SILU_MUL = 2
};

/* w4a16_gemm with a fused epilogue (W4A16_EPI_* flags).
 *   bias   device bf16 [N], 16-byte aligned; required with W4A16_EPI_BIAS,
 *          ignored otherwise
 *   y      device bf16 [B][N], or [B][N/2] with W4A16_EPI_SILU_MUL
 * Other arguments, the path choice and the workspace as for w4a16_gemm.
 * Errors: UNSUPPORTED for unknown flags, NULL / ALIGN for the bias, then as
 * w4a16_gemm.  The gated form needs a weight whose gate and up columns were
 * interleaved before quantisation (a column permutation of [W_gate | W_up]). */
w4a16_status w4a16_gemm_fused(const void *x, const void *packed, const void *scales,
                              int has_zeros, const void *bias, int epilogue, void *y, int B,
                              int K, int N, int group_size, void *workspace, size_t ws_bytes,
                              void *stream);

/* As w4a16_gemm, but with the kernel path forced (W4A16_PATH_*; AUTO = same
 * as w4a16_gemm).  For tests and ablations; the result must agree with
 * every other path within the GEMM error bound. */
w4a16_status w4a16_gemm_path(const void *x, const void *packed, const void *scales, int has_zeros,
                             void *y, int B, int K, int N, int group_size,
                             void *workspace, size_t ws_bytes, int path, void *stream);

/* Materialise the dequantised weights W[K][N] (bf16, row-major) from the
 * packed blob with the same device decode routine the GEMM kernels use, so
 * that every weight can be compared bit for bit with RNE_bf16((q - z) * s).
 * "When quantization pays -- and when it does not", section "Counting c from
 * the kernel, not from intuition": the magic-number decode gives the exact
 * integer (q - 8) before one bf16 multiply by the group scale; "Give Me BF16
 * or Give Me Death", "W4A16-INT Quantization": w = s * q per group of 128.
 *   w  device bf16 [K][N] (written) */
w4a16_status w4a16_dequant_ref(const void *packed, const void *scales, int has_zeros, void *w,
                               int K, int N, int group_size, void *stream);

/* fp16-activation variant ("Give Me BF16 or Give Me Death", "W4A16-INT
 * Quantization", paragraph "Inference with W4A16": fp16 weights, scales and
 * tensor-core products).  Same packed blob (w4a16_pack), same layouts,
 * shapes, workspace size (w4a16_workspace_bytes), path choice, errors and
 * device status as w4a16_gemm / w4a16_gemm_path, but
 *   x       device fp16 (IEEE binary16) [B][K]
 *   scales  device fp16 [K/128][N]
 *   y       device fp16 [B][N]
 * The weights are decoded with the fp16 magic number (1024.0, 0x6400: a code
 * OR-ed into its 10 fraction bits gives 1024 + q exactly) to
 * w = RNE_f16((q - z) * s), multiplied with fp16 tensor-core operands and
 * accumulated in fp32; y = RNE_f16 of the sum.  (The small-batch path scales
 * the fp32 sum of each 128-row group instead of each weight, which changes
 * the rounding of w, not the bound: |y - y_exact| stays within
 * 2e-3 * sum|x*w| + 2^-24 * (1 + sum|x|).)  No fused epilogue or grouped
 * form. */
w4a16_status w4a16_gemm_f16(const void *x, const void *packed, const void *scales, int has_zeros,
                            void *y, int B, int K, int N, int group_size, void *workspace,
                            size_t ws_bytes, void *stream);
w4a16_status w4a16_gemm_f16_path(const void *x, const void *packed, const void *scales,
                                 int has_zeros, void *y, int B, int K, int N, int group_size,
                                 void *workspace, size_t ws_bytes, int path, void *stream);

/* w4a16_dequant_ref for fp16 scales: W[K][N] as fp16, w = RNE_f16((q - z) *
 * s), through the fp16 GEMM kernels' decode routine.
 *   scales  device fp16 [K/128][N];  w  device fp16 [K][N] (written) */
w4a16_status w4a16_dequant_ref_f16(const void *packed, const void *scales, int has_zeros, void *w,
                                   int K, int N, int group_size, void *stream);

/* Grouped GEMM for mixture-of-experts layers: one launch computes, for every
 * expert e, y[r] = x[r] . dequant(W_e) for the rows r of x that belong to e.
 * Rows are grouped by expert: offsets (device int32 [E+1], non-decreasing,
 * offsets[0] = 0, offsets[E] = T) gives expert e the rows offsets[e] ..
 * offsets[e+1]-1 of x [T][K] and y [T][N]; an expert may have no rows.  The
 * offsets are read on the device, after the previous kernel on the stream has
 * finished, so the routing may come from that kernel.  A malformed table
 * cannot reach outside x and y: entries are clamped to [0, T] and a
 * decreasing entry is raised to the largest one before it (the experts' row
 * ranges stay disjoint); rows not covered by any expert are left unwritten.
 * "When quantization pays -- and when it does not", section "The three
 * regimes", mixture-of-experts paragraphs: a routed expert's GEMM sees only
 * the rows sent to it, B*k/E of them on average.
 *   packed     E packed blobs back to back, each w4a16_packed_bytes(K, N,
 *              128, has_zeros) bytes (from w4a16_pack)
 *   scales     bf16 [E][K/128][N]
 *   max_rows   an upper bound on one expert's rows; with the mean T/E it
 *              picks the batch tile (8, 16 or 32 rows: 8 when max_rows <= 8
 *              or T/E <= 5, 16 when max_rows <= 16 or T/E <= 10); an expert
 *              with more rows than the tile is computed correctly in more
 *              tiles (reading its weights once per tile)
 *   workspace  w4a16_grouped_workspace_bytes(T, E, max_rows, K, N, 128) bytes,
 *              same contract as w4a16_gemm's (zero-filled once, left zero)
 * Errors: UNSUPPORTED (group_size), SHAPE (K, N, T < 1, E outside 1..256,
 * max_rows < 1), NULL, ALIGN (16 bytes; offsets 4), WORKSPACE, CUDA. */
size_t w4a16_grouped_workspace_bytes(int T, int E, int max_rows, int K, int N, int group_size);
w4a16_status w4a16_gemm_grouped(const void *x, const int *offsets, int E, int T,
                                const void *packed, const void *scales, int has_zeros, void *y,
                                int max_rows, int K, int N, int group_size, void *workspace,
                                size_t ws_bytes, void *stream);

/* Offline quantizer for the symmetric format: bf16 weights -> canonical
 * codes and bf16 group scales, ready for w4a16_pack.  "Give Me BF16 or Give
 * Me Death", section "W4A16-INT Quantization", paragraph "Weight quantization
 * algorithm: GPTQ with MSE-optimal clipping", without the GPTQ update (which
 * needs calibration data): for each group of 128 consecutive weights along K
 * of each column, the clipping ratio alpha on the grid 1 - i/32 (i = 0..23)
 * whose round-to-nearest quantisation has the smallest sum of squared errors;
 * scale = RNE_bf16(alpha * max|x| / 7), code = clamp(rint(x / scale), -7, 7)
 * + 8 (codes 1..15; 8 with scale 0 for an all-zero group).  The error is
 * measured on RNE_bf16((code - 8) * scale), the weights the GEMM uses.  The
 * result is deterministic (binary32 division and rounding, binary64 error
 * sums in k order; ties keep the larger alpha).
 *   w        device bf16 [K][N], row-major (read)
 *   qweight  device uint32 [K/8][N], canonical layout (written)
 *   scales   device bf16 [K/128][N] (written)
 * Errors: UNSUPPORTED (group_size != 128), SHAPE (K % 128, N % 8), NULL,
 * ALIGN (16 bytes), CUDA (launch).  Asynchronous on stream. */
w4a16_status w4a16_quantize_rtn(const void *w, int K, int N, int group_size, uint32_t *qweight,
                                void *scales, void *stream);

/* Path w4a16_gemm would take for this shape on the current device
 * (W4A16_PATH_*), or -1 for invalid shapes.  The choice is made per shape
 * because the layer changes regime with the batch: "When quantization pays
 * -- and when it does not", sections "Model one decode step" and "The three
 * regimes" (weight-stream-bound at small B, tensor-core-bound past the ridge
 * batch), and the M-dependent kernel selection that page describes (a
 * small-batch kernel below a row threshold, the tiled tensor-core kernel
 * above it).  For tests and ablations the environment variable
 * W4A16_FORCE_PATH=skinny|tcgen05 (read once per process) overrides the
 * automatic choice of w4a16_gemm, w4a16_gemm_fused, w4a16_gemm_f16 and
 * w4a16_workspace_bytes alike; a forced tensor-core path is ignored on a
 * device without it. */
int w4a16_select_path(int B, int K, int N);

/* Name of the kernel w4a16_gemm launches for this shape on the current
 * device by automatic selection: "skinny_kernel" (small-batch split-K, 16 or
 * fewer rows) or "wide_kernel" (tensor cores, above 16 rows).  ("tc_kernel",
 * tensor cores with several issuing threads, runs only when
 * w4a16_gemm_path forces the tensor-core path at 16 or fewer rows.)  Both
 * tensor-core kernels keep the dequantised weight tile in tensor memory.
 * "invalid" for invalid shapes.  For logs and for
 * reporting which operator ran ("Quantization quality and performance":
 * report the operator actually used).  Never NULL; static storage. */
const char *w4a16_kernel_name(int B, int K, int N);

/* The launch plan w4a16_gemm uses for a shape, for logs and tests ("Quantization
 * quality and performance": report the operator actually used; the path and
 * its split change with the batch: "When quantization pays -- and when it
 * does not", "The three regimes").  num_sms = 0 plans for the current device
 * (its SM count and path availability); num_sms > 0 plans, without touching a
 * device, for a GB300-class device with that many SMs (the tensor-core path
 * assumed available).  Fields not used by the chosen kernel are 0. */
typedef struct {
    int kernel;          /* 0 skinny_kernel, 1 tc_kernel, 2 wide_kernel */
    int batch_rows;      /* batch rows per tile (small-batch kernel: 8, 16 or 32;
                            tensor-core kernels: the MMA's N) */
    int batch_tiles;     /* tiles along B */
    int col_tiles;       /* 128-column weight tiles */
    int k_splits;        /* K splits (1: no workspace accumulator) */
    int groups_per_split;/* 128-row groups of K per split (the last may be shorter) */
    int grid;            /* CTAs launched */
    int ctas_per_sm;     /* resident CTAs per SM the kernel is built for */
    int issuers;         /* MMA-issuing threads (wide kernel) */
    int acc_buffers;     /* accumulator sets in tensor memory (wide kernel) */
    int tile_slots;      /* dequantised weight tiles in tensor memory (wide kernel) */
    int x_slots;         /* activation blocks in shared memory (wide kernel) */
    int code_slots;      /* packed-code stages in shared memory */
    int block_rows;      /* K rows per pipeline block */
    int tmem_cols;       /* tensor-memory columns in use, of 512 (wide kernel) */
    size_t smem_bytes;   /* dynamic shared memory per CTA (small-batch and wide kernels) */
    size_t workspace_bytes; /* workspace this plan needs (<= w4a16_workspace_bytes) */
} w4a16_plan_info;

/* Fills *out.  W4A16_ERR_NULL for out == NULL; W4A16_ERR_SHAPE / _UNSUPPORTED as
 * w4a16_gemm validates (B, K, N, group_size); W4A16_ERR_CUDA if num_sms = 0 and
 * the device cannot be queried. */
w4a16_status w4a16_describe_plan(int B, int K, int N, int group_size, int num_sms,
                                 w4a16_plan_info *out);

/* Device-side status word of the GEMM kernels: W4A16_OK when every bounded
 * wait completed and every packed blob's tag matched its call, else
 * W4A16_ERR_TIMEOUT (a bounded wait ran out), W4A16_ERR_UNSUPPORTED (a GEMM
 * was given a blob whose tag does not describe it: another layout version,
 * shape or zero-point flag -- its output is then meaningless) or, in the
 * debug build only, W4A16_ERR_BOUNDS (an index check failed; the access was
 * skipped).  Synchronises
 * the current device; clears the word when `clear` != 0.  Returns
 * W4A16_ERR_CUDA if the query itself fails. */
w4a16_status w4a16_device_status(int clear);

/* w4a16_gemm for callers that cannot allocate device memory (the pages have
 * no counterpart; this is a deployment convenience).  Same arguments,
 * layouts and result as w4a16_gemm, but without a workspace argument: the
 * split-K scratch is a 4 MiB device array compiled into the library
 * (every GPU that loads the library holds it until the process exits).
 *  - Calls no cudaMalloc, cudaFree or allocating library routine.
 *  - The first call on a device looks the array's device address up for
 *    that device; make that first call before any stream capture.
 *  - Every call shares the one array and first clears (one memset on
 *    `stream`) every byte of it that the shape uses -- arrival counters,
 *    scheduler words and the fp32 split-K accumulator -- so a call whose
 *    bounded wait expired cannot leave partial sums for the next call; calls
 *    that may overlap on the GPU (different streams, or different host
 *    threads) race on it and must be serialised by the caller.
 *  - Returns W4A16_ERR_WORKSPACE when the shape needs more scratch than the
 *    array holds (w4a16_workspace_bytes() tells how much it needs). */
w4a16_status w4a16_gemm_static_scratch(const void *x, const void *packed, const void *scales,
                                       int has_zeros, void *y, int B, int K, int N,
                                       int group_size, void *stream);

/* Test hook for the bounded waits of the tensor-core kernel (no counterpart
 * on the pages).  Launches the tensor-core kernel on a valid problem (same
 * arguments and rules as w4a16_gemm_path with W4A16_PATH_TCGEN05), but its
 * MMA thread first waits on a barrier that nothing ever arrives at, limited
 * to wait_ms milliseconds (1..10000).  The wait expires, the kernel records
 * W4A16_ERR_TIMEOUT in the device status word (read it with
 * w4a16_device_status), lets its in-flight copies land, frees its tensor
 * memory and returns without writing y.  The CUDA context stays usable.
 * Returns W4A16_ERR_UNSUPPORTED where the tensor-core kernel is unavailable. */
w4a16_status w4a16_debug_forced_timeout(const void *x, const void *packed, const void *scales,
                                        int has_zeros, void *y, int B, int K, int N,
                                        int group_size, void *workspace, size_t ws_bytes,
                                        int wait_ms, void *stream);

/* 1 for the debug build of the library (compiled with W4A16_DEBUG), else 0.
 * In the debug build every global load, copy and store of the GEMM kernels is
 * preceded by a check of its index against the extent of the buffer it
 * touches; a failed check skips that access (so no wait is left hanging and
 * no memory outside the buffer is touched) and records W4A16_ERR_BOUNDS in
 * the device status word instead of trapping.  Same C ABI, same results. */
int w4a16_debug_build(void);

/* Test hook of the debug build (no counterpart on the pages): later GEMM
 * launches on this process tell their kernels that the packed codes end
 * `bytes` bytes earlier than they do (0 restores the true extent), so the
 * kernels' own checks skip the last copies and report W4A16_ERR_BOUNDS; the
 * memory touched stays inside the real blob and every wait still ends, but
 * the outputs of those launches are meaningless.  Returns
 * W4A16_ERR_UNSUPPORTED in the release build. */
w4a16_status w4a16_debug_shrink_code_bound(size_t bytes);

/* Checks a packed blob's tag against the layout version this library reads
 * and the call's shape: W4A16_OK, W4A16_ERR_UNSUPPORTED when the blob was
 * written for another layout version (or is not a packed blob), or
 * W4A16_ERR_SHAPE when K, N or the zero-point flag differ; NULL / ALIGN /
 * SHAPE / UNSUPPORTED for invalid arguments as everywhere.  For validating
 * stored weights when they are loaded: it copies the 16-byte tag to the host
 * and synchronises `stream`.  (The GEMMs check the tag on the device on every
 * call, see w4a16_device_status.) */
w4a16_status w4a16_packed_check(const void *packed, int K, int N, int group_size, int has_zeros,
                                void *stream);

/* Static description of a status code; never NULL. */
const char *w4a16_status_string(w4a16_status status);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H_ */
