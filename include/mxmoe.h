/*
 * mxmoe.h -- C ABI of libmxmoe.so, the GB300 (sm_103a) MXFP8 Mixture-of-Experts
 * training hot path: MXFP8 quantize, router, token permute/unpermute, block-scaled
 * grouped GEMM (forward, dgrad, wgrad), fused SwiGLU, and the MoE layer
 * forward/backward built from them.
 *
 * Sources (the method):
 *   [A] "1.5x faster MoE training on Blackwell with MXFP8 kernels built from
 *       scratch" (engineering.fyi), Overview; Key Questions Answered
 *       (microscaling; tcgen05.mma block-scaled MMA with TMEM accumulators);
 *       Common Pitfalls (quantization overhead).
 *   [B] pytorch/ao PR "[mxfp8 moe training] bench and profile mxfp8 a2a fwd
 *       and bwd separately", Stacked PRs (e8m0 -> fp32 scale decode) and
 *       Next steps (stay in MXFP8 through an "mxfp8 token shuffle kernel"
 *       and a scaled grouped GEMM that accepts pre-quantized operands).
 *   [C] OCP Microscaling Formats (MX) v1.0, section 6.3: blocks of 32
 *       elements, E4M3 elements, E8M0 shared scale 2^(floor(log2 amax) - 8).
 *
 * Conventions (every entry point):
 *   - Returns mx_status.  Host-detectable errors (null or misaligned pointer,
 *     bad sizes, wrong device) return before anything is enqueued.
 *   - Every pointer argument, unless documented otherwise, is DEVICE memory
 *     owned by the caller; the library never allocates or frees memory and
 *     keeps no state between calls.  Outputs must not alias inputs.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and runs asynchronously; nothing synchronizes the host, and
 *     group sizes stay on the device, so a sequence of calls can be captured
 *     into a CUDA graph and replayed.  Kernels are launched with programmatic
 *     dependent launch: each one waits for the previous work of the stream
 *     to complete before it touches memory, so stream order is kept, while
 *     its launch overlaps the end of that work.  Setting the environment
 *     variable MXMOE_PDL=0 before the first call launches them plainly.
 *   - Errors found on the device (expert id out of range, bad group offsets,
 *     a pipeline wait that timed out) are written to the optional
 *     `dev_status` word (device int32, nullable) as an mx_status value; the
 *     kernel skips the offending work.  The word is never cleared by the
 *     library: the caller zeroes it.
 *   - Matrices are row-major.  bf16 is IEEE bfloat16 (uint16 storage); fp8 is
 *     OCP E4M3FN (uint8); scales are E8M0 bytes (2^(b-127), 0xFF = NaN).
 *   - Sizes are int64_t; ids, counts and offsets are int32.
 *   - Device pointers must be 16-byte aligned (MX_ERR_ALIGNMENT otherwise),
 *     except scale arrays, which may start at any byte unless an entry point
 *     states otherwise.
 *   - Requires an sm_103 device (GB300); MX_ERR_UNSUPPORTED_DEVICE otherwise.
 */
#ifndef MXMOE_H
#define MXMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t mx_status;
typedef struct CUstream_st *mx_stream; /* same type as cudaStream_t */

#define MX_OK 0
#define MX_ERR_INVALID_ARG 1        /* null pointer, unknown enum, negative size */
#define MX_ERR_SHAPE 2              /* a dimension breaks a multiple-of-32/128/256 rule */
#define MX_ERR_ALIGNMENT 3          /* a pointer breaks its alignment rule (16 bytes unless stated) */
#define MX_ERR_UNSUPPORTED_DEVICE 4 /* current device is not sm_103 */
#define MX_ERR_CUDA 5               /* a CUDA runtime/driver call failed */
#define MX_ERR_DEVICE 6             /* device-detected: id out of range, bad offsets */
#define MX_ERR_TIMEOUT 7            /* device-detected: a bounded pipeline wait expired */
#define MX_ERR_WORKSPACE 8          /* workspace smaller than the size query returned */
#define MX_ERR_SCRATCH_LIMIT 9      /* problem needs more than an allocation-free entry point's fixed scratch */

/* quantize modes */
#define MX_MODE_ROW 1   /* blocks of 32 along each row                         */
#define MX_MODE_COL 2   /* blocks of 32 down each column, output transposed    */
#define MX_MODE_BOTH 3  /* both, from one read of the input                    */

/* scale layouts */
#define MX_SCALE_PLAIN 0    /* row-major [rows, cols/32]                             */
#define MX_SCALE_SWIZZLED 1 /* tiles of 128 rows x 4 scale columns (512 B), tile-row-
                               major; inside a tile byte (r%32)*16 + ((r%128)/32)*4 + c%4.
                               Rows padded to 128, scale columns to 4, padding 0x00.
                               This is the layout the block-scaled tensor-core MMA reads. */

/* element formats of an MX block (the scale rule takes the format's largest
 * power of two: 2^8 for E4M3, 2^15 for E5M2).  E4M3 is the MXFP8 of the
 * pages; E5M2 is the gradient option (two exponent bits more range, one
 * mantissa bit less), a variant the pages do not name. */
#define MX_ELEM_E4M3 0 /* OCP E4M3FN: max +-448, NaN 0x7F, no Inf          */
#define MX_ELEM_E5M2 1 /* OCP E5M2: max +-57344, Inf 0x7C, NaN 0x7F        */

/* grouped GEMM operations */
#define MX_GEMM_FWD 0   /* C[rows of e] = A[rows of e] . B[e]^T, rows grouped by offsets */
#define MX_GEMM_DGRAD 1 /* same contraction as FWD (operands differ, see mx_grouped_gemm) */
#define MX_GEMM_WGRAD 2 /* C[e] = X[:, tokens of e] . Y[:, tokens of e]^T                  */

/* output element types */
#define MX_OUT_BF16 0
#define MX_OUT_F32 1

/* permute kinds */
#define MX_PERMUTE_FP8 0        /* MXFP8 rows (E4M3 data + plain [T, H/32] scales) in, MXFP8 out */
#define MX_PERMUTE_BF16 1       /* bf16 rows in, bf16 rows out                                     */
#define MX_PERMUTE_BF16_QUANT 2 /* bf16 rows in, quantized (ROW mode) while moved, MXFP8 out        */

/* ------------------------------------------------------------------------ */
/* Library                                                                   */
/* ------------------------------------------------------------------------ */

/* Human-readable name of a status code (static string, never NULL). */
const char *mx_status_string(mx_status s);

/* ABI version of this header (bumped on any signature change). */
int32_t mx_abi_version(void);

/* MX_OK if the current CUDA device is an sm_103 part this library runs on. */
mx_status mx_check_device(void);

/*
 * Self-test of the device-side failure path (no counterpart on the pages:
 * it checks this library's own error handling).  Every pipeline wait in the
 * kernels is bounded; when a wait expires, the kernel writes MX_ERR_TIMEOUT to
 * dev_status, leaves its loops and exits with nothing in flight, so the CUDA
 * context stays usable.  This call runs one warp that waits, through the same
 * bounded wait, on an mbarrier that nothing ever arrives on, for timeout_ns
 * nanoseconds (at most 100 ms), then records MX_ERR_TIMEOUT in dev_status
 * (device int32, required).  Enqueued on `stream`; returns host errors only.
 */
mx_status mx_selftest_wait_timeout(int64_t timeout_ns, int32_t *dev_status, mx_stream stream);

/*
 * Self-test of the SwiGLU arithmetic (no counterpart on the pages: the pages
 * fix no precision for the SwiGLU step; this exposes the fp32 sigmoid the
 * fused SwiGLU forward and backward kernels use, so that its error can be
 * measured against an exact evaluation).  For each of the n bf16 values a[i]
 * (device, uint16 storage) writes three fp32 values to out[3i .. 3i+2]
 * (device):
 *   s = sigmoid(a) * 2^k,  1 - sigmoid(a),  2^-k,
 * with k = 64 for a < -64 and 0 otherwise (the kernels carry the 2^64 factor
 * until their last product, so that sigmoid(a) never leaves the fp32 normal
 * range; s * 2^-k is sigmoid(a)).  n >= 0; a and out may be NULL when n = 0.
 */
mx_status mx_selftest_sigmoid(const void *a, int64_t n, float *out, mx_stream stream);

/* Bytes of a scale array for `rows` x `cols` elements (cols % 32 == 0) in the
 * given layout: rows*cols/32 (PLAIN) or the padded tile size (SWIZZLED). */
int64_t mx_scale_bytes(int64_t rows, int64_t cols, int32_t layout);

/* ------------------------------------------------------------------------ */
/* Q: MXFP8 quantize  ([C] section 6.3; [A] Key Questions Answered on       */
/* microscaling; [B] Stacked PRs, quant kernels)                             */
/* ------------------------------------------------------------------------ */
/*
 * x: bf16 [batch, rows, cols].  For every 32-element block: amax over the
 * block; scale exponent e = floor(log2 amax) - 8 (amax = 0 -> -127), clamped to
 * [-127, 127], scale byte e + 127; each element becomes the E4M3 round-to-
 * nearest-even of x * 2^-e, saturated to +-448.  A block holding NaN or Inf
 * gets scale 0xFF and elements 0x7F.
 * elem = MX_ELEM_E5M2 instead: e = floor(log2 amax) - 15 and E5M2 elements
 * saturated to +-57344 (same clamp, NaN rule and layouts).
 *   ROW: q_row [batch, rows, cols], s_row [batch] x scale array(rows, cols).
 *        Needs cols % 32 == 0.
 *   COL: blocks of 32 consecutive rows of one column; stored transposed:
 *        q_col [batch, cols, rows], s_col [batch] x scale array(cols, rows).
 *        Needs rows % 32 == 0.
 *   BOTH: both outputs from one read of x.
 * Unused outputs may be NULL.  Sizes: rows, cols > 0 multiples of 32 for the
 * requested modes, batch >= 1.  For MX_SCALE_SWIZZLED each batch entry is one
 * padded scale array (mx_scale_bytes).
 */
mx_status mx_quantize(const void *x, int64_t batch, int64_t rows, int64_t cols,
                      int32_t mode, int32_t scale_layout, int32_t elem, uint8_t *q_row,
                      uint8_t *s_row, uint8_t *q_col, uint8_t *s_col,
                      mx_stream stream);

/* ------------------------------------------------------------------------ */
/* MXFP8 dequantize  ([B] Stacked PRs: the mxfp8 dequantization kernel and   */
/* the e8m0 -> fp32 scale decode; [C] section 6.3)                           */
/* ------------------------------------------------------------------------ */
/*
 * q: E4M3 [batch, rows, cols] with scales s in `scale_layout` (per batch
 * entry one scale array(rows, cols), as mx_quantize writes its ROW output; a
 * COL output dequantizes the same way into the transposed matrix).  Every
 * element becomes E4M3(q) * 2^(s - 127), the E8M0 decode of its block's
 * scale byte:
 *   MX_OUT_F32:  out fp32, exact (fp32 subnormals kept; overflow to +-Inf);
 *   MX_OUT_BF16: out bf16, that exact value rounded to nearest even once.
 * Scale byte 0xFF and the E4M3 NaN codes (0x7F, 0xFF) give NaN.
 * elem = MX_ELEM_E5M2: q holds E5M2 codes (their Inf and NaN codes decode as
 * such).
 * out [batch, rows, cols].  cols % 32 == 0 (cols % 128 == 0 is not needed:
 * the swizzled array's padding is not read); q and out 16-byte aligned.
 */
mx_status mx_dequantize(const uint8_t *q, const uint8_t *s, int64_t batch, int64_t rows,
                        int64_t cols, int32_t scale_layout, int32_t elem, int32_t out_dtype,
                        void *out, mx_stream stream);

/* ------------------------------------------------------------------------ */
/* Row-max-scaled FP8, for comparison with MX block scaling                  */
/* (NVIDIA/TransformerEngine issue "FP8 significantly slow down when scaling */
/* up to 1000+ GPUs": compute the row max, divide by it before the cast to   */
/* FP8, multiply it back after the GEMM)                                     */
/* ------------------------------------------------------------------------ */
/*
 * x: bf16 [rows, cols].  Per row: amax = max |x| over the row; the scale
 * s = amax / 448 (one IEEE fp32 division: the row max lands on E4M3's
 * largest finite value); each element becomes q = E4M3(x / s) (IEEE fp32
 * division, round to nearest even, saturating at +-448).  x is decoded as
 * E4M3(q) * s.  A zero row gets s = 1 (its elements encode as signed zeros);
 * a row holding NaN or Inf gets s = NaN and every byte 0x7F.
 * q: E4M3 [rows, cols]; row_scale: fp32 [rows].
 * rows >= 0 (0: nothing to do; pointers may be NULL), cols % 16 == 0,
 * cols <= 102400; x and q 16-byte aligned, row_scale 4-byte aligned.
 */
mx_status fp8_quantize_rowmax(const void *x, int64_t rows, int64_t cols, uint8_t *q,
                              float *row_scale, mx_stream stream);

/* ------------------------------------------------------------------------ */
/* R: router (helper; the pages name no router -- top-k with softmax gate)   */
/* ------------------------------------------------------------------------ */
/*
 * logits fp32 [T, E] -> ids int32 [T, k] (the k largest logits, ties to the
 * lower expert id, in decreasing order) and gate fp32 [T, k] = softmax over
 * all E logits evaluated at each chosen id.  1 <= k <= E <= 256.
 */
mx_status moe_route(const float *logits, int64_t T, int32_t E, int32_t k,
                    int32_t *ids, float *gate, mx_stream stream);

/* ------------------------------------------------------------------------ */
/* P1: expert grouping map ([B] Next steps: token shuffle)                   */
/* ------------------------------------------------------------------------ */
/*
 * ids int32 [T, k] -> counts int32 [E] (routed rows per expert),
 * offsets int32 [E+1] (exclusive prefix of counts rounded up to 128: group e
 * occupies rows offsets[e] .. offsets[e+1]-1), dst int32 [T*k] (row of routed
 * pair (t, j); order inside a group follows t*k + j), src int32 [rows_cap]
 * (t*k + j for a routed row, -1 for a pad row or a row past offsets[E]).
 * rows_cap >= moe_rows_cap(T, k, E).  `workspace` is device scratch of
 * moe_permute_map_workspace_size(T, k, E) bytes.  An id outside [0, E) sets
 * MX_ERR_DEVICE in dev_status and that pair gets dst = -1.
 */
int64_t moe_rows_cap(int64_t T, int32_t k, int32_t E);
int64_t moe_permute_map_workspace_size(int64_t T, int32_t k, int32_t E);
mx_status moe_permute_map(const int32_t *ids, int64_t T, int32_t k, int32_t E,
                          int64_t rows_cap, int32_t *counts, int32_t *offsets,
                          int32_t *dst, int32_t *src, void *workspace,
                          int64_t workspace_bytes, int32_t *dev_status,
                          mx_stream stream);

/*
 * Allocation-free variant of moe_permute_map (no counterpart on the pages: it
 * is a packaging choice of this library).  Same arguments and results as
 * moe_permute_map, minus the workspace: it is for callers that cannot hand
 * the library any scratch buffer -- code that only owns the input and output
 * buffers it was given (a plugin or callback inside another framework whose
 * device allocator it may not call, or a runtime with a fixed memory budget
 * decided up front).  Its scratch is a fixed array in the library's own
 * device memory, MOE_NOALLOC_SCRATCH_BYTES bytes, which every GPU that loads
 * the library keeps until the process exits:
 *   - problems whose moe_permute_map_workspace_size(T, k, E) exceeds that
 *     size are rejected with MX_ERR_SCRATCH_LIMIT before anything runs
 *     (2 * ceil(T*k / 1024) * E * 4 bytes: e.g. E = 16 allows T*k up to 2M);
 *   - the first call on each device looks the array's address up (a runtime
 *     call with that device current), so make that first call before any
 *     stream capture;
 *   - all calls on a device share the one array: calls whose work overlaps on
 *     the GPU (different streams, no ordering between them) race and corrupt
 *     each other's results; order them on one stream or with events;
 *   - every call fully rewrites the scratch it reads, so nothing in it has to
 *     start at zero; the library itself never allocates or frees memory here.
 */
#define MOE_NOALLOC_SCRATCH_BYTES (256 * 1024)
mx_status moe_permute_map_noalloc(const int32_t *ids, int64_t T, int32_t k,
                                  int32_t E, int64_t rows_cap, int32_t *counts,
                                  int32_t *offsets, int32_t *dst, int32_t *src,
                                  int32_t *dev_status, mx_stream stream);

/* ------------------------------------------------------------------------ */
/* P2: token permute ([B] Next steps: an MXFP8 token shuffle)               */
/* ------------------------------------------------------------------------ */
/*
 * Moves token rows into their expert groups: out row dst[t*k+j] = row t of x,
 * for every j; pad rows (src = -1) of out become 0 (data 0x00 and scale 0x00,
 * which is also the MXFP8 encoding of a zero row).  Each source row is read
 * once and written k times.
 *   MX_PERMUTE_FP8:        x = fp8 [T, H], x_scales = plain [T, H/32];
 *                          out = fp8 [rows_cap, H], out_scales in
 *                          `scale_layout` for (rows_cap, H).
 *   MX_PERMUTE_BF16:       x = bf16 [T, H] -> out bf16 [rows_cap, H];
 *                          x_scales and out_scales unused (NULL).
 *   MX_PERMUTE_BF16_QUANT: x = bf16 [T, H], quantized (ROW mode, as
 *                          mx_quantize) while moved -> out fp8 + out_scales.
 * H % 32 == 0 (fp8 outputs: H % 128 == 0 when swizzled).  dst, src from
 * moe_permute_map.
 */
mx_status moe_permute(int32_t kind, const void *x, const uint8_t *x_scales,
                      int64_t T, int64_t H, int32_t k, const int32_t *dst,
                      const int32_t *src, int64_t rows_cap, void *out,
                      uint8_t *out_scales, int32_t scale_layout,
                      mx_stream stream);

/* ------------------------------------------------------------------------ */
/* U: unpermute / combine                                                    */
/* ------------------------------------------------------------------------ */
/*
 * out[t] = bf16( sum_j gate[t,j] * y[dst[t*k+j]] ), products and sums in fp32
 * with j increasing from the j = 0 product, one round-to-nearest-even to bf16.
 * y bf16 [rows, H], gate fp32 [T, k] (NULL = all ones), out bf16 [T, H].
 * H % 8 == 0.
 */
mx_status moe_unpermute(const void *y, const int32_t *dst, const float *gate,
                        int64_t T, int64_t H, int32_t k, void *out,
                        mx_stream stream);

/* ------------------------------------------------------------------------ */
/* G: block-scaled grouped GEMM ([A] Key Questions Answered: tcgen05.mma     */
/* block-scaled MMA with TMEM accumulation; [B] Next steps: a scaled grouped */
/* GEMM taking pre-quantized operands and their scales)                      */
/* ------------------------------------------------------------------------ */
/*
 * All operands are MXFP8 with blocks of 32 along the contraction dimension
 * and scales in MX_SCALE_SWIZZLED layout; the scales are applied inside the
 * tensor-core MMA and products accumulate in fp32.  `offsets` int32 [E+1]
 * (device, multiples of 128, non-decreasing) delimits the expert groups.
 *
 * MX_GEMM_FWD / MX_GEMM_DGRAD (groups over rows):
 *   A  fp8 [M_cap, K], sA scales of (M_cap, K)
 *   B  fp8 [E, N, K],  sB scales of (E*N, K)
 *   C[r, :] = deq(A[r, :]) . deq(B[e])^T for offsets[e] <= r < offsets[e+1];
 *   C [M_cap, N] (rows >= offsets[E] are not written).
 *   FWD: A = activations quantized along K, B = weights quantized along K.
 *   DGRAD: A = output gradient quantized along N_fwd, B = weights quantized
 *   along N_fwd (the same call with the roles renamed).
 * MX_GEMM_WGRAD (groups over the contraction = tokens):
 *   A  fp8 [N, M_cap] (= X^T, quantized along tokens), sA scales of (N, M_cap)
 *   B  fp8 [K, M_cap] (= Y^T, quantized along tokens), sB scales of (K, M_cap)
 *   C[e] = sum over tokens r of group e of deq(A[:, r]) deq(B[:, r])^T,
 *   C [E, N, K]; an empty group writes zeros.
 * Sizes: M_cap % 128 == 0, N % 256 == 0, K % 128 == 0, 1 <= E <= 1024.
 * c_dtype: MX_OUT_BF16 (round-to-nearest-even) or MX_OUT_F32.
 * elem_a, elem_b: element formats of A and B (MX_ELEM_E4M3 or MX_ELEM_E5M2,
 * independently: the layer's E5M2 gradient option multiplies E5M2 gradients
 * by E4M3 weights or activations).
 * Alignment: A, B, sA, sB and C 16-byte aligned (the operands and their
 * scales are read by TMA).
 */
mx_status mx_grouped_gemm(int32_t op, const uint8_t *A, const uint8_t *sA,
                          const uint8_t *B, const uint8_t *sB,
                          const int32_t *offsets, int32_t E, int64_t M_cap,
                          int64_t N, int64_t K, void *C, int32_t c_dtype,
                          int32_t elem_a, int32_t elem_b, int32_t *dev_status,
                          mx_stream stream);

/*
 * Deterministic split-K weight gradient (a variant of MX_GEMM_WGRAD for
 * skewed or few output tiles): the same C[e] as mx_grouped_gemm(WGRAD), with
 * each group's tokens cut into `splits` 128-aligned chunks that separate
 * CTA pairs contract, chunk s of group e covering its 128-token blocks
 * [floor(n_e s / splits), floor(n_e (s+1) / splits)).  The partial products
 * (fp32, in `ws`) are summed in the order s = 0, 1, ..., splits-1, so the
 * result does not depend on scheduling; it differs from the unsplit call
 * only by fp32 rounding of the partial sums (splits = 1: bit-identical).
 * Operands as MX_GEMM_WGRAD (element formats elem_a, elem_b as in
 * mx_grouped_gemm); C fp32 [E, N, K].  1 <= splits <= 16,
 * E * splits <= 1024, N % 256 == 0, K % 256 == 0, M_cap % 128 == 0.
 * ws: device scratch of mx_wgrad_splitk_workspace_size(E, N, K, splits)
 * bytes, 16-byte aligned (MX_ERR_WORKSPACE if smaller).
 */
int64_t mx_wgrad_splitk_workspace_size(int32_t E, int64_t N, int64_t K, int32_t splits);
mx_status mx_grouped_gemm_wgrad_splitk(const uint8_t *A, const uint8_t *sA,
                                       const uint8_t *B, const uint8_t *sB,
                                       const int32_t *offsets, int32_t E, int64_t M_cap,
                                       int64_t N, int64_t K, int32_t splits, int32_t elem_a,
                                       int32_t elem_b, void *ws, int64_t ws_bytes, float *C,
                                       int32_t *dev_status, mx_stream stream);

/* ------------------------------------------------------------------------ */
/* S: SwiGLU between the expert projections (forward fused into GEMM1)       */
/* ------------------------------------------------------------------------ */
/*
 * Forward GEMM1 with fused SwiGLU epilogue.  Row-grouped like MX_GEMM_FWD with
 * B = the stacked [W1 | W3] weights quantized along H: B fp8 [E, 2F, H] (rows
 * 0..F-1 of each expert from W1^T, F..2F-1 from W3^T), sB scales of (E*2F, H).
 * Per row: a = x W1, b = x W3 accumulated in fp32 and rounded to bf16, saved to
 * ab bf16 [M_cap, 2F] (a in columns 0..F-1, b in F..2F-1); h = silu(a) * b in
 * fp32 (silu(a) = a / (1 + e^-a), the sigmoid of mx_selftest_sigmoid) is
 * quantized (ROW mode, blocks along F) into hq fp8 [M_cap, F] and hs
 * (MX_SCALE_SWIZZLED scales of (M_cap, F)).
 * F % 128 == 0, H % 128 == 0, M_cap % 128 == 0.  A, B, sA, sB, ab and hq
 * 16-byte aligned; hs may sit at any byte.
 */
mx_status moe_gemm1_swiglu(const uint8_t *A, const uint8_t *sA, const uint8_t *B,
                           const uint8_t *sB, const int32_t *offsets, int32_t E,
                           int64_t M_cap, int64_t F, int64_t H, void *ab,
                           uint8_t *hq, uint8_t *hs, int32_t *dev_status,
                           mx_stream stream);

/*
 * SwiGLU backward + quantization for the GEMM1 backward GEMMs.  dh fp32
 * [M_cap, F] (from the GEMM2 dgrad), ab bf16 [M_cap, 2F] (saved forward a|b).
 *   da = dh * b * s * (1 + a (1 - s)),  db = dh * silu(a),  s = sigmoid(a);
 *   dab = [da | db] [M_cap, 2F] is quantized ROW (blocks along 2F) into
 *   dab_rq / dab_rs and COL (blocks of 32 rows, transposed [2F, M_cap]) into
 *   dab_cq / dab_cs; h = silu(a) * b is recomputed and quantized COL into
 *   h_cq [F, M_cap] / h_cs.  All scales MX_SCALE_SWIZZLED.
 * `rows` = rows to process (<= M_cap, multiple of 128).  F % 32 == 0.
 * row_limit: optional device int32 (NULL = all `rows`): 128-row bands that
 * start at or past *row_limit are skipped and their outputs left untouched
 * (the layer passes offsets + E, the end of the routed rows).
 * grad_elem: element format of [da|db] (MX_ELEM_E4M3 or MX_ELEM_E5M2, the
 * gradient option); h is always E4M3.
 * Arithmetic: fp32; sigmoid(a) from the hardware's approximate base-2
 * exponential and reciprocal with an exactly rounded exponent (see
 * mx_selftest_sigmoid): a few fp32 ulps over bf16 a in [-128, 128].
 * Alignment: dh, ab, dab_rq, dab_cq and h_cq 16-byte aligned; the scale
 * arrays dab_rs, dab_cs and h_cs may sit at any byte.
 */
mx_status moe_swiglu_bwd(const float *dh, const void *ab, int64_t rows,
                         int64_t F, int32_t grad_elem, uint8_t *dab_rq, uint8_t *dab_rs,
                         uint8_t *dab_cq, uint8_t *dab_cs, uint8_t *h_cq,
                         uint8_t *h_cs, const int32_t *row_limit,
                         mx_stream stream);

/* ------------------------------------------------------------------------ */
/* Backward helpers (token shuffle of the gradients, gate gradient)          */
/* ------------------------------------------------------------------------ */
/*
 * Gather + quantize: builds the permuted matrix Z [rows_cap, H] row by row,
 *   Z[r] = bf16(gate[src[r]] * x[src[r] / k])   (fp32 product, RNE; gate NULL:
 *                                               Z[r] = x[src[r] / k] exactly)
 *   Z[r] = 0 where src[r] < 0 (pad rows and rows past the last group),
 * and quantizes it without storing it: ROW (blocks along H) into q_row
 * [rows_cap, H] / s_row, and/or COL (blocks of 32 rows, transposed) into
 * q_col [H, rows_cap] / s_col.  Scales are MX_SCALE_SWIZZLED.  Used for the
 * routed output gradient dY = gate * dOut (both layouts) and for the permuted
 * input x (COL, for wgrad).  x bf16 [T, H]; src from moe_permute_map.
 * H % 128 == 0, rows_cap % 128 == 0.  row_limit: optional device int32 (NULL
 * = all rows_cap rows): 128-row bands that start at or past *row_limit are
 * skipped and their outputs left untouched (the layer passes offsets + E).
 * elem: element format of both outputs (MX_ELEM_E4M3 or MX_ELEM_E5M2).
 */
mx_status moe_gather_quant(const void *x, const float *gate, const int32_t *src,
                           int64_t T, int64_t H, int32_t k, int64_t rows_cap,
                           int32_t mode, int32_t elem, uint8_t *q_row, uint8_t *s_row,
                           uint8_t *q_col, uint8_t *s_col,
                           const int32_t *row_limit, mx_stream stream);

/*
 * Gate gradient: d_gate[t,j] = sum_h dOut[t,h] * y[dst[t*k+j], h], fp32
 * accumulation in a fixed order (deterministic).  dOut bf16 [T, H], y bf16
 * [rows, H], d_gate fp32 [T, k].  H % 8 == 0.
 */
mx_status moe_gate_grad(const void *dOut, const void *y, const int32_t *dst,
                        int64_t T, int64_t H, int32_t k, float *d_gate,
                        mx_stream stream);

/* ------------------------------------------------------------------------ */
/* L: the MXFP8 MoE SwiGLU layer ([A] Overview: the MoE layer rewritten on   */
/* MXFP8 kernels, forward and backward)                                      */
/* ------------------------------------------------------------------------ */
/*
 * Dimensions: T tokens, H hidden, E experts, F FFN width, k experts per token.
 * H % 256 == 0, F % 256 == 0, T >= 0, 1 <= k <= min(E, 8), E <= 256.  T = 0 (an
 * empty batch) is valid: nothing is routed, the weight gradients are zero,
 * and the token arrays may be NULL.
 *
 * Weights (bf16, device): W13 [E, H, 2F] = [W1 | W3] stacked along the last
 * dim; W2 [E, F, H].  moe_layer_prep_weights quantizes them into the four
 * MXFP8 layouts the GEMMs read (forward: along H / along F; dgrad: along 2F /
 * along H), from one read of each weight, into `wq` (device scratch of
 * moe_layer_weights_size bytes).  Call it whenever the weights change.
 *
 * moe_layer_fwd: x bf16 [T, H].  If `logits` (fp32 [T, E]) is non-NULL the
 * router fills ids/gate; otherwise ids int32 [T, k] and gate fp32 [T, k]
 * (gate NULL = all ones) are inputs.  out bf16 [T, H].  Saves what the
 * backward needs in `ws` (moe_layer_workspace_size bytes).
 *
 * moe_layer_bwd: dOut bf16 [T, H] -> dX bf16 [T, H], dW13 [E, H, 2F] and dW2
 * [E, F, H] in `wgrad_dtype`, d_gate fp32 [T, k] (NULL: not computed).  Uses
 * the `ws` and `wq` of the matching forward.  grad_elem: element format of
 * the two gradient operands the backward quantizes, dY = gate * dOut and
 * [da|db] (MX_ELEM_E4M3; MX_ELEM_E5M2 is the gradient option); weights, h and
 * the permuted input stay E4M3.  wgrad_dtype: MX_OUT_F32 (fp32 weight
 * gradients, the reading for gradients that feed an optimizer) or
 * MX_OUT_BF16 (each element the fp32 accumulation rounded once to bf16: the
 * weight-gradient GEMMs then write half the bytes).
 */
int64_t moe_layer_weights_size(int64_t H, int64_t F, int32_t E);
int64_t moe_layer_workspace_size(int64_t T, int64_t H, int64_t F, int32_t E,
                                 int32_t k);
mx_status moe_layer_prep_weights(const void *W13, const void *W2, int64_t H,
                                 int64_t F, int32_t E, void *wq,
                                 int64_t wq_bytes, mx_stream stream);
mx_status moe_layer_fwd(const void *x, const float *logits, int32_t *ids,
                        float *gate, const void *wq, int64_t T, int64_t H,
                        int64_t F, int32_t E, int32_t k, void *ws,
                        int64_t ws_bytes, void *out, int32_t *dev_status,
                        mx_stream stream);
mx_status moe_layer_bwd(const void *x, const void *dOut, const float *gate,
                        const void *wq, int64_t T, int64_t H, int64_t F,
                        int32_t E, int32_t k, int32_t grad_elem, int32_t wgrad_dtype,
                        void *ws, int64_t ws_bytes, void *dX, void *dW13, void *dW2,
                        float *d_gate, int32_t *dev_status, mx_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* MXMOE_H */
