/*
 * fp8fg.h -- C ABI of libfp8fg.so: fine-grained E4M3 quantisation and
 * block-scaled FP8 GEMMs with per-128-K FP32 promotion, for NVIDIA B300
 * (sm_103a).
 *
 * The method is the FP8 mixed-precision training scheme described on the
 * scraped DeepSeek-V3 pages (cited as page + passage):
 *   page 1 = xn--9g3bo1gtkw0l8ubf92bgle.kr qna #85187,
 *   page 2 = inprokorea.com free #735329,
 *   page 5 = inprokorea.com free #890463.
 *
 * Conventions for every entry point
 *   - Memory: every pointer argument is a DEVICE pointer, except where stated.
 *     The caller owns and allocates all of it; the library allocates nothing
 *     per call.  (It keeps one device status word and, per device, a cached
 *     SM count; both live until the library is unloaded.)
 *   - Layout: tensors are dense, contiguous, row-major; no leading dimension.
 *   - Alignment: every pointer must be 16-byte aligned.
 *   - Sizes: int64_t, each dimension below 2^31; K % 128 == 0 everywhere.
 *   - Stream: `stream` is a cudaStream_t (NULL = the legacy default stream).
 *     Every call is asynchronous on it.  The return value reports argument
 *     validation and launch errors only; no kernel is launched when the
 *     arguments are rejected.
 *   - Device-detected errors (a pipeline wait that ran out of its cycle limit,
 *     bad expert offsets) are written to the library status word; the kernel
 *     then stops early without trapping.  fp8_get_device_status() reports and
 *     clears it.
 *   - There is no CPU fallback: without a CUDA device every call returns
 *     FP8FG_ERR_CUDA (after validation).
 */
#ifndef FP8FG_H_
#define FP8FG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FP8FG_OK = 0,
  FP8FG_ERR_INVALID_ARG = 1,      /* null pointer, negative size, unknown flag or dtype */
  FP8FG_ERR_UNSUPPORTED_SHAPE = 2,/* a dimension breaks a divisibility or size rule */
  FP8FG_ERR_MISALIGNED = 3,       /* a pointer is not 16-byte aligned */
  FP8FG_ERR_CUDA = 4,             /* a CUDA runtime/driver call failed (no device, launch) */
  FP8FG_ERR_TIMEOUT = 5,          /* device: a pipeline wait exceeded its cycle limit */
  FP8FG_ERR_BAD_OFFSETS = 6       /* device: expert offsets not 0..total, non-decreasing */
} fp8fg_status;

typedef enum { FP8FG_BF16 = 0, FP8FG_F32 = 1 } fp8fg_dtype;

/* flag bits */
#define FP8FG_POW2 1u          /* scales rounded up to an integral power of 2 */
#define FP8FG_TRANSPOSE 2u     /* act_quant: 128x1 tiles, transposed output */
#define FP8FG_B_TILE1x128 4u   /* GEMM: B carries 1x128 tile scales [N, K/128] */
#define FP8FG_WHOLE_K 8u       /* GEMM study mode: no per-128-K promotion (see below) */
#define FP8FG_STREAM_K 16u     /* fp8_blockscaled_gemm_ws: split the K slices even when it
                                  would not pay (tests, studies) */

/*
 * fp8_act_quant -- online 1x128 tile quantisation of activations to E4M3.
 * Source: page 1, Figure 7 (a) (one scale per token per 128 channels) and the
 * "Storage Format: float32" passage; page 2, passage on computing the maximum
 * absolute value online per 1x128 tile; pages 1 and 2, passage making the
 * scales integral powers of 2 for some activations (FP8FG_POW2); page 5,
 * backward-pass passage re-quantising into 128x1 tiles (FP8FG_TRANSPOSE).
 *
 * x      [M, K] BF16 or FP32 (x_dtype), row-major.
 * default: q [M, K] E4M3 codes (uint8), s [M, K/128] FP32, both row-major.
 *          Tile (r, t) = x[r, 128t .. 128t+127].
 * FP8FG_TRANSPOSE: requires M % 128 == 0; q [K, M], s [K, M/128] (row-major),
 *          tile (k, i) = x[128i .. 128i+127, k], i.e. act_quant of x^T.
 * Per tile: amax = max|x| (floored at 2^-64); s = amax/448 (IEEE FP32 divide);
 *          codes = E4M3_rne_satfinite(x * (448/amax)), one FP32 multiply each.
 *          FP8FG_POW2: s = 2^ceil(log2(amax/448)), multiplier 1/s (exact).
 * M may be 0 (nothing is launched).  Flags other than POW2|TRANSPOSE are
 * rejected.
 */
fp8fg_status fp8_act_quant(const void* x, fp8fg_dtype x_dtype, int64_t M, int64_t K,
                           uint8_t* q, float* s, unsigned flags, void* stream);

/*
 * fp8_requant_transpose -- backward re-quantisation of stored FP8 activations.
 * Source: page 5, backward-pass passage: the FP8 activations kept from the
 * forward pass are dequantised, transposed and quantised again in 128x1 tiles
 * (the operand layout the weight-gradient GEMM needs).
 *
 * q    [M, K] E4M3 codes with 1x128 scales s [M, K/128] (fp8_act_quant's
 *      output layout), M % 128 == 0, K % 128 == 0.
 * q_t  [K, M] codes, s_t [K, M/128] FP32: tile (k, i) = column k of the
 *      dequantised matrix, rows 128i .. 128i+127, as fp8_act_quant with
 *      FP8FG_TRANSPOSE would produce from it.
 * Dequantisation: x = fl32(decode(q) * s[row, k/128]) (one IEEE multiply;
 * E4M3 values are exact in FP32); then the scale rule of fp8_act_quant per
 * 128x1 tile.  Flags: FP8FG_POW2 only.  q must hold no NaN codes.
 * M may be 0 (nothing is launched).
 */
fp8fg_status fp8_requant_transpose(const uint8_t* q, const float* s, int64_t M, int64_t K,
                                   uint8_t* q_t, float* s_t, unsigned flags, void* stream);

/*
 * fp8_weight_quant -- online 128x128 block quantisation of weights to E4M3.
 * Source: page 1, Figure 7 (a) (one scale per 128 input x 128 output
 * channels) and "Storage Format" passage; page 2, online-amax passage.
 *
 * w    [N, K] BF16 or FP32, N % 128 == 0, K % 128 == 0.
 * q    [N, K] codes; s [N/128, K/128] FP32 (block (i, j) = rows 128i.., cols 128j..).
 * q_t  optional (NULL to skip) [K, N] codes = q transposed; s_t [K/128, N/128]
 *      = s transposed (both or neither).  These feed the Dgrad GEMM.
 * Scale rule as fp8_act_quant, per block; FP8FG_POW2 is honoured.
 */
fp8fg_status fp8_weight_quant(const void* w, fp8fg_dtype w_dtype, int64_t N, int64_t K,
                              uint8_t* q, float* s, uint8_t* q_t, float* s_t, unsigned flags,
                              void* stream);

/*
 * fp8_blockscaled_gemm -- C = A . B^T with per-128-K promotion.
 * Source: page 2, promotion passage (partial results copied to FP32 registers
 * and accumulated there; the garbled interval is read as 128, the K group of
 * the scales) and Figure 6 (Fprop, Dgrad and Wgrad all in FP8); page 2,
 * passage multiplying the per-group K scales in during dequantisation.
 *
 * a  [M, K] E4M3 codes, sa [M, K/128] FP32 (1x128 tiles).
 * b  [N, K] E4M3 codes; sb [N/128, K/128] FP32 (128x128 blocks, requires
 *    N % 128 == 0) or, with FP8FG_B_TILE1x128, sb [N, K/128] (1x128 tiles,
 *    requires N % 16 == 0).
 * c  [M, N] BF16 or FP32 (c_dtype), row-major.
 * C[m,n] = sum_kb P_kb[m,n] * sa[m,kb] * sb(n,kb), P_kb the tensor-core product
 * over K group kb; each P_kb is scaled and added into an FP32 accumulator; the
 * output is rounded once (RNE to BF16, or stored as FP32).
 * M >= 0 arbitrary (0: nothing launched); N >= 16; K >= 128.
 *
 * The dense kernel lets a launch queued after it with programmatic stream
 * serialisation start early (griddepcontrol.launch_dependents at its start);
 * such a kernel must wait for it (griddepcontrol.wait, or
 * cudaGridDependencySynchronize) before it reads C, as programmatic dependent
 * launch requires.  Launches without that attribute see the usual stream order.
 *
 * FP8FG_WHOLE_K (study mode, not with FP8FG_B_TILE1x128): the promotion the
 * pages prescribe is switched off.  All of K accumulates inside the tensor
 * core (one TMEM accumulator per tile) and the result is scaled once by
 * sa[0] * sb[0], i.e. per-tensor scales; sa and sb still have their usual
 * shapes but only their first element is read.  It measures the accumulation
 * error the promotion exists to avoid (page 2, passage on the limited
 * accumulation precision of FP8 tensor-core GEMMs and Figure 6).
 */
fp8fg_status fp8_blockscaled_gemm(const uint8_t* a, const float* sa, const uint8_t* b,
                                  const float* sb, void* c, fp8fg_dtype c_dtype, int64_t M,
                                  int64_t N, int64_t K, unsigned flags, void* stream);

/*
 * fp8_blockscaled_gemm_ws -- fp8_blockscaled_gemm with a caller-owned workspace
 * for a stream-K split of the work.  Same operation, arguments and rules as
 * fp8_blockscaled_gemm (page 2, promotion passage and Figure 6); flags within
 * FP8FG_B_TILE1x128 | FP8FG_STREAM_K.
 *
 * When the last wave of whole 128x256 output tiles would leave most SMs idle
 * for at least 40 of the 128-K slices (the Dgrad shape 4096 x 7168 x 18432: 896
 * tiles on 148 SMs), the full waves run as whole tiles and each leftover tile
 * is shared by its own group of SMs, which divide its 128-K slices evenly; a
 * shared tile is summed in FP32 from the group's partial sums, in a fixed
 * order, by a second kernel on the same stream (same result for every run;
 * one more FP32 addition per extra part than the whole-tile path).
 * FP8FG_STREAM_K applies the split whenever the tiles do not fill whole waves.
 *
 * A split call enqueues up to three kernels on `stream`: the whole tiles; the
 * shared tiles, launched with programmatic stream serialisation so that they
 * start on each SM as the first kernel's block there finishes (they read only
 * the inputs, and end only after the first kernel has); the fix-up.  Work
 * enqueued after the call sees all of C, as after any other call; the three
 * launches can be captured into a CUDA graph like a single one.
 *
 * workspace  DEVICE, 16-byte aligned, at least
 *            fp8_blockscaled_gemm_workspace_bytes(M, N, K, flags) bytes (the
 *            split needs 128 KB per SM of the current device: 18.5 MB on 148
 *            SMs), or NULL: then no split is made (FP8FG_STREAM_K then fails
 *            with FP8FG_ERR_INVALID_ARG).  Its contents on entry do not matter;
 *            it must not be used by another call running at the same time.
 * A non-NULL workspace smaller than needed: FP8FG_ERR_INVALID_ARG.
 */
fp8fg_status fp8_blockscaled_gemm_ws(const uint8_t* a, const float* sa, const uint8_t* b,
                                     const float* sb, void* c, fp8fg_dtype c_dtype, int64_t M,
                                     int64_t N, int64_t K, unsigned flags, void* workspace,
                                     size_t workspace_bytes, void* stream);

/*
 * fp8_blockscaled_gemm_workspace_bytes -- workspace bytes fp8_blockscaled_gemm_ws
 * uses for this shape and flags on the current device; 0 when it would not
 * split the work (or without a device, or for invalid sizes).
 */
size_t fp8_blockscaled_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, unsigned flags);

/*
 * fp8_blockscaled_gemm_noalloc -- fp8_blockscaled_gemm_ws for callers that
 * cannot allocate device memory when they call the GEMM: code running while a
 * memory pool is locked or a graph is being captured, allocators that must not
 * be re-entered, runtimes with a fixed memory budget decided up front.  The
 * pages have no counterpart of this entry point; it only changes where the
 * scratch of the stream-K split lives.
 *
 * Same operation, arguments, flags (FP8FG_B_TILE1x128, FP8FG_STREAM_K) and
 * results as fp8_blockscaled_gemm_ws given a large enough workspace; the
 * caller still passes every input and the output.  The split's partial tiles
 * go to a 20 MiB array of device memory that the library holds on every GPU
 * that loads it, until the process exits (the split needs 128 KB per SM, so
 * it covers devices of up to 160 SMs).  Nothing is allocated: no cudaMalloc,
 * no cudaFree, no allocating library call.
 *
 * - The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.
 * - Every call shares the array and it keeps the last call's contents; no
 *   part of it needs to start at zero (each SM of a split writes its whole
 *   slot before the fix-up kernel reads it).  Calls that overlap on the GPU
 *   (other streams, other threads) race on it: order them on one stream.
 * - A shape whose split on the current device would need more than the array
 *   holds (a device with more than 160 SMs): FP8FG_ERR_UNSUPPORTED_SHAPE,
 *   nothing launched.
 */
fp8fg_status fp8_blockscaled_gemm_noalloc(const uint8_t* a, const float* sa, const uint8_t* b,
                                          const float* sb, void* c, fp8fg_dtype c_dtype, int64_t M,
                                          int64_t N, int64_t K, unsigned flags, void* stream);

/*
 * fp8_blockscaled_gemm_quant -- fp8_blockscaled_gemm whose FP32 result is
 * quantised in the epilogue into 1x128 E4M3 tiles along N, the form in which
 * the next FP8 GEMM takes its activation input.  Source: page 2, fine-grained
 * quantisation passage (1x128 activation tiles, online amax, FP32 scales);
 * pages 1-2, power-of-2 passage (integral power-of-2 scales for the inputs the
 * pages name).  Reading: the tile is quantised from the FP32 accumulator, with
 * no BF16 rounding in between.
 *
 * a, sa, b, sb as fp8_blockscaled_gemm (flags may hold FP8FG_B_TILE1x128).
 * q  [M, N] E4M3 codes, row-major; s [M, N/128] FP32 dequantisation scales.
 * Per tile: amax = max |C| floored at 2^-64; s = amax/448 and codes
 * e4m3(C * (448/amax)) (IEEE division and multiply, RNE, saturating), or with
 * FP8FG_POW2 s = 2^ceil(log2(amax/448)) and codes e4m3(C / s).  Equal to
 * fp8_act_quant applied to the FP32 output of fp8_blockscaled_gemm.
 * Requires N % 128 == 0, K % 128 == 0, K >= 128; M >= 0 (0: nothing launched).
 * Pointers 16-byte aligned; the caller owns all memory.
 */
fp8fg_status fp8_blockscaled_gemm_quant(const uint8_t* a, const float* sa, const uint8_t* b,
                                        const float* sb, uint8_t* q, float* s, int64_t M,
                                        int64_t N, int64_t K, unsigned flags, void* stream);

/*
 * fp8_grouped_gemm -- fp8_blockscaled_gemm per routed expert over contiguous
 * row groups.  Source: page 2, passage quantising the activation before the
 * MoE up-projection for FP8 Fprop; page 5, MoE configuration passage (256
 * routed experts, 8 active per token, expert hidden size 2048).
 *
 * a        [total_rows, K] codes, rows grouped by expert; sa [total_rows, K/128].
 * offsets  DEVICE int32 [E+1]: expert e owns rows offsets[e] .. offsets[e+1]-1.
 *          Must satisfy offsets[0] == 0, non-decreasing, offsets[E] == total_rows;
 *          checked on the device (FP8FG_ERR_BAD_OFFSETS, nothing written).
 * b        [E, N, K] codes; sb [E, N/128, K/128] FP32 (128x128 blocks).
 * c        [total_rows, N] BF16 or FP32.  Rows of empty experts: none.
 * Requires 1 <= E <= 1024, N % 128 == 0; flags must be 0.  total_rows == 0:
 * nothing is launched (a, sa and c may be null; offsets are not read).
 */
fp8fg_status fp8_grouped_gemm(const uint8_t* a, const float* sa, const int32_t* offsets,
                              int32_t E, int64_t total_rows, const uint8_t* b, const float* sb,
                              void* c, fp8fg_dtype c_dtype, int64_t N, int64_t K, unsigned flags,
                              void* stream);

/*
 * fp8_grouped_gemm_swiglu_quant -- the routed up-projection followed by SwiGLU,
 * leaving h as the down-projection's FP8 input.  Source: page 2, passage
 * quantising the MoE up-projection input for FP8 Fprop and the power-of-2
 * passage naming the activations cached with integral power-of-2 scales; page
 * 5, MoE configuration passage (expert hidden size 2048).  Readings (the pages
 * name neither): the activation is SwiGLU, h = silu(g) * u, and each expert's
 * up-projection rows are its I gate rows followed by its I up rows.
 *
 * a, sa, offsets, E, total_rows as fp8_grouped_gemm (offsets checked on the
 * device, FP8FG_ERR_BAD_OFFSETS, nothing written).
 * b  [E, N, K] codes with N = 2I (gate rows 0..I-1, up rows I..2I-1);
 *    sb [E, N/128, K/128] FP32 (128x128 blocks).
 * q  [total_rows, I] E4M3 codes of h; s [total_rows, I/128] FP32 scales.
 * g and u are the FP32 accumulators of the promoted sums; h = g / (1 + e^-g) * u
 * in FP32 with the fast exponential and divide (relative error of silu at most
 * (4 + 1.2 |g|) 2^-23, a zero of the right sign below g = -87); per 1x128 tile of h the
 * activation quantiser's rules apply, power-of-2 scales with FP8FG_POW2 (the
 * pages' choice for this tensor).
 * Requires 1 <= E <= 1024, N % 256 == 0, K % 128 == 0; flags within FP8FG_POW2.
 * total_rows == 0: nothing is launched (a, sa, q and s may be null).
 */
fp8fg_status fp8_grouped_gemm_swiglu_quant(const uint8_t* a, const float* sa,
                                           const int32_t* offsets, int32_t E, int64_t total_rows,
                                           const uint8_t* b, const float* sb, uint8_t* q, float* s,
                                           int64_t N, int64_t K, unsigned flags, void* stream);

/*
 * fp8_get_device_status -- synchronises `stream`, then returns and clears the
 * library status word (FP8FG_OK, FP8FG_ERR_TIMEOUT or FP8FG_ERR_BAD_OFFSETS);
 * FP8FG_ERR_CUDA if the synchronisation itself failed.
 */
fp8fg_status fp8_get_device_status(void* stream);

/* Short English description of a status code (static storage). */
const char* fp8fg_status_string(fp8fg_status status);

/* ABI version of this header (bumped on any signature change or addition). */
int fp8fg_abi_version(void);

/*
 * fp8fg_set_wait_limit -- cycle limit of every pipeline wait in later launches
 * (default 2^32 cycles, about two seconds; 0 restores the default).  Also read
 * once from the environment variable FP8FG_WAIT_LIMIT_CYCLES.  Host-side only.
 * The waits with which a stopping GEMM block lets its own copies and MMAs
 * finish before it frees its memory use at least 2^27 cycles (~67 ms) even
 * when a smaller limit is set.
 */
void fp8fg_set_wait_limit(uint64_t cycles);

/*
 * fp8fg_selftest_wait_timeout -- failure-detection self-test.  Launches one
 * CTA that waits on an mbarrier nothing will ever arrive on, with the given
 * cycle limit (1 .. 2^31), so the wait must give up and record
 * FP8FG_ERR_TIMEOUT.  Read the result with fp8_get_device_status().
 */
fp8fg_status fp8fg_selftest_wait_timeout(uint32_t limit_cycles, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8FG_H_ */
