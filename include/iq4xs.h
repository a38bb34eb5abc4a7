/*
 * iq4xs.h -- C ABI of libiq4xs.so: IQ4_XS x Q8_1 batched matmul on GB300
 * (sm_103a).
 *
 *   y[M,N] = x[M,K] . W[N,K]^T
 *
 * W is IQ4_XS-quantized (136-byte super-blocks of 256 weights, 4.25 bits per
 * weight); x is quantized per 32 values to Q8_1 by iq4xs_quantize_q8_1 and the
 * product is formed from exact integer per-32-weight dot products, each
 * scaled by d_w*(ls-32)*d_x and accumulated in fp32.  The method is the one described on the V100TPS engine page
 * (agent-report.daedalus.work/V100TPS/engine.html): the kernel table at M=64
 * (quantize_q8_1 feeding the batched matmul), the new-kernel table (batched
 * IQ4_XS for 4 <= M <= 96) and the tile-geometry passage after it (sub-block
 * scale d*(ls-32), nibbles through kvalues_iq4nl, low nibbles = elements
 * 0-15 of a sub-block, high nibbles = 16-31).
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - All data pointers are DEVICE pointers owned by the caller.  The library
 *    never allocates, frees or retains them, and allocates nothing per call.
 *    Exception: the activations x (iq4xs_quantize_q8_1, iq4xs_linear) and
 *    the result y (iq4xs_matmul, iq4xs_linear) may instead be HOST memory
 *    the device can address -- page-locked host memory under unified
 *    addressing (cudaHostAlloc, cudaHostRegister), whose pointer is the
 *    device pointer -- in which case the quantizer reads x and the matmul
 *    writes y over the host-device link (NVLink-C2C on Grace-Blackwell)
 *    with no staging copy; results are bit-identical to device buffers.
 *    The library does not check which kind of memory it was given.
 *    A one-time per-device set-up (architecture check, the tensor-map encoder
 *    entry point, kernel attributes) runs on the first call made on a device.
 *  - `stream` is a cudaStream_t passed as an int64 (0 = legacy default
 *    stream).  Every call is asynchronous on that stream and never
 *    synchronizes; results are ready when the stream reaches that point.
 *  - The current CUDA device (cudaSetDevice) is the one used; it must be an
 *    sm_103 GPU (GB300) or the call returns IQ4XS_ERR_DEVICE.
 *  - Argument errors are detected on the host BEFORE any launch and are
 *    returned synchronously; nothing is launched and no output is touched.
 *    Launch failures return IQ4XS_ERR_CUDA.  A device-side bounded wait that
 *    ran out sets a device error word (see iq4xs_last_device_error) and the
 *    kernel returns without hanging; the outputs of that call are undefined.
 *  - Shapes: 1 <= M <= 32768; N >= 1; K a positive multiple of 256.
 *
 * Data layouts
 * ------------
 *  W (IQ4_XS): row-major [N][K/256] super-blocks, each 136 bytes:
 *      bytes 0-1   d         fp16, little endian
 *      bytes 2-3   scales_h  u16, little endian: bits 2j..2j+1 are the two
 *                            high bits of ls_j
 *      bytes 4-7   scales_l  u8[4]: low nibble of byte j/2 holds the four low
 *                            bits of ls_j for even j, high nibble for odd j
 *      bytes 8-135 qs        u8[128]: sub-block j uses bytes 16j..16j+15;
 *                            element i (0..15) is the low nibble of byte
 *                            16j+i, element 16+i the high nibble
 *      weight = fp32(d) * (ls_j - 32) * kvalues_iq4nl[nibble].
 *      Rows are K/256*136 bytes apart; W must be 16-byte aligned.
 *  Q8_1 activations (structure of arrays):
 *      qs  int8  [M][K]     q = round(x/d), ties away from zero
 *      ds  half2 [M][K/32]  {d = amax/127, s = d*sum(q)} each rounded to fp16
 *      Both matmul paths read these two arrays as they are (1.125 bytes per
 *      activation); qs must be 16-byte aligned, ds 4-byte aligned.
 *  Prepared tensor-core operand (opaque; iq4xs_quantize_q8_1_tc writes it
 *      beside qs and ds, iq4xs_matmul_tc_operand reads it): each value q*d
 *      (d the block's stored fp16 scale) held exactly as a pair of fp16
 *      values, tiled for the tcgen05 kernel; iq4xs_tc_operand_bytes(M, K) =
 *      4 * Mpad * K + 4 * Mpad * ceil(K/1024) bytes (Mpad = M rounded up to
 *      the tile height), 16-byte aligned.  It costs the quantizer one more
 *      write of 4 bytes per activation and spares every CTA of the matmul
 *      the conversion of the codes and the activation scaling.
 *  y: fp32 [M][ldy] row-major, ldy >= N; columns N..ldy-1 are not written.
 */
#ifndef IQ4XS_H
#define IQ4XS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    IQ4XS_OK = 0,
    IQ4XS_ERR_ARG = 1,     /* null pointer, bad size, ldx/ldy too small, bad enum */
    IQ4XS_ERR_ALIGN = 2,   /* a pointer lacks the alignment stated for it */
    IQ4XS_ERR_SHAPE = 3,   /* K not a multiple of 256, M out of range, or a shape
                              the requested path cannot take */
    IQ4XS_ERR_DEVICE = 4,  /* no CUDA device, or the current device is not sm_103 */
    IQ4XS_ERR_CUDA = 5,    /* a CUDA runtime/driver call or a launch failed */
    IQ4XS_ERR_TIMEOUT = 6, /* a bounded device wait ran out (iq4xs_last_device_error) */
    IQ4XS_ERR_BOUNDS = 7   /* bounds-checked build only: a checked device access
                              missed its buffer (iq4xs_last_device_error) */
} iq4xs_status;

typedef enum {
    IQ4XS_PATH_AUTO = 0,    /* iq4xs_select_path decides from (M, N, K)          */
    IQ4XS_PATH_DP4A = 1,    /* CUDA-core int8 dot products (small M)             */
    IQ4XS_PATH_TC = 2,      /* tcgen05 tensor cores: exact integer sub-block dots
                               in fp32 tensor memory, fp32 scale-in (larger M)   */
    IQ4XS_PATH_BASELINE = 3,/* advice from iq4xs_select_path only: above a
                               measured M, dequantizing W (iq4xs_dequantize) and
                               a dense bf16 GEMM in the caller's BLAS is faster,
                               at bf16 precision.  The library's own calls never
                               take it: iq4xs_matmul / iq4xs_linear run TC
                               there, and reject it as an explicit path.        */
    IQ4XS_PATH_MMA = 4      /* warp-level tensor-core MMA (mma.sync m16n8k16):
                               decoded weights go straight from the byte-table
                               lookup into the MMA's registers and every
                               sub-block's exact integer dot is scaled in from
                               registers (small and medium M; every weight
                               format)                                        */
} iq4xs_path;

/*
 * Weight formats (engine page, tile-geometry passage: an IQ4_XS 32-weight
 * sub-block is exactly one Q4_0 block -- 16 bytes of nibbles, low nibbles =
 * elements 0-15, high = 16-31 -- and the two differ only in the scale and in
 * the nibble's value; forum page on the Qwen3.5 engine: IQ4_NL is the
 * kvalues_iq4nl codebook on (32, 18) blocks).  Q4_0 and IQ4_NL share one
 * byte shape, row-major [N][K/32] blocks of 18 bytes:
 *      bytes 0-1   d    fp16, little endian
 *      bytes 2-17  qs   u8[16]: element i (0..15) is the low nibble of byte
 *                       2+i, element 16+i the high nibble
 *      Q4_0:   weight = fp32(d) * (nibble - 8)
 *      IQ4_NL: weight = fp32(d) * kvalues_iq4nl[nibble]
 * Rows are K/32*18 bytes apart; K must be a multiple of 256 here as for
 * IQ4_XS (rows are then 16-byte aligned), and W 16-byte aligned.
 */
typedef enum {
    IQ4XS_WTYPE_IQ4_XS = 0,
    IQ4XS_WTYPE_Q4_0 = 1,
    IQ4XS_WTYPE_IQ4_NL = 2
} iq4xs_wtype;

/* Bytes of an [N][K] weight matrix in format wtype; 0 if invalid. */
int64_t iq4xs_weight_bytes(int wtype, int64_t N, int64_t K);

/*
 * Q8_1 activation quantization (engine page, kernel table at M=64: the
 * activations enter the batched matmul through quantize_q8_1).
 *   x           fp32 [M][ldx], ldx >= K, 4-byte aligned, ldx*4 % 16 == 0 and
 *               x 16-byte aligned (rows are read as float4).
 *   qs, ds      outputs, layouts above; qs 16-byte aligned, ds 4-byte aligned.
 * Per block of 32: amax = max|x|, d = amax/127 (IEEE fp32 division),
 * q = d == 0 ? 0 : roundf(x/d), s = d*sum(q); d and s stored as fp16 (RNE).
 * Inputs must be finite (NaN/Inf give unspecified codes).
 */
int iq4xs_quantize_q8_1(const float* x, int64_t M, int64_t K, int64_t ldx,
                        int8_t* qs, void* ds, int64_t stream);

/*
 * iq4xs_quantize_q8_1 that also writes the prepared tensor-core operand
 * (layout above; padding rows written as zeros) for iq4xs_matmul_tc_operand.
 * tc_operand: iq4xs_tc_operand_bytes(M, K) bytes, 16-byte aligned, non-NULL.
 * qs and ds are written exactly as iq4xs_quantize_q8_1 writes them.
 */
int iq4xs_quantize_q8_1_tc(const float* x, int64_t M, int64_t K, int64_t ldx,
                           int8_t* qs, void* ds, void* tc_operand, int64_t stream);

/* Bytes of the prepared tensor-core operand for (M, K); 0 if invalid. */
int64_t iq4xs_tc_operand_bytes(int64_t M, int64_t K);

/*
 * Batched matmul y = x . W^T from IQ4_XS W and Q8_1 x (engine page,
 * new-kernel table and tile-geometry passage: per-32 sub-block integer dot
 * products scaled by d_w*(ls-32)*d_x into fp32).
 *   w       IQ4_XS [N][K/256] blocks, 16-byte aligned.
 *   qs, ds  Q8_1 activations as iq4xs_quantize_q8_1 writes them (qs 16-byte,
 *           ds 4-byte aligned), read on either path.
 *   M       activation rows; y fp32 [M][ldy] output, fully overwritten for
 *           columns < N.
 *   path    an iq4xs_path value: AUTO (the choice iq4xs_select_path makes),
 *           DP4A, TC or MMA; BASELINE is advice only and returns
 *           IQ4XS_ERR_ARG.
 * The TC and MMA paths need K % 512 == 0 (they stage W rows by tensor map,
 * whose row stride must be a multiple of 16 bytes: super-blocks in pairs),
 * else IQ4XS_ERR_SHAPE; DP4A takes any K % 256 == 0.  Every path takes
 * every weight format.
 * Result: each sub-block's dot sum_i kv*q is an exact integer on every path
 * (int32 on DP4A; on TC and MMA exact in the tensor core's fp32 accumulator,
 * every partial sum being an integer below 2^24); the scaled sub-block terms
 * are accumulated in fp32, so y differs from the fp64 definition by fp32
 * rounding and summation order only.
 */
int iq4xs_matmul(const void* w, int64_t N, int64_t K, const int8_t* qs, const void* ds,
                 int64_t M, float* y, int64_t ldy, int path, int64_t stream);

/*
 * The tensor-core matmul from the prepared operand (the faster form of the
 * TC path: the same kernel with d_x folded into exact fp16 hi / lo operand
 * pairs, four MMAs per 32-weight sub-block instead of two, no conversion in
 * the kernel and one FMA per result in its epilogue).  Each sub-block's
 * d_x*sum(kv*q) then carries the tensor core's fp32 accumulation rounding
 * (every product is exact); the bar is the same as iq4xs_matmul's.
 *   w           weights in format wtype (iq4xs_wtype), 16-byte aligned.
 *   tc_operand  from iq4xs_quantize_q8_1_tc for the same M and K.
 * K % 512 == 0, else IQ4XS_ERR_SHAPE; other errors as for iq4xs_matmul.
 */
int iq4xs_matmul_tc_operand(const void* w, int wtype, int64_t N, int64_t K,
                            const void* tc_operand, int64_t M, float* y, int64_t ldy,
                            int64_t stream);

/*
 * iq4xs_matmul for a weight in any iq4xs_wtype (IQ4XS_WTYPE_IQ4_XS is
 * iq4xs_matmul itself).  Both paths run the same tiles for every format; only
 * the decode differs (scale d per 18-byte block, nibble value q-8 or
 * kvalues_iq4nl[q]), so the result is, as for IQ4_XS, fp32 accumulation of
 * exact per-32-weight integer dots scaled by d_w * d_x.  The path choice
 * (AUTO) is the one iq4xs_select_path makes for IQ4_XS.  IQ4XS_ERR_ARG for
 * an unknown wtype.
 */
int iq4xs_matmul_wt(const void* w, int wtype, int64_t N, int64_t K, const int8_t* qs,
                    const void* ds, int64_t M, float* y, int64_t ldy, int path, int64_t stream);

/*
 * Grouped (mixture-of-experts) matmul in one launch: G experts, each with its
 * own IQ4_XS matrix and its own Q8_1 activation rows (forum page lcz.me post
 * 31556, the decode measurement of the grouped expert kernel: one call per
 * layer over the routed experts, because per-expert launches cost more than
 * the experts' bytes).  CUDA-core (DP4A) path: per-expert batches are small.
 *   w             G matrices, each [N][K/256] blocks as for iq4xs_matmul;
 *                 expert g starts at byte g * expert_stride (expert_stride
 *                 >= N*(K/256)*136 and a multiple of 16; w 16-byte aligned).
 *   qs, ds        Q8_1 rows of all experts (iq4xs_quantize_q8_1 over the
 *                 concatenated rows, grouped by expert).
 *   row_offsets   DEVICE int32 [G+1]: expert g owns rows
 *                 [row_offsets[g], row_offsets[g+1]); non-decreasing, read
 *                 by the kernel after the preceding grid completes (so it may
 *                 come from a routing kernel).
 *   total_rows    the number of rows, 1..32768 (row_offsets[G] <= total_rows); at most
 *                 min(G, total_rows) experts have rows, and the launch is
 *                 sized for that many (the kernels find the non-empty
 *                 experts themselves), so empty experts cost nothing.
 *   y             fp32 [rows][ldy]; the rows of every expert are written.
 * Path: the CUDA-core (DP4A) kernel, each expert computed with the batch
 * width its own row count selects, so the result per expert is
 * bit-identical to iq4xs_matmul on the DP4A path over the same rows; or,
 * when K % 512 == 0 and either total_rows >= min(G, 24) or the mean rows
 * per expert that has rows (total_rows / min(G, total_rows)) exceeds the
 * DP4A crossover of one expert's matrix size, a tensor-core form: the
 * warp-level MMA kernel in its grouped form (persistent: one CTA per SM
 * walks the layer's (expert, weight-row tile, activation tile) items, the
 * expert's rows in activation tiles of up to 32) below 32 mean rows per
 * expert slot, the tcgen05 kernel's grouped form from 32 on; each
 * sub-block's dot is exact as on those paths of iq4xs_matmul.
 */
int iq4xs_matmul_grouped(const void* w, int64_t expert_stride, int64_t G, int64_t N, int64_t K,
                         const int8_t* qs, const void* ds, const int32_t* row_offsets,
                         int64_t total_rows, float* y, int64_t ldy, int64_t stream);

/*
 * iq4xs_matmul_grouped with the path chosen by the caller: IQ4XS_PATH_AUTO
 * (the rule above), IQ4XS_PATH_DP4A, IQ4XS_PATH_MMA or IQ4XS_PATH_TC (the
 * last two need K % 512 == 0, else IQ4XS_ERR_SHAPE; qs 16-byte aligned);
 * other values IQ4XS_ERR_ARG.  IQ4XS_PATH_TC is the tcgen05 kernel in its
 * Q8_1 form: the layer's activation tiles (tc tile height from the mean
 * rows per expert slot, 16..128) each one CTA per 128 weight rows of its
 * expert, no K split; each sub-block's dot is exact as on that path of
 * iq4xs_matmul.
 */
int iq4xs_matmul_grouped_path(const void* w, int64_t expert_stride, int64_t G, int64_t N, int64_t K,
                              const int8_t* qs, const void* ds, const int32_t* row_offsets,
                              int64_t total_rows, float* y, int64_t ldy, int path, int64_t stream);

/*
 * iq4xs_matmul_grouped_path for experts in weight format wtype (an
 * iq4xs_wtype: every expert's N x K matrix in that format, expert_stride >=
 * iq4xs_weight_bytes(wtype, N, K)).  Q4_0 / IQ4_NL experts run on the DP4A
 * and warp-MMA forms (AUTO takes the warp-MMA form wherever it would take
 * the tcgen05 one for IQ4_XS; an explicit IQ4XS_PATH_TC returns
 * IQ4XS_ERR_SHAPE); each expert's result is that of iq4xs_matmul_wt on the
 * same path over its rows.  IQ4XS_ERR_ARG for an unknown format.
 */
int iq4xs_matmul_grouped_wt(const void* w, int wtype, int64_t expert_stride, int64_t G, int64_t N, int64_t K,
                            const int8_t* qs, const void* ds, const int32_t* row_offsets, int64_t total_rows,
                            float* y, int64_t ldy, int path, int64_t stream);

/*
 * The projection as one call: y = Q8_1(x) . W^T from fp32 activations
 * (engine page, kernel table at M=64: the projection op quantizes its
 * activations with quantize_q8_1 and runs the batched matmul).  Launches the
 * quantizer into `workspace` and then the matmul on the path
 * iq4xs_select_path picks; the second launch overlaps the first's tail
 * (programmatic dependent launch).
 *   x          fp32 [M][ldx], as for iq4xs_quantize_q8_1.
 *   workspace  device scratch owned by the caller, 16-byte aligned, of
 *              workspace_bytes >= iq4xs_linear_workspace_min_bytes(M, N, K)
 *              (M*K bytes of qs rounded up to 16, then M*K/32*4 bytes of ds
 *              rounded up to 16): its contents on return are those Q8_1
 *              activations.  On the TC path, with workspace_bytes >=
 *              iq4xs_linear_workspace_bytes(M, N, K) (the prepared operand
 *              after them), the faster prepared form runs
 *              (iq4xs_quantize_q8_1_tc + iq4xs_matmul_tc_operand); with less,
 *              the Q8_1 form (iq4xs_quantize_q8_1 + iq4xs_matmul).
 * Errors as for the two calls it makes; IQ4XS_ERR_ARG if the workspace is
 * too small.
 */
int iq4xs_linear(const void* w, int64_t N, int64_t K, const float* x, int64_t M, int64_t ldx,
                 float* y, int64_t ldy, void* workspace, int64_t workspace_bytes,
                 int64_t stream);

/*
 * iq4xs_linear for weights in format wtype (an iq4xs_wtype: W of
 * iq4xs_weight_bytes(wtype, N, K) bytes): the same workspace, path and
 * forms, the matmul that of iq4xs_matmul_wt (or, with the prepared operand,
 * iq4xs_matmul_tc_operand) for that format.  IQ4XS_ERR_ARG for an unknown
 * format.
 */
int iq4xs_linear_wt(const void* w, int wtype, int64_t N, int64_t K, const float* x, int64_t M, int64_t ldx,
                    float* y, int64_t ldy, void* workspace, int64_t workspace_bytes, int64_t stream);

/* Workspace bytes for iq4xs_linear's fastest form at (M, N, K), and the
 * least it accepts (the Q8_1 codes and scales); 0 if the shape is invalid. */
int64_t iq4xs_linear_workspace_bytes(int64_t M, int64_t N, int64_t K);
int64_t iq4xs_linear_workspace_min_bytes(int64_t M, int64_t N, int64_t K);

/*
 * iq4xs_linear without a caller workspace: the same projection, with its
 * scratch held in a fixed 8 MiB device array inside this library.  (The
 * source pages have no counterpart; this entry point serves callers that
 * cannot allocate device memory themselves -- a plugin inside a framework
 * that owns every device allocation, or a serving loop that must not
 * allocate once running, since cudaMalloc can synchronize the device, fail
 * under memory pressure, and is not allowed during stream capture.)
 *   - Allocates nothing and calls no allocating routine.  The array is
 *     created when the library is loaded and every GPU that loads it holds
 *     it until the process exits.
 *   - Size limit: iq4xs_linear_workspace_min_bytes(M, N, K), about
 *     1.125*M*K bytes, must not exceed iq4xs_linear_static_max_bytes()
 *     (8 MiB: M <= 428 at K = 17408, M <= 1456 at K = 5120); larger
 *     requests return IQ4XS_ERR_SHAPE and launch nothing.  Where the
 *     prepared tensor-core operand fits as well, the faster form runs.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before
 *     any stream capture.
 *   - Every call shares the one array and leaves its contents behind; calls
 *     that can overlap on the GPU (different streams, or different host
 *     threads without ordering) race on it.  Serialize them, e.g. on one
 *     stream.
 * Arguments and errors otherwise as for iq4xs_linear.
 */
int iq4xs_linear_static(const void* w, int64_t N, int64_t K, const float* x, int64_t M,
                        int64_t ldx, float* y, int64_t ldy, int64_t stream);

/* Bytes of the fixed scratch behind iq4xs_linear_static. */
int64_t iq4xs_linear_static_max_bytes(void);

/*
 * Dequantize W to a dense [N][K] matrix (engine page, kernel table at M=64:
 * dequantize_block_iq4_xs feeding a dense GEMM -- the baseline the batched
 * kernel replaces).  out_dtype 0 = fp32 (exact), 1 = bfloat16 (RNE of the
 * exact value).  out is 16-byte aligned, [N][K] row-major.
 */
int iq4xs_dequantize(const void* w, int64_t N, int64_t K, void* out, int out_dtype,
                     int64_t stream);

/* iq4xs_dequantize for a weight in any iq4xs_wtype (exact fp32, or bf16 RNE). */
int iq4xs_dequantize_wt(const void* w, int wtype, int64_t N, int64_t K, void* out,
                        int out_dtype, int64_t stream);

/*
 * Path choice for (M, N, K) (engine page, mmvq vs dequantize table: the
 * original dispatcher hard-coded its threshold at M=8 while the measured
 * crossover was M~15; the dequantize + GEMM route was the choice above it).
 * Host only, no device access.  For the matrix's weight-size class (N*K):
 * DP4A when M <= the calibrated DP4A crossover (iq4xs_set_crossover,
 * iq4xs_set_crossover_classes); MMA when M <= the calibrated warp-MMA
 * crossover (iq4xs_set_mma_crossover, iq4xs_set_mma_crossover_classes);
 * BASELINE when M >= the calibrated baseline threshold (0 = never); TC
 * otherwise.  K % 512 != 0 always gives DP4A (neither tensor-core path takes
 * it).  Q4_0 / IQ4_NL weights (iq4xs_matmul_wt with AUTO) take the same
 * path as IQ4_XS weights of the same shape.
 */
int iq4xs_select_path(int64_t M, int64_t N, int64_t K, int* path_out);

/*
 * The form iq4xs_matmul_grouped_wt takes with IQ4XS_PATH_AUTO for G experts
 * of N x K weights in format wtype over total_rows rows (the rule given
 * with iq4xs_matmul_grouped): IQ4XS_PATH_DP4A, IQ4XS_PATH_MMA or
 * IQ4XS_PATH_TC.  Host only, no device access.  IQ4XS_ERR_SHAPE for sizes
 * out of the call's range, IQ4XS_ERR_ARG for a null output or an unknown
 * format.
 */
int iq4xs_select_grouped_path(int64_t G, int64_t N, int64_t K, int64_t total_rows, int wtype, int* path_out);

/*
 * Install the measured crossover: DP4A is chosen for M <= m_max_dp4a.
 * Host only.  Defaults to 4 until a calibration sets it.  Thread-safe.
 */
int iq4xs_set_crossover(int64_t m_max_dp4a);

/*
 * Install measured crossovers per weight-size class: for a matrix of N*K
 * weights, the entry with the largest min_weights[i] <= N*K applies, and DP4A
 * is chosen for M <= m_max_dp4a[i]; matrices below every entry use the value
 * of iq4xs_set_crossover.  count = 0 clears the classes.  At most 16 entries,
 * min_weights[i] >= 1, 0 <= m_max_dp4a[i] <= 32768, else IQ4XS_ERR_ARG and
 * nothing changes.  Host only; the arrays are copied.  Thread-safe.
 */
int iq4xs_set_crossover_classes(const int64_t* min_weights, const int64_t* m_max_dp4a, int count);

/*
 * Install the measured warp-MMA crossover: above the DP4A range, MMA is
 * chosen for M <= m_max_mma (default 8 until a calibration sets it), TC
 * above.  Host only.  Thread-safe.  IQ4XS_ERR_ARG outside 0..32768.
 */
int iq4xs_set_mma_crossover(int64_t m_max_mma);

/*
 * The same per weight-size class, with the rules of
 * iq4xs_set_crossover_classes (at most 16 entries; count = 0 clears them).
 */
int iq4xs_set_mma_crossover_classes(const int64_t* min_weights, const int64_t* m_max_mma, int count);

/*
 * Install the measured upper threshold: iq4xs_select_path answers BASELINE
 * for M >= m_min_baseline (0 = never, the default until a calibration sets
 * it).  Host only.  Thread-safe.
 */
int iq4xs_set_baseline_threshold(int64_t m_min_baseline);

/*
 * Programmatic dependent launch (default on): each kernel lets the next one
 * in the stream start launching early, and a matmul begins streaming W before
 * the preceding kernel has finished (W is read before that wait, so W must
 * not be produced by a kernel that triggers its dependents early -- none of
 * this library's kernels writes W).  Off: every launch waits for the
 * preceding one in the usual way.  Host only; applies to later launches.
 */
int iq4xs_set_pdl(int enable);

/*
 * Read and clear the current device's error word, written by kernels whose
 * bounded waits ran out (2 s for a copy to land, 4 s for a hand-off between
 * the kernel's roles, 6 s for the final drains, so that the wait at the root
 * of a stall runs out first).  Synchronizes the current device.  Returns
 * IQ4XS_OK with *code_out = 0 when clean, IQ4XS_ERR_TIMEOUT with *code_out =
 * the code of the first wait that ran out since the last read, in the
 * tensor-core matmul:
 *   0x101 a W stage      0x102 an activation stage   0x103 a decoded unit
 *   0x104 a unit's MMAs  0x105 a free unit slot      0x106 the final drain
 *   0x107 the split-K slices of the other cluster ranks
 *   0x108 a stage of Q8_1 codes  0x109 a stage of activation scales;
 * in the warp-MMA matmul:
 *   0x10B a stage of weights and codes   0x10C a stage slot being freed.
 * (0x102 is a code stage's MMAs completing, which frees its slot.)
 */
int iq4xs_last_device_error(int* code_out);

/*
 * Bounds-checked debug build (no counterpart on the source pages; stands in
 * for a memory checker).  The same sources compiled with IQ4XS_BOUNDS_CHECK
 * defined give libiq4xs_bounds.so, with the same entry points.  There every
 * plain global load and store of every kernel, every TMA box origin and
 * every shared-memory range the kernels compute at run time is checked
 * against the extent the kernel derives from its own arguments (the sizes
 * this header states for each buffer).  A miss skips the access (a load
 * yields zero) and records code 0x200 + site in the device error word, so
 * iq4xs_last_device_error returns IQ4XS_ERR_BOUNDS.  The site number says
 * which access missed: 0x01-0x05 the quantizer (x, qs, ds, the prepared
 * operand, its span scales); 0x10-0x11 the dequantizer (W, out); 0x20-0x25
 * the dp4a matmul (W, qs, ds, y, row_offsets, an expert's rows outside y);
 * 0x30-0x39 the warp-MMA matmul (W box, W box alignment, code box, code box
 * alignment, ds, y, row_offsets, an expert's rows, shared-memory size,
 * split-K tile); 0x40-0x4A the tcgen05 matmul (W box, W box alignment,
 * code box, code box alignment, prepared operand, ds, y, span scales,
 * shared-memory size, split-K slices, grouped row_offsets or an expert's
 * rows).  A TMA box reaching past its tensor
 * is recorded but still copied (the copy unit fills the rest); a box origin
 * off the 16-byte grid is recorded and not copied, and that stage's bounded
 * wait then runs out.  Results are those of the normal build whenever
 * nothing is recorded.
 *
 * iq4xs_bounds_checked: *out = 1 in the checked build, 0 otherwise.
 * iq4xs_test_bounds_margin: checked build only (IQ4XS_ERR_ARG otherwise):
 * later launches treat the last `bytes` bytes of every global buffer as
 * outside it (copies the kernels wait for are still made), so a test can
 * see the checks fire on in-range accesses near a buffer's end without any
 * access leaving its buffer.  0 restores the exact extents.  Synchronizes
 * the current device.
 */
int iq4xs_bounds_checked(int* out);
int iq4xs_test_bounds_margin(int64_t bytes);

/*
 * Test hook for the bounded waits (no counterpart on the source pages): the
 * next tensor-core matmul launched after this call (on any thread; tcgen05
 * or warp MMA, dense or grouped) leaves W stage `stage` of every CTA
 * unissued (0-based: in units of 512 weights of each CTA's K range; in the
 * persistent grouped warp-MMA form, counted over the CTA's items one after
 * the other), so that the consumers' wait for it runs out after its 2 s
 * limit (the other roles' waits, longer, end on the abort it raises).  That
 * call's output is then undefined, every CTA still drains its copies (and,
 * on tcgen05, frees its tensor memory), and iq4xs_last_device_error
 * reports IQ4XS_ERR_TIMEOUT with code 0x101 (tcgen05) or 0x10B (warp MMA).
 * -1 disarms.  Host only.
 */
int iq4xs_test_skip_w_stage(int64_t stage);

/*
 * Test hook for the warp-MMA path's launch configuration (no counterpart on
 * the source pages): later MMA launches use rows_per_cta weight rows per CTA
 * (a multiple of 32, at most 256), k_splits CTAs per cluster along K (1..8,
 * capped at the K range's super-block pairs) and ctas_per_sm (1, or 2: the
 * half-shared-memory tiles) instead of the launch model's choice, so that
 * tests reach every configuration; a combination the activation tile cannot
 * take falls back to the nearest smaller tile height (at least 32 rows, at
 * most 128 from 24 activation rows on; two CTAs per SM only up to 64 rows at
 * 8 activation rows, 32 at 16 and 24, none above).  0 restores the model's
 * choice for that value.  Host only; applies to every thread's later
 * launches.  IQ4XS_ERR_ARG for other values.
 */
int iq4xs_test_mma_config(int64_t rows_per_cta, int64_t k_splits, int64_t ctas_per_sm);

/*
 * Measured launches of the warp-MMA path (no counterpart on the source
 * pages; written by the calibration, which times every configuration on
 * its shapes): `count` entries of six int64 each -- N, K, the activation
 * tile's rows (8, 16, 24 or 32), weight rows per CTA (a multiple of 32 up
 * to 256), CTAs per cluster along K (1..8) and CTAs per SM (1, 2).  A call
 * whose N, K and tile height match an entry launches that configuration
 * (when the tile width's configurations hold it and the K split fits K);
 * other calls use the launch model.  count = 0 clears the table; at most
 * 256 entries.  Replaces the whole table; IQ4XS_ERR_ARG (nothing
 * installed) for a value out of range.  Host only.
 */
int iq4xs_set_mma_launch_table(const int64_t* entries, int count);

/*
 * The launch the warp-MMA path makes for (M, N, K) on the current device
 * (no counterpart on the source pages; for tests and tuning): weight rows
 * per CTA, CTAs per cluster along K, and CTAs per SM, as the call would
 * take them (forced by iq4xs_test_mma_config, else from the measured
 * launch table, else from the launch model) for activation tiles of
 * min(32, M rounded up to 8) rows, for IQ4_XS weights (Q4_0 / IQ4_NL
 * launches take the same measured launch where the table holds the shape;
 * the model alone weighs their 6 % larger stages).  Host only; queries the
 * device's
 * cluster occupancy once per configuration.  IQ4XS_ERR_SHAPE unless K %
 * 512 == 0 and the sizes are in range; IQ4XS_ERR_ARG for null outputs.
 */
int iq4xs_mma_launch_config(int64_t M, int64_t N, int64_t K, int* rows_per_cta, int* k_splits, int* ctas_per_sm);

/* Static string for a status code. */
const char* iq4xs_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* IQ4XS_H */
