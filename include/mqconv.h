/*
 * mqconv.h -- C ABI of the MicroQonv quantize-once convolution library (sm_103a).
 *
 * The method (paper "MicroQonv: Reshaping Convolution Tensors for Efficient
 * Microscaling in Training and Inference", Facq, Ben Ali, Sentieys):
 * every convolution tensor -- activations X, weights W, output gradients
 * G_Y -- is quantized exactly once into square 8x8 microscaling blocks stored
 * channel-batch-first, and the three GEMMs of a training step run on those
 * packed blocks with an on-chip (implicit) im2col, so no im2col matrix and no
 * second quantization ever reaches device memory.
 *
 * Conventions shared by every entry point
 *   - All pointers documented as "device" are CUDA device pointers owned by the
 *     caller.  The library never allocates or frees memory.
 *   - Every call is asynchronous on `stream` (NULL = legacy default stream).
 *     Argument errors are reported synchronously by the return value and
 *     nothing is launched.  Errors found on the device (non-finite input, a
 *     bounded wait that expired) are OR-ed into a device status word that
 *     mqconv_device_status() reads and clears.
 *   - Batch N and every channel count must be multiples of 8 (the block edge);
 *     callers zero-pad otherwise.  All device pointers must be 16-byte aligned.
 *   - Element formats (codes): E2M1 (NVFP4), E2M3 (6-bit), E4M3 (8-bit).  Block
 *     scales are always E4M3; the per-tensor scale is one fp32.
 *
 * Packed tensor layout (mq_packed)
 *   Activations (role ACT) and gradients (role GRAD) with dims (N, C, H, W):
 *     blocks ordered [H][W][N/8][C/8]; inside a block element i = 8*n + c
 *     (channel fastest).  So every spatial position holds one contiguous run
 *     covering all its channels and all batch elements, the channel-batch-first
 *     storage of MicroQonv §IV-A, Fig. 3.
 *   Weights (role WEIGHT) with dims (Cout, Cin, Kh, Kw):
 *     blocks ordered [Kh][Kw][Cout/8][Cin/8]; element i = 8*co + ci (§IV-B:
 *     weights quantized along C_in and C_out).
 *   Code payload per block: E2M1 32 bytes (element i in byte i/2, low nibble
 *     for even i); E2M3 48 bytes (little-endian bit stream, element i at bits
 *     6i..6i+5); E4M3 64 bytes (byte i).  Scales: one E4M3 byte per block, in
 *     block order, in a separate array.
 *
 * Quantization (MicroQonv §II-D, §III-A, §IV-B)
 *   T_scale = fl32(amax / (maxB_ef * 448)), maxB_ef = 6 (E2M1), 7.5 (E2M3),
 *   448 (E4M3 codes); B_scale = RN_E4M3(amax_block / (maxB_ef * T_scale));
 *   code = RN(x / (B_scale * T_scale)).  Both roundings act on the exact real
 *   quotient, ties to even, saturating at the largest finite value.  A block
 *   whose scale rounds to zero (or T_scale = 0) gets magnitude-0 codes.  The
 *   sign bit of each code is the sign bit of its input.
 */
#ifndef MQCONV_H
#define MQCONV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MQCONV_ABI_VERSION 3

/* cudaStream_t without including CUDA headers */
typedef struct CUstream_st *mq_stream;

typedef enum {
  MQ_OK = 0,
  MQ_ERR_INVALID_ARG = 1,   /* null pointer, bad enum, inconsistent shapes */
  MQ_ERR_UNSUPPORTED = 2,   /* N or a channel count not a multiple of 8, too large */
  MQ_ERR_ALIGNMENT = 3,     /* a device pointer not 16-byte aligned */
  MQ_ERR_NONFINITE = 4,     /* device: Inf or NaN in a quantized input */
  MQ_ERR_TIMEOUT = 5,       /* device: a bounded wait inside a kernel expired */
  MQ_ERR_CUDA = 6,          /* a CUDA runtime call failed (launch error) */
  MQ_ERR_WORKSPACE = 7      /* workspace null or smaller than required */
} mq_status;

typedef enum { MQ_FMT_E2M1 = 4, MQ_FMT_E2M3 = 6, MQ_FMT_E4M3 = 8 } mq_format;
typedef enum { MQ_ROLE_ACT = 0, MQ_ROLE_WEIGHT = 1, MQ_ROLE_GRAD = 2 } mq_role;
typedef enum { MQ_DT_F32 = 0, MQ_DT_BF16 = 1 } mq_dtype;
typedef enum { MQ_LAYOUT_NCHW = 0, MQ_LAYOUT_HWCN = 1, MQ_LAYOUT_OIHW = 2 } mq_layout;

/* Rounding of the element codes (MicroQonv §III-A: Round is round-to-nearest
 * or stochastic; the paper rounds gradients stochastically).  Block scales
 * are always round-to-nearest (CastE4M3).  Stochastic rounding, as read
 * here:  q = fl32(|x| / fl32(B_scale * T_scale)) (IEEE fp32 division);
 * q >= maxB_ef gives the largest code; otherwise lo <= q < hi are the grid
 * values around q and the code is hi when r < 2^24 (q - lo) / (hi - lo),
 * else lo, with r the top 24 bits of word e % 4 of Philox4x32-10 (Salmon et
 * al., SC 2011) under key (seed low, seed high) at counter (e / 4 low,
 * e / 4 high, 0, 0), e = block * 64 + in-block index in packed order.  Every
 * step is exact, so a seed determines the codes bit for bit; the expected
 * code value is q to within 2^-24 of the grid spacing. */
typedef enum { MQ_ROUND_RN = 0, MQ_ROUND_SR = 1 } mq_rounding;

/* A tensor quantized once into packed 8x8 blocks (layout above). */
typedef struct {
  int32_t fmt;       /* mq_format of the codes */
  int32_t role;      /* mq_role */
  int64_t dims[4];   /* ACT/GRAD: (N, C, H, W); WEIGHT: (Cout, Cin, Kh, Kw) */
  void *codes;       /* device, mqconv_packed_code_bytes() bytes */
  uint8_t *scales;   /* device, mqconv_packed_scale_bytes() bytes */
  float *s_t;        /* device, one float: T_scale */
  void *decoded;     /* WEIGHT only, optional (else NULL): device fp16 copy of the
                        block values, mqconv_weight_decoded_bytes() bytes (below) */
} mq_packed;

/* Decoded weight copy (optional; role WEIGHT only).
 *   Blocks in the packed order [Kh][Kw][Cout/8][Cin/8], 128 bytes each: row r
 *   of a block (output channel 8*cog + r) holds eight fp16 values, input
 *   channels 8*cig .. 8*cig+7, each code * B_scale -- times 1/4 for E4M3
 *   codes, whose products can exceed the fp16 range -- without T_scale, which
 *   the convolutions apply in fp32.  Every value is exact in fp16.
 *   The convolutions decode the packed weight blocks on chip once per output
 *   tile; a small, deep layer has few output positions per weight block, so
 *   every tile repeats the same decode.  With the copy, mqconv_fwd,
 *   mqconv_dgrad and mqconv_dgrad_requant copy the weight operand straight
 *   into shared memory instead (same results, bit for bit).  It is a cache of
 *   codes and scales: mqconv_quantize_cbf rewrites it with them, and a caller
 *   that changes codes or scales otherwise calls mqconv_weight_decode.
 *   Must be 16-byte aligned (MQ_ERR_ALIGNMENT); non-NULL on a tensor of
 *   another role is MQ_ERR_INVALID_ARG. */

/* One convolution layer: cross-correlation, zero padding, square stride/pad.
 * Ho = (H + 2 pad - Kh) / stride + 1, Wo likewise (paperlayer summary of the
 * paper, §II-A "Forward Pass", generalised to stride and padding as §II-A
 * states the method allows). */
typedef struct {
  int64_t N, Cin, H, W, Cout, Kh, Kw, stride, pad;
} mq_conv_desc;

/* Optional fused epilogue of mqconv_fwd: requantize Y straight from the
 * accumulators into the next layer's activation blocks (role ACT, dims
 * (N, Cout, Ho, Wo)).  A global amax of Y cannot exist before Y does, so
 * T_scale is built from a caller-supplied statistic (e.g. the previous step's
 * amax, the Hindsight scheme the paper uses in §VII); the true amax of Y is
 * written to amax_out for the next step. */
typedef struct {
  int32_t fmt;            /* mq_format of the requantized Y */
  const float *amax_in;   /* device, 1 float: statistic T_scale is built from */
  const mq_packed *out;   /* packed Y (its fmt/role/dims must match) */
  float *amax_out;        /* device, 1 float or NULL: receives max|Y| */
  int32_t rounding;       /* mq_rounding of the element codes (MQ_ROUND_RN: 0) */
  uint64_t sr_seed;       /* Philox key of MQ_ROUND_SR; ignored otherwise */
} mq_requant;

int32_t mqconv_abi_version(void);
const char *mqconv_status_string(mq_status status);

/* Bytes of the code payload / scale array of a packed tensor.  dims as in
 * mq_packed.  Returns 0 for invalid arguments. */
size_t mqconv_packed_code_bytes(int32_t fmt, const int64_t dims[4]);
size_t mqconv_packed_scale_bytes(const int64_t dims[4]);
/* Bytes of the decoded weight copy of a packed weight tensor with dims
 * (Cout, Cin, Kh, Kw): 128 per block.  Returns 0 for invalid arguments. */
size_t mqconv_weight_decoded_bytes(const int64_t dims[4]);

/* (Re)write wq->decoded from wq's codes and scales (see "Decoded weight
 * copy").  wq: role WEIGHT, decoded non-NULL. */
mq_status mqconv_weight_decode(const mq_packed *wq, mq_stream stream);

/*
 * Quantize one dense tensor once (MicroQonv §III-A, §IV-B).
 *   src      device, fp32 or bf16 (dtype), dense in `layout`:
 *            ACT/GRAD: NCHW or HWCN ([H][W][C][N]); WEIGHT: OIHW.
 *   dst      packed output; dst->role, dst->fmt, dst->dims say what to produce.
 *   amax_in  device or NULL.  NULL: exact two-pass mode, T_scale from the
 *            tensor's own amax (amax_out must then be non-NULL; it receives
 *            that amax).  Non-NULL: one pass, T_scale from *amax_in; amax_out,
 *            if non-NULL, receives the measured amax.
 *   A WEIGHT dst with a decoded copy gets it rewritten after the codes.
 *   Non-finite input sets MQ_ERR_NONFINITE in the device status word (the
 *   output is then unspecified).
 */
mq_status mqconv_quantize_cbf(const void *src, int32_t dtype, int32_t layout, const mq_packed *dst,
                              const float *amax_in, float *amax_out, mq_stream stream);

/*
 * mqconv_quantize_cbf with stochastically rounded element codes (mq_rounding
 * above; MicroQonv §III-A, the paper's rounding of gradients), Philox key
 * `seed`.  T_scale, block scales, layouts, statistic modes and errors as for
 * mqconv_quantize_cbf.
 */
mq_status mqconv_quantize_cbf_sr(const void *src, int32_t dtype, int32_t layout, const mq_packed *dst,
                                 const float *amax_in, float *amax_out, uint64_t seed, mq_stream stream);

/*
 * Forward convolution on packed operands: Y = W_f * X' with X' the on-chip
 * channel-batch-first im2col of Xq (MicroQonv §IV-A:
 * Y_{fCout,N} = W_{fCout,Cin} . X'_{Cin,N}).
 *   xq  packed activations, role ACT, dims (N, Cin, H, W).
 *   wq  packed weights, role WEIGHT, dims (Cout, Cin, Kh, Kw); with a
 *       decoded copy, that copy is the weight operand (same results).
 *   y   device fp32 [Ho][Wo][Cout][N] (HWCN), or NULL when rq is given.
 *   rq  NULL, or the fused requantizing epilogue (see mq_requant).
 */
mq_status mqconv_fwd(const mq_conv_desc *desc, const mq_packed *xq, const mq_packed *wq, float *y,
                     const mq_requant *rq, mq_stream stream);

/*
 * Data gradient: G_X = col2im(W_f^T * G_Y) computed directly as the adjoint
 * convolution, i.e. G_Y correlated with the spatially flipped, channel-
 * transposed kernels (paperlayer summary §II-A "Backward Pass"; MicroQonv §IV-A:
 * G_X'_{Cin,N} = W^T_{fCout,Cin} . G_Y_{fCout,N}).
 *   wq   packed weights, role WEIGHT, dims (Cout, Cin, Kh, Kw); with a
 *        decoded copy, that copy is the weight operand (same results).
 *   dyq  packed output gradient, role GRAD, dims (N, Cout, Ho, Wo).
 *   dx   device fp32 [H][W][Cin][N] (HWCN).
 */
mq_status mqconv_dgrad(const mq_conv_desc *desc, const mq_packed *wq, const mq_packed *dyq, float *dx,
                       mq_stream stream);

/*
 * Data gradient with the fused requantizing epilogue: dX goes from the
 * accumulators straight into packed blocks of role GRAD, dims (N, Cin, H, W)
 * -- the output gradient G_Y of the layer below, quantized once (MicroQonv
 * §IV-B: gradients in (N, C) square blocks) -- without an fp32 round trip
 * through device memory.  As for the forward epilogue (mq_requant), T_scale
 * comes from the caller's statistic rq->amax_in (e.g. the previous step's
 * amax of dX) and the true amax is written to rq->amax_out.
 *   wq, dyq  as for mqconv_dgrad.
 *   dx       device fp32 [H][W][Cin][N], or NULL (only the packed result).
 *   rq       required; rq->out has role MQ_ROLE_GRAD.
 */
mq_status mqconv_dgrad_requant(const mq_conv_desc *desc, const mq_packed *wq, const mq_packed *dyq, float *dx,
                               const mq_requant *rq, mq_stream stream);

/*
 * Weight gradient: G_W = G_Y * X'^T (MicroQonv §IV-A: G_W_{fCout,Cin} =
 * G_Y_{fCout,N} . X'^T_{Cin,N}), reduced over (Ho, Wo, N).
 *   dyq  packed output gradient, role GRAD, dims (N, Cout, Ho, Wo).
 *   xq   packed activations, role ACT, dims (N, Cin, H, W).
 *   dw   device fp32 [Cout][Cin][Kh][Kw] (OIHW).
 *   workspace / ws_bytes  device scratch of at least
 *        mqconv_wgrad_workspace_bytes(desc) bytes for the split-K partial
 *        sums (reduced in a fixed order: results are deterministic).
 */
size_t mqconv_wgrad_workspace_bytes(const mq_conv_desc *desc);
mq_status mqconv_wgrad(const mq_conv_desc *desc, const mq_packed *dyq, const mq_packed *xq, float *dw,
                       void *workspace, size_t ws_bytes, mq_stream stream);

/*
 * Weight gradient that allocates nothing (this entry point has no counterpart
 * in the paper; it exists for callers of this library).
 *
 * Same result as mqconv_wgrad, up to the fp32 summation order of the split-K
 * partial sums, but without the workspace argument.  It is meant for callers
 * that cannot hand the library extra device memory: runtimes that own a fixed
 * device-memory budget and pass in only the inputs and outputs, allocators
 * that must not be bypassed or fragmented by side allocations, and code that
 * cannot accept the implicit device synchronisation a cudaMalloc/cudaFree may
 * bring.  The partial sums live in a built-in device array of
 * MQCONV_WGRAD_NOALLOC_SCRATCH_BYTES bytes that every GPU loading the library
 * reserves until the process exits; no cudaMalloc, cudaFree or other
 * allocating routine is called.
 *   dyq, xq, dw   as for mqconv_wgrad.
 *   Returns MQ_ERR_WORKSPACE, without launching, when one set of partial sums
 *   (Cout * Kh * Kw * Cin fp32) does not fit in the built-in array; when
 *   several sets are needed the reduction is split into fewer, longer chunks
 *   to fit.
 *   The first call on a device looks up the array's device address with that
 *   device current (cudaGetSymbolAddress); make that first call before any
 *   stream capture.  Every call overwrites the partial sums it reads, so no
 *   clearing is needed, but all calls share the one array: calls whose work
 *   overlaps on the GPU (e.g. on two streams at once) race and give wrong dW.
 */
#define MQCONV_WGRAD_NOALLOC_SCRATCH_BYTES (16u << 20)
mq_status mqconv_wgrad_noalloc(const mq_conv_desc *desc, const mq_packed *dyq, const mq_packed *xq, float *dw,
                               mq_stream stream);

/* Synchronize `stream`, copy the device status word (an OR of mq_status bit
 * flags 1 << MQ_ERR_*) to *host_status, and clear it. */
mq_status mqconv_device_status(mq_stream stream, int32_t *host_status);

/*
 * Test support for the failure detection (not part of the method; the paper
 * describes no runtime).  Every wait inside the convolution kernels is
 * bounded (2 s): when one expires, the kernel ORs 1 << MQ_ERR_TIMEOUT into
 * the device status word, lets the copies and MMAs it already issued land,
 * frees its tensor memory and returns, so the CUDA context stays usable and
 * the host learns of it from mqconv_device_status().
 *   what  MQ_INJECT_NONE, or MQ_INJECT_WITHHOLD_ACC_RELEASE: in every later
 *         launch of the halo forward / data-gradient kernel, the barrier of
 *         CTA 0's first accumulator slot expects one release more than its
 *         epilogue warps give, so the MMA issuer's wait to reuse that slot
 *         (on a second tile of CTA 0) can only expire.  Nothing traps or
 *         faults; only a plain barrier arrival is withheld.
 * The setting is process-wide and applies until changed; MQ_ERR_INVALID_ARG
 * for an unknown value.  Call with MQ_INJECT_NONE to restore normal
 * operation.
 */
#define MQ_INJECT_NONE 0
#define MQ_INJECT_WITHHOLD_ACC_RELEASE 1
mq_status mqconv_test_fault_inject(int32_t what);

#ifdef __cplusplus
}
#endif
#endif /* MQCONV_H */
