/*
 * coalesce.h -- C ABI of libcoalesce, a GB300 (sm_103a) library for a dense
 * GEMM with a fused bias + activation epilogue, and for a chained MLP whose
 * inter-layer activations never leave the chip.
 *
 * Plain C: pointers, 64-bit sizes and an opaque stream handle.  No C++ or
 * framework types cross this boundary.
 *
 * Common rules for every entry point
 * ----------------------------------
 * - All matrices are dense and row-major.  "Device pointer" means memory the
 *   current CUDA device can address (cudaMalloc, or a framework allocator on
 *   the same device).
 * - Ownership: the caller owns every buffer.  The library allocates no device
 *   memory: its only device state is one error word per device and the word
 *   coalesce_device_status moves it into (__device__ variables).  TMA descriptors are encoded on the host at each call and
 *   passed by value to the kernel.
 * - Asynchrony: work is enqueued on `stream` (a cudaStream_t cast to void*;
 *   NULL = the legacy default stream) and the call returns without a host
 *   synchronisation.  Outputs are valid once the stream reaches that point.
 * - Errors: every function returns COALESCE_OK (0) or a negative
 *   coalesce_status.  Argument checks happen before anything is enqueued; on an
 *   error nothing is launched and no output is touched.  There is no CPU
 *   fallback and no silent change of algorithm.
 * - Aliasing: outputs must not overlap inputs.
 * - Calls on different streams may run concurrently; the library's host state
 *   is guarded by a mutex.
 */
#ifndef COALESCE_H_
#define COALESCE_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type shared by A, B, bias and Y (GEMM) or x, W, b and out (MLP). */
typedef enum {
  COALESCE_F32 = 0,  /* IEEE fp32; GEMM only, computed with FP32 FMAs        */
  COALESCE_F16 = 1,  /* IEEE fp16 storage, fp32 accumulation, RNE downcast    */
  COALESCE_BF16 = 2  /* bfloat16 storage, fp32 accumulation, RNE downcast     */
} coalesce_dtype;

/* Epilogue activation, applied in fp32 to z = acc + bias. */
typedef enum {
  COALESCE_ACT_NONE = 0,     /* y = z                                        */
  COALESCE_ACT_RELU = 1,     /* y = max(z, 0)                                */
  COALESCE_ACT_GELU_ERF = 2, /* y = 0.5 z (1 + erf(z / sqrt 2))  (erf form)  */
  COALESCE_ACT_SOFTPLUS = 3  /* y = log(1 + e^z), beta = 1                   */
} coalesce_act;

typedef enum {
  COALESCE_OK = 0,
  COALESCE_ERR_INVALID_ARG = -1,   /* NULL required pointer, size <= 0, bad enum      */
  COALESCE_ERR_UNSUPPORTED = -2,   /* valid request this library does not implement   */
  COALESCE_ERR_MISALIGNED = -3,    /* base not 16-byte aligned / row stride not 16 B  */
  COALESCE_ERR_CUDA = -4,          /* the CUDA runtime reported an error              */
  COALESCE_ERR_DEVICE_TIMEOUT = -5 /* a kernel's bounded wait ran out (see status)    */
} coalesce_status;

/*
 * Y = act(A . B + bias)
 *
 * The fused GEMM + bias + activation of the "Coalesce" README ("Fusion study
 * (03_matmul_fused)": GEMM + bias + GELU in one kernel, equal to the matmul
 * followed by a separate elementwise kernel), with the bias-add and the
 * activation applied to the fp32 accumulator before a single store of Y (the
 * "Fuse Elementwise Ops" page, "Handle epilogue fusion into GEMM/conv").
 *
 *   M, N, K  sizes, each >= 1 (at most 2^31 - 1).
 *   dtype    coalesce_dtype of A, B, bias and Y.
 *   A        device pointer, [M, K] row-major.
 *   B        device pointer, [K, N] row-major.
 *   bias     device pointer to bias[N], broadcast over the M rows; NULL = 0.
 *   Y        device pointer, [M, N] row-major, written exactly once per element.
 *   act      coalesce_act.
 *   stream   cudaStream_t as void*, may be NULL.
 *
 * Paths: fp16/bf16 run on the tcgen05 tensor cores (TMA-fed operands, fp32
 * accumulators in tensor memory, fused epilogue); fp32 runs on a
 * register-tiled FFMA kernel (FP32-exact products, fp32 accumulation).
 * Alignment: A, B, bias and Y 16-byte aligned; row strides a multiple of
 * 16 bytes, i.e. K and N multiples of 8 (16-bit types) or 4 (fp32).
 * Returns COALESCE_OK, or INVALID_ARG / MISALIGNED / UNSUPPORTED / CUDA.
 */
int coalesce_gemm_bias_act(int64_t M, int64_t N, int64_t K, int dtype,
                           const void* A, const void* B, const void* bias,
                           void* Y, int act, void* stream);

/*
 * Y = act(Y + bias), in place, over a row-major [M, N] matrix.
 *
 * The separate elementwise pass of the UNFUSED sequence that the "Coalesce"
 * README's "Fusion study (03_matmul_fused)" compares the fused kernel with:
 * coalesce_gemm_bias_act(..., bias = NULL, act = NONE) followed by this call
 * computes what one fused coalesce_gemm_bias_act call computes, with Y making
 * one extra round trip through memory.  For fp32 the two orders give the same
 * bits; for fp16/bf16 the unfused order rounds the accumulator to the storage
 * type before the bias is added.  Used to measure what fusion saves.
 *
 *   M, N   sizes, >= 1; dtype a coalesce_dtype; Y device pointer [M, N];
 *   bias   device pointer to bias[N] or NULL (= 0); act a coalesce_act.
 * Alignment: Y and bias 16-byte aligned, N * sizeof(dtype) a multiple of 16.
 */
int coalesce_bias_act(int64_t M, int64_t N, int dtype, void* Y, const void* bias,
                      int act, void* stream);

/* Flags of coalesce_gemm_ex. */
typedef enum {
  COALESCE_GEMM_TRANS_A = 1,   /* A is given as At[K, M] row-major (A = At^T)  */
  COALESCE_GEMM_TRANS_B = 2,   /* B is given as Bt[N, K] row-major (B = Bt^T)  */
  COALESCE_GEMM_ACCUM_F32 = 4, /* Y is fp32 [M, N] and Y += A.B               */
  COALESCE_GEMM_DACT = 8       /* Y = (A.B) * act'(aux), aux[M, N] = act(z)  */
} coalesce_gemm_flags;

/*
 * The GEMM of coalesce_gemm_bias_act with transposed operands and two more
 * epilogues, for the MLP's backward pass (the "MLP Megakernel" README, "Key
 * ideas": above 32K rows the weight gradients are GEMMs interleaved with the
 * data-gradient computation).  fp16/bf16 operands, fp32 accumulation on the
 * tensor cores.
 *
 *   flags = 0           exactly coalesce_gemm_bias_act (aux must be NULL).
 *   TRANS_A / TRANS_B   operand layouts as above; combinable with any mode.
 *   ACCUM_F32           Y (fp32, [M, N]) += A.B; bias must be NULL and act
 *                       NONE.  The K range is split over all SMs and every
 *                       partial tile is added atomically, so the order of the
 *                       additions (and the last bits) may vary between calls.
 *                       The caller initialises Y (zero it for Y = A.B).
 *   DACT                Y (dtype, [M, N]) = (A.B) * act'(aux) where aux holds
 *                       the activation's OUTPUT h = act(z): softplus' =
 *                       1 - e^-h, ReLU' = [h > 0], NONE' = 1 (GELU returns
 *                       COALESCE_ERR_UNSUPPORTED: its derivative does not
 *                       follow from its output).  bias must be NULL.  Y may
 *                       be aux itself (in place), but must not overlap it
 *                       partly.
 *
 * Alignment: 16-byte pointers and row strides (A's row length K, or M with
 * TRANS_A; B's N, or K with TRANS_B; Y's N) multiples of 16 bytes.  Errors as
 * for coalesce_gemm_bias_act; COALESCE_F32 with any flag is UNSUPPORTED.
 */
int coalesce_gemm_ex(int64_t M, int64_t N, int64_t K, int dtype, unsigned flags,
                     const void* A, const void* B, const void* bias,
                     const void* aux, void* Y, int act, void* stream);

/*
 * out = h_{L-1} . W_L + b_L,  h_0 = x,  h_l = act(h_{l-1} . W_l + b_l)
 *
 * The chained MLP of the "MLP Megakernel" README ("Architecture":
 * out = softplus(softplus(x @ W1) @ W2) @ W3 and its 5-layer form; "Key
 * ideas": one persistent kernel, intermediates never reach global memory,
 * fp32 accumulation with 16-bit tensor-core operands).  Each layer adds its
 * bias; the last layer has a bias and no activation.
 *
 *   rows     number of rows, >= 1 (< 2^31).
 *   D        input width; H hidden width; O output width (the last layer's);
 *            each a multiple of 8 in [8, 256].  1 <= L <= 8 layers.  Widths
 *            that are not multiples of 64 run as if padded with zeros to the
 *            next multiple of 64 (a width of 72 costs what 128 does): the
 *            padding never reaches memory, and the results equal those of
 *            the unpadded chain.
 *   dtype    COALESCE_F16 or COALESCE_BF16: the type of x, every W_l and b_l,
 *            and out.  Accumulation is fp32; each intermediate h_l is rounded
 *            to dtype on chip to feed the next layer's tensor-core MMA.
 *            COALESCE_F32 returns COALESCE_ERR_UNSUPPORTED.
 *   x        device pointer, [rows, D] row-major.
 *   W        HOST array of L device pointers, each row-major in "x @ W"
 *            ([in, out]) form: W[0] is [D, H] (or [D, O] when L = 1), W[l] is
 *            [H, H] for 0 < l < L-1, W[L-1] is [H, O].
 *   b        HOST array of L device pointers to b_l (H elements, O for the
 *            last layer; an entry may be NULL = zero), or NULL for all-zero
 *            biases.
 *   out      device pointer, [rows, O] row-major; must not overlap x.
 *   act      activation between layers (coalesce_act; the workloads use
 *            COALESCE_ACT_SOFTPLUS).  With fp16, softplus is evaluated on
 *            packed fp16 pairs (max error 2e-3 + 2^-10 |y| per value against
 *            the exact function); every other case is evaluated in fp32.
 *   stream   cudaStream_t as void*, may be NULL.
 *
 * Weights of up to 160 KiB in all (2 bytes x the sum over layers of in x
 * out, with the widths rounded up to 64) stay in shared memory for the whole call when the ring of row tiles
 * fits beside them; otherwise they are streamed from L2 in 64-row chunks,
 * every row tile's intermediates still on chip.
 * Widths above 256, or L > 8, return COALESCE_ERR_UNSUPPORTED.
 * Alignment: every pointer 16-byte aligned and every width a multiple of 8
 * (COALESCE_ERR_MISALIGNED).
 */
int coalesce_mlp_fused_ex(int64_t rows, int64_t D, int64_t H, int64_t O, int L,
                          int dtype, const void* x, const void* const* W,
                          const void* const* b, void* out, int act,
                          void* stream);

/*
 * The pages' form of the chained MLP: coalesce_mlp_fused_ex with O = H and
 * dtype = COALESCE_F16 (the README's fp16 megakernel).  out is [rows, H].
 */
int coalesce_mlp_fused(int64_t rows, int64_t D, int64_t H, int L,
                       const void* x, const void* const* W,
                       const void* const* b, void* out, int act, void* stream);

/*
 * Training side of the chained MLP (the "MLP Megakernel" README: "Full
 * training" forward + backward; "Key ideas": activations kept for the
 * backward's derivative, weight gradients as GEMMs above 32K rows).  Shapes
 * as for coalesce_mlp_fused_ex (x [rows, D], W_0 [D, H] ... W_{L-1} [H, O],
 * b_l of the layer's output width), but any D, H, O that are multiples of 8,
 * and dtype COALESCE_F16 or COALESCE_BF16; act NONE, RELU or SOFTPLUS.
 *
 * coalesce_mlp_forward_train computes out like the fused MLP, layer by layer,
 * and stores every intermediate activation:
 *   h        HOST array of L-1 device pointers; h[l] ([rows, H], dtype)
 *            receives act(h_{l} W_l + b_l), the input of layer l+1.
 *
 * coalesce_mlp_backward, given dout = dLoss/dout [rows, O]:
 *   dW       HOST array of L device pointers to fp32 [in_l, out_l]: written
 *            (dLoss/dW_l, summed over rows).
 *   db       HOST array of L device pointers to fp32 [out_l] (entries may be
 *            NULL), or NULL: dLoss/db_l.
 *   dx       device pointer [rows, D] (dtype) for dLoss/dx, or NULL.
 *   h        the activations of the forward pass.  CONSUMED: their contents
 *            are unspecified afterwards (the layer-by-layer form overwrites
 *            them with the gradients w.r.t. the pre-activations).
 * Where D and H are at most 128, O at most 256 and the weight gradients fit
 * the 512 tensor-memory columns beside one 128 x max(D, H) accumulator (sum
 * over layers of out_l, plus max(D, H)), every width counted rounded up to a
 * multiple of 64, the whole backward is one fused kernel: each SM keeps its share of every dW_l
 * on chip across its row tiles, and dout, h and x are each read once.  Other
 * shapes run layer by layer on the GEMM kernels.
 * Sums over rows are atomic, so their rounding may differ between calls.
 * Each layer's derivative comes from the stored activation (softplus' =
 * 1 - e^-h), evaluated in fp32; the data gradients are rounded to dtype.
 * Errors as for coalesce_mlp_fused_ex; the library allocates nothing.
 */
int coalesce_mlp_forward_train(int64_t rows, int64_t D, int64_t H, int64_t O,
                               int L, int dtype, const void* x,
                               const void* const* W, const void* const* b,
                               void* const* h, void* out, int act,
                               void* stream);

int coalesce_mlp_backward(int64_t rows, int64_t D, int64_t H, int64_t O, int L,
                          int dtype, const void* x, const void* const* W,
                          void* const* h, const void* dout, void* dx,
                          float* const* dW, float* const* db, int act,
                          void* stream);

/*
 * Synchronise `stream`, then report and clear the device error word that
 * the kernels' bounded waits set when a wait runs out.  Returns COALESCE_OK,
 * COALESCE_ERR_DEVICE_TIMEOUT, or COALESCE_ERR_CUDA if the stream itself failed.
 *
 * The error word is per DEVICE, not per stream: a timeout raised by a kernel
 * on another stream of the same device is reported by whichever status call
 * reads the word first.  The word is read and cleared in one atomic exchange
 * (a one-thread kernel on `stream`), so no code is lost between the read and
 * the clear; two status calls that run at the same time on different streams
 * share one snapshot word, and one of them may report the other's result.
 */
int coalesce_device_status(void* stream);

/*
 * Measurement aid (not part of the computation): the FP32 FMA rate of this
 * device, against which the FP32 GEMM's roofline fraction is reported.
 * Enqueues one kernel on `stream` with 4 blocks of 256 threads per SM; every
 * thread runs 16 independent fp32 FMA chains for `iters` steps each (iters a
 * positive multiple of 8, at most 2^40), with no memory traffic in the loop.
 * *flop (host pointer) receives the number of floating-point operations the
 * kernel performs (2 per FMA); the caller times the kernel with events on
 * `stream`.  `sink` is a device pointer to one float that the kernel may
 * write (it is never read).  Returns COALESCE_OK, INVALID_ARG or CUDA.
 */
int coalesce_measure_ffma(int64_t iters, float* sink, double* flop, void* stream);

/*
 * Failure-detection self-test.  Launches one small kernel that waits, with the
 * same bounded mbarrier wait every kernel of this library uses, on a barrier
 * that nothing ever arrives on.  After limit_ns nanoseconds (1 us .. 10 s) the
 * wait gives up, records the timeout in the device error word and the kernel
 * returns normally; a following coalesce_device_status(stream) then reports
 * COALESCE_ERR_DEVICE_TIMEOUT and clears the word.  No fault, trap or hang is
 * involved and the CUDA context stays usable.  Returns COALESCE_OK once the
 * kernel is enqueued, INVALID_ARG for a limit out of range, or CUDA.
 */
int coalesce_selftest_wait_timeout(uint64_t limit_ns, void* stream);

/* Static, human-readable text for a status code (never NULL). */
const char* coalesce_status_string(int status);

/* Text describing the last failed call of this thread: a rejected argument,
 * an unsupported request or a CUDA error (never NULL; per thread). */
const char* coalesce_last_error(void);

/* Forget the per-device set-up (SM count, error-word address) so the next
 * call redoes it, e.g. after cudaDeviceReset.  Optional. */
void coalesce_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* COALESCE_H_ */
