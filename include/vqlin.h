/*
 * vqlin.h -- C ABI of the quantized linear projection library (libvqlin.so).
 *
 * The operations are the quantized linear projections that post-training
 * quantization of vision-language-action models runs on:
 *   - W4A4: online block-Hadamard rotation of the activations, dynamic
 *     per-token symmetric int4 activations, per-output-channel symmetric int4
 *     round-to-nearest (RTN) weights, native integer GEMM and a scale
 *     epilogue ("FoldQuantVLA: Native Low-Bit Quantization of
 *     Vision-Language-Action Models via Consistent Folding", abstract:
 *     block Hadamard transforms with dynamic per-token quantization, W4A4
 *     executed natively in integers);
 *   - W8A8: the same structure at eight bits, for the attention-output and
 *     feed-forward down projections kept at eight bits (same abstract);
 *   - W4A16: group-wise int4 weights dequantised inside the GEMM/GEMV, for the
 *     memory-bound action expert ("LoopQ: Fair, Closed-Loop Evaluation of
 *     Quantized Vision-Language-Action Models", abstract: the action expert
 *     is memory-bound, 63% of GPU time);
 *   - the 16-bit baseline projection (bf16 in, fp32 accumulate, bf16 out).
 * The rotation uses a normalised Hadamard matrix applied block-wise over
 * channels ("Omega-QVLA" technical summary, section "Rotazione Composita
 * SVD.Hadamard": normalised H, block-wise implementation).
 *
 * Conventions for every entry point
 *   - Tensor pointers are DEVICE pointers, allocated and owned by the
 *     caller, 16-byte aligned.  bf16 tensors are passed as uint16_t bit
 *     patterns.  All matrices are row-major: X [M, K], W [N, K] (nn.Linear
 *     layout), Y [M, N].
 *   - Symmetric codes lie in [-qmax, qmax] (qmax = 7 or 127) and are stored
 *     sign-magnitude.  Weight codes: an int4 code c is the nibble
 *     (c < 0) << 3 | |c|, two per byte with the even channel k in the low
 *     nibble ([N, K/2] bytes); an int8 code is the byte (c < 0) << 7 | |c|
 *     ([N, K]).  Activation codes are stored in the tensor-core operand
 *     encoding the GEMM consumes unchanged: an int4 code is the byte
 *     (c < 0) << 7 | |c| ([M, K] bytes, the e4m3 bits of c * 2^-9); an int8
 *     code is the 16-bit word (c < 0) << 15 | |c| ([M, K] uint16, the f16
 *     bits of c * 2^-24).  Asymmetric uint4 weight codes (W4A16) hold 8
 *     channels per little-endian 32-bit word: channel 2i in bits [4i, 4i+4),
 *     channel 2i+1 in bits [16+4i, 16+4i+4).  (The pages fix no packing;
 *     these layouts turn into exact tensor-core operands with a few bit
 *     operations.)
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     are asynchronous on it.  Argument checks happen on the host before any
 *     launch; a call that returns an error has launched nothing.
 *   - No entry point allocates device memory or falls back to the CPU.  An
 *     unsupported shape returns VQLIN_ERR_UNSUPPORTED_SHAPE.
 *   - Errors found on the device (a bounded wait that ran out) are recorded
 *     in a per-device status word read by vqlin_get_last_device_error().
 */
#ifndef VQLIN_H
#define VQLIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  VQLIN_OK = 0,
  VQLIN_ERR_INVALID_ARG = 1,       /* null pointer, bad enum value, negative size */
  VQLIN_ERR_UNSUPPORTED_SHAPE = 2, /* K not a multiple of the block/group, too large */
  VQLIN_ERR_MISALIGNED = 3,        /* a pointer is not 16-byte aligned */
  VQLIN_ERR_CUDA = 4,              /* a CUDA runtime or cuBLAS call failed */
  VQLIN_ERR_TIMEOUT = 5,           /* a bounded device-side wait ran out */
  VQLIN_ERR_DEVICE_ASSERT = 6      /* a device-side consistency check failed */
} vqlin_status;

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int vqlin_version(void);

/* Static, human-readable name of a status code. */
const char* vqlin_status_string(vqlin_status status);

/* Detail text of the last failing call on this host thread ("" if none).
 * The string stays valid until the next failing call on the thread. */
const char* vqlin_last_error_message(void);

/* Synchronises `stream`, then reads and clears the status word of the
 * current device.  Returns VQLIN_OK if no kernel recorded an error. */
vqlin_status vqlin_get_last_device_error(void* stream);

/*
 * Library state of the current device, made ahead of the first call: the
 * device status word's address and the cuBLASLt handle and 64 MiB workspace of
 * the bf16 baseline (vqlin_linear_bf16_ref).  Optional -- every call creates
 * what it needs on first use -- but calling it before capturing a CUDA graph
 * or timing keeps that one-time work out of them.  Returns VQLIN_ERR_CUDA if
 * there is no usable device.  The pages define no such call.
 */
vqlin_status vqlin_init(void);

/*
 * Releases what vqlin_init (or first use) created on every device: waits for
 * each such device's queued work, then destroys its cuBLASLt handle and frees
 * its workspace.  Device memory the caller owns is untouched.  A later call
 * creates the state again.  Must not run concurrently with other calls.
 */
vqlin_status vqlin_shutdown(void);

/*
 * Number of the library's own kernels launched (enqueued on a stream or
 * recorded into a CUDA graph being captured) since the library was loaded,
 * over all devices and threads.  A graph replay launches nothing through the
 * library and is not counted.  count: host pointer; VQLIN_ERR_INVALID_ARG if
 * null.  The pages define no such call.
 */
vqlin_status vqlin_kernel_launch_count(unsigned long long* count);

/*
 * Offline weight preparation: round-to-nearest quantization of W [N, K] bf16.
 * ("plain RTN", LoopQ abstract; rotation folded into the weights,
 * FoldQuantVLA abstract and Omega-QVLA "Rotazione Hadamard".)
 *
 * symmetric = 1 (bits 4 or 8, group_size 0):
 *   W~ = W . blockdiag(H_b / sqrt(b)) if hadamard_block b in {64, 128}
 *   (computed in float64, rounded once to float32), else W~ = W;
 *   s[n] = max_k |W~[n,k]| / qmax  (float32, qmax = 7 or 127);
 *   q = clamp(rint(W~ / s), -qmax, qmax), round half to even; a zero row
 *   gives s = 0 and codes 0.
 *   q_out: int4 [N, K/2] bytes or int8 [N, K]; scale_out: float [N];
 *   zero_out must be NULL.
 * symmetric = 0 (bits 4, group_size 64, 128 or 256, hadamard_block 0):
 *   per group of `group_size` consecutive channels of a row:
 *   lo = min(0, min W), hi = max(0, max W); s = (hi - lo) / 15 rounded up
 *   to bf16; z = clamp(rint(-lo / s), 0, 15); q = clamp(rint(W / s) + z, 0, 15);
 *   an all-zero group gives s = 1, z = 0.
 *   q_out: uint4 [N, K/2] bytes; scale_out, zero_out: bf16 [N, K/group_size].
 * Requires K % max(b, group_size, 32) == 0 and K <= 49152.
 */
vqlin_status vqlin_quantize_weights_rtn(const uint16_t* W, int N, int K, int bits,
                                        int symmetric, int group_size, int hadamard_block,
                                        void* q_out, void* scale_out, void* zero_out,
                                        void* stream);

/*
 * Channel scaling, the weight side (FoldQuantVLA abstract: channel scaling
 * folded consistently through the rotation, the weight rounding and native
 * integer execution): vqlin_quantize_weights_rtn, symmetric, of
 * W' = W . diag(c) -- each weight times channel_scale[k] in float64 before the
 * block rotation.  channel_scale: float [K] on the device, positive, finite
 * (c[k] = 1 everywhere gives vqlin_quantize_weights_rtn).  Pair it with
 * vqlin_act_hadamard_quant_scaled and the same c, so that x' . W'^T = x . W^T.
 */
vqlin_status vqlin_quantize_weights_rtn_scaled(const uint16_t* W, int N, int K, int bits, int hadamard_block,
                                               const float* channel_scale, void* q_out, float* scale_out,
                                               void* stream);

/*
 * Online activation kernel: block-Hadamard rotation + per-token quantization.
 * (FoldQuantVLA abstract: block Hadamard transforms with dynamic per-token
 * quantization; Omega-QVLA "Scalatura delle Attivazioni DiT per Passo":
 * per-step precomputed scales as the static alternative.)
 *
 *   x~ = x . blockdiag(H_b / sqrt(b)) (float32 fast Walsh-Hadamard transform;
 *        b = hadamard_block in {0, 64, 128}, 0 = no rotation);
 *   dynamic (static_scale == NULL): s[m] = max_k |x~[m,k]| / qmax;
 *   static: s[m] = *static_scale (ONE device float, > 0, finite);
 *   q = clamp(rint(x~ / s), -qmax, qmax), round half to even; s = 0 gives
 *   codes 0.
 * X: bf16 [M, K]; q_out: [M, K] bytes (bits 4) or [M, K] uint16 (bits 8) in
 * the activation-code encoding above; scale_out: float [M] (filled with the
 * static scale in static mode).
 * Requires K % max(b, 32) == 0 and K <= 65536.
 */
vqlin_status vqlin_act_hadamard_quant(const uint16_t* X, int M, int K, int bits,
                                      int hadamard_block, const float* static_scale,
                                      void* q_out, float* scale_out, void* stream);

/*
 * W4A4 projection: Y = bf16( (sum_k xq[m,k] * wq[n,k]) * sx[m] * sw[n] + bias[n] ).
 * The sum is exact in int32; the epilogue is float32 in that order, rounded
 * half to even to bf16.  (FoldQuantVLA abstract: native integer execution.)
 * xq: int4 activation codes [M, K] bytes; sx: float [M]; wq: int4 weight
 * codes [N, K/2]; sw: float [N];
 * bias: bf16 [N] or NULL; Y: bf16 [M, N].  Requires K % 128 == 0 and
 * K <= 65536.  Runs on the tcgen05 tensor cores (int4 codes as exact e4m3
 * operands); K may be split over a thread-block cluster, reduced on chip.
 */
vqlin_status vqlin_linear_w4a4(const uint8_t* xq, const float* sx, const uint8_t* wq,
                               const float* sw, const uint16_t* bias, uint16_t* Y,
                               int M, int N, int K, void* stream);

/*
 * W4A8 projection (QuantVLA's setting: int4 weights, int8 per-token
 * activations): Y = bf16( (sum_k xq[m,k] * wq[n,k]) * sx[m] * sw[n] + bias[n] )
 * with the int32 sum exact.  xq: int8 activation codes [M, K] uint16 (as for
 * vqlin_linear_w8a8, from vqlin_act_hadamard_quant with bits 8); wq: int4
 * weight codes [N, K/2] (as for vqlin_linear_w4a4, from
 * vqlin_quantize_weights_rtn with bits 4); the other arguments as for
 * vqlin_linear_w4a4.  Runs on the f16 tensor cores (exact subnormal operands;
 * float32 partial sums of at most 16384 channels stay below 2^24 and are added
 * up in int32).  Requires K % 64 == 0 and K <= 65536.
 */
vqlin_status vqlin_linear_w4a8(const uint16_t* xq, const float* sx, const uint8_t* wq,
                               const float* sw, const uint16_t* bias, uint16_t* Y,
                               int M, int N, int K, void* stream);

/*
 * W4A4 projection with the activations quantized on chip at a static scale
 * (Omega-QVLA "Scalatura delle Attivazioni DiT per Passo": per-step
 * precomputed activation scales; FoldQuantVLA abstract: block Hadamard
 * rotation and native integer execution).  Computes exactly what
 * vqlin_act_hadamard_quant(X, M, K, 4, hadamard_block, static_scale, xq_out, s)
 * followed by vqlin_linear_w4a4(xq_out, s, wq, sw, bias, Y, M, N, K) computes
 * (the same codes bit for bit, hence the same Y), in one kernel for up to 128
 * tokens when K < 4096 and the plan's clusters fit in one wave, otherwise as
 * the activation kernel followed by a GEMM on its codes (two launches).  The
 * one-launch kernel rotates and quantizes each activation tile once per
 * thread-block cluster, not once per CTA: the cluster's CTAs write the codes to
 * xq_out, meet at a cluster barrier and read the codes of their K range back
 * from L2.  So xq_out is both the code output and the kernel's exchange buffer.
 * X: bf16 [M, K]; static_scale: ONE device float (> 0, finite); hadamard_block
 * 64 or 128; wq, sw, bias, Y as for vqlin_linear_w4a4 (wq rotated with the same
 * block); xq_out: [M, K] bytes, caller-owned, receives the activation codes in
 * the int4 activation-code encoding (its previous contents are ignored).
 * Requires K % 128 == 0 and K <= 65536 (beyond 16384 channels: the activation
 * kernel, then the GEMM, two launches).
 */
vqlin_status vqlin_linear_w4a4_static(const uint16_t* X, const float* static_scale,
                                      int hadamard_block, const uint8_t* wq, const float* sw,
                                      const uint16_t* bias, uint16_t* Y, uint8_t* xq_out,
                                      int M, int N, int K, void* stream);

/*
 * vqlin_linear_w4a4_static with channel scaling (FoldQuantVLA abstract:
 * channel scaling combined with the block Hadamard transform): the
 * activations are divided by channel_scale[k] (IEEE float32 division of each
 * loaded value) before the rotation and static-scale quantization, on chip in
 * the one-launch kernel; wq must be quantized from W . diag(c) with the same c
 * (vqlin_quantize_weights_rtn_scaled), so that the projection stays x . W^T.
 * Computes exactly what vqlin_act_hadamard_quant_scaled(X, M, K, 4,
 * hadamard_block, channel_scale, static_scale, xq_out, s) followed by
 * vqlin_linear_w4a4 computes (same codes bit for bit, same Y).
 * channel_scale: float [K] on the device, positive, finite, 16-byte aligned;
 * VQLIN_ERR_INVALID_ARG if null.  Other arguments, layouts and errors as
 * vqlin_linear_w4a4_static.
 */
vqlin_status vqlin_linear_w4a4_static_scaled(const uint16_t* X, const float* static_scale,
                                             const float* channel_scale, int hadamard_block, const uint8_t* wq,
                                             const float* sw, const uint16_t* bias, uint16_t* Y, uint8_t* xq_out,
                                             int M, int N, int K, void* stream);

/*
 * The same projection as vqlin_linear_w4a4_static, for callers that cannot
 * allocate device memory: code that runs while a CUDA graph is being captured
 * (where an allocation is refused), plugins whose host hands them fixed
 * buffers and forbids allocations of their own, runtimes whose memory someone
 * else manages.  (It has no counterpart on the pages; it changes where the
 * kernel's exchange buffer lives, not what it computes.)
 *
 * Instead of a caller's code buffer it uses a fixed array of device memory
 * that belongs to the library: 1 MiB, reserved on every GPU that loads the
 * library until the process exits.  So M x K must be at most 1048576 (e.g. 64
 * tokens x 16384 channels); larger sizes return VQLIN_ERR_UNSUPPORTED_SHAPE.
 * It allocates nothing and calls no allocating routine.  Y equals what
 * vqlin_linear_w4a4_static computes for the same arguments; the codes are not
 * returned.
 *
 * - The first call on a device looks up the array's device address on that
 *   device (cudaGetSymbolAddress); make that first call before any stream
 *   capture that includes this entry point.
 * - Every call on a device shares the array, and the array keeps the last
 *   call's codes.  Nothing in it has to start at zero: each call writes every
 *   code it reads.  Calls whose kernels overlap on the GPU (different streams
 *   without ordering between them) race on the array and may compute wrong
 *   results; order them, for example on one stream.
 */
vqlin_status vqlin_linear_w4a4_static_noalloc(const uint16_t* X, const float* static_scale,
                                              int hadamard_block, const uint8_t* wq, const float* sw,
                                              const uint16_t* bias, uint16_t* Y, int M, int N, int K,
                                              void* stream);

/* W8A8 projection (FoldQuantVLA abstract: the attention-output and
 * feed-forward down projections kept at eight bits, native integer execution
 * with dynamic per-token activations): as vqlin_linear_w4a4 with int8
 * activation codes xq [M, K] uint16 and int8 weight codes wq [N, K] bytes
 * (exact f16 operands;
 * float32 partial sums cover at most 1024 channels, which bounds them below
 * 2^24, and are added up in int32).  Requires K % 64 == 0 and K <= 65536. */
vqlin_status vqlin_linear_w8a8(const uint16_t* xq, const float* sx, const uint8_t* wq,
                               const float* sw, const uint16_t* bias, uint16_t* Y,
                               int M, int N, int K, void* stream);

/*
 * W4A16 projection (weight-only int4, group-wise asymmetric; LoopQ abstract:
 * the batch-1 action expert is memory-bound, so weight bytes dominate and
 * plain RTN weight-only quantization targets it):
 *   Wdq[n,k] = (q[n,k] - z[n,k/g]) * s[n,k/g];
 *   Y = bf16( sum_k X[m,k] * Wdq[n,k] + bias[n] ), float32 accumulation.
 * X: bf16 [M, K]; wq: uint4 [N, K/2]; scales, zeros: bf16 [N, K/g];
 * group_size g in {64, 128, 256}; bias: bf16 [N] or NULL; Y: bf16 [M, N].
 * Requires K % 128 == 0 and K % g == 0.
 */
vqlin_status vqlin_linear_w4a16(const uint16_t* X, const uint8_t* wq, const uint16_t* scales,
                                const uint16_t* zeros, int group_size, const uint16_t* bias,
                                uint16_t* Y, int M, int N, int K, void* stream);

/*
 * 16-bit baseline projection (cuBLAS; LoopQ abstract: the 16-bit model the
 * quantized ones are timed against; FoldQuantVLA abstract: the floating-point
 * baseline): Y = bf16(X . W^T + bias), float32 accumulation.  X: bf16 [M, K]; W: bf16 [N, K]; bias: bf16 [N] or NULL.
 * Requires K % 8 == 0 and N % 8 == 0.
 */
vqlin_status vqlin_linear_bf16_ref(const uint16_t* X, const uint16_t* W, const uint16_t* bias,
                                   uint16_t* Y, int M, int N, int K, void* stream);

/* Test entry point: the int32 accumulators of the W4A8 GEMM (codes as for
 * vqlin_linear_w4a8) into acc [M, N] int32, caller-owned. */
vqlin_status vqlin_debug_gemm_w4a8_s32(const uint16_t* xq, const uint8_t* wq, int32_t* acc,
                                       int M, int N, int K, void* stream);

/*
 * Test entry point: the integer GEMM of vqlin_linear_w4a4 (bits 4) or
 * vqlin_linear_w8a8 (bits 8) with an epilogue that stores the int32
 * accumulators acc [M, N] instead of scaling them.
 */
vqlin_status vqlin_debug_gemm_s32(int bits, const void* xq, const void* wq, int32_t* acc,
                                  int M, int N, int K, void* stream);

/*
 * Test entry point of failure detection: launches the GEMM of
 * vqlin_debug_gemm_s32 with its tile producer withholding every load, so
 * that the consumers' bounded waits run out after limit_ns nanoseconds
 * (0 < limit_ns <= 2e9).  Nothing is left in flight; the kernel records
 * VQLIN_ERR_TIMEOUT in the device status word, frees its tensor memory and
 * returns.  The call itself returns VQLIN_OK once launched; the error is
 * read with vqlin_get_last_device_error().  acc [M, N] is not written.
 */
vqlin_status vqlin_debug_gemm_withheld_loads(int bits, const void* xq, const void* wq, int32_t* acc,
                                             int M, int N, int K, uint64_t limit_ns, void* stream);

/*
 * Channel scaling, the activation side (FoldQuantVLA abstract):
 * vqlin_act_hadamard_quant of x' = x . diag(1/c) -- each loaded value divided
 * by channel_scale[k] (IEEE float32 division) before the block rotation.
 * channel_scale: float [K] on the device, positive, finite, or NULL for none
 * (then exactly vqlin_act_hadamard_quant).  Other arguments as there.
 */
vqlin_status vqlin_act_hadamard_quant_scaled(const uint16_t* X, int M, int K, int bits, int hadamard_block,
                                             const float* channel_scale, const float* static_scale, void* q_out,
                                             float* scale_out, void* stream);

/*
 * The normalisation before the projection fused into the activation kernel
 * (Omega-QVLA technical summary, "Scalatura delle Attivazioni DiT per Passo":
 * the QKV projections follow an AdaLayerNorm).  Per token:
 *   x^ = (x - mean) / sqrt(var + eps)   (mean and population variance over
 *        the K channels, float32, no learned affine part),
 *   y  = x^ * (1 + ada_scale[k]) + ada_shift[k]   (the conditioning's
 *        modulation, one K-vector pair for every token of the call),
 * then exactly vqlin_act_hadamard_quant of y (rotation by blockdiag(H_b /
 * sqrt(b)), dynamic or static per-token quantization); y stays in float32 and
 * is never rounded to bf16.  ada_scale, ada_shift: float [K] on the device,
 * 16-byte aligned; eps >= 0.  Other arguments as vqlin_act_hadamard_quant.
 */
vqlin_status vqlin_act_adaln_hadamard_quant(const uint16_t* X, int M, int K, int bits, int hadamard_block,
                                            const float* ada_scale, const float* ada_shift, float eps,
                                            const float* static_scale, void* q_out, float* scale_out, void* stream);

/*
 * Composite SVD . Hadamard block rotation with a zig-zag channel permutation
 * (Omega-QVLA technical summary, "Rotazione Composita SVD.Hadamard": "Rotazione
 * SVD", "Rotazione Hadamard", "Implementazione a Blocchi").  Three calls:
 *
 * vqlin_composite_rotation_prepare (offline, from the bf16 weights W [N, K]):
 *   perm_out int32 [K]: perm_out[p] = the input channel at position p of the
 *     permuted order -- channels sorted by descending column norm (ties by
 *     index), dealt to the K/b blocks in boustrophedon rounds (round r gives
 *     sorted position r*nb + i to block i for even r, to nb - 1 - i for odd
 *     r; nb = K/b), round order kept inside a block;
 *   R_out float64 [K/b, b, b]: R_j = V_j . H_b / sqrt(b), V_j the right
 *     singular vectors of W's columns of block j (eigenvectors of the Gram
 *     matrix by cyclic Jacobi in float64), descending singular value, each
 *     column signed so its largest-magnitude entry is positive.  A column set
 *     of rank < b (N < b) has no unique null-space basis.  A Jacobi that does
 *     not converge in 40 sweeps records VQLIN_ERR_TIMEOUT in the status word.
 *   R_out is also the call's scratch (column norms, Gram matrices).
 * vqlin_quantize_weights_composite (offline): W~ = W[:, perm] . blockdiag(R_j)
 *   in float64, rounded once to float32, then per-output-channel symmetric RTN
 *   as in vqlin_quantize_weights_rtn: q_out packed as that call's symmetric
 *   layout ([N, K/2] int4 nibbles or [N, K] int8 bytes), scale_out float [N].
 * vqlin_act_composite_quant (online): x~ = x[:, perm] . blockdiag(R_j) in
 *   float32, then per-token dynamic quantization as vqlin_act_hadamard_quant:
 *   q_out [M, K] in the activation-code encoding, scale_out float [M].
 * The codes feed vqlin_linear_w4a4 / _w8a8 / _w4a8 unchanged: x~ . W~^T =
 * x . W^T.  b = block in {64, 128}, K % b == 0, K <= 49152.  Every buffer is a
 * device pointer owned by the caller, 16-byte aligned; scale_out doubles as
 * the per-row absmax accumulator while the call runs.
 */
vqlin_status vqlin_composite_rotation_prepare(const uint16_t* W, int N, int K, int block, int32_t* perm_out,
                                              double* R_out, void* stream);
vqlin_status vqlin_quantize_weights_composite(const uint16_t* W, int N, int K, int bits, int block,
                                              const int32_t* perm, const double* R, void* q_out, float* scale_out,
                                              void* stream);
vqlin_status vqlin_act_composite_quant(const uint16_t* X, int M, int K, int bits, int block, const int32_t* perm,
                                       const double* R, void* q_out, float* scale_out, void* stream);

/*
 * Test entry point of failure detection for the W4A16 tensor-core kernel
 * (M > 4, the sizes and layouts of vqlin_linear_w4a16, no bias): its tile
 * producer withholds every load, so the weight expanders', MMA issuers' and
 * group drains' bounded waits run out after limit_ns nanoseconds
 * (0 < limit_ns <= 2e9).  Nothing is left in flight; the kernel records
 * VQLIN_ERR_TIMEOUT in the device status word, frees its tensor memory and
 * returns.  The call returns VQLIN_OK once launched; the error is read with
 * vqlin_get_last_device_error().  Y is not written.  The pages define no such
 * call: it exists to test the bounded waits.
 */
vqlin_status vqlin_debug_w4a16_withheld_loads(const uint16_t* X, const uint8_t* wq, const uint16_t* scales,
                                              const uint16_t* zeros, int group_size, uint16_t* Y, int M, int N,
                                              int K, uint64_t limit_ns, void* stream);

/*
 * Measurement entry point: the dense rate of one tensor-core MMA kind on this
 * GPU, the roofline denominator of the projections (no passage of the pages
 * defines it; they name no GPU figure).  kind 0: tcgen05.mma kind::f8f6f4 with
 * e4m3 operands (K = 32 per instruction, the W4A4 GEMM); kind 1: kind::f16
 * with bf16 operands (K = 16, the W4A16 / W8A8 / W4A8 GEMMs).  `ctas` CTAs (one
 * per SM; 148 covers a B300) each issue iters x 4 back-to-back 128 x n x K
 * MMAs on operands resident on chip (A in tensor memory if a_in_tmem, else in
 * shared memory; n a multiple of 16 in [16, 256]) from `issuers` warps (1, 2
 * or 4), spread over `accumulators` independent accumulation chains (1, 2 or
 * 4, a multiple of issuers, accumulators * n <= 256).  cycles_dev: device buffer
 * of `ctas` int64, caller-owned (per-CTA SM-clock spans).  Outputs (host):
 * *tflops = flops / event time; *cycles_per_mma = average SM clocks per MMA
 * instruction of the CTA.  Synchronous (waits for the stream).
 */
vqlin_status vqlin_measure_mma_rate(int kind, int a_in_tmem, int n, int accumulators, int issuers,
                                    int iters, int ctas, long long* cycles_dev, double* tflops,
                                    double* cycles_per_mma, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* VQLIN_H */
