// Shared device helpers and internal launcher declarations of libvqlin.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/vqlin.h"

namespace vqlin {

// ---------------------------------------------------------------- host side

// Records a detail message for vqlin_last_error_message() and returns `st`.
vqlin_status fail(vqlin_status st, const char* fmt, ...);

// Host-side tally of the library's kernel launches: adds n to the count
// that vqlin_kernel_launch_count() reports when e is cudaSuccess; returns e.
cudaError_t launched(cudaError_t e, int n = 1);

// Address of the per-device status word (a __device__ int), for kernels that
// report bounded-wait timeouts.  Never null after a successful call.
int* device_status_word();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline unsigned ceil_div(long long a, long long b) { return (unsigned)((a + b - 1) / b); }

// 2-D tiled TMA descriptor: a [rows, inner] matrix of `dtype` elements whose
// rows are row_bytes apart, copied in boxes of box_inner x box_rows elements;
// out-of-range elements read as zero.  False if the driver rejects it
// (tmap.cu).
bool tmap_encoder_available();
bool encode_tmap_2d(CUtensorMap* tm, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                    uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows,
                    CUtensorMapSwizzle swizzle);

// Programmatic dependent launch of the library's kernels (on unless the
// environment sets VQLIN_PDL=0): each kernel may start while the previous one
// on the stream finishes, and waits for it before touching its outputs.
bool pdl_enabled();

// How many clusters of `cluster` CTAs of `kernel` (threads, dynamic shared
// memory) can be resident on the current device at once (cached; 0 if the
// query fails).
int max_active_clusters(const void* kernel, int threads, size_t dyn_smem, int cluster);

// Launchers (defined in the kernel files).  They assume validated arguments.
// chan: optional per-input-channel scale c [K] (x / c before the rotation;
// for weights W * c), null for none
cudaError_t launch_act_quant(const uint16_t* X, int M, int K, int bits, int hb,
                             const float* static_scale, void* q, float* s, cudaStream_t st,
                             const float* chan = nullptr, const float* ada_scale = nullptr,
                             const float* ada_shift = nullptr, float eps = 0.0f);
cudaError_t launch_weight_quant_sym(const uint16_t* W, int N, int K, int bits, int hb,
                                    void* q, float* s, cudaStream_t st, const float* chan = nullptr);
cudaError_t launch_weight_quant_asym(const uint16_t* W, int N, int K, int group,
                                     uint8_t* q, uint16_t* s, uint16_t* z, cudaStream_t st);
// Integer GEMM (tcgen05); acc == nullptr: bf16 epilogue into Y, else raw int32
// accumulators into acc.
vqlin_status launch_int_gemm(int bits, const void* xq, const float* sx, const void* wq,
                             const float* sw, const uint16_t* bias, uint16_t* Y, int32_t* acc,
                             int M, int N, int K, int* status, cudaStream_t st);
// W4A8 GEMM: int4 weight codes [N, K/2] (as for W4A4) against int8 activation
// codes [M, K] (16-bit operand words); acc == nullptr as above.
vqlin_status launch_int_gemm_w4a8(const void* xq, const float* sx, const void* wq, const float* sw,
                                  const uint16_t* bias, uint16_t* Y, int32_t* acc, int M, int N, int K, int* status,
                                  cudaStream_t st);
// W4A4 GEMM of activation codes quantized at one static scale (*static_scale
// applies to every token).
vqlin_status launch_int_gemm_static_scale(const void* xq, const float* static_scale, const void* wq, const float* sw,
                                          const uint16_t* bias, uint16_t* Y, int M, int N, int K, int* status,
                                          cudaStream_t st);
// W4A4 GEMM whose activations arrive as bf16 and are quantized on chip (block
// Hadamard of hb = 64 or 128 channels, one static scale) instead of by a
// separate activation kernel.
vqlin_status launch_int_gemm_static_act(const uint16_t* X, const float* static_scale, int hb, const void* wq,
                                       const float* sw, const uint16_t* bias, uint16_t* Y, int M, int N, int K,
                                       int* status, cudaStream_t st);
// The same GEMM with its producer withholding every tile load, so that the
// consumers' bounded waits run out after limit_ns (failure-detection test).
vqlin_status launch_int_gemm_withheld(int bits, const void* xq, const void* wq, int32_t* acc,
                                      int M, int N, int K, int* status, uint64_t limit_ns,
                                      cudaStream_t st);
// W4A16: CUDA-core GEMV (M <= 4) and tcgen05 dequant-GEMM (any M).
cudaError_t launch_w4a16_gemv(const uint16_t* X, const uint8_t* wq, const uint16_t* s,
                              const uint16_t* z, int group, const uint16_t* bias, uint16_t* Y,
                              int M, int N, int K, int* status, cudaStream_t st);
// withhold = 1: the tile producer issues nothing, so every bounded wait runs
// out after limit_ns (0: the default limit) -- the failure-detection test hook
vqlin_status launch_w4a16_tc(const uint16_t* X, const uint8_t* wq, const uint16_t* s,
                             const uint16_t* z, int group, const uint16_t* bias, uint16_t* Y,
                             int M, int N, int K, int* status, cudaStream_t st, int withhold = 0,
                             uint64_t limit_ns = 0);
constexpr int kW4a16GemvMaxM = 4;

// Few-token W4A4 (lowlat_tcgen05.cu): every operand of a CTA's K range stays
// on chip; at most 8 k-blocks of 128 channels per CTA and 16 CTAs along K.
constexpr int kLowlatMaxM = 128;
constexpr int kLowlatMaxK = 16384;
// Static-scale W4A4 whose activations are rotated and quantized on chip, once
// per cluster, into the code buffer xq_ws [M, K] (bytes, the activation
// kernel's encoding), which the CTAs then read back; any M, K <= kLowlatMaxK.
// chan (optional, float [K]): channel scaling, x / c[k] before the rotation.
vqlin_status launch_w4a4_static_lowlat(const uint16_t* X, const float* static_scale, int hb, uint8_t* xq_ws,
                                       const uint8_t* wq, const float* sw, const uint16_t* bias, uint16_t* Y, int M,
                                       int N, int K, int* status, cudaStream_t st, const float* chan = nullptr);
// The same kernel fed with the activation kernel's codes and per-token scales.
// Whether the few-token W4A4 kernel's plan fits one wave of clusters.
bool lowlat_one_wave(bool fused, int hb, int M, int N, int K);
// sx_step 1: per-token scales sx[m]; 0: one scale sx[0] for every token
vqlin_status launch_w4a4_codes_lowlat(const uint8_t* xq, const float* sx, const uint8_t* wq, const float* sw,
                                      const uint16_t* bias, uint16_t* Y, int M, int N, int K, int* status,
                                      cudaStream_t st, int sx_step = 1);
// Whether the static-scale projection at this K runs as the activation kernel
// plus the codes variant instead of the one-launch kernel.
bool static_two_launch(int K);

// Largest K each kernel supports (host-side shape checks).
constexpr int kActQuantMaxK = 65536;
constexpr int kWeightQuantMaxK = 49152;

// Composite SVD . Hadamard block rotation (b = 64 or 128, K % b == 0):
// P and R_j from the weights (float64, offline), weights rotated and
// quantized per output channel, activations rotated and quantized per token.
cudaError_t launch_composite_prepare(const uint16_t* W, int N, int K, int b, int* perm, double* R, int* status,
                                     cudaStream_t st);
cudaError_t launch_weight_quant_composite(const uint16_t* W, int N, int K, int bits, int b, const int* perm,
                                          const double* R, uint8_t* q, float* scale, cudaStream_t st);
cudaError_t launch_act_composite_quant(const uint16_t* X, int M, int K, int bits, int b, const int* perm,
                                       const double* R, void* q, float* scale, cudaStream_t st);
constexpr int kGemmW4MaxK = 65536;   // |acc| <= 49 K stays below 2^24
constexpr int kGemmW8MaxK = 65536;   // |acc| <= 127^2 K stays below 2^31

}  // namespace vqlin

// ---------------------------------------------------------------- device side

namespace vqlin_dev {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// 128-bit streaming load through the non-coherent path (read-only data).
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Two floats to bf16 (round to nearest even) in one paired conversion; lo in
// bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  const __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&t);
}

}  // namespace vqlin_dev
