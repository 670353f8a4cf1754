// Offline weight preparation: round-to-nearest (RTN) quantization.
//
// Method: "LoopQ" abstract (plain RTN weights), "FoldQuantVLA" abstract
// (rotation folded consistently into the weight rounding) and the
// "Omega-QVLA" summary (normalised Hadamard matrix, block-wise).
//
// Symmetric path (per output channel): one CTA per weight row.  The row is
// rotated block by block with a float64 fast Walsh-Hadamard transform in
// shared memory (the +-1 sums of bf16 values are exact in float64, so the
// rotated value is the float64 quotient by sqrt(b), rounded once to float32),
// kept in shared memory as float32, reduced to its absmax, then quantized.
// This path is offline and not timed, so it favours exactness over speed.
//
// Asymmetric path (weight-only int4, group-wise): one warp per group.
#include "common.cuh"

namespace {

using namespace vqlin_dev;

constexpr int kSymThreads = 256;

template <int BITS>
__global__ void __launch_bounds__(kSymThreads)
weight_quant_sym_kernel(const uint16_t* __restrict__ W, int K, int hb, const float* __restrict__ chan,
                        uint8_t* __restrict__ Q, float* __restrict__ S) {
  constexpr int qmax = (1 << (BITS - 1)) - 1;
  extern __shared__ float rowbuf[];      // K float32 rotated values
  __shared__ double tile[kSymThreads];   // one FWHT work tile
  __shared__ float red[kSymThreads / 32];
  const int n = blockIdx.x;
  const uint16_t* wrow = W + (size_t)n * K;
  const int t = threadIdx.x;

  if (hb == 0) {
    for (int k = t; k < K; k += kSymThreads) {
      const float w = __uint_as_float((uint32_t)wrow[k] << 16);
      rowbuf[k] = chan != nullptr ? __double2float_rn((double)w * (double)chan[k]) : w;
    }
  } else {
    // kSymThreads is a multiple of hb, so a tile holds whole Hadamard blocks
    const double denom = sqrt((double)hb);
    for (int k0 = 0; k0 < K; k0 += kSymThreads) {
      const int k = k0 + t;
      tile[t] = k < K ? (double)__uint_as_float((uint32_t)wrow[k] << 16) : 0.0;
      if (chan != nullptr && k < K) tile[t] *= (double)chan[k];  // channel scaling W' = W diag(c)
      for (int h = 1; h < hb; h <<= 1) {
        __syncthreads();
        if ((t & h) == 0) {
          double a = tile[t], b = tile[t + h];
          tile[t] = a + b;
          tile[t + h] = a - b;
        }
      }
      __syncthreads();
      if (k < K) rowbuf[k] = __double2float_rn(tile[t] / denom);
      __syncthreads();
    }
  }
  __syncthreads();

  float amax = 0.0f;
  for (int k = t; k < K; k += kSymThreads) amax = fmaxf(amax, fabsf(rowbuf[k]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((t & 31) == 0) red[t >> 5] = amax;
  __syncthreads();
  amax = 0.0f;
#pragma unroll
  for (int w = 0; w < kSymThreads / 32; ++w) amax = fmaxf(amax, red[w]);
  const float s = __fdiv_rn(amax, (float)qmax);
  if (t == 0) S[n] = s;

  // each thread quantizes pairs of channels (one int4 byte or two int8 bytes)
  for (int k = 2 * t; k < K; k += 2 * kSymThreads) {
    // sign-magnitude codes in [-qmax, qmax]: nibble (c < 0) << 3 | |c| or
    // byte (c < 0) << 7 | |c|
    uint32_t c[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float r = s > 0.0f ? rintf(__fdiv_rn(rowbuf[k + e], s)) : 0.0f;
      r = fminf(fmaxf(r, (float)(-qmax)), (float)qmax);
      c[e] = (uint32_t)fabsf(r) | (r < 0.0f ? (BITS == 4 ? 8u : 0x80u) : 0u);
    }
    if (BITS == 4) {
      Q[(size_t)n * (K / 2) + k / 2] = (uint8_t)(c[0] | (c[1] << 4));
    } else {
      *reinterpret_cast<uint16_t*>(Q + (size_t)n * K + k) = (uint16_t)(c[0] | (c[1] << 8));
    }
  }
}

// Smallest bf16 value >= x, for positive finite x (as a float32).
__device__ __forceinline__ float bf16_ceil(float x) {
  uint32_t b = __float_as_uint(x);
  if (b & 0xFFFFu) b = (b & 0xFFFF0000u) + 0x10000u;
  return __uint_as_float(b);
}

// One warp per (row, group).  EPL = group / 32 channels per lane (2, 4 or 8).
template <int EPL>
__global__ void __launch_bounds__(256)
weight_quant_asym_kernel(const uint16_t* __restrict__ W, int N, int K, uint8_t* __restrict__ Q,
                         uint16_t* __restrict__ Sg, uint16_t* __restrict__ Zg) {
  constexpr int group = 32 * EPL;
  const int G = K / group;
  const long long gid = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (gid >= (long long)N * G) return;
  const int n = (int)(gid / G), g = (int)(gid % G);
  const int lane = threadIdx.x & 31;
  const uint16_t* src = W + (size_t)n * K + (size_t)g * group + lane * EPL;
  float v[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) v[e] = __uint_as_float((uint32_t)src[e] << 16);
  float lo = 0.0f, hi = 0.0f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    lo = fminf(lo, v[e]);
    hi = fmaxf(hi, v[e]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  const float span = __fsub_rn(hi, lo);
  float s, z;
  if (span == 0.0f) {
    s = 1.0f;
    z = 0.0f;
  } else {
    s = bf16_ceil(__fdiv_rn(span, 15.0f));
    z = fminf(fmaxf(rintf(__fdiv_rn(-lo, s)), 0.0f), 15.0f);
  }
  if (lane == 0) {
    Sg[(size_t)n * G + g] = (uint16_t)(__float_as_uint(s) >> 16);   // exact: s is a bf16 value
    Zg[(size_t)n * G + g] = (uint16_t)(__float_as_uint(z) >> 16);   // exact: integer 0..15
  }
  // packed layout: per 8 channels one 32-bit word, channel 2i in bits
  // [4i, 4i+4) and channel 2i+1 in bits [16+4i, 16+4i+4); the lanes sharing a
  // word OR their nibbles together
  uint32_t word = 0;
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    float qf = rintf(__fdiv_rn(v[e], s)) + z;
    const uint32_t c = (uint32_t)fminf(fmaxf(qf, 0.0f), 15.0f);
    const int p = (lane * EPL + e) & 7;  // position inside the word
    word |= c << ((p & 1) * 16 + 4 * (p >> 1));
  }
  constexpr int LPW = EPL >= 8 ? 1 : 8 / EPL;  // lanes per word
#pragma unroll
  for (int o = 1; o < LPW; o <<= 1) word |= __shfl_xor_sync(0xffffffffu, word, o);
  if (EPL >= 8) {
    uint32_t* dst = reinterpret_cast<uint32_t*>(Q + (size_t)n * (K / 2) + (size_t)g * (group / 2)) + lane * (EPL / 8);
    dst[0] = word;
  } else if ((lane % LPW) == 0) {
    uint32_t* dst = reinterpret_cast<uint32_t*>(Q + (size_t)n * (K / 2) + (size_t)g * (group / 2)) + lane / LPW;
    *dst = word;
  }
}

}  // namespace

namespace vqlin {

cudaError_t launch_weight_quant_sym(const uint16_t* W, int N, int K, int bits, int hb,
                                    void* q, float* s, cudaStream_t st, const float* chan) {
  if (N == 0) return cudaSuccess;
  const size_t smem = (size_t)K * sizeof(float);
  cudaError_t e;
  if (bits == 4) {
    e = cudaFuncSetAttribute(weight_quant_sym_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    weight_quant_sym_kernel<4><<<N, kSymThreads, smem, st>>>(W, K, hb, chan, (uint8_t*)q, s);
  } else {
    e = cudaFuncSetAttribute(weight_quant_sym_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    weight_quant_sym_kernel<8><<<N, kSymThreads, smem, st>>>(W, K, hb, chan, (uint8_t*)q, s);
  }
  return launched(cudaGetLastError());
}

cudaError_t launch_weight_quant_asym(const uint16_t* W, int N, int K, int group, uint8_t* q,
                                     uint16_t* s, uint16_t* z, cudaStream_t st) {
  if (N == 0) return cudaSuccess;
  const long long groups = (long long)N * (K / group);
  const unsigned grid = ceil_div(groups, 8);
  switch (group) {
    case 64: weight_quant_asym_kernel<2><<<grid, 256, 0, st>>>(W, N, K, q, s, z); break;
    case 128: weight_quant_asym_kernel<4><<<grid, 256, 0, st>>>(W, N, K, q, s, z); break;
    default: weight_quant_asym_kernel<8><<<grid, 256, 0, st>>>(W, N, K, q, s, z); break;
  }
  return launched(cudaGetLastError());
}

}  // namespace vqlin
