// Weight-only int4 projection (W4A16), CUDA-core GEMV path for at most 4
// tokens (the tensor-core kernel in w4a16_tcgen05.cu serves larger M).
//
//   Wdq[n, k] = (q[n, k] - z[n, k/g]) * s[n, k/g]     (exact in float32)
//   Y[m, n]   = bf16(sum_k X[m, k] * Wdq[n, k] + bias[n]), float32 accumulation
//
// Method: "LoopQ" abstract (the action expert is memory-bound; weight bytes
// dominate), with group-wise asymmetric RTN weights.
//
// A warp owns 8 weight rows and up to 4 tokens.  Each lane covers 8
// consecutive channels of every 256-channel step (one 32-bit word of packed
// codes per row), keeps the 4 tokens' matching activations in registers and
// reuses them across its 8 rows; partial sums are reduced across lanes at the
// end.  Every packed weight byte is read from HBM once per token block.
#include "common.cuh"
#include "tc_ptx.cuh"

namespace {

using namespace vqlin_dev;

constexpr int ROWS_PER_WARP = 8;
constexpr int TOK = 4;
constexpr int WARPS = 8;

template <int GROUP>
__global__ void __launch_bounds__(WARPS * 32)
w4a16_gemv_kernel(const uint16_t* __restrict__ X, const uint8_t* __restrict__ Wq,
                  const uint16_t* __restrict__ Sg, const uint16_t* __restrict__ Zg,
                  const uint16_t* __restrict__ bias, uint16_t* __restrict__ Y, int M, int N, int K) {
  pdl_wait();  // X comes from the previous kernel; Y may still be read by it
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n0 = (blockIdx.x * WARPS + warp) * ROWS_PER_WARP;
  const int t0 = blockIdx.y * TOK;
  if (n0 >= N) return;
  const int G = K / GROUP;
  float acc[ROWS_PER_WARP][TOK];
#pragma unroll
  for (int r = 0; r < ROWS_PER_WARP; ++r)
#pragma unroll
    for (int t = 0; t < TOK; ++t) acc[r][t] = 0.0f;

  for (int k0 = 0; k0 < K; k0 += 256) {
    const int k = k0 + lane * 8;
    if (k >= K) continue;  // K % 128 == 0: only the upper half-warp of the last step idles
    float x[TOK][8];
#pragma unroll
    for (int t = 0; t < TOK; ++t) {
      uint4 raw = make_uint4(0, 0, 0, 0);
      if (t0 + t < M) raw = *reinterpret_cast<const uint4*>(X + (size_t)(t0 + t) * K + k);
      x[t][0] = bf16_lo(raw.x); x[t][1] = bf16_hi(raw.x);
      x[t][2] = bf16_lo(raw.y); x[t][3] = bf16_hi(raw.y);
      x[t][4] = bf16_lo(raw.z); x[t][5] = bf16_hi(raw.z);
      x[t][6] = bf16_lo(raw.w); x[t][7] = bf16_hi(raw.w);
    }
    const int g = k / GROUP;
#pragma unroll
    for (int r = 0; r < ROWS_PER_WARP; ++r) {
      const int n = n0 + r;
      if (n >= N) break;
      const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(Wq + (size_t)n * (K / 2) + k / 2));
      const float s = __uint_as_float((uint32_t)__ldg(Sg + (size_t)n * G + g) << 16);
      const float z = __uint_as_float((uint32_t)__ldg(Zg + (size_t)n * G + g) << 16);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        // channel 2i in bits [4i, 4i+4), channel 2i+1 in bits [16+4i, 16+4i+4)
        const float q = (float)((w >> ((e & 1) * 16 + 4 * (e >> 1))) & 0xFu);
        const float wd = (q - z) * s;  // exact: 5-bit integer times a bf16 value
#pragma unroll
        for (int t = 0; t < TOK; ++t) acc[r][t] = fmaf(x[t][e], wd, acc[r][t]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < ROWS_PER_WARP; ++r)
#pragma unroll
    for (int t = 0; t < TOK; ++t)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[r][t] += __shfl_xor_sync(0xffffffffu, acc[r][t], o);
  if (lane < ROWS_PER_WARP * TOK) {
    // lane -> (row, token); static indices via a select chain
    const int r = lane / TOK, t = lane % TOK;
    float v = 0.0f;
#pragma unroll
    for (int rr = 0; rr < ROWS_PER_WARP; ++rr)
#pragma unroll
      for (int tt = 0; tt < TOK; ++tt)
        if (rr == r && tt == t) v = acc[rr][tt];
    const int n = n0 + r, m = t0 + t;
    if (n < N && m < M) {
      if (bias) v += __uint_as_float((uint32_t)bias[n] << 16);
      Y[(size_t)m * N + n] = f32_to_bf16_rn(v);
    }
  }
}

}  // namespace

namespace vqlin {

cudaError_t launch_w4a16_gemv(const uint16_t* X, const uint8_t* wq, const uint16_t* s,
                         const uint16_t* z, int group, const uint16_t* bias, uint16_t* Y,
                         int M, int N, int K, int* /*status*/, cudaStream_t st) {
  if (M == 0 || N == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ceil_div(N, WARPS * ROWS_PER_WARP), ceil_div(M, TOK), 1);
  cfg.blockDim = dim3(WARPS * 32, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (group) {
    case 64: return cudaLaunchKernelEx(&cfg, w4a16_gemv_kernel<64>, X, wq, s, z, bias, Y, M, N, K);
    case 128: return cudaLaunchKernelEx(&cfg, w4a16_gemv_kernel<128>, X, wq, s, z, bias, Y, M, N, K);
    default: return cudaLaunchKernelEx(&cfg, w4a16_gemv_kernel<256>, X, wq, s, z, bias, Y, M, N, K);
  }
}

}  // namespace vqlin
