// Online activation kernel: block-Hadamard rotation + per-token quantization.
//
// Method: "FoldQuantVLA" abstract (block Hadamard transforms combined with
// dynamic per-token quantization) and the "Omega-QVLA" technical summary
// (normalised Hadamard matrix, applied block-wise over channels; per-step
// static activation scales as the alternative to dynamic ones).
//
// Work decomposition (one pass over HBM, every value stays in registers):
//   * a "unit" is 32 channels of one token held by one thread as four 8-channel
//     chunks (one 128-bit load each);
//   * a Hadamard block of b channels is spread over LPG = b/32 consecutive
//     lanes: lane l of the block holds chunks l, l+LPG, l+2LPG, l+3LPG, so
//     the 3 index bits inside a chunk and the 2 bits that pick the chunk are
//     butterflied in registers and only log2(LPG) stages use warp shuffles;
//   * the per-token absmax is reduced over the token's threads (shuffles, then
//     shared memory across warps); one CTA holds one or more whole tokens;
//   * optional channel scaling (FoldQuantVLA abstract: channel scaling
//     combined with the block Hadamard transform): x' = x / c per input
//     channel, an IEEE division of each loaded value, before the rotation;
//   * optional AdaLayerNorm before the rotation (Omega-QVLA summary: the QKV
//     projections follow an AdaLayerNorm): the token's mean and population
//     variance from its registers, then (x - mean)/sqrt(var + eps) * (1 +
//     scale[k]) + shift[k], kept in float32 (never rounded to bf16).
#include "act_codes.cuh"
#include "common.cuh"
#include "tc_ptx.cuh"

namespace {

using namespace vqlin_dev;

constexpr int kThreads = 256;

template <int HB>
struct BlockGeom {
  static constexpr int LPG = HB == 0 ? 1 : HB / 32;  // lanes per Hadamard block
  static constexpr int G = 32 * LPG;                   // channels per lane group
};

template <int BITS, int HB, int UPT, bool ADA>
__global__ void __launch_bounds__(512)
act_quant_kernel(const uint16_t* __restrict__ X, int M, int K, int tpr, int rpc,
                 const float* __restrict__ static_scale, const float* __restrict__ chan,
                 const float* __restrict__ ada_scale, const float* __restrict__ ada_shift, float eps,
                 uint8_t* __restrict__ Q, float* __restrict__ S) {
  using Geo = BlockGeom<HB>;
  constexpr int LPG = Geo::LPG, G = Geo::G;
  constexpr int qmax = (1 << (BITS - 1)) - 1;
  __shared__ float red[16];

  pdl_wait();     // X comes from the previous kernel; q and s may still be read by it
  pdl_trigger();
  const int r = threadIdx.x / tpr;  // token slot inside the CTA
  const int ut = threadIdx.x % tpr;
  const int m = blockIdx.x * rpc + r;
  const bool row_ok = (r < rpc) && (m < M);
  const int units = K / 32;
  const int lane = threadIdx.x & 31;

  float v[UPT][4][8];
  float amax = 0.0f;
  const uint16_t* xrow = X + (size_t)(row_ok ? m : 0) * K;

#pragma unroll
  for (int i = 0; i < UPT; ++i) {
    const int u = ut + i * tpr;
    const bool ok = row_ok && u < units;
    const int g = u / LPG, l = u % LPG;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint4 raw = make_uint4(0, 0, 0, 0);
      if (ok) raw = ldg_nc_v4(xrow + (size_t)g * G + (l + LPG * j) * 8);
      v[i][j][0] = bf16_lo(raw.x); v[i][j][1] = bf16_hi(raw.x);
      v[i][j][2] = bf16_lo(raw.y); v[i][j][3] = bf16_hi(raw.y);
      v[i][j][4] = bf16_lo(raw.z); v[i][j][5] = bf16_hi(raw.z);
      v[i][j][6] = bf16_lo(raw.w); v[i][j][7] = bf16_hi(raw.w);
      if (chan != nullptr && ok) {
        const float* cp = chan + (size_t)g * G + (l + LPG * j) * 8;
        const float4 c0 = __ldg(reinterpret_cast<const float4*>(cp));
        const float4 c1 = __ldg(reinterpret_cast<const float4*>(cp + 4));
        const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) v[i][j][e] = __fdiv_rn(v[i][j][e], c[e]);
      }
    }
    if (!ADA) {  // without the normalisation, rotate while the next unit's loads are in flight
      if (HB > 0) hadamard_unit<HB == 0 ? 128 : HB>(v[i], lane);
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[i][j][e]));
    }
  }

  // the token's sum over its tpr threads in a fixed order (shuffle tree, then
  // the warps' partials in warp order); every thread of the CTA calls it
  auto token_sum = [&](float x) -> float {
    if (tpr <= 32) {
      for (int o = tpr >> 1; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
      return x;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    __syncthreads();  // red may still be read by the previous reduction
    if (lane == 0) red[threadIdx.x >> 5] = x;
    __syncthreads();
    const int wpr = tpr >> 5, w0 = r * wpr;
    float t = 0.0f;
    if (r < rpc)
      for (int w = 0; w < wpr; ++w) t += red[w0 + w];
    return t;
  };

  if constexpr (ADA) {
    // AdaLayerNorm of the token before its rotation (the normalisation fused
    // into this kernel): (x - mean) / sqrt(var + eps) * (1 + scale) + shift,
    // mean and population variance over the K channels in float32 (two
    // passes over the registers)
    float s1 = 0.0f;
#pragma unroll
    for (int i = 0; i < UPT; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) s1 += v[i][j][e];
    const float mean = __fdiv_rn(token_sum(s1), (float)K);
    float s2 = 0.0f;
#pragma unroll
    for (int i = 0; i < UPT; ++i) {
      const bool ok = row_ok && ut + i * tpr < units;
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float d = ok ? v[i][j][e] - mean : 0.0f;
          s2 = fmaf(d, d, s2);
        }
    }
    const float var = __fdiv_rn(token_sum(s2), (float)K);
    const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(var + eps));
#pragma unroll
    for (int i = 0; i < UPT; ++i) {
      const int u = ut + i * tpr;
      if (!(row_ok && u < units)) continue;
      const int g = u / LPG, l = u % LPG;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const size_t ch = (size_t)g * G + (l + LPG * j) * 8;
        const float4 a0 = __ldg(reinterpret_cast<const float4*>(ada_scale + ch));
        const float4 a1 = __ldg(reinterpret_cast<const float4*>(ada_scale + ch + 4));
        const float4 b0 = __ldg(reinterpret_cast<const float4*>(ada_shift + ch));
        const float4 b1 = __ldg(reinterpret_cast<const float4*>(ada_shift + ch + 4));
        const float sc[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const float sh[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) v[i][j][e] = fmaf((v[i][j][e] - mean) * rstd, 1.0f + sc[e], sh[e]);
      }
    }
#pragma unroll
    for (int i = 0; i < UPT; ++i) {
      if (HB > 0) hadamard_unit<HB == 0 ? 128 : HB>(v[i], lane);
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[i][j][e]));
    }
  }

  float s;
  if (static_scale != nullptr) {
    s = __ldg(static_scale);
  } else {
    // per-token absmax over the token's tpr threads
    if (tpr <= 32) {
      for (int o = tpr >> 1; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    } else {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (ADA) __syncthreads();  // the normalisation's sums may still be read from red
      if (lane == 0) red[threadIdx.x >> 5] = amax;
      __syncthreads();
      const int wpr = tpr >> 5, w0 = r * wpr;
      amax = 0.0f;
      if (r < rpc)
        for (int w = 0; w < wpr; ++w) amax = fmaxf(amax, red[w0 + w]);
    }
    s = __fdiv_rn(amax, (float)qmax);
  }
  if (!row_ok) return;
  if (ut == 0 && S != nullptr) S[m] = s;
  const float inv_s = s > 0.0f ? __frcp_rn(s) : 0.0f;
  // rotated activations: the hardware conversions (see quantize_chunk_fast)
  const float kq = inv_s * (BITS == 4 ? 1.0f / 512.0f : 1.0f / 16777216.0f);

#pragma unroll
  for (int i = 0; i < UPT; ++i) {
    const int u = ut + i * tpr;
    if (u >= units) break;
    const int g = u / LPG, l = u % LPG;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t w[4];
      if (HB > 0)
        quantize_chunk_fast<BITS>(v[i][j], kq, w);
      else
        quantize_chunk<BITS>(v[i][j], s, inv_s, w);
      const size_t ch = (size_t)g * G + (l + LPG * j) * 8;  // first channel of the chunk
      if (BITS == 4) {
        *reinterpret_cast<uint2*>(Q + (size_t)m * K + ch) = make_uint2(w[0], w[1]);
      } else {
        *reinterpret_cast<uint4*>(Q + ((size_t)m * K + ch) * 2) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
}

template <int BITS, int HB>
cudaError_t launch_hb(const uint16_t* X, int M, int K, const float* ss, const float* chan, const float* ada_scale,
                      const float* ada_shift, float eps, void* q, float* s, cudaStream_t st) {
  const int units = K / 32;
  const int upt = units <= 512 ? 1 : (units <= 1024 ? 2 : 4);  // at most 512 threads per token
  int tpr = (units + upt - 1) / upt;
  // threads per token: a power of two up to a warp, else whole warps
  if (tpr <= 32) {
    int p = 1;
    while (p < tpr) p <<= 1;
    tpr = p;
  } else {
    tpr = (tpr + 31) / 32 * 32;
  }
  const int rpc = tpr >= kThreads ? 1 : kThreads / tpr;
  const int threads = rpc * tpr;
  const unsigned grid = vqlin::ceil_div(M, rpc);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = vqlin::pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  uint8_t* qb = static_cast<uint8_t*>(q);
  if (ada_scale != nullptr) {
    if (upt == 1)
      return cudaLaunchKernelEx(&cfg, act_quant_kernel<BITS, HB, 1, true>, X, M, K, tpr, rpc, ss, chan, ada_scale,
                                ada_shift, eps, qb, s);
    if (upt == 2)
      return cudaLaunchKernelEx(&cfg, act_quant_kernel<BITS, HB, 2, true>, X, M, K, tpr, rpc, ss, chan, ada_scale,
                                ada_shift, eps, qb, s);
    return cudaLaunchKernelEx(&cfg, act_quant_kernel<BITS, HB, 4, true>, X, M, K, tpr, rpc, ss, chan, ada_scale,
                              ada_shift, eps, qb, s);
  }
  if (upt == 1)
    return cudaLaunchKernelEx(&cfg, act_quant_kernel<BITS, HB, 1, false>, X, M, K, tpr, rpc, ss, chan, nullptr,
                              nullptr, 0.0f, qb, s);
  if (upt == 2)
    return cudaLaunchKernelEx(&cfg, act_quant_kernel<BITS, HB, 2, false>, X, M, K, tpr, rpc, ss, chan, nullptr,
                              nullptr, 0.0f, qb, s);
  return cudaLaunchKernelEx(&cfg, act_quant_kernel<BITS, HB, 4, false>, X, M, K, tpr, rpc, ss, chan, nullptr,
                            nullptr, 0.0f, qb, s);
}

}  // namespace

namespace vqlin {

cudaError_t launch_act_quant(const uint16_t* X, int M, int K, int bits, int hb,
                             const float* static_scale, void* q, float* s, cudaStream_t st, const float* chan,
                             const float* ada_scale, const float* ada_shift, float eps) {
  if (M == 0) return cudaSuccess;
  cudaError_t e;
  if (bits == 4) {
    if (hb == 0) e = launch_hb<4, 0>(X, M, K, static_scale, chan, ada_scale, ada_shift, eps, q, s, st);
    else if (hb == 64) e = launch_hb<4, 64>(X, M, K, static_scale, chan, ada_scale, ada_shift, eps, q, s, st);
    else e = launch_hb<4, 128>(X, M, K, static_scale, chan, ada_scale, ada_shift, eps, q, s, st);
  } else {
    if (hb == 0) e = launch_hb<8, 0>(X, M, K, static_scale, chan, ada_scale, ada_shift, eps, q, s, st);
    else if (hb == 64) e = launch_hb<8, 64>(X, M, K, static_scale, chan, ada_scale, ada_shift, eps, q, s, st);
    else e = launch_hb<8, 128>(X, M, K, static_scale, chan, ada_scale, ada_shift, eps, q, s, st);
  }
  return launched(e);
}

}  // namespace vqlin
