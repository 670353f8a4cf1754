// Weight-only int4 projection (W4A16) for a few tokens: a split-K GEMV on the
// CUDA cores (the tensor-core kernel in w4a16_tcgen05.cu serves more tokens).
//
//   Y[m, n] = bf16( sum_g s[n,g] * sum_{k in g} X[m,k] * (q[n,k] - z[n,g]) + bias[n] )
//
// Method: "LoopQ" abstract (the batch-1 action expert is memory-bound: weight
// bytes dominate), with group-wise asymmetric RTN weights.
//
// The kernel streams the packed weights once at HBM rate:
//   * work unit = 512 channels of one weight row, read by a half-warp with one
//     128-bit load per lane (32 channels = one group share; groups are >= 64
//     channels, so a lane's channels share one scale and zero point);
//   * a row block = RT rows; half-warp h works on row h % RT of a block and on
//     every KS-th unit of it (KS = 16 / RT, K split KS ways inside the CTA, so
//     that a half-warp has at most 8 units of a row);
//   * about two CTAs per SM stay resident and loop over row blocks; each lane
//     keeps the loads of the next block in flight while it computes the
//     current one (all of a block's weight loads are issued at once), and the
//     first block's loads go out before the previous kernel is waited for:
//     weights do not depend on it, so their latency overlaps it;
//   * (q - z) is exact: OR-ing a nibble pair with 0x4300 gives the bf16 values
//     128 + q, a bf16x2 subtraction of 128 + z leaves q - z, and the products
//     with X accumulate in float32 per group share, then times s;
//   * the KS partial sums of a row meet in shared memory and are added in a
//     fixed order (deterministic, no global scratch).
#include "common.cuh"
#include "tc_ptx.cuh"

namespace {

using namespace vqlin_dev;

constexpr int kThreads = 256;   // 16 half-warps
constexpr int kUnit = 512;      // channels of one work unit (16 lanes x 32)
constexpr int kMaxU = 8;        // units of a row one half-warp handles per block

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// bf16x2 bits of (128 + z, 128 + z) for the zero point stored at zp (a bf16
// holding an integer 0..15): 128 + z is the bf16 0x4300 + z.
__device__ __forceinline__ uint32_t zero_pair(const uint16_t* zp) {
  const uint32_t z = (uint32_t)__uint_as_float((uint32_t)__ldg(zp) << 16);
  const uint32_t h = 0x4300u + z;
  return h | (h << 16);
}

// The 8 channels of one packed word (channel 2i in bits 4i.., channel 2i+1 in
// bits 16 + 4i..) as float (q - z), channel order; zz = bf16x2 (128 + z).
__device__ __forceinline__ void dequant8(uint32_t w, uint32_t zz, float (&d)[8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t p = bf16x2_sub(((w >> (4 * i)) & 0x000F000Fu) | 0x43004300u, zz);
    d[2 * i] = bf16_lo(p);
    d[2 * i + 1] = bf16_hi(p);
  }
}

// The weight loads of one half-warp lane for one row block: units
// kp + KS u of its row (u < kMaxU), with their group scales and zero points.
struct UnitLoads {
  uint4 w[kMaxU];
  float s[kMaxU];
  uint32_t zz[kMaxU];
};

// Issues the loads of unit slot u for row n (nothing if the slot is empty).
template <int GROUP>
__device__ __forceinline__ void load_unit(UnitLoads& L, int u, const uint8_t* __restrict__ Wq,
                                          const uint16_t* __restrict__ Sg, const uint16_t* __restrict__ Zg, int n,
                                          bool row_ok, int kp, int ks, int li, int nunits, int K) {
  const int j = kp + ks * u;
  const int c = kUnit * j + 32 * li;
  L.w[u] = make_uint4(0, 0, 0, 0);
  L.s[u] = 0.0f;
  L.zz[u] = 0x43004300u;
  if (row_ok && j < nunits && c < K) {
    const int G = K / GROUP;
    L.w[u] = ldg_nc_v4(Wq + (size_t)n * (K / 2) + c / 2);
    const int g = c / GROUP;
    L.s[u] = __uint_as_float((uint32_t)__ldg(Sg + (size_t)n * G + g) << 16);
    L.zz[u] = zero_pair(Zg + (size_t)n * G + g);
  }
}

template <int MT, int GROUP>
__global__ void __launch_bounds__(kThreads, 2)
w4a16_gemv_kernel(const uint16_t* __restrict__ X, const uint8_t* __restrict__ Wq, const uint16_t* __restrict__ Sg,
                  const uint16_t* __restrict__ Zg, const uint16_t* __restrict__ bias, uint16_t* __restrict__ Y,
                  int M, int N, int K, int rt) {
  __shared__ float part[16][MT];
  const int tid = threadIdx.x, hw = tid >> 4, li = tid & 15;
  const int ks = 16 / rt;
  const int r = hw % rt, kp = hw / rt;
  const int nunits = (K + kUnit - 1) / kUnit;
  const int nblocks = (N + rt - 1) / rt;

  // one ring of slots: slot u holds unit u of the current block; once read,
  // it is refilled with unit u of the next block, so a lane keeps up to
  // kMaxU loads in flight across blocks
  UnitLoads L;
  int b = blockIdx.x;
  {
    const int n = b * rt + r;
#pragma unroll
    for (int u = 0; u < kMaxU; ++u)
      load_unit<GROUP>(L, u, Wq, Sg, Zg, n < N ? n : 0, b < nblocks && n < N, kp, ks, li, nunits, K);
  }
  pdl_wait();  // X comes from the previous kernel; Y may still be read by it
  pdl_trigger();

  for (; b < nblocks; b += gridDim.x) {
    const int nb = (b + (int)gridDim.x) * rt + r;  // this half-warp's row of the next block
    const bool nb_ok = b + (int)gridDim.x < nblocks && nb < N;
    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
#pragma unroll
    for (int u = 0; u < kMaxU; ++u) {
      const int j = kp + ks * u;
      const int c = kUnit * j + 32 * li;
      const bool live = j < nunits && c < K;
      const uint32_t ws[4] = {L.w[u].x, L.w[u].y, L.w[u].z, L.w[u].w};
      const uint32_t zz = L.zz[u];
      const float sc = L.s[u];
      load_unit<GROUP>(L, u, Wq, Sg, Zg, nb_ok ? nb : 0, nb_ok, kp, ks, li, nunits, K);
      if (!live) continue;
      // two independent chains per token
      float p0[MT], p1[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) p0[m] = p1[m] = 0.0f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // 8 channels per packed word
        float d[8];
        dequant8(ws[q], zz, d);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m < M) {
            const uint4 xr = *reinterpret_cast<const uint4*>(X + (size_t)m * K + c + 8 * q);
            p0[m] = fmaf(bf16_lo(xr.x), d[0], p0[m]);
            p1[m] = fmaf(bf16_hi(xr.x), d[1], p1[m]);
            p0[m] = fmaf(bf16_lo(xr.y), d[2], p0[m]);
            p1[m] = fmaf(bf16_hi(xr.y), d[3], p1[m]);
            p0[m] = fmaf(bf16_lo(xr.z), d[4], p0[m]);
            p1[m] = fmaf(bf16_hi(xr.z), d[5], p1[m]);
            p0[m] = fmaf(bf16_lo(xr.w), d[6], p0[m]);
            p1[m] = fmaf(bf16_hi(xr.w), d[7], p1[m]);
          }
        }
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[m] = fmaf(sc, p0[m] + p1[m], acc[m]);
    }
    // half-warp reduction (fixed order), then the KS partials of each row in
    // shared memory, added in order of the K phase
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], o);
    if (li == 0) {
#pragma unroll
      for (int m = 0; m < MT; ++m) part[hw][m] = acc[m];
    }
    __syncthreads();
    if (tid < rt * MT) {
      const int rr = tid / MT, m = tid % MT;
      const int nn = b * rt + rr;
      if (nn < N && m < M) {
        float y = 0.0f;
        for (int k = 0; k < ks; ++k) y += part[rr + rt * k][m];
        if (bias) y += __uint_as_float((uint32_t)bias[nn] << 16);
        Y[(size_t)m * N + nn] = f32_to_bf16_rn(y);
      }
    }
    __syncthreads();  // part is rewritten by the next block
  }
}

template <int MT>
cudaError_t launch_mt(const uint16_t* X, const uint8_t* wq, const uint16_t* s, const uint16_t* z, int group,
                      const uint16_t* bias, uint16_t* Y, int M, int N, int K, cudaStream_t st) {
  // K split KS = 16 / rt ways inside a CTA, so that a half-warp has at most
  // kMaxU units of a row; about two CTAs per SM loop over the row blocks
  const int nunits = (K + kUnit - 1) / kUnit;
  int ks = 1;
  while (ks < 16 && (nunits + ks - 1) / ks > kMaxU) ks <<= 1;
  const int rt = 16 / ks;
  const int nblocks = (N + rt - 1) / rt;
  const int grid = nblocks < 2 * 148 ? nblocks : 2 * 148;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = vqlin::pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (group) {
    case 64: return cudaLaunchKernelEx(&cfg, w4a16_gemv_kernel<MT, 64>, X, wq, s, z, bias, Y, M, N, K, rt);
    case 128: return cudaLaunchKernelEx(&cfg, w4a16_gemv_kernel<MT, 128>, X, wq, s, z, bias, Y, M, N, K, rt);
    default: return cudaLaunchKernelEx(&cfg, w4a16_gemv_kernel<MT, 256>, X, wq, s, z, bias, Y, M, N, K, rt);
  }
}

}  // namespace

namespace vqlin {

cudaError_t launch_w4a16_gemv(const uint16_t* X, const uint8_t* wq, const uint16_t* s, const uint16_t* z, int group,
                              const uint16_t* bias, uint16_t* Y, int M, int N, int K, int* /*status*/,
                              cudaStream_t st) {
  if (M == 0 || N == 0) return cudaSuccess;
  if (M <= 1) return launch_mt<1>(X, wq, s, z, group, bias, Y, M, N, K, st);
  if (M <= 2) return launch_mt<2>(X, wq, s, z, group, bias, Y, M, N, K, st);
  return launch_mt<4>(X, wq, s, z, group, bias, Y, M, N, K, st);  // M <= kW4a16GemvMaxM
}

}  // namespace vqlin
