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
#include <mutex>

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

// ---------------------------------------------------------------------------
// Variant with the activations staged on chip.  The tokens' activations are
// converted once per CTA to float32 in shared memory (float4 slots swizzled so
// that the 16 lanes of a half-warp, 128 bytes apart, hit different banks),
// with the sum of every 32-channel chunk beside them.  A nibble then becomes
// the float 16 + q with one shift and one logic operation (q in the mantissa
// bits 19..22 of 16.0), and the zero point leaves the inner loop:
//   sum_k x_k (q_k - z) = sum_k x_k (16 + q_k) - (16 + z) sum_k x_k
// over a lane's 32 channels (one group share).  About two thirds of the
// instructions per weight byte of the variant above.
constexpr int kThreads2 = 512;           // 32 half-warps
constexpr size_t kMaxXSmem = 200 * 1024;  // staged activations + chunk sums

__device__ __forceinline__ int xslot(int q) { return q ^ ((q >> 3) & 7); }

struct UnitLoads2 {
  uint4 w[kMaxU];
  float s[kMaxU];
  float zf[kMaxU];  // 16 + z
};

template <int GROUP>
__device__ __forceinline__ void load_unit2(UnitLoads2& L, int u, const uint8_t* __restrict__ Wq,
                                           const uint16_t* __restrict__ Sg, const uint16_t* __restrict__ Zg, int n,
                                           bool row_ok, int kp, int ks, int li, int nunits, int K) {
  const int j = kp + ks * u;
  const int c = kUnit * j + 32 * li;
  L.w[u] = make_uint4(0, 0, 0, 0);
  L.s[u] = 0.0f;
  L.zf[u] = 16.0f;
  if (row_ok && j < nunits && c < K) {
    const int G = K / GROUP;
    L.w[u] = ldg_nc_v4(Wq + (size_t)n * (K / 2) + c / 2);
    const int g = c / GROUP;
    L.s[u] = __uint_as_float((uint32_t)__ldg(Sg + (size_t)n * G + g) << 16);
    L.zf[u] = 16.0f + __uint_as_float((uint32_t)__ldg(Zg + (size_t)n * G + g) << 16);
  }
}

// The 8 channels of one packed word as the floats 16 + q, channel order.
__device__ __forceinline__ void nib16(uint32_t w, float (&f)[8]) {
  f[0] = __uint_as_float(((w << 19) & 0x00780000u) | 0x41800000u);
  f[1] = __uint_as_float(((w << 3) & 0x00780000u) | 0x41800000u);
  f[2] = __uint_as_float(((w << 15) & 0x00780000u) | 0x41800000u);
  f[3] = __uint_as_float(((w >> 1) & 0x00780000u) | 0x41800000u);
  f[4] = __uint_as_float(((w << 11) & 0x00780000u) | 0x41800000u);
  f[5] = __uint_as_float(((w >> 5) & 0x00780000u) | 0x41800000u);
  f[6] = __uint_as_float(((w << 7) & 0x00780000u) | 0x41800000u);
  f[7] = __uint_as_float(((w >> 9) & 0x00780000u) | 0x41800000u);
}

template <int MT, int GROUP>
__global__ void __launch_bounds__(kThreads2, 1)
w4a16_gemv_smem_kernel(const uint16_t* __restrict__ X, const uint8_t* __restrict__ Wq,
                       const uint16_t* __restrict__ Sg, const uint16_t* __restrict__ Zg,
                       const uint16_t* __restrict__ bias, uint16_t* __restrict__ Y, int M, int N, int K, int rt) {
  extern __shared__ float4 xsm[];  // [MT][K/4] swizzled, then chunk sums [MT][K/32]
  __shared__ float part[32][MT];
  const int K4 = K / 4, K32 = K / 32;
  float* xsum = reinterpret_cast<float*>(xsm + (size_t)MT * K4);
  const int tid = threadIdx.x, hw = tid >> 4, li = tid & 15;
  const int ks = 32 / rt;
  const int r = hw % rt, kp = hw / rt;
  const int nunits = (K + kUnit - 1) / kUnit;
  const int nblocks = (N + rt - 1) / rt;

  UnitLoads2 L;
  int b = blockIdx.x;
  {
    const int n = b * rt + r;
#pragma unroll
    for (int u = 0; u < kMaxU; ++u)
      load_unit2<GROUP>(L, u, Wq, Sg, Zg, n < N ? n : 0, b < nblocks && n < N, kp, ks, li, nunits, K);
  }
  pdl_wait();  // X comes from the previous kernel; Y may still be read by it
  pdl_trigger();

  // stage the activations: thread = one 32-channel chunk of one token
  for (int idx = tid; idx < MT * K32; idx += kThreads2) {
    const int m = idx / K32, cq = idx - m * K32;
    uint4 raw[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      raw[t] = make_uint4(0, 0, 0, 0);
      if (m < M) raw[t] = ldg_nc_v4(X + (size_t)m * K + 32 * cq + 8 * t);
    }
    float sum = 0.0f;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float4 lo = make_float4(bf16_lo(raw[t].x), bf16_hi(raw[t].x), bf16_lo(raw[t].y), bf16_hi(raw[t].y));
      const float4 hi = make_float4(bf16_lo(raw[t].z), bf16_hi(raw[t].z), bf16_lo(raw[t].w), bf16_hi(raw[t].w));
      sum += lo.x; sum += lo.y; sum += lo.z; sum += lo.w;
      sum += hi.x; sum += hi.y; sum += hi.z; sum += hi.w;
      xsm[(size_t)m * K4 + xslot(8 * cq + 2 * t)] = lo;
      xsm[(size_t)m * K4 + xslot(8 * cq + 2 * t + 1)] = hi;
    }
    xsum[m * K32 + cq] = sum;
  }
  __syncthreads();

  for (; b < nblocks; b += gridDim.x) {
    const int nb = (b + (int)gridDim.x) * rt + r;
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
      const float zf = L.zf[u], sc = L.s[u];
      load_unit2<GROUP>(L, u, Wq, Sg, Zg, nb_ok ? nb : 0, nb_ok, kp, ks, li, nunits, K);
      if (!live) continue;
      float p0[MT], p1[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) p0[m] = p1[m] = 0.0f;
      const int q0 = c / 4;
#pragma unroll
      for (int qw = 0; qw < 4; ++qw) {
        float f[8];
        nib16(ws[qw], f);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const float4 xa = xsm[(size_t)m * K4 + xslot(q0 + 2 * qw)];
          const float4 xb = xsm[(size_t)m * K4 + xslot(q0 + 2 * qw + 1)];
          p0[m] = fmaf(xa.x, f[0], p0[m]);
          p1[m] = fmaf(xa.y, f[1], p1[m]);
          p0[m] = fmaf(xa.z, f[2], p0[m]);
          p1[m] = fmaf(xa.w, f[3], p1[m]);
          p0[m] = fmaf(xb.x, f[4], p0[m]);
          p1[m] = fmaf(xb.y, f[5], p1[m]);
          p0[m] = fmaf(xb.z, f[6], p0[m]);
          p1[m] = fmaf(xb.w, f[7], p1[m]);
        }
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[m] = fmaf(sc, (p0[m] + p1[m]) - zf * xsum[m * K32 + c / 32], acc[m]);
    }
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

template <int MT, int GROUP>
cudaError_t launch_smem_g(const uint16_t* X, const uint8_t* wq, const uint16_t* s, const uint16_t* z,
                          const uint16_t* bias, uint16_t* Y, int M, int N, int K, cudaStream_t st) {
  const size_t smem = (size_t)MT * K * 4 + (size_t)MT * (K / 32) * 4;
  // function attributes are per device: set them once for every device used
  static std::mutex mu;
  static bool set[64] = {};
  static cudaError_t res[64] = {};
  static int occ[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int blocks_per_sm = 1, sms = 148;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!set[dev]) {
      res[dev] = cudaFuncSetAttribute(w4a16_gemv_smem_kernel<MT, GROUP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kMaxXSmem);
      set[dev] = true;
    }
    if (res[dev] != cudaSuccess) return res[dev];
    (void)occ;
  }
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, w4a16_gemv_smem_kernel<MT, GROUP>, kThreads2,
                                                    smem) != cudaSuccess || blocks_per_sm < 1)
    blocks_per_sm = 1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms = 148;
  const int slots = blocks_per_sm * sms;
  // K split ks ways inside a CTA (at most kMaxU units of a row per
  // half-warp), raised while that leaves at least two row blocks per slot
  const int nunits = (K + kUnit - 1) / kUnit;
  int ks = 1;
  while (ks < 32 && (nunits + ks - 1) / ks > kMaxU) ks <<= 1;
  while (ks < 32 && ks * 2 <= nunits && (N + 32 / (2 * ks) - 1) / (32 / (2 * ks)) <= 2 * slots &&
         (N + 32 / ks - 1) / (32 / ks) < 2 * slots)
    ks <<= 1;
  const int rt = 32 / ks;
  const int nblocks = (N + rt - 1) / rt;
  const int grid = nblocks < slots ? nblocks : slots;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads2, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = vqlin::pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, w4a16_gemv_smem_kernel<MT, GROUP>, X, wq, s, z, bias, Y, M, N, K, rt);
}

template <int MT>
cudaError_t launch_smem(const uint16_t* X, const uint8_t* wq, const uint16_t* s, const uint16_t* z, int group,
                        const uint16_t* bias, uint16_t* Y, int M, int N, int K, cudaStream_t st) {
  switch (group) {
    case 64: return launch_smem_g<MT, 64>(X, wq, s, z, bias, Y, M, N, K, st);
    case 128: return launch_smem_g<MT, 128>(X, wq, s, z, bias, Y, M, N, K, st);
    default: return launch_smem_g<MT, 256>(X, wq, s, z, bias, Y, M, N, K, st);
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
  const int mt = M <= 1 ? 1 : (M <= 2 ? 2 : 4);
  // one token and a large matrix: activations staged on chip (float32 plus
  // chunk sums) when they fit.  Timed on B300: 1 x 11008 x 4096 17.0 -> 15.6
  // us, 1 x 32768 x 4096 39.5 -> 35.0 us; at 4096 x 4096 the staging costs
  // more than it saves (6.8 -> 7.5 us).  With two or four tokens that
  // variant's registers spill at 512 threads, so those keep the other one.
  if (mt == 1 && (long long)N * K >= (32ll << 20) && (size_t)K * 4 + (size_t)(K / 32) * 4 <= kMaxXSmem)
    return launched(launch_smem<1>(X, wq, s, z, group, bias, Y, M, N, K, st));
  if (mt == 1) return launched(launch_mt<1>(X, wq, s, z, group, bias, Y, M, N, K, st));
  if (mt == 2) return launched(launch_mt<2>(X, wq, s, z, group, bias, Y, M, N, K, st));
  return launched(launch_mt<4>(X, wq, s, z, group, bias, Y, M, N, K, st));  // M <= kW4a16GemvMaxM
}

}  // namespace vqlin
