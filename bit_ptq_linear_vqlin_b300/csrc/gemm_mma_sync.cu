// Integer GEMM of the W4A4 / W8A8 projections on warp-level integer MMAs.
//
//   acc[m, n] = sum_k xq[m, k] * wq[n, k]        (exact int32)
//   Y[m, n]   = bf16(float(acc) * sx[m] * sw[n] + bias[n])
//
// Method: "FoldQuantVLA" abstract (native integer execution of W4A4 / W8A8
// projections after per-token activation and per-channel weight quantization).
//
// This is the portable baseline path: `mma.sync` m16n8k64 (s4) or m16n8k32
// (s8), fed from a 4-stage cp.async pipeline with an XOR-swizzled shared
// memory layout.  Both operands are K-major byte rows, so one kernel serves
// both widths: a 32-byte row segment is one MMA k-step in either format.
#include "common.cuh"

namespace {

using namespace vqlin_dev;

constexpr int BM = 128, BN = 128, BKB = 64;  // tile rows, tile cols, K bytes per stage
constexpr int STAGES = 4;
constexpr int THREADS = 256;                 // 8 warps: 2 (M) x 4 (N), warp tile 64 x 32
constexpr int kStageBytes = (BM + BN) * BKB;
constexpr int kSmemBytes = STAGES * kStageBytes;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Byte offset of 16-byte chunk c (0..3) of row r inside a 64-byte-row tile.
__device__ __forceinline__ int swz(int r, int c) { return r * BKB + ((c ^ ((r >> 1) & 3)) << 4); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
  const int n = pred ? 16 : 0;  // zero-fill when out of range
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

template <int BITS>
__device__ __forceinline__ void mma_int(int32_t (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  if (BITS == 4) {
    asm volatile(
        "mma.sync.aligned.m16n8k64.row.col.s32.s4.s4.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

template <int BITS, bool RAW>
__global__ void __launch_bounds__(THREADS)
int_gemm_kernel(const uint8_t* __restrict__ A, const float* __restrict__ sx,
                const uint8_t* __restrict__ B, const float* __restrict__ sw,
                const uint16_t* __restrict__ bias, uint16_t* __restrict__ Y,
                int32_t* __restrict__ acc_out, int M, int N, int K) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int kbytes = BITS == 4 ? K / 2 : K;
  const int ktiles = kbytes / BKB;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp >> 2, wn = warp & 3;

  auto load_stage = [&](int stage, int kt) {
    uint8_t* sa = smem + stage * kStageBytes;
    uint8_t* sb = sa + BM * BKB;
    const int kb = kt * BKB;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int idx = tid + i * THREADS;  // 512 chunks per operand tile
      const int r = idx >> 2, c = idx & 3;
      const int gm = m0 + r, gn = n0 + r;
      cp_async16(smem_u32(sa + swz(r, c)), A + (size_t)(gm < M ? gm : 0) * kbytes + kb + c * 16, gm < M);
      cp_async16(smem_u32(sb + swz(r, c)), B + (size_t)(gn < N ? gn : 0) * kbytes + kb + c * 16, gn < N);
    }
  };

  int32_t acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][j][e] = 0;

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < ktiles) load_stage(s, s);
    asm volatile("cp.async.commit_group;");
  }

  for (int kt = 0; kt < ktiles; ++kt) {
    asm volatile("cp.async.wait_group %0;" ::"n"(STAGES - 2));
    __syncthreads();
    const int nk = kt + STAGES - 1;
    if (nk < ktiles) load_stage(nk % STAGES, nk);
    asm volatile("cp.async.commit_group;");

    const uint8_t* sa = smem + (kt % STAGES) * kStageBytes;
    const uint8_t* sb = sa + BM * BKB;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {  // two 32-byte MMA k-steps per stage
      uint32_t af[4][4], bf[4][2];
#pragma unroll
      for (int mi = 0; mi < 4; ++mi) {
        const int r = wm * 64 + mi * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = ks * 2 + (lane >> 4);
        ldsm_x4(smem_u32(sa + swz(r, c)), af[mi][0], af[mi][1], af[mi][2], af[mi][3]);
      }
#pragma unroll
      for (int nj = 0; nj < 2; ++nj) {
        const int r = wn * 32 + nj * 16 + (lane & 7) + (lane >> 4) * 8;
        const int c = ks * 2 + ((lane >> 3) & 1);
        ldsm_x4(smem_u32(sb + swz(r, c)), bf[2 * nj][0], bf[2 * nj][1], bf[2 * nj + 1][0],
                bf[2 * nj + 1][1]);
      }
#pragma unroll
      for (int mi = 0; mi < 4; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) mma_int<BITS>(acc[mi][ni], af[mi], bf[ni][0], bf[ni][1]);
    }
  }
  asm volatile("cp.async.wait_group 0;");

  // epilogue: fragment (row g / g+8, cols 2t, 2t+1)
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int mi = 0; mi < 4; ++mi) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int row = m0 + wm * 64 + mi * 16 + g + half * 8;
      if (row >= M) continue;
      const float sxr = RAW ? 0.0f : __ldg(sx + row);
#pragma unroll
      for (int ni = 0; ni < 4; ++ni) {
        const int col = n0 + wn * 32 + ni * 8 + 2 * t;
        const int32_t a0 = acc[mi][ni][half * 2], a1 = acc[mi][ni][half * 2 + 1];
        if (RAW) {
          if (col < N) acc_out[(size_t)row * N + col] = a0;
          if (col + 1 < N) acc_out[(size_t)row * N + col + 1] = a1;
          continue;
        }
        float y0 = 0.0f, y1 = 0.0f;
        if (col < N) {
          y0 = (float)a0 * sxr * __ldg(sw + col);
          if (bias) y0 += __uint_as_float((uint32_t)bias[col] << 16);
        }
        if (col + 1 < N) {
          y1 = (float)a1 * sxr * __ldg(sw + col + 1);
          if (bias) y1 += __uint_as_float((uint32_t)bias[col + 1] << 16);
        }
        uint16_t* yp = Y + (size_t)row * N + col;
        if (col + 1 < N && (N % 2) == 0) {
          *reinterpret_cast<uint32_t*>(yp) = pack_bf16x2(y0, y1);
        } else {
          if (col < N) yp[0] = f32_to_bf16_rn(y0);
          if (col + 1 < N) yp[1] = f32_to_bf16_rn(y1);
        }
      }
    }
  }
}

template <int BITS, bool RAW>
cudaError_t launch_t(const void* xq, const float* sx, const void* wq, const float* sw,
                     const uint16_t* bias, uint16_t* Y, int32_t* acc, int M, int N, int K,
                     cudaStream_t st) {
  auto kern = int_gemm_kernel<BITS, RAW>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(vqlin::ceil_div(N, BN), vqlin::ceil_div(M, BM));
  kern<<<grid, THREADS, kSmemBytes, st>>>((const uint8_t*)xq, sx, (const uint8_t*)wq, sw, bias, Y,
                                           acc, M, N, K);
  return cudaGetLastError();
}

}  // namespace

namespace vqlin {

cudaError_t launch_int_gemm(int bits, const void* xq, const float* sx, const void* wq,
                            const float* sw, const uint16_t* bias, uint16_t* Y, int32_t* acc,
                            int M, int N, int K, int* /*status*/, cudaStream_t st) {
  if (M == 0 || N == 0) return cudaSuccess;
  if (bits == 4)
    return acc ? launch_t<4, true>(xq, sx, wq, sw, bias, Y, acc, M, N, K, st)
               : launch_t<4, false>(xq, sx, wq, sw, bias, Y, acc, M, N, K, st);
  return acc ? launch_t<8, true>(xq, sx, wq, sw, bias, Y, acc, M, N, K, st)
             : launch_t<8, false>(xq, sx, wq, sw, bias, Y, acc, M, N, K, st);
}

}  // namespace vqlin
