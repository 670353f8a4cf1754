// Dense tensor-core rate of the two MMA kinds the projections run on, measured
// by the library itself: kind::f8f6f4 with e4m3 operands (the W4A4 GEMM's
// int4 codes) and kind::f16 with bf16 or f16 operands (W8A8 / W4A8 codes,
// W4A16).  Every CTA (one per SM) issues back-to-back 128 x N x K MMAs on
// operands that stay on chip, so the figure is the instruction's throughput,
// with no memory traffic: the roofline denominator of the GEMMs, and the cost
// of one small-N MMA that bounds the few-token kernels.
#include "common.cuh"
#include "tc_ptx.cuh"

namespace {

using namespace vqlin_dev;

// A from shared memory (descriptor a), B from shared memory, D in tensor memory.
__device__ __forceinline__ void mma_ss_warp(bool f8, uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                            uint32_t accumulate) {
  if (f8)
    asm volatile(
        "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// One CTA per SM.  Shared memory: A tile [128 rows x 128 B] and B tile
// [n rows x 128 B], every element 1.0, 128-byte swizzled; A also held in
// tensor memory columns [256, 288).  Warps 0 .. issuers-1 each issue `iters`
// k-blocks of four MMAs (K = 32 e4m3 or 16 bf16 each, 128 bytes of every
// row); issuer w's MMA k accumulates into accumulator w * per + k % per
// (per = accumulators / issuers chains each, columns [that * n, ...)), then
// each issuer commits once; cycles[cta] = clock64 span of issuer 0.
__global__ void __launch_bounds__(128, 1)
mma_rate_kernel(int f8, int a_tmem, int n, int nacc, int issuers, int iters, long long* cycles, int* status) {
  extern __shared__ uint8_t smem_dyn[];
  __shared__ __align__(8) uint64_t done;
  __shared__ uint32_t s_tmem;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  uint8_t* a_tile = base;
  uint8_t* b_tile = base + 128 * 128;
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t one = f8 ? 0x38383838u : 0x3F803F80u;  // e4m3 / bf16 ones
  for (int i = tid; i < (128 + n) * 128 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(base)[i] = make_uint4(one, one, one, one);
  fence_proxy_async_smem();
  if (tid == 0) {
    mbar_init(&done, issuers);
    mbar_init_fence();
  }
  if (warp == 0) tmem_alloc(&s_tmem, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  {
    // A in tensor memory: warp w covers lanes 32w..32w+31, 32 columns
    uint32_t z[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = one;
    const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16) + 256;
    tmem_st_x16(ta, z);
    tmem_st_x16(ta + 16, z);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp < issuers) {
    const uint32_t id = idesc_f32acc(f8 ? 0u : 1u, 128, n);
    const uint64_t da = sdesc_sw128(a_tile), db = sdesc_sw128(b_tile);
    const uint32_t ta = tmem + 256;
    const int per = nacc / issuers;  // accumulation chains of this issuer
    uint32_t d[4], first[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      d[k] = tmem + (uint32_t)((warp * per + k % per) * n);
      first[k] = k < per ? 0u : 1u;
    }
    const long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
      // per MMA: 32 bytes along K (8 tensor-memory columns of A)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t acc = i > 0 ? 1u : first[k];
        if (a_tmem) {
          if (f8)
            mma_f8f6f4_ta_warp(d[k], ta + 8 * k, db + 2 * k, id, acc);
          else
            mma_f16_ta_warp(d[k], ta + 8 * k, db + 2 * k, id, acc);
        } else {
          mma_ss_warp(f8 != 0, d[k], da + 2 * k, db + 2 * k, id, acc);
        }
      }
    }
    tc_commit_warp(&done);
    const bool ok = mbar_wait_bounded(&done, 0, 2000000000ull, nullptr);
    const long long t1 = clock64();
    if (!ok && (tid & 31) == 0) atomicCAS(status, 0, (int)VQLIN_ERR_TIMEOUT);
    if (warp == 0 && (tid & 31) == 0) cycles[blockIdx.x] = t1 - t0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

extern "C" vqlin_status vqlin_measure_mma_rate(int kind, int a_in_tmem, int n, int accumulators, int issuers,
                                               int iters, int ctas, long long* cycles_dev, double* tflops,
                                               double* cycles_per_mma, void* stream) {
  if ((kind != 0 && kind != 1) || n < 16 || n > 256 || (n % 16) != 0 || iters < 1 || iters > (1 << 20) ||
      accumulators < 1 || accumulators > 4 || (accumulators & (accumulators - 1)) != 0 ||
      accumulators * n > 256 || issuers < 1 || issuers > accumulators || accumulators % issuers != 0 ||
      ctas < 1 || ctas > 4096 || cycles_dev == nullptr || tflops == nullptr || cycles_per_mma == nullptr)
    return vqlin::fail(VQLIN_ERR_INVALID_ARG, "measure_mma_rate: bad arguments");
  int* status = vqlin::device_status_word();
  if (status == nullptr) return vqlin::fail(VQLIN_ERR_CUDA, "no device status word");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t dyn = 1024 + (size_t)(128 + n) * 128;
  // one CTA per SM: ask for more than half of an SM's shared memory
  const size_t dyn_pad = dyn < 120 * 1024 ? 120 * 1024 : dyn;
  cudaError_t e = cudaFuncSetAttribute(mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn_pad);
  if (e != cudaSuccess) return vqlin::fail(VQLIN_ERR_CUDA, "measure_mma_rate: %s", cudaGetErrorString(e));
  cudaEvent_t a = nullptr, b = nullptr;
  vqlin_status out = VQLIN_OK;
  do {
    if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess) {
      out = vqlin::fail(VQLIN_ERR_CUDA, "measure_mma_rate: event creation failed");
      break;
    }
    mma_rate_kernel<<<ctas, 128, dyn_pad, st>>>(kind == 0, a_in_tmem, n, accumulators, issuers, 16, cycles_dev,
                                                 status);  // warm-up
    cudaEventRecord(a, st);
    mma_rate_kernel<<<ctas, 128, dyn_pad, st>>>(kind == 0, a_in_tmem, n, accumulators, issuers, iters, cycles_dev,
                                                 status);
    cudaEventRecord(b, st);
    e = cudaEventSynchronize(b);
    if (e != cudaSuccess) {
      out = vqlin::fail(VQLIN_ERR_CUDA, "measure_mma_rate: %s", cudaGetErrorString(e));
      break;
    }
    vqlin::launched(e, 2);
    float ms = 0.0f;
    cudaEventElapsedTime(&ms, a, b);
    const int kdim = kind == 0 ? 32 : 16;  // K of one MMA
    const double flops = 2.0 * 128.0 * n * kdim * 4.0 * iters * ctas * issuers;
    *tflops = flops / (ms * 1e-3) / 1e12;
    long long* h = new long long[ctas];
    e = cudaMemcpy(h, cycles_dev, sizeof(long long) * ctas, cudaMemcpyDeviceToHost);
    double avg = 0.0;
    for (int i = 0; i < ctas; ++i) avg += (double)h[i];
    delete[] h;
    if (e != cudaSuccess) {
      out = vqlin::fail(VQLIN_ERR_CUDA, "measure_mma_rate: %s", cudaGetErrorString(e));
      break;
    }
    *cycles_per_mma = avg / ctas / (4.0 * iters * issuers);
  } while (0);
  if (a) cudaEventDestroy(a);
  if (b) cudaEventDestroy(b);
  return out;
}
