// C ABI of libvqlin: argument validation, status reporting, dispatch.
//
// Every entry point checks its arguments on the host and launches nothing
// when they are invalid.  No entry point allocates per call; the only device
// memory the library owns is the cuBLASLt workspace of the bf16 baseline,
// created once per device by vqlin_init() or on first use, and released by
// vqlin_shutdown().
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <map>
#include <mutex>
#include <string>
#include <tuple>

#include <cublasLt.h>

#include "common.cuh"

// Per-device status word written by kernels whose bounded waits run out.
__device__ int g_vqlin_status = 0;

namespace vqlin {

namespace {

thread_local std::string t_last_error;

struct DeviceState {
  bool ready = false;
  cublasLtHandle_t lt = nullptr;
  void* workspace = nullptr;
  size_t workspace_bytes = 0;
  int* status_word = nullptr;
  std::map<std::tuple<int, int, int, bool>, cublasLtMatmulAlgo_t> algos;
};

std::mutex g_mu;
DeviceState g_dev[64];

vqlin_status cuda_fail(cudaError_t e, const char* what) {
  return fail(VQLIN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Returns the state of the current device, creating it on first use.
vqlin_status device_state(DeviceState** out, bool need_blas) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(VQLIN_ERR_CUDA, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& s = g_dev[dev];
  if (!s.status_word) {
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&s.status_word), g_vqlin_status);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status word)");
  }
  if (need_blas && !s.ready) {
    if (cublasLtCreate(&s.lt) != CUBLAS_STATUS_SUCCESS) return fail(VQLIN_ERR_CUDA, "cublasLtCreate failed");
    s.workspace_bytes = 64u << 20;
    e = cudaMalloc(&s.workspace, s.workspace_bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(cuBLASLt workspace)");
    s.ready = true;
  }
  *out = &s;
  return VQLIN_OK;
}

vqlin_status check_launch(cudaError_t e, const char* what) {
  return e == cudaSuccess ? VQLIN_OK : cuda_fail(e, what);
}

}  // namespace

vqlin_status fail(vqlin_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

namespace {
std::atomic<unsigned long long> g_launches{0};
}  // namespace

cudaError_t launched(cudaError_t e, int n) {
  if (e == cudaSuccess) g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed);
  return e;
}

int* device_status_word() {
  DeviceState* s = nullptr;
  return device_state(&s, false) == VQLIN_OK ? s->status_word : nullptr;
}

}  // namespace vqlin

extern "C" vqlin_status vqlin_kernel_launch_count(unsigned long long* count) {
  if (count == nullptr) return vqlin::fail(VQLIN_ERR_INVALID_ARG, "vqlin_kernel_launch_count: count is null");
  *count = vqlin::g_launches.load(std::memory_order_relaxed);
  return VQLIN_OK;
}

extern "C" vqlin_status vqlin_init(void) {
  vqlin::DeviceState* s = nullptr;
  return vqlin::device_state(&s, true);
}

extern "C" vqlin_status vqlin_shutdown(void) {
  int cur = -1;
  const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
  vqlin_status out = VQLIN_OK;
  std::lock_guard<std::mutex> lock(vqlin::g_mu);
  for (int d = 0; d < 64; ++d) {
    vqlin::DeviceState& s = vqlin::g_dev[d];
    if (!s.ready) continue;
    // the handle and workspace may still be in use by queued work on that device
    if (cudaSetDevice(d) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
      out = vqlin::fail(VQLIN_ERR_CUDA, "vqlin_shutdown: device %d did not synchronise", d);
    if (s.lt != nullptr) cublasLtDestroy(s.lt);
    if (s.workspace != nullptr) cudaFree(s.workspace);
    s.lt = nullptr;
    s.workspace = nullptr;
    s.workspace_bytes = 0;
    s.algos.clear();
    s.ready = false;
  }
  if (have_cur) cudaSetDevice(cur);
  return out;
}

using vqlin::fail;

#define REQUIRE(cond, code, ...)              \
  do {                                        \
    if (!(cond)) return fail(code, __VA_ARGS__); \
  } while (0)

#define REQUIRE_PTR(p) REQUIRE((p) != nullptr, VQLIN_ERR_INVALID_ARG, "%s is NULL", #p)
#define REQUIRE_ALIGNED(p) \
  REQUIRE(vqlin::aligned16(p), VQLIN_ERR_MISALIGNED, "%s is not 16-byte aligned", #p)

extern "C" {

int vqlin_version(void) { return 500; }

const char* vqlin_status_string(vqlin_status s) {
  switch (s) {
    case VQLIN_OK: return "VQLIN_OK";
    case VQLIN_ERR_INVALID_ARG: return "VQLIN_ERR_INVALID_ARG";
    case VQLIN_ERR_UNSUPPORTED_SHAPE: return "VQLIN_ERR_UNSUPPORTED_SHAPE";
    case VQLIN_ERR_MISALIGNED: return "VQLIN_ERR_MISALIGNED";
    case VQLIN_ERR_CUDA: return "VQLIN_ERR_CUDA";
    case VQLIN_ERR_TIMEOUT: return "VQLIN_ERR_TIMEOUT";
    case VQLIN_ERR_DEVICE_ASSERT: return "VQLIN_ERR_DEVICE_ASSERT";
  }
  return "VQLIN_ERR_UNKNOWN";
}

const char* vqlin_last_error_message(void) { return vqlin::t_last_error.c_str(); }

vqlin_status vqlin_get_last_device_error(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return vqlin::fail(VQLIN_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_vqlin_status, sizeof(int));
  if (e != cudaSuccess) return vqlin::fail(VQLIN_ERR_CUDA, "reading status word: %s", cudaGetErrorString(e));
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_vqlin_status, &zero, sizeof(int));
    if (e != cudaSuccess) return vqlin::fail(VQLIN_ERR_CUDA, "clearing status word: %s", cudaGetErrorString(e));
    return vqlin::fail(static_cast<vqlin_status>(v), "device reported status %d", v);
  }
  return VQLIN_OK;
}

vqlin_status vqlin_quantize_weights_rtn_scaled(const uint16_t* W, int N, int K, int bits, int hadamard_block,
                                               const float* channel_scale, void* q_out, float* scale_out,
                                               void* stream) {
  REQUIRE(N >= 0 && K > 0, VQLIN_ERR_INVALID_ARG, "bad sizes N=%d K=%d", N, K);
  REQUIRE(bits == 4 || bits == 8, VQLIN_ERR_INVALID_ARG, "bits must be 4 or 8 (got %d)", bits);
  REQUIRE(hadamard_block == 0 || hadamard_block == 64 || hadamard_block == 128, VQLIN_ERR_INVALID_ARG,
          "hadamard_block must be 0, 64 or 128 (got %d)", hadamard_block);
  REQUIRE(K % 32 == 0, VQLIN_ERR_UNSUPPORTED_SHAPE, "K=%d is not a multiple of 32", K);
  REQUIRE(hadamard_block == 0 || K % hadamard_block == 0, VQLIN_ERR_UNSUPPORTED_SHAPE,
          "K=%d is not a multiple of the Hadamard block %d", K, hadamard_block);
  REQUIRE(K <= vqlin::kWeightQuantMaxK, VQLIN_ERR_UNSUPPORTED_SHAPE, "K=%d exceeds %d", K,
          vqlin::kWeightQuantMaxK);
  if (N == 0) return VQLIN_OK;
  REQUIRE_PTR(W); REQUIRE_PTR(channel_scale); REQUIRE_PTR(q_out); REQUIRE_PTR(scale_out);
  REQUIRE_ALIGNED(W); REQUIRE_ALIGNED(channel_scale); REQUIRE_ALIGNED(q_out); REQUIRE_ALIGNED(scale_out);
  return vqlin::check_launch(vqlin::launch_weight_quant_sym(W, N, K, bits, hadamard_block, q_out, scale_out,
                                                           static_cast<cudaStream_t>(stream), channel_scale),
                             "weight_quant_sym");
}

vqlin_status vqlin_quantize_weights_rtn(const uint16_t* W, int N, int K, int bits, int symmetric,
                                        int group_size, int hadamard_block, void* q_out,
                                        void* scale_out, void* zero_out, void* stream) {
  REQUIRE(N >= 0 && K > 0, VQLIN_ERR_INVALID_ARG, "bad sizes N=%d K=%d", N, K);
  REQUIRE(bits == 4 || bits == 8, VQLIN_ERR_INVALID_ARG, "bits must be 4 or 8 (got %d)", bits);
  REQUIRE(hadamard_block == 0 || hadamard_block == 64 || hadamard_block == 128, VQLIN_ERR_INVALID_ARG,
          "hadamard_block must be 0, 64 or 128 (got %d)", hadamard_block);
  REQUIRE(K % 32 == 0, VQLIN_ERR_UNSUPPORTED_SHAPE, "K=%d is not a multiple of 32", K);
  REQUIRE(K <= vqlin::kWeightQuantMaxK, VQLIN_ERR_UNSUPPORTED_SHAPE, "K=%d exceeds %d", K,
          vqlin::kWeightQuantMaxK);
  if (N == 0) return VQLIN_OK;
  REQUIRE_PTR(W); REQUIRE_PTR(q_out); REQUIRE_PTR(scale_out);
  REQUIRE_ALIGNED(W); REQUIRE_ALIGNED(q_out); REQUIRE_ALIGNED(scale_out);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (symmetric) {
    REQUIRE(group_size == 0, VQLIN_ERR_INVALID_ARG, "symmetric weights are per channel (group_size 0)");
    REQUIRE(zero_out == nullptr, VQLIN_ERR_INVALID_ARG, "zero_out must be NULL for symmetric weights");
    REQUIRE(hadamard_block == 0 || K % hadamard_block == 0, VQLIN_ERR_UNSUPPORTED_SHAPE,
            "K=%d is not a multiple of the Hadamard block %d", K, hadamard_block);
    return vqlin::check_launch(vqlin::launch_weight_quant_sym(W, N, K, bits, hadamard_block, q_out,
                                                               static_cast<float*>(scale_out), st),
                               "weight_quant_sym");
  }
  REQUIRE(bits == 4, VQLIN_ERR_INVALID_ARG, "asymmetric weights are int4");
  REQUIRE(hadamard_block == 0, VQLIN_ERR_INVALID_ARG, "asymmetric (weight-only) weights are not rotated");
  REQUIRE(group_size == 64 || group_size == 128 || group_size == 256, VQLIN_ERR_INVALID_ARG,
          "group_size must be 64, 128 or 256 (got %d)", group_size);
  REQUIRE(K % group_size == 0, VQLIN_ERR_UNSUPPORTED_SHAPE, "K=%d is not a multiple of the group %d", K,
          group_size);
  REQUIRE_PTR(zero_out); REQUIRE_ALIGNED(zero_out);
  return vqlin::check_launch(
      vqlin::launch_weight_quant_asym(W, N, K, group_size, static_cast<uint8_t*>(q_out),
                                      static_cast<uint16_t*>(scale_out), static_cast<uint16_t*>(zero_out), st),
      "weight_quant_asym");
}

vqlin_status vqlin_act_hadamard_quant(const uint16_t* X, int M, int K, int bits, int hadamard_block,
                                      const float* static_scale, void* q_out, float* scale_out,
                                      void* stream) {
  return vqlin_act_hadamard_quant_scaled(X, M, K, bits, hadamard_block, nullptr, static_scale, q_out, scale_out,
                                         stream);
}

vqlin_status vqlin_act_hadamard_quant_scaled(const uint16_t* X, int M, int K, int bits, int hadamard_block,
                                             const float* channel_scale, const float* static_scale, void* q_out,
                                             float* scale_out, void* stream) {
  REQUIRE(M >= 0 && K > 0, VQLIN_ERR_INVALID_ARG, "bad sizes M=%d K=%d", M, K);
  REQUIRE(bits == 4 || bits == 8, VQLIN_ERR_INVALID_ARG, "bits must be 4 or 8 (got %d)", bits);
  REQUIRE(hadamard_block == 0 || hadamard_block == 64 || hadamard_block == 128, VQLIN_ERR_INVALID_ARG,
          "hadamard_block must be 0, 64 or 128 (got %d)", hadamard_block);
  REQUIRE(K % 32 == 0, VQLIN_ERR_UNSUPPORTED_SHAPE, "K=%d is not a multiple of 32", K);
  REQUIRE(hadamard_block == 0 || K % hadamard_block == 0, VQLIN_ERR_UNSUPPORTED_SHAPE,
          "K=%d is not a multiple of the Hadamard block %d", K, hadamard_block);
  REQUIRE(K <= vqlin::kActQuantMaxK, VQLIN_ERR_UNSUPPORTED_SHAPE, "K=%d exceeds %d", K, vqlin::kActQuantMaxK);
  if (M == 0) return VQLIN_OK;
  REQUIRE_PTR(X); REQUIRE_PTR(q_out); REQUIRE_PTR(scale_out);
  REQUIRE_ALIGNED(X); REQUIRE_ALIGNED(q_out);
  REQUIRE(vqlin::aligned16(scale_out) || (reinterpret_cast<uintptr_t>(scale_out) & 3) == 0,
          VQLIN_ERR_MISALIGNED, "scale_out is not 4-byte aligned");
  if (channel_scale != nullptr) REQUIRE_ALIGNED(channel_scale);
  return vqlin::check_launch(vqlin::launch_act_quant(X, M, K, bits, hadamard_block, static_scale, q_out,
                                                     scale_out, static_cast<cudaStream_t>(stream), channel_scale),
                             "act_hadamard_quant");
}

// bits: 4 (W4A4), 8 (W8A8); w4a8: int4 weights against int8 activations
static vqlin_status linear_int(int bits, const void* xq, const float* sx, const void* wq, const float* sw,
                               const uint16_t* bias, uint16_t* Y, int32_t* acc, int M, int N, int K,
                               void* stream, bool w4a8 = false) {
  REQUIRE(M >= 0 && N >= 0 && K > 0, VQLIN_ERR_INVALID_ARG, "bad sizes M=%d N=%d K=%d", M, N, K);
  const int kmul = bits == 4 ? 128 : 64;
  const int kmax = bits == 4 ? vqlin::kGemmW4MaxK : vqlin::kGemmW8MaxK;
  REQUIRE(K % kmul == 0, VQLIN_ERR_UNSUPPORTED_SHAPE, "K=%d is not a multiple of %d", K, kmul);
  REQUIRE(K <= kmax, VQLIN_ERR_UNSUPPORTED_SHAPE, "K=%d exceeds %d", K, kmax);
  if (M == 0 || N == 0) return VQLIN_OK;
  REQUIRE_PTR(xq); REQUIRE_PTR(wq);
  REQUIRE_ALIGNED(xq); REQUIRE_ALIGNED(wq);
  if (acc) {
    REQUIRE_ALIGNED(acc);
  } else {
    REQUIRE_PTR(sx); REQUIRE_PTR(sw); REQUIRE_PTR(Y);
    REQUIRE_ALIGNED(Y);
  }
  int* status = vqlin::device_status_word();
  REQUIRE(status != nullptr, VQLIN_ERR_CUDA, "no device status word");
  if (w4a8)
    return vqlin::launch_int_gemm_w4a8(xq, sx, wq, sw, bias, Y, acc, M, N, K, status,
                                       static_cast<cudaStream_t>(stream));
  // few tokens: the kernel that keeps every operand of its K range on chip
  if (bits == 4 && acc == nullptr && M <= vqlin::kLowlatMaxM && K <= vqlin::kLowlatMaxK &&
      vqlin::lowlat_one_wave(false, 128, M, N, K))
    return vqlin::launch_w4a4_codes_lowlat(static_cast<const uint8_t*>(xq), sx, static_cast<const uint8_t*>(wq), sw,
                                           bias, Y, M, N, K, status, static_cast<cudaStream_t>(stream));
  return vqlin::launch_int_gemm(bits, xq, sx, wq, sw, bias, Y, acc, M, N, K, status,
                                static_cast<cudaStream_t>(stream));
}

vqlin_status vqlin_linear_w4a4(const uint8_t* xq, const float* sx, const uint8_t* wq, const float* sw,
                               const uint16_t* bias, uint16_t* Y, int M, int N, int K, void* stream) {
  return linear_int(4, xq, sx, wq, sw, bias, Y, nullptr, M, N, K, stream);
}

vqlin_status vqlin_linear_w8a8(const uint16_t* xq, const float* sx, const uint8_t* wq, const float* sw,
                               const uint16_t* bias, uint16_t* Y, int M, int N, int K, void* stream) {
  return linear_int(8, xq, sx, wq, sw, bias, Y, nullptr, M, N, K, stream);
}

vqlin_status vqlin_linear_w4a8(const uint16_t* xq, const float* sx, const uint8_t* wq, const float* sw,
                               const uint16_t* bias, uint16_t* Y, int M, int N, int K, void* stream) {
  return linear_int(8, xq, sx, wq, sw, bias, Y, nullptr, M, N, K, stream, true);
}

vqlin_status vqlin_debug_gemm_w4a8_s32(const uint16_t* xq, const uint8_t* wq, int32_t* acc, int M, int N, int K,
                                       void* stream) {
  REQUIRE_PTR(acc);
  return linear_int(8, xq, nullptr, wq, nullptr, nullptr, nullptr, acc, M, N, K, stream, true);
}

// The static-scale W4A4 projection, optionally with channel scaling (chan).
static vqlin_status linear_w4a4_static_impl(const uint16_t* X, const float* static_scale, const float* chan,
                                     int hadamard_block, const uint8_t* wq, const float* sw, const uint16_t* bias,
                                     uint16_t* Y, uint8_t* xq_out, int M, int N, int K, void* stream) {
  REQUIRE(M >= 0 && N >= 0 && K > 0, VQLIN_ERR_INVALID_ARG, "bad sizes M=%d N=%d K=%d", M, N, K);
  REQUIRE(hadamard_block == 64 || hadamard_block == 128, VQLIN_ERR_INVALID_ARG,
          "hadamard_block must be 64 or 128 (got %d)", hadamard_block);
  REQUIRE(K % 128 == 0, VQLIN_ERR_UNSUPPORTED_SHAPE, "K=%d is not a multiple of 128", K);
  REQUIRE(K <= vqlin::kGemmW4MaxK, VQLIN_ERR_UNSUPPORTED_SHAPE, "K=%d exceeds %d", K, vqlin::kGemmW4MaxK);
  if (M == 0 || N == 0) return VQLIN_OK;
  REQUIRE_PTR(X); REQUIRE_PTR(static_scale); REQUIRE_PTR(wq); REQUIRE_PTR(sw); REQUIRE_PTR(Y); REQUIRE_PTR(xq_out);
  REQUIRE_ALIGNED(X); REQUIRE_ALIGNED(wq); REQUIRE_ALIGNED(Y); REQUIRE_ALIGNED(xq_out);
  if (chan != nullptr) REQUIRE_ALIGNED(chan);
  int* status = vqlin::device_status_word();
  REQUIRE(status != nullptr, VQLIN_ERR_CUDA, "no device status word");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (K <= vqlin::kLowlatMaxK && M <= vqlin::kLowlatMaxM && vqlin::lowlat_one_wave(true, hadamard_block, M, N, K)) {
    if (!vqlin::static_two_launch(K))
      return vqlin::launch_w4a4_static_lowlat(X, static_scale, hadamard_block, xq_out, wq, sw, bias, Y, M, N, K,
                                              status, st, chan);
    if (vqlin::lowlat_one_wave(false, 128, M, N, K)) {
      // long K: the activation kernel, then the few-token GEMM on its codes
      vqlin_status r = vqlin::check_launch(
          vqlin::launch_act_quant(X, M, K, 4, hadamard_block, static_scale, xq_out, nullptr, st, chan),
          "act_hadamard_quant");
      if (r != VQLIN_OK) return r;
      return vqlin::launch_w4a4_codes_lowlat(xq_out, static_scale, wq, sw, bias, Y, M, N, K, status, st, 0);
    }
  }
  // longer K or more than one wave: the activation kernel writes the codes,
  // the throughput GEMM uses them
  vqlin_status r = vqlin::check_launch(
      vqlin::launch_act_quant(X, M, K, 4, hadamard_block, static_scale, xq_out, nullptr, st, chan),
      "act_hadamard_quant");
  if (r != VQLIN_OK) return r;
  return vqlin::launch_int_gemm_static_scale(xq_out, static_scale, wq, sw, bias, Y, M, N, K, status, st);
}

vqlin_status vqlin_linear_w4a4_static(const uint16_t* X, const float* static_scale, int hadamard_block,
                                      const uint8_t* wq, const float* sw, const uint16_t* bias, uint16_t* Y,
                                      uint8_t* xq_out, int M, int N, int K, void* stream) {
  return linear_w4a4_static_impl(X, static_scale, nullptr, hadamard_block, wq, sw, bias, Y, xq_out, M, N, K, stream);
}

vqlin_status vqlin_linear_w4a4_static_scaled(const uint16_t* X, const float* static_scale,
                                             const float* channel_scale, int hadamard_block, const uint8_t* wq,
                                             const float* sw, const uint16_t* bias, uint16_t* Y, uint8_t* xq_out,
                                             int M, int N, int K, void* stream) {
  if (M > 0 && N > 0) REQUIRE_PTR(channel_scale);
  return linear_w4a4_static_impl(X, static_scale, channel_scale, hadamard_block, wq, sw, bias, Y, xq_out, M, N, K,
                                 stream);
}

vqlin_status vqlin_debug_gemm_s32(int bits, const void* xq, const void* wq, int32_t* acc, int M, int N, int K,
                                  void* stream) {
  REQUIRE(bits == 4 || bits == 8, VQLIN_ERR_INVALID_ARG, "bits must be 4 or 8 (got %d)", bits);
  REQUIRE_PTR(acc);
  return linear_int(bits, xq, nullptr, wq, nullptr, nullptr, nullptr, acc, M, N, K, stream);
}

vqlin_status vqlin_debug_gemm_withheld_loads(int bits, const void* xq, const void* wq, int32_t* acc, int M,
                                             int N, int K, uint64_t limit_ns, void* stream) {
  REQUIRE(bits == 4 || bits == 8, VQLIN_ERR_INVALID_ARG, "bits must be 4 or 8 (got %d)", bits);
  REQUIRE(M > 0 && N > 0 && K > 0, VQLIN_ERR_INVALID_ARG, "bad sizes M=%d N=%d K=%d", M, N, K);
  const int kmul = bits == 4 ? 128 : 64;
  const int kmax = bits == 4 ? vqlin::kGemmW4MaxK : vqlin::kGemmW8MaxK;
  REQUIRE(K % kmul == 0 && K <= kmax, VQLIN_ERR_UNSUPPORTED_SHAPE, "unsupported K=%d", K);
  REQUIRE(limit_ns > 0 && limit_ns <= 2000000000ull, VQLIN_ERR_INVALID_ARG, "limit_ns must be in (0, 2e9]");
  REQUIRE_PTR(xq); REQUIRE_PTR(wq); REQUIRE_PTR(acc);
  REQUIRE_ALIGNED(xq); REQUIRE_ALIGNED(wq); REQUIRE_ALIGNED(acc);
  int* status = vqlin::device_status_word();
  REQUIRE(status != nullptr, VQLIN_ERR_CUDA, "no device status word");
  return vqlin::launch_int_gemm_withheld(bits, xq, wq, acc, M, N, K, status, limit_ns,
                                         static_cast<cudaStream_t>(stream));
}

vqlin_status vqlin_act_adaln_hadamard_quant(const uint16_t* X, int M, int K, int bits, int hadamard_block,
                                            const float* ada_scale, const float* ada_shift, float eps,
                                            const float* static_scale, void* q_out, float* scale_out, void* stream) {
  REQUIRE(M >= 0 && K > 0, VQLIN_ERR_INVALID_ARG, "bad sizes M=%d K=%d", M, K);
  REQUIRE(bits == 4 || bits == 8, VQLIN_ERR_INVALID_ARG, "bits must be 4 or 8 (got %d)", bits);
  REQUIRE(hadamard_block == 0 || hadamard_block == 64 || hadamard_block == 128, VQLIN_ERR_INVALID_ARG,
          "hadamard_block must be 0, 64 or 128 (got %d)", hadamard_block);
  REQUIRE(K % 32 == 0, VQLIN_ERR_UNSUPPORTED_SHAPE, "K=%d is not a multiple of 32", K);
  REQUIRE(hadamard_block == 0 || K % hadamard_block == 0, VQLIN_ERR_UNSUPPORTED_SHAPE,
          "K=%d is not a multiple of the Hadamard block %d", K, hadamard_block);
  REQUIRE(K <= vqlin::kActQuantMaxK, VQLIN_ERR_UNSUPPORTED_SHAPE, "K=%d exceeds %d", K, vqlin::kActQuantMaxK);
  REQUIRE(eps >= 0.0f && eps == eps, VQLIN_ERR_INVALID_ARG, "eps must be a non-negative number");
  if (M == 0) return VQLIN_OK;
  REQUIRE_PTR(X); REQUIRE_PTR(ada_scale); REQUIRE_PTR(ada_shift); REQUIRE_PTR(q_out); REQUIRE_PTR(scale_out);
  REQUIRE_ALIGNED(X); REQUIRE_ALIGNED(ada_scale); REQUIRE_ALIGNED(ada_shift); REQUIRE_ALIGNED(q_out);
  REQUIRE((reinterpret_cast<uintptr_t>(scale_out) & 3) == 0, VQLIN_ERR_MISALIGNED, "scale_out is not 4-byte aligned");
  return vqlin::check_launch(vqlin::launch_act_quant(X, M, K, bits, hadamard_block, static_scale, q_out, scale_out,
                                                     static_cast<cudaStream_t>(stream), nullptr, ada_scale, ada_shift,
                                                     eps),
                             "act_adaln_hadamard_quant");
}

vqlin_status vqlin_composite_rotation_prepare(const uint16_t* W, int N, int K, int block, int32_t* perm_out,
                                              double* R_out, void* stream) {
  REQUIRE(N > 0 && K > 0, VQLIN_ERR_INVALID_ARG, "bad sizes N=%d K=%d", N, K);
  REQUIRE(block == 64 || block == 128, VQLIN_ERR_INVALID_ARG, "block must be 64 or 128 (got %d)", block);
  REQUIRE(K % block == 0, VQLIN_ERR_UNSUPPORTED_SHAPE, "K=%d is not a multiple of the block %d", K, block);
  REQUIRE(K <= vqlin::kWeightQuantMaxK, VQLIN_ERR_UNSUPPORTED_SHAPE, "K=%d exceeds %d", K, vqlin::kWeightQuantMaxK);
  REQUIRE_PTR(W); REQUIRE_PTR(perm_out); REQUIRE_PTR(R_out);
  REQUIRE_ALIGNED(W); REQUIRE_ALIGNED(perm_out); REQUIRE_ALIGNED(R_out);
  int* status = vqlin::device_status_word();
  REQUIRE(status != nullptr, VQLIN_ERR_CUDA, "no device status word");
  return vqlin::check_launch(vqlin::launch_composite_prepare(W, N, K, block, perm_out, R_out, status,
                                                             static_cast<cudaStream_t>(stream)),
                             "composite_rotation_prepare");
}

vqlin_status vqlin_quantize_weights_composite(const uint16_t* W, int N, int K, int bits, int block,
                                              const int32_t* perm, const double* R, void* q_out, float* scale_out,
                                              void* stream) {
  REQUIRE(N >= 0 && K > 0, VQLIN_ERR_INVALID_ARG, "bad sizes N=%d K=%d", N, K);
  REQUIRE(bits == 4 || bits == 8, VQLIN_ERR_INVALID_ARG, "bits must be 4 or 8 (got %d)", bits);
  REQUIRE(block == 64 || block == 128, VQLIN_ERR_INVALID_ARG, "block must be 64 or 128 (got %d)", block);
  REQUIRE(K % block == 0, VQLIN_ERR_UNSUPPORTED_SHAPE, "K=%d is not a multiple of the block %d", K, block);
  if (N == 0) return VQLIN_OK;
  REQUIRE_PTR(W); REQUIRE_PTR(perm); REQUIRE_PTR(R); REQUIRE_PTR(q_out); REQUIRE_PTR(scale_out);
  REQUIRE_ALIGNED(W); REQUIRE_ALIGNED(perm); REQUIRE_ALIGNED(R); REQUIRE_ALIGNED(q_out); REQUIRE_ALIGNED(scale_out);
  return vqlin::check_launch(vqlin::launch_weight_quant_composite(W, N, K, bits, block, perm, R,
                                                                  static_cast<uint8_t*>(q_out), scale_out,
                                                                  static_cast<cudaStream_t>(stream)),
                             "quantize_weights_composite");
}

vqlin_status vqlin_act_composite_quant(const uint16_t* X, int M, int K, int bits, int block, const int32_t* perm,
                                       const double* R, void* q_out, float* scale_out, void* stream) {
  REQUIRE(M >= 0 && K > 0, VQLIN_ERR_INVALID_ARG, "bad sizes M=%d K=%d", M, K);
  REQUIRE(bits == 4 || bits == 8, VQLIN_ERR_INVALID_ARG, "bits must be 4 or 8 (got %d)", bits);
  REQUIRE(block == 64 || block == 128, VQLIN_ERR_INVALID_ARG, "block must be 64 or 128 (got %d)", block);
  REQUIRE(K % block == 0, VQLIN_ERR_UNSUPPORTED_SHAPE, "K=%d is not a multiple of the block %d", K, block);
  if (M == 0) return VQLIN_OK;
  REQUIRE_PTR(X); REQUIRE_PTR(perm); REQUIRE_PTR(R); REQUIRE_PTR(q_out); REQUIRE_PTR(scale_out);
  REQUIRE_ALIGNED(X); REQUIRE_ALIGNED(perm); REQUIRE_ALIGNED(R); REQUIRE_ALIGNED(q_out); REQUIRE_ALIGNED(scale_out);
  return vqlin::check_launch(vqlin::launch_act_composite_quant(X, M, K, bits, block, perm, R, q_out, scale_out,
                                                               static_cast<cudaStream_t>(stream)),
                             "act_composite_quant");
}

vqlin_status vqlin_debug_w4a16_withheld_loads(const uint16_t* X, const uint8_t* wq, const uint16_t* scales,
                                              const uint16_t* zeros, int group_size, uint16_t* Y, int M, int N,
                                              int K, uint64_t limit_ns, void* stream) {
  REQUIRE(M > vqlin::kW4a16GemvMaxM && N > 0 && K > 0, VQLIN_ERR_INVALID_ARG,
          "bad sizes M=%d N=%d K=%d (the tensor-core kernel takes M > %d)", M, N, K, vqlin::kW4a16GemvMaxM);
  REQUIRE(group_size == 64 || group_size == 128 || group_size == 256, VQLIN_ERR_INVALID_ARG,
          "group_size must be 64, 128 or 256 (got %d)", group_size);
  REQUIRE(K % 128 == 0 && K % group_size == 0, VQLIN_ERR_UNSUPPORTED_SHAPE,
          "K=%d must be a multiple of 128 and of the group %d", K, group_size);
  REQUIRE(limit_ns > 0 && limit_ns <= 2000000000ull, VQLIN_ERR_INVALID_ARG, "limit_ns must be in (0, 2e9]");
  REQUIRE_PTR(X); REQUIRE_PTR(wq); REQUIRE_PTR(scales); REQUIRE_PTR(zeros); REQUIRE_PTR(Y);
  REQUIRE_ALIGNED(X); REQUIRE_ALIGNED(wq); REQUIRE_ALIGNED(scales); REQUIRE_ALIGNED(zeros); REQUIRE_ALIGNED(Y);
  int* status = vqlin::device_status_word();
  REQUIRE(status != nullptr, VQLIN_ERR_CUDA, "no device status word");
  return vqlin::launch_w4a16_tc(X, wq, scales, zeros, group_size, nullptr, Y, M, N, K, status,
                                static_cast<cudaStream_t>(stream), 1, limit_ns);
}

vqlin_status vqlin_linear_w4a16(const uint16_t* X, const uint8_t* wq, const uint16_t* scales,
                                const uint16_t* zeros, int group_size, const uint16_t* bias, uint16_t* Y,
                                int M, int N, int K, void* stream) {
  REQUIRE(M >= 0 && N >= 0 && K > 0, VQLIN_ERR_INVALID_ARG, "bad sizes M=%d N=%d K=%d", M, N, K);
  REQUIRE(group_size == 64 || group_size == 128 || group_size == 256, VQLIN_ERR_INVALID_ARG,
          "group_size must be 64, 128 or 256 (got %d)", group_size);
  REQUIRE(K % 128 == 0 && K % group_size == 0, VQLIN_ERR_UNSUPPORTED_SHAPE,
          "K=%d must be a multiple of 128 and of the group %d", K, group_size);
  if (M == 0 || N == 0) return VQLIN_OK;
  REQUIRE_PTR(X); REQUIRE_PTR(wq); REQUIRE_PTR(scales); REQUIRE_PTR(zeros); REQUIRE_PTR(Y);
  REQUIRE_ALIGNED(X); REQUIRE_ALIGNED(wq); REQUIRE_ALIGNED(scales); REQUIRE_ALIGNED(zeros); REQUIRE_ALIGNED(Y);
  int* status = vqlin::device_status_word();
  REQUIRE(status != nullptr, VQLIN_ERR_CUDA, "no device status word");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (M <= vqlin::kW4a16GemvMaxM)
    return vqlin::check_launch(vqlin::launch_w4a16_gemv(X, wq, scales, zeros, group_size, bias, Y, M, N, K, status, st),
                               "linear_w4a16");
  return vqlin::launch_w4a16_tc(X, wq, scales, zeros, group_size, bias, Y, M, N, K, status, st);
}

vqlin_status vqlin_linear_bf16_ref(const uint16_t* X, const uint16_t* W, const uint16_t* bias, uint16_t* Y,
                                   int M, int N, int K, void* stream) {
  REQUIRE(M >= 0 && N >= 0 && K > 0, VQLIN_ERR_INVALID_ARG, "bad sizes M=%d N=%d K=%d", M, N, K);
  REQUIRE(K % 8 == 0 && N % 8 == 0, VQLIN_ERR_UNSUPPORTED_SHAPE, "K=%d and N=%d must be multiples of 8", K, N);
  if (M == 0 || N == 0) return VQLIN_OK;
  REQUIRE_PTR(X); REQUIRE_PTR(W); REQUIRE_PTR(Y);
  REQUIRE_ALIGNED(X); REQUIRE_ALIGNED(W); REQUIRE_ALIGNED(Y);
  vqlin::DeviceState* ds = nullptr;
  vqlin_status s = vqlin::device_state(&ds, true);
  if (s != VQLIN_OK) return s;

  // Column-major view: Y^T [N, M] = W^T^T [N, K] x X^T [K, M].
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
  vqlin_status out = VQLIN_OK;
  const cublasOperation_t ta = CUBLAS_OP_T, tb = CUBLAS_OP_N;
  const cublasLtEpilogue_t epi = bias ? CUBLASLT_EPILOGUE_BIAS : CUBLASLT_EPILOGUE_DEFAULT;
  const float alpha = 1.0f, beta = 0.0f;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  do {
    if (cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS ||
        cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof(ta)) != CUBLAS_STATUS_SUCCESS ||
        cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof(tb)) != CUBLAS_STATUS_SUCCESS ||
        cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_EPILOGUE, &epi, sizeof(epi)) != CUBLAS_STATUS_SUCCESS) {
      out = fail(VQLIN_ERR_CUDA, "cuBLASLt descriptor setup failed");
      break;
    }
    if (bias && cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_BIAS_POINTER, &bias, sizeof(bias)) !=
                    CUBLAS_STATUS_SUCCESS) {
      out = fail(VQLIN_ERR_CUDA, "cuBLASLt bias pointer setup failed");
      break;
    }
    if (cublasLtMatrixLayoutCreate(&la, CUDA_R_16BF, K, N, K) != CUBLAS_STATUS_SUCCESS ||
        cublasLtMatrixLayoutCreate(&lb, CUDA_R_16BF, K, M, K) != CUBLAS_STATUS_SUCCESS ||
        cublasLtMatrixLayoutCreate(&lc, CUDA_R_16BF, N, M, N) != CUBLAS_STATUS_SUCCESS) {
      out = fail(VQLIN_ERR_CUDA, "cuBLASLt layout setup failed");
      break;
    }
    cublasLtMatmulAlgo_t algo;
    const auto key = std::make_tuple(M, N, K, bias != nullptr);
    bool have = false;
    {
      std::lock_guard<std::mutex> lock(vqlin::g_mu);
      auto it = ds->algos.find(key);
      if (it != ds->algos.end()) {
        algo = it->second;
        have = true;
      }
    }
    if (!have) {
      cublasLtMatmulPreference_t pref = nullptr;
      cublasLtMatmulHeuristicResult_t res;
      int n = 0;
      cublasLtMatmulPreferenceCreate(&pref);
      cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ds->workspace_bytes,
                                           sizeof(ds->workspace_bytes));
      cublasStatus_t hs = cublasLtMatmulAlgoGetHeuristic(ds->lt, op, la, lb, lc, lc, pref, 1, &res, &n);
      cublasLtMatmulPreferenceDestroy(pref);
      if (hs != CUBLAS_STATUS_SUCCESS || n == 0) {
        out = fail(VQLIN_ERR_CUDA, "cuBLASLt found no algorithm for M=%d N=%d K=%d", M, N, K);
        break;
      }
      algo = res.algo;
      std::lock_guard<std::mutex> lock(vqlin::g_mu);
      ds->algos[key] = algo;
    }
    cublasStatus_t ms = cublasLtMatmul(ds->lt, op, &alpha, W, la, X, lb, &beta, Y, lc, Y, lc, &algo,
                                       ds->workspace, ds->workspace_bytes, st);
    if (ms != CUBLAS_STATUS_SUCCESS) out = fail(VQLIN_ERR_CUDA, "cublasLtMatmul failed (%d)", (int)ms);
  } while (0);
  if (la) cublasLtMatrixLayoutDestroy(la);
  if (lb) cublasLtMatrixLayoutDestroy(lb);
  if (lc) cublasLtMatrixLayoutDestroy(lc);
  if (op) cublasLtMatmulDescDestroy(op);
  return out;
}

}  // extern "C"
