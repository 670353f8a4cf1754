// Weight-only int4 projection (W4A16) on the tcgen05 tensor cores.
//
//   Y[m, n] = bf16( sum_g s[n,g] * sum_{k in g} X[m,k] * (q[n,k] - z[n,g]) + bias[n] )
//
// which is sum_k X[m,k] * Wdq[n,k] with Wdq = (q - z) * s regrouped: the
// integer (q - z) is an exact bf16 operand, each group's partial sum is kept
// apart in tensor memory, and its scale is applied in float32 when it is
// drained.  No weight is rounded to bf16, so the only rounding besides the
// final one is float32 accumulation.
//
// Method: "LoopQ" abstract (the action expert is memory-bound, 63% of GPU
// time; weight bytes dominate), with group-wise asymmetric RTN weights.
//
// Packed weights: per 8 channels one 32-bit word, channel 2i in bits
// [4i, 4i+4) and channel 2i+1 in bits [16+4i, 16+4i+4), so one shift and one
// mask give the codes of two consecutive channels in the two halves of a
// word; OR with 0x4300 makes each half the bf16 value 128 + q, and a bf16x2
// subtraction of 128 + z leaves q - z exactly.
//
// Work decomposition (weights on the MMA's M side):
//   * one CTA: 128 output channels x BT tokens (BT in {16, 32, 64}) over a
//     range of whole groups of K; the S CTAs that split K form a cluster;
//   * warp 0: TMA producer; a stage holds the activation tile (bf16, written
//     by TMA directly in the 128-byte-swizzled MMA layout) and the packed
//     weight tile (32 bytes of each row per 64-channel k-block), each with a
//     barrier of its own: the weights of the first stages (and the CTA's zero
//     points and scales) are read and expanded before the previous kernel is
//     waited for, so in a chain of launches that work overlaps it;
//   * warps 2..9: expand the packed weights into bf16 (q - z) directly in
//     tensor memory (thread = weight row, tcgen05.st), the MMA's A operand;
//   * MMAs (kind::f16, bf16 x bf16 -> f32, A from tensor memory) from up to
//     four issuing warps (1, 14, 15, 16), issuer i taking every NI-th
//     quantization group of the CTA into an accumulator of its own: one
//     thread issues at most one tcgen05.mma per ~120 SM clocks on B300
//     whatever N, and a bf16 MMA covers only 16 channels, so a single issuer
//     bounded the kernel at a few tokens; an issuer reuses its accumulator
//     once the previous group in it has been drained;
//   * warps 10..13 and 17..20: drain each group's accumulator (in group
//     order), y += s[n,g] * partial, in registers, two warps per lane quadrant
//     with 32 tokens each, so that one tensor-memory round trip (~300 SM
//     clocks) covers a group; then the bias epilogue, with split K summed
//     over the cluster's shared memory in a fixed order (deterministic).
// Every wait is bounded in time (VQLIN_ERR_TIMEOUT in the status word).
#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace {

using namespace vqlin_dev;

constexpr int kTileN = 128;
constexpr int kKB = 64;           // channels per k-block (one 128-byte bf16 row)
constexpr int kRawRow = 32;       // packed weight bytes of one row per k-block
constexpr int kBRow = 128;        // activation bytes of one row per k-block
constexpr int kACols = 32;        // tensor-memory columns of one A stage
constexpr int kThreads = 672;     // 21 warps
constexpr int kExpandWarps = 8;
constexpr int kDrainThreads = 256;  // 8 warps
constexpr int kMaxIssuers = 4;
constexpr int kMaxSplit = 16;
constexpr int kMaxGroupsCta = 128;  // quantization groups of one CTA (zero points and scales in shared memory)
constexpr uint64_t kWaitLimitNs = 1000000000ull;

struct W4a16Args {
  const uint16_t* scales;  // bf16 [N, G]
  const uint16_t* zeros;   // bf16 [N, G]
  const uint16_t* bias;    // bf16 [N] or null
  uint16_t* Y;
  int* status;
  int M, N, K, G;          // G = K / group
  int stages;
  uint32_t tmem_cols;
  uint32_t a_col;          // first tensor-memory column of the A stages
  uint32_t acc_step;       // tensor-memory columns between the issuers' accumulators
  int issuers;             // MMA-issuing warps (1..4), one accumulator each
  int rows_per;            // split K: output channels each cluster rank owns
  int ng_max;              // quantization groups of the CTA with the most (<= kMaxGroupsCta)
  int withhold_loads;      // test hook: the producer issues nothing (every wait runs out)
  uint64_t wait_limit_ns;
};

__device__ __forceinline__ void record_timeout(int* status, volatile int* abort) {
  *abort = 1;
  atomicCAS(status, 0, (int)VQLIN_ERR_TIMEOUT);
}

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// 8 packed codes (one word) -> 8 bf16 values q - z (4 words), channel order.
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t zz, uint32_t* o) {
  o[0] = bf16x2_sub((w & 0x000F000Fu) | 0x43004300u, zz);
  o[1] = bf16x2_sub(((w >> 4) & 0x000F000Fu) | 0x43004300u, zz);
  o[2] = bf16x2_sub(((w >> 8) & 0x000F000Fu) | 0x43004300u, zz);
  o[3] = bf16x2_sub(((w >> 12) & 0x000F000Fu) | 0x43004300u, zz);
}

template <int BT, int GROUP>
__global__ void __launch_bounds__(kThreads, 1)
w4a16_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                const W4a16Args a) {
  constexpr int KB_PER_G = GROUP / kKB;
  constexpr uint32_t kBBytes = BT * kBRow;                       // a multiple of 2048
  constexpr uint32_t kStageBytes = kBBytes + kTileN * kRawRow;   // [B operand | packed A]
  extern __shared__ uint8_t smem_dyn[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float s_bias[kTileN];  // split K: the tile's bias, read by the reducing threads

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  const int NS = a.stages;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + (size_t)NS * kStageBytes);
  uint64_t* full = bars;              // TMA -> expanders (packed weight tile)
  uint64_t* aready = bars + NS;       // expanders -> MMA
  uint64_t* empty = bars + 2 * NS;    // MMA -> TMA
  uint64_t* fullx = bars + 3 * NS;    // TMA -> MMA (activation tile)
  uint64_t* accf = bars + 4 * NS;     // [issuer] MMA -> drain (a group accumulated)
  uint64_t* acce = accf + kMaxIssuers;  // [issuer] drain -> MMA (accumulator free)
  uint64_t* done = acce + kMaxIssuers;  // every MMA issued has completed
  // the CTA's zero points z (uint8) and scales (bf16 bits), [local group][row]
  uint8_t* zsm = reinterpret_cast<uint8_t*>(done + 1);
  uint16_t* ssm = reinterpret_cast<uint16_t*>(zsm + (size_t)a.ng_max * kTileN);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = (int)gridDim.z;
  const uint32_t rank = cluster_ctarank();
  const int n0 = blockIdx.x * kTileN, m0 = blockIdx.y * BT;
  const int g0 = (int)(((long long)rank * a.G) / S);
  const int g1 = (int)(((long long)(rank + 1) * a.G) / S);
  const int ng = g1 - g0;
  const int cnt = ng * KB_PER_G;            // k-blocks of this CTA
  const int kb0 = g0 * KB_PER_G;
  volatile int* abort = &s_abort;

  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&fullx[i], 1);
      mbar_init(&aready[i], kExpandWarps / 2);  // one group of four warps per k-block
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < kMaxIssuers; ++i) {
      mbar_init(&accf[i], 1);
      mbar_init(&acce[i], kDrainThreads / 32);
    }
    mbar_init(done, a.issuers);
    mbar_init_fence();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) tmem_alloc(&s_tmem, a.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  // drain warps: 32 tokens [32 half, 32 half + 32) of their lane quadrant
  constexpr int kHalfCols = BT < 32 ? BT : 32;
  const bool drain = (warp >= 10 && warp < 14) || warp >= 17;
  const int half = warp >= 17 ? 1 : 0;
  const int ncol = BT - 32 * half < kHalfCols ? BT - 32 * half : kHalfCols;  // <= 0: no tokens
  float y[kHalfCols];
#pragma unroll
  for (int c = 0; c < kHalfCols; ++c) y[c] = 0.0f;

  // Zero points (expanders) and scales and bias (drains) of the CTA's rows
  // and groups, read once before the previous kernel is waited for (weights
  // do not depend on it): loaded one group at a time inside the loops, their
  // global-memory latency stood between consecutive k-blocks.
  float bias_r = 0.0f;
  if (warp >= 2 && warp < 10) {
    const int t = tid - 64, row = t & (kTileN - 1), n = n0 + row;
    for (int g = t >> 7; g < ng; g += 2)
      zsm[g * kTileN + row] =
          n < a.N ? (uint8_t)__uint_as_float((uint32_t)__ldg(a.zeros + (size_t)n * a.G + g0 + g) << 16) : 0;
    named_barrier(1, kExpandWarps * 32);
  } else if (drain) {
    const int row = (warp & 3) * 32 + lane, n = n0 + row;
    for (int g = half; g < ng; g += 2) ssm[g * kTileN + row] = n < a.N ? __ldg(a.scales + (size_t)n * a.G + g0 + g) : 0;
    if (S == 1 && a.bias != nullptr && n < a.N) bias_r = __uint_as_float((uint32_t)__ldg(a.bias + n) << 16);
    if (S > 1 && half == 0)
      s_bias[row] = (a.bias != nullptr && n < a.N) ? __uint_as_float((uint32_t)__ldg(a.bias + n) << 16) : 0.0f;
    named_barrier(2, kDrainThreads);
  }

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && !a.withhold_loads) {
      int issued = 0;
      // weight tiles of the first stages before waiting for the previous
      // kernel: they are expanded into tensor memory while it still runs
      const int pre = cnt < NS ? cnt : NS;
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], kTileN * kRawRow);
        tma_load_2d(base + (size_t)i * kStageBytes + kBBytes, &tmW, (kb0 + i) * kRawRow, n0, &full[i]);
      }
      pdl_wait();
      // the next kernel may prepare once this one works; an earlier trigger
      // lets a chain of launches prefetch weights all at once
      pdl_trigger();
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&fullx[i], kBBytes);
        tma_load_2d(base + (size_t)i * kStageBytes, &tmX, (kb0 + i) * kKB, m0, &fullx[i]);
        ++issued;
      }
      int s = 0;        // stage of k-block i
      uint32_t ph = 0;  // parity of the release of stage s that k-block i waits for
      for (int i = pre; i < cnt; ++i) {
        if (!mbar_wait_bounded(&empty[s], ph, a.wait_limit_ns, abort)) {
          if (!*abort) record_timeout(a.status, abort);
          break;
        }
        uint8_t* st = base + (size_t)s * kStageBytes;
        mbar_arrive_expect_tx(&full[s], kTileN * kRawRow);
        tma_load_2d(st + kBBytes, &tmW, (kb0 + i) * kRawRow, n0, &full[s]);
        mbar_arrive_expect_tx(&fullx[s], kBBytes);
        tma_load_2d(st, &tmX, (kb0 + i) * kKB, m0, &fullx[s]);
        ++issued;
        if (++s == NS) {
          s = 0;
          ph ^= 1u;
        }
      }
      // copies in flight complete before the CTA may exit: once every MMA
      // has completed, every copy has landed; only a CTA that gave up checks
      // the last ones one by one
      const bool all_done = mbar_wait_bounded(done, 0, a.wait_limit_ns, abort);
      if (!all_done || *abort) {
        for (int i = issued > NS ? issued - NS : 0; i < issued; ++i)
          if (!mbar_wait_bounded(&full[i % NS], (i / NS) & 1, a.wait_limit_ns, nullptr) ||
              !mbar_wait_bounded(&fullx[i % NS], (i / NS) & 1, a.wait_limit_ns, nullptr))
            record_timeout(a.status, abort);
      }
    }
  } else if (warp == 1 || (warp >= 14 && warp - 13 < a.issuers)) {
    // ------------------------------------------------------------ MMA issuers
    // issuer i: local groups i, i + NI, ...; the whole warp runs the loop
    // (every wait decided by a vote) and one elected lane issues each MMA and
    // commit; ring stage and phase advance incrementally (no divisions in the
    // issue loop)
    const int NI = a.issuers;
    const int iss = warp == 1 ? 0 : warp - 13;
    const uint32_t id = idesc_f32acc(1u, kTileN, BT);  // bf16 x bf16 -> f32
    const uint64_t db0 = sdesc_sw128(base);
    const uint32_t ta0 = tmem + a.a_col;
    const uint32_t acc = tmem + (uint32_t)iss * a.acc_step;
    int s = (iss * KB_PER_G) % NS;                     // ring stage of this issuer's first k-block
    uint32_t ph = (uint32_t)(((iss * KB_PER_G) / NS) & 1);
    const int skip = (NI - 1) * KB_PER_G;              // k-blocks of the other issuers between two groups
    bool ok = true;
    int round = 0;
    for (int jl = iss; jl < ng && ok; jl += NI, ++round) {
      if (round > 0) {
        // the previous group in this accumulator has been drained
        ok = mbar_wait_bounded(&acce[iss], (uint32_t)((round - 1) & 1), a.wait_limit_ns, abort);
        if (!__all_sync(0xffffffffu, ok)) {
          if (!ok && !*abort) record_timeout(a.status, abort);
          ok = false;
          break;
        }
      }
      for (int kin = 0; kin < KB_PER_G; ++kin) {
        ok = mbar_wait_bounded(&aready[s], ph, a.wait_limit_ns, abort) &&
             mbar_wait_bounded(&fullx[s], ph, a.wait_limit_ns, abort);
        if (!__all_sync(0xffffffffu, ok)) {
          if (!ok && !*abort) record_timeout(a.status, abort);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t db = db0 + (uint64_t)(s * (kStageBytes >> 4));
        const uint32_t ta = ta0 + (uint32_t)(s * kACols);
        mma_f16_ta_warp(acc, ta, db, id, kin != 0 ? 1u : 0u);
        mma_f16_ta_warp(acc, ta + 8, db + 2, id, 1u);
        mma_f16_ta_warp(acc, ta + 16, db + 4, id, 1u);
        mma_f16_ta_warp(acc, ta + 24, db + 6, id, 1u);
        tc_commit_warp(&empty[s]);
        if (++s == NS) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      tc_commit_warp(&accf[iss]);
      s += skip;
      while (s >= NS) {
        s -= NS;
        ph ^= 1u;
      }
    }
    tc_commit_warp(done);  // tensor memory is freed only after every issuer's MMAs completed
  } else if (warp < 10) {
    // ------------------------------------------------- weight expanders (2..9)
    // thread = weight row; the two groups of four warps (one warp per lane
    // quadrant each) take alternate k-blocks and expand the whole row (32
    // packed bytes, 64 channels), so one group's tensor-memory stores are in
    // flight while the other expands
    const int q = warp & 3, gr = (warp - 2) >> 2;
    const int row = q * 32 + lane;
    const int sw = (row >> 2) & 1;  // 32-byte swizzle of the packed tile
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16) + a.a_col;
    // quantization group of this group's k-blocks: the next one differs by
    // jstep (one group per k-block: 2, else 1)
    constexpr int jstep = KB_PER_G == 1 ? 2 : 1;
    int jl = gr / KB_PER_G, kin = gr % KB_PER_G;
    int s = gr;        // stage of k-block i (NS >= 2)
    uint32_t ph = 0;   // phase parity of stage s
    for (int i = gr; i < cnt; i += 2) {
      const bool ok = mbar_wait_bounded(&full[s], ph, a.wait_limit_ns, abort);
      if (!__all_sync(0xffffffffu, ok)) {
        if (!ok && !*abort) record_timeout(a.status, abort);
        break;
      }
      const uint32_t zh = 0x4300u + zsm[jl * kTileN + row];  // bf16 128 + z
      const uint32_t zz = zh | (zh << 16);
      const uint8_t* rawrow = base + (size_t)s * kStageBytes + kBBytes + row * kRawRow;
      const uint4 c0 = *reinterpret_cast<const uint4*>(rawrow + (sw << 4));
      const uint4 c1 = *reinterpret_cast<const uint4*>(rawrow + ((1 ^ sw) << 4));
      uint32_t v[2][16];
      dequant_word(c0.x, zz, v[0]);
      dequant_word(c0.y, zz, v[0] + 4);
      dequant_word(c0.z, zz, v[0] + 8);
      dequant_word(c0.w, zz, v[0] + 12);
      dequant_word(c1.x, zz, v[1]);
      dequant_word(c1.y, zz, v[1] + 4);
      dequant_word(c1.z, zz, v[1] + 8);
      dequant_word(c1.w, zz, v[1] + 12);
      const uint32_t ta = trow + (uint32_t)(s * kACols);
      tmem_st_x16(ta, v[0]);
      tmem_st_x16(ta + 16, v[1]);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&aready[s]);
      s += 2;
      if (s >= NS) {
        s -= NS;
        ph ^= 1u;
      }
      kin += 2;
      if (kin >= KB_PER_G) {  // this group's next k-block is in another quantization group
        kin -= KB_PER_G * (kin / KB_PER_G);
        jl += jstep;
      }
    }
  } else if (drain) {
    // --------------------------------------- group drains (10..13, 17..20)
    const int q = warp & 3, row = q * 32 + lane;
    int iss = 0, round = 0;  // issuer of group jl and its round (no divisions)
    for (int jl = 0; jl < ng; ++jl) {
      const float sg = __uint_as_float((uint32_t)ssm[jl * kTileN + row] << 16);
      const bool ok = mbar_wait_bounded(&accf[iss], (uint32_t)(round & 1), a.wait_limit_ns, abort);
      if (!__all_sync(0xffffffffu, ok)) {
        if (!ok && !*abort) record_timeout(a.status, abort);
        break;
      }
      tc_fence_after();
      if (ncol > 0) {
        // every load of the group first, then one wait
        uint32_t v[2][16];
        const uint32_t src = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)iss * a.acc_step + (uint32_t)(32 * half);
        tmem_ld_x16(src, v[0]);
        if (kHalfCols > 16) tmem_ld_x16(src + 16, v[1]);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < kHalfCols; ++j) y[j] = fmaf(sg, __uint_as_float(v[j >> 4][j & 15]), y[j]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[iss]);
      if (++iss == a.issuers) {
        iss = 0;
        ++round;
      }
    }
  }

  // ---------------------------------------------------------------- epilogue
  __syncwarp();
  pdl_wait();  // global writes only once the previous kernel has finished
  if (S == 1) {
    if (drain && !*abort && ncol > 0) {
      const int row = (warp & 3) * 32 + lane, n = n0 + row;
      if (n < a.N) {
#pragma unroll
        for (int c = 0; c < kHalfCols; ++c) {
          const int m = m0 + 32 * half + c;
          if (c < ncol && m < a.M) a.Y[(size_t)m * a.N + n] = f32_to_bf16_rn(__fadd_rn(y[c], bias_r));
        }
      }
    }
    tc_fence_before();
    __syncthreads();
  } else {
    // Split K: each drain thread stores its partial row straight into the
    // shared memory of the cluster rank that owns the row (posted stores, no
    // round trip), as part[src][token][local row] over the owner's idle
    // stages; after the second cluster barrier every rank sums its rows'
    // slices from its own shared memory in source order (deterministic).
    float* part = reinterpret_cast<float*>(base);
    const int rows_per = a.rows_per;
    tc_fence_before();
    cluster_sync_all();  // every CTA of the cluster is past its stages before they are overwritten
    if (drain && !*abort && ncol > 0) {
      const int row = (warp & 3) * 32 + lane;
      const int owner = row / rows_per, lrow = row - owner * rows_per;
      const uint32_t dst = mapa_shared(smem_addr(part + ((size_t)rank * BT + 32 * half) * rows_per + lrow),
                                       (uint32_t)owner);
#pragma unroll
      for (int c = 0; c < kHalfCols; ++c)
        if (c < ncol) st_shared_cluster_f32(dst + (uint32_t)(c * rows_per * 4), y[c]);
    }
    cluster_sync_all();
    if (!*abort) {
      const int r0 = (int)rank * rows_per;
      const int nq = (min(kTileN, r0 + rows_per) - r0) / 4;
      const bool vec = (a.N & 3) == 0;
      for (int idx = tid; idx < nq * BT; idx += kThreads) {
        const int lr = 4 * (idx % nq), col = idx / nq;
        const int m = m0 + col, n = n0 + r0 + lr;
        if (m >= a.M || n >= a.N) continue;
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int cc = 0; cc < S; ++cc) {
          const float4 pv = *reinterpret_cast<const float4*>(part + ((size_t)cc * BT + col) * rows_per + lr);
          acc[0] += pv.x; acc[1] += pv.y; acc[2] += pv.z; acc[3] += pv.w;
        }
        uint16_t yo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) yo[e] = f32_to_bf16_rn(__fadd_rn(acc[e], s_bias[r0 + lr + e]));
        uint16_t* dst = a.Y + (size_t)m * a.N + n;
        if (vec) {
          *reinterpret_cast<uint2*>(dst) =
              make_uint2((uint32_t)yo[0] | ((uint32_t)yo[1] << 16), (uint32_t)yo[2] | ((uint32_t)yo[3] << 16));
        } else {
          for (int e = 0; e < 4 && n + e < a.N; ++e) dst[e] = yo[e];
        }
      }
    }
  }
  if (warp == 1) {
    if (!mbar_wait_bounded(done, 0, a.wait_limit_ns, nullptr)) record_timeout(a.status, abort);
    __syncwarp();
    tmem_dealloc(tmem, a.tmem_cols);
  }
}

// ------------------------------------------------------------------ host side

constexpr int kMaxSmem = 232448 - 4096;
constexpr size_t kSmemPerSm = 233472;

template <int BT>
constexpr size_t stage_bytes() {
  return (size_t)BT * kBRow + (size_t)kTileN * kRawRow;
}

template <int BT>
size_t smem_bytes(int stages, int ng_max) {
  return 1024 + stages * stage_bytes<BT>() + (4 * stages + 2 * kMaxIssuers + 1) * 8 + (size_t)ng_max * kTileN * 3;
}

template <int BT, int GROUP>
vqlin_status launch_t(const uint16_t* X, const uint8_t* wq, const uint16_t* s, const uint16_t* z,
                      const uint16_t* bias, uint16_t* Y, int M, int N, int K, int* status, cudaStream_t st,
                      int withhold, uint64_t limit_ns) {
  // function attributes are per device: set them once for every device used
  static std::mutex mu;
  static bool set[64] = {};
  static cudaError_t res[64] = {};
  cudaError_t attr_err = cudaSuccess;
  {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return vqlin::fail(VQLIN_ERR_CUDA, "w4a16: no device");
    std::lock_guard<std::mutex> lock(mu);
    if (!set[dev]) {
      res[dev] = cudaFuncSetAttribute(w4a16_tc_kernel<BT, GROUP>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
      if (res[dev] == cudaSuccess)
        res[dev] = cudaFuncSetAttribute(w4a16_tc_kernel<BT, GROUP>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      set[dev] = true;
    }
    attr_err = res[dev];
  }
  if (attr_err != cudaSuccess)
    return vqlin::fail(VQLIN_ERR_CUDA, "w4a16: cudaFuncSetAttribute: %s", cudaGetErrorString(attr_err));
  const int tiles_n = (N + kTileN - 1) / kTileN, tiles_m = (M + BT - 1) / BT;
  const int G = K / GROUP;
  int s_want = (148 + tiles_n * tiles_m - 1) / (tiles_n * tiles_m);
  s_want = s_want > 8 ? 8 : s_want;  // beyond 8 the reduction over the cluster costs more than it saves
  s_want = s_want > G ? G : s_want;
  // a CTA holds the zero points and scales of at most kMaxGroupsCta groups
  const int s_min = (G + kMaxGroupsCta - 1) / kMaxGroupsCta;
  if (s_min > kMaxSplit) return vqlin::fail(VQLIN_ERR_UNSUPPORTED_SHAPE, "w4a16: K=%d has too many groups", K);
  if (s_want < s_min) s_want = s_min;
  // Among the splits whose clusters are all resident at once (one wave), the
  // one of least estimated time, a fit to launches timed on B300 at 8 to 64
  // tokens: ~1.7 us fixed, ~0.27 us per k-block of a CTA (its pipeline ring
  // paces it), ~1 us for the cluster reduction when K is split, and ~0.035 us
  // per CTA (at 50 x 3072 x 1024 a split of 2 measured 5.03 us, of 4 5.44 us).  Splits other than powers of two (clusters of 3 or 6 CTAs timed
  // twice as slow) are left out unless the groups force one.  Without a
  // one-wave split, the smallest split.
  int S = 0, NS = 0, rows_per = 0, NI = 0;
  bool have_wave = false;
  double best = 0.0;
  uint32_t a_col = 0, cols = 0;
  const uint32_t acc_step = (uint32_t)((BT + 31) / 32 * 32);
  size_t dyn = 0;
  int ng_max = 0;
  for (int s_try = s_want; s_try >= s_min; --s_try) {
    if ((s_try & (s_try - 1)) != 0 && s_try != s_min) continue;
    const int groups = (G + s_try - 1) / s_try;  // of the CTA with the most
    const int per_cta = groups * (GROUP / kKB);
    // stages: up to 8, no more than the k-blocks a CTA runs, and enough that
    // the float partial tile of the split-K epilogue ([BT][128]) fits over them
    // (split K: s_try slices of [BT][rows_per] floats, rows_per rounded up to 4)
    const int rp_try = s_try > 1 ? ((kTileN + s_try - 1) / s_try + 3) & ~3 : kTileN;
    const size_t part_bytes = (size_t)(s_try > 1 ? s_try * rp_try : kTileN) * BT * 4;
    const int ns_min = (int)((part_bytes + stage_bytes<BT>() - 1) / stage_bytes<BT>());
    int ns = per_cta > 8 ? 8 : per_cta;
    if (ns < ns_min) ns = ns_min;
    if (ns < 2) ns = 2;
    // issuers: up to four, no more than the groups a CTA sums
    int ni = groups < kMaxIssuers ? groups : kMaxIssuers;
    if (ni < 1) ni = 1;
    // tensor memory: one accumulator per issuer, then one A slot per stage
    while (ni > 1 && (uint32_t)ni * acc_step + (uint32_t)(ns * kACols) > 512) --ni;
    while (ns > ns_min && ns > 2 && (uint32_t)ni * acc_step + (uint32_t)(ns * kACols) > 512) --ns;
    // A ring stage is reused by the k-block NS later.  mbarrier parity waits
    // tell only adjacent phases apart, so the role that waits for a stage's
    // next use must be the one that consumed its last use: the two expander
    // groups take alternate k-blocks (NS even), and issuer i takes whole
    // groups every NI groups (NS a multiple of NI x k-blocks per group; with
    // issuer 2 of 3 starting in a stage's second phase while its first was
    // still pending, a parity wait would pass at once).
    if (per_cta > ns) {
      if (ns & 1) ns += ns - 1 >= ns_min ? -1 : 1;  // the partial tile still fits
      while (ni > 1 && ns % (ni * (GROUP / kKB)) != 0) --ni;
    }
    const uint32_t ac = (uint32_t)ni * acc_step;
    uint32_t c = 32;
    while (c < ac + (uint32_t)(ns * kACols)) c <<= 1;
    if (c > 512 || smem_bytes<BT>(ns, groups) > (size_t)kMaxSmem) continue;
    // never more CTAs on an SM than its tensor memory holds (see the integer GEMM)
    size_t d = smem_bytes<BT>(ns, groups);
    const size_t dyn_floor = kSmemPerSm / (512 / c + 1) + 1;
    if (d < dyn_floor) d = dyn_floor;
    const int active = vqlin::max_active_clusters((const void*)w4a16_tc_kernel<BT, GROUP>, kThreads, d, s_try);
    const bool wave = tiles_n * tiles_m <= active;
    const int ctas = tiles_n * tiles_m * s_try;
    const double est = 1.7 + 0.27 * per_cta + (s_try > 1 ? 1.0 : 0.0) + 0.035 * ctas;
    const bool take = S == 0 || (wave && (!have_wave || est < best)) || (!wave && !have_wave && s_try < S);
    if (take) {
      S = s_try; NS = ns; a_col = ac; cols = c; dyn = d; NI = ni; ng_max = groups;
      rows_per = s_try > 1 ? ((kTileN + s_try - 1) / s_try + 3) & ~3 : kTileN;
      if (wave) {
        have_wave = true;
        best = est;
      }
    }
  }
  if (S == 0) return vqlin::fail(VQLIN_ERR_UNSUPPORTED_SHAPE, "w4a16: no tile plan for M=%d N=%d K=%d", M, N, K);

  CUtensorMap tmW, tmX;
  if (!vqlin::tmap_encoder_available())
    return vqlin::fail(VQLIN_ERR_CUDA, "w4a16: cuTensorMapEncodeTiled is unavailable");
  if (!vqlin::encode_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, (uint64_t)K / 2, (uint64_t)N, (uint64_t)K / 2,
                             kRawRow, kTileN, CU_TENSOR_MAP_SWIZZLE_32B) ||
      !vqlin::encode_tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2,
                             kKB, BT, CU_TENSOR_MAP_SWIZZLE_128B))
    return vqlin::fail(VQLIN_ERR_CUDA, "w4a16: tensor map encoding failed (M=%d N=%d K=%d)", M, N, K);

  W4a16Args a;
  a.scales = s; a.zeros = z; a.bias = bias; a.Y = Y; a.status = status;
  a.M = M; a.N = N; a.K = K; a.G = G; a.stages = NS; a.tmem_cols = cols; a.a_col = a_col;
  a.acc_step = acc_step; a.issuers = NI;
  a.rows_per = rows_per; a.ng_max = ng_max; a.wait_limit_ns = limit_ns; a.withhold_loads = withhold;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles_n, tiles_m, S);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = S;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = vqlin::pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = vqlin::launched(cudaLaunchKernelEx(&cfg, w4a16_tc_kernel<BT, GROUP>, tmW, tmX, a));
  if (e != cudaSuccess)
    return vqlin::fail(VQLIN_ERR_CUDA, "w4a16 launch (grid %d x %d x %d, %zu B smem): %s", tiles_n, tiles_m, S,
                       cfg.dynamicSmemBytes, cudaGetErrorString(e));
  return VQLIN_OK;
}

template <int BT>
vqlin_status launch_bt(const uint16_t* X, const uint8_t* wq, const uint16_t* s, const uint16_t* z, int group,
                       const uint16_t* bias, uint16_t* Y, int M, int N, int K, int* status, cudaStream_t st,
                       int withhold, uint64_t limit_ns) {
  switch (group) {
    case 64: return launch_t<BT, 64>(X, wq, s, z, bias, Y, M, N, K, status, st, withhold, limit_ns);
    case 128: return launch_t<BT, 128>(X, wq, s, z, bias, Y, M, N, K, status, st, withhold, limit_ns);
    default: return launch_t<BT, 256>(X, wq, s, z, bias, Y, M, N, K, status, st, withhold, limit_ns);
  }
}

}  // namespace

namespace vqlin {

vqlin_status launch_w4a16_tc(const uint16_t* X, const uint8_t* wq, const uint16_t* s, const uint16_t* z, int group,
                             const uint16_t* bias, uint16_t* Y, int M, int N, int K, int* status, cudaStream_t st,
                             int withhold, uint64_t limit_ns) {
  if (M == 0 || N == 0) return VQLIN_OK;
  if (limit_ns == 0) limit_ns = kWaitLimitNs;
  // token tile: the smallest of 16, 32, 64 that covers M in as few tiles as
  // possible (the drain warps keep BT float sums per thread in registers)
  const int tiles = (M + 63) / 64;
  const int per = (M + tiles - 1) / tiles;
  if (per <= 16) return launch_bt<16>(X, wq, s, z, group, bias, Y, M, N, K, status, st, withhold, limit_ns);
  if (per <= 32) return launch_bt<32>(X, wq, s, z, group, bias, Y, M, N, K, status, st, withhold, limit_ns);
  return launch_bt<64>(X, wq, s, z, group, bias, Y, M, N, K, status, st, withhold, limit_ns);
}

}  // namespace vqlin
