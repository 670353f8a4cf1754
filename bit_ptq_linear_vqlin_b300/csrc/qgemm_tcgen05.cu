// Integer GEMM of the W4A4 / W8A8 projections on the tcgen05 tensor cores.
//
//   acc[m, n] = sum_k xq[m, k] * wq[n, k]        (exact int32)
//   Y[m, n]   = bf16(((float)acc * sx[m]) * sw[n] + bias[n])
//
// Method: "FoldQuantVLA" abstract (W4A4 projections executed natively in
// integers after per-token activation and per-channel weight quantization;
// attention-output and FFN-down projections kept at W8A8).
//
// sm_103a has no integer tcgen05 MMA, so the integer codes ride in floating
// point operands whose products and sums are exact:
//   * int4 code c (sign-magnitude nibble s|mmm, |c| <= 7) is the e4m3 subnormal
//     byte s<<7 | mmm, value c * 2^-9; the MMA is kind::f8f6f4 and the float32
//     accumulator holds acc * 2^-18 exactly (|acc| <= 49 K < 2^24 for K < 342k);
//   * int8 code c (sign-magnitude byte, |c| <= 127) is the f16 subnormal
//     s<<15 | |c|, value c * 2^-24; the MMA is kind::f16 and the accumulator
//     holds acc * 2^-48 exactly while |acc| <= 127^2 * 1024 < 2^24, so every CTA
//     sums at most 1024 channels and longer K is split across the cluster.
// Conversions are a few bit operations per 32-bit word (no lookup table).
//
// Work decomposition (swap-AB: weights are the MMA's M side):
//   * one CTA computes 128 output channels x BT tokens (BT <= 256, a multiple
//     of 16) over a range of K; grid = (N/128, M/BT, S) with the S CTAs that
//     share an output tile forming one thread-block cluster (split K);
//   * warp 0: TMA producer of the packed code tiles (weights and activations,
//     64 bytes of each row per k-block) into a ring of raw stages;
//   * warps 2..5: unpack each raw stage into the MMA operand layout (128-byte
//     swizzled K-major rows) in a ring of operand stages;
//   * warp 1: allocates tensor memory and issues the MMAs (one thread), 4 per
//     k-block, accumulating 128 x BT float32 in tensor memory;
//   * epilogue: warps 2..5 convert the accumulator to int32 in shared memory;
//     after a cluster barrier each CTA of the cluster sums its slice of the
//     output channels over the cluster's shared memory (DSMEM) and applies the
//     scale epilogue, so split K needs no global scratch memory and the sum
//     is deterministic.
// Every wait is bounded in time; a wait that runs out records
// VQLIN_ERR_TIMEOUT in the device status word and the CTA winds down.
#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace {

using namespace vqlin_dev;

constexpr int kTileN = 128;       // output channels per CTA (MMA M)
constexpr int kRawRow = 64;       // packed bytes of one row per k-block
constexpr int kOpRow = 128;       // operand bytes of one row per k-block
constexpr int kThreads = 320;     // 10 warps
constexpr int kUnpackThreads = 256;
constexpr int kMaxSplit = 16;
constexpr int kOpStages = 2;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

struct QgemmArgs {
  const float* sx;
  const float* sw;
  const uint16_t* bias;
  uint16_t* Y;
  int32_t* acc;          // non-null: store raw int32 accumulators instead of Y
  int* status;
  int M, N, K;           // K in codes
  int bt;                // token tile
  int nkb;               // k-blocks over K
  int raw_stages;
  uint32_t tmem_cols;
  uint64_t wait_limit_ns;
  int withhold_loads;    // test hook: the producer issues nothing (waits run out)
  int tma_store;         // unsplit K: stage the bf16 tile and store it with TMA
  int push;              // split K: peers push int32 slices to the owning CTA
  int rows_per;          // split K: output channels each cluster rank owns
};

// Unpacks 8 packed bytes into 16 operand bytes.
//   int4: word w holds channels 0..7 (nibble s|mmm, even channel low).  The
//   e4m3 bytes of the even channels are (w & 0x07070707) | ((w << 4) &
//   0x80808080) and of the odd channels ((w >> 4) & 0x07070707) |
//   (w & 0x80808080); the chunk's channel order becomes 0,2,4,6,1,3,5,7, the
//   same permutation on both operands, which leaves every dot product
//   unchanged.
//   int8: byte s|mmmmmmm -> f16 s<<15 | mmmmmmm: prmt copies the byte and
//   replicates its sign bit into the high byte, a mask keeps bit 15 and 0..6.
template <int BITS>
__device__ __forceinline__ uint4 unpack8(uint2 in) {
  uint4 o;
  if (BITS == 4) {
    o.x = (in.x & 0x07070707u) | ((in.x << 4) & 0x80808080u);
    o.y = ((in.x >> 4) & 0x07070707u) | (in.x & 0x80808080u);
    o.z = (in.y & 0x07070707u) | ((in.y << 4) & 0x80808080u);
    o.w = ((in.y >> 4) & 0x07070707u) | (in.y & 0x80808080u);
  } else {
    o.x = __byte_perm(in.x, 0u, 0x9180) & 0x807F807Fu;
    o.y = __byte_perm(in.x, 0u, 0xB3A2) & 0x807F807Fu;
    o.z = __byte_perm(in.y, 0u, 0x9180) & 0x807F807Fu;
    o.w = __byte_perm(in.y, 0u, 0xB3A2) & 0x807F807Fu;
  }
  return o;
}

__device__ __forceinline__ void record_timeout(int* status, volatile int* abort) {
  *abort = 1;
  atomicCAS(status, 0, (int)VQLIN_ERR_TIMEOUT);
}

template <int BITS>
__global__ void __launch_bounds__(kThreads, 1)
qgemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
             const __grid_constant__ CUtensorMap tmY, const QgemmArgs a) {
  extern __shared__ uint8_t smem_dyn[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float s_sx[256], s_sw[kTileN], s_bias[kTileN];

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  const int bt = a.bt;
  const int rows = kTileN + bt;
  const uint32_t op_bytes = (uint32_t)rows * kOpRow;
  const uint32_t raw_bytes = (uint32_t)rows * kRawRow;
  const int R = a.raw_stages;
  uint8_t* op = base;
  uint8_t* raw = base + kOpStages * op_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(raw + (size_t)R * raw_bytes);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = bars + R;
  uint64_t* op_full = bars + 2 * R;
  uint64_t* op_empty = bars + 2 * R + kOpStages;
  uint64_t* acc_full = bars + 2 * R + 2 * kOpStages;
  uint64_t* scl_ready = acc_full + 1;
  uint64_t* red_full = acc_full + 2;  // push reduction: slices received
  // push reduction: recv[source rank][channel in the owned slice][token],
  // row stride bt + 4 words, after the barriers (not overlaying the rings,
  // which peers may still be using when slices arrive)
  const int ldr = bt + 4;
  int32_t* recv = reinterpret_cast<int32_t*>(bars + 2 * R + 2 * kOpStages + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = (int)gridDim.z;
  const uint32_t rank = cluster_ctarank();
  const int n0 = blockIdx.x * kTileN, m0 = blockIdx.y * bt;
  const int kb0 = (int)(((long long)rank * a.nkb) / S);
  const int kb1 = (int)(((long long)(rank + 1) * a.nkb) / S);
  const int cnt = kb1 - kb0;
  volatile int* abort = &s_abort;

  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < R; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], kUnpackThreads / 32);
    }
    for (int i = 0; i < kOpStages; ++i) {
      mbar_init(&op_full[i], kUnpackThreads / 32);
      mbar_init(&op_empty[i], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(scl_ready, 31);
    mbar_init(red_full, 1);
    mbar_init_fence();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) tmem_alloc(&s_tmem, a.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  if (tid == 0) pdl_trigger();
  const int r0_own = (int)rank * a.rows_per;
  const int nr_own = S > 1 ? max(0, min(kTileN, r0_own + a.rows_per) - r0_own) : 0;
  if (a.push) {
    // expect every peer's slice of the owned channels, then let peers know the
    // barrier exists (the matching cluster_wait is right before the pushes)
    if (tid == 0) mbar_arrive_expect_tx(red_full, (uint32_t)((S - 1) * nr_own * bt * 4));
    cluster_arrive();
  }

  if (warp == 0) {
    // lanes 1..31 stage the epilogue's per-token and per-channel scales and the
    // bias (float) while lane 0 produces; the epilogue reads them after a
    // CTA-wide or cluster-wide barrier
    if (lane > 0) {
      if (a.acc == nullptr) {
        for (int i = lane - 1; i < kTileN; i += 31) {
          const bool in = n0 + i < a.N;
          s_sw[i] = in ? __ldg(a.sw + n0 + i) : 0.0f;
          s_bias[i] = in && a.bias != nullptr ? __uint_as_float((uint32_t)__ldg(a.bias + n0 + i) << 16) : 0.0f;
        }
        pdl_wait();  // the per-token scales come from the previous kernel
        for (int i = lane - 1; i < bt; i += 31) s_sx[i] = m0 + i < a.M ? __ldg(a.sx + m0 + i) : 0.0f;
      }
      mbar_arrive(scl_ready);
    }
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued = 0;
      if (!a.withhold_loads) {
        // the weight tiles of the first stages do not depend on the previous
        // kernel: load them before waiting for it
        const int pre = cnt < R ? cnt : R;
        for (int i = 0; i < pre; ++i) {
          mbar_arrive_expect_tx(&raw_full[i], raw_bytes);
          tma_load_2d(raw + (size_t)i * raw_bytes, &tmW, (kb0 + i) * kRawRow, n0, &raw_full[i]);
        }
        pdl_wait();
        for (int i = 0; i < pre; ++i) {
          tma_load_2d(raw + (size_t)i * raw_bytes + kTileN * kRawRow, &tmX, (kb0 + i) * kRawRow, m0, &raw_full[i]);
          ++issued;
        }
        for (int i = pre; i < cnt; ++i) {
          const int s = i % R;
          if (!mbar_wait_bounded(&raw_empty[s], ((i / R) - 1) & 1, a.wait_limit_ns, abort)) {
            if (!*abort) record_timeout(a.status, abort);
            break;
          }
          mbar_arrive_expect_tx(&raw_full[s], raw_bytes);
          uint8_t* dst = raw + (size_t)s * raw_bytes;
          tma_load_2d(dst, &tmW, (kb0 + i) * kRawRow, n0, &raw_full[s]);
          tma_load_2d(dst + kTileN * kRawRow, &tmX, (kb0 + i) * kRawRow, m0, &raw_full[s]);
          ++issued;
        }
      } else {
        pdl_wait();
      }
      // copies still in flight complete before the CTA may exit
      for (int i = issued > R ? issued - R : 0; i < issued; ++i)
        if (!mbar_wait_bounded(&raw_full[i % R], (i / R) & 1, a.wait_limit_ns, nullptr))
          record_timeout(a.status, abort);
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f32acc(0u, kTileN, 0) ;
      const uint32_t id = idesc | ((uint32_t)(bt >> 3) << 17);
      for (int i = 0; i < cnt; ++i) {
        const int ps = i % kOpStages;
        if (!mbar_wait_bounded(&op_full[ps], (i / kOpStages) & 1, a.wait_limit_ns, abort)) {
          if (!*abort) record_timeout(a.status, abort);
          break;
        }
        tc_fence_after();
        const uint8_t* st = op + (size_t)ps * op_bytes;
        const uint64_t da = sdesc_sw128(st), db = sdesc_sw128(st + kTileN * kOpRow);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // +32 bytes along K inside the 128-byte swizzled row per MMA
          if (BITS == 4) mma_f8f6f4(tmem, da + 2 * j, db + 2 * j, id, (i | j) != 0);
          else mma_f16(tmem, da + 2 * j, db + 2 * j, id, (i | j) != 0);
        }
        tc_commit(&op_empty[ps]);
      }
      tc_commit(acc_full);
    }
  } else {
    // ------------------------------------------------------------ unpackers
    const int t = tid - 64;
    for (int i = 0; i < cnt; ++i) {
      const int s = i % R, ps = i % kOpStages;
      // warp-uniform exits: the per-warp arrival below needs every lane
      bool ok = mbar_wait_bounded(&raw_full[s], (i / R) & 1, a.wait_limit_ns, abort);
      if (ok && i >= kOpStages)
        ok = mbar_wait_bounded(&op_empty[ps], ((i / kOpStages) - 1) & 1, a.wait_limit_ns, abort);
      if (!__all_sync(0xffffffffu, ok)) {
        if (!ok && !*abort) record_timeout(a.status, abort);
        break;
      }
      const uint8_t* rs = raw + (size_t)s * raw_bytes;
      uint8_t* os = op + (size_t)ps * op_bytes;
      // thread t: chunk c = t % 8 of rows t/8 + 32 u; the swizzle term is the
      // same for all its rows (32 is a multiple of 8)
      {
        const int c = t & 7, r0 = t >> 3;
        const uint8_t* src = rs + r0 * kRawRow + c * 8;
        uint8_t* dst = os + r0 * kOpRow + ((c ^ (r0 & 7)) << 4);
#pragma unroll 4
        for (int r = r0; r < rows; r += 32) {
          const uint2 w = *reinterpret_cast<const uint2*>(src);
          *reinterpret_cast<uint4*>(dst) = unpack8<BITS>(w);
          src += 32 * kRawRow;
          dst += 32 * kOpRow;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();  // one arrival per warp, after every lane's writes and fence
      if (lane == 0) {
        mbar_arrive(&raw_empty[s]);
        mbar_arrive(&op_full[ps]);
      }
    }
  }

  // ---------------------------------------------------------------- epilogue
  __syncwarp();  // the single-thread roles rejoin their warps
  const float unit = BITS == 4 ? 262144.0f : 281474976710656.0f;  // 2^18, 2^48: accumulator -> integer
  const bool raw_out = a.acc != nullptr;
  bool go = false;
  if (warp >= 2) {
    const bool ok = mbar_wait_bounded(acc_full, 0, a.wait_limit_ns, nullptr) &&
                    mbar_wait_bounded(scl_ready, 0, a.wait_limit_ns, nullptr);
    if (!ok) record_timeout(a.status, abort);
    tc_fence_after();
    // warp-uniform decision: the tensor-memory loads below are warp-collective
    go = __all_sync(0xffffffffu, ok && !*abort);
  }
  pdl_wait();  // global writes only once the previous kernel has finished
  // warps 2..9: lane quadrant q of tensor memory, 16-column chunks h, h+2, ...
  const int q = warp & 3;
  const int h = (warp - 2) >> 2;
  const int row = q * 32 + lane;   // output channel inside the tile

  if (S == 1 && a.tma_store) {
    // bf16 tile [bt tokens][128 channels] staged over the idle rings, then one
    // TMA store (the tensor map clips the M and N tails)
    uint16_t* ystage = reinterpret_cast<uint16_t*>(base);
    if (warp >= 2) {
      if (go) {
        const float sw_n = s_sw[row], b_n = s_bias[row];
        for (int c0 = 16 * h; c0 < bt; c0 += 32) {
          uint32_t v[16];
          tmem_ld_x16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float acc = (float)__float2int_rn(__uint_as_float(v[j]) * unit);
            ystage[(c0 + j) * kTileN + row] = f32_to_bf16_rn(__fadd_rn(__fmul_rn(__fmul_rn(acc, s_sx[c0 + j]), sw_n), b_n));
          }
        }
        fence_proxy_async_smem();
      }
      named_barrier(1, kThreads - 64);
      if (tid == 64 && go) {
        tma_store_2d(&tmY, n0, m0, ystage);
        bulk_commit();
        bulk_wait_read();
      }
    }
    tc_fence_before();
    __syncthreads();
  } else if (S == 1) {
    // straight from tensor memory to global memory: thread = channel, 16
    // tokens per load; for each token the warp writes 32 consecutive channels
    if (warp >= 2 && go) {
      const int n = n0 + row;
      const float sw_n = s_sw[row], b_n = s_bias[row];
      for (int c0 = 16 * h; c0 < bt; c0 += 32) {
        uint32_t v[16];
        tmem_ld_x16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c0, v);
        tmem_ld_wait();
        if (n < a.N) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int m = m0 + c0 + j;
            if (m < a.M) {
              const int32_t acc = __float2int_rn(__uint_as_float(v[j]) * unit);
              if (raw_out) {
                a.acc[(size_t)m * a.N + n] = acc;
              } else {
                const float y = __fadd_rn(__fmul_rn(__fmul_rn((float)acc, s_sx[c0 + j]), sw_n), b_n);
                a.Y[(size_t)m * a.N + n] = f32_to_bf16_rn(y);
              }
            }
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();
  } else if (a.push) {
    // split K, push: every CTA sends each owner the int32 rows of the owner's
    // channel slice (st.async, counted on the owner's red_full); the owner sums
    // the S slices from its own shared memory.  No CTA reads a peer's shared
    // memory, so no closing cluster barrier is needed.
    cluster_wait();  // peers' red_full barriers are initialised
    if (warp >= 2 && go) {
      const int owner = row / a.rows_per, rr = row - owner * a.rows_per;
      const uint32_t off = (uint32_t)((rank * a.rows_per + rr) * ldr) * 4u;  // slot = this rank
      const uint32_t dst = mapa_shared(smem_addr(recv) + off, (uint32_t)owner);
      const uint32_t bar = mapa_shared(smem_addr(red_full), (uint32_t)owner);
      for (int c0 = 16 * h; c0 < bt; c0 += 32) {
        uint32_t v[16];
        tmem_ld_x16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c0, v);
        tmem_ld_wait();
        int4 w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          w[j] = make_int4(__float2int_rn(__uint_as_float(v[4 * j]) * unit),
                           __float2int_rn(__uint_as_float(v[4 * j + 1]) * unit),
                           __float2int_rn(__uint_as_float(v[4 * j + 2]) * unit),
                           __float2int_rn(__uint_as_float(v[4 * j + 3]) * unit));
        if (owner == (int)rank) {
#pragma unroll
          for (int j = 0; j < 4; ++j) *reinterpret_cast<int4*>(recv + (off / 4) + c0 + 4 * j) = w[j];
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) st_async_v4(dst + (uint32_t)(c0 + 4 * j) * 4u, w[j], bar);
        }
      }
    }
    __syncthreads();  // this CTA's own slice is in place
    if (nr_own > 0) {
      bool ok = mbar_wait_bounded(red_full, 0, a.wait_limit_ns, nullptr);
      if (!ok) record_timeout(a.status, abort);
      if (ok && !*abort) {
        for (int idx = tid; idx < nr_own * bt; idx += kThreads) {
          const int rr = idx % nr_own, col = idx / nr_own;
          const int m = m0 + col, n = n0 + r0_own + rr;
          if (m >= a.M || n >= a.N) continue;
          int32_t acc = 0;
          for (int c = 0; c < S; ++c) acc += recv[(c * a.rows_per + rr) * ldr + col];
          if (raw_out) {
            a.acc[(size_t)m * a.N + n] = acc;
          } else {
            const float y = __fadd_rn(__fmul_rn(__fmul_rn((float)acc, s_sx[col]), s_sw[r0_own + rr]),
                                      s_bias[r0_own + rr]);
            a.Y[(size_t)m * a.N + n] = f32_to_bf16_rn(y);
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();
  } else {
    // split K: int32 partial tile part[token][channel] in this CTA's shared
    // memory (it overlays the idle rings); after a cluster barrier, CTA r of
    // the cluster sums channels [r0, r0 + rows_per) over all S partials with
    // 16-byte DSMEM loads and writes them out.
    int32_t* part = reinterpret_cast<int32_t*>(base);
    if (warp >= 2 && go) {
      for (int c0 = 16 * h; c0 < bt; c0 += 32) {
        uint32_t v[16];
        tmem_ld_x16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) part[(c0 + j) * kTileN + row] = __float2int_rn(__uint_as_float(v[j]) * unit);
      }
    }
    tc_fence_before();
    cluster_sync_all();
    if (!*abort) {
      const int rows_per = a.rows_per;
      const int r0 = (int)rank * rows_per;
      const int nq = (min(kTileN, r0 + rows_per) - r0) / 4;  // 4-channel groups owned here
      const uint32_t part_s = smem_addr(part);
      const bool vec = (a.N & 3) == 0;
      for (int idx = tid; idx < nq * bt; idx += kThreads) {
        const int rr = r0 + 4 * (idx % nq), col = idx / nq;
        const int m = m0 + col, n = n0 + rr;
        if (m >= a.M || n >= a.N) continue;
        const uint32_t off = (uint32_t)(col * kTileN + rr) * 4u;
        int4 pv[kMaxSplit];
#pragma unroll
        for (int c = 0; c < kMaxSplit; ++c)
          if (c < S) pv[c] = ld_shared_cluster_v4(mapa_shared(part_s + off, (uint32_t)c));
        int32_t acc[4] = {0, 0, 0, 0};
#pragma unroll
        for (int c = 0; c < kMaxSplit; ++c)
          if (c < S) {
            acc[0] += pv[c].x; acc[1] += pv[c].y; acc[2] += pv[c].z; acc[3] += pv[c].w;
          }
        if (raw_out) {
          int32_t* dst = a.acc + (size_t)m * a.N + n;
          if (vec) {
            *reinterpret_cast<int4*>(dst) = make_int4(acc[0], acc[1], acc[2], acc[3]);
          } else {
            for (int e = 0; e < 4 && n + e < a.N; ++e) dst[e] = acc[e];
          }
        } else {
          uint16_t y[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            y[e] = f32_to_bf16_rn(__fadd_rn(__fmul_rn(__fmul_rn((float)acc[e], s_sx[col]), s_sw[rr + e]),
                                            s_bias[rr + e]));
          uint16_t* dst = a.Y + (size_t)m * a.N + n;
          if (vec) {
            *reinterpret_cast<uint2*>(dst) = make_uint2((uint32_t)y[0] | ((uint32_t)y[1] << 16),
                                                        (uint32_t)y[2] | ((uint32_t)y[3] << 16));
          } else {
            for (int e = 0; e < 4 && n + e < a.N; ++e) dst[e] = y[e];
          }
        }
      }
    }
    cluster_sync_all();  // peers have finished reading this CTA's shared memory
  }
  if (warp == 1) tmem_dealloc(tmem, a.tmem_cols);
}

// ------------------------------------------------------------------ host side

// Tensor map of a [rows, row_bytes] uint8 matrix, box = 64 bytes x box_rows,
// no swizzle; out-of-range rows read as zero.
bool make_tmap(CUtensorMap* tm, const void* ptr, int rows, int row_bytes, int box_rows) {
  return vqlin::encode_tmap_2d(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, ptr, (uint64_t)row_bytes, (uint64_t)rows,
                               (uint64_t)row_bytes, kRawRow, (uint32_t)box_rows, CU_TENSOR_MAP_SWIZZLE_NONE);
}

constexpr int kMaxSmem = 232448 - 4096;

// dynamic shared memory: alignment slack, operand and raw rings, barriers,
// and (push reduction) the receive buffer of S slices [rows_per][bt + 4] int32
size_t smem_bytes(int bt, int raw_stages, int S, int rows_per, bool push) {
  const size_t rows = kTileN + bt;
  size_t b = 1024 + kOpStages * rows * kOpRow + raw_stages * rows * kRawRow + (2 * raw_stages + 2 * kOpStages + 4) * 8;
  if (push) b += (size_t)S * rows_per * (bt + 4) * 4;
  return b;
}

template <int BITS>
vqlin_status launch_bits(const void* xq, const float* sx, const void* wq, const float* sw, const uint16_t* bias,
                         uint16_t* Y, int32_t* acc, int M, int N, int K, int* status, int withhold,
                         uint64_t limit_ns, cudaStream_t st) {
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(qgemm_kernel<BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(qgemm_kernel<BITS>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
  if (attr_err != cudaSuccess)
    return vqlin::fail(VQLIN_ERR_CUDA, "qgemm: cudaFuncSetAttribute: %s", cudaGetErrorString(attr_err));

  const int kb_codes = BITS == 4 ? 128 : 64;
  const int row_bytes = BITS == 4 ? K / 2 : K;
  const int nt = (M + 255) / 256;
  const int bt = ((M + nt - 1) / nt + 15) / 16 * 16;
  const int tiles_n = (N + kTileN - 1) / kTileN, tiles_m = (M + bt - 1) / bt;
  const int nkb = K / kb_codes;
  const int s_min = BITS == 8 ? (K + 1023) / 1024 : 1;
  int S = (148 + tiles_n * tiles_m - 1) / (tiles_n * tiles_m);
  S = S < s_min ? s_min : S;
  S = S > kMaxSplit ? kMaxSplit : S;
  S = S > nkb ? nkb : S;
  if (S < s_min)  // host checks keep K <= 16384 for int8
    return vqlin::fail(VQLIN_ERR_UNSUPPORTED_SHAPE, "qgemm: K=%d needs %d-way split", K, s_min);
  const int per_cta = (nkb + S - 1) / S;
  // channels each cluster rank owns in the split-K epilogue (a multiple of 4)
  const int rows_per = S > 1 ? ((kTileN + S - 1) / S + 3) & ~3 : kTileN;
  // raw stages: up to 6 within the shared-memory limit, no more than the
  // k-blocks a CTA runs, at least 2 (the int32 partial tile of the pull
  // epilogue overlays the rings and needs 2 raw stages' room for bt <= 256)
  const int r_cap = per_cta < 2 ? 2 : (per_cta > 6 ? 6 : per_cta);
  bool push = S > 1 && smem_bytes(bt, 2, S, rows_per, true) <= (size_t)kMaxSmem;
  int R = r_cap;
  while (R > 2 && smem_bytes(bt, R, S, rows_per, push) > (size_t)kMaxSmem) --R;
  const bool tma_store = S == 1 && acc == nullptr && (N % 8) == 0;
  uint32_t cols = 32;
  while ((int)cols < bt) cols <<= 1;

  CUtensorMap tmW, tmX, tmY;
  if (!vqlin::tmap_encoder_available())
    return vqlin::fail(VQLIN_ERR_CUDA, "qgemm: cuTensorMapEncodeTiled is unavailable");
  if (!make_tmap(&tmW, wq, N, row_bytes, kTileN) || !make_tmap(&tmX, xq, M, row_bytes, bt))
    return vqlin::fail(VQLIN_ERR_CUDA, "qgemm: tensor map encoding failed (M=%d N=%d K=%d)", M, N, K);
  if (tma_store) {
    if (!vqlin::encode_tmap_2d(&tmY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Y, (uint64_t)N, (uint64_t)M, (uint64_t)N * 2,
                               kTileN, (uint32_t)bt, CU_TENSOR_MAP_SWIZZLE_NONE))
      return vqlin::fail(VQLIN_ERR_CUDA, "qgemm: output tensor map encoding failed (M=%d N=%d)", M, N);
  } else {
    tmY = tmW;  // unused
  }

  QgemmArgs a;
  a.sx = sx; a.sw = sw; a.bias = bias; a.Y = Y; a.acc = acc; a.status = status;
  a.M = M; a.N = N; a.K = K; a.bt = bt; a.nkb = nkb; a.raw_stages = R; a.tmem_cols = cols;
  a.wait_limit_ns = limit_ns; a.withhold_loads = withhold;
  a.tma_store = tma_store ? 1 : 0; a.push = push ? 1 : 0; a.rows_per = rows_per;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles_n, tiles_m, S);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes(bt, R, S, rows_per, push);
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
  const cudaError_t e = cudaLaunchKernelEx(&cfg, qgemm_kernel<BITS>, tmW, tmX, tmY, a);
  if (e != cudaSuccess)
    return vqlin::fail(VQLIN_ERR_CUDA, "qgemm launch (grid %d x %d x %d, cluster %d, %zu B smem): %s", tiles_n,
                       tiles_m, S, S, cfg.dynamicSmemBytes, cudaGetErrorString(e));
  return VQLIN_OK;
}

}  // namespace

namespace vqlin {

vqlin_status launch_int_gemm(int bits, const void* xq, const float* sx, const void* wq, const float* sw,
                             const uint16_t* bias, uint16_t* Y, int32_t* acc, int M, int N, int K, int* status,
                             cudaStream_t st) {
  if (M == 0 || N == 0) return VQLIN_OK;
  if (bits == 4) return launch_bits<4>(xq, sx, wq, sw, bias, Y, acc, M, N, K, status, 0, kWaitLimitNs, st);
  return launch_bits<8>(xq, sx, wq, sw, bias, Y, acc, M, N, K, status, 0, kWaitLimitNs, st);
}

vqlin_status launch_int_gemm_withheld(int bits, const void* xq, const void* wq, int32_t* acc, int M, int N, int K,
                                     int* status, uint64_t limit_ns, cudaStream_t st) {
  if (bits == 4) return launch_bits<4>(xq, nullptr, wq, nullptr, nullptr, nullptr, acc, M, N, K, status, 1, limit_ns, st);
  return launch_bits<8>(xq, nullptr, wq, nullptr, nullptr, nullptr, acc, M, N, K, status, 1, limit_ns, st);
}

}  // namespace vqlin
