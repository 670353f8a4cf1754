// Few-token W4A4 projections (the batch-1 action expert: tens of tokens) on
// the tcgen05 tensor cores, built for latency rather than throughput.
//
//   acc[m, n] = sum_k xq[m, k] * wq[n, k]        (exact int32)
//   Y[m, n]   = bf16(((float)acc * sx[m]) * sw[n] + bias[n])
//
// Method: "FoldQuantVLA" abstract (block Hadamard transform, per-token
// quantization, native integer W4A4); "Omega-QVLA" technical summary, section
// "Scalatura delle Attivazioni DiT per Passo" (precomputed per-step activation
// scales for the action expert); "LoopQ" abstract (the batch-1 action expert
// is memory-bound and dominates GPU time).
//
// At a few tokens a projection moves well under a microsecond of HBM data and
// does even less arithmetic, so its time is the chain of latencies after the
// previous kernel finishes.  This kernel keeps that chain short:
//   * everything that does not depend on the previous kernel happens before
//     griddepcontrol.wait (programmatic dependent launch): every packed weight
//     tile of the CTA's K range is loaded by TMA and expanded into the MMA's A
//     operand in tensor memory, where all of it stays (at most 8 k-blocks of
//     128 channels = 256 columns);
//   * static-scale variant (FUSED): the bf16 activations are rotated (block
//     Hadamard) and quantized on chip exactly as the activation kernel does,
//     but each k-block of each token group is quantized once per cluster, not
//     once per CTA: the CTAs of a cluster split those units among their warps,
//     write the codes to the code buffer xq [M, K] in global memory (they stay
//     in L2), meet at one cluster barrier and then load the codes of their K
//     range by TMA.  Shared memory between CTAs would move these bytes at
//     about 16 bytes per clock per SM on B300; L2 at several times that and a
//     ~140 ns round trip, so L2 is the exchange medium;
//   * codes variant: the codes come from the activation kernel; their TMA loads
//     are issued right after the wait;
//   * K longer than 8 k-blocks is split over the cluster's z dimension (at most
//     16 CTAs per cluster) and reduced on chip: each split rank reads its
//     slice of every peer's int32 partial tile from distributed shared memory.
// Roles (14 warps): warp 0 loads tiles (lane 0) and stages the epilogue's
// scales (lanes 1..31); warps 2..9 expand the weights, then quantize
// activations, then run the epilogue (two per tensor-memory lane quadrant);
// warps 10..13 quantize.  (Sixteen warps with every warp in the epilogue
// measured slower.)  The MMAs come
// from up to four issuing warps (1, 10, 11, 12), each summing every NI-th
// k-block into an accumulator of its own: one thread issues at most one
// tcgen05.mma per ~116 SM clocks on B300 whatever its N, so at N = 64 tokens a
// single issuer reaches only a quarter of the tensor pipe's rate; four
// issuers reach all of it.  The accumulators hold integers x 2^-18 (exact),
// so the epilogue adds them exactly.
// Every mbarrier wait is bounded in time (VQLIN_ERR_TIMEOUT in the status
// word); every thread reaches every cluster barrier on every path.
#include <mutex>

#include "act_codes.cuh"
#include "common.cuh"
#include "tc_ptx.cuh"

namespace {

using namespace vqlin_dev;

constexpr int kTileN = 128;         // output channels per CTA (MMA M)
constexpr int kThreads = 448;       // 14 warps
constexpr int kExpandWarps = 8;     // warps 2..9
constexpr int kMaxKb = 8;           // k-blocks (128 channels) of one CTA: A resident in 8 x 32 columns
constexpr int kMaxCluster = 16;
constexpr int kWRow = 64;           // packed weight bytes of one row per k-block
constexpr int kBRow = 128;          // activation code bytes of one token per k-block
constexpr uint32_t kWTile = kTileN * kWRow;  // 8 KB
constexpr uint64_t kWaitLimitNs = 1000000000ull;

struct LowlatArgs {
  const uint16_t* X;            // FUSED: bf16 activations [M, K]
  const float* chan;            // FUSED with CHAN: channel factors c [K] (x / c before the rotation)
  const float* static_scale;    // FUSED: one device float
  const float* sx;              // codes variant: per-token scales [M] (sx_step 1) or one scale (0)
  int sx_step;
  const float* sw;
  const uint16_t* bias;
  uint16_t* Y;
  uint8_t* xq;                  // FUSED: code buffer [M, K] (written, then read back by TMA)
  int* status;
  int M, N, K;
  int bt;                       // token tile (multiple of 16, <= 128)
  int nkb;                      // k-blocks of K
  int cn;                       // CTAs of a cluster along N
  uint32_t tmem_cols;
  int rows_per;                 // split K: output channels each split rank owns
  int issuers;                  // MMA-issuing warps, one accumulator each (1, 2 or 4)
  uint64_t wait_limit_ns;
};

// 8 packed int4 weight bytes (sign-magnitude nibbles, even channel low) ->
// 4 words of e4m3 operand bytes s<<7 | |c| in channel order.
__device__ __forceinline__ void expand8_w4(uint32_t lo, uint32_t hi, uint32_t* o) {
  const uint32_t e0 = (lo & 0x07070707u) | ((lo << 4) & 0x80808080u);
  const uint32_t o0 = ((lo >> 4) & 0x07070707u) | (lo & 0x80808080u);
  const uint32_t e1 = (hi & 0x07070707u) | ((hi << 4) & 0x80808080u);
  const uint32_t o1 = ((hi >> 4) & 0x07070707u) | (hi & 0x80808080u);
  o[0] = __byte_perm(e0, o0, 0x5140);
  o[1] = __byte_perm(e0, o0, 0x7362);
  o[2] = __byte_perm(e1, o1, 0x5140);
  o[3] = __byte_perm(e1, o1, 0x7362);
}

__device__ __forceinline__ void record_timeout(int* status, volatile int* abort) {
  *abort = 1;
  atomicCAS(status, 0, (int)VQLIN_ERR_TIMEOUT);
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ float ldg_nc_f32(const float* p) {
  float r;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(r) : "l"(p));
  return r;
}

template <bool FUSED, int HB, bool CHAN = false>
__global__ void __launch_bounds__(kThreads, 1)
w4a4_lowlat_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmXq,
                   const LowlatArgs a) {
  extern __shared__ uint8_t smem_dyn[];
  __shared__ __align__(8) uint64_t s_bar[3 * kMaxKb + 3];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_unit;
  __shared__ __align__(16) float s_sx[128];
  __shared__ float s_sw[kTileN], s_bias[kTileN];

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  const int bt = a.bt;
  const uint32_t b_tile = (uint32_t)bt * kBRow;  // a multiple of 2048
  uint64_t* wfull = s_bar;                 // [kMaxKb] weight tile landed
  uint64_t* aready = s_bar + kMaxKb;       // [kMaxKb] A operand expanded into tensor memory
  uint64_t* bfull = s_bar + 2 * kMaxKb;    // [kMaxKb] activation codes landed
  uint64_t* acc_full = s_bar + 3 * kMaxKb; // every issuer's MMAs completed
  uint64_t* scl_ready = acc_full + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = (int)gridDim.z, split = (int)blockIdx.z;
  const int cx = (int)(blockIdx.x % (unsigned)a.cn);
  const uint32_t crank = cluster_ctarank();
  const uint32_t csize = (uint32_t)(a.cn * S);
  const int n0 = blockIdx.x * kTileN, m0 = blockIdx.y * bt;
  const bool live = n0 < a.N;  // clusters are padded along N; padded CTAs only quantize
  const int kb0 = (int)(((long long)split * a.nkb) / S);
  const int kb1 = (int)(((long long)(split + 1) * a.nkb) / S);
  const int cnt = live ? kb1 - kb0 : 0;
  const int mt = min(bt, a.M - m0);      // tokens of this tile
  const int NI = a.issuers;              // MMA issuers = accumulators
  const int n_acc = min(NI, cnt);        // accumulators that receive MMAs
  const uint32_t acc_step = (uint32_t)(((bt + 31) / 32) * 32);
  const uint32_t a_col = (uint32_t)NI * acc_step;  // A slots after the accumulators
  // B stages first (1024-aligned tiles), then the packed weight tiles
  const int cnt_max = (a.nkb + S - 1) / S;
  uint8_t* wbase = base + (size_t)cnt_max * b_tile;
  volatile int* abort = &s_abort;

  if (tid == 0) {
    s_abort = 0;
    s_unit = 0;
    for (int i = 0; i < kMaxKb; ++i) {
      mbar_init(&wfull[i], 1);
      mbar_init(&aready[i], kExpandWarps / 2);  // one group of four warps per k-block
      mbar_init(&bfull[i], 1);
    }
    mbar_init(acc_full, NI);
    mbar_init(scl_ready, 31);
    mbar_init_fence();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmXq);
  }
  if (warp == 1) tmem_alloc(&s_tmem, a.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  // Rotate + quantize units (k-block j, group of 8 tokens) of the cluster's
  // token tile; the units u = crank + csize * i are this CTA's, taken by its
  // warps from a shared counter.  Same Hadamard unit and rounding as the
  // activation kernel, so the codes equal its codes bit for bit.
  auto quantize_units = [&]() {
    constexpr int LPG = HB / 32;
    const int TG = (mt + 7) / 8;
    const int total = a.nkb * TG;
    const int rl = lane >> 2, l4 = lane & 3;
    const int g = l4 / LPG, l = l4 % LPG;  // Hadamard block inside the k-block; lane inside the block
    for (;;) {
      int ul = 0;
      if (lane == 0) ul = atomicAdd(&s_unit, 1);
      ul = __shfl_sync(0xffffffffu, ul, 0);
      const int u = (int)crank + (int)csize * ul;
      if (u >= total) break;
      const int j = u / TG, t8 = u - j * TG;
      const int r = t8 * 8 + rl;
      const bool ok = r < mt;
      const size_t row = (size_t)(m0 + (ok ? r : 0)) * a.K + (size_t)j * 128;
      uint4 raw[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        raw[c] = make_uint4(0, 0, 0, 0);
        if (ok) raw[c] = ldg_nc_v4(a.X + row + HB * g + 8 * (l + LPG * c));
      }
      // the scale's load is issued after the activations', so both are in flight together
      const float xs = ldg_nc_f32(a.static_scale);
      float v[4][8];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        v[c][0] = bf16_lo(raw[c].x); v[c][1] = bf16_hi(raw[c].x);
        v[c][2] = bf16_lo(raw[c].y); v[c][3] = bf16_hi(raw[c].y);
        v[c][4] = bf16_lo(raw[c].z); v[c][5] = bf16_hi(raw[c].z);
        v[c][6] = bf16_lo(raw[c].w); v[c][7] = bf16_hi(raw[c].w);
      }
      if (CHAN && ok) {
        // channel scaling: x / c[k] by IEEE division before the rotation, as
        // the activation kernel does
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float* cp = a.chan + (size_t)j * 128 + HB * g + 8 * (l + LPG * c);
          const float4 c0 = __ldg(reinterpret_cast<const float4*>(cp));
          const float4 c1 = __ldg(reinterpret_cast<const float4*>(cp + 4));
          const float cc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) v[c][e] = __fdiv_rn(v[c][e], cc[e]);
        }
      }
      hadamard_unit<HB>(v, lane);
      if (ok) {
        const float kq = (xs > 0.0f ? __frcp_rn(xs) : 0.0f) * (1.0f / 512.0f);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t w[4];
          quantize_chunk_fast<4>(v[c], kq, w);
          *reinterpret_cast<uint2*>(a.xq + row + HB * g + 8 * (l + LPG * c)) = make_uint2(w[0], w[1]);
        }
      }
    }
    // the codes are read by TMA (async proxy) in other CTAs after the barrier
    fence_proxy_async_global();
  };

  // MMA issuer i: k-blocks i, i + NI, ... into accumulator i (whole warp runs
  // the loop, one elected lane issues), then one commit on acc_full.
  auto issue_mmas = [&](int i) {
    const uint32_t id = idesc_f32acc(0u, kTileN, bt);  // e4m3 x e4m3 -> f32
    const uint64_t db0 = sdesc_sw128(base);
    const uint64_t dstep = (uint64_t)(b_tile >> 4);    // start-address field step per B tile
    const uint32_t d = tmem + (uint32_t)i * acc_step;
    for (int j = i; j < cnt; j += NI) {
      const bool ok = mbar_wait_bounded(&aready[j], 0, a.wait_limit_ns, abort) &&
                      mbar_wait_bounded(&bfull[j], 0, a.wait_limit_ns, abort);
      if (!__all_sync(0xffffffffu, ok)) {
        if (!ok && !*abort) record_timeout(a.status, abort);
        break;
      }
      tc_fence_after();
      const uint64_t db = db0 + (uint64_t)j * dstep;
      const uint32_t ta = tmem + a_col + (uint32_t)(j * 32);
      // per MMA: 8 tensor-memory columns of A, 32 bytes along the swizzled B row
      mma_f8f6f4_ta_warp(d, ta, db, id, j != i ? 1u : 0u);
      mma_f8f6f4_ta_warp(d, ta + 8, db + 2, id, 1u);
      mma_f8f6f4_ta_warp(d, ta + 16, db + 4, id, 1u);
      mma_f8f6f4_ta_warp(d, ta + 24, db + 6, id, 1u);
    }
    tc_commit_warp(acc_full);
  };

  if (warp == 0) {
    // ---------------------------------------------------- loads and scales
    auto load_codes = [&]() {
      for (int j = 0; j < cnt; ++j) {
        mbar_arrive_expect_tx(&bfull[j], b_tile);
        tma_load_2d(base + (size_t)j * b_tile, &tmXq, (kb0 + j) * kBRow, m0, &bfull[j]);
      }
    };
    // weight tiles, per-channel scales and bias do not depend on the previous
    // kernel: all of them are requested before waiting for it
    float wv[5], bv[5];
    if (lane == 0) {
      for (int j = 0; j < cnt; ++j) {
        mbar_arrive_expect_tx(&wfull[j], kWTile);
        tma_load_2d(wbase + (size_t)j * kWTile, &tmW, (kb0 + j) * kWRow, n0, &wfull[j]);
      }
    } else {
#pragma unroll
      for (int q = 0; q < 5; ++q) {
        const int i = lane - 1 + 31 * q;
        const bool in = i < kTileN && n0 + i < a.N;
        wv[q] = in ? __ldg(a.sw + n0 + i) : 0.0f;
        bv[q] = in && a.bias != nullptr ? __uint_as_float((uint32_t)__ldg(a.bias + n0 + i) << 16) : 0.0f;
      }
    }
    __syncwarp();
    pdl_wait();
    // the next kernel may start its own preparation now, while this one works:
    // triggering earlier lets a chain of launches prefetch their weights all at
    // once and slow this kernel's own loads
    if (lane == 0) pdl_trigger();
    if (!FUSED && lane == 0) load_codes();  // codes of the activation kernel
    if (lane > 0) {
      const float xs = FUSED ? __ldg(a.static_scale) : 0.0f;
      // token scales in the accumulator's unit: the float32 sums of e4m3
      // operands are integers x 2^-18 (unsplit K); split-K sums arrive as int32
      const float su = S == 1 ? 262144.0f : 1.0f;
#pragma unroll
      for (int q = 0; q < 5; ++q) {
        const int i = lane - 1 + 31 * q;
        if (i < kTileN) {
          s_sw[i] = wv[q];
          s_bias[i] = bv[q];
        }
        if (i < 128) s_sx[i] = i < mt ? (FUSED ? xs : __ldg(a.sx + (size_t)(m0 + i) * a.sx_step)) * su : 0.0f;
      }
      mbar_arrive(scl_ready);
    }
    __syncwarp();
    if (FUSED) {
      cluster_arrive();
      cluster_wait();  // every CTA of the cluster has written its codes
    }
    if (lane == 0) {
      if (FUSED && cnt > 0) {
        fence_proxy_async_global();
        load_codes();
      }
      // copies in flight complete before the CTA may exit: once every MMA
      // has completed, every copy has landed; only a CTA that gave up checks
      // them one by one.  (Checking the 2 x cnt barriers in turn kept this
      // warp from the final barrier ~1.5 us after the MMAs had finished.)
      const bool all_done = mbar_wait_bounded(acc_full, 0, a.wait_limit_ns, abort);
      if (!all_done || *abort) {
        for (int j = 0; j < cnt; ++j) {
          if (!mbar_wait_bounded(&wfull[j], 0, a.wait_limit_ns, nullptr)) record_timeout(a.status, abort);
          if (!mbar_wait_bounded(&bfull[j], 0, a.wait_limit_ns, nullptr)) record_timeout(a.status, abort);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer 0
    if (FUSED) {
      cluster_arrive();
      cluster_wait();
    }
    issue_mmas(0);
  } else {
    if (warp < 2 + kExpandWarps) {
      // ------------------------------------------ weight expanders (2..9)
      // thread = weight row; the two groups of four warps take alternate
      // k-blocks; the expanded A operand stays in its own slot
      const int q = warp & 3, grp = (warp - 2) >> 2;
      const int row = q * 32 + lane;
      const int sw = (row >> 1) & 3;  // 64-byte swizzle of the packed tile
      const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16) + a_col;
      for (int j = grp; j < cnt; j += 2) {
        const bool ok = mbar_wait_bounded(&wfull[j], 0, a.wait_limit_ns, abort);
        if (!__all_sync(0xffffffffu, ok)) {
          if (!ok && !*abort) record_timeout(a.status, abort);
          break;
        }
        const uint8_t* rawrow = wbase + (size_t)j * kWTile + row * kWRow;
        uint4 rw[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) rw[c] = *reinterpret_cast<const uint4*>(rawrow + ((c ^ sw) << 4));
        uint32_t v[2][16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          expand8_w4(rw[c].x, rw[c].y, &v[c >> 1][8 * (c & 1)]);
          expand8_w4(rw[c].z, rw[c].w, &v[c >> 1][8 * (c & 1) + 4]);
        }
        const uint32_t ta = trow + (uint32_t)(j * 32);
        tmem_st_x16(ta, v[0]);
        tmem_st_x16(ta + 16, v[1]);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&aready[j]);
      }
    }
    if (FUSED) {
      // ------------------------------- activation quantizers (2..13)
      pdl_wait();  // X and the static scale come from the previous kernel
      quantize_units();
      __syncwarp();
      cluster_arrive();
      cluster_wait();
    }
    // ---------------------------------------- MMA issuers 1..3 (10, 11, 12)
    if (warp >= 2 + kExpandWarps && warp - (1 + kExpandWarps) < NI) issue_mmas(warp - (1 + kExpandWarps));
  }

  // ---------------------------------------------------------------- epilogue
  // warps 2..9: lane quadrant q = warp % 4, token chunks 16 h + 32 i with
  // h = (warp - 2) / 4.  (One waiting warp releasing the others through a
  // named barrier measured about 1 us slower per launch.)
  __syncwarp();
  const bool epi = warp >= 2 && warp < 2 + kExpandWarps;  // the epilogue's warps
  bool go = false;
  if (epi) {
    const bool ok = mbar_wait_bounded(acc_full, 0, a.wait_limit_ns, nullptr) &&
                    mbar_wait_bounded(scl_ready, 0, a.wait_limit_ns, nullptr);
    if (!ok) record_timeout(a.status, abort);
    tc_fence_after();
    go = __all_sync(0xffffffffu, ok && !*abort && cnt > 0);
  }
  pdl_wait();  // global writes only once the previous kernel has finished
  const int q = warp & 3;
  const int cfirst = 16 * ((warp - 2) >> 2);
  const int row = q * 32 + lane;  // output channel inside the tile
  const uint32_t lanes_q = tmem + ((uint32_t)(q * 32) << 16);
  // the sum of the used accumulators over tokens c0 .. c0 + 15 (float, the
  // accumulator's unit; exact: integers x 2^-18 below 2^24)
  auto load_sum = [&](int c0, float (&f)[16]) {
    uint32_t v[4][16];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (i < n_acc) tmem_ld_x16(lanes_q + (uint32_t)i * acc_step + (uint32_t)c0, v[i]);  // warp-uniform
    tmem_ld_wait();
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      float t = __uint_as_float(v[0][jj]);
#pragma unroll
      for (int i = 1; i < 4; ++i)
        if (i < n_acc) t += __uint_as_float(v[i][jj]);
      f[jj] = t;
    }
  };

  if (S == 1) {
    // thread = channel, 16 tokens per tensor-memory load; each warp stages its
    // 16 tokens x 32 channels as bf16 over the dead operand tiles and writes
    // every token's 64 bytes as four 16-byte stores (a warp's 2-byte stores
    // to 16 token rows measured ~35 ns each)
    if (go) {
      const int n = n0 + row;
      const float sw_n = s_sw[row], b_n = s_bias[row];
      const bool vec = (a.N & 7) == 0;  // 16-byte aligned token rows
      uint16_t* stg = reinterpret_cast<uint16_t*>(base) + (warp - 2) * 512;
      for (int c0 = cfirst; c0 < bt; c0 += 32) {
        float f[16];
        load_sum(c0, f);
        // token scales into registers first: Y is a generic pointer, so a
        // shared-memory read after each store would be reissued and wait
        float sx[16];
#pragma unroll
        for (int jj = 0; jj < 16; jj += 4) {
          const float4 t = *reinterpret_cast<const float4*>(&s_sx[c0 + jj]);
          sx[jj] = t.x; sx[jj + 1] = t.y; sx[jj + 2] = t.z; sx[jj + 3] = t.w;
        }
        uint16_t yb[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) yb[jj] = f32_to_bf16_rn(fmaf(f[jj] * sx[jj], sw_n, b_n));
        if (vec) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) stg[jj * 32 + lane] = yb[jj];
          __syncwarp();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int tok = h * 8 + (lane >> 2), part = lane & 3;
            const int nn = n0 + q * 32 + part * 8;
            if (c0 + tok < mt && nn < a.N)
              *reinterpret_cast<uint4*>(a.Y + (size_t)(m0 + c0 + tok) * a.N + nn) =
                  *reinterpret_cast<const uint4*>(stg + tok * 32 + part * 8);
          }
          __syncwarp();
        } else if (n < a.N) {
          uint16_t* yp = a.Y + (size_t)(m0 + c0) * a.N + n;
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            if (c0 + jj < mt) yp[(size_t)jj * a.N] = yb[jj];
        }
      }
    }
    tc_fence_before();
    __syncthreads();
  } else {
    // split K among the S CTAs of this output tile (cluster ranks cx + cn *
    // r): split rank r owns channels [r rp, (r + 1) rp).  Every CTA writes its
    // int32 partial tile into its own shared memory as S slices
    // part[r][token][rp] over the dead operand tiles; after one cluster
    // barrier rank r reads slice r of every CTA of the tile (distributed
    // shared memory, 16-byte loads), adds them, scales and stores; a second
    // barrier keeps each CTA's shared memory alive until its peers have read
    // it.  Integer sums: exact in any order.  (Pushing the slices with one
    // bulk reduction per peer and waiting for them to land took 0.7 us more
    // at 50 x 1024 x 4096.)
    const int rp = a.rows_per;
    const uint32_t slice_words = (uint32_t)(bt * rp);
    const int own0 = split * rp;
    const int own_n = (live && own0 < kTileN) ? min(rp, kTileN - own0) : 0;
    uint32_t* part = reinterpret_cast<uint32_t*>(base);
    if (epi && live) {
      const int sl = row / rp, k = row - sl * rp;
      uint32_t* dst = part + (size_t)sl * slice_words + k;
      for (int c0 = cfirst; c0 < bt; c0 += 32) {
        float f[16];
        if (go) {
          load_sum(c0, f);
        } else {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) f[jj] = 0.0f;  // aborted: zeros (the status word reports it)
        }
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          // |sum| < 2^22: the integer sits in the low mantissa bits of
          // sum * 2^18 + 1.5 x 2^23 (exact)
          dst[(size_t)(c0 + jj) * rp] = (uint32_t)(__float_as_int(fmaf(f[jj], 262144.0f, 12582912.0f)) - 0x4B400000);
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    cluster_sync_all();  // every CTA's partial slices are in place
    if (own_n > 0 && !*abort) {
      const int nq = own_n / 4;
      const int total = nq * bt;
      const bool vec = (a.N & 3) == 0;
      const uint32_t mine = smem_addr(part + (size_t)split * slice_words);
      for (int idx = tid; idx < total; idx += kThreads) {
        const int c = idx / nq, k = 4 * (idx - c * nq);
        const int m = m0 + c, rr = own0 + k, n = n0 + rr;
        if (m >= a.M || n >= a.N) continue;
        const uint32_t src = mine + (uint32_t)((c * rp + k) * 4);
        int32_t acc[4] = {0, 0, 0, 0};
#pragma unroll 4
        for (int r = 0; r < S; ++r) {
          const float4 t = ld_shared_cluster_v4f(mapa_shared(src, (uint32_t)(cx + a.cn * r)));
          acc[0] += __float_as_int(t.x);
          acc[1] += __float_as_int(t.y);
          acc[2] += __float_as_int(t.z);
          acc[3] += __float_as_int(t.w);
        }
        const float sx_m = s_sx[c];
        float y[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) y[e] = fmaf((float)acc[e] * sx_m, s_sw[rr + e], s_bias[rr + e]);
        uint16_t* o = a.Y + (size_t)m * a.N + n;
        if (vec) {
          *reinterpret_cast<uint2*>(o) = make_uint2(pack_bf16x2_rn(y[0], y[1]), pack_bf16x2_rn(y[2], y[3]));
        } else {
          for (int e = 0; e < 4 && n + e < a.N; ++e) o[e] = f32_to_bf16_rn(y[e]);
        }
      }
    }
    __syncwarp();
    cluster_sync_all();  // peers have read this CTA's slices
  }
  if (warp == 1) tmem_dealloc(tmem, a.tmem_cols);
}

// ------------------------------------------------------------------ host side

constexpr int kMaxSmem = 232448 - 4096;
constexpr size_t kSmemPerSm = 233472;

struct LowlatPlan {
  int bt = 0, tiles_n = 0, tiles_n_pad = 0, tiles_m = 0, S = 0, cn = 0, rows_per = 0, issuers = 0;
  uint32_t cols = 0;
  size_t dyn = 0;
};

template <bool FUSED, int HB, bool CHAN = false>
void set_attrs_once(cudaError_t* err) {
  // function attributes are per device: set them for every device used
  static std::mutex mu;
  static bool done[64] = {};
  static cudaError_t res[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!done[dev]) {
    const auto kern = w4a4_lowlat_kernel<FUSED, HB, CHAN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    res[dev] = e;
    done[dev] = true;
  }
  *err = res[dev];
}

template <bool FUSED, int HB, bool CHAN = false>
bool make_plan(int M, int N, int K, LowlatPlan& p) {
  const auto kern = w4a4_lowlat_kernel<FUSED, HB, CHAN>;
  const int nkb = K / 128;
  const int S = (nkb + kMaxKb - 1) / kMaxKb;
  if (S < 1 || S > kMaxCluster) return false;
  const int cnt_max = (nkb + S - 1) / S;
  const int tiles_m = (M + 127) / 128;
  const int bt = ((M + tiles_m - 1) / tiles_m + 15) / 16 * 16;
  const int tiles_n = (N + kTileN - 1) / kTileN;
  const int rp = S > 1 ? ((kTileN + S - 1) / S + 3) & ~3 : kTileN;
  size_t need = (size_t)cnt_max * ((size_t)bt * kBRow + kWTile);
  need = need > (size_t)S * rp * bt * 4 ? need : (size_t)S * rp * bt * 4;  // split-K partial slices
  size_t dyn = 1024 + need;
  // tensor memory: one accumulator per MMA issuer (up to 4, no more than the
  // k-blocks of a CTA), then the CTA's A operand (32 columns per k-block)
  const uint32_t acc_step = (uint32_t)(((bt + 31) / 32) * 32);
  int issuers = 4;
  while (issuers > 1 && (issuers > cnt_max || (uint32_t)issuers * acc_step + (uint32_t)(cnt_max * 32) > 512))
    issuers >>= 1;
  uint32_t cols = 32;
  while (cols < (uint32_t)issuers * acc_step + (uint32_t)(cnt_max * 32)) cols <<= 1;
  if (cols > 512 || dyn > (size_t)kMaxSmem) return false;
  // never more CTAs on an SM than its 512 tensor-memory columns hold
  const size_t dyn_floor = kSmemPerSm / (512 / cols + 1) + 1;
  if (dyn < dyn_floor) dyn = dyn_floor;
  // cluster along N: as wide as the split allows (quantization shared by more
  // CTAs) while padding adds at most half as many CTAs again (a padded CTA
  // only quantizes: at 50 x 3072 x 1024 clusters of 16 with 8 padded CTAs
  // took 5.16 us against 5.60 us for clusters of 8; at 16 x 256 x 256 padding
  // 2 tiles to 16 CTAs cost more than it saved), and schedulable
  int cn = 0;
  for (int c = kMaxCluster / S; c >= 1; c >>= 1) {
    const int pad = (tiles_n + c - 1) / c * c;
    if (c > 1 && pad - tiles_n > (FUSED ? tiles_n / 2 : tiles_n / 4)) continue;
    if (FUSED || S > 1 || c == 1) {
      if (vqlin::max_active_clusters((const void*)kern, kThreads, dyn, c * S) <= 0 && c * S > 1) continue;
    }
    cn = c;
    break;
  }
  if (!FUSED) cn = 1;  // the codes variant shares nothing along N
  if (cn == 0) return false;
  if (!FUSED && S > 1 && vqlin::max_active_clusters((const void*)kern, kThreads, dyn, S) <= 0) return false;
  p.bt = bt; p.tiles_n = tiles_n; p.tiles_n_pad = (tiles_n + cn - 1) / cn * cn; p.tiles_m = tiles_m;
  p.S = S; p.cn = cn; p.rows_per = rp; p.cols = cols; p.dyn = dyn; p.issuers = issuers;
  return true;
}

template <bool FUSED, int HB, bool CHAN = false>
vqlin_status launch_lowlat(const uint16_t* X, const float* static_scale, const uint8_t* xq_in, const float* sx,
                           uint8_t* xq_ws, const uint8_t* wq, const float* sw, const uint16_t* bias, uint16_t* Y,
                           int M, int N, int K, int* status, cudaStream_t st, int sx_step = 1,
                           const float* chan = nullptr) {
  cudaError_t ae = cudaSuccess;
  set_attrs_once<FUSED, HB, CHAN>(&ae);
  if (ae != cudaSuccess)
    return vqlin::fail(VQLIN_ERR_CUDA, "w4a4 low-latency: cudaFuncSetAttribute: %s", cudaGetErrorString(ae));
  LowlatPlan p;
  if (!make_plan<FUSED, HB, CHAN>(M, N, K, p))
    return vqlin::fail(VQLIN_ERR_UNSUPPORTED_SHAPE, "w4a4 low-latency: no plan for M=%d N=%d K=%d", M, N, K);
  const uint8_t* codes = FUSED ? xq_ws : xq_in;
  CUtensorMap tmW, tmXq;
  if (!vqlin::tmap_encoder_available())
    return vqlin::fail(VQLIN_ERR_CUDA, "w4a4 low-latency: cuTensorMapEncodeTiled is unavailable");
  const bool ok = vqlin::encode_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, (uint64_t)K / 2, (uint64_t)N,
                                        (uint64_t)K / 2, kWRow, kTileN, CU_TENSOR_MAP_SWIZZLE_64B) &&
                  vqlin::encode_tmap_2d(&tmXq, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, (uint64_t)K, (uint64_t)M,
                                        (uint64_t)K, kBRow, (uint32_t)p.bt, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return vqlin::fail(VQLIN_ERR_CUDA, "w4a4 low-latency: tensor map encoding failed (M=%d N=%d K=%d)", M, N, K);

  LowlatArgs a;
  a.X = X; a.chan = chan; a.static_scale = static_scale; a.sx = sx; a.sx_step = sx_step; a.sw = sw; a.bias = bias;
  a.Y = Y;
  a.xq = xq_ws;
  a.status = status; a.M = M; a.N = N; a.K = K; a.bt = p.bt; a.nkb = K / 128; a.cn = p.cn;
  a.tmem_cols = p.cols; a.rows_per = p.rows_per; a.issuers = p.issuers; a.wait_limit_ns = kWaitLimitNs;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.tiles_n_pad, p.tiles_m, p.S);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = p.dyn;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.cn;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = p.S;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = vqlin::pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = vqlin::launched(cudaLaunchKernelEx(&cfg, w4a4_lowlat_kernel<FUSED, HB, CHAN>, tmW, tmXq, a));
  if (e != cudaSuccess)
    return vqlin::fail(VQLIN_ERR_CUDA, "w4a4 low-latency launch (grid %d x %d x %d, cluster %d x %d, %zu B): %s",
                       p.tiles_n_pad, p.tiles_m, p.S, p.cn, p.S, p.dyn, cudaGetErrorString(e));
  return VQLIN_OK;
}

}  // namespace

namespace vqlin {

vqlin_status launch_w4a4_static_lowlat(const uint16_t* X, const float* static_scale, int hb, uint8_t* xq_ws,
                                       const uint8_t* wq, const float* sw, const uint16_t* bias, uint16_t* Y, int M,
                                       int N, int K, int* status, cudaStream_t st, const float* chan) {
  if (M == 0 || N == 0) return VQLIN_OK;
  if (chan != nullptr) {
    if (hb == 64)
      return launch_lowlat<true, 64, true>(X, static_scale, nullptr, nullptr, xq_ws, wq, sw, bias, Y, M, N, K, status,
                                           st, 1, chan);
    return launch_lowlat<true, 128, true>(X, static_scale, nullptr, nullptr, xq_ws, wq, sw, bias, Y, M, N, K, status,
                                          st, 1, chan);
  }
  if (hb == 64)
    return launch_lowlat<true, 64>(X, static_scale, nullptr, nullptr, xq_ws, wq, sw, bias, Y, M, N, K, status, st);
  return launch_lowlat<true, 128>(X, static_scale, nullptr, nullptr, xq_ws, wq, sw, bias, Y, M, N, K, status, st);
}

// Whether the few-token kernel's plan runs as one wave of clusters: the kernel
// stages a CTA's whole K range of weights on chip before it waits for the
// previous launch, which pays off only when every CTA is resident at once
// (beyond that, its fixed per-CTA cost repeats every wave and the throughput
// GEMM streams the weights faster).
bool lowlat_one_wave(bool fused, int hb, int M, int N, int K) {
  LowlatPlan p;
  bool ok;
  int active = 0;
  cudaError_t ae = cudaSuccess;
  if (fused && hb == 64) {
    set_attrs_once<true, 64>(&ae);
    ok = ae == cudaSuccess && make_plan<true, 64>(M, N, K, p);
    if (ok) active = max_active_clusters((const void*)w4a4_lowlat_kernel<true, 64>, kThreads, p.dyn, p.cn * p.S);
  } else if (fused) {
    set_attrs_once<true, 128>(&ae);
    ok = ae == cudaSuccess && make_plan<true, 128>(M, N, K, p);
    if (ok) active = max_active_clusters((const void*)w4a4_lowlat_kernel<true, 128>, kThreads, p.dyn, p.cn * p.S);
  } else {
    set_attrs_once<false, 128>(&ae);
    ok = ae == cudaSuccess && make_plan<false, 128>(M, N, K, p);
    if (ok) active = max_active_clusters((const void*)w4a4_lowlat_kernel<false, 128>, kThreads, p.dyn, p.cn * p.S);
  }
  if (!ok) return false;
  const long long clusters = (long long)(p.tiles_n_pad / p.cn) * p.tiles_m;
  return clusters <= active;
}

vqlin_status launch_w4a4_codes_lowlat(const uint8_t* xq, const float* sx, const uint8_t* wq, const float* sw,
                                      const uint16_t* bias, uint16_t* Y, int M, int N, int K, int* status,
                                      cudaStream_t st, int sx_step) {
  if (M == 0 || N == 0) return VQLIN_OK;
  return launch_lowlat<false, 128>(nullptr, nullptr, xq, sx, nullptr, wq, sw, bias, Y, M, N, K, status, st,
                                   sx_step);
}

// Static-scale projection at long K: at 32 k-blocks or more the one-launch
// kernel's on-chip quantization and code exchange (spread over a split of 4
// or more) cost more than the activation kernel plus the codes variant
// (B300, 50 x 1024 x 4096: 8.8 us against 8.3 us); below, one launch wins.
bool static_two_launch(int K) { return K / 128 >= 32; }

}  // namespace vqlin

// ------------------------------------------- the projection that allocates nothing
//
// vqlin_linear_w4a4_static needs a caller-provided code buffer of M x K bytes,
// through which the CTAs of a cluster share the activation codes.  Some
// callers cannot provide one: code running while a CUDA graph is being
// captured (where a device allocation is refused), hosts that hand a plugin
// fixed buffers and forbid it any allocation of its own, and runtimes whose
// memory is managed by someone else.  For them this entry point keeps the
// exchange buffer in a fixed array of device memory that belongs to the
// library: every GPU that loads the library reserves it until the process
// exits, and every call on that GPU shares it.

namespace {

// Largest M x K (activation codes, one byte each) the array holds: 1 MiB, e.g.
// 64 tokens x 16384 channels or 256 tokens x 4096 channels.
constexpr size_t kNoAllocCodeBytes = size_t(1) << 20;

// The exchange buffer.  In host code this name is not a device address; the
// kernel gets the address that cudaGetSymbolAddress returns for the current
// device.
static __device__ __align__(256) uint8_t g_noalloc_codes[kNoAllocCodeBytes];

std::mutex g_noalloc_mu;
uint8_t* g_noalloc_ptr[64] = {};

// The device address of the array on the current device, looked up once per
// device (with that device current).
vqlin_status noalloc_codes_ptr(uint8_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return vqlin::fail(VQLIN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return vqlin::fail(VQLIN_ERR_CUDA, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_codes);
    if (e != cudaSuccess)
      return vqlin::fail(VQLIN_ERR_CUDA, "cudaGetSymbolAddress(code array): %s", cudaGetErrorString(e));
    g_noalloc_ptr[dev] = static_cast<uint8_t*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return VQLIN_OK;
}

}  // namespace

extern "C" vqlin_status vqlin_linear_w4a4_static_noalloc(const uint16_t* X, const float* static_scale,
                                                         int hadamard_block, const uint8_t* wq, const float* sw,
                                                         const uint16_t* bias, uint16_t* Y, int M, int N, int K,
                                                         void* stream) {
  if (M < 0 || N < 0 || K <= 0) return vqlin::fail(VQLIN_ERR_INVALID_ARG, "bad sizes M=%d N=%d K=%d", M, N, K);
  if (hadamard_block != 64 && hadamard_block != 128)
    return vqlin::fail(VQLIN_ERR_INVALID_ARG, "hadamard_block must be 64 or 128 (got %d)", hadamard_block);
  if (K % 128 != 0 || K > vqlin::kGemmW4MaxK)
    return vqlin::fail(VQLIN_ERR_UNSUPPORTED_SHAPE, "K=%d must be a multiple of 128 and at most %d", K,
                       vqlin::kGemmW4MaxK);
  if ((size_t)M * (size_t)K > kNoAllocCodeBytes)
    return vqlin::fail(VQLIN_ERR_UNSUPPORTED_SHAPE,
                       "M x K = %d x %d activation codes exceed the library's fixed %zu-byte code array "
                       "(use vqlin_linear_w4a4_static with a buffer of your own)",
                       M, K, kNoAllocCodeBytes);
  if (M == 0 || N == 0) return VQLIN_OK;
  if (X == nullptr || static_scale == nullptr || wq == nullptr || sw == nullptr || Y == nullptr)
    return vqlin::fail(VQLIN_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!vqlin::aligned16(X) || !vqlin::aligned16(wq) || !vqlin::aligned16(Y))
    return vqlin::fail(VQLIN_ERR_MISALIGNED, "X, wq and Y must be 16-byte aligned");
  int* status = vqlin::device_status_word();
  if (status == nullptr) return vqlin::fail(VQLIN_ERR_CUDA, "no device status word");
  uint8_t* codes = nullptr;
  const vqlin_status r = noalloc_codes_ptr(&codes);
  if (r != VQLIN_OK) return r;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the same dispatch as vqlin_linear_w4a4_static, the code buffer being the array
  if (K <= vqlin::kLowlatMaxK && M <= vqlin::kLowlatMaxM && vqlin::lowlat_one_wave(true, hadamard_block, M, N, K)) {
    if (!vqlin::static_two_launch(K))
      return vqlin::launch_w4a4_static_lowlat(X, static_scale, hadamard_block, codes, wq, sw, bias, Y, M, N, K,
                                              status, st);
    if (vqlin::lowlat_one_wave(false, 128, M, N, K)) {
      const cudaError_t e = vqlin::launch_act_quant(X, M, K, 4, hadamard_block, static_scale, codes, nullptr, st);
      if (e != cudaSuccess) return vqlin::fail(VQLIN_ERR_CUDA, "act_hadamard_quant: %s", cudaGetErrorString(e));
      return vqlin::launch_w4a4_codes_lowlat(codes, static_scale, wq, sw, bias, Y, M, N, K, status, st, 0);
    }
  }
  const cudaError_t e = vqlin::launch_act_quant(X, M, K, 4, hadamard_block, static_scale, codes, nullptr, st);
  if (e != cudaSuccess) return vqlin::fail(VQLIN_ERR_CUDA, "act_hadamard_quant: %s", cudaGetErrorString(e));
  return vqlin::launch_int_gemm_static_scale(codes, static_scale, wq, sw, bias, Y, M, N, K, status, st);
}
