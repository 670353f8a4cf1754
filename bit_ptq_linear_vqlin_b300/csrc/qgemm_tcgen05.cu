// Integer GEMM of the W4A4 / W8A8 projections on the tcgen05 tensor cores.
//
//   acc[m, n] = sum_k xq[m, k] * wq[n, k]        (exact int32)
//   Y[m, n]   = bf16(((float)acc * sx[m]) * sw[n] + bias[n])
//
// Method: "FoldQuantVLA" abstract (W4A4 projections executed natively in
// integers after per-token activation and per-channel weight quantization;
// attention-output and FFN-down projections kept at W8A8); W4A8 is the
// setting evaluated in the "QuantVLA: Scale-Calibrated Post-Training
// Quantization for Vision-Language-Action Models" summary (section 4).
//
// sm_103a has no integer tcgen05 MMA, so the integer codes ride in floating
// point operands whose products and sums are exact:
//   * int4 code c (|c| <= 7) is the e4m3 subnormal s<<7 | |c|, value c * 2^-9;
//     the MMA is kind::f8f6f4 and the float32 accumulator holds acc * 2^-18
//     exactly (|acc| <= 49 K < 2^24 for K < 342k);
//   * int8 code c (|c| <= 127) is the f16 subnormal s<<15 | |c|, value
//     c * 2^-24; the MMA is kind::f16 and the accumulator holds acc * 2^-48
//     exactly while |acc| <= 127^2 * 1024 < 2^24, so the MMAs accumulate
//     1024 channels at a time into one of two float32 buffers in tensor
//     memory, and four drain warps add each finished chunk, converted to
//     int32, into an int32 running sum there (exact for any K).
// Activation codes arrive already in that operand encoding (one byte per int4
// code, one 16-bit word per int8 code, written so by the activation kernel),
// so TMA copies them straight into the 128-byte-swizzled MMA layout.  Weight
// codes stay packed in HBM (4 or 8 bits) and are expanded on chip.
//
// Work decomposition (swap-AB: weights are the MMA's M side):
//   * one CTA computes 128 output channels x BT tokens (BT <= 256, a multiple
//     of 16) over a range of K; grid = (N/128, M/BT, S) with the S CTAs that
//     share an output tile forming one thread-block cluster (split K, S chosen
//     per shape by an estimate of its time);
//   * warp 0: TMA producer; a stage holds the activation operand tile and the
//     packed weight tile (64 bytes of each of the 128 rows, 64-byte swizzle);
//   * warps 2..9: expand the packed weights into the MMA's A operand directly
//     in tensor memory (thread = weight row, tcgen05.st), so the expanded
//     weights never pass through shared memory, whose bandwidth bounds the
//     kernel otherwise; the two groups of four warps take alternate k-blocks;
//   * warp 1: allocates tensor memory and issues the MMAs, 4 per k-block, A
//     from tensor memory, B from shared memory, accumulating 128 x BT float32
//     in tensor memory; the whole warp runs the issue loop and one elected lane
//     issues (a lone lane of a diverged warp issues too slowly);
//   * epilogue (warps 2..9): unsplit K stages the bf16 tile in shared memory
//     and writes it with one TMA store; split K writes the partial tile as
//     int32 slices over the idle stages and adds each slice into the cluster
//     rank that owns those channels with one bulk reduction (reduce-scatter in
//     shared memory), so split K needs no global scratch memory and its sum is
//     exact;
//   * variant W4 (W4A8): int4 weights (nibbles, 32 bytes per row and 64-channel
//     k-block) expanded to f16 operands against int8 activations; the sums
//     stay exact over 16384 channels (7 x 127 per product);
//   * variant FX (static-scale W4A4): the activations arrive as bf16 and warps
//     10..13 rotate and quantize each k-block's tile on chip into the B operand;
//     int8: warps 10..13 add each finished 1024-channel chunk into the int32
//     running sum (chunked plans) while the MMAs fill the other buffer.
// Every wait is bounded in time; a wait that runs out records
// VQLIN_ERR_TIMEOUT in the device status word and the CTA winds down.
#include <mutex>

#include "act_codes.cuh"
#include "common.cuh"
#include "tc_ptx.cuh"

namespace {

using namespace vqlin_dev;

constexpr int kTileN = 128;       // output channels per CTA (MMA M)
constexpr int kRawRow = 64;       // packed weight bytes of one row per k-block
constexpr int kBRow = 128;        // activation operand bytes of one row per k-block
constexpr int kACols = 32;        // tensor-memory columns of one A stage (128 bytes per row)
constexpr int kThreads = 320;     // 10 warps
constexpr int kThreadsFx = 448;   // 14 warps: + 4 activation-quantizer warps (static-scale W4A4)
                                  // or 4 chunk-drain warps (int8)
constexpr int kExpandWarps = 8;
constexpr int kQuantWarps = 4;
constexpr int kMaxSplit = 16;
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
  int stages;
  uint32_t tmem_cols;
  uint32_t a_col;        // first tensor-memory column of the A stages
  int chunk_kb;          // > 0: exact int32 chunking every chunk_kb k-blocks (int8)
  uint32_t d1_col;       // chunking: second float32 accumulator
  uint32_t r_col;        // chunking: int32 running sum
  uint64_t wait_limit_ns;
  int withhold_loads;    // test hook: the producer issues nothing (waits run out)
  int tma_store;         // unsplit K: stage the bf16 tile and store it with TMA
  int rows_per;          // split K: output channels each cluster rank owns
  const float* static_scale;  // on-chip activation quantization: the static scale (one float)
  int sx_step;           // 1: per-token scales sx[m]; 0: one scale sx[0] for every token
};

// Expands 8 packed bytes into 4 words of A operand in channel order.
//   int4: a word holds channels 0..7 (nibble s|mmm, even channel low); the
//   e4m3 bytes of the even channels are (w & 0x07070707) | ((w << 4) &
//   0x80808080), of the odd ones ((w >> 4) & 0x07070707) | (w & 0x80808080),
//   and two byte permutes interleave them back into channel order.
//   int8: byte s|mmmmmmm -> f16 s<<15 | mmmmmmm: prmt copies the byte and
//   replicates its sign bit into the high byte, a mask keeps bit 15 and 0..6.
template <int BITS>
__device__ __forceinline__ void expand8(uint32_t lo, uint32_t hi, uint32_t* o) {
  if (BITS == 4) {
    const uint32_t e0 = (lo & 0x07070707u) | ((lo << 4) & 0x80808080u);
    const uint32_t o0 = ((lo >> 4) & 0x07070707u) | (lo & 0x80808080u);
    const uint32_t e1 = (hi & 0x07070707u) | ((hi << 4) & 0x80808080u);
    const uint32_t o1 = ((hi >> 4) & 0x07070707u) | (hi & 0x80808080u);
    o[0] = __byte_perm(e0, o0, 0x5140);
    o[1] = __byte_perm(e0, o0, 0x7362);
    o[2] = __byte_perm(e1, o1, 0x5140);
    o[3] = __byte_perm(e1, o1, 0x7362);
  } else {
    o[0] = __byte_perm(lo, 0u, 0x9180) & 0x807F807Fu;
    o[1] = __byte_perm(lo, 0u, 0xB3A2) & 0x807F807Fu;
    o[2] = __byte_perm(hi, 0u, 0x9180) & 0x807F807Fu;
    o[3] = __byte_perm(hi, 0u, 0xB3A2) & 0x807F807Fu;
  }
}

// W4A8: one word of 8 packed int4 codes (nibble s|mmm, even channel in the low
// nibble of each byte) -> 4 words of f16 operand pairs s<<15 | mmm (the f16
// bits of c * 2^-24), channel order.
__device__ __forceinline__ void expand_nib_f16(uint32_t w, uint32_t* o) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t b = (w >> (8 * i)) & 0xFFu;
    const uint32_t t = (b & 0x0Fu) | ((b & 0xF0u) << 12);  // even channel bits 0..3, odd 16..19
    o[i] = (t & 0x00070007u) | ((t & 0x00080008u) << 12);
  }
}

__device__ __forceinline__ void record_timeout(int* status, volatile int* abort) {
  *abort = 1;
  atomicCAS(status, 0, (int)VQLIN_ERR_TIMEOUT);
}

// FX: the activations arrive as bf16 and warps 10..13 quantize them on chip
// (block Hadamard of HB channels, static scale) into the B operand.
// W4 (with BITS = 8): W4A8, int4 weights (packed nibbles, 32 bytes per row and
// k-block) against int8 activations, on the f16 MMAs.
template <int BITS, bool FX, int HB, bool W4>
__global__ void __launch_bounds__((FX || BITS == 8) ? kThreadsFx : kThreads, 1)
qgemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
             const __grid_constant__ CUtensorMap tmY, const QgemmArgs a) {
  extern __shared__ uint8_t smem_dyn[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ __align__(16) float s_sx[256];
  __shared__ float s_sw[kTileN], s_bias[kTileN];

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  const int bt = a.bt;
  const uint32_t b_bytes = (uint32_t)bt * kBRow;                  // a multiple of 2048
  constexpr int RAW = (BITS == 8 && W4) ? 32 : kRawRow;           // packed weight bytes per row and k-block
  const uint32_t xraw_off = b_bytes + kTileN * RAW;               // FX: bf16 activation tile
  // [B operand | packed A | (FX) bf16 activations, two 64-channel halves]
  const uint32_t stage_bytes = xraw_off + (FX ? (uint32_t)bt * 256u : 0u);
  constexpr int NT = (FX || BITS == 8) ? kThreadsFx : kThreads;
  const int NS = a.stages;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + (size_t)NS * stage_bytes);
  uint64_t* full = bars;               // TMA -> expanders (both tiles landed)
  uint64_t* aready = bars + NS;        // expanders -> MMA (A stage in tensor memory)
  uint64_t* empty = bars + 2 * NS;     // MMA -> TMA (stage consumed)
  uint64_t* bready = bars + 3 * NS;    // FX: quantizer -> MMA (B operand written)
  uint64_t* acc_full = bars + 4 * NS;
  uint64_t* scl_ready = acc_full + 1;
  uint64_t* accf = acc_full + 2;       // [2] chunking: MMA -> drain (chunk accumulated)
  uint64_t* acce = acc_full + 4;       // [2] chunking: drain -> MMA (accumulator free)
  uint64_t* red_full = acc_full + 6;   // split K: the peers' partial slices added in

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
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&aready[i], kExpandWarps / 2);  // one group of four warps per k-block
      mbar_init(&empty[i], 1);
      mbar_init(&bready[i], kQuantWarps);
    }
    mbar_init(acc_full, 1);
    mbar_init(scl_ready, 31);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&accf[i], 1);
      mbar_init(&acce[i], 4);  // the four chunk-drain warps
    }
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

  if (warp == 0) {
    // lanes 1..31 stage the epilogue's per-token and per-channel scales and the
    // bias (float) while lane 0 produces; the epilogue waits on scl_ready
    if (lane > 0) {
      if (a.acc == nullptr) {
        // every load of a lane is issued before any is used (one latency)
        float wv[5], bv[5], xv[9];
#pragma unroll
        for (int j = 0; j < 5; ++j) {
          const int i = lane - 1 + 31 * j;
          const bool in = i < kTileN && n0 + i < a.N;
          wv[j] = in ? __ldg(a.sw + n0 + i) : 0.0f;
          bv[j] = in && a.bias != nullptr ? __uint_as_float((uint32_t)__ldg(a.bias + n0 + i) << 16) : 0.0f;
        }
        pdl_wait();  // the per-token scales come from the previous kernel
        const float xs = FX ? __ldg(a.static_scale) : 0.0f;  // one scale for every token
#pragma unroll
        for (int j = 0; j < 9; ++j) {
          const int i = lane - 1 + 31 * j;
          xv[j] = i < bt && m0 + i < a.M ? (FX ? xs : __ldg(a.sx + (size_t)(m0 + i) * a.sx_step)) : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < 5; ++j) {
          const int i = lane - 1 + 31 * j;
          if (i < kTileN) {
            s_sw[i] = wv[j];
            s_bias[i] = bv[j];
          }
        }
        // token scales in the unit of the epilogue's accumulator value: float32
        // sums of int4 (int8) products are integers x 2^-18 (2^-48), scaled here
        // by 2^18 (2^48) once instead of per element; chunked int8 sums and all
        // split-K sums reach the epilogue as int32
        const float su = (S == 1 && (BITS == 4 || a.chunk_kb == 0)) ? (BITS == 4 ? 262144.0f : 281474976710656.0f)
                                                                      : 1.0f;
#pragma unroll
        for (int j = 0; j < 9; ++j) {
          const int i = lane - 1 + 31 * j;
          if (i < bt) s_sx[i] = xv[j] * su;
        }
      }
      mbar_arrive(scl_ready);
    }
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      constexpr int kXStep = BITS == 4 ? kBRow : kBRow / 2;  // activation elements per k-block
      // bytes one stage receives by TMA: packed weights and the activation
      // tile (operand codes, or bf16 when quantized on chip)
      const uint32_t tma_bytes = kTileN * RAW + (FX ? (uint32_t)bt * 256u : b_bytes);
      auto load_x = [&](uint8_t* st, int kb, uint64_t* bar) {
        if (FX) {
          tma_load_2d(st + xraw_off, &tmX, kb * 128, m0, bar);
          tma_load_2d(st + xraw_off + (uint32_t)bt * 128u, &tmX, kb * 128 + 64, m0, bar);
        } else {
          tma_load_2d(st, &tmX, kb * kXStep, m0, bar);
        }
      };
      int issued = 0;
      if (!a.withhold_loads) {
        // the weight tiles of the first stages do not depend on the previous
        // kernel: load them before waiting for it
        const int pre = cnt < NS ? cnt : NS;
        for (int i = 0; i < pre; ++i) {
          mbar_arrive_expect_tx(&full[i], tma_bytes);
          tma_load_2d(base + (size_t)i * stage_bytes + b_bytes, &tmW, (kb0 + i) * RAW, n0, &full[i]);
        }
        pdl_wait();
        // the next kernel may prepare once this one works; an earlier trigger
        // lets a chain of launches prefetch weights all at once
        pdl_trigger();
        for (int i = 0; i < pre; ++i) {
          load_x(base + (size_t)i * stage_bytes, kb0 + i, &full[i]);
          ++issued;
        }
        int s = 0;        // stage of k-block i
        uint32_t ph = 0;  // parity of the release of stage s that k-block i waits for
        for (int i = pre; i < cnt; ++i) {
          if (!mbar_wait_bounded(&empty[s], ph, a.wait_limit_ns, abort)) {
            if (!*abort) record_timeout(a.status, abort);
            break;
          }
          uint8_t* st = base + (size_t)s * stage_bytes;
          mbar_arrive_expect_tx(&full[s], tma_bytes);
          tma_load_2d(st + b_bytes, &tmW, (kb0 + i) * RAW, n0, &full[s]);
          load_x(st, kb0 + i, &full[s]);
          ++issued;
          if (++s == NS) {
            s = 0;
            ph ^= 1u;
          }
        }
      } else {
        pdl_wait();
        pdl_trigger();
      }
      // copies still in flight complete before the CTA may exit
      for (int i = issued > NS ? issued - NS : 0; i < issued; ++i)
        if (!mbar_wait_bounded(&full[i % NS], (i / NS) & 1, a.wait_limit_ns, nullptr))
          record_timeout(a.status, abort);
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    // the whole warp runs the loop (warp-uniform control flow, every wait
    // decided by a vote) and one elected lane issues each MMA and commit: a
    // single lane looping in a diverged warp issues MMAs too slowly to keep
    // the tensor core busy
    {
      const uint32_t id = idesc_f32acc(0u, kTileN, bt);  // e4m3 x e4m3 or f16 x f16 -> f32
      const int ck = BITS == 8 ? a.chunk_kb : 0;  // int4 sums never need chunking
      const uint64_t db0 = sdesc_sw128(base);
      const uint64_t dstep = (uint64_t)(stage_bytes >> 4);  // start-address field step per stage
      const uint32_t ta0 = tmem + a.a_col;
      int s = 0, kin = 0, c = 0;  // stage; k-block inside the chunk; chunk
      uint32_t ph = 0;            // phase parity of stage s
      for (int i = 0; i < cnt; ++i) {
        // chunking: chunk c accumulates into float32 buffer c & 1, which the
        // expanders drain into the int32 running sum before chunk c + 2 reuses it
        const uint32_t dacc = tmem + ((c & 1) ? a.d1_col : 0u);
        if (ck && kin == 0 && c >= 2) {
          const bool ok = mbar_wait_bounded(&acce[c & 1], ((c >> 1) - 1) & 1, a.wait_limit_ns, abort);
          if (!__all_sync(0xffffffffu, ok)) {
            if (!ok && !*abort) record_timeout(a.status, abort);
            break;
          }
        }
        const bool ok = mbar_wait_bounded(&aready[s], ph, a.wait_limit_ns, abort) &&
                        (!FX || mbar_wait_bounded(&bready[s], ph, a.wait_limit_ns, abort));
        if (!__all_sync(0xffffffffu, ok)) {
          if (!ok && !*abort) record_timeout(a.status, abort);
          break;
        }
        tc_fence_after();
        const uint64_t db = db0 + (uint64_t)s * dstep;
        const uint32_t ta = ta0 + (uint32_t)(s * kACols);
        // per MMA: 8 tensor-memory columns of A, 32 bytes along the swizzled B row
        if (BITS == 4) {
          mma_f8f6f4_ta_warp(dacc, ta, db, id, kin != 0 ? 1u : 0u);
          mma_f8f6f4_ta_warp(dacc, ta + 8, db + 2, id, 1u);
          mma_f8f6f4_ta_warp(dacc, ta + 16, db + 4, id, 1u);
          mma_f8f6f4_ta_warp(dacc, ta + 24, db + 6, id, 1u);
        } else {
          mma_f16_ta_warp(dacc, ta, db, id, kin != 0 ? 1u : 0u);
          mma_f16_ta_warp(dacc, ta + 8, db + 2, id, 1u);
          mma_f16_ta_warp(dacc, ta + 16, db + 4, id, 1u);
          mma_f16_ta_warp(dacc, ta + 24, db + 6, id, 1u);
        }
        tc_commit_warp(&empty[s]);
        ++kin;
        if (ck && (kin == ck || i == cnt - 1)) {
          tc_commit_warp(&accf[c & 1]);
          kin = 0;
          ++c;
        }
        if (++s == NS) {
          s = 0;
          ph ^= 1u;
        }
      }
      tc_commit_warp(acc_full);
    }
  } else if (warp < 2 + kExpandWarps) {
    // ------------------------------------------------- weight expanders (2..9)
    // thread = weight row (its warp's tensor-memory lane quadrant); the two
    // groups of four warps take alternate k-blocks, so one group's tensor
    // memory stores are in flight while the other group expands
    const int q = warp & 3, g = (warp - 2) >> 2;
    const int row = q * 32 + lane;
    // swizzle of the packed tile: 64-byte rows (int4 / int8 weights), or 32-byte
    // rows (W4A8: 64 channels of nibbles)
    const int sw = RAW == 64 ? (row >> 1) & 3 : (row >> 2) & 1;
    const uint32_t lanes = tmem + ((uint32_t)(q * 32) << 16);
    const uint32_t trow = lanes + a.a_col;
    int s = g;         // stage of k-block i (NS >= 2)
    uint32_t ph = 0;   // phase parity of stage s
    for (int i = g; i < cnt; i += 2) {
      const bool ok = mbar_wait_bounded(&full[s], ph, a.wait_limit_ns, abort);
      if (!__all_sync(0xffffffffu, ok)) {
        if (!ok && !*abort) record_timeout(a.status, abort);
        break;
      }
      const uint8_t* rawrow = base + (size_t)s * stage_bytes + b_bytes + row * RAW;
      uint32_t v[2][16];
      if (RAW == 32) {
        // W4A8: 16 bytes = 32 channels -> 16 f16 pair words per half
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const uint4 r = *reinterpret_cast<const uint4*>(rawrow + ((j ^ sw) << 4));
          expand_nib_f16(r.x, &v[j][0]);
          expand_nib_f16(r.y, &v[j][4]);
          expand_nib_f16(r.z, &v[j][8]);
          expand_nib_f16(r.w, &v[j][12]);
        }
      } else {
        uint4 rw[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) rw[j] = *reinterpret_cast<const uint4*>(rawrow + ((j ^ sw) << 4));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          expand8<BITS>(rw[j].x, rw[j].y, &v[j >> 1][8 * (j & 1)]);
          expand8<BITS>(rw[j].z, rw[j].w, &v[j >> 1][8 * (j & 1) + 4]);
        }
      }
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
    }
  } else if (BITS == 8) {
    // --------------------------------------------- int8 chunk drains (10..13)
    // Chunking: adds float32 chunk c (exact integers x 2^-48, each below 2^24)
    // into the int32 running sum in tensor memory, while the MMAs fill the
    // other float32 buffer; warp = lane quadrant, all bt columns.
    const int ck = a.chunk_kb;
    const int nch = ck > 0 ? (cnt + ck - 1) / ck : 0;
    const uint32_t lanes = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const float unit = 281474976710656.0f;  // 2^48: f16-operand accumulator -> integer
    for (int c = 0; c < nch; ++c) {
      const bool ok = mbar_wait_bounded(&accf[c & 1], (c >> 1) & 1, a.wait_limit_ns, abort);
      if (!__all_sync(0xffffffffu, ok)) {
        if (!ok && !*abort) record_timeout(a.status, abort);
        break;
      }
      tc_fence_after();
      const uint32_t src = lanes + ((c & 1) ? a.d1_col : 0u);
      for (int cb = 0; cb < bt; cb += 32) {
        const bool two = cb + 16 < bt;  // warp-uniform
        uint32_t v[2][16], r[2][16];
        tmem_ld_x16(src + (uint32_t)cb, v[0]);
        if (two) tmem_ld_x16(src + (uint32_t)(cb + 16), v[1]);
        if (c > 0) {
          tmem_ld_x16(lanes + a.r_col + (uint32_t)cb, r[0]);
          if (two) tmem_ld_x16(lanes + a.r_col + (uint32_t)(cb + 16), r[1]);
        }
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          if (u == 1 && !two) break;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            r[u][j] = (uint32_t)((c > 0 ? (int32_t)r[u][j] : 0) + __float2int_rn(__uint_as_float(v[u][j]) * unit));
          tmem_st_x16(lanes + a.r_col + (uint32_t)(cb + 16 * u), r[u]);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[c & 1]);
    }
  } else if (FX) {
    // --------------------------------------- activation quantizers (10..13)
    // The bf16 activation tile of each k-block (two 64-channel halves,
    // 128-byte swizzle) becomes the B operand: block Hadamard over HB
    // channels, then codes at the static scale, exactly as the standalone
    // activation kernel computes them.  Four lanes hold one token's 128
    // channels (32 each, the Hadamard unit layout); a warp takes 8 tokens per
    // pass, the four warps 32.
    constexpr int LPG = HB / 32;
    const int qw = warp - (2 + kExpandWarps);
    const int rl = lane >> 2, l4 = lane & 3;
    const int g = l4 / LPG, l = l4 % LPG;  // Hadamard block inside the k-block; lane inside the block
    pdl_wait();  // the static scale may come from the previous kernel
    const float xs = __ldg(a.static_scale);
    const float inv_s = xs > 0.0f ? __frcp_rn(xs) : 0.0f;
    int s = 0;
    uint32_t ph = 0;
    for (int i = 0; i < cnt; ++i) {
      const bool ok = mbar_wait_bounded(&full[s], ph, a.wait_limit_ns, abort);
      if (!__all_sync(0xffffffffu, ok)) {
        if (!ok && !*abort) record_timeout(a.status, abort);
        break;
      }
      const uint8_t* xr = base + (size_t)s * stage_bytes + xraw_off;
      uint8_t* bq = base + (size_t)s * stage_bytes;
      for (int r0 = qw * 8; r0 < bt; r0 += 8 * kQuantWarps) {  // warp-uniform
        const int r = r0 + rl, sw7 = r & 7;
        float v[4][8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int ch = HB * g + 8 * (l + LPG * j);  // first channel of chunk j
          const uint4 raw = *reinterpret_cast<const uint4*>(xr + (size_t)(ch >> 6) * bt * 128 + r * 128 +
                                                            ((((ch & 63) >> 3) ^ sw7) << 4));
          v[j][0] = bf16_lo(raw.x); v[j][1] = bf16_hi(raw.x);
          v[j][2] = bf16_lo(raw.y); v[j][3] = bf16_hi(raw.y);
          v[j][4] = bf16_lo(raw.z); v[j][5] = bf16_hi(raw.z);
          v[j][6] = bf16_lo(raw.w); v[j][7] = bf16_hi(raw.w);
        }
        hadamard_unit<HB>(v, lane);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t w[4];
          quantize_chunk<4>(v[j], xs, inv_s, w);
          const int ch = HB * g + 8 * (l + LPG * j);
          *reinterpret_cast<uint2*>(bq + r * 128 + ((((ch >> 4) ^ sw7)) << 4) + (ch & 8)) = make_uint2(w[0], w[1]);
        }
      }
      fence_proxy_async_smem();  // the MMA reads these bytes through the async proxy
      __syncwarp();
      if (lane == 0) mbar_arrive(&bready[s]);
      if (++s == NS) {
        s = 0;
        ph ^= 1u;
      }
    }
  }

  // ---------------------------------------------------------------- epilogue
  __syncwarp();  // the single-thread roles rejoin their warps
  const bool chunked = BITS == 8 && a.chunk_kb > 0;
  const float unit = BITS == 4 ? 262144.0f : 281474976710656.0f;  // 2^18, 2^48: accumulator -> integer
  const bool raw_out = a.acc != nullptr;
  const bool epi = warp >= 2 && warp < 2 + kExpandWarps;  // the epilogue's warps
  bool go = false;
  if (epi) {
    // chunked int8: the running sum is complete once the last chunk is drained
    const int nch = chunked ? (cnt + a.chunk_kb - 1) / a.chunk_kb : 0;
    const bool ok = mbar_wait_bounded(acc_full, 0, a.wait_limit_ns, nullptr) &&
                    mbar_wait_bounded(scl_ready, 0, a.wait_limit_ns, nullptr) &&
                    (nch == 0 || mbar_wait_bounded(&acce[(nch - 1) & 1], ((nch - 1) >> 1) & 1, a.wait_limit_ns, nullptr));
    if (!ok) record_timeout(a.status, abort);
    tc_fence_after();
    // warp-uniform decision: the tensor-memory loads below are warp-collective
    go = __all_sync(0xffffffffu, ok && !*abort);
  }
  pdl_wait();  // global writes only once the previous kernel has finished
  // warps 2..9: lane quadrant q of tensor memory, 16-column chunks 16h + 32k
  const int q = warp & 3;
  const int h = (warp - 2) >> 2;
  const int row = q * 32 + lane;  // output channel inside the tile
  const uint32_t lanes_q = tmem + ((uint32_t)(q * 32) << 16);
  // accumulator words of this thread's row in columns cb + 32u .. + 15, for
  // the u < 4 with cb + 32u < bt: four tensor-memory loads, one wait
  auto load4 = [&](int cb, uint32_t (&v)[4][16]) {
    const uint32_t src = lanes_q + (chunked ? a.r_col : 0u) + (uint32_t)cb;
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (cb + 32 * u < bt) tmem_ld_x16(src + (uint32_t)(32 * u), v[u]);  // warp-uniform
    tmem_ld_wait();
  };
  // the exact integer sum held by an accumulator word
  auto as_int = [&](uint32_t w) -> int32_t {
    return chunked ? (int32_t)w : __float2int_rn(__uint_as_float(w) * unit);
  };
  // the same sum as a float in the unit of s_sx (see the staging above)
  auto as_f = [&](uint32_t w) -> float { return chunked ? (float)(int32_t)w : __uint_as_float(w); };

  if (S == 1 && a.tma_store) {
    // bf16 tile [bt tokens][128 channels] staged over the idle stages, then one
    // TMA store (the tensor map clips the M and N tails)
    uint16_t* ystage = reinterpret_cast<uint16_t*>(base);
    if (epi) {
      if (go) {
        const float sw_n = s_sw[row], b_n = s_bias[row];
        for (int cb = 16 * h; cb < bt; cb += 128) {
          uint32_t v[4][16];
          load4(cb, v);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int c0 = cb + 32 * u;
            if (c0 >= bt) break;
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
              const float4 sx4 = *reinterpret_cast<const float4*>(&s_sx[c0 + j]);  // 4 token scales
              // two tokens of this channel per paired conversion to bf16
              const uint32_t p0 = pack_bf16x2_rn(fmaf(as_f(v[u][j]) * sx4.x, sw_n, b_n),
                                                 fmaf(as_f(v[u][j + 1]) * sx4.y, sw_n, b_n));
              const uint32_t p1 = pack_bf16x2_rn(fmaf(as_f(v[u][j + 2]) * sx4.z, sw_n, b_n),
                                                 fmaf(as_f(v[u][j + 3]) * sx4.w, sw_n, b_n));
              ystage[(c0 + j) * kTileN + row] = (uint16_t)p0;
              ystage[(c0 + j + 1) * kTileN + row] = (uint16_t)(p0 >> 16);
              ystage[(c0 + j + 2) * kTileN + row] = (uint16_t)p1;
              ystage[(c0 + j + 3) * kTileN + row] = (uint16_t)(p1 >> 16);
            }
          }
        }
        fence_proxy_async_smem();
      }
      named_barrier(1, kExpandWarps * 32);
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
    if (epi && go) {
      const int n = n0 + row;
      const float sw_n = s_sw[row], b_n = s_bias[row];
      for (int cb = 16 * h; cb < bt; cb += 128) {
        uint32_t v[4][16];
        load4(cb, v);
        if (n >= a.N) continue;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c0 = cb + 32 * u;
          if (c0 >= bt) break;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int m = m0 + c0 + j;
            if (m < a.M) {
              if (raw_out)
                a.acc[(size_t)m * a.N + n] = as_int(v[u][j]);
              else
                a.Y[(size_t)m * a.N + n] = f32_to_bf16_rn(fmaf(as_f(v[u][j]) * s_sx[c0 + j], sw_n, b_n));
            }
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();
  } else {
    // split K, reduce-scatter over the cluster: cluster rank r owns output
    // channels [r rp, (r + 1) rp).  Every CTA writes its 32-bit partial tile as
    // S slices part[r][token][rp] (over the idle stages; int4 and int8 sums as
    // int32), then adds slice r into rank r's slice with one bulk reduction
    // each; rank r scales and stores its slice once all S - 1 have landed.
    const int rp = a.rows_per;
    const uint32_t slice_words = (uint32_t)(bt * rp);
    const uint32_t slice_bytes = slice_words * 4u;
    const int own0 = (int)rank * rp;                                     // first owned channel
    const int own_n = own0 < kTileN ? min(rp, kTileN - own0) : 0;        // channels owned here
    uint32_t* part = reinterpret_cast<uint32_t*>(base);
    if (tid == 64 && own_n > 0) mbar_arrive_expect_tx(red_full, (uint32_t)(S - 1) * slice_bytes);
    if (epi && go) {
      const int sl = row / rp, k = row - sl * rp;
      uint32_t* dst = part + (size_t)sl * slice_words + k;
      for (int cb = 16 * h; cb < bt; cb += 128) {
        uint32_t v[4][16];
        load4(cb, v);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c0 = cb + 32 * u;
          if (c0 >= bt) break;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            uint32_t w;
            if (BITS == 4) {
              // |sum| < 2^22: the integer sits in the low mantissa bits of
              // sum + 1.5 x 2^23 (exact), no conversion instruction needed
              w = (uint32_t)(__float_as_int(fmaf(__uint_as_float(v[u][j]), unit, 12582912.0f)) - 0x4B400000);
            } else {
              w = (uint32_t)as_int(v[u][j]);
            }
            dst[(size_t)(c0 + j) * rp] = w;
          }
        }
      }
      fence_proxy_async_smem();  // the bulk reductions read and write these words
    }
    tc_fence_before();
    __syncwarp();
    cluster_sync_all();  // every CTA's partial slices are in place
    // the slices are sent even after an abort (their contents are then
    // meaningless), so every bulk reduction completes before any CTA exits
    const uint32_t part_s = smem_addr(part);
    if (tid >= 64 && tid < 64 + S) {
      const int r = tid - 64;
      if (r != (int)rank && r * rp < kTileN) {
        const uint32_t off = (uint32_t)r * slice_bytes;
        bulk_reduce_add_u32_to_peer(mapa_shared(part_s + off, (uint32_t)r), part_s + off, slice_bytes,
                                    mapa_shared(smem_addr(red_full), (uint32_t)r));
      }
    }
    bool got = true;
    if (own_n > 0) {
      got = mbar_wait_bounded(red_full, 0, a.wait_limit_ns, nullptr);
      if (!got) record_timeout(a.status, abort);
    }
    got = got && own_n > 0 && !*abort;
    // this CTA has all it receives: once every rank has arrived here, no
    // bulk reduction reads or writes any of the cluster's shared memory
    __syncwarp();
    cluster_arrive();
    if (got) {
      const int nq = own_n / 4;  // 4-channel groups owned here
      const int total = nq * bt;
      const bool vec = (a.N & 3) == 0;
      const uint32_t* mine = part + (size_t)rank * slice_words;
      for (int idx = tid; idx < total; idx += NT) {
        const int c = idx / nq, k = 4 * (idx - (idx / nq) * nq);
        const int m = m0 + c, rr = own0 + k, n = n0 + rr;
        if (m >= a.M || n >= a.N) continue;
        const uint4 t = *reinterpret_cast<const uint4*>(mine + (size_t)c * rp + k);
        const int32_t acc[4] = {(int32_t)t.x, (int32_t)t.y, (int32_t)t.z, (int32_t)t.w};
        if (raw_out) {
          int32_t* o = a.acc + (size_t)m * a.N + n;
          if (vec) {
            *reinterpret_cast<int4*>(o) = make_int4(acc[0], acc[1], acc[2], acc[3]);
          } else {
            for (int e = 0; e < 4 && n + e < a.N; ++e) o[e] = acc[e];
          }
        } else {
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
    }
    __syncwarp();
    cluster_wait();
  }
  if (warp == 1) tmem_dealloc(tmem, a.tmem_cols);
}

// ------------------------------------------------------------------ host side

// 227 KB opt-in per CTA, less room for the kernel's static shared memory
constexpr int kMaxSmem = 232448 - 4096;
constexpr size_t kSmemPerSm = 233472;  // shared memory of one SM

// one pipeline stage: B operand, packed weights (raw bytes per row) and (fx)
// the bf16 activation tile
size_t stage_bytes(int bt, bool fx, int raw) {
  return (size_t)bt * kBRow + (size_t)kTileN * raw + (fx ? (size_t)bt * 256 : 0);
}

size_t smem_bytes(int bt, int stages, bool fx, int raw) {
  return 1024 + stages * stage_bytes(bt, fx, raw) + (4 * stages + 7) * 8;
}

// FX: bf16 activations quantized on chip at a static scale (xq is the bf16
// activation matrix, sx the device pointer to the scale, HB the Hadamard block)
template <int BITS, bool FX = false, int HB = 128, bool W4 = false>
vqlin_status launch_bits(const void* xq, const float* sx, const void* wq, const float* sw, const uint16_t* bias,
                         uint16_t* Y, int32_t* acc, int M, int N, int K, int* status, int withhold,
                         uint64_t limit_ns, cudaStream_t st, int sx_step = 1) {
  constexpr int NT = (FX || BITS == 8) ? kThreadsFx : kThreads;
  const auto kern = qgemm_kernel<BITS, FX, HB, W4>;
  constexpr int RAW = (BITS == 8 && W4) ? 32 : kRawRow;
  // function attributes are per device: set them once for every device used
  static std::mutex attr_mu;
  static bool attr_set[64] = {};
  static cudaError_t attr_res[64] = {};
  cudaError_t attr_err = cudaSuccess;
  {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return vqlin::fail(VQLIN_ERR_CUDA, "qgemm: no device");
    std::lock_guard<std::mutex> lock(attr_mu);
    if (!attr_set[dev]) {
      attr_res[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
      if (attr_res[dev] == cudaSuccess)
        attr_res[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      attr_set[dev] = true;
    }
    attr_err = attr_res[dev];
  }
  if (attr_err != cudaSuccess)
    return vqlin::fail(VQLIN_ERR_CUDA, "qgemm: cudaFuncSetAttribute: %s", cudaGetErrorString(attr_err));

  const int kb_codes = BITS == 4 ? 128 : 64;
  const int w_row_bytes = (BITS == 4 || W4) ? K / 2 : K;
  // f16-operand sums are exact while below 2^24: 1024 channels of int8 x int8
  // (127^2 per product), 16384 of int4 x int8 (7 x 127)
  const int exact_ch = W4 ? 16384 : 1024;
  const int nkb = K / kb_codes;

  // One launch plan: token tile, K split, stages, tensor-memory columns and
  // shared memory.  Returns false if no plan fits; `one_wave` tells whether
  // all clusters are resident at once.
  struct Plan {
    bool chunked = false;
    int bt = 0, tiles_n = 0, tiles_m = 0, S = 0, NS = 0, rows_per = 0;
    uint32_t a_col = 0, cols = 0;
    size_t dyn = 0;
    bool one_wave = false;
  };
  // chunked: int8 beyond 1024 channels keeps two float32 accumulators and an
  // int32 running sum in tensor memory (token tile <= 128); otherwise every
  // CTA sums at most s_min-th of K (int8: <= 1024 channels)
  auto make_plan = [&](bool chunked, int s_min, Plan& p, int bt_force) -> bool {
    const int bt_max = chunked ? 128 : 256;
    const int nt = (M + bt_max - 1) / bt_max;
    const int bt = bt_force > 0 ? bt_force : ((M + nt - 1) / nt + 15) / 16 * 16;
    const int tiles_n = (N + kTileN - 1) / kTileN;
    const int tiles_m = (M + bt - 1) / bt;
    int s_want = (148 + tiles_n * tiles_m - 1) / (tiles_n * tiles_m);
    s_want = s_want < s_min ? s_min : s_want;
    s_want = s_want > kMaxSplit ? kMaxSplit : s_want;
    s_want = s_want > nkb ? nkb : s_want;
    if (s_want < s_min) return false;
    // Among the splits whose clusters are all resident at once (one wave),
    // the one of least estimated time: k-blocks per CTA x about 0.25 + 0.0004
    // bt us each (on-chip activation quantization: about 1.5 us), plus about
    // 1.2 + 0.008 bt + 0.17 S us for the split-K
    // epilogue (measured on B300 for 16 <= bt <= 208; at 50 tokens and 8
    // k-blocks no split is fastest).  With no one-wave split, the smallest.
    auto est_us = [&](int s) {
      // on-chip activation quantization costs far more per k-block than the MMAs
      const double t_kb = FX ? 1.5 : 0.25 + 0.0004 * bt;
      return ((nkb + s - 1) / s) * t_kb + (s > 1 ? 1.2 + 0.008 * bt + 0.17 * s : 0.0);
    };
    bool found = false, found_wave = false;
    double best = 0.0;
    for (int s_try = s_min; s_try <= s_want; ++s_try) {
      Plan q;
      const int per_cta = (nkb + s_try - 1) / s_try;
      // stages: up to 6 within the shared-memory limit, no more than the
      // k-blocks a CTA runs, and enough that the 32-bit partial tile of the
      // split-K epilogue (s_try slices of [bt][rows_per]) fits over them
      const int rp = s_try > 1 ? ((kTileN + s_try - 1) / s_try + 3) & ~3 : kTileN;
      const size_t part_bytes = (size_t)s_try * rp * bt * 4;
      const size_t sb = stage_bytes(bt, FX, RAW);
      const int ns_min = (int)((part_bytes + sb - 1) / sb);
      // tensor memory: accumulator [0, bt) (chunking: two float32 accumulators
      // and the int32 running sum), then one 32-column A slot per stage
      const uint32_t bt_pad = (uint32_t)((bt + 31) / 32 * 32);
      const uint32_t ac = chunked ? 3 * bt_pad : bt_pad;
      const int ns_tmem = (int)((512 - ac) / kACols);
      int ns = per_cta > 6 ? 6 : per_cta;
      if (ns > ns_tmem) ns = ns_tmem;
      if (ns < ns_min) ns = ns_min;
      if (ns < 2) ns = 2;
      while (ns > ns_min && ns > 2 && smem_bytes(bt, ns, FX, RAW) > (size_t)kMaxSmem) --ns;
      // A stage is reused by the k-block NS later, and the two expander groups
      // take alternate k-blocks: with NS odd, a group would wait on a stage
      // whose previous use belongs to the other group, where an mbarrier parity
      // wait cannot tell a pending phase from the one before it
      if (per_cta > ns && (ns & 1)) ns += ns - 1 >= ns_min && ns - 1 >= 2 ? -1 : 1;
      uint32_t c = 32;
      while (c < ac + (uint32_t)(ns * kACols)) c <<= 1;
      if (c > 512 || smem_bytes(bt, ns, FX, RAW) > (size_t)kMaxSmem) continue;
      // never more CTAs on an SM than its 512 tensor-memory columns hold: a
      // CTA blocked in tcgen05.alloc while its cluster peers wait for it could
      // otherwise wait on CTAs of another cluster in the same state
      size_t d = smem_bytes(bt, ns, FX, RAW);
      const size_t dyn_floor = kSmemPerSm / (512 / c + 1) + 1;
      if (d < dyn_floor) d = dyn_floor;
      q.chunked = chunked; q.bt = bt; q.tiles_n = tiles_n; q.tiles_m = tiles_m;
      q.S = s_try; q.NS = ns; q.a_col = ac; q.cols = c; q.dyn = d;
      q.rows_per = rp;
      const int active = vqlin::max_active_clusters((const void*)kern, NT, d, s_try);
      q.one_wave = tiles_n * tiles_m <= active;
      if (!found) {
        p = q;  // the smallest allowed split
        found = true;
      }
      if (q.one_wave && (!found_wave || est_us(s_try) < best)) {
        p = q;
        best = est_us(s_try);
        found_wave = true;
      }
    }
    return found;
  };
  // Many tokens on fewer tiles than SMs: also try the token tile (>= 96)
  // that puts the most CTAs in one wave, and keep it if a k-block-paced
  // estimate (0.25 us per k-block at 6 stages or more, longer with fewer,
  // + 0.0004 bt; a split adds 1.2 + 0.03 bt + 0.17 S us) is 5% lower.
  // Timed on B300: W8A8 816 x 2048 x 16384 85.9 -> 70.6 us (96 tokens, 144
  // CTAs, 6 stages instead of 4); W4A4 816 x 2560 x 2048 9.9 -> 8.7 us (128
  // tokens, 140 CTAs); W4A4 512 x 4096 x 4096 17.5 -> 13.3 us (160 tokens,
  // unsplit instead of split 2); a long K keeps its split (W4A8 512 x 4096 x
  // 11008: 37 us split against 54 us at 160 tokens unsplit).
  auto pick = [&](bool chunked, int s_min, Plan& out) -> bool {
    if (!make_plan(chunked, s_min, out, 0)) return false;
    if (M < 256 || out.tiles_n * out.tiles_m >= 148) return true;
    const int bt_max = chunked ? 128 : 256;
    int bt_fill = out.bt, best_tiles = out.tiles_n * out.tiles_m;
    for (int c = bt_max; c >= 96; c -= 16) {
      const int t = out.tiles_n * ((M + c - 1) / c);
      if (t <= 148 && t > best_tiles) {
        best_tiles = t;
        bt_fill = c;
      }
    }
    Plan alt;
    if (bt_fill == out.bt || !make_plan(chunked, s_min, alt, bt_fill) || !alt.one_wave) return true;
    auto est = [&](const Plan& q) {
      const double t_kb = 0.25 * (q.NS >= 6 ? 1.0 : 6.0 / q.NS) + 0.0004 * q.bt;
      return ((nkb + q.S - 1) / q.S) * t_kb + (q.S > 1 ? 1.2 + 0.03 * q.bt + 0.17 * q.S : 0.0);
    };
    if (est(alt) < 0.95 * est(out)) out = alt;
    return true;
  };
  Plan plan;
  bool have = false;
  if (BITS == 8 && K > exact_ch) {
    // int8 activations: split K over a cluster so no CTA sums more than
    // exact_ch channels if that runs in one wave, else chunk inside each CTA
    Plan split;
    if (pick(false, (K + exact_ch - 1) / exact_ch, split) && split.one_wave) {
      plan = split;
      have = true;
    } else {
      have = pick(true, 1, plan);
    }
  } else {
    have = pick(false, 1, plan);
  }
  if (!have) return vqlin::fail(VQLIN_ERR_UNSUPPORTED_SHAPE, "qgemm: no tile plan for M=%d N=%d K=%d", M, N, K);
  const bool chunked = plan.chunked;
  const int bt = plan.bt, tiles_n = plan.tiles_n, tiles_m = plan.tiles_m, S = plan.S, NS = plan.NS;
  const int rows_per = plan.rows_per;
  const uint32_t a_col = plan.a_col, cols = plan.cols;
  const size_t dyn = plan.dyn;
  const bool tma_store = S == 1 && acc == nullptr && (N % 8) == 0;

  CUtensorMap tmW, tmX, tmY;
  if (!vqlin::tmap_encoder_available())
    return vqlin::fail(VQLIN_ERR_CUDA, "qgemm: cuTensorMapEncodeTiled is unavailable");
  bool ok = vqlin::encode_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, (uint64_t)w_row_bytes, (uint64_t)N,
                                  (uint64_t)w_row_bytes, RAW, kTileN,
                                  RAW == 32 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B);
  if (FX)
    ok = ok && vqlin::encode_tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, xq, (uint64_t)K, (uint64_t)M,
                                     (uint64_t)K * 2, 64, (uint32_t)bt, CU_TENSOR_MAP_SWIZZLE_128B);
  else if (BITS == 4)
    ok = ok && vqlin::encode_tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, (uint64_t)K, (uint64_t)M, (uint64_t)K,
                                     kBRow, (uint32_t)bt, CU_TENSOR_MAP_SWIZZLE_128B);
  else
    ok = ok && vqlin::encode_tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_UINT16, xq, (uint64_t)K, (uint64_t)M,
                                     (uint64_t)K * 2, kBRow / 2, (uint32_t)bt, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return vqlin::fail(VQLIN_ERR_CUDA, "qgemm: tensor map encoding failed (M=%d N=%d K=%d)", M, N, K);
  if (tma_store) {
    if (!vqlin::encode_tmap_2d(&tmY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Y, (uint64_t)N, (uint64_t)M, (uint64_t)N * 2,
                               kTileN, (uint32_t)bt, CU_TENSOR_MAP_SWIZZLE_NONE))
      return vqlin::fail(VQLIN_ERR_CUDA, "qgemm: output tensor map encoding failed (M=%d N=%d)", M, N);
  } else {
    tmY = tmW;  // unused
  }

  QgemmArgs a;
  a.sx = FX ? nullptr : sx; a.static_scale = FX ? sx : nullptr; a.sw = sw; a.bias = bias; a.Y = Y; a.acc = acc; a.status = status;
  a.M = M; a.N = N; a.K = K; a.bt = bt; a.nkb = nkb; a.stages = NS; a.tmem_cols = cols; a.a_col = a_col;
  {
    const uint32_t bt_pad = (uint32_t)((bt + 31) / 32 * 32);
    a.chunk_kb = chunked ? exact_ch / kb_codes : 0;
    a.d1_col = bt_pad;
    a.r_col = 2 * bt_pad;
  }
  a.wait_limit_ns = limit_ns; a.withhold_loads = withhold;
  a.tma_store = tma_store ? 1 : 0; a.rows_per = rows_per; a.sx_step = sx_step;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles_n, tiles_m, S);
  cfg.blockDim = dim3(NT, 1, 1);
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
  const cudaError_t e = vqlin::launched(cudaLaunchKernelEx(&cfg, kern, tmW, tmX, tmY, a));
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

vqlin_status launch_int_gemm_w4a8(const void* xq, const float* sx, const void* wq, const float* sw,
                                  const uint16_t* bias, uint16_t* Y, int32_t* acc, int M, int N, int K, int* status,
                                  cudaStream_t st) {
  if (M == 0 || N == 0) return VQLIN_OK;
  return launch_bits<8, false, 128, true>(xq, sx, wq, sw, bias, Y, acc, M, N, K, status, 0, kWaitLimitNs, st);
}

vqlin_status launch_int_gemm_static_scale(const void* xq, const float* static_scale, const void* wq, const float* sw,
                                          const uint16_t* bias, uint16_t* Y, int M, int N, int K, int* status,
                                          cudaStream_t st) {
  if (M == 0 || N == 0) return VQLIN_OK;
  return launch_bits<4>(xq, static_scale, wq, sw, bias, Y, nullptr, M, N, K, status, 0, kWaitLimitNs, st, 0);
}

vqlin_status launch_int_gemm_static_act(const uint16_t* X, const float* static_scale, int hb, const void* wq,
                                       const float* sw, const uint16_t* bias, uint16_t* Y, int M, int N, int K,
                                       int* status, cudaStream_t st) {
  if (M == 0 || N == 0) return VQLIN_OK;
  if (hb == 64)
    return launch_bits<4, true, 64>(X, static_scale, wq, sw, bias, Y, nullptr, M, N, K, status, 0, kWaitLimitNs, st);
  return launch_bits<4, true, 128>(X, static_scale, wq, sw, bias, Y, nullptr, M, N, K, status, 0, kWaitLimitNs, st);
}

vqlin_status launch_int_gemm_withheld(int bits, const void* xq, const void* wq, int32_t* acc, int M, int N, int K,
                                      int* status, uint64_t limit_ns, cudaStream_t st) {
  if (bits == 4)
    return launch_bits<4>(xq, nullptr, wq, nullptr, nullptr, nullptr, acc, M, N, K, status, 1, limit_ns, st);
  return launch_bits<8>(xq, nullptr, wq, nullptr, nullptr, nullptr, acc, M, N, K, status, 1, limit_ns, st);
}

}  // namespace vqlin
