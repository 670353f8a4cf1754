// Composite SVD . Hadamard block rotation with a zig-zag channel permutation.
//
// Method: "Omega-QVLA" technical summary, "Rotazione Composita SVD.Hadamard":
// a rotation from the singular value decomposition of the weights ("Rotazione
// SVD") composed with a normalised Hadamard matrix ("Rotazione Hadamard"),
// applied block-wise over b channels after a zig-zag permutation of the
// channels by weight column norm ("Implementazione a Blocchi").
//
// Readings fixed here (the summary gives no orientation, sign or dealing rule):
//   * the projection is y = x . W^T with W [N, K]; the rotation acts on the K
//     input channels; V_j holds the right singular vectors of W restricted to
//     block j's channels (the eigenvectors of its Gram matrix W_j^T W_j), in
//     descending order of singular value, each column signed so that its
//     largest-magnitude entry (the first on ties) is positive;
//   * R_j = V_j . H_b / sqrt(b); activations x~ = x[:, P] . blockdiag(R_j)
//     (online), weights W~ = W[:, P] . blockdiag(R_j) (offline), so that
//     x~ . W~^T = x . W^T;
//   * P: channels sorted by descending column norm (ties by channel index),
//     dealt to the K/b blocks in boustrophedon rounds (round r gives sorted
//     position r nb + i to block i for even r, to block nb - 1 - i for odd r),
//     keeping round order inside a block.
//
// Kernels:
//   offline (preparation, float64, favouring exactness over speed):
//     colnorm  -- squared column norms, a fixed summation order;
//     zigzag   -- rank of every channel, then its place in P;
//     gram     -- G_j = W_j^T W_j per block (stored in the block's R slot);
//     jacobi   -- parallel cyclic Jacobi on G_j (round-robin pairs, b/2
//                 disjoint rotations per step), then order, signs and the
//                 Hadamard factor by a float64 fast Walsh-Hadamard transform;
//   offline and online (the same tiled code): rows gathered by P and rotated
//     by blockdiag(R_j), two passes -- the first reduces each row's absmax
//     into the scale buffer (an atomic max of non-negative float bits), the
//     second recomputes the identical values and writes the codes -- then a
//     last kernel turns the absmax into the scale.  Weights rotate in
//     float64 (rounded once to float32, the oracle's order of rounding);
//     activations in float32, the online arithmetic.
#include <mutex>

#include "common.cuh"

namespace {

using namespace vqlin_dev;

constexpr int kThreads = 256;

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// ---------------------------------------------------------------- offline: P

// nrm[k] = sum_n W[n, k]^2 (float64).  CTA: 32 columns x 8 row phases; the
// eight phase sums of a column are added in phase order (deterministic).
__global__ void __launch_bounds__(kThreads)
colnorm_kernel(const uint16_t* __restrict__ W, int N, int K, double* __restrict__ nrm) {
  __shared__ double part[8][32];
  const int c = threadIdx.x & 31, ph = threadIdx.x >> 5;
  const int k = blockIdx.x * 32 + c;
  double acc = 0.0;
  if (k < K)
    for (int n = ph; n < N; n += 8) {
      const double v = (double)bf16f(W[(size_t)n * K + k]);
      acc = fma(v, v, acc);
    }
  part[ph][c] = acc;
  __syncthreads();
  if (ph == 0 && k < K) {
    double s = 0.0;
    for (int p = 0; p < 8; ++p) s += part[p][c];
    nrm[k] = s;
  }
}

// perm[position] = channel.  Thread per channel: its rank in descending norm
// order (ties by channel index), then the zig-zag place of that rank.
__global__ void __launch_bounds__(kThreads)
zigzag_kernel(const double* __restrict__ nrm, int K, int b, int* __restrict__ perm) {
  __shared__ double tile[kThreads];
  const int k = blockIdx.x * kThreads + threadIdx.x;
  const double mine = k < K ? nrm[k] : 0.0;
  int rank = 0;
  for (int j0 = 0; j0 < K; j0 += kThreads) {
    __syncthreads();
    tile[threadIdx.x] = j0 + threadIdx.x < K ? nrm[j0 + threadIdx.x] : 0.0;
    __syncthreads();
    const int lim = K - j0 < kThreads ? K - j0 : kThreads;
    for (int t = 0; t < lim; ++t) {
      const double o = tile[t];
      const int j = j0 + t;
      rank += (o > mine || (o == mine && j < k)) ? 1 : 0;
    }
  }
  if (k < K) {
    const int nb = K / b;
    const int r = rank / nb, i = rank % nb;
    const int blk = (r & 1) ? nb - 1 - i : i;
    perm[blk * b + r] = k;
  }
}

// ------------------------------------------------------- offline: Gram blocks

// G_j[r][c] = sum_n W[n, P[j b + r]] W[n, P[j b + c]] into R[j] (float64).
// CTA per (block j, 32-row band of G_j); thread = (row r of the band, 1/8 of
// the columns), rows n of W staged 32 at a time (gathered, as float64).
template <int B>
__global__ void __launch_bounds__(kThreads)
gram_kernel(const uint16_t* __restrict__ W, int N, int K, const int* __restrict__ perm, double* __restrict__ R) {
  constexpr int CPT = B / 8;  // columns per thread
  __shared__ double wt[32][B + 1];
  const int j = blockIdx.x, band = blockIdx.y;
  const int r = band * 32 + (threadIdx.x & 31);
  const int c0 = (threadIdx.x >> 5) * CPT;
  const int* pj = perm + (size_t)j * B;
  double acc[CPT];
#pragma unroll
  for (int c = 0; c < CPT; ++c) acc[c] = 0.0;
  for (int n0 = 0; n0 < N; n0 += 32) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < 32 * B; idx += kThreads) {
      const int nn = idx / B, cc = idx % B, n = n0 + nn;
      wt[nn][cc] = n < N ? (double)bf16f(W[(size_t)n * K + pj[cc]]) : 0.0;
    }
    __syncthreads();
    for (int nn = 0; nn < 32; ++nn) {
      const double a = wt[nn][r];
#pragma unroll
      for (int c = 0; c < CPT; ++c) acc[c] = fma(a, wt[nn][c0 + c], acc[c]);
    }
  }
  double* G = R + (size_t)j * B * B;
#pragma unroll
  for (int c = 0; c < CPT; ++c) G[(size_t)r * B + c0 + c] = acc[c];
}

// ------------------------------------------------- offline: Jacobi and R_j

__device__ __forceinline__ int sidx(int i, int j) {  // packed symmetric storage
  return i <= j ? j * (j + 1) / 2 + i : i * (i + 1) / 2 + j;
}

// Pair k of round-robin step t over B players (B - 1 steps give every pair
// once): player B - 1 meets t, the others meet across the circle.
__device__ __forceinline__ void rr_pair(int t, int k, int B, int& p, int& q) {
  if (k == 0) {
    p = t;
    q = B - 1;
  } else {
    p = (t + k) % (B - 1);
    q = (t - k + (B - 1)) % (B - 1);
  }
}

template <int B>
constexpr size_t jacobi_smem() {
  return ((size_t)B * (B + 1) / 2 + (size_t)B * B + 4 * (B / 2)) * sizeof(double) + (B + 1) * sizeof(int);
}

// One CTA per block j: G_j (from R[j]) -> eigenvectors V_j by cyclic Jacobi
// (G <- J^T G J, V <- V J with J the product of B/2 disjoint plane rotations
// per step; a rotation zeroes G[p][q]: tau = (G_qq - G_pp) / (2 G_pq),
// t = sign(tau) / (|tau| + sqrt(1 + tau^2)), c = 1 / sqrt(1 + t^2), s = t c,
// the symmetric Schur step of the classical method), until a sweep applies
// no rotation (|G_pq| <= 1e-15 sqrt(G_pp G_qq) for every pair) or after 40
// sweeps; then R[j] = V_sorted . H_B / sqrt(B).
template <int B>
__global__ void __launch_bounds__(kThreads, 1)
jacobi_kernel(double* __restrict__ R, int* __restrict__ status) {
  constexpr int P = B / 2;
  extern __shared__ double jsm[];
  double* Gp = jsm;                              // B (B + 1) / 2
  double* V = Gp + B * (B + 1) / 2;              // B x B, row-major
  double* cs = V + B * B;                        // [P]
  double* sn = cs + P;
  double* tn = sn + P;
  double* lam = tn + P;                          // [P] spare (eigenvalue staging)
  int* colof = reinterpret_cast<int*>(lam + P);  // [B]: column of sorted position
  int* rotated = colof + B;
  const int tid = threadIdx.x;
  double* G = R + (size_t)blockIdx.x * B * B;

  for (int idx = tid; idx < B * B; idx += kThreads) {
    const int i = idx / B, j = idx % B;
    if (i <= j) Gp[sidx(i, j)] = G[idx];
    V[idx] = i == j ? 1.0 : 0.0;
  }
  __syncthreads();

  for (int sweep = 0; sweep < 40; ++sweep) {
    if (tid == 0) *rotated = 0;
    __syncthreads();
    for (int t = 0; t < B - 1; ++t) {
      // (a) the step's rotations
      if (tid < P) {
        int p, q;
        rr_pair(t, tid, B, p, q);
        const double app = Gp[sidx(p, p)], aqq = Gp[sidx(q, q)], apq = Gp[sidx(p, q)];
        double c = 1.0, s = 0.0, tt = 0.0;
        if (apq != 0.0 && fabs(apq) > 1e-15 * sqrt(fabs(app * aqq))) {
          const double tau = (aqq - app) / (2.0 * apq);
          tt = tau >= 0.0 ? 1.0 / (tau + sqrt(1.0 + tau * tau)) : -1.0 / (-tau + sqrt(1.0 + tau * tau));
          c = 1.0 / sqrt(1.0 + tt * tt);
          s = tt * c;
          *rotated = 1;
        }
        cs[tid] = c;
        sn[tid] = s;
        tn[tid] = tt;
      }
      __syncthreads();
      // (b) G <- J^T G J over 2 x 2 blocks of pair indices (a <= a2), V <- V J
      for (int idx = tid; idx < P * (P + 1) / 2; idx += kThreads) {
        int a2 = (int)((sqrt(8.0 * idx + 1.0) - 1.0) * 0.5);
        while (a2 * (a2 + 1) / 2 > idx) --a2;
        while ((a2 + 1) * (a2 + 2) / 2 <= idx) ++a2;
        const int a = idx - a2 * (a2 + 1) / 2;
        int p, q;
        rr_pair(t, a, B, p, q);
        if (a == a2) {
          const double tt = tn[a];
          if (tt != 0.0) {
            const double apq = Gp[sidx(p, q)];
            Gp[sidx(p, p)] -= tt * apq;
            Gp[sidx(q, q)] += tt * apq;
            Gp[sidx(p, q)] = 0.0;
          }
        } else {
          int r, u;
          rr_pair(t, a2, B, r, u);
          const double ca = cs[a], sa = sn[a], cb = cs[a2], sb = sn[a2];
          const double apr = Gp[sidx(p, r)], apu = Gp[sidx(p, u)];
          const double aqr = Gp[sidx(q, r)], aqu = Gp[sidx(q, u)];
          const double tpr = cb * apr - sb * apu, tpu = sb * apr + cb * apu;
          const double tqr = cb * aqr - sb * aqu, tqu = sb * aqr + cb * aqu;
          Gp[sidx(p, r)] = ca * tpr - sa * tqr;
          Gp[sidx(p, u)] = ca * tpu - sa * tqu;
          Gp[sidx(q, r)] = sa * tpr + ca * tqr;
          Gp[sidx(q, u)] = sa * tpu + ca * tqu;
        }
      }
      for (int idx = tid; idx < B * P; idx += kThreads) {
        const int i = idx / P, a = idx % P;
        if (tn[a] == 0.0) continue;
        int p, q;
        rr_pair(t, a, B, p, q);
        const double vp = V[i * B + p], vq = V[i * B + q];
        V[i * B + p] = cs[a] * vp - sn[a] * vq;
        V[i * B + q] = sn[a] * vp + cs[a] * vq;
      }
      __syncthreads();
    }
    const int any = *rotated;
    __syncthreads();
    if (!any) break;
    if (sweep == 39 && tid == 0) atomicCAS(status, 0, (int)VQLIN_ERR_TIMEOUT);  // did not converge
  }

  // order by eigenvalue (descending, ties by index) and the sign of each column
  if (tid < B) {
    const double mine = Gp[sidx(tid, tid)];
    int rank = 0;
    for (int j = 0; j < B; ++j) {
      const double o = Gp[sidx(j, j)];
      rank += (o > mine || (o == mine && j < tid)) ? 1 : 0;
    }
    colof[rank] = tid;
  }
  __syncthreads();
  double sgn_of_sorted = 1.0;  // thread c < B: sign of the column at sorted position c
  if (tid < B) {
    const int col = colof[tid];
    double best = -1.0, val = 0.0;
    for (int r = 0; r < B; ++r) {
      const double v = V[r * B + col];
      if (fabs(v) > best) {
        best = fabs(v);
        val = v;
      }
    }
    sgn_of_sorted = val < 0.0 ? -1.0 : 1.0;
  }
  __syncthreads();
  // reuse the packed G storage: per-thread signs, then one B-row buffer per warp
  double* sgn = Gp;
  if (tid < B) sgn[tid] = sgn_of_sorted;
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  double* u = Gp + B + warp * B;
  const double inv = 1.0 / sqrt((double)B);
  for (int r = warp; r < B; r += kThreads / 32) {
    for (int c = lane; c < B; c += 32) u[c] = sgn[c] * V[r * B + colof[c]];
    __syncwarp();
    for (int h = 1; h < B; h <<= 1) {
      for (int e = lane; e < B / 2; e += 32) {
        const int i0 = (e / h) * 2 * h + (e % h), i1 = i0 + h;
        const double x0 = u[i0], x1 = u[i1];
        u[i0] = x0 + x1;
        u[i1] = x0 - x1;
      }
      __syncwarp();
    }
    for (int l = lane; l < B; l += 32) G[(size_t)r * B + l] = u[l] * inv;
    __syncwarp();
  }
}

// ------------------------------------- rows rotated by blockdiag(R_j), quantized

__device__ __forceinline__ double fma_t(double a, double b, double c) { return fma(a, b, c); }
__device__ __forceinline__ float fma_t(float a, float b, float c) { return fmaf(a, b, c); }
__device__ __forceinline__ float to_f32(double v) { return __double2float_rn(v); }
__device__ __forceinline__ float to_f32(float v) { return v; }

// Rows per thread: float64 tiles are kept smaller (register and shared-memory
// footprint).
template <typename T>
constexpr int rows_per_thread() { return sizeof(T) == 8 ? 2 : 4; }
template <typename T, int B>
constexpr int tile_rows() { return rows_per_thread<T>() * (kThreads / (B / 8)); }
template <typename T, int B>
constexpr size_t rot_smem() { return ((size_t)B * B + (size_t)tile_rows<T, B>() * (B + 1)) * sizeof(T); }

// CTA: TR rows x block j.  PASS 0: each row's absmax (over its float32
// values) into amax_bits[row] by an atomic max; PASS 1: the codes, with
// s = absmax / qmax (IEEE division) and c = clamp(rint(v / s), -qmax, qmax).
// WEIGHT: packed sign-magnitude codes of the weight layout ([rows, K/2] int4
// nibbles, [rows, K] int8 bytes); else the activation operand encoding of the
// integer GEMM (one byte per int4 code, one 16-bit word per int8 code).
template <typename T, int B, int BITS, bool WEIGHT, int PASS>
__global__ void __launch_bounds__(kThreads)
rotate_rows_kernel(const uint16_t* __restrict__ X, int rows, int K, const int* __restrict__ perm,
                   const double* __restrict__ R, int* __restrict__ amax_bits, void* __restrict__ Q) {
  constexpr int qmax = (1 << (BITS - 1)) - 1;
  constexpr int CG = B / 8;                     // column groups of 8 channels
  constexpr int RPT = rows_per_thread<T>();
  constexpr int TR = tile_rows<T, B>();
  extern __shared__ __align__(16) uint8_t rsm[];
  T* Rs = reinterpret_cast<T*>(rsm);            // [B][B]
  T* xs = Rs + B * B;                           // [TR][B + 1]
  const int tid = threadIdx.x, j = blockIdx.y;
  const int row0 = blockIdx.x * TR;
  const int* pj = perm + (size_t)j * B;
  const double* Rj = R + (size_t)j * B * B;
  for (int idx = tid; idx < B * B; idx += kThreads) Rs[idx] = (T)Rj[idx];
  for (int idx = tid; idx < TR * B; idx += kThreads) {
    const int rr = idx / B, c = idx % B, row = row0 + rr;
    xs[rr * (B + 1) + c] = row < rows ? (T)bf16f(X[(size_t)row * K + pj[c]]) : (T)0;
  }
  __syncthreads();

  const int cg = tid % CG, rg = tid / CG;
  T acc[RPT][8];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[i][e] = (T)0;
  for (int r = 0; r < B; ++r) {
    T rv[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) rv[e] = Rs[r * B + 8 * cg + e];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const T xv = xs[(rg * RPT + i) * (B + 1) + r];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[i][e] = fma_t(xv, rv[e], acc[i][e]);
    }
  }

#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int row = row0 + rg * RPT + i;
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = to_f32(acc[i][e]);
    if (PASS == 0) {
      float m = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[e]));
#pragma unroll
      for (int o = CG / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (cg == 0 && row < rows) atomicMax(amax_bits + row, __float_as_int(m));
    } else if (row < rows) {
      const float s = __fdiv_rn(__int_as_float(amax_bits[row]), (float)qmax);
      uint32_t mag[8], neg[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float c = s > 0.0f ? rintf(__fdiv_rn(v[e], s)) : 0.0f;
        c = fminf(fmaxf(c, (float)(-qmax)), (float)qmax);
        mag[e] = (uint32_t)fabsf(c);
        neg[e] = c < 0.0f ? 1u : 0u;
      }
      const size_t col = (size_t)j * B + 8 * cg;
      if (WEIGHT && BITS == 4) {
        uint32_t w = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) w |= (mag[e] | (neg[e] << 3)) << (4 * e);
        *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(Q) + (size_t)row * (K / 2) + col / 2) = w;
      } else if (WEIGHT || BITS == 4) {
        // one byte per code: weight int8 (c < 0) << 7 | |c|; activation int4
        // s << 7 | |c| (the same bits)
        uint32_t w[2] = {0u, 0u};
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e >> 2] |= (mag[e] | (neg[e] << 7)) << (8 * (e & 3));
        *reinterpret_cast<uint2*>(static_cast<uint8_t*>(Q) + (size_t)row * K + col) = make_uint2(w[0], w[1]);
      } else {
        uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e >> 1] |= (mag[e] | (neg[e] << 15)) << (16 * (e & 1));
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(Q) + (size_t)row * K + col) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
}

// scale[row] = absmax / qmax, in place over the absmax bits.
template <int BITS>
__global__ void finalize_scale_kernel(int* __restrict__ bits_io, int rows) {
  constexpr int qmax = (1 << (BITS - 1)) - 1;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < rows) {
    const float s = __fdiv_rn(__int_as_float(bits_io[i]), (float)qmax);
    bits_io[i] = __float_as_int(s);
  }
}

// ------------------------------------------------------------------ host side

template <auto Fn>
cudaError_t set_smem_once(size_t bytes) {
  // function attributes are per device and per kernel: set once for each
  static std::mutex mu;
  static bool set[64] = {};
  static cudaError_t res[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!set[dev]) {
    res[dev] = cudaFuncSetAttribute(Fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    set[dev] = true;
  }
  return res[dev];
}

template <int B>
cudaError_t prepare_b(const uint16_t* W, int N, int K, int* perm, double* R, int* status, cudaStream_t st) {
  // column norms into the first K doubles of R (overwritten by the Gram blocks)
  colnorm_kernel<<<(K + 31) / 32, kThreads, 0, st>>>(W, N, K, R);
  zigzag_kernel<<<(K + kThreads - 1) / kThreads, kThreads, 0, st>>>(R, K, B, perm);
  gram_kernel<B><<<dim3(K / B, B / 32), kThreads, 0, st>>>(W, N, K, perm, R);
  cudaError_t e = set_smem_once<&jacobi_kernel<B>>(jacobi_smem<B>());
  if (e != cudaSuccess) return e;
  jacobi_kernel<B><<<K / B, kThreads, jacobi_smem<B>(), st>>>(R, status);
  return vqlin::launched(cudaGetLastError(), 4);
}

template <typename T, int B, int BITS, bool WEIGHT>
cudaError_t rotate_quant_b(const uint16_t* X, int rows, int K, const int* perm, const double* R, void* Q,
                           float* scale, cudaStream_t st) {
  constexpr size_t smem = rot_smem<T, B>();
  cudaError_t e = set_smem_once<&rotate_rows_kernel<T, B, BITS, WEIGHT, 0>>(smem);
  if (e == cudaSuccess) e = set_smem_once<&rotate_rows_kernel<T, B, BITS, WEIGHT, 1>>(smem);
  if (e != cudaSuccess) return e;
  int* amax = reinterpret_cast<int*>(scale);
  e = cudaMemsetAsync(amax, 0, sizeof(float) * (size_t)rows, st);
  if (e != cudaSuccess) return e;
  const dim3 grid((rows + tile_rows<T, B>() - 1) / tile_rows<T, B>(), K / B);
  rotate_rows_kernel<T, B, BITS, WEIGHT, 0><<<grid, kThreads, smem, st>>>(X, rows, K, perm, R, amax, Q);
  rotate_rows_kernel<T, B, BITS, WEIGHT, 1><<<grid, kThreads, smem, st>>>(X, rows, K, perm, R, amax, Q);
  finalize_scale_kernel<BITS><<<(rows + 255) / 256, 256, 0, st>>>(amax, rows);
  return vqlin::launched(cudaGetLastError(), 3);
}

template <typename T, bool WEIGHT>
cudaError_t rotate_quant(const uint16_t* X, int rows, int K, int bits, int b, const int* perm, const double* R,
                         void* Q, float* scale, cudaStream_t st) {
  if (b == 64)
    return bits == 4 ? rotate_quant_b<T, 64, 4, WEIGHT>(X, rows, K, perm, R, Q, scale, st)
                     : rotate_quant_b<T, 64, 8, WEIGHT>(X, rows, K, perm, R, Q, scale, st);
  return bits == 4 ? rotate_quant_b<T, 128, 4, WEIGHT>(X, rows, K, perm, R, Q, scale, st)
                   : rotate_quant_b<T, 128, 8, WEIGHT>(X, rows, K, perm, R, Q, scale, st);
}

}  // namespace

namespace vqlin {

cudaError_t launch_composite_prepare(const uint16_t* W, int N, int K, int b, int* perm, double* R, int* status,
                                     cudaStream_t st) {
  return b == 64 ? prepare_b<64>(W, N, K, perm, R, status, st) : prepare_b<128>(W, N, K, perm, R, status, st);
}

cudaError_t launch_weight_quant_composite(const uint16_t* W, int N, int K, int bits, int b, const int* perm,
                                          const double* R, uint8_t* q, float* scale, cudaStream_t st) {
  return rotate_quant<double, true>(W, N, K, bits, b, perm, R, q, scale, st);
}

cudaError_t launch_act_composite_quant(const uint16_t* X, int M, int K, int bits, int b, const int* perm,
                                       const double* R, void* q, float* scale, cudaStream_t st) {
  return rotate_quant<float, false>(X, M, K, bits, b, perm, R, q, scale, st);
}

}  // namespace vqlin
