// Observer statistics of attention rows (kv_attend_stats).
//
// What it computes, per query row, from the fp32 softmax p of sm_scale * q K^T
// over every key of the cache (the Catnip study, "Catnip Week 10 KV Cache
// Attention Study", section 实验设计 step 5 and its Structural / Effective /
// Numerical MXFP8 notes, and section "Q/K 与 probability quantization 的影响"):
//   entropy H = -sum p ln p and the entropy-equivalent support exp(H) / N;
//   the mass of the ceil(1 %, 5 %, 10 % of N) largest probabilities;
//   the share of probabilities that are exactly 0 in fp32 (structural zeros);
//   the MXFP8 probability path: p rounded to E4M3 with one E8M0 scale per 32
//     keys; the share of keys nonzero in fp32 but 0 there, 0.5 sum |p_mx - p|
//     and sum p_mx;
//   the MXFP8 Q/K path: q and every key rotated by the signed Hadamard
//     transform (x * signs) H / sqrt(D) when signs are given, both rounded to
//     E4M3 with one E8M0 scale per 32 along D; the total variation between its
//     softmax and p, and whether both rows have the same argmax.
//
// Three kernels. keys_kernel writes, once per (sequence, KV head), every key
// twice to workspace in fp32: as attention reads it (int4 part dequantized,
// window as stored) and on the MXFP8 Q/K path (rotated, rounded); warp per
// key, lane l holding features l*E .. l*E + E - 1 (E = D / 32), the Hadamard
// transform as E-wide in-thread butterflies followed by five lane-exchange
// stages. Both copies are stored in tiles of 32 keys, feature-major
// ([unit][tile][D][32]), transposed through shared memory. scores_kernel: one
// CTA per 16 query rows of a head and a range of key tiles; lane = key, so
// every tile row is one 128-byte load, read once for all 16 rows, and each
// lane keeps the 16 rows' dot products on both paths (q from shared memory,
// four features per broadcast load). stats_kernel: one CTA per query row;
// the reference score row comes from workspace into shared memory (for N up
// to kStagedTokens; longer rows are swept where they lie in the workspace,
// from L2), the MXFP8 Q/K row, which three passes read, stays in the
// workspace; the statistics are block reductions over them, and each top-k
// mass takes the k-th largest probability from a radix select over the
// float bits.

#include <cuda_fp8.h>
#include <math_constants.h>

#include <algorithm>

#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct StatsArgs {
  const uint8_t *k_codes;
  const float *k_scales;
  const void *k_window;
  const uint8_t *k_e8m0;
  int kwin;
  int Hkv, N, D, cut, Gs, Ws;
  int Hq, group, n_q;
  const void *q;
  int q_dtype;
  float sm_scale;
  const float *signs;  // [D] +-1, or nullptr: no rotation
  float *stats;        // [rows][KVQ_N_STATS]
  float *k_ref;        // workspace [units][T][D][32]: keys as attention reads them
  float *k_mx;         // workspace [units][T][D][32]: keys on the MXFP8 Q/K path
  float *s_ref;        // workspace [rows][N]: sm_scale * q k on the reference path
  float *s_mx;         // workspace [rows][N]: the same on the MXFP8 Q/K path
  int T;               // key tiles of 32 per unit
  int key_splits;      // scores_kernel CTAs per group of rows
  KernelCtl ctl;
};

constexpr int kRows = 16;  // query rows per scores_kernel CTA


__device__ __forceinline__ float key_value(const StatsArgs &a, long u, int j, int d) {
  if (j < a.cut) {
    const long g = u * a.Gs + (j >> 5);
    if (!in_bounds(a.ctl, a.k_codes + (g * kGroup + (j & 31)) * (a.D / 2) + d / 2, 1) ||
        !in_bounds(a.ctl, a.k_scales + g * a.D + d, sizeof(float)))
      return 0.0f;
    const uint8_t byte = a.k_codes[(g * kGroup + (j & 31)) * (a.D / 2) + d / 2];
    const int code = static_cast<int>((d & 1) ? (byte >> 4) : (byte & 15)) - 8;
    return static_cast<float>(code) * a.k_scales[g * a.D + d];
  }
  const long row = u * a.Ws + (j - a.cut);
  const size_t eb = a.kwin == KVQ_F32 ? 4 : a.kwin == KVQ_BF16 ? 2 : 1;
  if (!in_bounds(a.ctl, static_cast<const uint8_t *>(a.k_window) + (row * a.D + d) * eb, eb) ||
      (a.kwin == KVQ_MXFP8 &&
       !in_bounds(a.ctl, a.k_e8m0 + row * (a.D / kGroup) + d / kGroup, 1)))
    return 0.0f;
  if (a.kwin == KVQ_F32) return static_cast<const float *>(a.k_window)[row * a.D + d];
  if (a.kwin == KVQ_BF16)
    return load_f32(static_cast<const __nv_bfloat16 *>(a.k_window) + row * a.D + d);
  return mxfp8_value(static_cast<const uint8_t *>(a.k_window)[row * a.D + d],
                     a.k_e8m0[row * (a.D / kGroup) + d / kGroup]);
}

// Signed Hadamard transform of a D-vector spread over a warp, E per lane
// (element l*E + t in x[t]): multiply by the signs, butterflies over the low
// log2(E) index bits in registers, then over the five lane bits by shuffles.
template <int E>
__device__ __forceinline__ void signed_hadamard(float (&x)[E], const float *signs, int lane) {
#pragma unroll
  for (int t = 0; t < E; ++t) x[t] *= signs[lane * E + t];
#pragma unroll
  for (int b = 1; b < E; b <<= 1)
#pragma unroll
    for (int t = 0; t < E; ++t)
      if (!(t & b)) {
        const float lo = x[t], hi = x[t | b];
        x[t] = lo + hi;
        x[t | b] = lo - hi;
      }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const bool upper = lane & o;
#pragma unroll
    for (int t = 0; t < E; ++t) {
      const float other = __shfl_xor_sync(0xffffffffu, x[t], o);
      x[t] = upper ? other - x[t] : x[t] + other;
    }
  }
  const float norm = rsqrtf(static_cast<float>(E * 32));
#pragma unroll
  for (int t = 0; t < E; ++t) x[t] *= norm;
}

// MXFP8 rounding along D of a warp-spread vector: a 32-block is 32 / E lanes.
template <int E>
__device__ __forceinline__ void mxfp8_round_row(float (&x)[E]) {
  float amax = 0.0f;
#pragma unroll
  for (int t = 0; t < E; ++t) amax = fmaxf(amax, fabsf(x[t]));
#pragma unroll
  for (int o = 1; o < 32 / E; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int e = mxfp8_block_exp(amax);
  const float down = pow2_of(-e), up = pow2_of(e);
#pragma unroll
  for (int t = 0; t < E; ++t) x[t] = __fmul_rn(e4m3_value(mxfp8_code(x[t], down)), up);
}

// Both workspace copies of the 32 keys of tile blockIdx.x of unit
// blockIdx.y: warp w computes keys 4w .. 4w + 3 of the tile (zeros past N)
// into shared memory [2][D][33], then the CTA stores both [D][32] tiles with
// whole-row writes.
template <int E>
__global__ void __launch_bounds__(kThreads) keys_kernel(const StatsArgs a) {
  wait_prior_grid();
  allow_next_grid();
  extern __shared__ float tile[];  // [2][D][33]
  constexpr int D = 32 * E;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long u = blockIdx.y;
  const long o = (u * a.T + blockIdx.x) * D * 32;
  // the signs and this tile's two outputs (the same in every thread)
  if ((a.signs && !in_bounds(a.ctl, a.signs, sizeof(float) * D)) ||
      !in_bounds(a.ctl, a.k_ref + o, sizeof(float) * D * 32) ||
      !in_bounds(a.ctl, a.k_mx + o, sizeof(float) * D * 32))
    return;
  for (int kk = 0; kk < 4; ++kk) {
    const int c = 4 * warp + kk;  // key within the tile
    const int j = blockIdx.x * 32 + c;
    float x[E];
    if (j < a.N) {
#pragma unroll
      for (int t = 0; t < E; ++t) x[t] = key_value(a, u, j, lane * E + t);
    } else {
#pragma unroll
      for (int t = 0; t < E; ++t) x[t] = 0.0f;
    }
#pragma unroll
    for (int t = 0; t < E; ++t) tile[(lane * E + t) * 33 + c] = x[t];
    if (j < a.N) {
      if (a.signs) signed_hadamard<E>(x, a.signs, lane);
      mxfp8_round_row<E>(x);
    }
#pragma unroll
    for (int t = 0; t < E; ++t) tile[(D + lane * E + t) * 33 + c] = x[t];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < D * 32; i += kThreads) {
    a.k_ref[o + i] = tile[(i >> 5) * 33 + (i & 31)];
    a.k_mx[o + i] = tile[(D + (i >> 5)) * 33 + (i & 31)];
  }
}

// Scores of query rows i0 .. i0 + 15 of head blockIdx.y (sequence b, query
// head h) on both paths against the key tiles of split blockIdx.z. Rows past
// n_q are computed as zeros and not stored.
template <int E>
__global__ void __launch_bounds__(kThreads) scores_kernel(const StatsArgs a) {
  wait_prior_grid();
  allow_next_grid();
  constexpr int D = 32 * E;
  __shared__ __align__(16) float qf[kRows][D];
  __shared__ __align__(16) float qm[kRows][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long bh = blockIdx.y;  // b * Hq + h
  const int h = static_cast<int>(bh % a.Hq);
  const long u = (bh / a.Hq) * a.Hkv + h / a.group;
  const int i0 = blockIdx.x * kRows;
  const int nr = min(kRows, a.n_q - i0);
  const long row0 = bh * a.n_q + i0;
  const size_t qe = a.q_dtype == KVQ_F32 ? 4 : 2;
  // q rows, signs and score rows of the block (the same in every thread)
  if (!in_bounds(a.ctl, static_cast<const uint8_t *>(a.q) + row0 * D * qe, qe * D * nr) ||
      (a.signs && !in_bounds(a.ctl, a.signs, sizeof(float) * D)) ||
      !in_bounds(a.ctl, a.s_ref + row0 * a.N, sizeof(float) * a.N * nr) ||
      !in_bounds(a.ctl, a.s_mx + row0 * a.N, sizeof(float) * a.N * nr))
    return;
  for (int e = threadIdx.x; e < kRows * D; e += kThreads) {
    const int r = e / D, d = e % D;
    const long gi = (row0 + r) * D + d;
    qf[r][d] = r >= nr ? 0.0f
               : a.q_dtype == KVQ_F32 ? static_cast<const float *>(a.q)[gi]
                                      : load_f32(static_cast<const __nv_bfloat16 *>(a.q) + gi);
  }
  __syncthreads();
  for (int r = warp; r < kRows; r += kWarps) {
    float x[E];
#pragma unroll
    for (int t = 0; t < E; ++t) x[t] = qf[r][lane * E + t];
    if (a.signs) signed_hadamard<E>(x, a.signs, lane);
    mxfp8_round_row<E>(x);
#pragma unroll
    for (int t = 0; t < E; ++t) qm[r][lane * E + t] = x[t];
  }
  __syncthreads();

  const int per = (a.T + a.key_splits - 1) / a.key_splits;
  const int t_lo = blockIdx.z * per, t_hi = min(a.T, t_lo + per);
  // a warp takes two tiles per step (lane = key in each): every q load from
  // shared memory feeds both
  for (int t0 = t_lo + warp; t0 < t_hi; t0 += 2 * kWarps) {
    const int t1 = t0 + kWarps < t_hi ? t0 + kWarps : t0;
    if (!in_bounds(a.ctl, a.k_ref + (u * a.T + t0) * D * 32, sizeof(float) * D * 32) ||
        !in_bounds(a.ctl, a.k_mx + (u * a.T + t0) * D * 32, sizeof(float) * D * 32) ||
        !in_bounds(a.ctl, a.k_ref + (u * a.T + t1) * D * 32, sizeof(float) * D * 32) ||
        !in_bounds(a.ctl, a.k_mx + (u * a.T + t1) * D * 32, sizeof(float) * D * 32))
      continue;
    const float *kr0 = a.k_ref + (u * a.T + t0) * D * 32 + lane;
    const float *km0 = a.k_mx + (u * a.T + t0) * D * 32 + lane;
    const float *kr1 = a.k_ref + (u * a.T + t1) * D * 32 + lane;
    const float *km1 = a.k_mx + (u * a.T + t1) * D * 32 + lane;
    float ar[2][kRows], am[2][kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) ar[0][r] = am[0][r] = ar[1][r] = am[1][r] = 0.0f;
#pragma unroll 1
    for (int d = 0; d < D; d += 4) {
      float xr[2][4], xm[2][4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        xr[0][e] = __ldg(kr0 + (d + e) * 32);
        xm[0][e] = __ldg(km0 + (d + e) * 32);
        xr[1][e] = __ldg(kr1 + (d + e) * 32);
        xm[1][e] = __ldg(km1 + (d + e) * 32);
      }
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        const float4 f = *reinterpret_cast<const float4 *>(&qf[r][d]);
        const float4 g = *reinterpret_cast<const float4 *>(&qm[r][d]);
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          ar[x][r] = fmaf(f.x, xr[x][0], ar[x][r]);
          ar[x][r] = fmaf(f.y, xr[x][1], ar[x][r]);
          ar[x][r] = fmaf(f.z, xr[x][2], ar[x][r]);
          ar[x][r] = fmaf(f.w, xr[x][3], ar[x][r]);
          am[x][r] = fmaf(g.x, xm[x][0], am[x][r]);
          am[x][r] = fmaf(g.y, xm[x][1], am[x][r]);
          am[x][r] = fmaf(g.z, xm[x][2], am[x][r]);
          am[x][r] = fmaf(g.w, xm[x][3], am[x][r]);
        }
      }
    }
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const int j = (x ? t1 : t0) * 32 + lane;
      if ((x == 0 || t1 != t0) && j < a.N) {
#pragma unroll
        for (int r = 0; r < kRows; ++r)
          if (r < nr) {
            a.s_ref[(row0 + r) * a.N + j] = a.sm_scale * ar[x][r];
            a.s_mx[(row0 + r) * a.N + j] = a.sm_scale * am[x][r];
          }
      }
    }
  }
}

// ---- the same scores on the tensor cores (D = 128)
// mma.sync m16n8k8 with tf32 operands: 16 query rows are M, 8 keys of a tile
// N, 8 features K; a CTA takes 48 query rows, so that each key fragment read
// from L2 feeds three m-tiles (the key tiles are read once per 48 rows instead
// of once per 16). Reference path: each operand split into a tf32 high
// part and a tf32 low part (x = hi + lo to about 2^-22 of |x|), the product
// taken as hi.hi + hi.lo + lo.hi (three MMAs; the lo.lo term and the split
// residuals are below 2^-21 of a product). MXFP8 Q/K path: E4M3 values times
// a power of two have at most four significant bits, exact in tf32, so one
// MMA gives the exact products. Accumulation in fp32.
__device__ __forceinline__ uint32_t tf32_hi(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void mma_tf32(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

constexpr int kQPad = 132;  // floats per staged q row: lanes (g, t) read banks 4g + t
constexpr int kTcRows = 48;  // query rows per CTA: three m-tiles share each key fragment

struct ScoresTcSmem {
  float qf[kTcRows][128];
  uint32_t q_hi[kTcRows][kQPad], q_lo[kTcRows][kQPad], q_mx[kTcRows][kQPad];
};

__global__ void __launch_bounds__(kThreads) scores_tc_kernel(const StatsArgs a) {
  wait_prior_grid();
  allow_next_grid();
  constexpr int D = 128, E = 4, kM = kTcRows / 16;
  extern __shared__ __align__(16) uint8_t tc_smem_raw[];
  ScoresTcSmem &sm = *reinterpret_cast<ScoresTcSmem *>(tc_smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long bh = blockIdx.y;  // b * Hq + h
  const int h = static_cast<int>(bh % a.Hq);
  const long u = (bh / a.Hq) * a.Hkv + h / a.group;
  const int i0 = blockIdx.x * kTcRows;
  const int nr = min(kTcRows, a.n_q - i0);
  const long row0 = bh * a.n_q + i0;
  const size_t qe = a.q_dtype == KVQ_F32 ? 4 : 2;
  if (!in_bounds(a.ctl, static_cast<const uint8_t *>(a.q) + row0 * D * qe, qe * D * nr) ||
      (a.signs && !in_bounds(a.ctl, a.signs, sizeof(float) * D)) ||
      !in_bounds(a.ctl, a.s_ref + row0 * a.N, sizeof(float) * a.N * nr) ||
      !in_bounds(a.ctl, a.s_mx + row0 * a.N, sizeof(float) * a.N * nr))
    return;
  for (int e = threadIdx.x; e < kTcRows * D; e += kThreads) {
    const int r = e / D, d = e % D;
    const long gi = (row0 + r) * D + d;
    const float x = r >= nr ? 0.0f
                    : a.q_dtype == KVQ_F32 ? static_cast<const float *>(a.q)[gi]
                                           : load_f32(static_cast<const __nv_bfloat16 *>(a.q) + gi);
    sm.qf[r][d] = x;
    const uint32_t hi = tf32_hi(x);
    sm.q_hi[r][d] = hi;
    sm.q_lo[r][d] = tf32_hi(x - __uint_as_float(hi));
  }
  __syncthreads();
  for (int r = warp; r < kTcRows; r += kWarps) {
    float x[E];
#pragma unroll
    for (int t = 0; t < E; ++t) x[t] = sm.qf[r][lane * E + t];
    if (a.signs) signed_hadamard<E>(x, a.signs, lane);
    mxfp8_round_row<E>(x);
#pragma unroll
    for (int t = 0; t < E; ++t) sm.q_mx[r][lane * E + t] = __float_as_uint(x[t]);
  }
  __syncthreads();

  const int g = lane >> 2, t4 = lane & 3;
  const int per = (a.T + a.key_splits - 1) / a.key_splits;
  const int t_lo = blockIdx.z * per, t_hi = min(a.T, t_lo + per);
  for (int tile = t_lo + warp; tile < t_hi; tile += kWarps) {
    const float *kr = a.k_ref + (u * a.T + tile) * D * 32;
    const float *km = a.k_mx + (u * a.T + tile) * D * 32;
    if (!in_bounds(a.ctl, kr, sizeof(float) * D * 32) ||
        !in_bounds(a.ctl, km, sizeof(float) * D * 32))
      continue;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {  // keys 16 half .. 16 half + 15 of the tile
      float cr[kM][2][4], cm[kM][2][4];  // [m-tile][key group of 8][fragment]
#pragma unroll
      for (int m = 0; m < kM; ++m)
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int j = 0; j < 4; ++j) cr[m][n][j] = cm[m][n][j] = 0.0f;
#pragma unroll 2
      for (int k0 = 0; k0 < D; k0 += 8) {
        uint32_t bh[2][2], bl[2][2], bm[2][2];
#pragma unroll
        for (int n = 0; n < 2; ++n) {
          // B[k][key]: features k0 + t4 and k0 + t4 + 4 of key 16 half + 8n + g
          const int key = 16 * half + 8 * n + g;
          const float x0 = __ldg(kr + (k0 + t4) * 32 + key);
          const float x1 = __ldg(kr + (k0 + t4 + 4) * 32 + key);
          bm[n][0] = __float_as_uint(__ldg(km + (k0 + t4) * 32 + key));
          bm[n][1] = __float_as_uint(__ldg(km + (k0 + t4 + 4) * 32 + key));
          bh[n][0] = tf32_hi(x0);
          bh[n][1] = tf32_hi(x1);
          bl[n][0] = tf32_hi(x0 - __uint_as_float(bh[n][0]));
          bl[n][1] = tf32_hi(x1 - __uint_as_float(bh[n][1]));
        }
#pragma unroll
        for (int m = 0; m < kM; ++m) {
          const int ra = 16 * m + g, rb = ra + 8;
          const uint32_t ah[4] = {sm.q_hi[ra][k0 + t4], sm.q_hi[rb][k0 + t4],
                                  sm.q_hi[ra][k0 + t4 + 4], sm.q_hi[rb][k0 + t4 + 4]};
          const uint32_t al[4] = {sm.q_lo[ra][k0 + t4], sm.q_lo[rb][k0 + t4],
                                  sm.q_lo[ra][k0 + t4 + 4], sm.q_lo[rb][k0 + t4 + 4]};
          const uint32_t am[4] = {sm.q_mx[ra][k0 + t4], sm.q_mx[rb][k0 + t4],
                                  sm.q_mx[ra][k0 + t4 + 4], sm.q_mx[rb][k0 + t4 + 4]};
#pragma unroll
          for (int n = 0; n < 2; ++n) {
            mma_tf32(cr[m][n], al[0], al[1], al[2], al[3], bh[n][0], bh[n][1]);
            mma_tf32(cr[m][n], ah[0], ah[1], ah[2], ah[3], bl[n][0], bl[n][1]);
            mma_tf32(cr[m][n], ah[0], ah[1], ah[2], ah[3], bh[n][0], bh[n][1]);
            mma_tf32(cm[m][n], am[0], am[1], am[2], am[3], bm[n][0], bm[n][1]);
          }
        }
      }
      // C fragment: rows 16m + g (+ 8); keys 16 half + 8n + 2t4 (+ 1)
#pragma unroll
      for (int m = 0; m < kM; ++m)
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int r = 16 * m + g + 8 * (j >> 1);
            const int key = tile * 32 + 16 * half + 8 * n + 2 * t4 + (j & 1);
            if (r < nr && key < a.N) {
              a.s_ref[(row0 + r) * a.N + key] = a.sm_scale * cr[m][n][j];
              a.s_mx[(row0 + r) * a.N + key] = a.sm_scale * cm[m][n][j];
            }
          }
    }
  }
}

__device__ __forceinline__ float block_sum(float x, float *red) {
  x = warp_sum(x);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = x;
  __syncthreads();
  float t = 0.0f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) t += red[w];
  return t;
}

// Indices of the first maxima of a[0, n) and b[0, n) in one pass.
__device__ __forceinline__ void block_argmax2(const float *a, const float *b, int n, float *red,
                                              int *redi, int &ia, int &ib) {
  float best[2] = {-CUDART_INF_F, -CUDART_INF_F};
  int bi[2] = {0x7fffffff, 0x7fffffff};
  for (int j = threadIdx.x; j < n; j += kThreads) {
    if (a[j] > best[0]) {
      best[0] = a[j];
      bi[0] = j;
    }
    if (b[j] > best[1]) {
      best[1] = b[j];
      bi[1] = j;
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1)
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const float ob = __shfl_xor_sync(0xffffffffu, best[x], o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi[x], o);
      if (ob > best[x] || (ob == best[x] && oi < bi[x])) {
        best[x] = ob;
        bi[x] = oi;
      }
    }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0)
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      red[x * kWarps + warp] = best[x];
      redi[x * kWarps + warp] = bi[x];
    }
  __syncthreads();
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    float bb = red[x * kWarps];
    int ii = redi[x * kWarps];
    for (int w = 1; w < kWarps; ++w)
      if (red[x * kWarps + w] > bb || (red[x * kWarps + w] == bb && redi[x * kWarps + w] < ii)) {
        bb = red[x * kWarps + w];
        ii = redi[x * kWarps + w];
      }
    (x == 0 ? ia : ib) = ii;
  }
}

// 256-bucket histogram of bits [shift, shift + 8) of the keys of x[0, n)
// whose bits under `mask` equal `prefix`.
__device__ __forceinline__ void bucket_histogram(const float *x, int n, uint32_t prefix,
                                                 uint32_t mask, int shift, uint32_t *hist) {
  for (int i = threadIdx.x; i < 256; i += kThreads) hist[i] = 0u;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const uint32_t b = __float_as_uint(x[i]);
    if ((b & mask) == prefix) atomicAdd(&hist[(b >> shift) & 255u], 1u);
  }
  __syncthreads();
}

// The bucket d holding the k-th largest key: count above d < k <= count above
// d + hist[d]. Warp 0 scans (lane l owns buckets 8l .. 8l + 7) and leaves
// {d, k - count above d} in sel; every thread reads it after the barrier.
__device__ __forceinline__ void pick_bucket(const uint32_t *hist, int k, uint32_t *sel) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const uint32_t kk = static_cast<uint32_t>(k);
    uint32_t hb[8], tot = 0u;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      hb[e] = hist[8 * lane + e];
      tot += hb[e];
    }
    uint32_t above = tot;  // inclusive suffix sum over lanes >= lane
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_down_sync(0xffffffffu, above, o);
      if (lane + o < 32) above += v;
    }
    const uint32_t all = __shfl_sync(0xffffffffu, above, 0);
    uint32_t cum = above - tot;  // buckets of the lanes above
    bool found = false;
    uint32_t fd = 0u, fk = 0u;
#pragma unroll
    for (int e = 7; e >= 0; --e) {
      if (!found && cum < kk && cum + hb[e] >= kk) {
        found = true;
        fd = 8u * lane + e;
        fk = kk - cum;
      }
      cum += hb[e];
    }
    if (found) {
      sel[0] = fd;
      sel[1] = fk;
    }
    if (__ballot_sync(0xffffffffu, found) == 0u && lane == 0) {
      sel[0] = 0u;
      sel[1] = kk - (all - hb[0]);
    }
  }
  __syncthreads();
}

// Bits of the k-th largest of x[0, n) (all x >= 0, 1 <= k <= n) for three
// values of k: a radix select of four rounds of 8 bits each, the first
// round's histogram (all keys) shared by the three.
__device__ void kth_largest_bits3(const float *x, int n, const int (&k3)[3], uint32_t (&bits)[3],
                                  uint32_t *hist, uint32_t *hist_top, uint32_t *sel) {
  bucket_histogram(x, n, 0u, 0u, 24, hist_top);
#pragma unroll 1
  for (int which = 0; which < 3; ++which) {
    pick_bucket(hist_top, k3[which], sel);
    uint32_t prefix = sel[0] << 24, mask = 0xFF000000u;
    int k = static_cast<int>(sel[1]);
    __syncthreads();
#pragma unroll 1
    for (int shift = 16; shift >= 0; shift -= 8) {
      bucket_histogram(x, n, prefix, mask, shift, hist);
      pick_bucket(hist, k, sel);
      prefix |= sel[0] << shift;
      mask |= 255u << shift;
      k = static_cast<int>(sel[1]);
      __syncthreads();
    }
    bits[which] = prefix;
  }
}

// Rows of up to this many keys are staged in shared memory (64 KB).
constexpr int kStagedTokens = 16384;

template <bool kStaged>
__global__ void __launch_bounds__(kThreads) stats_kernel(const StatsArgs a) {
  wait_prior_grid();
  allow_next_grid();
  extern __shared__ float sm[];
  const long row = blockIdx.x;       // (b * Hq + h) * n_q + i
  // [N] each: scores, then p (reference path; staged in shared memory when it
  // fits) and the scores of the MXFP8 Q/K path (three passes read it: from L2)
  float *s_ref = kStaged ? sm : a.s_ref + row * a.N;
  float *s_mx = a.s_mx + row * a.N;
  __shared__ float red[2 * kWarps];
  __shared__ int redi[2 * kWarps];
  __shared__ uint32_t hist[256], hist_top[256], sel[2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the row's two score rows and its statistics (the same in every thread)
  if (!in_bounds(a.ctl, a.s_ref + row * a.N, sizeof(float) * a.N) ||
      !in_bounds(a.ctl, a.s_mx + row * a.N, sizeof(float) * a.N) ||
      !in_bounds(a.ctl, a.stats + row * KVQ_N_STATS, sizeof(float) * KVQ_N_STATS))
    return;
  if (kStaged)
    for (int j = threadIdx.x; j < a.N; j += kThreads) s_ref[j] = a.s_ref[row * a.N + j];
  __syncthreads();

  int am_ref, am_mx;
  block_argmax2(s_ref, s_mx, a.N, red, redi, am_ref, am_mx);
  const float mx_ref = s_ref[am_ref], mx_mx = s_mx[am_mx];
  __syncthreads();  // both maxima read before the rows are overwritten
  // the exponentials, kept in place of the scores
  float l_ref = 0.0f, l_mx = 0.0f;
  for (int j = threadIdx.x; j < a.N; j += kThreads) {
    const float er = expf(s_ref[j] - mx_ref), em = expf(s_mx[j] - mx_mx);
    s_ref[j] = er;
    s_mx[j] = em;
    l_ref += er;
    l_mx += em;
  }
  l_ref = block_sum(l_ref, red);
  l_mx = block_sum(l_mx, red);
  const float inv_ref = 1.0f / l_ref, inv_mx = 1.0f / l_mx;
  // p, structural zeros, entropy, Q/K-path TV
  float zeros = 0.0f, plogp = 0.0f, qk_tv = 0.0f;
  for (int j = threadIdx.x; j < a.N; j += kThreads) {
    const float p = s_ref[j] * inv_ref;
    const float p2 = s_mx[j] * inv_mx;
    s_ref[j] = p;
    zeros += p == 0.0f ? 1.0f : 0.0f;
    plogp += p > 0.0f ? p * logf(p) : 0.0f;
    qk_tv += fabsf(p2 - p);
  }
  zeros = block_sum(zeros, red);
  plogp = block_sum(plogp, red);
  qk_tv = block_sum(qk_tv, red);
  // the MXFP8 probability path: one warp per block of 32 keys, lane = key
  float p_zero = 0.0f, p_tv = 0.0f, p_sum = 0.0f;
  for (int b0 = warp * 32; b0 < a.N; b0 += kThreads) {
    const int j = b0 + lane;
    const float p = j < a.N ? s_ref[j] : 0.0f;
    const float pm = mxfp8_round_warp(p);
    p_zero += (p > 0.0f && pm == 0.0f) ? 1.0f : 0.0f;
    p_tv += fabsf(pm - p);
    p_sum += pm;
  }
  p_zero = block_sum(p_zero, red);
  p_tv = block_sum(p_tv, red);
  p_sum = block_sum(p_sum, red);

  // top-k masses: the k-th largest probability t by a radix select on the
  // float bits (monotone for p >= 0), then mass = sum(p > t) + (k - #(p > t)) t
  const int kk[3] = {(a.N + 99) / 100, (a.N * 5 + 99) / 100, (a.N * 10 + 99) / 100};
  uint32_t tb[3];
  kth_largest_bits3(s_ref, a.N, kk, tb, hist, hist_top, sel);
  float sum[3] = {0.0f, 0.0f, 0.0f}, cnt[3] = {0.0f, 0.0f, 0.0f};
  for (int j = threadIdx.x; j < a.N; j += kThreads) {
    const float p = s_ref[j];
    const uint32_t pb = __float_as_uint(p);
#pragma unroll
    for (int w = 0; w < 3; ++w)
      if (pb > tb[w]) {
        sum[w] += p;
        cnt[w] += 1.0f;
      }
  }
  float top[3];
#pragma unroll 1
  for (int w = 0; w < 3; ++w) {
    const float sw = block_sum(sum[w], red), cw = block_sum(cnt[w], red);
    top[w] = sw + (static_cast<float>(kk[w]) - cw) * __uint_as_float(tb[w]);
  }
  const float t1 = top[0], t5 = top[1], t10 = top[2];

  if (threadIdx.x == 0) {
    float *o = a.stats + row * KVQ_N_STATS;
    const float hnat = -plogp;
    o[KVQ_STAT_ENTROPY] = hnat;
    o[KVQ_STAT_SUPPORT] = expf(hnat) / static_cast<float>(a.N);
    o[KVQ_STAT_TOP1] = t1;
    o[KVQ_STAT_TOP5] = t5;
    o[KVQ_STAT_TOP10] = t10;
    o[KVQ_STAT_ZERO] = zeros / static_cast<float>(a.N);
    o[KVQ_STAT_P_ZERO] = p_zero / static_cast<float>(a.N);
    o[KVQ_STAT_P_TV] = 0.5f * p_tv;
    o[KVQ_STAT_P_SUM] = p_sum;
    o[KVQ_STAT_QK_TV] = 0.5f * qk_tv;
    o[KVQ_STAT_QK_AGREE] = am_ref == am_mx ? 1.0f : 0.0f;
  }
}


}  // namespace

int stats_max_tokens() { return 1 << 20; }

namespace {
size_t round256(size_t x) { return (x + 255) & ~size_t(255); }
}  // namespace

// Key tiles (both paths) and score rows (both paths).
size_t stats_workspace_bytes(const kvq_cache &c, int Hq, int n_q) {
  const size_t tiles = sizeof(float) * static_cast<size_t>(c.batch) * c.kv_heads *
                       ((c.n_tokens + 31) / 32) * 32 * c.head_dim;
  const size_t scores = sizeof(float) * static_cast<size_t>(c.batch) * Hq * n_q * c.n_tokens;
  return 2 * round256(tiles) + 2 * round256(scores);
}

int launch_attend_stats(const kvq_cache &c, const void *q, int q_dtype, int Hq, int n_q,
                        float sm_scale, const float *signs, float *stats, void *ws,
                        const KernelCtl &ctl, cudaStream_t s) {
  const CacheDims d = dims_of(c);
  StatsArgs a;
  a.ctl = ctl;
  a.k_codes = c.k_codes;
  a.k_scales = c.k_scales;
  a.k_window = c.k_window;
  a.k_e8m0 = c.k_window_e8m0;
  a.kwin = c.kwin_dtype;
  a.Hkv = d.Hkv;
  a.N = d.N;
  a.D = d.D;
  a.cut = d.cut;
  a.Gs = d.Gs;
  a.Ws = d.Ws;
  a.Hq = Hq;
  a.group = Hq / d.Hkv;
  a.n_q = n_q;
  a.q = q;
  a.q_dtype = q_dtype;
  a.sm_scale = sm_scale;
  a.signs = signs;
  a.stats = stats;
  a.T = (d.N + 31) / 32;
  const size_t tiles = round256(sizeof(float) * static_cast<size_t>(d.B) * d.Hkv * a.T * 32 * d.D);
  const size_t scores = round256(sizeof(float) * static_cast<size_t>(d.B) * Hq * n_q * d.N);
  uint8_t *w = static_cast<uint8_t *>(ws);
  a.k_ref = reinterpret_cast<float *>(w);
  a.k_mx = reinterpret_cast<float *>(w + tiles);
  a.s_ref = reinterpret_cast<float *>(w + 2 * tiles);
  a.s_mx = reinterpret_cast<float *>(w + 2 * tiles + scores);
  // about a thousand scoring CTAs, each over at least 8 key tiles
  const long row_blocks = static_cast<long>(d.B) * Hq * ((n_q + kRows - 1) / kRows);
  a.key_splits = static_cast<int>(
      std::max<long>(1, std::min<long>({(1024 + row_blocks - 1) / row_blocks, a.T / 8, 65535L})));
  const dim3 kgrid(static_cast<unsigned>(a.T), static_cast<unsigned>(d.B * d.Hkv));
  const size_t ksmem = sizeof(float) * 2 * d.D * 33;
  const dim3 sgrid(static_cast<unsigned>((n_q + kRows - 1) / kRows),
                   static_cast<unsigned>(d.B * Hq), static_cast<unsigned>(a.key_splits));
  const bool staged = d.N <= kStagedTokens;
  const size_t smem = staged ? sizeof(float) * static_cast<size_t>(d.N) : 0;
  const long rows = static_cast<long>(d.B) * Hq * n_q;
  switch (d.D / 32) {
#define KVQ_STATS_CASE(E)                                                                     \
  case E:                                                                                     \
    opt_in_smem(keys_kernel<E>, ksmem);                                            \
    launch_dependent(keys_kernel<E>, kgrid, dim3(kThreads), ksmem, s, a);                     \
    launch_dependent(scores_kernel<E>, sgrid, dim3(kThreads), 0, s, a);                       \
    break;
    KVQ_STATS_CASE(1)
    KVQ_STATS_CASE(2)
    KVQ_STATS_CASE(8)
#undef KVQ_STATS_CASE
    case 4: {  // D = 128: the scores on the tensor cores, 48 query rows per CTA
      opt_in_smem(keys_kernel<4>, ksmem);
      launch_dependent(keys_kernel<4>, kgrid, dim3(kThreads), ksmem, s, a);
      StatsArgs at = a;
      const long tc_blocks = static_cast<long>(d.B) * Hq * ((n_q + kTcRows - 1) / kTcRows);
      at.key_splits = static_cast<int>(std::max<long>(
          1, std::min<long>({(1024 + tc_blocks - 1) / tc_blocks, at.T / 8, 65535L})));
      const dim3 tgrid(static_cast<unsigned>((n_q + kTcRows - 1) / kTcRows),
                       static_cast<unsigned>(d.B * Hq), static_cast<unsigned>(at.key_splits));
      opt_in_smem(scores_tc_kernel, sizeof(ScoresTcSmem));
      launch_dependent(scores_tc_kernel, tgrid, dim3(kThreads), sizeof(ScoresTcSmem), s, at);
      break;
    }
    default:
      return -1;
  }
  if (staged) {
    opt_in_smem(stats_kernel<true>, smem);
    launch_dependent(stats_kernel<true>, dim3(static_cast<unsigned>(rows)), dim3(kThreads), smem,
                     s, a);
  } else {
    launch_dependent(stats_kernel<false>, dim3(static_cast<unsigned>(rows)), dim3(kThreads), 0, s,
                     a);
  }
  return 3;
}

}  // namespace kvq
