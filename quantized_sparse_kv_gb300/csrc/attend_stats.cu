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
// Two kernels. keys_kernel writes, once per (sequence, KV head), every key
// twice to workspace in fp32: as attention reads it (int4 part dequantized,
// window as stored) and on the MXFP8 Q/K path (rotated, rounded); warp per
// key, lane l holding features l*E .. l*E + E - 1 (E = D / 32), the Hadamard
// transform as E-wide in-thread butterflies followed by five lane-exchange
// stages. stats_kernel: one CTA (8 warps) per query row; warp w scores keys
// w, w + 8, ... on both paths from the workspace rows (whole rows per load,
// shuffle reductions); both score rows stay in shared memory, the statistics
// are block reductions over them, and each top-k mass takes the k-th largest
// probability from a radix select over the float bits.

#include <cuda_fp8.h>
#include <math_constants.h>

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
  float *k_ref;        // workspace [units][N][D]: keys as attention reads them
  float *k_mx;         // workspace [units][N][D]: keys on the MXFP8 Q/K path
};


__device__ __forceinline__ float key_value(const StatsArgs &a, long u, int j, int d) {
  if (j < a.cut) {
    const long g = u * a.Gs + (j >> 5);
    const uint8_t byte = a.k_codes[(g * kGroup + (j & 31)) * (a.D / 2) + d / 2];
    const int code = static_cast<int>((d & 1) ? (byte >> 4) : (byte & 15)) - 8;
    return static_cast<float>(code) * a.k_scales[g * a.D + d];
  }
  const long row = u * a.Ws + (j - a.cut);
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
  int e = -127;
  if (amax > 0.0f) {
    int ex;
    frexpf(amax, &ex);
    e = max(-127, min(127, ex - 1 - 8));
  }
#pragma unroll
  for (int t = 0; t < E; ++t) {
    const uint8_t c = static_cast<uint8_t>(
        __nv_cvt_float_to_fp8(ldexpf(x[t], -e), __NV_SATFINITE, __NV_E4M3));
    x[t] = mxfp8_value(c, static_cast<uint8_t>(e + 127));
  }
}

// Both workspace copies of key blockIdx.x * 8 + warp of unit blockIdx.y.
template <int E>
__global__ void __launch_bounds__(kThreads) keys_kernel(const StatsArgs a) {
  wait_prior_grid();
  allow_next_grid();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = blockIdx.x * kWarps + warp;
  if (j >= a.N) return;
  const long u = blockIdx.y;
  const long o = (u * a.N + j) * a.D + lane * E;
  float x[E];
#pragma unroll
  for (int t = 0; t < E; ++t) {
    x[t] = key_value(a, u, j, lane * E + t);
    a.k_ref[o + t] = x[t];
  }
  if (a.signs) signed_hadamard<E>(x, a.signs, lane);
  mxfp8_round_row<E>(x);
#pragma unroll
  for (int t = 0; t < E; ++t) a.k_mx[o + t] = x[t];
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

__device__ __forceinline__ float block_max(float x, float *red) {
  x = warp_max(x);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = x;
  __syncthreads();
  float t = -CUDART_INF_F;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) t = fmaxf(t, red[w]);
  return t;
}

// Index of the first maximum of s[0, n).
__device__ __forceinline__ int block_argmax(const float *s, int n, float *red, int *redi) {
  float best = -CUDART_INF_F;
  int bi = 0x7fffffff;
  for (int j = threadIdx.x; j < n; j += kThreads)
    if (s[j] > best) {
      best = s[j];
      bi = j;
    }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ob > best || (ob == best && oi < bi)) {
      best = ob;
      bi = oi;
    }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) {
    red[warp] = best;
    redi[warp] = bi;
  }
  __syncthreads();
  best = red[0];
  bi = redi[0];
  for (int w = 1; w < kWarps; ++w)
    if (red[w] > best || (red[w] == best && redi[w] < bi)) {
      best = red[w];
      bi = redi[w];
    }
  return bi;
}

// Bits of the k-th largest of x[0, n) (all x >= 0, 1 <= k <= n): four rounds
// of a 256-bucket histogram over the next 8 bits of the keys that still
// match the chosen prefix.
__device__ uint32_t kth_largest_bits(const float *x, int n, int k, uint32_t *hist,
                                     uint32_t *sel) {
  uint32_t prefix = 0u, mask = 0u;
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kThreads) hist[i] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kThreads) {
      const uint32_t b = __float_as_uint(x[i]);
      if ((b & mask) == prefix) atomicAdd(&hist[(b >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t cum = 0u, d = 255u;
      for (;; --d) {
        if (cum + hist[d] >= static_cast<uint32_t>(k) || d == 0u) break;
        cum += hist[d];
      }
      sel[0] = d;
      sel[1] = static_cast<uint32_t>(k) - cum;
    }
    __syncthreads();
    prefix |= sel[0] << shift;
    mask |= 255u << shift;
    k = static_cast<int>(sel[1]);
    __syncthreads();
  }
  return prefix;
}

template <int E>
__global__ void __launch_bounds__(kThreads) stats_kernel(const StatsArgs a) {
  wait_prior_grid();
  allow_next_grid();
  extern __shared__ float sm[];
  float *s_ref = sm;                 // [N]: scores, then p
  float *s_mx = sm + a.N;            // [N]: scores of the MXFP8 Q/K path
  __shared__ __align__(16) float qf[256];
  __shared__ __align__(16) float qm[256];
  __shared__ float red[kWarps];
  __shared__ int redi[kWarps];
  __shared__ uint32_t hist[256], sel[2];
  const long row = blockIdx.x;       // (b * Hq + h) * n_q + i
  const long bh = row / a.n_q;
  const int h = static_cast<int>(bh % a.Hq);
  const long u = (bh / a.Hq) * a.Hkv + h / a.group;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int D = a.D;

  for (int d = threadIdx.x; d < D; d += kThreads)
    qf[d] = a.q_dtype == KVQ_F32 ? static_cast<const float *>(a.q)[row * D + d]
                                 : load_f32(static_cast<const __nv_bfloat16 *>(a.q) + row * D + d);
  __syncthreads();
  if (warp == 0) {
    float x[E];
#pragma unroll
    for (int t = 0; t < E; ++t) x[t] = qf[lane * E + t];
    if (a.signs) signed_hadamard<E>(x, a.signs, lane);
    mxfp8_round_row<E>(x);
#pragma unroll
    for (int t = 0; t < E; ++t) qm[lane * E + t] = x[t];
  }
  __syncthreads();

  // scores of both paths: warp w takes keys w, w + 8, ..., two at a time;
  // lane l reads features l*E .. l*E + E - 1 of each (whole rows per load)
  float qa[E], qb[E];
#pragma unroll
  for (int t = 0; t < E; ++t) {
    qa[t] = qf[lane * E + t];
    qb[t] = qm[lane * E + t];
  }
  for (int j0 = 2 * warp; j0 < a.N; j0 += 2 * kWarps) {
    float dr[2], dm[2];
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const int j = min(j0 + x, a.N - 1);
      const float *kr = a.k_ref + (u * a.N + j) * D + lane * E;
      const float *km = a.k_mx + (u * a.N + j) * D + lane * E;
      dr[x] = dm[x] = 0.0f;
#pragma unroll
      for (int t = 0; t < E; ++t) {
        dr[x] = fmaf(qa[t], __ldg(kr + t), dr[x]);
        dm[x] = fmaf(qb[t], __ldg(km + t), dm[x]);
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1)
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        dr[x] += __shfl_xor_sync(0xffffffffu, dr[x], o);
        dm[x] += __shfl_xor_sync(0xffffffffu, dm[x], o);
      }
    if (lane == 0)
#pragma unroll
      for (int x = 0; x < 2; ++x)
        if (j0 + x < a.N) {
          s_ref[j0 + x] = a.sm_scale * dr[x];
          s_mx[j0 + x] = a.sm_scale * dm[x];
        }
  }
  __syncthreads();

  const int am_ref = block_argmax(s_ref, a.N, red, redi);
  const int am_mx = block_argmax(s_mx, a.N, red, redi);
  float mx_ref = -CUDART_INF_F, mx_mx = -CUDART_INF_F;
  for (int j = threadIdx.x; j < a.N; j += kThreads) {
    mx_ref = fmaxf(mx_ref, s_ref[j]);
    mx_mx = fmaxf(mx_mx, s_mx[j]);
  }
  mx_ref = block_max(mx_ref, red);
  mx_mx = block_max(mx_mx, red);
  float l_ref = 0.0f, l_mx = 0.0f;
  for (int j = threadIdx.x; j < a.N; j += kThreads) {
    l_ref += expf(s_ref[j] - mx_ref);
    l_mx += expf(s_mx[j] - mx_mx);
  }
  l_ref = block_sum(l_ref, red);
  l_mx = block_sum(l_mx, red);
  const float inv_ref = 1.0f / l_ref, inv_mx = 1.0f / l_mx;
  // p, structural zeros, entropy, Q/K-path TV
  float zeros = 0.0f, plogp = 0.0f, qk_tv = 0.0f;
  for (int j = threadIdx.x; j < a.N; j += kThreads) {
    const float p = expf(s_ref[j] - mx_ref) * inv_ref;
    const float p2 = expf(s_mx[j] - mx_mx) * inv_mx;
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
  float top[3];
#pragma unroll 1
  for (int which = 0; which < 3; ++which) {
    const uint32_t t = kth_largest_bits(s_ref, a.N, kk[which], hist, sel);
    const float tv = __uint_as_float(t);
    float sum = 0.0f, cnt = 0.0f;
    for (int j = threadIdx.x; j < a.N; j += kThreads) {
      const float p = s_ref[j];
      if (__float_as_uint(p) > t) {
        sum += p;
        cnt += 1.0f;
      }
    }
    sum = block_sum(sum, red);
    cnt = block_sum(cnt, red);
    top[which] = sum + (static_cast<float>(kk[which]) - cnt) * tv;
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

int stats_max_tokens() { return 16384; }

size_t stats_workspace_bytes(const kvq_cache &c) {
  const size_t one = sizeof(float) * static_cast<size_t>(c.batch) * c.kv_heads * c.n_tokens *
                     c.head_dim;
  return 2 * ((one + 255) & ~size_t(255));
}

int launch_attend_stats(const kvq_cache &c, const void *q, int q_dtype, int Hq, int n_q,
                        float sm_scale, const float *signs, float *stats, void *ws,
                        cudaStream_t s) {
  const CacheDims d = dims_of(c);
  StatsArgs a;
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
  const size_t one = (sizeof(float) * static_cast<size_t>(d.B) * d.Hkv * d.N * d.D + 255) &
                     ~size_t(255);
  a.k_ref = static_cast<float *>(ws);
  a.k_mx = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + one);
  const dim3 kgrid(static_cast<unsigned>((d.N + kWarps - 1) / kWarps),
                   static_cast<unsigned>(d.B * d.Hkv));
  const size_t smem = sizeof(float) * 2 * static_cast<size_t>(d.N);
  const long rows = static_cast<long>(d.B) * Hq * n_q;
  const dim3 grid(static_cast<unsigned>(rows));
  switch (d.D / 32) {
#define KVQ_STATS_CASE(E)                                                                     \
  case E:                                                                                     \
    launch_dependent(keys_kernel<E>, dim3(kgrid), dim3(kThreads), 0, s, a);                   \
    cudaFuncSetAttribute(stats_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,       \
                         static_cast<int>(smem));                                             \
    launch_dependent(stats_kernel<E>, dim3(grid), dim3(kThreads), smem, s, a);                \
    break;
    KVQ_STATS_CASE(1)
    KVQ_STATS_CASE(2)
    KVQ_STATS_CASE(4)
    KVQ_STATS_CASE(8)
#undef KVQ_STATS_CASE
    default:
      return -1;
  }
  return 2;
}

}  // namespace kvq
