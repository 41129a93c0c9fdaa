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
// One CTA (8 warps) per query row. Scores: warp w takes keys w, w + 8, ...;
// lane l holds features l*E .. l*E + E - 1 (E = D / 32) of the key, dequantized
// as the attention kernels read it, and the Hadamard transform runs as E-wide
// in-thread butterflies followed by five lane-exchange stages. Both score rows
// stay in shared memory; the statistics are block reductions over them, and
// the top-k masses come from a bitonic sort of p (padded to a power of two).
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
  int Hkv, N, D, cut, Gs, Ws, Np;
  int Hq, group, n_q;
  const void *q;
  int q_dtype;
  float sm_scale;
  const float *signs;  // [D] +-1, or nullptr: no rotation
  float *stats;        // [rows][KVQ_N_STATS]
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

template <int E>
__global__ void __launch_bounds__(kThreads) stats_kernel(const StatsArgs a) {
  extern __shared__ float sm[];
  float *s_ref = sm;                 // [Np]: scores, then p, then p sorted
  float *s_mx = sm + a.Np;           // [Np]: scores of the MXFP8 Q/K path
  __shared__ float qf[256], qm[256], red[kWarps];
  __shared__ int redi[kWarps];
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

  // scores of both paths, one key per warp at a time
  for (int j = warp; j < a.N; j += kWarps) {
    float x[E];
    float dot = 0.0f;
#pragma unroll
    for (int t = 0; t < E; ++t) {
      x[t] = key_value(a, u, j, lane * E + t);
      dot = fmaf(qf[lane * E + t], x[t], dot);
    }
    if (a.signs) signed_hadamard<E>(x, a.signs, lane);
    mxfp8_round_row<E>(x);
    float dm = 0.0f;
#pragma unroll
    for (int t = 0; t < E; ++t) dm = fmaf(qm[lane * E + t], x[t], dm);
    dot = warp_sum(dot);
    dm = warp_sum(dm);
    if (lane == 0) {
      s_ref[j] = a.sm_scale * dot;
      s_mx[j] = a.sm_scale * dm;
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

  // top-k masses: p sorted ascending (padding -1 goes first), sum the last k
  for (int j = a.N + threadIdx.x; j < a.Np; j += kThreads) s_ref[j] = -1.0f;
  __syncthreads();
  for (int k = 2; k <= a.Np; k <<= 1)
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      for (int i = threadIdx.x; i < a.Np; i += kThreads) {
        const int ixj = i ^ jj;
        if (ixj > i) {
          const float x = s_ref[i], y = s_ref[ixj];
          if (((i & k) == 0) ? (x > y) : (x < y)) {
            s_ref[i] = y;
            s_ref[ixj] = x;
          }
        }
      }
      __syncthreads();
    }
  const int k1 = (a.N + 99) / 100, k5 = (a.N * 5 + 99) / 100, k10 = (a.N * 10 + 99) / 100;
  float t1 = 0.0f, t5 = 0.0f, t10 = 0.0f;
  for (int r = threadIdx.x; r < k10; r += kThreads) {
    const float p = s_ref[a.Np - 1 - r];
    t10 += p;
    t5 += r < k5 ? p : 0.0f;
    t1 += r < k1 ? p : 0.0f;
  }
  t1 = block_sum(t1, red);
  t5 = block_sum(t5, red);
  t10 = block_sum(t10, red);

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

int pow2_at_least(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

}  // namespace

int stats_max_tokens() { return 16384; }

int launch_attend_stats(const kvq_cache &c, const void *q, int q_dtype, int Hq, int n_q,
                        float sm_scale, const float *signs, float *stats, cudaStream_t s) {
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
  a.Np = pow2_at_least(d.N);
  a.Hq = Hq;
  a.group = Hq / d.Hkv;
  a.n_q = n_q;
  a.q = q;
  a.q_dtype = q_dtype;
  a.sm_scale = sm_scale;
  a.signs = signs;
  a.stats = stats;
  const size_t smem = sizeof(float) * 2 * static_cast<size_t>(a.Np);
  const long rows = static_cast<long>(d.B) * Hq * n_q;
  const dim3 grid(static_cast<unsigned>(rows));
  switch (d.D / 32) {
#define KVQ_STATS_CASE(E)                                                                     \
  case E:                                                                                     \
    cudaFuncSetAttribute(stats_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,       \
                         static_cast<int>(smem));                                             \
    stats_kernel<E><<<grid, kThreads, smem, s>>>(a);                                          \
    break;
    KVQ_STATS_CASE(1)
    KVQ_STATS_CASE(2)
    KVQ_STATS_CASE(4)
    KVQ_STATS_CASE(8)
#undef KVQ_STATS_CASE
    default:
      return -1;
  }
  return 1;
}

}  // namespace kvq
