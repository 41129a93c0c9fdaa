// fp32 CUDA-core attention over a packed cache, for any supported shape.
//
// O = softmax(sm_scale * Q K^T) V over every token, K/V dequantized on the
// fly (int4 part) or read from the window, with per-row region masses
// (Catnip study, section "KV Cache 的实际作用": mass per region, all regions
// summing to 1). This is the exact path of the small head-dim workloads of the
// residual-window page (head dim 32, 16 queries, N up to 512) and of any shape
// the specialised kernels do not take.
//
// Layout (head dims above 64, or an MXFP8 K window): one CTA per (16 query
// rows, query head, sequence); 4 warps, 4 rows each. Keys stream through shared memory 32 at a time as fp32; lane j scores
// key j, the warp keeps an online softmax (running max, rescaled sum) and each
// lane owns D/32 output features.
#include <cuda_fp8.h>
#include <math_constants.h>

#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kTileKeys = 32;
constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 4;
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;

struct GenericArgs {
  const uint8_t *k_codes;
  const float *k_scales;
  const uint8_t *v_codes;
  const float *v_scales;
  const void *k_window;
  const void *v_window;
  const uint8_t *k_e8m0;
  int kwin, vwin;
  int Hkv, N, D, R, cut, Gk;
  int Gs, Vs, Ws;  // per-(sequence, head) strides: K groups, V rows, window rows
  int Hq, group, n_q;
  const void *q;
  int q_dtype;
  void *out;
  int out_dtype;
  float *mass;
  float sm_scale;
  Regions reg;
  KernelCtl ctl;
};

// Whether the int4 bytes and scales of element d of token t (unit u) lie in
// the call's buffers (see in_bounds; true outside debug builds).
__device__ __forceinline__ bool elem_ok(const GenericArgs &a, long u, int t, int d, int D) {
  const long g = u * a.Gs + t / kGroup, vr = u * a.Vs + t;
  return in_bounds(a.ctl, a.k_codes + (g * kGroup + t % kGroup) * (D / 2) + d / 2, 1) &&
         in_bounds(a.ctl, a.k_scales + g * D + d, sizeof(float)) &&
         in_bounds(a.ctl, a.v_codes + vr * (D / 2) + d / 2, 1) &&
         in_bounds(a.ctl, a.v_scales + vr * (D / 32) + d / 32, sizeof(float));
}
__device__ __forceinline__ bool win_elem_ok(const GenericArgs &a, long wi, long ei) {
  const size_t kb = a.kwin == KVQ_F32 ? 4 : a.kwin == KVQ_BF16 ? 2 : 1;
  const size_t vb = a.vwin == KVQ_F32 ? 4 : 2;
  return in_bounds(a.ctl, static_cast<const uint8_t *>(a.k_window) + wi * kb, kb) &&
         in_bounds(a.ctl, static_cast<const uint8_t *>(a.v_window) + wi * vb, vb) &&
         (a.kwin != KVQ_MXFP8 || in_bounds(a.ctl, a.k_e8m0 + ei, 1));
}

__device__ __forceinline__ float nib(uint8_t byte, int odd) {
  return static_cast<float>(static_cast<int>(odd ? (byte >> 4) : (byte & 15)) - 8);
}

__device__ __forceinline__ float window_value(const void *w, int dtype, long i) {
  return dtype == KVQ_F32 ? static_cast<const float *>(w)[i]
                          : bf16_to_f32(static_cast<const uint16_t *>(w)[i]);
}

template <int DPL>
__global__ void __launch_bounds__(kWarps * 32) generic_attend_kernel(GenericArgs a) {
  wait_prior_grid();
  allow_next_grid();
  constexpr int D = DPL * 32;
  extern __shared__ float sm[];
  float *Ks = sm;                        // [32][D+1]
  float *Vs = Ks + kTileKeys * (D + 1);  // [32][D]
  float *Qs = Vs + kTileKeys * D;        // [16][D]
  float *Ps = Qs + kRowsPerCta * D;      // [16][32]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y, b = blockIdx.z;
  const long u = static_cast<long>(b) * a.Hkv + h / a.group;
  const int q0 = blockIdx.x * kRowsPerCta;
  const long qbase = (static_cast<long>(b) * a.Hq + h) * a.n_q;

  for (int i = tid; i < kRowsPerCta * D; i += blockDim.x) {
    const int r = i / D, d = i % D;
    float x = 0.0f;
    const long gi = (qbase + q0 + r) * D + d;
    if (q0 + r < a.n_q &&
        in_bounds(a.ctl, static_cast<const uint8_t *>(a.q) + gi * (a.q_dtype == KVQ_F32 ? 4 : 2),
                  a.q_dtype == KVQ_F32 ? 4 : 2)) {
      x = a.q_dtype == KVQ_F32 ? static_cast<const float *>(a.q)[gi]
                               : bf16_to_f32(static_cast<const uint16_t *>(a.q)[gi]);
    }
    Qs[i] = x;
  }
  __syncthreads();
  if (a.kwin == KVQ_MXFP8) {  // Q takes the same MXFP8 rounding as the K window
    for (int r = warp; r < kRowsPerCta; r += kWarps)
      for (int j = 0; j < D / 32; ++j)
        Qs[r * D + 32 * j + lane] = mxfp8_round_warp(Qs[r * D + 32 * j + lane]);
    __syncthreads();
  }

  float m[kRowsPerWarp], l[kRowsPerWarp], rm[kRowsPerWarp], o[kRowsPerWarp][DPL];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    m[r] = -CUDART_INF_F;
    l[r] = 0.0f;
    rm[r] = 0.0f;
#pragma unroll
    for (int k = 0; k < DPL; ++k) o[r][k] = 0.0f;
  }

  for (int t0 = 0; t0 < a.N; t0 += kTileKeys) {
    __syncthreads();
    if (t0 + kTileKeys <= a.cut) {
      // whole tile in the int4 part: branch-free, so all its loads are in flight together
#pragma unroll 4
      for (int i = tid; i < kTileKeys * D; i += blockDim.x) {
        const int j = i / D, d = i % D, t = t0 + j;
        const int g = t / kGroup, r = t % kGroup;
        const long kb = ((u * a.Gs + g) * kGroup + r) * (D / 2) + d / 2;
        const long vb = (u * a.Vs + t) * (D / 2) + d / 2;
        const bool ok = elem_ok(a, u, t, d, D);
        Ks[j * (D + 1) + d] = ok ? nib(a.k_codes[kb], d & 1) * a.k_scales[(u * a.Gs + g) * D + d] : 0.0f;
        Vs[j * D + d] = ok ? nib(a.v_codes[vb], d & 1) * a.v_scales[(u * a.Vs + t) * (D / 32) + d / 32] : 0.0f;
      }
    } else
    for (int i = tid; i < kTileKeys * D; i += blockDim.x) {
      const int j = i / D, d = i % D, t = t0 + j;
      float kv = 0.0f, vv = 0.0f;
      if (t < a.cut && elem_ok(a, u, t, d, D)) {
        const int g = t / kGroup, r = t % kGroup;
        const long kb = ((u * a.Gs + g) * kGroup + r) * (D / 2) + d / 2;
        kv = nib(a.k_codes[kb], d & 1) * a.k_scales[(u * a.Gs + g) * D + d];
        const long vb = (u * a.Vs + t) * (D / 2) + d / 2;
        vv = nib(a.v_codes[vb], d & 1) * a.v_scales[(u * a.Vs + t) * (D / 32) + d / 32];
      } else if (t >= a.cut && t < a.N &&
                 win_elem_ok(a, (u * a.Ws + (t - a.cut)) * D + d,
                             (u * a.Ws + (t - a.cut)) * (D / 32) + d / 32)) {
        const long wi = (u * a.Ws + (t - a.cut)) * D + d;
        if (a.kwin == KVQ_MXFP8)
          kv = mxfp8_value(static_cast<const uint8_t *>(a.k_window)[wi],
                           a.k_e8m0[(u * a.Ws + (t - a.cut)) * (D / 32) + d / 32]);
        else
          kv = window_value(a.k_window, a.kwin, wi);
        vv = window_value(a.v_window, a.vwin, wi);
      }
      Ks[j * (D + 1) + d] = kv;
      Vs[j * D + d] = vv;
    }
    __syncthreads();

    const bool valid = t0 + lane < a.N;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const float *qr = Qs + (warp * kRowsPerWarp + r) * D;
      const float *kr = Ks + lane * (D + 1);
      float s = 0.0f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) s = fmaf(qr[d], kr[d], s);
      s = valid ? s * a.sm_scale : -CUDART_INF_F;
      const float m_new = fmaxf(m[r], warp_max(s));
      const float corr = expf(m[r] - m_new);
      const float p = valid ? expf(s - m_new) : 0.0f;
      l[r] = l[r] * corr + warp_sum(p);
      rm[r] *= corr;
      for (int k = 0; k < a.reg.n; ++k) {
        if (a.reg.b[k] < t0 + kTileKeys && a.reg.b[k + 1] > t0) {
          const int t = t0 + lane;
          const float ps = warp_sum((t >= a.reg.b[k] && t < a.reg.b[k + 1]) ? p : 0.0f);
          if (lane == k) rm[r] += ps;
        }
      }
#pragma unroll
      for (int k = 0; k < DPL; ++k) o[r][k] *= corr;
      m[r] = m_new;
      Ps[(warp * kRowsPerWarp + r) * kTileKeys + lane] = p;
    }
    __syncwarp();
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const float *pr = Ps + (warp * kRowsPerWarp + r) * kTileKeys;
      for (int j = 0; j < kTileKeys; ++j) {
        const float pj = pr[j];
#pragma unroll
        for (int k = 0; k < DPL; ++k) o[r][k] = fmaf(pj, Vs[j * D + lane + 32 * k], o[r][k]);
      }
    }
  }

#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int row = q0 + warp * kRowsPerWarp + r;
    if (row >= a.n_q) continue;
    const float inv = 1.0f / l[r];
    const long ob = (qbase + row) * D;
    if (!in_bounds(a.ctl,
                   static_cast<uint8_t *>(a.out) + ob * (a.out_dtype == KVQ_F32 ? 4 : 2),
                   D * (a.out_dtype == KVQ_F32 ? 4 : 2)) ||
        (a.mass && !in_bounds(a.ctl, a.mass + (qbase + row) * a.reg.n, sizeof(float) * a.reg.n)))
      continue;
#pragma unroll
    for (int k = 0; k < DPL; ++k) {
      const float x = o[r][k] * inv;
      if (a.out_dtype == KVQ_F32)
        static_cast<float *>(a.out)[ob + lane + 32 * k] = x;
      else
        static_cast<__nv_bfloat16 *>(a.out)[ob + lane + 32 * k] = __float2bfloat16_rn(x);
    }
    if (a.mass && lane < a.reg.n) a.mass[(qbase + row) * a.reg.n + lane] = rm[r] * inv;
  }
}

// Head dim 32, fp32 or bf16 windows, at most 4 regions: one CTA of 8 warps
// per query row; warp w takes the 32-key chunks w, w + 8, ..., lane j key
// t0 + j of a chunk, which it dequantizes on use and scores against the
// whole q row; a chunk's max and the running softmax state are shared across
// the warp, each lane keeps partial sums of O and of the region masses. At
// the end O is reduced across lanes through shared memory and the 8 warps'
// states are merged with the log-sum-exp rule.
constexpr int kSmallWarps = 8;  // warps per query row: each takes every 8th block of 32 keys
constexpr int kSmallRegions = 4;

template <int D>
__global__ void __launch_bounds__(kSmallWarps * 32) small_attend_kernel(GenericArgs a, long rows) {
  wait_prior_grid();
  allow_next_grid();
  __shared__ float red[kSmallWarps][32][D + 1];
  __shared__ float wm[kSmallWarps], wl[kSmallWarps], wr[kSmallWarps][kSmallRegions];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long row = blockIdx.x;  // over (b, h, i)
  const long bh = row / a.n_q;
  const int h = static_cast<int>(bh % a.Hq);
  const long b = bh / a.Hq;
  const long u = b * a.Hkv + h / a.group;
  const size_t qe = a.q_dtype == KVQ_F32 ? 4 : 2, oe = a.out_dtype == KVQ_F32 ? 4 : 2;
  // this row's q, output and masses (the same in every thread)
  if (!in_bounds(a.ctl, static_cast<const uint8_t *>(a.q) + row * D * qe, D * qe) ||
      !in_bounds(a.ctl, static_cast<uint8_t *>(a.out) + row * D * oe, D * oe) ||
      (a.mass && !in_bounds(a.ctl, a.mass + row * a.reg.n, sizeof(float) * a.reg.n)))
    return;

  float q[D];
#pragma unroll
  for (int d = 0; d < D; d += 4) {
    if (a.q_dtype == KVQ_F32) {
      const float4 x = *reinterpret_cast<const float4 *>(static_cast<const float *>(a.q) + row * D + d);
      q[d] = x.x; q[d + 1] = x.y; q[d + 2] = x.z; q[d + 3] = x.w;
    } else {
      const uint2 x = *reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(a.q) + row * D + d);
      q[d] = bf16_to_f32(x.x & 0xffffu); q[d + 1] = bf16_to_f32(x.x >> 16);
      q[d + 2] = bf16_to_f32(x.y & 0xffffu); q[d + 3] = bf16_to_f32(x.y >> 16);
    }
  }

  float m = -CUDART_INF_F, l = 0.0f, o[D], rm[kSmallRegions];
#pragma unroll
  for (int d = 0; d < D; ++d) o[d] = 0.0f;
#pragma unroll
  for (int k = 0; k < kSmallRegions; ++k) rm[k] = 0.0f;

  for (int t0 = 32 * warp; t0 < a.N; t0 += 32 * kSmallWarps) {
    const int t = t0 + lane;
    bool in_codes = t < a.cut, in_win = !in_codes && t < a.N;
    if (in_codes) {  // the token's code rows, scale group and V scales
      const long g = u * a.Gs + t / kGroup, vr = u * a.Vs + t;
      in_codes = in_bounds(a.ctl, a.k_codes + (g * kGroup + t % kGroup) * (D / 2), D / 2) &&
                 in_bounds(a.ctl, a.v_codes + vr * (D / 2), D / 2) &&
                 in_bounds(a.ctl, a.v_scales + vr * (D / 32), sizeof(float) * (D / 32)) &&
                 in_bounds(a.ctl, a.k_scales + g * D, sizeof(float) * D);
    } else if (in_win) {  // its window rows
      const long wr = (u * a.Ws + (t - a.cut)) * D;
      const size_t kb = a.kwin == KVQ_F32 ? 4 : 2, vb = a.vwin == KVQ_F32 ? 4 : 2;
      in_win = in_bounds(a.ctl, static_cast<const uint8_t *>(a.k_window) + wr * kb, D * kb) &&
               in_bounds(a.ctl, static_cast<const uint8_t *>(a.v_window) + wr * vb, D * vb);
    }
    // the key's K and V nibbles stay packed until used (8 registers, not 2D)
    uint32_t kw[D / 8], vw[D / 8];
    const float *ks = a.k_scales;
    float vs[D / 32];
    long wi = 0;
    if (in_codes) {
      const int g = t / kGroup, r = t % kGroup;
      const uint4 *kc = reinterpret_cast<const uint4 *>(a.k_codes + ((u * a.Gs + g) * kGroup + r) * (D / 2));
      const uint4 *vc = reinterpret_cast<const uint4 *>(a.v_codes + (u * a.Vs + t) * (D / 2));
#pragma unroll
      for (int w = 0; w < D / 32; ++w) {
        const uint4 x = kc[w], y = vc[w];
        kw[4 * w] = x.x; kw[4 * w + 1] = x.y; kw[4 * w + 2] = x.z; kw[4 * w + 3] = x.w;
        vw[4 * w] = y.x; vw[4 * w + 1] = y.y; vw[4 * w + 2] = y.z; vw[4 * w + 3] = y.w;
        vs[w] = a.v_scales[(u * a.Vs + t) * (D / 32) + w];
      }
      ks = a.k_scales + (u * a.Gs + g) * D;  // the same group for the whole warp: broadcast loads
    } else {
      wi = (u * a.Ws + (t - a.cut)) * D;
    }
    float s0 = 0.0f, s1 = 0.0f;
    if (in_codes) {
#pragma unroll
      for (int d = 0; d < D; d += 2) {
        const uint32_t w = kw[d >> 3];
        s0 = fmaf(q[d], static_cast<float>(static_cast<int>((w >> (4 * (d & 7))) & 15u) - 8) * ks[d], s0);
        s1 = fmaf(q[d + 1],
                  static_cast<float>(static_cast<int>((w >> (4 * ((d + 1) & 7))) & 15u) - 8) * ks[d + 1], s1);
      }
    } else if (in_win) {
#pragma unroll
      for (int d = 0; d < D; d += 2) {
        s0 = fmaf(q[d], window_value(a.k_window, a.kwin, wi + d), s0);
        s1 = fmaf(q[d + 1], window_value(a.k_window, a.kwin, wi + d + 1), s1);
      }
    }
    const bool valid = t < a.N;
    const float sc = valid ? (s0 + s1) * a.sm_scale : -CUDART_INF_F;
    const float m_new = fmaxf(m, warp_max(sc));
    const float p = valid ? expf(sc - m_new) : 0.0f;
    if (m_new != m) {  // warp-uniform
      const float corr = expf(m - m_new);
      l *= corr;
#pragma unroll
      for (int d = 0; d < D; ++d) o[d] *= corr;
#pragma unroll
      for (int k = 0; k < kSmallRegions; ++k) rm[k] *= corr;
      m = m_new;
    }
    l += p;
    if (in_codes) {
#pragma unroll
      for (int d = 0; d < D; ++d) {
        const float v = static_cast<float>(static_cast<int>((vw[d >> 3] >> (4 * (d & 7))) & 15u) - 8) * vs[d / 32];
        o[d] = fmaf(p, v, o[d]);
      }
    } else if (in_win) {
#pragma unroll
      for (int d = 0; d < D; ++d) o[d] = fmaf(p, window_value(a.v_window, a.vwin, wi + d), o[d]);
    }
#pragma unroll
    for (int k = 0; k < kSmallRegions; ++k)
      if (k < a.reg.n) rm[k] += (t >= a.reg.b[k] && t < a.reg.b[k + 1]) ? p : 0.0f;
  }

  // each warp's state: O through shared memory (lane d later sums feature
  // d), l and the region sums over the lanes
#pragma unroll
  for (int d = 0; d < D; ++d) red[warp][lane][d] = o[d];
  const float lw = warp_sum(l);
  float rw[kSmallRegions];
#pragma unroll
  for (int k = 0; k < kSmallRegions; ++k) rw[k] = warp_sum(rm[k]);
  if (lane == 0) {
    wm[warp] = m;
    wl[warp] = lw;
#pragma unroll
    for (int k = 0; k < kSmallRegions; ++k) wr[warp][k] = rw[k];
  }
  __syncthreads();
  // merge the warps (log-sum-exp); a warp that met no key has m = -inf
  float mx = -CUDART_INF_F;
#pragma unroll
  for (int w = 0; w < kSmallWarps; ++w) mx = fmaxf(mx, wm[w]);
  float cw[kSmallWarps], den = 0.0f;
#pragma unroll
  for (int w = 0; w < kSmallWarps; ++w) {
    cw[w] = wm[w] == -CUDART_INF_F ? 0.0f : expf(wm[w] - mx);
    den += cw[w] * wl[w];
  }
  const float inv = 1.0f / den;
  for (int d = threadIdx.x; d < D; d += kSmallWarps * 32) {
    float acc = 0.0f;
#pragma unroll
    for (int w = 0; w < kSmallWarps; ++w) {
      float sw = 0.0f;
#pragma unroll 8
      for (int j = 0; j < 32; ++j) sw += red[w][j][d];
      acc += cw[w] * sw;
    }
    const float x = acc * inv;
    if (a.out_dtype == KVQ_F32)
      static_cast<float *>(a.out)[row * D + d] = x;
    else
      static_cast<__nv_bfloat16 *>(a.out)[row * D + d] = __float2bfloat16_rn(x);
  }
  if (a.mass && threadIdx.x < a.reg.n && threadIdx.x < kSmallRegions) {
    float acc = 0.0f;
#pragma unroll
    for (int w = 0; w < kSmallWarps; ++w) acc += cw[w] * wr[w][threadIdx.x];
    a.mass[row * a.reg.n + threadIdx.x] = acc * inv;
  }
}

template <int DPL>
void launch_dpl(const GenericArgs &a, int B, cudaStream_t s) {
  constexpr int D = DPL * 32;
  const size_t smem = sizeof(float) * (kTileKeys * (D + 1) + kTileKeys * D + kRowsPerCta * D +
                                       kRowsPerCta * kTileKeys);
  opt_in_smem(generic_attend_kernel<DPL>, smem);
  dim3 grid((a.n_q + kRowsPerCta - 1) / kRowsPerCta, a.Hq, B);
  launch_dependent(generic_attend_kernel<DPL>, grid, dim3(kWarps * 32), smem, s, a);
}

}  // namespace

int launch_attend_generic(const kvq_cache &c, const void *q, int q_dtype, int Hq, int n_q,
                          float sm_scale, void *out, int out_dtype, const int32_t *bounds,
                          int n_regions, float *mass, const KernelCtl &ctl, cudaStream_t s) {
  const CacheDims d = dims_of(c);
  GenericArgs a;
  a.k_codes = c.k_codes;
  a.k_scales = c.k_scales;
  a.v_codes = c.v_codes;
  a.v_scales = c.v_scales;
  a.k_window = c.k_window;
  a.v_window = c.v_window;
  a.k_e8m0 = c.k_window_e8m0;
  a.kwin = c.kwin_dtype;
  a.vwin = c.vwin_dtype;
  a.Hkv = d.Hkv;
  a.N = d.N;
  a.D = d.D;
  a.R = d.R;
  a.cut = d.cut;
  a.Gk = d.Gk;
  a.Gs = d.Gs;
  a.Vs = d.Vs;
  a.Ws = d.Ws;
  a.Hq = Hq;
  a.group = Hq / d.Hkv;
  a.n_q = n_q;
  a.q = q;
  a.q_dtype = q_dtype;
  a.out = out;
  a.out_dtype = out_dtype;
  a.mass = mass;
  a.sm_scale = sm_scale;
  a.reg = make_regions(bounds, n_regions);
  a.ctl = ctl;
  if (d.D == 32 && c.kwin_dtype != KVQ_MXFP8 && a.reg.n <= kSmallRegions) {
    const long rows = static_cast<long>(d.B) * Hq * n_q;  // one CTA per query row
    launch_dependent(small_attend_kernel<32>, dim3(static_cast<unsigned>(rows)),
                     dim3(kSmallWarps * 32), 0, s, a, rows);
    return 1;
  }
  switch (d.D / 32) {
    case 1: launch_dpl<1>(a, d.B, s); break;
    case 2: launch_dpl<2>(a, d.B, s); break;
    case 3: launch_dpl<3>(a, d.B, s); break;
    case 4: launch_dpl<4>(a, d.B, s); break;
    case 5: launch_dpl<5>(a, d.B, s); break;
    case 6: launch_dpl<6>(a, d.B, s); break;
    case 7: launch_dpl<7>(a, d.B, s); break;
    default: launch_dpl<8>(a, d.B, s); break;
  }
  return 1;
}

}  // namespace kvq
