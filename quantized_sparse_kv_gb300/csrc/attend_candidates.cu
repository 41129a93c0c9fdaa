// Candidate attention: each query row attends exactly the keys listed for it.
//
// MiniCPM5-2B study (bjdmk.com.cn/news/5855973), section 6 (score -> top-C
// candidates -> exact attention inside the candidates) and section 9 (the
// decode kernel gathers the listed K/V rows and runs an online softmax). Here
// the gathered rows come from the int4 cache (dequantized on the fly) or from
// the float window.
//
// Layout (any head dim): one CTA per (query row, query head, sequence), 8 warps. Warp w
// takes candidates w, w+8, ...; lane l owns features [l*F, (l+1)*F) with
// F = D/32, so one candidate's K codes, K scales, V codes and V scales are
// read as contiguous warp-wide segments. Each warp keeps an online softmax in
// fp32; the 8 warp states are merged through shared memory at the end.
#include <math_constants.h>

#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kWarps = 8;

struct CandArgs {
  const uint8_t *k_codes;
  const float *k_scales;
  const uint8_t *v_codes;
  const float *v_scales;
  const void *k_window;
  const void *v_window;
  int kwin, vwin;
  int Hkv, N, R, cut, Gk;
  int Gs, Vs, Ws;  // per-(sequence, head) strides: K groups, V rows, window rows
  int Hq, group, n_q, C, validate;
  const void *q;
  int q_dtype;
  const int32_t *idx;
  void *out;
  int out_dtype;
  float scale_log2;
  int top_k, Cp;       // exact top-k inside the list (0: attend every listed key); Cp = pow2 >= C
  int block_q, lists_per_head;  // rows [k*block_q, (k+1)*block_q) of a head share list k
  int32_t *selected;   // [rows][top_k] kept positions, or nullptr
  KernelCtl ctl;
};

__device__ __forceinline__ float wval(const void *w, int dtype, long i) {
  return dtype == KVQ_F32 ? static_cast<const float *>(w)[i]
                          : bf16_to_f32(static_cast<const uint16_t *>(w)[i]);
}

template <int F>
__global__ void __launch_bounds__(kWarps * 32) cand_kernel(const CandArgs a) {
  wait_prior_grid();
  allow_next_grid();
  constexpr int D = F * 32;
  __shared__ float red_o[kWarps][D];
  __shared__ float red_m[kWarps], red_l[kWarps];
  extern __shared__ int32_t list[];  // the row's C indices (validate only)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const long u = static_cast<long>(b) * a.Hkv + h / a.group;
  const long row = (static_cast<long>(b) * a.Hq + h) * a.n_q + i;
  const int32_t *cand =
      a.idx + ((static_cast<long>(b) * a.Hq + h) * a.lists_per_head + i / a.block_q) * a.C;
  const int d0 = lane * F;

  float q[F];
#pragma unroll
  for (int k = 0; k < F; ++k) {
    const long gi = row * D + d0 + k;
    q[k] = (a.q_dtype == KVQ_F32 ? static_cast<const float *>(a.q)[gi]
                                 : bf16_to_f32(static_cast<const uint16_t *>(a.q)[gi])) *
           a.scale_log2;
  }

  if (a.validate) {
    for (int j = threadIdx.x; j < a.C; j += blockDim.x) list[j] = cand[j];
    __syncthreads();
    for (int j = threadIdx.x; j < a.C; j += blockDim.x) {
      const int32_t x = list[j];
      for (int jj = 0; jj < j; ++jj)
        if (list[jj] == x) {
          flag_error(a.ctl, KVQ_DEV_DUP);
          break;
        }
    }
  }

  float m = -CUDART_INF_F, l = 0.0f, o[F];
#pragma unroll
  for (int k = 0; k < F; ++k) o[k] = 0.0f;

  for (int c = warp; c < a.C; c += kWarps) {
    const int t = cand[c];
    if (t < 0 || t >= a.N) {
      if (lane == 0) flag_error(a.ctl, KVQ_DEV_INDEX);
      continue;
    }
    float kv[F], vv[F];
    if (t < a.cut) {
      const int g = t / kGroup, r = t % kGroup;
      const uint8_t *kc = a.k_codes + ((u * a.Gs + g) * kGroup + r) * (D / 2);
      const float *ks = a.k_scales + (u * a.Gs + g) * D;
      const uint8_t *vc = a.v_codes + (u * a.Vs + t) * (D / 2);
      const float *vs = a.v_scales + (u * a.Vs + t) * (D / 32);
#pragma unroll
      for (int k = 0; k < F; ++k) {
        const int d = d0 + k;
        const uint8_t kb = kc[d >> 1], vb = vc[d >> 1];
        kv[k] = static_cast<float>(static_cast<int>((d & 1) ? (kb >> 4) : (kb & 15)) - 8) * ks[d];
        vv[k] = static_cast<float>(static_cast<int>((d & 1) ? (vb >> 4) : (vb & 15)) - 8) *
                vs[d / 32];
      }
    } else {
      const long wr = u * a.Ws + (t - a.cut);
#pragma unroll
      for (int k = 0; k < F; ++k) {
        const long wi = wr * D + d0 + k;
        kv[k] = wval(a.k_window, a.kwin, wi);
        vv[k] = wval(a.v_window, a.vwin, wi);
      }
    }
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < F; ++k) s = fmaf(q[k], kv[k], s);
    s = warp_sum(s);
    const float mn = fmaxf(m, s);
    const float corr = exp2f(m - mn), p = exp2f(s - mn);
    l = l * corr + p;
#pragma unroll
    for (int k = 0; k < F; ++k) o[k] = o[k] * corr + p * vv[k];
    m = mn;
  }

  if (lane == 0) {
    red_m[warp] = m;
    red_l[warp] = l;
  }
#pragma unroll
  for (int k = 0; k < F; ++k) red_o[warp][d0 + k] = o[k];
  __syncthreads();
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float mx = -CUDART_INF_F;
    for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, red_m[w]);
    float acc = 0.0f, ls = 0.0f;
    for (int w = 0; w < kWarps; ++w) {
      if (red_m[w] == -CUDART_INF_F) continue;
      const float c = exp2f(red_m[w] - mx);
      acc += c * red_o[w][d];
      ls += c * red_l[w];
    }
    const float x = acc / ls;
    if (a.out_dtype == KVQ_F32)
      static_cast<float *>(a.out)[row * D + d] = x;
    else
      static_cast<__nv_bfloat16 *>(a.out)[row * D + d] = __float2bfloat16_rn(x);
  }
}

// Head dim 128 (4 features per lane): the row's index list is staged in shared
// memory, and each warp gathers kUnroll candidates per step with independent
// vector loads, so many rows are in flight per SM; the kUnroll dot products
// are reduced together and enter the online softmax as one update.
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kWarps * 32) cand128_kernel(const CandArgs a) {
  wait_prior_grid();
  allow_next_grid();
  constexpr int D = 128;
  __shared__ float red_o[kWarps][D];
  __shared__ float red_m[kWarps], red_l[kWarps];
  extern __shared__ int32_t list[];  // the row's C indices

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const long u = static_cast<long>(b) * a.Hkv + h / a.group;
  const long row = (static_cast<long>(b) * a.Hq + h) * a.n_q + i;
  const int32_t *cand =
      a.idx + ((static_cast<long>(b) * a.Hq + h) * a.lists_per_head + i / a.block_q) * a.C;
  for (int j = threadIdx.x; j < a.C; j += blockDim.x) list[j] = cand[j];

  float q[4];
  if (a.q_dtype == KVQ_F32) {
    const float4 x = reinterpret_cast<const float4 *>(static_cast<const float *>(a.q) + row * D)[lane];
    q[0] = x.x; q[1] = x.y; q[2] = x.z; q[3] = x.w;
  } else {
    const uint2 x = reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(a.q) + row * D)[lane];
    q[0] = bf16_to_f32(x.x & 0xffffu); q[1] = bf16_to_f32(x.x >> 16);
    q[2] = bf16_to_f32(x.y & 0xffffu); q[3] = bf16_to_f32(x.y >> 16);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) q[k] *= a.scale_log2;
  __syncthreads();

  if (a.validate) {
    for (int j = threadIdx.x; j < a.C; j += blockDim.x) {
      const int32_t x = list[j];
      for (int jj = 0; jj < j; ++jj)
        if (list[jj] == x) {
          flag_error(a.ctl, KVQ_DEV_DUP);
          break;
        }
    }
  }

  const uint8_t *kc_u = a.k_codes + u * a.Gs * kGroup * (D / 2);
  const float *ks_u = a.k_scales + u * a.Gs * D;
  const uint8_t *vc_u = a.v_codes + u * a.Vs * (D / 2);
  const float *vs_u = a.v_scales + u * a.Vs * (D / 32);
  const long wbase = u * a.Ws;

  float m = -CUDART_INF_F, l = 0.0f, o[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  const int tq_max = a.cut > 0 ? a.cut - 1 : 0;
  for (int c0 = warp * kUnroll; c0 < a.C; c0 += kWarps * kUnroll) {
    int tk[kUnroll];
    bool ok[kUnroll];
    bool any_win = false;
#pragma unroll
    for (int x = 0; x < kUnroll; ++x) {
      const int c = c0 + x;
      tk[x] = c < a.C ? list[c] : -1;
      ok[x] = c < a.C && tk[x] >= 0 && tk[x] < a.N;
      if (c < a.C && !ok[x] && lane == 0) flag_error(a.ctl, KVQ_DEV_INDEX);
      any_win |= ok[x] && tk[x] >= a.cut;
    }
    // int4 rows for every slot, branch-free: out-of-range or window slots read
    // a clamped, valid int4 row that is overwritten or masked below, so all
    // 4 x kUnroll loads are in flight together
    uint32_t kb[kUnroll], vb[kUnroll];
    float4 ks[kUnroll];
    float vs[kUnroll];
    if (a.cut > 0) {
#pragma unroll
      for (int x = 0; x < kUnroll; ++x) {
        const int t = min(max(tk[x], 0), tq_max);
        const int g = t / kGroup, r = t % kGroup;
        kb[x] = reinterpret_cast<const uint16_t *>(kc_u + (static_cast<long>(g) * kGroup + r) * (D / 2))[lane];
        ks[x] = reinterpret_cast<const float4 *>(ks_u + static_cast<long>(g) * D)[lane];
        vb[x] = reinterpret_cast<const uint16_t *>(vc_u + static_cast<long>(t) * (D / 2))[lane];
        vs[x] = vs_u[static_cast<long>(t) * (D / 32) + (lane >> 3)];
      }
    }
    float kv[kUnroll][4], vv[kUnroll][4], s[kUnroll];
#pragma unroll
    for (int x = 0; x < kUnroll; ++x) {
      if (a.cut > 0) {
        kv[x][0] = static_cast<float>(static_cast<int>(kb[x] & 15) - 8) * ks[x].x;
        kv[x][1] = static_cast<float>(static_cast<int>((kb[x] >> 4) & 15) - 8) * ks[x].y;
        kv[x][2] = static_cast<float>(static_cast<int>((kb[x] >> 8) & 15) - 8) * ks[x].z;
        kv[x][3] = static_cast<float>(static_cast<int>((kb[x] >> 12) & 15) - 8) * ks[x].w;
        vv[x][0] = static_cast<float>(static_cast<int>(vb[x] & 15) - 8) * vs[x];
        vv[x][1] = static_cast<float>(static_cast<int>((vb[x] >> 4) & 15) - 8) * vs[x];
        vv[x][2] = static_cast<float>(static_cast<int>((vb[x] >> 8) & 15) - 8) * vs[x];
        vv[x][3] = static_cast<float>(static_cast<int>((vb[x] >> 12) & 15) - 8) * vs[x];
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) kv[x][k] = vv[x][k] = 0.0f;
      }
    }
    if (any_win) {  // rare: rows of the float window
#pragma unroll
      for (int x = 0; x < kUnroll; ++x) {
        if (!(ok[x] && tk[x] >= a.cut)) continue;
        const long wr = (wbase + (tk[x] - a.cut)) * D;
        if (a.kwin == KVQ_F32) {
          const float4 kf = reinterpret_cast<const float4 *>(static_cast<const float *>(a.k_window) + wr)[lane];
          kv[x][0] = kf.x; kv[x][1] = kf.y; kv[x][2] = kf.z; kv[x][3] = kf.w;
        } else {
          const uint2 kw = reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(a.k_window) + wr)[lane];
          kv[x][0] = bf16_to_f32(kw.x & 0xffffu); kv[x][1] = bf16_to_f32(kw.x >> 16);
          kv[x][2] = bf16_to_f32(kw.y & 0xffffu); kv[x][3] = bf16_to_f32(kw.y >> 16);
        }
        if (a.vwin == KVQ_F32) {
          const float4 vf = reinterpret_cast<const float4 *>(static_cast<const float *>(a.v_window) + wr)[lane];
          vv[x][0] = vf.x; vv[x][1] = vf.y; vv[x][2] = vf.z; vv[x][3] = vf.w;
        } else {
          const uint2 vw = reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(a.v_window) + wr)[lane];
          vv[x][0] = bf16_to_f32(vw.x & 0xffffu); vv[x][1] = bf16_to_f32(vw.x >> 16);
          vv[x][2] = bf16_to_f32(vw.y & 0xffffu); vv[x][3] = bf16_to_f32(vw.y >> 16);
        }
      }
    }
#pragma unroll
    for (int x = 0; x < kUnroll; ++x)
      s[x] = q[0] * kv[x][0] + q[1] * kv[x][1] + q[2] * kv[x][2] + q[3] * kv[x][3];
#pragma unroll
    for (int off = 16; off; off >>= 1)
#pragma unroll
      for (int x = 0; x < kUnroll; ++x) s[x] += __shfl_xor_sync(0xffffffffu, s[x], off);
    float mn = m;
#pragma unroll
    for (int x = 0; x < kUnroll; ++x)
      if (ok[x]) mn = fmaxf(mn, s[x]);
    if (mn == -CUDART_INF_F) continue;  // nothing valid in this step
    const float corr = exp2f(m - mn);
    l *= corr;
#pragma unroll
    for (int k = 0; k < 4; ++k) o[k] *= corr;
#pragma unroll
    for (int x = 0; x < kUnroll; ++x) {
      const float p = ok[x] ? exp2f(s[x] - mn) : 0.0f;
      l += p;
#pragma unroll
      for (int k = 0; k < 4; ++k) o[k] = fmaf(p, vv[x][k], o[k]);
    }
    m = mn;
  }

  if (lane == 0) {
    red_m[warp] = m;
    red_l[warp] = l;
  }
  reinterpret_cast<float4 *>(red_o[warp])[lane] = make_float4(o[0], o[1], o[2], o[3]);
  __syncthreads();
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float mx = -CUDART_INF_F;
    for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, red_m[w]);
    float acc = 0.0f, ls = 0.0f;
    for (int w = 0; w < kWarps; ++w) {
      if (red_m[w] == -CUDART_INF_F) continue;
      const float c = exp2f(red_m[w] - mx);
      acc += c * red_o[w][d];
      ls += c * red_l[w];
    }
    const float x = acc / ls;
    if (a.out_dtype == KVQ_F32)
      static_cast<float *>(a.out)[row * D + d] = x;
    else
      static_cast<__nv_bfloat16 *>(a.out)[row * D + d] = __float2bfloat16_rn(x);
  }
}

template <int F>
void launch_f(const CandArgs &a, int B, cudaStream_t s) {
  dim3 grid(a.n_q, a.Hq, B);
  const size_t smem = a.validate ? sizeof(int32_t) * a.C : 0;
  launch_dependent(cand_kernel<F>, grid, dim3(kWarps * 32), smem, s, a);
}

// Exact top-k inside the candidates (MiniCPM study, section 6: the predictor's
// top-C list, then the true top-32 inside it by exact score). One CTA per
// (query row, query head, sequence): warp w scores candidates w, w + 8, ...
// into shared memory (lane l owns features l*F ..), the (score, list
// position) pairs are sorted by a bitonic sort (higher score first, ties to
// the position listed first), and the first top_k keys are attended: warp w
// takes kept keys w, w + 8, ... against the common maximum (the first sorted
// score), and the warps' sums meet in shared memory.
template <int F>
__global__ void __launch_bounds__(kWarps * 32) cand_topk_kernel(const CandArgs a) {
  wait_prior_grid();
  allow_next_grid();
  constexpr int D = F * 32;
  __shared__ float red_o[kWarps][D];
  __shared__ float red_l[kWarps];
  extern __shared__ float sc[];                       // [Cp] scores
  int32_t *pos = reinterpret_cast<int32_t *>(sc + a.Cp);  // [Cp] list positions
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const long u = static_cast<long>(b) * a.Hkv + h / a.group;
  const long row = (static_cast<long>(b) * a.Hq + h) * a.n_q + i;
  const int32_t *cand =
      a.idx + ((static_cast<long>(b) * a.Hq + h) * a.lists_per_head + i / a.block_q) * a.C;
  const int d0 = lane * F;

  float q[F];
#pragma unroll
  for (int k = 0; k < F; ++k) {
    const long gi = row * D + d0 + k;
    q[k] = (a.q_dtype == KVQ_F32 ? static_cast<const float *>(a.q)[gi]
                                 : bf16_to_f32(static_cast<const uint16_t *>(a.q)[gi])) *
           a.scale_log2;
  }
  for (int c = a.C + threadIdx.x; c < a.Cp; c += blockDim.x) {
    sc[c] = -CUDART_INF_F;
    pos[c] = 0x7fffffff;
  }
  // scores of every listed key (an index outside [0, N) scores -inf)
  for (int c = warp; c < a.C; c += kWarps) {
    const int t = cand[c];
    float s = -CUDART_INF_F;
    if (t >= 0 && t < a.N) {
      float part = 0.0f;
      if (t < a.cut) {
        const int g = t / kGroup, r = t % kGroup;
        const uint8_t *kc = a.k_codes + ((u * a.Gs + g) * kGroup + r) * (D / 2);
        const float *ks = a.k_scales + (u * a.Gs + g) * D;
#pragma unroll
        for (int k = 0; k < F; ++k) {
          const int d = d0 + k;
          const uint8_t kb = kc[d >> 1];
          part = fmaf(q[k],
                      static_cast<float>(static_cast<int>((d & 1) ? (kb >> 4) : (kb & 15)) - 8) *
                          ks[d],
                      part);
        }
      } else {
        const long wr = u * a.Ws + (t - a.cut);
#pragma unroll
        for (int k = 0; k < F; ++k) part = fmaf(q[k], wval(a.k_window, a.kwin, wr * D + d0 + k), part);
      }
      s = warp_sum(part);
    } else if (lane == 0) {
      flag_error(a.ctl, KVQ_DEV_INDEX);
    }
    if (lane == 0) {
      sc[c] = s;
      pos[c] = c;
    }
  }
  __syncthreads();
  // sort: element x before y when its score is higher, or equal and listed first
  for (int k = 2; k <= a.Cp; k <<= 1)
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      for (int e = threadIdx.x; e < a.Cp; e += blockDim.x) {
        const int f = e ^ jj;
        if (f > e) {
          const float se = sc[e], sf = sc[f];
          const int pe = pos[e], pf = pos[f];
          const bool f_first = sf > se || (sf == se && pf < pe);
          if (((e & k) == 0) == f_first) {
            sc[e] = sf;
            sc[f] = se;
            pos[e] = pf;
            pos[f] = pe;
          }
        }
      }
      __syncthreads();
    }
  const int kk = min(a.top_k, a.C);
  const float mx = sc[0];
  float l = 0.0f, o[F];
#pragma unroll
  for (int k = 0; k < F; ++k) o[k] = 0.0f;
  for (int r = warp; r < kk; r += kWarps) {
    if (sc[r] == -CUDART_INF_F) break;  // fewer valid keys than top_k
    const int t = cand[pos[r]];
    const float p = exp2f(sc[r] - mx);
    l += p;
    if (t < a.cut) {
      const uint8_t *vc = a.v_codes + (u * a.Vs + t) * (D / 2);
      const float *vs = a.v_scales + (u * a.Vs + t) * (D / 32);
#pragma unroll
      for (int k = 0; k < F; ++k) {
        const int d = d0 + k;
        const uint8_t vb = vc[d >> 1];
        o[k] = fmaf(p, static_cast<float>(static_cast<int>((d & 1) ? (vb >> 4) : (vb & 15)) - 8) *
                           vs[d / 32], o[k]);
      }
    } else {
      const long wr = u * a.Ws + (t - a.cut);
#pragma unroll
      for (int k = 0; k < F; ++k) o[k] = fmaf(p, wval(a.v_window, a.vwin, wr * D + d0 + k), o[k]);
    }
  }
  if (lane == 0) red_l[warp] = l;
#pragma unroll
  for (int k = 0; k < F; ++k) red_o[warp][d0 + k] = o[k];
  if (a.selected)
    for (int r = threadIdx.x; r < a.top_k; r += blockDim.x)
      a.selected[row * a.top_k + r] =
          (r < kk && sc[r] != -CUDART_INF_F) ? cand[pos[r]] : -1;
  __syncthreads();
  float ls = 0.0f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) ls += red_l[w];
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float acc = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) acc += red_o[w][d];
    const float x = acc / ls;
    if (a.out_dtype == KVQ_F32)
      static_cast<float *>(a.out)[row * D + d] = x;
    else
      static_cast<__nv_bfloat16 *>(a.out)[row * D + d] = __float2bfloat16_rn(x);
  }
}

}  // namespace

int candidates_topk_max() { return 4096; }

int launch_attend_candidates(const kvq_cache &c, const void *q, int q_dtype, int Hq, int n_q,
                             const int32_t *idx, int n_cand, int validate, float scale_log2,
                             void *out, int out_dtype, const KernelCtl &ctl, cudaStream_t s,
                             int top_k, int32_t *selected, int block_q) {
  const CacheDims d = dims_of(c);
  CandArgs a;
  a.k_codes = c.k_codes;
  a.k_scales = c.k_scales;
  a.v_codes = c.v_codes;
  a.v_scales = c.v_scales;
  a.k_window = c.k_window;
  a.v_window = c.v_window;
  a.kwin = c.kwin_dtype;
  a.vwin = c.vwin_dtype;
  a.Hkv = d.Hkv;
  a.N = d.N;
  a.R = d.R;
  a.cut = d.cut;
  a.Gk = d.Gk;
  a.Gs = d.Gs;
  a.Vs = d.Vs;
  a.Ws = d.Ws;
  a.Hq = Hq;
  a.group = Hq / d.Hkv;
  a.n_q = n_q;
  a.C = n_cand;
  a.validate = validate;
  a.q = q;
  a.q_dtype = q_dtype;
  a.idx = idx;
  a.out = out;
  a.out_dtype = out_dtype;
  a.scale_log2 = scale_log2;
  a.ctl = ctl;
  a.top_k = top_k;
  a.selected = selected;
  a.block_q = block_q;
  a.lists_per_head = (n_q + block_q - 1) / block_q;
  a.Cp = 1;
  while (a.Cp < n_cand) a.Cp <<= 1;
  if (top_k > 0) {
    const size_t smem = static_cast<size_t>(a.Cp) * (sizeof(float) + sizeof(int32_t));
    const dim3 grid(n_q, Hq, d.B);
    switch (d.D / 32) {
#define KVQ_TOPK_CASE(F)                                                                      \
  case F:                                                                                     \
    cudaFuncSetAttribute(cand_topk_kernel<F>, cudaFuncAttributeMaxDynamicSharedMemorySize,   \
                         static_cast<int>(smem));                                             \
    launch_dependent(cand_topk_kernel<F>, grid, dim3(kWarps * 32), smem, s, a);               \
    break;
      KVQ_TOPK_CASE(1)
      KVQ_TOPK_CASE(2)
      KVQ_TOPK_CASE(3)
      KVQ_TOPK_CASE(4)
      KVQ_TOPK_CASE(5)
      KVQ_TOPK_CASE(6)
      KVQ_TOPK_CASE(7)
      KVQ_TOPK_CASE(8)
#undef KVQ_TOPK_CASE
      default:
        return -1;
    }
    return 1;
  }
  if (d.D == 128) {
    launch_dependent(cand128_kernel, dim3(n_q, Hq, d.B), dim3(kWarps * 32),
                     sizeof(int32_t) * n_cand, s, a);
    return 1;
  }
  switch (d.D / 32) {
    case 1: launch_f<1>(a, d.B, s); break;
    case 2: launch_f<2>(a, d.B, s); break;
    case 3: launch_f<3>(a, d.B, s); break;
    case 4: launch_f<4>(a, d.B, s); break;
    case 5: launch_f<5>(a, d.B, s); break;
    case 6: launch_f<6>(a, d.B, s); break;
    case 7: launch_f<7>(a, d.B, s); break;
    default: launch_f<8>(a, d.B, s); break;
  }
  return 1;
}

}  // namespace kvq
