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

#include <algorithm>

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

// Whether the rows a listed key t of unit u reads (int4: its K code row, K
// scale group, V code row and V scales; window: its K and V rows) lie inside
// the call's buffers (see in_bounds; always true outside debug builds).
__device__ __forceinline__ bool cand_row_ok(const CandArgs &a, long u, int t, int D) {
  if (t < a.cut) {
    const long g = u * a.Gs + t / kGroup, vr = u * a.Vs + t;
    return in_bounds(a.ctl, a.k_codes + (g * kGroup + t % kGroup) * (D / 2), D / 2) &&
           in_bounds(a.ctl, a.k_scales + g * D, sizeof(float) * D) &&
           in_bounds(a.ctl, a.v_codes + vr * (D / 2), D / 2) &&
           in_bounds(a.ctl, a.v_scales + vr * (D / 32), sizeof(float) * (D / 32));
  }
  const long wr = (u * a.Ws + (t - a.cut)) * D;
  const size_t kb = a.kwin == KVQ_F32 ? 4 : 2, vb = a.vwin == KVQ_F32 ? 4 : 2;
  return in_bounds(a.ctl, static_cast<const uint8_t *>(a.k_window) + wr * kb, kb * D) &&
         in_bounds(a.ctl, static_cast<const uint8_t *>(a.v_window) + wr * vb, vb * D);
}

// The row's list, q row and output row inside the call's buffers.
__device__ __forceinline__ bool cand_io_ok(const CandArgs &a, const int32_t *cand, long row,
                                           int D) {
  const size_t qb = a.q_dtype == KVQ_F32 ? 4 : 2, ob = a.out_dtype == KVQ_F32 ? 4 : 2;
  return in_bounds(a.ctl, cand, sizeof(int32_t) * a.C) &&
         in_bounds(a.ctl, static_cast<const uint8_t *>(a.q) + row * D * qb, qb * D) &&
         in_bounds(a.ctl, static_cast<const uint8_t *>(a.out) + row * D * ob, ob * D);
}

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
  if (!cand_io_ok(a, cand, row, D)) return;  // the same in every thread

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
    if (!cand_row_ok(a, u, t, D)) continue;
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
  if (!cand_io_ok(a, cand, row, D)) return;  // the same in every thread
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
      ok[x] = ok[x] && cand_row_ok(a, u, tk[x], D);
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
        if (!cand_row_ok(a, u, t, D)) {  // debug builds only: the slot reads nothing
          kb[x] = vb[x] = 0u;
          ks[x] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          vs[x] = 0.0f;
          continue;
        }
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
  // the row's list, q, output and selected rows (the same in every thread)
  if (!cand_io_ok(a, cand, row, D) ||
      (a.selected && !in_bounds(a.ctl, a.selected + row * a.top_k, sizeof(int32_t) * a.top_k)))
    return;

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
    if (t >= 0 && t < a.N && cand_row_ok(a, u, t, D)) {
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
    } else if (lane == 0 && (t < 0 || t >= a.N)) {
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

// ------------------------------------------------------------------ union of a KV head's lists
// MiniCPM5-2B study, section 9: the decode kernel gathers only the listed K/V
// rows. With GQA the 8 query heads of a KV head list mostly different
// positions but share some (every list holds the sink positions) and share
// int4 K-scale groups. Three launches:
//   cand_union_build_kernel   the union of the 8 lists of each (sequence, KV
//                             head), one CTA per 32,768 positions: each listed
//                             position marks its head's bit in a byte per
//                             position, and the marked positions are written,
//                             in increasing order, with their head bits;
//   cand_union_kernel         the union split into equal pieces: each CTA
//                             reads the K/V rows of its piece once (each
//                             distinct row once per KV head; a K-scale group
//                             read by several rows is found in L2), scores
//                             them for all 8 heads on the tensor cores
//                             (tokens x heads), each head masked to the keys
//                             it listed, and leaves one partial (m, l, O) per
//                             head;
//   cand_union_combine_kernel the log-sum-exp merge of a KV head's pieces.
constexpr int kUT = 32;          // rows per round
constexpr int kURaw = 3;         // rounds of raw bytes in flight per loader thread
constexpr int kULoaders = 4;     // warps 2-5: asynchronous copies and bf16 conversion
constexpr int kUMma = 2;         // warps 0-1: one 16-row m-tile of each round each
constexpr int kUThreads = 32 * (kULoaders + kUMma);
constexpr int kUMaxList = 4096;  // bound of 8 x C, the union's size
constexpr int kUPart = 132;      // floats per (piece, head) partial: O[128], m, l, padding
constexpr int kUMaxPiece = 1024; // rows of one piece (staged in shared memory)
constexpr int kUW = 32768;       // positions per build slice: one mask byte each
constexpr int kUMaxSlices = 64;  // build slices per KV head (contexts up to 2 M positions)
constexpr int kUBuild = 512;     // threads of a build CTA

struct UnionArgs {
  const uint8_t *k_codes;
  const float *k_scales;
  const uint8_t *v_codes;
  const float *v_scales;
  const uint16_t *k_window, *v_window;  // bf16
  int Hkv, N, cut, Gs, Vs, Ws;
  int C, validate;
  const uint16_t *q;      // bf16 [B][Hkv * 8][128]
  const int32_t *idx;     // [B][Hkv * 8][C]
  int pieces;             // pieces per (sequence, KV head)
  int slices;             // build slices per (sequence, KV head)
  float scale_log2;
  int32_t *list_pos;      // [units][slices][8 C] positions of a slice (the first count)
  uint8_t *list_heads;    // [units][slices][8 C] their head bits
  int32_t *count;         // [units][slices]
  float *partials;        // [units][pieces][8][kUPart]
  void *out;
  int out_dtype;
  KernelCtl ctl;
};

// Number of nonzero bytes of w.
__device__ __forceinline__ int nonzero_bytes(uint32_t w) {
  return __popc((((w & 0x7f7f7f7fu) + 0x7f7f7f7fu) | w) & 0x80808080u);
}

struct __align__(16) BuildSmem {
  uint32_t mask[kUW / 4];        // byte j: head bits of position lo + j
  uint32_t summary[kUW / 512];   // bit c: 16-position chunk c is not empty
  uint16_t chunks[kUW / 16];     // the non-empty chunks, increasing
  int wsum[kUBuild / 32];
  int n_chunks;
};

// ---- union of the 8 lists of one (sequence, KV head), positions [lo, lo + kUW)
__global__ void __launch_bounds__(kUBuild) cand_union_build_kernel(const UnionArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  BuildSmem &sm = *reinterpret_cast<BuildSmem *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slice = blockIdx.x, u = blockIdx.y;
  const int lo = slice * kUW, hi = min(a.N, lo + kUW);
  const int n16 = (hi - lo + 15) >> 4;  // 16-position chunks of the slice
  allow_next_grid();
  for (int i = tid; i < n16; i += kUBuild)
    reinterpret_cast<uint4 *>(sm.mask)[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int i = tid; i < kUW / 512; i += kUBuild) sm.summary[i] = 0u;
  wait_prior_grid();
  __syncthreads();
  // ---- mark; the 8 lists are contiguous (8 C entries), read 4 entries per
  // 16-byte load when C is a multiple of 4, all of a thread's loads issued first
  const int b = u / a.Hkv, kvh = u % a.Hkv;
  const int32_t *lists = a.idx + (static_cast<long>(b) * a.Hkv * 8 + kvh * 8) * a.C;
  const int entries = 8 * a.C;
  const long lbase = (static_cast<long>(u) * a.slices + slice) * entries;
  // the 8 lists and this slice's outputs (the same in every thread)
  const bool io_ok = in_bounds(a.ctl, lists, sizeof(int32_t) * entries) &&
                     in_bounds(a.ctl, a.list_pos + lbase, sizeof(int32_t) * entries) &&
                     in_bounds(a.ctl, a.list_heads + lbase, entries) &&
                     in_bounds(a.ctl, a.count + static_cast<long>(u) * a.slices + slice, 4);
  if (!io_ok) return;
  auto mark = [&](int e, int t) {
    if (t < 0 || t >= a.N) {
      if (slice == 0) flag_error(a.ctl, KVQ_DEV_INDEX);
      return;
    }
    if (t < lo || t >= hi) return;
    const int j = t - lo;
    const uint32_t bit = 1u << (8 * (j & 3) + e / a.C);
    const uint32_t old = atomicOr(&sm.mask[j >> 2], bit);
    if (a.validate && (old & bit)) flag_error(a.ctl, KVQ_DEV_DUP);
    if (!old) atomicOr(&sm.summary[j >> 9], 1u << ((j >> 4) & 31));
  };
  if ((a.C & 3) == 0) {
    const int4 *l4 = reinterpret_cast<const int4 *>(lists);
    const int n4 = entries >> 2;
    for (int e0 = tid; e0 < n4; e0 += kUBuild * 2) {
      int4 tv[2];
#pragma unroll
      for (int x = 0; x < 2; ++x)
        tv[x] = e0 + kUBuild * x < n4 ? l4[e0 + kUBuild * x] : make_int4(0, 0, 0, 0);
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int e = 4 * (e0 + kUBuild * x);
        if (e >= entries) break;
        mark(e, tv[x].x);
        mark(e + 1, tv[x].y);
        mark(e + 2, tv[x].z);
        mark(e + 3, tv[x].w);
      }
    }
  } else {
    for (int e = tid; e < entries; e += kUBuild) mark(e, lists[e]);
  }
  __syncthreads();
  // ---- the non-empty chunks (warp 0, from the summary bits), then their bytes
  if (warp == 0) {
    int base = 0;
    for (int w0 = 0; w0 < kUW / 512; w0 += 32) {
      const uint32_t bits = sm.summary[w0 + lane];
      const int c = __popc(bits);
      int incl = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      int p = base + incl - c;
      for (uint32_t bb = bits; bb; bb &= bb - 1)
        sm.chunks[p++] = static_cast<uint16_t>(32 * (w0 + lane) + __ffs(bb) - 1);
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) sm.n_chunks = base;
  }
  __syncthreads();
  const int nch = sm.n_chunks;
  const int cpt = (nch + kUBuild - 1) / kUBuild;
  const int c0 = min(nch, tid * cpt), c1 = min(nch, c0 + cpt);
  int cnt = 0;
  for (int c = c0; c < c1; ++c) {
    const uint4 m4 = reinterpret_cast<const uint4 *>(sm.mask)[sm.chunks[c]];
    cnt += nonzero_bytes(m4.x) + nonzero_bytes(m4.y) + nonzero_bytes(m4.z) + nonzero_bytes(m4.w);
  }
  int incl = cnt;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) sm.wsum[warp] = incl;
  __syncthreads();
  int pos = incl - cnt, total = 0;
#pragma unroll
  for (int w = 0; w < kUBuild / 32; ++w) {
    pos += w < warp ? sm.wsum[w] : 0;
    total += sm.wsum[w];
  }
  for (int c = c0; c < c1; ++c) {
    const int ch = sm.chunks[c];
    const uint4 m4 = reinterpret_cast<const uint4 *>(sm.mask)[ch];
    const uint32_t mw[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
    for (int w = 0; w < 4; ++w)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t hb = (mw[w] >> (8 * k)) & 0xffu;
        if (hb) {
          if (pos < entries) {  // always: at most 8 C positions are listed
            a.list_pos[lbase + pos] = lo + 16 * ch + 4 * w + k;
            a.list_heads[lbase + pos] = static_cast<uint8_t>(hb);
          }
          ++pos;
        }
      }
  }
  if (tid == 0) a.count[static_cast<long>(u) * a.slices + slice] = min(total, entries);
}

// The raw bytes one loader thread copies for one round: 32 features (a chunk)
// of K and V of one position. int4 row: K codes, the 32 K scales of the
// chunk, V codes and the V scale; window row: K (bf16) over kc and the first
// 48 bytes of ks, V (bf16) over the rest of ks.
struct RawSlot {
  uint8_t kc[16];
  float ks[32];
  uint8_t vc[16];
  float vs;
  uint32_t pad[3];
};

// One stage of converted rows: K and V of kUT rows, bf16, 256 bytes a row
// with the 16-byte chunks of row r permuted by c ^ (r & 7), so that the 8
// rows an ldmatrix phase reads fall in distinct banks.
struct UnionStage {
  uint16_t k[kUT][128];
  uint16_t v[kUT][128];
};

struct __align__(16) UnionSmem {
  RawSlot raw[kURaw][32 * kULoaders];
  union {
    UnionStage stage[2];         // converted rows (during the rounds)
    float red_o[kUMma][8][128];  // the MMA warps' O (after the rounds)
  };
  int32_t pos[kUMaxPiece];       // the piece's positions
  uint8_t heads[kUMaxPiece];     // their head bits
  uint64_t full[2], empty[2];
  float red_m[kUMma][8], red_l[kUMma][8], red_c[kUMma][8];
};
static_assert(sizeof(UnionSmem) * 2 + 2048 <= 228 * 1024, "two union CTAs per SM");

// Byte offset of 16-byte chunk c (0..15) of row r in a stage array.
__device__ __forceinline__ uint32_t urow(int r, int c) {
  return static_cast<uint32_t>(r * 256 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int kPending>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory");
}

// Online softmax of one m-tile of scores s (rows g, g+8 = positions; heads
// 2t, 2t+1; masked entries -inf) into (m, l) of heads 2t, 2t+1; s becomes P.
// The reference maximum moves only when a score passes it by more than 2^8,
// so P stays below 2^8.
__device__ __forceinline__ void union_softmax(float (&s)[4], float (&m)[2], float (&l)[2],
                                              float (&o)[8][4]) {
  float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
  if (__any_sync(0xffffffffu, mx0 > m[0] + 8.0f || mx1 > m[1] + 8.0f)) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float n0 = fmaxf(m[0], mx0), n1 = fmaxf(m[1], mx1);
    // a head with no key yet keeps m = -inf (and so l = 0 and O = 0)
    const float c0 = n0 == -CUDART_INF_F ? 1.0f : fast_exp2(m[0] - n0);
    const float c1 = n1 == -CUDART_INF_F ? 1.0f : fast_exp2(m[1] - n1);
    m[0] = n0;
    m[1] = n1;
    l[0] *= c0;
    l[1] *= c1;
#pragma unroll
    for (int f = 0; f < 8; ++f) {
      o[f][0] *= c0;
      o[f][1] *= c1;
      o[f][2] *= c0;
      o[f][3] *= c1;
    }
  }
  s[0] = fast_exp2(s[0] - m[0]);
  s[1] = fast_exp2(s[1] - m[1]);
  s[2] = fast_exp2(s[2] - m[0]);
  s[3] = fast_exp2(s[3] - m[1]);
#pragma unroll
  for (int j = 0; j < 4; ++j) s[j] = s[j] == s[j] ? s[j] : 0.0f;  // -inf - -inf while m = -inf
  l[0] += s[0] + s[2];
  l[1] += s[1] + s[3];
}

// Issue the asynchronous copies of chunk cc of position t into a raw slot.
__device__ __forceinline__ void union_fetch(const UnionArgs &a, long u, int t, int cc,
                                            RawSlot &r) {
  if (t < a.cut) {
    const long grp = u * a.Gs + (t >> 5);
    const long vr = u * a.Vs + t;
    if (!in_bounds(a.ctl, a.k_codes + (grp * 32 + (t & 31)) * 64 + 16 * cc, 16) ||
        !in_bounds(a.ctl, a.k_scales + grp * 128 + 32 * cc, 128) ||
        !in_bounds(a.ctl, a.v_codes + vr * 64 + 16 * cc, 16) ||
        !in_bounds(a.ctl, a.v_scales + vr * 4 + cc, 4))
      return;
    cp_async16(smem_u32(r.kc), a.k_codes + (grp * 32 + (t & 31)) * 64 + 16 * cc);
    const float *ks = a.k_scales + grp * 128 + 32 * cc;
#pragma unroll
    for (int j = 0; j < 8; ++j) cp_async16(smem_u32(r.ks + 4 * j), ks + 4 * j);
    cp_async16(smem_u32(r.vc), a.v_codes + vr * 64 + 16 * cc);
    cp_async4(smem_u32(&r.vs), a.v_scales + vr * 4 + cc);
  } else {
    const long wr = (u * a.Ws + (t - a.cut)) * 128 + 32 * cc;
    if (!in_bounds(a.ctl, a.k_window + wr, 64) || !in_bounds(a.ctl, a.v_window + wr, 64)) return;
    uint8_t *dst = reinterpret_cast<uint8_t *>(&r);  // K: bytes 0..63, V: bytes 64..127
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      cp_async16(smem_u32(dst + 16 * j), a.k_window + wr + 8 * j);
      cp_async16(smem_u32(dst + 64 + 16 * j), a.v_window + wr + 8 * j);
    }
  }
}

// Convert a landed raw slot to bf16 into row `row` of a stage (int4 rows:
// x = code * scale, rounded once to bf16); zeros when !valid.
__device__ __forceinline__ void union_convert(const RawSlot &r, bool int4, bool valid, int cc,
                                              UnionStage &sg, int row) {
  uint8_t *kd = reinterpret_cast<uint8_t *>(sg.k), *vd = reinterpret_cast<uint8_t *>(sg.v);
  const uint4 kcw = *reinterpret_cast<const uint4 *>(r.kc);
  const uint4 vcw = *reinterpret_cast<const uint4 *>(r.vc);
  const uint32_t kw4[4] = {kcw.x, kcw.y, kcw.z, kcw.w}, vw4[4] = {vcw.x, vcw.y, vcw.z, vcw.w};
  const float vs = r.vs;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint4 ko, vo;
    if (!valid) {
      ko = vo = make_uint4(0u, 0u, 0u, 0u);
    } else if (int4) {
      // word w of the codes: features 8w..8w+7 of the chunk, low nibble first
      const float4 s0 = *reinterpret_cast<const float4 *>(r.ks + 8 * w);
      const float4 s1 = *reinterpret_cast<const float4 *>(r.ks + 8 * w + 4);
      const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
      uint32_t kp[4], vp[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float k0 = static_cast<float>(static_cast<int>((kw4[w] >> (8 * e)) & 15u) - 8);
        const float k1 = static_cast<float>(static_cast<int>((kw4[w] >> (8 * e + 4)) & 15u) - 8);
        const float v0 = static_cast<float>(static_cast<int>((vw4[w] >> (8 * e)) & 15u) - 8);
        const float v1 = static_cast<float>(static_cast<int>((vw4[w] >> (8 * e + 4)) & 15u) - 8);
        kp[e] = pack_bf2(k0 * sc[2 * e], k1 * sc[2 * e + 1]);
        vp[e] = pack_bf2(v0 * vs, v1 * vs);
      }
      ko = make_uint4(kp[0], kp[1], kp[2], kp[3]);
      vo = make_uint4(vp[0], vp[1], vp[2], vp[3]);
    } else {
      const uint8_t *raw = reinterpret_cast<const uint8_t *>(&r);
      ko = *reinterpret_cast<const uint4 *>(raw + 16 * w);
      vo = *reinterpret_cast<const uint4 *>(raw + 64 + 16 * w);
    }
    *reinterpret_cast<uint4 *>(kd + urow(row, 4 * cc + w)) = ko;
    *reinterpret_cast<uint4 *>(vd + urow(row, 4 * cc + w)) = vo;
  }
}

__global__ void __launch_bounds__(kUThreads, 2) cand_union_kernel(const UnionArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  UnionSmem &sm = *reinterpret_cast<UnionSmem *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int piece = blockIdx.x, u = blockIdx.y;
  allow_next_grid();
  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 32 * kULoaders);
      mbar_init(smem_u32(&sm.empty[s]), 32 * kUMma);
    }
    fence_mbar_init();
  }
  __shared__ int prefix[kUMaxSlices + 1];
  wait_prior_grid();  // the union lists of the build kernel (and whatever wrote q)
  // the q rows of the MMA warps: head g as B fragments (bf16 pairs of
  // features 16k + 2t.. and 16k + 2t + 8..)
  const int g = lane >> 2, t4 = lane & 3;
  uint32_t qb[8][2];
  // the unit's q rows, counts and lists (the same in every thread)
  const long lists_at = static_cast<long>(u) * a.slices * 8 * a.C;
  const bool io_ok = in_bounds(a.ctl, a.q + static_cast<long>(u) * 8 * 128, 8 * 128 * 2) &&
                     in_bounds(a.ctl, a.count + static_cast<long>(u) * a.slices, 4 * a.slices) &&
                     in_bounds(a.ctl, a.list_pos + lists_at, 4L * a.slices * 8 * a.C) &&
                     in_bounds(a.ctl, a.list_heads + lists_at, 1L * a.slices * 8 * a.C);
  if (!io_ok) return;
  if (warp < kUMma) {
    const uint32_t *qw =
        reinterpret_cast<const uint32_t *>(a.q + (static_cast<long>(u) * 8 + g) * 128);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      qb[k][0] = qw[8 * k + t4];
      qb[k][1] = qw[8 * k + t4 + 4];
    }
  }
  // ---- this piece: rows [r0, r1) of the KV head's union (its build slices'
  // lists one after another), staged in shared memory
  if (tid == 0) {
    int acc = 0;
    for (int sl = 0; sl < a.slices; ++sl) {
      prefix[sl] = acc;
      acc += a.count[static_cast<long>(u) * a.slices + sl];
    }
    prefix[a.slices] = acc;
  }
  __syncthreads();
  const int cnt = prefix[a.slices];
  const int r0 = static_cast<int>(static_cast<long>(piece) * cnt / a.pieces);
  const int r1 = static_cast<int>(static_cast<long>(piece + 1) * cnt / a.pieces);
  const int total = min(r1 - r0, kUMaxPiece);
  for (int i = tid; i < total; i += kUThreads) {
    const int row = r0 + i;
    int sl = 0;
    while (prefix[sl + 1] <= row) ++sl;
    const long at = (static_cast<long>(u) * a.slices + sl) * 8 * a.C + (row - prefix[sl]);
    sm.pos[i] = a.list_pos[at];
    sm.heads[i] = a.list_heads[at];
  }
  if (tid == 0 && r1 - r0 > kUMaxPiece) flag_error(a.ctl, KVQ_DEV_BOUNDS);  // not reached
  __syncthreads();

  const int rounds = (total + kUT - 1) / kUT;
  float m[2] = {-CUDART_INF_F, -CUDART_INF_F}, l[2] = {0.0f, 0.0f}, o[8][4];
#pragma unroll
  for (int f = 0; f < 8; ++f)
#pragma unroll
    for (int j = 0; j < 4; ++j) o[f][j] = 0.0f;
  if (warp >= kUMma) {
    // ---- loaders: thread -> (row tt, 32-feature chunk cc) of every round;
    // the raw bytes of kURaw rounds are in flight (asynchronous copies into
    // the thread's own slots), converted to bf16 as each lands
    const int pt = tid - 32 * kUMma, tt = pt >> 2, cc = pt & 3;
    auto fetch = [&](int r) {
      const int i = r * kUT + tt;
      if (r < rounds && i < total) union_fetch(a, u, sm.pos[i], cc, sm.raw[r % kURaw][pt]);
      cp_async_commit();  // one group per round, empty or not
    };
#pragma unroll
    for (int r = 0; r < kURaw; ++r) fetch(r);
    for (int r = 0; r < rounds; ++r) {
      const int st = r & 1;
      cp_async_wait<kURaw - 1>();  // this thread's copies of round r have landed
      if (r >= 2 && !mbar_wait(smem_u32(&sm.empty[st]), ((r - 2) >> 1) & 1, a.ctl.wait_limit_ns)) {
        flag_error(a.ctl, KVQ_DEV_TIMEOUT);
        break;
      }
      const int i = r * kUT + tt;
      const bool valid = i < total;
      const int t = valid ? sm.pos[i] : 0;
      union_convert(sm.raw[r % kURaw][pt], t < a.cut, valid, cc, sm.stage[st], tt);
      mbar_arrive(smem_u32(&sm.full[st]));
      fetch(r + kURaw);  // into the slot just converted
    }
    cp_async_wait<0>();
  } else {
    // ---- MMA warps: warp w takes rows 16w .. 16w + 15 of a round
    const int m0 = 16 * warp, mi = lane >> 3, rr = lane & 7;
    for (int r = 0; r < rounds; ++r) {
      const int st = r & 1;
      if (!mbar_wait(smem_u32(&sm.full[st]), (r >> 1) & 1, a.ctl.wait_limit_ns)) {
        flag_error(a.ctl, KVQ_DEV_TIMEOUT);
        break;
      }
      UnionStage &sg = sm.stage[st];
      const int base = r * kUT + m0;
      if (base < total) {
        float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        const int krow = m0 + rr + 8 * (mi & 1);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(smem_u32(reinterpret_cast<uint8_t *>(sg.k) + urow(krow, 2 * k + (mi >> 1))), a0,
                  a1, a2, a3);
          mma_bf16(s, a0, a1, a2, a3, qb[k][0], qb[k][1]);
        }
        const int ia = base + g, ib = ia + 8;
        const uint32_t ma = ia < total ? sm.heads[ia] : 0u, mb = ib < total ? sm.heads[ib] : 0u;
        s[0] = (ma >> (2 * t4)) & 1u ? s[0] * a.scale_log2 : -CUDART_INF_F;
        s[1] = (ma >> (2 * t4 + 1)) & 1u ? s[1] * a.scale_log2 : -CUDART_INF_F;
        s[2] = (mb >> (2 * t4)) & 1u ? s[2] * a.scale_log2 : -CUDART_INF_F;
        s[3] = (mb >> (2 * t4 + 1)) & 1u ? s[3] * a.scale_log2 : -CUDART_INF_F;
        union_softmax(s, m, l, o);
        const uint32_t pb0 = movmatrix_t(pack_bf2(s[0], s[1]));
        const uint32_t pb1 = movmatrix_t(pack_bf2(s[2], s[3]));
        const int vrow = m0 + rr + 8 * (mi >> 1);
#pragma unroll
        for (int f = 0; f < 8; ++f) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(smem_u32(reinterpret_cast<uint8_t *>(sg.v) + urow(vrow, 2 * f + (mi & 1))), a0,
                    a1, a2, a3);
          mma_bf16(o[f], a0, a1, a2, a3, pb0, pb1);
        }
      }
      mbar_arrive(smem_u32(&sm.empty[st]));
    }
  }
  __syncthreads();  // every round is done: the stages are free for the merge

  // ---- merge the MMA warps and leave one partial per head
  if (warp < kUMma) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
      l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
    }
    if (g == 0) {
      sm.red_m[warp][2 * t4] = m[0];
      sm.red_m[warp][2 * t4 + 1] = m[1];
      sm.red_l[warp][2 * t4] = l[0];
      sm.red_l[warp][2 * t4 + 1] = l[1];
    }
    // o[f][j]: feature 16f + g (+8 for j >= 2), head 2t (+1 for odd j)
#pragma unroll
    for (int f = 0; f < 8; ++f) {
      sm.red_o[warp][2 * t4][16 * f + g] = o[f][0];
      sm.red_o[warp][2 * t4 + 1][16 * f + g] = o[f][1];
      sm.red_o[warp][2 * t4][16 * f + g + 8] = o[f][2];
      sm.red_o[warp][2 * t4 + 1][16 * f + g + 8] = o[f][3];
    }
  }
  __syncthreads();
  if (tid < 8) {
    const int h = tid;
    float mx = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kUMma; ++w) mx = fmaxf(mx, sm.red_m[w][h]);
    float ls = 0.0f;
#pragma unroll
    for (int w = 0; w < kUMma; ++w) {
      const float c = sm.red_m[w][h] == -CUDART_INF_F ? 0.0f : exp2f(sm.red_m[w][h] - mx);
      sm.red_c[w][h] = c;
      ls += c * sm.red_l[w][h];
    }
    float *part = a.partials + ((static_cast<long>(u) * a.pieces + piece) * 8 + h) * kUPart;
    if (in_bounds(a.ctl, part, sizeof(float) * kUPart)) {
      part[128] = mx;
      part[129] = ls;
    }
  }
  __syncthreads();
  const bool part_ok = in_bounds(
      a.ctl, a.partials + (static_cast<long>(u) * a.pieces + piece) * 8 * kUPart,
      sizeof(float) * 8 * kUPart);
  for (int i = tid; part_ok && i < 8 * 128; i += kUThreads) {
    const int h = i >> 7, d = i & 127;
    float acc = 0.0f;
#pragma unroll
    for (int w = 0; w < kUMma; ++w) acc += sm.red_c[w][h] * sm.red_o[w][h][d];
    a.partials[((static_cast<long>(u) * a.pieces + piece) * 8 + h) * kUPart + d] = acc;
  }
}

// One warp per (sequence, query head): the log-sum-exp merge of the pieces'
// partials, normalised and stored.
__global__ void __launch_bounds__(256) cand_union_combine_kernel(const UnionArgs a) {
  wait_prior_grid();
  allow_next_grid();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x, h = warp;
  const float *base = a.partials + (static_cast<long>(u) * a.pieces * 8 + h) * kUPart;
  const long o = (static_cast<long>(u) * 8 + h) * 128 + 4 * lane;
  const size_t ob = a.out_dtype == KVQ_F32 ? 4 : 2;
  // the unit's partials and this head's output row (the same in every lane)
  if (!in_bounds(a.ctl, a.partials + static_cast<long>(u) * a.pieces * 8 * kUPart,
                 sizeof(float) * a.pieces * 8 * kUPart) ||
      !in_bounds(a.ctl, static_cast<uint8_t *>(a.out) + (o - 4 * lane) * ob, 128 * ob))
    return;
  float m = -CUDART_INF_F, l = 0.0f;
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  constexpr int kBatch = 8;  // pieces whose loads are in flight together
  for (int s0 = 0; s0 < a.pieces; s0 += kBatch) {
    float pm[kBatch], pl[kBatch];
    float4 po[kBatch];
#pragma unroll
    for (int x = 0; x < kBatch; ++x) {
      const float *p = base + static_cast<long>(min(s0 + x, a.pieces - 1)) * 8 * kUPart;
      const float2 ml = *reinterpret_cast<const float2 *>(p + 128);
      pm[x] = s0 + x < a.pieces ? ml.x : -CUDART_INF_F;
      pl[x] = ml.y;
      po[x] = reinterpret_cast<const float4 *>(p)[lane];
    }
    float nm = m;
#pragma unroll
    for (int x = 0; x < kBatch; ++x) nm = fmaxf(nm, pm[x]);
    if (nm == -CUDART_INF_F) continue;
    const float r = exp2f(m - nm);  // 0 while m is -inf
    l *= r;
    acc.x *= r;
    acc.y *= r;
    acc.z *= r;
    acc.w *= r;
#pragma unroll
    for (int x = 0; x < kBatch; ++x) {
      const float w = exp2f(pm[x] - nm);  // 0 for empty pieces
      l += w * pl[x];
      acc.x += w * po[x].x;
      acc.y += w * po[x].y;
      acc.z += w * po[x].z;
      acc.w += w * po[x].w;
    }
    m = nm;
  }
  const float inv = 1.0f / l;
  if (a.out_dtype == KVQ_F32) {
    reinterpret_cast<float4 *>(static_cast<float *>(a.out) + o)[0] =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  } else {
    __nv_bfloat16 *ob = static_cast<__nv_bfloat16 *>(a.out) + o;
    reinterpret_cast<uint2 *>(ob)[0] =
        make_uint2(pack_bf2(acc.x * inv, acc.y * inv), pack_bf2(acc.z * inv, acc.w * inv));
  }
}

struct UnionPlan {
  int pieces, slices;
  long units;
  size_t list_bytes, heads_bytes, count_bytes, part_bytes;
};

// Pieces per (sequence, KV head): one wave of the GPU's two resident CTAs
// per SM (pieces of a KV head have equal row counts, so a single wave is
// balanced), and none above kUMaxPiece rows.
UnionPlan union_plan(const kvq_cache &c, int n_cand, int num_sms) {
  UnionPlan p;
  p.units = static_cast<long>(c.batch) * c.kv_heads;
  const long rows = 8L * n_cand;
  long pieces = std::max<long>(1, 2L * num_sms / p.units);
  pieces = std::max(pieces, (rows + kUMaxPiece - 1) / kUMaxPiece);
  p.pieces = static_cast<int>(pieces);
  p.slices = static_cast<int>((c.n_tokens + kUW - 1) / kUW);
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  p.list_bytes = up(sizeof(int32_t) * p.units * p.slices * rows);
  p.heads_bytes = up(p.units * p.slices * rows);
  p.count_bytes = up(sizeof(int32_t) * p.units * p.slices);
  p.part_bytes = sizeof(float) * p.units * p.pieces * 8 * kUPart;
  return p;
}

}  // namespace

bool candidates_union_supported(const kvq_cache &c, int q_dtype, int Hq, int n_q, int n_cand) {
  const bool win_ok = c.recent == 0 || (c.kwin_dtype == KVQ_BF16 && c.vwin_dtype == KVQ_BF16);
  return c.head_dim == 128 && Hq == 8 * c.kv_heads && n_q == 1 && q_dtype == KVQ_BF16 &&
         8L * n_cand <= kUMaxList && win_ok && static_cast<long>(c.batch) * c.kv_heads <= 65535 &&
         (static_cast<long>(c.n_tokens) + kUW - 1) / kUW <= kUMaxSlices;
}

size_t candidates_union_workspace_bytes(const kvq_cache &c, int n_cand, int num_sms) {
  const UnionPlan p = union_plan(c, n_cand, num_sms);
  return p.list_bytes + p.heads_bytes + p.count_bytes + p.part_bytes;
}

int launch_candidates_union(const kvq_cache &c, const void *q, const int32_t *idx, int n_cand,
                            int validate, float scale_log2, void *out, int out_dtype, void *ws,
                            const KernelCtl &ctl, int num_sms, cudaStream_t s) {
  const CacheDims d = dims_of(c);
  const UnionPlan p = union_plan(c, n_cand, num_sms);
  UnionArgs a;
  a.k_codes = c.k_codes;
  a.k_scales = c.k_scales;
  a.v_codes = c.v_codes;
  a.v_scales = c.v_scales;
  a.k_window = static_cast<const uint16_t *>(c.k_window);
  a.v_window = static_cast<const uint16_t *>(c.v_window);
  a.Hkv = d.Hkv;
  a.N = d.N;
  a.cut = d.cut;
  a.Gs = d.Gs;
  a.Vs = d.Vs;
  a.Ws = d.Ws;
  a.C = n_cand;
  a.validate = validate;
  a.q = static_cast<const uint16_t *>(q);
  a.idx = idx;
  a.pieces = p.pieces;
  a.slices = p.slices;
  a.scale_log2 = scale_log2;
  uint8_t *w = static_cast<uint8_t *>(ws);
  a.list_pos = reinterpret_cast<int32_t *>(w);
  a.list_heads = w + p.list_bytes;
  a.count = reinterpret_cast<int32_t *>(w + p.list_bytes + p.heads_bytes);
  a.partials = reinterpret_cast<float *>(w + p.list_bytes + p.heads_bytes + p.count_bytes);
  a.out = out;
  a.out_dtype = out_dtype;
  a.ctl = ctl;
  const size_t build_smem = sizeof(BuildSmem);
  opt_in_smem(cand_union_build_kernel, build_smem);
  launch_dependent(cand_union_build_kernel, dim3(p.slices, static_cast<unsigned>(p.units)),
                   dim3(kUBuild), build_smem, s, a);
  const size_t smem = sizeof(UnionSmem);
  opt_in_smem(cand_union_kernel, smem);
  launch_dependent(cand_union_kernel, dim3(p.pieces, static_cast<unsigned>(p.units)),
                   dim3(kUThreads), smem, s, a);
  launch_dependent(cand_union_combine_kernel, dim3(static_cast<unsigned>(p.units)), dim3(256), 0,
                   s, a);
  return 3;
}

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
    opt_in_smem(cand_topk_kernel<F>, smem);                                             \
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
