// Split-K decode attention over an int4 KV cache: one query row per
// (sequence, query head), 8 query heads per KV head (GQA), head dim 128.
//
// What it computes: O = softmax(sm_scale * q K^T) V over all N tokens, K and V
// dequantized from grouped int4 (residual-window page, section 固定預算) or
// read from the bf16 window of the last R tokens; no mask.
//
// Work split. The cache of one (sequence, KV head) -- a "unit" -- is a list
// of items: its int4 groups (32 tokens: 2 KB K codes, 512 B K scales, 2 KB V
// codes, 512 B V scales) followed by its window tiles (16 tokens of bf16 K and
// V). All items of all units are laid end to end and the persistent grid
// (2 CTAs per SM) takes equal contiguous slices, so every SM streams the same
// number of bytes. A CTA emits one partial (running max m, sum l, unnormalised
// O for 8 heads) per unit its slice touches; combine_kernel merges them with
// the log-sum-exp rule.
//
// Inside a CTA. Warp 4 is the loader: one lane issues cp.async.bulk copies of
// each item into an 8-stage shared-memory ring, completing on mbarriers.
// Warps 0-3 take the items round robin. Scores use mma.sync m16n8k16 with the
// 16 tokens of a tile as M and the 8 query heads as N: the K scales of a group
// are folded into q (q' = q * s_k * sm_scale * log2 e, fp16), the nibbles are
// turned into fp16 codes with two bit masks and one subtraction, so the MMA sees
// codes in [-7, 7] exactly. P (fp16) is transposed in registers with movmatrix
// and multiplies V^T (features as M) whose codes are scaled by the token's V
// scale in fp16. The bf16 window uses bf16 MMAs with q and P split into
// hi + lo bf16 parts. Softmax runs in the log2 domain with fp32 state.
//
// Feature order. Within a thread, features are visited in a fixed permutation
// (the one that makes a 16-byte row slice of nibbles a ready MMA operand); the
// same permutation is used for q and K, and the output is written back in
// natural order.
#include <math_constants.h>

#include <algorithm>
#include <mutex>

#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kD = 128;
constexpr int kHeads = 8;              // query heads per KV head
constexpr int kConsumers = 4;          // consumer warps
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kStages = 8;
constexpr int kStageBytes = 8192;
constexpr int kWinTile = 16;           // window tokens per item
constexpr int kPartFloats = kD + 4;    // O[128], m, l per head, padded to 16 bytes
// int4 item layout inside a stage
constexpr int kOffKScale = 2048, kOffVCode = 2560, kOffVScale = 4608;

struct DecodeArgs {
  const uint8_t *k_codes;
  const float *k_scales;
  const uint8_t *v_codes;
  const float *v_scales;
  const uint16_t *k_window;
  const uint16_t *v_window;
  const void *q;
  int q_dtype;
  int Hkv, N, R, cut, Gk, Wt, ipu;  // ipu: items per unit = Gk + Wt
  long total_items;
  int num_ctas, max_units;
  float scale_log2;
  float *partials;                  // [num_ctas][max_units][8][132]
  KernelCtl ctl;
};

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t as_u32(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 as_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// Nibbles at bits 0-3 and 16-19 -> fp16 codes: 0x6400 | n is 1024 + n, n = code + 8.
__device__ __forceinline__ uint32_t dq_lo(uint32_t w) {
  const uint32_t x = (w & 0x000F000Fu) | 0x64006400u;
  return as_u32(__hsub2(as_h2(x), as_h2(0x64086408u)));  // 1032
}
// Nibbles at bits 4-7 and 20-23: 0x5400 | n << 4 is 64 + n.
__device__ __forceinline__ uint32_t dq_hi(uint32_t w) {
  const uint32_t x = (w & 0x00F000F0u) | 0x54005400u;
  return as_u32(__hsub2(as_h2(x), as_h2(0x54805480u)));  // 72
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  return as_u32(__floats2half2_rn(lo, hi));
}
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&b);
}
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// ------------------------------------------------------------------ per-warp state
struct WarpState {
  float o[8][4];  // PV accumulators: m-tile f (features), (row g|g+8) x (head 2t|2t+1)
  float m[2];     // running max, heads 2t and 2t+1 (log2 domain)
  float l[2];     // this thread's share of the running sum
};

__device__ __forceinline__ void state_reset(WarpState &st) {
#pragma unroll
  for (int f = 0; f < 8; ++f)
#pragma unroll
    for (int j = 0; j < 4; ++j) st.o[f][j] = 0.0f;
  st.m[0] = st.m[1] = -CUDART_INF_F;
  st.l[0] = st.l[1] = 0.0f;
}

// Online-softmax update with NT m-tiles of scores s[NT][4] (rows g, g+8 x heads
// 2t, 2t+1); masked scores are -inf. Turns s into probabilities in place.
template <int NT>
__device__ __forceinline__ void softmax_update(WarpState &st, float (&s)[NT][4]) {
  float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    mx0 = fmaxf(mx0, fmaxf(s[i][0], s[i][2]));
    mx1 = fmaxf(mx1, fmaxf(s[i][1], s[i][3]));
  }
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
  }
  const float n0 = fmaxf(st.m[0], mx0), n1 = fmaxf(st.m[1], mx1);
  const float c0 = exp2f(st.m[0] - n0), c1 = exp2f(st.m[1] - n1);
  st.m[0] = n0;
  st.m[1] = n1;
  float sum0 = 0.0f, sum1 = 0.0f;
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    s[i][0] = exp2f(s[i][0] - n0);
    s[i][1] = exp2f(s[i][1] - n1);
    s[i][2] = exp2f(s[i][2] - n0);
    s[i][3] = exp2f(s[i][3] - n1);
    sum0 += s[i][0] + s[i][2];
    sum1 += s[i][1] + s[i][3];
  }
  st.l[0] = st.l[0] * c0 + sum0;
  st.l[1] = st.l[1] * c1 + sum1;
  if (!__all_sync(0xffffffffu, c0 == 1.0f && c1 == 1.0f)) {
#pragma unroll
    for (int f = 0; f < 8; ++f) {
      st.o[f][0] *= c0;
      st.o[f][1] *= c1;
      st.o[f][2] *= c0;
      st.o[f][3] *= c1;
    }
  }
}

// ------------------------------------------------------------------ item bodies
// int4 group: 32 tokens (two m-tiles), `valid` of them real.
__device__ __forceinline__ void do_int4_item(WarpState &st, const uint8_t *stage,
                                             const float (&qr)[32], int valid, int g, int t) {
  const float *ks = reinterpret_cast<const float *>(stage + kOffKScale);
  // q' fragments for this group (features 32t .. 32t+31 of head g)
  uint32_t bq[8][2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 s0 = *reinterpret_cast<const float4 *>(ks + 32 * t + 8 * i);
    const float4 s1 = *reinterpret_cast<const float4 *>(ks + 32 * t + 8 * i + 4);
    const float x0 = qr[8 * i + 0] * s0.x, x1 = qr[8 * i + 1] * s0.y, x2 = qr[8 * i + 2] * s0.z,
                x3 = qr[8 * i + 3] * s0.w, x4 = qr[8 * i + 4] * s1.x, x5 = qr[8 * i + 5] * s1.y,
                x6 = qr[8 * i + 6] * s1.z, x7 = qr[8 * i + 7] * s1.w;
    bq[2 * i][0] = pack_h2(x0, x4);
    bq[2 * i][1] = pack_h2(x1, x5);
    bq[2 * i + 1][0] = pack_h2(x2, x6);
    bq[2 * i + 1][1] = pack_h2(x3, x7);
  }
  float s[2][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const int r0 = 16 * mt + g;
    const uint4 ka = *reinterpret_cast<const uint4 *>(stage + r0 * 64 + 16 * t);
    const uint4 kb = *reinterpret_cast<const uint4 *>(stage + (r0 + 8) * 64 + 16 * t);
    const uint32_t wa[4] = {ka.x, ka.y, ka.z, ka.w}, wb[4] = {kb.x, kb.y, kb.z, kb.w};
    s[mt][0] = s[mt][1] = s[mt][2] = s[mt][3] = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      mma_f16(s[mt], dq_lo(wa[i]), dq_lo(wb[i]), dq_hi(wa[i]), dq_hi(wb[i]), bq[2 * i][0],
              bq[2 * i][1]);
      const uint32_t a8 = wa[i] >> 8, b8 = wb[i] >> 8;
      mma_f16(s[mt], dq_lo(a8), dq_lo(b8), dq_hi(a8), dq_hi(b8), bq[2 * i + 1][0],
              bq[2 * i + 1][1]);
    }
    if (r0 >= valid) s[mt][0] = s[mt][1] = -CUDART_INF_F;
    if (r0 + 8 >= valid) s[mt][2] = s[mt][3] = -CUDART_INF_F;
  }
  softmax_update<2>(st, s);

  const uint8_t *vc = stage + kOffVCode;
  const float *vs = reinterpret_cast<const float *>(stage + kOffVScale);
  const uint2 zero8 = make_uint2(0x88888888u, 0x88888888u);  // code 0 everywhere
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const uint32_t b0 = movmatrix_t(pack_h2(s[mt][0], s[mt][1]));
    const uint32_t b1 = movmatrix_t(pack_h2(s[mt][2], s[mt][3]));
    const int ta = 16 * mt + 2 * t;  // tokens ta, ta+1, ta+8, ta+9
    const bool va = ta < valid, vb = ta + 1 < valid, vcv = ta + 8 < valid, vd = ta + 9 < valid;
    const uint2 za = va ? *reinterpret_cast<const uint2 *>(vc + ta * 64 + 8 * g) : zero8;
    const uint2 zb = vb ? *reinterpret_cast<const uint2 *>(vc + (ta + 1) * 64 + 8 * g) : zero8;
    const uint2 zc = vcv ? *reinterpret_cast<const uint2 *>(vc + (ta + 8) * 64 + 8 * g) : zero8;
    const uint2 zd = vd ? *reinterpret_cast<const uint2 *>(vc + (ta + 9) * 64 + 8 * g) : zero8;
    const float sa = va ? vs[ta * 4 + (g >> 1)] : 0.0f;
    const float sb = vb ? vs[(ta + 1) * 4 + (g >> 1)] : 0.0f;
    const float sc = vcv ? vs[(ta + 8) * 4 + (g >> 1)] : 0.0f;
    const float sd = vd ? vs[(ta + 9) * 4 + (g >> 1)] : 0.0f;
    const __half2 sab = __floats2half2_rn(sa, sb), scd = __floats2half2_rn(sc, sd);
    // feature f of this thread's 16 (16g + f): pairs (ta, ta+1) and (ta+8, ta+9)
    uint32_t pab[16], pcd[16];
    const uint32_t wab[2][2] = {{prmt(za.x, zb.x, 0x5410), prmt(za.x, zb.x, 0x7632)},
                                {prmt(za.y, zb.y, 0x5410), prmt(za.y, zb.y, 0x7632)}};
    const uint32_t wcd[2][2] = {{prmt(zc.x, zd.x, 0x5410), prmt(zc.x, zd.x, 0x7632)},
                                {prmt(zc.y, zd.y, 0x5410), prmt(zc.y, zd.y, 0x7632)}};
#pragma unroll
    for (int w = 0; w < 2; ++w)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int f = 8 * w + 4 * h;
        pab[f + 0] = as_u32(__hmul2(as_h2(dq_lo(wab[w][h])), sab));
        pab[f + 1] = as_u32(__hmul2(as_h2(dq_hi(wab[w][h])), sab));
        pab[f + 2] = as_u32(__hmul2(as_h2(dq_lo(wab[w][h] >> 8)), sab));
        pab[f + 3] = as_u32(__hmul2(as_h2(dq_hi(wab[w][h] >> 8)), sab));
        pcd[f + 0] = as_u32(__hmul2(as_h2(dq_lo(wcd[w][h])), scd));
        pcd[f + 1] = as_u32(__hmul2(as_h2(dq_hi(wcd[w][h])), scd));
        pcd[f + 2] = as_u32(__hmul2(as_h2(dq_lo(wcd[w][h] >> 8)), scd));
        pcd[f + 3] = as_u32(__hmul2(as_h2(dq_hi(wcd[w][h] >> 8)), scd));
      }
#pragma unroll
    for (int f = 0; f < 8; ++f) mma_f16(st.o[f], pab[f], pab[8 + f], pcd[f], pcd[8 + f], b0, b1);
  }
}

// bf16 window tile: 16 tokens, `valid` of them real.
__device__ __forceinline__ void do_window_item(WarpState &st, const uint8_t *stage,
                                               const float (&qr)[32], int valid, int g, int t) {
  const uint32_t *kw = reinterpret_cast<const uint32_t *>(stage);         // [16][64] words
  const uint32_t *vw = reinterpret_cast<const uint32_t *>(stage + 4096);  // [16][64] words
  float s[1][4] = {{0.0f, 0.0f, 0.0f, 0.0f}};
  const bool ra = g < valid, rb = g + 8 < valid;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    // features 32t + 8i .. +7 of rows g and g+8
    const uint4 a = ra ? *reinterpret_cast<const uint4 *>(kw + g * 64 + 16 * t + 4 * i)
                       : make_uint4(0, 0, 0, 0);
    const uint4 b = rb ? *reinterpret_cast<const uint4 *>(kw + (g + 8) * 64 + 16 * t + 4 * i)
                       : make_uint4(0, 0, 0, 0);
    const float q0 = qr[8 * i + 0], q1 = qr[8 * i + 1], q2 = qr[8 * i + 2], q3 = qr[8 * i + 3];
    const float q4 = qr[8 * i + 4], q5 = qr[8 * i + 5], q6 = qr[8 * i + 6], q7 = qr[8 * i + 7];
    const uint32_t h04 = pack_bf2(q0, q4), h15 = pack_bf2(q1, q5);
    const uint32_t h26 = pack_bf2(q2, q6), h37 = pack_bf2(q3, q7);
    const uint32_t l04 = pack_bf2(q0 - bf_lo(h04), q4 - bf_hi(h04));
    const uint32_t l15 = pack_bf2(q1 - bf_lo(h15), q5 - bf_hi(h15));
    const uint32_t l26 = pack_bf2(q2 - bf_lo(h26), q6 - bf_hi(h26));
    const uint32_t l37 = pack_bf2(q3 - bf_lo(h37), q7 - bf_hi(h37));
    // k-step 2i: features (0,4) and (1,5); k-step 2i+1: (2,6) and (3,7)
    const uint32_t a04 = prmt(a.x, a.z, 0x5410), a15 = prmt(a.x, a.z, 0x7632);
    const uint32_t b04 = prmt(b.x, b.z, 0x5410), b15 = prmt(b.x, b.z, 0x7632);
    const uint32_t a26 = prmt(a.y, a.w, 0x5410), a37 = prmt(a.y, a.w, 0x7632);
    const uint32_t b26 = prmt(b.y, b.w, 0x5410), b37 = prmt(b.y, b.w, 0x7632);
    mma_bf16(s[0], a04, b04, a15, b15, h04, h15);
    mma_bf16(s[0], a04, b04, a15, b15, l04, l15);
    mma_bf16(s[0], a26, b26, a37, b37, h26, h37);
    mma_bf16(s[0], a26, b26, a37, b37, l26, l37);
  }
  if (!ra) s[0][0] = s[0][1] = -CUDART_INF_F;
  if (!rb) s[0][2] = s[0][3] = -CUDART_INF_F;
  softmax_update<1>(st, s);

  const uint32_t xh0 = pack_bf2(s[0][0], s[0][1]), xh1 = pack_bf2(s[0][2], s[0][3]);
  const uint32_t xl0 = pack_bf2(s[0][0] - bf_lo(xh0), s[0][1] - bf_hi(xh0));
  const uint32_t xl1 = pack_bf2(s[0][2] - bf_lo(xh1), s[0][3] - bf_hi(xh1));
  const uint32_t bh0 = movmatrix_t(xh0), bh1 = movmatrix_t(xh1);
  const uint32_t bl0 = movmatrix_t(xl0), bl1 = movmatrix_t(xl1);
  const int ta = 2 * t;
  uint32_t zab[16], zcd[16];  // feature 16g + f, token pairs (ta, ta+1) and (ta+8, ta+9)
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int tk = ta + 8 * half;
    const bool v0 = tk < valid, v1 = tk + 1 < valid;
    uint32_t w0[8], w1[8];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint4 x = v0 ? *reinterpret_cast<const uint4 *>(vw + tk * 64 + 8 * g + 4 * j)
                         : make_uint4(0, 0, 0, 0);
      const uint4 y = v1 ? *reinterpret_cast<const uint4 *>(vw + (tk + 1) * 64 + 8 * g + 4 * j)
                         : make_uint4(0, 0, 0, 0);
      w0[4 * j + 0] = x.x; w0[4 * j + 1] = x.y; w0[4 * j + 2] = x.z; w0[4 * j + 3] = x.w;
      w1[4 * j + 0] = y.x; w1[4 * j + 1] = y.y; w1[4 * j + 2] = y.z; w1[4 * j + 3] = y.w;
    }
    uint32_t *z = half ? zcd : zab;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      z[2 * j] = prmt(w0[j], w1[j], 0x5410);
      z[2 * j + 1] = prmt(w0[j], w1[j], 0x7632);
    }
  }
#pragma unroll
  for (int f = 0; f < 8; ++f) {
    mma_bf16(st.o[f], zab[f], zab[8 + f], zcd[f], zcd[8 + f], bh0, bh1);
    mma_bf16(st.o[f], zab[f], zab[8 + f], zcd[f], zcd[8 + f], bl0, bl1);
  }
}

// ------------------------------------------------------------------ the kernel
struct __align__(16) DecodeSmem {
  uint8_t stage[kStages][kStageBytes];
  float red_o[kConsumers][kHeads][kD];
  float red_m[kConsumers][kHeads];
  float red_l[kConsumers][kHeads];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int abort_flag;
};

__device__ __forceinline__ void load_q(const DecodeArgs &a, long u, int g, int t,
                                       float (&qr)[32]) {
  const long row = u * kHeads + g;  // (b * Hkv + kvh) * 8 + g: query head kvh * 8 + g
  if (a.q_dtype == KVQ_F32) {
    const float *q = static_cast<const float *>(a.q) + row * kD + 32 * t;
#pragma unroll
    for (int i = 0; i < 32; ++i) qr[i] = q[i] * a.scale_log2;
  } else {
    const uint16_t *q = static_cast<const uint16_t *>(a.q) + row * kD + 32 * t;
#pragma unroll
    for (int i = 0; i < 32; ++i) qr[i] = bf16_to_f32(q[i]) * a.scale_log2;
  }
}

__device__ __forceinline__ bool aborted_flag(DecodeSmem &sm) {
  return *reinterpret_cast<volatile int *>(&sm.abort_flag) != 0;
}

__global__ void __launch_bounds__(kThreads, 2) decode_kernel(const DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  DecodeSmem &sm = *reinterpret_cast<DecodeSmem *>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long cta = blockIdx.x;
  const long lo = cta * a.total_items / a.num_ctas;
  const long hi = (cta + 1) * a.total_items / a.num_ctas;
  const long n_items = hi - lo;
  const long u_first = lo / a.ipu;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), 1);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumers) {
    // ---------------- loader
    if (lane == 0) {
      long k = 0;
      for (; k < n_items; ++k) {
        const int st = static_cast<int>(k % kStages);
        if (k >= kStages) {
          const uint32_t par = static_cast<uint32_t>((k / kStages - 1) & 1);
          if (!mbar_wait(smem_u32(&sm.empty[st]), par, a.ctl.wait_limit_ns)) {
            flag_error(a.ctl, KVQ_DEV_TIMEOUT);
            *reinterpret_cast<volatile int *>(&sm.abort_flag) = 1;
            break;
          }
        }
        if (aborted_flag(sm)) break;
        const long item = lo + k;
        if (item == a.ctl.drop_item) continue;  // test hook: this stage is never filled
        const long u = item / a.ipu;
        const int j = static_cast<int>(item % a.ipu);
        const uint32_t dst = smem_u32(sm.stage[st]);
        const uint32_t bar = smem_u32(&sm.full[st]);
        if (j < a.Gk) {
          const int valid = min(32, a.cut - 32 * j);
          const uint32_t vbytes = static_cast<uint32_t>(valid) * 64u;
          const uint32_t sbytes = static_cast<uint32_t>(valid) * 16u;
          mbar_arrive_expect_tx(bar, 2048u + 512u + vbytes + sbytes);
          bulk_g2s(dst, a.k_codes + (u * a.Gk + j) * 2048L, 2048u, bar);
          bulk_g2s(dst + kOffKScale, a.k_scales + (u * a.Gk + j) * 128L, 512u, bar);
          bulk_g2s(dst + kOffVCode, a.v_codes + (u * a.cut + 32L * j) * 64L, vbytes, bar);
          bulk_g2s(dst + kOffVScale, a.v_scales + (u * a.cut + 32L * j) * 4L, sbytes, bar);
        } else {
          const int w = j - a.Gk;
          const int valid = min(kWinTile, a.R - kWinTile * w);
          const uint32_t bytes = static_cast<uint32_t>(valid) * 256u;
          mbar_arrive_expect_tx(bar, 2u * bytes);
          bulk_g2s(dst, a.k_window + (u * a.R + kWinTile * w) * 128L, bytes, bar);
          bulk_g2s(dst + 4096, a.v_window + (u * a.R + kWinTile * w) * 128L, bytes, bar);
        }
      }
      // drain: copies still in flight must land before the CTA exits
      const long issued = k;
      for (long d = std::max(0L, issued - kStages); d < issued; ++d) {
        if (lo + d == a.ctl.drop_item) continue;
        mbar_wait(smem_u32(&sm.full[d % kStages]), static_cast<uint32_t>((d / kStages) & 1),
                  2000000000ull);
      }
    }
    return;
  }

  // ---------------- consumers
  const int g = lane >> 2, t = lane & 3;
  WarpState st;
  float qr[32];
  long k = warp;  // this warp's next item (CTA-relative)
  for (long u = u_first; u * a.ipu < hi; ++u) {
    state_reset(st);
    load_q(a, u, g, t, qr);
    const long u_end = std::min(hi, (u + 1) * a.ipu) - lo;  // CTA-relative end of unit u
    bool aborted = false;
    for (; k < u_end; k += kConsumers) {
      if (aborted_flag(sm)) {
        aborted = true;
        break;
      }
      const int s = static_cast<int>(k % kStages);
      if (!mbar_wait(smem_u32(&sm.full[s]), static_cast<uint32_t>((k / kStages) & 1),
                     a.ctl.wait_limit_ns)) {
        if (lane == 0) {
          flag_error(a.ctl, KVQ_DEV_TIMEOUT);
          *reinterpret_cast<volatile int *>(&sm.abort_flag) = 1;
        }
        aborted = true;
        break;
      }
      const int j = static_cast<int>((lo + k) % a.ipu);
      if (j < a.Gk)
        do_int4_item(st, sm.stage[s], qr, min(32, a.cut - 32 * j), g, t);
      else
        do_window_item(st, sm.stage[s], qr, min(kWinTile, a.R - kWinTile * (j - a.Gk)), g, t);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.empty[s]));
    }
    // ---- merge the 4 warps' states for unit u and write one partial
    float l0 = st.l[0], l1 = st.l[1];
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    if (g == 0) {
      sm.red_m[warp][2 * t] = st.m[0];
      sm.red_m[warp][2 * t + 1] = st.m[1];
      sm.red_l[warp][2 * t] = l0;
      sm.red_l[warp][2 * t + 1] = l1;
    }
#pragma unroll
    for (int f = 0; f < 8; ++f) {
      sm.red_o[warp][2 * t][16 * g + f] = st.o[f][0];
      sm.red_o[warp][2 * t + 1][16 * g + f] = st.o[f][1];
      sm.red_o[warp][2 * t][16 * g + 8 + f] = st.o[f][2];
      sm.red_o[warp][2 * t + 1][16 * g + 8 + f] = st.o[f][3];
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32));
    float *part = a.partials + ((cta * a.max_units + (u - u_first)) * kHeads) * kPartFloats;
    for (int i = threadIdx.x; i < kHeads * kD; i += kConsumers * 32) {
      const int h = i / kD, d = i % kD;
      float mx = -CUDART_INF_F;
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) mx = fmaxf(mx, sm.red_m[w][h]);
      float acc = 0.0f, lsum = 0.0f;
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) {
        const float c = (sm.red_m[w][h] == -CUDART_INF_F) ? 0.0f : exp2f(sm.red_m[w][h] - mx);
        acc += c * sm.red_o[w][h][d];
        lsum += c * sm.red_l[w][h];
      }
      part[h * kPartFloats + d] = acc;
      if (d == 0) {
        part[h * kPartFloats + kD] = mx;
        part[h * kPartFloats + kD + 1] = lsum;
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32));
    if (aborted || aborted_flag(sm)) break;
  }
}

// One warp per (unit, query head): merge the partials of every CTA whose
// slice overlaps the unit (log-sum-exp), normalise, store.
template <typename OT>
__global__ void __launch_bounds__(256) combine_kernel(const DecodeArgs a, OT *__restrict__ out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long u = blockIdx.x;
  const int h = warp;
  const long start = u * a.ipu, end = start + a.ipu;
  long c = start * a.num_ctas / a.total_items;
  while (c > 0 && (c * a.total_items / a.num_ctas) > start) --c;
  float m = -CUDART_INF_F, l = 0.0f, acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (; c < a.num_ctas; ++c) {
    const long clo = c * a.total_items / a.num_ctas, chi = (c + 1) * a.total_items / a.num_ctas;
    if (clo >= end) break;
    if (chi <= start) continue;
    const long slot = u - clo / a.ipu;
    if (slot < 0 || slot >= a.max_units) {
      if (lane == 0) flag_error(a.ctl, KVQ_DEV_BOUNDS);
      continue;
    }
    const float *p = a.partials + ((c * a.max_units + slot) * kHeads + h) * kPartFloats;
    const float pm = p[kD], pl = p[kD + 1];
    if (pm == -CUDART_INF_F) continue;
    const float nm = fmaxf(m, pm);
    const float c_old = exp2f(m - nm), c_new = exp2f(pm - nm);
    const float4 po = *reinterpret_cast<const float4 *>(p + 4 * lane);
    acc[0] = acc[0] * c_old + po.x * c_new;
    acc[1] = acc[1] * c_old + po.y * c_new;
    acc[2] = acc[2] * c_old + po.z * c_new;
    acc[3] = acc[3] * c_old + po.w * c_new;
    l = l * c_old + pl * c_new;
    m = nm;
  }
  const float inv = 1.0f / l;
  OT *o = out + (u * kHeads + h) * kD + 4 * lane;
#pragma unroll
  for (int i = 0; i < 4; ++i) store_from_f32(o + i, acc[i] * inv);
}

struct Plan {
  long total_items;
  int ipu, Wt, num_ctas, max_units;
};

Plan make_plan(const kvq_cache &c, int num_sms) {
  const CacheDims d = dims_of(c);
  Plan p;
  p.Wt = (d.R + kWinTile - 1) / kWinTile;
  p.ipu = d.Gk + p.Wt;
  p.total_items = static_cast<long>(d.B) * d.Hkv * p.ipu;
  p.num_ctas = static_cast<int>(std::min<long>(p.total_items, 2L * num_sms));
  const long per = (p.total_items + p.num_ctas - 1) / p.num_ctas;
  p.max_units = static_cast<int>((per + p.ipu - 1) / p.ipu + 1);
  return p;
}

}  // namespace

bool decode_supported(const kvq_cache &c, int q_dtype, int Hq, int n_q) {
  const bool win_ok = c.recent == 0 || (c.kwin_dtype == KVQ_BF16 && c.vwin_dtype == KVQ_BF16);
  return c.head_dim == kD && n_q == 1 && Hq == kHeads * c.kv_heads && win_ok &&
         (q_dtype == KVQ_BF16 || q_dtype == KVQ_F32) && c.n_tokens > 0;
}

size_t decode_workspace_bytes(const kvq_cache &c, int, int num_sms) {
  const Plan p = make_plan(c, num_sms);
  return sizeof(float) * static_cast<size_t>(p.num_ctas) * p.max_units * kHeads * kPartFloats;
}

int launch_attend_decode(const kvq_cache &c, const void *q, int q_dtype, float scale_log2,
                         void *out, int out_dtype, void *ws, const KernelCtl &ctl, int num_sms,
                         cudaStream_t s) {
  const CacheDims d = dims_of(c);
  const Plan p = make_plan(c, num_sms);
  DecodeArgs a;
  a.k_codes = c.k_codes;
  a.k_scales = c.k_scales;
  a.v_codes = c.v_codes;
  a.v_scales = c.v_scales;
  a.k_window = static_cast<const uint16_t *>(c.k_window);
  a.v_window = static_cast<const uint16_t *>(c.v_window);
  a.q = q;
  a.q_dtype = q_dtype;
  a.Hkv = d.Hkv;
  a.N = d.N;
  a.R = d.R;
  a.cut = d.cut;
  a.Gk = d.Gk;
  a.Wt = p.Wt;
  a.ipu = p.ipu;
  a.total_items = p.total_items;
  a.num_ctas = p.num_ctas;
  a.max_units = p.max_units;
  a.scale_log2 = scale_log2;
  a.partials = static_cast<float *>(ws);
  a.ctl = ctl;
  const size_t smem = sizeof(DecodeSmem);
  cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       static_cast<int>(smem));
  decode_kernel<<<p.num_ctas, kThreads, smem, s>>>(a);
  const unsigned units = static_cast<unsigned>(d.B) * d.Hkv;
  if (out_dtype == KVQ_F32)
    combine_kernel<float><<<units, kHeads * 32, 0, s>>>(a, static_cast<float *>(out));
  else
    combine_kernel<__nv_bfloat16><<<units, kHeads * 32, 0, s>>>(
        a, static_cast<__nv_bfloat16 *>(out));
  return 2;
}

// ------------------------------------------------------------------ library-owned scratch
// Scratch of kv_attend_decode_static: the split-K partials live in this
// file-scope device array instead of a caller-provided workspace. Every GPU
// that loads this module keeps the array until the process exits.
namespace {
constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];
std::mutex g_scratch_mu;
void *g_scratch_addr[64] = {};
}  // namespace

size_t decode_static_scratch_limit() { return kStaticScratchBytes; }

// In host code `g_decode_scratch` is only a host-side stand-in; the kernel
// needs its device address, resolved once per device with that device current.
cudaError_t decode_static_scratch(void **ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *ptr = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace kvq
