// Split-K decode attention over an int4 KV cache: one query row per
// (sequence, query head), 8 query heads per KV head (GQA), head dim 128.
//
// What it computes: O = softmax(sm_scale * q K^T) V over all N tokens, K and V
// dequantized from grouped int4 (residual-window page, section 固定預算) or
// read from the bf16 window of the last R tokens; no mask.
//
// Work split. The cache of one (sequence, KV head) -- a "unit" -- is a list
// of items: its int4 groups taken four at a time (128 tokens: 8 KB K codes,
// 2 KB K scales, 8 KB V codes, 2 KB V scales, one bulk copy each) followed by
// its window tiles (40 tokens of bf16 K and V). All items of all units are
// laid end to end and the persistent grid (3 CTAs per SM) takes equal
// contiguous slices, so every SM streams the same number of bytes. A CTA
// emits one partial (running max m, sum l, unnormalised O for 8 heads) per
// unit its slice touches, into the unit's slot for that CTA; combine_kernel,
// launched as a programmatic dependent of this grid, merges a unit's slots
// with the log-sum-exp rule.
//
// Inside a CTA. Warp 4 is the loader: one lane issues the copies of each item
// into a 3-stage shared-memory ring, completing on mbarriers. Consumer warp w
// takes group w of every item (window rows 10w..10w+9). Scores use mma.sync
// m16n8k16 with the 16 tokens of a tile as M and the 8 query heads as N: the
// K scales of a group are folded into q (q' = q * sm_scale * log2 e * s_k,
// fp16), the nibbles are turned into fp16 codes with two bit masks and one
// subtraction, so the MMA sees codes in [-7, 7] exactly. P (fp16) is
// transposed in registers with movmatrix and multiplies V^T (features as M)
// whose codes are scaled by the token's V scale in fp16. The bf16 window uses
// bf16 MMAs with q and P split into hi + lo bf16 parts. Softmax runs in the
// log2 domain with fp32 state.
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
#ifndef KVQ_DECODE_CTAS_PER_SM
#define KVQ_DECODE_CTAS_PER_SM 3
#endif
#ifndef KVQ_DECODE_STAGES
#define KVQ_DECODE_STAGES 3
#endif
constexpr int kStages = KVQ_DECODE_STAGES;          // ring depth per CTA
constexpr int kCtasPerSm = KVQ_DECODE_CTAS_PER_SM;  // resident CTAs per SM
constexpr int kGroupsPerItem = kConsumers;          // one K group per consumer warp
constexpr int kWinTile = 10;                        // window tokens per consumer warp
constexpr int kWinItem = kWinTile * kConsumers;     // window tokens per item
constexpr int kPartFloats = kD + 4;    // O[128], m, l per head, padded to 16 bytes
// int4 item (4 K groups = 128 tokens): K codes [4][2048], K scales [4][512],
// V codes [128][64], V scales [128][16]
constexpr int kOffKScale = 8192, kOffVCode = 10240, kOffVScale = 18432;
constexpr int kStageBytes = 20480;
// window item (40 tokens): K rows [40][256 B] at 0, V rows at kOffVWin
constexpr int kOffVWin = 10240;

struct DecodeArgs {
  const uint8_t *k_codes;
  const float *k_scales;
  const uint8_t *v_codes;
  const float *v_scales;
  const uint16_t *k_window;
  const uint16_t *v_window;
  const void *q;
  int q_dtype;
  int Hkv, N, R, cut, Gk, Wt, ipu;  // ipu: items per unit = ceil(Gk / 4) + Wt
  int Gi;                           // int4 items per unit = ceil(Gk / 4)
  int Gs, Vs, Ws;                   // per-unit strides: K groups, V rows, window rows
  int total_items;
  int num_ctas, max_ctas_per_unit;
  float scale_log2;
  float *partials;                  // [units][max_ctas_per_unit][8][132]
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

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t as_u32(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 as_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// (w & kMask) | kMagic as one three-input logic op.
template <uint32_t kMask, uint32_t kMagic>
__device__ __forceinline__ uint32_t and_or(uint32_t w) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(w), "n"(kMask), "n"(kMagic));
  return d;
}

// Nibbles at bits 0-3 and 16-19 -> fp16 codes: 0x6400 | n is 1024 + n, n = code + 8.
__device__ __forceinline__ uint32_t dq_lo(uint32_t w) {
  const uint32_t x = and_or<0x000F000Fu, 0x64006400u>(w);
  return as_u32(__hsub2(as_h2(x), as_h2(0x64086408u)));  // 1032
}
// Nibbles at bits 4-7 and 20-23: 0x5400 | n << 4 is 64 + n.
__device__ __forceinline__ uint32_t dq_hi(uint32_t w) {
  const uint32_t x = and_or<0x00F000F0u, 0x54005400u>(w);
  return as_u32(__hsub2(as_h2(x), as_h2(0x54805480u)));  // 72
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  return as_u32(__floats2half2_rn(lo, hi));
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
// The reference maximum m is only raised when some score of the tile exceeds
// it by more than kLazy (log2 units), so most tiles need no cross-lane
// reduction; probabilities are then at most 2^kLazy, well inside fp16, and
// the result is unchanged because O and l share the reference.
constexpr float kLazy = 8.0f;

template <int NT>
__device__ __forceinline__ void softmax_update(WarpState &st, float (&s)[NT][4]) {
  float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    mx0 = fmaxf(mx0, fmaxf(s[i][0], s[i][2]));
    mx1 = fmaxf(mx1, fmaxf(s[i][1], s[i][3]));
  }
  if (__any_sync(0xffffffffu, mx0 > st.m[0] + kLazy || mx1 > st.m[1] + kLazy)) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    const float n0 = fmaxf(st.m[0], mx0), n1 = fmaxf(st.m[1], mx1);
    const float c0 = fast_exp2(st.m[0] - n0), c1 = fast_exp2(st.m[1] - n1);
    st.m[0] = n0;
    st.m[1] = n1;
    st.l[0] *= c0;
    st.l[1] *= c1;
#pragma unroll
    for (int f = 0; f < 8; ++f) {
      st.o[f][0] *= c0;
      st.o[f][1] *= c1;
      st.o[f][2] *= c0;
      st.o[f][3] *= c1;
    }
  }
  float sum0 = 0.0f, sum1 = 0.0f;
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    s[i][0] = fast_exp2(s[i][0] - st.m[0]);
    s[i][1] = fast_exp2(s[i][1] - st.m[1]);
    s[i][2] = fast_exp2(s[i][2] - st.m[0]);
    s[i][3] = fast_exp2(s[i][3] - st.m[1]);
    sum0 += s[i][0] + s[i][2];
    sum1 += s[i][1] + s[i][3];
  }
  st.l[0] += sum0;
  st.l[1] += sum1;
}

// ------------------------------------------------------------------ item bodies
// int4 group: 32 tokens (two m-tiles), `valid` of them real; kFull: all 32.
// q of this thread: head g, features 32t + 8i + j, held as fp16 pairs
// qh[i][j] = (q[8i + j], q[8i + 4 + j]) in the MMA's feature order.
template <bool kFull>
__device__ __forceinline__ void do_int4_item(WarpState &st, const uint8_t *kc, const float *ks,
                                             const uint8_t *vc, const float *vs,
                                             const uint32_t (&qh)[4][4], int valid, int g, int t) {
  // q' = q * (K scale of the channel) for this group, as fp16 B fragments
  uint32_t bq[8][2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 s0 = *reinterpret_cast<const float4 *>(ks + 32 * t + 8 * i);
    const float4 s1 = *reinterpret_cast<const float4 *>(ks + 32 * t + 8 * i + 4);
    bq[2 * i][0] = as_u32(__hmul2(as_h2(qh[i][0]), __floats2half2_rn(s0.x, s1.x)));
    bq[2 * i][1] = as_u32(__hmul2(as_h2(qh[i][1]), __floats2half2_rn(s0.y, s1.y)));
    bq[2 * i + 1][0] = as_u32(__hmul2(as_h2(qh[i][2]), __floats2half2_rn(s0.z, s1.z)));
    bq[2 * i + 1][1] = as_u32(__hmul2(as_h2(qh[i][3]), __floats2half2_rn(s0.w, s1.w)));
  }
  float s[2][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const int r0 = 16 * mt + g;
    const uint4 ka = *reinterpret_cast<const uint4 *>(kc + r0 * 64 + 16 * t);
    const uint4 kb = *reinterpret_cast<const uint4 *>(kc + (r0 + 8) * 64 + 16 * t);
    const uint32_t wa[4] = {ka.x, ka.y, ka.z, ka.w}, wb[4] = {kb.x, kb.y, kb.z, kb.w};
    float e[4] = {0.0f, 0.0f, 0.0f, 0.0f}, o[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // two MMA chains
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      mma_f16(e, dq_lo(wa[i]), dq_lo(wb[i]), dq_hi(wa[i]), dq_hi(wb[i]), bq[2 * i][0],
              bq[2 * i][1]);
      const uint32_t a8 = wa[i] >> 8, b8 = wb[i] >> 8;
      mma_f16(o, dq_lo(a8), dq_lo(b8), dq_hi(a8), dq_hi(b8), bq[2 * i + 1][0],
              bq[2 * i + 1][1]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) s[mt][j] = e[j] + o[j];
    if (!kFull) {
      if (r0 >= valid) s[mt][0] = s[mt][1] = -CUDART_INF_F;
      if (r0 + 8 >= valid) s[mt][2] = s[mt][3] = -CUDART_INF_F;
    }
  }
  softmax_update<2>(st, s);

  const uint2 zero8 = make_uint2(0x88888888u, 0x88888888u);  // code 0 everywhere
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const uint32_t b0 = movmatrix_t(pack_h2(s[mt][0], s[mt][1]));
    const uint32_t b1 = movmatrix_t(pack_h2(s[mt][2], s[mt][3]));
    const int ta = 16 * mt + 2 * t;  // tokens ta, ta+1, ta+8, ta+9
    const bool va = kFull || ta < valid, vb = kFull || ta + 1 < valid;
    const bool vcv = kFull || ta + 8 < valid, vd = kFull || ta + 9 < valid;
    const uint2 za = va ? *reinterpret_cast<const uint2 *>(vc + ta * 64 + 8 * g) : zero8;
    const uint2 zb = vb ? *reinterpret_cast<const uint2 *>(vc + (ta + 1) * 64 + 8 * g) : zero8;
    const uint2 zc = vcv ? *reinterpret_cast<const uint2 *>(vc + (ta + 8) * 64 + 8 * g) : zero8;
    const uint2 zd = vd ? *reinterpret_cast<const uint2 *>(vc + (ta + 9) * 64 + 8 * g) : zero8;
    const float sa = va ? vs[ta * 4 + (g >> 1)] : 0.0f;
    const float sb = vb ? vs[(ta + 1) * 4 + (g >> 1)] : 0.0f;
    const float sc = vcv ? vs[(ta + 8) * 4 + (g >> 1)] : 0.0f;
    const float sd = vd ? vs[(ta + 9) * 4 + (g >> 1)] : 0.0f;
    const __half2 sab = __floats2half2_rn(sa, sb), scd = __floats2half2_rn(sc, sd);
    // Feature 16g + f of the token pair (ta, ta+1) comes from byte-permuted
    // words: f = 8w + 4h + j, w = which 8-byte word, h = low/high 2 bytes,
    // j = nibble position. M-tile f (f < 8) takes features 16g + f (row g)
    // and 16g + 8 + f (row g+8), so the A operands of one m-tile are built
    // right before its MMA.
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t sel = h ? 0x7632u : 0x5410u;
      const uint32_t xab0 = prmt(za.x, zb.x, sel), xab1 = prmt(za.y, zb.y, sel);
      const uint32_t xcd0 = prmt(zc.x, zd.x, sel), xcd1 = prmt(zc.y, zd.y, sel);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t a0 = j < 2 ? xab0 : xab0 >> 8, a1 = j < 2 ? xab1 : xab1 >> 8;
        const uint32_t c0 = j < 2 ? xcd0 : xcd0 >> 8, c1 = j < 2 ? xcd1 : xcd1 >> 8;
        const bool hi_nib = j & 1;
        const uint32_t r0 = as_u32(__hmul2(as_h2(hi_nib ? dq_hi(a0) : dq_lo(a0)), sab));
        const uint32_t r1 = as_u32(__hmul2(as_h2(hi_nib ? dq_hi(a1) : dq_lo(a1)), sab));
        const uint32_t r2 = as_u32(__hmul2(as_h2(hi_nib ? dq_hi(c0) : dq_lo(c0)), scd));
        const uint32_t r3 = as_u32(__hmul2(as_h2(hi_nib ? dq_hi(c1) : dq_lo(c1)), scd));
        mma_f16(st.o[4 * h + j], r0, r1, r2, r3, b0, b1);
      }
    }
  }
}

// bf16 window tile: 16 tokens, `valid` of them real.
__device__ __forceinline__ void do_window_item(WarpState &st, const uint32_t *kw,
                                               const uint32_t *vw, const uint32_t (&qh)[4][4],
                                               int valid, int g, int t) {
  // kw, vw: this warp's token rows, 64 words (128 bf16) each; rows >= valid unread
  float s[1][4] = {{0.0f, 0.0f, 0.0f, 0.0f}};
  const bool ra = g < valid, rb = g + 8 < valid;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    // features 32t + 8i .. +7 of rows g and g+8
    const uint4 a = ra ? *reinterpret_cast<const uint4 *>(kw + g * 64 + 16 * t + 4 * i)
                       : make_uint4(0, 0, 0, 0);
    const uint4 b = rb ? *reinterpret_cast<const uint4 *>(kw + (g + 8) * 64 + 16 * t + 4 * i)
                       : make_uint4(0, 0, 0, 0);
    const float2 f04 = __half22float2(as_h2(qh[i][0])), f15 = __half22float2(as_h2(qh[i][1]));
    const float2 f26 = __half22float2(as_h2(qh[i][2])), f37 = __half22float2(as_h2(qh[i][3]));
    const float q0 = f04.x, q4 = f04.y, q1 = f15.x, q5 = f15.y;
    const float q2 = f26.x, q6 = f26.y, q3 = f37.x, q7 = f37.y;
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
  // Word j of a token row slice holds features 16g + 2j, 2j+1. M-tiles 2j and
  // 2j+1 need words j (rows g) and 4 + j (rows g+8) of the tokens ta, ta+1,
  // ta+8, ta+9; invalid tokens read as zero.
  const bool v0 = ta < valid, v1 = ta + 1 < valid, v2 = ta + 8 < valid, v3 = ta + 9 < valid;
  const uint32_t *r0 = vw + ta * 64 + 8 * g, *r1 = r0 + 64, *r2 = r0 + 8 * 64, *r3 = r0 + 9 * 64;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t a_lo = v0 ? r0[j] : 0u, b_lo = v1 ? r1[j] : 0u;
    const uint32_t a_hi = v0 ? r0[4 + j] : 0u, b_hi = v1 ? r1[4 + j] : 0u;
    const uint32_t c_lo = v2 ? r2[j] : 0u, d_lo = v3 ? r3[j] : 0u;
    const uint32_t c_hi = v2 ? r2[4 + j] : 0u, d_hi = v3 ? r3[4 + j] : 0u;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const uint32_t sel = e ? 0x7632u : 0x5410u;
      const uint32_t x0 = prmt(a_lo, b_lo, sel), x1 = prmt(a_hi, b_hi, sel);
      const uint32_t x2 = prmt(c_lo, d_lo, sel), x3 = prmt(c_hi, d_hi, sel);
      mma_bf16(st.o[2 * j + e], x0, x1, x2, x3, bh0, bh1);
      mma_bf16(st.o[2 * j + e], x0, x1, x2, x3, bl0, bl1);
    }
  }
}

// ------------------------------------------------------------------ the kernel
struct __align__(16) DecodeSmem {
  uint8_t stage[kStages][kStageBytes];
  float red_o[kConsumers][kHeads / 2][kD];  // one half of the heads at a time
  float red_m[kConsumers][kHeads];
  float red_l[kConsumers][kHeads];
  float red_c[kConsumers][kHeads];  // merge weight of warp w's state for head h
  float red_mx[kHeads], red_ls[kHeads];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int abort_flag;
};

__device__ __forceinline__ void load_q(const DecodeArgs &a, int u, int g, int t,
                                       uint32_t (&qh)[4][4]) {
  const long row = static_cast<long>(u) * kHeads + g;  // query head kvh * 8 + g of sequence b
  float qr[32];
  if (a.q_dtype == KVQ_F32) {
    const float *q = static_cast<const float *>(a.q) + row * kD + 32 * t;
    const bool ok = in_bounds(a.ctl, q, 32 * sizeof(float));
#pragma unroll
    for (int i = 0; i < 32; ++i) qr[i] = ok ? q[i] * a.scale_log2 : 0.0f;
  } else {
    const uint16_t *q = static_cast<const uint16_t *>(a.q) + row * kD + 32 * t;
    const bool ok = in_bounds(a.ctl, q, 32 * sizeof(uint16_t));
#pragma unroll
    for (int i = 0; i < 32; ++i) qr[i] = ok ? bf16_to_f32(q[i]) * a.scale_log2 : 0.0f;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) qh[i][j] = pack_h2(qr[8 * i + j], qr[8 * i + 4 + j]);
}

// A bf16 query slice (this lane's 32 features of head g) as loaded, so that
// the next unit's loads can be issued before the current unit's merge and
// their latency hidden by it.
struct QRaw {
  uint4 w[4];
};

__device__ __forceinline__ void load_q_raw(const DecodeArgs &a, int u, int g, int t, QRaw &r) {
  if (a.q_dtype == KVQ_F32) return;  // fp32 rows are loaded when converted
  const long row = static_cast<long>(u) * kHeads + g;
  const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.q) + row * kD +
                                                   32 * t);
  const bool ok = in_bounds(a.ctl, p, 4 * sizeof(uint4));
#pragma unroll
  for (int i = 0; i < 4; ++i) r.w[i] = ok ? p[i] : make_uint4(0u, 0u, 0u, 0u);
}

// load_q from a prefetched bf16 slice (the same values).
__device__ __forceinline__ void q_from_raw(const DecodeArgs &a, int u, int g, int t,
                                           const QRaw &r, uint32_t (&qh)[4][4]) {
  if (a.q_dtype == KVQ_F32) {
    load_q(a, u, g, t, qh);
    return;
  }
  float qr[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w[4] = {r.w[i].x, r.w[i].y, r.w[i].z, r.w[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      qr[8 * i + 2 * j] = __uint_as_float(w[j] << 16) * a.scale_log2;
      qr[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u) * a.scale_log2;
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) qh[i][j] = pack_h2(qr[8 * i + j], qr[8 * i + 4 + j]);
}

__device__ __forceinline__ bool aborted_flag(DecodeSmem &sm) {
  return *reinterpret_cast<volatile int *>(&sm.abort_flag) != 0;
}

// Issue the copies of item `item` (unit u, index j within the unit) into a stage.
__device__ __forceinline__ void load_item(const DecodeArgs &a, int u, int j, uint32_t dst,
                                          uint32_t bar) {
  if (j < a.Gi) {
    const int g0 = kGroupsPerItem * j;
    const int ng = min(kGroupsPerItem, a.Gk - g0);
    const int t0 = 32 * g0;
    const int nt = min(32 * kGroupsPerItem, a.cut - t0);
    const long gi = static_cast<long>(u) * a.Gs + g0;
    const long ti = static_cast<long>(u) * a.Vs + t0;
    const uint32_t kb = 2048u * ng, sb = 512u * ng, vb = 64u * nt, wb = 16u * nt;
    // a copy whose source fails the bounds check is neither issued nor expected
    const bool ok0 = in_bounds(a.ctl, a.k_codes + gi * 2048, kb);
    const bool ok1 = in_bounds(a.ctl, a.k_scales + gi * 128, sb);
    const bool ok2 = in_bounds(a.ctl, a.v_codes + ti * 64, vb);
    const bool ok3 = in_bounds(a.ctl, a.v_scales + ti * 4, wb);
    mbar_arrive_expect_tx(bar, (ok0 ? kb : 0u) + (ok1 ? sb : 0u) + (ok2 ? vb : 0u) + (ok3 ? wb : 0u));
    if (ok0) bulk_g2s(dst, a.k_codes + gi * 2048, kb, bar);
    if (ok1) bulk_g2s(dst + kOffKScale, a.k_scales + gi * 128, sb, bar);
    if (ok2) bulk_g2s(dst + kOffVCode, a.v_codes + ti * 64, vb, bar);
    if (ok3) bulk_g2s(dst + kOffVScale, a.v_scales + ti * 4, wb, bar);
  } else {
    const int w0 = kWinItem * (j - a.Gi);
    const int nt = min(kWinItem, a.R - w0);
    const long wi = static_cast<long>(u) * a.Ws + w0;
    const uint32_t bytes = 256u * nt;
    const bool ok0 = in_bounds(a.ctl, a.k_window + wi * 128, bytes);
    const bool ok1 = in_bounds(a.ctl, a.v_window + wi * 128, bytes);
    mbar_arrive_expect_tx(bar, (ok0 ? bytes : 0u) + (ok1 ? bytes : 0u));
    if (ok0) bulk_g2s(dst, a.k_window + wi * 128, bytes, bar);
    if (ok1) bulk_g2s(dst + kOffVWin, a.v_window + wi * 128, bytes, bar);
  }
}

// First CTA of the persistent grid whose slice holds item x: the largest c
// with floor(c * T / C) <= x.
__device__ __forceinline__ int cta_of_item(const DecodeArgs &a, int x) {
  return static_cast<int>(((static_cast<long>(x) + 1) * a.num_ctas - 1) / a.total_items);
}

__device__ __forceinline__ float *partial_of(const DecodeArgs &a, int u, int slot) {
  return a.partials + (static_cast<long>(u) * a.max_ctas_per_unit + slot) * (kHeads * kPartFloats);
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm) decode_kernel(const DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  DecodeSmem &sm = *reinterpret_cast<DecodeSmem *>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const int lo = static_cast<int>(static_cast<long>(cta) * a.total_items / a.num_ctas);
  const int hi = static_cast<int>(static_cast<long>(cta + 1) * a.total_items / a.num_ctas);
  const int n_items = hi - lo;
  const int u_first = lo / a.ipu;

  // The combine launch may start placing its blocks as this grid drains; it
  // waits for the whole grid before reading any partial.
  allow_next_grid();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), kConsumers);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // The previous kernel may still be running (the last call's combine reads
  // the partial slots this grid rewrites; a kv_pack may be writing the cache).
  wait_prior_grid();

  if (warp == kConsumers) {
    // ---------------- loader: one lane walks the CTA's items in order
    if (lane == 0) {
      int k = 0, u = u_first, j = lo - u_first * a.ipu;
      for (; k < n_items; ++k) {
        const int st = k % kStages;
        if (k >= kStages) {
          const uint32_t par = static_cast<uint32_t>((k / kStages - 1) & 1);
          if (!mbar_wait(smem_u32(&sm.empty[st]), par, a.ctl.wait_limit_ns)) {
            flag_error(a.ctl, KVQ_DEV_TIMEOUT);
            *reinterpret_cast<volatile int *>(&sm.abort_flag) = 1;
            break;
          }
        }
        if (aborted_flag(sm)) break;
        if (lo + k != a.ctl.drop_item)  // test hook: a dropped stage is never filled
          load_item(a, u, j, smem_u32(sm.stage[st]), smem_u32(&sm.full[st]));
        if (++j == a.ipu) {
          j = 0;
          ++u;
        }
      }
      // drain: copies still in flight must land before the CTA exits
      for (int d = max(0, k - kStages); d < k; ++d) {
        if (lo + d == a.ctl.drop_item) continue;
        mbar_wait(smem_u32(&sm.full[d % kStages]), static_cast<uint32_t>((d / kStages) & 1),
                  2000000000ull);
      }
    }
    return;
  }

  // ---------------- consumers: warp w takes group w (or window rows 10w..) of every item
  const int g = lane >> 2, t = lane & 3;
  WarpState st;
  uint32_t qh[4][4];
  QRaw qraw;
  load_q_raw(a, u_first, g, t, qraw);
  int k = 0;  // CTA-relative item index
  for (int u = u_first; u * a.ipu < hi; ++u) {
    state_reset(st);
    q_from_raw(a, u, g, t, qraw, qh);
    const int u_end = min(hi, (u + 1) * a.ipu) - lo;  // CTA-relative end of unit u
    int j = lo + k - u * a.ipu;                        // item index within unit u
    bool aborted = false;
    for (; k < u_end; ++k, ++j) {
      if (aborted_flag(sm)) {
        aborted = true;
        break;
      }
      const int s = k % kStages;
      if (!mbar_wait(smem_u32(&sm.full[s]), static_cast<uint32_t>((k / kStages) & 1),
                     a.ctl.wait_limit_ns)) {
        if (lane == 0) {
          flag_error(a.ctl, KVQ_DEV_TIMEOUT);
          *reinterpret_cast<volatile int *>(&sm.abort_flag) = 1;
        }
        aborted = true;
        break;
      }
      const uint8_t *stg = sm.stage[s];
      if (j < a.Gi) {
        const int grp = kGroupsPerItem * j + warp;
        const int valid = a.cut - 32 * grp;
        const uint8_t *kc = stg + warp * 2048, *vc = stg + kOffVCode + warp * 2048;
        const float *ks = reinterpret_cast<const float *>(stg + kOffKScale + warp * 512);
        const float *vs = reinterpret_cast<const float *>(stg + kOffVScale + warp * 512);
        if (valid >= 32)
          do_int4_item<true>(st, kc, ks, vc, vs, qh, 32, g, t);
        else if (valid > 0)
          do_int4_item<false>(st, kc, ks, vc, vs, qh, valid, g, t);
      } else {
        const int r0 = kWinItem * (j - a.Gi) + kWinTile * warp;
        if (r0 < a.R)
          do_window_item(st, reinterpret_cast<const uint32_t *>(stg + warp * kWinTile * 256),
                         reinterpret_cast<const uint32_t *>(stg + kOffVWin + warp * kWinTile * 256),
                         qh, min(kWinTile, a.R - r0), g, t);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.empty[s]));
    }
    // the next unit's query rows are in flight during the merge
    if ((u + 1) * a.ipu < hi) load_q_raw(a, u + 1, g, t, qraw);
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
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32));
    // per head: the maximum over the warps, each warp's weight and the sum
    if (threadIdx.x < kHeads) {
      const int h = threadIdx.x;
      float mx = -CUDART_INF_F;
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) mx = fmaxf(mx, sm.red_m[w][h]);
      float lsum = 0.0f;
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) {
        const float c = (sm.red_m[w][h] == -CUDART_INF_F) ? 0.0f : exp2f(sm.red_m[w][h] - mx);
        sm.red_c[w][h] = c;
        lsum += c * sm.red_l[w][h];
      }
      sm.red_mx[h] = mx;
      sm.red_ls[h] = lsum;
    }
    // heads 0-3 live in lanes with t < 2, heads 4-7 in lanes with t >= 2:
    // merge one half at a time through red_o
    float *part = partial_of(a, u, cta - cta_of_item(a, u * a.ipu));
    const bool part_ok = in_bounds(a.ctl, part, sizeof(float) * kHeads * kPartFloats);
    for (int half = 0; half < 2; ++half) {
      if ((t >> 1) == half) {
        const int h0 = 2 * t - 4 * half;
        float4 *ra = reinterpret_cast<float4 *>(&sm.red_o[warp][h0][16 * g]);
        float4 *rb = reinterpret_cast<float4 *>(&sm.red_o[warp][h0 + 1][16 * g]);
        ra[0] = make_float4(st.o[0][0], st.o[1][0], st.o[2][0], st.o[3][0]);
        ra[1] = make_float4(st.o[4][0], st.o[5][0], st.o[6][0], st.o[7][0]);
        ra[2] = make_float4(st.o[0][2], st.o[1][2], st.o[2][2], st.o[3][2]);
        ra[3] = make_float4(st.o[4][2], st.o[5][2], st.o[6][2], st.o[7][2]);
        rb[0] = make_float4(st.o[0][1], st.o[1][1], st.o[2][1], st.o[3][1]);
        rb[1] = make_float4(st.o[4][1], st.o[5][1], st.o[6][1], st.o[7][1]);
        rb[2] = make_float4(st.o[0][3], st.o[1][3], st.o[2][3], st.o[3][3]);
        rb[3] = make_float4(st.o[4][3], st.o[5][3], st.o[6][3], st.o[7][3]);
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32));
      for (int i = threadIdx.x; i < (kHeads / 2) * kD; i += kConsumers * 32) {
        const int hh = i / kD, d = i % kD, h = 4 * half + hh;
        float acc = 0.0f;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) acc += sm.red_c[w][h] * sm.red_o[w][hh][d];
        if (!part_ok) continue;
        part[h * kPartFloats + d] = acc;
        if (d == 0) {
          part[h * kPartFloats + kD] = sm.red_mx[h];
          part[h * kPartFloats + kD + 1] = sm.red_ls[h];
        }
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32));
    }
    if (aborted || aborted_flag(sm)) break;
  }
}

// One warp per (unit, query head): merge the partials of the CTAs whose
// slices overlap the unit (log-sum-exp), normalise, store. The partials of
// unit u sit in consecutive slots, one per overlapping CTA; they are read
// sixteen at a time with all loads of a batch in flight together.
template <typename OT>
__global__ void __launch_bounds__(256) combine_kernel(const DecodeArgs a, OT *__restrict__ out) {
  wait_prior_grid();
  allow_next_grid();  // the next call's decode grid may be placed while this one runs
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x;
  const int h = warp;
  const int n = cta_of_item(a, (u + 1) * a.ipu - 1) - cta_of_item(a, u * a.ipu) + 1;
  const float *base = partial_of(a, u, 0) + h * kPartFloats;
  constexpr int kSlot = kHeads * kPartFloats;
#ifdef KVQ_DEBUG
  // the unit's partial slots and this head's output row (the same in every lane)
  if (!in_bounds(a.ctl, base - h * kPartFloats, sizeof(float) * n * kSlot) ||
      !in_bounds(a.ctl, out + (static_cast<long>(u) * kHeads + h) * kD, kD * sizeof(OT)))
    return;
#endif
  constexpr int kBatch = 16;
  float m = -CUDART_INF_F, l = 0.0f;
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (int c0 = 0; c0 < n; c0 += kBatch) {
    float pm[kBatch], pl[kBatch];
    float4 po[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const float *p = base + static_cast<long>(min(c0 + i, n - 1)) * kSlot;
      const float2 ml = *reinterpret_cast<const float2 *>(p + kD);
      pm[i] = c0 + i < n ? ml.x : -CUDART_INF_F;
      pl[i] = ml.y;
      po[i] = *reinterpret_cast<const float4 *>(p + 4 * lane);
    }
    float nm = m;
#pragma unroll
    for (int i = 0; i < kBatch; ++i) nm = fmaxf(nm, pm[i]);
    if (nm == -CUDART_INF_F) continue;
    const float r = exp2f(m - nm);  // 0 while m is -inf
    l *= r;
    acc.x *= r;
    acc.y *= r;
    acc.z *= r;
    acc.w *= r;
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const float w = exp2f(pm[i] - nm);  // 0 for empty and padded slots
      l += w * pl[i];
      acc.x += w * po[i].x;
      acc.y += w * po[i].y;
      acc.z += w * po[i].z;
      acc.w += w * po[i].w;
    }
    m = nm;
  }
  const float inv = 1.0f / l;
  OT *o = out + (static_cast<long>(u) * kHeads + h) * kD + 4 * lane;
  store_from_f32(o + 0, acc.x * inv);
  store_from_f32(o + 1, acc.y * inv);
  store_from_f32(o + 2, acc.z * inv);
  store_from_f32(o + 3, acc.w * inv);
}

// The same merge for units whose partials come from many CTAs (small
// batches, where each unit spans a large share of the grid): one block per
// (unit, query head), warp w merging slots w, w + 8, ..., then the eight
// warps' states merged through shared memory.
constexpr int kWideCombineAbove = 32;  // slots per unit above which it is used

template <typename OT>
__global__ void __launch_bounds__(256) combine_wide_kernel(const DecodeArgs a,
                                                           OT *__restrict__ out) {
  wait_prior_grid();
  allow_next_grid();
  __shared__ float sm_m[8], sm_l[8];
  __shared__ float4 sm_acc[8][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x, h = blockIdx.y;
  const int n = cta_of_item(a, (u + 1) * a.ipu - 1) - cta_of_item(a, u * a.ipu) + 1;
  const float *base = partial_of(a, u, 0) + h * kPartFloats;
  constexpr int kSlot = kHeads * kPartFloats;
#ifdef KVQ_DEBUG
  if (!in_bounds(a.ctl, base - h * kPartFloats, sizeof(float) * n * kSlot) ||
      !in_bounds(a.ctl, out + (static_cast<long>(u) * kHeads + h) * kD, kD * sizeof(OT)))
    return;
#endif
  constexpr int kBatch = 8;
  float m = -CUDART_INF_F, l = 0.0f;
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (int c0 = warp; c0 < n; c0 += 8 * kBatch) {
    float pm[kBatch], pl[kBatch];
    float4 po[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int c = c0 + 8 * i;
      const float *p = base + static_cast<long>(min(c, n - 1)) * kSlot;
      const float2 ml = *reinterpret_cast<const float2 *>(p + kD);
      pm[i] = c < n ? ml.x : -CUDART_INF_F;
      pl[i] = ml.y;
      po[i] = *reinterpret_cast<const float4 *>(p + 4 * lane);
    }
    float nm = m;
#pragma unroll
    for (int i = 0; i < kBatch; ++i) nm = fmaxf(nm, pm[i]);
    if (nm == -CUDART_INF_F) continue;
    const float r = exp2f(m - nm);  // 0 while m is -inf
    l *= r;
    acc.x *= r;
    acc.y *= r;
    acc.z *= r;
    acc.w *= r;
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const float w = exp2f(pm[i] - nm);  // 0 for empty and padded slots
      l += w * pl[i];
      acc.x += w * po[i].x;
      acc.y += w * po[i].y;
      acc.z += w * po[i].z;
      acc.w += w * po[i].w;
    }
    m = nm;
  }
  sm_acc[warp][lane] = acc;
  if (lane == 0) {
    sm_m[warp] = m;
    sm_l[warp] = l;
  }
  __syncthreads();
  if (warp != 0) return;
  float mx = -CUDART_INF_F;
#pragma unroll
  for (int w = 0; w < 8; ++w) mx = fmaxf(mx, sm_m[w]);
  float ls = 0.0f;
  float4 o4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const float c = sm_m[w] == -CUDART_INF_F ? 0.0f : exp2f(sm_m[w] - mx);
    const float4 x = sm_acc[w][lane];
    ls += c * sm_l[w];
    o4.x += c * x.x;
    o4.y += c * x.y;
    o4.z += c * x.z;
    o4.w += c * x.w;
  }
  const float inv = 1.0f / ls;
  OT *o = out + (static_cast<long>(u) * kHeads + h) * kD + 4 * lane;
  store_from_f32(o + 0, o4.x * inv);
  store_from_f32(o + 1, o4.y * inv);
  store_from_f32(o + 2, o4.z * inv);
  store_from_f32(o + 3, o4.w * inv);
}

struct Plan {
  int total_items;
  int ipu, Gi, Wt, num_ctas, max_ctas_per_unit;
  long units;
};

Plan make_plan(const kvq_cache &c, int num_sms) {
  const CacheDims d = dims_of(c);
  Plan p;
  p.Gi = (d.Gk + kGroupsPerItem - 1) / kGroupsPerItem;
  p.Wt = (d.R + kWinItem - 1) / kWinItem;
  p.ipu = p.Gi + p.Wt;
  p.units = static_cast<long>(d.B) * d.Hkv;
  const long total = p.units * p.ipu;
  p.total_items = static_cast<int>(std::min<long>(total, 1L << 30));
  p.num_ctas = static_cast<int>(std::min<long>(total, static_cast<long>(kCtasPerSm) * num_sms));
  // A unit's ipu items meet at most (ipu - 2) / min_per + 2 slices: the first
  // and last hold at least one of its items, the ones between all of theirs.
  const long min_per = total / p.num_ctas;
  p.max_ctas_per_unit = p.ipu >= 2 ? static_cast<int>((p.ipu - 2) / min_per + 2) : 1;
  return p;
}

}  // namespace

bool decode_supported(const kvq_cache &c, int q_dtype, int Hq, int n_q) {
  const bool win_ok = c.recent == 0 || (c.kwin_dtype == KVQ_BF16 && c.vwin_dtype == KVQ_BF16);
  const long items = static_cast<long>(c.batch) * c.kv_heads *
                    ((c.n_tokens - c.recent + 32 * kGroupsPerItem - 1) / (32 * kGroupsPerItem) +
                     (c.recent + kWinItem - 1) / kWinItem);
  return c.head_dim == kD && n_q == 1 && Hq == kHeads * c.kv_heads && win_ok &&
         (q_dtype == KVQ_BF16 || q_dtype == KVQ_F32) && c.n_tokens > 0 && items < (1L << 30);
}

size_t decode_workspace_bytes(const kvq_cache &c, int, int num_sms) {
  const Plan p = make_plan(c, num_sms);
  return sizeof(float) * static_cast<size_t>(p.units) * p.max_ctas_per_unit * kHeads * kPartFloats;
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
  a.Gs = d.Gs;
  a.Vs = d.Vs;
  a.Ws = d.Ws;
  a.Wt = p.Wt;
  a.Gi = p.Gi;
  a.ipu = p.ipu;
  a.total_items = p.total_items;
  a.num_ctas = p.num_ctas;
  a.max_ctas_per_unit = p.max_ctas_per_unit;
  a.scale_log2 = scale_log2;
  a.partials = static_cast<float *>(ws);
  a.ctl = ctl;
  const size_t smem = sizeof(DecodeSmem);
  opt_in_smem(decode_kernel, smem);
  // The combine grid's blocks may be placed while the decode grid drains; they
  // wait for it on the device.
  launch_dependent(decode_kernel, dim3(p.num_ctas), dim3(kThreads), smem, s, a);
  if (p.max_ctas_per_unit > kWideCombineAbove) {
    const dim3 grid(static_cast<unsigned>(p.units), kHeads);
    if (out_dtype == KVQ_F32)
      launch_dependent(combine_wide_kernel<float>, grid, dim3(256), 0, s, a,
                       static_cast<float *>(out));
    else
      launch_dependent(combine_wide_kernel<__nv_bfloat16>, grid, dim3(256), 0, s, a,
                       static_cast<__nv_bfloat16 *>(out));
  } else if (out_dtype == KVQ_F32) {
    launch_dependent(combine_kernel<float>, dim3(p.units), dim3(kHeads * 32), 0, s, a,
                     static_cast<float *>(out));
  } else {
    launch_dependent(combine_kernel<__nv_bfloat16>, dim3(p.units), dim3(kHeads * 32), 0, s, a,
                     static_cast<__nv_bfloat16 *>(out));
  }
  return 2;
}

// ------------------------------------------------------------------ library-owned scratch
// Scratch of kv_attend_decode_static: the split-K partials live in this
// file-scope device array instead of a caller-provided workspace. Every GPU
// that loads this module keeps the array until the process exits.
namespace {
constexpr size_t kStaticScratchBytes = KVQ_DECODE_STATIC_SCRATCH_BYTES;  // 8 MiB
static_assert(kStaticScratchBytes == (size_t(8) << 20), "the header states 8 MiB");
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];
std::mutex g_scratch_mu;
void *g_scratch_addr[64] = {};
}  // namespace

size_t decode_static_scratch_limit() { return kStaticScratchBytes; }

// In host code `g_decode_scratch` is only a host-side stand-in; the kernel
// needs its device address, resolved once per device with that device current.
// Resolving it loads this file's module on that device (with lazy module
// loading, the CUDA default, nothing is loaded before), which is when the
// 8 MiB are reserved. A failure leaves no sticky error behind: the runtime's
// last error is cleared so the caller's next successful call reports success.
cudaError_t decode_static_scratch(void **ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e;
  }
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return e;
    }
    g_scratch_addr[dev] = p;
  }
  *ptr = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace kvq
