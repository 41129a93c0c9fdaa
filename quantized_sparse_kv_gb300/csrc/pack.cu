// kv_pack kernels: grouped symmetric int4 for the tokens before the window and
// a copy (or MXFP8 encoding) of the last R tokens.
//
// Residual-window page ("KV殘差窗口", section 固定預算): group size 32, K per
// channel over 32-token groups, V per token over 32-feature groups, the last R
// tokens kept in floating point. Rounding: scale = amax / 7 rounded once to
// fp32; code = clamp(rint(x / scale), -7, 7) with the division correctly
// rounded (__fdiv_rn) and ties to even (__float2int_rn); a zero scale gives
// zero codes. MXFP8 K window: Catnip study, section "Q/K 与 probability
// quantization 的影响" (E4M3, E8M0 scale per 32 along the head dim).
#include <cuda_fp8.h>

#include <algorithm>

#include "int4_round.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

__device__ __forceinline__ float int4_scale(float amax) { return __fdiv_rn(amax, 7.0f); }

__device__ __forceinline__ int int4_code(float x, float scale) {
  if (scale == 0.0f) return 0;
  int c = __float2int_rn(__fdiv_rn(x, scale));
  return max(-7, min(7, c));
}

// Four consecutive elements as floats (one 8- or 16-byte load).
__device__ __forceinline__ void load4(const float *p, float (&x)[4]) {
  const float4 f = *reinterpret_cast<const float4 *>(p);
  x[0] = f.x;
  x[1] = f.y;
  x[2] = f.z;
  x[3] = f.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16 *p, float (&x)[4]) {
  const uint2 u = *reinterpret_cast<const uint2 *>(p);
  x[0] = __uint_as_float(u.x << 16);
  x[1] = __uint_as_float(u.x & 0xffff0000u);
  x[2] = __uint_as_float(u.y << 16);
  x[3] = __uint_as_float(u.y & 0xffff0000u);
}

// K, head dim 128: one CTA of 256 threads per (sequence*head, K group).
// Warp w holds tokens 4w..4w+3 and lane l channels 4l..4l+3, so every load
// of a warp is one whole token row; the per-channel maximum over the 32
// tokens is taken over the thread's four tokens and then across the eight
// warps in shared memory, and each thread writes 2 code bytes per token.
template <typename T>
__global__ void __launch_bounds__(256) pack_k128_kernel(const T *__restrict__ k, int N, int cut,
                                                        int Gs, long u0,
                                                        uint8_t *__restrict__ k_codes,
                                                        float *__restrict__ k_scales,
                                                        const KernelCtl ctl) {
  wait_prior_grid();
  allow_next_grid();
  constexpr int D = 128;
  __shared__ __align__(16) float part[8][D];
  __shared__ __align__(16) float scale[D];
  const int g = blockIdx.x;              // K group
  const long u = u0 + blockIdx.y;        // (sequence, head)
  const long ug = u * Gs + g;  // Gs: K groups per (sequence, head) in the arrays
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int valid = min(kGroup, cut - g * kGroup);
  const T *src = k + (u * N + static_cast<long>(g) * kGroup) * D + 4 * lane;
  float x[4][4];
  float m[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = 4 * warp + i;
    if (t < valid && in_bounds(ctl, src + static_cast<long>(t) * D, 4 * sizeof(T)))
      load4(src + static_cast<long>(t) * D, x[i]);
    else
      x[i][0] = x[i][1] = x[i][2] = x[i][3] = 0.0f;
#pragma unroll
    for (int e = 0; e < 4; ++e) m[e] = fmaxf(m[e], fabsf(x[i][e]));
  }
  *reinterpret_cast<float4 *>(&part[warp][4 * lane]) = make_float4(m[0], m[1], m[2], m[3]);
  __syncthreads();
  if (threadIdx.x < D) {
    float mx = part[0][threadIdx.x];
#pragma unroll
    for (int w = 1; w < 8; ++w) mx = fmaxf(mx, part[w][threadIdx.x]);
    const float sc = int4_scale(mx);
    scale[threadIdx.x] = sc;
    if (in_bounds(ctl, k_scales + ug * D + threadIdx.x, sizeof(float)))
      k_scales[ug * D + threadIdx.x] = sc;
  }
  __syncthreads();
  const float4 sc = *reinterpret_cast<const float4 *>(&scale[4 * lane]);
  const float s4[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t w = 0u;
#pragma unroll
    for (int e = 0; e < 4; ++e) w |= static_cast<uint32_t>(int4_code(x[i][e], s4[e]) + 8) << (4 * e);
    uint8_t *dst = k_codes + (ug * kGroup + 4 * warp + i) * (D / 2) + 2 * lane;
    if (in_bounds(ctl, dst, 2)) *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(w);
  }
}

// The K loads of one channel pair and token as they sit in memory: a bf16
// pair stays packed in one register until it is used (half the registers
// of two floats, so more groups are in flight per SM).
struct PairBF16 {
  uint32_t w;
  __device__ __forceinline__ void load(const __nv_bfloat16 *p) {
    w = *reinterpret_cast<const uint32_t *>(p);
  }
  __device__ __forceinline__ void zero() { w = 0u; }
  __device__ __forceinline__ float lo() const { return __uint_as_float(w << 16); }
  __device__ __forceinline__ float hi() const { return __uint_as_float(w & 0xffff0000u); }
};
struct PairF32 {
  float2 f;
  __device__ __forceinline__ void load(const float *p) { f = *reinterpret_cast<const float2 *>(p); }
  __device__ __forceinline__ void zero() { f = make_float2(0.0f, 0.0f); }
  __device__ __forceinline__ float lo() const { return f.x; }
  __device__ __forceinline__ float hi() const { return f.y; }
};
template <typename T> struct PairOf;
template <> struct PairOf<float> { using type = PairF32; };
template <> struct PairOf<__nv_bfloat16> { using type = PairBF16; };

// K: one thread per (sequence*head, K group, channel pair). A warp's threads
// read adjacent channel pairs of the same token (one 128-byte line per load
// for bf16), keep the group's 32 pairs in registers, and write the pair's
// byte for each of the 32 tokens (adjacent threads -> adjacent bytes) and
// its two scales.
template <typename T>
__global__ void __launch_bounds__(256) pack_k_kernel(const T *__restrict__ k, long tasks, int N,
                                                     int D, int cut, int Gk, int Gs,
                                                     uint8_t *__restrict__ k_codes,
                                                     float *__restrict__ k_scales,
                                                     const KernelCtl ctl) {
  wait_prior_grid();
  allow_next_grid();
  const long task = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x;
  if (task >= tasks) return;
  const int pairs = D / 2;
  const int p = static_cast<int>(task % pairs);
  const long ugk = task / pairs;  // unit * Gk + g
  const int g = static_cast<int>(ugk % Gk);
  const long u = ugk / Gk;
  const long ug = u * Gs + g;     // position in the arrays
  const int valid = min(kGroup, cut - g * kGroup);
  const T *src = k + (u * N + static_cast<long>(g) * kGroup) * D + 2 * p;
  typename PairOf<T>::type x[kGroup];
#pragma unroll
  for (int t = 0; t < kGroup; ++t) {
    if (t < valid && in_bounds(ctl, src + static_cast<long>(t) * D, 2 * sizeof(T)))
      x[t].load(src + static_cast<long>(t) * D);
    else
      x[t].zero();
  }
  float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
  for (int t = 0; t < kGroup; ++t) {
    a0 = fmaxf(a0, fabsf(x[t].lo()));
    a1 = fmaxf(a1, fabsf(x[t].hi()));
  }
  const float s0 = int4_scale(a0), s1 = int4_scale(a1);
  if (in_bounds(ctl, k_scales + ug * D + 2 * p, 2 * sizeof(float)))
    *reinterpret_cast<float2 *>(k_scales + ug * D + 2 * p) = make_float2(s0, s1);
  uint8_t *dst = k_codes + ug * (kGroup * D / 2) + p;
  if (!in_bounds(ctl, dst, (kGroup - 1) * (D / 2) + 1)) return;
#pragma unroll
  for (int t = 0; t < kGroup; ++t)
    dst[t * (D / 2)] =
        static_cast<uint8_t>((int4_code(x[t].lo(), s0) + 8) | ((int4_code(x[t].hi(), s1) + 8) << 4));
}

// V: one thread per (token, 32-feature group) of the quantized part; 32 values
// in (16-byte loads), 16 code bytes and one scale out. The grid is (position
// within a slice of the unit's tokens, unit), so indices stay 32-bit.
template <typename T>
__global__ void __launch_bounds__(256) pack_v_kernel(const T *__restrict__ v, long u0, int t0,
                                                     int nt, int N, int D, int Vs,
                                                     uint8_t *__restrict__ v_codes,
                                                     float *__restrict__ v_scales,
                                                     const KernelCtl ctl) {
  wait_prior_grid();
  allow_next_grid();
  const int groups = D / kGroup;
  const unsigned task = blockIdx.x * blockDim.x + threadIdx.x;  // (token, group) in the slice
  if (task >= static_cast<unsigned>(nt) * groups) return;
  const int t = t0 + static_cast<int>(task / groups);  // token < cut
  const int j = static_cast<int>(task % groups);
  const long u = u0 + blockIdx.y;
  const long row = u * Vs + t;  // Vs: V rows per (sequence, head) in the arrays
  const T *src = v + (u * N + t) * D + j * kGroup;
  const bool src_ok = in_bounds(ctl, src, kGroup * sizeof(T));
  float x[kGroup];
#pragma unroll
  for (int i = 0; i < kGroup / 4; ++i) {
    float f[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (src_ok) load4(src + 4 * i, f);
    x[4 * i] = f[0];
    x[4 * i + 1] = f[1];
    x[4 * i + 2] = f[2];
    x[4 * i + 3] = f[3];
  }
  float amax = 0.0f;
#pragma unroll
  for (int e = 0; e < kGroup; ++e) amax = fmaxf(amax, fabsf(x[e]));
  const float s = int4_scale(amax);
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int e = 0; e < kGroup; ++e)
    w[e >> 3] |= static_cast<uint32_t>(int4_code(x[e], s) + 8) << (4 * (e & 7));
  uint8_t *cd = v_codes + row * (D / 2) + j * (kGroup / 2);
  if (in_bounds(ctl, cd, 16)) *reinterpret_cast<uint4 *>(cd) = make_uint4(w[0], w[1], w[2], w[3]);
  if (in_bounds(ctl, v_scales + row * groups + j, sizeof(float))) v_scales[row * groups + j] = s;
}

// ------------------------------------------------------------------ bf16, D = 128
// The int4 part of a bf16 cache with D = 128 in one persistent kernel. A work
// item is one 32-token group of one (sequence, head): its K rows and its V
// rows are two contiguous 8 KB tiles. One loader lane streams both tiles of
// each item into a ring of shared-memory stages with 1-D bulk copies; warps
// 0-3 quantize the K tile (warp w: tokens 8w..8w+7, lane l: channels
// 4l..4l+3, so each shared-memory load of a warp is one whole row; the four
// warps' per-channel maxima meet in shared memory behind an mbarrier) and
// warps 4-7 the V tile (lane: one token and one 32-feature group).
//
// Same codes and scales as the kernels above, without a division per
// element (int4_round.cuh: a reciprocal and one correction step, exact on
// bf16 inputs for the groups recip_ok admits); other groups take the
// division.
constexpr int kPkStages = 6;
constexpr int kPkTile = kGroup * 128 * 2;  // bytes of one tile: 32 rows of 128 bf16
constexpr int kPkWorkers = 8;              // warps 0-3 K, 4-7 V; warp 8 loads
constexpr int kPkThreads = 32 * (kPkWorkers + 1);
constexpr int kPkCtasPerSm = 2;

struct PackSmem {
  uint8_t k[kPkStages][kPkTile];
  uint8_t v[kPkStages][kPkTile];
  uint64_t full[kPkStages], empty[kPkStages];
  int abort_flag;
};

__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// One code byte by the division (the groups recip_ok leaves out).
__device__ __forceinline__ uint32_t code_byte_div(uint32_t w, float s_lo, float s_hi) {
  return static_cast<uint32_t>(int4_code(bf_hi(w), s_hi) + 8) * 16u +
         static_cast<uint32_t>(int4_code(bf_lo(w), s_lo) + 8);
}

// The division path of one K lane (out of line, reading its column of the
// tile again: rare).
__device__ __noinline__ void pack_k_quarter_div(const uint8_t *src, int h, int valid, float a0,
                                                float a1, float *scales, uint8_t *dst,
                                                const KernelCtl ctl) {
  const float s0 = int4_scale(a0), s1 = int4_scale(a1);
  if (h == 0 && in_bounds(ctl, scales, 2 * sizeof(float)))
    *reinterpret_cast<float2 *>(scales) = make_float2(s0, s1);
#pragma unroll 1
  for (int i = 0; i < 16; ++i) {
    const uint32_t x = 16 * h + i < valid ? *reinterpret_cast<const uint32_t *>(src + i * 256) : 0u;
    if (in_bounds(ctl, dst + i * 64, 1)) dst[i * 64] = static_cast<uint8_t>(code_byte_div(x, s0, s1));
  }
}

// K warp kw of one item: channels 32kw..32kw+31 of the tile. Lane (w, h) =
// (lane % 16, lane / 16) holds the channel pair 32kw + 2w, +1 of rows
// 16h..16h+15 in registers; one lane exchange joins the two halves' maxima.
template <bool kRagged>
__device__ __forceinline__ void pack_k_quarter(const uint8_t *tile, int kw, int lane, int valid,
                                               long ug, uint8_t *__restrict__ k_codes,
                                               float *__restrict__ k_scales,
                                               const KernelCtl &ctl) {
  const int w = lane & 15, h = lane >> 4;
  const uint8_t *src = tile + 16 * h * 256 + 64 * kw + 4 * w;
  uint32_t x[16];
  uint32_t m = 0u;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    x[i] = *reinterpret_cast<const uint32_t *>(src + i * 256);
    if (kRagged && 16 * h + i >= valid) x[i] = 0u;  // rows past the cut
    m = max_bf16x2(m, x[i] & 0x7fff7fffu);
  }
  m = max_bf16x2(m, __shfl_xor_sync(~0u, m, 16));
  const float a0 = bf_lo(m), a1 = bf_hi(m);
  float *scales = k_scales + ug * 128 + 32 * kw + 2 * w;
  uint8_t *dst = k_codes + (ug * kGroup + 16 * h) * 64 + 16 * kw + w;
  if (!(recip_ok(a0) && recip_ok(a1))) {
    pack_k_quarter_div(src, h, valid, a0, a1, scales, dst, ctl);
    return;
  }
  const float s0 = scale_recip(a0), s1 = scale_recip(a1);
  const float r0 = recip_of(s0), r1 = recip_of(s1);
  if (h == 0 && in_bounds(ctl, scales, 2 * sizeof(float)))
    *reinterpret_cast<float2 *>(scales) = make_float2(s0, s1);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t b = code_byte_recip(x[i], -s0, -s1, r0, r1);
    if (in_bounds(ctl, dst + i * 64, 1)) dst[i * 64] = static_cast<uint8_t>(b);
  }
}

// One V lane's group by the division (out of line, reading its 64 bytes of
// shared memory again: rare).
__device__ __noinline__ void pack_v_group_div(const uint8_t *src, float amax, bool store,
                                              uint8_t *dst, float *scale, const KernelCtl ctl) {
  const float s = int4_scale(amax);
  uint32_t o[4];
#pragma unroll 1
  for (int i = 0; i < 4; ++i) {
    const uint4 w = *reinterpret_cast<const uint4 *>(src + 16 * i);
    const uint32_t e[4] = {w.x, w.y, w.z, w.w};
    uint32_t b[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) b[q] = code_byte_div(e[q], s, s);
    o[i] = __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040), 0x5410);
  }
  if (!store) return;
  if (in_bounds(ctl, dst, 16)) *reinterpret_cast<uint4 *>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
  if (in_bounds(ctl, scale, sizeof(float))) *scale = s;
}

// V warp vw of one item: lane (token 8 vw + lane / 4, feature group lane % 4).
// Its four 16-byte loads are taken in a rotated order so that the eight lanes
// of each shared-memory phase hit eight different bank quads.
__device__ __forceinline__ void pack_v_tile(const uint8_t *tile, int vw, int lane, int valid,
                                            long row0, uint8_t *__restrict__ v_codes,
                                            float *__restrict__ v_scales, const KernelCtl &ctl) {
  const int t = 8 * vw + (lane >> 2), j = lane & 3;
  const int rot = ((j >> 1) + 2 * (t & 1)) & 3;
  const uint8_t *src = tile + t * 256 + 64 * j;
  uint4 w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = *reinterpret_cast<const uint4 *>(src + 16 * ((i + rot) & 3));
  uint32_t m[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    m[i] = max_bf16x2(max_bf16x2(w[i].x & 0x7fff7fffu, w[i].y & 0x7fff7fffu),
                      max_bf16x2(w[i].z & 0x7fff7fffu, w[i].w & 0x7fff7fffu));
  const uint32_t mm = max_bf16x2(max_bf16x2(m[0], m[1]), max_bf16x2(m[2], m[3]));
  const float amax = fmaxf(bf_lo(mm), bf_hi(mm));
  const long row = row0 + t;
  uint8_t *dst = v_codes + row * 64 + 16 * j;
  float *scale = v_scales + row * 4 + j;
  if (!recip_ok(amax)) {
    pack_v_group_div(src, amax, t < valid, dst, scale, ctl);
    return;
  }
  const float s = scale_recip(amax), r = recip_of(s);
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t e[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
    uint32_t b[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) b[q] = code_byte_recip(e[q], -s, -s, r, r);
    o[i] = __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040), 0x5410);
  }
  // o[i] holds 16-byte piece (i + rot) & 3: rotate back by rot
  uint32_t p[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) p[c] = (rot & 1) ? o[(c + 3) & 3] : o[c];
#pragma unroll
  for (int c = 0; c < 4; ++c) o[c] = (rot & 2) ? p[(c + 2) & 3] : p[c];
  if (t >= valid) return;  // rows past the cut belong to the window
  if (in_bounds(ctl, dst, 16)) *reinterpret_cast<uint4 *>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
  if (in_bounds(ctl, scale, sizeof(float))) *scale = s;
}

// The items of a CTA: it = blockIdx.x + n * gridDim.x, as (unit u, group g)
// advanced without a division (du, dg: gridDim.x = du * Gk + dg).
struct ItemWalk {
  int u, g;
  __device__ __forceinline__ void start(int Gk) {
    u = static_cast<int>(blockIdx.x) / Gk;
    g = static_cast<int>(blockIdx.x) - u * Gk;
  }
  __device__ __forceinline__ void next(int Gk, int du, int dg) {
    u += du;
    g += dg;
    if (g >= Gk) {
      g -= Gk;
      ++u;
    }
  }
};

// Every worker warp takes part in every item of the CTA, in order (so each
// waits on each phase of a stage's barrier and none can run a phase ahead):
// K warp w a quarter of the channels of the K tile, V warp w a quarter of
// the rows of the V tile; a stage is free again after the eight arrivals.
__global__ void __launch_bounds__(kPkThreads, kPkCtasPerSm)
    pack_kv128_bf16_kernel(const __nv_bfloat16 *__restrict__ k,
                           const __nv_bfloat16 *__restrict__ v, int N, int cut, int Gk, int Gs,
                           int Vs, int items, int du, int dg, uint8_t *__restrict__ k_codes,
                           float *__restrict__ k_scales, uint8_t *__restrict__ v_codes,
                           float *__restrict__ v_scales, const KernelCtl ctl) {
  extern __shared__ __align__(128) uint8_t pk_smem_raw[];
  PackSmem &sm = *reinterpret_cast<PackSmem *>(pk_smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  allow_next_grid();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPkStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), kPkWorkers);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  wait_prior_grid();  // the previous kernel may still be reading the cache
  ItemWalk at;
  at.start(Gk);

  if (warp == kPkWorkers) {
    // ---------------- loader
    if (lane == 0) {
      int n = 0;
      for (int it = blockIdx.x; it < items; it += gridDim.x, ++n, at.next(Gk, du, dg)) {
        const int st = n % kPkStages;
        if (n >= kPkStages &&
            !mbar_wait(smem_u32(&sm.empty[st]), static_cast<uint32_t>((n / kPkStages - 1) & 1),
                       ctl.wait_limit_ns)) {
          flag_error(ctl, KVQ_DEV_TIMEOUT);
          *reinterpret_cast<volatile int *>(&sm.abort_flag) = 1;
          break;
        }
        if (*reinterpret_cast<volatile int *>(&sm.abort_flag)) break;
        if (it == ctl.drop_item) continue;  // test hook: a dropped stage is never filled
        const uint32_t bytes = static_cast<uint32_t>(min(kGroup, cut - at.g * kGroup)) * 256u;
        const long e0 = (static_cast<long>(at.u) * N + static_cast<long>(at.g) * kGroup) * 128;
        const bool ok_k = in_bounds(ctl, k + e0, bytes), ok_v = in_bounds(ctl, v + e0, bytes);
        mbar_arrive_expect_tx(smem_u32(&sm.full[st]), (ok_k + ok_v) * bytes);
        if (ok_k) bulk_g2s(smem_u32(sm.k[st]), k + e0, bytes, smem_u32(&sm.full[st]));
        if (ok_v) bulk_g2s(smem_u32(sm.v[st]), v + e0, bytes, smem_u32(&sm.full[st]));
      }
      // drain: copies still in flight must land before the CTA exits
      for (int d = max(0, n - kPkStages); d < n; ++d) {
        if (static_cast<long>(blockIdx.x) + static_cast<long>(d) * gridDim.x == ctl.drop_item)
          continue;
        mbar_wait(smem_u32(&sm.full[d % kPkStages]), static_cast<uint32_t>((d / kPkStages) & 1),
                  2000000000ull);
      }
    }
    return;
  }

  // ---------------- workers (every decision on a wait is taken by the whole warp)
  const bool is_k = warp < 4;
  int n = 0;
  for (int it = blockIdx.x; it < items; it += gridDim.x, ++n, at.next(Gk, du, dg)) {
    const int st = n % kPkStages;
    if (__any_sync(~0u, *reinterpret_cast<volatile int *>(&sm.abort_flag) != 0)) break;
    if (!__all_sync(~0u, mbar_wait(smem_u32(&sm.full[st]),
                                   static_cast<uint32_t>((n / kPkStages) & 1), ctl.wait_limit_ns))) {
      if (lane == 0) {
        flag_error(ctl, KVQ_DEV_TIMEOUT);
        *reinterpret_cast<volatile int *>(&sm.abort_flag) = 1;
      }
      break;
    }
    const int valid = min(kGroup, cut - at.g * kGroup);
    if (is_k) {
      const long ug = static_cast<long>(at.u) * Gs + at.g;
      if (valid == kGroup)
        pack_k_quarter<false>(sm.k[st], warp, lane, valid, ug, k_codes, k_scales, ctl);
      else
        pack_k_quarter<true>(sm.k[st], warp, lane, valid, ug, k_codes, k_scales, ctl);
    } else {
      pack_v_tile(sm.v[st], warp - 4, lane, valid,
                  static_cast<long>(at.u) * Vs + static_cast<long>(at.g) * kGroup, v_codes,
                  v_scales, ctl);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sm.empty[st]));
  }
}

// Window copy with dtype change (fp32 <-> bf16, nearest even).
// Ws: window rows per (sequence, head) in the arrays.
template <typename TI, typename TO>
__global__ void window_copy_kernel(const TI *__restrict__ x, long rows, int N, int D, int R,
                                   int Ws, TO *__restrict__ w, const KernelCtl ctl) {
  wait_prior_grid();
  allow_next_grid();
  const long n = rows * D;
  for (long i = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long>(gridDim.x) * blockDim.x) {
    const long row = i / D, d = i % D;
    const long u = row / R, t = row % R;
    const TI *src = x + (u * N + (N - R) + t) * D + d;
    TO *dst = w + (u * Ws + t) * D + d;
    if (in_bounds(ctl, src, sizeof(TI)) && in_bounds(ctl, dst, sizeof(TO)))
      store_from_f32(dst, load_f32(src));
  }
}

// MXFP8 window: one warp per (token, 32-feature block). Block exponent
// e = floor(log2 amax) - 8 clamped to [-127, 127] (-127 for a zero block);
// elements x * 2^-e rounded to E4M3, nearest even, saturating at 448.
template <typename TI>
__global__ void __launch_bounds__(256) window_mxfp8_kernel(const TI *__restrict__ x, long rows,
                                                           int N, int D, int R, int Ws,
                                                           uint8_t *__restrict__ codes,
                                                           uint8_t *__restrict__ e8m0,
                                                           const KernelCtl ctl) {
  wait_prior_grid();
  allow_next_grid();
  const int groups = D / kGroup;
  const long task = static_cast<long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
  if (task >= rows * groups) return;
  const int lane = threadIdx.x & 31;
  const long row = task / groups;
  const int j = static_cast<int>(task % groups);
  const long u = row / R, t = row % R;
  const TI *src = x + (u * N + (N - R) + t) * D + j * kGroup + lane;
  const float val = in_bounds(ctl, src, sizeof(TI)) ? load_f32(src) : 0.0f;
  const int e = mxfp8_block_exp(warp_max(fabsf(val)));
  const long dst = u * Ws + t;
  if (in_bounds(ctl, codes + dst * D + j * kGroup + lane, 1))
    codes[dst * D + j * kGroup + lane] = mxfp8_code(val, pow2_of(-e));
  if (lane == 0 && in_bounds(ctl, e8m0 + dst * groups + j, 1))
    e8m0[dst * groups + j] = static_cast<uint8_t>(e + 127);
}

bool aligned16_ptr(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The fused bf16 kernel for the int4 part, when the cache takes it: D = 128,
// every array on a 16-byte boundary (the bulk copies and the vector stores).
bool pack_fused(const __nv_bfloat16 *k, const __nv_bfloat16 *v, const kvq_cache &c,
                const CacheDims &d, const KernelCtl &ctl, int num_sms, cudaStream_t s) {
  const long items = static_cast<long>(d.B) * d.Hkv * d.Gk;
  if (d.D != 128 || items >= (1L << 30) || !aligned16_ptr(k) || !aligned16_ptr(v) ||
      !aligned16_ptr(c.k_codes) || !aligned16_ptr(c.k_scales) || !aligned16_ptr(c.v_codes) ||
      !aligned16_ptr(c.v_scales))
    return false;
  const size_t smem = sizeof(PackSmem);
  if (opt_in_smem(pack_kv128_bf16_kernel, smem) != cudaSuccess) return false;
  const int grid = static_cast<int>(std::min<long>(items, static_cast<long>(kPkCtasPerSm) * num_sms));
  launch_dependent(pack_kv128_bf16_kernel, dim3(grid), dim3(kPkThreads), smem, s, k, v, d.N, d.cut,
                   d.Gk, d.Gs, d.Vs, static_cast<int>(items), grid / d.Gk, grid % d.Gk, c.k_codes,
                   c.k_scales, c.v_codes, c.v_scales, ctl);
  return true;
}
bool pack_fused(const float *, const float *, const kvq_cache &, const CacheDims &,
                const KernelCtl &, int, cudaStream_t) {
  return false;
}

template <typename T>
int pack_typed(const T *k, const T *v, const kvq_cache &c, const KernelCtl &ctl, int num_sms,
               cudaStream_t s) {
  const CacheDims d = dims_of(c);
  const long units = static_cast<long>(d.B) * d.Hkv;
  int launches = 0;
  if (d.cut > 0 && pack_fused(k, v, c, d, ctl, num_sms, s)) {
    ++launches;
  } else if (d.cut > 0) {
    if (d.D == 128) {
      for (long u0 = 0; u0 < units; u0 += 65535) {  // grid.y holds at most 65,535 units
        const unsigned nu = static_cast<unsigned>(std::min<long>(65535, units - u0));
        launch_dependent(pack_k128_kernel<T>, dim3(d.Gk, nu), dim3(256), 0, s, k, d.N, d.cut, d.Gs,
                         u0, c.k_codes, c.k_scales, ctl);
        ++launches;
      }
    } else {
      const long ktasks = units * d.Gk * (d.D / 2);
      const unsigned kblocks = static_cast<unsigned>((ktasks + 255) / 256);
      launch_dependent(pack_k_kernel<T>, dim3(kblocks), dim3(256), 0, s, k, ktasks, d.N, d.D, d.cut, d.Gk, d.Gs, c.k_codes, c.k_scales, ctl);
      ++launches;
    }
    // V: per launch at most 65,535 units (grid.y) and 2^24 tokens of each,
    // so the thread index within a unit's slice fits 32 bits
    constexpr int kSlice = 1 << 24;
    for (long u0 = 0; u0 < units; u0 += 65535) {
      const unsigned nu = static_cast<unsigned>(std::min<long>(65535, units - u0));
      for (int t0 = 0; t0 < d.cut; t0 += kSlice) {
        const int nt = std::min(kSlice, d.cut - t0);
        const long vthreads = static_cast<long>(nt) * (d.D / kGroup);
        launch_dependent(pack_v_kernel<T>, dim3(static_cast<unsigned>((vthreads + 255) / 256), nu),
                         dim3(256), 0, s, v, u0, t0, nt, d.N, d.D, d.Vs, c.v_codes, c.v_scales,
                         ctl);
        ++launches;
      }
    }
  }
  if (d.R > 0) {
    const long rows = units * d.R;
    const unsigned blocks =
        static_cast<unsigned>(std::min<long>((rows * d.D + 255) / 256, 1L << 20));
    if (c.kwin_dtype == KVQ_MXFP8) {
      const long tasks = rows * (d.D / kGroup);
      launch_dependent(window_mxfp8_kernel<T>, dim3(static_cast<unsigned>((tasks + 7) / 8)),
                       dim3(256), 0, s, k, rows, d.N, d.D, d.R, d.Ws,
                       static_cast<uint8_t *>(c.k_window), c.k_window_e8m0, ctl);
    } else if (c.kwin_dtype == KVQ_F32) {
      launch_dependent(window_copy_kernel<T, float>, dim3(blocks), dim3(256), 0, s, k, rows, d.N,
                       d.D, d.R, d.Ws, static_cast<float *>(c.k_window), ctl);
    } else {
      launch_dependent(window_copy_kernel<T, __nv_bfloat16>, dim3(blocks), dim3(256), 0, s,
          k, rows, d.N, d.D, d.R, d.Ws, static_cast<__nv_bfloat16 *>(c.k_window), ctl);
    }
    if (c.vwin_dtype == KVQ_F32) {
      launch_dependent(window_copy_kernel<T, float>, dim3(blocks), dim3(256), 0, s, v, rows, d.N,
                       d.D, d.R, d.Ws, static_cast<float *>(c.v_window), ctl);
    } else {
      launch_dependent(window_copy_kernel<T, __nv_bfloat16>, dim3(blocks), dim3(256), 0, s,
          v, rows, d.N, d.D, d.R, d.Ws, static_cast<__nv_bfloat16 *>(c.v_window), ctl);
    }
    launches += 2;
  }
  return launches;
}

// ------------------------------------------------------------------ kv_append
// The tokens of one (sequence, head) as an append sees them: the current
// window rows followed by the new ones, S[i] = window row i for i < R_old and
// new row i - R_old after. The oldest 32m of them become int4 groups
// Gk_old .. Gk_old + m - 1 (and V rows cut_old .. cut_old + 32m - 1) by the
// kv_pack rule; S[32m ..] is the new window.
struct AppendArgs {
  const void *k_new, *v_new;  // [units][T][D] in in_dtype
  int in_dtype, kwin, vwin;
  uint8_t *k_codes;
  float *k_scales;
  uint8_t *v_codes;
  float *v_scales;
  void *k_window, *v_window;
  int D, T, R_old, m, Gk_old, cut_old, Gs, Vs, Ws;
  KernelCtl ctl;
};

// Eight consecutive elements from element e0 of a window or of the new rows,
// as floats: one 16-byte load for bf16, two for fp32 (e0 is a multiple of 8
// and every row starts on a 16-byte boundary).
__device__ __forceinline__ void load8_as(const void *base, long e0, int dt, float (&x)[8]) {
  if (dt == KVQ_F32) {
    const float4 lo = *reinterpret_cast<const float4 *>(static_cast<const float *>(base) + e0);
    const float4 hi = *reinterpret_cast<const float4 *>(static_cast<const float *>(base) + e0 + 4);
    x[0] = lo.x, x[1] = lo.y, x[2] = lo.z, x[3] = lo.w;
    x[4] = hi.x, x[5] = hi.y, x[6] = hi.z, x[7] = hi.w;
  } else {
    const uint4 w = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(base) + e0);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(ws[i] << 16);
      x[2 * i + 1] = __uint_as_float(ws[i] & 0xffff0000u);
    }
  }
}

__device__ __forceinline__ void store8_as(void *base, long e0, int dt, const float (&x)[8]) {
  if (dt == KVQ_F32) {
    float *o = static_cast<float *>(base) + e0;
    *reinterpret_cast<float4 *>(o) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4 *>(o + 4) = make_float4(x[4], x[5], x[6], x[7]);
  } else {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 b = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t *>(&b);
    }
    *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(base) + e0) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Elements d0 .. d0 + 7 of token i of the append sequence S.
__device__ __forceinline__ void seq8(const AppendArgs &a, const void *win, const void *fresh,
                                     int win_dt, long u, int i, int d0, float (&x)[8]) {
  // (debug builds: a row outside the call's buffers reads as zeros)
  if (i < a.R_old) {
    const long e0 = (u * a.Ws + i) * a.D + d0;
    const size_t eb = win_dt == KVQ_F32 ? 4 : 2;
    if (in_bounds(a.ctl, static_cast<const uint8_t *>(win) + e0 * eb, 8 * eb)) {
      load8_as(win, e0, win_dt, x);
      return;
    }
  } else {
    const long e0 = (u * a.T + (i - a.R_old)) * a.D + d0;
    const size_t eb = a.in_dtype == KVQ_F32 ? 4 : 2;
    if (in_bounds(a.ctl, static_cast<const uint8_t *>(fresh) + e0 * eb, 8 * eb)) {
      load8_as(fresh, e0, a.in_dtype, x);
      return;
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) x[e] = 0.0f;
}

constexpr int kAppendThreads = 256;
// 8-element pieces of a 32-token group per thread: 32 * D / 8 / 256, D <= 256
constexpr int kStagePieces = 4;

// The group's 32 tokens of S into shared memory as floats, rows of D + 1
// (the padding spreads a column over the banks). Every load of a thread is
// issued before its first store.
__device__ __forceinline__ void stage_group(const AppendArgs &a, const void *win,
                                            const void *fresh, int win_dt, long u, int gi,
                                            float *xs) {
  const int D = a.D, pieces = kGroup * D / 8;
  float x[kStagePieces][8];
#pragma unroll
  for (int k = 0; k < kStagePieces; ++k) {
    const int pc = threadIdx.x + k * kAppendThreads;
    if (pc < pieces) seq8(a, win, fresh, win_dt, u, kGroup * gi + pc * 8 / D, pc * 8 % D, x[k]);
  }
#pragma unroll
  for (int k = 0; k < kStagePieces; ++k) {
    const int pc = threadIdx.x + k * kAppendThreads;
    if (pc < pieces) {
      float *row = xs + (pc * 8 / D) * (D + 1) + pc * 8 % D;
#pragma unroll
      for (int e = 0; e < 8; ++e) row[e] = x[k][e];
    }
  }
}

// One CTA per (migrated group gi, unit). The group's 32 tokens are staged in
// shared memory as floats, K then V; K takes a thread per channel pair and
// token slice, V one thread per (token, 32-feature block).
__global__ void __launch_bounds__(kAppendThreads) append_migrate_kernel(const AppendArgs a) {
  wait_prior_grid();
  allow_next_grid();
  extern __shared__ float xs[];  // [32][D + 1]
  const int gi = blockIdx.x;
  const long u = blockIdx.y;
  const long grp = u * a.Gs + a.Gk_old + gi;
  const int D = a.D, ld = D + 1;
  stage_group(a, a.k_window, a.k_new, a.kwin, u, gi, xs);
  __syncthreads();
  // K: thread (pair p, slice q) takes channels 2p, 2p + 1 over tokens
  // q * tq .. q * tq + tq - 1; the per-channel maxima meet in shared memory.
  __shared__ float2 kmax[kAppendThreads];
  const int np = D / 2, nq = kAppendThreads / np, tq = kGroup / nq;
  const int p = threadIdx.x % np, q = threadIdx.x / np;
  float a0 = 0.0f, a1 = 0.0f;
  for (int t = q * tq; t < q * tq + tq; ++t) {
    a0 = fmaxf(a0, fabsf(xs[t * ld + 2 * p]));
    a1 = fmaxf(a1, fabsf(xs[t * ld + 2 * p + 1]));
  }
  kmax[threadIdx.x] = make_float2(a0, a1);
  __syncthreads();
  for (int r = 0; r < nq; ++r) {
    a0 = fmaxf(a0, kmax[r * np + p].x);
    a1 = fmaxf(a1, kmax[r * np + p].y);
  }
  const float s0 = int4_scale(a0), s1 = int4_scale(a1);
  if (q == 0 && in_bounds(a.ctl, a.k_scales + grp * D + 2 * p, 2 * sizeof(float))) {
    a.k_scales[grp * D + 2 * p] = s0;
    a.k_scales[grp * D + 2 * p + 1] = s1;
  }
  for (int t = q * tq; t < q * tq + tq; ++t)
    if (in_bounds(a.ctl, a.k_codes + (grp * kGroup + t) * (D / 2) + p, 1))
      a.k_codes[(grp * kGroup + t) * (D / 2) + p] = static_cast<uint8_t>(
        (int4_code(xs[t * ld + 2 * p], s0) + 8) | ((int4_code(xs[t * ld + 2 * p + 1], s1) + 8) << 4));
  __syncthreads();
  stage_group(a, a.v_window, a.v_new, a.vwin, u, gi, xs);
  __syncthreads();
  const int blocks = D / kGroup;
  for (int task = threadIdx.x; task < kGroup * blocks; task += blockDim.x) {
    const int t = task / blocks, j = task % blocks;
    const long row = u * a.Vs + a.cut_old + kGroup * gi + t;
    const float *x = xs + t * ld + kGroup * j;
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < kGroup; ++e) amax = fmaxf(amax, fabsf(x[e]));
    const float sc = int4_scale(amax);
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int e = 0; e < kGroup; ++e)
      w[e >> 3] |= static_cast<uint32_t>(int4_code(x[e], sc) + 8) << (4 * (e & 7));
    uint8_t *cd = a.v_codes + row * (D / 2) + j * (kGroup / 2);
    if (in_bounds(a.ctl, cd, 16)) *reinterpret_cast<uint4 *>(cd) = make_uint4(w[0], w[1], w[2], w[3]);
    if (in_bounds(a.ctl, a.v_scales + row * blocks + j, sizeof(float)))
      a.v_scales[row * blocks + j] = sc;
  }
}

// The new window, rows [0, R_new) = S[32m ..], one CTA per unit, 32 rows per
// step with a barrier between steps. With m > 0 a step reads rows at least 32
// above those it writes, and a row written at step s was read at step s - m,
// before the barrier; with m = 0 the old rows stay and only new ones are
// written. A step moves 8-element pieces, all of a thread's loads before its
// stores.
__global__ void __launch_bounds__(kAppendThreads) append_window_kernel(const AppendArgs a,
                                                                       int R_new) {
  wait_prior_grid();
  allow_next_grid();
  const long u = blockIdx.x;
  const int D = a.D;
  for (int r0 = a.m == 0 ? a.R_old : 0; r0 < R_new; r0 += kGroup) {
    const int pieces = min(kGroup, R_new - r0) * D / 8;
    float kx[kStagePieces][8], vx[kStagePieces][8];
#pragma unroll
    for (int k = 0; k < kStagePieces; ++k) {
      const int pc = threadIdx.x + k * kAppendThreads;
      if (pc < pieces) {
        const int i = kGroup * a.m + r0 + pc * 8 / D, d0 = pc * 8 % D;
        seq8(a, a.k_window, a.k_new, a.kwin, u, i, d0, kx[k]);
        seq8(a, a.v_window, a.v_new, a.vwin, u, i, d0, vx[k]);
      }
    }
#pragma unroll
    for (int k = 0; k < kStagePieces; ++k) {
      const int pc = threadIdx.x + k * kAppendThreads;
      if (pc < pieces) {
        const long o = (u * a.Ws + r0 + pc * 8 / D) * D + pc * 8 % D;
        const size_t kb = a.kwin == KVQ_F32 ? 4 : 2, vb = a.vwin == KVQ_F32 ? 4 : 2;
        if (in_bounds(a.ctl, static_cast<uint8_t *>(a.k_window) + o * kb, 8 * kb))
          store8_as(a.k_window, o, a.kwin, kx[k]);
        if (in_bounds(a.ctl, static_cast<uint8_t *>(a.v_window) + o * vb, 8 * vb))
          store8_as(a.v_window, o, a.vwin, vx[k]);
      }
    }
    __syncthreads();
  }
}

}  // namespace

int launch_pack(const void *k, const void *v, int in_dtype, const kvq_cache &c,
                const KernelCtl &ctl, int num_sms, cudaStream_t s) {
  if (in_dtype == KVQ_F32)
    return pack_typed(static_cast<const float *>(k), static_cast<const float *>(v), c, ctl,
                      num_sms, s);
  return pack_typed(static_cast<const __nv_bfloat16 *>(k), static_cast<const __nv_bfloat16 *>(v),
                    c, ctl, num_sms, s);
}

int launch_append(const kvq_cache &c, const void *k_new, const void *v_new, int in_dtype,
                  int n_new, int m, int R_new, const KernelCtl &ctl, cudaStream_t s) {
  const CacheDims d = dims_of(c);
  const long units = static_cast<long>(d.B) * d.Hkv;
  AppendArgs a;
  a.k_new = k_new;
  a.v_new = v_new;
  a.in_dtype = in_dtype;
  a.kwin = c.kwin_dtype;
  a.vwin = c.vwin_dtype;
  a.k_codes = c.k_codes;
  a.k_scales = c.k_scales;
  a.v_codes = c.v_codes;
  a.v_scales = c.v_scales;
  a.k_window = c.k_window;
  a.v_window = c.v_window;
  a.D = d.D;
  a.T = n_new;
  a.R_old = d.R;
  a.m = m;
  a.Gk_old = d.Gk;
  a.cut_old = d.cut;
  a.Gs = d.Gs;
  a.Vs = d.Vs;
  a.Ws = d.Ws;
  a.ctl = ctl;
  int launches = 0;
  if (m > 0) {
    const size_t smem = sizeof(float) * kGroup * (d.D + 1);
    launch_dependent(append_migrate_kernel,
                     dim3(static_cast<unsigned>(m), static_cast<unsigned>(units)),
                     dim3(kAppendThreads), smem, s, a);
    ++launches;
  }
  launch_dependent(append_window_kernel, dim3(static_cast<unsigned>(units)),
                   dim3(kAppendThreads), 0, s, a, R_new);
  return launches + 1;
}

}  // namespace kvq
