// Chunk attention on the fifth-generation tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes: for every query row of a chunk, O = softmax(sm_scale * Q
// K^T) V over all keys of a cache whose window holds every token (bf16 K and
// V), plus the per-row softmax mass on each key region -- the Catnip study's
// chunk of 2,340 queries (6 latent frames) over 6,240 keys laid out [sink 1560
// | recent 2340 | current 2340] (section "KV Cache 的实际作用"), no mask.
//
// Variants of the same kernel body: bf16 Q/K over 128-key tiles (an
// all-window cache; an int4-history cache, whose history tiles are first
// expanded to bf16 in workspace; block-shared candidate lists gathered to
// bf16), and MXFP8 Q/K over 112-key tiles (QK^T as a block-scaled MMA).
//
// One CTA per (128 query rows, query head); 12 warps:
//   warp 0      TMA producer: Q once, then the K tiles (a ring of two stages,
//               three with MXFP8; a stage is refilled once its QK MMA ends),
//               128B-swizzled in 64-feature boxes;
//   warp 1      allocates 512 TMEM columns and one lane issues the MMAs;
//   warp 2      TMA producer: the V tiles (the same ring sizes; a stage is
//               refilled once its PV MMA ends);
//   warps 4-7   softmax group A: key tiles 0, 2, 4, ...
//   warps 8-11  softmax group B: key tiles 1, 3, 5, ...
// Each softmax group g owns TMEM S_g (128 columns) and O_g (128 columns) and
// a P buffer in shared memory; its chain per tile is S = Q K^T (MMA) ->
// softmax (thread r owns query row r = TMEM lane r) -> O_g += P V (MMA, V as
// the MN-major operand), and the two groups' chains interleave so the tensor
// core works on one group while the other exponentiates. P is taken against
// a fixed reference per row and group, set from the first 32 scores the
// group sees; a tile that would push P past 2^64 raises the reference,
// rescales O_g and the sums, and is redone from its scores (still in TMEM).
// Region masses (up to 16 regions) are summed per row as the keys stream by:
// one running sum for the region under the current key, the finished
// regions' sums kept per thread. At the end each group leaves its row state
// (reference, sum, region sums) in shared memory and merges both groups' O
// for half of the columns, normalises and stores them; group A stores the
// region masses.
// Every mbarrier wait is bounded; on timeout the CTA flags KVQ_DEV_TIMEOUT,
// stops, drains its copies and MMAs and frees TMEM.
#include <cuda.h>
#include <math_constants.h>

#include <algorithm>
#include <mutex>

#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kBM = 128;          // query rows per CTA
constexpr int kDim = 128;         // head dim
constexpr int kMaxRegions = 16;
constexpr uint32_t kHalfBytes = 128u * 128u;     // 16 KB: 128 rows x 128 B (P, bf16 Q and K)
constexpr float kRedoThreshold = 64.0f;           // log2 units: P stays below 2^64
constexpr float kRedoBound = 18446744073709551616.0f;  // 2^64

// Tile geometry of the two variants. bf16 Q/K: 128-key tiles, Q and K tiles
// as two 64-feature halves of 128 B rows. MXFP8 Q/K: E4M3 rows of 128 B
// (one swizzle row per token), 112-key tiles: S then takes 112 TMEM columns
// per group, which leaves columns 496-511 free for the E8M0 scale vectors.
template <bool kMx>
struct Tile {
  static constexpr int BN = kMx ? 112 : 128;                         // keys per tile
  static constexpr int KStages = kMx ? 3 : 2;                        // K tile ring
  static constexpr int VStages = kMx ? 3 : 2;                        // V tile ring
  static constexpr uint32_t QBytes = kMx ? 128u * 128u : 2u * kHalfBytes;
  static constexpr uint32_t KBytes = kMx ? BN * 128u : 2u * kHalfBytes;
  static constexpr uint32_t VHalf = BN * 128u;                       // 64 features x BN rows
  static constexpr uint32_t VBytes = 2u * VHalf;
};

// Scale-factor block of a 128-row (or key) MXFP8 tile as the tensor core reads
// it from TMEM: byte (r % 32) * 16 + (r / 32) * 4 + b holds the E8M0 scale of
// row r and 32-feature block b. tcgen05.cp (32 rows x 16 B, replicated to the
// four lane quadrants) moves it to four TMEM columns: lane r % 32 (+ 32 q),
// column r / 32, byte b; the MMA picks byte b through its scale-factor ids.
__host__ __device__ constexpr uint32_t sf_offset(int r, int b) {
  return static_cast<uint32_t>((r % 32) * 16 + (r / 32) * 4 + b);
}

constexpr int kBN = Tile<false>::BN;  // key tile of the bf16 variant (int4 history, lists)

template <bool kMx>
struct __align__(1024) ChunkSmem {
  static constexpr int kKStages = Tile<kMx>::KStages;
  static constexpr int kVStages = Tile<kMx>::VStages;
  uint8_t q[Tile<kMx>::QBytes];             // bf16: 2 x [128 rows][128 B]; MXFP8: [128][128 B]
  uint8_t k[kKStages][Tile<kMx>::KBytes];   // swizzled like q, BN rows
  uint8_t v[kVStages][Tile<kMx>::VBytes];   // 2 x [BN rows][128 B] (64 features each)
  uint8_t p[2][2 * kHalfBytes];             // P (bf16) of group A and B, K-major A operand
  uint8_t sfa[kMx ? 512 : 16];              // MXFP8: Q scale block
  uint8_t sfb[kKStages][kMx ? 512 : 16];    // MXFP8: K scale block per stage
  uint64_t q_full;
  uint64_t k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[2], s_free[2], p_full[2], o_done[2], mma_done;
  uint32_t tmem_base;
  int abort_flag;
  int rb[kMaxRegions + 1];                  // region bounds (a copy of ChunkArgs::reg.b)
};

// The two groups' row states for the final merge, laid over the Q tile and
// the first K stage (contiguous), which no copy or MMA touches any more once
// a group has seen its last PV complete: every QK MMA was issued before it.
struct MergeState {
  float m[kBM], l[kBM];
  float r[kMaxRegions][kBM];
};
static_assert(2 * sizeof(MergeState) <= Tile<false>::QBytes + Tile<false>::KBytes &&
                  2 * sizeof(MergeState) <= Tile<true>::QBytes + Tile<true>::KBytes,
              "merge states fit over Q and K stage 0");

struct ChunkArgs {
  int n_q, n_kv, q_heads, kv_group, n_tiles;
  // block-shared candidate lists: 0, or the 128-row query tiles per list;
  // K/V row set of CTA (x, y) is then list y * lists_per_head + x / tiles_per_list
  int tiles_per_list, lists_per_head;
  // key tiles below hist_tiles come from the K/V maps; the later ones from
  // the window maps, at row key - win_off (an int4-history cache whose
  // expanded history is followed by its bf16 window read in place)
  int hist_tiles, win_off;
  float scale_log2;
  void *out;
  int out_dtype;
  float *mass;
  Regions reg;
  KernelCtl ctl;
  // MXFP8 only: Q scale blocks [hq][q tiles][512 B]; K window scales
  // [unit][Ws][4] (E8M0 bytes) with Ws rows per unit
  const uint8_t *q_sf;
  const uint8_t *k_e8m0;
  int k_ws;
};

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Block-scaled E4M3 x E4M3 MMA: the E8M0 scale vectors of A (rows) and B
// (keys) are read from TMEM at sfa / sfb; the byte used (the 32-feature block)
// is chosen by the scale-factor ids in the instruction descriptor.
__device__ __forceinline__ void tc_mma_mx(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// Shared-memory descriptor without swizzle (rows of 16 B, 8-row groups 128 B
// apart): the source of a scale-block copy.
__device__ __forceinline__ uint64_t smem_desc_plain(uint32_t addr) {
  uint64_t d = static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(16u >> 4) << 16;
  d |= static_cast<uint64_t>(128u >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// A 512-byte scale block (32 rows x 16 B) to four TMEM columns, replicated to
// all four lane quadrants; ordered before the MMAs this thread issues next.
__device__ __forceinline__ void tc_copy_sf(uint32_t taddr, uint32_t src) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr),
               "l"(smem_desc_plain(src))
               : "memory");
}

// 32 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Registers written by tcgen05.ld hold valid data only after tcgen05.wait::ld;
// this empty asm, placed after the wait, keeps the compiler from moving any
// use of them above it.
__device__ __forceinline__ void reg_fence(float (&v)[32]) {
  asm volatile(""
               : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]),
                 "+f"(v[6]), "+f"(v[7]), "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]),
                 "+f"(v[12]), "+f"(v[13]), "+f"(v[14]), "+f"(v[15]), "+f"(v[16]), "+f"(v[17]),
                 "+f"(v[18]), "+f"(v[19]), "+f"(v[20]), "+f"(v[21]), "+f"(v[22]), "+f"(v[23]),
                 "+f"(v[24]), "+f"(v[25]), "+f"(v[26]), "+f"(v[27]), "+f"(v[28]), "+f"(v[29]),
                 "+f"(v[30]), "+f"(v[31])::"memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: 128B swizzle, version 1 (bits 46-48).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulator, M=128,
// N=n, A K-major, B K-major (b_mn_major = 0) or MN-major (1).
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t b_mn_major, uint32_t n = 128) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn_major << 16) | ((n >> 3) << 17) |
         ((128u >> 4) << 24);
}

// Instruction descriptor, kind::mxf8f6f4 block-scaled: E4M3 A and B (format
// 0), both K-major, N=n, UE8M0 scales (bit 23), M=128; the scale-factor ids of
// B (bits 4-5) and A (bits 29-30) select byte `blk` of the scale vectors.
__host__ __device__ constexpr uint32_t idesc_mx(uint32_t n, uint32_t blk) {
  return (blk << 4) | ((n >> 3) << 17) | (1u << 23) | ((128u >> 4) << 24) | (blk << 29);
}

__device__ __forceinline__ bool cta_aborted(int *abort_flag) {
  return *reinterpret_cast<volatile int *>(abort_flag) != 0;
}

__device__ __forceinline__ bool wait_or_abort(int *abort_flag, uint32_t bar, uint32_t parity,
                                              const KernelCtl &ctl) {
  if (mbar_wait(bar, parity, ctl.wait_limit_ns)) return true;
  flag_error(ctl, KVQ_DEV_TIMEOUT);
  *reinterpret_cast<volatile int *>(abort_flag) = 1;
  return false;
}

// Byte offset of 16-byte chunk c (0..7) of row r inside a 128B-swizzled
// [rows][128 B] region that starts on a 1024-byte boundary.
__device__ __forceinline__ uint32_t swz(uint32_t r, uint32_t c) {
  return r * 128u + ((c ^ (r & 7u)) << 4);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&b);
}

// Scale 128 fp32 TMEM columns of this thread's lane by f.
__device__ __forceinline__ void scale_tmem_row(uint32_t taddr, float f) {
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    float v[32];
    tmem_ld32(taddr + 32u * c, v);
    tmem_wait_ld();
    reg_fence(v);
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] *= f;
    tmem_st32(taddr + 32u * c, v);
  }
  tmem_wait_st();
}

// Maximum of the first `valid` of this lane's 128 score columns.
__device__ __forceinline__ float row_max(uint32_t taddr, int valid) {
  float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    float v[32];
    tmem_ld32(taddr + 32u * c, v);
    tmem_wait_ld();
    reg_fence(v);
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      mx0 = fmaxf(mx0, 32 * c + e < valid ? v[e] : -CUDART_INF_F);
      mx1 = fmaxf(mx1, 32 * c + e + 1 < valid ? v[e + 1] : -CUDART_INF_F);
    }
  }
  return fmaxf(mx0, mx1);
}

// Paired fp32 arithmetic (one instruction for two lanes of work):
// (y0, y1) = (x0, x1) * (s, s) + (n, n), and (a0, a1) += (x0, x1).
__device__ __forceinline__ void fma2(float &y0, float &y1, float x0, float x1, float s, float n) {
  asm("{\n\t.reg .b64 x, s, n, y;\n\t"
      "mov.b64 x, {%2, %3};\n\tmov.b64 s, {%4, %4};\n\tmov.b64 n, {%5, %5};\n\t"
      "fma.rn.f32x2 y, x, s, n;\n\tmov.b64 {%0, %1}, y;\n\t}"
      : "=f"(y0), "=f"(y1)
      : "f"(x0), "f"(x1), "f"(s), "f"(n));
}
__device__ __forceinline__ void add2(float &a0, float &a1, float x0, float x1) {
  asm("{\n\t.reg .b64 a, x;\n\t"
      "mov.b64 a, {%0, %1};\n\tmov.b64 x, {%2, %3};\n\t"
      "add.rn.f32x2 a, a, x;\n\tmov.b64 {%0, %1}, a;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(x0), "f"(x1));
}

// Running region sums of one row. The keys a softmax group sees arrive in
// increasing order, so the region under the current key only moves forward:
// `cur` sums region k, and a region that has been left is stored in done[]
// (indexed at run time, so it lives in local memory; it is written once per
// region, not per key). k is the same in every thread of a group.
struct RegionAcc {
  int k;
  float cur;
  float *done;
};

// Move to the region holding key `pos`, storing the sums of those passed.
__device__ __forceinline__ void region_seek(RegionAcc &r, const int *rb, int n, int pos) {
  while (r.k + 1 < n && rb[r.k + 1] <= pos) {
    r.done[r.k] = r.cur;
    r.cur = 0.0f;
    ++r.k;
  }
}

// Sum of v[e] for lo <= e < hi.
__device__ __forceinline__ float range_sum(const float (&v)[32], int lo, int hi) {
  float a = 0.0f, b = 0.0f;
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    a += (e >= lo && e < hi) ? v[e] : 0.0f;
    b += (e + 1 >= lo && e + 1 < hi) ? v[e + 1] : 0.0f;
  }
  return a + b;
}

// 32 columns of the pass: P = 2^(s * scale + neg_m) for the valid ones (0
// beyond), raw maximum, P to shared memory as bf16, the chunk's sum. Region
// sums: byte c of offs is the offset of the one region bound inside chunk c
// (32: none); psum then receives the sum of the chunk's keys before it, and
// the caller does the accounting once P is handed over. With kSplit (some
// chunk of the tile holds two or more bounds) the chunk's keys are added to
// the region sums here instead, split at every bound inside the chunk.
template <bool kSplit, bool kMax = true>
__device__ __forceinline__ void softmax_chunk(float (&v)[32], int c, int valid, int t0,
                                              float scale, float neg_m, const int *rb, int nreg,
                                              uint32_t offs, uint8_t *p, int row, float &cs,
                                              float &psum, RegionAcc &racc, float &mx0,
                                              float &mx1) {
  float ps4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  if (32 * c + 32 <= valid) {
    if (kMax) {
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        mx0 = fmaxf(mx0, v[e]);
        mx1 = fmaxf(mx1, v[e + 1]);
      }
    }
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      fma2(v[e], v[e + 1], v[e], v[e + 1], scale, neg_m);
      v[e] = fast_exp2(v[e]);
      v[e + 1] = fast_exp2(v[e + 1]);
      if (e & 2)
        add2(ps4[2], ps4[3], v[e], v[e + 1]);
      else
        add2(ps4[0], ps4[1], v[e], v[e + 1]);
    }
  } else if (32 * c + 16 == valid) {
    // exactly 16 keys (the last chunk of a 112-key tile)
    if (kMax) {
#pragma unroll
      for (int e = 0; e < 16; e += 2) {
        mx0 = fmaxf(mx0, v[e]);
        mx1 = fmaxf(mx1, v[e + 1]);
      }
    }
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
      fma2(v[e], v[e + 1], v[e], v[e + 1], scale, neg_m);
      v[e] = fast_exp2(v[e]);
      v[e + 1] = fast_exp2(v[e + 1]);
      if (e & 2)
        add2(ps4[2], ps4[3], v[e], v[e + 1]);
      else
        add2(ps4[0], ps4[1], v[e], v[e + 1]);
    }
#pragma unroll
    for (int e = 16; e < 32; ++e) v[e] = 0.0f;
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const bool in = 32 * c + e < valid;
      if (kMax) {
        if (e & 1)
          mx1 = fmaxf(mx1, in ? v[e] : -CUDART_INF_F);
        else
          mx0 = fmaxf(mx0, in ? v[e] : -CUDART_INF_F);
      }
      v[e] = in ? fast_exp2(fmaf(v[e], scale, neg_m)) : 0.0f;
      ps4[e & 3] += v[e];
    }
  }
#pragma unroll
  for (int q8 = 0; q8 < 4; ++q8) {
    const int chunk = 4 * c + q8;  // 16-byte chunk of the row, 0..15
    uint4 w;
    w.x = pack_bf16x2(v[8 * q8 + 0], v[8 * q8 + 1]);
    w.y = pack_bf16x2(v[8 * q8 + 2], v[8 * q8 + 3]);
    w.z = pack_bf16x2(v[8 * q8 + 4], v[8 * q8 + 5]);
    w.w = pack_bf16x2(v[8 * q8 + 6], v[8 * q8 + 7]);
    *reinterpret_cast<uint4 *>(p + (chunk >> 3) * kHalfBytes + swz(row, chunk & 7)) = w;
  }
  cs = (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
  if (!kSplit) {
    const int off = static_cast<int>((offs >> (8 * c)) & 0xffu);
    if (off < 32) psum = range_sum(v, 0, off);
  } else {
    const int start = t0 + 32 * c;
    region_seek(racc, rb, nreg, start);
    int lo = 0;
    while (racc.k + 1 < nreg && rb[racc.k + 1] < start + 32) {  // a bound inside the chunk
      const int o = rb[racc.k + 1] - start;
      racc.done[racc.k] = racc.cur + range_sum(v, lo, o);
      racc.cur = 0.0f;
      ++racc.k;
      lo = o;
    }
    racc.cur += lo == 0 ? cs : range_sum(v, lo, 32);
  }
}

// The pass over the 128 score columns of this thread's row, up to the last
// chunk: chunks 0-2 are exponentiated and stored while the TMEM load of the
// next is in flight; chunk 3 is left raw in v3, and mx is its raw maximum, so
// that the caller can release S before finishing it. cs[c]: sum of chunk c.
// With set_ref (a group's first tile) the reference is taken from chunk 0's
// maximum, stored in ref_out, and used for the whole tile.
template <bool kSplit>
__device__ __forceinline__ void softmax_pass_head(uint32_t taddr, int valid, int t0, float scale,
                                                  float neg_m, const int *rb, int nreg,
                                                  uint32_t offs, uint8_t *p, int row,
                                                  float (&cs)[4], float (&psum)[4],
                                                  RegionAcc &racc, float (&v3)[32], float &mx,
                                                  bool set_ref, float &ref_out) {
  float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
  float va[32];
  tmem_ld32(taddr, va);
  tmem_wait_ld();
  reg_fence(va);
  tmem_ld32(taddr + 32u, v3);
  if (set_ref) {  // chunk 0 holds at least one valid key
    float r0 = -CUDART_INF_F, r1 = -CUDART_INF_F;
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      r0 = fmaxf(r0, e < valid ? va[e] : -CUDART_INF_F);
      r1 = fmaxf(r1, e + 1 < valid ? va[e + 1] : -CUDART_INF_F);
    }
    const float ref = fmaxf(r0, r1) * scale;  // scale > 0 keeps the order
    ref_out = ref;
    neg_m = -ref;
  }
  softmax_chunk<kSplit, false>(va, 0, valid, t0, scale, neg_m, rb, nreg, offs, p, row, cs[0],
                               psum[0], racc, mx0, mx1);
  tmem_wait_ld();
  reg_fence(v3);
  tmem_ld32(taddr + 64u, va);
  softmax_chunk<kSplit, false>(v3, 1, valid, t0, scale, neg_m, rb, nreg, offs, p, row, cs[1],
                               psum[1], racc, mx0, mx1);
  tmem_wait_ld();
  reg_fence(va);
  tmem_ld32(taddr + 96u, v3);
  softmax_chunk<kSplit, false>(va, 2, valid, t0, scale, neg_m, rb, nreg, offs, p, row, cs[2],
                               psum[2], racc, mx0, mx1);
  tmem_wait_ld();
  reg_fence(v3);
  if (valid >= 128) {
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      mx0 = fmaxf(mx0, v3[e]);
      mx1 = fmaxf(mx1, v3[e + 1]);
    }
  } else if (valid == 112) {
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
      mx0 = fmaxf(mx0, v3[e]);
      mx1 = fmaxf(mx1, v3[e + 1]);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      mx0 = fmaxf(mx0, 96 + e < valid ? v3[e] : -CUDART_INF_F);
      mx1 = fmaxf(mx1, 97 + e < valid ? v3[e + 1] : -CUDART_INF_F);
    }
  }
  mx = fmaxf(mx0, mx1);
}

// The kernel body, for bf16 Q/K (kind::f16 QK) and MXFP8 Q/K (block-scaled
// kind::mxf8f6f4 QK); PV is a bf16 kind::f16 MMA in both.
template <bool kMx>
__device__ __forceinline__ void chunk_body(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                                           const CUtensorMap &tm_v, const CUtensorMap &tm_kw,
                                           const CUtensorMap &tm_vw, const ChunkArgs &a) {
  using T = Tile<kMx>;
  constexpr int BN = T::BN;
  constexpr int kKStages = T::KStages, kVStages = T::VStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // dynamic shared memory is only 16-byte aligned: round up to 1024
  const uint32_t base = smem_u32(smem_raw);
  ChunkSmem<kMx> &sm =
      *reinterpret_cast<ChunkSmem<kMx> *>(smem_raw + (((base + 1023u) & ~1023u) - base));
  int *const abort_flag = &sm.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = blockIdx.x * kBM;
  const int hq = blockIdx.y;                 // b * q_heads + h
  const int hkv = a.tiles_per_list
                      ? hq * a.lists_per_head + static_cast<int>(blockIdx.x) / a.tiles_per_list
                      : (hq / a.q_heads) * (a.q_heads / a.kv_group) + (hq % a.q_heads) / a.kv_group;
  const int nt = a.n_tiles;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.q_full), kMx ? 32 : 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(smem_u32(&sm.k_full[s]), kMx ? 32 : 1);
      mbar_init(smem_u32(&sm.k_empty[s]), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(smem_u32(&sm.v_full[s]), 1);
      mbar_init(smem_u32(&sm.v_empty[s]), 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(smem_u32(&sm.s_full[g]), 1);
      mbar_init(smem_u32(&sm.s_free[g]), 128);
      mbar_init(smem_u32(&sm.p_full[g]), 128);
      mbar_init(smem_u32(&sm.o_done[g]), 1);
    }
    mbar_init(smem_u32(&sm.mma_done), 1);
    sm.abort_flag = 0;
#pragma unroll
    for (int i = 0; i <= kMaxRegions; ++i) sm.rb[i] = a.reg.b[i];
    fence_mbar_init();
  }
  if (kMx && warp == 3) {
    // the scale slots of rows 112-127 of a key block are never written:
    // give them a valid scale (1.0) once, so no byte is ever NaN
    for (int i = lane; i < kKStages * 128; i += 32)
      reinterpret_cast<uint32_t *>(sm.sfb)[i] = 0x7f7f7f7fu;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                     smem_u32(&sm.tmem_base))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The barriers and TMEM are set up while the previous kernel drains; its
  // outputs (the expanded or gathered K and V rows, the MXFP8 Q) are read
  // only after this.
  wait_prior_grid();
  allow_next_grid();
  const uint32_t tmem = sm.tmem_base;
  // bf16: group g's S at columns 256g, O at 256g + 128. MXFP8: O at 128g, S
  // (112 columns) at 256 + 128g, Q scales at 496, K scales of stage s at 500 + 4s.
  auto t_s = [&](int g) { return tmem + (kMx ? 256u + 128u * g : 256u * g); };
  auto t_o = [&](int g) { return tmem + (kMx ? 128u * g : 256u * g + 128u); };
  const uint32_t t_sfa = tmem + 496u;
  auto t_sfb = [&](int st) { return tmem + 500u + 4u * st; };

  if (warp == 0) {
    // ------------------------------------------------ TMA producer: Q, then K tiles
    // With MXFP8 every lane also moves scale bytes into the stage's scale
    // block and arrives on its barrier (32 arrivals); lane 0 posts the
    // copy's byte count first so that the phase waits for the copy too.
    const uint32_t qb = smem_u32(&sm.q_full);
    if (lane == 0) {
      if (kMx)
        mbar_expect_tx(qb, T::QBytes);
      else
        mbar_arrive_expect_tx(qb, T::QBytes);
      tma_load_3d(smem_u32(sm.q), &tm_q, 0, q0, hq, qb);
      if (!kMx) tma_load_3d(smem_u32(sm.q) + kHalfBytes, &tm_q, 64, q0, hq, qb);
    }
    // MXFP8: the K scales of a tile are loaded into registers one tile ahead
    // (lane l holds keys l, l + 32, l + 64, l + 96; 1.0 past the last key)
    uint32_t sfw[4] = {0u, 0u, 0u, 0u};
    auto load_sf = [&](int kj) {
      const int valid = min(BN, a.n_kv - kj * BN);
      const uint32_t *e8 = reinterpret_cast<const uint32_t *>(a.k_e8m0) +
                           static_cast<long>(hkv) * a.k_ws + kj * BN;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        sfw[i] = lane + 32 * i < valid && in_bounds(a.ctl, e8 + lane + 32 * i, 4)
                     ? e8[lane + 32 * i]
                     : 0x7f7f7f7fu;
    };
    if (kMx) {
      // the Q tile's scale block, laid out by the prologue as the MMA reads it
      const uint4 *src = reinterpret_cast<const uint4 *>(
          a.q_sf + (static_cast<long>(hq) * gridDim.x + blockIdx.x) * 512);
      reinterpret_cast<uint4 *>(sm.sfa)[lane] =
          in_bounds(a.ctl, src + lane, 16) ? src[lane] : make_uint4(0x7f7f7f7fu, 0x7f7f7f7fu,
                                                                    0x7f7f7f7fu, 0x7f7f7f7fu);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(qb);
      if (nt > 0) load_sf(0);
    }
    // a stage is reused once the MMA reading it has completed
    int kj = 0;
    for (; kj < nt; ++kj) {
      const int st = kj % kKStages, use = kj / kKStages;
      // every lane waits: with MXFP8 every lane then writes the stage's scales
      bool go = use == 0 ||
                wait_or_abort(abort_flag, smem_u32(&sm.k_empty[st]), (use - 1) & 1, a.ctl);
      go = __all_sync(0xffffffffu, go) && !cta_aborted(abort_flag);
      if (!go) break;
      const uint32_t fb = smem_u32(&sm.k_full[st]);
      if (lane == 0) {
        if (kMx)
          mbar_expect_tx(fb, T::KBytes);
        else
          mbar_arrive_expect_tx(fb, T::KBytes);
        const bool hist = kj < a.hist_tiles;
        const CUtensorMap *mk = hist ? &tm_k : &tm_kw;
        const int ky = hist ? kj * BN : kj * BN - a.win_off;
        tma_load_3d(smem_u32(sm.k[st]), mk, 0, ky, hkv, fb);
        if (!kMx) tma_load_3d(smem_u32(sm.k[st]) + kHalfBytes, mk, 64, ky, hkv, fb);
      }
      if (kMx) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (lane + 32 * i < BN)
            *reinterpret_cast<uint32_t *>(sm.sfb[st] + sf_offset(lane + 32 * i, 0)) = sfw[i];
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(fb);
        if (kj + 1 < nt) load_sf(kj + 1);
      }
    }
    // drain: the copies of the last stages must land before the CTA exits
    if (lane == 0) {
      mbar_wait(qb, 0, 2000000000ull);
      for (int d = (kj > kKStages ? kj - kKStages : 0); d < kj; ++d)
        mbar_wait(smem_u32(&sm.k_full[d % kKStages]), (d / kKStages) & 1, 2000000000ull);
    }
  } else if (warp == 2) {
    // ------------------------------------------------ TMA producer: V tiles
    if (lane == 0) {
      int vj = 0;
      for (; vj < nt; ++vj) {
        const int st = vj % kVStages, use = vj / kVStages;
        if (use > 0 &&
            !wait_or_abort(abort_flag, smem_u32(&sm.v_empty[st]), (use - 1) & 1, a.ctl))
          break;
        if (cta_aborted(abort_flag)) break;
        const uint32_t fb = smem_u32(&sm.v_full[st]);
        mbar_arrive_expect_tx(fb, T::VBytes);
        const bool hist = vj < a.hist_tiles;
        const CUtensorMap *mv = hist ? &tm_v : &tm_vw;
        const int vy = hist ? vj * BN : vj * BN - a.win_off;
        tma_load_3d(smem_u32(sm.v[st]), mv, 0, vy, hkv, fb);
        tma_load_3d(smem_u32(sm.v[st]) + T::VHalf, mv, 64, vy, hkv, fb);
      }
      for (int d = (vj > kVStages ? vj - kVStages : 0); d < vj; ++d)
        mbar_wait(smem_u32(&sm.v_full[d % kVStages]), (d / kVStages) & 1, 2000000000ull);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_bf16(0), id_pv = idesc_bf16(1);
      const uint32_t qa = smem_u32(sm.q);
      bool ok = wait_or_abort(abort_flag, smem_u32(&sm.q_full), 0, a.ctl);
      if (kMx && ok) {
        tc_fence_after();
        tc_copy_sf(t_sfa, smem_u32(sm.sfa));
      }
      // S_j = Q K_j^T into group j % 2's S
      auto issue_s = [&](int j) -> bool {
        const int st = j % kKStages, g = j & 1;
        if (!wait_or_abort(abort_flag, smem_u32(&sm.k_full[st]), (j / kKStages) & 1, a.ctl))
          return false;
        tc_fence_after();
        const uint32_t ka = smem_u32(sm.k[st]);
        if (kMx) {
          tc_copy_sf(t_sfb(st), smem_u32(sm.sfb[st]));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_mx(t_s(g), smem_desc(qa + 32u * kk, 16, 1024), smem_desc(ka + 32u * kk, 16, 1024),
                      idesc_mx(BN, kk), t_sfa, t_sfb(st), kk > 0 ? 1u : 0u);
        } else {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32u;
            tc_mma_f16(t_s(g), smem_desc(qa + off, 16, 1024), smem_desc(ka + off, 16, 1024),
                       id_qk, kk > 0 ? 1u : 0u);
          }
        }
        tc_commit(smem_u32(&sm.s_full[g]));
        tc_commit(smem_u32(&sm.k_empty[st]));
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok && nt > 1) ok = issue_s(1);
      for (int j = 0; ok && j < nt; ++j) {
        const int st = j % kVStages, g = j & 1, i = j >> 1;
        // S_g can take tile j + 2 as soon as group g holds tile j's scores in
        // registers, before its P is written
        if (j + 2 < nt &&
            (!wait_or_abort(abort_flag, smem_u32(&sm.s_free[g]), i & 1, a.ctl) || !issue_s(j + 2))) {
          ok = false;
          break;
        }
        // O_g += P_g V_j once group g has written P for tile j
        if (!wait_or_abort(abort_flag, smem_u32(&sm.p_full[g]), i & 1, a.ctl) ||
            !wait_or_abort(abort_flag, smem_u32(&sm.v_full[st]), (j / kVStages) & 1, a.ctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t pa = smem_u32(sm.p[g]), va = smem_u32(sm.v[st]);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t ad = smem_desc(pa + (kk >> 2) * kHalfBytes + (kk & 3) * 32u, 16, 1024);
          const uint64_t bd = smem_desc(va + kk * 2048u, T::VHalf, 1024);
          tc_mma_f16(t_o(g), ad, bd, id_pv, (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(smem_u32(&sm.o_done[g]));
        tc_commit(smem_u32(&sm.v_empty[st]));
      }
      // all MMAs of this CTA complete before TMEM is released
      tc_commit(smem_u32(&sm.mma_done));
      mbar_wait(smem_u32(&sm.mma_done), 0, 2000000000ull);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------ softmax groups
    const int g = (warp - 4) >> 2;           // 0: even tiles, 1: odd tiles
    const int quad = warp & 3;               // TMEM lanes 32*quad .. +31
    const int row = quad * 32 + lane;        // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_row = t_s(g) + lane_off, o_row = t_o(g) + lane_off;
    const int my_tiles = (nt - g + 1) >> 1;  // tiles g, g+2, ...
    // Row state: P is taken against a reference m_used, set from the row's
    // maximum over the first 32 scores of its first tile and kept while P stays below
    // 2^kRedoThreshold (bf16 P and the fp32 sums have the range for it, so no
    // running maximum is kept); a tile that would pass that bound raises the
    // reference to its maximum and is redone.
    float m_used = -CUDART_INF_F, l = 0.0f;
    const int nreg = a.reg.n;
    const int *rb = sm.rb;
    float done[kMaxRegions];
    RegionAcc racc;
    racc.k = 0;
    racc.cur = 0.0f;
    racc.done = done;
    bool ok = true;
    for (int i = 0; i < my_tiles; ++i) {
      const int j = 2 * i + g;
      if (!wait_or_abort(abort_flag, smem_u32(&sm.s_full[g]), i & 1, a.ctl)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int valid = min(BN, a.n_kv - j * BN);
      const int t0 = j * BN;
      // O_g += P V of the previous tile must be done before P_g is rewritten
      // or O_g is rescaled
      if (i >= 1 && !wait_or_abort(abort_flag, smem_u32(&sm.o_done[g]), (i - 1) & 1, a.ctl)) {
        ok = false;
        break;
      }
      // Regions of the tile (the same for every row of the group): `whole`
      // when it lies inside one region; otherwise offs holds, per 32-key
      // chunk, the offset of the one bound strictly inside it (32: none),
      // and `split` is set when some chunk holds two or more (tiny regions:
      // accounted key by key during the pass, from a state kept so that a
      // redone tile is counted once).
      bool whole = true, split = false;
      uint32_t offs = 0x20202020u;
      if (nreg > 0) {
        region_seek(racc, rb, nreg, t0);
        for (int b = racc.k + 1; b < nreg && rb[b] < t0 + valid; ++b) {
          whole = false;
          const int o = rb[b] - t0, c = o >> 5, oc = o & 31;
          if (oc == 0) continue;  // a bound on a chunk start needs no split
          if (((offs >> (8 * c)) & 0xffu) != 32u) split = true;
          offs = (offs & ~(0xffu << (8 * c))) | (static_cast<uint32_t>(oc) << (8 * c));
        }
      }
      const int k_before = racc.k;
      const float cur_before = racc.cur;
      // one pass: P = 2^(s * scale - m_used) -> shared memory, sums; the
      // group's first tile sets m_used from its first 32 scores
      float cs[4], psum[4], v3[32], mx, dummy0 = 0.0f, dummy1 = 0.0f;
      bool set_ref = i == 0;
      for (;;) {
        if (split)
          softmax_pass_head<true>(s_row, valid, t0, a.scale_log2, -m_used, rb, nreg, offs,
                                  sm.p[g], row, cs, psum, racc, v3, mx, set_ref, m_used);
        else
          softmax_pass_head<false>(s_row, valid, t0, a.scale_log2, -m_used, rb, nreg, offs,
                                   sm.p[g], row, cs, psum, racc, v3, mx, set_ref, m_used);
        // A chunk sum bounds each of its P values: chunks 0-2 are checked by
        // their sums, chunk 3 by its raw maximum.
        const float big = fmaxf(fmaxf(cs[0], cs[1]), cs[2]);
        if (!__any_sync(0xffffffffu,
                        !(big <= kRedoBound) || mx * a.scale_log2 > m_used + kRedoThreshold))
          break;
        // far above the reference for some row (P could overflow): the warp
        // takes the tile maxima now and redoes the tile from its scores, still
        // in TMEM (TMEM access is warp-wide); O_g is idle, its last MMA is
        // done. The new reference is the tile's maximum, so a second pass
        // never redoes again.
        const float m_new = fmaxf(m_used, row_max(s_row, valid) * a.scale_log2);
        const float f = fast_exp2(m_used - m_new);
        m_used = m_new;
        l *= f;
        racc.k = k_before;
        racc.cur = cur_before * f;
        for (int k = 0; k < k_before; ++k) done[k] *= f;
        if (i >= 1) {
          tc_fence_after();
          scale_tmem_row(o_row, f);
        }
        set_ref = false;
      }
      // every score of the tile is in registers: S_g may take the next tile
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.s_free[g]));
      if (split)
        softmax_chunk<true, false>(v3, 3, valid, t0, a.scale_log2, -m_used, rb, nreg, offs,
                                   sm.p[g], row, cs[3], psum[3], racc, dummy0, dummy1);
      else
        softmax_chunk<false, false>(v3, 3, valid, t0, a.scale_log2, -m_used, rb, nreg, offs,
                                    sm.p[g], row, cs[3], psum[3], racc, dummy0, dummy1);
      // P is complete: hand it to the MMA warp, then do the bookkeeping
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.p_full[g]));
      const float tile_sum = (cs[0] + cs[1]) + (cs[2] + cs[3]);
      l += tile_sum;
      if (nreg > 0 && !split) {
        if (whole) {
          racc.cur += tile_sum;
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            region_seek(racc, rb, nreg, t0 + 32 * c);
            if (((offs >> (8 * c)) & 0xffu) < 32u) {  // the chunk ends one region
              done[racc.k] = racc.cur + psum[c];
              racc.cur = cs[c] - psum[c];
              ++racc.k;
            } else {
              racc.cur += cs[c];
            }
          }
        }
      }
    }
    // ---- epilogue: each group leaves its row state in shared memory, then
    // merges both groups' O for half of the columns (group g: 64g .. 64g + 63)
    const bool mine_ok =
        ok && (my_tiles == 0 ||
               wait_or_abort(abort_flag, smem_u32(&sm.o_done[g]), (my_tiles - 1) & 1, a.ctl));
    // A group's last PV is issued after the last QK, so once it has completed
    // no MMA reads Q or K stage 0 any more and the group may write over them.
    MergeState *ms = reinterpret_cast<MergeState *>(sm.q);
    if (mine_ok && my_tiles > 0) {
      ms[g].m[row] = m_used;
      ms[g].l[row] = l;
      if (nreg > 0) {
        region_seek(racc, rb, nreg, a.n_kv);  // store the open regions' sums
        done[racc.k] = racc.cur;
        for (int k = 0; k < nreg; ++k) ms[g].r[k][row] = done[k];
      }
    }
    tc_fence_before();
    asm volatile("bar.sync 2, 256;" ::: "memory");
    const int other = 1 - g;
    const int other_tiles = (nt - other + 1) >> 1;
    if (mine_ok &&
        (other_tiles == 0 ||
         wait_or_abort(abort_flag, smem_u32(&sm.o_done[other]), (other_tiles - 1) & 1, a.ctl))) {
      tc_fence_after();
      const bool have_b = nt > 1;  // group B processed at least one tile (group A always)
      const float ma = ms[0].m[row], mb = have_b ? ms[1].m[row] : -CUDART_INF_F;
      const float mm = fmaxf(ma, mb);
      const float fa = exp2f(ma - mm);
      const float fb = have_b ? exp2f(mb - mm) : 0.0f;
      const float inv = 1.0f / (fa * ms[0].l[row] + (have_b ? fb * ms[1].l[row] : 0.0f));
      const int qrow = q0 + row;
      const long obase = (static_cast<long>(hq) * a.n_q + qrow) * kDim;
#pragma unroll
      for (int c = 2 * g; c < 2 * g + 2; ++c) {
        float va[32], vb[32];
        tmem_ld32(t_o(0) + lane_off + 32u * c, va);
        if (have_b) tmem_ld32(t_o(1) + lane_off + 32u * c, vb);
        tmem_wait_ld();
        reg_fence(va);
        if (have_b) reg_fence(vb);
#pragma unroll
        for (int e = 0; e < 32; ++e) va[e] = (fa * va[e] + (have_b ? fb * vb[e] : 0.0f)) * inv;
        const size_t ob = a.out_dtype == KVQ_F32 ? 4 : 2;
        if (qrow < a.n_q &&
            in_bounds(a.ctl, static_cast<uint8_t *>(a.out) + (obase + 32 * c) * ob, 32 * ob)) {
          if (a.out_dtype == KVQ_F32) {
            float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(a.out) + obase + 32 * c);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              o[e] = make_float4(va[4 * e], va[4 * e + 1], va[4 * e + 2], va[4 * e + 3]);
          } else {
            uint4 *o =
                reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) + obase + 32 * c);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              o[e] = make_uint4(pack_bf16x2(va[8 * e], va[8 * e + 1]),
                                pack_bf16x2(va[8 * e + 2], va[8 * e + 3]),
                                pack_bf16x2(va[8 * e + 4], va[8 * e + 5]),
                                pack_bf16x2(va[8 * e + 6], va[8 * e + 7]));
          }
        }
      }
      if (g == 0 && a.mass && qrow < a.n_q &&
          in_bounds(a.ctl, a.mass + (static_cast<long>(hq) * a.n_q + qrow) * a.reg.n,
                    sizeof(float) * nreg))
        for (int k = 0; k < nreg; ++k)
          a.mass[(static_cast<long>(hq) * a.n_q + qrow) * a.reg.n + k] =
              (fa * ms[0].r[k][row] + (have_b ? fb * ms[1].r[k][row] : 0.0f)) * inv;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

__global__ void __launch_bounds__(384, 1)
    chunk_bf16_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_kw,
                      const __grid_constant__ CUtensorMap tm_vw, const ChunkArgs a) {
  chunk_body<false>(tm_q, tm_k, tm_v, tm_kw, tm_vw, a);
}

__global__ void __launch_bounds__(384, 1)
    chunk_mxfp8_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const ChunkArgs a) {
  chunk_body<true>(tm_q, tm_k, tm_v, tm_k, tm_v, a);
}

// ------------------------------------------------------------------ MXFP8 Q prologue
// The MXFP8 path (Catnip study, section "Q/K 与 probability quantization 的影响":
// E4M3 elements with an E8M0 scale per 32 features) takes K as kv_pack stored
// it (E4M3 window + E8M0 bytes) and rounds Q to MXFP8 with the same rule here:
// E4M3 codes [hq][n_q][128] and, per 128-row query tile, the scale block in
// the layout the tensor core reads (sf_offset). Rows of the last tile past
// n_q get scale 1.0 (their codes are zero: the TMA fills rows past the end).
// Four lanes per 32-value block, 8 values each (16-byte loads); the block
// maximum takes two shuffles, after which every value follows the rule
// kv_pack applies to an MXFP8 K window in the exact steps of
// mxfp8_round_warp, two values per E4M3 conversion.
__global__ void __launch_bounds__(256) q_mxfp8_kernel(const __nv_bfloat16 *__restrict__ q,
                                                     int n_q, int q_tiles, long n_blocks,
                                                     uint8_t *__restrict__ codes,
                                                     uint8_t *__restrict__ sf,
                                                     const KernelCtl ctl) {
  wait_prior_grid();
  allow_next_grid();
  const long tid = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long blk = tid >> 2;                   // (hq, padded row, 32-feature block)
  const bool live = blk < n_blocks;
  const int kb = static_cast<int>(blk & 3);
  const long prow = blk >> 2;                  // hq * q_tiles * 128 + padded row
  const int r = static_cast<int>(prow % (static_cast<long>(q_tiles) * kBM));
  const long hq = prow / (static_cast<long>(q_tiles) * kBM);
  const bool real = live && r < n_q;
  const long src = (hq * n_q + r) * kDim + 32 * kb + 8 * (tid & 3);
  const uint4 u = real && in_bounds(ctl, q + src, 16) ? *reinterpret_cast<const uint4 *>(q + src)
                                                     : make_uint4(0, 0, 0, 0);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  float x[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    x[2 * j] = __uint_as_float(w[j] << 16);
    x[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
  }
  float amax = 0.0f;
#pragma unroll
  for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  if (!live) return;
  const int ex = mxfp8_block_exp(amax);
  if ((tid & 3) == 0) {
    const int t = r / kBM;
    uint8_t *dst = sf + (hq * q_tiles + t) * 512 + sf_offset(r % kBM, kb);
    if (in_bounds(ctl, dst, 1)) *dst = static_cast<uint8_t>(real ? ex + 127 : 127);
  }
  if (!real) return;
  const float down = pow2_of(-ex);
  uint32_t o[2] = {0u, 0u};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __nv_fp8x2_storage_t c = __nv_cvt_float2_to_fp8x2(
        make_float2(__fmul_rn(x[2 * j], down), __fmul_rn(x[2 * j + 1], down)), __NV_SATFINITE,
        __NV_E4M3);
    o[j >> 1] |= static_cast<uint32_t>(c) << (16 * (j & 1));
  }
  if (in_bounds(ctl, codes + src, 8)) *reinterpret_cast<uint2 *>(codes + src) = make_uint2(o[0], o[1]);
}

// ------------------------------------------------------------------ int4 history
// A cache whose older tokens are grouped int4 (residual-window page, section
// 固定預算) and whose last R tokens are a bf16 window -- the layout of the
// Catnip study's cache with the sink and recent regions compressed -- has the
// key tiles that hold int4 tokens expanded to contiguous bf16 K and V rows
// [unit][N][128] in workspace (N here: the history rounded up to whole
// 128-key tiles, the first window rows of the last one included): x = code * s,
// exact in fp32, rounded once to bf16 (the precision the tensor cores take
// anyway). The chunk kernel reads those tiles from workspace and the later
// ones from the window in place.
struct HistArgs {
  const uint8_t *k_codes;   // [unit][Gk][32][64]
  const float *k_scales;    // [unit][Gk][128]
  const uint8_t *v_codes;   // [unit][cut][64]
  const float *v_scales;    // [unit][cut][4]
  const uint16_t *k_window, *v_window;  // [unit][R][128] bf16
  uint16_t *k_out, *v_out;  // [unit][N][128] bf16
  int N, R, cut, Gk;        // N: rows expanded
  int Gs, Vs, Ws;  // per-unit strides: K groups, V rows, window rows
  KernelCtl ctl;
};

__device__ __forceinline__ float nib(uint32_t w, int e) {
  return static_cast<float>(static_cast<int>((w >> (4 * e)) & 0xFu) - 8);
}

// One thread per (token, 8 features) of unit blockIdx.y: 16-byte stores.
__global__ void __launch_bounds__(256) history_to_bf16_kernel(const HistArgs a) {
  wait_prior_grid();
  allow_next_grid();
  const int i = blockIdx.x * 256 + threadIdx.x;
  if (i >= a.N * 16) return;
  const long u = blockIdx.y;
  const int t = i >> 4, q = i & 15;  // token, feature slice 8q..8q+7
  uint4 ko = make_uint4(0u, 0u, 0u, 0u), vo = ko;
  if (t < a.cut) {
    const long grp = u * a.Gs + (t >> 5);
    const long row = u * a.Vs + t;
    if (!in_bounds(a.ctl, a.k_codes + (grp * 32 + (t & 31)) * 64 + 4 * q, 4) ||
        !in_bounds(a.ctl, a.k_scales + grp * 128 + 8 * q, 32) ||
        !in_bounds(a.ctl, a.v_codes + row * 64 + 4 * q, 4) ||
        !in_bounds(a.ctl, a.v_scales + row * 4 + (q >> 2), 4))
      return;
    // byte j of the slice holds features 8q + 2j (low nibble) and 8q + 2j + 1
    const uint32_t kc =
        *reinterpret_cast<const uint32_t *>(a.k_codes + (grp * 32 + (t & 31)) * 64 + 4 * q);
    const float4 s0 = *reinterpret_cast<const float4 *>(a.k_scales + grp * 128 + 8 * q);
    const float4 s1 = *reinterpret_cast<const float4 *>(a.k_scales + grp * 128 + 8 * q + 4);
    ko = make_uint4(pack_bf16x2(nib(kc, 0) * s0.x, nib(kc, 1) * s0.y),
                    pack_bf16x2(nib(kc, 2) * s0.z, nib(kc, 3) * s0.w),
                    pack_bf16x2(nib(kc, 4) * s1.x, nib(kc, 5) * s1.y),
                    pack_bf16x2(nib(kc, 6) * s1.z, nib(kc, 7) * s1.w));
    const uint32_t vc = *reinterpret_cast<const uint32_t *>(a.v_codes + row * 64 + 4 * q);
    const float vs = a.v_scales[row * 4 + (q >> 2)];
    vo = make_uint4(pack_bf16x2(nib(vc, 0) * vs, nib(vc, 1) * vs),
                    pack_bf16x2(nib(vc, 2) * vs, nib(vc, 3) * vs),
                    pack_bf16x2(nib(vc, 4) * vs, nib(vc, 5) * vs),
                    pack_bf16x2(nib(vc, 6) * vs, nib(vc, 7) * vs));
  } else {
    const long w = (u * a.Ws + (t - a.cut)) * 128 + 8 * q;
    if (in_bounds(a.ctl, a.k_window + w, 16)) ko = *reinterpret_cast<const uint4 *>(a.k_window + w);
    if (in_bounds(a.ctl, a.v_window + w, 16)) vo = *reinterpret_cast<const uint4 *>(a.v_window + w);
  }
  const long o = (u * a.N + t) * 128 + 8 * q;
  if (in_bounds(a.ctl, a.k_out + o, 16)) *reinterpret_cast<uint4 *>(a.k_out + o) = ko;
  if (in_bounds(a.ctl, a.v_out + o, 16)) *reinterpret_cast<uint4 *>(a.v_out + o) = vo;
}

// ------------------------------------------------------------------ block-shared candidate lists
// Candidate prefill with one list per block of query rows (MiniCPM study,
// section 9: its prefill kernel re-gathered a head's candidate rows for every
// query block and lost to dense attention; the fix it names is a
// block-shared candidate layout with the rows tiled through on-chip memory).
// Every list's K and V rows are gathered once, dequantized to bf16, into
// workspace [list][C][128]; the tensor-core kernel then runs each 128-row
// query tile against its list as if it were a cache of C tokens.
struct ListArgs {
  const uint8_t *k_codes;
  const float *k_scales;
  const uint8_t *v_codes;
  const float *v_scales;
  const void *k_window, *v_window;
  int kwin, vwin;
  const int32_t *idx;  // [lists][C], or nullptr: the kept ranges below, one list per unit
  uint16_t *k_out, *v_out;  // [lists][C][128] bf16
  int N, cut, Gs, Vs, Ws, Hkv, Hq, group, lists_per_head, C;
  int n_ranges;
  int range_lo[16], range_hi[16];  // kept key ranges, in order
  KernelCtl ctl;
};

// Position of the c-th kept key when the list is a set of key ranges.
__device__ __forceinline__ int kept_position(const ListArgs &a, int c) {
  for (int r = 0; r < a.n_ranges; ++r) {
    const int len = a.range_hi[r] - a.range_lo[r];
    if (c < len) return a.range_lo[r] + c;
    c -= len;
  }
  return -1;
}

__device__ __forceinline__ float win_value(const void *w, int dt, long i) {
  return dt == KVQ_F32 ? static_cast<const float *>(w)[i]
                       : __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t *>(w)[i]) << 16);
}

// One thread per (listed key, 8 features) of list blockIdx.y.
__global__ void __launch_bounds__(256) gather_lists_bf16_kernel(const ListArgs a) {
  wait_prior_grid();
  allow_next_grid();
  const int i = blockIdx.x * 256 + threadIdx.x;
  if (i >= a.C * 16) return;
  const long l = blockIdx.y;
  const int c = i >> 4, q8 = i & 15;
  const long bh = l / a.lists_per_head;  // b * Hq + h
  const long u = a.idx ? (bh / a.Hq) * a.Hkv + (bh % a.Hq) / a.group : l;
  const int t = a.idx ? (in_bounds(a.ctl, a.idx + l * a.C + c, 4) ? a.idx[l * a.C + c] : -1)
                     : kept_position(a, c);
  float kx[8], vx[8];
  const long grp = u * a.Gs + (t >> 5);
  const long wrow = (u * a.Ws + (t - a.cut)) * 128 + 8 * q8;
  const size_t kwb = a.kwin == KVQ_F32 ? 4 : 2, vwb = a.vwin == KVQ_F32 ? 4 : 2;
  const bool in_ok =
      t >= 0 && t < a.N &&
      (t < a.cut
           ? in_bounds(a.ctl, a.k_codes + (grp * 32 + (t & 31)) * 64 + 4 * q8, 4) &&
                 in_bounds(a.ctl, a.v_codes + (u * a.Vs + t) * 64 + 4 * q8, 4) &&
                 in_bounds(a.ctl, a.v_scales + (u * a.Vs + t) * 4 + (q8 >> 2), 4) &&
                 in_bounds(a.ctl, a.k_scales + grp * 128 + 8 * q8, 32)
           : in_bounds(a.ctl, static_cast<const uint8_t *>(a.k_window) + wrow * kwb, 8 * kwb) &&
                 in_bounds(a.ctl, static_cast<const uint8_t *>(a.v_window) + wrow * vwb, 8 * vwb));
  if (t < 0 || t >= a.N || !in_ok) {
    if (q8 == 0 && (t < 0 || t >= a.N)) flag_error(a.ctl, KVQ_DEV_INDEX);
#pragma unroll
    for (int e = 0; e < 8; ++e) kx[e] = vx[e] = 0.0f;
  } else if (t < a.cut) {
    const uint32_t kc =
        *reinterpret_cast<const uint32_t *>(a.k_codes + (grp * 32 + (t & 31)) * 64 + 4 * q8);
    const uint32_t vc = *reinterpret_cast<const uint32_t *>(a.v_codes + (u * a.Vs + t) * 64 + 4 * q8);
    const float vs = a.v_scales[(u * a.Vs + t) * 4 + (q8 >> 2)];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      kx[e] = nib(kc, e) * a.k_scales[grp * 128 + 8 * q8 + e];
      vx[e] = nib(vc, e) * vs;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      kx[e] = win_value(a.k_window, a.kwin, wrow + e);
      vx[e] = win_value(a.v_window, a.vwin, wrow + e);
    }
  }
  const long o = (l * a.C + c) * 128 + 8 * q8;
  if (!in_bounds(a.ctl, a.k_out + o, 16) || !in_bounds(a.ctl, a.v_out + o, 16)) return;
  *reinterpret_cast<uint4 *>(a.k_out + o) =
      make_uint4(pack_bf16x2(kx[0], kx[1]), pack_bf16x2(kx[2], kx[3]), pack_bf16x2(kx[4], kx[5]),
                 pack_bf16x2(kx[6], kx[7]));
  *reinterpret_cast<uint4 *>(a.v_out + o) =
      make_uint4(pack_bf16x2(vx[0], vx[1]), pack_bf16x2(vx[2], vx[3]), pack_bf16x2(vx[4], vx[5]),
                 pack_bf16x2(vx[6], vx[7]));
}

// ------------------------------------------------------------------ host side
using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

// [heads][rows][128] bf16 as a 3-D map, box 64 features x 128 rows x 1 head;
// consecutive heads are head_rows rows apart (>= rows).
bool make_map(CUtensorMap *m, const void *ptr, int rows, int heads, long head_rows,
              int box_rows = 128) {
  EncodeTiled enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kDim), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(heads)};
  const cuuint64_t strides[2] = {kDim * 2ull, static_cast<cuuint64_t>(head_rows) * kDim * 2ull};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [heads][rows][128] bytes (E4M3) as a 3-D map, box 128 bytes x box_rows x 1:
// one 128B-swizzled row per token.
bool make_map_e4m3(CUtensorMap *m, const void *ptr, int rows, int heads, long head_rows,
                   int box_rows) {
  EncodeTiled enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kDim), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(heads)};
  const cuuint64_t strides[2] = {kDim * 1ull, static_cast<cuuint64_t>(head_rows) * kDim};
  const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// All-window caches (bf16 K, or MXFP8 K) and int4-history caches whose window,
// if any, is bf16.
bool chunk_supported(const kvq_cache &c, int q_dtype, int Hq, int n_q) {
  const bool all_window = c.recent == c.n_tokens && c.vwin_dtype == KVQ_BF16 &&
                          (c.kwin_dtype == KVQ_BF16 || c.kwin_dtype == KVQ_MXFP8);
  const bool history = c.recent < c.n_tokens &&
                       (c.recent == 0 || (c.kwin_dtype == KVQ_BF16 && c.vwin_dtype == KVQ_BF16));
  return (all_window || history) && c.head_dim == kDim && q_dtype == KVQ_BF16 && n_q >= 64 &&
         Hq % c.kv_heads == 0 && encoder() != nullptr;
}

static bool has_history(const kvq_cache &c) { return c.recent < c.n_tokens; }

// Rows of an int4-history cache expanded to bf16: the key tiles that hold an
// int4 token, i.e. the history rounded up to whole tiles (the first window
// rows of the last such tile included); later tiles are read from the window.
static int expanded_rows(const kvq_cache &c) {
  const int cut = c.n_tokens - c.recent;
  return std::min(c.n_tokens, (cut + kBN - 1) / kBN * kBN);
}

// MXFP8: E4M3 codes of Q [hq][n_q][128] (256-byte aligned size), then the Q
// scale blocks [hq][query tiles][512]. int4 history: bf16 K and V of the
// expanded rows.
static size_t q_codes_bytes(const kvq_cache &c, int Hq, int n_q) {
  return (static_cast<size_t>(c.batch) * Hq * n_q * kDim + 255) & ~size_t(255);
}

size_t chunk_workspace_bytes(const kvq_cache &c, int Hq, int n_q) {
  if (has_history(c)) {
    const size_t kb = static_cast<size_t>(c.batch) * c.kv_heads * expanded_rows(c) * kDim * 2;
    return 2 * ((kb + 255) & ~size_t(255));
  }
  if (c.kwin_dtype != KVQ_MXFP8) return 0;
  const size_t tiles = static_cast<size_t>((n_q + kBM - 1) / kBM);
  return q_codes_bytes(c, Hq, n_q) + static_cast<size_t>(c.batch) * Hq * tiles * 512;
}

int chunk_max_regions() { return kMaxRegions; }

// MXFP8 Q/K: Q rounded to E4M3 + E8M0 in workspace, then the block-scaled
// kernel over the cache's E4M3 K window and bf16 V window in place.
static int launch_chunk_mxfp8(const kvq_cache &c, const void *q, int Hq, int n_q,
                              float scale_log2, void *out, int out_dtype, const int32_t *bounds,
                              int n_regions, float *mass, void *ws, const KernelCtl &ctl,
                              cudaStream_t s) {
  using T = Tile<true>;
  const int q_tiles = (n_q + kBM - 1) / kBM;
  const long hq_rows = static_cast<long>(c.batch) * Hq;
  uint8_t *codes = static_cast<uint8_t *>(ws);
  uint8_t *sf = codes + q_codes_bytes(c, Hq, n_q);
  const long n_blocks = hq_rows * q_tiles * kBM * 4;  // 32-feature blocks, padded rows
  launch_dependent(q_mxfp8_kernel, dim3(static_cast<unsigned>((n_blocks * 4 + 255) / 256)),
                   dim3(256), 0, s, static_cast<const __nv_bfloat16 *>(q), n_q, q_tiles,
                   n_blocks, codes, sf, ctl);
  const int Ws = dims_of(c).Ws;
  CUtensorMap tq, tk, tv;
  if (!make_map_e4m3(&tq, codes, n_q, static_cast<int>(hq_rows), n_q, kBM) ||
      !make_map_e4m3(&tk, c.k_window, c.n_tokens, c.batch * c.kv_heads, Ws, T::BN) ||
      !make_map(&tv, c.v_window, c.n_tokens, c.batch * c.kv_heads, Ws, T::BN))
    return -1;
  ChunkArgs a;
  a.n_q = n_q;
  a.n_kv = c.n_tokens;
  a.q_heads = Hq;
  a.kv_group = Hq / c.kv_heads;
  a.n_tiles = (c.n_tokens + T::BN - 1) / T::BN;
  a.scale_log2 = scale_log2;
  a.out = out;
  a.out_dtype = out_dtype;
  a.mass = mass;
  a.reg = make_regions(bounds, n_regions);
  a.ctl = ctl;
  a.tiles_per_list = 0;
  a.lists_per_head = 0;
  a.hist_tiles = 0x7fffffff;
  a.win_off = 0;
  a.q_sf = sf;
  a.k_e8m0 = c.k_window_e8m0;
  a.k_ws = Ws;
  static_assert(sizeof(ChunkSmem<true>) + 1024 <= 232448, "chunk kernel shared memory");
  const size_t smem = sizeof(ChunkSmem<true>) + 1024;
  opt_in_smem(chunk_mxfp8_kernel, smem);
  dim3 grid(q_tiles, static_cast<unsigned>(hq_rows));
  launch_dependent(chunk_mxfp8_kernel, grid, dim3(384), smem, s, tq, tk, tv, a);
  return 2;
}

int launch_attend_chunk(const kvq_cache &c, const void *q, int Hq, int n_q, float scale_log2,
                        void *out, int out_dtype, const int32_t *bounds, int n_regions,
                        float *mass, void *ws, const KernelCtl &ctl, cudaStream_t s) {
  int launches = 1;
  const void *kptr = c.k_window, *vptr = c.v_window, *qptr = q;
  int hist_rows = 0;  // rows read from the expanded history (0: none)
  if (has_history(c)) {
    const CacheDims d = dims_of(c);
    hist_rows = expanded_rows(c);
    const size_t kb =
        (static_cast<size_t>(d.B) * d.Hkv * hist_rows * kDim * 2 + 255) & ~size_t(255);
    HistArgs h;
    h.k_codes = c.k_codes;
    h.k_scales = c.k_scales;
    h.v_codes = c.v_codes;
    h.v_scales = c.v_scales;
    h.k_window = static_cast<const uint16_t *>(c.k_window);
    h.v_window = static_cast<const uint16_t *>(c.v_window);
    h.k_out = static_cast<uint16_t *>(ws);
    h.v_out = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(ws) + kb);
    h.N = hist_rows;
    h.R = d.R;
    h.cut = d.cut;
    h.Gk = d.Gk;
    h.Gs = d.Gs;
    h.Vs = d.Vs;
    h.Ws = d.Ws;
    h.ctl = ctl;
    const dim3 grid(static_cast<unsigned>((hist_rows * 16 + 255) / 256),
                    static_cast<unsigned>(d.B * d.Hkv));
    launch_dependent(history_to_bf16_kernel, grid, dim3(256), 0, s, h);
    kptr = h.k_out;
    vptr = h.v_out;
    launches += 1;
  } else if (c.kwin_dtype == KVQ_MXFP8) {
    return launch_chunk_mxfp8(c, q, Hq, n_q, scale_log2, out, out_dtype, bounds, n_regions, mass,
                              ws, ctl, s);
  }
  CUtensorMap tq, tk, tv, tkw, tvw;
  // expanded K and V (history, MXFP8) are tight; an all-window cache keeps
  // its window stride
  const int Ws = dims_of(c).Ws;
  const int rows = hist_rows ? hist_rows : c.n_tokens;
  const long k_rows = kptr == c.k_window ? Ws : rows;
  const long v_rows = vptr == c.v_window ? Ws : rows;
  if (!make_map(&tq, qptr, n_q, c.batch * Hq, n_q) ||
      !make_map(&tk, kptr, rows, c.batch * c.kv_heads, k_rows) ||
      !make_map(&tv, vptr, rows, c.batch * c.kv_heads, v_rows))
    return -1;
  // the window of an int4-history cache, read in place after the expanded tiles
  const bool split = hist_rows > 0 && hist_rows < c.n_tokens;
  if (split) {
    if (!make_map(&tkw, c.k_window, c.recent, c.batch * c.kv_heads, Ws) ||
        !make_map(&tvw, c.v_window, c.recent, c.batch * c.kv_heads, Ws))
      return -1;
  } else {
    tkw = tk;
    tvw = tv;
  }
  ChunkArgs a;
  a.n_q = n_q;
  a.n_kv = c.n_tokens;
  a.q_heads = Hq;
  a.kv_group = Hq / c.kv_heads;
  a.n_tiles = (c.n_tokens + kBN - 1) / kBN;
  a.scale_log2 = scale_log2;
  a.out = out;
  a.out_dtype = out_dtype;
  a.mass = mass;
  a.reg = make_regions(bounds, n_regions);
  a.ctl = ctl;
  a.tiles_per_list = 0;
  a.lists_per_head = 0;
  a.hist_tiles = split ? hist_rows / kBN : 0x7fffffff;
  a.win_off = split ? c.n_tokens - c.recent : 0;
  a.q_sf = nullptr;
  a.k_e8m0 = nullptr;
  a.k_ws = 0;
  static_assert(sizeof(ChunkSmem<false>) + 1024 <= 232448, "chunk kernel shared memory");
  const size_t smem = sizeof(ChunkSmem<false>) + 1024;
  opt_in_smem(chunk_bf16_kernel, smem);
  dim3 grid((n_q + kBM - 1) / kBM, c.batch * Hq);
  launch_dependent(chunk_bf16_kernel, grid, dim3(384), smem, s, tq, tk, tv, tkw, tvw, a);
  return launches;
}

// Tensor-core path of kv_attend_candidates_block: D = 128, bf16 q, lists of
// block_q (a multiple of 128) query rows.
bool candidate_lists_supported(const kvq_cache &c, int q_dtype, int block_q) {
  return c.head_dim == kDim && q_dtype == KVQ_BF16 && block_q % kBM == 0 &&
         c.kwin_dtype != KVQ_MXFP8 && encoder() != nullptr;
}

size_t candidate_lists_workspace_bytes(long lists, int C) {
  const size_t kb = static_cast<size_t>(lists) * C * kDim * 2;
  return 2 * ((kb + 255) & ~size_t(255));
}

int launch_candidate_lists(const kvq_cache &c, const void *q, int Hq, int n_q,
                           const int32_t *idx, int C, int block_q, float scale_log2, void *out,
                           int out_dtype, void *ws, const KernelCtl &ctl, cudaStream_t s) {
  const CacheDims d = dims_of(c);
  const int lists_per_head = (n_q + block_q - 1) / block_q;
  const long lists = static_cast<long>(d.B) * Hq * lists_per_head;
  const size_t kb = (static_cast<size_t>(lists) * C * kDim * 2 + 255) & ~size_t(255);
  ListArgs g;
  g.k_codes = c.k_codes;
  g.k_scales = c.k_scales;
  g.v_codes = c.v_codes;
  g.v_scales = c.v_scales;
  g.k_window = c.k_window;
  g.v_window = c.v_window;
  g.kwin = c.kwin_dtype;
  g.vwin = c.vwin_dtype;
  g.idx = idx;
  g.k_out = static_cast<uint16_t *>(ws);
  g.v_out = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(ws) + kb);
  g.N = d.N;
  g.cut = d.cut;
  g.Gs = d.Gs;
  g.Vs = d.Vs;
  g.Ws = d.Ws;
  g.Hkv = d.Hkv;
  g.Hq = Hq;
  g.group = Hq / d.Hkv;
  g.lists_per_head = lists_per_head;
  g.C = C;
  g.ctl = ctl;
  launch_dependent(gather_lists_bf16_kernel,
                   dim3(static_cast<unsigned>((C * 16 + 255) / 256), static_cast<unsigned>(lists)),
                   dim3(256), 0, s, g);
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, q, n_q, d.B * Hq, n_q) ||
      !make_map(&tk, g.k_out, C, static_cast<int>(lists), C) ||
      !make_map(&tv, g.v_out, C, static_cast<int>(lists), C))
    return -1;
  const CUtensorMap tkw = tk, tvw = tv;  // no window read in place
  ChunkArgs a;
  a.n_q = n_q;
  a.n_kv = C;
  a.q_heads = Hq;
  a.kv_group = 1;
  a.n_tiles = (C + kBN - 1) / kBN;
  a.scale_log2 = scale_log2;
  a.out = out;
  a.out_dtype = out_dtype;
  a.mass = nullptr;
  a.reg = make_regions(nullptr, 0);
  a.ctl = ctl;
  a.tiles_per_list = block_q / kBM;
  a.lists_per_head = lists_per_head;
  a.hist_tiles = 0x7fffffff;
  a.win_off = 0;
  a.q_sf = nullptr;
  a.k_e8m0 = nullptr;
  a.k_ws = 0;
  const size_t smem = sizeof(ChunkSmem<false>) + 1024;
  opt_in_smem(chunk_bf16_kernel, smem);
  dim3 grid((n_q + kBM - 1) / kBM, d.B * Hq);
  launch_dependent(chunk_bf16_kernel, grid, dim3(384), smem, s, tq, tk, tv, tkw, tvw, a);
  return 2;
}

// kv_attend_region_drop: every (sequence, KV head)'s keys outside the dropped
// regions gathered once to bf16 (a list of C keys per unit), then the chunk
// kernel over them with the usual GQA mapping.
size_t region_drop_workspace_bytes(const kvq_cache &c, int kept) {
  return candidate_lists_workspace_bytes(static_cast<long>(c.batch) * c.kv_heads, kept);
}

int launch_region_drop(const kvq_cache &c, const void *q, int Hq, int n_q, const int32_t *bounds,
                       int n_regions, uint32_t drop_mask, float scale_log2, void *out,
                       int out_dtype, void *ws, const KernelCtl &ctl, cudaStream_t s) {
  const CacheDims d = dims_of(c);
  const long units = static_cast<long>(d.B) * d.Hkv;
  ListArgs g;
  g.n_ranges = 0;
  int C = 0;
  for (int r = 0; r < n_regions && r < 16; ++r) {
    if (drop_mask & (1u << r)) continue;
    if (g.n_ranges > 0 && g.range_hi[g.n_ranges - 1] == bounds[r]) {
      g.range_hi[g.n_ranges - 1] = bounds[r + 1];  // adjacent kept regions: one range
    } else {
      g.range_lo[g.n_ranges] = bounds[r];
      g.range_hi[g.n_ranges] = bounds[r + 1];
      ++g.n_ranges;
    }
    C += bounds[r + 1] - bounds[r];
  }
  if (C == 0) return -1;
  const size_t kb = (static_cast<size_t>(units) * C * kDim * 2 + 255) & ~size_t(255);
  g.k_codes = c.k_codes;
  g.k_scales = c.k_scales;
  g.v_codes = c.v_codes;
  g.v_scales = c.v_scales;
  g.k_window = c.k_window;
  g.v_window = c.v_window;
  g.kwin = c.kwin_dtype;
  g.vwin = c.vwin_dtype;
  g.idx = nullptr;
  g.k_out = static_cast<uint16_t *>(ws);
  g.v_out = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(ws) + kb);
  g.N = d.N;
  g.cut = d.cut;
  g.Gs = d.Gs;
  g.Vs = d.Vs;
  g.Ws = d.Ws;
  g.Hkv = d.Hkv;
  g.Hq = Hq;
  g.group = Hq / d.Hkv;
  g.lists_per_head = 1;
  g.C = C;
  g.ctl = ctl;
  launch_dependent(gather_lists_bf16_kernel,
                   dim3(static_cast<unsigned>((C * 16 + 255) / 256), static_cast<unsigned>(units)),
                   dim3(256), 0, s, g);
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, q, n_q, d.B * Hq, n_q) ||
      !make_map(&tk, g.k_out, C, static_cast<int>(units), C) ||
      !make_map(&tv, g.v_out, C, static_cast<int>(units), C))
    return -1;
  const CUtensorMap tkw = tk, tvw = tv;  // no window read in place
  ChunkArgs a;
  a.n_q = n_q;
  a.n_kv = C;
  a.q_heads = Hq;
  a.kv_group = Hq / d.Hkv;
  a.n_tiles = (C + kBN - 1) / kBN;
  a.scale_log2 = scale_log2;
  a.out = out;
  a.out_dtype = out_dtype;
  a.mass = nullptr;
  a.reg = make_regions(nullptr, 0);
  a.ctl = ctl;
  a.tiles_per_list = 0;
  a.lists_per_head = 0;
  a.hist_tiles = 0x7fffffff;
  a.win_off = 0;
  a.q_sf = nullptr;
  a.k_e8m0 = nullptr;
  a.k_ws = 0;
  const size_t smem = sizeof(ChunkSmem<false>) + 1024;
  opt_in_smem(chunk_bf16_kernel, smem);
  dim3 grid((n_q + kBM - 1) / kBM, d.B * Hq);
  launch_dependent(chunk_bf16_kernel, grid, dim3(384), smem, s, tq, tk, tv, tkw, tvw, a);
  return 2;
}

}  // namespace kvq
