// Device helpers shared by the kvq kernels: error reporting, bounded mbarrier
// waits, 1-D bulk copies (TMA) and small conversions. sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <tuple>
#include <vector>

#include "../../include/kvq.h"

namespace kvq {

constexpr int kGroup = 32;

#ifdef KVQ_DEBUG
constexpr int kMaxBufs = 16;  // buffers one call may register for the bounds checks
#endif

// Launch-wide settings every kernel receives by value.
struct KernelCtl {
  int32_t *dev_status;      // may be nullptr
  uint64_t wait_limit_ns;   // bound of every mbarrier wait
  int32_t drop_item;        // test hook: loader skips this work item (-1: none)
#ifdef KVQ_DEBUG
  // The device buffers of the call ([lo, hi) byte ranges): the cache's
  // arrays, q, the outputs, index lists, workspace.
  int32_t n_bufs;
  uintptr_t buf_lo[kMaxBufs], buf_hi[kMaxBufs];
#endif
};

__host__ __device__ __forceinline__ void flag_error(const KernelCtl &ctl, int bit) {
#ifdef __CUDA_ARCH__
  if (ctl.dev_status) atomicOr(ctl.dev_status, bit);
#else
  if (ctl.dev_status) *ctl.dev_status |= bit;  // host: the check's own tests
#endif
}

// Bounds check of a global access. In a build with KVQ_DEBUG defined: true
// when the bytes [p, p + bytes) lie inside one buffer of the call; otherwise
// KVQ_DEV_BOUNDS is set and the caller leaves the access out (a load reads
// zeros, a store is dropped, a bulk copy is not issued and not expected), so
// a wrong index is reported instead of touching memory. Every kernel checks
// each contiguous range it derives from its indices (a row, a chunk, a copy)
// before the accesses inside it. Other builds: true, and the check
// compiles away.
__host__ __device__ __forceinline__ bool in_bounds(const KernelCtl &ctl, const void *p,
                                                   size_t bytes) {
#ifdef KVQ_DEBUG
  const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = a + bytes;
  for (int i = 0; i < ctl.n_bufs; ++i)
    if (a >= ctl.buf_lo[i] && b <= ctl.buf_hi[i] && b >= a) return true;
  flag_error(ctl, KVQ_DEV_BOUNDS);
  return false;
#else
  (void)ctl;
  (void)p;
  (void)bytes;
  return true;
#endif
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ dependent launches
// Every kvq kernel is started with launch_dependent(): its blocks may be
// placed on the SMs while the kernel before it on the stream drains, which
// hides the launch gap between back-to-back kernels. Such a kernel calls
// wait_prior_grid() in every thread before its first access to global memory;
// the wait returns once the previous kernel has completed and its writes are
// visible (at once for an ordinary launch). allow_next_grid() lets the next
// dependent launch start placing its blocks; it changes no memory ordering.
__device__ __forceinline__ void wait_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_next_grid() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block,
                                    size_t smem, cudaStream_t s, Args &&...args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Raise the transaction count of the current phase without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but a thread whose phase has not completed is suspended
// until it completes or about hint_ns nanoseconds pass, instead of returning
// at once: a waiting warp takes no issue slots from the warps doing the work.
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity,
                                                   uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete, for at most about
// limit_ns nanoseconds of global time (the last suspension may overshoot by
// up to 100 us). Returns false when the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (mbar_try_wait_hint(bar, parity, 100000u)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// 2^x on the SFU (ex2.approx: about 2 ulp, subnormal results flushed to 0,
// 2^-inf = 0). Every caller rounds the result to 16 bits afterwards.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------ bulk copy
// 1-D global -> shared copy completing on an mbarrier (tx bytes). Both
// addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// ------------------------------------------------------------------ conversions
__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

template <typename T>
__device__ __forceinline__ float load_f32(const T *p);
template <>
__device__ __forceinline__ float load_f32<float>(const float *p) {
  return *p;
}
template <>
__device__ __forceinline__ float load_f32<__nv_bfloat16>(const __nv_bfloat16 *p) {
  return __bfloat162float(*p);
}

template <typename T>
__device__ __forceinline__ void store_from_f32(T *p, float x);
template <>
__device__ __forceinline__ void store_from_f32<float>(float *p, float x) {
  *p = x;
}
template <>
__device__ __forceinline__ void store_from_f32<__nv_bfloat16>(__nv_bfloat16 *p, float x) {
  *p = __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// ------------------------------------------------------------------ warp MMA (mma.sync)
// D += A B, m16n8k16, bf16 operands, fp32 accumulators. With g = lane / 4 and
// t = lane % 4: a0 = A(g, 2t..2t+1), a1 = A(g+8, 2t..), a2 = A(g, 2t+8..),
// a3 = A(g+8, 2t+8..); b0 = B(2t..2t+1, g), b1 = B(2t+8..2t+9, g);
// c0, c1 = C(g, 2t..2t+1), c2, c3 = C(g+8, 2t..2t+1).
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 matrix of 16-bit pairs held one row pair per lane.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&b);
}

// Four 8x8 16-bit matrices from shared memory: lane i gives the address of
// row i % 8 of matrix i / 8; register j receives matrix j (transposed with
// ldsm_x4_t).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Value of an E4M3 byte times 2^(e8m0 - 127), computed exactly in fp32
// (E4M3 has 3 mantissa bits; the power of two is applied with ldexpf).
__device__ __forceinline__ float mxfp8_value(uint8_t code, uint8_t e8m0) {
  const int e = (code >> 3) & 0xF;
  const int m = code & 0x7;
  float mag = (e == 0) ? ldexpf(static_cast<float>(m), -9)
                       : ldexpf(static_cast<float>(8 + m), e - 10);
  if ((code & 0x7F) == 0x7F) mag = __int_as_float(0x7fc00000);
  return ldexpf((code & 0x80) ? -mag : mag, static_cast<int>(e8m0) - 127);
}

// MXFP8 (E4M3 elements, one E8M0 scale 2^e per 32-value block, the OCP MX
// rule): e = clamp(floor(log2 amax) - 8, -127, 127), -127 for a zero block.
// The exponent is read from the float bits when amax is normal (frexpf for a
// subnormal or non-finite maximum), so every step below is exact: x * 2^-e
// (the power of two is normal since e <= 119; a product below the normal
// range, rounded as ldexpf would, has code 0), the saturating conversion to
// E4M3, the exact E4M3 -> f16 conversion back, and the product with 2^e (an
// E4M3 value has at most 4 significant bits and the result stays above 2^-136).
__device__ __forceinline__ int mxfp8_block_exp(float amax) {
  const int be = static_cast<int>(__float_as_uint(amax) >> 23);  // biased exponent, amax >= 0
  if (be >= 1 && be <= 254) return max(-127, be - 135);       // frexp exponent be - 126
  if (!(amax > 0.0f)) return -127;
  int f;
  frexpf(amax, &f);
  return max(-127, min(127, f - 1 - 8));
}
__device__ __forceinline__ float pow2_of(int e) {  // 2^e for e in [-127, 127]
  return e > -127 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23)
                  : __uint_as_float(0x00400000u);
}
__device__ __forceinline__ uint8_t mxfp8_code(float x, float down) {  // down = 2^-e
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(__fmul_rn(x, down), __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float e4m3_value(uint8_t c) {
  uint32_t f16x2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f16x2) : "h"(static_cast<unsigned short>(c)));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(f16x2 & 0xffffu)));
}

// Round x to MXFP8 inside a warp (lane = position in the 32-block) and return
// the dequantized value: the same rule kv_pack applies to an MXFP8 K window.
__device__ __forceinline__ float mxfp8_round_warp(float x) {
  const int e = mxfp8_block_exp(warp_max(fabsf(x)));
  return __fmul_rn(e4m3_value(mxfp8_code(x, pow2_of(-e))), pow2_of(e));
}

// Let `kernel` take `bytes` of dynamic shared memory on the current device.
// The attribute is set once per (kernel, device) and size, so a call that
// launches the kernel again costs a lookup, not a driver call.
template <typename Kernel>
inline cudaError_t opt_in_smem(Kernel *kernel, size_t bytes) {
  static std::mutex mu;
  static std::vector<std::tuple<const void *, int, size_t>> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  const void *fn = reinterpret_cast<const void *>(kernel);
  std::lock_guard<std::mutex> lock(mu);
  for (const auto &d : done)
    if (std::get<0>(d) == fn && std::get<1>(d) == dev && std::get<2>(d) >= bytes) return cudaSuccess;
  const cudaError_t r = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(bytes));
  if (r == cudaSuccess) done.emplace_back(fn, dev, bytes);
  return r;
}

}  // namespace kvq
