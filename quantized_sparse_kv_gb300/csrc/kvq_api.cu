// C ABI entry points: argument checks, kernel choice, launch accounting.
// Declarations and the meaning of every argument are in include/kvq.h.
#include <math.h>

#include "kvq_internal.h"

namespace {

thread_local int32_t g_last_launches = 0;
thread_local const char *g_last_path = "";
thread_local uint64_t g_wait_limit_ns = 0;
thread_local int32_t g_drop_item = -1;

constexpr uint64_t kDefaultWaitNs = 1000000000ull;  // one second
constexpr double kLog2e = 1.4426950408889634;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  if (dev < 64) cache[dev] = n;
  return n;
}

kvq::KernelCtl make_ctl(int32_t *dev_status) {
  kvq::KernelCtl c;
  c.dev_status = dev_status;
  c.wait_limit_ns = g_wait_limit_ns ? g_wait_limit_ns : kDefaultWaitNs;
  c.drop_item = g_drop_item;
#ifdef KVQ_DEBUG
  c.n_bufs = 0;
#endif
  return c;
}

// The bounds-check table of a KVQ_DEBUG build: each device buffer of the
// call, as [p, p + bytes). Other builds keep no table and these do nothing.
void ctl_add(kvq::KernelCtl &c, const void *p, size_t bytes) {
#ifdef KVQ_DEBUG
  if (!p || bytes == 0 || c.n_bufs >= kvq::kMaxBufs) return;
  c.buf_lo[c.n_bufs] = reinterpret_cast<uintptr_t>(p);
  c.buf_hi[c.n_bufs] = reinterpret_cast<uintptr_t>(p) + bytes;
  ++c.n_bufs;
#else
  (void)c;
  (void)p;
  (void)bytes;
#endif
}

// Bytes of rows x d elements of type dt.
size_t rows_bytes(long rows, int d, int32_t dt) {
  return static_cast<size_t>(rows) * static_cast<size_t>(d) *
         (dt == KVQ_F32 ? 4u : dt == KVQ_BF16 ? 2u : 1u);
}

bool shape_ok(int32_t batch, int32_t kv_heads, int32_t n_tokens, int32_t head_dim, int32_t recent,
              int32_t kwin, int32_t vwin) {
  if (batch < 1 || kv_heads < 1 || n_tokens < 1) return false;
  if (head_dim < 32 || head_dim > 256 || head_dim % 32) return false;
  if (recent < 0 || recent > n_tokens) return false;
  if (kwin != KVQ_F32 && kwin != KVQ_BF16 && kwin != KVQ_MXFP8) return false;
  if (vwin != KVQ_F32 && vwin != KVQ_BF16) return false;
  return true;
}

size_t elem_bytes(int32_t dt) { return dt == KVQ_F32 ? 4 : dt == KVQ_BF16 ? 2 : 1; }

// Validates the cache descriptor's shape and the pointers its arrays need.
kvq_status check_cache(const kvq_cache *c) {
  if (!c) return KVQ_ERR_ARG;
  if (!shape_ok(c->batch, c->kv_heads, c->n_tokens, c->head_dim, c->recent, c->kwin_dtype,
                c->vwin_dtype))
    return KVQ_ERR_ARG;
  const int cut = c->n_tokens - c->recent;
  if (c->cap_groups < 0 || c->cap_window < 0) return KVQ_ERR_ARG;
  if (c->cap_groups > 0 && (c->cap_groups < (cut + 31) / 32 || c->cap_window < c->recent))
    return KVQ_ERR_ARG;
  if (c->cap_groups == 0 && c->cap_window != 0) return KVQ_ERR_ARG;
  if (cut > 0) {
    if (!c->k_codes || !c->k_scales || !c->v_codes || !c->v_scales) return KVQ_ERR_ARG;
    if (!aligned16(c->k_codes) || !aligned16(c->k_scales) || !aligned16(c->v_codes) ||
        !aligned16(c->v_scales))
      return KVQ_ERR_ALIGN;
  }
  if (c->recent > 0) {
    if (!c->k_window || !c->v_window) return KVQ_ERR_ARG;
    if (c->kwin_dtype == KVQ_MXFP8 && !c->k_window_e8m0) return KVQ_ERR_ARG;
    if (!aligned16(c->k_window) || !aligned16(c->v_window)) return KVQ_ERR_ALIGN;
    if (c->kwin_dtype == KVQ_MXFP8 && !aligned16(c->k_window_e8m0)) return KVQ_ERR_ALIGN;
  }
  return KVQ_OK;
}

kvq_status finish(int launches, const char *path) {
  if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  g_last_launches = launches;
  g_last_path = path;
  return KVQ_OK;
}

// The calls that fill a cache (kv_pack, kv_append) come before any decode,
// so they reserve the static decode scratch of the current device (loading
// its module) before a runtime hands the rest of HBM to its own pool. A
// failure here is not the caller's: it is cleared and kv_attend_decode_static
// retries, returning KVQ_ERR_CUDA if the array still cannot be had.
void reserve_static_scratch() {
  void *p = nullptr;
  (void)kvq::decode_static_scratch(&p);
}

float resolve_scale(float sm_scale, int head_dim) {
  return sm_scale > 0.0f ? sm_scale
                         : static_cast<float>(1.0 / sqrt(static_cast<double>(head_dim)));
}

// The cache's arrays, at the sizes its shape (and reserved room) gives.
void ctl_add_cache(kvq::KernelCtl &c, const kvq_cache &k) {
#ifdef KVQ_DEBUG
  size_t sz[8];
  const kvq_status st =
      k.cap_groups > 0
          ? kvq_cache_sizes_reserved(k.batch, k.kv_heads, k.head_dim, k.kwin_dtype, k.vwin_dtype,
                                     k.cap_groups, k.cap_window, sz)
          : kvq_cache_sizes(k.batch, k.kv_heads, k.n_tokens, k.head_dim, k.recent, k.kwin_dtype,
                            k.vwin_dtype, sz);
  if (st != KVQ_OK) return;
  ctl_add(c, k.k_codes, sz[0]);
  ctl_add(c, k.k_scales, sz[1]);
  ctl_add(c, k.v_codes, sz[2]);
  ctl_add(c, k.v_scales, sz[3]);
  ctl_add(c, k.k_window, sz[4]);
  ctl_add(c, k.v_window, sz[5]);
  ctl_add(c, k.k_window_e8m0, sz[6]);
#else
  (void)c;
  (void)k;
#endif
}

}  // namespace

extern "C" {

kvq_status kvq_cache_sizes(int32_t batch, int32_t kv_heads, int32_t n_tokens, int32_t head_dim,
                           int32_t recent, int32_t kwin_dtype, int32_t vwin_dtype,
                           size_t sizes[8]) {
  if (!sizes || !shape_ok(batch, kv_heads, n_tokens, head_dim, recent, kwin_dtype, vwin_dtype))
    return KVQ_ERR_ARG;
  const size_t units = static_cast<size_t>(batch) * kv_heads;
  const size_t cut = static_cast<size_t>(n_tokens - recent);
  const size_t gk = (cut + 31) / 32;
  const size_t d = static_cast<size_t>(head_dim);
  sizes[0] = units * gk * 32 * d / 2;                 // k_codes
  sizes[1] = units * gk * d * sizeof(float);          // k_scales
  sizes[2] = units * cut * d / 2;                     // v_codes
  sizes[3] = units * cut * (d / 32) * sizeof(float);  // v_scales
  sizes[4] = units * recent * d * elem_bytes(kwin_dtype);
  sizes[5] = units * recent * d * elem_bytes(vwin_dtype);
  sizes[6] = kwin_dtype == KVQ_MXFP8 ? units * recent * (d / 32) : 0;
  sizes[7] = 16;                                      // {N, D, R, 32}
  return KVQ_OK;
}

kvq_status kvq_cache_sizes_reserved(int32_t batch, int32_t kv_heads, int32_t head_dim,
                                    int32_t kwin_dtype, int32_t vwin_dtype, int32_t cap_groups,
                                    int32_t cap_window, size_t sizes[8]) {
  if (!sizes || cap_groups < 1 || cap_window < 0 ||
      !shape_ok(batch, kv_heads, 1, head_dim, 0, kwin_dtype, vwin_dtype))
    return KVQ_ERR_ARG;
  const size_t units = static_cast<size_t>(batch) * kv_heads;
  const size_t gs = static_cast<size_t>(cap_groups), ws = static_cast<size_t>(cap_window);
  const size_t d = static_cast<size_t>(head_dim);
  sizes[0] = units * gs * 32 * d / 2;
  sizes[1] = units * gs * d * sizeof(float);
  sizes[2] = units * gs * 32 * d / 2;
  sizes[3] = units * gs * 32 * (d / 32) * sizeof(float);
  sizes[4] = units * ws * d * elem_bytes(kwin_dtype);
  sizes[5] = units * ws * d * elem_bytes(vwin_dtype);
  sizes[6] = kwin_dtype == KVQ_MXFP8 ? units * ws * (d / 32) : 0;
  sizes[7] = 16;
  return KVQ_OK;
}

size_t kvq_cache_bytes(int32_t batch, int32_t kv_heads, int32_t n_tokens, int32_t head_dim,
                       int32_t recent, int32_t kwin_dtype, int32_t vwin_dtype) {
  size_t s[8];
  if (kvq_cache_sizes(batch, kv_heads, n_tokens, head_dim, recent, kwin_dtype, vwin_dtype, s) !=
      KVQ_OK)
    return 0;
  size_t total = 0;
  for (int i = 0; i < 8; ++i) total += s[i];
  return total;
}

kvq_status kv_pack(const void *k, const void *v, int32_t in_dtype, kvq_cache *cache,
                   int32_t *dev_status, kvq_stream_t stream) {
  const kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (in_dtype != KVQ_F32 && in_dtype != KVQ_BF16) return KVQ_ERR_ARG;
  if (!k || !v) return KVQ_ERR_ARG;
  if (!aligned16(k) || !aligned16(v) || (dev_status && !aligned16(dev_status)))
    return KVQ_ERR_ALIGN;
  cache->header[0] = static_cast<uint32_t>(cache->n_tokens);
  cache->header[1] = static_cast<uint32_t>(cache->head_dim);
  cache->header[2] = static_cast<uint32_t>(cache->recent);
  cache->header[3] = 32u;
  reserve_static_scratch();
  kvq::KernelCtl ctl = make_ctl(dev_status);
  ctl_add_cache(ctl, *cache);
  const long units = static_cast<long>(cache->batch) * cache->kv_heads;
  ctl_add(ctl, k, rows_bytes(units * cache->n_tokens, cache->head_dim, in_dtype));
  ctl_add(ctl, v, rows_bytes(units * cache->n_tokens, cache->head_dim, in_dtype));
  const int n = kvq::launch_pack(k, v, in_dtype, *cache, ctl, sm_count(),
                                 reinterpret_cast<cudaStream_t>(stream));
  return finish(n, "pack");
}

kvq_status kv_append(kvq_cache *cache, const void *k_new, const void *v_new, int32_t in_dtype,
                     int32_t n_new, int32_t window, int32_t *dev_status, kvq_stream_t stream) {
  const kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (in_dtype != KVQ_F32 && in_dtype != KVQ_BF16) return KVQ_ERR_ARG;
  if (n_new < 1 || window < 0 || !k_new || !v_new) return KVQ_ERR_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || (dev_status && !aligned16(dev_status)))
    return KVQ_ERR_ALIGN;
  if (cache->cap_groups <= 0) return KVQ_ERR_UNSUPPORTED;
  if ((cache->kwin_dtype != KVQ_F32 && cache->kwin_dtype != KVQ_BF16) ||
      (cache->vwin_dtype != KVQ_F32 && cache->vwin_dtype != KVQ_BF16))
    return KVQ_ERR_UNSUPPORTED;
  const int cut = cache->n_tokens - cache->recent;
  if (cut % 32) return KVQ_ERR_UNSUPPORTED;  // a padded last K group cannot grow
  if (n_new > 0x7fffffff - cache->n_tokens) return KVQ_ERR_ARG;
  const int n2 = cache->n_tokens + n_new;
  int cut2 = n2 > window ? 32 * ((n2 - window) / 32) : 0;
  if (cut2 < cut) cut2 = cut;
  const int r2 = n2 - cut2, m = (cut2 - cut) / 32;
  if (cut2 / 32 > cache->cap_groups || r2 > cache->cap_window) return KVQ_ERR_WORKSPACE;
  if (m > 0 && static_cast<long>(cache->batch) * cache->kv_heads > 65535)
    return KVQ_ERR_UNSUPPORTED;
  reserve_static_scratch();
  kvq::KernelCtl ctl = make_ctl(dev_status);
  ctl_add_cache(ctl, *cache);
  const long units = static_cast<long>(cache->batch) * cache->kv_heads;
  ctl_add(ctl, k_new, rows_bytes(units * n_new, cache->head_dim, in_dtype));
  ctl_add(ctl, v_new, rows_bytes(units * n_new, cache->head_dim, in_dtype));
  const int n = kvq::launch_append(*cache, k_new, v_new, in_dtype, n_new, m, r2, ctl,
                                   reinterpret_cast<cudaStream_t>(stream));
  const kvq_status done = finish(n, "append");
  if (done != KVQ_OK) return done;
  cache->n_tokens = n2;
  cache->recent = r2;
  cache->header[0] = static_cast<uint32_t>(n2);
  cache->header[1] = static_cast<uint32_t>(cache->head_dim);
  cache->header[2] = static_cast<uint32_t>(r2);
  cache->header[3] = 32u;
  return KVQ_OK;
}

kvq_status kv_attend(const kvq_cache *cache, const void *q, int32_t q_dtype, int32_t q_heads,
                     int32_t n_q, float sm_scale, void *out, int32_t out_dtype,
                     const int32_t *region_bounds, int32_t n_regions, float *region_mass,
                     void *workspace, size_t *ws_bytes, int32_t *dev_status,
                     kvq_stream_t stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (!ws_bytes) return KVQ_ERR_ARG;
  if (q_heads < 1 || q_heads % cache->kv_heads || n_q < 1) return KVQ_ERR_ARG;
  if ((q_dtype != KVQ_F32 && q_dtype != KVQ_BF16) ||
      (out_dtype != KVQ_F32 && out_dtype != KVQ_BF16))
    return KVQ_ERR_ARG;
  if (region_bounds) {
    if (n_regions < 1 || n_regions > 16 || !region_mass) return KVQ_ERR_ARG;
    if (region_bounds[0] != 0 || region_bounds[n_regions] != cache->n_tokens) return KVQ_ERR_ARG;
    for (int i = 0; i < n_regions; ++i)
      if (region_bounds[i + 1] <= region_bounds[i]) return KVQ_ERR_ARG;
    if (!aligned16(region_mass)) return KVQ_ERR_ALIGN;
  }
  const bool regions = region_bounds != nullptr;
  const float scale = resolve_scale(sm_scale, cache->head_dim);
  const int sms = sm_count();

  enum { GENERIC, DECODE, CHUNK } path = GENERIC;
  // the chunk kernel's grid is (query tiles, batch * q_heads)
  if (kvq::chunk_supported(*cache, q_dtype, q_heads, n_q) &&
      static_cast<long>(cache->batch) * q_heads <= 65535 &&
      (!regions || n_regions <= kvq::chunk_max_regions()))
    path = CHUNK;
  else if (!regions && kvq::decode_supported(*cache, q_dtype, q_heads, n_q))
    path = DECODE;
  // the fp32 kernel's grid is (row blocks, q_heads, batch)
  if (path == GENERIC && (q_heads > 65535 || cache->batch > 65535)) return KVQ_ERR_UNSUPPORTED;
  size_t need = 0;
  if (path == DECODE) need = kvq::decode_workspace_bytes(*cache, q_heads, sms);
  if (path == CHUNK) need = kvq::chunk_workspace_bytes(*cache, q_heads, n_q);
  if (!workspace) {
    *ws_bytes = need;
    return KVQ_OK;
  }
  if (*ws_bytes < need) return KVQ_ERR_WORKSPACE;
  if (!q || !out) return KVQ_ERR_ARG;
  if (!aligned16(q) || !aligned16(out) || !aligned16(workspace) ||
      (dev_status && !aligned16(dev_status)))
    return KVQ_ERR_ALIGN;

  kvq::KernelCtl ctl = make_ctl(dev_status);
  {
    const long rows = static_cast<long>(cache->batch) * q_heads * n_q;
    ctl_add_cache(ctl, *cache);
    ctl_add(ctl, q, rows_bytes(rows, cache->head_dim, q_dtype));
    ctl_add(ctl, out, rows_bytes(rows, cache->head_dim, out_dtype));
    if (regions) ctl_add(ctl, region_mass, rows_bytes(rows, n_regions, KVQ_F32));
    ctl_add(ctl, workspace, *ws_bytes);
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (path == CHUNK) {
    const int n = kvq::launch_attend_chunk(*cache, q, q_heads, n_q,
                                           static_cast<float>(scale * kLog2e), out, out_dtype,
                                           region_bounds, n_regions, region_mass, workspace, ctl, s);
    if (n < 0) return KVQ_ERR_CUDA;
    return finish(n, cache->recent < cache->n_tokens   ? "chunk_int4"
                     : cache->kwin_dtype == KVQ_MXFP8 ? "chunk_mxfp8"
                                                      : "chunk_bf16");
  }
  if (path == DECODE) {
    const int n = kvq::launch_attend_decode(*cache, q, q_dtype,
                                            static_cast<float>(scale * kLog2e), out, out_dtype,
                                            workspace, ctl, sms, s);
    return finish(n, "decode");
  }
  const int n = kvq::launch_attend_generic(*cache, q, q_dtype, q_heads, n_q, scale, out,
                                           out_dtype, region_bounds, n_regions, region_mass, ctl, s);
  return finish(n, "generic");
}

kvq_status kv_attend_stats(const kvq_cache *cache, const void *q, int32_t q_dtype,
                           int32_t q_heads, int32_t n_q, float sm_scale,
                           const float *hadamard_signs, float *stats, void *workspace,
                           size_t *ws_bytes, int32_t *dev_status, kvq_stream_t stream) {
  const kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (!ws_bytes) return KVQ_ERR_ARG;
  if (q_heads < 1 || q_heads % cache->kv_heads || n_q < 1) return KVQ_ERR_ARG;
  if (q_dtype != KVQ_F32 && q_dtype != KVQ_BF16) return KVQ_ERR_ARG;
  const int d = cache->head_dim;
  if ((d & (d - 1)) != 0 || cache->n_tokens > kvq::stats_max_tokens()) return KVQ_ERR_UNSUPPORTED;
  if (static_cast<long>(cache->batch) * q_heads * n_q > 0x7fffffffL) return KVQ_ERR_UNSUPPORTED;
  if (static_cast<long>(cache->batch) * q_heads > 65535) return KVQ_ERR_UNSUPPORTED;  // grid.y
  const size_t need = kvq::stats_workspace_bytes(*cache, q_heads, n_q);
  if (!workspace) {
    *ws_bytes = need;
    return KVQ_OK;
  }
  if (*ws_bytes < need) return KVQ_ERR_WORKSPACE;
  if (!q || !stats) return KVQ_ERR_ARG;
  if (!aligned16(q) || !aligned16(stats) || !aligned16(workspace) ||
      (hadamard_signs && !aligned16(hadamard_signs)) || (dev_status && !aligned16(dev_status)))
    return KVQ_ERR_ALIGN;
  const float scale = resolve_scale(sm_scale, d);
  kvq::KernelCtl ctl = make_ctl(dev_status);
  {
    const long rows = static_cast<long>(cache->batch) * q_heads * n_q;
    ctl_add_cache(ctl, *cache);
    ctl_add(ctl, q, rows_bytes(rows, d, q_dtype));
    ctl_add(ctl, stats, rows_bytes(rows, KVQ_N_STATS, KVQ_F32));
    ctl_add(ctl, hadamard_signs, rows_bytes(1, d, KVQ_F32));
    ctl_add(ctl, workspace, *ws_bytes);
  }
  const int n = kvq::launch_attend_stats(*cache, q, q_dtype, q_heads, n_q, scale, hadamard_signs,
                                         stats, workspace, ctl,
                                         reinterpret_cast<cudaStream_t>(stream));
  if (n < 0) return KVQ_ERR_UNSUPPORTED;
  return finish(n, "stats");
}

kvq_status kv_attend_candidates(const kvq_cache *cache, const void *q, int32_t q_dtype,
                                int32_t q_heads, int32_t n_q, const int32_t *idx,
                                int32_t n_cand, int32_t validate, float sm_scale, void *out,
                                int32_t out_dtype, void *workspace, size_t *ws_bytes,
                                int32_t *dev_status, kvq_stream_t stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (!ws_bytes) return KVQ_ERR_ARG;
  if (q_heads < 1 || q_heads % cache->kv_heads || n_q < 1 || n_cand < 1) return KVQ_ERR_ARG;
  if ((q_dtype != KVQ_F32 && q_dtype != KVQ_BF16) ||
      (out_dtype != KVQ_F32 && out_dtype != KVQ_BF16))
    return KVQ_ERR_ARG;
  if (cache->recent > 0 && cache->kwin_dtype == KVQ_MXFP8) return KVQ_ERR_UNSUPPORTED;
  // the grid is (query rows, q_heads, batch)
  if (n_cand > 65536 || q_heads > 65535 || cache->batch > 65535) return KVQ_ERR_UNSUPPORTED;
  const int sms = sm_count();
  const bool uni = kvq::candidates_union_supported(*cache, q_dtype, q_heads, n_q, n_cand);
  const size_t need = uni ? kvq::candidates_union_workspace_bytes(*cache, n_cand, sms) : 0;
  if (!workspace) {
    *ws_bytes = need;
    return KVQ_OK;
  }
  if (*ws_bytes < need) return KVQ_ERR_WORKSPACE;
  if (!q || !out || !idx) return KVQ_ERR_ARG;
  if (!aligned16(q) || !aligned16(out) || !aligned16(idx) || !aligned16(workspace) ||
      (dev_status && !aligned16(dev_status)))
    return KVQ_ERR_ALIGN;
  const float scale = resolve_scale(sm_scale, cache->head_dim);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  kvq::KernelCtl ctl = make_ctl(dev_status);
  {
    const long rows = static_cast<long>(cache->batch) * q_heads * n_q;
    ctl_add_cache(ctl, *cache);
    ctl_add(ctl, q, rows_bytes(rows, cache->head_dim, q_dtype));
    ctl_add(ctl, out, rows_bytes(rows, cache->head_dim, out_dtype));
    ctl_add(ctl, idx, rows_bytes(rows, n_cand, KVQ_F32));
    ctl_add(ctl, workspace, *ws_bytes);
  }
  if (uni) {
    const int n = kvq::launch_candidates_union(*cache, q, idx, n_cand, validate,
                                               static_cast<float>(scale * kLog2e), out, out_dtype,
                                               workspace, ctl, sms, s);
    return finish(n, "candidates_union");
  }
  const int n = kvq::launch_attend_candidates(*cache, q, q_dtype, q_heads, n_q, idx, n_cand,
                                              validate, static_cast<float>(scale * kLog2e), out,
                                              out_dtype, ctl, s);
  return finish(n, "candidates");
}

kvq_status kv_attend_candidates_topk(const kvq_cache *cache, const void *q, int32_t q_dtype,
                                     int32_t q_heads, int32_t n_q, const int32_t *idx,
                                     int32_t n_cand, int32_t top_k, float sm_scale, void *out,
                                     int32_t out_dtype, int32_t *selected, int32_t *dev_status,
                                     kvq_stream_t stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (q_heads < 1 || q_heads % cache->kv_heads || n_q < 1 || n_cand < 1) return KVQ_ERR_ARG;
  if (top_k < 1 || top_k > n_cand) return KVQ_ERR_ARG;
  if ((q_dtype != KVQ_F32 && q_dtype != KVQ_BF16) ||
      (out_dtype != KVQ_F32 && out_dtype != KVQ_BF16))
    return KVQ_ERR_ARG;
  if (!q || !out || !idx) return KVQ_ERR_ARG;
  if (cache->recent > 0 && cache->kwin_dtype == KVQ_MXFP8) return KVQ_ERR_UNSUPPORTED;
  if (n_cand > kvq::candidates_topk_max() || q_heads > 65535 || cache->batch > 65535)
    return KVQ_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(out) || !aligned16(idx) || (selected && !aligned16(selected)) ||
      (dev_status && !aligned16(dev_status)))
    return KVQ_ERR_ALIGN;
  const float scale = resolve_scale(sm_scale, cache->head_dim);
  kvq::KernelCtl ctl = make_ctl(dev_status);
  {
    const long rows = static_cast<long>(cache->batch) * q_heads * n_q;
    ctl_add_cache(ctl, *cache);
    ctl_add(ctl, q, rows_bytes(rows, cache->head_dim, q_dtype));
    ctl_add(ctl, out, rows_bytes(rows, cache->head_dim, out_dtype));
    ctl_add(ctl, idx, rows_bytes(rows, n_cand, KVQ_F32));
    ctl_add(ctl, selected, rows_bytes(rows, top_k, KVQ_F32));
  }
  const int n = kvq::launch_attend_candidates(
      *cache, q, q_dtype, q_heads, n_q, idx, n_cand, 0, static_cast<float>(scale * kLog2e), out,
      out_dtype, ctl, reinterpret_cast<cudaStream_t>(stream), top_k, selected);
  if (n < 0) return KVQ_ERR_UNSUPPORTED;
  return finish(n, "candidates_topk");
}

kvq_status kv_attend_candidates_block(const kvq_cache *cache, const void *q, int32_t q_dtype,
                                      int32_t q_heads, int32_t n_q, const int32_t *idx,
                                      int32_t n_cand, int32_t block_q, float sm_scale, void *out,
                                      int32_t out_dtype, void *workspace, size_t *ws_bytes,
                                      int32_t *dev_status, kvq_stream_t stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (!ws_bytes) return KVQ_ERR_ARG;
  if (q_heads < 1 || q_heads % cache->kv_heads || n_q < 1 || n_cand < 1 || block_q < 1)
    return KVQ_ERR_ARG;
  if ((q_dtype != KVQ_F32 && q_dtype != KVQ_BF16) ||
      (out_dtype != KVQ_F32 && out_dtype != KVQ_BF16))
    return KVQ_ERR_ARG;
  if (cache->recent > 0 && cache->kwin_dtype == KVQ_MXFP8) return KVQ_ERR_UNSUPPORTED;
  if (n_cand > 65536 || q_heads > 65535 || cache->batch > 65535) return KVQ_ERR_UNSUPPORTED;
  const long lists = static_cast<long>(cache->batch) * q_heads * ((n_q + block_q - 1) / block_q);
  const bool tensor = kvq::candidate_lists_supported(*cache, q_dtype, block_q) && lists <= 65535;
  const size_t need = tensor ? kvq::candidate_lists_workspace_bytes(lists, n_cand) : 0;
  if (!workspace) {
    *ws_bytes = need;
    return KVQ_OK;
  }
  if (*ws_bytes < need) return KVQ_ERR_WORKSPACE;
  if (!q || !out || !idx) return KVQ_ERR_ARG;
  if (!aligned16(q) || !aligned16(out) || !aligned16(idx) || !aligned16(workspace) ||
      (dev_status && !aligned16(dev_status)))
    return KVQ_ERR_ALIGN;
  const float scale = resolve_scale(sm_scale, cache->head_dim);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  kvq::KernelCtl ctl = make_ctl(dev_status);
  {
    const long rows = static_cast<long>(cache->batch) * q_heads * n_q;
    ctl_add_cache(ctl, *cache);
    ctl_add(ctl, q, rows_bytes(rows, cache->head_dim, q_dtype));
    ctl_add(ctl, out, rows_bytes(rows, cache->head_dim, out_dtype));
    ctl_add(ctl, idx, rows_bytes(lists, n_cand, KVQ_F32));
    ctl_add(ctl, workspace, *ws_bytes);
  }
  if (tensor) {
    const int n = kvq::launch_candidate_lists(*cache, q, q_heads, n_q, idx, n_cand, block_q,
                                              static_cast<float>(scale * kLog2e), out, out_dtype,
                                              workspace, ctl, s);
    if (n < 0) return KVQ_ERR_CUDA;
    return finish(n, "candidates_block_tensor");
  }
  const int n = kvq::launch_attend_candidates(*cache, q, q_dtype, q_heads, n_q, idx, n_cand, 0,
                                              static_cast<float>(scale * kLog2e), out, out_dtype,
                                              ctl, s, 0, nullptr, block_q);
  return finish(n, "candidates_block");
}

kvq_status kv_attend_region_drop(const kvq_cache *cache, const void *q, int32_t q_dtype,
                                 int32_t q_heads, int32_t n_q, float sm_scale,
                                 const int32_t *region_bounds, int32_t n_regions,
                                 uint32_t drop_mask, void *out, int32_t out_dtype,
                                 void *workspace, size_t *ws_bytes, int32_t *dev_status,
                                 kvq_stream_t stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (!ws_bytes || !region_bounds) return KVQ_ERR_ARG;
  if (q_heads < 1 || q_heads % cache->kv_heads || n_q < 1) return KVQ_ERR_ARG;
  if (n_regions < 1 || n_regions > 16) return KVQ_ERR_ARG;
  if (region_bounds[0] != 0 || region_bounds[n_regions] != cache->n_tokens) return KVQ_ERR_ARG;
  for (int i = 0; i < n_regions; ++i)
    if (region_bounds[i + 1] <= region_bounds[i]) return KVQ_ERR_ARG;
  if (out_dtype != KVQ_F32 && out_dtype != KVQ_BF16) return KVQ_ERR_ARG;
  int kept = 0;
  for (int r = 0; r < n_regions; ++r)
    if (!(drop_mask & (1u << r))) kept += region_bounds[r + 1] - region_bounds[r];
  if (kept == 0 || (drop_mask >> n_regions) != 0) return KVQ_ERR_ARG;
  if (!kvq::candidate_lists_supported(*cache, q_dtype, 128) || q_heads > 65535 ||
      static_cast<long>(cache->batch) * cache->kv_heads > 65535)
    return KVQ_ERR_UNSUPPORTED;
  const size_t need = kvq::region_drop_workspace_bytes(*cache, kept);
  if (!workspace) {
    *ws_bytes = need;
    return KVQ_OK;
  }
  if (*ws_bytes < need) return KVQ_ERR_WORKSPACE;
  if (!q || !out) return KVQ_ERR_ARG;
  if (!aligned16(q) || !aligned16(out) || !aligned16(workspace) ||
      (dev_status && !aligned16(dev_status)))
    return KVQ_ERR_ALIGN;
  const float scale = resolve_scale(sm_scale, cache->head_dim);
  kvq::KernelCtl ctl = make_ctl(dev_status);
  {
    const long rows = static_cast<long>(cache->batch) * q_heads * n_q;
    ctl_add_cache(ctl, *cache);
    ctl_add(ctl, q, rows_bytes(rows, cache->head_dim, q_dtype));
    ctl_add(ctl, out, rows_bytes(rows, cache->head_dim, out_dtype));
    ctl_add(ctl, workspace, *ws_bytes);
  }
  const int n = kvq::launch_region_drop(*cache, q, q_heads, n_q, region_bounds, n_regions,
                                        drop_mask, static_cast<float>(scale * kLog2e), out,
                                        out_dtype, workspace, ctl,
                                        reinterpret_cast<cudaStream_t>(stream));
  if (n < 0) return KVQ_ERR_CUDA;
  return finish(n, "region_drop");
}

kvq_status kv_attend_decode_static(const kvq_cache *cache, const void *q, int32_t q_dtype,
                                   int32_t q_heads, float sm_scale, void *out,
                                   int32_t out_dtype, int32_t *dev_status, kvq_stream_t stream) {
  kvq_status st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (q_heads < 1 || q_heads % cache->kv_heads) return KVQ_ERR_ARG;
  if ((q_dtype != KVQ_F32 && q_dtype != KVQ_BF16) ||
      (out_dtype != KVQ_F32 && out_dtype != KVQ_BF16))
    return KVQ_ERR_ARG;
  if (!kvq::decode_supported(*cache, q_dtype, q_heads, 1)) return KVQ_ERR_UNSUPPORTED;
  if (!q || !out) return KVQ_ERR_ARG;
  if (!aligned16(q) || !aligned16(out) || (dev_status && !aligned16(dev_status)))
    return KVQ_ERR_ALIGN;
  const int sms = sm_count();
  if (kvq::decode_workspace_bytes(*cache, q_heads, sms) > kvq::decode_static_scratch_limit())
    return KVQ_ERR_WORKSPACE;
  void *scratch = nullptr;
  if (kvq::decode_static_scratch(&scratch) != cudaSuccess) return KVQ_ERR_CUDA;
  const float scale = resolve_scale(sm_scale, cache->head_dim);
  kvq::KernelCtl ctl = make_ctl(dev_status);
  {
    const long rows = static_cast<long>(cache->batch) * q_heads;
    ctl_add_cache(ctl, *cache);
    ctl_add(ctl, q, rows_bytes(rows, cache->head_dim, q_dtype));
    ctl_add(ctl, out, rows_bytes(rows, cache->head_dim, out_dtype));
    ctl_add(ctl, scratch, kvq::decode_static_scratch_limit());
  }
  const int n = kvq::launch_attend_decode(*cache, q, q_dtype, static_cast<float>(scale * kLog2e),
                                          out, out_dtype, scratch, ctl, sms,
                                          reinterpret_cast<cudaStream_t>(stream));
  return finish(n, "decode_static");
}

int32_t kvq_last_launch_count(void) { return g_last_launches; }

const char *kvq_last_path(void) { return g_last_path; }

int32_t kvq_debug_checks(void) {
#ifdef KVQ_DEBUG
  return 1;
#else
  return 0;
#endif
}

void kvq_debug_set(uint32_t wait_limit_ns, int32_t drop_item) {
  g_wait_limit_ns = wait_limit_ns;
  g_drop_item = drop_item;
}

}  // extern "C"
