// Host-side launchers implemented by the kernel files and called by the C ABI
// layer (kvq_api.cu). Arguments are already validated when these run.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/kvq.h"
#include "kvq_common.cuh"

namespace kvq {

// Shape of a cache, derived once from a kvq_cache. Gs, Vs and Ws are the
// per-(sequence, head) strides of the K-group, V-row and window arrays: the
// sizes themselves for a tight cache, the reserved counts for one laid out
// for kv_append.
struct CacheDims {
  int B, Hkv, N, D, R, cut, Gk;
  int Gs, Vs, Ws;
};

inline CacheDims dims_of(const kvq_cache &c) {
  CacheDims d;
  d.B = c.batch;
  d.Hkv = c.kv_heads;
  d.N = c.n_tokens;
  d.D = c.head_dim;
  d.R = c.recent;
  d.cut = c.n_tokens - c.recent;
  d.Gk = (d.cut + kGroup - 1) / kGroup;
  d.Gs = c.cap_groups > 0 ? c.cap_groups : d.Gk;
  d.Vs = c.cap_groups > 0 ? kGroup * c.cap_groups : d.cut;
  d.Ws = c.cap_window > 0 ? c.cap_window : d.R;
  return d;
}

// Region bounds live in a small by-value struct so kernels need no extra copy.
struct Regions {
  int n;      // number of regions, 0 = none
  int b[17];  // bounds b[0] = 0 < ... < b[n] = N
};

inline Regions make_regions(const int32_t *bounds, int n) {
  Regions r{};
  r.n = bounds ? n : 0;
  if (bounds)
    for (int i = 0; i <= r.n && i < 17; ++i) r.b[i] = bounds[i];
  return r;
}

// pack.cu
int launch_pack(const void *k, const void *v, int in_dtype, const kvq_cache &c,
                const KernelCtl &ctl, int num_sms, cudaStream_t s);

// pack.cu: kv_append on a cache with reserved room: n_new tokens per
// (sequence, head) after the current ones; m groups of the oldest window
// tokens become int4 and the window becomes R_new rows.
int launch_append(const kvq_cache &c, const void *k_new, const void *v_new, int in_dtype,
                  int n_new, int m, int R_new, const KernelCtl &ctl, cudaStream_t s);

// attend_generic.cu: fp32 CUDA-core attention for any supported shape.
int launch_attend_generic(const kvq_cache &c, const void *q, int q_dtype, int Hq, int n_q,
                          float sm_scale, void *out, int out_dtype, const int32_t *bounds,
                          int n_regions, float *mass, const KernelCtl &ctl, cudaStream_t s);

// attend_decode.cu: split-K decode for D = 128, 8 query heads per KV head, one query.
bool decode_supported(const kvq_cache &c, int q_dtype, int Hq, int n_q);
size_t decode_workspace_bytes(const kvq_cache &c, int Hq, int num_sms);
int launch_attend_decode(const kvq_cache &c, const void *q, int q_dtype, float scale_log2,
                         void *out, int out_dtype, void *ws, const KernelCtl &ctl, int num_sms,
                         cudaStream_t s);

// attend_decode.cu: the same decode kernels with the partials in a static
// device array (kv_attend_decode_static).
size_t decode_static_scratch_limit();
cudaError_t decode_static_scratch(void **ptr);

// attend_candidates.cu
// top_k > 0: attend only the top_k listed keys by exact score (selected, if
// not null, receives their positions); n_cand <= candidates_topk_max() then.
int launch_attend_candidates(const kvq_cache &c, const void *q, int q_dtype, int Hq, int n_q,
                             const int32_t *idx, int n_cand, int validate, float scale_log2,
                             void *out, int out_dtype, const KernelCtl &ctl, cudaStream_t s,
                             int top_k = 0, int32_t *selected = nullptr, int block_q = 1);
int candidates_topk_max();

// attend_candidates.cu: one pass per (sequence, KV head) over the union of its
// 8 query heads' lists (D = 128, bf16 q, one query row, 8 x C <= 4096).
bool candidates_union_supported(const kvq_cache &c, int q_dtype, int Hq, int n_q, int n_cand);
size_t candidates_union_workspace_bytes(const kvq_cache &c, int n_cand, int num_sms);
int launch_candidates_union(const kvq_cache &c, const void *q, const int32_t *idx, int n_cand,
                            int validate, float scale_log2, void *out, int out_dtype, void *ws,
                            const KernelCtl &ctl, int num_sms, cudaStream_t s);

// attend_chunk.cu: kv_attend_candidates_block on the tensor cores (lists of
// block_q query rows gathered once to bf16 in workspace).
bool candidate_lists_supported(const kvq_cache &c, int q_dtype, int block_q);
size_t candidate_lists_workspace_bytes(long lists, int C);
int launch_candidate_lists(const kvq_cache &c, const void *q, int Hq, int n_q,
                           const int32_t *idx, int C, int block_q, float scale_log2, void *out,
                           int out_dtype, void *ws, const KernelCtl &ctl, cudaStream_t s);
// kv_attend_region_drop (same conditions as the block lists, block_q = any).
size_t region_drop_workspace_bytes(const kvq_cache &c, int kept);
int launch_region_drop(const kvq_cache &c, const void *q, int Hq, int n_q, const int32_t *bounds,
                       int n_regions, uint32_t drop_mask, float scale_log2, void *out,
                       int out_dtype, void *ws, const KernelCtl &ctl, cudaStream_t s);

// attend_chunk.cu: tcgen05 chunk attention over an all-window bf16 / MXFP8 cache.
bool chunk_supported(const kvq_cache &c, int q_dtype, int Hq, int n_q);
size_t chunk_workspace_bytes(const kvq_cache &c, int Hq, int n_q);
int chunk_max_regions();
int launch_attend_chunk(const kvq_cache &c, const void *q, int Hq, int n_q, float scale_log2,
                        void *out, int out_dtype, const int32_t *bounds, int n_regions,
                        float *mass, void *ws, const KernelCtl &ctl, cudaStream_t s);

// attend_stats.cu: observer statistics of attention rows (kv_attend_stats).
int stats_max_tokens();
size_t stats_workspace_bytes(const kvq_cache &c, int Hq, int n_q);
int launch_attend_stats(const kvq_cache &c, const void *q, int q_dtype, int Hq, int n_q,
                        float sm_scale, const float *signs, float *stats, void *ws,
                        const KernelCtl &ctl, cudaStream_t s);

}  // namespace kvq
