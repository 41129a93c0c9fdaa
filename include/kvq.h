/*
 * kvq.h -- C ABI of the compressed-KV-cache attention library (sm_103a).
 *
 * The cache follows "KV殘差窗口：最近Token一定值得高精度嗎？" (huhohoo.com,
 * kv-residual-window), section 固定預算，先問它保護了誰: the tokens before the
 * last R are stored as grouped symmetric int4 (group 32, no zero point, K per
 * channel over 32-token groups, V per token over 32-feature groups) and the
 * last R tokens stay in floating point. Attention always covers the whole
 * context, or exactly a listed set of candidate keys (MiniCPM5-2B study,
 * bjdmk.com.cn/news/5855973, sections 6 and 9). The chunk layout and the
 * per-row region mass follow "Catnip Week 10 KV Cache Attention Study"
 * (cappuccino.cafe/kv-attn.html), section "KV Cache 的实际作用"; MXFP8 Q/K
 * (E4M3 elements, one E8M0 scale per 32 along the head dim) follows its section
 * "Q/K 与 probability quantization 的影响".
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    never allocates, never frees and never synchronises. Every pointer must be
 *    16-byte aligned (else KVQ_ERR_ALIGN).
 *  - Tensors are dense, row-major, in the index order written beside them.
 *  - GQA: query head h reads KV head h / (q_heads / kv_heads); q_heads must be
 *    a multiple of kv_heads.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream) and runs asynchronously.
 *  - Argument errors are returned before anything is enqueued. Errors a kernel
 *    detects are OR-ed as KVQ_DEV_* bits into *dev_status (a device int32 the
 *    caller zeroes beforehand and reads after synchronising); kernels never
 *    trap and every wait in them is bounded.
 *  - sm_scale <= 0 selects 1/sqrt(head_dim). There is no mask.
 *  - head_dim is a multiple of 32 in [32, 256].
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *kvq_stream_t; /* same type as cudaStream_t */

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_ARG = 1,         /* bad shape, dtype, count or NULL pointer */
  KVQ_ERR_ALIGN = 2,       /* a pointer is not 16-byte aligned */
  KVQ_ERR_UNSUPPORTED = 3, /* a valid combination this build has no kernel for */
  KVQ_ERR_WORKSPACE = 4,   /* workspace given but smaller than required */
  KVQ_ERR_CUDA = 5         /* a launch failed (cudaGetLastError) */
} kvq_status;

/* Bits OR-ed into *dev_status by kernels. */
enum {
  KVQ_DEV_INDEX = 1,   /* a candidate index outside [0, n_tokens) (that key is skipped) */
  KVQ_DEV_DUP = 2,     /* a candidate list holds the same index twice (validate only) */
  KVQ_DEV_TIMEOUT = 4, /* a bounded wait ran out; the outputs of that launch are invalid */
  KVQ_DEV_BOUNDS = 8   /* an address range a kernel derived lay outside the call's buffers
                          (checked in the KVQ_DEBUG build, kvq_debug_checks); outputs invalid */
};

typedef enum { KVQ_F32 = 0, KVQ_BF16 = 1, KVQ_MXFP8 = 2 } kvq_dtype;

/*
 * A packed cache of `batch` sequences x `kv_heads` heads, each holding
 * `n_tokens` (N) tokens of `head_dim` (D) features, the last `recent` (R)
 * tokens kept in the window. With cut = N - R and Gk = ceil(cut / 32):
 *
 *   k_codes  [batch][kv_heads][Gk][32][D/2]   uint8: token-group major; byte i
 *            of a token row holds channels 2i (low nibble) and 2i+1 (high
 *            nibble) as code + 8 (codes in [-7, 7]); padding tokens of the last
 *            group hold code 0.
 *   k_scales [batch][kv_heads][Gk][D]         float: one scale per (group, channel).
 *   v_codes  [batch][kv_heads][cut][D/2]      uint8: same nibble order, per token.
 *   v_scales [batch][kv_heads][cut][D/32]     float: one scale per (token, 32 features).
 *   k_window [batch][kv_heads][R][D]          kwin_dtype: F32, BF16, or MXFP8
 *            (E4M3 bytes, with k_window_e8m0 [batch][kv_heads][R][D/32] holding
 *            the E8M0 block-scale bytes, exponent + 127).
 *   v_window [batch][kv_heads][R][D]          vwin_dtype: F32 or BF16.
 *   header   {N, D, R, 32}: the 16 bytes of shape metadata, filled by kv_pack.
 *
 * Pointers for empty arrays (cut == 0 or R == 0) may be NULL.
 */
typedef struct kvq_cache {
  int32_t batch, kv_heads, n_tokens, head_dim, recent;
  int32_t kwin_dtype, vwin_dtype;
  uint8_t *k_codes;
  float *k_scales;
  uint8_t *v_codes;
  float *v_scales;
  void *k_window;
  void *v_window;
  uint8_t *k_window_e8m0;
  uint32_t header[4];
  /* Room reserved per (sequence, head) for kv_append; 0 and 0 = a tight cache
   * whose arrays are exactly the sizes above. With cap_groups > 0 the
   * per-(sequence, head) strides become cap_groups K groups (k_codes,
   * k_scales), 32 * cap_groups V rows (v_codes, v_scales) and cap_window
   * window rows (k_window, v_window, k_window_e8m0); rows past Gk, cut and R
   * are unused. Both are then required, with cap_groups >= Gk and
   * cap_window >= R. */
  int32_t cap_groups;
  int32_t cap_window;
} kvq_cache;

/* Array sizes of a cache, in bytes (host only, no GPU needed):
 * sizes[0..7] = k_codes, k_scales, v_codes, v_scales, k_window, v_window,
 * k_window_e8m0, header. Returns KVQ_ERR_ARG for an invalid shape. */
KVQ_API kvq_status kvq_cache_sizes(int32_t batch, int32_t kv_heads, int32_t n_tokens,
                                   int32_t head_dim, int32_t recent, int32_t kwin_dtype,
                                   int32_t vwin_dtype, size_t sizes[8]);

/* Array sizes of a cache laid out for kv_append, with cap_groups >= 1 K groups
 * (and 32 * cap_groups V rows) and cap_window window rows reserved per
 * (sequence, head); same order as kvq_cache_sizes. KVQ_ERR_ARG for an invalid
 * shape. */
KVQ_API kvq_status kvq_cache_sizes_reserved(int32_t batch, int32_t kv_heads, int32_t head_dim,
                                            int32_t kwin_dtype, int32_t vwin_dtype,
                                            int32_t cap_groups, int32_t cap_window,
                                            size_t sizes[8]);

/* Total payload in bytes: the sum of kvq_cache_sizes (header included). */
KVQ_API size_t kvq_cache_bytes(int32_t batch, int32_t kv_heads, int32_t n_tokens,
                               int32_t head_dim, int32_t recent, int32_t kwin_dtype,
                               int32_t vwin_dtype);

/*
 * kv_pack -- quantize K and V into `cache` (residual-window page, section
 * 固定預算). k, v: [batch][kv_heads][N][D] in in_dtype (F32 or BF16), device.
 * For each (sequence, head): tokens [0, cut) are quantized, tokens [cut, N)
 * are copied into the window (rounded to nearest even when the window type is
 * narrower; E4M3 with an E8M0 scale per 32 features for an MXFP8 K window).
 * int4 rule: scale = amax / 7 rounded to fp32, code = clamp(rint(x / scale),
 * -7, 7) with the division correctly rounded in fp32 and ties to even; a zero
 * scale gives all-zero codes. Inputs are expected finite: the code of a NaN
 * or infinite element is unspecified (the group's other elements follow the
 * rule; a NaN does not enter amax). The cache's shape fields and array
 * pointers are read; header[] is written. dev_status may be NULL.
 */
KVQ_API kvq_status kv_pack(const void *k, const void *v, int32_t in_dtype, kvq_cache *cache,
                           int32_t *dev_status, kvq_stream_t stream);

/*
 * kv_append -- add n_new tokens per (sequence, head) to a cache laid out with
 * reserved room (cap_groups > 0), as decoding produces them. The pages build
 * the cache once and leave this online update out ("KV殘差窗口", section
 * 適用邊界：本輪沒有測在線更新: the oldest window entries are not migrated
 * into the quantized part token by token); this call is that update, with
 * the cache layout and quantization rule of kv_pack.
 * k_new, v_new: [batch][kv_heads][n_new][D] in in_dtype (F32 or BF16), device.
 * The window grows by n_new; then, while it holds at least `window` + 32
 * tokens, its oldest 32 become one more int4 K group and 32 more V rows (the
 * kv_pack rule applied to the window's values, so the result equals kv_pack
 * of the whole sequence whenever the window type holds the inputs exactly --
 * BF16 inputs with a BF16 window, or an F32 window). Afterwards N - R is the
 * largest multiple of 32 leaving at least `window` tokens in the window (and
 * never less than before), so R lies in [window, window + 31] once
 * N >= window.
 * On success the call updates cache->n_tokens, cache->recent and header[]
 * (host fields) and enqueues the kernels on `stream`.
 * Errors: KVQ_ERR_UNSUPPORTED for a tight cache (cap_groups == 0), an MXFP8
 * K window, an int4 part whose last K group is padded ((N - R) % 32 != 0) or
 * more than 65,535 (sequence, head) pairs when groups migrate;
 * KVQ_ERR_WORKSPACE when the reserved room (cap_groups, cap_window) is too
 * small for the result; the cache is then left unchanged.
 */
KVQ_API kvq_status kv_append(kvq_cache *cache, const void *k_new, const void *v_new,
                             int32_t in_dtype, int32_t n_new, int32_t window,
                             int32_t *dev_status, kvq_stream_t stream);

/*
 * kv_attend -- O = softmax(sm_scale * Q K^T) V over all N tokens of the cache,
 * with K, V dequantized (int4 part) or taken from the window.
 * q:   [batch][q_heads][n_q][D] in q_dtype (F32 or BF16), device.
 * out: [batch][q_heads][n_q][D] in out_dtype (F32 or BF16), device.
 * region_bounds: HOST array of n_regions + 1 increasing token positions
 *   starting at 0 and ending at N, or NULL; region_mass: device float
 *   [batch][q_heads][n_q][n_regions] receiving, per query row, the softmax
 *   mass on tokens [b_k, b_{k+1}) (n_regions <= 16). For an MXFP8 K window, Q
 *   is quantized the same way (E4M3 + E8M0 per 32) before QK^T.
 * workspace: device scratch of *ws_bytes bytes. With workspace == NULL the
 *   call only stores the required size in *ws_bytes and returns KVQ_OK
 *   (enqueueing nothing); to run, pass a non-NULL workspace even when the
 *   required size is 0.
 * Kernel choice: one query row per (sequence, head) with 8 query heads per KV
 *   head and D = 128 runs the split-K decode kernels; with bf16 q, D = 128
 *   and at least 64 query rows, a bf16 or MXFP8 window covering all tokens,
 *   or an int4 part followed by a bf16 window (the key tiles holding int4
 *   tokens are expanded to bf16 in the workspace, the others read in place),
 *   runs the tensor-core chunk kernel (when batch * q_heads <= 65,535);
 *   everything else runs the fp32 kernel, which needs q_heads and batch
 *   <= 65,535 (else KVQ_ERR_UNSUPPORTED).
 */
KVQ_API kvq_status kv_attend(const kvq_cache *cache, const void *q, int32_t q_dtype,
                             int32_t q_heads, int32_t n_q, float sm_scale, void *out,
                             int32_t out_dtype, const int32_t *region_bounds, int32_t n_regions,
                             float *region_mass, void *workspace, size_t *ws_bytes,
                             int32_t *dev_status, kvq_stream_t stream);

/* Columns of kv_attend_stats' output, one row of KVQ_N_STATS floats per query. */
enum {
  KVQ_STAT_ENTROPY = 0,  /* H = -sum p ln p (nats) */
  KVQ_STAT_SUPPORT = 1,  /* exp(H) / N: entropy-equivalent share of the keys */
  KVQ_STAT_TOP1 = 2,     /* mass of the ceil(1 % of N) largest probabilities */
  KVQ_STAT_TOP5 = 3,     /* ... ceil(5 %) */
  KVQ_STAT_TOP10 = 4,    /* ... ceil(10 %) */
  KVQ_STAT_ZERO = 5,     /* share of probabilities exactly 0 in fp32 */
  KVQ_STAT_P_ZERO = 6,   /* share of keys nonzero in fp32 but 0 on the MXFP8 P path */
  KVQ_STAT_P_TV = 7,     /* 0.5 sum |p_mx - p| on the MXFP8 P path */
  KVQ_STAT_P_SUM = 8,    /* sum p_mx (the P-path proxy row sum) */
  KVQ_STAT_QK_TV = 9,    /* 0.5 sum |p_qk - p|, p_qk from MXFP8 Q/K */
  KVQ_STAT_QK_AGREE = 10, /* 1 when p_qk and p have the same argmax (first index), else 0 */
  KVQ_N_STATS = 11
};

/*
 * kv_attend_stats -- observer statistics of attention rows (Catnip study,
 * "Catnip Week 10 KV Cache Attention Study", section 实验设计 step 5 with its
 * Structural / Effective / Numerical MXFP8 notes, and section "Q/K 与
 * probability quantization 的影响"). For each query row, p is the fp32
 * softmax of sm_scale * q K^T over all N keys of the cache, K as kv_attend
 * reads it. The MXFP8 P path rounds p to E4M3 with one E8M0 scale per 32
 * consecutive keys (the scale rule of the MXFP8 K window). The MXFP8 Q/K path
 * rotates q and every key by the signed Hadamard transform
 * x -> (x * signs) H / sqrt(D) (H the Sylvester Hadamard matrix of order D)
 * when hadamard_signs is not NULL, rounds both to MXFP8 along D and takes the
 * softmax of their scores (p_qk).
 * q: [batch][q_heads][n_q][D] in q_dtype (F32 or BF16), device; typically a
 *   sample of query rows. hadamard_signs: device float [D] of +-1, or NULL.
 * stats: device float [batch][q_heads][n_q][KVQ_N_STATS], see KVQ_STAT_*.
 * workspace/ws_bytes as kv_attend (it holds every key twice in fp32, as
 * attention reads it and on the MXFP8 Q/K path, and both score rows of
 * every query row: about 8 x B x Hkv x N x D + 8 x B x q_heads x n_q x N
 * bytes).
 * Restrictions (else KVQ_ERR_UNSUPPORTED): D in {32, 64, 128, 256},
 * N <= 1,048,576, batch * q_heads <= 65,535. A row's reference scores are
 * swept in shared memory up to 16,384 keys, longer rows in place in the
 * workspace (slower).
 */
KVQ_API kvq_status kv_attend_stats(const kvq_cache *cache, const void *q, int32_t q_dtype,
                                   int32_t q_heads, int32_t n_q, float sm_scale,
                                   const float *hadamard_signs, float *stats, void *workspace,
                                   size_t *ws_bytes, int32_t *dev_status, kvq_stream_t stream);

/*
 * kv_attend_candidates -- exact attention of each query row over its own
 * candidate keys only (MiniCPM5-2B study, sections 6 and 9): row (b, h, i)
 * attends the n_cand token positions idx[b][h][i][:] (int32, device) and no
 * other key. Lists hold distinct positions in any order. An index outside
 * [0, N) is skipped and flagged KVQ_DEV_INDEX; with validate != 0 duplicate
 * positions are flagged KVQ_DEV_DUP (the output of that row is then invalid).
 * An MXFP8 K window, n_cand > 65,536 and q_heads or batch above 65,535 are
 * not supported (KVQ_ERR_UNSUPPORTED). Other arguments as for kv_attend.
 * Kernel choice: with D = 128, bf16 q, one query row, 8 query heads per KV
 * head, a bf16 window (or none) and 8 x n_cand <= 4096, one pass per
 * (sequence, KV head) covers the union of its 8 query heads' lists, reading
 * each distinct row and K-scale group once and scoring it for all 8 heads on
 * the tensor cores (bf16 operands, the int4 rows rounded once to bf16); it
 * needs workspace for per-slice partials (query it with workspace == NULL).
 * Other shapes run a per-row fp32 kernel and need none.
 */
KVQ_API kvq_status kv_attend_candidates(const kvq_cache *cache, const void *q, int32_t q_dtype,
                                        int32_t q_heads, int32_t n_q, const int32_t *idx,
                                        int32_t n_cand, int32_t validate, float sm_scale,
                                        void *out, int32_t out_dtype, void *workspace,
                                        size_t *ws_bytes, int32_t *dev_status,
                                        kvq_stream_t stream);

/*
 * kv_attend_candidates_topk -- the two-stage form of candidate attention
 * (MiniCPM5-2B study, section 6: a predictor proposes top-C candidates, then
 * the true top-32 inside them is taken by exact score): each query row scores
 * its n_cand listed keys exactly (sm_scale * q . k, keys as kv_attend reads
 * them), keeps the top_k highest (equal scores: the key listed first) and
 * attends exactly over those. q, idx, out as kv_attend_candidates; positions
 * outside [0, N) score -inf (flagged KVQ_DEV_INDEX) and are never kept.
 * selected: device int32 [batch][q_heads][n_q][top_k] receiving the kept
 *   positions in score order (-1 past the valid ones), or NULL.
 * Restrictions: 1 <= top_k <= n_cand <= 4096 (else KVQ_ERR_ARG /
 * KVQ_ERR_UNSUPPORTED); an MXFP8 K window is not supported. No workspace.
 */
KVQ_API kvq_status kv_attend_candidates_topk(const kvq_cache *cache, const void *q,
                                             int32_t q_dtype, int32_t q_heads, int32_t n_q,
                                             const int32_t *idx, int32_t n_cand, int32_t top_k,
                                             float sm_scale, void *out, int32_t out_dtype,
                                             int32_t *selected, int32_t *dev_status,
                                             kvq_stream_t stream);

/*
 * kv_attend_candidates_block -- candidate attention for many query rows
 * (prefill) with one candidate list per block of block_q consecutive query
 * rows of a head. The MiniCPM5-2B study (section 9) found its prefill kernel,
 * which gathered a head's candidate rows again for every query block, slower
 * than dense attention, and names the fix: a block-shared candidate layout
 * with the rows tiled through on-chip memory. Row i of head h of sequence b
 * attends exactly over the keys of list idx[b][h][i / block_q][0 .. n_cand).
 * idx: device int32 [batch][q_heads][ceil(n_q / block_q)][n_cand] of distinct
 *   positions in [0, N) (others are flagged KVQ_DEV_INDEX; such a list's rows
 *   are then invalid). q, out as kv_attend.
 * With D = 128, bf16 q, block_q a multiple of 128 and no MXFP8 K window,
 * every list's K and V rows are gathered once into workspace as bf16 and the
 * rows attend them on the tensor cores; otherwise the fp32 candidate kernel
 * runs with the shared lists (no workspace). workspace/ws_bytes as kv_attend.
 */
KVQ_API kvq_status kv_attend_candidates_block(const kvq_cache *cache, const void *q,
                                              int32_t q_dtype, int32_t q_heads, int32_t n_q,
                                              const int32_t *idx, int32_t n_cand, int32_t block_q,
                                              float sm_scale, void *out, int32_t out_dtype,
                                              void *workspace, size_t *ws_bytes,
                                              int32_t *dev_status, kvq_stream_t stream);

/*
 * kv_attend_region_drop -- the local output ablation the Catnip study
 * recommends ("Catnip Week 10 KV Cache Attention Study", section
 * 当前判断与下一步优化空间: drop sink, drop recent or drop all history,
 * renormalise P, compare the attention output): O over the keys of the regions
 * NOT set in drop_mask only, the softmax renormalised over them.
 * region_bounds: HOST array of n_regions + 1 increasing positions from 0 to N
 * (n_regions <= 16); bit r of drop_mask drops region r (at least one key must
 * remain). q, out, workspace/ws_bytes as kv_attend. The kept keys of every
 * (sequence, KV head) are gathered once to bf16 in workspace and attended on
 * the tensor cores: D = 128, bf16 q and no MXFP8 K window, else
 * KVQ_ERR_UNSUPPORTED.
 */
KVQ_API kvq_status kv_attend_region_drop(const kvq_cache *cache, const void *q, int32_t q_dtype,
                                         int32_t q_heads, int32_t n_q, float sm_scale,
                                         const int32_t *region_bounds, int32_t n_regions,
                                         uint32_t drop_mask, void *out, int32_t out_dtype,
                                         void *workspace, size_t *ws_bytes, int32_t *dev_status,
                                         kvq_stream_t stream);

/*
 * kv_attend_decode_static -- the decode case of kv_attend (one query row per
 * sequence and head, 8 query heads per KV head, D = 128, bf16 or no window)
 * for callers that cannot allocate device memory: a serving runtime that has
 * already handed all free HBM to its KV-cache pool (any further cudaMalloc
 * fails), or a latency-critical caller that cannot afford cudaMalloc's
 * implicit device synchronisation. The pages have no counterpart; it exists
 * only for those callers.
 * Same q / out / dtype / dev_status / stream rules as kv_attend; no
 * workspace argument. The split-K partials go to a scratch array of
 * KVQ_DECODE_STATIC_SCRATCH_BYTES (8 MiB) that the library keeps in device
 * memory on every GPU that loads it, until the process exits. A call whose
 * partials need more (batch * kv_heads above 992 on a
 * 152-SM GPU) returns KVQ_ERR_WORKSPACE and enqueues nothing; other
 * unsupported shapes return KVQ_ERR_UNSUPPORTED. Nothing is allocated, by
 * the library or by any library it calls.
 * The array's device address is looked up (cudaGetSymbolAddress) once per
 * device, with that device current, by the first kv_pack or kv_append on the
 * device, or else by the first call of this entry point; make that first call
 * before any stream capture. The lookup loads the library's decode module on
 * the device (CUDA loads modules lazily by default), and that load is what
 * takes the 8 MiB: a runtime that hands all free HBM to its KV-cache pool
 * should pack (or append to) a cache first, as it must before decoding anyway.
 * If the lookup fails, the call returns KVQ_ERR_CUDA with the CUDA error
 * cleared. The looked-up address is kept for the life of the process: do not
 * use the library across a cudaDeviceReset on that device.
 * Every call reads scratch it wrote itself in the
 * same call, so nothing needs clearing between calls, but all calls share
 * the one array: calls that overlap on the GPU (different streams, no
 * ordering between them) race and corrupt each other's results.
 */
#define KVQ_DECODE_STATIC_SCRATCH_BYTES (8u << 20)
KVQ_API kvq_status kv_attend_decode_static(const kvq_cache *cache, const void *q,
                                           int32_t q_dtype, int32_t q_heads, float sm_scale,
                                           void *out, int32_t out_dtype, int32_t *dev_status,
                                           kvq_stream_t stream);

/* Number of kernel launches the last successful call on this thread enqueued. */
KVQ_API int32_t kvq_last_launch_count(void);

/* Name of the kernel family the last successful call on this thread used
 * ("pack", "decode", "chunk_bf16", "chunk_mxfp8", "generic", "candidates");
 * a static string. */
KVQ_API const char *kvq_last_path(void);

/*
 * Test hook: bound every mbarrier wait of the next launches on this thread to
 * `wait_limit_ns` nanoseconds (0 restores the default of one second), and,
 * when drop_item >= 0, make the loader of the decode kernel and of the bf16
 * kv_pack kernel skip the copy of that work item so that the wait on it can
 * only run out. Used by the failure tests.
 */
KVQ_API void kvq_debug_set(uint32_t wait_limit_ns, int32_t drop_item);

/*
 * 1 when this library was built with KVQ_DEBUG (libkvq_debug.so), else 0. In
 * that build every kernel checks each global address range it derives from
 * its indices (a row, a chunk, a bulk copy) against the device buffers the
 * call passed -- the cache's arrays at the sizes its shape gives, q, the
 * outputs, index lists and the workspace at the size given in *ws_bytes --
 * and, for a range outside them, sets KVQ_DEV_BOUNDS in *dev_status and
 * leaves the access out (a load reads zeros, a store is dropped, a bulk copy
 * is neither issued nor waited for), so a wrong index is reported instead of
 * faulting. TMA tile copies are bounded by their tensor maps. The checks cost
 * time; the outputs of a call that reports no error are those of the other
 * build.
 */
KVQ_API int32_t kvq_debug_checks(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
