/*
 * pkv.h - C ABI of a GB300 (sm_103a) library for the paged KV-cache attention
 * step of an LLM serving engine: store new tokens' K/V into a paged pool,
 * then run decode or extend (chunked-prefill) attention through page tables.
 *
 * The operations follow the Mini-SGLang pages:
 *  - "Code Notes: mini-sglang", Engine Layer table, BaseKVCachePool row:
 *    the pool is ONE tensor (2, num_layers, num_pages, page_size, heads,
 *    head_dim) (index 0 = K, 1 = V), and store_kv() writes it at out_loc
 *    indices.
 *  - same page, Scheduler Layer table, TableManager row: one page_table row
 *    per request; CacheManager row: free_slots are token positions (slots).
 *  - same page, Engine Layer table, BaseAttnBackend row: prefill and decode
 *    are separate attention calls; Scheduler Layer table, PrefillManager row
 *    and "Introduction", Key Features (Chunked Prefill, Radix Cache): a prompt
 *    chunk attends over its cached, possibly shared, prefix plus itself.
 *  - same page, Engine Layer table, GraphRunner row: decode is replayed from
 *    CUDA graphs, so every call here is asynchronous on the given stream,
 *    never synchronises, never allocates and never changes the current
 *    device.
 *
 * Conventions for every call:
 *  - Pointers marked "device" are device memory owned by the caller. The
 *    library keeps no pointer after a call returns.
 *  - bf16 tensors are row-major and contiguous unless a stride is given.
 *    All integer tables (page_table, out_loc, seq_lens, qo_indptr,
 *    table_idx) are int32; address arithmetic is int64 throughout.
 *  - Layout of the pool (element offset, all int64):
 *      ((((c * L + layer) * num_pages + page) * page_size + off) * Hkv + h) * D + d
 *    with c = 0 for K and 1 for V. A slot is page * page_size + off.
 *  - A page_table entry is a physical page id: key i of a row lives at page
 *    row[i / page_size], offset i % page_size. For page_size 1 an entry is
 *    the slot itself. Entries past a row's seq_len are never read.
 *  - GQA: q head h reads kv head h / (Hq / Hkv).
 *  - lse outputs are natural-log log-sum-exp of the scaled scores, fp32.
 *  - Host-visible arguments are validated: a bad one returns
 *    PKV_ERR_INVALID_ARG (or PKV_ERR_UNSUPPORTED for a valid but unsupported
 *    shape) and launches nothing. A failed launch returns PKV_ERR_CUDA.
 *    pkv_last_error() gives a one-line reason for the last failure on the
 *    calling thread.
 *  - Device-resident values (page_table entries, out_loc, seq_lens,
 *    qo_indptr) are bounds-checked on the device: an out-of-range value is
 *    skipped (its key is treated as absent, its store is dropped), never
 *    dereferenced, and a bit is set in the device error word that
 *    pkv_read_device_errors() returns.
 *  - Supported: head_dim 64 or 128; Hq / Hkv = 1..8 (decode) or 1..16
 *    (extend); any page_size >= 1; the current device must be compute
 *    capability 10.3 (pkv_init checks it).
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,
  PKV_ERR_UNSUPPORTED = 2,
  PKV_ERR_WORKSPACE_TOO_SMALL = 3,
  PKV_ERR_CUDA = 4
} pkv_status;

/* Bits of the device error word (pkv_read_device_errors). */
#define PKV_DEVERR_OUT_LOC_RANGE 0x1    /* kv_store: out_loc outside the pool  */
#define PKV_DEVERR_PAGE_RANGE 0x2       /* a page_table entry outside the pool */
#define PKV_DEVERR_SEQ_LEN_RANGE 0x4    /* seq_len < 0 or past the row's stride */
#define PKV_DEVERR_INDPTR 0x8           /* qo_indptr not monotone / prefix < 0 */
#define PKV_DEVERR_TABLE_IDX_RANGE 0x10 /* table_idx negative                  */
#define PKV_DEVERR_TIMEOUT 0x20         /* a bounded in-kernel wait gave up     */

/* The KV pool (one tensor, see the layout above). base: device, bf16,
 * 16-byte aligned. Passed by pointer; the library does not keep it. */
typedef struct {
  void *base;
  int32_t num_layers;
  int64_t num_pages;
  int32_t page_size;
  int32_t num_kv_heads;
  int32_t head_dim;
} pkv_pool;

/* Checks that the current device is compute capability 10.3 and caches its
 * SM count. PKV_ERR_UNSUPPORTED otherwise. Every other call performs the
 * same check lazily; calling this first only moves it out of the hot path. */
pkv_status pkv_init(void);

/* Human-readable name of a status code (static string). */
const char *pkv_status_string(pkv_status s);

/* One-line reason for the last non-OK status returned on this thread
 * (thread-local static buffer, valid until the next failing call). */
const char *pkv_last_error(void);

/*
 * store_kv ("Code Notes: mini-sglang", Engine Layer table, BaseKVCachePool
 * row): for i < num_tokens,
 *   pool[0, layer, out_loc[i]] = k[i]   and   pool[1, layer, out_loc[i]] = v[i]
 * k, v: device bf16 [num_tokens, Hkv, D], token rows kv_row_stride elements
 * apart (>= Hkv * D, a multiple of 8), heads and dims contiguous, 16-byte
 * aligned (so k and v may be column slices of a fused QKV output).
 * out_loc: device int32 [num_tokens], flat slots. Two tokens with the same
 * slot give an unspecified one of the two rows. Bits are copied unchanged.
 */
pkv_status pkv_kv_store(const pkv_pool *pool, int32_t layer, const void *k, const void *v,
                        int64_t kv_row_stride, const int32_t *out_loc, int64_t num_tokens,
                        cudaStream_t stream);

/*
 * Bytes of device workspace pkv_paged_decode_attn needs for these host-side
 * sizes on the current device (0 when no request is split). The split plan
 * depends only on these arguments and the device's SM count, never on
 * device data, so the call stays graph-capturable.
 * max_seq_len_hint: an upper bound on every seq_len of the call; it sets how
 * finely long rows are split. A value < 1 means "no bound known" and
 * disables splitting (correct, but one CTA per request and head group).
 */
size_t pkv_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t max_seq_len_hint);

/*
 * Decode attention ("Code Notes: mini-sglang", Engine Layer table,
 * BaseAttnBackend and BaseKVCachePool rows; Scheduler Layer table,
 * TableManager row). For request b < batch and q head h < num_q_heads, with
 * row = page_table + (table_idx ? table_idx[b] : b) * table_stride and
 * n = seq_lens[b]:
 *   s_i = scale * <q[b,h,:], K[key i of row, h / g, :]>    for i < n
 *   o[b,h,:] = sum_i softmax(s)_i V[key i of row, h / g, :]
 *   lse[b,h] = log sum_i exp(s_i)
 * n = 0 gives o = 0 and lse = -inf. The newest token must already be in
 * the pool (call pkv_kv_store first, on the same stream).
 * q, o: device bf16 [batch, Hq, D], 16-byte aligned. lse: device fp32
 * [batch, Hq] or NULL. page_table: device int32 [rows, table_stride].
 * table_idx: device int32 [batch] or NULL (row b). seq_lens: device int32
 * [batch]. Long rows are split across CTAs (split-KV) and merged by
 * log-sum-exp; the partial states live in the caller's workspace (device,
 * 256-byte aligned, >= pkv_decode_workspace_size(...) bytes, contents
 * irrelevant on entry). A seq_len above max_seq_len_hint is still computed
 * correctly, only with less parallelism.
 */
pkv_status pkv_paged_decode_attn(const pkv_pool *pool, int32_t layer, const void *q, void *o,
                                 float *lse, const int32_t *page_table, int64_t table_stride,
                                 const int32_t *table_idx, const int32_t *seq_lens,
                                 int32_t batch, int32_t num_q_heads, float scale,
                                 int32_t max_seq_len_hint, void *workspace,
                                 size_t workspace_bytes, cudaStream_t stream);

/*
 * One decode step with store_kv fused in ("Code Notes: mini-sglang", Engine
 * Layer table, BaseKVCachePool row: the new token's K and V are written into
 * the pool, then attention reads the pool; GraphRunner row: decode steps are
 * launch-bound, so one launch fewer matters). For every request b the new
 * rows k_new[b, :, :] and v_new[b, :, :] (device bf16, [batch, Hkv, D] with
 * kv_row_stride elements between requests, 16-byte aligned, stride >= Hkv*D
 * and a multiple of 8) are stored at key position seq_lens[b] - 1 of its
 * page_table row (the slot P * row[(n-1)/P] + (n-1)%P, n = seq_lens[b]),
 * then attention runs exactly as pkv_paged_decode_attn (same arguments,
 * workspace from pkv_decode_workspace_size). Equivalent to pkv_kv_store with
 * out_loc[b] = that slot followed by pkv_paged_decode_attn; requests with
 * seq_lens[b] = 0 store nothing. A bad page id at that position is flagged
 * (PKV_DEVERR_PAGE_RANGE) and nothing is stored for it.
 */
pkv_status pkv_paged_decode_attn_store(const pkv_pool *pool, int32_t layer, const void *q,
                                       const void *k_new, const void *v_new,
                                       int64_t kv_row_stride, void *o, float *lse,
                                       const int32_t *page_table, int64_t table_stride,
                                       const int32_t *table_idx, const int32_t *seq_lens,
                                       int32_t batch, int32_t num_q_heads, float scale,
                                       int32_t max_seq_len_hint, void *workspace,
                                       size_t workspace_bytes, cudaStream_t stream);

/* Size of the library-owned scratch used by pkv_paged_decode_attn_noalloc. */
#define PKV_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * Decode attention that allocates nothing and takes no workspace. The pages
 * have no counterpart to this call: it exists for callers that cannot
 * allocate device memory or hand the library a workspace, such as a plugin
 * running inside a host framework that owns all device memory and gives the
 * plugin no allocation hook, or a serving loop that must never call
 * cudaMalloc because it can synchronise the device and can fail with
 * out-of-memory in the middle of a step.
 *
 * Same arguments and results as pkv_paged_decode_attn, minus the workspace:
 * the split-KV partial states go to a fixed scratch array in device memory
 * that the library owns (PKV_NOALLOC_SCRATCH_BYTES = 32 MiB, held by every
 * GPU that loads the library until the process exits).
 *  - If the split plan for these sizes needs more than that
 *    (pkv_decode_workspace_size(...) > PKV_NOALLOC_SCRATCH_BYTES), the call
 *    returns PKV_ERR_WORKSPACE_TOO_SMALL and launches nothing; lower batch
 *    or max_seq_len_hint, or use pkv_paged_decode_attn.
 *  - The first call on a device looks up the scratch array's device address
 *    (cudaGetSymbolAddress, with that device current). Make that first call
 *    before any stream capture begins.
 *  - Every call on a device shares the one array and it keeps whatever the
 *    last call left; nothing in it needs to start at zero. Calls whose
 *    kernels can overlap on the GPU (different streams without ordering
 *    between them) race on the array: order them on one stream.
 */
pkv_status pkv_paged_decode_attn_noalloc(const pkv_pool *pool, int32_t layer, const void *q,
                                         void *o, float *lse, const int32_t *page_table,
                                         int64_t table_stride, const int32_t *table_idx,
                                         const int32_t *seq_lens, int32_t batch,
                                         int32_t num_q_heads, float scale,
                                         int32_t max_seq_len_hint, cudaStream_t stream);

/*
 * Bytes of device workspace pkv_paged_extend_attn needs: the visible K and V
 * rows of every request, gathered once out of the paged pool into one
 * contiguous run per (request, kv head), each request's seq_len rounded up
 * to 128 rows, the requests' runs back to back ([2][Hkv][C][head_dim] bf16,
 * C = max_total_keys_hint rounded up to 128, plus 128 per request), then the
 * attention's block schedule. So the size follows the keys present, not
 * batch x the longest request. Depends only on these host-side sizes:
 *   max_seq_len_hint     a bound on every seq_len (>= 1; it sets the
 *                        schedule's cost buckets: scheduling only);
 *   max_total_keys_hint  a bound on the sum of the call's seq_lens; < 1: no
 *                        sum known, batch x max_seq_len_hint is used.
 * Returns 0 for invalid sizes.
 */
size_t pkv_extend_workspace_size(int32_t batch, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t max_seq_len_hint, int64_t max_total_keys_hint);

/*
 * Extend (chunked-prefill) attention ("Code Notes: mini-sglang", Scheduler
 * Layer table, PrefillManager row; "Introduction", Key Features, Chunked
 * Prefill and Radix Cache). Request r < batch owns queries qo_indptr[r] ..
 * qo_indptr[r+1]-1 of q (chunk length c_r); seq_lens[r] counts its cached
 * prefix plus the chunk, so the prefix is p_r = seq_lens[r] - c_r and the
 * chunk's keys are already stored (pkv_kv_store) at positions p_r .. p_r +
 * c_r - 1 of its row. Chunk query j attends to keys 0 .. p_r + j (full
 * prefix, causal within the chunk):
 *   o[t,h,:], lse[t,h] = attention of q[t,h,:] over those keys (as decode).
 * q, o: device bf16 [total_q, Hq, D], 16-byte aligned; lse: device fp32
 * [total_q, Hq] or NULL; qo_indptr: device int32 [batch + 1], qo_indptr[0]
 * = 0, non-decreasing, qo_indptr[batch] = total_q. Other tables as for
 * decode. max_seq_len_hint: a bound on every seq_len of the call (< 1: the
 * row capacity table_stride * page_size); it only sets how finely the
 * attention's blocks are sorted by cost, and a longer request is still
 * computed. max_total_keys_hint: a bound on the sum of the seq_lens (< 1:
 * batch x max_seq_len_hint); a request whose rounded-up keys, counted in
 * request order, would go past it is not computed (its outputs are
 * unspecified) and PKV_DEVERR_SEQ_LEN_RANGE is flagged, as it is for a
 * seq_len outside [0, table_stride * page_size]. workspace: device, 256-byte
 * aligned, at least pkv_extend_workspace_size(batch, Hkv, D,
 * max_seq_len_hint, max_total_keys_hint) bytes (with the same effective
 * bounds), contents irrelevant on entry.
 */
pkv_status pkv_paged_extend_attn(const pkv_pool *pool, int32_t layer, const void *q,
                                 const int32_t *qo_indptr, void *o, float *lse,
                                 const int32_t *page_table, int64_t table_stride,
                                 const int32_t *table_idx, const int32_t *seq_lens,
                                 int32_t batch, int32_t total_q, int32_t num_q_heads,
                                 float scale, int32_t max_seq_len_hint,
                                 int64_t max_total_keys_hint, void *workspace,
                                 size_t workspace_bytes, cudaStream_t stream);

/*
 * One extend step with store_kv fused in ("Code Notes: mini-sglang", Engine
 * Layer table, BaseKVCachePool row: the chunk's new K and V are written into
 * the pool, then attention reads the pool). k_new, v_new: device bf16
 * [total_q, Hkv, D], row t holding the new K / V of query token t
 * (kv_row_stride elements between tokens, 16-byte aligned, stride >= Hkv*D
 * and a multiple of 8). For each request r the rows qo_indptr[r] + j,
 * j < c_r, are stored at key position p_r + j of its page_table row (the slot
 * P * row[i/P] + i%P, i = p_r + j), and attention runs exactly as
 * pkv_paged_extend_attn with the same arguments and workspace. Equivalent
 * to pkv_kv_store with out_loc[qo_indptr[r] + j] = that slot followed by
 * pkv_paged_extend_attn, provided no other request's row of the call holds
 * those slots. A bad page id at a chunk position is flagged
 * (PKV_DEVERR_PAGE_RANGE) and that token is not stored; a request whose
 * qo_indptr pair is malformed (PKV_DEVERR_INDPTR) or whose keys go past the
 * bounds (PKV_DEVERR_SEQ_LEN_RANGE) stores nothing.
 */
pkv_status pkv_paged_extend_attn_store(const pkv_pool *pool, int32_t layer, const void *q,
                                       const void *k_new, const void *v_new,
                                       int64_t kv_row_stride, const int32_t *qo_indptr, void *o,
                                       float *lse, const int32_t *page_table,
                                       int64_t table_stride, const int32_t *table_idx,
                                       const int32_t *seq_lens, int32_t batch, int32_t total_q,
                                       int32_t num_q_heads, float scale,
                                       int32_t max_seq_len_hint, int64_t max_total_keys_hint,
                                       void *workspace, size_t workspace_bytes,
                                       cudaStream_t stream);

/*
 * Bytes of device workspace pkv_paged_cascade_decode_attn needs: fp32 partial
 * states per (request, q head), one per suffix split and one per key range
 * the shared prefixes are cut into. Depends only on these host-side sizes
 * (max_prefix_len_hint >= 1) and the device's SM count.
 */
size_t pkv_cascade_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t num_groups,
                                  int32_t max_prefix_len_hint, int32_t max_suffix_len_hint);

/*
 * Cascade decode over shared prefixes ("Introduction", Key Features, Radix
 * Cache: requests that share a prefix share its KV entries; "Code Notes:
 * mini-sglang", Scheduler Layer table, CacheManager row). Requests are
 * partitioned into groups: group k's members are requests
 * members[member_indptr[k]] .. members[member_indptr[k+1] - 1], and every
 * request is a member of exactly one group. Request b of group k attends,
 * as in pkv_paged_decode_attn, to the concatenation of
 *   the group's shared prefix: prefix_lens[k] keys of row k of
 *     prefix_page_table ([num_groups, prefix_table_stride] int32), then
 *   its own suffix: seq_lens[b] keys of row table_idx[b] (or b) of page_table,
 * i.e. o[b,h,:], lse[b,h] = attention of q[b,h,:] over those keys. The
 * prefix is attended once per group for all its members together (tensor
 * cores, one 128-row query tile per 128 / (Hq/Hkv) members and kv head, its
 * K/V read from the pool once per kv head), the suffix per request
 * (split-KV decode), and the states are merged by log-sum-exp. A group may have prefix_lens[k] = 0. Requires Hq/Hkv <= 8 and
 * Hkv in {1, 2} or a multiple of 4 (as decode). Tables and q/o/lse as for
 * decode; member_indptr: device int32 [num_groups + 1], member_indptr[0] = 0,
 * non-decreasing, member_indptr[num_groups] <= batch; members: device int32,
 * a permutation of 0 .. batch - 1 laid out by member_indptr (trusted: a
 * request in no group gets an unspecified result, one in two groups a racy
 * one; a member index outside the batch is skipped and flagged
 * PKV_DEVERR_INDPTR). max_prefix_len_hint: a bound on every prefix_lens
 * entry (< 1: the row capacity prefix_table_stride * page_size); with
 * max_suffix_len_hint it sets how the prefix is cut into key ranges (host
 * sizes only); a longer prefix is still computed. A prefix length outside
 * [0, prefix_table_stride * page_size] is flagged (PKV_DEVERR_SEQ_LEN_RANGE)
 * and its members get their suffix's attention alone. max_suffix_len_hint
 * sizes the suffix split plan as max_seq_len_hint does for decode. workspace:
 * device, 256-byte aligned, at least pkv_cascade_workspace_size(...) bytes
 * (with the same effective prefix bound). Every kernel runs on `stream`:
 * the shared-prefix kernel first, then the suffix decode, which starts as
 * soon as every prefix CTA is running and fills the SMs those leave free,
 * then the merge.
 */
pkv_status pkv_paged_cascade_decode_attn(
    const pkv_pool *pool, int32_t layer, const void *q, void *o, float *lse,
    const int32_t *prefix_page_table, int64_t prefix_table_stride, const int32_t *prefix_lens,
    const int32_t *member_indptr, const int32_t *members, int32_t num_groups,
    const int32_t *page_table, int64_t table_stride, const int32_t *table_idx,
    const int32_t *seq_lens, int32_t batch, int32_t num_q_heads, float scale,
    int32_t max_prefix_len_hint, int32_t max_suffix_len_hint, void *workspace,
    size_t workspace_bytes, cudaStream_t stream);

/*
 * Merge of two attention states over disjoint key sets (the log-sum-exp
 * combination split-KV decode uses internally, exported so callers can
 * compose attention over a shared prefix with attention over a private
 * suffix). For each row and head:
 *   lse = log(exp(lse_a) + exp(lse_b))
 *   o   = exp(lse_a - lse) * o_a + exp(lse_b - lse) * o_b
 * A state with lse = -inf contributes nothing; two such states give o = 0,
 * lse = -inf. o_a, o_b: device fp32 [rows, heads, head_dim]; lse_a, lse_b:
 * device fp32 [rows, heads]. o_out: device [rows, heads, head_dim], bf16 if
 * o_out_is_bf16 else fp32 (may alias o_a or o_b when fp32). lse_out: device
 * fp32 [rows, heads] or NULL (may alias lse_a or lse_b). head_dim must be a
 * multiple of 4 and every pointer 16-byte aligned (lse pointers 4-byte).
 */
pkv_status pkv_merge_lse(const float *o_a, const float *lse_a, const float *o_b,
                         const float *lse_b, void *o_out, int32_t o_out_is_bf16,
                         float *lse_out, int64_t rows, int32_t heads, int32_t head_dim,
                         cudaStream_t stream);

/*
 * Reads and clears the device error word of the current device (see the
 * PKV_DEVERR_* bits) into *flags. This call SYNCHRONISES the device: it is
 * a debugging aid, not part of the hot path.
 */
pkv_status pkv_read_device_errors(uint32_t *flags);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
