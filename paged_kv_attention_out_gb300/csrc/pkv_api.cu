// pkv_api.cu - the C ABI declared in include/pkv.h: argument validation,
// per-device facts (compute capability, SM count), the decode split plan,
// and the kernel launches. No call here allocates, synchronises (except
// pkv_read_device_errors, documented as a debugging aid) or changes the
// current device.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>

#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

thread_local char g_last_error[256] = "";

// Device error word (PKV_DEVERR_* bits), one per device that loads the library.
__device__ unsigned int g_device_errors;

struct DevInfo {
  bool init = false;
  pkv_status status = PKV_OK;
  int sm_count = 0;
  unsigned *err = nullptr;
};

constexpr int kMaxDevices = 64;
DevInfo g_dev[kMaxDevices];
std::mutex g_mu;

pkv_status fail(pkv_status s, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return s;
}

pkv_status cuda_fail(cudaError_t e, const char *what) {
  return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Facts about the current device, computed once per device.
pkv_status device_info(DevInfo **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PKV_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  DevInfo &d = g_dev[dev];
  if (!d.init) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3) {
      d.status = PKV_ERR_UNSUPPORTED;
    } else {
      void *p = nullptr;
      if ((e = cudaGetSymbolAddress(&p, g_device_errors)) != cudaSuccess)
        return cuda_fail(e, "cudaGetSymbolAddress(device error word)");
      d.err = static_cast<unsigned *>(p);
      d.status = PKV_OK;
    }
    d.sm_count = sms;
    d.init = true;
  }
  if (d.status != PKV_OK)
    return fail(d.status, "device %d is not compute capability 10.3 (sm_103a)", dev);
  *out = &d;
  return PKV_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

pkv_status check_pool(const pkv_pool *pool, int32_t layer, pkv::PoolGeom *g) {
  if (!pool) return fail(PKV_ERR_INVALID_ARG, "pool is NULL");
  if (!pool->base) return fail(PKV_ERR_INVALID_ARG, "pool->base is NULL");
  if (!aligned(pool->base, 16)) return fail(PKV_ERR_INVALID_ARG, "pool->base not 16-byte aligned");
  if (pool->num_layers <= 0 || pool->num_pages <= 0 || pool->page_size <= 0 ||
      pool->num_kv_heads <= 0)
    return fail(PKV_ERR_INVALID_ARG, "pool sizes must be positive");
  if (pool->head_dim != 64 && pool->head_dim != 128)
    return fail(PKV_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", pool->head_dim);
  if (layer < 0 || layer >= pool->num_layers)
    return fail(PKV_ERR_INVALID_ARG, "layer %d outside [0, %d)", layer, pool->num_layers);
  const int64_t slots = pool->num_pages * static_cast<int64_t>(pool->page_size);
  if (slots / pool->page_size != pool->num_pages || slots > (int64_t(1) << 40))
    return fail(PKV_ERR_INVALID_ARG, "pool too large");
  g->base = pool->base;
  g->slots = slots;
  g->plane = slots * pool->num_kv_heads * pool->head_dim;
  g->num_layers = pool->num_layers;
  g->page_size = pool->page_size;
  g->hkv = pool->num_kv_heads;
  g->d = pool->head_dim;
  return PKV_OK;
}

int32_t effective_hint(int32_t hint) { return hint < 1 ? 1 : hint; }

}  // namespace

namespace pkv {
pkv_status fail_status(pkv_status s, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return s;
}
}  // namespace pkv

extern "C" {

pkv_status pkv_init(void) {
  DevInfo *d = nullptr;
  return device_info(&d);
}

const char *pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
    case PKV_ERR_WORKSPACE_TOO_SMALL: return "PKV_ERR_WORKSPACE_TOO_SMALL";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
  }
  return "PKV_UNKNOWN_STATUS";
}

const char *pkv_last_error(void) { return g_last_error; }

pkv_status pkv_kv_store(const pkv_pool *pool, int32_t layer, const void *k, const void *v,
                        int64_t kv_row_stride, const int32_t *out_loc, int64_t num_tokens,
                        cudaStream_t stream) {
  pkv::PoolGeom g;
  pkv_status s = check_pool(pool, layer, &g);
  if (s != PKV_OK) return s;
  if (num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "num_tokens < 0");
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !out_loc) return fail(PKV_ERR_INVALID_ARG, "k, v and out_loc must be non-NULL");
  if (!aligned(k, 16) || !aligned(v, 16))
    return fail(PKV_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
  if (!aligned(out_loc, 4)) return fail(PKV_ERR_INVALID_ARG, "out_loc must be 4-byte aligned");
  if (kv_row_stride < static_cast<int64_t>(g.hkv) * g.d || kv_row_stride % 8 != 0)
    return fail(PKV_ERR_INVALID_ARG, "kv_row_stride %lld must be >= Hkv*D and a multiple of 8",
                static_cast<long long>(kv_row_stride));
  DevInfo *d = nullptr;
  if ((s = device_info(&d)) != PKV_OK) return s;
  cudaError_t e = pkv::launch_kv_store(g, layer, k, v, kv_row_stride, out_loc, num_tokens,
                                       d->sm_count, d->err, stream);
  return e == cudaSuccess ? PKV_OK : cuda_fail(e, "kv_store launch");
}

size_t pkv_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t max_seq_len_hint) {
  if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      num_q_heads % num_kv_heads != 0)
    return 0;
  DevInfo *d = nullptr;
  if (device_info(&d) != PKV_OK) return 0;
  return pkv::plan_decode(batch, num_q_heads, num_kv_heads, head_dim,
                          effective_hint(max_seq_len_hint), d->sm_count)
      .workspace_bytes;
}

// Decode, optionally with the step's new key / value rows stored first
// (k_new != NULL: the fused store of pkv_paged_decode_attn_store).
static pkv_status decode_call(const pkv_pool *pool, int32_t layer, const void *q,
                              const void *k_new, const void *v_new, int64_t kv_row_stride,
                              void *o, float *lse, const int32_t *page_table,
                              int64_t table_stride, const int32_t *table_idx,
                              const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                              float scale, int32_t max_seq_len_hint, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
  pkv::PoolGeom g;
  pkv_status s = check_pool(pool, layer, &g);
  if (s != PKV_OK) return s;
  if (batch < 0) return fail(PKV_ERR_INVALID_ARG, "batch < 0");
  if (num_q_heads <= 0 || num_q_heads % g.hkv != 0)
    return fail(PKV_ERR_INVALID_ARG, "num_q_heads %d is not a positive multiple of Hkv %d",
                num_q_heads, g.hkv);
  const int group = num_q_heads / g.hkv;
  if (group > 8) return fail(PKV_ERR_UNSUPPORTED, "decode supports Hq/Hkv <= 8, got %d", group);
  if (g.hkv < 4 ? (4 % g.hkv != 0) : (g.hkv % 4 != 0))
    return fail(PKV_ERR_UNSUPPORTED, "decode supports Hkv in {1, 2} or a multiple of 4, got %d",
                g.hkv);
  if (batch > 65535) return fail(PKV_ERR_UNSUPPORTED, "decode batch %d > 65535", batch);
  if (table_stride <= 0) return fail(PKV_ERR_INVALID_ARG, "table_stride must be positive");
  if (!isfinite(scale)) return fail(PKV_ERR_INVALID_ARG, "scale is not finite");
  if (batch == 0) return PKV_OK;
  if (!q || !o || !page_table || !seq_lens)
    return fail(PKV_ERR_INVALID_ARG, "q, o, page_table and seq_lens must be non-NULL");
  if (!aligned(q, 16) || !aligned(o, 16))
    return fail(PKV_ERR_INVALID_ARG, "q and o must be 16-byte aligned");
  if (!aligned(page_table, 4) || !aligned(seq_lens, 4) || !aligned(lse, 4) ||
      !aligned(table_idx, 4))
    return fail(PKV_ERR_INVALID_ARG, "int32/fp32 tables must be 4-byte aligned");
  DevInfo *d = nullptr;
  if ((s = device_info(&d)) != PKV_OK) return s;
  const pkv::DecodePlan plan = pkv::plan_decode(batch, num_q_heads, g.hkv, g.d,
                                                effective_hint(max_seq_len_hint), d->sm_count);
  if (plan.workspace_bytes > 0) {
    if (!workspace)
      return fail(PKV_ERR_WORKSPACE_TOO_SMALL, "workspace is NULL, %zu bytes needed",
                  plan.workspace_bytes);
    if (workspace_bytes < plan.workspace_bytes)
      return fail(PKV_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes, %zu needed", workspace_bytes,
                  plan.workspace_bytes);
    if (!aligned(workspace, 256))
      return fail(PKV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  }
  cudaError_t e = pkv::launch_decode(g, layer, q, o, lse, page_table, table_stride, table_idx,
                                     seq_lens, batch, num_q_heads, scale, plan, workspace, d->err,
                                     stream, k_new, v_new, kv_row_stride);
  return e == cudaSuccess ? PKV_OK : cuda_fail(e, "decode launch");
}

pkv_status pkv_paged_decode_attn(const pkv_pool *pool, int32_t layer, const void *q, void *o,
                                 float *lse, const int32_t *page_table, int64_t table_stride,
                                 const int32_t *table_idx, const int32_t *seq_lens,
                                 int32_t batch, int32_t num_q_heads, float scale,
                                 int32_t max_seq_len_hint, void *workspace,
                                 size_t workspace_bytes, cudaStream_t stream) {
  return decode_call(pool, layer, q, nullptr, nullptr, 0, o, lse, page_table, table_stride,
                     table_idx, seq_lens, batch, num_q_heads, scale, max_seq_len_hint, workspace,
                     workspace_bytes, stream);
}

pkv_status pkv_paged_decode_attn_store(const pkv_pool *pool, int32_t layer, const void *q,
                                       const void *k_new, const void *v_new,
                                       int64_t kv_row_stride, void *o, float *lse,
                                       const int32_t *page_table, int64_t table_stride,
                                       const int32_t *table_idx, const int32_t *seq_lens,
                                       int32_t batch, int32_t num_q_heads, float scale,
                                       int32_t max_seq_len_hint, void *workspace,
                                       size_t workspace_bytes, cudaStream_t stream) {
  if (batch > 0) {
    if (!k_new || !v_new) return fail(PKV_ERR_INVALID_ARG, "k_new and v_new must be non-NULL");
    if (!aligned(k_new, 16) || !aligned(v_new, 16))
      return fail(PKV_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
    if (pool && (kv_row_stride < static_cast<int64_t>(pool->num_kv_heads) * pool->head_dim ||
                 kv_row_stride % 8 != 0))
      return fail(PKV_ERR_INVALID_ARG, "kv_row_stride %lld must be >= Hkv*D and a multiple of 8",
                  static_cast<long long>(kv_row_stride));
  }
  return decode_call(pool, layer, q, batch > 0 ? k_new : nullptr, v_new, kv_row_stride, o, lse,
                     page_table, table_stride, table_idx, seq_lens, batch, num_q_heads, scale,
                     max_seq_len_hint, workspace, workspace_bytes, stream);
}

static size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

size_t pkv_cascade_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t num_groups,
                                  int32_t max_prefix_len_hint, int32_t max_suffix_len_hint) {
  if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || num_groups <= 0 ||
      num_q_heads % num_kv_heads != 0 || max_prefix_len_hint < 1)
    return 0;
  DevInfo *d = nullptr;
  if (device_info(&d) != PKV_OK) return 0;
  const pkv::DecodePlan plan = pkv::plan_cascade_suffix(
      batch, num_q_heads, num_kv_heads, head_dim, effective_hint(max_suffix_len_hint), d->sm_count);
  const int32_t ks = pkv::cascade_prefix_splits(batch, num_q_heads, num_kv_heads, num_groups,
                                                max_prefix_len_hint, max_suffix_len_hint,
                                                d->sm_count);
  return align256(pkv::cascade_partial_bytes(batch, num_q_heads, head_dim, plan.splits + ks));
}

pkv_status pkv_paged_cascade_decode_attn(
    const pkv_pool *pool, int32_t layer, const void *q, void *o, float *lse,
    const int32_t *prefix_page_table, int64_t prefix_table_stride, const int32_t *prefix_lens,
    const int32_t *member_indptr, const int32_t *members, int32_t num_groups,
    const int32_t *page_table, int64_t table_stride, const int32_t *table_idx,
    const int32_t *seq_lens, int32_t batch, int32_t num_q_heads, float scale,
    int32_t max_prefix_len_hint, int32_t max_suffix_len_hint, void *workspace,
    size_t workspace_bytes, cudaStream_t stream) {
  pkv::PoolGeom g;
  pkv_status s = check_pool(pool, layer, &g);
  if (s != PKV_OK) return s;
  if (batch < 0 || num_groups < 0) return fail(PKV_ERR_INVALID_ARG, "batch and num_groups must be >= 0");
  if (num_q_heads <= 0 || num_q_heads % g.hkv != 0)
    return fail(PKV_ERR_INVALID_ARG, "num_q_heads %d is not a positive multiple of Hkv %d",
                num_q_heads, g.hkv);
  const int group = num_q_heads / g.hkv;
  if (group > 8) return fail(PKV_ERR_UNSUPPORTED, "cascade decode supports Hq/Hkv <= 8, got %d", group);
  if (g.hkv < 4 ? (4 % g.hkv != 0) : (g.hkv % 4 != 0))
    return fail(PKV_ERR_UNSUPPORTED, "decode supports Hkv in {1, 2} or a multiple of 4, got %d",
                g.hkv);
  if (batch > 65535 || num_groups >= 65535)
    return fail(PKV_ERR_UNSUPPORTED, "cascade decode: batch %d or groups %d too large", batch,
                num_groups);
  if (table_stride <= 0 || prefix_table_stride <= 0)
    return fail(PKV_ERR_INVALID_ARG, "table strides must be positive");
  if (!isfinite(scale)) return fail(PKV_ERR_INVALID_ARG, "scale is not finite");
  if (batch == 0) return PKV_OK;
  if (num_groups == 0)
    return fail(PKV_ERR_INVALID_ARG, "cascade decode needs every request in a group (num_groups 0)");
  if (!q || !o || !page_table || !seq_lens || !prefix_page_table || !prefix_lens ||
      !member_indptr || !members)
    return fail(PKV_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned(q, 16) || !aligned(o, 16))
    return fail(PKV_ERR_INVALID_ARG, "q and o must be 16-byte aligned");
  if (!aligned(page_table, 4) || !aligned(seq_lens, 4) || !aligned(lse, 4) ||
      !aligned(table_idx, 4) || !aligned(prefix_page_table, 4) || !aligned(prefix_lens, 4) ||
      !aligned(member_indptr, 4) || !aligned(members, 4))
    return fail(PKV_ERR_INVALID_ARG, "int32/fp32 tables must be 4-byte aligned");
  const int64_t prefix_row_capacity = prefix_table_stride * g.page_size;
  int64_t pcap = max_prefix_len_hint >= 1 ? max_prefix_len_hint : prefix_row_capacity;
  if (pcap > prefix_row_capacity) pcap = prefix_row_capacity;
  if (pcap > (int64_t(1) << 30)) pcap = int64_t(1) << 30;
  if (static_cast<int64_t>(pkv::cascade_prefix_blocks(batch, num_q_heads, g.hkv, num_groups)) >
      65535)
    return fail(PKV_ERR_UNSUPPORTED, "cascade: too many member blocks in one call");
  DevInfo *d = nullptr;
  if ((s = device_info(&d)) != PKV_OK) return s;
  const pkv::DecodePlan plan = pkv::plan_cascade_suffix(
      batch, num_q_heads, g.hkv, g.d, effective_hint(max_suffix_len_hint), d->sm_count);
  const int32_t ks = pkv::cascade_prefix_splits(batch, num_q_heads, g.hkv, num_groups,
                                                static_cast<int32_t>(pcap), max_suffix_len_hint,
                                                d->sm_count);
  const int32_t slots = plan.splits + ks;
  const size_t need = align256(pkv::cascade_partial_bytes(batch, num_q_heads, g.d, slots));
  if (!workspace)
    return fail(PKV_ERR_WORKSPACE_TOO_SMALL, "workspace is NULL, %zu bytes needed", need);
  if (workspace_bytes < need)
    return fail(PKV_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes, %zu needed", workspace_bytes,
                need);
  if (!aligned(workspace, 256)) return fail(PKV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  float *part_o = nullptr, *part_lse = nullptr;
  pkv::cascade_partial_ptrs(workspace, batch, num_q_heads, g.d, slots, &part_o, &part_lse);
  // All on `stream`, in this order:
  // 1. the shared-prefix states of every member (slots splits .. splits +
  //    ks - 1): each group's prefix once per kv head and key range, K/V read
  //    from the pool by the tensor-core prefix kernel;
  cudaError_t e = pkv::launch_cascade_prefix(
      g, layer, q, prefix_page_table, prefix_table_stride, prefix_lens, member_indptr, members,
      num_groups, batch, num_q_heads, scale, part_o, part_lse, slots, plan.splits, ks, d->err,
      stream);
  if (e != cudaSuccess) return cuda_fail(e, "cascade prefix launch");
  // 2. the suffix partial states (slots 0 .. splits - 1): split-KV decode,
  //    started as soon as every prefix CTA is running (it reads nothing the
  //    prefix kernel writes; its last request's split-0 CTAs wait for that
  //    kernel at their exit, so this grid completes after it);
  float *po = nullptr, *pl = nullptr;
  e = pkv::launch_cascade_suffix(g, layer, q, o, lse, page_table, table_stride, table_idx,
                                 seq_lens, batch, num_q_heads, scale, plan, ks, workspace, d->err,
                                 stream, &po, &pl);
  if (e != cudaSuccess) return cuda_fail(e, "cascade suffix launch");
  // 3. the merge of every request's suffix splits and prefix states.
  e = pkv::launch_cascade_merge(g, layer, q, o, lse, page_table, table_stride, table_idx,
                                seq_lens, batch, num_q_heads, scale, plan, ks, part_o, part_lse,
                                d->err, stream);
  return e == cudaSuccess ? PKV_OK : cuda_fail(e, "cascade merge launch");
}

size_t pkv_extend_workspace_size(int32_t batch, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t max_seq_len_hint, int64_t max_total_keys_hint) {
  if (batch <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_seq_len_hint < 1) return 0;
  return pkv::extend_layout(batch, num_kv_heads, head_dim, max_seq_len_hint, max_total_keys_hint)
      .total_bytes;
}

// Extend with (k_new != NULL) or without the fused store of the chunk's K/V.
static pkv_status extend_call(const pkv_pool *pool, int32_t layer, const void *q,
                              const void *k_new, const void *v_new, int64_t kv_row_stride,
                              const int32_t *qo_indptr, void *o, float *lse,
                              const int32_t *page_table, int64_t table_stride,
                              const int32_t *table_idx, const int32_t *seq_lens, int32_t batch,
                              int32_t total_q, int32_t num_q_heads, float scale,
                              int32_t max_seq_len_hint, int64_t max_total_keys_hint,
                              void *workspace, size_t workspace_bytes, cudaStream_t stream) {
  pkv::PoolGeom g;
  pkv_status s = check_pool(pool, layer, &g);
  if (s != PKV_OK) return s;
  if (batch < 0 || total_q < 0) return fail(PKV_ERR_INVALID_ARG, "batch and total_q must be >= 0");
  if (num_q_heads <= 0 || num_q_heads % g.hkv != 0)
    return fail(PKV_ERR_INVALID_ARG, "num_q_heads %d is not a positive multiple of Hkv %d",
                num_q_heads, g.hkv);
  const int group = num_q_heads / g.hkv;
  if (group > 16) return fail(PKV_ERR_UNSUPPORTED, "extend supports Hq/Hkv <= 16, got %d", group);
  if (batch >= 65535) return fail(PKV_ERR_UNSUPPORTED, "extend supports batch < 65535");
  if (g.hkv > 65535) return fail(PKV_ERR_UNSUPPORTED, "too many kv heads");
  if (table_stride <= 0) return fail(PKV_ERR_INVALID_ARG, "table_stride must be positive");
  if (!isfinite(scale)) return fail(PKV_ERR_INVALID_ARG, "scale is not finite");
  if (batch == 0 || total_q == 0) return PKV_OK;
  if (!q || !o || !qo_indptr || !page_table || !seq_lens)
    return fail(PKV_ERR_INVALID_ARG, "q, o, qo_indptr, page_table and seq_lens must be non-NULL");
  if (!aligned(q, 16) || !aligned(o, 16))
    return fail(PKV_ERR_INVALID_ARG, "q and o must be 16-byte aligned");
  if (!aligned(page_table, 4) || !aligned(seq_lens, 4) || !aligned(lse, 4) ||
      !aligned(table_idx, 4) || !aligned(qo_indptr, 4))
    return fail(PKV_ERR_INVALID_ARG, "int32/fp32 tables must be 4-byte aligned");
  const int64_t row_capacity = table_stride * g.page_size;
  int64_t cap = max_seq_len_hint >= 1 ? max_seq_len_hint : row_capacity;
  if (cap > row_capacity) cap = row_capacity;
  if (cap > (int64_t(1) << 30)) return fail(PKV_ERR_UNSUPPORTED, "sequence capacity too large");
  if (max_total_keys_hint > (int64_t(1) << 40))
    return fail(PKV_ERR_UNSUPPORTED, "max_total_keys_hint too large");
  const pkv::ExtendLayout lay = pkv::extend_layout(batch, g.hkv, g.d, cap, max_total_keys_hint);
  if (2 * g.hkv * lay.cap_rows >= (int64_t(1) << 31) || lay.max_blocks >= (int64_t(1) << 28))
    return fail(PKV_ERR_UNSUPPORTED, "extend: kv heads x key bound too large (%lld rows)",
                static_cast<long long>(2 * g.hkv * lay.cap_rows));
  const size_t need = lay.total_bytes;
  if (!workspace)
    return fail(PKV_ERR_WORKSPACE_TOO_SMALL, "workspace is NULL, %zu bytes needed", need);
  if (workspace_bytes < need)
    return fail(PKV_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes, %zu needed", workspace_bytes,
                need);
  if (!aligned(workspace, 256)) return fail(PKV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const int64_t tpc = 2 * (128 / group);  // chunk tokens per CTA (two 128-row query tiles)
  if ((static_cast<int64_t>(total_q) + tpc - 1) / tpc + batch > 65535)
    return fail(PKV_ERR_UNSUPPORTED, "extend: too many query tiles in one call");
  DevInfo *d = nullptr;
  if ((s = device_info(&d)) != PKV_OK) return s;
  pkv::ExtendMode mode;
  mode.k_new = k_new;
  mode.v_new = v_new;
  mode.kv_row_stride = kv_row_stride;
  cudaError_t e = pkv::launch_extend(g, layer, q, qo_indptr, o, lse, page_table, table_stride,
                                     table_idx, seq_lens, batch, total_q, num_q_heads, scale, lay,
                                     workspace, d->sm_count, d->err, stream, mode);
  return e == cudaSuccess ? PKV_OK : cuda_fail(e, "extend launch");
}

pkv_status pkv_paged_extend_attn(const pkv_pool *pool, int32_t layer, const void *q,
                                 const int32_t *qo_indptr, void *o, float *lse,
                                 const int32_t *page_table, int64_t table_stride,
                                 const int32_t *table_idx, const int32_t *seq_lens,
                                 int32_t batch, int32_t total_q, int32_t num_q_heads,
                                 float scale, int32_t max_seq_len_hint,
                                 int64_t max_total_keys_hint, void *workspace,
                                 size_t workspace_bytes, cudaStream_t stream) {
  return extend_call(pool, layer, q, nullptr, nullptr, 0, qo_indptr, o, lse, page_table,
                     table_stride, table_idx, seq_lens, batch, total_q, num_q_heads, scale,
                     max_seq_len_hint, max_total_keys_hint, workspace, workspace_bytes, stream);
}

pkv_status pkv_paged_extend_attn_store(const pkv_pool *pool, int32_t layer, const void *q,
                                       const void *k_new, const void *v_new,
                                       int64_t kv_row_stride, const int32_t *qo_indptr, void *o,
                                       float *lse, const int32_t *page_table,
                                       int64_t table_stride, const int32_t *table_idx,
                                       const int32_t *seq_lens, int32_t batch, int32_t total_q,
                                       int32_t num_q_heads, float scale,
                                       int32_t max_seq_len_hint, int64_t max_total_keys_hint,
                                       void *workspace, size_t workspace_bytes,
                                       cudaStream_t stream) {
  if (batch > 0 && total_q > 0) {
    if (!k_new || !v_new) return fail(PKV_ERR_INVALID_ARG, "k_new and v_new must be non-NULL");
    if (!aligned(k_new, 16) || !aligned(v_new, 16))
      return fail(PKV_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
    if (pool && (kv_row_stride < static_cast<int64_t>(pool->num_kv_heads) * pool->head_dim ||
                 kv_row_stride % 8 != 0))
      return fail(PKV_ERR_INVALID_ARG, "kv_row_stride %lld must be >= Hkv*D and a multiple of 8",
                  static_cast<long long>(kv_row_stride));
  }
  return extend_call(pool, layer, q, batch > 0 && total_q > 0 ? k_new : nullptr, v_new,
                     kv_row_stride, qo_indptr, o, lse, page_table, table_stride, table_idx,
                     seq_lens, batch, total_q, num_q_heads, scale, max_seq_len_hint,
                     max_total_keys_hint, workspace, workspace_bytes, stream);
}

pkv_status pkv_merge_lse(const float *o_a, const float *lse_a, const float *o_b,
                         const float *lse_b, void *o_out, int32_t o_out_is_bf16,
                         float *lse_out, int64_t rows, int32_t heads, int32_t head_dim,
                         cudaStream_t stream) {
  if (rows < 0 || heads <= 0 || head_dim <= 0 || head_dim % 4 != 0)
    return fail(PKV_ERR_INVALID_ARG, "rows >= 0, heads > 0 and head_dim a positive multiple of 4");
  if (rows == 0) return PKV_OK;
  if (!o_a || !lse_a || !o_b || !lse_b || !o_out)
    return fail(PKV_ERR_INVALID_ARG, "o_a, lse_a, o_b, lse_b and o_out must be non-NULL");
  if (!aligned(o_a, 16) || !aligned(o_b, 16) || !aligned(o_out, 16))
    return fail(PKV_ERR_INVALID_ARG, "o pointers must be 16-byte aligned");
  if (!aligned(lse_a, 4) || !aligned(lse_b, 4) || !aligned(lse_out, 4))
    return fail(PKV_ERR_INVALID_ARG, "lse pointers must be 4-byte aligned");
  DevInfo *d = nullptr;
  pkv_status s = device_info(&d);
  if (s != PKV_OK) return s;
  cudaError_t e = pkv::launch_merge(o_a, lse_a, o_b, lse_b, o_out, o_out_is_bf16 != 0, lse_out,
                                    rows, heads, head_dim, d->sm_count, stream);
  return e == cudaSuccess ? PKV_OK : cuda_fail(e, "merge launch");
}

pkv_status pkv_read_device_errors(uint32_t *flags) {
  if (!flags) return fail(PKV_ERR_INVALID_ARG, "flags is NULL");
  DevInfo *d = nullptr;
  pkv_status s = device_info(&d);
  if (s != PKV_OK) return s;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  unsigned v = 0;
  if ((e = cudaMemcpyFromSymbol(&v, g_device_errors, sizeof v)) != cudaSuccess)
    return cuda_fail(e, "read device error word");
  const unsigned zero = 0;
  if ((e = cudaMemcpyToSymbol(g_device_errors, &zero, sizeof zero)) != cudaSuccess)
    return cuda_fail(e, "clear device error word");
  *flags = v;
  return PKV_OK;
}

}  // extern "C"
