// pkv_internal.h - launchers shared between the C ABI (pkv_api.cu) and the
// kernel translation units. Arguments arrive here already validated.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// Pool geometry as the kernels use it.
struct PoolGeom {
  const void *base;   // bf16 pool
  int64_t plane;      // elements of one (c, layer) plane: num_pages * page_size * Hkv * D
  int64_t slots;      // num_pages * page_size
  int32_t num_layers;
  int32_t page_size;
  int32_t hkv;
  int32_t d;
};

struct DecodePlan {
  int32_t heads_per_cta;   // kv heads one CTA covers
  int32_t warps_per_head;  // warps that share one kv head's keys
  int32_t head_groups;     // Hkv / heads_per_cta
  int32_t chunk;           // keys per split (multiple of 16)
  int32_t splits;          // splits per request (grid.y)
  size_t workspace_bytes;  // 0 when splits == 1
};

DecodePlan plan_decode(int32_t batch, int32_t hq, int32_t hkv, int32_t d, int32_t max_seq_len,
                       int32_t sm_count);

cudaError_t launch_kv_store(const PoolGeom &g, int32_t layer, const void *k, const void *v,
                            int64_t row_stride, const int32_t *out_loc, int64_t n,
                            int32_t sm_count, unsigned *err, cudaStream_t stream);

cudaError_t launch_decode(const PoolGeom &g, int32_t layer, const void *q, void *o, float *lse,
                          const int32_t *page_table, int64_t table_stride,
                          const int32_t *table_idx, const int32_t *seq_lens, int32_t batch,
                          int32_t hq, float scale, const DecodePlan &plan, void *workspace,
                          unsigned *err, cudaStream_t stream, const void *k_new = nullptr,
                          const void *v_new = nullptr, int64_t kv_row_stride = 0);

// Cascade decode: suffix partial states for split slots 0 .. splits - 1 of
// [B, Hq, splits + 1] (decode_kernel, always partial), then the merge of those
// with slot `splits`, the shared-prefix state written by the extend kernel.
size_t cascade_partial_bytes(int32_t batch, int32_t hq, int32_t d, int32_t slots);
// Key ranges the shared prefix of a cascade is cut into, from host sizes only.
int32_t cascade_prefix_splits(int32_t batch, int32_t hq, int32_t hkv, int32_t num_groups,
                              int32_t max_prefix, int32_t sm_count);
cudaError_t launch_cascade_suffix(const PoolGeom &g, int32_t layer, const void *q, void *o,
                                  float *lse, const int32_t *page_table, int64_t table_stride,
                                  const int32_t *table_idx, const int32_t *seq_lens,
                                  int32_t batch, int32_t hq, float scale, const DecodePlan &plan,
                                  int32_t prefix_slots, void *partials, unsigned *err,
                                  cudaStream_t stream, float **part_o, float **part_lse);
cudaError_t launch_cascade_merge(const PoolGeom &g, int32_t layer, const void *q, void *o,
                                 float *lse, const int32_t *page_table, int64_t table_stride,
                                 const int32_t *table_idx, const int32_t *seq_lens, int32_t batch,
                                 int32_t hq, float scale, const DecodePlan &plan,
                                 int32_t prefix_slots, float *part_o, float *part_lse,
                                 unsigned *err, cudaStream_t stream);

// Where the extend kernel's queries come from and where its results go. The
// defaults are the extend call: chunk token t of request r is q row
// qo_indptr[r] + t, causal, bf16 o and lse. The cascade's shared-prefix
// attention sets members (token t of group r is request members[qo_indptr[r]
// + t]), causal = 0 (every member sees all seq_lens[r] prefix keys) and
// writes fp32 partial states into slot `pslot` of [B, Hq, pstride].
struct ExtendMode {
  int32_t causal = 1;
  const int32_t *members = nullptr;
  float *part_o = nullptr;
  float *part_lse = nullptr;
  int32_t pstride = 0;
  int32_t pslot = 0;
  int32_t key_splits = 1;  // non-causal: key ranges per block (slots pslot .. + key_splits - 1)
  // causal only: store_kv fused into the gather (chunk rows of k_new / v_new,
  // kv_row_stride elements apart, written into the pool at their slots)
  const void *k_new = nullptr;
  const void *v_new = nullptr;
  int64_t kv_row_stride = 0;
  // the gather reads nothing the previous kernel on the stream writes: it
  // may run beside that kernel (its dependency wait moves to its exit)
  int32_t overlap_previous = 0;
};

// Gathered-K/V workspace of the extend call: [2][batch][hkv][s_pad][d] bf16,
// s_pad = capacity rounded up to 128.
int64_t extend_s_pad(int32_t capacity);
size_t extend_workspace_bytes(int32_t batch, int32_t hkv, int32_t d, int32_t capacity);

cudaError_t launch_extend(const PoolGeom &g, int32_t layer, const void *q,
                          const int32_t *qo_indptr, void *o, float *lse,
                          const int32_t *page_table, int64_t table_stride,
                          const int32_t *table_idx, const int32_t *seq_lens, int32_t batch,
                          int32_t total_q, int32_t hq, float scale, int32_t capacity,
                          void *workspace, int32_t sm_count, unsigned *err, cudaStream_t stream,
                          const ExtendMode &mode = ExtendMode());

cudaError_t launch_merge(const float *o_a, const float *lse_a, const float *o_b,
                         const float *lse_b, void *o_out, bool out_bf16, float *lse_out,
                         int64_t rows, int32_t heads, int32_t head_dim, int32_t sm_count,
                         cudaStream_t stream);

// Records a one-line reason for pkv_last_error() and returns s.
pkv_status fail_status(pkv_status s, const char *fmt, ...);

}  // namespace pkv
