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
  int32_t sm_count;        // of the device the plan was made for
};

DecodePlan plan_decode(int32_t batch, int32_t hq, int32_t hkv, int32_t d, int32_t max_seq_len,
                       int32_t sm_count);
// The split plan of a cascade's suffix decode (host scalars only).
DecodePlan plan_cascade_suffix(int32_t batch, int32_t hq, int32_t hkv, int32_t d,
                               int32_t max_seq_len, int32_t sm_count);

cudaError_t launch_kv_store(const PoolGeom &g, int32_t layer, const void *k, const void *v,
                            int64_t row_stride, const int32_t *out_loc, int64_t n,
                            int32_t sm_count, unsigned *err, cudaStream_t stream);

cudaError_t launch_decode(const PoolGeom &g, int32_t layer, const void *q, void *o, float *lse,
                          const int32_t *page_table, int64_t table_stride,
                          const int32_t *table_idx, const int32_t *seq_lens, int32_t batch,
                          int32_t hq, float scale, const DecodePlan &plan, void *workspace,
                          unsigned *err, cudaStream_t stream, const void *k_new = nullptr,
                          const void *v_new = nullptr, int64_t kv_row_stride = 0);

// Cascade decode: the shared-prefix states of every member (cascade.cu,
// slots splits .. splits + key ranges - 1 of [B, Hq, slots]), the suffix
// partial states in slots 0 .. splits - 1 (decode_kernel, always partial),
// then the merge of all of them per (request, q head).
size_t cascade_partial_bytes(int32_t batch, int32_t hq, int32_t d, int32_t slots);
void cascade_partial_ptrs(void *partials, int32_t batch, int32_t hq, int32_t d, int32_t slots,
                          float **part_o, float **part_lse);
// Key ranges the shared prefix of a cascade is cut into, from host sizes only.
int32_t cascade_prefix_splits(int32_t batch, int32_t hq, int32_t hkv, int32_t num_groups,
                              int32_t max_prefix, int32_t max_suffix, int32_t sm_count);
// Upper bound on the shared-prefix CTAs per (kv head, key range): member
// blocks of 128 / (Hq / Hkv) members, cut per group.
int32_t cascade_prefix_blocks(int32_t batch, int32_t hq, int32_t hkv, int32_t num_groups);
cudaError_t launch_cascade_prefix(const PoolGeom &g, int32_t layer, const void *q,
                                  const int32_t *prefix_table, int64_t prefix_stride,
                                  const int32_t *prefix_lens, const int32_t *member_indptr,
                                  const int32_t *members, int32_t num_groups, int32_t batch,
                                  int32_t hq, float scale, float *part_o, float *part_lse,
                                  int32_t pstride, int32_t pslot, int32_t key_splits,
                                  unsigned *err, cudaStream_t stream);
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

// Options of the extend call: store_kv fused into the gather (the chunk's
// rows of k_new / v_new, kv_row_stride elements apart, are written into the
// pool at their slots and attended in the same call).
struct ExtendMode {
  const void *k_new = nullptr;
  const void *v_new = nullptr;
  int64_t kv_row_stride = 0;
};

// Workspace of the extend call, from host scalars only: the gathered K/V
// runs ([2][Hkv][cap_rows][D] bf16, every request's keys rounded up to 128,
// back to back in request order), then (256-byte aligned) the block schedule
// and the run offsets.
struct ExtendLayout {
  int64_t cap_rows;     // rows of one (K or V, kv head) region
  int64_t nbuck;        // cost buckets of the block schedule
  int64_t max_blocks;   // bound on the schedule's blocks
  uint64_t kv_bytes;
  uint64_t plan_offset;
  uint64_t total_bytes;
};
// max_seq: a bound on every seq_len (sets the schedule's cost buckets);
// max_total_keys: a bound on their sum (< 1: batch x max_seq).
ExtendLayout extend_layout(int32_t batch, int32_t hkv, int32_t d, int64_t max_seq,
                           int64_t max_total_keys);

cudaError_t launch_extend(const PoolGeom &g, int32_t layer, const void *q,
                          const int32_t *qo_indptr, void *o, float *lse,
                          const int32_t *page_table, int64_t table_stride,
                          const int32_t *table_idx, const int32_t *seq_lens, int32_t batch,
                          int32_t total_q, int32_t hq, float scale, const ExtendLayout &lay,
                          void *workspace, int32_t sm_count, unsigned *err, cudaStream_t stream,
                          const ExtendMode &mode = ExtendMode());

cudaError_t launch_merge(const float *o_a, const float *lse_a, const float *o_b,
                         const float *lse_b, void *o_out, bool out_bf16, float *lse_out,
                         int64_t rows, int32_t heads, int32_t head_dim, int32_t sm_count,
                         cudaStream_t stream);

// Records a one-line reason for pkv_last_error() and returns s.
pkv_status fail_status(pkv_status s, const char *fmt, ...);

}  // namespace pkv
