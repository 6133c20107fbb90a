// decode.cu - paged GQA decode attention with split-KV and a log-sum-exp merge.
//
// What it computes ("Code Notes: mini-sglang", Engine Layer table,
// BaseAttnBackend / BaseKVCachePool rows; Scheduler Layer table, TableManager
// row): for every request b and q head h, softmax attention of q[b,h] over
// the first seq_len[b] keys of its page_table row, on kv head h / g.
//
// Design (HBM-bound: every K/V byte is read once, 4 flops per byte at g=4):
//  * Grid (kv-head group, split, request). A CTA of 4 warps covers up to 4
//    kv heads of one request over one split (a contiguous key range), so the
//    CTA's loads of one token are one contiguous 1 KB (4 heads x 256 B) run.
//  * Each warp streams 16-key tiles of its kv head through its own 2-stage
//    cp.async pipeline (16-byte chunks, zero-filled past the end, slots
//    resolved from the page table one key per lane) into XOR-swizzled shared
//    memory. No CTA-wide barrier inside the loop.
//  * Scores are S^T = K q^T on the m16n8k16 tensor-core MMA with keys as the
//    M dimension and the g <= 8 q heads of the group as N: the MMA work is
//    exact at g = 8 and the FMA pipe is left free. The bf16 probabilities go
//    through movmatrix to become the B operand of O^T += V^T P^T (V^T from
//    ldmatrix.trans). Online softmax runs in the log2 domain; per-thread sums
//    are reduced across lanes only once, at the end.
//  * Warps sharing a head, then splits, are merged by log-sum-exp: in shared
//    memory inside the CTA, and by a small second kernel across splits (the
//    partial states sit in the caller's workspace and are mostly L2 hits).
//  * The split size comes from host scalars only (batch, heads, a bound on
//    seq_len, SM count), so the call never syncs and is graph-capturable.
#include <math.h>

#include "decode_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

#ifndef PKV_DECODE_UNITS_PER_SM
#define PKV_DECODE_UNITS_PER_SM 8  // split sizing: CTAs of work per SM at max length
#endif
#ifndef PKV_DECODE_MIN_SPLIT_TILES
#define PKV_DECODE_MIN_SPLIT_TILES 8  // smallest split, in 16-key tiles
#endif
#ifndef PKV_MERGE_BATCH
#define PKV_MERGE_BATCH 16  // partial rows the merge loads in its first round trip
#endif

template <int D>
__global__ void __launch_bounds__(kDecodeThreads, (kDecodeStages <= 3 ? 2 : 1)) decode_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  if (!a.defer_wait) grid_dependency_wait();  // inputs may come from the previous kernel (store_kv)
  grid_dependents_launch();  // the split merge may be scheduled as CTAs drain
  decode_body<D, kDecodeStages>(a, blockIdx.x, blockIdx.y, blockIdx.z, threadIdx.x, smem,
                                [] { __syncthreads(); });
  if (a.defer_wait && blockIdx.y == 0 && blockIdx.z == gridDim.z - 1) grid_dependency_wait();
}

// Cross-split merge: one warp per (request, q head) with more than one
// split; with a cascade's shared-prefix states in slots splits .. pstride - 1,
// every (request, q head) merges its suffix splits with those. Lane s holds
// the lse of state s; the partial rows of up to kMergeBatch states are
// loaded together with the lse values, so the common case costs one
// round trip to L2 after the decode grid completes. The grid holds at most
// one wave of CTAs; a warp takes (request, q head) pairs warp-stride.
constexpr int kMergeBatch = PKV_MERGE_BATCH;
constexpr int kMergeThreads = 128;
#ifndef PKV_MERGE_CTAS_PER_SM
#define PKV_MERGE_CTAS_PER_SM 16  // resident merge CTAs per SM the grid is sized for
#endif


template <int D>
__device__ __forceinline__ void merge_pair(const DecodeArgs &a, int64_t bh, int lane);

template <int D>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(const DecodeArgs a, int32_t batch) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t pairs = static_cast<int64_t>(batch) * a.hq;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * (kMergeThreads / 32);
  int64_t bh = static_cast<int64_t>(blockIdx.x) * (kMergeThreads / 32) + warp;
  // seq_lens and table_idx are inputs of the call (complete before any
  // decode CTA passed its own dependency wait): the first pair's are read
  // before the wait.
  if (bh < pairs) (void)row_info(a, static_cast<int>(bh / a.hq), false);
  grid_dependency_wait();  // the partial states come from decode_kernel
  for (; bh < pairs; bh += stride) merge_pair<D>(a, bh, lane);
}

template <int D>
__device__ __forceinline__ void merge_pair(const DecodeArgs &a, int64_t bh, int lane) {
  const int b = static_cast<int>(bh / a.hq);
  const RowInfo ri = row_info(a, b, false);
  const int n = ri.nsplit;
  if (n <= 1 && !a.force_partial) return;
  // suffix splits in slots 0 .. n - 1, shared-prefix states (cascade) in
  // slots splits .. pstride - 1: state s < n is slot s, state n + e is slot
  // splits + e
  const int total = n + (a.pstride - a.splits);
  const float *pl = a.part_lse + bh * a.pstride;
  const float *po = a.part_o + bh * a.pstride * D + lane * 4;
  auto slot = [&](int st) { return st < n ? st : a.splits + (st - n); };
  const bool row_lane = lane < D / 4;
  float4 v[kMergeBatch];
#pragma unroll
  for (int u = 0; u < kMergeBatch; ++u)
    v[u] = (row_lane && u < total)
               ? *reinterpret_cast<const float4 *>(po + static_cast<int64_t>(slot(u)) * D)
               : make_float4(0.f, 0.f, 0.f, 0.f);
  float lse_l = lane < total ? pl[slot(lane)] : -INFINITY;
  float M = lse_l;
  for (int s = lane + 32; s < total; s += 32) M = fmaxf(M, pl[slot(s)]);
#pragma unroll
  for (int x = 16; x > 0; x >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, x));
  const float ref = M == -INFINITY ? 0.f : M;
  const float e_l = lane < total ? expf(lse_l - ref) : 0.f;
  float L = e_l;
  for (int s = lane + 32; s < total; s += 32) L += expf(pl[slot(s)] - ref);
#pragma unroll
  for (int x = 16; x > 0; x >>= 1) L += __shfl_xor_sync(0xffffffffu, L, x);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int u = 0; u < kMergeBatch; ++u) {
    const float w = __shfl_sync(0xffffffffu, e_l, u) * inv;
    O.x += w * v[u].x;
    O.y += w * v[u].y;
    O.z += w * v[u].z;
    O.w += w * v[u].w;
  }
  // Beyond the first batch (long rows, cascade prefix states): batches of
  // eight rows, all loads of a batch issued before their weights are used.
  for (int s0 = kMergeBatch; s0 < total; s0 += 8) {
    float4 x[8];
    float w[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int st = s0 + u;
      const bool in = st < total;
      x[u] = (row_lane && in)
                 ? *reinterpret_cast<const float4 *>(po + static_cast<int64_t>(slot(st)) * D)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
      w[u] = in && st >= 32 ? pl[slot(st)] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int st = s0 + u;
      const float e = st < 32 ? __shfl_sync(0xffffffffu, e_l, st & 31)
                              : (st < total ? expf(w[u] - ref) : 0.f);
      const float wt = e * inv;
      O.x += wt * x[u].x;
      O.y += wt * x[u].y;
      O.z += wt * x[u].z;
      O.w += wt * x[u].w;
    }
  }
  if (row_lane) {
    uint2 packed;
    packed.x = pack_bf16(O.x, O.y);
    packed.y = pack_bf16(O.z, O.w);
    *reinterpret_cast<uint2 *>(a.o + bh * D + lane * 4) = packed;
  }
  if (lane == 0 && a.lse) a.lse[bh] = L > 0.f ? ref + logf(L) : -INFINITY;
}

// The same merge for plans with at most kNarrowStates states per (request,
// q head) (suffix splits plus cascade prefix slots): a group of D / 16 lanes
// per pair, 16 columns per lane, 32 / (D / 16) pairs per warp. A quarter of
// the warps of decode_merge_kernel at about its registers per thread, so a
// batch of a few hundred requests is merged by one wave of CTAs right after
// the decode grid completes.
constexpr int kNarrowStates = 4;
#ifndef PKV_MERGE_NARROW
#define PKV_MERGE_NARROW 1  // 0: every merge through decode_merge_kernel
#endif

template <int D>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_narrow_kernel(const DecodeArgs a,
                                                                           int32_t batch) {
  constexpr int kLanes = D / 16;       // lanes per (request, q head) pair
  constexpr int kPairs = 32 / kLanes;  // pairs per warp
  static_assert(kNarrowStates <= kLanes, "one lse per lane of a pair's group");
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int grp = lane / kLanes;  // pair of this lane within the warp
  const int sl = lane % kLanes;   // lane within the pair's group
  const int64_t pairs = static_cast<int64_t>(batch) * a.hq;
  const int64_t bh =
      (static_cast<int64_t>(blockIdx.x) * (kMergeThreads / 32) + warp) * kPairs + grp;
  int n = 0, total = 0;
  if (bh < pairs) {
    // seq_lens and table_idx are inputs of the call: read before the wait
    n = row_info(a, static_cast<int>(bh / a.hq), false).nsplit;
    total = (n <= 1 && !a.force_partial) ? 0 : n + (a.pstride - a.splits);
  }
  grid_dependency_wait();  // the partial states come from decode_kernel
  // total is uniform over a pair's group; every lane of the warp takes part
  // in the shuffles (those of groups with nothing to merge on zeros).
  auto slot = [&](int st) { return st < n ? st : a.splits + (st - n); };
  const int64_t bhc = total > 0 ? bh : 0;
  const float *pl = a.part_lse + bhc * a.pstride;
  const float *po = a.part_o + bhc * a.pstride * D + sl * 16;
  float4 v[kNarrowStates][4];
#pragma unroll
  for (int st = 0; st < kNarrowStates; ++st)
#pragma unroll
    for (int c = 0; c < 4; ++c)
      v[st][c] = st < total ? *reinterpret_cast<const float4 *>(
                                  po + static_cast<int64_t>(slot(st)) * D + c * 4)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
  const float lse_l = sl < total ? pl[slot(sl)] : -INFINITY;
  float M = lse_l;
#pragma unroll
  for (int x = kLanes / 2; x > 0; x >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, x, kLanes));
  const float ref = M == -INFINITY ? 0.f : M;
  const float e_l = sl < total ? expf(lse_l - ref) : 0.f;
  float L = e_l;
#pragma unroll
  for (int x = kLanes / 2; x > 0; x >>= 1) L += __shfl_xor_sync(0xffffffffu, L, x, kLanes);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  float o[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i] = 0.f;
#pragma unroll
  for (int st = 0; st < kNarrowStates; ++st) {
    const float w = __shfl_sync(0xffffffffu, e_l, st, kLanes) * inv;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      o[4 * c] += w * v[st][c].x;
      o[4 * c + 1] += w * v[st][c].y;
      o[4 * c + 2] += w * v[st][c].z;
      o[4 * c + 3] += w * v[st][c].w;
    }
  }
  if (total == 0) return;  // one split: decode_kernel wrote o itself
  uint4 *dst = reinterpret_cast<uint4 *>(a.o + bh * D + sl * 16);
  dst[0] = make_uint4(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]), pack_bf16(o[4], o[5]),
                      pack_bf16(o[6], o[7]));
  dst[1] = make_uint4(pack_bf16(o[8], o[9]), pack_bf16(o[10], o[11]), pack_bf16(o[12], o[13]),
                      pack_bf16(o[14], o[15]));
  if (sl == 0 && a.lse) a.lse[bh] = L > 0.f ? ref + logf(L) : -INFINITY;
}

}  // namespace

static DecodePlan plan_splits(int32_t batch, int32_t hq, int32_t hkv, int32_t d,
                              int32_t max_seq_len, int32_t sm_count, int32_t units_per_sm);

DecodePlan plan_decode(int32_t batch, int32_t hq, int32_t hkv, int32_t d, int32_t max_seq_len,
                       int32_t sm_count) {
  return plan_splits(batch, hq, hkv, d, max_seq_len, sm_count, PKV_DECODE_UNITS_PER_SM);
}

#ifndef PKV_CASCADE_UNITS_PER_SM
#define PKV_CASCADE_UNITS_PER_SM PKV_DECODE_UNITS_PER_SM
#endif

DecodePlan plan_cascade_suffix(int32_t batch, int32_t hq, int32_t hkv, int32_t d,
                               int32_t max_seq_len, int32_t sm_count) {
  return plan_splits(batch, hq, hkv, d, max_seq_len, sm_count, PKV_CASCADE_UNITS_PER_SM);
}

static DecodePlan plan_splits(int32_t batch, int32_t hq, int32_t hkv, int32_t d,
                              int32_t max_seq_len, int32_t sm_count, int32_t units_per_sm) {
  (void)hq;
  DecodePlan p{};
  p.sm_count = sm_count;
  p.heads_per_cta = hkv >= kDecodeWarps ? kDecodeWarps : hkv;
  p.warps_per_head = kDecodeWarps / p.heads_per_cta;
  p.head_groups = hkv / p.heads_per_cta;
  const int64_t max_seq = max_seq_len < 1 ? 1 : max_seq_len;
  const int64_t tiles = (max_seq + kDecodeTileKeys - 1) / kDecodeTileKeys;
  // Aim for about PKV_DECODE_UNITS_PER_SM CTAs of work per SM if every
  // request were max_seq long, with at least PKV_DECODE_MIN_SPLIT_TILES tiles
  // per split so partial states stay a few percent of the KV bytes.
  const int64_t units = static_cast<int64_t>(batch) * p.head_groups * tiles;
  const int64_t target = static_cast<int64_t>(sm_count > 0 ? sm_count : 1) * units_per_sm;
  int64_t chunk_tiles = (units + target - 1) / target;
  if (chunk_tiles < PKV_DECODE_MIN_SPLIT_TILES) chunk_tiles = PKV_DECODE_MIN_SPLIT_TILES;
  int64_t splits = (tiles + chunk_tiles - 1) / chunk_tiles;
  while (splits > 65535) {
    chunk_tiles *= 2;
    splits = (tiles + chunk_tiles - 1) / chunk_tiles;
  }
  p.chunk = static_cast<int32_t>(chunk_tiles * kDecodeTileKeys);
  p.splits = static_cast<int32_t>(splits);
  if (p.splits > 1) {
    const size_t rows = static_cast<size_t>(batch) * hq * p.splits;
    const size_t o_bytes = (rows * d * sizeof(float) + 255) & ~size_t(255);
    const size_t l_bytes = (rows * sizeof(float) + 255) & ~size_t(255);
    p.workspace_bytes = o_bytes + l_bytes;
  } else {
    p.workspace_bytes = 0;
  }
  return p;
}

static DecodeArgs decode_args(const PoolGeom &g, int32_t layer, const void *q, void *o,
                              float *lse, const int32_t *page_table, int64_t table_stride,
                              const int32_t *table_idx, const int32_t *seq_lens, int32_t hq,
                              float scale, const DecodePlan &plan, unsigned *err) {
  DecodeArgs a{};
  a.pool = static_cast<const __nv_bfloat16 *>(g.base);
  a.plane = g.plane;
  a.slots = g.slots;
  a.num_layers = g.num_layers;
  a.layer = layer;
  a.page_size = g.page_size;
  a.hkv = g.hkv;
  a.q = static_cast<const __nv_bfloat16 *>(q);
  a.o = static_cast<__nv_bfloat16 *>(o);
  a.lse = lse;
  a.page_table = page_table;
  a.table_stride = table_stride;
  a.table_idx = table_idx;
  a.seq_lens = seq_lens;
  a.hq = hq;
  a.group = hq / g.hkv;
  a.scale_log2 = scale * kLog2e;
  a.heads_per_cta = plan.heads_per_cta;
  a.warps_per_head = plan.warps_per_head;
  a.chunk = plan.chunk;
  a.splits = plan.splits;
  a.pstride = plan.splits;
  a.force_partial = 0;
  a.err = err;
  return a;
}

static cudaError_t launch_decode_main(const DecodeArgs &a, const PoolGeom &g,
                                      const DecodePlan &plan, int32_t batch, cudaStream_t stream) {
  cudaError_t e;
  const dim3 grid(plan.head_groups, plan.splits, batch);
  if (g.d == 128) {
    e = cudaFuncSetAttribute(decode_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DecodeSmem<128>::kTotal);
    if (e != cudaSuccess) return e;
    e = launch_pdl(decode_kernel<128>, grid, dim3(kDecodeThreads), DecodeSmem<128>::kTotal, stream, a);
  } else {
    e = cudaFuncSetAttribute(decode_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DecodeSmem<64>::kTotal);
    if (e != cudaSuccess) return e;
    e = launch_pdl(decode_kernel<64>, grid, dim3(kDecodeThreads), DecodeSmem<64>::kTotal, stream, a);
  }
  return e;
}

static cudaError_t launch_decode_merge(const DecodeArgs &a, const PoolGeom &g, int32_t batch,
                                       int32_t sm_count, cudaStream_t stream) {
  const int64_t pairs = static_cast<int64_t>(batch) * a.hq;
  if (PKV_MERGE_NARROW && a.pstride <= kNarrowStates) {
    const int64_t per_cta = (kMergeThreads / 32) * (32 / (g.d / 16));
    const dim3 ngrid(static_cast<unsigned>((pairs + per_cta - 1) / per_cta));
    if (g.d == 128)
      return launch_pdl(decode_merge_narrow_kernel<128>, ngrid, dim3(kMergeThreads), 0, stream, a,
                        batch);
    return launch_pdl(decode_merge_narrow_kernel<64>, ngrid, dim3(kMergeThreads), 0, stream, a,
                      batch);
  }
  int64_t ctas = (pairs + 3) / 4;
  const int64_t wave = static_cast<int64_t>(sm_count > 0 ? sm_count : 1) * PKV_MERGE_CTAS_PER_SM;
  if (ctas > wave) ctas = wave;
  const dim3 mgrid(static_cast<unsigned>(ctas));
  if (g.d == 128) return launch_pdl(decode_merge_kernel<128>, mgrid, dim3(128), 0, stream, a, batch);
  return launch_pdl(decode_merge_kernel<64>, mgrid, dim3(128), 0, stream, a, batch);
}

cudaError_t launch_decode(const PoolGeom &g, int32_t layer, const void *q, void *o, float *lse,
                          const int32_t *page_table, int64_t table_stride,
                          const int32_t *table_idx, const int32_t *seq_lens, int32_t batch,
                          int32_t hq, float scale, const DecodePlan &plan, void *workspace,
                          unsigned *err, cudaStream_t stream, const void *k_new,
                          const void *v_new, int64_t kv_row_stride) {
  DecodeArgs a = decode_args(g, layer, q, o, lse, page_table, table_stride, table_idx, seq_lens,
                             hq, scale, plan, err);
  a.k_new = static_cast<const __nv_bfloat16 *>(k_new);
  a.v_new = static_cast<const __nv_bfloat16 *>(v_new);
  a.kv_row_stride = kv_row_stride;
  // the pool is the caller's writable buffer (store_kv writes it too)
  a.pool_w = const_cast<__nv_bfloat16 *>(static_cast<const __nv_bfloat16 *>(g.base));
  if (plan.splits > 1) {
    const size_t rows = static_cast<size_t>(batch) * hq * plan.splits;
    const size_t o_bytes = (rows * g.d * sizeof(float) + 255) & ~size_t(255);
    a.part_o = static_cast<float *>(workspace);
    a.part_lse = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + o_bytes);
  }
  cudaError_t e = launch_decode_main(a, g, plan, batch, stream);
  if (e != cudaSuccess || plan.splits <= 1) return e;
  return launch_decode_merge(a, g, batch, plan.sm_count, stream);
}

size_t cascade_partial_bytes(int32_t batch, int32_t hq, int32_t d, int32_t slots) {
  const size_t rows = static_cast<size_t>(batch) * hq * static_cast<size_t>(slots);
  return ((rows * d * sizeof(float) + 255) & ~size_t(255)) +
         ((rows * sizeof(float) + 255) & ~size_t(255));
}

void cascade_partial_ptrs(void *partials, int32_t batch, int32_t hq, int32_t d, int32_t slots,
                          float **part_o, float **part_lse) {
  const size_t rows = static_cast<size_t>(batch) * hq * static_cast<size_t>(slots);
  *part_o = static_cast<float *>(partials);
  *part_lse = reinterpret_cast<float *>(static_cast<uint8_t *>(partials) +
                                        ((rows * d * sizeof(float) + 255) & ~size_t(255)));
}

cudaError_t launch_cascade_suffix(const PoolGeom &g, int32_t layer, const void *q, void *o,
                                  float *lse, const int32_t *page_table, int64_t table_stride,
                                  const int32_t *table_idx, const int32_t *seq_lens,
                                  int32_t batch, int32_t hq, float scale, const DecodePlan &plan,
                                  int32_t prefix_slots, void *partials, unsigned *err,
                                  cudaStream_t stream, float **part_o, float **part_lse) {
  DecodeArgs a = decode_args(g, layer, q, o, lse, page_table, table_stride, table_idx, seq_lens,
                             hq, scale, plan, err);
  a.pstride = plan.splits + prefix_slots;
  a.force_partial = 1;
  a.defer_wait = 1;
  cascade_partial_ptrs(partials, batch, hq, g.d, a.pstride, &a.part_o, &a.part_lse);
  *part_o = a.part_o;
  *part_lse = a.part_lse;
  return launch_decode_main(a, g, plan, batch, stream);
}

cudaError_t launch_cascade_merge(const PoolGeom &g, int32_t layer, const void *q, void *o,
                                 float *lse, const int32_t *page_table, int64_t table_stride,
                                 const int32_t *table_idx, const int32_t *seq_lens, int32_t batch,
                                 int32_t hq, float scale, const DecodePlan &plan,
                                 int32_t prefix_slots, float *part_o, float *part_lse,
                                 unsigned *err, cudaStream_t stream) {
  DecodeArgs a = decode_args(g, layer, q, o, lse, page_table, table_stride, table_idx, seq_lens,
                             hq, scale, plan, err);
  a.pstride = plan.splits + prefix_slots;
  a.force_partial = 1;
  a.part_o = part_o;
  a.part_lse = part_lse;
  return launch_decode_merge(a, g, batch, plan.sm_count, stream);
}

}  // namespace pkv
