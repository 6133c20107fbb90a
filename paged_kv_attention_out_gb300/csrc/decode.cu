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

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

// Tuning constants (compile-time; the defaults are the measured best on GB300).
#ifndef PKV_DECODE_STAGES
#define PKV_DECODE_STAGES 2  // cp.async pipeline depth per warp
#endif
#ifndef PKV_DECODE_UNITS_PER_SM
#define PKV_DECODE_UNITS_PER_SM 8  // split sizing: CTAs of work per SM at max length
#endif
#ifndef PKV_DECODE_WARPS
#define PKV_DECODE_WARPS 4  // warps per CTA (each on one kv head)
#endif
#ifndef PKV_DECODE_MIN_SPLIT_TILES
#define PKV_DECODE_MIN_SPLIT_TILES 8  // smallest split, in 16-key tiles
#endif
#ifndef PKV_MERGE_BATCH
#define PKV_MERGE_BATCH 16  // partial rows the merge loads in its first round trip
#endif

constexpr int kWarps = PKV_DECODE_WARPS;
constexpr int kThreads = kWarps * 32;
constexpr int kTileKeys = 16;
constexpr int kStages = PKV_DECODE_STAGES;

template <int D>
struct DecodeSmem {
  static constexpr int kTileBytes = kTileKeys * D * 2;  // one K (or V) tile
  static constexpr int kStageBytes = 2 * kTileBytes;    // K + V
  static constexpr int kWarpBytes = kStages * kStageBytes;
  static constexpr int kTotal = kWarps * kWarpBytes;
  // epilogue reuse of a warp's region: O^T [8][D] fp32 + m[8] + l[8]
  static_assert(8 * D * 4 + 64 <= kWarpBytes, "epilogue does not fit");
};

struct DecodeArgs {
  const __nv_bfloat16 *pool;
  int64_t plane;
  int64_t slots;
  int32_t num_layers;
  int32_t layer;
  int32_t page_size;
  int32_t hkv;
  const __nv_bfloat16 *q;
  __nv_bfloat16 *o;
  float *lse;
  const int32_t *page_table;
  int64_t table_stride;
  const int32_t *table_idx;
  const int32_t *seq_lens;
  int32_t hq;
  int32_t group;
  float scale_log2;
  int32_t heads_per_cta;
  int32_t warps_per_head;
  int32_t chunk;
  int32_t splits;
  int32_t pstride;        // partial slots per (request, q head): splits, or more when
                          // slots splits .. pstride - 1 hold shared-prefix states (cascade)
  int32_t force_partial;  // write partial states even for one split (cascade)
  float *part_o;    // [B, Hq, pstride, D]
  float *part_lse;  // [B, Hq, pstride] (natural log)
  unsigned *err;
  // store_kv fused into the step (may be null): request b's new key and
  // value rows k_new[b], v_new[b] (row stride kv_row_stride elements) go to
  // key seq_len - 1 of its row before it is attended
  const __nv_bfloat16 *k_new;
  const __nv_bfloat16 *v_new;
  int64_t kv_row_stride;
  __nv_bfloat16 *pool_w;
  // Cascade suffix: the previous kernel on the stream (the shared-prefix
  // attention) writes nothing this kernel reads, so the CTAs do not wait for
  // it at entry; the split-0 CTAs of the last request wait for it at exit,
  // so this grid still completes after it (and the merge after both).
  int32_t defer_wait;
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t ld_b32(const __nv_bfloat16 *p) {
  return *reinterpret_cast<const uint32_t *>(p);
}

// Request-level facts every CTA (and the merge kernel) derives the same way.
struct RowInfo {
  const int32_t *row;
  int seq;
  int nsplit;
};

__device__ __forceinline__ RowInfo row_info(const DecodeArgs &a, int b, bool report) {
  RowInfo r;
  int row_id = a.table_idx ? a.table_idx[b] : b;
  int seq = a.seq_lens[b];
  const int64_t max_keys = a.table_stride * a.page_size;
  if (row_id < 0) {
    if (report) flag_error(a.err, kErrTableIdx);
    row_id = 0;
    seq = 0;
  }
  if (seq < 0 || seq > max_keys) {
    if (report) flag_error(a.err, kErrSeqLen);
    seq = seq < 0 ? 0 : static_cast<int>(max_keys);
  }
  r.row = a.page_table + static_cast<int64_t>(row_id) * a.table_stride;
  r.seq = seq;
  int n = (seq + a.chunk - 1) / a.chunk;
  r.nsplit = n < 1 ? 1 : (n > a.splits ? a.splits : n);
  return r;
}

template <int D>
__global__ void __launch_bounds__(kThreads, (kStages <= 3 ? 2 : 1)) decode_kernel(const DecodeArgs a) {
  using S = DecodeSmem<D>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.y;
  const int b = blockIdx.z;

  if (!a.defer_wait) grid_dependency_wait();  // inputs may come from the previous kernel (store_kv)
  grid_dependents_launch();  // the split merge may be scheduled as CTAs drain
  const RowInfo ri = row_info(a, b, split == 0 && blockIdx.x == 0 && threadIdx.x == 0);
  if (split >= ri.nsplit) return;
  if (a.k_new) {
    // Fused store: the split holding key seq - 1 writes the new token's K and
    // V rows of its kv heads first; no other CTA reads that key of these heads.
    if (split == ri.nsplit - 1 && ri.seq > 0) {
      const int pos = ri.seq - 1;
      const int pe = __ldg(ri.row + pos / a.page_size);
      const int64_t slot = static_cast<int64_t>(pe) * a.page_size + pos % a.page_size;
      if (pe < 0 || slot >= a.slots) {
        if (threadIdx.x == 0) flag_error(a.err, kErrPage);
      } else {
        constexpr int kCh = D / 8;  // 16-byte chunks per head row
        for (int i = threadIdx.x; i < a.heads_per_cta * 2 * kCh; i += kThreads) {
          const int ch = i % kCh;
          const int c = (i / kCh) & 1;
          const int h = blockIdx.x * a.heads_per_cta + i / kCh / 2;
          const __nv_bfloat16 *src =
              (c ? a.v_new : a.k_new) + static_cast<int64_t>(b) * a.kv_row_stride + h * D + ch * 8;
          __nv_bfloat16 *dst = a.pool_w + (static_cast<int64_t>(c) * a.num_layers + a.layer) * a.plane +
                               slot * a.hkv * D + h * D + ch * 8;
          *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
        }
      }
      __threadfence();  // visible to this CTA's copies (and the GPU) before they read it
    }
    __syncthreads();
  }
  const int key_begin = split * a.chunk;
  const int key_end = (split == ri.nsplit - 1) ? ri.seq : key_begin + a.chunk;

  const int head_slot = warp % a.heads_per_cta;
  const int sub = warp / a.heads_per_cta;
  const int kvh = blockIdx.x * a.heads_per_cta + head_slot;
  const int ntiles = (key_end - key_begin + kTileKeys - 1) / kTileKeys;
  const int my_tiles = ntiles > sub ? (ntiles - sub + a.warps_per_head - 1) / a.warps_per_head : 0;

  // q of the group as the MMA B operand: k = head dim, n = q head in group.
  uint32_t bq[D / 16][2];
  {
    const int n = lane >> 2;
    const int kk = (lane & 3) * 2;
    const bool valid = n < a.group;
    const __nv_bfloat16 *qp =
        a.q + (static_cast<int64_t>(b) * a.hq + kvh * a.group + (valid ? n : 0)) * D;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      bq[ks][0] = valid ? ld_b32(qp + ks * 16 + kk) : 0u;
      bq[ks][1] = valid ? ld_b32(qp + ks * 16 + kk + 8) : 0u;
    }
  }

  float acc[D / 16][4];
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  uint8_t *wsm = smem + warp * S::kWarpBytes;
  const uint32_t wbase = smem_addr(wsm);
  const int64_t slot_stride = static_cast<int64_t>(a.hkv) * D;
  const __nv_bfloat16 *kbase =
      a.pool + static_cast<int64_t>(a.layer) * a.plane + static_cast<int64_t>(kvh) * D;
  const __nv_bfloat16 *vbase =
      a.pool + (static_cast<int64_t>(a.num_layers) + a.layer) * a.plane +
      static_cast<int64_t>(kvh) * D;
  const int P = a.page_size;

  // Page-table entry of this lane's key of warp tile j (lanes 0..15), or -1
  // past the end. Loaded one tile before its copies are issued, so the index
  // load is off the critical path of the copy stream.
  auto load_entry = [&](int j) -> int {
    int e = -1;
    if (lane < kTileKeys && j < my_tiles) {
      const int key = key_begin + (sub + j * a.warps_per_head) * kTileKeys + lane;
      if (key < key_end) e = __ldg(ri.row + ((P == 1) ? key : key / P));
    }
    return e;
  };
  auto issue = [&](int j, int entry, int stage) {
    const int k0 = key_begin + (sub + j * a.warps_per_head) * kTileKeys;
    long long slot = -1;
    if (lane < kTileKeys && k0 + lane < key_end) {
      const int key = k0 + lane;
      const int off = (P == 1) ? 0 : key % P;
      const long long s = static_cast<long long>(entry) * P + off;
      if (entry < 0 || s >= a.slots) {
        flag_error(a.err, kErrPage);
      } else {
        slot = s;
      }
    }
    constexpr int CPK = D / 8;      // 16-byte chunks per key row
    constexpr int KPI = 32 / CPK;   // keys per warp instruction
    const int chunk = lane % CPK;
    const uint32_t st = wbase + stage * S::kStageBytes;
#pragma unroll
    for (int it = 0; it < kTileKeys / KPI; ++it) {
      const int r = it * KPI + lane / CPK;
      const long long s = __shfl_sync(0xffffffffu, slot, r);
      const bool ok = s >= 0;
      const int64_t off = ok ? s * slot_stride + chunk * 8 : 0;
      const uint32_t dk = st + swz<D>(r, chunk);
      cp_async_16(dk, ok ? kbase + off : a.pool, ok ? 16 : 0);
      cp_async_16(dk + S::kTileBytes, ok ? vbase + off : a.pool, ok ? 16 : 0);
    }
  };

  int next_entry;
  {
    int e[kStages - 1];
#pragma unroll
    for (int j = 0; j < kStages - 1; ++j) e[j] = load_entry(j);
    next_entry = load_entry(kStages - 1);
#pragma unroll
    for (int j = 0; j < kStages - 1; ++j) {
      if (j < my_tiles) issue(j, e[j], j);
      cp_async_commit();
    }
  }

  const int r0 = lane >> 2;
  for (int j = 0; j < my_tiles; ++j) {
    const int jn = j + kStages - 1;
    if (jn < my_tiles) issue(jn, next_entry, jn % kStages);
    cp_async_commit();
    next_entry = load_entry(jn + 1);
    cp_async_wait<kStages - 1>();
    __syncwarp();

    const uint32_t kst = wbase + (j % kStages) * S::kStageBytes;
    const uint32_t vst = kst + S::kTileBytes;
    const int k0 = key_begin + (sub + j * a.warps_per_head) * kTileKeys;

    // S^T[16 keys][8 heads] = K_tile . q^T
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldmatrix_x4(kst + swz<D>((lane & 7) + ((lane >> 3) & 1) * 8, ks * 2 + (lane >> 4)), a0,
                  a1, a2, a3);
      mma_bf16_16816(s, a0, a1, a2, a3, bq[ks][0], bq[ks][1]);
    }
    // s[0]: key r0, head n0; s[1]: key r0, head n0+1; s[2], s[3]: key r0 + 8.
    const bool ok0 = k0 + r0 < key_end;
    const bool ok1 = k0 + r0 + 8 < key_end;
    s[0] = ok0 ? s[0] * a.scale_log2 : -INFINITY;
    s[1] = ok0 ? s[1] * a.scale_log2 : -INFINITY;
    s[2] = ok1 ? s[2] * a.scale_log2 : -INFINITY;
    s[3] = ok1 ? s[3] * a.scale_log2 : -INFINITY;
    float mx0 = fmaxf(s[0], s[2]);
    float mx1 = fmaxf(s[1], s[3]);
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, x));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, x));
    }
    const float mn0 = fmaxf(m0, mx0);
    const float mn1 = fmaxf(m1, mx1);
    const float ref0 = mn0 == -INFINITY ? 0.f : mn0;
    const float ref1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = fast_exp2(m0 - ref0);
    const float al1 = fast_exp2(m1 - ref1);
    const float p0 = fast_exp2(s[0] - ref0);
    const float p1 = fast_exp2(s[1] - ref1);
    const float p2 = fast_exp2(s[2] - ref0);
    const float p3 = fast_exp2(s[3] - ref1);
    l0 = l0 * al0 + (p0 + p2);
    l1 = l1 * al1 + (p1 + p3);
    m0 = mn0;
    m1 = mn1;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      acc[mt][0] *= al0;
      acc[mt][1] *= al1;
      acc[mt][2] *= al0;
      acc[mt][3] *= al1;
    }
    // P^T as the B operand (k = key, n = head): transpose the two 8x8 halves.
    const uint32_t bp0 = movmatrix_trans(pack_bf16(p0, p1));
    const uint32_t bp1 = movmatrix_trans(pack_bf16(p2, p3));
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      uint32_t a0, a1, a2, a3;
      ldmatrix_x4_trans(vst + swz<D>((lane & 7) + (lane >> 4) * 8, mt * 2 + ((lane >> 3) & 1)),
                        a0, a1, a2, a3);
      mma_bf16_16816(acc[mt], a0, a1, a2, a3, bp0, bp1);
    }
    __syncwarp();
  }
  cp_async_wait<0>();
  __syncwarp();

#pragma unroll
  for (int x = 4; x < 32; x <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, x);
    l1 += __shfl_xor_sync(0xffffffffu, l1, x);
  }

  // Per-warp state to shared memory: O^T [8 heads][D], m[8], l[8] (log2 domain).
  float *so = reinterpret_cast<float *>(wsm);
  float *sm_m = so + 8 * D;
  float *sm_l = sm_m + 8;
  const int n0 = (lane & 3) * 2;
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    so[n0 * D + mt * 16 + r0] = acc[mt][0];
    so[(n0 + 1) * D + mt * 16 + r0] = acc[mt][1];
    so[n0 * D + mt * 16 + r0 + 8] = acc[mt][2];
    so[(n0 + 1) * D + mt * 16 + r0 + 8] = acc[mt][3];
  }
  if (lane < 4) {
    sm_m[n0] = m0;
    sm_m[n0 + 1] = m1;
    sm_l[n0] = l0;
    sm_l[n0 + 1] = l1;
  }
  __syncthreads();

  // Merge the warps that share a kv head; write the final or the partial state.
  const bool final_out = ri.nsplit == 1 && !a.force_partial;
  const int items = a.heads_per_cta * a.group * (D / 4);
  for (int it = threadIdx.x; it < items; it += kThreads) {
    const int d4 = it % (D / 4);
    const int n = (it / (D / 4)) % a.group;
    const int hs = it / (D / 4) / a.group;
    float M = -INFINITY;
    for (int w = 0; w < a.warps_per_head; ++w) {
      const float *base = reinterpret_cast<const float *>(smem + (hs + w * a.heads_per_cta) * S::kWarpBytes);
      M = fmaxf(M, base[8 * D + n]);
    }
    const float ref = M == -INFINITY ? 0.f : M;
    float L = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int w = 0; w < a.warps_per_head; ++w) {
      const float *base = reinterpret_cast<const float *>(smem + (hs + w * a.heads_per_cta) * S::kWarpBytes);
      const float sc = fast_exp2(base[8 * D + n] - ref);
      L += base[8 * D + 8 + n] * sc;
      const float4 v = *reinterpret_cast<const float4 *>(base + n * D + d4 * 4);
      O.x += v.x * sc;
      O.y += v.y * sc;
      O.z += v.z * sc;
      O.w += v.w * sc;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    O.x *= inv;
    O.y *= inv;
    O.z *= inv;
    O.w *= inv;
    const float lse_nat = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
    const int h = (blockIdx.x * a.heads_per_cta + hs) * a.group + n;
    const int64_t bh = static_cast<int64_t>(b) * a.hq + h;
    if (final_out) {
      uint2 packed;
      packed.x = pack_bf16(O.x, O.y);
      packed.y = pack_bf16(O.z, O.w);
      *reinterpret_cast<uint2 *>(a.o + bh * D + d4 * 4) = packed;
      if (d4 == 0 && a.lse) a.lse[bh] = lse_nat;
    } else {
      *reinterpret_cast<float4 *>(a.part_o + (bh * a.pstride + split) * D + d4 * 4) = O;
      if (d4 == 0) a.part_lse[bh * a.pstride + split] = lse_nat;
    }
  }
  if (a.defer_wait && split == 0 && b == static_cast<int>(gridDim.z) - 1) grid_dependency_wait();
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
  p.heads_per_cta = hkv >= kWarps ? kWarps : hkv;
  p.warps_per_head = kWarps / p.heads_per_cta;
  p.head_groups = hkv / p.heads_per_cta;
  const int64_t max_seq = max_seq_len < 1 ? 1 : max_seq_len;
  const int64_t tiles = (max_seq + kTileKeys - 1) / kTileKeys;
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
  p.chunk = static_cast<int32_t>(chunk_tiles * kTileKeys);
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
    e = launch_pdl(decode_kernel<128>, grid, dim3(kThreads), DecodeSmem<128>::kTotal, stream, a);
  } else {
    e = cudaFuncSetAttribute(decode_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DecodeSmem<64>::kTotal);
    if (e != cudaSuccess) return e;
    e = launch_pdl(decode_kernel<64>, grid, dim3(kThreads), DecodeSmem<64>::kTotal, stream, a);
  }
  return e;
}

static cudaError_t launch_decode_merge(const DecodeArgs &a, const PoolGeom &g, int32_t batch,
                                       int32_t sm_count, cudaStream_t stream) {
  const int64_t pairs = static_cast<int64_t>(batch) * a.hq;
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
