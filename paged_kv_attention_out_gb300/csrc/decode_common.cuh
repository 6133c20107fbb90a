// decode_common.cuh - the split-KV decode unit shared by the decode kernel
// (decode.cu) and the cascade kernel (cascade.cu): its arguments, shared
// memory layout, per-request facts and the body that attends one split of
// one request for one group of kv heads ("Code Notes: mini-sglang", Engine
// Layer table, BaseAttnBackend / BaseKVCachePool rows; Scheduler Layer
// table, TableManager row). The design notes are in decode.cu.
#pragma once

#include <math.h>

#include "pkv_common.cuh"

namespace pkv {

// Tuning constants of the decode unit (compile-time; the defaults are the
// measured best on GB300).
#ifndef PKV_DECODE_STAGES
#define PKV_DECODE_STAGES 2  // cp.async pipeline depth per warp
#endif
#ifndef PKV_KV_EVICT_FIRST
#define PKV_KV_EVICT_FIRST 1  // K/V tiles read with the L2 evict-first policy
#endif
#ifndef PKV_DECODE_WARPS
#define PKV_DECODE_WARPS 4  // warps per CTA (each on one kv head)
#endif

constexpr int kDecodeWarps = PKV_DECODE_WARPS;
constexpr int kDecodeThreads = kDecodeWarps * 32;
constexpr int kDecodeTileKeys = 16;
constexpr int kDecodeStages = PKV_DECODE_STAGES;

template <int D, int kSt = kDecodeStages>
struct DecodeSmem {
  static constexpr int kTileBytes = kDecodeTileKeys * D * 2;  // one K (or V) tile
  static constexpr int kStageBytes = 2 * kTileBytes;    // K + V
  static constexpr int kWarpBytes = kSt * kStageBytes;
  static constexpr int kTotal = kDecodeWarps * kWarpBytes;
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

__device__ __forceinline__ float decode_exp2(float x) {
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

// One decode unit: kv-head group hg (heads_per_cta kv heads), split `split`
// of request b, computed by kDecodeThreads threads (tid 0 .. kDecodeThreads - 1, whole
// warps) in `smem` (DecodeSmem<D, kSt>::kTotal bytes, 128-byte aligned);
// sync() is a barrier over exactly those threads.
template <int D, int kSt, typename Sync>
__device__ __forceinline__ void decode_body(const DecodeArgs &a, int hg, int split, int b,
                                            int tid, uint8_t *smem, Sync sync) {
  using S = DecodeSmem<D, kSt>;
  constexpr int kStages = kSt;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const RowInfo ri = row_info(a, b, split == 0 && hg == 0 && tid == 0);
  if (split >= ri.nsplit) return;
  if (a.k_new) {
    // Fused store: the split holding key seq - 1 writes the new token's K and
    // V rows of its kv heads first; no other CTA reads that key of these heads.
    if (split == ri.nsplit - 1 && ri.seq > 0) {
      const int pos = ri.seq - 1;
      const int pe = __ldg(ri.row + pos / a.page_size);
      const int64_t slot = static_cast<int64_t>(pe) * a.page_size + pos % a.page_size;
      if (pe < 0 || slot >= a.slots) {
        if (tid == 0) flag_error(a.err, kErrPage);
      } else {
        constexpr int kCh = D / 8;  // 16-byte chunks per head row
        for (int i = tid; i < a.heads_per_cta * 2 * kCh; i += kDecodeThreads) {
          const int ch = i % kCh;
          const int c = (i / kCh) & 1;
          const int h = hg * a.heads_per_cta + i / kCh / 2;
          const __nv_bfloat16 *src =
              (c ? a.v_new : a.k_new) + static_cast<int64_t>(b) * a.kv_row_stride + h * D + ch * 8;
          __nv_bfloat16 *dst = a.pool_w + (static_cast<int64_t>(c) * a.num_layers + a.layer) * a.plane +
                               slot * a.hkv * D + h * D + ch * 8;
          *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
        }
      }
      __threadfence();  // visible to this CTA's copies (and the GPU) before they read it
    }
    sync();
  }
  const int key_begin = split * a.chunk;
  const int key_end = (split == ri.nsplit - 1) ? ri.seq : key_begin + a.chunk;

  const int head_slot = warp % a.heads_per_cta;
  const int sub = warp / a.heads_per_cta;
  const int kvh = hg * a.heads_per_cta + head_slot;
  const int ntiles = (key_end - key_begin + kDecodeTileKeys - 1) / kDecodeTileKeys;
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
  // Each K/V byte is read once: its L2 lines go first (the partial states
  // the merge reads back and the page-table rows stay).
  const uint64_t kv_policy = PKV_KV_EVICT_FIRST ? l2_evict_first_policy() : 0ull;

  // Page-table entry of this lane's key of warp tile j (lanes 0..15), or -1
  // past the end. Loaded one tile before its copies are issued, so the index
  // load is off the critical path of the copy stream.
  auto load_entry = [&](int j) -> int {
    int e = -1;
    if (lane < kDecodeTileKeys && j < my_tiles) {
      const int key = key_begin + (sub + j * a.warps_per_head) * kDecodeTileKeys + lane;
      if (key < key_end) e = __ldg(ri.row + ((P == 1) ? key : key / P));
    }
    return e;
  };
  auto issue = [&](int j, int entry, int stage) {
    const int k0 = key_begin + (sub + j * a.warps_per_head) * kDecodeTileKeys;
    long long slot = -1;
    if (lane < kDecodeTileKeys && k0 + lane < key_end) {
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
    for (int it = 0; it < kDecodeTileKeys / KPI; ++it) {
      const int r = it * KPI + lane / CPK;
      const long long s = __shfl_sync(0xffffffffu, slot, r);
      const bool ok = s >= 0;
      const int64_t off = ok ? s * slot_stride + chunk * 8 : 0;
      const uint32_t dk = st + swz<D>(r, chunk);
      if (PKV_KV_EVICT_FIRST) {
        cp_async_16_hint(dk, ok ? kbase + off : a.pool, ok ? 16 : 0, kv_policy);
        cp_async_16_hint(dk + S::kTileBytes, ok ? vbase + off : a.pool, ok ? 16 : 0, kv_policy);
      } else {
        cp_async_16(dk, ok ? kbase + off : a.pool, ok ? 16 : 0);
        cp_async_16(dk + S::kTileBytes, ok ? vbase + off : a.pool, ok ? 16 : 0);
      }
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
    const int k0 = key_begin + (sub + j * a.warps_per_head) * kDecodeTileKeys;

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
    const float al0 = decode_exp2(m0 - ref0);
    const float al1 = decode_exp2(m1 - ref1);
    const float p0 = decode_exp2(s[0] - ref0);
    const float p1 = decode_exp2(s[1] - ref1);
    const float p2 = decode_exp2(s[2] - ref0);
    const float p3 = decode_exp2(s[3] - ref1);
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
  sync();

  // Merge the warps that share a kv head; write the final or the partial state.
  const bool final_out = ri.nsplit == 1 && !a.force_partial;
  const int items = a.heads_per_cta * a.group * (D / 4);
  for (int it = tid; it < items; it += kDecodeThreads) {
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
      const float sc = decode_exp2(base[8 * D + n] - ref);
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
    const int h = (hg * a.heads_per_cta + hs) * a.group + n;
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
}

}  // namespace pkv
