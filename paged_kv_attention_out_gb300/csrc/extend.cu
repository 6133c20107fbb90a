// extend.cu - paged extend (chunked-prefill) attention on tcgen05 / TMEM.
//
// What it computes ("Code Notes: mini-sglang", Scheduler Layer table,
// PrefillManager row; "Introduction", Key Features, Chunked Prefill and Radix
// Cache): request r's chunk of c_r new queries sits after a cached prefix of
// p_r = seq_len[r] - c_r keys; chunk query j attends to keys 0 .. p_r + j of
// the request's page_table row (full prefix, causal within the chunk).
//
// Tiling. A CTA owns one 128-row query tile of one kv head: 128 / g chunk
// tokens x the g q heads that read that kv head, so every gathered K/V tile
// feeds g heads. It walks the visible keys in tiles of 128:
//   S_j  = Q K_j^T            tcgen05.mma, M=128 N=128 K=D, fp32 in TMEM
//   P_j  = exp2(scale*S_j - m) softmax warps, one thread per query row, bf16
//                             into shared memory
//   O   += P_j V_j            tcgen05.mma, M=128 N=D K=128, fp32 in TMEM
// Roles (288 threads):
//   warps 0-3  softmax: thread r owns row r of S and O (TMEM lane r); online
//              softmax in the log2 domain with a lazy rescale (O is rescaled
//              only when the row max grows by more than 2^8), causal and
//              range masks only on tiles that cross a row's last key, then
//              the epilogue O / l -> bf16 and lse.
//   warp 4     TMEM allocation and the single MMA-issuing thread; S is
//              double-buffered in TMEM so QK^T of tile j+1 runs while the
//              softmax works on tile j.
//   warps 5-8  producers: gather K_j and V_j rows through the page table
//              with 16-byte cp.async into the SW128 shared layout (zero fill
//              past the end), two stages deep.
// Every hand-off is an mbarrier; every wait is bounded (tc_common.cuh).
#include <math.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"
#include "tc_common.cuh"

namespace pkv {
namespace {

constexpr int kM = 128;  // query rows per CTA
constexpr int kN = 128;  // keys per K/V tile
constexpr int kSoftmaxWarps = 8;  // two per SM sub-partition: a row's columns are split
constexpr int kMmaWarp = kSoftmaxWarps;
constexpr int kProducerWarps = 4;
constexpr int kProducerBase = (kSoftmaxWarps + 1) * 32;
constexpr int kThreads = (kSoftmaxWarps + 1 + kProducerWarps) * 32;
constexpr int kProducers = kProducerWarps * 32;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct Smem {
  static constexpr int kQ = 0;
  static constexpr int kQBytes = kM * D * 2;
  static constexpr int kTileBytes = kN * D * 2;
  static constexpr int kKV = kQ + kQBytes;  // stage s: K at kKV + s*2*tile, V after it
  static constexpr int kP = kKV + 4 * kTileBytes;
  static constexpr int kPBytes = kM * kN * 2;
  static constexpr int kBars = kP + kPBytes;
  static constexpr int kBarCount = 17;
  // + alignment slack; never below 116 KB, so one CTA (and one 512-column
  // TMEM allocation) per SM even for head_dim 64
  static constexpr int kNeed = kBars + kBarCount * 8 + 16 + 1024;
  static constexpr int kTotal = kNeed > 116 * 1024 ? kNeed : 116 * 1024;
};

// TMEM columns: S buffers at 0 and 128, O at 256.
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemO = 256;

// Barrier indices.
enum : int {
  kBarKFull = 0,   // [2] producers: K tile landed
  kBarVFull = 2,   // [2] producers: V tile landed
  kBarKVEmpty = 4, // [2] MMA: stage consumed (after PV)
  kBarSFull = 6,   // [2] MMA: S tile ready
  kBarSFree = 8,   // [2] softmax: S tile read
  kBarPFull = 10,  // softmax: P written
  kBarODone = 11,  // MMA: PV finished
  kBarTeardown = 12,  // MMA: everything issued has finished (abort path)
  kBarPair = 13,      // [4] softmax: the two warps of a lane quarter exchanged a value
};

struct ExtendArgs {
  const __nv_bfloat16 *pool;
  int64_t plane;
  int64_t slots;
  int32_t num_layers;
  int32_t layer;
  int32_t page_size;
  int32_t hkv;
  const __nv_bfloat16 *q;
  const int32_t *qo_indptr;
  __nv_bfloat16 *o;
  float *lse;
  const int32_t *page_table;
  int64_t table_stride;
  const int32_t *table_idx;
  const int32_t *seq_lens;
  int32_t batch;
  int32_t total_q;
  int32_t hq;
  int32_t group;
  int32_t tokens_per_cta;  // floor(128 / group)
  float scale_log2;
  unsigned *err;
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) extend_tc_kernel(const ExtendArgs a) {
  using S = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_req, s_j0, s_c, s_p, s_row;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float s_pair[2][2][kM];  // [parity][column half][row] values exchanged in a pair
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int kvh = blockIdx.x;

  grid_dependency_wait();  // the chunk's K/V may come from the previous kernel (store_kv)
  if (tid == 0) {
    // Which (request, token tile) this CTA owns; tiles are taken from the end.
    const int tile = static_cast<int>(gridDim.y) - 1 - static_cast<int>(blockIdx.y);
    int acc = 0;
    int req = -1, j0 = 0, c = 0, p = 0, row = 0;
    for (int r = 0; r < a.batch; ++r) {
      const int beg = a.qo_indptr[r];
      const int end = a.qo_indptr[r + 1];
      const int cr = end - beg;
      if (cr < 0 || end > a.total_q || beg < 0) {
        if (kvh == 0 && blockIdx.y == 0) flag_error(a.err, kErrIndptr);
        break;
      }
      const int nt = (cr + a.tokens_per_cta - 1) / a.tokens_per_cta;
      if (tile < acc + nt) {
        req = r;
        j0 = (tile - acc) * a.tokens_per_cta;
        c = cr;
        p = a.seq_lens[r] - cr;
        row = a.table_idx ? a.table_idx[r] : r;
        break;
      }
      acc += nt;
    }
    if (req >= 0) {
      const int64_t max_keys = a.table_stride * a.page_size;
      if (p < 0 || static_cast<int64_t>(p) + c > max_keys || row < 0) {
        if (kvh == 0) {
          flag_error(a.err, p < 0 ? kErrIndptr : (row < 0 ? kErrTableIdx : kErrSeqLen));
        }
        req = -1;
      }
    }
    s_req = req;
    s_j0 = j0;
    s_c = c;
    s_p = p;
    s_row = row;
    s_abort = 0;
  }
  __syncthreads();
  const int req = s_req;
  if (req < 0) return;

  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bars = sbase + S::kBars;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  volatile int *abort = &s_abort;

  const int j0 = s_j0, c = s_c, p = s_p;
  const int32_t *row_pages = a.page_table + static_cast<int64_t>(s_row) * a.table_stride;
  const int t_base = a.qo_indptr[req];
  const int tokens = min(a.tokens_per_cta, c - j0);
  const int n_keys = p + j0 + tokens;  // keys the last token of the tile sees
  const int n_tiles = (n_keys + kN - 1) / kN;

  if (tid == 0) {
    mbar_init(bar(kBarKFull + 0), kProducers);
    mbar_init(bar(kBarKFull + 1), kProducers);
    mbar_init(bar(kBarVFull + 0), kProducers);
    mbar_init(bar(kBarVFull + 1), kProducers);
    mbar_init(bar(kBarKVEmpty + 0), 1);
    mbar_init(bar(kBarKVEmpty + 1), 1);
    mbar_init(bar(kBarSFull + 0), 1);
    mbar_init(bar(kBarSFull + 1), 1);
    mbar_init(bar(kBarSFree + 0), kSoftmaxWarps * 32);
    mbar_init(bar(kBarSFree + 1), kSoftmaxWarps * 32);
    mbar_init(bar(kBarPFull), kSoftmaxWarps * 32);
    mbar_init(bar(kBarODone), 1);
    mbar_init(bar(kBarTeardown), 1);
    for (int q = 0; q < 4; ++q) mbar_init(bar(kBarPair + q), 64);
    mbar_init_fence();
  }
  if (warp == kMmaWarp) tmem_alloc(smem_addr(&s_tmem), kTmemCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = s_tmem;

  if (warp >= kSoftmaxWarps + 1) {
    // ------------------------------------------------------------ producers
    const int pt = tid - kProducerBase;
    constexpr int CPK = D / 8;                 // 16-byte chunks per row
    constexpr int kRowsPerPass = kProducers / CPK;
    constexpr int kPasses = kN / kRowsPerPass;  // rows handled per thread per tile
    const int ch = pt % CPK;
    const int r0 = pt / CPK;
    const int64_t slot_stride = static_cast<int64_t>(a.hkv) * D;
    const __nv_bfloat16 *kbase =
        a.pool + static_cast<int64_t>(a.layer) * a.plane + static_cast<int64_t>(kvh) * D + ch * 8;
    const __nv_bfloat16 *vbase = a.pool + (static_cast<int64_t>(a.num_layers) + a.layer) * a.plane +
                                 static_cast<int64_t>(kvh) * D + ch * 8;
    const int P = a.page_size;
    // Q tile: row r -> token j0 + r / g, q head kvh * g + r % g.
    for (int i = 0; i < kM / kRowsPerPass; ++i) {
      const int r = r0 + i * kRowsPerPass;
      const int t = r / a.group, hh = r % a.group;
      const bool ok = t < tokens;
      const __nv_bfloat16 *src =
          ok ? a.q + (static_cast<int64_t>(t_base + j0 + t) * a.hq + kvh * a.group + hh) * D + ch * 8
             : a.q;
      cp_async_16(sbase + S::kQ + sw128_offset(kM, r, ch * 8), src, ok ? 16 : 0);
    }
    cp_async_commit();
    // Page-table entries of this thread's rows, loaded one tile ahead.
    int entry[kPasses];
#pragma unroll
    for (int i = 0; i < kPasses; ++i) {
      const int key = r0 + i * kRowsPerPass;
      entry[i] = key < n_keys ? __ldg(row_pages + ((P == 1) ? key : key / P)) : -1;
    }
    for (int j = 0; j < n_tiles; ++j) {
      const int s = j & 1;
      if (j >= 2 && !mbar_wait(bar(kBarKVEmpty + s), ((j >> 1) - 1) & 1, abort)) {
        *abort = 1;
        break;
      }
      int64_t off[kPasses];
#pragma unroll
      for (int i = 0; i < kPasses; ++i) {
        const int key = j * kN + r0 + i * kRowsPerPass;
        const long long sl = static_cast<long long>(entry[i]) * P + ((P == 1) ? 0 : key % P);
        const bool ok = key < n_keys && entry[i] >= 0 && sl < a.slots;
        if (key < n_keys && !ok) flag_error(a.err, kErrPage);
        off[i] = ok ? sl * slot_stride : -1;
        const int nkey = key + kN;  // same row of tile j + 1
        entry[i] = nkey < n_keys ? __ldg(row_pages + ((P == 1) ? nkey : nkey / P)) : -1;
      }
      const uint32_t kst = sbase + S::kKV + s * 2 * S::kTileBytes;
      const uint32_t vst = kst + S::kTileBytes;
#pragma unroll
      for (int i = 0; i < kPasses; ++i) {
        const int r = r0 + i * kRowsPerPass;
        cp_async_16(kst + sw128_offset(kN, r, ch * 8), off[i] >= 0 ? kbase + off[i] : a.pool,
                    off[i] >= 0 ? 16 : 0);
      }
      cp_async_commit();
#pragma unroll
      for (int i = 0; i < kPasses; ++i) {
        const int r = r0 + i * kRowsPerPass;
        cp_async_16(vst + sw128_offset(kN, r, ch * 8), off[i] >= 0 ? vbase + off[i] : a.pool,
                    off[i] >= 0 ? 16 : 0);
      }
      cp_async_commit();
      cp_async_wait<1>();  // K_j (and V_{j-1}, Q) landed
      fence_async_shared();
      mbar_arrive(bar(kBarKFull + s));
      if (j >= 1) mbar_arrive(bar(kBarVFull + (s ^ 1)));
    }
    cp_async_wait<0>();
    fence_async_shared();
    if (!*abort && n_tiles > 0) mbar_arrive(bar(kBarVFull + ((n_tiles - 1) & 1)));
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = umma_idesc_bf16(kM, kN, 0, 0);
      constexpr uint32_t idesc_pv = umma_idesc_bf16(kM, D, 0, 1);
      auto pv = [&](int i) -> bool {
        const int s = i & 1;
        if (!mbar_wait(bar(kBarPFull), i & 1, abort)) return false;
        if (!mbar_wait(bar(kBarVFull + s), (i >> 1) & 1, abort)) return false;
        tc_fence_after_sync();
        const uint32_t vst = sbase + S::kKV + s * 2 * S::kTileBytes + S::kTileBytes;
#pragma unroll
        for (int ks = 0; ks < kN / 16; ++ks) {
          const uint64_t da = umma_desc_sw128(sbase + S::kP + (ks >> 2) * (kM * 128) + (ks & 3) * 32, 16, 1024);
          const uint64_t db = umma_desc_sw128(vst + ks * 2048, kN * 128, 1024);
          umma_bf16_ss(tmem + kTmemO, da, db, idesc_pv, (i > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit(bar(kBarODone));
        umma_commit(bar(kBarKVEmpty + s));
        return true;
      };
      bool ok = true;
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int s = j & 1;
        ok = mbar_wait(bar(kBarKFull + s), (j >> 1) & 1, abort);
        if (ok && j >= 2) ok = mbar_wait(bar(kBarSFree + s), ((j >> 1) - 1) & 1, abort);
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t kst = sbase + S::kKV + s * 2 * S::kTileBytes;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t da = umma_desc_sw128(sbase + S::kQ + (ks >> 2) * (kM * 128) + (ks & 3) * 32, 16, 1024);
          const uint64_t db = umma_desc_sw128(kst + (ks >> 2) * (kN * 128) + (ks & 3) * 32, 16, 1024);
          umma_bf16_ss(tmem + kTmemS + s * kN, da, db, idesc_qk, ks > 0 ? 1u : 0u);
        }
        umma_commit(bar(kBarSFull + s));
        if (j >= 1) ok = pv(j - 1);
      }
      if (ok && n_tiles > 0) ok = pv(n_tiles - 1);
      if (!ok) {
        *abort = 1;
        flag_error(a.err, kErrTimeout);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    // Warp w owns TMEM lanes 32 * (w % 4) .. + 31 (query rows) and half
    // hc = w / 4 of the key columns of each S tile (and of the O columns).
    // The two warps of a lane quarter combine their row maxima through
    // s_pair and an mbarrier each tile.
    const int quarter = warp & 3;
    const int hc = warp >> 2;
    const int r = quarter * 32 + lane;  // query row == TMEM lane
    const int t = r / a.group;
    const bool valid = t < tokens;
    const int limit = p + j0 + (valid ? t : 0);  // last key this row may see
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    constexpr int kCols = kN / 2;  // S columns (keys) per thread
    constexpr int kOCols = D / 2;  // O columns per thread
    const uint32_t pair_bar = bar(kBarPair + quarter);
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    int pair_phase = 0;
    // Exchange one float with the partner warp (bounded wait; warp-uniform ok).
    auto exchange = [&](float mine, bool &good) -> float {
      float *slot = s_pair[pair_phase & 1][0];
      slot[hc * kM + r] = mine;
      mbar_arrive(pair_bar);
      good = mbar_wait_warp(pair_bar, pair_phase & 1, abort);
      const float other = good ? slot[(hc ^ 1) * kM + r] : mine;
      ++pair_phase;
      return other;
    };
    for (int j = 0; j < n_tiles && ok; ++j) {
      const int s = j & 1;
      if (!(ok = mbar_wait_warp(bar(kBarSFull + s), (j >> 1) & 1, abort))) break;
      tc_fence_after_sync();
      const int key0 = j * kN + hc * kCols;
      const bool full = key0 + kCols - 1 <= limit;
      float v[kCols];
      {
        float a0[32], a1[32];
        tmem_ld32(tmem + lane_base + kTmemS + s * kN + hc * kCols, a0);
        tmem_ld32(tmem + lane_base + kTmemS + s * kN + hc * kCols + 32, a1);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          v[i] = a0[i];
          v[32 + i] = a1[i];
        }
      }
      tc_fence_before_sync();
      mbar_arrive(bar(kBarSFree + s));  // S tile read: QK^T of tile j + 2 may overwrite it
      if (!full) {
#pragma unroll
        for (int i = 0; i < kCols; ++i)
          if (key0 + i > limit) v[i] = -INFINITY;
      }
      // Row max of the raw scores (scale > 0 commutes with max), 8 chains.
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = v[k];
#pragma unroll
      for (int i = 8; i < kCols; ++i) mx[i & 7] = fmaxf(mx[i & 7], v[i]);
      float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                       fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      mt = fmaxf(mt, exchange(mt, ok));
      if (!ok) break;
      mt *= a.scale_log2;
      if (j >= 1) {
        if (!(ok = mbar_wait_warp(bar(kBarODone), (j - 1) & 1, abort))) break;
        tc_fence_after_sync();
      }
      if (j == 0) {
        m_used = mt;  // first tile: key 0 is always visible, so mt is finite
      } else if (__any_sync(0xffffffffu, mt > m_used + kRescaleThreshold)) {
        // Warp-uniform (tcgen05.ld/st are .sync.aligned): every lane rescales
        // its row by its own factor, 1 where the row max did not move.
        const float m_new = fmaxf(m_used, mt);
        const float f = fast_exp2(m_used - m_new);
        l *= f;
        m_used = m_new;
#pragma unroll 1
        for (int cb = 0; cb < kOCols / 16; ++cb) {
          float o[16];
          const uint32_t oaddr = tmem + lane_base + kTmemO + hc * kOCols + cb * 16;
          tmem_ld16(oaddr, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] *= f;
          tmem_st16(oaddr, o);
        }
        tmem_st_wait();
      }
      // P = exp2(s * scale - m) as bf16 into P region hc (keys hc*64 .. +63).
      const float neg_m = -m_used;
      float sum[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) sum[k] = 0.f;
      const uint32_t prow = sbase + S::kP;
#pragma unroll
      for (int c8 = 0; c8 < kCols / 8; ++c8) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i0 = c8 * 8 + 2 * e;
          const float p0 = fast_exp2(fmaf(v[i0], a.scale_log2, neg_m));
          const float p1 = fast_exp2(fmaf(v[i0 + 1], a.scale_log2, neg_m));
          sum[(2 * e) & 7] += p0;
          sum[(2 * e + 1) & 7] += p1;
          w[e] = pack_bf16(p0, p1);
        }
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                         prow + sw128_offset(kM, r, hc * kCols + c8 * 8)),
                     "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                     : "memory");
      }
      l += ((sum[0] + sum[1]) + (sum[2] + sum[3])) + ((sum[4] + sum[5]) + (sum[6] + sum[7]));
      fence_async_shared();
      tc_fence_before_sync();
      mbar_arrive(bar(kBarPFull));
    }
    if (ok) l += exchange(l, ok);  // row sum over both column halves
    if (ok && n_tiles > 0) ok = mbar_wait_warp(bar(kBarODone), (n_tiles - 1) & 1, abort);
    if (!ok) {
      *abort = 1;
      flag_error(a.err, kErrTimeout);
    } else {
      tc_fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int64_t orow =
          static_cast<int64_t>(t_base + j0 + t) * a.hq + kvh * a.group + (r % a.group);
#pragma unroll
      for (int cb = 0; cb < kOCols / 32; ++cb) {
        float o[32];
        tmem_ld32(tmem + lane_base + kTmemO + hc * kOCols + cb * 32, o);
        tmem_ld_wait();
        if (valid) {
          uint4 *dst = reinterpret_cast<uint4 *>(a.o + orow * D + hc * kOCols + cb * 32);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 u;
            u.x = pack_bf16(o[q4 * 8 + 0] * inv, o[q4 * 8 + 1] * inv);
            u.y = pack_bf16(o[q4 * 8 + 2] * inv, o[q4 * 8 + 3] * inv);
            u.z = pack_bf16(o[q4 * 8 + 4] * inv, o[q4 * 8 + 5] * inv);
            u.w = pack_bf16(o[q4 * 8 + 6] * inv, o[q4 * 8 + 7] * inv);
            dst[q4] = u;
          }
        }
      }
      if (valid && hc == 0 && a.lse)
        a.lse[orow] = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
    }
  }

  // Teardown: every role has left its loop (normally or through the abort
  // flag); wait for this thread's copies, then free TMEM once no MMA is in
  // flight (the MMA thread's last commit was waited on by the softmax, or
  // the abort path below waits for it).
  cp_async_wait<0>();
  if (warp == kMmaWarp && lane == 0 && *abort) {
    // Tracks every MMA this thread issued; they need no other input to finish.
    umma_commit(bar(kBarTeardown));
    int never = 0;
    mbar_wait(bar(kBarTeardown), 0, &never);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_extend(const PoolGeom &g, int32_t layer, const void *q,
                          const int32_t *qo_indptr, void *o, float *lse,
                          const int32_t *page_table, int64_t table_stride,
                          const int32_t *table_idx, const int32_t *seq_lens, int32_t batch,
                          int32_t total_q, int32_t hq, float scale, int32_t sm_count,
                          unsigned *err, cudaStream_t stream) {
  (void)sm_count;
  ExtendArgs a{};
  a.pool = static_cast<const __nv_bfloat16 *>(g.base);
  a.plane = g.plane;
  a.slots = g.slots;
  a.num_layers = g.num_layers;
  a.layer = layer;
  a.page_size = g.page_size;
  a.hkv = g.hkv;
  a.q = static_cast<const __nv_bfloat16 *>(q);
  a.qo_indptr = qo_indptr;
  a.o = static_cast<__nv_bfloat16 *>(o);
  a.lse = lse;
  a.page_table = page_table;
  a.table_stride = table_stride;
  a.table_idx = table_idx;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.total_q = total_q;
  a.hq = hq;
  a.group = hq / g.hkv;
  a.tokens_per_cta = kM / a.group;
  a.scale_log2 = scale * kLog2e;
  a.err = err;
  const int64_t tiles =
      (static_cast<int64_t>(total_q) + a.tokens_per_cta - 1) / a.tokens_per_cta + batch;
  if (tiles > 65535) return cudaErrorInvalidConfiguration;
  const dim3 grid(g.hkv, static_cast<unsigned>(tiles));
  cudaError_t e;
  if (g.d == 128) {
    e = cudaFuncSetAttribute(extend_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Smem<128>::kTotal);
    if (e != cudaSuccess) return e;
    e = launch_pdl(extend_tc_kernel<128>, grid, dim3(kThreads), Smem<128>::kTotal, stream, a);
  } else {
    e = cudaFuncSetAttribute(extend_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Smem<64>::kTotal);
    if (e != cudaSuccess) return e;
    e = launch_pdl(extend_tc_kernel<64>, grid, dim3(kThreads), Smem<64>::kTotal, stream, a);
  }
  return e;
}

}  // namespace pkv
