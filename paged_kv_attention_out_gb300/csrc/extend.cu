// extend.cu - paged extend (chunked-prefill) attention on tcgen05 / TMEM / TMA.
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
//   P_j  = exp2(scale*S_j - m) softmax warps, bf16 into one of two shared
//                             P buffers (the softmax runs a tile ahead of PV)
//   O   += P_j V_j            tcgen05.mma, M=128 N=D K=128, fp32 in TMEM
// Roles (416 threads):
//   warps 0-7  softmax: warp w owns TMEM lanes 32 (w % 4) .. + 31 (query
//              rows) and half w / 4 of each row's key columns; online
//              softmax in the log2 domain with a lazy rescale (O is rescaled
//              only when a row max grows by more than 2^8), masks only on
//              tiles that cross a row's last key, then O / l -> bf16 and lse.
//   warp 8     TMEM allocation and the single MMA-issuing thread; S is
//              double-buffered in TMEM so QK^T of tile j+1 runs while the
//              softmax works on tile j.
//   warps 9-12 producers: TMA tile::gather4 loads (4 rows per instruction,
//              128-byte swizzle, zeros for keys past the end) of the Q rows
//              and, through the page table, of the K rows (warps 9-10) and V
//              rows (warps 11-12) of each tile. TMA issue is serialised per
//              warp, so four warps issue; a K buffer is refilled once its
//              QK^T is done, a V buffer once its PV is done.
// Every hand-off is an mbarrier; every wait is bounded (tc_common.cuh).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "pkv_common.cuh"
#include "pkv_internal.h"
#include "tc_common.cuh"

namespace pkv {
namespace {

constexpr int kM = 128;  // query rows per CTA
constexpr int kN = 128;  // keys per K/V tile
constexpr int kSoftmaxWarps = 8;  // two per SM sub-partition: a row's columns are split
constexpr int kMmaWarp = kSoftmaxWarps;
constexpr int kProducerWarp = kSoftmaxWarps + 1;  // warps +0, +1: K (and Q); +2, +3: V
constexpr int kProducerWarps = 4;
constexpr int kThreads = (kSoftmaxWarps + 1 + kProducerWarps) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct Smem {
  static constexpr int kQ = 0;
  static constexpr int kQBytes = kM * D * 2;
  static constexpr int kTileBytes = kN * D * 2;
  static constexpr int kKV = kQ + kQBytes;  // stage s: K at kKV + s*2*tile, V after it
  static constexpr int kP = kKV + 4 * kTileBytes;  // P buffer b at kP + b * kPBytes
  static constexpr int kPBytes = kM * kN * 2;
  static constexpr int kBars = kP + 2 * kPBytes;
  // + alignment slack; never below 116 KB, so one CTA (and one 512-column
  // TMEM allocation) per SM even for head_dim 64
  static constexpr int kNeed = kBars + 32 * 8 + 16 + 1024;
  static constexpr int kTotal = kNeed > 116 * 1024 ? kNeed : 116 * 1024;
};

// TMEM columns: S buffers at 0 and 128, O at 256, and 4 scratch columns at
// 384 where the two softmax warps of a lane quarter exchange row values.
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemO = 256;
constexpr uint32_t kTmemX = 384;

// Barrier indices. Every barrier that is waited on with a parity completes
// at most once between two waits of the same waiter (so a waiter is never
// two phases behind): per-buffer barriers for everything double-buffered.
enum : int {
  kBarKFull = 0,      // [2] producers: K tile landed (TMA bytes)
  kBarVFull = 2,      // [2] producers: V tile landed (TMA bytes)
  kBarKEmpty = 4,     // [2] MMA: K buffer consumed (after QK^T)
  kBarVEmpty = 6,     // [2] MMA: V buffer consumed (after PV)
  kBarSFull = 8,      // [2] MMA: S tile ready
  kBarSFree = 10,     // [2] softmax: S tile read
  kBarPFull = 12,     // [2] softmax: P buffer written
  kBarPFree = 14,     // [2] MMA: PV that read P buffer b finished (and all before it)
  kBarTeardown = 16,  // MMA: everything issued has finished (abort path)
  kBarPair = 17,      // [4] softmax: the two warps of a lane quarter exchanged a value
  kBarQFull = 21,     // producers: Q tile landed (TMA bytes)
  kBarCount = 22,
};

struct ExtendArgs {
  int64_t slots;         // pool slots per (c, layer) plane
  int32_t num_layers;
  int32_t layer;
  int32_t page_size;
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

// pool_map: the pool as a 2-D bf16 tensor [2 * L * slots rows][Hkv * D]
// (row (c * L + layer) * slots + slot); q_map: q as [total_q * Hq rows][D].
// Both with box {64, 1} and 128-byte swizzle.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    extend_tc_kernel(const __grid_constant__ CUtensorMap pool_map,
                     const __grid_constant__ CUtensorMap q_map, const ExtendArgs a) {
  using S = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_req, s_j0, s_c, s_p, s_row;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
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
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarKFull + i), 2);  // one expect_tx arrival per issuing warp
      mbar_init(bar(kBarVFull + i), 2);
      mbar_init(bar(kBarKEmpty + i), 1);
      mbar_init(bar(kBarVEmpty + i), 1);
      mbar_init(bar(kBarSFull + i), 1);
      mbar_init(bar(kBarSFree + i), kSoftmaxWarps * 32);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarPFull + i), kSoftmaxWarps * 32);
      mbar_init(bar(kBarPFree + i), 1);
    }
    mbar_init(bar(kBarTeardown), 1);
    for (int q = 0; q < 4; ++q) mbar_init(bar(kBarPair + q), 64);
    mbar_init(bar(kBarQFull), 2);
    mbar_init_fence();
  }
  if (warp == kMmaWarp) tmem_alloc(smem_addr(&s_tmem), kTmemCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = s_tmem;

  if (warp >= kProducerWarp) {
    // ------------------------------------------------------------ producers
    // Producer warp pw (0..3): pw 0-1 load Q and K tiles, pw 2-3 V tiles.
    // In a tile, warp w2 = pw & 1 covers row groups 16 w2 .. 16 w2 + 15
    // (4 rows each); lane l takes group 16 w2 + (l & 15) and 64-column half
    // l >> 4. Rows that must read as zero (past the end, bad page ids) get
    // row -1.
    const int pw = warp - kProducerWarp;
    const bool is_k = pw < 2;
    const int grp = 16 * (pw & 1) + (lane & 15);
    const int h = lane >> 4;
    constexpr int kHalves = D / 64;
    const bool active = h < kHalves;
    const int P = a.page_size;
    const int plane = (is_k ? 0 : a.num_layers) + a.layer;
    const int plane_base = plane * static_cast<int>(a.slots);
    const int xcol = kvh * D + h * 64;
    // destination of rows 4 grp .. 4 grp + 3 inside a SW128 region
    const uint32_t row_off =
        static_cast<uint32_t>(h * (kN * 128) + (grp >> 1) * 1024 + (grp & 1) * 512);
    constexpr uint32_t kWarpBytes = S::kTileBytes / 2;  // each of the two warps' share
    bool ok = true;
    if (is_k) {
      int qr[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = 4 * grp + e;
        const int t = r / a.group;
        qr[e] = t < tokens ? (t_base + j0 + t) * a.hq + kvh * a.group + (r % a.group) : -1;
      }
      if (lane == 0) mbar_arrive_expect_tx(bar(kBarQFull), S::kQBytes / 2);
      __syncwarp();
      if (active)
        tma_gather4(sbase + S::kQ + static_cast<uint32_t>(h * (kM * 128) + (grp >> 1) * 1024 +
                                                         (grp & 1) * 512),
                    &q_map, h * 64, qr[0], qr[1], qr[2], qr[3], bar(kBarQFull));
    }
    // Pool rows of this lane's 4 keys of tile j (-1 where the key is past
    // the end or its page id is out of range): one division per tile, then
    // the keys walk through the page.
    auto rows_of = [&](int j, int (&rr)[4]) {
      const int k0 = j * kN + 4 * grp;
      int pidx = k0 / P;
      int off = k0 - pidx * P;
      int ent = -1, ent_idx = -1;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (off == P) {
          ++pidx;
          off = 0;
        }
        rr[e] = -1;
        if (k0 + e < n_keys) {
          if (pidx != ent_idx) {
            ent = __ldg(row_pages + pidx);
            ent_idx = pidx;
          }
          const long long sl = static_cast<long long>(ent) * P + off;
          if (ent >= 0 && sl < a.slots) {
            rr[e] = plane_base + static_cast<int>(sl);
          } else if (is_k && h == 0) {
            flag_error(a.err, kErrPage);
          }
        }
        ++off;
      }
    };
    const int full_bar = is_k ? kBarKFull : kBarVFull;
    const int empty_bar = is_k ? kBarKEmpty : kBarVEmpty;
    const int buf_off = is_k ? 0 : S::kTileBytes;
    int rr[4];
    rows_of(0, rr);
    int issued = 0;
    for (int j = 0; j < n_tiles; ++j) {
      const int s = j & 1;
      if (j >= 2 && !(ok = mbar_wait_warp(bar(empty_bar + s), ((j >> 1) - 1) & 1, abort))) break;
      if (lane == 0) mbar_arrive_expect_tx(bar(full_bar + s), kWarpBytes);
      __syncwarp();
      if (active)
        tma_gather4(sbase + S::kKV + s * 2 * S::kTileBytes + buf_off + row_off, &pool_map, xcol,
                    rr[0], rr[1], rr[2], rr[3], bar(full_bar + s));
      ++issued;
      if (j + 1 < n_tiles) rows_of(j + 1, rr);
    }
    if (!ok) *abort = 1;
    if (*abort && lane == 0) {
      // Let every issued copy land before the CTA can exit: TMA writes to
      // this CTA's shared memory need no other input to finish.
      int never = 0;
      if (is_k) mbar_wait(bar(kBarQFull), 0, &never);
      for (int t = issued > 2 ? issued - 2 : 0; t < issued; ++t)
        mbar_wait(bar(full_bar + (t & 1)), (t >> 1) & 1, &never);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = umma_idesc_bf16(kM, kN, 0, 0);
      constexpr uint32_t idesc_pv = umma_idesc_bf16(kM, D, 0, 1);
      // Descriptors are built once; a k-step adds its byte offset / 16 to the
      // start-address field (addresses stay below 256 KB, so no carry).
      const uint64_t dq = umma_desc_sw128(sbase + S::kQ, 16, 1024);
      const uint64_t dp = umma_desc_sw128(sbase + S::kP, 16, 1024);
      const uint64_t dk0 = umma_desc_sw128(sbase + S::kKV, 16, 1024);
      const uint64_t dv0 = umma_desc_sw128(sbase + S::kKV + S::kTileBytes, kN * 128, 1024);
      constexpr uint64_t kStageStep = (2 * S::kTileBytes) >> 4;
      auto kstep = [](int ks, int rows) -> uint64_t {
        return static_cast<uint64_t>(((ks >> 2) * (rows * 128) + (ks & 3) * 32) >> 4);
      };
      auto pv = [&](int i) -> bool {
        const int s = i & 1;
        if (!mbar_wait(bar(kBarPFull + s), (i >> 1) & 1, abort)) return false;
        if (!mbar_wait(bar(kBarVFull + s), (i >> 1) & 1, abort)) return false;
        tc_fence_after_sync();
        const uint64_t dv = dv0 + s * kStageStep;
        const uint64_t dpb = dp + s * static_cast<uint64_t>(S::kPBytes >> 4);
#pragma unroll
        for (int ks = 0; ks < kN / 16; ++ks)
          umma_bf16_ss(tmem + kTmemO, dpb + kstep(ks, kM), dv + ks * (2048 >> 4), idesc_pv,
                       (i > 0 || ks > 0) ? 1u : 0u);
        umma_commit(bar(kBarPFree + s));
        umma_commit(bar(kBarVEmpty + s));
        return true;
      };
      bool ok = mbar_wait(bar(kBarQFull), 0, abort);
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int s = j & 1;
        ok = mbar_wait(bar(kBarKFull + s), (j >> 1) & 1, abort);
        if (ok && j >= 2) ok = mbar_wait(bar(kBarSFree + s), ((j >> 1) - 1) & 1, abort);
        if (!ok) break;
        tc_fence_after_sync();
        const uint64_t dk = dk0 + s * kStageStep;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          umma_bf16_ss(tmem + kTmemS + s * kN, dq + kstep(ks, kM), dk + kstep(ks, kN), idesc_qk,
                       ks > 0 ? 1u : 0u);
        umma_commit(bar(kBarSFull + s));
        umma_commit(bar(kBarKEmpty + s));
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
    // spare TMEM columns and an mbarrier each tile.
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
    // Exchange one float with the partner warp through a TMEM scratch column
    // (bounded wait; warp-uniform ok).
    auto exchange = [&](float mine, bool &good) -> float {
      const uint32_t col = tmem + lane_base + kTmemX + 2 * (pair_phase & 1);
      tmem_st1(col + hc, mine);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(pair_bar);
      good = mbar_wait_warp(pair_bar, pair_phase & 1, abort);
      float other = mine;
      if (good) {
        tc_fence_after_sync();
        other = tmem_ld1(col + (hc ^ 1));
        tmem_ld_wait();
      }
      ++pair_phase;
      return other;
    };
    for (int j = 0; j < n_tiles && ok; ++j) {
      const int s = j & 1;
      if (!(ok = mbar_wait_warp(bar(kBarSFull + s), (j >> 1) & 1, abort))) break;
      tc_fence_after_sync();
      const int key0 = j * kN + hc * kCols;
      const uint32_t srow = tmem + lane_base + kTmemS + s * kN + hc * kCols;
      // Pass 1: row max of the raw scores (scale > 0 commutes with max).
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
      for (int cb = 0; cb < kCols / 16; ++cb) {
        float v[16];
        tmem_ld16(srow + cb * 16, v);
        tmem_ld_wait();
        const int kb = key0 + cb * 16;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          mx[i & 3] = fmaxf(mx[i & 3], kb + i <= limit ? v[i] : -INFINITY);
      }
      float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      mt = fmaxf(mt, exchange(mt, ok));
      if (!ok) break;
      mt *= a.scale_log2;
      if (j == 0) {
        m_used = mt;  // first tile: key 0 is always visible, so mt is finite
      } else if (__any_sync(0xffffffffu, mt > m_used + kRescaleThreshold)) {
        // O may only change once every PV so far is done: PV_{j-1} finished
        // implies all earlier ones did (commits track all prior MMAs).
        if (!(ok = mbar_wait_warp(bar(kBarPFree + ((j - 1) & 1)), ((j - 1) >> 1) & 1, abort)))
          break;
        tc_fence_after_sync();
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
      // Pass 2: P = exp2(s * scale - m) as bf16 into region hc of P buffer
      // j & 1, once the PV that last read that buffer (tile j - 2) is done.
      if (j >= 2) {
        if (!(ok = mbar_wait_warp(bar(kBarPFree + s), ((j >> 1) - 1) & 1, abort))) break;
      }
      const float neg_m = -m_used;
      float sum[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t prow = sbase + S::kP + s * S::kPBytes;
#pragma unroll 1
      for (int cb = 0; cb < kCols / 16; ++cb) {
        float v[16];
        tmem_ld16(srow + cb * 16, v);
        tmem_ld_wait();
        const int kb = key0 + cb * 16;
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float p0 = kb + 2 * e <= limit ? fast_exp2(fmaf(v[2 * e], a.scale_log2, neg_m)) : 0.f;
          const float p1 =
              kb + 2 * e + 1 <= limit ? fast_exp2(fmaf(v[2 * e + 1], a.scale_log2, neg_m)) : 0.f;
          sum[(2 * e) & 3] += p0;
          sum[(2 * e + 1) & 3] += p1;
          w[e] = pack_bf16(p0, p1);
        }
        const int col = hc * kCols + cb * 16;
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(prow + sw128_offset(kM, r, col)),
                     "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                     : "memory");
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                         prow + sw128_offset(kM, r, col + 8)),
                     "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                     : "memory");
      }
      l += (sum[0] + sum[1]) + (sum[2] + sum[3]);
      tc_fence_before_sync();
      mbar_arrive(bar(kBarSFree + s));  // S tile read: QK^T of tile j + 2 may overwrite it
      fence_async_shared();
      mbar_arrive(bar(kBarPFull + s));
    }
    if (ok) l += exchange(l, ok);  // row sum over both column halves
    if (ok && n_tiles > 0)
      ok = mbar_wait_warp(bar(kBarPFree + ((n_tiles - 1) & 1)), ((n_tiles - 1) >> 1) & 1, abort);
    if (!ok) {
      *abort = 1;
      flag_error(a.err, kErrTimeout);
    } else {
      tc_fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int64_t orow =
          static_cast<int64_t>(t_base + j0 + t) * a.hq + kvh * a.group + (r % a.group);
#pragma unroll 1
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
  // flag); free TMEM once no MMA is in flight (the MMA thread's last commit
  // was waited on by the softmax, or the abort path below waits for it).
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

// cuTensorMapEncodeTiled from the driver, looked up once per process.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A 2-D bf16 tensor of `rows` rows of `cols` elements (row-major), read 4
// rows x 64 columns at a time with 128-byte swizzle; zeros outside.
bool gather_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, 1};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
  a.slots = g.slots;
  a.num_layers = g.num_layers;
  a.layer = layer;
  a.page_size = g.page_size;
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
  const uint64_t pool_rows = 2ull * static_cast<uint64_t>(g.num_layers) * g.slots;
  const uint64_t q_rows = static_cast<uint64_t>(total_q) * hq;
  if (pool_rows >= (1ull << 31) || q_rows >= (1ull << 31)) return cudaErrorInvalidValue;
  CUtensorMap pool_map, q_map;
  if (!gather_map(&pool_map, g.base, pool_rows, static_cast<uint64_t>(g.hkv) * g.d) ||
      !gather_map(&q_map, q, q_rows, static_cast<uint64_t>(g.d)))
    return cudaErrorInvalidValue;
  const int64_t tiles =
      (static_cast<int64_t>(total_q) + a.tokens_per_cta - 1) / a.tokens_per_cta + batch;
  if (tiles > 65535) return cudaErrorInvalidConfiguration;
  const dim3 grid(g.hkv, static_cast<unsigned>(tiles));
  cudaError_t e;
  if (g.d == 128) {
    e = cudaFuncSetAttribute(extend_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Smem<128>::kTotal);
    if (e != cudaSuccess) return e;
    e = launch_pdl(extend_tc_kernel<128>, grid, dim3(kThreads), Smem<128>::kTotal, stream,
                   pool_map, q_map, a);
  } else {
    e = cudaFuncSetAttribute(extend_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Smem<64>::kTotal);
    if (e != cudaSuccess) return e;
    e = launch_pdl(extend_tc_kernel<64>, grid, dim3(kThreads), Smem<64>::kTotal, stream,
                   pool_map, q_map, a);
  }
  return e;
}

}  // namespace pkv
