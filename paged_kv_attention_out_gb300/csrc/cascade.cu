// cascade.cu - the shared-prefix half of cascade decode: each group's prefix
// attended once for all of its member requests, on tcgen05 / TMEM, with the
// prefix K/V read straight from the paged pool.
//
// What it computes ("Introduction", Key Features, Radix Cache: requests that
// share a prefix share its KV entries; "Code Notes: mini-sglang", Scheduler
// Layer table, CacheManager row): for group k, whose prefix is the first
// prefix_lens[k] keys of row k of the prefix page table, every member request
// b and q head h, the attention state of q[b,h] over one key range of that
// prefix, as an fp32 partial state (o normalised over the range, natural-log
// lse) in the slot that the cascade's merge combines with b's suffix decode.
// A key range with no key gives o = 0, lse = -inf.
//
// Tiling. A CTA owns one query tile of 128 rows, up to 128 / g members x the
// g q heads that read one kv head (one TMEM lane per row), and one key range.
// Every 128-key K/V tile it loads feeds all 128 rows: 128 FLOPs per byte at
// g = 4 x 32 members, below the tensor core's ridge point, so the kernel is
// bound by the bytes it gathers, and it reads each prefix byte once per kv
// head with no staging copy. Per key tile j:
//   S  = Q K_j^T      tcgen05.mma SS, M=128 N=128 K=D, fp32 in TMEM
//   P  = exp2(scale*S - m), bf16 back into TMEM over S (softmax warps)
//   O += P V_j        tcgen05.mma TS, A = P from TMEM, M=128 N=D K=128
// Roles (288 threads):
//   warps 0-3  softmax: one query row per thread (TMEM lane), log2-domain
//              online softmax with a lazy rescale of O; a mask only on the
//              tile that holds the prefix's last key; then the partial state.
//   warp 4     TMEM allocation and the single MMA-issuing thread.
//   warps 5-8  producers: the members' Q rows once, then per key tile the K
//              and V rows of the kv head, gathered through the prefix page
//              table with 16-byte cp.async into 128-byte-swizzled shared
//              memory (three stages, all in flight). Each producer thread's
//              copies of a stage arrive on its barrier when they land
//              (cp.async.mbarrier.arrive); the MMA thread fences the async
//              proxy after its wait; a stage is refilled once the MMAs
//              reading it are done.
// Every hand-off is an mbarrier; every wait is bounded (tc_common.cuh).
#include <math.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"
#include "tc_common.cuh"

namespace pkv {
namespace {

constexpr int kM = 128;  // query rows per CTA (= TMEM lanes)
constexpr int kN = 128;  // keys per K/V tile
#ifndef PKV_PREFIX_STAGES
#define PKV_PREFIX_STAGES 3
#endif
constexpr int kStages = PKV_PREFIX_STAGES;
constexpr int kSoftmaxWarps = 4;
constexpr int kMmaWarp = kSoftmaxWarps;
constexpr int kProducerWarp0 = kSoftmaxWarps + 1;
#ifndef PKV_PREFIX_PRODUCER_WARPS
#define PKV_PREFIX_PRODUCER_WARPS 4
#endif
constexpr int kProducerWarps = PKV_PREFIX_PRODUCER_WARPS;
constexpr int kKeysPerWarp = kN / kProducerWarps;  // keys of a tile one producer warp copies
static_assert(kKeysPerWarp * kProducerWarps == kN && kKeysPerWarp <= 32, "producer split");
constexpr int kProducerThreads = kProducerWarps * 32;
constexpr int kThreads = (kSoftmaxWarps + 1 + kProducerWarps) * 32;
constexpr uint32_t kTmemCols = 256;  // S / P at columns 0 .. 127, O at 128 .. 128 + D - 1
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemO = 128;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
#ifndef PKV_PREFIX_EVICT_FIRST
#define PKV_PREFIX_EVICT_FIRST 1  // prefix K/V read with the L2 evict-first policy
#endif
#ifndef PKV_PREFIX_MAX_SPLITS
#define PKV_PREFIX_MAX_SPLITS 64  // key ranges per group at most
#endif

template <int D>
struct PrefixSmem {
  static constexpr int kQ = 0;
  static constexpr int kQBytes = kM * D * 2;
  static constexpr int kTileBytes = kN * D * 2;  // one K or V tile
  static constexpr int kKV = kQ + kQBytes;       // stage s: K at kKV + 2 s tile, V after it
  static constexpr int kBars = kKV + kStages * 2 * kTileBytes;
  static constexpr int kTotal = kBars + 16 * 8 + 1024;  // + barriers + alignment slack
};

enum : int {
  kBarFull = 0,                  // [kStages] producers: K and V of the stage landed
  kBarEmpty = kStages,           // [kStages] MMA: every MMA reading the stage done
  kBarQFull = 2 * kStages,       // producers: Q landed (and sign-folded)
  kBarSFull = 2 * kStages + 1,   // MMA: S ready (and every earlier MMA done)
  kBarPFull = 2 * kStages + 2,   // softmax: P written to TMEM (and O rescaled)
  kBarOFull = 2 * kStages + 3,   // MMA: every MMA done, O final
  kBarTeardown = 2 * kStages + 4,
};

struct PrefixArgs {
  const __nv_bfloat16 *pool;  // plane (c, layer) starts at ((c * L + layer) * slots) rows
  int64_t slots;
  int32_t num_layers;
  int32_t layer;
  int32_t page_size;
  int32_t hkv;
  const int32_t *prefix_table;
  int64_t prefix_stride;
  const int32_t *prefix_lens;
  const int32_t *member_indptr;
  const int32_t *members;
  int32_t num_groups;
  int32_t batch;
  const __nv_bfloat16 *q;
  int32_t hq;
  int32_t group;             // q heads per kv head
  int32_t members_per_tile;  // floor(128 / group)
  float scale_log2;          // |scale| log2(e) (log2(e) for scale 0), > 0
  int32_t q_mode;            // 0: q as given, 1: negated (scale < 0), 2: zeroed (scale 0)
  float *part_o;             // [B, Hq, pstride, D] fp32
  float *part_lse;           // [B, Hq, pstride] fp32
  int32_t pstride;
  int32_t pslot;       // slot of key range 0; range z writes slot pslot + z
  int32_t key_splits;  // key ranges per group (gridDim.z)
  unsigned *err;
};

// Block `rank` of the grid's y dimension: groups in order, each cut into
// blocks of members_per_tile members. One warp; returns the group (-1 past
// the last block), the block's first member index into `members`, the
// group's member end and its prefix length, all from one round of loads. A
// group whose member_indptr pair is malformed has no block.
struct BlockInfo {
  int group, first, end, plen;
};

__device__ BlockInfo locate_block(const PrefixArgs &a, int rank, bool report) {
  const int lane = threadIdx.x & 31;
  const int mpt = a.members_per_tile;
  int base = 0;
  BlockInfo out{-1, 0, 0, 0};
  for (int k0 = 0; k0 < a.num_groups; k0 += 32) {
    const int k = k0 + lane;
    int nb = 0, beg = 0, end = 0, plen = 0;
    if (k < a.num_groups) {
      beg = a.member_indptr[k];
      end = a.member_indptr[k + 1];
      plen = a.prefix_lens[k];
      if (beg < 0 || end < beg || end > a.batch) {
        if (report) flag_error(a.err, kErrIndptr);
      } else {
        nb = (end - beg + mpt - 1) / mpt;
      }
    }
    int inc = nb;  // inclusive scan over the 32 groups of this round
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += v;
    }
    const int total = __shfl_sync(0xffffffffu, inc, 31);
    if (rank < base + total) {  // warp-uniform
      const unsigned who = __ballot_sync(0xffffffffu, rank >= base + inc - nb && rank < base + inc);
      const int src = __ffs(who) - 1;
      const int start = __shfl_sync(0xffffffffu, base + inc - nb, src);
      out.group = k0 + src;
      out.first = __shfl_sync(0xffffffffu, beg, src) + (rank - start) * mpt;
      out.end = __shfl_sync(0xffffffffu, end, src);
      out.plen = __shfl_sync(0xffffffffu, plen, src);
      break;
    }
    base += total;
  }
  return out;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) cascade_prefix_kernel(const PrefixArgs a) {
  using S = PrefixSmem<D>;
  constexpr int kChunks = D / 8;  // 16-byte chunks per row
  extern __shared__ uint8_t smem_raw[];
  __shared__ BlockInfo s_blk;
  __shared__ int64_t s_qrow[kM];  // q_row() of every query row (producers)
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int kvh = blockIdx.x;
  const int z = blockIdx.z;

  // The pool and q may come from earlier kernels on the stream (store_kv);
  // once every CTA has passed this wait, the suffix decode may start.
  grid_dependency_wait();
  grid_dependents_launch();
  if (warp == 0) {
    const BlockInfo bi = locate_block(a, blockIdx.y, blockIdx.x == 0 && blockIdx.z == 0);
    if (lane == 0) {
      s_blk = bi;
      s_abort = 0;
    }
  }
  __syncthreads();
  const int k = s_blk.group;
  if (k < 0) return;
  const int beg = s_blk.first;                             // first member of the tile
  const int nm = min(a.members_per_tile, s_blk.end - beg);  // members in the tile
  int plen = s_blk.plen;
  const bool report = kvh == 0 && z == 0 && tid == 0;
  if (plen < 0 || plen > a.prefix_stride * a.page_size) {
    if (report) flag_error(a.err, kErrSeqLen);
    plen = 0;  // state of an empty prefix: the member keeps its suffix's result
  }
  // Key range z: tiles tile0 .. tile0 + n_tiles - 1 of the prefix.
  const int nk = (plen + kN - 1) / kN;
  const int per = (nk + a.key_splits - 1) / a.key_splits;
  const int tile0 = z * per;
  const int n_tiles = max(0, min(nk, tile0 + per) - tile0);
  const int32_t *prow = a.prefix_table + static_cast<int64_t>(k) * a.prefix_stride;

  // Query row r of the tile: member r / g, q head kvh * g + r % g; the row of
  // q and of the partial state, -1 for a padding row, -2 for a member index
  // outside the batch (skipped and flagged).
  auto q_row = [&](int r) -> int64_t {
    const int m = r / a.group;
    if (m >= a.members_per_tile || m >= nm) return -1;
    const int b = a.members[beg + m];
    if (b < 0 || b >= a.batch) return -2;
    return static_cast<int64_t>(b) * a.hq + kvh * a.group + r % a.group;
  };
  if (warp < kSoftmaxWarps && z == 0 && q_row(tid) == -2) flag_error(a.err, kErrIndptr);

  if (n_tiles == 0) {  // no key in this range: o = 0, lse = -inf
    if (warp < kSoftmaxWarps) {
      const int64_t bh = q_row(tid);
      if (bh >= 0) {
        const int64_t prow_o = bh * a.pstride + a.pslot + z;
        for (int d = 0; d < D; d += 4)
          *reinterpret_cast<float4 *>(a.part_o + prow_o * D + d) = make_float4(0.f, 0.f, 0.f, 0.f);
        a.part_lse[prow_o] = -INFINITY;
      }
    }
    return;
  }

  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bars = sbase + S::kBars;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  volatile int *abort = &s_abort;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarFull + s), kProducerThreads);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    mbar_init(bar(kBarQFull), kProducerThreads);
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarPFull), kSoftmaxWarps * 32);
    mbar_init(bar(kBarOFull), 1);
    mbar_init(bar(kBarTeardown), 1);
    mbar_init_fence();
  }
  if (warp == kMmaWarp) tmem_alloc(smem_addr(&s_tmem), kTmemCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = s_tmem;

  if (warp >= kProducerWarp0) {
    // ------------------------------------------------------------ producers
    const int pt = tid - kProducerWarp0 * 32;
    const int pw = pt >> 5;  // producer warp: keys kKeysPerWarp pw .. + kKeysPerWarp - 1 of a tile
    bool ok = true;
    const int64_t row_elems = static_cast<int64_t>(a.hkv) * D;
    const __nv_bfloat16 *kbase =
        a.pool + static_cast<int64_t>(a.layer) * a.slots * row_elems + kvh * D;
    const __nv_bfloat16 *vbase =
        a.pool + (static_cast<int64_t>(a.num_layers) + a.layer) * a.slots * row_elems + kvh * D;
    // The slot of this lane's key of tile j (lane l of warp pw holds key
    // kKeysPerWarp pw + l % kKeysPerWarp), -1 past the prefix or for a bad
    // page id.
    auto key_slot_of = [&](int j) -> long long {
      const int key = (tile0 + j) * kN + pw * kKeysPerWarp + lane % kKeysPerWarp;
      if (key >= plen) return -1;
      const int pidx = key / a.page_size;
      const int ent = __ldg(prow + pidx);
      const long long s = static_cast<long long>(ent) * a.page_size + (key - pidx * a.page_size);
      if (ent < 0 || s >= a.slots) {
        flag_error(a.err, kErrPage);
        return -1;
      }
      return s;
    };
    // The first tile's page entries and the rows' member ids are loaded
    // together, before any copy is issued (each copy's asm is a compiler
    // barrier, so loads placed between copies would run one after another).
    long long slot = key_slot_of(0);
    for (int r = pt; r < kM; r += kProducerThreads) s_qrow[r] = q_row(r);
    named_barrier_sync(1, kProducerThreads);
    // Q: 128 rows x kChunks chunks; consecutive threads take consecutive
    // chunks of a row (coalesced 16-byte pieces).
    for (int c = pt; c < kM * kChunks; c += kProducerThreads) {
      const int r = c / kChunks, ch = c % kChunks;
      const int64_t qr = s_qrow[r];
      cp_async_16(sbase + S::kQ + sw128_offset(kM, r, ch * 8),
                  qr >= 0 ? a.q + qr * D + ch * 8 : a.q, qr >= 0 ? 16 : 0);
    }
    if (a.q_mode != 0) {
      // Fold the softmax scale's sign into Q once its rows have landed: the
      // row max is taken on raw scores, which needs a positive scale (scale *
      // q.k = |scale| * (-q).k exactly; scale 0 makes every score 0, as q = 0
      // does). Each thread rewrites the chunks it copied.
      cp_async_wait_all();
      for (int c = pt; c < kM * kChunks; c += kProducerThreads) {
        const int r = c / kChunks, cq = c % kChunks;
        uint4 *p = reinterpret_cast<uint4 *>(smem + S::kQ + sw128_offset(kM, r, cq * 8));
        uint4 w = *p;
        if (a.q_mode == 1) {
          w.x ^= 0x80008000u;
          w.y ^= 0x80008000u;
          w.z ^= 0x80008000u;
          w.w ^= 0x80008000u;
        } else {
          w = make_uint4(0u, 0u, 0u, 0u);
        }
        *p = w;
      }
      fence_async_shared();
      mbar_arrive(bar(kBarQFull));
    } else {
      cp_async_mbar_arrive(bar(kBarQFull));  // arrives once this thread's Q copies land
    }
    // K/V tiles: every stage in flight at once. A thread's arrive on a stage's
    // barrier fires when all its copies so far have landed; the MMA thread
    // makes them visible to the tensor core with a proxy fence after its wait.
    constexpr int kKeysPerInstr = 32 / kChunks;  // keys one warp instruction covers
    const int ch = lane % kChunks;
    // each prefix byte is read once per call: its L2 lines go first
    const uint64_t kv_policy = PKV_PREFIX_EVICT_FIRST ? l2_evict_first_policy() : 0ull;
    for (int j = 0; j < n_tiles; ++j) {
      const int s = j % kStages;
      if (j >= kStages &&
          !(ok = mbar_wait_warp(bar(kBarEmpty + s), ((j / kStages) - 1) & 1, abort)))
        break;
      const uint32_t kst = sbase + S::kKV + s * 2 * S::kTileBytes;
#pragma unroll
      for (int it = 0; it < kKeysPerWarp / kKeysPerInstr; ++it) {
        const int kl = it * kKeysPerInstr + lane / kChunks;  // key within this warp's share
        const long long sl = __shfl_sync(0xffffffffu, slot, kl);
        const int kk = pw * kKeysPerWarp + kl;  // key within the tile
        const bool kv_ok = sl >= 0;
        const int64_t off = kv_ok ? sl * row_elems + ch * 8 : 0;
        const uint32_t dst = kst + sw128_offset(kN, kk, ch * 8);
        if (PKV_PREFIX_EVICT_FIRST) {
          cp_async_16_hint(dst, kv_ok ? kbase + off : a.pool, kv_ok ? 16 : 0, kv_policy);
          cp_async_16_hint(dst + S::kTileBytes, kv_ok ? vbase + off : a.pool, kv_ok ? 16 : 0,
                           kv_policy);
        } else {
          cp_async_16(dst, kv_ok ? kbase + off : a.pool, kv_ok ? 16 : 0);
          cp_async_16(dst + S::kTileBytes, kv_ok ? vbase + off : a.pool, kv_ok ? 16 : 0);
        }
      }
      cp_async_mbar_arrive(bar(kBarFull + s));
      if (j + 1 < n_tiles) slot = key_slot_of(j + 1);  // next tile's page entry, off the copy path
    }
    cp_async_wait_all();  // every copy has landed before the CTA may exit
    if (!ok) *abort = 1;
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // S(0); then per tile j >= 1: PV(j - 1) once P(j - 1) is in TMEM, S(j)
    // once tile j has landed. tcgen05.mma ops of one thread run in issue
    // order, so S(j) overwrites P(j - 1) only after PV(j - 1) has read it,
    // and a completed S(j) implies a completed PV(j - 1) (O is then stable).
    if (lane == 0) {
      constexpr uint32_t idesc_qk = umma_idesc_bf16(kM, kN, 0, 0);
      constexpr uint32_t idesc_pv = umma_idesc_bf16(kM, D, 0, 1);
      const uint64_t dq = umma_desc_sw128(sbase + S::kQ, 16, 1024);
      const uint64_t dk0 = umma_desc_sw128(sbase + S::kKV, 16, 1024);
      const uint64_t dv0 = umma_desc_sw128(sbase + S::kKV + S::kTileBytes, kN * 128, 1024);
      constexpr uint64_t kStageStep = (2 * S::kTileBytes) >> 4;
      auto kstep = [](int ks, int rows) -> uint64_t {
        return static_cast<uint64_t>(((ks >> 2) * (rows * 128) + (ks & 3) * 32) >> 4);
      };
      auto qk = [&](int j) {
        const uint64_t dk = dk0 + (j % kStages) * kStageStep;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          umma_bf16_ss(tmem + kTmemS, dq + kstep(ks, kM), dk + kstep(ks, kN), idesc_qk,
                       ks > 0 ? 1u : 0u);
        umma_commit(bar(kBarSFull));
      };
      auto pv = [&](int j) {
        const uint64_t dv = dv0 + (j % kStages) * kStageStep;
#pragma unroll
        for (int ks = 0; ks < kN / 16; ++ks)
          umma_bf16_ts(tmem + kTmemO, tmem + kTmemS + ks * 8, dv + ks * (2048 >> 4), idesc_pv,
                       (j > 0 || ks > 0) ? 1u : 0u);
        umma_commit(bar(kBarEmpty + j % kStages));
      };
      bool ok = mbar_wait_fast(bar(kBarQFull), 0, abort) && mbar_wait_fast(bar(kBarFull), 0, abort);
      if (ok) {
        fence_async_shared();  // Q and tile 0, written by cp.async, read by tcgen05.mma
        tc_fence_after_sync();
        qk(0);
      }
      for (int j = 1; j < n_tiles && ok; ++j) {
        if (!(ok = mbar_wait_fast(bar(kBarPFull), (j - 1) & 1, abort))) break;
        tc_fence_after_sync();
        pv(j - 1);
        if (!(ok = mbar_wait_fast(bar(kBarFull + j % kStages), (j / kStages) & 1, abort))) break;
        fence_async_shared();  // tile j, written by cp.async, read by tcgen05.mma
        tc_fence_after_sync();
        qk(j);
      }
      if (ok && (ok = mbar_wait_fast(bar(kBarPFull), (n_tiles - 1) & 1, abort))) {
        tc_fence_after_sync();
        pv(n_tiles - 1);
        umma_commit(bar(kBarOFull));
      }
      if (!ok) {
        *abort = 1;
        flag_error(a.err, kErrTimeout);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int r = tid;  // query row == TMEM lane (warps 0-3)
    const int64_t bh = q_row(r);
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t srow = tmem + lane_base + kTmemS;
    const uint32_t orow_t = tmem + lane_base + kTmemO;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      if (!(ok = mbar_wait_warp(bar(kBarSFull), j & 1, abort))) break;
      tc_fence_after_sync();
      // Row max of the raw scores; scale_log2 > 0 commutes with max. The
      // loads return the max of the columns they read; the tile holding the
      // prefix's last key (CTA-uniform) takes the max after the mask.
      float v[kN], mx0, mx1, mx2, mx3;
      tmem_ld32_max(srow + 0, *reinterpret_cast<float(*)[32]>(&v[0]), mx0);
      tmem_ld32_max(srow + 32, *reinterpret_cast<float(*)[32]>(&v[32]), mx1);
      tmem_ld32_max(srow + 64, *reinterpret_cast<float(*)[32]>(&v[64]), mx2);
      tmem_ld32_max(srow + 96, *reinterpret_cast<float(*)[32]>(&v[96]), mx3);
      tmem_ld_wait();
      const int key0 = (tile0 + j) * kN;
      if (key0 + kN > plen) {
#pragma unroll
        for (int cc = 0; cc < kN; ++cc) v[cc] = key0 + cc < plen ? v[cc] : -INFINITY;
        mx0 = fmaxf(v[0], v[1]);
        mx1 = fmaxf(v[2], v[3]);
        mx2 = fmaxf(v[4], v[5]);
        mx3 = fmaxf(v[6], v[7]);
#pragma unroll
        for (int cc = 8; cc < kN; cc += 8) {
          mx0 = max3f(mx0, v[cc], v[cc + 1]);
          mx1 = max3f(mx1, v[cc + 2], v[cc + 3]);
          mx2 = max3f(mx2, v[cc + 4], v[cc + 5]);
          mx3 = max3f(mx3, v[cc + 6], v[cc + 7]);
        }
      }
      const float mt = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * a.scale_log2;
      // Lazy rescale: move the reference max only when some row's max grew
      // by more than 2^kRescaleThreshold (warp-uniform: tcgen05.ld/st are
      // .sync.aligned).
      const bool rescale = j > 0 && __any_sync(0xffffffffu, mt > m_used + kRescaleThreshold);
      float f = 1.f;
      if (j == 0) {
        m_used = mt;
      } else if (rescale) {
        const float m_new = fmaxf(m_used, mt);
        f = m_used == -INFINITY ? 0.f : fast_exp2(m_used - m_new);
        m_used = m_new;
      }
      const float nm_ = m_used == -INFINITY ? 0.f : -m_used;
      float sa0 = 0.f, sa1 = 0.f, sb0 = 0.f, sb1 = 0.f;
#pragma unroll
      for (int cc = 0; cc < kN; cc += 32) {
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float y0, y1;
          fma2(y0, y1, v[cc + 2 * e], v[cc + 2 * e + 1], a.scale_log2, nm_);
          y0 = fast_exp2(y0);
          y1 = fast_exp2(y1);
          if (e & 1)
            add2(sb0, sb1, y0, y1);
          else
            add2(sa0, sa1, y0, y1);
          w[e] = pack_bf16(y0, y1);
        }
        tmem_st16u(srow + cc / 2, w);  // P: keys cc .. cc + 31 -> columns cc / 2 ..
      }
      l = l * f + ((sa0 + sa1) + (sb0 + sb1));
      if (rescale) {
        // O is stable: S(j) completed, so did PV(j - 1) before it.
#pragma unroll 1
        for (int cb = 0; cb < D / 32; ++cb) {
          float o[32];
          tmem_ld32(orow_t + cb * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int qq = 0; qq < 32; ++qq) o[qq] *= f;
          tmem_st32(orow_t + cb * 32, o);
        }
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(kBarPFull));
    }
    if (ok) ok = mbar_wait_warp(bar(kBarOFull), 0, abort);
    if (!ok) {
      *abort = 1;
      flag_error(a.err, kErrTimeout);
    } else {
      // O / l through shared memory (the K/V stages are free: every MMA is
      // done), so that each store instruction writes whole rows of the
      // partial state instead of 16 bytes of 32 different rows.
      tc_fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      constexpr int kStride = D + 4;  // floats per staged row (16-byte skew: no bank conflicts)
      float *stage = reinterpret_cast<float *>(smem + S::kKV) + warp * 32 * kStride;
#pragma unroll 1
      for (int cb = 0; cb < D / 32; ++cb) {
        float o[32];
        tmem_ld32(orow_t + cb * 32, o);
        tmem_ld_wait();
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
          *reinterpret_cast<float4 *>(stage + lane * kStride + cb * 32 + q4 * 4) =
              make_float4(o[q4 * 4] * inv, o[q4 * 4 + 1] * inv, o[q4 * 4 + 2] * inv,
                          o[q4 * 4 + 3] * inv);
      }
      __syncwarp();
      constexpr int kLanesPerRow = D / 4;  // one float4 per lane
      constexpr int kRowsPerStore = 32 / kLanesPerRow;
      for (int rr0 = 0; rr0 < 32; rr0 += kRowsPerStore) {
        const int rr = rr0 + lane / kLanesPerRow;  // row of this warp
        const int64_t rbh = __shfl_sync(0xffffffffu, bh, rr);
        if (rbh >= 0) {
          const int c4 = (lane % kLanesPerRow) * 4;
          *reinterpret_cast<float4 *>(a.part_o + (rbh * a.pstride + a.pslot + z) * D + c4) =
              *reinterpret_cast<const float4 *>(stage + rr * kStride + c4);
        }
      }
      if (bh >= 0)
        a.part_lse[bh * a.pstride + a.pslot + z] =
            l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
    }
  }

  // Teardown: every role has left its loop (normally or through the abort
  // flag); free TMEM once no MMA is in flight.
  if (warp == kMmaWarp && lane == 0 && *abort) {
    umma_commit(bar(kBarTeardown));  // tracks every MMA this thread issued
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

template <int D>
cudaError_t launch_prefix(const PrefixArgs &a, dim3 grid, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(cascade_prefix_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       PrefixSmem<D>::kTotal);
  if (e != cudaSuccess) return e;
  return launch_pdl(cascade_prefix_kernel<D>, grid, dim3(kThreads), PrefixSmem<D>::kTotal,
                    stream, a);
}

}  // namespace

int32_t cascade_prefix_splits(int32_t batch, int32_t hq, int32_t hkv, int32_t num_groups,
                              int32_t max_prefix, int32_t max_suffix, int32_t sm_count) {
  // The prefix CTAs (one per SM) and the suffix decode's CTAs share the GPU
  // and both are bound by the bytes they gather, so the prefix gets about its
  // share of the bytes in SMs: key ranges per (member block, kv head) =
  // SMs x prefix / (prefix + suffix) / CTAs, from the host bounds, at least
  // one, at most one wave, each range at least two key tiles long.
  const int64_t mpt = kM / (hq / hkv);
  int64_t blocks = (static_cast<int64_t>(batch) + mpt - 1) / mpt;
  if (blocks < num_groups) blocks = num_groups;
  const int64_t ctas = static_cast<int64_t>(hkv) * (blocks > 0 ? blocks : 1);
  const int64_t sms = sm_count > 0 ? sm_count : 1;
  const double pre = static_cast<double>(num_groups) * (max_prefix > 0 ? max_prefix : 0);
  const double suf = static_cast<double>(batch) * (max_suffix > 1 ? max_suffix : 1);
  int64_t ks = static_cast<int64_t>(static_cast<double>(sms) * pre / (pre + suf) /
                                    static_cast<double>(ctas) + 0.5);
  const int64_t wave = sms / ctas;
  const int64_t nk = (static_cast<int64_t>(max_prefix > 0 ? max_prefix : 0) + kN - 1) / kN;
  if (ks > wave) ks = wave;
  if (ks > nk / 2) ks = nk / 2;
  if (ks > PKV_PREFIX_MAX_SPLITS) ks = PKV_PREFIX_MAX_SPLITS;
  return static_cast<int32_t>(ks < 1 ? 1 : ks);
}

int32_t cascade_prefix_blocks(int32_t batch, int32_t hq, int32_t hkv, int32_t num_groups) {
  const int64_t mpt = kM / (hq / hkv);
  return static_cast<int32_t>((static_cast<int64_t>(batch) + mpt - 1) / mpt + num_groups);
}

cudaError_t launch_cascade_prefix(const PoolGeom &g, int32_t layer, const void *q,
                                  const int32_t *prefix_table, int64_t prefix_stride,
                                  const int32_t *prefix_lens, const int32_t *member_indptr,
                                  const int32_t *members, int32_t num_groups, int32_t batch,
                                  int32_t hq, float scale, float *part_o, float *part_lse,
                                  int32_t pstride, int32_t pslot, int32_t key_splits,
                                  unsigned *err, cudaStream_t stream) {
  PrefixArgs a{};
  a.pool = static_cast<const __nv_bfloat16 *>(g.base);
  a.slots = g.slots;
  a.num_layers = g.num_layers;
  a.layer = layer;
  a.page_size = g.page_size;
  a.hkv = g.hkv;
  a.prefix_table = prefix_table;
  a.prefix_stride = prefix_stride;
  a.prefix_lens = prefix_lens;
  a.member_indptr = member_indptr;
  a.members = members;
  a.num_groups = num_groups;
  a.batch = batch;
  a.q = static_cast<const __nv_bfloat16 *>(q);
  a.hq = hq;
  a.group = hq / g.hkv;
  a.members_per_tile = kM / a.group;
  a.q_mode = scale > 0.f ? 0 : (scale < 0.f ? 1 : 2);
  a.scale_log2 = scale > 0.f ? scale * kLog2e : (scale < 0.f ? -scale * kLog2e : kLog2e);
  a.part_o = part_o;
  a.part_lse = part_lse;
  a.pstride = pstride;
  a.pslot = pslot;
  a.key_splits = key_splits;
  a.err = err;
  const dim3 grid(g.hkv, cascade_prefix_blocks(batch, hq, g.hkv, num_groups), key_splits);
  return g.d == 128 ? launch_prefix<128>(a, grid, stream) : launch_prefix<64>(a, grid, stream);
}

}  // namespace pkv
