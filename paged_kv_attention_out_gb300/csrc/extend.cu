// extend.cu - paged extend (chunked-prefill) attention on tcgen05 / TMEM / TMA.
//
// What it computes ("Code Notes: mini-sglang", Scheduler Layer table,
// PrefillManager row; "Introduction", Key Features, Chunked Prefill and Radix
// Cache): request r's chunk of c_r new queries sits after a cached prefix of
// p_r = seq_len[r] - c_r keys; chunk query j attends to keys 0 .. p_r + j of
// the request's page_table row (full prefix, causal within the chunk).
//
// Two kernels per call:
//   extend_gather_kernel  copies each request's visible K and V rows, for
//       every kv head, out of the paged pool into a contiguous run of the
//       workspace (zero rows up to the next multiple of 128 keys), reading
//       the pool once per call. The runs of the requests lie back to back in
//       request order, [2][Hkv][cap_rows][D], so the workspace is sized by the
//       keys present (a host bound on their sum), not by batch x max length;
//       two waves of resident CTAs loop over 16-row chunks of that space,
//       finding each chunk's request by a prefix sum of the rounded lengths;
//       the first CTA builds the block schedule meanwhile; pool rows are
//       read with an L2 evict-first policy and the workspace rows written
//       with evict-last, since the attention reads them right after;
//   extend_tc_persistent_kernel  the attention, which then reads every
//       128-key K or V tile with plain 2-D TMA boxes instead of row gathers;
//       one CTA per SM takes blocks of the schedule as work items.
//
// Tiling. A block (work item) is two 128-row query tiles X = 0, 1 of one kv
// head; a tile holds 128 / g chunk tokens x the g q heads that read that kv
// head, so every K/V tile loaded feeds 2 x 128 query rows. It walks the
// visible keys in tiles of 128; per key tile j and query tile X:
//   S_X  = Q_X K_j^T           tcgen05.mma, M=128 N=128 K=D, fp32 in TMEM
//   P_X  = exp2(scale*S_X - m) softmax warps of tile X, bf16 back into TMEM
//                              over the first half of S_X
//   O_X += P_X V_j             tcgen05.mma with A = P_X from TMEM, M=128
//                              N=D K=128, fp32 in TMEM
// While the softmax of one query tile runs, the tensor core works on the
// other's MMAs.
// Roles (320 threads):
//   warps 0-7  softmax: query tile X = warp / 4; warp w owns TMEM lanes
//              32 (w % 4) .. + 31 (query rows), one whole row per thread;
//              log2-domain online softmax with a lazy rescale (O_X is
//              rescaled only when a row max grows by more than 2^8), masks
//              only on tiles that cross some row's last key; then O / l ->
//              bf16 and lse.
//   warp 8     TMEM allocation and the single MMA-issuing thread.
//   warp 9     producer: takes the work items, then per item the Q tiles
//              (3-D TMA boxes) and the K and V tiles (2-D TMA boxes of 128
//              keys x 64 columns, 128-byte swizzle) into two stages; a stage
//              is refilled once every MMA that reads it is done.
// Every hand-off is an mbarrier; every wait is bounded (tc_common.cuh).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "pkv_common.cuh"
#include "pkv_internal.h"
#include "tc_common.cuh"

namespace pkv {
namespace {

constexpr int kM = 128;       // query rows per query tile (= TMEM lanes)
constexpr int kQTiles = 2;    // query tiles per CTA, sharing every K/V tile
constexpr int kN = 128;       // keys per K/V tile
constexpr int kSoftmaxWarps = 8;  // warps 4X .. 4X + 3 serve query tile X
constexpr int kMmaWarp = kSoftmaxWarps;
constexpr int kProducerWarp = kSoftmaxWarps + 1;  // loads Q, K and V
constexpr int kProducerWarps = 1;
constexpr int kThreads = (kSoftmaxWarps + 1 + kProducerWarps) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct Smem {
  static constexpr int kQ = 0;  // query tile X at kQ + X * kQBytes
  static constexpr int kQBytes = kM * D * 2;
  static constexpr int kTileBytes = kN * D * 2;
  static constexpr int kKV = kQ + kQTiles * kQBytes;  // stage s: K at kKV + s*2*tile, V after it
  static constexpr int kBars = kKV + 4 * kTileBytes;
  // + alignment slack; never below 116 KB, so one CTA (and one 512-column
  // TMEM allocation) per SM even for head_dim 64
  static constexpr int kNeed = kBars + 32 * 8 + 1024;
  static constexpr int kTotal = kNeed > 116 * 1024 ? kNeed : 116 * 1024;
};

// TMEM columns: S_X (fp32 scores of query tile X) at 128 X, O_X at 256 + D X.
// P_X (bf16 pairs, one 32-bit column per two keys) overwrites the first 64
// columns of S_X once the softmax has read S_X into registers; the P V MMA
// takes it from there as its A operand.
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemO = 256;

struct GatherArgs {
  const __nv_bfloat16 *pool;  // plane (c, layer) starts at ((c * L + layer) * slots) rows
  int64_t slots;
  int32_t num_layers;
  int32_t layer;
  int32_t page_size;
  int32_t hkv;
  const int32_t *page_table;
  int64_t table_stride;
  const int32_t *table_idx;
  const int32_t *seq_lens;
  int32_t batch;
  int64_t row_capacity;  // table_stride * page_size: a longer seq_len is invalid
  int32_t cap_rows;      // rows of one (K or V, kv head) region of the workspace
  int32_t nbuck;         // cost buckets of the block schedule
  int32_t max_blocks;    // bound on the schedule's blocks
  __nv_bfloat16 *ws;
  unsigned *err;
  // block schedule (built by the planner CTA, read by the attention)
  const int32_t *qo_indptr;
  int32_t total_q;
  int32_t tokens_per_tile;
  int32_t *plan;
  // Fused store (k_new != nullptr): the chunk's keys p_r .. seq_r - 1 are
  // taken from rows qo_indptr[r] .. of k_new / v_new and also written into
  // the pool at their page-table slots.
  const __nv_bfloat16 *k_new;
  const __nv_bfloat16 *v_new;
  int64_t kv_row_stride;
  __nv_bfloat16 *pool_w;
};

struct ExtendArgs {
  const int32_t *qo_indptr;
  __nv_bfloat16 *o;
  float *lse;
  const int32_t *seq_lens;
  int32_t batch;
  int32_t hkv;
  int32_t total_q;
  int32_t hq;
  int32_t group;
  int32_t tokens_per_tile;  // floor(128 / group) chunk tokens per query tile
  int32_t cap_rows;
  int32_t nbuck;
  int32_t max_blocks;
  float scale_log2;  // |scale| * log2(e) (log2(e) when scale is 0), always > 0
  // How the softmax scale's sign reaches the scores: the row max is taken
  // on raw scores, which needs scale_log2 > 0, so a negative scale negates
  // Q in shared memory (scale * q.k = |scale| * (-q).k, exactly) and a zero
  // scale zeroes it (every score 0, as for q = 0). 0: Q as given.
  int32_t q_mode;
  unsigned *err;
  int32_t *plan;  // the persistent form takes its work items from plan[1]
};

constexpr int kGatherKeys = 16;     // keys per chunk of a gather CTA (two per warp)
constexpr int kGatherWaves = 2;     // copying CTAs: this many waves of resident CTAs
constexpr int kGatherThreads = 256;

// Workspace run of request r, kv head h, K (c = 0) or V (c = 1): the
// request's seq_len rounded up to 128 rows of D elements, starting at row
// (c * Hkv + h) * cap_rows + off_r, where off_r is the sum of the rounded
// lengths of requests 0 .. r - 1 (a seq_len outside [0, row capacity] has
// none). A request whose run would end past cap_rows is not gathered or
// attended (flagged). Rows seq_len .. (seq_len rounded up to 128) - 1 are
// written as zeros so a tile never holds stale bits (a NaN there would
// survive P = 0 in P V).
__device__ __forceinline__ int64_t run_rows(const GatherArgs &a, int seq) {
  return (seq >= 0 && seq <= a.row_capacity) ? ((static_cast<int64_t>(seq) + 127) & ~int64_t(127))
                                             : 0;
}

// Longest-first block schedule. A "block" is one attention CTA's work: two
// query tiles (2 * tokens_per_tile chunk tokens) of one request. Its cost is
// the number of (query tile, key tile) pairs it computes plus two for its
// prologue and epilogue; blocks are counting-sorted by cost, largest first,
// so the longest CTAs start in the first wave and the tail is short. Layout
// (int32): plan[0] = block count; the histogram at kPlanHist (nbuck
// entries); then (request, first token, cost) per block in request order;
// then the sorted (request, first token) pairs; then off_r per request.
constexpr int kPlanHist = 16;

__host__ __device__ inline int64_t plan_ints(int64_t batch, int64_t nbuck, int64_t max_blocks) {
  return kPlanHist + nbuck + 5 * max_blocks + batch;
}
__host__ __device__ inline int64_t plan_sorted(int64_t nbuck, int64_t max_blocks) {
  return kPlanHist + nbuck + 3 * max_blocks;
}
__host__ __device__ inline int64_t plan_offsets(int64_t nbuck, int64_t max_blocks) {
  return kPlanHist + nbuck + 5 * max_blocks;
}

// Block-wide inclusive scan of one int64 per thread (kGatherThreads threads);
// returns the thread's inclusive sum and writes the round's total.
__device__ __forceinline__ int64_t block_scan(int64_t v, int64_t *s_warp, int64_t *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int64_t u = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += u;
  }
  if (lane == 31) s_warp[warp] = v;
  __syncthreads();
  int64_t before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kGatherThreads / 32; ++w) {
    before += w < warp ? s_warp[w] : 0;
    all += s_warp[w];
  }
  __syncthreads();  // s_warp may be reused by the caller's next round
  *total = all;
  return v + before;
}

__device__ void plan_blocks(const GatherArgs &a) {
  __shared__ int s_first_bad;
  __shared__ int s_part[kGatherThreads];
  __shared__ int64_t s_warp[kGatherThreads / 32];
  const int tid = threadIdx.x;
  const int per = 2 * a.tokens_per_tile;
  const int nbuck = a.nbuck;
  int *hist = a.plan + kPlanHist;
  int *ent = hist + nbuck;                // 3 per block, request order
  int *sorted = ent + 3 * a.max_blocks;   // 2 per block, by cost
  int *offsets = a.plan + plan_offsets(nbuck, a.max_blocks);
  if (tid == 0) s_first_bad = a.batch;
  for (int i = tid; i < nbuck; i += kGatherThreads) hist[i] = 0;
  __syncthreads();
  // The schedule covers the requests before the first malformed qo_indptr entry.
  for (int r = tid; r < a.batch; r += kGatherThreads) {
    const int beg = a.qo_indptr[r], end = a.qo_indptr[r + 1];
    if (beg < 0 || end < beg || end > a.total_q) atomicMin(&s_first_bad, r);
  }
  __syncthreads();
  if (tid == 0 && s_first_bad < a.batch) flag_error(a.err, kErrIndptr);
  const int nreq = s_first_bad;
  // Run offsets and block offsets: running scans over all requests,
  // kGatherThreads at a time (the gather CTAs find their runs by the same
  // run-offset scan).
  int base = 0;
  int64_t run_base = 0;
  for (int r0 = 0; r0 < a.batch; r0 += kGatherThreads) {
    const int r = r0 + tid;
    int nb = 0, c = 0, p = 0;
    int64_t rows = 0;
    bool placed = false;
    if (r < a.batch) {
      const int seq = a.seq_lens[r];
      rows = run_rows(a, seq);
      if (rows == 0 && seq != 0) flag_error(a.err, kErrSeqLen);  // outside [0, row capacity]
      if (r < nreq) {
        c = a.qo_indptr[r + 1] - a.qo_indptr[r];
        p = seq - c;  // the cached prefix
        if (p < 0) flag_error(a.err, kErrIndptr);
      }
    }
    int64_t round_rows;
    const int64_t run_end = run_base + block_scan(rows, s_warp, &round_rows);
    if (r < a.batch) {
      placed = run_end <= a.cap_rows;
      if (rows > 0 && !placed) flag_error(a.err, kErrSeqLen);  // past the workspace's key bound
      offsets[r] = placed ? static_cast<int>(run_end - rows) : 0;
      if (r < nreq && p >= 0 && rows > 0 && placed) nb = (c + per - 1) / per;
    }
    run_base += round_rows;
    s_part[tid] = nb;
    __syncthreads();
    for (int off = 1; off < kGatherThreads; off <<= 1) {  // inclusive scan
      const int v = tid >= off ? s_part[tid - off] : 0;
      __syncthreads();
      s_part[tid] += v;
      __syncthreads();
    }
    const int first = base + s_part[tid] - nb;
    for (int i = 0; i < nb; ++i) {
      const int j0 = i * per;
      const int tokens = min(per, c - j0);
      const int tok0 = min(a.tokens_per_tile, tokens);
      const int tok1 = max(0, tokens - a.tokens_per_tile);
      const int n0 = (p + j0 + tok0 + 127) / 128;
      const int n1 = tok1 == 0 ? 0 : (p + j0 + a.tokens_per_tile + tok1 + 127) / 128;
      const int cost = min(n0 + n1 + 2, nbuck - 1);
      const int b = first + i;
      ent[3 * b] = r;
      ent[3 * b + 1] = j0;
      ent[3 * b + 2] = cost;
      atomicAdd(&hist[cost], 1);
    }
    base += s_part[kGatherThreads - 1];
    __syncthreads();
  }
  const int nblk = base;
  // Exclusive scan of the histogram from the largest cost down gives each
  // bucket's first rank; thread t owns a contiguous run of buckets.
  const int run = (nbuck + kGatherThreads - 1) / kGatherThreads;
  int sum = 0;
  for (int i = 0; i < run; ++i) {
    const int k = nbuck - 1 - (tid * run + i);
    if (k >= 0) sum += hist[k];
  }
  s_part[tid] = sum;
  __syncthreads();
  for (int off = 1; off < kGatherThreads; off <<= 1) {
    const int v = tid >= off ? s_part[tid - off] : 0;
    __syncthreads();
    s_part[tid] += v;
    __syncthreads();
  }
  int start = s_part[tid] - sum;
  for (int i = 0; i < run; ++i) {
    const int k = nbuck - 1 - (tid * run + i);
    if (k >= 0) {
      const int h = hist[k];
      hist[k] = start;
      start += h;
    }
  }
  __syncthreads();
  for (int b = tid; b < nblk; b += kGatherThreads) {
    const int pos = atomicAdd(&hist[ent[3 * b + 2]], 1);
    sorted[2 * pos] = ent[3 * b];
    sorted[2 * pos + 1] = ent[3 * b + 1];
  }
  if (tid == 0) {
    a.plan[0] = nblk;
    a.plan[1] = 0;  // the persistent attention's work-item counter
  }
}

// kStore: the fused store (a.k_new != nullptr), a separate instantiation so
// the plain gather keeps its lean inner loop.
template <int D, bool kStore>
__device__ __forceinline__ void gather_body(const GatherArgs &a);
template <int D, bool kStore>
__device__ __forceinline__ bool gather_rows(const GatherArgs &a, int64_t pos);

template <int D, bool kStore>
__global__ void __launch_bounds__(kGatherThreads)
    extend_gather_kernel(const GatherArgs a) {
  grid_dependency_wait();  // the chunk's K/V may come from the previous kernel (store_kv)
  grid_dependents_launch();
  gather_body<D, kStore>(a);
}

// Read-only 16-byte load / 16-byte store with an L2 eviction-priority
// policy (createpolicy): the pool rows are read once per call (evict first),
// the workspace rows are read again by the attention right after (evict last).
__device__ __forceinline__ uint4 ldg_nc_hint(const uint4 *p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}
__device__ __forceinline__ void st_hint(uint4 *p, uint4 v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w), "l"(policy)
               : "memory");
}
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// The first CTA builds the schedule (dispatched before the copying CTAs);
// the others copy 16-row chunks of the key space, chunk c by CTA 1 + c mod
// (grid - 1), so a grid of whole waves finishes together.
template <int D, bool kStore>
__device__ __forceinline__ void gather_body(const GatherArgs &a) {
  if (blockIdx.x == 0) {
    plan_blocks(a);
    return;
  }
  const int64_t chunks = a.cap_rows / kGatherKeys;
  for (int64_t c = blockIdx.x - 1; c < chunks; c += gridDim.x - 1)
    if (!gather_rows<D, kStore>(a, c * kGatherKeys)) break;
}

// Copies rows pos .. pos + 15 of the key space. Returns false once pos lies
// past every run (so does every later chunk).
template <int D, bool kStore>
__device__ __forceinline__ bool gather_rows(const GatherArgs &a, int64_t pos) {
  // The request whose run holds these 16 rows (runs are multiples of 128
  // rows, so they never straddle two requests): the same scan of the
  // rounded lengths as the planner's, kGatherThreads requests per round.
  __shared__ int64_t s_warp[kGatherThreads / 32];
  __shared__ int s_r;
  __shared__ int64_t s_off;
  __syncthreads();  // the previous chunk's s_r / s_off are read
  if (threadIdx.x == 0) s_r = -1;
  int64_t run_base = 0;
  for (int r0 = 0; r0 < a.batch; r0 += kGatherThreads) {
    const int rr = r0 + static_cast<int>(threadIdx.x);
    const int64_t rows = rr < a.batch ? run_rows(a, a.seq_lens[rr]) : 0;
    int64_t round_rows;
    const int64_t run_end = run_base + block_scan(rows, s_warp, &round_rows);
    if (rows > 0 && pos >= run_end - rows && pos < run_end) {
      s_r = rr;
      s_off = run_end - rows;
    }
    run_base += round_rows;
    if (pos < run_base) break;  // uniform: found in this round (or in no run)
  }
  __syncthreads();
  const int r = s_r;
  if (r < 0) return false;  // past the last run
  const int64_t off = s_off;
  const int seq = a.seq_lens[r];
  if (off + run_rows(a, seq) > a.cap_rows) return false;  // past the key bound (flagged by the planner)
  const int key0 = static_cast<int>(pos - off);
  const int row = a.table_idx ? a.table_idx[r] : r;
  if (row < 0) {
    if (key0 == 0 && threadIdx.x == 0) flag_error(a.err, kErrTableIdx);  // once per request
    return true;
  }
  const int32_t *row_pages = a.page_table + static_cast<int64_t>(row) * a.table_stride;
  // Fused store: keys from new_key0 on are the chunk's, key k is row
  // new_row0 + k of k_new / v_new. A malformed qo_indptr pair (flagged by the
  // planner) stores nothing and reads the pool as the unfused call would.
  int new_key0 = seq;
  int64_t new_row0 = 0;
  if (kStore) {
    const int beg = a.qo_indptr[r], end = a.qo_indptr[r + 1];
    if (beg >= 0 && end >= beg && end <= a.total_q && end - beg <= seq) {
      new_key0 = seq - (end - beg);
      new_row0 = static_cast<int64_t>(beg) - new_key0;
    }
  }
  // One warp per key: its K row and V row (Hkv * D contiguous elements each
  // in the pool); 16-byte chunk `ch` of a row goes to kv head ch / (D / 8)'s run.
  constexpr int kChunks = D / 8;  // 16-byte chunks per head row
  const int nch = a.hkv * kChunks;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t row_elems = static_cast<int64_t>(a.hkv) * D;
  const int64_t run_elems = static_cast<int64_t>(a.cap_rows) * D;  // one kv head's region
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  constexpr int kUnroll = 4;  // chunks per lane per row in flight (x 2 rows)
  const uint64_t pol_read = l2_evict_first_policy();
  const uint64_t pol_write = l2_evict_last_policy();
  for (int kk = warp; kk < kGatherKeys; kk += kGatherThreads / 32) {
    const int key = key0 + kk;
    // the key's K row (c = 0) and V row (c = 1) are copied together
    const uint4 *src[2] = {nullptr, nullptr};
    uint4 *store[2] = {nullptr, nullptr};  // fused store: the key's pool rows
    if (key < seq) {
      const int pidx = key / a.page_size;
      const int ent = __ldg(row_pages + pidx);
      const int64_t slot = static_cast<int64_t>(ent) * a.page_size + (key - pidx * a.page_size);
      const bool slot_ok = ent >= 0 && slot < a.slots;
      if (kStore && key >= new_key0) {
        const int64_t nrow = (new_row0 + key) * a.kv_row_stride;
        src[0] = reinterpret_cast<const uint4 *>(a.k_new + nrow);
        src[1] = reinterpret_cast<const uint4 *>(a.v_new + nrow);
      }
      if (slot_ok) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int64_t prow = (static_cast<int64_t>(c) * a.num_layers + a.layer) * a.slots + slot;
          if (kStore && key >= new_key0)
            store[c] = reinterpret_cast<uint4 *>(a.pool_w + prow * row_elems);
          else
            src[c] = reinterpret_cast<const uint4 *>(a.pool + prow * row_elems);
        }
      } else if (lane == 0) {
        flag_error(a.err, kErrPage);
      }
    }
    for (int ch0 = lane; ch0 < nch; ch0 += 32 * kUnroll) {
      uint4 v[2][kUnroll];
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int ch = ch0 + 32 * u;
          v[c][u] = (src[c] != nullptr && ch < nch) ? ldg_nc_hint(src[c] + ch, pol_read) : zero;
        }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        __nv_bfloat16 *dst = a.ws + static_cast<int64_t>(c) * a.hkv * run_elems +
                             (off + key) * D;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int ch = ch0 + 32 * u;
          if (ch < nch) {
            st_hint(reinterpret_cast<uint4 *>(dst + (ch / kChunks) * run_elems + (ch % kChunks) * 8),
                    v[c][u], pol_write);
            if (kStore && store[c] != nullptr) store[c][ch] = v[c][u];
          }
        }
      }
    }
  }
  return true;
}

// TMA tile load (as tma_load_2d) with an L2 eviction-priority policy
// (createpolicy): the K/V workspace tiles are read again by every block of
// their request, so they are kept (evict last) ahead of Q and O, which are
// touched once.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const void *tmap, int x, int y,
                                                 uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// ------------------------------------------------------------ attention
// One CTA per SM pulls work items, (kv head, block) pairs in longest-first
// order, from a counter the planner zeroes (plan[1]); item i is block
// i / Hkv of the schedule on kv head i % Hkv. The roles run the per-tile
// pipeline described at the top, continued across items: the producer publishes the next
// item (a two-slot descriptor ring) and loads its Q tiles as soon as every
// S MMA of the current item is done, and its K/V tiles through the same
// two-stage ring; the MMA thread issues the next item's first S while the
// softmax warps write the current item's output, and its first P V once
// they have read O. So a CTA's prologue (barrier setup, TMEM allocation,
// the Q and first K/V loads) is paid once per SM, not once per block.
// Every barrier keeps one phase sequence across items: tile counters for
// the K/V stages and S/P hand-offs, item counters for the rest, counted per
// query tile where a tile may sit out an item (no tokens), so a waiter is
// never two phases behind (a barrier waited on with a parity completes at
// most once between two waits of the same waiter).

enum : int {
  kPBarFull = 0,        // [2] producer: K and V tiles of stage s landed (TMA bytes)
  kPBarEmpty = 2,       // [2] MMA: every MMA reading stage s done
  kPBarSFull = 4,       // [2] MMA: S_X ready
  kPBarPFull = 6,       // [2] softmax X: P_X in TMEM (and O_X rescaled)
  kPBarOFull = 8,       // [2] MMA: every MMA of the item on query tile X done
  kPBarOEmpty = 10,     // [2] softmax X: O_X read out (the item's output written)
  kPBarItemFull = 12,   // [2] producer: descriptor slot written
  kPBarItemEmpty = 14,  // [2] MMA thread + one lane per softmax warp: slot read
  kPBarQFull = 16,      // producer: the item's Q tiles landed (TMA bytes)
  kPBarQReady = 17,     // softmax warps: Q negated / zeroed in place (q_mode != 0)
  kPBarQEmpty = 18,     // MMA: every S = Q K^T of the item done (Q may be reloaded)
  kPBarTeardown = 19,   // MMA: everything issued has finished (abort path)
  kPBarCount = 20,
};
static_assert(kPBarCount <= 32, "barrier area of Smem");

constexpr std::integral_constant<int, 0> kTile0{};
constexpr std::integral_constant<int, 1> kTile1{};

// One work item as the producer publishes it (req < 0: no more items).
struct ItemDesc {
  int req, kvh, j0, c, p, off, t_base;
};

// The item's split into query tiles and key tiles: query tile X holds
// tokens X tpt .. X tpt + tok_X - 1 of the item and walks key tiles
// 0 .. n_X - 1 (n_1 = 0 when it holds no token).
struct ItemGeom {
  int tokens, n0, n1, n_tiles;
};

__device__ __forceinline__ ItemGeom item_geom(const ItemDesc &d, int tpt) {
  ItemGeom g;
  g.tokens = min(kQTiles * tpt, d.c - d.j0);
  const int tok1 = max(0, min(tpt, g.tokens - tpt));
  const int tok0 = min(tpt, g.tokens);
  g.n0 = (d.p + d.j0 + tok0 + kN - 1) / kN;
  g.n1 = tok1 == 0 ? 0 : (d.p + d.j0 + tpt + tok1 + kN - 1) / kN;
  g.n_tiles = max(g.n0, g.n1);
  return g;
}

__device__ __forceinline__ ItemDesc shfl_desc(ItemDesc d) {
  d.req = __shfl_sync(0xffffffffu, d.req, 0);
  d.kvh = __shfl_sync(0xffffffffu, d.kvh, 0);
  d.j0 = __shfl_sync(0xffffffffu, d.j0, 0);
  d.c = __shfl_sync(0xffffffffu, d.c, 0);
  d.p = __shfl_sync(0xffffffffu, d.p, 0);
  d.off = __shfl_sync(0xffffffffu, d.off, 0);
  d.t_base = __shfl_sync(0xffffffffu, d.t_base, 0);
  return d;
}

// q3_map: q as a 3-D bf16 tensor [total_q][Hq][D], box {64, g, 128 / g}
// (one query tile's half: its tokens x the g q heads of one kv head, rows in
// (token, head) order as the tile's rows), 128-byte swizzle.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    extend_tc_persistent_kernel(const __grid_constant__ CUtensorMap kv_map,
                                const __grid_constant__ CUtensorMap q3_map, const ExtendArgs a) {
  using S = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ ItemDesc s_item[2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  // Per softmax warp: items taken, S tiles taken, items that used its query
  // tile (kept here, not in registers, across the warp's key-tile loop).
  __shared__ int s_sm_state[kSoftmaxWarps][3];
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int tpt = a.tokens_per_tile;

  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bars = sbase + S::kBars;
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  volatile int *abort = &s_abort;

  // Set-up that needs nothing from the gather kernel runs before the wait.
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kPBarFull + i), 1);  // the producer's expect_tx arrival
      mbar_init(bar(kPBarEmpty + i), 1);
      mbar_init(bar(kPBarSFull + i), 1);
      mbar_init(bar(kPBarPFull + i), 128);  // the four warps of one query tile
      mbar_init(bar(kPBarOFull + i), 1);
      mbar_init(bar(kPBarOEmpty + i), 128);
      mbar_init(bar(kPBarItemFull + i), 1);
      mbar_init(bar(kPBarItemEmpty + i), 1 + kSoftmaxWarps);
    }
    mbar_init(bar(kPBarQFull), 1);
    mbar_init(bar(kPBarQReady), kSoftmaxWarps * 32);
    mbar_init(bar(kPBarQEmpty), 1);
    mbar_init(bar(kPBarTeardown), 1);
    s_abort = 0;
    mbar_init_fence();
  }
  {
    // Rows g * tpt .. 127 of a query tile (group not dividing 128) are
    // never loaded: zero them once, so those rows' scores stay finite.
    constexpr int kHalves = D / 64;
    const int pad_rows = kM - a.group * tpt;
    for (int i = tid; i < kQTiles * kHalves * pad_rows * 8; i += kThreads) {
      const int chunk = i & 7, row = (i >> 3) % pad_rows, region = (i >> 3) / pad_rows;
      *reinterpret_cast<uint4 *>(smem + S::kQ + region * (kM * 128) + (kM - pad_rows + row) * 128 +
                                 chunk * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_async_shared();  // generic-proxy writes, read by tcgen05.mma
  }
  if (warp == kMmaWarp) tmem_alloc(smem_addr(&s_tmem), kTmemCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = s_tmem;
  grid_dependency_wait();  // the schedule and the K/V runs come from the gather kernel

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // Per item: take the next item from the counter and publish it; once
    // every S of the previous item is done, load the item's two Q tiles
    // (lane l: rows 4 l .. 4 l + 3 of each, both 64-column halves; rows past
    // the item's tokens read as zeros); then its K and V tiles, tile g of
    // the CTA into stage g % 2 once every MMA reading that stage (tile
    // g - 2) is done. Lane 0 issues the loads.
    constexpr int kHalves = D / 64;
    const uint64_t kv_policy = l2_evict_last_policy();
    const int total_items = a.hkv * a.plan[0];
    const int *sorted = a.plan + plan_sorted(a.nbuck, a.max_blocks);
    const int *offs = a.plan + plan_offsets(a.nbuck, a.max_blocks);
    unsigned *counter = reinterpret_cast<unsigned *>(a.plan + 1);
    bool ok = true;
    uint32_t g = 0;  // K/V tiles issued (all items)
    int q_loads = 0;
    for (int k = 0;; ++k) {
      const int slot = k & 1;
      if (k >= 2 &&
          !(ok = mbar_wait_warp(bar(kPBarItemEmpty + slot), ((k >> 1) - 1) & 1, abort)))
        break;
      ItemDesc d{-1, 0, 0, 0, 0, 0, 0};
      if (lane == 0) {
        const int i = static_cast<int>(atomicAdd(counter, 1u));
        if (i < total_items) {
          const int rank = i / a.hkv;
          d.kvh = i - rank * a.hkv;
          d.req = sorted[2 * rank];
          d.j0 = sorted[2 * rank + 1];
          d.t_base = a.qo_indptr[d.req];
          d.c = a.qo_indptr[d.req + 1] - d.t_base;
          d.p = a.seq_lens[d.req] - d.c;
          d.off = offs[d.req];
        }
        s_item[slot] = d;
        mbar_arrive(bar(kPBarItemFull + slot));  // release: the slot's contents
      }
      d = shfl_desc(d);
      if (d.req < 0) break;
      const ItemGeom ig = item_geom(d, tpt);
      if (k >= 1 && !(ok = mbar_wait_warp(bar(kPBarQEmpty), (k - 1) & 1, abort))) break;
      if (lane == 0) {
        // Query tile x: tokens t_base + j0 + x tpt .. + tpt - 1, the g q heads
        // of this kv head, as one 3-D box per 64-column half. Rows of tokens
        // past the item (the next request's, or zeros past the last token)
        // belong to no output row.
        const uint32_t box_bytes = static_cast<uint32_t>(a.group * tpt) * 128u;
        mbar_arrive_expect_tx(bar(kPBarQFull), kQTiles * kHalves * box_bytes);
#pragma unroll
        for (int x = 0; x < kQTiles; ++x)
#pragma unroll
          for (int h = 0; h < kHalves; ++h)
            tma_load_3d(sbase + S::kQ + static_cast<uint32_t>(x * S::kQBytes + h * (kM * 128)),
                        &q3_map, h * 64, d.kvh * a.group, d.t_base + d.j0 + x * tpt,
                        bar(kPBarQFull));
      }
      __syncwarp();
      ++q_loads;
      // first workspace rows of this request's K and V runs for this kv head
      const int k_run = d.kvh * a.cap_rows + d.off;
      const int v_run = (a.hkv + d.kvh) * a.cap_rows + d.off;
      for (int j = 0; j < ig.n_tiles; ++j, ++g) {
        const int st = static_cast<int>(g & 1);
        if (g >= 2 && !(ok = mbar_wait_warp(bar(kPBarEmpty + st), ((g >> 1) - 1) & 1, abort)))
          break;
        if (lane == 0) {
          const uint32_t dst = sbase + S::kKV + st * 2 * S::kTileBytes;
          mbar_arrive_expect_tx(bar(kPBarFull + st), 2 * S::kTileBytes);
#pragma unroll
          for (int h = 0; h < kHalves; ++h) {
            tma_load_2d_hint(dst + h * (kN * 128), &kv_map, h * 64, k_run + j * kN,
                             bar(kPBarFull + st), kv_policy);
            tma_load_2d_hint(dst + S::kTileBytes + h * (kN * 128), &kv_map, h * 64,
                             v_run + j * kN, bar(kPBarFull + st), kv_policy);
          }
        }
        __syncwarp();
      }
      if (!ok) break;
    }
    if (!ok) *abort = 1;
    if (*abort && lane == 0) {
      // Let every issued copy land before the CTA can exit: TMA writes to
      // this CTA's shared memory need no other input to finish.
      int never = 0;
      if (q_loads > 0) mbar_wait(bar(kPBarQFull), (q_loads - 1) & 1, &never);
      for (uint32_t t = g > 2 ? g - 2 : 0; t < g; ++t)
        mbar_wait(bar(kPBarFull + (t & 1)), (t >> 1) & 1, &never);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // Per item: S_0(0), S_1(0), then per key tile j PV_0(j), S_0(j+1),
    // PV_1(j), S_1(j+1). tcgen05.mma ops of one thread run in issue order, so
    // S_X(j+1) overwrites P_X(j) only after PV_X(j) has read it, and a
    // completed S_X(j+1) implies a completed PV_X(j) (O_X is then stable). Across items: the next item's S_X(0) may
    // run while softmax X writes the previous output (it only reads O_X);
    // its first PV_X waits until that output has been read out of O_X.
    if (lane == 0) {
      constexpr uint32_t idesc_qk = umma_idesc_bf16(kM, kN, 0, 0);
      constexpr uint32_t idesc_pv = umma_idesc_bf16(kM, D, 0, 1);
      const uint64_t dq0 = umma_desc_sw128(sbase + S::kQ, 16, 1024);
      const uint64_t dk0 = umma_desc_sw128(sbase + S::kKV, 16, 1024);
      const uint64_t dv0 = umma_desc_sw128(sbase + S::kKV + S::kTileBytes, kN * 128, 1024);
      constexpr uint64_t kStageStep = (2 * S::kTileBytes) >> 4;
      auto kstep = [](int ks, int rows) -> uint64_t {
        return static_cast<uint64_t>(((ks >> 2) * (rows * 128) + (ks & 3) * 32) >> 4);
      };
      auto qk = [&](int x, uint32_t gt) {  // S_x from CTA tile gt's K
        const uint64_t dq = dq0 + static_cast<uint64_t>((x * S::kQBytes) >> 4);
        const uint64_t dk = dk0 + (gt & 1) * kStageStep;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          umma_bf16_ss(tmem + kTmemS + x * kN, dq + kstep(ks, kM), dk + kstep(ks, kN), idesc_qk,
                       ks > 0 ? 1u : 0u);
        umma_commit(bar(kPBarSFull + x));
      };
      // Per query tile (scalars): P V products issued and items that used
      // the tile, over all items.
      int pv_count0 = 0, pv_count1 = 0, uses0 = 0, uses1 = 0;
      // O_x += P_x V(tile gt), j = the item's key tile; the item's first
      // product overwrites O_x once the previous item's output is read out.
      auto pv = [&](auto xc, int j, uint32_t gt) -> bool {
        constexpr int x = decltype(xc)::value;
        int &pv_count = x == 0 ? pv_count0 : pv_count1;
        const int uses = x == 0 ? uses0 : uses1;
        if (j == 0 && uses > 0 && !mbar_wait_fast(bar(kPBarOEmpty + x), (uses - 1) & 1, abort))
          return false;
        if (!mbar_wait_fast(bar(kPBarPFull + x), pv_count & 1, abort)) return false;
        ++pv_count;
        tc_fence_after_sync();
        const uint64_t dv = dv0 + (gt & 1) * kStageStep;
#pragma unroll
        for (int ks = 0; ks < kN / 16; ++ks)
          umma_bf16_ts(tmem + kTmemO + x * D, tmem + kTmemS + x * kN + ks * 8,
                       dv + ks * (2048 >> 4), idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
        return true;
      };
      uint32_t g = 0;  // K/V tiles consumed (all items)
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int slot = k & 1;
        if (!(ok = mbar_wait_fast(bar(kPBarItemFull + slot), (k >> 1) & 1, abort))) break;
        const ItemDesc d = s_item[slot];
        mbar_arrive(bar(kPBarItemEmpty + slot));
        if (d.req < 0) break;
        const ItemGeom ig = item_geom(d, tpt);
        const int n0 = ig.n0, n1 = ig.n1, n_tiles = ig.n_tiles;
        const uint32_t g0 = g;
        ok = mbar_wait_fast(bar(a.q_mode ? kPBarQReady : kPBarQFull), k & 1, abort) &&
             mbar_wait_fast(bar(kPBarFull + (g0 & 1)), (g0 >> 1) & 1, abort);
        if (!ok) break;
        tc_fence_after_sync();
        qk(0, g0);
        if (n1 > 0) qk(1, g0);
        if (n_tiles == 1) umma_commit(bar(kPBarQEmpty));
        for (int j = 0; j < n_tiles && ok; ++j) {
          const uint32_t gj = g0 + static_cast<uint32_t>(j);
          const bool next = j + 1 < n_tiles;
          if (j < n0) ok = pv(kTile0, j, gj);
          // O_0 is final once its last product is done (not held for tile 1's)
          if (ok && j == n0 - 1) umma_commit(bar(kPBarOFull + 0));
          if (ok && next) ok = mbar_wait_fast(bar(kPBarFull + ((gj + 1) & 1)), ((gj + 1) >> 1) & 1, abort);
          if (!ok) break;
          tc_fence_after_sync();
          if (next && j + 1 < n0) qk(0, gj + 1);
          if (j < n1 && !(ok = pv(kTile1, j, gj))) break;
          if (j == n1 - 1) umma_commit(bar(kPBarOFull + 1));
          umma_commit(bar(kPBarEmpty + (gj & 1)));
          if (next && j + 1 < n1) qk(1, gj + 1);
          if (j + 2 == n_tiles) umma_commit(bar(kPBarQEmpty));  // every S of the item issued
        }
        g = g0 + static_cast<uint32_t>(n_tiles);
        ++uses0;
        if (n1 > 0) ++uses1;
      }
      if (!ok) {
        *abort = 1;
        flag_error(a.err, kErrTimeout);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    // Query tile x = warp / 4; warp w owns TMEM lanes 32 (w % 4) .. + 31,
    // one query row per thread, whole rows of S; per item the key-tile loop,
    // then the item's output, then O_x is handed back.
    const int quarter = warp & 3;
    const int x = warp >> 2;
    const int r = quarter * 32 + lane;  // query row == TMEM lane
    const int tt = r / a.group;         // token within the query tile
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t srow = tmem + lane_base + kTmemS + x * kN;
    const uint32_t orow_t = tmem + lane_base + kTmemO + x * D;
    int *state = s_sm_state[warp];  // [0] items, [1] S tiles, [2] items that used tile x
    if (lane == 0) state[0] = state[1] = state[2] = 0;
    __syncwarp();
    bool ok = true;
    for (;;) {
      const int k = state[0];
      const int slot = k & 1;
      if (!(ok = mbar_wait_warp(bar(kPBarItemFull + slot), (k >> 1) & 1, abort))) break;
      const ItemDesc d = s_item[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kPBarItemEmpty + slot));
      if (d.req < 0) break;
      const ItemGeom ig = item_geom(d, tpt);
      const int n_x = x == 0 ? ig.n0 : ig.n1;
      const int tok = x * tpt + tt;  // token within the item
      const int qtok = (tt < tpt && tok < ig.tokens) ? d.t_base + d.j0 + tok : -1;
      const bool valid = qtok >= 0;
      // last key of the tile's first token, and the last key this row may see
      const int min_limit = d.p + d.j0 + x * tpt;
      const int limit = min_limit + (valid ? tt : 0);
      float m_used = -INFINITY, l = 0.f;
      if (a.q_mode != 0) {
        // Fold the softmax scale's sign into the item's Q (both query tiles,
        // all eight softmax warps), before its first S = Q K^T is issued.
        if (!(ok = mbar_wait_warp(bar(kPBarQFull), k & 1, abort))) break;
        uint4 *qs = reinterpret_cast<uint4 *>(smem + S::kQ);
        const uint32_t flip = 0x80008000u;  // the sign bits of a bf16 pair
        for (int i = tid; i < kQTiles * S::kQBytes / 16; i += kSoftmaxWarps * 32) {
          uint4 w = qs[i];
          if (a.q_mode == 1) {
            w.x ^= flip;
            w.y ^= flip;
            w.z ^= flip;
            w.w ^= flip;
          } else {
            w = make_uint4(0u, 0u, 0u, 0u);
          }
          qs[i] = w;
        }
        fence_async_shared();  // generic-proxy writes, read next by tcgen05.mma
        mbar_arrive(bar(kPBarQReady));
      }
      const int s_par = state[1] & 1;  // parity of this item's first S tile
      for (int j = 0; ok && j < n_x; ++j) {
        if (!(ok = mbar_wait_warp(bar(kPBarSFull + x), (s_par ^ j) & 1, abort))) break;
        tc_fence_after_sync();
        // Row max of the raw scores; scale_log2 > 0 commutes with max (a
        // negative or zero softmax scale was folded into Q, see q_mode).
        // The loads return the max of the columns they read; a tile that
        // crosses some row's last key (warp-uniform) takes the max after
        // the mask instead, so a hidden key never sets the reference.
        float v[kN], mx0, mx1, mx2, mx3;
        tmem_ld32_max(srow + 0, *reinterpret_cast<float(*)[32]>(&v[0]), mx0);
        tmem_ld32_max(srow + 32, *reinterpret_cast<float(*)[32]>(&v[32]), mx1);
        tmem_ld32_max(srow + 64, *reinterpret_cast<float(*)[32]>(&v[64]), mx2);
        tmem_ld32_max(srow + 96, *reinterpret_cast<float(*)[32]>(&v[96]), mx3);
        tmem_ld_wait();
        const int key0 = j * kN;
        if (key0 + kN - 1 > min_limit) {
#pragma unroll
          for (int cc = 0; cc < kN; ++cc) v[cc] = key0 + cc <= limit ? v[cc] : -INFINITY;
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
        // Lazy rescale: move the reference max only when a row's max grew by
        // more than 2^kRescaleThreshold (warp-uniform: tcgen05.ld/st are
        // .sync.aligned, so every lane takes part, with factor 1 where its
        // row did not move).
        const bool rescale = j > 0 && __any_sync(0xffffffffu, mt > m_used + kRescaleThreshold);
        float f = 1.f;
        if (j == 0) {
          m_used = mt;  // may be -inf: a row with no visible key in this tile
        } else if (rescale) {
          const float m_new = fmaxf(m_used, mt);
          f = m_used == -INFINITY ? 0.f : fast_exp2(m_used - m_new);
          m_used = m_new;
        }
        const float nm = m_used == -INFINITY ? 0.f : -m_used;
        float sa0 = 0.f, sa1 = 0.f, sb0 = 0.f, sb1 = 0.f;
#pragma unroll
        for (int cc = 0; cc < kN; cc += 32) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float y0, y1;
            fma2(y0, y1, v[cc + 2 * e], v[cc + 2 * e + 1], a.scale_log2, nm);
            y0 = fast_exp2(y0);
            y1 = fast_exp2(y1);
            if (e & 1)
              add2(sb0, sb1, y0, y1);
            else
              add2(sa0, sa1, y0, y1);
            w[e] = pack_bf16(y0, y1);
          }
          tmem_st16u(srow + cc / 2, w);  // P_x: keys cc .. cc + 31 -> columns cc/2 ..
        }
        l = l * f + ((sa0 + sa1) + (sb0 + sb1));
        if (rescale) {
          // O_x is stable: S_x(j) completed, so did PV_x(j - 1) before it.
#pragma unroll 1
          for (int cb = 0; cb < D / 32; ++cb) {
            float o[32];
            tmem_ld32(orow_t + cb * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] *= f;
            tmem_st32(orow_t + cb * 32, o);
          }
        }
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(bar(kPBarPFull + x));
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) {
        state[0] = k + 1;
        state[1] += n_x;
      }
      __syncwarp();
      if (n_x == 0) continue;
      if (!(ok = mbar_wait_warp(bar(kPBarOFull + x), state[2] & 1, abort))) break;
      tc_fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int64_t orow =
          static_cast<int64_t>(valid ? qtok : 0) * a.hq + d.kvh * a.group + (r % a.group);
      {
        // The whole row of O at once (the score registers are free here):
        // one TMEM round trip instead of one per 32 columns.
        float o[D];
#pragma unroll
        for (int cb = 0; cb < D / 32; ++cb)
          tmem_ld32(orow_t + cb * 32, *reinterpret_cast<float(*)[32]>(&o[cb * 32]));
        tmem_ld_wait();
        if (valid) {
          uint4 *dst = reinterpret_cast<uint4 *>(a.o + orow * D);
#pragma unroll
          for (int q8 = 0; q8 < D / 8; ++q8) {
            uint4 u;
            u.x = pack_bf16(o[q8 * 8 + 0] * inv, o[q8 * 8 + 1] * inv);
            u.y = pack_bf16(o[q8 * 8 + 2] * inv, o[q8 * 8 + 3] * inv);
            u.z = pack_bf16(o[q8 * 8 + 4] * inv, o[q8 * 8 + 5] * inv);
            u.w = pack_bf16(o[q8 * 8 + 6] * inv, o[q8 * 8 + 7] * inv);
            dst[q8] = u;
          }
        }
      }
      if (valid && a.lse) a.lse[orow] = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
      tc_fence_before_sync();
      mbar_arrive(bar(kPBarOEmpty + x));  // O_x read out: the next item may overwrite it
      __syncwarp();
      if (lane == 0) ++state[2];
      __syncwarp();
    }
    if (!ok) {
      *abort = 1;
      flag_error(a.err, kErrTimeout);
    }
  }

  // Teardown: every role has left its item loop (normally or through the
  // abort flag); free TMEM once no MMA is in flight.
  if (warp == kMmaWarp && lane == 0 && *abort) {
    umma_commit(bar(kPBarTeardown));  // tracks every MMA this thread issued
    int never = 0;
    mbar_wait(bar(kPBarTeardown), 0, &never);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Copying CTAs of one gather variant resident on an SM at once (looked up
// once per variant).
template <int D, bool kStore>
int gather_ctas_per_sm() {
  static const int n = [] {
    int b = 0;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, extend_gather_kernel<D, kStore>,
                                                         kGatherThreads, 0) == cudaSuccess &&
                   b > 0
               ? b
               : 1;
  }();
  return n;
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

// q [total_q][Hq][D] bf16 as a 3-D tensor, box {64, g, tpt}, 128-byte
// swizzle; zeros outside.
bool q3_map_of(CUtensorMap *m, const void *q, uint64_t total_q, uint64_t hq, uint64_t d,
               uint32_t g, uint32_t tpt) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {d, hq, total_q};
  cuuint64_t strides[2] = {d * 2, hq * d * 2};
  cuuint32_t box[3] = {64, g, tpt};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A 2-D bf16 tensor of `rows` rows of `cols` elements (row-major), read in
// boxes of box_rows rows x 64 columns with 128-byte swizzle; zeros outside.
bool bf16_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

ExtendLayout extend_layout(int32_t batch, int32_t hkv, int32_t d, int64_t max_seq,
                           int64_t max_total_keys) {
  ExtendLayout l{};
  const int64_t seq_pad = ((max_seq > 0 ? max_seq : 1) + 127) & ~int64_t(127);
  const int64_t total = max_total_keys >= 1 ? max_total_keys : static_cast<int64_t>(batch) * seq_pad;
  // Every request's run is its seq_len rounded up to 128: at most 127 rows
  // more per request than the keys present.
  l.cap_rows = ((total + 127) & ~int64_t(127)) + 128 * static_cast<int64_t>(batch);
  l.nbuck = 2 * (seq_pad / 128) + 4;
  l.max_blocks = l.cap_rows / 16 + batch;  // a block holds >= 16 chunk tokens (group <= 16)
  l.kv_bytes = 2ull * static_cast<uint64_t>(hkv) * static_cast<uint64_t>(l.cap_rows) *
               static_cast<uint64_t>(d) * 2ull;
  l.plan_offset = (l.kv_bytes + 255) & ~uint64_t(255);
  l.total_bytes = l.plan_offset + 4ull * static_cast<uint64_t>(plan_ints(batch, l.nbuck, l.max_blocks));
  return l;
}

cudaError_t launch_extend(const PoolGeom &g, int32_t layer, const void *q,
                          const int32_t *qo_indptr, void *o, float *lse,
                          const int32_t *page_table, int64_t table_stride,
                          const int32_t *table_idx, const int32_t *seq_lens, int32_t batch,
                          int32_t total_q, int32_t hq, float scale, const ExtendLayout &lay,
                          void *workspace, int32_t sm_count, unsigned *err, cudaStream_t stream,
                          const ExtendMode &mode) {
  const uint64_t ws_rows = 2ull * static_cast<uint64_t>(g.hkv) * static_cast<uint64_t>(lay.cap_rows);
  const uint64_t q_rows = static_cast<uint64_t>(total_q) * hq;
  if (ws_rows >= (1ull << 31) || q_rows >= (1ull << 31) || lay.max_blocks >= (int64_t(1) << 28))
    return cudaErrorInvalidValue;

  GatherArgs ga{};
  ga.pool = static_cast<const __nv_bfloat16 *>(g.base);
  ga.slots = g.slots;
  ga.num_layers = g.num_layers;
  ga.layer = layer;
  ga.page_size = g.page_size;
  ga.hkv = g.hkv;
  ga.page_table = page_table;
  ga.table_stride = table_stride;
  ga.table_idx = table_idx;
  ga.seq_lens = seq_lens;
  ga.batch = batch;
  ga.row_capacity = table_stride * g.page_size;
  ga.cap_rows = static_cast<int32_t>(lay.cap_rows);
  ga.nbuck = static_cast<int32_t>(lay.nbuck);
  ga.max_blocks = static_cast<int32_t>(lay.max_blocks);
  ga.ws = static_cast<__nv_bfloat16 *>(workspace);
  ga.err = err;
  ga.qo_indptr = qo_indptr;
  ga.total_q = total_q;
  ga.tokens_per_tile = kM / (hq / g.hkv);
  ga.k_new = static_cast<const __nv_bfloat16 *>(mode.k_new);
  ga.v_new = static_cast<const __nv_bfloat16 *>(mode.v_new);
  ga.kv_row_stride = mode.kv_row_stride;
  ga.pool_w = static_cast<__nv_bfloat16 *>(const_cast<void *>(g.base));
  ga.plan = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(workspace) + lay.plan_offset);

  ExtendArgs a{};
  a.qo_indptr = qo_indptr;
  a.o = static_cast<__nv_bfloat16 *>(o);
  a.lse = lse;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.hkv = g.hkv;
  a.total_q = total_q;
  a.hq = hq;
  a.group = hq / g.hkv;
  a.tokens_per_tile = kM / a.group;
  a.cap_rows = ga.cap_rows;
  a.nbuck = ga.nbuck;
  a.max_blocks = ga.max_blocks;
  a.q_mode = scale > 0.f ? 0 : (scale < 0.f ? 1 : 2);
  a.scale_log2 = scale > 0.f ? scale * kLog2e : (scale < 0.f ? -scale * kLog2e : kLog2e);
  a.err = err;
  a.plan = ga.plan;
  CUtensorMap kv_map, q_map;
  if (!bf16_map(&kv_map, workspace, ws_rows, static_cast<uint64_t>(g.d), kN) ||
      !q3_map_of(&q_map, q, static_cast<uint64_t>(total_q), static_cast<uint64_t>(hq),
                 static_cast<uint64_t>(g.d), static_cast<uint32_t>(a.group),
                 static_cast<uint32_t>(a.tokens_per_tile)))
    return cudaErrorInvalidValue;
  const int64_t per_cta = static_cast<int64_t>(kQTiles) * a.tokens_per_tile;
  const int64_t tiles = (static_cast<int64_t>(total_q) + per_cta - 1) / per_cta + batch;
  if (tiles > 65535 || batch >= 65535) return cudaErrorInvalidConfiguration;
  // the planner, then two waves of copying CTAs (twice as many as are
  // resident at once) looping over the 16-row chunks
  const int64_t chunks = lay.cap_rows / kGatherKeys;
  const int per_sm = g.d == 128 ? (ga.k_new ? gather_ctas_per_sm<128, true>() : gather_ctas_per_sm<128, false>())
                                : (ga.k_new ? gather_ctas_per_sm<64, true>() : gather_ctas_per_sm<64, false>());
  const int64_t copiers = std::min<int64_t>(
      chunks, static_cast<int64_t>(sm_count > 0 ? sm_count : 1) * per_sm * kGatherWaves);
  const dim3 ggrid(static_cast<unsigned>(1 + copiers));
  // attention: one CTA per SM (whole-SM shared memory), at most one per work item
  const int64_t items = static_cast<int64_t>(g.hkv) * tiles;
  const dim3 pgrid(static_cast<unsigned>(std::min<int64_t>(sm_count > 0 ? sm_count : 1, items)));
  cudaError_t e;
  if (g.d == 128) {
    e = ga.k_new ? launch_pdl(extend_gather_kernel<128, true>, ggrid, dim3(kGatherThreads), 0,
                              stream, ga)
                 : launch_pdl(extend_gather_kernel<128, false>, ggrid, dim3(kGatherThreads), 0,
                              stream, ga);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(extend_tc_persistent_kernel<128>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<128>::kTotal);
    if (e != cudaSuccess) return e;
    e = launch_pdl(extend_tc_persistent_kernel<128>, pgrid, dim3(kThreads), Smem<128>::kTotal,
                   stream, kv_map, q_map, a);
  } else {
    e = ga.k_new ? launch_pdl(extend_gather_kernel<64, true>, ggrid, dim3(kGatherThreads), 0,
                              stream, ga)
                 : launch_pdl(extend_gather_kernel<64, false>, ggrid, dim3(kGatherThreads), 0,
                              stream, ga);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(extend_tc_persistent_kernel<64>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<64>::kTotal);
    if (e != cudaSuccess) return e;
    e = launch_pdl(extend_tc_persistent_kernel<64>, pgrid, dim3(kThreads), Smem<64>::kTotal,
                   stream, kv_map, q_map, a);
  }
  return e;
}

}  // namespace pkv
