// extend.cu - paged extend (chunked-prefill) attention.
//
// What it computes ("Code Notes: mini-sglang", Scheduler Layer table,
// PrefillManager row; "Introduction", Key Features, Chunked Prefill and Radix
// Cache): request r's chunk of c_r new queries sits after a cached prefix of
// p_r = seq_len[r] - c_r keys; chunk query j attends to keys 0 .. p_r + j of
// the request's page_table row (full prefix, causal within the chunk).
//
// This version tiles on the m16n8k16 tensor-core MMA:
//  * A CTA (4 warps) owns 64 query rows of one kv head: 64 / g chunk tokens
//    x the g q heads that read that kv head, so each gathered K/V tile feeds
//    g q heads at once.
//  * K/V tiles of 64 keys are gathered through the page table with 16-byte
//    cp.async (zero fill past the end) into XOR-swizzled shared memory, two
//    stages deep; Q stays in registers as MMA A fragments.
//  * S = Q K^T and O += P V per warp (16 rows), online softmax in the log2
//    domain, causal mask only on tiles that cross the diagonal.
//  * CTAs are issued from the end of each request's chunk backwards, so the
//    longest key ranges start first.
#include <math.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kRows = kWarps * 16;  // query rows per CTA
constexpr int kKeys = 64;           // keys per K/V tile
constexpr int kStages = 2;

template <int D>
struct ExtendSmem {
  static constexpr int kTileBytes = kKeys * D * 2;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kQBytes = kRows * D * 2;
  static constexpr int kTotal = kStages * kStageBytes + kQBytes;
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
  int32_t tokens_per_cta;  // floor(64 / group)
  float scale_log2;
  unsigned *err;
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2) extend_kernel(const ExtendArgs a) {
  using S = ExtendSmem<D>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_req, s_j0, s_c, s_p, s_row;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int kvh = blockIdx.x;

  grid_dependency_wait();  // the chunk's K/V may come from the previous kernel (store_kv)
  // Which (request, token tile) this CTA owns; tiles are taken from the end.
  if (tid == 0) {
    const int tile = static_cast<int>(gridDim.y) - 1 - static_cast<int>(blockIdx.y);
    int acc = 0;
    int req = -1, j0 = 0, c = 0, p = 0, row = 0;
    for (int r = 0; r < a.batch; ++r) {
      const int beg = a.qo_indptr[r];
      const int end = a.qo_indptr[r + 1];
      const int cr = end - beg;
      if (cr < 0 || end > a.total_q) {
        if (blockIdx.x == 0 && blockIdx.y == 0) flag_error(a.err, kErrIndptr);
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
        if (kvh == 0) flag_error(a.err, p < 0 ? kErrIndptr : (row < 0 ? kErrTableIdx : kErrSeqLen));
        req = -1;
      }
    }
    s_req = req;
    s_j0 = j0;
    s_c = c;
    s_p = p;
    s_row = row;
  }
  __syncthreads();
  const int req = s_req;
  if (req < 0) return;
  const int j0 = s_j0, c = s_c, p = s_p;
  const int32_t *row = a.page_table + static_cast<int64_t>(s_row) * a.table_stride;
  const int t_base = a.qo_indptr[req];
  const int tokens = min(a.tokens_per_cta, c - j0);
  const int n_keys = p + j0 + tokens;         // keys the last token of the tile sees
  const int n_tiles = (n_keys + kKeys - 1) / kKeys;
  const int diag_start = p + j0;              // keys below this are seen by every row

  const uint32_t sbase = smem_addr(smem);
  const uint32_t qs = sbase + kStages * S::kStageBytes;
  constexpr int CPK = D / 8;

  // Q rows: row r -> token j0 + r / g, q head kvh * g + r % g.
  for (int idx = tid; idx < kRows * CPK; idx += kThreads) {
    const int r = idx / CPK, ch = idx % CPK;
    const int t = r / a.group, hh = r % a.group;
    const bool ok = t < tokens;
    const __nv_bfloat16 *src =
        ok ? a.q + (static_cast<int64_t>(t_base + j0 + t) * a.hq + kvh * a.group + hh) * D + ch * 8
           : a.q;
    cp_async_16(qs + swz<D>(r, ch), src, ok ? 16 : 0);
  }

  const int64_t slot_stride = static_cast<int64_t>(a.hkv) * D;
  const __nv_bfloat16 *kbase =
      a.pool + static_cast<int64_t>(a.layer) * a.plane + static_cast<int64_t>(kvh) * D;
  const __nv_bfloat16 *vbase = a.pool + (static_cast<int64_t>(a.num_layers) + a.layer) * a.plane +
                               static_cast<int64_t>(kvh) * D;
  const int P = a.page_size;

  auto issue = [&](int kt, int stage) {
    const uint32_t st = sbase + stage * S::kStageBytes;
    for (int idx = tid; idx < kKeys * CPK; idx += kThreads) {
      const int r = idx / CPK, ch = idx % CPK;
      const int key = kt * kKeys + r;
      bool ok = key < n_keys;
      int64_t off = 0;
      if (ok) {
        const int pi = (P == 1) ? key : key / P;
        const long long pg = row[pi];
        const long long s = pg * P + (key - pi * P);
        if (pg < 0 || s >= a.slots) {
          if (ch == 0) flag_error(a.err, kErrPage);
          ok = false;
        } else {
          off = s * slot_stride + ch * 8;
        }
      }
      const uint32_t d = st + swz<D>(r, ch);
      cp_async_16(d, ok ? kbase + off : a.pool, ok ? 16 : 0);
      cp_async_16(d + S::kTileBytes, ok ? vbase + off : a.pool, ok ? 16 : 0);
    }
  };

  issue(0, 0);
  cp_async_commit();  // group 0: Q + tile 0

  // This thread's two rows: ra = 16 * warp + lane / 4 and rb = ra + 8.
  const int ra = warp * 16 + (lane >> 2);
  const int rb = ra + 8;
  const int ta = ra / a.group, tb = rb / a.group;
  const bool va = ta < tokens, vb = tb < tokens;
  const int lim_a = p + j0 + ta;  // last key row a may see
  const int lim_b = p + j0 + tb;

  uint32_t qa[D / 16][4];
  float acc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;

  for (int kt = 0; kt < n_tiles; ++kt) {
    if (kt + 1 < n_tiles) issue(kt + 1, (kt + 1) % kStages);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (kt == 0) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        ldmatrix_x4(qs + swz<D>(warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, ks * 2 + (lane >> 4)),
                    qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
    }
    const uint32_t kst = sbase + (kt % kStages) * S::kStageBytes;
    const uint32_t vst = kst + S::kTileBytes;

    float s[kKeys / 8][4];
#pragma unroll
    for (int nt = 0; nt < kKeys / 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
      for (int np = 0; np < kKeys / 16; ++np) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(kst + swz<D>(np * 16 + (lane & 7) + (lane >> 4) * 8, ks * 2 + ((lane >> 3) & 1)),
                    b0, b1, b2, b3);
        mma_bf16_16816(s[2 * np], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
        mma_bf16_16816(s[2 * np + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
      }
    }

    const bool need_mask = (kt + 1) * kKeys > diag_start + 1 || (kt + 1) * kKeys > n_keys;
    float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < kKeys / 8; ++nt) {
      const int key = kt * kKeys + nt * 8 + (lane & 3) * 2;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float xa = s[nt][e] * a.scale_log2;
        float xb = s[nt][2 + e] * a.scale_log2;
        if (need_mask) {
          if (!va || key + e > lim_a) xa = -INFINITY;
          if (!vb || key + e > lim_b) xb = -INFINITY;
        }
        s[nt][e] = xa;
        s[nt][2 + e] = xb;
        mxa = fmaxf(mxa, xa);
        mxb = fmaxf(mxb, xb);
      }
    }
    mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 1));
    mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 2));
    mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
    mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
    const float mna = fmaxf(ma, mxa), mnb = fmaxf(mb, mxb);
    const float refa = mna == -INFINITY ? 0.f : mna;
    const float refb = mnb == -INFINITY ? 0.f : mnb;
    const float ala = fast_exp2(ma - refa), alb = fast_exp2(mb - refb);
    ma = mna;
    mb = mnb;
    float suma = 0.f, sumb = 0.f;
    uint32_t pa[kKeys / 16][4];
#pragma unroll
    for (int nt = 0; nt < kKeys / 8; ++nt) {
      const float p0 = fast_exp2(s[nt][0] - refa), p1 = fast_exp2(s[nt][1] - refa);
      const float p2 = fast_exp2(s[nt][2] - refb), p3 = fast_exp2(s[nt][3] - refb);
      suma += p0 + p1;
      sumb += p2 + p3;
      pa[nt / 2][(nt & 1) * 2 + 0] = pack_bf16(p0, p1);
      pa[nt / 2][(nt & 1) * 2 + 1] = pack_bf16(p2, p3);
    }
    la = la * ala + suma;
    lb = lb * alb + sumb;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      acc[i][0] *= ala;
      acc[i][1] *= ala;
      acc[i][2] *= alb;
      acc[i][3] *= alb;
    }
#pragma unroll
    for (int kk = 0; kk < kKeys / 16; ++kk) {
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(vst + swz<D>(kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, dp * 2 + (lane >> 4)),
                          b0, b1, b2, b3);
        mma_bf16_16816(acc[2 * dp], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b0, b1);
        mma_bf16_16816(acc[2 * dp + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b2, b3);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  la += __shfl_xor_sync(0xffffffffu, la, 1);
  la += __shfl_xor_sync(0xffffffffu, la, 2);
  lb += __shfl_xor_sync(0xffffffffu, lb, 1);
  lb += __shfl_xor_sync(0xffffffffu, lb, 2);
  const float inva = la > 0.f ? 1.f / la : 0.f;
  const float invb = lb > 0.f ? 1.f / lb : 0.f;
  const int64_t orow_a = static_cast<int64_t>(t_base + j0 + ta) * a.hq + kvh * a.group + ra % a.group;
  const int64_t orow_b = static_cast<int64_t>(t_base + j0 + tb) * a.hq + kvh * a.group + rb % a.group;
#pragma unroll
  for (int i = 0; i < D / 8; ++i) {
    const int d = i * 8 + (lane & 3) * 2;
    if (va)
      *reinterpret_cast<uint32_t *>(a.o + orow_a * D + d) = pack_bf16(acc[i][0] * inva, acc[i][1] * inva);
    if (vb)
      *reinterpret_cast<uint32_t *>(a.o + orow_b * D + d) = pack_bf16(acc[i][2] * invb, acc[i][3] * invb);
  }
  if (a.lse && (lane & 3) == 0) {
    if (va) a.lse[orow_a] = la > 0.f ? (ma + __log2f(la)) * kLn2 : -INFINITY;
    if (vb) a.lse[orow_b] = lb > 0.f ? (mb + __log2f(lb)) * kLn2 : -INFINITY;
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
  a.tokens_per_cta = kRows / a.group;
  a.scale_log2 = scale * kLog2e;
  a.err = err;
  const int64_t tiles = (static_cast<int64_t>(total_q) + a.tokens_per_cta - 1) / a.tokens_per_cta + batch;
  if (tiles > 65535) return cudaErrorInvalidConfiguration;
  const dim3 grid(g.hkv, static_cast<unsigned>(tiles));
  cudaError_t e;
  if (g.d == 128) {
    e = cudaFuncSetAttribute(extend_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             ExtendSmem<128>::kTotal);
    if (e != cudaSuccess) return e;
    e = launch_pdl(extend_kernel<128>, grid, dim3(kThreads), ExtendSmem<128>::kTotal, stream, a);
  } else {
    e = cudaFuncSetAttribute(extend_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             ExtendSmem<64>::kTotal);
    if (e != cudaSuccess) return e;
    e = launch_pdl(extend_kernel<64>, grid, dim3(kThreads), ExtendSmem<64>::kTotal, stream, a);
  }
  return e;
}

}  // namespace pkv
