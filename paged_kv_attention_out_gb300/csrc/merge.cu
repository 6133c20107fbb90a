// merge.cu - log-sum-exp merge of two attention states over disjoint key sets.
//
// Exported as pkv_merge_lse so a caller can combine attention over a shared
// (radix-cached) prefix with attention over a private suffix ("Introduction",
// Key Features, Radix Cache): lse = log(e^lse_a + e^lse_b) and
// o = e^(lse_a - lse) o_a + e^(lse_b - lse) o_b. A state with lse = -inf
// contributes nothing. Pure streaming: 2 * rows * heads * (D + 1) fp32 in,
// rows * heads * D out. One warp per (row, head); every lane reads both lse
// values before lane 0 writes, so lse_out may alias an input.
#include <math.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__global__ void __launch_bounds__(256)
    merge_kernel(const float *__restrict__ o_a, const float *__restrict__ lse_a,
                 const float *__restrict__ o_b, const float *__restrict__ lse_b, void *o_out,
                 int out_bf16, float *lse_out, int64_t pairs, int32_t head_dim) {
  grid_dependency_wait();  // the states may come from the previous kernel
  const int lane = threadIdx.x & 31;
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t rh = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5);
       rh < pairs; rh += warps_total) {
    const float la = lse_a[rh];
    const float lb = lse_b[rh];
    __syncwarp();
    float wa, wb, lse;
    if (la == -INFINITY && lb == -INFINITY) {
      wa = wb = 0.f;
      lse = -INFINITY;
    } else if (la == -INFINITY) {
      wa = 0.f;
      wb = 1.f;
      lse = lb;
    } else if (lb == -INFINITY) {
      wa = 1.f;
      wb = 0.f;
      lse = la;
    } else {
      const float m = fmaxf(la, lb);
      const float ea = expf(la - m), eb = expf(lb - m);
      const float z = ea + eb;
      wa = ea / z;
      wb = eb / z;
      lse = m + logf(z);
    }
    const int64_t base = rh * head_dim;
    for (int d = lane * 4; d < head_dim; d += 128) {
      float4 va = make_float4(0.f, 0.f, 0.f, 0.f), vb = va;
      if (wa != 0.f) va = *reinterpret_cast<const float4 *>(o_a + base + d);
      if (wb != 0.f) vb = *reinterpret_cast<const float4 *>(o_b + base + d);
      float4 r;
      r.x = wa * va.x + wb * vb.x;
      r.y = wa * va.y + wb * vb.y;
      r.z = wa * va.z + wb * vb.z;
      r.w = wa * va.w + wb * vb.w;
      if (out_bf16) {
        uint2 packed;
        packed.x = pack_bf16(r.x, r.y);
        packed.y = pack_bf16(r.z, r.w);
        *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(o_out) + base + d) = packed;
      } else {
        *reinterpret_cast<float4 *>(static_cast<float *>(o_out) + base + d) = r;
      }
    }
    if (lane == 0 && lse_out) lse_out[rh] = lse;
  }
}

}  // namespace

cudaError_t launch_merge(const float *o_a, const float *lse_a, const float *o_b,
                         const float *lse_b, void *o_out, bool out_bf16, float *lse_out,
                         int64_t rows, int32_t heads, int32_t head_dim, int32_t sm_count,
                         cudaStream_t stream) {
  const int64_t pairs = rows * heads;
  const int threads = 256;
  int64_t blocks = (pairs + 7) / 8;
  const int64_t cap = static_cast<int64_t>(sm_count) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(merge_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream,
                    o_a, lse_a, o_b, lse_b, o_out, out_bf16 ? 1 : 0, lse_out, pairs, head_dim);
}

}  // namespace pkv
