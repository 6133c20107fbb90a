// kv_store.cu - store_kv: scatter each new token's K and V rows into the
// paged pool at its out_loc slot ("Code Notes: mini-sglang", Engine Layer
// table, BaseKVCachePool row).
//
// A token's K (or V) row for all kv heads is Hkv * D contiguous bf16 in both
// the source and the pool, so the copy is a gather-free scatter of 16-byte
// chunks: consecutive threads move consecutive chunks of one row, which
// makes both the read and the write fully coalesced. The kernel is
// HBM/latency bound (2 * N * Hkv * D * 2 bytes read and written); at decode
// sizes it is a few microseconds and launch-bound, which is what CUDA-graph
// replay of the decode step is for.
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__global__ void __launch_bounds__(256)
    kv_store_kernel(__nv_bfloat16 *__restrict__ pool, int64_t plane, int64_t slots,
                    int32_t layer, int32_t num_layers, const __nv_bfloat16 *__restrict__ k,
                    const __nv_bfloat16 *__restrict__ v, int64_t row_stride,
                    const int32_t *__restrict__ out_loc, int64_t n, int32_t chunks_per_row,
                    unsigned *err) {
  grid_dependency_wait();    // k, v, out_loc may come from the previous kernel
  grid_dependents_launch();  // let the attention kernel that follows get scheduled
  const int64_t total = n * 2 * chunks_per_row;
  const int64_t row_elems = static_cast<int64_t>(chunks_per_row) * 8;
  for (int64_t w = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; w < total;
       w += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t ch = w % chunks_per_row;
    const int64_t rest = w / chunks_per_row;
    const int c = static_cast<int>(rest % 2);  // 0 = K, 1 = V
    const int64_t i = rest / 2;
    const int64_t slot = out_loc[i];
    if (slot < 0 || slot >= slots) {  // never write outside the pool
      if (ch == 0 && c == 0) flag_error(err, kErrOutLoc);
      continue;
    }
    const __nv_bfloat16 *src = (c ? v : k) + i * row_stride + ch * 8;
    __nv_bfloat16 *dst = pool + (static_cast<int64_t>(c) * num_layers + layer) * plane +
                         slot * row_elems + ch * 8;
    *reinterpret_cast<uint4 *>(dst) = __ldg(reinterpret_cast<const uint4 *>(src));
  }
}

}  // namespace

cudaError_t launch_kv_store(const PoolGeom &g, int32_t layer, const void *k, const void *v,
                            int64_t row_stride, const int32_t *out_loc, int64_t n,
                            int32_t sm_count, unsigned *err, cudaStream_t stream) {
  const int32_t chunks = g.hkv * g.d / 8;
  const int64_t total = n * 2 * chunks;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(sm_count) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(kv_store_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0,
                    stream, static_cast<__nv_bfloat16 *>(const_cast<void *>(g.base)), g.plane,
                    g.slots, layer, g.num_layers, static_cast<const __nv_bfloat16 *>(k),
                    static_cast<const __nv_bfloat16 *>(v), row_stride, out_loc, n, chunks, err);
}

}  // namespace pkv
