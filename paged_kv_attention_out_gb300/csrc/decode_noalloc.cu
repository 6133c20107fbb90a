// decode_noalloc.cu - decode attention for callers that cannot allocate.
//
// pkv_paged_decode_attn needs a caller-provided workspace for the partial
// states of split rows. Some callers have no way to provide one: a plugin
// inside a host framework that owns all device memory and offers the plugin
// no allocation hook, or a latency-critical serving loop where cudaMalloc is
// forbidden because it can synchronise the device and can fail with
// out-of-memory in the middle of a step. This file gives them
// pkv_paged_decode_attn_noalloc, which runs the same kernels with the split
// scratch taken from a fixed array in device memory that this library owns.
//
// The array is a file-scope static __device__ buffer of kScratchBytes; every
// GPU that loads the library holds it until the process exits. Host code
// cannot use the array's name as a device address, so each device looks up
// the real address once, with that device current, via cudaGetSymbolAddress.
// Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <stdio.h>

#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

constexpr size_t kScratchBytes = PKV_NOALLOC_SCRATCH_BYTES;

// Split-KV partial states (o and lse of every split) of the no-alloc decode.
// Shared by every call on a device; holds whatever the last call left there.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_decode_scratch on the current device (looked up once
// per device, with that device current).
pkv_status scratch_for_current_device(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return pkv::fail_status(PKV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return pkv::fail_status(PKV_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || !p)
      return pkv::fail_status(PKV_ERR_CUDA, "cudaGetSymbolAddress(decode scratch): %s",
                              cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_paged_decode_attn_noalloc(
    const pkv_pool *pool, int32_t layer, const void *q, void *o, float *lse,
    const int32_t *page_table, int64_t table_stride, const int32_t *table_idx,
    const int32_t *seq_lens, int32_t batch, int32_t num_q_heads, float scale,
    int32_t max_seq_len_hint, cudaStream_t stream) {
  if (pool) {
    const size_t need = pkv_decode_workspace_size(batch, num_q_heads, pool->num_kv_heads,
                                                  pool->head_dim, max_seq_len_hint);
    if (need > kScratchBytes)
      return pkv::fail_status(
          PKV_ERR_WORKSPACE_TOO_SMALL,
          "no-alloc decode: the split state needs %zu bytes but the static scratch holds %zu; "
          "lower batch or max_seq_len_hint, or call pkv_paged_decode_attn with a workspace",
          need, kScratchBytes);
  }
  void *scratch = nullptr;
  const pkv_status s = scratch_for_current_device(&scratch);
  if (s != PKV_OK) return s;
  // The split partials need no zeroing: every split writes its own slot before
  // the merge reads it, within the same call.
  return pkv_paged_decode_attn(pool, layer, q, o, lse, page_table, table_stride, table_idx,
                               seq_lens, batch, num_q_heads, scale, max_seq_len_hint, scratch,
                               kScratchBytes, stream);
}
