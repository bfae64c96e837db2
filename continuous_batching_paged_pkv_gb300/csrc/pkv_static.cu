// pkv_attention_no_alloc: pkv_attention with its scratch in a file-scope
// device array, for callers that must not allocate device memory.
//
// Some callers cannot hand the library a workspace they allocated: a host
// process that reserves all device memory in its own arena at start-up and
// forbids further cudaMalloc, or a latency-critical serving loop that may not
// allocate (and so may not synchronise) between steps. For them this entry
// point keeps the span partials in `g_pkv_scratch`, a fixed array that every
// GPU loading this library holds until the process exits.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "pkv.h"

namespace {

static __device__ __align__(256) unsigned char g_pkv_scratch[PKV_NO_ALLOC_SCRATCH_BYTES];

// Device address of g_pkv_scratch per device, looked up once with that device
// current. In host code the array's name is only a host-side stand-in, so the
// kernels must get this address instead.
void *scratch_address(pkv_status *status) {
  static void *addr[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *status = PKV_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pkv_scratch) != cudaSuccess || !p) {
      *status = PKV_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = p;
  }
  *status = PKV_OK;
  return addr[dev];
}

}  // namespace

extern "C" pkv_status pkv_attention_no_alloc(
    const void *q, const int32_t *cu_seqlens_q, int32_t num_seqs, int64_t total_q, const int32_t *seq_slot,
    const int32_t *context_lens, const int32_t *block_tables, int32_t max_slots, int32_t max_blocks_per_slot,
    int32_t block_size, const void *k_pool, const void *v_pool, int64_t num_blocks, int32_t num_q_heads,
    int32_t num_kv_heads, int32_t head_dim, float scale, const int32_t *work, const pkv_work_info *info,
    void *out, uint32_t *device_status, pkv_stream_t stream) {
  if (!info) return PKV_ERR_INVALID_ARG;
  // Reject steps whose partials do not fit before touching the GPU.
  if (info->workspace_bytes > PKV_NO_ALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE_TOO_SMALL;
  pkv_status st = PKV_OK;
  void *scratch = scratch_address(&st);
  if (st != PKV_OK) return st;
  return pkv_attention(q, cu_seqlens_q, num_seqs, total_q, seq_slot, context_lens, block_tables, max_slots,
                       max_blocks_per_slot, block_size, k_pool, v_pool, num_blocks, num_q_heads, num_kv_heads,
                       head_dim, scale, work, info, out, scratch, PKV_NO_ALLOC_SCRATCH_BYTES, device_status, stream);
}
