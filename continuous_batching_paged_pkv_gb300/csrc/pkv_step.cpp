// Host-staged step: the step's inputs travel to the device as one copy from a
// single host staging buffer, the work list is planned straight into that
// buffer, and the output comes back as one copy (or, on request, the kernels
// write the output straight to host memory, and for small steps without
// prompt chunks also read the staging buffer in place). Everything is
// enqueued on the caller's stream; nothing here synchronises.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

constexpr uint64_t kAlign = 256;

uint64_t align_up(uint64_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

// Device address of host memory the device can reach (page-locked under unified
// addressing), or nullptr.
void *device_view(void *host) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, host) != cudaSuccess) {
    cudaGetLastError();  // clear the error of an unknown pointer
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

}  // namespace

extern "C" {

pkv_status pkv_stage_layout_init(pkv_stage_layout *layout, int64_t total_q, int32_t num_seqs,
                                 int32_t max_slots, int32_t max_blocks_per_slot,
                                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim) {
  if (!layout || total_q < 0 || num_seqs < 0 || max_slots <= 0 || max_blocks_per_slot <= 0 ||
      num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return PKV_ERR_INVALID_ARG;
  // every size below stays far from 2^64 under these bounds
  if (total_q > (int64_t(1) << 31) || num_q_heads > 4096 || head_dim > 4096 ||
      int64_t(max_slots) * max_blocks_per_slot > (int64_t(1) << 34))
    return PKV_ERR_INVALID_ARG;
  std::memset(layout, 0, sizeof(*layout));
  layout->total_q = total_q;
  layout->num_seqs = num_seqs;
  layout->max_slots = max_slots;
  layout->max_blocks_per_slot = max_blocks_per_slot;
  layout->num_q_heads = num_q_heads;
  layout->num_kv_heads = num_kv_heads;
  layout->head_dim = head_dim;
  const uint64_t T = static_cast<uint64_t>(total_q);
  uint64_t off = 0;
  auto take = [&off](uint64_t bytes) {
    const uint64_t at = off;
    off = align_up(off + bytes);
    return at;
  };
  layout->q = take(T * num_q_heads * head_dim * 2);
  layout->k_new = take(T * num_kv_heads * head_dim * 2);
  layout->v_new = take(T * num_kv_heads * head_dim * 2);
  layout->slot_mapping = take(T * 8);
  layout->cu_seqlens_q = take((static_cast<uint64_t>(num_seqs) + 1) * 4);
  layout->seq_slot = take(static_cast<uint64_t>(num_seqs) * 4);
  layout->context_lens = take(static_cast<uint64_t>(max_slots) * 4);
  layout->block_tables = take(static_cast<uint64_t>(max_slots) * max_blocks_per_slot * 4);
  layout->work = off;
  return PKV_OK;
}

pkv_status pkv_step(const pkv_stage_layout *layout, void *host_stage, uint64_t host_stage_bytes,
                    void *device_stage, uint64_t device_stage_bytes, void *k_pool, void *v_pool,
                    int64_t num_blocks, int32_t block_size, float scale, void *workspace,
                    uint64_t workspace_bytes, void *out, void *out_host, uint32_t *device_status,
                    pkv_stream_t stream, pkv_work_info *info_out, uint32_t options) {
  if (!layout || !host_stage || !device_stage || host_stage_bytes < layout->work ||
      (reinterpret_cast<uintptr_t>(device_stage) & (kAlign - 1)) != 0)
    return PKV_ERR_INVALID_ARG;
  const pkv_stage_layout &L = *layout;
  uint8_t *h = static_cast<uint8_t *>(host_stage);
  const int32_t *cu = reinterpret_cast<const int32_t *>(h + L.cu_seqlens_q);
  if (cu[L.num_seqs] != L.total_q) return PKV_ERR_INVALID_ARG;

  // 1. the work list, planned into the staging buffer
  pkv_work_info info;
  std::memset(&info, 0, sizeof(info));
  const int64_t capacity = static_cast<int64_t>((host_stage_bytes - L.work) / 4);
  pkv_status st = pkv_plan_work(cu, L.num_seqs, reinterpret_cast<const int32_t *>(h + L.seq_slot),
                                reinterpret_cast<const int32_t *>(h + L.context_lens), L.max_slots,
                                L.max_blocks_per_slot, block_size, L.num_q_heads, L.num_kv_heads, L.head_dim,
                                reinterpret_cast<int32_t *>(h + L.work), capacity, &info);
  if (info_out) *info_out = info;
  if (st != PKV_OK) return st;
  const uint64_t bytes = L.work + static_cast<uint64_t>(info.work_words) * 4;
  if (bytes > device_stage_bytes || info.workspace_bytes > workspace_bytes) return PKV_ERR_WORKSPACE_TOO_SMALL;
  if (L.total_q > 0 && !out) return PKV_ERR_INVALID_ARG;

  // 2. one copy in, or (small steps without prompt chunks, on request) the
  //    staged inputs read in place; on request the output goes straight to
  //    out_host
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *d = nullptr;
  void *out_dev = out;
  bool out_direct = false;  // the kernels write the output rows straight into out_host
  if (options & PKV_STEP_IN_PLACE) {
    void *outv = out_host ? device_view(out_host) : out;
    if (outv) {
      out_dev = outv;
      out_direct = out_host != nullptr;
      if (info.num_prefill_items == 0 && bytes <= PKV_STEP_IN_PLACE_MAX_BYTES)
        d = static_cast<uint8_t *>(device_view(host_stage));
    }
  }
  const bool in_place = d != nullptr;
  if (!in_place) {
    if (cudaMemcpyAsync(device_stage, host_stage, bytes, cudaMemcpyHostToDevice, cs) != cudaSuccess)
      return PKV_ERR_CUDA;
    d = static_cast<uint8_t *>(device_stage);
  }

  // 3-4. the cache write, then attention, from the staged copies
  st = pkv_cache_write(d + L.k_new, d + L.v_new, reinterpret_cast<const int64_t *>(d + L.slot_mapping), L.total_q,
                       k_pool, v_pool, num_blocks, block_size, L.num_kv_heads, L.head_dim, device_status, stream);
  if (st != PKV_OK) return st;
  st = pkv::attention(d + L.q, reinterpret_cast<const int32_t *>(d + L.cu_seqlens_q), L.num_seqs, L.total_q,
                      reinterpret_cast<const int32_t *>(d + L.seq_slot),
                      reinterpret_cast<const int32_t *>(d + L.context_lens),
                      reinterpret_cast<const int32_t *>(d + L.block_tables), L.max_slots, L.max_blocks_per_slot,
                      block_size, k_pool, v_pool, num_blocks, L.num_q_heads, L.num_kv_heads, L.head_dim, scale,
                      reinterpret_cast<const int32_t *>(d + L.work), &info, out_dev, workspace, workspace_bytes,
                      device_status, stream, out_direct);
  if (st != PKV_OK) return st;

  // 5. one copy out (none when the output went straight to out_host)
  if (out_host && L.total_q > 0 && !out_direct) {
    const uint64_t out_bytes = static_cast<uint64_t>(L.total_q) * L.num_q_heads * L.head_dim * 2;
    if (cudaMemcpyAsync(out_host, out, out_bytes, cudaMemcpyDeviceToHost, cs) != cudaSuccess) return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

}  // extern "C"
