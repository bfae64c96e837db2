// Internal interfaces between the C-ABI layer (pkv_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "pkv.h"

namespace pkv {

// Keys per 16-row sub-tile: the unit every kernel loads with one TMA box per
// 64-column half of head_dim.
constexpr int kSubKeys = 16;

struct StepArgs {
  const void *q;
  const void *k_pool;
  const void *v_pool;
  const int32_t *cu_seqlens_q;
  const int32_t *seq_slot;
  const int32_t *context_lens;
  const int32_t *block_tables;
  int32_t num_seqs, max_slots, max_blocks_per_slot, block_size;
  int64_t num_blocks, total_q;
  int32_t num_q_heads, num_kv_heads, group, head_dim;
  int32_t decode_rows_max;  // most rows of a segment on the decode path (1 for plain decode)
  float scale_log2;  // softmax scale times log2(e)
  const int32_t *work;
  void *out;
  float *partial_acc;  // [num_partials][Hq][D]
  float *partial_ml;   // [num_partials][Hq][2]  (running max in log2 units, sum)
  uint32_t *status;
  // Workspace word the decode kernel hands out tasks from past its first
  // three static rounds (nullptr: every task is assigned statically). The
  // launch zeroes it on the stream first.
  uint32_t *task_counter;
  // The chunk kernel's K/V pool is written by the kernel right before it (the
  // 8-bit and 4-bit paths' widening pass): wait for it before any K/V load.
  // Otherwise only the tiles holding this step's rows wait for the cache write.
  int32_t kv_from_previous;
  // `out` is page-locked host memory reached through its device address: the
  // chunk kernel then stages its rows in shared memory and stores whole rows,
  // which the host link carries at its copy rate (one 16-byte piece of 32
  // different rows per store it carries far slower).
  int32_t out_on_host;
};

// pkv_attention with the output's location: out_on_host marks `out` as host
// memory (pkv_step's output written straight to the caller's host buffer).
pkv_status attention(const void *q, const int32_t *cu_seqlens_q, int32_t num_seqs, int64_t total_q,
                     const int32_t *seq_slot, const int32_t *context_lens, const int32_t *block_tables,
                     int32_t max_slots, int32_t max_blocks_per_slot, int32_t block_size, const void *k_pool,
                     const void *v_pool, int64_t num_blocks, int32_t num_q_heads, int32_t num_kv_heads,
                     int32_t head_dim, float scale, const int32_t *work, const pkv_work_info *info, void *out,
                     void *workspace, uint64_t workspace_bytes, uint32_t *device_status, pkv_stream_t stream,
                     bool out_on_host);

// Rows of more spans than this are merged with four lanes per column.
constexpr int kLongMergeSpans = 64;

// Bytes of workspace after the span partials: the decode kernel's task counter.
constexpr uint64_t kCounterBytes = 256;

cudaError_t launch_cache_write(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                               int64_t num_tokens, void *k_pool, void *v_pool, int64_t num_blocks,
                               int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                               uint32_t *status, cudaStream_t stream);

cudaError_t launch_copy_blocks(const int32_t *pairs, int64_t num_pairs, void *const *arrays,
                               const int64_t *block_bytes, int32_t num_arrays, int64_t num_blocks, uint32_t *status,
                               cudaStream_t stream);

// `beside_chunk`: the chunk kernel of the same step runs at the same time
// (head_dim 128 takes the small per-SM footprint described below).
cudaError_t launch_decode(const StepArgs &a, const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                          int32_t num_items, const int32_t *items, bool beside_chunk, cudaStream_t stream);

// One CTA per (row of a multi-span segment, group of q heads): merges that
// row's span partials. The first `num_long` items (rows of more than two
// span groups) may take four lanes per column.
cudaError_t launch_merge(const StepArgs &a, int32_t num_items, int32_t num_long, const int32_t *items,
                         cudaStream_t stream);

// Block-scaled pools (bits = 8, or 4 at head_dim 128): quantising cache write,
// decode over the codes, and the widening of prompt-chunk histories into a
// bf16 scratch pool.
cudaError_t launch_cache_write_quant(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                                  int64_t num_tokens, void *k_codes, void *k_scales, void *v_codes, void *v_scales,
                                  int64_t num_blocks, int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t bits, uint32_t *status, cudaStream_t stream);
cudaError_t launch_decode_quant(const StepArgs &a, const CUtensorMap &tmap_k_codes, const CUtensorMap &tmap_v_codes,
                             const void *k_scales, const void *v_scales, int32_t num_items, const int32_t *items,
                             int32_t bits, cudaStream_t stream);
cudaError_t launch_widen_quant(const StepArgs &a, const void *k_codes, const void *k_scales, const void *v_codes,
                            const void *v_scales, void *k_out, void *v_out, int32_t *scratch_table,
                            int64_t scratch_blocks, int32_t num_items, const int32_t *items, int32_t bits,
                            cudaStream_t stream);

cudaError_t launch_prefill(const StepArgs &a, const CUtensorMap &tmap_q, int32_t rows_per_tile,
                           int32_t num_items, const int32_t *items, cudaStream_t stream);
// head_dim 128: items are tile pairs, run by clusters of two CTAs.
// `beside_decode`: the step also has decode rows, whose kernel runs at the
// same time; the chunk kernel then keeps fewer K/V stages so that a decode CTA
// fits beside each of its CTAs.
cudaError_t launch_prefill_pair(const StepArgs &a, const CUtensorMap &tmap_q, const CUtensorMap &tmap_k,
                                const CUtensorMap &tmap_v, int32_t rows_per_tile, int32_t num_items,
                                const int32_t *items, bool beside_decode, cudaStream_t stream);

// A step with both prompt chunks and decode rows (head_dim 128) runs one CTA
// of each kernel on every SM: the chunk kernel with kPairStagesBesideDecode
// K/V stages (129 KiB of shared memory, 7 warps x 232 registers), the decode
// kernel with kDecodeWarpsBesideChunk warps of kDecodeStagesBesideChunk
// stages (81 KiB, 2 warps x at most 208 registers); together they stay within
// an SM's 228 KiB of shared memory and 64 Ki registers. The tensor-bound chunk
// tiles and the HBM-bound decode streams then share every SM instead of
// queueing for SMs.
constexpr int kPairStagesBesideDecode = 3;
constexpr int kDecodeWarpsBesideChunk = 4;
constexpr int kDecodeStagesBesideChunk = 2;

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel in the stream drains; it calls griddepcontrol.wait
// before touching any input.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Raises a kernel's dynamic shared-memory limit to `smem`, once per device,
// and asks for the largest shared-memory carve-out of the SM's L1 storage: a
// CTA of another kernel can join an SM only under the carve-out that SM was
// configured with, so the kernels meant to share SMs (a chunk CTA beside a
// decode CTA) must all ask for the same, largest one.
// `done` holds one bit per device (devices past 63 set the attributes on every
// call); two host threads racing on a first call both set them, which is harmless.
template <typename Kernel>
cudaError_t allow_smem_once(Kernel *kernel, int smem, std::atomic<uint64_t> &done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev >= 0 && dev < 64 ? 1ull << dev : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Positions per prefill tile: whole GQA groups fit one 128-row MMA tile.
inline int32_t prefill_rows_per_tile(int32_t group) { return 128 / group; }

}  // namespace pkv
