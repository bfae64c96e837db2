// C-ABI entry points of libpkv that touch the GPU: argument validation on the
// host, TMA tensor-map encoding, kernel launches on the caller's stream (plus
// one library-owned stream per device, forked from and joined back to the
// caller's stream, when a step has both prompt chunks and decode rows), and
// the one synchronising call that reads the device status word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

using EncodeFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeFn encoder() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// A side stream per device for the decode kernels of a step that also has
// prompt chunks: the chunk kernel (tensor-bound) leaves SMs idle and frees
// more as its tiles finish, and the decode kernel (HBM-bound) only needs the
// cache write that precedes the call. The fork and join are events; the mutex
// keeps each call's record/wait pairs together when calls come from several
// host threads.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  std::mutex mu;
  bool ok = false;
};

SideStream *side_stream() {
  static SideStream sides[64];
  static std::once_flag once[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  SideStream *s = &sides[dev];
  std::call_once(once[dev], [s] {
    s->ok = cudaStreamCreateWithFlags(&s->stream, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&s->fork, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&s->join, cudaEventDisableTiming) == cudaSuccess;
  });
  return s->ok ? s : nullptr;
}

bool supported_shape(int32_t block_size, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim) {
  if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0) return false;
  const int32_t g = num_q_heads / num_kv_heads;
  return g >= 1 && g <= 16 && (head_dim == 64 || head_dim == 128) &&
         (block_size == 16 || block_size == 32 || block_size == 64);
}

// Pool tensor [num_blocks*Hkv*bs rows][D] -> boxes of 16 rows x 64 columns, 128B swizzle.
bool encode_pool(CUtensorMap *m, const void *pool, int64_t rows, int32_t head_dim) {
  EncodeFn enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(pkv::kSubKeys)};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(pool), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Key pool at head_dim 128 for the chunk kernel, seen as five dimensions
// (column within a 64-column half, key within 8, half, group of 8 keys within
// the block, block x kv head): one box is a whole 16-key sub-tile, 4 KiB,
// landing as [key group][half][8 keys][128 B] in shared memory, so each
// 8-key group of either half is one 128-byte-swizzle atom.
bool encode_pool_subtiles(CUtensorMap *m, const void *pool, int64_t block_heads, int32_t block_size) {
  EncodeFn enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[5] = {64, 8, 2, static_cast<cuuint64_t>(block_size / 8), static_cast<cuuint64_t>(block_heads)};
  cuuint64_t strides[4] = {256, 128, 2048, static_cast<cuuint64_t>(block_size) * 256};
  cuuint32_t box[5] = {64, 8, 2, static_cast<cuuint32_t>(pkv::kSubKeys / 8), 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(pool), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 8-bit codes [rows][D] -> boxes of 16 whole rows; 128-byte swizzle for
// 128-byte rows (D = 128), 64-byte swizzle for 64-byte rows (D = 64).
// Code rows of head_dim * bits / 8 bytes (128 or 64), 16-row boxes with the
// matching swizzle (128B or 64B).
bool encode_codes(CUtensorMap *m, const void *codes, int64_t rows, int32_t head_dim, int32_t bits) {
  EncodeFn enc = encoder();
  if (!enc) return false;
  const int32_t row_bytes = head_dim * bits / 8;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(row_bytes), static_cast<cuuint32_t>(pkv::kSubKeys)};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(codes), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q [T][Hq][D] -> boxes of (64 columns, G heads, P positions), 128B swizzle.
bool encode_q(CUtensorMap *m, const void *q, int64_t total_q, int32_t hq, int32_t d, int32_t g, int32_t p) {
  EncodeFn enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(hq), static_cast<cuuint64_t>(total_q)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(hq) * d * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(g), static_cast<cuuint32_t>(p)};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

uint64_t align256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

}  // namespace

extern "C" {

pkv_status pkv_cache_write(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                           int64_t num_tokens, void *k_pool, void *v_pool, int64_t num_blocks,
                           int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                           uint32_t *device_status, pkv_stream_t stream) {
  if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0) return PKV_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping || !k_pool || !v_pool) return PKV_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
      !aligned(slot_mapping, 8))
    return PKV_ERR_INVALID_ARG;
  cudaError_t e = pkv::launch_cache_write(k_new, v_new, slot_mapping, num_tokens, k_pool, v_pool, num_blocks,
                                          block_size, num_kv_heads, head_dim, device_status,
                                          reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_attention(const void *q, const int32_t *cu_seqlens_q, int32_t num_seqs, int64_t total_q,
                         const int32_t *seq_slot, const int32_t *context_lens, const int32_t *block_tables,
                         int32_t max_slots, int32_t max_blocks_per_slot, int32_t block_size,
                         const void *k_pool, const void *v_pool, int64_t num_blocks, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, float scale, const int32_t *work,
                         const pkv_work_info *info, void *out, void *workspace, uint64_t workspace_bytes,
                         uint32_t *device_status, pkv_stream_t stream) {
  return pkv::attention(q, cu_seqlens_q, num_seqs, total_q, seq_slot, context_lens, block_tables, max_slots,
                        max_blocks_per_slot, block_size, k_pool, v_pool, num_blocks, num_q_heads, num_kv_heads,
                        head_dim, scale, work, info, out, workspace, workspace_bytes, device_status, stream, false);
}

}  // extern "C"

pkv_status pkv::attention(const void *q, const int32_t *cu_seqlens_q, int32_t num_seqs, int64_t total_q,
                          const int32_t *seq_slot, const int32_t *context_lens, const int32_t *block_tables,
                          int32_t max_slots, int32_t max_blocks_per_slot, int32_t block_size, const void *k_pool,
                          const void *v_pool, int64_t num_blocks, int32_t num_q_heads, int32_t num_kv_heads,
                          int32_t head_dim, float scale, const int32_t *work, const pkv_work_info *info, void *out,
                          void *workspace, uint64_t workspace_bytes, uint32_t *device_status, pkv_stream_t stream,
                          bool out_on_host) {
  if (!info || num_seqs < 0 || total_q < 0 || max_slots <= 0 || max_blocks_per_slot <= 0 || num_blocks <= 0)
    return PKV_ERR_INVALID_ARG;
  if (!supported_shape(block_size, num_q_heads, num_kv_heads, head_dim)) return PKV_ERR_UNSUPPORTED;
  const int64_t rows = num_blocks * num_kv_heads * block_size;
  if (rows > INT32_MAX || total_q > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  const int64_t items = static_cast<int64_t>(info->num_decode_items) + info->num_prefill_items +
                        info->num_combine_items + info->num_scratch_items;
  if (info->num_decode_items < 0 || info->num_prefill_items < 0 || info->num_combine_items < 0 ||
      info->num_scratch_items < 0 || info->num_partials < 0 ||
      info->work_words != items * PKV_WORK_WORDS_PER_ITEM)
    return PKV_ERR_INVALID_ARG;
  if (items == 0 || total_q == 0) return PKV_OK;
  if (!q || !cu_seqlens_q || !seq_slot || !context_lens || !block_tables || !k_pool || !v_pool || !work || !out)
    return PKV_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16) ||
      !aligned(work, 16))
    return PKV_ERR_INVALID_ARG;
  const uint64_t acc_bytes = align256(uint64_t(info->num_partials) * num_q_heads * head_dim * 4);
  const uint64_t ml_bytes = align256(uint64_t(info->num_partials) * num_q_heads * 8);
  const uint64_t need = info->num_partials == 0 ? 0 : acc_bytes + ml_bytes + pkv::kCounterBytes;
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 256)))
    return PKV_ERR_WORKSPACE_TOO_SMALL;
  if ((info->num_combine_items > 0) != (info->num_partials > 0)) return PKV_ERR_INVALID_ARG;
  if (info->num_long_combine_items < 0 || info->num_long_combine_items > info->num_combine_items)
    return PKV_ERR_INVALID_ARG;
  // a decode-path segment's (row, q head) columns fit one 16-column tile
  if (info->decode_rows_max < 0 ||
      (info->num_decode_items > 0 && info->decode_rows_max * (num_q_heads / num_kv_heads) > 16))
    return PKV_ERR_INVALID_ARG;

  pkv::StepArgs a{};
  a.q = q;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.cu_seqlens_q = cu_seqlens_q;
  a.seq_slot = seq_slot;
  a.context_lens = context_lens;
  a.block_tables = block_tables;
  a.num_seqs = num_seqs;
  a.max_slots = max_slots;
  a.max_blocks_per_slot = max_blocks_per_slot;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.total_q = total_q;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.group = num_q_heads / num_kv_heads;
  a.head_dim = head_dim;
  a.decode_rows_max = info->decode_rows_max;
  const float s = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(head_dim));
  a.scale_log2 = s * 1.4426950408889634f;
  a.work = work;
  a.out = out;
  a.out_on_host = out_on_host ? 1 : 0;
  a.partial_acc = static_cast<float *>(workspace);
  a.partial_ml = need ? reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + acc_bytes) : nullptr;
  a.status = device_status;
  a.task_counter =
      need ? reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(workspace) + acc_bytes + ml_bytes) : nullptr;

  CUtensorMap tk, tv, tq, tks;
  if (!encode_pool(&tk, k_pool, rows, head_dim) || !encode_pool(&tv, v_pool, rows, head_dim))
    return PKV_ERR_CUDA;
  const int32_t rpt = pkv::prefill_rows_per_tile(a.group);
  if (info->num_prefill_items > 0 &&
      (!encode_q(&tq, q, total_q, num_q_heads, head_dim, a.group, rpt) ||
       (head_dim == 128 && !encode_pool_subtiles(&tks, k_pool, num_blocks * num_kv_heads, block_size))))
    return PKV_ERR_CUDA;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int32_t *dec = work;
  const int32_t *pre = dec + static_cast<int64_t>(info->num_decode_items) * PKV_WORK_WORDS_PER_ITEM;
  const int32_t *comb = pre + static_cast<int64_t>(info->num_prefill_items) * PKV_WORK_WORDS_PER_ITEM;
  // Both kinds of rows: the chunk kernel goes first on the caller's stream (its
  // CTAs take their SMs first), the decode and merge kernels run beside it on
  // the side stream from the same starting point, and the caller's stream
  // waits for them before anything it enqueues next.
  SideStream *side = (info->num_prefill_items > 0 && info->num_decode_items > 0) ? side_stream() : nullptr;
  std::unique_lock<std::mutex> lock;
  if (side) lock = std::unique_lock<std::mutex>(side->mu);
  // With decode segments of at most 8 (row, q head) columns, a CTA of each
  // kernel fits on every SM, so both kinds of rows share all SMs.
  const bool beside = side && head_dim == 128 && a.group * (a.decode_rows_max > 1 ? a.decode_rows_max : 1) <= 8;
  cudaError_t e = side ? cudaEventRecord(side->fork, st) : cudaSuccess;
  if (e == cudaSuccess)
    e = head_dim == 128 ? pkv::launch_prefill_pair(a, tq, tks, tv, rpt, info->num_prefill_items, pre, beside, st)
                        : pkv::launch_prefill(a, tq, rpt, info->num_prefill_items, pre, st);
  cudaStream_t dst = side ? side->stream : st;
  if (e == cudaSuccess && side) e = cudaStreamWaitEvent(side->stream, side->fork, 0);
  if (e == cudaSuccess) e = pkv::launch_decode(a, tk, tv, info->num_decode_items, dec, beside, dst);
  if (e == cudaSuccess) e = pkv::launch_merge(a, info->num_combine_items, info->num_long_combine_items, comb, dst);
  if (side) {
    // join even after a failed launch, so the caller's stream never runs ahead of queued work
    const cudaError_t j = cudaEventRecord(side->join, side->stream);
    const cudaError_t w = j == cudaSuccess ? cudaStreamWaitEvent(st, side->join, 0) : j;
    if (e == cudaSuccess) e = w;
  }
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" {

pkv_status pkv_copy_blocks(const int32_t *pairs, int64_t num_pairs, void *const *arrays,
                           const int64_t *block_bytes, int32_t num_arrays, int64_t num_blocks,
                           uint32_t *device_status, pkv_stream_t stream) {
  if (num_pairs < 0 || num_arrays < 1 || num_arrays > 4 || num_blocks <= 0 || !arrays || !block_bytes)
    return PKV_ERR_INVALID_ARG;
  if (num_pairs == 0) return PKV_OK;
  if (!pairs || !aligned(pairs, 8)) return PKV_ERR_INVALID_ARG;
  for (int32_t a = 0; a < num_arrays; ++a)
    if (!arrays[a] || !aligned(arrays[a], 16) || block_bytes[a] <= 0 || block_bytes[a] % 16 != 0)
      return PKV_ERR_INVALID_ARG;
  cudaError_t e = pkv::launch_copy_blocks(pairs, num_pairs, arrays, block_bytes, num_arrays, num_blocks,
                                          device_status, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// The block-scaled pools' entry points share these bodies; `bits` is 8, or 4
// (head_dim 128 only).
static pkv_status cache_write_quant(int32_t bits, const void *k_new, const void *v_new, const int64_t *slot_mapping,
                                    int64_t num_tokens, int8_t *k_codes, void *k_scales, int8_t *v_codes,
                                    void *v_scales, int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                                    int32_t head_dim, uint32_t *device_status, pkv_stream_t stream) {
  if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0) return PKV_ERR_INVALID_ARG;
  if ((head_dim != 64 && head_dim != 128) || (bits == 4 && head_dim != 128)) return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping || !k_codes || !v_codes || !k_scales || !v_scales)
    return PKV_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_codes, 16) || !aligned(v_codes, 16) ||
      !aligned(k_scales, 16) || !aligned(v_scales, 16) || !aligned(slot_mapping, 8))
    return PKV_ERR_INVALID_ARG;
  cudaError_t e = pkv::launch_cache_write_quant(k_new, v_new, slot_mapping, num_tokens, k_codes, k_scales, v_codes,
                                             v_scales, num_blocks, block_size, num_kv_heads, head_dim, bits,
                                             device_status, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_cache_write_q8(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                              int64_t num_tokens, int8_t *k_codes, void *k_scales, int8_t *v_codes, void *v_scales,
                              int64_t num_blocks, int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                              uint32_t *device_status, pkv_stream_t stream) {
  return cache_write_quant(8, k_new, v_new, slot_mapping, num_tokens, k_codes, k_scales, v_codes, v_scales,
                           num_blocks, block_size, num_kv_heads, head_dim, device_status, stream);
}

pkv_status pkv_cache_write_q4(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                              int64_t num_tokens, uint8_t *k_codes, void *k_scales, uint8_t *v_codes, void *v_scales,
                              int64_t num_blocks, int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                              uint32_t *device_status, pkv_stream_t stream) {
  return cache_write_quant(4, k_new, v_new, slot_mapping, num_tokens, reinterpret_cast<int8_t *>(k_codes), k_scales,
                           reinterpret_cast<int8_t *>(v_codes), v_scales, num_blocks, block_size, num_kv_heads,
                           head_dim, device_status, stream);
}

static pkv_status attention_quant(int32_t bits, const void *q, const int32_t *cu_seqlens_q, int32_t num_seqs,
                                  int64_t total_q, const int32_t *seq_slot, const int32_t *context_lens,
                                  const int32_t *block_tables, int32_t max_slots, int32_t max_blocks_per_slot,
                                  int32_t block_size, const int8_t *k_codes, const void *k_scales,
                                  const int8_t *v_codes, const void *v_scales, int64_t num_blocks,
                                  int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, float scale,
                                  const int32_t *work, const pkv_work_info *info, void *out, void *workspace,
                                  uint64_t workspace_bytes, uint32_t *device_status, pkv_stream_t stream) {
  if (!info || num_seqs < 0 || total_q < 0 || max_slots <= 0 || max_blocks_per_slot <= 0 || num_blocks <= 0)
    return PKV_ERR_INVALID_ARG;
  if (!supported_shape(block_size, num_q_heads, num_kv_heads, head_dim) || (bits == 4 && head_dim != 128))
    return PKV_ERR_UNSUPPORTED;
  const int64_t rows = num_blocks * num_kv_heads * block_size;
  if (rows > INT32_MAX || total_q > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  const int64_t items = static_cast<int64_t>(info->num_decode_items) + info->num_prefill_items +
                        info->num_combine_items + info->num_scratch_items;
  if (info->num_decode_items < 0 || info->num_prefill_items < 0 || info->num_combine_items < 0 ||
      info->num_scratch_items < 0 || info->num_partials < 0 || info->scratch_blocks < 0 ||
      info->work_words != items * PKV_WORK_WORDS_PER_ITEM ||
      (info->num_prefill_items > 0) != (info->num_scratch_items > 0))
    return PKV_ERR_INVALID_ARG;
  if (items == 0 || total_q == 0) return PKV_OK;
  if (!q || !cu_seqlens_q || !seq_slot || !context_lens || !block_tables || !k_codes || !v_codes || !k_scales ||
      !v_scales || !work || !out)
    return PKV_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_codes, 16) || !aligned(v_codes, 16) || !aligned(k_scales, 16) ||
      !aligned(v_scales, 16) || !aligned(out, 16) || !aligned(work, 16))
    return PKV_ERR_INVALID_ARG;
  const uint64_t acc_bytes = align256(uint64_t(info->num_partials) * num_q_heads * head_dim * 4);
  const uint64_t ml_bytes = align256(uint64_t(info->num_partials) * num_q_heads * 8);
  const uint64_t part_bytes = info->num_partials == 0 ? 0 : acc_bytes + ml_bytes + pkv::kCounterBytes;
  const uint64_t sb = static_cast<uint64_t>(info->scratch_blocks);
  const uint64_t scratch_pool = align256(sb * num_kv_heads * block_size * head_dim * 2);
  const uint64_t table_bytes = align256(uint64_t(max_slots) * max_blocks_per_slot * 4);
  const uint64_t need = part_bytes + (sb ? 2 * scratch_pool + table_bytes : 0);
  if (need != info->workspace_bytes_q8) return PKV_ERR_INVALID_ARG;  // info from another shape
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 256)))
    return PKV_ERR_WORKSPACE_TOO_SMALL;
  if ((info->num_combine_items > 0) != (info->num_partials > 0)) return PKV_ERR_INVALID_ARG;
  if (info->num_long_combine_items < 0 || info->num_long_combine_items > info->num_combine_items)
    return PKV_ERR_INVALID_ARG;
  if (info->decode_rows_max < 0 ||
      (info->num_decode_items > 0 && info->decode_rows_max * (num_q_heads / num_kv_heads) > 16))
    return PKV_ERR_INVALID_ARG;
  if (sb && sb * num_kv_heads * block_size > INT32_MAX) return PKV_ERR_UNSUPPORTED;

  pkv::StepArgs a{};
  a.q = q;
  a.k_pool = k_codes;
  a.v_pool = v_codes;
  a.cu_seqlens_q = cu_seqlens_q;
  a.seq_slot = seq_slot;
  a.context_lens = context_lens;
  a.block_tables = block_tables;
  a.num_seqs = num_seqs;
  a.max_slots = max_slots;
  a.max_blocks_per_slot = max_blocks_per_slot;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.total_q = total_q;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.group = num_q_heads / num_kv_heads;
  a.head_dim = head_dim;
  a.decode_rows_max = info->decode_rows_max;
  const float s = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(head_dim));
  a.scale_log2 = s * 1.4426950408889634f;
  a.work = work;
  a.out = out;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  a.partial_acc = info->num_partials ? reinterpret_cast<float *>(ws) : nullptr;
  a.partial_ml = info->num_partials ? reinterpret_cast<float *>(ws + acc_bytes) : nullptr;
  a.status = device_status;
  a.task_counter = info->num_partials ? reinterpret_cast<uint32_t *>(ws + acc_bytes + ml_bytes) : nullptr;

  // The chunk kernel reads a bf16 scratch pool: the chunk segments' histories,
  // widened block by block, with a scratch block table in the same shape.
  pkv::StepArgs c = a;
  c.kv_from_previous = 1;  // the widening pass right before the chunk kernel fills its K/V
  void *scratch_k = nullptr, *scratch_v = nullptr;
  int32_t *scratch_table = nullptr;
  if (sb) {
    scratch_k = ws + part_bytes;
    scratch_v = ws + part_bytes + scratch_pool;
    scratch_table = reinterpret_cast<int32_t *>(ws + part_bytes + 2 * scratch_pool);
    c.k_pool = scratch_k;
    c.v_pool = scratch_v;
    c.block_tables = scratch_table;
    c.num_blocks = static_cast<int64_t>(sb);
  }

  CUtensorMap tkc, tvc, tq, tk, tv;
  if (info->num_decode_items > 0 &&
      (!encode_codes(&tkc, k_codes, rows, head_dim, bits) || !encode_codes(&tvc, v_codes, rows, head_dim, bits)))
    return PKV_ERR_CUDA;
  const int32_t rpt = pkv::prefill_rows_per_tile(a.group);
  if (info->num_prefill_items > 0) {
    const int64_t srows = static_cast<int64_t>(sb) * num_kv_heads * block_size;
    if (!encode_q(&tq, q, total_q, num_q_heads, head_dim, a.group, rpt) ||
        !encode_pool(&tv, scratch_v, srows, head_dim) ||
        (head_dim == 128 ? !encode_pool_subtiles(&tk, scratch_k, static_cast<int64_t>(sb) * num_kv_heads, block_size)
                         : !encode_pool(&tk, scratch_k, srows, head_dim)))
      return PKV_ERR_CUDA;
  }

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int32_t *dec = work;
  const int32_t *pre = dec + static_cast<int64_t>(info->num_decode_items) * PKV_WORK_WORDS_PER_ITEM;
  const int32_t *comb = pre + static_cast<int64_t>(info->num_prefill_items) * PKV_WORK_WORDS_PER_ITEM;
  const int32_t *scr = comb + static_cast<int64_t>(info->num_combine_items) * PKV_WORK_WORDS_PER_ITEM;
  SideStream *side = (info->num_prefill_items > 0 && info->num_decode_items > 0) ? side_stream() : nullptr;
  std::unique_lock<std::mutex> lock;
  if (side) lock = std::unique_lock<std::mutex>(side->mu);
  cudaError_t e = side ? cudaEventRecord(side->fork, st) : cudaSuccess;
  if (e == cudaSuccess && info->num_prefill_items > 0) {
    e = pkv::launch_widen_quant(a, k_codes, k_scales, v_codes, v_scales, scratch_k, scratch_v, scratch_table,
                             static_cast<int64_t>(sb), info->num_scratch_items, scr, bits, st);
    if (e == cudaSuccess)
      e = head_dim == 128 ? pkv::launch_prefill_pair(c, tq, tk, tv, rpt, info->num_prefill_items, pre, false, st)
                          : pkv::launch_prefill(c, tq, rpt, info->num_prefill_items, pre, st);
  }
  cudaStream_t dst = side ? side->stream : st;
  if (e == cudaSuccess && side) e = cudaStreamWaitEvent(side->stream, side->fork, 0);
  if (e == cudaSuccess)
    e = pkv::launch_decode_quant(a, tkc, tvc, k_scales, v_scales, info->num_decode_items, dec, bits, dst);
  if (e == cudaSuccess) e = pkv::launch_merge(a, info->num_combine_items, info->num_long_combine_items, comb, dst);
  if (side) {
    const cudaError_t j = cudaEventRecord(side->join, side->stream);
    const cudaError_t w = j == cudaSuccess ? cudaStreamWaitEvent(st, side->join, 0) : j;
    if (e == cudaSuccess) e = w;
  }
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_attention_q8(const void *q, const int32_t *cu_seqlens_q, int32_t num_seqs, int64_t total_q,
                            const int32_t *seq_slot, const int32_t *context_lens, const int32_t *block_tables,
                            int32_t max_slots, int32_t max_blocks_per_slot, int32_t block_size,
                            const int8_t *k_codes, const void *k_scales, const int8_t *v_codes, const void *v_scales,
                            int64_t num_blocks, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                            float scale, const int32_t *work, const pkv_work_info *info, void *out, void *workspace,
                            uint64_t workspace_bytes, uint32_t *device_status, pkv_stream_t stream) {
  return attention_quant(8, q, cu_seqlens_q, num_seqs, total_q, seq_slot, context_lens, block_tables, max_slots,
                         max_blocks_per_slot, block_size, k_codes, k_scales, v_codes, v_scales, num_blocks,
                         num_q_heads, num_kv_heads, head_dim, scale, work, info, out, workspace, workspace_bytes,
                         device_status, stream);
}

pkv_status pkv_attention_q4(const void *q, const int32_t *cu_seqlens_q, int32_t num_seqs, int64_t total_q,
                            const int32_t *seq_slot, const int32_t *context_lens, const int32_t *block_tables,
                            int32_t max_slots, int32_t max_blocks_per_slot, int32_t block_size,
                            const uint8_t *k_codes, const void *k_scales, const uint8_t *v_codes,
                            const void *v_scales, int64_t num_blocks, int32_t num_q_heads, int32_t num_kv_heads,
                            int32_t head_dim, float scale, const int32_t *work, const pkv_work_info *info, void *out,
                            void *workspace, uint64_t workspace_bytes, uint32_t *device_status, pkv_stream_t stream) {
  return attention_quant(4, q, cu_seqlens_q, num_seqs, total_q, seq_slot, context_lens, block_tables, max_slots,
                         max_blocks_per_slot, block_size, reinterpret_cast<const int8_t *>(k_codes), k_scales,
                         reinterpret_cast<const int8_t *>(v_codes), v_scales, num_blocks, num_q_heads, num_kv_heads,
                         head_dim, scale, work, info, out, workspace, workspace_bytes, device_status, stream);
}

pkv_status pkv_check_device_status(uint32_t *device_status, pkv_stream_t stream, uint32_t *bits_out) {
  if (!device_status) return PKV_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t bits = 0;
  if (cudaMemcpyAsync(&bits, device_status, sizeof(bits), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemsetAsync(device_status, 0, sizeof(bits), st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (bits_out) *bits_out = bits;
  if (bits == 0) return PKV_OK;
  return (bits & PKV_DEV_TIMEOUT) ? PKV_ERR_DEVICE_TIMEOUT : PKV_ERR_DEVICE_INDEX;
}

}  // extern "C"
