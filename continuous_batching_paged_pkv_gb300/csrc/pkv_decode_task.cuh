// Work-item bookkeeping shared by the split-KV decode kernels (bf16 and
// 8-bit pools): one task is (decode segment, key span of PKV_SPLIT_KEYS keys,
// kv head). A warp expands a task (issues the loads of its metadata and block
// IDs), then finalises it (checks the metadata against the work item and
// derives the key range and the pool row of each 16-key sub-tile).
#pragma once

#include <cuda_runtime.h>

#include "pkv_internal.h"

namespace pkv {
namespace {

// One task's metadata. Scalars are uniform across the warp; `bid` is per lane:
// the physical block of the task's sub-tile number `lane`.
struct Task {
  int t;  // task index, -1 if none
  int seg, slot, span, pbase, g;
  int row0, row1, L, sslot;
  int nrows;  // rows of the segment (1, or a short run of causal rows)
  int key0, key1, units;
  int bid;  // per lane: block of sub-tile `lane`
  int row;  // per lane: tensor-map row of sub-tile `lane`, -1 if its block ID is outside the pool
  bool raw_ok, finalized, ok;
  bool reads_new;  // the span reaches this step's rows (written by the kernel before in the stream)
};

__device__ __forceinline__ int4 load_item(const int32_t *items, int t, int hkv) {
  return __ldg(reinterpret_cast<const int4 *>(items) + t / hkv);
}

// Issue every load the task needs; nothing here waits for a result.
__device__ __forceinline__ void expand(Task &T, int t, int4 raw, const StepArgs &a, int lane) {
  T.t = t;
  T.finalized = false;
  T.ok = false;
  T.reads_new = true;
  T.units = 0;
  T.bid = 0;
  T.row = -1;
  if (t < 0) return;
  T.seg = raw.x;
  T.slot = raw.y;
  T.span = raw.z;
  T.pbase = raw.w;
  T.g = t % a.num_kv_heads;
  T.key0 = T.span * PKV_SPLIT_KEYS;
  T.raw_ok = T.seg >= 0 && T.seg < a.num_seqs && T.slot >= 0 && T.slot < a.max_slots && T.span >= 0;
  if (!T.raw_ok) return;
  T.row0 = __ldg(a.cu_seqlens_q + T.seg);
  T.row1 = __ldg(a.cu_seqlens_q + T.seg + 1);
  T.L = __ldg(a.context_lens + T.slot);
  T.sslot = __ldg(a.seq_slot + T.seg);
  const int64_t key = static_cast<int64_t>(T.key0) + lane * kSubKeys;
  if (lane * kSubKeys < PKV_SPLIT_KEYS && key < static_cast<int64_t>(a.max_blocks_per_slot) * a.block_size)
    T.bid = __ldg(a.block_tables + static_cast<int64_t>(T.slot) * a.max_blocks_per_slot + key / a.block_size);
}

// Check the metadata against the work item and derive the key range.
__device__ __forceinline__ void finalize(Task &T, const StepArgs &a, int lane, int max_cols, int max_rows) {
  if (T.finalized) return;
  T.finalized = true;
  if (T.t < 0) return;
  T.nrows = T.row1 - T.row0;
  T.ok = T.raw_ok && T.sslot == T.slot && T.nrows >= 1 && T.nrows <= max_rows && T.nrows * a.group <= max_cols && T.nrows <= T.L &&
         T.L >= 1 &&
         static_cast<int64_t>(T.L) <= static_cast<int64_t>(a.max_blocks_per_slot) * a.block_size &&
         T.key0 < T.L && T.row0 >= 0 && static_cast<int64_t>(T.row0) + T.nrows <= a.total_q;
  if (!T.ok) {
    if (lane == 0 && a.status) atomicOr(a.status, PKV_DEV_BAD_SEGMENT);
    return;
  }
  T.key1 = min(T.L, T.key0 + PKV_SPLIT_KEYS);
  T.units = (T.key1 - T.key0 + kSubKeys - 1) / kSubKeys;
  T.reads_new = T.key1 > T.L - T.nrows;
  const bool in_pool = T.bid >= 0 && T.bid < a.num_blocks;
  T.row = in_pool ? (T.bid * a.num_kv_heads + T.g) * a.block_size + (T.key0 + lane * kSubKeys) % a.block_size : -1;
  if (lane < T.units && !in_pool && a.status) atomicOr(a.status, PKV_DEV_BAD_BLOCK);
}

}  // namespace
}  // namespace pkv
