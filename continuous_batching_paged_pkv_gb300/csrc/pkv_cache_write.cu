// Cache write: append each new row's key and value to its pool row.
//
// Lucebox, "Continuous batching: Qwen3.8-27B at 301 tok/s across five
// clients, up to 1.97x llama.cpp", §Chunked prefill is a slot phase: every
// selected chunk (and every decode row) appends directly to its slot's paged
// KV; §Paged KV and paged attention: the pool is fixed-size physical blocks.
//
// One thread moves one 16-byte vector (8 bf16). Consecutive threads cover
// consecutive vectors of one (token, kv head) row, so reads of k_new/v_new
// and writes into the pool are both fully coalesced 16-byte accesses; the
// kernel is a pure HBM copy with no arithmetic on the values.
#include <cuda_runtime.h>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

__global__ void __launch_bounds__(256) cache_write_kernel(
    const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
    const int64_t *__restrict__ slot_mapping, int64_t num_tokens, uint4 *__restrict__ k_pool,
    uint4 *__restrict__ v_pool, int64_t pool_rows, int32_t block_size, int32_t num_kv_heads,
    int32_t vec_per_row, uint32_t *__restrict__ status) {
  grid_dependency_wait();  // k_new / v_new / slot_mapping may come from the previous kernel
  // The attention call may start now: everything before this kernel has
  // finished, so it can read its step metadata and q at once and wait for
  // this kernel only before it reads the rows written here.
  launch_dependents();
  // Vector index over [2 (k, v)][num_tokens][num_kv_heads][vec_per_row].
  const int64_t per_tensor = num_tokens * num_kv_heads * vec_per_row;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       i < 2 * per_tensor; i += stride) {
    const bool is_v = i >= per_tensor;
    const int64_t j = is_v ? i - per_tensor : i;
    const int64_t c = j % vec_per_row;
    const int64_t th = j / vec_per_row;  // token * num_kv_heads + head
    const int64_t h = th % num_kv_heads;
    const int64_t t = th / num_kv_heads;
    const int64_t s = __ldg(slot_mapping + t);
    if (s < 0) continue;
    if (s >= pool_rows) {
      if (status && c == 0 && h == 0 && !is_v) atomicOr(status, PKV_DEV_BAD_SLOT_MAPPING);
      continue;
    }
    const int64_t block = s / block_size, row = s % block_size;
    const int64_t dst = ((block * num_kv_heads + h) * block_size + row) * vec_per_row + c;
    if (is_v)
      v_pool[dst] = __ldg(v_new + j);
    else
      k_pool[dst] = __ldg(k_new + j);
  }
}

// Copy-on-write: whole blocks, source -> destination, in up to four pool
// arrays at once (mlxcel manual, "Continuous batching", §Paged KV cache and
// prefix sharing: a shared block branches by copy when a sequence's contents
// diverge from it). A block is contiguous in every pool array ([block][...]),
// so one block is block_bytes[a] / 16 consecutive 16-byte vectors.
struct CopyArrays {
  uint4 *base[4];
  int64_t vecs[4];  // 16-byte vectors per block
  int32_t count;
};

__global__ void __launch_bounds__(256) copy_blocks_kernel(const int32_t *__restrict__ pairs, int64_t num_pairs,
                                                          const CopyArrays arrays, int64_t num_blocks,
                                                          uint32_t *__restrict__ status) {
  grid_dependency_wait();  // the pairs and the source blocks come from earlier work
  launch_dependents();
  for (int64_t pi = blockIdx.y; pi < num_pairs; pi += gridDim.y) {
    const int32_t src = __ldg(pairs + 2 * pi), dst = __ldg(pairs + 2 * pi + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks || src == dst) {
      if (status && threadIdx.x == 0 && blockIdx.x == 0) atomicOr(status, PKV_DEV_BAD_BLOCK);
      continue;
    }
    for (int a = 0; a < arrays.count; ++a) {
      const int64_t n = arrays.vecs[a];
      const uint4 *s = arrays.base[a] + src * n;
      uint4 *d = arrays.base[a] + dst * n;
      for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
           i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        d[i] = __ldg(s + i);
    }
  }
}

}  // namespace

cudaError_t launch_copy_blocks(const int32_t *pairs, int64_t num_pairs, void *const *arrays,
                               const int64_t *block_bytes, int32_t num_arrays, int64_t num_blocks, uint32_t *status,
                               cudaStream_t stream) {
  CopyArrays ca{};
  ca.count = num_arrays;
  int64_t most = 0;
  for (int a = 0; a < num_arrays; ++a) {
    ca.base[a] = static_cast<uint4 *>(arrays[a]);
    ca.vecs[a] = block_bytes[a] / 16;
    most = ca.vecs[a] > most ? ca.vecs[a] : most;
  }
  const int64_t x = (most + 255) / 256;
  const int64_t y = num_pairs < 4096 ? num_pairs : 4096;
  return launch_pdl(copy_blocks_kernel, dim3(static_cast<unsigned>(x > 0 ? x : 1), static_cast<unsigned>(y)),
                    dim3(256), 0, stream, pairs, num_pairs, ca, num_blocks, status);
}

cudaError_t launch_cache_write(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                               int64_t num_tokens, void *k_pool, void *v_pool, int64_t num_blocks,
                               int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                               uint32_t *status, cudaStream_t stream) {
  const int32_t vec_per_row = head_dim * 2 / 16;
  const int64_t vectors = 2 * num_tokens * num_kv_heads * vec_per_row;
  const int threads = 256;
  int64_t blocks = (vectors + threads - 1) / threads;
  if (blocks > 152 * 16) blocks = 152 * 16;  // grid-stride beyond 16 CTAs per SM
  return launch_pdl(cache_write_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream,
                    static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new), slot_mapping, num_tokens,
                    static_cast<uint4 *>(k_pool), static_cast<uint4 *>(v_pool), num_blocks * block_size, block_size,
                    num_kv_heads, vec_per_row, status);
}

}  // namespace pkv
