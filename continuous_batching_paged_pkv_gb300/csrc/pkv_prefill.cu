// Prompt-chunk attention on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Lucebox, "Continuous batching: Qwen3.8-27B at 301 tok/s across five
// clients, up to 1.97x llama.cpp", §Chunked prefill is a slot phase (a chunk
// of a prompt appends to its slot and attends the slot's whole history) and
// §Packing unequal prompt chunks together (per-query causal positions let
// prompt rows share the call with decode rows). Tutorial 15, "Continuous
// Batching and Scheduling", §9 Summary: prefill is large matrix products.
//
// One CTA per (chunk tile, kv head). The tile's M = 128 rows are P query
// positions x G grouped q heads (row m = position m/G, head m%G), so every
// K/V tile is shared by the whole GQA group. Keys come in tiles of 128
// (8 TMA boxes of 16 rows per half of head_dim, straight from the pool
// rows the block table names, 128-byte swizzle).
//
//   warp 0 (one lane)  TMA producer: Q once, then K/V tiles into a 2-stage ring
//   warp 1 (one lane)  MMA issuer:   S_j = Q K_j^T   (SS form, fp32 in TMEM)
//                                     O  += P_j V_j   (A = P from TMEM, B = V smem)
//   warps 2-5          softmax: thread = TMEM lane = row; reads S_j, masks the
//                      causal/ragged edge, keeps (max, sum), writes P_j as bf16
//                      over S_j in TMEM; rescales O only when the running max
//                      grew by more than 2^8; final normalisation and store.
//
// TMEM columns: [0,128) S/P buffer 0, [128,256) S/P buffer 1, [256,256+D) O.
// Every mbarrier wait is bounded; on expiry the CTA records PKV_DEV_TIMEOUT,
// drains its MMAs and frees TMEM before returning.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kKeysPerTile = 128;
constexpr int kSubPerTile = kKeysPerTile / kSubKeys;  // 8
constexpr int kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > 256x

template <int D>
struct PrefillLayout {
  static constexpr int kHalves = D / 64;
  static constexpr int kQHalf = 128 * 128;              // 128 rows x 128 B
  static constexpr int kQBytes = kHalves * kQHalf;
  static constexpr int kKVHalf = kKeysPerTile * 128;    // 128 keys x 128 B
  static constexpr int kKVBytes = kHalves * kKVHalf;    // one K (or V) tile
  static constexpr int kStageBytes = 2 * kKVBytes;
  static constexpr int kBarOffset = kQBytes + 2 * kStageBytes;
  static constexpr int kSmem = kBarOffset + 256 + 1024;  // barriers/flags + alignment slack
};

enum Bar : int {
  kQFull = 0,
  kKVFull = 1,    // +stage
  kKVEmpty = 3,   // +stage
  kSFull = 5,     // +buffer
  kPReady = 7,    // +buffer
  kPVDone = 9,    // +buffer
  kDrain = 11,
  kNumBars = 12
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > 1000000000ull) {
        *abort = 1;
        return false;
      }
    }
  }
}

template <int D>
__global__ void __launch_bounds__(192, 1) prefill_kernel(const __grid_constant__ CUtensorMap tmap_q,
                                                         const __grid_constant__ CUtensorMap tmap_k,
                                                         const __grid_constant__ CUtensorMap tmap_v,
                                                         const StepArgs a,
                                                         const int32_t *__restrict__ items,
                                                         int rows_per_tile) {
  using Lay = PrefillLayout<D>;
  constexpr int H = Lay::kHalves;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint8_t *sQ = smem;
  uint8_t *sKV = smem + Lay::kQBytes;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + Lay::kBarOffset);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + kNumBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.y;
  launch_dependents();
  grid_dependency_wait();  // every input may come from the previous kernel in the stream
  const int4 it = reinterpret_cast<const int4 *>(items)[blockIdx.x];
  const int seg = it.x, slot = it.y, tile = it.z;
  const int G = a.group, P = rows_per_tile;

  bool bad = seg < 0 || seg >= a.num_seqs || slot < 0 || slot >= a.max_slots || tile < 0;
  int row0 = 0, n = 0, L = 0;
  if (!bad) {
    row0 = a.cu_seqlens_q[seg];
    n = a.cu_seqlens_q[seg + 1] - row0;
    L = a.context_lens[slot];
    bad = a.seq_slot[seg] != slot || n < 2 || n > L ||
          static_cast<int64_t>(L) > static_cast<int64_t>(a.max_blocks_per_slot) * a.block_size ||
          tile * P >= n || row0 < 0 || static_cast<int64_t>(row0) + n > a.total_q;
  }
  if (bad) {
    if (threadIdx.x == 0 && a.status) atomicOr(a.status, PKV_DEV_BAD_SEGMENT);
    return;
  }
  const int pos0 = tile * P;                 // first query row of the tile within the segment
  const int rows = min(P, n - pos0);         // query positions present in this tile
  const int kv_end = L - n + pos0 + rows;    // keys [0, kv_end) are visible to some row
  const int ntiles = (kv_end + kKeysPerTile - 1) / kKeysPerTile;
  const int32_t *bt_row = a.block_tables + static_cast<int64_t>(slot) * a.max_blocks_per_slot;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(bar + i, (i == kPReady || i == kPReady + 1) ? 128 : 1);
    fence_barrier_init();
    *abort_flag = 0;
  }
  // Rows of the Q tile beyond G*P whole groups stay zero.
  {
    const int qrows = G * P;
    const int chunks = (128 - qrows) * 8;  // 16-byte chunks per half
    for (int i = threadIdx.x; i < chunks * H; i += blockDim.x) {
      const int h = i / chunks, rem = i % chunks;
      *reinterpret_cast<uint4 *>(sQ + h * Lay::kQHalf + (qrows + rem / 8) * 128 + (rem % 8) * 16) =
          make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tmap_q);
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
      mbar_arrive_expect_tx(bar + kQFull, H * G * P * 128);
      for (int h = 0; h < H; ++h)
        tma_load_3d(sQ + h * Lay::kQHalf, &tmap_q, h * 64, g * G, row0 + pos0, bar + kQFull);
      for (int j = 0; j < ntiles; ++j) {
        const int s = j & 1;
        if (j >= 2 && !wait_or_abort(bar + kKVEmpty + s, ((j - 2) >> 1) & 1, abort_flag)) break;
        const int kt0 = j * kKeysPerTile;
        const int units = min(kSubPerTile, (kv_end - kt0 + kSubKeys - 1) / kSubKeys);
        uint8_t *sK = sKV + s * Lay::kStageBytes;
        uint8_t *sV = sK + Lay::kKVBytes;
        mbar_arrive_expect_tx(bar + kKVFull + s, units * H * 2 * kSubKeys * 128);
        for (int u = 0; u < units; ++u) {
          const int key = kt0 + u * kSubKeys;
          int blk = __ldg(bt_row + key / a.block_size);
          if (blk < 0 || blk >= a.num_blocks) {
            if (a.status) atomicOr(a.status, PKV_DEV_BAD_BLOCK);
            blk = 0;  // load something in range; the flag already marks the output invalid
          }
          const int row = (blk * a.num_kv_heads + g) * a.block_size + key % a.block_size;
          for (int h = 0; h < H; ++h) {
            tma_load_2d(sK + h * Lay::kKVHalf + u * kSubKeys * 128, &tmap_k, h * 64, row, bar + kKVFull + s);
            tma_load_2d(sV + h * Lay::kKVHalf + u * kSubKeys * 128, &tmap_v, h * 64, row, bar + kKVFull + s);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, kKeysPerTile, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, 0, 1);
      const uint32_t q_base = smem_addr(sQ);
      auto issue_pv = [&](int jj) -> bool {
        const int sp = jj & 1;
        if (!wait_or_abort(bar + kPReady + sp, (jj >> 1) & 1, abort_flag)) return false;
        tc_fence_after();
        const int valid = min(kKeysPerTile, kv_end - jj * kKeysPerTile);
        const int ksteps = (valid + kSubKeys - 1) / kSubKeys;
        const uint32_t v_base = smem_addr(sKV + sp * Lay::kStageBytes + Lay::kKVBytes);
        for (int ks = 0; ks < ksteps; ++ks) {
          const uint64_t bdesc = smem_desc_sw128(v_base + ks * kSubKeys * 128, Lay::kKVHalf, 1024);
          tc_mma_ts(tmem + 256, tmem + sp * 128 + ks * 8, bdesc, idesc_pv, (jj > 0 || ks > 0) ? 1u : 0u);
        }
        tc_commit(bar + kPVDone + sp);
        tc_commit(bar + kKVEmpty + sp);
        return true;
      };
      bool ok = wait_or_abort(bar + kQFull, 0, abort_flag);
      tc_fence_after();
      for (int j = 0; ok && j < ntiles; ++j) {
        const int s = j & 1;
        if (j >= 2 && !(ok = wait_or_abort(bar + kPVDone + s, ((j - 2) >> 1) & 1, abort_flag))) break;
        if (!(ok = wait_or_abort(bar + kKVFull + s, (j >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        const uint32_t k_base = smem_addr(sKV + s * Lay::kStageBytes);
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * Lay::kQHalf + (kk & 3) * 32;
          const uint32_t koff = (kk >> 2) * Lay::kKVHalf + (kk & 3) * 32;
          tc_mma_ss(tmem + s * 128, smem_desc_sw128(q_base + off, 16, 1024),
                    smem_desc_sw128(k_base + koff, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar + kSFull + s);
        if (j >= 1 && !(ok = issue_pv(j - 1))) break;
      }
      if (ok) issue_pv(ntiles - 1);
      tc_commit(bar + kDrain);
      if (!wait_or_abort(bar + kDrain, 0, abort_flag) && a.status) atomicOr(a.status, PKV_DEV_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int qw = warp & 3;
    const int mrow = qw * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(qw * 32) << 16;
    const int pos = mrow / G, hh = mrow % G;
    const bool row_valid = mrow < G * P && pos < rows;
    const int p_row = L - n + pos0 + pos;  // last visible key of this row (inclusive)
    const float sl2 = a.scale_log2;
    float m_used = -INFINITY, lsum = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int s = j & 1;
      if (!(ok = wait_or_abort(bar + kSFull + s, (j >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      uint32_t sv[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_base + s * 128 + c * 32, sv[c]);
      tmem_wait_ld();
      const int lim = min(p_row, L - 1) - j * kKeysPerTile;
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float x = (c * 32 + i) <= lim ? __uint_as_float(sv[c][i]) * sl2 : -INFINITY;
          sv[c][i] = __float_as_uint(x);
          mx = fmaxf(mx, x);
        }
      const float m_new = fmaxf(m_used, mx);
      const bool need = j > 0 && m_new > m_used + kRescaleThreshold;
      if (j == 0) m_used = m_new;
      if (__any_sync(0xffffffffu, need)) {
        // O must hold P_{j-1} V_{j-1} before it is rescaled.
        if (!(ok = wait_or_abort(bar + kPVDone + ((j - 1) & 1), ((j - 1) >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        const float corr = need ? exp2f(m_used - m_new) : 1.f;
        if (need) m_used = m_new;
        lsum *= corr;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(tmem + lane_base + 256 + c * 32, ov);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * corr);
          tmem_st32(tmem + lane_base + 256 + c * 32, ov);
        }
      }
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const __nv_bfloat16 p0 = __float2bfloat16_rn(exp2f(__uint_as_float(sv[c][2 * i]) - m_used));
          const __nv_bfloat16 p1 = __float2bfloat16_rn(exp2f(__uint_as_float(sv[c][2 * i + 1]) - m_used));
          rs += __bfloat162float(p0) + __bfloat162float(p1);
          pk[i] = static_cast<uint32_t>(__bfloat16_as_ushort(p0)) |
                  (static_cast<uint32_t>(__bfloat16_as_ushort(p1)) << 16);
        }
        tmem_st16(tmem + lane_base + s * 128 + c * 16, pk);
      }
      lsum += rs;
      if (j == ntiles - 1) {
        // Zero V rows past the last visible key inside the final 16-key step:
        // a partly filled block may hold stale or NaN rows there.
        const int valid = kv_end - j * kKeysPerTile;
        const int tail = (kSubKeys - valid % kSubKeys) % kSubKeys;
        if (tail) {
          if (!(ok = wait_or_abort(bar + kKVFull + s, (j >> 1) & 1, abort_flag))) break;
          uint8_t *sV = sKV + s * Lay::kStageBytes + Lay::kKVBytes;
          const int tid = threadIdx.x - 64;
          for (int i = tid; i < tail * 8 * H; i += 128) {
            const int h = i / (tail * 8), rem = i % (tail * 8);
            *reinterpret_cast<uint4 *>(sV + h * Lay::kKVHalf + (valid + rem / 8) * 128 + (rem % 8) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar + kPReady + s);
    }
    if (ok && wait_or_abort(bar + kPVDone + ((ntiles - 1) & 1), ((ntiles - 1) >> 1) & 1, abort_flag)) {
      tc_fence_after();
      const float inv = 1.f / lsum;
      __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(a.out) +
                            (static_cast<size_t>(row0 + pos0 + pos) * a.num_q_heads + g * G + hh) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(tmem + lane_base + 256 + c * 32, ov);
        tmem_wait_ld();
        if (row_valid) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv, __uint_as_float(ov[2 * i + 1]) * inv);
          uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0 && a.status) atomicOr(a.status, PKV_DEV_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_prefill_t(const StepArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                             const CUtensorMap &tv, int32_t rows_per_tile, int32_t num_items,
                             const int32_t *items, cudaStream_t stream) {
  constexpr int smem = PrefillLayout<D>::kSmem;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(static_cast<unsigned>(num_items), static_cast<unsigned>(a.num_kv_heads));
  return launch_pdl(prefill_kernel<D>, grid, dim3(192), smem, stream, tq, tk, tv, a, items, rows_per_tile);
}

}  // namespace

cudaError_t launch_prefill(const StepArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                           const CUtensorMap &tv, int32_t rows_per_tile, int32_t num_items,
                           const int32_t *items, cudaStream_t stream) {
  if (num_items <= 0) return cudaSuccess;
  if (a.head_dim == 128) return launch_prefill_t<128>(a, tq, tk, tv, rows_per_tile, num_items, items, stream);
  return launch_prefill_t<64>(a, tq, tk, tv, rows_per_tile, num_items, items, stream);
}

}  // namespace pkv
