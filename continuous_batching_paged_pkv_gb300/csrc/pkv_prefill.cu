// Prompt-chunk attention on the 5th-generation tensor cores (tcgen05 + TMEM),
// one CTA per query tile; serves head_dim 64 (head_dim 128 runs on SM pairs).
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
// K/V tile is shared by the whole GQA group. Keys come in tiles of 128.
//
//   warps 0-1          producers: Q once by TMA; each 128-key K/V tile as 4096
//                      16-byte cp.async copies straight from the pool rows the
//                      block table names, written in the 128-byte-swizzled
//                      layout the tensor core reads (keys past the context are
//                      zero-filled); three stages. A TMA issue costs its thread
//                      hundreds of cycles and a 2 KiB box is the largest this
//                      pool layout allows, which caps TMA near 44 GB/s per SM;
//                      mostly L2-resident K/V needs more than that.
//   warp 2 (one lane)  MMA issuer:   S_j  = Q K_j^T   (SS form, fp32 in TMEM)
//                                     O   += P_j V_j   (A = P from TMEM, B = V smem)
//                                     l   += P_j 1     (A = P from TMEM, B = ones)
//   warps 3-6          softmax: thread = TMEM lane = row; reads S_j, masks the
//                      causal/ragged edge on the tiles that need it, writes
//                      P_j = 2^(s*scale*log2e - m) as bf16 over S_j in TMEM;
//                      rescales O and l only when the running max grew by more
//                      than 2^8; final normalisation and store.
//
// The row sums come from the tensor core: an extra N = 16 MMA of P against a
// tile of ones accumulates, next to O, exactly the bf16-rounded P the output
// uses, so the softmax threads keep no running sum.
//
// TMEM columns: [0,128) S/P buffer 0, [128,256) S/P buffer 1, [256,256+D) O,
// [256+D, 256+D+16) l (all 16 columns equal). Every mbarrier wait is bounded;
// on expiry the CTA records PKV_DEV_TIMEOUT, drains its MMAs and frees TMEM
// before returning.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kKeysPerTile = 128;
constexpr int kTmemCols = 512;
constexpr int kOCol = 256;                 // O accumulator; l follows at kOCol + D
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > 256x
constexpr uint32_t kFull = 0xffffffffu;
constexpr uint32_t kNegInfBits = 0xff800000u;
constexpr uint32_t kSleepNs = 20000;
constexpr int kStages = 3;            // K/V tiles in flight
constexpr int kProducerLanes = 64;    // warps 0-1
constexpr int kThreads = 224;         // 2 producer warps, 1 MMA warp, 4 softmax warps

template <int D>
struct PrefillLayout {
  static constexpr int kHalves = D / 64;
  static constexpr int kQHalf = 128 * 128;              // 128 rows x 128 B
  static constexpr int kQBytes = kHalves * kQHalf;
  static constexpr int kKVHalf = kKeysPerTile * 128;    // 128 keys x 128 B
  static constexpr int kKVBytes = kHalves * kKVHalf;    // one K (or V) tile
  static constexpr int kStageBytes = 2 * kKVBytes;
  static constexpr int kOnesOffset = kQBytes + kStages * kStageBytes;  // 1 KiB of bf16 ones
  static constexpr int kBarOffset = kOnesOffset + 1024;
  static constexpr int kSmem = kBarOffset + 256 + 1024;  // barriers/flags + alignment slack
};

enum Bar : int {
  kQFull = 0,
  kKVFull = 1,    // +stage (3)
  kKVEmpty = 4,   // +stage (3)
  kSFull = 7,     // +buffer (2)
  kPReady = 9,    // +buffer (2)
  kPVDone = 11,   // +buffer (2)
  kDrain = 13,
  kNumBars = 14
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Wait that also gives up as soon as another role has aborted. The thread may
// sleep in the hardware until the phase completes.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort) {
  if (mbar_try_wait_sleep(bar, parity, kSleepNs)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_sleep(bar, parity, kSleepNs)) return true;
    if ((i & 15u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > 1000000000ull) {
        *abort = 1;
        return false;
      }
    }
  }
}

// Same, for a whole warp: every lane agrees on the outcome (the TMEM loads and
// stores that follow are warp-collective).
__device__ __forceinline__ bool warp_wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort) {
  return __all_sync(kFull, wait_or_abort(bar, parity, abort));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ CUtensorMap tmap_q,
                                                              const StepArgs a,
                                                              const int32_t *__restrict__ items,
                                                              int rows_per_tile) {
  using Lay = PrefillLayout<D>;
  constexpr int H = Lay::kHalves;
  constexpr int kLCol = kOCol + D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint8_t *sQ = smem;
  uint8_t *sKV = smem + Lay::kQBytes;
  uint8_t *sOnes = smem + Lay::kOnesOffset;
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
    for (int i = 0; i < kNumBars; ++i) {
      const bool p_ready = i == kPReady || i == kPReady + 1;
      const bool kv_full = i >= kKVFull && i < kKVFull + kStages;
      mbar_init(bar + i, p_ready ? 128 : (kv_full ? kProducerLanes : 1));
    }
    fence_barrier_init();
    *abort_flag = 0;
  }
  // Rows of the Q tile beyond G*P whole groups stay zero; the ones tile for the row sums.
  {
    const int qrows = G * P;
    const int chunks = (128 - qrows) * 8;  // 16-byte chunks per half
    for (int i = threadIdx.x; i < chunks * H; i += blockDim.x) {
      const int h = i / chunks, rem = i % chunks;
      *reinterpret_cast<uint4 *>(sQ + h * Lay::kQHalf + (qrows + rem / 8) * 128 + (rem % 8) * 16) =
          make_uint4(0, 0, 0, 0);
    }
    const uint32_t one2 = 0x3F803F80u;  // two bf16 1.0
    for (int i = threadIdx.x; i < 1024 / 16; i += blockDim.x)
      *reinterpret_cast<uint4 *>(sOnes + i * 16) = make_uint4(one2, one2, one2, one2);
    fence_proxy_async_smem();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 2) {
    // ------------------------------------------------------------ producers
    // Producer lane p copies, for k = 0..63, the 16-byte chunk p % 8 of row
    // (k % 2) * 8 + p / 8 of sub-tile (k / 2) % 8, half (k / 16) % 2, tensor
    // k / 32 (K then V): consecutive lanes read consecutive 16 bytes of a row.
    const int p = threadIdx.x;  // 0..63
    const uint8_t *kp = static_cast<const uint8_t *>(a.k_pool);
    const uint8_t *vp = static_cast<const uint8_t *>(a.v_pool);
    const int64_t row_bytes = static_cast<int64_t>(D) * 2;
    // Pool rows of the 16-key sub-tiles, four tiles per warp-wide load: lane l
    // covers sub-tile l % 8 of tile t0 + l / 8. The block IDs of the next group
    // are loaded raw one group ahead and turned into rows (checked against the
    // pool: -1 when outside it, the status word reports it) only when that
    // group comes into use, so no block-table latency is ever waited on.
    auto group_ids = [&](int t0) -> int {
      const int key = (t0 + (lane >> 3)) * kKeysPerTile + (lane & 7) * kSubKeys;
      return key < kv_end ? __ldg(bt_row + key / a.block_size) : 0;
    };
    auto group_rows = [&](int t0, int blk) -> int {
      const int key = (t0 + (lane >> 3)) * kKeysPerTile + (lane & 7) * kSubKeys;
      if (key >= kv_end) return 0;
      if (blk < 0 || blk >= a.num_blocks) {
        if (a.status && warp == 0) atomicOr(a.status, PKV_DEV_BAD_BLOCK);
        return -1;
      }
      return (blk * a.num_kv_heads + g) * a.block_size + key % a.block_size;
    };
    int rows_cur = group_rows(0, group_ids(0)), ids_next = group_ids(4);
    if (threadIdx.x == 0) {
      prefetch_tensormap(&tmap_q);
      mbar_arrive_expect_tx(bar + kQFull, H * G * P * 128);
      for (int h = 0; h < H; ++h)
        tma_load_3d(sQ + h * Lay::kQHalf, &tmap_q, h * 64, g * G, row0 + pos0, bar + kQFull);
    }
    const int c = p & 7;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int s = j % kStages;
      if (j >= kStages && !(ok = warp_wait_or_abort(bar + kKVEmpty + s, ((j - kStages) / kStages) & 1, abort_flag)))
        break;
      if (j > 0 && (j & 3) == 0) {
        rows_cur = group_rows(j, ids_next);
        ids_next = group_ids(j + 4);
      }
      const int kt0 = j * kKeysPerTile;
      const uint32_t sK = smem_addr(sKV + s * Lay::kStageBytes);
      const uint32_t sV = sK + Lay::kKVBytes;
#pragma unroll 4
      for (int k = 0; k < 64; ++k) {
        const int t = k >> 5, h = (k >> 4) & 1, u = (k >> 1) & 7;
        const int r = ((k & 1) << 3) + (p >> 3);
        const int urow = __shfl_sync(kFull, rows_cur, (j & 3) * 8 + u);
        if (h < H) {
          const bool valid = kt0 + u * kSubKeys + r < kv_end && urow >= 0;
          const int64_t off = (static_cast<int64_t>(valid ? urow : 0) + (valid ? r : 0)) * row_bytes + h * 128 + c * 16;
          const uint32_t dst = (t ? sV : sK) + h * Lay::kKVHalf + (u * kSubKeys + r) * 128 + ((c ^ (r & 7)) << 4);
          cp_async_16_zfill(dst, (t ? vp : kp) + off, valid);
        }
      }
      cp_async_commit();
      if (j >= 1) {
        // Tile j-1 has landed: make it visible to the tensor core and publish it.
        cp_async_wait<1>();
        fence_proxy_async_smem();
        mbar_arrive(bar + kKVFull + (j - 1) % kStages);
      }
    }
    cp_async_wait<0>();  // also on abort: no copy may still target shared memory at exit
    if (ok) {
      fence_proxy_async_smem();
      mbar_arrive(bar + kKVFull + (ntiles - 1) % kStages);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, kKeysPerTile, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, 0, 1);
      constexpr uint32_t idesc_l = idesc_bf16_f32(128, 16, 0, 0);
      const uint32_t q_base = smem_addr(sQ);
      const uint64_t ones_desc = smem_desc_noswz(smem_addr(sOnes), 128, 256);
      auto issue_pv = [&](int jj) -> bool {
        const int sp = jj & 1;
        if (!wait_or_abort(bar + kPReady + sp, (jj >> 1) & 1, abort_flag)) return false;
        tc_fence_after();
        const int valid = min(kKeysPerTile, kv_end - jj * kKeysPerTile);
        const int ksteps = (valid + kSubKeys - 1) / kSubKeys;
        const uint32_t v_base = smem_addr(sKV + (jj % kStages) * Lay::kStageBytes + Lay::kKVBytes);
        for (int ks = 0; ks < ksteps; ++ks) {
          const uint64_t bdesc = smem_desc_sw128(v_base + ks * kSubKeys * 128, Lay::kKVHalf, 1024);
          const uint32_t acc = (jj > 0 || ks > 0) ? 1u : 0u;
          tc_mma_ts(tmem + kOCol, tmem + sp * 128 + ks * 8, bdesc, idesc_pv, acc);
          tc_mma_ts(tmem + kLCol, tmem + sp * 128 + ks * 8, ones_desc, idesc_l, acc);
        }
        tc_commit(bar + kPVDone + sp);
        tc_commit(bar + kKVEmpty + jj % kStages);
        return true;
      };
      bool ok = wait_or_abort(bar + kQFull, 0, abort_flag);
      tc_fence_after();
      for (int j = 0; ok && j < ntiles; ++j) {
        const int s = j & 1;
        if (j >= 2 && !(ok = wait_or_abort(bar + kPVDone + s, ((j - 2) >> 1) & 1, abort_flag))) break;
        if (!(ok = wait_or_abort(bar + kKVFull + j % kStages, (j / kStages) & 1, abort_flag))) break;
        tc_fence_after();
        const uint32_t k_base = smem_addr(sKV + (j % kStages) * Lay::kStageBytes);
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
    float m_used = -INFINITY;  // log2 units
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int s = j & 1;
      if (!(ok = warp_wait_or_abort(bar + kSFull + s, (j >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      uint32_t sv[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_base + s * 128 + c * 32, sv[c]);
      tmem_wait_ld();
      // Causal / ragged edge: only tiles that reach past some row's last key need a mask.
      const int lim = min(p_row, kv_end - 1) - j * kKeysPerTile;
      if (!__all_sync(kFull, lim >= kKeysPerTile - 1)) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (c * 32 + i > lim) sv[c][i] = kNegInfBits;
      }
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], __uint_as_float(sv[c][i]));
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * sl2;
      const float m_new = fmaxf(m_used, mx);
      const bool need = j > 0 && m_new > m_used + kRescaleThreshold;
      if (j == 0) m_used = m_new;
      if (__any_sync(kFull, need)) {
        // O and l must hold tile j-1's products before they are rescaled.
        if (!(ok = warp_wait_or_abort(bar + kPVDone + ((j - 1) & 1), ((j - 1) >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        const float corr = need ? ex2_approx(m_used - m_new) : 1.f;
        if (need) m_used = m_new;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(tmem + lane_base + kOCol + c * 32, ov);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * corr);
          tmem_st32(tmem + lane_base + kOCol + c * 32, ov);
        }
        uint32_t lv[16];
        tmem_ld16(tmem + lane_base + kLCol, lv);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) lv[i] = __float_as_uint(__uint_as_float(lv[i]) * corr);
        tmem_st16(tmem + lane_base + kLCol, lv);
      }
      const float nm = -m_used;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(ex2_approx(fmaf(__uint_as_float(sv[c][2 * i]), sl2, nm)),
                              ex2_approx(fmaf(__uint_as_float(sv[c][2 * i + 1]), sl2, nm)));
        tmem_st16(tmem + lane_base + s * 128 + c * 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar + kPReady + s);
    }
    if (ok && warp_wait_or_abort(bar + kPVDone + ((ntiles - 1) & 1), ((ntiles - 1) >> 1) & 1, abort_flag)) {
      tc_fence_after();
      uint32_t lv[16];
      tmem_ld16(tmem + lane_base + kLCol, lv);
      tmem_wait_ld();
      const float inv = 1.f / __uint_as_float(lv[0]);
      __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(a.out) +
                            (static_cast<size_t>(row0 + pos0 + pos) * a.num_q_heads + g * G + hh) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(tmem + lane_base + kOCol + c * 32, ov);
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
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_prefill_t(const StepArgs &a, const CUtensorMap &tq, int32_t rows_per_tile, int32_t num_items,
                             const int32_t *items, cudaStream_t stream) {
  constexpr int smem = PrefillLayout<D>::kSmem;
  static std::atomic<uint64_t> configured{0};  // one bit per device
  if (const cudaError_t e = allow_smem_once(prefill_kernel<D>, smem, configured); e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(num_items), static_cast<unsigned>(a.num_kv_heads));
  return launch_pdl(prefill_kernel<D>, grid, dim3(kThreads), smem, stream, tq, a, items, rows_per_tile);
}

}  // namespace

cudaError_t launch_prefill(const StepArgs &a, const CUtensorMap &tq, int32_t rows_per_tile, int32_t num_items,
                           const int32_t *items, cudaStream_t stream) {
  if (num_items <= 0) return cudaSuccess;
  if (a.head_dim != 64) return cudaErrorInvalidValue;  // head_dim 128 runs on SM pairs
  return launch_prefill_t<64>(a, tq, rows_per_tile, num_items, items, stream);
}

}  // namespace pkv
