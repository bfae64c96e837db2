// Prompt-chunk attention for head_dim 128 on SM pairs (tcgen05 cta_group::2).
//
// Lucebox, "Continuous batching: Qwen3.8-27B at 301 tok/s across five
// clients, up to 1.97x llama.cpp", §Chunked prefill is a slot phase (a chunk
// of a prompt appends to its slot and attends the slot's whole history) and
// §Packing unequal prompt chunks together (per-query causal positions let
// prompt rows share the call with decode rows). Tutorial 15, "Continuous
// Batching and Scheduling", §9 Summary: prefill is large matrix products.
//
// A cluster of two CTAs on two SMs runs two consecutive 128-row query tiles
// of one (segment, kv head): rows are P query positions x G grouped q heads
// (row m = position m/G, head m%G). The even CTA issues M = 256 MMAs that
// span both tiles. B operands are split by N between the CTAs, so each SM
// loads half of every K/V tile: the keys [64r, 64r+64) of K and the head_dim
// columns [64r, 64r+64) of V, for CTA r. The TMA unit's cost is mostly per
// box (about 70 SM cycles for a 2 KiB box): a K sub-tile (16 keys, both
// halves of head_dim) is one 4 KiB box through a five-dimensional view of the
// pool, a V sub-tile half one 2 KiB box (the half belongs to one CTA), so an
// SM takes 12 boxes per tile. A 128-row tile alone would need about 60 B/clk
// to keep its tensor core busy, a pair needs half of that per SM.
//
//   warp 0 (32 lanes)  TMA producer, both CTAs: Q once, then per 128-key tile
//                      12 boxes of this CTA's parts, counted on the even
//                      CTA's barriers; six stages.
//   warp 1 (one lane)  QK issuer, even CTA only: S_j = Q K_j^T (SS, M 256,
//                      N 128 keys) into S/P buffer j % 3, as soon as that
//                      buffer's previous P V product has finished.
//   warp 6 (one lane)  PV issuer, even CTA only: O += P_j V_j (TS, A = P in
//                      TMEM, N 128 = head_dim) as soon as P_j is written.
//                      A tcgen05.mma issue blocks its thread until the tensor
//                      pipe takes it, so one thread issuing both streams would
//                      serialise them with its waits; two issuers keep the
//                      pipe fed. Commits arrive on the barriers of both CTAs.
//   warps 2-5          softmax, both CTAs: thread = TMEM lane = row; masks the
//                      causal/ragged edge, writes P_j = 2^(s*scale*log2e - m)
//                      as bf16 over S_j, keeps the row sum l in fp32 registers,
//                      rescales O and l only when the running max grew by more
//                      than 2^8; final normalisation and store.
//
// The rows past a segment's last tile (an odd tile count) belong to a CTA that
// still loads its halves and runs the softmax, but stores nothing.
//
// TMEM columns (same in both CTAs): [128b, 128b+128) S/P buffer b for b < 3,
// [384,512) O. Every mbarrier wait is
// bounded; on expiry the CTA records PKV_DEV_TIMEOUT and both CTAs still meet
// at the closing cluster barrier, after the MMAs drained, before TMEM is freed.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int D = 128;
constexpr int kKeysPerTile = 128;
constexpr int kSubPerTile = kKeysPerTile / kSubKeys;  // 8 sub-tiles of 16 keys
constexpr int kTmemCols = 512;
constexpr int kSBufs = 3;      // S/P buffers in TMEM
constexpr int kOCol = 384;
// Warps 0-3 (one warpgroup): softmax, one per TMEM lane quarter. Warps 4-7:
// TMA producer, QK issuer, PV issuer, and one idle warp that completes the
// warpgroup. The kernel launches with kLaunchRegs registers per thread; the
// softmax warpgroup then raises its share to kSoftmaxRegs and the other
// warpgroup lowers its own to kOtherRegs (the sum is unchanged), so each SM
// sub-partition holds one softmax warp and one other warp in 9,728 registers
// and keeps room for a decode warp of the same step beside them.
constexpr int kThreads = 256;
constexpr int kWarpProducer = 4, kWarpQK = 5, kWarpPV = 6;
constexpr int kLaunchRegs = 152, kSoftmaxRegs = 216, kOtherRegs = 88;
static_assert(kSoftmaxRegs + kOtherRegs == 2 * kLaunchRegs, "register shares must add up to the launch's");
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > 256x
constexpr uint32_t kFull = 0xffffffffu;
constexpr uint32_t kNegInfBits = 0xff800000u;

// NST K/V tiles in flight: six when the chunk kernel has its SMs to itself (the
// producer runs well ahead of the MMAs), three when a decode CTA shares each SM.
template <int NST>
struct Layout {
  static constexpr int kStages = NST;
  static constexpr int kQHalf = 128 * 128;                 // 128 rows x 128 B: one 64-column half of D
  static constexpr int kQBytes = 2 * kQHalf;
  static constexpr int kKSub = kSubKeys * 256;              // one 16-key sub-tile of K: [2 groups][2 halves][8 keys][128 B]
  static constexpr int kKBytes = (kKeysPerTile / 2 / kSubKeys) * kKSub;  // this CTA's 64 keys
  static constexpr int kVBytes = kKeysPerTile * 128;       // 128 keys x this CTA's 64 columns
  static constexpr int kStageBytes = kKBytes + kVBytes;    // 32 KiB: 4 K boxes of 4 KiB, 8 V boxes of 2 KiB
  static constexpr int kBarOffset = kQBytes + kStages * kStageBytes;
  static constexpr int kSmem = kBarOffset + 256 + 1024;    // barriers/flags + alignment slack
};
static_assert(Layout<6>::kSmem <= 232448, "dynamic shared memory per CTA");

// Barrier indices for NST stages.
template <int NST>
struct Bars {
  static constexpr int kQFull = 0;                     // even CTA: both Q tiles
  static constexpr int kKVFull = 1;                    // +stage; even CTA: both CTAs' halves of a K/V tile
  static constexpr int kKVEmpty = kKVFull + NST;       // +stage; both CTAs
  static constexpr int kSFull = kKVEmpty + NST;        // +buffer (3); both CTAs
  static constexpr int kPReady = kSFull + kSBufs;      // +buffer (3); even CTA: one arrival per softmax warp of the pair
  static constexpr int kPVDone = kPReady + kSBufs;     // +buffer (3); both CTAs
  static constexpr int kDrain = kPVDone + kSBufs;      // QK issuer's MMAs complete
  static constexpr int kDrainPV = kDrain + 1;          // PV issuer's MMAs complete
  static constexpr int kNumBars = kDrainPV + 1;
  static_assert(kNumBars * 8 + 8 <= 256, "barriers, TMEM address and abort flag fit their 256 bytes");
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Wait that also gives up as soon as another role of this CTA has aborted.
// `cluster` selects cluster-scope acquire (barriers the other CTA arrives on).
// Plain try_wait (no suspend-time hint): every wait here is on the critical
// path of the tile pipeline, and a suspended thread can resume late.
template <bool cluster = false>
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort) {
  auto poll = [&]() { return cluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  if (poll()) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (poll()) return true;
    if ((i & 15u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > 1000000000ull) {
        *abort = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool warp_wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort) {
  return __all_sync(kFull, wait_or_abort(bar, parity, abort));
}

template <int NST>
__global__ void __maxnreg__(kLaunchRegs) prefill_pair_kernel(const __grid_constant__ CUtensorMap tmap_q,
                                                                   const __grid_constant__ CUtensorMap tmap_k,
                                                                   const __grid_constant__ CUtensorMap tmap_v,
                                                                   const StepArgs a,
                                                                   const int32_t *__restrict__ items,
                                                                   int rows_per_tile) {
  using Lay = Layout<NST>;
  constexpr int kStages = NST;
  constexpr int kQFull = Bars<NST>::kQFull, kKVFull = Bars<NST>::kKVFull, kKVEmpty = Bars<NST>::kKVEmpty;
  constexpr int kSFull = Bars<NST>::kSFull, kPReady = Bars<NST>::kPReady, kPVDone = Bars<NST>::kPVDone;
  constexpr int kDrain = Bars<NST>::kDrain, kDrainPV = Bars<NST>::kDrainPV, kNumBars = Bars<NST>::kNumBars;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint8_t *sQ = smem;
  uint8_t *sKV = smem + Lay::kQBytes;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + Lay::kBarOffset);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + kNumBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.y;
  const uint32_t rank = cluster_ctarank();  // 0 issues the MMAs
  // The work item, step metadata, q and the cached history are final when this
  // grid starts (the kernel before it in the stream, the cache write, signals
  // dependents only after its own wait); only the keys this step appends come
  // from that kernel, and the producer waits for it before loading the first
  // tile that holds them (before the first tile at all when the K/V source is
  // a scratch pool the previous kernel fills).
  launch_dependents();
  const int4 it = reinterpret_cast<const int4 *>(items)[blockIdx.x >> 1];
  const int seg = it.x, slot = it.y, tile0 = it.z;
  const int G = a.group, P = rows_per_tile;

  // Both CTAs of the pair read the same item, so they agree on `bad` and leave together.
  bool bad = seg < 0 || seg >= a.num_seqs || slot < 0 || slot >= a.max_slots || tile0 < 0;
  int row0 = 0, n = 0, L = 0;
  if (!bad) {
    row0 = a.cu_seqlens_q[seg];
    n = a.cu_seqlens_q[seg + 1] - row0;
    L = a.context_lens[slot];
    bad = a.seq_slot[seg] != slot || n < 2 || n > L ||
          static_cast<int64_t>(L) > static_cast<int64_t>(a.max_blocks_per_slot) * a.block_size ||
          tile0 * P >= n || row0 < 0 || static_cast<int64_t>(row0) + n > a.total_q;
  }
  if (bad) {
    if (threadIdx.x == 0 && rank == 0 && a.status) atomicOr(a.status, PKV_DEV_BAD_SEGMENT);
    return;
  }
  const int q_tiles = (n + P - 1) / P;
  const int tile = tile0 + static_cast<int>(rank);
  const bool present = tile < q_tiles;              // else: rows past the segment, nothing stored
  const int pos0 = (present ? tile : tile0) * P;    // first query row of this CTA's tile
  const int rows = present ? min(P, n - pos0) : 0;
  const int last = min(tile0 + 1, q_tiles - 1);     // the pair's last present tile
  const int kv_end = L - n + min(n, (last + 1) * P);  // keys [0, kv_end) are visible to some row of the pair
  const int ntiles = (kv_end + kKeysPerTile - 1) / kKeysPerTile;
  const int32_t *bt_row = a.block_tables + static_cast<int64_t>(slot) * a.max_blocks_per_slot;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(bar + i, (i >= kPReady && i < kPReady + kSBufs) ? 8 : 1);
    fence_barrier_init();
    *abort_flag = 0;
  }
  // Rows of the Q tile beyond G*P whole groups stay zero.
  {
    const int qrows = G * P;
    const int chunks = (128 - qrows) * 8;  // 16-byte chunks per half
    for (int i = threadIdx.x; i < chunks * 2; i += blockDim.x) {
      const int h = i / chunks, rem = i % chunks;
      *reinterpret_cast<uint4 *>(sQ + h * Lay::kQHalf + (qrows + rem / 8) * 128 + (rem % 8) * 16) =
          make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  if (warp == kWarpQK) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers initialised and Q padding written in both CTAs
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 4) {
   setmaxnreg_dec<kOtherRegs>();
   if (warp == kWarpProducer) {
    // ------------------------------------------------------------ producer
    // Pool rows of the 16-key sub-tiles, four tiles per warp-wide load: lane l
    // covers sub-tile l % 8 of tile t0 + l / 8. The block IDs of the next group
    // are loaded raw one group ahead and turned into rows (checked against the
    // pool: 0 when outside it, the status word reports it) only when that
    // group comes into use, so no block-table latency is ever waited on.
    auto group_ids = [&](int t0) -> int {
      const int key = (t0 + (lane >> 3)) * kKeysPerTile + (lane & 7) * kSubKeys;
      return key < kv_end ? __ldg(bt_row + key / a.block_size) : 0;
    };
    auto group_rows = [&](int t0, int blk) -> int {
      const int key = (t0 + (lane >> 3)) * kKeysPerTile + (lane & 7) * kSubKeys;
      if (key >= kv_end) return 0;
      if (blk < 0 || blk >= a.num_blocks) {
        if (a.status) atomicOr(a.status, PKV_DEV_BAD_BLOCK);
        return 0;
      }
      return (blk * a.num_kv_heads + g) * a.block_size + key % a.block_size;
    };
    int rows_cur = group_rows(0, group_ids(0)), ids_next = group_ids(4);
    const uint32_t q_full = cluster_addr(bar + kQFull, 0);
    if (lane == 0) {
      prefetch_tensormap(&tmap_q);
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
      if (rank == 0) mbar_arrive_expect_tx(bar + kQFull, 2 * 2 * G * P * 128);
      for (int h = 0; h < 2; ++h)
        tma_load_3d_pair(sQ + h * Lay::kQHalf, &tmap_q, h * 64, g * G, row0 + pos0, q_full);
    }
    // Lane l < 4 loads K sub-tile 4r + l (both halves of head_dim, one box);
    // lane 8 <= l < 16 loads V sub-tile l-8, this CTA's half of head_dim.
    const bool is_k = lane < 4, is_v = lane >= 8 && lane < 16;
    const int u = is_k ? static_cast<int>(rank) * 4 + lane : lane - 8;
    const int dst_off = is_k ? lane * Lay::kKSub : Lay::kKBytes + (lane - 8) * kSubKeys * 128;
    const int bs_shift = 31 - __clz(a.block_size);  // block sizes are powers of two
    bool waited = false;
    for (int j = 0; j < ntiles; ++j) {
      const int s = j % kStages;
      if (j >= kStages && !warp_wait_or_abort(bar + kKVEmpty + s, ((j - kStages) / kStages) & 1, abort_flag)) break;
      if (j > 0 && (j & 3) == 0) {
        rows_cur = group_rows(j, ids_next);
        ids_next = group_ids(j + 4);
      }
      const int kt0 = j * kKeysPerTile;
      const int vs = min(kSubPerTile, (kv_end - kt0 + kSubKeys - 1) / kSubKeys);  // sub-tiles with a visible key
      const uint32_t kv_full = cluster_addr(bar + kKVFull + s, 0);
      // The pair loads 4 boxes per visible sub-tile: two K halves (one CTA) and two V halves (one each).
      if (rank == 0 && lane == 0) mbar_arrive_expect_tx(bar + kKVFull + s, vs * 4 * 2048);
      const int urow = __shfl_sync(kFull, rows_cur, (j & 3) * 8 + (u & 7));
      // wait for the kernel before: at the first tile holding rows the cache write appends, or at once
      // when that kernel wrote the whole K/V source
      if (!waited && (a.kv_from_previous || (j + 1) * kKeysPerTile > L - n)) {
        grid_dependency_wait();
        waited = true;
      }
      if (is_k && u < vs)
        tma_load_5d_pair(sKV + s * Lay::kStageBytes + dst_off, &tmap_k, 0, 0, 0, (urow & (a.block_size - 1)) >> 3,
                         urow >> bs_shift, kv_full);
      if (is_v && u < vs)
        tma_load_2d_pair(sKV + s * Lay::kStageBytes + dst_off, &tmap_v, static_cast<int>(rank) * 64, urow, kv_full);
    }
  } else if (warp == kWarpQK) {
    // ------------------------------------------------------------ QK issuer
    if (rank == 0 && lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(256, kKeysPerTile, 0, 0);
      const uint32_t q_base = smem_addr(sQ);
      bool ok = wait_or_abort(bar + kQFull, 0, abort_flag);
      tc_fence_after();
      for (int j = 0; ok && j < ntiles; ++j) {
        const int s = j % kSBufs;
        // S buffer s last held P_{j-3}: its product with V must have finished.
        if (j >= kSBufs && !(ok = wait_or_abort(bar + kPVDone + s, ((j - kSBufs) / kSBufs) & 1, abort_flag))) break;
        if (!(ok = wait_or_abort(bar + kKVFull + j % kStages, (j / kStages) & 1, abort_flag))) break;
        tc_fence_after();
        const uint32_t k_base = smem_addr(sKV + (j % kStages) * Lay::kStageBytes);
        for (int kk = 0; kk < D / 16; ++kk) {
          // K: 8-key groups 2048 B apart, the second half of head_dim 1024 B after the first
          const uint32_t qoff = (kk >> 2) * Lay::kQHalf + (kk & 3) * 32;
          const uint32_t koff = (kk >> 2) * 1024 + (kk & 3) * 32;
          tc_mma_ss_pair(tmem + s * 128, smem_desc_sw128(q_base + qoff, 16, 1024),
                         smem_desc_sw128(k_base + koff, 16, 2048), idesc_qk, kk > 0 ? 1u : 0u);
        }
        tc_commit_pair(bar + kSFull + s);
      }
      tc_commit_pair(bar + kDrain);
      if (!wait_or_abort(bar + kDrain, 0, abort_flag) && a.status) atomicOr(a.status, PKV_DEV_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == kWarpPV) {
    // ------------------------------------------------------------ PV issuer
    if (rank == 0 && lane == 0) {
      constexpr uint32_t idesc_pv = idesc_bf16_f32(256, D, 0, 1);
      for (int j = 0; j < ntiles; ++j) {
        const int sp = j % kSBufs;
        // P_j written by all eight softmax warps of the pair; V_j has landed (S_j used K_j of the same stage).
        if (!wait_or_abort<true>(bar + kPReady + sp, (j / kSBufs) & 1, abort_flag)) break;
        tc_fence_after();
        const int valid = min(kKeysPerTile, kv_end - j * kKeysPerTile);
        const int ksteps = (valid + kSubKeys - 1) / kSubKeys;
        const uint32_t v_base = smem_addr(sKV + (j % kStages) * Lay::kStageBytes + Lay::kKBytes);
        for (int ks = 0; ks < ksteps; ++ks) {
          const uint64_t bdesc = smem_desc_sw128(v_base + ks * kSubKeys * 128, Lay::kVBytes, 1024);
          tc_mma_ts_pair(tmem + kOCol, tmem + sp * 128 + ks * 8, bdesc, idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
        }
        tc_commit_pair(bar + kPVDone + sp);
        tc_commit_pair(bar + kKVEmpty + j % kStages);
      }
      tc_commit_pair(bar + kDrainPV);
      if (!wait_or_abort(bar + kDrainPV, 0, abort_flag) && a.status) atomicOr(a.status, PKV_DEV_TIMEOUT);
    }
    __syncwarp();
   }
  } else {
    // ------------------------------------------------------------ softmax
    setmaxnreg_inc<kSoftmaxRegs>();
    const int qw = warp;
    const int mrow = qw * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(qw * 32) << 16;
    const int pos = mrow / G;
    const int p_row = L - n + pos0 + pos;  // last visible key of this row (inclusive)
    const float sl2 = a.scale_log2;
    const uint32_t p_ready0 = cluster_addr(bar + kPReady, 0);
    float m_used = -INFINITY;  // log2 units
    bool ok = true;
    float l_sum = 0.f, l_odd = 0.f;  // row sum, as even and odd columns (packed adds)
    for (int j = 0; j < ntiles; ++j) {
      const int s = j % kSBufs;
      if (!(ok = warp_wait_or_abort(bar + kSFull + s, (j / kSBufs) & 1, abort_flag))) break;
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
      // Row max: three-input max, four independent chains.
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; i += 2)
          mx4[(i >> 1) & 3] = max3(mx4[(i >> 1) & 3], __uint_as_float(sv[c][i]), __uint_as_float(sv[c][i + 1]));
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * sl2;
      const float m_new = fmaxf(m_used, mx);
      const bool need = j > 0 && m_new > m_used + kRescaleThreshold;
      if (j == 0) m_used = m_new;
      if (__any_sync(kFull, need)) {
        // O must hold tile j-1's products before it is rescaled.
        if (!(ok = warp_wait_or_abort(bar + kPVDone + (j - 1) % kSBufs, ((j - 1) / kSBufs) & 1, abort_flag))) break;
        tc_fence_after();
        const float corr = need ? ex2_approx(m_used - m_new) : 1.f;
        if (need) m_used = m_new;
        l_sum *= corr;
        l_odd *= corr;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(tmem + lane_base + kOCol + c * 32, ov);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * corr);
          tmem_st32(tmem + lane_base + kOCol + c * 32, ov);
        }
      }
      const float nm = -m_used;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float x0, x1;
          fma2(x0, x1, __uint_as_float(sv[c][2 * i]), __uint_as_float(sv[c][2 * i + 1]), sl2, sl2, nm, nm);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          add2(l_sum, l_odd, p0, p1);
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st16(tmem + lane_base + s * 128 + c * 16, pk);
      }
      if (j == ntiles - 1) {
        // Zero this CTA's V rows past the last visible key inside the final
        // 16-key step: a partly filled block may hold stale or NaN rows there,
        // and 0 * NaN would reach O. The tile's data has landed (S_j exists).
        const int valid = kv_end - j * kKeysPerTile;
        const int tail = (kSubKeys - valid % kSubKeys) % kSubKeys;
        if (tail) {
          uint8_t *sV = sKV + (j % kStages) * Lay::kStageBytes + Lay::kKBytes;
          for (int i = threadIdx.x; i < tail * 8; i += 128)
            *reinterpret_cast<uint4 *>(sV + (valid + i / 8) * 128 + (i % 8) * 16) = make_uint4(0, 0, 0, 0);
          fence_proxy_async_smem();
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      // Only the last tile also wrote shared memory (the V tail) for the MMA to read.
      if (lane == 0) {
        if (j == ntiles - 1)
          mbar_arrive_cluster(p_ready0 + s * 8);
        else
          mbar_arrive_remote_cta_release(p_ready0 + s * 8);
      }
    }
    if (ok && warp_wait_or_abort(bar + kPVDone + (ntiles - 1) % kSBufs, ((ntiles - 1) / kSBufs) & 1, abort_flag)) {
      tc_fence_after();
      const float inv = 1.f / (l_sum + l_odd);
      constexpr int kRowBytes = D * 2, kChunks = kRowBytes / 16;
      if (!a.out_on_host) {
        // each thread stores its own row, 64 bytes per TMEM load (the loads are warp-wide)
        const bool row_valid = mrow < G * P && pos < rows;
        uint4 *orow = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(a.out) +
                                                (static_cast<size_t>(row0 + pos0 + pos) * a.num_q_heads + g * G +
                                                 mrow % G) * D);
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
#pragma unroll
            for (int v = 0; v < 4; ++v)
              orow[c * 4 + v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      } else {
        // Output in host memory: the rows leave through shared memory, the Q
        // tile (no longer read once the last P.V is done, its S consumed
        // above). Each warp stages its 32 rows (16-byte chunk k of row r at
        // chunk k ^ (r % 16), which keeps the banks apart both ways), then a
        // half-warp stores one whole 256-byte row per instruction.
        static_assert(kChunks == 16 && 4 * 32 * kRowBytes <= Lay::kQBytes, "four warps' rows fit in the Q tile");
        uint8_t *stage = sQ + qw * 32 * kRowBytes;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(tmem + lane_base + kOCol + c * 32, ov);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv, __uint_as_float(ov[2 * i + 1]) * inv);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            *reinterpret_cast<uint4 *>(stage + lane * kRowBytes + (((c * 4 + v) ^ (lane & 15)) << 4)) =
                make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
        __syncwarp();
        const int k = lane % kChunks;
#pragma unroll 4
        for (int r0 = 0; r0 < 32; r0 += 32 / kChunks) {
          const int r = r0 + lane / kChunks, mr = qw * 32 + r;
          const int rpos = mr / G, rhh = mr % G;
          if (mr < G * P && rpos < rows) {
            const uint4 v = *reinterpret_cast<const uint4 *>(stage + r * kRowBytes + ((k ^ (r & 15)) << 4));
            reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(a.out) +
                                      (static_cast<size_t>(row0 + pos0 + rpos) * a.num_q_heads + g * G + rhh) *
                                          D)[k] = v;
          }
        }
      }
    }
  }

  tc_fence_before();
  cluster_sync();  // both CTAs are done with TMEM and the MMAs have drained
  if (*abort_flag && threadIdx.x == 0 && a.status) atomicOr(a.status, PKV_DEV_TIMEOUT);
  if (warp == kWarpQK) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

template <int NST>
cudaError_t launch_pair_t(const StepArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                          int32_t rows_per_tile, int32_t num_items, const int32_t *items, cudaStream_t stream) {
  constexpr int smem = Layout<NST>::kSmem;
  static std::atomic<uint64_t> configured{0};  // one bit per device
  if (const cudaError_t e = allow_smem_once(prefill_pair_kernel<NST>, smem, configured); e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * num_items), static_cast<unsigned>(a.num_kv_heads));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, prefill_pair_kernel<NST>, tq, tk, tv, a, items, rows_per_tile);
}

}  // namespace

cudaError_t launch_prefill_pair(const StepArgs &a, const CUtensorMap &tq, const CUtensorMap &tk,
                                const CUtensorMap &tv, int32_t rows_per_tile, int32_t num_items,
                                const int32_t *items, bool beside_decode, cudaStream_t stream) {
  if (num_items <= 0) return cudaSuccess;
  return beside_decode ? launch_pair_t<kPairStagesBesideDecode>(a, tq, tk, tv, rows_per_tile, num_items, items, stream)
                       : launch_pair_t<6>(a, tq, tk, tv, rows_per_tile, num_items, items, stream);
}

}  // namespace pkv
