// Split-KV decode attention (persistent warps) and the span merge.
//
// Lucebox, "Continuous batching: Qwen3.8-27B at 301 tok/s across five
// clients, up to 1.97x llama.cpp", §Paged KV and paged attention: attention
// follows each sequence's block table in logical order over the shared pool.
// mlxcel manual, "Continuous batching", §Paged KV cache and prefix sharing:
// batched paged decode reads blocks in place (a block-table kernel) instead
// of rebuilding a contiguous window every step.
//
// Decode kernel. A task is one (decode segment, key span of PKV_SPLIT_KEYS
// keys, kv head). The grid is one CTA per SM with eight warps (four to six,
// with deeper rings, on steps with few tasks); every warp is
// an independent worker taking tasks t = w, w + W, w + 2W (W = all warps; the
// work list is sorted longest first and consecutive tasks go to different
// SMs), then, on steps with more tasks, the next unclaimed task from a counter
// in the workspace: some SMs stream faster than others, and claiming keeps
// them all busy to the end. A warp streams its tasks' 16-key K/V sub-tiles
// through its own three-stage ring in shared memory with TMA (64-column x 16-row boxes,
// 128-byte swizzle) straight from the pool rows the block table names. The
// ring keeps flowing across task boundaries: the next task's metadata and
// block IDs load while the current task computes, and its first sub-tiles are
// requested before the current task ends. Eight warps x three 8 KiB stages
// keep ~192 KiB of K/V in flight per SM, enough to cover HBM latency; a step
// with four to six tasks per SM runs four to six warps with six to four
// stages, so its busy warps keep about as much in flight.
//
// Math per sub-tile: warp-level bf16 MMA (m16n8k16), fp32 accumulation,
//   S^T[16 keys][8 heads] = K[16 keys][D] * Q^T[D][8 heads]   (GQA group on N)
//   O^T[D][8 heads]      += V^T[D][16 keys] * P^T[16 keys][8 heads]
// with an online softmax per head in the exp2 domain; P^T reaches the second
// MMA's B operand through an in-register 8x8 transpose (movmatrix). The
// running output is rescaled only when a head's max grows by more than 2^8.
//
// A segment may also be a short run of causal rows (n rows with n x group <=
// 16, e.g. draft tokens being verified): the MMA columns are then the (row,
// q head) pairs, all rows share every K/V sub-tile the warp loads, and row i
// masks the keys past L - n + i. Such a run can leave a row with no visible
// key in the last span; its partial is (max -inf, sum 0) and the merge gives
// it weight 0.
//
// A single-span segment's result goes straight to the output; otherwise each
// span writes a partial (unnormalised sum, reference max, denominator) and the
// merge kernel, launched right behind the decode kernel (programmatic
// dependent launch), combines the spans of each (segment, q head) in a fixed
// order. Nothing depends on timing or on other segments: results are
// deterministic and independent of the rest of the batch.
//
// Keys past the context in a partly filled block are masked to -inf in S and
// their V values zeroed in registers, so stale or NaN pool rows never reach
// the output.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "pkv_decode_task.cuh"
#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kWarps = 8;  // independent workers per CTA on steps that fill every warp
constexpr uint32_t kFull = 0xffffffffu;
constexpr float kRescale = 8.0f;  // log2 units

// NW warps per CTA, each with a ring of NST stages (0: 24 KiB per warp).
template <int D, int NW = kWarps, int NST = 0>
struct DecodeCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kHalfBytes = kSubKeys * 128;        // 16 rows x 128 B
  static constexpr int kTileBytes = kHalves * kHalfBytes;  // one K (or V) sub-tile
  static constexpr int kStageBytes = 2 * kTileBytes;       // K then V
  static constexpr int kStages = NST > 0 ? NST : (24 * 1024) / kStageBytes;  // default 3 (D=128) or 6 (D=64)
  static constexpr int kWarpRing = kStages * kStageBytes;
  static constexpr int kSmem = NW * kWarpRing + NW * kStages * 8 + 1024;
  static_assert(kSmem <= 227 * 1024, "ring does not fit in shared memory");
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Q^T fragments (B operand): column c = nt*8 + lane/4 is (row c / G, head
// c % G) of the segment; d = kk*16 + (lane%4)*2 (+8). Columns past rows x G are zero.
template <int D, int NT, bool MULTI>
__device__ __forceinline__ void load_q(uint32_t (&qf)[NT][D / 16][2], const Task &T, const StepArgs &a,
                                       int lane) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int col = nt * 8 + (lane >> 2);
    const bool valid = col < (MULTI ? T.nrows : 1) * a.group;
    const int i = MULTI && valid ? col / a.group : 0, h = !MULTI ? col : valid ? col % a.group : 0;
    const uint16_t *qrow = static_cast<const uint16_t *>(a.q) +
                           ((static_cast<size_t>(T.row0) + i) * a.num_q_heads + T.g * a.group + h) * D;
    const uint32_t *qp = reinterpret_cast<const uint32_t *>(qrow) + (lane & 3);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qf[nt][kk][0] = valid ? __ldg(qp + kk * 8) : 0u;
      qf[nt][kk][1] = valid ? __ldg(qp + kk * 8 + 4) : 0u;
    }
  }
}

// NT: 8-column MMA tiles of (row, q head) columns; MULTI: segments may hold
// more than one row (otherwise every segment is a single decode row).
// NW, NS: warps per CTA and stages per warp ring. A warp's stream of
// sub-tiles is latency-bound (its ring's bytes per HBM round trip), so steps
// with fewer tasks than warps run fewer warps with deeper rings; the math of
// a task does not depend on them.
template <int D, int NT, bool MULTI, int NW, int NS>
__global__ void __launch_bounds__(NW * 32, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                  const StepArgs a, const int32_t *__restrict__ items, int num_items) {
  using Cfg = DecodeCfg<D, NW, NS>;
  constexpr int KT = D / 16;  // k-steps of QK^T, m-tiles of PV
  constexpr int NST = Cfg::kStages;
  constexpr int kMaxRows = MULTI ? 16 : 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t *ring = smem + warp * Cfg::kWarpRing;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + NW * Cfg::kWarpRing) + warp * NST;

  // The span merge may launch now; it waits for this grid before reading.
  launch_dependents();
  const int hkv = a.num_kv_heads;
  const int num_tasks = num_items * hkv;
  const int stride = gridDim.x * NW;
  const int t0 = warp * gridDim.x + blockIdx.x;
  if (t0 >= num_tasks) return;
  if (lane == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(full + s, 1);
    fence_barrier_init();
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }
  __syncwarp();
  // Metadata, q and the history rows are final when this grid starts (the
  // kernel before it in the stream signals dependents only after its own
  // wait); the rows written by that kernel itself (this step's K/V, the last
  // span of each row) are read only after waiting for it, in issue().
  bool waited = false;

  // A warp's tasks: t0, t0 + stride, t0 + 2 stride, then (with a task
  // counter) 3 stride + the counter's next value, else t0 + 3 stride, ...
  // A is current, B expanded, tC the task whose work item is in rawC.
  uint32_t *const counter = a.task_counter;
  Task A, B;
  int4 rawC = make_int4(0, 0, 0, 0);
  expand(A, t0, load_item(items, t0, hkv), a, lane);
  int tC;
  {
    const int t1 = t0 + stride;
    expand(B, t1 < num_tasks ? t1 : -1, t1 < num_tasks ? load_item(items, t1, hkv) : rawC, a, lane);
    tC = t1 + stride;
    if (tC < num_tasks) rawC = load_item(items, tC, hkv);
  }
  finalize(A, a, lane, 8 * NT, kMaxRows);
  uint32_t qA[NT][KT][2], qB[NT][KT][2];
  if (A.ok) load_q<D, NT, MULTI>(qA, A, a, lane);
  bool qB_loaded = false;

  int P = 0, C = 0, pa = 0, pb = 0;
  int pstage = 0;  // P % NST
  // Each history row is read once per step: its L2 lines go first, which keeps
  // the span partials this grid writes in L2 for the merge.
  const uint64_t policy = l2_evict_first_policy();
  auto issue = [&](const Task &T, int u) {
    // only the sub-tiles holding this step's rows wait for the cache write
    if (!waited && T.reads_new && T.key0 + (u + 1) * kSubKeys > T.L - T.nrows) {
      grid_dependency_wait();
      waited = true;
    }
    const int row = __shfl_sync(kFull, T.row, u);
    if (lane == 0) {
      uint64_t *bar = full + pstage;
      uint8_t *dst = ring + pstage * Cfg::kStageBytes;
      if (row >= 0) {
        mbar_arrive_expect_tx(bar, Cfg::kStageBytes);
#pragma unroll
        for (int h = 0; h < Cfg::kHalves; ++h) {
          tma_load_2d_hint(dst + h * Cfg::kHalfBytes, &tmap_k, h * 64, row, bar, policy);
          tma_load_2d_hint(dst + Cfg::kTileBytes + h * Cfg::kHalfBytes, &tmap_v, h * 64, row, bar, policy);
        }
      } else {
        mbar_arrive(bar);  // nothing loaded; the consumer masks this sub-tile out
      }
    }
    ++P;
    pstage = pstage + 1 == NST ? 0 : pstage + 1;
  };
  auto issue_next = [&]() -> bool {
    if (pa < A.units) {
      issue(A, pa++);
      return true;
    }
    if (B.t >= 0) {
      if (!B.finalized) {
        finalize(B, a, lane, 8 * NT, kMaxRows);
        if (B.ok) {
          load_q<D, NT, MULTI>(qB, B, a, lane);
          qB_loaded = true;
        }
      }
      if (pb < B.units) {
        issue(B, pb++);
        return true;
      }
    }
    return false;
  };
  while (P - C < NST && issue_next()) {
  }

  // Per-lane byte offsets of the swizzled ldmatrix rows inside a 64-column
  // half, for K (A operand, rows = keys) and V (transposed A operand).
  // Row r's 16-byte chunk c sits at chunk c ^ (r % 8) (128-byte swizzle).
  uint32_t koff[4], voff[4];
  {
    const int j = lane >> 3;
    const int rk = (lane & 7) + ((j & 1) << 3), rv = (lane & 7) + ((j >> 1) << 3);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      koff[q] = rk * 128 + ((((q << 1) + (j >> 1)) ^ (rk & 7)) << 4);
      voff[q] = rv * 128 + ((((q << 1) + (j & 1)) ^ (rv & 7)) << 4);
    }
  }
  const uint32_t ring_addr = smem_addr(ring);
  const float sl2 = a.scale_log2;
  const int G = a.group;
  const int ka = lane >> 2, kb = ka + 8, k0 = (lane & 3) * 2;
  int cstage = 0;
  uint32_t cphase = 0;  // (C / NST) & 1

  while (A.t >= 0) {
    // Claim the task after tC now; the answer is needed only when A is done.
    uint32_t claim = 0;
    if (counter && tC < num_tasks && lane == 0) claim = atomicAdd(counter, 1u);
    // m: the reference max each head's sums are scaled to (log2 units); it is
    // only raised when a head's running max exceeds it by more than 2^8, so
    // exp2(x - m) <= 256 and the sums stay exact up to rounding.
    float m[NT][2], l[NT][2], acc[NT][KT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m[nt][0] = m[nt][1] = -INFINITY;
      l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < KT; ++mt) acc[nt][mt][0] = acc[nt][mt][1] = acc[nt][mt][2] = acc[nt][mt][3] = 0.f;
    }

    // Row i of the segment sees keys up to L - rows + i. Byte nt*2 + c holds
    // the row of this thread's column (nt, c); padding columns take the last
    // row and so see every key.
    const int nrows = MULTI ? A.nrows : 1;
    uint32_t colrow = 0;
    if (MULTI) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int col = nt * 8 + (lane & 3) * 2 + c;
          const int i = col < nrows * G ? col / G : nrows - 1;
          colrow |= static_cast<uint32_t>(i & 0xFF) << (8 * (nt * 2 + c));
        }
    }

    for (int u = 0; u < A.units; ++u) {
      const int stage = cstage;
      if (!mbar_wait(full + stage, cphase)) {
        if (lane == 0 && a.status) atomicOr(a.status, PKV_DEV_TIMEOUT);
        return;
      }
      const int row = __shfl_sync(kFull, A.row, u);
      const int kbase = A.key0 + u * kSubKeys;
      // keys of the sub-tile that take part (0 for a block ID outside the pool)
      const int v = row >= 0 ? min(kSubKeys, A.key1 - kbase) : 0;
      const int vis0 = A.L - nrows - kbase + 1;  // keys of the sub-tile row 0 sees
      const uint32_t kaddr = ring_addr + stage * Cfg::kStageBytes;

      // S^T = K Q^T, split over two accumulators to halve the MMA chain.
      float s0[NT][4], s1[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) s0[nt][i] = s1[nt][i] = 0.f;
#pragma unroll
      for (int kk = 0; kk < KT; ++kk) {
        uint32_t af[4];
        ldmatrix_x4(af, kaddr + (kk >> 2) * Cfg::kHalfBytes + koff[kk & 3]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16_16816((kk & 1) ? s1[nt] : s0[nt], af, qA[nt][kk][0], qA[nt][kk][1]);
      }

      // Online softmax; this thread holds keys lane/4 and lane/4 + 8 of heads
      // (lane%4)*2 + {0, 1}. A column's maximum moves only when a logit passes
      // it by the lazy margin: each lane tests its own two keys, and only then
      // does the warp reduce the column maxima.
      float x[NT][2][2];
      bool need = false;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          // causal limit of this column's row (a single row sees the whole span)
          const int vis = MULTI ? min(v, vis0 + static_cast<int>((colrow >> (8 * (nt * 2 + c))) & 0xFF)) : v;
          x[nt][c][0] = ka < vis ? (s0[nt][c] + s1[nt][c]) * sl2 : -INFINITY;
          x[nt][c][1] = kb < vis ? (s0[nt][c + 2] + s1[nt][c + 2]) * sl2 : -INFINITY;
          need |= fmaxf(x[nt][c][0], x[nt][c][1]) > m[nt][c] + kRescale;
        }
      if (__any_sync(kFull, need)) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            float t = fmaxf(x[nt][c][0], x[nt][c][1]);
            t = fmaxf(t, __shfl_xor_sync(kFull, t, 4));
            t = fmaxf(t, __shfl_xor_sync(kFull, t, 8));
            t = fmaxf(t, __shfl_xor_sync(kFull, t, 16));
            if (t > m[nt][c] + kRescale) {
              const float corr = exp2f(m[nt][c] - t);
              m[nt][c] = t;
              l[nt][c] *= corr;
#pragma unroll
              for (int mt = 0; mt < KT; ++mt) {
                acc[nt][mt][c] *= corr;
                acc[nt][mt][c + 2] *= corr;
              }
            }
          }
      }
      uint32_t pf[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float m0 = m[nt][0] == -INFINITY ? 0.f : m[nt][0];
        const float m1 = m[nt][1] == -INFINITY ? 0.f : m[nt][1];
        uint32_t pk[2];  // keys ka / kb: heads (c=0, c=1) packed as bf16x2
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          pk[i] = pack_bf16x2(exp2f(x[nt][0][i] - m0), exp2f(x[nt][1][i] - m1));
          l[nt][0] += __uint_as_float(pk[i] << 16);
          l[nt][1] += __uint_as_float(pk[i] & 0xFFFF0000u);
        }
        pf[nt][0] = movmatrix_trans(pk[0]);
        pf[nt][1] = movmatrix_trans(pk[1]);
      }

      // O^T += V^T P^T; V rows of keys that do not take part are zeroed.
      const bool part = v < kSubKeys;
      const uint32_t mlo = (k0 < v ? 0x0000FFFFu : 0u) | (k0 + 1 < v ? 0xFFFF0000u : 0u);
      const uint32_t mhi = (k0 + 8 < v ? 0x0000FFFFu : 0u) | (k0 + 9 < v ? 0xFFFF0000u : 0u);
#pragma unroll
      for (int mt = 0; mt < KT; ++mt) {
        uint32_t af[4];
        ldmatrix_x4_trans(af, kaddr + Cfg::kTileBytes + (mt >> 2) * Cfg::kHalfBytes + voff[mt & 3]);
        if (part) {
          af[0] &= mlo;
          af[1] &= mlo;
          af[2] &= mhi;
          af[3] &= mhi;
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc[nt][mt], af, pf[nt][0], pf[nt][1]);
      }
      // Refill the ring by one. The stage's shared-memory reads are complete:
      // every ldmatrix result has been consumed by an MMA before the warp
      // converges here, so the next TMA write cannot overtake them.
      __syncwarp();
      ++C;
      if (++cstage == NST) {
        cstage = 0;
        cphase ^= 1u;
      }
      issue_next();
    }

    // ---- finish task A: the output row, or this span's partial ----
    if (A.ok) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float t = l[nt][c];
          t += __shfl_xor_sync(kFull, t, 4);
          t += __shfl_xor_sync(kFull, t, 8);
          t += __shfl_xor_sync(kFull, t, 16);
          l[nt][c] = t;
        }
      const int hbase = A.g * G;
      if (A.pbase < 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int col = nt * 8 + (lane & 3) * 2 + c;
            if (col < nrows * G) {
              const int i = MULTI ? col / G : 0, hh = MULTI ? col % G : col;
              __nv_bfloat16 *out = reinterpret_cast<__nv_bfloat16 *>(a.out) +
                                   ((static_cast<size_t>(A.row0) + i) * a.num_q_heads + hbase) * D + (lane >> 2);
              const float inv = 1.f / l[nt][c];
#pragma unroll
              for (int mt = 0; mt < KT; ++mt) {
                out[static_cast<size_t>(hh) * D + mt * 16] = __float2bfloat16_rn(acc[nt][mt][c] * inv);
                out[static_cast<size_t>(hh) * D + mt * 16 + 8] = __float2bfloat16_rn(acc[nt][mt][c + 2] * inv);
              }
            }
          }
      } else {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int col = nt * 8 + (lane & 3) * 2 + c;
            if (col < nrows * G) {
              // partial entry of (span, row i)
              const int i = MULTI ? col / G : 0, hh = MULTI ? col % G : col;
              const size_t pi = static_cast<size_t>(A.pbase + A.span * nrows + i) * a.num_q_heads + hbase;
              float *pacc = a.partial_acc + (pi + hh) * D + (lane >> 2);
#pragma unroll
              for (int mt = 0; mt < KT; ++mt) {
                pacc[mt * 16] = acc[nt][mt][c];
                pacc[mt * 16 + 8] = acc[nt][mt][c + 2];
              }
              if (lane < 4) {
                a.partial_ml[(pi + hh) * 2] = m[nt][c];
                a.partial_ml[(pi + hh) * 2 + 1] = l[nt][c];
              }
            }
          }
      }
    }

    // ---- advance: B becomes current, the task after it is expanded ----
    const int next_t = tC < num_tasks ? tC : num_tasks;
    int after = num_tasks;
    if (next_t < num_tasks) {
      if (counter) {
        const uint32_t c = __shfl_sync(kFull, claim, 0);
        after = c < static_cast<uint32_t>(num_tasks) ? 3 * stride + static_cast<int>(c) : num_tasks;
        if (after > num_tasks) after = num_tasks;
      } else {
        after = next_t + stride;
      }
    }
    A = B;
    pa = pb;
    pb = 0;
    if (A.t >= 0) {
      if (!A.finalized) finalize(A, a, lane, 8 * NT, kMaxRows);
      if (qB_loaded) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int kk = 0; kk < KT; ++kk) {
            qA[nt][kk][0] = qB[nt][kk][0];
            qA[nt][kk][1] = qB[nt][kk][1];
          }
      } else if (A.ok) {
        load_q<D, NT, MULTI>(qA, A, a, lane);
      }
    }
    qB_loaded = false;
    expand(B, next_t < num_tasks ? next_t : -1, rawC, a, lane);
    tC = after;
    if (tC < num_tasks) rawC = load_item(items, tC, hkv);
    while (P - C < NST && issue_next()) {
    }
  }
}

// Span merge. A row's result is fixed by its spans alone, whichever kernel
// below merges it, so it never depends on the step around it:
//   M   = the largest span max (exact), w_i = 2^(m_i - M) (0 for an empty span);
//   per group g of 8 consecutive spans, from zero and in span order,
//         L_g = sum l_i * w_i and A_g = sum acc_i * w_i (fused multiply-adds);
//   L = sum_g L_g and A = sum_g A_g, added in group order from zero;
//   out = bf16(A * (1 / L)).
// merge_small_kernel spreads a row's groups over four adjacent lanes per
// column (for the short steps, where merge latency is on the critical path);
// merge_wide_kernel gives each thread all groups of its columns and stages
// the spans' (max, denominator) pairs in shared memory (for steps with
// thousands of merges). Both take one float4 of columns per thread.
constexpr int kMergeThreads = 128;
constexpr int kGroup = 8;   // spans per group
constexpr int kPiece = 64;  // spans staged in shared memory at a time (a multiple of kGroup)

struct MergeRow {
  int row, spans, pbase, nrows;
  bool bad;
};

// Decode a merge item and check it against the step metadata.
__device__ __forceinline__ MergeRow merge_row(const StepArgs &a, const int32_t *items, int item) {
  const int4 it = __ldg(reinterpret_cast<const int4 *>(items) + item);
  // word 2: spans | row index << 16 | (rows - 1) << 24; word 3: the partial
  // entry of (span 0, this row); span s of the row is entry word3 + s * rows.
  MergeRow r;
  const int seg = it.x, slot = it.y;
  r.pbase = it.w;
  r.spans = it.z & 0xFFFF;
  const int ri = (it.z >> 16) & 0xFF;
  r.nrows = ((it.z >> 24) & 0xFF) + 1;
  r.row = 0;
  r.bad = seg < 0 || seg >= a.num_seqs || slot < 0 || slot >= a.max_slots || r.spans < 2 || r.pbase < 0 ||
          ri >= r.nrows;
  if (!r.bad) {
    const int row0 = __ldg(a.cu_seqlens_q + seg);
    const int L = __ldg(a.context_lens + slot);
    r.row = row0 + ri;
    r.bad = __ldg(a.seq_slot + seg) != slot || __ldg(a.cu_seqlens_q + seg + 1) - row0 != r.nrows ||
            (L + PKV_SPLIT_KEYS - 1) / PKV_SPLIT_KEYS != r.spans || row0 < 0 || row0 + r.nrows > a.total_q ||
            r.nrows > L;
  }
  return r;
}

__device__ __forceinline__ float span_weight(float m, float M) { return m == -INFINITY ? 0.f : exp2f(m - M); }

__device__ __forceinline__ void fold_span(float &lg, float4 &ag, float l, const float4 &acc, float w) {
  lg = __fmaf_rn(l, w, lg);
  ag.x = __fmaf_rn(acc.x, w, ag.x);
  ag.y = __fmaf_rn(acc.y, w, ag.y);
  ag.z = __fmaf_rn(acc.z, w, ag.z);
  ag.w = __fmaf_rn(acc.w, w, ag.w);
}

__device__ __forceinline__ void add_group(float &lt, float4 &at, float lg, const float4 &ag) {
  lt = __fadd_rn(lt, lg);
  at.x = __fadd_rn(at.x, ag.x);
  at.y = __fadd_rn(at.y, ag.y);
  at.z = __fadd_rn(at.z, ag.z);
  at.w = __fadd_rn(at.w, ag.w);
}

template <int D>
__device__ __forceinline__ void store_merged(const StepArgs &a, int row, int h, int col, float lt, const float4 &at) {
  const float inv = 1.f / lt;
  uint2 packed;
  packed.x = pack_bf16x2(__fmul_rn(at.x, inv), __fmul_rn(at.y, inv));
  packed.y = pack_bf16x2(__fmul_rn(at.z, inv), __fmul_rn(at.w, inv));
  *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(a.out) +
                             (static_cast<size_t>(row) * a.num_q_heads + h) * D + 4 * col) = packed;
}

// Four lanes per float4 column: lane w of a column folds groups w, w + 4,
// ...; the column's maximum and its ordered group sums go across the four
// lanes by shuffles. 128 threads hold D / 4 columns x 4 lanes of 128 / D q heads.
template <int D>
__device__ __forceinline__ void merge_small_body(const StepArgs &a, const int32_t *__restrict__ items, int item,
                                                 int head_group) {
  constexpr int F = D / 4;             // float4 columns per q head
  constexpr int WPH = F / 8;           // warps per q head (8 columns per warp)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = head_group * (kMergeThreads / (4 * F)) + warp / WPH;
  const int col = (warp % WPH) * 8 + (lane >> 2), w = lane & 3;
  // The work item and step metadata are final when this grid starts (the
  // decode kernel starts only after everything before the cache write has
  // finished); only the partials need the decode grid to finish (the wait below).
  const MergeRow r = merge_row(a, items, item);
  grid_dependency_wait();  // partials come from the decode kernel
  if (r.bad) {
    if (threadIdx.x == 0 && a.status) atomicOr(a.status, PKV_DEV_BAD_SEGMENT);
    return;
  }
  if (h >= a.num_q_heads) return;  // whole warps
  const int hq = a.num_q_heads;
  const uint32_t stride = static_cast<uint32_t>(r.nrows) * hq;  // entries between spans
  const size_t e0 = static_cast<size_t>(r.pbase) * hq + h;
  const float2 *ml = reinterpret_cast<const float2 *>(a.partial_ml) + e0;
  const float4 *acc = reinterpret_cast<const float4 *>(a.partial_acc + e0 * D) + col;
  const int groups = (r.spans + kGroup - 1) / kGroup, rounds = (groups + 3) / 4;

  float mi[kGroup], li[kGroup];
  float4 ai[kGroup];
  auto load_group = [&](int g) {
#pragma unroll
    for (int k = 0; k < kGroup; ++k) {
      const int i = g * kGroup + k;
      mi[k] = -INFINITY;
      li[k] = 0.f;
      if (i < r.spans) {
        const float2 v = __ldg(ml + static_cast<size_t>(static_cast<uint32_t>(i) * stride));
        mi[k] = v.x;
        li[k] = v.y;
        ai[k] = __ldg(acc + static_cast<size_t>(static_cast<uint32_t>(i) * stride) * F);
      }
    }
  };
  float M = -INFINITY;
  if (rounds == 1) {
    load_group(w);
#pragma unroll
    for (int k = 0; k < kGroup; ++k) M = fmaxf(M, mi[k]);
  } else {
    for (int g = w; g < groups; g += 4)
#pragma unroll
      for (int k = 0; k < kGroup; ++k) {
        const int i = g * kGroup + k;
        if (i < r.spans) M = fmaxf(M, __ldg(ml + static_cast<size_t>(static_cast<uint32_t>(i) * stride)).x);
      }
  }
  M = fmaxf(M, __shfl_xor_sync(kFull, M, 1));
  M = fmaxf(M, __shfl_xor_sync(kFull, M, 2));

  float lt = 0.f;
  float4 at = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int rd = 0; rd < rounds; ++rd) {
    const int g = rd * 4 + w;
    if (rounds > 1) load_group(g);
    float lg = 0.f;
    float4 ag = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kGroup; ++k)
      if (g * kGroup + k < r.spans) fold_span(lg, ag, li[k], ai[k], span_weight(mi[k], M));
    // groups 4 rd .. 4 rd + 3 in order, from the four lanes of this column
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int src = (lane & ~3) | j;
      const float lj = __shfl_sync(kFull, lg, src);
      float4 aj;
      aj.x = __shfl_sync(kFull, ag.x, src);
      aj.y = __shfl_sync(kFull, ag.y, src);
      aj.z = __shfl_sync(kFull, ag.z, src);
      aj.w = __shfl_sync(kFull, ag.w, src);
      if (rd * 4 + j < groups) add_group(lt, at, lj, aj);
    }
  }
  if (w == 0) store_merged<D>(a, r.row, h, col, lt, at);
}

// One-dimensional grids, item-major: every head group of the first (longest)
// rows is issued before any CTA of a later row.
template <int D>
__global__ void __launch_bounds__(kMergeThreads) merge_small_kernel(const StepArgs a,
                                                                    const int32_t *__restrict__ items, int groups) {
  merge_small_body<D>(a, items, static_cast<int>(blockIdx.x) / groups, static_cast<int>(blockIdx.x) % groups);
}

// One thread per float4 column; 128 threads hold 128 / (D / 4) q heads. The
// CTA stages its heads' (max, denominator) pairs kPiece spans at a time in
// shared memory; each thread reads the maxima from there, then folds its
// groups in order, each group's eight sums loaded at once.
template <int D>
__device__ __forceinline__ void merge_wide_body(const StepArgs &a, const int32_t *__restrict__ items, int item,
                                                int head_group) {
  constexpr int F = D / 4;                // float4 columns per q head
  constexpr int HPC = kMergeThreads / F;  // q heads per CTA
  __shared__ float s_m[HPC][kPiece], s_l[HPC][kPiece];
  const int hl = static_cast<int>(threadIdx.x) / F, col = threadIdx.x % F;
  const int h0 = head_group * HPC, h = h0 + hl;
  const MergeRow r = merge_row(a, items, item);
  grid_dependency_wait();  // partials come from the decode kernel
  if (r.bad) {  // uniform over the CTA
    if (threadIdx.x == 0 && a.status) atomicOr(a.status, PKV_DEV_BAD_SEGMENT);
    return;
  }
  const int hq = a.num_q_heads;
  const bool live = h < hq;
  const uint32_t stride = static_cast<uint32_t>(r.nrows) * hq;
  const float2 *ml = reinterpret_cast<const float2 *>(a.partial_ml) + static_cast<size_t>(r.pbase) * hq;
  const float4 *acc =
      reinterpret_cast<const float4 *>(a.partial_acc + (static_cast<size_t>(r.pbase) * hq + (live ? h : 0)) * D) +
      col;
  const int spans = r.spans;

  float4 ai[kGroup];
  auto load_sums = [&](int g) {
#pragma unroll
    for (int k = 0; k < kGroup; ++k) {
      const int i = g * kGroup + k;
      if (live && i < spans) ai[k] = __ldg(acc + static_cast<size_t>(static_cast<uint32_t>(i) * stride) * F);
    }
  };
  auto stage = [&](int p0, int n) {  // (max, denominator) of spans p0 .. p0 + n - 1 of the CTA's heads
    __syncthreads();
    for (int idx = threadIdx.x; idx < HPC * n; idx += kMergeThreads) {
      const int hh = idx / n, i = idx % n;
      float2 v = make_float2(-INFINITY, 0.f);
      if (h0 + hh < hq) v = __ldg(ml + static_cast<size_t>(static_cast<uint32_t>(p0 + i) * stride) + h0 + hh);
      s_m[hh][i] = v.x;
      s_l[hh][i] = v.y;
    }
    __syncthreads();
  };
  load_sums(0);  // the first group's sums do not depend on the maxima
  float M = -INFINITY;
  for (int p0 = 0; p0 < spans; p0 += kPiece) {
    const int n = min(kPiece, spans - p0);
    stage(p0, n);
    for (int i = 0; i < n; ++i) M = fmaxf(M, s_m[hl][i]);
  }
  float lt = 0.f;
  float4 at = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int p0 = 0; p0 < spans; p0 += kPiece) {
    const int n = min(kPiece, spans - p0);
    if (spans > kPiece) stage(p0, n);  // otherwise still staged from the max pass
    for (int c0 = 0; c0 < n; c0 += kGroup) {
      const int g = (p0 + c0) / kGroup;
      if (g > 0) load_sums(g);
      float lg = 0.f;
      float4 ag = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < kGroup; ++k)
        if (c0 + k < n) fold_span(lg, ag, s_l[hl][c0 + k], ai[k], span_weight(s_m[hl][c0 + k], M));
      add_group(lt, at, lg, ag);
    }
  }
  if (live) store_merged<D>(a, r.row, h, col, lt, at);
}

template <int D>
__global__ void __launch_bounds__(kMergeThreads) merge_wide_kernel(const StepArgs a,
                                                                   const int32_t *__restrict__ items, int groups) {
  merge_wide_body<D>(a, items, static_cast<int>(blockIdx.x) / groups, static_cast<int>(blockIdx.x) % groups);
}

// Both layouts in one grid: the first `num_long` items (rows of more than two
// span groups, first in the list) take four lanes per column, the rest one;
// the grid's first long_ctas CTAs are the long items' (item, head group)s.
template <int D>
__global__ void __launch_bounds__(kMergeThreads) merge_mixed_kernel(const StepArgs a,
                                                                    const int32_t *__restrict__ items,
                                                                    int num_long, int long_groups, int wide_groups) {
  const int b = static_cast<int>(blockIdx.x), long_ctas = num_long * long_groups;
  if (b < long_ctas)
    merge_small_body<D>(a, items, b / long_groups, b % long_groups);
  else
    merge_wide_body<D>(a, items, num_long + (b - long_ctas) / wide_groups, (b - long_ctas) % wide_groups);
}

int sm_count() {
  static int count[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    count[dev] = n;
  }
  return count[dev];
}

template <int D, int NT, bool MULTI, int NW = kWarps, int NS = 0>
cudaError_t launch_decode_t(const StepArgs &a, const CUtensorMap &tk, const CUtensorMap &tv, int32_t num_items,
                            const int32_t *items, cudaStream_t stream) {
  constexpr int smem = DecodeCfg<D, NW, NS>::kSmem;
  static std::atomic<uint64_t> configured{0};  // one bit per device
  if (const cudaError_t e = allow_smem_once(decode_kernel<D, NT, MULTI, NW, NS>, smem, configured);
      e != cudaSuccess)
    return e;
  const int64_t tasks = static_cast<int64_t>(num_items) * a.num_kv_heads;
  const int grid = static_cast<int>(tasks < sm_count() ? tasks : sm_count());
  // Past three static rounds, warps take tasks from the workspace counter, so
  // SMs that stream faster take more and all finish together.
  StepArgs b = a;
  if (b.task_counter && tasks > 3ll * grid * NW) {
    const cudaError_t e = cudaMemsetAsync(b.task_counter, 0, sizeof(uint32_t), stream);
    if (e != cudaSuccess) return e;
  } else {
    b.task_counter = nullptr;
  }
  return launch_pdl(decode_kernel<D, NT, MULTI, NW, NS>, dim3(grid), dim3(NW * 32), smem, stream, tk, tv, b, items,
                    num_items);
}

// Single-row decode at head_dim 128: with at most 4, 5 or 6 tasks per SM,
// 4 warps x 6 stages, 5 x 5 or 6 x 4 (192-200 KiB of rings) keep more bytes
// in flight per busy warp than 8 x 3.
template <int NT>
cudaError_t launch_decode_128(const StepArgs &a, const CUtensorMap &tk, const CUtensorMap &tv, int32_t num_items,
                              const int32_t *items, cudaStream_t stream) {
  const int64_t tasks = static_cast<int64_t>(num_items) * a.num_kv_heads;
  const int64_t per_sm = (tasks + sm_count() - 1) / sm_count();
  if (per_sm <= 4) return launch_decode_t<128, NT, false, 4, 6>(a, tk, tv, num_items, items, stream);
  if (per_sm == 5) return launch_decode_t<128, NT, false, 5, 5>(a, tk, tv, num_items, items, stream);
  if (per_sm == 6) return launch_decode_t<128, NT, false, 6, 4>(a, tk, tv, num_items, items, stream);
  return launch_decode_t<128, NT, false>(a, tk, tv, num_items, items, stream);
}

}  // namespace

cudaError_t launch_decode(const StepArgs &a, const CUtensorMap &tk, const CUtensorMap &tv, int32_t num_items,
                          const int32_t *items, bool beside_chunk, cudaStream_t stream) {
  if (num_items <= 0) return cudaSuccess;
  // one column per (row, q head) of a segment: 8 columns per tile, 16 at most
  const bool multi = a.decode_rows_max > 1;
  const bool wide = a.group * (multi ? a.decode_rows_max : 1) > 8;
  if (beside_chunk && a.head_dim == 128 && !wide) {
    // one 8-column tile (at most ~208 registers): small enough to share an SM with a chunk CTA
    constexpr int W = kDecodeWarpsBesideChunk, S = kDecodeStagesBesideChunk;
    return multi ? launch_decode_t<128, 1, true, W, S>(a, tk, tv, num_items, items, stream)
                 : launch_decode_t<128, 1, false, W, S>(a, tk, tv, num_items, items, stream);
  }
  const int v = (a.head_dim == 128 ? 4 : 0) + (wide ? 2 : 0) + (multi ? 1 : 0);
  switch (v) {
    case 0: return launch_decode_t<64, 1, false>(a, tk, tv, num_items, items, stream);
    case 1: return launch_decode_t<64, 1, true>(a, tk, tv, num_items, items, stream);
    case 2: return launch_decode_t<64, 2, false>(a, tk, tv, num_items, items, stream);
    case 3: return launch_decode_t<64, 2, true>(a, tk, tv, num_items, items, stream);
    case 4: return launch_decode_128<1>(a, tk, tv, num_items, items, stream);
    case 5: return launch_decode_t<128, 1, true>(a, tk, tv, num_items, items, stream);
    case 6: return launch_decode_128<2>(a, tk, tv, num_items, items, stream);
    default: return launch_decode_t<128, 2, true>(a, tk, tv, num_items, items, stream);
  }
}

cudaError_t launch_merge(const StepArgs &a, int32_t num_items, int32_t num_long, const int32_t *items,
                         cudaStream_t stream) {
  if (num_items <= 0) return cudaSuccess;
  const int f = a.head_dim / 4;  // float4 columns per q head
  const dim3 block(kMergeThreads);
  const int small_groups = (a.num_q_heads * 4 * f + kMergeThreads - 1) / kMergeThreads;
  const int wide_groups = (a.num_q_heads * f + kMergeThreads - 1) / kMergeThreads;
  // Four lanes per column while that fits one wave of CTAs (six per SM at
  // their 80 registers), else one, except for the rows of more than
  // kLongMergeSpans spans (first in the list): their group chain would
  // otherwise set the kernel's end.
  const int64_t small_ctas = static_cast<int64_t>(num_items) * small_groups;
  if (small_ctas <= 6ll * sm_count()) {
    const dim3 grid(static_cast<unsigned>(small_ctas));
    if (a.head_dim == 128) return launch_pdl(merge_small_kernel<128>, grid, block, 0, stream, a, items, small_groups);
    return launch_pdl(merge_small_kernel<64>, grid, block, 0, stream, a, items, small_groups);
  }
  if (num_long <= 0) {
    const dim3 grid(static_cast<unsigned>(static_cast<int64_t>(num_items) * wide_groups));
    if (a.head_dim == 128) return launch_pdl(merge_wide_kernel<128>, grid, block, 0, stream, a, items, wide_groups);
    return launch_pdl(merge_wide_kernel<64>, grid, block, 0, stream, a, items, wide_groups);
  }
  const int64_t ctas = static_cast<int64_t>(num_long) * small_groups +
                       static_cast<int64_t>(num_items - num_long) * wide_groups;
  const dim3 grid(static_cast<unsigned>(ctas));
  if (a.head_dim == 128)
    return launch_pdl(merge_mixed_kernel<128>, grid, block, 0, stream, a, items, num_long, small_groups, wide_groups);
  return launch_pdl(merge_mixed_kernel<64>, grid, block, 0, stream, a, items, num_long, small_groups, wide_groups);
}

}  // namespace pkv
