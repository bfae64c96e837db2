// Split-KV decode attention and the span combine.
//
// Lucebox, "Continuous batching: Qwen3.8-27B at 301 tok/s across five
// clients, up to 1.97x llama.cpp", §Paged KV and paged attention: attention
// follows each sequence's block table in logical order over the shared pool.
// mlxcel manual, "Continuous batching", §Paged KV cache and prefix sharing:
// batched paged decode reads blocks in place (a block-table kernel) instead
// of rebuilding a contiguous window every step.
//
// Work: one CTA per (decode segment, key span of PKV_SPLIT_KEYS keys, kv head).
// The span is cut into 16-key sub-tiles; warp w takes sub-tiles w, w+4, ...
// Each warp keeps its own 3-stage ring in shared memory: lane 0 issues two TMA
// boxes (64 columns x 16 rows, 128-byte swizzle) per half of head_dim for K
// and V of the next sub-tile, straight from the pool row the block table
// names. The math is warp-level bf16 MMA (m16n8k16) with fp32 accumulation:
//   S^T[16 keys][8 heads] = K[16 keys][D] * Q^T[D][8 heads]   (GQA group on N)
//   O^T[D][8 heads]      += V^T[D][16 keys] * P^T[16 keys][8 heads]
// with an online softmax per head in the exp2 domain. P^T reaches the B
// operand of the second MMA through an in-register 8x8 transpose (movmatrix).
// The four warps merge in a fixed order; spans merge in span order in the
// combine kernel. Nothing depends on timing or on the other segments, so the
// result is deterministic and independent of batch composition.
//
// Keys past the context in a partially filled block are masked to -inf in S
// and their V values are zeroed in registers, so stale or NaN pool rows never
// reach the output.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kWarps = 4;
constexpr int kStages = 3;

template <int D>
struct DecodeLayout {
  static constexpr int kHalves = D / 64;
  static constexpr int kHalfBytes = kSubKeys * 128;           // 16 rows x 128 B
  static constexpr int kTileBytes = kHalves * kHalfBytes;     // one K (or V) sub-tile
  static constexpr int kStageBytes = 2 * kTileBytes;          // K then V
  static constexpr int kRingBytes = kWarps * kStages * kStageBytes;
};

template <int NT>
__host__ __device__ constexpr int merge_bytes(int d) {
  return kWarps * 8 * NT * d * 4;
}

template <int D, int NT>
constexpr int decode_smem_bytes() {
  constexpr int ring = DecodeLayout<D>::kRingBytes;
  constexpr int merge = merge_bytes<NT>(D);
  constexpr int body = ring > merge ? ring : merge;
  // + barriers + per-warp (m, l) + 1 KiB for manual 1024-byte alignment
  return body + kWarps * kStages * 8 + 2 * kWarps * 8 * NT * 4 + 1024;
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void store_bf16(void *out, size_t idx, float x) {
  reinterpret_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(x);
}

__device__ __forceinline__ float bf16_round(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

template <int D, int NT>
__global__ void __launch_bounds__(128) decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                                     const __grid_constant__ CUtensorMap tmap_v,
                                                     const StepArgs a,
                                                     const int32_t *__restrict__ items) {
  using Lay = DecodeLayout<D>;
  constexpr int KT = D / 16;  // k-steps of QK^T, m-tiles of PV
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  constexpr int kBody = Lay::kRingBytes > merge_bytes<NT>(D) ? Lay::kRingBytes : merge_bytes<NT>(D);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kBody);
  float *red_m = reinterpret_cast<float *>(bars + kWarps * kStages);
  float *red_l = red_m + kWarps * 8 * NT;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.y;
  const int4 it = reinterpret_cast<const int4 *>(items)[blockIdx.x];
  const int seg = it.x, slot = it.y, span = it.z, pbase = it.w;

  // ---- segment metadata (uniform across the CTA) ----
  bool bad = seg < 0 || seg >= a.num_seqs || slot < 0 || slot >= a.max_slots;
  int row0 = 0, L = 0;
  if (!bad) {
    row0 = a.cu_seqlens_q[seg];
    const int n = a.cu_seqlens_q[seg + 1] - row0;
    L = a.context_lens[slot];
    bad = a.seq_slot[seg] != slot || n != 1 || L < 1 ||
          static_cast<int64_t>(L) > static_cast<int64_t>(a.max_blocks_per_slot) * a.block_size ||
          span * PKV_SPLIT_KEYS >= L || row0 < 0 || row0 >= a.total_q;
  }
  if (bad) {
    if (threadIdx.x == 0 && a.status) atomicOr(a.status, PKV_DEV_BAD_SEGMENT);
    return;
  }
  const int key0 = span * PKV_SPLIT_KEYS;
  const int key1 = min(L, key0 + PKV_SPLIT_KEYS);
  const int units = (key1 - key0 + kSubKeys - 1) / kSubKeys;
  const int my_units = units > warp ? (units - warp + kWarps - 1) / kWarps : 0;

  // Lane i holds the physical block of this warp's i-th sub-tile.
  const int32_t *bt_row = a.block_tables + static_cast<int64_t>(slot) * a.max_blocks_per_slot;
  int my_block = 0;
  bool my_ok = true;
  if (lane < my_units) {
    my_block = __ldg(bt_row + (key0 + kSubKeys * (warp + kWarps * lane)) / a.block_size);
    my_ok = my_block >= 0 && my_block < a.num_blocks;
    if (!my_ok && a.status) atomicOr(a.status, PKV_DEV_BAD_BLOCK);
  }

  uint64_t *wbar = bars + warp * kStages;
  uint8_t *wring = smem + warp * kStages * Lay::kStageBytes;
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(wbar + s, 1);
    fence_barrier_init();
  }
  __syncwarp();

  // Q^T fragments (B operand): head = nt*8 + lane/4, d = kk*16 + (lane%4)*2 (+8).
  uint32_t qf[NT][KT][2];
  {
    const uint16_t *qrow = static_cast<const uint16_t *>(a.q) +
                           (static_cast<size_t>(row0) * a.num_q_heads + g * a.group) * D;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int head = nt * 8 + (lane >> 2);
      const uint32_t *qp = reinterpret_cast<const uint32_t *>(qrow + head * D) + (lane & 3);
#pragma unroll
      for (int kk = 0; kk < KT; ++kk) {
        qf[nt][kk][0] = head < a.group ? __ldg(qp + kk * 8) : 0u;
        qf[nt][kk][1] = head < a.group ? __ldg(qp + kk * 8 + 4) : 0u;
      }
    }
  }

  auto issue = [&](int i) {
    const int blk = __shfl_sync(0xffffffffu, my_block, i);
    const bool ok = __shfl_sync(0xffffffffu, my_ok ? 1 : 0, i) != 0;
    if (lane == 0) {
      const int stage = i % kStages;
      uint8_t *dst = wring + stage * Lay::kStageBytes;
      uint64_t *bar = wbar + stage;
      const int key = key0 + kSubKeys * (warp + kWarps * i);
      if (ok) {
        const int row = (blk * a.num_kv_heads + g) * a.block_size + key % a.block_size;
        mbar_arrive_expect_tx(bar, Lay::kStageBytes);
#pragma unroll
        for (int h = 0; h < Lay::kHalves; ++h) {
          tma_load_2d(dst + h * Lay::kHalfBytes, &tmap_k, h * 64, row, bar);
          tma_load_2d(dst + Lay::kTileBytes + h * Lay::kHalfBytes, &tmap_v, h * 64, row, bar);
        }
      } else {
        mbar_arrive(bar);  // nothing to load; the consumer skips this sub-tile
      }
    }
  };

  float m[NT][2], l[NT][2], acc[NT][KT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m[nt][0] = m[nt][1] = -INFINITY;
    l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) acc[nt][mt][0] = acc[nt][mt][1] = acc[nt][mt][2] = acc[nt][mt][3] = 0.f;
  }

  if (lane == 0 && warp == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }
  for (int i = 0; i < my_units && i < kStages; ++i) issue(i);

  bool timed_out = false;
  const float sl2 = a.scale_log2;
  for (int i = 0; i < my_units; ++i) {
    const int stage = i % kStages;
    if (!mbar_wait(wbar + stage, (i / kStages) & 1)) {
      timed_out = true;
      break;
    }
    const bool ok = __shfl_sync(0xffffffffu, my_ok ? 1 : 0, i) != 0;
    const int kbase = key0 + kSubKeys * (warp + kWarps * i);
    const int valid = min(kSubKeys, key1 - kbase);
    if (ok) {
      const uint32_t kaddr = smem_addr(wring + stage * Lay::kStageBytes);
      const uint32_t vaddr = kaddr + Lay::kTileBytes;
      const int j = lane >> 3;

      // S^T = K Q^T : A = K sub-tile rows (keys), 16 columns of d per k-step.
      float s[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
      {
        const int r = (lane & 7) + ((j & 1) << 3);
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) {
          const int chunk = ((kk & 3) << 1) + (j >> 1);
          uint32_t af[4];
          ldmatrix_x4(af, kaddr + (kk >> 2) * Lay::kHalfBytes + r * 128 + ((chunk ^ (r & 7)) << 4));
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(s[nt], af, qf[nt][kk][0], qf[nt][kk][1]);
        }
      }

      // Online softmax; thread holds keys lane/4 (+8) for heads (lane%4)*2 + {0,1}.
      const int ka = lane >> 2, kb = ka + 8;
      uint32_t pb[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const float xa = ka < valid ? s[nt][c] * sl2 : -INFINITY;
          const float xb = kb < valid ? s[nt][c + 2] * sl2 : -INFINITY;
          float mx = fmaxf(xa, xb);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mnew = fmaxf(m[nt][c], mx);
          const float corr = exp2f(m[nt][c] - mnew);
          m[nt][c] = mnew;
          const float pa = bf16_round(exp2f(xa - mnew));
          const float pbv = bf16_round(exp2f(xb - mnew));
          l[nt][c] = l[nt][c] * corr + pa + pbv;
#pragma unroll
          for (int mt = 0; mt < KT; ++mt) {
            acc[nt][mt][c] *= corr;
            acc[nt][mt][c + 2] *= corr;
          }
          s[nt][c] = pa;
          s[nt][c + 2] = pbv;
        }
        pb[nt][0] = movmatrix_trans(pack_bf16x2(s[nt][0], s[nt][1]));
        pb[nt][1] = movmatrix_trans(pack_bf16x2(s[nt][2], s[nt][3]));
      }

      // O^T += V^T P^T : A = V^T via transposed ldmatrix of the V sub-tile.
      const int k0 = (lane & 3) * 2;
      const uint32_t mlo = (k0 < valid ? 0x0000FFFFu : 0u) | (k0 + 1 < valid ? 0xFFFF0000u : 0u);
      const uint32_t mhi = (k0 + 8 < valid ? 0x0000FFFFu : 0u) | (k0 + 9 < valid ? 0xFFFF0000u : 0u);
      const int r = (lane & 7) + ((j >> 1) << 3);
#pragma unroll
      for (int mt = 0; mt < KT; ++mt) {
        const int chunk = ((mt & 3) << 1) + (j & 1);
        uint32_t af[4];
        ldmatrix_x4_trans(af, vaddr + (mt >> 2) * Lay::kHalfBytes + r * 128 + ((chunk ^ (r & 7)) << 4));
        af[0] &= mlo;
        af[1] &= mlo;
        af[2] &= mhi;
        af[3] &= mhi;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc[nt][mt], af, pb[nt][0], pb[nt][1]);
      }
    }
    // Release the stage: order this warp's reads before the next TMA write.
    fence_proxy_async_smem();
    __syncwarp();
    if (i + kStages < my_units) issue(i + kStages);
  }

  const bool any_timeout = __syncthreads_or(timed_out);
  if (any_timeout) {
    if (threadIdx.x == 0 && a.status) atomicOr(a.status, PKV_DEV_TIMEOUT);
    return;
  }

  // Row sums over the 8 lanes that share a head column.
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float v = l[nt][c];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      l[nt][c] = v;
    }

  // ---- merge the four warps (fixed order), reusing the ring as scratch ----
  float *red_acc = reinterpret_cast<float *>(smem);  // [warp][8*NT heads][D]
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int hh = nt * 8 + (lane & 3) * 2 + c;
      if (lane < 4) {
        red_m[warp * 8 * NT + hh] = m[nt][c];
        red_l[warp * 8 * NT + hh] = l[nt][c];
      }
      float *dst = red_acc + (warp * 8 * NT + hh) * D + (lane >> 2);
#pragma unroll
      for (int mt = 0; mt < KT; ++mt) {
        dst[mt * 16] = acc[nt][mt][c];
        dst[mt * 16 + 8] = acc[nt][mt][c + 2];
      }
    }
  __syncthreads();

  const int G = a.group;
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int hh = idx / D, d = idx % D;
    float mmax = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mmax = fmaxf(mmax, red_m[w * 8 * NT + hh]);
    float lsum = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = exp2f(red_m[w * 8 * NT + hh] - mmax);
      lsum += red_l[w * 8 * NT + hh] * f;
      o += red_acc[(w * 8 * NT + hh) * D + d] * f;
    }
    const int head = g * G + hh;
    if (pbase < 0) {
      store_bf16(a.out, (static_cast<size_t>(row0) * a.num_q_heads + head) * D + d, o / lsum);
    } else {
      const size_t pi = static_cast<size_t>(pbase + span) * a.num_q_heads + head;
      a.partial_acc[pi * D + d] = o;
      if (d == 0) {
        a.partial_ml[pi * 2] = mmax;
        a.partial_ml[pi * 2 + 1] = lsum;
      }
    }
  }
}

// One CTA per (segment with several spans, q head); one thread per column.
__global__ void __launch_bounds__(128) combine_kernel(const StepArgs a,
                                                      const int32_t *__restrict__ items) {
  const int4 it = reinterpret_cast<const int4 *>(items)[blockIdx.x];
  const int seg = it.x, slot = it.y, spans = it.z, pbase = it.w;
  const int h = blockIdx.y, d = threadIdx.x;
  const int D = a.head_dim;
  bool bad = seg < 0 || seg >= a.num_seqs || slot < 0 || slot >= a.max_slots || spans < 1;
  int row0 = 0;
  if (!bad) {
    row0 = a.cu_seqlens_q[seg];
    bad = a.seq_slot[seg] != slot || a.cu_seqlens_q[seg + 1] - row0 != 1 || row0 >= a.total_q;
  }
  if (bad) {
    if (threadIdx.x == 0 && a.status) atomicOr(a.status, PKV_DEV_BAD_SEGMENT);
    return;
  }
  if (d >= D) return;
  const size_t base = static_cast<size_t>(pbase) * a.num_q_heads + h;
  float mmax = -INFINITY;
  for (int i = 0; i < spans; ++i)
    mmax = fmaxf(mmax, a.partial_ml[(base + static_cast<size_t>(i) * a.num_q_heads) * 2]);
  float lsum = 0.f, o = 0.f;
  for (int i = 0; i < spans; ++i) {
    const size_t pi = base + static_cast<size_t>(i) * a.num_q_heads;
    const float f = exp2f(a.partial_ml[pi * 2] - mmax);
    lsum += a.partial_ml[pi * 2 + 1] * f;
    o += a.partial_acc[pi * D + d] * f;
  }
  store_bf16(a.out, (static_cast<size_t>(row0) * a.num_q_heads + h) * D + d, o / lsum);
}

template <int D, int NT>
cudaError_t launch_decode_t(const StepArgs &a, const CUtensorMap &tk, const CUtensorMap &tv,
                            int32_t num_items, const int32_t *items, cudaStream_t stream) {
  constexpr int smem = decode_smem_bytes<D, NT>();
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, NT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(static_cast<unsigned>(num_items), static_cast<unsigned>(a.num_kv_heads));
  decode_kernel<D, NT><<<grid, 128, smem, stream>>>(tk, tv, a, items);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const StepArgs &a, const CUtensorMap &tk, const CUtensorMap &tv,
                          int32_t num_items, const int32_t *items, cudaStream_t stream) {
  if (num_items <= 0) return cudaSuccess;
  const bool wide = a.group > 8;
  if (a.head_dim == 128)
    return wide ? launch_decode_t<128, 2>(a, tk, tv, num_items, items, stream)
                : launch_decode_t<128, 1>(a, tk, tv, num_items, items, stream);
  return wide ? launch_decode_t<64, 2>(a, tk, tv, num_items, items, stream)
              : launch_decode_t<64, 1>(a, tk, tv, num_items, items, stream);
}

cudaError_t launch_combine(const StepArgs &a, int32_t num_items, const int32_t *items,
                           cudaStream_t stream) {
  if (num_items <= 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>(num_items), static_cast<unsigned>(a.num_q_heads));
  combine_kernel<<<grid, 128, 0, stream>>>(a, items);
  return cudaGetLastError();
}

}  // namespace pkv
