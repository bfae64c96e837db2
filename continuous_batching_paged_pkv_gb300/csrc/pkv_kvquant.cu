// Block-scaled KV pools (8-bit codes; 4-bit codes at head_dim 128): the
// quantising cache write, split-KV decode attention straight from the codes,
// and the widening of prompt-chunk histories into a bf16 scratch pool for the
// tensor-core chunk kernel. Every kernel is templated on the code width.
//
// Lucebox, "Continuous batching: Qwen3.8-27B at 301 tok/s across five
// clients, up to 1.97x llama.cpp", §Qwen3.8-27B DFlash2 on the R9700 (vs
// llama.cpp) and §DeepSeek V4 Flash on Strix Halo and two GPUs: the pages
// serve from 8-bit and 4-bit KV caches without defining the formats. This
// library's 8-bit format: every pool row (token, kv head) is cut into groups
// of 32 values; a group keeps one power-of-two scale d, the smallest at or
// above amax / 127 (at least 2^-126), stored as a bfloat16 (exact), and 32
// int8 codes round_half_even(x / d) clamped to [-127, 127]. The power-of-two
// ceiling is this library's own rule: x / d is exact and every code * d is a
// bfloat16 number, so widening codes to bf16 loses nothing; the price is up to
// one bit at the group maximum, whose code lands in [64, 127] rather than at
// 127. Codes live in [num_blocks][Hkv][bs][D] int8, scales in
// [num_blocks][Hkv][bs][D / 32] bf16: a row costs D + D / 16 bytes instead of
// 2 D, so decode reads 53% of the bf16 pool's bytes. The 4-bit format keeps
// the groups and the scale rule with 7 in place of 127 and stores the codes as
// two's complement nibbles, two per byte, the even value in the low nibble
// ([num_blocks][Hkv][bs][D / 2] bytes): a row costs D / 2 + D / 16 bytes.
//
// Decode kernel (same task pipeline as the bf16 decode kernel: persistent
// warps, a TMA ring per warp, work sorted longest first). Per 16-key sub-tile
// a stage holds the K and V codes (TMA, swizzled like the bf16 tiles) and
// their scales (one bulk copy each). Both products are fp16 MMAs over offset
// codes: an 8-bit code c enters as the fp16 integer 1152 + c (its byte XOR
// 0x80 placed under the exponent of 1024.0), a 4-bit code as 1032 + c (its
// nibble XOR 8), one or two integer instructions per pair of codes and no
// float subtraction. The offsets come out in fp32:
//   S^T = K Q^T: the accumulator of each scale group starts at -offset times
//   the sum of that group's query values, so it ends at the group's partial
//   dot product; the group scales then fold the partial sums into a logit. Q
//   is widened to fp16 after a power-of-two rescale per column (max |q'| <
//   2^15), undone in the softmax scale, so fp16's range never clips a query.
//   O^T += V^T P'^T with P' = 2^7 p dv / Dref: p the softmax weight (at most
//   2^8 under the lazy rescale), dv the key's V scale of the group and Dref
//   the largest V scale the task has met in that group (a running maximum;
//   the group's accumulators are rescaled when it grows), so P' < 2^15 fits
//   fp16. After each m-tile's MMA a second one with A = -offset (each row's
//   own offset) and the same P' subtracts offset times the sub-tile's P' sums,
//   so the accumulator never carries more than one sub-tile's offset; the
//   task's end multiplies by Dref (the 2^7 cancels against the row sum, which
//   adds the same scaled weights).
// head_dim is permuted inside each tile so that every thread reads whole
// words of codes: the permutation is undone in the output address, and for
// 4-bit K by loading q in the same order (a thread's K word holds dims
// 32 g + 8 j .. + 7, paired (0, 4), (1, 5), (2, 6), (3, 7) in the MMA).
// 4-bit codes in odd nibbles are placed without a shift as 1152 + 16 c: for
// K the matching q values are taken at 1/16 (exact), for V the offset MMA
// takes 1152 on those rows and the output takes 1/16 of them.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "pkv_decode_task.cuh"
#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kWarpsQuant = 8;
constexpr uint32_t kAll = 0xffffffffu;
constexpr float kRescaleQuant = 8.0f;  // log2 units, as in the bf16 decode kernel

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// ---- quantising cache write ---------------------------------------------------

// One warp per (k or v, token, kv head) row; lane l holds D/32 consecutive
// values, so one scale group spans 1024/D lanes. BITS = 8: one code per byte;
// BITS = 4: codes in [-7, 7], two per byte, the even value in the low nibble.
template <int D, int BITS>
__global__ void __launch_bounds__(256) cache_write_quant_kernel(
    const __nv_bfloat16 *__restrict__ k_new, const __nv_bfloat16 *__restrict__ v_new,
    const int64_t *__restrict__ slot_mapping, int64_t num_tokens, int8_t *__restrict__ k_codes,
    __nv_bfloat16 *__restrict__ k_scales, int8_t *__restrict__ v_codes, __nv_bfloat16 *__restrict__ v_scales,
    int64_t pool_rows, int32_t block_size, int32_t num_kv_heads, uint32_t *__restrict__ status) {
  grid_dependency_wait();
  launch_dependents();  // as the bf16 cache write: everything before this kernel has finished
  constexpr int VPL = D / 32;       // values per lane
  constexpr int LPG = 32 / VPL;     // lanes per scale group
  const int lane = threadIdx.x & 31;
  const int64_t per_tensor = num_tokens * num_kv_heads;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32; w < 2 * per_tensor;
       w += warps) {
    const bool is_v = w >= per_tensor;
    const int64_t th = is_v ? w - per_tensor : w;
    const int64_t t = th / num_kv_heads, h = th % num_kv_heads;
    const int64_t s = __ldg(slot_mapping + t);
    if (s < 0) continue;
    if (s >= pool_rows) {
      if (status && lane == 0 && h == 0 && !is_v) atomicOr(status, PKV_DEV_BAD_SLOT_MAPPING);
      continue;
    }
    const __nv_bfloat16 *src = (is_v ? v_new : k_new) + th * D + lane * VPL;
    float x[VPL];
    if constexpr (VPL == 4) {
      const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(src));
      x[0] = bf16_bits_to_float(raw.x & 0xFFFFu);
      x[1] = bf16_bits_to_float(raw.x >> 16);
      x[2] = bf16_bits_to_float(raw.y & 0xFFFFu);
      x[3] = bf16_bits_to_float(raw.y >> 16);
    } else {
      const uint32_t raw = __ldg(reinterpret_cast<const uint32_t *>(src));
      x[0] = bf16_bits_to_float(raw & 0xFFFFu);
      x[1] = bf16_bits_to_float(raw >> 16);
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int o = 1; o < LPG; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kAll, amax, o));
    // d: the smallest power of two >= amax / Q (float32 quotient), at least 2^-126
    constexpr float Q = BITS == 8 ? 127.f : 7.f;
    const uint32_t tb = __float_as_uint(__fdiv_rn(amax, Q));
    const uint32_t te = tb & 0x7F800000u;
    uint32_t db = (tb & 0x007FFFFFu) == 0 ? tb : te + 0x00800000u;
    if (te == 0) db = 0x00800000u;
    if (tb == 0) db = 0;
    const float d = __uint_as_float(db);
    const __nv_bfloat16 dq = __ushort_as_bfloat16(static_cast<unsigned short>(db >> 16));
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      float c = d > 0.f ? rintf(__fdiv_rn(x[i], d)) : 0.f;
      c = fminf(fmaxf(c, -Q), Q);
      packed |= (static_cast<uint32_t>(static_cast<int32_t>(c)) & ((1u << BITS) - 1)) << (BITS * i);
    }
    const int64_t blk = s / block_size, row = s % block_size;
    const int64_t prow = (blk * num_kv_heads + h) * block_size + row;
    int8_t *dst = (is_v ? v_codes : k_codes) + (prow * D + lane * VPL) * BITS / 8;
    if constexpr (VPL * BITS == 32)
      *reinterpret_cast<uint32_t *>(dst) = packed;
    else if constexpr (VPL * BITS == 16)
      *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(packed);
    else
      *reinterpret_cast<uint8_t *>(dst) = static_cast<uint8_t>(packed);
    if (lane % LPG == 0) (is_v ? v_scales : k_scales)[prow * (D / 32) + lane / LPG] = dq;
  }
}

// ---- prompt-chunk histories widened into a bf16 scratch pool ------------------

// Item (segment, slot, first scratch block, blocks). CTA (item, y) widens the
// item's logical blocks y, y + gridDim.y, ... : block j of the slot becomes
// scratch block first + j, and the scratch table row of the slot points there.
template <int D, int BITS>
__global__ void __launch_bounds__(256) widen_quant_kernel(const StepArgs a, const int32_t *__restrict__ items,
                                                       const int8_t *__restrict__ k_codes,
                                                       const __nv_bfloat16 *__restrict__ k_scales,
                                                       const int8_t *__restrict__ v_codes,
                                                       const __nv_bfloat16 *__restrict__ v_scales,
                                                       __nv_bfloat16 *__restrict__ k_out,
                                                       __nv_bfloat16 *__restrict__ v_out,
                                                       int32_t *__restrict__ scratch_table, int64_t scratch_blocks) {
  const int4 it = __ldg(reinterpret_cast<const int4 *>(items) + blockIdx.x);
  const int seg = it.x, slot = it.y, first = it.z, nblk = it.w;
  bool ok = seg >= 0 && seg < a.num_seqs && slot >= 0 && slot < a.max_slots && first >= 0 && nblk >= 1 &&
            static_cast<int64_t>(first) + nblk <= scratch_blocks && nblk <= a.max_blocks_per_slot;
  if (ok) {
    const int L = __ldg(a.context_lens + slot);
    ok = __ldg(a.seq_slot + seg) == slot && (L + a.block_size - 1) / a.block_size == nblk;
  }
  grid_dependency_wait();  // the codes come from the cache write before this kernel
  launch_dependents();
  if (!ok) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && a.status) atomicOr(a.status, PKV_DEV_BAD_SEGMENT);
    return;
  }
  constexpr int NG = D / 32;
  const int64_t rows = static_cast<int64_t>(a.num_kv_heads) * a.block_size;  // rows of one block
  const int64_t vecs = rows * (D / 8);                                      // 8 values per vector
  for (int j = blockIdx.y; j < nblk; j += gridDim.y) {
    const int bid = __ldg(a.block_tables + static_cast<int64_t>(slot) * a.max_blocks_per_slot + j);
    const bool in_pool = bid >= 0 && bid < a.num_blocks;
    if (!in_pool && threadIdx.x == 0 && a.status) atomicOr(a.status, PKV_DEV_BAD_BLOCK);
    if (threadIdx.x == 0) scratch_table[static_cast<int64_t>(slot) * a.max_blocks_per_slot + j] = first + j;
    const int64_t src_row0 = static_cast<int64_t>(in_pool ? bid : 0) * rows;
    const int64_t dst_row0 = static_cast<int64_t>(first + j) * rows;
    for (int64_t i = threadIdx.x; i < 2 * vecs; i += blockDim.x) {
      const bool is_v = i >= vecs;
      const int64_t e = is_v ? i - vecs : i;
      const int64_t r = e / (D / 8), c8 = e % (D / 8);
      uint4 outv = make_uint4(0, 0, 0, 0);
      if (in_pool) {
        const int8_t *codes = (is_v ? v_codes : k_codes) + ((src_row0 + r) * D + c8 * 8) * BITS / 8;
        const __nv_bfloat16 *sc = (is_v ? v_scales : k_scales) + (src_row0 + r) * NG + (c8 * 8) / 32;
        const float d = __bfloat162float(*sc);
        uint32_t w[4];
        if constexpr (BITS == 8) {
          const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(codes));
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t word = q < 2 ? raw.x : raw.y;
            const int b0 = (q & 1) * 2;
            const float lo = static_cast<float>(static_cast<int8_t>((word >> (8 * b0)) & 0xFF)) * d;
            const float hi = static_cast<float>(static_cast<int8_t>((word >> (8 * (b0 + 1))) & 0xFF)) * d;
            w[q] = pack_bf16x2(lo, hi);
          }
        } else {  // eight nibbles, value 2q in the low nibble of byte q; sign-extended by shifts
          const uint32_t raw = __ldg(reinterpret_cast<const uint32_t *>(codes));
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float lo = static_cast<float>(static_cast<int32_t>(raw << (28 - 8 * q)) >> 28) * d;
            const float hi = static_cast<float>(static_cast<int32_t>(raw << (24 - 8 * q)) >> 28) * d;
            w[q] = pack_bf16x2(lo, hi);
          }
        }
        outv = make_uint4(w[0], w[1], w[2], w[3]);
      }
      *reinterpret_cast<uint4 *>((is_v ? v_out : k_out) + (dst_row0 + r) * D + c8 * 8) = outv;
    }
  }
}

// ---- split-KV decode over the codes ---------------------------------------------

// NW warps per CTA (the ring depth follows from the shared memory they share).
template <int D, int NW, int BITS>
struct QuantCfg {
  static constexpr int kGroups = D / 32;
  static constexpr int kCodeBytes = kSubKeys * D * BITS / 8;   // K (or V) codes of one sub-tile
  static constexpr int kScaleBytes = kSubKeys * kGroups * 2;   // their scales
  static constexpr int kRowBytes = D * BITS / 8;               // one key's codes (128 or 64 bytes)
  static constexpr int kStages = (D * BITS == 1024 ? 48 : 96) / NW;  // 6 or 12 at eight warps
  static constexpr int kVc = kStages * kCodeBytes;             // offsets inside a warp's ring
  static constexpr int kKs = 2 * kStages * kCodeBytes;
  static constexpr int kVs = kKs + kStages * kScaleBytes;
  static constexpr int kWarpRing = ((kVs + kStages * kScaleBytes) + 1023) / 1024 * 1024;
  static constexpr int kStageTx = 2 * kCodeBytes + 2 * kScaleBytes;
  static constexpr int kSmem = NW * kWarpRing + NW * kStages * 8 + 1024;
  static_assert(kSmem <= 232448, "decode ring exceeds shared memory");
};

// Byte (row, col) of a swizzled sub-tile of codes: 128-byte rows with the
// 128-byte swizzle (D = 128) or 64-byte rows with the 64-byte swizzle (D = 64).
template <int D>
__device__ __forceinline__ uint32_t code_off(int row, int col) {
  if constexpr (D == 128)
    return row * 128 + ((((col >> 4) ^ (row & 7))) << 4) + (col & 15);
  else
    return row * 64 + ((((col >> 4) ^ ((row >> 1) & 3))) << 4) + (col & 15);
}

// Offset under which a code enters the fp16 MMAs: 1152 + c (8-bit), 1032 + c (4-bit).
template <int BITS>
constexpr float kCodeOffset = BITS == 8 ? 1152.f : 1032.f;

// Four 8-bit codes (a word, two's complement) -> two fp16 pairs of 1152 + code:
// lo holds codes 0 and 1, hi codes 2 and 3.
__device__ __forceinline__ void codes_to_f16_off(uint32_t w, uint32_t &lo, uint32_t &hi) {
  const uint32_t u = w ^ 0x80808080u;  // offset by 128
  lo = prmt(u, 0x64646464u, 0x4140u);   // under the exponent of 1024.0
  hi = prmt(u, 0x64646464u, 0x4342u);
}

// Byte J of word x and of word y (8-bit codes) -> the fp16 pair (1152 + x_J, 1152 + y_J).
template <int J>
__device__ __forceinline__ uint32_t code_pair_f16_off(uint32_t x, uint32_t y) {
  constexpr uint32_t sel = J | (J << 4) | ((4 + J) << 8) | ((4 + J) << 12);
  return (prmt(x, y, sel) & 0x00FF00FFu) ^ 0x64806480u;
}

// Nibble 0 of both 16-bit halves of x (4-bit codes) -> the fp16 pair of 1032 + code.
__device__ __forceinline__ uint32_t nibble_lo_f16_off(uint32_t x) { return (x & 0x000F000Fu) ^ 0x64086408u; }

// Nibble 1 of both 16-bit halves of x -> the fp16 pair of 1152 + 16 code (the
// nibble, XOR 8, lands in mantissa bits 4..7 under the exponent of 1024.0).
__device__ __forceinline__ uint32_t nibble_hi_f16_off(uint32_t x) { return (x & 0x00F000F0u) ^ 0x64806480u; }

// Scale of group g from bf16 pairs packed two per word, as fp32.
template <int G2>
__device__ __forceinline__ float group_scale(const uint32_t (&w)[G2], int g) {
  return __uint_as_float((g & 1) ? (w[g >> 1] & 0xFFFF0000u) : (w[g >> 1] << 16));
}

// Q'^T fragments (B operand, fp16) for k-step kk = 2 g + h: thread (column
// lane/4, j = lane%4) holds, for 8-bit codes, q[column][32 g + 16 h + 4 j +
// 0..3] ((0, 1) in the first register, (2, 3) in the second); for 4-bit codes,
// with p = 32 g + 8 j, (p + 2 h, p + 2 h + 4) and (p + 2 h + 1, p + 2 h + 5),
// the pairs the nibble words give. Scaled by 2^sh (per column) so that
// max |q'| < 2^15; `inv` receives 2^-sh.
template <int D, int NT, bool MULTI, int BITS>
__device__ __forceinline__ void load_q_quant(uint32_t (&qf)[NT][D / 16][2], float (&inv)[NT], const Task &T,
                                          const StepArgs &a, int lane) {
  constexpr int KT = D / 16;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int col = nt * 8 + (lane >> 2);
    const bool valid = col < (MULTI ? T.nrows : 1) * a.group;
    const int i = MULTI && valid ? col / a.group : 0, h = !MULTI ? col : valid ? col % a.group : 0;
    const __nv_bfloat16 *qrow = static_cast<const __nv_bfloat16 *>(a.q) +
                                ((static_cast<size_t>(T.row0) + i) * a.num_q_heads + T.g * a.group + h) * D;
    const int j = lane & 3;
    uint32_t raw[KT][2];  // bf16 pairs in fragment order
    if constexpr (BITS == 8) {
#pragma unroll
      for (int kk = 0; kk < KT; ++kk) {
        const uint2 r = valid ? __ldg(reinterpret_cast<const uint2 *>(qrow + 32 * (kk >> 1) + 16 * (kk & 1) + 4 * j))
                              : make_uint2(0, 0);
        raw[kk][0] = r.x;
        raw[kk][1] = r.y;
      }
    } else {
#pragma unroll
      for (int g = 0; g < KT / 2; ++g) {
        const __nv_bfloat16 *p = qrow + 32 * g + 8 * j;
        const uint2 r0 = valid ? __ldg(reinterpret_cast<const uint2 *>(p)) : make_uint2(0, 0);      // dims 0..3
        const uint2 r1 = valid ? __ldg(reinterpret_cast<const uint2 *>(p + 4)) : make_uint2(0, 0);  // dims 4..7
        raw[2 * g][0] = prmt(r0.x, r1.x, 0x5410u);      // (0, 4)
        raw[2 * g][1] = prmt(r0.x, r1.x, 0x7632u);      // (1, 5)
        raw[2 * g + 1][0] = prmt(r0.y, r1.y, 0x5410u);  // (2, 6)
        raw[2 * g + 1][1] = prmt(r0.y, r1.y, 0x7632u);  // (3, 7)
      }
    }
    float mx = 0.f;
#pragma unroll
    for (int kk = 0; kk < KT; ++kk)
#pragma unroll
      for (int b = 0; b < 2; ++b)
        mx = fmaxf(mx, fmaxf(fabsf(bf16_bits_to_float(raw[kk][b] & 0xFFFFu)), fabsf(bf16_bits_to_float(raw[kk][b] >> 16))));
    mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 2));
    // exponent of mx (its float bits; 0 and subnormals read as -127)
    const int e = static_cast<int>((__float_as_uint(mx) >> 23) & 0xFF) - 127;
    const int sh = mx > 0.f ? min(126, max(-126, 14 - e)) : 0;
    const float f = __uint_as_float(static_cast<uint32_t>(sh + 127) << 23);
    inv[nt] = __uint_as_float(static_cast<uint32_t>(127 - sh) << 23);
#pragma unroll
    for (int kk = 0; kk < KT; ++kk)
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const float fb = BITS == 4 && b == 1 ? f * 0.0625f : f;  // 4-bit odd nibbles enter as 16 c
        __half2 v = __floats2half2_rn(bf16_bits_to_float(raw[kk][b] & 0xFFFFu) * fb,
                                      bf16_bits_to_float(raw[kk][b] >> 16) * fb);
        qf[nt][kk][b] = *reinterpret_cast<uint32_t *>(&v);
      }
  }
}

// The q rows of task T's columns pulled into L1 ahead of load_q_quant (the
// four threads of a column cover its D * 2 bytes).
template <int D, int NT, bool MULTI>
__device__ __forceinline__ void prefetch_q(const Task &T, const StepArgs &a, int lane) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int col = nt * 8 + (lane >> 2);
    if (col < (MULTI ? T.nrows : 1) * a.group) {
      const int i = MULTI ? col / a.group : 0, h = MULTI ? col % a.group : col;
      const char *p = reinterpret_cast<const char *>(static_cast<const __nv_bfloat16 *>(a.q) +
                                                     ((static_cast<size_t>(T.row0) + i) * a.num_q_heads +
                                                      T.g * a.group + h) * D) +
                      (lane & 3) * (D / 2);
      asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
    }
  }
}

// Start value of each scale group's S^T accumulator: -offset times the sum of
// the group's 32 query values (the fp16 values the MMA reads) of columns
// 2 (lane % 4) + c, which removes the code offset from the group's dot product.
template <int D, int NT, int BITS>
__device__ __forceinline__ void key_offsets(float (&kinit)[D / 32][NT][4], const uint32_t (&qf)[NT][D / 16][2],
                                            int lane) {
  const int jq = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int g = 0; g < D / 32; ++g) {
      // first registers of a k-step meet codes at offset kCodeOffset, second
      // ones 1152 (4-bit odd nibbles, whose q values are at 1/16)
      float s = 0.f;
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&qf[nt][2 * g + h][b]));
          s += (b == 0 ? kCodeOffset<BITS> : 1152.f) * (f.x + f.y);
        }
      s += __shfl_xor_sync(kAll, s, 1);  // the four threads of a column hold its 32 values
      s += __shfl_xor_sync(kAll, s, 2);
      // the accumulator layout: (key ka, column 2 jq), (ka, 2 jq + 1), (kb, 2 jq), (kb, 2 jq + 1)
      kinit[g][nt][0] = kinit[g][nt][2] = -__shfl_sync(kAll, s, (2 * jq) * 4);
      kinit[g][nt][1] = kinit[g][nt][3] = -__shfl_sync(kAll, s, (2 * jq + 1) * 4);
    }
}

template <int D, int NT, bool MULTI, int NW, int BITS>
__global__ void __launch_bounds__(NW * 32, 1)
    decode_quant_kernel(const __grid_constant__ CUtensorMap tmap_kc, const __grid_constant__ CUtensorMap tmap_vc,
                     const StepArgs a, const __nv_bfloat16 *__restrict__ k_scales,
                     const __nv_bfloat16 *__restrict__ v_scales, const int32_t *__restrict__ items, int num_items) {
  using Cfg = QuantCfg<D, NW, BITS>;
  static_assert(BITS == 8 || D == 128, "4-bit codes need head_dim 128 (64-byte code rows)");
  constexpr int RB = Cfg::kRowBytes;  // code row layout: 128-byte rows (128B swizzle) or 64-byte (64B)
  constexpr int KT = D / 16;  // k-steps of QK^T, m-tiles of PV
  constexpr int NG = Cfg::kGroups;
  constexpr int NG2 = NG / 2;  // words of packed bf16 scales per key
  constexpr int NST = Cfg::kStages;
  constexpr int kMaxRows = MULTI ? 16 : 1;
  constexpr float kHeadroom = 7.f;  // log2 of the factor that lifts P' towards fp16's top
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t *ring = smem + warp * Cfg::kWarpRing;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + NW * Cfg::kWarpRing) + warp * NST;

  launch_dependents();  // the span merge may launch now; it waits for this grid before reading
  const int hkv = a.num_kv_heads;
  const int num_tasks = num_items * hkv;
  const int stride = gridDim.x * NW;
  const int t0 = warp * gridDim.x + blockIdx.x;
  if (t0 >= num_tasks) return;
  if (lane == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(full + s, 1);
    fence_barrier_init();
    prefetch_tensormap(&tmap_kc);
    prefetch_tensormap(&tmap_vc);
  }
  __syncwarp();
  bool waited = false;  // rows written by the kernel before (this step's) are read after its wait

  // Tasks as in the bf16 decode kernel: three static rounds, then (with a
  // task counter) 3 stride + the counter's next value. A current, B
  // expanded, tC the task whose work item is in rawC.
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
  uint32_t qA[NT][KT][2];
  float invA[NT];
  if (A.ok) load_q_quant<D, NT, MULTI, BITS>(qA, invA, A, a, lane);

  int P = 0, C = 0, pa = 0, pb = 0;
  int pstage = 0;
  // Each history row is read once per step: its L2 lines go first, which keeps
  // the span partials this grid writes in L2 for the merge.
  const uint64_t policy = l2_evict_first_policy();
  auto issue = [&](const Task &T, int u) {
    // only the sub-tiles holding this step's rows wait for the cache write
    if (!waited && T.reads_new && T.key0 + (u + 1) * kSubKeys > T.L - T.nrows) {
      grid_dependency_wait();
      waited = true;
    }
    const int row = __shfl_sync(kAll, T.row, u);
    if (lane == 0) {
      uint64_t *bar = full + pstage;
      if (row >= 0) {
        mbar_arrive_expect_tx(bar, Cfg::kStageTx);
        tma_load_2d_hint(ring + pstage * Cfg::kCodeBytes, &tmap_kc, 0, row, bar, policy);
        tma_load_2d_hint(ring + Cfg::kVc + pstage * Cfg::kCodeBytes, &tmap_vc, 0, row, bar, policy);
        bulk_load(ring + Cfg::kKs + pstage * Cfg::kScaleBytes, k_scales + static_cast<int64_t>(row) * NG,
                  Cfg::kScaleBytes, bar);
        bulk_load(ring + Cfg::kVs + pstage * Cfg::kScaleBytes, v_scales + static_cast<int64_t>(row) * NG,
                  Cfg::kScaleBytes, bar);
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
        if (B.ok) prefetch_q<D, NT, MULTI>(B, a, lane);  // loaded when B becomes current
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

  const uint32_t ring_addr = smem_addr(ring);
  const float sl2 = a.scale_log2;
  const int G = a.group;
  const int ka = lane >> 2, kb = ka + 8, jq = lane & 3, k0 = jq * 2, r = lane >> 2;
  // per-thread code offsets inside a sub-tile (rows kb = ka + 8 and k0 + 8 share the swizzle phase)
  const uint32_t koff = code_off<RB>(ka, 4 * jq);  // + group/half chunk below
  // V codes of group 0 (dims 4 r .. + 3) in rows k0 and k0 + 1; group g XORs g << kGroupShift into the chunk bits
  constexpr int kGroupShift = BITS == 8 ? 5 : 4;  // 32 or 16 bytes of codes per scale group
  const uint32_t voff0 = code_off<RB>(k0, BITS == 8 ? 4 * r : 2 * r);
  const uint32_t voff1 = code_off<RB>(k0 + 1, BITS == 8 ? 4 * r : 2 * r);
  // fp16 pairs of -offset (-1152 or -1032): A of the MMA that takes the code offset out of O^T
  // (rows r + 8 of a 4-bit m-tile hold odd nibbles, at 1152 + 16 c)
  constexpr uint32_t kNegOffLo = BITS == 8 ? 0xE480E480u : 0xE408E408u;
  const uint32_t kNegOff[4] = {kNegOffLo, 0xE480E480u, kNegOffLo, 0xE480E480u};
  int cstage = 0;
  uint32_t cphase = 0;

  while (A.t >= 0) {
    // Claim the task after tC now; the answer is needed only when A is done.
    uint32_t claim = 0;
    if (counter && tC < num_tasks && lane == 0) claim = atomicAdd(counter, 1u);
    float m[NT][2], l[NT][2], acc[NT][KT][4];
    float mr[NT][2], m0h[NT][2];  // per column: m + the lazy margin, and (m, 0 before any key) - headroom
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m[nt][0] = m[nt][1] = -INFINITY;
      mr[nt][0] = mr[nt][1] = -INFINITY;
      m0h[nt][0] = m0h[nt][1] = -kHeadroom;
      l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < KT; ++mt) acc[nt][mt][0] = acc[nt][mt][1] = acc[nt][mt][2] = acc[nt][mt][3] = 0.f;
    }
    // running maximum V scale of each group (packed bf16 bits, 0 before the first) and its reciprocal
    uint32_t vref[NG2];
    float vinv[NG];
#pragma unroll
    for (int i = 0; i < NG2; ++i) vref[i] = 0u;
#pragma unroll
    for (int g = 0; g < NG; ++g) vinv[g] = 0.f;
    float kinit[NG][NT][4];
    key_offsets<D, NT, BITS>(kinit, qA, lane);
    const int nrows = MULTI ? A.nrows : 1;
    uint32_t colrow = 0;
    if (MULTI) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int col = nt * 8 + jq * 2 + c;
          const int i = col < nrows * G ? col / G : nrows - 1;
          colrow |= static_cast<uint32_t>(i & 0xFF) << (8 * (nt * 2 + c));
        }
    }
    // softmax scale of this thread's columns (2 jq + c): scale * log2(e) / 2^sh of the column
    float sl2c[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 2; ++c) sl2c[nt][c] = sl2 * __shfl_sync(kAll, invA[nt], (jq * 2 + c) * 4);

    for (int u = 0; u < A.units; ++u) {
      const int stage = cstage;
      if (!mbar_wait(full + stage, cphase)) {
        if (lane == 0 && a.status) atomicOr(a.status, PKV_DEV_TIMEOUT);
        return;
      }
      const int row = __shfl_sync(kAll, A.row, u);
      const int kbase = A.key0 + u * kSubKeys;
      const int v = row >= 0 ? min(kSubKeys, A.key1 - kbase) : 0;
      const int vis0 = A.L - nrows - kbase + 1;
      // this thread's K words of rows ka (and kb, 8 rows on) at chunk 0; a chunk index is XORed into
      // the swizzled chunk bits (the stage base is a multiple of 128)
      const uint32_t kbase0 = ring_addr + stage * Cfg::kCodeBytes + koff;
      const uint32_t vc = ring_addr + Cfg::kVc + stage * Cfg::kCodeBytes;
      const uint32_t ks = ring_addr + Cfg::kKs + stage * Cfg::kScaleBytes;
      const uint32_t vs = ring_addr + Cfg::kVs + stage * Cfg::kScaleBytes;

      // group scales of keys ka and kb (packed bf16); V scales zero past the sub-tile's keys
      uint32_t kwa[NG2], kwb[NG2], vwa[NG2], vwb[NG2];
      if constexpr (NG == 4) {
        const uint2 x0 = lds64(ks + ka * 8), x1 = lds64(ks + kb * 8);
        const uint2 y0 = lds64(vs + ka * 8), y1 = lds64(vs + kb * 8);
        kwa[0] = x0.x; kwa[1] = x0.y; kwb[0] = x1.x; kwb[1] = x1.y;
        vwa[0] = y0.x; vwa[1] = y0.y; vwb[0] = y1.x; vwb[1] = y1.y;
      } else {
        kwa[0] = lds32(ks + ka * 4); kwb[0] = lds32(ks + kb * 4);
        vwa[0] = lds32(vs + ka * 4); vwb[0] = lds32(vs + kb * 4);
      }
#pragma unroll
      for (int i = 0; i < NG2; ++i) {
        vwa[i] = ka < v ? vwa[i] : 0u;
        vwb[i] = kb < v ? vwb[i] : 0u;
      }

      // S^T = K Q^T per scale group over the offset codes, each group's
      // accumulator starting at -offset * its query sum; the group scales fold
      // the partial sums into the logits of keys ka (0, 1) and kb (2, 3)
      float sacc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        float sg[NT][4];  // the group's first MMA starts from kinit (no copy: kinit lives on)
        if constexpr (BITS == 8) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // chunk 2g + h of rows ka / kb: the swizzle XORs the chunk index
            const int kk = 2 * g + h;
            const uint32_t ka_addr = kbase0 ^ (static_cast<uint32_t>(kk) << 4);
            const uint32_t wa = lds32(ka_addr);
            const uint32_t wb = lds32(ka_addr + 8 * RB);
            uint32_t af[4];
            codes_to_f16_off(wa, af[0], af[2]);
            codes_to_f16_off(wb, af[1], af[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              if (h == 0)
                mma_f16_16816_from(sg[nt], af, qA[nt][kk][0], qA[nt][kk][1], kinit[g][nt][0], kinit[g][nt][1],
                                   kinit[g][nt][2], kinit[g][nt][3]);
              else
                mma_f16_16816(sg[nt], af, qA[nt][kk][0], qA[nt][kk][1]);
            }
          }
        } else {
          // chunk g of rows ka / kb holds dims 32 g .. 32 g + 31; this thread's word holds dims 32 g + 8 jq + 0..7
          const uint32_t ka_addr = kbase0 ^ (static_cast<uint32_t>(g) << 4);
          const uint32_t wa = lds32(ka_addr);
          const uint32_t wb = lds32(ka_addr + 8 * RB);
          const uint32_t wa8 = wa >> 8, wb8 = wb >> 8;  // nibbles 2, 3 (and 6, 7) into place
          const uint32_t a0[4] = {nibble_lo_f16_off(wa), nibble_lo_f16_off(wb), nibble_hi_f16_off(wa),
                                  nibble_hi_f16_off(wb)};
          const uint32_t a1[4] = {nibble_lo_f16_off(wa8), nibble_lo_f16_off(wb8), nibble_hi_f16_off(wa8),
                                  nibble_hi_f16_off(wb8)};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma_f16_16816_from(sg[nt], a0, qA[nt][2 * g][0], qA[nt][2 * g][1], kinit[g][nt][0], kinit[g][nt][1],
                               kinit[g][nt][2], kinit[g][nt][3]);
            mma_f16_16816(sg[nt], a1, qA[nt][2 * g + 1][0], qA[nt][2 * g + 1][1]);
          }
        }
        const float dka = group_scale(kwa, g), dkb = group_scale(kwb, g);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          fma2(sacc[nt][0], sacc[nt][1], dka, dka, sg[nt][0], sg[nt][1], sacc[nt][0], sacc[nt][1]);
          fma2(sacc[nt][2], sacc[nt][3], dkb, dkb, sg[nt][2], sg[nt][3], sacc[nt][2], sacc[nt][3]);
        }
      }

      // online softmax (keys ka, kb of columns 2 jq + c); the warp reduces the
      // column maxima only when some lane's logit passes its column's maximum
      // by the lazy margin
      float x[NT][2][2];
      bool need = false;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int vis = MULTI ? min(v, vis0 + static_cast<int>((colrow >> (8 * (nt * 2 + c))) & 0xFF)) : v;
          x[nt][c][0] = ka < vis ? sacc[nt][c] * sl2c[nt][c] : -INFINITY;
          x[nt][c][1] = kb < vis ? sacc[nt][c + 2] * sl2c[nt][c] : -INFINITY;
          need |= fmaxf(x[nt][c][0], x[nt][c][1]) > mr[nt][c];
        }
      if (__any_sync(kAll, need)) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            float t = fmaxf(x[nt][c][0], x[nt][c][1]);
            t = fmaxf(t, __shfl_xor_sync(kAll, t, 4));
            t = fmaxf(t, __shfl_xor_sync(kAll, t, 8));
            t = fmaxf(t, __shfl_xor_sync(kAll, t, 16));
            if (t > mr[nt][c]) {
              const float corr = ex2_approx(m[nt][c] - t);
              m[nt][c] = t;
              mr[nt][c] = t + kRescaleQuant;
              m0h[nt][c] = t - kHeadroom;
              l[nt][c] *= corr;
#pragma unroll
              for (int mt = 0; mt < KT; ++mt) {
                acc[nt][mt][c] *= corr;
                acc[nt][mt][c + 2] *= corr;
              }
            }
          }
      }

      // Dref: the running maximum V scale per group; a group's accumulators follow it when it grows
      {
        uint32_t vn[NG2], grow = 0;
#pragma unroll
        for (int i = 0; i < NG2; ++i) {
          vn[i] = max_u16x2(max_u16x2(vwa[i], vwb[i]), vref[i]);  // positive bf16: bit order is value order
          grow |= vn[i] ^ vref[i];
        }
        if (__any_sync(kAll, grow != 0)) {
#pragma unroll
          for (int i = 0; i < NG2; ++i)
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) vn[i] = max_u16x2(vn[i], __shfl_xor_sync(kAll, vn[i], o));
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            const float dn = group_scale(vn, g), dold = group_scale(vref, g);
            if (dn != dold) {
              const float inv = __frcp_rn(dn);  // exact: dn is a power of two >= 2^-126
              const float f = dold * inv;       // 0 when the group had no scale yet (its sums are 0)
              vinv[g] = inv;
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  acc[nt][2 * g][e] *= f;
                  acc[nt][2 * g + 1][e] *= f;
                }
            }
          }
#pragma unroll
          for (int i = 0; i < NG2; ++i) vref[i] = vn[i];
        }
      }

      // P' = 2^7 p dv / Dref (fp32), one fp16 copy of P'^T per V scale group
      float ra[NG], rb[NG];
#pragma unroll
      for (int i = 0; i < NG2; ++i) {
        mul2(ra[2 * i], ra[2 * i + 1], group_scale(vwa, 2 * i), group_scale(vwa, 2 * i + 1), vinv[2 * i], vinv[2 * i + 1]);
        mul2(rb[2 * i], rb[2 * i + 1], group_scale(vwb, 2 * i), group_scale(vwb, 2 * i + 1), vinv[2 * i], vinv[2 * i + 1]);
      }
      uint32_t pf[NG][NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float m0 = m0h[nt][0], m1 = m0h[nt][1];
        const float p00 = ex2_approx(x[nt][0][0] - m0), p01 = ex2_approx(x[nt][0][1] - m0);  // column c=0: ka, kb
        const float p10 = ex2_approx(x[nt][1][0] - m1), p11 = ex2_approx(x[nt][1][1] - m1);  // column c=1
        add2(l[nt][0], l[nt][1], p00, p10);
        add2(l[nt][0], l[nt][1], p01, p11);
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          float a0, a1, b0, b1;
          mul2(a0, a1, p00, p10, ra[g], ra[g]);
          mul2(b0, b1, p01, p11, rb[g], rb[g]);
          pf[g][nt][0] = movmatrix_trans(pack_f16x2(a0, a1));
          pf[g][nt][1] = movmatrix_trans(pack_f16x2(b0, b1));
        }
      }

      // O^T += V^T P'^T over the offset codes, then -offset * P' sums; m-tile
      // 2g + h, rows r / r + 8: head_dim 32 g + 4 r + 2 h (+ 1); keys k0, k0 + 1 (+ 8).
      // rows k0 and k0 + 1 of group 0; a group's chunk differs only in the
      // bits the swizzle XORs (the stage base is a multiple of 128), and rows
      // k0 + 8, k0 + 9 sit 8 rows further with the same swizzle phase
      const uint32_t va0 = vc + voff0, va1 = vc + voff1;
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        uint32_t af0[4], af1[4];
        const uint32_t ga0 = va0 ^ (static_cast<uint32_t>(g) << kGroupShift);
        const uint32_t ga1 = va1 ^ (static_cast<uint32_t>(g) << kGroupShift);
        if constexpr (BITS == 8) {
          const uint32_t u0 = lds32(ga0);
          const uint32_t u1 = lds32(ga1);
          const uint32_t u8 = lds32(ga0 + 8 * RB);
          const uint32_t u9 = lds32(ga1 + 8 * RB);
          af0[0] = code_pair_f16_off<0>(u0, u1);
          af0[1] = code_pair_f16_off<1>(u0, u1);
          af0[2] = code_pair_f16_off<0>(u8, u9);
          af0[3] = code_pair_f16_off<1>(u8, u9);
          af1[0] = code_pair_f16_off<2>(u0, u1);
          af1[1] = code_pair_f16_off<3>(u0, u1);
          af1[2] = code_pair_f16_off<2>(u8, u9);
          af1[3] = code_pair_f16_off<3>(u8, u9);
        } else {
          // the four codes of dims 32 g + 4 r .. + 3 of a key are one 16-bit word (byte 16 g + 2 r)
          const uint32_t x01 = lds16(ga0) | (lds16(ga1) << 16);
          const uint32_t x89 = lds16(ga0 + 8 * RB) | (lds16(ga1 + 8 * RB) << 16);
          const uint32_t y01 = x01 >> 8, y89 = x89 >> 8;  // nibbles 2, 3 into place
          af0[0] = nibble_lo_f16_off(x01);
          af0[1] = nibble_hi_f16_off(x01);  // rows r + 8: 16 c
          af0[2] = nibble_lo_f16_off(x89);
          af0[3] = nibble_hi_f16_off(x89);
          af1[0] = nibble_lo_f16_off(y01);
          af1[1] = nibble_hi_f16_off(y01);
          af1[2] = nibble_lo_f16_off(y89);
          af1[3] = nibble_hi_f16_off(y89);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma_f16_16816(acc[nt][2 * g], af0, pf[g][nt][0], pf[g][nt][1]);
          mma_f16_16816(acc[nt][2 * g + 1], af1, pf[g][nt][0], pf[g][nt][1]);
          mma_f16_16816(acc[nt][2 * g], kNegOff, pf[g][nt][0], pf[g][nt][1]);
          mma_f16_16816(acc[nt][2 * g + 1], kNegOff, pf[g][nt][0], pf[g][nt][1]);
        }
      }
      __syncwarp();  // every read of this stage is consumed before the ring refills it
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
          t += __shfl_xor_sync(kAll, t, 4);
          t += __shfl_xor_sync(kAll, t, 8);
          t += __shfl_xor_sync(kAll, t, 16);
          l[nt][c] = t;
        }
      const int hbase = A.g * G;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int col = nt * 8 + jq * 2 + c;
          if (col < nrows * G) {
            const int i = MULTI ? col / G : 0, hh = MULTI ? col % G : col;
            // o = acc * Dref: sum over keys of p dv code, times 2^7
            float o[NG][4];
#pragma unroll
            for (int g = 0; g < NG; ++g) {
              const float d = group_scale(vref, g);
              const float d8 = BITS == 4 ? d * 0.0625f : d;  // rows r + 8 of 4-bit codes carry 16 c
              o[g][0] = acc[nt][2 * g][c] * d;
              o[g][1] = acc[nt][2 * g][c + 2] * d8;
              o[g][2] = acc[nt][2 * g + 1][c] * d;
              o[g][3] = acc[nt][2 * g + 1][c + 2] * d8;
            }
            if (A.pbase < 0) {
              __nv_bfloat16 *out = reinterpret_cast<__nv_bfloat16 *>(a.out) +
                                   ((static_cast<size_t>(A.row0) + i) * a.num_q_heads + hbase + hh) * D + 4 * r;
              const float inv = 1.f / l[nt][c];  // l also carries the 2^7
#pragma unroll
              for (int g = 0; g < NG; ++g) {
                uint2 pk;
                pk.x = pack_bf16x2(o[g][0] * inv, o[g][1] * inv);
                pk.y = pack_bf16x2(o[g][2] * inv, o[g][3] * inv);
                *reinterpret_cast<uint2 *>(out + 32 * g) = pk;
              }
            } else {
              // span partials in the merge's units: sums of p dv code and of p
              constexpr float kDown = 1.f / 128.f;
              const size_t pi = (static_cast<size_t>(A.pbase + A.span * nrows + i) * a.num_q_heads + hbase + hh);
              float *pacc = a.partial_acc + pi * D + 4 * r;
#pragma unroll
              for (int g = 0; g < NG; ++g)
                *reinterpret_cast<float4 *>(pacc + 32 * g) =
                    make_float4(o[g][0] * kDown, o[g][1] * kDown, o[g][2] * kDown, o[g][3] * kDown);
              if (r == 0) {
                a.partial_ml[pi * 2] = m[nt][c];
                a.partial_ml[pi * 2 + 1] = l[nt][c] * kDown;
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
        const uint32_t c = __shfl_sync(kAll, claim, 0);
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
      if (A.ok) load_q_quant<D, NT, MULTI, BITS>(qA, invA, A, a, lane);
    }
    expand(B, next_t < num_tasks ? next_t : -1, rawC, a, lane);
    tC = after;
    if (tC < num_tasks) rawC = load_item(items, tC, hkv);
    while (P - C < NST && issue_next()) {
    }
  }
}

template <int D, int NT, bool MULTI, int NW, int BITS>
cudaError_t launch_decode_quant_w(const StepArgs &a, const CUtensorMap &tk, const CUtensorMap &tv,
                               const void *k_scales, const void *v_scales, int32_t num_items, const int32_t *items,
                               int grid, cudaStream_t stream) {
  constexpr int smem = QuantCfg<D, NW, BITS>::kSmem;
  static std::atomic<uint64_t> configured{0};  // one bit per device
  if (const cudaError_t e = allow_smem_once(decode_quant_kernel<D, NT, MULTI, NW, BITS>, smem, configured);
      e != cudaSuccess)
    return e;
  const int64_t tasks = static_cast<int64_t>(num_items) * a.num_kv_heads;
  StepArgs b = a;  // past three static rounds, tasks come from the workspace counter
  if (b.task_counter && tasks > 3ll * grid * NW) {
    const cudaError_t e = cudaMemsetAsync(b.task_counter, 0, sizeof(uint32_t), stream);
    if (e != cudaSuccess) return e;
  } else {
    b.task_counter = nullptr;
  }
  return launch_pdl(decode_quant_kernel<D, NT, MULTI, NW, BITS>, dim3(grid), dim3(NW * 32), smem, stream, tk, tv, b,
                    static_cast<const __nv_bfloat16 *>(k_scales), static_cast<const __nv_bfloat16 *>(v_scales),
                    items, num_items);
}

// Eight warps (six stages at head_dim 128 with 8-bit codes, twice that with
// 4-bit ones); single-row, single-tile steps with more than three rounds of
// tasks run 12 warps instead: the code conversions make a warp's sub-tile a
// long dependent chain, and more warps per scheduler hide it once every warp
// has work (a small step's few busy warps stream faster through deeper rings).
template <int D, int NT, bool MULTI, int BITS>
cudaError_t launch_decode_quant_t(const StepArgs &a, const CUtensorMap &tk, const CUtensorMap &tv,
                               const void *k_scales, const void *v_scales, int32_t num_items, const int32_t *items,
                               cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 148;
  const int64_t tasks = static_cast<int64_t>(num_items) * a.num_kv_heads;
  const int grid = static_cast<int>(tasks < sms ? tasks : sms);
  if constexpr (D == 128 && NT == 1 && !MULTI) {
    if (tasks > 3ll * grid * 12)
      return launch_decode_quant_w<D, NT, MULTI, 12, BITS>(a, tk, tv, k_scales, v_scales, num_items, items, grid,
                                                         stream);
  }
  return launch_decode_quant_w<D, NT, MULTI, kWarpsQuant, BITS>(a, tk, tv, k_scales, v_scales, num_items, items, grid,
                                                           stream);
}

}  // namespace

cudaError_t launch_cache_write_quant(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                                  int64_t num_tokens, void *k_codes, void *k_scales, void *v_codes, void *v_scales,
                                  int64_t num_blocks, int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t bits, uint32_t *status, cudaStream_t stream) {
  const int64_t rows = 2 * num_tokens * num_kv_heads;
  int64_t blocks = (rows + 7) / 8;  // 8 warps per CTA, one row each
  if (blocks > 152 * 16) blocks = 152 * 16;
  const dim3 grid(static_cast<unsigned>(blocks));
  auto *kn = static_cast<const __nv_bfloat16 *>(k_new);
  auto *vn = static_cast<const __nv_bfloat16 *>(v_new);
  auto *kc = static_cast<int8_t *>(k_codes);
  auto *vc = static_cast<int8_t *>(v_codes);
  auto *ksc = static_cast<__nv_bfloat16 *>(k_scales);
  auto *vsc = static_cast<__nv_bfloat16 *>(v_scales);
  const int64_t prows = num_blocks * block_size;
  if (bits == 4)
    return launch_pdl(cache_write_quant_kernel<128, 4>, grid, dim3(256), 0, stream, kn, vn, slot_mapping, num_tokens,
                      kc, ksc, vc, vsc, prows, block_size, num_kv_heads, status);
  if (head_dim == 128)
    return launch_pdl(cache_write_quant_kernel<128, 8>, grid, dim3(256), 0, stream, kn, vn, slot_mapping, num_tokens,
                      kc, ksc, vc, vsc, prows, block_size, num_kv_heads, status);
  return launch_pdl(cache_write_quant_kernel<64, 8>, grid, dim3(256), 0, stream, kn, vn, slot_mapping, num_tokens, kc,
                    ksc, vc, vsc, prows, block_size, num_kv_heads, status);
}

cudaError_t launch_widen_quant(const StepArgs &a, const void *k_codes, const void *k_scales, const void *v_codes,
                            const void *v_scales, void *k_out, void *v_out, int32_t *scratch_table,
                            int64_t scratch_blocks, int32_t num_items, const int32_t *items, int32_t bits,
                            cudaStream_t stream) {
  if (num_items <= 0) return cudaSuccess;
  // about four CTAs per SM over all items; a CTA whose first block is past its item's end exits
  const int per_item = (4 * 152 + num_items - 1) / num_items;
  const dim3 grid(static_cast<unsigned>(num_items),
                  static_cast<unsigned>(per_item < 1 ? 1 : per_item > 512 ? 512 : per_item));
  auto *kc = static_cast<const int8_t *>(k_codes);
  auto *vc = static_cast<const int8_t *>(v_codes);
  auto *ksc = static_cast<const __nv_bfloat16 *>(k_scales);
  auto *vsc = static_cast<const __nv_bfloat16 *>(v_scales);
  auto *ko = static_cast<__nv_bfloat16 *>(k_out);
  auto *vo = static_cast<__nv_bfloat16 *>(v_out);
  if (bits == 4)
    return launch_pdl(widen_quant_kernel<128, 4>, grid, dim3(256), 0, stream, a, items, kc, ksc, vc, vsc, ko, vo,
                      scratch_table, scratch_blocks);
  if (a.head_dim == 128)
    return launch_pdl(widen_quant_kernel<128, 8>, grid, dim3(256), 0, stream, a, items, kc, ksc, vc, vsc, ko, vo,
                      scratch_table, scratch_blocks);
  return launch_pdl(widen_quant_kernel<64, 8>, grid, dim3(256), 0, stream, a, items, kc, ksc, vc, vsc, ko, vo,
                    scratch_table, scratch_blocks);
}

cudaError_t launch_decode_quant(const StepArgs &a, const CUtensorMap &tk, const CUtensorMap &tv, const void *k_scales,
                             const void *v_scales, int32_t num_items, const int32_t *items, int32_t bits,
                             cudaStream_t stream) {
  if (num_items <= 0) return cudaSuccess;
  const bool multi = a.decode_rows_max > 1;
  const bool wide = a.group * (multi ? a.decode_rows_max : 1) > 8;
  const int v = (wide ? 2 : 0) + (multi ? 1 : 0);
  if (bits == 4) {  // head_dim 128 only
    switch (v) {
      case 0: return launch_decode_quant_t<128, 1, false, 4>(a, tk, tv, k_scales, v_scales, num_items, items, stream);
      case 1: return launch_decode_quant_t<128, 1, true, 4>(a, tk, tv, k_scales, v_scales, num_items, items, stream);
      case 2: return launch_decode_quant_t<128, 2, false, 4>(a, tk, tv, k_scales, v_scales, num_items, items, stream);
      default: return launch_decode_quant_t<128, 2, true, 4>(a, tk, tv, k_scales, v_scales, num_items, items, stream);
    }
  }
  switch (v + (a.head_dim == 128 ? 4 : 0)) {
    case 0: return launch_decode_quant_t<64, 1, false, 8>(a, tk, tv, k_scales, v_scales, num_items, items, stream);
    case 1: return launch_decode_quant_t<64, 1, true, 8>(a, tk, tv, k_scales, v_scales, num_items, items, stream);
    case 2: return launch_decode_quant_t<64, 2, false, 8>(a, tk, tv, k_scales, v_scales, num_items, items, stream);
    case 3: return launch_decode_quant_t<64, 2, true, 8>(a, tk, tv, k_scales, v_scales, num_items, items, stream);
    case 4: return launch_decode_quant_t<128, 1, false, 8>(a, tk, tv, k_scales, v_scales, num_items, items, stream);
    case 5: return launch_decode_quant_t<128, 1, true, 8>(a, tk, tv, k_scales, v_scales, num_items, items, stream);
    case 6: return launch_decode_quant_t<128, 2, false, 8>(a, tk, tv, k_scales, v_scales, num_items, items, stream);
    default: return launch_decode_quant_t<128, 2, true, 8>(a, tk, tv, k_scales, v_scales, num_items, items, stream);
  }
}

}  // namespace pkv
