"""Oracle for the 8-bit and 4-bit block-scaled KV pools -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this module; the CUDA library never calls it and shares no code
with it.

The pages run their KV caches quantised (Lucebox, "Continuous batching ...",
§DeepSeek V4 Flash on Strix Halo and two GPUs: 4-bit KV; §Qwen3.8-27B DFlash2
on the R9700 (vs llama.cpp): 8-bit KV) but do not define the formats. The
reading taken here is the plainest block-scaled one, with B bits per code and
Q = 2^(B-1) - 1 (127 for 8 bits, 7 for 4 bits):

* each pool row (one token, one kv head, head_dim values) is cut into groups
  of 32 consecutive values;
* a group stores one power-of-two scale ``d`` (kept as a bfloat16, which
  holds it exactly) and 32 signed codes in [-Q, Q]; the value a code stands
  for is ``code * d``;
* quantising a group of bfloat16 values ``x`` (all steps in float32, the
  precision the codes are decided in):
    amax = max |x|;  t = amax / Q;  d = the smallest power of two >= t
    (at least 2^-126; 0 when amax is 0);
    code = clamp(round_half_even(x / d), -Q, Q), or 0 when d is 0.
  This power-of-two ceiling is this library's own reading (the pages fix no
  rule). It makes x / d exact, |x - code * d| <= d / 2, and every value a code
  stands for exactly a bfloat16 number (at most 7 significant bits times a
  power of two), so attention may widen codes to bfloat16 without rounding.
  Its cost: rounding the scale up leaves the group maximum's code anywhere in
  [(Q + 1) / 2, Q] rather than at Q, up to one bit of precision lost there.
* storage: 8-bit codes one per byte; 4-bit codes two per byte, the code of
  the even value in the low nibble, each a 4-bit two's complement number
  (``pack_nibbles``). Scales are stored as in the 8-bit pool.

Attention over such a pool is ordinary causal grouped-query attention over the
dequantised values ``code * d`` (exact in double), computed here in float64
with a plain per-segment gather through the block table.
"""

from __future__ import annotations

import numpy as np

GROUP = 32  # values per scale
CODE_MAX = 127  # 8-bit codes


def code_max(bits: int) -> int:
    if bits not in (8, 4):
        raise ValueError(f"{bits}-bit codes are not a format of this pool")
    return (1 << (bits - 1)) - 1


def _widen(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def _pow2_ceil(t) -> np.ndarray:
    """Smallest power of two >= t (float32 t >= 0), at least 2^-126; 0 for t == 0. Float32 bits."""
    b = np.ascontiguousarray(t, dtype=np.float32).view(np.uint32)
    exp_bits = b & np.uint32(0x7F800000)
    up = np.where((b & np.uint32(0x007FFFFF)) == 0, b, exp_bits + np.uint32(0x00800000))
    up = np.where(exp_bits == 0, np.uint32(0x00800000), up)  # below 2^-126
    return np.where(b == 0, np.uint32(0), up).astype(np.uint32)


def quantize(x_bits, bits: int = 8):
    """bf16 bits ``[..., D]`` -> (codes int8 ``[..., D]`` in [-Q, Q], scale bits uint16 ``[..., D / 32]``)."""
    q = code_max(bits)
    x = _widen(x_bits)
    d_len = x.shape[-1]
    if d_len % GROUP:
        raise ValueError(f"head_dim {d_len} is not a multiple of {GROUP}")
    g = x.reshape(*x.shape[:-1], d_len // GROUP, GROUP)
    amax = np.abs(g).max(axis=-1)
    d32 = _pow2_ceil((amax / np.float32(q)).astype(np.float32))
    d_bits = (d32 >> 16).astype(np.uint16)  # a power of two: its bfloat16 is exact
    df = _widen(d_bits)[..., None]
    safe = np.where(df > 0, df, np.float32(1))
    r = np.where(df > 0, g / safe, np.float32(0)).astype(np.float32)
    codes = np.clip(np.rint(r), -q, q).astype(np.int8)
    return codes.reshape(x.shape), d_bits


def dequantize(codes, scale_bits) -> np.ndarray:
    """The values codes stand for, in float64 (exact)."""
    c = np.asarray(codes, dtype=np.int8)
    s = _widen(scale_bits).astype(np.float64)
    g = c.reshape(*c.shape[:-1], c.shape[-1] // GROUP, GROUP).astype(np.float64)
    return (g * s[..., None]).reshape(c.shape)


def pack_nibbles(codes) -> np.ndarray:
    """4-bit storage of codes in [-8, 7] ``[..., D]``: uint8 ``[..., D / 2]``, even value in the low nibble."""
    c = np.asarray(codes, dtype=np.int8).astype(np.int16) & 0xF
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed) -> np.ndarray:
    """Inverse of ``pack_nibbles``: int8 codes ``[..., 2 * D2]``."""
    p = np.asarray(packed, dtype=np.uint8).astype(np.int16)
    lo, hi = p & 0xF, p >> 4
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), np.int16)
    out[..., 0::2], out[..., 1::2] = lo, hi
    return np.where(out >= 8, out - 16, out).astype(np.int8)


def empty_pool(num_blocks, num_kv_heads, block_size, head_dim, bits: int = 8):
    """(codes, scales) pools filled with a recognisable pattern for rows never written.

    Codes are kept one per int8 here; the unused code -2^(B-1) marks rows never written."""
    codes = np.full((num_blocks, num_kv_heads, block_size, head_dim), -(code_max(bits) + 1), np.int8)
    scales = np.full((num_blocks, num_kv_heads, block_size, head_dim // GROUP), 0x7FC1, np.uint16)  # NaN
    return codes, scales


def cache_write(k_codes, k_scales, v_codes, v_scales, k_new, v_new, mapping, bits: int = 8) -> None:
    """Quantise new rows ``[T, Hkv, D]`` (bf16 bits) into the pools at pool rows ``mapping`` (< 0: skip)."""
    nb, hkv, bs, d = k_codes.shape
    mapping = np.asarray(mapping, dtype=np.int64)
    if np.any(mapping >= nb * bs):
        raise ValueError("slot mapping past the pool")
    kq, ks = quantize(k_new, bits)
    vq, vs = quantize(v_new, bits)
    for t, s in enumerate(mapping):
        if s < 0:
            continue
        blk, row = divmod(int(s), bs)
        k_codes[blk, :, row, :] = kq[t]
        k_scales[blk, :, row, :] = ks[t]
        v_codes[blk, :, row, :] = vq[t]
        v_scales[blk, :, row, :] = vs[t]


def attention_paged(q, cu_seqlens_q, seq_slot, context_lens, block_tables, k_codes, k_scales, v_codes,
                    v_scales, scale: float, *, num_q_heads: int, rows=None) -> np.ndarray:
    """float64 ``[T, Hq, D]``; rows outside ``rows`` (if given) are NaN.

    Segment s (slot c, n rows, L = context_lens[c]): row i sits at position
    L - n + i and attends keys 0..L-n+i of slot c, gathered block by block in
    logical order; q head h reads kv head h // (Hq / Hkv).
    """
    nb, hkv, bs, d = k_codes.shape
    qf = _widen(q).astype(np.float64)
    T = qf.shape[0]
    out = np.full((T, num_q_heads, d), np.nan)
    keep = None if rows is None else set(int(r) for r in rows)
    G = num_q_heads // hkv
    cu = np.asarray(cu_seqlens_q)
    for s, slot in enumerate(np.asarray(seq_slot)):
        r0, r1 = int(cu[s]), int(cu[s + 1])
        n, L = r1 - r0, int(context_lens[slot])
        if n == 0:
            continue
        blocks = np.asarray(block_tables[slot][: -(-L // bs)], dtype=np.int64)
        if np.any(blocks < 0) or np.any(blocks >= nb):
            raise ValueError(f"segment {s}: block id outside the pool")
        # [nblk, Hkv, bs, D] -> [nblk * bs, Hkv, D], first L positions
        k = dequantize(k_codes[blocks], k_scales[blocks]).transpose(0, 2, 1, 3).reshape(-1, hkv, d)[:L]
        v = dequantize(v_codes[blocks], v_scales[blocks]).transpose(0, 2, 1, 3).reshape(-1, hkv, d)[:L]
        for i in range(n):
            row = r0 + i
            if keep is not None and row not in keep:
                continue
            p = L - n + i
            for h in range(num_q_heads):
                sc = scale * (k[: p + 1, h // G, :] @ qf[row, h, :])
                w = np.exp(sc - sc.max())
                out[row, h, :] = (w @ v[: p + 1, h // G, :]) / w.sum()
    return out
