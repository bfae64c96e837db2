"""Pins for the 8-bit and 4-bit block-scaled KV oracle (``oracle.kvquant``).

The format is this library's reading (the pages run 8-bit and 4-bit KV caches
without defining them): groups of 32 values, one power-of-two scale (the
smallest at or above amax / Q), codes rounded half to even into [-Q, Q], with
Q = 127 for 8-bit and 7 for 4-bit codes. The pins tie the oracle to facts that
hold independently of its code, for both code widths:

* the error bound of round-to-nearest: |x - code * d| <= d / 2, with d a power
  of two in [amax / Q, 2 amax / Q);
* every dequantised value is exactly a bfloat16 number;
* exact reconstruction of groups that are integer multiples of a power of two
  with one value at +-Q of them;
* the 4-bit storage: two's complement nibbles, the even value low, by hand;
* the half-way cases, which must round to even;
* zero groups, and groups at the ends of bfloat16's range;
* attention over an exactly representable quantised pool equals the bf16
  oracle (pinned elsewhere) on the same values;
* attention over any quantised pool equals a numpy brute force over the
  dequantised contiguous history.
"""

import numpy as np
import pytest

import oracle
from oracle import kvquant as KQ
from continuous_batching_paged_pkv_gb300 import workloads as W


def _bits(x):
    return W.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


BITS = [8, 4]
QMAX = {8: 127, 4: 7}


@pytest.mark.parametrize("nbits", BITS)
def test_error_bound_and_code_range(nbits):
    Q = QMAX[nbits]
    rng = np.random.default_rng(0)
    x = rng.standard_normal((64, 4, 128)).astype(np.float32) * (10.0 ** rng.integers(-30, 30, (64, 1, 1)))
    bits = _bits(x)
    xf = W.bf16_bits_to_f32(bits).astype(np.float64)
    codes, sb = KQ.quantize(bits, nbits)
    d = W.bf16_bits_to_f32(sb).astype(np.float64)
    assert codes.dtype == np.int8 and sb.shape == (64, 4, 4)
    assert codes.min() >= -Q and codes.max() <= Q
    err = np.abs(xf.reshape(64, 4, 4, 32) - codes.reshape(64, 4, 4, 32) * d[..., None])
    assert np.all(err <= d[..., None] / 2)
    # d is a power of two between amax / Q and twice that, so the largest code is in [(Q + 1) / 2, Q]
    amax = np.abs(xf.reshape(64, 4, 4, 32)).max(axis=-1)
    assert np.all(np.frexp(d)[0] == 0.5)
    assert np.all((d >= amax / Q) & (d < 2 * amax / Q * (1 + 1e-6)))
    top = np.abs(codes.reshape(64, 4, 4, 32)).max(axis=-1)
    assert np.all((top >= (Q + 1) // 2) & (top <= Q))
    # each dequantised value is a bfloat16 number: widening to bf16 loses nothing
    deq = KQ.dequantize(codes, sb).astype(np.float32)
    assert np.array_equal(W.bf16_bits_to_f32(W.f32_to_bf16_bits(deq)), deq)


@pytest.mark.parametrize("nbits", BITS)
@pytest.mark.parametrize("e", [-120, -24, -7, 0, 5, 100])
def test_power_of_two_multiples_are_exact(e, nbits):
    Q = QMAX[nbits]
    rng = np.random.default_rng(e + 1000)
    k = rng.integers(-Q, Q + 1, (8, 2, 64))
    k[..., 0] = Q
    k[..., 32] = -Q
    x = np.ldexp(k.astype(np.float64), e)
    codes, sb = KQ.quantize(_bits(x), nbits)
    assert np.array_equal(codes, k.astype(np.int8))
    assert np.all(W.bf16_bits_to_f32(sb).astype(np.float64) == 2.0 ** e)
    assert np.array_equal(KQ.dequantize(codes, sb), x)


@pytest.mark.parametrize("nbits,top,want", [(8, 62.5, 62), (4, 6.5, 6)])
def test_half_way_values_round_to_even(nbits, top, want):
    k = np.zeros(32)
    k[0] = QMAX[nbits]
    halves = np.array([0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, top])
    k[1:1 + len(halves)] = halves
    codes, _ = KQ.quantize(_bits(np.ldexp(k, -3)), nbits)
    assert codes[1:1 + len(halves)].tolist() == [0, 2, 2, 4, 0, -2, -2, want]


def test_nibble_storage_by_hand():
    # -8 -> 0x8, 7 -> 0x7, -1 -> 0xF, 0 -> 0x0, 3 -> 0x3, -7 -> 0x9; even value in the low nibble
    codes = np.array([[-8, 7, -1, 0, 3, -7]], np.int8)
    packed = KQ.pack_nibbles(codes)
    assert packed.tolist() == [[0x78, 0x0F, 0x93]]
    assert np.array_equal(KQ.unpack_nibbles(packed), codes)
    every = np.arange(-8, 8, dtype=np.int8).reshape(1, 16)
    assert np.array_equal(KQ.unpack_nibbles(KQ.pack_nibbles(every)), every)


@pytest.mark.parametrize("nbits", BITS)
def test_zero_group_and_range_ends(nbits):
    Q = QMAX[nbits]
    x = np.zeros((4, 64), np.float32)
    x[1, :32] = np.linspace(-3e38, 3e38, 32)    # near the top of bfloat16's range
    x[2, :32] = np.linspace(-1e-35, 1e-35, 32)  # scale still a normal number
    x[3, :32] = np.linspace(-1e-38, 1e-38, 32)  # scale subnormal: fewer code levels, same bound
    codes, sb = KQ.quantize(_bits(x), nbits)
    assert np.all(codes[0] == 0) and np.all(sb[0] == 0) and np.all(codes[1:, 32:] == 0)
    for r in (1, 2, 3):
        xf = W.bf16_bits_to_f32(_bits(x[r, :32])).astype(np.float64)
        d = float(W.bf16_bits_to_f32(sb[r, :1])[0])
        assert np.frexp(d)[0] == 0.5 and d >= 2.0 ** -126
        if r < 3:
            assert codes[r, 0] == -codes[r, 31] and (Q + 1) // 2 <= codes[r, 31] <= Q
        assert np.all(np.abs(xf - codes[r, :32] * d) <= d / 2)


def _exact_step(rng, shapes, hq, hkv, d, e=-6, Q=127):
    """A random step whose K/V are k * 2^e with +-Q in every group (bf16-exact and exact in the format)."""
    w = W.random_step(int(rng.integers(1 << 30)), shapes, num_q_heads=hq, num_kv_heads=hkv, head_dim=d)
    for slot in w.hist_k:
        for arr in (w.hist_k[slot], w.hist_v[slot]):
            k = rng.integers(-Q, Q + 1, arr.shape)
            k[..., ::32] = Q * rng.choice([-1, 1], k[..., ::32].shape)
            arr[...] = _bits(np.ldexp(k.astype(np.float64), e))
    return w


def _q8_step(w, nbits=8):
    st = oracle.prepare_step(w)
    kq, ks = KQ.empty_pool(w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim, nbits)
    vq, vs = KQ.empty_pool(w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim, nbits)
    segs = [(s.slot, s.q_len, s.ctx) for s in w.segments]
    hk = np.concatenate([w.hist_k[slot][:c] for slot, _, c in segs])
    hv = np.concatenate([w.hist_v[slot][:c] for slot, _, c in segs])
    allrows = oracle.pack([(slot, c, c) for slot, _, c in segs])
    m = oracle.slot_mapping(st.block_tables, allrows.token_slot, allrows.token_pos, w.block_size, w.num_blocks)
    KQ.cache_write(kq, ks, vq, vs, hk, hv, m, nbits)
    return st, (kq, ks, vq, vs)


@pytest.mark.parametrize("nbits", BITS)
def test_attention_on_exact_pool_equals_bf16_oracle(oracle_lib, nbits):
    rng = np.random.default_rng(5)
    w = _exact_step(rng, [(1, 37), (16, 80), (1, 5), (3, 300)], 8, 2, 64, Q=QMAX[nbits])
    st, (kq, ks, vq, vs) = _q8_step(w, nbits)
    got = KQ.attention_paged(w.q, st.packed.cu_seqlens_q, st.packed.seq_slot, st.context_lens, st.block_tables,
                             kq, ks, vq, vs, w.scale, num_q_heads=w.num_q_heads)
    ref = oracle.step_attention(w, st)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("nbits", BITS)
def test_attention_equals_bruteforce_on_dequantised_history(nbits):
    rng = np.random.default_rng(6)
    w = W.random_step(17, [(1, 70), (12, 40), (2, 2)], num_q_heads=6, num_kv_heads=2, head_dim=64)
    st, (kq, ks, vq, vs) = _q8_step(w, nbits)
    got = KQ.attention_paged(w.q, st.packed.cu_seqlens_q, st.packed.seq_slot, st.context_lens, st.block_tables,
                             kq, ks, vq, vs, w.scale, num_q_heads=w.num_q_heads)
    qf = W.bf16_bits_to_f32(w.q).astype(np.float64)
    for s, seg in enumerate(w.segments):
        kf = KQ.dequantize(*KQ.quantize(w.hist_k[seg.slot][: seg.ctx], nbits))
        vf = KQ.dequantize(*KQ.quantize(w.hist_v[seg.slot][: seg.ctx], nbits))
        r0 = int(st.packed.cu_seqlens_q[s])
        n, L = seg.q_len, seg.ctx
        mask = np.arange(L)[None, :] <= (L - n + np.arange(n))[:, None]
        for h in range(w.num_q_heads):
            sc = w.scale * (qf[r0:r0 + n, h, :] @ kf[:, h // 3, :].T)
            sc = np.where(mask, sc, -np.inf)
            p = np.exp(sc - sc.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            np.testing.assert_allclose(got[r0:r0 + n, h, :], p @ vf[:, h // 3, :], rtol=0, atol=1e-12)
    del rng
