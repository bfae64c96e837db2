"""GPU parity of the 8-bit and 4-bit block-scaled KV pools against ``oracle.kvquant``.

* ``pkv_cache_write_q8`` / ``_q4`` must be bit-exact: codes (4-bit: two's
  complement nibbles, the even value low, as ``oracle.kvquant.pack_nibbles``
  stores them) and scales of every pool row, including rows never written
  (which keep their fill);
* ``pkv_attention_q8`` / ``_q4`` must match attention over the dequantised pool within
  the attention tolerance (max abs 2e-2, relative L2 1e-2), on decode rows,
  verify runs, prompt chunks (widened into the bf16 scratch pool) and mixed
  steps, over the same shapes as the bf16 path.
"""

import zlib

import numpy as np
import pytest

import oracle
from oracle import kvquant as KQ
from continuous_batching_paged_pkv_gb300 import binding as B
from continuous_batching_paged_pkv_gb300 import build as libbuild
from continuous_batching_paged_pkv_gb300 import runtime as R
from continuous_batching_paged_pkv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
MAX_REL_L2 = 1e-2


@pytest.fixture(scope="module", autouse=True)
def cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    libbuild.build()
    oracle.build()
    return torch


def _oracle_pool(w, bits=8):
    """The oracle's block-scaled pool after the step's cache write (history, then the step's rows)."""
    st = oracle.prepare_step(w)
    kq, ks = KQ.empty_pool(w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim, bits)
    vq, vs = KQ.empty_pool(w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim, bits)
    segs = [(s.slot, s.q_len, s.ctx) for s in w.segments]
    hk = np.concatenate([w.hist_k[slot][:c - ql] for slot, ql, c in segs])
    hv = np.concatenate([w.hist_v[slot][:c - ql] for slot, ql, c in segs])
    KQ.cache_write(kq, ks, vq, vs, hk, hv, st.history_mapping, bits)
    nk = np.concatenate([w.hist_k[slot][c - ql:c] for slot, ql, c in segs])
    nv = np.concatenate([w.hist_v[slot][c - ql:c] for slot, ql, c in segs])
    KQ.cache_write(kq, ks, vq, vs, nk, nv, st.new_mapping, bits)
    return st, (kq, ks, vq, vs)


def _run(w, rows=None, check_pool=True, bits=8):
    import torch

    ds = R.prepare(w, kv=f"q{bits}")
    R.run_step(ds)
    torch.cuda.synchronize()
    assert B.pkv_check_device_status(ds.status) == 0
    st, (kq, ks, vq, vs) = _oracle_pool(w, bits)
    if check_pool:
        got = [ds.k_pool.cpu().numpy(), ds.k_scales.view(torch.int16).cpu().numpy().view(np.uint16),
               ds.v_pool.cpu().numpy(), ds.v_scales.view(torch.int16).cpu().numpy().view(np.uint16)]
        stored = (kq, ks, vq, vs) if bits == 8 else (KQ.pack_nibbles(kq), ks, KQ.pack_nibbles(vq), vs)
        for g, e, nm in zip(got, stored, ("k codes", "k scales", "v codes", "v scales")):
            assert np.array_equal(g, e), f"{w.name}: {nm} differ from the oracle's"
    ref = KQ.attention_paged(w.q, st.packed.cu_seqlens_q, st.packed.seq_slot, st.context_lens, st.block_tables,
                             kq, ks, vq, vs, w.scale, num_q_heads=w.num_q_heads, rows=rows)
    out = R.out_f32(ds)
    if rows is not None:
        out, ref = out[rows], ref[rows]
    assert np.isfinite(out).all(), f"{w.name}: non-finite output"
    err = np.abs(out - ref).max()
    rel = np.linalg.norm(out - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err <= MAX_ABS and rel <= MAX_REL_L2, f"{w.name}: max abs {err:.3e}, rel L2 {rel:.3e}"
    return ds


def test_tiny_step_q8():
    _run(W.tiny(0))


SHAPES = {
    "decode rows across spans": [(1, 1), (1, 17), (1, 257), (1, 511), (1, 1025), (1, 3000)],
    "verify runs": [(2, 257), (3, 258), (4, 513), (2, 2), (8, 520)],
    "long verify runs": [(12, 600), (16, 1000), (9, 257), (13, 13)],
    "prompt chunks": [(33, 100), (129, 300), (7, 7), (200, 200)],
    "mixed": [(40, 333), (1, 700), (1, 64), (9, 9), (2, 300)],
}


@pytest.mark.parametrize("case", sorted(SHAPES))
@pytest.mark.parametrize("heads,d", [((4, 2), 64), ((32, 8), 128), ((40, 8), 128), ((8, 8), 64), ((64, 8), 128),
                                     ((16, 1), 128)])
def test_shapes_q8(case, heads, d):
    hq, hkv = heads
    w = W.random_step(zlib.crc32(f"q8/{case}/{hq}/{hkv}/{d}".encode()) % 1000, SHAPES[case], num_q_heads=hq,
                      num_kv_heads=hkv, head_dim=d)
    _run(w)


def test_peaked_softmax_q8():
    w = W.random_step(6, [(1, 900), (64, 700)], num_q_heads=32, num_kv_heads=8, head_dim=128)
    w.q = W.f32_to_bf16_bits(W.bf16_bits_to_f32(w.q) * 8.0)
    _run(w)


def test_rows_of_different_magnitudes_q8():
    """Each (token, kv head) row scaled by 10^k, k in [-2, 2]: every group gets its own scale.

    Outputs then reach ~100, where bf16's own output rounding is ~0.4, so the
    absolute bound is taken relative to the output's magnitude (2e-2 * max |ref|);
    the relative L2 bound is unchanged.
    """
    rng = np.random.default_rng(3)
    w = W.random_step(8, [(1, 300), (16, 90), (3, 260)], num_q_heads=32, num_kv_heads=8, head_dim=128)
    for slot in w.hist_k:
        for arr in (w.hist_k[slot], w.hist_v[slot]):
            f = (10.0 ** rng.integers(-2, 3, arr.shape[:-1] + (1,))).astype(np.float32)
            arr[...] = W.f32_to_bf16_bits((W.bf16_bits_to_f32(arr) * f).astype(np.float32))
    global MAX_ABS
    saved = MAX_ABS
    try:
        st, (kq, ks, vq, vs) = _oracle_pool(w)
        ref = KQ.attention_paged(w.q, st.packed.cu_seqlens_q, st.packed.seq_slot, st.context_lens,
                                 st.block_tables, kq, ks, vq, vs, w.scale, num_q_heads=w.num_q_heads)
        MAX_ABS = 2e-2 * max(1.0, float(np.abs(ref).max()))
        _run(w)
    finally:
        MAX_ABS = saved


def test_decode_five_clients_q8():
    # the bench's contexts and heads on a smaller pool (the pool size changes no result)
    _run(W.make_step("decode5", 0, pool_blocks=4096))


def test_mixed_step_q8():
    w = W.make_step("mixed", 0, pool_blocks=4096)
    rows = sorted({0, 1, 255, 256, 511, *range(512, w.total_q)})
    _run(w, rows=rows)


def test_many_rows_q8():
    """A step with more than three rounds of decode tasks per warp: the 12-warp kernel and the task counter."""
    ctxs = [int(c) for c in np.random.default_rng(41).integers(1500, 2600, 360)]
    w = W.random_step(41, [(1, c) for c in ctxs], num_q_heads=16, num_kv_heads=2, head_dim=128)
    rows = sorted({0, 1, 2, 100, 200, 358, 359})
    _run(w, rows=rows)



# ---- 4-bit pool (head_dim 128) ----------------------------------------------------

@pytest.mark.parametrize("case", sorted(SHAPES))
@pytest.mark.parametrize("heads", [(32, 8), (40, 8), (64, 8), (16, 1)])
def test_shapes_q4(case, heads):
    hq, hkv = heads
    w = W.random_step(zlib.crc32(f"q4/{case}/{hq}/{hkv}".encode()) % 1000, SHAPES[case], num_q_heads=hq,
                      num_kv_heads=hkv, head_dim=128)
    _run(w, bits=4)


def test_peaked_softmax_q4():
    w = W.random_step(6, [(1, 900), (64, 700)], num_q_heads=32, num_kv_heads=8, head_dim=128)
    w.q = W.f32_to_bf16_bits(W.bf16_bits_to_f32(w.q) * 8.0)
    _run(w, bits=4)


def test_decode_five_clients_q4():
    _run(W.make_step("decode5", 0, pool_blocks=4096), bits=4)


def test_mixed_step_q4():
    w = W.make_step("mixed", 0, pool_blocks=4096)
    rows = sorted({0, 1, 255, 256, 511, *range(512, w.total_q)})
    _run(w, rows=rows, bits=4)


def test_many_rows_q4():
    ctxs = [int(c) for c in np.random.default_rng(43).integers(1500, 2600, 360)]
    w = W.random_step(43, [(1, c) for c in ctxs], num_q_heads=16, num_kv_heads=2, head_dim=128)
    _run(w, rows=sorted({0, 1, 2, 100, 200, 358, 359}), bits=4)


def test_q4_rejects_head_dim_64():
    with pytest.raises(B.PkvError):
        R.prepare(W.tiny(0), kv="q4")  # head_dim 64: the 4-bit pool is head_dim 128 only


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("bs", [32, 64])
def test_other_block_sizes_quant(bits, bs):
    w = W.random_step(bs + bits, [(1, 700), (40, 333), (1, 64), (9, 9), (3, 260)], num_q_heads=32, num_kv_heads=8,
                      head_dim=128, block_size=bs)
    _run(w, bits=bits)
