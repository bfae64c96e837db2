"""GPU parity: the CUDA path against the CPU oracle, element by element.

Cache writes must be bit-exact (whole pool, including rows never written,
which keep their NaN sentinel). Attention must satisfy, over the output,
max |gpu - oracle| <= 2e-2 and ||gpu - oracle||_2 / ||oracle||_2 <= 1e-2
(bf16 inputs, fp32 softmax and accumulation, bf16 output). Invariants the
pages fix are checked bit for bit on the GPU: packed order, physical block
permutation, batch of one, slot reuse.
"""

import zlib

import numpy as np
import pytest

import oracle
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


def assert_close(got, ref, rows=None, what=""):
    if rows is not None:
        got, ref = got[rows], ref[rows]
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err.max() <= MAX_ABS, f"{what}: max abs {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"
    assert rel <= MAX_REL_L2, f"{what}: rel L2 {rel:.3e}"


def run_and_check(w, *, full_pool=True, rows=None):
    import torch

    ds = R.prepare(w)
    R.run_step(ds)
    torch.cuda.synchronize()
    assert B.pkv_check_device_status(ds.status) == 0
    st = oracle.prepare_step(w)
    np.testing.assert_array_equal(ds.lowered.cu_seqlens_q, st.packed.cu_seqlens_q)
    np.testing.assert_array_equal(ds.lowered.seq_slot, st.packed.seq_slot)
    np.testing.assert_array_equal(ds.lowered.slot_mapping, st.new_mapping)
    if full_pool:
        kp, vp = R.pool_bits(ds)
        assert np.array_equal(kp, st.k_pool), "K pool differs from the oracle's"
        assert np.array_equal(vp, st.v_pool), "V pool differs from the oracle's"
    else:
        used = np.unique(np.concatenate([w.blocks[s.slot] for s in w.segments]))
        extra = np.random.default_rng(0).choice(w.num_blocks, 64, replace=False)
        check = np.unique(np.concatenate([used, extra]))
        idx = torch.from_numpy(check).to(ds.k_pool.device)
        kp = ds.k_pool.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16)
        vp = ds.v_pool.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(kp, st.k_pool[check]) and np.array_equal(vp, st.v_pool[check])
    ref = oracle.step_attention(w, st, rows=rows)
    got = R.out_f32(ds)
    assert_close(got, ref, rows, w.name)
    return ds, got, ref


def test_tiny_step():
    ds, got, ref = run_and_check(W.tiny(0))
    # a decode row at context 5 and one at 37, a 16-row chunk at offset 64
    assert got.shape == (18, 4, 64)


def test_decode_five_clients():
    run_and_check(W.decode5(0))


def test_mixed_chunk_and_decode():
    run_and_check(W.mixed(0))


@pytest.mark.slow
def test_large_decode_batch():
    run_and_check(W.decode256(0), full_pool=False)


def test_full_2048_row_chunk_at_offset_6144():
    """The chunk size taken while nothing decodes, every element against the oracle:
    2048 rows [6144, 8192) of an 8192-token prompt, 32 q / 8 kv heads, head_dim 128."""
    run_and_check(W.chunk2048(0), full_pool=False)


def test_full_2048_row_chunk_beside_decode_rows():
    """A 2048-row chunk at offset 4096 packed with decode rows and a short verify run."""
    w = W.random_step(2048, [(2048, 6144), (1, 3000), (3, 700), (1, 17)], num_q_heads=32, num_kv_heads=8,
                      head_dim=128)
    run_and_check(w, full_pool=False)


EDGE_SHAPES = {
    "single key and tiny contexts": [(1, 1), (1, 2), (1, 15), (1, 16), (1, 17)],
    "span boundaries": [(1, 511), (1, 512), (1, 513), (1, 1024), (1, 1025), (1, 1536)],
    "chunks with ragged tails": [(2, 2), (31, 40), (32, 32), (33, 100), (129, 300), (7, 7)],
    "whole prompt as one chunk": [(200, 200), (128, 128), (1, 300)],
    # short causal runs (verify rows); at small groups they take the decode path,
    # and a run across a span boundary leaves its first rows with an empty last span
    "verify runs": [(2, 257), (3, 258), (4, 257), (4, 513), (8, 520), (16, 777), (5, 5), (2, 2)],
    # runs of several row groups (ragged last group, across span boundaries), and one just past the limit
    "long verify runs": [(12, 600), (16, 1000), (9, 257), (7, 513), (20, 700), (33, 800), (64, 300), (13, 13)],
}


@pytest.mark.parametrize("case", sorted(EDGE_SHAPES))
@pytest.mark.parametrize("heads,d", [((4, 2), 64), ((32, 8), 128), ((40, 8), 128), ((8, 8), 64),
                                     ((64, 8), 128), ((16, 1), 128)])
def test_edge_shapes(case, heads, d):
    hq, hkv = heads
    w = W.random_step(zlib.crc32(f"{case}/{hq}/{hkv}/{d}".encode()) % 1000, EDGE_SHAPES[case], num_q_heads=hq, num_kv_heads=hkv,
                      head_dim=d)
    run_and_check(w)


@pytest.mark.parametrize("bs", [32, 64])
def test_other_block_sizes(bs):
    w = W.random_step(bs, [(1, 700), (40, 333), (1, 64), (9, 9)], num_q_heads=32, num_kv_heads=8,
                      head_dim=128, block_size=bs)
    run_and_check(w)


def test_single_key_output_is_exactly_the_value():
    w = W.random_step(5, [(1, 1)], num_q_heads=8, num_kv_heads=2, head_dim=128)
    ds, got, ref = run_and_check(w)
    v0 = W.bf16_bits_to_f32(w.hist_v[0][0])  # [Hkv, D]
    np.testing.assert_array_equal(got[0], np.repeat(v0, 4, axis=0))


def test_peaked_softmax():
    w = W.random_step(6, [(1, 900), (64, 700)], num_q_heads=32, num_kv_heads=8, head_dim=128)
    w.q = W.f32_to_bf16_bits(W.bf16_bits_to_f32(w.q) * 8.0)
    run_and_check(w)


# ---- invariants, bit for bit on the GPU ---------------------------------------------

def _out_rows(w, got):
    res, start = {}, 0
    for s in w.segments:
        res[s.slot] = got[start:start + s.q_len]
        start += s.q_len
    return res


SHAPES = [(1, 700), (64, 300), (1, 37), (17, 80), (1, 5000), (3, 3)]


def _gpu_out(w):
    import torch

    ds = R.prepare(w)
    R.run_step(ds)
    torch.cuda.synchronize()
    assert B.pkv_check_device_status(ds.status) == 0
    return R.out_f32(ds)


def test_packed_order_does_not_change_results():
    w = W.random_step(21, SHAPES, num_q_heads=32, num_kv_heads=8, head_dim=128)
    base = _out_rows(w, _gpu_out(w))
    r = W.random_step(21, SHAPES, num_q_heads=32, num_kv_heads=8, head_dim=128)
    order = [4, 2, 0, 5, 3, 1]
    rows = {}
    start = 0
    for s in w.segments:
        rows[s.slot] = w.q[start:start + s.q_len]
        start += s.q_len
    r.segments = [w.segments[i] for i in order]
    r.q = np.concatenate([rows[s.slot] for s in r.segments])
    got = _out_rows(r, _gpu_out(r))
    for slot in base:
        np.testing.assert_array_equal(got[slot], base[slot])


def test_physical_block_permutation_does_not_change_results():
    a = W.random_step(22, SHAPES, num_q_heads=32, num_kv_heads=8, head_dim=128)
    b = W.random_step(22, SHAPES, num_q_heads=32, num_kv_heads=8, head_dim=128)
    perm = np.random.default_rng(1).permutation(a.num_blocks).astype(np.int32)
    b.blocks = {s: perm[ids] for s, ids in a.blocks.items()}
    np.testing.assert_array_equal(_gpu_out(a), _gpu_out(b))


def test_batch_of_one_equals_in_batch():
    w = W.random_step(23, SHAPES, num_q_heads=32, num_kv_heads=8, head_dim=128)
    full = _out_rows(w, _gpu_out(w))
    start = 0
    for seg in list(w.segments):
        one = W.random_step(23, SHAPES, num_q_heads=32, num_kv_heads=8, head_dim=128)
        one.segments = [seg]
        one.q = w.q[start:start + seg.q_len]
        start += seg.q_len
        np.testing.assert_array_equal(_gpu_out(one), full[seg.slot])


@pytest.mark.parametrize("heads,d", [((16, 2), 64), ((8, 1), 128)])
def test_merge_kernels_agree_bit_for_bit(heads, d):
    """A step of many split rows is merged by the many-row kernel (one lane per column, four for
    rows of more than 64 spans); the same rows in a step of their own are merged by the few-row
    kernel. Both follow one fixed order of operations, so the rows must come out bit-identical --
    also for rows of more than 32 spans (several rounds per lane) and of more than 64 spans
    (several shared-memory pieces in the one-lane layout, the four-lane layout in the mixed one)."""
    hq, hkv = heads
    ctxs = [int(c) for c in np.random.default_rng(31).integers(300, 2500, 150)] + [9000, 17000, 20001, 513]
    shapes = [(1, c) for c in ctxs]
    w = W.random_step(31, shapes, num_q_heads=hq, num_kv_heads=hkv, head_dim=d)
    # more four-lane CTAs (8 per row here) than one wave of six per SM on 152 SMs: the full step
    # takes the one-lane layout, with its rows of more than 64 spans (17000, 20001) in four lanes
    assert len(ctxs) * 8 > 6 * 152
    _, got_full, _ = run_and_check(w, full_pool=False, rows=[0, 1, 150, 151, 152, 153])
    full = _out_rows(w, got_full)
    pick = [150, 151, 152, 3]
    sub = W.random_step(31, shapes, num_q_heads=hq, num_kv_heads=hkv, head_dim=d)
    sub.segments = [w.segments[i] for i in pick]
    sub.q = np.concatenate([w.q[i:i + 1] for i in pick])  # one row per segment, in packed order
    got = _out_rows(sub, _gpu_out(sub))
    for i in pick:
        slot = w.segments[i].slot
        np.testing.assert_array_equal(got[slot], full[slot])


def test_slot_reuse_leaves_other_slots_bit_identical():
    """B retires; a new sequence D takes B's slot and blocks. A's and C's pool rows and outputs stay."""
    import torch

    w = W.tiny(0)
    ds = R.prepare(w)
    R.run_step(ds)
    torch.cuda.synchronize()
    out_a_c = R.out_f32(ds)[16:].copy()
    a_c = torch.from_numpy(np.concatenate([w.blocks[0], w.blocks[2]])).cuda()
    keep_k = ds.k_pool.index_select(0, a_c).clone()
    keep_v = ds.v_pool.index_select(0, a_c).clone()

    ds.pool.release(1)
    assert ds.pool.admit(1, 40) == B.PKV_OK
    rng = np.random.default_rng(9)
    d_k = W.f32_to_bf16_bits(rng.standard_normal((40, 2, 64), dtype=np.float32))
    d_v = W.f32_to_bf16_bits(rng.standard_normal((40, 2, 64), dtype=np.float32))
    d_q = W.f32_to_bf16_bits(rng.standard_normal((1, 4, 64), dtype=np.float32))
    low_hist = ds.pool.lower([(1, 39)])
    B.pkv_cache_write(R._bf16_tensor(d_k[:39], "cuda"), R._bf16_tensor(d_v[:39], "cuda"),
                      R._i64(low_hist.slot_mapping, "cuda"), ds.k_pool, ds.v_pool)
    # next step: D decodes its 40th row, A and C decode one more row too
    extra = {s: W.f32_to_bf16_bits(rng.standard_normal((1, 2, 64), dtype=np.float32)) for s in (0, 2)}
    low = ds.pool.lower([(1, 1), (0, 1), (2, 1)])
    k_new = np.concatenate([d_k[39:], extra[0], extra[2]])
    v_new = np.concatenate([d_v[39:], extra[0], extra[2]])
    B.pkv_cache_write(R._bf16_tensor(k_new, "cuda"), R._bf16_tensor(v_new, "cuda"),
                      R._i64(low.slot_mapping, "cuda"), ds.k_pool, ds.v_pool)
    # A's and C's already-written rows did not move
    k_after = ds.k_pool.index_select(0, a_c)
    for i, blk in enumerate(np.concatenate([w.blocks[0], w.blocks[2]])):
        rows_written = (low.slot_mapping // 16 == blk)
        if not rows_written.any():
            assert torch.equal(k_after[i].view(torch.int16), keep_k[i].view(torch.int16))
    # Attention for the previous step's A and C rows is unchanged when recomputed with the old contexts.
    bt = torch.from_numpy(ds.pool.block_tables()).cuda()
    ctx_old = torch.from_numpy(ds.lowered.context_lens).cuda()
    q_ac = ds.q[16:].contiguous()
    cu = torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda")
    ss = torch.tensor([0, 2], dtype=torch.int32, device="cuda")
    work, info = B.pkv_plan_work(np.array([0, 1, 2]), np.array([0, 2]), ds.lowered.context_lens,
                                 max_slots=w.max_slots, max_blocks_per_slot=w.max_blocks_per_slot,
                                 block_size=16, num_q_heads=4, num_kv_heads=2, head_dim=64)
    out = torch.empty_like(q_ac)
    B.pkv_attention(q_ac, cu, ss, ctx_old, bt, ds.k_pool, ds.v_pool, torch.from_numpy(work).cuda(), info, out,
                    None, scale=w.scale)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.float().cpu().numpy(), out_a_c)
    del keep_v


# ---- failure detection: invalid indices are reported, never faulted on ----------------

def test_bad_block_id_sets_device_status_and_context_survives():
    import torch

    w = W.random_step(30, [(1, 600), (20, 90)], num_q_heads=32, num_kv_heads=8, head_dim=128)
    ds = R.prepare(w)
    bt = ds.block_tables.clone()
    bt[0, 3] = w.num_blocks + 7        # decode span
    bt[1, 2] = -5                      # chunk tile
    B.pkv_attention(ds.q, ds.cu_seqlens_q, ds.seq_slot, ds.context_lens, bt, ds.k_pool, ds.v_pool, ds.work,
                    ds.info, ds.out, ds.workspace, scale=w.scale, device_status=ds.status)
    bits = B.pkv_check_device_status(ds.status)
    assert bits & 0x2
    # the context is still healthy: a correct step right after passes parity
    run_and_check(W.tiny(1))


def test_bad_slot_mapping_sets_device_status():
    import torch

    w = W.tiny(0)
    ds = R.prepare(w)
    sm = ds.slot_mapping.clone()
    sm[3] = w.num_blocks * w.block_size + 100
    B.pkv_cache_write(ds.k_new, ds.v_new, sm, ds.k_pool, ds.v_pool, device_status=ds.status)
    assert B.pkv_check_device_status(ds.status) & 0x1
    torch.cuda.synchronize()


def test_empty_step_launches_nothing():
    import torch

    w = W.tiny(0)
    ds = R.prepare(w)
    empty = torch.empty((0, 2, 64), dtype=torch.bfloat16, device="cuda")
    B.pkv_cache_write(empty, empty, torch.empty(0, dtype=torch.int64, device="cuda"), ds.k_pool, ds.v_pool)
    info = B.WorkInfo()
    B.pkv_attention(ds.q[:0], torch.zeros(1, dtype=torch.int32, device="cuda"),
                    torch.zeros(0, dtype=torch.int32, device="cuda"), ds.context_lens, ds.block_tables,
                    ds.k_pool, ds.v_pool, torch.zeros(4, dtype=torch.int32, device="cuda"), info, ds.out[:0])
    torch.cuda.synchronize()
