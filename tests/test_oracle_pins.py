"""Pins for the CPU oracle: each test ties it to something other than itself.

* a numpy brute force that builds the contiguous history, the full score
  matrix and an explicit causal mask matrix (a different algorithm and data
  path from the oracle's per-row walk of the block table);
* torch's scaled_dot_product_attention in float64 on the CPU (a library
  routine), with grouped heads expanded by repeat_interleave;
* closed forms: one visible key, zero query, equal keys, one dominant key;
* invariants the pages fix: paged = contiguous, independence from the physical
  block permutation, batch of one = inside a batch, packed order, slot reuse
  (Lucebox, "Continuous batching ...", §Keeping track of each request and
  §Paged KV and paged attention; mlxcel manual, §Paged KV cache and prefix
  sharing);
* the pages' worked examples under tests/golden/;
* mutation checks: plausible mistakes planted in a copy of the oracle's C
  source make at least one pin fail.
"""

import os
import subprocess

import numpy as np
import pytest

from continuous_batching_paged_pkv_gb300 import workloads as W
from tests.conftest import golden

import oracle
from oracle import churn


def _f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def brute_force(q, k, v, scale):
    """q [n,Hq,D], k/v [L,Hkv,D] (bf16 bits) -> [n,Hq,D] via full masked score matrices."""
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    n, hq, d = qf.shape
    L, hkv, _ = kf.shape
    g = hq // hkv
    mask = np.arange(L)[None, :] <= (L - n + np.arange(n))[:, None]
    out = np.empty((n, hq, d))
    for h in range(hq):
        s = scale * (qf[:, h, :] @ kf[:, h // g, :].T)
        s = np.where(mask, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ vf[:, h // g, :]
    return out


def _rand(rng, shape):
    return W.f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


CASES = [  # (n, L, Hq, Hkv, D)
    (1, 1, 2, 1, 8), (1, 37, 4, 2, 64), (16, 80, 4, 2, 64), (5, 5, 4, 4, 16),
    (7, 40, 6, 2, 32), (3, 19, 8, 1, 8), (12, 12, 5, 5, 16),
]


@pytest.mark.parametrize("n,L,hq,hkv,d", CASES)
def test_dense_matches_bruteforce(oracle_lib, n, L, hq, hkv, d):
    rng = np.random.default_rng(n * 1000 + L)
    q, k, v = _rand(rng, (n, hq, d)), _rand(rng, (L, hkv, d)), _rand(rng, (L, hkv, d))
    for mult in (1.0, 8.0):  # diffuse and peaked softmax
        qq = W.f32_to_bf16_bits(W.bf16_bits_to_f32(q) * mult)
        got = oracle.attention_dense(qq, k, v, 1 / np.sqrt(d))
        ref = brute_force(qq, k, v, 1 / np.sqrt(d))
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("n,L,hq,hkv,d", CASES)
def test_dense_matches_torch_sdpa_float64(oracle_lib, n, L, hq, hkv, d):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7 + n + L)
    q, k, v = _rand(rng, (n, hq, d)), _rand(rng, (L, hkv, d)), _rand(rng, (L, hkv, d))
    scale = 1 / np.sqrt(d)
    got = oracle.attention_dense(q, k, v, scale)
    g = hq // hkv
    tq = torch.from_numpy(_f64(q)).permute(1, 0, 2)
    tk = torch.from_numpy(_f64(k)).permute(1, 0, 2).repeat_interleave(g, dim=0)
    tv = torch.from_numpy(_f64(v)).permute(1, 0, 2).repeat_interleave(g, dim=0)
    mask = torch.arange(L)[None, :] <= (L - n + torch.arange(n))[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
    np.testing.assert_allclose(got, ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def _segment_dense(w, seg):
    qrows = _rows_of(w, seg)
    return oracle.attention_dense(w.q[qrows], w.hist_k[seg.slot], w.hist_v[seg.slot], w.scale)


def _rows_of(w, seg):
    start = 0
    for s in w.segments:
        if s is seg:
            return slice(start, start + s.q_len)
        start += s.q_len
    raise KeyError


SHAPES = [(1, 37), (16, 80), (1, 5), (33, 33), (3, 50), (1, 1), (20, 64)]


def test_paged_equals_contiguous_bitwise(oracle_lib):
    w = W.random_step(11, SHAPES, num_q_heads=6, num_kv_heads=2, head_dim=32)
    st = oracle.prepare_step(w)
    out = oracle.step_attention(w, st)
    for seg in w.segments:
        np.testing.assert_array_equal(out[_rows_of(w, seg)], _segment_dense(w, seg))


def test_tiny_step_paged_equals_bruteforce(oracle_lib):
    w = W.tiny(0)
    st = oracle.prepare_step(w)
    out = oracle.step_attention(w, st)
    for seg in w.segments:
        ref = brute_force(w.q[_rows_of(w, seg)], w.hist_k[seg.slot], w.hist_v[seg.slot], w.scale)
        np.testing.assert_allclose(out[_rows_of(w, seg)], ref, rtol=0, atol=1e-12)


def test_invariant_under_block_permutation(oracle_lib):
    a = W.random_step(5, SHAPES, head_dim=16)
    b = W.random_step(5, SHAPES, head_dim=16)
    perm = np.random.default_rng(99).permutation(a.num_blocks).astype(np.int32)
    b.blocks = {s: perm[ids] for s, ids in a.blocks.items()}
    assert any(not np.array_equal(a.blocks[s], b.blocks[s]) for s in a.blocks)
    oa = oracle.step_attention(a, oracle.prepare_step(a))
    ob = oracle.step_attention(b, oracle.prepare_step(b))
    np.testing.assert_array_equal(oa, ob)


def test_batch_of_one_equals_in_batch(oracle_lib):
    w = W.random_step(6, SHAPES, head_dim=16)
    full = oracle.step_attention(w, oracle.prepare_step(w))
    for seg in w.segments:
        one = W.random_step(6, SHAPES, head_dim=16)
        rows = _rows_of(w, seg)
        one.segments = [seg]
        one.q = w.q[rows]
        got = oracle.step_attention(one, oracle.prepare_step(one))
        np.testing.assert_array_equal(got, full[rows])


def test_packed_order_does_not_matter(oracle_lib):
    w = W.random_step(8, SHAPES, head_dim=16)
    full = oracle.step_attention(w, oracle.prepare_step(w))
    r = W.random_step(8, SHAPES, head_dim=16)
    order = [6, 0, 3, 5, 1, 4, 2]
    r.segments = [w.segments[i] for i in order]
    r.q = np.concatenate([w.q[_rows_of(w, w.segments[i])] for i in order])
    got = oracle.step_attention(r, oracle.prepare_step(r))
    for seg in w.segments:
        np.testing.assert_array_equal(got[_rows_of(r, seg)], full[_rows_of(w, seg)])


def test_slot_reuse_leaves_other_slots_bitwise(oracle_lib):
    """B finishes; its blocks go to a new sequence D in the same slot. A and C do not move."""
    w = W.tiny(0)
    st = oracle.prepare_step(w)
    before = oracle.step_attention(w, st)
    a_c_blocks = np.concatenate([w.blocks[0], w.blocks[2]])
    pool_a_c = (st.k_pool[a_c_blocks].copy(), st.v_pool[a_c_blocks].copy())

    # D takes B's slot and (in reverse order) B's blocks, with its own history.
    w2 = W.tiny(0)
    rng = np.random.default_rng(3)
    w2.blocks[1] = w.blocks[1][::-1][:3].copy()
    w2.hist_k[1] = _rand(rng, (40, 2, 64))
    w2.hist_v[1] = _rand(rng, (40, 2, 64))
    w2.segments = [W.Segment(1, 8, 40), w.segments[1], w.segments[2]]
    w2.q = np.concatenate([_rand(rng, (8, 4, 64)), w.q[16:]])
    st2 = oracle.prepare_step(w2)
    after = oracle.step_attention(w2, st2)
    np.testing.assert_array_equal(after[8:], before[16:])
    np.testing.assert_array_equal(st2.k_pool[a_c_blocks], pool_a_c[0])
    np.testing.assert_array_equal(st2.v_pool[a_c_blocks], pool_a_c[1])


# ---- closed forms ----------------------------------------------------------

def test_single_key_returns_its_value_exactly(oracle_lib):
    rng = np.random.default_rng(1)
    q, k, v = _rand(rng, (1, 4, 16)), _rand(rng, (1, 2, 16)), _rand(rng, (1, 2, 16))
    out = oracle.attention_dense(q, k, v, 0.25)
    for h in range(4):
        np.testing.assert_array_equal(out[0, h], _f64(v[0, h // 2]))


def test_zero_query_gives_causal_prefix_means(oracle_lib):
    rng = np.random.default_rng(2)
    n, L = 6, 20
    q = np.zeros((n, 4, 16), np.uint16)
    k, v = _rand(rng, (L, 2, 16)), _rand(rng, (L, 2, 16))
    out = oracle.attention_dense(q, k, v, 0.25)
    vf = _f64(v)
    for i in range(n):
        p = L - n + i
        for h in range(4):
            np.testing.assert_allclose(out[i, h], vf[: p + 1, h // 2].mean(axis=0), rtol=0, atol=1e-14)


def test_equal_keys_give_uniform_weights(oracle_lib):
    rng = np.random.default_rng(3)
    L = 25
    q = _rand(rng, (1, 2, 8))
    k = np.repeat(_rand(rng, (1, 1, 8)), L, axis=0)
    v = _rand(rng, (L, 1, 8))
    out = oracle.attention_dense(q, k, v, 0.5)
    np.testing.assert_allclose(out[0, 0], _f64(v)[:, 0].mean(axis=0), rtol=0, atol=1e-14)


def test_dominant_key_selects_its_value(oracle_lib):
    rng = np.random.default_rng(4)
    L, d = 30, 8
    k = np.zeros((L, 1, d), np.uint16)
    star = 17
    k[star, 0, :] = W.f32_to_bf16_bits(np.full(d, 8.0, np.float32))
    q = W.f32_to_bf16_bits(np.full((1, 1, d), 8.0, np.float32))  # score 512*scale vs 0
    v = _rand(rng, (L, 1, d))
    out = oracle.attention_dense(q, k, v, 1.0)
    np.testing.assert_allclose(out[0, 0], _f64(v)[star, 0], rtol=0, atol=1e-12)


# ---- cache write and slot mapping -----------------------------------------

def test_block_table_example_from_the_page(oracle_lib):
    g = golden("block_table_example.json")
    bs = 16
    names = list(g["tables"])
    bt = np.full((len(names), 4), -1, np.int32)
    for i, nm in enumerate(names):
        bt[i, : len(g["tables"][nm])] = g["tables"][nm]
    used = sorted(sum(g["tables"].values(), []) + g["free_pool"])
    assert used == list(range(10))
    for i, nm in enumerate(names):
        n_tok = len(g["tables"][nm]) * bs
        pos = np.arange(n_tok, dtype=np.int32)
        sm = oracle.slot_mapping(bt, np.full(n_tok, i, np.int32), pos, bs, 10)
        # every token of logical block j lands in physical block tables[nm][j], rows in order
        np.testing.assert_array_equal(sm // bs, np.repeat(g["tables"][nm], bs))
        np.testing.assert_array_equal(sm % bs, np.tile(np.arange(bs), len(g["tables"][nm])))


def test_cache_write_touches_only_mapped_rows(oracle_lib):
    rng = np.random.default_rng(5)
    nb, hkv, bs, d = 6, 2, 4, 8
    kp = np.full((nb, hkv, bs, d), oracle.SENTINEL, np.uint16)
    vp = kp.copy()
    mapping = np.array([5, -1, 17, 0, 23], np.int64)
    kn, vn = _rand(rng, (5, hkv, d)), _rand(rng, (5, hkv, d))
    oracle.cache_write(kp, vp, kn, vn, mapping)
    written = np.zeros((nb, bs), bool)
    for t, s in enumerate(mapping):
        if s < 0:
            continue
        written[s // bs, s % bs] = True
        np.testing.assert_array_equal(kp[s // bs, :, s % bs], kn[t])
        np.testing.assert_array_equal(vp[s // bs, :, s % bs], vn[t])
    assert (kp.transpose(0, 2, 1, 3)[~written] == oracle.SENTINEL).all()
    assert (vp.transpose(0, 2, 1, 3)[~written] == oracle.SENTINEL).all()


def test_cache_write_rejects_rows_past_the_pool(oracle_lib):
    kp = np.zeros((2, 1, 4, 8), np.uint16)
    with pytest.raises(oracle.OracleError):
        oracle.cache_write(kp, kp.copy(), np.zeros((1, 1, 8), np.uint16),
                           np.zeros((1, 1, 8), np.uint16), np.array([8], np.int64))


def test_paged_attention_rejects_bad_block_ids(oracle_lib):
    w = W.tiny(0)
    st = oracle.prepare_step(w)
    bt = st.block_tables.copy()
    bt[0, 1] = 99
    with pytest.raises(oracle.OracleError):
        oracle.attention_paged(w.q, st.packed.cu_seqlens_q, st.packed.seq_slot, st.context_lens, bt,
                               st.k_pool, st.v_pool, w.scale, num_q_heads=4)


def test_sentinel_never_reaches_outputs(oracle_lib):
    w = W.tiny(0)
    out = oracle.step_attention(w, oracle.prepare_step(w))
    assert np.isfinite(out).all()


def test_packing_example_from_the_page(oracle_lib):
    g = golden("packing_example.json")
    segs = [(i, s["rows"], s["rows"] + 7) for i, s in enumerate(g["segments"])]
    p = oracle.pack(segs)
    widths = np.diff(p.cu_seqlens_q)
    np.testing.assert_array_equal(widths, [s["rows"] for s in g["segments"]])
    assert p.cu_seqlens_q[-1] == 512 + 512 + 180 + 1 + 1  # no padding of E
    np.testing.assert_array_equal(p.seq_slot, np.arange(5))


def test_row_mask_computes_only_selected_rows(oracle_lib):
    w = W.tiny(0)
    st = oracle.prepare_step(w)
    full = oracle.step_attention(w, st)
    part = oracle.step_attention(w, st, rows=[0, 15, 17])
    np.testing.assert_array_equal(part[[0, 15, 17]], full[[0, 15, 17]])
    assert np.isnan(part[1]).all()


def test_thread_count_does_not_change_results(oracle_lib):
    w = W.random_step(12, SHAPES, head_dim=16)
    st = oracle.prepare_step(w)
    one = oracle.step_attention(w, st, threads=1)
    many = oracle.step_attention(w, st, threads=5)
    np.testing.assert_array_equal(one, many)


# ---- the churn replay's scheduling rules ------------------------------------

class _Req:
    def __init__(self, rid, arrival_step, prompt_len, output_len, priority=0, prefix=(-1, 0)):
        self.rid, self.arrival_step = rid, arrival_step
        self.prompt_len, self.output_len = prompt_len, output_len
        self.priority = priority
        self.prefix_id, self.prefix_len = prefix


def _run_steps(r, n):
    out = []
    for _ in range(n):
        rows = r.plan()
        out.append(rows)
        r.commit(rows)
    return out


# ---- budget rules (mlxcel manual, §Preemptive eviction and the decode-headroom
# section), hand-worked scenarios ---------------------------------------------

def test_watermark_holds_back_admission_only_while_decoding():
    # A (prompt 15: one block with its first decode row) decodes from step 1; B arrives at step 1.
    # 100 blocks, F = 0.10: B is admitted only if 99 free - its blocks >= 10.
    def live_after(b_blocks, watermark=0.10, with_a=True):
        reqs = ([_Req(0, 0, 15, 50)] if with_a else []) + [_Req(1, 1 if with_a else 0, b_blocks * 16 - 1, 1)]
        r = churn.ChurnReplay(reqs, max_slots=4, num_blocks=100, block_size=16, watermark=watermark)
        _run_steps(r, 1 if not with_a else 1)
        r.plan()
        return [x.rid for x in r.live], [q[1] for q in r.queue]

    assert live_after(85) == ([0, 1], [])   # 99 - 85 = 14 >= 10
    assert live_after(89) == ([0, 1], [])   # 99 - 89 = 10 >= 10: exactly at the floor
    assert live_after(90) == ([0], [1])     # 99 - 90 = 9 < 10: waits
    assert live_after(90, watermark=0.0) == ([0, 1], [])
    # with nothing decoding the watermark does not apply
    r = churn.ChurnReplay([_Req(1, 0, 99 * 16 - 1, 1)], max_slots=4, num_blocks=100, block_size=16,
                          watermark=0.10)
    r.plan()
    assert [x.rid for x in r.live] == [1]


@pytest.mark.parametrize("policy,victim", [("longest-first", 1), ("lowest-priority", 0)])
def test_priority_preemption_picks_the_policy_victim(policy, victim):
    # two slots; X (prio 0) and Y (prio 0 / 1) decode; Z (prio 2) arrives and finds no slot
    reqs = [_Req(0, 0, 15, 100, 0), _Req(1, 0, 15, 100, 1 if policy == "lowest-priority" else 0),
            _Req(2, 6, 15, 100, 2)]
    r = churn.ChurnReplay(reqs, max_slots=2, num_blocks=64, block_size=16, preemption=policy)
    # X generates one token fewer than Y: Y gets its first token one step earlier
    r.live[0:0] = []
    _run_steps(r, 6)
    by = {x.rid: x for x in r.live}
    gen = {k: v.generated for k, v in by.items()}
    if policy == "longest-first":  # equal priority 0: the most generated tokens, ties to the latest admitted
        assert gen[0] == gen[1]
    rows = r.plan()
    assert r.preempted == [victim] and sorted(x.rid for x in r.live) == sorted({0, 1, 2} - {victim})
    # the victim waits with its prompt plus the tokens it generated, in arrival order
    assert r.queue[0][1] == victim and r.queue[0][2] == 15 + gen[victim] and r.queue[0][6] == gen[victim]
    assert any(x.rid == 2 and x.prefill for x in rows)


# ---- prompt-prefix cache (mlxcel manual, §Paged KV cache and prefix sharing), by hand ----

def test_prefix_donated_in_whole_blocks_and_adopter_charged_for_its_suffix():
    # A's shared prefix is 40 tokens: its whole blocks, 32 tokens (2 blocks), are cached.
    reqs = [_Req(0, 0, 60, 3, prefix=(0, 40)), _Req(1, 1, 50, 2, prefix=(0, 40))]
    r = churn.ChurnReplay(reqs, max_slots=4, num_blocks=64, block_size=16, prefix_cache=2)
    _run_steps(r, 1)                     # A: 4 blocks, prefills 60 rows, donates 2 of them
    assert r.free_blocks == 60 and r.cache[0].nb == 2 and r.cache[0].refs == 2
    rows = r.plan()                      # B adopts: ceil(51 / 16) - 2 = 2 fresh blocks, prefill from 32
    assert r.free_blocks == 58 and r.cache[0].refs == 3
    assert [(x.rid, x.begin, x.n, x.prefill) for x in rows] == [(1, 32, 18, True), (0, 60, 1, False)]
    r.commit(rows)
    _run_steps(r, 1)                     # both retire; the cached prefix keeps its 2 blocks
    assert r.finished == [0, 1] and r.free_blocks == 62 and r.cache[0].refs == 1
    assert r.cache_events == [(0, "donate", 0), (1, "adopt", 0)]


def test_cold_prefix_is_evicted_before_anyone_is_preempted():
    # 4 blocks. A caches 2 blocks and retires; D and E take the other two; D's decode then
    # opens a block: the cold prefix goes, nobody is preempted.
    reqs = [_Req(0, 0, 33, 2, prefix=(0, 32)), _Req(1, 1, 14, 50), _Req(2, 2, 14, 50)]
    r = churn.ChurnReplay(reqs, max_slots=4, num_blocks=4, block_size=16, prefix_cache=2)
    _run_steps(r, 4)
    assert r.free_blocks == 0 and r.cache[0].refs == 1
    r.plan()
    assert r.cache_events[-1] == (4, "drop-headroom", 0) and r.preempted == [] and 0 not in r.cache
    assert r.free_blocks == 1  # the 2 freed blocks, minus the one D's row opens


def test_admission_evicts_cold_prefixes_but_spares_the_heads_own():
    base = [_Req(0, 0, 33, 2, prefix=(0, 32))]
    # a head with no prefix needing 3 blocks (2 free): the cold prefix goes
    r = churn.ChurnReplay(base + [_Req(1, 2, 40, 2)], max_slots=4, num_blocks=4, block_size=16, prefix_cache=2)
    _run_steps(r, 2)
    r.plan()
    assert r.cache_events[-1] == (2, "drop-admission", 0) and [x.rid for x in r.live] == [1]
    # a head that would adopt that prefix (3 fresh blocks on top of it) waits instead
    r = churn.ChurnReplay(base + [_Req(1, 2, 70, 2, prefix=(0, 32))], max_slots=4, num_blocks=4, block_size=16,
                          prefix_cache=2)
    _run_steps(r, 2)
    r.plan()
    assert 0 in r.cache and r.live == [] and [q[1] for q in r.queue] == [1]


def test_full_prefix_cache_drops_the_least_recently_used():
    reqs = [_Req(0, 0, 20, 1, prefix=(0, 16)), _Req(1, 1, 20, 1, prefix=(1, 16))]
    r = churn.ChurnReplay(reqs, max_slots=4, num_blocks=8, block_size=16, prefix_cache=1)
    _run_steps(r, 2)
    assert r.cache_events == [(0, "donate", 0), (1, "drop-capacity", 0), (1, "donate", 1)]
    assert list(r.cache) == [1] and r.free_blocks == 7


def test_decode_headroom_preempts_the_least_progress():
    # 4 blocks in all: A and B each reserve 1 (prompt 14 + 1 row) and decode into block 2 at position 16
    reqs = [_Req(0, 0, 14, 50), _Req(1, 0, 14, 50), _Req(2, 1, 14, 50)]
    r = churn.ChurnReplay(reqs, max_slots=4, num_blocks=4, block_size=16)
    _run_steps(r, 1)          # A, B prefill (generated 1 each); C not yet arrived
    _run_steps(r, 1)          # C admitted (1 block, free 1) and prefills; A, B decode at 14
    rows = r.plan()           # A, B at 15: still in block 1
    r.commit(rows)
    rows = r.plan()           # A, B open block 2 (two blocks, one free): C has the least progress
    assert r.preempted == [2] and {x.rid for x in rows} == {0, 1}
    assert r.free_blocks == 0 and r.queue[0][1] == 2


def test_re_prefill_resumes_where_the_request_stopped():
    reqs = [_Req(0, 0, 14, 6), _Req(1, 0, 14, 50), _Req(2, 1, 14, 50)]
    r = churn.ChurnReplay(reqs, max_slots=4, num_blocks=4, block_size=16)
    seen_gen, refill = {}, None
    for _ in range(12):  # C: prefill, one decode, preempted at its first block crossing, back at step 6
        rows = r.plan()
        if r.preempted and 2 not in seen_gen:
            seen_gen[2] = r.queue[0][6]  # generated tokens kept while it waits
        for x in rows:
            if x.rid == 2 and 2 in seen_gen and refill is None:
                refill = x
        r.commit(rows)
    assert r.preempted[0] == 2 and 0 in r.finished
    # once back, C prefills its prompt plus the tokens it had generated, from position 0
    g = seen_gen[2]
    assert g >= 1 and refill.prefill and refill.begin == 0 and refill.n == 14 + g
    c = next(x for x in r.live if x.rid == 2)
    assert c.decoding and c.generated == g + 1 + (c.pos - (14 + g))


def test_chunk_schedule_example_from_the_page():
    g = golden("chunk_schedule_example.json")
    # A (rid 0) and B (rid 1) are decoding with long outputs; C (rid 2) arrives.
    reqs = [_Req(0, 0, 16, 10_000), _Req(1, 0, 16, 10_000), _Req(2, 1, g["prompt_tokens"]["C"], 50)]
    r = churn.ChurnReplay(reqs, max_slots=8, num_blocks=10_000, block_size=16)
    r.commit(r.plan())  # step 0: A and B prefill together
    steps = []
    while True:
        rows = r.plan()
        steps.append(rows)
        r.commit(rows)
        if not any(x.prefill for x in rows):
            break
    for want, got in zip(g["printed_steps"], steps):
        pre = [x for x in got if x.prefill]
        assert [(x.rid, x.begin, x.begin + x.n) for x in pre] == [(2, want["prefill"][1], want["prefill"][2])]
        assert [x.rid for x in got if not x.prefill] == [0, 1]
    final = steps[-2]
    assert [x.begin + x.n for x in final if x.prefill] == [g["final"]["prefill_ends_at"]]
    assert [x.rid for x in final if not x.prefill] == [0, 1]
    assert [x.rid for x in steps[-1]] == [0, 1, 2] and all(x.n == 1 for x in steps[-1])
    assert all(x.n == g["chunk"] for s in steps[:-2] for x in s if x.prefill)


def test_fifo_admission_example_from_the_page():
    g = golden("fifo_admission_example.json")
    bs = 16
    d_tokens = g["queue"][0]["blocks"] * bs - 1  # needs ceil((p + 1) / bs) = 100 blocks
    e_tokens = g["queue"][1]["blocks"] * bs - 1
    reqs = [_Req(0, 0, d_tokens, 1), _Req(1, 0, e_tokens, 1)]
    r = churn.ChurnReplay(reqs, max_slots=8, num_blocks=g["free_blocks"], block_size=bs)
    assert r.plan() == []
    assert [q[1] for q in r.queue] == [0, 1] and r.free_blocks == g["free_blocks"]  # (arrival, rid, ...)


def test_chunk_size_rule_from_the_page():
    g = golden("chunk_size_rule.json")
    r = churn.ChurnReplay([_Req(0, 0, 8192, 3)], max_slots=4, num_blocks=4096, block_size=16)
    first = r.plan()
    assert [x.n for x in first] == [g["no_decoder"]]
    r2 = churn.ChurnReplay([_Req(0, 0, 16, 100), _Req(1, 1, 8192, 3)], max_slots=4,
                           num_blocks=4096, block_size=16)
    r2.commit(r2.plan())
    rows = r2.plan()
    assert [x.n for x in rows if x.prefill] == [g["decoding"]]


def test_retirement_returns_slot_and_blocks():
    reqs = [_Req(0, 0, 20, 1), _Req(1, 0, 40, 3)]
    r = churn.ChurnReplay(reqs, max_slots=2, num_blocks=100, block_size=16)
    rows = r.plan()
    assert [(x.rid, x.n) for x in rows] == [(0, 20), (1, 40)]
    assert r.free_blocks == 100 - 2 - 3
    assert r.commit(rows) == [0]           # one output token: done after its prompt
    assert r.free_slots == 1 and r.free_blocks == 100 - 3
    assert [(x.rid, x.begin) for x in r.plan()] == [(1, 40)]
    r.commit([churn.Row(1, 40, 1, False)])
    rows = r.plan()
    assert r.commit(rows) == [1]
    assert r.free_slots == 2 and r.free_blocks == 100


def test_decode_growth_takes_a_block_at_block_boundaries():
    r = churn.ChurnReplay([_Req(0, 0, 31, 40)], max_slots=1, num_blocks=10, block_size=16)
    r.commit(r.plan())          # prompt of 31 -> reservation ceil(32/16) = 2 blocks
    assert r.free_blocks == 8
    r.commit(r.plan())          # decode row at position 31: still block 1
    assert r.free_blocks == 8
    r.commit(r.plan())          # position 32 opens block 2
    assert r.free_blocks == 7


# ---- mutation checks: the pins above notice plausible mistakes --------------

MUTANTS = {
    "causal boundary excludes the diagonal": ("for (int32_t j = 0; j <= p; ++j) {\n        const uint16_t *kj",
                                              "for (int32_t j = 0; j < p + (p == 0); ++j) {\n        const uint16_t *kj"),
    "scale dropped": ("scores[j] = scale * dot;", "scores[j] = dot;"),
    "wrong kv head for grouped queries": ("dense_ctx c = {k, v, num_kv_heads, head_dim, h / G};",
                                          "dense_ctx c = {k, v, num_kv_heads, head_dim, h % num_kv_heads};"),
    "row inside block off by one": ("int64_t row = j % c->block_size;",
                                    "int64_t row = (j + 1) % c->block_size;"),
    "diagonal term dropped from the denominator": ("denom += w;", "denom += (j < p ? w : 0.0);"),
    "keys read in place of values": ("const uint16_t *vj = value_row(ctx, j);", "const uint16_t *vj = key_row(ctx, j);"),
    "position of chunk rows shifted": ("int32_t p = L - n + i;\n        for (int32_t h = g * G;",
                                       "int32_t p = L - n + i - (i > 0);\n        for (int32_t h = g * G;"),
}


def _build_mutant(tmp_path, old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "pkv_oracle.c")).read()
    assert src.count(old) == 1, old
    path = tmp_path / "m.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "m.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", "-o", str(so), str(path), "-lm"],
                   check=True)
    return so


def _pins_pass(so) -> bool:
    """Run a few pins against the shared object at ``so``; True if all hold."""
    saved_lib, saved_build = oracle._lib, oracle.build
    oracle._lib = None
    oracle.build = lambda force=False: str(so)
    try:
        oracle._load()
        test_dense_matches_bruteforce(None, 16, 80, 4, 2, 64)
        test_dense_matches_bruteforce(None, 3, 19, 8, 1, 8)
        test_tiny_step_paged_equals_bruteforce(None)
        test_paged_equals_contiguous_bitwise(None)
        return True
    except AssertionError:
        return False
    finally:
        oracle._lib, oracle.build = saved_lib, saved_build


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(oracle_lib, tmp_path, name):
    old, new = MUTANTS[name]
    so = _build_mutant(tmp_path, old, new)
    assert not _pins_pass(so), f"pins missed the planted mistake: {name}"
    assert _pins_pass(oracle.build()), "the unmodified oracle must pass its pins"


# ---- the churn replay's row-subset attention ---------------------------------
# The churn checks compare kernel rows with ContiguousHistory.attend(keep=...),
# which computes each kept row as the last row of a shorter prefix. Pinned here
# against the brute force over the whole contiguous history (a masked score
# matrix, no prefix slicing), with histories built by several appends.

def _subset_pin(history_cls) -> bool:
    """True if ``history_cls.attend(keep=...)`` matches the brute force on every case."""
    rng = np.random.default_rng(2024)
    for n, chunks, hq, hkv, d in [(1, [5, 1], 4, 2, 16), (7, [16, 9, 7], 6, 2, 32), (64, [100, 37, 64], 4, 1, 16)]:
        h = history_cls()
        for c in chunks:
            h.append(7, _rand(rng, (c, hkv, d)), _rand(rng, (c, hkv, d)))
        k, v = np.concatenate(h.k[7]), np.concatenate(h.v[7])
        q = _rand(rng, (n, hq, d))
        keep = sorted({0, n - 1} | set(int(i) for i in rng.choice(n, size=min(n, 5), replace=False)))
        for mult in (1.0, 8.0):
            qq = W.f32_to_bf16_bits(W.bf16_bits_to_f32(q) * mult)
            got = h.attend(7, qq, 1 / np.sqrt(d), keep=keep)
            ref = brute_force(qq, k, v, 1 / np.sqrt(d))
            if not np.allclose(got[keep], ref[keep], rtol=0, atol=1e-12):
                return False
            rest = [i for i in range(n) if i not in keep]
            if rest and not np.isnan(got[rest]).all():
                return False
            if not np.allclose(h.attend(7, qq, 1 / np.sqrt(d)), ref, rtol=0, atol=1e-12):
                return False
    return True


def test_history_subset_rows_match_bruteforce(oracle_lib):
    assert _subset_pin(churn.ContiguousHistory)


HISTORY_MUTANTS = {
    "kept row sees one key fewer": ("L = len(k) - n + i + 1", "L = len(k) - n + i"),
    "kept row sees one key more": ("L = len(k) - n + i + 1", "L = min(len(k), len(k) - n + i + 2)"),
    "kept row takes the first row's prefix": ("L = len(k) - n + i + 1", "L = len(k) - n + 1"),
    "kept row answers with the wrong query": ("attention_dense(q_rows[i:i + 1]", "attention_dense(q_rows[n - 1:n]"),
}


@pytest.mark.parametrize("name", sorted(HISTORY_MUTANTS))
def test_history_subset_planted_mistakes_are_caught(oracle_lib, name):
    import inspect
    import textwrap

    old, new = HISTORY_MUTANTS[name]
    src = textwrap.dedent(inspect.getsource(churn.ContiguousHistory.attend))
    assert src.count(old) == 1, old
    ns = dict(vars(churn))
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    mutant = type("MutantHistory", (churn.ContiguousHistory,), {"attend": ns["attend"]})
    assert not _subset_pin(mutant), f"pin missed the planted mistake: {name}"
